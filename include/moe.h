/*
 * bit_moe_expert_gb300 -- C ABI of a GB300 (sm_103a) mixture-of-experts layer
 * whose expert weights are 4-bit groupwise-affine quantised.
 *
 * The operation (sources: the web pages "Perplexity's Lily Beats MLX-LM on
 * MacBook M5. Because It Only Runs One Model." -- sections "Why
 * Qwen3.6-35B-A3B is a weird workload", "Prefill: keep routing on the GPU,
 * dequantize in flight" and "Decode: minimize bytes per token" -- and
 * "Perplexity builds a custom engine for Qwen on M5 Macs"):
 *
 *   routing   for each token t, the k experts with the largest router logits
 *             (ties to the lower expert index) and weights w = softmax over
 *             the experts renormalised over the selected k;
 *   layout    a histogram of assignments per expert, its exclusive prefix
 *             scan, a stable scatter that groups each expert's rows together
 *             and a tile block map, all on the GPU with no host round trip;
 *   experts   Y[t] = sum_j w[t][j] * FFN_{e(t,j)}(x_t) + FFN_shared(x_t), with
 *             FFN(x) = (silu(x Wg^T) * (x Wu^T)) Wd^T and every weight
 *             w = q * scale + bias, q a 4-bit code, one bf16 scale and one
 *             bf16 bias per group of 64 consecutive weights along K.
 *
 * Conventions for every entry point
 *   - All array pointers are DEVICE pointers, owned by the caller, and must be
 *     16-byte aligned.  The library never allocates, frees or synchronises on
 *     these paths (moe_check_status is the one synchronising call).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL means the legacy
 *     default stream) and may be captured into a CUDA graph.
 *   - Kernels are launched with programmatic dependent launch: a call's kernel
 *     may start while the previous kernel on the stream is finishing, and
 *     reads weights (expert codes and group parameters, router rows) before
 *     waiting for it; activations, logits and routing are read only after.
 *     Weights written by a kernel must therefore be separated from the call
 *     that reads them by something other than a kernel launch (an event wait,
 *     a copy, a memset, another stream's completion), or the environment
 *     variable MOE_PDL=0 turns the early starts off.
 *   - Argument checks happen on the host before anything is launched; a failed
 *     check returns a status and launches nothing.  Errors that only the device
 *     can see (a non-finite logit, a bounded wait that expired) are recorded in
 *     a status word at the start of the workspace and read by moe_check_status.
 *   - Integers in device arrays are int32 (no int64 anywhere).
 *   - bf16 values travel as uint16_t bit patterns.
 */
#ifndef BIT_MOE_EXPERT_GB300_MOE_H
#define BIT_MOE_EXPERT_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Identical to cudaStream_t. */
typedef struct CUstream_st* moe_stream;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a size, pointer or alignment precondition failed */
  MOE_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels implement */
  MOE_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or smaller than queried */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device-side wait expired (device status word) */
  MOE_ERR_NONFINITE = 6    /* a router logit was NaN or infinite (device status word) */
} moe_status;

/* Human-readable name of a status.  Never NULL. */
const char* moe_status_string(moe_status s);

/* ------------------------------------------------------------------ weights
 * One stacked packed matrix of E experts with N rows and K columns (K a
 * multiple of 64), b = 4, 3 or 2 bits per code:
 *   q   uint32 [E][K/64][N][2b]  the codes, group-major: the 2b words of row
 *                            n, columns 64g .. 64g+63 sit at [e][g][n][..];
 *                            inside a word the codes are interleaved so that
 *                            one mask takes two adjacent columns into the
 *                            halves of a register: with 4-bit codes the code
 *                            of column 8j+2p sits in bits 4p and that of
 *                            column 8j+2p+1 in bits 4p+16 (p = 0..3); with
 *                            2-bit codes the code of column 16j+2p sits in
 *                            bits 2p and that of column 16j+2p+1 in bits
 *                            2p+16 (p = 0..7).  3-bit codes are two planes
 *                            in the row's six words: words 0..3 hold the low
 *                            two bits exactly as 2-bit codes, and the high
 *                            bit of column 16j+2p+h (h = 0, 1) sits in bit
 *                            16h + 8(j%2) + p of word 4 + j/2.  Build it once
 *                            per weight set with moe_prepack_codes (4-bit)
 *                            or moe_prepack_codes_bits from the row-major
 *                            [E][N][K*b/32] checkpoint layout (each row one
 *                            bit stream, code k at bits b*k .. b*k+b-1, so a
 *                            3-bit code may straddle two words);
 *   sb  uint32 [E][K/64][N]  the group parameters, transposed so one group of
 *                            many rows is contiguous: bits 0..15 hold the bf16
 *                            scale and bits 16..31 the bf16 bias of rows n,
 *                            columns 64g .. 64g+63.  Build it once per weight
 *                            set with moe_prepack_scales.
 * Gate and up projections have N = I, K = d; the down projection has N = d,
 * K = I.
 */
typedef struct {
  const uint32_t* q;
  const uint32_t* sb;
} moe_qmat;

typedef struct {
  moe_qmat gate;
  moe_qmat up;
  moe_qmat down;
  int n_experts;
  int bits; /* bits per code of all three matrices: 4 (or 0), 3 or 2; a
               shared expert has the routed experts' width */
} moe_experts;

/* Bytes of the sb array for E experts of an N x K matrix: E * (K/64) * N * 4. */
size_t moe_prepack_bytes(int E, int N, int K);

/* Reorder row-major codes q [E][N][K/8] (the checkpoint layout: row n holds
 * its K/8 words) into the group-major layout qp [E][K/64][N][8] that
 * moe_forward reads: the 32-byte piece of every row for one group of 64
 * columns becomes contiguous, so one group of many rows is one contiguous
 * block, and the codes inside each word are interleaved (see above).  A pure
 * data movement (same size, E*N*K/2 bytes); bit-exact.  Both
 * pointers 16-byte aligned device memory, not overlapping.  Sizes: E >= 1,
 * N >= 1, K a positive multiple of 64.  Returns MOE_ERR_INVALID_ARG on a bad
 * size or pointer. */
moe_status moe_prepack_codes(const uint32_t* q, int E, int N, int K, uint32_t* qp, moe_stream stream);

/* moe_prepack_codes for b = `bits` bits per code (4, 3 or 2): q
 * [E][N][K*b/32] -> qp [E][K/64][N][2b], the codes of each word interleaved
 * (3-bit codes split into planes; see above); E*N*K*b/8 bytes.
 * MOE_ERR_INVALID_ARG for any other width. */
moe_status moe_prepack_codes_bits(const uint32_t* q, int E, int N, int K, int bits, uint32_t* qp,
                                  moe_stream stream);

/* Transpose and interleave per-group bf16 scale and bias, both laid out
 * [E][N][K/64] as in the checkpoint, into sb [E][K/64][N] (see above).  A pure
 * data movement; bit-exact.  Sizes: E >= 1, N >= 1, K a positive multiple of
 * 64.  Returns MOE_ERR_INVALID_ARG on a bad size or pointer. */
moe_status moe_prepack_scales(const uint16_t* scale, const uint16_t* bias, int E, int N, int K,
                              uint32_t* sb, moe_stream stream);

/* Expanded weights of one prepacked matrix m (E experts, N rows, K columns, b =
 * `bits` bits per code): W[e][n][k] = q * scale + bias as fp16 (uint16 bit
 * patterns, row-major [E][N][K], 2*E*N*K bytes, caller-owned device memory,
 * 16-byte aligned).  The value is formed in fp32 with one fused multiply-add
 * and rounded to fp16 once (exact for the synthetic weights, whose values
 * need at most 11 significant bits); values beyond the fp16 range become
 * infinities.  The layer itself never does this -- "Perplexity's Lily Beats
 * MLX-LM on MacBook M5", section "Prefill: keep routing on the GPU, dequantize
 * in flight": dequantising inside the GEMM instead of expanding the weights
 * first gave +77.4% at 512 tokens -- it serves that comparison's unfused arm
 * and checks of a weight set.  Asynchronous; allocates nothing.
 * MOE_ERR_INVALID_ARG on a bad size, width or pointer. */
moe_status moe_dequant_experts(const moe_qmat* m, int E, int N, int K, int bits, uint16_t* W, moe_stream stream);

/* ------------------------------------------------------------------ routing
 * Output arrays of moe_route, all caller-owned device memory:
 *   ids        int32 [T][k]  selected experts, descending logit, lower index
 *                            first among equal logits
 *   w          float [T][k]  renormalised routing weights: exp(l - l_max) summed
 *                            over the selection in fp64, rounded once to fp32
 *   counts     int32 [E]     assignments per expert (sum = T*k)
 *   offsets    int32 [E+1]   exclusive prefix sum of counts; offsets[E] = T*k
 *   perm       int32 [T*k]   permuted row p holds assignment a = t*k + j;
 *                            rows of one expert are contiguous
 *                            ([offsets[e], offsets[e+1])) and in ascending a
 *   inv_perm   int32 [T*k]   inv_perm[perm[p]] = p
 *   block_map  int32 [moe_route_max_blocks(...)][3]  one entry per tile:
 *                            (expert, first permuted row, rows <= block_rows),
 *                            experts ascending, tiles of an expert in order
 *   num_blocks int32 [1]     number of valid block_map entries
 * block_rows records the tile height moe_route was called with; moe_forward
 * reads it.  When T = 0 the arrays of length T*k may be NULL.
 */
typedef struct {
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* block_map;
  int32_t* num_blocks;
  int block_rows;
} moe_routing;

/* Upper bound on num_blocks: ceil(T*k / block_rows) + E. */
int moe_route_max_blocks(int T, int E, int k, int block_rows);

/* Workspace bytes moe_route needs.  A workspace is caller-owned device memory,
 * 256-byte aligned, zero-filled ONCE before its first use; every call leaves it
 * ready for the next.  Calls sharing a workspace must be stream-ordered. */
size_t moe_route_workspace_bytes(int T, int E, int k);

/* fp32 router logits [T][E] (row-major) -> all arrays of *out.  One kernel
 * launch, no host synchronisation.  Preconditions: T >= 0 (T = 0 writes zero
 * counts, offsets and num_blocks), 1 <= E <= 1024, 1 <= k <= min(E, 32),
 * 1 <= block_rows <= 128 (the tile height of moe_forward's tensor-core path,
 * T > 4, whose MMA N is the tile's row count rounded up to 16).  Logits must
 * be finite: a NaN or infinity leaves a
 * deterministic but meaningless selection and records MOE_ERR_NONFINITE in
 * the workspace status word.  Sets out->block_rows. */
moe_status moe_route(const float* logits, int T, int E, int k, int block_rows, moe_routing* out,
                     void* ws, size_t ws_bytes, moe_stream stream);

/* ------------------------------------------------------------------ routing without a workspace
 * moe_route_noalloc: no counterpart on the source pages.  It computes exactly
 * what moe_route computes, into the same caller-owned output arrays, for
 * callers that cannot allocate device memory -- for example code hosted by a
 * framework that owns all device memory and forbids cudaMalloc once it has
 * started, or code that runs while a stream is being captured into a CUDA
 * graph, where allocating is not allowed.  Instead of a workspace it uses one
 * scratch array compiled into the library: MOE_ROUTE_NOALLOC_SCRATCH_BYTES of
 * device memory on every GPU that loads the library, held until the process
 * exits.
 *   - Limits: T*k <= MOE_ROUTE_NOALLOC_MAX_ASSIGNMENTS and
 *     ceil(T/32)*E <= MOE_ROUTE_NOALLOC_MAX_HIST; larger sizes return
 *     MOE_ERR_UNSUPPORTED and launch nothing.  Other preconditions and errors
 *     as for moe_route.
 *   - The first call on a device looks up the scratch array's device address
 *     (with that device current).  Make that first call before any stream
 *     capture.  The address is kept per device together with the CUDA context
 *     it belongs to; after cudaDeviceReset (a new context) the next call looks
 *     it up again, so that call, too, must come before any capture.
 *   - Every call shares the one array and leaves its contents behind; each call
 *     first clears the part that must start at zero (cudaMemsetAsync on
 *     `stream`).  Calls that overlap on the GPU -- on different streams or from
 *     different host threads -- race and produce wrong results: keep them
 *     ordered on one stream.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - Device-side errors (a non-finite logit: MOE_ERR_NONFINITE; a bounded
 *     wait of the routing kernel that expired: MOE_ERR_TIMEOUT, after which
 *     the outputs are meaningless) are recorded in a status word inside the
 *     scratch array.  The word keeps the first error until
 *     moe_route_noalloc_check_status reads and clears it; the call itself
 *     still returns MOE_OK, because it does not wait for the GPU. */
#define MOE_ROUTE_NOALLOC_MAX_ASSIGNMENTS 65536
#define MOE_ROUTE_NOALLOC_MAX_HIST 65536
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (256 + 4 * (MOE_ROUTE_NOALLOC_MAX_HIST + MOE_ROUTE_NOALLOC_MAX_ASSIGNMENTS))
moe_status moe_route_noalloc(const float* logits, int T, int E, int k, int block_rows, moe_routing* out,
                             moe_stream stream);

/* Synchronises `stream`, returns the first device-side error recorded by
 * moe_route_noalloc calls on the current device since the last check
 * (MOE_OK if none) and clears it.  Allocates nothing.  For tests and
 * debugging, like moe_check_status; it must not run while a stream is being
 * captured. */
moe_status moe_route_noalloc_check_status(moe_stream stream);

/* ------------------------------------------------------------------ experts
 * Workspace bytes moe_forward needs for these sizes (I_shared = 0: no shared
 * expert).  Same rules as the routing workspace: zero-filled once before first
 * use, 256-byte aligned, one in-flight call per workspace. */
size_t moe_forward_workspace_bytes(int T, int d, int I, int E, int k, int I_shared);

/* bf16 X [T][d] (row-major) -> bf16 Y [T][d].
 *   routed   E = routed->n_experts experts, I columns of intermediate
 *   shared   NULL, or one always-on expert (n_experts = 1) with I_shared
 *   r        the routing written by moe_route for the same T, E, k on this
 *            stream (block_rows <= 128, as moe_route accepts; a routing
 *            struct claiming more is refused with MOE_ERR_UNSUPPORTED)
 * Preconditions: T >= 0 (T = 0 does nothing), d, I and I_shared multiples of
 * 64 (I_shared = 0 iff shared is NULL), 1 <= k <= min(E, 32), E <= 1024.
 * Path: T <= 4 runs the decode kernel (every active expert's bytes streamed
 * once, one launch; warp-level tensor-core MMAs fed from the 4-bit codes, the
 * gate/up projections in bf16 with x exact, h rounded to fp16 for the down
 * projection; with one token and d <= 2048 the gate/up codes are loaded
 * straight into registers, MOE_DECODE_REG=0 keeps them on the shared-memory
 * stage ring the other token counts use, with the same result bits); larger T runs the grouped tensor-core GEMM (tcgen05,
 * dequantisation fused, SwiGLU fused into the gate/up epilogue; the down
 * projection writes each expert's output rows in fp32 and a separate combine
 * kernel sums each token's rows with its routing weights and the shared
 * expert, in slot order, into bf16 Y).  The
 * environment variable MOE_PATH=gemv|gemm overrides the choice (gemv with
 * T > 4 returns MOE_ERR_UNSUPPORTED; for A/B
 * measurements and tests).  Arithmetic: fp32 accumulation; on the GEMM path X,
 * the dequantised weights and the SwiGLU output are rounded to fp16 as
 * tensor-core operands (a value outside the fp16 range is recorded as
 * MOE_ERR_UNSUPPORTED); Y is rounded to bf16 once. */
moe_status moe_forward(const uint16_t* X, int T, int d, int I, int k, const moe_experts* routed,
                       const moe_experts* shared, int I_shared, const moe_routing* r, uint16_t* Y,
                       void* ws, size_t ws_bytes, moe_stream stream);

/* ------------------------------------------------------------------ router projection
 * logits[t][e] = sum_i X[t][i] * W_r[e][i]: the router's score of expert e for
 * token t ("Perplexity's Lily Beats MLX-LM on MacBook M5", section "Why
 * Qwen3.6-35B-A3B is a weird workload": a router scores the 256 experts and
 * picks 8; the score is read as a linear map of the token's hidden state).
 *   X       bf16 [T][d] row-major (device)
 *   W_r     bf16 [E][d] row-major, one row per expert (device, caller-owned)
 *   logits  fp32 [T][E] row-major (device, caller-owned), written
 * Preconditions: T >= 0 (T = 0 does nothing), d a multiple of 64,
 * 1 <= E <= 1024, X and W_r 16-byte aligned.  Arithmetic: bf16 products
 * accumulated in fp32 (on the CUDA cores up to 32 tokens, else on the tensor
 * cores); the additions are not in index order, so the logits agree with an
 * exact sum to within fp32 accumulation error, not bit for bit.  The result
 * does not depend on timing: the same call gives the same bits.  More than
 * 32 tokens with E a multiple of 128, d of 256 and logits 16-byte aligned take
 * the fifth-generation tensor cores (environment variable MOE_ROUTER_TC=0
 * keeps the warp-level MMA kernel, for comparisons); a device-side wait there
 * that gives up leaves NaN in the affected logits, which moe_route then
 * reports as MOE_ERR_NONFINITE.  Asynchronous on `stream`; allocates
 * nothing. */
moe_status moe_router_logits(const uint16_t* X, int T, int d, const uint16_t* W_r, int E, float* logits,
                             moe_stream stream);

/* moe_router_logits, then moe_route on the logits it wrote (two launches on
 * `stream`, the second started by the first on the device).  Same arguments,
 * results and errors as the two calls; `logits` receives the scores. */
moe_status moe_route_x(const uint16_t* X, int T, int d, const uint16_t* W_r, int E, int k, int block_rows,
                       float* logits, moe_routing* out, void* ws, size_t ws_bytes, moe_stream stream);

/* ------------------------------------------------------------------ wide top-K
 * The K largest entries of each row of logits [T][V] (fp32, row-major, device):
 * values [T][K] (fp32) and indices [T][K] (int32), caller-owned device arrays,
 * in descending order, a lower index first among equal values (-0.0 equals
 * +0.0; a value is copied from its entry).  "Squeezing a 26B diffusion LLM onto
 * a Mac", section "The optimizations that worked", item 1: the sampler needs
 * only the top ~64 candidates of 262,144 logits per canvas position, found by
 * a two-stage chunk-max selection that is exact.  Exact here too (no
 * approximation): chunk maxima of 256 entries, the K best chunks, then the top
 * K of their entries.
 * Preconditions: T >= 0 (T = 0 does nothing), 1 <= K <= 64 (MOE_ERR_UNSUPPORTED
 * above), K <= V <= 2^20 (MOE_ERR_UNSUPPORTED above), no NaN entries (a NaN
 * orders above +inf), logits 4-byte aligned.  Asynchronous; allocates
 * nothing. */
moe_status moe_topk_wide(const float* logits, int T, int V, int K, float* values, int32_t* indices,
                         moe_stream stream);

/* ------------------------------------------------------------------ whole layer
 * Workspace bytes moe_layer needs (the forward workspace followed by a routing
 * workspace); same rules: zero-filled once, 256-byte aligned, one in-flight
 * call per workspace. */
size_t moe_layer_workspace_bytes(int T, int d, int I, int E, int k, int I_shared);

/* moe_route followed by moe_forward on the same stream, with the same
 * arguments and results: r receives every routing output and Y the layer
 * output.  E = routed->n_experts.  When the decode kernel takes the call
 * (1 <= T <= 4, E <= 256, its shared-memory plan fits, MOE_PATH not "gemm")
 * this is ONE launch: every CTA of the decode kernel selects the tokens'
 * experts itself with the routing kernel's arithmetic, and one of its CTAs
 * writes the routing outputs.  Otherwise it launches the routing kernel and
 * then the moe_forward kernels.  Device-side errors of both parts go to the
 * status word at the start of ws (read it with moe_check_status(ws, ...)). */
moe_status moe_layer(const float* logits, const uint16_t* X, int T, int d, int I, int k, int block_rows,
                     const moe_experts* routed, const moe_experts* shared, int I_shared, moe_routing* r,
                     uint16_t* Y, void* ws, size_t ws_bytes, moe_stream stream);

/* The whole layer from the hidden state: moe_router_logits(X, W_r) into
 * `logits` (fp32 [T][E], caller-owned), then moe_layer on those logits (two
 * launches on `stream`, or more when moe_layer takes more).  E =
 * routed->n_experts; W_r is bf16 [E][d]; every other argument, result and
 * error as for moe_router_logits and moe_layer. */
moe_status moe_layer_x(const uint16_t* X, int T, int d, const uint16_t* W_r, int I, int k, int block_rows,
                       const moe_experts* routed, const moe_experts* shared, int I_shared, float* logits,
                       moe_routing* r, uint16_t* Y, void* ws, size_t ws_bytes, moe_stream stream);

/* Synchronises `stream`, returns the status recorded in the workspace of a
 * previous moe_route, moe_forward or moe_layer call (MOE_OK if none) and clears it.  For
 * tests and debugging; never needed on the hot path. */
moe_status moe_check_status(void* ws, moe_stream stream);

/* Number of streaming multiprocessors the library sizes its persistent grids
 * for on the current device (0 if no device).  Informational. */
int moe_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif
