"""GB300-native 4-bit groupwise-affine mixture-of-experts layer (sm_103a)."""
