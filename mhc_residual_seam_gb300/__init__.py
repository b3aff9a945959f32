"""GB300-native delayed mHC seam (sm_103a CUDA behind a C ABI)."""
