"""GB300-native ReplaySSM prefix materialization (sm_103a CUDA, C-ABI library)."""
