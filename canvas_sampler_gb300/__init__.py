"""GB300-native canvas sampler for uniform-state text diffusion (sm_103a CUDA behind a C ABI)."""
