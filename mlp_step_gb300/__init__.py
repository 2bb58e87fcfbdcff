"""GB300-native MLP training step: CUDA kernels behind a C ABI, and a thin binding."""
