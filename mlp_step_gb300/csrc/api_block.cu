// Placeholder entry points of the block path (filled in by the block kernels).
#include "kernels.cuh"

extern "C" {

size_t mlp_block_workspace_bytes(int T, int d, int hidden) {
  (void)T; (void)d; (void)hidden;
  return 0;
}

mlp_status mlp_block_fwd(const void*, const void*, const void*, int, int, int, float, float, void*,
                         float*, void*) {
  return MLP_ERR_UNSUPPORTED_SHAPE;
}

mlp_status mlp_block_bwd(const void*, const float*, const void*, const void*, const void*, int, int,
                         int, float, float, void*, float*, float*, void*, size_t, void*) {
  return MLP_ERR_UNSUPPORTED_SHAPE;
}

size_t mlp_stack_param_count(int n_blocks, int d, int hidden) {
  if (n_blocks <= 0 || d <= 0 || hidden <= 0) return 0;
  return (size_t)n_blocks * 2 * d * hidden;
}

size_t mlp_stack_workspace_bytes(int, int, int, int) { return 0; }

mlp_status mlp_stack_train_step(int, int, int, int, float, float, const void*, const void*, float*,
                                float*, float*, void*, float, float, float*, void*, size_t, void*) {
  return MLP_ERR_UNSUPPORTED_SHAPE;
}

}  // extern "C"
