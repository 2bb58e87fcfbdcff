// Softmax cross entropy of one row of at most NC logits held by one thread
// ("Capstone 5: train a network with your CUDA kernels", "The minimum model"
// and "Read the worked reference": subtract the row maximum before
// exponentiating; fp32 throughout).  Shared by the loss epilogue of the
// logits GEMM and by the one-row-per-thread loss kernel, so the two paths give
// bit-identical results.  The maximum and the sum of exponentials are
// pairwise trees over the NC slots (a fixed order, short dependency chains:
// the row is one thread's serial work on the critical path of a step).
#pragma once

#include "common.cuh"

namespace mlp {

struct MaxAt {
  float v;
  int i;
};

// the larger value; among equal values the lower index
__device__ __forceinline__ MaxAt max_at(MaxAt a, MaxAt b) {
  return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

// z: the row's logits in slots [0, C) (others ignored).  label is clamped into
// [0, C).  Returns the row loss m + ln(sum exp(z - m)) - z_label; d receives
// (softmax - onehot) * inv_norm in slots [0, C) and 0 past C; argmax the
// index of the maximum (lowest among ties).
template <int NC>
__device__ __forceinline__ float xent_row_small(const float (&z)[NC], int C, int label,
                                                float inv_norm, float (&d)[NC], int& argmax) {
  label = label < 0 ? 0 : (label >= C ? C - 1 : label);
  MaxAt t[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) t[j] = MaxAt{j < C ? z[j] : -INFINITY, j};
#pragma unroll
  for (int w = NC / 2; w > 0; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = max_at(t[j], t[j + w]);
  const float mx = t[0].v;
  argmax = t[0].i;
  float zy = 0.f;
#pragma unroll
  for (int j = 0; j < NC; ++j)
    if (j == label) zy = z[j];
  float e[NC], s[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    e[j] = j < C ? expf(z[j] - mx) : 0.f;
    s[j] = e[j];
  }
#pragma unroll
  for (int w = NC / 2; w > 0; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) s[j] += s[j + w];
#pragma unroll
  for (int j = 0; j < NC; ++j)
    d[j] = j < C ? (e[j] / s[0] - (j == label ? 1.f : 0.f)) * inv_norm : 0.f;
  return mx + logf(s[0]) - zy;
}

}  // namespace mlp
