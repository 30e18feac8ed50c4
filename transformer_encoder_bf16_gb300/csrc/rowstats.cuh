// rowstats.cuh -- the LayerNorm row arithmetic, shared by the LayerNorm kernel
// and the GEMM that normalises its activation tiles on load, so that both
// produce bit-identical normalised values.
//
// Bias-free LayerNorm ("perf(model): exact Metal speed-ups of the forward pass
// - #45": the encoder has no biases): mean first, then the mean of squared
// deviations about it (two passes), rstd = 1 / sqrt(var + eps), and
// y = ((x - mean) * rstd) * gamma, every operation rounded to fp32 on its own
// (explicit _rn intrinsics: no fused multiply-add, whatever the call site).
#pragma once

#include <cuda_bf16.h>

namespace laya {

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// One warp, one row of 256 * V values: lane holds chunks lane + 32 c (c < V)
// of 8 values each, loaded from `row`.  Returns mean and rstd in every lane.
template <int V>
__device__ __forceinline__ void row_stats(const uint4* row, int lane, float eps, float (&v)[V][8],
                                          float& mean, float& rstd) {
#pragma unroll
  for (int c = 0; c < V; ++c) bf16x8_to_f32(row[lane + 32 * c], v[c]);
  // four independent partial sums per lane (short dependency chains), added
  // in a fixed order, then across the warp
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < V; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) s4[i & 3] = __fadd_rn(s4[i & 3], v[c][i]);
  const float s = __fadd_rn(__fadd_rn(s4[0], s4[1]), __fadd_rn(s4[2], s4[3]));
  mean = __fdiv_rn(warp_allsum(s), static_cast<float>(256 * V));
  float q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < V; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float d = __fsub_rn(v[c][i], mean);
      q4[i & 3] = __fadd_rn(q4[i & 3], __fmul_rn(d, d));
    }
  const float q = __fadd_rn(__fadd_rn(q4[0], q4[1]), __fadd_rn(q4[2], q4[3]));
  const float var = __fdiv_rn(warp_allsum(q), static_cast<float>(256 * V));
  rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
}

__device__ __forceinline__ float ln_apply(float x, float mean, float rstd, float g) {
  return __fmul_rn(__fmul_rn(__fsub_rn(x, mean), rstd), g);
}

}  // namespace laya
