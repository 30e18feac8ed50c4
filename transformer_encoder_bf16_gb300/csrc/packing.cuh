// packing.cuh -- the packed-token layout of the layer-by-layer path.
//
// A batch of B rows padded to S tokens carries sum(len) valid tokens.  The
// kernels keep only those: row b's tokens occupy activation rows
// [cu(b), cu(b) + len(b)), cu(b) = the lengths of the rows before it summed,
// so the projections, norms and attention skip the padding entirely (the
// pages leave padded positions without meaning; "Run Laya encoder and
// decision layers on CUDA", "Test Result").  A token's position for RoPE and
// for the attention window is still its index s in its row (the embedding
// kernel records it per packed token for the RoPE epilogue).  Every kernel
// recomputes cu from the device lengths (B <= 16 additions), so no kernel
// depends on another for the layout.  Lengths outside [1, S] are clamped
// exactly as the attention kernel clamps them.
#pragma once

#include <cstdint>

namespace laya {

__device__ __forceinline__ int packed_len(const int32_t* lens, int b, int S) {
  const int l = lens[b];
  return l < 1 ? 1 : (l > S ? S : l);
}

// cu(b): the first activation row of row b.
__device__ __forceinline__ int packed_start(const int32_t* lens, int b, int S) {
  int c = 0;
  for (int i = 0; i < b; ++i) c += packed_len(lens, i, S);
  return c;
}

// Number of valid tokens of the batch.
__device__ __forceinline__ int packed_total(const int32_t* lens, int B, int S) {
  return packed_start(lens, B, S);
}

// The first packed row of every batch row, held in registers, so that a
// token's position in its row is found by compares alone (no dependent load
// on the way to the RoPE table rows it selects).  B <= 16.
struct RowStarts {
  int cu[16];
  __device__ __forceinline__ void init(const int32_t* lens, int B, int S) {
    int c = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      cu[k] = k < B ? c : 0x7fffffff;
      if (k < B) c += packed_len(lens, k, S);
    }
  }
  // index of packed token t in its row
  __device__ __forceinline__ int pos(int t) const {
    int base = 0;
#pragma unroll
    for (int k = 1; k < 16; ++k) base = cu[k] <= t ? cu[k] : base;
    return t - base;
  }
};

}  // namespace laya
