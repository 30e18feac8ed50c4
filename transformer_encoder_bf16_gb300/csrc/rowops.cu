// rowops.cu -- memory-bound row kernels: embedding gather + LayerNorm,
// LayerNorm, RoPE; and the host-side RoPE table.
//
// LayerNorm: bias-free, y = (x - mean) * (1 / sqrt(var + eps)) * gamma with
// the mean first and the variance about it second, fp32, one BF16 rounding
// ("perf(model): exact Metal speed-ups of the forward pass - #45": the encoder
// has no biases).  One warp per row, 16-byte vector loads: for hidden 1024
// each lane holds 32 values in registers, so the row is read from HBM once.
//
// RoPE: rotate-half pairs (i, i + 32) of every 64-wide q and k head, at the
// token's index in its padded row, with fp32 tables; each product and the sum
// are rounded separately (no FMA) and the result once to BF16, so the result
// is bit-identical to the CPU oracle ("[Performance]: Optimize native
// Rust/CUDA Laya inference #66", "Starting evidence": bitwise RoPE checks at
// both tables).  Grid (pair, head, token) with 32-bit indices, the geometry
// "perf(model): exact Metal speed-ups of the forward pass - #45" found fast.
#include <cmath>
#include <cstring>

#include "internal.h"
#include "packing.cuh"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace laya {

namespace {

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// V = hidden / 256 chunks of 8 BF16 per lane.  ids != nullptr selects the
// embedding form: row t reads emb[ids[t]].  lens != nullptr selects packed
// tokens (packing.cuh): the embedding form reads padded row t = b * S + s and
// writes packed row cu(b) + s (s < len(b) only); the plain form covers the
// sum(len) packed rows.
template <int V>
__global__ void __launch_bounds__(128) layernorm_kernel(const bf16* src,
                                                        const bf16* __restrict__ gamma, int M,
                                                        float eps, bf16* dst,
                                                        const int32_t* __restrict__ ids,
                                                        int vocab, int* err,
                                                        const int32_t* __restrict__ lens, int B,
                                                        int S, int32_t* __restrict__ pos,
                                                        uint64_t* stamp) {
  ptx::grid_launch_dependents();
  constexpr int H = 256 * V;
  const int row = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  // gamma is a weight, not an output of the previous kernel: its loads are
  // in flight while that kernel finishes
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  uint4 gr[V];
#pragma unroll
  for (int c = 0; c < V; ++c) gr[c] = __ldg(g4 + lane + 32 * c);
  ptx::grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) record_stamp(stamp);
  if (row >= M) return;
  int orow = row;  // output row
  if (lens != nullptr) {
    if (ids != nullptr) {
      const int b = row / S, s = row - b * S;
      if (s >= packed_len(lens, b, S)) return;  // padding: not kept
      orow = packed_start(lens, b, S) + s;
      if (pos != nullptr && lane == 0) pos[orow] = s;
    } else if (row >= packed_total(lens, B, S)) {
      return;
    }
  }
  const bf16* in;
  if (ids != nullptr) {
    int id = ids[row];
    if (id < 0 || id >= vocab) {
      if (lane == 0 && err != nullptr) atomicCAS(err, 0, kDevBadId);
      id = 0;
    }
    in = src + static_cast<size_t>(id) * H;
  } else {
    in = src + static_cast<size_t>(row) * H;
  }
  float v[V][8];
  float mean, rstd;
  row_stats<V>(reinterpret_cast<const uint4*>(in), lane, eps, v, mean, rstd);

  uint4* out4 = reinterpret_cast<uint4*>(dst + static_cast<size_t>(orow) * H);
#pragma unroll
  for (int c = 0; c < V; ++c) {
    float g[8], y[8];
    unpack8(gr[c], g);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = ln_apply(v[c][i], mean, rstd, g[i]);
    out4[lane + 32 * c] = pack8(y);
  }
}

// threadIdx.x = group of 8 pairs (pairs 8 x .. 8 x + 7 of the 32), threadIdx.y
// = head-part (q heads, then k heads), blockIdx.x = token: a (half-dim, head,
// row) grid with 32-bit indices.  Each thread moves 16 bytes of each half of
// its head (x1 = pairs' first members, x2 = second members) and two 32-byte
// table rows, so a warp reads and writes whole 128-byte heads.
__global__ void __launch_bounds__(256) rope_kernel(bf16* qkv, const float* __restrict__ cos_t,
                                                   const float* __restrict__ sin_t, int S,
                                                   int heads) {
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  const uint32_t i0 = threadIdx.x * 8u;
  const uint32_t hp = threadIdx.y;
  if (hp >= 2u * static_cast<uint32_t>(heads)) return;
  const uint32_t t = blockIdx.x;
  const uint32_t s = t % static_cast<uint32_t>(S);
  const uint32_t H = static_cast<uint32_t>(heads) * 64u;
  const uint32_t part = hp / static_cast<uint32_t>(heads);
  const uint32_t n = hp - part * static_cast<uint32_t>(heads);
  bf16* p = qkv + t * 3u * H + part * H + n * 64u + i0;
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint4 b = *reinterpret_cast<const uint4*>(p + 32);
  const float4* c4 = reinterpret_cast<const float4*>(cos_t + s * 32u + i0);
  const float4* s4 = reinterpret_cast<const float4*>(sin_t + s * 32u + i0);
  const float4 ca = __ldg(c4), cb = __ldg(c4 + 1), sa = __ldg(s4), sb = __ldg(s4 + 1);
  const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
  const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
  float x1[8], x2[8], y1[8], y2[8];
  unpack8(a, x1);
  unpack8(b, x2);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    y1[k] = __fsub_rn(__fmul_rn(x1[k], cv[k]), __fmul_rn(x2[k], sv[k]));
    y2[k] = __fadd_rn(__fmul_rn(x2[k], cv[k]), __fmul_rn(x1[k], sv[k]));
  }
  *reinterpret_cast<uint4*>(p) = pack8(y1);
  *reinterpret_cast<uint4*>(p + 32) = pack8(y2);
}

// Padded output from packed rows: out[b * S + s] = x[cu(b) + s] for s < len(b),
// 0 for the padding.  Rows of `chunks` 16-byte units (BF16 or fp32 values);
// one warp per padded row, 16-byte copies.
__global__ void __launch_bounds__(128) unpack_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ lens, int B,
                                                          int S, int chunks,
                                                          uint4* __restrict__ out,
                                                          uint64_t* stamp) {
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) record_stamp(stamp);
  const int row = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * S) return;
  const int b = row / S, s = row - b * S;
  uint4* dst = out + static_cast<size_t>(row) * chunks;
  if (s < packed_len(lens, b, S)) {
    const uint4* src = x + static_cast<size_t>(packed_start(lens, b, S) + s) * chunks;
    for (int c = lane; c < chunks; c += 32) dst[c] = src[c];
  } else {
    for (int c = lane; c < chunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
  }
}

// out[m] = x[idx[m]] for m < n: rows of `chunks` 16-byte units, one warp per row.
__global__ void __launch_bounds__(128) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ idx, int n,
                                                          int chunks, uint4* __restrict__ out,
                                                          uint64_t* stamp) {
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) record_stamp(stamp);
  const int row = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const uint4* src = x + static_cast<size_t>(idx[row]) * chunks;
  uint4* dst = out + static_cast<size_t>(row) * chunks;
  for (int c = lane; c < chunks; c += 32) dst[c] = src[c];
}

cudaError_t launch_cfg(const void* fn, dim3 grid, dim3 block, size_t smem, Launch l,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int V>
cudaError_t launch_ln_v(const bf16* src, const bf16* gamma, int M, float eps, bf16* dst,
                        const int32_t* ids, int vocab, int* err, const Packing& pk, Launch l) {
  const int rows_per_block = 4;
  dim3 grid((M + rows_per_block - 1) / rows_per_block), block(32 * rows_per_block);
  const int32_t* lens = pk.lens;
  int B = pk.B, S = pk.S;
  int32_t* pos = pk.pos;
  uint64_t* stamp = l.stamp;
  void* args[] = {(void*)&src, (void*)&gamma, (void*)&M,    (void*)&eps, (void*)&dst,
                  (void*)&ids, (void*)&vocab, (void*)&err,  (void*)&lens, (void*)&B,
                  (void*)&S,   (void*)&pos,   (void*)&stamp};
  return launch_cfg(reinterpret_cast<const void*>(&layernorm_kernel<V>), grid, block, 0, l,
                    args);
}

cudaError_t launch_ln(const bf16* src, const bf16* gamma, int M, int H, float eps, bf16* dst,
                      const int32_t* ids, int vocab, int* err, const Packing& pk, Launch l) {
  switch (H / 256) {
    case 1: return launch_ln_v<1>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 2: return launch_ln_v<2>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 3: return launch_ln_v<3>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 4: return launch_ln_v<4>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 5: return launch_ln_v<5>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 6: return launch_ln_v<6>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 7: return launch_ln_v<7>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    case 8: return launch_ln_v<8>(src, gamma, M, eps, dst, ids, vocab, err, pk, l);
    default: return cudaErrorInvalidValue;
  }
}

float bf16_round_host(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u) {
    u = (u & 0xffff0000u) | 0x00400000u;
  } else {
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
  }
  float y;
  std::memcpy(&y, &u, 4);
  return y;
}

// The end mark of a profiled forward pass: one thread records when the last
// kernel before it has completed.
__global__ void stamp_kernel(uint64_t* stamp) {
  ptx::grid_dependency_wait();
  record_stamp(stamp);
}

}  // namespace

cudaError_t launch_stamp(Launch l) {
  uint64_t* stamp = l.stamp;
  void* args[] = {(void*)&stamp};
  return launch_cfg(reinterpret_cast<const void*>(&stamp_kernel), dim3(1), dim3(32), 0, l, args);
}

bool rowops_supported_hidden(int H) { return H >= 256 && H <= 2048 && H % 256 == 0; }

cudaError_t launch_embed_layernorm(const bf16* emb, const bf16* gamma, const int32_t* ids, int M,
                                   int H, int vocab, float eps, bf16* x, int* err, Launch l,
                                   const Packing& pk) {
  if (M <= 0 || ids == nullptr) return cudaErrorInvalidValue;
  return launch_ln(emb, gamma, M, H, eps, x, ids, vocab, err, pk, l);
}

cudaError_t launch_layernorm(const bf16* x, const bf16* gamma, int M, int H, float eps, bf16* y,
                             Launch l, const Packing& pk) {
  if (M <= 0) return cudaErrorInvalidValue;
  return launch_ln(x, gamma, M, H, eps, y, nullptr, 0, nullptr, pk, l);
}

cudaError_t launch_unpack_rows(const void* x, const int32_t* lens, int B, int S, int row_bytes,
                               void* out, Launch l) {
  if (B <= 0 || S <= 0 || lens == nullptr || row_bytes <= 0 || row_bytes % 16 != 0)
    return cudaErrorInvalidValue;
  const int rows_per_block = 4;
  const int chunks = row_bytes / 16;
  dim3 grid((B * S + rows_per_block - 1) / rows_per_block), block(32 * rows_per_block);
  uint64_t* stamp = l.stamp;
  void* args[] = {(void*)&x,      (void*)&lens, (void*)&B,    (void*)&S,
                  (void*)&chunks, (void*)&out,  (void*)&stamp};
  return launch_cfg(reinterpret_cast<const void*>(&unpack_rows_kernel), grid, block, 0, l, args);
}

cudaError_t launch_gather_rows(const void* x, const int32_t* idx, int n, int row_bytes, void* out,
                               Launch l) {
  if (n <= 0 || idx == nullptr || row_bytes <= 0 || row_bytes % 16 != 0)
    return cudaErrorInvalidValue;
  const int rows_per_block = 4;
  const int chunks = row_bytes / 16;
  dim3 grid((n + rows_per_block - 1) / rows_per_block), block(32 * rows_per_block);
  uint64_t* stamp = l.stamp;
  void* args[] = {(void*)&x, (void*)&idx, (void*)&n, (void*)&chunks, (void*)&out, (void*)&stamp};
  return launch_cfg(reinterpret_cast<const void*>(&gather_rows_kernel), grid, block, 0, l, args);
}

cudaError_t unpack_node_retarget(cudaGraphExec_t exec, cudaGraphNode_t node, const void* old_out,
                                 void* new_out) {
  cudaKernelNodeParams p = {};
  cudaError_t e = cudaGraphKernelNodeGetParams(node, &p);
  if (e != cudaSuccess) return e;
  if (p.func != reinterpret_cast<const void*>(&unpack_rows_kernel) || p.kernelParams == nullptr)
    return cudaErrorInvalidValue;
  // arguments: x, lens, B, S, chunks, out, stamp
  if (*static_cast<void* const*>(p.kernelParams[5]) != old_out) return cudaErrorInvalidValue;
  void* args[7] = {p.kernelParams[0], p.kernelParams[1], p.kernelParams[2], p.kernelParams[3],
                   p.kernelParams[4], &new_out,          p.kernelParams[6]};
  p.kernelParams = args;
  p.extra = nullptr;
  e = cudaGraphExecKernelNodeSetParams(exec, node, &p);
  if (e == cudaSuccess) e = cudaGraphKernelNodeSetParams(node, &p);  // keep the template in step
  return e;
}

cudaError_t launch_rope(bf16* qkv, const float* cos_t, const float* sin_t, int B, int S,
                        int heads, Launch l) {
  const int M = B * S;
  if (M <= 0 || heads <= 0) return cudaErrorInvalidValue;
  if (2 * heads > 64) return cudaErrorInvalidValue;
  dim3 block(4, 2 * heads), grid(M);
  void* args[] = {(void*)&qkv, (void*)&cos_t, (void*)&sin_t, (void*)&S, (void*)&heads};
  return launch_cfg(reinterpret_cast<const void*>(&rope_kernel), grid, block, 0, l, args);
}

void rope_table_host(double theta, int max_seq, int half, int bf16_round, float* cos_t,
                     float* sin_t) {
  for (int p = 0; p < max_seq; ++p) {
    for (int i = 0; i < half; ++i) {
      const double inv_freq = std::pow(theta, -2.0 * i / static_cast<double>(2 * half));
      const double angle = static_cast<double>(p) * inv_freq;
      float c = static_cast<float>(std::cos(angle));
      float s = static_cast<float>(std::sin(angle));
      if (bf16_round) {
        c = bf16_round_host(c);
        s = bf16_round_host(s);
      }
      cos_t[static_cast<size_t>(p) * half + i] = c;
      sin_t[static_cast<size_t>(p) * half + i] = s;
    }
  }
}

}  // namespace laya
