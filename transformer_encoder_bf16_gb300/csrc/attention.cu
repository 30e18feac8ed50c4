// attention.cu -- masked softmax attention, flash-style (online softmax, no
// score matrix in memory), one CTA per (64-query tile, head, row).
//
//   ctx_i = sum_j softmax_j(q_i . k_j / 8) v_j,
//   j visible iff j < len[b] and (global or |i - j| <= half_window)
//
// Sources: "perf(model): exact Metal speed-ups of the forward pass - #45" --
// the mask is one (b,1,1,s) key-padding row broadcast over every query, and the
// context is written straight into (b, s, h, hd) order, so no transpose follows;
// "Run Laya encoder and decision layers on CUDA", "Test Result" -- queries whose
// visible keys are all padding are excluded from checks (context 0 here).
// Local layers visit only the three 64-key tiles that can hold visible keys.
// Query tiles that lie wholly in the padding of their row are written as 0.
//
// Tensor cores: QK^T and PV run on mma.sync m16n8k16 (BF16 in, fp32 out); P
// is rounded to BF16 for the PV product.  Softmax in fp32 with exp2.
//
// RoPE fused: with tables given, each Q tile and each K tile is rotated in
// shared memory right after it lands, with exactly the arithmetic of the
// stand-alone RoPE kernel (fp32 products and sum each rounded, one BF16
// rounding), so attention sees bit-identical q and k while the packed
// projection in memory is read once and never rewritten.
#include "internal.h"
#include "packing.cuh"
#include "ptx.cuh"

namespace laya {

namespace {

constexpr int kQ = 64;    // queries per CTA (4 warps x 16)
constexpr int kKT = 64;   // keys per tile
constexpr int kLd = 72;   // shared row stride in BF16 (64 + 8: conflict-free ldmatrix)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Copy a 64 x 64 BF16 tile (rows row0.., columns col0..) of the packed
// projection into shared memory; rows at or beyond S are zero-filled.
__device__ __forceinline__ void load_tile(uint32_t sdst, const bf16* base, int row0, int S,
                                          size_t ld, int tid) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = tid + 128 * r;
    const int row = c >> 3, ch = c & 7;
    const bool valid = row0 + row < S;
    const bf16* src = base + static_cast<size_t>(valid ? row0 + row : 0) * ld + ch * 8;
    cp_async16(sdst + static_cast<uint32_t>(row * kLd + ch * 8) * 2u, src, valid);
  }
}

// Rotate pairs (i, i + 32) of a 64 x 64 tile in shared memory whose first row
// is at position row0; rows at or beyond S (zero-filled) are left alone.
__device__ __forceinline__ void rope_tile(bf16* tile, int row0, int S,
                                          const float* __restrict__ cos_t,
                                          const float* __restrict__ sin_t, int tid) {
#pragma unroll 4
  for (int r = 0; r < 16; ++r) {
    const int idx = tid + 128 * r;
    const int row = idx >> 5, i = idx & 31;
    const int pos = row0 + row;
    if (pos < S) {
      bf16* p = tile + row * kLd + i;
      const float x1 = __bfloat162float(p[0]);
      const float x2 = __bfloat162float(p[32]);
      const float c = cos_t[pos * 32 + i];
      const float sn = sin_t[pos * 32 + i];
      p[0] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, sn)));
      p[32] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, sn)));
    }
  }
}

__global__ void __launch_bounds__(128, 4) attention_kernel(const bf16* __restrict__ qkv,
                                                        const int32_t* __restrict__ lengths,
                                                        int S, int heads, int global,
                                                        int half_window, bf16* __restrict__ ctx,
                                                        int* err, const float* __restrict__ cos_t,
                                                        const float* __restrict__ sin_t,
                                                        int packed, int warm, uint64_t* stamp) {
  __shared__ __align__(128) bf16 sQ[kQ * kLd];
  __shared__ __align__(128) bf16 sK[2][kKT * kLd];
  __shared__ __align__(128) bf16 sV[2][kKT * kLd];

  ptx::grid_launch_dependents();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = blockIdx.x * kQ;
  const int n = blockIdx.y;
  const int b = blockIdx.z;
  const int H = heads * 64;
  const size_t ld = static_cast<size_t>(3) * H;
  // The lengths are an input of the whole forward (uploaded before its first
  // kernel), not an output of the previous kernel: everything up to the
  // dependency wait below uses only them.
  const int len_in = lengths[b];
  const bool bad_len = len_in < 1 || len_in > S;
  const int len = len_in < 1 ? 1 : (len_in > S ? S : len_in);
  // padded rows: row b starts at token b S and rows up to S exist (padding
  // tokens are read as keys, masked); packed rows (packing.cuh): row b starts
  // at cu(b) and only its len tokens are read or written (the next row
  // follows), so tiles are cut at len
  const size_t r0 = packed ? static_cast<size_t>(packed_start(lengths, b, S))
                           : static_cast<size_t>(b) * S;
  const int rows = packed ? len : S;
  const bf16* rowbase = qkv + r0 * ld;
  bf16* out = ctx + r0 * H + static_cast<size_t>(n) * 64;
  const bool pad_tile = q0 >= len;

  int kbeg = 0, kend = len;
  if (!global) {
    kbeg = q0 - half_window > 0 ? q0 - half_window : 0;
    const int hi = q0 + kQ - 1 + half_window + 1;
    kend = hi < len ? hi : len;
  }
  const int kt0 = kbeg / kKT;
  const int kt1 = (kend + kKT - 1) / kKT;

  const uint32_t sq = ptx::smem_u32(sQ);
  const uint32_t sk0 = ptx::smem_u32(sK[0]), sk1 = ptx::smem_u32(sK[1]);
  const uint32_t sv0 = ptx::smem_u32(sV[0]), sv1 = ptx::smem_u32(sV[1]);
  const int g = lane >> 2, c4 = lane & 3;
  const float scale_log2 = 0.125f * 1.4426950408889634f;
  const int qi0 = q0 + warp * 16 + g;  // query of accumulator rows 0 (and +8)

  // Pass 0 (warm launches) runs the tile computation once over whatever
  // shared memory holds, stores nothing, and reads no output of earlier
  // kernels: it executes, while the previous kernel finishes (programmatic
  // dependent launch), the same instructions as the live pass 1, whose
  // instruction fetches then hit.
#pragma unroll 1
  for (int pass = (pad_tile || !warm) ? 1 : 0; pass < 2; ++pass) {
  const bool live = pass == 1;
  if (live) {
    ptx::grid_dependency_wait();
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_stamp(stamp);
    if (bad_len && tid == 0 && err != nullptr) atomicCAS(err, 0, kDevBadLength);
    if (pad_tile) {
      if (packed) return;  // no such tokens
      // the whole tile is padding: defined zeros
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int c = tid + 128 * r;
        const int row = c >> 3, ch = c & 7;
        if (q0 + row < S)
          *reinterpret_cast<uint4*>(out + static_cast<size_t>(q0 + row) * H + ch * 8) =
              make_uint4(0, 0, 0, 0);
      }
      return;
    }
    load_tile(sq, rowbase + n * 64, q0, rows, ld, tid);
    load_tile(sk0, rowbase + H + n * 64, kt0 * kKT, rows, ld, tid);
    load_tile(sv0, rowbase + 2 * H + n * 64, kt0 * kKT, rows, ld, tid);
    cp_async_commit();
  }

  uint32_t qf[4][4];
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

  const int kt_end = live ? kt1 : kt0 + 1;
  for (int kt = kt0; kt < kt_end; ++kt) {
    const int buf = (kt - kt0) & 1;
    const bool prefetch = kt + 1 < kt_end;
    if (!live) {
    } else if (prefetch) {
      load_tile(buf ? sk0 : sk1, rowbase + H + n * 64, (kt + 1) * kKT, rows, ld, tid);
      load_tile(buf ? sv0 : sv1, rowbase + 2 * H + n * 64, (kt + 1) * kKT, rows, ld, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (cos_t != nullptr) {
      if (kt == kt0) rope_tile(sQ, q0, rows, cos_t, sin_t, tid);
      rope_tile(buf ? sK[1] : sK[0], kt * kKT, rows, cos_t, sin_t, tid);
      __syncthreads();
    }
    if (kt == kt0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int row = warp * 16 + (lane & 15);
        const int col = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(sq + static_cast<uint32_t>(row * kLd + col) * 2u, qf[kk][0], qf[kk][1],
                qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t skb = buf ? sk1 : sk0;
    const uint32_t svb = buf ? sv1 : sv0;

    // S = Q K^T for 16 queries x 64 keys per warp
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t r0, r1, r2, r3;
        const int key = j * 8 + (lane & 7);
        const int dim = h2 * 32 + (lane >> 3) * 8;
        ldsm_x4(skb + static_cast<uint32_t>(key * kLd + dim) * 2u, r0, r1, r2, r3);
        mma16816(s[j], qf[2 * h2], r0, r1);
        mma16816(s[j], qf[2 * h2 + 1], r2, r3);
      }
    }

    // mask, scale and online softmax (rows g and g + 8 of this warp's tile)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qi = qi0 + (e >> 1) * 8;
        const int kj = kt * kKT + j * 8 + 2 * c4 + (e & 1);
        int dist = qi - kj;
        dist = dist < 0 ? -dist : dist;
        const bool vis = kj < len && (global || dist <= half_window);
        s[j][e] = vis ? s[j][e] * scale_log2 : -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], s[j][e]);
      }
    }
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mnew = fmaxf(m[r], mx[r]);
      alpha[r] = (mnew == -INFINITY) ? 1.f : exp2f(m[r] - mnew);
      m[r] = mnew;
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        const float p = (m[r] == -INFINITY) ? 0.f : exp2f(s[j][e] - m[r]);
        s[j][e] = p;
        ls[r] += p;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) l[r] = l[r] * alpha[r] + ls[r];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int jd = 0; jd < 8; jd += 2) {
        uint32_t r0, r1, r2, r3;
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int dim = jd * 8 + (lane >> 4) * 8;
        ldsm_x4_t(svb + static_cast<uint32_t>(key * kLd + dim) * 2u, r0, r1, r2, r3);
        mma16816(o[jd], pa, r0, r1);
        mma16816(o[jd + 1], pa, r2, r3);
      }
    }
    __syncthreads();
  }

  // normalise and store
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  const float inv0 = l[0] > 0.f ? 1.f / l[0] : 0.f;
  const float inv1 = l[1] > 0.f ? 1.f / l[1] : 0.f;
#pragma unroll
  for (int jd = 0; jd < 8; ++jd) {
    const int d = jd * 8 + 2 * c4;
    if (live && qi0 < rows)
      *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(qi0) * H + d) =
          pack_bf16(o[jd][0] * inv0, o[jd][1] * inv0);
    if (live && qi0 + 8 < rows)
      *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(qi0 + 8) * H + d) =
          pack_bf16(o[jd][2] * inv1, o[jd][3] * inv1);
  }
  }  // pass
}


// Attention over a subset of query rows ("perf(model): exact Metal speed-ups
// of the forward pass - #45": the last layer attends only from its marker
// rows, with the (b, 1, 1, s) key-padding row broadcast over them).  Slot
// m = b * kmax + r (r < kmax) is query token q_tok[m] (its row in qkv) at
// position q_pos[m] of row b; keys and values are row b's tokens.  One CTA per
// (64 slots of one row, head, row): the gathered Q tile, every key tile of
// the row (masked by the window on local layers), online softmax as above;
// ctx_rows[m] receives the context of slot m.
__global__ void __launch_bounds__(128) attention_rows_kernel(
    const bf16* __restrict__ qkv, const int32_t* __restrict__ lengths,
    const int32_t* __restrict__ q_tok, const int32_t* __restrict__ q_pos, int S, int kmax,
    int heads, int global, int half_window, int packed, bf16* __restrict__ ctx_rows, int* err,
    uint64_t* stamp) {
  __shared__ __align__(128) bf16 sQ[kQ * kLd];
  __shared__ __align__(128) bf16 sK[2][kKT * kLd];
  __shared__ __align__(128) bf16 sV[2][kKT * kLd];
  ptx::grid_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = blockIdx.x * kQ;  // first slot of this CTA within the row's kmax
  const int n = blockIdx.y;
  const int b = blockIdx.z;
  if (r0 >= kmax) return;
  const int nq = kmax - r0 < kQ ? kmax - r0 : kQ;
  const int m0 = b * kmax + r0;
  const int H = heads * 64;
  const size_t ld = static_cast<size_t>(3) * H;
  const int len_in = lengths[b];
  const bool bad_len = len_in < 1 || len_in > S;
  const int len = len_in < 1 ? 1 : (len_in > S ? S : len_in);
  const size_t rb = packed ? static_cast<size_t>(packed_start(lengths, b, S))
                           : static_cast<size_t>(b) * S;
  const int rows = packed ? len : S;
  const bf16* rowbase = qkv + rb * ld;
  const int g = lane >> 2, c4 = lane & 3;
  const int qr0 = warp * 16 + g;  // slot (within the CTA) of accumulator rows 0 and +8
  const int pos0 = qr0 < nq ? q_pos[m0 + qr0] : 0;
  const int pos1 = qr0 + 8 < nq ? q_pos[m0 + qr0 + 8] : 0;
  const float scale_log2 = 0.125f * 1.4426950408889634f;
  const uint32_t sq = ptx::smem_u32(sQ);
  const uint32_t sk0 = ptx::smem_u32(sK[0]), sk1 = ptx::smem_u32(sK[1]);
  const uint32_t sv0 = ptx::smem_u32(sV[0]), sv1 = ptx::smem_u32(sV[1]);

  ptx::grid_dependency_wait();
  if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_stamp(stamp);
  if (bad_len && tid == 0 && err != nullptr) atomicCAS(err, 0, kDevBadLength);
  // the gathered Q tile: slot rows past nq are zero
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = tid + 128 * r;
    const int row = c >> 3, ch = c & 7;
    const bool valid = row < nq;
    const bf16* src = qkv + static_cast<size_t>(valid ? q_tok[m0 + row] : 0) * ld + n * 64 + ch * 8;
    cp_async16(sq + static_cast<uint32_t>(row * kLd + ch * 8) * 2u, src, valid);
  }
  const int kt1 = (len + kKT - 1) / kKT;
  load_tile(sk0, rowbase + H + n * 64, 0, rows, ld, tid);
  load_tile(sv0, rowbase + 2 * H + n * 64, 0, rows, ld, tid);
  cp_async_commit();

  uint32_t qf[4][4];
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  for (int kt = 0; kt < kt1; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < kt1) {
      load_tile(buf ? sk0 : sk1, rowbase + H + n * 64, (kt + 1) * kKT, rows, ld, tid);
      load_tile(buf ? sv0 : sv1, rowbase + 2 * H + n * 64, (kt + 1) * kKT, rows, ld, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int row = warp * 16 + (lane & 15);
        const int col = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(sq + static_cast<uint32_t>(row * kLd + col) * 2u, qf[kk][0], qf[kk][1],
                qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t skb = buf ? sk1 : sk0;
    const uint32_t svb = buf ? sv1 : sv0;
    float sc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t x0, x1, x2, x3;
        const int key = j * 8 + (lane & 7);
        const int dim = h2 * 32 + (lane >> 3) * 8;
        ldsm_x4(skb + static_cast<uint32_t>(key * kLd + dim) * 2u, x0, x1, x2, x3);
        mma16816(sc[j], qf[2 * h2], x0, x1);
        mma16816(sc[j], qf[2 * h2 + 1], x2, x3);
      }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qp = (e >> 1) ? pos1 : pos0;
        const int kj = kt * kKT + j * 8 + 2 * c4 + (e & 1);
        int dist = qp - kj;
        dist = dist < 0 ? -dist : dist;
        const bool vis = kj < len && (global || dist <= half_window);
        sc[j][e] = vis ? sc[j][e] * scale_log2 : -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], sc[j][e]);
      }
    }
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mnew = fmaxf(m[r], mx[r]);
      alpha[r] = (mnew == -INFINITY) ? 1.f : exp2f(m[r] - mnew);
      m[r] = mnew;
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        const float p = (m[r] == -INFINITY) ? 0.f : exp2f(sc[j][e] - m[r]);
        sc[j][e] = p;
        ls[r] += p;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) l[r] = l[r] * alpha[r] + ls[r];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int jd = 0; jd < 8; jd += 2) {
        uint32_t x0, x1, x2, x3;
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int dim = jd * 8 + (lane >> 4) * 8;
        ldsm_x4_t(svb + static_cast<uint32_t>(key * kLd + dim) * 2u, x0, x1, x2, x3);
        mma16816(o[jd], pa, x0, x1);
        mma16816(o[jd + 1], pa, x2, x3);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  const float inv0 = l[0] > 0.f ? 1.f / l[0] : 0.f;
  const float inv1 = l[1] > 0.f ? 1.f / l[1] : 0.f;
  bf16* out = ctx_rows + static_cast<size_t>(m0) * H + static_cast<size_t>(n) * 64;
#pragma unroll
  for (int jd = 0; jd < 8; ++jd) {
    const int d = jd * 8 + 2 * c4;
    if (qr0 < nq)
      *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(qr0) * H + d) =
          pack_bf16(o[jd][0] * inv0, o[jd][1] * inv0);
    if (qr0 + 8 < nq)
      *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(qr0 + 8) * H + d) =
          pack_bf16(o[jd][2] * inv1, o[jd][3] * inv1);
  }
}
}  // namespace

cudaError_t launch_attention(const bf16* qkv, const int32_t* lengths, int B, int S, int heads,
                             int global, int half_window, bf16* ctx, int* err, Launch l,
                             const float* cos_t, const float* sin_t, bool packed) {
  if (B <= 0 || S <= 0 || heads <= 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((S + kQ - 1) / kQ, heads, B);
  cfg.blockDim = dim3(128);
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.pdl ? 1 : 0;
  // the dry pass is free only while the previous kernel runs: with
  // programmatic dependent launch and a grid that is resident at once (one
  // wave of four CTAs per SM); a later wave would pay for it
  const long long ctas = static_cast<long long>(cfg.gridDim.x) * heads * B;
  const int warm = (l.pdl && ctas <= 4ll * device_sm_count()) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attention_kernel, qkv, lengths, S, heads, global, half_window,
                            ctx, err, cos_t, sin_t, packed ? 1 : 0, warm, l.stamp);
}

}  // namespace laya

namespace laya {

cudaError_t launch_attention_rows(const bf16* qkv, const int32_t* lengths, const int32_t* q_tok,
                                  const int32_t* q_pos, int B, int S, int kmax, int heads,
                                  int global, int half_window, bool packed, bf16* ctx_rows,
                                  int* err, Launch l) {
  if (B <= 0 || S <= 0 || kmax <= 0 || heads <= 0 || half_window < 0)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((kmax + kQ - 1) / kQ, heads, B);
  cfg.blockDim = dim3(128);
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attention_rows_kernel, qkv, lengths, q_tok, q_pos, S, kmax,
                            heads, global, half_window, packed ? 1 : 0, ctx_rows, err, l.stamp);
}

}  // namespace laya
