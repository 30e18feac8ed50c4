// attention_tc.cu -- masked softmax attention on the 5th-generation tensor
// cores, flash-style, with warp-specialised roles inside each CTA.
//
//   ctx_i = sum_j softmax_j(q_i . k_j / 8) v_j,
//   j visible iff j < len[b] and (global or |i - j| <= half_window)
//
// Sources: "perf(model): exact Metal speed-ups of the forward pass - #45" (one
// key-padding row broadcast over every query; the context is written straight
// into (b, s, h, hd) order); "Run Laya encoder and decision layers on CUDA",
// "Test Result" (queries whose visible keys are all padding: context 0 here).
//
// One CTA per (128-query tile, head, row); keys in tiles of 128.  Roles:
//   warp 0     TMA: the Q tile once, K and V tiles into a two-stage ring;
//   warp 1     owns TMEM; one thread issues S_j = Q K_j^T (tcgen05.mma, fp32
//              in TMEM, two S buffers) ahead of the softmax, and
//              O_j = P_j V_j (V as an MN-major operand: its [keys][64 dims]
//              tile is already that layout) into one of two O buffers;
//   warps 2-5  softmax, one thread per query row (its TMEM lane): the 128
//              scores of S_j in one TMEM load, mask, running maximum and sum
//              (exp2, fp32), the BF16 row of P_j into shared memory in the
//              128-byte swizzled K-major layout (two buffers), then the
//              previous tile's O_{j-1} folded into fp32 registers after
//              rescaling.
// So the QK^T of tile j + 1 and the PV of tile j - 1 run on the tensor cores
// while the softmax of tile j runs.  P is rounded to BF16 for the PV product
// (the row sums are not).  Local layers visit the two key tiles that cover
// [q0 - w, q0 + 128 + w) (w = 64) inside the row; global layers the tiles
// below len.  Query
// rows outside the row (partial tiles of packed rows) are computed and not
// stored; padded query rows of the padded layout are stored (0 where no key
// is visible).  Every wait is bounded (ptx::mbar_wait): an expired wait raises the
// CTA's abort flag and the device error word, every role then leaves its loop,
// the TMA and MMA threads wait (bounded) for their copies and products in
// flight, and TMEM is released.
#include "internal.h"
#include "packing.cuh"
#include "ptx.cuh"

namespace laya {

namespace {

constexpr int kThreads = 192;
constexpr int kQT = 128;                    // queries per CTA (MMA M)
constexpr int kKT = 128;                    // keys per tile (MMA N of Q K^T)
constexpr uint32_t kTile = 128u * 128u;     // bytes of a [128 x 64] BF16 tile
// shared memory (1024-byte aligned): Q | K[2] | V[2] | P[2] (two 64-key halves each) | barriers
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTile;
constexpr uint32_t kOffV = kOffK + 2 * kTile;
constexpr uint32_t kOffP = kOffV + 2 * kTile;
constexpr uint32_t kOffBar = kOffP + 4 * kTile;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;  // + alignment slack
// TMEM: S[b] at columns 128 b, O[b] at 256 + 64 b
constexpr uint32_t kTmemCols = 512;

// Barrier slots (8 bytes each) from kOffBar.
enum : uint32_t {
  kBarQ = 0,
  kBarKvFull = 1,   // + b
  kBarKvEmpty = 3,  // + b
  kBarSFull = 5,    // + b
  kBarSEmpty = 7,   // + b
  kBarPFull = 9,    // + b
  kBarPEmpty = 11,  // + b
  kBarOFull = 13,   // + b
  kBarOEmpty = 15,  // + b
  kBarDone = 17,    // every MMA of the CTA has completed
  kBarCount = 18
};

// Descriptor of a V tile as an MN-major operand (the 64 dims contiguous, keys
// down the rows, 128-byte swizzle): groups of 8 keys are 1024 bytes apart,
// carried in both offset fields.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(1024 >> 4) << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

struct AttnArgs {
  const int32_t* lengths;
  int S, heads, global, half_window, packed;
  bf16* ctx;
  int* err;
  uint64_t* stamp;
};

__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  const uint32_t bar0 = sb + kOffBar;
  auto bar = [&](uint32_t slot) { return bar0 + 8u * slot; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kBarCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  ptx::grid_launch_dependents();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = blockIdx.x * kQT;
  const int n = blockIdx.y;
  const int b = blockIdx.z;
  const int S = a.S;
  const int H = a.heads * 64;
  const int w = a.half_window;
  // The lengths are an input of the whole forward (uploaded before its first
  // kernel), not an output of the previous kernel: read before the wait.
  const int len_in = a.lengths[b];
  const bool bad_len = len_in < 1 || len_in > S;
  const int len = len_in < 1 ? 1 : (len_in > S ? S : len_in);
  if (q0 >= len) {
    if (a.packed) return;  // no such tokens
    // the whole tile is padding: defined zeros
    ptx::grid_dependency_wait();
    bf16* out = a.ctx + (static_cast<size_t>(b) * S) * H + static_cast<size_t>(n) * 64;
    for (int r = tid; r < kQT * 8; r += kThreads) {
      const int row = q0 + (r >> 3);
      if (row < S)
        reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * H)[r & 7] =
            make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  // first token of this row in the projection: packed rows start at cu(b)
  const int row0 = a.packed ? packed_start(a.lengths, b, S) : b * S;
  // key tiles of 128 from kbase: global, [0, len); local, the keys of
  // [q0 - w, q0 + 128 + w) inside [0, len) (two tiles when w <= 64)
  const int kbase = a.global ? 0 : max(0, q0 - w);
  const int kend = a.global ? len : min(len, q0 + kQT + w);
  const int nk = (kend - kbase + kKT - 1) / kKT;
  const int rows = a.packed ? len : S;  // query rows of this row that exist

  if (tid == 0) {
    for (uint32_t i = 0; i < kBarCount; ++i) ptx::mbar_init(bar(i), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(kBarSEmpty + i), 4);  // one arrival per softmax warp
      ptx::mbar_init(bar(kBarPFull + i), 4);
      ptx::mbar_init(bar(kBarOEmpty + i), 4);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm_qkv);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA
      const uint64_t pol = ptx::policy_evict_last();
      ptx::grid_dependency_wait();  // q, k, v are written by the previous kernel
      if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_stamp(a.stamp);
      if (bad_len && a.err != nullptr) atomicCAS(a.err, 0, kDevBadLength);
      ptx::mbar_arrive_expect_tx(bar(kBarQ), kTile);
      ptx::tma_load_2d(sb + kOffQ, &tm_qkv, bar(kBarQ), n * 64, row0 + q0, pol);
      int issued = 0;
      for (int j = 0; j < nk; ++j) {
        const int s = j & 1;
        if (j >= 2 && !ptx::mbar_wait(bar(kBarKvEmpty + s), ((j >> 1) - 1) & 1, abort_flag, a.err,
                                      kDevWaitEmpty, kWaitLimitNs))
          break;
        const int krow = row0 + kbase + j * kKT;
        ptx::mbar_arrive_expect_tx(bar(kBarKvFull + s), 2 * kTile);
        ptx::tma_load_2d(sb + kOffK + s * kTile, &tm_qkv, bar(kBarKvFull + s), H + n * 64, krow,
                         pol);
        ptx::tma_load_2d(sb + kOffV + s * kTile, &tm_qkv, bar(kBarKvFull + s), 2 * H + n * 64,
                         krow, pol);
        issued = j + 1;
      }
      // no copy may still be in flight into shared memory at exit (a flag of
      // our own, so that an abort does not cut these waits short)
      volatile int drain = 0;
      ptx::mbar_wait(bar(kBarQ), 0, &drain, nullptr, 0, kWaitLimitNs);
      for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
        ptx::mbar_wait(bar(kBarKvFull + (j & 1)), (j >> 1) & 1, &drain, nullptr, 0, kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      const uint32_t idesc_s = ptx::idesc_bf16(kQT, kKT);               // Q K^T: both K-major
      const uint32_t idesc_o = ptx::idesc_bf16(kQT, 64) | (1u << 16);   // P V: V MN-major
      auto issue_pv = [&](int t) -> bool {
        const int s = t & 1;
        if (!ptx::mbar_wait(bar(kBarPFull + s), (t >> 1) & 1, abort_flag, a.err, kDevWaitFull,
                            kWaitLimitNs))
          return false;
        if (t >= 2 && !ptx::mbar_wait(bar(kBarOEmpty + s), ((t >> 1) - 1) & 1, abort_flag, a.err,
                                      kDevWaitAccum, kWaitLimitNs))
          return false;
        ptx::tc_fence_after();
        const uint32_t p = sb + kOffP + s * 2 * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 256 + 64 * s,
                        ptx::sdesc_sw128(p + (kk >> 2) * kTile + (kk & 3) * 32),
                        sdesc_sw128_mn(sb + kOffV + s * kTile + kk * 2048), idesc_o,
                        kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(kBarOFull + s));
        ptx::mma_commit(bar(kBarPEmpty + s));
        ptx::mma_commit(bar(kBarKvEmpty + s));
        return true;
      };
      bool ok = ptx::mbar_wait(bar(kBarQ), 0, abort_flag, a.err, kDevWaitFull, kWaitLimitNs);
      for (int j = 0; j < nk && ok; ++j) {
        const int s = j & 1;
        ok = ptx::mbar_wait(bar(kBarKvFull + s), (j >> 1) & 1, abort_flag, a.err, kDevWaitFull,
                            kWaitLimitNs);
        if (ok && j >= 2)
          ok = ptx::mbar_wait(bar(kBarSEmpty + s), ((j >> 1) - 1) & 1, abort_flag, a.err,
                              kDevWaitAccum, kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_bf16(tmem + 128 * s, ptx::sdesc_sw128(sb + kOffQ + kk * 32),
                        ptx::sdesc_sw128(sb + kOffK + s * kTile + kk * 32), idesc_s,
                        kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(kBarSFull + s));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(nk - 1);
      // every product issued so far has completed before TMEM is released
      ptx::mma_commit(bar(kBarDone));
      volatile int drain = 0;
      ptx::mbar_wait(bar(kBarDone), 0, &drain, nullptr, 0, kWaitLimitNs);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;  // this thread's query row and TMEM lane
    const int i = q0 + row;          // its position in the row
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const float scale_log2 = 0.125f * 1.4426950408889634f;
    float o[64];
#pragma unroll
    for (int d = 0; d < 64; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f;  // running maximum (scaled, log2 domain) and sum
    float m_ref = -INFINITY;       // the maximum o is relative to
    float m_tile[2] = {-INFINITY, -INFINITY};  // the maximum each O buffer's P used
    bool ok = true;
    // adds O_t (relative to the maximum its P used) to o
    auto fold = [&](int t) -> bool {
      const int s = t & 1;
      if (!ptx::mbar_wait(bar(kBarOFull + s), (t >> 1) & 1, abort_flag, a.err, kDevWaitAccum,
                          kWaitLimitNs))
        return false;
      ptx::tc_fence_after();
      float ot[64];
      ptx::tmem_ld64(lane_base + 256 + 64 * s, ot);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarOEmpty + s));
      const float mt = m_tile[s];
      if (mt != -INFINITY) {
        const float c = m_ref == -INFINITY ? 0.f : exp2f(m_ref - mt);
#pragma unroll
        for (int d = 0; d < 64; ++d) o[d] = o[d] * c + ot[d];
        m_ref = mt;
      }
      return true;
    };
    for (int j = 0; j < nk && ok; ++j) {
      const int s = j & 1;
      if (!ptx::mbar_wait(bar(kBarSFull + s), (j >> 1) & 1, abort_flag, a.err, kDevWaitAccum,
                          kWaitLimitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float sc[128];
      ptx::tmem_ld128(lane_base + 128 * s, sc);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarSEmpty + s));
      // visible columns of this row: [lo, hi) (keys kstart + c)
      const int kstart = kbase + j * kKT;
      int lo = -kstart, hi = len - kstart;
      if (!a.global) {
        lo = max(lo, i - w - kstart);
        hi = min(hi, i + w + 1 - kstart);
      }
      float mx = -INFINITY;
      if (lo <= 0 && hi >= kKT) {
#pragma unroll
        for (int c = 0; c < kKT; ++c) {
          sc[c] *= scale_log2;
          mx = fmaxf(mx, sc[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKT; ++c) {
          sc[c] = (c >= lo && c < hi) ? sc[c] * scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[c]);
        }
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = m_new == -INFINITY ? 1.f : exp2f(m - m_new);
      m = m_new;
      m_tile[s] = m_new;
      if (j >= 2 && !ptx::mbar_wait(bar(kBarPEmpty + s), ((j >> 1) - 1) & 1, abort_flag, a.err,
                                    kDevWaitAccum, kWaitLimitNs)) {
        ok = false;
        break;
      }
      // P row: keys [0, 64) in half 0, [64, 128) in half 1; 16-byte chunk c
      // of row r sits at chunk c ^ (r % 8)
      uint8_t* prow = smem + kOffP + s * 2 * kTile + static_cast<uint32_t>(row) * 128u;
      float ls = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < kKT / 8; ++c8) {
        uint4 pk;
        __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = sc[c8 * 8 + 2 * e], x1 = sc[c8 * 8 + 2 * e + 1];
          const float p0 = m_new == -INFINITY ? 0.f : exp2f(x0 - m_new);
          const float p1 = m_new == -INFINITY ? 0.f : exp2f(x1 - m_new);
          ls += p0 + p1;
          p2[e] = __floats2bfloat162_rn(p0, p1);
        }
        const int half = c8 >> 3, ch = c8 & 7;
        *reinterpret_cast<uint4*>(prow + half * kTile + ((ch ^ (row & 7)) << 4)) = pk;
      }
      l = l * alpha + ls;
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarPFull + s));
      if (j >= 1) ok = fold(j - 1);
    }
    if (ok) ok = fold(nk - 1);
    if (ok && *abort_flag == 0 && i < rows) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* o4 = reinterpret_cast<uint4*>(a.ctx + static_cast<size_t>(row0 + i) * H +
                                           static_cast<size_t>(n) * 64);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 pk;
        __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          p2[e] = __floats2bfloat162_rn(o[c * 8 + 2 * e] * inv, o[c * 8 + 2 * e + 1] * inv);
        o4[c] = pk;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t attention_tc_smem_bytes() { return kSmem; }

cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, const int32_t* lengths, int B, int S,
                                int heads, int global, int half_window, bf16* ctx, int* err,
                                Launch l, bool packed) {
  if (B <= 0 || S <= 0 || heads <= 0 || half_window < 0) return cudaErrorInvalidValue;
  static cudaError_t configured = cudaErrorNotReady;
  if (configured != cudaSuccess) {
    configured = cudaFuncSetAttribute(attention_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (configured != cudaSuccess) return configured;
  }
  AttnArgs a;
  a.lengths = lengths;
  a.S = S;
  a.heads = heads;
  a.global = global;
  a.half_window = half_window;
  a.packed = packed ? 1 : 0;
  a.ctx = ctx;
  a.err = err;
  a.stamp = l.stamp;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((S + kQT - 1) / kQT, heads, B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attention_tc_kernel, tm_qkv, a);
}

}  // namespace laya
