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
//   warp 0     TMA: the Q tile once, K tiles into a two-stage ring (the next
//              K tile loads while Q K^T of the current one runs), V tiles into
//              a two-stage ring;
//   warp 1     owns TMEM; one thread issues S_j = Q K_j^T (tcgen05.mma, fp32
//              in TMEM) as soon as the softmax has read S_{j-1}, and
//              O += P_j V_j into an fp32 accumulator in TMEM, with P_j read
//              from TMEM as the A operand (V as an MN-major operand: its
//              [keys][64 dims] tile is already that layout);
//   warps 2-5  softmax, one thread per query row (its TMEM lane): the 128
//              scores of S_j in one TMEM load, mask, running maximum, P_j =
//              2^(s - m) rounded to BF16 and stored into TMEM (one row per
//              lane, two keys per 32-bit column), fp32 row sum.
// The QK^T of tile j + 1 runs on the tensor cores while the softmax of tile j
// runs.  The maximum the exponents use is raised only when a row's running
// maximum exceeds it by more than 8 (log2 units), and only then is that row of
// O rescaled in TMEM (before the next P V): the normalisation divides by a sum
// taken against the same maximum, so the result is the same softmax, with
// probabilities below 2^8 before normalisation.  P is rounded to BF16 for the
// P V product (the row sums are not).
//
// Shared memory (80 KB) and TMEM (256 columns: S 128, O 64, P 64) are sized
// so that two CTAs share an SM: one CTA's softmax overlaps the other's loads
// and products, and its start-up the other's tail.
//
// Local layers visit the key tiles of [q0 - w, q0 + 128 + w) inside the row
// (two tiles when w <= 64); global layers the tiles below len.  Query rows
// outside the row (partial tiles of packed rows) are computed and not stored;
// padded query rows of the padded layout are stored (0 where no key is
// visible).  Every wait is bounded (ptx::mbar_wait): an expired wait raises the
// CTA's abort flag and the device error word, every role then leaves its loop,
// the TMA and MMA threads wait (bounded) for their copies and products in
// flight, and TMEM is released.
#include "internal.h"
#include "packing.cuh"
#include "ptx.cuh"

namespace laya {

namespace {

constexpr int kThreads = 192;
constexpr int kQT = 128;                 // queries per CTA (MMA M)
constexpr int kKT = 128;                 // keys per tile (MMA N of Q K^T)
constexpr uint32_t kTile = 128u * 128u;  // bytes of a [128 x 64] BF16 tile
// shared memory (1024-byte aligned): Q | K[2] | V[2] | barriers
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTile;
constexpr uint32_t kOffV = kOffK + 2 * kTile;
constexpr uint32_t kOffBar = kOffV + 2 * kTile;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;  // + alignment slack
// TMEM: S at columns [0, 128), O at [128, 192), P (BF16 pairs) at [192, 256)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 192;
// the maximum the exponents use is raised only beyond this margin (log2)
constexpr float kRescaleMargin = 8.f;

// Barrier slots (8 bytes each) from kOffBar.
enum : uint32_t {
  kBarQ = 0,
  kBarKFull = 1,   // + b
  kBarKEmpty = 3,  // + b
  kBarVFull = 5,   // + b
  kBarVEmpty = 7,  // + b
  kBarSFull = 9,
  kBarSEmpty = 10,
  kBarPFull = 11,
  kBarPvDone = 12,  // P_j V_j has completed: P may be rewritten, O read or rescaled
  kBarDone = 13,    // every MMA of the CTA has completed
  kBarCount = 14
};

// Descriptor of a V tile as an MN-major operand (the 64 dims contiguous, keys
// down the rows, 128-byte swizzle): groups of 8 keys are 1024 bytes apart,
// carried in both offset fields.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(1024 >> 4) << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// 2^x by the special-function unit (approximate, flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

// Two fp32 lanes in one instruction (sm_100 f32x2 arithmetic).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n"
      " .reg .b64 ra, rb, rc, rd;\n"
      " mov.b64 ra, {%2, %3};\n"
      " mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n"
      " mov.b64 {%0, %1}, rd;\n"
      "}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

struct AttnArgs {
  const int32_t* lengths;
  int S, heads, global, half_window, packed;
  bf16* ctx;
  int* err;
  uint64_t* stamp;
};

__global__ void __launch_bounds__(kThreads, 2)
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
  // [q0 - w, q0 + 128 + w) inside [0, len)
  const int kbase = a.global ? 0 : max(0, q0 - w);
  const int kend = a.global ? len : min(len, q0 + kQT + w);
  const int nk = (kend - kbase + kKT - 1) / kKT;
  const int rows = a.packed ? len : S;  // query rows of this row that exist

  if (tid == 0) {
    for (uint32_t i = 0; i < kBarCount; ++i) ptx::mbar_init(bar(i), 1);
    ptx::mbar_init(bar(kBarSEmpty), 4);  // one arrival per softmax warp
    ptx::mbar_init(bar(kBarPFull), 4);
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
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nk; ++j) {
        const int krow = row0 + kbase + j * kKT;
        const int s = j & 1;
        if (j >= 2 && !ptx::mbar_wait(bar(kBarKEmpty + s), ((j >> 1) - 1) & 1, abort_flag, a.err,
                                      kDevWaitEmpty, kWaitLimitNs))
          break;
        ptx::mbar_arrive_expect_tx(bar(kBarKFull + s), kTile);
        ptx::tma_load_2d(sb + kOffK + s * kTile, &tm_qkv, bar(kBarKFull + s), H + n * 64, krow, pol);
        k_issued = j + 1;
        if (j >= 2 && !ptx::mbar_wait(bar(kBarVEmpty + s), ((j >> 1) - 1) & 1, abort_flag, a.err,
                                      kDevWaitEmpty, kWaitLimitNs))
          break;
        ptx::mbar_arrive_expect_tx(bar(kBarVFull + s), kTile);
        ptx::tma_load_2d(sb + kOffV + s * kTile, &tm_qkv, bar(kBarVFull + s), 2 * H + n * 64,
                         krow, pol);
        v_issued = j + 1;
      }
      // no copy may still be in flight into shared memory at exit (a flag of
      // our own, so that an abort does not cut these waits short)
      volatile int drain = 0;
      ptx::mbar_wait(bar(kBarQ), 0, &drain, nullptr, 0, kWaitLimitNs);
      for (int j = k_issued > 2 ? k_issued - 2 : 0; j < k_issued; ++j)
        ptx::mbar_wait(bar(kBarKFull + (j & 1)), (j >> 1) & 1, &drain, nullptr, 0, kWaitLimitNs);
      for (int j = v_issued > 2 ? v_issued - 2 : 0; j < v_issued; ++j)
        ptx::mbar_wait(bar(kBarVFull + (j & 1)), (j >> 1) & 1, &drain, nullptr, 0, kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      const uint32_t idesc_s = ptx::idesc_bf16(kQT, kKT);               // Q K^T: both K-major
      const uint32_t idesc_o = ptx::idesc_bf16(kQT, 64) | (1u << 16);   // P V: V MN-major
      auto issue_pv = [&](int t) -> bool {
        const int s = t & 1;
        if (!ptx::mbar_wait(bar(kBarPFull), t & 1, abort_flag, a.err, kDevWaitFull, kWaitLimitNs) ||
            !ptx::mbar_wait(bar(kBarVFull + s), (t >> 1) & 1, abort_flag, a.err, kDevWaitFull,
                            kWaitLimitNs))
          return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // keys 16 kk ..: P columns 8 kk .. (two keys a column)
          ptx::mma_bf16_ta(tmem + kColO, tmem + kColP + 8 * kk,
                           sdesc_sw128_mn(sb + kOffV + s * kTile + kk * 2048), idesc_o,
                           (t > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(kBarPvDone));
        ptx::mma_commit(bar(kBarVEmpty + s));
        return true;
      };
      bool ok = ptx::mbar_wait(bar(kBarQ), 0, abort_flag, a.err, kDevWaitFull, kWaitLimitNs);
      for (int j = 0; j < nk && ok; ++j) {
        ok = ptx::mbar_wait(bar(kBarKFull + (j & 1)), (j >> 1) & 1, abort_flag, a.err, kDevWaitFull,
                            kWaitLimitNs);
        // S is single-buffered: the softmax must have read S_{j-1}
        if (ok && j >= 1)
          ok = ptx::mbar_wait(bar(kBarSEmpty), (j - 1) & 1, abort_flag, a.err, kDevWaitAccum,
                              kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_bf16(tmem, ptx::sdesc_sw128(sb + kOffQ + kk * 32),
                        ptx::sdesc_sw128(sb + kOffK + (j & 1) * kTile + kk * 32), idesc_s,
                        kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(kBarSFull));
        ptx::mma_commit(bar(kBarKEmpty + (j & 1)));
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
    // Scores stay in the raw domain until the exponent: p = 2^(s * scale - m)
    // is one FFMA and one ex2 per score; maxima and sums use several
    // independent accumulators.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;  // this thread's query row and TMEM lane
    const int i = q0 + row;          // its position in the row
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const float scale_log2 = 0.125f * 1.4426950408889634f;
    float m = -INFINITY;  // the maximum the exponents use (scaled, log2 domain)
    float l = 0.f;        // the row sum against m
    bool ok = true;
    for (int j = 0; j < nk && ok; ++j) {
      if (!ptx::mbar_wait(bar(kBarSFull), j & 1, abort_flag, a.err, kDevWaitAccum, kWaitLimitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float sc[128];
      ptx::tmem_ld128(lane_base, sc);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarSEmpty));
      // visible columns of this row: [lo, hi) (keys kstart + c)
      const int kstart = kbase + j * kKT;
      int lo = -kstart, hi = len - kstart;
      if (!a.global) {
        lo = max(lo, i - w - kstart);
        hi = min(hi, i + w + 1 - kstart);
      }
      // (one-sided where one bound is outside the tile: the usual case, the
      // lower bound in a window's first tile, the upper one in its last)
      if (lo > 0 && hi >= kKT) {
#pragma unroll
        for (int c = 0; c < kKT; ++c)
          if (c < lo) sc[c] = -INFINITY;
      } else if (lo <= 0 && hi < kKT) {
#pragma unroll
        for (int c = 0; c < kKT; ++c)
          if (c >= hi) sc[c] = -INFINITY;
      } else if (lo > 0) {
        const uint32_t span = static_cast<uint32_t>(max(hi - lo, 0));
#pragma unroll
        for (int c = 0; c < kKT; ++c)
          if (static_cast<uint32_t>(c - lo) >= span) sc[c] = -INFINITY;
      }
      // row maximum with three-input max: eight independent accumulators
      float mxa[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxa[k] = fmaxf(sc[k], sc[k + 8]);
#pragma unroll
      for (int c = 16; c < kKT; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mxa[k] = fmax3(mxa[k], sc[c + k], sc[c + 8 + k]);
      const float mx =
          fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])) *
          scale_log2;
      // raise the exponents' maximum only when the row has gone beyond it by
      // the margin (or had none): then O and l are rescaled to the new one
      float alpha = 1.f;
      if (mx > m + kRescaleMargin) {
        alpha = m == -INFINITY ? 0.f : ex2(m - mx);
        m = mx;
      }
      const float mu = m == -INFINITY ? 0.f : m;  // a fully masked row gives p = 0
      // P_{j-1} V_{j-1} must have completed before P is rewritten and O read
      if (j >= 1) {
        if (!ptx::mbar_wait(bar(kBarPvDone), (j - 1) & 1, abort_flag, a.err, kDevWaitAccum,
                            kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      // the P row into TMEM: keys 2c and 2c + 1 as the BF16 pair of column c,
      // in two halves of 32 columns; exponents' arguments and the row sum two
      // keys per instruction
      float lsa[4] = {0.f, 0.f, 0.f, 0.f};
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 nmu2 = make_float2(-mu, -mu);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = ffma2(make_float2(sc[64 * h2 + 2 * c], sc[64 * h2 + 2 * c + 1]), sc2, nmu2);
          const float p0 = ex2(x.x), p1 = ex2(x.y);
          lsa[c & 3] += p0 + p1;
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
          pk[c] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&b2));
        }
        ptx::tmem_st32(lane_base + kColP + 32 * h2, pk);
      }
      l = l * alpha + ((lsa[0] + lsa[1]) + (lsa[2] + lsa[3]));
      // the scores are dead by now: rescale this warp's rows of O if any moved
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        float ov[64];
        ptx::tmem_ld64(lane_base + kColO, ov);
#pragma unroll
        for (int d = 0; d < 64; ++d) ov[d] *= alpha;
        ptx::tmem_st64(lane_base + kColO, ov);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarPFull));
    }
    if (ok)
      ok = ptx::mbar_wait(bar(kBarPvDone), (nk - 1) & 1, abort_flag, a.err, kDevWaitAccum,
                          kWaitLimitNs);
    if (ok) {
      ptx::tc_fence_after();
      float ov[64];
      ptx::tmem_ld64(lane_base + kColO, ov);
      if (*abort_flag == 0 && i < rows) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4* o4 = reinterpret_cast<uint4*>(a.ctx + static_cast<size_t>(row0 + i) * H +
                                             static_cast<size_t>(n) * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 pk;
          __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            p2[e] = __floats2bfloat162_rn(ov[c * 8 + 2 * e] * inv, ov[c * 8 + 2 * e + 1] * inv);
          o4[c] = pk;
        }
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
