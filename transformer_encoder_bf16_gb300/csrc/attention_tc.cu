// attention_tc.cu -- masked softmax attention on the 5th-generation tensor
// cores: one CTA per (128-query tile, head, row), S = Q K^T and O = P V by
// tcgen05.mma with fp32 accumulators in TMEM, Q/K/V tiles brought in by TMA.
//
//   ctx_i = sum_j softmax_j(q_i . k_j / 8) v_j,
//   j visible iff j < len[b] and (global or |i - j| <= half_window)
//
// Sources: "perf(model): exact Metal speed-ups of the forward pass - #45" (one
// key-padding row broadcast over every query; context written straight into
// (b, s, h, hd) order); "Run Laya encoder and decision layers on CUDA", "Test
// Result" (queries with no visible key: context 0 here).
//
// Per key tile of 128 keys: TMA K and V (double-buffered) -> S = Q K^T into
// TMEM (128 x 128 fp32) -> each of the 128 threads owns one query row: it
// reads its 128 scores with tcgen05.ld, masks them, updates its running
// maximum and sum (exp2, fp32) and writes its row of P (BF16) into shared
// memory in the 128-byte swizzled K-major layout -> O_tile = P V into TMEM
// (V used as an MN-major operand: its TMA tile is [keys][64 dims]) -> the
// thread adds its row of O_tile into fp32 registers after rescaling.  P is
// rounded to BF16 for the P V product (the sum of probabilities is not).
// Local layers visit only the key tiles that can hold visible keys; query
// tiles wholly in the padding of their row are written as 0.
#include "internal.h"
#include "ptx.cuh"

namespace laya {

namespace {

constexpr int kAQ = 128;        // queries per CTA (MMA M)
constexpr int kAK = 128;        // keys per tile
constexpr int kAThreads = 128;  // one thread per query row
constexpr uint32_t kTile16 = 128u * 128u;  // bytes of a [128 x 64] BF16 tile
// shared memory: Q | K[2] | V[2] | P (two 64-key halves) | barriers
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTile16;
constexpr uint32_t kOffV = kOffK + 2 * kTile16;
constexpr uint32_t kOffP = kOffV + 2 * kTile16;
constexpr uint32_t kOffBar = kOffP + 2 * kTile16;
constexpr uint32_t kAttnSmem = kOffBar + 128 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;                    // S: 128 columns, O: 64 columns

// Descriptor of the V tile as an MN-major operand (the 64 dims contiguous,
// keys down the rows, 128-byte swizzle): groups of 8 keys are 1024 bytes
// apart.  Both offset fields carry that stride.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(1024 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ bool sync_and_check(volatile int* abort_flag) {
  __syncthreads();
  return *abort_flag == 0;
}

__global__ void __launch_bounds__(kAThreads, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const int32_t* __restrict__ lengths,
                        int S, int heads, int global, int half_window, bf16* __restrict__ ctx,
                        int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const uint32_t bar_q = ptx::smem_u32(bars);        // Q landed
  const uint32_t bar_kv0 = bar_q + 8;                // K/V buffer 0, 1 landed
  const uint32_t bar_s = bar_q + 24;                 // S = Q K^T done
  const uint32_t bar_o = bar_q + 32;                 // O_tile = P V done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 72);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int q0 = blockIdx.x * kAQ;
  const int n = blockIdx.y;
  const int b = blockIdx.z;
  const int H = heads * 64;

  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  int len = lengths[b];
  if (len < 1 || len > S) {
    if (tid == 0 && err != nullptr) atomicCAS(err, 0, kDevBadLength);
    len = len < 1 ? 1 : S;
  }
  bf16* out = ctx + static_cast<size_t>(b) * S * H + static_cast<size_t>(n) * 64;
  const int i = q0 + tid;  // this thread's query

  if (q0 >= len) {
    // the whole tile is padding: defined zeros
    if (i < S) {
      uint4* o4 = reinterpret_cast<uint4*>(out + static_cast<size_t>(i) * H);
#pragma unroll
      for (int c = 0; c < 8; ++c) o4[c] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  int kbeg = 0, kend = len;
  if (!global) {
    kbeg = q0 - half_window > 0 ? q0 - half_window : 0;
    const int hi = q0 + kAQ - 1 + half_window + 1;
    kend = hi < len ? hi : len;
  }
  const int kt0 = kbeg / kAK, kt1 = (kend + kAK - 1) / kAK;
  const int row0 = b * S;  // first token of this row in the packed projection

  if (tid == 0) {
    ptx::mbar_init(bar_q, 1);
    ptx::mbar_init(bar_kv0, 1);
    ptx::mbar_init(bar_kv0 + 8, 1);
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_o, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm_qkv);
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem;            // S: columns [0, 128)
  const uint32_t t_o = tmem + 128;      // O_tile: columns [128, 192)
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  const uint64_t pol = ptx::policy_evict_last();
  auto load_kv = [&](int kt, int buf) {
    const uint32_t bar = bar_kv0 + 8u * buf;
    ptx::mbar_arrive_expect_tx(bar, 2 * kTile16);
    ptx::tma_load_2d(sb + kOffK + buf * kTile16, &tm_qkv, bar, H + n * 64, row0 + kt * kAK, pol);
    ptx::tma_load_2d(sb + kOffV + buf * kTile16, &tm_qkv, bar, 2 * H + n * 64, row0 + kt * kAK, pol);
  };
  // thread 0's count of key tiles requested and of those it saw land
  int kv_issued = 0, kv_landed = 0;
  bool q_landed = false;
  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(bar_q, kTile16);
    ptx::tma_load_2d(sb + kOffQ, &tm_qkv, bar_q, n * 64, row0 + q0, pol);
    load_kv(kt0, 0);
    kv_issued = 1;
  }

  const uint32_t idesc_s = ptx::idesc_bf16(kAQ, kAK);                 // Q K^T: both K-major
  const uint32_t idesc_o = ptx::idesc_bf16(kAQ, 64) | (1u << 16);     // P V: B (V) MN-major
  const float scale_log2 = 0.125f * 1.4426950408889634f;
  float o[64];
#pragma unroll
  for (int d = 0; d < 64; ++d) o[d] = 0.f;
  float m = -INFINITY, l = 0.f;
  bool ok = true;

  for (int kt = kt0; kt < kt1 && ok; ++kt) {
    const int it = kt - kt0;
    const int buf = it & 1;
    const uint32_t ph = static_cast<uint32_t>(it) & 1u;  // phase of bar_s / bar_o this step
    if (tid == 0) {
      if (it == 0) q_landed = ptx::mbar_wait(bar_q, 0, abort_flag, err, kDevWaitFull, kWaitLimitNs);
      if ((it > 0 || q_landed) &&
          ptx::mbar_wait(bar_kv0 + 8u * buf, static_cast<uint32_t>(it >> 1) & 1u, abort_flag, err,
                         kDevWaitFull, kWaitLimitNs)) {
        kv_landed = it + 1;
        // prefetch the next key tile into the other buffer (its previous
        // contents were consumed by the P V product of the previous step)
        if (kt + 1 < kt1) {
          load_kv(kt + 1, buf ^ 1);
          kv_issued = it + 2;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_bf16(t_s, ptx::sdesc_sw128(sb + kOffQ + kk * 32),
                        ptx::sdesc_sw128(sb + kOffK + buf * kTile16 + kk * 32), idesc_s,
                        kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar_s);
      }
    }
    ok = ptx::mbar_wait(bar_s, ph, abort_flag, err, kDevWaitAccum, kWaitLimitNs);
    if (!sync_and_check(abort_flag)) break;
    ptx::tc_fence_after();

    // ---- softmax on this thread's row, 128 scores read from TMEM in chunks
    // of 16: once for the maximum, once more for the probabilities
    float mx = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float t16[16];
      ptx::tmem_ld16(t_s + lane_base + c * 16, t16);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int key = kt * kAK + c * 16 + j;
        int dist = i - key;
        dist = dist < 0 ? -dist : dist;
        const bool vis = key < len && (global || dist <= half_window);
        if (vis) mx = fmaxf(mx, t16[j] * scale_log2);
      }
    }
    const float mnew = fmaxf(m, mx);
    const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m - mnew);
    m = mnew;
    float ls = 0.f;
    // P row: keys [0, 64) in half 0, [64, 128) in half 1; 16-byte chunk j of
    // row r sits at chunk j ^ (r % 8)
    uint8_t* prow = smem + kOffP + static_cast<uint32_t>(tid) * 128u;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float t16[16];
      ptx::tmem_ld16(t_s + lane_base + c * 16, t16);
      uint4 pk[2];
      __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float pe[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int j = 2 * e + h2;
          const int key = kt * kAK + c * 16 + j;
          int dist = i - key;
          dist = dist < 0 ? -dist : dist;
          const bool vis = key < len && (global || dist <= half_window);
          pe[h2] = (vis && m != -INFINITY) ? exp2f(t16[j] * scale_log2 - m) : 0.f;
          ls += pe[h2];
        }
        p2[e] = __floats2bfloat162_rn(pe[0], pe[1]);
      }
      const int half = c >> 2;
      const int ch0 = 2 * (c & 3);
      uint8_t* base = prow + half * kTile16;
      *reinterpret_cast<uint4*>(base + ((ch0 ^ (tid & 7)) << 4)) = pk[0];
      *reinterpret_cast<uint4*>(base + (((ch0 + 1) ^ (tid & 7)) << 4)) = pk[1];
    }
    l = l * alpha + ls;
#pragma unroll
    for (int d = 0; d < 64; ++d) o[d] *= alpha;
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();  // P complete, S read by every thread

    if (tid == 0) {
      ptx::tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_bf16(t_o, ptx::sdesc_sw128(sb + kOffP + (kk >> 2) * kTile16 + (kk & 3) * 32),
                      sdesc_sw128_mn(sb + kOffV + buf * kTile16 + kk * 2048), idesc_o,
                      kk > 0 ? 1u : 0u);
      ptx::mma_commit(bar_o);
    }
    ok = ptx::mbar_wait(bar_o, ph, abort_flag, err, kDevWaitAccum, kWaitLimitNs);
    if (!sync_and_check(abort_flag)) break;
    ptx::tc_fence_after();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float t16[16];
      ptx::tmem_ld16(t_o + lane_base + c * 16, t16);
#pragma unroll
      for (int j = 0; j < 16; ++j) o[c * 16 + j] += t16[j];
    }
    ptx::tc_fence_before();
    __syncthreads();  // O_tile read by every thread before the next P V overwrites it
  }

  if (ok && *abort_flag == 0 && i < S) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4* o4 = reinterpret_cast<uint4*>(out + static_cast<size_t>(i) * H);
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
  // no copy may still be in flight into shared memory at exit.  Every copy
  // is waited for in the loop unless it ended early; then wait here for the
  // rest, with a flag of our own so that the abort does not cut these waits.
  if (tid == 0) {
    volatile int drain_flag = 0;
    if (!q_landed)
      ptx::mbar_wait(bar_q, 0, &drain_flag, nullptr, 0, kWaitLimitNs);
    for (int t = kv_landed; t < kv_issued; ++t)
      ptx::mbar_wait(bar_kv0 + 8u * (t & 1), static_cast<uint32_t>(t >> 1) & 1u, &drain_flag,
                     nullptr, 0, kWaitLimitNs);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t attention_tc_smem_bytes() { return kAttnSmem; }

cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, const int32_t* lengths, int B, int S,
                                int heads, int global, int half_window, bf16* ctx, int* err,
                                Launch l) {
  if (B <= 0 || S <= 0 || heads <= 0) return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((S + kAQ - 1) / kAQ, heads, B);
  cfg.blockDim = dim3(kAThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attention_tc_kernel, tm_qkv, lengths, S, heads, global,
                            half_window, ctx, err);
}

}  // namespace laya
