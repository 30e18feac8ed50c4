// gemm.cu -- the four projections of an encoder layer on the 5th-generation
// tensor cores: tcgen05.mma with fp32 accumulators in TMEM, operands staged in
// shared memory by TMA (128-byte swizzle), fused epilogues.
//
//   y[t, f] = epilogue( sum_k x[t, k] * w[f, k] )      (w in nn.Linear layout)
//
// Orientation: the MMA's M side (128 rows) is always 128 output features f of
// the weight, and its N side is a tile of nt tokens t (16..256).  One kernel
// thus serves 48-token requests (nt = 48: no padding to 128 tokens) and
// 8192-token batches (nt = 256) alike; the accumulator lane is the feature, so
// a warp's epilogue stores 32 consecutive features of a token row (64 bytes).
//
// Epilogues ("[RFC]: Native Laya inference with Rust and CUDA #14": fused GEMM
// epilogues; "[Performance]: Optimize native Rust/CUDA Laya inference #66",
// "Implementation priorities": keep fp32 accumulation and BF16 rounding):
//   plain     y = bf16(acc)                    QKV projection
//   residual  y = bf16(r + acc)                attention output, MLP down (in place)
//   GeGLU     y = bf16(gelu(acc_in) * acc_gate) MLP up: two weight tiles (rows f and
//             I + f of the up-projection) feed two TMEM accumulators
//
// Split-K for short sequences, where the weights are the traffic and too few
// tiles exist to occupy every SM ("Implementation priorities": smaller tiles
// for the short shapes): the K blocks are divided among the CTAs of a thread-
// block cluster along z.  Each CTA parks its fp32 partial tile in its own
// shared memory; after a cluster barrier every CTA sums one slice of rows over
// all partials in rank order (deterministic) through distributed shared
// memory and runs the epilogue for it.  No global scratch, no atomics.
//
// Roles (192 threads): warp 0 lane 0 issues TMA, warp 1 owns TMEM and its lane
// 0 issues the MMAs, warps 2-5 drain TMEM (warp w reads TMEM lanes
// 32 * (w % 4) .. + 31).  Every wait is bounded (see ptx::mbar_wait).
//
// With programmatic dependent launch the producer loads the first pipeline
// stages of WEIGHTS before waiting for the previous kernel, so weight streaming
// overlaps the tail of the kernel before it; activations are loaded after.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace laya {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;                 // features per tile
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row of BF16
constexpr uint32_t kATileBytes = kBM * kBK * 2;
constexpr int kMaxSplits = 8;            // portable cluster size
constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kCtrlBytes = 256;

struct GemmArgs {
  int M, N, k_blocks, nt, splits, stages;
  uint32_t tmem_cols;
  uint32_t ctrl_offset;  // bytes from the aligned smem base to barriers
  bf16* y;
  const bf16* residual;
  int* err;
};

__device__ __forceinline__ float gelu_erf(float z) {
  return (0.5f * z) * (1.0f + erff(z * 0.70710678118654752f));
}

template <int KIND>
__device__ __forceinline__ void store_out(const GemmArgs& a, int t, int f, float v, float g) {
  const size_t o = static_cast<size_t>(t) * a.N + f;
  if (KIND == kGemmPlain) {
    a.y[o] = __float2bfloat16_rn(v);
  } else if (KIND == kGemmResidual) {
    a.y[o] = __float2bfloat16_rn(__bfloat162float(a.residual[o]) + v);
  } else {
    a.y[o] = __float2bfloat16_rn(gelu_erf(v) * g);
  }
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w2,
                   const __grid_constant__ CUtensorMap tm_x, const GemmArgs a) {
  constexpr int NA = (KIND == kGemmGeglu) ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t b_bytes = static_cast<uint32_t>(a.nt) * kBK * 2;
  const uint32_t stage_bytes = NA * kATileBytes + b_bytes;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.ctrl_offset);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * a.stages;
  const uint32_t accum_bar = empty0 + 8u * a.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * a.stages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int f_tile = blockIdx.x, t_tile = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * a.k_blocks / a.splits;
  const int kb1 = (split + 1) * a.k_blocks / a.splits;
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      ptx::mbar_init(full0 + 8u * i, 1);
      ptx::mbar_init(empty0 + 8u * i, 1);
    }
    ptx::mbar_init(accum_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_w);
    if (NA == 2) ptx::prefetch_tmap(&tm_w2);
    ptx::prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), a.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::grid_launch_dependents();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      const int pre = nkb < a.stages ? nkb : a.stages;
      // weights of the first stages do not depend on the previous kernel
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = sbase + i * stage_bytes;
        const uint32_t fb = full0 + 8u * i;
        const int kc = (kb0 + i) * kBK;
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
        ptx::tma_load_2d(st, &tm_w, fb, kc, f_tile * kBM, pol_w);
        if (NA == 2) ptx::tma_load_2d(st + kATileBytes, &tm_w2, fb, kc, f_tile * kBM, pol_w);
      }
      ptx::grid_dependency_wait();
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = sbase + i * stage_bytes;
        ptx::tma_load_2d(st + NA * kATileBytes, &tm_x, full0 + 8u * i, (kb0 + i) * kBK,
                         t_tile * a.nt, pol_x);
      }
      int issued = pre;
      for (int i = pre; i < nkb; ++i) {
        const int s = i % a.stages;
        const uint32_t ph = static_cast<uint32_t>(i / a.stages) & 1u;
        if (!ptx::mbar_wait(empty0 + 8u * s, ph ^ 1u, abort_flag, a.err, kDevWaitEmpty,
                            kWaitLimitNs))
          break;
        const uint32_t st = sbase + s * stage_bytes;
        const uint32_t fb = full0 + 8u * s;
        const int kc = (kb0 + i) * kBK;
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
        ptx::tma_load_2d(st, &tm_w, fb, kc, f_tile * kBM, pol_w);
        if (NA == 2) ptx::tma_load_2d(st + kATileBytes, &tm_w2, fb, kc, f_tile * kBM, pol_w);
        ptx::tma_load_2d(st + NA * kATileBytes, &tm_x, fb, kc, t_tile * a.nt, pol_x);
        issued = i + 1;
      }
      // no copy may still be in flight into this CTA's shared memory at exit
      for (int i = (issued > a.stages ? issued - a.stages : 0); i < issued; ++i)
        ptx::mbar_wait(full0 + 8u * (i % a.stages), static_cast<uint32_t>(i / a.stages) & 1u,
                       abort_flag, a.err, kDevWaitFull, kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = ptx::idesc_bf16(kBM, a.nt);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % a.stages;
        const uint32_t ph = static_cast<uint32_t>(i / a.stages) & 1u;
        if (!ptx::mbar_wait(full0 + 8u * s, ph, abort_flag, a.err, kDevWaitFull, kWaitLimitNs))
          break;
        ptx::tc_fence_after();
        const uint32_t st = sbase + s * stage_bytes;
        const uint32_t sb = st + NA * kATileBytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t bdesc = ptx::sdesc_sw128(sb + kk * 32);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          ptx::mma_bf16(tmem, ptx::sdesc_sw128(st + kk * 32), bdesc, idesc, acc);
          if (NA == 2)
            ptx::mma_bf16(tmem + static_cast<uint32_t>(a.nt),
                          ptx::sdesc_sw128(st + kATileBytes + kk * 32), bdesc, idesc, acc);
        }
        ptx::mma_commit(empty0 + 8u * s);
      }
      ptx::mma_commit(accum_bar);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int f = f_tile * kBM + row;
    const int t_base = t_tile * a.nt;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool ok = ptx::mbar_wait(accum_bar, 0, abort_flag, a.err, kDevWaitAccum, kWaitLimitNs);
    ptx::tc_fence_after();
    if (ok) {
      if (a.splits == 1) {
        ptx::grid_dependency_wait();  // residual / output of earlier kernels
        for (int c0 = 0; c0 < a.nt; c0 += 16) {
          float v[16], g[16];
          ptx::tmem_ld16(tq + c0, v);
          if (NA == 2) ptx::tmem_ld16(tq + a.nt + c0, g);
          if (f < a.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = t_base + c0 + j;
              if (t < a.M) store_out<KIND>(a, t, f, v[j], NA == 2 ? g[j] : 0.f);
            }
          }
        }
      } else {
        // park the partial tile: part[(c * 128) + row], c = token column
        float* part = reinterpret_cast<float*>(smem);
        for (int c0 = 0; c0 < a.nt; c0 += 16) {
          float v[16];
          ptx::tmem_ld16(tq + c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) part[(c0 + j) * kBM + row] = v[j];
          if (NA == 2) {
            ptx::tmem_ld16(tq + a.nt + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) part[(a.nt + c0 + j) * kBM + row] = v[j];
          }
        }
      }
    }
  }

  if (a.splits > 1) {
    __syncwarp();
    ptx::cluster_sync();  // every partial of the cluster is parked
    if (warp >= 2) {
      ptx::grid_dependency_wait();
      const uint32_t S = static_cast<uint32_t>(a.splits);
      const uint32_t rank = ptx::cluster_ctarank();
      const int r0 = static_cast<int>(rank * kBM / S);
      const int r1 = static_cast<int>((rank + 1) * kBM / S);
      const int nrows = r1 - r0;
      const int total = nrows * a.nt;
      const int t_base = t_tile * a.nt;
      uint32_t remote[kMaxSplits];
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s) remote[s] = s < a.splits ? ptx::mapa(sbase, s) : 0u;
      for (int e = threadIdx.x - 64; e < total; e += kThreads - 64) {
        const int rr = e % nrows;
        const int c = e / nrows;
        const int row = r0 + rr;
        const int f = f_tile * kBM + row;
        const int t = t_base + c;
        const uint32_t off = static_cast<uint32_t>(c * kBM + row) * 4u;
        const uint32_t off2 = static_cast<uint32_t>((a.nt + c) * kBM + row) * 4u;
        float v = 0.f, g = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) {
          if (s < a.splits) {
            v += ptx::ld_dsmem_f32(remote[s] + off);
            if (NA == 2) g += ptx::ld_dsmem_f32(remote[s] + off2);
          }
        }
        if (f < a.N && t < a.M) store_out<KIND>(a, t, f, v, g);
      }
    }
    __syncwarp();
    ptx::cluster_sync();  // nobody leaves while its partial may still be read
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, a.tmem_cols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

uint32_t pow2_cols(uint32_t n) {
  uint32_t c = 32;
  while (c < n) c <<= 1;
  return c;
}

template <int KIND>
cudaError_t launch_kind(const GemmPlan& p, const GemmOperands& o, Launch l) {
  static bool configured = false;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<KIND>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemLimit));
      if (e != cudaSuccess) return e;
      configured = true;
    }
  }
  GemmArgs a;
  a.M = p.M;
  a.N = p.N;
  a.k_blocks = p.k_blocks;
  a.nt = p.nt;
  a.splits = p.splits;
  a.stages = p.stages;
  a.tmem_cols = p.tmem_cols;
  const int na = KIND == kGemmGeglu ? 2 : 1;
  const size_t stage_bytes = static_cast<size_t>(na) * kATileBytes + static_cast<size_t>(p.nt) * 128;
  size_t data = stage_bytes * p.stages;
  const size_t part = p.splits > 1 ? static_cast<size_t>(na) * p.nt * kBM * 4 : 0;
  if (part > data) data = part;
  a.ctrl_offset = static_cast<uint32_t>(data);
  a.y = o.y;
  a.residual = o.residual;
  a.err = o.err;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.feat_tiles, p.token_tiles, p.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = 1;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = p.splits;
  ++n;
  if (l.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<KIND>, o.w, o.w2, o.x, a);
}

}  // namespace

namespace {

// Fills everything that follows from (M, N, K, kind, nt, splits); false if the
// tile does not fit in shared memory or TMEM.
bool finish_plan(GemmPlan* r) {
  const int na = r->kind == kGemmGeglu ? 2 : 1;
  const size_t stage_bytes = static_cast<size_t>(na) * kATileBytes + static_cast<size_t>(r->nt) * 128;
  const int max_kb = (r->k_blocks + r->splits - 1) / r->splits;  // K blocks of the largest split
  const size_t budget = kSmemLimit - kCtrlBytes - 1024;
  int stages = static_cast<int>(budget / stage_bytes);
  if (stages > 8) stages = 8;
  if (stages > max_kb) stages = max_kb;
  if (stages < 1) return false;
  r->stages = stages;
  size_t data = stage_bytes * stages;
  const size_t part = r->splits > 1 ? static_cast<size_t>(na) * r->nt * kBM * 4 : 0;
  if (part > budget) return false;
  if (part > data) data = part;
  r->smem_bytes = data + kCtrlBytes + 1024;
  r->tmem_cols = pow2_cols(static_cast<uint32_t>(na * r->nt));
  if (r->tmem_cols > 512) return false;
  // Never let more CTAs share an SM than its 512 TMEM columns can hold: a CTA
  // blocked in tcgen05.alloc while a cluster peer on the same SM holds TMEM at
  // a cluster barrier would never proceed.  Shared memory is the lever: each
  // resident CTA takes smem_bytes + 1 KB of the SM's 228 KB.
  const size_t sm_smem = 228 * 1024;
  const size_t max_resident = 512 / r->tmem_cols;
  const size_t floor_bytes = sm_smem / (max_resident + 1) + 1;  // (max+1) CTAs cannot fit
  if (r->smem_bytes + 1024 < floor_bytes) r->smem_bytes = floor_bytes - 1024;
  return r->smem_bytes <= kSmemLimit;
}

}  // namespace

bool plan_gemm(int M, int N, int K, int kind, int num_sms, int force_splits, int force_nt,
               GemmPlan* p) {
  if (M <= 0 || N <= 0 || K <= 0 || K % kBK != 0 || N % 8 != 0) return false;
  if (kind < kGemmPlain || kind > kGemmGeglu) return false;
  if (force_nt > 0 && (force_nt % 16 != 0 || force_nt > 256)) return false;
  if (num_sms <= 0) num_sms = 148;
  // token tiling: the fewest tiles of at most 256 tokens, evened out; one more
  // tile at a time while a split-K partial would not fit in shared memory
  for (int tt = (M + 255) / 256; tt <= (M + 15) / 16; ++tt) {
    GemmPlan r;
    r.M = M;
    r.N = N;
    r.K = K;
    r.kind = kind;
    r.k_blocks = K / kBK;
    if (force_nt > 0) {
      r.nt = force_nt;
    } else {
      const int per = (M + tt - 1) / tt;
      r.nt = (per + 15) / 16 * 16;
    }
    r.token_tiles = (M + r.nt - 1) / r.nt;
    r.feat_tiles = (N + kBM - 1) / kBM;
    const int tiles = r.token_tiles * r.feat_tiles;
    int splits;
    if (force_splits > 0) {
      splits = force_splits;
    } else {
      splits = tiles >= num_sms ? 1 : num_sms / tiles;
      // keep at least two K blocks per CTA so that each split still pipelines
      if (splits > r.k_blocks / 2) splits = r.k_blocks / 2;
    }
    if (splits < 1) splits = 1;
    if (splits > kMaxSplits) splits = kMaxSplits;
    if (splits > r.k_blocks) splits = r.k_blocks;
    if (force_splits > 0 && splits != force_splits) return false;
    r.splits = splits;
    if (finish_plan(&r)) {
      *p = r;
      return true;
    }
    if (force_nt > 0) return false;
  }
  return false;
}

bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t row_stride_bytes, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr || base == nullptr) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || row_stride_bytes % 16 != 0) return false;
  if (box_rows == 0 || box_rows > 256) return false;
  std::memset(m, 0, sizeof(*m));
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const GemmPlan& p, const GemmOperands& o, Launch l) {
  switch (p.kind) {
    case kGemmPlain: return launch_kind<kGemmPlain>(p, o, l);
    case kGemmResidual: return launch_kind<kGemmResidual>(p, o, l);
    case kGemmGeglu: return launch_kind<kGemmGeglu>(p, o, l);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace laya
