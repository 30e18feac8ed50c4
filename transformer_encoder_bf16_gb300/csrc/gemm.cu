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
//   GeGLU-il  the same values from ONE 128-row weight tile holding 64 rows of
//             each half, interleaved 16 by 16 (so that a feature's two values
//             sit 16 lanes apart in one warp): one MMA per K step instead of
//             two, an accumulator of nt columns instead of 2 nt (so token
//             tiles up to 256 still double-buffer), a third less shared-memory
//             traffic
//
// Split-K for short sequences, where the weights are the traffic and too few
// tiles exist to occupy every SM ("Implementation priorities": smaller tiles
// for the short shapes): the K blocks are divided among the CTAs of a thread-
// block cluster along z.  Each CTA writes its fp32 partial tile to a global
// workspace (L2-resident) in slice layout (see slice_g0); after a cluster
// barrier (release / acquire) every CTA fetches its slice of all partials with
// one bulk copy per split, sums it in rank order (deterministic, no atomics)
// and runs the epilogue for it.  (Measured slower on this GPU: parking the
// partials in shared memory and reading them through DSMEM, and pushing the
// slices into the reducers' shared memory with DSMEM bulk copies.)
//
// Roles: warp 0 lane 0 issues TMA, warp 1 owns TMEM and its lane 0 issues the
// MMAs, the other warps drain TMEM (warp w reads TMEM lanes 32 * (w % 4) ..
// + 31): warps 2-5 of the 192-thread split kernel, warps 2-9 of the 320-thread
// persistent kernel (two warps per lane quarter, each taking half of a
// chunk's token columns).  Every wait is bounded (see ptx::mbar_wait).
//
// With programmatic dependent launch the producer loads the first pipeline
// stages of WEIGHTS before waiting for the previous kernel, so weight streaming
// overlaps the tail of the kernel before it; activations are loaded after.
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"
#include "packing.cuh"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace laya {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;                 // features per tile
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row of BF16
constexpr uint32_t kATileBytes = kBM * kBK * 2;
constexpr int kMaxSplits = 16;           // split-K cluster size (above 8: non-portable, opted in)
constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kCtrlBytes = 256;
constexpr size_t kLnStatsBytes = 256 * 8;  // [nt <= 256][mean, rstd] for LayerNorm on load
constexpr int kEpiBatch = 4;             // epilogue units whose loads are issued together
constexpr int kChunk = 32;               // staging epilogue: token columns per drain step
constexpr int kPThreads = 320;           // persistent kernel: 2 issuing warps + 8 epilogue warps
constexpr int kPEpi = kPThreads - 64;    // its epilogue threads
// per epilogue thread and chunk: units of (token, 8 features) and RoPE units
// of (token, 8 pairs)
constexpr int kPUnits = kChunk * (kBM / 8) / kPEpi;
constexpr int kRopeUnits = kChunk * (kBM / 16) / kPEpi;
static_assert(kPUnits * kPEpi == kChunk * (kBM / 8) && kRopeUnits * kPEpi == kChunk * (kBM / 16),
              "a chunk divides evenly among the epilogue threads");
// fp32 staging tiles are token-major with a padded row of kSld floats: the
// padding spreads the rows of consecutive tokens over different banks for
// the 16-byte reads of the vector phase (and the DSMEM reads of split-K).
constexpr int kSld = kBM + 4;
// the persistent kernel's double-buffered fp32 staging (plain and residual kinds)
constexpr size_t kStagingBytes = 2ull * kChunk * kSld * 4;
constexpr bool staged_epilogue(int kind) { return kind == kGemmPlain || kind == kGemmResidual; }

struct GemmArgs {
  int M, N, k_blocks, nt, splits, stages;
  int feat_tiles, token_tiles;  // persistent kernel: tile = f + feat_tiles * t
  uint32_t tmem_cols;
  uint32_t ctrl_offset;  // bytes from the aligned smem base to barriers
  bf16* y;
  const bf16* residual;
  float* y_f32;  // residual kind: if set, the fp32 sums are stored here instead of y
  int* err;
  float* partials;  // split-K workspace: [tile][split] fp32 partial tiles in slice layout
  // RoPE in the epilogue (plain kind): output features below rope_cols are
  // q|k heads of 64, rotated with the [pos, 32] tables at pos = token % rope_S
  // (packed tokens: pos = rope_pos[token], the index of the token in its row)
  const float* rope_cos;
  const float* rope_sin;
  int rope_S, rope_cols;
  const int32_t* rope_pos;  // packed tokens: position of each token (else t % rope_S)
  // packed tokens (packing.cuh): the valid token count sum(len) replaces M,
  // token tiles past it do nothing; null: all M rows
  const int32_t* lens;
  int lens_B, lens_S;
  // LayerNorm on load (split kernel): the activation tiles TMA brings in are
  // rows of ln_x, normalised in shared memory before the MMA reads them
  const bf16* ln_x;
  const bf16* ln_gamma;
  float ln_eps;
  uint64_t* stamp;  // profiling: release time of the dependency wait (first CTA)
  uint64_t wait_ns;  // bound of every wait on a barrier
  // failure-path test hook: the first CTA's producer never issues its first
  // stage, so the MMA issuer's wait for it runs out (no fault, no trap)
  int withhold;
};

// Position in a ring of n stages, advanced without division (the stage
// count is a runtime value, and a division in the single-thread producer and
// MMA loops costs more issue slots than the loop's real work).
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  int n;
  __device__ explicit RingPos(int stages, int start = 0) : n(stages) {
    s = start % n;
    ph = static_cast<uint32_t>(start / n) & 1u;
  }
  __device__ __forceinline__ void next() {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

__device__ __forceinline__ float gelu_erf(float z) {
  return (0.5f * z) * (1.0f + erff(z * 0.70710678118654752f));
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// gelu(a) * g over four values, out of line: the split-K epilogue runs once
// per launch with a cold instruction cache, so it keeps one copy of the erf
// code instead of one per unrolled element.
__device__ __noinline__ float4 geglu4(float4 a, float4 g) {
  return make_float4(gelu_erf(a.x) * g.x, gelu_erf(a.y) * g.y, gelu_erf(a.z) * g.z,
                     gelu_erf(a.w) * g.w);
}

__device__ __forceinline__ void load8_smem(const float* p, float (&v)[8]) {
  const float4 lo = reinterpret_cast<const float4*>(p)[0];
  const float4 hi = reinterpret_cast<const float4*>(p)[1];
  v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
  v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
}

// Split-K reduction slices.  The groups of a 128-feature tile (8 features
// each; a RoPE tile pairs features fo..fo+7 with fo+32..fo+39 into groups of
// 16, fo = 64 (p / 4) + 8 (p % 4) for pair group p) are divided among the
// cluster's CTAs: rank r reduces groups [r ng / splits, (r + 1) ng / splits).
// A CTA's partial tile is laid out slice by slice, so that the part of every
// split's partial one rank reduces is one contiguous block:
//   [slice r][half][token column c][feature of the slice],
// a slice's features in group order (a RoPE slice: the low 8 features of each
// of its pair groups, then the high 8 of each).
// Slice r starts at float g0(r) * gw * halves * nt, gw the group width.
__device__ __forceinline__ int slice_g0(int r, int ngroups, int splits) {
  return r * ngroups / splits;
}

// Shared memory the split-K reduction needs: the widest rank's slice of every
// split's partial (a RoPE tile's 16-wide groups bound the plain 8-wide ones).
constexpr size_t split_reduce_bytes(int na, int nt, int splits) {
  return static_cast<size_t>(splits) * na * nt * ((8 + splits - 1) / splits) * 16 * 4;
}

// The rank whose slice holds group g: the largest r with g0(r) <= g.
__device__ __forceinline__ int slice_owner(int g, int ngroups, int splits) {
  return ((g + 1) * splits - 1) / ngroups;
}


// What the epilogues write and read besides the accumulator (from GemmArgs).
struct EpiOut {
  bf16* y;
  float* y_f32;
  const bf16* residual;
  int N;
  const float* rope_cos;
  const float* rope_sin;
  int rope_S;
  const int32_t* rope_pos;
};

__device__ __forceinline__ EpiOut epi_out(const GemmArgs& a) {
  return EpiOut{a.y, a.y_f32, a.residual, a.N, a.rope_cos, a.rope_sin, a.rope_S, a.rope_pos};
}

// The eight consecutive table entries (cos, sin) a RoPE unit of token t and
// pair index i0 (a multiple of 8) needs: 32-byte aligned.  padded: take the
// position from the padded layout (t % rope_S) even for packed tokens.
struct RopeRow {
  float4 c0, c1, s0, s1;
};

__device__ __forceinline__ RopeRow rope_row_at(const EpiOut& e, int pos, int i0) {
  const float4* ct = reinterpret_cast<const float4*>(e.rope_cos + static_cast<size_t>(pos) * 32 + i0);
  const float4* st = reinterpret_cast<const float4*>(e.rope_sin + static_cast<size_t>(pos) * 32 + i0);
  return RopeRow{__ldg(ct), __ldg(ct + 1), __ldg(st), __ldg(st + 1)};
}

__device__ __forceinline__ RopeRow rope_row(const EpiOut& e, int t, int i0, bool padded = false) {
  const int pos = (e.rope_pos != nullptr && !padded) ? e.rope_pos[t] : t % e.rope_S;
  const float4* ct = reinterpret_cast<const float4*>(e.rope_cos + static_cast<size_t>(pos) * 32 + i0);
  const float4* st = reinterpret_cast<const float4*>(e.rope_sin + static_cast<size_t>(pos) * 32 + i0);
  return RopeRow{__ldg(ct), __ldg(ct + 1), __ldg(st), __ldg(st + 1)};
}

// Round to BF16 (the value the projection stores), then rotate the pair
// (x1, x2) = (feature i, feature i + 32) of a head exactly as the RoPE kernel
// does: fp32 products and sum each rounded, one BF16 rounding of the result.
// f1 is the output column of the first member of eight consecutive pairs.
__device__ __forceinline__ void rope_apply_store16(const EpiOut& a, int t, int f1, const RopeRow& r,
                                                   const float (&v1)[8], const float (&v2)[8],
                                                   bool live = true) {
  const float cv[8] = {r.c0.x, r.c0.y, r.c0.z, r.c0.w, r.c1.x, r.c1.y, r.c1.z, r.c1.w};
  const float sv[8] = {r.s0.x, r.s0.y, r.s0.z, r.s0.w, r.s1.x, r.s1.y, r.s1.z, r.s1.w};
  uint4 o1, o2;
  __nv_bfloat16* p1 = reinterpret_cast<__nv_bfloat16*>(&o1);
  __nv_bfloat16* p2 = reinterpret_cast<__nv_bfloat16*>(&o2);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float x1 = __bfloat162float(__float2bfloat16_rn(v1[i]));
    const float x2 = __bfloat162float(__float2bfloat16_rn(v2[i]));
    const float c = cv[i], sn = sv[i];
    p1[i] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, sn)));
    p2[i] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, sn)));
  }
  if (!live) return;
  bf16* row = a.y + static_cast<size_t>(t) * a.N;
  *reinterpret_cast<uint4*>(row + f1) = o1;
  *reinterpret_cast<uint4*>(row + f1 + 32) = o2;
}

// Eight consecutive output features of token t: one BF16 rounding each into
// y, or (residual kind with y_f32 set) the fp32 values themselves.
template <int KIND>
__device__ __forceinline__ void store8(const EpiOut& a, int t, int f, const float (&o)[8]) {
  const size_t e = static_cast<size_t>(t) * a.N + f;
  if (KIND == kGemmResidual && a.y_f32 != nullptr) {
    float4* d = reinterpret_cast<float4*>(a.y_f32 + e);
    d[0] = make_float4(o[0], o[1], o[2], o[3]);
    d[1] = make_float4(o[4], o[5], o[6], o[7]);
    return;
  }
  uint4 packed;
  __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
  for (int i = 0; i < 4; ++i) p2[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
  *reinterpret_cast<uint4*>(a.y + e) = packed;
}

// mean and rstd of row t of ln_x (K = 256 * V values), one warp.
template <int V>
__device__ __forceinline__ void ln_row(const GemmArgs& a, int t, int lane, float& mean, float& rstd) {
  float v[V][8];
  row_stats<V>(reinterpret_cast<const uint4*>(a.ln_x + static_cast<size_t>(t) * (256 * V)), lane,
               a.ln_eps, v, mean, rstd);
}

__device__ __forceinline__ void ln_row_any(const GemmArgs& a, int t, int lane, float& mean,
                                           float& rstd) {
  switch (a.k_blocks / 4) {
    case 1: ln_row<1>(a, t, lane, mean, rstd); break;
    case 2: ln_row<2>(a, t, lane, mean, rstd); break;
    case 3: ln_row<3>(a, t, lane, mean, rstd); break;
    case 4: ln_row<4>(a, t, lane, mean, rstd); break;
    case 5: ln_row<5>(a, t, lane, mean, rstd); break;
    case 6: ln_row<6>(a, t, lane, mean, rstd); break;
    case 7: ln_row<7>(a, t, lane, mean, rstd); break;
    default: ln_row<8>(a, t, lane, mean, rstd); break;
  }
}

// Split-K epilogue, step 1: this thread's feature row of the fp32 partial
// (GeGLU: both halves) from TMEM into its slice of the workspace, `width`
// floats between token columns.
//
// Steps 1 and 2 run once per launch at the short shapes that use split-K, a
// few microseconds after the instruction cache last held them.  They are out
// of line so that a dry call (live = false) made while the main loop runs
// executes the very instructions of the live call and brings them into the
// instruction cache: a dry call reads TMEM before the accumulator is there,
// sends its stores to the scratch words `dry` (shared memory nothing else
// uses then) and reads no output of earlier kernels.
template <int NA>
__device__ __noinline__ void split_drain(uint32_t tq, float* part, int width, int nt, float* dry,
                                         bool live) {
  float* dst = live ? part : dry;
  const int w = live ? width : 0;
#pragma unroll 1
  for (int c0 = 0; c0 < nt; c0 += 16) {
    float v[16];
    ptx::tmem_ld16(tq + c0, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) dst[(c0 + j) * w] = v[j];
    if (NA == 2) {
      ptx::tmem_ld16(tq + nt + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[(nt + c0 + j) * w] = v[j];
    }
  }
}

// Split-K epilogue, step 2: the units of this rank's slice (8 features of one
// token; a RoPE tile: 8 pairs), summed over the splits in split order from 0
// out of `red` ([split][half][token column][width], sstride floats between
// splits), then the kind's epilogue and the store.  A dry call (see
// split_drain) reads the residual and the RoPE table at padded-layout
// positions and stores into `dry` (512 bytes) with a zero row stride.
template <int KIND, int NA>
__device__ __noinline__ void split_epilogue(EpiOut eo, const float* red, int width, int sstride,
                                            int splits, int nt, int g0, int ng, int units,
                                            int t_base, int Meff, int f_base, bool rope_tile,
                                            int tid_e, float* dry, bool live) {
  const int N = eo.N;  // row stride of the residual and the output
  if (!live) {
    // stores land in `dry`: row stride 0, columns within the tile
    eo.y = reinterpret_cast<bf16*>(dry);
    if (eo.y_f32 != nullptr) eo.y_f32 = dry;
    eo.N = 0;
  }
  if (KIND == kGemmPlain && rope_tile) {
    // unit = token column c, pair group p: features (fo, fo + 32), fo = 64 (p / 4) + 8 (p % 4)
#pragma unroll 1
    for (int u = tid_e; u < units; u += kThreads - 64) {
      const int c = u / ng;
      const int pg = g0 + u % ng;
      const int fo = 64 * (pg >> 2) + 8 * (pg & 3);
      const int t = t_base + c;
      if (t >= Meff) continue;
      const RopeRow rr = rope_row(eo, t, fo & 31, !live);  // in flight during the sums
      const float4* q = reinterpret_cast<const float4*>(red + c * width + (pg - g0) * 8);
      const int h4 = width / 8;  // float4s from a low feature to its high partner
      float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0, s2 = s0, s3 = s0;
#pragma unroll 1
      for (int sp = 0; sp < splits; ++sp, q += sstride / 4) {
        s0 = add4(s0, q[0]);
        s1 = add4(s1, q[1]);
        s2 = add4(s2, q[h4]);
        s3 = add4(s3, q[h4 + 1]);
      }
      const float v1[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const float v2[8] = {s2.x, s2.y, s2.z, s2.w, s3.x, s3.y, s3.z, s3.w};
      rope_apply_store16(eo, live ? t : 0, (live ? f_base : 0) + fo, rr, v1, v2);
    }
    return;
  }
#pragma unroll 1
  for (int u = tid_e; u < units; u += kThreads - 64) {
    const int c = u / ng;
    const int grp = g0 + u % ng;
    const int t = t_base + c;
    const int f = f_base + grp * 8;
    if (t >= Meff || f >= N) continue;
    uint4 res = make_uint4(0u, 0u, 0u, 0u);
    if (KIND == kGemmResidual)  // issued before the sums
      res = *reinterpret_cast<const uint4*>(eo.residual + static_cast<size_t>(t) * N + f);
    // the GeGLU gate half follows each split's first half, nt token columns on
    const float4* q = reinterpret_cast<const float4*>(red + c * width + (grp - g0) * 8);
    const int hoff4 = nt * width / 4;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo, glo = lo, ghi = lo;
#pragma unroll 1
    for (int sp = 0; sp < splits; ++sp, q += sstride / 4) {
      lo = add4(lo, q[0]);
      hi = add4(hi, q[1]);
      if (NA == 2) {
        glo = add4(glo, q[hoff4]);
        ghi = add4(ghi, q[hoff4 + 1]);
      }
    }
    if (NA == 2) {
      lo = geglu4(lo, glo);
      hi = geglu4(hi, ghi);
    }
    float o[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    if (KIND == kGemmResidual) {
      const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&res);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 rf = __bfloat1622float2(r2[i]);
        o[2 * i] = rf.x + o[2 * i];
        o[2 * i + 1] = rf.y + o[2 * i + 1];
      }
    }
    store8<KIND>(eo, live ? t : 0, live ? f : grp * 8, o);
  }
}

// (launch bounds: two CTAs per SM, so that with programmatic dependent
// launch the next projection's CTAs fit beside this one's and stream their
// weights while it finishes)
template <int KIND>
__global__ void __launch_bounds__(kThreads, 2)
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
  const uint32_t xform0 = accum_bar + 8u;  // LayerNorm on load: stage normalised
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * a.stages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t red_bar = full0 + 8u * (3 * a.stages + 2);  // split-K slices landed
  const uint32_t done_bar = full0 + 8u * (3 * a.stages + 3);  // every MMA completed
  const bool ln = a.ln_x != nullptr;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int f_tile = blockIdx.x, t_tile = blockIdx.y, split = blockIdx.z;
  // tokens this launch covers (packed: the valid ones); a token tile past
  // them has nothing to do (its whole cluster shares the tile and leaves)
  const int Meff = a.lens != nullptr ? packed_total(a.lens, a.lens_B, a.lens_S) : a.M;
  if (t_tile * a.nt >= Meff) return;
  const int kb0 = split * a.k_blocks / a.splits;
  const int kb1 = (split + 1) * a.k_blocks / a.splits;
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      ptx::mbar_init(full0 + 8u * i, 1);
      ptx::mbar_init(empty0 + 8u * i, 1);
      ptx::mbar_init(xform0 + 8u * i, kThreads - 64);
    }
    ptx::mbar_init(accum_bar, 1);
    ptx::mbar_init(red_bar, 1);
    ptx::mbar_init(done_bar, 1);
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
  bool epi_ok = false;
  bool red_failed = false;

  // split-K geometry (see slice_g0).  Drain side: the slice this thread's
  // feature row (TMEM lane) belongs to; reduce side: this rank's slice.
  const bool rope_tile = KIND == kGemmPlain && a.rope_cos != nullptr && f_tile * kBM < a.rope_cols;
  const int gw = rope_tile ? 16 : 8;
  const int ngroups = kBM / gw;  // RoPE: pairs of groups (f, f + 32)
  const int erow = threadIdx.x & 127;  // epilogue warps: TMEM lane (warp % 4) * 32 + lane
  const int drain_grp = rope_tile ? 4 * (erow >> 6) + ((erow & 31) >> 3) : erow >> 3;
  int drain_width = 0, red_g0 = 0, red_g1 = ngroups, red_width = 0;
  float* drain_part = nullptr;
  if (a.splits > 1) {
    const int r = slice_owner(drain_grp, ngroups, a.splits);
    const int sg0 = slice_g0(r, ngroups, a.splits);
    drain_width = (slice_g0(r + 1, ngroups, a.splits) - sg0) * gw;
    // feature of the slice: group-major; a RoPE slice holds the low 8 of each
    // pair group first, then the high 8 (a warp's rows stay contiguous)
    const int in_slice = rope_tile ? ((erow & 32) ? drain_width / 2 : 0) +
                                         (drain_grp - sg0) * 8 + (erow & 7)
                                   : (drain_grp - sg0) * 8 + (erow & 7);
    const int tile = t_tile * gridDim.x + f_tile;
    drain_part = a.partials + (static_cast<size_t>(tile) * a.splits + split) * NA * a.nt * kBM +
                 static_cast<size_t>(sg0) * gw * NA * a.nt + in_slice;
    const int rank = static_cast<int>(ptx::cluster_ctarank());
    red_g0 = slice_g0(rank, ngroups, a.splits);
    red_g1 = slice_g0(rank + 1, ngroups, a.splits);
    red_width = (red_g1 - red_g0) * gw;
  }
  const int red_units = (red_g1 - red_g0) * a.nt;
  const int red_sstride = NA * a.nt * red_width;  // floats between splits in the reduce buffer
  // scratch for dry calls: the LayerNorm-statistics area, unused without LayerNorm on load
  float* dry = reinterpret_cast<float*>(smem + a.ctrl_offset + kCtrlBytes);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      const int pre = nkb < a.stages ? nkb : a.stages;
      const bool wh = a.withhold && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
      // weights of the first stages do not depend on the previous kernel
      for (int i = 0; i < pre; ++i) {
        if (wh && i == 0) continue;
        const uint32_t st = sbase + i * stage_bytes;
        const uint32_t fb = full0 + 8u * i;
        const int kc = (kb0 + i) * kBK;
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
        ptx::tma_load_2d(st, &tm_w, fb, kc, f_tile * kBM, pol_w);
        if (NA == 2) ptx::tma_load_2d(st + kATileBytes, &tm_w2, fb, kc, f_tile * kBM, pol_w);
      }
      ptx::grid_dependency_wait();
      if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_stamp(a.stamp);
      for (int i = 0; i < pre; ++i) {
        if (wh && i == 0) continue;
        const uint32_t st = sbase + i * stage_bytes;
        ptx::tma_load_2d(st + NA * kATileBytes, &tm_x, full0 + 8u * i, (kb0 + i) * kBK,
                         t_tile * a.nt, pol_x);
      }
      int issued = pre;
      RingPos rp(a.stages, pre);
      for (int i = pre; i < nkb; ++i, rp.next()) {
        const int s = rp.s;
        if (!ptx::mbar_wait(empty0 + 8u * s, rp.ph ^ 1u, abort_flag, a.err, kDevWaitEmpty,
                            a.wait_ns))
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
      // no copy may still be in flight into this CTA's shared memory at exit:
      // wait for the last stages issued, with a flag of our own so that an
      // abort does not cut these waits short
      volatile int drain = 0;
      for (int i = (issued > a.stages ? issued - a.stages : 0); i < issued; ++i)
        if (!(wh && i == 0))
          ptx::mbar_wait(full0 + 8u * (i % a.stages), static_cast<uint32_t>(i / a.stages) & 1u,
                         &drain, nullptr, 0, a.wait_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = ptx::idesc_bf16(kBM, a.nt);
      // descriptors of stage 0; stage s and K step kk add s * stage_bytes and
      // kk * 32 bytes to the start-address field (in 16-byte units)
      const uint64_t da0 = ptx::sdesc_sw128(sbase);
      const uint64_t db0 = ptx::sdesc_sw128(sbase + NA * kATileBytes);
      const uint64_t stage_units = stage_bytes >> 4;
      RingPos rp(a.stages);
      for (int i = 0; i < nkb; ++i, rp.next()) {
        const int s = rp.s;
        if (!ptx::mbar_wait((ln ? xform0 : full0) + 8u * s, rp.ph, abort_flag, a.err, kDevWaitFull,
                            a.wait_ns))
          break;
        ptx::tc_fence_after();
        const uint64_t da = da0 + static_cast<uint64_t>(s) * stage_units;
        const uint64_t db = db0 + static_cast<uint64_t>(s) * stage_units;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          ptx::mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, acc);
          if (NA == 2)
            ptx::mma_bf16(tmem + static_cast<uint32_t>(a.nt), da + (kATileBytes >> 4) + 2 * kk,
                          db + 2 * kk, idesc, acc);
        }
        ptx::mma_commit(empty0 + 8u * s);
      }
      ptx::mma_commit(accum_bar);
      // every product issued has completed before TMEM is released (an abort
      // may leave no other thread waiting for them)
      ptx::mma_commit(done_bar);
      volatile int drain = 0;
      ptx::mbar_wait(done_bar, 0, &drain, nullptr, 0, a.wait_ns);
    }
  } else {
    // ------------------------------------------- epilogue phase 1: drain TMEM
    // fp32 tile staged token-major in shared memory: stg[c * kSld + row] for
    // token column c and feature row (the pipeline stages are free by now).
    // Split-K parks the raw partial (GeGLU: both halves); otherwise the
    // GeGLU product is formed here.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    if (a.splits > 1 && !ln) {
      // dry calls while the main loop runs (see split_drain)
      split_drain<NA>(tq, drain_part, drain_width, a.nt, dry, false);
      split_epilogue<KIND, NA>(epi_out(a), reinterpret_cast<const float*>(smem), red_width,
                               red_sstride, a.splits, a.nt, red_g0, red_g1 - red_g0, red_units,
                               t_tile * a.nt, Meff, f_tile * kBM, rope_tile,
                               static_cast<int>(threadIdx.x) - 64, dry, false);
    }
    // LayerNorm input and residual are written by earlier kernels; waiting
    // here, while the main loop runs, keeps the wait off the epilogue's path
    ptx::grid_dependency_wait();
    if (ln) {
      // ---- LayerNorm on load: row statistics, then normalise each stage
      const int tid_e = threadIdx.x - 64;
      float* stats = reinterpret_cast<float*>(smem + a.ctrl_offset + kCtrlBytes);
      for (int r = warp - 2; r < a.nt; r += 4) {
        const int t = t_tile * a.nt + r;
        float mean = 0.f, rstd = 0.f;
        if (t < Meff) ln_row_any(a, t, lane, mean, rstd);
        if (lane == 0) {
          stats[2 * r] = mean;
          stats[2 * r + 1] = rstd;
        }
      }
      ptx::named_barrier_sync(1, kThreads - 64);
      RingPos rp(a.stages);
      for (int i = 0; i < nkb; ++i, rp.next()) {
        const int s = rp.s;
        if (!ptx::mbar_wait(full0 + 8u * s, rp.ph, abort_flag, a.err, kDevWaitFull, a.wait_ns))
          break;
        // B tile: nt rows of 128 bytes; 16-byte chunk j of row r sits at j ^ (r % 8)
        uint8_t* bt = smem + static_cast<size_t>(s) * stage_bytes + NA * kATileBytes;
        const int kc = (kb0 + i) * kBK;
        for (int u = tid_e; u < a.nt * 8; u += kThreads - 64) {
          const int r = u >> 3, pc = u & 7, j = pc ^ (r & 7);
          uint4* p = reinterpret_cast<uint4*>(bt + r * 128 + pc * 16);
          float xv[8], g[8];
          bf16x8_to_f32(*p, xv);
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.ln_gamma + kc + 8 * j), g);
          const float mean = stats[2 * r], rstd = stats[2 * r + 1];
          uint4 o;
          __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o2[e] = __floats2bfloat162_rn(ln_apply(xv[2 * e], mean, rstd, g[2 * e]),
                                          ln_apply(xv[2 * e + 1], mean, rstd, g[2 * e + 1]));
          *p = o;
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(xform0 + 8u * s);
      }
    }
    epi_ok = ptx::mbar_wait(accum_bar, 0, abort_flag, a.err, kDevWaitAccum, a.wait_ns);
    // the TMEM loads below are warp-collective: after an abort, lanes that
    // polled at different moments must still agree
    epi_ok = __all_sync(0xffffffffu, epi_ok);
    ptx::tc_fence_after();
    if (epi_ok && a.splits > 1) {
      // partial tile to the workspace, this thread's row into its owner's slice
      split_drain<NA>(tq, drain_part, drain_width, a.nt, dry, true);
    } else if (epi_ok) {
      float* stg = reinterpret_cast<float*>(smem);
      for (int c0 = 0; c0 < a.nt; c0 += 16) {
        float v[16];
        ptx::tmem_ld16(tq + c0, v);
        if (NA == 2) {
          float g[16];
          ptx::tmem_ld16(tq + a.nt + c0, g);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = gelu_erf(v[j]) * g[j];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) stg[(c0 + j) * kSld + row] = v[j];
      }
    }
    if (a.splits == 1) ptx::named_barrier_sync(1, kThreads - 64);
  }

  if (a.splits > 1) {
    __syncwarp();
    ptx::cluster_sync();  // every partial of the cluster is in the workspace (release/acquire)
  }

  if (warp >= 2 && epi_ok) {
    // ------------------------------- epilogue phase 2: 16-byte vector stores
    // unit = 8 consecutive features of one token; consecutive threads take
    // consecutive units of a token row, so loads and stores are coalesced.
    // Split-K: this CTA finishes the feature groups of its slice of the tile,
    // summing the partials of every CTA of the cluster in rank order.
    const int tid_e = threadIdx.x - 64;
    const int t_base = t_tile * a.nt;
    const EpiOut eo = epi_out(a);
    if (a.splits > 1) {
      // this rank's slice of every split's partial into the idle ring:
      // [split][half][token column][width]
      const uint32_t bytes = static_cast<uint32_t>(red_sstride) * 4u;
      if (tid_e == 0) {
        // the partials were written by the other CTAs of the cluster with
        // ordinary stores (ordered before the cluster barrier above)
        ptx::fence_proxy_async_global();
        const size_t pstride = static_cast<size_t>(NA) * a.nt * kBM;  // floats between splits
        const float* src = a.partials +
                           static_cast<size_t>(t_tile * gridDim.x + f_tile) * a.splits * pstride +
                           static_cast<size_t>(red_g0) * gw * NA * a.nt;
        ptx::mbar_arrive_expect_tx(red_bar, bytes * static_cast<uint32_t>(a.splits));
        for (int sp = 0; sp < a.splits; ++sp)
          ptx::bulk_load(sbase + static_cast<uint32_t>(sp) * bytes, src + sp * pstride, bytes,
                         red_bar);
      }
      if (!ptx::mbar_wait(red_bar, 0, abort_flag, a.err, kDevWaitReduce, a.wait_ns))
        red_failed = true;
      else
        split_epilogue<KIND, NA>(eo, reinterpret_cast<const float*>(smem), red_width, red_sstride,
                                 a.splits, a.nt, red_g0, red_g1 - red_g0, red_units, t_base, Meff,
                                 f_tile * kBM, rope_tile, tid_e, dry, true);
    } else {
    // one CTA per tile: the fp32 tile staged by phase 1 (GeGLU applied)
    const int ng = ngroups;
    const int units = red_units;
    const float* stg = reinterpret_cast<const float*>(smem);
    if (rope_tile) {
      // unit = token column c, pair group p: features (fo, fo + 32), fo = 64 (p / 4) + 8 (p % 4)
      for (int u = tid_e; u < units; u += kThreads - 64) {
        const int c = u / ng;
        const int pg = u % ng;
        const int fo = 64 * (pg >> 2) + 8 * (pg & 3);
        const int t = t_base + c;
        if (t >= Meff) continue;
        const RopeRow rr = rope_row(eo, t, fo & 31);
        float v1[8], v2[8];
        load8_smem(stg + c * kSld + fo, v1);
        load8_smem(stg + c * kSld + fo + 32, v2);
        rope_apply_store16(eo, t, f_tile * kBM + fo, rr, v1, v2);
      }
    } else
    for (int u0 = tid_e; u0 < units; u0 += (kThreads - 64) * kEpiBatch) {
      float v[kEpiBatch][8];
      uint4 res[kEpiBatch];
      int tok[kEpiBatch], fea[kEpiBatch];
      // loads first (the output may alias the residual: keep every load of
      // the batch ahead of its stores)
#pragma unroll
      for (int b = 0; b < kEpiBatch; ++b) {
        const int u = u0 + (kThreads - 64) * b;
        tok[b] = -1;
        if (u < units) {
          const int c = u / ng;
          const int grp = u % ng;
          {
            // the staged tile (GeGLU already applied)
            const float4* p4 = reinterpret_cast<const float4*>(stg + c * kSld + grp * 8);
            const float4 lo = p4[0], hi = p4[1];
            v[b][0] = lo.x; v[b][1] = lo.y; v[b][2] = lo.z; v[b][3] = lo.w;
            v[b][4] = hi.x; v[b][5] = hi.y; v[b][6] = hi.z; v[b][7] = hi.w;
          }
          const int t = t_base + c;
          const int f = f_tile * kBM + grp * 8;
          if (t < Meff && f < a.N) {
            tok[b] = t;
            fea[b] = f;
            if (KIND == kGemmResidual)
              res[b] = *reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(t) * a.N + f);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kEpiBatch; ++b) {
        if (tok[b] < 0) continue;
        float o[8];
        if (KIND == kGemmResidual) {
          const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&res[b]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 rf = __bfloat1622float2(r2[i]);
            o[2 * i] = rf.x + v[b][2 * i];
            o[2 * i + 1] = rf.y + v[b][2 * i + 1];
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = v[b][i];
        }
        store8<KIND>(eo, tok[b], fea[b], o);
      }
    }
    }  // one CTA per tile
    if (red_failed && a.splits > 1 && threadIdx.x == 64) {
      // no bulk copy may still be landing in this CTA's shared memory at exit
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(red_bar, 0) && ptx::globaltimer_ns() - t0 < a.wait_ns) {
      }
    }
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

// Persistent variant for splits == 1: one CTA per SM walks the output tiles
// (tile = feature tile + feat_tiles * token tile, strided by gridDim.x).  Two
// TMEM accumulators alternate, so the epilogue of one tile overlaps the main
// loop of the next; the TMA ring runs continuously across tiles.
//
// Two epilogues.  Plain and residual kinds stage the accumulator through
// shared memory (32 token columns at a time, fp32) and store 16-byte
// vectors, reading the residual and the RoPE table rows as 16-byte vectors
// too.  The GeGLU kinds, which read nothing from global memory, go from TMEM
// straight to global memory: shared-memory bandwidth is what the main loop's
// TMA writes and MMA reads already use up, and staging there slowed their
// MMAs by a third.  There a thread owns one accumulator row (an output
// feature) and loads 16 token columns at a time; for each token the warp's
// lanes store consecutive features.  GeGLU-il's two rows of a feature (GELU
// and gate half) are loaded as lanes l and l + 16 of one warp (a 4-D tensor
// map interleaves the weight rows 16 by 16): one shuffle brings them together.
// (Stores of 2 bytes per lane were measured slower than the staged 16-byte
// vectors for the plain and residual kinds, whose reads of the residual and
// the RoPE tables then become 2- and 4-byte loads per lane and token.)
//
// PAIR != 0: the CTAs run in clusters of two that share one operand tile of
// every stage, brought in once by the first CTA and multicast by TMA into both
// CTAs' shared memory (halving the L2-to-SM traffic of that operand); each
// CTA's MMA issuer releases a stage in both CTAs (multicast commit), so a
// stage is refilled only when both have consumed it.
//   PAIR == 1: the two feature tiles of a pair with the same token tile (the
//              token tile, B, is shared);
//   PAIR == 2: the two token tiles of a pair with the same feature tile (the
//              weight tiles, A, are shared).
//   PAIR == 3: one MMA for the pair (tcgen05 cta_group::2, 256 weight rows):
//              each CTA loads its 128 weight rows and HALF of the shared token
//              tile (halving that operand's traffic into each SM, not only
//              out of L2), the first CTA issues the MMAs for both, and each
//              CTA's TMEM holds its 128 features x nt tokens.  Both CTAs'
//              loads count on the first CTA's full barriers; both CTAs'
//              epilogues hand the accumulator back on its barriers.
// With an odd tile count the last pair's second tile lies past N (its weight
// rows load as zeros) or past the tokens; its outputs are not stored.
template <int KIND, int PAIR>
__global__ void __launch_bounds__(kPThreads, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_w2,
                           const __grid_constant__ CUtensorMap tm_x, const GemmArgs a) {
  constexpr int NA = (KIND == kGemmGeglu) ? 2 : 1;
  constexpr bool TWO = PAIR == 3;  // one cta_group::2 MMA per pair
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  // this CTA's token rows of a stage (TWO: half the tile)
  const uint32_t b_bytes = static_cast<uint32_t>(TWO ? a.nt / 2 : a.nt) * kBK * 2;
  const uint32_t stage_bytes = NA * kATileBytes + b_bytes;
  float* staging = reinterpret_cast<float*>(smem + static_cast<size_t>(a.stages) * stage_bytes);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.ctrl_offset);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * a.stages;
  const uint32_t accf0 = empty0 + 8u * a.stages;  // accumulator b ready: accf0 + 8b
  const uint32_t acce0 = accf0 + 16u;             // accumulator b drained: acce0 + 8b
  const uint32_t done_bar = acce0 + 16u;          // every MMA completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * a.stages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // tokens this launch covers (packed: the valid ones) and their tiles.  The
  // walk: work item w = first, first + step, ... < tiles; feature tile and
  // token tile of an item from tile_of (PAIR: items are feature-tile pairs)
  const int Meff = a.lens != nullptr ? packed_total(a.lens, a.lens_B, a.lens_S) : a.M;
  const int ttiles = (Meff + a.nt - 1) / a.nt;
  const int fwalk = (PAIR == 1 || TWO) ? (a.feat_tiles + 1) / 2 : a.feat_tiles;
  const int twalk = PAIR == 2 ? (ttiles + 1) / 2 : ttiles;
  const int tiles = fwalk * twalk;
  const int rank = PAIR ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  const int first = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  auto tile_of = [&](int item, int& ft, int& tt) {
    const int f = item % fwalk, t = item / fwalk;
    ft = (PAIR == 1 || TWO) ? 2 * f + rank : f;
    tt = PAIR == 2 ? 2 * t + rank : t;
  };
  const int KB = a.k_blocks;
  const uint32_t acc_cols = static_cast<uint32_t>(NA * a.nt);  // one accumulator's columns

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      ptx::mbar_init(full0 + 8u * i, 1);
      // PAIR 1, 2: both CTAs' MMAs release it; TWO: the first CTA's MMA for both
      ptx::mbar_init(empty0 + 8u * i, (PAIR == 1 || PAIR == 2) ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf0 + 8u * b, 1);
      // every epilogue thread arrives (TWO: both CTAs')
      ptx::mbar_init(acce0 + 8u * b, (TWO ? 2 : 1) * kPEpi);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_w);
    if (NA == 2) ptx::prefetch_tmap(&tm_w2);
    ptx::prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    if (TWO) {
      ptx::tmem_alloc_cg2(ptx::smem_u32(tmem_slot), a.tmem_cols);
      ptx::tmem_relinquish_cg2();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), a.tmem_cols);
      ptx::tmem_relinquish();
    }
  }
  // PAIR: both CTAs' barriers are initialised before either multicasts into the other
  if (PAIR) ptx::cluster_sync();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::grid_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  // an epilogue thread hands accumulator b back to the MMA issuer (TWO: to
  // the first CTA's barrier, from both CTAs)
  auto release_acc = [&](int b) {
    if (TWO)
      ptx::mbar_arrive_cluster(ptx::mapa(acce0 + 8u * b, 0));
    else
      ptx::mbar_arrive(acce0 + 8u * b);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      // each operand tile: loaded by this CTA alone, or (the shared one of a
      // pair) by the first CTA of the pair into both
      const bool loads_a = PAIR != 2 || rank == 0;
      const bool loads_b = PAIR != 1 || rank == 0;
      auto load = [&](bool mc, uint32_t dst, const CUtensorMap* m, uint32_t fb, int kc, int row,
                      uint64_t pol) {
        if (TWO)
          ptx::tma_load_2d_cg2(dst, m, fb, kc, row, pol);
        else if (mc)
          ptx::tma_load_2d_mc(dst, m, fb, kc, row, static_cast<uint16_t>(0x3), pol);
        else
          ptx::tma_load_2d(dst, m, fb, kc, row, pol);
      };
      // the barrier a stage's bytes count on (TWO: the first CTA's) and the
      // bytes it expects (TWO: both CTAs'; only the first CTA arms it)
      auto fbar = [&](int s) {
        return TWO ? ptx::mapa(full0 + 8u * s, 0) : full0 + 8u * s;
      };
      const bool arms = !TWO || rank == 0;
      const uint32_t expect = TWO ? 2 * stage_bytes : stage_bytes;
      auto load_a = [&](uint32_t st, uint32_t fb, int kc, int f) {
        if (KIND == kGemmGegluIl) {
          // blocks 4f .. 4f + 3 of 16 features, each as GELU rows then gate
          // rows: (k, row, half, block) from (kc, 0, 0, 4f)
          if (TWO)
            ptx::tma_load_4d_cg2(st, &tm_w, fb, kc, 0, 0, 4 * f, pol_w);
          else if (PAIR == 2)
            ptx::tma_load_4d_mc(st, &tm_w, fb, kc, 0, 0, 4 * f, static_cast<uint16_t>(0x3), pol_w);
          else
            ptx::tma_load_4d(st, &tm_w, fb, kc, 0, 0, 4 * f, pol_w);
          return;
        }
        load(PAIR == 2, st, &tm_w, fb, kc, f * kBM, pol_w);
        if (NA == 2) load(PAIR == 2, st + kATileBytes, &tm_w2, fb, kc, f * kBM, pol_w);
      };
      // token rows from t (TWO: this CTA's half of the tile)
      auto load_b = [&](uint32_t dst, uint32_t fb, int kc, int t) {
        load(PAIR == 1, dst, &tm_x, fb, kc, TWO ? t + rank * (a.nt / 2) : t, pol_x);
      };
      int issued = 0;
      const bool wh = a.withhold && blockIdx.x == 0;
      if (first < tiles) {
        // weights of the first stages of the first tile before the dependency wait
        const int pre = KB < a.stages ? KB : a.stages;
        int f0, t0;
        tile_of(first, f0, t0);
        for (int i = 0; i < pre; ++i) {
          if (wh && i == 0) continue;
          const uint32_t st = sbase + i * stage_bytes;
          if (arms) ptx::mbar_arrive_expect_tx(full0 + 8u * i, expect);
          if (loads_a) load_a(st, fbar(i), i * kBK, f0);
        }
        ptx::grid_dependency_wait();
        if (blockIdx.x == 0) record_stamp(a.stamp);
        for (int i = 0; i < pre; ++i)
          if (!(wh && i == 0) && loads_b)
            load_b(sbase + i * stage_bytes + NA * kATileBytes, fbar(i), i * kBK, t0 * a.nt);
        issued = pre;
        int it = 0;
        bool stop = false;
        RingPos rp(a.stages);
        for (int item = first; item < tiles && !stop; item += step) {
          int ft, tt;
          tile_of(item, ft, tt);
          for (int kb = 0; kb < KB; ++kb, ++it, rp.next()) {
            if (it < pre) continue;  // issued above
            const int s = rp.s;
            if (!ptx::mbar_wait(empty0 + 8u * s, rp.ph ^ 1u, abort_flag, a.err, kDevWaitEmpty,
                                a.wait_ns)) {
              stop = true;
              break;
            }
            const uint32_t st = sbase + s * stage_bytes;
            const uint32_t fb = fbar(s);
            if (arms) ptx::mbar_arrive_expect_tx(full0 + 8u * s, expect);
            if (loads_a) load_a(st, fb, kb * kBK, ft);
            if (loads_b) load_b(st + NA * kATileBytes, fb, kb * kBK, tt * a.nt);
            issued = it + 1;
          }
        }
      }
      // no copy may still be in flight at exit (a flag of our own: an abort
      // must not cut these waits short).  TWO: the second CTA's copies count
      // on the first CTA's barriers, which the first CTA waits for, and
      // neither CTA leaves before the final cluster barrier.
      volatile int drain = 0;
      if (arms)
        for (int i = (issued > a.stages ? issued - a.stages : 0); i < issued; ++i)
          if (!(wh && i == 0))
            ptx::mbar_wait(full0 + 8u * (i % a.stages), static_cast<uint32_t>(i / a.stages) & 1u,
                           &drain, nullptr, 0, a.wait_ns);
    }
  } else if (warp == 1) {
    // TWO: the pair's MMAs are issued by the first CTA alone
    if (lane == 0 && (!TWO || rank == 0)) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = ptx::idesc_bf16(TWO ? 2 * kBM : kBM, a.nt);
      const uint64_t da0 = ptx::sdesc_sw128(sbase);
      const uint64_t db0 = ptx::sdesc_sw128(sbase + NA * kATileBytes);
      const uint64_t stage_units = stage_bytes >> 4;
      RingPos rp(a.stages);
      int it = 0, lt = 0;
      bool stop = false;
      for (int item = first; item < tiles && !stop; item += step, ++lt) {
        const int b = lt & 1;
        const int use = lt >> 1;
        if (lt >= 2) {
          const uint32_t par = static_cast<uint32_t>(use - 1) & 1u;
          const bool ok = TWO ? ptx::mbar_wait_cluster(acce0 + 8u * b, par, abort_flag, a.err,
                                                       kDevWaitAccum, a.wait_ns)
                              : ptx::mbar_wait(acce0 + 8u * b, par, abort_flag, a.err,
                                               kDevWaitAccum, a.wait_ns);
          if (!ok) break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b) * acc_cols;
        for (int kb = 0; kb < KB; ++kb, ++it, rp.next()) {
          const int s = rp.s;
          if (!ptx::mbar_wait(full0 + 8u * s, rp.ph, abort_flag, a.err, kDevWaitFull, a.wait_ns)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t da = da0 + static_cast<uint64_t>(s) * stage_units;
          const uint64_t db = db0 + static_cast<uint64_t>(s) * stage_units;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            if (TWO) {
              ptx::mma_bf16_cg2(d, da + 2 * kk, db + 2 * kk, idesc, acc);
              if (NA == 2)
                ptx::mma_bf16_cg2(d + static_cast<uint32_t>(a.nt), da + (kATileBytes >> 4) + 2 * kk,
                                  db + 2 * kk, idesc, acc);
            } else {
              ptx::mma_bf16(d, da + 2 * kk, db + 2 * kk, idesc, acc);
              if (NA == 2)
                ptx::mma_bf16(d + static_cast<uint32_t>(a.nt), da + (kATileBytes >> 4) + 2 * kk,
                              db + 2 * kk, idesc, acc);
            }
          }
          // PAIR: the stage is free only once both CTAs have consumed it
          // (TWO: once the pair's MMA has, in both CTAs)
          if (TWO)
            ptx::mma_commit_cg2_mc(empty0 + 8u * s, static_cast<uint16_t>(0x3));
          else if (PAIR)
            ptx::mma_commit_mc(empty0 + 8u * s, static_cast<uint16_t>(0x3));
          else
            ptx::mma_commit(empty0 + 8u * s);
        }
        if (TWO)
          ptx::mma_commit_cg2_mc(accf0 + 8u * b, static_cast<uint16_t>(0x3));
        else
          ptx::mma_commit(accf0 + 8u * b);
      }
      // every product issued has completed before TMEM is released
      if (TWO)
        ptx::mma_commit_cg2(done_bar);
      else
        ptx::mma_commit(done_bar);
      volatile int drain = 0;
      ptx::mbar_wait(done_bar, 0, &drain, nullptr, 0, a.wait_ns);
    }
  } else {
    if constexpr (staged_epilogue(KIND)) {
      // ------------------------------------------------ epilogue (staged)
      // Chunks of kChunk token columns: TMEM -> fp32 staging in shared memory
      // -> 16-byte stores.  The two warps of a TMEM lane quarter drain 16
      // columns each.  What a chunk reads from global memory (the residual, the
      // RoPE table rows) is requested when the chunk before it starts, across
      // tiles too, so that its latency overlaps that whole chunk.
      const int q = warp & 3;
      const int half = (warp - 2) >> 2;
      const int row = q * 32 + lane;
      const int tid_e = threadIdx.x - 64;
      const EpiOut eo = epi_out(a);
      ptx::grid_dependency_wait();  // residual written by earlier kernels
      uint4 res_cur[kPUnits], res_nxt[kPUnits];
      RopeRow rr_cur[kRopeUnits], rr_nxt[kRopeUnits];
      // RoPE positions by arithmetic: packed tokens from the row starts, else t mod S
      RowStarts rs;
      const bool rope_packed = a.rope_pos != nullptr && a.lens != nullptr;
      if (KIND == kGemmPlain && a.rope_cos != nullptr && rope_packed) rs.init(a.lens, a.lens_B, a.lens_S);
      // global reads of chunk c0 of work item `item` into (res, rr)
      auto prefetch = [&](int item, int c0, uint4 (&res)[kPUnits], RopeRow (&rr)[kRopeUnits]) {
        if (item >= tiles) return;
        int ft, tt;
        tile_of(item, ft, tt);
        const int ncols = a.nt - c0 < kChunk ? a.nt - c0 : kChunk;
        if (KIND == kGemmResidual) {
  #pragma unroll
          for (int k = 0; k < kPUnits; ++k) {
            const int u = tid_e + kPEpi * k;
            const int c = u / (kBM / 8), grp = u % (kBM / 8);
            const int t = tt * a.nt + c0 + c;
            const int f = ft * kBM + grp * 8;
            if (u < ncols * (kBM / 8) && t < Meff && f < a.N)
              res[k] = *reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(t) * a.N + f);
          }
        }
        if (KIND == kGemmPlain && a.rope_cos != nullptr && ft * kBM < a.rope_cols) {
  #pragma unroll
          for (int k = 0; k < kRopeUnits; ++k) {
            const int u = tid_e + kPEpi * k;
            const int c = u / (kBM / 16), pg = u % (kBM / 16);
            const int t = tt * a.nt + c0 + c;
            if (u < ncols * (kBM / 16) && t < Meff)
              rr[k] = rope_row_at(eo, rope_packed ? rs.pos(t) : t % a.rope_S, 8 * (pg & 3));
          }
        }
      };
      prefetch(first, 0, res_cur, rr_cur);
      int lt = 0, cc = 0;
      for (int item = first; item < tiles; item += step, ++lt) {
        const int b = lt & 1;
        const int use = lt >> 1;
        ptx::mbar_wait(accf0 + 8u * b, static_cast<uint32_t>(use) & 1u, abort_flag, a.err,
                       kDevWaitAccum, a.wait_ns);
        // all epilogue threads leave together: whoever gave up raised the flag
        // before this barrier, so everyone reads the same value after it
        ptx::named_barrier_sync(1, kPEpi);
        if (*abort_flag) break;
        ptx::tc_fence_after();
        int ft, tt;
        tile_of(item, ft, tt);
        const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b) * acc_cols;
        const bool rope_tile =
            KIND == kGemmPlain && a.rope_cos != nullptr && ft * kBM < a.rope_cols;
        for (int c0 = 0; c0 < a.nt; c0 += kChunk, ++cc) {
          float* buf = staging + (cc & 1) * (kChunk * kSld);
          const int ncols = a.nt - c0 < kChunk ? a.nt - c0 : kChunk;
          // the next chunk's global reads (of this tile, or the next tile's first)
          if (c0 + kChunk < a.nt)
            prefetch(item, c0 + kChunk, res_nxt, rr_nxt);
          else
            prefetch(item + step, 0, res_nxt, rr_nxt);
          const int j0 = 16 * half;  // ncols is a multiple of 16
          if (j0 < ncols) {
            float v[16];
            ptx::tmem_ld16(tq + c0 + j0, v);
  #pragma unroll
            for (int j = 0; j < 16; ++j) buf[(j0 + j) * kSld + row] = v[j];
          }
          if (c0 + kChunk >= a.nt) {
            // every TMEM read of this tile is complete: hand the accumulator back
            ptx::tc_fence_before();
            release_acc(b);
          }
          ptx::named_barrier_sync(1, kPEpi);
          // 16-byte vector stores: 8 features of one token per unit
          if (rope_tile) {
  #pragma unroll
            for (int k = 0; k < kRopeUnits; ++k) {
              const int u = tid_e + kPEpi * k;
              const int c = u / (kBM / 16), pg = u % (kBM / 16);
              const int fo = 64 * (pg >> 2) + 8 * (pg & 3);
              const int t = tt * a.nt + c0 + c;
              if (u < ncols * (kBM / 16) && t < Meff) {
                float v1[8], v2[8];
                load8_smem(buf + c * kSld + fo, v1);
                load8_smem(buf + c * kSld + fo + 32, v2);
                rope_apply_store16(eo, t, ft * kBM + fo, rr_cur[k], v1, v2);
              }
            }
          } else {
            const int units = ncols * (kBM / 8);
  #pragma unroll
            for (int k = 0; k < kPUnits; ++k) {
              const int u = tid_e + kPEpi * k;
              if (u >= units) continue;
              const int c = u / (kBM / 8), grp = u % (kBM / 8);
              const int t = tt * a.nt + c0 + c;
              const int f = ft * kBM + grp * 8;
              if (t >= Meff || f >= a.N) continue;
              float o[8];
              load8_smem(buf + c * kSld + grp * 8, o);
              if (KIND == kGemmResidual) {
                const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&res_cur[k]);
  #pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 rf = __bfloat1622float2(r2[i]);
                  o[2 * i] = rf.x + o[2 * i];
                  o[2 * i + 1] = rf.y + o[2 * i + 1];
                }
              }
              store8<KIND>(eo, t, f, o);
            }
          }
  #pragma unroll
          for (int k = 0; k < kPUnits; ++k) res_cur[k] = res_nxt[k];
  #pragma unroll
          for (int k = 0; k < kRopeUnits; ++k) rr_cur[k] = rr_nxt[k];
        }
      }
    } else {
      // ------------------------------------------------ epilogue (direct)
      // The two warps of a TMEM lane quarter take alternate blocks of token
      // columns.
      const int q = warp & 3;
      const int half = (warp - 2) >> 2;
      const int lrow = q * 32 + lane;         // accumulator row (TMEM lane)
      const bool upper = (lane & 16) != 0;    // GeGLU-il: the gate row of the pair
      ptx::grid_dependency_wait();            // the output may be read by earlier kernels
      int lt = 0;
      for (int item = first; item < tiles; item += step, ++lt) {
        const int b = lt & 1;
        const int use = lt >> 1;
        ptx::mbar_wait(accf0 + 8u * b, static_cast<uint32_t>(use) & 1u, abort_flag, a.err,
                       kDevWaitAccum, a.wait_ns);
        // all epilogue threads leave together: whoever gave up raised the flag
        // before this barrier, so everyone reads the same value after it
        ptx::named_barrier_sync(1, kPEpi);
        if (*abort_flag) break;
        ptx::tc_fence_after();
        int ft, tt;
        tile_of(item, ft, tt);
        const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b) * acc_cols;
        // the output feature of this accumulator row
        const int f = KIND == kGemmGegluIl ? ft * 64 + (lrow >> 5) * 16 + (lrow & 15) : ft * kBM + lrow;
        const bool f_ok = f < a.N;
        unsigned short* yb = reinterpret_cast<unsigned short*>(a.y);
        // GeGLU-il, 16 token columns from t0: lanes l < 16 hold the GELU half,
        // l + 16 the gate half of the same feature; the lower lanes finish
        // even tokens, the upper odd ones
        auto il16 = [&](const float* v, int t0) {
          float o[16];
  #pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = __shfl_xor_sync(0xffffffffu, v[j], 16);
  #pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float h = upper ? o[2 * jj + 1] : v[2 * jj];
            const float gt = upper ? v[2 * jj + 1] : o[2 * jj];
            const int t = t0 + 2 * jj + (upper ? 1 : 0);
            const float val = gelu_erf(h) * gt;
            if (t < Meff && f_ok)
              yb[static_cast<size_t>(t) * a.N + f] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
          }
        };
        int c_first = 16 * half;
        if (KIND == kGemmGegluIl) {
          // whole blocks of 64 columns in one TMEM load each (one wait per 64
          // columns instead of per 16: the load latency under the main loop's
          // TMEM traffic is what bounds this epilogue); the two warps of a
          // lane quarter alternate blocks, the last partial block goes 16 by 16
          const int full64 = a.nt / 64;
          for (int blk = half; blk < full64; blk += 2) {
            float v64[64];
            ptx::tmem_ld64(tq + blk * 64, v64);
  #pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) il16(v64 + 16 * g4, tt * a.nt + blk * 64 + 16 * g4);
          }
          c_first = full64 * 64 + 16 * half;
        }
        for (int c = c_first; c < a.nt; c += 32) {
          const int t0 = tt * a.nt + c;
          float v[16];
          if (NA == 2) {
            float g[16];
            ptx::tmem_ld16x2(tq + c, tq + a.nt + c, v, g);
  #pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = t0 + j;
              const float val = gelu_erf(v[j]) * g[j];
              if (t < Meff && f_ok)
                yb[static_cast<size_t>(t) * a.N + f] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
            }
          } else {
            ptx::tmem_ld16(tq + c, v);
            il16(v, t0);
          }
        }
        // every TMEM read of this tile by this thread is complete: its share
        // of the accumulator goes back to the MMA issuer
        ptx::tc_fence_before();
        release_acc(b);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // PAIR: neither CTA leaves while the other may still multicast into it or
  // arrive on its barriers
  if (PAIR) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (TWO)
      ptx::tmem_dealloc_cg2(tmem, a.tmem_cols);
    else
      ptx::tmem_dealloc(tmem, a.tmem_cols);
  }
}

cudaError_t configure_kernels();

uint32_t pow2_cols(uint32_t n) {
  uint32_t c = 32;
  while (c < n) c <<= 1;
  return c;
}

template <int KIND>
cudaError_t launch_kind(const GemmPlan& p, const GemmOperands& o, Launch l) {
  cudaError_t ce = configure_kernels();
  if (ce != cudaSuccess) return ce;
  GemmArgs a;
  a.M = p.M;
  a.N = p.N;
  a.k_blocks = p.k_blocks;
  a.nt = p.nt;
  a.splits = p.splits;
  a.stages = p.stages;
  a.feat_tiles = p.feat_tiles;
  a.token_tiles = p.token_tiles;
  a.tmem_cols = p.tmem_cols;
  const int na = KIND == kGemmGeglu ? 2 : 1;
  const size_t stage_bytes =
      static_cast<size_t>(na) * kATileBytes + static_cast<size_t>(p.x_box()) * 128;
  size_t data = stage_bytes * p.stages;
  if (p.persistent) {
    if (staged_epilogue(KIND)) data += kStagingBytes;
  } else {
    const size_t part = p.splits == 1 ? static_cast<size_t>(p.nt) * kSld * 4
                                      : split_reduce_bytes(na, p.nt, p.splits);
    if (part > data) data = part;
  }
  a.ctrl_offset = static_cast<uint32_t>(data);
  a.y = o.y;
  a.residual = o.residual;
  a.y_f32 = KIND == kGemmResidual ? o.y_f32 : nullptr;
  a.err = o.err;
  a.partials = o.partials;
  a.rope_cos = o.rope_cos;
  a.rope_sin = o.rope_sin;
  a.rope_S = o.rope_S;
  a.rope_cols = o.rope_cols;
  a.lens = o.lens;
  a.lens_B = o.lens_B;
  a.lens_S = o.lens_S;
  a.rope_pos = o.rope_pos;
  a.ln_x = o.ln_x;
  a.ln_gamma = o.ln_gamma;
  a.ln_eps = o.ln_eps;
  a.stamp = l.stamp;
  a.wait_ns = o.wait_ns;
  a.withhold = o.withhold ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(p.persistent ? kPThreads : kThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (p.persistent) {
    cfg.gridDim = dim3(p.grid_ctas, 1, 1);
    if (p.pair) {
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = 2;
      attr[n].val.clusterDim.y = 1;
      attr[n].val.clusterDim.z = 1;
      ++n;
    }
  } else {
    cfg.gridDim = dim3(p.feat_tiles, p.token_tiles, p.splits);
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = p.splits;
    ++n;
  }
  if (l.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  if (p.persistent && p.pair == 1)
    return cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<KIND, 1>, o.w, o.w2, o.x, a);
  if (p.persistent && p.pair == 2)
    return cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<KIND, 2>, o.w, o.w2, o.x, a);
  if (p.persistent && p.pair == 3)
    return cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<KIND, 3>, o.w, o.w2, o.x, a);
  if (p.persistent)
    return cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<KIND, 0>, o.w, o.w2, o.x, a);
  if constexpr (KIND == kGemmGegluIl) {
    return cudaErrorInvalidValue;  // persistent plans only
  } else {
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<KIND>, o.w, o.w2, o.x, a);
  }
}

}  // namespace

namespace {

const void* kernel_ptr(int kind) {
  switch (kind) {
    case kGemmPlain: return reinterpret_cast<const void*>(&gemm_tc_kernel<kGemmPlain>);
    case kGemmResidual: return reinterpret_cast<const void*>(&gemm_tc_kernel<kGemmResidual>);
    default: return reinterpret_cast<const void*>(&gemm_tc_kernel<kGemmGeglu>);
  }
}

const void* persistent_ptr(int kind, int pair) {
  switch (kind) {
    case kGemmPlain:
      return pair == 1   ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmPlain, 1>)
             : pair == 2 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmPlain, 2>)
             : pair == 3 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmPlain, 3>)
                         : reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmPlain, 0>);
    case kGemmResidual:
      return pair == 1   ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmResidual, 1>)
             : pair == 2 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmResidual, 2>)
             : pair == 3 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmResidual, 3>)
                         : reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmResidual, 0>);
    case kGemmGeglu:
      return pair == 1   ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGeglu, 1>)
             : pair == 2 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGeglu, 2>)
             : pair == 3 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGeglu, 3>)
                         : reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGeglu, 0>);
    default:
      return pair == 1   ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGegluIl, 1>)
             : pair == 2 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGegluIl, 2>)
             : pair == 3 ? reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGegluIl, 3>)
                         : reinterpret_cast<const void*>(&gemm_persistent_kernel<kGemmGegluIl, 0>);
  }
}

// Clusters of two persistent CTAs with this shared memory that can be
// resident at once; -1 when there is no device to ask.
int max_active_pairs(int kind, size_t smem, int mode);

// Opt every kernel variant into the full dynamic shared memory once.
cudaError_t configure_kernels() {
  static cudaError_t status = cudaErrorNotReady;
  static std::once_flag once;
  std::call_once(once, [] {
    status = cudaSuccess;
    for (int k = kGemmPlain; k <= kGemmGegluIl && status == cudaSuccess; ++k) {
      if (k <= kGemmGeglu) {
        status = cudaFuncSetAttribute(kernel_ptr(k), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmemLimit));
        // split-K clusters of up to 16 CTAs (the portable limit is 8)
        if (status == cudaSuccess)
          status = cudaFuncSetAttribute(kernel_ptr(k),
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      }
      for (int pair = 0; pair < 4 && status == cudaSuccess; ++pair)
        status = cudaFuncSetAttribute(persistent_ptr(k, pair),
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmemLimit));
    }
  });
  return status;
}

// How many clusters of `splits` CTAs with this shared memory can be resident
// at once on the current device; -1 when there is no device to ask.
int max_active_clusters(int kind, size_t smem, int splits) {
  static std::mutex mu;
  static std::map<std::tuple<int, size_t, int>, int> cache;
  const auto key = std::make_tuple(kind, smem, splits);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && configure_kernels() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = splits;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel_ptr(kind), &cfg) != cudaSuccess) n = -1;
  }
  cudaGetLastError();  // a failed query must not leave a sticky-looking error behind
  std::lock_guard<std::mutex> g(mu);
  cache[key] = n;
  return n;
}

int max_active_pairs(int kind, size_t smem, int mode) {
  static std::mutex mu;
  static std::map<std::tuple<int, size_t, int>, int> cache;
  const auto key = std::make_tuple(kind, smem, mode);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && configure_kernels() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, persistent_ptr(kind, mode), &cfg) != cudaSuccess) n = -1;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> g(mu);
  cache[key] = n;
  return n;
}

}  // namespace

namespace {

// Fills everything that follows from (M, N, K, kind, nt, splits); false if the
// tile does not fit in shared memory or TMEM.
bool finish_plan(GemmPlan* r) {
  const int na = r->kind == kGemmGeglu ? 2 : 1;
  const size_t stage_bytes = static_cast<size_t>(na) * kATileBytes + static_cast<size_t>(r->x_box()) * 128;
  const size_t budget = kSmemLimit - kCtrlBytes - kLnStatsBytes - 1024;
  if (r->persistent) {
    // ring of stages (+ the staging of the plain and residual epilogues); two
    // accumulators in TMEM
    const size_t staging = staged_epilogue(r->kind) ? kStagingBytes : 0;
    int stages = static_cast<int>((budget - staging) / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages > r->k_blocks) stages = r->k_blocks;
    if (stages < 2 && r->k_blocks >= 2) return false;
    if (stages < 1) return false;
    r->stages = stages;
    r->smem_bytes = stage_bytes * stages + staging + kCtrlBytes + 1024;
    r->tmem_cols = pow2_cols(static_cast<uint32_t>(2 * na * r->nt));
    return r->tmem_cols <= 512 && r->smem_bytes <= kSmemLimit;
  }
  const int max_kb = (r->k_blocks + r->splits - 1) / r->splits;  // K blocks of the largest split
  // at most ~110 KB of stages, so that two CTAs (this projection's and the
  // next one's, under programmatic dependent launch) share an SM
  const size_t split_budget = 110 * 1024;
  int stages = static_cast<int>((budget < split_budget ? budget : split_budget) / stage_bytes);
  if (stages > 8) stages = 8;
  if (stages > max_kb) stages = max_kb;
  if (stages < 1) return false;
  r->stages = stages;
  size_t data = stage_bytes * stages;
  // fp32 staging tile of the epilogue, or (split-K) this rank's slices of the
  // cluster's partials, both in the idle ring once the accumulator is ready
  const size_t part = r->splits > 1 ? split_reduce_bytes(na, r->nt, r->splits)
                                    : static_cast<size_t>(r->nt) * kSld * 4;
  if (part > budget) return false;
  if (part > data) data = part;
  r->workspace_bytes = r->splits > 1 ? static_cast<size_t>(r->feat_tiles) * r->token_tiles *
                                           r->splits * na * r->nt * kBM * 4
                                     : 0;
  r->smem_bytes = data + kCtrlBytes + kLnStatsBytes + 1024;
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
               GemmPlan* p, bool allow_persistent, double split_cost) {
  if (M <= 0 || N <= 0 || K <= 0 || K % kBK != 0 || N % 8 != 0) return false;
  if (kind < kGemmPlain || kind > kGemmGegluIl) return false;
  // the interleaved GeGLU: persistent (unsplit) plans over 64-feature tiles
  if (kind == kGemmGegluIl && (!allow_persistent || N % 64 != 0 || force_splits > 1)) return false;
  if (force_nt > 0 && (force_nt % 16 != 0 || force_nt > 256)) return false;
  if (force_splits > 0 && (force_splits > kMaxSplits || force_splits > K / kBK)) return false;
  if (num_sms <= 0) num_sms = 148;
  const int na = kind == kGemmGeglu ? 2 : 1;
  // Candidates: every token tile nt (a multiple of 16 up to 256) x split-K
  // factor.  Split 1 runs the persistent kernel (one CTA per SM walking the
  // tiles, epilogue overlapped with the next tile's main loop); splits > 1
  // run one CTA per (tile, split) in clusters.  Cost in units of one 16 KB
  // weight tile streamed by one CTA:
  //   persistent: ceil(tiles / CTAs) x (K blocks x unit + 0.3) + 2
  //   split:      waves x (K blocks per split x unit + split_cost + partial
  //               round trip),
  // a wave being as many clusters as the device can hold at once.
  GemmPlan best;
  double best_cost = 0.0;
  bool found = false;
  const int nt_max = ((M + 15) / 16) * 16 < 256 ? ((M + 15) / 16) * 16 : 256;
  for (int nt = 16; nt <= nt_max; nt += 16) {
    if (force_nt > 0 && nt != force_nt) continue;
    GemmPlan r;
    r.M = M;
    r.N = N;
    r.K = K;
    r.kind = kind;
    r.k_blocks = K / kBK;
    r.nt = nt;
    r.token_tiles = (M + nt - 1) / nt;
    r.feat_tiles = kind == kGemmGegluIl ? N / 64 : (N + kBM - 1) / kBM;
    const int tiles = r.token_tiles * r.feat_tiles;
    const double unit = (na * kATileBytes + static_cast<double>(nt) * 128.0) / kATileBytes;
    const int s_lo = force_splits > 0 ? force_splits : 1;
    const int s_hi = force_splits > 0                   ? force_splits
                     : (tiles >= num_sms || kind == kGemmGegluIl) ? 1
                                                                   : kMaxSplits;
    for (int S = s_lo; S <= s_hi && S <= r.k_blocks; ++S) {
      GemmPlan c = r;
      c.splits = S;
      c.persistent = (S == 1) && allow_persistent;
      if (!finish_plan(&c)) continue;
      double cost;
      if (c.persistent) {
        c.grid_ctas = tiles < num_sms ? tiles : num_sms;
        const int per_cta = (tiles + c.grid_ctas - 1) / c.grid_ctas;
        cost = per_cta * (c.k_blocks * unit + 0.3) + 2.0;
      } else {
        int mac = max_active_clusters(kind, c.smem_bytes, S);
        if (mac <= 0) mac = num_sms / S;  // no device to ask: one CTA per SM
        if (mac <= 0) continue;
        const int waves = (tiles + mac - 1) / mac;
        const int kb_per = (c.k_blocks + S - 1) / S;
        // + the partial tile written to and read back from L2 (about half the
        //   cost of streaming the same bytes from HBM)
        const double partial = 0.5 * na * c.nt * kBM * 4.0 / kATileBytes;
        cost = waves * (kb_per * unit + split_cost + partial);
      }
      if (!found || cost < best_cost - 1e-9) {
        best = c;
        best_cost = cost;
        found = true;
      }
    }
  }
  if (!found) return false;
  *p = best;
  return true;
}

bool make_pair_plan(GemmPlan* p, int mode) {
  if (!p->persistent || p->pair != 0 || mode < 1 || mode > 3) return false;
  GemmPlan q = *p;
  q.pair = mode;
  // mode 3: a CTA's stage holds half the token tile (more stages fit)
  if (mode == 3 && !finish_plan(&q)) return false;
  const int pairs_max = max_active_pairs(q.kind, q.smem_bytes, mode);
  if (pairs_max <= 0) return false;
  const int items = mode == 2 ? q.feat_tiles * ((q.token_tiles + 1) / 2)
                              : ((q.feat_tiles + 1) / 2) * q.token_tiles;
  q.grid_ctas = 2 * (items < pairs_max ? items : pairs_max);
  *p = q;
  return true;
}

int plan_candidates(int M, int N, int K, int kind, int num_sms, GemmPlan* out, int max_out) {
  // the model's choice under a range of split-K overhead weights, and the
  // best plan without split-K: distinct plans only
  const double costs[] = {2.0, 8.0, 16.0, 32.0};
  int n = 0;
  auto add = [&](const GemmPlan& c) {
    for (int i = 0; i < n; ++i)
      if (out[i].nt == c.nt && out[i].splits == c.splits && out[i].persistent == c.persistent)
        return;
    if (n < max_out) out[n++] = c;
  };
  for (double sc : costs) {
    GemmPlan c;
    if (plan_gemm(M, N, K, kind, num_sms, 0, 0, &c, true, sc)) add(c);
  }
  GemmPlan c;
  if (plan_gemm(M, N, K, kind, num_sms, 1, 0, &c, true)) add(c);
  // persistent plans with more, smaller tiles per CTA: the largest token tile
  // that gives each CTA k tiles, k = 2..4 (the last tile's epilogue is the
  // part no main loop hides, and it shrinks with the tile)
  const int sms = num_sms > 0 ? num_sms : 148;
  const int ftiles = kind == kGemmGegluIl ? N / 64 : (N + kBM - 1) / kBM;
  for (int k = 2; k <= 4; ++k) {
    int pick = 0;
    for (int nt = 16; nt <= 256; nt += 16) {
      const int tiles = ((M + nt - 1) / nt) * ftiles;
      if ((tiles + sms - 1) / sms <= k) {
        pick = nt;
        break;
      }
    }
    if (pick > 0 && plan_gemm(M, N, K, kind, num_sms, 1, pick, &c, true)) add(c);
  }
  // the persistent candidates again in clusters of two: one two-CTA MMA per
  // pair first, then the multicast pairings
  const int base = n;
  for (int mode : {3, 1, 2})
    for (int i = 0; i < base && n < max_out; ++i) {
      GemmPlan pp = out[i];
      if (pp.persistent && make_pair_plan(&pp, mode)) out[n++] = pp;
    }
  return n;
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

bool make_tmap_geglu_il(CUtensorMap* m, const void* w, uint64_t N, uint64_t K) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr || w == nullptr || N == 0 || N % 64 != 0 || K == 0 || (K * 2) % 16 != 0)
    return false;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) != 0) return false;
  std::memset(m, 0, sizeof(*m));
  // (k, row in a block of 16, half, block): a box of 4 blocks is 128 rows,
  // 16 GELU rows then the 16 gate rows of the same features, four times
  const cuuint64_t dims[4] = {K, 16, 2, N / 16};
  const cuuint64_t strides[3] = {K * 2, N * K * 2, 16 * K * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kBK), 16, 2, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm(const GemmPlan& p, const GemmOperands& o, Launch l) {
  // the TMA box must match the shared-memory stage the plan reserves for it
  if (o.x_box_rows != p.x_box()) return cudaErrorInvalidValue;
  // split-K needs its workspace, 16-byte aligned
  if (p.splits > 1 && (o.partials == nullptr || o.partials_bytes < p.workspace_bytes ||
                       (reinterpret_cast<uintptr_t>(o.partials) & 15u) != 0))
    return cudaErrorInvalidValue;
  // LayerNorm on load: split kernel only, K a multiple of 256 up to 2048
  if (o.ln_x != nullptr &&
      (p.persistent || o.ln_gamma == nullptr || p.K % 256 != 0 || p.K > 2048))
    return cudaErrorInvalidValue;
  // RoPE in the epilogue: plain kind, whole 64-wide heads in whole 128-feature tiles
  if (o.rope_cos != nullptr &&
      (p.kind != kGemmPlain || o.rope_sin == nullptr || o.rope_S < 1 || o.rope_cols % kBM != 0))
    return cudaErrorInvalidValue;
  switch (p.kind) {
    case kGemmPlain: return launch_kind<kGemmPlain>(p, o, l);
    case kGemmResidual: return launch_kind<kGemmResidual>(p, o, l);
    case kGemmGeglu: return launch_kind<kGemmGeglu>(p, o, l);
    case kGemmGegluIl: return launch_kind<kGemmGegluIl>(p, o, l);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_node_retarget(cudaGraphExec_t exec, cudaGraphNode_t node, const void* old_y,
                               void* new_y) {
  cudaKernelNodeParams p = {};
  cudaError_t e = cudaGraphKernelNodeGetParams(node, &p);
  if (e != cudaSuccess) return e;
  const void* split = reinterpret_cast<const void*>(&gemm_tc_kernel<kGemmResidual>);
  if ((p.func != split && p.func != persistent_ptr(kGemmResidual, 0) &&
       p.func != persistent_ptr(kGemmResidual, 1) && p.func != persistent_ptr(kGemmResidual, 2) &&
       p.func != persistent_ptr(kGemmResidual, 3)) ||
      p.kernelParams == nullptr)
    return cudaErrorInvalidValue;
  // arguments: weight map, gate map, activation map, GemmArgs
  GemmArgs a = *static_cast<const GemmArgs*>(p.kernelParams[3]);
  bool hit = false;
  if (a.y == old_y) {
    a.y = static_cast<bf16*>(new_y);
    hit = true;
  }
  if (a.y_f32 != nullptr && a.y_f32 == old_y) {
    a.y_f32 = static_cast<float*>(new_y);
    hit = true;
  }
  if (!hit) return cudaErrorInvalidValue;
  void* args[4] = {p.kernelParams[0], p.kernelParams[1], p.kernelParams[2], &a};
  p.kernelParams = args;
  p.extra = nullptr;
  e = cudaGraphExecKernelNodeSetParams(exec, node, &p);
  if (e == cudaSuccess) e = cudaGraphKernelNodeSetParams(node, &p);  // keep the template in step
  return e;
}

}  // namespace laya
