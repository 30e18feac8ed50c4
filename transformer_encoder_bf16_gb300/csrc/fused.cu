// fused.cu -- the whole forward pass of a short request (at most 128 tokens)
// as ONE persistent kernel: one CTA per SM in clusters of four, launched
// cooperatively (every CTA resident), each walking the same phase program
//
//   E:   x = LN_emb(E[ids])                    rows spread over every CTA
//   per layer l (FN first when l is the first decision layer):
//   FN:  x = LN_final(x)
//   QKV: qkv = RoPE(LN_attn(x) Wqkv^T)         split-K tiles, LN applied on load
//   ATT: ctx = attention(qkv)                  one (row, head) per CTA, mma.sync
//   O:   x = x + ctx Wo^T
//   UP:  g = gelu(LN_mlp(x) Win^T) * (LN_mlp(x) Wgate^T)
//   DN:  x = x + g Wdown^T                     (last layer: into out)
//
// The layer equations are those of the layer-by-layer path (encoder.cu); what
// differs is the schedule.  At a few dozen tokens every projection is a
// stream of weights past a tiny activation matrix, and a chain of separate
// kernels is bound by launch and drain latency, not by HBM.  Here the weights
// never wait: a producer thread per CTA streams its share of the weight tiles
// of the coming phases through an 8-slot ring by TMA, as far ahead as the
// ring allows; only the small activation tiles wait for the previous phase.
// ("Implementation priorities" of "[Performance]: Optimize native Rust/CUDA
// Laya inference #66": the short-sequence shapes are weight-streaming bound.)
//
// Roles (256 threads):
//   warp 0 lane 0   weight producer (TMA, 16 KB tiles [128 features x 64 k])
//   warp 1          TMEM owner; lane 0 issues tcgen05.mma into two fp32
//                   accumulators (double-buffered, 256 columns each)
//   warps 2-5       epilogue: drain TMEM, split-K partials, reductions and
//                   fused epilogues; attention; embedding and final-norm rows
//   warps 6-7       activation loader: reads x / ctx / g (L2), applies the
//                   LayerNorm, writes [nt x 64] BF16 tiles in the 128-byte
//                   swizzled K-major layout the MMA reads
//
// Split-K inside a thread-block cluster of four CTAs.  Each 128-feature tile
// of a projection belongs to one cluster (a host-side greedy assignment
// balances the weight bytes of the clusters); its K range is split among the
// cluster's four CTAs.  Each CTA drains its fp32 partial tile from TMEM into
// its own shared memory (token-major), tells its peers (remote mbarrier
// arrivals, release at cluster scope), and reduces one quarter of the
// tokens by reading the four partials through distributed shared memory, in
// rank order (deterministic); the fused epilogue (RoPE, GeGLU, residual) then
// writes BF16 to global memory.  The residual epilogues also write, per token
// and 128-feature slice, the mean and the sum of squared deviations of the
// stored BF16 values; the next LayerNorm combines the slices (Chan et al.'s
// pairwise update) instead of re-reading the row.
//
// Phase order.  Each CTA counts itself on the phase's ready counter after its
// last output of the phase is written (release); readers of a phase's outputs
// wait for the count (acquire).  Counters only grow: a launch waits for
// generation x CTAs, the generation being one more than the previous launch's
// (kept in device memory and advanced by CTA 0 once every CTA has finished).
// Every wait is bounded by a time limit; on expiry the kernel records an
// error, raises a grid-wide abort word that every other wait also watches,
// drains its copies and frees its TMEM.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace laya {

namespace {

constexpr int kFThreads = 256;
constexpr int kFBM = 128;                   // features per tile (MMA M)
constexpr int kFBK = 64;                    // K per k-block
constexpr int kWSlots = 8;                  // weight ring
constexpr int kASlotsMax = 4;               // activation ring slots (see Ctl::nas)
constexpr uint32_t kWSlotBytes = kFBM * kFBK * 2;   // 16 KB
constexpr uint32_t kARingBytes = 64 * 1024;          // activation ring
constexpr uint32_t kASlotBytes = kARingBytes / kASlotsMax;  // up to 128 token rows
constexpr uint32_t kAttnBytes = 2 * 128 * 128;      // K and V of one head, <= 128 keys
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffA = kOffW + kWSlots * kWSlotBytes;
constexpr uint32_t kOffAttn = kOffA + kARingBytes;
constexpr uint32_t kOffLn = kOffAttn + kAttnBytes;  // [128 tokens][mean, rstd]
constexpr uint32_t kOffCtrl = kOffLn + 128 * 8;
constexpr uint32_t kCtrlBytes = 512;
constexpr uint32_t kFusedSmem = kOffCtrl + kCtrlBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;                            // two accumulators of 256
constexpr int kGammaPre = 4;  // loader: gamma chunks of a unit's first k-blocks loaded up front
constexpr int kCluster = 4;   // CTAs per cluster = K splits of a tile
// split-K staging of this CTA's partial tile: the activation ring and the
// attention tiles, both idle while a cluster reduces (contiguous, 96 KB)
constexpr uint32_t kOffRed = kOffA;
constexpr uint32_t kRedBytes = kOffLn - kOffA;

enum PhaseKind : int { kPhEmbed, kPhFinal, kPhQkv, kPhAttn, kPhOut, kPhUp, kPhDown };
enum MapIdx : int { kMapQkv = 0, kMapOut = 1, kMapUpIn = 2, kMapUpGate = 3, kMapDown = 4 };

// Device error codes of this kernel (first error wins).
enum FusedError : int {
  kFErrWeight = 11,   // weight producer: no free ring slot
  kFErrMma = 12,      // MMA issuer: operand tile never arrived
  kFErrDrain = 13,    // epilogue: accumulator never completed
  kFErrAct = 14,      // loader: activation slot never freed
  kFErrPhase = 15,    // a phase's ready count never reached
  kFErrTile = 16,     // a cluster peer's partial (or its release of ours) never came
};

struct Phase {
  int kind, layer, idx;  // idx: position in the program (ready counter index)
  int gemm;              // 0..3 for the four projections, -1 otherwise
};

struct Ctl {
  uint32_t wfull, wempty, afull, aempty, accfull, accempty, mma_done;
  uint32_t aload;      // activation tile landed (TMA), per ring slot
  uint32_t kvbar;      // attention Q, K and V tiles landed
  uint32_t red_ready;  // every CTA of the cluster has staged its partial (4 arrivals)
  uint32_t red_done;   // every CTA of the cluster has read this CTA's partial (4 arrivals)
  volatile int* cta_abort;
  uint32_t* tmem_slot;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

__device__ __forceinline__ uint4 ldcg16(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

// Arrival on the mbarrier at shared::cluster address `bar` (this CTA's or a
// peer's), releasing this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// mbarrier phase test with acquire ordering at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void cluster_arrive_wait() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void sts32f(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 BF16, row) * B (16x8 BF16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float gelu_erf(float z) {
  return (0.5f * z) * (1.0f + erff(z * 0.70710678118654752f));
}

// Raises the grid-wide abort and records `code` (first error wins).
__device__ __forceinline__ void raise_abort(const FusedArgs& a, const Ctl& c, int code) {
  *c.cta_abort = 1;
  atomicExch(a.sync + 2, 1u);
  if (a.err) atomicCAS(a.err, 0, code);
}

__device__ __forceinline__ bool aborted(const FusedArgs& a, const Ctl& c) {
  if (*c.cta_abort) return true;
  if (ld_volatile_u32(a.sync + 2) != 0) {
    *c.cta_abort = 1;
    return true;
  }
  return false;
}

// Waits are bounded in SM clock cycles (a cheap, SM-local counter; the global
// timer is slow to read and would delay noticing a completed barrier): the
// limit is kWaitLimitCycles (about 2 s at the top clock, longer when the
// clock is lower).  They poll only on-chip state (the mbarrier or counter,
// the CTA's abort flag) for the first kSlowWaitCycles; only a wait that long
// also reads the grid-wide abort word (a global load, kept off the fast path).
constexpr long long kWaitLimitCycles = 4000000000ll;
constexpr long long kSlowWaitCycles = 40000;

// Bounded wait on an mbarrier phase that also gives up when the grid aborts.
__device__ bool fwait(const FusedArgs& a, const Ctl& c, uint32_t bar, uint32_t parity, int code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t n = 0;
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.cta_abort) return false;
    const long long dt = clock64() - t0;
    if (dt > kSlowWaitCycles && (++n & 255u) == 0 && aborted(a, c)) return false;
    if (dt > kWaitLimitCycles) {
      raise_abort(a, c, code);
      return false;
    }
  }
}

// As fwait, acquiring at cluster scope (barriers that cluster peers arrive on).
__device__ bool fwait_cluster(const FusedArgs& a, const Ctl& c, uint32_t bar, uint32_t parity,
                              int code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*c.cta_abort) return false;
    const long long dt = clock64() - t0;
    if (dt > kSlowWaitCycles && (++n & 255u) == 0 && aborted(a, c)) return false;
    if (dt > kWaitLimitCycles) {
      raise_abort(a, c, code);
      return false;
    }
  }
}

// Bounded wait until *ctr reaches target (wrap-safe), with acquire ordering.
__device__ bool wait_count(const FusedArgs& a, const Ctl& c, const uint32_t* ctr, uint32_t target,
                           int code) {
  if (static_cast<int32_t>(ld_acquire(ctr) - target) >= 0) return true;
  const long long t0 = clock64();
  uint32_t n = 0;
  while (true) {
    if (static_cast<int32_t>(ld_acquire(ctr) - target) >= 0) return true;
    if (*c.cta_abort) return false;
    const long long dt = clock64() - t0;
    if (dt > kSlowWaitCycles && (++n & 15u) == 0 && aborted(a, c)) return false;
    if (dt > kWaitLimitCycles) {
      raise_abort(a, c, code);
      return false;
    }
  }
}

// ------------------------------------------------------- the phase program

// Phase number idx of the program: 0 is the embedding; then per layer the
// final norm (first decision layer only), QKV, attention, out, up, down.
__device__ __forceinline__ Phase phase_at(const FusedArgs& a, int idx) {
  Phase p{kPhEmbed, 0, idx, -1};
  if (idx == 0) return p;
  int r = idx - 1;
  const bool fn = a.final_gamma != nullptr && a.L > a.n_enc;
  const int before = 5 * a.n_enc;  // phases of the encoder layers
  if (fn && r >= before) {
    if (r == before) {
      p.kind = kPhFinal;
      p.layer = a.n_enc;
      return p;
    }
    r -= 1;
  }
  p.layer = r / 5;
  const int k = r % 5;
  p.kind = k == 0 ? kPhQkv : k == 1 ? kPhAttn : k == 2 ? kPhOut : k == 3 ? kPhUp : kPhDown;
  p.gemm = k == 0 ? 0 : k == 1 ? -1 : k - 1;
  return p;
}

// Calls f(Phase) for every phase in order (one call site, so that the body
// is compiled once); stops early when f returns false.
template <class F>
__device__ __forceinline__ void walk(const FusedArgs& a, F&& f) {
  const int n = 1 + 5 * a.L + ((a.final_gamma != nullptr && a.L > a.n_enc) ? 1 : 0);
#pragma unroll 1
  for (int idx = 0; idx < n; ++idx)
    if (!f(phase_at(a, idx))) return;
}

__device__ __forceinline__ int gemm_na(int gemm) { return gemm == 2 ? 2 : 1; }

// The tile of projection `gemm` this CTA's cluster computes (-1: none) and
// this CTA's k-block range of it (its rank's quarter of K).
__device__ __forceinline__ int cluster_tile(const FusedArgs& a, int gemm, int& k0, int& k1) {
  const int t = a.cluster_tile[gemm][blockIdx.x / kCluster];
  const int r = static_cast<int>(blockIdx.x % kCluster);
  const int kb = a.plan[gemm].kb;
  k0 = r * kb / kCluster;
  k1 = (r + 1) * kb / kCluster;
  return t == 255 ? -1 : t;
}

__device__ __forceinline__ bool layer_global(const FusedArgs& a, int l) {
  return l >= a.n_enc || (l % a.global_every) == 0;
}

// ------------------------------------------------------------ row phases

// One warp, one row of H = 32 * VPL values; lane holds [lane * VPL, +VPL).
// Normalises x with gamma, stores BF16 to y and the per-128-feature slice
// statistics (mean, sum of squared deviations) of the stored values.
__device__ void ln_row_store(const FusedArgs& a, const bf16* src, bool src_cg, const bf16* gamma,
                             int t, bf16* y, int lane) {
  const int vpl = a.H / 32;  // 8, 16 or 32
  const int nc = vpl / 8;
  float v[32];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < nc) {
      const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<size_t>(lane) * vpl) + c;
      const uint4 u = src_cg ? __ldcg(p) : __ldg(p);
      bf16x8_to_f32(u, v + 8 * c);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < vpl) s += v[i];
  const float mean = warp_allsum(s) / static_cast<float>(a.H);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < vpl) {
      const float d = v[i] - mean;
      q += d * d;
    }
  const float var = warp_allsum(q) / static_cast<float>(a.H);
  const float rstd = 1.0f / sqrtf(var + a.eps);
  // normalised BF16 values: stored, and summed for the slice statistics
  // (all of a lane's values lie in one 128-feature slice); the second pass
  // recomputes the same rounded values instead of keeping them
  const uint4* gp = reinterpret_cast<const uint4*>(gamma + lane * vpl);
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < nc) {
      float gm[8];
      bf16x8_to_f32(__ldg(gp + c), gm);
      uint4 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o2[e] = __floats2bfloat162_rn(ln_apply(v[8 * c + 2 * e], mean, rstd, gm[2 * e]),
                                      ln_apply(v[8 * c + 2 * e + 1], mean, rstd, gm[2 * e + 1]));
        const float2 back = __bfloat1622float2(o2[e]);
        ss += back.x + back.y;
      }
      reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * a.H + lane * vpl)[c] = o;
    }
  }
  // slice statistics: the 128 / vpl lanes of a slice are consecutive
  const int lps = 128 / vpl;
  for (int o = lps >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float ms = ss / 128.f;
  float qs = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (c < nc) {
      float gm[8];
      bf16x8_to_f32(__ldg(gp + c), gm);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float rv = __bfloat162float(__float2bfloat16_rn(ln_apply(v[8 * c + i], mean, rstd, gm[i])));
        const float d = rv - ms;
        qs += d * d;
      }
    }
  }
  for (int o = lps >> 1; o > 0; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
  if ((lane % lps) == 0) {
    const int slice = lane / lps;
    float2* st = reinterpret_cast<float2*>(a.stats) + static_cast<size_t>(t) * (a.H / 128) + slice;
    *st = make_float2(ms, qs);
  }
}

// ------------------------------------------------------------- attention

// One warp: queries [q0, q0 + 16) of row b, head n, against the K and V
// tiles staged in shared memory (swizzled [key][64 dims], sk keys, zero
// beyond S).  S <= 128: every score fits in registers, one softmax pass.
__device__ void attn_warp(const FusedArgs& a, uint32_t sQ, uint32_t sK, uint32_t sV, int b, int n,
                          int q0, int len, bool global, int lane) {
  const int S = a.S, H = a.H;
  const int g = lane >> 2, tig = lane & 3;
  const int i0 = q0 + g, i1 = q0 + g + 8;
  // Q fragments from the swizzled tile: matrix (lane / 8) of an x4 load is
  // (rows q0 + 8 ((lane / 8) & 1) + lane % 8, dims 16 kk + 8 (lane / 16))
  uint32_t qa[4][4];
  {
    const int qr = q0 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int chunk = 2 * kk + (lane >> 4);
      ldmatrix_x4(sQ + qr * 128 + ((chunk ^ (qr & 7)) << 4), qa[kk][0], qa[kk][1], qa[kk][2],
                  qa[kk][3]);
    }
  }
  // keys in halves of 64 with an online softmax (running maximum and sum per
  // query row; the accumulator is rescaled when the maximum grows)
  const float scale = 0.125f * 1.4426950408889634f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[8][4];
#pragma unroll
  for (int d = 0; d < 8; ++d) acc[d][0] = acc[d][1] = acc[d][2] = acc[d][3] = 0.f;
#pragma unroll 1
  for (int kh = 0; kh * 64 < S; ++kh) {
    float sc[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
      sc[jt][0] = sc[jt][1] = sc[jt][2] = sc[jt][3] = 0.f;
      const int key = kh * 64 + 8 * jt + g;
      if (kh * 64 + 8 * jt < S) {
        const uint32_t row = sK + key * 128;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t b0 = lds32(row + (((2 * kk) ^ (key & 7)) << 4) + tig * 4);
          const uint32_t b1 = lds32(row + (((2 * kk + 1) ^ (key & 7)) << 4) + tig * 4);
          mma16816(sc[jt], qa[kk], b0, b1);
        }
      }
    }
    float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kh * 64 + 8 * jt + tig * 2 + (e & 1);
        const int qi = e < 2 ? i0 : i1;
        const int dist = qi > key ? qi - key : key - qi;
        const bool vis = key < len && (global || dist <= a.half_window);
        sc[jt][e] = vis ? sc[jt][e] * scale : -INFINITY;
      }
      t0 = fmaxf(t0, fmaxf(sc[jt][0], sc[jt][1]));
      t1 = fmaxf(t1, fmaxf(sc[jt][2], sc[jt][3]));
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o));
    }
    const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
    const float al0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
    const float al1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = e < 2 ? m0 : m1;
        const float pv = sc[jt][e] == -INFINITY ? 0.f : exp2f(sc[jt][e] - m);
        sc[jt][e] = pv;
        if (e < 2) s0 += pv; else s1 += pv;
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    l0 = l0 * al0 + s0;
    l1 = l1 * al1 + s1;
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      acc[d][0] *= al0;
      acc[d][1] *= al0;
      acc[d][2] *= al1;
      acc[d][3] *= al1;
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (kh * 64 + 16 * ks < S) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * ks][0], sc[2 * ks][1]);
        pa[1] = pack_bf16(sc[2 * ks][2], sc[2 * ks][3]);
        pa[2] = pack_bf16(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
        pa[3] = pack_bf16(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
        // matrix (lane / 8): keys 16 ks + 8 ((lane / 8) & 1) + lane % 8, dims 8 (dt + lane / 16)
        const int key = kh * 64 + 16 * ks + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int dt = 0; dt < 8; dt += 2) {
          const int chunk = dt + (lane >> 4);
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(sV + key * 128 + ((chunk ^ (key & 7)) << 4), r0, r1, r2, r3);
          mma16816(acc[dt], pa, r0, r1);
          mma16816(acc[dt + 1], pa, r2, r3);
        }
      }
    }
  }
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  bf16* out0 = a.ctx + (static_cast<size_t>(b) * S + i0) * H + n * 64 + tig * 2;
  bf16* out1 = a.ctx + (static_cast<size_t>(b) * S + i1) * H + n * 64 + tig * 2;
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    if (i0 < S)
      *reinterpret_cast<uint32_t*>(out0 + 8 * d) = pack_bf16(acc[d][0] * inv0, acc[d][1] * inv0);
    if (i1 < S)
      *reinterpret_cast<uint32_t*>(out1 + 8 * d) = pack_bf16(acc[d][2] * inv1, acc[d][3] * inv1);
  }
}

// ------------------------------------------------------- split-K reduce

// Sum over the cluster's CTAs, in rank order, of the 8 fp32 values at byte
// offset `off` of each CTA's staged partial (stg[r]: shared::cluster address
// of rank r's staging).  Every load is issued before the first add.
__device__ __forceinline__ void cluster_sum8(const uint32_t (&stg)[kCluster], uint32_t off,
                                             float (&v)[8]) {
  float t[kCluster][8];
#pragma unroll
  for (int r = 0; r < kCluster; ++r) ptx::ld_dsmem_f32x8(stg[r] + off, t[r]);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = t[0][i];
#pragma unroll
  for (int r = 1; r < kCluster; ++r)
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] += t[r][i];
}

// Epilogue of tokens [c0, c0 + n) of tile f of the projection of phase ph.
// The cluster's partials of the chunk of columns starting at token cb0 are
// staged token-major, [half][token - cb0][128] fp32 with wch tokens per
// half, in every CTA of the cluster (stg).  128 epilogue threads (etid);
// loops run a warp-uniform number of times.  xpre: the residual of this
// thread's first unit, already loaded (or null).
__device__ void epilogue_chunk(const FusedArgs& a, const Phase& ph, int f, int c0, int n, int cb0,
                               int wch, const uint32_t (&stg)[kCluster], int etid,
                               const uint4* xpre) {
  const int H = a.H;
  if (ph.kind == kPhQkv && f * kFBM < 2 * H) {
    // q and k: unit = token c, pair group pg (features fo..fo+7 and
    // fo+32..fo+39 of one head), rotated after the BF16 rounding
    const bool glob = layer_global(a, ph.layer);
    const float* cos_t = a.rope + (glob ? 0 : 2) * static_cast<size_t>(a.max_seq) * 32;
    const float* sin_t = cos_t + static_cast<size_t>(a.max_seq) * 32;
    for (int u = etid; u < n * 8; u += 128) {
      const int c = c0 + u / 8, pg = u % 8;
      const int fo = 64 * (pg >> 2) + 8 * (pg & 3);
      const int pos = c % a.S;
      const int i0 = fo & 31;
      const float4* ct = reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(pos) * 32 + i0);
      const float4* st = reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(pos) * 32 + i0);
      const float4 ca = __ldg(ct), cb = __ldg(ct + 1), sa = __ldg(st), sb = __ldg(st + 1);
      const uint32_t off = static_cast<uint32_t>((c - cb0) * kFBM + fo) * 4u;
      float v1[8], v2[8];
      cluster_sum8(stg, off, v1);
      cluster_sum8(stg, off + 32u * 4u, v2);
      const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
      const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
      uint4 o1, o2;
      __nv_bfloat16* p1 = reinterpret_cast<__nv_bfloat16*>(&o1);
      __nv_bfloat16* p2 = reinterpret_cast<__nv_bfloat16*>(&o2);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x1 = __bfloat162float(__float2bfloat16_rn(v1[i]));
        const float x2 = __bfloat162float(__float2bfloat16_rn(v2[i]));
        p1[i] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(x1, cv[i]), __fmul_rn(x2, sv[i])));
        p2[i] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(x2, cv[i]), __fmul_rn(x1, sv[i])));
      }
      bf16* row = a.qkv + static_cast<size_t>(c) * (3 * H) + f * kFBM;
      *reinterpret_cast<uint4*>(row + fo) = o1;
      *reinterpret_cast<uint4*>(row + fo + 32) = o2;
    }
    return;
  }
  if (ph.kind == kPhQkv || ph.kind == kPhUp) {
    // v of the QKV projection (plain), or the GeGLU product; unit = token c,
    // group grp of 8 features
    const bool up = ph.kind == kPhUp;
    const int N = up ? a.I : 3 * H;
    bf16* y = up ? a.g : a.qkv;
    for (int u = etid; u < n * 16; u += 128) {
      const int c = c0 + u / 16, grp = u % 16;
      const int fe = f * kFBM + grp * 8;
      if (fe >= N) continue;
      const uint32_t off = static_cast<uint32_t>((c - cb0) * kFBM + grp * 8) * 4u;
      float v[8];
      cluster_sum8(stg, off, v);
      uint4 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
      if (up) {
        float gt[8];
        cluster_sum8(stg, off + static_cast<uint32_t>(wch) * kFBM * 4u, gt);  // gate half
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o2[e] = __floats2bfloat162_rn(gelu_erf(v[2 * e]) * gt[2 * e],
                                        gelu_erf(v[2 * e + 1]) * gt[2 * e + 1]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      }
      *reinterpret_cast<uint4*>(y + static_cast<size_t>(c) * N + fe) = o;
    }
    return;
  }
  // residual epilogues (out-projection, down-projection): y = bf16(x + acc),
  // then the slice statistics of token c over this tile's 128 features; the
  // 16 units of a token are 16 consecutive lanes (128 is a multiple of 16)
  const bool last = ph.kind == kPhDown && ph.layer == a.L - 1;
  bf16* y = last ? a.out : a.x;
  const int total = n * 16;
  for (int b0 = 0; b0 < total; b0 += 128) {
    const int u = b0 + etid;
    const bool valid = u < total;
    const int c = c0 + (valid ? u / 16 : 0), grp = u % 16;
    const size_t goff = static_cast<size_t>(c) * H + f * kFBM + grp * 8;
    float r[8];
    if (valid) {
      // the first pass's residual was loaded by the caller (xpre)
      const uint4 xres = (xpre != nullptr && b0 == 0) ? *xpre : ldcg16(a.x + goff);
      float v[8], xr[8];
      cluster_sum8(stg, static_cast<uint32_t>((c - cb0) * kFBM + grp * 8) * 4u, v);
      bf16x8_to_f32(xres, xr);
      uint4 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o2[e] = __floats2bfloat162_rn(xr[2 * e] + v[2 * e], xr[2 * e + 1] + v[2 * e + 1]);
        const float2 back = __bfloat1622float2(o2[e]);
        r[2 * e] = back.x;
        r[2 * e + 1] = back.y;
      }
      *reinterpret_cast<uint4*>(y + goff) = o;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = 0.f;
    }
    if (last) continue;
    float sm = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) sm += r[i];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    const float ms = sm / 128.f;
    float q = 0.f;
    if (valid)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float d = r[i] - ms;
        q += d * d;
      }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    if (valid && grp == 0)
      reinterpret_cast<float2*>(a.stats)[static_cast<size_t>(c) * (H / 128) + f] =
          make_float2(ms, q);
  }
}

// ------------------------------------------------------------------ roles

__device__ void role_weights(const FusedArgs& a, const Ctl& c, uint32_t sbase) {
  const uint64_t pol = ptx::policy_evict_first();
  uint32_t wi = 0;
  walk(a, [&](const Phase& ph) -> bool {
    if (ph.gemm < 0) return true;
    int k0, k1;
    const int f = cluster_tile(a, ph.gemm, k0, k1);
    if (f < 0) return true;
    const FusedLayer& lw = a.layers[ph.layer];
    const CUtensorMap* m0 = &lw.maps[ph.gemm == 0 ? kMapQkv : ph.gemm == 1 ? kMapOut
                                     : ph.gemm == 2 ? kMapUpIn : kMapDown];
    const CUtensorMap* m1 = &lw.maps[kMapUpGate];
    const int na = gemm_na(ph.gemm);
    for (int kb = k0; kb < k1; ++kb) {
      for (int h = 0; h < na; ++h) {
        const uint32_t slot = wi % kWSlots;
        const uint32_t par = (wi / kWSlots) & 1u;
        if (!fwait(a, c, c.wempty + 8u * slot, par ^ 1u, kFErrWeight)) return false;
        ptx::mbar_arrive_expect_tx(c.wfull + 8u * slot, kWSlotBytes);
        ptx::tma_load_2d(sbase + kOffW + slot * kWSlotBytes, h == 0 ? m0 : m1,
                         c.wfull + 8u * slot, kb * kFBK, f * kFBM, pol);
        ++wi;
      }
    }
    return true;
  });
  // no copy may still be in flight into shared memory at exit (bounded, and
  // not cut short by an abort: the copies land whatever the other roles do)
  const uint32_t first = wi > static_cast<uint32_t>(kWSlots) ? wi - kWSlots : 0u;
  for (uint32_t i = first; i < wi; ++i) {
    const uint32_t slot = i % kWSlots;
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(c.wfull + 8u * slot, (i / kWSlots) & 1u))
      if (clock64() - t0 > kWaitLimitCycles) break;
  }
}

__device__ void role_mma(const FusedArgs& a, const Ctl& c, uint32_t sbase, uint32_t tmem) {
  uint32_t wi = 0, ai = 0, ui = 0;
  const uint32_t idesc = ptx::idesc_bf16(kFBM, a.nt);
  const uint64_t dA0 = ptx::sdesc_sw128(sbase + kOffA), dW0 = ptx::sdesc_sw128(sbase + kOffW);
  walk(a, [&](const Phase& ph) -> bool {
    if (ph.gemm < 0) return true;
    int k0, k1;
    if (cluster_tile(a, ph.gemm, k0, k1) < 0) return true;
    const int na = gemm_na(ph.gemm);
    const uint32_t buf = ui & 1u;
    if (!fwait(a, c, c.accempty + 8u * buf, ((ui >> 1) & 1u) ^ 1u, kFErrMma)) return false;
    ptx::tc_fence_after();
    const uint32_t d = tmem + buf * 256u;
    for (int kb = k0; kb < k1; ++kb) {
      const uint32_t as = ai % kASlotsMax;
      if (!fwait(a, c, c.afull + 8u * as, (ai / kASlotsMax) & 1u, kFErrMma)) return false;
      for (int h = 0; h < na; ++h)
        if (!fwait(a, c, c.wfull + 8u * ((wi + h) % kWSlots), ((wi + h) / kWSlots) & 1u, kFErrMma))
          return false;
      ptx::tc_fence_after();
      // descriptors: the start-address field advances by 16-byte units
      const uint64_t da = dA0 + static_cast<uint64_t>(as) * (kASlotBytes >> 4);
      const uint64_t dw0 = dW0 + static_cast<uint64_t>(wi % kWSlots) * (kWSlotBytes >> 4);
      const uint64_t dw1 = dW0 + static_cast<uint64_t>((wi + 1) % kWSlots) * (kWSlotBytes >> 4);
#pragma unroll
      for (int kk = 0; kk < kFBK / 16; ++kk) {
        const uint32_t acc = (kb > k0 || kk > 0) ? 1u : 0u;
        ptx::mma_bf16(d, dw0 + 2 * kk, da + 2 * kk, idesc, acc);
        if (na == 2) ptx::mma_bf16(d + 128u, dw1 + 2 * kk, da + 2 * kk, idesc, acc);
      }
      // the slots are free once these MMAs have read them
      for (int h = 0; h < na; ++h) ptx::mma_commit(c.wempty + 8u * ((wi + h) % kWSlots));
      ptx::mma_commit(c.aempty + 8u * as);
      wi += na;
      ++ai;
    }
    ptx::mma_commit(c.accfull + 8u * buf);
    ++ui;
    return true;
  });
}

__device__ void role_loader(const FusedArgs& a, const Ctl& c, uint32_t sbase, uint8_t* smem,
                            uint32_t gen) {
  const int ltid = threadIdx.x - 192;  // 0..63
  float2* lnst = reinterpret_cast<float2*>(smem + kOffLn);
  volatile int* phase_ok = reinterpret_cast<volatile int*>(c.tmem_slot + 3);
  const uint64_t pol = ptx::policy_evict_last();
  uint32_t ai = 0;
  const int nt = a.nt, M = a.M;
  const uint32_t tile_bytes = static_cast<uint32_t>(nt) * kFBK * 2;
  walk(a, [&](const Phase& ph) -> bool {
    if (ph.gemm < 0) return true;
    int k0, k1;
    if (cluster_tile(a, ph.gemm, k0, k1) < 0) return true;  // no unit of this phase here
    const FusedLayer& lw = a.layers[ph.layer];
    const bf16* gamma = ph.kind == kPhQkv ? lw.attn_norm : ph.kind == kPhUp ? lw.mlp_norm : nullptr;
    // gamma chunk j = ltid % 8 of the first k-blocks, requested before the
    // wait below (the vectors are not kept in L2 from one forward to the next)
    const int j = ltid & 7;
    uint4 gpre[kGammaPre];
    if (gamma != nullptr) {
#pragma unroll
      for (int i = 0; i < kGammaPre; ++i)
        if (k0 + i < k1)
          gpre[i] = __ldg(reinterpret_cast<const uint4*>(gamma + (k0 + i) * kFBK + j * 8));
    }
    // inputs of this phase: every CTA done with the previous phase
    if (ltid == 0) {
      const bool ok = wait_count(a, c, a.ready + (ph.idx - 1), gen * gridDim.x, kFErrPhase);
      ptx::fence_proxy_async_global();
      *phase_ok = ok ? 1 : 0;
    }
    ptx::named_barrier_sync(2, 64);
    if (!*phase_ok) return false;
    // activations: x (normalised here unless attn_norm is null: identity), ctx, g
    const CUtensorMap* tm = ph.kind == kPhOut ? &a.tm_ctx : ph.kind == kPhDown ? &a.tm_g : &a.tm_x;
    {
      // every k-block's raw tile requested at once (as ring slots allow)
      if (ltid == 0) {
        uint32_t ti = ai;
        for (int kb = k0; kb < k1 && kb - k0 < kASlotsMax; ++kb, ++ti) {
          const uint32_t as = ti % kASlotsMax;
          if (!fwait(a, c, c.aempty + 8u * as, ((ti / kASlotsMax) & 1u) ^ 1u, kFErrAct)) break;
          ptx::mbar_arrive_expect_tx(c.aload + 8u * as, tile_bytes);
          ptx::tma_load_2d(sbase + kOffA + as * kASlotBytes, tm, c.aload + 8u * as, kb * kFBK, 0,
                           pol);
        }
      }
      if (gamma != nullptr) {
        // mean and rstd of every token from the slice statistics
        const int T8 = a.H / 128;
        for (int t = ltid; t < M; t += 64) {
          const float2* st = reinterpret_cast<const float2*>(a.stats) + static_cast<size_t>(t) * T8;
          float2 sl[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) sl[i] = i < T8 ? __ldcg(st + i) : make_float2(0.f, 0.f);
          float msum = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) msum += sl[i].x;
          const float mean = msum / static_cast<float>(T8);
          float m2 = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < T8) {
              const float d = sl[i].x - mean;
              m2 += sl[i].y + 128.f * d * d;
            }
          const float var = m2 / static_cast<float>(a.H);
          lnst[t] = make_float2(mean, 1.0f / sqrtf(var + a.eps));
        }
        ptx::named_barrier_sync(2, 64);
      }
      for (int kb = k0; kb < k1; ++kb, ++ai) {
        const uint32_t as = ai % kASlotsMax;
        if (ltid == 0 && kb - k0 >= kASlotsMax) {
          // beyond the ring: request this tile once its slot is free
          if (!fwait(a, c, c.aempty + 8u * as, ((ai / kASlotsMax) & 1u) ^ 1u, kFErrAct)) return false;
          ptx::mbar_arrive_expect_tx(c.aload + 8u * as, tile_bytes);
          ptx::tma_load_2d(sbase + kOffA + as * kASlotBytes, tm, c.aload + 8u * as, kb * kFBK, 0,
                           pol);
        }
        if (!fwait(a, c, c.aload + 8u * as, (ai / kASlotsMax) & 1u, kFErrAct)) return false;
        if (gamma != nullptr) {
          // LayerNorm in place: thread ltid takes 16-byte chunk j = ltid % 8 of
          // token rows ltid / 8 + 8 i (row r's chunk j sits at j ^ (r % 8))
          const uint32_t slot = sbase + kOffA + as * kASlotBytes;
          float gm[8];
          uint4 graw;
#pragma unroll
          for (int i = 0; i < kGammaPre; ++i)
            if (kb - k0 == i) graw = gpre[i];
          if (kb - k0 >= kGammaPre)
            graw = __ldg(reinterpret_cast<const uint4*>(gamma + kb * kFBK + j * 8));
          bf16x8_to_f32(graw, gm);
          for (int r = ltid >> 3; r < M; r += 8) {
            const uint32_t addr = slot + r * 128 + ((j ^ (r & 7)) << 4);
            uint4 v = lds128(addr);
            float xv[8];
            bf16x8_to_f32(v, xv);
            const float2 mr = lnst[r];
            __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              o2[q] = __floats2bfloat162_rn(ln_apply(xv[2 * q], mr.x, mr.y, gm[2 * q]),
                                            ln_apply(xv[2 * q + 1], mr.x, mr.y, gm[2 * q + 1]));
            sts128(addr, v);
          }
          ptx::fence_proxy_async_smem();
        }
        ptx::mbar_arrive(c.afull + 8u * as);
      }
    }
    return true;
  });
}

__device__ void role_epilogue(const FusedArgs& a, const Ctl& c, uint32_t sbase, uint32_t tmem,
                              uint32_t gen) {
  const int etid = threadIdx.x - 64;  // 0..127
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;             // TMEM lanes 32 q .. 32 q + 31
  const int row = q * 32 + lane;      // feature row of the accumulator
  volatile int* flag = reinterpret_cast<volatile int*>(c.tmem_slot + 2);
  const uint32_t G = gridDim.x;
  const uint32_t target = gen * G;
  uint32_t ui = 0, kvi = 0, stg_uses = 0;
  const uint64_t kv_pol = ptx::policy_evict_last();
  // every epilogue thread takes a decision thread 0 made
  auto agree = [&](bool v) -> bool {
    if (etid == 0) *flag = v ? 1 : 0;
    ptx::named_barrier_sync(1, 128);
    const bool r = *flag != 0;
    ptx::named_barrier_sync(1, 128);
    return r;
  };
  auto signal = [&](int idx) {
    ptx::named_barrier_sync(1, 128);
    if (etid == 0) red_release_add(a.ready + idx, 1u);
  };
  const int gw = blockIdx.x * 4 + (warp - 2);  // global epilogue warp
  walk(a, [&](const Phase& ph) -> bool {
    // every phase but the first starts by acquiring the previous phase's
    // completion: the outputs of every earlier phase are then visible here,
    // and every read of them by any CTA is finished
    if (ph.kind != kPhEmbed &&
        !agree(etid != 0 || wait_count(a, c, a.ready + (ph.idx - 1), target, kFErrPhase)))
      return false;
    if (ph.kind == kPhEmbed || ph.kind == kPhFinal) {
      for (int t = gw; t < a.M; t += 4 * G) {
        if (ph.kind == kPhEmbed) {
          int id = a.ids[t];
          if (id < 0 || id >= a.vocab) {
            if (lane == 0 && a.err) atomicCAS(a.err, 0, kDevBadId);
            id = id < 0 ? 0 : a.vocab - 1;
          }
          ln_row_store(a, a.emb + static_cast<size_t>(id) * a.H, false, a.emb_gamma, t, a.x, lane);
        } else {
          ln_row_store(a, a.x + static_cast<size_t>(t) * a.H, true, a.final_gamma, t, a.x, lane);
        }
      }
      signal(ph.idx);
      return true;
    }
    if (ph.kind == kPhAttn) {
      const bool glob = layer_global(a, ph.layer);
      // Q, K, V tiles of one (row, head): the first activation slot (idle in
      // this phase) and the attention area
      const uint32_t sQ = sbase + kOffA, sK = sbase + kOffAttn, sV = sK + 16384u;
      const int S = a.S, H = a.H;
      if (etid == 0) ptx::fence_proxy_async_global();  // qkv was written by other CTAs
      for (int u = blockIdx.x; u < a.B * a.heads; u += G) {
        const int b = u / a.heads, n = u % a.heads;
        int len = a.lens[b];
        if (len < 1 || len > S) {
          if (etid == 0 && a.err) atomicCAS(a.err, 0, kDevBadLength);
          len = len < 1 ? 1 : S;
        }
        // K and V of (b, n): 128 key rows each by TMA, landing in the 128-byte
        // swizzled layout (rows past S are other tokens or zero; masked)
        if (etid == 0) {
          ptx::mbar_arrive_expect_tx(c.kvbar, 3u * 128u * 128u);
          ptx::tma_load_2d(sQ, &a.tm_qkv, c.kvbar, n * 64, b * S, kv_pol);
          ptx::tma_load_2d(sK, &a.tm_qkv, c.kvbar, H + n * 64, b * S, kv_pol);
          ptx::tma_load_2d(sV, &a.tm_qkv, c.kvbar, 2 * H + n * 64, b * S, kv_pol);
        }
        if (!agree(fwait(a, c, c.kvbar, kvi & 1u, kFErrPhase))) return false;
        ++kvi;
        ptx::named_barrier_sync(1, 128);
        for (int qb = warp - 2; qb * 16 < S; qb += 4)
          attn_warp(a, sQ, sK, sV, b, n, qb * 16, len, glob, lane);
        ptx::named_barrier_sync(1, 128);  // K/V read before the next unit overwrites them
      }
      signal(ph.idx);
      return true;
    }
    // ---- GEMM phase: this CTA's quarter of K of its cluster's tile (if any)
    int k0, k1;
    const int f = cluster_tile(a, ph.gemm, k0, k1);
    bool ok = true;
    if (f >= 0) {
      const int na = gemm_na(ph.gemm);
      const int rank = static_cast<int>(blockIdx.x % kCluster);
      const uint32_t buf = ui & 1u;
      const bool resid = ph.kind == kPhOut || ph.kind == kPhDown;
      // token columns in chunks whose partial (both halves) fits the staging
      const int cw = static_cast<int>(kRedBytes / (static_cast<uint32_t>(na) * kFBM * 4)) & ~15;
      // the residual of this thread's first unit of the first chunk, loaded
      // while the MMAs run
      uint4 xpre = make_uint4(0, 0, 0, 0);
      {
        const int wch = a.M < cw ? a.M : cw;
        const int c0 = rank * wch / kCluster, c1 = (rank + 1) * wch / kCluster;
        if (resid && etid < (c1 - c0) * 16)
          xpre = ldcg16(a.x + static_cast<size_t>(c0 + etid / 16) * a.H + f * kFBM + (etid % 16) * 8);
      }
      ok = agree(fwait(a, c, c.accfull + 8u * buf, (ui >> 1) & 1u, kFErrDrain));
      if (!ok) return false;
      ptx::tc_fence_after();
      const uint32_t tq = tmem + buf * 256u + (static_cast<uint32_t>(q * 32) << 16);
      uint32_t stg[kCluster];
#pragma unroll
      for (int r = 0; r < kCluster; ++r) stg[r] = ptx::mapa(sbase + kOffRed, r);
      for (int cb0 = 0; cb0 < a.M && ok; cb0 += cw) {
        const int ce = a.M - cb0 < cw ? a.M : cb0 + cw;  // columns [cb0, ce)
        const int wch = ce - cb0;
        const int c0 = cb0 + rank * wch / kCluster, c1 = cb0 + (rank + 1) * wch / kCluster;
        // the staging is free once every peer has read the previous partial
        if (stg_uses > 0)
          ok = agree(fwait_cluster(a, c, c.red_done, (stg_uses - 1) & 1u, kFErrTile));
        if (!ok) break;
        for (int h = 0; h < na; ++h) {
          for (int cb = cb0; cb < ce; cb += 16) {
            float v[16];
            ptx::tmem_ld16(tq + h * 128u + cb, v);
            const uint32_t srow = sbase + kOffRed + ((h * wch + (cb - cb0)) * kFBM + row) * 4u;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (cb + j < ce) sts32f(srow + j * kFBM * 4u, v[j]);
          }
        }
        ptx::named_barrier_sync(1, 128);
        if (etid == 0)
          for (int r = 0; r < kCluster; ++r) mbar_arrive_cluster(ptx::mapa(c.red_ready, r));
        ok = agree(fwait_cluster(a, c, c.red_ready, stg_uses & 1u, kFErrTile));
        if (!ok) break;
        epilogue_chunk(a, ph, f, c0, c1 - c0, cb0, wch, stg, etid, cb0 == 0 ? &xpre : nullptr);
        ptx::named_barrier_sync(1, 128);
        if (etid == 0)
          for (int r = 0; r < kCluster; ++r) mbar_arrive_cluster(ptx::mapa(c.red_done, r));
        ++stg_uses;
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.accempty + 8u * buf);
      ++ui;
    }
    if (!ok) return false;
    signal(ph.idx);
    return true;
  });
}

__global__ void __launch_bounds__(kFThreads, 1)
    fused_forward_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffCtrl);
  Ctl c;
  c.wfull = ptx::smem_u32(bars);
  c.wempty = c.wfull + 8u * kWSlots;
  c.afull = c.wempty + 8u * kWSlots;
  c.aempty = c.afull + 8u * kASlotsMax;
  c.accfull = c.aempty + 8u * kASlotsMax;
  c.accempty = c.accfull + 16u;
  c.mma_done = c.accempty + 16u;
  c.aload = c.mma_done + 8u;
  c.kvbar = c.aload + 8u * kASlotsMax;
  c.red_ready = c.kvbar + 8u;
  c.red_done = c.red_ready + 8u;
  c.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kWSlots + 3 * kASlotsMax + 8);

  c.cta_abort = reinterpret_cast<volatile int*>(c.tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWSlots; ++i) {
      ptx::mbar_init(c.wfull + 8u * i, 1);
      ptx::mbar_init(c.wempty + 8u * i, 1);
    }
    for (int i = 0; i < kASlotsMax; ++i) {
      ptx::mbar_init(c.afull + 8u * i, 64);
      ptx::mbar_init(c.aempty + 8u * i, 1);
      ptx::mbar_init(c.aload + 8u * i, 1);
    }
    ptx::mbar_init(c.kvbar, 1);
    ptx::mbar_init(c.red_ready, kCluster);  // one arrival from each CTA of the cluster
    ptx::mbar_init(c.red_done, kCluster);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(c.accfull + 8u * i, 1);
      ptx::mbar_init(c.accempty + 8u * i, 128);
    }
    ptx::mbar_init(c.mma_done, 1);
    *c.cta_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(c.tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  // generation of this launch: one more than the last completed launch's
  const uint32_t gen = ld_volatile_u32(a.sync) + 1u;
  ptx::tc_fence_before();
  __syncthreads();
  cluster_arrive_wait();  // peers' barriers are initialised before any remote arrival
  ptx::tc_fence_after();
  const uint32_t tmem = *c.tmem_slot;

  if (warp == 0) {
    if (lane == 0) role_weights(a, c, sbase);
  } else if (warp == 1) {
    if (lane == 0) {
      role_mma(a, c, sbase, tmem);
      // every MMA this thread issued is complete before TMEM is freed
      ptx::mma_commit(c.mma_done);
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(c.mma_done, 0))
        if (clock64() - t0 > kWaitLimitCycles) break;
    }
  } else if (warp < 6) {
    role_epilogue(a, c, sbase, tmem, gen);
    if (threadIdx.x == 64) {
      // finished: CTA 0 advances the generation once every CTA is
      red_release_add(a.sync + 1, 1u);
      if (blockIdx.x == 0 && *c.cta_abort == 0 &&
          wait_count(a, c, a.sync + 1, gen * gridDim.x, kFErrPhase)) {
        __threadfence();
        atomicExch(a.sync, gen);
      }
    }
  } else {
    role_loader(a, c, sbase, smem, gen);
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_arrive_wait();  // no peer reads this CTA's shared memory any more
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool plan_fused(int M, int H, int I, int heads, int n_clusters, FusedPlanOut* out) {
  if (M < 1 || M > 128 || n_clusters < 1 || n_clusters > kFusedMaxClusters) return false;
  if (!(H == 256 || H == 512 || H == 1024) || heads * 64 != H) return false;
  if (I < 64 || I % 64 != 0) return false;
  FusedPlanOut o{};
  o.nt = (M + 15) & ~15;
  o.n_clusters = n_clusters;
  const int tiles[4] = {3 * H / kFBM, H / kFBM, (I + kFBM - 1) / kFBM, H / kFBM};
  const int kbs[4] = {H / kFBK, H / kFBK, H / kFBK, I / kFBK};
  const int na[4] = {1, 1, 2, 1};
  for (int i = 0; i < 4; ++i) {
    // every tile on its own cluster; every CTA of a cluster with k-blocks
    if (tiles[i] > n_clusters || tiles[i] > 255 || kbs[i] < kCluster) return false;
    o.plan[i].tiles = tiles[i];
    o.plan[i].kb = kbs[i];
  }
  std::memset(o.cluster_tile, 255, sizeof(o.cluster_tile));
  // Placement for weight prefetch: a cluster's producer streams the weights
  // of its next tile while earlier phases run, so no cluster should hold
  // tiles of two consecutive projections.  The down- and out-projections
  // share clusters [0, a0) (out, up, down: separated by up), the up-projection
  // takes the next clusters and QKV the last ones (up, down, QKV: separated
  // by down), when that fits.
  const int a0 = std::max(tiles[3], tiles[1]);
  if (a0 + tiles[2] <= n_clusters && tiles[0] <= n_clusters - a0) {
    for (int t = 0; t < tiles[3]; ++t) o.cluster_tile[3][t] = static_cast<uint8_t>(t);
    for (int t = 0; t < tiles[1]; ++t) o.cluster_tile[1][t] = static_cast<uint8_t>(t);
    for (int t = 0; t < tiles[2]; ++t) o.cluster_tile[2][a0 + t] = static_cast<uint8_t>(t);
    for (int t = 0; t < tiles[0]; ++t)
      o.cluster_tile[0][n_clusters - tiles[0] + t] = static_cast<uint8_t>(t);
    *out = o;
    return true;
  }
  // otherwise: heaviest projection first, each tile to the cluster with the
  // fewest weight bytes so far that has no tile of that projection
  int order[4] = {0, 1, 2, 3};
  std::stable_sort(order, order + 4,
                   [&](int x, int y) { return kbs[x] * na[x] > kbs[y] * na[y]; });
  long long load[kFusedMaxClusters] = {};
  for (int oi = 0; oi < 4; ++oi) {
    const int g = order[oi];
    for (int t = 0; t < tiles[g]; ++t) {
      int best = -1;
      for (int cl = 0; cl < n_clusters; ++cl)
        if (o.cluster_tile[g][cl] == 255 && (best < 0 || load[cl] < load[best])) best = cl;
      o.cluster_tile[g][best] = static_cast<uint8_t>(t);
      load[best] += static_cast<long long>(kbs[g]) * na[g];
    }
  }
  *out = o;
  return true;
}

cudaError_t launch_fused(const FusedArgs& a, int n_clusters, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fused_forward_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * kCluster);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fused_forward_kernel, a);
}

int fused_max_clusters() {
  static int cached = -1;
  if (cached >= 0) return cached;
  cudaError_t e = cudaFuncSetAttribute(fused_forward_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
  int n = 0;
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCluster);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = kFusedSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, fused_forward_kernel, &cfg);
  }
  cached = (e == cudaSuccess && n > 0) ? (n < kFusedMaxClusters ? n : kFusedMaxClusters) : 0;
  return cached;
}

}  // namespace laya
