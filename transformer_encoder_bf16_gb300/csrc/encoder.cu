// encoder.cu -- the handle behind laya_enc_*: configuration checks, RoPE
// tables, TMA descriptors over the caller's weights, per-shape workspaces with
// CUDA Graph capture and replay, and the layer loop.
//
// Layer loop (one forward pass, all on the caller's stream):
//   x = LN(E[ids])                                       embedding + norm
//   for each of the n_enc encoder and n_dec decision layers l:
//     if l == n_enc and final_norm:  x = LN_final(x)
//     h   = (l == 0 and first_attn_norm_identity) ? x : LN_attn(x)
//     qkv = RoPE(h Wqkv^T)            GEMM, plain epilogue with RoPE on q and k
//                                     (RoPE of q and k in the same epilogue: global table
//                                     iff decision layer or l % global_every == 0)
//     ctx = attention(qkv, lengths)   sliding window on local layers
//     x   = x + ctx Wo^T              GEMM, residual epilogue (in place)
//     h   = LN_mlp(x)
//     g   = gelu(h Wup_in^T) * (h Wup_gate^T)   GEMM, GeGLU epilogue
//     x   = x + g Wdown^T             GEMM, residual epilogue (last layer: into out)
// Sources: "Run Laya encoder and decision layers on CUDA" ("Purpose",
// "H800 comparison"); "[RFC]: Native Laya inference with Rust and CUDA #14"
// ("Design": separate QKV, RoPE and attention launches; per-shape CUDA Graphs
// with two warm-ups before a synchronous capture; an LRU cache of four shapes
// and 512 MiB of workspaces); "[Performance]: Optimize native Rust/CUDA Laya
// inference #66" ("Implementation priorities": grouped uploads with safe host
// buffer lifetimes, resolved handles reused).  The norm placement, GeGLU half
// order and layer-0 identity norm are readings of pages that do not write the
// layer equations out; the CPU oracle states the same readings.
#include <algorithm>
#include <chrono>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/laya_ops.h"
#include "internal.h"

namespace laya {

namespace {

constexpr int kMaxShapes = 4;
constexpr size_t kMaxWorkspaceBytes = 512ull << 20;

struct LayerMaps {
  CUtensorMap wqkv, wo, wup_in, wup_gate, wdown;
  CUtensorMap wup_il;  // the up-projection as interleaved 128-row tiles (kGemmGegluIl)
  const bf16* attn_norm;
  const bf16* mlp_norm;
};

struct Workspace {
  int B = 0, S = 0, M = 0;
  // marker rows (laya_enc_run_markers): the last layer after its QKV runs on
  // Mk = B * kmax slots only; kmax = 0 for the full forward
  int kmax = 0, Mk = 0;
  int32_t* mtok = nullptr;  // device staging [Mk]: each slot's token row in the activations
  int32_t* mpos = nullptr;  // device staging [Mk]: each slot's position in its row
  bf16 *xm = nullptr, *ctxm = nullptr, *hm = nullptr, *gm = nullptr;  // slot rows
  GemmPlan p_mo, p_mup, p_mdn;
  CUtensorMap tm_ctxm, tm_hm, tm_gm;
  void* block = nullptr;  // one device allocation for every buffer below
  size_t bytes = 0;
  bf16 *x = nullptr, *h = nullptr, *qkv = nullptr, *ctx = nullptr, *g = nullptr;
  int32_t* ids = nullptr;   // device staging [M], followed by
  int32_t* lens = nullptr;  // device staging [B]
  int32_t* pos = nullptr;   // packed tokens: each token's index in its row [M]
  int32_t* host = nullptr;  // pinned staging [M + B]
  float* partials = nullptr;  // split-K workspace shared by the four GEMMs (stream-ordered)
  size_t partials_bytes = 0;
  cudaEvent_t staged = nullptr;   // the last upload from `host` has been consumed
  cudaEvent_t done = nullptr;     // the last forward using this workspace has finished
  GemmPlan p_qkv, p_o, p_up, p_dn;
  // plan tuning (tune_plans): candidate plans of each projection, timed on
  // the first run of the shape; p_* above are the chosen ones
  static constexpr int kMaxCand = 32;
  GemmPlan cand[7][kMaxCand];
  int ncand[7] = {};
  bool tuned = false;
  // activation operand of each GEMM; the TMA box height is that GEMM's own
  // token tile (plans may differ: a GeGLU split-K partial can force a smaller tile)
  CUtensorMap tm_x_qkv, tm_h_qkv, tm_ctx_o, tm_h_up, tm_g_dn;
  CUtensorMap tm_qkv_attn;  // the projection as the tcgen05 attention reads it (box 128 rows)
  // packed tokens (packing.cuh) for batches of several rows: the kernels skip
  // the padding and a last kernel writes the padded output
  bool packed = false;
  // profiling (laya_enc_set_profiling): one release time per launch plus the
  // end mark, the class of each launch, and a graph of the stamped launches
  uint64_t* stamps = nullptr;
  std::vector<int> prof_class;
  cudaGraphExec_t prof_exec = nullptr;
  void* prof_out = nullptr;
  bool prof_pending = false;  // a profiled forward is enqueued and not yet folded
  cudaGraphExec_t exec = nullptr;
  cudaGraph_t graph = nullptr;         // the template exec was instantiated from
  cudaGraphNode_t out_node = nullptr;  // its last launch, the one writing the output
  void* graph_out = nullptr;
  uint64_t last_use = 0;
};

}  // namespace
}  // namespace laya

struct laya_enc_handle {
  laya_enc_config cfg;
  int L = 0;
  int device = 0;
  int num_sms = 0;
  const laya::bf16* tok_emb = nullptr;
  const laya::bf16* emb_norm = nullptr;
  const laya::bf16* final_norm = nullptr;
  std::vector<laya::LayerMaps> layers;
  float* rope = nullptr;  // device: cos_g, sin_g, cos_l, sin_l, each [max_seq, 32]
  int* err = nullptr;     // device error word
  cudaStream_t capture_stream = nullptr;
  std::vector<laya::Workspace*> cache;
  uint64_t tick = 0;
  laya_enc_cache_stats stats = {};  // counters of the workspace / graph cache
  bool graphs = true;
  bool pdl = true;
  bool attn_tc = true;  // attention on tcgen05 (false: the mma.sync kernel, env LAYA_ATTN_MMA_SYNC=1)
  bool tune = true;     // time candidate projection plans on a shape's first run (env LAYA_NO_TUNE=1: off)
  bool geglu_il = false;  // the up-projection can also run as interleaved tiles (I % 64 == 0)
  bool poisoned = false;
  std::string last_error;
  bool fail_next_run = false;  // test hook: the next run fails as a CUDA error would
  // failure-path test hooks on the device: the bound of the GEMM kernels'
  // barrier waits, and the next run's first projection withholding a stage
  uint64_t wait_ns = laya::kWaitLimitNs;
  bool withhold_next_run = false;
  // profiling: per-class totals of the stamped runs folded so far
  bool profiling = false;
  double prof_ms[LAYA_PROF_CLASSES] = {};
  int prof_count[LAYA_PROF_CLASSES] = {};
};

namespace laya {
namespace {

thread_local std::string g_create_error = "no error";

int fail(laya_enc_handle* h, int code, const std::string& msg) {
  if (h) {
    h->last_error = msg;
    if (code == LAYA_E_CUDA || code == LAYA_E_DEVICE) h->poisoned = true;
  } else {
    g_create_error = msg;
  }
  return code;
}

int cuda_fail(laya_enc_handle* h, cudaError_t e, const char* what) {
  return fail(h, LAYA_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && v[0] != '0';
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

void free_workspace(Workspace* w) {
  if (!w) return;
  if (w->done) cudaEventSynchronize(w->done);
  if (w->prof_exec) cudaGraphExecDestroy(w->prof_exec);
  if (w->exec) cudaGraphExecDestroy(w->exec);
  if (w->graph) cudaGraphDestroy(w->graph);
  if (w->staged) cudaEventDestroy(w->staged);
  if (w->done) cudaEventDestroy(w->done);
  if (w->host) cudaFreeHost(w->host);
  if (w->block) cudaFree(w->block);
  delete w;
}

// The projections of a workspace by slot: QKV, out, up, down, then the
// marker-row out, up and down.
enum GemmSlot : int { kGemmQkv = 0, kGemmOut, kGemmUp, kGemmDown, kGemmMarkerOut, kGemmMarkerUp,
                      kGemmMarkerDown };

GemmPlan* gemm_slot(Workspace* w, int g) {
  GemmPlan* p[7] = {&w->p_qkv, &w->p_o, &w->p_up, &w->p_dn, &w->p_mo, &w->p_mup, &w->p_mdn};
  return p[g];
}

int kernel_count(const laya_enc_config& c, const Workspace& w) {
  const int L = c.n_encoder_layers + c.n_decision_layers;
  // per layer: attention norm (not at an identity layer 0), QKV, attention,
  // out-proj, MLP norm, up, down
  int n = 1 + 7 * L - (c.first_attn_norm_identity ? 1 : 0);
  if (c.final_norm && c.n_decision_layers > 0) n += 1;
  if (w.kmax > 0) n += 1;          // marker rows: the slot gather
  else if (w.packed) n += 1;       // the padded output
  return n;
}

// Activations, staging and split-K workspace for one (B, S) shape, and the
// GEMM plans for it.
int workspace_layout(const laya_enc_handle* h, int B, int S, int kmax, Workspace* w,
                     size_t* total) {
  const laya_enc_config& c = h->cfg;
  const int M = B * S;
  const int H = c.hidden, I = c.intermediate;
  w->B = B;
  w->S = S;
  w->M = M;
  w->kmax = kmax;
  w->Mk = B * kmax;
  const int Mk = w->Mk;
  w->packed = B > 1;
  if (!plan_gemm(M, 3 * H, H, kGemmPlain, h->num_sms, 0, 0, &w->p_qkv) ||
      !plan_gemm(M, H, H, kGemmResidual, h->num_sms, 0, 0, &w->p_o) ||
      !plan_gemm(M, I, H, kGemmGeglu, h->num_sms, 0, 0, &w->p_up) ||
      !plan_gemm(M, H, I, kGemmResidual, h->num_sms, 0, 0, &w->p_dn))
    return LAYA_E_INVAL;
  if (kmax > 0 && (!plan_gemm(Mk, H, H, kGemmResidual, h->num_sms, 0, 0, &w->p_mo) ||
                   !plan_gemm(Mk, I, H, kGemmGeglu, h->num_sms, 0, 0, &w->p_mup) ||
                   !plan_gemm(Mk, H, I, kGemmResidual, h->num_sms, 0, 0, &w->p_mdn)))
    return LAYA_E_INVAL;
  // candidates for the timing on the first run (the model's choice first)
  for (int g = 0; g < 7; ++g) {
    GemmPlan* pg = gemm_slot(w, g);
    w->ncand[g] = 0;
    if (g >= kGemmMarkerOut && kmax == 0) continue;
    // the model's choice first (kept unless another candidate is clearly faster)
    w->cand[g][0] = *pg;
    w->ncand[g] = 1;
    // the up-projection also as one interleaved weight tile per 64 features
    if (pg->kind == kGemmGeglu && h->geglu_il)
      w->ncand[g] += plan_candidates(pg->M, pg->N, pg->K, kGemmGegluIl, h->num_sms,
                                     w->cand[g] + w->ncand[g], 12);
    w->ncand[g] += plan_candidates(pg->M, pg->N, pg->K, pg->kind, h->num_sms,
                                   w->cand[g] + w->ncand[g], Workspace::kMaxCand - w->ncand[g]);
    // distinct plans only
    int n = 0;
    for (int k = 0; k < w->ncand[g]; ++k) {
      const GemmPlan& c = w->cand[g][k];
      bool dup = false;
      for (int j = 0; j < n && !dup; ++j) {
        const GemmPlan& d = w->cand[g][j];
        dup = d.kind == c.kind && d.nt == c.nt && d.splits == c.splits &&
              d.persistent == c.persistent && d.pair == c.pair;
      }
      if (!dup) w->cand[g][n++] = c;
    }
    w->ncand[g] = n;
  }
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  const size_t ox = take(static_cast<size_t>(M) * H * 2);
  const size_t oh = take(static_cast<size_t>(M) * H * 2);
  const size_t oq = take(static_cast<size_t>(M) * 3 * H * 2);
  const size_t oc = take(static_cast<size_t>(M) * H * 2);
  const size_t og = take(static_cast<size_t>(M) * I * 2);
  // ids, lengths, slot tokens, slot positions: adjacent, one upload
  const size_t oi = take(static_cast<size_t>(M + B + 2 * Mk) * 4);
  const size_t opos = take(static_cast<size_t>(M) * 4);
  const size_t oxm = take(static_cast<size_t>(Mk) * H * 2);
  const size_t ocm = take(static_cast<size_t>(Mk) * H * 2);
  const size_t ohm = take(static_cast<size_t>(Mk) * H * 2);
  const size_t ogm = take(static_cast<size_t>(Mk) * I * 2);
  // split-K partials: room for the largest candidate of any projection
  size_t pbytes = 0;
  for (int g = 0; g < 7; ++g) {
    if (g >= kGemmMarkerOut && kmax == 0) continue;
    pbytes = std::max(pbytes, gemm_slot(w, g)->workspace_bytes);
    for (int k = 0; k < w->ncand[g]; ++k) pbytes = std::max(pbytes, w->cand[g][k].workspace_bytes);
  }
  const size_t ostamp = take(static_cast<size_t>(kernel_count(c, *w) + 1) * sizeof(uint64_t));
  const size_t op = take(pbytes);
  *total = off;
  if (w->block) {
    char* base = static_cast<char*>(w->block);
    w->x = reinterpret_cast<bf16*>(base + ox);
    w->h = reinterpret_cast<bf16*>(base + oh);
    w->qkv = reinterpret_cast<bf16*>(base + oq);
    w->ctx = reinterpret_cast<bf16*>(base + oc);
    w->g = reinterpret_cast<bf16*>(base + og);
    w->ids = reinterpret_cast<int32_t*>(base + oi);
    w->lens = w->ids + M;
    w->mtok = w->lens + B;
    w->mpos = w->mtok + Mk;
    w->pos = reinterpret_cast<int32_t*>(base + opos);
    if (kmax > 0) {
      w->xm = reinterpret_cast<bf16*>(base + oxm);
      w->ctxm = reinterpret_cast<bf16*>(base + ocm);
      w->hm = reinterpret_cast<bf16*>(base + ohm);
      w->gm = reinterpret_cast<bf16*>(base + ogm);
    }
    w->partials = pbytes ? reinterpret_cast<float*>(base + op) : nullptr;
    w->partials_bytes = pbytes;
    w->stamps = reinterpret_cast<uint64_t*>(base + ostamp);
  }
  return LAYA_OK;
}

// Folds the stamps of the last profiled forward on workspace w into the
// per-class totals: launch k is charged the time from its release (the
// completion of launch k - 1) to the release of launch k + 1, so the charges
// of one forward add up to its time from the first kernel's start to the
// last kernel's completion, with the overlap the graph replay has.
cudaError_t prof_fold(laya_enc_handle* h, Workspace* w) {
  if (!w->prof_pending) return cudaSuccess;
  cudaError_t e = cudaEventSynchronize(w->done);
  if (e != cudaSuccess) return e;
  const size_t n = w->prof_class.size();
  std::vector<uint64_t> t(n + 1);
  e = cudaMemcpy(t.data(), w->stamps, sizeof(uint64_t) * (n + 1), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  for (size_t k = 0; k < n; ++k) {
    const double ms = t[k + 1] > t[k] ? static_cast<double>(t[k + 1] - t[k]) * 1e-6 : 0.0;
    h->prof_ms[w->prof_class[k]] += ms;
    h->prof_count[w->prof_class[k]] += 1;
  }
  w->prof_pending = false;
  return cudaSuccess;
}

cudaError_t prof_fold_all(laya_enc_handle* h) {
  for (Workspace* w : h->cache) {
    cudaError_t e = prof_fold(h, w);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// What one forward pass writes besides its workspace.
struct RunOut {
  void* out = nullptr;      // BF16 [B, S, H], or fp32 when cfg.out_fp32
  bf16* capture = nullptr;  // debug: [L, B, S, H], the residual stream entering each layer
  bool withhold = false;    // failure-path test (laya_enc_debug_withhold_next_run)
};

// Enqueues one forward pass.  out is written by the last residual sum
// directly, or through the packed rows it leaves in x (fp32: in the qkv
// buffer, which that layer's attention no longer needs).  profiling: every
// launch records its release time in w->stamps (see prof_fold), and an end
// mark follows the last launch.
cudaError_t enqueue_forward(laya_enc_handle* h, Workspace* w, const RunOut& ro,
                            cudaStream_t stream, bool profiling) {
  const laya_enc_config& c = h->cfg;
  const int H = c.hidden;
  const int M = w->M;
  const bool pdl = h->pdl;
  void* out = ro.out;
  const float* cos_g = h->rope;
  const float* sin_g = h->rope + static_cast<size_t>(c.max_seq) * 32;
  const float* cos_l = sin_g + static_cast<size_t>(c.max_seq) * 32;
  const float* sin_l = cos_l + static_cast<size_t>(c.max_seq) * 32;
  if (profiling) w->prof_class.clear();
  int idx = 0;
  // launch options of the next launch; `cls` is its profiling class
  auto next = [&](int cls, bool first = false) {
    Launch l{stream, first ? false : pdl, nullptr};
    if (profiling) {
      l.stamp = w->stamps + idx;
      w->prof_class.push_back(cls);
    }
    ++idx;
    return l;
  };
  cudaError_t e;
#define LAYA_LAUNCH(call)             \
  do {                                \
    e = (call);                       \
    if (e != cudaSuccess) return e;   \
  } while (0)

  Packing pk;
  pk.lens = w->lens;
  pk.B = w->B;
  pk.S = w->S;
  if (w->packed) pk.pos = w->pos;
  else pk.lens = nullptr;
  // debug capture of the stream entering each layer: padded layout, padding 0
  auto capture = [&](int li) -> cudaError_t {
    if (ro.capture == nullptr) return cudaSuccess;
    bf16* dst = ro.capture + static_cast<size_t>(li) * w->B * w->S * H;
    return launch_unpack_rows(w->x, w->lens, w->B, w->S, H * 2, dst, next(LAYA_PROF_OUTPUT));
  };
  LAYA_LAUNCH(launch_embed_layernorm(h->tok_emb, h->emb_norm, w->ids, M, H, c.vocab, c.ln_eps,
                                     w->x, h->err, next(LAYA_PROF_EMBED_NORM, true), pk));
  for (int li = 0; li < h->L; ++li) {
    const LayerMaps& lw = h->layers[li];
    const bool dec = li >= c.n_encoder_layers;
    const bool glob = dec || (li % c.global_every == 0);
    LAYA_LAUNCH(capture(li));
    if (li == c.n_encoder_layers && c.final_norm)
      LAYA_LAUNCH(launch_layernorm(w->x, h->final_norm, M, H, c.ln_eps, w->x,
                                   next(LAYA_PROF_NORM), pk));
    GemmOperands o;
    o.err = h->err;
    o.wait_ns = h->wait_ns;
    o.withhold = ro.withhold && li == 0;  // the first projection of the forward
    o.partials = w->partials;
    o.partials_bytes = w->partials_bytes;
    o.lens = pk.lens;
    o.lens_B = pk.B;
    o.lens_S = pk.S;
    o.rope_pos = pk.pos;  // read by the RoPE epilogue only
    const CUtensorMap* qkv_in = &w->tm_h_qkv;
    if (li == 0 && c.first_attn_norm_identity) {
      qkv_in = &w->tm_x_qkv;
    } else {
      LAYA_LAUNCH(launch_layernorm(w->x, lw.attn_norm, M, H, c.ln_eps, w->h,
                                   next(LAYA_PROF_NORM), pk));
    }
    o.w = lw.wqkv;
    o.w2 = lw.wqkv;
    o.x = *qkv_in;
    o.x_box_rows = w->p_qkv.x_box();
    o.y = w->qkv;
    // RoPE in the QKV epilogue: q and k columns [0, 2H) leave the GEMM rotated
    o.rope_cos = glob ? cos_g : cos_l;
    o.rope_sin = glob ? sin_g : sin_l;
    o.rope_S = w->S;
    o.rope_cols = 2 * H;
    LAYA_LAUNCH(launch_gemm(w->p_qkv, o, next(LAYA_PROF_QKV)));
    o.withhold = false;
    o.rope_cos = o.rope_sin = nullptr;
    if (li == h->L - 1 && w->kmax > 0) {
      // marker rows: everything after the keys and values is row-wise, so the
      // rest of the last layer runs on the Mk slot rows alone
      LAYA_LAUNCH(launch_gather_rows(w->x, w->mtok, w->Mk, H * 2, w->xm, next(LAYA_PROF_OUTPUT)));
      LAYA_LAUNCH(launch_attention_rows(w->qkv, w->lens, w->mtok, w->mpos, w->B, w->S, w->kmax,
                                        c.heads, glob ? 1 : 0, c.local_half_window, w->packed,
                                        w->ctxm, h->err, next(LAYA_PROF_ATTN)));
      GemmOperands om;
      om.err = h->err;
      om.wait_ns = h->wait_ns;
      om.partials = w->partials;
      om.partials_bytes = w->partials_bytes;
      om.w = lw.wo;
      om.w2 = lw.wo;
      om.x = w->tm_ctxm;
      om.x_box_rows = w->p_mo.x_box();
      om.y = w->xm;
      om.residual = w->xm;
      LAYA_LAUNCH(launch_gemm(w->p_mo, om, next(LAYA_PROF_OUT)));
      LAYA_LAUNCH(launch_layernorm(w->xm, lw.mlp_norm, w->Mk, H, c.ln_eps, w->hm,
                                   next(LAYA_PROF_NORM)));
      om.w = w->p_mup.kind == kGemmGegluIl ? lw.wup_il : lw.wup_in;
      om.w2 = lw.wup_gate;
      om.x = w->tm_hm;
      om.x_box_rows = w->p_mup.x_box();
      om.y = w->gm;
      om.residual = nullptr;
      LAYA_LAUNCH(launch_gemm(w->p_mup, om, next(LAYA_PROF_UP)));
      om.w = lw.wdown;
      om.w2 = lw.wdown;
      om.x = w->tm_gm;
      om.x_box_rows = w->p_mdn.x_box();
      om.y = static_cast<bf16*>(out);
      om.residual = w->xm;
      if (c.out_fp32) om.y_f32 = static_cast<float*>(out);
      LAYA_LAUNCH(launch_gemm(w->p_mdn, om, next(LAYA_PROF_DOWN)));
      break;
    }
    if (h->attn_tc)
      LAYA_LAUNCH(launch_attention_tc(w->tm_qkv_attn, w->lens, w->B, w->S, c.heads, glob ? 1 : 0,
                                      c.local_half_window, w->ctx, h->err, next(LAYA_PROF_ATTN),
                                      w->packed));
    else
      LAYA_LAUNCH(launch_attention(w->qkv, w->lens, w->B, w->S, c.heads, glob ? 1 : 0,
                                   c.local_half_window, w->ctx, h->err, next(LAYA_PROF_ATTN),
                                   nullptr, nullptr, w->packed));
    o.w = lw.wo;
    o.w2 = lw.wo;
    o.x = w->tm_ctx_o;
    o.x_box_rows = w->p_o.x_box();
    o.y = w->x;
    o.residual = w->x;
    LAYA_LAUNCH(launch_gemm(w->p_o, o, next(LAYA_PROF_OUT)));
    LAYA_LAUNCH(launch_layernorm(w->x, lw.mlp_norm, M, H, c.ln_eps, w->h, next(LAYA_PROF_NORM),
                                 pk));
    o.w = w->p_up.kind == kGemmGegluIl ? lw.wup_il : lw.wup_in;
    o.w2 = lw.wup_gate;
    o.x = w->tm_h_up;
    o.x_box_rows = w->p_up.x_box();
    o.y = w->g;
    o.residual = nullptr;
    LAYA_LAUNCH(launch_gemm(w->p_up, o, next(LAYA_PROF_UP)));
    o.w = lw.wdown;
    o.w2 = lw.wdown;
    o.x = w->tm_g_dn;
    o.x_box_rows = w->p_dn.x_box();
    const bool last = li == h->L - 1;
    o.y = (last && !w->packed) ? static_cast<bf16*>(out) : w->x;
    o.residual = w->x;
    if (last && c.out_fp32)
      o.y_f32 = w->packed ? reinterpret_cast<float*>(w->qkv) : static_cast<float*>(out);
    LAYA_LAUNCH(launch_gemm(w->p_dn, o, next(LAYA_PROF_DOWN)));
  }
  if (w->packed && w->kmax == 0)
    LAYA_LAUNCH(launch_unpack_rows(c.out_fp32 ? static_cast<const void*>(w->qkv) : w->x, w->lens,
                                   w->B, w->S, H * (c.out_fp32 ? 4 : 2), out,
                                   next(LAYA_PROF_OUTPUT)));
  if (profiling) {
    // the end mark: released when the last launch has completed
    Launch l{stream, pdl, w->stamps + idx};
    LAYA_LAUNCH(launch_stamp(l));
  }
#undef LAYA_LAUNCH
  return cudaSuccess;
}

// TMA descriptors over the workspace activations; each GEMM's box height is
// its plan's token tile.
bool build_activation_maps(const laya_enc_handle* h, Workspace* w) {
  const laya_enc_config& c = h->cfg;
  const int M = w->M;
  auto box = [](const GemmPlan& p) { return static_cast<uint32_t>(p.x_box()); };
  const uint64_t ldh = c.hidden * 2ull, ldi = c.intermediate * 2ull;
  bool ok = make_tmap_bf16_2d(&w->tm_x_qkv, w->x, M, c.hidden, ldh, box(w->p_qkv)) &&
            make_tmap_bf16_2d(&w->tm_h_qkv, w->h, M, c.hidden, ldh, box(w->p_qkv)) &&
            make_tmap_bf16_2d(&w->tm_ctx_o, w->ctx, M, c.hidden, ldh, box(w->p_o)) &&
            make_tmap_bf16_2d(&w->tm_h_up, w->h, M, c.hidden, ldh, box(w->p_up)) &&
            make_tmap_bf16_2d(&w->tm_g_dn, w->g, M, c.intermediate, ldi, box(w->p_dn)) &&
            make_tmap_bf16_2d(&w->tm_qkv_attn, w->qkv, M, 3ull * c.hidden, 3 * ldh, 128);
  if (ok && w->kmax > 0) {
    const int Mk = w->Mk;
    ok = make_tmap_bf16_2d(&w->tm_ctxm, w->ctxm, Mk, c.hidden, ldh, box(w->p_mo)) &&
         make_tmap_bf16_2d(&w->tm_hm, w->hm, Mk, c.hidden, ldh, box(w->p_mup)) &&
         make_tmap_bf16_2d(&w->tm_gm, w->gm, Mk, c.intermediate, ldi, box(w->p_mdn));
  }
  return ok;
}

// Plans chosen by timing, shared by every handle of the process so that two
// handles running the same shape take the same plans (and give the same
// bits): (M, N, K, kind, rows of the batch or 0 for marker slots) -> (token
// tile, split-K factor, paired CTAs, kind run).
std::mutex g_tuned_mu;
std::map<std::tuple<int, int, int, int, int>, std::tuple<int, int, int, int>> g_tuned;

// The choices can also live in a text file named by the environment variable
// LAYA_PLAN_CACHE (one line per shape: M N K kind rows, then token tile,
// split-K, pairing, kind run), read once per process before the first
// tuning and rewritten after every tuning that adds a shape: a second
// process (a profiler's run, say, whose timings would differ) then runs the
// plans the first one chose.  A line whose plan is not among a shape's
// candidates is ignored (the model's plan runs, untimed).
const char* plan_cache_path() {
  const char* p = std::getenv("LAYA_PLAN_CACHE");
  return (p != nullptr && p[0] != '\0') ? p : nullptr;
}

void load_plan_cache() {  // with g_tuned_mu held
  static bool loaded = false;
  if (loaded) return;
  loaded = true;
  const char* path = plan_cache_path();
  if (path == nullptr) return;
  std::ifstream in(path);
  int M, N, K, kind, rows, nt, splits, pair, krun;
  while (in >> M >> N >> K >> kind >> rows >> nt >> splits >> pair >> krun)
    g_tuned.emplace(std::make_tuple(M, N, K, kind, rows), std::make_tuple(nt, splits, pair, krun));
}

void save_plan_cache() {  // with g_tuned_mu held
  const char* path = plan_cache_path();
  if (path == nullptr) return;
  std::ofstream out(path, std::ios::trunc);
  for (const auto& e : g_tuned)
    out << std::get<0>(e.first) << ' ' << std::get<1>(e.first) << ' ' << std::get<2>(e.first)
        << ' ' << std::get<3>(e.first) << ' ' << std::get<4>(e.first) << ' '
        << std::get<0>(e.second) << ' ' << std::get<1>(e.second) << ' ' << std::get<2>(e.second)
        << ' ' << std::get<3>(e.second) << '\n';
}

// Times the candidate plans of each projection on the first run of a shape,
// on `stream` after that run's input upload (the packed row lengths are real,
// the activations are the workspace's), and keeps the fastest; the model's
// choice stays unless another candidate is faster by more than 5 %.  Each
// candidate is launched as in the forward (programmatic dependent launch,
// layer-0 weights), into scratch outputs of the workspace.
int marker_or_b(const Workspace* w, int g) { return g >= kGemmMarkerOut ? 0 : w->B; }

int tune_plans(laya_enc_handle* h, Workspace* w, cudaStream_t stream) {
  const laya_enc_config& c = h->cfg;
  const int H = c.hidden;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  const LayerMaps& lw = h->layers[0];
  const uint64_t ldh = H * 2ull, ldi = c.intermediate * 2ull;
  for (int g = 0; g < 7 && e == cudaSuccess; ++g) {
    if (w->ncand[g] <= 0) continue;
    GemmPlan* slot = gemm_slot(w, g);
    const auto key = std::make_tuple(slot->M, slot->N, slot->K, slot->kind, marker_or_b(w, g));
    {
      std::lock_guard<std::mutex> lk(g_tuned_mu);
      load_plan_cache();
      auto it = g_tuned.find(key);
      if (it != g_tuned.end()) {
        for (int k = 0; k < w->ncand[g]; ++k)
          if (w->cand[g][k].nt == std::get<0>(it->second) &&
              w->cand[g][k].splits == std::get<1>(it->second) &&
              w->cand[g][k].pair == std::get<2>(it->second) &&
              w->cand[g][k].kind == std::get<3>(it->second))
            *slot = w->cand[g][k];
        continue;
      }
    }
    const bool marker = g >= kGemmMarkerOut;
    const int rows = marker ? w->Mk : w->M;
    double best_ms = 0.0;
    int best = 0;
    for (int k = 0; k < w->ncand[g] && e == cudaSuccess; ++k) {
      const GemmPlan& p = w->cand[g][k];
      GemmOperands o;
      o.err = h->err;
      o.wait_ns = h->wait_ns;
      o.partials = w->partials;
      o.partials_bytes = w->partials_bytes;
      if (!marker && w->packed) {
        o.lens = w->lens;
        o.lens_B = w->B;
        o.lens_S = w->S;
      }
      o.x_box_rows = p.x_box();
      const uint32_t nt = static_cast<uint32_t>(p.x_box());  // activation box rows
      bool ok = true;
      switch (g) {
        case kGemmQkv:
          o.w = o.w2 = lw.wqkv;
          ok = make_tmap_bf16_2d(&o.x, w->h, rows, H, ldh, nt);
          o.y = w->qkv;
          o.rope_cos = h->rope;
          o.rope_sin = h->rope + static_cast<size_t>(c.max_seq) * 32;
          o.rope_S = w->S;
          o.rope_cols = 2 * H;
          o.rope_pos = w->packed ? w->pos : nullptr;
          break;
        case kGemmOut:
        case kGemmMarkerOut:
          o.w = o.w2 = lw.wo;
          ok = make_tmap_bf16_2d(&o.x, marker ? w->ctxm : w->ctx, rows, H, ldh, nt);
          o.residual = marker ? w->xm : w->x;
          o.y = marker ? w->hm : w->h;
          break;
        case kGemmUp:
        case kGemmMarkerUp:
          o.w = p.kind == kGemmGegluIl ? lw.wup_il : lw.wup_in;
          o.w2 = lw.wup_gate;
          ok = make_tmap_bf16_2d(&o.x, marker ? w->hm : w->h, rows, H, ldh, nt);
          o.y = marker ? w->gm : w->g;
          break;
        default:
          o.w = o.w2 = lw.wdown;
          ok = make_tmap_bf16_2d(&o.x, marker ? w->gm : w->g, rows, c.intermediate, ldi, nt);
          o.residual = marker ? w->xm : w->x;
          o.y = marker ? w->hm : w->h;
          break;
      }
      if (!ok) {
        e = cudaErrorInvalidValue;
        break;
      }
      const Launch l{stream, h->pdl, nullptr};
      for (int r = 0; r < 3 && e == cudaSuccess; ++r) e = launch_gemm(p, o, l);
      if (e == cudaSuccess) e = cudaEventRecord(e0, stream);
      for (int r = 0; r < 12 && e == cudaSuccess; ++r) e = launch_gemm(p, o, l);
      if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
      if (e == cudaSuccess) e = cudaEventSynchronize(e1);
      float ms = 0.f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
      if (e != cudaSuccess) break;
      if (k == 0 || ms < best_ms * (best == 0 ? 0.95 : 1.0)) {
        best_ms = ms;
        best = k;
      }
    }
    if (e != cudaSuccess) break;
    *slot = w->cand[g][best];
    std::lock_guard<std::mutex> lk(g_tuned_mu);
    g_tuned.emplace(key, std::make_tuple(slot->nt, slot->splits, slot->pair, slot->kind));
    save_plan_cache();
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail(h, e, "plan tuning");
  if (!build_activation_maps(h, w)) return fail(h, LAYA_E_CUDA, "tensor map encoding failed");
  w->tuned = true;
  return LAYA_OK;
}

int get_workspace(laya_enc_handle* h, int B, int S, int kmax, Workspace** out) {
  for (Workspace* w : h->cache) {
    if (w->B == B && w->S == S && w->kmax == kmax) {
      w->last_use = ++h->tick;
      *out = w;
      return LAYA_OK;
    }
  }
  const auto t_setup = std::chrono::steady_clock::now();
  Workspace* w = new (std::nothrow) Workspace();
  if (!w) return fail(h, LAYA_E_NOMEM, "workspace: host allocation failed");
  size_t bytes = 0;
  if (workspace_layout(h, B, S, kmax, w, &bytes) != LAYA_OK) {
    delete w;
    return fail(h, LAYA_E_INVAL, "no GEMM plan for this shape");
  }
  // evict least-recently-used shapes beyond four or 512 MiB
  auto used = [&]() {
    size_t s = 0;
    for (Workspace* x : h->cache) s += x->bytes;
    return s;
  };
  while (!h->cache.empty() && (h->cache.size() >= static_cast<size_t>(kMaxShapes) ||
                               used() + bytes > kMaxWorkspaceBytes)) {
    auto it = std::min_element(h->cache.begin(), h->cache.end(),
                               [](Workspace* a, Workspace* b) { return a->last_use < b->last_use; });
    free_workspace(*it);
    h->cache.erase(it);
    ++h->stats.evicted;
  }
  cudaError_t e = cudaMalloc(&w->block, bytes);
  if (e != cudaSuccess) {
    delete w;
    return fail(h, LAYA_E_NOMEM, std::string("workspace: ") + cudaGetErrorString(e));
  }
  w->bytes = bytes;
  workspace_layout(h, B, S, kmax, w, &bytes);
  e = cudaHostAlloc(reinterpret_cast<void**>(&w->host), sizeof(int32_t) * (w->M + B + 2 * w->Mk),
                    cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&w->staged, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&w->done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemset(w->block, 0, w->bytes);
  if (e != cudaSuccess) {
    free_workspace(w);
    return fail(h, LAYA_E_NOMEM, std::string("workspace: ") + cudaGetErrorString(e));
  }
  const bool ok = build_activation_maps(h, w);
  if (!ok) {
    free_workspace(w);
    return fail(h, LAYA_E_CUDA, "workspace: tensor map encoding failed");
  }
  w->last_use = ++h->tick;
  h->cache.push_back(w);
  ++h->stats.created;
  h->stats.setup_ms += std::chrono::duration<double, std::milli>(
                           std::chrono::steady_clock::now() - t_setup).count();
  *out = w;
  return LAYA_OK;
}

// Captures one forward pass of w into a graph.  sink: the capture's last
// launch (the one writing out), null if it cannot be told.
int capture_graph(laya_enc_handle* h, Workspace* w, void* out, bool profiling,
                  cudaGraph_t* graph, cudaGraphExec_t* exec, cudaGraphNode_t* sink) {
  *graph = nullptr;
  *exec = nullptr;
  *sink = nullptr;
  cudaError_t e = cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamBeginCapture");
  RunOut ro;
  ro.out = out;
  cudaError_t el = enqueue_forward(h, w, ro, h->capture_stream, profiling);
  // the capture's single open dependency is the last launch
  if (el == cudaSuccess) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t* deps = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(h->capture_stream, &st, nullptr, nullptr, &deps, nullptr, &nd) ==
            cudaSuccess &&
        nd == 1)
      *sink = deps[0];
    else
      cudaGetLastError();
  }
  e = cudaStreamEndCapture(h->capture_stream, graph);
  if (el != cudaSuccess) {
    if (*graph) cudaGraphDestroy(*graph);
    *graph = nullptr;
    return cuda_fail(h, el, "launch during capture");
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamEndCapture");
  e = cudaGraphInstantiate(exec, *graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(*graph);
    *graph = nullptr;
    *exec = nullptr;
    return cuda_fail(h, e, "cudaGraphInstantiate");
  }
  return LAYA_OK;
}

int run_common(laya_enc_handle* h, Workspace* w, const RunOut& ro, cudaStream_t stream) {
  void* out = ro.out;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamIsCapturing");
  if (!w->tuned) {
    if (cap == cudaStreamCaptureStatusNone && h->tune) {
      const auto t_tune = std::chrono::steady_clock::now();
      const int rc = tune_plans(h, w, stream);
      if (rc != LAYA_OK) return rc;
      h->stats.capture_ms += std::chrono::duration<double, std::milli>(
                                 std::chrono::steady_clock::now() - t_tune).count();
    }
    w->tuned = true;  // inside a caller's capture: the model's plans stay
  }
  const bool profiling = h->profiling && cap == cudaStreamCaptureStatusNone && !ro.capture;
  if (profiling) {
    e = prof_fold_all(h);
    if (e != cudaSuccess) return cuda_fail(h, e, "profiling stamps");
  }
  if (!h->graphs || cap != cudaStreamCaptureStatusNone || ro.capture != nullptr || ro.withhold) {
    e = enqueue_forward(h, w, ro, stream, profiling);
    if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  } else if (profiling) {
    // the same launches with release stamps, in a graph of their own
    if (w->prof_exec == nullptr || w->prof_out != out) {
      if (w->prof_exec) cudaGraphExecDestroy(w->prof_exec);
      w->prof_exec = nullptr;
      cudaGraph_t g = nullptr;
      cudaGraphNode_t sink = nullptr;
      const int rc = capture_graph(h, w, out, true, &g, &w->prof_exec, &sink);
      if (rc != LAYA_OK) return rc;
      cudaGraphDestroy(g);
      w->prof_out = out;
    }
    e = cudaGraphLaunch(w->prof_exec, stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGraphLaunch");
  } else {
    // a new output buffer for a captured shape: repoint the launch that
    // writes the output instead of capturing again
    if (w->exec != nullptr && w->graph_out != out && w->out_node != nullptr) {
      const cudaError_t er =
          (w->packed && w->kmax == 0)
              ? unpack_node_retarget(w->exec, w->out_node, w->graph_out, out)
              : gemm_node_retarget(w->exec, w->out_node, w->graph_out, out);
      if (er == cudaSuccess) {
        w->graph_out = out;
        ++h->stats.retargets;
      } else {
        cudaGetLastError();  // not retargetable: capture again below
      }
    }
    if (w->exec == nullptr || w->graph_out != out) {
      const auto t_cap = std::chrono::steady_clock::now();
      if (w->exec == nullptr) {
        // two eager warm-up passes before the first capture of a shape
        for (int i = 0; i < 2; ++i) {
          e = enqueue_forward(h, w, ro, stream, false);
          if (e != cudaSuccess) return cuda_fail(h, e, "warm-up launch");
        }
      }
      e = cudaStreamSynchronize(stream);
      if (e != cudaSuccess) return cuda_fail(h, e, "warm-up");
      if (w->exec) {
        cudaGraphExecDestroy(w->exec);
        w->exec = nullptr;
      }
      if (w->graph) {
        cudaGraphDestroy(w->graph);
        w->graph = nullptr;
        w->out_node = nullptr;
      }
      const int rc = capture_graph(h, w, out, false, &w->graph, &w->exec, &w->out_node);
      if (rc != LAYA_OK) return rc;
      w->graph_out = out;
      ++h->stats.captures;
      h->stats.capture_ms += std::chrono::duration<double, std::milli>(
                                 std::chrono::steady_clock::now() - t_cap).count();
    }
    e = cudaGraphLaunch(w->exec, stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGraphLaunch");
  }
  e = cudaEventRecord(w->done, stream);
  if (e != cudaSuccess && cap == cudaStreamCaptureStatusNone)
    return cuda_fail(h, e, "cudaEventRecord");
  if (profiling) w->prof_pending = true;
  return LAYA_OK;
}

int check_run_args(laya_enc_handle* h, int B, int S, void* out) {
  if (!h) return LAYA_E_INVAL;
  if (h->poisoned) return fail(h, LAYA_E_POISONED, "handle is poisoned by an earlier error");
  if (B < 1 || B > h->cfg.max_batch)
    return fail(h, LAYA_E_INVAL, "batch outside [1, max_batch]");
  if (S < 1 || S > h->cfg.max_seq) return fail(h, LAYA_E_INVAL, "seq outside [1, max_seq]");
  if (!out || (reinterpret_cast<uintptr_t>(out) & 15u) != 0)
    return fail(h, LAYA_E_INVAL, "out_hidden must be a 16-byte aligned device pointer");
  return LAYA_OK;
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace laya

using laya::bf16;

extern "C" {

int laya_enc_abi_version(void) { return LAYA_ENC_ABI_VERSION; }

int laya_enc_validate_config(const laya_enc_config* c) {
  if (!c) return LAYA_E_INVAL;
  if (!laya::rowops_supported_hidden(c->hidden)) return LAYA_E_INVAL;
  if (c->head_dim != 64 || c->heads < 1 || c->heads * c->head_dim != c->hidden) return LAYA_E_INVAL;
  if (c->intermediate < 64 || c->intermediate % 64 != 0) return LAYA_E_INVAL;
  if (c->vocab < 1) return LAYA_E_INVAL;
  if (c->n_encoder_layers < 1 || c->n_decision_layers < 0) return LAYA_E_INVAL;
  if (c->n_encoder_layers + c->n_decision_layers > 256) return LAYA_E_INVAL;
  if (c->global_every < 1 || c->local_half_window < 0) return LAYA_E_INVAL;
  if (!(c->theta_global > 0.f) || !(c->theta_local > 0.f) || !(c->ln_eps > 0.f))
    return LAYA_E_INVAL;
  if (c->max_batch < 1 || c->max_batch > 16 || c->max_seq < 1 || c->max_seq > 512)
    return LAYA_E_INVAL;
  if ((c->rope_table_bf16 | 1) != 1 || (c->first_attn_norm_identity | 1) != 1 ||
      (c->final_norm | 1) != 1 || (c->out_fp32 | 1) != 1)
    return LAYA_E_INVAL;
  return LAYA_OK;
}

int laya_enc_create(const laya_enc_config* cfg, const laya_enc_weights* wts,
                    laya_enc_handle** out) {
  using namespace laya;
  if (out) *out = nullptr;
  if (!out || !cfg || !wts) return fail(nullptr, LAYA_E_INVAL, "null argument");
  if (laya_enc_validate_config(cfg) != LAYA_OK)
    return fail(nullptr, LAYA_E_INVAL, "unsupported configuration");
  const int L = cfg->n_encoder_layers + cfg->n_decision_layers;
  if (wts->n_layers != L || !wts->layers)
    return fail(nullptr, LAYA_E_INVAL, "weights.n_layers does not match the configuration");
  auto aligned = [](const void* p) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
  };
  if (!aligned(wts->tok_emb) || !aligned(wts->emb_norm) ||
      (cfg->final_norm && !aligned(wts->final_norm)))
    return fail(nullptr, LAYA_E_INVAL, "embedding or norm weights missing or misaligned");
  for (int l = 0; l < L; ++l) {
    const laya_enc_layer_weights& lw = wts->layers[l];
    const bool need_attn_norm = !(l == 0 && cfg->first_attn_norm_identity);
    if ((need_attn_norm && !aligned(lw.attn_norm)) || !aligned(lw.wqkv) || !aligned(lw.wo) ||
        !aligned(lw.mlp_norm) || !aligned(lw.wup) || !aligned(lw.wdown))
      return fail(nullptr, LAYA_E_INVAL,
                  "layer " + std::to_string(l) + ": weight missing or not 16-byte aligned");
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(nullptr, LAYA_E_CUDA, cudaGetErrorString(e));
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(nullptr, LAYA_E_UNSUPPORTED,
                "device compute capability " + std::to_string(major) + "." +
                    std::to_string(minor) + " is not 10.3 (GB300)");

  laya_enc_handle* h = new (std::nothrow) laya_enc_handle();
  if (!h) return fail(nullptr, LAYA_E_NOMEM, "host allocation failed");
  h->cfg = *cfg;
  h->L = L;
  h->device = dev;
  h->num_sms = device_sm_count();
  h->graphs = !env_flag("LAYA_EAGER");
  h->pdl = !env_flag("LAYA_NO_PDL");
  h->attn_tc = !env_flag("LAYA_ATTN_MMA_SYNC");
  h->tune = !env_flag("LAYA_NO_TUNE");
  h->geglu_il = cfg->intermediate % 64 == 0;
  h->tok_emb = static_cast<const bf16*>(wts->tok_emb);
  h->emb_norm = static_cast<const bf16*>(wts->emb_norm);
  h->final_norm = static_cast<const bf16*>(wts->final_norm);
  const int H = cfg->hidden, I = cfg->intermediate;
  h->layers.resize(L);
  bool ok = true;
  for (int l = 0; l < L && ok; ++l) {
    const laya_enc_layer_weights& lw = wts->layers[l];
    LayerMaps& m = h->layers[l];
    m.attn_norm = static_cast<const bf16*>(lw.attn_norm);
    m.mlp_norm = static_cast<const bf16*>(lw.mlp_norm);
    const char* up = static_cast<const char*>(lw.wup);
    ok = make_tmap_bf16_2d(&m.wqkv, lw.wqkv, 3ull * H, H, H * 2ull, 128) &&
         make_tmap_bf16_2d(&m.wo, lw.wo, H, H, H * 2ull, 128) &&
         make_tmap_bf16_2d(&m.wup_in, up, I, H, H * 2ull, 128) &&
         make_tmap_bf16_2d(&m.wup_gate, up + static_cast<size_t>(I) * H * 2, I, H, H * 2ull,
                           128) &&
         make_tmap_bf16_2d(&m.wdown, lw.wdown, H, I, I * 2ull, 128);
    if (ok && h->geglu_il) h->geglu_il = make_tmap_geglu_il(&m.wup_il, lw.wup, I, H);
  }
  if (!ok) {
    delete h;
    return fail(nullptr, LAYA_E_CUDA, "weight tensor map encoding failed");
  }
  const size_t tab = static_cast<size_t>(cfg->max_seq) * 32;
  std::vector<float> host(4 * tab);
  rope_table_host(cfg->theta_global, cfg->max_seq, 32, cfg->rope_table_bf16, host.data(),
                  host.data() + tab);
  rope_table_host(cfg->theta_local, cfg->max_seq, 32, cfg->rope_table_bf16, host.data() + 2 * tab,
                  host.data() + 3 * tab);
  e = cudaMalloc(&h->rope, 4 * tab * sizeof(float));
  if (e == cudaSuccess)
    e = cudaMemcpy(h->rope, host.data(), 4 * tab * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMalloc(&h->err, 4 * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, 4 * sizeof(int));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    std::string msg = std::string("create: ") + cudaGetErrorString(e);
    laya_enc_destroy(h);
    return fail(nullptr, LAYA_E_NOMEM, msg);
  }
  h->last_error = "no error";
  *out = h;
  return LAYA_OK;
}

static int run_impl(laya_enc_handle* h, const int32_t* ids, const int32_t* lengths, int B, int S,
                    const int32_t* markers, int kmax, const laya::RunOut& ro, void* stream_v,
                    bool device_inputs) {
  using namespace laya;
  int rc = check_run_args(h, B, S, ro.out);
  if (rc != LAYA_OK) return rc;
  if (!ids || !lengths) return fail(h, LAYA_E_INVAL, "null token_ids or lengths");
  if (!device_inputs) {
    for (int b = 0; b < B; ++b)
      if (lengths[b] < 1 || lengths[b] > S)
        return fail(h, LAYA_E_INVAL, "lengths[" + std::to_string(b) + "] outside [1, seq]");
    const int64_t M = static_cast<int64_t>(B) * S;
    for (int64_t t = 0; t < M; ++t)
      if (ids[t] < 0 || ids[t] >= h->cfg.vocab)
        return fail(h, LAYA_E_INVAL, "token id outside [0, vocab)");
  }
  if (kmax > 0) {
    if (!markers) return fail(h, LAYA_E_INVAL, "null marker_pos");
    if (static_cast<int64_t>(B) * kmax > LAYA_ENC_MAX_MARKERS)
      return fail(h, LAYA_E_INVAL, "batch * kmax exceeds LAYA_ENC_MAX_MARKERS");
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < kmax; ++j) {
        const int p = markers[b * kmax + j];
        if (p < -1 || p >= lengths[b])
          return fail(h, LAYA_E_INVAL, "marker_pos[" + std::to_string(b * kmax + j) +
                                           "] is not a valid token of its row (nor -1)");
      }
  }
  if (h->fail_next_run) {
    h->fail_next_run = false;
    return cuda_fail(h, cudaErrorLaunchFailure, "injected failure (test hook)");
  }
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  Workspace* w = nullptr;
  rc = get_workspace(h, B, S, kmax, &w);
  if (rc != LAYA_OK) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  RunOut run = ro;
  if (h->withhold_next_run) {
    h->withhold_next_run = false;
    run.withhold = true;
  }
  const size_t nid = static_cast<size_t>(w->M) * sizeof(int32_t);
  const size_t nlen = static_cast<size_t>(B) * sizeof(int32_t);
  if (device_inputs) {
    e = cudaMemcpyAsync(w->ids, ids, nid, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(w->lens, lengths, nlen, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "input copy");
  } else {
    // the previous upload from the pinned buffer must have been consumed
    e = cudaEventSynchronize(w->staged);
    if (e != cudaSuccess) return cuda_fail(h, e, "staging wait");
    std::memcpy(w->host, ids, nid);
    std::memcpy(w->host + w->M, lengths, nlen);
    // marker slots: the token row of each slot in the activations (packed
    // rows start at the earlier rows' lengths summed) and its position; an
    // empty slot reads its row's first token
    int32_t* mtok = w->host + w->M + B;
    int32_t* mpos = mtok + w->Mk;
    int cu = 0;
    for (int b = 0; b < B && kmax > 0; ++b) {
      const int start = w->packed ? cu : b * S;
      for (int j = 0; j < kmax; ++j) {
        const int p = markers[b * kmax + j] < 0 ? 0 : markers[b * kmax + j];
        mtok[b * kmax + j] = start + p;
        mpos[b * kmax + j] = p;
      }
      cu += lengths[b];
    }
    // ids, lengths and marker slots are adjacent on both sides: one grouped upload
    e = cudaMemcpyAsync(w->ids, w->host, nid + nlen + 2 * sizeof(int32_t) * w->Mk,
                        cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "input upload");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(stream, &cap);
    if (cap == cudaStreamCaptureStatusNone) {
      e = cudaEventRecord(w->staged, stream);
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventRecord");
    }
  }
  return run_common(h, w, run, stream);
}

int laya_enc_run(laya_enc_handle* h, const int32_t* token_ids, const int32_t* lengths, int batch,
                 int seq, void* out_hidden, void* stream) {
  laya::RunOut ro;
  ro.out = out_hidden;
  return run_impl(h, token_ids, lengths, batch, seq, nullptr, 0, ro, stream, false);
}

int laya_enc_run_device(laya_enc_handle* h, const int32_t* token_ids_dev,
                        const int32_t* lengths_dev, int batch, int seq, void* out_hidden,
                        void* stream) {
  laya::RunOut ro;
  ro.out = out_hidden;
  return run_impl(h, token_ids_dev, lengths_dev, batch, seq, nullptr, 0, ro, stream, true);
}

int laya_enc_run_markers(laya_enc_handle* h, const int32_t* token_ids, const int32_t* lengths,
                         int batch, int seq, const int32_t* marker_pos, int kmax,
                         void* out_markers, void* stream) {
  if (!h) return LAYA_E_INVAL;
  if (kmax < 1 || kmax > LAYA_ENC_MAX_MARKERS)
    return laya::fail(h, LAYA_E_INVAL, "kmax outside [1, LAYA_ENC_MAX_MARKERS]");
  laya::RunOut ro;
  ro.out = out_markers;
  return run_impl(h, token_ids, lengths, batch, seq, marker_pos, kmax, ro, stream, false);
}

int laya_enc_debug_capture(laya_enc_handle* h, const int32_t* token_ids, const int32_t* lengths,
                           int batch, int seq, void* out_hidden, void* states, void* stream) {
  if (!h) return LAYA_E_INVAL;
  if (!states || (reinterpret_cast<uintptr_t>(states) & 15u) != 0)
    return laya::fail(h, LAYA_E_INVAL, "states must be a 16-byte aligned device pointer");
  laya::RunOut ro;
  ro.out = out_hidden;
  ro.capture = static_cast<laya::bf16*>(states);
  return run_impl(h, token_ids, lengths, batch, seq, nullptr, 0, ro, stream, false);
}

int laya_enc_check(laya_enc_handle* h, void* stream) {
  using namespace laya;
  if (!h) return LAYA_E_INVAL;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, h->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "error word read");
  if (word != 0) return fail(h, LAYA_E_DEVICE, "kernel reported device error " + std::to_string(word));
  if (h->poisoned) return fail(h, LAYA_E_POISONED, "handle is poisoned by an earlier error");
  return LAYA_OK;
}

int laya_enc_debug_fail_next_run(laya_enc_handle* h) {
  if (!h) return LAYA_E_INVAL;
  h->fail_next_run = true;
  return LAYA_OK;
}

int laya_enc_debug_set_wait_limit_ns(laya_enc_handle* h, uint64_t ns) {
  if (!h) return LAYA_E_INVAL;
  if (ns == 0) ns = laya::kWaitLimitNs;
  if (ns < 1000000ull || ns > 10000000000ull)
    return laya::fail(h, LAYA_E_INVAL, "wait limit outside [1 ms, 10 s]");
  h->wait_ns = ns;
  return LAYA_OK;
}

int laya_enc_debug_withhold_next_run(laya_enc_handle* h) {
  if (!h) return LAYA_E_INVAL;
  h->withhold_next_run = true;
  return LAYA_OK;
}

int laya_enc_set_graphs(laya_enc_handle* h, int enabled) {
  if (!h) return LAYA_E_INVAL;
  h->graphs = enabled != 0;
  return LAYA_OK;
}

int laya_enc_get_cache_stats(const laya_enc_handle* h, laya_enc_cache_stats* out) {
  if (!h || !out) return LAYA_E_INVAL;
  *out = h->stats;
  out->shapes = static_cast<int32_t>(h->cache.size());
  out->max_shapes = laya::kMaxShapes;
  out->bytes = 0;
  for (const laya::Workspace* w : h->cache) out->bytes += w->bytes;
  out->max_bytes = laya::kMaxWorkspaceBytes;
  return LAYA_OK;
}

int laya_enc_set_profiling(laya_enc_handle* h, int enabled) {
  if (!h) return LAYA_E_INVAL;
  if (!enabled && h->profiling) {
    cudaError_t e = laya::prof_fold_all(h);
    if (e != cudaSuccess) return laya::cuda_fail(h, e, "profiling stamps");
  }
  h->profiling = enabled != 0;
  return LAYA_OK;
}

int laya_enc_profile_read(laya_enc_handle* h, double* ms, int* launches, int n) {
  if (!h || !ms || !launches || n < 1 || n > LAYA_PROF_CLASSES) return LAYA_E_INVAL;
  cudaError_t e = laya::prof_fold_all(h);
  if (e != cudaSuccess) return laya::cuda_fail(h, e, "profiling stamps");
  for (int c = 0; c < n; ++c) {
    ms[c] = h->prof_ms[c];
    launches[c] = h->prof_count[c];
  }
  for (int c = 0; c < LAYA_PROF_CLASSES; ++c) {
    h->prof_ms[c] = 0.0;
    h->prof_count[c] = 0;
  }
  return LAYA_OK;
}

int laya_enc_launch_count(const laya_enc_handle* h, int batch, int seq) {
  if (!h || batch < 1 || batch > h->cfg.max_batch || seq < 1 || seq > h->cfg.max_seq)
    return LAYA_E_INVAL;
  laya::Workspace w;
  size_t b = 0;
  if (laya::workspace_layout(h, batch, seq, 0, &w, &b) != LAYA_OK) return LAYA_E_INVAL;
  return laya::kernel_count(h->cfg, w);
}

int laya_enc_get_plans(const laya_enc_handle* h, int batch, int seq, int32_t* out) {
  if (!h || !out) return LAYA_E_INVAL;
  for (const laya::Workspace* w : h->cache) {
    if (w->B != batch || w->S != seq || w->kmax != 0) continue;
    const laya::GemmPlan* p[4] = {&w->p_qkv, &w->p_o, &w->p_up, &w->p_dn};
    for (int g = 0; g < 4; ++g) {
      out[5 * g + 0] = p[g]->nt;
      out[5 * g + 1] = p[g]->splits;
      out[5 * g + 2] = p[g]->pair;
      out[5 * g + 3] = p[g]->ctas();
      out[5 * g + 4] = p[g]->kind;
    }
    return LAYA_OK;
  }
  return LAYA_E_INVAL;
}

int laya_enc_workspace_bytes(const laya_enc_handle* h, int batch, int seq, size_t* bytes) {
  if (!h || !bytes || batch < 1 || batch > h->cfg.max_batch || seq < 1 || seq > h->cfg.max_seq)
    return LAYA_E_INVAL;
  laya::Workspace w;
  size_t b = 0;
  if (laya::workspace_layout(h, batch, seq, 0, &w, &b) != LAYA_OK) return LAYA_E_INVAL;
  *bytes = b;
  return LAYA_OK;
}

int laya_enc_destroy(laya_enc_handle* h) {
  if (!h) return LAYA_OK;
  for (laya::Workspace* w : h->cache) laya::free_workspace(w);
  h->cache.clear();
  if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  if (h->rope) cudaFree(h->rope);
  if (h->err) cudaFree(h->err);
  delete h;
  return LAYA_OK;
}

const char* laya_enc_last_error(const laya_enc_handle* h) {
  if (!h) return laya::g_create_error.c_str();
  return h->last_error.c_str();
}

}  // extern "C"
