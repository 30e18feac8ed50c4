// internal.h -- declarations shared by the translation units of liblaya_enc.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/laya_enc.h"

namespace laya {

using bf16 = __nv_bfloat16;

// Device error word codes (first error wins; the host maps any of them to
// LAYA_E_DEVICE).
enum DeviceError : int {
  kDevOk = 0,
  kDevWaitFull = 1,     // GEMM: MMA issuer gave up waiting for a TMA stage
  kDevWaitEmpty = 2,    // GEMM: producer gave up waiting for a free stage
  kDevWaitAccum = 3,    // GEMM: epilogue gave up waiting for the accumulator
  kDevBadId = 4,        // embedding: token id outside [0, vocab)
  kDevBadLength = 5,    // attention: row length outside [1, S]
  kDevWaitReduce = 6,   // GEMM: epilogue gave up waiting for the split-K partial slices
};

// Upper bound on any device-side wait, in nanoseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Launch options shared by every launcher.
struct Launch {
  cudaStream_t stream = nullptr;
  bool pdl = false;  // programmatic dependent launch (overlap with the previous kernel)
  // Profiling: non-null, the kernel's first CTA writes the %globaltimer value
  // at which its dependency wait returned (the previous kernel's completion)
  uint64_t* stamp = nullptr;
};

// Records the release time of a kernel (see Launch::stamp): called by one
// thread of the kernel's first CTA right after its dependency wait.
__device__ __forceinline__ void record_stamp(uint64_t* stamp) {
  if (stamp != nullptr) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    *stamp = t;
  }
}

// A kernel that only records its release time: the end mark of a profiled
// forward pass.
cudaError_t launch_stamp(Launch l);

// Packed tokens (packing.cuh): lens non-null selects them for B rows of S.
struct Packing {
  const int32_t* lens = nullptr;
  int B = 0, S = 0;
  int32_t* pos = nullptr;  // written by the packed embedding: each token's index in its row
};

// ----------------------------------------------------------- row kernels ---
cudaError_t launch_embed_layernorm(const bf16* emb, const bf16* gamma, const int32_t* ids, int M,
                                   int H, int vocab, float eps, bf16* x, int* err, Launch l,
                                   const Packing& pk = Packing());
cudaError_t launch_layernorm(const bf16* x, const bf16* gamma, int M, int H, float eps, bf16* y,
                             Launch l, const Packing& pk = Packing());
// out [B*S rows of row_bytes] (padded) from packed rows x; row_bytes a
// multiple of 16.
cudaError_t launch_unpack_rows(const void* x, const int32_t* lens, int B, int S, int row_bytes,
                               void* out, Launch l);
cudaError_t launch_rope(bf16* qkv, const float* cos_t, const float* sin_t, int B, int S,
                        int heads, Launch l);
// out[m] = x[idx[m]] for m < n, rows of row_bytes (a multiple of 16).
cudaError_t launch_gather_rows(const void* x, const int32_t* idx, int n, int row_bytes, void* out,
                               Launch l);
bool rowops_supported_hidden(int H);

// ------------------------------------------------------------- attention ---
// cos_t/sin_t non-null: RoPE is applied to q and k inside the kernel.
// packed: qkv and ctx hold packed tokens (packing.cuh) instead of B rows of S.
cudaError_t launch_attention(const bf16* qkv, const int32_t* lengths, int B, int S, int heads,
                             int global, int half_window, bf16* ctx, int* err, Launch l,
                             const float* cos_t = nullptr, const float* sin_t = nullptr,
                             bool packed = false);

// Attention from a subset of query rows: slot m = b * kmax + r is query token
// q_tok[m] (its row in qkv) at position q_pos[m] of row b; ctx_rows [B*kmax, H].
cudaError_t launch_attention_rows(const bf16* qkv, const int32_t* lengths, const int32_t* q_tok,
                                  const int32_t* q_pos, int B, int S, int kmax, int heads,
                                  int global, int half_window, bool packed, bf16* ctx_rows,
                                  int* err, Launch l);

// tcgen05 attention: tm_qkv maps the projection [rows, 3H] (padded: B*S rows;
// packed: the packed tokens) with a box of 128 rows x 64 columns
// (make_tmap_bf16_2d(..., box_rows = 128)).
cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, const int32_t* lengths, int B, int S,
                                int heads, int global, int half_window, bf16* ctx, int* err,
                                Launch l, bool packed = false);

// ------------------------------------------------------------------ GEMM ---
// kGemmGegluIl: GeGLU with both halves in one 128-row weight tile (rows
// 0..63 the GELU half, 64..127 the gate half of the same 64 output features),
// read from the unchanged [2N, K] weight through a 4-D tensor map
// (make_tmap_geglu_il); persistent plans only, N a multiple of 64.
enum GemmKind : int { kGemmPlain = 0, kGemmResidual = 1, kGemmGeglu = 2, kGemmGegluIl = 3 };

struct GemmPlan {
  int M = 0, N = 0, K = 0, kind = 0;
  int nt = 0;            // tokens per tile (MMA N)
  int token_tiles = 0;   // ceil(M / nt)
  int feat_tiles = 0;    // ceil(N / 128) (kGemmGegluIl: N / 64)
  int splits = 1;        // split-K factor = cluster size along z
  int stages = 0;        // pipeline depth
  bool persistent = false;  // one CTA per SM walks the tiles (splits == 1)
  int pair = 0;  // persistent CTAs in clusters of two sharing an operand tile by TMA multicast:
                 // 1 the token tile (feature-tile pairs), 2 the weight tiles (token-tile pairs);
                 // 3 one cta_group::2 MMA per feature-tile pair, each CTA loading half the tokens
  int grid_ctas = 0;     // persistent: CTAs launched
  size_t workspace_bytes = 0;  // split-K partial tiles (0 when splits == 1)
  int k_blocks = 0;      // K / 64
  uint32_t tmem_cols = 0;
  size_t smem_bytes = 0;
  int ctas() const { return persistent ? grid_ctas : feat_tiles * token_tiles * splits; }
  // rows of the activation box a CTA loads per stage (pair 3: half the token tile)
  int x_box() const { return pair == 3 ? nt / 2 : nt; }
};

// Chooses tile and split for an M x N x K projection; force_* > 0 override.
// Returns false if the shape is unsupported.
bool plan_gemm(int M, int N, int K, int kind, int num_sms, int force_splits, int force_nt,
               GemmPlan* p, bool allow_persistent = true, double split_cost = 2.0);

// A persistent plan run as clusters of two CTAs sharing an operand tile
// (mode 1: the token tile; mode 2: the weight tiles; mode 3: one two-CTA MMA
// per pair of feature tiles, each CTA loading half of the token tile); false
// if the device cannot hold such clusters.
bool make_pair_plan(GemmPlan* p, int mode);

// Distinct plans worth timing for one projection shape (at most max_out):
// the planner's choice under several weights of the split-K overhead, and the
// best plan without split-K.  Returns how many were written.
int plan_candidates(int M, int N, int K, int kind, int num_sms, GemmPlan* out, int max_out);

// Tensor-map encoder (driver entry point resolved through the runtime).
bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t row_stride_bytes, uint32_t box_rows);

// The [2N, K] GeGLU weight (rows [0, N) the GELU half, [N, 2N) the gate) as
// 4-D (k, row in a block of 16, half, block): a box of (64, 16, 2, 4) is the
// 128-row tile of kGemmGegluIl, the 16 GELU rows of a block of features
// followed by its 16 gate rows.  N a multiple of 64.
bool make_tmap_geglu_il(CUtensorMap* m, const void* w, uint64_t N, uint64_t K);

struct GemmOperands {
  CUtensorMap w;       // weights [N, K] (GeGLU: the GELU half; kGemmGegluIl: make_tmap_geglu_il)
  CUtensorMap w2;      // GeGLU gate half [N, K]; unused otherwise
  CUtensorMap x;       // activations [M, K], box rows = plan.nt
  int x_box_rows = 0;  // the box height x was encoded with (plan.x_box()); launch_gemm checks it
  bf16* y = nullptr;   // output [M, N]
  const bf16* residual = nullptr;
  float* y_f32 = nullptr;  // residual kind: fp32 output [M, N] in place of y (16-byte aligned)
  int* err = nullptr;
  float* partials = nullptr;   // split-K workspace (plan.workspace_bytes, 16-byte aligned)
  size_t partials_bytes = 0;
  // plain kind only: rotate output columns [0, rope_cols) as q|k heads of 64
  const float* rope_cos = nullptr;  // [>= rope_S, 32]
  const float* rope_sin = nullptr;
  int rope_S = 0;     // position of token t is t % rope_S
  int rope_cols = 0;  // a multiple of 128
  // LayerNorm on load (non-persistent plans): x maps ln_x, the GEMM computes
  // bf16(LN(ln_x) * ln_gamma) in shared memory, bit-identical to the LN kernel
  const bf16* ln_x = nullptr;
  const bf16* ln_gamma = nullptr;
  float ln_eps = 0.f;
  // packed tokens (packing.cuh): rows [0, sum(len)) of x and y hold the valid
  // tokens of lens_B rows of lens_S; token tiles past them are skipped
  const int32_t* lens = nullptr;
  int lens_B = 0, lens_S = 0;
  const int32_t* rope_pos = nullptr;  // packed tokens: RoPE position of each token
  uint64_t wait_ns = kWaitLimitNs;    // bound of every barrier wait
  bool withhold = false;  // failure-path test: the first CTA never issues its first stage
};

cudaError_t launch_gemm(const GemmPlan& p, const GemmOperands& o, Launch l);

// Graph nodes that write the forward's output: point the captured launch
// (a residual GEMM, or the unpack of packed rows) at new output memory in
// the instantiated graph and its template, in place of old output memory.
// cudaErrorInvalidValue if the node is not such a launch or does not write
// old output memory; the graph is then unchanged.
cudaError_t gemm_node_retarget(cudaGraphExec_t exec, cudaGraphNode_t node, const void* old_y,
                               void* new_y);
cudaError_t unpack_node_retarget(cudaGraphExec_t exec, cudaGraphNode_t node, const void* old_out,
                                 void* new_out);

// Host RoPE table (shared by create() and the op-level entry point).
void rope_table_host(double theta, int max_seq, int half, int bf16_round, float* cos_t,
                     float* sin_t);

int device_sm_count();

}  // namespace laya
