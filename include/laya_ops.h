/*
 * laya_ops.h -- C ABI of the single steps of the Laya encoder forward pass.
 *
 * These are the kernels laya_enc_run composes, exposed one by one so that each
 * can be checked against the CPU oracle at the same BF16 storage points.  All
 * pointers named *_dev or documented as device memory are DEVICE pointers,
 * 16-byte aligned; BF16 tensors are row-major; `stream` is a cudaStream_t.
 * Every call returns 0 or a negative LAYA_E_* code (laya_enc.h); on an
 * argument error nothing is enqueued.  Calls are asynchronous.
 */
#ifndef LAYA_OPS_H_
#define LAYA_OPS_H_

#include <stddef.h>
#include <stdint.h>

#include "laya_enc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Embedding gather + bias-free LayerNorm:
 *   x[t] = bf16( LN(emb[ids[t]]) * gamma ),  LN(v) = (v - mean) / sqrt(var + eps)
 * with mean and variance over the hidden dimension (two passes, fp32).
 * Sources: "Run Laya encoder and decision layers on CUDA", "H800 comparison"
 * (token embedding is part of the timed stack); "perf(model): exact Metal
 * speed-ups of the forward pass - #45" (the encoder has no biases).
 * emb [vocab, H], gamma [H], ids_dev int32 [M], x [M, H].  H a multiple of 256,
 * at most 2048.  An id outside [0, vocab) reads row 0 and sets *err_dev to
 * LAYA_E_DEVICE (err_dev may be NULL). */
int laya_op_embed_layernorm(const void* emb, const void* gamma,
                            const int32_t* ids_dev, int M, int H, int vocab,
                            float eps, void* x, int* err_dev, void* stream);

/* Bias-free LayerNorm of M rows: y[t] = bf16(LN(x[t]) * gamma).  x and y may
 * be the same buffer.  Same source and limits as above. */
int laya_op_layernorm(const void* x, const void* gamma, int M, int H, float eps,
                      void* y, void* stream);

/* Host-side RoPE table, the one laya_enc_create uploads: for position p in
 * [0, max_seq) and pair i in [0, half): angle = p * theta^(-2i / (2 half)) in
 * fp64, cos and sin in fp64, rounded to fp32 and, if bf16 != 0, to BF16 values
 * (kept as fp32).  Layout [max_seq, half] into host arrays.
 * Sources: "[Performance]: Optimize native Rust/CUDA Laya inference #66",
 * "Starting evidence" (separate global and local tables); "Laya native CUDA
 * worker", "Prepare the checkpoint and bundle" (BF16 rounding of the table). */
int laya_op_rope_table(double theta, int max_seq, int half, int bf16,
                       float* cos_host, float* sin_host);

/* RoPE in place on the q and k slices of a packed projection qkv [B*S, 3H]
 * (q at columns [0, H), k at [H, 2H), v untouched), head n at columns n*D.
 * Pairs (i, i + D/2); position of token (b, s) is s:
 *   y_i = bf16(x_i c - x_{i+D/2} s),  y_{i+D/2} = bf16(x_{i+D/2} c + x_i s)
 * with each product and the sum rounded to fp32 separately (no FMA).
 * cos_dev, sin_dev: fp32 [>= S, D/2] device tables, 16-byte aligned.  A
 * (half-dim, head, row) grid with 32-bit indices: one thread per (8 pairs,
 * head, token), 16-byte loads and stores; heads <= 32.
 * Sources: "[RFC]: Native Laya inference with Rust and CUDA #14", "Design"
 * (separate QKV, RoPE and attention launches); "perf(model): exact Metal
 * speed-ups of the forward pass - #45" (a (half-dim, head, row) grid with
 * 32-bit indices).  head_dim must be 64. */
int laya_op_rope(void* qkv, const float* cos_dev, const float* sin_dev, int B,
                 int S, int heads, int head_dim, void* stream);

/* Softmax attention per (row b, head n):
 *   ctx_i = sum_j softmax_j(q_i . k_j / sqrt(D)) v_j
 * over keys j < lengths[b] and, if global == 0, |i - j| <= half_window.
 * A query with no visible key gets ctx = 0.  Query tiles that lie wholly in
 * the padding of their row are written as 0 (padded positions carry no
 * meaning).  qkv [B*S, 3H] as above (after RoPE), lengths_dev int32 [B] with
 * values in [1, S], ctx [B*S, H] BF16 written as [B, S, heads*D] (no
 * transpose).  Sources: "perf(model): exact Metal speed-ups of the forward
 * pass - #45" (one (b,1,1,s) key-padding row broadcast over every query;
 * output written with (b, s, h, hd) strides); "Run Laya encoder and decision
 * layers on CUDA", "Test Result" (empty-key padding rows).  head_dim 64. */
int laya_op_attention(const void* qkv, const int32_t* lengths_dev, int B, int S,
                      int heads, int head_dim, int global, int half_window,
                      void* ctx, void* stream);

/* laya_op_attention from a subset of query rows ("perf(model): exact Metal
 * speed-ups of the forward pass - #45": attention over a subset of query rows
 * gets its own entry point; the marker-row last layer attends from the marker
 * rows only, with the (b, 1, 1, s) key-padding row of its batch row broadcast
 * over them).  Slot m = b * kmax + r (r < kmax) is query token q_tok_dev[m] (a
 * row of qkv, normally b * S + q_pos_dev[m]) at position q_pos_dev[m] of row
 * b (the window's reference on local layers); keys and values are row b's
 * tokens below lengths[b].  qkv [B*S, 3H] and lengths_dev as for
 * laya_op_attention; q_tok_dev, q_pos_dev: DEVICE int32 [B*kmax]; ctx_rows:
 * DEVICE BF16 [B*kmax, H], slot m's context.  B * kmax <=
 * LAYA_ENC_MAX_MARKERS.  Same arithmetic as laya_op_attention (mma.sync
 * tiles, key tiles in the same order), so a slot's context equals that
 * kernel's context of the same query row bit for bit. */
int laya_op_attention_rows(const void* qkv, const int32_t* lengths_dev,
                           const int32_t* q_tok_dev, const int32_t* q_pos_dev, int B,
                           int S, int kmax, int heads, int head_dim, int global,
                           int half_window, void* ctx_rows, void* stream);

/* laya_op_attention on the 5th-generation tensor cores: S = Q K^T and O = P V
 * by tcgen05.mma with fp32 accumulators in tensor memory, one CTA per 128
 * queries of one head and row with warp-specialised roles (TMA, MMA issue,
 * softmax), Q/K/V tiles brought in by TMA.  Same arguments, layouts, mask and
 * results contract as laya_op_attention; P is rounded to BF16 for the P V
 * product (the row sums are not).  qkv must be 16-byte aligned with B*S rows
 * of 3*heads*64 BF16 values.  Returns LAYA_E_INVAL for bad arguments,
 * LAYA_E_CUDA when the launch fails.
 * Sources: as laya_op_attention. */
int laya_op_attention_tc(const void* qkv, const int32_t* lengths_dev, int B, int S,
                         int heads, int head_dim, int global, int half_window,
                         void* ctx, void* stream);

/* RoPE and attention in one kernel: the q and k of each tile are rotated in
 * shared memory (same arithmetic as laya_op_rope, bit-identical values) and
 * attended as in laya_op_attention; qkv in memory is not modified.  cos_dev,
 * sin_dev: fp32 [>= S, 32] device tables.  (laya_enc_run rotates q and k once,
 * in the QKV projection's epilogue, instead: every K tile would otherwise be
 * rotated once per query tile.)
 * Sources: as laya_op_rope and laya_op_attention. */
int laya_op_attention_rope(const void* qkv, const int32_t* lengths_dev,
                           const float* cos_dev, const float* sin_dev, int B,
                           int S, int heads, int head_dim, int global,
                           int half_window, void* ctx, void* stream);

/* Linear projection on the tensor cores (tcgen05, TMEM accumulators, TMA):
 *   a = x . w^T  (x [M, K], w [N_w, K] in nn.Linear layout, fp32 accumulate)
 * kind 0 (plain):    y [M, N] = bf16(a),             N_w = N
 * kind 1 (residual): y [M, N] = bf16(residual + a),  N_w = N; residual may be y
 * kind 2 (GeGLU):    y [M, N] = bf16(gelu(a[:, :N]) * a[:, N:]), N_w = 2N,
 *                    gelu(z) = z/2 (1 + erf(z / sqrt 2))
 * kind 3 (GeGLU, interleaved tiles): the kind 2 result bit for bit, from the
 *                    same w, computed with 64 rows of each half in one
 *                    128-row weight tile (one MMA per K step); N a multiple
 *                    of 64, unsplit plans only (splits <= 1)
 * K a multiple of 64; N a multiple of 8.  splits <= 0 and tile_tokens <= 0
 * pick the library's plan; positive values force them (tile_tokens a multiple
 * of 16, at most 256; splits at most 16 and at most K/64).  workspace: device
 * scratch of at least laya_op_linear_workspace_size() bytes, 16-byte aligned,
 * caller-owned (NULL allowed when that size is 0): split-K writes its fp32
 * partial tiles there and the CTAs of each cluster sum them in split order,
 * so results do not depend on timing.  The contents need no initialisation
 * and are garbage afterwards; concurrent calls must not share it.
 * Sources: "[Performance]: Optimize native Rust/CUDA Laya inference #66",
 * "Implementation priorities" (the four encoder GEMMs; small tiles for short
 * sequences, preserving fp32 accumulation and BF16 rounding); "[RFC]: Native
 * Laya inference with Rust and CUDA #14" (fused GEMM epilogues). */
int laya_op_linear(const void* x, int M, int K, const void* w, int N, int kind,
                   const void* residual, void* y, void* workspace,
                   size_t workspace_bytes, int splits, int tile_tokens,
                   void* stream);

/* laya_op_linear with the choice of the persistent kernel's pairing (splits
 * must be 1 when paired != 0): the one-CTA-per-SM kernel runs in clusters of
 * two CTAs that share one operand tile of every pipeline stage, read from L2
 * once and multicast by TMA into both (halving the L2-to-SM traffic of that
 * operand).  paired = 1: the two CTAs take the two feature tiles of a pair
 * with the same token tile (the token tile is shared); paired = 2: the two
 * token tiles of a pair with the same feature tile (the weight tiles are
 * shared); paired = 3: the pair computes one 256-feature tile with one
 * two-CTA MMA (tcgen05 cta_group::2), each CTA loading its 128 weight rows
 * and half of the token tile.  laya_enc_run's first run of a shape may pick
 * any of them by timing.  Same arithmetic and results as paired = 0, bit for
 * bit.
 * LAYA_E_UNSUPPORTED if the device cannot hold such clusters.
 * Sources: as laya_op_linear. */
int laya_op_linear_ex(const void* x, int M, int K, const void* w, int N, int kind,
                      const void* residual, void* y, void* workspace,
                      size_t workspace_bytes, int splits, int tile_tokens, int paired,
                      void* stream);

/* Workspace bytes laya_op_linear (and the _ln / _rope forms) need for this
 * shape and plan; 0 when the plan does not split K. */
int laya_op_linear_workspace_size(int M, int K, int N, int kind, int splits,
                                  int tile_tokens, size_t* bytes);

/* A projection whose input is LayerNorm'd on load: the GEMM reads rows of
 * x_raw [M, K] and computes h = bf16(LN(x_raw) * gamma) in shared memory with
 * exactly the arithmetic of laya_op_layernorm, so y equals laya_op_layernorm
 * followed by laya_op_linear bit for bit; kinds as laya_op_linear.  The
 * split-K kernel is used (laya_enc_run launches its norms as separate
 * kernels).  K a multiple of 256, at most 2048.  Sources: as laya_op_layernorm and
 * laya_op_linear. */
int laya_op_linear_ln(const void* x_raw, const void* gamma, float eps, int M,
                      int K, const void* w, int N, int kind,
                      const void* residual, void* y, void* workspace,
                      size_t workspace_bytes, int splits, int tile_tokens,
                      void* stream);

/* The QKV projection as laya_enc_run runs it: kind 0 (plain) with RoPE
 * applied in the epilogue to output columns [0, rope_cols) (the q and k heads
 * of 64): each value is rounded to BF16 as the plain projection stores it,
 * then rotated with exactly the arithmetic of laya_op_rope at position
 * token % S, so y equals laya_op_linear followed by laya_op_rope bit for bit.
 * rope_cols a multiple of 128 and at most N; cos_dev, sin_dev fp32 [>= S, 32].
 * Sources: as laya_op_linear and laya_op_rope. */
int laya_op_linear_rope(const void* x, int M, int K, const void* w, int N,
                        const float* cos_dev, const float* sin_dev, int S,
                        int rope_cols, void* y, void* workspace,
                        size_t workspace_bytes, int splits, int tile_tokens,
                        void* stream);

/* laya_op_linear for callers that cannot allocate device memory.  The pages
 * have no counterpart: this entry point exists for library users who must not
 * call cudaMalloc (code under a device-memory budget owned by a host
 * framework, or latency-critical loops where an allocation could synchronise
 * the device) and cannot keep a workspace of their own.  Same arguments and
 * results as laya_op_linear, minus the workspace: split-K partial tiles go to
 * a fixed 16 MiB device array inside the library (every GPU that loads the
 * library holds it until the process exits).  A plan needing more than that
 * (laya_op_linear_workspace_size > 16 MiB) is rejected with LAYA_E_INVAL and
 * nothing is enqueued.  The first call on a device looks the array's address
 * up (cudaGetSymbolAddress) and keeps it: make that first call before any
 * stream capture.  All calls share the array and it keeps the last call's
 * contents (nothing in it needs to start at zero); calls whose kernels
 * overlap on the GPU race.  Allocates nothing: no cudaMalloc or cudaFree. */
int laya_op_linear_noalloc(const void* x, int M, int K, const void* w, int N,
                           int kind, const void* residual, void* y, int splits,
                           int tile_tokens, void* stream);

/* The plan laya_op_linear picks by default: tokens per tile, split-K factor
 * and the number of CTAs (feature tiles x token tiles x splits) on a device
 * with num_sms SMs.  Host-only. */
int laya_op_linear_plan(int M, int K, int N, int kind, int num_sms,
                        int* tile_tokens, int* splits, int* ctas);

#ifdef __cplusplus
}
#endif

#endif /* LAYA_OPS_H_ */
