// ops_abi.cu -- the single-step entry points declared in laya_ops.h.  They
// validate arguments on the host and launch the same kernels laya_enc_run
// uses; nothing here computes on the CPU.
#include <cstring>

#include "../../include/laya_ops.h"
#include "internal.h"

using laya::bf16;

namespace {

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int rc_of(cudaError_t e) { return e == cudaSuccess ? LAYA_OK : LAYA_E_CUDA; }

}  // namespace

extern "C" {

int laya_op_embed_layernorm(const void* emb, const void* gamma, const int32_t* ids_dev, int M,
                            int H, int vocab, float eps, void* x, int* err_dev, void* stream) {
  if (!al16(emb) || !al16(gamma) || !ids_dev || !al16(x) || M < 1 || vocab < 1 ||
      !laya::rowops_supported_hidden(H) || !(eps > 0.f))
    return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_embed_layernorm(static_cast<const bf16*>(emb),
                                            static_cast<const bf16*>(gamma), ids_dev, M, H, vocab,
                                            eps, static_cast<bf16*>(x), err_dev, l));
}

int laya_op_layernorm(const void* x, const void* gamma, int M, int H, float eps, void* y,
                      void* stream) {
  if (!al16(x) || !al16(gamma) || !al16(y) || M < 1 || !laya::rowops_supported_hidden(H) ||
      !(eps > 0.f))
    return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_layernorm(static_cast<const bf16*>(x), static_cast<const bf16*>(gamma),
                                      M, H, eps, static_cast<bf16*>(y), l));
}

int laya_op_rope_table(double theta, int max_seq, int half, int bf16_round, float* cos_host,
                       float* sin_host) {
  if (!(theta > 0.0) || max_seq < 1 || half < 1 || !cos_host || !sin_host) return LAYA_E_INVAL;
  laya::rope_table_host(theta, max_seq, half, bf16_round ? 1 : 0, cos_host, sin_host);
  return LAYA_OK;
}

int laya_op_rope(void* qkv, const float* cos_dev, const float* sin_dev, int B, int S, int heads,
                 int head_dim, void* stream) {
  if (!al16(qkv) || !al16(cos_dev) || !al16(sin_dev) || B < 1 || S < 1 || heads < 1 ||
      heads > 32 || head_dim != 64)
    return LAYA_E_INVAL;
  if (static_cast<long long>(B) * S > 0x7fffffffLL) return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_rope(static_cast<bf16*>(qkv), cos_dev, sin_dev, B, S, heads, l));
}

int laya_op_attention(const void* qkv, const int32_t* lengths_dev, int B, int S, int heads,
                      int head_dim, int global, int half_window, void* ctx, void* stream) {
  if (!al16(qkv) || !lengths_dev || !al16(ctx) || B < 1 || S < 1 || heads < 1 ||
      head_dim != 64 || half_window < 0 || B > 65535 || heads > 65535)
    return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_attention(static_cast<const bf16*>(qkv), lengths_dev, B, S, heads,
                                      global ? 1 : 0, half_window, static_cast<bf16*>(ctx),
                                      nullptr, l));
}

int laya_op_attention_rows(const void* qkv, const int32_t* lengths_dev, const int32_t* q_tok_dev,
                           const int32_t* q_pos_dev, int B, int S, int kmax, int heads,
                           int head_dim, int global, int half_window, void* ctx_rows,
                           void* stream) {
  if (!al16(qkv) || !lengths_dev || !q_tok_dev || !q_pos_dev || !al16(ctx_rows) || B < 1 ||
      S < 1 || kmax < 1 || static_cast<long long>(B) * kmax > LAYA_ENC_MAX_MARKERS || heads < 1 ||
      head_dim != 64 || half_window < 0 || heads > 65535)
    return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_attention_rows(static_cast<const bf16*>(qkv), lengths_dev, q_tok_dev,
                                           q_pos_dev, B, S, kmax, heads, global ? 1 : 0,
                                           half_window, false, static_cast<bf16*>(ctx_rows),
                                           nullptr, l));
}

int laya_op_attention_tc(const void* qkv, const int32_t* lengths_dev, int B, int S, int heads,
                         int head_dim, int global, int half_window, void* ctx, void* stream) {
  if (!al16(qkv) || !lengths_dev || !al16(ctx) || B < 1 || S < 1 || heads < 1 ||
      head_dim != 64 || half_window < 0 || B > 65535 || heads > 65535)
    return LAYA_E_INVAL;
  CUtensorMap tm;
  const uint64_t cols = 3ull * heads * 64;
  if (!laya::make_tmap_bf16_2d(&tm, qkv, static_cast<uint64_t>(B) * S, cols, cols * 2, 128))
    return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_attention_tc(tm, lengths_dev, B, S, heads, global ? 1 : 0, half_window,
                                         static_cast<bf16*>(ctx), nullptr, l));
}

int laya_op_attention_rope(const void* qkv, const int32_t* lengths_dev, const float* cos_dev,
                           const float* sin_dev, int B, int S, int heads, int head_dim, int global,
                           int half_window, void* ctx, void* stream) {
  if (!al16(qkv) || !lengths_dev || !cos_dev || !sin_dev || !al16(ctx) || B < 1 || S < 1 ||
      heads < 1 || head_dim != 64 || half_window < 0 || B > 65535 || heads > 65535)
    return LAYA_E_INVAL;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_attention(static_cast<const bf16*>(qkv), lengths_dev, B, S, heads,
                                      global ? 1 : 0, half_window, static_cast<bf16*>(ctx),
                                      nullptr, l, cos_dev, sin_dev));
}

int laya_op_linear_plan(int M, int K, int N, int kind, int num_sms, int* tile_tokens,
                        int* splits, int* ctas) {
  laya::GemmPlan p;
  if (!laya::plan_gemm(M, N, K, kind, num_sms, 0, 0, &p)) return LAYA_E_INVAL;
  if (tile_tokens) *tile_tokens = p.nt;
  if (splits) *splits = p.splits;
  if (ctas) *ctas = p.ctas();
  return LAYA_OK;
}

int laya_op_linear_workspace_size(int M, int K, int N, int kind, int splits, int tile_tokens,
                                  size_t* bytes) {
  laya::GemmPlan p;
  if (!bytes || !laya::plan_gemm(M, N, K, kind, laya::device_sm_count(), splits, tile_tokens, &p))
    return LAYA_E_INVAL;
  *bytes = p.workspace_bytes;
  return LAYA_OK;
}

int laya_op_linear(const void* x, int M, int K, const void* w, int N, int kind,
                   const void* residual, void* y, void* workspace, size_t workspace_bytes,
                   int splits, int tile_tokens, void* stream) {
  return laya_op_linear_ex(x, M, K, w, N, kind, residual, y, workspace, workspace_bytes, splits,
                           tile_tokens, 0, stream);
}

int laya_op_linear_ex(const void* x, int M, int K, const void* w, int N, int kind,
                      const void* residual, void* y, void* workspace, size_t workspace_bytes,
                      int splits, int tile_tokens, int paired, void* stream) {
  if (!al16(x) || !al16(w) || !al16(y)) return LAYA_E_INVAL;
  if (kind == laya::kGemmResidual && !al16(residual)) return LAYA_E_INVAL;
  if (paired < 0 || paired > 3 || (paired && splits != 1)) return LAYA_E_INVAL;
  laya::GemmPlan p;
  if (!laya::plan_gemm(M, N, K, kind, laya::device_sm_count(), splits, tile_tokens, &p))
    return LAYA_E_INVAL;
  if (paired && !laya::make_pair_plan(&p, paired)) return LAYA_E_UNSUPPORTED;
  laya::GemmOperands o;
  const uint64_t ldk = static_cast<uint64_t>(K) * 2;
  bool ok = laya::make_tmap_bf16_2d(&o.x, x, M, K, ldk, static_cast<uint32_t>(p.x_box()));
  if (kind == laya::kGemmGegluIl) {
    ok = ok && laya::make_tmap_geglu_il(&o.w, w, N, K);
    o.w2 = o.w;
  } else {
    ok = ok && laya::make_tmap_bf16_2d(&o.w, w, N, K, ldk, 128);
    if (kind == laya::kGemmGeglu) {
      const char* gate = static_cast<const char*>(w) + static_cast<size_t>(N) * K * 2;
      ok = ok && laya::make_tmap_bf16_2d(&o.w2, gate, N, K, ldk, 128);
    } else {
      o.w2 = o.w;
    }
  }
  if (!ok) return LAYA_E_INVAL;
  o.x_box_rows = p.x_box();
  o.y = static_cast<bf16*>(y);
  o.residual = static_cast<const bf16*>(residual);
  o.err = nullptr;
  if (p.workspace_bytes > workspace_bytes || (p.workspace_bytes && !al16(workspace)))
    return LAYA_E_INVAL;
  o.partials = static_cast<float*>(workspace);
  o.partials_bytes = workspace_bytes;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_gemm(p, o, l));
}

int laya_op_linear_ln(const void* x_raw, const void* gamma, float eps, int M, int K, const void* w,
                      int N, int kind, const void* residual, void* y, void* workspace,
                      size_t workspace_bytes, int splits, int tile_tokens, void* stream) {
  if (!al16(x_raw) || !al16(gamma) || !al16(w) || !al16(y) || !(eps > 0.f) || K % 256 != 0 ||
      K > 2048)
    return LAYA_E_INVAL;
  if (kind == laya::kGemmResidual && !al16(residual)) return LAYA_E_INVAL;
  laya::GemmPlan p;
  if (!laya::plan_gemm(M, N, K, kind, laya::device_sm_count(), splits, tile_tokens, &p, false))
    return LAYA_E_INVAL;
  laya::GemmOperands o;
  const uint64_t ldk = static_cast<uint64_t>(K) * 2;
  bool ok = laya::make_tmap_bf16_2d(&o.w, w, N, K, ldk, 128) &&
            laya::make_tmap_bf16_2d(&o.x, x_raw, M, K, ldk, static_cast<uint32_t>(p.nt));
  if (kind == laya::kGemmGeglu) {
    const char* gate = static_cast<const char*>(w) + static_cast<size_t>(N) * K * 2;
    ok = ok && laya::make_tmap_bf16_2d(&o.w2, gate, N, K, ldk, 128);
  } else {
    o.w2 = o.w;
  }
  if (!ok) return LAYA_E_INVAL;
  o.x_box_rows = p.x_box();
  o.y = static_cast<bf16*>(y);
  o.residual = static_cast<const bf16*>(residual);
  o.ln_x = static_cast<const bf16*>(x_raw);
  o.ln_gamma = static_cast<const bf16*>(gamma);
  o.ln_eps = eps;
  if (p.workspace_bytes > workspace_bytes || (p.workspace_bytes && !al16(workspace)))
    return LAYA_E_INVAL;
  o.partials = static_cast<float*>(workspace);
  o.partials_bytes = workspace_bytes;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_gemm(p, o, l));
}

int laya_op_linear_rope(const void* x, int M, int K, const void* w, int N, const float* cos_dev,
                        const float* sin_dev, int S, int rope_cols, void* y, void* workspace,
                        size_t workspace_bytes, int splits, int tile_tokens, void* stream) {
  if (!al16(x) || !al16(w) || !al16(y) || !cos_dev || !sin_dev || S < 1 || S > 65535 ||
      rope_cols < 0 || rope_cols % 128 != 0 || rope_cols > N)
    return LAYA_E_INVAL;
  laya::GemmPlan p;
  if (!laya::plan_gemm(M, N, K, laya::kGemmPlain, laya::device_sm_count(), splits, tile_tokens,
                       &p))
    return LAYA_E_INVAL;
  laya::GemmOperands o;
  const uint64_t ldk = static_cast<uint64_t>(K) * 2;
  if (!laya::make_tmap_bf16_2d(&o.w, w, N, K, ldk, 128) ||
      !laya::make_tmap_bf16_2d(&o.x, x, M, K, ldk, static_cast<uint32_t>(p.nt)))
    return LAYA_E_INVAL;
  o.w2 = o.w;
  o.x_box_rows = p.x_box();
  o.y = static_cast<bf16*>(y);
  o.rope_cos = cos_dev;
  o.rope_sin = sin_dev;
  o.rope_S = S;
  o.rope_cols = rope_cols;
  if (p.workspace_bytes > workspace_bytes || (p.workspace_bytes && !al16(workspace)))
    return LAYA_E_INVAL;
  o.partials = static_cast<float*>(workspace);
  o.partials_bytes = workspace_bytes;
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return rc_of(laya::launch_gemm(p, o, l));
}

}  // extern "C"
