/*
 * laya_enc.h -- C ABI of the Laya BF16 encoder forward pass on one GB300 (sm_103a).
 *
 * The library runs token embedding, the encoder layers and the decision layers
 * of a bidirectional transformer encoder over a right-padded batch of rows
 * (at most max_batch rows of at most max_seq tokens, with per-row lengths used
 * as a key-padding mask) and leaves the final hidden states in a caller-owned
 * device buffer.
 *
 * Sources for the operation:
 *  - "Run Laya encoder and decision layers on CUDA" (PR #49), sections
 *    "Purpose" and "H800 comparison": embedding + 28 encoder layers + 2
 *    decision transformer layers, hidden states left on the GPU.
 *  - "[RFC]: Native Laya inference with Rust and CUDA #14", section "Design"
 *    and the C-ABI discussion under "Activity": an ABI version call, int
 *    return codes, work queued on a caller-supplied stream so that it can be
 *    captured in a CUDA Graph; per-shape graph capture and replay with an LRU
 *    cache of at most four shapes and 512 MiB of workspaces.
 *  - "Laya native CUDA worker", section "Start and check": at most 16 rows and
 *    512 tokens per row; invalid input is a client error; a native failure
 *    stops the executor.
 *  - "[Performance]: Optimize native Rust/CUDA Laya inference #66", section
 *    "Implementation priorities": group uploads and keep safe host-buffer
 *    lifetimes.
 * The per-layer arithmetic (pre-norm layers, GeGLU MLP, rotate-half RoPE with
 * separate global and local tables, local layers with a sliding window) is the
 * same definition as the CPU oracle of this repository; see laya_ops.h for
 * each step.
 *
 * Conventions.  Every function returns 0 on success and a negative LAYA_E_*
 * code on failure.  On an argument error nothing is enqueued and the output
 * buffer is untouched.  Device pointers must be 16-byte aligned.  A handle is
 * not thread-safe: calls on one handle must be serialised by the caller.
 */
#ifndef LAYA_ENC_H_
#define LAYA_ENC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LAYA_ENC_ABI_VERSION 3

/* Error codes (negative). */
#define LAYA_OK 0
#define LAYA_E_INVAL (-1)       /* bad argument or configuration */
#define LAYA_E_NOMEM (-2)       /* device or pinned host allocation failed */
#define LAYA_E_CUDA (-3)        /* a CUDA call failed; the handle is poisoned */
#define LAYA_E_POISONED (-4)    /* the handle saw an earlier CUDA/device error */
#define LAYA_E_UNSUPPORTED (-5) /* device is not compute capability 10.3 */
#define LAYA_E_DEVICE (-6)      /* a kernel reported an error (bounded wait expired,
                                   id out of range); the handle is poisoned */

/* Model shape.  Plain old data; all fields must be set.
 * Full model: hidden 1024, heads 16, head_dim 64, intermediate 2624,
 * vocab 50368, 28 encoder + 2 decision layers, global_every 3,
 * local_half_window 64, theta_global 160000, theta_local 10000, ln_eps 1e-5,
 * max_batch 16, max_seq 512, rope_table_bf16 1, first_attn_norm_identity 1,
 * final_norm 1, out_fp32 0.
 * Supported: hidden a multiple of 256 and at most 2048, head_dim 64,
 * heads * head_dim == hidden, intermediate a multiple of 64,
 * max_seq <= 512, max_batch <= 16. */
typedef struct {
  int32_t hidden, heads, head_dim, intermediate, vocab;
  int32_t n_encoder_layers, n_decision_layers;
  int32_t global_every;      /* encoder layer l is global iff l % global_every == 0;
                                decision layers are always global */
  int32_t local_half_window; /* local layers: query i sees key j iff |i - j| <= this */
  float theta_global, theta_local, ln_eps;
  int32_t max_batch, max_seq;
  int32_t rope_table_bf16;          /* 1: RoPE table values rounded to BF16 (kept fp32) */
  int32_t first_attn_norm_identity; /* 1: encoder layer 0 projects x without LayerNorm */
  int32_t final_norm;               /* 1: LayerNorm after the last encoder layer */
  int32_t out_fp32; /* 0: out_hidden is BF16.  1 (parity mode): out_hidden is
                       fp32 and receives the last residual sum of the last
                       layer before its BF16 rounding (every earlier storage
                       point unchanged), so that tolerances on the final hidden
                       states ("[Performance]: Optimize native Rust/CUDA Laya
                       inference #66", "Starting evidence") can be read
                       without that last rounding.  Rounding this output to
                       BF16 gives the out_fp32 = 0 result bit for bit. */
} laya_enc_config;

/* Per-layer weights: device pointers to BF16 data in nn.Linear layout
 * [out_features, in_features], row-major.  Caller-owned; they must stay valid
 * and unchanged until laya_enc_destroy. */
typedef struct {
  const void* attn_norm; /* [hidden]; NULL at encoder layer 0 when
                            first_attn_norm_identity is set */
  const void* wqkv;      /* [3*hidden, hidden]: rows q | k | v, head-major inside */
  const void* wo;        /* [hidden, hidden] */
  const void* mlp_norm;  /* [hidden] */
  const void* wup;       /* [2*intermediate, hidden]: rows [0, I) go through
                            GELU, rows [I, 2I) are the gate */
  const void* wdown;     /* [hidden, intermediate] */
} laya_enc_layer_weights;

typedef struct {
  const void* tok_emb;    /* [vocab, hidden] */
  const void* emb_norm;   /* [hidden] */
  const void* final_norm; /* [hidden] (may be NULL if final_norm == 0) */
  int32_t n_layers;       /* must equal n_encoder_layers + n_decision_layers */
  const laya_enc_layer_weights* layers; /* host array of n_layers entries */
} laya_enc_weights;

typedef struct laya_enc_handle laya_enc_handle;

/* Returns LAYA_ENC_ABI_VERSION. */
int laya_enc_abi_version(void);

/* Validates the configuration without touching a GPU.  0 or LAYA_E_INVAL. */
int laya_enc_validate_config(const laya_enc_config* cfg);

/* Creates a handle on the current CUDA device: checks the device (10.3),
 * builds the global and local RoPE tables on the host and uploads them, and
 * builds TMA descriptors over the caller's weights (no weight copy).
 * Switches read from the environment here: LAYA_EAGER=1 (no CUDA Graphs),
 * LAYA_NO_PDL=1 (no programmatic dependent launch), LAYA_NO_TUNE=1 (see
 * laya_enc_run), LAYA_ATTN_MMA_SYNC=1 (attention on the mma.sync kernel
 * instead of the tcgen05 one).  Results stay within the same tolerances
 * under each of them.
 * *out is set to NULL on failure. */
int laya_enc_create(const laya_enc_config* cfg, const laya_enc_weights* weights,
                    laya_enc_handle** out);

/* Runs the forward pass on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  token_ids: HOST int32 [batch * seq], row-major;
 * lengths: HOST int32 [batch], each in [1, seq], positions >= length are
 * padding.  out_hidden: DEVICE BF16 [batch, seq, hidden] (fp32 when
 * cfg.out_fp32), caller-owned;
 * valid positions receive the final hidden states, padded positions receive
 * finite values of no meaning.  The host arrays are copied into library-owned
 * pinned memory before the call returns and may be reused at once.  The call
 * is asynchronous; synchronise `stream` before reading out_hidden.
 * The first call of a (batch, seq) shape allocates its workspace, times the
 * candidate plans of each projection once per process (unless env
 * LAYA_NO_TUNE=1; env LAYA_PLAN_CACHE=<file> keeps the chosen plans in a text
 * file that later processes read instead of timing again; the file is not
 * locked: processes sharing one file at the same time may each time a shape,
 * the last writer's lines stand, and reading stops at the first line that
 * does not parse), runs two eager
 * warm-up passes and captures a CUDA Graph (unless graphs are off); later
 * calls replay it.  If `stream` is itself capturing, the kernels are launched
 * into the caller's capture instead. */
int laya_enc_run(laya_enc_handle* h, const int32_t* token_ids,
                 const int32_t* lengths, int batch, int seq, void* out_hidden,
                 void* stream);

/* Most marker slots one laya_enc_run_markers call takes ("Laya native CUDA
 * worker", "Start and check": at most 2048 markers per request). */
#define LAYA_ENC_MAX_MARKERS 2048

/* The forward pass with the last layer at marker rows only ("perf(model):
 * exact Metal speed-ups of the forward pass - #45": only the marker positions
 * reach the scorer; keys and values need every position, but everything after
 * them is row-wise and attention is independent per query row, so the last
 * layer attends from, projects and runs its MLP on the batch * kmax marker
 * rows alone).  token_ids, lengths: as laya_enc_run (HOST).  marker_pos: HOST
 * int32 [batch * kmax]; marker_pos[b * kmax + j] is a position in [0,
 * lengths[b]) of row b, or -1 for an empty slot.  out_markers: DEVICE BF16
 * [batch * kmax, hidden] (fp32 when cfg.out_fp32), caller-owned; slot
 * b * kmax + j receives the final hidden state of token (b, marker_pos), the
 * value laya_enc_run leaves at out_hidden[b, marker_pos] up to the order of
 * fp32 sums in the last layer's projections; empty slots receive finite values
 * of no meaning.  batch * kmax <= LAYA_ENC_MAX_MARKERS; a marker on padding
 * (>= lengths[b]) or below -1 is LAYA_E_INVAL.  The workspace and graph cache
 * is keyed by (batch, seq, kmax).  Otherwise as laya_enc_run. */
int laya_enc_run_markers(laya_enc_handle* h, const int32_t* token_ids,
                         const int32_t* lengths, int batch, int seq,
                         const int32_t* marker_pos, int kmax, void* out_markers,
                         void* stream);

/* As laya_enc_run, with token_ids and lengths in DEVICE memory (int32, same
 * layouts).  Ids cannot be checked on the host: an out-of-range id or length
 * is clamped by the kernels and reported as LAYA_E_DEVICE by laya_enc_check. */
int laya_enc_run_device(laya_enc_handle* h, const int32_t* token_ids_dev,
                        const int32_t* lengths_dev, int batch, int seq,
                        void* out_hidden, void* stream);

/* Synchronises `stream` and reads the device error word.  Returns 0, or
 * LAYA_E_DEVICE (and poisons the handle) if a kernel flagged an error. */
int laya_enc_check(laya_enc_handle* h, void* stream);

/* Test hook for the failure path: the next laya_enc_run / laya_enc_run_device
 * on this handle enqueues nothing and fails with LAYA_E_CUDA as a failed
 * launch would, poisoning the handle ("Laya native CUDA worker", "Start and
 * check": a native failure stops the executor); later calls return
 * LAYA_E_POISONED.  No device fault is involved. */
int laya_enc_debug_fail_next_run(laya_enc_handle* h);

/* Test hooks for the device-side failure path ("Laya native CUDA worker",
 * "Start and check": a native failure stops the executor).  Every wait of a
 * kernel on a barrier is bounded; when one runs out, the kernel raises its
 * CTA's abort flag and the device error word, every role of the CTA leaves
 * its loop, the copies and tensor-core products in flight are waited for and
 * tensor memory is released, so the kernel returns and the context stays
 * usable; laya_enc_check then returns LAYA_E_DEVICE and poisons the handle.
 * set_wait_limit_ns: the bound of the projections' barrier waits, in [1 ms,
 * 10 s]; 0 restores the default of 2 s.
 * withhold_next_run: in the next laya_enc_run / _run_device on this handle
 * (launched eagerly), the first CTA of the first projection never issues the
 * copy of its first pipeline stage, so the wait for that stage runs out after
 * the limit.  No trap, no fault, no invalid access is involved. */
int laya_enc_debug_set_wait_limit_ns(laya_enc_handle* h, uint64_t ns);
int laya_enc_debug_withhold_next_run(laya_enc_handle* h);

/* 1: use CUDA Graphs (default, unless env LAYA_EAGER=1); 0: eager launches. */
int laya_enc_set_graphs(laya_enc_handle* h, int enabled);

/* The per-shape workspace and CUDA Graph cache ("[RFC]: Native Laya inference
 * with Rust and CUDA #14", "Design": capture per shape, replay, an LRU of at
 * most four shapes and 512 MiB of workspaces).  The first run of a shape
 * allocates its workspace (evicting least-recently-used shapes until both
 * bounds hold, after waiting for their last forward), runs two eager warm-up
 * passes and captures a graph.  A later run of a captured shape with a
 * different out_hidden re-points the graph's last launch (the one writing
 * out_hidden) instead of capturing again.  Counters since create; times are
 * host wall-clock. */
typedef struct {
  int32_t shapes;       /* workspaces resident now (<= max_shapes) */
  int32_t max_shapes;   /* 4 */
  uint64_t bytes;       /* device bytes they hold (<= max_bytes) */
  uint64_t max_bytes;   /* 512 MiB */
  uint64_t created;     /* workspaces allocated */
  uint64_t evicted;     /* workspaces freed to make room */
  uint64_t captures;    /* graphs captured and instantiated */
  uint64_t retargets;   /* graphs re-pointed at a new out_hidden */
  double setup_ms;      /* time spent creating workspaces */
  double capture_ms;    /* time spent in first-run warm-ups, captures and
                           instantiations */
} laya_enc_cache_stats;

int laya_enc_get_cache_stats(const laya_enc_handle* h, laya_enc_cache_stats* out);

/* Number of kernel launches one forward pass of this shape makes. */
int laya_enc_launch_count(const laya_enc_handle* h, int batch, int seq);

/* The projection plans in use for a (batch, seq) shape that has a workspace
 * (after its first run, which times the candidate plans): for QKV, out-proj,
 * up and down in turn, five values each into out[20]: tokens per tile,
 * split-K factor, pairing (0 none, 1 CTA pairs sharing the token tile, 2
 * sharing the weight tiles), CTAs launched, and the kernel kind as
 * laya_op_linear numbers it (the up-projection: 2, or 3 for the interleaved
 * weight tiles).  LAYA_E_INVAL if the shape has no workspace. */
int laya_enc_get_plans(const laya_enc_handle* h, int batch, int seq, int32_t* out);

/* Bytes of device workspace a (batch, seq) shape uses (activations, split-K
 * partials, staging). */
int laya_enc_workspace_bytes(const laya_enc_handle* h, int batch, int seq,
                             size_t* bytes);

/* Kernel classes reported by the profiling calls below. */
#define LAYA_PROF_EMBED_NORM 0 /* embedding gather + LayerNorm */
#define LAYA_PROF_NORM 1       /* LayerNorm (attention, MLP and final norms) */
#define LAYA_PROF_QKV 2        /* QKV projection (RoPE in its epilogue) */
#define LAYA_PROF_ROPE 3       /* stand-alone RoPE (not launched by the forward) */
#define LAYA_PROF_ATTN 4       /* attention */
#define LAYA_PROF_OUT 5        /* attention output projection + residual */
#define LAYA_PROF_UP 6         /* MLP up-projection + GeGLU */
#define LAYA_PROF_DOWN 7       /* MLP down-projection + residual */
#define LAYA_PROF_OUTPUT 8     /* copies into the caller's layout (padded output rows) */
#define LAYA_PROF_CLASSES 9

/* Measurement aid.  While enabled, laya_enc_run / laya_enc_run_device launch
 * the same kernels as without it (same plans, same programmatic dependent
 * launch, replayed from a graph of their own when graphs are on), except that
 * the first CTA of every kernel records the %globaltimer value at which its
 * dependency wait returned, i.e. when the kernel before it completed, and a
 * one-thread kernel marks the completion of the last.  Launch k is charged
 * the time from its own release to the release of launch k + 1, so the
 * charges of a forward add up to its device time with the overlap of the
 * graph replay.  Each run first folds the previous profiled run's stamps
 * into per-class totals (waiting for that run to finish). */
int laya_enc_set_profiling(laya_enc_handle* h, int enabled);

/* Folds in the last run, then returns and clears the totals: ms[c] (device
 * time) and launches[c] for classes c < n (n <= LAYA_PROF_CLASSES). */
int laya_enc_profile_read(laya_enc_handle* h, double* ms, int* launches, int n);

/* Debug aid for per-layer parity: runs the forward as laya_enc_run does (host
 * token_ids and lengths, out_hidden written the same way) but eagerly, and
 * also writes `states`: DEVICE BF16 [L, batch, seq, hidden] (L = encoder +
 * decision layers), caller-owned, where states[l] is the residual stream
 * entering layer l in the padded layout (states[0]: the embedding output;
 * states[n_encoder_layers]: the stream before the final norm).  Padded
 * positions hold 0.  With out_hidden, this gives the input and the output of
 * every layer, so that a checker can run one layer at a time on the GPU's own
 * state.  Same argument errors as laya_enc_run; states must be 16-byte
 * aligned. */
int laya_enc_debug_capture(laya_enc_handle* h, const int32_t* token_ids,
                           const int32_t* lengths, int batch, int seq, void* out_hidden,
                           void* states, void* stream);

/* Frees the handle and every workspace and graph it owns.  NULL is allowed. */
int laya_enc_destroy(laya_enc_handle* h);

/* Message of the last error on this handle (or of the last failed create when
 * h is NULL).  Never NULL; the string lives until the next call. */
const char* laya_enc_last_error(const laya_enc_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* LAYA_ENC_H_ */
