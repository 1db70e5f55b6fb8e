/*
 * rlt.h -- C ABI of the B300 implementation of the Recurrent Looped
 * Transformer (RLT) hot path: the causal encoder with memory projection (the
 * producer) and the batched recurrent decoder transition with its scoring head.
 *
 * Sources (page title, section):
 *  - "Understanding and Applying the Recurrent Looped Transformer
 *    Architecture", "How the Architecture Works": H_t = (s_t, C_t^D),
 *    H_0 = (s_*, empty), (s_t, C_t^D) = D_phi(Merge(e_t, s_{t-1}), M_<=t,
 *    C_{t-1}^D, t), p(x_{t+1} | x_{1:t}) = softmax(W_o RMSNorm_o(s_t));
 *    "Three forms of context" (window W includes the current token,
 *    cross-attention reads memory through the current position);
 *    "Basic Usage" (prompt prefill = parallel encode, then recur through every
 *    prompt token); "Current-Policy Reinforcement Learning Replay" (score an
 *    action before consuming it; temperature and truncation in the behaviour
 *    log-probability; caches are stale after a weight update).
 *  - "Princeton Researcher Proposes Recurrent Looped Transformer to Carry
 *    Decoder State Across Tokens", architecture and design-principle
 *    paragraphs (token-parallel encoder and memory projection in G groups,
 *    tied encoder/decoder weights, decoder sequential in t and batched across
 *    independent sequences, Proposition 3.1: the prompt/response split does
 *    not change the state).
 *
 * Conventions
 *  - All tensors are caller-owned device memory (PyTorch allocates them); the
 *    library borrows the pointers for the duration of a call and allocates no
 *    device memory.  Every call is asynchronous on the given CUDA stream.
 *  - Matrices are row-major W[out][in] (y = x W^T).  "dtype" below is float32
 *    when config.dtype == RLT_F32 and bfloat16 when RLT_BF16; norm gains, the
 *    gate bias and s_* are always float32.  Pointers must be 16-byte aligned.
 *  - Per-layer tensors are stacked on a leading layer axis L = n_layers
 *    (L_E = L_D; encoder layer l and decoder layer l share W_qkv, W_O, W_1,
 *    W_3, W_2).
 *  - Return values: RLT_OK (0) or a negative RLT_E* code.  The library never
 *    aborts, traps or exits.  Device-side conditions (a bounded wait that gave
 *    up, an out-of-range token id) are recorded in a flag inside the workspace
 *    and read with rlt_status().
 */
#ifndef RLT_H_
#define RLT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(RLT_BUILD)
#define RLT_API __attribute__((visibility("default")))
#else
#define RLT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* rlt_stream_t;   /* a cudaStream_t; NULL = legacy default stream */

enum {
  RLT_OK = 0,
  RLT_EINVAL = -1,      /* bad argument: null pointer, shape, alignment, config */
  RLT_ESTALE = -2,      /* state.version differs from the model's version */
  RLT_ERANGE = -3,      /* state.pos + n exceeds the encoded length T_mem */
  RLT_ECUDA = -4,       /* a CUDA runtime call or launch failed */
  RLT_ETIMEOUT = -5,    /* device flag: a bounded wait gave up */
  RLT_EBOUNDS = -6,     /* device flag: an index (token or action id) was out of range */
  RLT_EWORKSPACE = -7,  /* workspace smaller than rlt_workspace_size() */
  RLT_EUNSUPPORTED = -8 /* shape outside what the kernels are built for */
};

enum { RLT_F32 = 0, RLT_BF16 = 1 };
enum { RLT_GATE_LEARNED = 0, RLT_GATE_DISCARD_S = 1 };
enum { RLT_MEM_FINAL = 0, RLT_MEM_PER_LAYER = 1 };

/* Model shape.  d_model = n_heads * head_dim; head_dim even and <= 128;
 * mem_groups is 1 (memory shared by all decoder layers) or n_layers (one
 * group per layer).  gate_mode RLT_GATE_DISCARD_S forces the merge gate z to
 * 0 (u_t = e_t) and exists for the equivalence checks; RLT_GATE_LEARNED is
 * z = sigmoid(W_g [e_t; s_{t-1}] + b_g), u_t = z * s_{t-1} + (1 - z) * e_t.
 * mem_source picks where the memory groups are projected from: RLT_MEM_FINAL
 * (every group from the final encoder output e; "Princeton Researcher
 * Proposes Recurrent Looped Transformer ...", architecture paragraph: decoder
 * keys and values from the final encoder states) or RLT_MEM_PER_LAYER (group
 * l from RMSNorm_e of the encoder's residual stream after layer l, the other
 * reading of the configurations with per-layer memory projections; needs
 * mem_groups == n_layers). */
typedef struct rlt_config {
  int32_t d_model, n_layers, n_heads, head_dim, d_ffn, window, mem_groups, vocab;
  int32_t dtype;          /* RLT_F32 or RLT_BF16 */
  float rms_eps;          /* RMSNorm: x / sqrt(mean(x^2) + eps) * g */
  float rope_theta;       /* rotate-half RoPE base on encoder and decoder self-attention */
  int32_t gate_mode;
  int32_t mem_source;     /* RLT_MEM_FINAL or RLT_MEM_PER_LAYER */
} rlt_config;

/* Weights: device pointers, borrowed for the model's lifetime (the caller
 * keeps them alive and calls rlt_model_set_version after changing them). */
typedef struct rlt_weights {
  const void* tok_emb;          /* [V][d]        dtype   token embedding */
  const float* s_star;          /* [d]           f32     learned start state s_* */
  const void* W_g;              /* [d][2d]       dtype   merge gate, input [e_t; s_{t-1}] */
  const float* b_g;             /* [d]           f32     merge gate bias */
  const void* W_qkv;            /* [L][3d][d]    dtype   rows [q; k; v], head-major (tied) */
  const void* W_O;              /* [L][d][d]     dtype   self-attention output (tied) */
  const void* W_1;              /* [L][f][d]     dtype   SwiGLU gate branch (tied) */
  const void* W_3;              /* [L][f][d]     dtype   SwiGLU linear branch (tied) */
  const void* W_2;              /* [L][d][f]     dtype   SwiGLU down projection (tied) */
  const void* W_Qx;             /* [L][d][d]     dtype   cross-attention query (decoder only) */
  const void* W_Ox;             /* [L][d][d]     dtype   cross-attention output (decoder only) */
  const void* W_K;              /* [G][d][d]     dtype   memory key projection per group */
  const void* W_V;              /* [G][d][d]     dtype   memory value projection per group */
  const void* W_o;              /* [V][d]        dtype   output head */
  const float* enc_attn_norm;   /* [L][d] */
  const float* enc_ffn_norm;    /* [L][d] */
  const float* enc_norm;        /* [d]   final encoder norm producing e */
  const float* dec_attn_norm;   /* [L][d] */
  const float* dec_xattn_norm;  /* [L][d] */
  const float* dec_ffn_norm;    /* [L][d] */
  const float* head_norm;       /* [d]   RMSNorm_o */
} rlt_weights;

/* Recurrent state H_t = (s_t, C_t^D) of B sequences advancing in lockstep.
 * All device buffers are caller-owned.  ring_k/ring_v hold the per-layer SWA
 * cache as a ring of W slots: entry of position p (0-based) lives in slot
 * p mod W, after RoPE for keys.  pos and version are host-side fields the
 * library reads and updates. */
typedef struct rlt_state {
  int32_t batch;          /* B */
  int32_t pos;            /* tokens consumed so far (t of s_t) */
  uint64_t version;       /* model version the state was built under */
  float* s;               /* [B][d]              f32    s_t */
  void* ring_k;           /* [L][B][H][W][hd]    dtype  keys after RoPE */
  void* ring_v;           /* [L][B][H][W][hd]    dtype  values */
} rlt_state;

typedef struct rlt_model rlt_model;   /* opaque host object */

/* Validates the config and weight pointers and keeps them.  Creates host-side
 * resources only (a capture stream, graph cache); no device allocation. */
RLT_API int rlt_model_create(const rlt_config* cfg, const rlt_weights* w, uint64_t version,
                     rlt_model** out);
/* Declares that the weights changed: every state built earlier becomes stale
 * (rlt_decode_steps then returns RLT_ESTALE). */
RLT_API int rlt_model_set_version(rlt_model* m, uint64_t version);
RLT_API void rlt_model_destroy(rlt_model* m);

/* Bytes of workspace rlt_encode / rlt_decode_steps need for B sequences of up
 * to T_max positions.  The workspace also holds the device status flag.  A
 * workspace serves one call at a time (calls that share it must be ordered
 * on one stream). */
RLT_API int rlt_workspace_size(const rlt_model* m, int32_t B, int32_t T_max, size_t* bytes);
/* Clears the device status flag of a fresh workspace (call once after
 * allocating it, before the first rlt_encode / rlt_decode_steps). */
RLT_API int rlt_workspace_init(void* ws, size_t ws_bytes, rlt_stream_t stream);
/* Byte sizes of the state buffers (s, each of ring_k / ring_v) for B sequences. */
RLT_API int rlt_state_sizes(const rlt_model* m, int32_t B, size_t* s_bytes, size_t* ring_bytes);

/* H_0: s = s_* for every sequence, ring slots filled with NaN (never read
 * before written), pos = 0, version = model version. */
RLT_API int rlt_state_init(const rlt_model* m, rlt_state* st, rlt_stream_t stream);

/* Token-parallel causal encoder and memory projection over positions 0..T-1:
 *   tokens [B][T] int32 (device), e [B][T][d] dtype,
 *   mem [G][2][B][H][T][hd] dtype (index 0 keys, 1 values; no RoPE).
 * Memory depends only on the tokens. */
RLT_API int rlt_encode(const rlt_model* m, const int32_t* tokens, int32_t B, int32_t T,
               void* e, void* mem, void* ws, size_t ws_bytes, rlt_stream_t stream);

/* Advances every sequence of st by n tokens: for i in 0..n-1 the token at
 * position p = st->pos + i is consumed (step t = p + 1, reading e[:, p] and
 * memory positions 0..p), then the head scores actions[b][i], the token that
 * follows, before it is consumed:
 *   logp[b][i]      = l_a/T - LSE_topk(l/T)   (-inf if a is outside the top-k;
 *                     top_k = 0 means no truncation)
 *   logp_full[b][i] = l_a/T - LSE(l/T)
 *   argmax[b][i]    = argmax_v l_v (lowest id on ties)
 * where l = W_o RMSNorm_o(s_t) and T = temperature.  An action < 0 gives NaN.
 * Any output pointer may be NULL.  emit_steps (HOST array, n_emit entries,
 * each in [0, n)) selects steps whose logits are written to
 * logits[n_emit][B][V] (f32).  e is [B][T_mem][d], mem [G][2][B][H][T_mem][hd].
 * Requires st->pos + n <= T_mem and st->version == model version.  Splitting
 * n across calls gives bit-identical results (Proposition 3.1). */
RLT_API int rlt_decode_steps(const rlt_model* m, rlt_state* st, const void* e, const void* mem,
                     int32_t T_mem, int32_t n, const int32_t* actions, float temperature,
                     int32_t top_k, float* logp, float* logp_full, int32_t* argmax,
                     const int32_t* emit_steps, int32_t n_emit, float* logits,
                     void* ws, size_t ws_bytes, rlt_stream_t stream);

/* Decoder path of rlt_decode_steps (both compute the transition above; the
 * step stays sequential in t while independent sequences share the launch -
 * "Princeton Researcher Proposes Recurrent Looped Transformer ...", design
 * principles paragraph).
 *  RLT_DECODE_GRAPH  one step is captured as a CUDA graph of per-operation
 *                    kernels (tensor-core projections with split-K clusters,
 *                    attention, norms, head) and replayed n times.  Every
 *                    configuration.
 *  RLT_DECODE_FUSED  one persistent launch runs all n steps: one thread-block
 *                    cluster per group of at most 16 sequences, the
 *                    projections split by rows across the cluster's CTAs and
 *                    exchanged through distributed shared memory, the next
 *                    phase's weights streamed from L2 while the current one
 *                    computes.  bf16 models whose per-CTA working set fits in
 *                    shared memory (small widths); rlt_decode_steps returns
 *                    RLT_EUNSUPPORTED otherwise.  The same values are
 *                    stored in bf16 as on the graph path; sums run in
 *                    another order, so the two paths agree to rounding, not
 *                    bitwise.  Splitting n across calls is bit-identical
 *                    within this path.
 *                    On this path rlt_generate runs too: per token the draw,
 *                    the incremental encoder step (embedding, every encoder
 *                    layer against the encoder cache, RMSNorm_e, the memory
 *                    rows) and the decoder step, all n tokens in one launch.
 *  RLT_DECODE_AUTO   the graph path.
 * cluster_size 0 lets the fused path choose per call among 16, 8, 4, 2, 1
 * CTAs per cluster: the most sequences per cluster whose working set fits in
 * shared memory, the fewest waves of clusters the device holds at once, then
 * the largest cluster; 1, 2, 4, 8 or 16 forces the cluster size.
 * Host-side setting of the model object; not thread-safe with concurrent
 * calls on the same model.  Errors: RLT_EINVAL (null model, unknown path or
 * cluster size). */
enum { RLT_DECODE_AUTO = 0, RLT_DECODE_GRAPH = 1, RLT_DECODE_FUSED = 2 };
RLT_API int rlt_set_decode_path(rlt_model* m, int32_t path, int32_t cluster_size);

/* The fused path's plan for B sequences: CTAs per cluster, sequences per
 * cluster, clusters, and dynamic shared memory per CTA.  RLT_EUNSUPPORTED
 * when the fused path does not take this model (fp32 models, widths whose
 * working set exceeds shared memory, head counts that are neither a multiple
 * nor a divisor of the cluster size).  Any output pointer may be NULL. */
RLT_API int rlt_fused_plan(const rlt_model* m, int32_t B, int32_t* cluster_size, int32_t* seqs_per_cluster,
                           int32_t* clusters, int32_t* smem_bytes);

/* Cross-attention of one decoder layer (the step that reads encoder memory),
 * as a standalone call: for every sequence b and head h,
 *   out[b][h*hd + i] = sum_{j < t} softmax_j(q[b][h] . K[b][h][j] / sqrt(hd)) V[b][h][j][i]
 * i.e. attention to memory positions 1..t (the current position included).
 *   q     [B][d] f32 (the projected query, no RoPE)
 *   mem_k [B][H][T_mem][hd] dtype, mem_v same layout (one group's plane of the
 *         memory written by rlt_encode)
 *   out   [B][d] dtype;  1 <= t <= T_mem.
 * Partial results and per-(b, h) arrival counters go to the workspace
 * (rlt_workspace_size(m, B, T_mem)). */
RLT_API int rlt_cross_attention(const rlt_model* m, const float* q, const void* mem_k, const void* mem_v,
                                int32_t B, int32_t T_mem, int32_t t, void* out, void* ws, size_t ws_bytes,
                                rlt_stream_t stream);

/* Dense projection on the tensor cores: the kernel behind every projection of
 * the encoder and of the decoder step of bf16 models, exposed so that it can
 * be tested and timed on its own.
 *   W3 == NULL:  C[m][n] = sum_k A[m][k] W[n][k]                       (n < N)
 *   W3 != NULL:  C[m][j] = silu(sum_k A[m][k] W[j][k]) * sum_k A[m][k] W3[j][k]
 *                (the SwiGLU pair W_1, W_3 of one FFN layer; j < N)
 * A [M][lda] bf16, W and W3 [N][ldw] bf16 (row pitches multiples of 8
 * elements), C [M][ldc] f32.  K may be any positive size (zero padded).  The
 * model must be a bf16 model; the workspace must hold
 * rlt_workspace_size(m, 1, 1) bytes (split-K partials and counters). */
RLT_API int rlt_linear(const rlt_model* m, const void* A, int32_t lda, int32_t M, int32_t K, const void* W,
                       const void* W3, int32_t ldw, int32_t N, float* C, int32_t ldc, void* ws, size_t ws_bytes,
                       rlt_stream_t stream);

/* Allocation-free variant of rlt_cross_attention, for callers that cannot
 * allocate device memory (no cudaMalloc, no torch allocator): same result,
 * same q / mem_k / mem_v / out layouts, but the partial results live in a
 * fixed 16 MiB array inside the library, so no workspace is passed and the
 * shape comes as plain sizes (n_heads, head_dim, dtype = RLT_F32/RLT_BF16).
 * The pages have no counterpart: this is an integration convenience.
 *  - Limit: round_up(4 * B * n_heads, 256) + B * n_heads * 32 * (head_dim + 2)
 *    * 4 bytes (arrival counters and up to 32 partial results per (b, h)) must
 *    fit in 16 MiB - 256 B, i.e. B * n_heads <= 1007 at head_dim 128; larger
 *    requests return RLT_EUNSUPPORTED.
 *  - The first call on a device looks up the array's device address (set-up);
 *    make that first call before any stream capture.  The address is kept
 *    for the life of the process: do not use the entry point on a device
 *    after cudaDeviceReset (or another teardown of its primary context).
 *  - Every call shares the array: calls that overlap on the GPU race.
 *  - Device-side conditions (a bounded wait that gave up) go to a status word
 *    inside the array, not to a workspace: read and clear it with
 *    rlt_cross_attention_noalloc_status (it synchronises the stream and
 *    returns RLT_OK, RLT_ETIMEOUT, or RLT_ECUDA when the set-up or the read
 *    fails).  The first condition recorded wins until it is read.
 *  - Allocates nothing; its launches are not included in rlt_launch_count(). */
RLT_API int rlt_cross_attention_noalloc(const float* q, const void* mem_k, const void* mem_v, int32_t B,
                                        int32_t n_heads, int32_t head_dim, int32_t dtype, int32_t T_mem,
                                        int32_t t, void* out, rlt_stream_t stream);
RLT_API int rlt_cross_attention_noalloc_status(rlt_stream_t stream);

/* Generation ("Understanding and Applying the Recurrent Looped Transformer
 * Architecture", "Prompt prefill" and "Autoregressive generation"): the
 * prompt is encoded token-parallel and consumed by the decoder; then each new
 * token is drawn from the current state's distribution, encoded
 * incrementally against the encoder's key/value cache, and consumed through
 * the decoder exactly once.  bf16 models (RLT_EUNSUPPORTED otherwise).
 *
 * rlt_encode_kv: rlt_encode of positions 0..T-1 into buffers with room for
 *   T_max positions, also keeping every encoder layer's keys (after RoPE) and
 *   values: e [B][T_max][d], mem [G][2][B][H][T_max][hd], enc_kv
 *   [L][2][B][H][T_max][hd], all dtype; workspace rlt_workspace_size(m, B,
 *   T_max).  The prompt is then consumed with rlt_decode_steps(..., e, mem,
 *   T_mem = T_max, n = T, ...).
 * rlt_generate: from st (pos = p tokens consumed) draws, encodes and consumes
 *   n tokens (positions p..p+n-1), writing them to tokens [B][n] and, when
 *   logp is given, the log-probability of each under the distribution it was
 *   drawn from (temperature, top-k as in rlt_decode_steps) to logp [B][n].
 *   Draw i of sequence b uses the uniform number of (seed, b, position) - a
 *   SplitMix64 counter - and the token is the first id, in id order, at which
 *   the cumulative weight of the (top-k) set passes it; so the tokens do not
 *   depend on how generation is split into calls.  Requires p + n <= T_max,
 *   e / mem / enc_kv holding positions 0..p-1 (rlt_encode_kv, then earlier
 *   rlt_generate calls); writes positions p..p+n-1 of them.  Errors as
 *   rlt_decode_steps. */
RLT_API int rlt_encode_kv(const rlt_model* m, const int32_t* tokens, int32_t B, int32_t T, int32_t T_max, void* e,
                          void* mem, void* enc_kv, void* ws, size_t ws_bytes, rlt_stream_t stream);
RLT_API int rlt_generate(const rlt_model* m, rlt_state* st, void* e, void* mem, void* enc_kv, int32_t T_max,
                         int32_t n, uint64_t seed, float temperature, int32_t top_k, int32_t* tokens, float* logp,
                         void* ws, size_t ws_bytes, rlt_stream_t stream);

/* Exact prefix snapshots ("Recurrent Looped Transformer: A New Architecture
 * for Infinite Context Reasoning", "Training and Serving Considerations";
 * "Princeton Researcher Proposes Recurrent Looped Transformer ...",
 * training and serving paragraph): what a multi-turn server keeps to resume a
 * prefix - the encoder's output and memory, the whole decoder state, the
 * position, the window convention and the weight version - and may reuse
 * across requests because the state does not depend on how the computation
 * was split; a weight update invalidates it.
 *
 * A snapshot of a state at position pos holds everything needed to continue
 * decoding from there: s_pos, both window caches (ring slots by position mod
 * W, W recorded), pos, and the encoder output e and memory M of positions
 * 1..pos, tagged with the model version and shape; optionally also the
 * encoder's key/value cache of positions 1..pos (rlt_encode_kv, rlt_generate),
 * which is what continuing generation needs.  Restoring it and decoding (or
 * generating) on gives bit-identical states, tokens and log-probabilities to
 * never having stopped (Proposition 3.1), also for another request that
 * shares the prefix (the encoder, its cache and the memory of positions <= pos
 * depend only on those tokens).
 *   snap: caller-owned device buffer of rlt_snapshot_size(m, B, pos,
 *         with_enc_kv) bytes, 16-byte aligned; layout private to the library
 *         (a header, then s, ring K, ring V, e [B][pos][d],
 *         M [G][2][B][H][pos][hd], and with the cache section
 *         [L][2][B][H][pos][hd]).
 *   e [B][T_mem][d], mem [G][2][B][H][T_mem][hd] and enc_kv
 *         [L][2][B][H][T_mem][hd]: the encoder buffers of rlt_encode /
 *         rlt_encode_kv; save reads and restore writes their rows 0..pos-1.
 *         enc_kv NULL: no cache section (save), the snapshot holds none
 *         (restore: a snapshot with the section needs enc_kv, one without it
 *         takes enc_kv NULL).
 * rlt_snapshot_save copies asynchronously on the stream (nothing is read on
 * the host).  rlt_snapshot_restore reads the snapshot's header (it
 * synchronises the stream for that), checks it against the model and the
 * state, then copies asynchronously and sets st->pos and st->version.
 * Errors: RLT_EINVAL (null or misaligned pointer, buffer too small, batch or
 * shape mismatch, pos > T_mem, not a snapshot, cache section asked for and
 * absent or present and not asked for, with_enc_kv not 0 or 1), RLT_ESTALE
 * (the snapshot, or st for save, was taken under another model version). */
RLT_API int rlt_snapshot_size(const rlt_model* m, int32_t B, int32_t pos, int32_t with_enc_kv, size_t* bytes);
RLT_API int rlt_snapshot_save(const rlt_model* m, const rlt_state* st, const void* e, const void* mem,
                              const void* enc_kv, int32_t T_mem, void* snap, size_t snap_bytes, rlt_stream_t stream);
RLT_API int rlt_snapshot_restore(const rlt_model* m, const void* snap, size_t snap_bytes, rlt_state* st,
                                 void* e, void* mem, void* enc_kv, int32_t T_mem, rlt_stream_t stream);

/* Backpropagation through time of the decoder recurrence, teacher forced
 * ("Recurrent Looped Transformer: A New Architecture for Infinite Context
 * Reasoning", "Training and Serving Considerations": training backpropagates
 * through time; "Princeton Researcher Proposes Recurrent Looped Transformer
 * ...", training paragraph: the state Jacobian has cross terms through the
 * decoder's keys and values, so a truncated scheme names every tensor it
 * detaches; "Understanding and Applying the Recurrent Looped Transformer
 * Architecture", "Current-Policy Reinforcement Learning Replay": gradients
 * pass through the recurrent outputs, the decoder key-value entries and the
 * encoder memory).
 *
 * From H_0 = (s_*, empty cache), steps t = 1..n consume positions 0..n-1 of
 * e [B][T_mem][d] with memory mem [G][2][B][H][T_mem][hd] (dtype, as written
 * by rlt_encode), the head scoring actions [B][n] (int32, device) exactly as
 * rlt_decode_steps does (temperature, top_k):
 *   loss = - sum over (b, t) with 0 <= a < V of lp_t(a_{b,t})      (f32 [1])
 *   logp [B][n] = lp (NaN for a < 0; -inf for an action outside the top-k
 *                 set, whose gradient then keeps only the set's terms); may be NULL
 *   grads: d loss / d every decoder parameter, fp32, the parameters' shapes
 *          (W_qkv, W_O, W_1, W_3, W_2 get the decoder's use of the tied
 *          matrices only; the encoder's use is the encoder backward's);
 *          all fields required, overwritten
 *   d_e  [B][T_mem][d] f32, d_mem [G][2][B][H][T_mem][hd] f32: gradients of
 *          the encoder output and memory (rows past n zero); may be NULL.
 * Named detach points (all off: full BPTT):
 *   detach_s_every = k > 0: s_t enters step t+1 as a constant when t % k == 0;
 *   RLT_DETACH_CACHE: the window keys/values of earlier positions enter later
 *     steps as constants (each step keeps the gradient of its own entry);
 *   RLT_DETACH_MEMORY: the memory is a constant (d_mem stays zero).
 * Execution (flags): each step's launches are captured once as a CUDA graph
 * (on the model's capture stream; one graph for the recording step and one
 * per slot of a 16-step block) and replayed on the caller's stream;
 * RLT_BPTT_NO_GRAPHS launches them one by one instead (same results).
 * Memory gradient: on bf16 models with head_dim 32, 64 or 128 it runs on the
 * tensor cores (bf16 MMA operands: the queries, output gradients, P and dS
 * rounded to bf16); RLT_BPTT_CORE_MEMGRAD keeps it on CUDA cores in fp32.
 * Work: a forward pass recording s_t and every position's keys and values,
 * then a reverse pass that recomputes each step's activations; workspace
 * rlt_bptt_workspace_size(m, B, n) bytes (its first 256 bytes are the status
 * word, cleared by rlt_workspace_init).  Errors: RLT_EINVAL (null or
 * misaligned pointer, n > T_mem, bad temperature / top_k / flags),
 * RLT_EWORKSPACE, RLT_EUNSUPPORTED (bf16 model with vocab not a multiple of
 * 8, or B * n_heads > 65535); an action >= V sets RLT_EBOUNDS in the status
 * word and counts as absent. */
enum { RLT_DETACH_CACHE = 1, RLT_DETACH_MEMORY = 2, RLT_BPTT_NO_GRAPHS = 4, RLT_BPTT_CORE_MEMGRAD = 8 };
typedef struct rlt_grads {
  float *W_g, *b_g, *W_qkv, *W_O, *W_Qx, *W_Ox, *W_1, *W_3, *W_2, *W_o;
  float *dec_attn_norm, *dec_xattn_norm, *dec_ffn_norm, *head_norm, *s_star;
} rlt_grads;
RLT_API int rlt_bptt_workspace_size(const rlt_model* m, int32_t B, int32_t n, size_t* bytes);
RLT_API int rlt_bptt(const rlt_model* m, const void* e, const void* mem, int32_t T_mem, int32_t B, int32_t n,
                     const int32_t* actions, float temperature, int32_t top_k, int32_t detach_s_every,
                     int32_t flags, float* loss, float* logp, const rlt_grads* grads, float* d_e,
                     float* d_mem, void* ws, size_t ws_bytes, rlt_stream_t stream);

/* Failure injection for the bounded device waits, so that their give-up
 * path can be exercised without a GPU fault (a wait whose arrival never
 * comes).  Every wait of the library's kernels on a copy, an MMA or a cluster
 * peer is bounded by a clock budget (about one second); a wait that runs out
 * records RLT_ETIMEOUT in the workspace's status word, waits (bounded) for
 * the launch's other copies in flight, frees its tensor memory and returns.
 * This call arms that path for the next launch of one kernel through its
 * standalone entry point on this model:
 *   RLT_KERNEL_XATTN  rlt_cross_attention: one warp never requests its first
 *                     value chunk;
 *   RLT_KERNEL_GEMM   rlt_linear (bf16 models): the first CTA never requests
 *                     its first A tile (its split-K cluster peers then wait on
 *                     it at the cluster barrier until it gives up and arrives);
 *   RLT_KERNEL_NORM_PROJ  rlt_decode_steps (bf16 models, batches of up to 128
 *                     sequences, whose projections build their RMSNorm input
 *                     in the kernel): in the layer-0 QKV projection the first
 *                     CTA never requests the fp32 rows of its first k-block,
 *                     so the group converting them and then the MMA give up;
 *                     every step of that call repeats it (call with n = 1);
 *                     calls that build no such projection (fp32 models,
 *                     more than 128 sequences) leave it armed;
 * and gives every wait of that launch budget_cycles clock cycles (1e3 ..
 * 4e9) instead of the default.  The launch's output is then unspecified and
 * rlt_status() of its workspace returns RLT_ETIMEOUT; later launches are not
 * affected (one-shot; the attention's arrival counters are cleared by every
 * rlt_cross_attention call).  Host-side setting, not thread-safe with
 * concurrent calls on the same model.  Errors: RLT_EINVAL (null model,
 * unknown kernel, budget out of range), RLT_EUNSUPPORTED (RLT_KERNEL_GEMM or
 * RLT_KERNEL_NORM_PROJ on an fp32 model). */
enum { RLT_KERNEL_XATTN = 1, RLT_KERNEL_GEMM = 2, RLT_KERNEL_NORM_PROJ = 3 };
RLT_API int rlt_debug_withhold_copy(rlt_model* m, int32_t kernel, int64_t budget_cycles);

/* Synchronises the stream, returns the device status recorded in the workspace
 * (RLT_OK, RLT_ETIMEOUT or RLT_EBOUNDS) and clears it. */
RLT_API int rlt_status(void* ws, rlt_stream_t stream);

RLT_API const char* rlt_strerror(int code);

/* Per-launch timing of one kernel class inside rlt_decode_steps, with CUDA
 * events recorded on the launching stream (event-record nodes of the captured
 * step, re-pointed to fresh events on every replay).  rlt_timer_arm enables it
 * for up to max_launches launches; rlt_timer_read synchronises the device,
 * writes the per-launch durations in milliseconds (in launch order) and
 * disarms.  Classes: RLT_TIMER_XATTN (cross-attention, partial + combine),
 * RLT_TIMER_SWA, RLT_TIMER_GEMM (every decoder GEMM), RLT_TIMER_HEAD (norm,
 * head GEMM and log-softmax reduction), RLT_TIMER_STEP (a whole step). */
enum { RLT_TIMER_OFF = 0, RLT_TIMER_XATTN = 1, RLT_TIMER_SWA = 2, RLT_TIMER_GEMM = 3,
       RLT_TIMER_HEAD = 4, RLT_TIMER_STEP = 5 };
RLT_API int rlt_timer_arm(rlt_model* m, int32_t kernel_class, int32_t max_launches);
RLT_API int rlt_timer_read(rlt_model* m, float* ms, int32_t cap, int32_t* n_out);

/* Number of kernels this library has enqueued in this process (graph nodes
 * count once per graph launch). */
RLT_API uint64_t rlt_launch_count(void);

/* ABI version of this header (major * 100 + minor). */
RLT_API int rlt_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RLT_H_ */
