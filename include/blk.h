/*
 * blk.h — C ABI of a GB300 (sm_103a) library for the forward pass of one
 * Llama-style decoder block.
 *
 * The block (nnterp encyclopedia "arcee", "The block, in order"; the
 * "LlamaForCausalLM-32L-4096d" sheet, "Implementing it"):
 *
 *   h   = x + o_proj(attn(rope(qk_norm(q_proj(n1))), rope(qk_norm(k_proj(n1))), v_proj(n1)))
 *         with n1 = rmsnorm(x, input_layernorm)
 *   out = h + down_proj(act(...(rmsnorm(h, post_attention_layernorm))))
 *
 * act is gated SiLU (silu(gate) * up, the sheet's pseudo-code), squared ReLU
 * ("arcee": relu(up)^2) or xIELU ("apertus", "The MLP has no gate").
 * q_norm/k_norm are optional per-head RMSNorms before the rotary ("apertus",
 * "Queries and keys are normed per head, before the rotary"). Attention is
 * causal softmax(q k^T / sqrt(head_dim)) v with key/value head j serving query
 * heads j*G .. j*G+G-1, G = num_heads / num_kv_heads ("arcee", "Grouped-query
 * attention, 128-wide heads").
 *
 * The "afmoe" block variant (dense MLP), four descriptor options:
 *   sliding_window  attention over the last W positions ("Rotary runs on the
 *                   sliding-window blocks only": 2048 on Trinity Nano and Mini)
 *   no_rope         no rotary on q and k (afmoe's whole-prefix blocks)
 *   attn_gate       o_proj reads heads * sigmoid(n1 W_attn_gate^T), one gate value
 *                   per channel of every head ("Attention: per-head q/k norms and a
 *                   sigmoid gate on every head")
 *   sandwich_norm   h   = x + rmsnorm(o_proj(...), post_attn_g)
 *                   out = h + rmsnorm(down_proj(...), post_mlp_g)
 *                   ("The block, in order"); the MLP's input norm stays ln2_g
 *                   (afmoe's pre_mlp_layernorm).
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers are CUDA device addresses owned by the
 *    caller; the library never frees or keeps them past the call. Host
 *    pointers (descriptors, weight tables) are read during the call only.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls enqueue work and return; they never synchronise, except
 *    blk_last_status, which reads a device word synchronously.
 *  - Return values are blk_status codes; no exceptions cross the ABI and the
 *    library never exits the process. blk_error_string() names a code;
 *    blk_last_error_message() gives the detail of the last failure on this
 *    thread.
 *  - Activation tensors are row-major with the innermost dimension contiguous.
 *    Weights are PyTorch Linear weights: [out_features, in_features] row-major,
 *    used as h @ W^T, no bias.
 *  - Every device pointer must be 16-byte aligned (TMA and 128-bit loads);
 *    otherwise the call returns BLK_ERR_ALIGNMENT.
 *  - Element type is the descriptor's dtype (fp32 or bf16) for every tensor of
 *    a call, including weights, gains and the KV cache.
 */
#ifndef BLK_H_
#define BLK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BLK_OK = 0,
  BLK_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, inconsistent shape */
  BLK_ERR_UNSUPPORTED = 2,  /* a shape/dtype combination this build has no kernel for */
  BLK_ERR_ALIGNMENT = 3,    /* a pointer not 16-byte aligned */
  BLK_ERR_CACHE_FULL = 4,   /* a decode step would write past the KV cache capacity */
  BLK_ERR_CUDA = 5,         /* a CUDA runtime/driver call or a launch failed */
  BLK_ERR_TIMEOUT = 6,      /* a device-side wait hit its iteration budget (blk_last_status) */
  BLK_ERR_WORKSPACE = 7     /* workspace missing or smaller than blk_workspace_bytes() */
} blk_status;

typedef enum {
  BLK_ACT_SWIGLU = 0, /* silu(h W_gate^T) * (h W_up^T)  ("LlamaForCausalLM-32L-4096d") */
  BLK_ACT_RELU2 = 1,  /* relu(h W_up^T)^2              ("arcee") */
  BLK_ACT_XIELU = 2   /* xielu(h W_up^T)               ("apertus") */
} blk_act;

typedef enum { BLK_F32 = 0, BLK_BF16 = 1 } blk_dtype;

/* Block description, in the pages' config keys (hidden_size, num_attention_heads,
 * num_key_value_heads, head_dim, intermediate_size, hidden_act, rms_norm_eps,
 * rope_theta). */
/* Stretched rotaries (the pages name them with their settings: YaRN factor 20
 * over 4096 positions on "arcee", "Loading and positions"; llama3 factor 8 over
 * 8192, rope_theta 12,000,000 on "apertus"). Both keep fast components, divide
 * slow ones by the factor and blend in between, after their published
 * definitions: llama3 linearly in the turn count over the original context,
 * YaRN (as its published implementation, which transformers runs) linearly in
 * the pair index between the floored and ceiled indices where the components
 * make rope_high and rope_low turns; YaRN also multiplies cos and sin by
 * 0.1 ln(factor) + 1. */
typedef enum {
  BLK_ROPE_PLAIN = 0,
  BLK_ROPE_YARN = 1,   /* rope_low / rope_high: turns over the original context (1 and 32) */
  BLK_ROPE_LLAMA3 = 2  /* rope_low / rope_high: low_freq_factor and high_freq_factor (1 and 4) */
} blk_rope_type;

typedef struct {
  int hidden;        /* hidden_size D */
  int n_heads;       /* num_attention_heads H */
  int n_kv_heads;    /* num_key_value_heads Hkv; H % Hkv == 0 */
  int head_dim;      /* d; even */
  int ffn;           /* intermediate_size F */
  float rope_theta;  /* RoPE base (10000 in the pages' configs) */
  float eps;         /* rms_norm_eps, used by both block norms and q/k norms */
  blk_act act;
  float xielu_alpha_p; /* EFFECTIVE alpha_p (after softplus), see blk_xielu_effective */
  float xielu_alpha_n; /* EFFECTIVE alpha_n (after beta + softplus) */
  float xielu_beta;    /* 0.5 on the pages */
  float xielu_eps;     /* -1e-6 on the pages */
  int qk_norm;       /* 1: per-head RMSNorm of q and k over head_dim before RoPE */
  blk_dtype dtype;   /* storage type of every tensor; accumulation is fp32 */
  int max_batch;     /* largest batch a call may pass */
  int max_seq;       /* largest rotary position + 1 a call may use (prefill length, or cache length + 1) */
  blk_rope_type rope_type;  /* BLK_ROPE_PLAIN ignores the four fields below */
  float rope_factor;        /* >= 1 */
  int rope_orig_max_pos;    /* the original context length the scaling stretches */
  float rope_low, rope_high;
  /* the "afmoe" options (0 = off for each) */
  int sliding_window;  /* W > 0: query at position p sees keys at positions p - W + 1 .. p */
  int no_rope;         /* 1: no rotary (needs rope_type BLK_ROPE_PLAIN) */
  int attn_gate;       /* 1: sigmoid gate on the head outputs (weights.w_attn_gate) */
  int sandwich_norm;   /* 1: post-norms of both sublayers (weights.post_attn_g, post_mlp_g); on the
                          bf16 path it needs prepared weights (see blk_prepare_weights) */
} blk_desc;

/* Block weights: device pointers in the descriptor's dtype.
 * Shapes: ln1_g, ln2_g [D]; wq [H*d, D]; wk, wv [Hkv*d, D]; q_norm_g, k_norm_g
 * [d] (ignored unless qk_norm); wo [D, H*d]; w_gate [F, D] (SWIGLU only, else
 * NULL); w_up [F, D]; w_down [D, F]; w_attn_gate [H*d, D] (attn_gate only);
 * post_attn_g, post_mlp_g [D] (sandwich_norm only; afmoe's
 * post_attention_layernorm and post_mlp_layernorm). */
typedef struct {
  const void *ln1_g, *wq, *wk, *wv, *q_norm_g, *k_norm_g, *wo, *ln2_g;
  const void *w_gate, *w_up, *w_down;
  const void* prepared; /* NULL, or the buffer blk_prepare_weights filled for these weights */
  const void *w_attn_gate, *post_attn_g, *post_mlp_g;
} blk_weights;

/* KV cache: k, v are [batch, Hkv, capacity, d] in the descriptor's dtype,
 * holding keys AFTER k_norm and RoPE. lens is a device int array [batch]:
 * positions already filled. A forward over T new tokens per sequence puts token
 * t at position lens[b] + t, writes its key and value at slot lens[b] + t,
 * lets it attend to slots 0 .. lens[b] + t (causal over the cache and the new
 * tokens) and then adds T to lens[b] on the device. T == 1 is a decode step;
 * T > 1 is a prefill chunk (bf16 path). The pages have no cache: this is the
 * prefill block restricted to the new rows, earlier keys read from the cache. */
typedef struct {
  void *k, *v;
  int capacity;
  int *lens;
} blk_kv_cache;

/* Optional debug outputs of blk_forward (nnterp tap names, "arcee", "The API").
 * Any member may be NULL. Device pointers in the descriptor's dtype:
 *   attention_queries [B,H,T,d], attention_keys / attention_values [B,Hkv,T,d]
 *   (prefill only), attention_head_outputs [B,T,H,d] (before the attention
 *   gate), attention_output, layer_mid, mlp_output [B,T,D] (after the sandwich
 *   post-norms), mlp_neurons [B,T,F].
 * Requesting taps may launch extra copies; it does not change layer_output. */
typedef struct {
  void *attention_queries, *attention_keys, *attention_values;
  void *attention_head_outputs, *attention_output, *layer_mid;
  void *mlp_neurons, *mlp_output;
} blk_taps;

typedef struct blk_handle blk_handle;

/* Validates the descriptor and builds the handle: it owns a small device
 * status word and the RoPE cos/sin table (max_seq x head_dim/2, fp32, computed
 * in double on the host). No weights are copied. Requires a current CUDA
 * device. Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
blk_status blk_create(const blk_desc* desc, blk_handle** out);

/* Optional one-time weight preparation (bf16 path), the step an inference
 * engine does when it loads a model: fp16 copies of wq, wk, wv (and
 * w_attn_gate), wo, w_gate and w_up are written to `prepared`, a caller-owned
 * device buffer of at least blk_prepared_bytes(h) bytes. With weights.prepared
 * set, the o_proj and MLP-up GEMMs of prefills and prefill chunks, and the
 * Q/K/V, o_proj and MLP-up GEMMs of decode steps (and of sandwich-block
 * prefills) take fp16 operands (the input norm's rows, the attention output and
 * the MLP's normed input in fp16 too): 3 more mantissa bits than bf16 at the
 * same tensor-core rate and the same bytes streamed. The conversion is exact for every bf16 weight with
 * 2^-17 <= |w| <= 65504; smaller ones move by at most 2^-25. The input norm's
 * fp16 rows are normalized before rounding, so they stay finite when
 * max|ln1_g| * sqrt(D) <= 65504 (likewise ln2_g on a sandwich block); larger
 * gains are refused. The copies must be refreshed whenever the bf16 weights
 * change. Synchronises `stream` (it checks the ranges).
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED (fp32 handle, or a
 * weight or gain outside those ranges: then use the weights unprepared), CUDA. */
size_t blk_prepared_bytes(const blk_handle* h);
blk_status blk_prepare_weights(blk_handle* h, const blk_weights* w, void* prepared, size_t bytes, void* stream);

/* Frees the handle and its device tables. Safe on NULL. Synchronises nothing:
 * the caller must ensure no work using the handle is still in flight. */
blk_status blk_destroy(blk_handle* h);

/* Bytes of caller-owned device workspace blk_forward needs for this batch and
 * sequence length; decode != 0 when a cache is passed (a decode step when
 * seq == 1; a prefill chunk needs the same as a prefill of seq tokens).
 * Returns 0 for invalid sizes. */
size_t blk_workspace_bytes(const blk_handle* h, int batch, int seq, int decode);

/* The whole block: out[B,T,D] = block(x[B,T,D]).
 * cache == NULL: prefill, positions 0..T-1 per sequence, causal.
 * cache != NULL: T new tokens per sequence over the cache (see blk_kv_cache):
 * a decode step (T == 1) or a prefill chunk (T > 1; bf16 only; its keys and
 * values go to the cache, so the key/value taps are refused).
 * workspace: device scratch of at least blk_workspace_bytes(h, B, T, cache!=NULL).
 * out must not alias x. taps may be NULL. A sandwich_norm block on the bf16
 * path needs weights.prepared: each post-norm scales its sublayer's output to
 * the size of the residual stream, and with it the rounding of that sublayer's
 * GEMM operands; bf16 operands (all that bf16 weights allow) would spend the
 * whole bf16 tolerance there, so such calls return UNSUPPORTED.
 * Errors: INVALID_ARG, ALIGNMENT,
 * UNSUPPORTED, WORKSPACE, CACHE_FULL (checked on the host when the caller
 * passes host_lens_max >= 0, the largest lens[b] before the call; a prefill
 * chunk requires it), CUDA. */
blk_status blk_forward(blk_handle* h, const void* x, int batch, int seq, const blk_weights* w,
                       blk_kv_cache* cache, int host_lens_max, void* out, void* workspace,
                       size_t workspace_bytes, const blk_taps* taps, void* stream);

/* A padded prefill batch (nnterp's attention_mask, "arcee", "The API": [batch
 * seq], zeros are padding). attention_mask: device int32 [B, T], 16-byte
 * aligned; the ones of each row form one contiguous run [lo_b, hi_b) (left
 * padding, right padding, or both). Key j of sequence b is visible to query t
 * iff lo_b <= j < hi_b and j <= t (and within the sliding window), and row t
 * takes rotary position t - lo_b, so every real row equals the row of the
 * unpadded sequence. Padding rows are computed like the others and carry no
 * meaning: rows before lo_b see no key (their head outputs are zero), rows from
 * hi_b on see the real keys. A row whose ones are not contiguous sets the
 * status word to INVALID_ARG (blk_last_status) and is treated as its hull.
 * Otherwise as blk_forward without a cache (same workspace). Errors: those of
 * blk_forward. */
blk_status blk_forward_masked(blk_handle* h, const void* x, int batch, int seq, const int* attention_mask,
                              const blk_weights* w, void* out, void* workspace, size_t workspace_bytes,
                              const blk_taps* taps, void* stream);

/* The model around the block ("LlamaForCausalLM-32L-4096d" sheet, "Implementing
 * it": embed_tokens, the decoder layers, norm, lm_head), all layers of one
 * handle's shape. Device pointers in the handle's dtype, row-major:
 *   embed   [vocab, D]   token embeddings (embed_tokens)
 *   layers  [n_layers]   host array of per-layer weights (blk_weights)
 *   norm_g  [D]          final RMSNorm gain
 *   lm_head [vocab, D]   output projection (may equal embed when tied) */
typedef struct {
  const void* embed;
  const blk_weights* layers;
  int n_layers;
  const void* norm_g;
  const void* lm_head;
  int vocab;
} blk_model;

/* Workspace for blk_model_forward: one layer's blk_workspace_bytes plus two
 * [B, T, D] activation buffers and the final norm's output. */
size_t blk_model_workspace_bytes(const blk_handle* h, int batch, int seq, int decode);

/* logits[B, T, vocab] = lm_head(norm(layers(embed[tokens]))). tokens: device
 * int32 [B, T]; an id outside [0, vocab) embeds as zeros and sets the status
 * word to INVALID_ARG (blk_last_status). caches: NULL (prefill from position 0)
 * or a host array of n_layers KV caches with T new tokens after lens[b] (as in
 * blk_forward; each layer's cache needs its own lens array, since each layer
 * advances its own). Errors: those of blk_forward, WORKSPACE, CUDA. */
blk_status blk_model_forward(blk_handle* h, const blk_model* m, const int* tokens, int batch, int seq,
                             blk_kv_cache* caches, int host_lens_max, void* logits, void* workspace,
                             size_t workspace_bytes, void* stream);

/* A recorded forward: the launches one blk_forward makes for fixed arguments,
 * captured once into a CUDA graph so that replaying it costs one launch. */
typedef struct blk_graph blk_graph;

/* Records blk_forward(h, x, ..., taps) with exactly these arguments (captured on
 * a private stream; nothing runs now) and instantiates the graph. Replays read
 * and write the same buffers, so the caller refreshes inputs in place between
 * replays. A decode graph bumps lens on every replay, as blk_forward does. If
 * profiling is on for h, the graph also records the per-stage events and
 * blk_profile_collect reads them after a replay (keep profiling on while the
 * graph exists). Errors: those of blk_forward, CUDA. */
blk_status blk_forward_graph_create(blk_handle* h, const void* x, int batch, int seq, const blk_weights* w,
                                    blk_kv_cache* cache, int host_lens_max, void* out, void* workspace,
                                    size_t workspace_bytes, const blk_taps* taps, blk_graph** out_graph);

/* Enqueues one replay on the caller's stream. Errors: INVALID_ARG, CUDA. */
blk_status blk_graph_launch(blk_graph* g, void* stream);

/* Frees the graph (the caller ensures no replay is in flight). Safe on NULL. */
blk_status blk_graph_destroy(blk_graph* g);

/* Stage: RMSNorm of each row (nnterp "input_layernorm" / "post_attention_layernorm"):
 * y[r, :] = x[r, :] / sqrt(mean(x[r, :]^2) + eps) * g, statistics in fp32.
 * x, y [rows, n], g [n], device, dtype elements; n % 8 == 0 (bf16) or n % 4 == 0
 * (fp32), n <= 16384. y may alias x. */
blk_status blk_rmsnorm(const void* x, const void* g, int rows, int n, float eps, void* y,
                       blk_dtype dtype, void* stream);

/* Stage: Q/K/V projections of normed rows y[B*T, D], optional per-head q/k
 * RMSNorm, RoPE at positions pos0[b] + t (pos0: device int[B], NULL = 0), and the
 * scatter to head-major layouts q [B,H,T,d], k, v [B,Hkv,T,d].
 * workspace: device scratch of blk_stage_workspace_bytes(h, B*T). */
blk_status blk_qkv_rope(blk_handle* h, const void* y, const blk_weights* w, int batch, int seq,
                        const int* pos0, void* q, void* k, void* v, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Stage: causal grouped-query attention.
 * q [B,H,Tq,d]; k, v with row stride kv_stride rows per (b, kv head):
 * element (b, j, s, :) at ((b*Hkv + j)*kv_stride + s)*d. kv_lens: device int[B]
 * with the number of valid keys per sequence, or NULL for kv_len = Tq (plain
 * prefill). Query i of sequence b sits at position kv_len[b] - Tq + i and sees
 * keys at positions <= its own. Output o [B,Tq,H,d] (nnterp attention_head_outputs).
 * workspace: device scratch of blk_stage_workspace_bytes(h, B*Tq). */
blk_status blk_attn_gqa(blk_handle* h, const void* q, const void* k, const void* v, int batch,
                        int seq_q, int kv_stride, const int* kv_lens, void* o, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Stage: MLP sublayer with the residual add of its rows:
 * out[r] = resid[r] + down(act(h_normed[r])) for rows r < rows, shapes [rows, D].
 * workspace: device scratch of blk_stage_workspace_bytes(h, rows).
 * out may not alias h_normed; it may alias resid. On the bf16 path a
 * sandwich_norm handle returns UNSUPPORTED (its bf16 h_normed rounding would be
 * scaled up by the post-norm; blk_forward runs such blocks on prepared weights). */
blk_status blk_mlp(blk_handle* h, const void* resid, const void* h_normed, const blk_weights* w,
                   int rows, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* Scratch bytes a stage entry point needs for `rows` token rows. */
size_t blk_stage_workspace_bytes(const blk_handle* h, int rows);

/* Device-side status after the caller has synchronised the stream: BLK_OK, or
 * BLK_ERR_TIMEOUT if a kernel's bounded wait gave up (its outputs are then
 * invalid). Clears the word. Reads device memory synchronously. */
blk_status blk_last_status(blk_handle* h);

/* Host helper for xIELU ("apertus"): stored parameters -> effective values
 * alpha_p = softplus(raw_p), alpha_n = beta + softplus(raw_n). */
void blk_xielu_effective(float raw_alpha_p, float raw_alpha_n, float beta, float* alpha_p,
                         float* alpha_n);

/* Allocation-free decode attention. This entry point has no counterpart in the
 * paper; it exists for callers that cannot call cudaMalloc: for instance a host
 * plugin interface that hands over only input and output pointers and no
 * workspace, a runtime that has already given all device memory to its own
 * pool, or a latency-critical loop that cannot afford cudaMalloc's implicit
 * device synchronisation. Such a caller cannot create a handle (blk_create
 * allocates), so this call needs none.
 *
 * It computes the same thing as blk_attn_gqa with kv_lens and seq_q == 1 on
 * the bf16 path: for each sequence b and query head h, o[b, h, :] =
 * softmax(q[b, h] . k[b, j, s] / sqrt(d), s < kv_lens[b]) @ v[b, j, s, :] with
 * j = h / (n_heads / n_kv_heads). q [B, H, 1, 128] and o [B, H, 128] (i.e.
 * [B, 1, H, 128]); k, v [B, Hkv, kv_stride, 128]; kv_lens device int[B] with
 * 1 <= kv_lens[b] <= kv_stride; all bf16 device pointers, 16-byte aligned.
 *
 * Its per-split partial results and its work counter live in one file-scope
 * 16 MiB device array that every GPU loading the library holds until exit. The
 * limit is batch * n_heads * (head_dim + 2) * 4 bytes <= 16 MiB - 256 (e.g.
 * 64 x 32 heads); larger calls return BLK_ERR_UNSUPPORTED with that reason.
 * Every call shares the array and it keeps the last call's contents; each call
 * zeroes the counter (cudaMemsetAsync on `stream`) and writes every partial it
 * reads, but calls that overlap on the GPU (other streams, other host threads)
 * race on it and must be serialised by the caller. The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture. It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 * A device-side wait that runs out (the limit of blk_debug_set_wait_timeout_ns,
 * 2 s by default) cannot be returned by this asynchronous call, and there is no
 * handle to read a status from: the call then writes NaN to every element of o
 * (the status word that decides it sits in the same array, zeroed per call).
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA. */
blk_status blk_attn_decode_noalloc(const void* q, const void* k, const void* v, const int* kv_lens, int batch,
                                   int n_heads, int n_kv_heads, int head_dim, int kv_stride, void* o, void* stream);

/* Static name of a status code. */
const char* blk_error_string(blk_status s);

/* Detail of the last failing call on the calling thread ("" if none). */
const char* blk_last_error_message(void);

/* Debug knob: wall-time limit, in nanoseconds, of every device-side mbarrier
 * wait in later launches; <= 0 restores the default (2 s). A wait that runs
 * out records BLK_ERR_TIMEOUT in the handle's status word (blk_last_status),
 * makes every role of its CTA stop, then waits (with a separate 2 s limit) for
 * the CTA's copies and MMAs in flight, frees its TMEM and returns, leaving the
 * CUDA context usable; the outputs of that call are invalid. Process-wide. */
void blk_debug_set_wait_timeout_ns(long long ns);

/* Status of the debug GEMM entry point (blk_debug_gemm_bf16, which has no
 * handle), read after the caller has synchronised: BLK_OK or BLK_ERR_TIMEOUT.
 * Clears the word. Reads device memory synchronously. Errors: CUDA. */
blk_status blk_debug_last_status(void);

/* Per-stage device timing of later blk_forward calls on this handle: when on,
 * each stage's launches are bracketed by CUDA events recorded on the caller's
 * stream (the stages of a call run back to back; recording adds no sync).
 * Errors: INVALID_ARG, CUDA. */
blk_status blk_profile_enable(blk_handle* h, int on);

/* Waits for the last profiled blk_forward on the handle, adds its per-stage
 * times to running totals and copies, for i < min(max_stages, stage count):
 * total_ms[i] (milliseconds summed over collected calls), launches[i] (kernel
 * launches summed likewise). Returns the number of stages of that call's path
 * (prefill or decode), or -1 on error. Either array may be NULL. */
int blk_profile_collect(blk_handle* h, double* total_ms, long long* launches, int max_stages);

/* Name of stage i of the last profiled path ("" when out of range). */
const char* blk_profile_stage_name(const blk_handle* h, int i);

/* Zeroes the running totals. */
void blk_profile_reset(blk_handle* h);

/* Debug/test entry: the bare tcgen05 GEMM, c[M, N] = bf16(a[M, K] @ b[N, K]^T)
 * with fp32 accumulation, all bf16 row-major device pointers, N-tile bn in
 * {64, 128, 192, 224, 256}, split_k >= 1 (bn == 64 only: fp32 partial sums are then
 * written to c as float [split_k][N][M] instead). K % 8 == 0. pair != 0: CTA pairs
 * (tcgen05 cta_group::2, 256-row tiles, bn in {192, 224, 256}, split_k == 1).
 * Errors: INVALID_ARG, ALIGNMENT, CUDA. */
blk_status blk_debug_gemm_bf16(const void* a, const void* b, void* c, int M, int N, int K, int bn, int split_k,
                               int pair, void* stream);

/* Library version string. */
const char* blk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BLK_H_ */
