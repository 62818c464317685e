/*
 * spec.h -- C ABI of the greedy speculative-decoding verify pass on one GB300.
 *
 * The library runs the data-parallel hot path of speculative decoding on a
 * decoder-only transformer: a block of n = 1..16 tokens (the last accepted
 * token plus n-1 drafted ones) goes through every layer against a paged KV
 * cache in one pass, the LM head gives one argmax per position, and the
 * greedy accept rule returns how many drafts match.  The same kernels run a
 * kept-layer subset of the model as a layer-skip self-speculative draft with
 * shared weights, and MoE layers read their routed experts either once per
 * (token, slot) or once per pass.
 *
 * Sources (by page title and section):
 *  - "I built self-speculative decoding for MLX ..." (MLX self-speculation
 *    post), "Code -> the implementation": the draft is the model with a
 *    contiguous middle block of layers skipped, sharing weights; greedy
 *    self-speculation is lossless.
 *  - "LayerSkip: Enabling Early Exit Inference and Self-Speculative Decoding",
 *    4.3.1-4.3.2: drafting with a layer subset, verifying all drafts in one
 *    parallel pass, accepting up to the first mismatch plus the verifier's
 *    token.
 *  - "mlx-dflash" README, "Architecture" and "Apple Silicon Optimizations":
 *    verify [last_token] + drafts in one pass (block of 16), greedy cumprod
 *    match, advance by accept_len + 1, crop caches on rejection, keep token
 *    ids on the device.
 *  - "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel
 *    Bandwidth and the Best Draft Length" (abstract): per-slot engines read an
 *    expert once per (token, slot), deduplicating engines once per pass.
 *
 * Conventions for every call:
 *  - Pointers named d_* are device pointers; all other pointers are host
 *    pointers.  Device work is enqueued on the handle's CUDA stream and is
 *    asynchronous unless stated; the caller synchronises that stream before
 *    reading outputs.
 *  - Argument errors are detected on the host, return a status, change no
 *    state and enqueue nothing.  spec_last_error() then describes the error
 *    (thread-local string, valid until the next call on that thread).
 *  - Weights are bfloat16, row-major [out_features][in_features].  Logits are
 *    float32.  Token ids are int32 in [0, vocab).
 *  - The library owns its packed weight copies, KV caches and scratch; the
 *    caller owns every buffer it passes in.
 *  - A device-side wait that gives up (bounded spin) records SPEC_ERR_TIMEOUT
 *    in the handle; the next call that synchronises (spec_kv_len,
 *    spec_check_error) reports it.
 */
#ifndef SPEC_H
#define SPEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_MAX_BLOCK 16 /* largest verify block n (DFlash README: block_size=16) */

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* bad pointer, size, shape or id                  */
    SPEC_ERR_CAPACITY = 2,    /* the pass would run past max_ctx                  */
    SPEC_ERR_STATE = 3,       /* call not valid in the handle's current state     */
    SPEC_ERR_CUDA = 4,        /* a CUDA runtime call failed (message has details) */
    SPEC_ERR_TIMEOUT = 5,     /* a bounded device wait gave up                    */
    SPEC_ERR_OOM = 6          /* device allocation failed                         */
} spec_status;

enum { SPEC_MOE_PER_SLOT = 0, SPEC_MOE_DEDUP = 1 };
enum { SPEC_CACHE_TARGET = 0, SPEC_CACHE_DRAFT = 1 };

/* Model shape.  A dense model has n_experts = 0.  In an MoE model, layers
 * l >= first_moe_layer use a softmax router over n_experts, top_k routed
 * SwiGLU experts of width expert_ffn and n_shared_experts shared experts of
 * the same width; earlier layers use a dense SwiGLU FFN of width ffn_dim.
 * Shape rules (checked): d_model is a multiple of 128 up to 8192; n_heads*head_dim,
 * ffn_dim and expert_ffn are multiples of 64; head_dim is 64 or 128; n_heads is a multiple of
 * n_kv_heads with at most 4 query heads per kv head; n_experts <= 64;
 * top_k <= 8; 1 <= max_ctx <= 65536. */
typedef struct spec_model_config {
    int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    float rope_theta; /* RoPE base (rotate-half pairing) */
    float norm_eps;   /* RMSNorm epsilon                 */
    int32_t tied_embeddings;
    int32_t n_experts, top_k, expert_ffn, n_shared_experts, first_moe_layer;
    int32_t max_ctx; /* KV capacity in tokens per cache */
} spec_model_config;

/* Device pointers of one layer's weights.  Dense-FFN layers set w_gate,
 * w_up, w_down; MoE layers set router and the host arrays e_* (n_experts
 * device pointers each) and s_* (n_shared_experts device pointers each). */
typedef struct spec_layer_weights {
    const void* attn_norm; /* [d]                     */
    const void* ffn_norm;  /* [d]                     */
    const void* wq;        /* [n_heads*head_dim][d]    */
    const void* wk;        /* [n_kv_heads*head_dim][d] */
    const void* wv;        /* [n_kv_heads*head_dim][d] */
    const void* wo;        /* [d][n_heads*head_dim]    */
    const void* w_gate;    /* [ffn_dim][d]             */
    const void* w_up;      /* [ffn_dim][d]             */
    const void* w_down;    /* [d][ffn_dim]             */
    const void* router;    /* [n_experts][d]           */
    const void* const* e_gate; /* [n_experts] -> [expert_ffn][d] */
    const void* const* e_up;   /* [n_experts] -> [expert_ffn][d] */
    const void* const* e_down; /* [n_experts] -> [d][expert_ffn] */
    const void* const* s_gate; /* [n_shared]  -> [expert_ffn][d] */
    const void* const* s_up;   /* [n_shared]  -> [expert_ffn][d] */
    const void* const* s_down; /* [n_shared]  -> [d][expert_ffn] */
} spec_layer_weights;

typedef struct spec_weights {
    const void* embed;      /* [vocab][d]                          */
    const void* lm_head;    /* [vocab][d], NULL when tied to embed */
    const void* final_norm; /* [d]                                 */
    const spec_layer_weights* layers; /* host array [n_layers]     */
} spec_weights;

typedef struct spec_model* spec_handle;

/* Build a model on the current CUDA device.
 * Repacks every weight into the library's streaming layout (library-owned
 * device memory), allocates the target KV cache (all layers) and the draft KV
 * cache (kept layers), and synchronises `cuda_stream` before returning, so
 * the caller may free its weight buffers afterwards.
 * draft_layers: host array of n_draft_layers increasing layer indices, the
 * kept layers of the self-speculative draft (first and last layer kept); NULL
 * or 0 layers means no draft.  cuda_stream: a cudaStream_t (NULL = legacy
 * default stream).  On success *out holds the handle. */
spec_status spec_model_create(const spec_model_config* cfg, const spec_weights* w, const int32_t* draft_layers,
                              int32_t n_draft_layers, void* cuda_stream, spec_handle* out);

/* Free everything the handle owns.  Synchronises its stream. */
spec_status spec_model_destroy(spec_handle h);

/* Replace the draft's kept-layer plan (same rules as in create) and empty the
 * draft cache.  Synchronous. */
spec_status spec_set_draft_plan(spec_handle h, const int32_t* draft_layers, int32_t n_draft_layers);

/* Change the stream later calls enqueue on. */
spec_status spec_set_stream(spec_handle h, void* cuda_stream);

/* Prefill: run d_tokens[0..m) at positions len..len+m-1 of the TARGET cache
 * (all layers) and, when a draft plan exists, of the DRAFT cache, in blocks
 * of up to 16 tokens.  Writes the target's argmax at the last position to
 * d_next_token[0].  Both caches must hold the same length before the call. */
spec_status spec_prefill(spec_handle h, const int32_t* d_tokens, int32_t m, int32_t* d_next_token);

/* One draft step (MLX post: the draft is the kept-layer subset): run
 * d_tokens[0..n), n in {1, 2}, at the DRAFT cache's next positions through the
 * draft plan, append their k/v, and write the argmax of the last position to
 * d_draft_token[0].  n = 2 catches the draft up on a token it has not seen
 * (after a fully accepted block) or re-feeds the token at the rolled-back
 * position. */
spec_status spec_draft_step(spec_handle h, const int32_t* d_tokens, int32_t n, int32_t* d_draft_token);

/* The verify pass (LayerSkip 4.3.2; DFlash README "Verify" and "Accept").
 * d_block[0..n): the last accepted token followed by n-1 drafts, n in 1..16,
 * placed at TARGET positions p..p+n-1 where p is the target cache length.
 * Every layer runs on all n positions in one pass and appends their k/v.
 * Outputs:
 *   d_argmax[0..n)  argmax of each position's logits (lowest id on ties);
 *   d_accept_len[0] number of leading j < n-1 with d_block[j+1] == d_argmax[j];
 *   d_logits_opt    NULL or [n][vocab] float32 logits;
 *   d_expert_ids_opt NULL or [n_layers][n][top_k] int32 routed ids (MoE; -1 on
 *                   dense layers);
 *   d_next_pair_opt NULL or int32[2] = {d_block[k], d_argmax[k]} with
 *                   k = accept_len: the token at the last kept position and the
 *                   new last accepted token, ready for spec_draft_step(n=2).
 *                   May alias d_block - 1 (written after the block is read).
 * The cache is NOT rolled back; call spec_kv_rollback afterwards. */
spec_status spec_verify_step(spec_handle h, const int32_t* d_block, int32_t n, int32_t* d_argmax,
                             int32_t* d_accept_len, float* d_logits_opt, int32_t* d_expert_ids_opt,
                             int32_t* d_next_pair_opt);

/* KV rollback (DFlash README: caches cropped precisely on rejection).
 * which = SPEC_CACHE_TARGET or SPEC_CACHE_DRAFT.
 * new_len >= 0: keep positions [0, new_len); new_len must not exceed the
 *   length the host knows the cache may hold.
 * new_len = -1: device-side rollback after the last spec_verify_step with
 *   k = its accept_len and p its first position: TARGET keeps p+k+1
 *   positions, DRAFT keeps min(p+k, its length) positions (one less than the
 *   target, so the next spec_draft_step(n=2) re-feeds the last kept token and
 *   the new one without a host round trip). */
spec_status spec_kv_rollback(spec_handle h, int32_t which, int32_t new_len);

/* MoE expert-read mode: SPEC_MOE_PER_SLOT (one read per token and slot) or
 * SPEC_MOE_DEDUP (one read per distinct expert per pass).  Both give
 * bitwise identical outputs.  The shared experts are read once per pass in
 * either mode. */
spec_status spec_moe_mode(spec_handle h, int32_t mode);

/* Shared prefix cache (LayerSkip summary, section 4.3.3, "Single KV
 * Cache").  The draft plan's leading layers 0..E-1 (E = the length of its
 * contiguous prefix 0, 1, 2, ...) compute exactly what the target computes
 * for the same tokens, so with enable != 0 the draft uses the target's KV
 * cache for them and keeps its own cache only for its other layers (E fewer
 * slots are allocated).  Values the draft writes ahead of the target are the
 * ones the target's verify writes again (the passes are batch-invariant).
 * Reallocates the draft cache and sets its length to 0 (prefill again);
 * drops captured launch sequences; synchronises the stream.  SPEC_ERR_STATE
 * without a draft plan.  A later spec_set_draft_plan keeps the setting. */
spec_status spec_share_prefix(spec_handle h, int32_t enable);

/* Hidden-state taps (mlx-dflash README, "Architecture": the draft's context
 * features are taken from the target's hidden states at chosen layers).
 * After this call every target verify pass also writes, for each of its n
 * rows, the residual stream after layer layers[t] (fp32, the value the next
 * layer's norm reads) to d_out[(t * 16 + row) * d_model ...].  Rows n..15
 * are left untouched; prefill and draft passes write nothing.
 *   layers  host array of `count` distinct layer indices in [0, n_layers);
 *   count   0..n_layers; 0 switches the taps off (layers, d_out may be NULL);
 *   d_out   device buffer of count * 16 * d_model floats, 16-byte aligned,
 *           CALLER-owned; it must stay valid while taps are on.
 * Synchronises the stream and drops captured launch sequences.  Errors:
 * SPEC_ERR_INVALID_ARG (range, duplicates, alignment, NULL), state unchanged. */
spec_status spec_set_taps(spec_handle h, const int32_t* layers, int32_t count, float* d_out);

/* Block-draft conditioning (mlx-dflash README, "Architecture": the target's
 * hidden states at chosen layers -> fc -> context features; the draft's
 * attention is full over the context).  For a handle that serves as the
 * block draft, with the reading that each of its layers derives the keys and
 * values of a context position from that position's feature exactly as it
 * does from a token's residual stream (its input norm, k/v projections, RoPE
 * at the position):
 *
 * spec_set_context_fc: d_fc = bf16 [d_model][n_in * d_model] row-major
 *   (device, caller-owned, read once and repacked; input index t*d_model + i
 *   is element i of tap t).  n_in in 1..8.  Once per handle (SPEC_ERR_STATE
 *   on a second call).  Synchronises the stream.
 *
 * spec_context_append: d_taps = fp32 [n_in][16][d_model] (the layout
 *   spec_set_taps writes), rows 0..m-1 used, m in 1..16, 16-byte aligned.
 *   feature[r] = fc . bf16(concat_t taps[t][r]) (fp32); then every layer
 *   writes k/v of positions p..p+m-1 of the TARGET cache (p its length) and
 *   the length becomes p+m.  Asynchronous on the handle's stream.  Errors:
 *   SPEC_ERR_STATE (no fc), SPEC_ERR_INVALID_ARG, SPEC_ERR_CAPACITY.
 * The draft block itself is then an ordinary spec_verify_step of
 * [last token, mask x 15] on this handle, followed by spec_kv_rollback of
 * its TARGET cache to p+m. */
spec_status spec_set_context_fc(spec_handle h, const uint16_t* d_fc, int32_t n_in);
spec_status spec_context_append(spec_handle h, const float* d_taps, int32_t m);

/* Batched sequences (LayerSkip summary, "Critical Assessment": in batched
 * inference one verify pass serves several sequences, which raises the
 * flops per weight byte read).  One pass verifies the
 * blocks of nseq independent sequences: every weight is read once for all
 * nseq * n rows, while each sequence attends only to its own cache.
 *
 * spec_batch_reserve: allocates target caches for nseq (1..16) sequences of
 *   max_ctx positions each, next to the handle's own caches.  Once per
 *   handle (SPEC_ERR_STATE on a second call).  Synchronises the stream.
 * spec_batch_kv_load / spec_batch_kv_export: as spec_kv_load/export, for
 *   sequence `seq` (0..reserved-1) and layer `slot`.
 * spec_batch_set_len: sets sequence seq's length (synchronises the stream).
 * spec_batch_len: synchronises and returns sequence seq's device length.
 * spec_verify_batch: d_blocks = int32 [nseq][n] (sequence q's block: its
 *   last accepted token then n-1 drafts, at positions len_q .. len_q+n-1),
 *   nseq * n <= 16.  Outputs d_argmax [nseq][n], d_accept [nseq] (the greedy
 *   cumulative-product rule per sequence), d_logits_opt NULL or
 *   [nseq*n][vocab].  Each sequence's length then becomes len_q + accept_q + 1
 *   on the device (the rollback rule of spec_kv_rollback, applied here).
 *   Row j of sequence q is bitwise the row a single-sequence verify of the
 *   same block on the same cache gives.  Errors: SPEC_ERR_INVALID_ARG,
 *   SPEC_ERR_CAPACITY; state unchanged. */
spec_status spec_batch_reserve(spec_handle h, int32_t nseq);
spec_status spec_batch_kv_load(spec_handle h, int32_t seq, int32_t slot, const void* d_k, const void* d_v, int32_t ctx);
spec_status spec_batch_kv_export(spec_handle h, int32_t seq, int32_t slot, void* d_k, void* d_v, int32_t ctx);
spec_status spec_batch_set_len(spec_handle h, int32_t seq, int32_t len);
spec_status spec_batch_len(spec_handle h, int32_t seq, int32_t* out_len);
spec_status spec_verify_batch(spec_handle h, const int32_t* d_blocks, int32_t nseq, int32_t n, int32_t* d_argmax,
                              int32_t* d_accept, float* d_logits_opt);

/* Sampled verification (LayerSkip summary, 4.3.2 "Self-Verification": with
 * sampling, rejection sampling keeps the output distribution exactly the full
 * model's; the pages give the property, and the rule here is the standard
 * one of speculative sampling).  With p_j = softmax(target_logits[j] / T) and
 * q_j = softmax(draft_logits[j] / T), the draft x = d_block[j+1] (drawn from
 * q_j by the caller) is accepted when u_j * q_j(x) < p_j(x), tested in the log
 * domain from the logits; at the first rejection j the next token is drawn
 * from norm(max(0, p_j - q_j)) (from p_j where p_j == q_j), after a full
 * accept from p_{n-1}.  A draw with uniform u is the smallest index whose
 * running weight sum exceeds u times the total.
 *   d_target_logits  float32 [n][vocab] (e.g. spec_verify_step's logits);
 *   d_draft_logits   float32 [n-1][vocab] (e.g. spec_draft_step_logits'
 *                    rows), NULL only when n == 1;
 *   d_block          int32 [n]: the last accepted token, then the drafts;
 *   n                1..16; with n == 1 the call draws one token from p_0
 *                    (plain sampling, or a draft's own proposal);
 *   temperature      > 0 and finite;
 *   d_uniforms       float64 [n] in [0, 1): u_0 .. u_{n-2} for the accept
 *                    tests, then the draw's; CALLER-supplied, so a run is
 *                    reproducible and the random source is the caller's;
 *   d_accept_len[0]  the number of accepted drafts k;
 *   d_next_token[0]  the token drawn at position k.
 * Uses the handle's scratch (four small launches on its stream); the vocab
 * is the handle's.  Argument errors: SPEC_ERR_INVALID_ARG, nothing enqueued. */
spec_status spec_accept_sampled(spec_handle h, const float* d_target_logits, const float* d_draft_logits,
                                const int32_t* d_block, int32_t n, float temperature, const double* d_uniforms,
                                int32_t* d_accept_len, int32_t* d_next_token);

/* Thread-local description of the last error. */
const char* spec_last_error(void);

/* ---- inspection, test and benchmark calls ---- */

/* spec_draft_step that also writes the draft's logits: d_logits_opt NULL or
 * [n][vocab] float32, row i the logits of d_tokens[i] after the kept layers,
 * the final norm and the LM head (the row whose argmax spec_draft_step
 * returns is the last).  Same arguments, errors and state change otherwise. */
spec_status spec_draft_step_logits(spec_handle h, const int32_t* d_tokens, int32_t n, int32_t* d_draft_token,
                                   float* d_logits_opt);

/* Synchronise the stream and report a device-side error recorded by a
 * bounded wait (SPEC_ERR_TIMEOUT) or a CUDA error. */
spec_status spec_check_error(spec_handle h);

/* Synchronise the stream and return the device-side cache length. */
spec_status spec_kv_len(spec_handle h, int32_t which, int32_t* out_len);

/* Load keys/values of one cache slot (target: slot = layer; draft: slot =
 * index in the draft plan) at positions [0, ctx): d_k, d_v are bf16
 * [ctx][n_kv_heads][head_dim].  Sets nothing else; call spec_kv_set_len
 * afterwards. */
spec_status spec_kv_load(spec_handle h, int32_t which, int32_t slot, const void* d_k, const void* d_v, int32_t ctx);

/* Read back keys/values of one slot at positions [0, ctx) into bf16
 * [ctx][n_kv_heads][head_dim] buffers. */
spec_status spec_kv_export(spec_handle h, int32_t which, int32_t slot, void* d_k, void* d_v, int32_t ctx);

/* Set a cache's length (positions [0, len) are taken as valid). */
spec_status spec_kv_set_len(spec_handle h, int32_t which, int32_t len);

/* Force the routed experts of the next passes: d_ids is [n_layers][16][top_k]
 * int32 (rows of dense layers ignored; row j applies to block position j),
 * copied at the call; gates become the router probabilities at those ids.
 * NULL returns to computed top-k routing. */
spec_status spec_moe_force_routing(spec_handle h, const int32_t* d_ids);

/* Number of the library's kernel launches enqueued by the last call. */
int32_t spec_last_launch_count(spec_handle h);

/* Benchmark hook: while enabled, every streaming-GEMM launch is bracketed by
 * CUDA events on the handle's stream (this serialises those launches with
 * their neighbours).  enable = 0 stops recording. */
spec_status spec_profile_enable(spec_handle h, int32_t enable);

/* Synchronise the stream and return, for the recorded launches of one kind:
 * the summed event time in ms, the summed bytes and the launch count, and
 * drop those records.  kind = -1: every dense launch (GEMMs outside the expert
 * FFN); -2: all; 0..7: one GEMM epilogue kind.  Bytes are algorithmic (weights + activation operand + outputs,
 * each once); for expert launches they are the expert bytes the launch
 * requests (one expert per (token, slot) in per-slot mode, one per distinct
 * expert in dedup mode, counted from forced routing ids), plus each shared
 * expert once. */
spec_status spec_profile_read(spec_handle h, int32_t kind, double* total_ms, double* total_bytes, int32_t* launches);

/* Benchmark hook.  While enabled, every pass runs its kernels as separate
 * launches (no graph replay) and every GEMM and attention launch records
 * global-timer stamps (nanoseconds) per CTA: entry, inputs ready (after
 * waiting for the previous kernel), main work done (GEMM: last weight stage
 * consumed; attention: K/V slabs arrived), exit.  Stamps a kernel has no
 * point for are 0.
 * Each pass overwrites the previous record.  Allocates the trace buffer on
 * enable; synchronous. */
spec_status spec_trace_enable(spec_handle h, int32_t enable);

/* Copy the last traced pass's stamps ([nctas][nphase][4]) to the host array
 * out (capacity entries).  nphase is the number of traced launches; nctas is
 * 512 slots per launch (unused slots hold zeros).  Synchronises the stream. */
spec_status spec_trace_read(spec_handle h, long long* out, int32_t capacity, int32_t* nphase, int32_t* nctas);

/* Kind of each traced launch of the last traced pass (count
 * entries): 0..7 the GEMM epilogue kind (0 QKV, 1 residual, 2 SwiGLU, 3 LM
 * head, 4 router, 5 expert gate-up, 6 expert down, 7 store), 16 attention
 * partials, 17 attention chunk merge, 18 embedding, 19 accept. */
spec_status spec_trace_kinds(spec_handle h, int32_t* out, int32_t capacity, int32_t* count);

/* Greedy accept from caller-computed logits, without any device allocation.
 * The pages have no counterpart to this call.  It serves callers that cannot
 * allocate device memory where they need the accept decision: a process
 * whose memory pool already owns the device, a serving loop that forbids
 * allocation after warm-up, or a thread that must not stall the device with
 * cudaMalloc.  It computes what the accept step of spec_verify_step computes:
 * d_argmax[j] = argmax of row j of d_logits ([n][vocab] float32, lowest id on
 * ties) and d_accept_len[0] = number of leading j < n-1 with
 * d_block[j+1] == d_argmax[j]; the caller passes and owns all five buffers.
 * Limits: 1 <= n <= 16 and 1 <= vocab <= 2,097,152; other sizes, or a null
 * pointer, return SPEC_ERR_INVALID_ARG and enqueue nothing.
 * Scratch: a fixed 128 KB array inside the library, which every GPU that
 * loads the library holds until the process exits; no cudaMalloc, cudaFree or
 * allocating library routine is called.  The first call on a device looks up
 * that array's device address with the device current (and so does the first
 * call after a device reset, which gives the device a new context), so make
 * the first call on each device before any stream capture.  All calls on a device share the
 * array: calls whose kernels can overlap on the GPU (different streams with
 * no ordering between them) race; calls on one stream are ordered and safe.
 * Each call overwrites every scratch entry it reads, so nothing has to start
 * at zero.  Asynchronous on cuda_stream (a cudaStream_t, NULL = default). */
spec_status spec_accept_from_logits_noalloc(const float* d_logits, int32_t n, int32_t vocab, const int32_t* d_block,
                                            int32_t* d_argmax, int32_t* d_accept_len, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_H */
