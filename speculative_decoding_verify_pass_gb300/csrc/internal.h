// Internal interface between the host runtime (api.cu) and the kernel
// translation units.  Plain structs of device pointers and sizes, one
// launcher per kernel family; every launcher enqueues on the given stream with
// programmatic dependent launch and returns the CUDA error of the launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace sv {

// Epilogue kinds of the streaming GEMM.
enum EpiKind : int {
    EPI_QKV = 0,            // rstd scale, RoPE on q/k, q -> qbuf, k/v -> paged cache
    EPI_RESID = 1,          // x += acc; next-norm operand + sum-of-squares partials
    EPI_SWIGLU = 2,         // silu(rstd*gate) * (rstd*up) -> next operand
    EPI_LMHEAD = 3,         // rstd scale, optional logits, per-tile argmax partials
    EPI_ROUTER = 4,         // softmax over experts, top-k ids and gates
    EPI_EXPERT_SWIGLU = 5,  // per work item: SwiGLU rows of its tokens -> item operand
    EPI_EXPERT_DOWN = 6,    // per work item: rows of its tokens -> y_slot
    EPI_STORE = 7           // acc -> fp32 rows (shared-expert output)
};

// A weight matrix [N][K] repacked as tiles of 128 rows x 64 k in the order the
// tensor core reads them: [tile][kblock][8-row group (16)][8-k group (8)][row (8)][8 bf16].
// Launch tracing: a traced launch gets kTraceCtas x 4 slots; CTA c writes
// global-timer stamps at trace[c*4 + k]: k = 0 entry, 1 inputs ready (after
// the dependency wait), 2 main work done, 3 exit (0 where a kernel has no such
// point).
constexpr int kTraceCtas = 512;
// Kind codes of traced launches other than GEMMs (GEMMs report their EPI_* kind).
constexpr int kTraceAttnPartial = 16, kTraceAttnCombine = 17, kTraceEmbed = 18, kTraceAccept = 19;

__device__ __forceinline__ long long trace_clock() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

struct PackedMat {
    uint8_t* p = nullptr;
    int N = 0, K = 0, T = 0, KBs = 0;
    size_t bytes() const { return (size_t)T * KBs * kStageWBytes; }
};

struct GemmParams {
    const uint8_t* W;          // packed weights (items mode: expert e at W + e*w_item_stride)
    long long w_item_stride;
    int T, KBs, N;
    const uint8_t* X;          // fragment-ordered operand [KBs][2 KB bf16 | 4 KB fp32] (items: + item*x_item_stride)
    int x_f32;                 // operand holds fp32 x*gain; rstd is applied and bf16 rounding done on read
    long long x_item_stride;
    int n;                     // tokens (1..16)
    int items_mode;            // 0: stream-K over T*KBs; 1: (item, tile) units
    int grid;                  // CTAs launched
    float* partials;           // stream-K partial tiles [2*grid][128*16]
    int* counters;             // [T], zero between launches
    DevState* st;
    int which;                 // cache whose length gives the positions
    int epi;
    // input normalisation (rstd applied in the epilogue)
    const float* ss_in;        // [16][ss_in_tiles] sum-of-squares partials of x
    int ss_in_tiles;
    int norm_dim;              // 0: no normalisation
    float norm_eps;
    // EPI_QKV
    int n_heads, n_kv_heads, head_dim;
    int tile0;                 // first 128-row tile of the full q|k|v matrix that W starts at (k/v only: q rows skipped)
    // batched sequences (seq_len != null): row r is token r % rows_per_seq of
    // sequence r / rows_per_seq, at position seq_len[seq] + token, whose
    // logical pages start at seq * seq_pages of the block table
    const int* seq_len;
    int rows_per_seq, seq_pages;
    const float2* rope;        // [max_pos][head_dim/2] (cos, sin)
    uint16_t* qbuf;            // [16][n_heads*head_dim]
    uint16_t* kpool;           // this layer's pages [page][n_kv_heads][64][head_dim]
    uint16_t* vpool;
    const int* block_table;
    // EPI_RESID
    float* x;                  // [16][d]
    int d;
    const uint16_t* g_next;    // gain of the norm that consumes x next
    uint8_t* xf_out;           // next GEMM's operand
    float* ss_out;             // [16][d/128]
    float* tap;                // optional: the new residual rows, fp32 [16][d] (hidden-state tap)
    // EPI_LMHEAD
    float* logits;             // optional [n][vocab]
    float* amax_val;           // [16][T]
    int* amax_idx;
    // EPI_ROUTER / experts
    int n_experts, top_k;
    int n_shared;              // shared experts: work items n_experts.. of every expert launch, all tokens
    int* route_ids;            // [16][top_k]
    float* route_gates;
    const int* forced_ids;     // [16][top_k] or null
    int* debug_ids;            // [n][top_k] or null
    int moe_mode;
    float* y_slot;             // [16][top_k + n_shared][d]
    float* y_store;            // [16][N] (EPI_STORE)
    uint8_t* xe;               // expert-down operands [item][KBs_down][2 KB]
    long long xe_stride;
    long long* trace;          // optional: this launch's [kTraceCtas][4] stamps (see kTraceCtas)
};

struct AttnParams {
    const uint16_t* qbuf;      // [16][Hq*hd]
    const uint16_t* kpool;     // [page][Hkv][64][hd]
    const uint16_t* vpool;
    const int* block_table;
    float* part_o;             // [Hkv][nch][64][hd]
    float2* part_ml;           // [Hkv][nch][64] (max (log2 domain), sum)
    uint8_t* xf_out;           // O-projection operand
    DevState* st;
    int which, n, n_heads, n_kv_heads, head_dim, nch;
    int num_sms;               // the partial kernel's grid: about one CTA per SM
    int groups;                // S: chunk c's partial is group c mod S's (fixed per model, <= nch)
    float scale_log2;          // log2(e) / sqrt(hd)
    // batched sequences (seq_len != null): n rows per sequence, nseq of them;
    // sequence s: positions from seq_len[s], logical pages from s * seq_pages,
    // query rows s*n.., partials at s * n_kv_heads * nch * 64 rows
    const int* seq_len;
    int nseq, seq_pages;
    long long* trace;          // optional stamps of the partial kernel, then of the combine kernel
};

// Launchers (stream, PDL).  Return cudaSuccess or the launch error.
cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl);
cudaError_t gemm_configure(int device);  // shared-memory opt-in, once per device
cudaError_t attention_configure(int device);
int gemm_threads();
size_t gemm_smem_bytes();

struct EmbedParams {
    const int* tokens;         // device [n]
    const uint16_t* embed;     // [V][d]
    int n, d, vocab;
    float* x;
    const uint16_t* g_next;
    uint8_t* xf_out;
    float* ss_out;
    DevState* st;
};
cudaError_t launch_embed(const EmbedParams& p, cudaStream_t s, bool pdl);

struct CombineParams {           // MoE: x += sum_s gate*y_slot[s] + sum_t y_slot[top_k + t]
    float* x;
    const float* y_slot;       // [16][top_k + n_shared][d]
    const float* gates;
    int n, d, top_k, n_shared;
    const uint16_t* g_next;
    uint8_t* xf_out;
    float* ss_out;
    float* tap;                // optional: the new residual rows, fp32 [16][d] (hidden-state tap)
};
cudaError_t launch_moe_combine(const CombineParams& p, cudaStream_t s, bool pdl);

// Block-draft conditioning (context append): the tapped hidden states
// [n_in][16][d] as one fp32 operand of K = n_in*d (xfrag32_offset order, gain 1),
// and fp32 rows [16][d] as a layer's normalised operand (x*gain + sum of
// squares, as the embedding kernel writes them).
struct ConcatParams {
    const float* taps;         // [n_in][16][d]
    int n_in, d;
    uint8_t* xf_out;           // [n_in*d/64][4 KB]
};
cudaError_t launch_concat_taps(const ConcatParams& p, cudaStream_t s, bool pdl);
struct RowsParams {
    float* x;                  // [16][d], rows < n read (and rewritten unchanged)
    int n, d;
    const uint16_t* g_next;
    uint8_t* xf_out;
    float* ss_out;
};
cudaError_t launch_rows_operand(const RowsParams& p, cudaStream_t s, bool pdl);

enum AcceptMode : int { ACC_VERIFY = 0, ACC_DRAFT = 1, ACC_PREFILL = 2, ACC_BATCH = 3 };
struct AcceptParams {
    const float* amax_val;     // [16][T]
    const int* amax_idx;
    int T, n, mode, which;
    const int* block;          // verify: d_block
    int* out_argmax;           // verify: [n]
    int* out_accept;           // verify: [1]
    int* out_pair;             // verify: [2] or null
    int* out_token;            // draft / prefill: [1]
    DevState* st;
    // ACC_BATCH: nseq sequences of n / nseq rows; out_accept[nseq]; each
    // sequence keeps seq_len[s] + accept + 1 positions
    int* seq_len;
    int nseq;
};
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t s, bool pdl);

// len[which] += n (a pass without LM head).
cudaError_t launch_advance(DevState* st, int which, int n, cudaStream_t s, bool pdl);
// Rollback: new_len >= 0 sets it; -1 applies the device rule of spec_kv_rollback.
cudaError_t launch_rollback(DevState* st, int which, int new_len, cudaStream_t s, bool pdl);

struct PackSrc {
    const uint16_t* src[4];
    int rows[4];               // rows of each source
    int cols;                  // K of each source
    int nsrc;
    int mode;                  // 0 row concat, 1 gate/up interleave by 64
};
cudaError_t launch_pack(const PackSrc& s, const PackedMat& m, cudaStream_t st);

// Logical [ctx][Hkv][hd] bf16 <-> paged pool in the K (is_v false) or V
// page layout (kv_off_k / kv_off_v).
cudaError_t launch_kv_io(uint16_t* pool, const int* block_table, uint16_t* logical, int ctx, int hkv, int hd,
                         bool to_pool, bool is_v, cudaStream_t s);

// Sampled verification (sampling.cu): rejection-sampling accept from the
// target's and the draft's logits and caller-supplied uniforms.
struct SampleParams {
    const float* target;       // [n][vocab] target logits
    const float* draft;        // [n-1][vocab] draft logits (null when n == 1)
    const int* block;          // [n]: last accepted token, then the drafts
    const double* uniforms;    // [n]: one per accept test, then the draw's
    int n, vocab, chunks;
    float temperature;
    float2* stats;             // [2n-1][chunks] (max of l/T, sum of exp(l/T - max)) per chunk
    double2* row_stat;         // [2n-1] (max, log of the sum) per row
    double* chunk_sum;         // [2][chunks] the draw's weight sums per chunk (and p's)
    int* decision;             // [2]: row k of the draw, and 1 (from p) or 0 (residual)
    int* out_accept;
    int* out_token;
};
int sample_chunks(int vocab);
cudaError_t launch_sample_accept(const SampleParams& p, cudaStream_t s, bool pdl);

// Sets the thread-local message returned by spec_last_error (api.cu).
void set_last_error(const char* msg);

}  // namespace sv
