// Host runtime of the verify-pass library: the C ABI of include/spec.h.
//
// A handle owns the packed weights, the target and draft KV caches (paged,
// 64 positions per page, identity block table over a pool sized for
// max_ctx), the activation and scratch buffers, and a small device state
// block with the cache lengths.  Every pass is a fixed sequence of kernel
// launches on the handle's stream with programmatic dependent launch; kernels
// read positions from the device state, so no host value changes between
// steps and a decode loop needs no host round trip.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "internal.h"
#include "spec.h"

using namespace sv;

namespace {

thread_local std::string g_err;

spec_status fail(spec_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

#define CU(call)                                                                                       \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess)                                                                         \
            return fail(e_ == cudaErrorMemoryAllocation ? SPEC_ERR_OOM : SPEC_ERR_CUDA, "%s: %s (%s:%d)", #call, \
                        cudaGetErrorString(e_), __FILE__, __LINE__);                                   \
    } while (0)

enum PassMode { PASS_VERIFY, PASS_DRAFT, PASS_PREFILL_LAST, PASS_PREFILL_MID };

struct LayerW {
    bool moe = false;
    PackedMat qkv, o, gu, down;         // dense FFN in gu/down
    PackedMat router;                   // MoE
    PackedMat egu, edown;               // geometry of one expert; routed experts then shared ones, at a fixed stride
    long long egu_stride = 0, edown_stride = 0;
    uint16_t* attn_norm = nullptr;
    uint16_t* ffn_norm = nullptr;
};

}  // namespace

struct spec_model {
    spec_model_config c{};
    cudaStream_t stream = nullptr;
    int device = 0, num_sms = 0;
    bool pdl = true;
    std::vector<LayerW> L;
    PackedMat lm;
    uint16_t* embed = nullptr;
    uint16_t* final_norm = nullptr;
    float2* rope = nullptr;
    int max_pages = 0, nch = 0;
    int* block_table = nullptr;
    size_t pool_elems = 0;              // elements of one layer's K (or V) pool
    uint16_t *kt = nullptr, *vt = nullptr, *kd = nullptr, *vd = nullptr;
    std::vector<int> plan_full, plan_draft;
    float* x = nullptr;
    uint8_t *xf_norm = nullptr, *xf_o = nullptr, *xf_down = nullptr, *xe = nullptr;
    long long xe_stride = 0;
    uint16_t* qbuf = nullptr;
    float* ss = nullptr;
    float* attn_o = nullptr;
    float2* attn_ml = nullptr;
    float* gpart = nullptr;
    int* gcnt = nullptr;
    int max_T = 0;
    float* amax_val = nullptr;
    int* amax_idx = nullptr;
    int* route_ids = nullptr;
    float* route_gates = nullptr;
    int* forced = nullptr;
    bool forced_on = false;
    // batched sequences (spec_batch_reserve): target caches of their own
    int bat_cap = 0;                    // sequences reserved
    uint16_t *kb = nullptr, *vb = nullptr;   // [layer][bat_cap * max_pages pages][Hkv][64][hd]
    int* bt_b = nullptr;                // identity table over bat_cap * max_pages pages
    int* seq_len = nullptr;             // device [16]
    std::vector<int> bat_host_len;      // upper bounds of the device lengths
    float* battn_o = nullptr;           // attention partials of all sequences
    float2* battn_ml = nullptr;
    int bat_nseq = 0;                   // > 0 while a batched pass is built
    PackedMat ctx_fc;                   // block-draft conditioning: fc [d][ctx_n_in*d]
    int ctx_n_in = 0;
    uint8_t* xf_ctx = nullptr;          // its operand: the concatenated taps, fp32 (xfrag32_offset order)
    std::vector<int> tap_of_layer;      // hidden-state taps: slot of each layer in tap_out, or -1
    float* tap_out = nullptr;           // caller's [count][16][d_model] fp32 buffer
    int tap_count = 0;
    float* y_slot = nullptr;
    DevState* st = nullptr;
    int moe_mode = SPEC_MOE_DEDUP;
    int host_len[2] = {0, 0};   // upper bounds of the device lengths
    bool len_exact[2] = {true, true};
    int launches = 0;
    long long* trace = nullptr;         // phase timestamps of the last traced pass
    size_t trace_cap = 0;
    bool tracing = false;               // the current pass records launch stamps
    std::vector<int32_t> trace_kinds;   // per traced launch
    bool profiling = false;
    bool use_graphs = true;             // replay captured launch sequences (SPEC_GRAPHS=0: direct launches)
    cudaStream_t cap_stream = nullptr;  // private stream used only for capture
    struct GraphEntry {
        cudaGraphExec_t exec;
        int launches;
    };
    std::map<std::vector<uintptr_t>, GraphEntry> graphs;
    struct ProfRec {
        cudaEvent_t a, b;
        double bytes;
        int kind;   // EPI_* of the GEMM launch
    };
    std::vector<int32_t> forced_host;   // host copy of forced routing ids
    std::vector<ProfRec> prof;
    std::vector<void*> allocs;
    std::vector<void*> draft_allocs;
    float2* samp_stats = nullptr;       // sampled verification scratch (sampling.cu)
    double2* samp_rows = nullptr;
    double* samp_sums = nullptr;
    int* samp_decision = nullptr;
    bool share_prefix = false;          // the draft's leading layers 0..n_shared-1 use the target's caches
    int n_shared = 0;                   // layers the draft plan shares with the target as a contiguous prefix
};

namespace {
}  // namespace

void sv::set_last_error(const char* msg) { g_err = msg ? msg : ""; }

namespace {

spec_status dalloc(spec_model* h, void** p, size_t bytes, std::vector<void*>* owner = nullptr) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) return fail(SPEC_ERR_OOM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
    (owner ? *owner : h->allocs).push_back(*p);
    e = cudaMemsetAsync(*p, 0, bytes, h->stream);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

template <class T>
spec_status dalloc_t(spec_model* h, T** p, size_t count, std::vector<void*>* owner = nullptr) {
    return dalloc(h, reinterpret_cast<void**>(p), count * sizeof(T), owner);
}

PackedMat geometry(int N, int K) {
    PackedMat m;
    m.N = N;
    m.K = K;
    m.T = (N + kTileRows - 1) / kTileRows;
    m.KBs = K / kKBlock;
    return m;
}

spec_status pack_into(spec_model* h, PackedMat& m, const PackSrc& src) {
    CU(launch_pack(src, m, h->stream));
    if (m.T > h->max_T) h->max_T = m.T;
    return SPEC_OK;
}

spec_status alloc_packed(spec_model* h, PackedMat& m, int N, int K) {
    m = geometry(N, K);
    spec_status s = dalloc(h, reinterpret_cast<void**>(&m.p), m.bytes());
    if (m.T > h->max_T) h->max_T = m.T;
    return s;
}

PackSrc src_rows(std::initializer_list<const void*> ptrs, std::initializer_list<int> rows, int cols, int mode) {
    PackSrc s{};
    int i = 0;
    for (const void* p : ptrs) s.src[i++] = static_cast<const uint16_t*>(p);
    i = 0;
    for (int r : rows) s.rows[i++] = r;
    s.nsrc = i;
    s.cols = cols;
    s.mode = mode;
    return s;
}

spec_status copy_vec(spec_model* h, uint16_t** dst, const void* src, size_t count) {
    spec_status s = dalloc_t(h, dst, count);
    if (s != SPEC_OK) return s;
    CU(cudaMemcpyAsync(*dst, src, count * 2, cudaMemcpyDeviceToDevice, h->stream));
    return SPEC_OK;
}

spec_status validate_config(const spec_model_config* c) {
    if (!c) return fail(SPEC_ERR_INVALID_ARG, "null config");
    if (c->n_layers < 1 || c->d_model < 128 || c->d_model % 128 || c->d_model > 8192)
        return fail(SPEC_ERR_INVALID_ARG, "d_model must be a multiple of 128 in 128..8192");
    if (c->head_dim != 64 && c->head_dim != 128) return fail(SPEC_ERR_INVALID_ARG, "head_dim must be 64 or 128");
    if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads || c->n_heads / c->n_kv_heads > 4)
        return fail(SPEC_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads with at most 4 per kv head");
    if ((c->n_heads * c->head_dim) % 64) return fail(SPEC_ERR_INVALID_ARG, "n_heads*head_dim must be a multiple of 64");
    if (c->vocab < 1) return fail(SPEC_ERR_INVALID_ARG, "vocab must be positive");
    if (c->max_ctx < 1 || c->max_ctx > 65536) return fail(SPEC_ERR_INVALID_ARG, "max_ctx must be in 1..65536");
    if (!(c->norm_eps > 0.f) || !(c->rope_theta > 1.f)) return fail(SPEC_ERR_INVALID_ARG, "bad norm_eps or rope_theta");
    const bool has_dense = c->n_experts == 0 || c->first_moe_layer > 0;
    if (has_dense && (c->ffn_dim < 64 || c->ffn_dim % 64)) return fail(SPEC_ERR_INVALID_ARG, "ffn_dim must be a positive multiple of 64");
    if (c->n_experts < 0 || c->n_experts > kMaxExperts) return fail(SPEC_ERR_INVALID_ARG, "n_experts must be in 0..64");
    if (c->n_experts > 0) {
        if (c->top_k < 1 || c->top_k > kMaxTopK || c->top_k > c->n_experts) return fail(SPEC_ERR_INVALID_ARG, "top_k must be in 1..min(8, n_experts)");
        if (c->expert_ffn < 64 || c->expert_ffn % 64) return fail(SPEC_ERR_INVALID_ARG, "expert_ffn must be a positive multiple of 64");
        if (c->n_shared_experts < 0 || c->n_shared_experts > kMaxShared)
            return fail(SPEC_ERR_INVALID_ARG, "n_shared_experts must be 0..%d", kMaxShared);
        if (c->first_moe_layer < 0) return fail(SPEC_ERR_INVALID_ARG, "first_moe_layer must be >= 0");
    }
    return SPEC_OK;
}

spec_status validate_plan(const spec_model* h, const int32_t* layers, int32_t n) {
    if (n == 0) return SPEC_OK;
    if (!layers || n < 0 || n > h->c.n_layers) return fail(SPEC_ERR_INVALID_ARG, "bad draft plan size");
    for (int i = 0; i < n; ++i) {
        if (layers[i] < 0 || layers[i] >= h->c.n_layers) return fail(SPEC_ERR_INVALID_ARG, "draft layer %d out of range", layers[i]);
        if (i && layers[i] <= layers[i - 1]) return fail(SPEC_ERR_INVALID_ARG, "draft layers must increase");
    }
    if (layers[0] != 0 || layers[n - 1] != h->c.n_layers - 1)
        return fail(SPEC_ERR_INVALID_ARG, "draft plan must keep the first and the last layer");
    return SPEC_OK;
}

// The K (kv = 0) or V (kv = 1) pool of cache `which`, slot `si` (plan index;
// the layer itself for the target).  With a shared prefix the draft's first
// n_shared slots are the target's pools of the same layers (LayerSkip
// summary 4.3.3: one KV cache for the layers both stages run identically).
uint16_t* kv_pool(spec_model* h, int which, int si, int kv) {
    if (which == 0) return (kv ? h->vt : h->kt) + h->pool_elems * si;
    if (h->share_prefix && si < h->n_shared) return (kv ? h->vt : h->kt) + h->pool_elems * si;
    const int own = h->share_prefix ? si - h->n_shared : si;
    return (kv ? h->vd : h->kd) + h->pool_elems * own;
}

spec_status alloc_draft(spec_model* h, const int32_t* layers, int32_t n) {
    for (void* p : h->draft_allocs) cudaFree(p);
    h->draft_allocs.clear();
    h->kd = h->vd = nullptr;
    h->plan_draft.assign(layers, layers + n);
    h->n_shared = 0;
    while (h->n_shared < n && layers[h->n_shared] == h->n_shared) ++h->n_shared;
    const int own = h->share_prefix ? n - h->n_shared : n;   // slots the draft keeps for itself
    if (own > 0) {
        spec_status s;
        if ((s = dalloc_t(h, &h->kd, h->pool_elems * own, &h->draft_allocs)) != SPEC_OK) return s;
        if ((s = dalloc_t(h, &h->vd, h->pool_elems * own, &h->draft_allocs)) != SPEC_OK) return s;
    }
    h->host_len[1] = 0;
    h->len_exact[1] = true;
    return SPEC_OK;
}

// Refresh the host's view of the device lengths (synchronises the stream).
spec_status sync_lengths(spec_model* h) {
    CU(cudaStreamSynchronize(h->stream));
    DevState st;
    CU(cudaMemcpy(&st, h->st, sizeof(st), cudaMemcpyDeviceToHost));
    h->host_len[0] = st.len[0];
    h->host_len[1] = st.len[1];
    h->len_exact[0] = h->len_exact[1] = true;
    return SPEC_OK;
}

spec_status check_capacity(spec_model* h, int which, int n) {
    if (h->host_len[which] + n <= h->c.max_ctx) return SPEC_OK;
    if (!h->len_exact[which]) {
        spec_status s = sync_lengths(h);
        if (s != SPEC_OK) return s;
        if (h->host_len[which] + n <= h->c.max_ctx) return SPEC_OK;
    }
    return fail(SPEC_ERR_CAPACITY, "cache %d holds %d positions; %d more exceed max_ctx %d", which, h->host_len[which], n,
                h->c.max_ctx);
}

GemmParams base_params(spec_model* h, int which, int n) {
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.n = n;
    p.st = h->st;
    p.which = which;
    p.partials = h->gpart;
    p.counters = h->gcnt;
    p.d = h->c.d_model;
    p.norm_eps = h->c.norm_eps;
    p.ss_in = h->ss;
    p.ss_in_tiles = h->c.d_model / kTileRows;
    p.ss_out = h->ss;
    p.x = h->x;
    p.n_heads = h->c.n_heads;
    p.n_kv_heads = h->c.n_kv_heads;
    p.head_dim = h->c.head_dim;
    p.n_experts = h->c.n_experts;
    p.top_k = h->c.top_k;
    p.n_shared = h->c.n_experts > 0 ? h->c.n_shared_experts : 0;
    p.moe_mode = h->moe_mode;
    return p;
}

void set_mat(spec_model* h, GemmParams& p, const PackedMat& m, const uint8_t* X, int epi, int grid_cap) {
    p.W = m.p;
    p.T = m.T;
    p.KBs = m.KBs;
    p.N = m.N;
    p.X = X;
    p.x_f32 = (X == h->xf_norm) ? 1 : 0;   // normalised operands are kept in fp32
    p.epi = epi;
    p.items_mode = 0;
    const long long I = (long long)m.T * m.KBs;
    // at most 160 CTAs may share one tile in the stream-K fixup
    long long cap = grid_cap < 159ll * m.T ? grid_cap : 159ll * m.T;
    p.grid = (int)(I < cap ? I : cap);
}

// Algorithmic bytes of one dense GEMM launch: weights once, the activation
// operand once, the outputs once (fp32 residual read+write for EPI_RESID).
double gemm_bytes(const GemmParams& p) {
    const double w = (double)p.N * p.KBs * kKBlock * 2.0;
    const double xin = (double)p.n * p.KBs * kKBlock * (p.x_f32 ? 4.0 : 2.0);
    double out = 0.0;
    switch (p.epi) {
        case EPI_QKV: out = (double)p.n * p.N * 2.0; break;
        case EPI_RESID: out = (double)p.n * p.N * (4.0 + 4.0 + 2.0); break;
        case EPI_SWIGLU: out = (double)p.n * (p.N / 2) * 2.0; break;
        case EPI_LMHEAD: out = p.logits ? (double)p.n * p.N * 4.0 : (double)p.n * p.T * 8.0; break;
        case EPI_STORE: out = (double)p.n * p.N * 4.0; break;
        default: out = 0.0;
    }
    return w + xin + out;
}

// Expert weight bytes one items-mode launch requests: per-slot reads one
// expert per (token, slot), dedup one per distinct expert (needs the ids on
// the host, i.e. forced routing; otherwise the per-slot count is reported);
// both read every shared expert once.
double expert_launch_bytes(spec_model* h, const GemmParams& p, int layer) {
    const double per = (double)p.N * p.KBs * kKBlock * 2.0;
    const int K = h->c.top_k, n = p.n;
    int items = n * K;
    if (p.moe_mode == SPEC_MOE_DEDUP && h->forced_on && !h->forced_host.empty()) {
        unsigned long long used = 0ull;
        for (int j = 0; j < n; ++j)
            for (int s = 0; s < K; ++s) used |= 1ull << (h->forced_host[((size_t)layer * kMaxBlock + j) * K + s] & 63);
        items = __builtin_popcountll(used);
    }
    items += h->c.n_shared_experts;   // shared experts: once per launch in both modes
    return items * per + (double)n * p.KBs * kKBlock * 2.0;
}

// Chunk groups of the attention partials: about the SMs per kv head (one
// wave of partial CTAs for a single sequence), at most the chunks a cache
// holds.  Fixed per model, so every pass groups a position's chunk alike.
int attn_groups(const spec_model* h) {
    int g = (h->num_sms + h->c.n_kv_heads - 1) / h->c.n_kv_heads;
    if (g < 1) g = 1;
    return g < h->nch ? g : h->nch;
}

// Next launch slot of a traced pass (nullptr when not tracing or full).
long long* trace_slot(spec_model* h, int kind, int slots = 1) {
    if (!h->trace || !h->tracing) return nullptr;
    const size_t per = (size_t)kTraceCtas * 4;
    if ((h->trace_kinds.size() + slots) * per > h->trace_cap) return nullptr;
    long long* t = h->trace + h->trace_kinds.size() * per;
    for (int i = 0; i < slots; ++i) h->trace_kinds.push_back(kind + i);
    return t;
}

spec_status gemm(spec_model* h, const GemmParams& p_in, int layer = -1) {
    // the GEMM kernels fix the work-item mode by epilogue kind (expert kinds walk item lists)
    const bool items_kind = p_in.epi == EPI_EXPERT_SWIGLU || p_in.epi == EPI_EXPERT_DOWN;
    if ((p_in.items_mode != 0) != items_kind) return fail(SPEC_ERR_STATE, "internal: GEMM kind %d with item mode %d", p_in.epi, p_in.items_mode);
    GemmParams p = p_in;
    p.trace = trace_slot(h, p.epi);
    const bool rec = h->profiling;
    spec_model::ProfRec r{};
    if (rec) {
        CU(cudaEventCreate(&r.a));
        CU(cudaEventCreate(&r.b));
        CU(cudaEventRecord(r.a, h->stream));
    }
    CU(launch_gemm(p, h->stream, h->pdl));
    ++h->launches;
    if (rec) {
        CU(cudaEventRecord(r.b, h->stream));
        r.bytes = p.items_mode ? expert_launch_bytes(h, p, layer) : gemm_bytes(p);
        r.kind = p.epi;
        h->prof.push_back(r);
    }
    return SPEC_OK;
}

// One pass of n tokens through a plan (target: all layers; draft: kept layers).
spec_status run_pass_launch(spec_model* h, int which, const int32_t* d_tokens, int n, PassMode mode,
                            int32_t* d_argmax, int32_t* d_accept, float* d_logits, int32_t* d_ids, int32_t* d_pair,
                            int32_t* d_token, const int32_t* d_block);

void clear_graphs(spec_model* h) {
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second.exec);
    h->graphs.clear();
}

// One pass: the per-phase launch sequence, replayed from a captured CUDA
// graph when possible.
spec_status run_pass(spec_model* h, int which, const int32_t* d_tokens, int n, PassMode mode, int32_t* d_argmax,
                     int32_t* d_accept, float* d_logits, int32_t* d_ids, int32_t* d_pair, int32_t* d_token,
                     const int32_t* d_block) {
    if (h->trace) {  // a traced pass runs its launches directly, each with its own stamp slots
        h->tracing = true;
        h->trace_kinds.clear();
        CU(cudaMemsetAsync(h->trace, 0, h->trace_cap * sizeof(long long), h->stream));
        return run_pass_launch(h, which, d_tokens, n, mode, d_argmax, d_accept, d_logits, d_ids, d_pair, d_token,
                               d_block);
    }
    if (!h->use_graphs || h->profiling)
        return run_pass_launch(h, which, d_tokens, n, mode, d_argmax, d_accept, d_logits, d_ids, d_pair, d_token,
                               d_block);
    const std::vector<uintptr_t> key = {(uintptr_t)which, (uintptr_t)n, (uintptr_t)mode, (uintptr_t)d_tokens,
                                        (uintptr_t)d_argmax, (uintptr_t)d_accept, (uintptr_t)d_logits,
                                        (uintptr_t)d_ids, (uintptr_t)d_pair, (uintptr_t)d_token, (uintptr_t)d_block,
                                        (uintptr_t)h->moe_mode, (uintptr_t)h->forced_on, (uintptr_t)h->tap_out,
                                        (uintptr_t)h->tap_count, (uintptr_t)h->bat_nseq};
    auto f = h->graphs.find(key);
    if (f == h->graphs.end()) {
        if (h->graphs.size() >= 256) clear_graphs(h);
        cudaStream_t user = h->stream;
        h->stream = h->cap_stream;
        h->launches = 0;
        CU(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
        spec_status s = run_pass_launch(h, which, d_tokens, n, mode, d_argmax, d_accept, d_logits, d_ids, d_pair,
                                        d_token, d_block);
        cudaGraph_t graph = nullptr;
        const cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
        h->stream = user;
        if (s != SPEC_OK) {
            if (graph) cudaGraphDestroy(graph);
            return s;
        }
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(e));
        cudaGraphExec_t exec = nullptr;
        const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (ei != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(ei));
        f = h->graphs.emplace(key, spec_model::GraphEntry{exec, h->launches}).first;
    }
    CU(cudaGraphLaunch(f->second.exec, h->stream));
    h->launches = f->second.launches;
    return SPEC_OK;
}

spec_status run_pass_launch(spec_model* h, int which, const int32_t* d_tokens, int n, PassMode mode,
                            int32_t* d_argmax, int32_t* d_accept, float* d_logits, int32_t* d_ids, int32_t* d_pair,
                            int32_t* d_token, const int32_t* d_block) {
    const spec_model_config& c = h->c;
    const std::vector<int>& plan = which == 0 ? h->plan_full : h->plan_draft;
    const int d = c.d_model, hd = c.head_dim;
    const int G = h->num_sms;
    const bool pdl = h->pdl;
    spec_status s;

    {
        EmbedParams e{};
        e.tokens = d_tokens;
        e.embed = h->embed;
        e.n = n;
        e.d = d;
        e.vocab = c.vocab;
        e.x = h->x;
        e.g_next = h->L[plan[0]].attn_norm;
        e.xf_out = h->xf_norm;
        e.ss_out = h->ss;
        e.st = h->st;
        CU(launch_embed(e, h->stream, pdl));
        ++h->launches;
    }
    if (d_ids) CU(cudaMemsetAsync(d_ids, 0xFF, sizeof(int32_t) * (size_t)c.n_layers * n * (c.top_k > 0 ? c.top_k : 1), h->stream));

    for (size_t si = 0; si < plan.size(); ++si) {
        const int l = plan[si];
        LayerW& W = h->L[l];
        const uint16_t* g_after = (si + 1 < plan.size()) ? h->L[plan[si + 1]].attn_norm : h->final_norm;
        // hidden-state tap: the residual stream after this layer, target verify passes only
        float* tap = (which == 0 && mode == PASS_VERIFY && h->tap_count > 0 && h->tap_of_layer[l] >= 0)
                         ? h->tap_out + (size_t)h->tap_of_layer[l] * kMaxBlock * d
                         : nullptr;
        uint16_t* kpool = kv_pool(h, which, which == 0 ? l : (int)si, 0);
        uint16_t* vpool = kv_pool(h, which, which == 0 ? l : (int)si, 1);
        const bool bat = h->bat_nseq > 0;   // batched sequences: their own caches, positions and pages
        const int rps = bat ? n / h->bat_nseq : n;
        if (bat) {
            kpool = h->kb + h->pool_elems * h->bat_cap * l;
            vpool = h->vb + h->pool_elems * h->bat_cap * l;
        }

        // QKV (attn RMSNorm scale, RoPE, paged KV append)
        GemmParams p = base_params(h, which, n);
        set_mat(h, p, W.qkv, h->xf_norm, EPI_QKV, G);
        p.norm_dim = d;
        p.rope = h->rope;
        p.qbuf = h->qbuf;
        p.kpool = kpool;
        p.vpool = vpool;
        p.block_table = bat ? h->bt_b : h->block_table;
        if (bat) {
            p.seq_len = h->seq_len;
            p.rows_per_seq = rps;
            p.seq_pages = h->max_pages;
        }
        if ((s = gemm(h, p)) != SPEC_OK) return s;

        AttnParams a{};
        a.qbuf = h->qbuf;
        a.kpool = kpool;
        a.vpool = vpool;
        a.block_table = bat ? h->bt_b : h->block_table;
        a.part_o = bat ? h->battn_o : h->attn_o;
        a.part_ml = bat ? h->battn_ml : h->attn_ml;
        a.xf_out = h->xf_o;
        a.st = h->st;
        a.which = which;
        a.n = rps;
        if (bat) {
            a.seq_len = h->seq_len;
            a.nseq = h->bat_nseq;
            a.seq_pages = h->max_pages;
        }
        a.n_heads = c.n_heads;
        a.n_kv_heads = c.n_kv_heads;
        a.head_dim = hd;
        a.nch = h->nch;
        a.num_sms = h->num_sms;
        a.groups = attn_groups(h);
        a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)hd));
        a.trace = trace_slot(h, kTraceAttnPartial, 2);
        CU(launch_attention(a, h->stream, pdl));
        h->launches += 2;

        // O projection + residual; next operand = ffn-normed x
        p = base_params(h, which, n);
        set_mat(h, p, W.o, h->xf_o, EPI_RESID, G);
        p.g_next = W.ffn_norm;
        p.xf_out = h->xf_norm;
        if ((s = gemm(h, p)) != SPEC_OK) return s;

        if (!W.moe) {
            p = base_params(h, which, n);
            set_mat(h, p, W.gu, h->xf_norm, EPI_SWIGLU, G);
            p.norm_dim = d;
            p.xf_out = h->xf_down;
            if ((s = gemm(h, p)) != SPEC_OK) return s;
            p = base_params(h, which, n);
            set_mat(h, p, W.down, h->xf_down, EPI_RESID, G);
            p.g_next = g_after;
            p.xf_out = h->xf_norm;
            p.tap = tap;
            if ((s = gemm(h, p)) != SPEC_OK) return s;
        } else {
            const int K = c.top_k;
            // router: softmax + top-k
            p = base_params(h, which, n);
            set_mat(h, p, W.router, h->xf_norm, EPI_ROUTER, G);
            p.norm_dim = d;
            p.route_ids = h->route_ids;
            p.route_gates = h->route_gates;
            p.forced_ids = h->forced_on ? h->forced + (size_t)l * kMaxBlock * K : nullptr;
            p.debug_ids = (d_ids && which == 0) ? d_ids + (size_t)l * n * K : nullptr;
            if ((s = gemm(h, p)) != SPEC_OK) return s;
            // routed experts, gate/up: per-slot or deduplicated work items; the
            // shared experts are further items of the same launches
            p = base_params(h, which, n);
            set_mat(h, p, W.egu, h->xf_norm, EPI_EXPERT_SWIGLU, G);
            p.items_mode = 1;
            p.grid = G;
            p.w_item_stride = W.egu_stride;
            p.x_item_stride = 0;
            p.norm_dim = d;
            p.route_ids = h->route_ids;
            p.xe = h->xe;
            p.xe_stride = h->xe_stride;
            if ((s = gemm(h, p, l)) != SPEC_OK) return s;
            p = base_params(h, which, n);
            set_mat(h, p, W.edown, h->xe, EPI_EXPERT_DOWN, G);
            p.items_mode = 1;
            p.grid = G;
            p.w_item_stride = W.edown_stride;
            p.x_item_stride = h->xe_stride;
            p.route_ids = h->route_ids;
            p.y_slot = h->y_slot;
            if ((s = gemm(h, p, l)) != SPEC_OK) return s;
            CombineParams cb{};
            cb.x = h->x;
            cb.y_slot = h->y_slot;
            cb.n_shared = c.n_shared_experts;
            cb.gates = h->route_gates;
            cb.n = n;
            cb.d = d;
            cb.top_k = K;
            cb.g_next = g_after;
            cb.xf_out = h->xf_norm;
            cb.ss_out = h->ss;
            cb.tap = tap;
            CU(launch_moe_combine(cb, h->stream, pdl));
            ++h->launches;
        }
    }

    if (mode == PASS_PREFILL_MID) {
        CU(launch_advance(h->st, which, n, h->stream, pdl));
        ++h->launches;
        return SPEC_OK;
    }
    GemmParams p = base_params(h, which, n);
    set_mat(h, p, h->lm, h->xf_norm, EPI_LMHEAD, G);
    p.norm_dim = d;
    p.logits = d_logits;
    p.amax_val = h->amax_val;
    p.amax_idx = h->amax_idx;
    if ((s = gemm(h, p)) != SPEC_OK) return s;

    AcceptParams ap{};
    ap.amax_val = h->amax_val;
    ap.amax_idx = h->amax_idx;
    ap.T = h->lm.T;
    ap.n = n;
    ap.which = which;
    ap.st = h->st;
    ap.mode = mode == PASS_VERIFY ? ACC_VERIFY : (mode == PASS_DRAFT ? ACC_DRAFT : ACC_PREFILL);
    ap.block = d_block;
    ap.out_argmax = d_argmax;
    ap.out_accept = d_accept;
    ap.out_pair = d_pair;
    ap.out_token = d_token;
    if (h->bat_nseq > 0) {
        ap.mode = ACC_BATCH;
        ap.seq_len = h->seq_len;
        ap.nseq = h->bat_nseq;
    }
    CU(launch_accept(ap, h->stream, pdl));
    ++h->launches;
    return SPEC_OK;
}

void free_all(spec_model* h) {
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second.exec);
    h->graphs.clear();
    if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
    h->cap_stream = nullptr;
    if (h->trace) cudaFree(h->trace);
    h->trace = nullptr;
    for (void* p : h->draft_allocs) cudaFree(p);
    for (void* p : h->allocs) cudaFree(p);
    h->allocs.clear();
    h->draft_allocs.clear();
}

}  // namespace

extern "C" {

const char* spec_last_error(void) { return g_err.c_str(); }

spec_status spec_model_create(const spec_model_config* cfg, const spec_weights* w, const int32_t* draft_layers,
                              int32_t n_draft_layers, void* cuda_stream, spec_handle* out) {
    if (!out) return fail(SPEC_ERR_INVALID_ARG, "null output handle");
    *out = nullptr;
    spec_status s = validate_config(cfg);
    if (s != SPEC_OK) return s;
    if (!w || !w->embed || !w->final_norm || !w->layers) return fail(SPEC_ERR_INVALID_ARG, "missing weights");
    const spec_model_config& c = *cfg;
    for (int l = 0; l < c.n_layers; ++l) {
        const spec_layer_weights& lw = w->layers[l];
        if (!lw.attn_norm || !lw.ffn_norm || !lw.wq || !lw.wk || !lw.wv || !lw.wo)
            return fail(SPEC_ERR_INVALID_ARG, "layer %d: missing attention weights", l);
        const bool moe = c.n_experts > 0 && l >= c.first_moe_layer;
        if (!moe && (!lw.w_gate || !lw.w_up || !lw.w_down)) return fail(SPEC_ERR_INVALID_ARG, "layer %d: missing FFN weights", l);
        if (moe) {
            if (!lw.router || !lw.e_gate || !lw.e_up || !lw.e_down) return fail(SPEC_ERR_INVALID_ARG, "layer %d: missing expert weights", l);
            for (int e = 0; e < c.n_experts; ++e)
                if (!lw.e_gate[e] || !lw.e_up[e] || !lw.e_down[e]) return fail(SPEC_ERR_INVALID_ARG, "layer %d expert %d: null", l, e);
            if (c.n_shared_experts > 0) {
                if (!lw.s_gate || !lw.s_up || !lw.s_down) return fail(SPEC_ERR_INVALID_ARG, "layer %d: missing shared experts", l);
                for (int e = 0; e < c.n_shared_experts; ++e)
                    if (!lw.s_gate[e] || !lw.s_up[e] || !lw.s_down[e]) return fail(SPEC_ERR_INVALID_ARG, "layer %d shared %d: null", l, e);
            }
        }
    }
    if (!c.tied_embeddings && !w->lm_head) return fail(SPEC_ERR_INVALID_ARG, "untied model needs lm_head");

    spec_model* h = new spec_model();
    h->c = c;
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    {
        spec_status vs = validate_plan(h, draft_layers, n_draft_layers);
        if (vs != SPEC_OK) {
            delete h;
            return vs;
        }
    }
#define TRY(x)                     \
    do {                           \
        spec_status t_ = (x);      \
        if (t_ != SPEC_OK) {       \
            free_all(h);           \
            delete h;              \
            return t_;             \
        }                          \
    } while (0)
#define TRYCU(x) TRY(([&]() -> spec_status { CU(x); return SPEC_OK; })())

    TRYCU(cudaGetDevice(&h->device));
    cudaDeviceProp prop;
    TRYCU(cudaGetDeviceProperties(&prop, h->device));
    if (prop.major != 10 || prop.minor != 3) {
        std::string msg = "this library is built for sm_103a (GB300); device is sm_" + std::to_string(prop.major) +
                          std::to_string(prop.minor);
        delete h;
        return fail(SPEC_ERR_CUDA, "%s", msg.c_str());
    }
    h->num_sms = prop.multiProcessorCount;
    if (const char* e = std::getenv("SPEC_NO_PDL")) h->pdl = !(e[0] == '1');
    if (const char* e = std::getenv("SPEC_GRAPHS")) h->use_graphs = !(e[0] == '0');
    TRYCU(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
    TRYCU(gemm_configure(h->device));
    TRYCU(attention_configure(h->device));

    const int d = c.d_model, hd = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads;
    const int qw = Hq * hd, kw = Hkv * hd;
    const int S = c.n_experts > 0 ? c.n_shared_experts : 0;
    const int fe = c.expert_ffn;

    // ---- weights ----
    TRY(copy_vec(h, &h->embed, w->embed, (size_t)c.vocab * d));
    TRY(copy_vec(h, &h->final_norm, w->final_norm, d));
    TRY(alloc_packed(h, h->lm, c.vocab, d));
    TRY(pack_into(h, h->lm, src_rows({c.tied_embeddings ? w->embed : w->lm_head}, {c.vocab}, d, 0)));
    h->L.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const spec_layer_weights& lw = w->layers[l];
        LayerW& W = h->L[l];
        W.moe = c.n_experts > 0 && l >= c.first_moe_layer;
        TRY(copy_vec(h, &W.attn_norm, lw.attn_norm, d));
        TRY(copy_vec(h, &W.ffn_norm, lw.ffn_norm, d));
        TRY(alloc_packed(h, W.qkv, qw + 2 * kw, d));
        TRY(pack_into(h, W.qkv, src_rows({lw.wq, lw.wk, lw.wv}, {qw, kw, kw}, d, 0)));
        TRY(alloc_packed(h, W.o, d, qw));
        TRY(pack_into(h, W.o, src_rows({lw.wo}, {d}, qw, 0)));
        if (!W.moe) {
            TRY(alloc_packed(h, W.gu, 2 * c.ffn_dim, d));
            TRY(pack_into(h, W.gu, src_rows({lw.w_gate, lw.w_up}, {c.ffn_dim, c.ffn_dim}, d, 1)));
            TRY(alloc_packed(h, W.down, d, c.ffn_dim));
            TRY(pack_into(h, W.down, src_rows({lw.w_down}, {d}, c.ffn_dim, 0)));
        } else {
            TRY(alloc_packed(h, W.router, c.n_experts, d));
            TRY(pack_into(h, W.router, src_rows({lw.router}, {c.n_experts}, d, 0)));
            // experts: one contiguous region per layer, expert e at e * stride
            PackedMat g1 = geometry(2 * fe, d), d1 = geometry(d, fe);
            W.egu_stride = (long long)g1.bytes();
            W.edown_stride = (long long)d1.bytes();
            W.egu = g1;
            W.edown = d1;
            TRY(dalloc(h, reinterpret_cast<void**>(&W.egu.p), g1.bytes() * (c.n_experts + S)));
            TRY(dalloc(h, reinterpret_cast<void**>(&W.edown.p), d1.bytes() * (c.n_experts + S)));
            if (g1.T > h->max_T) h->max_T = g1.T;
            if (d1.T > h->max_T) h->max_T = d1.T;
            for (int e = 0; e < c.n_experts + S; ++e) {   // shared expert t at index n_experts + t
                PackedMat ge = g1, de = d1;
                ge.p = W.egu.p + e * W.egu_stride;
                de.p = W.edown.p + e * W.edown_stride;
                const bool sh = e >= c.n_experts;
                const int t = e - c.n_experts;
                TRY(pack_into(h, ge, src_rows({sh ? lw.s_gate[t] : lw.e_gate[e], sh ? lw.s_up[t] : lw.e_up[e]},
                                              {fe, fe}, d, 1)));
                TRY(pack_into(h, de, src_rows({sh ? lw.s_down[t] : lw.e_down[e]}, {d}, fe, 0)));
            }
        }
    }

    // ---- caches ----
    h->nch = (c.max_ctx + kAttnChunk - 1) / kAttnChunk;
    h->max_pages = h->nch * (kAttnChunk / kPageSize);
    h->pool_elems = (size_t)h->max_pages * Hkv * kPageSize * hd;
    TRY(dalloc_t(h, &h->kt, h->pool_elems * c.n_layers));
    TRY(dalloc_t(h, &h->vt, h->pool_elems * c.n_layers));
    {
        std::vector<int> bt(h->max_pages);
        for (int i = 0; i < h->max_pages; ++i) bt[i] = i;
        TRY(dalloc_t(h, &h->block_table, h->max_pages));
        TRYCU(cudaMemcpyAsync(h->block_table, bt.data(), sizeof(int) * bt.size(), cudaMemcpyHostToDevice, h->stream));
        TRYCU(cudaStreamSynchronize(h->stream));
    }
    {
        // RoPE table, rotate-half pairing: angle = pos * theta^(-2i/hd), in double
        const int half = hd / 2;
        std::vector<float2> tab((size_t)c.max_ctx * half);
        for (int p = 0; p < c.max_ctx; ++p)
            for (int i = 0; i < half; ++i) {
                const double ang = (double)p * std::pow((double)c.rope_theta, -2.0 * i / (double)hd);
                tab[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
        TRY(dalloc_t(h, &h->rope, tab.size()));
        TRYCU(cudaMemcpyAsync(h->rope, tab.data(), sizeof(float2) * tab.size(), cudaMemcpyHostToDevice, h->stream));
        TRYCU(cudaStreamSynchronize(h->stream));
    }
    h->plan_full.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) h->plan_full[l] = l;
    TRY(alloc_draft(h, draft_layers, n_draft_layers));

    // ---- activations and scratch ----
    const int ffn_max = std::max(c.ffn_dim, 64);
    TRY(dalloc_t(h, &h->x, (size_t)kMaxBlock * d));
    TRY(dalloc_t(h, &h->xf_norm, (size_t)(d / kKBlock) * kStageX32Bytes));
    TRY(dalloc_t(h, &h->xf_o, (size_t)(qw / kKBlock) * kStageXBytes));
    TRY(dalloc_t(h, &h->xf_down, (size_t)(ffn_max / kKBlock) * kStageXBytes));
    TRY(dalloc_t(h, &h->qbuf, (size_t)kMaxBlock * qw));
    TRY(dalloc_t(h, &h->ss, (size_t)kMaxBlock * (d / kTileRows)));
    TRY(dalloc_t(h, &h->attn_o, (size_t)Hkv * 2 * h->nch * 64 * hd));
    TRY(dalloc_t(h, &h->attn_ml, (size_t)Hkv * 2 * h->nch * 64));
    TRY(dalloc_t(h, &h->gpart, (size_t)2 * h->num_sms * kTileRows * kMaxBlock));
    TRY(dalloc_t(h, &h->gcnt, (size_t)h->max_T + 1));
    TRY(dalloc_t(h, &h->amax_val, (size_t)kMaxBlock * h->lm.T));
    TRY(dalloc_t(h, &h->amax_idx, (size_t)kMaxBlock * h->lm.T));
    TRY(dalloc_t(h, &h->st, 1));
    {
        const int ch = sample_chunks(c.vocab);
        TRY(dalloc_t(h, &h->samp_stats, (size_t)(2 * kMaxBlock - 1) * ch));
        TRY(dalloc_t(h, &h->samp_rows, (size_t)(2 * kMaxBlock - 1)));
        TRY(dalloc_t(h, &h->samp_sums, (size_t)2 * ch));
        TRY(dalloc_t(h, &h->samp_decision, 2));
    }
    if (c.n_experts > 0) {
        const int K = c.top_k;
        TRY(dalloc_t(h, &h->route_ids, (size_t)kMaxBlock * K));
        TRY(dalloc_t(h, &h->route_gates, (size_t)kMaxBlock * K));
        TRY(dalloc_t(h, &h->forced, (size_t)c.n_layers * kMaxBlock * K));
        TRY(dalloc_t(h, &h->y_slot, (size_t)kMaxBlock * (K + S) * d));
        h->xe_stride = (long long)(fe / kKBlock) * kStageXBytes;
        TRY(dalloc_t(h, &h->xe, (size_t)h->xe_stride * (kMaxBlock * K + S)));
    }
    TRYCU(cudaStreamSynchronize(h->stream));
    TRYCU(cudaGetLastError());
#undef TRY
#undef TRYCU
    *out = h;
    return SPEC_OK;
}

spec_status spec_model_destroy(spec_handle h) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    cudaStreamSynchronize(h->stream);
    free_all(h);
    delete h;
    return SPEC_OK;
}

spec_status spec_set_draft_plan(spec_handle h, const int32_t* draft_layers, int32_t n_draft_layers) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    spec_status s = validate_plan(h, draft_layers, n_draft_layers);
    if (s != SPEC_OK) return s;
    CU(cudaStreamSynchronize(h->stream));
    clear_graphs(h);
    if ((s = alloc_draft(h, draft_layers, n_draft_layers)) != SPEC_OK) return s;
    h->launches = 0;
    CU(launch_rollback(h->st, 1, 0, h->stream, false));
    CU(cudaStreamSynchronize(h->stream));
    return SPEC_OK;
}

spec_status spec_set_stream(spec_handle h, void* cuda_stream) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    return SPEC_OK;
}

spec_status spec_prefill(spec_handle h, const int32_t* d_tokens, int32_t m, int32_t* d_next_token) {
    if (!h || !d_tokens || !d_next_token || m < 1) return fail(SPEC_ERR_INVALID_ARG, "bad prefill arguments");
    spec_status s;
    if ((s = check_capacity(h, 0, m)) != SPEC_OK) return s;
    const bool draft = !h->plan_draft.empty();
    if (draft && (s = check_capacity(h, 1, m)) != SPEC_OK) return s;
    h->launches = 0;
    for (int off = 0; off < m; off += kMaxBlock) {
        const int cn = std::min(kMaxBlock, m - off);
        const bool last = off + cn == m;
        s = run_pass(h, 0, d_tokens + off, cn, last ? PASS_PREFILL_LAST : PASS_PREFILL_MID, nullptr, nullptr, nullptr,
                     nullptr, nullptr, last ? d_next_token : nullptr, nullptr);
        if (s != SPEC_OK) return s;
    }
    h->host_len[0] += m;
    if (draft) {
        for (int off = 0; off < m; off += kMaxBlock) {
            const int cn = std::min(kMaxBlock, m - off);
            s = run_pass(h, 1, d_tokens + off, cn, PASS_PREFILL_MID, nullptr, nullptr, nullptr, nullptr, nullptr,
                         nullptr, nullptr);
            if (s != SPEC_OK) return s;
        }
        h->host_len[1] += m;
    }
    return SPEC_OK;
}

spec_status spec_draft_step(spec_handle h, const int32_t* d_tokens, int32_t n, int32_t* d_draft_token) {
    return spec_draft_step_logits(h, d_tokens, n, d_draft_token, nullptr);
}

spec_status spec_draft_step_logits(spec_handle h, const int32_t* d_tokens, int32_t n, int32_t* d_draft_token,
                                   float* d_logits_opt) {
    if (!h || !d_tokens || !d_draft_token) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (n < 1 || n > 2) return fail(SPEC_ERR_INVALID_ARG, "draft step takes 1 or 2 tokens");
    if (h->plan_draft.empty()) return fail(SPEC_ERR_STATE, "model has no draft plan");
    spec_status s = check_capacity(h, 1, n);
    if (s != SPEC_OK) return s;
    h->launches = 0;
    s = run_pass(h, 1, d_tokens, n, PASS_DRAFT, nullptr, nullptr, d_logits_opt, nullptr, nullptr, d_draft_token,
                 nullptr);
    if (s == SPEC_OK) h->host_len[1] += n;
    return s;
}

spec_status spec_verify_step(spec_handle h, const int32_t* d_block, int32_t n, int32_t* d_argmax, int32_t* d_accept_len,
                             float* d_logits_opt, int32_t* d_expert_ids_opt, int32_t* d_next_pair_opt) {
    if (!h || !d_block || !d_argmax || !d_accept_len) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (n < 1 || n > SPEC_MAX_BLOCK) return fail(SPEC_ERR_INVALID_ARG, "block size %d outside 1..16", n);
    if (d_expert_ids_opt && h->c.n_experts == 0) return fail(SPEC_ERR_INVALID_ARG, "dense model has no expert ids");
    spec_status s = check_capacity(h, 0, n);
    if (s != SPEC_OK) return s;
    h->launches = 0;
    s = run_pass(h, 0, d_block, n, PASS_VERIFY, d_argmax, d_accept_len, d_logits_opt, d_expert_ids_opt, d_next_pair_opt,
                 nullptr, d_block);
    if (s == SPEC_OK) h->host_len[0] += n;
    return s;
}

spec_status spec_accept_sampled(spec_handle h, const float* d_target_logits, const float* d_draft_logits,
                                const int32_t* d_block, int32_t n, float temperature, const double* d_uniforms,
                                int32_t* d_accept_len, int32_t* d_next_token) {
    if (!h || !d_target_logits || !d_block || !d_uniforms || !d_accept_len || !d_next_token)
        return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (n < 1 || n > SPEC_MAX_BLOCK) return fail(SPEC_ERR_INVALID_ARG, "block size %d outside 1..16", n);
    if (n > 1 && !d_draft_logits) return fail(SPEC_ERR_INVALID_ARG, "draft logits needed for n > 1");
    if (!(temperature > 0.f) || !std::isfinite(temperature))
        return fail(SPEC_ERR_INVALID_ARG, "temperature must be positive and finite");
    SampleParams p{};
    p.target = d_target_logits;
    p.draft = n > 1 ? d_draft_logits : nullptr;
    p.block = d_block;
    p.uniforms = d_uniforms;
    p.n = n;
    p.vocab = h->c.vocab;
    p.chunks = sample_chunks(h->c.vocab);
    p.temperature = temperature;
    p.stats = h->samp_stats;
    p.row_stat = h->samp_rows;
    p.chunk_sum = h->samp_sums;
    p.decision = h->samp_decision;
    p.out_accept = d_accept_len;
    p.out_token = d_next_token;
    h->launches = 0;
    CU(launch_sample_accept(p, h->stream, h->pdl));
    h->launches = 4;
    return SPEC_OK;
}

spec_status spec_kv_rollback(spec_handle h, int32_t which, int32_t new_len) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (which != SPEC_CACHE_TARGET && which != SPEC_CACHE_DRAFT) return fail(SPEC_ERR_INVALID_ARG, "bad cache id");
    if (which == SPEC_CACHE_DRAFT && h->plan_draft.empty()) return fail(SPEC_ERR_STATE, "model has no draft plan");
    if (new_len < -1) return fail(SPEC_ERR_INVALID_ARG, "bad length %d", new_len);
    if (new_len >= 0 && new_len > h->host_len[which]) {
        spec_status s = h->len_exact[which] ? SPEC_OK : sync_lengths(h);
        if (s != SPEC_OK) return s;
        if (new_len > h->host_len[which])
            return fail(SPEC_ERR_INVALID_ARG, "rollback to %d beyond the %d cached positions", new_len, h->host_len[which]);
    }
    h->launches = 0;
    CU(launch_rollback(h->st, which, new_len, h->stream, h->pdl));
    h->launches = 1;
    if (new_len >= 0) {
        h->host_len[which] = new_len;
        h->len_exact[which] = true;
    } else {
        h->len_exact[which] = false;   // known on the device only; host keeps the upper bound
    }
    return SPEC_OK;
}

spec_status spec_moe_mode(spec_handle h, int32_t mode) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (mode != SPEC_MOE_PER_SLOT && mode != SPEC_MOE_DEDUP) return fail(SPEC_ERR_INVALID_ARG, "bad MoE mode");
    if (h->c.n_experts == 0) return fail(SPEC_ERR_STATE, "dense model");
    h->moe_mode = mode;
    return SPEC_OK;
}

spec_status spec_share_prefix(spec_handle h, int32_t enable) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (h->plan_draft.empty()) return fail(SPEC_ERR_STATE, "model has no draft plan");
    CU(cudaStreamSynchronize(h->stream));
    clear_graphs(h);
    h->share_prefix = enable != 0;
    const std::vector<int32_t> plan = h->plan_draft;
    spec_status s = alloc_draft(h, plan.data(), (int32_t)plan.size());
    if (s != SPEC_OK) return s;
    CU(launch_rollback(h->st, 1, 0, h->stream, false));
    CU(cudaStreamSynchronize(h->stream));
    return SPEC_OK;
}

spec_status spec_set_taps(spec_handle h, const int32_t* layers, int32_t count, float* d_out) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (count < 0 || count > h->c.n_layers) return fail(SPEC_ERR_INVALID_ARG, "tap count %d out of range", count);
    if (count > 0 && (!layers || !d_out)) return fail(SPEC_ERR_INVALID_ARG, "null tap layers or output");
    if (count > 0 && (reinterpret_cast<uintptr_t>(d_out) & 15))
        return fail(SPEC_ERR_INVALID_ARG, "tap output not 16-byte aligned");
    std::vector<int> of(h->c.n_layers, -1);
    for (int t = 0; t < count; ++t) {
        const int l = layers[t];
        if (l < 0 || l >= h->c.n_layers) return fail(SPEC_ERR_INVALID_ARG, "tap layer %d out of range", l);
        if (of[l] >= 0) return fail(SPEC_ERR_INVALID_ARG, "tap layer %d listed twice", l);
        of[l] = t;
    }
    CU(cudaStreamSynchronize(h->stream));
    clear_graphs(h);
    h->tap_of_layer = of;
    h->tap_out = count > 0 ? d_out : nullptr;
    h->tap_count = count;
    return SPEC_OK;
}

spec_status spec_batch_reserve(spec_handle h, int32_t nseq) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (nseq < 1 || nseq > kMaxBlock) return fail(SPEC_ERR_INVALID_ARG, "nseq must be in 1..16");
    if (h->bat_cap) return fail(SPEC_ERR_STATE, "batch caches are already reserved");
    const spec_model_config& c = h->c;
    const size_t pages = (size_t)nseq * h->max_pages;
    const size_t parts = (size_t)nseq * c.n_kv_heads * h->nch * 64;
    spec_status s;
    if ((s = dalloc_t(h, &h->kb, h->pool_elems * nseq * c.n_layers)) != SPEC_OK) return s;
    if ((s = dalloc_t(h, &h->vb, h->pool_elems * nseq * c.n_layers)) != SPEC_OK) return s;
    if ((s = dalloc_t(h, &h->bt_b, pages)) != SPEC_OK) return s;
    if ((s = dalloc_t(h, &h->seq_len, (size_t)kMaxBlock)) != SPEC_OK) return s;
    if ((s = dalloc_t(h, &h->battn_o, parts * c.head_dim)) != SPEC_OK) return s;
    if ((s = dalloc_t(h, &h->battn_ml, parts)) != SPEC_OK) return s;
    std::vector<int> bt(pages);
    for (size_t i = 0; i < pages; ++i) bt[i] = (int)i;
    CU(cudaMemcpyAsync(h->bt_b, bt.data(), sizeof(int) * bt.size(), cudaMemcpyHostToDevice, h->stream));
    CU(cudaStreamSynchronize(h->stream));
    h->bat_cap = nseq;
    h->bat_host_len.assign(nseq, 0);
    return SPEC_OK;
}

static spec_status batch_kv_io(spec_handle h, int32_t seq, int32_t slot, void* dk, void* dv, int32_t ctx, bool load) {
    if (!h || !dk || !dv) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (seq < 0 || seq >= h->bat_cap) return fail(SPEC_ERR_INVALID_ARG, "sequence %d not reserved", seq);
    if (slot < 0 || slot >= h->c.n_layers) return fail(SPEC_ERR_INVALID_ARG, "slot %d out of range", slot);
    if (ctx < 0 || ctx > h->c.max_ctx) return fail(SPEC_ERR_INVALID_ARG, "ctx %d out of range", ctx);
    const size_t off = h->pool_elems * ((size_t)h->bat_cap * slot + seq);   // the sequence's own pages
    CU(launch_kv_io(h->kb + off, h->block_table, static_cast<uint16_t*>(dk), ctx, h->c.n_kv_heads, h->c.head_dim, load,
                    false, h->stream));
    CU(launch_kv_io(h->vb + off, h->block_table, static_cast<uint16_t*>(dv), ctx, h->c.n_kv_heads, h->c.head_dim, load,
                    true, h->stream));
    return SPEC_OK;
}

spec_status spec_batch_kv_load(spec_handle h, int32_t seq, int32_t slot, const void* d_k, const void* d_v, int32_t ctx) {
    return batch_kv_io(h, seq, slot, const_cast<void*>(d_k), const_cast<void*>(d_v), ctx, true);
}

spec_status spec_batch_kv_export(spec_handle h, int32_t seq, int32_t slot, void* d_k, void* d_v, int32_t ctx) {
    return batch_kv_io(h, seq, slot, d_k, d_v, ctx, false);
}

spec_status spec_batch_set_len(spec_handle h, int32_t seq, int32_t len) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (seq < 0 || seq >= h->bat_cap) return fail(SPEC_ERR_INVALID_ARG, "sequence %d not reserved", seq);
    if (len < 0 || len > h->c.max_ctx) return fail(SPEC_ERR_INVALID_ARG, "length %d out of range", len);
    const int32_t v = len;
    CU(cudaMemcpyAsync(h->seq_len + seq, &v, sizeof(v), cudaMemcpyHostToDevice, h->stream));
    CU(cudaStreamSynchronize(h->stream));
    h->bat_host_len[seq] = len;
    return SPEC_OK;
}

spec_status spec_batch_len(spec_handle h, int32_t seq, int32_t* out_len) {
    if (!h || !out_len) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (seq < 0 || seq >= h->bat_cap) return fail(SPEC_ERR_INVALID_ARG, "sequence %d not reserved", seq);
    CU(cudaStreamSynchronize(h->stream));
    int32_t v = 0;
    CU(cudaMemcpy(&v, h->seq_len + seq, sizeof(v), cudaMemcpyDeviceToHost));
    h->bat_host_len[seq] = v;
    *out_len = v;
    return SPEC_OK;
}

spec_status spec_verify_batch(spec_handle h, const int32_t* d_blocks, int32_t nseq, int32_t n, int32_t* d_argmax,
                              int32_t* d_accept, float* d_logits_opt) {
    if (!h || !d_blocks || !d_argmax || !d_accept) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (nseq < 1 || nseq > h->bat_cap) return fail(SPEC_ERR_INVALID_ARG, "nseq %d outside the %d reserved", nseq, h->bat_cap);
    if (n < 1 || nseq * n > kMaxBlock) return fail(SPEC_ERR_INVALID_ARG, "nseq * n must be in 1..16");
    bool synced = false;
    for (int q = 0; q < nseq; ++q) {
        if (h->bat_host_len[q] + n <= h->c.max_ctx) continue;
        if (!synced) {   // the host's bounds may be stale after device-side accepts
            CU(cudaStreamSynchronize(h->stream));
            std::vector<int32_t> lens(h->bat_cap);
            CU(cudaMemcpy(lens.data(), h->seq_len, sizeof(int32_t) * h->bat_cap, cudaMemcpyDeviceToHost));
            for (int t = 0; t < h->bat_cap; ++t) h->bat_host_len[t] = lens[t];
            synced = true;
        }
        if (h->bat_host_len[q] + n > h->c.max_ctx)
            return fail(SPEC_ERR_CAPACITY, "sequence %d holds %d positions; %d more exceed max_ctx %d", q,
                        h->bat_host_len[q], n, h->c.max_ctx);
    }
    h->launches = 0;
    h->bat_nseq = nseq;
    spec_status s = run_pass(h, 0, d_blocks, nseq * n, PASS_VERIFY, d_argmax, d_accept, d_logits_opt, nullptr, nullptr,
                             nullptr, d_blocks);
    h->bat_nseq = 0;
    if (s == SPEC_OK)
        for (int q = 0; q < nseq; ++q) h->bat_host_len[q] += n;
    return s;
}

spec_status spec_set_context_fc(spec_handle h, const uint16_t* d_fc, int32_t n_in) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (!d_fc || n_in < 1 || n_in > 8) return fail(SPEC_ERR_INVALID_ARG, "fc must be given for 1..8 tapped layers");
    if (h->ctx_n_in) return fail(SPEC_ERR_STATE, "the context projection is already set");
    const int d = h->c.d_model;
    spec_status s;
    if ((s = alloc_packed(h, h->ctx_fc, d, n_in * d)) != SPEC_OK) return s;
    if ((s = pack_into(h, h->ctx_fc, src_rows({d_fc}, {d}, n_in * d, 0))) != SPEC_OK) return s;
    if ((s = dalloc(h, reinterpret_cast<void**>(&h->xf_ctx), (size_t)n_in * d / kKBlock * kStageX32Bytes)) != SPEC_OK)
        return s;
    CU(cudaStreamSynchronize(h->stream));
    h->ctx_n_in = n_in;
    return SPEC_OK;
}

spec_status spec_context_append(spec_handle h, const float* d_taps, int32_t m) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (!h->ctx_n_in) return fail(SPEC_ERR_STATE, "no context projection (spec_set_context_fc)");
    if (!d_taps || (reinterpret_cast<uintptr_t>(d_taps) & 15)) return fail(SPEC_ERR_INVALID_ARG, "null or unaligned taps");
    if (m < 1 || m > kMaxBlock) return fail(SPEC_ERR_INVALID_ARG, "m must be in 1..16");
    spec_status s = check_capacity(h, 0, m);
    if (s != SPEC_OK) return s;
    const spec_model_config& c = h->c;
    const int d = c.d_model, G = h->num_sms;
    const bool pdl = h->pdl;
    h->launches = 0;
    ConcatParams cp{d_taps, h->ctx_n_in, d, h->xf_ctx};
    CU(launch_concat_taps(cp, h->stream, pdl));
    ++h->launches;
    // features = fc . bf16(concatenated taps), fp32 rows into the residual buffer
    GemmParams p = base_params(h, 0, m);
    set_mat(h, p, h->ctx_fc, h->xf_ctx, EPI_STORE, G);
    p.x_f32 = 1;
    p.y_store = h->x;
    if ((s = gemm(h, p)) != SPEC_OK) return s;
    for (int l = 0; l < c.n_layers; ++l) {
        LayerW& W = h->L[l];
        RowsParams rp{h->x, m, d, W.attn_norm, h->xf_norm, h->ss};
        CU(launch_rows_operand(rp, h->stream, pdl));
        ++h->launches;
        // this layer's k/v of the context positions; when the q rows fill whole
        // tiles the GEMM starts at the first k/v tile and never reads them
        p = base_params(h, 0, m);
        PackedMat kv = W.qkv;
        const int qw = c.n_heads * c.head_dim;
        if (qw % kTileRows == 0) {
            kv.p = W.qkv.p + (size_t)(qw / kTileRows) * W.qkv.KBs * kStageWBytes;
            kv.T = W.qkv.T - qw / kTileRows;
        }
        set_mat(h, p, kv, h->xf_norm, EPI_QKV, G);
        p.N = W.qkv.N;
        if (qw % kTileRows == 0) p.tile0 = qw / kTileRows;
        p.norm_dim = d;
        p.rope = h->rope;
        p.qbuf = h->qbuf;
        p.kpool = h->kt + h->pool_elems * l;
        p.vpool = h->vt + h->pool_elems * l;
        p.block_table = h->block_table;
        if ((s = gemm(h, p)) != SPEC_OK) return s;
    }
    CU(launch_advance(h->st, 0, m, h->stream, pdl));
    ++h->launches;
    h->host_len[0] += m;
    return SPEC_OK;
}

spec_status spec_check_error(spec_handle h) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    CU(cudaStreamSynchronize(h->stream));
    CU(cudaGetLastError());
    int err = 0;
    CU(cudaMemcpy(&err, &h->st->error, sizeof(int), cudaMemcpyDeviceToHost));
    if (err) {
        int zero = 0;
        CU(cudaMemcpy(&h->st->error, &zero, sizeof(int), cudaMemcpyHostToDevice));
        CU(cudaMemset(h->gcnt, 0, sizeof(int) * (h->max_T + 1)));
        return fail(err == 10 ? SPEC_ERR_INVALID_ARG : SPEC_ERR_TIMEOUT,
                    err == 10 ? "a token id outside [0, vocab) was replaced by 0" : "device error code %d", err);
    }
    return SPEC_OK;
}

spec_status spec_kv_len(spec_handle h, int32_t which, int32_t* out_len) {
    if (!h || !out_len || (which != 0 && which != 1)) return fail(SPEC_ERR_INVALID_ARG, "bad arguments");
    spec_status s = sync_lengths(h);
    if (s != SPEC_OK) return s;
    *out_len = h->host_len[which];
    return SPEC_OK;
}

static spec_status kv_io(spec_handle h, int32_t which, int32_t slot, void* dk, void* dv, int32_t ctx, bool load) {
    if (!h || !dk || !dv) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (which != 0 && which != 1) return fail(SPEC_ERR_INVALID_ARG, "bad cache id");
    const int nslots = which == 0 ? h->c.n_layers : (int)h->plan_draft.size();
    if (slot < 0 || slot >= nslots) return fail(SPEC_ERR_INVALID_ARG, "slot %d out of range", slot);
    if (ctx < 0 || ctx > h->c.max_ctx) return fail(SPEC_ERR_INVALID_ARG, "ctx %d out of range", ctx);
    uint16_t* kp = kv_pool(h, which, slot, 0);
    uint16_t* vp = kv_pool(h, which, slot, 1);
    CU(launch_kv_io(kp, h->block_table, static_cast<uint16_t*>(dk), ctx, h->c.n_kv_heads, h->c.head_dim, load, false,
                    h->stream));
    CU(launch_kv_io(vp, h->block_table, static_cast<uint16_t*>(dv), ctx, h->c.n_kv_heads, h->c.head_dim, load, true,
                    h->stream));
    return SPEC_OK;
}

spec_status spec_kv_load(spec_handle h, int32_t which, int32_t slot, const void* d_k, const void* d_v, int32_t ctx) {
    return kv_io(h, which, slot, const_cast<void*>(d_k), const_cast<void*>(d_v), ctx, true);
}

spec_status spec_kv_export(spec_handle h, int32_t which, int32_t slot, void* d_k, void* d_v, int32_t ctx) {
    return kv_io(h, which, slot, d_k, d_v, ctx, false);
}

spec_status spec_kv_set_len(spec_handle h, int32_t which, int32_t len) {
    if (!h || (which != 0 && which != 1)) return fail(SPEC_ERR_INVALID_ARG, "bad arguments");
    if (len < 0 || len > h->c.max_ctx) return fail(SPEC_ERR_INVALID_ARG, "length %d out of range", len);
    CU(launch_rollback(h->st, which, len, h->stream, false));
    h->host_len[which] = len;
    h->len_exact[which] = true;
    return SPEC_OK;
}

spec_status spec_moe_force_routing(spec_handle h, const int32_t* d_ids) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    if (h->c.n_experts == 0) return fail(SPEC_ERR_STATE, "dense model");
    if (!d_ids) {
        h->forced_on = false;
        return SPEC_OK;
    }
    const size_t count = (size_t)h->c.n_layers * kMaxBlock * h->c.top_k;
    std::vector<int32_t> ids(count);
    CU(cudaStreamSynchronize(h->stream));
    CU(cudaMemcpy(ids.data(), d_ids, count * sizeof(int32_t), cudaMemcpyDeviceToHost));
    const int K = h->c.top_k;
    for (int l = h->c.first_moe_layer; l < h->c.n_layers; ++l)
        for (int j = 0; j < kMaxBlock; ++j) {
            const int32_t* r = &ids[((size_t)l * kMaxBlock + j) * K];
            for (int s = 0; s < K; ++s) {
                if (r[s] < 0 || r[s] >= h->c.n_experts) return fail(SPEC_ERR_INVALID_ARG, "forced expert id %d out of range", r[s]);
                for (int t = 0; t < s; ++t)
                    if (r[t] == r[s]) return fail(SPEC_ERR_INVALID_ARG, "forced ids of a token must be distinct");
            }
        }
    CU(cudaMemcpyAsync(h->forced, ids.data(), count * sizeof(int32_t), cudaMemcpyHostToDevice, h->stream));
    CU(cudaStreamSynchronize(h->stream));
    h->forced_host = ids;
    h->forced_on = true;
    return SPEC_OK;
}

int32_t spec_last_launch_count(spec_handle h) { return h ? h->launches : -1; }

spec_status spec_profile_enable(spec_handle h, int32_t enable) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    h->profiling = enable != 0;
    return SPEC_OK;
}

spec_status spec_trace_enable(spec_handle h, int32_t enable) {
    if (!h) return fail(SPEC_ERR_INVALID_ARG, "null handle");
    CU(cudaStreamSynchronize(h->stream));
    if (enable && !h->trace) {
        h->trace_cap = (size_t)h->num_sms * 4096 * 4;
        CU(cudaMalloc(&h->trace, h->trace_cap * sizeof(long long)));
    } else if (!enable && h->trace) {
        cudaFree(h->trace);
        h->trace = nullptr;
        h->trace_cap = 0;
    }
    return SPEC_OK;
}

spec_status spec_trace_read(spec_handle h, long long* out, int32_t capacity, int32_t* nphase, int32_t* nctas) {
    if (!h || !out || !nphase || !nctas) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (!h->trace || !h->tracing) return fail(SPEC_ERR_STATE, "no traced pass");
    CU(cudaStreamSynchronize(h->stream));
    // separate launches: device layout [launch][kTraceCtas][4] -> [kTraceCtas][launch][4]
    const size_t nl = h->trace_kinds.size();
    if (nl == 0) return fail(SPEC_ERR_STATE, "no traced pass");
    const size_t count = (size_t)kTraceCtas * nl * 4;
    if ((size_t)capacity < count) return fail(SPEC_ERR_INVALID_ARG, "need %zu entries", count);
    std::vector<long long> dev(count);
    CU(cudaMemcpy(dev.data(), h->trace, count * sizeof(long long), cudaMemcpyDeviceToHost));
    for (size_t l = 0; l < nl; ++l)
        for (size_t c = 0; c < (size_t)kTraceCtas; ++c)
            for (int k = 0; k < 4; ++k) out[(c * nl + l) * 4 + k] = dev[(l * kTraceCtas + c) * 4 + k];
    *nphase = (int32_t)nl;
    *nctas = kTraceCtas;
    return SPEC_OK;
}

spec_status spec_trace_kinds(spec_handle h, int32_t* out, int32_t capacity, int32_t* count) {
    if (!h || !out || !count) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    if (!h->trace || !h->tracing) return fail(SPEC_ERR_STATE, "no traced pass");
    const size_t nl = h->trace_kinds.size();
    if ((size_t)capacity < nl) return fail(SPEC_ERR_INVALID_ARG, "need %zu entries", nl);
    for (size_t i = 0; i < nl; ++i) out[i] = h->trace_kinds[i];
    *count = (int32_t)nl;
    return SPEC_OK;
}

spec_status spec_profile_read(spec_handle h, int32_t kind, double* total_ms, double* total_bytes, int32_t* launches) {
    if (!h || !total_ms || !total_bytes || !launches) return fail(SPEC_ERR_INVALID_ARG, "null argument");
    CU(cudaStreamSynchronize(h->stream));
    double ms = 0.0, bytes = 0.0;
    int count = 0;
    std::vector<spec_model::ProfRec> keep;
    for (auto& r : h->prof) {
        const bool take = kind == -1 ? (r.kind != EPI_EXPERT_SWIGLU && r.kind != EPI_EXPERT_DOWN) : (kind == -2 || r.kind == kind);
        if (!take) {
            keep.push_back(r);
            continue;
        }
        float t = 0.f;
        CU(cudaEventElapsedTime(&t, r.a, r.b));
        ms += t;
        bytes += r.bytes;
        ++count;
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    *total_ms = ms;
    *total_bytes = bytes;
    *launches = count;
    h->prof = keep;
    return SPEC_OK;
}

}  // extern "C"
