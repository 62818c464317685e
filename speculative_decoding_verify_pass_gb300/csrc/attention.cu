// Grouped-query attention of a verify block over the paged KV cache.
//
// Query token j of the block sits at position p+j and attends to keys
// 0..p+j (causal inside the block; LayerSkip summary 4.3.2: all drafted
// positions are verified in one parallel pass).  The work is split over fixed
// absolute chunks of 128 positions (two 64-position pages); a CTA takes
// every gridDim.y-th chunk of one kv head (about one CTA per SM in all) and
// loads the next chunk's slabs while it computes one.  Per chunk:
//  * both pages' K and V slabs arrive by 1-D bulk copies (they are contiguous
//    in the page layout, and stored chunk-swizzled so fragment loads are
//    bank-conflict free);
//  * the n*G query rows (G query heads per kv head, <= 64 rows) are taken 16
//    at a time; the 8 warps split S = Q K^T by keys (16 each) and O = P V by
//    output dimensions (16 each), on bf16 tensor-core MMA with fp32
//    accumulation, P as a bf16 high part plus a bf16 low part;
//  * the CTA merges one (row max, row sum, unnormalised O) per row into the
//    partial of the chunk's group (chunk mod S, S fixed per model: about the
//    SMs per kv head); a merge kernel (one warp per query head and token)
//    combines the groups in increasing order.
// Chunk boundaries are absolute positions and the grouping depends on
// nothing else, so a query's result does not depend on the block size n or
// on how many sequences share the pass; chunks entirely past a query's last
// key contribute exactly zero.
#include <math.h>

#include "attn_core.cuh"

namespace sv {

namespace {

constexpr int kAttnThreads = attn_core::kAttnUnitThreads;  // 8 warps: 4 row groups x 2 pages

// C: warps per group of 16 query rows (8, 4 or 2 as 1, 2 or up to 4 groups
// are present; attn_core::attn_unit_c), chosen by the host from n * G.
template <int HD, int C>
__global__ void __maxnreg__(192) attn_partial_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr int kBuf = 2 * kAttnChunk * HD;     // one chunk's K and V slabs (elements)
    uint16_t* slabs = reinterpret_cast<uint16_t*>(smem_raw);   // two buffers
    __shared__ uint64_t bar[2];

    // Chunk c belongs to group c mod S (S = p.groups, fixed per model); the
    // group's partial merges its chunks in increasing order.  CTA (h, y)
    // takes the groups y, y + gridDim.y, ... of kv head h, chunk after
    // chunk, loading the next chunk's slabs while it computes one.
    const int h = blockIdx.x, y = blockIdx.y, ystep = gridDim.y, sq = blockIdx.z;   // sq: sequence
    const int tid = threadIdx.x;
    const int cta = (sq * gridDim.y + y) * gridDim.x + h;
    long long* tr = (p.trace && cta < kTraceCtas && tid == 0) ? p.trace + (size_t)cta * 4 : nullptr;
    if (tr) tr[0] = trace_clock();
    // The cache length and the keys/values of positions before it were
    // written by kernels that completed before the preceding QKV kernel
    // passed its own dependency wait, so they may be read before ours; only
    // the block's new rows (positions >= pos0) come from the QKV kernel.
    const int pos0 = p.seq_len ? p.seq_len[sq] : p.st->len[p.which];
    const int total = pos0 + p.n;
    const int* btab = p.block_table + (p.seq_len ? sq * p.seq_pages : 0);
    const int S = p.groups;
    const int need = (total + kAttnChunk - 1) / kAttnChunk;   // chunks holding keys of this pass
    const int gmax = need < S ? need : S;                      // groups holding them
    if (y >= gmax || total > p.nch * kAttnChunk) {
        pdl_wait();
        pdl_launch_dependents();
        if (total > p.nch * kAttnChunk && tid == 0) atomicCAS(&p.st->error, 0, 20);  // beyond the pages
        if (tr) tr[3] = trace_clock();
        return;
    }
    // this CTA's chunks in order: (group, chunk); group -1 ends the list
    auto step = [&](int2 t) -> int2 {
        if (t.x < 0) return t;
        if (t.y + S < need) return make_int2(t.x, t.y + S);
        const int g = t.x + ystep;
        return g < gmax ? make_int2(g, g) : make_int2(-1, -1);
    };
    constexpr uint32_t kSlab = kPageSize * HD * 2;
    // page pg (0, 1) of chunk c into buffer b: K then V slab
    auto issue = [&](int c, int b, int pg) {
        const int page = btab[c * (kAttnChunk / kPageSize) + pg];
        const size_t off = ((size_t)(page * p.n_kv_heads + h) * kPageSize) * HD;
        uint16_t* sk = slabs + b * kBuf;
        bulk_g2s(sk + pg * kPageSize * HD, p.kpool + off, kSlab, &bar[b]);
        bulk_g2s(sk + kAttnChunk * HD + pg * kPageSize * HD, p.vpool + off, kSlab, &bar[b]);
    };
    const int2 first = make_int2(y, y), second = step(first);
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar[0], 4 * kSlab);
        if (second.x >= 0) mbar_arrive_expect_tx(&bar[1], 4 * kSlab);
        // fully cached pages (no new row of this pass): load now
        for (int pg = 0; pg < 2; ++pg) {
            if (first.y * kAttnChunk + (pg + 1) * kPageSize <= pos0) issue(first.y, 0, pg);
            if (second.x >= 0 && second.y * kAttnChunk + (pg + 1) * kPageSize <= pos0) issue(second.y, 1, pg);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tr) tr[1] = trace_clock();
    if (tid == 0)
        for (int pg = 0; pg < 2; ++pg) {   // pages that hold new rows
            if (first.y * kAttnChunk + (pg + 1) * kPageSize > pos0) issue(first.y, 0, pg);
            if (second.x >= 0 && second.y * kAttnChunk + (pg + 1) * kPageSize > pos0) issue(second.y, 1, pg);
        }
    // the unit's query rows into shared memory (one round trip for all row groups)
    float* scratch = reinterpret_cast<float*>(smem_raw + 2 * kBuf * 2);
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem_raw + 2 * kBuf * 2 + attn_core::kAttnScratchBytes);
    // the running partial of the current chunk group: [64 rows][HD] + [64]
    float* run_o = reinterpret_cast<float*>(smem_raw + 2 * kBuf * 2 + attn_core::kAttnScratchBytes +
                                            kMaxBlock * 4 * attn_core::q_stride<HD>() * 2);
    float2* run_ml = reinterpret_cast<float2*>(run_o + 64 * HD);
    const int G = p.n_heads / p.n_kv_heads, R = p.n * G;
    const uint16_t* qsrc = p.qbuf + (size_t)sq * p.n * p.n_heads * HD;   // this sequence's query rows
    for (int c = tid; c < R * (HD / 8); c += kAttnThreads) {
        const int r = c / (HD / 8), q = c % (HD / 8);
        cp_async16(qs + r * attn_core::q_stride<HD>() + q * 8,
                   qsrc + ((size_t)(r / G) * p.n_heads + h * G + r % G) * HD + q * 8);
    }
    cp_async_wait_all();
    __syncthreads();
    const size_t seq_base = (size_t)sq * p.n_kv_heads * p.nch * 64;
    int2 cur = first, ahead = step(second);
    for (int i = 0; cur.x >= 0; ++i) {
        const int b = i & 1;
        const uint16_t* sk = slabs + b * kBuf;
        const uint16_t* svv = sk + kAttnChunk * HD;
        auto wait = [&] {
            mbar_wait(&bar[b], (uint32_t)((i >> 1) & 1), &p.st->error, 3);
            if (tr && i == 0) tr[2] = trace_clock();
        };
        const int2 nxt = step(cur);
        attn_core::attn_unit_c<HD, C>(p, sk, sk + kPageSize * HD, svv, svv + kPageSize * HD, scratch, qs, h, cur.y,
                                      pos0, p.n, seq_base, cur.x, cur.y != cur.x, nxt.x != cur.x, run_o, run_ml,
                                      tid, wait);
        __syncthreads();   // every warp is done with buffer b, the scratch and the running partial
        if (tid == 0 && ahead.x >= 0) {   // the chunk after next into the freed buffer
            mbar_arrive_expect_tx(&bar[b], 4 * kSlab);
            issue(ahead.y, b, 0);
            issue(ahead.y, b, 1);
        }
        cur = nxt;
        ahead = step(ahead);
    }
    if (tr) tr[3] = trace_clock();
}

// Two rows (query head, token) per CTA, one warp each: the group partials
// of a row merged in group order.  At most 184 registers a thread, so that a
// merge CTA (64 threads) fits beside a streaming-GEMM CTA (384 threads at up
// to 136): the next GEMM's CTAs must find room to prefetch their weights
// while the merge runs.
template <int HD>
__global__ void __maxnreg__(184) attn_combine_kernel(const __grid_constant__ AttnParams p) {
    long long* tr = (p.trace && blockIdx.x < kTraceCtas && threadIdx.x == 0)
                        ? p.trace + (size_t)(kTraceCtas + blockIdx.x) * 4 : nullptr;
    if (tr) tr[0] = trace_clock();
    pdl_wait();
    pdl_launch_dependents();
    if (tr) tr[1] = trace_clock();
    const int total = p.st->len[p.which] + p.n;   // batched passes: per sequence, in comb_rows
    int nc = (total + kAttnChunk - 1) / kAttnChunk;
    if (nc > p.nch) nc = p.nch;
    if (nc > p.groups) nc = p.groups;              // partials: one per chunk group
    constexpr int kWarps = attn_core::kAttnCombThreads / 32;
    attn_core::comb_rows<HD>(p, blockIdx.x * kWarps + (threadIdx.x >> 5), gridDim.x * kWarps, threadIdx.x & 31, nc);
    if (tr) tr[3] = trace_clock();
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

// Two chunks' slabs + scratch + query rows + the running group partial,
// padded so that two units never share an SM: a unit's slab loads then have
// a whole SM's share of HBM bandwidth.
constexpr int attn_smem_used(int hd) {
    return 2 * 2 * kAttnChunk * hd * 2 + attn_core::kAttnScratchBytes + kMaxBlock * 4 * (hd + 8) * 2 +
           64 * hd * 4 + 64 * 8;
}
constexpr int attn_smem(int hd) { return attn_smem_used(hd) > 116 * 1024 ? attn_smem_used(hd) : 116 * 1024; }

cudaError_t attention_configure(int device) {
    (void)device;
    const void* fns[6] = {(const void*)attn_partial_kernel<128, 8>, (const void*)attn_partial_kernel<128, 4>,
                          (const void*)attn_partial_kernel<128, 2>, (const void*)attn_partial_kernel<64, 8>,
                          (const void*)attn_partial_kernel<64, 4>, (const void*)attn_partial_kernel<64, 2>};
    for (int k = 0; k < 6; ++k) {
        const cudaError_t e = cudaFuncSetAttribute(fns[k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   attn_smem(k < 3 ? 128 : 64));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl) {
    AttnParams q = p;
    void* args[] = {&q};
    cudaError_t e;
    const int nseq = p.seq_len ? p.nseq : 1;
    // about one CTA per SM over (kv head, sequence), each taking every
    // gridDim.y-th chunk group: a long context no longer runs in several waves
    int ysplit = (p.num_sms + p.n_kv_heads * nseq - 1) / (p.n_kv_heads * nseq);
    if (ysplit < 1) ysplit = 1;
    if (ysplit > p.groups) ysplit = p.groups;
    const dim3 g1((unsigned)p.n_kv_heads, (unsigned)ysplit, (unsigned)nseq);
    const dim3 g2((unsigned)((nseq * p.n_heads * p.n + attn_core::kAttnCombThreads / 32 - 1) / (attn_core::kAttnCombThreads / 32)));
    const int nrg = (p.n * (p.n_heads / p.n_kv_heads) + 15) / 16;   // groups of 16 query rows
    const int ci = nrg <= 1 ? 0 : (nrg <= 2 ? 1 : 2);                 // C = 8, 4, 2
    const void* fn128[3] = {(const void*)attn_partial_kernel<128, 8>, (const void*)attn_partial_kernel<128, 4>,
                            (const void*)attn_partial_kernel<128, 2>};
    const void* fn64[3] = {(const void*)attn_partial_kernel<64, 8>, (const void*)attn_partial_kernel<64, 4>,
                           (const void*)attn_partial_kernel<64, 2>};
    if (p.head_dim == 128)
        e = launch_pdl(fn128[ci], g1, dim3(kAttnThreads), attn_smem(128), s, pdl, args);
    else if (p.head_dim == 64)
        e = launch_pdl(fn64[ci], g1, dim3(kAttnThreads), attn_smem(64), s, pdl, args);
    else
        return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    const void* comb = p.head_dim == 128 ? (const void*)attn_combine_kernel<128> : (const void*)attn_combine_kernel<64>;
    return launch_pdl(comb, g2, dim3(attn_core::kAttnCombThreads), 0, s, pdl, args);
}

}  // namespace sv
