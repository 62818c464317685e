// Grouped-query attention of a verify block over the paged KV cache.
//
// Query token j of the block sits at position p+j and attends to keys
// 0..p+j (causal inside the block; LayerSkip summary 4.3.2: all drafted
// positions are verified in one parallel pass).  The work is split over fixed
// absolute chunks of 128 positions (two 64-position pages), one CTA per
// (kv head, chunk):
//  * both pages' K and V slabs arrive by 1-D bulk copies (they are contiguous
//    in the page layout, and stored chunk-swizzled so fragment loads are
//    bank-conflict free);
//  * the n*G query rows (G query heads per kv head, <= 64 rows) are taken 16
//    at a time; the 8 warps split S = Q K^T by keys (16 each) and O = P V by
//    output dimensions (16 each), on bf16 tensor-core MMA with fp32
//    accumulation, P as a bf16 high part plus a bf16 low part;
//  * the CTA writes one (row max, row sum, unnormalised O) per row; a merge
//    kernel (one warp per query head and token) combines the chunks in
//    increasing order.
// Chunk boundaries are absolute positions, so a query's result does not
// depend on the block size n; chunks entirely past a query's last key
// contribute exactly zero.
#include <math.h>

#include "attn_core.cuh"

namespace sv {

namespace {

constexpr int kAttnThreads = attn_core::kAttnUnitThreads;  // 8 warps: 4 row groups x 2 pages

template <int HD>
__global__ void __maxnreg__(192) attn_partial_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint16_t* sk = reinterpret_cast<uint16_t*>(smem_raw);
    uint16_t* svv = sk + kAttnChunk * HD;
    __shared__ uint64_t bar;

    const int h = blockIdx.x, chunk = blockIdx.y, sq = blockIdx.z;   // sq: sequence (batched passes)
    const int tid = threadIdx.x;
    const int cta = (sq * gridDim.y + chunk) * gridDim.x + h;
    long long* tr = (p.trace && cta < kTraceCtas && tid == 0) ? p.trace + (size_t)cta * 4 : nullptr;
    if (tr) tr[0] = trace_clock();
    // The cache length and the keys/values of positions before it were
    // written by kernels that completed before the preceding QKV kernel
    // passed its own dependency wait, so they may be read before ours; only
    // the block's new rows (positions >= pos0) come from the QKV kernel.
    const int pos0 = p.seq_len ? p.seq_len[sq] : p.st->len[p.which];
    const int total = pos0 + p.n;
    const int* btab = p.block_table + (p.seq_len ? sq * p.seq_pages : 0);
    const int start = chunk * kAttnChunk;
    if (start >= total || total > p.nch * kAttnChunk) {
        pdl_wait();
        pdl_launch_dependents();
        if (total > p.nch * kAttnChunk && tid == 0) atomicCAS(&p.st->error, 0, 20);  // beyond the pages
        if (tr) tr[3] = trace_clock();
        return;
    }
    constexpr uint32_t kSlab = kPageSize * HD * 2;
    auto issue = [&](int pg) {
        const int page = btab[start / kPageSize + pg];
        const size_t off = ((size_t)(page * p.n_kv_heads + h) * kPageSize) * HD;
        bulk_g2s(sk + pg * kPageSize * HD, p.kpool + off, kSlab, &bar);
        bulk_g2s(svv + pg * kPageSize * HD, p.vpool + off, kSlab, &bar);
    };
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar, 4 * kSlab);
        for (int pg = 0; pg < 2; ++pg)
            if (start + (pg + 1) * kPageSize <= pos0) issue(pg);  // fully cached page: load now
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tr) tr[1] = trace_clock();
    if (tid == 0)
        for (int pg = 0; pg < 2; ++pg)
            if (start + (pg + 1) * kPageSize > pos0) issue(pg);   // holds new rows
    // the unit's query rows into shared memory (one round trip for all row groups)
    float* scratch = reinterpret_cast<float*>(smem_raw + 2 * kAttnChunk * HD * 2);
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem_raw + 2 * kAttnChunk * HD * 2 + attn_core::kAttnScratchBytes);
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
    attn_core::attn_unit<HD>(p, sk, sk + kPageSize * HD, svv, svv + kPageSize * HD, scratch, qs, 4, h, chunk, pos0, p.n,
                             seq_base, tid,
                             [&] {
                                 mbar_wait(&bar, 0, &p.st->error, 3);
                                 if (tr) tr[2] = trace_clock();
                             });
    if (tr) tr[3] = trace_clock();
}

// Two rows (query head, token) per CTA, one warp each: the chunk partials
// of a row merged in chunk order.  At most 184 registers a thread, so that a
// merge CTA (64 threads) fits beside a streaming-GEMM CTA (320 threads at up
// to 168): the next GEMM's CTAs must find room to prefetch their weights
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

// Slabs + scratch, padded so that two units never share an SM: a unit's
// slab loads then have a whole SM's share of HBM bandwidth.
constexpr int attn_smem_used(int hd) {
    return 2 * kAttnChunk * hd * 2 + attn_core::kAttnScratchBytes + kMaxBlock * 4 * (hd + 8) * 2;  // slabs, scratch, q
}
constexpr int attn_smem(int hd) { return attn_smem_used(hd) > 116 * 1024 ? attn_smem_used(hd) : 116 * 1024; }

cudaError_t attention_configure(int device) {
    (void)device;
    cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_smem(128));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_partial_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem(64));
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl) {
    AttnParams q = p;
    void* args[] = {&q};
    cudaError_t e;
    const int nseq = p.seq_len ? p.nseq : 1;
    const dim3 g1((unsigned)p.n_kv_heads, (unsigned)p.nch, (unsigned)nseq);
    const dim3 g2((unsigned)((nseq * p.n_heads * p.n + attn_core::kAttnCombThreads / 32 - 1) / (attn_core::kAttnCombThreads / 32)));
    if (p.head_dim == 128)
        e = launch_pdl((const void*)attn_partial_kernel<128>, g1, dim3(kAttnThreads), attn_smem(128), s, pdl, args);
    else if (p.head_dim == 64)
        e = launch_pdl((const void*)attn_partial_kernel<64>, g1, dim3(kAttnThreads), attn_smem(64), s, pdl, args);
    else
        return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    const void* comb = p.head_dim == 128 ? (const void*)attn_combine_kernel<128> : (const void*)attn_combine_kernel<64>;
    return launch_pdl(comb, g2, dim3(attn_core::kAttnCombThreads), 0, s, pdl, args);
}

}  // namespace sv
