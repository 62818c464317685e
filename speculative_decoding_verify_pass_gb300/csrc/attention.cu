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
//  * the n*G query rows of the kv head's G query heads (<= 64) are split over
//    4 warps of 16 rows; S = Q K^T and O = P V run on bf16 tensor-core MMA
//    with fp32 accumulation, P rounded to bf16;
//  * each CTA writes (row max, row sum, unnormalised O) for its chunk, and a
//    combine kernel merges the chunks in increasing order.
// Chunk boundaries are absolute positions, so a query's result does not
// depend on the block size n; chunks entirely past a query's last key
// contribute exactly zero.
#include <math.h>

#include "internal.h"

namespace sv {

namespace {

constexpr int kAttnThreads = 128;
constexpr int kMaxChunks = 512;  // 65536 positions / 128

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_partial_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint16_t* sk = reinterpret_cast<uint16_t*>(smem_raw);
    uint16_t* svv = sk + kAttnChunk * HD;
    __shared__ uint64_t bar;

    const int h = blockIdx.x, chunk = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();
    pdl_wait();
    const int pos0 = p.st->len[p.which];
    const int total = pos0 + p.n;
    const int start = chunk * kAttnChunk;
    if (start >= total) return;
    if (total > p.nch * kAttnChunk) {  // positions beyond the allocated pages
        if (tid == 0) atomicCAS(&p.st->error, 0, 20);
        return;
    }
    const int G = p.n_heads / p.n_kv_heads;
    const int R = p.n * G;
    constexpr uint32_t kSlab = kPageSize * HD * 2;

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar, 4 * kSlab);
        for (int pg = 0; pg < 2; ++pg) {
            const int page = p.block_table[start / kPageSize + pg];
            const size_t off = ((size_t)(page * p.n_kv_heads + h) * kPageSize) * HD;
            bulk_g2s(sk + pg * kPageSize * HD, p.kpool + off, kSlab, &bar);
            bulk_g2s(svv + pg * kPageSize * HD, p.vpool + off, kSlab, &bar);
        }
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, &p.st->error, 3);
    (void)ok;

    const int r0 = warp * 16;
    if (r0 >= R) return;
    const int g = lane >> 2, cc = lane & 3;
    const int rA = r0 + g, rB = rA + 8;
    const uint16_t* qa = nullptr;
    const uint16_t* qb = nullptr;
    if (rA < R) qa = p.qbuf + ((size_t)(rA / G) * p.n_heads + h * G + rA % G) * HD;
    if (rB < R) qb = p.qbuf + ((size_t)(rB / G) * p.n_heads + h * G + rB % G) * HD;

    uint32_t qf[HD / 16][4];
#pragma unroll
    for (int k16 = 0; k16 < HD / 16; ++k16) {
        qf[k16][0] = qa ? *reinterpret_cast<const uint32_t*>(qa + k16 * 16 + 2 * cc) : 0u;
        qf[k16][1] = qb ? *reinterpret_cast<const uint32_t*>(qb + k16 * 16 + 2 * cc) : 0u;
        qf[k16][2] = qa ? *reinterpret_cast<const uint32_t*>(qa + k16 * 16 + 8 + 2 * cc) : 0u;
        qf[k16][3] = qb ? *reinterpret_cast<const uint32_t*>(qb + k16 * 16 + 8 + 2 * cc) : 0u;
    }

    // S = Q K^T over the chunk's 128 keys (16 tiles of 8 keys)
    float s[16][4];
#pragma unroll
    for (int n8 = 0; n8 < 16; ++n8) {
        s[n8][0] = s[n8][1] = s[n8][2] = s[n8][3] = 0.f;
        const int key = n8 * 8 + g;
        const uint16_t* krow = sk + key * HD;
#pragma unroll
        for (int k16 = 0; k16 < HD / 16; ++k16) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + (((2 * k16) ^ g) << 3) + 2 * cc);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + (((2 * k16 + 1) ^ g) << 3) + 2 * cc);
            mma_bf16_16816(s[n8], qf[k16], b0, b1);
        }
    }

    // causal mask by absolute position, row max
    const int limA = rA < R ? pos0 + rA / G : -1;
    const int limB = rB < R ? pos0 + rB / G : -1;
    float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
    for (int n8 = 0; n8 < 16; ++n8)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int kp = start + n8 * 8 + 2 * cc + e;
            if (kp > limA) s[n8][e] = -INFINITY;
            if (kp > limB) s[n8][2 + e] = -INFINITY;
            mA = fmaxf(mA, s[n8][e]);
            mB = fmaxf(mB, s[n8][2 + e]);
        }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, o));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, o));
    }
    const float k2 = p.scale_log2;
    const float msA = (mA == -INFINITY) ? -1e30f : mA * k2;
    const float msB = (mB == -INFINITY) ? -1e30f : mB * k2;
    float lA = 0.f, lB = 0.f;
#pragma unroll
    for (int n8 = 0; n8 < 16; ++n8) {
        s[n8][0] = exp2f(s[n8][0] * k2 - msA);
        s[n8][1] = exp2f(s[n8][1] * k2 - msA);
        s[n8][2] = exp2f(s[n8][2] * k2 - msB);
        s[n8][3] = exp2f(s[n8][3] * k2 - msB);
        lA += s[n8][0] + s[n8][1];
        lB += s[n8][2] + s[n8][3];
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, o);
        lB += __shfl_xor_sync(0xffffffffu, lB, o);
    }

    // O = P V (P as bf16 A fragments straight from the S accumulators)
    float o[HD / 8][4];
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t pa[4] = {pack_bf16x2(s[2 * kk][0], s[2 * kk][1]), pack_bf16x2(s[2 * kk][2], s[2 * kk][3]),
                                pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
        const int key = kk * 16 + (mi & 1) * 8 + ri;
#pragma unroll
        for (int np = 0; np < HD / 16; ++np) {
            const int chunk16 = np * 2 + (mi >> 1);
            uint32_t r[4];
            ldmatrix_x4_trans(r, smem_u32(svv + key * HD + ((chunk16 ^ ri) << 3)));
            mma_bf16_16816(o[2 * np], pa, r[0], r[1]);
            mma_bf16_16816(o[2 * np + 1], pa, r[2], r[3]);
        }
    }

    const size_t base = (size_t)(h * p.nch + chunk) * 64;
    if (rA < R) {
        float* dst = p.part_o + (base + rA) * HD;
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) = make_float2(o[t][0], o[t][1]);
        if (cc == 0) p.part_ml[base + rA] = make_float2(msA, lA);
    }
    if (rB < R) {
        float* dst = p.part_o + (base + rB) * HD;
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) = make_float2(o[t][2], o[t][3]);
        if (cc == 0) p.part_ml[base + rB] = make_float2(msB, lB);
    }
}

// One CTA per (query head, token): merge the chunks in increasing order and
// write the bf16 attention output into the O projection's operand.
template <int HD>
__global__ void __launch_bounds__(HD) attn_combine_kernel(const __grid_constant__ AttnParams p) {
    __shared__ float w_s[kMaxChunks];
    __shared__ float l_s[kMaxChunks];
    const int qh = blockIdx.x, j = blockIdx.y, dim = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    const int G = p.n_heads / p.n_kv_heads;
    const int h = qh / G, r = j * G + qh % G;
    const int total = p.st->len[p.which] + p.n;
    int nc = (total + kAttnChunk - 1) / kAttnChunk;
    if (nc > p.nch) nc = p.nch;
    if (nc > kMaxChunks) nc = kMaxChunks;
    // all chunk statistics in parallel, then the merge weights
    for (int c = dim; c < nc; c += HD) {
        const float2 ml = p.part_ml[(size_t)(h * p.nch + c) * 64 + r];
        w_s[c] = ml.x;
        l_s[c] = ml.y;
    }
    __syncthreads();
    float M = -1e30f;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, w_s[c]);
    float L = 0.f;
    for (int c = 0; c < nc; ++c) L += exp2f(w_s[c] - M) * l_s[c];
    __syncthreads();
    for (int c = dim; c < nc; c += HD) w_s[c] = exp2f(w_s[c] - M);
    __syncthreads();
    // unnormalised outputs: independent loads, summed in chunk order
    const float* po = p.part_o + ((size_t)h * p.nch * 64 + r) * HD + dim;
    const size_t cstride = (size_t)64 * HD;
    float O = 0.f;
    int c = 0;
    for (; c + 8 <= nc; c += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = po[(size_t)(c + u) * cstride];
#pragma unroll
        for (int u = 0; u < 8; ++u) O += w_s[c + u] * v[u];
    }
    for (; c < nc; ++c) O += w_s[c] * po[(size_t)c * cstride];
    const int k = qh * HD + dim;
    *reinterpret_cast<uint16_t*>(p.xf_out + (size_t)(k >> 6) * kStageXBytes + xfrag_offset(j, k & 63)) = f2bf(O / L);
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

cudaError_t attention_configure(int device) {
    (void)device;
    cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         2 * kAttnChunk * 128 * 2);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_partial_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                2 * kAttnChunk * 64 * 2);
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl) {
    AttnParams q = p;
    void* args[] = {&q};
    cudaError_t e;
    const dim3 g1((unsigned)p.n_kv_heads, (unsigned)p.nch), g2((unsigned)p.n_heads, (unsigned)p.n);
    if (p.head_dim == 128) {
        e = launch_pdl((const void*)attn_partial_kernel<128>, g1, dim3(kAttnThreads), 2 * kAttnChunk * 128 * 2, s, pdl,
                       args);
        if (e != cudaSuccess) return e;
        return launch_pdl((const void*)attn_combine_kernel<128>, g2, dim3(128), 0, s, pdl, args);
    }
    if (p.head_dim == 64) {
        e = launch_pdl((const void*)attn_partial_kernel<64>, g1, dim3(kAttnThreads), 2 * kAttnChunk * 64 * 2, s, pdl,
                       args);
        if (e != cudaSuccess) return e;
        return launch_pdl((const void*)attn_combine_kernel<64>, g2, dim3(64), 0, s, pdl, args);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sv
