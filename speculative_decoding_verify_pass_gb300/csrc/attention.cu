// Grouped-query attention of a verify block over the paged KV cache, on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Query token j of the block sits at position p+j and attends to keys
// 0..p+j (causal inside the block; LayerSkip summary 4.3.2: all drafted
// positions are verified in one parallel pass).  The work is split over fixed
// absolute chunks of 128 positions (two 64-position pages); a CTA takes the
// chunk groups y, y + gridDim.y, ... of one kv head (group g holds the chunks
// c with c mod S = g, S fixed per model: about the SMs per kv head) and loads
// the next chunk's pages while it computes one.  The block's n*G query rows
// of the kv head (R <= 64) are the narrow side of every product, so keys and
// head dimensions run along the 128 tensor-memory lanes.  Per chunk:
//  * the chunk's K and V pages arrive by 1-D bulk copies; the cache keeps
//    them in the tensor core's canonical K-major layout (K: rows = positions,
//    k = dims; V: rows = dims, k = positions), so each slab is an MMA operand
//    as it lies;
//  * one thread issues S^T = K Q^T (M = 128 keys, N = R rounded up to 16,
//    K = head dim) into tensor memory;
//  * every key's thread reads its S^T row; the row maximum over the chunk's
//    visible keys is exact (an integer warp reduction, then across the four
//    lane quadrants); P = exp2(S*scale*log2e - max) is kept as a bf16 high
//    part plus a bf16 low part (~16 significant bits) and written as P^T, an
//    MN-major operand (a 16-byte core-matrix row holds one key's 8 query
//    rows; each column quad of 4 rows writes half of one);
//  * the row sum of P is exact in 24-bit fixed point (each P rounded to a
//    multiple of 2^-24, integer sums over the warp and the four quadrants),
//    so it is the same whatever the order of the terms;
//  * the issuing thread runs O^T = V^T P^T (M = head dims, N as above, K = 128
//    keys, high part then low part) into tensor memory;
//  * while those MMAs run, one thread per query row takes the row's merge
//    weights, running max and running sum;
//  * every head dimension's thread merges O into the running partial of the
//    chunk group (in tensor memory) or, for the group's last chunk, writes
//    the group's unnormalised O and, per row, (max, sum) to global memory; a
//    merge kernel (one warp per query head and token) combines the groups in
//    increasing order.
// Chunk boundaries are absolute positions, the grouping depends on nothing
// else, and a query row's arithmetic never involves another row, so a
// query's result does not depend on the block size n or on how many
// sequences share the pass; chunks entirely past a query's last key
// contribute exactly zero.
#include <math.h>

#include "attn_core.cuh"

namespace sv {

namespace {

constexpr int kRowWarps = 16;                     // four per TMEM lane quadrant: column quads hc, hc + 4, ..
constexpr int kIssuerWarp = kRowWarps;            // bulk copies and MMAs (one elected thread)
constexpr int kAttnThreads = 32 * (kRowWarps + 1);
constexpr int kMaxRows = 64;                      // n * G query rows per kv head (G <= 4, n <= 16)

// Shared memory, from the dynamic base: Q [64 rows][HD] K-major (rows x
// dims); P^T high and low parts [64 rows][128 keys], MN-major (8-row groups
// 2 KB apart, 8-key groups 128 bytes apart, each 16-byte row of a core matrix
// = one key's 8 query rows); then two chunk buffers (K page 0, K page 1, V
// page 0, V page 1).  For HD = 64 an M = 128 MMA over V^T reads 64 rows past
// a V page (their results are never read): the tail pad keeps that inside the
// allocation.
template <int HD>
struct AttnLayout {
    static constexpr int kQ = 0;
    static constexpr int kPh = kMaxRows * HD * 2;
    static constexpr int kPl = kPh + kMaxRows * kAttnChunk * 2;
    static constexpr int kBuf = kPl + kMaxRows * kAttnChunk * 2;
    static constexpr uint32_t kSlab = kPageSize * HD * 2;   // one page of K or V
    static constexpr int kBufBytes = 4 * kSlab;
    static constexpr int kBytes = kBuf + 2 * kBufBytes + (HD < 128 ? (int)kSlab : 0);
    static constexpr uint32_t kSbo = (HD / 8) * 128;        // Q and K: next 8-row group
};
// tensor-memory columns (of 256): S^T, O^T, the group's running O^T
constexpr uint32_t kColS = 0, kColO = 64, kColRun = 128, kTmemCols = 256;
constexpr float kFix = 16777216.f;   // 2^24: the fixed-point scale of the row sums

// The bounded mbarrier wait, out of line: one copy of its polling loop.
__device__ __noinline__ bool wait_bar(uint64_t* bar, uint32_t parity, int* err, int site) {
    return mbar_wait(bar, parity, err, site);
}

// Bounded wait used only after a failed one: lets copies or MMAs already in
// flight finish before the CTA releases its memory.
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 20) && !mbar_try_wait(bar, parity); ++i) __nanosleep(64);
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_partial_kernel(const __grid_constant__ AttnParams p) {
    using L = AttnLayout<HD>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full[2], s_done, p_ready, o_done;
    __shared__ uint32_t tmem_base;
    __shared__ __align__(16) float xmax[4][kMaxRows];   // per lane quadrant (32 keys) and row: max of S
    __shared__ __align__(16) float2 xw[kMaxRows];       // per row: this chunk's merge weights (w_run, w_chunk)
    __shared__ __align__(16) uint32_t xl[4][kMaxRows];  // per lane quadrant and row: fixed-point sum of P
    __shared__ __align__(16) float rowm[2][kMaxRows];   // per row: the group's running max, by chunk parity
    __shared__ __align__(16) float rowl[2][kMaxRows];   // and running sum
    __shared__ __align__(16) int lastkey[kMaxRows];     // per row: its last visible key position (-1: no row)

    const int h = blockIdx.x, y = blockIdx.y, ystep = gridDim.y, sq = blockIdx.z;   // sq: sequence
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = (sq * gridDim.y + y) * gridDim.x + h;
    long long* trc = (p.trace && cta < kTraceCtas) ? p.trace + (size_t)cta * 4 : nullptr;
    long long* tr = tid == 0 ? trc : nullptr;
    if (tr) tr[0] = trace_clock();
    int* err = &p.st->error;
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
        if (total > p.nch * kAttnChunk && tid == 0) atomicCAS(err, 0, 20);  // beyond the pages
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
    uint8_t* qs = smem_raw + L::kQ;
    uint8_t* ph = smem_raw + L::kPh;
    uint8_t* pl = smem_raw + L::kPl;
    uint8_t* bufs = smem_raw + L::kBuf;
    // page pg (0, 1) of chunk c into buffer b: the K slab, then the V slab
    auto issue = [&](int c, int b, int pg) {
        const int page = btab[c * (kAttnChunk / kPageSize) + pg];
        const size_t off = ((size_t)(page * p.n_kv_heads + h) * kPageSize) * HD;
        uint8_t* dst = bufs + b * L::kBufBytes;
        bulk_g2s(dst + pg * L::kSlab, p.kpool + off, L::kSlab, &full[b]);
        bulk_g2s(dst + (2 + pg) * L::kSlab, p.vpool + off, L::kSlab, &full[b]);
    };
    const int G = p.n_heads / p.n_kv_heads, R = p.n * G;
    const int Rp = (R + 15) & ~15;    // MMA N: the rows rounded up to 16
    const int2 first = make_int2(y, y), second = step(first);
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&s_done, 1);
        mbar_init(&o_done, 1);
        mbar_init(&p_ready, kRowWarps);
        fence_barrier_init();
    }
    if (warp == kIssuerWarp) tmem_alloc(&tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == kIssuerWarp) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[0], 4 * L::kSlab);
            if (second.x >= 0) mbar_arrive_expect_tx(&full[1], 4 * L::kSlab);
            for (int pg = 0; pg < 2; ++pg) {   // fully cached pages (no new row of this pass): load now
                if (first.y * kAttnChunk + (pg + 1) * kPageSize <= pos0) issue(first.y, 0, pg);
                if (second.x >= 0 && second.y * kAttnChunk + (pg + 1) * kPageSize <= pos0) issue(second.y, 1, pg);
            }
        }
        pdl_wait();
        pdl_launch_dependents();
        if (lane == 0)
            for (int pg = 0; pg < 2; ++pg) {   // pages that hold new rows
                if (first.y * kAttnChunk + (pg + 1) * kPageSize > pos0) issue(first.y, 0, pg);
                if (second.x >= 0 && second.y * kAttnChunk + (pg + 1) * kPageSize > pos0) issue(second.y, 1, pg);
            }
    } else {
        pdl_wait();
        pdl_launch_dependents();
        if (tr) tr[1] = trace_clock();
        // the query rows (row r: token r / G, query head h*G + r % G),
        // K-major; rows R..63 zero
        const uint16_t* qsrc = p.qbuf + (size_t)sq * p.n * p.n_heads * HD;
        for (int c = tid; c < kMaxRows * (HD / 8); c += 32 * kRowWarps) {
            const int r = c / (HD / 8), d8 = c % (HD / 8);
            uint8_t* dst = qs + ((r >> 3) * (HD / 8) + d8) * 128 + (r & 7) * 16;
            if (r < R)
                cp_async16(dst, qsrc + ((size_t)(r / G) * p.n_heads + h * G + r % G) * HD + d8 * 8);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        // P^T zero (its live 8-row groups are rewritten every chunk)
        for (int c = tid; c < 2 * kMaxRows * kAttnChunk / 8; c += 32 * kRowWarps)
            *reinterpret_cast<uint4*>(ph + c * 16) = make_uint4(0u, 0u, 0u, 0u);   // P_hi then P_lo
        if (tid < kMaxRows) lastkey[tid] = tid < R ? pos0 + tid / G : -1;
        cp_async_wait_all();
        fence_proxy_async_smem();   // the tensor core reads Q and P^T
    }
    __syncthreads();

    if (warp == kIssuerWarp) {
        // ---------------- bulk copies and MMAs (one thread) ----------------
        if (lane == 0) {
            const uint32_t idS = umma_idesc_bf16(128, Rp);
            const uint32_t idO = umma_idesc_bf16(128, Rp) | (1u << 16);   // B = P^T, MN-major
            const uint32_t qa = smem_u32(qs), pha = smem_u32(ph), pla = smem_u32(pl), ba = smem_u32(bufs);
            // descriptors advance by adding (bytes >> 4) to their start-address field
            const uint64_t dq = umma_desc_kmajor(qa, 128, L::kSbo);
            const uint64_t dk0 = umma_desc_kmajor(ba, 128, L::kSbo);
            const uint64_t dv0 = umma_desc_kmajor(ba + 2 * L::kSlab, 128, 8 * 128);
            const uint64_t dph = umma_desc_kmajor(pha, 128, 16 * 128), dpl = umma_desc_kmajor(pla, 128, 16 * 128);
            // S^T = K Q^T: K = HD in steps of 16 (two core matrices, 256 bytes)
            auto issue_S = [&](int b) {
                const uint64_t dk = dk0 + (uint64_t)(b * L::kBufBytes >> 4);
#pragma unroll
                for (int ks = 0; ks < HD / 16; ++ks) umma_bf16_id(tmem + kColS, dk + ks * 16, dq + ks * 16, idS, ks > 0);
                umma_commit(&s_done);
            };
            // O^T = V^T P^T: K = 128 keys in steps of 16 (V page kk/4, its
            // 8-position groups 2(kk%4), +1; the next 8-dim group 1 KB on;
            // P^T's next 8-row group 2 KB on), the high part, then the low part
            auto issue_O = [&](int b) {
                const uint64_t dv = dv0 + (uint64_t)(b * L::kBufBytes >> 4);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kAttnChunk / 16; ++kk) {
                        const uint64_t pd = (part ? dpl : dph) + kk * 16;
                        umma_bf16_id(tmem + kColO, dv + (uint64_t)(((kk >> 2) * L::kSlab + (kk & 3) * 256) >> 4), pd, idO,
                                     (part | kk) != 0);
                    }
                umma_commit(&o_done);
            };
            bool ok = wait_bar(&full[0], 0, err, 3);
            if (trc) trc[2] = trace_clock();
            tc_fence_after();
            int armed = 2, waited = 1, s_commits = 0, o_commits = 0;   // chunk copies set up / waited for
            if (ok) {
                issue_S(0);
                ++s_commits;
            }
            int2 cur = first, nxt = second, ahead = step(second);
            for (int i = 0; cur.x >= 0; ++i) {
                const int b = i & 1;
                ok = ok && wait_bar(&p_ready, i & 1, err, 21);   // P^T of chunk i is in shared memory
                tc_fence_after();
                if (ok) {
                    issue_O(b);
                    ++o_commits;
                }
                if (nxt.x >= 0) {   // S^T of the next chunk while this one is merged
                    ok = ok && wait_bar(&full[b ^ 1], ((i + 1) >> 1) & 1, err, 22);
                    if (ok) ++waited;
                    tc_fence_after();
                    if (ok) {
                        issue_S(b ^ 1);
                        ++s_commits;
                    }
                }
                if (ahead.x >= 0) {   // the chunk after next into buffer b once O^T has read it
                    ok = ok && wait_bar(&o_done, i & 1, err, 23);
                    if (ok) {
                        mbar_arrive_expect_tx(&full[b], 4 * L::kSlab);
                        issue(ahead.y, b, 0);
                        issue(ahead.y, b, 1);
                        ++armed;
                    }
                }
                cur = nxt;
                nxt = ahead;
                ahead = step(ahead);
            }
            if (!ok) {   // a wait gave up: let what is in flight land before the CTA ends
                for (int c = waited; c < armed && c < waited + 2; ++c) drain(&full[c & 1], (c >> 1) & 1);
                if (s_commits) drain(&s_done, (s_commits - 1) & 1);
                if (o_commits) drain(&o_done, (o_commits - 1) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---- one thread per key (softmax) and per head dimension (merge) ----
        // The warp's column quads (4 query rows each): 4 q4 .. +3 for q4 = hc, hc + 4, ...
        const int qd = warp & 3, hc = warp >> 2;      // lane quadrant, first column quad
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        const int key = qd * 32 + lane;               // this thread's key in the chunk (TMEM lane)
        const int d = qd * 32 + lane;                 // and head dimension in the merge
        const bool dims = d < HD;                     // lanes holding head dimensions (HD = 64: quadrants 0, 1)
        const float k2 = p.scale_log2;
        const size_t seq_base = (size_t)sq * p.n_kv_heads * p.nch * 64;
        const int nquad = (R + 3) >> 2;               // column quads holding live rows
        // this key's 16-byte row of a P^T core matrix
        const int pkey = (key >> 3) * 128 + (key & 7) * 16;
        bool ok = true;
        int2 cur = first;
        for (int i = 0; cur.x >= 0; ++i) {
            const int2 nx = step(cur);
            const bool accumulate = cur.y != cur.x, flush = nx.x != cur.x;
            const int par = i & 1;
            const int kp = cur.y * kAttnChunk + key;  // this key's position
            ok = ok && wait_bar(&s_done, i & 1, err, 24);
            tc_fence_after();
#pragma unroll 1
            for (int q4 = hc; q4 < nquad; q4 += 4) {   // this quadrant's maximum of each row
                float v[4];
                tmem_ld4(tl + kColS + 4 * q4, v);
                const int4 lim = *reinterpret_cast<const int4*>(&lastkey[4 * q4]);
                const float m0 = warp_max_exact(kp > lim.x ? -INFINITY : v[0]);   // past the row's last key: none
                const float m1 = warp_max_exact(kp > lim.y ? -INFINITY : v[1]);
                const float m2 = warp_max_exact(kp > lim.z ? -INFINITY : v[2]);
                const float m3 = warp_max_exact(kp > lim.w ? -INFINITY : v[3]);
                if (lane == 0) *reinterpret_cast<float4*>(&xmax[qd][4 * q4]) = make_float4(m0, m1, m2, m3);
            }
            named_bar_sync(1, 32 * kRowWarps);   // every quadrant's maxima are in
#pragma unroll 1
            for (int q4 = hc; q4 < nquad; q4 += 4) {   // P = exp2(S * scale * log2 e - max), high and low parts
                float v[4];
                tmem_ld4(tl + kColS + 4 * q4, v);
                const int4 lim = *reinterpret_cast<const int4*>(&lastkey[4 * q4]);
                const int lims[4] = {lim.x, lim.y, lim.z, lim.w};
                const float4 a0 = *reinterpret_cast<const float4*>(&xmax[0][4 * q4]);
                const float4 a1 = *reinterpret_cast<const float4*>(&xmax[1][4 * q4]);
                const float4 a2 = *reinterpret_cast<const float4*>(&xmax[2][4 * q4]);
                const float4 a3 = *reinterpret_cast<const float4*>(&xmax[3][4 * q4]);
                const float M[4] = {fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x)), fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y)),
                                    fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z)), fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w))};
                float ms[4], pv[4], hv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ms[j] = M[j] == -INFINITY ? -1e30f : M[j] * k2;   // -1e30: no visible key
                    pv[j] = kp > lims[j] ? 0.f : ex2_approx(v[j] * k2 - ms[j]);
                    hv[j] = bf_round(pv[j]);
                }
                // the quadrant's fixed-point sums of P per row (exact)
                const uint32_t s0 = warp_sum_u32(__float2uint_rn(pv[0] * kFix)), s1 = warp_sum_u32(__float2uint_rn(pv[1] * kFix));
                const uint32_t s2 = warp_sum_u32(__float2uint_rn(pv[2] * kFix)), s3 = warp_sum_u32(__float2uint_rn(pv[3] * kFix));
                if (lane == 0) *reinterpret_cast<uint4*>(&xl[qd][4 * q4]) = make_uint4(s0, s1, s2, s3);
                const int off = (q4 >> 1) * 2048 + pkey + (q4 & 1) * 8;   // the 8-row group, this quad's half
                *reinterpret_cast<uint2*>(ph + off) = make_uint2(pack_bf16x2(hv[0], hv[1]), pack_bf16x2(hv[2], hv[3]));
                *reinterpret_cast<uint2*>(pl + off) =
                    make_uint2(pack_bf16x2(pv[0] - hv[0], pv[1] - hv[1]), pack_bf16x2(pv[2] - hv[2], pv[3] - hv[3]));
            }
            fence_proxy_async_smem();   // P^T is read by the tensor core
            tc_fence_before();          // the S^T reads are done before the next S^T is written
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_ready);
            named_bar_sync(1, 32 * kRowWarps);   // every quadrant's sums of P are in
            const size_t prow = seq_base + ((size_t)h * p.nch + cur.x) * 64;   // the group's partial rows
            if (tid < R) {
                // one thread per row, while the O^T MMAs run (off the lane
                // quadrants' loops, which would otherwise all wait for the
                // warps that did this): the chunk's merge weights in the log2
                // domain, the group's running max and running sum
                const int c = tid;
                const float M = fmaxf(fmaxf(xmax[0][c], xmax[1][c]), fmaxf(xmax[2][c], xmax[3][c]));
                const float msj = M == -INFINITY ? -1e30f : M * k2;
                float w1 = 0.f, w2 = 1.f, mn = msj;
                if (accumulate) {
                    const float mr = rowm[par][c];
                    mn = fmaxf(mr, msj);
                    w1 = ex2_approx(mr - mn);
                    w2 = ex2_approx(msj - mn);
                }
                xw[c] = make_float2(w1, w2);
                const float lc = (float)(xl[0][c] + xl[1][c] + xl[2][c] + xl[3][c]) * (1.f / kFix);
                const float ln = accumulate ? rowl[par][c] * w1 + lc * w2 : lc;
                if (flush) p.part_ml[prow + c] = make_float2(mn, ln);
                rowm[par ^ 1][c] = mn;
                rowl[par ^ 1][c] = ln;
            }
            ok = ok && wait_bar(&o_done, i & 1, err, 25);
            tc_fence_after();
            named_bar_sync(1, 32 * kRowWarps);   // this chunk's weights are in
#pragma unroll 1
            for (int q4 = hc; q4 < nquad; q4 += 4) {   // merge into the group's running O, or write it out
                if (dims) {
                    float o[4];
                    tmem_ld4(tl + kColO + 4 * q4, o);
                    if (accumulate) {
                        float run[4];
                        tmem_ld4(tl + kColRun + 4 * q4, run);
                        const float4 wa = *reinterpret_cast<const float4*>(&xw[4 * q4]);
                        const float4 wb = *reinterpret_cast<const float4*>(&xw[4 * q4 + 2]);
                        o[0] = run[0] * wa.x + o[0] * wa.y;
                        o[1] = run[1] * wa.z + o[1] * wa.w;
                        o[2] = run[2] * wb.x + o[2] * wb.y;
                        o[3] = run[3] * wb.z + o[3] * wb.w;
                    }
                    if (flush) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (4 * q4 + j < R) p.part_o[(prow + 4 * q4 + j) * HD + d] = o[j];
                    } else {
                        tmem_st4(tl + kColRun + 4 * q4, o);
                    }
                }
            }
            cur = nx;
        }
    }
    tc_fence_before();
    __syncthreads();   // every TMEM access of the CTA is done
    if (warp == kIssuerWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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

cudaError_t attention_configure(int device) {
    (void)device;
    cudaError_t e = cudaFuncSetAttribute((const void*)attn_partial_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, AttnLayout<128>::kBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute((const void*)attn_partial_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnLayout<64>::kBytes);
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s, bool pdl) {
    AttnParams q = p;
    void* args[] = {&q};
    cudaError_t e;
    const int nseq = p.seq_len ? p.nseq : 1;
    if (p.n * (p.n_heads / p.n_kv_heads) > kMaxRows) return cudaErrorInvalidValue;
    // about one CTA per SM over (kv head, sequence), each taking every
    // gridDim.y-th chunk group: a long context no longer runs in several waves
    int ysplit = (p.num_sms + p.n_kv_heads * nseq - 1) / (p.n_kv_heads * nseq);
    if (ysplit < 1) ysplit = 1;
    if (ysplit > p.groups) ysplit = p.groups;
    const dim3 g1((unsigned)p.n_kv_heads, (unsigned)ysplit, (unsigned)nseq);
    const dim3 g2((unsigned)((nseq * p.n_heads * p.n + attn_core::kAttnCombThreads / 32 - 1) / (attn_core::kAttnCombThreads / 32)));
    if (p.head_dim == 128)
        e = launch_pdl((const void*)attn_partial_kernel<128>, g1, dim3(kAttnThreads), AttnLayout<128>::kBytes, s, pdl, args);
    else if (p.head_dim == 64)
        e = launch_pdl((const void*)attn_partial_kernel<64>, g1, dim3(kAttnThreads), AttnLayout<64>::kBytes, s, pdl, args);
    else
        return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    const void* comb = p.head_dim == 128 ? (const void*)attn_combine_kernel<128> : (const void*)attn_combine_kernel<64>;
    return launch_pdl(comb, g2, dim3(attn_core::kAttnCombThreads), 0, s, pdl, args);
}

}  // namespace sv
