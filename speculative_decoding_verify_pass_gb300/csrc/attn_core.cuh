// Attention building blocks of the attention kernels (attention.cu).
//
// A unit is (kv head h, 128-position chunk c); its 8 warps split each group
// of 16 query rows by keys for S = Q K^T and by output dimensions for O = P V
// (bf16 tensor-core MMA, fp32 accumulation).  The unit writes one partial
// (row max, row sum, unnormalised O) per row into the slot of its chunk's
// group (chunk mod S, S fixed per model), merging it into the chunks of the
// group that came before; the grouping depends only on absolute positions,
// so a query's result never depends on the block size.  A merge step
// combines the groups of a row in increasing order.
#pragma once

#include <math.h>

#include "internal.h"

namespace sv {
namespace attn_core {

constexpr int kAttnUnitThreads = 256;  // 8 warps (named barrier 1)
constexpr int kAttnCombThreads = 64;   // merge kernel: 2 warps, one merged row each

// Shared-memory scratch of one row-group slot: row maxima and row sums per
// key group [8][16] and the P fragments [8 key groups][32 lanes][8 words].
constexpr int kAttnSlotBytes = 2 * 8 * 16 * 4 + 8 * 32 * 8 * 4;
constexpr int kAttnScratchBytes = 4 * kAttnSlotBytes;  // up to 4 row groups at once
// Query rows in shared memory are padded by 8 elements so that the eight rows
// a fragment load touches fall in different banks.
template <int HD>
__host__ __device__ constexpr int q_stride() { return HD + 8; }

// Merging two partials of one row, (m1, l1, O1) then (m2, l2, O2), maxima in
// the log2 domain (-1e30 for a row with no key): with M = max(m1, m2), each
// part is weighted by exp2(m - M).  A part with no key gets weight exactly
// zero and the other weight exactly one, so merging an empty chunk changes
// nothing.
__device__ __forceinline__ float2 merge2(float2 o1, float m1, float2 o2, float m2) {
    const float M = fmaxf(m1, m2);
    const float w1 = exp2f(m1 - M), w2 = exp2f(m2 - M);
    return make_float2(o1.x * w1 + o2.x * w2, o1.y * w1 + o2.y * w2);
}
__device__ __forceinline__ float2 merge_ml(float2 a, float2 b) {
    const float M = fmaxf(a.x, b.x);
    return make_float2(M, a.y * exp2f(a.x - M) + b.y * exp2f(b.x - M));
}

// One unit (kv head h, 128-position chunk) with all 8 warps.  sk0/sk1 and
// sv0/sv1 are the K and V slabs of the chunk's two pages.
//
// The n*G query rows are taken in groups of 16.  C warps cooperate on a row
// group (C = 8, 4 or 2 as 1, 2 or up to 4 groups are present; C = 8 always
// when `slots` is 1, the groups then taken one after another).  The chunk's
// 128 keys are 8 key groups of 16 and the head dimension is split in tiles of
// 16; a warp takes 8/C key groups for S = Q K^T and a 1/C share of the dim
// tiles for O = P V.  For every C the arithmetic of a row is the same:
//  - S per key group: two MMA chains (even / odd k16 steps), added;
//  - row max over all keys (exact); P = exp2(S*scale*log2e - max), kept as a
//    bf16 high part plus a bf16 low part (~16 significant bits);
//  - row sum: within a key group over its 16 keys in a fixed lane order,
//    then over the key groups in order;
//  - O per dim tile: four MMA chains (P high / low x even / odd key group)
//    over the key groups in order, then (c0 + c1) + (c2 + c3).
// So a row's result depends neither on the block size nor on C.  The unit
// writes one partial (row max in the log2 domain, row sum, unnormalised O)
// per row.  wait_slabs() is called once, after the first query fragments are
// requested and before any slab is read.  The attention kernel picks C from
// the number of row groups.  qs, when given, holds the unit's
// query rows in shared memory ([R][HD+8]); otherwise they are read from
// global memory.  scratch holds `slots` slot areas of kAttnSlotBytes.
template <int HD, int C, class WaitSlabs>
__device__ __forceinline__ void attn_unit_c(const AttnParams& a, const uint16_t* sk0, const uint16_t* sk1,
                                            const uint16_t* sv0, const uint16_t* sv1, float* scratch,
                                            const uint16_t* qs, int h, int chunk, int pos0, int n, size_t seq_base,
                                            int group, bool accumulate, bool flush, float* run_o, float2* run_ml,
                                            int tid, WaitSlabs& wait_slabs) {
    constexpr int kTiles = HD / 16;                                   // dim tiles
    constexpr int par = 8 / C;                                        // row groups at once
    constexpr int kgs = 8 / C;                                        // key groups per warp
    constexpr int tpw = kTiles / C > 0 ? kTiles / C : 1;              // dim tiles per warp
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, cc = lane & 3;
    const int G = a.n_heads / a.n_kv_heads;
    const int R = n * G;
    const int nrg = (R + 15) / 16;
    const int slot = warp / C, sub = warp % C;
    float* smax = scratch + slot * (kAttnSlotBytes / 4);              // [8][16]
    float* ssum = smax + 128;                                         // [8][16]
    uint32_t* pf = reinterpret_cast<uint32_t*>(smax + 256);           // [8][32][8]
    const float k2 = a.scale_log2;
    // the partial of (kv head h, chunk group) runs in shared memory (run_o
    // [row][HD], run_ml [row]): with `accumulate` it already holds the group's
    // earlier chunks and this chunk is merged into it; with `flush` (the
    // group's last chunk of this pass) it is then written to global memory
    const size_t base = seq_base + ((size_t)h * a.nch + group) * 64;
    // barrier of the C warps sharing a slot (the whole CTA when C = 8)
    auto slot_sync = [&] {
        if (C == 8)
            named_bar_sync(1, kAttnUnitThreads);
        else
            named_bar_sync(2 + slot, 32 * C);
    };
    bool waited = false;
    for (int rg0 = 0; rg0 < nrg; rg0 += par) {
        const int rg = rg0 + slot;
        const bool act = rg < nrg;   // whole slots idle only in the last round
        const int rA = rg * 16 + g, rB = rA + 8;
        uint32_t qf[HD / 16][4];
        if (act) {
            const uint16_t* qa = rA >= R ? nullptr
                                 : qs ? qs + (size_t)rA * q_stride<HD>()
                                      : a.qbuf + ((size_t)(rA / G) * a.n_heads + h * G + rA % G) * HD;
            const uint16_t* qb = rB >= R ? nullptr
                                 : qs ? qs + (size_t)rB * q_stride<HD>()
                                      : a.qbuf + ((size_t)(rB / G) * a.n_heads + h * G + rB % G) * HD;
#pragma unroll
            for (int k16 = 0; k16 < HD / 16; ++k16) {
                qf[k16][0] = qa ? *reinterpret_cast<const uint32_t*>(qa + k16 * 16 + 2 * cc) : 0u;
                qf[k16][1] = qb ? *reinterpret_cast<const uint32_t*>(qb + k16 * 16 + 2 * cc) : 0u;
                qf[k16][2] = qa ? *reinterpret_cast<const uint32_t*>(qa + k16 * 16 + 8 + 2 * cc) : 0u;
                qf[k16][3] = qb ? *reinterpret_cast<const uint32_t*>(qb + k16 * 16 + 8 + 2 * cc) : 0u;
            }
        }
        if (!waited) {
            wait_slabs();
            waited = true;
        }
        const int limA = rA < R ? pos0 + rA / G : -1;
        const int limB = rB < R ? pos0 + rB / G : -1;
        // the group's earlier maxima, read before any thread of the slot
        // writes the merged ones (after the slot's next barrier)
        float moA = -1e30f, moB = -1e30f;
        if (accumulate && act) {
            if (rA < R) moA = run_ml[rA].x;
            if (rB < R) moB = run_ml[rB].x;
        }
        float s[kgs][2][4];   // this warp's key groups
        if (act) {
#pragma unroll
            for (int q = 0; q < kgs; ++q) {
                const int kg = sub * kgs + q;
                const uint16_t* sk = kg < 4 ? sk0 : sk1;
                float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    const uint16_t* krow = sk + ((kg & 3) * 16 + t * 8 + g) * HD;
#pragma unroll
                    for (int k16 = 0; k16 < HD / 16; ++k16) {
                        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + (((2 * k16) ^ g) << 3) + 2 * cc);
                        const uint32_t b1 =
                            *reinterpret_cast<const uint32_t*>(krow + (((2 * k16 + 1) ^ g) << 3) + 2 * cc);
                        mma_bf16_16816(s2[k16 & 1], qf[k16], b0, b1);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[q][t][e] = s2[0][e] + s2[1][e];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kp = chunk * kAttnChunk + kg * 16 + t * 8 + 2 * cc + e;
                        if (kp > limA) s[q][t][e] = -INFINITY;
                        if (kp > limB) s[q][t][2 + e] = -INFINITY;
                        mA = fmaxf(mA, s[q][t][e]);
                        mB = fmaxf(mB, s[q][t][2 + e]);
                    }
                }
#pragma unroll
                for (int off = 1; off <= 2; off <<= 1) {
                    mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
                    mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, off));
                }
                if (cc == 0) {
                    smax[kg * 16 + g] = mA;
                    smax[kg * 16 + g + 8] = mB;
                }
            }
        }
        slot_sync();
        float MA = -INFINITY, MB = -INFINITY;
#pragma unroll
        for (int kg = 0; kg < 8; ++kg) {
            MA = fmaxf(MA, smax[kg * 16 + g]);
            MB = fmaxf(MB, smax[kg * 16 + g + 8]);
        }
        const float msA = (MA == -INFINITY) ? -1e30f : MA * k2;
        const float msB = (MB == -INFINITY) ? -1e30f : MB * k2;
        if (act) {
#pragma unroll
            for (int q = 0; q < kgs; ++q) {
                const int kg = sub * kgs + q;
                float lA = 0.f, lB = 0.f;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    s[q][t][0] = exp2f(s[q][t][0] * k2 - msA);
                    s[q][t][1] = exp2f(s[q][t][1] * k2 - msA);
                    s[q][t][2] = exp2f(s[q][t][2] * k2 - msB);
                    s[q][t][3] = exp2f(s[q][t][3] * k2 - msB);
                    lA += s[q][t][0] + s[q][t][1];
                    lB += s[q][t][2] + s[q][t][3];
                }
#pragma unroll
                for (int off = 1; off <= 2; off <<= 1) {
                    lA += __shfl_xor_sync(0xffffffffu, lA, off);
                    lB += __shfl_xor_sync(0xffffffffu, lB, off);
                }
                if (cc == 0) {
                    ssum[kg * 16 + g] = lA;
                    ssum[kg * 16 + g + 8] = lB;
                }
                // S accumulator layout = m16k16 A layout: P of key group kg
                const float src[8] = {s[q][0][0], s[q][0][1], s[q][0][2], s[q][0][3],
                                      s[q][1][0], s[q][1][1], s[q][1][2], s[q][1][3]};
                float hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    hi[e] = bf_round(src[e]);
                    lo[e] = src[e] - hi[e];
                }
                uint4* dst = reinterpret_cast<uint4*>(pf + (kg * 32 + lane) * 8);
                dst[0] = make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]), pack_bf16x2(hi[4], hi[5]),
                                    pack_bf16x2(hi[6], hi[7]));
                dst[1] = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]), pack_bf16x2(lo[4], lo[5]),
                                    pack_bf16x2(lo[6], lo[7]));
            }
        }
        slot_sync();
        if (act) {
            const int mi = lane >> 3, ri = lane & 7;
            for (int q = 0; q < tpw; ++q) {
                const int tile = sub * tpw + q;
                if (tile >= kTiles) break;
                float oc[4][2][4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int t = 0; t < 2; ++t) oc[c4][t][0] = oc[c4][t][1] = oc[c4][t][2] = oc[c4][t][3] = 0.f;
                const int chunk16 = tile * 2 + (mi >> 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint4* src = reinterpret_cast<const uint4*>(pf + (kk * 32 + lane) * 8);
                    const uint4 h4 = src[0], l4 = src[1];
                    const uint32_t ph[4] = {h4.x, h4.y, h4.z, h4.w};
                    const uint32_t pl[4] = {l4.x, l4.y, l4.z, l4.w};
                    const uint16_t* svv = kk < 4 ? sv0 : sv1;
                    const int key = (kk & 3) * 16 + (mi & 1) * 8 + ri;
                    uint32_t r[4];
                    ldmatrix_x4_trans(r, smem_u32(svv + key * HD + ((chunk16 ^ ri) << 3)));
                    const int pp = kk & 1;
                    mma_bf16_16816(oc[pp][0], ph, r[0], r[1]);
                    mma_bf16_16816(oc[pp][1], ph, r[2], r[3]);
                    mma_bf16_16816(oc[2 + pp][0], pl, r[0], r[1]);
                    mma_bf16_16816(oc[2 + pp][1], pl, r[2], r[3]);
                }
                // this thread owns the same elements of the running partial
                // for every chunk, so it merges them without a barrier
                if (rA < R) {
                    float* run = run_o + rA * HD + tile * 16;
                    float* dst = a.part_o + (base + rA) * HD + tile * 16;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        float2 v = make_float2((oc[0][t][0] + oc[1][t][0]) + (oc[2][t][0] + oc[3][t][0]),
                                               (oc[0][t][1] + oc[1][t][1]) + (oc[2][t][1] + oc[3][t][1]));
                        if (accumulate) v = merge2(*reinterpret_cast<const float2*>(run + t * 8 + 2 * cc), moA, v, msA);
                        if (flush)
                            *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) = v;
                        else
                            *reinterpret_cast<float2*>(run + t * 8 + 2 * cc) = v;
                    }
                }
                if (rB < R) {
                    float* run = run_o + rB * HD + tile * 16;
                    float* dst = a.part_o + (base + rB) * HD + tile * 16;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        float2 v = make_float2((oc[0][t][2] + oc[1][t][2]) + (oc[2][t][2] + oc[3][t][2]),
                                               (oc[0][t][3] + oc[1][t][3]) + (oc[2][t][3] + oc[3][t][3]));
                        if (accumulate) v = merge2(*reinterpret_cast<const float2*>(run + t * 8 + 2 * cc), moB, v, msB);
                        if (flush)
                            *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) = v;
                        else
                            *reinterpret_cast<float2*>(run + t * 8 + 2 * cc) = v;
                    }
                }
            }
            if (sub == 0 && cc == 0) {
                float LA = 0.f, LB = 0.f;
#pragma unroll
                for (int kg = 0; kg < 8; ++kg) {
                    LA += ssum[kg * 16 + g];
                    LB += ssum[kg * 16 + g + 8];
                }
                if (rA < R) {
                    float2 ml = make_float2(msA, LA);
                    if (accumulate) ml = merge_ml(run_ml[rA], ml);
                    if (flush) a.part_ml[base + rA] = ml;
                    else run_ml[rA] = ml;
                }
                if (rB < R) {
                    float2 ml = make_float2(msB, LB);
                    if (accumulate) ml = merge_ml(run_ml[rB], ml);
                    if (flush) a.part_ml[base + rB] = ml;
                    else run_ml[rB] = ml;
                }
            }
        }
        if (rg0 + par < nrg) slot_sync();   // the slot's scratch is reused by the next round
    }
}

// Rows (query head, token) u0, u0+ustep, ...: one warp per row merges the nc
// chunk partials in chunk order and writes the bf16 output into the O
// projection's operand.  Each lane owns HD/32 consecutive dimensions.  The
// first kFirst chunks' partial outputs are loaded together with the chunk
// statistics (their addresses do not depend on them), so a row of up to
// kFirst chunks costs one round trip to L2 and issues no load after it: the
// next GEMM's weight prefetch starts with this kernel, and a load queued
// behind it waits microseconds.  Every lane reads every chunk's
// (max, sum) (uniform loads) and forms the same weights; the sums run in
// chunk order, so a row's result does not depend on the block size.
template <int HD>
__device__ __forceinline__ void comb_rows(const AttnParams& a, int u0, int ustep, int lane, int nc) {
    constexpr int V = HD / 32;   // dimensions per lane: 4 (hd 128) or 2 (hd 64)
    constexpr int kFirst = 20;
    const int G = a.n_heads / a.n_kv_heads;
    const int nseq = a.seq_len ? a.nseq : 1;
    const int per = a.n_heads * a.n;            // rows of one sequence
    const int U = per * nseq;
    const size_t cstride = (size_t)64 * HD;
    for (int u = u0; u < U; u += ustep) {
        const int sq = u / per, uu = u - sq * per;
        const int qh = uu % a.n_heads, jl = uu / a.n_heads;
        const int j = sq * a.n + jl;              // the row of the pass
        if (a.seq_len) {                          // this sequence's own chunk count
            const int tot = a.seq_len[sq] + a.n;
            nc = (tot + kAttnChunk - 1) / kAttnChunk;
            if (nc > a.nch) nc = a.nch;
            if (nc > a.groups) nc = a.groups;
        }
        const int h = qh / G, r = jl * G + qh % G;
        const size_t sbase = (size_t)sq * a.n_kv_heads * a.nch * 64;
        const float2* ml = a.part_ml + sbase + (size_t)h * a.nch * 64 + r;
        const float* po = a.part_o + (sbase + (size_t)h * a.nch * 64 + r) * HD + lane * V;
        // the first kFirst chunks' outputs and (max, sum) in one sweep of
        // independent loads (one L2 round trip), later chunks' maxima after
        float ob[kFirst][V];
        float2 sf[kFirst];
#pragma unroll
        for (int t = 0; t < kFirst; ++t) {
            if (t < nc) {
                if constexpr (V == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(po + (size_t)t * cstride);
                    ob[t][0] = v.x; ob[t][1] = v.y; ob[t][2] = v.z; ob[t][3] = v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(po + (size_t)t * cstride);
                    ob[t][0] = v.x; ob[t][1] = v.y;
                }
                sf[t] = ml[(size_t)t * 64];
            }
        }
        float M = -1e30f;
#pragma unroll
        for (int t = 0; t < kFirst; ++t)
            if (t < nc) M = fmaxf(M, sf[t].x);
        for (int c0 = kFirst; c0 < nc; c0 += 8) {   // longer rows: eight statistics loads in flight
            float m[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) m[t] = c0 + t < nc ? ml[(size_t)(c0 + t) * 64].x : -1e30f;
#pragma unroll
            for (int t = 0; t < 8; ++t) M = fmaxf(M, m[t]);
        }
        float L = 0.f, O[V];
#pragma unroll
        for (int e = 0; e < V; ++e) O[e] = 0.f;
#pragma unroll
        for (int t = 0; t < kFirst; ++t) {
            if (t < nc) {
                const float2 st = sf[t];
                const float w = exp2f(st.x - M);
                L += w * st.y;
#pragma unroll
                for (int e = 0; e < V; ++e) O[e] += w * ob[t][e];
            }
        }
        for (int c0 = kFirst; c0 < nc; c0 += 8) {   // longer rows: eight chunks in flight
            float ov[8][V];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (c0 + t < nc) {
#pragma unroll
                    for (int e = 0; e < V; ++e) ov[t][e] = po[(size_t)(c0 + t) * cstride + e];
                }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (c0 + t < nc) {
                    const float2 st = ml[(size_t)(c0 + t) * 64];
                    const float w = exp2f(st.x - M);
                    L += w * st.y;
#pragma unroll
                    for (int e = 0; e < V; ++e) O[e] += w * ov[t][e];
                }
            }
        }
        const int k = qh * HD + lane * V;
#pragma unroll
        for (int e = 0; e < V; e += 2) {
            const int kk = (k + e) & 63;
            *reinterpret_cast<uint32_t*>(a.xf_out + (size_t)((k + e) >> 6) * kStageXBytes + xfrag_offset(j, kk)) =
                pack_bf16x2(O[e] / L, O[e + 1] / L);
        }
    }
}

}  // namespace attn_core
}  // namespace sv
