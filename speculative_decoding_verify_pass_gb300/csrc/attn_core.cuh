// Attention building blocks shared by the standalone attention kernels and
// the persistent pass kernel.
//
// A unit is (kv head h, 128-position chunk c).  Its 8 warps split the work as
// 4 groups of 16 query rows x the chunk's 2 pages of 64 keys; each warp runs
// S = Q K^T and O = P V on bf16 tensor-core MMA with fp32 accumulation (P as
// a bf16 high part plus a bf16 low part, ~16 significant bits).  The
// two pages of a row group are then merged in shared memory (page 0 first)
// and the unit writes one partial (row max, row sum, unnormalised O) per row:
// partials are indexed by absolute chunk, so a query's result never depends on
// the block size.  A merge step combines the chunks of a row in increasing
// chunk order.
#pragma once

#include <math.h>

#include "internal.h"

namespace sv {
namespace attn_core {

constexpr int kAttnUnitThreads = 256;  // 8 warps (named barrier 1)
constexpr int kAttnCombThreads = 64;   // merge kernel: 2 warps, one merged row each

// One warp's 16 rows (row group rg) against one 64-key page slab (keys
// key0..key0+63 in absolute positions).  Outputs stay in registers.
template <int HD>
__device__ __forceinline__ void attn_rows(const AttnParams& a, const uint16_t* sk, const uint16_t* svv, int h,
                                          int key0, int pos0, int rg, int lane, float (&o)[HD / 8][4], float& msA,
                                          float& lA, float& msB, float& lB) {
    const int G = a.n_heads / a.n_kv_heads;
    const int R = a.n * G;
    const int g = lane >> 2, cc = lane & 3;
    const int rA = rg * 16 + g, rB = rA + 8;
    const uint16_t* qa = rA < R ? a.qbuf + ((size_t)(rA / G) * a.n_heads + h * G + rA % G) * HD : nullptr;
    const uint16_t* qb = rB < R ? a.qbuf + ((size_t)(rB / G) * a.n_heads + h * G + rB % G) * HD : nullptr;
    uint32_t qf[HD / 16][4];
#pragma unroll
    for (int k16 = 0; k16 < HD / 16; ++k16) {
        qf[k16][0] = qa ? *reinterpret_cast<const uint32_t*>(qa + k16 * 16 + 2 * cc) : 0u;
        qf[k16][1] = qb ? *reinterpret_cast<const uint32_t*>(qb + k16 * 16 + 2 * cc) : 0u;
        qf[k16][2] = qa ? *reinterpret_cast<const uint32_t*>(qa + k16 * 16 + 8 + 2 * cc) : 0u;
        qf[k16][3] = qb ? *reinterpret_cast<const uint32_t*>(qb + k16 * 16 + 8 + 2 * cc) : 0u;
    }
    float s[8][4];
#pragma unroll
    for (int n8 = 0; n8 < 8; ++n8) {
        s[n8][0] = s[n8][1] = s[n8][2] = s[n8][3] = 0.f;
        const uint16_t* krow = sk + (n8 * 8 + g) * HD;
#pragma unroll
        for (int k16 = 0; k16 < HD / 16; ++k16) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + (((2 * k16) ^ g) << 3) + 2 * cc);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + (((2 * k16 + 1) ^ g) << 3) + 2 * cc);
            mma_bf16_16816(s[n8], qf[k16], b0, b1);
        }
    }
    const int limA = rA < R ? pos0 + rA / G : -1;
    const int limB = rB < R ? pos0 + rB / G : -1;
    float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
    for (int n8 = 0; n8 < 8; ++n8)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int kp = key0 + n8 * 8 + 2 * cc + e;
            if (kp > limA) s[n8][e] = -INFINITY;
            if (kp > limB) s[n8][2 + e] = -INFINITY;
            mA = fmaxf(mA, s[n8][e]);
            mB = fmaxf(mB, s[n8][2 + e]);
        }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, off));
    }
    const float k2 = a.scale_log2;
    msA = (mA == -INFINITY) ? -1e30f : mA * k2;
    msB = (mB == -INFINITY) ? -1e30f : mB * k2;
    lA = 0.f;
    lB = 0.f;
#pragma unroll
    for (int n8 = 0; n8 < 8; ++n8) {
        s[n8][0] = exp2f(s[n8][0] * k2 - msA);
        s[n8][1] = exp2f(s[n8][1] * k2 - msA);
        s[n8][2] = exp2f(s[n8][2] * k2 - msB);
        s[n8][3] = exp2f(s[n8][3] * k2 - msB);
        lA += s[n8][0] + s[n8][1];
        lB += s[n8][2] + s[n8][3];
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, off);
        lB += __shfl_xor_sync(0xffffffffu, lB, off);
    }
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    const int mi = lane >> 3, ri = lane & 7;
    // P = P_hi + P_lo, both bf16: two MMAs keep ~16 bits of the fp32 weights
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        float hi[8], lo[8];
        const float src[8] = {s[2 * kk][0], s[2 * kk][1], s[2 * kk][2], s[2 * kk][3],
                              s[2 * kk + 1][0], s[2 * kk + 1][1], s[2 * kk + 1][2], s[2 * kk + 1][3]};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            hi[e] = bf_round(src[e]);
            lo[e] = src[e] - hi[e];
        }
        const uint32_t ph[4] = {pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]), pack_bf16x2(hi[4], hi[5]),
                                pack_bf16x2(hi[6], hi[7])};
        const uint32_t pl[4] = {pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]), pack_bf16x2(lo[4], lo[5]),
                                pack_bf16x2(lo[6], lo[7])};
        const int key = kk * 16 + (mi & 1) * 8 + ri;
#pragma unroll
        for (int np = 0; np < HD / 16; ++np) {
            const int chunk16 = np * 2 + (mi >> 1);
            uint32_t r[4];
            ldmatrix_x4_trans(r, smem_u32(svv + key * HD + ((chunk16 ^ ri) << 3)));
            mma_bf16_16816(o[2 * np], ph, r[0], r[1]);
            mma_bf16_16816(o[2 * np + 1], ph, r[2], r[3]);
            mma_bf16_16816(o[2 * np], pl, r[0], r[1]);
            mma_bf16_16816(o[2 * np + 1], pl, r[2], r[3]);
        }
    }
}

// One unit with all 256 threads of the group (named barrier 1).  sk0/sk1 and
// sv0/sv1 are the K and V slabs of the chunk's two pages; after the first
// barrier they are reused as scratch (sk1 and sv1: page-1 outputs of row
// groups 0-1 and 2-3; sk0: their row statistics).
template <int HD>
__device__ __forceinline__ void attn_unit(const AttnParams& a, uint16_t* sk0, uint16_t* sk1, uint16_t* sv0, uint16_t* sv1,
                                          int h, int chunk, int pos0, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    const int half = warp >> 2, rg = warp & 3;
    const int R = a.n * (a.n_heads / a.n_kv_heads);
    const bool active = rg * 16 < R;
    float o[HD / 8][4];
    float msA = -1e30f, lA = 0.f, msB = -1e30f, lB = 0.f;
    if (active)
        attn_rows<HD>(a, half ? sk1 : sk0, half ? sv1 : sv0, h, chunk * kAttnChunk + half * kPageSize, pos0, rg, lane,
                      o, msA, lA, msB, lB);
    named_bar_sync(1, kAttnUnitThreads);  // every slab read is done: slabs become scratch
    const int g = lane >> 2, cc = lane & 3;
    float* obuf = reinterpret_cast<float*>((rg < 2) ? sk1 : sv1) + (rg & 1) * 16 * HD;  // [16][HD]
    float* mlbuf = reinterpret_cast<float*>(sk0) + rg * 16 * 2;                          // [16][2]
    if (half == 1 && active) {
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) {
            *reinterpret_cast<float2*>(obuf + g * HD + t * 8 + 2 * cc) = make_float2(o[t][0], o[t][1]);
            *reinterpret_cast<float2*>(obuf + (g + 8) * HD + t * 8 + 2 * cc) = make_float2(o[t][2], o[t][3]);
        }
        if (cc == 0) {
            mlbuf[g * 2] = msA;
            mlbuf[g * 2 + 1] = lA;
            mlbuf[(g + 8) * 2] = msB;
            mlbuf[(g + 8) * 2 + 1] = lB;
        }
    }
    named_bar_sync(1, kAttnUnitThreads);
    if (half != 0 || !active) return;
    const int rA = rg * 16 + g, rB = rA + 8;
    const float m1A = mlbuf[g * 2], l1A = mlbuf[g * 2 + 1];
    const float m1B = mlbuf[(g + 8) * 2], l1B = mlbuf[(g + 8) * 2 + 1];
    const float MA = fmaxf(msA, m1A), MB = fmaxf(msB, m1B);
    const float a0A = exp2f(msA - MA), a1A = exp2f(m1A - MA);
    const float a0B = exp2f(msB - MB), a1B = exp2f(m1B - MB);
    const size_t base = ((size_t)h * a.nch + chunk) * 64;
    if (rA < R) {
        float* dst = a.part_o + (base + rA) * HD;
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) {
            const float2 p1 = *reinterpret_cast<const float2*>(obuf + g * HD + t * 8 + 2 * cc);
            *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) =
                make_float2(a0A * o[t][0] + a1A * p1.x, a0A * o[t][1] + a1A * p1.y);
        }
        if (cc == 0) a.part_ml[base + rA] = make_float2(MA, a0A * lA + a1A * l1A);
    }
    if (rB < R) {
        float* dst = a.part_o + (base + rB) * HD;
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) {
            const float2 p1 = *reinterpret_cast<const float2*>(obuf + (g + 8) * HD + t * 8 + 2 * cc);
            *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) =
                make_float2(a0B * o[t][2] + a1B * p1.x, a0B * o[t][3] + a1B * p1.y);
        }
        if (cc == 0) a.part_ml[base + rB] = make_float2(MB, a0B * lB + a1B * l1B);
    }
}

// Rows (query head, token) u0, u0+ustep, ...: one warp per row merges the nc
// chunk partials in chunk order and writes the bf16 output into the O
// projection's operand.  Each lane owns HD/32 consecutive dimensions.  The
// first kFirst chunks' partial outputs are loaded together with the chunk
// statistics (their addresses do not depend on them), so a row of up to
// kFirst chunks costs one round trip to L2.  Every lane reads every chunk's
// (max, sum) (uniform loads) and forms the same weights; the sums run in
// chunk order, so a row's result does not depend on the block size.
template <int HD>
__device__ __forceinline__ void comb_rows(const AttnParams& a, int u0, int ustep, int lane, int nc) {
    constexpr int V = HD / 32;   // dimensions per lane: 4 (hd 128) or 2 (hd 64)
    constexpr int kFirst = 24;
    const int G = a.n_heads / a.n_kv_heads;
    const int U = a.n_heads * a.n;
    const size_t cstride = (size_t)64 * HD;
    for (int u = u0; u < U; u += ustep) {
        const int qh = u % a.n_heads, j = u / a.n_heads;
        const int h = qh / G, r = j * G + qh % G;
        const float2* ml = a.part_ml + (size_t)h * a.nch * 64 + r;
        const float* po = a.part_o + ((size_t)h * a.nch * 64 + r) * HD + lane * V;
        float ob[kFirst][V];
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
            }
        }
        float M = -1e30f;
        for (int c0 = 0; c0 < nc; c0 += 8) {   // statistics: eight loads in flight
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
                const float2 st = ml[(size_t)t * 64];
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
