// Attention building blocks shared by the attention kernels (attention.cu):
// the merge of the chunk-group partials.
//
// The partial kernel leaves, per query row and chunk group (chunk mod S, S
// fixed per model), the row maximum in the log2 domain (-1e30 for a row with
// no visible key), the row sum and the unnormalised output.  The merge
// combines a row's groups in increasing group order; the grouping depends
// only on absolute positions, so a query's result never depends on the block
// size.
#pragma once

#include <math.h>

#include "internal.h"

namespace sv {
namespace attn_core {

constexpr int kAttnCombThreads = 64;   // merge kernel: 2 warps, one merged row each

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
