// Core of the weight-streaming GEMM (gemm.cu): stage ring layout, stream-K /
// work-item iterators, expert work lists and the fused epilogues.
#pragma once

#include <math.h>

#include "internal.h"

namespace sv {
namespace gemm_core {

constexpr int kStages = 10;  // 160 KB of weights in flight per SM
// Weight stages requested before the dependency wait.  The next kernel's
// weight prefetch overlaps this kernel's tail, whose few L2 round trips
// queue behind it; of 5, 6, 8 and the whole ring of 10, eight was best on
// the Llama-3.1-8B verify (0.8% at every n = 1..16 against ten).
constexpr int kPreStages = 8;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kConverterWarps = 2;   // convert alternate fp32 operand stages
constexpr int kThreads = kConsumers + 64 + 32 * kConverterWarps;  // + producer, MMA issuer, converters
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kIssuerWarp = kConsumerWarps + 1;
constexpr int kConverterWarp0 = kConsumerWarps + 2;
constexpr int kReadGroup = 4;        // stage accumulators a consumer warp reads per wait
constexpr int kAccCols = 16;   // TMEM columns of one stage's accumulator (N = 16 token columns)
constexpr uint32_t kTmemCols = 256;   // power of two >= kStages * kAccCols
constexpr int kCsLd = 20;  // padded row stride of the fp32 tile
constexpr int kMaxItems = kMaxBlock * kMaxTopK + kMaxShared;
constexpr int kPartFloats = kTileRows * kMaxBlock;
constexpr int kMaxContrib = 160;  // CTAs that can share one tile (the host caps the grid at 159 per tile)

struct Item {
    int expert;
    int mask;               // tokens routed to this item
    signed char slot[kMaxBlock];  // slot of the expert in each token's top-k
};

struct __align__(128) GemmSmem {
    uint8_t w[kStages][kStageWBytes];
    uint8_t x[kStages][kStageX32Bytes];
    float cs[kTileRows * kCsLd];
    uint64_t full[kStages];    // weights and operand of the stage have landed (bulk copies)
    uint64_t ready[kStages];   // fp32 operand stage converted to bf16 in place (normalised operands)
    uint64_t mdone[kStages];   // the stage's MMAs completed: its shared memory is free, its accumulator readable
    uint64_t tfree[kStages];   // every consumer warp has read the stage's accumulator
    uint64_t empty[kStages];   // mma.sync path: every consumer warp is done with the stage
    uint32_t tmem_base;        // TMEM address of the accumulator ring (kStages x kAccCols columns)
    float rstd[kMaxBlock];     // applied in the epilogue (bf16 operands)
    float rstd_op[kMaxBlock];  // applied to fp32 operands before rounding
    int slots[kMaxContrib];
    int flag;
    int pos0;                  // cache length at the pass's start (first new position)
    int n_items;
    int emask[kMaxExperts];    // dedup work list: tokens routed to each expert
    int eidx[kMaxExperts];     // and each present expert's item
    unsigned eball[2];         // experts present, by warp of 32
    Item items[kMaxItems];
};

// Iterates the stages of one CTA: stream-K range or strided (item, tile) units.
struct StageIter {
    long long it, end;
    int u, U, step;
    int T, KBs;
    bool items;
    int tile, item, b, b1;
    bool valid;

    __device__ __forceinline__ bool next_seg() {
        if (!items) {
            if (it >= end) return false;
            tile = (int)(it / KBs);
            b = (int)(it % KBs);
            long long rem = end - it;
            b1 = (int)((long long)b + rem < (long long)KBs ? (long long)b + rem : (long long)KBs);
            item = 0;
            it += b1 - b;
            return true;
        }
        if (u >= U) return false;
        item = u / T;
        tile = u % T;
        b = 0;
        b1 = KBs;
        u += step;
        return true;
    }
    // items: the launch walks (item, tile) units (expert kinds; the callers
    // pass a compile-time constant so dense kernels carry no item code)
    __device__ __forceinline__ void init(const GemmParams& p, int n_items, bool items_mode) {
        T = p.T;
        KBs = p.KBs;
        items = items_mode;
        if (!items) {
            long long I = (long long)p.T * p.KBs;
            it = (long long)blockIdx.x * I / p.grid;
            end = (long long)(blockIdx.x + 1) * I / p.grid;
        } else {
            // k = ceil(U / grid) units per CTA, on the fewest CTAs that hold
            // them at k each: no CTA runs a second round alone while others
            // idle (176 units on 152 CTAs: 88 CTAs take 2 each)
            U = n_items * p.T;
            const int per = (U + p.grid - 1) / p.grid;
            const int active = per ? (U + per - 1) / per : 0;
            step = active;
            u = (int)blockIdx.x < active ? (int)blockIdx.x : U;
        }
        valid = next_seg();
    }
    __device__ __forceinline__ void advance() {
        if (++b >= b1) valid = next_seg();
    }
};

// The expert work list of one launch, built by all `nthreads` threads of the
// CTA (call before any role split; contains CTA barriers).  Per slot: item
// j*k + s is token j's s-th expert.  Dedup: one item per distinct expert in
// ascending id, with the tokens that route to it and their slots.  In both
// modes the shared experts follow as one item each (expert n_experts + t,
// every token, output slot k + t), read once per launch.
__device__ __forceinline__ void add_shared_items(const GemmParams& p, GemmSmem& sm, int first) {
    for (int t = 0; t < p.n_shared; ++t) {
        Item& it = sm.items[first + t];
        it.expert = p.n_experts + t;
        it.mask = (1 << p.n) - 1;
        for (int j = 0; j < kMaxBlock; ++j) it.slot[j] = j < p.n ? (signed char)(p.top_k + t) : (signed char)-1;
    }
}

__device__ __forceinline__ void build_items(const GemmParams& p, GemmSmem& sm, int tid, int nthreads) {
    const int n = p.n, k = p.top_k, nk = n * k;
    int* ids = sm.slots;                  // the block's routing, [n][k] (<= 96 entries)
    for (int i = tid; i < nk; i += nthreads) ids[i] = p.route_ids[i];
    __syncthreads();
    if (p.moe_mode == 0) {
        for (int i = tid; i < nk; i += nthreads) {
            const int j = i / k;
            Item& it = sm.items[i];
            it.expert = ids[i];
            it.mask = 1 << j;
            for (int t = 0; t < kMaxBlock; ++t) it.slot[t] = -1;
            it.slot[j] = (signed char)(i % k);
        }
        if (tid == 0) {
            add_shared_items(p, sm, nk);
            sm.n_items = nk + p.n_shared;
        }
        return;
    }
    // dedup, every step one pass of independent threads: the tokens routed
    // to each expert (shared-memory ORs), each present expert's place in
    // ascending id (a ballot over the 64 experts), then each (token, rank)'s slot
    for (int e = tid; e < kMaxExperts; e += nthreads) sm.emask[e] = 0;
    __syncthreads();
    for (int i = tid; i < nk; i += nthreads) atomicOr(&sm.emask[ids[i] & 63], 1 << (i / k));
    __syncthreads();
    if (tid < kMaxExperts) {   // kMaxExperts = 64: two warps
        const bool present = sm.emask[tid] != 0;
        const unsigned bal = __ballot_sync(0xffffffffu, present);
        if ((tid & 31) == 0) sm.eball[tid >> 5] = bal;
    }
    __syncthreads();
    if (tid < kMaxExperts && sm.emask[tid] != 0) {
        const int w = tid >> 5;
        const int idx = (w ? __popc(sm.eball[0]) : 0) + __popc(sm.eball[w] & ((1u << (tid & 31)) - 1u));
        sm.eidx[tid] = idx;
        Item& it = sm.items[idx];
        it.expert = tid;
        it.mask = sm.emask[tid];
        for (int t = 0; t < kMaxBlock; ++t) it.slot[t] = -1;
    }
    __syncthreads();
    for (int i = tid; i < nk; i += nthreads) sm.items[sm.eidx[ids[i] & 63]].slot[i / k] = (signed char)(i % k);
    if (tid == 0) {
        const int cnt = __popc(sm.eball[0]) + __popc(sm.eball[1]);
        add_shared_items(p, sm, cnt);
        sm.n_items = cnt + p.n_shared;
    }
}

// Stream-K ownership: CTA owning flattened iteration i, and its range start.
__device__ __forceinline__ int sk_owner(long long i, long long I, int G) { return (int)(((i + 1) * G - 1) / I); }
__device__ __forceinline__ long long sk_start(int c, long long I, int G) { return (long long)c * I / G; }

// ------------------------------------------------------------- epilogues ---
template <int EPI>
__device__ __forceinline__ void epilogue(const GemmParams& p, GemmSmem& sm, int tile, int item, int tid) {
    const float* cs = sm.cs;
    const int warp = tid >> 5, lane = tid & 31;
    if constexpr (EPI == EPI_QKV) {
        const int hd = p.head_dim, half = hd >> 1;
        const int Nq = p.n_heads * hd, Nk = p.n_kv_heads * hd;
        const int pos0 = sm.pos0;
        constexpr int kJobs = 64 * kMaxBlock / kConsumers;  // rotation pairs per thread, at most
        // all global loads (rotation, page) first: one round trip, then the stores
        float2 cn[kJobs];
        int page[kJobs], posj[kJobs];
#pragma unroll
        for (int u = 0; u < kJobs; ++u) {
            const int job = tid + u * kConsumers;
            cn[u] = make_float2(1.f, 0.f);
            page[u] = 0;
            posj[u] = 0;
            if (job >= 64 * p.n) continue;
            const int j = job >> 6, pr = job & 63;
            const int hl = pr / half, i = pr - hl * half;
            const int R = (tile + p.tile0) * kTileRows + hl * hd + i;
            // batched sequences: this row's own sequence, position and page range
            int pos = pos0 + j, pg0 = 0;
            if (p.seq_len) {
                const int sq = j / p.rows_per_seq;
                pos = p.seq_len[sq] + (j - sq * p.rows_per_seq);
                pg0 = sq * p.seq_pages;
            }
            posj[u] = pos;
            if (R < p.N && R < Nq + Nk) cn[u] = p.rope[(size_t)pos * half + i];
            if (R < p.N && R >= Nq) page[u] = p.block_table[pg0 + pos / kPageSize];
        }
#pragma unroll
        for (int u = 0; u < kJobs; ++u) {
            const int job = tid + u * kConsumers;
            if (job >= 64 * p.n) continue;
            const int j = job >> 6, pr = job & 63;
            const int hl = pr / half, i = pr - hl * half;
            const int ra = hl * hd + i, rb = ra + half;
            const int R = (tile + p.tile0) * kTileRows + ra;
            if (R >= p.N) continue;
            const float rs = sm.rstd[j];
            float va = cs[ra * kCsLd + j] * rs, vb = cs[rb * kCsLd + j] * rs;
            const int pos = posj[u];
            if (R < Nq + Nk) {
                const float na = va * cn[u].x - vb * cn[u].y;
                const float nb = vb * cn[u].x + va * cn[u].y;
                va = na;
                vb = nb;
            }
            if (R < Nq) {
                uint16_t* q = p.qbuf + (size_t)j * Nq + (R / hd) * hd;
                q[i] = f2bf(va);
                q[i + half] = f2bf(vb);
            } else {
                const bool isk = R < Nq + Nk;
                const int kvh = (R - (isk ? Nq : Nq + Nk)) / hd;
                const int slot = pos % kPageSize;
                uint16_t* base =
                    (isk ? p.kpool : p.vpool) + ((size_t)(page[u] * p.n_kv_heads + kvh) * kPageSize) * hd;
                base[isk ? kv_off_k(slot, i, hd) : kv_off_v(slot, i)] = f2bf(va);
                base[isk ? kv_off_k(slot, i + half, hd) : kv_off_v(slot, i + half)] = f2bf(vb);
            }
        }
    } else if constexpr (EPI == EPI_RESID) {
        const int j = tid >> 4, rg = tid & 15;
        float ssum = 0.f;
        if (j < p.n) {
            const int R0 = tile * kTileRows + rg * 8;
            float* xr = p.x + (size_t)j * p.d + R0;
            // every load first (one round trip), then the stores
            const float4 x0 = *reinterpret_cast<const float4*>(xr);
            const float4 x1 = *reinterpret_cast<const float4*>(xr + 4);
            const uint4 gq = *reinterpret_cast<const uint4*>(p.g_next + R0);   // 8 bf16 gains
            const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
            float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[e] += cs[(rg * 8 + e) * kCsLd + j];
                ssum += v[e] * v[e];
                const int R = R0 + e;
                const float g = __uint_as_float((e & 1) ? (gw[e >> 1] & 0xFFFF0000u) : (gw[e >> 1] << 16));
                *reinterpret_cast<float*>(p.xf_out + (size_t)(R >> 6) * kStageX32Bytes + xfrag32_offset(j, R & 63)) =
                    v[e] * g;
            }
            *reinterpret_cast<float4*>(xr) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(xr + 4) = make_float4(v[4], v[5], v[6], v[7]);
            if (p.tap) {
                float* tr = p.tap + (size_t)j * p.d + R0;
                *reinterpret_cast<float4*>(tr) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(tr + 4) = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
        if (rg == 0 && j < p.n) p.ss_out[j * (p.d / kTileRows) + tile] = ssum;
    } else if constexpr (EPI == EPI_SWIGLU || EPI == EPI_EXPERT_SWIGLU) {
        int mask = (1 << p.n) - 1;
        uint8_t* out = p.xf_out;
        if constexpr (EPI == EPI_EXPERT_SWIGLU) {
            mask = sm.items[item].mask;
            out = p.xe + (size_t)item * p.xe_stride;
        }
        out += (size_t)tile * kStageXBytes;
        const int rows = (EPI == EPI_EXPERT_SWIGLU) ? kMaxBlock : p.n;
        for (int job = tid; job < 64 * rows; job += kConsumers) {
            const int j = job >> 6, i = job & 63;
            float a = 0.f;
            if ((mask >> j) & 1) {
                const float rs = sm.rstd[j];
                const float gt = cs[i * kCsLd + j] * rs;
                const float up = cs[(64 + i) * kCsLd + j] * rs;
                a = gt / (1.f + expf(-gt)) * up;
            }
            *reinterpret_cast<uint16_t*>(out + xfrag_offset(j, i)) = f2bf(a);
        }
    } else if constexpr (EPI == EPI_LMHEAD) {
        const int j = tid >> 4, rg = tid & 15;
        float best = -INFINITY;
        int bidx = 0x7fffffff;
        if (j < p.n) {
            const float rs = sm.rstd[j];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = rg * 8 + e, v = tile * kTileRows + r;
                if (v < p.N) {
                    const float lv = cs[r * kCsLd + j] * rs;
                    if (p.logits) p.logits[(size_t)j * p.N + v] = lv;
                    if (lv > best) {
                        best = lv;
                        bidx = v;
                    }
                }
            }
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
            if (ov > best || (ov == best && oi < bidx)) {
                best = ov;
                bidx = oi;
            }
        }
        if (rg == 0 && j < p.n) {
            p.amax_val[j * p.T + tile] = best;
            p.amax_idx[j * p.T + tile] = bidx;
        }
    } else if constexpr (EPI == EPI_ROUTER) {
        const int E = p.n_experts, K = p.top_k;
        for (int j = warp; j < p.n; j += kConsumerWarps) {
            const float rs = sm.rstd[j];
            const float l0 = lane < E ? cs[lane * kCsLd + j] * rs : -INFINITY;
            const float l1 = lane + 32 < E ? cs[(lane + 32) * kCsLd + j] * rs : -INFINITY;
            float mx = fmaxf(l0, l1);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float p0 = lane < E ? expf(l0 - mx) : 0.f;
            float p1 = lane + 32 < E ? expf(l1 - mx) : 0.f;
            float den = p0 + p1;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            p0 = p0 / den;
            p1 = p1 / den;
            bool t0 = false, t1 = false;
            for (int s = 0; s < K; ++s) {
                int e;
                if (p.forced_ids) {
                    e = p.forced_ids[j * K + s];
                } else {
                    float bv = -1.f;
                    int bi = 0x7fffffff;
                    if (!t0 && lane < E) {
                        bv = p0;
                        bi = lane;
                    }
                    if (!t1 && lane + 32 < E && p1 > bv) {
                        bv = p1;
                        bi = lane + 32;
                    }
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                        if (ov > bv || (ov == bv && oi < bi)) {
                            bv = ov;
                            bi = oi;
                        }
                    }
                    e = bi;
                }
                e = e < 0 ? 0 : (e >= E ? E - 1 : e);
                if (e == lane) t0 = true;
                if (e == lane + 32) t1 = true;
                const float gate = __shfl_sync(0xffffffffu, e < 32 ? p0 : p1, e & 31);
                if (lane == 0) {
                    p.route_ids[j * K + s] = e;
                    p.route_gates[j * K + s] = gate;
                    if (p.debug_ids) p.debug_ids[j * K + s] = e;
                }
            }
        }
    } else if constexpr (EPI == EPI_EXPERT_DOWN) {
        const Item& it = sm.items[item];
        for (int job = tid; job < kTileRows * kMaxBlock; job += kConsumers) {
            const int j = job >> 7, r = job & 127;
            const int R = tile * kTileRows + r;
            if (((it.mask >> j) & 1) && R < p.N)
                p.y_slot[((size_t)j * (p.top_k + p.n_shared) + it.slot[j]) * p.d + R] = cs[r * kCsLd + j];
        }
    } else if constexpr (EPI == EPI_STORE) {
        for (int job = tid; job < kTileRows * p.n; job += kConsumers) {
            const int j = job >> 7, r = job & 127;
            const int R = tile * kTileRows + r;
            if (R < p.N) p.y_store[(size_t)j * p.N + R] = cs[r * kCsLd + j];
        }
    }
    (void)warp;
    (void)lane;
}



// Accumulators of one tile segment -> the shared fp32 tile cs[row][token].
// tcgen05 consumers: thread (warp w, lane l) holds weight row 32*(w%4) + l,
// token columns 8*(w/4) .. +7 (its TMEM lane and columns).
__device__ __forceinline__ void store_acc_tc(GemmSmem& sm, const float (&acc)[8], int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    float* crow = sm.cs + (32 * (warp & 3) + lane) * kCsLd + 8 * (warp >> 2);
    *reinterpret_cast<float4*>(crow) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(crow + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
}
// mma.sync consumers: warp w holds rows 16w..16w+15 in the m16n8 accumulator
// distribution, acc0 for tokens 0..7 and acc1 for tokens 8..15.
__device__ __forceinline__ void store_acc_mma(GemmSmem& sm, const float (&acc0)[4], const float (&acc1)[4], int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    float* cs = sm.cs;
    const int r0 = warp * 16 + g;
    cs[r0 * kCsLd + 2 * c] = acc0[0];
    cs[r0 * kCsLd + 2 * c + 1] = acc0[1];
    cs[(r0 + 8) * kCsLd + 2 * c] = acc0[2];
    cs[(r0 + 8) * kCsLd + 2 * c + 1] = acc0[3];
    cs[r0 * kCsLd + 8 + 2 * c] = acc1[0];
    cs[r0 * kCsLd + 8 + 2 * c + 1] = acc1[1];
    cs[(r0 + 8) * kCsLd + 8 + 2 * c] = acc1[2];
    cs[(r0 + 8) * kCsLd + 8 + 2 * c + 1] = acc1[3];
}

// After the accumulators are in cs: for a tile split between CTAs
// (stream-K), the other contributors publish their partials and the first
// contributor sums all partials in contributor order.  Returns true when
// this CTA holds the complete tile (and must run the epilogue), false
// otherwise.
__device__ __forceinline__ bool finish_tile(const GemmParams& p, GemmSmem& sm, int tile, int b0, int b1, int tid) {
    const long long I = (long long)p.T * p.KBs;
        float* cs = sm.cs;
        named_bar_sync(1, kConsumers);

        if (!p.items_mode && !(b0 == 0 && b1 == p.KBs)) {
            // Split tile.  Contributors cf..cl cover it in k order; the tile is
            // cf's last segment, so cf reduces: every other contributor stores
            // its partial and signals with one release-add (no round trip);
            // cf keeps its own partial in shared memory, waits for the others
            // and sums all partials in contributor order.
            const int cf = sk_owner((long long)tile * p.KBs, I, p.grid);
            const int cl = sk_owner((long long)tile * p.KBs + p.KBs - 1, I, p.grid);
            const int ncontrib = cl - cf + 1;
            const int me = blockIdx.x;
            // partial tile stored as [128 rows][pc cols], pc = 8 (n <= 8) or 16;
            // thread tid owns 8 consecutive floats: row tid*8/pc, cols (tid*8)%pc..+7
            const int pc = p.n > 8 ? 16 : 8;
            const bool owner = tid * 8 < kTileRows * pc;
            const int prow = (tid * 8) / pc, pcol = (tid * 8) % pc;
            if (me != cf) {
                const int myslot = 2 * me + ((sk_start(me, I, p.grid) / p.KBs == tile) ? 0 : 1);
                if (owner) {
                    const float* crow = cs + prow * kCsLd + pcol;
                    float4* dst = reinterpret_cast<float4*>(p.partials + (size_t)myslot * kPartFloats + tid * 8);
                    __stcg(dst, make_float4(crow[0], crow[1], crow[2], crow[3]));
                    __stcg(dst + 1, make_float4(crow[4], crow[5], crow[6], crow[7]));
                }
                named_bar_sync(1, kConsumers);
                if (tid == 0) red_release_add(&p.counters[tile], 1);
                return false;
            }
            if (tid < ncontrib && tid < kMaxContrib) {
                const int cc = cf + tid;
                sm.slots[tid] = 2 * cc + ((sk_start(cc, I, p.grid) / p.KBs == tile) ? 0 : 1);
            }
            if (tid == 0) {
                int* err = &p.st->error;
                uint32_t i = 0;
                while (ld_acquire_gpu_i32(&p.counters[tile]) < ncontrib - 1) {
                    if (++i > 64) __nanosleep(64);
                    if (i > (1u << 25) || ((i & 1023) == 0 && *reinterpret_cast<volatile int*>(err) != 0)) {
                        atomicCAS(err, 0, 8);
                        break;
                    }
                }
                p.counters[tile] = 0;  // every contributor has arrived: ready for the next launch
            }
            named_bar_sync(1, kConsumers);
            if (owner) {
                float* wrow = cs + prow * kCsLd + pcol;
                float4 s0 = make_float4(wrow[0], wrow[1], wrow[2], wrow[3]);   // cf's own partial first
                float4 s1 = make_float4(wrow[4], wrow[5], wrow[6], wrow[7]);
                for (int base = 1; base < ncontrib; base += 8) {  // up to 8 contributors' loads in flight
                    float4 v[8][2];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (base + u < ncontrib) {
                            const int sl = (base + u < kMaxContrib) ? sm.slots[base + u] : 0;
                            const float4* src = reinterpret_cast<const float4*>(p.partials + (size_t)sl * kPartFloats + tid * 8);
                            v[u][0] = __ldcg(src);
                            v[u][1] = __ldcg(src + 1);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (base + u < ncontrib) {
                            s0.x += v[u][0].x; s0.y += v[u][0].y; s0.z += v[u][0].z; s0.w += v[u][0].w;
                            s1.x += v[u][1].x; s1.y += v[u][1].y; s1.z += v[u][1].z; s1.w += v[u][1].w;
                        }
                    }
                }
                wrow[0] = s0.x; wrow[1] = s0.y; wrow[2] = s0.z; wrow[3] = s0.w;
                wrow[4] = s1.x; wrow[5] = s1.y; wrow[6] = s1.z; wrow[7] = s1.w;
            }
            named_bar_sync(1, kConsumers);
        }
        return true;
}

// rstd[j] = rsqrt(sum_t ss_in[j][t] / norm_dim + eps) for the block's rows:
// every partial is loaded in one parallel sweep (one L2 round trip), then
// each row sums its partials from shared memory in tile order.  Uses the
// fp32 tile buffer as scratch, so call it before the tile loop.
__device__ __forceinline__ void compute_rstd(const GemmParams& p, GemmSmem& sm, int tid) {
    const int tiles = p.ss_in_tiles;
    const bool norm = p.norm_dim > 0;
    float* buf = sm.cs;
    if (norm) {
        const int total = p.n * tiles;  // <= 16 * 64 (d <= 8192)
        for (int i = tid; i < total && i < kTileRows * kCsLd; i += kConsumers) buf[i] = p.ss_in[i];
    }
    named_bar_sync(1, kConsumers);
    if (tid < kMaxBlock) {
        float r = 1.f;
        if (norm && tid < p.n) {
            float s = 0.f;
            for (int t = 0; t < tiles; ++t) s += buf[tid * tiles + t];
            r = rsqrtf(s / (float)p.norm_dim + p.norm_eps);
        }
        if (p.x_f32) {
            sm.rstd_op[tid] = r;
            sm.rstd[tid] = 1.f;
        } else {
            sm.rstd_op[tid] = 1.f;
            sm.rstd[tid] = r;
        }
    }
    named_bar_sync(1, kConsumers);
}

// P ring stages at once on the mma.sync path, fragments loaded with
// ldmatrix from the canonical layout (weights and operand alike: a core
// matrix of 8 rows x 16 bytes is one 8x8 b16 matrix).  Warp `warp` owns weight
// rows 16*warp..+15; per k16 step its A fragment is the core matrices (row
// groups 2w, 2w+1) x (k groups 2k16, 2k16+1), its B fragment the token
// group(s) x the same k groups.  The stages' MMA chains are independent, so
// issuing them interleaved hides the tensor-core latency of a single chain;
// each stage's four k16 products start from zero, and the stage sums enter
// the running accumulator in stage order (round-to-nearest adds).
template <int P, bool TWO>
__device__ __forceinline__ void mma_stages(const GemmSmem& sm, const int (&st)[4], int warp, int lane,
                                           float (&run0)[4], float (&run1)[4]) {
    float acc0[P][4], acc1[P][4];
#pragma unroll
    for (int u = 0; u < P; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc0[u][i] = acc1[u][i] = 0.f;
    const int mi = lane >> 3, r = lane & 7;
    // A: matrix mi = (row group 2w + (mi & 1), k group 2k16 + (mi >> 1))
    const int a_off = ((2 * warp + (mi & 1)) * 8 + (mi >> 1)) * 128 + r * 16;
    // B (x4 for two token groups): matrix mi = (token group mi >> 1, k group 2k16 + (mi & 1))
    const int b_off = ((mi >> 1) * 8 + (mi & 1)) * 128 + r * 16;
#pragma unroll
    for (int k16 = 0; k16 < 4; ++k16) {
#pragma unroll
        for (int u = 0; u < P; ++u) {
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(sm.w[st[u]]) + a_off + k16 * 256);
            if constexpr (TWO) {
                uint32_t b[4];
                ldmatrix_x4(b, smem_u32(sm.x[st[u]]) + b_off + k16 * 256);
                mma_bf16_16816(acc0[u], a, b[0], b[1]);
                mma_bf16_16816(acc1[u], a, b[2], b[3]);
            } else {
                uint32_t b[2];
                ldmatrix_x2(b, smem_u32(sm.x[st[u]]) + (b_off & 255) + k16 * 256);
                mma_bf16_16816(acc0[u], a, b[0], b[1]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < P; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            run0[i] += acc0[u][i];
            if constexpr (TWO) run1[i] += acc1[u][i];
        }
}

// Converts one ring stage's fp32 operand (x*gain, xfrag32_offset order) in
// place into the bf16 operand of x*gain*rstd (xfrag_offset order, the layout
// the MMA reads), by one warp: unit u (8 values of one row) moves from bytes
// 32u.. to 16u..; every lane reads all its units before any lane writes
// (__syncwarp orders the reads before the other lanes' writes).  The rounding
// is the normalisation's: fp32 product, then bf16 round-to-nearest-even.
template <bool TWO>
__device__ __forceinline__ void convert_stage(uint8_t* xs, const float* rstd_op, int lane) {
    constexpr int kUnits = TWO ? 4 : 2;   // 64 units (rows 0..7) or 128 (rows 0..15) per stage
    float4 v[kUnits][2];
#pragma unroll
    for (int t = 0; t < kUnits; ++t) {
        const int u = lane + 32 * t;
        v[t][0] = *reinterpret_cast<const float4*>(xs + u * 32);
        v[t][1] = *reinterpret_cast<const float4*>(xs + u * 32 + 16);
    }
    __syncwarp();
#pragma unroll
    for (int t = 0; t < kUnits; ++t) {
        const int u = lane + 32 * t;
        const float r = rstd_op[((u >> 6) << 3) | (u & 7)];
        *reinterpret_cast<uint4*>(xs + u * 16) =
            make_uint4(pack_bf16x2(v[t][0].x * r, v[t][0].y * r), pack_bf16x2(v[t][0].z * r, v[t][0].w * r),
                       pack_bf16x2(v[t][1].x * r, v[t][1].y * r), pack_bf16x2(v[t][1].z * r, v[t][1].w * r));
    }
}

}  // namespace gemm_core
}  // namespace sv
