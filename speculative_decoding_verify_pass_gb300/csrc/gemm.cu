// Weight-streaming skinny GEMM for the verify pass: Y[n][N] = X[n][K] . W^T
// with n <= 16 tokens and bf16 weights read exactly once.
//
// The verify pass of speculative decoding (LayerSkip summary 4.3.2; DFlash
// README "Verify") multiplies a block of at most 16 token rows by every weight
// matrix of the model, so each GEMM moves N*K*2 bytes of weights for only
// 2*n*N*K flops: the kernel is bound by HBM bandwidth, and its job is to keep
// enough weight bytes in flight.
//
// Design (one CTA per SM, 8 consumer warps + 1 producer warp):
//  * Weights are repacked once into 16 KB stages (128 rows x 64 k) laid out in
//    mma.m16n8k16 A-fragment order, so a stage is one contiguous 1-D bulk copy
//    (TMA engine, mbarrier completion) and each consumer lane reads its
//    fragment with one 16-byte shared load.
//  * The activation operand (n x 64 per stage, <= 2 KB) is kept by the
//    producing kernel in B-fragment order and bulk-copied next to the weights.
//  * An 8-deep ring of stages keeps 128 KB of weights in flight per SM.  The
//    CTA takes over half of the SM's shared memory on purpose: a persistent
//    grid with a static split must not have two of its CTAs on one SM.
//  * Work split: stream-K over the flattened (tile, k-block) space, each CTA
//    one contiguous range; a tile split between CTAs is summed by the last CTA
//    to arrive, in fixed contributor order (deterministic, and independent of
//    n, so row i of a verify pass equals a one-token decode bitwise).  MoE
//    expert GEMMs instead take whole (item, tile) units, so per-slot and
//    deduplicated schedules share every reduction order.
//  * The fused epilogue (RMSNorm scale, RoPE + paged KV append, residual add,
//    SwiGLU, LM-head argmax partials, router softmax/top-k) runs on the
//    finished 128 x 16 fp32 tile in shared memory.
//  * Programmatic dependent launch: the producer issues the first weight
//    stages before waiting on the previous kernel.
#include <math.h>

#include "internal.h"

namespace sv {

namespace {

constexpr int kStages = 8;  // 128 KB of weights in flight per SM
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kCsLd = 20;  // padded row stride of the fp32 tile
constexpr int kMaxItems = kMaxBlock * kMaxTopK;
constexpr int kPartFloats = kTileRows * kMaxBlock;
constexpr int kMaxContrib = 64;  // CTAs that can share one tile (checked on the host)

struct Item {
    int expert;
    int mask;               // tokens routed to this item
    signed char slot[kMaxBlock];  // slot of the expert in each token's top-k
};

struct __align__(128) GemmSmem {
    uint8_t w[kStages][kStageWBytes];
    uint8_t x[kStages][kStageXBytes];
    float cs[kTileRows * kCsLd];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    float rstd[kMaxBlock];
    int slots[kMaxContrib];
    int flag;
    int n_items;
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

    __device__ bool next_seg() {
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
    __device__ void init(const GemmParams& p, int n_items) {
        T = p.T;
        KBs = p.KBs;
        items = p.items_mode != 0;
        if (!items) {
            long long I = (long long)p.T * p.KBs;
            it = (long long)blockIdx.x * I / p.grid;
            end = (long long)(blockIdx.x + 1) * I / p.grid;
        } else {
            u = blockIdx.x;
            U = n_items * p.T;
            step = p.grid;
        }
        valid = next_seg();
    }
    __device__ void advance() {
        if (++b >= b1) valid = next_seg();
    }
};

__device__ __forceinline__ void build_items(const GemmParams& p, GemmSmem& sm) {
    const int n = p.n, k = p.top_k;
    int cnt = 0;
    if (p.moe_mode == 0) {  // per slot: one item per (token, slot)
        for (int j = 0; j < n; ++j)
            for (int s = 0; s < k; ++s) {
                Item& it = sm.items[cnt++];
                it.expert = p.route_ids[j * k + s];
                it.mask = 1 << j;
                for (int t = 0; t < kMaxBlock; ++t) it.slot[t] = -1;
                it.slot[j] = (signed char)s;
            }
    } else {  // dedup: one item per distinct expert, ascending id
        unsigned long long used = 0ull;
        for (int j = 0; j < n; ++j)
            for (int s = 0; s < k; ++s) used |= 1ull << (p.route_ids[j * k + s] & 63);
        for (int e = 0; e < kMaxExperts; ++e) {
            if (!((used >> e) & 1ull)) continue;
            Item& it = sm.items[cnt++];
            it.expert = e;
            it.mask = 0;
            for (int t = 0; t < kMaxBlock; ++t) it.slot[t] = -1;
            for (int j = 0; j < n; ++j)
                for (int s = 0; s < k; ++s)
                    if (p.route_ids[j * k + s] == e) {
                        it.mask |= 1 << j;
                        it.slot[j] = (signed char)s;
                    }
        }
    }
    sm.n_items = cnt;
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
        const int pos0 = p.st->len[p.which];
        for (int job = tid; job < 64 * p.n; job += kConsumers) {
            const int j = job >> 6, pr = job & 63;
            const int hl = pr / half, i = pr - hl * half;
            const int ra = hl * hd + i, rb = ra + half;
            const int R = tile * kTileRows + ra;
            if (R >= p.N) continue;
            const float rs = sm.rstd[j];
            float va = cs[ra * kCsLd + j] * rs, vb = cs[rb * kCsLd + j] * rs;
            const int pos = pos0 + j;
            if (R < Nq + Nk) {
                const float2 cn = p.rope[(size_t)pos * half + i];
                const float na = va * cn.x - vb * cn.y;
                const float nb = vb * cn.x + va * cn.y;
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
                const int page = p.block_table[pos / kPageSize], slot = pos % kPageSize;
                uint16_t* base = (isk ? p.kpool : p.vpool) + ((size_t)(page * p.n_kv_heads + kvh) * kPageSize) * hd;
                base[kv_swz(slot, i, hd)] = f2bf(va);
                base[kv_swz(slot, i + half, hd)] = f2bf(vb);
            }
        }
    } else if constexpr (EPI == EPI_RESID) {
        const int j = tid >> 4, rg = tid & 15;
        float ssum = 0.f;
        if (j < p.n) {
            const int R0 = tile * kTileRows + rg * 8;
            float* xr = p.x + (size_t)j * p.d + R0;
            float4 x0 = *reinterpret_cast<float4*>(xr);
            float4 x1 = *reinterpret_cast<float4*>(xr + 4);
            float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[e] += cs[(rg * 8 + e) * kCsLd + j];
                ssum += v[e] * v[e];
                const int R = R0 + e;
                *reinterpret_cast<uint16_t*>(p.xf_out + (size_t)(R >> 6) * kStageXBytes + xfrag_offset(j, R & 63)) =
                    f2bf(v[e] * bf2f(p.g_next[R]));
            }
            *reinterpret_cast<float4*>(xr) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(xr + 4) = make_float4(v[4], v[5], v[6], v[7]);
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
                p.y_slot[((size_t)j * p.top_k + it.slot[j]) * p.d + R] = cs[r * kCsLd + j];
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

// --------------------------------------------------------------- kernel ---
template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = &p.st->error;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (p.items_mode) {  // the work list depends on the router's output
        pdl_wait();
        if (tid == 0) build_items(p, sm);
        __syncthreads();
    }
    const int n_items = p.items_mode ? sm.n_items : 0;
    const uint32_t xb = p.n > 8 ? (uint32_t)kStageXBytes : (uint32_t)(kStageXBytes / 2);

    if (warp == kConsumerWarps) {
        // ---------------- producer: one lane issues every bulk copy ----------------
        if (lane == 0) {
            StageIter it;
            it.init(p, n_items);
            int q = 0;
            bool aborted = false;
            auto w_src = [&](const StageIter& s) {
                const long long e = p.items_mode ? (long long)sm.items[s.item].expert : 0ll;
                return p.W + e * p.w_item_stride + ((long long)s.tile * p.KBs + s.b) * kStageWBytes;
            };
            auto x_src = [&](const StageIter& s) {
                return p.X + (long long)s.item * p.x_item_stride + (long long)s.b * kStageXBytes;
            };
            if (!p.items_mode) {
                // weights do not depend on the previous kernel: start streaming them now
                int pre = 0;
                int pre_b[kStages];
                while (it.valid && pre < kStages) {
                    mbar_arrive_expect_tx(&sm.full[pre], kStageWBytes + xb);
                    bulk_g2s(sm.w[pre], w_src(it), kStageWBytes, &sm.full[pre]);
                    pre_b[pre] = it.b;
                    ++pre;
                    it.advance();
                }
                pdl_wait();
                for (int i = 0; i < pre; ++i)
                    bulk_g2s(sm.x[i], p.X + (long long)pre_b[i] * kStageXBytes, xb, &sm.full[i]);
                q = pre;
            }
            while (it.valid) {
                const int s = q % kStages;
                if (q >= kStages && !aborted) {
                    if (!mbar_wait(&sm.empty[s], ((q / kStages) & 1) ^ 1, err, 2)) aborted = true;
                }
                mbar_arrive_expect_tx(&sm.full[s], kStageWBytes + xb);
                bulk_g2s(sm.w[s], w_src(it), kStageWBytes, &sm.full[s]);
                bulk_g2s(sm.x[s], x_src(it), xb, &sm.full[s]);
                ++q;
                it.advance();
            }
        }
        return;
    }

    // -------------------- consumers: 8 warps, 16 weight rows each --------------------
    if (!p.items_mode) pdl_wait();
    if (tid < kMaxBlock) {
        float r = 1.f;
        if (p.norm_dim > 0 && tid < p.n) {
            float s = 0.f;
            for (int t = 0; t < p.ss_in_tiles; ++t) s += p.ss_in[tid * p.ss_in_tiles + t];
            r = rsqrtf(s / (float)p.norm_dim + p.norm_eps);
        }
        sm.rstd[tid] = r;
    }
    named_bar_sync(1, kConsumers);

    StageIter it;
    it.init(p, n_items);
    const bool two = p.n > 8;
    const int g = lane >> 2, c = lane & 3;
    int q = 0;
    bool aborted = false;
    const long long I = (long long)p.T * p.KBs;

    while (it.valid) {
        const int tile = it.tile, item = it.item, b0 = it.b, b1 = it.b1;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int b = b0; b < b1; ++b, ++q) {
            const int s = q % kStages;
            if (!aborted && !mbar_wait(&sm.full[s], (q / kStages) & 1, err, 1)) aborted = true;
            const uint8_t* ws = sm.w[s] + warp * 2048 + lane * 16;
            const uint8_t* xs = sm.x[s] + lane * 8;
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16) {
                const uint4 a4 = *reinterpret_cast<const uint4*>(ws + k16 * 512);
                const uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w};
                const uint2 bv = *reinterpret_cast<const uint2*>(xs + k16 * 256);
                mma_bf16_16816(acc0, a, bv.x, bv.y);
                if (two) {
                    const uint2 bw = *reinterpret_cast<const uint2*>(xs + 1024 + k16 * 256);
                    mma_bf16_16816(acc1, a, bw.x, bw.y);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        // the segment of the CTA's range that lies in this tile is done
        it.valid = it.next_seg();

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
        named_bar_sync(1, kConsumers);

        if (!p.items_mode && !(b0 == 0 && b1 == p.KBs)) {
            // split tile: publish the partial; the last contributor to arrive
            // sums all partials in contributor order
            const int cf = sk_owner((long long)tile * p.KBs, I, p.grid);
            const int cl = sk_owner((long long)tile * p.KBs + p.KBs - 1, I, p.grid);
            const int ncontrib = cl - cf + 1;
            const int me = blockIdx.x;
            const int myslot = 2 * me + ((sk_start(me, I, p.grid) / p.KBs == tile) ? 0 : 1);
            // thread tid owns partial elements [tid*8, tid*8+8): row tid/2, cols (tid&1)*8..+7
            const float* crow = cs + (tid >> 1) * kCsLd + (tid & 1) * 8;
            float4* dst = reinterpret_cast<float4*>(p.partials + (size_t)myslot * kPartFloats) + tid * 2;
            __stcg(dst, make_float4(crow[0], crow[1], crow[2], crow[3]));
            __stcg(dst + 1, make_float4(crow[4], crow[5], crow[6], crow[7]));
            if (tid < ncontrib && tid < kMaxContrib) {
                const int cc = cf + tid;
                sm.slots[tid] = 2 * cc + ((sk_start(cc, I, p.grid) / p.KBs == tile) ? 0 : 1);
            }
            __threadfence();
            named_bar_sync(1, kConsumers);
            if (tid == 0) {
                const int old = atomicAdd(&p.counters[tile], 1);
                sm.flag = (old == cl - cf) ? 1 : 0;
            }
            named_bar_sync(1, kConsumers);
            if (!sm.flag) continue;
            __threadfence();
            float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
            for (int base = 0; base < ncontrib; base += 4) {
                float4 v[4][2];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (base + u < ncontrib) {
                        const int sl = (base + u < kMaxContrib) ? sm.slots[base + u] : 0;
                        const float4* src = reinterpret_cast<const float4*>(p.partials + (size_t)sl * kPartFloats) + tid * 2;
                        v[u][0] = __ldcg(src);
                        v[u][1] = __ldcg(src + 1);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (base + u < ncontrib) {
                        s0.x += v[u][0].x; s0.y += v[u][0].y; s0.z += v[u][0].z; s0.w += v[u][0].w;
                        s1.x += v[u][1].x; s1.y += v[u][1].y; s1.z += v[u][1].z; s1.w += v[u][1].w;
                    }
                }
            }
            float* wrow = cs + (tid >> 1) * kCsLd + (tid & 1) * 8;
            wrow[0] = s0.x; wrow[1] = s0.y; wrow[2] = s0.z; wrow[3] = s0.w;
            wrow[4] = s1.x; wrow[5] = s1.y; wrow[6] = s1.z; wrow[7] = s1.w;
            if (tid == 0) p.counters[tile] = 0;
            named_bar_sync(1, kConsumers);
        }
        epilogue<EPI>(p, sm, tile, item, tid);
        named_bar_sync(1, kConsumers);
    }
}

template <int EPI>
cudaError_t launch_one(const GemmParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(GemmSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<EPI>, p);
}

template <int EPI>
cudaError_t configure_one() {
    return cudaFuncSetAttribute(gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(GemmSmem));
}

}  // namespace

int gemm_threads() { return kThreads; }
size_t gemm_smem_bytes() { return sizeof(GemmSmem); }

cudaError_t gemm_configure(int device) {
    (void)device;
    cudaError_t e;
    if ((e = configure_one<EPI_QKV>()) != cudaSuccess) return e;
    if ((e = configure_one<EPI_RESID>()) != cudaSuccess) return e;
    if ((e = configure_one<EPI_SWIGLU>()) != cudaSuccess) return e;
    if ((e = configure_one<EPI_LMHEAD>()) != cudaSuccess) return e;
    if ((e = configure_one<EPI_ROUTER>()) != cudaSuccess) return e;
    if ((e = configure_one<EPI_EXPERT_SWIGLU>()) != cudaSuccess) return e;
    if ((e = configure_one<EPI_EXPERT_DOWN>()) != cudaSuccess) return e;
    return configure_one<EPI_STORE>();
}

cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s, bool pdl) {
    switch (p.epi) {
        case EPI_QKV: return launch_one<EPI_QKV>(p, s, pdl);
        case EPI_RESID: return launch_one<EPI_RESID>(p, s, pdl);
        case EPI_SWIGLU: return launch_one<EPI_SWIGLU>(p, s, pdl);
        case EPI_LMHEAD: return launch_one<EPI_LMHEAD>(p, s, pdl);
        case EPI_ROUTER: return launch_one<EPI_ROUTER>(p, s, pdl);
        case EPI_EXPERT_SWIGLU: return launch_one<EPI_EXPERT_SWIGLU>(p, s, pdl);
        case EPI_EXPERT_DOWN: return launch_one<EPI_EXPERT_DOWN>(p, s, pdl);
        case EPI_STORE: return launch_one<EPI_STORE>(p, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sv
