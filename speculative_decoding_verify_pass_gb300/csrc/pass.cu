// Persistent pass kernel: a whole verify / draft / prefill pass of a dense
// model in one cooperative launch.
//
// A pass is a chain of dependent phases (embed; per layer QKV, attention,
// attention merge, O, gate-up, down; LM head; accept).  Launched as separate
// kernels, every phase pays its pipeline fill, its tail and a launch gap, and
// the HBM pipe drains in between.  Here one CTA per SM runs every phase;
// phases are separated by a grid barrier (an arrival counter, bounded waits),
// and all stages of all phases flow through one 11-deep shared-memory ring in
// a fixed order:
//  * GEMM phases contribute their stream-K k-block stages (16 KB of weights
//    plus the activation operand), attention phases contribute the K and V
//    page slabs of their (kv head, 128-position chunk) units;
//  * a weight-producer warp reserves ring slots in that order and streams
//    weights immediately -- weights never depend on an earlier phase, so the
//    next layer's weights are already arriving while the current phase ends;
//  * a dependency-producer warp issues the copies that do depend on earlier
//    phases (activation operands, KV slabs) once the consumer warps have
//    observed the grid barrier in front of their phase;
//  * the 8 consumer warps run the MMA main loop, the fixups and the fused
//    epilogues exactly as the per-kernel path does, plus the attention,
//    merge, embedding and accept work.
// Every wait is bounded; a wait that gives up records an error code and the
// kernel still runs to its end.
#include <math.h>

#include "gemm_core.cuh"

namespace sv {

namespace {

using namespace gemm_core;

constexpr int kPassThreads = kConsumers + 64;  // 8 consumer warps + 2 producer warps
constexpr int kWarpW = kConsumerWarps;
constexpr int kWarpX = kConsumerWarps + 1;

struct __align__(128) PassSmem {
    GemmSmem g;
    GemmParams gp;   // the current GEMM phase (consumers' copy, IO pointers patched)
    int w_issued;    // ring stages whose slot the weight producer has reserved
    int phase_ok;    // phases whose predecessors are all complete
    int am[kMaxBlock];
};

__device__ __forceinline__ int ld_acquire_cta(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_cta(int* p, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ long long globaltimer() {
    long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Bounded wait until *p >= target (p in shared memory, written by another warp).
__device__ __forceinline__ void wait_smem_ge(const int* p, int target, int* err, int site) {
    if (ld_acquire_cta(p) >= target) return;
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (ld_acquire_cta(p) >= target) return;
        if (i > 32) __nanosleep(64);
        if ((i & 1023) == 1023 && *reinterpret_cast<volatile int*>(err) != 0) return;
    }
    atomicCAS(err, 0, site);
}

// Bounded wait until the global arrival counter reaches target.
__device__ __forceinline__ void wait_global_ge(const int* p, int target, int* err, int site) {
    if (ld_acquire_gpu(p) >= target) return;
    for (uint32_t i = 0; i < (1u << 25); ++i) {
        if (ld_acquire_gpu(p) >= target) return;
        if (i > 16) __nanosleep(i < 1024 ? 32 : 128);
        if ((i & 1023) == 1023 && *reinterpret_cast<volatile int*>(err) != 0) return;
    }
    atomicCAS(err, 0, site);
}

// This CTA's ring stages of one phase, in order.
struct PhaseIter {
    int kind;
    StageIter gi;
    int u, U, step, sub;
    bool valid;
    __device__ void init(const PhaseDesc& D, int nc) {
        kind = D.kind;
        valid = false;
        if (kind == PH_GEMM) {
            if ((int)blockIdx.x < D.g.grid) {
                gi.init(D.g, 0);
                valid = gi.valid;
            }
        } else if (kind == PH_ATTN) {
            U = D.a.n_kv_heads * nc;
            u = blockIdx.x;
            step = gridDim.x;
            sub = 0;
            valid = u < U;
        }
    }
    __device__ void advance() {
        if (kind == PH_GEMM) {
            gi.advance();
            valid = gi.valid;
        } else if (++sub == 4) {  // K page 0, K page 1, V page 0, V page 1
            sub = 0;
            u += step;
            valid = u < U;
        }
    }
};

// ------------------------------------------------------------------ phases ---
__device__ void embed_phase(const EmbedParams& e, const int* tokens, int tid) {
    const int tiles = e.d / kTileRows;
    const int j = tid >> 4, rg = tid & 15;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        float ssum = 0.f;
        if (j < e.n) {
            int tok = tokens[j];
            if (tok < 0 || tok >= e.vocab) {
                atomicCAS(&e.st->error, 0, 10);
                tok = 0;
            }
            const int R0 = tile * kTileRows + rg * 8;
            const uint4 raw = *reinterpret_cast<const uint4*>(e.embed + (size_t)tok * e.d + R0);
            const uint16_t* b = reinterpret_cast<const uint16_t*>(&raw);
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                v[q] = bf2f(b[q]);
                ssum += v[q] * v[q];
                const int R = R0 + q;
                *reinterpret_cast<uint16_t*>(e.xf_out + (size_t)(R >> 6) * kStageXBytes + xfrag_offset(j, R & 63)) =
                    f2bf(v[q] * bf2f(e.g_next[R]));
            }
            float* xr = e.x + (size_t)j * e.d + R0;
            *reinterpret_cast<float4*>(xr) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(xr + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
        if (rg == 0 && j < e.n) e.ss_out[j * tiles + tile] = ssum;
    }
}

__device__ void gemm_phase(const GemmParams& gp, PassSmem& sm, int& q, bool& aborted, int tid, int* err,
                           long long* tr) {
    if ((int)blockIdx.x >= gp.grid) return;
    const int warp = tid >> 5, lane = tid & 31;
    StageIter it;
    it.init(gp, 0);
    const bool two = gp.n > 8;
    while (it.valid) {
        const int tile = it.tile, b0 = it.b, b1 = it.b1;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int b = b0; b < b1; ++b, ++q) {
            const int s = q % kStages;
            if (!aborted && !mbar_wait(&sm.g.full[s], (q / kStages) & 1, err, 1)) aborted = true;
            const uint8_t* ws = sm.g.w[s] + warp * 2048 + lane * 16;
            const uint8_t* xs = sm.g.x[s] + lane * 8;
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
            if (lane == 0) mbar_arrive(&sm.g.empty[s]);
        }
        it.valid = it.next_seg();
        if (tr && tid == 0 && !it.valid) tr[3] = globaltimer();
        if (!finish_tile(gp, sm.g, tile, b0, b1, acc0, acc1, tid)) continue;
        epilogue_any(gp.epi, gp, sm.g, tile, 0, tid);
        named_bar_sync(1, kConsumers);
    }
}

// One warp: 16 query rows (row group rg) against the 64 keys of one page slab.
template <int HD>
__device__ __forceinline__ void attn_warp(const AttnParams& a, const uint16_t* sk, const uint16_t* svv, int h,
                                          int page_idx, int pos0, int rg, int lane) {
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
    const int start = page_idx * kPageSize;
    const int limA = rA < R ? pos0 + rA / G : -1;
    const int limB = rB < R ? pos0 + rB / G : -1;
    float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
    for (int n8 = 0; n8 < 8; ++n8)
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
    const float k2 = a.scale_log2;
    const float msA = (mA == -INFINITY) ? -1e30f : mA * k2;
    const float msB = (mB == -INFINITY) ? -1e30f : mB * k2;
    float lA = 0.f, lB = 0.f;
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
    for (int o = 1; o <= 2; o <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, o);
        lB += __shfl_xor_sync(0xffffffffu, lB, o);
    }
    float o[HD / 8][4];
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
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
    const size_t base = ((size_t)h * (2 * a.nch) + page_idx) * 64;
    if (rA < R) {
        float* dst = a.part_o + (base + rA) * HD;
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) = make_float2(o[t][0], o[t][1]);
        if (cc == 0) a.part_ml[base + rA] = make_float2(msA, lA);
    }
    if (rB < R) {
        float* dst = a.part_o + (base + rB) * HD;
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) *reinterpret_cast<float2*>(dst + t * 8 + 2 * cc) = make_float2(o[t][2], o[t][3]);
        if (cc == 0) a.part_ml[base + rB] = make_float2(msB, lB);
    }
}

// Units (kv head, 128-position chunk); warps 0-3 take page 0 and warps 4-7
// page 1 of the chunk, each for 16 of the up to 64 query rows.
__device__ void attn_phase(const AttnParams& a, PassSmem& sm, int& q, bool& aborted, int tid, int nc, int pos0,
                           int* err) {
    const int warp = tid >> 5, lane = tid & 31;
    const int U = a.n_kv_heads * nc;
    const int R = a.n * (a.n_heads / a.n_kv_heads);
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int h = u / nc, c = u % nc;
        for (int t = 0; t < 4; ++t) {
            const int s = (q + t) % kStages;
            if (!aborted && !mbar_wait(&sm.g.full[s], ((q + t) / kStages) & 1, err, 3)) aborted = true;
        }
        const int half = warp >> 2, rg = warp & 3;
        if (rg * 16 < R) {
            const uint16_t* sk = reinterpret_cast<const uint16_t*>(sm.g.w[(q + half) % kStages]);
            const uint16_t* svv = reinterpret_cast<const uint16_t*>(sm.g.w[(q + 2 + half) % kStages]);
            if (a.head_dim == 128)
                attn_warp<128>(a, sk, svv, h, 2 * c + half, pos0, rg, lane);
            else
                attn_warp<64>(a, sk, svv, h, 2 * c + half, pos0, rg, lane);
        }
        __syncwarp();
        if (lane == 0)
            for (int t = 0; t < 4; ++t) mbar_arrive(&sm.g.empty[(q + t) % kStages]);
        q += 4;
    }
}

// One CTA per (query head, token): merge the 64-position page partials in
// page order and write the bf16 output into the O projection's operand.
// Threads split the pages (fixed assignment), partial sums combine in a
// fixed order, so the result is deterministic and independent of n.
__device__ void comb_phase(const AttnParams& a, PassSmem& sm, int tid, int nc) {
    const int G = a.n_heads / a.n_kv_heads;
    const int HD = a.head_dim;
    const int np = 2 * nc, NP = 2 * a.nch;
    const int U = a.n_heads * a.n;
    const int groups = kConsumers / HD;        // page groups: 2 (hd 128) or 4 (hd 64)
    const int dim = tid % HD, grp = tid / HD;
    float* red = sm.g.cs;                      // scratch: [kConsumers] + [groups][HD]
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int qh = u % a.n_heads, j = u / a.n_heads;
        const int h = qh / G, r = j * G + qh % G;
        const float2* ml = a.part_ml + (size_t)h * NP * 64 + r;
        float M = -1e30f;
        for (int pi = tid; pi < np; pi += kConsumers) M = fmaxf(M, ml[(size_t)pi * 64].x);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if ((tid & 31) == 0) red[tid >> 5] = M;
        named_bar_sync(1, kConsumers);
        M = red[0];
        for (int w = 1; w < kConsumerWarps; ++w) M = fmaxf(M, red[w]);
        float L = 0.f;
        for (int pi = tid; pi < np; pi += kConsumers) {
            const float2 v = ml[(size_t)pi * 64];
            L += exp2f(v.x - M) * v.y;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        named_bar_sync(1, kConsumers);
        if ((tid & 31) == 0) red[tid >> 5] = L;
        named_bar_sync(1, kConsumers);
        L = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) L += red[w];
        // this thread: dimension `dim` over pages grp, grp+groups, ...
        const float* po = a.part_o + ((size_t)h * NP * 64 + r) * HD + dim;
        const size_t pstride = (size_t)64 * HD;
        float O = 0.f;
        int pi = grp;
        for (; pi + 7 * groups < np; pi += 8 * groups) {
            float v[8], m8[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                v[t] = po[(size_t)(pi + t * groups) * pstride];
                m8[t] = ml[(size_t)(pi + t * groups) * 64].x;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) O += exp2f(m8[t] - M) * v[t];
        }
        for (; pi < np; pi += groups) O += exp2f(ml[(size_t)pi * 64].x - M) * po[(size_t)pi * pstride];
        named_bar_sync(1, kConsumers);
        red[kConsumers + grp * HD + dim] = O;
        named_bar_sync(1, kConsumers);
        if (grp == 0) {
            float tot = 0.f;
            for (int gg = 0; gg < groups; ++gg) tot += red[kConsumers + gg * HD + dim];
            const int k = qh * HD + dim;
            *reinterpret_cast<uint16_t*>(a.xf_out + (size_t)(k >> 6) * kStageXBytes + xfrag_offset(j, k & 63)) =
                f2bf(tot / L);
        }
        named_bar_sync(1, kConsumers);
    }
}

__device__ void accept_phase(const PassParams& P, PassSmem& sm, int tid, int pos0) {
    const int warp = tid >> 5, lane = tid & 31;
    for (int j = warp; j < P.n; j += kConsumerWarps) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        int t = lane;
        for (; t + 7 * 32 < P.lm_T; t += 8 * 32) {
            float v[8];
            int ix[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                v[u] = P.amax_val[j * P.lm_T + t + u * 32];
                ix[u] = P.amax_idx[j * P.lm_T + t + u * 32];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (v[u] > best || (v[u] == best && ix[u] < bi)) {
                    best = v[u];
                    bi = ix[u];
                }
        }
        for (; t < P.lm_T; t += 32) {
            const float v = P.amax_val[j * P.lm_T + t];
            const int i = P.amax_idx[j * P.lm_T + t];
            if (v > best || (v == best && i < bi)) {
                best = v;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > best || (ov == best && oi < bi)) {
                best = ov;
                bi = oi;
            }
        }
        if (lane == 0) sm.am[j] = bi == 0x7fffffff ? 0 : bi;
    }
    named_bar_sync(1, kConsumers);
    if (tid != 0) return;
    DevState* st = P.st;
    if (P.mode == ACC_VERIFY) {
        int k = 0;
        while (k < P.n - 1 && P.block[k + 1] == sm.am[k]) ++k;
        const int tok_k = P.block[k];
        for (int j = 0; j < P.n; ++j) P.out_argmax[j] = sm.am[j];
        *P.out_accept = k;
        if (P.out_pair) {
            P.out_pair[0] = tok_k;
            P.out_pair[1] = sm.am[k];
        }
        st->verify_pos = pos0;
        st->verify_accept = k;
    } else if (P.out_token) {
        *P.out_token = sm.am[P.n - 1];
    }
    st->len[P.which] = pos0 + P.n;
}

// ------------------------------------------------------------------ kernel ---
__global__ void __launch_bounds__(kPassThreads, 1) pass_kernel(const __grid_constant__ PassParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PassSmem& sm = *reinterpret_cast<PassSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = &P.st->error;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.g.full[s], 1);
            mbar_init(&sm.g.empty[s], kConsumerWarps);
        }
        sm.w_issued = 0;
        sm.phase_ok = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int pos0 = P.st->len[P.which];
    const int nc_need = (pos0 + P.n + kAttnChunk - 1) / kAttnChunk;
    const int nc = nc_need < P.nch ? nc_need : P.nch;  // never index past the allocated pages
    const int G = gridDim.x;

    if (warp == kWarpW) {
        // ---- weight producer: reserves every ring slot in order, streams weights ----
        if (lane == 0) {
            int q = 0;
            bool aborted = false;
            for (int ph = 0; ph < P.nphase; ++ph) {
                const PhaseDesc& D = P.phases[ph];
                PhaseIter it;
                it.init(D, nc);
                const uint32_t xb = P.n > 8 ? (uint32_t)kStageXBytes : (uint32_t)(kStageXBytes / 2);
                const uint32_t slab = (uint32_t)(kPageSize * D.a.head_dim * 2);
                while (it.valid) {
                    const int s = q % kStages;
                    if (q >= kStages && !aborted &&
                        !mbar_wait(&sm.g.empty[s], ((q / kStages) & 1) ^ 1, err, 4))
                        aborted = true;
                    if (D.kind == PH_GEMM) {
                        mbar_arrive_expect_tx(&sm.g.full[s], kStageWBytes + xb);
                        bulk_g2s(sm.g.w[s], D.g.W + ((long long)it.gi.tile * D.g.KBs + it.gi.b) * kStageWBytes,
                                 kStageWBytes, &sm.g.full[s]);
                    } else {
                        mbar_arrive_expect_tx(&sm.g.full[s], slab);
                        const int h = it.u / nc, c = it.u % nc;
                        if ((c + 1) * kAttnChunk <= pos0) {
                            // only previously cached positions: no dependency on this pass
                            const int page = D.a.block_table[2 * c + (it.sub & 1)];
                            const size_t off = ((size_t)(page * D.a.n_kv_heads + h) * kPageSize) * D.a.head_dim;
                            bulk_g2s(sm.g.w[s], (it.sub >= 2 ? D.a.vpool : D.a.kpool) + off, slab, &sm.g.full[s]);
                        }
                    }
                    st_release_cta(&sm.w_issued, q + 1);
                    ++q;
                    it.advance();
                }
            }
        }
        return;
    }
    if (warp == kWarpX) {
        // ---- dependency producer: operands and KV slabs after the phase barrier ----
        if (lane == 0) {
            int q = 0;
            for (int ph = 0; ph < P.nphase; ++ph) {
                const PhaseDesc& D = P.phases[ph];
                PhaseIter it;
                it.init(D, nc);
                if (!it.valid) continue;
                wait_smem_ge(&sm.phase_ok, ph, err, 5);
                fence_proxy_async();
                const uint32_t xb = P.n > 8 ? (uint32_t)kStageXBytes : (uint32_t)(kStageXBytes / 2);
                const int hd = D.a.head_dim;
                const uint32_t slab = (uint32_t)(kPageSize * hd * 2);
                while (it.valid) {
                    wait_smem_ge(&sm.w_issued, q + 1, err, 6);
                    const int s = q % kStages;
                    if (D.kind == PH_GEMM) {
                        bulk_g2s(sm.g.x[s], D.g.X + (long long)it.gi.b * kStageXBytes, xb, &sm.g.full[s]);
                    } else {
                        const int h = it.u / nc, c = it.u % nc;
                        if ((c + 1) * kAttnChunk > pos0) {  // holds this pass's new keys
                            const int page = D.a.block_table[2 * c + (it.sub & 1)];
                            const size_t off = ((size_t)(page * D.a.n_kv_heads + h) * kPageSize) * hd;
                            bulk_g2s(sm.g.w[s], (it.sub >= 2 ? D.a.vpool : D.a.kpool) + off, slab, &sm.g.full[s]);
                        }
                    }
                    ++q;
                    it.advance();
                }
            }
        }
        return;
    }

    // ---------------------------- consumers ----------------------------
    int q = 0;
    bool aborted = false;
    if (pos0 + P.n > P.nch * kAttnChunk && tid == 0) atomicCAS(err, 0, 20);
    for (int ph = 0; ph < P.nphase; ++ph) {
        const PhaseDesc& D = P.phases[ph];
        long long* tr = P.trace ? P.trace + ((size_t)blockIdx.x * P.nphase + ph) * 4 : nullptr;
        if (tr && tid == 0) tr[0] = globaltimer();
        if (ph > 0) {
            if (tid == 0) {
                wait_global_ge(&P.gbar[0], ph * G, err, 7);
                st_release_cta(&sm.phase_ok, ph);
            }
            named_bar_sync(1, kConsumers);
        }
        if (tr && tid == 0) {
            tr[1] = globaltimer();
            tr[3] = 0;
        }
        const int kind = D.kind;
        if (kind == PH_EMBED) {
            embed_phase(D.e, P.tokens, tid);
        } else if (kind == PH_GEMM) {
            // this phase's parameters into shared memory, IO pointers patched
            const int words = (int)(sizeof(GemmParams) / 4);
            const int* srcw = reinterpret_cast<const int*>(&D.g);
            int* dstw = reinterpret_cast<int*>(&sm.gp);
            for (int i = tid; i < words; i += kConsumers) dstw[i] = srcw[i];
            named_bar_sync(1, kConsumers);
            if (tid == 0 && sm.gp.epi == EPI_LMHEAD) sm.gp.logits = P.logits;
            compute_rstd(sm.gp, sm.g, tid);
            gemm_phase(sm.gp, sm, q, aborted, tid, err, tr);
        } else if (kind == PH_ATTN) {
            attn_phase(D.a, sm, q, aborted, tid, nc, pos0, err);
        } else if (kind == PH_COMB) {
            comb_phase(D.a, sm, tid, nc);
        } else if (kind == PH_ACCEPT) {
            if (blockIdx.x == 0) accept_phase(P, sm, tid, pos0);
        } else if (kind == PH_ADVANCE) {
            if (blockIdx.x == 0 && tid == 0) P.st->len[P.which] = pos0 + P.n;
        }
        named_bar_sync(1, kConsumers);
        if (tid == 0) {
            if (tr) tr[2] = globaltimer();  // tr[3]: when the last stage was consumed (0: no stages)
            red_release_add(&P.gbar[0], 1);
        }
    }
    if (tid == 0) {
        const int old = atomicAdd(&P.gbar[1], 1);
        if (old == G - 1) {  // every CTA is past its last wait
            atomicExch(&P.gbar[0], 0);
            atomicExch(&P.gbar[1], 0);
        }
    }
}

}  // namespace

size_t pass_smem_bytes() { return sizeof(PassSmem); }

cudaError_t pass_configure(int device) {
    (void)device;
    return cudaFuncSetAttribute(pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(PassSmem));
}

cudaError_t launch_pass(const PassParams& p, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kPassThreads);
    cfg.dynamicSmemBytes = sizeof(PassSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pass_kernel, p);
}

}  // namespace sv
