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

#include "attn_core.cuh"
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
                gi.init(D.g, 0, false);   // dense phases only
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
                *reinterpret_cast<float*>(e.xf_out + (size_t)(R >> 6) * kStageX32Bytes + xfrag32_offset(j, R & 63)) =
                    v[q] * bf2f(e.g_next[R]);
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
    it.init(gp, 0, false);
    const bool two = gp.n > 8;
    const bool f32 = gp.x_f32 != 0;
    const float ra0 = sm.g.rstd_op[lane >> 2], ra1 = sm.g.rstd_op[8 + (lane >> 2)];
    while (it.valid) {
        const int tile = it.tile, b0 = it.b, b1 = it.b1;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int b = b0; b < b1; ++b, ++q) {
            const int s = q % kStages;
            if (!aborted && !mbar_wait(&sm.g.full[s], (q / kStages) & 1, err, 1)) aborted = true;
            mma_stage(sm.g, s, warp, lane, two, f32, ra0, ra1, acc0, acc1);
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

// Units (kv head, 128-position chunk) over the ring's four slabs (K and V of
// the chunk's two pages); see attn_core::attn_unit.
__device__ void attn_phase(const AttnParams& a, PassSmem& sm, int& q, bool& aborted, int tid, int nc, int pos0,
                           int* err) {
    const int lane = tid & 31;
    const int U = a.n_kv_heads * nc;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int h = u / nc, c = u % nc;
        for (int t = 0; t < 4; ++t) {
            const int s = (q + t) % kStages;
            if (!aborted && !mbar_wait(&sm.g.full[s], ((q + t) / kStages) & 1, err, 3)) aborted = true;
        }
        uint16_t* k0 = reinterpret_cast<uint16_t*>(sm.g.w[q % kStages]);
        uint16_t* k1 = reinterpret_cast<uint16_t*>(sm.g.w[(q + 1) % kStages]);
        uint16_t* v0 = reinterpret_cast<uint16_t*>(sm.g.w[(q + 2) % kStages]);
        uint16_t* v1 = reinterpret_cast<uint16_t*>(sm.g.w[(q + 3) % kStages]);
        static_assert(attn_core::kAttnSlotBytes <= (int)sizeof(sm.g.cs), "attention scratch must fit the tile buffer");
        auto ready = [] {};   // the slab stages were waited for above
        if (a.head_dim == 128)
            attn_core::attn_unit_c<128, 8>(a, k0, k1, v0, v1, sm.g.cs, nullptr, h, c, pos0, a.n, 0, tid, ready);
        else
            attn_core::attn_unit_c<64, 8>(a, k0, k1, v0, v1, sm.g.cs, nullptr, h, c, pos0, a.n, 0, tid, ready);
        __syncwarp();
        if (lane == 0)
            for (int t = 0; t < 4; ++t) mbar_arrive(&sm.g.empty[(q + t) % kStages]);
        q += 4;
    }
}

__device__ void comb_phase(const AttnParams& a, PassSmem& sm, int tid, int nc) {
    (void)sm;
    const int w0 = blockIdx.x * kConsumerWarps + (tid >> 5), ws = gridDim.x * kConsumerWarps;
    if (a.head_dim == 128)
        attn_core::comb_rows<128>(a, w0, ws, tid & 31, nc);
    else
        attn_core::comb_rows<64>(a, w0, ws, tid & 31, nc);
}

__device__ void accept_phase(const PassParams& P, PassSmem& sm, int tid, int pos0) {
    const int warp = tid >> 5, lane = tid & 31;
    for (int j = warp; j < P.n; j += kConsumerWarps) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int t0 = lane; t0 < P.lm_T; t0 += 8 * 32) {  // predicated batches: eight loads in flight per lane
            float v[8];
            int ix[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u * 32;
                v[u] = t < P.lm_T ? P.amax_val[j * P.lm_T + t] : -INFINITY;
                ix[u] = t < P.lm_T ? P.amax_idx[j * P.lm_T + t] : 0x7fffffff;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (v[u] > best || (v[u] == best && ix[u] < bi)) {
                    best = v[u];
                    bi = ix[u];
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
                const uint32_t xb = x_stage_bytes(P.n, D.g.x_f32);
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
                const uint32_t xb = x_stage_bytes(P.n, D.g.x_f32);
                const long long xstride = x_kblock_stride(D.g.x_f32);
                const int hd = D.a.head_dim;
                const uint32_t slab = (uint32_t)(kPageSize * hd * 2);
                while (it.valid) {
                    wait_smem_ge(&sm.w_issued, q + 1, err, 6);
                    const int s = q % kStages;
                    if (D.kind == PH_GEMM) {
                        bulk_g2s(sm.g.x[s], D.g.X + (long long)it.gi.b * xstride, xb, &sm.g.full[s]);
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
            if (tid == 0) sm.g.pos0 = pos0;
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
