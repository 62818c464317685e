// Weight-streaming skinny GEMM for the verify pass: Y[n][N] = X[n][K] . W^T
// with n <= 16 tokens and bf16 weights read exactly once.
//
// The verify pass of speculative decoding (LayerSkip summary 4.3.2; DFlash
// README "Verify") multiplies a block of at most 16 token rows by every weight
// matrix of the model, so each GEMM moves N*K*2 bytes of weights for only
// 2*n*N*K flops: the kernel is bound by HBM bandwidth, and its job is to keep
// enough weight bytes in flight.
//
// Design (one CTA per SM, 8 consumer warps + 1 producer warp + 1 converter /
// MMA-issuing warp):
//  * Weights are repacked once into 16 KB stages (128 rows x 64 k) in the
//    tensor core's canonical K-major core-matrix layout, so a stage is one
//    contiguous 1-D bulk copy (TMA engine, mbarrier completion) that the MMA
//    reads in place through a shared-memory matrix descriptor.
//  * The activation operand (n x 64 per stage) is kept by the producing kernel
//    in the same layout and bulk-copied next to the weights: bf16 (<= 2 KB)
//    for plain operands, fp32 x*gain (<= 4 KB) for RMS-normalised ones, which
//    the converter warp scales by rstd and rounds to bf16 in place, once per
//    stage.
//  * One lane of that warp issues the stage's MMAs (tcgen05.mma, M = 128
//    weight rows, N = 16 token columns, four K = 16 steps, fp32 accumulation
//    in tensor memory) into an accumulator of the stage's own, and commits
//    them to the stage's mbarrier: the producer then refills the stage and the
//    consumer warps read the stage sum (tcgen05.ld) and add it to their fp32
//    running sums in stage order.  Every stage sum starts from zero, so a
//    row's result is the same whatever n is, and the rounding of the running
//    sum is round-to-nearest rather than the tensor core's own.
//  * A 10-deep ring of stages keeps 160 KB of weights in flight per SM.  The
//    CTA takes over half of the SM's shared memory on purpose: a persistent
//    grid with a static split must not have two of its CTAs on one SM.
//  * Work split: stream-K over the flattened (tile, k-block) space, each CTA
//    one contiguous range; a tile split between CTAs is summed by its first
//    contributor (for which it is the last segment), in fixed contributor
//    order (deterministic, and independent of n, so row i of a verify pass
//    equals a one-token decode bitwise).  MoE
//    expert GEMMs instead take whole (item, tile) units, so per-slot and
//    deduplicated schedules share every reduction order.
//  * The fused epilogue (RMSNorm scale, RoPE + paged KV append, residual add,
//    SwiGLU, LM-head argmax partials, router softmax/top-k) runs on the
//    finished 128 x 16 fp32 tile in shared memory.
//  * Programmatic dependent launch: the producer issues the first weight
//    stages before waiting on the previous kernel.
#include <math.h>
#include <stdlib.h>

#include "gemm_core.cuh"

namespace sv {

namespace {

using namespace gemm_core;

// --------------------------------------------------------------- kernel ---
// Warp roles: warps 0..7 consume (run the MMAs on the mma.sync path, or read
// the stage accumulators from TMEM on the tcgen05 path; then the fixup and
// the epilogue), warp 8 produces (one lane issues the bulk copies), one lane
// of warp 9 issues the tcgen05 MMAs, warps 10..11 convert alternate fp32
// operand stages.  TWO: n > 8, a second group of 8 token columns (a
// compile-time choice, as the work per stage differs).  TC: the tcgen05 path.

// Registers are capped so that a GEMM CTA (384 threads) and an attention-merge
// CTA (64 threads at up to 184 registers) fit on one SM together: the next
// GEMM's CTAs then take their SMs, and stream their first stages, while the
// merge is still running.
constexpr int kMaxRegs = 136;
constexpr int kGroup = 2;   // mma.sync path: ring stages a consumer warp may take at once

template <int EPI, bool TWO, bool TC>
__global__ void __maxnreg__(kMaxRegs) gemm_kernel(const __grid_constant__ GemmParams p) {
    // work items (expert launches) are a property of the epilogue kind, fixed at
    // compile time: the dense kernels carry none of the item-list code
    constexpr bool kItems = EPI == EPI_EXPERT_SWIGLU || EPI == EPI_EXPERT_DOWN;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = &p.st->error;
    long long* tr = (p.trace && blockIdx.x < kTraceCtas) ? p.trace + (size_t)blockIdx.x * 4 : nullptr;
    if (tr && tid == 0) tr[0] = trace_clock();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.ready[s], 1);
            mbar_init(&sm.mdone[s], 1);
            mbar_init(&sm.tfree[s], kConsumerWarps);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    if (TC && warp == kIssuerWarp) tmem_alloc(&sm.tmem_base, kTmemCols);
    if constexpr (TC) tc_fence_before();
    __syncthreads();
    if constexpr (TC) tc_fence_after();
    const uint32_t tmem = TC ? sm.tmem_base : 0u;

    if constexpr (kItems) {  // the work list depends on the router's output
        pdl_wait();
        pdl_launch_dependents();
        build_items(p, sm, tid, kThreads);
        __syncthreads();
    }
    const int n_items = kItems ? sm.n_items : 0;
    const uint32_t xb = x_stage_bytes(p.n, p.x_f32);
    const long long xstride = x_kblock_stride(p.x_f32);
    // fp32 operands reach the MMAs converted (ready barrier)
    uint64_t* gate = p.x_f32 ? sm.ready : sm.full;

    if (warp >= kConverterWarp0) {
        // ------- converters: fp32 operand stages -> bf16 in place; warp c takes
        // the stages q with q % kConverterWarps == c -------
        if (!p.x_f32) return;
        const int cw = warp - kConverterWarp0;
        named_bar_sync(2, kConsumers + 32 * kConverterWarps);   // the consumers' rstd is in shared memory
        StageIter it;
        it.init(p, n_items, kItems);
        bool aborted = false;
        for (int q = 0; it.valid; ++q, it.advance()) {
            if (q % kConverterWarps != cw) continue;
            const int s = q % kStages;
            const bool ok = aborted || mbar_wait(&sm.full[s], (q / kStages) & 1, err, 4);
            aborted = __any_sync(0xffffffffu, !ok) || aborted;
            if (!aborted) convert_stage<TWO>(sm.x[s], sm.rstd_op, lane);
            if constexpr (TC) fence_proxy_async_smem();   // the MMA reads these writes through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ready[s]);
        }
        return;
    }

    if (warp == kIssuerWarp) {
        if constexpr (!TC) return;
        // ------- MMA issue: one lane issues each stage's four k16 MMAs (M 128
        // weight rows, N 16 token columns) into the stage's own TMEM
        // accumulator, starting from zero, and commits them to mdone[s] -------
        int issued = -1;
        if (lane == 0) {
            StageIter it;
            it.init(p, n_items, kItems);
            bool aborted = false;
            for (int q = 0; it.valid && !aborted; ++q, it.advance()) {
                const int s = q % kStages;
                const uint32_t ph = (q / kStages) & 1;
                if (!mbar_wait(&gate[s], ph, err, 4)) aborted = true;
                if (!aborted && q >= kStages && !mbar_wait(&sm.tfree[s], ph ^ 1, err, 5)) aborted = true;
                if (aborted) break;
                tc_fence_after();
                const uint64_t ad = umma_desc(smem_u32(sm.w[s])), bd = umma_desc(smem_u32(sm.x[s]));
                const uint32_t dt = tmem + (uint32_t)(s * kAccCols);
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16) umma_bf16(dt, ad + 16 * k16, bd + 16 * k16, k16 > 0 ? 1u : 0u);
                umma_commit(&sm.mdone[s]);
                issued = q;
            }
            // the last MMAs complete before TMEM is released
            if (issued >= 0) mbar_wait(&sm.mdone[issued % kStages], (issued / kStages) & 1, err, 6);
        }
        __syncwarp();
        named_bar_sync(3, kConsumers + 32);   // the consumers have read every accumulator
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
        return;
    }

    if (warp == kProducerWarp) {
        // ---------------- producer: one lane issues every bulk copy ----------------
        if (lane == 0) {
            // a slot is free once its previous stage is consumed: the MMAs that
            // read it completed (tcgen05) or every consumer warp is done (mma.sync)
            uint64_t* slot_free = TC ? sm.mdone : sm.empty;
            StageIter it;
            it.init(p, n_items, kItems);
            int q = 0;
            bool aborted = false;
            auto w_src = [&](const StageIter& s) {
                const long long e = kItems ? (long long)sm.items[s.item].expert : 0ll;
                return p.W + e * p.w_item_stride + ((long long)s.tile * p.KBs + s.b) * kStageWBytes;
            };
            auto x_src = [&](const StageIter& s) {
                return p.X + (long long)s.item * p.x_item_stride + (long long)s.b * xstride;
            };
            if constexpr (!kItems) {
                // weights do not depend on the previous kernel: start streaming them now
                int pre = 0;
                int pre_b[kPreStages];
                while (it.valid && pre < kPreStages) {
                    mbar_arrive_expect_tx(&sm.full[pre], kStageWBytes + xb);
                    bulk_g2s(sm.w[pre], w_src(it), kStageWBytes, &sm.full[pre]);
                    pre_b[pre] = it.b;
                    ++pre;
                    it.advance();
                }
                pdl_wait();
                pdl_launch_dependents();
                for (int i = 0; i < pre; ++i)
                    bulk_g2s(sm.x[i], p.X + (long long)pre_b[i] * xstride, xb, &sm.full[i]);
                q = pre;
            }
            while (it.valid) {
                const int s = q % kStages;
                if (q >= kStages && !aborted) {
                    if (!mbar_wait(&slot_free[s], ((q / kStages) & 1) ^ 1, err, 2)) aborted = true;
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

    // -------------------- consumers: 8 warps --------------------
    // the cache length is not written by the preceding kernel (trigger rule)
    if constexpr (EPI == EPI_QKV) {
        if (tid == 0) sm.pos0 = p.st->len[p.which];   // published by compute_rstd's barriers
    }
    if constexpr (!kItems) {
        pdl_wait();
        pdl_launch_dependents();
    }
    compute_rstd(p, sm, tid);
    if (p.x_f32) named_bar_arrive(2, kConsumers + 32 * kConverterWarps);   // release the converters
    if (tr && tid == 0) tr[1] = trace_clock();

    StageIter it;
    it.init(p, n_items, kItems);
    // tcgen05: warp w reads its 32 TMEM lanes, token columns 8*(w/4).. of every
    // stage accumulator; for n <= 8 the warps 4..7 have no columns to read
    const bool reads = TWO || warp < 4;
    const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(8 * (warp >> 2));
    int q = 0;
    bool aborted = false;

    while (it.valid) {
        const int tile = it.tile, item = it.item, b0 = it.b, b1 = it.b1;
        if constexpr (TC) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int b = b0; b < b1;) {
                // up to kReadGroup stages per wait: a commit completes only after
                // every MMA issued before it, so the last stage's barrier covers
                // the earlier ones
                const int g = (b1 - b >= 4) ? 4 : (b1 - b >= 2 ? 2 : 1);
                const int ql = q + g - 1;
                const bool ok = aborted || mbar_wait(&sm.mdone[ql % kStages], (ql / kStages) & 1, err, 1);
                aborted = __any_sync(0xffffffffu, !ok) || aborted;
                tc_fence_after();
                if (reads && !aborted) {
                    // each stage's sum over its 64 k (four k16 MMAs from zero)
                    // enters the running sum with an ordinary round-to-nearest
                    // fp32 add, in stage order, as in a one-token pass
                    if (g == 4) {
                        float v[4][8];
                        tmem_ld8x4(tlane + (uint32_t)((q % kStages) * kAccCols),
                                   tlane + (uint32_t)(((q + 1) % kStages) * kAccCols),
                                   tlane + (uint32_t)(((q + 2) % kStages) * kAccCols),
                                   tlane + (uint32_t)(((q + 3) % kStages) * kAccCols), v);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[i] += v[u][i];
                    } else if (g == 2) {
                        float v[2][8];
                        tmem_ld8x2(tlane + (uint32_t)((q % kStages) * kAccCols),
                                   tlane + (uint32_t)(((q + 1) % kStages) * kAccCols), v);
#pragma unroll
                        for (int u = 0; u < 2; ++u)
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[i] += v[u][i];
                    } else {
                        float v[8];
                        tmem_ld8(tlane + (uint32_t)((q % kStages) * kAccCols), v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] += v[i];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    for (int u = 0; u < g; ++u) mbar_arrive(&sm.tfree[(q + u) % kStages]);
                b += g;
                q += g;
            }
            store_acc_tc(sm, acc, tid);
        } else {
            float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int b = b0; b < b1;) {
                // the next stage, and as many of the following ones (up to
                // kGroup in all) as have already landed
                int st[4];
                st[0] = q % kStages;
                if (!aborted && !mbar_wait(&gate[st[0]], (q / kStages) & 1, err, 1)) aborted = true;
                int m = 1;
                while (m < kGroup && b + m < b1) {
                    const int qq = q + m;
                    if (!aborted && !mbar_test(&gate[qq % kStages], (qq / kStages) & 1)) break;
                    st[m++] = qq % kStages;
                }
                if (m == 2) mma_stages<2, TWO>(sm, st, warp, lane, acc0, acc1);
                else mma_stages<1, TWO>(sm, st, warp, lane, acc0, acc1);
                __syncwarp();
                if (lane == 0)
                    for (int u = 0; u < m; ++u) mbar_arrive(&sm.empty[st[u]]);
                b += m;
                q += m;
            }
            store_acc_mma(sm, acc0, acc1, tid);
        }
        // the segment of the CTA's range that lies in this tile is done
        it.valid = it.next_seg();
        if (tr && tid == 0 && !it.valid) tr[2] = trace_clock();

        if (!finish_tile(p, sm, tile, b0, b1, tid)) continue;
        epilogue<EPI>(p, sm, tile, item, tid);
        named_bar_sync(1, kConsumers);
    }
    if constexpr (TC) {
        tc_fence_before();
        named_bar_arrive(3, kConsumers + 32);   // TMEM may be released
    }
    if (tr && tid == 0) tr[3] = trace_clock();
}

// Which MMA path a launch takes: SPEC_GEMM_TC=1 forces tcgen05 for every
// block size, =0 forces mma.sync; by default blocks of more than kTcMinN
// tokens use tcgen05.  Measured on the Llama-3.1-8B shape at context 4096,
// the tcgen05 pipeline (converter -> issuer -> MMA -> commit -> TMEM read per
// stage) is slower than the mma.sync consumers at every block size up to 16
// (4168 against 3950 us per verify at n = 16), so by default no block takes it.
// Both paths give bitwise the same stage sums, so the choice never changes a
// result.
constexpr int kTcMinN = kMaxBlock;

template <int EPI>
cudaError_t launch_one(const GemmParams& p, cudaStream_t s, bool pdl, int tc_mode) {
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
    const bool tc = tc_mode == 1 || (tc_mode < 0 && p.n > kTcMinN);
    if (p.n > 8) return tc ? cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, true, true>, p)
                           : cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, true, false>, p);
    return tc ? cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, false, true>, p)
              : cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, false, false>, p);
}

template <int EPI>
cudaError_t configure_one() {
    const int bytes = (int)sizeof(GemmSmem);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<EPI, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<EPI, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<EPI, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
        cudaSuccess)
        return e;
    return cudaFuncSetAttribute(gemm_kernel<EPI, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

int g_tc_mode = -1;

}  // namespace

int gemm_threads() { return kThreads; }
size_t gemm_smem_bytes() { return sizeof(GemmSmem); }

cudaError_t gemm_configure(int device) {
    (void)device;
    if (const char* v = std::getenv("SPEC_GEMM_TC")) g_tc_mode = v[0] == '1' ? 1 : (v[0] == '0' ? 0 : -1);
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
        case EPI_QKV: return launch_one<EPI_QKV>(p, s, pdl, g_tc_mode);
        case EPI_RESID: return launch_one<EPI_RESID>(p, s, pdl, g_tc_mode);
        case EPI_SWIGLU: return launch_one<EPI_SWIGLU>(p, s, pdl, g_tc_mode);
        case EPI_LMHEAD: return launch_one<EPI_LMHEAD>(p, s, pdl, g_tc_mode);
        case EPI_ROUTER: return launch_one<EPI_ROUTER>(p, s, pdl, g_tc_mode);
        case EPI_EXPERT_SWIGLU: return launch_one<EPI_EXPERT_SWIGLU>(p, s, pdl, g_tc_mode);
        case EPI_EXPERT_DOWN: return launch_one<EPI_EXPERT_DOWN>(p, s, pdl, g_tc_mode);
        case EPI_STORE: return launch_one<EPI_STORE>(p, s, pdl, g_tc_mode);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sv
