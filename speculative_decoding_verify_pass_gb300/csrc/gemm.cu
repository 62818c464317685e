// Weight-streaming skinny GEMM for the verify pass: Y[n][N] = X[n][K] . W^T
// with n <= 16 tokens and bf16 weights read exactly once.
//
// The verify pass of speculative decoding (LayerSkip summary 4.3.2; DFlash
// README "Verify") multiplies a block of at most 16 token rows by every weight
// matrix of the model, so each GEMM moves N*K*2 bytes of weights for only
// 2*n*N*K flops: the kernel is bound by HBM bandwidth, and its job is to keep
// enough weight bytes in flight.
//
// Design (one CTA per SM, 8 consumer warps + 1 producer warp + 1 operand
// converter warp):
//  * Weights are repacked once into 16 KB stages (128 rows x 64 k) laid out in
//    mma.m16n8k16 A-fragment order, so a stage is one contiguous 1-D bulk copy
//    (TMA engine, mbarrier completion) and each consumer lane reads its
//    fragment with one 16-byte shared load.
//  * The activation operand (n x 64 per stage) is kept by the producing kernel
//    in B-fragment order and bulk-copied next to the weights: bf16 (<= 2 KB)
//    for plain operands, fp32 x*gain (<= 4 KB) for RMS-normalised ones, which
//    the converter warp scales by rstd and rounds to bf16 in place, once per
//    stage, before releasing the stage to the consumers.
//  * A consumer warp takes the next stage together with the one after it when
//    that one has already landed, and runs the two stages' MMA chains
//    interleaved (the arithmetic of each stage is unchanged); the kernel is
//    instantiated separately for one and two n8 token tiles.
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

#include "gemm_core.cuh"

namespace sv {

namespace {

using namespace gemm_core;

constexpr int kGroup = 2;   // ring stages a consumer warp may take at once (4: slower, register cap)

// --------------------------------------------------------------- kernel ---
template <int EPI, bool TWO>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
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
            mbar_init(&sm.empty[s], kConsumerWarps);
            mbar_init(&sm.ready[s], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if constexpr (kItems) {  // the work list depends on the router's output
        pdl_wait();
        pdl_launch_dependents();
        build_items(p, sm, tid, kThreads);
        __syncthreads();
    }
    const int n_items = kItems ? sm.n_items : 0;
    const uint32_t xb = x_stage_bytes(p.n, p.x_f32);
    const long long xstride = x_kblock_stride(p.x_f32);

    if (warp == kConsumerWarps + 1) {
        // ------- converter: fp32 operand stages -> bf16 fragments, once per stage -------
        if (!p.x_f32) return;
        named_bar_sync(2, kConsumers + 32);   // the consumers' rstd is in shared memory
        StageIter it;
        it.init(p, n_items, kItems);
        bool aborted = false;
        for (int q = 0; it.valid; ++q) {
            const int s = q % kStages;
            if (!aborted && !mbar_wait(&sm.full[s], (q / kStages) & 1, err, 4)) aborted = true;
            convert_stage<TWO>(sm.x[s], sm.rstd_op, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ready[s]);
            it.advance();
        }
        return;
    }

    if (warp == kConsumerWarps) {
        // ---------------- producer: one lane issues every bulk copy ----------------
        if (lane == 0) {
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
                int pre_b[kStages];
                while (it.valid && pre < kStages) {
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
    // the cache length is not written by the preceding kernel (trigger rule)
    if constexpr (EPI == EPI_QKV) {
        if (tid == 0) sm.pos0 = p.st->len[p.which];   // published by compute_rstd's barriers
    }
    if constexpr (!kItems) {
        pdl_wait();
        pdl_launch_dependents();
    }
    compute_rstd(p, sm, tid);
    if (p.x_f32) named_bar_arrive(2, kConsumers + 32);   // release the converter
    if (tr && tid == 0) tr[1] = trace_clock();

    StageIter it;
    it.init(p, n_items, kItems);
    // fp32 operands reach the consumers already converted (ready barrier)
    uint64_t* gate = p.x_f32 ? sm.ready : sm.full;
    int q = 0;
    bool aborted = false;

    while (it.valid) {
        const int tile = it.tile, item = it.item, b0 = it.b, b1 = it.b1;
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
            if (kGroup >= 4 && m == 4) mma_stages<4, TWO>(sm, st, warp, lane, acc0, acc1);
            else if (kGroup >= 3 && m == 3) mma_stages<3, TWO>(sm, st, warp, lane, acc0, acc1);
            else if (kGroup >= 2 && m == 2) mma_stages<2, TWO>(sm, st, warp, lane, acc0, acc1);
            else mma_stages<1, TWO>(sm, st, warp, lane, acc0, acc1);
            __syncwarp();
            if (lane == 0)
                for (int u = 0; u < m; ++u) mbar_arrive(&sm.empty[st[u]]);
            b += m;
            q += m;
        }
        // the segment of the CTA's range that lies in this tile is done
        it.valid = it.next_seg();
        if (tr && tid == 0 && !it.valid) tr[2] = trace_clock();

        if (!finish_tile(p, sm, tile, b0, b1, acc0, acc1, tid)) continue;
        epilogue<EPI>(p, sm, tile, item, tid);
        named_bar_sync(1, kConsumers);
    }
    if (tr && tid == 0) tr[3] = trace_clock();
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
    if (p.n > 8) return cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, true>, p);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, false>, p);
}

template <int EPI>
cudaError_t configure_one() {
    const cudaError_t e = cudaFuncSetAttribute(gemm_kernel<EPI, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)sizeof(GemmSmem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_kernel<EPI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(GemmSmem));
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
