// Greedy accept from caller-computed logits, without any device allocation.
//
// Some callers cannot allocate device memory at the point where they need
// the accept decision: code running inside a memory pool that owns the whole
// device, a serving loop under a strict no-allocation rule after warm-up, or
// a host thread that must not call cudaMalloc because it would synchronise
// the device.  This entry point needs nothing from the caller except the
// logits, the verify block and the two outputs: its scratch (per-chunk row
// maxima) lives in a fixed file-scope device array that every GPU loading the
// library holds until process exit.
//
// It performs the same reduction as the accept step of spec_verify_step: the
// argmax of each logit row (lowest id on ties) and the count of leading
// drafts that equal the previous row's argmax.
#include <cuda.h>

#include <mutex>

#include "internal.h"
#include "spec.h"

namespace sv {
namespace {

constexpr int kNaThreads = 256;
constexpr int kNaPerThread = 8;
constexpr int kNaChunk = kNaThreads * kNaPerThread;        // vocab entries per CTA and row
constexpr int kNaMaxChunks = 1024;                          // -> vocab <= 2,097,152
constexpr int kNaMaxVocab = kNaChunk * kNaMaxChunks;

struct NaPartial {
    float val;
    int idx;
};

// 16 rows x 1024 chunks x 8 bytes = 128 KB, shared by every call on a device.
static __device__ __align__(256) NaPartial g_noalloc_scratch[kMaxBlock * kNaMaxChunks];

// Per device: the array's device address and the context it was looked up
// in.  A device reset ends the context; the next call runs in a new one,
// where the module (and the array) may sit at another address, so a changed
// context id triggers a fresh lookup.
struct NaAddr {
    unsigned long long ctx_id;
    void* ptr;
};
std::mutex g_na_mutex;
NaAddr g_na_addr[64] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the calling thread's current context (driver entry points fetched
// through the runtime, so the library needs no link against libcuda); 0 if
// the driver cannot tell, in which case the first address stays in use.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur && get_id && get_cur(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
    return 0;
}

__device__ __forceinline__ void na_better(float& bv, int& bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// Stage 1: CTA (chunk c, row j) -> (max, lowest argmax) of its 2048 logits.
__global__ void __launch_bounds__(kNaThreads) na_chunk_kernel(const float* __restrict__ logits, int n, int vocab,
                                                              int chunks, NaPartial* scratch) {
    const int c = blockIdx.x, j = blockIdx.y, tid = threadIdx.x;
    __shared__ float sv_[kNaThreads / 32];
    __shared__ int si_[kNaThreads / 32];
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const float* row = logits + (size_t)j * vocab;
    const int base = c * kNaChunk;
#pragma unroll
    for (int u = 0; u < kNaPerThread; ++u) {
        const int v = base + u * kNaThreads + tid;
        if (v < vocab) na_better(bv, bi, row[v], v);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        na_better(bv, bi, ov, oi);
    }
    if ((tid & 31) == 0) {
        sv_[tid >> 5] = bv;
        si_[tid >> 5] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kNaThreads / 32; ++w) na_better(bv, bi, sv_[w], si_[w]);
        scratch[j * kNaMaxChunks + c] = NaPartial{bv, bi};
    }
    (void)n;
    (void)chunks;
}

// Stage 2: one warp per row reduces the chunk maxima; thread 0 applies the
// greedy accept rule.
__global__ void __launch_bounds__(512) na_accept_kernel(int n, int chunks, const int* block, int* out_argmax,
                                                        int* out_accept, const NaPartial* scratch) {
    __shared__ int am[kMaxBlock];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < n) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int c = lane; c < chunks; c += 32) {
            const NaPartial q = scratch[warp * kNaMaxChunks + c];
            na_better(bv, bi, q.val, q.idx);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            na_better(bv, bi, ov, oi);
        }
        if (lane == 0) am[warp] = bi == 0x7fffffff ? 0 : bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int k = 0;
        while (k < n - 1 && block[k + 1] == am[k]) ++k;
        for (int j = 0; j < n; ++j) out_argmax[j] = am[j];
        *out_accept = k;
    }
}

}  // namespace
}  // namespace sv

extern "C" spec_status spec_accept_from_logits_noalloc(const float* d_logits, int32_t n, int32_t vocab,
                                                       const int32_t* d_block, int32_t* d_argmax,
                                                       int32_t* d_accept_len, void* cuda_stream) {
    using namespace sv;
    if (!d_logits || !d_block || !d_argmax || !d_accept_len) {
        set_last_error("spec_accept_from_logits_noalloc: null pointer");
        return SPEC_ERR_INVALID_ARG;
    }
    if (n < 1 || n > SPEC_MAX_BLOCK) {
        set_last_error("spec_accept_from_logits_noalloc: n must be in 1..16");
        return SPEC_ERR_INVALID_ARG;
    }
    if (vocab < 1 || vocab > kNaMaxVocab) {
        set_last_error("spec_accept_from_logits_noalloc: vocab must be in 1..2097152 (fixed scratch size)");
        return SPEC_ERR_INVALID_ARG;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        set_last_error("spec_accept_from_logits_noalloc: no current CUDA device");
        return SPEC_ERR_CUDA;
    }
    void* scratch = nullptr;
    {
        // Once per device (and again after a device reset), with that device
        // current: the array's device address (its name in host code only
        // stands in for it).
        std::lock_guard<std::mutex> lock(g_na_mutex);
        const unsigned long long ctx_id = current_context_id();
        if (!g_na_addr[dev].ptr || g_na_addr[dev].ctx_id != ctx_id) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                set_last_error(cudaGetErrorString(e));
                return SPEC_ERR_CUDA;
            }
            g_na_addr[dev] = NaAddr{ctx_id, p};
        }
        scratch = g_na_addr[dev].ptr;
    }
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int chunks = (vocab + kNaChunk - 1) / kNaChunk;
    NaPartial* part = static_cast<NaPartial*>(scratch);
    na_chunk_kernel<<<dim3((unsigned)chunks, (unsigned)n), kNaThreads, 0, s>>>(d_logits, n, vocab, chunks, part);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        na_accept_kernel<<<1, 512, 0, s>>>(n, chunks, d_block, d_argmax, d_accept_len, part);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return SPEC_ERR_CUDA;
    }
    return SPEC_OK;
}
