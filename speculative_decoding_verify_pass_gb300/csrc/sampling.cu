// Sampled verification: the rejection-sampling accept step.
//
// The LayerSkip summary (4.3.2, "Self-Verification") states that with
// sampling, rejection sampling keeps the output distribution exactly the
// full model's.  The rule is the standard one of speculative sampling:
// draft x_{j+1}, drawn from q_j = softmax(draft_logits[j] / T), is accepted
// when u_j * q_j(x) < p_j(x), p_j = softmax(target_logits[j] / T) (the test
// u_j < min(1, p/q) written without the division, evaluated in the log
// domain); at the first rejection the next token is drawn from
// norm(max(0, p_j - q_j)), after a full accept from p_{n-1}.  A draw with the
// uniform u is the smallest index whose running weight sum exceeds u times
// the total (inverse CDF).  The uniforms are inputs.
//
// Four small launches over the vocabulary:
//  1. samp_stats_kernel: per (row, 2048-entry chunk) the maximum of l/T and
//     the sum of exp(l/T - max), for the n target rows and n-1 draft rows;
//  2. samp_decide_kernel: one CTA merges each row's chunk statistics in
//     chunk order and runs the accept tests; it writes accept_len and which
//     row, and how, the next token is drawn from;
//  3. samp_weights_kernel: per chunk, fp64 sums of the draw's weights (the
//     residual max(0, p - q), or p), in a fixed order;
//  4. samp_pick_kernel: one CTA walks the chunk sums in order to the chunk
//     where the running sum passes u * total, then scans that chunk.
#include <math.h>

#include "internal.h"

namespace sv {
namespace {

constexpr int kSampThreads = 256;
constexpr int kSampPer = 8;
constexpr int kSampChunk = kSampThreads * kSampPer;   // vocabulary entries per chunk

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Row r < n: target row r; r >= n: draft row r - n.
__device__ __forceinline__ const float* samp_row(const SampleParams& p, int r) {
    return r < p.n ? p.target + (size_t)r * p.vocab : p.draft + (size_t)(r - p.n) * p.vocab;
}

__global__ void __launch_bounds__(kSampThreads) samp_stats_kernel(const __grid_constant__ SampleParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int c = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const float* row = samp_row(p, r);
    __shared__ float red[kSampThreads / 32];
    float z[kSampPer];
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < kSampPer; ++e) {
        const int v = c * kSampChunk + e * kSampThreads + tid;
        z[e] = v < p.vocab ? row[v] / p.temperature : -INFINITY;
        m = fmaxf(m, z[e]);
    }
    m = warp_max(m);
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    float cm = red[0];
#pragma unroll
    for (int w = 1; w < kSampThreads / 32; ++w) cm = fmaxf(cm, red[w]);
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < kSampPer; ++e) s += z[e] == -INFINITY ? 0.f : expf(z[e] - cm);
    s = warp_sum_f(s);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        float cs = 0.f;
        for (int w = 0; w < kSampThreads / 32; ++w) cs += red[w];
        p.stats[(size_t)r * p.chunks + c] = make_float2(cm, cs);
    }
}

__global__ void __launch_bounds__(64) samp_decide_kernel(const __grid_constant__ SampleParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int rows = 2 * p.n - 1;
    // each row's statistics merged in chunk order: max M, sum S of exp(l/T - M)
    if (tid < rows) {
        const float2* st = p.stats + (size_t)tid * p.chunks;
        float M = -INFINITY;
        for (int c = 0; c < p.chunks; ++c) M = fmaxf(M, st[c].x);
        double S = 0.0;
        for (int c = 0; c < p.chunks; ++c)
            if (st[c].x != -INFINITY) S += (double)st[c].y * exp((double)st[c].x - (double)M);
        p.row_stat[tid] = make_double2((double)M, log(S));   // (max, log of the sum)
    }
    __syncthreads();
    if (tid == 0) {
        int k = p.n - 1, mode = 1;   // mode 1: draw from p of row k; 0: from the residual of row k
        for (int j = 0; j + 1 < p.n; ++j) {
            const int x = p.block[j + 1];
            const double2 ts = p.row_stat[j], ds = p.row_stat[p.n + j];
            const double lp = ((double)p.target[(size_t)j * p.vocab + x] / (double)p.temperature - ts.x) - ts.y;
            const double lq = ((double)p.draft[(size_t)j * p.vocab + x] / (double)p.temperature - ds.x) - ds.y;
            if (!(log(p.uniforms[j]) + lq < lp)) {
                k = j;
                mode = 0;
                break;
            }
        }
        p.decision[0] = k;
        p.decision[1] = mode;
        *p.out_accept = k;
    }
}

// Weight of entry v for the decided draw, as a double: p(v), or max(0, p(v) - q(v)).
__device__ __forceinline__ double samp_weight(const SampleParams& p, int k, int mode, int v) {
    const double2 ts = p.row_stat[k];
    const double pv = exp((double)p.target[(size_t)k * p.vocab + v] / (double)p.temperature - ts.x - ts.y);
    if (mode) return pv;
    const double2 ds = p.row_stat[p.n + k];
    const double qv = exp((double)p.draft[(size_t)k * p.vocab + v] / (double)p.temperature - ds.x - ds.y);
    return pv > qv ? pv - qv : 0.0;
}

__global__ void __launch_bounds__(kSampThreads) samp_weights_kernel(const __grid_constant__ SampleParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int c = blockIdx.x, tid = threadIdx.x;
    const int k = p.decision[0], mode = p.decision[1];
    __shared__ double red[2][kSampThreads / 32];
    double s = 0.0, sp = 0.0;
    for (int e = 0; e < kSampPer; ++e) {   // thread tid owns entries c*chunk + tid*8 .. +7
        const int v = c * kSampChunk + tid * kSampPer + e;
        if (v < p.vocab) {
            s += samp_weight(p, k, mode, v);
            if (!mode) sp += samp_weight(p, k, 1, v);
        }
    }
    s = warp_sum_d(s);
    sp = warp_sum_d(sp);
    if ((tid & 31) == 0) {
        red[0][tid >> 5] = s;
        red[1][tid >> 5] = sp;
    }
    __syncthreads();
    if (tid == 0) {
        double a = 0.0, b = 0.0;
        for (int w = 0; w < kSampThreads / 32; ++w) {
            a += red[0][w];
            b += red[1][w];
        }
        p.chunk_sum[c] = a;
        p.chunk_sum[p.chunks + c] = b;   // p's own sums: the residual's fallback when p == q
    }
}

__global__ void __launch_bounds__(kSampThreads) samp_pick_kernel(const __grid_constant__ SampleParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int k = p.decision[0];
    __shared__ int sc_chunk, sc_mode;
    __shared__ double sc_base, sc_target;
    __shared__ double tsum[kSampThreads];
    if (tid == 0) {
        int mode = p.decision[1];
        double total = 0.0;
        for (int c = 0; c < p.chunks; ++c) total += p.chunk_sum[c];
        const double* sums = p.chunk_sum;
        if (!mode && !(total > 0.0)) {   // p == q: the residual is empty, draw from p
            mode = 1;
            sums = p.chunk_sum + p.chunks;
            total = 0.0;
            for (int c = 0; c < p.chunks; ++c) total += sums[c];
        }
        const double t = p.uniforms[p.n - 1] * total;
        double run = 0.0;
        int c = 0;
        for (; c < p.chunks - 1; ++c) {
            if (run + sums[c] > t) break;
            run += sums[c];
        }
        sc_chunk = c;
        sc_mode = mode;
        sc_base = run;
        sc_target = t;
    }
    __syncthreads();
    const int c = sc_chunk, mode = sc_mode;
    double w[kSampPer];
    double mine = 0.0;
    for (int e = 0; e < kSampPer; ++e) {
        const int v = c * kSampChunk + tid * kSampPer + e;
        w[e] = v < p.vocab ? samp_weight(p, k, mode, v) : 0.0;
        mine += w[e];
    }
    tsum[tid] = mine;
    __syncthreads();
    if (tid == 0) {   // exclusive running sums over the threads, in thread order
        double run = sc_base;
        for (int i = 0; i < kSampThreads; ++i) {
            const double v = tsum[i];
            tsum[i] = run;
            run += v;
        }
    }
    __syncthreads();
    // the first entry whose running sum exceeds the target; the lowest index wins
    __shared__ int found;
    if (tid == 0) found = 0x7fffffff;
    __syncthreads();
    double run = tsum[tid];
    for (int e = 0; e < kSampPer; ++e) {
        run += w[e];
        const int v = c * kSampChunk + tid * kSampPer + e;
        if (run > sc_target && v < p.vocab && w[e] > 0.0) {
            atomicMin(&found, v);
            break;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int tok = found;
        if (tok == 0x7fffffff) {   // rounding left the target past the end: the last entry with weight
            tok = 0;
            for (int v = p.vocab - 1; v >= 0; --v)
                if (samp_weight(p, k, mode, v) > 0.0) {
                    tok = v;
                    break;
                }
        }
        *p.out_token = tok;
    }
}

cudaError_t launch_k(const void* fn, dim3 grid, dim3 block, cudaStream_t s, bool pdl, const SampleParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    SampleParams q = p;
    void* args[] = {&q};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

int sample_chunks(int vocab) { return (vocab + kSampChunk - 1) / kSampChunk; }

cudaError_t launch_sample_accept(const SampleParams& p, cudaStream_t s, bool pdl) {
    cudaError_t e;
    if ((e = launch_k((const void*)samp_stats_kernel, dim3((unsigned)p.chunks, (unsigned)(2 * p.n - 1)),
                      dim3(kSampThreads), s, pdl, p)) != cudaSuccess)
        return e;
    if ((e = launch_k((const void*)samp_decide_kernel, dim3(1), dim3(64), s, pdl, p)) != cudaSuccess) return e;
    if ((e = launch_k((const void*)samp_weights_kernel, dim3((unsigned)p.chunks), dim3(kSampThreads), s, pdl, p)) !=
        cudaSuccess)
        return e;
    return launch_k((const void*)samp_pick_kernel, dim3(1), dim3(kSampThreads), s, pdl, p);
}

}  // namespace sv
