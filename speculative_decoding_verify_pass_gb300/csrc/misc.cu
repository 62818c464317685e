// Small kernels around the streaming GEMMs: token embedding, MoE combine,
// argmax reduction + greedy accept, cache-length updates, weight repacking
// and KV-cache import/export.
#include <math.h>

#include "internal.h"

namespace sv {

namespace {

cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Writes row j's 8 values starting at R0 into the residual, the next GEMM's
// operand (x * gain, fp32, xfrag32_offset order; the consumer applies rstd and
// rounds) and returns their sum of squares.
__device__ __forceinline__ float store_residual8(float* xr, const float (&v)[8], int j, int R0, const uint16_t* g_next,
                                                 uint8_t* xf_out) {
    float ssum = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        ssum += v[e] * v[e];
        const int R = R0 + e;
        *reinterpret_cast<float*>(xf_out + (size_t)(R >> 6) * kStageX32Bytes + xfrag32_offset(j, R & 63)) =
            v[e] * bf2f(g_next[R]);
    }
    *reinterpret_cast<float4*>(xr) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(xr + 4) = make_float4(v[4], v[5], v[6], v[7]);
    return ssum;
}

// x[j] = embed[token_j] (bf16 -> fp32); one CTA per 128 columns, 16 threads
// per token each owning 8 columns.
__global__ void __launch_bounds__(256) embed_kernel(const __grid_constant__ EmbedParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int tile = blockIdx.x, tid = threadIdx.x;
    const int j = tid >> 4, rg = tid & 15;
    float ssum = 0.f;
    if (j < p.n) {
        int tok = p.tokens[j];
        if (tok < 0 || tok >= p.vocab) {
            atomicCAS(&p.st->error, 0, 10);
            tok = 0;
        }
        const int R0 = tile * kTileRows + rg * 8;
        const uint4 raw = *reinterpret_cast<const uint4*>(p.embed + (size_t)tok * p.d + R0);
        const uint16_t* b = reinterpret_cast<const uint16_t*>(&raw);
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = bf2f(b[e]);
        ssum = store_residual8(p.x + (size_t)j * p.d + R0, v, j, R0, p.g_next, p.xf_out);
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (rg == 0 && j < p.n) p.ss_out[j * (p.d / kTileRows) + tile] = ssum;
}

// Tapped hidden states -> one fp32 GEMM operand over K = n_in*d: element
// (row j, k = t*d + i) = taps[t][j][i].  One CTA per 128 k, 16 threads per
// row each owning 8 k (which never straddle two taps: d is a multiple of 128).
__global__ void __launch_bounds__(256) concat_taps_kernel(const __grid_constant__ ConcatParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int j = threadIdx.x >> 4, rg = threadIdx.x & 15;
    const int k0 = blockIdx.x * kTileRows + rg * 8;
    const int t = k0 / p.d, i0 = k0 - t * p.d;
    const float* src = p.taps + ((size_t)t * kMaxBlock + j) * p.d + i0;
    const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int k = k0 + e;
        *reinterpret_cast<float*>(p.xf_out + (size_t)(k >> 6) * kStageX32Bytes + xfrag32_offset(j, k & 63)) = v[e];
    }
}

// Rows x[j] (j < n) as the operand of a normalised GEMM: x*gain and the
// sum-of-squares partials, exactly as the embedding kernel writes them.
__global__ void __launch_bounds__(256) rows_operand_kernel(const __grid_constant__ RowsParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int tile = blockIdx.x, tid = threadIdx.x;
    const int j = tid >> 4, rg = tid & 15;
    float ssum = 0.f;
    if (j < p.n) {
        const int R0 = tile * kTileRows + rg * 8;
        float* xr = p.x + (size_t)j * p.d + R0;
        const float4 a = *reinterpret_cast<const float4*>(xr), b = *reinterpret_cast<const float4*>(xr + 4);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        ssum = store_residual8(xr, v, j, R0, p.g_next, p.xf_out);
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (rg == 0 && j < p.n) p.ss_out[j * (p.d / kTileRows) + tile] = ssum;
}

// MoE layer output: x[j] += sum_s gate[j][s] * y_slot[j][s] (routed slots in
// rank order) + y_slot[j][top_k] + y_slot[j][top_k + 1] (shared experts, in
// order), then the next norm's operand and sum-of-squares.
__global__ void __launch_bounds__(256) moe_combine_kernel(const __grid_constant__ CombineParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int tile = blockIdx.x, tid = threadIdx.x;
    const int j = tid >> 4, rg = tid & 15;
    float ssum = 0.f;
    if (j < p.n) {
        const int R0 = tile * kTileRows + rg * 8;
        float* xr = p.x + (size_t)j * p.d + R0;
        // all slot rows at once (independent loads), then the sum in slot order
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int slots = p.top_k + p.n_shared;
        float4 ys[kMaxTopK + kMaxShared][2];
        float gs[kMaxTopK];
#pragma unroll
        for (int s = 0; s < kMaxTopK + kMaxShared; ++s) {
            if (s < slots) {
                const float* src = p.y_slot + ((size_t)j * slots + s) * p.d + R0;
                ys[s][0] = *reinterpret_cast<const float4*>(src);
                ys[s][1] = *reinterpret_cast<const float4*>(src + 4);
            }
            if (s < kMaxTopK && s < p.top_k) gs[s] = p.gates[j * p.top_k + s];
        }
        // routed slots weighted by their gates, then the shared experts' slots
#pragma unroll
        for (int s = 0; s < kMaxTopK + kMaxShared; ++s) {
            if (s < slots) {
                const float a[8] = {ys[s][0].x, ys[s][0].y, ys[s][0].z, ys[s][0].w,
                                    ys[s][1].x, ys[s][1].y, ys[s][1].z, ys[s][1].w};
                if (s < kMaxTopK && s < p.top_k) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] += gs[s < kMaxTopK ? s : 0] * a[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] += a[e];
                }
            }
        }
        const float4 x0 = *reinterpret_cast<const float4*>(xr), x1 = *reinterpret_cast<const float4*>(xr + 4);
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = xv[e] + y[e];
        if (p.tap) {
            float* tr = p.tap + (size_t)j * p.d + R0;
            *reinterpret_cast<float4*>(tr) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(tr + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
        ssum = store_residual8(xr, v, j, R0, p.g_next, p.xf_out);
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (rg == 0 && j < p.n) p.ss_out[j * (p.d / kTileRows) + tile] = ssum;
}

// Per-token argmax over the LM head's tile partials (lowest id on ties), then
// the greedy accept rule and the cache-length bookkeeping.
__global__ void __launch_bounds__(512) accept_kernel(const __grid_constant__ AcceptParams p) {
    __shared__ int am[kMaxBlock];
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < p.n) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int t0 = lane; t0 < p.T; t0 += 8 * 32) {  // predicated batches: eight loads in flight per lane
            float v[8];
            int ix[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u * 32;
                v[u] = t < p.T ? p.amax_val[warp * p.T + t] : -INFINITY;
                ix[u] = t < p.T ? p.amax_idx[warp * p.T + t] : 0x7fffffff;
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
        if (lane == 0) am[warp] = bi == 0x7fffffff ? 0 : bi;
    }
    __syncthreads();
    if (p.mode == ACC_BATCH) {   // one thread per sequence: its rows are s*per .. s*per+per-1
        const int per = p.n / p.nseq, sq = threadIdx.x;
        if (sq >= p.nseq) return;
        const int* blk = p.block + sq * per;
        const int* a = am + sq * per;
        int k = 0;
        while (k < per - 1 && blk[k + 1] == a[k]) ++k;
        for (int j = 0; j < per; ++j) p.out_argmax[sq * per + j] = a[j];
        p.out_accept[sq] = k;
        p.seq_len[sq] += k + 1;   // the accepted drafts and the bonus token's position are kept
        return;
    }
    if (threadIdx.x != 0) return;
    DevState* st = p.st;
    const int pos0 = st->len[p.which];
    if (p.mode == ACC_VERIFY) {
        int k = 0;
        while (k < p.n - 1 && p.block[k + 1] == am[k]) ++k;   // cumulative product of matches
        const int tok_k = p.block[k];
        for (int j = 0; j < p.n; ++j) p.out_argmax[j] = am[j];
        *p.out_accept = k;
        if (p.out_pair) {
            p.out_pair[0] = tok_k;
            p.out_pair[1] = am[k];
        }
        st->verify_pos = pos0;
        st->verify_accept = k;
    } else if (p.out_token) {
        *p.out_token = am[p.n - 1];
    }
    st->len[p.which] = pos0 + p.n;
}

__global__ void advance_kernel(DevState* st, int which, int n) {
    pdl_wait();
    pdl_launch_dependents();
    st->len[which] += n;
}

__global__ void rollback_kernel(DevState* st, int which, int new_len) {
    pdl_wait();
    pdl_launch_dependents();
    if (new_len >= 0) {
        st->len[which] = new_len;
    } else if (which == 0) {
        st->len[0] = st->verify_pos + st->verify_accept + 1;
    } else {
        const int keep = st->verify_pos + st->verify_accept;
        if (keep < st->len[1]) st->len[1] = keep;
    }
}

// Logical row r of the packed matrix -> source element (or zero).
__device__ __forceinline__ uint16_t pack_fetch(const PackSrc& s, int N, int r, int k) {
    if (r >= N) return 0;
    int row = r;
    int first = 0, count = s.nsrc;
    if (s.mode == 1) {  // tile t rows 0..63 = gate rows t*64.., rows 64..127 = up rows t*64..
        const int t = r >> 7, i = r & 127;
        row = t * 64 + (i & 63);
        first = (i < 64) ? 0 : s.nsrc / 2;
        count = s.nsrc / 2;
    }
    for (int q = first; q < first + count; ++q) {
        if (row < s.rows[q]) return s.src[q][(size_t)row * s.cols + k];
        row -= s.rows[q];
    }
    return 0;
}

// One thread per 16-byte chunk (8 consecutive k of one row) of the packed
// layout: a stage is [8-row group (16)][8-k group (8)][row (8)][8 k], the
// tensor core's canonical K-major layout (see xfrag_offset).
__global__ void pack_kernel(PackSrc s, uint8_t* out, int N, int T, int KBs) {
    const long long total = (long long)T * KBs * (kStageWBytes / 16);
    for (long long ch = blockIdx.x * (long long)blockDim.x + threadIdx.x; ch < total;
         ch += (long long)gridDim.x * blockDim.x) {
        const int r8 = (int)(ch & 7), k8 = (int)((ch >> 3) & 7), m8 = (int)((ch >> 6) & 15);
        const long long tb = ch >> 10;
        const int b = (int)(tb % KBs), t = (int)(tb / KBs);
        const int r = t * kTileRows + m8 * 8 + r8;
        const int k0 = b * kKBlock + k8 * 8;
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = pack_fetch(s, N, r, k0 + e);
        *reinterpret_cast<uint4*>(out + ch * 16) = *reinterpret_cast<const uint4*>(v);
    }
}

__global__ void kv_io_kernel(uint16_t* pool, const int* bt, uint16_t* logical, int ctx, int hkv, int hd, int to_pool,
                             int is_v) {
    const long long total = (long long)ctx * hkv * hd;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int dim = (int)(i % hd);
        const int h = (int)((i / hd) % hkv);
        const int pos = (int)(i / ((long long)hd * hkv));
        const int slot = pos % kPageSize;
        const size_t pi = ((size_t)(bt[pos / kPageSize] * hkv + h) * kPageSize) * hd +
                          (is_v ? kv_off_v(slot, dim) : kv_off_k(slot, dim, hd));
        if (to_pool)
            pool[pi] = logical[i];
        else
            logical[i] = pool[pi];
    }
}

}  // namespace

cudaError_t launch_embed(const EmbedParams& p, cudaStream_t s, bool pdl) {
    EmbedParams q = p;
    void* args[] = {&q};
    return launch_ex((const void*)embed_kernel, dim3((unsigned)(p.d / kTileRows)), dim3(256), 0, s, pdl, args);
}

cudaError_t launch_moe_combine(const CombineParams& p, cudaStream_t s, bool pdl) {
    CombineParams q = p;
    void* args[] = {&q};
    return launch_ex((const void*)moe_combine_kernel, dim3((unsigned)(p.d / kTileRows)), dim3(256), 0, s, pdl, args);
}

cudaError_t launch_concat_taps(const ConcatParams& p, cudaStream_t s, bool pdl) {
    ConcatParams q = p;
    void* args[] = {&q};
    return launch_ex((const void*)concat_taps_kernel, dim3((unsigned)(p.n_in * p.d / kTileRows)), dim3(256), 0, s, pdl,
                     args);
}

cudaError_t launch_rows_operand(const RowsParams& p, cudaStream_t s, bool pdl) {
    RowsParams q = p;
    void* args[] = {&q};
    return launch_ex((const void*)rows_operand_kernel, dim3((unsigned)(p.d / kTileRows)), dim3(256), 0, s, pdl, args);
}

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t s, bool pdl) {
    AcceptParams q = p;
    void* args[] = {&q};
    return launch_ex((const void*)accept_kernel, dim3(1), dim3(512), 0, s, pdl, args);
}

cudaError_t launch_advance(DevState* st, int which, int n, cudaStream_t s, bool pdl) {
    void* args[] = {&st, &which, &n};
    return launch_ex((const void*)advance_kernel, dim3(1), dim3(1), 0, s, pdl, args);
}

cudaError_t launch_rollback(DevState* st, int which, int new_len, cudaStream_t s, bool pdl) {
    void* args[] = {&st, &which, &new_len};
    return launch_ex((const void*)rollback_kernel, dim3(1), dim3(1), 0, s, pdl, args);
}

cudaError_t launch_pack(const PackSrc& src, const PackedMat& m, cudaStream_t st) {
    const long long total = (long long)m.T * m.KBs * (kStageWBytes / 16);
    long long blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    pack_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, m.p, m.N, m.T, m.KBs);
    return cudaGetLastError();
}

cudaError_t launch_kv_io(uint16_t* pool, const int* bt, uint16_t* logical, int ctx, int hkv, int hd, bool to_pool,
                         bool is_v, cudaStream_t s) {
    const long long total = (long long)ctx * hkv * hd;
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    kv_io_kernel<<<(unsigned)blocks, 256, 0, s>>>(pool, bt, logical, ctx, hkv, hd, to_pool ? 1 : 0, is_v ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace sv
