// Device-side building blocks shared by the verify-pass kernels (sm_103a).
//
// Layout constants, inline-PTX wrappers (mbarrier, bulk async copies, bf16
// tensor-core MMA, programmatic dependent launch) and the device state word
// block that holds the cache lengths so captured passes need no host values.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

// ---------------------------------------------------------------- layout ---
constexpr int kMaxBlock = 16;        // tokens per pass (verify block n <= 16)
constexpr int kTileRows = 128;       // weight rows per streamed tile
constexpr int kKBlock = 64;          // k elements per streamed stage
constexpr int kStageWBytes = kTileRows * kKBlock * 2;   // 16 KB of weights
constexpr int kStageXBytes = kMaxBlock * kKBlock * 2;   // 2 KB of bf16 activations
constexpr int kStageX32Bytes = kMaxBlock * kKBlock * 4; // 4 KB of fp32 activations (normalised operands)
constexpr int kPageSize = 64;        // KV positions per page
constexpr int kAttnChunk = 128;      // positions per attention work item
constexpr int kMaxExperts = 64;
constexpr int kMaxTopK = 8;
constexpr int kMaxShared = 2;       // shared experts per MoE layer

// Device state: cache lengths and the last verify's outcome.  Kernels read
// positions from here, so one launch sequence serves every step.
struct DevState {
    int len[2];          // [target, draft] valid positions
    int verify_pos;      // first position of the last verify block
    int verify_accept;   // its accept_len
    int error;           // nonzero: a bounded wait gave up (code = site)
    int pad[3];
};

// ------------------------------------------------------------ bf16 utils ---
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float bf_round(float f) { return bf2f(f2bf(f)); }

// Byte offset of activation element (row j, k) inside one 64-wide k-block of
// the fragment-ordered operand layout: [n8 tile][k16][lane][b0b1, b2b3].
// This is exactly the order in which mma.m16n8k16's B fragments are read,
// so the streaming GEMM loads each fragment with one 8-byte shared load.
__device__ __forceinline__ int xfrag_offset(int j, int kk) {
    const int n8 = j >> 3, g = j & 7;
    const int k16 = kk >> 4, kin = kk & 15;
    const int half = kin >> 3, c = (kin & 7) >> 1, e = kin & 1;
    const int lane = g * 4 + c;
    return (((n8 * 4 + k16) * 32 + lane) * 8) + half * 4 + e * 2;
}

// fp32 variant for operands that a normalisation scales before rounding:
// [n8 tile][k16][lane][b0, b1, b2, b3 as floats], 16 bytes per lane.
__device__ __forceinline__ int xfrag32_offset(int j, int kk) {
    const int n8 = j >> 3, g = j & 7;
    const int k16 = kk >> 4, kin = kk & 15;
    const int half = kin >> 3, c = (kin & 7) >> 1, e = kin & 1;
    const int lane = g * 4 + c;
    return (((n8 * 4 + k16) * 32 + lane) * 16) + (half * 2 + e) * 4;
}

// Bytes of one operand stage (n rows, bf16 or fp32) and one k-block's stride.
__host__ __device__ __forceinline__ uint32_t x_stage_bytes(int n, int f32) {
    const uint32_t base = n > 8 ? (uint32_t)kStageXBytes : (uint32_t)(kStageXBytes / 2);
    return f32 ? 2 * base : base;
}
__host__ __device__ __forceinline__ long long x_kblock_stride(int f32) {
    return f32 ? (long long)kStageX32Bytes : (long long)kStageXBytes;
}

// Element offset of (key slot, dim) inside one KV page slab [64][hd]: 16-byte
// chunks of a row are XOR-permuted by (slot & 7), so the attention kernel's
// fragment loads from the bulk-copied slab hit distinct shared-memory banks.
__device__ __forceinline__ int kv_swz(int slot, int dim, int hd) {
    return slot * hd + ((((dim >> 3) ^ (slot & 7))) << 3) + (dim & 7);
}

// ----------------------------------------------------------- PTX helpers ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (after recording `site`
// in the device error word) if the phase does not complete within the bound;
// callers then carry on without the data so every thread still reaches the
// kernel's end.  The bound (~2^24 polls with back-off) is far above any
// legitimate wait.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(i < 4096 ? 32 : 256);
        // once any wait of the launch has given up, stop waiting at all
        if ((i & 1023) == 1023 && err && *reinterpret_cast<volatile int*>(err) != 0) return false;
    }
    if (err) atomicCAS(err, 0, site);
    return false;
}

// 1-D bulk async copy global -> shared, completing on an mbarrier (TMA engine).
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Release-ordered reduction at GPU scope (no return value, no round trip):
// every write the CTA made before the preceding CTA barrier is visible to a
// thread that acquires the counter afterwards.
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu_i32(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Asynchronous 16-byte global -> shared copy (completes at cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}


// Programmatic dependent launch: let the next kernel start its prologue, and
// wait for the previous kernel's writes before reading them.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace sv
