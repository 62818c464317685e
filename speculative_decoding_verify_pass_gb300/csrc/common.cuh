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
// a bf16 GEMM operand: the tensor core's canonical K-major layout without
// swizzle, [8-row group][8-k group][row][8 k] -- "core matrices" of 8 rows x
// 16 bytes, 128 bytes each, the next core matrix along k 128 bytes further
// and the next 8-row group 1024 bytes further.  The streaming GEMM's MMA reads
// a stage of this layout straight from shared memory.
__device__ __forceinline__ int xfrag_offset(int j, int kk) {
    return ((((j >> 3) * 8 + (kk >> 3)) * 8 + (j & 7)) * 16) + (kk & 7) * 2;
}

// fp32 variant for operands that a normalisation scales before rounding: the
// same order with 32-byte units (8 floats of one row), so that the GEMM's
// converter turns unit u of 32 bytes into unit u of 16 bytes in place.
__device__ __forceinline__ int xfrag32_offset(int j, int kk) {
    return ((((j >> 3) * 8 + (kk >> 3)) * 8 + (j & 7)) * 32) + (kk & 7) * 4;
}

// Bytes of one operand stage (n rows, bf16 or fp32) and one k-block's stride.
__host__ __device__ __forceinline__ uint32_t x_stage_bytes(int n, int f32) {
    const uint32_t base = n > 8 ? (uint32_t)kStageXBytes : (uint32_t)(kStageXBytes / 2);
    return f32 ? 2 * base : base;
}
__host__ __device__ __forceinline__ long long x_kblock_stride(int f32) {
    return f32 ? (long long)kStageX32Bytes : (long long)kStageXBytes;
}

// Element offsets of (key slot, dim) inside one KV page slab (64 positions of
// one kv head, hd dims), in the tensor core's canonical K-major layout: core
// matrices of 8 rows x 8 bf16 (128 contiguous bytes).  K is the key operand
// of S = Q K^T (rows = positions, k = dims): [8-position group][8-dim
// group][position][8 dims].  V is the value operand of O = P V (rows = dims,
// k = positions): [8-dim group][8-position group][dim][8 positions].  A
// bulk-copied slab is an MMA operand as it lies.
__host__ __device__ __forceinline__ int kv_off_k(int slot, int dim, int hd) {
    return ((((slot >> 3) * (hd >> 3)) + (dim >> 3)) << 6) + ((slot & 7) << 3) + (dim & 7);
}
__host__ __device__ __forceinline__ int kv_off_v(int slot, int dim) {
    return ((((dim >> 3) << 3) + (slot >> 3)) << 6) + ((dim & 7) << 3) + (slot & 7);
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

// ---------------------------------------------------- tcgen05 (sm_100+) ---
// The fifth-generation tensor core: one thread issues an MMA whose operands
// come from shared memory through matrix descriptors and whose fp32
// accumulator lives in tensor memory (TMEM, 128 lanes x 512 columns of 32 bit
// per SM); warps read the accumulator back with tcgen05.ld.

// Allocate `ncols` TMEM columns (a power of two >= 32); the base address is
// written to shared memory.  One whole warp executes it.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Order tcgen05 operations around thread synchronisation (barriers, mbarrier waits).
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make this thread's ordinary shared-memory writes visible to the tensor core
// (the async proxy) before an MMA reads them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, unswizzled operand in the
// layout of xfrag_offset: core matrices 128 bytes apart along k (leading
// byte offset) and 1024 bytes apart per 8-row group (stride byte offset);
// bits 46..48 hold the fixed value 0b001.  Adding 16 advances the start
// address by 256 bytes, one k16 step.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(1024u >> 4) << 32) |
           (1ull << 46);
}

// The same for any core-matrix strides: lbo along k, sbo per 8-row group.
__device__ __forceinline__ uint64_t umma_desc_kmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both
// operands K-major: M (bits 24..28: M >> 4) x N (bits 17..22: N >> 3).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(uint32_t m, uint32_t n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}
constexpr uint32_t kUmmaIdescM128N16 = umma_idesc_bf16(128, 16);

// D[tmem] (+)= A[128 x 16] * B[16 x 16]^T; accumulate = 0 starts from zero.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kUmmaIdescM128N16), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A * B^T under instruction descriptor idesc.
__device__ __forceinline__ void umma_bf16_id(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when every MMA this thread issued so far has
// completed, i.e. its shared-memory operands may be overwritten and its
// accumulator read.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 8 consecutive fp32 columns at each of G TMEM addresses of this warp's 32
// lanes (lane i of the warp reads TMEM lane (warp % 4) * 32 + i), then one
// wait for all G loads.
__device__ __forceinline__ void tmem_ld8x2(uint32_t t0, uint32_t t1, float (&v)[2][8]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(t0), "r"(t1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i >> 3][i & 7] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld8x4(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3, float (&v)[4][8]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t0), "r"(t1), "r"(t2), "r"(t3)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i >> 3][i & 7] = __uint_as_float(r[i]);
}

// 8 consecutive fp32 columns of this warp's 32 TMEM lanes (lane i of the
// warp reads TMEM lane (warp % 4) * 32 + i), waiting for the load.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 4 consecutive fp32 columns of this warp's 32 TMEM lanes, waiting for the
// load; and the matching store.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const float (&v)[4]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
        : "memory");
}

// 2^x by the hardware's approximate base-2 exponential (one instruction;
// results below the smallest normal flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sum of v over the 32 lanes of a warp (integer: exact, in no particular order).
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
    uint32_t r;
    asm volatile("redux.sync.add.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

// Exact maximum of v over the 32 lanes of a warp: floats mapped to ints in
// the same order (negative values' magnitude bits flipped), one integer
// warp reduction, mapped back.
__device__ __forceinline__ float warp_max_exact(float v) {
    int k = __float_as_int(v);
    k = k >= 0 ? k : k ^ 0x7FFFFFFF;
    int m;
    asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(m) : "r"(k));
    return __int_as_float(m >= 0 ? m : m ^ 0x7FFFFFFF);
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four (x4) or two (x2) 8x8 b16 matrices from shared memory: lanes 8i..8i+7
// give the row addresses of matrix i (16 contiguous bytes each); register i
// receives matrix i in the mma fragment distribution (lane 4g+c holds row g,
// columns 2c, 2c+1).
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
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
