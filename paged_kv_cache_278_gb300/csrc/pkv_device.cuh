// pkv_device.cuh -- small inline-PTX helpers shared by the sm_103a kernels:
// mbarrier set-up and bounded waits, 1-D bulk copies (the TMA engine's
// non-tensor form) from global into shared memory, and the per-translation-unit
// device error word.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace pkv {

constexpr unsigned kFullMask = 0xffffffffu;

// A wait on an mbarrier gives up after this many nanoseconds of %globaltimer,
// records PKV_DEV_WAIT_TIMEOUT and lets the kernel finish instead of hanging.
// PKV_WAIT_TEST (a separate test build of the library, never the product) makes
// one wait of the decode kernel run out on purpose and shortens the limit to 1 ms.
#ifndef PKV_WAIT_TEST
#define PKV_WAIT_TEST 0
#endif
constexpr uint64_t kWaitLimitNs = PKV_WAIT_TEST ? 1000000ull : 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later asynchronous-proxy writes to the same bytes (buffer reuse).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D tensor-map copy of one box into shared memory, completion counted on `bar` in bytes.
// x (innermost, elements) must make a 16-byte-aligned offset.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tensor_map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(tensor_map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 3-D tensor-map copy of one box into shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tensor_map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(tensor_map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t bits) {
    __half2 h = *reinterpret_cast<__half2 *>(&bits);
    return __half22float2(h);
}

__device__ __forceinline__ float lds32f(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Two signed int8 values -> an exact fp16x2.  `biased` holds four int8 bytes XOR 0x80 (value + 128
// as unsigned); `sel` picks bytes (0x4140: bytes 0 and 1, 0x4342: bytes 2 and 3).  Each picked byte
// becomes the low mantissa byte of 0x64xx = 1024 + byte, and subtracting 1152 leaves the integer.
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t biased, uint32_t sel) {
    const uint32_t h = __byte_perm(biased, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

// Symmetric int8 code of x for the row scale s = max|k| / 127: round-half-even(x / s) in
// [-127, 127] with IEEE float32 division; 0 when s == 0.
__device__ __forceinline__ int quantize_int8(float x, float s) {
    if (s == 0.f) return 0;
    const int c = __float2int_rn(__fdiv_rn(x, s));
    return c > 127 ? 127 : (c < -127 ? -127 : c);
}

// Four E4M3 codes (8-bit floating point: sign, 4 exponent bits with bias 7, 3 fraction bits,
// largest finite 448) -> two fp16x2, exactly (every E4M3 value is an fp16 value): bytes 0, 1 go
// to the low and high half of lo, bytes 2, 3 to those of hi.  One hardware conversion per pair.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// E4M3 codes of x / s for the row scale s = max|x| / 448: the nearest code (ties to the even
// code, the sign kept when rounding to zero), |x / s| clamped to 448, with IEEE float32
// division; code 0 when s == 0.  lo goes to bits 0-7, hi to bits 8-15.
__device__ __forceinline__ uint32_t quantize_e4m3x2(float lo, float hi, float s) {
    if (s == 0.f) return 0u;
    const float ylo = __fdiv_rn(lo, s), yhi = __fdiv_rn(hi, s);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(yhi), "f"(ylo));
    return r;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += a (16x16 fp16, row-major) * b (16x8 fp16, column-major), fp32 accumulators (warp-wide MMA)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (c0, c1) += (a0, a1) * (b0, b1): one packed two-lane fp32 FMA (Blackwell FFMA2), each lane
// rounded exactly like fmaf.
__device__ __forceinline__ void fma2(float &c0, float &c1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory) --------------------

// Allocate / free `ncols` tensor-memory columns (a power of two >= 32) for this CTA; executed by
// every thread of one warp.  The allocated base address is written to the shared-memory slot.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte swizzle: rows of 128 B
// (64 fp16 of K), 8-row groups 1024 B apart (stride byte offset), the leading byte offset unused
// (each MMA's 16-element K slice lies inside one 128-byte row), descriptor version 1, layout 2
// (128-byte swizzle).  The tile must start on a 1024-byte boundary; a K step inside the row
// advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t umma_desc_k_sw128(uint32_t smem_addr) {
    return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Shared-memory matrix descriptor of an MN-major operand tile in the 128-byte swizzle: 64 elements of
// the M/N dimension per 128-byte row, rows along K, 8-row groups `sbo` bytes apart (stride byte
// offset) and 64-wide M/N slabs `lbo` bytes apart (leading byte offset), descriptor version 1,
// layout 2.  The start must lie on a 1024-byte boundary.
__device__ __forceinline__ uint64_t umma_desc_mn_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16 with fp16 A and B (both K-major), fp32 accumulation, M x N;
// bit 16 set makes B MN-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane (warp w of a warpgroup reads
// lanes 32 (w % 4) .. + 31); the load and its completion wait are one statement so no use of the
// registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}

// Release-acquire increment at GPU scope; returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *addr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx.ftz.f32: one instruction;
// subnormal results flush to zero).  For softmax weights in [0, 1] whose products are split into
// fp16 hi + lo parts; the attention results it feeds are checked against the float64 oracle.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: let the next kernel in the stream start launching now, and
// (in that kernel) wait until the preceding grid has completed and its writes are visible.
// Both are no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// First error wins; later ones are dropped.
__device__ __forceinline__ void record_error(int *word, int code) { atomicCAS(word, 0, code); }

}  // namespace pkv
