// pq_tcgen05.cuh -- inline-PTX pieces shared by the two tcgen05 GEMM kernels
// (prefill tiles and narrow-M tiles): TMA tensor copies, UMMA descriptors and
// issue, TMEM loads, the nibble -> e4m3 expansion, packed f32x2 arithmetic and
// the host-side tensor-map encoder entry point.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pq_device.cuh"

namespace pq {
namespace tc {

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand in the canonical SWIZZLE_128B layout: 8-row atoms of 1024 B
// (stride byte offset 1024), descriptor version 1, layout type 2 (128B swizzle).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f8f6f4 instruction descriptor: D fp32 (bits 4-5 = 1), A and B e4m3
// (type 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f8(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accum) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}

// K-major operand without swizzle (layout type 0): 8-row x 16-byte core
// matrices, lbo = byte distance between core matrices adjacent along K, sbo =
// between core matrices adjacent along M/N; descriptor version 1.
__device__ __forceinline__ uint64_t desc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// kind::f16 instruction descriptor with bf16 A and B (type 1 at bits 7-9 and
// 10-12), D fp32, both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accum) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}

// x ~ hi + mid + lo, each the bf16 rounding (to nearest even) of what the
// previous parts leave (those differences are exact in fp32), as raw bf16
// bits: 24 significant bits between them.
__device__ __forceinline__ void bf16_split3(float x, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const float r1 = __fsub_rn(x, __bfloat162float(h));
    const __nv_bfloat16 m = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(m));
    hi = __bfloat16_as_ushort(h);
    mid = __bfloat16_as_ushort(m);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

// Non-blocking test of three mbarrier phases issued back to back, so their
// shared-memory round trips overlap (acquire on success).
__device__ __forceinline__ uint32_t mbar_test3(uint64_t *b0, uint32_t p0, uint64_t *b1, uint32_t p1,
                                               uint64_t *b2, uint32_t p2) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred q0, q1, q2;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n"
        "and.pred q0, q0, q1;\nand.pred q0, q0, q2;\nselp.u32 %0, 1, 0, q0;\n}"
        : "=r"(r)
        : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1), "r"(smem_u32(b2)), "r"(p2)
        : "memory");
    return r;
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n.reg .pred p;\n.reg .b32 r;\nelect.sync r|p, 0xffffffff;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 4-byte asynchronous global -> shared copy (zero-fill when !valid; the source
// is then not read) and the arrival on an mbarrier once all of this thread's
// copies have landed (the arrival is part of the barrier's expected count).
__device__ __forceinline__ void cp_async4(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait for two phases: one overlapped test of both first, then each
// barrier in turn (the common case, both complete, costs one round trip).
__device__ __forceinline__ uint32_t mbar_test2(uint64_t *b0, uint32_t p0, uint64_t *b1, uint32_t p1) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred q0, q1;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n"
        "and.pred q0, q0, q1;\nselp.u32 %0, 1, 0, q0;\n}"
        : "=r"(r)
        : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1)
        : "memory");
    return r;
}
__device__ __forceinline__ bool wait2_or_abort(uint64_t *b0, uint32_t p0, uint64_t *b1, uint32_t p1,
                                               volatile int *abort_flag, const WaitBound &wb) {
    if (mbar_test2(b0, p0, b1, p1)) return true;
    return wait_or_abort(b0, p0, abort_flag, wb) && wait_or_abort(b1, p1, abort_flag, wb);
}
// Bounded wait for three phases: one overlapped test first, then each barrier
// in turn (the common case, all three complete, costs one round trip).
__device__ __forceinline__ bool wait3_or_abort(uint64_t *b0, uint32_t p0, uint64_t *b1, uint32_t p1,
                                               uint64_t *b2, uint32_t p2, volatile int *abort_flag,
                                               const WaitBound &wb) {
    if (mbar_test3(b0, p0, b1, p1, b2, p2)) return true;
    return wait_or_abort(b0, p0, abort_flag, wb) && wait_or_abort(b1, p1, abort_flag, wb) &&
           wait_or_abort(b2, p2, abort_flag, wb);
}



// PTX prmt in its default mode (the __byte_perm intrinsic only uses the low
// three bits of each selector nibble).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Sixteen packed nibbles -> sixteen e4m3 bytes in k order, each the e4m3
// value c * 2^-9: a byte holding a nibble c alone is exactly that e4m3 number
// (bit 3 is the lowest exponent bit, so codes 0..7 are the subnormals
// m * 2^-9 and 8..15 the normals (1 + m/8) * 2^-6).  The packed layout puts
// k0 + b in the low and k0 + b + 4 in the high nibble of byte b of each word
// (k0 = 0, 8), so one AND gives k0..k0+3 in byte order and a shift and an AND
// give k0+4..k0+7: 6 instructions per 16 weights.  The MMA result is
// therefore 2^-9 * sum a * c; the fold multiplies its weight scale by 2^9.
constexpr float kNibbleScale = 512.0f;

__device__ __forceinline__ uint4 expand16(uint2 pk) {
    return make_uint4(pk.x & 0x0F0F0F0Fu, (pk.x >> 4) & 0x0F0F0F0Fu, pk.y & 0x0F0F0F0Fu,
                      (pk.y >> 4) & 0x0F0F0F0Fu);
}

// int5 weights: sixteen packed low nibbles plus their sixteen fifth bits ->
// sixteen e4m3 bytes of value (c - 16) * 2^-9, c = nibble + 16 * bit, in k
// order.  Fifth bit 1: c - 16 is the nibble itself, the byte of expand16.
// Fifth bit 0: c - 16 = -(16 - nibble) with 16 - nibble in 1..16, and that
// magnitude alone in a byte is again its own e4m3 value times 2^-9 (16 ->
// 0x10 = 2^-5), so the byte is 0x80 | (16 - nibble) = 0x90 - nibble (no
// borrow leaves a byte).  hs is the 32-k fifth-bit block word shifted right by
// 4h for the 16-k half h it covers, so that bit q of byte j is the fifth bit
// of k = 4q + j of these sixteen (bit 4 + q: the other half's, or nothing).
// Shifting it left by 7 - q puts the bits of word q's four k on the four
// byte top bits (every other bit lands below a top bit), and the
// sign-replicating byte permute widens them to byte masks.
__device__ __forceinline__ uint4 expand16_int5(uint2 pk, uint32_t hs) {
    const uint4 e = expand16(pk);
    uint32_t nib[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t msk = prmt(hs << (7 - q), 0u, 0xBA98u);
        nib[q] = (nib[q] & msk) | ((0x90909090u - nib[q]) & ~msk);
    }
    return make_uint4(nib[0], nib[1], nib[2], nib[3]);
}

__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFF))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
// ---------------------------------------------------------------- fold pieces
// Wait for the thread's outstanding TMEM loads, carrying the registers
// through the wait so their uses stay after it.
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}
// Wait for the thread's outstanding TMEM loads, carrying two load buffers
// through the wait so their uses stay after it.
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[16], uint32_t (&t)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(t[0]), "+r"(t[1]), "+r"(t[2]), "+r"(t[3]), "+r"(t[4]),
                   "+r"(t[5]), "+r"(t[6]), "+r"(t[7]), "+r"(t[8]), "+r"(t[9]), "+r"(t[10]), "+r"(t[11]),
                   "+r"(t[12]), "+r"(t[13]), "+r"(t[14]), "+r"(t[15])
                 :
                 : "memory");
}
// 16x256b.x4 TMEM load (no wait): for repetition j (columns 8j..8j+7 of the
// address), d[4j], d[4j+1] = lane base + g4, columns 8j + 2c4 + {0, 1};
// d[4j+2], d[4j+3] = lane base + 8 + g4, same columns (g4 = lane / 4, c4 = lane % 4).
__device__ __forceinline__ void tmem_issue256(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Packed ops, kept in program order (volatile) so each chunk's chains are
// issued stage by stage.
__device__ __forceinline__ uint64_t fmul2v(uint64_t a, uint64_t b) {
    uint64_t d;
    asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t ffma2v(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// 32x32b.x16 TMEM load (no wait): thread t of the warp receives lane
// (lane base + t), 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_issue32x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// ---------------------------------------------------------------- host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace tc
}  // namespace pq
