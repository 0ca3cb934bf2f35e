// pq_gemm_tc.cu -- prefill uint4 x e4m3 group GEMM on the 5th-generation
// tensor cores (tcgen05 MMA, TMEM accumulators, TMA), sm_103a.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Design"
// items 1 (zero point as a row-sum correction, SZ table), 2 (per-group fp8
// activation scales folded once per 128-k slab) and 4 (partition select per
// n-block, one launch for any P); the "Prefill kernel attribution + fix" notes
// (the per-slab fold is the cost to watch) and the A-tiled kernel's choice of
// slab = scale group = 128 k.
//
// One CTA computes a 128 (tokens) x 128 (output features) tile of y.  Per
// 128-k group kb (a "slab"):
//   TMA warp     loads A[p][m0:m0+128][128kb:+128] (e4m3, 128B-swizzled,
//                zero-filled past M), the packed weight tile w[n0:n0+128]
//                [64kb:+64] and the slab's 128 SZ words (16 octets x 8 words
//                of the [N/8][G][8] table) into stage s.
//   expand warps turn each nibble c into the e4m3 code of c (0..15 are exact
//                in e4m3) in the canonical K-major SWIZZLE_128B layout the MMA
//                reads, and convert the SZ words to fp32 (sc, zscale + 8 sc).
//   MMA warp     issues 4 x tcgen05.mma m128n128k32 (kind::f8f6f4, fp32
//                accumulate) into one of two TMEM accumulators, so the MMAs of
//                slab kb+1 run while slab kb is folded.
//   fold warps   tcgen05.ld the slab's D' = sum_k dec(a) * c and fold it into
//                fp32 registers: acc += asg * (sc * D' - (zscale + 8 sc) * rs),
//                which equals asg * (sc * D - zscale * rs) with D the sum over
//                (c - 8): D' = D + 8 * rs exactly, and zscale + 8 sc is exact in
//                fp32.
// Epilogue: bf16 rows < M are stored; nothing else is written.
//
// Every wait is bounded (%globaltimer); a wait that gives up marks the CTA as
// aborted, lets in-flight copies and MMAs finish, frees TMEM, fills its tile
// with NaN and reports through the optional status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pq_device.cuh"
#include "pq_internal.h"

namespace pq {
namespace {

constexpr int BM = 128, BN = 128, BK = 128;
constexpr int kStages = 4;
constexpr int kFoldWarps = 8;     // warps 0..7: warp w folds rows 32(w%4).., columns 64(w/4)..
constexpr int kExpWarps = 4;      // warps 8..11
constexpr int kTmaWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr uint32_t kABytes = BM * BK;
constexpr uint32_t kBpBytes = BN * BK / 2;
constexpr uint32_t kBxBytes = BN * BK;
constexpr uint32_t kSzBytes = BN * 4;
constexpr uint32_t kTxBytes = kABytes + kBpBytes + kSzBytes;
constexpr uint32_t kTmemCols = 256;

struct __align__(1024) Stage {
    uint8_t a[kABytes];       // 128 rows x 128 B, SWIZZLE_128B (TMA)
    uint8_t bx[kBxBytes];     // 128 rows x 128 B, SWIZZLE_128B (expand warps)
    uint8_t bp[kBpBytes];     // 128 rows x 64 B packed nibbles (TMA)
    uint32_t sz[BN];          // f16 (sc, zscale) per column (bulk copy)
    float4 szf[BN / 2];       // (sc[n], sc[n+1], zs8[n], zs8[n+1]) for even n
};

struct Ctrl {
    uint64_t full_tma[kStages];
    uint64_t full_b[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = kStages * sizeof(Stage) + sizeof(Ctrl) + 1024;

struct TcParams {
    const float *asg;
    const float *rs;
    const uint32_t *sz;
    __nv_bfloat16 *y;
    unsigned int *status;
    int M, N, K, pb1, pb2, ldy;
};

// ---------------------------------------------------------------- PTX helpers
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

// kind::f8f6f4 instruction descriptor: D fp32, A and B e4m3, both K-major,
// N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait carries
// the registers so no use can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void set_abort(Ctrl *ctl, unsigned int *status, unsigned int code) {
    if (status) atomicOr(status, code);
    *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
}

// e4m3 codes of 4 nibbles (selector bits 0..15): nibble c < 8 picks byte c of
// the low table, c >= 8 picks byte c-8 of the high table; PRMT's sign mode
// (selector bit 3) turns the other table's byte into 0x00 since every entry
// has a clear sign bit.
// (PTX prmt in its default mode honours the sign-replicate bit of each
// selector nibble; the __byte_perm intrinsic only uses the low three bits.)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t expand4(uint32_t sel, uint32_t sel_x8) {
    constexpr uint32_t kLo0 = 0x44403800u, kLo1 = 0x4E4C4A48u;   // e4m3(0..7)
    constexpr uint32_t kHi0 = 0x53525150u, kHi1 = 0x57565554u;   // e4m3(8..15)
    return prmt(kLo0, kLo1, sel) | prmt(kHi0, kHi1, sel_x8);
}

__device__ __forceinline__ uint4 expand16(uint2 pk) {
    const uint32_t x0 = pk.x, x1 = pk.y;
    const uint32_t y0 = x0 ^ 0x88888888u, y1 = x1 ^ 0x88888888u;
    uint4 o;
    o.x = expand4(x0, y0);
    o.y = expand4(x0 >> 16, y0 >> 16);
    o.z = expand4(x1, y1);
    o.w = expand4(x1 >> 16, y1 >> 16);
    return o;
}

__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFF))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmS, const TcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Stage *stg = reinterpret_cast<Stage *>(base);
    Ctrl *ctl = reinterpret_cast<Ctrl *>(base + kStages * sizeof(Stage));
    volatile int *abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int M = prm.M, N = prm.N, G = prm.K / BK;
    const int p = (n0 >= prm.pb1) + (n0 >= prm.pb2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full_tma[s], 1);
            mbar_init(&ctl->full_b[s], kExpWarps);
            mbar_init(&ctl->empty[s], 1 + kFoldWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tmem_full[b], 1);
            mbar_init(&ctl->tmem_empty[b], kFoldWarps);
        }
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == kTmaWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_map(&tmA);
            prefetch_map(&tmB);
            prefetch_map(&tmS);
            int issued = 0;
            // first stages: weights and SZ (load-time tables) before the
            // preceding kernel has finished, activations after pdl_wait
            const int pre = G < kStages ? G : kStages;
            for (int kb = 0; kb < pre; ++kb) {
                mbar_arrive_expect_tx(&ctl->full_tma[kb], kTxBytes);
                tma_load_2d(stg[kb].bp, &tmB, kb * (BK / 2), n0, &ctl->full_tma[kb]);
                tma_load_2d(stg[kb].sz, &tmS, 8 * kb, n0 / 8, &ctl->full_tma[kb]);
            }
            pdl_wait();
            for (int kb = 0; kb < pre; ++kb) tma_load_3d(stg[kb].a, &tmA, kb * BK, m0, p, &ctl->full_tma[kb]);
            issued = pre;
            for (int kb = pre; kb < G; ++kb) {
                const int s = kb % kStages, use = kb / kStages;
                if (!wait_or_abort(&ctl->empty[s], (use - 1) & 1, abort_flag)) {
                    set_abort(ctl, prm.status, kStatusWaitEmpty);
                    break;
                }
                mbar_arrive_expect_tx(&ctl->full_tma[s], kTxBytes);
                tma_load_3d(stg[s].a, &tmA, kb * BK, m0, p, &ctl->full_tma[s]);
                tma_load_2d(stg[s].bp, &tmB, kb * (BK / 2), n0, &ctl->full_tma[s]);
                tma_load_2d(stg[s].sz, &tmS, 8 * kb, n0 / 8, &ctl->full_tma[s]);
                issued = kb + 1;
            }
            if (*abort_flag) {   // let issued copies land before shared memory is released
                for (int s = 0; s < kStages && s < issued; ++s) {
                    const int last = (issued - 1 - s) / kStages;
                    if (!mbar_wait(&ctl->full_tma[s], last & 1) && prm.status)
                        atomicOr(prm.status, kStatusDrain);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int committed = 0;
            for (int kb = 0; kb < G; ++kb) {
                const int s = kb % kStages, use = kb / kStages;
                const int b = kb & 1, tuse = kb >> 1;
                if (!wait_or_abort(&ctl->full_tma[s], use & 1, abort_flag) ||
                    !wait_or_abort(&ctl->full_b[s], use & 1, abort_flag)) {
                    set_abort(ctl, prm.status, kStatusWaitFull);
                    break;
                }
                if (tuse > 0 && !wait_or_abort(&ctl->tmem_empty[b], (tuse - 1) & 1, abort_flag)) {
                    set_abort(ctl, prm.status, kStatusWaitTmem);
                    break;
                }
                tc_fence_after();
                const uint64_t ad = desc_sw128(smem_u32(stg[s].a));
                const uint64_t bd = desc_sw128(smem_u32(stg[s].bx));
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk)     // +32 bytes along K inside the swizzle row
                    mma_f8(tmem + (uint32_t)(b * BN), ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk),
                           kk > 0 ? 1u : 0u);
                mma_commit(&ctl->empty[s]);
                mma_commit(&ctl->tmem_full[b]);
                committed = kb + 1;
            }
            if (*abort_flag && committed > 0) {   // MMAs must finish before TMEM is freed
                const int kb = committed - 1;
                if (!mbar_wait(&ctl->tmem_full[kb & 1], (kb >> 1) & 1) && prm.status)
                    atomicOr(prm.status, kStatusDrain);
            }
        }
    } else if (warp >= kFoldWarps) {
        // ------------------------------------------------ nibble expansion
        const int et = threadIdx.x - kFoldWarps * 32;    // 0..127
        const int chunk = et & 7;
        for (int kb = 0; kb < G; ++kb) {
            const int s = kb % kStages, use = kb / kStages;
            if (!wait_or_abort(&ctl->full_tma[s], use & 1, abort_flag)) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                break;
            }
            Stage &st = stg[s];
            if (et < BN / 2) {
                const uint32_t w0 = st.sz[2 * et], w1 = st.sz[2 * et + 1];
                const float sc0 = f16lo(w0), sc1 = f16lo(w1);
                st.szf[et] = make_float4(sc0, sc1, f16hi(w0) + 8.0f * sc0, f16hi(w1) + 8.0f * sc1);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = (et >> 3) + 16 * i;
                const uint2 pk = *reinterpret_cast<const uint2 *>(st.bp + row * (BK / 2) + chunk * 8);
                *reinterpret_cast<uint4 *>(st.bx + row * BK + ((chunk ^ (row & 7)) << 4)) = expand16(pk);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->full_b[s]);
        }
    } else {
        // ------------------------------------------------ fold warps
        const int q = warp & 3, h = warp >> 2;
        const int row = 32 * q + lane;
        const int m = m0 + row;
        const bool live = m < M;
        const float *asg_p = prm.asg + (size_t)p * G * M + m;
        const float *rs_p = prm.rs + (size_t)p * G * M + m;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        pdl_wait();        // asg and rs are the preceding prologue's output
        float sa_next = live ? __ldg(asg_p) : 0.0f, r_next = live ? __ldg(rs_p) : 0.0f;
        for (int kb = 0; kb < G; ++kb) {
            const int s = kb % kStages, use = kb / kStages;
            const int b = kb & 1, tuse = kb >> 1;
            const float sa = sa_next, nr = -r_next;
            if (kb + 1 < G && live) {
                sa_next = __ldg(asg_p + (size_t)(kb + 1) * M);
                r_next = __ldg(rs_p + (size_t)(kb + 1) * M);
            }
            if (!wait_or_abort(&ctl->full_b[s], use & 1, abort_flag) ||
                !wait_or_abort(&ctl->tmem_full[b], tuse & 1, abort_flag)) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                break;
            }
            tc_fence_after();
            const float4 *zf = stg[s].szf + 32 * h;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float d[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 64 * h + 32 * half), d);
                if (half == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tmem_empty[b]);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float4 z = zf[16 * half + j];
                    const int c = 32 * half + 2 * j;
                    const float t0 = fmaf(z.z, nr, d[2 * j] * z.x);
                    const float t1 = fmaf(z.w, nr, d[2 * j + 1] * z.y);
                    acc[c] = fmaf(sa, t0, acc[c]);
                    acc[c + 1] = fmaf(sa, t1, acc[c + 1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->empty[s]);
        }
        pdl_trigger();
        // epilogue: bf16 row segment of 64 columns
        if (live) {
            const bool bad = *abort_flag != 0;
            uint4 *dst = reinterpret_cast<uint4 *>(prm.y + (size_t)m * prm.ldy + n0 + 64 * h);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t wv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float lo = acc[8 * i + 2 * j], hi = acc[8 * i + 2 * j + 1];
                    if (bad) lo = hi = __int_as_float(0x7FC00000);
                    const __nv_bfloat162 v2 = __floats2bfloat162_rn(lo, hi);
                    wv[j] = *reinterpret_cast<const uint32_t *>(&v2);
                }
                dst[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

pq_status launch_gemm_tc(const void *a, const float *asg, const float *rs, int M, int N, int K,
                         int P, int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                         unsigned int *dev_status, void *stream, int sm_count) {
    (void)sm_count;
    auto enc = encode_fn();
    if (!enc) return fail(PQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    CUtensorMap tmA, tmB, tmS;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)M, (cuuint64_t)P};
        const cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)K * (cuuint64_t)M};
        const cuuint32_t box[3] = {BK, BM, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        const CUresult r = enc(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(a), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for A: CUresult %d", (int)r);
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        const cuuint32_t box[2] = {BK / 2, BN};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(w), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for w: CUresult %d", (int)r);
    }
    {
        // SZ table [N/8][G][8] words: box = the 8 words of group kb for 16 octets
        const cuuint64_t dims[2] = {(cuuint64_t)(8 * (K / 128)), (cuuint64_t)(N / 8)};
        const cuuint64_t strides[1] = {(cuuint64_t)(32 * (K / 128))};
        const cuuint32_t box[2] = {8, BN / 8};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(sz), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for sz: CUresult %d", (int)r);
    }
    TcParams prm{};
    prm.asg = asg;
    prm.rs = rs;
    prm.sz = static_cast<const uint32_t *>(sz);
    prm.y = static_cast<__nv_bfloat16 *>(y);
    prm.status = dev_status;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.pb1 = pb1;
    prm.pb2 = pb2;
    prm.ldy = ldy;
    const dim3 grid(N / BN, (M + BM - 1) / BM);
    if (grid.y > 65535) return fail(PQ_ERR_SHAPE, "pq_gemm_tc: M = %d too large", M);
    cudaError_t e = cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = launch_pdl(tc_kernel, grid, dim3(kThreads), kSmemBytes, static_cast<cudaStream_t>(stream), tmA, tmB,
                   tmS, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "tc launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

}  // namespace pq
