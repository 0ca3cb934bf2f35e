// pq_gemm_skinny.cu -- decode-band (M <= 16) uint4 x e4m3 group GEMM on CUDA
// cores, streaming the 4.25-bit/weight operands from HBM once.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Design"
// items 1 (zero point as a row-sum correction: per group
// acc += asg * (sc * D - zscale * rowsum), SZ table in one 4-byte load),
// 2 (per-group activation scales folded per 128-k group) and 4 (partition
// of a column from two boundary columns, one launch for any P).
//
// Work split.  A CTA owns a run of column octets (8 output features) for an
// M-tile of MT tokens.  Compute warp kw covers k in [1024 kw, 1024 kw + 1024):
// lane l owns the 32 consecutive k at 1024 kw + 32 l (one quarter of group
// 8 kw + l/4) and keeps that slice of the MT activation rows in registers for
// the whole launch (as f16 pairs; e4m3 converts to f16 exactly).  A producer
// warp streams each octet's weight rows (8 x K/2 contiguous bytes) and its SZ
// words (G x 32 contiguous bytes) into a shared-memory ring with bulk copies
// (cp.async.bulk + mbarrier transaction counts), so the weight stream is
// independent of register pressure.
//
// Consumer groups.  A CTA may hold up to three groups of nkw compute warps
// that share its producer and its ring: octet i of the CTA's run goes to group
// i mod ngrp and ring stage i mod S (S a multiple of ngrp, so a stage always
// serves the same group and no waiter can fall two phases behind).  The launch
// prefers three one-group CTAs per SM and falls back to one CTA with three
// groups.  Measured on decode gate_up (M = 1, K = 5120, N = 17408):
//   - GEMM alone, back to back: the three-group CTA is faster, 11.0 vs
//     11.6 us.  Its groups take the SM's octets round robin and finish within
//     about one octet of each other.  Three separate CTAs on one SM finish up
//     to 2.5 us apart, because the first one served runs its whole range ahead.
//   - Decode step after the prologue: three separate CTAs are faster, 14.4 vs
//     16.0 us.  As soon as the first of them exits, the next launch's CTA
//     takes its place and prefetches weights during this launch's tail and
//     the next prologue.  A whole-SM CTA leaves no such room.
//
// Arithmetic.  A weight nibble c is turned into an f16 *subnormal* whose bits
// are the nibble (value c * 2^-24) by one AND per two nibbles -- no integer to
// float conversion and no bias subtraction -- and multiplied into an fp32
// accumulator with the mixed-precision fma.rn.f32.f16 (exact product, one
// rounding per add).  Nibbles sitting in bits 4..7 of a half are used in place
// as 16 * c * 2^-24, against activations pre-divided by 16 (exact in f16), so
// every product is a * c * 2^-24.  So per group and token the lanes compute
// D' = sum a * c = D + 8 * rs exactly up to fp32 addition, and the fold uses
// sc * D - zscale * rs = sc * D' - (zscale + 8 sc) * rs, where zscale + 8 sc
// is exact in fp32.  The four lanes of a group first sum their partials of the
// octet's 8 columns with a butterfly that hands 2 columns to each lane, so
// each lane folds only its 2 columns; a second butterfly over the 8 groups of
// the warp finishes the sum (9 exchanges per 8 columns in all), shared memory
// reduces the k-warps in a fixed order (deterministic), and the bf16 result is
// stored once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pq_device.cuh"
#include "pq_internal.h"

namespace pq {
namespace {

constexpr int kMaxK = kSkinnyMaxK;    // 16 compute warps + producer; pq_gemm sends larger K to the narrow tcgen05 kernel
constexpr int kSmemBudget = 220 * 1024;    // per SM, over all resident CTAs

struct SkinnyParams {
    const uint8_t *a;
    const float *asg;
    const float *rs;
    const uint8_t *w;
    const uint8_t *whi;     // int5: fifth-bit planes [N][K/8] (else null)
    const uint32_t *sz;     // [N/8][G][8] words: f16 scale | f16 zscale << 16
    __nv_bfloat16 *y;
    unsigned int *status;
    int M, N, K, G, pb1, pb2, ldy;
    int oct_per_cta, n_oct, nkw, ngrp, stages;
    // a stage: the octet's nibble rows (w_bytes), its fifth-bit rows (h_bytes,
    // int5 only) and its SZ words (from sz_off)
    uint32_t stage_bytes, w_bytes, h_bytes, sz_off;
    WaitBound wait;           // the pipeline waits' bound
};

__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two_codes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_codes));
    return r;
}

// (a.lo / 16, a.hi / 16): exact for the e4m3 range (>= 2^-13 stays normal in f16)
__device__ __forceinline__ uint32_t hmul2_sixteenth(uint32_t a) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(0x2C002C00u));
    return r;
}

// v shifted left by s bits (right by -s when s < 0); s is a compile-time
// constant after unrolling
__device__ __forceinline__ uint32_t shift_bits(uint32_t v, int s) { return s >= 0 ? v << s : v >> -s; }

// acc_lo += a.lo * b.lo, acc_hi += a.hi * b.hi with f16 operands and fp32 accumulators
__device__ __forceinline__ void fma2_f32_f16(float &acc_lo, float &acc_hi, uint32_t a, uint32_t b) {
    asm("{\n.reg .f16 al, ah, bl, bh;\n"
        "mov.b32 {al, ah}, %2;\n"
        "mov.b32 {bl, bh}, %3;\n"
        "fma.rn.f32.f16 %0, al, bl, %0;\n"
        "fma.rn.f32.f16 %1, ah, bh, %1;\n}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(a), "r"(b));
}

__device__ __forceinline__ float half_lo(uint32_t w) {
    float f;
    asm("{\n.reg .f16 l, h;\nmov.b32 {l, h}, %1;\ncvt.f32.f16 %0, l;\n}" : "=f"(f) : "r"(w));
    return f;
}
__device__ __forceinline__ float half_hi(uint32_t w) {
    float f;
    asm("{\n.reg .f16 l, h;\nmov.b32 {l, h}, %1;\ncvt.f32.f16 %0, h;\n}" : "=f"(f) : "r"(w));
    return f;
}

// Keep half of a lane's NC values, exchanging the other half with the lane
// whose index differs in bit `mask`: out[i] = own kept value + partner's
// value of the same column.  Lanes with the bit clear keep the lower half.
template <int NC>
__device__ __forceinline__ void split_step(const float (&in)[NC], float (&out)[NC / 2], int lane, int mask) {
    const bool hi = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < NC / 2; ++i) {
        const float send = hi ? in[i] : in[i + NC / 2];
        const float keep = hi ? in[i + NC / 2] : in[i];
        out[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, mask);
    }
}

// The producer: lane 0 of the last warp streams the CTA's octets, in order,
// into the S-stage ring: each octet's weight rows (8 x K/2 contiguous bytes)
// and its SZ words (G x 32 contiguous bytes) with two bulk copies completing
// on full[s]; a stage is refilled once its consumer group has released it on
// empty[s].  (Weights and SZ words are load-time tables, not written by the
// preceding kernel, so they stream before its completion.)  Returns the
// number of octets issued.
__device__ __forceinline__ int produce_octets(const SkinnyParams &prm, uint8_t *smem, uint64_t *full,
                                               uint64_t *empty, volatile int *abort_flag, int oct0,
                                               int noct) {
    const int S = prm.stages, K = prm.K, G = prm.G;
    int issued = 0;
    for (int i = 0, s = 0, use = 0; i < noct; ++i) {     // s = i mod S, use = i / S
        if (i > 0 && ++s == S) {
            s = 0;
            ++use;
        }
        if (*abort_flag) break;
        if (use > 0 && !wait_or_abort(&empty[s], (use - 1) & 1, abort_flag, prm.wait)) {
            if (prm.status) atomicOr(prm.status, kStatusWaitEmpty);
            *abort_flag = 1;
            break;
        }
        uint8_t *st = smem + (size_t)s * prm.stage_bytes;
        const int o = oct0 + i;
        mbar_arrive_expect_tx(&full[s], prm.stage_bytes);
        bulk_g2s(st, prm.w + (size_t)o * 8 * (K / 2), prm.w_bytes, &full[s]);
        if (prm.h_bytes) bulk_g2s(st + prm.w_bytes, prm.whi + (size_t)o * prm.h_bytes, prm.h_bytes, &full[s]);
        bulk_g2s(st + prm.sz_off, prm.sz + (size_t)o * G * 8, 32u * (uint32_t)G, &full[s]);
        issued = i + 1;
    }
    return issued;
}

template <int MT, int kBits>
__global__ void skinny_kernel(const SkinnyParams prm) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int nkw = prm.nkw, S = prm.stages, ngrp = prm.ngrp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * prm.stage_bytes);
    uint64_t *empty = full + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + S);
    float *ypart = reinterpret_cast<float *>(empty + S + 2);

    // balanced contiguous octet range of this CTA
    const int oct0 = (int)(((long long)blockIdx.x * prm.n_oct) / gridDim.x);
    const int noct = (int)(((long long)(blockIdx.x + 1) * prm.n_oct) / gridDim.x) - oct0;
    const int ncol = prm.oct_per_cta * 8;
    const int m0 = blockIdx.y * MT;
    const int K = prm.K, G = prm.G, M = prm.M;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nkw);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    pdl_trigger();
    int issued = 0;     // octets the producer issued, for the drain after a give-up
    if (warp == ngrp * nkw) {
        if (lane == 0) issued = produce_octets(prm, smem, full, empty, abort_flag, oct0, noct);
    } else {
        // ---------------- compute warps ----------------
        const int grp = warp / nkw, kw = warp - grp * nkw;
        const int k0 = 1024 * kw + 32 * lane;
        const bool kvalid = k0 < K;
        const int g = kvalid ? (k0 >> 7) : 0;
        pdl_wait();        // a, asg, rs are the preceding prologue's output
        uint32_t A[MT][16];
        // per row of this lane's group: 2^24 asg, asg * rs and zo * asg * rs,
        // zo = 8 (int4: the codes are summed raw, so zscale + 8 sc) or 16
        // (int5: zscale + 16 sc)
        constexpr float kZOff = kBits == 5 ? 16.0f : 8.0f;
        float asg24_r[MT], ar_r[MT], arz_r[MT];
        int cur_p = -1;
        // s = i mod S and use = i / S, stepped without a division (S is a
        // multiple of ngrp, so s wraps back to grp)
        for (int i = grp, s = grp, use = 0; i < noct; i += ngrp) {
            if (i > grp && (s += ngrp) >= S) {
                s -= S;
                ++use;
            }
            const int n0 = (oct0 + i) * 8;
            const int p = (n0 >= prm.pb1) + (n0 >= prm.pb2);
            if (p != cur_p) {
                cur_p = p;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const int row = m0 + m;
                    uint32_t u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    asg24_r[m] = 0.0f;
                    ar_r[m] = 0.0f;
                    arz_r[m] = 0.0f;
                    if (kvalid && row < M) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            prm.a + ((size_t)p * M + row) * K + k0);
                        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                        u[0] = v0.x; u[1] = v0.y; u[2] = v0.z; u[3] = v0.w;
                        u[4] = v1.x; u[5] = v1.y; u[6] = v1.z; u[7] = v1.w;
                        const float sa = __ldg(prm.asg + ((size_t)p * G + g) * M + row);
                        asg24_r[m] = sa * 16777216.0f;
                        ar_r[m] = sa * __ldg(prm.rs + ((size_t)p * G + g) * M + row);
                        arz_r[m] = kZOff * ar_r[m];
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // activation bytes k0..k0+7 (k0 = 8q) -> the pairs of the
                        // masked weight halves: word byte b holds k0 + b (low
                        // nibble) and k0 + b + 4 (high nibble), so the masks below
                        // give (k0, k0+2), 16 (k0+4, k0+6) and, after the 8-bit
                        // shift, (k0+1, k0+3), 16 (k0+5, k0+7)
                        const uint32_t t01 = __byte_perm(u[2 * q], u[2 * q + 1], 0x6420);
                        const uint32_t t23 = __byte_perm(u[2 * q], u[2 * q + 1], 0x7531);
                        // the partners of the high nibbles (used in place as 16 c)
                        // are divided by 16 -- exact in f16 -- so every product is
                        // a * c * 2^-24
                        A[m][4 * q + 0] = f16x2_from_e4m3x2(t01 & 0xFFFF);
                        A[m][4 * q + 1] = hmul2_sixteenth(f16x2_from_e4m3x2(t01 >> 16));
                        A[m][4 * q + 2] = f16x2_from_e4m3x2(t23 & 0xFFFF);
                        A[m][4 * q + 3] = hmul2_sixteenth(f16x2_from_e4m3x2(t23 >> 16));
                    }
                }
            }
            // warp-uniform: the shuffles below need the whole warp
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&full[s], use & 1, abort_flag, prm.wait))) {
                if (lane == 0) {
                    if (prm.status) atomicOr(prm.status, kStatusWaitFull);
                    *abort_flag = 1;
                }
                break;
            }
            const uint8_t *st = smem + (size_t)s * prm.stage_bytes;
            // dot products of the 8 columns: lane partials in units of 2^-24
            float S[MT][8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 wv = make_uint4(0, 0, 0, 0);
                if (kvalid) wv = *reinterpret_cast<const uint4 *>(st + (size_t)j * (K / 2) + (k0 >> 1));
                float acc[MT][2];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0.0f;
                const uint32_t wq[4] = {wv.x, wv.y, wv.z, wv.w};
                // int5: the fifth bits of this lane's 32 k, one 32-k block word
                // (bit 8j' + q' of the word: k = 4q' + j')
                uint32_t hw = 0;
                if constexpr (kBits == 5)
                    if (kvalid) hw = *reinterpret_cast<const uint32_t *>(st + prm.w_bytes + (size_t)j * (K / 8) + (k0 >> 3));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t x = wq[q], x8 = x >> 8;
                    uint32_t lo = x & 0x000F000Fu, hi = x & 0x00F000F0u;
                    uint32_t lo2 = x8 & 0x000F000Fu, hi2 = x8 & 0x00F000F0u;
                    if constexpr (kBits == 5) {
                        // Each fifth bit joins its nibble in the same f16 half: at
                        // bit 4 above a low nibble (c = nibble + 16 b) and at bit 8
                        // above a high nibble used as 16 nibble, so the one FMA
                        // multiplies the 5-bit code (mantissa bits 0..8, still a
                        // subnormal).  The shifts bring the bits of k = 8q + {0, 2},
                        // {4, 6}, {1, 3}, {5, 7} to those places.
                        lo |= shift_bits(hw, 4 - 2 * q) & 0x00100010u;
                        hi |= shift_bits(hw, 7 - 2 * q) & 0x01000100u;
                        lo2 |= (hw >> (4 + 2 * q)) & 0x00100010u;
                        hi2 |= (hw >> (2 * q + 1)) & 0x01000100u;
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        fma2_f32_f16(acc[m][0], acc[m][1], A[m][4 * q + 0], lo);
                        fma2_f32_f16(acc[m][0], acc[m][1], A[m][4 * q + 1], hi);
                        fma2_f32_f16(acc[m][0], acc[m][1], A[m][4 * q + 2], lo2);
                        fma2_f32_f16(acc[m][0], acc[m][1], A[m][4 * q + 3], hi2);
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) S[m][j] = acc[m][0] + acc[m][1];
            }
            // this lane's group folds columns cb, cb+1 (cb even): the SZ words of
            // (octet, group g) are contiguous, one 8-byte load
            const int cb = 4 * ((lane >> 1) & 1) + 2 * (lane & 1);
            const uint2 szp = *reinterpret_cast<const uint2 *>(st + prm.sz_off + 32 * g + 4 * cb);
            // the stage is refilled by a bulk copy (the async proxy): order this
            // warp's reads of it before that write, then release it
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const float sc0 = half_lo(szp.x), zs0 = half_hi(szp.x);
            const float sc1 = half_lo(szp.y), zs1 = half_hi(szp.y);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // sum the 4 lanes of the group, splitting the columns on the way:
                // bit 1 keeps 4 of 8, bit 0 keeps 2 of 4 (columns cb, cb+1)
                float h4[4], h2[2];
                split_step<8>(S[m], h4, lane, 2);
                split_step<4>(h4, h2, lane, 1);
                // fold (once per group and column): asg * (sc * D' - (zs + zo sc) * rs)
                // with D' = 2^24 * sum
                float f[2];
                f[0] = fmaf(sc0 * asg24_r[m], h2[0], -fmaf(sc0, arz_r[m], zs0 * ar_r[m]));
                f[1] = fmaf(sc1 * asg24_r[m], h2[1], -fmaf(sc1, arz_r[m], zs1 * ar_r[m]));
                // sum the 8 groups of the warp: bit 4 keeps 1 of 2, bits 3 and 2 add
                float h1[1];
                split_step<2>(f, h1, lane, 16);
                float t = h1[0];
                t += __shfl_xor_sync(0xFFFFFFFFu, t, 8);
                t += __shfl_xor_sync(0xFFFFFFFFu, t, 4);
                if ((lane & 12) == 0)          // lanes 0-3 and 16-19 hold column cb + bit 4
                    ypart[(kw * MT + m) * ncol + 8 * i + cb + ((lane >> 4) & 1)] = t;
            }
        }
    }
    __syncthreads();

    // reduce the k-warps in a fixed order and store bf16 rows (NaN after an abort)
    const bool bad = *abort_flag != 0;
    // after a give-up (the flag is final once every warp has left its loop):
    // every copy already issued lands before shared memory is released (these
    // waits keep the full bound)
    if (bad && warp == ngrp * nkw && lane == 0) {
        for (int s = 0; s < S && s < issued; ++s) {
            const int last_use = (issued - 1 - s) / S;
            if (!mbar_wait(&full[s], last_use & 1) && prm.status) atomicOr(prm.status, kStatusDrain);
        }
    }
    const int cols = noct * 8;
    for (int e = threadIdx.x; e < MT * cols; e += blockDim.x) {
        const int m = e / cols, c = e - m * cols;
        if (m0 + m >= M) continue;
        float v = 0.0f;
        for (int k = 0; k < nkw; ++k) v += ypart[(k * MT + m) * ncol + c];
        if (bad) v = __int_as_float(0x7FC00000);
        prm.y[(size_t)(m0 + m) * prm.ldy + oct0 * 8 + c] = __float2bfloat16_rn(v);
    }
}

using SkinnyFn = void (*)(SkinnyParams);

// Registers per thread (allocation granule of 8) and the thread limit of a
// kernel, or false if its attributes cannot be read.
bool kernel_limits(SkinnyFn k, int *regs, int *max_threads) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    *regs = (fa.numRegs + 7) / 8 * 8;
    *max_threads = fa.maxThreadsPerBlock;
    return true;
}

// Whether kernel k fits the register file with `warps` warps.
bool fits_registers(SkinnyFn k, int warps) {
    int regs, max_threads;
    if (!kernel_limits(k, &regs, &max_threads)) return false;
    return regs * 32 * warps <= 65536 && 32 * warps <= max_threads;
}

// Launch kernel k (mt rows per M-tile) over the octet ring.  Three consumer
// groups per SM (the more compute warps per SM, the more load latency is
// hidden): preferably three one-group CTAs, else one CTA with three groups,
// else fewer, each group with 2..4 ring stages; shared memory and registers
// per SM are kept under their limits.  CTAs per M-tile: a whole multiple of
// the SM count when there are enough octets, each with a balanced octet
// range.
pq_status launch_ring(SkinnyFn k, int mt, SkinnyParams prm, int sm_count, cudaStream_t stream) {
    const int mtiles = (prm.M + mt - 1) / mt;
    const int sms = sm_count > 0 ? sm_count : 1;
    auto smem_for = [&](int stages, int opc) {
        return (size_t)stages * prm.stage_bytes + 16 * (size_t)stages + 16 +
               (size_t)prm.nkw * mt * opc * 8 * 4;
    };
    // (groups per CTA, CTAs per SM) in order of preference
    constexpr int kConfigs[5][2] = {{1, 3}, {3, 1}, {1, 2}, {2, 1}, {1, 1}};
    for (const auto &cfg : kConfigs) {
        const int ngrp = cfg[0], per_sm = cfg[1];
        const int warps = ngrp * prm.nkw + 1;
        if (!fits_registers(k, warps * per_sm)) continue;
        int ctas = sms * per_sm / mtiles;
        if (ctas < 1) ctas = 1;
        if (ctas > prm.n_oct) ctas = prm.n_oct;
        const int opc = (prm.n_oct + ctas - 1) / ctas;
        int spg = 4;
        while (spg > 2 && smem_for(ngrp * spg, opc) * per_sm > (size_t)kSmemBudget) --spg;
        const size_t smem = smem_for(ngrp * spg, opc);
        if (smem * per_sm > (size_t)kSmemBudget) continue;
        prm.ngrp = ngrp;
        prm.stages = ngrp * spg;
        prm.oct_per_cta = opc;
        const dim3 grid(ctas, mtiles);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return fail(PQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        e = launch_pdl(k, grid, dim3(32 * warps), smem, stream, prm);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "skinny launch: %s", cudaGetErrorString(e));
        return PQ_OK;
    }
    return fail(PQ_ERR_SHAPE, "pq_gemm_skinny: K = %d needs too much shared memory", prm.K);
}

}  // namespace

pq_status launch_gemm_skinny(const void *a, const float *asg, const float *rs, int M, int N, int K,
                             int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                             int ldy, unsigned int *dev_status, void *stream, int sm_count,
                             const void *whi) {
    (void)P;
    if (K > kMaxK) return fail(PQ_ERR_SHAPE, "pq_gemm_skinny: K = %d > %d", K, kMaxK);
    SkinnyParams prm{};
    prm.a = static_cast<const uint8_t *>(a);
    prm.asg = asg;
    prm.rs = rs;
    prm.w = static_cast<const uint8_t *>(w);
    prm.whi = static_cast<const uint8_t *>(whi);
    prm.sz = static_cast<const uint32_t *>(sz);
    prm.y = static_cast<__nv_bfloat16 *>(y);
    prm.status = dev_status;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.G = K / 128;
    prm.pb1 = pb1;
    prm.pb2 = pb2;
    prm.ldy = ldy;
    prm.wait = pipeline_wait_bound();
    prm.n_oct = N / 8;
    prm.nkw = (K + 1023) / 1024;
    prm.w_bytes = (uint32_t)(8 * (K / 2));
    prm.h_bytes = whi ? (uint32_t)(8 * (K / 8)) : 0u;      // int5: the octet's fifth-bit rows
    prm.sz_off = prm.w_bytes + prm.h_bytes;
    prm.stage_bytes = prm.sz_off + 32u * (uint32_t)prm.G;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // rows per M-tile: the smallest power of two >= M (at most 8; int5 at most
    // 4) whose instantiation fits the register file with one group of k-warps
    const int w1 = prm.nkw + 1;
    if (whi) {
        if (M == 1 && fits_registers(skinny_kernel<1, 5>, w1)) return launch_ring(skinny_kernel<1, 5>, 1, prm, sm_count, st);
        if (M <= 2 && fits_registers(skinny_kernel<2, 5>, w1)) return launch_ring(skinny_kernel<2, 5>, 2, prm, sm_count, st);
        if (fits_registers(skinny_kernel<4, 5>, w1)) return launch_ring(skinny_kernel<4, 5>, 4, prm, sm_count, st);
        if (fits_registers(skinny_kernel<2, 5>, w1)) return launch_ring(skinny_kernel<2, 5>, 2, prm, sm_count, st);
        if (fits_registers(skinny_kernel<1, 5>, w1)) return launch_ring(skinny_kernel<1, 5>, 1, prm, sm_count, st);
        return fail(PQ_ERR_CUDA, "pq_gemm5_skinny: no instantiation fits K = %d", K);
    }
    if (M == 1 && fits_registers(skinny_kernel<1, 4>, w1)) return launch_ring(skinny_kernel<1, 4>, 1, prm, sm_count, st);
    if (M <= 2 && fits_registers(skinny_kernel<2, 4>, w1)) return launch_ring(skinny_kernel<2, 4>, 2, prm, sm_count, st);
    if (M <= 4 && fits_registers(skinny_kernel<4, 4>, w1)) return launch_ring(skinny_kernel<4, 4>, 4, prm, sm_count, st);
    if (fits_registers(skinny_kernel<8, 4>, w1)) return launch_ring(skinny_kernel<8, 4>, 8, prm, sm_count, st);
    if (fits_registers(skinny_kernel<4, 4>, w1)) return launch_ring(skinny_kernel<4, 4>, 4, prm, sm_count, st);
    if (fits_registers(skinny_kernel<2, 4>, w1)) return launch_ring(skinny_kernel<2, 4>, 2, prm, sm_count, st);
    if (fits_registers(skinny_kernel<1, 4>, w1)) return launch_ring(skinny_kernel<1, 4>, 1, prm, sm_count, st);
    return fail(PQ_ERR_CUDA, "pq_gemm_skinny: no instantiation fits K = %d", K);
}

}  // namespace pq
