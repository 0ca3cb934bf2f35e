// pq_rotate_quant.cu -- the fused prologue: channel scale, eight layers of
// Givens rotations per 128-channel group, per-(token, group) amax, e4m3 encode
// and code-domain row-sums, for up to three partitions, in one launch.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Design"
// items 2 (per-group fp8 activation scales, no cross-block sync) and 3 (fused
// prologue; records read once per chunk; row-sum = sum of what the codes decode
// to), "Gates passed" (the scale is amax times the fp32 reciprocal of 448; the
// outputs match a CPU evaluation bit for bit) and "2026-09-15: hardware e4m3
// convert" (the hardware round-to-nearest-even convert, wrapped so that a NaN
// gives code zero, a negative zero gives positive zero and magnitudes
// saturate at 448).
//
// Layout on the GPU (M > 16).  One CTA owns a tile of 64 tokens x one
// 128-group x one partition (the partition is the grid's z dimension).  The
// tile is held in shared memory as v[k][token pair] (two fp32 values, tokens
// 2l and 2l+1, per 8-byte word): in a Givens layer lane l of a warp works on
// its two tokens of one pair at a time, so the 32 lanes touch consecutive
// 8-byte words, free of bank conflicts whatever the pair permutation is.
// Each of the 8 warps owns 8 of the 64 slots of every layer.  The records come
// in the packer's chained order: the channel a slot keeps from one layer is
// the first channel of its pair in the next, so each slot holds that value in
// registers and exchanges only the other one through shared memory -- one
// 8-byte load and one store per slot and layer instead of two of each.  The
// records of (p, g) are decoded once into byte offsets and fp32 coefficient
// pairs, one per output, in the space of the consumed x tile.  The layers are
// separated by __syncthreads.  Every multiply, add, subtract and divide is a
// separately rounded IEEE operation (explicit .rn intrinsics), so results are
// bit-identical to an fp32 CPU evaluation in the same order.
//
// Decode band (M <= 16): 64 threads per token, thread t owns pair t of every
// layer and keeps its 8 records in registers; one CTA per (token block, group,
// partition), so at M = 1 the whole prologue is one short dependent chain.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pq_device.cuh"
#include "pq_internal.h"

namespace pq {
namespace {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
    float2 f;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(f.x), "=f"(f.y) : "r"(addr) : "memory");
    return f;
}
__device__ __forceinline__ void sts_f32x2(uint32_t addr, float2 f) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(f.x), "f"(f.y) : "memory");
}

// Many tokens: lane l holds tokens 2l and 2l+1 of the CTA's 64 (adjacent, so
// every shared-memory access moves both with one 8-byte instruction); warp w
// rotates pairs 8w..8w+7 of every layer.
constexpr int kTok = 64;              // tokens per CTA
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kPairsPerWarp = 64 / kWarps;     // pairs of a layer per warp
constexpr int kBatch = 4;                      // pairs loaded together before any store
constexpr int kChPerWarp = 128 / kWarps;       // channels per warp in the fill and the quantise
static_assert(kPairsPerWarp % kBatch == 0 && kChPerWarp % 16 == 0, "work split");
constexpr int kXsStride = 65;         // words per staged x row (64 + 1 pad)
constexpr int kCodeStride = 144;      // bytes per staged code row

// A decoded record: per slot the two outputs as coefficient pairs on the
// slot's two operands, out1 = fl(fl(x1 a) + fl(y1 b)), out2 = fl(fl(x2 a) +
// fl(y2 b)), and two byte offsets into v (see rotate_quant_kernel).
struct __align__(16) Smem {
    float2 v[128][kTok / 2];          // 32 KB, v[k][token pair]: (token 2l, token 2l+1)
    union {
        uint32_t xs[kTok][kXsStride]; // x tile, two bf16 per word (before the fill)
        struct {                      // the records of (p, g), during the layers
            float4 coef[8][64];       // (x1, y1, x2, y2)
            uint2 off[8][64];         // byte offsets of v rows
        } rec;
        struct {                      // after the layers
            uint8_t codes[kTok][kCodeStride];   // e4m3 codes
            float red_max[kWarps][kTok];        // per-warp amax
            int red_sum[kWarps][kTok];          // per-warp row-sums (x 2^9)
        };
    };
    float cs[128];
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float bf16_round(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

__device__ __forceinline__ uint32_t bf16_pack2(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

__device__ __forceinline__ float half_to_float(uint16_t h) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

// e4m3 encode of two values: hardware RNE convert with saturation to +-448,
// NaN -> 0x00 and any zero result (either sign) -> 0x00.  Returns
// (code(hi) << 8) | code(lo).
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    uint32_t c = r;
    if (hi != hi) c &= 0x00FFu;
    if (lo != lo) c &= 0xFF00u;
    if ((c & 0x7F00u) == 0) c &= 0x00FFu;
    if ((c & 0x007Fu) == 0) c &= 0xFF00u;
    return c;
}

// Correctly rounded a / b from y = RN(1/b) with multiply-adds only, after
// Markstein's theorem (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990): if q
// is within one ulp of a / b and y within half an ulp of 1 / b, then
// RN(q + (a - b q) y), with the residual exact in one fused multiply-add, is
// RN(a / b).  q0 = RN(a y) can be off by up to 1.5 ulp, so a first correction
// makes it faithful and a second one exact.  This holds while no step
// underflows or overflows: the callers keep b within [2^-60, 2^60]
// (quot_ok) and |a / b| <= 448; where |a / b| is below ~2^-100 the last bit
// may differ, and the e4m3 encoder maps every such value to 0 either way.
// Checked against IEEE division on 5 * 10^8 pairs including halfway cases.
// Used where one scale serves a whole CTA (the per-token pass C); in the
// per-group quantisers, where each lane has its own scale, the IEEE divide
// measured faster.
__device__ __forceinline__ bool quot_ok(float b) { return b >= 0x1p-60f && b <= 0x1p60f; }
__device__ __forceinline__ float quot_rn(float a, float b, float y) {
    const float q0 = __fmul_rn(a, y);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, b, a), y, q0);
    return __fmaf_rn(__fmaf_rn(-q1, b, a), y, q1);
}
// a / b rounded to nearest: quot_rn where it is exact, else the IEEE divide
__device__ __forceinline__ float div_scale(float a, float b, float y, bool ok) {
    return ok ? quot_rn(a, b, y) : __fdiv_rn(a, b);
}

// acc + the values of the four e4m3 codes of word w.  The hardware convert
// gives each value exactly in f16 (every e4m3 value is one), and the mixed
// f16 -> f32 multiply-add by 1 adds it exactly while the sum stays a multiple
// of 2^-9 below 2^14 (24 significant bits): so for up to 32 codes the result
// is the exact sum, whatever the order.
__device__ __forceinline__ float e4m3x4_accumulate(uint32_t w, float acc) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w >> 16)));
    asm("{\n.reg .f16 a0, a1, a2, a3, one;\n"
        "mov.b16 one, 0x3C00;\n"
        "mov.b32 {a0, a1}, %1;\n"
        "mov.b32 {a2, a3}, %2;\n"
        "fma.rn.f32.f16 %0, a0, one, %0;\n"
        "fma.rn.f32.f16 %0, a1, one, %0;\n"
        "fma.rn.f32.f16 %0, a2, one, %0;\n"
        "fma.rn.f32.f16 %0, a3, one, %0;\n}"
        : "+f"(acc)
        : "r"(h01), "r"(h23));
    return acc;
}

// dec(code) * 2^9 as an integer (exact; |value| <= 448 * 512)
__device__ __forceinline__ int e4m3_times512(uint32_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    const int mag = e == 0 ? m : ((8 | m) << (e - 1));
    return (c & 0x80) ? -mag : mag;
}

// One Givens pair, each product and sum rounded on its own:
//   vi' = fl(fl(c*vi) + fl(s*vj)),  vj' = fl(fl(c*vj) - fl(s*vi))
__device__ __forceinline__ void givens(float c, float s, float &vi, float &vj) {
    const float ni = __fadd_rn(__fmul_rn(c, vi), __fmul_rn(s, vj));
    const float nj = __fsub_rn(__fmul_rn(c, vj), __fmul_rn(s, vi));
    vi = ni;
    vj = nj;
}

// (fl(fl(x a.x) + fl(y b.x)), fl(fl(x a.y) + fl(y b.y))): one output of a
// Givens pair for two tokens, each product and the sum rounded on its own
__device__ __forceinline__ float2 rot2(float x, float y, float2 a, float2 b) {
    return make_float2(__fadd_rn(__fmul_rn(x, a.x), __fmul_rn(y, b.x)),
                       __fadd_rn(__fmul_rn(x, a.y), __fmul_rn(y, b.y)));
}

// kRot = false: the per-group quantisation (codes, asg, rs).
// kRot = true: pass A of the per-token path -- the rotated rows rounded to
// bf16 into xr [P][M][K] and each group's scale fl(max |xr| * fl(1/448)) into
// asg (the token-quant pass reads them back); a and rs are not touched.
template <bool kRot>
__global__ void __launch_bounds__(kThreads, 4)
rotate_quant_kernel(const uint16_t *__restrict__ x, int M, int K, int ldx, int P,
                    const uint2 *__restrict__ rec, const uint16_t *__restrict__ cs,
                    uint8_t *__restrict__ a, float *__restrict__ asg, float *__restrict__ rs,
                    uint16_t *__restrict__ xr) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m0 = blockIdx.x * kTok, g = blockIdx.y, G = K >> 7;
    const float inv448 = __fdiv_rn(1.0f, 448.0f);
    pdl_wait();        // x may be the previous kernel's output
    pdl_trigger();

    // x tile (64 rows of 256 bytes): issued together with the records and scales
    constexpr int kXv = kTok * 16 / kThreads;     // 16-byte pieces of the tile per thread
    uint4 xv[kXv];
#pragma unroll
    for (int it = 0; it < kXv; ++it) {
        const int c = tid + it * kThreads, row = c >> 4, q = c & 15;
        xv[it] = make_uint4(0, 0, 0, 0);
        if (m0 + row < M)
            xv[it] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(m0 + row) * ldx + 128 * g) + q);
    }

    {
        const int p = blockIdx.z;      // one partition per CTA: partitions run side by side
        constexpr int kRv = 256 / kThreads;           // 16-byte pieces of the 8 x 64 records
        uint4 rv[kRv];
#pragma unroll
        for (int it = 0; it < kRv; ++it) {
            const int c = tid + it * kThreads, r = c >> 5, q = c & 31;
            rv[it] = __ldg(reinterpret_cast<const uint4 *>(rec + ((size_t)(p * 8 + r) * G + g) * 64) + q);
        }
        const uint16_t csv = tid < 128 ? __ldg(cs + (size_t)p * K + 128 * g + tid) : (uint16_t)0;
#pragma unroll
        for (int it = 0; it < kXv; ++it) {
            const int c = tid + it * kThreads, row = c >> 4, q = c & 15;
            uint32_t *d = &sm.xs[row][4 * q];
            d[0] = xv[it].x; d[1] = xv[it].y; d[2] = xv[it].z; d[3] = xv[it].w;
        }
        if (tid < 128) sm.cs[tid] = half_to_float(csv);
        __syncthreads();

        // v[k][t] = x[t][k] * cs[k] (exact: bf16 x f16 fits in 24 bits)
#pragma unroll 4
        for (int q = 0; q < kChPerWarp / 2; ++q) {
            const int kw = (kChPerWarp / 2) * warp + q;   // word index: channels 2kw, 2kw+1
            const uint32_t w0 = sm.xs[2 * lane][kw], w1 = sm.xs[2 * lane + 1][kw];
            sm.v[2 * kw][lane] = make_float2(__fmul_rn(bf16lo(w0), sm.cs[2 * kw]),
                                             __fmul_rn(bf16lo(w1), sm.cs[2 * kw]));
            sm.v[2 * kw + 1][lane] = make_float2(__fmul_rn(bf16hi(w0), sm.cs[2 * kw + 1]),
                                                 __fmul_rn(bf16hi(w1), sm.cs[2 * kw + 1]));
        }
        __syncthreads();     // the x tile is consumed: its space takes the records

        // Records in chained order (pq_pack): slot t of a layer rotates the
        // pair (u, v); from layer 1 on, u is the channel slot t kept in
        // registers from the layer before.  Decoded per layer kind, with
        // u' = c u + s v -> (c, s) and v' = c v - s u -> (-s, c) on (u, v):
        //   layer 0:  operands (kept channel, other) both loaded: off = (kept,
        //             other); out1 is kept, out2 stored at the other;
        //   1..6:     operands (u held, v loaded from off.x); out1 is kept,
        //             out2 (the other channel's output) stored at off.y;
        //   7:        operands (u held, v from off.x); u' stored at off.y, v'
        //             at off.x.
        // The reversals are exact: fl(-s a) = -fl(s a) and x - y = x + (-y).
        // Channel bytes are masked to 0..127, so every offset stays in v.
#pragma unroll
        for (int it = 0; it < kRv; ++it) {
            const int c = tid + it * kThreads, r = c >> 5, q = c & 31;
            const uint32_t w0[2] = {rv[it].x, rv[it].z}, w1[2] = {rv[it].y, rv[it].w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t u = (w0[h] & 0x7F) * (uint32_t)(kTok * 4);
                const uint32_t v = ((w0[h] >> 8) & 0x7F) * (uint32_t)(kTok * 4);
                const bool keep_v = (w0[h] >> 16) & 1;
                const float cc = half_to_float((uint16_t)(w1[h] & 0xFFFFu));
                const float ss = half_to_float((uint16_t)(w1[h] >> 16));
                float4 cf;
                uint2 of;
                if (r == 0) {
                    of = keep_v ? make_uint2(v, u) : make_uint2(u, v);
                    cf = keep_v ? make_float4(cc, -ss, ss, cc) : make_float4(cc, ss, -ss, cc);
                } else if (r < 7) {
                    of = make_uint2(v, keep_v ? u : v);
                    cf = keep_v ? make_float4(-ss, cc, cc, ss) : make_float4(cc, ss, -ss, cc);
                } else {
                    of = make_uint2(v, u);
                    cf = make_float4(cc, ss, -ss, cc);
                }
                sm.rec.coef[r][2 * q + h] = cf;
                sm.rec.off[r][2 * q + h] = of;
            }
        }
        __syncthreads();

        // eight Givens layers.  Warp w owns slots 8w..8w+7 of every layer and
        // keeps one value per slot (for both tokens of the lane) in kv; the
        // pairs of one layer are disjoint, so a warp reads all operands of a
        // batch of slots before writing any result.
        const uint32_t vlane = smem_addr(&sm.v[0][lane]);
        const int s0 = kPairsPerWarp * warp;
        float2 kv[kPairsPerWarp];
#pragma unroll
        for (int half = 0; half < kPairsPerWarp / kBatch; ++half) {
            float2 va[kBatch], vb[kBatch];
            float4 cf[kBatch];
            uint32_t ob[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const uint2 o = sm.rec.off[0][s0 + kBatch * half + q];
                cf[q] = sm.rec.coef[0][s0 + kBatch * half + q];
                ob[q] = vlane + o.y;
                va[q] = lds_f32x2(vlane + o.x);
                vb[q] = lds_f32x2(ob[q]);
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                kv[kBatch * half + q] = rot2(cf[q].x, cf[q].y, va[q], vb[q]);
                sts_f32x2(ob[q], rot2(cf[q].z, cf[q].w, va[q], vb[q]));
            }
        }
        __syncthreads();
        for (int r = 1; r < 7; ++r) {
#pragma unroll
            for (int half = 0; half < kPairsPerWarp / kBatch; ++half) {
                float2 vb[kBatch];
                float4 cf[kBatch];
                uint32_t os[kBatch];
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const uint2 o = sm.rec.off[r][s0 + kBatch * half + q];
                    cf[q] = sm.rec.coef[r][s0 + kBatch * half + q];
                    os[q] = vlane + o.y;
                    vb[q] = lds_f32x2(vlane + o.x);
                }
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const float2 va = kv[kBatch * half + q];
                    kv[kBatch * half + q] = rot2(cf[q].x, cf[q].y, va, vb[q]);
                    sts_f32x2(os[q], rot2(cf[q].z, cf[q].w, va, vb[q]));
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int half = 0; half < kPairsPerWarp / kBatch; ++half) {
            float2 vb[kBatch];
            float4 cf[kBatch];
            uint32_t oa[kBatch], os[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const uint2 o = sm.rec.off[7][s0 + kBatch * half + q];
                cf[q] = sm.rec.coef[7][s0 + kBatch * half + q];
                oa[q] = vlane + o.x;
                os[q] = vlane + o.y;
                vb[q] = lds_f32x2(oa[q]);
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const float2 va = kv[kBatch * half + q];
                sts_f32x2(os[q], rot2(cf[q].x, cf[q].y, va, vb[q]));
                sts_f32x2(oa[q], rot2(cf[q].z, cf[q].w, va, vb[q]));
            }
        }
        __syncthreads();

        // quantise: warp w takes channels kChPerWarp w .. + kChPerWarp - 1 of
        // both tokens of the lane
        constexpr int kC = kChPerWarp;
        float2 vals[kC];
        float amax0 = 0.0f, amax1 = 0.0f;
        if constexpr (kRot) {
            // bf16 rows straight to xr (64 contiguous bytes per token and
            // warp); amax over the rounded values
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                uint32_t pk[kC / 2];
                float am = 0.0f;
#pragma unroll
                for (int q = 0; q < kC / 2; ++q) {
                    const float2 lo = sm.v[kC * warp + 2 * q][lane], hi = sm.v[kC * warp + 2 * q + 1][lane];
                    pk[q] = bf16_pack2(t ? lo.y : lo.x, t ? hi.y : hi.x);
                    am = fmaxf(am, fmaxf(fabsf(bf16lo(pk[q])), fabsf(bf16hi(pk[q]))));
                }
                const int tok = 2 * lane + t;
                sm.red_max[warp][tok] = am;
                if (m0 + tok < M) {
                    uint4 *dst = reinterpret_cast<uint4 *>(xr + ((size_t)p * M + m0 + tok) * K + 128 * g + kC * warp);
#pragma unroll
                    for (int q = 0; q < kC / 8; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            __syncthreads();
            if (tid < kTok && m0 + tid < M) {
                float amax = sm.red_max[0][tid];
#pragma unroll
                for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, sm.red_max[w][tid]);
                asg[((size_t)p * G + g) * M + m0 + tid] = __fmul_rn(amax, inv448);
            }
        } else {
#pragma unroll
            for (int q = 0; q < kC; ++q) {
                vals[q] = sm.v[kC * warp + q][lane];
                amax0 = fmaxf(amax0, fabsf(vals[q].x));
                amax1 = fmaxf(amax1, fabsf(vals[q].y));
            }
            sm.red_max[warp][2 * lane] = amax0;
            sm.red_max[warp][2 * lane + 1] = amax1;
            __syncthreads();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int tok = 2 * lane + t;
                float amax = sm.red_max[0][tok];
#pragma unroll
                for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, sm.red_max[w][tok]);
                const float scale = __fmul_rn(amax, inv448);
                uint32_t packed[kC / 4];
                float vsum = 0.0f;     // exact: kC codes
#pragma unroll
                for (int q = 0; q < kC / 4; ++q) {
                    uint32_t word = 0;
                    if (scale != 0.0f) {
                        const float e0 = t ? vals[4 * q].y : vals[4 * q].x, e1 = t ? vals[4 * q + 1].y : vals[4 * q + 1].x;
                        const float e2 = t ? vals[4 * q + 2].y : vals[4 * q + 2].x, e3 = t ? vals[4 * q + 3].y : vals[4 * q + 3].x;
                        const uint32_t c01 = e4m3x2(__fdiv_rn(e1, scale), __fdiv_rn(e0, scale));
                        const uint32_t c23 = e4m3x2(__fdiv_rn(e3, scale), __fdiv_rn(e2, scale));
                        word = c01 | (c23 << 16);
                    }
                    packed[q] = word;
                    vsum = e4m3x4_accumulate(word, vsum);
                }
                const int sum512 = __float2int_rn(__fmul_rn(vsum, 512.0f));
                uint4 *cdst = reinterpret_cast<uint4 *>(&sm.codes[tok][kC * warp]);
#pragma unroll
                for (int q = 0; q < kC / 16; ++q)
                    cdst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                sm.red_sum[warp][tok] = sum512;
                if (warp == 0 && m0 + tok < M) asg[((size_t)p * G + g) * M + m0 + tok] = scale;
            }
            __syncthreads();

            // stores: 128-byte code rows, then one row-sum per token
            for (int c = tid; c < kTok * 8; c += kThreads) {
                const int row = c >> 3, q = c & 7;
                if (m0 + row < M)
                    reinterpret_cast<uint4 *>(a + ((size_t)p * M + m0 + row) * K + 128 * g)[q] =
                        *reinterpret_cast<const uint4 *>(&sm.codes[row][16 * q]);
            }
            if (tid < kTok && m0 + tid < M) {
                const size_t o = ((size_t)p * G + g) * M + m0 + tid;
                int s = 0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) s += sm.red_sum[w][tid];
                rs[o] = __fmul_rn(__int2float_rn(s), 1.0f / 512.0f);
            }
        }  // !kRot
    }
}

// The decode-band tail shared by the small kernels: token tt's 128 scaled
// values of group g are in v[tt] (written by all 64 threads of the token, then
// __syncthreads); eight Givens layers through shared memory, amax, the e4m3
// codes and the exact row-sum, stored for partition p.
template <int T>
__device__ __forceinline__ void small_rotate_quant_tail(float (&v)[T][128], float (&red_max)[T][2],
                                                        int (&red_sum)[T][2], const uint2 (&r8)[8], int tt,
                                                        int t, int lane, int half, int m, int g, int p,
                                                        int M, int K, bool live, uint8_t *__restrict__ a,
                                                        float *__restrict__ asg, float *__restrict__ rs) {
    const int G = K >> 7;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = r8[r].x & 0xFF, j = (r8[r].x >> 8) & 0xFF;
        float vi = v[tt][i], vj = v[tt][j];
        givens(half_to_float((uint16_t)(r8[r].y & 0xFFFF)), half_to_float((uint16_t)(r8[r].y >> 16)),
               vi, vj);
        v[tt][i] = vi;
        v[tt][j] = vj;
        __syncthreads();
    }
    const float e0 = v[tt][2 * t], e1 = v[tt][2 * t + 1];
    float amax = fmaxf(fabsf(e0), fabsf(e1));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) red_max[tt][half] = amax;
    __syncthreads();
    amax = fmaxf(red_max[tt][0], red_max[tt][1]);
    const float scale = __fmul_rn(amax, __fdiv_rn(1.0f, 448.0f));
    uint32_t c2 = 0;
    if (scale != 0.0f) c2 = e4m3x2(__fdiv_rn(e1, scale), __fdiv_rn(e0, scale));
    int sum512 = e4m3_times512(c2 & 0xFF) + e4m3_times512(c2 >> 8);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum512 += __shfl_xor_sync(0xFFFFFFFFu, sum512, o);
    if (lane == 0) red_sum[tt][half] = sum512;
    __syncthreads();
    if (live) {
        reinterpret_cast<uint16_t *>(a + ((size_t)p * M + m) * K + 128 * g)[t] = (uint16_t)c2;
        if (t == 0) {
            const size_t o = ((size_t)p * G + g) * M + m;
            asg[o] = scale;
            rs[o] = __fmul_rn(__int2float_rn(red_sum[tt][0] + red_sum[tt][1]), 1.0f / 512.0f);
        }
    }
}

template <int T>
__global__ void __launch_bounds__(64 * T)
rotate_quant_small_kernel(const uint16_t *__restrict__ x, int M, int K, int ldx,
                          const uint2 *__restrict__ rec, const uint16_t *__restrict__ cs,
                          uint8_t *__restrict__ a, float *__restrict__ asg, float *__restrict__ rs) {
    __shared__ float v[T][128];
    __shared__ float red_max[T][2];
    __shared__ int red_sum[T][2];
    const int tid = threadIdx.x, tt = tid >> 6, t = tid & 63, lane = tid & 31, half = (tid >> 5) & 1;
    const int m = blockIdx.x * T + tt, g = blockIdx.y, p = blockIdx.z, G = K >> 7;
    const bool live = m < M;
    pdl_trigger();

    // the load-time tables first (channel-scale pair, the 8 records of pair t):
    // they are read while the preceding kernel may still be running
    const uint32_t cw = __ldg(reinterpret_cast<const uint32_t *>(cs + (size_t)p * K + 128 * g) + t);
    uint2 r8[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) r8[r] = __ldg(rec + ((size_t)(p * 8 + r) * G + g) * 64 + t);
    pdl_wait();        // x may be the previous kernel's output; a, asg, rs may still be read by it
    const uint32_t xw = live ? __ldg(reinterpret_cast<const uint32_t *>(x + (size_t)m * ldx + 128 * g) + t) : 0u;

    v[tt][2 * t] = __fmul_rn(bf16lo(xw), half_to_float((uint16_t)(cw & 0xFFFF)));
    v[tt][2 * t + 1] = __fmul_rn(bf16hi(xw), half_to_float((uint16_t)(cw >> 16)));
    __syncthreads();
    small_rotate_quant_tail<T>(v, red_max, red_sum, r8, tt, t, lane, half, m, g, p, M, K, live, a, asg, rs);
}

// ---------------------------------------------------------------------------
// Fused producer: residual add + Gemma RMSNorm + channel scale + rotation +
// per-group quant ("2026-09-02/03: rotation stream (fused add + RMSNorm +
// rotate + quant producers)").  Per row:
//   s = bf16(x + r)  (the new residual);  ss = sum of s^2 (order below);
//   inv = 1 / sqrt(ss / K + eps)  (correctly rounded sqrt and division);
//   h = bf16((s * inv) * (1 + gamma));  then the pq_rotate_quant steps on h.
// Order of ss: thread t of a row's 64 holds channels 2t, 2t+1 of each
// 128-group and sums fl(s^2 + s'^2) over the groups in order (its lane sum);
// the 64 lane sums are added pairwise by recursive halving: the xor tree over
// each warp, then warp 0's + warp 1's.
// ---------------------------------------------------------------------------

// s of the two channels of a lane, from the x and residual words
__device__ __forceinline__ float2 residual_add(uint32_t xw, uint32_t rw) {
    return make_float2(bf16_round(__fadd_rn(bf16lo(xw), bf16lo(rw))),
                       bf16_round(__fadd_rn(bf16hi(xw), bf16hi(rw))));
}

// This lane's sum over the groups, in order, of fl(s^2 + s'^2) for its
// channel pair, with x and residual words read through rd(gg) -> (xw, rw).
template <class Read>
__device__ __forceinline__ float lane_sumsq(int G, Read rd) {
    float acc = 0.0f;
    int gg = 0;
    for (; gg + 8 <= G; gg += 8) {
        uint2 w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = rd(gg + j);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 s = residual_add(w[j].x, w[j].y);
            acc = __fadd_rn(acc, __fadd_rn(__fmul_rn(s.x, s.x), __fmul_rn(s.y, s.y)));
        }
    }
    for (; gg < G; ++gg) {
        const uint2 w = rd(gg);
        const float2 s = residual_add(w.x, w.y);
        acc = __fadd_rn(acc, __fadd_rn(__fmul_rn(s.x, s.x), __fmul_rn(s.y, s.y)));
    }
    return acc;
}

// The pairwise sum of the row's 64 lane sums: the xor tree over the warp
// (every lane ends with the warp's sum), written to wsum[half]; after a
// __syncthreads, row_inv_rms adds warp 0's and warp 1's.
__device__ __forceinline__ void warp_pairwise(float acc, int lane, int half, float *wsum) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
    if (lane == 0) wsum[half] = acc;
}

// 1 / sqrt(ss / K + eps) from the two warps' sums
__device__ __forceinline__ float row_inv_rms(const float *wsum, int K, float eps) {
    const float ss = __fadd_rn(wsum[0], wsum[1]);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps)));
}

// 16-byte asynchronous global -> shared copy, zero-filled when !valid (the
// source is then not read)
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

// Decode band: one CTA per (token block, group, partition) as the small
// kernel, each recomputing the whole row's norm (the row is read from L2);
// partition 0 writes the new residual and h of its group.
template <int T>
__global__ void __launch_bounds__(64 * T)
add_rms_rotate_quant_small_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ res, int M,
                                  int K, int ldx, const uint16_t *__restrict__ gamma, float eps,
                                  const uint2 *__restrict__ rec, const uint16_t *__restrict__ cs,
                                  uint16_t *__restrict__ res_out, uint16_t *__restrict__ h_out,
                                  uint8_t *__restrict__ a, float *__restrict__ asg, float *__restrict__ rs) {
    // dynamic shared memory: each token's x row and residual row [T][2][K]
    // (bf16), staged with one wave of copies
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ float v[T][128];
    __shared__ float red_max[T][2];
    __shared__ int red_sum[T][2];
    __shared__ float wsum[T][2];
    const int tid = threadIdx.x, tt = tid >> 6, t = tid & 63, lane = tid & 31, half = (tid >> 5) & 1;
    const int m = blockIdx.x * T + tt, g = blockIdx.y, p = blockIdx.z, G = K >> 7;
    const bool live = m < M;
    uint16_t *rows = reinterpret_cast<uint16_t *>(dsm);
    pdl_trigger();

    // load-time tables first: channel scales, records, Gemma weights
    const uint32_t cw = __ldg(reinterpret_cast<const uint32_t *>(cs + (size_t)p * K + 128 * g) + t);
    const uint32_t gw = __ldg(reinterpret_cast<const uint32_t *>(gamma + 128 * g) + t);
    uint2 r8[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) r8[r] = __ldg(rec + ((size_t)(p * 8 + r) * G + g) * 64 + t);
    pdl_wait();        // x and res may be the previous kernel's output

    uint16_t *xs = rows + (size_t)tt * 2 * K, *rsm = xs + K;
    {
        const uint16_t *xrow = x + (size_t)m * ldx, *rrow = res + (size_t)m * ldx;
        for (int c = t; c < K / 8; c += 64) {      // 16-byte chunks of 8 values
            cp_async16(xs + 8 * c, live ? xrow + 8 * c : x, live);
            cp_async16(rsm + 8 * c, live ? rrow + 8 * c : res, live);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncthreads();
    const uint32_t *xs32 = reinterpret_cast<const uint32_t *>(xs), *rs32 = reinterpret_cast<const uint32_t *>(rsm);
    warp_pairwise(lane_sumsq(G, [&](int gg) { return make_uint2(xs32[64 * gg + t], rs32[64 * gg + t]); }), lane,
                  half, wsum[tt]);
    const uint32_t xk = xs32[64 * g + t], rk = rs32[64 * g + t];
    __syncthreads();
    const float inv = row_inv_rms(wsum[tt], K, eps);
    const float2 s = residual_add(xk, rk);
    const float h0 = bf16_round(__fmul_rn(__fmul_rn(s.x, inv), __fadd_rn(1.0f, bf16lo(gw))));
    const float h1 = bf16_round(__fmul_rn(__fmul_rn(s.y, inv), __fadd_rn(1.0f, bf16hi(gw))));
    if (live && p == 0) {
        reinterpret_cast<uint32_t *>(res_out + (size_t)m * K + 128 * g)[t] = bf16_pack2(s.x, s.y);
        reinterpret_cast<uint32_t *>(h_out + (size_t)m * K + 128 * g)[t] = bf16_pack2(h0, h1);
    }
    v[tt][2 * t] = __fmul_rn(h0, half_to_float((uint16_t)(cw & 0xFFFF)));
    v[tt][2 * t + 1] = __fmul_rn(h1, half_to_float((uint16_t)(cw >> 16)));
    __syncthreads();
    small_rotate_quant_tail<T>(v, red_max, red_sum, r8, tt, t, lane, half, m, g, p, M, K, live, a, asg, rs);
}

// Above the decode band: the norm alone, four rows per CTA (64 threads per
// row), writing the new residual and h; pq_rotate_quant's kernel follows.
__global__ void __launch_bounds__(256)
add_rms_norm_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ res, int M, int K, int ldx,
                    const uint16_t *__restrict__ gamma, float eps, uint16_t *__restrict__ res_out,
                    uint16_t *__restrict__ h_out) {
    __shared__ float wsum[4][2];
    const int tid = threadIdx.x, tt = tid >> 6, t = tid & 63, lane = tid & 31, half = (tid >> 5) & 1;
    const int m = blockIdx.x * 4 + tt, G = K >> 7;
    const bool live = m < M;
    pdl_wait();        // x and res may be the previous kernel's output
    pdl_trigger();
    const uint16_t *xrow = x + (size_t)m * ldx, *rrow = res + (size_t)m * ldx;
    const uint32_t *x32 = reinterpret_cast<const uint32_t *>(xrow), *r32 = reinterpret_cast<const uint32_t *>(rrow);
    warp_pairwise(lane_sumsq(G, [&](int gg) {
                      return live ? make_uint2(__ldg(x32 + 64 * gg + t), __ldg(r32 + 64 * gg + t)) : make_uint2(0u, 0u);
                  }),
                  lane, half, wsum[tt]);
    __syncthreads();
    if (!live) return;
    const float inv = row_inv_rms(wsum[tt], K, eps);
    for (int gg = 0; gg < G; ++gg) {
        const float2 s = residual_add(__ldg(reinterpret_cast<const uint32_t *>(xrow + 128 * gg) + t),
                                      __ldg(reinterpret_cast<const uint32_t *>(rrow + 128 * gg) + t));
        const uint32_t gw = __ldg(reinterpret_cast<const uint32_t *>(gamma + 128 * gg) + t);
        const float h0 = __fmul_rn(__fmul_rn(s.x, inv), __fadd_rn(1.0f, bf16lo(gw)));
        const float h1 = __fmul_rn(__fmul_rn(s.y, inv), __fadd_rn(1.0f, bf16hi(gw)));
        reinterpret_cast<uint32_t *>(res_out + (size_t)m * K + 128 * gg)[t] = bf16_pack2(s.x, s.y);
        reinterpret_cast<uint32_t *>(h_out + (size_t)m * K + 128 * gg)[t] = bf16_pack2(h0, h1);
    }
}

// ---------------------------------------------------------------------------
// silu-mul producer ("2026-09-03: rotation stream 2 (silu-mul, GDN gated norm,
// attention gate fused with rotate+quant)", its first mode): the merged gate/up
// output y holds g in columns [0, I) and u in [I, 2I);
//   act = bf16(bf16(g / (1 + exp(-g))) * u),  then the pq_rotate_quant steps
// on act (K = I).  exp is the fixed sequence below, so the result is the
// same bits on any IEEE fp32 machine that follows it.
// ---------------------------------------------------------------------------

// exp(x) in fp32: Cody-Waite reduction n = rint(x log2 e),
// r = (x - n ln2_hi) - n ln2_lo (ln2_hi has 13 trailing zero bits, so n ln2_hi
// is exact), the degree-6 Taylor polynomial of exp in Horner form and an
// exact scaling by 2^n; x > 88 gives +inf and x < -103 gives 0.  Every step
// is a separately rounded IEEE operation.
__device__ __forceinline__ float exp32_fixed(float x) {
    if (x > 88.0f) return __int_as_float(0x7F800000);
    if (x < -103.0f) return 0.0f;
    const float n = rintf(__fmul_rn(x, 1.44269502f));
    const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, 0.693145751953125f)), __fmul_rn(n, 1.42860677e-06f));
    float q = __fmul_rn(r, 1.0f / 720.0f);
    q = __fmul_rn(r, __fadd_rn(1.0f / 120.0f, q));
    q = __fmul_rn(r, __fadd_rn(1.0f / 24.0f, q));
    q = __fmul_rn(r, __fadd_rn(1.0f / 6.0f, q));
    q = __fmul_rn(r, __fadd_rn(0.5f, q));
    q = __fmul_rn(r, __fadd_rn(1.0f, q));
    q = __fadd_rn(1.0f, q);
    return ldexpf(q, (int)n);
}

__device__ __forceinline__ float silu_mul1(float g, float u) {
    const float sg = bf16_round(__fdiv_rn(g, __fadd_rn(1.0f, exp32_fixed(-g))));
    return bf16_round(__fmul_rn(sg, u));
}

// Decode band: the small prologue's grid; partition 0 also writes act.
template <int T>
__global__ void __launch_bounds__(64 * T)
silu_mul_rotate_quant_small_kernel(const uint16_t *__restrict__ y, int M, int I, int ldy,
                                   const uint2 *__restrict__ rec, const uint16_t *__restrict__ cs,
                                   uint16_t *__restrict__ act_out, uint8_t *__restrict__ a,
                                   float *__restrict__ asg, float *__restrict__ rs) {
    __shared__ float v[T][128];
    __shared__ float red_max[T][2];
    __shared__ int red_sum[T][2];
    const int tid = threadIdx.x, tt = tid >> 6, t = tid & 63, lane = tid & 31, half = (tid >> 5) & 1;
    const int m = blockIdx.x * T + tt, g = blockIdx.y, p = blockIdx.z, G = I >> 7;
    const bool live = m < M;
    pdl_trigger();
    const uint32_t cw = __ldg(reinterpret_cast<const uint32_t *>(cs + (size_t)p * I + 128 * g) + t);
    uint2 r8[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) r8[r] = __ldg(rec + ((size_t)(p * 8 + r) * G + g) * 64 + t);
    pdl_wait();        // y may be the previous kernel's output
    const uint16_t *yrow = y + (size_t)m * ldy;
    const uint32_t gw = live ? __ldg(reinterpret_cast<const uint32_t *>(yrow + 128 * g) + t) : 0u;
    const uint32_t uw = live ? __ldg(reinterpret_cast<const uint32_t *>(yrow + I + 128 * g) + t) : 0u;
    const float a0 = silu_mul1(bf16lo(gw), bf16lo(uw)), a1 = silu_mul1(bf16hi(gw), bf16hi(uw));
    if (live && p == 0) reinterpret_cast<uint32_t *>(act_out + (size_t)m * I + 128 * g)[t] = bf16_pack2(a0, a1);
    v[tt][2 * t] = __fmul_rn(a0, half_to_float((uint16_t)(cw & 0xFFFF)));
    v[tt][2 * t + 1] = __fmul_rn(a1, half_to_float((uint16_t)(cw >> 16)));
    __syncthreads();
    small_rotate_quant_tail<T>(v, red_max, red_sum, r8, tt, t, lane, half, m, g, p, M, I, live, a, asg, rs);
}

// Above the band: act elementwise, two channels per thread; blockIdx.x
// walks a row's channel pairs, blockIdx.y the rows.  pq_rotate_quant's
// kernel on act follows.
__global__ void __launch_bounds__(256)
silu_mul_kernel(const uint16_t *__restrict__ y, int M, int I, int ldy, uint16_t *__restrict__ act_out) {
    pdl_wait();        // y may be the previous kernel's output
    pdl_trigger();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;   // channel pair
    if (c >= I / 2) return;
    for (int m = blockIdx.y; m < M; m += gridDim.y) {
        const uint16_t *yrow = y + (size_t)m * ldy;
        const uint32_t gw = __ldg(reinterpret_cast<const uint32_t *>(yrow) + c);
        const uint32_t uw = __ldg(reinterpret_cast<const uint32_t *>(yrow + I) + c);
        reinterpret_cast<uint32_t *>(act_out + (size_t)m * I)[c] =
            bf16_pack2(silu_mul1(bf16lo(gw), bf16lo(uw)), silu_mul1(bf16hi(gw), bf16hi(uw)));
    }
}

__global__ void e4m3_encode_kernel(const float *__restrict__ in, uint8_t *__restrict__ out,
                                   size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x * 2;
    for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 2; i < n; i += stride) {
        const float lo = in[i];
        const float hi = (i + 1 < n) ? in[i + 1] : 0.0f;
        const uint32_t c = e4m3x2(hi, lo);
        out[i] = (uint8_t)(c & 0xFF);
        if (i + 1 < n) out[i + 1] = (uint8_t)(c >> 8);
    }
}

// ---------------------------------------------------------------------------
// Pass C of the per-token path ("Numbers", the per-token prefill item, pass
// C): for every row, As = max over the groups of pass A's group scales,
// a = e4m3(fl(xr / As)) (all 0 when As = 0), and per group the exact sum of
// what the codes decode to (plain row-sums: the token scale is applied in the
// GEMM's epilogue).  One CTA of 128 threads per (row, partition): thread t
// takes the 8 channels of chunk c8 = c0 + t, so the 16 lanes of a half-warp
// hold one group.  gsc and rs may be the same buffer: the CTA reads all of its
// row's group scales before the barrier and writes the row-sums after it, and
// no other CTA touches the row.
// ---------------------------------------------------------------------------
constexpr int kTqThreads = 128;

__device__ __forceinline__ uint32_t e4m3x4_scaled(uint2 w, float as, float rcp, bool ok) {
    return e4m3x2(div_scale(bf16hi(w.x), as, rcp, ok), div_scale(bf16lo(w.x), as, rcp, ok)) |
           (e4m3x2(div_scale(bf16hi(w.y), as, rcp, ok), div_scale(bf16lo(w.y), as, rcp, ok)) << 16);
}

__global__ void __launch_bounds__(kTqThreads)
token_quant_kernel(const uint16_t *__restrict__ xr, int M, int K, const float *gsc, uint8_t *__restrict__ a,
                   float *__restrict__ As, float *rs) {
    __shared__ float wmax[kTqThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int m = blockIdx.x, p = blockIdx.y, G = K >> 7;
    pdl_wait();        // xr and the group scales are the preceding pass's output
    pdl_trigger();
    float as = 0.0f;
    for (int g = t; g < G; g += kTqThreads) as = fmaxf(as, gsc[((size_t)p * G + g) * M + m]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) as = fmaxf(as, __shfl_xor_sync(0xFFFFFFFFu, as, o));
    if (lane == 0) wmax[warp] = as;
    __syncthreads();   // every group scale of the row has been read
    as = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    if (t == 0) As[(size_t)p * M + m] = as;
    const bool ok = quot_ok(as);
    const float rcp = __frcp_rn(as);
    const uint16_t *row = xr + ((size_t)p * M + m) * K;
    uint8_t *arow = a + ((size_t)p * M + m) * K;
    for (int c0 = 0; c0 < 16 * G; c0 += kTqThreads) {
        const int c8 = c0 + t, g = c8 >> 4;
        const bool valid = c8 < 16 * G;
        int sum512 = 0;
        if (valid) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row) + c8);
            uint32_t lo = 0, hi = 0;
            if (as != 0.0f) {
                lo = e4m3x4_scaled(make_uint2(v.x, v.y), as, rcp, ok);
                hi = e4m3x4_scaled(make_uint2(v.z, v.w), as, rcp, ok);
            }
            reinterpret_cast<uint2 *>(arow)[c8] = make_uint2(lo, hi);
            sum512 = __float2int_rn(__fmul_rn(e4m3x4_accumulate(hi, e4m3x4_accumulate(lo, 0.0f)), 512.0f));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sum512 += __shfl_xor_sync(0xFFFFFFFFu, sum512, o);
        if ((lane & 15) == 0 && valid) rs[((size_t)p * G + g) * M + m] = __fmul_rn(__int2float_rn(sum512), 1.0f / 512.0f);
    }
}

}  // namespace

pq_status launch_rotate_quant(const void *x, int M, int K, int ldx, int P, const void *rec,
                              const void *cs, void *a, float *asg, float *rs, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    const uint2 *rp = static_cast<const uint2 *>(rec);
    const uint16_t *cp = static_cast<const uint16_t *>(cs);
    uint8_t *ap = static_cast<uint8_t *>(a);
    if (K / 128 > 65535) return fail(PQ_ERR_SHAPE, "pq_rotate_quant: K = %d too large", K);
    cudaError_t e;
    if (M <= 16) {
        // decode band: 64 threads per token, partitions in parallel
        if (M == 1)
            e = launch_pdl(rotate_quant_small_kernel<1>, dim3(1, K / 128, P), dim3(64), 0, st, xp, M, K, ldx,
                           rp, cp, ap, asg, rs);
        else if (M == 2)
            e = launch_pdl(rotate_quant_small_kernel<2>, dim3(1, K / 128, P), dim3(128), 0, st, xp, M, K,
                           ldx, rp, cp, ap, asg, rs);
        else
            e = launch_pdl(rotate_quant_small_kernel<4>, dim3((M + 3) / 4, K / 128, P), dim3(256), 0, st, xp,
                           M, K, ldx, rp, cp, ap, asg, rs);
    } else {
        const dim3 grid((M + kTok - 1) / kTok, K / 128, P);
        if (grid.x > 0x7FFFFFFF) return fail(PQ_ERR_SHAPE, "pq_rotate_quant: M = %d too large", M);
        e = cudaFuncSetAttribute(rotate_quant_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(Smem));
        if (e == cudaSuccess)
            e = launch_pdl(rotate_quant_kernel<false>, grid, dim3(kThreads), sizeof(Smem), st, xp, M, K, ldx, P,
                           rp, cp, ap, asg, rs, (uint16_t *)nullptr);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "rotate_quant launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

pq_status launch_rotate_tokquant(const void *x, int M, int K, int ldx, int P, const void *rec, const void *cs,
                                 void *xr, void *a, float *As, float *rs, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint16_t *xrp = static_cast<uint16_t *>(xr);
    if (K / 128 > 65535) return fail(PQ_ERR_SHAPE, "pq_rotate_tokquant: K = %d too large", K);
    // pass A: rotation into xr, group scales into rs
    const dim3 grid((M + kTok - 1) / kTok, K / 128, P);
    cudaError_t e = cudaFuncSetAttribute(rotate_quant_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(Smem));
    if (e == cudaSuccess)
        e = launch_pdl(rotate_quant_kernel<true>, grid, dim3(kThreads), sizeof(Smem), st,
                       static_cast<const uint16_t *>(x), M, K, ldx, P, static_cast<const uint2 *>(rec),
                       static_cast<const uint16_t *>(cs), (uint8_t *)nullptr, rs, (float *)nullptr, xrp);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "rotate_tokquant pass A launch: %s", cudaGetErrorString(e));
    // pass C: token scale, codes, row-sums
    e = launch_pdl(token_quant_kernel, dim3(M, P), dim3(kTqThreads), 0, st,
                   (const uint16_t *)xrp, M, K, (const float *)rs, static_cast<uint8_t *>(a), As, rs);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "rotate_tokquant pass C launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

pq_status launch_add_rms_rotate_quant(const void *x, const void *res, const void *gamma, float eps, int M,
                                      int K, int ldx, int P, const void *rec, const void *cs, void *res_out,
                                      void *h, void *a, float *asg, float *rs, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t *xp = static_cast<const uint16_t *>(x), *rp = static_cast<const uint16_t *>(res);
    const uint16_t *gp = static_cast<const uint16_t *>(gamma), *cp = static_cast<const uint16_t *>(cs);
    const uint2 *recp = static_cast<const uint2 *>(rec);
    uint16_t *rop = static_cast<uint16_t *>(res_out), *hp = static_cast<uint16_t *>(h);
    uint8_t *ap = static_cast<uint8_t *>(a);
    const int G = K / 128;
    if (G > 65535) return fail(PQ_ERR_SHAPE, "pq_add_rms_rotate_quant: K = %d too large", K);
    cudaError_t e;
    const int Tsmall = M == 1 ? 1 : (M == 2 ? 2 : 4);
    const size_t small_smem = (size_t)Tsmall * 2 * K * 2;
    if (M <= 16 && small_smem <= 160 * 1024) {
        // decode band: one fused launch
        const int T = M == 1 ? 1 : (M == 2 ? 2 : 4);
        const size_t smem = (size_t)T * 2 * K * 2;
        const dim3 grid((M + T - 1) / T, G, P), block(64 * T);
        if (T == 1) {
            e = cudaFuncSetAttribute(add_rms_rotate_quant_small_kernel<1>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e == cudaSuccess)
                e = launch_pdl(add_rms_rotate_quant_small_kernel<1>, grid, block, smem, st, xp, rp, M, K, ldx, gp,
                               eps, recp, cp, rop, hp, ap, asg, rs);
        } else if (T == 2) {
            e = cudaFuncSetAttribute(add_rms_rotate_quant_small_kernel<2>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e == cudaSuccess)
                e = launch_pdl(add_rms_rotate_quant_small_kernel<2>, grid, block, smem, st, xp, rp, M, K, ldx, gp,
                               eps, recp, cp, rop, hp, ap, asg, rs);
        } else {
            e = cudaFuncSetAttribute(add_rms_rotate_quant_small_kernel<4>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e == cudaSuccess)
                e = launch_pdl(add_rms_rotate_quant_small_kernel<4>, grid, block, smem, st, xp, rp, M, K, ldx, gp,
                               eps, recp, cp, rop, hp, ap, asg, rs);
        }
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "add_rms_rotate_quant launch: %s", cudaGetErrorString(e));
        return PQ_OK;
    }
    // above it: the norm, then the prologue on h (chained by programmatic
    // dependent launch; the prologue waits for the norm before reading h)
    e = launch_pdl(add_rms_norm_kernel, dim3((M + 3) / 4), dim3(256), 0, st, xp, rp, M, K, ldx, gp, eps, rop, hp);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "add_rms_norm launch: %s", cudaGetErrorString(e));
    return launch_rotate_quant(h, M, K, K, P, rec, cs, a, asg, rs, stream);
}

pq_status launch_silu_mul_rotate_quant(const void *y, int M, int I, int ldy, int P, const void *rec,
                                       const void *cs, void *act, void *a, float *asg, float *rs,
                                       void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t *yp = static_cast<const uint16_t *>(y), *cp = static_cast<const uint16_t *>(cs);
    const uint2 *recp = static_cast<const uint2 *>(rec);
    uint16_t *actp = static_cast<uint16_t *>(act);
    uint8_t *ap = static_cast<uint8_t *>(a);
    const int G = I / 128;
    if (G > 65535) return fail(PQ_ERR_SHAPE, "pq_silu_mul_rotate_quant: I = %d too large", I);
    cudaError_t e;
    if (M <= 16) {
        if (M == 1)
            e = launch_pdl(silu_mul_rotate_quant_small_kernel<1>, dim3(1, G, P), dim3(64), 0, st, yp, M, I, ldy,
                           recp, cp, actp, ap, asg, rs);
        else if (M == 2)
            e = launch_pdl(silu_mul_rotate_quant_small_kernel<2>, dim3(1, G, P), dim3(128), 0, st, yp, M, I, ldy,
                           recp, cp, actp, ap, asg, rs);
        else
            e = launch_pdl(silu_mul_rotate_quant_small_kernel<4>, dim3((M + 3) / 4, G, P), dim3(256), 0, st, yp, M,
                           I, ldy, recp, cp, actp, ap, asg, rs);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "silu_mul_rotate_quant launch: %s", cudaGetErrorString(e));
        return PQ_OK;
    }
    const dim3 grid((unsigned)((I / 2 + 255) / 256), (unsigned)(M < 65535 ? M : 65535));
    e = launch_pdl(silu_mul_kernel, grid, dim3(256), 0, st, yp, M, I, ldy, actp);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "silu_mul launch: %s", cudaGetErrorString(e));
    return launch_rotate_quant(act, M, I, I, P, rec, cs, a, asg, rs, stream);
}

pq_status launch_e4m3_encode(const float *in, uint8_t *out, size_t n, void *stream) {
    e4m3_encode_kernel<<<1216, 256, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "e4m3_encode launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

// ------------------------------------------------ the per-token prologue without caller scratch
// The bf16 rotated rows that pass A hands to pass C live in this fixed array
// instead of a caller buffer.  It is part of the library's device image, so
// every GPU that loads the library holds its 16 MiB until the process exits.
// Pass A writes every element pass C reads, so nothing in it needs clearing.
static __device__ __align__(256) uint16_t g_tokquant_xr[PQ_TOKQUANT_NOALLOC_MAX_ELEMS];

namespace {
// Device address of g_tokquant_xr on the current device.  In host code the
// symbol names a host-side stand-in, never device memory, so the address is
// looked up once per device (with that device current) and cached.
pq_status tokquant_scratch(void **out) {
    static std::mutex mu;
    static void *cached[64];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return fail(PQ_ERR_ARCH, "cudaGetDevice: %s", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 64 && cached[dev]) {
        *out = cached[dev];
        return PQ_OK;
    }
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_tokquant_xr);
    if (e != cudaSuccess || !ptr) {
        cudaGetLastError();
        return fail(PQ_ERR_CUDA, "cudaGetSymbolAddress(g_tokquant_xr): %s", cudaGetErrorString(e));
    }
    if (dev < 64) cached[dev] = ptr;
    *out = ptr;
    return PQ_OK;
}
}  // namespace

pq_status launch_rotate_tokquant_noalloc(const void *x, int M, int K, int ldx, int P, const void *rec,
                                         const void *cs, void *a, float *As, float *rs, void *stream) {
    void *xr = nullptr;
    const pq_status st = tokquant_scratch(&xr);
    if (st != PQ_OK) return st;
    return launch_rotate_tokquant(x, M, K, ldx, P, rec, cs, xr, a, As, rs, stream);
}

}  // namespace pq
