// pq_rotate_quant.cu -- the fused prologue: channel scale, eight layers of
// Givens rotations per 128-channel group, per-(token, group) amax, e4m3 encode
// and code-domain row-sums, for up to three partitions, in one launch.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Design"
// items 2 (per-group fp8 activation scales, no cross-block sync) and 3 (fused
// prologue; records read once per chunk; row-sum = sum of what the codes decode
// to), "Gates passed" (scale = amax * (1/448.f), bit-exact to a CPU reference),
// and "2026-09-15: hardware e4m3 convert" (NaN -> 0, -0 -> +0, clamp +-448,
// then the hardware round-to-nearest-even convert).
//
// Layout on the GPU.  One CTA owns a tile of 32 tokens x one 128-group and
// loops over the partitions.  The tile is held in shared memory as
// v[k][token] (fp32), token fastest: in a Givens layer every warp works on one
// pair (i, j) at a time with lane = token, so the 32 lanes read v[i][0..31]
// and v[j][0..31] -- consecutive words, free of bank conflicts whatever the
// pair permutation is.  Each of the 4 warps takes 16 of the 64 disjoint pairs
// of a layer; the layers are separated by __syncthreads.  Every multiply, add,
// subtract and divide is a separately rounded IEEE operation (explicit .rn
// intrinsics; the packed f32x2 forms are .rn as well), so results are
// bit-identical to an fp32 CPU evaluation in the same order.
#include <cuda_runtime.h>

#include <cstdint>

#include "pq_internal.h"

namespace pq {
namespace {

constexpr int kTok = 32;              // tokens per CTA (lane = token)
constexpr int kWarps = 4;             // warp w rotates pairs 16w..16w+15 of each layer
constexpr int kThreads = kTok * kWarps;
constexpr int kXsStride = 65;         // words per staged x row (64 + 1 pad)
constexpr int kCodeStride = 144;      // bytes per staged code row

struct __align__(16) Smem {
    float v[128][kTok];               // 16 KB
    uint32_t xs[kTok][kXsStride];     // x tile, two bf16 per word
    uint2 rec[8][64];                 // records of (p, g)
    float cs[128];
    uint8_t codes[kTok][kCodeStride];
    float red_max[kWarps][kTok];
    int red_sum[kWarps][kTok];
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

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

// dec(code) * 2^9 as an integer (exact; |value| <= 448 * 512)
__device__ __forceinline__ int e4m3_times512(uint32_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    const int mag = e == 0 ? m : ((8 | m) << (e - 1));
    return (c & 0x80) ? -mag : mag;
}

__global__ void __launch_bounds__(kThreads)
rotate_quant_kernel(const uint16_t *__restrict__ x, int M, int K, int ldx, int P,
                    const uint2 *__restrict__ rec, const uint16_t *__restrict__ cs,
                    uint8_t *__restrict__ a, float *__restrict__ asg, float *__restrict__ rs) {
    __shared__ Smem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m0 = blockIdx.x * kTok, g = blockIdx.y, G = K >> 7;

    // x tile -> shared (bf16 pairs); tokens past M read as zero
    for (int c = tid; c < kTok * 16; c += kThreads) {
        const int row = c >> 4, q = c & 15;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (m0 + row < M)
            val = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(m0 + row) * ldx + 128 * g) + q);
        uint32_t *d = &sm.xs[row][4 * q];
        d[0] = val.x; d[1] = val.y; d[2] = val.z; d[3] = val.w;
    }
    const float inv448 = __fdiv_rn(1.0f, 448.0f);

    for (int p = 0; p < P; ++p) {
        // records of (p, g): 8 layers x 64 x 8 B, and the group's channel scales
        for (int c = tid; c < 8 * 32; c += kThreads) {
            const int r = c >> 5, q = c & 31;
            const uint4 val = __ldg(reinterpret_cast<const uint4 *>(
                                        rec + ((size_t)(p * 8 + r) * G + g) * 64) + q);
            sm.rec[r][2 * q] = make_uint2(val.x, val.y);
            sm.rec[r][2 * q + 1] = make_uint2(val.z, val.w);
        }
        sm.cs[tid] = half_to_float(__ldg(cs + (size_t)p * K + 128 * g + tid));
        __syncthreads();

        // v[k][t] = x[t][k] * cs[k] (exact: bf16 x f16 fits in 24 bits)
#pragma unroll 4
        for (int q = 0; q < 16; ++q) {
            const int kw = 16 * warp + q;                 // word index: channels 2kw, 2kw+1
            const uint32_t wv = sm.xs[lane][kw];
            sm.v[2 * kw][lane] = __fmul_rn(bf16lo(wv), sm.cs[2 * kw]);
            sm.v[2 * kw + 1][lane] = __fmul_rn(bf16hi(wv), sm.cs[2 * kw + 1]);
        }
        __syncthreads();

        // eight Givens layers; pairs of one layer are disjoint, so a warp reads
        // all 32 operands of its 16 pairs before writing any result
        for (int r = 0; r < 8; ++r) {
            float vi[16], vj[16];
            int ii[16], jj[16];
            float cc[16], ss[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint2 rr = sm.rec[r][16 * warp + q];
                ii[q] = rr.x & 0xFF;
                jj[q] = (rr.x >> 8) & 0xFF;
                cc[q] = half_to_float((uint16_t)(rr.y & 0xFFFF));
                ss[q] = half_to_float((uint16_t)(rr.y >> 16));
                vi[q] = sm.v[ii[q]][lane];
                vj[q] = sm.v[jj[q]][lane];
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float ni = __fadd_rn(__fmul_rn(cc[q], vi[q]), __fmul_rn(ss[q], vj[q]));
                const float nj = __fsub_rn(__fmul_rn(cc[q], vj[q]), __fmul_rn(ss[q], vi[q]));
                sm.v[ii[q]][lane] = ni;
                sm.v[jj[q]][lane] = nj;
            }
            __syncthreads();
        }

        // quantise: warp w takes channels 32w..32w+31 of every token
        float vals[32];
        float amax = 0.0f;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            vals[q] = sm.v[32 * warp + q][lane];
            amax = fmaxf(amax, fabsf(vals[q]));
        }
        sm.red_max[warp][lane] = amax;
        __syncthreads();
        amax = fmaxf(fmaxf(sm.red_max[0][lane], sm.red_max[1][lane]),
                     fmaxf(sm.red_max[2][lane], sm.red_max[3][lane]));
        const float scale = __fmul_rn(amax, inv448);
        uint32_t packed[8];
        int sum512 = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t word = 0;
            if (scale != 0.0f) {
                const uint32_t c01 = e4m3x2(__fdiv_rn(vals[4 * q + 1], scale),
                                            __fdiv_rn(vals[4 * q], scale));
                const uint32_t c23 = e4m3x2(__fdiv_rn(vals[4 * q + 3], scale),
                                            __fdiv_rn(vals[4 * q + 2], scale));
                word = c01 | (c23 << 16);
            }
            packed[q] = word;
#pragma unroll
            for (int b = 0; b < 4; ++b) sum512 += e4m3_times512((word >> (8 * b)) & 0xFF);
        }
        uint4 *cdst = reinterpret_cast<uint4 *>(&sm.codes[lane][32 * warp]);
        cdst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        cdst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        sm.red_sum[warp][lane] = sum512;
        __syncthreads();

        // stores: 128-byte code rows, then one scale and one row-sum per token
        for (int c = tid; c < kTok * 8; c += kThreads) {
            const int row = c >> 3, q = c & 7;
            if (m0 + row < M)
                reinterpret_cast<uint4 *>(a + ((size_t)p * M + m0 + row) * K + 128 * g)[q] =
                    *reinterpret_cast<const uint4 *>(&sm.codes[row][16 * q]);
        }
        if (m0 + lane < M) {
            const size_t o = ((size_t)p * G + g) * M + m0 + lane;
            if (warp == 0) asg[o] = scale;
            if (warp == 1) {
                const int s = sm.red_sum[0][lane] + sm.red_sum[1][lane] + sm.red_sum[2][lane] +
                              sm.red_sum[3][lane];
                rs[o] = __fmul_rn(__int2float_rn(s), 1.0f / 512.0f);
            }
        }
        __syncthreads();
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

}  // namespace

pq_status launch_rotate_quant(const void *x, int M, int K, int ldx, int P, const void *rec,
                              const void *cs, void *a, float *asg, float *rs, void *stream) {
    const dim3 grid((M + kTok - 1) / kTok, K / 128);
    if (grid.x > 0x7FFFFFFF || grid.y > 65535)
        return fail(PQ_ERR_SHAPE, "pq_rotate_quant: grid (%u, %u) too large", grid.x, grid.y);
    rotate_quant_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(x), M, K, ldx, P, static_cast<const uint2 *>(rec),
        static_cast<const uint16_t *>(cs), static_cast<uint8_t *>(a), asg, rs);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "rotate_quant launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

pq_status launch_e4m3_encode(const float *in, uint8_t *out, size_t n, void *stream) {
    e4m3_encode_kernel<<<1216, 256, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "e4m3_encode launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

}  // namespace pq
