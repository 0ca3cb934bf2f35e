// pq_abi.cpp -- host side of libpq: status strings, per-thread error text,
// device checks, argument validation, the load-time packer and GEMM dispatch.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", sections
// "Format" (checkpoint layouts, nibble order 0,2,4,6,1,3,5,7, raw zero
// points, pairs local to each 128 group) and "Design" items 1 (SZ table of
// (scale, scale*(zp-8))), 3 (8-byte rotation records {i|j<<8, cos, sin}) and
// 4 (partition select from two boundary columns).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pq_internal.h"

namespace pq {

namespace {
thread_local std::string g_err;

const char *kStatusText[] = {
    "ok",
    "a required pointer is NULL",
    "a size or leading dimension is out of range",
    "a pointer or leading dimension breaks the alignment rule",
    "a pairs row is not a permutation of 0..127",
    "partition count or boundaries are inconsistent",
    "no sm_103 device is current",
    "a CUDA runtime call failed",
    "a pointer is not directly usable by the device",
};
}  // namespace

pq_status fail(pq_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

void clear_error() { g_err.clear(); }

namespace {
// 0: the product bound kWaitLimitNs; otherwise the test bound in ns.
std::atomic<unsigned long long> g_test_wait_ns{0};
}  // namespace

WaitBound pipeline_wait_bound() {
    const unsigned long long t = g_test_wait_ns.load(std::memory_order_relaxed);
    if (t == 0) return WaitBound{kWaitLimitNs, kSuspendHintNs};
    return WaitBound{t, t < kSuspendHintNs ? (uint32_t)t : kSuspendHintNs};
}

pq_status check_device(int *sm_count) {
    // Per-device cache of (checked, ok, SMs); devices are few and fixed.
    static std::mutex mu;
    static int cached_sm[64];
    static int cached_ok[64];   // 0 unknown, 1 ok, -1 wrong arch
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return fail(PQ_ERR_ARCH, "cudaGetDevice: %s", cudaGetErrorString(e));
    }
    if (dev < 64) {
        std::lock_guard<std::mutex> lk(mu);
        if (cached_ok[dev] == 1) {
            if (sm_count) *sm_count = cached_sm[dev];
            return PQ_OK;
        }
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        e = cudaGetLastError();
        return fail(PQ_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    }
    if (major != 10 || minor != 3)
        return fail(PQ_ERR_ARCH, "device %d is sm_%d%d; libpq is built for sm_103a only", dev,
                    major, minor);
    if (dev < 64) {
        std::lock_guard<std::mutex> lk(mu);
        cached_ok[dev] = 1;
        cached_sm[dev] = sms;
    }
    if (sm_count) *sm_count = sms;
    return PQ_OK;
}

static pq_status check_partitions(int P, int N, int pb1, int pb2) {
    if (P < 1 || P > PQ_MAX_PARTITIONS)
        return fail(PQ_ERR_PARTITION, "P = %d outside 1..%d", P, PQ_MAX_PARTITIONS);
    if (pb1 % 128 || pb2 % 128)
        return fail(PQ_ERR_PARTITION, "pb1 = %d, pb2 = %d must be multiples of 128", pb1, pb2);
    bool ok = false;
    if (P == 1) ok = (pb1 == N && pb2 == N);
    if (P == 2) ok = (pb1 > 0 && pb1 < N && pb2 == N);
    if (P == 3) ok = (pb1 > 0 && pb1 < pb2 && pb2 < N);
    if (!ok)
        return fail(PQ_ERR_PARTITION, "pb1 = %d, pb2 = %d do not describe %d partitions of N = %d",
                    pb1, pb2, P, N);
    return PQ_OK;
}

pq_status check_gemm_args(const void *a, const float *asg, const float *rs, int M, int N, int K,
                          int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                          int ldy) {
    if (!a || !asg || !rs || !w || !sz || !y) return fail(PQ_ERR_NULL, "NULL buffer");
    if (M < 1 || N < 128 || K < 128 || N % 128 || K % 128)
        return fail(PQ_ERR_SHAPE, "M = %d, N = %d, K = %d (need M >= 1, N and K positive "
                    "multiples of 128)", M, N, K);
    if ((long long)K * 128 > (1ll << 31) || (long long)M * N > (1ll << 40))
        return fail(PQ_ERR_SHAPE, "sizes too large");
    if (ldy < N) return fail(PQ_ERR_SHAPE, "ldy = %d < N = %d", ldy, N);
    pq_status st = check_partitions(P, N, pb1, pb2);
    if (st != PQ_OK) return st;
    if (!aligned(a, 16) || !aligned(w, 16) || !aligned(sz, 16) || !aligned(y, 16) ||
        !aligned(asg, 4) || !aligned(rs, 4) || ldy % 8)
        return fail(PQ_ERR_ALIGN, "a, w, sz, y need 16-byte alignment, asg/rs 4-byte, ldy a "
                    "multiple of 8");
    return PQ_OK;
}

// ---------------------------------------------------------------------------
// load-time packer
// ---------------------------------------------------------------------------

// double -> IEEE binary16 bits, round to nearest even, by integer manipulation
// of the binary64 encoding.
static uint16_t half_bits_rne(double d) {
    uint64_t u;
    std::memcpy(&u, &d, 8);
    const uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    const uint64_t mag = u & 0x7FFFFFFFFFFFFFFFull;
    if (mag > 0x7FF0000000000000ull) return sign | 0x7E00;          // NaN
    if ((mag >> 52) == 0) return sign;                                // zero / binary64 subnormal
    const int e = (int)(mag >> 52) - 1023;                            // value in [2^e, 2^(e+1))
    if (e >= 16) return sign | 0x7C00;
    const uint64_t sig = (mag & ((1ull << 52) - 1)) | (1ull << 52);   // 53-bit significand
    const int qexp = (e < -14 ? -14 : e) - 10;                        // exponent of one f16 ulp
    const int drop = qexp - (e - 52);                                 // >= 42
    if (drop > 63) return sign;
    uint64_t n = sig >> drop;
    const uint64_t rem = sig & ((1ull << drop) - 1), half = 1ull << (drop - 1);
    if (rem > half || (rem == half && (n & 1))) n++;
    if (e < -14) return sign | (uint16_t)n;                           // n <= 1024 (1024 = min normal)
    const uint32_t bits = ((uint32_t)(e + 15) << 10) + (uint32_t)(n - 1024);   // n == 2048 carries
    return bits >= 0x7C00 ? (uint16_t)(sign | 0x7C00) : (uint16_t)(sign | bits);
}

static double half_value(uint16_t h) {
    const int e = (h >> 10) & 31, m = h & 1023;
    double v = e == 0 ? std::ldexp((double)m, -24) : std::ldexp((double)(m | 1024), e - 25);
    return (h & 0x8000) ? -v : v;
}

// AWQ interleave: slot s of a packed word holds column kAwqOrder[s] of its octet.
static const int kAwqOrder[8] = {0, 2, 4, 6, 1, 3, 5, 7};

}  // namespace pq

using namespace pq;

extern "C" int pq_abi_version(void) { return PQ_ABI_VERSION; }

extern "C" const char *pq_status_string(int status) {
    if (status < 0 || status > (int)PQ_ERR_ACCESS) return "unknown status";
    return kStatusText[status];
}

extern "C" const char *pq_last_error(void) { return g_err.c_str(); }

extern "C" pq_status pq_pack_sizes(int K, int N, int P, size_t *rec_bytes, size_t *sz_bytes,
                                   size_t *w_bytes) {
    clear_error();
    if (K < 128 || N < 128 || K % 128 || N % 128)
        return fail(PQ_ERR_SHAPE, "K = %d, N = %d must be positive multiples of 128", K, N);
    if (P < 1 || P > PQ_MAX_PARTITIONS) return fail(PQ_ERR_PARTITION, "P = %d outside 1..3", P);
    const size_t G = (size_t)K / 128;
    if (rec_bytes) *rec_bytes = (size_t)P * 8 * G * 64 * 8;
    if (sz_bytes) *sz_bytes = G * (size_t)N * 4;
    if (w_bytes) *w_bytes = (size_t)N * (size_t)K / 2;
    return PQ_OK;
}

// Both packers: int4 (qweight_hi == NULL) or int5 (the fifth-bit planes
// qweight_hi [K][N/32], qzeros_hi [G][N/32], column 32w + j in bit j).
static pq_status pack_layer(int K, int N, int P, const int32_t *qweight, const int32_t *qzeros,
                            const int32_t *qweight_hi, const int32_t *qzeros_hi, const uint16_t *scales,
                            const int16_t *pairs, const uint16_t *theta, void *rec, void *sz, void *w,
                            void *whi) {
    pq_status st = pq_pack_sizes(K, N, P, nullptr, nullptr, nullptr);
    if (st != PQ_OK) return st;
    const int G = K / 128, W8 = N / 8, W32 = N / 32;
    const bool int5 = qweight_hi != nullptr;
    const int offset = int5 ? 16 : 8;       // the code's midpoint: c - 8 (int4), c - 16 (int5)

    // pairs: every (p, layer, group) row a permutation of 0..127
    for (int row = 0; row < P * 8 * G; ++row) {
        const int16_t *pr = pairs + (size_t)row * 128;   // rows are contiguous 128-entry blocks
        uint64_t seen[2] = {0, 0};
        for (int t = 0; t < 128; ++t) {
            const int v = pr[t];
            if (v < 0 || v > 127 || ((seen[v >> 6] >> (v & 63)) & 1))
                return fail(PQ_ERR_PAIRS, "pairs row (p=%d, layer=%d, group=%d) is not a "
                            "permutation of 0..127", row / (8 * G), (row / G) % 8, row % G);
            seen[v >> 6] |= 1ull << (v & 63);
        }
    }

    // rotation records: [p][layer][g][slot] = {u, v, keep, 0, f16 cos, f16 sin},
    // in chained order (pq.h): layer 0 in the pages' order; slot t of layer
    // r + 1 holds the pair of the channel that slot t keeps from layer r, that
    // channel first (u), the sine negated where this reverses the pages' pair.
    // The kept channels of a layer are chosen along the alternating cycles of
    // the two layers' pairings, walked from the lowest unvisited channel:
    // cycle x0 -r- y0 -(r+1)- x1 -r- y1 ... keeps y0, y1, ..., so that every
    // pair of layer r + 1 receives exactly one kept channel.
    uint8_t *ro = static_cast<uint8_t *>(rec);
    for (int p = 0; p < P; ++p)
        for (int g = 0; g < G; ++g) {
            int u[64], v[64], src[64];      // this layer's slots: channels, pages' pair index
            bool rev[64];                   // (u, v) is the pages' pair reversed
            const int16_t *p0 = pairs + (size_t)p * 8 * K + 128 * g;
            for (int t = 0; t < 64; ++t) {
                u[t] = p0[2 * t];
                v[t] = p0[2 * t + 1];
                src[t] = t;
                rev[t] = false;
            }
            for (int r = 0; r < 8; ++r) {
                const size_t pl = (size_t)p * 8 + r;
                uint8_t keep_v[64] = {};
                int nu[64], nv[64], nsrc[64];
                bool nrev[64];
                if (r < 7) {
                    const int16_t *pn = pairs + (pl + 1) * K + 128 * g;
                    int mate[128], slot[128], mate_n[128], pair_n[128];
                    for (int t = 0; t < 64; ++t) {
                        mate[u[t]] = v[t];
                        mate[v[t]] = u[t];
                        slot[u[t]] = slot[v[t]] = t;
                        const int a = pn[2 * t], b = pn[2 * t + 1];
                        mate_n[a] = b;
                        mate_n[b] = a;
                        pair_n[a] = pair_n[b] = t;
                    }
                    bool seen[128] = {};
                    for (int c0 = 0; c0 < 128; ++c0) {
                        if (seen[c0]) continue;
                        int x = c0;
                        do {
                            const int y = mate[x], t = slot[x], tn = pair_n[y];
                            seen[x] = seen[y] = true;
                            keep_v[t] = (uint8_t)(y == v[t]);
                            nu[t] = y;
                            nv[t] = mate_n[y];
                            nsrc[t] = tn;
                            nrev[t] = pn[2 * tn] != y;
                            x = mate_n[y];
                        } while (x != c0);
                    }
                }
                for (int t = 0; t < 64; ++t) {
                    const double th = half_value(theta[pl * (K / 2) + 64 * g + src[t]]);
                    const uint16_t c = half_bits_rne(std::cos(th));
                    const uint16_t s = (uint16_t)(half_bits_rne(std::sin(th)) ^ (rev[t] ? 0x8000u : 0u));
                    uint8_t *o = ro + ((pl * G + g) * 64 + t) * 8;
                    o[0] = (uint8_t)u[t];
                    o[1] = (uint8_t)v[t];
                    o[2] = keep_v[t];
                    o[3] = 0;
                    o[4] = (uint8_t)(c & 0xFF);
                    o[5] = (uint8_t)(c >> 8);
                    o[6] = (uint8_t)(s & 0xFF);
                    o[7] = (uint8_t)(s >> 8);
                }
                if (r < 7)
                    for (int t = 0; t < 64; ++t) {
                        u[t] = nu[t];
                        v[t] = nv[t];
                        src[t] = nsrc[t];
                        rev[t] = nrev[t];
                    }
            }
        }

    // SZ table: (sc, f16(sc * (zp - offset))), the product exact in fp32, one
    // word per (column, group) at [n/8][g][n%8]
    uint32_t *so = static_cast<uint32_t *>(sz);
    for (int g = 0; g < G; ++g)
        for (int w8 = 0; w8 < W8; ++w8) {
            const uint32_t zw = (uint32_t)qzeros[(size_t)g * W8 + w8];
            for (int s = 0; s < 8; ++s) {
                const int j = kAwqOrder[s];
                const int n = 8 * w8 + j;
                int zp = (int)((zw >> (4 * s)) & 15u);
                if (int5) zp += 16 * (int)(((uint32_t)qzeros_hi[(size_t)g * W32 + n / 32] >> (n % 32)) & 1u);
                const uint16_t sc = scales[(size_t)g * N + n];
                const float prod = (float)half_value(sc) * (float)(zp - offset);
                so[((size_t)w8 * G + g) * 8 + j] = (uint32_t)sc | ((uint32_t)half_bits_rne((double)prod) << 16);
            }
        }

    // weights: per run of eight k (k0 = 8t), byte 4t + b of row n holds
    // c[k0 + b][n] (low nibble) and c[k0 + b + 4][n] (high nibble), so that
    // masking a word's low and high nibbles yields k0..k0+3 and k0+4..k0+7 in
    // byte order
    uint8_t *wo = static_cast<uint8_t *>(w);
    for (int k0 = 0; k0 < K; k0 += 8)
        for (int b = 0; b < 4; ++b) {
            const int32_t *r0 = qweight + (size_t)(k0 + b) * W8;
            const int32_t *r1 = qweight + (size_t)(k0 + b + 4) * W8;
            for (int w8 = 0; w8 < W8; ++w8) {
                const uint32_t a0 = (uint32_t)r0[w8], a1 = (uint32_t)r1[w8];
                for (int s = 0; s < 8; ++s) {
                    const int n = 8 * w8 + kAwqOrder[s];
                    wo[(size_t)n * (K / 2) + k0 / 2 + b] =
                        (uint8_t)(((a0 >> (4 * s)) & 15u) | (((a1 >> (4 * s)) & 15u) << 4));
                }
            }
        }

    // int5: fifth bits whi[n][K/8] in 4-byte blocks of 32 k.  Byte j of a
    // block collects the bits of k = 4q + j (q = 0..7) at bit q, so that one
    // left shift moves the bits of four consecutive k to the top bits of the
    // four bytes (the expansion's byte masks)
    if (int5) {
        uint8_t *ho = static_cast<uint8_t *>(whi);
        for (int k32 = 0; k32 < K; k32 += 32)
            for (int n = 0; n < N; ++n)
                for (int j = 0; j < 4; ++j) {
                    uint32_t b = 0;
                    for (int q = 0; q < 8; ++q)
                        b |= (((uint32_t)qweight_hi[(size_t)(k32 + 4 * q + j) * W32 + n / 32] >> (n % 32)) & 1u) << q;
                    ho[(size_t)n * (K / 8) + k32 / 8 + j] = (uint8_t)b;
                }
    }
    return PQ_OK;
}

extern "C" pq_status pq_pack(int K, int N, int P, const int32_t *qweight, const int32_t *qzeros,
                             const uint16_t *scales, const int16_t *pairs, const uint16_t *theta,
                             void *rec, void *sz, void *w) {
    clear_error();
    if (!qweight || !qzeros || !scales || !pairs || !theta || !rec || !sz || !w)
        return fail(PQ_ERR_NULL, "pq_pack: NULL pointer");
    return pack_layer(K, N, P, qweight, qzeros, nullptr, nullptr, scales, pairs, theta, rec, sz, w, nullptr);
}

extern "C" pq_status pq_pack5(int K, int N, int P, const int32_t *qweight, const int32_t *qzeros,
                              const int32_t *qweight_hi, const int32_t *qzeros_hi, const uint16_t *scales,
                              const int16_t *pairs, const uint16_t *theta, void *rec, void *sz, void *w,
                              void *whi) {
    clear_error();
    if (!qweight || !qzeros || !qweight_hi || !qzeros_hi || !scales || !pairs || !theta || !rec || !sz || !w ||
        !whi)
        return fail(PQ_ERR_NULL, "pq_pack5: NULL pointer");
    return pack_layer(K, N, P, qweight, qzeros, qweight_hi, qzeros_hi, scales, pairs, theta, rec, sz, w, whi);
}

extern "C" pq_status pq_rotate_quant(const void *x, int M, int K, int ldx, int P, const void *rec,
                                     const void *cs, void *a, float *asg, float *rs,
                                     void *stream) {
    clear_error();
    if (!x || !rec || !cs || !a || !asg || !rs) return fail(PQ_ERR_NULL, "NULL buffer");
    if (M < 1 || K < 128 || K % 128 || ldx < K)
        return fail(PQ_ERR_SHAPE, "M = %d, K = %d, ldx = %d", M, K, ldx);
    if ((long long)M * K > (1ll << 40)) return fail(PQ_ERR_SHAPE, "sizes too large");
    if (P < 1 || P > PQ_MAX_PARTITIONS) return fail(PQ_ERR_PARTITION, "P = %d outside 1..3", P);
    if (!aligned(x, 16) || !aligned(rec, 16) || !aligned(cs, 16) || !aligned(a, 16) ||
        !aligned(asg, 4) || !aligned(rs, 4) || ldx % 8)
        return fail(PQ_ERR_ALIGN, "x, rec, cs, a need 16-byte alignment, asg/rs 4-byte, ldx a "
                    "multiple of 8");
    pq_status st = check_device(nullptr);
    if (st != PQ_OK) return st;
    return launch_rotate_quant(x, M, K, ldx, P, rec, cs, a, asg, rs, stream);
}

// Whether [a, a + na) and [b, b + nb) share a byte.
static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

extern "C" pq_status pq_add_rms_rotate_quant(const void *x, const void *residual, const void *gamma, float eps,
                                             int M, int K, int ldx, int P, const void *rec, const void *cs,
                                             void *residual_out, void *h, void *a, float *asg, float *rs,
                                             void *stream) {
    clear_error();
    if (!x || !residual || !gamma || !rec || !cs || !residual_out || !h || !a || !asg || !rs)
        return fail(PQ_ERR_NULL, "NULL buffer");
    if (M < 1 || K < 128 || K % 128 || ldx < K)
        return fail(PQ_ERR_SHAPE, "M = %d, K = %d, ldx = %d", M, K, ldx);
    if ((long long)M * ldx > (1ll << 40)) return fail(PQ_ERR_SHAPE, "sizes too large");
    if (!(eps >= 0.0f) || eps > 3.0e38f) return fail(PQ_ERR_SHAPE, "eps must be finite and >= 0");
    if (P < 1 || P > PQ_MAX_PARTITIONS) return fail(PQ_ERR_PARTITION, "P = %d outside 1..3", P);
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(gamma, 16) || !aligned(rec, 16) ||
        !aligned(cs, 16) || !aligned(residual_out, 16) || !aligned(h, 16) || !aligned(a, 16) ||
        !aligned(asg, 4) || !aligned(rs, 4) || ldx % 8)
        return fail(PQ_ERR_ALIGN, "x, residual, gamma, rec, cs, residual_out, h, a need 16-byte "
                    "alignment, asg/rs 4-byte, ldx a multiple of 8");
    const size_t in_bytes = ((size_t)(M - 1) * ldx + K) * 2, out_bytes = (size_t)M * K * 2;
    if (overlaps(residual_out, out_bytes, x, in_bytes) || overlaps(residual_out, out_bytes, residual, in_bytes) ||
        overlaps(h, out_bytes, x, in_bytes) || overlaps(h, out_bytes, residual, in_bytes))
        return fail(PQ_ERR_SHAPE, "residual_out and h must not overlap x or residual");
    pq_status st = check_device(nullptr);
    if (st != PQ_OK) return st;
    return launch_add_rms_rotate_quant(x, residual, gamma, eps, M, K, ldx, P, rec, cs, residual_out, h, a, asg,
                                       rs, stream);
}

extern "C" pq_status pq_silu_mul_rotate_quant(const void *y, int M, int I, int ldy, int P, const void *rec,
                                              const void *cs, void *act, void *a, float *asg, float *rs,
                                              void *stream) {
    clear_error();
    if (!y || !rec || !cs || !act || !a || !asg || !rs) return fail(PQ_ERR_NULL, "NULL buffer");
    if (M < 1 || I < 128 || I % 128 || ldy < 2 * I)
        return fail(PQ_ERR_SHAPE, "M = %d, I = %d, ldy = %d", M, I, ldy);
    if ((long long)M * ldy > (1ll << 40)) return fail(PQ_ERR_SHAPE, "sizes too large");
    if (P < 1 || P > PQ_MAX_PARTITIONS) return fail(PQ_ERR_PARTITION, "P = %d outside 1..3", P);
    if (!aligned(y, 16) || !aligned(rec, 16) || !aligned(cs, 16) || !aligned(act, 16) || !aligned(a, 16) ||
        !aligned(asg, 4) || !aligned(rs, 4) || ldy % 8)
        return fail(PQ_ERR_ALIGN, "y, rec, cs, act, a need 16-byte alignment, asg/rs 4-byte, ldy a "
                    "multiple of 8");
    if (overlaps(act, (size_t)M * I * 2, y, ((size_t)(M - 1) * ldy + 2 * I) * 2))
        return fail(PQ_ERR_SHAPE, "act must not overlap y");
    pq_status st = check_device(nullptr);
    if (st != PQ_OK) return st;
    return launch_silu_mul_rotate_quant(y, M, I, ldy, P, rec, cs, act, a, asg, rs, stream);
}

extern "C" pq_status pq_rotate_tokquant(const void *x, int M, int K, int ldx, int P, const void *rec,
                                        const void *cs, void *xr, void *a, float *As, float *rs, void *stream) {
    clear_error();
    if (!x || !rec || !cs || !xr || !a || !As || !rs) return fail(PQ_ERR_NULL, "NULL buffer");
    if (M < 1 || K < 128 || K % 128 || ldx < K)
        return fail(PQ_ERR_SHAPE, "M = %d, K = %d, ldx = %d", M, K, ldx);
    if ((long long)M * ldx > (1ll << 40)) return fail(PQ_ERR_SHAPE, "sizes too large");
    if (P < 1 || P > PQ_MAX_PARTITIONS) return fail(PQ_ERR_PARTITION, "P = %d outside 1..3", P);
    if (!aligned(x, 16) || !aligned(rec, 16) || !aligned(cs, 16) || !aligned(xr, 16) || !aligned(a, 16) ||
        !aligned(As, 4) || !aligned(rs, 4) || ldx % 8)
        return fail(PQ_ERR_ALIGN, "x, rec, cs, xr, a need 16-byte alignment, As/rs 4-byte, ldx a "
                    "multiple of 8");
    if (overlaps(xr, (size_t)P * M * K * 2, x, ((size_t)(M - 1) * ldx + K) * 2))
        return fail(PQ_ERR_SHAPE, "xr must not overlap x");
    pq_status st = check_device(nullptr);
    if (st != PQ_OK) return st;
    return launch_rotate_tokquant(x, M, K, ldx, P, rec, cs, xr, a, As, rs, stream);
}

extern "C" pq_status pq_rotate_tokquant_noalloc(const void *x, int M, int K, int ldx, int P, const void *rec,
                                                const void *cs, void *a, float *As, float *rs, void *stream) {
    clear_error();
    if (!x || !rec || !cs || !a || !As || !rs) return fail(PQ_ERR_NULL, "NULL buffer");
    if (M < 1 || K < 128 || K % 128 || ldx < K)
        return fail(PQ_ERR_SHAPE, "M = %d, K = %d, ldx = %d", M, K, ldx);
    if ((long long)M * ldx > (1ll << 40)) return fail(PQ_ERR_SHAPE, "sizes too large");
    if (P < 1 || P > PQ_MAX_PARTITIONS) return fail(PQ_ERR_PARTITION, "P = %d outside 1..3", P);
    if ((unsigned long long)P * (unsigned long long)M * (unsigned long long)K > PQ_TOKQUANT_NOALLOC_MAX_ELEMS)
        return fail(PQ_ERR_SHAPE,
                    "pq_rotate_tokquant_noalloc: P * M * K = %llu exceeds its fixed scratch of %u elements; "
                    "use pq_rotate_tokquant with a caller buffer",
                    (unsigned long long)P * M * K, (unsigned)PQ_TOKQUANT_NOALLOC_MAX_ELEMS);
    if (!aligned(x, 16) || !aligned(rec, 16) || !aligned(cs, 16) || !aligned(a, 16) || !aligned(As, 4) ||
        !aligned(rs, 4) || ldx % 8)
        return fail(PQ_ERR_ALIGN, "x, rec, cs, a need 16-byte alignment, As/rs 4-byte, ldx a multiple of 8");
    pq_status st = check_device(nullptr);
    if (st != PQ_OK) return st;
    return launch_rotate_tokquant_noalloc(x, M, K, ldx, P, rec, cs, a, As, rs, stream);
}

extern "C" pq_status pq_gemm_ptok(const void *a, const float *As, const float *rs, int M, int N, int K,
                                  int P, int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                                  unsigned int *dev_status, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, As, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    return launch_gemm_tc(a, As, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream, sms, true);
}

extern "C" pq_status pq_e4m3_encode(const float *in, uint8_t *out, size_t n, void *stream) {
    clear_error();
    if (!in || !out) return fail(PQ_ERR_NULL, "NULL buffer");
    if (!aligned(in, 4)) return fail(PQ_ERR_ALIGN, "in needs 4-byte alignment");
    pq_status st = check_device(nullptr);
    if (st != PQ_OK) return st;
    if (n == 0) return PQ_OK;
    return launch_e4m3_encode(in, out, n, stream);
}

extern "C" int pq_gemm_skinny_max_m(void) { return kSkinnyMaxM; }

extern "C" pq_status pq_gemm_skinny(const void *a, const float *asg, const float *rs, int M,
                                    int N, int K, int P, int pb1, int pb2, const void *w,
                                    const void *sz, void *y, int ldy, unsigned int *dev_status,
                                    void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (M > kSkinnyMaxM) return fail(PQ_ERR_SHAPE, "pq_gemm_skinny: M = %d > %d", M, kSkinnyMaxM);
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    return launch_gemm_skinny(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream,
                              sms);
}

extern "C" pq_status pq_gemm_tc(const void *a, const float *asg, const float *rs, int M, int N,
                                int K, int P, int pb1, int pb2, const void *w, const void *sz,
                                void *y, int ldy, unsigned int *dev_status, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    return launch_gemm_tc(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream, sms);
}

extern "C" pq_status pq_gemm_tcn(const void *a, const float *asg, const float *rs, int M, int N,
                                 int K, int P, int pb1, int pb2, const void *w, const void *sz,
                                 void *y, int ldy, unsigned int *dev_status, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (M > kTcnMaxM) return fail(PQ_ERR_SHAPE, "pq_gemm_tcn: M = %d > %d", M, kTcnMaxM);
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    return launch_gemm_tcn(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream);
}

extern "C" pq_status pq_gemm5_tc(const void *a, const float *asg, const float *rs, int M, int N, int K,
                                 int P, int pb1, int pb2, const void *w, const void *whi, const void *sz,
                                 void *y, int ldy, unsigned int *dev_status, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (!whi) return fail(PQ_ERR_NULL, "NULL whi");
    if (!aligned(whi, 16)) return fail(PQ_ERR_ALIGN, "whi needs 16-byte alignment");
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    return launch_gemm_tc(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream, sms, false, whi);
}

extern "C" pq_status pq_gemm5_tcn(const void *a, const float *asg, const float *rs, int M, int N, int K,
                                  int P, int pb1, int pb2, const void *w, const void *whi, const void *sz,
                                  void *y, int ldy, unsigned int *dev_status, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (!whi) return fail(PQ_ERR_NULL, "NULL whi");
    if (!aligned(whi, 16)) return fail(PQ_ERR_ALIGN, "whi needs 16-byte alignment");
    if (M > kTcnMaxM) return fail(PQ_ERR_SHAPE, "pq_gemm5_tcn: M = %d > %d", M, kTcnMaxM);
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    st = check_device(nullptr);
    if (st != PQ_OK) return st;
    return launch_gemm_tcn(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream, whi);
}

extern "C" pq_status pq_gemm5_skinny(const void *a, const float *asg, const float *rs, int M, int N, int K,
                                     int P, int pb1, int pb2, const void *w, const void *whi, const void *sz,
                                     void *y, int ldy, unsigned int *dev_status, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (!whi) return fail(PQ_ERR_NULL, "NULL whi");
    if (!aligned(whi, 16)) return fail(PQ_ERR_ALIGN, "whi needs 16-byte alignment");
    if (M > kSkinnyMaxM) return fail(PQ_ERR_SHAPE, "pq_gemm5_skinny: M = %d > %d", M, kSkinnyMaxM);
    if (dev_status && !aligned(dev_status, 4)) return fail(PQ_ERR_ALIGN, "dev_status alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    return launch_gemm_skinny(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, dev_status, stream, sms, whi);
}

extern "C" pq_status pq_gemm5(const void *a, const float *asg, const float *rs, int M, int N, int K, int P,
                              int pb1, int pb2, const void *w, const void *whi, const void *sz, void *y,
                              int ldy, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    if (!whi) return fail(PQ_ERR_NULL, "NULL whi");
    if (!aligned(whi, 16)) return fail(PQ_ERR_ALIGN, "whi needs 16-byte alignment");
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    // As pq_gemm: M = 1 on the CUDA-core kernel (fewest instructions per
    // weight); 2 <= M <= 16 on the narrow tensor-core kernel when its
    // 128-feature tiles cover at least half the SMs, else on the CUDA-core
    // kernel; any M <= 16 with K above the CUDA-core limit on the narrow
    // kernel; M > 16 on the prefill kernel.
    if (M <= kSkinnyMaxM) {
        if ((M >= 2 && M <= kTcnMaxM && 2 * (N / 128) >= sms) || K > kSkinnyMaxK)
            return launch_gemm_tcn(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, nullptr, stream, whi);
        return launch_gemm_skinny(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, nullptr, stream, sms, whi);
    }
    return launch_gemm_tc(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, nullptr, stream, sms, false, whi);
}

extern "C" pq_status pq_gemm(const void *a, const float *asg, const float *rs, int M, int N, int K,
                             int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                             int ldy, void *stream) {
    clear_error();
    pq_status st = check_gemm_args(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy);
    if (st != PQ_OK) return st;
    int sms = 0;
    st = check_device(&sms);
    if (st != PQ_OK) return st;
    // M = 1: the CUDA-core kernel streams the weights with the fewest instructions.
    // 2 <= M <= 16: the narrow tensor-core kernel, when its 128-feature tiles cover
    // at least half the SMs (it streams each tile from one SM); otherwise the
    // CUDA-core kernel, which spreads 8-feature octets over every SM.
    // Any M <= 16 with K above the CUDA-core kernel's limit: the narrow kernel.
    // M > 16: the prefill tensor-core kernel.
    if (M <= kSkinnyMaxM) {
        if ((M >= 2 && M <= kTcnMaxM && 2 * (N / 128) >= sms) || K > kSkinnyMaxK)
            return launch_gemm_tcn(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, nullptr, stream);
        return launch_gemm_skinny(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, nullptr, stream,
                                  sms);
    }
    return launch_gemm_tc(a, asg, rs, M, N, K, P, pb1, pb2, w, sz, y, ldy, nullptr, stream, sms);
}

extern "C" pq_status pq_test_set_wait_limit_ns(unsigned long long ns) {
    clear_error();
    if (ns > pq::kWaitLimitNs) return pq::fail(PQ_ERR_SHAPE, "wait limit %llu ns above the product bound", ns);
    pq::g_test_wait_ns.store(ns, std::memory_order_relaxed);
    return PQ_OK;
}

extern "C" pq_status pq_check_device_access(const void *p) {
    clear_error();
    if (!p) return pq::fail(PQ_ERR_NULL, "NULL pointer");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return pq::fail(PQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    }
    cudaPointerAttributes at{};
    e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return pq::fail(PQ_ERR_CUDA, "cudaPointerGetAttributes: %s", cudaGetErrorString(e));
    }
    switch (at.type) {
        case cudaMemoryTypeManaged:
            return PQ_OK;
        case cudaMemoryTypeDevice:
            if (at.device == dev) return PQ_OK;
            return pq::fail(PQ_ERR_ACCESS, "device memory of device %d, current device %d", at.device, dev);
        case cudaMemoryTypeHost:
            if (at.devicePointer == p) return PQ_OK;
            return pq::fail(PQ_ERR_ACCESS, "page-locked host memory not mapped at the same device address");
        default:
            return pq::fail(PQ_ERR_ACCESS, "pageable host memory");
    }
}
