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
// One CTA computes a 256 (tokens) x 128 (output features) tile of y as two
// M=128 halves that share the B tile.  Per 128-k group kb (a "slab"):
//   TMA warp     loads A[p][m0:m0+256][128kb:+128] (e4m3, 128B-swizzled,
//                zero-filled past M), the packed weight tile w[n0:n0+128]
//                [64kb:+64] and the slab's 128 SZ words (16 octets x 8 words
//                of the [N/8][G][8] table) into stage s.
//   row warps    load the slab's per-row asg and rs (one slab ahead of their
//                stores) into a ring slot of their own, up to the ring's depth
//                ahead: asg for the fold, and the zero-point MMA's row
//                operand, -rs / 2 as three bf16 parts.
//   expand warps turn each nibble c into the e4m3 byte of value c * 2^-9 (the
//                nibble alone in its byte) in the canonical K-major
//                SWIZZLE_128B layout the MMA reads, and write per column the
//                fold's 2^9 sc' and the zero-point MMA's column operand: the
//                bf16 parts of zq = 2^-9 (zscale + 8 sc) / sc'.  sc' = sc, or
//                1 where sc = 0, whose codes are masked to 0.
//   MMA warp     per half: 4 tcgen05.mma m128n128k32 (kind::f8f6f4, fp32
//                accumulate), then one m128n128k16 kind::f16 (bf16) MMA of the
//                zero-point operands into the same accumulator, so TMEM holds
//                D'' = 2^-9 (sum_k dec(a) c - rs * zq); two accumulator sets,
//                so the MMAs of slab kb+1 run while slab kb is folded.
//   fold warps   tcgen05.ld D'' and fold it into fp32 registers with packed
//                f32x2 operations: acc += (asg * 2^9 sc') * D''.  That is
//                asg * (sc * D' - (zscale + 8 sc) * rs) with D' = sum dec(a) c
//                = D + 8 rs, D the sum over (c - 8): the zero point of the
//                method, moved onto the tensor core, leaves two fp32 operations
//                per element and slab instead of three.
// Zero-point operand precision: with rs = h + m + l and zq = zh + zm + zl
// (bf16_split3, 24 significant bits each), k = 0..5 of the row operand carry
// -(h, h, m, h, l, m) / 2 against (zh, zm, zh, zl, zh, zm) in the column
// operand, and the MMA reads each row's eight values twice (its two K core
// matrices are the same bytes): every product of parts whose orders sum to
// <= 2, so the MMA adds -rs * zq to about 2^-24 relative (products are exact,
// sums fp32).
// The fold warps raise their register budget (setmaxnreg) to hold the 128
// accumulators; the others lower theirs.
// Epilogue: bf16 rows < M are stored; nothing else is written.
// Per-token mode (the "Numbers" section's PTOK GEMM: one activation scale As
// per token and partition, plain row-sums): the row warps load rs only, the
// fold is acc += (2^9 sc') * D'' (one packed operation per two elements) and
// the epilogue multiplies each row by its As.
// int5 weights ("2026-09-10: int5 W5A8 ParoQuant": low nibbles as for int4,
// fifth bits in [N][K/8] planes): each stage also receives the slab's
// 16-byte x 128-row fifth-bit box, the expansion writes the e4m3 bytes of
// (c - 16) * 2^-9 (expand16_int5), and zq drops its 8 sc term.
// Persistent grid: when the last round of tiles would fill at most half the
// grid, its tiles run as 128-row half items (per-group kernels only).
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
#include "pq_tcgen05.cuh"

namespace pq {
namespace {

constexpr int BM = 256, BN = 128, BK = 128;    // BM = two M=128 MMA halves
constexpr int kStages = 3;
constexpr int kFoldWarps = 8;     // warps 0..7: warp w folds rows 128(w/4) + 32(w%4)..+31, all columns
constexpr int kExpWarps = 4;      // warps 8..11
// row warps 12 and 13 (tile half 0, 1), TMA warp 14, MMA warp 15
constexpr int kRowWarp = 12, kTmaWarp = 14, kMmaWarp = 15;
constexpr int kThreads = 16 * 32;
constexpr uint32_t kFoldRegs = 216, kOtherRegs = 40;   // 256 * 216 + 256 * 40 = 65536
constexpr uint32_t kABytes = BM * BK;
constexpr uint32_t kBpBytes = BN * BK / 2;
constexpr uint32_t kBxBytes = BN * BK;
constexpr uint32_t kSzBytes = BN * 4;
constexpr uint32_t kTxBytes = kABytes + kBpBytes + kSzBytes;
constexpr uint32_t kTmemCols = 512;    // 2 buffers x 2 halves x 128 columns

// int5 weights: the fifth bits of the slab, 128 rows x 16 B (one bit per k)
constexpr uint32_t kBhBytes = BN * BK / 8;

template <int kBits>
struct __align__(1024) StageT {
    uint8_t a[kABytes];       // 256 rows x 128 B, SWIZZLE_128B (TMA); half h at 16 KB * h
    uint8_t bx[kBxBytes];     // 128 rows x 128 B, SWIZZLE_128B (expand warps)
    uint8_t bp[kBpBytes];     // 128 rows x 64 B packed nibbles (TMA)
    uint32_t sz[BN];          // f16 (sc, zscale) per column
    uint8_t bh[kBits == 5 ? kBhBytes : 16];   // int5: fifth-bit planes (TMA)
};

// A slab's scales and zero-point operands, in a ring of their own so a stage
// is free as soon as its MMAs complete (the fold lags the MMA).  The column
// part comes from the expansion warps; the row part is loaded from global
// memory by the row warps, which run up to a ring's depth ahead, so no
// global-load latency reaches the fold warps.
constexpr int kSzfRing = 4;
// The zero-point MMA's operands: K = 16 bf16, K-major without swizzle, 8-row
// x 16-byte core matrices 128 bytes apart along M/N.  The two core matrices
// along K are the same bytes (leading byte offset 0), so each row's eight
// values enter the sum twice; the row operand carries -rs / 2.
constexpr uint32_t kZLbo = 0, kZSbo = 128;
struct __align__(128) SzfSlot {
    uint8_t za[BM * 16];      // row operand: (h, h, m, h, l, m, 0, 0) of -rs / 2 (row warps)
    uint8_t zb[BN * 16];      // column operand: (zh, zm, zh, zl, zh, zm, 0, 0) of zq (expand warps)
    // 2^9 sc' per column and asg per tile row (0 past M; per-token: unused),
    // each stored in the order a fold thread reads them (col_slot, row_slot),
    // so that it loads a 32-column step's scales and its four rows' asg with
    // 16-byte loads, one conflict-free wavefront each
    float col[BN];
    float row[BM];
};
// column n: pair P = n / 2 is read by fold lane c4 = P % 4 in step cb = P / 16
// as element j = (P / 4) % 4 of its eight floats at (4 cb + c4) * 8
__device__ __forceinline__ int col_slot(int n) {
    const int P = n >> 1;
    return ((((P >> 4) * 4 + (P & 3)) * 4 + ((P >> 2) & 3)) << 1) + (n & 1);
}
// tile row 128 h + 32 q + 8 ri + g4 is read by fold warp (h, q), lane group g4,
// as element ri of its four floats at ((4 h + q) * 8 + g4) * 4
__device__ __forceinline__ int row_slot(int row) {
    const int h = row >> 7, q = (row >> 5) & 3, ri = (row >> 3) & 3, g4 = row & 7;
    return ((h * 4 + q) * 8 + g4) * 4 + ri;
}

struct Ctrl {
    uint64_t full_tma[kStages];
    uint64_t full_b[kStages];
    uint64_t empty[kStages];
    uint64_t szf_full[kSzfRing];
    uint64_t szf_empty[kSzfRing];
    uint64_t rows_full[kSzfRing];   // the row warps have written a slab's asg and zero-point row operand
    uint64_t tmem_full[2][2];     // [m-half][accumulator buffer]
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int abort;
    int issued;               // slabs the TMA producer issued (the drain after a give-up)
};

template <int kBits>
constexpr size_t smem_bytes() {
    return kStages * sizeof(StageT<kBits>) + kSzfRing * sizeof(SzfSlot) + sizeof(Ctrl) + 1024;
}
static_assert(smem_bytes<4>() <= 232448 && smem_bytes<5>() <= 232448, "shared memory per CTA");

struct TcParams {
    const float *asg;         // asg [P][G][M]; per-token: As [P][M]
    const float *rs;
    const uint32_t *sz;
    __nv_bfloat16 *y;
    unsigned int *status;
    int M, N, K, pb1, pb2, ldy;
    WaitBound wait;           // the pipeline waits' bound
};

// ---------------------------------------------------------------- PTX helpers
using namespace tc;
constexpr uint32_t kIdesc = idesc_f8(128, BN);     // one M=128 half x BN columns
constexpr uint32_t kIdescZ = idesc_bf16(128, BN);  // the zero-point MMA of a half

__device__ __forceinline__ void set_abort(Ctrl *ctl, unsigned int *status, unsigned int code) {
    if (status) atomicOr(status, code);
    *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
}

// Named barrier 1 over the whole CTA, reached by every role once it has left
// its loop.  From then on the abort flag is final, so the TMA producer and the
// MMA warp know whether the copies and MMAs they issued must still be waited
// for (a consumer that gave up never saw them land) before shared and tensor
// memory are released.  Those drain waits keep the full bound.
__device__ __forceinline__ void roles_done() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// Packed fp32 pair operations for the fold; not volatile, so the compiler
// interleaves the independent chains of a step.
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// The fold of one 16x256b.x4 load: four column pairs j for two rows (lo:
// d[4j], d[4j+1]; hi: d[4j+2], d[4j+3]).  The accumulator holds
// D'' = 2^-9 (sum_k dec(a) c - rs zq) of the slab (the zero-point MMA added
// the second term), so with z[j] = the (2^9 sc') pair of column pair j and
// sa = the row's asg splat:
//   acc += (sa * z) * D'' = asg * (sc' sum_k dec(a) c - zs8 rs)
// which is asg * (sc * D - zscale * rs) with D = sum over (c - 8) (int5:
// c - 16 is fed directly and zs8 = zscale).  Two packed operations per two
// elements.
__device__ __forceinline__ void fold_block(const uint32_t (&d)[16], const uint64_t (&z)[4], uint64_t *acc_lo,
                                           uint64_t *acc_hi, uint64_t sa_lo, uint64_t sa_hi) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc_lo[j] = ffma2(fmul2(sa_lo, z[j]), f2pack(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1])),
                          acc_lo[j]);
        acc_hi[j] = ffma2(fmul2(sa_hi, z[j]), f2pack(__uint_as_float(d[4 * j + 2]), __uint_as_float(d[4 * j + 3])),
                          acc_hi[j]);
    }
}

// The per-token fold: the token scale is applied in the epilogue, so
// acc += z * D'': one packed operation per two elements.
__device__ __forceinline__ void fold_block_tok(const uint32_t (&d)[16], const uint64_t (&z)[4], uint64_t *acc_lo,
                                               uint64_t *acc_hi) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc_lo[j] = ffma2(z[j], f2pack(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1])), acc_lo[j]);
        acc_hi[j] = ffma2(z[j], f2pack(__uint_as_float(d[4 * j + 2]), __uint_as_float(d[4 * j + 3])), acc_hi[j]);
    }
}

// Work items.  Tiles are numbered output-feature tile fastest; CTA c takes
// items c, c + gridDim.x, ...  When the last round would hold at most half
// the grid (rem = ntiles % gridDim.x <= gridDim.x / 2), its rem tiles become
// 2 rem half items of 128 rows each, so that round takes about half as long.
// A half item uses the M = 128 MMA half 0 and the fold warps of half 0; half
// 1's MMAs are not issued and its fold warps only keep the barriers in step.
// kSplit = false (the per-token kernel, where it measured slower) keeps whole
// tiles throughout.
template <bool kSplit>
__device__ __forceinline__ bool split_round(int ntiles) {
    const int C = (int)gridDim.x, rem = ntiles % C;
    return kSplit && rem > 0 && 2 * rem <= C;
}
template <bool kSplit>
__device__ __forceinline__ int item_count(int ntiles) {
    return split_round<kSplit>(ntiles) ? ntiles + ntiles % (int)gridDim.x : ntiles;
}
// Whether item i of this CTA is a half item (see tile_coords).
template <bool kSplit>
__device__ __forceinline__ bool is_half_item(int i, int ntiles) {
    return split_round<kSplit>(ntiles) && (int)blockIdx.x + i * (int)gridDim.x >= ntiles - ntiles % (int)gridDim.x;
}
// Item i of this CTA: n0, m0 (the item's first row), partition p, and
// half_item (true for a 128-row half item).
template <bool kSplit>
__device__ __forceinline__ void tile_coords(int i, int ntn, int ntiles, int pb1, int pb2, int &n0, int &m0,
                                            int &p, bool &half_item) {
    const int C = (int)gridDim.x, t = (int)blockIdx.x + i * C;
    const int rem = ntiles % C, nfull = ntiles - rem;
    int tile = t, hsel = 0;
    half_item = split_round<kSplit>(ntiles) && t >= nfull;
    if (half_item) {
        tile = nfull + ((t - nfull) >> 1);
        hsel = (t - nfull) & 1;
    }
    n0 = (tile % ntn) * BN;
    m0 = (tile / ntn) * BM + hsel * (BM / 2);
    p = (n0 >= pb1) + (n0 >= pb2);
}

// ---------------------------------------------------------------- kernel
// Persistent: CTA c walks tiles t = c, c + gridDim.x, ... (output-feature
// tile fastest, so the CTAs running at once share activation rows and the
// weight tiles stay L2-resident).  All pipelines run continuously across tile
// boundaries; slab counter it = (tile index) * G + kb.
template <bool kTok, int kBits>
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmH,
          const TcParams prm) {
    using Stage = StageT<kBits>;
    constexpr uint32_t kTx = kTxBytes + (kBits == 5 ? kBhBytes : 0u);
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (SWIZZLE_128B tiles), offset from the shared
    // array itself so that every access stays a shared-memory instruction
    const uint32_t smem_off = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((smem_off + 1023u) & ~1023u) - smem_off);
    Stage *stg = reinterpret_cast<Stage *>(base);
    SzfSlot *szf = reinterpret_cast<SzfSlot *>(base + kStages * sizeof(Stage));
    Ctrl *ctl = reinterpret_cast<Ctrl *>(base + kStages * sizeof(Stage) + kSzfRing * sizeof(SzfSlot));
    volatile int *abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = prm.M, G = prm.K / BK;
    const int ntn = prm.N / BN, ntiles = ntn * ((M + BM - 1) / BM);
    const int nitems = item_count<!kTok>(ntiles);
    const int my_tiles = (int)blockIdx.x < nitems ? (nitems - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_tiles * G;
    const int pb1 = prm.pb1, pb2 = prm.pb2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full_tma[s], 1);
            mbar_init(&ctl->full_b[s], kExpWarps);
            mbar_init(&ctl->empty[s], 1);            // the MMA commit
        }
        for (int r = 0; r < kSzfRing; ++r) {
            mbar_init(&ctl->szf_full[r], kExpWarps);
            mbar_init(&ctl->rows_full[r], 64);              // every lane of the two row warps
            mbar_init(&ctl->szf_empty[r], kFoldWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tmem_full[0][b], 1);
            mbar_init(&ctl->tmem_full[1][b], 1);
            mbar_init(&ctl->tmem_empty[b], kFoldWarps);
        }
        ctl->abort = 0;
        ctl->issued = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();
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

    if (warp >= kFoldWarps) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kTmaWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_map(&tmA);
            prefetch_map(&tmB);
            prefetch_map(&tmS);
            if constexpr (kBits == 5) prefetch_map(&tmH);
            // slab coordinates, stepped without divisions: tile ti of this
            // CTA, group kb
            int ti = 0, kb = 0, n0 = 0, m0 = 0, p = 0;
            bool half_item;
            if (total > 0) tile_coords<!kTok>(0, ntn, ntiles, pb1, pb2, n0, m0, p, half_item);
            auto next_slab = [&]() {
                if (++kb == G) {
                    kb = 0;
                    if (++ti < my_tiles) tile_coords<!kTok>(ti, ntn, ntiles, pb1, pb2, n0, m0, p, half_item);
                }
            };
            // first stages: weights and SZ (load-time tables) before the
            // preceding kernel has finished, activations after pdl_wait
            const int pre = total < kStages ? total : kStages;
            int pre_kb[kStages], pre_m0[kStages], pre_p[kStages];
            for (int it = 0; it < pre; ++it) {
                pre_kb[it] = kb;
                pre_m0[it] = m0;
                pre_p[it] = p;
                mbar_arrive_expect_tx(&ctl->full_tma[it], kTx);
                tma_load_2d(stg[it].bp, &tmB, kb * (BK / 2), n0, &ctl->full_tma[it]);
                tma_load_2d(stg[it].sz, &tmS, 8 * kb, n0 / 8, &ctl->full_tma[it]);
                if constexpr (kBits == 5) tma_load_2d(stg[it].bh, &tmH, kb * (BK / 8), n0, &ctl->full_tma[it]);
                next_slab();
            }
            pdl_wait();
            for (int it = 0; it < pre; ++it)
                tma_load_3d(stg[it].a, &tmA, pre_kb[it] * BK, pre_m0[it], pre_p[it], &ctl->full_tma[it]);
            int issued = pre;
            for (int it = pre, s = 0, par = 0; it < total; ++it) {   // s = it % kStages, par = (it / kStages - 1) & 1
                if (!wait_or_abort(&ctl->empty[s], (uint32_t)par, abort_flag, prm.wait)) {
                    set_abort(ctl, prm.status, kStatusWaitEmpty);
                    break;
                }
                mbar_arrive_expect_tx(&ctl->full_tma[s], kTx);
                tma_load_3d(stg[s].a, &tmA, kb * BK, m0, p, &ctl->full_tma[s]);
                tma_load_2d(stg[s].bp, &tmB, kb * (BK / 2), n0, &ctl->full_tma[s]);
                tma_load_2d(stg[s].sz, &tmS, 8 * kb, n0 / 8, &ctl->full_tma[s]);
                if constexpr (kBits == 5) tma_load_2d(stg[s].bh, &tmH, kb * (BK / 8), n0, &ctl->full_tma[s]);
                issued = it + 1;
                next_slab();
                if (++s == kStages) {
                    s = 0;
                    par ^= 1;
                }
            }
            ctl->issued = issued;
        }
        roles_done();
        if (*abort_flag && lane == 0) {   // after a give-up: every issued copy lands first
            const int issued = ctl->issued;
            for (int s = 0; s < kStages && s < issued; ++s) {
                const int last = (issued - 1 - s) / kStages;
                if (!mbar_wait(&ctl->full_tma[s], last & 1) && prm.status) atomicOr(prm.status, kStatusDrain);
            }
        }
    } else if (warp == kRowWarp || warp == kRowWarp + 1) {
        // ------------------------------------------------ per-row scales
        // asg and rs of a slab's rows into the slab's ring slot, up to a
        // ring's depth ahead: asg for the fold warps, and -rs / 2 split into
        // three bf16 parts as the zero-point MMA's row operand.  Row warp hw
        // covers tile half hw; lane l rows 128 hw + l + 32 u (u = 0..3).  The
        // loads of slab it + 1 are issued before slab it is stored, so their
        // latency overlaps the wait for the slab's slot.
        const int row0 = (BM / 2) * (warp - kRowWarp) + lane;
        const int rslot0 = row_slot(row0);    // row row0 + 32 u sits at rslot0 + 32 u
        pdl_wait();        // asg and rs are the preceding prologue's output
        int ti = 0, kb = 0, n0 = 0, m0 = 0, p = 0;   // the slab whose rows are loaded next
        bool half_item;
        uint32_t ok = 0;            // bit u: row row0 + 32 u of that slab's tile is below M
        size_t off = 0;             // (p * G + kb) * M
        auto tile_start = [&]() {
            tile_coords<!kTok>(ti, ntn, ntiles, pb1, pb2, n0, m0, p, half_item);
            ok = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) ok |= (m0 + row0 + 32 * u < M ? 1u : 0u) << u;
            off = (size_t)p * G * (size_t)M;
        };
        float av[4], rv[4];         // the slab it's asg and rs (0 past M)
        auto load = [&](float (&a)[4], float (&rr)[4]) {
            const float *ga = prm.asg + off + m0 + row0, *gr = prm.rs + off + m0 + row0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool v = (ok >> u) & 1u;
                a[u] = (!kTok && v) ? __ldg(ga + 32 * u) : 0.0f;
                rr[u] = v ? __ldg(gr + 32 * u) : 0.0f;
            }
            if (++kb == G) {
                kb = 0;
                if (++ti < my_tiles) tile_start();
            } else {
                off += (size_t)M;
            }
        };
        if (total > 0) {
            tile_start();
            load(av, rv);
        }
        for (int it = 0, r = 0, ruse = 0; it < total; ++it) {   // r = it % kSzfRing, ruse = it / kSzfRing
            float an[4], rn[4];
            if (it + 1 < total) load(an, rn);
            // lanes decide on their own (nothing below is warp-wide), so each
            // lane that gives up reports it
            if (ruse > 0 && !wait_or_abort(&ctl->szf_empty[r], (ruse - 1) & 1, abort_flag, prm.wait)) {
                set_abort(ctl, prm.status, kStatusWaitEmpty);
                break;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int row = row0 + 32 * u;
                if constexpr (!kTok) szf[r].row[rslot0 + 32 * u] = av[u];
                // rs = h + m + l (bf16 parts): the row operand (h, h, m, h, l, m)
                // of -rs / 2 against (zh, zm, zh, zl, zh, zm) in the column
                // operand; the MMA reads the eight values twice (kZLbo = 0), so
                // it adds -(every product of parts whose orders sum to <= 2) =
                // -rs * zq to about 2^-24 relative
                uint32_t h, m, l;
                bf16_split3(-0.5f * rv[u], h, m, l);
                *reinterpret_cast<uint4 *>(szf[r].za + (row >> 3) * kZSbo + (row & 7) * 16) =
                    make_uint4(h | (h << 16), m | (h << 16), l | (m << 16), 0u);
            }
            fence_proxy_async_smem();     // the row operand is read by the tensor core
            mbar_arrive(&ctl->rows_full[r]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                av[u] = an[u];
                rv[u] = rn[u];
            }
            if (++r == kSzfRing) {
                r = 0;
                ++ruse;
            }
        }
        roles_done();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (so the descriptors stay warp-uniform)
        // and one elected lane issues the MMAs and commits.  full_b implies
        // full_tma and the slab's row operand: the expand warps waited for
        // both before they arrived on full_b, after writing the column operand.
        int committed = 0;
        int tim = 0, kbm = 0;       // tile and group of slab it
        bool half_item = false;
        // the bounded waits below start their clocks only once the preceding
        // kernel has completed, so a long predecessor cannot run them out
        pdl_wait();
        for (int it = 0; it < total; ++it) {
            const int s = it % kStages, use = it / kStages;
            const int b = it & 1, tuse = it >> 1;
            const int r = it % kSzfRing;
            // the accumulator's first use waits on nothing: the phase before
            // the first reads as complete
            const bool ok = __all_sync(0xFFFFFFFFu,
                                       wait2_or_abort(&ctl->full_b[s], use & 1, &ctl->tmem_empty[b], (tuse - 1) & 1,
                                                      abort_flag, prm.wait));
            if (!ok) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull | kStatusWaitTmem);
                break;
            }
            tc_fence_after();
            const uint64_t ad0 = desc_sw128(smem_u32(stg[s].a));
            const uint64_t ad1 = desc_sw128(smem_u32(stg[s].a + kABytes / 2));
            const uint64_t bd = desc_sw128(smem_u32(stg[s].bx));
            const uint64_t za0 = desc_noswz(smem_u32(szf[r].za), kZLbo, kZSbo);
            const uint64_t za1 = desc_noswz(smem_u32(szf[r].za + BM * 8), kZLbo, kZSbo);
            const uint64_t zbd = desc_noswz(smem_u32(szf[r].zb), kZLbo, kZSbo);
            const uint32_t d0 = tmem + (uint32_t)(b * 2 * BN), d1 = d0 + BN;
            if (kbm == 0) half_item = is_half_item<!kTok>(tim, ntiles);   // once per tile
            if (elect_one()) {
                // half 0, then half 1, each committed on its own so the two
                // fold warp groups start half a slab apart; each half's chain
                // ends with the zero-point MMA (bf16, K = 16).  A half item
                // issues half 0 only; half 1's commit still signals its fold
                // warps, which then only release the buffer.
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk)   // +32 bytes along K inside the swizzle row
                    mma_f8(d0, ad0 + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, kk > 0 ? 1u : 0u);
                mma_bf16(d0, za0, zbd, kIdescZ, 1u);
                mma_commit(&ctl->tmem_full[0][b]);
                if (!half_item) {
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk)
                        mma_f8(d1, ad1 + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, kk > 0 ? 1u : 0u);
                    mma_bf16(d1, za1, zbd, kIdescZ, 1u);
                }
                // A stage that is never refilled gets no release: nothing would wait
                // for that arrival, and an arrival still in flight when the CTA
                // exits would land in the shared memory of the next CTA on this SM.
                if (it + kStages < total) mma_commit(&ctl->empty[s]);
                mma_commit(&ctl->tmem_full[1][b]);
            }
            __syncwarp();
            committed = it + 1;
            if (++kbm == G) {
                kbm = 0;
                ++tim;
            }
        }
        roles_done();
        if (*abort_flag && committed > 0 && lane == 0) {
            // after a give-up: the last slab's three commits land first (later
            // commits complete after earlier ones)
            const int it = committed - 1;
            if (!mbar_wait(&ctl->tmem_full[0][it & 1], (it >> 1) & 1) && prm.status)
                atomicOr(prm.status, kStatusDrain);
            if (!mbar_wait(&ctl->tmem_full[1][it & 1], (it >> 1) & 1) && prm.status)
                atomicOr(prm.status, kStatusDrain);
            if (it + kStages < total && !mbar_wait(&ctl->empty[it % kStages], (it / kStages) & 1) && prm.status)
                atomicOr(prm.status, kStatusDrain);
        }
    } else if (warp >= kFoldWarps && warp < kFoldWarps + kExpWarps) {
        // ------------------------------------------------ nibble expansion
        const int et = threadIdx.x - kFoldWarps * 32;    // 0..127
        const int chunk = et & 7;
        pdl_wait();        // as for the MMA warp: the wait clocks start after the predecessor
        for (int it = 0; it < total; ++it) {
            const int s = it % kStages, use = it / kStages;
            const int r = it % kSzfRing, ruse = it / kSzfRing;
            // the stage's copies, the ring slot free (its previous slab folded;
            // the phase before the first reads as complete) and the slab's row
            // operand written (so that full_b, below, implies it for the MMA);
            // warp-uniform, so the warp stays converged for its votes and syncs
            if (!__all_sync(0xFFFFFFFFu, wait3_or_abort(&ctl->full_tma[s], use & 1, &ctl->szf_empty[r],
                                                        (ruse - 1) & 1, &ctl->rows_full[r], ruse & 1, abort_flag,
                                                        prm.wait))) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                break;
            }
            Stage &st = stg[s];
            const uint32_t wcol = st.sz[et];   // column et's SZ word, read before full_b frees the stage
            // A column with sc = 0 dequantizes to -zscale whatever its codes, so
            // its codes must not reach the MMA: the fold then scales it by
            // 2^9 * 1 and the zero-point MMA alone gives -zscale * rs.  Lane l
            // checks row 4w + l % 4 + 16 (l / 4) of this warp's 32 rows.
            const bool any_zero_sc = __any_sync(
                0xFFFFFFFFu, (st.sz[4 * (et >> 5) + (lane & 3) + 16 * (lane >> 2)] & 0x7FFFu) == 0u);
            // the packed loads of a batch first (the stores below could alias
            // them as far as the compiler knows), then expand and store; int5
            // takes its eight rows in two batches of four, which keeps its
            // fifth-bit words within the role's 40 registers
            constexpr int kLoadBatch = kBits == 5 ? 4 : 8;
#pragma unroll
            for (int i0 = 0; i0 < 8; i0 += kLoadBatch) {
                uint2 pk[kLoadBatch];
                uint32_t hb[kLoadBatch];  // int5: the fifth-bit block word of the same 16 k, shifted for expand16_int5
#pragma unroll
                for (int u = 0; u < kLoadBatch; ++u) {
                    const int row = (et >> 3) + 16 * (i0 + u);
                    pk[u] = *reinterpret_cast<const uint2 *>(st.bp + row * (BK / 2) + chunk * 8);
                    if constexpr (kBits == 5)
                        hb[u] = *reinterpret_cast<const uint32_t *>(st.bh + row * (BK / 8) + (chunk >> 1) * 4) >>
                                (4 * (chunk & 1));
                }
#pragma unroll
                for (int u = 0; u < kLoadBatch; ++u) {
                    const int row = (et >> 3) + 16 * (i0 + u);
                    uint4 e;
                    if constexpr (kBits == 5)
                        e = expand16_int5(pk[u], hb[u]);
                    else
                        e = expand16(pk[u]);
                    if (any_zero_sc && (st.sz[row] & 0x7FFFu) == 0u) e = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(st.bx + row * BK + ((chunk ^ (row & 7)) << 4)) = e;
                }
            }
            // column et: the fold's 2^9 sc' (the MMA sums a * c * 2^-9, see
            // expand16; sc' = sc, or 1 where sc = 0) and the zero-point MMA's
            // column operand (zh, zm, zh, zl, zh, zm): the bf16 parts of
            // zq = 2^-9 zs8 / sc' with zs8 = zscale + 8 sc (int4: the MMA sums
            // raw c, so the -8 moves here; int5 feeds c - 16 itself, so
            // zs8 = zscale).  zq only corrects, so a quotient to 2 ulp (about
            // 2^-23 relative) is accurate enough.
            {
                const float sc = f16lo(wcol);
                const float sce = sc != 0.0f ? sc : 1.0f;
                const float zs8 = kBits == 5 ? f16hi(wcol) : f16hi(wcol) + 8.0f * sc;
                const float zq = __fdividef(zs8, sce) * (1.0f / kNibbleScale);
                uint32_t h, m, l;
                bf16_split3(zq, h, m, l);
                *reinterpret_cast<uint4 *>(szf[r].zb + (et >> 3) * kZSbo + (et & 7) * 16) =
                    make_uint4(h | (m << 16), h | (l << 16), h | (m << 16), 0u);
                szf[r].col[col_slot(et)] = kNibbleScale * sce;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctl->full_b[s]);
                mbar_arrive(&ctl->szf_full[r]);
            }
        }
        roles_done();
    } else if (warp < kFoldWarps) {
        // ------------------------------------------------ fold warps
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFoldRegs));
        // 16x256b TMEM loads: thread (g4, c4) of the warp holds rows
        // 128h + 32q + 8i + g4 (i = 0..3) and column pairs 8J + 2c4 (J = 0..15),
        // so each per-column scale load serves four rows.
        const int q = warp & 3, h = warp >> 2;
        const int g4 = lane >> 2, c4 = lane & 3;
        const int row0 = 128 * h + 32 * q + g4;
        pdl_wait();        // y may still be read by the preceding kernel
        bool bad = false;
        for (int i = 0; i < my_tiles; ++i) {
            int n0, m0, p;
            bool half_item;
            tile_coords<!kTok>(i, ntn, ntiles, pb1, pb2, n0, m0, p, half_item);
            const int mb = m0 + row0;     // rows mb + 8 * ri
            if (half_item && h == 1) {
                // a half item: nothing to fold here; keep the barriers in step
                for (int kb = 0; kb < G && !bad; ++kb) {
                    const int it = i * G + kb;
                    const int b = it & 1, tuse = it >> 1;
                    const int r = it % kSzfRing, ruse = it / kSzfRing;
                    if (!__all_sync(0xFFFFFFFFu, wait2_or_abort(&ctl->szf_full[r], ruse & 1, &ctl->tmem_full[h][b],
                                                                tuse & 1, abort_flag, prm.wait))) {
                        if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                        bad = true;
                        break;
                    }
                    tc_fence_after();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&ctl->tmem_empty[b]);
                        mbar_arrive(&ctl->szf_empty[r]);
                    }
                }
                if (i == my_tiles - 1) pdl_trigger();
                continue;
            }
            uint64_t acc[4][16];
#pragma unroll
            for (int ri = 0; ri < 4; ++ri)
#pragma unroll
                for (int J = 0; J < 16; ++J) acc[ri][J] = 0;
            for (int kb = 0; kb < G && !bad; ++kb) {
                const int it = i * G + kb;
                const int b = it & 1, tuse = it >> 1;
                const int r = it % kSzfRing, ruse = it / kSzfRing;
                // the slab's column values (szf_full; the expand warps arrived on
                // it after seeing the row warps' rows_full, so the row values
                // are there too) and its accumulator; warp-uniform: the TMEM
                // loads and syncs below need the whole warp
                if (!__all_sync(0xFFFFFFFFu, wait2_or_abort(&ctl->szf_full[r], ruse & 1, &ctl->tmem_full[h][b],
                                                            tuse & 1, abort_flag, prm.wait))) {
                    if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                    bad = true;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 2 * BN + h * BN);
                // four steps (32-column block cb), each two 16x256b.x4 loads
                // (16-lane halves sh = 0, 1) in flight behind one wait
                // per row: the asg splat (per-token: none, As is applied at the end)
                uint64_t sa2[4] = {0, 0, 0, 0};
                if constexpr (!kTok) {
                    const float4 v = *reinterpret_cast<const float4 *>(szf[r].row + row_slot(row0));
                    sa2[0] = f2pack(v.x, v.x);
                    sa2[1] = f2pack(v.y, v.y);
                    sa2[2] = f2pack(v.z, v.z);
                    sa2[3] = f2pack(v.w, v.w);
                }
                // column pairs 8 J + 2 c4 (J = 4 cb + j, j = 0..3) of step cb:
                // eight floats at (4 cb + c4) * 8 (col_slot)
                const float4 *cf = reinterpret_cast<const float4 *>(szf[r].col) + 2 * c4;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t d0[16], d1[16];
                    tmem_issue256(taddr + 32 * cb, d0);
                    tmem_issue256(taddr + ((uint32_t)16 << 16) + 32 * cb, d1);
                    uint64_t z[4];
                    {
                        const float4 v01 = cf[8 * cb], v23 = cf[8 * cb + 1];
                        z[0] = f2pack(v01.x, v01.y);
                        z[1] = f2pack(v01.z, v01.w);
                        z[2] = f2pack(v23.x, v23.y);
                        z[3] = f2pack(v23.z, v23.w);
                    }
                    tmem_wait32(d0, d1);
                    if (cb == 3) {       // every load of this buffer has completed
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctl->tmem_empty[b]);
                    }
                    if constexpr (kTok) {
                        fold_block_tok(d0, z, acc[0] + 4 * cb, acc[1] + 4 * cb);
                        fold_block_tok(d1, z, acc[2] + 4 * cb, acc[3] + 4 * cb);
                    } else {
                        fold_block(d0, z, acc[0] + 4 * cb, acc[1] + 4 * cb, sa2[0], sa2[1]);
                        fold_block(d1, z, acc[2] + 4 * cb, acc[3] + 4 * cb, sa2[2], sa2[3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->szf_empty[r]);
            }
            if (i == my_tiles - 1) pdl_trigger();
            bad = __any_sync(0xFFFFFFFFu, bad || *abort_flag != 0);     // one verdict per warp
            // epilogue: bf16 pairs (NaN once the CTA has aborted); per-token:
            // times the row's As first
#pragma unroll
            for (int ri = 0; ri < 4; ++ri) {
                if (mb + 8 * ri >= M) continue;
                uint32_t *dst = reinterpret_cast<uint32_t *>(prm.y + (size_t)(mb + 8 * ri) * prm.ldy + n0 + 2 * c4);
                float as = 1.0f;
                if constexpr (kTok) as = __ldg(prm.asg + (size_t)p * M + mb + 8 * ri);
#pragma unroll
                for (int J = 0; J < 16; ++J) {
                    float2 v = f2unpack(acc[ri][J]);
                    if constexpr (kTok) {
                        v.x *= as;
                        v.y *= as;
                    }
                    if (bad) v.x = v.y = __int_as_float(0x7FC00000);
                    const __nv_bfloat162 v2 = __floats2bfloat162_rn(v.x, v.y);
                    dst[4 * J] = *reinterpret_cast<const uint32_t *>(&v2);
                }
            }
        }
        roles_done();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side
}  // namespace

pq_status launch_gemm_tc(const void *a, const float *asg, const float *rs, int M, int N, int K,
                         int P, int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                         unsigned int *dev_status, void *stream, int sm_count, bool per_token,
                         const void *whi) {
    (void)sm_count;
    const bool int5 = whi != nullptr;
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
    CUtensorMap tmH = tmB;        // int4: never read
    if (int5) {
        // fifth-bit planes [N][K/8] bytes: box = one slab (16 B) of 128 rows
        const cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)(K / 8)};
        const cuuint32_t box[2] = {BK / 8, BN};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmH, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(whi), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for whi: CUresult %d", (int)r);
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
    prm.wait = pipeline_wait_bound();
    const long long ntiles = (long long)(N / BN) * ((M + BM - 1) / BM);
    if (ntiles > 0x7FFFFFFF) return fail(PQ_ERR_SHAPE, "pq_gemm_tc: M = %d too large", M);
    const int ctas = (int)(ntiles < sm_count ? ntiles : (sm_count > 0 ? sm_count : 1));
    const dim3 grid(ctas);
    auto kern = int5 ? (per_token ? tc_kernel<true, 5> : tc_kernel<false, 5>)
                     : (per_token ? tc_kernel<true, 4> : tc_kernel<false, 4>);
    const size_t smem = int5 ? smem_bytes<5>() : smem_bytes<4>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = launch_pdl(kern, grid, dim3(kThreads), smem, static_cast<cudaStream_t>(stream), tmA, tmB, tmS, tmH,
                   prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "tc launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

}  // namespace pq
