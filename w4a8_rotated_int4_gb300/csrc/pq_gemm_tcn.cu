// pq_gemm_tcn.cu -- narrow-M (decode band) uint4 x e4m3 group GEMM on the
// 5th-generation tensor cores, sm_103a.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Design"
// items 1 (zero point as a row-sum correction, SZ table), 2 (per-group fp8
// activation scales folded once per 128-k group) and 4 (partition select per
// n-block); int5 weights as in the prefill kernel ("2026-09-10: int5 W5A8
// ParoQuant": (c - 16) fed to the MMA, the correction -zscale), with the
// packed nibbles sharing their bytes with the expanded tile.  Same arithmetic
// as the prefill kernel; the operands swap roles so that a handful of tokens
// still fills the MMA:
//
//   D'[n][m] = sum_{k in group} c[n][k] * dec(a[m][k])     (c in 0..15, exact)
//   y[m][n] += asg[m,g] * (sc[g,n] * D' - (zscale + 8 sc)[g,n] * rs[m,g])
//
// One CTA owns 128 output features (the MMA's M = 128 rows are weight rows)
// and streams all K/128 groups of its weights; up to 16 tokens are the MMA's
// N = 16 columns (rows past M are zero-filled by the TMA).  Per group:
//   TMA warp     packed weights w[n0:+128][64g:+64], the group's SZ words and
//                the activation tile a[p][0:16][128g:+128] (SWIZZLE_128B)
//                into one of kStages stages.
//   expand warps nibble c -> the e4m3 byte of value c * 2^-9 (the nibble alone
//                in its byte) in the canonical K-major SWIZZLE_128B layout
//                (the MMA's A operand), and the SZ words -> fp32
//                (2^9 sc, -(zscale + 8 sc)) into a ring slot of their own.
//   row warp     cp.async of the group's per-token (asg, rs) into a deeper ring.
//   MMA warps    4 x tcgen05.mma m128n16k32 (kind::f8f6f4, fp32 accumulate)
//                into one of four 16-column TMEM accumulators (one per MMA warp).
//   fold warps   one thread per output feature: tcgen05.ld 32x32b.x16 and
//                acc[m] += asg[m] * (sc * D'[m] - zs8 * rs[m]) for m < M.
// The weights are read exactly once, so the kernel is bound by HBM when the
// grid covers the GPU.
//
// Every wait is bounded (%globaltimer); a wait that gives up marks the CTA as
// aborted, lets in-flight copies and MMAs finish, frees TMEM, writes NaN to
// its outputs and reports through the optional status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pq_device.cuh"
#include "pq_internal.h"
#include "pq_tcgen05.cuh"

namespace pq {
namespace {

using namespace tc;

constexpr int NN = 128;           // output features per CTA (the MMA's M)
constexpr int MT = 16;            // token columns (the MMA's N)
constexpr int BK = 128;           // one scale group per slab
constexpr int kStages = 8;
constexpr int kSzfRing = 4;       // column scales, written by the expand warps (slot = group)
constexpr int kRowRing = 16;      // per-token scales, copied by the row warp (latency of global loads)
// A single thread issues an MMA only every ~100 cycles, so four MMA warps
// (one per SM sub-partition) take turns: warp j issues the slabs it = j mod 4
// into TMEM accumulator j.
// TMA: issuing a tensor copy costs one thread ~120 cycles, so kTmaWarps
// producers take the slabs in turn (warp t fills the stages s = t mod kTmaWarps)
constexpr int kTmaWarps = 2, kRowWarp = kTmaWarps;
constexpr int kMmaWarp0 = kRowWarp + 1, kMmaWarps = 4;    // warps 3..6, one per sub-partition
// expansion: kExpGroups groups of 4 warps, group e expands slabs it = e mod kExpGroups,
// so that several slabs are expanded at once
constexpr int kExpWarp0 = kMmaWarp0 + kMmaWarps, kExpWarps = 4, kExpGroups = 4;   // warps 7..22
// fold: kFoldSets sets of 4 warps (warps 23..30), set f folds the slabs
// it = f mod kFoldSets into accumulators of its own, summed at the end; warp w
// reads TMEM lane quarter w % 4 (each set covers all four)
constexpr int kFoldWarp0 = kExpWarp0 + kExpWarps * kExpGroups, kFoldWarps = 4, kFoldSets = 2;
constexpr int kThreads = (kFoldWarp0 + kFoldWarps * kFoldSets) * 32;
// An mbarrier parity wait cannot tell phase u+1 from phase u-1, so a waiter must
// never wait for a barrier's next use before it has seen the previous one.  Each
// stage and each scale slot is therefore always served by the same expand group
// and the same MMA warp, which take their slabs in order.
static_assert(kStages % kExpGroups == 0 && kStages % kMmaWarps == 0 && kStages % kTmaWarps == 0,
              "stage ownership");
// TMEM accumulators: slab it uses buffer it % kTmemBufs, issued by MMA warp
// it % kMmaWarps and folded by set it % kFoldSets (each buffer keeps its owners)
constexpr int kTmemBufs = 8;
static_assert(kTmemBufs % kMmaWarps == 0 && kTmemBufs % kFoldSets == 0, "accumulator ownership");
constexpr uint32_t kBxBytes = NN * BK;        // expanded weights, 128 rows x 128 B
constexpr uint32_t kAaBytes = MT * BK;        // activations, 16 rows x 128 B
constexpr uint32_t kBpBytes = NN * BK / 2;    // packed weights, 128 rows x 64 B
constexpr uint32_t kSzBytes = NN * 4;
constexpr uint32_t kTxBytes = kBpBytes + kAaBytes + kSzBytes;
constexpr uint32_t kTmemCols = 128;           // 8 accumulators x 16 columns
constexpr uint32_t kIdescN = idesc_f8(NN, MT);

constexpr uint32_t kBhBytes = NN * BK / 8;    // int5: fifth bits, 128 rows x 16 B

template <int kBits>
struct __align__(1024) StageT {
    uint8_t bx[kBxBytes];     // SWIZZLE_128B, written by the expand warps
    uint8_t aa[kAaBytes];     // SWIZZLE_128B, written by the TMA
    uint8_t bp[kBpBytes];
    uint32_t sz[NN];
};
// int5 stages add the fifth-bit tile; to keep eight stages the packed nibbles
// share their bytes with the expanded tile (the expansion group reads all of
// them, meets on bp_read, then writes the tile over them).
template <>
struct __align__(1024) StageT<5> {
    union {
        uint8_t bx[kBxBytes];
        uint8_t bp[kBpBytes];
    };
    uint8_t aa[kAaBytes];
    uint32_t sz[NN];
    uint8_t bh[kBhBytes];     // fifth bits, 128 rows x 16 B (TMA)
};

struct __align__(16) SzfSlot {
    float2 col[NN];           // (sc[n], -(zscale[n] + 8 sc[n]))
};
struct __align__(16) RowSlot {
    float2 row[MT];           // (asg[m], rs[m]), 0 past M
};

struct Ctrl {
    uint64_t full_tma[kStages];
    uint64_t full_b[kStages];
    uint64_t empty[kStages];
    uint64_t bp_read[kStages];   // int5: the group's packed loads are done
    uint64_t szf_full[kSzfRing];
    uint64_t szf_empty[kSzfRing];
    uint64_t row_full[kRowRing];
    uint64_t row_empty[kRowRing];
    uint64_t tmem_full[kTmemBufs];
    uint64_t tmem_empty[kTmemBufs];
    uint32_t tmem_base;
    int abort;
};

template <int kBits>
constexpr size_t smem_bytes() {
    return kStages * sizeof(StageT<kBits>) + kSzfRing * sizeof(SzfSlot) + kRowRing * sizeof(RowSlot) +
           sizeof(Ctrl) + 1024;
}
static_assert(smem_bytes<4>() <= 227 * 1024 && smem_bytes<5>() <= 227 * 1024, "shared memory budget");
static_assert(kSzfRing % kExpGroups == 0 && kSzfRing % kFoldSets == 0 && kRowRing % kFoldSets == 0,
              "scale slot ownership");

struct TcnParams {
    const float *asg;
    const float *rs;
    __nv_bfloat16 *y;
    unsigned int *status;
    int M, N, K, pb1, pb2, ldy;
};

__device__ __forceinline__ void set_abort(Ctrl *ctl, unsigned int *status, unsigned int code) {
    if (status) atomicOr(status, code);
    *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
}

template <int kBits>
__global__ void __launch_bounds__(kThreads, 1)
tcn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmH,
           const TcnParams prm) {
    using Stage = StageT<kBits>;
    constexpr uint32_t kTx = kTxBytes + (kBits == 5 ? kBhBytes : 0u);
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (SWIZZLE_128B tiles), offset from the shared
    // array itself so that every access stays a shared-memory instruction
    const uint32_t smem_off = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((smem_off + 1023u) & ~1023u) - smem_off);
    Stage *stg = reinterpret_cast<Stage *>(base);
    SzfSlot *szf = reinterpret_cast<SzfSlot *>(base + kStages * sizeof(Stage));
    RowSlot *rows = reinterpret_cast<RowSlot *>(base + kStages * sizeof(Stage) + kSzfRing * sizeof(SzfSlot));
    Ctrl *ctl = reinterpret_cast<Ctrl *>(reinterpret_cast<uint8_t *>(rows) + kRowRing * sizeof(RowSlot));
    volatile int *abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = prm.M, G = prm.K / BK;
    const int n0 = blockIdx.x * NN;
    const int p = (n0 >= prm.pb1 ? 1 : 0) + (n0 >= prm.pb2 ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full_tma[s], 1);
            mbar_init(&ctl->full_b[s], kExpWarps);
            mbar_init(&ctl->empty[s], 1);            // the MMA commit
            mbar_init(&ctl->bp_read[s], kExpWarps);
        }
        for (int r = 0; r < kSzfRing; ++r) {
            mbar_init(&ctl->szf_full[r], kExpWarps);
            mbar_init(&ctl->szf_empty[r], kFoldWarps);
        }
        for (int r = 0; r < kRowRing; ++r) {
            mbar_init(&ctl->row_full[r], 32);               // the row warp's cp.async arrivals
            mbar_init(&ctl->row_empty[r], kFoldWarps);
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&ctl->tmem_full[b], 1);
            mbar_init(&ctl->tmem_empty[b], kFoldWarps);
        }
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp0) {
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
    pdl_trigger();     // the next kernel may start its own load-time prefetch

    if (warp < kTmaWarps) {
        // ------------------------------------------------ TMA producers
        if (lane == 0) {
            const int tw = warp;
            prefetch_map(&tmA);
            prefetch_map(&tmB);
            prefetch_map(&tmS);
            if constexpr (kBits == 5) prefetch_map(&tmH);
            // first stages: weights and SZ (load-time tables) before the
            // preceding kernel has finished, activations after pdl_wait
            const int pre = G < kStages ? G : kStages;
            int last = -1;             // the last slab this producer issued
            for (int it = tw; it < pre; it += kTmaWarps) {
                mbar_arrive_expect_tx(&ctl->full_tma[it], kTx);
                tma_load_2d(stg[it].bp, &tmB, it * (BK / 2), n0, &ctl->full_tma[it]);
                tma_load_2d(stg[it].sz, &tmS, 8 * it, n0 / 8, &ctl->full_tma[it]);
                if constexpr (kBits == 5) tma_load_2d(stg[it].bh, &tmH, it * (BK / 8), n0, &ctl->full_tma[it]);
            }
            pdl_wait();
            for (int it = tw; it < pre; it += kTmaWarps) {
                tma_load_3d(stg[it].aa, &tmA, it * BK, 0, p, &ctl->full_tma[it]);
                last = it;
            }
            for (int it = pre + tw; it < G; it += kTmaWarps) {   // pre is a multiple of kTmaWarps here
                const int s = it % kStages, use = it / kStages;
                if (!wait_or_abort(&ctl->empty[s], (use - 1) & 1, abort_flag)) {
                    set_abort(ctl, prm.status, kStatusWaitEmpty);
                    break;
                }
                mbar_arrive_expect_tx(&ctl->full_tma[s], kTx);
                tma_load_2d(stg[s].bp, &tmB, it * (BK / 2), n0, &ctl->full_tma[s]);
                tma_load_2d(stg[s].sz, &tmS, 8 * it, n0 / 8, &ctl->full_tma[s]);
                if constexpr (kBits == 5) tma_load_2d(stg[s].bh, &tmH, it * (BK / 8), n0, &ctl->full_tma[s]);
                tma_load_3d(stg[s].aa, &tmA, it * BK, 0, p, &ctl->full_tma[s]);
                last = it;
            }
            if (*abort_flag) {   // let this producer's copies land before shared memory is released
                for (int it = last; it >= 0 && it > last - kStages; it -= kTmaWarps) {
                    if (!mbar_wait(&ctl->full_tma[it % kStages], (it / kStages) & 1) && prm.status)
                        atomicOr(prm.status, kStatusDrain);
                }
            }
        }
    } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMmaWarps) {
        // ------------------------------------------------ MMA issuers
        // full_b implies full_tma: the expand warps waited for the stage's
        // copies (activations included) before they arrived on full_b
        // The whole warp runs the loop (so the descriptors stay warp-uniform)
        // and one elected lane issues the MMAs and commits.
        const int j = warp - kMmaWarp0;
        int committed = -1;
        // the bounded waits below start their clocks only once the preceding
        // kernel has completed, so a long predecessor cannot run them out
        pdl_wait();
        for (int it = j; it < G; it += kMmaWarps) {
            const int s = it % kStages, use = it / kStages;
            const int b = it % kTmemBufs, tuse = it / kTmemBufs;
            // full_b, and the accumulator's release by the fold (its first use
            // waits on nothing: the phase before the first reads as complete)
            const bool ok = __all_sync(0xFFFFFFFFu,
                                       wait2_or_abort(&ctl->full_b[s], use & 1, &ctl->tmem_empty[b], (tuse - 1) & 1,
                                                      abort_flag));
            if (!ok) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull | kStatusWaitTmem);
                break;
            }
            tc_fence_after();
            const uint64_t ad = desc_sw128(smem_u32(stg[s].bx));
            const uint64_t bd = desc_sw128(smem_u32(stg[s].aa));
            const uint32_t d = tmem + (uint32_t)(b * MT);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk)   // +32 bytes along K inside the swizzle row
                    mma_f8(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdescN, kk > 0 ? 1u : 0u);
                // A stage that is never refilled gets no release: nothing would wait
                // for that arrival, and an arrival still in flight when the CTA
                // exits would land in the shared memory of the next CTA on this SM.
                if (it + kStages < G) mma_commit(&ctl->empty[s]);
                mma_commit(&ctl->tmem_full[b]);
            }
            __syncwarp();
            committed = it;
        }
        if (*abort_flag && committed >= 0 && lane == 0) {   // MMAs and their arrivals must land before exit
            if (!mbar_wait(&ctl->tmem_full[committed % kTmemBufs], (committed / kTmemBufs) & 1) && prm.status)
                atomicOr(prm.status, kStatusDrain);
            if (committed + kStages < G &&
                !mbar_wait(&ctl->empty[committed % kStages], (committed / kStages) & 1) && prm.status)
                atomicOr(prm.status, kStatusDrain);
        }
    } else if (warp == kRowWarp) {
        // ------------------------------------------------ per-token scales
        pdl_wait();        // asg and rs are the preceding prologue's output
        for (int it = 0; it < G; ++it) {
            const int r = it % kRowRing, ruse = it / kRowRing;
            if (ruse > 0 && !wait_or_abort(&ctl->row_empty[r], (ruse - 1) & 1, abort_flag)) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitEmpty);
                break;
            }
            if (lane < MT) {
                const size_t off = ((size_t)p * G + (size_t)it) * (size_t)M;
                const bool ok = lane < M;     // tokens past M are zero-filled
                cp_async4(&rows[r].row[lane].x, ok ? prm.asg + off + lane : prm.asg, ok);
                cp_async4(&rows[r].row[lane].y, ok ? prm.rs + off + lane : prm.rs, ok);
            }
            cp_async_arrive(&ctl->row_full[r]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy outlives the CTA
    } else if (warp >= kExpWarp0 && warp < kExpWarp0 + kExpWarps * kExpGroups) {
        // ------------------------------------------------ nibble expansion
        const int eg = (warp - kExpWarp0) / kExpWarps;   // this warp's group
        const int et = threadIdx.x - (kExpWarp0 + kExpWarps * eg) * 32;   // 0..127
        const int chunk = et & 7;
        pdl_wait();        // as for the MMA warps: the wait clocks start after the predecessor
        for (int it = eg; it < G; it += kExpGroups) {
            const int s = it % kStages, use = it / kStages;
            if (!wait_or_abort(&ctl->full_tma[s], use & 1, abort_flag)) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                break;
            }
            Stage &st = stg[s];
            uint32_t w0 = 0, w1 = 0;
            if (et < NN / 2) {            // read the SZ words now: the stage may be refilled after full_b
                w0 = st.sz[2 * et];
                w1 = st.sz[2 * et + 1];
            }
            // all eight packed loads first (the stores below could alias them
            // as far as the compiler knows), then expand and store
            uint2 pk[8];
            uint32_t hb[8];           // int5: the fifth bits of the same 16 k
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pk[i] = *reinterpret_cast<const uint2 *>(st.bp + ((et >> 3) + 16 * i) * (BK / 2) + chunk * 8);
                if constexpr (kBits == 5)
                    hb[i] = *reinterpret_cast<const uint16_t *>(st.bh + ((et >> 3) + 16 * i) * (BK / 8) + chunk * 2);
            }
            if constexpr (kBits == 5) {
                // bp and bx share bytes: every warp of the group has its packed
                // words in registers before any warp overwrites them.  A stage's
                // next use needs the MMA of this one, which needs all four
                // warps past this wait, so the parity never aliases.
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->bp_read[s]);
                if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&ctl->bp_read[s], use & 1, abort_flag))) {
                    if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                    break;
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = (et >> 3) + 16 * i;
                uint4 e;
                if constexpr (kBits == 5)
                    e = expand16_int5(pk[i], hb[i]);
                else
                    e = expand16(pk[i]);
                *reinterpret_cast<uint4 *>(st.bx + row * BK + ((chunk ^ (row & 7)) << 4)) = e;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->full_b[s]);
            // fp32 column scales for the fold, into the ring slot of this group
            const int r = it % kSzfRing, ruse = it / kSzfRing;
            if (ruse > 0 && !wait_or_abort(&ctl->szf_empty[r], (ruse - 1) & 1, abort_flag)) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                break;
            }
            if (et < NN / 2) {
                const float sc0 = f16lo(w0), sc1 = f16lo(w1);
                // word j of the slab's SZ box is octet j / 8, column j % 8: column n = j
                // the MMA sums a * c * 2^-9 (expand16), so sc carries 2^9; int5
                // feeds c - 16 itself (expand16_int5), so its correction is zscale
                const float o8 = kBits == 5 ? 0.0f : 8.0f;
                szf[r].col[2 * et] = make_float2(kNibbleScale * sc0, -(f16hi(w0) + o8 * sc0));
                szf[r].col[2 * et + 1] = make_float2(kNibbleScale * sc1, -(f16hi(w1) + o8 * sc1));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->szf_full[r]);
        }
    } else if (warp >= kFoldWarp0 && warp < kFoldWarp0 + kFoldWarps * kFoldSets) {
        // ------------------------------------------------ fold warps
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int n = 32 * q + lane;         // output feature within the tile
        const int fs = (warp - kFoldWarp0) / kFoldWarps;
        pdl_wait();        // y may still be read by the preceding kernel
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        bool bad = false;
        for (int it = fs; it < G; it += kFoldSets) {
            const int b = it % kTmemBufs, tuse = it / kTmemBufs;
            const int r = it % kSzfRing, ruse = it / kSzfRing;
            const int rr = it % kRowRing, rruse = it / kRowRing;
            if (!wait3_or_abort(&ctl->row_full[rr], rruse & 1, &ctl->szf_full[r], ruse & 1,
                                &ctl->tmem_full[b], tuse & 1, abort_flag)) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                bad = true;
                break;
            }
            tc_fence_after();
            uint32_t d[16];
            tmem_issue32x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * MT), d);
            const float2 cz = szf[r].col[n];
            tmem_wait16(d);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tmem_empty[b]);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    const float2 rv = rows[rr].row[m];    // (asg, rs), the same for every lane
                    const float t = fmaf(cz.y, rv.y, cz.x * __uint_as_float(d[m]));
                    acc[m] = fmaf(rv.x, t, acc[m]);
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctl->szf_empty[r]);
                mbar_arrive(&ctl->row_empty[rr]);
            }
        }
        // the sets meet in shared memory, in stage 0's expanded-weight buffer:
        // it is free only once BOTH sets have seen their last slab (then every
        // expansion and MMA has completed) -- a set that finishes first must
        // not write while the other set's last slab may still be in stage 0
        float *part = reinterpret_cast<float *>(stg[0].bx);      // [kFoldSets - 1][MT][NN]
        asm volatile("bar.sync 1, %0;" ::"n"(kFoldWarps * kFoldSets * 32) : "memory");
        if (fs > 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) part[((fs - 1) * MT + m) * NN + n] = acc[m];
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kFoldWarps * kFoldSets * 32) : "memory");
        if (fs == 0) {
            bad = bad || *abort_flag != 0;
            for (int f = 1; f < kFoldSets; ++f) {
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] += part[((f - 1) * MT + m) * NN + n];
            }
            // epilogue: one bf16 per token (NaN once the CTA has aborted)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    const float v = bad ? __int_as_float(0x7FC00000) : acc[m];
                    prm.y[(size_t)m * prm.ldy + n0 + n] = __float2bfloat16_rn(v);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
}

}  // namespace

pq_status launch_gemm_tcn(const void *a, const float *asg, const float *rs, int M, int N, int K,
                          int P, int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                          unsigned int *dev_status, void *stream, const void *whi) {
    if (M > MT) return fail(PQ_ERR_SHAPE, "pq_gemm_tcn: M = %d > %d", M, MT);
    const bool int5 = whi != nullptr;
    auto enc = encode_fn();
    if (!enc) return fail(PQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    CUtensorMap tmA, tmB, tmS;
    {
        // activations [P][M][K]; a box of 16 token rows, rows past M read as zero
        const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)M, (cuuint64_t)P};
        const cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)K * (cuuint64_t)M};
        const cuuint32_t box[3] = {BK, MT, 1};
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
        const cuuint32_t box[2] = {BK / 2, NN};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(w), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for w: CUresult %d", (int)r);
    }
    {
        // SZ table [N/8][G][8] words: box = the 8 words of one group for 16 octets
        const cuuint64_t dims[2] = {(cuuint64_t)(8 * (K / 128)), (cuuint64_t)(N / 8)};
        const cuuint64_t strides[1] = {(cuuint64_t)(32 * (K / 128))};
        const cuuint32_t box[2] = {8, NN / 8};
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
        const cuuint32_t box[2] = {BK / 8, NN};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmH, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(whi), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for whi: CUresult %d", (int)r);
    }
    TcnParams prm{};
    prm.asg = asg;
    prm.rs = rs;
    prm.y = static_cast<__nv_bfloat16 *>(y);
    prm.status = dev_status;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.pb1 = pb1;
    prm.pb2 = pb2;
    prm.ldy = ldy;
    auto kern = int5 ? tcn_kernel<5> : tcn_kernel<4>;
    const size_t smem = int5 ? smem_bytes<5>() : smem_bytes<4>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = launch_pdl(kern, dim3(N / NN), dim3(kThreads), smem, static_cast<cudaStream_t>(stream), tmA, tmB, tmS,
                   tmH, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PQ_ERR_CUDA, "tcn launch: %s", cudaGetErrorString(e));
    return PQ_OK;
}

}  // namespace pq
