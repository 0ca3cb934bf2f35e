// pq_gemm_tcn.cu -- narrow-M (decode band) uint4 x e4m3 group GEMM on the
// 5th-generation tensor cores, sm_103a.
//
// Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Design"
// items 1 (zero point as a row-sum correction, SZ table), 2 (per-group fp8
// activation scales folded once per 128-k group) and 4 (partition select per
// n-block); int5 weights as in the prefill kernel ("2026-09-10: int5 W5A8
// ParoQuant": (c - 16) fed to the MMA, the correction -zscale).  Same arithmetic
// as the prefill kernel; the operands swap roles so that a handful of tokens
// still fills the MMA:
//
//   D'[n][m] = sum_{k in group} c[n][k] * dec(a[m][k])     (c in 0..15, exact)
//   y[m][n] += asg[m,g] * (sc[g,n] * D' - (zscale + 8 sc)[g,n] * rs[m,g])
//
// One CTA owns 128 output features (the MMA's M = 128 rows are weight rows)
// and streams all K/128 groups ("slabs") of its weights; up to 16 tokens are
// the MMA's N = 16 columns (rows past M are zero-filled by the TMA).  Roles:
//   weight TMA   two warps take the slabs in turn: packed weights
//                w[n0:+128][64g:+64], the slab's SZ words (and int5 fifth
//                bits) into the weight ring, which an expand group frees as
//                soon as it has read the slab into registers -- so the weight
//                stream runs up to a ring's depth ahead of the MMAs
//   act. TMA     the activation tile a[p][0:16][128g:+128] (SWIZZLE_128B) into
//                the operand ring, whose slots the MMAs free
//   expand warps 4 groups of 4 warps, group e takes slabs g = e mod 4: nibble
//                c -> the e4m3 byte of value c * 2^-9 (the nibble alone in its
//                byte) in the canonical K-major SWIZZLE_128B layout (the MMA's
//                A operand) in the operand ring, and the slab's SZ words into
//                a batch slot for the fold
//   row warp     cp.async of each batch's per-token (asg, rs)
//   MMA warps    4 warps, warp j takes slabs g = j mod 4: 4 x tcgen05.mma
//                m128n16k32 (kind::f8f6f4, fp32 accumulate) into column
//                block j of the batch's TMEM buffer
//   fold warps   2 sets of 4, set f takes batches f mod 2 (a batch is 4
//                consecutive slabs): one thread per output feature, one
//                barrier test per batch, tcgen05.ld 32x32b.x16 per slab and
//                acc[m] += asg[m] * (2^9 sc * D'[m] - zs8 * rs[m]) for m < M.
// Thread 0 issues the first ring of weight copies as soon as the barriers are
// initialised, ahead of the TMEM allocation, and the dependent launch is
// triggered only after the fold loop: a CTA fills its SM, and a dependent grid
// launched earlier crowds onto the SMs this grid leaves idle.
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

// Two rings.  A slab's packed weights only feed the expansion, so they sit in
// the weight ring only until the expansion has read them; the expanded tile
// and the activation tile feed the MMA and sit in the operand ring until its
// MMAs complete.  The weight ring is therefore free to run far ahead of the
// MMAs and hides the HBM latency, while the operand ring only spans
// expansion -> MMA.
// A weight slot holds kWSlabs consecutive slabs: one box of 128 rows x
// (64 kWSlabs) bytes.  One slab per slot measured fastest (two gave fewer,
// larger copies and a slower stream).
constexpr int kWSlabs = 1;
// int5 weight slots carry the fifth-bit planes too, so int5 keeps four of them
// to leave room for eight operand slots.  (Four operand slots measured slower;
// a version with four once raced because a weight slot was released to the
// TMA after generic reads with no proxy fence, which every release now has.)
template <int kBits>
constexpr int kWSlotsOf = kBits == 5 ? 4 : 8;   // weight ring (packed weights, SZ words, fifth bits), kWSlabs slabs each
template <int kBits>
constexpr int kXSlotsOf = 8;      // operand ring (expanded tile, activation tile)
// Accumulators, column scales and per-token scales are handed to the fold in
// batches of kBatch consecutive slabs (slab it belongs to batch it / kBatch),
// so each fold set tests one set of barriers per batch instead of per slab.
constexpr int kBatch = 4;
constexpr int kSzfSlots = 2;      // batch slots of raw SZ words, written by the expand warps
constexpr int kRowSlots = 4;      // batch slots of per-token scales, copied by the row warp
// Warps.  Issuing a tensor copy costs one thread ~120 cycles, so two weight
// producers take the slabs in turn; a third producer loads activation tiles
// as operand slots free up.  A single thread issues an MMA only every ~100
// cycles, so four MMA warps (one per SM sub-partition) take turns: warp j
// issues the slabs it = j mod 4.
constexpr int kTmaWWarps = 2, kTmaAWarp = kTmaWWarps, kRowWarp = kTmaAWarp + 1;
constexpr int kMmaWarp0 = kRowWarp + 1, kMmaWarps = 4;                               // warps 4..7
// expansion: kExpGroups groups of 4 warps, group e expands slabs it = e mod kExpGroups
constexpr int kExpWarp0 = kMmaWarp0 + kMmaWarps, kExpWarps = 4, kExpGroups = 4;   // warps 8..23
// fold: kFoldSets sets of 4 warps (warps 24..31), set f folds the batches
// k = f mod kFoldSets into accumulators of its own, summed at the end; warp w
// reads TMEM lane quarter w % 4 (each set covers all four)
constexpr int kFoldWarp0 = kExpWarp0 + kExpWarps * kExpGroups, kFoldWarps = 4, kFoldSets = 2;
constexpr int kThreads = (kFoldWarp0 + kFoldWarps * kFoldSets) * 32;
static_assert(kThreads <= 1024, "block size");
// An mbarrier parity wait cannot tell phase u+1 from phase u-1, so a waiter must
// never wait for a barrier's next use before it has seen the previous one.  Each
// slot is therefore always served by the same expand group, MMA warp and
// producer, which take their slabs in order.
static_assert((kWSlotsOf<4> * kWSlabs) % kExpGroups == 0 && (kWSlotsOf<5> * kWSlabs) % kExpGroups == 0 &&
                  kExpGroups % kWSlabs == 0 && kWSlotsOf<4> % kTmaWWarps == 0 && kWSlotsOf<5> % kTmaWWarps == 0 &&
                  kXSlotsOf<4> % kExpGroups == 0 && kXSlotsOf<5> % kExpGroups == 0 &&
                  kXSlotsOf<4> % kMmaWarps == 0 && kXSlotsOf<5> % kMmaWarps == 0,
              "slot ownership");
// TMEM accumulators: batch k uses buffer k % kTmemBufs (kBatch x 16 columns,
// slab it of the batch at column 16 (it % kBatch)); fold set f folds the
// batches k = f mod kFoldSets (each buffer and slot keeps its owners)
constexpr int kTmemBufs = 4;
static_assert(kBatch == kMmaWarps && kBatch == kExpGroups, "one slab of each batch per MMA warp and expand group");
static_assert(kTmemBufs % kFoldSets == 0 && kSzfSlots % kFoldSets == 0 && kRowSlots % kFoldSets == 0,
              "accumulator and slot ownership");
constexpr uint32_t kBxBytes = NN * BK;        // expanded weights, 128 rows x 128 B
constexpr uint32_t kAaBytes = MT * BK;        // activations, 16 rows x 128 B
constexpr uint32_t kBpBytes = NN * BK / 2;    // packed weights, 128 rows x 64 B
constexpr uint32_t kSzBytes = NN * 4;
constexpr uint32_t kBhBytes = NN * BK / 8;    // int5: fifth bits, 128 rows x 16 B
constexpr uint32_t kTmemCols = kTmemBufs * kBatch * MT;   // 4 buffers x 4 slabs x 16 columns = 256
constexpr uint32_t kIdescN = idesc_f8(NN, MT);

template <int kBits>
struct __align__(128) WSlotT {
    uint8_t bp[kWSlabs * kBpBytes];     // 128 rows x (64 kWSlabs) B packed nibbles (TMA)
    uint32_t sz[kWSlabs * NN];          // SZ words: octet o, slab u, column c at (o * kWSlabs + u) * 8 + c (TMA)
    uint8_t bh[kBits == 5 ? kWSlabs * kBhBytes : 16];   // int5: fifth bits, 128 rows x (16 kWSlabs) B (TMA)
};
struct __align__(1024) XSlot {
    uint8_t bx[kBxBytes];     // SWIZZLE_128B, written by the expand warps
    uint8_t aa[kAaBytes];     // SWIZZLE_128B, written by the TMA
};
constexpr uint32_t kTxW4 = kWSlabs * (kBpBytes + kSzBytes), kTxW5 = kTxW4 + kWSlabs * kBhBytes;

struct __align__(16) SzfSlot {
    uint32_t w[kBatch][NN];   // SZ word (f16 sc | f16 zscale << 16) of column n, per slab of the batch
};
struct __align__(16) RowSlot {
    float2 row[kBatch][MT];   // (asg[m], rs[m]) per slab of the batch, 0 past M
};

constexpr int kWMax = 8, kXMax = 8;
struct Ctrl {
    uint64_t w_full[kWMax];        // a slab's weights have landed (TMA transaction count)
    uint64_t w_empty[kWMax];       // the expand group has read them
    uint64_t x_full_a[kXMax];      // the activation tile has landed (TMA)
    uint64_t x_full_b[kXMax];      // the expanded tile is written
    uint64_t x_empty[kXMax];       // the slab's MMAs have completed
    uint64_t szf_full[kSzfSlots];
    uint64_t szf_empty[kSzfSlots];
    uint64_t row_full[kRowSlots];
    uint64_t row_empty[kRowSlots];
    uint64_t tmem_full[kTmemBufs];
    uint64_t tmem_empty[kTmemBufs];
    uint64_t drain[kMmaWarps];     // abort only: an MMA warp's last commit
    uint32_t tmem_base;
    int abort;
};

template <int kBits>
constexpr size_t smem_bytes() {
    return kXSlotsOf<kBits> * sizeof(XSlot) + kWSlotsOf<kBits> * sizeof(WSlotT<kBits>) +
           kSzfSlots * sizeof(SzfSlot) + kRowSlots * sizeof(RowSlot) + sizeof(Ctrl) + 1024;
}
static_assert(smem_bytes<4>() <= 227 * 1024 && smem_bytes<5>() <= 227 * 1024, "shared memory budget");

struct TcnParams {
    const float *asg;
    const float *rs;
    __nv_bfloat16 *y;
    unsigned int *status;
    int M, N, K, pb1, pb2, ldy;
    WaitBound wait;           // the pipeline waits' bound
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
    using WSlot = WSlotT<kBits>;
    constexpr int kW = kWSlotsOf<kBits>, kX = kXSlotsOf<kBits>;
    constexpr uint32_t kTxW = kBits == 5 ? kTxW5 : kTxW4;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (SWIZZLE_128B tiles), offset from the shared
    // array itself so that every access stays a shared-memory instruction
    const uint32_t smem_off = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((smem_off + 1023u) & ~1023u) - smem_off);
    XSlot *xs = reinterpret_cast<XSlot *>(base);
    WSlot *ws = reinterpret_cast<WSlot *>(base + kX * sizeof(XSlot));
    SzfSlot *szf = reinterpret_cast<SzfSlot *>(base + kX * sizeof(XSlot) + kW * sizeof(WSlot));
    RowSlot *rows = reinterpret_cast<RowSlot *>(reinterpret_cast<uint8_t *>(szf) + kSzfSlots * sizeof(SzfSlot));
    Ctrl *ctl = reinterpret_cast<Ctrl *>(reinterpret_cast<uint8_t *>(rows) + kRowSlots * sizeof(RowSlot));
    volatile int *abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = prm.M, G = prm.K / BK;
    const int nbatch = (G + kBatch - 1) / kBatch;
    const int nwb = (G + kWSlabs - 1) / kWSlabs;     // weight blocks of kWSlabs slabs
    const int n0 = blockIdx.x * NN;
    const int p = (n0 >= prm.pb1 ? 1 : 0) + (n0 >= prm.pb2 ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kW; ++s) {
            mbar_init(&ctl->w_full[s], 1);
            mbar_init(&ctl->w_empty[s], kExpWarps * kWSlabs);   // the expand groups of the slot's slabs
        }
        for (int s = 0; s < kX; ++s) {
            mbar_init(&ctl->x_full_a[s], 1);
            mbar_init(&ctl->x_full_b[s], kExpWarps);
            mbar_init(&ctl->x_empty[s], 1);            // the MMA commit
        }
        for (int r = 0; r < kSzfSlots; ++r) {
            mbar_init(&ctl->szf_full[r], kExpWarps * kExpGroups);   // every expand warp, once per batch
            mbar_init(&ctl->szf_empty[r], kFoldWarps);
        }
        for (int r = 0; r < kRowSlots; ++r) {
            mbar_init(&ctl->row_full[r], 32);               // the row warp's cp.async arrivals
            mbar_init(&ctl->row_empty[r], kFoldWarps);
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&ctl->tmem_full[b], kMmaWarps);       // one commit (or arrival) per MMA warp and batch
            mbar_init(&ctl->tmem_empty[b], kFoldWarps);
        }
        for (int w = 0; w < kMmaWarps; ++w) mbar_init(&ctl->drain[w], 1);
        ctl->abort = 0;
        fence_mbar_init();
        // The first ring's worth of weight blocks, before the tensor-memory
        // allocation and the block-wide barrier: load-time tables that need no
        // wait, so the first HBM round trip overlaps the CTA's setup.  The
        // producers below continue from block kW on.
        prefetch_map(&tmB);
        prefetch_map(&tmS);
        if constexpr (kBits == 5) prefetch_map(&tmH);
        for (int wb = 0; wb < kW && wb < nwb; ++wb) {
            const int it = wb * kWSlabs;
            mbar_arrive_expect_tx(&ctl->w_full[wb], kTxW);
            tma_load_2d(ws[wb].bp, &tmB, it * (BK / 2), n0, &ctl->w_full[wb]);
            tma_load_2d(ws[wb].sz, &tmS, 8 * it, n0 / 8, &ctl->w_full[wb]);
            if constexpr (kBits == 5) tma_load_2d(ws[wb].bh, &tmH, it * (BK / 8), n0, &ctl->w_full[wb]);
        }
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

    // the last block (weight producers) or slab (activation producer) issued
    // and the last slab an MMA warp committed, for the drain after a give-up
    int last = -1;
    if (warp < kTmaWWarps) {
        // ------------------------------------------------ weight producers
        // Weights, SZ words and fifth bits are load-time tables, not written by
        // the preceding kernel, so they stream without waiting for it.
        if (lane == 0) {
            const int tw = warp;
            // weight block wb = slabs kWSlabs wb .. +kWSlabs-1 (a box past K
            // reads as zero); this warp owns the blocks wb = tw (mod
            // kTmaWWarps), those below kW issued at the start by thread 0
            for (int wb = tw; wb < kW && wb < nwb; wb += kTmaWWarps) last = wb;
            for (int wb = tw + kW; wb < nwb; wb += kTmaWWarps) {
                const int s = wb % kW, use = wb / kW;
                if (use > 0 && !wait_or_abort(&ctl->w_empty[s], (use - 1) & 1, abort_flag, prm.wait)) {
                    set_abort(ctl, prm.status, kStatusWaitEmpty);
                    break;
                }
                const int it = wb * kWSlabs;
                mbar_arrive_expect_tx(&ctl->w_full[s], kTxW);
                tma_load_2d(ws[s].bp, &tmB, it * (BK / 2), n0, &ctl->w_full[s]);
                tma_load_2d(ws[s].sz, &tmS, 8 * it, n0 / 8, &ctl->w_full[s]);
                if constexpr (kBits == 5) tma_load_2d(ws[s].bh, &tmH, it * (BK / 8), n0, &ctl->w_full[s]);
                last = wb;
            }
        }
    } else if (warp == kTmaAWarp) {
        // ------------------------------------------------ activation producer
        if (lane == 0) {
            prefetch_map(&tmA);
            pdl_wait();        // the activations are the preceding prologue's output
            for (int it = 0; it < G; ++it) {
                const int s = it % kX, use = it / kX;
                if (use > 0 && !wait_or_abort(&ctl->x_empty[s], (use - 1) & 1, abort_flag, prm.wait)) {
                    set_abort(ctl, prm.status, kStatusWaitEmpty);
                    break;
                }
                mbar_arrive_expect_tx(&ctl->x_full_a[s], kAaBytes);
                tma_load_3d(xs[s].aa, &tmA, it * BK, 0, p, &ctl->x_full_a[s]);
                last = it;
            }
        }
    } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMmaWarps) {
        // ------------------------------------------------ MMA issuers
        // The whole warp runs the loop (so the descriptors stay warp-uniform)
        // and one elected lane issues the MMAs and commits.
        const int j = warp - kMmaWarp0;
        // the bounded waits below start their clocks only once the preceding
        // kernel has completed, so a long predecessor cannot run them out
        pdl_wait();
        for (int k = 0; k < nbatch; ++k) {
            const int it = k * kBatch + j;          // this warp's slab of batch k
            const int s = it % kX, use = it / kX;
            const int b = k % kTmemBufs, tuse = k / kTmemBufs;
            // the accumulator buffer's release by the fold (its first use
            // waits on nothing: the phase before the first reads as complete)
            // and, for a slab that exists, the expanded and activation tiles
            const bool ok = __all_sync(
                0xFFFFFFFFu, it < G ? wait3_or_abort(&ctl->x_full_b[s], use & 1, &ctl->x_full_a[s], use & 1,
                                                     &ctl->tmem_empty[b], (tuse - 1) & 1, abort_flag, prm.wait)
                                    : wait_or_abort(&ctl->tmem_empty[b], (tuse - 1) & 1, abort_flag, prm.wait));
            if (!ok) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull | kStatusWaitTmem);
                break;
            }
            tc_fence_after();
            if (it >= G) {
                // past the last slab: arrive without an MMA so the batch's
                // barrier still completes (the buffer is free, so this use's
                // previous phase has completed)
                if (lane == 0) mbar_arrive(&ctl->tmem_full[b]);
                continue;
            }
            const uint64_t ad = desc_sw128(smem_u32(xs[s].bx));
            const uint64_t bd = desc_sw128(smem_u32(xs[s].aa));
            const uint32_t d = tmem + (uint32_t)(b * kBatch * MT + j * MT);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk)   // +32 bytes along K inside the swizzle row
                    mma_f8(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdescN, kk > 0 ? 1u : 0u);
                // A slot that is never refilled gets no release: nothing would wait
                // for that arrival, and an arrival still in flight when the CTA
                // exits would land in the shared memory of the next CTA on this SM.
                if (it + kX < G) mma_commit(&ctl->x_empty[s]);
                mma_commit(&ctl->tmem_full[b]);
            }
            __syncwarp();
            last = it;
        }
    } else if (warp == kRowWarp) {
        // ------------------------------------------------ per-token scales
        pdl_wait();        // asg and rs are the preceding prologue's output
        for (int k = 0; k < nbatch; ++k) {
            const int r = k % kRowSlots, ruse = k / kRowSlots;
            // lanes decide on their own (nothing below is warp-wide), so each
            // lane that gives up reports it
            if (ruse > 0 && !wait_or_abort(&ctl->row_empty[r], (ruse - 1) & 1, abort_flag, prm.wait)) {
                set_abort(ctl, prm.status, kStatusWaitEmpty);
                break;
            }
            if (lane < MT) {
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj) {
                    const int it = k * kBatch + jj;
                    const size_t off = ((size_t)p * G + (size_t)it) * (size_t)M;
                    const bool ok = lane < M && it < G;     // tokens past M and slabs past G read as zero
                    cp_async4(&rows[r].row[jj][lane].x, ok ? prm.asg + off + lane : prm.asg, ok);
                    cp_async4(&rows[r].row[jj][lane].y, ok ? prm.rs + off + lane : prm.rs, ok);
                }
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
        for (int k = 0; k < nbatch; ++k) {
            const int it = k * kBatch + eg;         // this group's slab of batch k
            uint32_t wcol = 0;        // column et's SZ word
            const int wb = it / kWSlabs, wu = it % kWSlabs;
            const int ws_i = wb % kW, wuse = wb / kW;
            if (it >= G && wb * kWSlabs < G) {
                // a slab past K in a weight block that holds an earlier slab:
                // release this group's share of the slot once it has landed
                // (so the arrival counts for this use)
                if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&ctl->w_full[ws_i], wuse & 1, abort_flag, prm.wait))) {
                    if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                    break;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->w_empty[ws_i]);
            }
            if (it < G) {
                const int xs_i = it % kX, xuse = it / kX;
                // the slab's weights: read everything into registers, then
                // release the weight slot
                if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&ctl->w_full[ws_i], wuse & 1, abort_flag, prm.wait))) {
                    if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                    break;
                }
                const WSlot &wsl = ws[ws_i];
                wcol = wsl.sz[((et >> 3) * kWSlabs + wu) * 8 + (et & 7)];
                uint2 pk[8];
                uint32_t hb[8];           // int5: the fifth-bit block word of the same 16 k, shifted for expand16_int5
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = (et >> 3) + 16 * i;
                    pk[i] = *reinterpret_cast<const uint2 *>(wsl.bp + row * (kWSlabs * BK / 2) + wu * (BK / 2) +
                                                             chunk * 8);
                    if constexpr (kBits == 5)
                        hb[i] = *reinterpret_cast<const uint32_t *>(wsl.bh + row * (kWSlabs * BK / 8) +
                                                                    wu * (BK / 8) + (chunk >> 1) * 4) >>
                                (4 * (chunk & 1));
                }
                // The slot is refilled by the TMA (the async proxy), so these
                // generic reads must be ordered before that write by a proxy
                // fence, which waits for them to land.  int5 (four weight
                // slots) releases here, with a fence of its own; int4 (eight
                // slots, where the later release costs nothing) releases after
                // the operand stores, behind the fence those need anyway.
                if constexpr (kBits == 5) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->w_empty[ws_i]);
                }
                // the operand slot free (its previous slab's MMAs complete; the
                // phase before the first reads as complete)
                if (xuse > 0 && !__all_sync(0xFFFFFFFFu, wait_or_abort(&ctl->x_empty[xs_i], (xuse - 1) & 1, abort_flag, prm.wait))) {
                    if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                    break;
                }
                XSlot &xsl = xs[xs_i];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = (et >> 3) + 16 * i;
                    uint4 e;
                    if constexpr (kBits == 5)
                        e = expand16_int5(pk[i], hb[i]);
                    else
                        e = expand16(pk[i]);
                    *reinterpret_cast<uint4 *>(xsl.bx + row * BK + ((chunk ^ (row & 7)) << 4)) = e;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctl->x_full_b[xs_i]);
                    if constexpr (kBits != 5) mbar_arrive(&ctl->w_empty[ws_i]);
                }
            }
            // the slab's SZ words for the fold (word j of the SZ box is octet
            // j / 8, column j % 8: column n = j), into the batch slot; every
            // expand warp arrives once per batch, slab or not
            const int r = k % kSzfSlots, ruse = k / kSzfSlots;
            if (ruse > 0 &&
                !__all_sync(0xFFFFFFFFu, wait_or_abort(&ctl->szf_empty[r], (ruse - 1) & 1, abort_flag, prm.wait))) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                break;
            }
            szf[r].w[eg][et] = wcol;
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
        // the MMA sums a * c * 2^-9 (expand16), so sc carries 2^9; int5 feeds
        // c - 16 itself (expand16_int5), so its correction is -zscale
        const float o8 = kBits == 5 ? 0.0f : 8.0f;
        for (int k = fs; k < nbatch; k += kFoldSets) {
            const int b = k % kTmemBufs, tuse = k / kTmemBufs;
            const int r = k % kSzfSlots, ruse = k / kSzfSlots;
            const int rr = k % kRowSlots, rruse = k / kRowSlots;
            // warp-uniform: the TMEM loads and syncs below need the whole warp
            if (!__all_sync(0xFFFFFFFFu, wait3_or_abort(&ctl->row_full[rr], rruse & 1, &ctl->szf_full[r], ruse & 1,
                                                        &ctl->tmem_full[b], tuse & 1, abort_flag, prm.wait))) {
                if (lane == 0) set_abort(ctl, prm.status, kStatusWaitFull);
                bad = true;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj) {
                uint32_t d[16];
                tmem_issue32x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * kBatch * MT + jj * MT), d);
                const uint32_t w = szf[r].w[jj][n];
                tmem_wait16(d);
                if (jj == kBatch - 1) {      // every load of this buffer has completed
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tmem_empty[b]);
                }
                if (k * kBatch + jj < G) {
                    const float sc = f16lo(w);
                    const float z = kNibbleScale * sc, zz = -(f16hi(w) + o8 * sc);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < M) {
                            const float2 rv = rows[rr].row[jj][m];    // (asg, rs), the same for every lane
                            const float t = fmaf(zz, rv.y, z * __uint_as_float(d[m]));
                            acc[m] = fmaf(rv.x, t, acc[m]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctl->szf_empty[r]);
                mbar_arrive(&ctl->row_empty[rr]);
            }
        }
        // Dependent launch only now, as the CTA is about to finish: a CTA of
        // this kernel fills its SM, so a dependent grid launched earlier
        // crowds its CTAs onto the SMs this grid leaves idle (N/128 tiles
        // against the SM count) and runs them there, several to an SM, once
        // this grid completes.  A following prologue then took up to 3 us
        // longer (decode M = 16: step 21.2 against 19.6 us).
        pdl_trigger();
        // the sets meet in shared memory, in operand slot 0's expanded-weight
        // buffer: it is free only once BOTH sets have seen their last batch
        // (then every expansion and MMA has completed) -- a set that finishes
        // first must not write while the other set's last slab may still be in
        // slot 0
        float *part = reinterpret_cast<float *>(xs[0].bx);      // [kFoldSets - 1][MT][NN]
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
    // After a give-up anywhere in the CTA -- the flag is final once every role
    // has left its loop -- the copies and MMAs already issued must land before
    // shared and tensor memory are released.  These waits keep the full bound.
    if (*abort_flag) {
        if (warp < kTmaWWarps && lane == 0) {
            // this producer's blocks are last, last - 2, ...; each slot's latest
            for (int wb = last; wb >= 0 && wb > last - kW; wb -= kTmaWWarps)
                if (!mbar_wait(&ctl->w_full[wb % kW], (wb / kW) & 1) && prm.status) atomicOr(prm.status, kStatusDrain);
        } else if (warp == kTmaAWarp && lane == 0) {
            for (int it = last; it >= 0 && it > last - kX; --it)
                if (!mbar_wait(&ctl->x_full_a[it % kX], (it / kX) & 1) && prm.status)
                    atomicOr(prm.status, kStatusDrain);
        } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMmaWarps && last >= 0) {
            // one more commit, on a barrier of this warp's own: it completes
            // once every MMA this warp's issuing lane issued has completed
            const int j = warp - kMmaWarp0;
            if (elect_one()) mma_commit(&ctl->drain[j]);
            __syncwarp();
            if (lane == 0 && !mbar_wait(&ctl->drain[j], 0) && prm.status) atomicOr(prm.status, kStatusDrain);
        }
        // every MMA warp's drain ends before the tensor memory is freed (the
        // flag is final, so every thread takes this branch)
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (warp == kMmaWarp0) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
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
        const cuuint32_t box[2] = {kWSlabs * BK / 2, NN};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(w), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for w: CUresult %d", (int)r);
    }
    {
        // SZ table [N/8][G][8] words: box = the 8 words of kWSlabs groups for 16 octets
        const cuuint64_t dims[2] = {(cuuint64_t)(8 * (K / 128)), (cuuint64_t)(N / 8)};
        const cuuint64_t strides[1] = {(cuuint64_t)(32 * (K / 128))};
        const cuuint32_t box[2] = {8 * kWSlabs, NN / 8};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(sz), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PQ_ERR_CUDA, "tensor map for sz: CUresult %d", (int)r);
    }
    CUtensorMap tmH = tmB;        // int4: never read
    if (int5) {
        // fifth-bit planes [N][K/8] bytes: box = kWSlabs slabs (16 B each) of 128 rows
        const cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)(K / 8)};
        const cuuint32_t box[2] = {kWSlabs * BK / 8, NN};
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
    prm.wait = pipeline_wait_bound();
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
