/*
 * pq.h -- C ABI of libpq, a single-GPU (GB300, sm_103a) implementation of the
 * ParoQuant (PARO) W4A8 rotated-int4 linear layer
 *
 *     y = ((x * channel_scales) R^T) dequant(Q)^T
 *
 * R is eight layers of pairwise Givens rotations local to each 128-channel
 * group, Q is AWQ-packed uint4 with asymmetric zero points and group size 128.
 *
 * Source: the web page "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log":
 *   [Format]   section "Format"
 *   [Identity] the "Inference identity" paragraph of "Format"
 *   [D1]..[D4] section "Design", items 1 (zero point as a row-sum correction,
 *              SZ table), 2 (per-group fp8 activation scales), 3 (fused
 *              prologue, rotation records, software e4m3), 4 (partition select)
 *   [Gates]    section "Gates passed" (scale = amax * (1/448.f), rows past M
 *              untouched, bf16-floor GEMM tolerance)
 *   [CVT]      section "2026-09-15: hardware e4m3 convert in the producers"
 *   [PTOK]     section "Numbers", the per-token prefill item (pass A, pass C,
 *              the PTOK GEMM with As in the epilogue)
 *   [INT5]     section "2026-09-10: int5 W5A8 ParoQuant" (5-bit codes: low
 *              nibbles in the int4 words, the fifth bit in bit planes;
 *              c - 16 exact in e4m3)
 *
 * Conventions for every call:
 *   - Sizes are element counts.  G = K / 128.  "f16" = IEEE binary16,
 *     "bf16" = bfloat16, "e4m3" = OCP FP8 E4M3FN, all little-endian.
 *   - Every buffer is owned by the caller, who allocates and frees it.  The
 *     library allocates no memory (host or device), keeps no state besides a
 *     per-thread error string, and may be called from several host threads.
 *     The one exception is pq_rotate_tokquant_noalloc, whose scratch is a
 *     fixed array in the library's device image (see there).
 *   - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream) and never synchronise.  All
 *     argument checks run on the host before any launch; a failed check
 *     returns a status and launches nothing.  A launch failure returns
 *     PQ_ERR_CUDA.  Faults inside a kernel surface at the caller's next
 *     synchronisation, as for any CUDA kernel.
 *   - Kernels are launched as programmatic dependents (programmatic stream
 *     serialization).  Each kernel may read its load-time tables while the
 *     preceding kernel in the stream is still running, if that kernel signals
 *     early completion (all kernels here do), and waits for the preceding
 *     kernel before it reads anything else or writes anything:
 *     pq_rotate_quant may read `rec` and `cs` early, then waits before reading
 *     `x` and writing `a`, `asg`, `rs`; pq_gemm may stream `w` and `sz` early,
 *     then waits before reading `a`, `asg`, `rs` or writing `y`.  So `rec` and
 *     `cs` must not be written by the kernel issued right before
 *     pq_rotate_quant, nor `w` and `sz` by the one right before pq_gemm.
 *     The relaxation survives CUDA-graph capture.
 *   - Device pointers must be 16-byte aligned unless stated otherwise.
 *   - Inputs (x, channel scales, angles, scales) are finite; results for
 *     non-finite inputs are unspecified.
 *   - No call aborts, traps or prints.
 */
#ifndef PQ_H
#define PQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1: pack, prologue, the three GEMM kernels, the e4m3 encoder.
 * 2: adds the fused producers, the per-token path (pq_rotate_tokquant,
 *    pq_gemm_ptok) and int5 weights (pq_pack5, pq_gemm5*); version 1's calls
 *    are unchanged.
 * 3: adds pq_rotate_tokquant_noalloc; earlier calls are unchanged.
 * 4: adds the test hook pq_test_set_wait_limit_ns.
 * 5: adds pq_check_device_access and the status PQ_ERR_ACCESS.
 * 6: the byte layouts of w (pq_pack, pq_pack5) and whi (pq_pack5) change: a
 *    word's low nibbles hold four consecutive k and its high nibbles the next
 *    four, and whi is laid out in 32-k blocks; weights packed by an earlier
 *    version must be packed again.  Signatures are unchanged.
 * 7: adds pq_gemm5_skinny.
 * 8: the records of pq_pack and pq_pack5 are stored in chained order (see
 *    pq_pack) with a keep flag in byte 2; records packed by an earlier
 *    version must be packed again.  Signatures are unchanged. */
#define PQ_ABI_VERSION 8

/* Largest number of distinct rotations (partitions) one GEMM launch serves
 * ([Format] and the "Traps hit" note: the GEMM's limit applies to distinct
 * rotations). */
#define PQ_MAX_PARTITIONS 3

typedef enum pq_status {
    PQ_OK = 0,
    PQ_ERR_NULL = 1,      /* a required pointer is NULL                         */
    PQ_ERR_SHAPE = 2,     /* M/N/K/ld out of range, K or N not a multiple of 128 */
    PQ_ERR_ALIGN = 3,     /* a pointer or leading dimension breaks alignment    */
    PQ_ERR_PAIRS = 4,     /* a pairs row is not a permutation of 0..127         */
    PQ_ERR_PARTITION = 5, /* P outside 1..3 or pb1/pb2 inconsistent with P      */
    PQ_ERR_ARCH = 6,      /* no device, or the current device is not sm_103     */
    PQ_ERR_CUDA = 7,      /* a CUDA runtime call or launch failed               */
    PQ_ERR_ACCESS = 8     /* a pointer is not directly usable by the device     */
} pq_status;

/* ABI version of the loaded library (PQ_ABI_VERSION of its build). */
int pq_abi_version(void);

/* Static description of a status code; never NULL. */
const char *pq_status_string(int status);

/* Message of the last failed call on this host thread ("" if none). The
 * pointer stays valid until the next pq_* call on the same thread. */
const char *pq_last_error(void);

/* ------------------------------------------------------------------------ */
/* Load time (host)                                                         */
/* ------------------------------------------------------------------------ */

/* Byte sizes of pq_pack's three outputs for a K x N layer with P rotations:
 *   rec_bytes = P * 8 * G * 64 * 8, sz_bytes = G * N * 4, w_bytes = N * K / 2.
 * Any of the out pointers may be NULL.  Errors: PQ_ERR_SHAPE, PQ_ERR_PARTITION. */
pq_status pq_pack_sizes(int K, int N, int P, size_t *rec_bytes, size_t *sz_bytes,
                        size_t *w_bytes);

/*
 * Host packer: turns one checkpoint projection into the kernels' load-time
 * tables.  Pure and deterministic; all pointers are HOST memory, the outputs
 * sized by pq_pack_sizes.
 *
 * Inputs, as stored by the checkpoint ([Format]):
 *   qweight  int32 [K][N/8]   AWQ-packed codes: word slot i (bits 4i..4i+3)
 *                             holds column 8w + order[i], order = 0,2,4,6,1,3,5,7
 *   qzeros   int32 [G][N/8]   zero points, same packing, used raw (no +1)
 *   scales   f16   [G][N]     group scales
 *   pairs    int16 [P][8][K]  Givens pair indices local to each 128-group: in
 *                             layer r, group g, entries 2t and 2t+1 form pair t;
 *                             each (p, r, g) row is a permutation of 0..127
 *   theta    f16   [P][8][K/2] angle of pair t of group g at index 64g + t
 *
 * Outputs:
 *   rec  [P][8][G][64] records of 8 bytes ([D3]): bytes u, v, keep, 0, then
 *        uint16 f16(cos theta), uint16 f16(+-sin theta); cos/sin are evaluated
 *        in double precision (host libm) and rounded once to f16 (nearest,
 *        ties to even).  A record (u, v, c, s) rotates as
 *            v[u], v[v] = fl(fl(c*v[u]) + fl(s*v[v])), fl(fl(c*v[v]) - fl(s*v[u]))
 *        so a pages' pair (i, j) may be stored as (j, i) with its sine negated
 *        (bit-identical results).  Chained order, per (p, g): layer 0 lists
 *        the pairs in the pages' order t = 0..63 as (i, j); for r < 7, keep
 *        (bit 0 of byte 2) names the output of slot t that the next layer
 *        uses first (0: u, 1: v), and slot t of layer r + 1 holds the pair
 *        containing that channel, with it as u.  Every pair of layer r + 1
 *        receives exactly one kept channel: the kept channels are taken along
 *        the alternating cycles of the two layers' pairings, each cycle walked
 *        from its lowest channel c0 over its layer-r pair (c0, y0), keeping
 *        y0, then from y0's layer-(r+1) partner over its layer-r pair, and so
 *        on.  keep is 0 in layer 7.  Within a layer the order of the pairs
 *        does not change the result (they are disjoint), but the prologues
 *        rely on the chained order and the keep flags: records in another
 *        order give wrong results.
 *   sz   the SZ table ([D1]): for column n and group g the f16 pair
 *        (sc, f16(sc * (zp - 8))) -- the product is taken in fp32 (exact) and
 *        rounded once to f16 -- stored as one 4-byte word (scale in the low
 *        half) at word index ((n / 8) * G + g) * 8 + n % 8, i.e. laid out
 *        [N/8][G][8]: the words of one column octet over all groups are
 *        contiguous (one 32-byte sector per group and octet).
 *   w    [N][K/2] bytes (raw codes 0..15): each run of eight codes k = 8t ..
 *        8t+7 of row n fills bytes 4t .. 4t+3, byte 4t + b holding c[8t+b][n]
 *        in its low nibble and c[8t+b+4][n] in its high nibble (so a word's
 *        low nibbles are four consecutive k, as are its high nibbles).
 *
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE (K, N not positive multiples of 128),
 * PQ_ERR_PARTITION (P outside 1..3), PQ_ERR_PAIRS (a pairs row is not a
 * permutation; nothing useful is written in that case).
 */
pq_status pq_pack(int K, int N, int P, const int32_t *qweight, const int32_t *qzeros,
                  const uint16_t *scales, const int16_t *pairs, const uint16_t *theta,
                  void *rec, void *sz, void *w);

/*
 * Host packer for int5 weights ([INT5]).  As pq_pack, plus the fifth bits:
 *   qweight, qzeros  the low nibbles of the 5-bit codes and zero points, in
 *                    pq_pack's AWQ packing
 *   qweight_hi       int32 [K][N/32]: bit j of word w = the fifth bit of the
 *                    code of column 32w + j
 *   qzeros_hi        int32 [G][N/32]: the zero points' fifth bits, same order
 * so c = nibble + 16 * bit and zp likewise (0..31).  Outputs:
 *   rec, w   as pq_pack (w holds the low nibbles)
 *   sz       as pq_pack with zscale = f16(sc * (zp - 16))
 *   whi      [N][K/8] bytes (N * K / 8) in 4-byte blocks of 32 k: for
 *            k = 32t + 4q + j (q in 0..7, j in 0..3) the fifth bit of c[k][n]
 *            is bit q of byte 4t + j of row n
 * Errors: as pq_pack.
 */
pq_status pq_pack5(int K, int N, int P, const int32_t *qweight, const int32_t *qzeros,
                   const int32_t *qweight_hi, const int32_t *qzeros_hi, const uint16_t *scales,
                   const int16_t *pairs, const uint16_t *theta, void *rec, void *sz, void *w,
                   void *whi);

/* ------------------------------------------------------------------------ */
/* Per forward (device)                                                     */
/* ------------------------------------------------------------------------ */

/*
 * Fused prologue ([D2], [D3], [Gates]): for every partition p, token m < M and
 * group g, in one launch:
 *   v[k]  = x[m][128g+k] * cs[p][128g+k]                  (fp32, exact)
 *   for r = 0..7, for each pair t of (p, r, g) with record (i, j, c, s):
 *       v[i], v[j] = fl(fl(c*v[i]) + fl(s*v[j])), fl(fl(c*v[j]) - fl(s*v[i]))
 *   amax  = max_k |v[k]|,  asg = fl(amax * fl(1/448))
 *   a[k]  = e4m3(fl(v[k] / asg))  -- RNE, |q| saturated at 448, NaN -> 0,
 *           zero results as 0x00 ([CVT]); all codes 0x00 when asg == 0
 *   rs    = fl32(exact sum of the values the 128 codes decode to)
 * Every multiply, add and divide is a separately rounded IEEE fp32 operation,
 * so the outputs are bit-identical to a CPU evaluation in that order.
 *
 *   x    bf16 [M][ldx] (device), ldx >= K, ldx a multiple of 8
 *   rec  device copy of pq_pack's rec for these P rotations
 *   cs   f16 [P][K] (device) channel scales, stored pre-inverted (multiplied)
 *   a    e4m3 [P][M][K] (device, written)
 *   asg  fp32 [P][G][M] (device, written; 4-byte aligned)
 *   rs   fp32 [P][G][M] (device, written; 4-byte aligned)
 * Exactly P*M*K code bytes and P*G*M scales/row-sums are written; nothing else.
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE (M < 1, K not a positive multiple of 128,
 * ldx < K), PQ_ERR_ALIGN, PQ_ERR_PARTITION (P outside 1..3), PQ_ERR_ARCH,
 * PQ_ERR_CUDA.
 */
pq_status pq_rotate_quant(const void *x, int M, int K, int ldx, int P, const void *rec,
                          const void *cs, void *a, float *asg, float *rs, void *stream);

/*
 * Fused producer ([LOG] "2026-09-02/03: rotation stream (fused add + RMSNorm
 * + rotate + quant producers)"): residual add + Gemma RMSNorm + the
 * pq_rotate_quant steps, for every row m < M:
 *   s[k]  = bf16(fl(x[m][k] + residual[m][k]))          -> residual_out
 *   ss    = sum of s[k]^2: lane t of 64 sums fl(s^2 + s'^2) of its channel
 *           pair (128g+2t, 128g+2t+1) over the groups in order (fp32), then
 *           the 64 lane sums are added pairwise by recursive halving (fp32)
 *   inv   = fl(1 / fl(sqrt(fl(fl(ss / K) + eps))))      (IEEE sqrt, divide)
 *   h[k]  = bf16(fl(fl(s[k] * inv) * fl(1 + gamma[k])))  -> h
 *   then a, asg, rs = pq_rotate_quant of h (all P partitions).
 * Every step is a separately rounded IEEE operation, so the outputs are
 * bit-identical to a CPU evaluation in that order.  M <= 16 runs one fused
 * launch (each CTA recomputes its row's norm); larger M runs a norm kernel
 * and then pq_rotate_quant's kernel on h.
 *
 *   x, residual    bf16 [M][ldx] (device), ldx >= K, ldx a multiple of 8
 *   gamma          bf16 [K] (device): the RMSNorm weight, applied as (1 + gamma)
 *   eps            >= 0 and finite; a row of zeros needs eps > 0
 *   rec, cs        as for pq_rotate_quant
 *   residual_out   bf16 [M][K] (device, written); must not overlap x or
 *                  residual (other CTAs still read the whole input rows)
 *   h              bf16 [M][K] (device, written): the normed rows
 *   a, asg, rs     as written by pq_rotate_quant
 * Programmatic dependent launch: gamma, rec and cs may be read before the
 * preceding kernel completes; x and residual are read after it.
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE (M < 1, K not a positive multiple of 128,
 * ldx < K, eps negative or not finite, residual_out overlapping an input),
 * PQ_ERR_ALIGN, PQ_ERR_PARTITION, PQ_ERR_ARCH, PQ_ERR_CUDA.
 */
pq_status pq_add_rms_rotate_quant(const void *x, const void *residual, const void *gamma, float eps,
                                  int M, int K, int ldx, int P, const void *rec, const void *cs,
                                  void *residual_out, void *h, void *a, float *asg, float *rs,
                                  void *stream);

/*
 * silu-mul producer ([LOG] "2026-09-03: rotation stream 2 (silu-mul, GDN
 * gated norm, attention gate fused with rotate+quant)", MODE 0): for every
 * row m < M and channel k < I of the merged gate/up output y (gate g in
 * columns [0, I), up u in [I, 2I)):
 *   e      = exp32(-g)   -- a fixed fp32 sequence: n = rint(fl(x log2 e)),
 *            r = fl(fl(x - n ln2_hi) - n ln2_lo) with ln2_hi =
 *            0.693145751953125, ln2_lo = 1.42860677e-06, the degree-6 Taylor
 *            polynomial of exp in Horner form, exact scaling by 2^n; x > 88
 *            gives +inf, x < -103 gives 0
 *   act[k] = bf16(fl(bf16(fl(g / fl(1 + e))) * u))
 *   then a, asg, rs = pq_rotate_quant of act with K = I.
 * Every step is a separately rounded IEEE operation, so the outputs are
 * bit-identical to a CPU evaluation in that order.  M <= 16 runs one launch;
 * larger M runs an elementwise kernel and then pq_rotate_quant's kernel.
 *
 *   y        bf16 [M][ldy] (device), ldy >= 2*I, ldy a multiple of 8
 *   I        the down projection's K: a positive multiple of 128
 *   rec, cs  as for pq_rotate_quant, for K = I
 *   act      bf16 [M][I] (device, written); must not overlap y
 *   a, asg, rs  as written by pq_rotate_quant
 * Programmatic dependent launch: rec and cs may be read before the preceding
 * kernel completes; y is read after it.
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE (M < 1, I not a positive multiple of
 * 128, ldy < 2*I, act overlapping y), PQ_ERR_ALIGN, PQ_ERR_PARTITION,
 * PQ_ERR_ARCH, PQ_ERR_CUDA.
 */
pq_status pq_silu_mul_rotate_quant(const void *y, int M, int I, int ldy, int P, const void *rec,
                                   const void *cs, void *act, void *a, float *asg, float *rs,
                                   void *stream);

/*
 * uint4 x e4m3 group GEMM ([D1], [D2], [D4]):
 *   p(n)   = (n >= pb1) + (n >= pb2)
 *   D      = sum_{k in g} dec(a[p(n)][m][k]) * (c[k][n] - 8)
 *   y[m][n] = bf16( sum_g asg[p][g][m] * (sc[g][n] * D - zs[g][n] * rs[p][g][m]) )
 * with (sc, zs) the f16 pair of column n, group g in the SZ table.  Accumulation is fp32 (tensor-core
 * fp32 accumulation within a 128-k group on the tensor-core path); the result
 * is within the bf16 output floor of the fp64 value (norm-wise relative error
 * <= 2e-3 is the gate).
 *
 *   a, asg, rs  as written by pq_rotate_quant (P partitions)
 *   w, sz       device copies of pq_pack's outputs
 *   y           bf16 [M][ldy] (device, written), ldy >= N, ldy a multiple of 8;
 *               only y[0..M-1][0..N-1] is written
 *   pb1, pb2    partition boundaries, multiples of 128:
 *               P = 1: pb1 = pb2 = N;  P = 2: 0 < pb1 < pb2 = N;
 *               P = 3: 0 < pb1 < pb2 < N
 * Dispatch (one launch in every case; S = the device's SM count):
 *   M = 1, K <= 16384                   -> pq_gemm_skinny (CUDA cores)
 *   2 <= M <= 16, 2 * (N / 128) >= S    -> pq_gemm_tcn (narrow tensor-core kernel)
 *   2 <= M <= 16, 2 * (N / 128) < S,
 *     K <= 16384                        -> pq_gemm_skinny
 *   M <= 16, K > 16384                  -> pq_gemm_tcn
 *   M > 16                              -> pq_gemm_tc (prefill tensor-core kernel)
 * Layouts differ from a plain [G][N][2] SZ table and [P][M][G] scales on
 * purpose: the SZ words are octet-major ([N/8][G][8], see pq_pack) and asg/rs
 * are [P][G][M], so that each kernel reads them with one contiguous copy.
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE, PQ_ERR_ALIGN, PQ_ERR_PARTITION,
 * PQ_ERR_ARCH, PQ_ERR_CUDA.
 */
pq_status pq_gemm(const void *a, const float *asg, const float *rs, int M, int N, int K, int P,
                  int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                  void *stream);

/* Largest M that pq_gemm may send to the CUDA-core decode kernel (see the
 * dispatch rule of pq_gemm; pq_gemm_skinny itself also needs K <= 16384). */
int pq_gemm_skinny_max_m(void);

/*
 * The GEMM kernels behind pq_gemm, callable on their own (same arguments and
 * result).  pq_gemm_skinny (CUDA cores; weights streamed once, exact products
 * accumulated in fp32) accepts 1 <= M <= 16; pq_gemm_tcn (tensor cores,
 * operands swapped: 128 output features x up to 16 tokens per MMA, weights
 * streamed once) accepts 1 <= M <= 16; pq_gemm_tc (tensor cores, 256-token x
 * 128-feature tiles) accepts any M >= 1.  A larger M returns PQ_ERR_SHAPE, and
 * so does pq_gemm_skinny for K > 16384.
 *
 * dev_status (device, 4-byte aligned, may be NULL): every wait inside the
 * kernels is bounded; a wait that gives up (never expected) ORs a nonzero
 * code into *dev_status, the affected output tile is filled with NaN, and the
 * kernel returns.  The caller zeroes *dev_status beforehand.
 */
pq_status pq_gemm_skinny(const void *a, const float *asg, const float *rs, int M, int N, int K,
                         int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                         int ldy, unsigned int *dev_status, void *stream);
pq_status pq_gemm_tc(const void *a, const float *asg, const float *rs, int M, int N, int K,
                     int P, int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                     unsigned int *dev_status, void *stream);
pq_status pq_gemm_tcn(const void *a, const float *asg, const float *rs, int M, int N, int K,
                      int P, int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                      unsigned int *dev_status, void *stream);

/*
 * Per-token activation scales, prologue ([PTOK] pass A and pass C).  For
 * every partition p, row m < M:
 *   v     = the pq_rotate_quant rotation of x[m] * cs[p] (fp32, same steps)
 *   xr[k] = bf16(v[k])                        (round to nearest even)
 *   asg_g = fl(max_{k in g} |xr[k]| * fl(1/448))  for every group g
 *   As    = max_g asg_g
 *   a[k]  = e4m3(fl(xr[k] / As))              (all 0 when As == 0; [CVT])
 *   rs_g  = sum_{k in g} dec(a[k])            (exact, then rounded to fp32)
 * Two launches: pass A writes xr and the group scales (into rs); pass C reads
 * them back and writes a, As and the row-sums over them.  Every step is a
 * separately rounded IEEE operation, so the outputs are bit-identical to a CPU
 * evaluation in that order.
 *
 *   x, rec, cs  as for pq_rotate_quant
 *   xr          bf16 [P][M][K] (device, written): the rotated rows, the
 *               scratch between the passes; must not overlap x
 *   a           e4m3 [P][M][K] (device, written)
 *   As          fp32 [P][M] (device, written; 4-byte aligned)
 *   rs          fp32 [P][G][M] (device, written; 4-byte aligned): plain
 *               row-sums, no activation scale in them
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE (M < 1, K not a positive multiple of 128,
 * ldx < K, xr overlapping x), PQ_ERR_ALIGN, PQ_ERR_PARTITION, PQ_ERR_ARCH,
 * PQ_ERR_CUDA.
 */
pq_status pq_rotate_tokquant(const void *x, int M, int K, int ldx, int P, const void *rec,
                             const void *cs, void *xr, void *a, float *As, float *rs, void *stream);

/*
 * pq_rotate_tokquant for callers that cannot allocate device memory.  It has
 * no counterpart in the engineering log: it exists for code that must not
 * call cudaMalloc or any allocator -- for instance a plugin inside an engine
 * that owns every byte of device memory through its own pool, a caller that
 * only receives its input and output tensors, or a latency-critical path
 * where an allocation could synchronise the device.  Such a caller cannot
 * provide pq_rotate_tokquant's xr scratch.  This entry point keeps the
 * rotated rows in a fixed bf16 array inside the library instead (16 MiB of
 * device memory on every GPU that loads the library, held until the process
 * exits), and allocates nothing itself.
 *
 * Same result and arguments as pq_rotate_tokquant, without xr:
 *   x, rec, cs, a, As, rs   as for pq_rotate_tokquant
 * Limits and rules:
 *   - P * M * K <= PQ_TOKQUANT_NOALLOC_MAX_ELEMS; a larger problem returns
 *     PQ_ERR_SHAPE and launches nothing (use pq_rotate_tokquant).
 *   - Every call on a device uses the same array, and a call leaves its rows
 *     there; each call overwrites every element it reads, so old contents do
 *     not matter.  Calls whose kernels overlap on the GPU (different streams
 *     without ordering between them, or several host threads) race on the
 *     array and give wrong results: order them on one stream.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress, which may load the
 *     library's device code); make that first call before any stream capture.
 * Errors: as pq_rotate_tokquant, plus PQ_ERR_SHAPE for P * M * K above the
 * limit and PQ_ERR_CUDA if the address lookup fails.
 */
#define PQ_TOKQUANT_NOALLOC_MAX_ELEMS (8u * 1024u * 1024u)
pq_status pq_rotate_tokquant_noalloc(const void *x, int M, int K, int ldx, int P, const void *rec,
                                     const void *cs, void *a, float *As, float *rs, void *stream);

/*
 * The GEMM on per-token scales ([PTOK] "PTOK GEMM"):
 *   y[m][n] = bf16( As[p][m] * sum_g (sc[g][n] * D - zs[g][n] * rs[p][g][m]) )
 * with p, D, sc, zs as for pq_gemm and a, As, rs from pq_rotate_tokquant.
 * The tcgen05 prefill kernel with the group fold reduced to one fp32 multiply-
 * add per element and slab and As applied once in the epilogue; any M >= 1.
 * Arguments, dev_status and errors as for pq_gemm_tc.
 */
pq_status pq_gemm_ptok(const void *a, const float *As, const float *rs, int M, int N, int K, int P,
                       int pb1, int pb2, const void *w, const void *sz, void *y, int ldy,
                       unsigned int *dev_status, void *stream);

/*
 * uint4 x e4m3 group GEMM on int5 weights ([INT5]): pq_gemm's result with
 *   D = sum_{k in g} dec(a[p(n)][m][k]) * (c[k][n] - 16),  c in 0..31,
 *   y[m][n] = bf16( sum_g asg[p][g][m] * (sc[g][n] * D - zs[g][n] * rs[p][g][m]) )
 * and (sc, zs) from pq_pack5's SZ table.  The tensor cores take (c - 16) * 2^-9
 * itself, exact in e4m3.  Tolerance and arguments as pq_gemm, plus
 *   w, whi, sz  device copies of pq_pack5's outputs (whi 16-byte aligned)
 * pq_gemm5 dispatches as pq_gemm: M = 1 to the CUDA-core kernel
 * (pq_gemm5_skinny); 2 <= M <= 16 to the narrow tensor-core kernel
 * (pq_gemm5_tcn) when its 128-feature tiles cover at least half the SMs, else
 * to the CUDA-core kernel; any M <= 16 with K > 16384 to the narrow kernel;
 * M > 16 to the prefill tensor-core kernel (pq_gemm5_tc).  pq_gemm5_tcn and
 * pq_gemm5_skinny accept 1 <= M <= 16 (the CUDA-core kernel K <= 16384): it
 * is pq_gemm_skinny with each fifth bit ORed into the f16 word of its nibble
 * (bit 4 above a low nibble, bit 8 above a high one), so the same FMA takes
 * the 5-bit code.  dev_status as for pq_gemm_tc.
 * Errors: PQ_ERR_NULL, PQ_ERR_SHAPE, PQ_ERR_ALIGN, PQ_ERR_PARTITION,
 * PQ_ERR_ARCH, PQ_ERR_CUDA.
 */
pq_status pq_gemm5(const void *a, const float *asg, const float *rs, int M, int N, int K, int P,
                   int pb1, int pb2, const void *w, const void *whi, const void *sz, void *y, int ldy,
                   void *stream);
pq_status pq_gemm5_tc(const void *a, const float *asg, const float *rs, int M, int N, int K, int P,
                      int pb1, int pb2, const void *w, const void *whi, const void *sz, void *y,
                      int ldy, unsigned int *dev_status, void *stream);
pq_status pq_gemm5_tcn(const void *a, const float *asg, const float *rs, int M, int N, int K, int P,
                       int pb1, int pb2, const void *w, const void *whi, const void *sz, void *y,
                       int ldy, unsigned int *dev_status, void *stream);
pq_status pq_gemm5_skinny(const void *a, const float *asg, const float *rs, int M, int N, int K, int P,
                          int pb1, int pb2, const void *w, const void *whi, const void *sz, void *y,
                          int ldy, unsigned int *dev_status, void *stream);

/*
 * The prologue's device e4m3 encoder applied to n fp32 values ([CVT]: NaN ->
 * 0x00, clamp to +-448, round to nearest even, zero results as 0x00).  For the
 * exhaustive check of the encoder; in/out device pointers, 4-byte and 1-byte
 * alignment suffice.  Errors: PQ_ERR_NULL, PQ_ERR_ARCH, PQ_ERR_CUDA.
 */
pq_status pq_e4m3_encode(const float *in, uint8_t *out, size_t n, void *stream);

/*
 * Test hook, not for production use (the pages have no counterpart).  Sets
 * the bound of the GEMM kernels' pipeline waits (see dev_status above) for
 * every launch made after the call, process-wide: ns = 0 restores the
 * product bound of 2 s; 0 < ns <= 2e9 shortens it, so that on a healthy GPU
 * the waits give up and the give-up path (status code, NaN tile, release of
 * tensor memory, return) runs.  The waits that let in-flight copies and MMAs
 * land after a give-up keep 2 s.  Not thread-safe with respect to launches
 * on other threads.  Errors: PQ_ERR_SHAPE for ns > 2e9.
 */
pq_status pq_test_set_wait_limit_ns(unsigned long long ns);

/*
 * Whether kernels on the current device can dereference p directly (no
 * counterpart in the pages; a helper for zero-copy inputs and outputs).  Every
 * device pointer argument of the calls above may point to memory of the
 * current device, to managed memory, or to page-locked host memory that is
 * mapped into the device's address space at the same address (on this
 * platform the host's memory is reached over a coherent link): the kernels
 * then read x from, or write y to, host memory directly, and the bytes cross
 * the link inside the kernels.  Such host buffers must stay allocated and
 * page-locked until the kernels have finished.  This call checks the start
 * address only (cudaPointerGetAttributes); it launches nothing.
 * Returns PQ_OK, PQ_ERR_NULL, PQ_ERR_ACCESS (pageable host memory, host memory
 * mapped at another address, or another device's memory) or PQ_ERR_CUDA.
 */
pq_status pq_check_device_access(const void *p);

#ifdef __cplusplus
}
#endif

#endif /* PQ_H */
