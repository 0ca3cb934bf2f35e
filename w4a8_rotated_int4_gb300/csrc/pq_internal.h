// pq_internal.h -- declarations shared by the translation units of libpq.
// Not part of the public ABI (that is include/pq.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "pq.h"

namespace pq {

// Records the message for pq_last_error() on this thread and returns `st`.
pq_status fail(pq_status st, const char *fmt, ...);
// Clears the thread's message (start of every public call).
void clear_error();

// PQ_OK if the current device is compute capability 10.3, else PQ_ERR_ARCH /
// PQ_ERR_CUDA with a message.  Also returns the SM count of that device.
pq_status check_device(int *sm_count);

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validation shared by the GEMM entry points.
pq_status check_gemm_args(const void *a, const float *asg, const float *rs, int M, int N, int K,
                          int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                          int ldy);

// Kernel launchers (one per translation unit).
pq_status launch_add_rms_rotate_quant(const void *x, const void *res, const void *gamma, float eps, int M,
                                      int K, int ldx, int P, const void *rec, const void *cs, void *res_out,
                                      void *h, void *a, float *asg, float *rs, void *stream);
pq_status launch_silu_mul_rotate_quant(const void *y, int M, int I, int ldy, int P, const void *rec,
                                       const void *cs, void *act, void *a, float *asg, float *rs, void *stream);
pq_status launch_rotate_quant(const void *x, int M, int K, int ldx, int P, const void *rec,
                              const void *cs, void *a, float *asg, float *rs, void *stream);
pq_status launch_rotate_tokquant(const void *x, int M, int K, int ldx, int P, const void *rec, const void *cs,
                                 void *xr, void *a, float *As, float *rs, void *stream);
pq_status launch_rotate_tokquant_noalloc(const void *x, int M, int K, int ldx, int P, const void *rec,
                                         const void *cs, void *a, float *As, float *rs, void *stream);
pq_status launch_e4m3_encode(const float *in, uint8_t *out, size_t n, void *stream);
pq_status launch_gemm_skinny(const void *a, const float *asg, const float *rs, int M, int N,
                             int K, int P, int pb1, int pb2, const void *w, const void *sz,
                             void *y, int ldy, unsigned int *dev_status, void *stream,
                             int sm_count, const void *whi = nullptr);
pq_status launch_gemm_tc(const void *a, const float *asg, const float *rs, int M, int N, int K,
                         int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                         int ldy, unsigned int *dev_status, void *stream, int sm_count,
                         bool per_token = false, const void *whi = nullptr);

pq_status launch_gemm_tcn(const void *a, const float *asg, const float *rs, int M, int N, int K,
                          int P, int pb1, int pb2, const void *w, const void *sz, void *y,
                          int ldy, unsigned int *dev_status, void *stream, const void *whi = nullptr);

// Give up a wait after this many nanoseconds of %globaltimer (never reached by
// a correct pipeline; it bounds the damage of a bug to one slow launch).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// One try_wait; the thread may be suspended by the hardware for up to
// kSuspendHintNs while the phase is incomplete (it resumes as soon as the
// phase completes), so waiting warps do not spin on the issue slots.
constexpr uint32_t kSuspendHintNs = 100000u;

// The bound of a kernel's pipeline waits, passed in its parameters: kWaitLimitNs
// in every product launch.  A test entry point may shorten it so that the
// give-up path runs on a healthy GPU; `hint` (the try_wait suspend hint) is
// then shortened too, so that one suspended try_wait cannot outlast the bound.
// The waits that drain in-flight copies and MMAs after a give-up always keep
// kWaitLimitNs.
struct WaitBound {
    unsigned long long ns;
    uint32_t hint;
};

// The bound every launch puts in its kernel parameters: {kWaitLimitNs,
// kSuspendHintNs} unless pq_test_set_wait_limit_ns has shortened it.
WaitBound pipeline_wait_bound();

constexpr int kSkinnyMaxM = 16;   // largest M the CUDA-core decode kernel accepts
constexpr int kSkinnyMaxK = 16384;   // largest K it accepts (one compute warp per 1024 k, plus the producer)
constexpr int kTcnMaxM = 16;      // largest M the narrow tensor-core kernel accepts

}  // namespace pq
