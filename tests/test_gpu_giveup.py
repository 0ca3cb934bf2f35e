"""The GEMM kernels' give-up path, run on a healthy GPU.

Every wait inside the GEMM kernels is bounded (2 s of %globaltimer).  A wait
that runs out ORs a code into the status word, the CTA stops, lets the copies
and MMAs it already issued land (those drain waits keep the full bound),
frees its tensor memory, writes NaN over its outputs and returns.  Here the
test hook pq_test_set_wait_limit_ns shortens the pipeline waits to 100 ns, far
below one HBM round trip under load, on problems where every CTA streams many
stages through its ring (so its producers and consumers do wait), and the
waits give up in a correct pipeline: each kernel must then return promptly with a nonzero
status word and no drain failure, every output element must be NaN or the
value of a normal launch, nothing outside y may be written, and the next
launch with the normal bound must reproduce the normal result bit for bit.

Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log",
"2026-09-03: rotation stream 3" (spin waits that deadlocked the device):
every wait here has a bound and a reported way out.
"""
import ctypes as C
import time

import numpy as np
import pytest

import pqgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

STATUS_DRAIN = 8           # a drain wait ran out: an issued copy or MMA did not land
SHORT_NS = 100
CANARY = 3.0


@pytest.fixture(scope="module")
def pq():
    import __graft_entry__
    __graft_entry__.build()
    import w4a8_rotated_int4_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def build_case(pq, orc, path, M, K, N):
    """Device operands for one path and the fp64 oracle result."""
    bits = 5 if path.endswith("5") else 4
    prob = pqgen.make_problem(M, K, N, seed=M + K + N + bits, bits=bits)
    x_d = dev_u16(prob.x).view(torch.bfloat16)
    if bits == 5:
        rec, sz, w, whi = pq.pq_pack5(prob.qweight, prob.qzeros, prob.qweight_hi, prob.qzeros_hi,
                                      prob.scales, prob.pairs, prob.theta)
        t = orc.pack5(prob)
    else:
        rec, sz, w = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta)
        whi = None
        t = orc.pack(prob)
    rec_d, sz_d, w_d = torch.from_numpy(rec).cuda(), dev_u16(sz), torch.from_numpy(w).cuda()
    whi_d = torch.from_numpy(whi).cuda() if whi is not None else None
    cs_d = dev_u16(prob.cs)
    if path == "ptok":
        _, a, s, rs = pq.pq_rotate_tokquant(x_d, rec_d, cs_d)
        _, a_o, s_o, rs_o = orc.rotate_tokquant(prob.x, prob.cs, t["rec"])
        y64 = orc.gemm_ptok_f64(a_o, s_o, rs_o, t["codes"], t["sz"], prob.pb1, prob.pb2)
    else:
        a, s, rs = pq.pq_rotate_quant(x_d, rec_d, cs_d)
        a_o, s_o, rs_o = orc.rotate_quant(prob.x, prob.cs, t["rec"])
        f = orc.gemm5_f64 if bits == 5 else orc.gemm_f64
        y64 = f(a_o, s_o, rs_o, t["codes"], t["sz"], prob.pb1, prob.pb2)
    name = {"skinny": "pq_gemm_skinny", "tcn": "pq_gemm_tcn", "tc": "pq_gemm_tc", "ptok": "pq_gemm_ptok",
            "tc5": "pq_gemm5_tc", "tcn5": "pq_gemm5_tcn", "skinny5": "pq_gemm5_skinny"}[path]
    fn = getattr(pq.lib(), name)
    P = a.shape[0]

    def launch(y, ldy, status):
        """Through the C ABI: y is the [M, ldy] buffer, N < ldy columns written."""
        ptrs = [C.c_void_p(a.data_ptr()), C.c_void_p(s.data_ptr()), C.c_void_p(rs.data_ptr())]
        dims = [M, N, K, P, prob.pb1, prob.pb2]
        wts = [C.c_void_p(w_d.data_ptr())] + ([C.c_void_p(whi_d.data_ptr())] if bits == 5 else [])
        tail = [C.c_void_p(sz_d.data_ptr()), C.c_void_p(y.data_ptr()), ldy, C.c_void_p(status.data_ptr()),
                C.c_void_p(torch.cuda.current_stream().cuda_stream)]
        pq._check(fn(*ptrs, *dims, *wts, *tail), name)

    return launch, y64


def run(launch, M, N):
    """One launch into a canary-filled y with a leading dimension past N;
    returns (y [M, N] as bf16 bits, status, seconds, canary intact)."""
    ybuf = torch.full((M + 2, N + 64), CANARY, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    launch(ybuf, N + 64, status)
    torch.cuda.synchronize()
    dt = time.monotonic() - t0
    yb = ybuf.view(torch.int16).cpu().numpy()
    canary = np.int16(torch.tensor([CANARY], dtype=torch.bfloat16).view(torch.int16).item())
    outside_ok = bool((yb[M:] == canary).all() and (yb[:M, N:] == canary).all())
    return yb[:M, :N].copy(), int(status.item()), dt, outside_ok


def is_nan_bf16(bits):
    return ((bits.astype(np.uint16) & 0x7F80) == 0x7F80) & ((bits.astype(np.uint16) & 0x007F) != 0)


GIVEUP_CASES = [  # path, M, K, N: several ring turns per CTA
    ("skinny", 1, 5120, 17408),
    ("skinny", 3, 2048, 16384),
    ("skinny5", 1, 5120, 17408),
    ("tcn", 4, 5120, 8192),
    ("tcn5", 16, 2048, 4096),
    ("tc", 300, 4096, 2048),
    ("ptok", 300, 4096, 2048),
    ("tc5", 256, 2048, 1024),
]


@pytest.mark.parametrize("path,M,K,N", GIVEUP_CASES)
def test_short_wait_bound_gives_up_cleanly(pq, orc, path, M, K, N):
    launch, y64 = build_case(pq, orc, path, M, K, N)
    ref, st, _, ok = run(launch, M, N)
    assert st == 0 and ok
    yf = torch.from_numpy(ref).view(torch.bfloat16).float().numpy()
    rel = float(np.linalg.norm(yf - y64) / max(np.linalg.norm(y64), 1e-300))
    assert rel <= 2e-3, "normal launch: rel err %.3e" % rel

    outcomes = []
    try:
        pq.pq_test_set_wait_limit_ns(SHORT_NS)
        # the waits race the copies, so a launch could in principle finish
        # untouched; a few tries make a give-up certain in practice
        for _ in range(5):
            y, st, dt, ok = run(launch, M, N)
            outcomes.append((st, dt))
            assert ok, "%s wrote outside y after giving up" % path
            assert dt < 10.0, "%s took %.1f s to give up" % (path, dt)
            nan = is_nan_bf16(y)
            # every element is NaN (its CTA gave up) or the normal result
            assert np.array_equal(y[~nan], ref[~nan]), "%s: a non-NaN output differs" % path
            if st != 0:
                assert st & STATUS_DRAIN == 0, "%s: a drain wait ran out (status %d)" % (path, st)
                assert nan.any(), "%s: status %d but no NaN output" % (path, st)
                break
    finally:
        pq.pq_test_set_wait_limit_ns(0)
    assert any(s != 0 for s, _ in outcomes), "%s: no wait gave up at %d ns: %s" % (path, SHORT_NS, outcomes)

    # the normal bound again: the context and the library are unharmed
    for _ in range(2):
        y, st, _, ok = run(launch, M, N)
        assert st == 0 and ok
        assert np.array_equal(y, ref), "%s: launch after the give-up differs" % path


def test_wait_bound_hook_rejects_above_product_bound(pq):
    with pytest.raises(pq.PQError):
        pq.pq_test_set_wait_limit_ns(2_000_000_001)
    pq.pq_test_set_wait_limit_ns(0)
