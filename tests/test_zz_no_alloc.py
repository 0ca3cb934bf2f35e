"""pq_rotate_tokquant_noalloc, the per-token prologue for callers that cannot
allocate device memory (an engine plugin whose host owns every byte through
its own pool, a caller handed only its tensors, a path where an allocation
could stall the device).  It keeps the rotated rows in a fixed array inside
the library instead of the caller's xr buffer.

The test calls it through the C ABI (ctypes, no Python wrapper) twice in a
row on different inputs -- the second call finds the first call's rows still
in the shared array -- and compares each call's codes, token scales and
row-sums with pq_rotate_tokquant on a caller-supplied xr: they must be
bit-identical, the tolerance of every prologue test.  It also checks that a
problem above the array's size is refused before anything runs.  This file
sorts last so a run that stops at the first failure has run every other test
first; it passes on its own as well.
"""
import ctypes as C

import numpy as np
import pytest

import pqgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pq():
    import __graft_entry__
    __graft_entry__.build()
    import w4a8_rotated_int4_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def _ptr(t):
    return C.c_void_p(t.data_ptr())


@pytest.mark.parametrize("M,K,P", [(37, 640, 1), (300, 5120, 3)])
def test_noalloc_matches_caller_scratch_twice(pq, M, K, P):
    L = pq.lib()
    G = K // 128
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((11, 12)):
        prob = pqgen.make_problem(M, K, 128 * P, P=P, seed=seed + M)
        rec, _, _ = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta)
        x = torch.from_numpy(prob.x.view(np.int16)).cuda().view(torch.bfloat16)
        cs = torch.from_numpy(prob.cs.view(np.int16)).cuda()
        rec_d = torch.from_numpy(rec).cuda()
        # reference: the existing entry point with a caller-supplied xr
        xr_ref = torch.empty((P, M, K), dtype=torch.bfloat16, device="cuda")
        a_ref = torch.empty((P, M, K), dtype=torch.uint8, device="cuda")
        As_ref = torch.empty((P, M), dtype=torch.float32, device="cuda")
        rs_ref = torch.empty((P, G, M), dtype=torch.float32, device="cuda")
        st = L.pq_rotate_tokquant(_ptr(x), M, K, K, P, _ptr(rec_d), _ptr(cs), _ptr(xr_ref), _ptr(a_ref),
                                  _ptr(As_ref), _ptr(rs_ref), stream)
        assert st == 0, L.pq_last_error().decode()
        # the entry point without scratch, outputs pre-filled with garbage
        a = torch.full((P, M, K), 0xA5, dtype=torch.uint8, device="cuda")
        As = torch.full((P, M), float("nan"), dtype=torch.float32, device="cuda")
        rs = torch.full((P, G, M), float("nan"), dtype=torch.float32, device="cuda")
        st = L.pq_rotate_tokquant_noalloc(_ptr(x), M, K, K, P, _ptr(rec_d), _ptr(cs), _ptr(a), _ptr(As),
                                          _ptr(rs), stream)
        assert st == 0, L.pq_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(a, a_ref), "call %d: codes differ" % call
        assert np.array_equal(As.cpu().numpy().view(np.uint32), As_ref.cpu().numpy().view(np.uint32)), \
            "call %d: token scales differ" % call
        assert np.array_equal(rs.cpu().numpy().view(np.uint32), rs_ref.cpu().numpy().view(np.uint32)), \
            "call %d: row-sums differ" % call


def test_noalloc_refuses_problems_above_its_scratch(pq):
    L = pq.lib()
    K, P = 1024, 1
    M = 8 * 1024 * 1024 // K + 1          # one row over the fixed array
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    cs = torch.zeros((P, K), dtype=torch.int16, device="cuda")
    rec = torch.zeros((P * 8 * (K // 128) * 64 * 8,), dtype=torch.uint8, device="cuda")
    a = torch.empty((P, M, K), dtype=torch.uint8, device="cuda")
    As = torch.empty((P, M), dtype=torch.float32, device="cuda")
    rs = torch.empty((P, K // 128, M), dtype=torch.float32, device="cuda")
    st = L.pq_rotate_tokquant_noalloc(_ptr(x), M, K, K, P, _ptr(rec), _ptr(cs), _ptr(a), _ptr(As), _ptr(rs),
                                      C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert pq.STATUS[st] == "PQ_ERR_SHAPE"
    assert b"fixed scratch" in L.pq_last_error()
