"""Host-side checks of libpq that need no GPU: the library loads and exports
every symbol include/pq.h declares, the host packer is byte-equal to the
oracle's independent packer, and every argument check returns its status
without touching device memory."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import pqgen
import w4a8_rotated_int4_gb300 as pq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build_library()
    return pq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "pq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pq_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(pq.EXPORTS)
    assert pq.pq_abi_version() == 8
    for s in range(9):
        assert L.pq_status_string(s)
    assert L.pq_status_string(99) == b"unknown status"


@pytest.mark.parametrize("shape", [(256, 128, 1), (384, 256, 2), (640, 384, 3), (1024, 1024, 1)])
def test_pack_byte_equal_to_oracle(L, orc, shape):
    K, N, P = shape
    prob = pqgen.make_problem(2, K, N, P=P, seed=K + N + P)
    rec, sz, w = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta)
    t = orc.pack(prob)
    assert np.array_equal(rec, t["rec_kernel"])
    assert np.array_equal(sz, t["sz_kernel"])
    assert np.array_equal(w, t["w"])


@pytest.mark.parametrize("shape", [(256, 128, 1), (640, 384, 3), (5120, 1024, 2)])
def test_pack5_byte_equal_to_oracle(L, orc, shape):
    """int5 packer: records, SZ (zp - 16), low nibbles and fifth-bit planes."""
    K, N, P = shape
    prob = pqgen.make_problem(2, K, N, P=P, seed=K + N + P + 5, bits=5)
    rec, sz, w, whi = pq.pq_pack5(prob.qweight, prob.qzeros, prob.qweight_hi, prob.qzeros_hi, prob.scales,
                                  prob.pairs, prob.theta)
    t = orc.pack5(prob)
    assert np.array_equal(rec, t["rec_kernel"])
    assert np.array_equal(sz, t["sz_kernel"])
    assert np.array_equal(w, t["w"])
    assert np.array_equal(whi, t["whi"])
    nul = C.c_void_p(0)
    assert L.pq_pack5(K, N, P, *([nul] * 11)) == 1


@pytest.mark.parametrize("pattern", ["identity", "alternate", "reversed", "mixed"])
def test_pack_chained_records_structured_pairings(L, orc, pattern):
    """The packer's chained record order against the oracle's on pairings with
    structure: the same pairs in every layer, an alternation that makes one
    cycle through all channels, reversed repeats, and random rows between them."""
    K, N, P = 256, 128, 2
    prob = pqgen.make_problem(1, K, N, P=P, seed=41)
    ident = np.arange(128, dtype=np.int16)
    shifted = np.roll(ident, -1)
    swapped = ident.reshape(64, 2)[:, ::-1].reshape(-1).copy()
    rows = {"identity": [ident] * 8, "alternate": [ident, shifted] * 4,
            "reversed": [ident, swapped] * 4}
    pairs = prob.pairs.copy()
    for p in range(P):
        for g in range(K // 128):
            seq = rows.get(pattern)
            for r in range(8):
                if seq is not None:
                    pairs[p, r, 128 * g:128 * g + 128] = seq[r]
                elif r % 2 == 0:
                    pairs[p, r, 128 * g:128 * g + 128] = [ident, shifted, swapped][(p + g + r // 2) % 3]
    rec, _, _ = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, pairs, prob.theta)
    assert np.array_equal(rec, orc.chain_records(orc.records(pairs, prob.theta)))


def test_pack_special_angles_and_scales(L, orc):
    """Angles and scales at the edges of f16: zero, subnormal, large, negative."""
    prob = pqgen.make_problem(1, 256, 256, seed=3)
    th = prob.theta.copy()
    specials = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x3C00, 0xBC00, 0x4248,
                         0x7BFF, 0xFBFF, 0x3555, 0x2E66], dtype=np.uint16)
    th.reshape(-1)[:len(specials)] = specials
    sc = prob.scales.copy()
    sc.reshape(-1)[:6] = np.array([0x0001, 0x03FF, 0x0400, 0x7BFF, 0x3C00, 0x0000], dtype=np.uint16)
    rec, szt, w = pq.pq_pack(prob.qweight, prob.qzeros, sc, prob.pairs, th)
    assert np.array_equal(rec, orc.chain_records(orc.records(prob.pairs, th)))
    assert np.array_equal(szt, orc.sz_kernel_layout(orc.sz_table(sc, prob.qzeros)))


def test_pack_sizes_and_errors(L):
    assert pq.pq_pack_sizes(5120, 17408, 1) == (8 * 40 * 64 * 8, 40 * 17408 * 4, 17408 * 2560)
    for args, st in [((100, 128, 1), 2), ((256, 130, 1), 2), ((256, 128, 0), 5), ((256, 128, 4), 5)]:
        with pytest.raises(pq.PQError) as e:
            pq.pq_pack_sizes(*args)
        assert e.value.status == st
    prob = pqgen.make_problem(1, 256, 128, seed=4)
    bad = prob.pairs.copy()
    bad[0, 5, 200] = bad[0, 5, 201]
    with pytest.raises(pq.PQError) as e:
        pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, bad, prob.theta)
    assert e.value.status == 4 and b"layer=5, group=1" in L.pq_last_error()
    bad[0, 5, 200] = -1
    with pytest.raises(pq.PQError):
        pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, bad, prob.theta)
    nul = C.c_void_p(0)
    assert L.pq_pack(256, 128, 1, nul, nul, nul, nul, nul, nul, nul, nul) == 1


# fake, 256-byte aligned addresses: every case below must be rejected by the
# host checks before any pointer is used.  They run only where no GPU is
# visible, so a case that wrongly passed the checks could never launch.
A, S = C.c_void_p(0x100000), C.c_void_p(0x200000)


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except ImportError:
        return True


cpu_only = pytest.mark.skipif(not _no_gpu(), reason="fake device pointers: CPU-only host checks")


@pytest.mark.parametrize("case,status", [
    (dict(a=None), 1), (dict(y=None), 1), (dict(M=0), 2), (dict(N=100), 2), (dict(K=200), 2),
    (dict(ldy=100), 2), (dict(P=0), 5), (dict(P=4), 5), (dict(P=2, pb1=128, pb2=128), 5),
    (dict(P=1, pb1=128, pb2=256), 5), (dict(P=3, pb1=128, pb2=64), 5),
    (dict(P=3, pb1=256, pb2=128), 5), (dict(P=2, pb1=100, pb2=256), 5),
    (dict(a=C.c_void_p(0x100004)), 3), (dict(asg=C.c_void_p(0x200002)), 3), (dict(ldy=260), 3),
])
@cpu_only
def test_gemm_argument_checks(L, case, status):
    args = dict(a=A, asg=S, rs=S, M=4, N=256, K=256, P=1, pb1=256, pb2=256, w=A, sz=A, y=A, ldy=256)
    args.update(case)
    order = ["a", "asg", "rs", "M", "N", "K", "P", "pb1", "pb2", "w", "sz", "y", "ldy"]
    vals = [args[k] for k in order]
    assert L.pq_gemm(*vals, None) == status
    assert L.pq_gemm_tc(*vals, None, None) == status
    assert L.pq_gemm_skinny(*vals, None, None) == status
    assert L.pq_gemm_ptok(*vals, None, None) == status
    v5 = vals[:10] + [A] + vals[10:]             # whi after w
    assert L.pq_gemm5(*v5, None) == status
    assert L.pq_gemm5_tc(*v5, None, None) == status
    assert L.pq_gemm5_skinny(*v5, None, None) == status
    assert L.pq_last_error()


@cpu_only
def test_skinny_rejects_large_m(L):
    vals = [A, S, S, 17, 256, 256, 1, 256, 256, A, A, A, 256]
    assert L.pq_gemm_skinny(*vals, None, None) == 2
    assert pq.pq_gemm_skinny_max_m() == 16


@pytest.mark.parametrize("case,status", [
    (dict(x=None), 1), (dict(M=0), 2), (dict(K=100), 2), (dict(ldx=128, K=256), 2),
    (dict(P=0), 5), (dict(P=4), 5), (dict(x=C.c_void_p(0x100008)), 3), (dict(ldx=260), 3),
    (dict(asg=C.c_void_p(0x200001)), 3),
])
@cpu_only
def test_rotate_quant_argument_checks(L, case, status):
    args = dict(x=A, M=4, K=256, ldx=256, P=1, rec=A, cs=A, a=A, asg=S, rs=S)
    args.update(case)
    order = ["x", "M", "K", "ldx", "P", "rec", "cs", "a", "asg", "rs"]
    assert L.pq_rotate_quant(*[args[k] for k in order], None) == status


X2, R2, O2, H2 = (C.c_void_p(0x300000), C.c_void_p(0x400000), C.c_void_p(0x500000),
                  C.c_void_p(0x600000))


@pytest.mark.parametrize("case,status", [
    (dict(x=None), 1), (dict(gamma=None), 1), (dict(res_out=None), 1), (dict(h=None), 1),
    (dict(M=0), 2), (dict(K=100), 2), (dict(ldx=128, K=256), 2),
    (dict(eps=-1e-6), 2), (dict(eps=float("nan")), 2), (dict(eps=float("inf")), 2),
    # the outputs may not overlap the inputs (other CTAs still read whole rows)
    (dict(res_out=R2), 2), (dict(res_out=C.c_void_p(0x300000 + 512)), 2), (dict(h=X2), 2),
    (dict(P=0), 5), (dict(P=4), 5), (dict(x=C.c_void_p(0x300008)), 3), (dict(ldx=260), 3),
    (dict(gamma=C.c_void_p(0x100004)), 3), (dict(asg=C.c_void_p(0x200001)), 3),
])
@cpu_only
def test_add_rms_rotate_quant_argument_checks(L, case, status):
    args = dict(x=X2, res=R2, gamma=A, eps=1e-6, M=4, K=256, ldx=256, P=1, rec=A, cs=A, res_out=O2, h=H2,
                a=A, asg=S, rs=S)
    args.update(case)
    order = ["x", "res", "gamma", "eps", "M", "K", "ldx", "P", "rec", "cs", "res_out", "h", "a", "asg", "rs"]
    vals = [args[k] for k in order]
    assert L.pq_add_rms_rotate_quant(*vals, None) == status
    assert L.pq_last_error()


@pytest.mark.parametrize("case,status", [
    (dict(y=None), 1), (dict(act=None), 1), (dict(M=0), 2), (dict(I=100), 2), (dict(ldy=256 + 128), 2),
    (dict(act=C.c_void_p(0x300000 + 1024)), 2),          # act overlapping y
    (dict(P=0), 5), (dict(P=4), 5), (dict(y=C.c_void_p(0x300008)), 3), (dict(ldy=516), 3),
    (dict(rs=C.c_void_p(0x200002)), 3),
])
@cpu_only
def test_silu_mul_rotate_quant_argument_checks(L, case, status):
    args = dict(y=X2, M=4, I=256, ldy=512, P=1, rec=A, cs=A, act=O2, a=A, asg=S, rs=S)
    args.update(case)
    order = ["y", "M", "I", "ldy", "P", "rec", "cs", "act", "a", "asg", "rs"]
    assert L.pq_silu_mul_rotate_quant(*[args[k] for k in order], None) == status
    assert L.pq_last_error()


@pytest.mark.parametrize("case,status", [
    (dict(x=None), 1), (dict(xr=None), 1), (dict(As=None), 1), (dict(M=0), 2), (dict(K=100), 2),
    (dict(ldx=128, K=256), 2), (dict(xr=C.c_void_p(0x300000 + 1024)), 2),     # xr overlapping x
    (dict(P=0), 5), (dict(P=4), 5), (dict(x=C.c_void_p(0x300008)), 3), (dict(xr=C.c_void_p(0x500008)), 3),
    (dict(ldx=260), 3), (dict(As=C.c_void_p(0x200002)), 3),
])
@cpu_only
def test_rotate_tokquant_argument_checks(L, case, status):
    args = dict(x=X2, M=4, K=256, ldx=256, P=1, rec=A, cs=A, xr=O2, a=A, As=S, rs=S)
    args.update(case)
    order = ["x", "M", "K", "ldx", "P", "rec", "cs", "xr", "a", "As", "rs"]
    assert L.pq_rotate_tokquant(*[args[k] for k in order], None) == status
    assert L.pq_last_error()


def test_device_calls_without_gpu_report_arch(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    vals = [A, S, S, 4, 256, 256, 1, 256, 256, A, A, A, 256]
    assert L.pq_gemm(*vals, None) == 6
    assert L.pq_rotate_quant(A, 4, 256, 256, 1, A, A, A, S, S, None) == 6
    assert L.pq_add_rms_rotate_quant(X2, R2, A, 1e-6, 4, 256, 256, 1, A, A, O2, H2, A, S, S, None) == 6
    assert L.pq_silu_mul_rotate_quant(X2, 4, 256, 512, 1, A, A, O2, A, S, S, None) == 6
    assert L.pq_rotate_tokquant(X2, 4, 256, 256, 1, A, A, O2, A, S, S, None) == 6
    assert L.pq_gemm_ptok(*vals, None, None) == 6
    v5 = vals[:10] + [A] + vals[10:]
    assert L.pq_gemm5(*v5, None) == 6 and L.pq_gemm5_tcn(*v5, None, None) == 6
    assert L.pq_gemm5_skinny(*v5, None, None) == 6
    assert L.pq_gemm5(*(vals[:10] + [None] + vals[10:]), None) == 1
    assert L.pq_e4m3_encode(S, A, 16, None) == 6
    with pytest.raises(pq.PQError) as e:
        pq._check(6, "probe")
    assert "PQ_ERR_ARCH" in str(e.value)
