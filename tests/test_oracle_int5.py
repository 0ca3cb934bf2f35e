"""Pins of the oracle's int5 (W5A8) weight format and GEMM.

Page: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", section
"2026-09-10: int5 W5A8 ParoQuant": 5-bit codes c with the low nibbles in the
int4 AWQ words and the fifth bit in [K, N/32] int32 planes; (c - 16) runs
-16..15 and every value of that range is exact in e4m3, so the GEMM algebra of
the int4 path carries over with 16 in place of 8.

The pins: single-bit planes against the stated bit order, a round trip
through a packer written here from the page's AWQ slot order, numpy's binary16
rounding for the SZ table, brute-force dense matmul on a tiny layer, and the
offset-8 GEMM as a plausible slip that must fail.
"""
import numpy as np
import pytest

import pqgen

AWQ_ORDER = [0, 2, 4, 6, 1, 3, 5, 7]     # word slot i holds column AWQ_ORDER[i] of its octet


def _pack_awq(codes):
    """codes uint8 [rows, N] (0..15) -> int32 [rows, N/8], slot i <- column AWQ_ORDER[i]."""
    rows, N = codes.shape
    w = np.zeros((rows, N // 8), dtype=np.uint32)
    for i, col in enumerate(AWQ_ORDER):
        w |= codes[:, col::8].astype(np.uint32) << np.uint32(4 * i)
    return w.view(np.int32)


def _pack_plane(bits):
    """bits uint8 [rows, N] (0/1) -> int32 [rows, N/32], column 32w + j in bit j."""
    rows, N = bits.shape
    w = np.zeros((rows, N // 32), dtype=np.uint64)
    for j in range(32):
        w |= bits[:, j::32].astype(np.uint64) << np.uint64(j)
    return w.astype(np.uint32).view(np.int32)


def test_plane_single_bits(orc):
    """Bit j of plane word w is the fifth bit of column 32w + j."""
    N = 96
    for w in range(3):
        for j in (0, 1, 7, 8, 15, 16, 30, 31):
            plane = np.zeros((1, N // 32), dtype=np.uint32)
            plane[0, w] = np.uint32(1) << np.uint32(j)
            bits = orc.unpack_plane(plane.view(np.int32), N)[0]
            assert bits.sum() == 1 and bits[32 * w + j] == 1, (w, j)


def test_codes5_round_trip_through_independent_packer(orc):
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 32, size=(6, 128), dtype=np.uint8)
    lo, hi = _pack_awq(codes & 15), _pack_plane(codes >> 4)
    assert np.array_equal(orc.codes5(lo, hi, 128), codes)


def test_signed_codes_exact_in_e4m3(orc):
    """Every c - 16, c in 0..31, is an e4m3 value (alone and scaled by 2^-9):
    the property the page gives for using (c - 16) as the MMA operand."""
    dec = orc.e4m3_decode_table()
    for c in range(32):
        for unit in (1.0, 2.0 ** -9):
            v = np.float32((c - 16) * unit)
            assert dec[orc.e4m3_encode(v)] == v, c
    # and 17, the first value past the range on the positive side, is not
    assert dec[orc.e4m3_encode(np.float32(17.0))] != 17.0


def test_sz5_against_numpy(orc):
    rng = np.random.default_rng(6)
    G, N = 4, 256
    zp = rng.integers(0, 32, size=(G, N), dtype=np.uint8)
    zp[0, :32] = np.arange(32)                       # every zero point at least once
    scales = pqgen.f16_bits(rng.uniform(0.002, 0.02, size=(G, N)))
    scales[1, :4] = pqgen.f16_bits(np.array([0.0, 65504.0, 2.0 ** -24, 1.0]))
    sz = orc.sz5_table(scales, _pack_awq(zp & 15), _pack_plane(zp >> 4))
    sc = scales.view(np.float16).astype(np.float32)
    with np.errstate(over="ignore"):          # 65504 * 15 rounds to +inf in binary16
        want = (sc * (zp.astype(np.float32) - np.float32(16))).astype(np.float16).view(np.uint16)
    assert np.array_equal(sz[..., 0], scales)
    assert np.array_equal(sz[..., 1], want)
    assert np.all(sz[0, 16, 1] == 0)                  # zp = 16 -> zscale 0


def test_repack5_layout(orc):
    prob = pqgen.make_problem(4, 512, 256, seed=12, bits=5)
    codes = orc.codes5(prob.qweight, prob.qweight_hi, 256)      # [K, N]
    w, whi = orc.repack5(prob.qweight, prob.qweight_hi)
    back = np.empty((256, 64, 8), dtype=np.uint8)      # byte 4t + b: codes 8t + b, 8t + b + 4
    back[:, :, 0:4] = (w & 15).reshape(256, 64, 4)
    back[:, :, 4:8] = (w >> 4).reshape(256, 64, 4)
    back = back.reshape(256, 512)
    # fifth bit of k = 32t + 16h + 4q + j: bit 4h + q of byte 4t + j
    k = np.arange(512)
    byte = 4 * (k // 32) + k % 4
    sh = 4 * ((k % 32) // 16) + (k % 16) // 4
    fifth = (whi[:, byte] >> sh[None, :].astype(np.uint8)) & 1                   # [N, K]
    back += 16 * fifth.astype(np.uint8)
    # one bit by hand: k = 53 = 32 + 16 + 4 + 1 sits in byte 5, bit 5
    assert (whi[7, 5] >> 5) & 1 == codes[53, 7] >> 4
    assert np.array_equal(back, codes.T)
    assert 0.4 < (codes >= 16).mean() < 0.6


def _dequant_dense5(prob, tab):
    codes = tab["codes"].astype(np.float64)                       # [K, N]
    zp = np.repeat(tab["zp"].astype(np.float64), 128, axis=0)
    sc = np.repeat(prob.scales.view(np.float16).astype(np.float64), 128, axis=0)
    return ((codes - zp) * sc).T


@pytest.mark.parametrize("P,pb", [(1, None), (3, (128, 256))])
def test_gemm5_brute_force_tiny(orc, P, pb):
    prob = pqgen.make_problem(4, 256, 384 if P == 3 else 128, P=P, pb=pb, seed=21, bits=5)
    tab = orc.pack5(prob)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, tab["rec"])
    W = _dequant_dense5(prob, tab)                                # [N, K]
    dec = orc.e4m3_decode_table()
    y_bf = np.empty((prob.M, prob.N))
    for n in range(prob.N):
        p = (n >= prob.pb1) + (n >= prob.pb2)
        A = dec[a[p]] * np.repeat(asg[p].T.astype(np.float64), 128, axis=1)
        y_bf[:, n] = A @ W[n]
    y_fmt = orc.gemm_format_f64(a, asg, tab["codes"], tab["zp"], prob.scales, prob.pb1, prob.pb2)
    assert np.max(np.abs(y_fmt - y_bf)) <= 1e-12 * np.max(np.abs(y_bf))
    y_tab = orc.gemm5_f64(a, asg, rs, tab["codes"], tab["sz"], prob.pb1, prob.pb2)
    zs_exact = prob.scales.view(np.float16).astype(np.float64) * (tab["zp"].astype(np.float64) - 16)
    bound = np.zeros_like(y_bf)
    for n in range(prob.N):
        p = (n >= prob.pb1) + (n >= prob.pb2)
        for g in range(prob.G):
            bound[:, n] += np.abs(asg[p, g].astype(np.float64) * rs[p, g]) * 2.0 ** -11 * abs(zs_exact[g, n])
    assert np.all(np.abs(y_tab - y_bf) <= bound * 1.0001 + 1e-15)
    assert orc.rel_err(y_tab, y_bf) < 1e-3
    # the int4 offset on int5 codes is a plausible slip: far off
    y_off8 = orc.gemm_f64(a, asg, rs, tab["codes"], tab["sz"], prob.pb1, prob.pb2)
    assert orc.rel_err(y_off8, y_bf) > 1e-2


def test_gemm5_sampled_equals_full(orc):
    prob = pqgen.make_problem(7, 256, 256, P=2, seed=14, pb=(128, 256), bits=5)
    tab = orc.pack5(prob)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, tab["rec"])
    y = orc.gemm5_f64(a, asg, rs, tab["codes"], tab["sz"], 128, 256)
    ms = np.array([0, 6, 3, 2])
    ns = np.array([0, 255, 128, 127])
    assert np.array_equal(orc.gemm5_f64_sampled(ms, ns, a, asg, rs, tab["codes"], tab["sz"], 128, 256),
                          y[ms, ns])
