"""Pins of the CPU oracle to things other than itself.

Each test ties one oracle function to a fact the pages or mathematics fix:
values printed in tests/golden (with their source), library routines
(numpy's binary16 conversion, torch's float8_e4m3fn conversion, numpy matmul),
exhaustive enumeration, closed forms, and brute force on tiny inputs.  The
cases are chosen so that a plausible slip (a swapped nibble slot, a dropped
term, a wrong sign or index, a transposed operand, a missing rounding step)
fails at least one of them.

Pages: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", sections
"Format", "Inference identity", "Design" 1-4, "Gates passed", and
"2026-09-15: hardware e4m3 convert in the producers".
"""
import json
import math
import os

import numpy as np
import pytest

import pqgen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ f16 / bf16
def test_f16_decode_all_patterns_match_numpy(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero kept
    assert math.copysign(1.0, orc.f16_to_double(0x8000)) == -1.0


def test_f16_rounding_matches_numpy_rne(orc):
    rng = np.random.default_rng(7)
    # random doubles across the whole f16 range, exact halfway points, subnormals, overflow
    vals = list(rng.standard_normal(4000) * np.exp2(rng.integers(-26, 17, 4000)))
    h = np.arange(0, 0x7C00, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals += list((lo + hi) / 2)            # ties: must go to the even pattern
    vals += [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -25 * 1.0001, 2.0 ** -24,
             3 * 2.0 ** -25, 0.0, -0.0]
    vals = np.array(vals, dtype=np.float64)
    vals = np.concatenate([vals, -vals])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f16_from_double(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ e4m3
def test_e4m3_decode_golden_and_table(orc):
    g = _golden("e4m3_ocp.json")
    for code, val in g["decode"]:
        got = orc.e4m3_decode(int(code, 16))
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    tab = orc.e4m3_decode_table()
    assert all(math.isnan(tab[int(c, 16)]) for c in g["nan_codes"])
    assert int(np.isfinite(tab).sum()) == g["finite_count"]
    pos = tab[:127]
    assert np.all(np.diff(pos) > 0)          # codes 0..126 increase strictly
    assert np.array_equal(tab[128:255], -pos)  # sign bit mirrors


def test_e4m3_decode_matches_torch(orc):
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_decode_table()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.array_equal(got[fin], ref[fin])


def test_e4m3_encode_golden(orc):
    for v, code in _golden("e4m3_ocp.json")["encode"]:
        assert orc.e4m3_encode(np.float32(v)) == int(code, 16), v


def test_e4m3_round_trip_all_codes(orc):
    """encode(decode(c)) == c for every finite code except -0 (0x80 -> 0x00)."""
    for c in range(256):
        v = orc.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert orc.e4m3_encode(np.float32(v)) == (0 if c == 0x80 else c), hex(c)


def test_e4m3_encode_nearest_value_all_2_32(orc):
    """Nearest-value optimality with ties to even over every binary32 pattern
    (binary search over the decoded table, an algorithm independent of the
    encoder's exponent/quantum arithmetic)."""
    bad, first = orc.e4m3_check_range(0, 1 << 32)
    assert bad == 0, "first disagreement at 0x%08x" % first


def test_e4m3_encode_matches_torch_conversion(orc):
    """torch's float -> float8_e4m3fn conversion (RNE, non-saturating) agrees
    with the oracle after the pages' wrapper (clamp +-448, zero -> 0x00)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add every value within +-2 ulp of each e4m3 grid point and midpoint
    tab = orc.e4m3_decode_table()[:127]
    mids = np.concatenate([tab, (tab[:-1] + tab[1:]) / 2]).astype(np.float32)
    near = mids.view(np.uint32)[:, None].astype(np.int64) + np.arange(-2, 3)[None, :]
    near = near[(near >= 0)].astype(np.uint32).view(np.float32)
    f = np.concatenate([f, near, -near]).astype(np.float32)
    t = torch.from_numpy(f).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    t = np.where((t & 0x7F) == 0, 0, t).astype(np.uint8)
    got = np.array([orc.e4m3_encode(float(v)) for v in f[:20000]], dtype=np.uint8)
    assert np.array_equal(got, t[:20000])
    # the rest in bulk through the exhaustive checker's own range API is already
    # covered; check the remaining near-boundary values one by one as well
    got2 = np.array([orc.e4m3_encode(float(v)) for v in f[-2 * len(near):]], dtype=np.uint8)
    assert np.array_equal(got2, t[-2 * len(near):])


# ------------------------------------------------------------------ AWQ format
def test_awq_unpack_golden(orc):
    for case in _golden("awq_unpack.json")["cases"]:
        w = np.array([[int(case["word_hex"], 16)]], dtype=np.uint32).view(np.int32)
        assert list(orc.unpack_awq(w, 8)[0]) == case["codes_by_column"], case


def test_repack_round_trip(orc):
    prob = pqgen.make_problem(4, 256, 128, seed=11)
    codes = orc.unpack_awq(prob.qweight, 128)          # [K, N]
    w = orc.repack(prob.qweight)                        # [N, K/2]
    # byte 4t + b of a row: code 8t + b (low nibble), code 8t + b + 4 (high)
    lo = (w & 15).astype(np.uint8).reshape(128, 32, 4)
    hi = (w >> 4).astype(np.uint8).reshape(128, 32, 4)
    back = np.empty((128, 32, 8), dtype=np.uint8)
    back[:, :, 0:4] = lo
    back[:, :, 4:8] = hi
    assert np.array_equal(back.reshape(128, 256), codes.T)
    # one byte by hand: row 5, bytes 4..7 hold codes 8..15
    assert w[5, 6] == codes[10, 5] | (codes[14, 5] << 4)


# ------------------------------------------------------------------ records
def _rec_fields(rec):
    ij = rec[..., 0].astype(np.int64) | (rec[..., 1].astype(np.int64) << 8) | \
        (rec[..., 2].astype(np.int64) << 16) | (rec[..., 3].astype(np.int64) << 24)
    c16 = (rec[..., 4].astype(np.uint16) | (rec[..., 5].astype(np.uint16) << 8))
    s16 = (rec[..., 6].astype(np.uint16) | (rec[..., 7].astype(np.uint16) << 8))
    return ij & 0xFF, (ij >> 8) & 0xFF, ij >> 16, c16, s16


def test_records_layout_and_trig(orc):
    prob = pqgen.make_problem(1, 384, 128, P=2, seed=5)
    rec = orc.records(prob.pairs, prob.theta)
    assert rec.shape == (2, 8, 3, 64, 8)
    i, j, upper, c16, s16 = _rec_fields(rec)
    assert np.all(upper == 0)
    pr = prob.pairs.reshape(2, 8, 3, 64, 2)
    assert np.array_equal(i, pr[..., 0]) and np.array_equal(j, pr[..., 1])
    th = prob.theta.reshape(2, 8, 3, 64).view(np.float16).astype(np.float64)
    assert np.array_equal(c16, np.cos(th).astype(np.float16).view(np.uint16))
    assert np.array_equal(s16, np.sin(th).astype(np.float16).view(np.uint16))
    c = c16.view(np.float16).astype(np.float64)
    s = s16.view(np.float16).astype(np.float64)
    assert np.max(np.abs(c * c + s * s - 1)) <= 2.0 ** -10


def test_records_special_angles(orc):
    K = 128
    pairs = np.tile(np.arange(128, dtype=np.int16), (1, 8, 1))
    theta = np.zeros((1, 8, 64), dtype=np.uint16)
    th = np.array([0.0, 0.5, -0.5, 0.25, -0.25, 1e-3, -1e-3, 0.49951171875])
    theta[0, :, :8] = np.float16(th).view(np.uint16)
    rec = orc.records(pairs, theta)
    _, _, _, c16, s16 = _rec_fields(rec)
    assert c16[0, 0, 0, 0] == 0x3C00 and s16[0, 0, 0, 0] == 0x0000      # theta = 0 -> (1, 0)
    assert c16[0, 0, 0, 1] == c16[0, 0, 0, 2]                             # cos even
    assert s16[0, 0, 0, 2] == (s16[0, 0, 0, 1] ^ 0x8000)                  # sin odd
    assert s16[0, 0, 0, 6] == (s16[0, 0, 0, 5] ^ 0x8000)


def test_pairs_validation(orc):
    prob = pqgen.make_problem(1, 256, 128, seed=1)
    assert orc.check_pairs(prob.pairs)
    bad = prob.pairs.copy()
    bad[0, 3, 130] = bad[0, 3, 131]
    assert not orc.check_pairs(bad)
    with pytest.raises(ValueError):
        orc.records(bad, prob.theta)
    bad2 = prob.pairs.copy()
    bad2[0, 0, 5] = 128
    assert not orc.check_pairs(bad2)


# ------------------------------------------------- chained record order
def _check_chain(plain, chained):
    """The chained records hold the same rotation as the plain ones: per
    layer the same pairs with the same cosines and the sines of reversed
    pairs negated, layer 0 unchanged, and every kept channel leads the next
    layer's slot, one kept channel per next-layer pair."""
    pi, pj, pup, pc, ps = _rec_fields(plain)
    ci, cj, cup, cc, cs_ = _rec_fields(chained)
    assert np.all(pup == 0)
    keep = cup & 0xFF
    assert np.all(cup >> 8 == 0) and np.all((keep == 0) | (keep == 1)) and np.all(keep[:, 7] == 0)
    P, L, G, T = pi.shape
    for p in range(P):
        for g in range(G):
            for r in range(L):
                want = {}
                for t in range(T):
                    want[(int(pi[p, r, g, t]), int(pj[p, r, g, t]))] = (int(pc[p, r, g, t]), int(ps[p, r, g, t]))
                for t in range(T):
                    u, v = int(ci[p, r, g, t]), int(cj[p, r, g, t])
                    if (u, v) in want:
                        assert want.pop((u, v)) == (int(cc[p, r, g, t]), int(cs_[p, r, g, t]))
                    else:
                        assert want.pop((v, u)) == (int(cc[p, r, g, t]), int(cs_[p, r, g, t]) ^ 0x8000)
                assert not want
                if r + 1 < L:
                    kept = [int(cj[p, r, g, t]) if keep[p, r, g, t] else int(ci[p, r, g, t]) for t in range(T)]
                    assert [int(ci[p, r + 1, g, t]) for t in range(T)] == kept


def test_chain_records_valid(orc):
    prob = pqgen.make_problem(1, 384, 128, P=3, seed=21)
    plain = orc.records(prob.pairs, prob.theta)
    chained = orc.chain_records(plain)
    _check_chain(plain, chained)
    assert np.array_equal(chained[:, 0, ..., :2], plain[:, 0, ..., :2])
    assert np.array_equal(chained[:, 0, ..., 4:], plain[:, 0, ..., 4:])


def test_chain_records_hand_examples(orc):
    """Small pairings worked by hand."""
    theta = np.zeros((1, 8, 64), dtype=np.uint16)
    theta[0, :, :] = np.float16(0.25).view(np.uint16)
    sin_bits = int(np.float16(np.sin(np.float64(np.float16(0.25)))).view(np.uint16))
    neg = sin_bits ^ 0x8000
    t = np.arange(64)
    ident = np.arange(128, dtype=np.int16)                      # (0,1), (2,3), ...
    shifted = np.roll(ident, -1)                                # (1,2), (3,4), ..., (127,0)
    swapped = ident.reshape(64, 2)[:, ::-1].reshape(-1).copy()  # (1,0), (3,2), ...

    # identity / shifted alternating: one cycle through all channels.
    # 0 -> 1: the walk from 0 keeps 1, 3, 5, ... (each slot's second channel);
    #   slot t of layer 1 is shifted's pair (2t+1, 2t+2) in its own order.
    # 1 -> 2: the walk from 0 meets slot 63 = (127, 0) and keeps 127, then
    #   125, ...: every slot keeps its first channel 2t+1, which leads
    #   identity's pair (2t, 2t+1) reversed (sine negated).
    # 2 -> 3: the walk from 0 meets slot 0 = (1, 0) and keeps 1: first again.
    ch = orc.chain_records(orc.records(np.stack([ident, shifted] * 4)[None], theta))
    i, j, up, c16, s16 = _rec_fields(ch)
    assert np.array_equal(up[0, :, 0], np.array([1] + [0] * 7)[:, None] * np.ones((1, 64), np.int64))
    for r in (1, 3, 5, 7):
        assert np.array_equal(i[0, r, 0], 2 * t + 1) and np.array_equal(j[0, r, 0], (2 * t + 2) % 128)
        assert np.all(s16[0, r, 0] == sin_bits)
    for r in (2, 4, 6):
        assert np.array_equal(i[0, r, 0], 2 * t + 1) and np.array_equal(j[0, r, 0], 2 * t)
        assert np.all(s16[0, r, 0] == neg)

    # the same pairs, the odd layers given reversed: cycles of length two;
    # 0 -> 1 keeps 2t+1, which is first in swapped's (2t+1, 2t): no negation
    ch = orc.chain_records(orc.records(np.stack([ident, swapped] * 4)[None], theta))
    i, j, up, c16, s16 = _rec_fields(ch)
    assert np.all(up[0, 0, 0] == 1)
    assert np.array_equal(i[0, 1, 0], 2 * t + 1) and np.array_equal(j[0, 1, 0], 2 * t)
    assert np.all(s16[0, 1, 0] == sin_bits)

    # the same pairs in the same order in every layer: layer 0 keeps 2t+1,
    # which then leads (2t+1, 2t) in every later layer, kept as the first
    ch = orc.chain_records(orc.records(np.stack([ident] * 8)[None], theta))
    i, j, up, c16, s16 = _rec_fields(ch)
    assert np.all(up[0, 0, 0] == 1) and np.all(up[0, 1:, 0] == 0)
    for r in range(1, 8):
        assert np.array_equal(i[0, r, 0], 2 * t + 1) and np.array_equal(j[0, r, 0], 2 * t)
        assert np.all(s16[0, r, 0] == neg)
    assert np.all(c16 == c16[0, 0, 0, 0])


def test_chain_records_rotate_identically(orc):
    """The oracle's prologue gives the same bits with the chained records as
    with the pages' order (the reversal with a negated sine is exact)."""
    prob = pqgen.make_problem(37, 640, 128, P=2, seed=8)
    plain = orc.records(prob.pairs, prob.theta)
    chained = orc.chain_records(plain)
    assert not np.array_equal(plain, chained)
    for x1, x2 in zip(orc.rotate_quant(prob.x, prob.cs, plain), orc.rotate_quant(prob.x, prob.cs, chained)):
        assert np.array_equal(np.asarray(x1).view(np.uint8), np.asarray(x2).view(np.uint8))


# ------------------------------------------------------------------ SZ table
def test_sz_exhaustive_against_numpy(orc):
    """(sc, f16(sc*(zp-8))) for every positive finite f16 scale and zp 0..15."""
    sc = np.arange(1, 0x7C00, dtype=np.uint32).astype(np.uint16)      # all positive finite f16
    G = 16
    n = len(sc)
    N = (n + 127) // 128 * 128
    scales = np.zeros((G, N), dtype=np.uint16)
    scales[:, :n] = sc[None, :]
    zp = np.repeat(np.arange(16, dtype=np.uint32)[:, None], N // 8, axis=1)   # row g: zp = g
    qzeros = np.zeros((G, N // 8), dtype=np.uint32)
    for slot in range(8):
        qzeros |= zp << np.uint32(4 * slot)
    sz = orc.sz_table(scales, qzeros.view(np.int32))
    scf = sc.view(np.float16).astype(np.float32)
    for g in range(G):
        with np.errstate(over="ignore"):
            ref = (scf * np.float32(g - 8)).astype(np.float16).view(np.uint16)
        assert np.array_equal(sz[g, :n, 0], sc)
        assert np.array_equal(sz[g, :n, 1], ref), g


# ------------------------------------------------------------------ rotation
def _dense_R(rec, p, g):
    """fp64 128x128 matrix of layers 0..7 of (p, g) built from the record
    values: each layer maps x_i -> c x_i + s x_j, x_j -> -s x_i + c x_j."""
    i, j, _, c16, s16 = _rec_fields(rec[p, :, g])
    c = c16.view(np.float16).astype(np.float64)
    s = s16.view(np.float16).astype(np.float64)
    R = np.eye(128)
    for r in range(8):
        L = np.zeros((128, 128))
        for t in range(64):
            a, b = i[r, t], j[r, t]
            L[a, a] = c[r, t]
            L[a, b] = s[r, t]
            L[b, a] = -s[r, t]
            L[b, b] = c[r, t]
        R = L @ R
    return R


def test_rotation_fp32_vs_dense_fp64(orc):
    prob = pqgen.make_problem(1, 256, 128, P=2, seed=9)
    rec = orc.records(prob.pairs, prob.theta)
    rng = np.random.default_rng(0)
    for p in range(2):
        for g in range(2):
            R = _dense_R(rec, p, g)
            v = rng.standard_normal(128).astype(np.float32)
            got = orc.rotate_group_f32(rec, p, g, v).astype(np.float64)
            ref = R @ v.astype(np.float64)
            # 8 layers of 3 roundings each on values of size ~|v|
            assert np.max(np.abs(got - ref)) <= 64 * 2.0 ** -24 * np.max(np.abs(v)) * 4
            # the layer's own fp64 norm identity: sum v'^2 = sum (c^2+s^2)(vi^2+vj^2)
            i, j, _, c16, s16 = _rec_fields(rec[p, :, g])
            w = v.astype(np.float64)
            for r in range(8):
                c = c16[r].view(np.float16).astype(np.float64)
                s = s16[r].view(np.float16).astype(np.float64)
                w2 = w.copy()
                w2[i[r]] = c * w[i[r]] + s * w[j[r]]
                w2[j[r]] = c * w[j[r]] - s * w[i[r]]
                lhs = np.sum(w2 ** 2)
                rhs = np.sum((c * c + s * s) * (w[i[r]] ** 2 + w[j[r]] ** 2))
                assert abs(lhs - rhs) <= 1e-12 * rhs
                w = w2


def test_rotation_identity_layers_is_exact(orc):
    prob = pqgen.make_problem(1, 128, 128, seed=2)
    theta = np.zeros_like(prob.theta)
    rec = orc.records(prob.pairs, theta)
    v = np.random.default_rng(1).standard_normal(128).astype(np.float32)
    assert np.array_equal(orc.rotate_group_f32(rec, 0, 0, v), v)


def test_identity_rotate_activations_equals_rotate_weights(orc):
    """y = ((x*cs) R^T) W^T == (x*cs) (W R)^T ... i.e. moving the rotation onto
    the weight rows as the transposed layers (7..0, negated angles); fp64,
    no quantisation, <= 1e-12 relative (page: "Inference identity")."""
    prob = pqgen.make_problem(3, 384, 256, P=3, seed=4, pb=(128, 256))
    W = np.random.default_rng(2).standard_normal((256, 384))
    y1 = orc.linear_rotx_f64(prob.x, prob.cs, prob.pairs, prob.theta, W, 128, 256)
    y2 = orc.linear_rotw_f64(prob.x, prob.cs, prob.pairs, prob.theta, W, 128, 256)
    assert np.linalg.norm(y1 - y2) <= 1e-12 * np.linalg.norm(y1)
    # and a transposed (wrong) direction does not satisfy it
    theta_neg = (prob.theta ^ np.uint16(0x8000))
    y3 = orc.linear_rotw_f64(prob.x, prob.cs, prob.pairs, theta_neg, W, 128, 256)
    assert np.linalg.norm(y1 - y3) > 1e-3 * np.linalg.norm(y1)


# ------------------------------------------------------------------ prologue
def _torch_quant(v, scale_const=None):
    """Per-group e4m3 quantisation of fp32 rows v [R, 128] with torch ops:
    scale = amax * fl(1/448), q = v / scale, torch's e4m3 conversion after the
    pages' wrapper, row-sum as the fp32 rounding of the fp64 sum of decodes."""
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(448.0, dtype=torch.float32)
    amax = t.abs().amax(dim=1)
    scale = amax * inv
    q = t / scale[:, None]
    codes = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    codes = torch.where((codes & 0x7F) == 0, torch.zeros_like(codes), codes)
    codes = torch.where(scale[:, None] == 0, torch.zeros_like(codes), codes)
    dec = codes.view(torch.float8_e4m3fn).to(torch.float64)
    rs = dec.sum(dim=1).to(torch.float32)
    return codes.numpy(), scale.numpy(), rs.numpy()


def test_prologue_theta_zero_is_plain_group_quant(orc):
    prob = pqgen.make_problem(5, 256, 128, P=2, seed=6)
    theta = np.zeros_like(prob.theta)
    rec = orc.records(prob.pairs, theta)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, rec)
    x = orc.bf16_bits_to_f32(prob.x)
    for p in range(2):
        v = x * prob.cs[p].view(np.float16).astype(np.float32)[None, :]
        codes, scale, rsum = _torch_quant(v.reshape(-1, 128))
        assert np.array_equal(a[p].reshape(-1, 128), codes)
        assert np.array_equal(asg[p].T.reshape(-1), scale)       # asg is [G, M]
        assert np.array_equal(rs[p].T.reshape(-1), rsum)


def test_prologue_rotated_quant_matches_torch_and_dense(orc):
    prob = pqgen.make_problem(6, 384, 128, P=3, seed=8, pb=(128, 128))
    rec = orc.records(prob.pairs, prob.theta)
    a, asg, rs, v = orc.rotate_quant(prob.x, prob.cs, rec, want_v=True)
    x = orc.bf16_bits_to_f32(prob.x).astype(np.float64)
    for p in range(3):
        codes, scale, rsum = _torch_quant(v[p].reshape(-1, 128))
        assert np.array_equal(a[p].reshape(-1, 128), codes)
        assert np.array_equal(asg[p].T.reshape(-1), scale)
        assert np.array_equal(rs[p].T.reshape(-1), rsum)
        for g in range(3):
            R = _dense_R(rec, p, g)
            xs = x[:, 128 * g:128 * g + 128] * prob.cs[p, 128 * g:128 * g + 128].view(np.float16)
            ref = xs @ R.T
            err = np.abs(v[p][:, 128 * g:128 * g + 128] - ref)
            assert np.max(err) <= 2e-6 * np.max(np.abs(xs))


def test_prologue_pow2_scaling_and_zero_group(orc):
    prob = pqgen.make_problem(4, 256, 128, seed=12)
    rec = orc.records(prob.pairs, prob.theta)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, rec)
    x4 = pqgen.to_bf16_bits(orc.bf16_bits_to_f32(prob.x) * np.float32(4.0))
    a4, asg4, rs4 = orc.rotate_quant(x4, prob.cs, rec)
    assert np.array_equal(a, a4) and np.array_equal(rs, rs4) and np.array_equal(asg4, asg * 4)
    x0 = prob.x.copy()
    x0[1, 128:] = 0
    a0, asg0, rs0 = orc.rotate_quant(x0, prob.cs, rec)
    assert np.all(a0[0, 1, 128:] == 0) and asg0[0, 1, 1] == 0 and rs0[0, 1, 1] == 0
    # untouched groups unchanged
    assert np.array_equal(a0[0, 0], a[0, 0]) and np.array_equal(a0[0, 1, :128], a[0, 1, :128])


def test_subnormal_heavy_inputs_produce_subnormal_codes(orc):
    prob = pqgen.make_problem(8, 256, 128, seed=2, x_mode="sparse", theta_range=1e-4)
    rec = orc.records(prob.pairs, prob.theta)
    a, _, _ = orc.rotate_quant(prob.x, prob.cs, rec)
    sub = ((a & 0x78) == 0) & ((a & 7) != 0)
    assert sub.mean() > 0.5


# ------------------------------------------------------------------ GEMM
def _dequant_dense(orc, prob, tab):
    """W [N, K] = (c - zp) * sc in fp64 (format-true, zero point exact)."""
    K, N = prob.K, prob.N
    codes = tab["codes"].astype(np.float64)                       # [K, N]
    zp = np.repeat(tab["zp"].astype(np.float64), 128, axis=0)     # [K, N]
    sc = np.repeat(prob.scales.view(np.float16).astype(np.float64), 128, axis=0)
    return ((codes - zp) * sc).T


def test_gemm_brute_force_tiny(orc):
    """Tiny workload: materialise W = (c-zp)*sc and A = dec*asg, triple-loop
    via matmul, compare with the fold form (format-true to 1e-12, table-true
    to the f16 rounding of zscale)."""
    prob = pqgen.config_problem("tiny")
    tab = orc.pack(prob)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, tab["rec"])
    dec = orc.e4m3_decode_table()[a[0]]                           # [M, K]
    A = dec * np.repeat(asg[0].T.astype(np.float64), 128, axis=1)
    W = _dequant_dense(orc, prob, tab)
    y_bf = A @ W.T
    y_fmt = orc.gemm_format_f64(a, asg, tab["codes"], tab["zp"], prob.scales, prob.pb1, prob.pb2)
    assert np.max(np.abs(y_fmt - y_bf)) <= 1e-12 * np.max(np.abs(y_bf))
    y_tab = orc.gemm_f64(a, asg, rs, tab["codes"], tab["sz"], prob.pb1, prob.pb2)
    # |zs_f16 - sc*(zp-8)| <= 2^-11 |sc*(zp-8)|, times |asg * rs| per group
    zs_exact = prob.scales.view(np.float16).astype(np.float64) * (tab["zp"].astype(np.float64) - 8)
    bound = np.zeros_like(y_bf)
    for g in range(prob.G):
        bound += np.abs(asg[0, g].astype(np.float64) * rs[0, g])[:, None] * \
            (2.0 ** -11 * np.abs(zs_exact[g]))[None, :]
    assert np.all(np.abs(y_tab - y_bf) <= bound * 1.0001 + 1e-15)
    assert orc.rel_err(y_tab, y_bf) < 1e-3
    # a dropped zero-point term would be far off
    sz_nozp = tab["sz"].copy()
    sz_nozp[..., 1] = 0
    y_bad = orc.gemm_f64(a, asg, rs, tab["codes"], sz_nozp, prob.pb1, prob.pb2)
    assert orc.rel_err(y_bad, y_bf) > 1e-2


def test_gemm_all_codes_eight_is_zero(orc):
    M, K, N = 3, 256, 128
    a = pqgen.random_codes(1, M, K, seed=1)
    asg = pqgen.random_scales(1, K // 128, M, seed=1)
    rs = np.zeros((1, K // 128, M), dtype=np.float32)
    for g in range(K // 128):
        rs[0, g] = orc.e4m3_decode_table()[a[0][:, 128 * g:128 * g + 128]].sum(axis=1)
    codes = np.full((K, N), 8, dtype=np.uint8)
    sc = np.full((K // 128, N), 0x2000, dtype=np.uint16)
    sz = np.stack([sc, np.zeros_like(sc)], axis=-1)                 # zp = 8 -> zscale 0
    y = orc.gemm_f64(a, asg, rs, codes, sz, N, N)
    assert np.all(y == 0)


def test_gemm_partitions_equal_sliced_launches(orc):
    """Merged P=3 GEMM == three single-partition GEMMs on column slices."""
    prob = pqgen.make_problem(5, 256, 384, P=3, seed=13, pb=(128, 256))
    tab = orc.pack(prob)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, tab["rec"])
    y = orc.gemm_f64(a, asg, rs, tab["codes"], tab["sz"], 128, 256)
    for p, (lo, hi) in enumerate([(0, 128), (128, 256), (256, 384)]):
        ys = orc.gemm_f64(a[p:p + 1], asg[p:p + 1], rs[p:p + 1],
                          np.ascontiguousarray(tab["codes"][:, lo:hi]),
                          np.ascontiguousarray(tab["sz"][:, lo:hi]), 128, 128)
        assert np.array_equal(y[:, lo:hi], ys)
    # and the partitions really differ
    assert not np.array_equal(a[0], a[1])


def test_gemm_sampled_equals_full(orc):
    prob = pqgen.make_problem(7, 256, 256, P=2, seed=14, pb=(128, 256))
    tab = orc.pack(prob)
    a, asg, rs = orc.rotate_quant(prob.x, prob.cs, tab["rec"])
    y = orc.gemm_f64(a, asg, rs, tab["codes"], tab["sz"], 128, 256)
    ms = np.array([0, 6, 3, 2])
    ns = np.array([0, 255, 128, 127])
    ys = orc.gemm_f64_sampled(ms, ns, a, asg, rs, tab["codes"], tab["sz"], 128, 256)
    assert np.array_equal(ys, y[ms, ns])


def test_end_to_end_against_unquantised_layer(orc):
    """The quantised layer tracks the exact fp64 layer to the e4m3 activation
    floor (the pages report ~2.6e-2 for real activations)."""
    prob = pqgen.make_problem(16, 512, 256, seed=15)
    tab = orc.pack(prob)
    _, _, _, y = orc.layer(prob, tab)
    W = _dequant_dense(orc, prob, tab)
    y_exact = orc.linear_rotx_f64(prob.x, prob.cs, prob.pairs, prob.theta, W, 256, 256)
    e = orc.rel_err(y, y_exact)
    assert 1e-3 < e < 6e-2
