"""Pins of the oracle's fused producer (residual add + Gemma RMSNorm + rotate
+ quant) to things other than itself: torch's bfloat16 rounding and its
rms_norm, exact sums, closed forms and exact scaling identities.

Page: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", section
"2026-09-02/03: rotation stream (fused add + RMSNorm + rotate + quant
producers)": one producer does residual add + Gemma RMSNorm (vLLM's op order)
+ channel scale + rotation + per-group quant and returns (hs, residual, A,
ASG, RS).  The summation order and the rsqrt rounding are readings (R16).
"""
import math

import numpy as np
import pytest

import pqgen

torch = pytest.importorskip("torch")


def bf16_bits(f32):
    """torch's float32 -> bfloat16 rounding (RNE), as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def problem(M, K, P=1, seed=0, scale=1.0):
    prob = pqgen.make_problem(M, K, 256, P=P, seed=seed)
    rng = np.random.default_rng(seed + 100)
    res = bf16_bits(rng.standard_normal((M, K)).astype(np.float32) * np.float32(scale))
    gamma = bf16_bits(rng.standard_normal(K).astype(np.float32) * np.float32(0.2))
    return prob, res, gamma


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(3)
    f = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 1000,
                        # exact ties: 1 + 2^-8 (tie to 1), 1 + 3 * 2^-8 (tie to 1 + 2^-6)
                        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)], np.float32)])
    got = np.array([orc.bf16_from_float(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, bf16_bits(f))
    assert got[-3] == 0x3F80 and got[-2] == 0x3F82 and got[-1] == 0xBF80


def test_row_sumsq_exact_cases(orc):
    # equal powers of two: every partial sum is exact, the total is K c^2
    for K, c in ((128, 0.5), (5120, 2.0 ** -6), (896, 3.0)):
        s = np.full(K, c, dtype=np.float32)
        assert orc.row_sumsq(s) == np.float32(K * c * c)
    # a few nonzero entries: every partial sum is exact
    s = np.zeros(512, np.float32)
    s[[5, 200, 300, 511]] = [2.0, -3.0, 0.25, 1.0]
    assert orc.row_sumsq(s) == np.float32(4 + 9 + 0.0625 + 1)


def test_row_sumsq_within_pairwise_bound(orc):
    rng = np.random.default_rng(4)
    for K in (128, 1024, 5120):
        s = bf16_to_f32(bf16_bits(rng.standard_normal(K).astype(np.float32)))
        exact = math.fsum(float(v) * float(v) for v in s)
        got = float(orc.row_sumsq(s))
        # per lane: G sequential adds of pair sums; then 6 pairwise levels
        depth = K // 128 + 1 + 6
        assert abs(got - exact) <= depth * 2.0 ** -24 * exact * 1.01


def test_residual_and_norm_match_torch(orc):
    M, K = 6, 1024
    prob, res, gamma = problem(M, K, seed=5)
    t = orc.pack(prob)
    eps = 1e-6
    res_out, h, a, asg, rs = orc.add_rms_rotate_quant(prob.x, res, gamma, eps, prob.cs, t["rec"])
    xs = torch.from_numpy(bf16_to_f32(prob.x)).to(torch.bfloat16)
    rr = torch.from_numpy(bf16_to_f32(res)).to(torch.bfloat16)
    s = xs + rr                                   # bf16 add: fp32 sum rounded once
    assert np.array_equal(res_out, s.view(torch.int16).numpy().view(np.uint16))
    w = 1.0 + torch.from_numpy(bf16_to_f32(gamma))
    ref = torch.nn.functional.rms_norm(s.float(), (K,), w, eps)
    # the same formula with another reduction order and rsqrt: within one
    # bf16 step of the fp32 reference (plus a hair for the reference's own
    # rounding)
    got = torch.from_numpy(bf16_to_f32(h))
    step = 2.0 ** -7 * ref.abs()
    assert bool(((got - ref).abs() <= step * 1.01 + 1e-30).all())


def test_quant_stage_is_rotate_quant_of_h(orc):
    M, K, P = 4, 512, 3
    prob, res, gamma = problem(M, K, P=P, seed=6)
    t = orc.pack(prob)
    res_out, h, a, asg, rs = orc.add_rms_rotate_quant(prob.x, res, gamma, 1e-5, prob.cs, t["rec"])
    a2, asg2, rs2 = orc.rotate_quant(h, prob.cs, t["rec"])
    assert np.array_equal(a, a2) and np.array_equal(asg, asg2) and np.array_equal(rs, rs2)


def test_zero_rows_and_zero_weight(orc):
    M, K = 3, 256
    prob, res, gamma = problem(M, K, seed=7)
    t = orc.pack(prob)
    res0 = prob.x.copy() ^ np.uint16(0x8000)     # x + (-x) = 0 in every channel
    _, h, a, asg, rs = orc.add_rms_rotate_quant(prob.x, res0, gamma, 1e-6, prob.cs, t["rec"])
    assert not h.any() and not a.any() and not asg.any() and not rs.any()
    # Gemma weight -1: (1 + w) = 0 zeroes every normed value
    gneg = np.full(K, 0xBF80, dtype=np.uint16)   # bf16 -1.0
    _, h, a, asg, rs = orc.add_rms_rotate_quant(prob.x, res, gneg, 1e-6, prob.cs, t["rec"])
    assert not (h & 0x7FFF).any() and not a.any() and not asg.any()


def test_scaling_by_two_leaves_h_unchanged(orc):
    # with eps = 0: s -> 2s makes ss -> 4 ss, sqrt -> 2 sqrt, inv -> inv / 2
    # exactly, so h is bit-identical; a dropped square or a missing 1/K breaks it
    M, K = 4, 640
    prob, res, gamma = problem(M, K, seed=8)
    t = orc.pack(prob)
    x2 = bf16_bits(bf16_to_f32(prob.x) * 2)
    r2 = bf16_bits(bf16_to_f32(res) * 2)
    o1 = orc.add_rms_rotate_quant(prob.x, res, gamma, 0.0, prob.cs, t["rec"])
    o2 = orc.add_rms_rotate_quant(x2, r2, gamma, 0.0, prob.cs, t["rec"])
    assert np.array_equal(o1[1], o2[1])
    assert np.array_equal(bf16_to_f32(o2[0]), 2 * bf16_to_f32(o1[0]))


def test_norm_of_constant_row_is_one(orc):
    # s = c everywhere (power of two), gamma = 0, eps = 0: h = sign(c) exactly
    M, K = 2, 384
    prob, _, _ = problem(M, K, seed=9)
    t = orc.pack(prob)
    x = np.full((M, K), 0x3E80, dtype=np.uint16)       # 0.25
    x[1] = 0xC100                                      # -8.0
    zero = np.zeros((M, K), dtype=np.uint16)
    _, h, _, _, _ = orc.add_rms_rotate_quant(x, zero, np.zeros(K, np.uint16), 0.0, prob.cs, t["rec"])
    assert (h[0] == 0x3F80).all() and (h[1] == 0xBF80).all()


# ---------------------------------------------------------------- silu-mul producer
# Page: same log, "2026-09-03: rotation stream 2 (silu-mul, GDN gated norm,
# attention gate fused with rotate+quant)": MODE 0 is silu(g)*u with a
# bf16-rounded silu and a bf16 product, then the rotate_quant body.  The exp
# routine is a reading (R17) fixed so both implementations agree bit for bit.
def test_exp32_accuracy(orc):
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001), [0.0, -1e-8, 1e-8, 0.5, -0.5, 1.0]])
    for x in xs:
        x = float(np.float32(x))
        got, ref = orc.exp32(x), math.exp(x)
        assert abs(got - ref) <= 2.0 ** -22 * ref, (x, got, ref)
    assert orc.exp32(0.0) == 1.0
    assert orc.exp32(89.0) == math.inf and orc.exp32(-104.0) == 0.0


def test_silu_mul_matches_torch(orc):
    rng = np.random.default_rng(11)
    g = bf16_bits(np.concatenate([rng.standard_normal(3000).astype(np.float32) * 4,
                                  np.array([0.0, 50.0, -100.0, 1.0, -1.0], np.float32)]))
    u = bf16_bits(rng.standard_normal(g.size).astype(np.float32) * 2)
    got = np.array([orc.silu_mul(int(a), int(b)) for a, b in zip(g, u)], dtype=np.uint16)
    gt = torch.from_numpy(bf16_to_f32(g)).to(torch.bfloat16)
    ut = torch.from_numpy(bf16_to_f32(u)).to(torch.bfloat16)
    ref = (torch.nn.functional.silu(gt.float()).to(torch.bfloat16) * ut).float().numpy()
    gotf = bf16_to_f32(got)
    # another exp can move the bf16 silu by one step, and the product by one more
    assert np.all(np.abs(gotf - ref) <= 2.0 ** -6 * np.abs(ref) + 1e-37)
    assert np.mean(gotf == ref) > 0.99
    # special values: silu(0) = 0; silu(50) = 50 exactly; silu(-100) = -0
    assert gotf[-5] == 0.0
    assert gotf[-4] == bf16_to_f32(bf16_bits(np.float32(50.0) * bf16_to_f32(u[-4:-3])))[0]
    assert gotf[-3] == 0.0


def test_silu_mul_quant_stage_is_rotate_quant(orc):
    M, I, P = 3, 384, 2
    prob = pqgen.make_problem(M, I, 256, P=P, seed=12, pb=(128, 256))
    t = orc.pack(prob)
    rng = np.random.default_rng(13)
    y = bf16_bits(rng.standard_normal((M, 2 * I + 64)).astype(np.float32) * 3)
    act, a, asg, rs = orc.silu_mul_rotate_quant(y, prob.cs, t["rec"])
    expect = np.array([[orc.silu_mul(int(y[m, k]), int(y[m, I + k])) for k in range(I)] for m in range(M)],
                      dtype=np.uint16)
    assert np.array_equal(act, expect)
    a2, asg2, rs2 = orc.rotate_quant(act, prob.cs, t["rec"])
    assert np.array_equal(a, a2) and np.array_equal(asg, asg2) and np.array_equal(rs, rs2)


# ---------------------------------------------------------------- per-token scales
# Page: same log, "PER-TOKEN PREFILL (v3, BUILT)": pass A rotates into a bf16
# scratch with group amaxes, pass C takes As = max_g asg, encodes and forms
# plain row-sums, and the PTOK GEMM applies As in the epilogue (reading R18).
def test_tokquant_steps_match_independent_pieces(orc):
    M, K, P = 5, 640, 2
    prob = pqgen.make_problem(M, K, 256, P=P, seed=14, pb=(128, 256))
    t = orc.pack(prob)
    xr, a, As, rs = orc.rotate_tokquant(prob.x, prob.cs, t["rec"])
    # the rotation is the per-group prologue's (pinned on its own)
    _, _, _, v = orc.rotate_quant(prob.x, prob.cs, t["rec"], want_v=True)
    assert np.array_equal(xr, bf16_bits(v))
    xrf = bf16_to_f32(xr)
    G = K // 128
    amax = np.abs(xrf.reshape(P, M, G, 128)).max(axis=3)
    asg = (amax * np.float32(np.float32(1.0) / np.float32(448.0))).astype(np.float32)
    assert np.array_equal(As, asg.max(axis=2))
    # codes: the pinned encoder on fl32(xr / As); row-sums: exact sums of the decoded codes
    q = (xrf / As[:, :, None]).astype(np.float32)
    enc = np.array([orc.e4m3_encode(float(v)) for v in q.ravel()], dtype=np.uint8).reshape(q.shape)
    assert np.array_equal(a, enc)
    dec = orc.e4m3_decode_table()[a.astype(np.int64)]
    exact = dec.reshape(P, M, G, 128).sum(axis=3)
    assert np.array_equal(rs, np.transpose(exact, (0, 2, 1)).astype(np.float32))


def test_ptok_gemm_is_the_group_gemm_with_one_scale(orc):
    # with asg[g] = As for every group the per-group GEMM (pinned) is the same
    # sum; only the fp64 association differs
    M, K, N, P = 4, 512, 384, 3
    prob = pqgen.make_problem(M, K, N, P=P, seed=15, pb=(128, 256))
    t = orc.pack(prob)
    _, a, As, rs = orc.rotate_tokquant(prob.x, prob.cs, t["rec"])
    G = K // 128
    asg = np.repeat(As[:, None, :], G, axis=1).astype(np.float32)
    y1 = orc.gemm_ptok_f64(a, As, rs, t["codes"], t["sz"], 128, 256)
    y2 = orc.gemm_f64(a, asg, rs, t["codes"], t["sz"], 128, 256)
    assert np.allclose(y1, y2, rtol=1e-12, atol=1e-12 * np.abs(y2).max())
    ms = np.array([0, 3, 1], np.int32)
    ns = np.array([5, 200, 383], np.int32)
    ys = orc.gemm_ptok_f64_sampled(ms, ns, a, As, rs, t["codes"], t["sz"], 128, 256)
    assert np.array_equal(ys, y1[ms, ns])
