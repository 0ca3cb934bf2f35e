"""GPU parity gates: the CUDA path through the C ABI against the CPU oracle.

* prologue (codes, per-group scales, row-sums): byte-equal on every workload,
  ragged M, three partitions, subnormal-heavy inputs;
* device e4m3 encoder: equal to the oracle's encoder on all 2^32 fp32 patterns;
* GEMM (CUDA-core decode kernel and tcgen05 kernel): norm-wise relative error
  <= 2e-3 against the fp64 oracle (the bf16 output floor; the engineering log
  reports 1.65-1.71e-3 for its kernels), plus an elementwise bound, on full
  small problems and on sampled outputs at the full workload sizes;
* metamorphic cases: merged P=3 == three sliced launches (bit-identical),
  all-eight codes with zero point 8 give 0 to within fp32 rounding, rows are
  independent,
  rows past M and columns past N are never written.

Source: "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log", "Gates passed"
(prologue bit-exact vs CPU, GEMM at the bf16 floor on all shapes incl.
3-partition QKV and subnormal-heavy codes, rows past M untouched) and
"Traps hit" ("clear every output between variants": outputs here are
pre-filled with a canary).
"""
import numpy as np
import pytest

import pqgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CANARY = 0xA5


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


class Problem:
    """A generated layer: device tables from the product packer, host tables
    from the oracle's independent packer (checked byte-equal)."""

    def __init__(self, pq, orc, prob, check_pack=True):
        self.prob = prob
        self.rec, self.sz, self.w = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales,
                                               prob.pairs, prob.theta)
        self.t = orc.pack(prob)
        if check_pack:
            assert np.array_equal(self.rec, self.t["rec_kernel"])
            assert np.array_equal(self.sz, self.t["sz_kernel"])
            assert np.array_equal(self.w, self.t["w"])
        self.rec_d = torch.from_numpy(self.rec).cuda()
        self.sz_d = dev_u16(self.sz)
        self.w_d = torch.from_numpy(self.w).cuda()
        self.cs_d = dev_u16(prob.cs)
        self.x_d = dev_u16(prob.x).view(torch.bfloat16)


def canary_outputs(P, M, K, G, pad=64):
    """Outputs inside larger canary-filled buffers (views keep 16-byte alignment)."""
    a_buf = torch.full((P * M * K + 2 * pad,), CANARY, dtype=torch.uint8, device="cuda")
    s_buf = torch.full((P * G * M + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    r_buf = torch.full((P * G * M + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    a = a_buf[pad:pad + P * M * K].view(P, M, K)
    asg = s_buf[pad:pad + P * G * M].view(P, G, M)
    rs = r_buf[pad:pad + P * G * M].view(P, G, M)
    return (a_buf, s_buf, r_buf), (a, asg, rs), pad


def check_guards(bufs, pad):
    a_buf, s_buf, r_buf = [b.cpu() for b in bufs]
    assert bool((a_buf[:pad] == CANARY).all()) and bool((a_buf[-pad:] == CANARY).all())
    for b in (s_buf, r_buf):
        assert bool(torch.isnan(b[:pad]).all()) and bool(torch.isnan(b[-pad:]).all())


# ---------------------------------------------------------------- encoder
def test_e4m3_device_encoder_all_2_32(pq, orc):
    chunk = 1 << 28
    for lo in range(0, 1 << 32, chunk):
        bits = torch.arange(lo, lo + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        got = pq.pq_e4m3_encode(bits.view(torch.float32)).cpu().numpy()
        want = orc.e4m3_encode_range(lo, lo + chunk)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, "pattern 0x%08x: gpu %02x oracle %02x" % (
            lo + bad[0], got[bad[0]], want[bad[0]])
        del bits


# ---------------------------------------------------------------- prologue
PROLOGUE_CASES = [
    ("tiny", dict()),
    ("decode", dict(M=1)),
    ("decode", dict(M=4)),
    ("decode", dict(M=16)),
    ("prefill", dict()),
    ("prefill", dict(x_sigma=1e-4)),                          # literal N(0, 1e-4) variant
    ("prefill", dict(M=333, x_mode="sparse", theta_range=1e-4)),   # subnormal-heavy codes
    ("down", dict()),
    ("qkv", dict()),
    ("qkv", dict(M=33)),
    ("qkv", dict(M=2)),                   # three partitions in the decode-band kernel
    ("decode", dict(M=5)),
    ("prefill", dict(M=17)),              # first size of the many-token kernel
]


@pytest.mark.parametrize("name,over", PROLOGUE_CASES,
                         ids=["%s-%s" % (n, "-".join("%s%s" % kv for kv in o.items()))
                              for n, o in PROLOGUE_CASES])
def test_prologue_bit_exact(pq, orc, name, over):
    c = dict(pqgen.CONFIGS[name])
    c.update(over)
    c["N"] = 128                                   # the prologue does not depend on N
    c["pb"] = {1: (128, 128), 3: None}[c["P"]]
    if c["P"] == 3:
        c["N"] = 384
        c["pb"] = (128, 256)
    prob = pqgen.make_problem(**c)
    P, M, K, G = prob.P, prob.M, prob.K, prob.G
    rec = orc.records(prob.pairs, prob.theta)
    rec_p, _, _ = pq.pq_pack(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta)
    assert np.array_equal(orc.chain_records(rec), rec_p)
    bufs, (a, asg, rs), pad = canary_outputs(P, M, K, G)
    pq.pq_rotate_quant(dev_u16(prob.x).view(torch.bfloat16), torch.from_numpy(orc.chain_records(rec)).cuda(),
                       dev_u16(prob.cs), a=a, asg=asg, rs=rs)
    torch.cuda.synchronize()
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, rec)
    a_g = a.cpu().numpy()
    assert np.array_equal(a_g, a_o), "codes differ at %s" % (np.argwhere(a_g != a_o)[:3].tolist(),)
    assert np.array_equal(asg.cpu().numpy().view(np.uint32), asg_o.view(np.uint32))
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), rs_o.view(np.uint32))
    check_guards(bufs, pad)
    if over.get("x_mode") == "sparse":
        sub = ((a_o & 0x78) == 0) & ((a_o & 7) != 0)
        assert sub.mean() > 0.5


def test_prologue_tiny_and_huge_scales(pq, orc):
    """Groups whose scale falls below 2^-60 (the kernels then divide with the
    IEEE divide) or sits near it, and huge values, in both quantisers (the
    many-token prologue and the per-token pass C): bit-exact either way."""
    M, K = 40, 512
    prob = pqgen.make_problem(M, K, 128, seed=77)
    xf = (prob.x.astype(np.uint32) << 16).view(np.float32).copy()
    for r, f in zip(range(0, M, 4), (1e-16, 3e-17, 1e-18, 1e-22, 1e-30, 1e-36, 1e30, 4e35, 1e-17, 2e-17)):
        xf[r] *= np.float32(f)
    x = pqgen.to_bf16_bits(xf)
    rec = orc.records(prob.pairs, prob.theta)
    xd, rd, cd = dev_u16(x).view(torch.bfloat16), torch.from_numpy(orc.chain_records(rec)).cuda(), dev_u16(prob.cs)
    a, asg, rs = pq.pq_rotate_quant(xd, rd, cd)
    _, a2, As, rs2 = pq.pq_rotate_tokquant(xd, rd, cd)
    torch.cuda.synchronize()
    a_o, asg_o, rs_o = orc.rotate_quant(x, prob.cs, rec)
    _, a2_o, As_o, rs2_o = orc.rotate_tokquant(x, prob.cs, rec)
    assert (asg_o[asg_o > 0] < 2.0 ** -60).any() and (asg_o >= 2.0 ** -60).any()
    assert np.array_equal(a.cpu().numpy(), a_o) and np.array_equal(rs.cpu().numpy(), rs_o)
    assert np.array_equal(asg.cpu().numpy(), asg_o)
    assert np.array_equal(a2.cpu().numpy(), a2_o) and np.array_equal(rs2.cpu().numpy(), rs2_o)
    assert np.array_equal(As.cpu().numpy(), As_o)


def test_prologue_strided_x(pq, orc):
    """ldx > K: only the first K columns of each row are read."""
    prob = pqgen.make_problem(37, 384, 128, seed=21)
    xw = np.full((37, 384 + 64), 0x7FC0, dtype=np.uint16)     # NaN padding must never be read
    xw[:, :384] = prob.x
    rec = orc.records(prob.pairs, prob.theta)
    a, asg, rs = pq.pq_rotate_quant(dev_u16(xw).view(torch.bfloat16), torch.from_numpy(orc.chain_records(rec)).cuda(),
                                    dev_u16(prob.cs))
    a_o, asg_o, rs_o = orc.rotate_quant(xw, prob.cs, rec)
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(asg.cpu().numpy(), asg_o) and np.array_equal(rs.cpu().numpy(), rs_o)


# ---------------------------------------------------------------- fused producer
def producer_inputs(M, K, ldx, seed):
    """Residual rows and a Gemma weight for the fused producer (bf16 bits)."""
    rng = np.random.default_rng(seed + 1000)
    r = rng.standard_normal((M, ldx)).astype(np.float32) * np.float32(0.7)
    res = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w = rng.standard_normal(K).astype(np.float32) * np.float32(0.2)
    gamma = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return res, gamma


PRODUCER_CASES = [  # M, K, P, ldx pad
    (1, 5120, 1, 0), (2, 1024, 3, 0), (3, 896, 2, 64), (4, 256, 1, 0), (16, 5120, 1, 0),
    (17, 640, 3, 0), (100, 1152, 1, 64), (7, 16384, 1, 0),
]


@pytest.mark.parametrize("M,K,P,pad", PRODUCER_CASES)
def test_add_rms_rotate_quant_bit_exact(pq, orc, M, K, P, pad):
    N = 384 if P == 3 else 256
    pb = (128, 256) if P == 3 else ((128, 256) if P == 2 else None)
    prob = pqgen.make_problem(M, K, N, P=P, seed=M + K + P, pb=pb)
    ldx = K + pad
    xw = np.full((M, ldx), 0x7FC0, dtype=np.uint16)        # NaN padding must never be read
    xw[:, :K] = prob.x
    res, gamma = producer_inputs(M, K, ldx, M * 7 + K)
    res[:, K:] = 0x7FC0
    rec = orc.records(prob.pairs, prob.theta)
    G = K // 128
    bufs, (a, asg, rs), gpad = canary_outputs(P, M, K, G)
    ro, h, a, asg, rs = pq.pq_add_rms_rotate_quant(
        dev_u16(xw).view(torch.bfloat16), dev_u16(res).view(torch.bfloat16), dev_u16(gamma).view(torch.bfloat16),
        1e-6, torch.from_numpy(orc.chain_records(rec)).cuda(), dev_u16(prob.cs), a=a, asg=asg, rs=rs)
    torch.cuda.synchronize()
    ro_o, h_o, a_o, asg_o, rs_o = orc.add_rms_rotate_quant(xw, res, gamma, 1e-6, prob.cs, rec)
    u16 = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(u16(ro), ro_o), "residual differs"
    assert np.array_equal(u16(h), h_o), "normed rows differ at %s" % (np.argwhere(u16(h) != h_o)[:3].tolist(),)
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(asg.cpu().numpy().view(np.uint32), asg_o.view(np.uint32))
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), rs_o.view(np.uint32))
    check_guards(bufs, gpad)


def test_add_rms_rotate_quant_feeds_the_gemm(pq, orc):
    """The producer's outputs are a valid pq_gemm input: the layer matches the
    oracle's GEMM of the oracle's producer outputs."""
    M, K, N = 1, 5120, 1024
    prob = pqgen.make_problem(M, K, N, seed=77)
    L = Problem(pq, orc, prob)
    res, gamma = producer_inputs(M, K, K, 77)
    _, _, a, asg, rs = pq.pq_add_rms_rotate_quant(
        L.x_d, dev_u16(res).view(torch.bfloat16), dev_u16(gamma).view(torch.bfloat16), 1e-6, L.rec_d, L.cs_d)
    y = pq.pq_gemm(a, asg, rs, L.w_d, L.sz_d)
    torch.cuda.synchronize()
    _, _, a_o, asg_o, rs_o = orc.add_rms_rotate_quant(prob.x, res, gamma, 1e-6, prob.cs, L.t["rec"])
    y64 = orc.gemm_f64(a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], N, N)
    assert_close(y.float().cpu().numpy(), y64, "producer -> pq_gemm")


SILU_CASES = [  # M, I, P, ldy pad
    (1, 8704, 1, 0), (2, 384, 3, 64), (5, 1024, 2, 0), (16, 256, 1, 0), (17, 640, 1, 128), (300, 1152, 3, 0),
]


@pytest.mark.parametrize("M,I,P,pad", SILU_CASES)
def test_silu_mul_rotate_quant_bit_exact(pq, orc, M, I, P, pad):
    N = 384 if P == 3 else 256
    pb = (128, 256) if P in (2, 3) else None
    prob = pqgen.make_problem(M, I, N, P=P, seed=M + I + 3 * P, pb=pb)
    rng = np.random.default_rng(M * 5 + I)
    ldy = 2 * I + pad
    yv = rng.standard_normal((M, ldy)).astype(np.float32) * np.float32(3.0)
    y = torch.from_numpy(yv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    y[:, 2 * I:] = 0x7FC0                                    # padding must never be read
    rec = orc.records(prob.pairs, prob.theta)
    G = I // 128
    bufs, (a, asg, rs), gpad = canary_outputs(P, M, I, G)
    act, a, asg, rs = pq.pq_silu_mul_rotate_quant(dev_u16(y).view(torch.bfloat16), torch.from_numpy(orc.chain_records(rec)).cuda(),
                                                  dev_u16(prob.cs), a=a, asg=asg, rs=rs)
    torch.cuda.synchronize()
    act_o, a_o, asg_o, rs_o = orc.silu_mul_rotate_quant(y, prob.cs, rec)
    got = act.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, act_o), "act differs at %s" % (np.argwhere(got != act_o)[:3].tolist(),)
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(asg.cpu().numpy().view(np.uint32), asg_o.view(np.uint32))
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), rs_o.view(np.uint32))
    check_guards(bufs, gpad)


def test_mlp_chain_matches_oracle(pq, orc):
    """norm producer -> gate_up GEMM -> silu-mul producer -> down GEMM at
    decode, against the oracle's chain (each GEMM to its 2e-3 gate; the
    producers' inputs are the GPU's own GEMM outputs, so the comparison of
    the down projection is against the oracle run on those)."""
    M, K, I = 2, 1024, 512
    up = pqgen.make_problem(M, K, 2 * I, seed=31)
    down = pqgen.make_problem(M, I, K, seed=32)
    Lu, Ld = Problem(pq, orc, up), Problem(pq, orc, down)
    res, gamma = producer_inputs(M, K, K, 31)
    _, _, a1, s1, r1 = pq.pq_add_rms_rotate_quant(Lu.x_d, dev_u16(res).view(torch.bfloat16),
                                                  dev_u16(gamma).view(torch.bfloat16), 1e-6, Lu.rec_d, Lu.cs_d)
    y1 = pq.pq_gemm(a1, s1, r1, Lu.w_d, Lu.sz_d)
    act, a2, s2, r2 = pq.pq_silu_mul_rotate_quant(y1, Ld.rec_d, Ld.cs_d)
    y2 = pq.pq_gemm(a2, s2, r2, Ld.w_d, Ld.sz_d)
    torch.cuda.synchronize()
    _, _, a1o, s1o, r1o = orc.add_rms_rotate_quant(up.x, res, gamma, 1e-6, up.cs, Lu.t["rec"])
    assert np.array_equal(a1.cpu().numpy(), a1o)
    y1_64 = orc.gemm_f64(a1o, s1o, r1o, Lu.t["codes"], Lu.t["sz"], 2 * I, 2 * I)
    assert_close(y1.float().cpu().numpy(), y1_64, "gate_up")
    y1_bits = y1.view(torch.int16).cpu().numpy().view(np.uint16)
    act_o, a2o, s2o, r2o = orc.silu_mul_rotate_quant(y1_bits, down.cs, Ld.t["rec"])
    assert np.array_equal(act.view(torch.int16).cpu().numpy().view(np.uint16), act_o)
    y2_64 = orc.gemm_f64(a2o, s2o, r2o, Ld.t["codes"], Ld.t["sz"], K, K)
    assert_close(y2.float().cpu().numpy(), y2_64, "down")


# ---------------------------------------------------------------- GEMM helpers
def gemm_paths(pq, M):
    paths = [("tc", pq.pq_gemm_tc)]
    if M <= pq.pq_gemm_skinny_max_m():
        paths.append(("skinny", pq.pq_gemm_skinny))
        paths.append(("tcn", pq.pq_gemm_tcn))
    return paths


def run_gemm(fn, a, asg, rs, L, pb1, pb2, M, N, ldy=None, fill=float("nan")):
    ldy = ldy or N
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ybuf = torch.full((M + 3, ldy), fill, dtype=torch.bfloat16, device="cuda")
    y = ybuf[:M]
    # a strided y view: pass the storage with its leading dimension
    import ctypes as C
    import w4a8_rotated_int4_gb300 as m
    lib = m.lib()
    name = {m.pq_gemm_tc: "pq_gemm_tc", m.pq_gemm_skinny: "pq_gemm_skinny",
            m.pq_gemm_tcn: "pq_gemm_tcn", m.pq_gemm_ptok: "pq_gemm_ptok"}[fn]
    P = a.shape[0]
    K = a.shape[2]
    st = getattr(lib, name)(C.c_void_p(a.data_ptr()), C.c_void_p(asg.data_ptr()),
                            C.c_void_p(rs.data_ptr()), M, N, K, P, pb1, pb2,
                            C.c_void_p(L.w_d.data_ptr()), C.c_void_p(L.sz_d.data_ptr()),
                            C.c_void_p(y.data_ptr()), ldy, C.c_void_p(status.data_ptr()),
                            C.c_void_p(torch.cuda.current_stream().cuda_stream))
    m._check(st, name)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %d" % int(status.item())
    yb = ybuf.float().cpu().numpy()
    # nothing outside [0, M) x [0, N) was written
    assert np.isnan(yb[M:]).all()
    if ldy > N:
        assert np.isnan(yb[:M, N:]).all()
    return yb[:M, :N]


def assert_close(y, y64, what):
    rel = float(np.linalg.norm(y - y64) / max(np.linalg.norm(y64), 1e-300))
    rms = float(np.sqrt(np.mean(y64 ** 2)))
    # elementwise: bf16 rounding (<= 2^-8 relative) plus fp32 accumulation noise
    bound = 2.0 ** -8 * np.abs(y64) * 1.001 + 1e-3 * rms
    worst = float(np.max(np.abs(y - y64) - bound))
    assert np.isfinite(y).all(), what + ": non-finite output"
    assert rel <= 2e-3, "%s: rel err %.3e" % (what, rel)
    assert worst <= 0, "%s: elementwise excess %.3e (rms %.3e)" % (what, worst, rms)
    return rel


# ---------------------------------------------------------------- GEMM, full oracle
GEMM_SMALL = [  # M, K, N, P, pb
    (4, 256, 128, 1, None), (1, 1024, 256, 1, None), (3, 640, 384, 1, None),
    (16, 1152, 512, 1, None), (7, 512, 384, 3, (128, 256)), (12, 384, 512, 2, (256, 512)),
    (129, 512, 256, 1, None), (200, 896, 384, 3, (128, 256)), (256, 1024, 512, 1, None),
    (33, 1152, 256, 1, None), (18, 8704, 128, 1, None),
    # several octets per CTA of the decode kernel and partition switches
    # inside a CTA's run; M = 2 runs its three-group CTAs (unequal group loads)
    (1, 1152, 8448, 3, (2048, 4992)), (3, 640, 6016, 2, (2944, 6016)), (6, 384, 4096, 1, None),
    (2, 5120, 8448, 2, (4096, 8448)),
]


@pytest.mark.parametrize("M,K,N,P,pb", GEMM_SMALL)
def test_gemm_full_vs_oracle(pq, orc, M, K, N, P, pb):
    prob = pqgen.make_problem(M, K, N, P=P, pb=pb, seed=M * 7 + K + N)
    L = Problem(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    y64 = orc.gemm_f64(a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1, prob.pb2)
    for name, fn in gemm_paths(pq, M):
        y = run_gemm(fn, a, asg, rs, L, prob.pb1, prob.pb2, M, N, ldy=N + 64)
        assert_close(y, y64, "%s M=%d K=%d N=%d P=%d" % (name, M, K, N, P))


@pytest.mark.parametrize("M", [1, 3])
def test_gemm_dispatch_beyond_skinny_k(pq, orc, M):
    """pq_gemm at M <= 16 with K above the CUDA-core kernel's limit (16384):
    the dispatcher must hand it to the narrow tensor-core kernel, which has no
    K limit, and the result must stay within the bf16 floor.  The CUDA-core
    kernel itself refuses that K."""
    K, N = 17408, 256
    prob = pqgen.make_problem(M, K, N, seed=K + M)
    L = Problem(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    y64 = orc.gemm_f64(a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1, prob.pb2)
    y = pq.pq_gemm(a, asg, rs, L.w_d, L.sz_d)
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), y64, "pq_gemm M=%d K=%d" % (M, K))
    with pytest.raises(pq.PQError) as e:
        pq.pq_gemm_skinny(a, asg, rs, L.w_d, L.sz_d)
    assert e.value.status == 2
    del e      # the traceback holds this frame: no cycle may keep its CUDA objects alive


@pytest.mark.parametrize("subnormal", [False, True])
def test_gemm_random_codes(pq, orc, subnormal):
    """Codes drawn uniformly from all 254 finite e4m3 codes (incl. 0x80 and
    subnormals), or only from the 16 zero/subnormal codes."""
    M, K, N, P = 24, 1024, 384, 2
    prob = pqgen.make_problem(M, K, N, P=P, pb=(128, 384), seed=5)
    L = Problem(pq, orc, prob)
    a_o = pqgen.random_codes(P, M, K, seed=6, subnormal_only=subnormal)
    asg_o = pqgen.random_scales(P, K // 128, M, seed=7)
    dec = orc.e4m3_decode_table()[a_o]
    rs_o = dec.reshape(P, M, K // 128, 128).sum(axis=3).transpose(0, 2, 1).astype(np.float32)
    y64 = orc.gemm_f64(a_o, asg_o, np.ascontiguousarray(rs_o), L.t["codes"], L.t["sz"], 128, 384)
    a = torch.from_numpy(a_o).cuda()
    asg = torch.from_numpy(asg_o).cuda()
    rs = torch.from_numpy(np.ascontiguousarray(rs_o)).cuda()
    for name, fn in gemm_paths(pq, M):
        assert_close(run_gemm(fn, a, asg, rs, L, 128, 384, M, N), y64, name)


def test_gemm_zero_point_eight_gives_zero(pq, orc):
    """All codes 8 with zero point 8: every weight is 0, so y = 0.  The kernels
    form D' = sum a*c and subtract 8*rs, so the zero is reached to within the
    fp32 rounding of the two sums: |y| <= 2^-21 * sum_g asg * 8 sc |rs|."""
    M, K, N = 9, 512, 256
    prob = pqgen.make_problem(M, K, N, seed=8)
    eights = np.int32(np.uint32(0x88888888).view(np.int32))
    prob["qweight"] = np.full_like(prob.qweight, eights)
    prob["qzeros"] = np.full_like(prob.qzeros, eights)
    L = Problem(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    sc = prob.scales.view(np.float16).astype(np.float64)                       # [G, N]
    mag = np.einsum("gm,gn->mn", np.abs(asg[0].cpu().numpy().astype(np.float64) *
                                        rs[0].cpu().numpy()), 8 * sc)
    for name, fn in gemm_paths(pq, M):
        y = run_gemm(fn, a, asg, rs, L, N, N, M, N)
        assert np.all(np.abs(y) <= 2.0 ** -21 * mag), name
        # and a non-trivial weight moves it far away from zero
        assert float(np.max(mag)) > 1e-3


@pytest.mark.parametrize("M", [300, 3])
def test_gemm_zero_scale_groups(pq, orc, M):
    """A group whose scale is 0 (either sign) dequantizes to -zscale whatever
    its codes.  The packer never writes one with a nonzero zscale, so the SZ
    table is edited by hand here; every path must still match the oracle
    (the prefill kernel masks such codes and folds the zero point apart)."""
    K, N = 512, 256
    G = K // 128
    prob = pqgen.make_problem(M, K, N, seed=21 + M)
    L = Problem(pq, orc, prob)
    rng = np.random.default_rng(5)
    sz = L.t["sz"].copy()                                    # [G, N, 2] f16 bits
    pick = rng.random((G, N)) < 0.15
    zs = (rng.standard_normal((G, N)) * 0.02).astype(np.float16).view(np.uint16)
    sz[..., 0][pick] = np.where(rng.random(int(pick.sum())) < 0.5, 0x0000, 0x8000)
    sz[..., 1][pick] = zs[pick]
    L.sz_d = dev_u16(np.ascontiguousarray(sz.reshape(G, N // 8, 8, 2).transpose(1, 0, 2, 3)))
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    y64 = orc.gemm_f64(a.cpu().numpy(), asg.cpu().numpy(), rs.cpu().numpy(), L.t["codes"], sz, N, N)
    for name, fn in gemm_paths(pq, M):
        y = run_gemm(fn, a, asg, rs, L, N, N, M, N)
        assert_close(y, y64, "%s zero-scale groups M=%d" % (name, M))


@pytest.mark.parametrize("M,K,N", [(512, 256, 10240), (300, 384, 10240)])
def test_gemm_tc_split_last_round(pq, orc, M, K, N):
    """160 tiles on 152 CTAs: the last 8 tiles run as 16 half items (128 rows
    each; at M = 300 one half of each lies past M).  Every output of the
    per-group, per-token and int5 prefill kernels against the oracle."""
    prob = pqgen.make_problem(M, K, N, P=2, pb=(N // 2, N), seed=M + K)
    L = Problem(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    y64 = orc.gemm_f64(a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], N // 2, N)
    assert_close(run_gemm(pq.pq_gemm_tc, a, asg, rs, L, N // 2, N, M, N), y64, "tc split")
    _, a_t, As, rs_t = pq.pq_rotate_tokquant(L.x_d, L.rec_d, L.cs_d)
    _, a_to, As_o, rs_to = orc.rotate_tokquant(prob.x, prob.cs, L.t["rec"])
    y64t = orc.gemm_ptok_f64(a_to, As_o, rs_to, L.t["codes"], L.t["sz"], N // 2, N)
    assert_close(run_gemm(pq.pq_gemm_ptok, a_t, As, rs_t, L, N // 2, N, M, N), y64t, "ptok split")
    p5 = pqgen.make_problem(M, K, N, P=2, pb=(N // 2, N), seed=M + K, bits=5)
    L5 = Problem5(pq, orc, p5)
    y64_5 = orc.gemm5_f64(a_o, asg_o, rs_o, L5.t["codes"], L5.t["sz"], N // 2, N)
    assert_close(run_gemm5("pq_gemm5_tc", a, asg, rs, L5, N // 2, N, M, N), y64_5, "int5 split")


def test_gemm_merged_equals_sliced(pq, orc):
    """One P=3 launch == three P=1 launches on the column slices, bit for bit."""
    M, K, N = 40, 640, 512
    prob = pqgen.make_problem(M, K, N, P=3, pb=(256, 384), seed=9)
    L = Problem(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    for Mx in (M, 5):
        for name, fn in gemm_paths(pq, Mx):
            aa, ss, rr = a[:, :Mx].contiguous(), asg[:, :, :Mx].contiguous(), rs[:, :, :Mx].contiguous()
            y = run_gemm(fn, aa, ss, rr, L, 256, 384, Mx, N)
            for p, (lo, hi) in enumerate([(0, 256), (256, 384), (384, 512)]):
                Ls = type("S", (), {})()
                Ls.w_d = L.w_d[lo:hi].contiguous()
                Ls.sz_d = L.sz_d[lo // 8:hi // 8].contiguous()
                ys = run_gemm(fn, aa[p:p + 1].contiguous(), ss[p:p + 1].contiguous(),
                              rr[p:p + 1].contiguous(), Ls, hi - lo, hi - lo, Mx, hi - lo)
                assert np.array_equal(y[:, lo:hi], ys), (name, Mx, p)


def test_gemm_rows_independent(pq, orc):
    M, K, N = 150, 512, 256
    prob = pqgen.make_problem(M, K, N, seed=10)
    L = Problem(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    a2, asg2, rs2 = a.clone(), asg.clone(), rs.clone()
    g = torch.Generator(device="cpu").manual_seed(0)
    a2[:, 1::2] = torch.randint(0, 126, a2[:, 1::2].shape, generator=g).to(torch.uint8).cuda()
    asg2[:, :, 1::2] *= 3
    for Mx in (M, 16):
        for name, fn in gemm_paths(pq, Mx):
            y1 = run_gemm(fn, a[:, :Mx].contiguous(), asg[:, :, :Mx].contiguous(),
                          rs[:, :, :Mx].contiguous(), L, N, N, Mx, N)
            y2 = run_gemm(fn, a2[:, :Mx].contiguous(), asg2[:, :, :Mx].contiguous(),
                          rs2[:, :, :Mx].contiguous(), L, N, N, Mx, N)
            assert np.array_equal(y1[0::2], y2[0::2]), name


# ---------------------------------------------------------------- full workloads, sampled
FULL = [("decode", 1), ("decode", 4), ("decode", 16), ("prefill", None), ("down", None),
        ("qkv", None), ("tiny", None)]


def _samples(M, N, pb1, pb2, count, seed):
    r = np.random.default_rng(seed)
    ms = list(r.integers(0, M, count)) + [0, M - 1] * 4
    ns = list(r.integers(0, N, count)) + [0, N - 1, pb1 - 1, min(pb1, N - 1), pb2 - 1,
                                          min(pb2, N - 1), 127, min(128, N - 1)]
    return np.array(ms[:len(ns)]), np.array(ns)


@pytest.mark.parametrize("name,M", FULL, ids=["%s-%s" % f for f in FULL])
def test_full_workload_sampled(pq, orc, name, M):
    """At the benchmarked sizes and launch configuration: prologue bit-exact
    (full), GEMM on 3000 sampled outputs against the fp64 oracle."""
    prob = pqgen.config_problem(name, M=M)
    L = Problem(pq, orc, prob, check_pack=(name != "down"))
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    y = pq.pq_gemm(a, asg, rs, L.w_d, L.sz_d, prob.pb1, prob.pb2)
    torch.cuda.synchronize()
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(asg.cpu().numpy(), asg_o) and np.array_equal(rs.cpu().numpy(), rs_o)
    ms, ns = _samples(prob.M, prob.N, prob.pb1, prob.pb2, 3000, 11)
    y64 = orc.gemm_f64_sampled(ms, ns, a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1,
                               prob.pb2)
    yg = y.float().cpu().numpy()[ms, ns]
    assert_close(yg, y64, "%s M=%d" % (name, prob.M))
    if prob.M <= pq.pq_gemm_skinny_max_m():      # the other paths on the same inputs
        for tag, fn in (("tc", pq.pq_gemm_tc), ("skinny", pq.pq_gemm_skinny), ("tcn", pq.pq_gemm_tcn)):
            y2 = fn(a, asg, rs, L.w_d, L.sz_d, prob.pb1, prob.pb2)
            assert_close(y2.float().cpu().numpy()[ms, ns], y64, "%s %s M=%d" % (tag, name, prob.M))


# ---------------------------------------------------------------- per-token scales
TOKQUANT_CASES = [  # M, K, P, pb, zero rows, generator knobs
    (4, 256, 1, None, (), {}),
    (1, 5120, 1, None, (), dict(outlier_frac=0.01)),
    (5, 1152, 1, None, (2,), {}),
    (64, 384, 3, (128, 256), (), {}),
    (65, 640, 2, (256, 384), (0, 64), {}),
    (333, 1024, 1, None, (), dict(x_mode="sparse", theta_range=1e-4)),
    (2048, 5120, 1, None, (7,), {}),
    (512, 5120, 3, (6144, 7168), (), {}),
]


def tokquant_problem(M, K, P, pb, zero_rows, knobs, N=None, seed=None):
    N = N or (384 if P == 3 else 128 * P)
    if pb is not None and pb[1] >= N:
        N = pb[1] + 128 if P == 3 else pb[1]
    prob = pqgen.make_problem(M, K, N, P=P, pb=pb, seed=seed if seed is not None else M + K, **knobs)
    x = prob.x.copy()
    for r in zero_rows:
        x[r] = 0
    return prob, x


@pytest.mark.parametrize("M,K,P,pb,zero_rows,knobs", TOKQUANT_CASES,
                         ids=["M%d-K%d-P%d" % c[:3] for c in TOKQUANT_CASES])
def test_rotate_tokquant_bit_exact(pq, orc, M, K, P, pb, zero_rows, knobs):
    """Per-token prologue: the bf16 rotated rows, codes, token scales and
    plain row-sums bit-identical to the oracle; nothing outside them written."""
    prob, x = tokquant_problem(M, K, P, pb, zero_rows, knobs)
    G = K // 128
    rec = orc.records(prob.pairs, prob.theta)
    pad = 64
    xr_buf = torch.full((P * M * K + 2 * pad,), -1, dtype=torch.int16, device="cuda")
    as_buf = torch.full((P * M + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    bufs, (a, _, rs), _ = canary_outputs(P, M, K, G, pad)
    xr = xr_buf[pad:pad + P * M * K].view(P, M, K).view(torch.bfloat16)
    As = as_buf[pad:pad + P * M].view(P, M)
    pq.pq_rotate_tokquant(dev_u16(x).view(torch.bfloat16), torch.from_numpy(orc.chain_records(rec)).cuda(), dev_u16(prob.cs),
                          xr=xr, a=a, As=As, rs=rs)
    torch.cuda.synchronize()
    xr_o, a_o, As_o, rs_o = orc.rotate_tokquant(x, prob.cs, rec)
    xr_g = xr.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(xr_g, xr_o), "xr differs at %s" % (np.argwhere(xr_g != xr_o)[:3].tolist(),)
    a_g = a.cpu().numpy()
    assert np.array_equal(a_g, a_o), "codes differ at %s" % (np.argwhere(a_g != a_o)[:3].tolist(),)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_o.view(np.uint32))
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), rs_o.view(np.uint32))
    a_buf, r_buf = bufs[0].cpu(), bufs[2].cpu()
    assert bool((a_buf[:pad] == CANARY).all()) and bool((a_buf[-pad:] == CANARY).all())
    assert bool(torch.isnan(r_buf[:pad]).all()) and bool(torch.isnan(r_buf[-pad:]).all())
    xb, ab = xr_buf.cpu(), as_buf.cpu()
    assert bool((xb[:pad] == -1).all()) and bool((xb[-pad:] == -1).all())
    assert bool(torch.isnan(ab[:pad]).all()) and bool(torch.isnan(ab[-pad:]).all())
    for r in zero_rows:
        assert (As_o[:, r] == 0).all() and (a_o[:, r] == 0).all()
    if knobs.get("x_mode") == "sparse":
        sub = ((a_o & 0x78) == 0) & ((a_o & 7) != 0)
        assert sub.mean() > 0.3


def test_rotate_tokquant_long_rows(pq, orc):
    """928 groups per row (K = 118784): the token scale spans more groups than
    a CTA of pass C has threads."""
    M, K = 3, 118784
    prob = pqgen.make_problem(M, K, 128, seed=K + M)
    rec = orc.records(prob.pairs, prob.theta)
    xr, a, As, rs = pq.pq_rotate_tokquant(dev_u16(prob.x).view(torch.bfloat16), torch.from_numpy(orc.chain_records(rec)).cuda(),
                                          dev_u16(prob.cs))
    torch.cuda.synchronize()
    xr_o, a_o, As_o, rs_o = orc.rotate_tokquant(prob.x, prob.cs, rec)
    assert np.array_equal(xr.view(torch.int16).cpu().numpy().view(np.uint16), xr_o)
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_o.view(np.uint32))
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), rs_o.view(np.uint32))


PTOK_GEMM = [  # M, K, N, P, pb
    (1, 1024, 256, 1, None), (7, 512, 384, 3, (128, 256)), (129, 512, 256, 1, None),
    (200, 896, 384, 3, (128, 256)), (256, 1024, 512, 1, None), (300, 1152, 384, 2, (256, 384)),
    (33, 8704, 128, 1, None),
]


@pytest.mark.parametrize("M,K,N,P,pb", PTOK_GEMM)
def test_gemm_ptok_vs_oracle(pq, orc, M, K, N, P, pb):
    prob = pqgen.make_problem(M, K, N, P=P, pb=pb, seed=M * 5 + K + N)
    x = prob.x.copy()
    x[M // 2] = 0                                  # a token with As = 0
    L = Problem(pq, orc, prob)
    _, a, As, rs = pq.pq_rotate_tokquant(dev_u16(x).view(torch.bfloat16), L.rec_d, L.cs_d)
    _, a_o, As_o, rs_o = orc.rotate_tokquant(x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    y64 = orc.gemm_ptok_f64(a_o, As_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1, prob.pb2)
    y = run_gemm(pq.pq_gemm_ptok, a, As, rs, L, prob.pb1, prob.pb2, M, N, ldy=N + 64)
    assert (y[M // 2] == 0).all()
    assert_close(y, y64, "ptok M=%d K=%d N=%d P=%d" % (M, K, N, P))


@pytest.mark.parametrize("name", ["prefill", "down", "qkv"])
def test_ptok_full_workload_sampled(pq, orc, name):
    """At the benchmarked sizes: the per-token prologue bit-exact (full), the
    per-token GEMM on 3000 sampled outputs against the fp64 oracle."""
    prob = pqgen.config_problem(name)
    L = Problem(pq, orc, prob, check_pack=(name != "down"))
    xr, a, As, rs = pq.pq_rotate_tokquant(L.x_d, L.rec_d, L.cs_d)
    y = pq.pq_gemm_ptok(a, As, rs, L.w_d, L.sz_d, prob.pb1, prob.pb2)
    torch.cuda.synchronize()
    xr_o, a_o, As_o, rs_o = orc.rotate_tokquant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(xr.view(torch.int16).cpu().numpy().view(np.uint16), xr_o)
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(As.cpu().numpy(), As_o) and np.array_equal(rs.cpu().numpy(), rs_o)
    ms, ns = _samples(prob.M, prob.N, prob.pb1, prob.pb2, 3000, 13)
    y64 = orc.gemm_ptok_f64_sampled(ms, ns, a_o, As_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1, prob.pb2)
    assert_close(y.float().cpu().numpy()[ms, ns], y64, "ptok %s M=%d" % (name, prob.M))


# ---------------------------------------------------------------- int5 weights
class Problem5:
    """A generated int5 layer: device tables from pq_pack5, host tables from
    the oracle's packer (checked byte-equal)."""

    def __init__(self, pq, orc, prob, check_pack=True):
        self.prob = prob
        self.rec, self.sz, self.w, self.whi = pq.pq_pack5(prob.qweight, prob.qzeros, prob.qweight_hi,
                                                          prob.qzeros_hi, prob.scales, prob.pairs, prob.theta)
        self.t = orc.pack5(prob)
        if check_pack:
            assert np.array_equal(self.rec, self.t["rec_kernel"])
            assert np.array_equal(self.sz, self.t["sz_kernel"])
            assert np.array_equal(self.w, self.t["w"])
            assert np.array_equal(self.whi, self.t["whi"])
        self.rec_d = torch.from_numpy(self.rec).cuda()
        self.sz_d = dev_u16(self.sz)
        self.w_d = torch.from_numpy(self.w).cuda()
        self.whi_d = torch.from_numpy(self.whi).cuda()
        self.cs_d = dev_u16(prob.cs)
        self.x_d = dev_u16(prob.x).view(torch.bfloat16)


def run_gemm5(name, a, asg, rs, L, pb1, pb2, M, N, ldy=None):
    """An int5 GEMM path (pq_gemm5_tc, _tcn or _skinny) through the C ABI into a
    NaN-filled strided y."""
    import ctypes as C
    import w4a8_rotated_int4_gb300 as m
    ldy = ldy or N
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ybuf = torch.full((M + 3, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    P, K = a.shape[0], a.shape[2]
    st = getattr(m.lib(), name)(C.c_void_p(a.data_ptr()), C.c_void_p(asg.data_ptr()), C.c_void_p(rs.data_ptr()),
                                M, N, K, P, pb1, pb2, C.c_void_p(L.w_d.data_ptr()), C.c_void_p(L.whi_d.data_ptr()),
                                C.c_void_p(L.sz_d.data_ptr()), C.c_void_p(ybuf.data_ptr()), ldy,
                                C.c_void_p(status.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    m._check(st, name)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %d" % int(status.item())
    yb = ybuf.float().cpu().numpy()
    assert np.isnan(yb[M:]).all()
    if ldy > N:
        assert np.isnan(yb[:M, N:]).all()
    return yb[:M, :N]


def gemm5_paths(M):
    return ["pq_gemm5_tc"] + (["pq_gemm5_tcn", "pq_gemm5_skinny"] if M <= 16 else [])


INT5_SMALL = [  # M, K, N, P, pb
    (1, 1024, 256, 1, None), (4, 256, 128, 1, None), (16, 1152, 512, 1, None), (7, 512, 384, 3, (128, 256)),
    (12, 384, 512, 2, (256, 512)), (129, 512, 256, 1, None), (200, 896, 384, 3, (128, 256)),
    (256, 1024, 512, 1, None), (33, 8704, 128, 1, None), (3, 5120, 1024, 1, None),
]


@pytest.mark.parametrize("M,K,N,P,pb", INT5_SMALL)
def test_gemm5_vs_oracle(pq, orc, M, K, N, P, pb):
    prob = pqgen.make_problem(M, K, N, P=P, pb=pb, seed=M * 3 + K + N, bits=5)
    L = Problem5(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    y64 = orc.gemm5_f64(a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1, prob.pb2)
    for name in gemm5_paths(M):
        y = run_gemm5(name, a, asg, rs, L, prob.pb1, prob.pb2, M, N, ldy=N + 64)
        assert_close(y, y64, "%s M=%d K=%d N=%d P=%d" % (name, M, K, N, P))
    y = pq.pq_gemm5(a, asg, rs, L.w_d, L.whi_d, L.sz_d, prob.pb1, prob.pb2)
    assert_close(y.float().cpu().numpy(), y64, "pq_gemm5 M=%d" % M)


@pytest.mark.parametrize("M", [300, 3])
def test_gemm5_zero_scale_groups(pq, orc, M):
    """int5 columns whose scale is 0 dequantize to -zscale (set by hand here)."""
    K, N = 512, 256
    G = K // 128
    prob = pqgen.make_problem(M, K, N, seed=41 + M, bits=5)
    L = Problem5(pq, orc, prob)
    rng = np.random.default_rng(7)
    sz = L.t["sz"].copy()
    pick = rng.random((G, N)) < 0.15
    zs = (rng.standard_normal((G, N)) * 0.02).astype(np.float16).view(np.uint16)
    sz[..., 0][pick] = np.where(rng.random(int(pick.sum())) < 0.5, 0x0000, 0x8000)
    sz[..., 1][pick] = zs[pick]
    L.sz_d = dev_u16(np.ascontiguousarray(sz.reshape(G, N // 8, 8, 2).transpose(1, 0, 2, 3)))
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    y64 = orc.gemm5_f64(a.cpu().numpy(), asg.cpu().numpy(), rs.cpu().numpy(), L.t["codes"], sz, N, N)
    for name in gemm5_paths(M):
        assert_close(run_gemm5(name, a, asg, rs, L, N, N, M, N), y64, "%s zero-scale M=%d" % (name, M))


def test_gemm5_all_fifth_bits_equal_int4(pq, orc):
    """With every fifth bit set, int5 codes and zero points are the int4 ones
    plus 16: the same layer.  The two SZ tables round zscale to f16 from
    different products (sc * zp vs sc * (zp - 8)), so the int5 and int4
    oracles agree to that rounding only; the GPU is held to the int5 one."""
    M, K, N = 16, 512, 256
    prob = pqgen.make_problem(M, K, N, seed=3)
    p5 = pqgen.Problem(dict(prob))
    p5["qweight_hi"] = np.full((K, N // 32), -1, dtype=np.int32)
    p5["qzeros_hi"] = np.full((K // 128, N // 32), -1, dtype=np.int32)
    L4, L5 = Problem(pq, orc, prob), Problem5(pq, orc, p5)
    assert np.array_equal(L4.w, L5.w) and (L5.whi == 0xFF).all()
    a, asg, rs = pq.pq_rotate_quant(L4.x_d, L4.rec_d, L4.cs_d)
    a_h, s_h, r_h = a.cpu().numpy(), asg.cpu().numpy(), rs.cpu().numpy()
    y4 = orc.gemm_f64(a_h, s_h, r_h, L4.t["codes"], L4.t["sz"], N, N)
    y64 = orc.gemm5_f64(a_h, s_h, r_h, L5.t["codes"], L5.t["sz"], N, N)
    assert orc.rel_err(y64, y4) < 1e-3
    for name in ("pq_gemm5_tc", "pq_gemm5_tcn", "pq_gemm5_skinny"):
        assert_close(run_gemm5(name, a, asg, rs, L5, N, N, M, N), y64, name)


@pytest.mark.parametrize("name,M", [("decode", 1), ("decode", 16), ("prefill", None), ("qkv", None)])
def test_gemm5_full_workload_sampled(pq, orc, name, M):
    """int5 weights at the benchmarked sizes: 3000 sampled outputs against the
    fp64 oracle (packer checked byte-equal)."""
    prob = pqgen.config_problem(name, M=M, bits=5)
    L = Problem5(pq, orc, prob)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    y = pq.pq_gemm5(a, asg, rs, L.w_d, L.whi_d, L.sz_d, prob.pb1, prob.pb2)
    torch.cuda.synchronize()
    a_o, asg_o, rs_o = orc.rotate_quant(prob.x, prob.cs, L.t["rec"])
    assert np.array_equal(a.cpu().numpy(), a_o)
    ms, ns = _samples(prob.M, prob.N, prob.pb1, prob.pb2, 3000, 17)
    y64 = orc.gemm5_f64_sampled(ms, ns, a_o, asg_o, rs_o, L.t["codes"], L.t["sz"], prob.pb1, prob.pb2)
    assert_close(y.float().cpu().numpy()[ms, ns], y64, "int5 %s M=%d" % (name, prob.M))
    if prob.M <= 16:      # the CUDA-core int5 kernel on the same inputs
        ys = pq.pq_gemm5_skinny(a, asg, rs, L.w_d, L.whi_d, L.sz_d, prob.pb1, prob.pb2)
        torch.cuda.synchronize()
        assert_close(ys.float().cpu().numpy()[ms, ns], y64, "int5 skinny %s M=%d" % (name, prob.M))


# ---------------------------------------------------------------- graph API
@pytest.mark.parametrize("M", [1, 3, 40])
def test_layer_graph_replays_the_step(pq, orc, M):
    """PQLinear.make_graph: each replay copies the pinned input in, runs the
    prologue and GEMM, and copies y out; bit-equal to the eager call, also
    after new values are written into the pinned input."""
    prob = pqgen.make_problem(M, 512, 256, seed=55 + M)
    layer = pq.PQLinear(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta, prob.cs)
    xh = torch.from_numpy(prob.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((M, 256), dtype=torch.bfloat16).pin_memory()
    step = layer.make_graph(xh, yh)
    for seed in (55 + M, 155 + M):
        x = pqgen.make_problem(M, 512, 256, seed=seed).x
        xh.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        yh.fill_(float("nan"))
        step()
        torch.cuda.synchronize()
        y_eager = layer(dev_u16(x).view(torch.bfloat16))
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_eager.cpu().view(torch.int16))
        t = orc.pack(prob)
        a_o, asg_o, rs_o = orc.rotate_quant(x, prob.cs, t["rec"])
        assert_close(yh.float().numpy(), orc.gemm_f64(a_o, asg_o, rs_o, t["codes"], t["sz"], 256, 256),
                     "graph M=%d" % M)


@pytest.mark.parametrize("M,N", [(1, 256), (4, 17408), (40, 512)])
def test_layer_graph_zero_copy(pq, orc, M, N):
    """make_graph(zero_copy=True): the prologue reads x from the pinned host
    buffer and the GEMM writes y into the pinned host buffer directly; every
    replay must equal the eager call bit for bit, also after new values are
    written into the pinned input, and the host buffers must pass the access
    check that pageable memory fails."""
    K = 512
    prob = pqgen.make_problem(M, K, N, seed=75 + M)
    layer = pq.PQLinear(prob.qweight, prob.qzeros, prob.scales, prob.pairs, prob.theta, prob.cs)
    xh = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
    yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    pq.pq_check_device_access(xh)
    pq.pq_check_device_access(yh)
    pq.pq_check_device_access(layer.w)
    with pytest.raises(pq.PQError) as e:
        pq.pq_check_device_access(torch.empty((M, K), dtype=torch.bfloat16))   # pageable
    assert e.value.status == 8
    del e      # the traceback holds this frame, and the frame will hold the graph
    step = layer.make_graph(xh, yh, zero_copy=True)
    for seed in (75 + M, 175 + M, 275 + M):
        x = pqgen.make_problem(M, K, N, seed=seed).x
        xh.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        yh.fill_(float("nan"))
        step()
        torch.cuda.synchronize()
        y_eager = layer(dev_u16(x).view(torch.bfloat16))
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_eager.cpu().view(torch.int16)), seed
    t = orc.pack(prob)
    a_o, asg_o, rs_o = orc.rotate_quant(x, prob.cs, t["rec"])
    ms, ns = _samples(M, N, N, N, 1000, 3)
    y64 = orc.gemm_f64_sampled(ms, ns, a_o, asg_o, rs_o, t["codes"], t["sz"], N, N)
    assert_close(yh.float().numpy()[ms, ns], y64, "zero-copy graph M=%d" % M)


# ---------------------------------------------------------------- repeated launches
@pytest.mark.parametrize("path", ["skinny", "tcn", "tc"])
def test_gemm_repeated_graph_launches_status_clean(pq, orc, path):
    """Many back-to-back launches chained by programmatic dependent launch,
    replayed from a CUDA graph over rotating buffers: every bounded wait in
    every launch must succeed (status word stays 0) and the last results must
    still match the first ones bit for bit."""
    M, K, N = 4, 5120, 17408
    prob = pqgen.make_problem(M, K, N, seed=12)
    L = Problem(pq, orc, prob, check_pack=False)
    fn = {"skinny": pq.pq_gemm_skinny, "tcn": pq.pq_gemm_tcn, "tc": pq.pq_gemm_tc}[path]
    C = 7
    acts = [pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d) for _ in range(C)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(C)]
    st = torch.zeros((C, 1), dtype=torch.int32, device="cuda")
    fn(*acts[0], L.w_d, L.sz_d, N, N, y=ys[0], dev_status=st[0])
    torch.cuda.synchronize()
    ref = ys[0].clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(C):
            fn(*acts[j], L.w_d, L.sz_d, N, N, y=ys[j], dev_status=st[j])
    reps = 300 if path != "tc" else 40
    for _ in range(reps):
        g.replay()
    torch.cuda.synchronize()
    assert int(st.abs().sum().item()) == 0, "a bounded wait gave up: %s" % st.flatten().tolist()
    for j in range(C):
        assert torch.equal(ys[j], ref), j


@pytest.mark.parametrize("K", [1152, 2176])
@pytest.mark.parametrize("M", [1, 16])
def test_gemm_tail_slabs_repeated(pq, orc, M, K):
    """K/128 one past a multiple of the kernels' stage counts, so the last slab
    reuses a stage while other warps finish: twenty launches per path must
    all match the fp64 oracle and each other bit for bit."""
    N = 512
    prob = pqgen.make_problem(M, K, N, seed=13)
    L = Problem(pq, orc, prob, check_pack=False)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    torch.cuda.synchronize()
    y64 = orc.gemm_f64(a.cpu().numpy(), asg.cpu().numpy(), rs.cpu().numpy(), L.t["codes"], L.t["sz"], N, N)
    for name, fn in gemm_paths(pq, M):
        first = run_gemm(fn, a, asg, rs, L, N, N, M, N)
        assert_close(first, y64, "%s M=%d K=%d" % (name, M, K))
        for _ in range(20):
            y = run_gemm(fn, a, asg, rs, L, N, N, M, N)
            assert np.array_equal(y, first), name


@pytest.mark.parametrize("bits,M", [(5, 4), (5, 16), (4, 4), (4, 16)])
def test_narrow_kernel_repeated_launches_bit_identical(pq, orc, bits, M):
    """The narrow tensor-core kernel at the decode gate_up size: eight launches
    must give bit-identical outputs (a ring-ownership race shows up as run-to-run
    differences in a few columns), and the first must match the fp64 oracle on
    sampled outputs."""
    K, N = 5120, 17408
    prob = pqgen.make_problem(M, K, N, seed=41 + M + bits, bits=bits)
    L = (Problem5 if bits == 5 else Problem)(pq, orc, prob, check_pack=False)
    a, asg, rs = pq.pq_rotate_quant(L.x_d, L.rec_d, L.cs_d)
    name = "pq_gemm5_tcn" if bits == 5 else None
    outs = []
    for _ in range(8):
        if bits == 5:
            y = run_gemm5(name, a, asg, rs, L, N, N, M, N)
        else:
            y = run_gemm(pq.pq_gemm_tcn, a, asg, rs, L, N, N, M, N)
        outs.append(y)
    for j in range(1, 8):
        assert np.array_equal(outs[j], outs[0]), "launch %d differs" % j
    ms, ns = _samples(M, N, N, N, 2000, 17)
    a_h, s_h, r_h = a.cpu().numpy(), asg.cpu().numpy(), rs.cpu().numpy()
    if bits == 5:
        y64 = orc.gemm5_f64_sampled(ms, ns, a_h, s_h, r_h, L.t["codes"], L.t["sz"], N, N)
    else:
        y64 = orc.gemm_f64_sampled(ms, ns, a_h, s_h, r_h, L.t["codes"], L.t["sz"], N, N)
    assert_close(outs[0][ms, ns], y64, "tcn int%d M=%d" % (bits, M))
