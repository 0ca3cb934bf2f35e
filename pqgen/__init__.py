"""Seeded synthetic inputs for the ParoQuant W4A8 rotated-int4 linear layer.

This module only draws random numbers and lays them out in the checkpoint
format the ParoQuant engineering log describes ("ParoQuant (PARO) W4A8 on
gfx1201 -- engineering log", section "Format"):

* ``x``        bf16 ``[M, K]`` activations (returned as uint16 bit patterns)
* ``qweight``  int32 ``[K, N/8]``, eight 4-bit codes per word
* ``qzeros``   int32 ``[K/128, N/8]``, eight 4-bit zero points per word
* ``scales``   f16 ``[K/128, N]`` group scales (uint16 bit patterns)
* ``pairs``    int16 ``[P, 8, K]``, per 128-channel group a permutation of 0..127
* ``theta``    f16 ``[P, 8, K/2]`` Givens angles (uint16 bit patterns)
* ``cs``       f16 ``[P, K]`` channel scales, stored pre-inverted (uint16 bits)

With ``bits=5`` (int5 weights, "2026-09-10: int5 W5A8 ParoQuant"): ``qweight``
and ``qzeros`` hold the low nibbles, and ``qweight_hi`` int32 ``[K, N/32]`` and
``qzeros_hi`` int32 ``[K/128, N/32]`` the fifth bits, 32 columns per word.
Every nibble and every fifth bit is an independent uniform draw, so the codes
are uniform 0..31 and the zero points uniform 0..31.

It holds none of the method's arithmetic: no rotation, no quantisation, no
unpacking.  Every nibble of ``qweight`` is an independent uniform code 0..15
and every nibble of ``qzeros`` an independent uniform zero point 2..14, so the
position of a column inside a word never has to be known here.

Each tensor is drawn from ``numpy.random.default_rng([seed, tensor_id, p])``
with a fixed ``tensor_id`` per tensor, so draws do not depend on the order in
which tensors are generated or on the other shapes.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "TENSOR_IDS", "CONFIGS", "Problem", "make_problem", "to_bf16_bits",
    "f16_bits", "random_codes", "config_problem",
]

# fixed ids: never renumber (stored fixtures and seeds depend on them)
TENSOR_IDS = {
    "x": 1, "qweight": 2, "qzeros": 3, "scales": 4, "pairs": 5, "theta": 6,
    "cs": 7, "outliers": 8, "codes": 9, "asg": 10, "sparse": 11,
    "qweight_hi": 12, "qzeros_hi": 13, "qzeros5": 14,
}

# The five workloads: (M, K, N, P, partition boundaries, extra knobs).
# seed = workload index - 1.
CONFIGS = {
    "tiny":     dict(M=4, K=256, N=128, P=1, seed=0),
    "decode":   dict(M=1, K=5120, N=17408, P=1, seed=1, outlier_frac=0.01),
    "prefill":  dict(M=2048, K=5120, N=17408, P=1, seed=2),
    "down":     dict(M=8192, K=8704, N=5120, P=1, seed=3),
    "qkv":      dict(M=512, K=5120, N=8192, P=3, seed=4, pb=(6144, 7168)),
}


def _rng(seed: int, name: str, p: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), TENSOR_IDS[name], int(p)])


def to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (input preparation)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    # finite inputs only: u + 0x7FFF + lsb cannot overflow 32 bits below the NaN range
    r = (u + (np.uint32(0x7FFF) + lsb)) >> np.uint32(16)
    return r.astype(np.uint16)


def f16_bits(f: np.ndarray) -> np.ndarray:
    """float -> IEEE binary16 bit patterns (numpy's own RNE conversion)."""
    return np.ascontiguousarray(np.asarray(f, dtype=np.float64).astype(np.float16)).view(np.uint16)


def _nibble_words(rng: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """int32 words whose eight nibbles are independent uniform integers in [lo, hi]."""
    nib = rng.integers(lo, hi + 1, size=tuple(shape) + (8,), dtype=np.uint32)
    w = np.zeros(tuple(shape), dtype=np.uint32)
    for i in range(8):
        w |= nib[..., i] << np.uint32(4 * i)
    return w.view(np.int32)


class Problem(dict):
    """A dict of generated tensors plus the shape fields (attribute access)."""

    def __getattr__(self, k):
        try:
            return self[k]
        except KeyError as e:
            raise AttributeError(k) from e


def make_problem(M: int, K: int, N: int, P: int = 1, seed: int = 0,
                 pb=None, outlier_frac: float = 0.0, x_sigma: float = 1.0,
                 x_mode: str = "normal", theta_range: float = 0.5, bits: int = 4) -> Problem:
    """Generate one synthetic linear layer and its input activations.

    x_mode: "normal"  -- x ~ N(0, x_sigma^2)
            "sparse"  -- per 128-group one channel ~ N(0,1) and the other 127
                         ~ N(0, 1e-5^2): with |theta| <~ 1e-5 the group scale is
                         set by the one large channel and most codes of the
                         group land in the e4m3 subnormal range
    """
    if K % 128 or N % 128:
        raise ValueError("K and N must be multiples of 128")
    if bits not in (4, 5):
        raise ValueError("bits must be 4 or 5")
    G = K // 128
    # activations, drawn and rounded to bf16 in row blocks (same stream as one draw)
    r = _rng(seed, "x")
    if outlier_frac > 0:
        n_out = int(round(outlier_frac * K))
        out_ch = _rng(seed, "outliers").choice(K, size=n_out, replace=False)
    x = np.empty((M, K), dtype=np.uint16)
    if x_mode == "sparse":
        hot = np.empty((0,), dtype=np.int64)
    for r0 in range(0, M, 256):
        rows = min(256, M - r0)
        if x_mode == "normal":
            xf = r.standard_normal((rows, K), dtype=np.float32)
            if x_sigma != 1.0:
                xf *= np.float32(x_sigma)
        elif x_mode == "sparse":
            xf = r.standard_normal((rows, K), dtype=np.float32) * np.float32(1e-5)
            hot = r.integers(0, 128, size=(rows, G))
            vals = r.standard_normal((rows, G), dtype=np.float32)
            ri = np.repeat(np.arange(rows), G)
            ci = np.tile(np.arange(G), rows) * 128 + hot.reshape(-1)
            xf[ri, ci] = vals.reshape(-1)
        else:
            raise ValueError(x_mode)
        if outlier_frac > 0:
            xf[:, out_ch] *= np.float32(20.0)
        x[r0:r0 + rows] = to_bf16_bits(xf)
    # weights (checkpoint format)
    # eight independent uniform codes 0..15 per word == one uniform 32-bit word
    qweight = _rng(seed, "qweight").integers(0, 1 << 32, size=(K, N // 8),
                                             dtype=np.uint64).astype(np.uint32).view(np.int32)
    if bits == 4:
        qzeros = _nibble_words(_rng(seed, "qzeros"), (G, N // 8), 2, 14)
    else:
        qzeros = _nibble_words(_rng(seed, "qzeros5"), (G, N // 8), 0, 15)
    scales = f16_bits(_rng(seed, "scales").uniform(0.002, 0.02, size=(G, N)))
    # rotations, one per partition
    pairs = np.empty((P, 8, K), dtype=np.int16)
    theta = np.empty((P, 8, K // 2), dtype=np.uint16)
    cs = np.empty((P, K), dtype=np.uint16)
    for p in range(P):
        rp = _rng(seed, "pairs", p)
        for layer in range(8):
            for g in range(G):
                pairs[p, layer, g * 128:(g + 1) * 128] = rp.permutation(128).astype(np.int16)
        theta[p] = f16_bits(_rng(seed, "theta", p).uniform(-theta_range, theta_range,
                                                              size=(8, K // 2))).reshape(8, K // 2)
        cs[p] = f16_bits(_rng(seed, "cs", p).uniform(0.5, 2.0, size=K))
    if pb is None:
        pb = {1: (N, N), 2: (N // 2 // 128 * 128, N), 3: None}[P]
        if pb is None:
            third = (N // 3) // 128 * 128
            pb = (third, 2 * third)
    prob = Problem(M=M, K=K, N=N, P=P, G=G, seed=seed, pb1=int(pb[0]), pb2=int(pb[1]),
                   x=x, qweight=qweight, qzeros=qzeros, scales=scales,
                   pairs=pairs, theta=theta, cs=cs, bits=bits)
    if bits == 5:
        def plane(name, rows):
            return _rng(seed, name).integers(0, 1 << 32, size=(rows, N // 32),
                                             dtype=np.uint64).astype(np.uint32).view(np.int32)
        prob["qweight_hi"] = plane("qweight_hi", K)
        prob["qzeros_hi"] = plane("qzeros_hi", G)
    return prob


def config_problem(name: str, M: int | None = None, **over) -> Problem:
    """The named workload (optionally with another M or knobs)."""
    c = dict(CONFIGS[name])
    if M is not None:
        c["M"] = M
    c.update(over)
    return make_problem(**c)


# all 254 finite e4m3 bit patterns (0x7F and 0xFF are the NaN codes)
_FINITE_E4M3 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def random_codes(P: int, M: int, K: int, seed: int, subnormal_only: bool = False) -> np.ndarray:
    """e4m3 activation codes [P, M, K] drawn uniformly from the finite code set
    (or from the 16 subnormal/zero codes 0x00-0x07, 0x80-0x87)."""
    r = _rng(seed, "codes")
    if subnormal_only:
        pool = np.array(list(range(8)) + [0x80 + i for i in range(8)], dtype=np.uint8)
    else:
        pool = _FINITE_E4M3
    return pool[r.integers(0, len(pool), size=(P, M, K))]


def random_scales(P: int, G: int, M: int, seed: int) -> np.ndarray:
    """Positive fp32 per-(partition, group, token) activation scales [P, G, M]."""
    return _rng(seed, "asg").uniform(1e-3, 1e-2, size=(P, G, M)).astype(np.float32)
