"""numpy front end of the plain CPU oracle (``oracle/pq_oracle.c``).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``w4a8_rotated_int4_gb300``) never imports it, and this package never imports
the product.

Every function follows one step of the method described on the page
"ParoQuant (PARO) W4A8 on gfx1201 -- engineering log" (sections "Format",
"Inference identity", "Design" 1-4, "Gates passed"); the C file's header
lists the readings taken where the page is silent.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, library routines, exhaustive enumeration, brute force).  The
one exception is bit-level agreement of the fp32 rotation with the pages' own
kernel, which prints no worked values: parity unpinned against the pages for
that detail; it is pinned against the stated operation order only.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        vp, i32, u64 = C.c_void_p, C.c_int, C.c_uint64
        L.orc_f16_to_double.restype = C.c_double
        L.orc_f16_to_double.argtypes = [C.c_uint16]
        L.orc_f16_from_double.restype = C.c_uint16
        L.orc_f16_from_double.argtypes = [C.c_double]
        L.orc_e4m3_decode.restype = C.c_double
        L.orc_e4m3_decode.argtypes = [C.c_uint8]
        L.orc_e4m3_encode.restype = C.c_uint8
        L.orc_e4m3_encode.argtypes = [C.c_float]
        L.orc_unpack_awq.argtypes = [i32, i32, vp, vp]
        L.orc_check_pairs.argtypes = [i32, i32, vp]
        L.orc_records.argtypes = [i32, i32, vp, vp, vp]
        L.orc_sz.argtypes = [i32, i32, vp, vp, vp]
        L.orc_repack.argtypes = [i32, i32, vp, vp]
        L.orc_unpack_plane.argtypes = [i32, i32, vp, vp]
        L.orc_codes5.argtypes = [i32, i32, vp, vp, vp]
        L.orc_sz5.argtypes = [i32, i32, vp, vp, vp, vp]
        L.orc_repack5.argtypes = [i32, i32, vp, vp, vp, vp]
        L.orc_gemm5_f64.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.orc_gemm5_f64_sampled.argtypes = [i32, vp, vp, i32, i32, i32, i32, i32,
                                            vp, vp, vp, vp, vp, vp]
        L.orc_rotate_group_f32.argtypes = [vp, i32, i32, i32, vp]
        L.orc_rotate_quant.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.orc_bf16_from_float.restype = C.c_uint16
        L.orc_bf16_from_float.argtypes = [C.c_float]
        L.orc_row_sumsq.restype = C.c_float
        L.orc_row_sumsq.argtypes = [i32, vp]
        L.orc_add_rms_rotate_quant.argtypes = [i32, i32, i32, i32, vp, vp, vp, C.c_float, vp, vp,
                                               vp, vp, vp, vp, vp]
        L.orc_exp32.restype = C.c_float
        L.orc_exp32.argtypes = [C.c_float]
        L.orc_silu_mul.restype = C.c_uint16
        L.orc_silu_mul.argtypes = [C.c_uint16, C.c_uint16]
        L.orc_silu_mul_rotate_quant.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.orc_rotate_tokquant.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.orc_gemm_ptok_f64.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.orc_gemm_ptok_f64_sampled.argtypes = [i32, vp, vp, i32, i32, i32, i32, i32,
                                                vp, vp, vp, vp, vp, vp]
        L.orc_gemm_f64.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.orc_gemm_f64_sampled.argtypes = [i32, vp, vp, i32, i32, i32, i32, i32,
                                           vp, vp, vp, vp, vp, vp]
        L.orc_gemm_format_f64.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.orc_linear_rotx_f64.argtypes = [i32] * 6 + [vp] * 6
        L.orc_linear_rotw_f64.argtypes = [i32] * 6 + [vp] * 6
        L.orc_e4m3_check_range.restype = C.c_longlong
        L.orc_e4m3_check_range.argtypes = [u64, u64, C.POINTER(C.c_uint32)]
        L.orc_e4m3_encode_range.argtypes = [u64, u64, vp]
        L.orc_num_threads.restype = i32
        L.orc_set_num_threads.argtypes = [i32]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars
def f16_to_double(h: int) -> float:
    return lib().orc_f16_to_double(int(h))


def f16_from_double(x: float) -> int:
    return int(lib().orc_f16_from_double(float(x)))


def e4m3_decode(c: int) -> float:
    return lib().orc_e4m3_decode(int(c))


def e4m3_encode(q: float) -> int:
    return int(lib().orc_e4m3_encode(float(q)))


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_check_range(lo: int, hi: int):
    """(#disagreements, first bad pattern) of the encoder against nearest-value
    search over binary32 patterns [lo, hi)."""
    first = C.c_uint32(0)
    bad = lib().orc_e4m3_check_range(lo, hi, C.byref(first))
    return int(bad), int(first.value)


def e4m3_encode_range(lo: int, hi: int) -> np.ndarray:
    """Oracle codes of the binary32 patterns [lo, hi)."""
    out = np.empty(hi - lo, dtype=np.uint8)
    lib().orc_e4m3_encode_range(lo, hi, _p(out))
    return out


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- format
def unpack_awq(packed: np.ndarray, N: int) -> np.ndarray:
    packed = _c(packed, np.int32)
    rows = packed.shape[0]
    out = np.empty((rows, N), dtype=np.uint8)
    lib().orc_unpack_awq(rows, N, _p(packed), _p(out))
    return out


def check_pairs(pairs: np.ndarray) -> bool:
    pairs = _c(pairs, np.int16)
    P, _, K = pairs.shape
    return lib().orc_check_pairs(P, K, _p(pairs)) == 0


def records(pairs: np.ndarray, theta: np.ndarray) -> np.ndarray:
    """Rotation records [P, 8, G, 64] x 8 bytes (as uint8 [P, 8, G, 64, 8])."""
    pairs = _c(pairs, np.int16)
    theta = _c(theta, np.uint16)
    P, _, K = pairs.shape
    out = np.zeros((P, 8, K // 128, 64, 8), dtype=np.uint8)
    rc = lib().orc_records(P, K, _p(pairs), _p(theta), _p(out))
    if rc != 0:
        raise ValueError("orc_records failed with code %d" % rc)
    return out


def chain_records(rec: np.ndarray) -> np.ndarray:
    """The records [P, 8, G, 64, 8] rearranged into the library's chained
    storage order (a layout of this library, not a step of the method).

    Layer 0 keeps the given order.  Between layers r and r + 1 the two
    pairings form alternating cycles; taking the cycles by their lowest
    channel c0, the walk goes c0 -> its layer-r partner y (kept: byte 2 of
    that layer-r record = 1 if y is its second channel) -> y's layer-(r+1)
    partner -> ... until it is back at c0.  Slot t of layer r + 1 is the
    layer-(r+1) pair holding the channel slot t kept, that channel first;
    a pair stored reversed gets its sine's sign bit flipped, which leaves the
    rotation unchanged because fl(-a) = -fl(a) and x - y = x + (-y) exactly.
    """
    rec = np.asarray(rec, dtype=np.uint8)
    P, L, G, T, _ = rec.shape
    out = np.zeros_like(rec)
    for p in range(P):
        for g in range(G):
            # the current layer's slots as (first, second, cos bits, sin bits)
            cur = [(int(rec[p, 0, g, t, 0]), int(rec[p, 0, g, t, 1]),
                    int(rec[p, 0, g, t, 4]) | int(rec[p, 0, g, t, 5]) << 8,
                    int(rec[p, 0, g, t, 6]) | int(rec[p, 0, g, t, 7]) << 8) for t in range(T)]
            for r in range(L):
                keep_second = [0] * T
                if r + 1 < L:
                    nxt = {}                 # channel -> (partner, cos, sin, is first in the given order)
                    for t in range(T):
                        i, j = int(rec[p, r + 1, g, t, 0]), int(rec[p, r + 1, g, t, 1])
                        c = int(rec[p, r + 1, g, t, 4]) | int(rec[p, r + 1, g, t, 5]) << 8
                        s = int(rec[p, r + 1, g, t, 6]) | int(rec[p, r + 1, g, t, 7]) << 8
                        nxt[i] = (j, c, s, True)
                        nxt[j] = (i, c, s, False)
                    where = {}               # channel -> (slot, partner) in layer r
                    for t, (u, v, _, _) in enumerate(cur):
                        where[u] = (t, v)
                        where[v] = (t, u)
                    new = [None] * T
                    done = set()
                    for c0 in range(2 * T):
                        if c0 in done:
                            continue
                        x = c0
                        while True:
                            t, y = where[x]
                            done.update((x, y))
                            keep_second[t] = 1 if y == cur[t][1] else 0
                            partner, c, s, first = nxt[y]
                            new[t] = (y, partner, c, s if first else s ^ 0x8000)
                            x = partner
                            if x == c0:
                                break
                for t, (u, v, c, s) in enumerate(cur):
                    out[p, r, g, t] = (u, v, keep_second[t], 0, c & 0xFF, c >> 8, s & 0xFF, s >> 8)
                if r + 1 < L:
                    cur = new
    return out


def sz_table(scales: np.ndarray, qzeros: np.ndarray) -> np.ndarray:
    """SZ table [G, N, 2] f16 bit patterns (scale, scale*(zp-8))."""
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.int32)
    G, N = scales.shape
    out = np.empty((G, N, 2), dtype=np.uint16)
    lib().orc_sz(G, N, _p(scales), _p(qzeros), _p(out))
    return out


def sz_kernel_layout(sz: np.ndarray) -> np.ndarray:
    """The SZ table [G, N, 2] rearranged into the library's storage order
    [N/8, G, 8, 2] (one contiguous 32-byte run per column octet and group)."""
    G, N, _ = sz.shape
    return np.ascontiguousarray(sz.reshape(G, N // 8, 8, 2).transpose(1, 0, 2, 3))


def repack(qweight: np.ndarray) -> np.ndarray:
    """Kernel weight bytes [N, K/2]."""
    qweight = _c(qweight, np.int32)
    K, N8 = qweight.shape
    out = np.empty((N8 * 8, K // 2), dtype=np.uint8)
    lib().orc_repack(K, N8 * 8, _p(qweight), _p(out))
    return out


# ---------------------------------------------------------------- int5 weights
def unpack_plane(plane: np.ndarray, N: int) -> np.ndarray:
    """Fifth-bit plane int32 [rows, N/32] -> bits uint8 [rows, N]."""
    plane = _c(plane, np.int32)
    out = np.empty((plane.shape[0], N), dtype=np.uint8)
    lib().orc_unpack_plane(plane.shape[0], N, _p(plane), _p(out))
    return out


def codes5(lo: np.ndarray, hi: np.ndarray, N: int) -> np.ndarray:
    """5-bit codes uint8 [rows, N] from the nibble words and the plane."""
    lo = _c(lo, np.int32)
    hi = _c(hi, np.int32)
    out = np.empty((lo.shape[0], N), dtype=np.uint8)
    lib().orc_codes5(lo.shape[0], N, _p(lo), _p(hi), _p(out))
    return out


def sz5_table(scales: np.ndarray, qzeros: np.ndarray, qzeros_hi: np.ndarray) -> np.ndarray:
    """SZ table of int5 weights [G, N, 2] f16 (scale, scale*(zp-16))."""
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.int32)
    qzeros_hi = _c(qzeros_hi, np.int32)
    G, N = scales.shape
    out = np.empty((G, N, 2), dtype=np.uint16)
    lib().orc_sz5(G, N, _p(scales), _p(qzeros), _p(qzeros_hi), _p(out))
    return out


def repack5(qweight: np.ndarray, qweight_hi: np.ndarray):
    """Kernel layouts (w [N, K/2] low nibbles, whi [N, K/8] fifth bits)."""
    qweight = _c(qweight, np.int32)
    qweight_hi = _c(qweight_hi, np.int32)
    K, N8 = qweight.shape
    N = N8 * 8
    w = np.empty((N, K // 2), dtype=np.uint8)
    whi = np.empty((N, K // 8), dtype=np.uint8)
    lib().orc_repack5(K, N, _p(qweight), _p(qweight_hi), _p(w), _p(whi))
    return w, whi


def gemm5_f64(a, asg, rs, codes, sz, pb1, pb2) -> np.ndarray:
    a = _c(a, np.uint8); asg = _c(asg, np.float32); rs = _c(rs, np.float32)
    codes = _c(codes, np.uint8); sz = _c(sz, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_gemm5_f64(M, N, K, pb1, pb2, _p(a), _p(asg), _p(rs), _p(codes), _p(sz), _p(y))
    return y


def gemm5_f64_sampled(ms, ns, a, asg, rs, codes, sz, pb1, pb2) -> np.ndarray:
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    a = _c(a, np.uint8); asg = _c(asg, np.float32); rs = _c(rs, np.float32)
    codes = _c(codes, np.uint8); sz = _c(sz, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty(len(ms), dtype=np.float64)
    lib().orc_gemm5_f64_sampled(len(ms), _p(ms), _p(ns), M, N, K, pb1, pb2, _p(a), _p(asg), _p(rs),
                                _p(codes), _p(sz), _p(y))
    return y


def pack5(prob) -> dict:
    """Oracle's own load-time tables for a generated int5 problem."""
    sz = sz5_table(prob["scales"], prob["qzeros"], prob["qzeros_hi"])
    w, whi = repack5(prob["qweight"], prob["qweight_hi"])
    rec = records(prob["pairs"], prob["theta"])
    return dict(rec=rec, rec_kernel=chain_records(rec), sz=sz, sz_kernel=sz_kernel_layout(sz),
                w=w, whi=whi, codes=codes5(prob["qweight"], prob["qweight_hi"], prob["N"]),
                zp=codes5(prob["qzeros"], prob["qzeros_hi"], prob["N"]))


# ---------------------------------------------------------------- prologue
def rotate_group_f32(rec: np.ndarray, p: int, g: int, v: np.ndarray) -> np.ndarray:
    rec = _c(rec, np.uint8)
    G = rec.shape[2]
    v = _c(v, np.float32).copy()
    lib().orc_rotate_group_f32(_p(rec), G, p, g, _p(v))
    return v


def rotate_quant(x: np.ndarray, cs: np.ndarray, rec: np.ndarray, want_v: bool = False):
    """(a e4m3 [P,M,K], asg f32 [P,G,M], rs f32 [P,G,M][, v f32 [P,M,K]])."""
    x = _c(x, np.uint16)
    cs = _c(cs, np.uint16)
    rec = _c(rec, np.uint8)
    M, ldx = x.shape
    P, K = cs.shape
    G = K // 128
    a = np.empty((P, M, K), dtype=np.uint8)
    asg = np.empty((P, G, M), dtype=np.float32)
    rs = np.empty((P, G, M), dtype=np.float32)
    v = np.empty((P, M, K), dtype=np.float32) if want_v else None
    lib().orc_rotate_quant(M, K, ldx, P, _p(x), _p(cs), _p(rec), _p(a), _p(asg), _p(rs),
                           _p(v) if want_v else None)
    return (a, asg, rs, v) if want_v else (a, asg, rs)


# ------------------------------------------------- fused producer (reading R16)
def bf16_from_float(f: float) -> int:
    return int(lib().orc_bf16_from_float(f))


def row_sumsq(s: np.ndarray) -> np.float32:
    """fp32 sum of squares of one row of bf16 values (reading R16 order)."""
    s = _c(s, np.float32)
    return np.float32(lib().orc_row_sumsq(s.shape[0], _p(s)))


def add_rms_rotate_quant(x, res, gamma, eps, cs, rec):
    """Residual add + Gemma RMSNorm + rotate + quant (reading R16).
    x, res bf16 bits [M, ldx]; gamma bf16 bits [K]; eps float; cs f16 bits
    [P, K].  Returns (res_out bf16 [M,K], h bf16 [M,K], a, asg, rs)."""
    x = _c(x, np.uint16)
    res = _c(res, np.uint16)
    gamma = _c(gamma, np.uint16)
    cs = _c(cs, np.uint16)
    rec = _c(rec, np.uint8)
    M, ldx = x.shape
    assert res.shape == x.shape
    P, K = cs.shape
    G = K // 128
    res_out = np.empty((M, K), dtype=np.uint16)
    h = np.empty((M, K), dtype=np.uint16)
    a = np.empty((P, M, K), dtype=np.uint8)
    asg = np.empty((P, G, M), dtype=np.float32)
    rs = np.empty((P, G, M), dtype=np.float32)
    lib().orc_add_rms_rotate_quant(M, K, ldx, P, _p(x), _p(res), _p(gamma), float(eps), _p(cs),
                                   _p(rec), _p(res_out), _p(h), _p(a), _p(asg), _p(rs))
    return res_out, h, a, asg, rs


# ------------------------------------------------- silu-mul producer (reading R17)
def exp32(x: float) -> float:
    return float(lib().orc_exp32(x))


def silu_mul(g: int, u: int) -> int:
    """bf16 bits of bf16(bf16(silu(g)) * u) for bf16 bits g, u."""
    return int(lib().orc_silu_mul(g, u))


def silu_mul_rotate_quant(y, cs, rec):
    """y bf16 bits [M, ldy] with gate in [0, I) and up in [I, 2I), I = K of
    cs.  Returns (act bf16 [M,I], a, asg, rs)."""
    y = _c(y, np.uint16)
    cs = _c(cs, np.uint16)
    rec = _c(rec, np.uint8)
    M, ldy = y.shape
    P, I = cs.shape
    assert ldy >= 2 * I
    G = I // 128
    act = np.empty((M, I), dtype=np.uint16)
    a = np.empty((P, M, I), dtype=np.uint8)
    asg = np.empty((P, G, M), dtype=np.float32)
    rs = np.empty((P, G, M), dtype=np.float32)
    lib().orc_silu_mul_rotate_quant(M, I, ldy, P, _p(y), _p(cs), _p(rec), _p(act), _p(a), _p(asg), _p(rs))
    return act, a, asg, rs


# ------------------------------------------------- per-token scales (reading R18)
def rotate_tokquant(x, cs, rec):
    """(xr bf16 [P,M,K], a e4m3 [P,M,K], As f32 [P,M], rs f32 [P,G,M])."""
    x = _c(x, np.uint16)
    cs = _c(cs, np.uint16)
    rec = _c(rec, np.uint8)
    M, ldx = x.shape
    P, K = cs.shape
    G = K // 128
    xr = np.empty((P, M, K), dtype=np.uint16)
    a = np.empty((P, M, K), dtype=np.uint8)
    As = np.empty((P, M), dtype=np.float32)
    rs = np.empty((P, G, M), dtype=np.float32)
    lib().orc_rotate_tokquant(M, K, ldx, P, _p(x), _p(cs), _p(rec), _p(xr), _p(a), _p(As), _p(rs))
    return xr, a, As, rs


def gemm_ptok_f64(a, As, rs, codes, sz, pb1, pb2) -> np.ndarray:
    a = _c(a, np.uint8); As = _c(As, np.float32); rs = _c(rs, np.float32)
    codes = _c(codes, np.uint8); sz = _c(sz, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_gemm_ptok_f64(M, N, K, pb1, pb2, _p(a), _p(As), _p(rs), _p(codes), _p(sz), _p(y))
    return y


def gemm_ptok_f64_sampled(ms, ns, a, As, rs, codes, sz, pb1, pb2) -> np.ndarray:
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    a = _c(a, np.uint8); As = _c(As, np.float32); rs = _c(rs, np.float32)
    codes = _c(codes, np.uint8); sz = _c(sz, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty(len(ms), dtype=np.float64)
    lib().orc_gemm_ptok_f64_sampled(len(ms), _p(ms), _p(ns), M, N, K, pb1, pb2, _p(a), _p(As), _p(rs),
                                    _p(codes), _p(sz), _p(y))
    return y


# ---------------------------------------------------------------- GEMM
def gemm_f64(a, asg, rs, codes, sz, pb1, pb2) -> np.ndarray:
    a = _c(a, np.uint8); asg = _c(asg, np.float32); rs = _c(rs, np.float32)
    codes = _c(codes, np.uint8); sz = _c(sz, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_gemm_f64(M, N, K, pb1, pb2, _p(a), _p(asg), _p(rs), _p(codes), _p(sz), _p(y))
    return y


def gemm_f64_sampled(ms, ns, a, asg, rs, codes, sz, pb1, pb2) -> np.ndarray:
    ms = _c(ms, np.int32); ns = _c(ns, np.int32)
    a = _c(a, np.uint8); asg = _c(asg, np.float32); rs = _c(rs, np.float32)
    codes = _c(codes, np.uint8); sz = _c(sz, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty(len(ms), dtype=np.float64)
    lib().orc_gemm_f64_sampled(len(ms), _p(ms), _p(ns), M, N, K, pb1, pb2, _p(a), _p(asg),
                               _p(rs), _p(codes), _p(sz), _p(y))
    return y


def gemm_format_f64(a, asg, codes, zp, scales, pb1, pb2) -> np.ndarray:
    a = _c(a, np.uint8); asg = _c(asg, np.float32); codes = _c(codes, np.uint8)
    zp = _c(zp, np.uint8); scales = _c(scales, np.uint16)
    P, M, K = a.shape
    N = codes.shape[1]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_gemm_format_f64(M, N, K, pb1, pb2, _p(a), _p(asg), _p(codes), _p(zp), _p(scales),
                              _p(y))
    return y


def linear_rotx_f64(x, cs, pairs, theta, W, pb1, pb2) -> np.ndarray:
    x = _c(x, np.uint16); cs = _c(cs, np.uint16); pairs = _c(pairs, np.int16)
    theta = _c(theta, np.uint16); W = _c(W, np.float64)
    M, K = x.shape
    N = W.shape[0]
    P = cs.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_linear_rotx_f64(M, K, N, P, pb1, pb2, _p(x), _p(cs), _p(pairs), _p(theta), _p(W),
                              _p(y))
    return y


def linear_rotw_f64(x, cs, pairs, theta, W, pb1, pb2) -> np.ndarray:
    x = _c(x, np.uint16); cs = _c(cs, np.uint16); pairs = _c(pairs, np.int16)
    theta = _c(theta, np.uint16); W = _c(W, np.float64)
    M, K = x.shape
    N = W.shape[0]
    P = cs.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_linear_rotw_f64(M, K, N, P, pb1, pb2, _p(x), _p(cs), _p(pairs), _p(theta), _p(W),
                              _p(y))
    return y


# ---------------------------------------------------------------- whole layer
def pack(prob) -> dict:
    """Oracle's own load-time tables for a generated problem."""
    sz = sz_table(prob["scales"], prob["qzeros"])
    rec = records(prob["pairs"], prob["theta"])
    return dict(rec=rec, rec_kernel=chain_records(rec),
                sz=sz, sz_kernel=sz_kernel_layout(sz),
                w=repack(prob["qweight"]),
                codes=unpack_awq(prob["qweight"], prob["N"]),
                zp=unpack_awq(prob["qzeros"], prob["N"]))


def layer(prob, tables=None):
    """Prologue + fp64 GEMM on a generated problem: (a, asg, rs, y64)."""
    t = tables or pack(prob)
    a, asg, rs = rotate_quant(prob["x"], prob["cs"], t["rec"])
    y = gemm_f64(a, asg, rs, t["codes"], t["sz"], prob["pb1"], prob["pb2"])
    return a, asg, rs, y


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def rel_err(y, y64) -> float:
    """Norm-wise relative error ||y - y64||_F / ||y64||_F."""
    y = np.asarray(y, dtype=np.float64)
    d = np.linalg.norm((y - y64).ravel())
    n = np.linalg.norm(np.asarray(y64, dtype=np.float64).ravel())
    return float(d / n) if n > 0 else float(d)


__all__ = [k for k in dir() if not k.startswith("_")]
