"""Python binding of libpq: the ParoQuant (PARO) W4A8 rotated-int4 linear layer
on one GB300 (sm_103a).

    y = ((x * channel_scales) R^T) dequant(Q)^T

The functions mirror the C ABI in include/pq.h one to one (same names, same
argument order after marshalling).  This module only converts arguments:
numpy arrays for the host packer, torch CUDA tensors (device memory) and the
current torch stream for the device calls.  Every step of the layer runs in
libpq's CUDA kernels; there is no fallback.  If libpq.so has not been built the
first call raises PQError.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpq.so")

# Every symbol include/pq.h declares.
EXPORTS = (
    "pq_abi_version", "pq_status_string", "pq_last_error", "pq_pack_sizes", "pq_pack",
    "pq_rotate_quant", "pq_add_rms_rotate_quant", "pq_silu_mul_rotate_quant", "pq_gemm", "pq_gemm_skinny_max_m", "pq_gemm_skinny",
    "pq_gemm_tc",
    "pq_gemm_tcn",
    "pq_rotate_tokquant", "pq_rotate_tokquant_noalloc", "pq_gemm_ptok",
    "pq_pack5", "pq_gemm5", "pq_gemm5_tc", "pq_gemm5_tcn", "pq_gemm5_skinny",
    "pq_e4m3_encode", "pq_test_set_wait_limit_ns", "pq_check_device_access",
)

STATUS = {0: "PQ_OK", 1: "PQ_ERR_NULL", 2: "PQ_ERR_SHAPE", 3: "PQ_ERR_ALIGN", 4: "PQ_ERR_PAIRS",
          5: "PQ_ERR_PARTITION", 6: "PQ_ERR_ARCH", 7: "PQ_ERR_CUDA", 8: "PQ_ERR_ACCESS"}


class PQError(RuntimeError):
    """A libpq call returned a non-zero status (or the library is missing)."""

    def __init__(self, msg, status=None):
        super().__init__(msg)
        self.status = status


_lib = None


def lib() -> C.CDLL:
    """The loaded libpq.so (raises PQError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise PQError("libpq.so is not built (run __graft_entry__.build() or "
                      "python w4a8_rotated_int4_gb300/build.py)")
    L = C.CDLL(LIB_PATH)
    vp, i32, st, u64 = C.c_void_p, C.c_int, C.c_size_t, C.POINTER(C.c_size_t)
    L.pq_abi_version.restype = i32
    L.pq_abi_version.argtypes = []
    L.pq_status_string.restype = C.c_char_p
    L.pq_status_string.argtypes = [i32]
    L.pq_last_error.restype = C.c_char_p
    L.pq_last_error.argtypes = []
    L.pq_pack_sizes.restype = i32
    L.pq_pack_sizes.argtypes = [i32, i32, i32, u64, u64, u64]
    L.pq_pack.restype = i32
    L.pq_pack.argtypes = [i32, i32, i32] + [vp] * 8
    L.pq_rotate_quant.restype = i32
    L.pq_rotate_quant.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    L.pq_add_rms_rotate_quant.restype = i32
    L.pq_add_rms_rotate_quant.argtypes = [vp, vp, vp, C.c_float, i32, i32, i32, i32] + [vp] * 8
    L.pq_silu_mul_rotate_quant.restype = i32
    L.pq_silu_mul_rotate_quant.argtypes = [vp, i32, i32, i32, i32] + [vp] * 7
    L.pq_gemm.restype = i32
    L.pq_gemm.argtypes = [vp, vp, vp] + [i32] * 6 + [vp, vp, vp, i32, vp]
    L.pq_gemm_skinny_max_m.restype = i32
    L.pq_gemm_skinny_max_m.argtypes = []
    for name in ("pq_gemm_skinny", "pq_gemm_tc", "pq_gemm_tcn"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [vp, vp, vp] + [i32] * 6 + [vp, vp, vp, i32, vp, vp]
    L.pq_rotate_tokquant.restype = i32
    L.pq_rotate_tokquant.argtypes = [vp, i32, i32, i32, i32] + [vp] * 7
    L.pq_rotate_tokquant_noalloc.restype = i32
    L.pq_rotate_tokquant_noalloc.argtypes = [vp, i32, i32, i32, i32] + [vp] * 6
    L.pq_gemm_ptok.restype = i32
    L.pq_gemm_ptok.argtypes = [vp, vp, vp] + [i32] * 6 + [vp, vp, vp, i32, vp, vp]
    L.pq_pack5.restype = i32
    L.pq_pack5.argtypes = [i32, i32, i32] + [vp] * 11
    L.pq_gemm5.restype = i32
    L.pq_gemm5.argtypes = [vp, vp, vp] + [i32] * 6 + [vp, vp, vp, vp, i32, vp]
    for name in ("pq_gemm5_tc", "pq_gemm5_tcn", "pq_gemm5_skinny"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [vp, vp, vp] + [i32] * 6 + [vp, vp, vp, vp, i32, vp, vp]
    L.pq_e4m3_encode.restype = i32
    L.pq_e4m3_encode.argtypes = [vp, vp, st, vp]
    L.pq_test_set_wait_limit_ns.restype = i32
    L.pq_test_set_wait_limit_ns.argtypes = [C.c_ulonglong]
    L.pq_check_device_access.restype = i32
    L.pq_check_device_access.argtypes = [vp]
    _lib = L
    return L


def _check(status: int, what: str) -> None:
    if status != 0:
        L = lib()
        raise PQError("%s: %s (%s): %s" % (what, STATUS.get(status, status),
                                           L.pq_status_string(status).decode(),
                                           L.pq_last_error().decode()), status)


def pq_abi_version() -> int:
    return int(lib().pq_abi_version())


def pq_gemm_skinny_max_m() -> int:
    return int(lib().pq_gemm_skinny_max_m())


# ---------------------------------------------------------------- host packer
def _np_ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def pq_pack_sizes(K: int, N: int, P: int):
    r, s, w = C.c_size_t(), C.c_size_t(), C.c_size_t()
    _check(lib().pq_pack_sizes(K, N, P, C.byref(r), C.byref(s), C.byref(w)), "pq_pack_sizes")
    return r.value, s.value, w.value


def pq_pack(qweight: np.ndarray, qzeros: np.ndarray, scales: np.ndarray, pairs: np.ndarray,
            theta: np.ndarray):
    """Host packer.  Inputs in checkpoint layout (f16 tensors as uint16 bit
    patterns); returns (rec uint8 [P,8,G,64,8], sz uint16 [N/8,G,8,2],
    w uint8 [N,K/2])."""
    qweight = np.ascontiguousarray(qweight, dtype=np.int32)
    qzeros = np.ascontiguousarray(qzeros, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    pairs = np.ascontiguousarray(pairs, dtype=np.int16)
    theta = np.ascontiguousarray(theta, dtype=np.uint16)
    K, N = qweight.shape[0], qweight.shape[1] * 8
    if pairs.ndim == 2:
        pairs = pairs[None]
        theta = theta[None]
    P = pairs.shape[0]
    G = K // 128
    nr, ns, nw = pq_pack_sizes(K, N, P)
    rec = np.empty((P, 8, G, 64, 8), dtype=np.uint8)
    sz = np.empty((N // 8, G, 8, 2), dtype=np.uint16)
    w = np.empty((N, K // 2), dtype=np.uint8)
    assert rec.nbytes == nr and sz.nbytes == ns and w.nbytes == nw
    _check(lib().pq_pack(K, N, P, _np_ptr(qweight), _np_ptr(qzeros), _np_ptr(scales),
                         _np_ptr(pairs), _np_ptr(theta), _np_ptr(rec), _np_ptr(sz), _np_ptr(w)),
           "pq_pack")
    return rec, sz, w


def pq_pack5(qweight, qzeros, qweight_hi, qzeros_hi, scales, pairs, theta):
    """Host packer for int5 weights: pq_pack's inputs plus the fifth-bit planes
    qweight_hi int32 [K, N/32] and qzeros_hi int32 [G, N/32].  Returns
    (rec, sz, w, whi uint8 [N, K/8])."""
    qweight = np.ascontiguousarray(qweight, dtype=np.int32)
    qzeros = np.ascontiguousarray(qzeros, dtype=np.int32)
    qweight_hi = np.ascontiguousarray(qweight_hi, dtype=np.int32)
    qzeros_hi = np.ascontiguousarray(qzeros_hi, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    pairs = np.ascontiguousarray(pairs, dtype=np.int16)
    theta = np.ascontiguousarray(theta, dtype=np.uint16)
    K, N = qweight.shape[0], qweight.shape[1] * 8
    if pairs.ndim == 2:
        pairs = pairs[None]
        theta = theta[None]
    P = pairs.shape[0]
    G = K // 128
    if qweight_hi.shape != (K, N // 32) or qzeros_hi.shape != (G, N // 32):
        raise PQError("pq_pack5: fifth-bit planes must be [K, N/32] and [G, N/32]")
    rec = np.empty((P, 8, G, 64, 8), dtype=np.uint8)
    sz = np.empty((N // 8, G, 8, 2), dtype=np.uint16)
    w = np.empty((N, K // 2), dtype=np.uint8)
    whi = np.empty((N, K // 8), dtype=np.uint8)
    _check(lib().pq_pack5(K, N, P, _np_ptr(qweight), _np_ptr(qzeros), _np_ptr(qweight_hi), _np_ptr(qzeros_hi),
                          _np_ptr(scales), _np_ptr(pairs), _np_ptr(theta), _np_ptr(rec), _np_ptr(sz),
                          _np_ptr(w), _np_ptr(whi)), "pq_pack5")
    return rec, sz, w, whi


# ---------------------------------------------------------------- device calls
def _torch():
    import torch
    return torch


def _dptr(t) -> C.c_void_p:
    if not t.is_cuda:
        raise PQError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise PQError("expected a contiguous tensor")
    return C.c_void_p(t.data_ptr())


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _expect(t, what, dtype=None, shape=None, nbytes=None):
    """Raise PQError unless tensor t has the given dtype, shape and byte size:
    the C ABI takes raw pointers, so a mis-sized tensor would be read or
    written out of bounds on the device."""
    if dtype is not None and t.dtype != dtype:
        raise PQError("%s: dtype %s, expected %s" % (what, t.dtype, dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise PQError("%s: shape %s, expected %s" % (what, tuple(t.shape), tuple(shape)))
    if nbytes is not None and _nbytes(t) != nbytes:
        raise PQError("%s: %d bytes, expected %d" % (what, _nbytes(t), nbytes))


def _rotation_args(x, rec, cs, what):
    """Checks shared by the prologues: x bf16 [M, ldx], cs 2-byte [P, K],
    rec pq_pack's record table for (P, K).  Returns (M, ldx, P, K, G)."""
    torch = _torch()
    _expect(x, what + " x", dtype=torch.bfloat16)
    if x.dim() != 2:
        raise PQError("%s x: expected a 2-D [M, ldx] tensor" % what)
    if cs.dim() != 2 or cs.element_size() != 2:
        raise PQError("%s cs: expected a 2-byte [P, K] tensor" % what)
    M, ldx = x.shape
    P, K = cs.shape
    if K % 128 or K < 128 or ldx < K:
        raise PQError("%s: K = %d must be a positive multiple of 128 and <= ldx = %d" % (what, K, ldx))
    G = K // 128
    _expect(rec, what + " rec", nbytes=P * 8 * G * 64 * 8)
    return M, ldx, P, K, G


def _quant_outputs(what, P, M, K, G, a, asg, rs):
    torch = _torch()
    _expect(a, what + " a", dtype=torch.uint8, shape=(P, M, K))
    _expect(asg, what + " asg", dtype=torch.float32, shape=(P, G, M))
    _expect(rs, what + " rs", dtype=torch.float32, shape=(P, G, M))


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def pq_rotate_quant(x, rec, cs, a=None, asg=None, rs=None, stream=None):
    """x bf16 [M, ldx>=K] (CUDA), rec uint8 (device copy of pq_pack's rec),
    cs f16 [P, K].  Returns (a uint8 [P,M,K] e4m3 codes, asg f32 [P,G,M], rs f32 [P,G,M])."""
    torch = _torch()
    M, ldx, P, K, G = _rotation_args(x, rec, cs, "pq_rotate_quant")
    dev = x.device
    if a is None:
        a = torch.empty((P, M, K), dtype=torch.uint8, device=dev)
    if asg is None:
        asg = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    if rs is None:
        rs = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    _quant_outputs("pq_rotate_quant", P, M, K, G, a, asg, rs)
    _check(lib().pq_rotate_quant(_dptr(x), M, K, ldx, P, _dptr(rec), _dptr(cs), _dptr(a),
                                 _dptr(asg), _dptr(rs), _stream(stream)), "pq_rotate_quant")
    return a, asg, rs


def pq_add_rms_rotate_quant(x, residual, gamma, eps, rec, cs, residual_out=None, h=None, a=None,
                            asg=None, rs=None, stream=None):
    """Residual add + Gemma RMSNorm + rotate + quant in one call.
    x, residual bf16 [M, ldx>=K] (CUDA, same strides), gamma bf16 [K], eps
    float, rec and cs as for pq_rotate_quant.  Returns (residual_out bf16
    [M,K], h bf16 [M,K], a uint8 [P,M,K], asg f32 [P,G,M], rs f32 [P,G,M])."""
    torch = _torch()
    M, ldx, P, K, G = _rotation_args(x, rec, cs, "pq_add_rms_rotate_quant")
    if tuple(residual.shape) != (M, ldx) or residual.stride(0) != x.stride(0):
        raise PQError("residual must have x's shape and row stride")
    _expect(residual, "pq_add_rms_rotate_quant residual", dtype=torch.bfloat16)
    _expect(gamma, "pq_add_rms_rotate_quant gamma", dtype=torch.bfloat16, nbytes=2 * K)
    dev = x.device
    if residual_out is None:
        residual_out = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if h is None:
        h = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if a is None:
        a = torch.empty((P, M, K), dtype=torch.uint8, device=dev)
    if asg is None:
        asg = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    if rs is None:
        rs = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    _expect(residual_out, "pq_add_rms_rotate_quant residual_out", dtype=torch.bfloat16, shape=(M, K))
    _expect(h, "pq_add_rms_rotate_quant h", dtype=torch.bfloat16, shape=(M, K))
    _quant_outputs("pq_add_rms_rotate_quant", P, M, K, G, a, asg, rs)
    _check(lib().pq_add_rms_rotate_quant(_dptr(x), _dptr(residual), _dptr(gamma), C.c_float(eps), M, K,
                                         x.stride(0), P, _dptr(rec), _dptr(cs), _dptr(residual_out),
                                         _dptr(h), _dptr(a), _dptr(asg), _dptr(rs), _stream(stream)),
           "pq_add_rms_rotate_quant")
    return residual_out, h, a, asg, rs


def pq_silu_mul_rotate_quant(y, rec, cs, act=None, a=None, asg=None, rs=None, stream=None):
    """silu(gate) * up + rotate + quant.  y bf16 [M, ldy >= 2I] (CUDA): the
    merged gate/up output, gate in columns [0, I) and up in [I, 2I); rec and
    cs for the down projection (cs f16 [P, I]).  Returns (act bf16 [M, I],
    a uint8 [P, M, I], asg f32 [P, G, M], rs f32 [P, G, M])."""
    torch = _torch()
    _expect(y, "pq_silu_mul_rotate_quant y", dtype=torch.bfloat16)
    if y.dim() != 2 or cs.dim() != 2 or cs.element_size() != 2:
        raise PQError("pq_silu_mul_rotate_quant: y must be 2-D [M, ldy], cs a 2-byte [P, I] tensor")
    M, ldy = y.shape
    P, I = cs.shape
    if I % 128 or I < 128 or ldy < 2 * I:
        raise PQError("pq_silu_mul_rotate_quant: I = %d must be a positive multiple of 128, ldy >= 2I" % I)
    G = I // 128
    _expect(rec, "pq_silu_mul_rotate_quant rec", nbytes=P * 8 * G * 64 * 8)
    dev = y.device
    if act is None:
        act = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
    if a is None:
        a = torch.empty((P, M, I), dtype=torch.uint8, device=dev)
    if asg is None:
        asg = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    if rs is None:
        rs = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    _expect(act, "pq_silu_mul_rotate_quant act", dtype=torch.bfloat16, shape=(M, I))
    _quant_outputs("pq_silu_mul_rotate_quant", P, M, I, G, a, asg, rs)
    _check(lib().pq_silu_mul_rotate_quant(_dptr(y), M, I, y.stride(0), P, _dptr(rec), _dptr(cs), _dptr(act),
                                          _dptr(a), _dptr(asg), _dptr(rs), _stream(stream)),
           "pq_silu_mul_rotate_quant")
    return act, a, asg, rs


def _gemm_args(a, asg, rs, w, sz, pb1, pb2, y, per_token=False, whi=None):
    """Shapes of a GEMM call, checked against (P, M, K) from a and N from w:
    a uint8 [P, M, K]; asg, rs f32 [P, G, M] (per-token: As f32 [P, M]);
    w uint8 [N, K/2]; sz G * N 4-byte words; whi uint8 [N, K/8]; y bf16
    [M, >= N]."""
    torch = _torch()
    if a.dim() != 3 or w.dim() != 2:
        raise PQError("GEMM: a must be [P, M, K] and w [N, K/2]")
    P, M, K = a.shape
    N = w.shape[0]
    G = K // 128
    _expect(a, "GEMM a", dtype=torch.uint8)
    _expect(w, "GEMM w", dtype=torch.uint8, shape=(N, K // 2))
    _expect(asg, "GEMM As" if per_token else "GEMM asg", dtype=torch.float32,
            shape=(P, M) if per_token else (P, G, M))
    _expect(rs, "GEMM rs", dtype=torch.float32, shape=(P, G, M))
    _expect(sz, "GEMM sz", nbytes=4 * G * N)
    if whi is not None:
        _expect(whi, "GEMM whi", dtype=torch.uint8, nbytes=N * K // 8)
    if pb1 is None:
        pb1 = pb2 = N
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _expect(y, "GEMM y", dtype=torch.bfloat16)
    if y.dim() != 2 or y.shape[0] != M or y.shape[1] < N:
        raise PQError("GEMM y: shape %s, expected [%d, >= %d]" % (tuple(y.shape), M, N))
    return P, M, K, N, pb1, pb2, y


def pq_gemm(a, asg, rs, w, sz, pb1=None, pb2=None, y=None, stream=None):
    """y bf16 [M, N] = group GEMM of the prologue outputs with the packed weights."""
    P, M, K, N, pb1, pb2, y = _gemm_args(a, asg, rs, w, sz, pb1, pb2, y)
    _check(lib().pq_gemm(_dptr(a), _dptr(asg), _dptr(rs), M, N, K, P, pb1, pb2, _dptr(w),
                         _dptr(sz), _dptr(y), y.stride(0), _stream(stream)), "pq_gemm")
    return y


def _status_ptr(dev_status):
    if dev_status is None:
        return None
    if _nbytes(dev_status) < 4:
        raise PQError("dev_status: needs at least one 4-byte word")
    return _dptr(dev_status)


def _gemm_path(fn, name, a, asg, rs, w, sz, pb1, pb2, y, dev_status, stream, per_token=False):
    P, M, K, N, pb1, pb2, y = _gemm_args(a, asg, rs, w, sz, pb1, pb2, y, per_token=per_token)
    st = _status_ptr(dev_status)
    _check(fn(_dptr(a), _dptr(asg), _dptr(rs), M, N, K, P, pb1, pb2, _dptr(w), _dptr(sz),
              _dptr(y), y.stride(0), st, _stream(stream)), name)
    return y


def pq_gemm_skinny(a, asg, rs, w, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    return _gemm_path(lib().pq_gemm_skinny, "pq_gemm_skinny", a, asg, rs, w, sz, pb1, pb2, y,
                      dev_status, stream)


def pq_gemm_tc(a, asg, rs, w, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    return _gemm_path(lib().pq_gemm_tc, "pq_gemm_tc", a, asg, rs, w, sz, pb1, pb2, y,
                      dev_status, stream)


def pq_gemm_tcn(a, asg, rs, w, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    return _gemm_path(lib().pq_gemm_tcn, "pq_gemm_tcn", a, asg, rs, w, sz, pb1, pb2, y,
                      dev_status, stream)


def _tokquant_outputs(what, P, M, K, G, a, As, rs):
    torch = _torch()
    _expect(a, what + " a", dtype=torch.uint8, shape=(P, M, K))
    _expect(As, what + " As", dtype=torch.float32, shape=(P, M))
    _expect(rs, what + " rs", dtype=torch.float32, shape=(P, G, M))


def pq_rotate_tokquant(x, rec, cs, xr=None, a=None, As=None, rs=None, stream=None):
    """Per-token prologue: x bf16 [M, ldx>=K] (CUDA), rec, cs as for
    pq_rotate_quant.  Returns (xr bf16 [P,M,K] rotated rows, a uint8 [P,M,K]
    e4m3 codes, As f32 [P,M] token scales, rs f32 [P,G,M] plain row-sums)."""
    torch = _torch()
    M, ldx, P, K, G = _rotation_args(x, rec, cs, "pq_rotate_tokquant")
    dev = x.device
    if xr is None:
        xr = torch.empty((P, M, K), dtype=torch.bfloat16, device=dev)
    if a is None:
        a = torch.empty((P, M, K), dtype=torch.uint8, device=dev)
    if As is None:
        As = torch.empty((P, M), dtype=torch.float32, device=dev)
    if rs is None:
        rs = torch.empty((P, G, M), dtype=torch.float32, device=dev)
    _expect(xr, "pq_rotate_tokquant xr", dtype=torch.bfloat16, shape=(P, M, K))
    _tokquant_outputs("pq_rotate_tokquant", P, M, K, G, a, As, rs)
    _check(lib().pq_rotate_tokquant(_dptr(x), M, K, ldx, P, _dptr(rec), _dptr(cs), _dptr(xr), _dptr(a),
                                    _dptr(As), _dptr(rs), _stream(stream)), "pq_rotate_tokquant")
    return xr, a, As, rs


def pq_rotate_tokquant_noalloc(x, rec, cs, a, As, rs, stream=None):
    """pq_rotate_tokquant with the library's fixed scratch instead of xr:
    for callers that cannot allocate device memory, so every output (a uint8
    [P,M,K], As f32 [P,M], rs f32 [P,G,M]) is the caller's; P * M * K must not
    exceed the library's limit.  Returns (a, As, rs)."""
    M, ldx, P, K, G = _rotation_args(x, rec, cs, "pq_rotate_tokquant_noalloc")
    _tokquant_outputs("pq_rotate_tokquant_noalloc", P, M, K, G, a, As, rs)
    _check(lib().pq_rotate_tokquant_noalloc(_dptr(x), M, K, ldx, P, _dptr(rec), _dptr(cs), _dptr(a),
                                            _dptr(As), _dptr(rs), _stream(stream)),
           "pq_rotate_tokquant_noalloc")
    return a, As, rs


def pq_gemm_ptok(a, As, rs, w, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    """y bf16 [M, N] from the per-token prologue's outputs (As in the epilogue)."""
    return _gemm_path(lib().pq_gemm_ptok, "pq_gemm_ptok", a, As, rs, w, sz, pb1, pb2, y,
                      dev_status, stream, per_token=True)


def pq_gemm5(a, asg, rs, w, whi, sz, pb1=None, pb2=None, y=None, stream=None):
    """y bf16 [M, N]: the group GEMM on int5 weights (pq_pack5's w, whi, sz)."""
    P, M, K, N, pb1, pb2, y = _gemm_args(a, asg, rs, w, sz, pb1, pb2, y, whi=whi)
    _check(lib().pq_gemm5(_dptr(a), _dptr(asg), _dptr(rs), M, N, K, P, pb1, pb2, _dptr(w), _dptr(whi),
                          _dptr(sz), _dptr(y), y.stride(0), _stream(stream)), "pq_gemm5")
    return y


def _gemm5_path(fn, name, a, asg, rs, w, whi, sz, pb1, pb2, y, dev_status, stream):
    P, M, K, N, pb1, pb2, y = _gemm_args(a, asg, rs, w, sz, pb1, pb2, y, whi=whi)
    st = _status_ptr(dev_status)
    _check(fn(_dptr(a), _dptr(asg), _dptr(rs), M, N, K, P, pb1, pb2, _dptr(w), _dptr(whi), _dptr(sz),
              _dptr(y), y.stride(0), st, _stream(stream)), name)
    return y


def pq_gemm5_tc(a, asg, rs, w, whi, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    return _gemm5_path(lib().pq_gemm5_tc, "pq_gemm5_tc", a, asg, rs, w, whi, sz, pb1, pb2, y, dev_status,
                       stream)


def pq_gemm5_tcn(a, asg, rs, w, whi, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    return _gemm5_path(lib().pq_gemm5_tcn, "pq_gemm5_tcn", a, asg, rs, w, whi, sz, pb1, pb2, y, dev_status,
                       stream)


def pq_gemm5_skinny(a, asg, rs, w, whi, sz, pb1=None, pb2=None, y=None, dev_status=None, stream=None):
    return _gemm5_path(lib().pq_gemm5_skinny, "pq_gemm5_skinny", a, asg, rs, w, whi, sz, pb1, pb2, y,
                       dev_status, stream)


def pq_e4m3_encode(x, out=None, stream=None):
    """The prologue's device e4m3 encoder on an fp32 CUDA tensor."""
    torch = _torch()
    _expect(x, "pq_e4m3_encode x", dtype=torch.float32)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _expect(out, "pq_e4m3_encode out", dtype=torch.uint8, nbytes=x.numel())
    _check(lib().pq_e4m3_encode(_dptr(x), _dptr(out), x.numel(), _stream(stream)),
           "pq_e4m3_encode")
    return out


def pq_test_set_wait_limit_ns(ns):
    """Test hook: the GEMM kernels' pipeline-wait bound in ns (0 = product bound)."""
    _check(lib().pq_test_set_wait_limit_ns(int(ns)), "pq_test_set_wait_limit_ns")


def pq_check_device_access(t):
    """Raise PQError unless kernels on the current device can dereference the
    storage of tensor t (or the integer address t) directly: memory of the
    current device, managed memory, or page-locked host memory mapped at the
    same address."""
    ptr = t.data_ptr() if hasattr(t, "data_ptr") else int(t)
    _check(lib().pq_check_device_access(C.c_void_p(ptr)), "pq_check_device_access")


class PQLinear:
    """One packed projection resident in device memory: pq_pack once, then
    forward(x) = pq_rotate_quant + pq_gemm on the current stream."""

    def __init__(self, qweight, qzeros, scales, pairs, theta, cs, pb=None, device="cuda"):
        torch = _torch()
        rec, sz, w = pq_pack(qweight, qzeros, scales, pairs, theta)
        self.P, self.K, self.N = rec.shape[0], w.shape[1] * 2, w.shape[0]
        self.pb1, self.pb2 = pb if pb is not None else (self.N, self.N)
        self.rec = torch.from_numpy(rec).to(device)
        self.sz = torch.from_numpy(sz.view(np.int16)).to(device)
        self.w = torch.from_numpy(w).to(device)
        self.cs = torch.from_numpy(np.ascontiguousarray(cs, dtype=np.uint16).view(np.int16)
                                   .reshape(self.P, self.K)).to(device)

    @classmethod
    def from_tables(cls, rec, sz, w, cs, pb=None):
        """A layer over device tables already packed by pq_pack (rec uint8, sz
        and cs int16 bit patterns, w uint8, all on one CUDA device)."""
        self = cls.__new__(cls)
        self.rec, self.sz, self.w, self.cs = rec, sz, w, cs
        self.P, self.K, self.N = rec.shape[0], w.shape[1] * 2, w.shape[0]
        self.pb1, self.pb2 = pb if pb is not None else (self.N, self.N)
        return self

    def forward(self, x, y=None, stream=None):
        a, asg, rs = pq_rotate_quant(x, self.rec, self.cs, stream=stream)
        return pq_gemm(a, asg, rs, self.w, self.sz, self.pb1, self.pb2, y=y, stream=stream)

    __call__ = forward

    def make_graph(self, x_host, y_host, zero_copy=False):
        """One step as a CUDA graph on pinned host buffers x_host (bf16 [M, K])
        and y_host (bf16 [M, N]).  Returns a function that replays the step on
        the current stream; each replay reads whatever x_host holds then.  The
        device buffers live as long as the returned function.

        zero_copy=False: copy x_host to the device, the prologue and the GEMM,
        copy y back to y_host.  zero_copy=True: the prologue reads x straight
        from x_host and the GEMM writes y straight into y_host (page-locked
        host memory mapped at the same device address, checked with
        pq_check_device_access), so the bytes cross the host link inside the
        kernels and the step has no copy operations.

        The returned function owns a CUDA graph: release it (and anything that
        keeps it alive, such as a reference cycle) outside any stream capture.
        A graph destroyed while another global-mode capture is running
        invalidates that capture."""
        torch = _torch()
        dev = self.w.device
        M, K = x_host.shape
        G = K // 128
        if K != self.K or tuple(y_host.shape) != (M, self.N):
            raise PQError("make_graph: x_host must be [M, %d] and y_host [M, %d]" % (self.K, self.N))
        for t, what in ((x_host, "x_host"), (y_host, "y_host")):
            if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_pinned() or not t.is_contiguous():
                raise PQError("make_graph: %s must be a contiguous page-locked bf16 host tensor" % what)
            if zero_copy:
                pq_check_device_access(t)
        x_dev = None if zero_copy else torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        y_dev = None if zero_copy else torch.empty((M, self.N), dtype=torch.bfloat16, device=dev)
        a = torch.empty((self.P, M, K), dtype=torch.uint8, device=dev)
        asg = torch.empty((self.P, G, M), dtype=torch.float32, device=dev)
        rs = torch.empty((self.P, G, M), dtype=torch.float32, device=dev)

        if zero_copy:
            def body():
                L, st = lib(), _stream(None)
                _check(L.pq_rotate_quant(C.c_void_p(x_host.data_ptr()), M, K, K, self.P, _dptr(self.rec),
                                         _dptr(self.cs), _dptr(a), _dptr(asg), _dptr(rs), st), "pq_rotate_quant")
                _check(L.pq_gemm(_dptr(a), _dptr(asg), _dptr(rs), M, self.N, K, self.P, self.pb1, self.pb2,
                                 _dptr(self.w), _dptr(self.sz), C.c_void_p(y_host.data_ptr()), self.N, st),
                       "pq_gemm")
        else:
            def body():
                x_dev.copy_(x_host, non_blocking=True)
                pq_rotate_quant(x_dev, self.rec, self.cs, a=a, asg=asg, rs=rs)
                pq_gemm(a, asg, rs, self.w, self.sz, self.pb1, self.pb2, y=y_dev)
                y_host.copy_(y_dev, non_blocking=True)

        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            body()                                  # first run outside the capture
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            body()

        def replay():
            graph.replay()

        replay.buffers = (graph, x_dev, y_dev, a, asg, rs, x_host, y_host)
        return replay
