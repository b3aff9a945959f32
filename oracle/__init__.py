"""ctypes front end of the seam oracle -- TEST INFRASTRUCTURE ONLY.

The oracle (``mhc_oracle.c``) is a plain, single-threaded double-precision CPU
restatement of the delayed mHC seam.  Only the test-suite, the smoke check and
the benchmark's CPU-baseline leg may import this package; the product path
never does.  It shares no code with the CUDA library.

Functions mirror the C entry points and take/return numpy arrays (bf16 values
travel as their uint16 bit patterns).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libmhc_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc -O2 (no fast-math) into oracle/_build."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = bind(C.CDLL(build()))
    return _lib


def bind(cdll):
    """Declare the C signatures on a loaded oracle library."""
    L = cdll
    P = C.c_void_p
    L.mhc_oracle_bf16_rne.restype = C.c_uint16
    L.mhc_oracle_bf16_rne.argtypes = [C.c_double]
    L.mhc_oracle_bf16_to_double.restype = C.c_double
    L.mhc_oracle_bf16_to_double.argtypes = [C.c_uint16]
    L.mhc_oracle_e4m3_rne_satfinite.restype = C.c_uint8
    L.mhc_oracle_e4m3_rne_satfinite.argtypes = [C.c_double]
    L.mhc_oracle_ue8m0_exponent.restype = C.c_int
    L.mhc_oracle_ue8m0_exponent.argtypes = [C.c_double, C.c_double]
    L.mhc_oracle_quant_ue8m0.restype = C.c_int
    L.mhc_oracle_quant_ue8m0.argtypes = [P, C.c_int64, C.c_int, C.c_double, P, P]
    L.mhc_oracle_e4m3_decode.restype = C.c_double
    L.mhc_oracle_e4m3_decode.argtypes = [C.c_uint8]
    L.mhc_oracle_grid_ue8m0.restype = C.c_int
    L.mhc_oracle_grid_ue8m0.argtypes = [P, C.c_int64, C.c_int, C.c_double, P]
    L.mhc_oracle_sinkhorn.restype = None
    L.mhc_oracle_sinkhorn.argtypes = [C.c_int, P, C.c_int]
    L.mhc_oracle_sigmoid.restype = C.c_double
    L.mhc_oracle_sigmoid.argtypes = [C.c_double]
    L.mhc_oracle_seam.restype = C.c_int
    L.mhc_oracle_seam.argtypes = [C.c_int64, C.c_int] + [P] * 9 + [C.c_double, C.c_int, C.c_int] + [P] * 7
    L.mhc_oracle_seam_unshifted.restype = C.c_int
    L.mhc_oracle_seam_unshifted.argtypes = [C.c_int64, C.c_int] + [P] * 7 + [C.c_double, C.c_int] + [P] * 5
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _u16(a) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor or of a uint16 array."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def _f32(a) -> np.ndarray:
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def bf16_rne(v: float) -> int:
    return int(lib().mhc_oracle_bf16_rne(float(v)))


def bf16_to_float(b: int) -> float:
    return float(lib().mhc_oracle_bf16_to_double(int(b)))


def e4m3(v: float) -> int:
    return int(lib().mhc_oracle_e4m3_rne_satfinite(float(v)))


def ue8m0_exponent(amax: float, amax_floor: float = 1e-10) -> int:
    return int(lib().mhc_oracle_ue8m0_exponent(float(amax), float(amax_floor)))


def sigmoid(z: float) -> float:
    return float(lib().mhc_oracle_sigmoid(float(z)))


def sinkhorn(M: np.ndarray, iters: int = 20) -> np.ndarray:
    """Sinkhorn rounds on each n x n matrix of ``M`` (shape [..., n, n])."""
    M = np.array(M, dtype=np.float64, copy=True)
    n = M.shape[-1]
    flat = M.reshape(-1, n, n)
    for b in range(flat.shape[0]):
        m = np.ascontiguousarray(flat[b])
        lib().mhc_oracle_sinkhorn(n, _ptr(m), int(iters))
        flat[b] = m
    return flat.reshape(M.shape)


def carried_gates(pre_logits, post_logits, comb_logits, iters: int = 20):
    """Carried-gate inputs from U(-1,1) draws, in the form the seam itself
    emits: pre = sigmoid, post = 2 sigmoid, comb = Sinkhorn20(exp(.)), fp32."""
    sig = np.vectorize(sigmoid, otypes=[np.float64])
    pre = sig(np.asarray(pre_logits, np.float64)).astype(np.float32)
    post = (2.0 * sig(np.asarray(post_logits, np.float64))).astype(np.float32)
    comb = sinkhorn(np.exp(np.asarray(comb_logits, np.float64)), iters).astype(np.float32)
    return pre, post, comb


def quant_ue8m0(x, amax_floor: float = 1e-10):
    """Per-32 ue8m0 quantisation of bf16 rows: returns (codes u8 [rows,H],
    scales u8 [rows,H/32])."""
    xb = _u16(x)
    rows, H = xb.shape
    codes = np.zeros((rows, H), np.uint8)
    scales = np.zeros((rows, H // 32), np.uint8)
    rc = lib().mhc_oracle_quant_ue8m0(_ptr(xb), rows, H, float(amax_floor), _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("H must be a multiple of 32")
    return codes, scales


def e4m3_decode(code: int) -> float:
    """Value of one e4m3fn code (NaN for 0x7F / 0xFF)."""
    return float(lib().mhc_oracle_e4m3_decode(int(code)))


def grid_ue8m0(x, amax_floor: float = 1e-10) -> np.ndarray:
    """fp8_grid output of bf16 rows: per 32-group, bf16(decode(code) * 2^e) as
    uint16 bits [rows, H]."""
    xb = _u16(x)
    rows, H = xb.shape
    grid = np.zeros((rows, H), np.uint16)
    rc = lib().mhc_oracle_grid_ue8m0(_ptr(xb), rows, H, float(amax_floor), _ptr(grid))
    if rc != 0:
        raise ValueError("H must be a multiple of 32")
    return grid


def seam(R, Y, post_prev, comb_prev, pre_prev, fn, bias, alpha, gamma, eps: float,
         sinkhorn_iters: int = 20, rprime_unrounded: bool = False, want_x: bool = False) -> dict:
    """Run the oracle seam.  bf16 inputs may be torch bf16 tensors or uint16
    bit arrays; fp32 inputs may be tensors or arrays.  Returns a dict with
    ``residual_out`` [T,4,H] and ``norm`` [T,H] as uint16 bits, ``pre``,
    ``post`` [T,4], ``comb`` [T,4,4], ``rstd`` [T,2] in float64 and
    optionally ``x`` [T,H] float64.  ``comb_prev`` None (with ``Y`` and
    ``post_prev`` None) is the identity form of the first block: R' = R."""
    Rb = _u16(R)
    T, n, H = Rb.shape
    assert n == 4
    Yb = None if Y is None else _u16(Y)
    post_a, comb_a, pre_a = _f32(post_prev), _f32(comb_prev), _f32(pre_prev)
    fn_a, bias_a, alpha_a = _f32(fn), _f32(bias), _f32(alpha)
    gb = _u16(gamma)
    out = {
        "residual_out": np.zeros((T, 4, H), np.uint16),
        "norm": np.zeros((T, H), np.uint16),
        "pre": np.zeros((T, 4)),
        "post": np.zeros((T, 4)),
        "comb": np.zeros((T, 4, 4)),
        "rstd": np.zeros((T, 2)),
    }
    x = np.zeros((T, H)) if want_x else None
    rc = lib().mhc_oracle_seam(T, H, _ptr(Rb), _ptr(Yb), _ptr(post_a), _ptr(comb_a), _ptr(pre_a),
                               _ptr(fn_a), _ptr(bias_a), _ptr(alpha_a), _ptr(gb), float(eps),
                               int(sinkhorn_iters), int(bool(rprime_unrounded)),
                               _ptr(out["residual_out"]), _ptr(out["norm"]), _ptr(out["pre"]),
                               _ptr(out["post"]), _ptr(out["comb"]), _ptr(out["rstd"]), _ptr(x))
    if rc != 0:
        raise ValueError("oracle rejected the inputs (NULL operand, half-present post inputs, or Y without comb)")
    if want_x:
        out["x"] = x
    return out


def seam_unshifted(R, Y, post_prev, comb_prev, fn, bias, alpha, eps: float, sinkhorn_iters: int = 20) -> dict:
    """The unshifted ordering: post-mix with the carried comb and post, gates
    from R', and the layer input x = sum_i pre[i] R'[i] with the fresh pre,
    bf16 with no norm.  Returns ``residual_out`` [T,4,H] and ``x`` [T,H] as
    uint16 bits and ``pre``, ``post`` [T,4], ``comb`` [T,4,4] in float64."""
    Rb = _u16(R)
    T, n, H = Rb.shape
    assert n == 4
    Yb = None if Y is None else _u16(Y)
    post_a, comb_a = _f32(post_prev), _f32(comb_prev)
    fn_a, bias_a, alpha_a = _f32(fn), _f32(bias), _f32(alpha)
    out = {
        "residual_out": np.zeros((T, 4, H), np.uint16),
        "x": np.zeros((T, H), np.uint16),
        "pre": np.zeros((T, 4)),
        "post": np.zeros((T, 4)),
        "comb": np.zeros((T, 4, 4)),
    }
    rc = lib().mhc_oracle_seam_unshifted(T, H, _ptr(Rb), _ptr(Yb), _ptr(post_a), _ptr(comb_a), _ptr(fn_a),
                                         _ptr(bias_a), _ptr(alpha_a), float(eps), int(sinkhorn_iters),
                                         _ptr(out["residual_out"]), _ptr(out["x"]), _ptr(out["pre"]),
                                         _ptr(out["post"]), _ptr(out["comb"]))
    if rc != 0:
        raise ValueError("oracle rejected the inputs (NULL operand, half-present post inputs, or Y without comb)")
    return out
