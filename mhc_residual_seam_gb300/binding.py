"""ctypes binding of libmhcseam (include/mhc_seam.h): argument marshalling only.

Every function has the name of its C entry point and takes torch tensors
(device memory) plus plain numbers; it passes ``data_ptr()`` values and the
CUDA stream handle through, and raises ``MhcError`` on a non-zero status.
There is no fallback: if the library cannot be built or loaded, the first call
raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re

from . import build as _build

MHC_OUT_BF16 = 0
MHC_OUT_MXFP8 = 1
MHC_OUT_FP8_GRID = 2
STATUS_NAMES = {
    0: "MHC_OK", -1: "MHC_ERR_NULL", -2: "MHC_ERR_SHAPE", -3: "MHC_ERR_ALIGN", -4: "MHC_ERR_INCOMPLETE_POST",
    -5: "MHC_ERR_WORKSPACE", -6: "MHC_ERR_CAPTURE", -7: "MHC_ERR_TIMEOUT", -8: "MHC_ERR_CUDA", -9: "MHC_ERR_ALIAS",
    -10: "MHC_ERR_CONFIG",
}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mhc_seam.h")


class MhcError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class MhcConfig(C.Structure):
    """mhc_config: zero in a field means the policy decides."""
    _fields_ = [("path", C.c_int), ("block_m", C.c_int), ("cols_per_cta", C.c_int), ("sinkhorn_iters", C.c_int),
                ("amax_floor", C.c_float), ("spin_limit", C.c_longlong), ("projection", C.c_int),
                ("wave_split", C.c_int)]


_lib = None


def lib():
    """Load (building first if needed) the in-tree libmhcseam.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P, I64, I = C.c_void_p, C.c_int64, C.c_int
        L.mhc_workspace_bytes.restype = C.c_size_t
        L.mhc_workspace_bytes.argtypes = [I64, I, P]
        L.mhc_workspace_bytes_unshifted.restype = C.c_size_t
        L.mhc_workspace_bytes_unshifted.argtypes = [I64, I, P]
        L.mhc_workspace_init.restype = I
        L.mhc_workspace_init.argtypes = [P, C.c_size_t, P]
        L.mhc_check_status.restype = I
        L.mhc_check_status.argtypes = [P, P]
        L.mhc_packed_fn_bytes.restype = C.c_size_t
        L.mhc_packed_fn_bytes.argtypes = [I]
        L.mhc_pack_fn.restype = I
        L.mhc_pack_fn.argtypes = [P, P, I, P]
        L.mhc_seam.restype = I
        L.mhc_seam.argtypes = [P] * 10 + [C.c_float, I64, I, I] + [P] * 7 + [P, C.c_size_t, P, P]
        L.mhc_seam_unshifted.restype = I
        L.mhc_seam_unshifted.argtypes = [P] * 8 + [C.c_float, I64, I] + [P] * 6 + [C.c_size_t, P, P]
        L.mhc_seam_noalloc.restype = I
        L.mhc_seam_noalloc.argtypes = [P] * 9 + [C.c_float, I64, I, I] + [P] * 7 + [P, P]
        L.mhc_noalloc_check_status.restype = I
        L.mhc_noalloc_check_status.argtypes = [P]
        L.mhc_quant_ue8m0.restype = I
        L.mhc_quant_ue8m0.argtypes = [P, I64, I, C.c_float, P, P, P]
        L.mhc_copy.restype = I
        L.mhc_copy.argtypes = [P, P, C.c_size_t, P]
        L.mhc_last_launch_count.restype = I
        L.mhc_last_launch_count.argtypes = []
        L.mhc_last_wave_parts.restype = I
        L.mhc_last_wave_parts.argtypes = []
        L.mhc_last_error_string.restype = C.c_char_p
        L.mhc_last_error_string.argtypes = []
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the entry points the C header declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mhc_[a-z0-9_]+)\s*\(", src)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != 0:
        raise MhcError(rc, lib().mhc_last_error_string().decode())


def _cfg(cfg):
    if cfg is None:
        return None
    if isinstance(cfg, dict):
        cfg = MhcConfig(**cfg)
    return C.byref(cfg)


def mhc_workspace_bytes(T: int, H: int, cfg=None) -> int:
    return int(lib().mhc_workspace_bytes(int(T), int(H), _cfg(cfg)))


def mhc_workspace_init(ws, stream=None) -> None:
    _check(lib().mhc_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def mhc_check_status(ws, stream=None) -> None:
    _check(lib().mhc_check_status(_ptr(ws), _stream(stream)))


def mhc_packed_fn_bytes(H: int) -> int:
    return int(lib().mhc_packed_fn_bytes(int(H)))


def mhc_pack_fn(fn, fn_packed, stream=None) -> None:
    H = fn.shape[0] // 4
    _check(lib().mhc_pack_fn(_ptr(fn), _ptr(fn_packed), H, _stream(stream)))


def mhc_seam(R, Y, post_prev, comb_prev, pre_prev, fn, fn_packed, bias, alpha, gamma, eps: float, out_mode: int,
             residual_out, norm, fp8_codes, e8m0_scales, pre_out, post_out, comb_out, workspace, cfg=None,
             stream=None, T: int | None = None, H: int | None = None) -> None:
    """One seam call; T and H default to R's shape [T, 4, H]."""
    if T is None:
        T = R.shape[0]
    if H is None:
        H = R.shape[-1]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().mhc_seam(_ptr(R), _ptr(Y), _ptr(post_prev), _ptr(comb_prev), _ptr(pre_prev), _ptr(fn),
                          _ptr(fn_packed), _ptr(bias), _ptr(alpha), _ptr(gamma), float(eps), int(T), int(H),
                          int(out_mode), _ptr(residual_out), _ptr(norm), _ptr(fp8_codes), _ptr(e8m0_scales),
                          _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _ptr(workspace), ws_bytes, _cfg(cfg),
                          _stream(stream)))


def mhc_seam_unshifted(R, Y, post_prev, comb_prev, fn, fn_packed, bias, alpha, eps: float, residual_out, x_out,
                       pre_out, post_out, comb_out, workspace, cfg=None, stream=None, T: int | None = None,
                       H: int | None = None) -> None:
    """One seam call in the unshifted ordering (x with the fresh pre, no norm);
    T and H default to R's shape [T, 4, H]."""
    if T is None:
        T = R.shape[0]
    if H is None:
        H = R.shape[-1]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().mhc_seam_unshifted(_ptr(R), _ptr(Y), _ptr(post_prev), _ptr(comb_prev), _ptr(fn), _ptr(fn_packed),
                                    _ptr(bias),
                                    _ptr(alpha), float(eps), int(T), int(H), _ptr(residual_out), _ptr(x_out),
                                    _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _ptr(workspace), ws_bytes,
                                    _cfg(cfg), _stream(stream)))


def mhc_workspace_bytes_unshifted(T: int, H: int, cfg=None) -> int:
    return int(lib().mhc_workspace_bytes_unshifted(int(T), int(H), _cfg(cfg)))


def mhc_seam_noalloc(R, Y, post_prev, comb_prev, pre_prev, fn, bias, alpha, gamma, eps: float, out_mode: int,
                     residual_out, norm, fp8_codes, e8m0_scales, pre_out, post_out, comb_out, cfg=None,
                     stream=None, T: int | None = None, H: int | None = None) -> None:
    """mhc_seam on the split path with the library's own static scratch, for
    callers that cannot allocate device memory (no workspace argument)."""
    if T is None:
        T = R.shape[0]
    if H is None:
        H = R.shape[-1]
    _check(lib().mhc_seam_noalloc(_ptr(R), _ptr(Y), _ptr(post_prev), _ptr(comb_prev), _ptr(pre_prev), _ptr(fn),
                                  _ptr(bias), _ptr(alpha), _ptr(gamma), float(eps), int(T), int(H), int(out_mode),
                                  _ptr(residual_out), _ptr(norm), _ptr(fp8_codes), _ptr(e8m0_scales),
                                  _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _cfg(cfg), _stream(stream)))


def mhc_noalloc_check_status(stream=None) -> None:
    _check(lib().mhc_noalloc_check_status(_stream(stream)))


def mhc_quant_ue8m0(x, codes, scales, amax_floor: float = 0.0, stream=None) -> None:
    rows, H = x.shape
    _check(lib().mhc_quant_ue8m0(_ptr(x), rows, H, float(amax_floor), _ptr(codes), _ptr(scales), _stream(stream)))


def mhc_copy(src, dst, nbytes: int | None = None, stream=None) -> None:
    if nbytes is None:
        nbytes = src.numel() * src.element_size()
    _check(lib().mhc_copy(_ptr(src), _ptr(dst), int(nbytes), _stream(stream)))


def mhc_last_launch_count() -> int:
    return int(lib().mhc_last_launch_count())


def mhc_last_wave_parts() -> int:
    return int(lib().mhc_last_wave_parts())


def mhc_last_error_string() -> str:
    return lib().mhc_last_error_string().decode()


# ----------------------------------------------------------- allocation ----
def alloc_outputs(T: int, H: int, out_mode: int, device, cfg=None, unshifted: bool = False) -> dict:
    """Output tensors and an initialised workspace for one seam call (with
    ``unshifted``, for mhc_seam_unshifted: ``norm`` then receives x)."""
    import torch
    o = {
        "residual_out": torch.empty((T, 4, H), dtype=torch.bfloat16, device=device),
        "norm": torch.empty((T, H), dtype=torch.bfloat16, device=device),
        # mxfp8: e4m3 codes; fp8_grid: the bf16 grid (written through the same argument)
        "fp8_codes": (torch.empty((T, H), dtype=torch.uint8, device=device) if out_mode == MHC_OUT_MXFP8 else
                      torch.empty((T, H), dtype=torch.bfloat16, device=device) if out_mode == MHC_OUT_FP8_GRID
                      else None),
        "e8m0_scales": torch.empty((T, H // 32), dtype=torch.uint8, device=device) if out_mode == MHC_OUT_MXFP8 else None,
        "pre_out": torch.empty((T, 4), dtype=torch.float32, device=device),
        "post_out": torch.empty((T, 4), dtype=torch.float32, device=device),
        "comb_out": torch.empty((T, 4, 4), dtype=torch.float32, device=device),
    }
    nbytes = mhc_workspace_bytes_unshifted(T, H, cfg) if unshifted else mhc_workspace_bytes(T, H, cfg)
    o["workspace"] = torch.empty((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=device)
    mhc_workspace_init(o["workspace"])
    return o
