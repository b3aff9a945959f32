"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a and loads, it exports every entry point include/mhc_seam.h declares,
and the argument checks reject bad calls before anything touches CUDA.  The
pointers below are fake addresses; every call here fails validation first."""
import ctypes as C
import subprocess

import pytest

from mhc_residual_seam_gb300 import binding as B

FAKE = 0x10000000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def L():
    return B.lib()


def test_exports_every_declared_symbol(L):
    names = B.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", B._build.LIB], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in nm.splitlines() if " T " in l}
    assert set(names) <= exported


def test_config_struct_layout_matches_c():
    assert C.sizeof(B.MhcConfig) == 40
    assert B.MhcConfig.spin_limit.offset == 24
    assert B.MhcConfig.projection.offset == 32
    assert B.MhcConfig.wave_split.offset == 36


def _seam(L, **over):
    T, H = over.pop("T", 4), over.pop("H", 64)
    args = dict(R=FAKE, Y=FAKE + 0x100000, post_prev=FAKE + 0x200000, comb_prev=FAKE + 0x300000,
                pre_prev=FAKE + 0x400000, fn=FAKE + 0x500000, fn_packed=None, bias=FAKE + 0x600000,
                alpha=FAKE + 0x700000, gamma=FAKE + 0x800000, eps=1e-6, T=T, H=H, out_mode=0,
                residual_out=FAKE + 0x900000, norm=FAKE + 0xA00000, codes=None, scales=None,
                pre_out=FAKE + 0xB00000, post_out=FAKE + 0xC00000, comb_out=FAKE + 0xD00000,
                ws=FAKE + 0xE00000, ws_bytes=1 << 30, cfg=None)
    args.update(over)
    a = args
    return L.mhc_seam(a["R"], a["Y"], a["post_prev"], a["comb_prev"], a["pre_prev"], a["fn"], a["fn_packed"],
                      a["bias"], a["alpha"], a["gamma"], a["eps"], a["T"], a["H"], a["out_mode"],
                      a["residual_out"], a["norm"], a["codes"], a["scales"], a["pre_out"], a["post_out"],
                      a["comb_out"], a["ws"], a["ws_bytes"], a["cfg"], None)


def test_shape_errors(L):
    assert _seam(L, T=-1) == -2
    assert _seam(L, H=0) == -2
    assert _seam(L, H=12) == -2                 # H % 8
    assert _seam(L, H=40, out_mode=1) == -2     # mxfp8 needs H % 32
    assert _seam(L, out_mode=7) == -10


def test_empty_input_is_ok_without_launch(L):
    assert _seam(L, T=0, R=None, Y=None, post_prev=None, ws=None) == 0
    assert L.mhc_last_launch_count() == 0


def test_incomplete_post_is_rejected(L):
    assert _seam(L, Y=None) == -4
    assert _seam(L, post_prev=None) == -4
    assert "post_prev" in L.mhc_last_error_string().decode()
    assert _seam(L, comb_prev=None) == -4        # Y and post without comb: not the identity form
    assert "identity form" in L.mhc_last_error_string().decode()


def test_identity_form_ignores_residual_out(L):
    # comb, Y and post all NULL: the identity form; residual_out may be NULL or
    # anything (it is not written), so the call gets as far as the workspace check
    ident = dict(comb_prev=None, Y=None, post_prev=None, ws_bytes=1)
    assert _seam(L, residual_out=None, **ident) == -5
    assert _seam(L, residual_out=FAKE + 16, **ident) == -5   # would alias R in the other forms
    assert _seam(L, comb_prev=None, Y=None, post_prev=None, pre_prev=None) == -1


def _unsh(L, **over):
    args = dict(R=FAKE, Y=FAKE + 0x100000, post_prev=FAKE + 0x200000, comb_prev=FAKE + 0x300000, fn=FAKE + 0x500000,
                fn_packed=None, bias=FAKE + 0x600000, alpha=FAKE + 0x700000, eps=1e-6, T=4, H=64, residual_out=FAKE + 0x900000,
                x_out=FAKE + 0xA00000, pre_out=FAKE + 0xB00000, post_out=FAKE + 0xC00000, comb_out=FAKE + 0xD00000,
                ws=FAKE + 0xE00000, ws_bytes=1 << 30, cfg=None)
    args.update(over)
    a = args
    return L.mhc_seam_unshifted(a["R"], a["Y"], a["post_prev"], a["comb_prev"], a["fn"], a["fn_packed"], a["bias"],
                                a["alpha"],
                                a["eps"], a["T"], a["H"], a["residual_out"], a["x_out"], a["pre_out"], a["post_out"],
                                a["comb_out"], a["ws"], a["ws_bytes"], a["cfg"], None)


def test_unshifted_argument_rules(L):
    assert _unsh(L, T=0, R=None, ws=None) == 0
    assert _unsh(L, x_out=None) == -1
    assert _unsh(L, Y=None) == -4
    assert _unsh(L, comb_prev=None) == -4
    assert _unsh(L, x_out=FAKE + 0x100000) == -9          # x over Y
    # the split path keeps R' (8 bytes per element) in shared memory: a tile the
    # delayed seam takes is refused here
    big = B.MhcConfig(block_m=32, cols_per_cta=640)
    assert _unsh(L, H=5120, cfg=C.byref(big)) == -10
    assert _seam(L, H=5120, cfg=C.byref(big), ws_bytes=1) == -5
    # the streaming path's workspace: the status header, the split last round's 776 KiB and
    # the item scheduler's 128-byte counter row
    assert L.mhc_workspace_bytes_unshifted(4096, 5120, None) == L.mhc_workspace_bytes(4096, 5120, None) == 256 + 776 * 1024 + 128
    p1 = B.MhcConfig(path=1)
    need = L.mhc_workspace_bytes_unshifted(4096, 5120, C.byref(p1))
    assert need > 256 and _unsh(L, T=4096, H=5120, cfg=C.byref(p1), ws_bytes=need - 1) == -5


def test_null_and_alignment(L):
    assert _seam(L, gamma=None) == -1
    assert _seam(L, out_mode=1) == -1           # mxfp8 without codes/scales
    assert _seam(L, R=FAKE + 2) == -3
    assert _seam(L, norm=FAKE + 0xA00008) == -3
    assert _seam(L, bias=FAKE + 0x600002) == -3


def test_alias_rules(L):
    # residual_out partly overlapping R is rejected; exactly R is allowed (in place)
    assert _seam(L, residual_out=FAKE + 16) == -9
    assert _seam(L, norm=FAKE + 0x100000) == -9  # norm over Y
    assert _seam(L, pre_out=FAKE + 0xC00000) == -9  # two outputs overlap


def test_workspace_rules(L):
    need = L.mhc_workspace_bytes(4, 64, None)
    assert need >= 256
    assert _seam(L, ws_bytes=need - 1) == -5
    assert _seam(L, ws=None) == -5
    assert L.mhc_workspace_init(None, 1024, None) == -5


def test_config_validation(L):
    for bad in (dict(path=5), dict(path=-1), dict(block_m=3), dict(block_m=64), dict(cols_per_cta=48), dict(spin_limit=-1),
                dict(sinkhorn_iters=-2), dict(amax_floor=-1.0), dict(projection=3), dict(wave_split=-1),
                dict(wave_split=65)):
        cfg = B.MhcConfig(**bad)
        assert _seam(L, cfg=C.byref(cfg)) == -10, bad
    cfg = B.MhcConfig(path=3, projection=1)     # clusters of 16 run the tcgen05 projection only
    assert _seam(L, H=5120, fn_packed=FAKE + 0xF00000, cfg=C.byref(cfg)) == -10


def test_workspace_grows_with_tokens_and_columns(L):
    p1 = B.MhcConfig(path=1)
    a = L.mhc_workspace_bytes(4, 5120, C.byref(p1))      # split path forced
    b = L.mhc_workspace_bytes(64, 5120, C.byref(p1))
    c = L.mhc_workspace_bytes(1024, 5120, None)          # streaming path: status word + split last round
    d = L.mhc_workspace_bytes(1024, 5120, C.byref(p1))
    stream = 256 + 776 * 1024 + 128
    assert 256 < a < b < d and c == stream
    # small T: the automatic policy's workspace covers both paths it may take
    # (the split path without fn_packed, clusters of 16 with it)
    assert L.mhc_workspace_bytes(4, 5120, None) == max(a, stream)
    p3 = B.MhcConfig(path=3)
    assert L.mhc_workspace_bytes(4, 5120, C.byref(p3)) == stream
    cfg = B.MhcConfig(block_m=8, cols_per_cta=64)
    assert L.mhc_workspace_bytes(64, 5120, C.byref(cfg)) == 256 + 8 * (((64 + 128 + 80 * 8 * 128) + 255) // 256 * 256)


def test_packed_fn_and_quant_arg_checks(L):
    assert L.mhc_packed_fn_bytes(5120) == 48 * 4 * 5120 * 2
    assert L.mhc_pack_fn(None, FAKE, 64, None) == -1
    assert L.mhc_pack_fn(FAKE, FAKE + 0x100000, 12, None) == -2
    assert L.mhc_quant_ue8m0(FAKE, 4, 40, 0.0, FAKE + 0x100000, FAKE + 0x200000, None) == -2
    assert L.mhc_quant_ue8m0(FAKE + 8, 4, 64, 0.0, FAKE + 0x100000, FAKE + 0x200000, None) == -3
    assert L.mhc_quant_ue8m0(FAKE, 0, 64, 0.0, None, None, None) == 0
    assert L.mhc_copy(FAKE, FAKE + 8, 64, None) == -3
    assert L.mhc_copy(FAKE, FAKE + 16, 64, None) == -9
