"""The C-ABI library loads and exports every entry point include/moe.h
declares; host-side argument checks work without a GPU."""
import ctypes
import os
import re

import pytest

import dropless_grouped_gemm_gb300 as M
from dropless_grouped_gemm_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return M.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "moe_grouped_mlp_fwd" in names and len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def test_version(L):
    assert "sm_103a" in M.version()


def test_host_argument_errors(L):
    vp = ctypes.c_void_p
    # E = 0, k > E, bad align: rejected before anything touches the GPU
    assert L.moe_grouped_mlp_fwd(None, None, 0, 0, 64, 64, None, None, 0, 0, None, None, None,
                                 None, None, None, None) == -3
    assert L.moe_grouped_mlp_fwd(None, None, 4, 128, 96, 64, None, None, 0, 0, None, None, None,
                                 None, None, None, None) == -3    # d not a multiple of 64
    assert L.moe_grouped_mlp_fwd(None, None, 4, 128, 64, 64, None, None, 7, 0, None, None, None,
                                 None, None, None, None) == -4    # bad act
    assert L.moe_grouped_mlp_fwd(None, None, 4, 128, 64, 64, None, None, 0, 2, None, None, None,
                                 None, None, None, None) == -1    # MXFP8 without its buffers
    assert L.moe_mx_quantize_weights(None, 4, 96, 128, None, None, None, None) == -3
    assert L.moe_mx_quantize(None, 64, 48, None, 2, None, None, None, None, None, None) == -3
    # tiled scales: widths in 128-column groups; at least one copy requested
    assert L.moe_mx_quantize_tiled(vp(16), 64, 96, vp(16), 2, vp(16), vp(16), None, None, vp(16),
                                   None) == -3
    assert L.moe_mx_quantize_tiled(vp(16), 64, 128, vp(16), 2, None, None, None, None, vp(16),
                                   None) == -1
    assert L.moe_mx_quantize_tiled(vp(16), 64, 128, vp(16), 2, vp(16), None, None, None, vp(16),
                                   None) == -1
    assert L.moe_route_offsets(None, 4, 3, 2, 1, 12, None, None, None, None, None, None, 0, None,
                               None) == -3                  # k > E
    assert L.moe_route_offsets(None, 4, 2, 8, 0, 12, None, None, None, None, None, None, 0, None,
                               None) == -3                  # align 0
    assert L.moe_permute(None, None, None, 4, 1, 100, 4, None, None) == -3
    # token-order permute: same size rules; both maps (row_of_pair only when T > 0)
    assert L.moe_permute_tokens(None, None, None, None, 4, 1, 100, 4, None, None) == -3
    assert L.moe_permute_tokens(vp(16), None, None, vp(16), 4, 1, 64, 4, vp(16), None) == -1
    assert L.moe_permute_tokens(vp(16), None, vp(16), None, 4, 1, 64, 4, vp(16), None) == -1
    assert L.moe_permute_tokens(vp(16), None, vp(16), vp(16), 4, 0, 64, 4, vp(16), None) == -3
    assert L.moe_permute_tokens(vp(8), None, vp(16), vp(16), 4, 1, 64, 4, vp(16), None) == -2
    assert L.moe_permute_tokens(None, None, None, None, 4, 1, 64, 0, None, None) == 0  # nothing to do
    assert L.moe_unpermute(vp(16), None, vp(16), 2, 1, 64, 4, None, None, None, None) == -1
    # MXFP8 backward: sizes need multiples of 128 (d, n) and 32 (M_cap); mx required
    assert L.moe_grouped_mlp_bwd_mx(None, None, None, vp(16), 4, 128, 192, 128, 0, 0, None, None,
                                    None, vp(16), vp(16), vp(16), None) == -3
    assert L.moe_grouped_mlp_bwd_mx(None, None, None, vp(16), 4, 100, 128, 128, 0, 0, None, None,
                                    None, vp(16), vp(16), vp(16), None) == -3
    assert L.moe_grouped_mlp_bwd_mx(None, None, None, vp(16), 4, 128, 128, 128, 0, 0, None, None,
                                    None, vp(16), vp(16), vp(16), None) == -1
    assert L.moe_mx_quantize_weights_rowwise(vp(16), 100, 128, None, 0, vp(16), vp(16), None) == -3
    # with routing offsets: rows must split into E experts of a multiple of 128 rows each
    assert L.moe_mx_quantize_weights_rowwise(vp(16), 384, 128, vp(16), 2, vp(16), vp(16), None) == -3
    assert L.moe_mx_quantize_weights_rowwise(vp(16), 384, 128, vp(16), 0, vp(16), vp(16), None) == -3
    assert L.moe_mx_quantize_weights_rowwise(vp(16), 512, 128, None, 3, None, vp(16), None) == -1


def test_accumulate_flag_host_checks(L):
    """MOE_FLAG_ACCUMULATE_DW is the backward flag (and, for the MXFP8
    backward alone, MOE_FLAG_MX_SEPARATE_DH_QUANT); an unknown bit is
    refused.  With no rows at all an accumulating backward has nothing to
    add and returns before any CUDA call (all pointers are dummies)."""
    vp = ctypes.c_void_p
    d = vp(256)
    bwd = lambda flags, M_cap: L.moe_grouped_mlp_bwd(d, d, d, d, d, 2, M_cap, 128, 128, d, d, 0,
                                                     flags, d, d, d, d, None, d, None)
    routed = lambda flags, M_cap: L.moe_grouped_mlp_bwd_routed(
        d, d, d, d, d, d, 2, M_cap, 128, 128, d, d, 0, flags, d, d, d, d, d, d, None, d, None)
    mxb = lambda flags, M_cap: L.moe_grouped_mlp_bwd_mx(d, d, d, d, 2, M_cap, 128, 128, 0, flags,
                                                         d, d, d, d, d, d, None)
    for f in (bwd, routed, mxb):
        assert f(16, 256) == -4
        assert f(M.FLAG_ACCUMULATE_DW | 1, 256) == -4
        assert f(M.FLAG_ACCUMULATE_DW, 0) == 0
    for f in (bwd, routed):
        assert f(M.FLAG_MX_SEPARATE_DH_QUANT, 256) == -4
    assert mxb(M.FLAG_ACCUMULATE_DW | M.FLAG_MX_SEPARATE_DH_QUANT, 0) == 0


def test_mx_bwd_workspace_too_small(L):
    """A workspace smaller than moe_mx_bwd_workspace_size is refused before
    any launch (all pointers are dummies: nothing is dereferenced)."""
    vp = ctypes.c_void_p
    need = M.mx_bwd_workspace_size(256, 128, 128, "swiglu")
    assert need >= 256 * (3 * 128 + 2 * 256)
    st = M.MxBwd(256, 256, 256, 256, 256, 256, 256, need - 1)
    assert L.moe_grouped_mlp_bwd_mx(vp(256), vp(256), vp(256), vp(256), 2, 256, 128, 128, 0, 0,
                                    ctypes.byref(st), vp(256), vp(256), vp(256), vp(256),
                                    vp(256), None) == -6


def test_workspace_size_host_only(L):
    assert M.route_workspace_size(4096, 8, 256) >= 8 * 256 * 4
    assert M.route_workspace_size(0, 1, 4) == 4 * 4


def test_header_compiles_as_c(tmp_path):
    """include/moe.h is a C ABI: it compiles as strict C99 (no C++ types or
    defaults leak into it), with every warning an error."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "use_moe.c"
    src.write_text('#include "moe.h"\n'
                   "int main(void) {\n"
                   "  moe_mx_bwd b;\n"
                   "  (void)b;\n"
                   "  return moe_version() != 0 ? 0 : 1;\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(root, "include"), "-c", str(src),
                        "-o", str(tmp_path / "use_moe.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_layer_workspace_size_is_the_larger_part(L):
    """moe_workspace_size: the routing layout's scratch, or the MXFP8
    backward's when that is larger and requested; host-only."""
    T, k, E, M_cap, d, n = 4096, 8, 256, 32768 + 256 * 31, 7168, 2048
    r = L.moe_route_workspace_size(T, k, E)
    m = L.moe_mx_bwd_workspace_size(M_cap, d, n, 0)
    assert r > 0 and m > r
    assert L.moe_workspace_size(T, k, E, M_cap, d, n, 0, 0) == r
    assert L.moe_workspace_size(T, k, E, M_cap, d, n, 0, M.FLAG_MXFP8) == m
    assert M.workspace_size(T, k, E, M_cap, d, n, "swiglu", mxfp8=True) == m
    assert L.moe_workspace_size(0, 0, 0, 0, 0, 0, 0, M.FLAG_MXFP8) == 0


def test_mx_bwd_workspace_layout(L):
    """moe_mx_bwd_workspace_layout: 11 sections, 256-byte aligned, in the
    documented order, sized as the documented shapes, ending within the
    workspace size; invalid sizes give 0; host-only."""
    M_cap, d, n = 1024, 256, 128
    for act, n1 in (("swiglu", 2 * n), ("srelu", n)):
        lay = M.mx_bwd_workspace_layout(M_cap, d, n, act)
        sizes = {"dy_q": M_cap * d, "dy_s": M_cap * d // 8, "dy_qT": M_cap * d,
                 "dy_sT": M_cap * d // 8, "x_qT": M_cap * d, "x_sT": M_cap * d // 8,
                 "a_sT": M_cap * n // 8, "dh_q": M_cap * n1, "dh_s": M_cap * n1 // 8,
                 "dh_qT": M_cap * n1, "dh_sT": M_cap * n1 // 8}
        names = list(M.MX_BWD_SECTIONS)
        assert lay["bytes"] == M.mx_bwd_workspace_size(M_cap, d, n, act)
        for a, b in zip(names, names[1:]):
            assert lay[a] % 256 == 0 and lay[b] >= lay[a] + sizes[a], (a, b)
        assert lay[names[0]] == 0 and lay[names[-1]] + sizes[names[-1]] <= lay["bytes"]
    offs = (ctypes.c_size_t * 11)()
    assert L.moe_mx_bwd_workspace_layout(64, 0, 128, 0, offs) == 0
    assert L.moe_mx_bwd_workspace_layout(64, 128, 128, 0, None) == 0
