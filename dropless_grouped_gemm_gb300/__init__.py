"""GB300-native dropless MoE expert MLP: Python binding of libmoe.

Argument marshalling only: every step of the path runs in libmoe's CUDA
kernels (``csrc/``).  PyTorch supplies device memory and the current CUDA
stream.  There is no CPU fallback: if ``libmoe.so`` is missing or a call
fails, an exception is raised.

Functions mirror the C ABI in ``include/moe.h``:

    route_offsets      -> moe_route_offsets
    permute            -> moe_permute (moe_permute_tokens with row_of_pair)
    unpermute          -> moe_unpermute
    grouped_mlp_fwd    -> moe_grouped_mlp_fwd
    grouped_mlp_bwd    -> moe_grouped_mlp_bwd
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "ACT", "FLAG_SAVE_H", "DEV_BAD_EXPERT", "DEV_OVERFLOW", "DEV_TIMEOUT", "DEV_BAD_OFFSETS",
    "lib", "lib_path", "version", "last_launch_count", "route_workspace_size", "workspace_size",
    "route_offsets",
    "router_topk",
    "permute", "unpermute", "grouped_mlp_fwd", "grouped_mlp_bwd", "MoeError",
    "FLAG_MXFP8", "MxFwd", "mx_quantize_weights", "mx_quantize", "mx_buffers",
    "MxBwd", "mx_quantize_weights_rowwise", "mx_quantize_tiled", "mx_bwd_workspace_size", "grouped_mlp_bwd_mx",
    "grouped_mlp_bwd_routed", "router_grad_rows", "mx_quantize_weights2", "FLAG_ACCUMULATE_DW",
    "grouped_gemm", "activation", "activation_bwd", "grouped_mlp_fwd_gather",
    "grouped_mlp_bwd_routed_gather", "route_logits", "FLAG_MX_SEPARATE_DH_QUANT",
    "mx_bwd_workspace_layout", "set_pair_mma",
]

ACT = {"swiglu": 0, "geglu": 1, "srelu": 2}
FLAG_SAVE_H = 1
FLAG_MXFP8 = 2
FLAG_ACCUMULATE_DW = 4
FLAG_MX_SEPARATE_DH_QUANT = 8
DEV_BAD_EXPERT, DEV_OVERFLOW, DEV_TIMEOUT, DEV_BAD_OFFSETS = 1, 2, 4, 8
_RC = {-1: "MOE_E_NULL", -2: "MOE_E_ALIGN", -3: "MOE_E_SIZE", -4: "MOE_E_ARG",
       -5: "MOE_E_CUDA", -6: "MOE_E_WORKSPACE"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class MoeError(RuntimeError):
    pass


class MxFwd(ctypes.Structure):
    """moe_mx_fwd: MXFP8 buffers of the forward (device pointers)."""
    _fields_ = [("w2_q", ctypes.c_void_p), ("w2_s", ctypes.c_void_p), ("a_q", ctypes.c_void_p),
                ("a_s", ctypes.c_void_p), ("a_qT", ctypes.c_void_p), ("a_sT", ctypes.c_void_p),
                ("y_q", ctypes.c_void_p), ("y_s", ctypes.c_void_p)]


class MxBwd(ctypes.Structure):
    """moe_mx_bwd: MXFP8 operands and workspace of the backward (device pointers)."""
    _fields_ = [("a_qT", ctypes.c_void_p), ("a_sT", ctypes.c_void_p), ("w2_q", ctypes.c_void_p),
                ("w2_s", ctypes.c_void_p), ("w1_q", ctypes.c_void_p), ("w1_s", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
                ("dx_q", ctypes.c_void_p), ("dx_s", ctypes.c_void_p)]


def lib_path() -> str:
    return os.path.join(_HERE, "libmoe.so")


def lib():
    """The loaded libmoe (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        p = lib_path()
        if not os.path.exists(p):
            raise MoeError(f"{p} is missing: build it with dropless_grouped_gemm_gb300.build.build()")
        L = ctypes.CDLL(p)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_version.restype = ctypes.c_char_p
        L.moe_version.argtypes = []
        L.moe_last_launch_count.restype = i32
        L.moe_last_launch_count.argtypes = []
        L.moe_router_topk.restype = i32
        L.moe_router_topk.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_route_logits.restype = i32
        L.moe_route_logits.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                       sz, vp, vp]
        L.moe_route_workspace_size.restype = sz
        L.moe_route_workspace_size.argtypes = [i32, i32, i32]
        L.moe_route_offsets.restype = i32
        L.moe_route_offsets.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz,
                                        vp, vp]
        L.moe_permute.restype = i32
        L.moe_permute.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
        L.moe_permute_tokens.restype = i32
        L.moe_permute_tokens.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]
        L.moe_unpermute.restype = i32
        L.moe_unpermute.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.moe_grouped_mlp_fwd.restype = i32
        L.moe_grouped_mlp_fwd.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, i32, i32, vp, vp, vp,
                                          vp, vp, vp, vp]
        L.moe_mx_quantize_weights.restype = i32
        L.moe_mx_quantize_weights.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.moe_mx_quantize.restype = i32
        L.moe_mx_quantize.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_set_launch_events.restype = i32
        L.moe_set_launch_events.argtypes = [vp, i32]
        L.moe_launch_events_used.restype = i32
        L.moe_launch_events_used.argtypes = []
        L.moe_grouped_mlp_bwd.restype = i32
        L.moe_grouped_mlp_bwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, i32, i32,
                                          vp, vp, vp, vp, vp, vp, vp]
        L.moe_mx_quantize_weights2.restype = i32
        L.moe_mx_quantize_weights2.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.moe_mx_quantize_tiled.restype = i32
        L.moe_mx_quantize_tiled.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_mx_quantize_weights_rowwise.restype = i32
        L.moe_mx_quantize_weights_rowwise.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp]
        L.moe_mx_bwd_workspace_size.restype = sz
        L.moe_mx_bwd_workspace_size.argtypes = [i32, i32, i32, i32]
        L.moe_set_pair_mma.restype = i32
        L.moe_set_pair_mma.argtypes = [i32]
        L.moe_mx_bwd_workspace_layout.restype = sz
        L.moe_mx_bwd_workspace_layout.argtypes = [i32, i32, i32, i32, vp]
        L.moe_workspace_size.restype = sz
        L.moe_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
        L.moe_grouped_mlp_bwd_mx.restype = i32
        L.moe_grouped_mlp_bwd_mx.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp,
                                             vp, vp, vp, vp, vp]
        L.moe_grouped_mlp_bwd_routed.restype = i32
        L.moe_grouped_mlp_bwd_routed.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp,
                                                 vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_grouped_mlp_fwd_gather.restype = i32
        L.moe_grouped_mlp_fwd_gather.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, i32, vp, vp,
                                                 i32, i32, vp, vp, vp, vp, vp, vp]
        L.moe_grouped_mlp_bwd_routed_gather.restype = i32
        L.moe_grouped_mlp_bwd_routed_gather.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, i32, i32,
                                                        i32, i32, vp, vp, i32, i32, vp, vp, vp, vp,
                                                        vp, vp, vp, vp, vp]
        L.moe_grouped_gemm.restype = i32
        L.moe_grouped_gemm.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp, vp]
        L.moe_activation.restype = i32
        L.moe_activation.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp]
        L.moe_activation_bwd.restype = i32
        L.moe_activation_bwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
        L.moe_router_grad_rows.restype = i32
        L.moe_router_grad_rows.argtypes = [vp, i32, vp, i32, i32, i32, vp, vp]
        L.moe_selftest_bounded_wait.restype = i32
        L.moe_selftest_bounded_wait.argtypes = [i32, vp, vp, vp]
        _LIB = L
    return _LIB


def version() -> str:
    return lib().moe_version().decode()


def last_launch_count() -> int:
    return int(lib().moe_last_launch_count())


def _check(rc: int, what: str):
    if rc != 0:
        raise MoeError(f"{what} failed: {_RC.get(rc, rc)}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, ndim=None):
    if t is None:
        return
    if not t.is_cuda:
        raise MoeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MoeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MoeError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise MoeError(f"{name} must have {ndim} dims")


def _err_word(err, device):
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=device)
    _need(err, torch.int32, "err")
    return err


def router_topk(logits: torch.Tensor, k: int, stream=None):
    """Top-k experts per token and their softmax weights (moe_router_topk).
    Returns (topk_idx int32 [T, k], probs float32 [T, k])."""
    _need(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    probs = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    rc = lib().moe_router_topk(_ptr(logits), T, E, k, _ptr(idx), _ptr(probs), _stream(stream))
    _check(rc, "moe_router_topk")
    return idx, probs


def route_workspace_size(T: int, k: int, E: int) -> int:
    return int(lib().moe_route_workspace_size(T, k, E))


def workspace_size(T: int, k: int, E: int, M_cap: int, d: int, n: int, act: str = "swiglu",
                   mxfp8: bool = False) -> int:
    """Device scratch for one layer's calls (moe_workspace_size): the routing
    layout's and, with ``mxfp8``, the MXFP8 backward's, one buffer for both."""
    return int(lib().moe_workspace_size(T, k, E, M_cap, d, n, ACT[act],
                                        FLAG_MXFP8 if mxfp8 else 0))


def route_offsets(topk_idx: torch.Tensor, E: int, align: int = 1, M_cap: int | None = None,
                  err: torch.Tensor | None = None, out: dict | None = None,
                  workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Routing layout on the device (see moe_route_offsets).  Returns a dict
    of device tensors: counts, offsets, row_of_pair, pair_of_row, true_total,
    err."""
    _need(topk_idx, torch.int32, "topk_idx", 2)
    T, k = topk_idx.shape
    if M_cap is None:
        M_cap = T * k + E * (align - 1)
    dev = topk_idx.device
    o = out if out is not None else {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "row_of_pair": torch.empty(T * k, dtype=torch.int32, device=dev),
        "pair_of_row": torch.empty(M_cap, dtype=torch.int32, device=dev),
        "true_total": torch.empty(1, dtype=torch.int32, device=dev),
    }
    o["err"] = _err_word(err if err is not None else o.get("err"), dev)
    ws_bytes = route_workspace_size(T, k, E)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    rc = lib().moe_route_offsets(_ptr(topk_idx), T, k, E, align, M_cap, _ptr(o["counts"]),
                                 _ptr(o["offsets"]), _ptr(o["row_of_pair"]), _ptr(o["pair_of_row"]),
                                 _ptr(o["true_total"]), _ptr(workspace), workspace.numel(),
                                 _ptr(o["err"]), _stream(stream))
    _check(rc, "moe_route_offsets")
    return o


def route_logits(logits: torch.Tensor, k: int, align: int = 1, M_cap: int | None = None,
                 err: torch.Tensor | None = None, out: dict | None = None,
                 workspace: torch.Tensor | None = None, stream=None) -> dict:
    """The router fused into the routing layout (see moe_route_logits):
    from logits [T, E] float32 to the dict of route_offsets plus topk_idx
    [T, k] and probs [T, k]."""
    _need(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    if M_cap is None:
        M_cap = T * k + E * (align - 1)
    dev = logits.device
    o = out if out is not None else {
        "topk_idx": torch.empty((T, k), dtype=torch.int32, device=dev),
        "probs": torch.empty((T, k), dtype=torch.float32, device=dev),
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "row_of_pair": torch.empty(T * k, dtype=torch.int32, device=dev),
        "pair_of_row": torch.empty(M_cap, dtype=torch.int32, device=dev),
        "true_total": torch.empty(1, dtype=torch.int32, device=dev),
    }
    o["err"] = _err_word(err if err is not None else o.get("err"), dev)
    ws_bytes = route_workspace_size(T, k, E)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    rc = lib().moe_route_logits(_ptr(logits), T, E, k, align, M_cap, _ptr(o["topk_idx"]),
                                _ptr(o["probs"]), _ptr(o["counts"]), _ptr(o["offsets"]),
                                _ptr(o["row_of_pair"]), _ptr(o["pair_of_row"]),
                                _ptr(o["true_total"]), _ptr(workspace), workspace.numel(),
                                _ptr(o["err"]), _stream(stream))
    _check(rc, "moe_route_logits")
    return o


def permute(src: torch.Tensor, pair_of_row: torch.Tensor, k: int, scale: torch.Tensor | None = None,
            out: torch.Tensor | None = None, stream=None,
            row_of_pair: torch.Tensor | None = None) -> torch.Tensor:
    """Expert-major gather (see moe_permute).  With ``row_of_pair`` (the
    routing layout's inverse map) the copy runs in token order
    (moe_permute_tokens), reading each token row once."""
    _need(src, torch.bfloat16, "src", 2)
    _need(pair_of_row, torch.int32, "pair_of_row")
    _need(row_of_pair, torch.int32, "row_of_pair")
    _need(scale, torch.float32, "scale")
    T, d = src.shape
    M_cap = pair_of_row.numel()
    if out is None:
        out = torch.empty((M_cap, d), dtype=torch.bfloat16, device=src.device)
    _need(out, torch.bfloat16, "out", 2)
    if row_of_pair is not None:
        if row_of_pair.numel() != T * k:
            raise MoeError("row_of_pair must hold T*k entries")
        rc = lib().moe_permute_tokens(_ptr(src), _ptr(scale), _ptr(row_of_pair), _ptr(pair_of_row),
                                      T, k, d, M_cap, _ptr(out), _stream(stream))
        _check(rc, "moe_permute_tokens")
        return out
    rc = lib().moe_permute(_ptr(src), _ptr(scale), _ptr(pair_of_row), T, k, d, M_cap, _ptr(out),
                           _stream(stream))
    _check(rc, "moe_permute")
    return out


def unpermute(src: torch.Tensor, row_of_pair: torch.Tensor, T: int, k: int,
              probs: torch.Tensor | None = None, out: torch.Tensor | None = None,
              dO: torch.Tensor | None = None, dprobs: torch.Tensor | None = None,
              combine: bool = True, stream=None):
    """Combine and/or router-score gradient (see moe_unpermute).  Returns
    (out, dprobs); either may be None."""
    _need(src, torch.bfloat16, "src", 2)
    _need(row_of_pair, torch.int32, "row_of_pair")
    _need(probs, torch.float32, "probs")
    _need(dO, torch.bfloat16, "dO")
    d = src.shape[1]
    if combine and out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=src.device)
    if not combine:
        out = None
    if dO is not None and dprobs is None:
        dprobs = torch.empty((T, k), dtype=torch.float32, device=src.device)
    _need(out, torch.bfloat16, "out")
    _need(dprobs, torch.float32, "dprobs")
    rc = lib().moe_unpermute(_ptr(src), _ptr(probs), _ptr(row_of_pair), T, k, d, src.shape[0],
                             _ptr(out),
                             _ptr(dO), _ptr(dprobs), _stream(stream))
    _check(rc, "moe_unpermute")
    return out, dprobs


def grouped_mlp_fwd(x_perm: torch.Tensor, offsets: torch.Tensor, W1: torch.Tensor,
                    W2: torch.Tensor, act: str = "swiglu", save_h: bool = False,
                    h_saved: torch.Tensor | None = None, a: torch.Tensor | None = None,
                    y_perm: torch.Tensor | None = None, err: torch.Tensor | None = None,
                    mx: dict | None = None, amax: torch.Tensor | None = None, stream=None):
    """Grouped expert MLP forward (see moe_grouped_mlp_fwd).  With ``mx`` (a
    dict of uint8 device tensors w2_q, w2_s, a_q, a_s and optionally a_qT,
    a_sT; see ``mx_buffers``) the MXFP8 path runs.  ``amax`` (a float32
    device tensor of one element) is raised to max |A|.  Returns
    (h_saved or None, a, y_perm, err)."""
    if amax is not None:
        _need(amax, torch.float32, "amax")
    _need(x_perm, torch.bfloat16, "x_perm", 2)
    _need(offsets, torch.int32, "offsets", 1)
    _need(W1, torch.bfloat16, "W1", 3)
    _need(W2, torch.bfloat16, "W2", 3)
    M_cap, d = x_perm.shape
    E, n, d2 = W2.shape
    n1 = n if act == "srelu" else 2 * n
    if d2 != d or tuple(W1.shape) != (E, d, n1) or offsets.numel() != E + 1:
        raise MoeError("inconsistent shapes")
    dev = x_perm.device
    if save_h and h_saved is None:
        h_saved = torch.empty((M_cap, n1), dtype=torch.bfloat16, device=dev)
    if a is None:
        a = torch.empty((M_cap, n), dtype=torch.bfloat16, device=dev)
    if y_perm is None:
        y_perm = torch.empty((M_cap, d), dtype=torch.bfloat16, device=dev)
    err = _err_word(err, dev)
    flags = FLAG_SAVE_H if save_h else 0
    mxs = None
    if mx is not None:
        names = ("w2_q", "w2_s", "a_q", "a_s", "a_qT", "a_sT", "y_q", "y_s")
        for k_ in names:
            _need(mx.get(k_), torch.uint8, k_)
        mxs = MxFwd(*[(mx[k_].data_ptr() if mx.get(k_) is not None else None) for k_ in names])
        flags |= FLAG_MXFP8
    rc = lib().moe_grouped_mlp_fwd(_ptr(x_perm), _ptr(offsets), E, M_cap, d, n, _ptr(W1), _ptr(W2),
                                   ACT[act], flags, _ptr(h_saved) if save_h else None, _ptr(a),
                                   _ptr(y_perm), ctypes.byref(mxs) if mxs is not None else None,
                                   _ptr(amax), _ptr(err), _stream(stream))
    _check(rc, "moe_grouped_mlp_fwd")
    return (h_saved if save_h else None), a, y_perm, err


def grouped_mlp_fwd_gather(x: torch.Tensor, pair_of_row: torch.Tensor, k: int,
                           offsets: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor,
                           act: str = "swiglu", save_h: bool = False, h_saved=None, a=None,
                           y_perm=None, err=None, amax=None, stream=None):
    """Grouped expert MLP forward reading the token rows of x [T, d] through
    the routing map (moe_grouped_mlp_fwd_gather): no permuted copy of x.
    Returns (h_saved or None, a, y_perm, err) like ``grouped_mlp_fwd``."""
    if amax is not None:
        _need(amax, torch.float32, "amax")
    _need(x, torch.bfloat16, "x", 2)
    _need(pair_of_row, torch.int32, "pair_of_row", 1)
    _need(offsets, torch.int32, "offsets", 1)
    _need(W1, torch.bfloat16, "W1", 3)
    _need(W2, torch.bfloat16, "W2", 3)
    T, d = x.shape
    M_cap = pair_of_row.numel()
    E, n, d2 = W2.shape
    n1 = n if act == "srelu" else 2 * n
    if d2 != d or tuple(W1.shape) != (E, d, n1) or offsets.numel() != E + 1:
        raise MoeError("inconsistent shapes")
    dev = x.device
    if save_h and h_saved is None:
        h_saved = torch.empty((M_cap, n1), dtype=torch.bfloat16, device=dev)
    if a is None:
        a = torch.empty((M_cap, n), dtype=torch.bfloat16, device=dev)
    if y_perm is None:
        y_perm = torch.empty((M_cap, d), dtype=torch.bfloat16, device=dev)
    err = _err_word(err, dev)
    if T == 0:      # the library reads nothing of x then, but needs an address
        x = torch.zeros((1, d), dtype=torch.bfloat16, device=dev)
    rc = lib().moe_grouped_mlp_fwd_gather(
        _ptr(x), T, k, _ptr(pair_of_row), _ptr(offsets), E, M_cap, d, n, _ptr(W1), _ptr(W2),
        ACT[act], FLAG_SAVE_H if save_h else 0, _ptr(h_saved) if save_h else None, _ptr(a),
        _ptr(y_perm), _ptr(amax), _ptr(err), _stream(stream))
    _check(rc, "moe_grouped_mlp_fwd_gather")
    return (h_saved if save_h else None), a, y_perm, err


def _bwd_flags(accumulate_dw: bool, dW1, dW2) -> int:
    if not accumulate_dw:
        return 0
    if dW1 is None or dW2 is None:
        raise ValueError("accumulate_dw needs the dW1 and dW2 to accumulate into")
    return FLAG_ACCUMULATE_DW


def grouped_mlp_bwd(x_perm, h_saved, a, dy_perm, offsets, W1, W2, act: str = "swiglu",
                    dh=None, dx_perm=None, dW1=None, dW2=None, err=None, amax=None, stream=None,
                    accumulate_dw: bool = False):
    """Grouped expert MLP backward (see moe_grouped_mlp_bwd).  Returns
    (dh, dx_perm, dW1, dW2, err).  accumulate_dw: add this step's weight
    gradients to the given dW1, dW2 (MOE_FLAG_ACCUMULATE_DW)."""
    flags = _bwd_flags(accumulate_dw, dW1, dW2)
    for t, nm in ((x_perm, "x_perm"), (h_saved, "h_saved"), (a, "a"), (dy_perm, "dy_perm"),
                  (W1, "W1"), (W2, "W2")):
        _need(t, torch.bfloat16, nm)
    _need(offsets, torch.int32, "offsets", 1)
    M_cap, d = x_perm.shape
    E, n, _ = W2.shape
    n1 = n if act == "srelu" else 2 * n
    dev = x_perm.device
    if dh is None:
        dh = torch.empty((M_cap, n1), dtype=torch.bfloat16, device=dev)
    if dx_perm is None:
        dx_perm = torch.empty((M_cap, d), dtype=torch.bfloat16, device=dev)
    if dW1 is None:
        dW1 = torch.empty((E, d, n1), dtype=torch.bfloat16, device=dev)
    if dW2 is None:
        dW2 = torch.empty((E, n, d), dtype=torch.bfloat16, device=dev)
    err = _err_word(err, dev)
    rc = lib().moe_grouped_mlp_bwd(_ptr(x_perm), _ptr(h_saved), _ptr(a), _ptr(dy_perm),
                                   _ptr(offsets), E, M_cap, d, n, _ptr(W1), _ptr(W2), ACT[act], flags,
                                   _ptr(dh), _ptr(dx_perm), _ptr(dW1), _ptr(dW2), _ptr(amax),
                                   _ptr(err), _stream(stream))
    _check(rc, "moe_grouped_mlp_bwd")
    return dh, dx_perm, dW1, dW2, err


def mx_buffers(E: int, n: int, d: int, M_cap: int, device, transposed: bool = True,
               quantize_y: bool = False) -> dict:
    """Allocate the uint8 buffers of moe_mx_fwd (sizes as moe.h states)."""
    u8 = torch.uint8
    b = {"w2_q": torch.empty((E, n, d), dtype=u8, device=device),
         "w2_s": torch.empty(E * (n // 32) * d, dtype=u8, device=device),
         "a_q": torch.empty((M_cap, n), dtype=u8, device=device),
         "a_s": torch.empty((M_cap // 32) * (n // 128) * 512, dtype=u8, device=device)}
    if transposed:
        b["a_qT"] = torch.empty((n, M_cap), dtype=u8, device=device)
        b["a_sT"] = torch.empty((n, M_cap // 32), dtype=u8, device=device)
    if quantize_y:
        b["y_q"] = torch.empty((M_cap, d), dtype=u8, device=device)
        b["y_s"] = torch.empty((M_cap, d // 32), dtype=u8, device=device)
    return b


def _offsets_arg(offsets, E):
    if offsets is None:
        return None
    _need(offsets, torch.int32, "offsets", 1)
    if offsets.numel() != E + 1:
        raise ValueError(f"offsets has {offsets.numel()} entries, want E+1 = {E + 1}")
    return offsets


def mx_quantize_weights(W2: torch.Tensor, w2_q: torch.Tensor | None = None,
                        w2_s: torch.Tensor | None = None, stream=None, offsets=None):
    """MXFP8 codes and MMA-tiled scales of W2 [E, n, d] (moe_mx_quantize_weights).
    With the routing ``offsets``, experts without rows are skipped (left as
    they were in w2_q / w2_s)."""
    _need(W2, torch.bfloat16, "W2", 3)
    E, n, d = W2.shape
    offsets = _offsets_arg(offsets, E)
    if w2_q is None:
        w2_q = torch.empty((E, n, d), dtype=torch.uint8, device=W2.device)
    if w2_s is None:
        w2_s = torch.empty(E * (n // 32) * d, dtype=torch.uint8, device=W2.device)
    _need(w2_q, torch.uint8, "w2_q")
    _need(w2_s, torch.uint8, "w2_s")
    rc = lib().moe_mx_quantize_weights(_ptr(W2), E, n, d, _ptr(offsets), _ptr(w2_q), _ptr(w2_s),
                                       _stream(stream))
    _check(rc, "moe_mx_quantize_weights")
    return w2_q, w2_s


def mx_quantize(src: torch.Tensor, offsets: torch.Tensor, transposed: bool = True,
                err: torch.Tensor | None = None, stream=None):
    """Group-aware MXFP8 quantisation (moe_mx_quantize).  Returns
    (q, s, qT, sT, err); qT/sT are None unless ``transposed``."""
    _need(src, torch.bfloat16, "src", 2)
    _need(offsets, torch.int32, "offsets", 1)
    rows, cols = src.shape
    dev = src.device
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=dev)
    qT = torch.empty((cols, rows), dtype=torch.uint8, device=dev) if transposed else None
    sT = torch.empty((cols, rows // 32), dtype=torch.uint8, device=dev) if transposed else None
    err = _err_word(err, dev)
    rc = lib().moe_mx_quantize(_ptr(src), rows, cols, _ptr(offsets), offsets.numel() - 1, _ptr(q),
                               _ptr(s), _ptr(qT), _ptr(sT), _ptr(err), _stream(stream))
    _check(rc, "moe_mx_quantize")
    return q, s, qT, sT, err


def mx_quantize_tiled(src: torch.Tensor, offsets: torch.Tensor, rowwise: bool = True,
                      transposed: bool = True, err: torch.Tensor | None = None, stream=None):
    """Group-aware MXFP8 quantisation with the scales in the block-scaled
    GEMM's layouts (moe_mx_quantize_tiled).  Returns (q, s, qT, sT, err);
    q/s are None unless ``rowwise``, qT/sT None unless ``transposed``; s and
    sT are rows*cols/8 bytes each."""
    _need(src, torch.bfloat16, "src", 2)
    _need(offsets, torch.int32, "offsets", 1)
    if not (rowwise or transposed):
        raise ValueError("at least one copy")
    rows, cols = src.shape
    dev = src.device
    u8 = torch.uint8
    q = torch.empty((rows, cols), dtype=u8, device=dev) if rowwise else None
    s = torch.empty(rows * cols // 8, dtype=u8, device=dev) if rowwise else None
    qT = torch.empty((cols, rows), dtype=u8, device=dev) if transposed else None
    sT = torch.empty(rows * cols // 8, dtype=u8, device=dev) if transposed else None
    err = _err_word(err, dev)
    rc = lib().moe_mx_quantize_tiled(_ptr(src), rows, cols, _ptr(offsets), offsets.numel() - 1,
                                     _ptr(q), _ptr(s), _ptr(qT), _ptr(sT), _ptr(err),
                                     _stream(stream))
    _check(rc, "moe_mx_quantize_tiled")
    return q, s, qT, sT, err


def mx_quantize_weights_rowwise(W: torch.Tensor, q: torch.Tensor | None = None,
                                s: torch.Tensor | None = None, stream=None, offsets=None):
    """MXFP8 codes of a weight with blocks along its last axis and scales in
    weight tiles (moe_mx_quantize_weights_rowwise); W is [E, R, K] or [R, K].
    With the routing ``offsets`` (W then [E, R, K]), experts without rows
    are skipped (left as they were in q / s)."""
    _need(W, torch.bfloat16, "W")
    K = W.shape[-1]
    rows = W.numel() // K
    E = W.shape[0] if offsets is not None else 0
    if offsets is not None and W.dim() != 3:
        raise ValueError("offsets needs W as [E, R, K]")
    offsets = _offsets_arg(offsets, E) if offsets is not None else None
    if q is None:
        q = torch.empty(tuple(W.shape), dtype=torch.uint8, device=W.device)
    if s is None:
        s = torch.empty(rows * K // 32, dtype=torch.uint8, device=W.device)
    _need(q, torch.uint8, "q")
    _need(s, torch.uint8, "s")
    rc = lib().moe_mx_quantize_weights_rowwise(_ptr(W), rows, K, _ptr(offsets), E, _ptr(q), _ptr(s),
                                               _stream(stream))
    _check(rc, "moe_mx_quantize_weights_rowwise")
    return q, s


def mx_bwd_workspace_size(M_cap: int, d: int, n: int, act: str = "swiglu") -> int:
    return int(lib().moe_mx_bwd_workspace_size(M_cap, d, n, ACT[act]))


PAIR_NEVER, PAIR_AUTO, PAIR_ALWAYS = 0, 1, 2


def set_pair_mma(mode: int) -> int:
    """moe_set_pair_mma: 0 never, 1 automatic (default), 2 always pair the
    two CTAs of a cluster with 2-SM MMAs; returns the previous mode."""
    rc = int(lib().moe_set_pair_mma(int(mode)))
    _check(rc if rc < 0 else 0, "moe_set_pair_mma")
    return rc


MX_BWD_SECTIONS = ("dy_q", "dy_s", "dy_qT", "dy_sT", "x_qT", "x_sT", "a_sT", "dh_q", "dh_s",
                   "dh_qT", "dh_sT")


def mx_bwd_workspace_layout(M_cap: int, d: int, n: int, act: str = "swiglu") -> dict:
    """Byte offsets of the MXFP8 backward's quantised operands inside its
    workspace (moe_mx_bwd_workspace_layout), by section name, plus "bytes"."""
    offs = (ctypes.c_size_t * len(MX_BWD_SECTIONS))()
    total = int(lib().moe_mx_bwd_workspace_layout(M_cap, d, n, ACT[act], offs))
    if total == 0:
        raise MoeError("moe_mx_bwd_workspace_layout: invalid sizes")
    out = {nm: int(offs[i]) for i, nm in enumerate(MX_BWD_SECTIONS)}
    out["bytes"] = total
    return out


def grouped_mlp_bwd_mx(x_perm, h_saved, dy_perm, offsets, mx: dict, act: str = "swiglu",
                       dh=None, dx_perm=None, dW1=None, dW2=None, err=None, workspace=None,
                       stream=None, accumulate_dw: bool = False, separate_dh_quant: bool = False):
    """MXFP8 grouped expert MLP backward (moe_grouped_mlp_bwd_mx).  ``mx``
    holds uint8 tensors a_qT, a_sT (the forward's transposed copy), w2_q, w2_s
    (W2 with blocks along d) and w1_q, w1_s (W1 with blocks along n1).
    Returns (dh, dx_perm, dW1, dW2, err).  accumulate_dw as in
    grouped_mlp_bwd; separate_dh_quant selects the unfused control (dH
    quantised in its own pass, MOE_FLAG_MX_SEPARATE_DH_QUANT)."""
    flags = _bwd_flags(accumulate_dw, dW1, dW2)
    if separate_dh_quant:
        flags |= FLAG_MX_SEPARATE_DH_QUANT
    for t, nm in ((x_perm, "x_perm"), (h_saved, "h_saved"), (dy_perm, "dy_perm")):
        _need(t, torch.bfloat16, nm)
    _need(offsets, torch.int32, "offsets", 1)
    for k_ in ("a_qT", "a_sT", "w2_q", "w2_s", "w1_q", "w1_s"):
        _need(mx.get(k_), torch.uint8, k_)
    M_cap, d = x_perm.shape
    E = offsets.numel() - 1
    n = mx["a_qT"].shape[0]
    n1 = h_saved.shape[1]
    dev = x_perm.device
    if dh is None:
        dh = torch.empty((M_cap, n1), dtype=torch.bfloat16, device=dev)
    if dx_perm is None:
        dx_perm = torch.empty((M_cap, d), dtype=torch.bfloat16, device=dev)
    if dW1 is None:
        dW1 = torch.empty((E, d, n1), dtype=torch.bfloat16, device=dev)
    if dW2 is None:
        dW2 = torch.empty((E, n, d), dtype=torch.bfloat16, device=dev)
    err = _err_word(err, dev)
    need = mx_bwd_workspace_size(M_cap, d, n, act)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _need(workspace, torch.uint8, "workspace")
    for k_ in ("dx_q", "dx_s"):
        _need(mx.get(k_), torch.uint8, k_)
    st = MxBwd(mx["a_qT"].data_ptr(), mx["a_sT"].data_ptr(), mx["w2_q"].data_ptr(),
               mx["w2_s"].data_ptr(), mx["w1_q"].data_ptr(), mx["w1_s"].data_ptr(),
               workspace.data_ptr(), workspace.numel(),
               mx["dx_q"].data_ptr() if mx.get("dx_q") is not None else None,
               mx["dx_s"].data_ptr() if mx.get("dx_s") is not None else None)
    rc = lib().moe_grouped_mlp_bwd_mx(_ptr(x_perm), _ptr(h_saved), _ptr(dy_perm), _ptr(offsets),
                                      E, M_cap, d, n, ACT[act], flags, ctypes.byref(st), _ptr(dh),
                                      _ptr(dx_perm), _ptr(dW1), _ptr(dW2), _ptr(err),
                                      _stream(stream))
    _check(rc, "moe_grouped_mlp_bwd_mx")
    return dh, dx_perm, dW1, dW2, err


def grouped_mlp_bwd_routed(x_perm, h_saved, do_perm, pair_of_row, probs, offsets, W1, W2,
                           act: str = "swiglu", dh=None, a_scaled=None, ds_part=None,
                           dx_perm=None, dW1=None, dW2=None, err=None, amax=None, stream=None,
                           accumulate_dw: bool = False):
    """Backward with the router gradient inside the expert MLP
    (moe_grouped_mlp_bwd_routed).  do_perm is the gathered dO without the
    router probability.  Returns (dh, a_scaled, ds_part, dx_perm, dW1, dW2,
    err).  accumulate_dw as in grouped_mlp_bwd."""
    flags = _bwd_flags(accumulate_dw, dW1, dW2)
    for t, nm in ((x_perm, "x_perm"), (h_saved, "h_saved"), (do_perm, "do_perm"), (W1, "W1"),
                  (W2, "W2")):
        _need(t, torch.bfloat16, nm)
    _need(pair_of_row, torch.int32, "pair_of_row", 1)
    _need(probs, torch.float32, "probs")
    _need(offsets, torch.int32, "offsets", 1)
    M_cap, d = x_perm.shape
    E, n, _ = W2.shape
    n1 = n if act == "srelu" else 2 * n
    dev = x_perm.device
    bf = torch.bfloat16
    if dh is None:
        dh = torch.empty((M_cap, n1), dtype=bf, device=dev)
    if a_scaled is None:
        a_scaled = torch.empty((M_cap, n), dtype=bf, device=dev)
    if ds_part is None:
        ds_part = torch.empty((M_cap, (n + 127) // 128), dtype=torch.float32, device=dev)
    if dx_perm is None:
        dx_perm = torch.empty((M_cap, d), dtype=bf, device=dev)
    if dW1 is None:
        dW1 = torch.empty((E, d, n1), dtype=bf, device=dev)
    if dW2 is None:
        dW2 = torch.empty((E, n, d), dtype=bf, device=dev)
    err = _err_word(err, dev)
    rc = lib().moe_grouped_mlp_bwd_routed(
        _ptr(x_perm), _ptr(h_saved), _ptr(do_perm), _ptr(pair_of_row), _ptr(probs), _ptr(offsets),
        E, M_cap, d, n, _ptr(W1), _ptr(W2), ACT[act], flags, _ptr(dh), _ptr(a_scaled), _ptr(ds_part),
        _ptr(dx_perm), _ptr(dW1), _ptr(dW2), _ptr(amax), _ptr(err), _stream(stream))
    _check(rc, "moe_grouped_mlp_bwd_routed")
    return dh, a_scaled, ds_part, dx_perm, dW1, dW2, err


def grouped_mlp_bwd_routed_gather(x, dO, pair_of_row, k: int, h_saved, probs, offsets, W1, W2,
                                  act: str = "swiglu", dh=None, a_scaled=None, ds_part=None,
                                  dx_perm=None, dW1=None, dW2=None, err=None, amax=None,
                                  stream=None, accumulate_dw: bool = False):
    """Routed backward reading x [T, d] and dO [T, d] through the routing map
    (moe_grouped_mlp_bwd_routed_gather): no permuted copies.  Returns (dh,
    a_scaled, ds_part, dx_perm, dW1, dW2, err) like
    ``grouped_mlp_bwd_routed``."""
    flags = _bwd_flags(accumulate_dw, dW1, dW2)
    for t, nm in ((x, "x"), (dO, "dO"), (h_saved, "h_saved"), (W1, "W1"), (W2, "W2")):
        _need(t, torch.bfloat16, nm)
    _need(pair_of_row, torch.int32, "pair_of_row", 1)
    _need(probs, torch.float32, "probs")
    _need(offsets, torch.int32, "offsets", 1)
    T, d = x.shape
    M_cap = pair_of_row.numel()
    E, n, _ = W2.shape
    n1 = n if act == "srelu" else 2 * n
    dev = x.device
    bf = torch.bfloat16
    if dh is None:
        dh = torch.empty((M_cap, n1), dtype=bf, device=dev)
    if a_scaled is None:
        a_scaled = torch.empty((M_cap, n), dtype=bf, device=dev)
    if ds_part is None:
        ds_part = torch.empty((M_cap, (n + 127) // 128), dtype=torch.float32, device=dev)
    if dx_perm is None:
        dx_perm = torch.empty((M_cap, d), dtype=bf, device=dev)
    if dW1 is None:
        dW1 = torch.empty((E, d, n1), dtype=bf, device=dev)
    if dW2 is None:
        dW2 = torch.empty((E, n, d), dtype=bf, device=dev)
    err = _err_word(err, dev)
    if T == 0:      # nothing of x or dO is read then, but the maps need addresses
        x = dO = torch.zeros((1, d), dtype=bf, device=dev)
    rc = lib().moe_grouped_mlp_bwd_routed_gather(
        _ptr(x), _ptr(dO), T, k, _ptr(h_saved), _ptr(pair_of_row), _ptr(probs), _ptr(offsets), E,
        M_cap, d, n, _ptr(W1), _ptr(W2), ACT[act], flags, _ptr(dh), _ptr(a_scaled), _ptr(ds_part),
        _ptr(dx_perm), _ptr(dW1), _ptr(dW2), _ptr(amax), _ptr(err), _stream(stream))
    _check(rc, "moe_grouped_mlp_bwd_routed_gather")
    return dh, a_scaled, ds_part, dx_perm, dW1, dW2, err


def router_grad_rows(ds_part, row_of_pair, T: int, k: int, dprobs=None, stream=None):
    """dprobs [T, k] from the routed backward's partials (moe_router_grad_rows)."""
    _need(ds_part, torch.float32, "ds_part", 2)
    _need(row_of_pair, torch.int32, "row_of_pair", 1)
    M_cap, n_parts = ds_part.shape
    if dprobs is None:
        dprobs = torch.empty((T, k), dtype=torch.float32, device=ds_part.device)
    rc = lib().moe_router_grad_rows(_ptr(ds_part), n_parts, _ptr(row_of_pair), T, k, M_cap,
                                    _ptr(dprobs), _stream(stream))
    _check(rc, "moe_router_grad_rows")
    return dprobs


def mx_quantize_weights2(W2: torch.Tensor, w2_q=None, w2_s=None, w2_q_rows=None, w2_s_rows=None,
                         stream=None, offsets=None):
    """Both MXFP8 copies of W2 [E, n, d] from one read (moe_mx_quantize_weights2):
    blocks along n (w2_q, w2_s; forward FC2) and along d (w2_q_rows,
    w2_s_rows; backward FC2-dgrad).  Returns the four tensors.  With the
    routing ``offsets``, experts without rows are skipped."""
    _need(W2, torch.bfloat16, "W2", 3)
    E, n, d = W2.shape
    offsets = _offsets_arg(offsets, E)
    u8 = torch.uint8
    dev = W2.device
    if w2_q is None:
        w2_q = torch.empty((E, n, d), dtype=u8, device=dev)
    if w2_s is None:
        w2_s = torch.empty(E * (n // 32) * d, dtype=u8, device=dev)
    if w2_q_rows is None:
        w2_q_rows = torch.empty((E, n, d), dtype=u8, device=dev)
    if w2_s_rows is None:
        w2_s_rows = torch.empty(E * n * d // 32, dtype=u8, device=dev)
    for t, nm in ((w2_q, "w2_q"), (w2_s, "w2_s"), (w2_q_rows, "w2_q_rows"), (w2_s_rows, "w2_s_rows")):
        _need(t, u8, nm)
    rc = lib().moe_mx_quantize_weights2(_ptr(W2), E, n, d, _ptr(offsets), _ptr(w2_q), _ptr(w2_s),
                                        _ptr(w2_q_rows), _ptr(w2_s_rows), _stream(stream))
    _check(rc, "moe_mx_quantize_weights2")
    return w2_q, w2_s, w2_q_rows, w2_s_rows


# ----------------------------------------------------------------- unfused pieces

def grouped_gemm(a, offsets, B, b_layout: str = "kn", out=None, err=None, stream=None):
    """Plain grouped GEMM (moe_grouped_gemm): out_e = a_e B_e with B [E, K, N]
    ("kn"), or B stored [E, N, K] and out_e = a_e B_e^T ("nk").  Returns
    (out, err)."""
    _need(a, torch.bfloat16, "a", 2)
    _need(B, torch.bfloat16, "B", 3)
    _need(offsets, torch.int32, "offsets", 1)
    layout = {"kn": 0, "nk": 1}[b_layout]
    M_cap, K = a.shape
    E = B.shape[0]
    N = B.shape[2] if layout == 0 else B.shape[1]
    if out is None:
        out = torch.empty((M_cap, N), dtype=torch.bfloat16, device=a.device)
    err = _err_word(err, a.device)
    rc = lib().moe_grouped_gemm(_ptr(a), _ptr(offsets), E, M_cap, K, N, _ptr(B), layout, _ptr(out),
                                _ptr(err), _stream(stream))
    _check(rc, "moe_grouped_gemm")
    return out, err


def activation(h, offsets, act: str = "swiglu", a=None, stream=None):
    """A = act(H) as its own memory pass (moe_activation)."""
    _need(h, torch.bfloat16, "h", 2)
    _need(offsets, torch.int32, "offsets", 1)
    M_cap, n1 = h.shape
    n = n1 if act == "srelu" else n1 // 2
    if a is None:
        a = torch.empty((M_cap, n), dtype=torch.bfloat16, device=h.device)
    rc = lib().moe_activation(_ptr(h), _ptr(offsets), offsets.numel() - 1, M_cap, n, ACT[act],
                              _ptr(a), _stream(stream))
    _check(rc, "moe_activation")
    return a


def activation_bwd(h, da, offsets, act: str = "swiglu", dh=None, stream=None):
    """dH = act'(H; dA) as its own memory pass (moe_activation_bwd)."""
    _need(h, torch.bfloat16, "h", 2)
    _need(da, torch.bfloat16, "da", 2)
    _need(offsets, torch.int32, "offsets", 1)
    M_cap, n = da.shape
    if dh is None:
        dh = torch.empty_like(h)
    rc = lib().moe_activation_bwd(_ptr(h), _ptr(da), _ptr(offsets), offsets.numel() - 1, M_cap, n,
                                  ACT[act], _ptr(dh), _stream(stream))
    _check(rc, "moe_activation_bwd")
    return dh
