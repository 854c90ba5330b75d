"""GB300 (sm_103a) sparse Mixture-of-Experts FFN layer.

Python binding of the C ABI in ``include/moe.h`` (``libmoe_gb300.so``).  The
functions keep the C names and only marshal arguments: tensors become device
pointers, ``None`` becomes NULL, the stream defaults to torch's current
stream.  Every step of the layer runs in the library's CUDA kernels; there is
no fallback of any kind, and loading fails loudly when the library is absent.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libmoe_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG_DIR), "include", "moe.h")

MOE_F32, MOE_BF16, MOE_FP8_E4M3, MOE_FP8_E4M3_NK, MOE_FP8_E4M3_NK_A8 = 0, 1, 2, 3, 4
MOE_ACT_SWIGLU, MOE_ACT_GEGLU_TANH = 0, 1
MOE_OK = 0
MOE_DEV_BAD_EXPERT_ID = 0x1
MOE_DEV_BAD_OFFSETS = 0x2
MOE_DEV_BAD_DEST = 0x4
MOE_DEV_NONFINITE_LOGIT = 0x8
MOE_DEV_WAIT_TIMEOUT = 0x10
WS_SLOTS = ["logits", "topk_ids", "topk_w", "counts", "offsets", "sorted_rows", "dest",
            "x_perm", "h", "y_perm", "h_shared", "s", "x16", "tok_inv", "row_inv"]

_DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16, "fp8_e4m3": MOE_FP8_E4M3,
           "fp8_e4m3_nk": MOE_FP8_E4M3_NK, "fp8_e4m3_nk_a8": MOE_FP8_E4M3_NK_A8}
_ACTS = {"swiglu": MOE_ACT_SWIGLU, "geglu_tanh": MOE_ACT_GEGLU_TANH}


class MoEConfig(ctypes.Structure):
    """Mirror of moe_config_t."""

    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "D", "E", "k", "I", "I_shared", "act", "act_dtype", "w_dtype", "renormalize")]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} returned {status}: {text}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_SIGS = {
    "moe_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(MoEConfig)]),
    "moe_workspace_offset": (ctypes.c_size_t, [ctypes.POINTER(MoEConfig), ctypes.c_int]),
    "moe_route": (ctypes.c_int, [ctypes.POINTER(MoEConfig)] + [_P] * 6 + [_P, ctypes.c_size_t, _P]),
    "moe_permute": (ctypes.c_int, [ctypes.POINTER(MoEConfig)] + [_P] * 7 + [_P, ctypes.c_size_t, _P]),
    "moe_grouped_ffn": (ctypes.c_int, [ctypes.POINTER(MoEConfig)] + [_P] * 15 + [_P, ctypes.c_size_t, _P]),
    "moe_finalize": (ctypes.c_int, [ctypes.POINTER(MoEConfig)] + [_P] * 5 + [_P, ctypes.c_size_t, _P]),
    "moe_layer": (ctypes.c_int, [ctypes.POINTER(MoEConfig)] + [_P] * 12 + [_P, ctypes.c_size_t, _P]),
    "moe_read_device_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_layer_launch_count": (ctypes.c_int, [ctypes.POINTER(MoEConfig)]),
    "moe_set_trace_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    "moe_permute_noalloc": (ctypes.c_int, [ctypes.POINTER(MoEConfig)] + [_P] * 7 + [_P]),
    "moe_set_option": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "moe_pack_weights_nk": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P]),
}
MOE_OPT_PAIR_TILES = 1
MOE_OPT_GATHER_A = 2
MOE_OPT_DECODE_KERNEL = 3
MOE_OPT_PDL = 4
MOE_OPT_SHARED_STREAM = 5
MOE_OPT_FUSED_COMBINE = 6
MOE_OPT_TILE_ORDER = 7
MOE_OPT_SHARED_IN_GEMM = 9
MOE_OPT_FUSED_ROUTING = 10
MOE_OPT_B_PREFETCH = 11
MOE_OPT_DYNAMIC_TILES = 12
MOE_OPT_SHARED_CTAS = 13


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmoe_gb300.so (raises when it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() "
                           "(or python -m mixture_experts_layer_gating_gb300._build)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def header_symbols(header: str = HEADER_PATH):
    """Function names declared in include/moe.h."""
    txt = open(header).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", txt, flags=re.M)))


def make_config(T: int, D: int, E: int, k: int, I: int, I_shared: int = 0, act: str = "swiglu",
                act_dtype: str = "bf16", w_dtype: str = "bf16", renormalize: bool = True) -> MoEConfig:
    return MoEConfig(T, D, E, k, I, I_shared, _ACTS[act], _DTYPES[act_dtype], _DTYPES[w_dtype],
                     1 if renormalize else 0)


def config_from_shape(shape, fp8_layout: str = "kn") -> MoEConfig:
    """MoEConfig from a workloads.MoEShape-like object.  For fp8 weights,
    fp8_layout "nk" selects MOE_FP8_E4M3_NK (weights packed by pack_weights_nk)
    and "nk_a8" MOE_FP8_E4M3_NK_A8 (the same weights, W8A8 activations)."""
    if fp8_layout not in ("kn", "nk", "nk_a8"):
        raise ValueError("fp8_layout is 'kn', 'nk' or 'nk_a8'")
    w = shape.w_dtype
    if w == "fp8_e4m3" and fp8_layout == "nk":
        w = "fp8_e4m3_nk"
    if w == "fp8_e4m3" and fp8_layout == "nk_a8":
        w = "fp8_e4m3_nk_a8"
    return make_config(shape.T, shape.D, shape.E, shape.k, shape.I, shape.I_shared, shape.act,
                       shape.act_dtype, w, shape.renormalize)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws(ws):
    return _ptr(ws), (ws.numel() * ws.element_size() if hasattr(ws, "numel") else 0)


def _check(fn: str, st: int):
    if st != MOE_OK:
        raise MoEError(fn, st, load_library().moe_status_string(st).decode())


def moe_workspace_size(cfg: MoEConfig) -> int:
    return int(load_library().moe_workspace_size(ctypes.byref(cfg)))


def moe_workspace_offset(cfg: MoEConfig, which: int) -> int:
    return int(load_library().moe_workspace_offset(ctypes.byref(cfg), which))


def moe_layer_launch_count(cfg: MoEConfig) -> int:
    return int(load_library().moe_layer_launch_count(ctypes.byref(cfg)))


def moe_set_trace_events(events) -> None:
    """Record one of ``events`` (torch.cuda.Event) at every kernel boundary of
    the following moe_layer calls; None switches it off."""
    lib = load_library()
    if not events:
        lib.moe_set_trace_events(None, 0)
        moe_set_trace_events._keep = None
        return
    for e in events:  # force creation of the underlying cudaEvent_t
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    moe_set_trace_events._keep = arr
    lib.moe_set_trace_events(arr, len(events))


def moe_set_option(option: int, value: int) -> int:
    """Set a kernel-variant option (e.g. MOE_OPT_PAIR_TILES); returns the old value."""
    r = int(load_library().moe_set_option(option, value))
    if r < 0:
        raise MoEError("moe_set_option", r, moe_status_string(r))
    return r


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_route(cfg, x, Wg, logit_bias, logits, topk_ids, topk_w, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_route", load_library().moe_route(
        ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logit_bias), _ptr(logits), _ptr(topk_ids),
        _ptr(topk_w), wp, wb, _stream(stream)))


def moe_permute(cfg, topk_ids, x, counts, offsets, sorted_rows, dest, x_perm, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_permute", load_library().moe_permute(
        ctypes.byref(cfg), _ptr(topk_ids), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(sorted_rows),
        _ptr(dest), _ptr(x_perm), wp, wb, _stream(stream)))


def moe_permute_noalloc(cfg, topk_ids, x, counts, offsets, sorted_rows, dest, x_perm, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device
    memory: its scratch is a fixed array inside the library (see include/moe.h
    for the size limit and the rule that overlapping calls race)."""
    _check("moe_permute_noalloc", load_library().moe_permute_noalloc(
        ctypes.byref(cfg), _ptr(topk_ids), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(sorted_rows),
        _ptr(dest), _ptr(x_perm), _stream(stream)))


def moe_grouped_ffn(cfg, x_perm, offsets, W13, s13, W2, s2, h, y_perm, x=None, W13s=None,
                    s13s=None, W2s=None, s2s=None, h_s=None, s_out=None, ws=None, stream=None):
    wp, wb = _ws(ws)
    _check("moe_grouped_ffn", load_library().moe_grouped_ffn(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(W13), _ptr(s13), _ptr(W2), _ptr(s2),
        _ptr(h), _ptr(y_perm), _ptr(x), _ptr(W13s), _ptr(s13s), _ptr(W2s), _ptr(s2s), _ptr(h_s),
        _ptr(s_out), wp, wb, _stream(stream)))


def moe_finalize(cfg, y_perm, dest, topk_w, s, out, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_finalize", load_library().moe_finalize(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(dest), _ptr(topk_w), _ptr(s), _ptr(out), wp, wb,
        _stream(stream)))


def moe_layer(cfg, x, Wg, logit_bias, W13, s13, W2, s2, W13s, s13s, W2s, s2s, out, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_layer", load_library().moe_layer(
        ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logit_bias), _ptr(W13), _ptr(s13), _ptr(W2),
        _ptr(s2), _ptr(W13s), _ptr(s13s), _ptr(W2s), _ptr(s2s), _ptr(out), wp, wb,
        _stream(stream)))


def moe_pack_weights_nk(W, G: int, K: int, N: int, W_nk, stream=None) -> None:
    _check("moe_pack_weights_nk", load_library().moe_pack_weights_nk(
        _ptr(W), G, K, N, _ptr(W_nk), _stream(stream)))


def pack_weights_nk(W, stream=None):
    """A new [G, N, K] (or [N, K]) copy of the one-byte [G, K, N] (or [K, N])
    weight tensor W, written by moe_pack_weights_nk on W's device."""
    import torch

    if W.element_size() != 1:
        raise ValueError("pack_weights_nk takes one-byte (e4m3) weights")
    if W.dim() not in (2, 3):
        raise ValueError("pack_weights_nk takes [K, N] or [G, K, N] weights")
    Wg = W if W.dim() == 3 else W.unsqueeze(0)
    G, K, N = Wg.shape
    out = torch.empty((G, N, K), dtype=W.dtype, device=W.device)
    moe_pack_weights_nk(Wg, G, K, N, out, stream)
    return out if W.dim() == 3 else out[0]


def moe_read_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error flags."""
    flags = ctypes.c_int32(0)
    st = load_library().moe_read_device_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    if st not in (MOE_OK, -4):
        _check("moe_read_device_status", st)
    return int(flags.value)


def alloc_workspace(cfg: MoEConfig, device=None):
    """A zero-filled uint8 torch workspace of moe_workspace_size(cfg) bytes."""
    import torch

    n = moe_workspace_size(cfg)
    if n == 0:
        raise ValueError("invalid MoE configuration")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def workspace_view(ws, cfg: MoEConfig, slot: str, shape, dtype):
    """A typed view of one of moe_layer's intermediates inside the workspace."""
    import torch

    off = moe_workspace_offset(cfg, WS_SLOTS.index(slot))
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).view(*shape)
