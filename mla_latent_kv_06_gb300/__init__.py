"""Thin Python binding of libmla.so (the C ABI in include/mla.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  Functions take
CUDA tensors, check dtype/shape/contiguity, allocate outputs and workspace
with torch when the caller gives none, and enqueue on the current stream.
There is no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmla.so")

MLA_F32, MLA_BF16 = 0, 1
MLA_OK, MLA_ERR_INVALID, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_DEVICE = 0, -1, -2, -3, -4
MLA_DEV_BAD_LENGTH, MLA_DEV_BAD_INDEX, MLA_DEV_TIMEOUT = 1, 2, 4

# Every symbol declared in include/mla.h.
EXPORTS = (
    "mla_last_error", "mla_abi_version", "mla_device_status", "mla_set_wait_limit_ns",
    "mla_set_kernel_events", "mla_last_launch_names",
    "mla_decode_absorbed_workspace_size", "mla_decode_absorbed", "mla_decode_launch_count",
    "mla_sparse_decode_workspace_size", "mla_sparse_decode", "mla_sparse_decode_layers_workspace_size",
    "mla_sparse_decode_layers",
    "mla_prefill_naive_workspace_size", "mla_prefill_naive", "mla_prefill_naive_noalloc",
    "dsa_index_scores", "dsa_topk_select_workspace_size", "dsa_topk_select",
    "mla_cache_append", "dsa_index_key_append",
    "mla_decode_paged_workspace_size", "mla_decode_paged", "mla_sparse_decode_paged", "mla_cache_append_paged",
    "dsa_select_workspace_size", "dsa_select",
    "mla_o_proj_workspace_size", "mla_o_proj", "mla_decode_oproj_workspace_size", "mla_decode_oproj",
    "mla_decode_fp8_workspace_size", "mla_decode_fp8", "mla_decode_fp8_paged", "mla_cache_append_fp8",
    "mla_cache_append_fp8_paged",
)


class MlaDims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("qk_nope", ctypes.c_int), ("qk_rope", ctypes.c_int),
                ("kv_lora", ctypes.c_int), ("v_head", ctypes.c_int), ("scale", ctypes.c_float),
                ("rope_base", ctypes.c_float)]


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmla status {code}: {msg}")
        self.code = code


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_DP = ctypes.POINTER(MlaDims)
_PP = ctypes.POINTER(ctypes.c_void_p)  # host array of device pointers


def _declare(lib: ctypes.CDLL) -> None:
    sig = {
        "mla_last_error": (ctypes.c_char_p, []),
        "mla_abi_version": (_I, []),
        "mla_device_status": (_I, [_P, ctypes.POINTER(_I)]),
        "mla_set_wait_limit_ns": (None, [ctypes.c_longlong]),
        "mla_set_kernel_events": (_I, [ctypes.POINTER(ctypes.c_void_p), _I]),
        "mla_last_launch_names": (ctypes.c_char_p, []),
        "mla_decode_absorbed_workspace_size": (_SZ, [_DP, _I, _I, _I, _I]),
        "mla_decode_launch_count": (_I, [_DP, _I, _I, _I, _I]),
        "mla_decode_absorbed": (_I, [_DP, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _SZ, _P]),
        "mla_sparse_decode_workspace_size": (_SZ, [_DP, _I, _I, _I, _I]),
        "mla_sparse_decode": (_I, [_DP, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P,
                                   _SZ, _P]),
        "mla_sparse_decode_layers_workspace_size": (_SZ, [_DP, _I, _I, _I, _I, _I]),
        "mla_sparse_decode_layers": (_I, [_DP, _I, _I, _I, _I, _PP, _PP, _PP, _I, _P, _PP, _P, _P, _I, _PP, _PP, _I,
                                          _PP, _P, _SZ, _P]),
        "mla_prefill_naive_workspace_size": (_SZ, [_DP, _I, _I, _I, _I]),
        "mla_prefill_naive": (_I, [_DP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
        "mla_prefill_naive_noalloc": (_I, [_DP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
        "dsa_index_scores": (_I, [_I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P]),
        "dsa_topk_select_workspace_size": (_SZ, [_I, _I, _I, _I]),
        "dsa_topk_select": (_I, [_I, _I, _P, _I, _P, _I, _P, _P, _P, _SZ, _P]),
        "mla_cache_append": (_I, [_DP, _I, _I, _I, _P, _P, ctypes.c_float, _I, _P, _P, _P, _P]),
        "dsa_index_key_append": (_I, [_I, _I, _I, _I, _P, _P, _P, ctypes.c_float, ctypes.c_float, _I, _P,
                                      _P, _P]),
        "mla_decode_paged_workspace_size": (_SZ, [_DP, _I, _I, _I, _I, _I]),
        "mla_decode_paged": (_I, [_DP, _I, _I, _I, _P, _P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _SZ, _P]),
        "mla_sparse_decode_paged": (_I, [_DP, _I, _I, _I, _P, _P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _I, _P,
                                         _P, _SZ, _P]),
        "mla_cache_append_paged": (_I, [_DP, _I, _I, _I, _P, _P, ctypes.c_float, _P, _P, _I, _I, _P, _I, _P, _P]),
        "dsa_select_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
        "dsa_select": (_I, [_I, _I, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _SZ, _P]),
        "mla_o_proj_workspace_size": (_SZ, [_I, _I, _I, _I]),
        "mla_o_proj": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
        "mla_decode_oproj_workspace_size": (_SZ, [_DP, _I, _I, _I, _I, _I]),
        "mla_decode_oproj": (_I, [_DP, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _SZ, _P]),
        "mla_decode_fp8_workspace_size": (_SZ, [_DP, _I, _I, _I]),
        "mla_decode_fp8": (_I, [_DP, _I, _I, _P, _P, _P, ctypes.c_float, _I, _P, _P, _P, _P, _SZ, _P]),
        "mla_decode_fp8_paged": (_I, [_DP, _I, _I, _P, _P, _P, ctypes.c_float, _I, _I, _P, _I, _P, _P, _P, _P,
                                      _SZ, _P]),
        "mla_cache_append_fp8": (_I, [_DP, _I, _I, _P, _P, ctypes.c_float, ctypes.c_float, _I, _P, _P, _P, _P]),
        "mla_cache_append_fp8_paged": (_I, [_DP, _I, _I, _P, _P, ctypes.c_float, ctypes.c_float, _P, _P, _I, _I,
                                            _P, _I, _P, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmla.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        _declare(lib)
        _lib = lib
    return _lib


def lib() -> ctypes.CDLL:
    return load()


def _check(rc: int) -> None:
    if rc != MLA_OK:
        raise MlaError(rc, lib().mla_last_error().decode(errors="replace"))


def make_dims(dims) -> MlaDims:
    """Accepts workload.Dims or any object with the same fields."""
    scale = getattr(dims, "scale", None)
    return MlaDims(dims.H, dims.qk_nope, dims.qk_rope, dims.kv_lora, dims.v_head,
                   float(scale) if scale else 0.0, float(getattr(dims, "rope_base", 10000.0)))


# ------------------------------------------------------------------ helpers
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return MLA_F32
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _workspace(nbytes: int, device, ws):
    torch = _torch()
    if nbytes == 0:
        return ws, 0
    if ws is None or ws.numel() * ws.element_size() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device flag word."""
    flags = _I(0)
    rc = lib().mla_device_status(_stream(stream), ctypes.byref(flags))
    if rc not in (MLA_OK, MLA_ERR_DEVICE):
        _check(rc)
    return flags.value


def set_wait_limit_ns(ns: int) -> None:
    lib().mla_set_wait_limit_ns(int(ns))


_event_array = None


def set_kernel_events(events) -> None:
    """Record these torch.cuda.Event objects around the kernels of every later
    call on this thread (see mla_set_kernel_events); None switches it off."""
    global _event_array
    if not events:
        _event_array = None
        lib().mla_set_kernel_events(None, 0)
        return
    for e in events:
        if not e.cuda_event:
            e.record()  # torch creates the CUDA event lazily
    _event_array = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    lib().mla_set_kernel_events(_event_array, len(events))


def last_launch_names():
    """Kernels launched by the last call on this thread, in order."""
    return [n for n in lib().mla_last_launch_names().decode().split(",") if n]


# ------------------------------------------------------------------ ops
def kernels_per_call(kind: str, dims, B: int = 1, S: int = 1, dtype: int = MLA_BF16) -> int:
    """Kernels one decode ("decode") or sparse-decode ("sparse") call launches."""
    d = make_dims(dims)
    return lib().mla_decode_launch_count(ctypes.byref(d), dtype, B, S, 1 if kind == "sparse" else 0)


def decode_workspace_size(dims, dtype: int, B: int, S: int, T_cap: int) -> int:
    d = make_dims(dims)
    return lib().mla_decode_absorbed_workspace_size(ctypes.byref(d), dtype, B, S, T_cap)


def decode_absorbed(q, Lc, Rc, T, kv_b, dims, out=None, workspace=None, stream=None):
    """Weight-absorbed decode; q [B,S,H,qk], Lc [B,T_cap,kv_lora], Rc [B,T_cap,qk_rope]."""
    torch = _torch()
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    T_cap = Lc.shape[1]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_decode_absorbed_workspace_size(ctypes.byref(d), code, B, S, T_cap)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_decode_absorbed(ctypes.byref(d), code, B, S, _ptr(q), _ptr(Lc), _ptr(Rc), T_cap,
                                     _ptr(T), _ptr(kv_b), _ptr(out), _ptr(workspace), wsb,
                                     _stream(stream)))
    return out


def sparse_decode(q, Lc, Rc, T, kv_b, sel, nsel, dims, out=None, workspace=None, stream=None):
    """Absorbed decode over the keys sel[b,s,:nsel[b,s]] (sel [B,S,topk] int32)."""
    torch = _torch()
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    T_cap = Lc.shape[1]
    topk = sel.shape[2]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_sparse_decode_workspace_size(ctypes.byref(d), code, B, S, topk)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_sparse_decode(ctypes.byref(d), code, B, S, _ptr(q), _ptr(Lc), _ptr(Rc), T_cap,
                                   _ptr(T), _ptr(kv_b), _ptr(sel), _ptr(nsel), topk, _ptr(out),
                                   _ptr(workspace), wsb, _stream(stream)))
    return out


def sparse_decode_layers(layers, T, sel, nsel, dims, outs=None, w_o=None, ys=None, workspace=None, stream=None):
    """Sparse decode of L layers over one selection: layers is a list of
    (q, Lc, Rc, kv_b) per layer.  With w_o (a list of L [hidden, H*v_head]
    weights) each layer's output is also projected.  Returns the list of L
    outputs [B,S,H,v_head], and with w_o also the list of L projections
    [B*S, hidden]."""
    torch = _torch()
    L = len(layers)
    q0, Lc0 = layers[0][0], layers[0][1]
    B, S, H = q0.shape[0], q0.shape[1], q0.shape[2]
    T_cap = Lc0.shape[1]
    topk = sel.shape[2]
    code = _dtype_code(q0)
    for q, Lc, Rc, kv_b in layers:
        if q.shape != q0.shape or Lc.shape != Lc0.shape or q.dtype != q0.dtype:
            raise ValueError("every layer needs the shapes and dtype of layer 0")
    if outs is None:
        outs = [torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q0.device) for _ in range(L)]
    hidden = 0
    if w_o is not None:
        if len(w_o) != L:
            raise ValueError("one projection weight per layer")
        hidden = w_o[0].shape[0]
        if ys is None:
            ys = [torch.empty(B * S, hidden, dtype=torch.float32, device=q0.device) for _ in range(L)]
    d = make_dims(dims)
    need = lib().mla_sparse_decode_layers_workspace_size(ctypes.byref(d), code, B, S, topk, hidden)
    workspace, wsb = _workspace(need, q0.device, workspace)

    def arr(ts):
        return (ctypes.c_void_p * L)(*[_ptr(t) for t in ts])

    _check(lib().mla_sparse_decode_layers(
        ctypes.byref(d), code, L, B, S, arr([x[0] for x in layers]), arr([x[1] for x in layers]),
        arr([x[2] for x in layers]), T_cap, _ptr(T), arr([x[3] for x in layers]), _ptr(sel), _ptr(nsel), topk,
        arr(outs), arr(w_o) if w_o is not None else None, hidden, arr(ys) if w_o is not None else None,
        _ptr(workspace), wsb, _stream(stream)))
    return (outs, ys) if w_o is not None else outs


def prefill_naive(q, Lc, Rc, kv_b, dims, pos_base: int, out=None, workspace=None, stream=None):
    """Non-absorbed prefill of S new tokens at pos_base; Lc/Rc hold Tk = pos_base + S rows."""
    torch = _torch()
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_prefill_naive_workspace_size(ctypes.byref(d), code, B, S, pos_base)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_prefill_naive(ctypes.byref(d), code, B, S, pos_base, _ptr(q), _ptr(Lc), _ptr(Rc),
                                   _ptr(kv_b), _ptr(out), _ptr(workspace), wsb, _stream(stream)))
    return out


def index_scores(q_idx, w, Ic, T, out=None, stream=None):
    """DSA indexer scores [B,S,T_cap] (fp32; -inf past each query's position)."""
    torch = _torch()
    B, S, n_ih, hd = q_idx.shape
    T_cap = Ic.shape[1]
    if out is None:
        out = torch.empty(B, S, T_cap, dtype=torch.float32, device=q_idx.device)
    _check(lib().dsa_index_scores(B, S, n_ih, hd, _ptr(q_idx), _ptr(w), _ptr(Ic), T_cap, _ptr(T),
                                  _ptr(out), _stream(stream)))
    return out


def topk_select(scores, T, topk: int, S: Optional[int] = None, sel=None, nsel=None,
                workspace=None, stream=None) -> Tuple[object, object]:
    """Causal top-k selection: (sel [B,S,topk] ascending then -1, nsel [B,S])."""
    torch = _torch()
    B, S_, T_cap = scores.shape
    S = S_ if S is None else S
    if sel is None:
        sel = torch.empty(B, S, topk, dtype=torch.int32, device=scores.device)
    if nsel is None:
        nsel = torch.empty(B, S, dtype=torch.int32, device=scores.device)
    need = lib().dsa_topk_select_workspace_size(B, S, T_cap, topk)
    workspace, wsb = _workspace(need, scores.device, workspace)
    _check(lib().dsa_topk_select(B, S, _ptr(scores), T_cap, _ptr(T), topk, _ptr(sel), _ptr(nsel),
                                 _ptr(workspace), wsb, _stream(stream)))
    return sel, nsel


def cache_append(comp, kv_a_ln, T, Lc, Rc, dims, rms_eps: float, stream=None):
    """Writes the S new tokens of each sequence into Lc/Rc in place at rows
    T[b]-S+s: comp [B,S,kv_lora+qk_rope] (the kv_a output), kv_a_ln [kv_lora]."""
    B, S = comp.shape[0], comp.shape[1]
    T_cap = Lc.shape[1]
    code = _dtype_code(comp)
    for t in (kv_a_ln, Lc, Rc):
        if t.dtype != comp.dtype:
            raise TypeError("comp, kv_a_ln, Lc and Rc must share one dtype")
    d = make_dims(dims)
    _check(lib().mla_cache_append(ctypes.byref(d), code, B, S, _ptr(comp), _ptr(kv_a_ln), float(rms_eps),
                                  T_cap, _ptr(T), _ptr(Lc), _ptr(Rc), _stream(stream)))
    return Lc, Rc


def index_key_append(k_idx, ln_w, ln_b, T, Ic, rope_dim: int, ln_eps: float = 1e-6,
                     rope_base: float = 10000.0, stream=None):
    """Writes the indexer keys of the S new tokens (k_idx [B,S,index_hd] fp32)
    into Ic [B,T_cap,index_hd] in place: LayerNorm, then RoPE on the last rope_dim."""
    B, S, hd = k_idx.shape
    T_cap = Ic.shape[1]
    _check(lib().dsa_index_key_append(B, S, hd, int(rope_dim), _ptr(k_idx), _ptr(ln_w), _ptr(ln_b),
                                      float(ln_eps), float(rope_base), T_cap, _ptr(T), _ptr(Ic),
                                      _stream(stream)))
    return Ic


def o_proj(x, w_o, y=None, workspace=None, stream=None):
    """y [R, hidden] = x [R, in_dim] (fp32) times w_o [hidden, in_dim]^T."""
    torch = _torch()
    x2 = x.reshape(-1, x.shape[-1]) if x.dim() == 2 else x.reshape(x.shape[0] * x.shape[1], -1)
    R, in_dim = x2.shape
    hidden = w_o.shape[0]
    code = _dtype_code(w_o)
    if y is None:
        y = torch.empty(R, hidden, dtype=torch.float32, device=x.device)
    need = lib().mla_o_proj_workspace_size(R, in_dim, hidden, code)
    workspace, wsb = _workspace(need, x.device, workspace)
    _check(lib().mla_o_proj(R, in_dim, hidden, code, _ptr(w_o), _ptr(x2), _ptr(y), _ptr(workspace), wsb,
                            _stream(stream)))
    return y


def decode_oproj(q, Lc, Rc, T, kv_b, w_o, dims, y=None, workspace=None, stream=None):
    """mla_decode_absorbed then the output projection: y [B, S, hidden]."""
    torch = _torch()
    B, S = q.shape[0], q.shape[1]
    T_cap = Lc.shape[1]
    hidden = w_o.shape[0]
    code = _dtype_code(q)
    if y is None:
        y = torch.empty(B, S, hidden, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_decode_oproj_workspace_size(ctypes.byref(d), code, B, S, T_cap, hidden)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_decode_oproj(ctypes.byref(d), code, B, S, _ptr(q), _ptr(Lc), _ptr(Rc), T_cap, _ptr(T),
                                  _ptr(kv_b), _ptr(w_o), hidden, _ptr(y), _ptr(workspace), wsb, _stream(stream)))
    return y


def select(q_idx, w, Ic, T, topk: int, scores=None, sel=None, nsel=None, workspace=None, stream=None):
    """Fused DSA selection: index scores then causal top-k -> (scores, sel, nsel)."""
    torch = _torch()
    B, S, n_ih, hd = q_idx.shape
    T_cap = Ic.shape[1]
    dev = q_idx.device
    if scores is None:
        scores = torch.empty(B, S, T_cap, dtype=torch.float32, device=dev)
    if sel is None:
        sel = torch.empty(B, S, topk, dtype=torch.int32, device=dev)
    if nsel is None:
        nsel = torch.empty(B, S, dtype=torch.int32, device=dev)
    need = lib().dsa_select_workspace_size(B, S, n_ih, hd, T_cap, topk)
    workspace, wsb = _workspace(need, dev, workspace)
    _check(lib().dsa_select(B, S, n_ih, hd, _ptr(q_idx), _ptr(w), _ptr(Ic), T_cap, _ptr(T), topk, _ptr(scores),
                            _ptr(sel), _ptr(nsel), _ptr(workspace), wsb, _stream(stream)))
    return scores, sel, nsel


# ------------------------------------------------------------------ paged cache
def decode_paged(q, Lc_pages, Rc_pages, block_table, T, kv_b, dims, out=None, workspace=None, stream=None):
    """Absorbed decode over a page pool: Lc_pages [num_pages, page_size, kv_lora],
    Rc_pages [num_pages, page_size, qk_rope], block_table [B, max_pages] int32."""
    torch = _torch()
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    num_pages, page_size = Lc_pages.shape[0], Lc_pages.shape[1]
    max_pages = block_table.shape[1]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_decode_paged_workspace_size(ctypes.byref(d), code, B, S, max_pages, page_size)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_decode_paged(ctypes.byref(d), code, B, S, _ptr(q), _ptr(Lc_pages), _ptr(Rc_pages), num_pages,
                                  page_size, _ptr(block_table), max_pages, _ptr(T), _ptr(kv_b), _ptr(out),
                                  _ptr(workspace), wsb, _stream(stream)))
    return out


def sparse_decode_paged(q, Lc_pages, Rc_pages, block_table, T, kv_b, sel, nsel, dims, out=None, workspace=None,
                        stream=None):
    """Absorbed decode over the selected keys of a paged cache (sel holds token indices)."""
    torch = _torch()
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    num_pages, page_size = Lc_pages.shape[0], Lc_pages.shape[1]
    max_pages = block_table.shape[1]
    topk = sel.shape[2]
    code = _dtype_code(q)
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_sparse_decode_workspace_size(ctypes.byref(d), code, B, S, topk)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_sparse_decode_paged(ctypes.byref(d), code, B, S, _ptr(q), _ptr(Lc_pages), _ptr(Rc_pages),
                                         num_pages, page_size, _ptr(block_table), max_pages, _ptr(T), _ptr(kv_b),
                                         _ptr(sel), _ptr(nsel), topk, _ptr(out), _ptr(workspace), wsb,
                                         _stream(stream)))
    return out


def cache_append_paged(comp, kv_a_ln, block_table, T, Lc_pages, Rc_pages, dims, rms_eps: float, stream=None):
    """mla_cache_append into the page pools (in place)."""
    B, S = comp.shape[0], comp.shape[1]
    num_pages, page_size = Lc_pages.shape[0], Lc_pages.shape[1]
    code = _dtype_code(comp)
    for t in (kv_a_ln, Lc_pages, Rc_pages):
        if t.dtype != comp.dtype:
            raise TypeError("comp, kv_a_ln and the pools must share one dtype")
    d = make_dims(dims)
    _check(lib().mla_cache_append_paged(ctypes.byref(d), code, B, S, _ptr(comp), _ptr(kv_a_ln), float(rms_eps),
                                        _ptr(Lc_pages), _ptr(Rc_pages), num_pages, page_size, _ptr(block_table),
                                        block_table.shape[1], _ptr(T), _stream(stream)))
    return Lc_pages, Rc_pages


# ------------------------------------------------------------- FP8 latent cache
def _need_bf16(*ts):
    torch = _torch()
    for t in ts:
        if t.dtype != torch.bfloat16:
            raise TypeError("the FP8 cache entry points take bf16 q, Rc, kv_b and comp")


def _need_u8(t):
    torch = _torch()
    if t.dtype != torch.uint8:
        raise TypeError("the FP8 latent cache holds uint8 E4M3 codes")


def decode_fp8(q, Lc8, Rc, T, kv_b, dims, lat_scale: float, out=None, workspace=None, stream=None):
    """Absorbed decode over an FP8 latent cache: Lc8 [B, T_cap, kv_lora] uint8
    E4M3 codes (latent = lat_scale * code), Rc [B, T_cap, qk_rope] bf16."""
    torch = _torch()
    _need_bf16(q, Rc, kv_b)
    _need_u8(Lc8)
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    T_cap = Lc8.shape[1]
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_decode_fp8_workspace_size(ctypes.byref(d), B, S, T_cap)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_decode_fp8(ctypes.byref(d), B, S, _ptr(q), _ptr(Lc8), _ptr(Rc), float(lat_scale), T_cap,
                                _ptr(T), _ptr(kv_b), _ptr(out), _ptr(workspace), wsb, _stream(stream)))
    return out


def decode_fp8_paged(q, Lc8_pages, Rc_pages, block_table, T, kv_b, dims, lat_scale: float, out=None,
                     workspace=None, stream=None):
    """decode_fp8 over page pools: Lc8_pages [num_pages, page_size, kv_lora] uint8,
    Rc_pages [num_pages, page_size, qk_rope] bf16, block_table [B, max_pages] int32."""
    torch = _torch()
    _need_bf16(q, Rc_pages, kv_b)
    _need_u8(Lc8_pages)
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    num_pages, page_size = Lc8_pages.shape[0], Lc8_pages.shape[1]
    max_pages = block_table.shape[1]
    if out is None:
        out = torch.empty(B, S, H, dims.v_head, dtype=torch.float32, device=q.device)
    d = make_dims(dims)
    need = lib().mla_decode_fp8_workspace_size(ctypes.byref(d), B, S, max_pages * page_size)
    workspace, wsb = _workspace(need, q.device, workspace)
    _check(lib().mla_decode_fp8_paged(ctypes.byref(d), B, S, _ptr(q), _ptr(Lc8_pages), _ptr(Rc_pages),
                                      float(lat_scale), num_pages, page_size, _ptr(block_table), max_pages, _ptr(T),
                                      _ptr(kv_b), _ptr(out), _ptr(workspace), wsb, _stream(stream)))
    return out


def cache_append_fp8(comp, kv_a_ln, T, Lc8, Rc, dims, rms_eps: float, lat_scale: float, stream=None):
    """mla_cache_append into the FP8 cache (in place): Lc8 uint8 codes, Rc bf16."""
    _need_bf16(comp, kv_a_ln, Rc)
    _need_u8(Lc8)
    B, S = comp.shape[0], comp.shape[1]
    d = make_dims(dims)
    _check(lib().mla_cache_append_fp8(ctypes.byref(d), B, S, _ptr(comp), _ptr(kv_a_ln), float(rms_eps),
                                      float(lat_scale), Lc8.shape[1], _ptr(T), _ptr(Lc8), _ptr(Rc), _stream(stream)))
    return Lc8, Rc


def cache_append_fp8_paged(comp, kv_a_ln, block_table, T, Lc8_pages, Rc_pages, dims, rms_eps: float,
                           lat_scale: float, stream=None):
    """cache_append_fp8 into the page pools (in place)."""
    _need_bf16(comp, kv_a_ln, Rc_pages)
    _need_u8(Lc8_pages)
    B, S = comp.shape[0], comp.shape[1]
    num_pages, page_size = Lc8_pages.shape[0], Lc8_pages.shape[1]
    d = make_dims(dims)
    _check(lib().mla_cache_append_fp8_paged(ctypes.byref(d), B, S, _ptr(comp), _ptr(kv_a_ln), float(rms_eps),
                                            float(lat_scale), _ptr(Lc8_pages), _ptr(Rc_pages), num_pages, page_size,
                                            _ptr(block_table), block_table.shape[1], _ptr(T), _stream(stream)))
    return Lc8_pages, Rc_pages
