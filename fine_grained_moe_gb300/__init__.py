"""Python binding of the GB300 batch-1 fine-grained MoE verify-step library.

A thin ctypes layer over the C ABI in ``include/fgm.h``: it turns torch CUDA
tensors into device pointers, picks the current CUDA stream and raises on a
non-zero status. Every stage of the step runs in the CUDA library
``libfgm.so``; there is no other implementation in this package, so calling
any function without the built library raises.

Build the library with ``python -m fine_grained_moe_gb300.build`` (or the
repository's ``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import traffic  # noqa: F401  (byte accounting used by the benchmark)

HIDDEN = 2816
FFN = 704
EXPERTS = 128
N_EXPERTS = 129
TOPK = 8
MAX_M = 8
MAX_LAYERS = 48

STATUS_NONFINITE_LOGITS = 1
STATUS_WAIT_TIMEOUT = 2
PATH_FUSED = 0    # one persistent cooperative kernel per call (TMA ring + mma.sync tiles; tcgen05 down products at M <= 5)
PATH_STAGED = 1   # one launch per stage, fp32 CUDA-core arithmetic
PATH_FUSED_TC = 2  # as PATH_FUSED, with the FP8 lm_head on tcgen05 tensor-memory tiles fed by TMA tensor copies
PATH_FUSED_MMA = 3  # as PATH_FUSED, with the down products on mma.sync at every M (comparison path)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfgm.so")
_lib = None


class FgmError(RuntimeError):
    pass


class fgm_layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("router_w", "router_b", "gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]


class fgm_mlp(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")] + \
               [("width", ctypes.c_int)]


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FgmError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run python -m fine_grained_moe_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        vp, ci, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        LP = ctypes.POINTER(fgm_layer)
        sig = {
            "fgm_workspace_bytes": (sz, [ci, i64]),
            "fgm_workspace_init": (ci, [vp, sz, vp]),
            "fgm_moe_layer_fwd": (ci, [LP, vp, vp, ci, vp, vp, vp, sz, vp]),
            "fgm_moe_layer_fwd_noalloc": (ci, [LP, vp, vp, ci, vp, vp, vp]),
            "fgm_moe_stack_fwd": (ci, [LP, ci, vp, vp, ci, vp, vp, sz, vp]),
            "fgm_moe_layer_dense_fwd": (ci, [LP, ctypes.POINTER(fgm_mlp), vp, vp, ci, vp, vp, vp, sz, vp]),
            "fgm_moe_stack_dense_fwd": (ci, [LP, ctypes.POINTER(fgm_mlp), ci, vp, vp, ci, vp, vp, sz, vp]),
            "fgm_verify_step_dense": (ci, [LP, ctypes.POINTER(fgm_mlp), ci, vp, i64, vp, vp, ci, vp, vp, vp, sz,
                                           vp]),
            "fgm_lm_head_argmax": (ci, [vp, i64, vp, ci, vp, vp, vp, sz, vp]),
            "fgm_lm_head_argmax_fp8": (ci, [vp, vp, i64, vp, ci, vp, vp, vp, sz, vp]),
            "fgm_spec_verify": (ci, [vp, vp, ci, vp, vp]),
            "fgm_verify_step": (ci, [LP, ci, vp, i64, vp, vp, ci, vp, vp, vp, sz, vp]),
            "fgm_verify_step_host": (ci, [LP, ci, vp, i64, vp, vp, ci, vp, vp, sz, vp]),
            "fgm_verify_step_fp8_head": (ci, [LP, ci, vp, vp, i64, vp, vp, ci, vp, vp, vp, sz, vp]),
            "fgm_lm_head_sample": (ci, [vp, i64, vp, ci, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "fgm_verify_step_sample": (ci, [LP, ci, vp, i64, vp, vp, ci, ctypes.c_float, vp, vp, vp, vp, vp, vp,
                                            sz, vp]),
            "fgm_read_status": (ci, [vp, sz, ci, vp, vp]),
            "fgm_select_path": (ci, [ci]),
            "fgm_set_phase_trace": (ci, [vp, sz]),
            "fgm_debug_stall_next_launch": (ci, []),
            "fgm_debug_stall_next_launch_at": (ci, [ci]),
            "fgm_read_wait_report": (ci, [vp, sz, vp, vp]),
            "fgm_set_wait_limit_ns": (ctypes.c_longlong, [ctypes.c_longlong]),
            "fgm_last_error": (ctypes.c_char_p, []),
            "fgm_version": (ci, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        msg = lib().fgm_last_error().decode(errors="replace")
        raise FgmError(f"fgm error {rc}: {msg}")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise FgmError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise FgmError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _m(x: torch.Tensor) -> int:
    if x.dim() != 2 or x.shape[1] != HIDDEN or x.dtype != torch.bfloat16:
        raise FgmError(f"expected bf16 [M, {HIDDEN}] activations, got {tuple(x.shape)} {x.dtype}")
    return int(x.shape[0])


def _check_like(name: str, t: torch.Tensor, x: torch.Tensor) -> None:
    """Output rows must match the input rows: bf16 [M, 2816] on x's device."""
    if tuple(t.shape) != tuple(x.shape) or t.dtype != torch.bfloat16 or t.device != x.device:
        raise FgmError(f"{name}: expected bf16 {tuple(x.shape)} on {x.device}, got "
                       f"{tuple(t.shape)} {t.dtype} on {t.device}")


def _check_topk(M: int, x: torch.Tensor, topk_ids: torch.Tensor | None, topk_w: torch.Tensor | None) -> None:
    """Optional routing outputs: int32 / float32 [M, 8] on x's device."""
    for name, t, dt in (("topk_ids", topk_ids, torch.int32), ("topk_w", topk_w, torch.float32)):
        if t is not None and (tuple(t.shape) != (M, TOPK) or t.dtype != dt or t.device != x.device):
            raise FgmError(f"{name}: expected {dt} [{M}, {TOPK}] on {x.device}, got "
                           f"{tuple(t.shape)} {t.dtype} on {t.device}")


def select_path(path: int) -> int:
    """Selects the execution path (PATH_FUSED, PATH_STAGED, PATH_FUSED_TC or PATH_FUSED_MMA); returns the previous one."""
    return int(lib().fgm_select_path(int(path)))


def set_wait_limit_ns(ns: int) -> int:
    """Bound on every wait inside the persistent kernel (ns < 0 only queries)."""
    return int(lib().fgm_set_wait_limit_ns(int(ns)))


def set_phase_trace(buf: torch.Tensor | None) -> None:
    """Profiling aid: record per-CTA phase timestamps of later persistent-kernel
    launches into an int64 CUDA tensor (None stops)."""
    if buf is None:
        _check(lib().fgm_set_phase_trace(None, 0))
    else:
        if buf.dtype != torch.int64:
            raise FgmError("trace buffer must be int64")
        _check(lib().fgm_set_phase_trace(_ptr(buf), buf.numel()))


def debug_stall_next_launch(layer: int = 0) -> None:
    """Test hook: the next persistent-kernel launch waits, at the start of
    ``layer``, on a barrier that can never complete, so its wait limit must run
    out."""
    if layer == 0:
        _check(lib().fgm_debug_stall_next_launch())
    else:
        _check(lib().fgm_debug_stall_next_launch_at(int(layer)))


def workspace_bytes(M: int = MAX_M, V: int = 0) -> int:
    return int(lib().fgm_workspace_bytes(int(M), int(V)))


class Workspace:
    """Device scratch for the library's calls (one per concurrent stream)."""

    def __init__(self, device=None, M: int = MAX_M, V: int = 0):
        self.nbytes = workspace_bytes(M, V)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.t = self.buf[off:off + self.nbytes]
        _check(lib().fgm_workspace_init(_ptr(self.t), self.nbytes, _stream(None)))

    @property
    def ptr(self):
        return _ptr(self.t)

    def wait_report(self) -> list[int]:
        """{site, block, warp, index} of the first wait that ran out (see fgm.h)."""
        out = (ctypes.c_int32 * 4)()
        _check(lib().fgm_read_wait_report(self.ptr, self.nbytes, out, _stream(None)))
        return list(out)

    def status(self, clear: bool = True) -> int:
        out = ctypes.c_int32(0)
        _check(lib().fgm_read_status(self.ptr, self.nbytes, int(clear), ctypes.byref(out), _stream(None)))
        return int(out.value)


@dataclass
class Layer:
    """One layer's device tensors (see ``fgm_layer`` in include/fgm.h)."""
    router_w: torch.Tensor
    router_b: torch.Tensor | None
    gate_q: torch.Tensor
    gate_s: torch.Tensor
    up_q: torch.Tensor
    up_s: torch.Tensor
    down_q: torch.Tensor
    down_s: torch.Tensor

    @classmethod
    def from_dict(cls, p: dict) -> "Layer":
        return cls(**{k: p[k] for k in ("router_w", "router_b", "gate_q", "gate_s", "up_q", "up_s",
                                        "down_q", "down_s")})

    def struct(self) -> fgm_layer:
        shapes = {"router_w": ((EXPERTS, HIDDEN), torch.bfloat16),
                  "gate_q": ((N_EXPERTS, FFN, HIDDEN), torch.uint8),
                  "up_q": ((N_EXPERTS, FFN, HIDDEN), torch.uint8),
                  "down_q": ((N_EXPERTS, HIDDEN, FFN), torch.uint8),
                  "gate_s": ((N_EXPERTS, FFN), torch.float32),
                  "up_s": ((N_EXPERTS, FFN), torch.float32),
                  "down_s": ((N_EXPERTS, HIDDEN), torch.float32)}
        for name, (shape, dt) in shapes.items():
            t = getattr(self, name)
            if tuple(t.shape) != shape or t.dtype != dt:
                raise FgmError(f"{name}: expected {shape} {dt}, got {tuple(t.shape)} {t.dtype}")
        if self.router_b is not None and (tuple(self.router_b.shape) != (EXPERTS,)
                                          or self.router_b.dtype != torch.float32):
            raise FgmError("router_b: expected float32 [128]")
        return fgm_layer(*[(_ptr(getattr(self, n)) or ctypes.c_void_p(0)).value for n in
                           ("router_w", "router_b", "gate_q", "gate_s", "up_q", "up_s", "down_q",
                            "down_s")])


def _layers_array(layers) -> ctypes.Array:
    structs = [(l if isinstance(l, Layer) else Layer.from_dict(l)).struct() for l in layers]
    arr = (fgm_layer * len(structs))(*structs)
    return arr


def _ws(ws: Workspace | None, device) -> Workspace:
    return ws if ws is not None else Workspace(device)


# ---------------------------------------------------------------- entry points
def moe_layer_fwd(layer, x: torch.Tensor, y: torch.Tensor | None = None,
                  topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None,
                  ws: Workspace | None = None, stream=None) -> torch.Tensor:
    """One MoE layer (no norm, no residual) on bf16 x[M, 2816]; returns bf16 y."""
    M = _m(x)
    y = torch.empty_like(x) if y is None else y
    _check_like("y", y, x)
    _check_topk(M, x, topk_ids, topk_w)
    ws = _ws(ws, x.device)
    L = (layer if isinstance(layer, Layer) else Layer.from_dict(layer)).struct()
    _check(lib().fgm_moe_layer_fwd(ctypes.byref(L), _ptr(x), _ptr(y), M, _ptr(topk_ids), _ptr(topk_w),
                                   ws.ptr, ws.nbytes, _stream(stream)))
    return y


def _mlp_struct(mlp: dict) -> fgm_mlp:
    W = int(mlp["gate_q"].shape[0])
    shapes = {"gate_q": ((W, HIDDEN), torch.uint8), "up_q": ((W, HIDDEN), torch.uint8),
              "down_q": ((HIDDEN, W), torch.uint8), "gate_s": ((W,), torch.float32),
              "up_s": ((W,), torch.float32), "down_s": ((HIDDEN,), torch.float32)}
    for name, (shape, dt) in shapes.items():
        t = mlp[name]
        if tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous():
            raise FgmError(f"dense {name}: expected contiguous {shape} {dt}, got {tuple(t.shape)} {t.dtype}")
    return fgm_mlp(*[_ptr(mlp[n]).value for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")],
                   W)


def moe_layer_dense_fwd(layer, dense: dict, x: torch.Tensor, y: torch.Tensor | None = None,
                        topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None,
                        ws: Workspace | None = None, stream=None) -> torch.Tensor:
    """One MoE layer with the always-on dense MLP `dense` (gate_q/up_q [W, 2816],
    down_q [2816, W], fp32 row scales; W a multiple of 704 up to 2112) in place
    of the shared expert; returns bf16 y."""
    M = _m(x)
    y = torch.empty_like(x) if y is None else y
    _check_like("y", y, x)
    _check_topk(M, x, topk_ids, topk_w)
    ws = _ws(ws, x.device)
    L = (layer if isinstance(layer, Layer) else Layer.from_dict(layer)).struct()
    D = _mlp_struct(dense)
    _check(lib().fgm_moe_layer_dense_fwd(ctypes.byref(L), ctypes.byref(D), _ptr(x), _ptr(y), M, _ptr(topk_ids),
                                         _ptr(topk_w), ws.ptr, ws.nbytes, _stream(stream)))
    return y


def moe_layer_fwd_noalloc(layer, x: torch.Tensor, y: torch.Tensor,
                          topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """moe_layer_fwd on the library's built-in device scratch instead of a
    Workspace, for callers that must not allocate while they run (``y`` is
    therefore required). At most 8 tokens. Calls whose GPU work overlaps on
    one device race on that scratch; make the first call on a device before
    any stream capture starts, since it looks the scratch up."""
    M = _m(x)
    _check_like("y", y, x)
    _check_topk(M, x, topk_ids, topk_w)
    L = (layer if isinstance(layer, Layer) else Layer.from_dict(layer)).struct()
    _check(lib().fgm_moe_layer_fwd_noalloc(ctypes.byref(L), _ptr(x), _ptr(y), M, _ptr(topk_ids),
                                           _ptr(topk_w), _stream(stream)))
    return y


def moe_stack_fwd(layers, x: torch.Tensor, y: torch.Tensor | None = None,
                  ids_trace: torch.Tensor | None = None, ws: Workspace | None = None,
                  stream=None) -> torch.Tensor:
    """The stack h <- h + layer(RMSNorm(h)) over ``layers``; returns bf16 h."""
    M = _m(x)
    y = torch.empty_like(x) if y is None else y
    _check_like("y", y, x)
    if ids_trace is not None and (tuple(ids_trace.shape) != (len(layers), M, TOPK)
                                  or ids_trace.dtype != torch.int32 or ids_trace.device != x.device):
        raise FgmError(f"ids_trace: expected int32 [{len(layers)}, {M}, {TOPK}] on {x.device}")
    ws = _ws(ws, x.device)
    arr = _layers_array(layers)
    _check(lib().fgm_moe_stack_fwd(arr, len(arr), _ptr(x), _ptr(y), M, _ptr(ids_trace), ws.ptr,
                                   ws.nbytes, _stream(stream)))
    return y


def _mlps_array(mlps, n_layers: int) -> ctypes.Array:
    if len(mlps) != n_layers:
        raise FgmError(f"mlps: expected one dense MLP per layer ({n_layers}), got {len(mlps)}")
    return (fgm_mlp * n_layers)(*[_mlp_struct(m) for m in mlps])


def moe_stack_dense_fwd(layers, mlps, x: torch.Tensor, y: torch.Tensor | None = None,
                        ids_trace: torch.Tensor | None = None, ws: Workspace | None = None,
                        stream=None) -> torch.Tensor:
    """The stack with the dense MLP ``mlps[l]`` (dicts as for moe_layer_dense_fwd)
    in place of layer l's shared expert; returns bf16 h."""
    M = _m(x)
    y = torch.empty_like(x) if y is None else y
    _check_like("y", y, x)
    if ids_trace is not None and (tuple(ids_trace.shape) != (len(layers), M, TOPK)
                                  or ids_trace.dtype != torch.int32 or ids_trace.device != x.device):
        raise FgmError(f"ids_trace: expected int32 [{len(layers)}, {M}, {TOPK}] on {x.device}")
    ws = _ws(ws, x.device)
    arr = _layers_array(layers)
    mlp_arr = _mlps_array(mlps, len(arr))
    _check(lib().fgm_moe_stack_dense_fwd(arr, mlp_arr, len(arr), _ptr(x), _ptr(y), M, _ptr(ids_trace), ws.ptr,
                                         ws.nbytes, _stream(stream)))
    return y


def lm_head_argmax(emb: torch.Tensor, h: torch.Tensor, argmax: torch.Tensor | None = None,
                   maxlogit: torch.Tensor | None = None, ws: Workspace | None = None,
                   stream=None) -> torch.Tensor:
    """argmax_v emb[v] . h[t] for each of the M rows of bf16 h; returns int32 [M]."""
    M = _m(h)
    V = int(emb.shape[0])
    argmax = torch.empty(M, dtype=torch.int32, device=h.device) if argmax is None else argmax
    ws = _ws(ws, h.device)
    _check(lib().fgm_lm_head_argmax(_ptr(emb), V, _ptr(h), M, _ptr(argmax), _ptr(maxlogit), ws.ptr,
                                    ws.nbytes, _stream(stream)))
    return argmax


def _fp8_rows(emb_q: torch.Tensor, emb_s: torch.Tensor) -> int:
    if emb_q.dim() != 2 or emb_q.shape[1] != HIDDEN or emb_q.dtype != torch.uint8:
        raise FgmError(f"expected uint8 [V, {HIDDEN}] E4M3 codes, got {tuple(emb_q.shape)} {emb_q.dtype}")
    if emb_s.dtype != torch.float32 or tuple(emb_s.shape) != (emb_q.shape[0],):
        raise FgmError(f"expected fp32 [{emb_q.shape[0]}] row scales, got {tuple(emb_s.shape)} {emb_s.dtype}")
    return int(emb_q.shape[0])


def lm_head_argmax_fp8(emb_q: torch.Tensor, emb_s: torch.Tensor, h: torch.Tensor,
                       argmax: torch.Tensor | None = None, maxlogit: torch.Tensor | None = None,
                       ws: Workspace | None = None, stream=None) -> torch.Tensor:
    """argmax_v emb_s[v] * (e4m3(emb_q[v]) . h[t]) for each of the M rows of bf16 h;
    returns int32 [M]."""
    M = _m(h)
    V = _fp8_rows(emb_q, emb_s)
    argmax = torch.empty(M, dtype=torch.int32, device=h.device) if argmax is None else argmax
    ws = _ws(ws, h.device)
    _check(lib().fgm_lm_head_argmax_fp8(_ptr(emb_q), _ptr(emb_s), V, _ptr(h), M, _ptr(argmax),
                                        _ptr(maxlogit), ws.ptr, ws.nbytes, _stream(stream)))
    return argmax


def _sample_args(M: int, V: int, device, draft, u_acc, u_next, z, out):
    if u_next is None or u_next.dtype != torch.float32 or u_next.numel() != M:
        raise FgmError(f"u_next must be fp32 [{M}]")
    if M > 1 and (draft is None or u_acc is None or u_acc.dtype != torch.float32 or u_acc.numel() != M - 1
                  or draft.dtype != torch.int32 or draft.numel() != M - 1):
        raise FgmError(f"draft (int32) and u_acc (fp32) must have M - 1 = {M - 1} elements")
    z = torch.empty((M, V), dtype=torch.float32, device=device) if z is None else z
    if z.dtype != torch.float32 or tuple(z.shape) != (M, V) or not z.is_contiguous():
        raise FgmError(f"z must be contiguous fp32 [{M}, {V}]")
    out = torch.empty(2, dtype=torch.int32, device=device) if out is None else out
    return z, out


def lm_head_sample(emb: torch.Tensor, h: torch.Tensor, T: float, draft: torch.Tensor | None,
                   u_acc: torch.Tensor | None, u_next: torch.Tensor, z: torch.Tensor | None = None,
                   argmax: torch.Tensor | None = None, out: torch.Tensor | None = None,
                   ws: Workspace | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Speculative sampling verify at temperature T on the lm_head logits of the
    M bf16 rows h; returns (out int32 [2] = {accepted drafts, emitted token},
    z fp32 [M, V] logits)."""
    M = _m(h)
    V = int(emb.shape[0])
    z, out = _sample_args(M, V, h.device, draft, u_acc, u_next, z, out)
    ws = _ws(ws, h.device)
    _check(lib().fgm_lm_head_sample(_ptr(emb), V, _ptr(h), M, float(T), _ptr(draft) if M > 1 else None,
                                    _ptr(u_acc) if M > 1 else None, _ptr(u_next), _ptr(z), _ptr(argmax),
                                    _ptr(out), ws.ptr, ws.nbytes, _stream(stream)))
    return out, z


def verify_step_sample(layers, emb: torch.Tensor, x: torch.Tensor, T: float, draft: torch.Tensor | None,
                       u_acc: torch.Tensor | None, u_next: torch.Tensor, z: torch.Tensor | None = None,
                       argmax: torch.Tensor | None = None, out: torch.Tensor | None = None,
                       ws: Workspace | None = None, stream=None, _arr=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Stack + final RMSNorm + lm_head + speculative sampling at temperature T;
    returns (out int32 [2] = {accepted drafts, emitted token}, z fp32 [M, V])."""
    M = _m(x)
    V = int(emb.shape[0])
    z, out = _sample_args(M, V, x.device, draft, u_acc, u_next, z, out)
    ws = _ws(ws, x.device)
    arr = _layers_array(layers) if _arr is None else _arr
    _check(lib().fgm_verify_step_sample(arr, len(arr), _ptr(emb), V, _ptr(x), _ptr(draft) if M > 1 else None, M,
                                        float(T), _ptr(u_acc) if M > 1 else None, _ptr(u_next), _ptr(z),
                                        _ptr(argmax), _ptr(out), ws.ptr, ws.nbytes, _stream(stream)))
    return out, z


def spec_verify(target: torch.Tensor, draft: torch.Tensor, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Greedy acceptance; returns int32 [2] = {accepted drafts, next token}."""
    M = int(target.shape[0])
    out = torch.empty(2, dtype=torch.int32, device=target.device) if out is None else out
    _check(lib().fgm_spec_verify(_ptr(target), _ptr(draft) if M > 1 else None, M, _ptr(out),
                                 _stream(stream)))
    return out


def verify_step(layers, emb: torch.Tensor, x: torch.Tensor, draft: torch.Tensor | None,
                out: torch.Tensor | None = None, argmax: torch.Tensor | None = None,
                ws: Workspace | None = None, stream=None, _arr=None) -> torch.Tensor:
    """Stack + final RMSNorm + lm_head argmax + greedy acceptance; returns int32
    [2] = {accepted drafts, next token} on the device."""
    M = _m(x)
    out = torch.empty(2, dtype=torch.int32, device=x.device) if out is None else out
    ws = _ws(ws, x.device)
    arr = _layers_array(layers) if _arr is None else _arr
    _check(lib().fgm_verify_step(arr, len(arr), _ptr(emb), int(emb.shape[0]), _ptr(x),
                                 _ptr(draft) if M > 1 else None, M, _ptr(argmax), _ptr(out), ws.ptr,
                                 ws.nbytes, _stream(stream)))
    return out


def verify_step_dense(layers, mlps, emb: torch.Tensor, x: torch.Tensor, draft: torch.Tensor | None,
                      out: torch.Tensor | None = None, argmax: torch.Tensor | None = None,
                      ws: Workspace | None = None, stream=None, _arr=None, _mlp_arr=None) -> torch.Tensor:
    """verify_step on the stack with a dense MLP per layer (see moe_stack_dense_fwd);
    returns int32 [2] = {accepted drafts, next token} on the device."""
    M = _m(x)
    out = torch.empty(2, dtype=torch.int32, device=x.device) if out is None else out
    ws = _ws(ws, x.device)
    arr = _layers_array(layers) if _arr is None else _arr
    mlp_arr = _mlps_array(mlps, len(arr)) if _mlp_arr is None else _mlp_arr
    _check(lib().fgm_verify_step_dense(arr, mlp_arr, len(arr), _ptr(emb), int(emb.shape[0]), _ptr(x),
                                       _ptr(draft) if M > 1 else None, M, _ptr(argmax), _ptr(out), ws.ptr,
                                       ws.nbytes, _stream(stream)))
    return out


def mlps_array(mlps):
    """Pre-marshalled dense MLP table, reusable across calls (pass as ``_mlp_arr``)."""
    return _mlps_array(mlps, len(mlps))


def verify_step_fp8_head(layers, emb_q: torch.Tensor, emb_s: torch.Tensor, x: torch.Tensor,
                         draft: torch.Tensor | None, out: torch.Tensor | None = None,
                         argmax: torch.Tensor | None = None, ws: Workspace | None = None, stream=None,
                         _arr=None) -> torch.Tensor:
    """verify_step with the FP8 lm_head (E4M3 rows emb_q, fp32 row scales emb_s);
    returns int32 [2] = {accepted drafts, next token} on the device."""
    M = _m(x)
    V = _fp8_rows(emb_q, emb_s)
    out = torch.empty(2, dtype=torch.int32, device=x.device) if out is None else out
    ws = _ws(ws, x.device)
    arr = _layers_array(layers) if _arr is None else _arr
    _check(lib().fgm_verify_step_fp8_head(arr, len(arr), _ptr(emb_q), _ptr(emb_s), V, _ptr(x),
                                          _ptr(draft) if M > 1 else None, M, _ptr(argmax), _ptr(out),
                                          ws.ptr, ws.nbytes, _stream(stream)))
    return out


def verify_step_host(layers, emb: torch.Tensor, x_host: torch.Tensor, draft_host: torch.Tensor | None,
                     out_host: torch.Tensor | None = None, ws: Workspace | None = None,
                     stream=None, _arr=None) -> torch.Tensor:
    """verify_step with host (ideally pinned) x/draft/out; synchronises."""
    if x_host.is_cuda:
        raise FgmError("x_host must be a host tensor")
    M = int(x_host.shape[0])
    out_host = torch.empty(2, dtype=torch.int32) if out_host is None else out_host
    ws = _ws(ws, emb.device)
    arr = _layers_array(layers) if _arr is None else _arr
    dp = ctypes.c_void_p(draft_host.data_ptr()) if (draft_host is not None and M > 1) else None
    _check(lib().fgm_verify_step_host(arr, len(arr), _ptr(emb), int(emb.shape[0]),
                                      ctypes.c_void_p(x_host.data_ptr()), dp, M,
                                      ctypes.c_void_p(out_host.data_ptr()), ws.ptr, ws.nbytes,
                                      _stream(stream)))
    return out_host


def layers_array(layers):
    """Pre-marshalled layer table, reusable across calls (pass as ``_arr``)."""
    return _layers_array(layers)
