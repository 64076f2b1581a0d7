"""Oracle for the batch-1 fine-grained MoE verify step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, the smoke check and the
benchmark's CPU-baseline leg, never by the product package. The arithmetic
lives in ``oracle.c`` (plain C, fp64 accumulation, formula decoding of E4M3
and bf16); this module only marshals numpy arrays.

What each function follows is stated in ``oracle.c``; the short version:
router = softmax over all experts, top-k (ties to the lower index),
renormalised; expert = GELU-tanh(gate) * up then down, each weight row
dequantised from E4M3 with its fp32 row scale; layer = routed experts
weighted by the router plus the shared expert with weight 1; stack layer =
h + layer(RMSNorm(h)); lm_head = bf16 embedding rows dotted with the final
hidden rows, argmax with ties to the lower index (the FP8 variant: E4M3
rows times their fp32 row scale); greedy verify = longest
draft prefix equal to the target argmax of the preceding position.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O3, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-D_DEFAULT_SOURCE",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("F", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("n_shared", ctypes.c_int)]


class _Layer(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_b", ctypes.c_void_p),
                ("gate_q", ctypes.c_void_p), ("gate_s", ctypes.c_void_p),
                ("up_q", ctypes.c_void_p), ("up_s", ctypes.c_void_p),
                ("down_q", ctypes.c_void_p), ("down_s", ctypes.c_void_p)]


class _Mlp(ctypes.Structure):
    _fields_ = [("F", ctypes.c_int),
                ("gate_q", ctypes.c_void_p), ("gate_s", ctypes.c_void_p),
                ("up_q", ctypes.c_void_p), ("up_s", ctypes.c_void_p),
                ("down_q", ctypes.c_void_p), ("down_s", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, ci, cd = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.fgmo_e4m3_decode.restype = cd
        L.fgmo_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.fgmo_e4m3_encode.restype = ctypes.c_uint8
        L.fgmo_e4m3_encode.argtypes = [cd]
        L.fgmo_bf16_round.restype = ctypes.c_uint16
        L.fgmo_bf16_round.argtypes = [cd]
        L.fgmo_gelu_tanh.restype = cd
        L.fgmo_gelu_tanh.argtypes = [cd]
        for name in ("fgmo_e4m3_decode_array", "fgmo_e4m3_encode_array", "fgmo_bf16_round_array",
                     "fgmo_gelu_tanh_array"):
            getattr(L, name).argtypes = [vp, i64, vp]
            getattr(L, name).restype = None
        L.fgmo_quantize_rows.argtypes = [vp, i64, i64, vp, vp]
        L.fgmo_rmsnorm.argtypes = [vp, ci, ci, cd, vp]
        L.fgmo_router_token.restype = cd
        L.fgmo_router_token.argtypes = [vp, vp, vp, ci, ci, ci, vp, vp, vp]
        L.fgmo_expert_token.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Layer), ci, vp, vp]
        L.fgmo_mlp_token.argtypes = [ci, ctypes.POINTER(_Mlp), vp, vp]
        L.fgmo_moe_layer_dense.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Layer),
                                           ctypes.POINTER(_Mlp), vp, ci, vp, vp, vp, vp, vp]
        L.fgmo_moe_layer.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Layer), vp, ci, vp,
                                     vp, vp, vp, vp]
        L.fgmo_stack_layer.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Layer), vp, ci, cd,
                                       vp, vp, vp]
        L.fgmo_lm_head.argtypes = [vp, i64, ci, vp, ci, vp, vp, vp]
        L.fgmo_lm_head_fp8.argtypes = [vp, vp, i64, ci, vp, ci, vp, vp, vp]
        L.fgmo_spec_verify.argtypes = [vp, vp, ci, vp]
        L.fgmo_lm_head_logits.argtypes = [vp, i64, ci, vp, ci, vp]
        L.fgmo_spec_sample.argtypes = [vp, i64, ci, cd, vp, vp, vp, vp, vp]
        L.fgmo_num_threads.restype = ci
        L.fgmo_set_num_threads.argtypes = [ci]
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().fgmo_num_threads()


def set_num_threads(n: int) -> None:
    lib().fgmo_set_num_threads(int(n))


# ---------------------------------------------------------------- formats
def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().fgmo_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float64)
    out = np.empty(v.shape, np.uint8)
    lib().fgmo_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def bf16_round(values) -> np.ndarray:
    """Nearest bf16 bit patterns (uint16) of fp64 values, ties to even."""
    v = _c(values, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().fgmo_bf16_round_array(_p(v), v.size, _p(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (the upper half of a binary32)."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gelu_tanh(x) -> np.ndarray:
    v = _c(x, np.float64)
    out = np.empty(v.shape, np.float64)
    lib().fgmo_gelu_tanh_array(_p(v), v.size, _p(out))
    return out


def quantize_rows(w) -> tuple[np.ndarray, np.ndarray]:
    """Per-row E4M3 quantiser: returns (codes uint8 like w, scales float32 [rows])."""
    w = _c(w, np.float32)
    cols = w.shape[-1]
    rows = w.size // cols
    q = np.empty(w.shape, np.uint8)
    s = np.empty(w.shape[:-1], np.float32)
    lib().fgmo_quantize_rows(_p(w), rows, cols, _p(q), _p(s))
    return q, s


def rmsnorm(h, eps: float = 1e-6) -> np.ndarray:
    h = _c(h, np.float64)
    M, H = h.shape
    out = np.empty_like(h)
    lib().fgmo_rmsnorm(_p(h), M, H, eps, _p(out))
    return out


# ---------------------------------------------------------------- model
@dataclass
class LayerParams:
    """Host copies of one layer's parameters (see ``oracle.c`` for layouts)."""
    router_w: np.ndarray          # uint16 bf16 bits [E, H]
    router_b: np.ndarray | None   # float32 [E]
    gate_q: np.ndarray            # uint8 [E+S, F, H]
    gate_s: np.ndarray            # float32 [E+S, F]
    up_q: np.ndarray
    up_s: np.ndarray
    down_q: np.ndarray            # uint8 [E+S, H, F]
    down_s: np.ndarray            # float32 [E+S, H]
    k: int = 8
    n_shared: int = 1

    def __post_init__(self):
        self.router_w = _c(self.router_w, np.uint16)
        if self.router_b is not None:
            self.router_b = _c(self.router_b, np.float32)
        for n in ("gate_q", "up_q", "down_q"):
            setattr(self, n, _c(getattr(self, n), np.uint8))
        for n in ("gate_s", "up_s", "down_s"):
            setattr(self, n, _c(getattr(self, n), np.float32))
        E, H = self.router_w.shape
        n_all, F, H2 = self.gate_q.shape
        assert H2 == H and n_all == E + self.n_shared
        assert self.up_q.shape == self.gate_q.shape
        assert self.down_q.shape == (n_all, H, F)
        assert self.gate_s.shape == (n_all, F) and self.up_s.shape == (n_all, F)
        assert self.down_s.shape == (n_all, H)

    @property
    def dims(self) -> _Dims:
        E, H = self.router_w.shape
        return _Dims(H, self.gate_q.shape[1], E, self.k, self.n_shared)

    def _struct(self) -> _Layer:
        return _Layer(_p(self.router_w), _p(self.router_b), _p(self.gate_q), _p(self.gate_s),
                      _p(self.up_q), _p(self.up_s), _p(self.down_q), _p(self.down_s))


@dataclass
class LayerOut:
    y: np.ndarray        # float64 [M, H]
    ids: np.ndarray      # int32 [M, k]
    w: np.ndarray        # float64 [M, k]
    margin: np.ndarray   # float64 [M]: k-th minus (k+1)-th logit
    logits: np.ndarray | None = None


@dataclass
class MlpParams:
    """A gated-GELU MLP of any width F (E4M3 rows, fp32 row scales)."""
    gate_q: np.ndarray   # uint8 [F, H]
    gate_s: np.ndarray   # float32 [F]
    up_q: np.ndarray     # uint8 [F, H]
    up_s: np.ndarray     # float32 [F]
    down_q: np.ndarray   # uint8 [H, F]
    down_s: np.ndarray   # float32 [H]

    def __post_init__(self):
        for n in ("gate_q", "up_q", "down_q"):
            setattr(self, n, _c(getattr(self, n), np.uint8))
        for n in ("gate_s", "up_s", "down_s"):
            setattr(self, n, _c(getattr(self, n), np.float32))
        F, H = self.gate_q.shape
        assert self.up_q.shape == (F, H) and self.down_q.shape == (H, F)
        assert self.gate_s.shape == (F,) and self.up_s.shape == (F,) and self.down_s.shape == (H,)

    @property
    def H(self) -> int:
        return self.gate_q.shape[1]

    def _struct(self) -> _Mlp:
        return _Mlp(self.gate_q.shape[0], _p(self.gate_q), _p(self.gate_s), _p(self.up_q), _p(self.up_s),
                    _p(self.down_q), _p(self.down_s))


def mlp_token(mlp: MlpParams, x) -> np.ndarray:
    """The MLP on one token x[H]."""
    x = _c(x, np.float64)
    out = np.empty(mlp.H, np.float64)
    m = mlp._struct()
    lib().fgmo_mlp_token(mlp.H, ctypes.byref(m), _p(x), _p(out))
    return out


def router_token(layer: LayerParams, x) -> tuple[np.ndarray, np.ndarray, float, np.ndarray]:
    x = _c(x, np.float64)
    d = layer.dims
    ids = np.empty(d.k, np.int32)
    w = np.empty(d.k, np.float64)
    logits = np.empty(d.E, np.float64)
    m = lib().fgmo_router_token(_p(x), _p(layer.router_w), _p(layer.router_b), d.H, d.E, d.k,
                                _p(ids), _p(w), _p(logits))
    return ids, w, m, logits


def expert_token(layer: LayerParams, expert: int, x) -> np.ndarray:
    x = _c(x, np.float64)
    d = layer.dims
    out = np.empty(d.H, np.float64)
    s = layer._struct()
    lib().fgmo_expert_token(ctypes.byref(d), ctypes.byref(s), int(expert), _p(x), _p(out))
    return out


def moe_layer(layer: LayerParams, x, dense_shared: MlpParams | None = None) -> LayerOut:
    """One MoE layer on x[M, H] (no norm, no residual). With ``dense_shared``
    that MLP is the always-on part in place of the layer's shared expert."""
    x = _c(x, np.float64)
    M = x.shape[0]
    d = layer.dims
    y = np.empty((M, d.H), np.float64)
    ids = np.empty((M, d.k), np.int32)
    w = np.empty((M, d.k), np.float64)
    margin = np.empty(M, np.float64)
    logits = np.empty((M, d.E), np.float64)
    s = layer._struct()
    if dense_shared is None:
        lib().fgmo_moe_layer(ctypes.byref(d), ctypes.byref(s), _p(x), M, _p(y), _p(ids), _p(w),
                             _p(margin), _p(logits))
    else:
        assert dense_shared.H == d.H
        m = dense_shared._struct()
        lib().fgmo_moe_layer_dense(ctypes.byref(d), ctypes.byref(s), ctypes.byref(m), _p(x), M, _p(y),
                                   _p(ids), _p(w), _p(margin), _p(logits))
    return LayerOut(y, ids, w, margin, logits)


def stack_layer(layer: LayerParams, h, eps: float = 1e-6) -> LayerOut:
    """One layer of the stack: returns h + layer(RMSNorm(h)) in ``y``."""
    h = np.array(h, dtype=np.float64, order="C", copy=True)
    M = h.shape[0]
    d = layer.dims
    ids = np.empty((M, d.k), np.int32)
    w = np.empty((M, d.k), np.float64)
    margin = np.empty(M, np.float64)
    s = layer._struct()
    lib().fgmo_stack_layer(ctypes.byref(d), ctypes.byref(s), _p(h), M, eps, _p(ids), _p(w),
                           _p(margin))
    return LayerOut(h, ids, w, margin)


def lm_head(emb_bits, h) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Tied lm_head argmax: returns (argmax int32 [M], max logit [M], top-1 minus top-2 [M])."""
    e = _c(emb_bits, np.uint16)
    h = _c(h, np.float64)
    V, H = e.shape
    M = h.shape[0]
    assert h.shape[1] == H and 1 <= M <= 16
    am = np.empty(M, np.int32)
    mx = np.empty(M, np.float64)
    mg = np.empty(M, np.float64)
    lib().fgmo_lm_head(_p(e), V, H, _p(h), M, _p(am), _p(mx), _p(mg))
    return am, mx, mg


def lm_head_fp8(q, scale, h) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """FP8 lm_head argmax over E4M3 rows q [V, H] with fp32 row scales [V]:
    returns (argmax int32 [M], max logit [M], top-1 minus top-2 [M])."""
    q = _c(q, np.uint8)
    sc = _c(scale, np.float32)
    h = _c(h, np.float64)
    V, H = q.shape
    M = h.shape[0]
    assert sc.shape == (V,) and h.shape[1] == H and 1 <= M <= 16
    am = np.empty(M, np.int32)
    mx = np.empty(M, np.float64)
    mg = np.empty(M, np.float64)
    lib().fgmo_lm_head_fp8(_p(q), _p(sc), V, H, _p(h), M, _p(am), _p(mx), _p(mg))
    return am, mx, mg


def spec_verify(target, draft) -> tuple[int, int]:
    """Greedy acceptance: (accepted drafts a, next token target[a])."""
    t = _c(target, np.int32)
    d = _c(draft, np.int32)
    M = t.shape[0]
    assert d.shape[0] == M - 1
    out = np.empty(2, np.int32)
    lib().fgmo_spec_verify(_p(t), _p(d) if d.size else None, M, _p(out))
    return int(out[0]), int(out[1])


def lm_head_logits(emb_bits, h) -> np.ndarray:
    """All logits of the bf16 tied lm_head: float64 [M, V]."""
    e = _c(emb_bits, np.uint16)
    h = _c(h, np.float64)
    V, H = e.shape
    M = h.shape[0]
    assert h.shape[1] == H and 1 <= M <= 16
    z = np.empty((M, V), np.float64)
    lib().fgmo_lm_head_logits(_p(e), V, H, _p(h), M, _p(z))
    return z


def spec_sample(z, T: float, draft, u_acc, u_next) -> tuple[int, int, float, float]:
    """Speculative sampling verify at temperature T > 0 with a deterministic
    drafter, on logits z [M, V] and caller-supplied uniforms u_acc [M-1],
    u_next [M]. Returns (accepted drafts a, emitted token, accept margin,
    inverse-CDF gap)."""
    z = _c(z, np.float64)
    M, V = z.shape
    d = _c(draft, np.int32)
    ua = _c(u_acc, np.float64)
    un = _c(u_next, np.float64)
    assert d.shape == (M - 1,) and ua.shape == (M - 1,) and un.shape == (M,) and T > 0
    assert ((d >= 0) & (d < V)).all()
    out = np.empty(2, np.int32)
    mg = np.empty(2, np.float64)
    lib().fgmo_spec_sample(_p(z), V, M, float(T), _p(d) if d.size else None, _p(ua) if ua.size else None,
                           _p(un), _p(out), _p(mg))
    return int(out[0]), int(out[1]), float(mg[0]), float(mg[1])
