"""ctypes wrapper of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product library. The oracle shares
no code with the CUDA path; both read the same seeded weights (``inputs``).
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_P = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads",
                                           "head_dim", "ffn", "vocab")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("qk_norm", ctypes.c_int), ("act", ctypes.c_int)]


_LAYER_KEYS = ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate_up", "w_down")


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("lm_head", _P), ("final_norm", _P)] + [(k, _PP) for k in _LAYER_KEYS]


def _open(path: str):
    L = ctypes.CDLL(path)
    i32, f32, u16 = ctypes.c_int, ctypes.c_float, ctypes.c_uint16
    L.orc_create.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), i32]
    L.orc_create.restype = _P
    L.orc_destroy.argtypes = [_P]
    L.orc_len.argtypes = [_P]
    L.orc_threads.argtypes = []
    L.orc_forward.argtypes = [_P, i32, _P]
    L.orc_prefill.argtypes = [_P, _P, i32, _P, _P]
    L.orc_decode.argtypes = [_P, i32, _P, _P]
    L.orc_verify.argtypes = [_P, _P, i32, _P, _P, _P, _P]
    L.orc_truncate.argtypes = [_P, i32]
    L.orc_kv.argtypes = [_P, i32, i32, _P, _P]
    L.orc_bruteforce.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), _P, i32, _P]
    L.orc_layer.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), i32, i32, i32, _P, _P,
                            _P, _P, _P, _P]
    L.orc_head.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), _P, _P]
    L.orc_bf16.argtypes = [f32]
    L.orc_bf16.restype = u16
    L.orc_f32.argtypes = [u16]
    L.orc_f32.restype = f32
    L.orc_argmax.argtypes = [_P, i32]
    L.orc_rmsnorm.argtypes = [_P, _P, i32, f32, _P]
    L.orc_linear.argtypes = [_P, _P, i32, i32, _P]
    L.orc_rope.argtypes = [_P, i32, i32, f32]
    L.orc_attend.argtypes = [_P, _P, _P, i32, i32, i32, _P]
    L.orc_silu.argtypes = [f32]
    L.orc_silu.restype = f32
    L.orc_gelu_tanh.argtypes = [f32]
    L.orc_gelu_tanh.restype = f32
    L.orc_glu.argtypes = [_P, _P, i32, i32, _P]
    return L


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise RuntimeError(f"{_LIB} is missing: run __graft_entry__.build() first")
        _lib = _open(_LIB)
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the wrapper against another build of oracle.c (used by the tests
    that plant a mistake in a copy of the oracle and expect the pins to fail)."""
    global _lib
    saved = lib()
    _lib = _open(path)
    try:
        yield
    finally:
        _lib = saved


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


# ------------------------------------------------------------ single ops
def bf16(x: float) -> int:
    return int(lib().orc_bf16(float(x)))


def f32(b: int) -> float:
    return float(lib().orc_f32(int(b)))


def argmax(v) -> int:
    v = np.ascontiguousarray(v, dtype=np.float32)
    return int(lib().orc_argmax(_ptr(v), v.size))


def rmsnorm(x_bits, g_bits, eps: float) -> np.ndarray:
    x, g = _u16(x_bits), _u16(g_bits)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(g), x.size, eps, _ptr(y))
    return y


def linear(W_bits, x_bits) -> np.ndarray:
    W, x = _u16(W_bits), _u16(x_bits)
    y = np.empty(W.shape[0], dtype=np.uint16)
    lib().orc_linear(_ptr(W), _ptr(x), W.shape[0], W.shape[1], _ptr(y))
    return y


def rope(x_bits, pos: int, theta: float) -> np.ndarray:
    x = _u16(x_bits).copy()
    lib().orc_rope(_ptr(x), x.size, pos, theta)
    return x


def attend(q_bits, K_bits, V_bits) -> np.ndarray:
    q, K, V = _u16(q_bits), _u16(K_bits), _u16(V_bits)
    out = np.empty(q.size, dtype=np.uint16)
    lib().orc_attend(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.size, K.shape[1], _ptr(out))
    return out


def silu(x: float) -> float:
    return float(lib().orc_silu(x))


def gelu_tanh(x: float) -> float:
    return float(lib().orc_gelu_tanh(x))


def glu(gate_bits, up_bits, act: int) -> np.ndarray:
    g, u = _u16(gate_bits), _u16(up_bits)
    a = np.empty_like(g)
    lib().orc_glu(_ptr(g), _ptr(u), g.size, int(act), _ptr(a))
    return a


def threads() -> int:
    return int(lib().orc_threads())


def bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 values (plain widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bits(x) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (the oracle's own rounding)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.array([lib().orc_bf16(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


# ------------------------------------------------------------- the model
class _Bound:
    """ctypes structs + every array they point into, kept alive together."""

    def __init__(self, hw):
        c = hw.cfg
        self.cfg = _Config(c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.ffn,
                           c.vocab, c.rms_eps, c.rope_theta, c.qk_norm, c.act)
        self.keep = []
        L = max(c.n_layers, 1)

        def arr(key, layer=-1):
            a = hw.get(key, layer)
            if a is None:
                return None
            a = _u16(a)
            self.keep.append(a)
            return a.ctypes.data

        w = _Weights()
        w.embed = arr("embed")
        w.lm_head = arr("lm_head")
        w.final_norm = arr("final_norm")
        for k in _LAYER_KEYS:
            ptrs = (ctypes.c_void_p * L)(*[arr(k, l) for l in range(c.n_layers)])
            self.keep.append(ptrs)
            setattr(w, k, ctypes.cast(ptrs, _PP))
        self.w = w


class OracleModel:
    """One sequence's decoder state on the CPU (dense per-position cache)."""

    def __init__(self, hw, max_len: int):
        self.hw = hw
        self.V = hw.cfg.vocab
        self._b = _Bound(hw)
        self._L = lib()
        self._m = self._L.orc_create(ctypes.byref(self._b.cfg), ctypes.byref(self._b.w), max_len)
        if not self._m:
            raise ValueError("orc_create rejected the configuration")

    def __del__(self):
        if getattr(self, "_m", None):
            self._L.orc_destroy(self._m)
            self._m = None

    def __len__(self) -> int:
        return int(self._L.orc_len(self._m))

    def _check(self, rc, what):
        if rc != 0:
            raise ValueError(f"{what} failed (rc={rc})")

    def prefill(self, tokens):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        lg = np.empty(self.V, dtype=np.float32)
        nxt = np.zeros(1, dtype=np.int32)
        self._check(self._L.orc_prefill(self._m, _ptr(t), t.size, _ptr(lg), _ptr(nxt)), "prefill")
        return lg, int(nxt[0])

    def decode(self, token: int):
        lg = np.empty(self.V, dtype=np.float32)
        nxt = np.zeros(1, dtype=np.int32)
        self._check(self._L.orc_decode(self._m, int(token), _ptr(lg), _ptr(nxt)), "decode")
        return lg, int(nxt[0])

    def verify(self, tokens):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        K = t.size
        lg = np.empty((K, self.V), dtype=np.float32)
        am = np.empty(K, dtype=np.int32)
        n = np.zeros(1, dtype=np.int32)
        c = np.zeros(1, dtype=np.int32)
        self._check(self._L.orc_verify(self._m, _ptr(t), K, _ptr(lg), _ptr(am), _ptr(n), _ptr(c)),
                    "verify")
        return lg, am, int(n[0]), int(c[0])

    def truncate(self, new_len: int):
        self._check(self._L.orc_truncate(self._m, int(new_len)), "truncate")

    def kv(self, layer: int, pos: int):
        c = self.hw.cfg
        k = np.empty(c.n_kv_heads * c.head_dim, dtype=np.uint16)
        v = np.empty_like(k)
        self._check(self._L.orc_kv(self._m, layer, pos, _ptr(k), _ptr(v)), "kv")
        return k, v


def bruteforce(hw, tokens) -> np.ndarray:
    """Logits [n, vocab] of every prefix, recomputed layer-major with no cache."""
    b = _Bound(hw)
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    lg = np.empty((t.size, hw.cfg.vocab), dtype=np.float32)
    rc = lib().orc_bruteforce(ctypes.byref(b.cfg), ctypes.byref(b.w), _ptr(t), t.size, _ptr(lg))
    if rc != 0:
        raise ValueError("bruteforce rejected its arguments")
    return lg


class LayerOracle:
    """One layer, or the final head, of the oracle applied to given inputs:
    the per-token pass cut at a layer boundary (teacher forcing)."""

    def __init__(self, hw):
        self.hw = hw
        self._b = _Bound(hw)

    def layer(self, layer: int, pos: int, x_in, k_cache=None, v_cache=None):
        """Rows x_in (bf16 bits [K, hidden]) at positions pos .. pos+K-1 through
        layer ``layer``, over that layer's cached K/V of positions 0 .. pos-1
        (bf16 bits [pos, n_kv_heads * head_dim]). Returns (x_out, k, v): the
        rows after the layer and their own K and V."""
        c = self.hw.cfg
        x = _u16(x_in).reshape(-1, c.hidden)
        K = x.shape[0]
        row = c.n_kv_heads * c.head_dim
        kc = None if k_cache is None else _u16(k_cache).reshape(-1, row)
        vc = None if v_cache is None else _u16(v_cache).reshape(-1, row)
        if pos > 0 and (kc is None or vc is None or kc.shape[0] < pos or vc.shape[0] < pos):
            raise ValueError("the cache must hold every position before pos")
        xo = np.empty_like(x)
        ko = np.empty((K, row), dtype=np.uint16)
        vo = np.empty_like(ko)
        rc = lib().orc_layer(ctypes.byref(self._b.cfg), ctypes.byref(self._b.w), int(layer), int(pos),
                             K, 0 if kc is None else _ptr(kc), 0 if vc is None else _ptr(vc),
                             _ptr(x), _ptr(xo), _ptr(ko), _ptr(vo))
        if rc != 0:
            raise ValueError("orc_layer rejected its arguments")
        return xo, ko, vo

    def head(self, x):
        """Final RMSNorm + LM head of residual-stream rows x (bf16 bits [K, hidden]):
        logits [K, vocab] (bf16 values)."""
        c = self.hw.cfg
        xs = _u16(x).reshape(-1, c.hidden)
        out = np.empty((xs.shape[0], c.vocab), dtype=np.float32)
        for r in range(xs.shape[0]):
            xr = np.ascontiguousarray(xs[r])
            if lib().orc_head(ctypes.byref(self._b.cfg), ctypes.byref(self._b.w), _ptr(xr),
                              _ptr(out[r])) != 0:
                raise ValueError("orc_head rejected its arguments")
        return out
