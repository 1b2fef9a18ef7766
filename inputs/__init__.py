"""Seeded synthetic inputs shared by the CPU oracle and the GPU path.

Holds no arithmetic of the decoding method: model shapes, the weight
generator (``svgen.h``: counter-based splitmix64 + sum-of-twelve-uniforms
normals, bf16 bit patterns), uniform random prompts and the draft windows fed
to verify (the target's own greedy chain with slots replaced at random).

The weights are the inputs of both sides of every parity test; random numbers
of the workload (prompt ids, which draft slots are corrupted and by what) are
drawn here and passed in as plain token ids.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_HOST = os.path.join(_HERE, "libsvgen.so")
_LIB_DEV = os.path.join(_HERE, "libsvgen_dev.so")

MASK64 = (1 << 64) - 1

# tensor ids (svgen.h)
T_EMBED, T_LM_HEAD, T_FINAL_NORM, T_LAYER_BASE = 1, 2, 3, 100
ATTN_NORM, WQKV, Q_NORM, K_NORM, WO, FFN_NORM, W_GATE_UP, W_DOWN = range(8)
# streams of the workload's random token ids (not weights)
T_PREFIX = 7001
T_DRAFT = 7002


@dataclass(frozen=True)
class ModelConfig:
    """Decoder shape. act: 0 = SwiGLU, 1 = GeGLU with tanh-approximated GELU."""

    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    qk_norm: int = 1
    act: int = 0
    tie_embeddings: int = 1
    weight_std: float = 0.02

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def layer_params(self) -> int:
        h, d = self.hidden, self.head_dim
        return (self.qkv_rows * h + h * self.n_q_heads * d + 2 * self.ffn * h + h * self.ffn)

    def weight_bytes(self) -> int:
        """Bytes of every linear weight plus the LM head, each counted once."""
        return 2 * (self.n_layers * self.layer_params() + self.vocab * self.hidden)

    def kv_bytes_per_token(self) -> int:
        return self.n_layers * 2 * self.n_kv_heads * self.head_dim * 2


# Shapes of the workloads on the pages (names say what they are).
TINY = ModelConfig("tiny", 2, 256, 4, 2, 64, 704, 1024, rope_theta=1e4, qk_norm=1)
QWEN3_0P6B = ModelConfig("qwen3-0.6b-shape", 28, 1024, 16, 8, 128, 3072, 151936,
                         rope_theta=1e6, qk_norm=1, tie_embeddings=1)
QWEN3_8B = ModelConfig("qwen3-8b-shape", 36, 4096, 32, 8, 128, 12288, 151936,
                       rope_theta=1e6, qk_norm=1, tie_embeddings=0)
GEMMA_LIKE = ModelConfig("gemma-like", 35, 1536, 8, 1, 256, 6144, 262144,
                         rope_theta=1e4, qk_norm=0, act=1, tie_embeddings=1)
CONFIGS = {c.name: c for c in (TINY, QWEN3_0P6B, QWEN3_8B, GEMMA_LIKE)}


def shrink(cfg: ModelConfig, **kw) -> ModelConfig:
    """A copy of ``cfg`` with some fields changed (e.g. fewer layers)."""
    return replace(cfg, **kw)


# ---------------------------------------------------------------- generator
def mix64(x: int) -> int:
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream(seed: int, tensor_id: int) -> int:
    return mix64(mix64(seed & MASK64) ^ ((tensor_id * 0xD1B54A32D192ED03) & MASK64))


def draw(st: int, counter: int) -> int:
    return mix64((st + counter) & MASK64)


def uniform01(st: int, counter: int) -> float:
    """Top 53 bits of a draw as a double in [0, 1)."""
    return (draw(st, counter) >> 11) * (1.0 / (1 << 53))


_host_lib = None
_dev_lib = None


def host_lib():
    global _host_lib
    if _host_lib is None:
        if not os.path.exists(_LIB_HOST):
            raise RuntimeError(f"{_LIB_HOST} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(_LIB_HOST)
        u64, dbl, i32 = ctypes.c_uint64, ctypes.c_double, ctypes.c_int
        for fn in ("svg_fill_weights", "svg_fill_gains"):
            getattr(lib, fn).argtypes = [ctypes.c_void_p, u64, u64, u64, dbl, i32]
            getattr(lib, fn).restype = i32
        lib.svg_fill_tokens.argtypes = [ctypes.c_void_p, u64, u64, u64, ctypes.c_uint32]
        lib.svg_fill_tokens.restype = i32
        lib.svg_weight_at.argtypes = [u64, u64, u64, dbl]
        lib.svg_weight_at.restype = ctypes.c_uint16
        lib.svg_gain_at.argtypes = [u64, u64, u64, dbl]
        lib.svg_gain_at.restype = ctypes.c_uint16
        lib.svg_draw_at.argtypes = [u64, u64, u64]
        lib.svg_draw_at.restype = u64
        _host_lib = lib
    return _host_lib


def dev_lib():
    global _dev_lib
    if _dev_lib is None:
        if not os.path.exists(_LIB_DEV):
            raise RuntimeError(f"{_LIB_DEV} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(_LIB_DEV)
        lib.svg_dev_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint64, ctypes.c_double, ctypes.c_int,
                                     ctypes.c_void_p]
        lib.svg_dev_fill.restype = ctypes.c_int
        _dev_lib = lib
    return _dev_lib


def _nthreads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def layer_tensor(layer: int, which: int) -> int:
    return T_LAYER_BASE + 16 * layer + which


def tensor_specs(cfg: ModelConfig):
    """(key, layer, tensor id, shape, kind) of every weight; kind 'w' or 'g'."""
    h, d = cfg.hidden, cfg.head_dim
    specs = [("embed", -1, T_EMBED, (cfg.vocab, h), "w")]
    if not cfg.tie_embeddings:
        specs.append(("lm_head", -1, T_LM_HEAD, (cfg.vocab, h), "w"))
    specs.append(("final_norm", -1, T_FINAL_NORM, (h,), "g"))
    for l in range(cfg.n_layers):
        specs += [
            ("attn_norm", l, layer_tensor(l, ATTN_NORM), (h,), "g"),
            ("wqkv", l, layer_tensor(l, WQKV), (cfg.qkv_rows, h), "w"),
        ]
        if cfg.qk_norm:
            specs += [("q_norm", l, layer_tensor(l, Q_NORM), (d,), "g"),
                      ("k_norm", l, layer_tensor(l, K_NORM), (d,), "g")]
        specs += [
            ("wo", l, layer_tensor(l, WO), (h, cfg.n_q_heads * d), "w"),
            ("ffn_norm", l, layer_tensor(l, FFN_NORM), (h,), "g"),
            ("w_gate_up", l, layer_tensor(l, W_GATE_UP), (2 * cfg.ffn, h), "w"),
            ("w_down", l, layer_tensor(l, W_DOWN), (h, cfg.ffn), "w"),
        ]
    return specs


@dataclass
class HostWeights:
    """bf16 bit patterns (numpy uint16) of one seeded model."""

    cfg: ModelConfig
    seed: int
    gain_std: float
    tensors: dict = field(default_factory=dict)  # (key, layer) -> ndarray

    def get(self, key: str, layer: int = -1):
        if key == "lm_head" and self.cfg.tie_embeddings:
            key = "embed"
        return self.tensors.get((key, layer))


def host_weights(cfg: ModelConfig, seed: int = 0, gain_std: float = 0.0,
                 nthreads: int | None = None) -> HostWeights:
    """Generate every weight on the host. gain_std = 0 gives unit norm gains."""
    lib = host_lib()
    nt = nthreads or _nthreads()
    hw = HostWeights(cfg, seed, gain_std)
    for key, layer, tid, shape, kind in tensor_specs(cfg):
        arr = np.empty(shape, dtype=np.uint16)
        n = arr.size
        if kind == "w":
            lib.svg_fill_weights(arr.ctypes.data, n, seed, tid, cfg.weight_std, nt)
        else:
            lib.svg_fill_gains(arr.ctypes.data, n, seed, tid, gain_std, nt)
        hw.tensors[(key, layer)] = arr
    return hw


def device_fill(ptr: int, n: int, seed: int, tensor_id: int, stdv: float, kind: int,
                stream_ptr: int = 0) -> None:
    """Fill n bf16 values at device pointer ``ptr`` (kind 0 weight, 1 gain)."""
    rc = dev_lib().svg_dev_fill(ctypes.c_void_p(ptr), n, seed, tensor_id, stdv, kind,
                                ctypes.c_void_p(stream_ptr))
    if rc != 0:
        raise RuntimeError(f"svg_dev_fill failed with CUDA error {rc}")


# ------------------------------------------------------------- token inputs
def prefix_tokens(seq: int, n: int, vocab: int) -> list[int]:
    """Uniform random prompt of sequence ``seq`` (seed 1000 + seq)."""
    st = stream(1000 + seq, T_PREFIX)
    return [draw(st, i) % vocab for i in range(n)]


def corrupt_slot(seq: int, step: int, slot: int, true_tok: int, p: float, vocab: int):
    """Draft slot ``slot`` of verify step ``step``: the true token, or with
    probability p a uniform id different from it (seed 2000 + seq)."""
    st = stream(2000 + seq, T_DRAFT)
    c = (step * 64 + slot) * 2
    if uniform01(st, c) < p:
        return (true_tok + 1 + draw(st, c + 1) % (vocab - 1)) % vocab, True
    return true_tok, False


def window(chain: list[int], i: int, K: int, *, seq: int = 0, step: int = 0, p: float = 0.0,
           vocab: int = 2, reject_at: int | None = None):
    """Verify rows for the pending token chain[i]: [chain[i], d_1 .. d_{K-1}].

    Draft d_j is chain[i + j] unless corrupted. ``reject_at`` (0-based draft
    slot) forces that one draft to be wrong and every other one right; else
    each draft is corrupted independently with probability p. Returns
    (tokens, expected n_accepted).
    """
    toks = [chain[i]]
    n_exp = None
    for j in range(1, K):
        true_tok = chain[i + j]
        if reject_at is not None:
            bad = (j - 1) == reject_at
            tok = (true_tok + 1) % vocab if bad else true_tok
        else:
            tok, bad = corrupt_slot(seq, step, j, true_tok, p, vocab)
        if bad and n_exp is None:
            n_exp = j - 1
        toks.append(tok)
    if n_exp is None:
        n_exp = K - 1
    return toks, n_exp


def schedule(chain: list[int], K: int, n_steps: int, **kw):
    """Windows of n_steps consecutive verify steps along ``chain`` (chain[0]
    is the pending token after the prompt). Returns a list of
    (chain index, tokens, expected n_accepted); the next step starts at
    chain index i + n + 1."""
    out, i = [], 0
    for s in range(n_steps):
        if i + K > len(chain):
            break
        toks, n = window(chain, i, K, step=s, **kw)
        out.append((i, toks, n))
        i += n + 1
    return out


# ------------------------------------------------------------ device copies
def device_weights(cfg: ModelConfig, seed: int = 0, gain_std: float = 0.0, host: HostWeights = None,
                   device: str = "cuda"):
    """Weights as CUDA bf16 tensors keyed (name, layer): copied from ``host``
    when given, else generated in device memory by the device implementation of
    the same generator (bit-identical by construction)."""
    import torch
    out = {}
    for key, layer, tid, shape, kind in tensor_specs(cfg):
        if host is not None:
            a = host.tensors[(key, layer)]
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
            out[(key, layer)] = t.to(device)
        else:
            t = torch.empty(shape, dtype=torch.bfloat16, device=device)
            if kind == "w":
                device_fill(t.data_ptr(), t.numel(), seed, tid, cfg.weight_std, 0)
            else:
                device_fill(t.data_ptr(), t.numel(), seed, tid, gain_std, 1)
            out[(key, layer)] = t
    if host is None:
        torch.cuda.synchronize()
    return out
