"""An independent float64 decoder built from PyTorch library routines.

Used only to pin the oracle: embedding lookup, ``F.rms_norm``,
``F.linear``, ``F.scaled_dot_product_attention`` (causal, grouped-query with
``enable_gqa``), ``F.silu`` and ``F.gelu(approximate="tanh")`` are library
calls; only rotate-half RoPE is written out. No bf16 rounding anywhere, so
the oracle must agree with it up to accumulated bf16 rounding.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _t(bits) -> torch.Tensor:
    f = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return torch.from_numpy(f.astype(np.float64))


def _rope(x: torch.Tensor, theta: float) -> torch.Tensor:
    """x: [heads, n, d]; position of row t is t."""
    n, d = x.shape[1], x.shape[2]
    half = d // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.arange(n, dtype=torch.float64)[:, None] * inv[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return torch.cat([a * c - b * s, b * c + a * s], dim=-1)


def logits(hw, tokens) -> np.ndarray:
    """Logits [n, vocab] of every prefix of ``tokens`` under weights ``hw``."""
    cfg = hw.cfg
    d, Hq, Hkv, H, Fd = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads, cfg.hidden, cfg.ffn
    ids = torch.tensor(list(tokens), dtype=torch.long)
    n = ids.numel()
    x = F.embedding(ids, _t(hw.get("embed")))
    for l in range(cfg.n_layers):
        y = F.rms_norm(x, (H,), weight=_t(hw.get("attn_norm", l)), eps=cfg.rms_eps)
        qkv = F.linear(y, _t(hw.get("wqkv", l)))
        q = qkv[:, : Hq * d].reshape(n, Hq, d).transpose(0, 1)
        k = qkv[:, Hq * d:(Hq + Hkv) * d].reshape(n, Hkv, d).transpose(0, 1)
        v = qkv[:, (Hq + Hkv) * d:].reshape(n, Hkv, d).transpose(0, 1)
        if cfg.qk_norm:
            q = F.rms_norm(q, (d,), weight=_t(hw.get("q_norm", l)), eps=cfg.rms_eps)
            k = F.rms_norm(k, (d,), weight=_t(hw.get("k_norm", l)), eps=cfg.rms_eps)
        q, k = _rope(q, cfg.rope_theta), _rope(k, cfg.rope_theta)
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True,
                                           enable_gqa=True)[0]
        o = o.transpose(0, 1).reshape(n, Hq * d)
        x = x + F.linear(o, _t(hw.get("wo", l)))
        y = F.rms_norm(x, (H,), weight=_t(hw.get("ffn_norm", l)), eps=cfg.rms_eps)
        gu = F.linear(y, _t(hw.get("w_gate_up", l)))
        g, u = gu[:, :Fd], gu[:, Fd:]
        act = F.silu(g) if cfg.act == 0 else F.gelu(g, approximate="tanh")
        x = x + F.linear(act * u, _t(hw.get("w_down", l)))
    y = F.rms_norm(x, (H,), weight=_t(hw.get("final_norm")), eps=cfg.rms_eps)
    return F.linear(y, _t(hw.get("lm_head"))).numpy()
