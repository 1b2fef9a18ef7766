"""Shared set-up of the GPU tests: seeded models on the device, contexts, and
the comparisons against the CPU oracle."""
from __future__ import annotations

import numpy as np

import inputs
import oracle

TOL_LOGIT = 0.05      # |GPU logit - oracle logit| bound
ARGMAX_MARGIN = 0.1   # argmax must agree where the oracle's top-2 margin exceeds this


def make(cfg, seed=0, gain_std=0.1, host=True):
    """(host weights or None, device weights) of a seeded model."""
    hw = inputs.host_weights(cfg, seed=seed, gain_std=gain_std) if host else None
    dw = inputs.device_weights(cfg, seed=seed, gain_std=gain_std, host=hw)
    return hw, dw


def context(cfg, dw, max_k=8, max_seq=512, max_pages=None, shuffle=None, kv_delayed=False):
    import greedy_speculative_decode_gb300 as sv
    ctx = sv.Context(cfg, dw, max_k=max_k, max_seq=max_seq, max_pages=max_pages, kv_delayed=kv_delayed)
    if shuffle is not None:
        ctx.shuffle_pages(shuffle)
    return ctx


def logits_buf(rows, vocab):
    import torch
    return torch.full((rows, vocab), float("nan"), dtype=torch.float32, device="cuda")


def assert_close_to_oracle(gpu_logits, orc_logits, what=""):
    g = np.asarray(gpu_logits, dtype=np.float64)
    o = np.asarray(orc_logits, dtype=np.float64)
    assert g.shape == o.shape, what
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU logits"
    err = np.max(np.abs(g - o))
    assert err <= TOL_LOGIT, f"{what}: max |dlogit| = {err}"
    g2, o2 = np.atleast_2d(g), np.atleast_2d(o)
    top2 = np.sort(o2, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > ARGMAX_MARGIN
    assert np.array_equal(g2.argmax(1)[sure], o2.argmax(1)[sure]), f"{what}: argmax differs"
    # logits are bf16 values
    assert np.array_equal(oracle.bits_to_f32(oracle.f32_to_bits(g2[:1].astype(np.float32))),
                          g2[:1].astype(np.float32)), f"{what}: logits are not bf16 values"
    return err


def decisive(orc_logits, rows) -> bool:
    """True if the oracle's top-2 margin exceeds ARGMAX_MARGIN on every row in
    ``rows``: only then is its greedy choice, and so its acceptance count, one
    the GPU must reproduce (closer calls are bf16 near-ties)."""
    o = np.atleast_2d(np.asarray(orc_logits, dtype=np.float64))
    top2 = np.sort(o[list(rows)], axis=1)[:, -2:]
    return bool(np.all(top2[:, 1] - top2[:, 0] > ARGMAX_MARGIN))


def bits(t):
    """Raw bytes of a CUDA tensor as a numpy uint8 array (for exact comparisons)."""
    import torch
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def commit(ctx, tokens, pending):
    """Commit ``tokens`` one at a time: a decode where the token is the
    pending greedy token, else a one-token prefill (the library takes tokens
    the model did not choose only through prefill).  Returns the new pending
    token."""
    for tok in tokens:
        pending = ctx.decode(tok) if tok == pending else ctx.prefill([tok])
    return pending


def greedy_chain_gpu(ctx, prompt, n):
    """Prefill `prompt` then decode greedily; returns [t0, t1, ...] (n tokens),
    leaving ctx at len(prompt) + n - 1 committed tokens."""
    t = ctx.prefill(prompt)
    chain = [t]
    for _ in range(n - 1):
        t = ctx.decode(t)
        chain.append(t)
    return chain
