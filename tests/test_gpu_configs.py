"""GPU parity on the shapes of the larger workloads: the Qwen3-0.6B-, Qwen3-8B-
and Gemma-like models at full width (every weight matrix, head layout and the
full vocabulary, so the same kernels and K partitions as the full models) with
two layers, so that the CPU oracle finishes in seconds; and long-context
acceptance patterns, checked bit-exactly against single-token decode."""
import numpy as np
import pytest

import inputs
import oracle
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _decode_rows(ctx, first, n, vocab):
    """Greedy decode of n tokens from `first`; returns (chain, per-step logits)."""
    lg1 = gh.logits_buf(1, vocab)
    t, chain, rows = first, [first], []
    for _ in range(n):
        t = ctx.decode(t, logits=lg1)
        rows.append(lg1.clone())
        chain.append(t)
    return chain, rows


def _verify_against_oracle_and_decode(cfg, hw, dw, plen, K, steps, p, seq):
    """Verify windows drawn from the target's own greedy chain (each draft slot
    replaced with probability p) on one context, against the CPU oracle
    (logits within tolerance, same acceptance and correction) and against the
    GPU's single-token decode of the same prefixes (accepted rows bit-equal)."""
    prompt = inputs.prefix_tokens(seq, plen, cfg.vocab)
    max_seq = plen + steps * K + 16
    dec = gh.context(cfg, dw, max_k=max(K, 8), max_seq=max_seq)
    chain, rows = _decode_rows(dec, dec.prefill(prompt), steps * K + 1, cfg.vocab)
    ver = gh.context(cfg, dw, max_k=max(K, 8), max_seq=max_seq, shuffle=seq + 13)
    ver.prefill(prompt)
    orc = oracle.OracleModel(hw, max_seq)
    orc.prefill(prompt)
    lg = gh.logits_buf(K, cfg.vocab)
    for (i, toks, n_exp) in inputs.schedule(chain, K, steps, seq=seq, p=p, vocab=cfg.vocab):
        n, corr = ver.verify(toks, logits=lg)
        lo, am, n_o, c_o = orc.verify(toks)
        assert n == n_exp and corr == chain[i + n + 1], (i, n, n_exp)
        gh.assert_close_to_oracle(lg.cpu().numpy(), lo, f"{cfg.name} verify at {i}")
        if gh.decisive(lo, range(max(n, n_o) + 1)):
            assert (n, corr) == (n_o, c_o), (i, n, n_o)
        if n_o != n:  # a near-tie decided differently: put the oracle on the GPU's path
            orc.truncate(len(ver) - (n + 1))
            orc.prefill(toks[:n + 1])
        assert len(orc) == len(ver)
        for r in range(n + 1):
            assert torch.equal(lg[r], rows[i + r][0]), f"{cfg.name}: row {r} at {i} != decode"
    return ver


@pytest.fixture(scope="module")
def qwen06():
    cfg = inputs.shrink(inputs.QWEN3_0P6B, n_layers=2)
    return (cfg,) + gh.make(cfg, seed=0, gain_std=0.1)


@pytest.fixture(scope="module")
def qwen8b():
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=2)
    return (cfg,) + gh.make(cfg, seed=0, gain_std=0.1)


@pytest.fixture(scope="module")
def gemma():
    cfg = inputs.shrink(inputs.GEMMA_LIKE, n_layers=2)
    return (cfg,) + gh.make(cfg, seed=0, gain_std=0.1)


@pytest.mark.parametrize("K", [4, 5])
def test_qwen06_shape_verify(qwen06, K):
    """0.6B-shaped workload: gamma = 4 drafts read as K = 5 rows, and K = 4;
    prefix of 260 ids (past the first 256-position attention split)."""
    cfg, hw, dw = qwen06
    _verify_against_oracle_and_decode(cfg, hw, dw, plen=260, K=K, steps=4, p=0.6, seq=K)


def test_qwen8b_shape_verify():
    """8B-shaped workload (the benchmark's weight shapes, K partitions and
    kernels) with one layer: K = 4 verify steps against the oracle and against
    decode.  (Each further 4096-wide layer adds rounding-order noise on both
    sides; two layers already reach |dlogit| of about 0.06.)"""
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=1)
    hw, dw = gh.make(cfg, seed=0, gain_std=0.1)
    _verify_against_oracle_and_decode(cfg, hw, dw, plen=40, K=4, steps=3, p=0.6, seq=3)


@pytest.mark.parametrize("K", [8, 16])
def test_gemma_like_three_histories(gemma, K):
    """Gemma-like block verify at the failing prefix length of 87 ids: the
    same committed prefix built by one-token commits, by accepted K = 8 blocks
    and by one prefill gives bit-identical logits and K/V; the verify matches
    the oracle (head_dim 256, one KV head, GeGLU, no QK-norm)."""
    cfg, hw, dw = gemma
    prompt = inputs.prefix_tokens(40, 9, cfg.vocab)
    ref = gh.context(cfg, dw, max_k=16, max_seq=160)
    chain = gh.greedy_chain_gpu(ref, prompt, 80 + K)
    committed = prompt + chain[:78]
    probe = chain[78:78 + K]
    a = gh.context(cfg, dw, max_k=16, max_seq=160, shuffle=1)
    gh.commit(a, committed[1:], a.prefill(committed[:1]))
    b = gh.context(cfg, dw, max_k=16, max_seq=160, shuffle=2)
    b.prefill(prompt)
    i, pending = 0, None
    while len(b) + 8 <= len(committed):
        n, pending = b.verify(chain[i:i + 8])
        assert n == 7
        i += 8
    gh.commit(b, committed[len(b):], pending)
    c = gh.context(cfg, dw, max_k=16, max_seq=160, shuffle=3)
    c.prefill(committed)
    assert len(a) == len(b) == len(c) == len(committed) == 87
    outs = []
    for ctx in (a, b, c):
        lg = gh.logits_buf(K, cfg.vocab)
        n, corr = ctx.verify(probe, logits=lg)
        assert n == K - 1 and corr == chain[78 + K]
        outs.append(lg)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    for layer in range(cfg.n_layers):
        ka, va = a.kv_read(layer, 0, len(a))
        for other in (b, c):
            ko, vo = other.kv_read(layer, 0, len(other))
            assert torch.equal(ka.view(torch.int16), ko.view(torch.int16))
            assert torch.equal(va.view(torch.int16), vo.view(torch.int16))
    orc = oracle.OracleModel(hw, 160)
    orc.prefill(committed)
    lo, am, n_o, c_o = orc.verify(probe)
    gh.assert_close_to_oracle(outs[0].cpu().numpy(), lo, f"gemma-like K={K}")
    if gh.decisive(lo, range(K)):
        assert n_o == K - 1 and c_o == chain[78 + K]


def test_tiny_long_prefix_matches_oracle():
    """4096-id prefix (sixteen attention splits) on the tiny model against the
    oracle, verify of 8 rows."""
    cfg = inputs.TINY
    hw, dw = gh.make(cfg, seed=0, gain_std=0.1)
    prompt = inputs.prefix_tokens(50, 4096, cfg.vocab)
    ctx = gh.context(cfg, dw, max_k=32, max_seq=4200, shuffle=5)
    t = ctx.prefill(prompt)
    orc = oracle.OracleModel(hw, 4200)
    _, to = orc.prefill(prompt)
    assert t == to
    toks = [t, 1, 2, 3, 4, 5, 6, 7]
    lg = gh.logits_buf(8, cfg.vocab)
    n, c = ctx.verify(toks, logits=lg)
    lo, am, n_o, c_o = orc.verify(toks)
    assert (n, c) == (n_o, c_o)
    gh.assert_close_to_oracle(lg.cpu().numpy(), lo, "tiny, 4096-id prefix")


@pytest.mark.parametrize("plen", [4096, 32768])
def test_long_context_forced_patterns(qwen8b, plen):
    """8B-shaped long-context stress: K in {1, 2, 4, 8, 16}, acceptance forced
    to all-accept, reject at slot 0 and reject at slot K/2, each followed by
    the in-call truncation; every accepted row equals single-token decode and
    the committed K/V equals that of a context that only decoded."""
    cfg, hw, dw = qwen8b
    prompt = inputs.prefix_tokens(60 + plen % 7, plen, cfg.vocab)
    Ks = [1, 2, 4, 8, 16]
    n_chain = sum(Ks) * 3 + 4
    dec = gh.context(cfg, dw, max_k=16, max_seq=plen + n_chain + 32)
    chain, rows = _decode_rows(dec, dec.prefill(prompt), n_chain, cfg.vocab)
    ver = gh.context(cfg, dw, max_k=16, max_seq=plen + n_chain + 32, shuffle=plen)
    ver.prefill(prompt)
    i = 0  # chain index of the pending token
    for K in Ks:
        for reject_at in (None, 0, K // 2):
            if reject_at is not None and reject_at >= K - 1:
                continue  # no draft slot to reject
            toks, n_exp = inputs.window(chain, i, K, vocab=cfg.vocab, reject_at=reject_at)
            lg = gh.logits_buf(K, cfg.vocab)
            n, corr = ver.verify(toks, logits=lg)
            assert n == n_exp and corr == chain[i + n + 1], (plen, K, reject_at, n, n_exp)
            for r in range(n + 1):
                assert torch.equal(lg[r], rows[i + r][0]), (plen, K, reject_at, r)
            i += n + 1
            assert len(ver) == plen + i
    assert i > 0
    for layer in range(cfg.n_layers):
        kd, vd = dec.kv_read(layer, plen - 16, i + 16)
        kv, vv = ver.kv_read(layer, plen - 16, i + 16)
        assert torch.equal(kd.view(torch.int16), kv.view(torch.int16))
        assert torch.equal(vd.view(torch.int16), vv.view(torch.int16))


def test_gemma_like_long_context_crosses_attention_forms(gemma):
    """head_dim 256 at a 4100-id prefix (17 attention splits): a 32-row
    verify runs the attention form whose CTAs take several items and the
    long split merge, single-token decode the one-item form; every accepted
    row equals decode bit for bit, and so does the committed K/V."""
    cfg, hw, dw = gemma
    plen = 4100
    prompt = inputs.prefix_tokens(61, plen, cfg.vocab)
    dec = gh.context(cfg, dw, max_k=32, max_seq=plen + 80)
    chain, rows = _decode_rows(dec, dec.prefill(prompt), 50, cfg.vocab)
    ver = gh.context(cfg, dw, max_k=32, max_seq=plen + 80, shuffle=11)
    ver.prefill(prompt)
    for K, reject_at in ((32, None), (16, 5)):
        i = len(ver) - plen
        toks, n_exp = inputs.window(chain, i, K, vocab=cfg.vocab, reject_at=reject_at)
        lg = gh.logits_buf(K, cfg.vocab)
        n, corr = ver.verify(toks, logits=lg)
        assert n == n_exp and corr == chain[i + n + 1], (K, n, n_exp)
        for r in range(n + 1):
            assert torch.equal(lg[r], rows[i + r][0]), (K, r)
    m = len(ver) - plen
    for layer in range(cfg.n_layers):
        kd, vd = dec.kv_read(layer, plen - 8, m + 8)
        kv, vv = ver.kv_read(layer, plen - 8, m + 8)
        assert torch.equal(kd.view(torch.int16), kv.view(torch.int16))
        assert torch.equal(vd.view(torch.int16), vv.view(torch.int16))
