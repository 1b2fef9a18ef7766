"""The benchmark's low-rate verify audit ("Phase 23: Speculative Verify
Parity", section 4 item 2: a sampled audit of verify rows against target
decode) run on the GPU: every audited row of a real schedule must be
bit-identical to single-token decode, and its mismatch report must carry the
top-5 ids and logits of both sides."""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _steps(cfg, dw, K=4, prefix=40, n_steps=8):
    ctx = gh.context(cfg, dw, max_k=8, max_seq=prefix + 64 + 2 * K)
    prompt = inputs.prefix_tokens(84, prefix, cfg.vocab)
    t = ctx.prefill(prompt)
    chain = [t]
    for _ in range(n_steps * K + K):
        chain.append(ctx.decode(chain[-1]))
    ctx.truncate(prefix)
    sq = {"ctx": ctx, "prompt": prompt, "chain": chain}
    sched = inputs.schedule(chain, K, n_steps, seq=0, p=0.5, vocab=cfg.vocab)
    return [(sq, i, toks, n) for (i, toks, n) in sched], ctx


def test_audit_finds_every_row_bit_identical():
    import bench
    cfg = inputs.TINY
    _, dw = gh.make(cfg, seed=0, gain_std=0.1, host=False)
    steps, ctx = _steps(cfg, dw)
    aud = bench.audit(steps, 0, len(steps), 2, 40, 4, cfg.vocab)
    assert aud["rows"] == 4 * len(range(0, len(steps), 2))
    assert aud["bitwise_equal"] == aud["rows"] and aud["mismatches"] == []
    assert len(ctx) == 40 + steps[-2][1]  # the audit leaves the context at the audited step's prefix


def test_audit_reports_a_mismatch_with_both_top5():
    """The comparison is swapped for one that rejects row 1 (a mistake planted
    in the host-side comparison, not in the GPU path): the report keeps the
    top-5 (id, logit) lists of both sides, largest first."""
    import bench
    cfg = inputs.TINY
    _, dw = gh.make(cfg, seed=0, gain_std=0.1, host=False)
    steps, _ = _steps(cfg, dw)
    calls = {"n": 0}

    def same(a, b):
        calls["n"] += 1
        return calls["n"] % 4 != 2 and torch.equal(a, b)

    aud = bench.audit(steps, 0, 4, 1, 40, 4, cfg.vocab, same=same)
    assert aud["rows"] == 16 and aud["bitwise_equal"] == 12
    ex = aud["mismatches"][0]
    assert ex["row"] == 1 and ex["max_abs_diff"] == 0.0
    for side in ("verify_top5", "decode_top5"):
        assert len(ex[side]) == 5
        vals = [v for _, v in ex[side]]
        assert vals == sorted(vals, reverse=True)
    assert ex["verify_top5"] == ex["decode_top5"]
