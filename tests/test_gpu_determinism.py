"""Run-to-run and context-to-context bit-exactness at a production width.

A rare shared-memory hazard (TMA overwriting a stage that ldmatrix was still
ordered against) once made about one step in thirty differ in a few values
on the Qwen3-8B shape. These tests repeat the same step many times and build
the same prefix in independent contexts; every repeat must match exactly."""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wide():
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=6)
    dw = inputs.device_weights(cfg, seed=0, gain_std=0.0)
    return cfg, dw


def test_repeated_steps_identical(wide):
    cfg, dw = wide
    prompt = inputs.prefix_tokens(0, 600, cfg.vocab)
    ctx = gh.context(cfg, dw, max_k=32, max_seq=700)
    t = ctx.prefill(prompt)
    ref1, ref4 = None, None
    l1, l4 = gh.logits_buf(1, cfg.vocab), gh.logits_buf(4, cfg.vocab)
    for rep in range(40):
        ctx.decode(t, logits=l1)
        ctx.truncate(600)
        ctx.verify([t, 11, 12, 13], logits=l4)
        ctx.truncate(600)
        if ref1 is None:
            ref1, ref4 = l1.clone(), l4.clone()
        else:
            assert torch.equal(ref1, l1), f"decode repeat {rep} differs"
            assert torch.equal(ref4, l4), f"verify repeat {rep} differs"
    assert torch.equal(ref4[0], ref1[0])


def test_independent_contexts_identical(wide):
    cfg, dw = wide
    prompt = inputs.prefix_tokens(1, 700, cfg.vocab)
    outs = []
    for rep in range(3):
        ctx = gh.context(cfg, dw, max_k=32, max_seq=800, shuffle=rep)
        t = ctx.prefill(prompt)
        chain = [t]
        for _ in range(6):
            chain.append(ctx.decode(chain[-1]))
        kv = [ctx.kv_read(l, 0, len(ctx)) for l in range(cfg.n_layers)]
        outs.append((chain, kv))
        ctx.close()
    for chain, kv in outs[1:]:
        assert chain == outs[0][0]
        for (k, v), (k0, v0) in zip(kv, outs[0][1]):
            assert torch.equal(k.view(torch.int16), k0.view(torch.int16))
            assert torch.equal(v.view(torch.int16), v0.view(torch.int16))
