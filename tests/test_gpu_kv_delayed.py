"""Delayed K/V write-through (sv_config kv_delayed = 1) against
write-then-truncate, on the GPU through the C-ABI.

"Phase B decision — post-v4", section "Phase C gating item (new)", lists as
candidate C0 a verify that computes its logits without committing K/V, the
K/V being committed once the acceptance decision is made, so that no later
argmax conditions on rejected draft rows.  "Phase 23: Speculative Verify
Parity" section 2 instead writes the whole window and truncates to the
accepted prefix (steps 1 and 5).  In this library both protocols compute the
same thing: the tests run the same steps both ways and require identical
logits, argmax, acceptance and cache contents (zero past the length), bit
for bit, through the synchronous and the asynchronous call, on shuffled
pages and with windows that straddle two page boundaries.
"""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _kv(ctx, cfg, first, count):
    out = []
    for layer in range(cfg.n_layers):
        k, v = ctx.kv_read(layer, first, count)
        out.append((k.view(torch.int16).clone(), v.view(torch.int16).clone()))
    return out


def _same_kv(a, b):
    return all(torch.equal(x[0], y[0]) and torch.equal(x[1], y[1]) for x, y in zip(a, b))


def _pages_end(n):
    return (n + 15) // 16 * 16


def _sync_run(cfg, dw, prompt, K, n_steps, p, delayed, shuffle, max_pages=None):
    """Verify steps along the greedy chain of `prompt` with drafts corrupted
    at rate p; per step: (tokens, n, correction, logits, cache to the end of
    the last page the sequence keeps)."""
    ref = gh.context(cfg, dw, max_k=K, max_seq=512)
    chain = gh.greedy_chain_gpu(ref, prompt, 160)
    ref.close()
    ctx = gh.context(cfg, dw, max_k=K, max_seq=512, max_pages=max_pages, shuffle=shuffle,
                     kv_delayed=delayed)
    assert ctx.prefill(prompt) == chain[0]
    out, i = [], 0
    for s in range(n_steps):
        if i + K > len(chain):
            break
        toks, n_exp = inputs.window(chain, i, K, seq=11, step=s, p=p, vocab=cfg.vocab)
        lg = gh.logits_buf(K, cfg.vocab)
        n, corr = ctx.verify(toks, logits=lg)
        assert n == n_exp and corr == chain[i + n + 1]
        out.append((toks, n, corr, lg, _kv(ctx, cfg, 0, _pages_end(len(ctx)))))
        i += n + 1
    # a single-row step commits its row directly in either mode
    lg = gh.logits_buf(1, cfg.vocab)
    nxt = ctx.decode(out[-1][2], logits=lg)
    out.append(([out[-1][2]], 0, nxt, lg, _kv(ctx, cfg, 0, _pages_end(len(ctx)))))
    ctx.close()
    return out


@pytest.mark.parametrize("K,prompt_len,shuffle", [(8, 45, None), (32, 47, 5), (32, 30, None)])
def test_delayed_matches_write_then_truncate_tiny(K, prompt_len, shuffle):
    """TINY model; K = 32 from position 47 spans pages 2, 3 and 4."""
    cfg = inputs.TINY
    _, dw = gh.make(cfg, seed=2, gain_std=0.1, host=False)
    prompt = inputs.prefix_tokens(90 + K, prompt_len, cfg.vocab)
    a = _sync_run(cfg, dw, prompt, K, 6, 0.25, False, shuffle)
    b = _sync_run(cfg, dw, prompt, K, 6, 0.25, True, shuffle)
    assert len(a) == len(b) >= 3
    assert any(s[1] < K - 1 for s in a), "no step rejected a draft"
    for s, (x, y) in enumerate(zip(a, b)):
        assert x[0] == y[0] and x[1:3] == y[1:3], f"step {s}: acceptance differs"
        assert torch.equal(x[3], y[3]), f"step {s}: logits differ"
        assert _same_kv(x[4], y[4]), f"step {s}: cache differs"


@pytest.mark.parametrize("shape", ["qwen3-8b-shape", "gemma-like"])
def test_delayed_matches_wide_layers(shape):
    """8B-shaped (8 kv heads of 128) and Gemma-like (one kv head of 256)
    layers, 2 layers, shuffled pages of a 32-page pool (ids 0..31; the
    scratch pages are ids 32..34), after a 300-token prompt prefilled in
    128-row blocks."""
    cfg = inputs.shrink(inputs.CONFIGS[shape], n_layers=2, vocab=32768)
    _, dw = gh.make(cfg, seed=3, gain_std=0.1, host=False)
    prompt = inputs.prefix_tokens(95, 300, cfg.vocab)
    a = _sync_run(cfg, dw, prompt, 16, 5, 0.2, False, 9, max_pages=32)
    b = _sync_run(cfg, dw, prompt, 16, 5, 0.2, True, 9, max_pages=32)
    for s, (x, y) in enumerate(zip(a, b)):
        assert x[1:3] == y[1:3], f"step {s}: acceptance differs"
        assert torch.equal(x[3], y[3]), f"step {s}: logits differ"
        assert _same_kv(x[4], y[4]), f"step {s}: cache differs"


def test_delayed_async_matches_and_stale_step_commits_nothing():
    """The asynchronous call with device-resident windows: five steps, one
    of them with a stale tokens[0], which commits nothing in either mode."""
    import greedy_speculative_decode_gb300 as sv
    cfg = inputs.TINY
    _, dw = gh.make(cfg, seed=4, gain_std=0.1, host=False)
    prompt = inputs.prefix_tokens(97, 41, cfg.vocab)
    ref = gh.context(cfg, dw, max_k=8, max_seq=256)
    chain = gh.greedy_chain_gpu(ref, prompt, 80)
    ref.close()
    sched = inputs.schedule(chain, 8, 4, seq=3, p=0.3, vocab=cfg.vocab)
    rows = [t for _, t, _ in sched]
    stale = [(chain[sched[2][0]] + 1) % cfg.vocab] + rows[2][1:]
    rows = rows[:2] + [stale] + rows[2:]
    results = {}
    for delayed in (False, True):
        ctx = gh.context(cfg, dw, max_k=8, max_seq=256, kv_delayed=delayed)
        ctx.prefill(prompt)
        ctx.reserve(41 + 8 * len(rows))
        toks = torch.tensor(rows, dtype=torch.int32, device="cuda")
        res = torch.zeros((len(rows), 4), dtype=torch.int32, device="cuda")
        lg = torch.full((len(rows), 8, cfg.vocab), float("nan"), dtype=torch.float32, device="cuda")
        for j in range(len(rows)):
            ctx.verify_async(toks[j], 8, res[j], logits=lg[j])
        with pytest.raises(sv.SvError) as e:
            ctx.sync()
        assert e.value.code == sv.SV_E_STATE
        n = len(ctx)
        results[delayed] = (res.cpu(), lg, n, _kv(ctx, cfg, 0, _pages_end(41 + 8 * len(rows))))
        ctx.close()
    (ra, la, na, ka), (rb, lb, nb, kb) = results[False], results[True]
    assert torch.equal(ra, rb) and na == nb
    assert ra[2][0] == -1 and ra[2][3] == 8
    assert [int(r[0]) for i, r in enumerate(ra) if i != 2] == [n for _, _, n in sched]
    for j in range(len(rows)):  # the stale step's logits are computed all the same
        assert torch.equal(la[j], lb[j]), f"step {j}: logits differ"
    assert _same_kv(ka, kb)


def test_delayed_kernel_count():
    cfg = inputs.TINY
    _, dw = gh.make(cfg, seed=0, gain_std=0.1, host=False)
    a = gh.context(cfg, dw, max_k=8, max_seq=64)
    b = gh.context(cfg, dw, max_k=8, max_seq=64, kv_delayed=True)
    assert b.kernels_per_step(8) == a.kernels_per_step(8) + 1
    assert b.kernels_per_step(1) == a.kernels_per_step(1)   # a decode step commits its row directly
    assert b.kernels_per_step(8, with_head=False) == a.kernels_per_step(8, with_head=False)


def test_delayed_draft_verify_loop_matches():
    """sv_spec_generate with an 8B-shaped target (one layer, 32768 ids) in
    delayed mode and a 0.6B-shaped drafter of other weights, so that drafts
    are rejected, commits the same tokens, counts and cache as with
    write-then-truncate."""
    import greedy_speculative_decode_gb300 as sv
    tcfg = inputs.shrink(inputs.QWEN3_8B, n_layers=1, vocab=32768)
    dcfg = inputs.shrink(inputs.QWEN3_0P6B, n_layers=2, vocab=32768)
    _, tw = gh.make(tcfg, seed=0, gain_std=0.1, host=False)
    _, dw = gh.make(dcfg, seed=1, gain_std=0.1, host=False)
    prompt = inputs.prefix_tokens(82, 40, tcfg.vocab)
    out = []
    for delayed in (False, True):
        tgt = gh.context(tcfg, tw, max_k=8, max_seq=128, kv_delayed=delayed)
        drf = gh.context(dcfg, dw, max_k=8, max_seq=128)
        pending = tgt.prefill(prompt)
        drf.prefill(prompt)
        toks, nxt, st = sv.spec_generate(tgt, drf, pending, 4, 40)
        out.append((toks, nxt, st, _kv(tgt, tcfg, 0, _pages_end(len(tgt)))))
        tgt.close()
        drf.close()
    assert out[0][:3] == out[1][:3]
    assert out[0][2]["accepted"] < out[0][2]["proposed"], "no draft was rejected"
    assert _same_kv(out[0][3], out[1][3])
