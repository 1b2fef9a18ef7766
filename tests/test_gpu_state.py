"""The boundary's state rules on the GPU, through the C-ABI.

A verify window starts with the pending token: the target's greedy token
after the committed sequence ("Phase 23: Speculative Verify Parity",
section 2: the draft window that step 1 writes follows the known-correct
next token).  sv_verify and sv_decode reject any other tokens[0] with
SV_E_STATE and change nothing; the asynchronous call commits nothing for such
a step and reports it at sv_sync.  Rejected rows leave zeros behind
(section 2 step 5 truncates the cache to the accepted prefix): every slot
past the length reads zero.
"""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tiny():
    cfg = inputs.TINY
    _, dw = gh.make(cfg, seed=0, gain_std=0.1, host=False)
    return cfg, dw


def _kv_bytes(ctx, cfg, first, count):
    out = []
    for layer in range(cfg.n_layers):
        k, v = ctx.kv_read(layer, first, count)
        out.append((k.view(torch.int16).clone(), v.view(torch.int16).clone()))
    return out


def _expect(code, fn, *a):
    import greedy_speculative_decode_gb300 as sv
    with pytest.raises(sv.SvError) as e:
        fn(*a)
    assert e.value.code == code, str(e.value)
    return str(e.value)


def test_stale_pending_token_is_state_error(tiny):
    import greedy_speculative_decode_gb300 as sv
    cfg, dw = tiny
    ctx = gh.context(cfg, dw, max_k=8, max_seq=128)
    t = ctx.prefill(inputs.prefix_tokens(80, 30, cfg.vocab))
    before = _kv_bytes(ctx, cfg, 0, 32)
    wrong = (t + 1) % cfg.vocab
    msg = _expect(sv.SV_E_STATE, ctx.verify, [wrong, 1, 2, 3])
    assert str(t) in msg
    _expect(sv.SV_E_STATE, ctx.decode, wrong)
    assert len(ctx) == 30
    after = _kv_bytes(ctx, cfg, 0, 32)
    assert all(torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) for a, b in zip(before, after))
    # the pending token itself is accepted, and the next pending is the correction
    n, corr = ctx.verify([t, 1, 2, 3])
    _expect(sv.SV_E_STATE, ctx.decode, (corr + 1) % cfg.vocab)
    nxt = ctx.decode(corr)
    # a shorter length forgets the pending token: any window may follow
    ctx.truncate(len(ctx) - 2)
    ctx.verify([(nxt + 5) % cfg.vocab, 4])
    # truncation to the same length keeps it
    keep = ctx.decode(ctx.prefill([9]))
    ctx.truncate(len(ctx))
    _expect(sv.SV_E_STATE, ctx.decode, (keep + 1) % cfg.vocab)
    ctx.decode(keep)


def test_rejected_rows_and_truncated_positions_read_zero(tiny):
    """pos = 32 (a page boundary), K = 8 with the first draft wrong: rows
    33..39 are written then zeroed in every layer, and stay on the sequence's
    last page, which sv_kv_read reads to its end."""
    cfg, dw = tiny
    ctx = gh.context(cfg, dw, max_k=8, max_seq=128)
    ref = gh.context(cfg, dw, max_k=8, max_seq=128)
    prompt = inputs.prefix_tokens(81, 32, cfg.vocab)
    chain = gh.greedy_chain_gpu(ref, prompt, 10)
    ctx.prefill(prompt)
    toks, n_exp = inputs.window(chain, 0, 8, vocab=cfg.vocab, reject_at=0)
    n, corr = ctx.verify(toks)
    assert (n, corr) == (n_exp, chain[1]) == (0, chain[1])
    assert len(ctx) == 33
    for k, v in _kv_bytes(ctx, cfg, 33, 15):  # the rest of page 2
        assert not k.any() and not v.any()
    for k, v in _kv_bytes(ctx, cfg, 32, 1):   # the pending row was committed
        assert k.any() and v.any()
    # a truncation zeroes what it removes, on pages it keeps
    ctx.prefill(chain[1:6])
    ctx.truncate(35)
    for k, v in _kv_bytes(ctx, cfg, 35, 13):
        assert not k.any() and not v.any()


def test_async_step_with_stale_pending_commits_nothing(tiny):
    import greedy_speculative_decode_gb300 as sv
    cfg, dw = tiny
    ctx = gh.context(cfg, dw, max_k=8, max_seq=128)
    t = ctx.prefill(inputs.prefix_tokens(82, 40, cfg.vocab))
    ctx.reserve(64)
    good = torch.tensor([t, 3, 4, 5], dtype=torch.int32, device="cuda")
    bad = torch.tensor([(t + 1) % cfg.vocab, 3, 4, 5], dtype=torch.int32, device="cuda")
    res = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    ctx.verify_async(bad, 4, res[0])
    ctx.verify_async(good, 4, res[1])   # still the right window: the bad one changed nothing
    msg = _expect(sv.SV_E_STATE, ctx.sync)
    assert "committed nothing" in msg
    r = res.cpu().tolist()
    assert r[0][0] == -1 and r[0][1] == t and r[0][2] == 40 and r[0][3] == 8
    assert r[1][3] == 0 and r[1][2] == 40 + r[1][0] + 1
    assert len(ctx) == r[1][2]
    ctx.sync()                          # the error was reported once
    for k, v in _kv_bytes(ctx, cfg, len(ctx), 64 - len(ctx)):
        assert not k.any() and not v.any()
    ctx.decode(r[1][1])                 # the pending token is the good step's correction
