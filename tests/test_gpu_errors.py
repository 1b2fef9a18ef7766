"""Error paths of the C-ABI: every rejected call returns its code, names the
reason, and leaves the sequence (length, K/V bytes, next results) unchanged."""
import dataclasses

import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tiny():
    cfg = inputs.TINY
    hw, dw = gh.make(cfg, seed=0, gain_std=0.1, host=False)
    return cfg, dw


def _codes():
    import greedy_speculative_decode_gb300 as sv
    return sv


def _expect(code, fn, *args, **kw):
    sv = _codes()
    with pytest.raises(sv.SvError) as e:
        fn(*args, **kw)
    assert e.value.code == code, str(e.value)
    return str(e.value)


def _snapshot(ctx, cfg):
    out = [len(ctx)]
    for layer in range(cfg.n_layers):
        k, v = ctx.kv_read(layer, 0, len(ctx))
        out.append((k.clone(), v.clone()))
    return out


def _same(a, b):
    if a[0] != b[0]:
        return False
    return all(torch.equal(x[0].view(torch.int16), y[0].view(torch.int16)) and
               torch.equal(x[1].view(torch.int16), y[1].view(torch.int16)) for x, y in zip(a[1:], b[1:]))


def test_bad_arguments_are_rejected_and_change_nothing(tiny):
    cfg, dw = tiny
    sv = _codes()
    ctx = gh.context(cfg, dw, max_k=8, max_seq=64)
    t = ctx.prefill(inputs.prefix_tokens(70, 20, cfg.vocab))
    before = _snapshot(ctx, cfg)
    _expect(sv.SV_E_INVAL, ctx.verify, [t] + [1] * 8)          # K = 9 > max_k
    _expect(sv.SV_E_INVAL, ctx.verify, [])                     # K = 0
    _expect(sv.SV_E_INVAL, ctx.verify, [t, cfg.vocab])         # token out of range
    _expect(sv.SV_E_INVAL, ctx.verify, [t, -1])
    _expect(sv.SV_E_INVAL, ctx.prefill, [1] * 45)              # 20 + 45 > max_seq
    _expect(sv.SV_E_INVAL, ctx.truncate, 21)                   # beyond the length
    _expect(sv.SV_E_INVAL, ctx.truncate, -1)
    _expect(sv.SV_E_INVAL, ctx.kv_read, 0, 20, 13)             # past the allocated pages (32)
    _expect(sv.SV_E_INVAL, ctx.kv_read, cfg.n_layers, 0, 1)    # no such layer
    assert _same(before, _snapshot(ctx, cfg))
    # the context still works, and gives what a fresh one gives
    lg_a = gh.logits_buf(4, cfg.vocab)
    na, ca = ctx.verify([t, 5, 6, 7], logits=lg_a)
    fresh = gh.context(cfg, dw, max_k=8, max_seq=64)
    fresh.prefill(inputs.prefix_tokens(70, 20, cfg.vocab))
    lg_b = gh.logits_buf(4, cfg.vocab)
    nb, cb = fresh.verify([t, 5, 6, 7], logits=lg_b)
    assert (na, ca) == (nb, cb) and torch.equal(lg_a, lg_b)


def test_page_pool_exhaustion_is_nomem_and_recoverable(tiny):
    """A pool of 3 pages holds 48 positions: a longer sequence is refused
    with SV_E_NOMEM, the context is unchanged, and truncation frees pages."""
    cfg, dw = tiny
    sv = _codes()
    ctx = gh.context(cfg, dw, max_k=8, max_seq=256, max_pages=3)
    t = ctx.prefill(inputs.prefix_tokens(71, 41, cfg.vocab))
    before = _snapshot(ctx, cfg)
    msg = _expect(sv.SV_E_NOMEM, ctx.prefill, [1] * 8)        # 49 > 48
    assert "page" in msg
    _expect(sv.SV_E_NOMEM, ctx.verify, [t] + [2] * 7)         # 41 + 8 > 48
    assert _same(before, _snapshot(ctx, cfg))
    n, c = ctx.verify([t] + [2] * 6)                          # exactly 48 fits
    assert len(ctx) == 41 + n + 1
    ctx.truncate(16)                                          # frees the pages past 16
    ctx.prefill([3] * 32)                                     # 48 again
    assert len(ctx) == 48


def test_async_pending_is_state_error(tiny):
    cfg, dw = tiny
    sv = _codes()
    ctx = gh.context(cfg, dw, max_k=8, max_seq=128)
    t = ctx.prefill(inputs.prefix_tokens(72, 30, cfg.vocab))
    toks = torch.tensor([t, 4, 5, 6], dtype=torch.int32, device="cuda")
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    ctx.reserve(len(ctx) + 4)
    ctx.verify_async(toks, 4, res)
    msg = _expect(sv.SV_E_STATE, ctx.verify, [t, 4, 5, 6])
    assert "sync" in msg
    ctx.sync()
    assert len(ctx) == 30 + int(res[0]) + 1 == int(res[2])
    assert int(res[3]) == 0
    ctx.decode(int(res[1]))                                  # usable again


def test_bad_configurations_are_rejected(tiny):
    cfg, dw = tiny
    sv = _codes()
    bad = [
        dataclasses.replace(cfg, hidden=200),          # not a multiple of 128
        dataclasses.replace(cfg, n_q_heads=3),         # not a multiple of the KV heads
        dataclasses.replace(cfg, head_dim=96),         # unsupported head size
        dataclasses.replace(cfg, ffn=700),             # not a multiple of 64
        dataclasses.replace(cfg, n_layers=0, vocab=0), # no vocabulary
    ]
    for c in bad:
        with pytest.raises(sv.SvError) as e:
            sv.Context(c, dw, max_k=8, max_seq=64)
        assert e.value.code == sv.SV_E_INVAL, c
    with pytest.raises(sv.SvError) as e:
        sv.Context(cfg, dw, max_k=33, max_seq=64)  # more rows than a step holds (32)
    assert e.value.code == sv.SV_E_INVAL


def test_a_partial_that_never_arrives_times_out_and_a_new_context_works(monkeypatch):
    """Failure detection without a fault: with the test switch, one CTA of the
    step's first linear withholds its split-tile partial, so the tile's
    reducer polls a tag that nothing sets.  Its wait is bounded (2 s): the
    kernel gives up, raises the timeout bit and returns, the call reports
    SV_E_CUDA, and the device stays usable -- a new context computes what a
    context that never saw the switch computes."""
    sv = _codes()
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=1, vocab=8192)  # split tiles in the QKV linear
    _, dw = gh.make(cfg, seed=0, gain_std=0.1, host=False)
    prompt = inputs.prefix_tokens(73, 6, cfg.vocab)
    ref = gh.context(cfg, dw, max_k=8, max_seq=64)
    t_ref = ref.prefill(prompt)
    lg_ref = gh.logits_buf(4, cfg.vocab)
    ref.verify([t_ref, 1, 2, 3], logits=lg_ref)
    monkeypatch.setenv("SV_TEST_WITHHOLD_PARTIAL", "1")
    bad = gh.context(cfg, dw, max_k=8, max_seq=64)
    msg = _expect(sv.SV_E_CUDA, bad.prefill, prompt)
    assert "status 0x1" in msg and "timeout" in msg
    bad.close()
    monkeypatch.delenv("SV_TEST_WITHHOLD_PARTIAL")
    fresh = gh.context(cfg, dw, max_k=8, max_seq=64)
    assert fresh.prefill(prompt) == t_ref
    lg = gh.logits_buf(4, cfg.vocab)
    fresh.verify([t_ref, 1, 2, 3], logits=lg)
    assert torch.equal(lg, lg_ref)
