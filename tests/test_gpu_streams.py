"""A context created on a stream of the caller's runs every call on that
stream (no stream of its own, no event join): same results, bit for bit, as
a context on the default stream, and asynchronous verify steps ordered with
the caller's own work on the stream without any synchronisation in between."""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_caller_stream_matches_default_stream():
    cfg = inputs.shrink(inputs.CONFIGS["qwen3-0.6b-shape"], n_layers=2, vocab=32768)
    _, dw = gh.make(cfg, seed=11, gain_std=0.1, host=False)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    import greedy_speculative_decode_gb300 as sv
    a = sv.Context(cfg, dw, max_k=8, max_seq=512)
    b = sv.Context(cfg, dw, max_k=8, max_seq=512, stream=side)
    prompt = inputs.prefix_tokens(5, 200, cfg.vocab)
    pa = a.prefill(prompt)
    with torch.cuda.stream(side):
        pb = b.prefill(prompt)
    assert pa == pb
    chain = [pa]
    for _ in range(12):
        chain.append(a.decode(chain[-1]))
    # the same windows through the asynchronous call on the caller's stream:
    # windows written, verified and read back by work queued on `side` only
    gen = torch.Generator().manual_seed(3)
    windows, expect = [], []
    i = 0
    while i + 4 < len(chain):
        toks = [chain[i]] + [chain[i + 1 + j] if torch.rand((), generator=gen) < 0.6 else (chain[i + 1 + j] + 1)
                             % cfg.vocab for j in range(3)]
        n = 0
        while n < 3 and toks[1 + n] == chain[i + 1 + n]:
            n += 1
        windows.append(toks)
        expect.append((n, chain[i + n + 1]))
        i += n + 1
    la = gh.logits_buf(4, cfg.vocab)
    b.reserve(len(prompt) + len(chain) + 8)  # asynchronous steps take no pages of their own
    with torch.cuda.stream(side):
        win = torch.tensor(windows, dtype=torch.int32, device="cuda")
        res = torch.full((len(windows), 4), -1, dtype=torch.int32, device="cuda")
        lb = torch.empty((len(windows), 4, cfg.vocab), dtype=torch.float32, device="cuda")
        for j in range(len(windows)):
            b.verify_async(win[j], 4, res[j], lb[j])
        got = res[:, :2].clone()  # queued behind the verify steps on the same stream
    side.synchronize()
    b.sync()
    assert [tuple(x) for x in got.cpu().tolist()] == expect
    # the default-stream context, step by step: the same logits, bit for bit
    a.truncate(len(prompt))
    for j, toks in enumerate(windows):
        n, corr = a.verify(toks, logits=la)
        assert (n, corr) == expect[j]
        assert torch.equal(la.view(torch.int32), lb[j].view(torch.int32)), j
    assert len(a) == len(b)


@pytest.mark.parametrize("graphs", [True, False])
def test_async_and_sync_calls_alternate(graphs, monkeypatch):
    """The asynchronous call reads the caller's token buffer and writes its
    result buffer from inside the step (the step graph's embedding and accept
    nodes re-pointed at each call's buffers; or, without graphs, the kernels
    launched with them).  Alternating it with the synchronous call on the same
    step shape, with a new pair of buffers each time, gives the results and
    logits of synchronous calls alone; host buffers are refused."""
    import greedy_speculative_decode_gb300 as sv
    cfg = inputs.CONFIGS["tiny"]
    _, dw = gh.make(cfg, seed=4, gain_std=0.1, host=False)
    if not graphs:
        monkeypatch.setenv("SV_NO_GRAPHS", "1")
    a = gh.context(cfg, dw, max_k=8, max_seq=256)
    monkeypatch.delenv("SV_NO_GRAPHS", raising=False)
    ref = gh.context(cfg, dw, max_k=8, max_seq=256)
    prompt = inputs.prefix_tokens(9, 37, cfg.vocab)
    pa = a.prefill(prompt)
    assert ref.prefill(prompt) == pa
    chain = [pa]
    for _ in range(40):
        chain.append(ref.decode(chain[-1]))
    ref.truncate(len(prompt))
    la, lr = gh.logits_buf(4, cfg.vocab), gh.logits_buf(4, cfg.vocab)
    i, step = 0, 0
    while i + 4 < len(chain):
        toks = [chain[i], chain[i + 1], chain[i + 2] if step % 3 else (chain[i + 2] + 7) % cfg.vocab,
                chain[i + 3]]
        expect = ref.verify(toks, logits=lr)
        if step % 2 == 0:
            tok_dev = torch.tensor(toks, dtype=torch.int32, device="cuda")
            res = torch.full((4,), -5, dtype=torch.int32, device="cuda")
            a.reserve(len(a) + 4)  # (sync released the pages past the length)
            a.verify_async(tok_dev, 4, res, la)
            a.sync()
            r = res.cpu().tolist()
            got = (r[0], r[1])
            assert r[2] == len(prompt) + i + r[0] + 1 and r[3] == 0
        else:
            got = a.verify(toks, logits=la)
        assert got == expect, step
        assert torch.equal(la.view(torch.int32), lr.view(torch.int32)), step
        assert len(a) == len(ref)
        i += got[0] + 1
        step += 1
    assert step >= 8
    host_toks = torch.tensor([chain[i], 1, 2, 3], dtype=torch.int32)
    res = torch.zeros((4,), dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SvError) as e:
        a.verify_async(host_toks, 4, res)
    assert e.value.code == sv.SV_E_INVAL
    assert a.verify([chain[i]]) == ref.verify([chain[i]])  # nothing changed by the refused call
