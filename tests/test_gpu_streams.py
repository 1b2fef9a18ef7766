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
