"""GPU path vs the CPU oracle, and bit-exactness of block verify against
single-token decode, on seeded tiny models (all through the C-ABI)."""
import numpy as np
import pytest

import inputs
import oracle
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tiny():
    cfg = inputs.TINY
    hw, dw = gh.make(cfg, seed=0, gain_std=0.1)
    return cfg, hw, dw


def test_prefill_and_decode_match_oracle(tiny):
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(0, 32, cfg.vocab)
    ctx = gh.context(cfg, dw, max_k=8, max_seq=128)
    orc = oracle.OracleModel(hw, 128)
    lg = gh.logits_buf(1, cfg.vocab)
    t = ctx.prefill(prompt, logits=lg)
    lo, to = orc.prefill(prompt)
    gh.assert_close_to_oracle(lg.cpu().numpy()[0], lo, "prefill")
    assert t == to
    for step in range(12):
        t_gpu = ctx.decode(t, logits=lg)
        lo, t_orc = orc.decode(t)
        gh.assert_close_to_oracle(lg.cpu().numpy()[0], lo, f"decode {step}")
        assert t_gpu == t_orc
        t = t_gpu
    assert len(ctx) == len(orc) == 32 + 12


def test_verify_steps_match_decode_and_oracle(tiny):
    """The tiny workload: 16 verify steps of K=4 over the target's own greedy
    chain with each draft slot replaced with probability 0.5."""
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(0, 32, cfg.vocab)
    K, steps = 4, 16
    # the greedy chain and its decode logits, on the GPU
    dec = gh.context(cfg, dw, max_k=8, max_seq=256)
    lg1 = gh.logits_buf(1, cfg.vocab)
    t = dec.prefill(prompt)
    chain, dec_logits = [t], []
    for _ in range(steps * K + 1):
        t = dec.decode(t, logits=lg1)
        dec_logits.append(lg1.clone())
        chain.append(t)
    sched = inputs.schedule(chain, K, steps, seq=0, p=0.5, vocab=cfg.vocab)
    ver = gh.context(cfg, dw, max_k=8, max_seq=256, shuffle=7)
    ver.prefill(prompt)
    orc = oracle.OracleModel(hw, 256)
    orc.prefill(prompt)
    lgK = gh.logits_buf(K, cfg.vocab)
    accepted = 0
    for (i, toks, n_exp) in sched:
        n, corr = ver.verify(toks, logits=lgK)
        lo, am, n_o, c_o = orc.verify(toks)
        assert n == n_exp == n_o, (i, toks, n, n_exp, n_o)
        assert corr == chain[i + n + 1] == c_o
        g = lgK.cpu().numpy()
        gh.assert_close_to_oracle(g, lo, f"verify at chain index {i}")
        for r in range(n + 1):  # rows whose prefix is on the greedy chain
            assert torch.equal(lgK[r], dec_logits[i + r][0]), f"row {r} != decode at {i + r}"
        accepted += n
        assert len(ver) == len(orc) == len(prompt) + i + n + 1
    assert accepted > 0


@pytest.mark.parametrize("K", [1, 2, 3, 7, 8, 9, 16, 17, 32])
def test_rows_bit_identical_to_decode_for_every_width(tiny, K):
    """All-accept verify of K rows equals K single-token decodes, byte for byte,
    including K that use one, two and four 8-column mma tiles."""
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(1, 45, cfg.vocab)
    dec = gh.context(cfg, dw, max_k=32, max_seq=256)
    lg1 = gh.logits_buf(1, cfg.vocab)
    t = dec.prefill(prompt)
    chain, rows = [t], []
    for _ in range(K):
        t = dec.decode(t, logits=lg1)
        rows.append(lg1.clone())
        chain.append(t)
    ver = gh.context(cfg, dw, max_k=32, max_seq=256, shuffle=K)
    ver.prefill(prompt)
    lgK = gh.logits_buf(K, cfg.vocab)
    n, corr = ver.verify(chain[:K], logits=lgK)
    assert n == K - 1 and corr == chain[K]
    for r in range(K):
        assert torch.equal(lgK[r], rows[r][0]), f"row {r}"
    for layer in range(cfg.n_layers):
        kd, vd = dec.kv_read(layer, 0, len(dec))
        kv, vv = ver.kv_read(layer, 0, len(ver))
        assert torch.equal(kd.view(torch.int16), kv.view(torch.int16))
        assert torch.equal(vd.view(torch.int16), vv.view(torch.int16))


def test_k1_verify_equals_decode(tiny):
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(2, 20, cfg.vocab)
    a = gh.context(cfg, dw)
    b = gh.context(cfg, dw)
    t = a.prefill(prompt)
    b.prefill(prompt)
    la, lb = gh.logits_buf(1, cfg.vocab), gh.logits_buf(1, cfg.vocab)
    n, c = a.verify([t], logits=la)
    nd = b.decode(t, logits=lb)
    assert n == 0 and c == nd and torch.equal(la, lb)


def test_row0_ignores_later_rows(tiny):
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(3, 30, cfg.vocab)
    outs = []
    for drafts in ([1, 2, 3], [900, 17, 5], [0, 0, 0], [4, 4, 4, 4, 4, 4, 4]):
        ctx = gh.context(cfg, dw)
        t0 = ctx.prefill(prompt)
        lg = gh.logits_buf(1 + len(drafts), cfg.vocab)
        ctx.verify([t0] + drafts, logits=lg)
        outs.append(lg[0].clone())
    assert all(torch.equal(outs[0], o) for o in outs)


def test_three_cache_histories_identical(tiny):
    """The same committed prefix built by one-token commits, by accepted
    8-row blocks and by one prefill gives identical logits and K/V bytes."""
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(4, 9, cfg.vocab)
    # reference greedy chain
    ref = gh.context(cfg, dw, max_k=16, max_seq=256)
    chain = gh.greedy_chain_gpu(ref, prompt, 90)
    committed = prompt + chain[:78]  # 87 ids, the length of the page's failing prefix
    probe = chain[78:78 + 8]         # a verify window after that prefix
    # (a) one-token commits
    a = gh.context(cfg, dw, max_k=16, max_seq=256, shuffle=1)
    gh.commit(a, committed[1:], a.prefill(committed[:1]))
    # (b) accepted 8-row blocks: prompt, then K=8 all-accept verifies along the chain
    b = gh.context(cfg, dw, max_k=16, max_seq=256, shuffle=2)
    b.prefill(prompt)
    i, pending = 0, None
    while len(b) + 8 <= len(committed):
        n, pending = b.verify(chain[i:i + 8])
        assert n == 7
        i += 8
    gh.commit(b, committed[len(b):], pending)
    # (c) one fresh prefill
    c = gh.context(cfg, dw, max_k=16, max_seq=256, shuffle=3)
    c.prefill(committed)
    assert len(a) == len(b) == len(c) == len(committed)
    outs = []
    for ctx in (a, b, c):
        lg = gh.logits_buf(8, cfg.vocab)
        ctx.verify(probe, logits=lg)
        outs.append(lg)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    for layer in range(cfg.n_layers):
        ka, va = a.kv_read(layer, 0, len(committed))
        for other in (b, c):
            ko, vo = other.kv_read(layer, 0, len(committed))
            assert torch.equal(ka.view(torch.int16), ko.view(torch.int16))
            assert torch.equal(va.view(torch.int16), vo.view(torch.int16))


def test_truncate_then_verify_equals_fresh(tiny):
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(5, 40, cfg.vocab)
    ref = gh.context(cfg, dw, max_k=16, max_seq=256)
    chain = gh.greedy_chain_gpu(ref, prompt, 30)
    x = gh.context(cfg, dw, max_k=16, max_seq=256)
    x.prefill(prompt)
    toks, n_exp = inputs.window(chain, 0, 8, vocab=cfg.vocab, reject_at=2)
    n, corr = x.verify(toks)
    assert n == n_exp == 2 and corr == chain[3]
    # rejected rows are zeroed: the pages hold nothing beyond the length
    x.truncate(len(prompt) + 2)
    lg_x = gh.logits_buf(6, cfg.vocab)
    nx, cx = x.verify(chain[2:8], logits=lg_x)
    y = gh.context(cfg, dw, max_k=16, max_seq=256)
    y.prefill(prompt + chain[:2])
    lg_y = gh.logits_buf(6, cfg.vocab)
    ny, cy = y.verify(chain[2:8], logits=lg_y)
    assert (nx, cx) == (ny, cy) and torch.equal(lg_x, lg_y)
    for layer in range(cfg.n_layers):
        kx, vx = x.kv_read(layer, 0, len(x))
        ky, vy = y.kv_read(layer, 0, len(y))
        assert torch.equal(kx.view(torch.int16), ky.view(torch.int16))
        assert torch.equal(vx.view(torch.int16), vy.view(torch.int16))


@pytest.mark.parametrize("plen", [1, 15, 16, 17, 63, 64, 65, 255, 256, 257, 511, 700])
def test_ragged_prefix_lengths(tiny, plen):
    """Prefixes that end inside or at the edge of a page, a warp's 64
    positions and a 256-position split; verify of 5 rows across the edge."""
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(6, plen, cfg.vocab)
    ctx = gh.context(cfg, dw, max_k=8, max_seq=1024, shuffle=plen)
    t = ctx.prefill(prompt)
    orc = oracle.OracleModel(hw, 1024)
    _, to = orc.prefill(prompt)
    assert t == to
    toks = [t, 3, 5, 7, 11]
    lg = gh.logits_buf(5, cfg.vocab)
    n, c = ctx.verify(toks, logits=lg)
    lo, am, no, co = orc.verify(toks)
    assert (n, c) == (no, co)
    gh.assert_close_to_oracle(lg.cpu().numpy(), lo, f"prefix {plen}")


def test_decode_past_split_boundaries_bitexact(tiny):
    """Verify rows that straddle a 256-position split equal decodes."""
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(7, 250, cfg.vocab)
    dec = gh.context(cfg, dw, max_k=16, max_seq=512)
    t = dec.prefill(prompt)
    lg1 = gh.logits_buf(1, cfg.vocab)
    chain, rows = [t], []
    for _ in range(12):
        t = dec.decode(t, logits=lg1)
        rows.append(lg1.clone())
        chain.append(t)
    ver = gh.context(cfg, dw, max_k=16, max_seq=512, shuffle=11)
    ver.prefill(prompt)
    lg = gh.logits_buf(12, cfg.vocab)
    n, _ = ver.verify(chain[:12], logits=lg)
    assert n == 11
    for r in range(12):
        assert torch.equal(lg[r], rows[r][0]), r


def test_prefill_blocks_do_not_depend_on_max_k(tiny):
    """Prefill runs 32-row blocks whatever max_k is: a 100-token prompt
    committed by contexts with max_k 1, 4 and 32 gives the same next token
    and the same K/V as committing it one decode at a time."""
    cfg, hw, dw = tiny
    prompt = inputs.prefix_tokens(77, 100, cfg.vocab)
    ref = gh.context(cfg, dw, max_k=1, max_seq=128)
    nxt = gh.commit(ref, prompt[1:], ref.prefill(prompt[:1]))
    for mk in (1, 4, 32):
        ctx = gh.context(cfg, dw, max_k=mk, max_seq=128, shuffle=mk)
        assert ctx.prefill(prompt) == nxt, mk
        for layer in range(cfg.n_layers):
            ka, va = ref.kv_read(layer, 0, 100)
            kb, vb = ctx.kv_read(layer, 0, 100)
            assert torch.equal(ka.view(torch.int16), kb.view(torch.int16)), (mk, layer)
            assert torch.equal(va.view(torch.int16), vb.view(torch.int16)), (mk, layer)
