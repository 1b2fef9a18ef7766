"""The tcgen05 form of the linear (blocks of 9 to 32 rows, and prefill blocks
of up to 128) against the mma.sync form: the same prefill and verify steps on
two contexts, one with the tcgen05 form switched off (SV_NO_TC=1, which also
cuts prefills into 32-row blocks), give byte-identical logits, K/V,
acceptance and corrections.  Run on the full-width 0.6B-, 8B- and Gemma-like
shapes cut to two layers, so every weight shape, head layout, K partition and
split-tile exchange of the full models goes through both forms."""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", params=["qwen3-0.6b-shape", "qwen3-8b-shape", "gemma-like"])
def model(request):
    cfg = inputs.shrink(inputs.CONFIGS[request.param], n_layers=2)
    _, dw = gh.make(cfg, seed=3, gain_std=0.1, host=False)
    return cfg, dw


def _pair(cfg, dw, monkeypatch, max_seq):
    tc = gh.context(cfg, dw, max_k=32, max_seq=max_seq, shuffle=5)
    monkeypatch.setenv("SV_NO_TC", "1")
    ref = gh.context(cfg, dw, max_k=32, max_seq=max_seq, shuffle=9)
    monkeypatch.delenv("SV_NO_TC")
    return tc, ref


def _same_cache(cfg, a, b):
    assert len(a) == len(b)
    for layer in range(cfg.n_layers):
        ka, va = a.kv_read(layer, 0, len(a))
        kb, vb = b.kv_read(layer, 0, len(b))
        assert torch.equal(ka.view(torch.int16), kb.view(torch.int16)), layer
        assert torch.equal(va.view(torch.int16), vb.view(torch.int16)), layer


@pytest.mark.parametrize("K", [9, 12, 16, 17, 24, 32])
def test_verify_identical_with_and_without_tcgen05(model, monkeypatch, K):
    cfg, dw = model
    prompt = inputs.prefix_tokens(40 + K, 300 + K, cfg.vocab)  # prefill: 32-row blocks and a ragged one
    tc, ref = _pair(cfg, dw, monkeypatch, max_seq=300 + K + 3 * K + 8)
    p_tc, p_ref = tc.prefill(prompt), ref.prefill(prompt)
    assert p_tc == p_ref
    _same_cache(cfg, tc, ref)
    gen = torch.Generator().manual_seed(K)
    pending = p_tc
    for step in range(3):
        drafts = torch.randint(0, cfg.vocab, (K - 1,), generator=gen).tolist()
        if step == 1:  # a window that accepts some drafts: the target's own continuation
            drafts[: K // 2] = [pending] * (K // 2)
        lg_tc, lg_ref = gh.logits_buf(K, cfg.vocab), gh.logits_buf(K, cfg.vocab)
        r_tc = tc.verify([pending] + drafts, logits=lg_tc)
        r_ref = ref.verify([pending] + drafts, logits=lg_ref)
        assert r_tc == r_ref, step
        assert torch.equal(lg_tc.view(torch.int32), lg_ref.view(torch.int32)), step
        _same_cache(cfg, tc, ref)
        pending = r_tc[1]


@pytest.mark.parametrize("K", [16, 32])
def test_rows_of_a_wide_block_equal_decode(model, monkeypatch, K):
    """Each row of a 16- or 32-row all-accept verify on the tcgen05 form
    equals the single-token decode of its prefix (mma.sync, one token row),
    bit for bit."""
    cfg, dw = model
    prompt = inputs.prefix_tokens(91, 70, cfg.vocab)
    dec = gh.context(cfg, dw, max_k=32, max_seq=70 + K + 8)
    lg1 = gh.logits_buf(1, cfg.vocab)
    t = dec.prefill(prompt)
    chain, rows = [t], []
    for _ in range(K):
        t = dec.decode(t, logits=lg1)
        rows.append(lg1.clone())
        chain.append(t)
    ver = gh.context(cfg, dw, max_k=32, max_seq=70 + K + 8, shuffle=2)
    ver.prefill(prompt)
    lgK = gh.logits_buf(K, cfg.vocab)
    n, corr = ver.verify(chain[:K], logits=lgK)
    assert n == K - 1 and corr == chain[K]
    for r in range(K):
        assert torch.equal(lgK[r].view(torch.int32), rows[r][0].view(torch.int32)), f"row {r}"
    _same_cache(cfg, dec, ver)


@pytest.mark.parametrize("n", [87, 300, 1024])
def test_prefill_in_wide_blocks_equals_one_token_commits(model, n):
    """A prompt committed by sv_prefill, whose blocks of up to 128 rows run
    the tcgen05 linears with a 128-column accumulator (the 8B and Gemma-like
    shapes stream more k-blocks per CTA than the ring has stages, so every
    stage is reused), leaves the same K/V and next token as one-token
    commits."""
    cfg, dw = model
    import greedy_speculative_decode_gb300 as sv
    assert max(sv.prefill_blocks(n)) > sv.MAX_K
    prompt = inputs.prefix_tokens(500 + n, n, cfg.vocab)
    ref = gh.context(cfg, dw, max_k=4, max_seq=n + 8)
    t = None
    for tok in prompt:  # one-row commits of forced ids (a one-token prefill is a one-row step)
        t = ref.prefill([tok])
    big = gh.context(cfg, dw, max_k=4, max_seq=n + 8, shuffle=7)
    assert big.prefill(prompt) == t
    _same_cache(cfg, ref, big)


def test_wide_prefill_repeats_exactly(model):
    """Sixteen prefills of one 300-token prompt (blocks of 128, 128, 32 and 12
    rows) into one context, truncated to zero in between so that the graphs
    replay and the pages are reused, each equal to the first byte for byte:
    a race in the 128-row form (ring stage reuse, the accumulator hand-off,
    the chunked read-back, the split-tile exchange) would show up as a rare
    difference here."""
    cfg, dw = model
    prompt = inputs.prefix_tokens(77, 300, cfg.vocab)
    ctx = gh.context(cfg, dw, max_k=4, max_seq=320, shuffle=3)
    first = None
    for rep in range(16):
        ctx.truncate(0)
        lg = gh.logits_buf(1, cfg.vocab)
        t = ctx.prefill(prompt, logits=lg)
        kv = [tuple(x.view(torch.int16).clone() for x in ctx.kv_read(layer, 0, 300)) for layer in range(cfg.n_layers)]
        if first is None:
            first = (t, lg.clone(), kv)
            continue
        assert t == first[0], f"repeat {rep}: next token"
        assert torch.equal(lg.view(torch.int32), first[1].view(torch.int32)), f"repeat {rep}: logits"
        for layer in range(cfg.n_layers):
            assert torch.equal(kv[layer][0], first[2][layer][0]), f"repeat {rep}: K of layer {layer}"
            assert torch.equal(kv[layer][1], first[2][layer][1]), f"repeat {rep}: V of layer {layer}"
