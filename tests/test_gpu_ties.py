"""Exact ties in the greedy argmax on the GPU.

The greedy rule takes the largest bf16 logit and, among equal ones, the
lowest token id: the Gemma page's position-60 table ("Shape and cache
history in Gemma block verification", section "Same-prefix controls") has a
one-token row with logits 22.75 = 22.75 that selects the lower id 12630 over
54945, and the decode row of "Phase 23: Speculative Verify Parity" section 1
lists two equal 24.500 logits.  The GPU takes the argmax in two stages (per
128-id tile inside the LM head, then across tiles in the accept kernel), so a
tie can meet inside one tile, across tiles of one CTA, or across CTAs.

Each case copies the LM-head row of a row's winning id into another id, so
both ids get the same logit, and checks that verify (argmax, acceptance and
correction), single-token decode, the allocation-free LM head and the oracle's
head on the GPU's own final hidden state all pick the lower id.
"""
import numpy as np
import pytest

import inputs
import oracle
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CFG = inputs.shrink(inputs.QWEN3_8B, n_layers=1)  # full width, untied 151,936-id head
PROMPT = inputs.prefix_tokens(90, 40, CFG.vocab)
SEED = 7


@pytest.fixture(scope="module")
def base():
    hw, dw = gh.make(CFG, seed=SEED, gain_std=0.1)
    ctx = gh.context(CFG, dw, max_k=8, max_seq=96)
    t = ctx.prefill(PROMPT)
    lg = gh.logits_buf(4, CFG.vocab)
    ctx.verify([t, 11, 12, 13], logits=lg)
    winner = int(lg[0].argmax())
    ctx.close()
    return hw, dw, t, winner


def _partner(a, kind):
    V, tile = CFG.vocab, 128
    if kind == "other_cta":      # half the vocabulary away: another CTA's range
        return (a + V // 2) % V
    if kind == "same_tile":      # the same 128-id tile
        j = (a % tile + 64) % tile
        return (a // tile) * tile + j
    if kind == "adjacent_tile":  # the last id of the previous tile (or first of the next)
        return (a // tile) * tile - 1 if a >= tile else tile
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["other_cta", "same_tile", "adjacent_tile"])
def test_exact_tie_goes_to_the_lower_id(base, kind):
    import greedy_speculative_decode_gb300 as sv
    hw, dw0, t, a = base
    i = _partner(a, kind)
    assert i != a
    lo_id, hi_id = min(i, a), max(i, a)
    # the same model with LM-head row i replaced by row a
    dw = dict(dw0)
    head = dw0[("lm_head", -1)].clone()
    head[i] = head[a]
    dw[("lm_head", -1)] = head
    hw = inputs.HostWeights(hw.cfg, hw.seed, hw.gain_std, dict(hw.tensors))
    hw.tensors[("lm_head", -1)] = hw.tensors[("lm_head", -1)].copy()
    hw.tensors[("lm_head", -1)][i] = hw.tensors[("lm_head", -1)][a]

    ctx = gh.context(CFG, dw, max_k=8, max_seq=96)
    trace = torch.zeros((CFG.n_layers + 1, 4, CFG.hidden), dtype=torch.bfloat16, device="cuda")
    ctx.trace_hidden(trace, 4)
    assert ctx.prefill(PROMPT) == t
    lg = gh.logits_buf(4, CFG.vocab)
    # draft 1 is the higher id of the tied pair: rejected, correction = the lower id
    n, corr = ctx.verify([t, hi_id, 5, 6], logits=lg)
    x_final = trace[CFG.n_layers].clone()
    ctx.trace_hidden(None)
    assert float(lg[0, i]) == float(lg[0, a]) == float(lg[0].max()), "the copied rows must tie"
    assert (n, corr) == (0, lo_id), (kind, a, i, n, corr)
    # draft 1 = the lower id: accepted
    ctx.truncate(len(PROMPT))
    n2, _ = ctx.verify([t, lo_id, 5, 6])
    assert n2 >= 1
    # single-token decode of the same prefix picks it too
    dec = gh.context(CFG, dw, max_k=8, max_seq=96)
    dec.prefill(PROMPT)
    lg1 = gh.logits_buf(1, CFG.vocab)
    assert dec.decode(t, logits=lg1) == lo_id
    assert torch.equal(lg1[0], lg[0])
    # the allocation-free LM head on the same final hidden rows
    lgn = gh.logits_buf(4, CFG.vocab)
    am = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    sv.lm_head_noalloc(x_final, dw[("final_norm", -1)], head, lgn, am, eps=CFG.rms_eps)
    torch.cuda.synchronize()
    assert int(am[0]) == lo_id and torch.equal(lgn, lg)
    # the oracle's head on the GPU's own final hidden state: same tie, same choice
    xo = x_final.view(torch.int16).cpu().numpy().view(np.uint16)
    lo = oracle.LayerOracle(hw).head(xo[:1])[0]
    assert lo[i] == lo[a] and int(np.argmax(lo)) == lo_id
    assert oracle.argmax(lo) == lo_id
    gh.assert_close_to_oracle(lg[0].cpu().numpy(), lo, f"tie {kind}")


def test_one_step_apart_goes_to_the_larger(base):
    """A near-tie one bf16 step apart: row i = row a with one weight changed so
    that its logit lands one bf16 step above; verify, decode and the
    allocation-free head all pick i, and their logits are identical."""
    import greedy_speculative_decode_gb300 as sv
    hw, dw0, t, a = base
    i = _partner(a, "other_cta")
    ctx0 = gh.context(CFG, dw0, max_k=8, max_seq=96)
    trace = torch.zeros((CFG.n_layers + 1, 1, CFG.hidden), dtype=torch.bfloat16, device="cuda")
    ctx0.trace_hidden(trace, 1)
    ctx0.prefill(PROMPT)
    lg0 = gh.logits_buf(1, CFG.vocab)
    ctx0.decode(t, logits=lg0)
    top = float(lg0[0, a])
    # the normalised final row the head multiplies: y = bf16(bf16(x * rstd) * g)
    x = trace[CFG.n_layers, 0].float()
    rstd = 1.0 / torch.sqrt((x * x).mean() + CFG.rms_eps)
    y = ((x * rstd).bfloat16().float() * dw0[("final_norm", -1)].float()).bfloat16().float()
    k = int(torch.argmax(y.abs()))
    step = 2.0 ** (np.floor(np.log2(abs(top))) - 7)  # one bf16 step at the logit's magnitude
    head = dw0[("lm_head", -1)].clone()
    head[i] = head[a]
    w_new = (float(head[i, k]) + 1.5 * step / float(y[k]))
    head[i, k] = torch.tensor(w_new, dtype=torch.bfloat16)
    dw = dict(dw0)
    dw[("lm_head", -1)] = head
    ctx = gh.context(CFG, dw, max_k=8, max_seq=96)
    ctx.prefill(PROMPT)
    lg = gh.logits_buf(4, CFG.vocab)
    n, corr = ctx.verify([t, a, 5, 6], logits=lg)
    li, la = float(lg[0, i]), float(lg[0, a])
    assert li > la, (li, la)
    assert (n, corr) == (0, i)
    dec = gh.context(CFG, dw, max_k=8, max_seq=96)
    dec.prefill(PROMPT)
    lg1 = gh.logits_buf(1, CFG.vocab)
    assert dec.decode(t, logits=lg1) == i and torch.equal(lg1[0], lg[0])
    lgn = gh.logits_buf(1, CFG.vocab)
    am = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    sv.lm_head_noalloc(trace[CFG.n_layers].clone(), dw[("final_norm", -1)], head, lgn, am,
                       eps=CFG.rms_eps)
    torch.cuda.synchronize()
    assert int(am[0]) == i and torch.equal(lgn[0], lg[0])
