"""The allocation-free LM-head call (sv_lm_head_noalloc) against the context
path that owns its buffers.

Callers of the allocation-free call are those that may not cudaMalloc: code
inside a process whose device memory another allocator has already reserved
(a serving runtime's pool or a plugin in it), and latency-critical code that
cannot take the synchronisation an allocation may bring. For a model with no
layers, sv_verify computes exactly embed -> final RMSNorm -> LM head ->
argmax, with the same K split and rounding, so its logits are the reference
for this call on the same rows, bit for bit: this call runs the mma.sync form
of the linear at every row count, the context the tcgen05 form for 9..32
rows, and the two forms are bit-identical.
This file is collected last so a failure here leaves every other test run.
"""
import pytest

import inputs
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _compare(cfg, tokens, seed):
    import greedy_speculative_decode_gb300 as sv
    dw = inputs.device_weights(cfg, seed=seed, gain_std=0.1)
    K = len(tokens)
    ctx = gh.context(cfg, dw, max_k=32, max_seq=64)
    ref = gh.logits_buf(K, cfg.vocab)
    ctx.verify(tokens, logits=ref)
    ref_am = ref.argmax(dim=1).to(torch.int32)
    ctx.close()
    x = dw[("embed", -1)][torch.tensor(tokens, device="cuda")].contiguous()
    gain = dw[("final_norm", -1)]
    w = dw.get(("lm_head", -1), dw[("embed", -1)])
    for call in range(2):  # two calls in a row share the fixed scratch array
        lg = gh.logits_buf(K, cfg.vocab)
        am = torch.full((K,), -1, dtype=torch.int32, device="cuda")
        st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        sv.lm_head_noalloc(x, gain, w, lg, am, st, eps=cfg.rms_eps)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: kernel status {int(st.item())}"
        err = (lg.double() - ref.double()).abs().max().item()
        assert torch.equal(lg, ref), f"call {call}: logits differ from the context's (max {err})"
        assert torch.equal(am, ref_am), f"call {call}: argmax differs"


def test_no_alloc_lm_head_matches_context_tiny():
    cfg = inputs.shrink(inputs.TINY, n_layers=0)
    _compare(cfg, [5, 77, 901, 3, 1023], seed=3)


def test_no_alloc_lm_head_matches_context_wide():
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=0, vocab=32768)
    _compare(cfg, [11, 2049, 30000, 7], seed=4)


def test_no_alloc_lm_head_matches_context_32_rows():
    """32 rows: the four-token-tile kernel with its own ring and window
    geometry, against the context's LM head on the same rows."""
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=0, vocab=32768)
    _compare(cfg, [(7919 * j + 11) % 32768 for j in range(32)], seed=5)


def test_no_alloc_lm_head_matches_context_full_vocab():
    """The 151,936-id vocabulary of the 8B-shaped model (1187 tiles, split
    tiles between neighbouring CTAs) fits the fixed scratch."""
    cfg = inputs.shrink(inputs.QWEN3_8B, n_layers=0)
    _compare(cfg, [3, 151935, 70000, 12, 99999], seed=6)


def test_no_alloc_rejects_shapes_beyond_the_scratch():
    """32 rows of a 3,000,000-id vocabulary: the argmax partials alone
    (8 bytes per row per 128-id tile) take 6 MB, the split-tile slots
    (4 bytes per tile row and padded row per CTA) 2.5 MB: more than the
    fixed 8 MiB."""
    import greedy_speculative_decode_gb300 as sv
    V = 3_000_000
    x = torch.zeros((32, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.ones((128,), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((V, 128), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((32, V), dtype=torch.float32, device="cuda")
    with pytest.raises(sv.SvError) as e:
        sv.lm_head_noalloc(x, g, w, lg)
    assert e.value.code == sv.SV_E_NOMEM


def test_no_alloc_rejects_mismatched_buffers_before_any_device_work():
    """The C call takes raw pointers; the binding checks what they point to
    (a too-small logits buffer would be written out of bounds)."""
    import greedy_speculative_decode_gb300 as sv
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones((256,), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((1024, 256), dtype=torch.bfloat16, device="cuda")
    bad = [
        dict(logits=torch.empty((4, 1000), dtype=torch.float32, device="cuda")),   # too few ids
        dict(logits=torch.empty((4, 1024), dtype=torch.bfloat16, device="cuda")),  # wrong dtype
        dict(logits=torch.empty((1024, 4), dtype=torch.float32, device="cuda").t()),  # strided
        dict(argmax=torch.empty((3,), dtype=torch.int32, device="cuda")),
        dict(status=torch.empty((1,), dtype=torch.int64, device="cuda")),
        dict(gain=torch.ones((128,), dtype=torch.bfloat16, device="cuda")),
    ]
    for kw in bad:
        args = dict(x=x, gain=g, w=w, logits=torch.empty((4, 1024), dtype=torch.float32, device="cuda"))
        args.update(kw)
        with pytest.raises(ValueError):
            sv.lm_head_noalloc(**args)
