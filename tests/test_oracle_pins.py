"""Pins of the CPU oracle to facts it does not define itself.

Every test here runs on the CPU (no GPU marker). They tie the oracle to:
values printed on the pages (tests/golden), closed forms, textbook special
cases, PyTorch library routines in float64, and brute-force recomputation.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import inputs
import oracle
from tests import torch_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append([c.strip() for c in line.split("|")])
    return out


def _bits(x):
    return oracle.f32_to_bits(np.asarray(x, dtype=np.float32))


# --------------------------------------------------------- bf16 rounding
@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (1.0 + 2.0 ** -8, 0x3F80),             # halfway, even neighbour below
    (1.0 + 3 * 2.0 ** -8, 0x3F82),         # halfway, even neighbour above
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # just above halfway rounds up
    (1.0 + 2.0 ** -8 - 2.0 ** -20, 0x3F80),  # just below halfway rounds down
    (float("inf"), 0x7F80), (3.4e38, 0x7F80),  # above the largest bf16 -> inf
    (22.8, 0x41B6), (22.8125, 0x41B6),     # 22.75 = 0x41B6; 22.8125 ties to even
])
def test_bf16_round_nearest_even(x, bits):
    assert oracle.bf16(x) == bits


def test_bf16_nan_stays_nan():
    b = oracle.bf16(float("nan"))
    assert (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


def test_page_logits_are_bf16_values():
    """Every logit the pages print is a bf16 value, spaced 0.125 in [16, 32)."""
    vals = [float(r[2]) for r in _rows("p3_position60_table.txt")]
    vals += [float(r[3]) for r in _rows("p3_position60_table.txt")]
    vals += [float(r[1]) for r in _rows("p3_position54_receipt.txt")]
    vals += [float(r[2]) for r in _rows("p3_position54_receipt.txt")]
    for r in _rows("p2_verify_decode_top2.txt"):
        vals += [float(p.split(":")[1]) for p in r[1].split(",")]
    for v in vals:
        assert 16.0 <= v < 32.0
        assert oracle.f32(oracle.bf16(v)) == v
        assert (v * 8.0) == int(v * 8.0)


# --------------------------------------------------------- argmax ties
def _two_logit_vector(a_id, a, b_id, b, vocab=262144, fill=-10.0):
    v = np.full(vocab, fill, dtype=np.float32)
    v[a_id], v[b_id] = a, b
    return v


@pytest.mark.parametrize("row", _rows("p3_position60_table.txt") + [
    ["receipt54", *r] for r in _rows("p3_position54_receipt.txt")])
def test_argmax_matches_page_selection(row):
    l12630, l54945, selected = float(row[2]), float(row[3]), int(row[4])
    v = _two_logit_vector(12630, l12630, 54945, l54945)
    assert oracle.argmax(v) == selected


def test_decode_tie_lists_lower_id_first():
    rows = {r[0]: r[1] for r in _rows("p2_verify_decode_top2.txt")}
    (i0, v0), (i1, v1) = [(int(p.split(":")[0]), float(p.split(":")[1]))
                          for p in rows["decode"].split(",")]
    assert v0 == v1 and i0 < i1
    v = _two_logit_vector(i0, v0, i1, v1, vocab=151936)
    assert oracle.argmax(v) == i0
    (j0, w0), (j1, w1) = [(int(p.split(":")[0]), float(p.split(":")[1]))
                          for p in rows["verify"].split(",")]
    assert oracle.argmax(_two_logit_vector(j0, w0, j1, w1, vocab=151936)) == j0
    assert w0 - w1 == 0.125  # one bf16 step at this magnitude


# --------------------------------------------------------- single ops
def test_rmsnorm_constant_vector():
    """x = c everywhere: x / sqrt(mean(x^2) + eps) = sign(c) c/sqrt(c^2+eps)."""
    for c, g in [(2.0, 1.0), (-3.0, 1.0), (0.75, 0.5), (5.0, -1.25)]:
        x = _bits(np.full(64, c))
        gg = _bits(np.full(64, g))
        y = oracle.bits_to_f32(oracle.rmsnorm(x, gg, 1e-6))
        expect = math.copysign(1.0, c) * g
        assert np.all(y == np.float32(expect)), (c, g, y[:4])


def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(1)
    x = _bits(rng.normal(0, 3, 300))
    g = _bits(rng.uniform(0.5, 1.5, 300))
    y = oracle.bits_to_f32(oracle.rmsnorm(x, g, 1e-6)).astype(np.float64)
    ref = F.rms_norm(torch.from_numpy(oracle.bits_to_f32(x).astype(np.float64)), (300,),
                     weight=torch.from_numpy(oracle.bits_to_f32(g).astype(np.float64)),
                     eps=1e-6).numpy()
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)


def _bf16_equal_fraction(got_bits, ref64):
    """Fraction of bf16 outputs equal to a float64 reference cast to bf16 by
    the library (torch's own round-to-nearest-even), and the largest gap in
    bf16 steps."""
    ref = torch.from_numpy(np.asarray(ref64, dtype=np.float64)).to(torch.bfloat16)
    ref_bits = ref.view(torch.int16).numpy().view(np.uint16)
    got = np.asarray(got_bits, dtype=np.uint16)
    # bf16 values of one sign are ordered like their bit patterns
    gap = np.abs(got.astype(np.int64) - ref_bits.astype(np.int64))
    same_sign = (got >> 15) == (ref_bits >> 15)
    return float(np.mean(got == ref_bits)), int(np.max(np.where(same_sign, gap, 0)))


def test_rmsnorm_rounding_points_match_library_casts():
    """The stated rounding path of the RMSNorm, bf16(bf16(x * rstd) * g), against
    float64 library arithmetic (F.rms_norm) cast to bf16 by the library at the
    same two points.  The oracle's fp32 intermediates differ from float64 by
    an fp32 rounding, which moves a bf16 result only near a rounding boundary:
    a few outputs in a thousand.  Dropping either rounding moves a large
    share of them (the gains are not 1)."""
    rng = np.random.default_rng(11)
    n = 4096
    x = _bits(rng.normal(0, 2.0, n))
    g = _bits(rng.uniform(0.5, 1.5, n))
    xf = torch.from_numpy(oracle.bits_to_f32(x).astype(np.float64))
    gf = torch.from_numpy(oracle.bits_to_f32(g).astype(np.float64))
    t = F.rms_norm(xf, (n,), eps=1e-6).to(torch.bfloat16).to(torch.float64)
    ref = (t * gf).numpy()
    frac, gap = _bf16_equal_fraction(oracle.rmsnorm(x, g, 1e-6), ref)
    assert frac >= 0.99 and gap <= 1, (frac, gap)


@pytest.mark.parametrize("act", [0, 1])
def test_glu_rounding_points_match_library_casts(act):
    """The gated unit's stated rounding path, bf16(bf16(act(g)) * u), against
    float64 F.silu / F.gelu(tanh) with the library's bf16 casts at the same
    points (same reasoning as the RMSNorm case)."""
    rng = np.random.default_rng(12 + act)
    n = 4096
    gb = _bits(rng.normal(0, 1.3, n))
    ub = _bits(rng.normal(0, 1.3, n))
    gf = torch.from_numpy(oracle.bits_to_f32(gb).astype(np.float64))
    uf = torch.from_numpy(oracle.bits_to_f32(ub).astype(np.float64))
    a = F.silu(gf) if act == 0 else F.gelu(gf, approximate="tanh")
    ref = (a.to(torch.bfloat16).to(torch.float64) * uf).numpy()
    frac, gap = _bf16_equal_fraction(oracle.glu(gb, ub, act), ref)
    assert frac >= 0.99 and gap <= 1, (act, frac, gap)


def test_linear_matches_matmul():
    rng = np.random.default_rng(2)
    W = _bits(rng.normal(0, 0.05, (37, 300)))
    x = _bits(rng.normal(0, 1, 300))
    y = oracle.bits_to_f32(oracle.linear(W, x)).astype(np.float64)
    ref = oracle.bits_to_f32(W).astype(np.float64) @ oracle.bits_to_f32(x).astype(np.float64)
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)
    # row r depends on W[r] only: swapping two rows swaps two outputs
    W2 = W.copy()
    W2[[3, 7]] = W2[[7, 3]]
    y2 = oracle.linear(W2, x)
    y1 = oracle.linear(W, x)
    assert y2[3] == y1[7] and y2[7] == y1[3]


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(3)
    x = _bits(rng.normal(0, 1, 128))
    assert np.array_equal(oracle.rope(x, 0, 1e6), x)


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6), (256, 1e4)])
def test_rope_basis_vectors(d, theta):
    """e_i turns into (cos a, sin a) on the pair (i, i + d/2), a = p theta^(-2i/d)."""
    for i in (0, 1, d // 4, d // 2 - 1):
        for p in (1, 7, 1000, 32767):
            x = np.zeros(d, dtype=np.float32)
            x[i] = 1.0
            y = oracle.bits_to_f32(oracle.rope(_bits(x), p, theta))
            a = p * theta ** (-2.0 * i / d)
            assert abs(y[i] - math.cos(a)) <= 2.0 ** -8
            assert abs(y[i + d // 2] - math.sin(a)) <= 2.0 ** -8
            others = np.delete(y, [i, i + d // 2])
            assert np.all(others == 0.0)


def test_rope_depends_on_relative_position_only():
    rng = np.random.default_rng(4)
    d = 128
    q = _bits(rng.normal(0, 1, d))
    k = _bits(rng.normal(0, 1, d))
    dots = []
    for m, n in [(5, 2), (105, 102), (3005, 3002)]:
        qm = oracle.bits_to_f32(oracle.rope(q, m, 1e4)).astype(np.float64)
        kn = oracle.bits_to_f32(oracle.rope(k, n, 1e4)).astype(np.float64)
        dots.append(qm @ kn)
    # bf16 rounding of the rotated vectors moves a dot product by about
    # 2^-8 * |q| |k| / sqrt(d); a one-position shift moves it by much more.
    tol = 2.0 ** -8 * np.linalg.norm(oracle.bits_to_f32(q)) * \
        np.linalg.norm(oracle.bits_to_f32(k)) / math.sqrt(d)
    assert max(dots) - min(dots) <= 2 * tol
    for m in (4, 6):
        qm = oracle.bits_to_f32(oracle.rope(q, m, 1e4)).astype(np.float64)
        k2 = oracle.bits_to_f32(oracle.rope(k, 2, 1e4)).astype(np.float64)
        assert abs(qm @ k2 - dots[0]) > 10 * tol


def test_attention_single_position_returns_value():
    rng = np.random.default_rng(5)
    q, k, v = (_bits(rng.normal(0, 1, 64)) for _ in range(3))
    out = oracle.attend(q, k[None], v[None])
    assert np.array_equal(out, v)


def test_attention_equal_scores_average_values():
    rng = np.random.default_rng(6)
    q = _bits(rng.normal(0, 1, 64))
    k = _bits(rng.normal(0, 1, 64))
    v0, v1 = _bits(rng.normal(0, 1, 64)), _bits(rng.normal(0, 1, 64))
    out = oracle.attend(q, np.stack([k, k]), np.stack([v0, v1]))
    mean = (oracle.bits_to_f32(v0).astype(np.float64) + oracle.bits_to_f32(v1)) / 2
    assert np.array_equal(out, _bits(mean))


def test_attention_matches_sdpa():
    rng = np.random.default_rng(7)
    d, n = 128, 50
    q = _bits(rng.normal(0, 1, d))
    K = _bits(rng.normal(0, 1, (n, d)))
    V = _bits(rng.normal(0, 1, (n, d)))
    out = oracle.bits_to_f32(oracle.attend(q, K, V)).astype(np.float64)
    f = lambda a: torch.from_numpy(oracle.bits_to_f32(a).astype(np.float64))
    ref = F.scaled_dot_product_attention(f(q)[None, None], f(K)[None], f(V)[None])[0, 0].numpy()
    assert np.all(np.abs(out - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-4)


def test_activations():
    assert oracle.silu(0.0) == 0.0 and oracle.gelu_tanh(0.0) == 0.0
    for x in np.linspace(-12, 12, 97):
        x = float(np.float32(x))
        s = float(F.silu(torch.tensor(x, dtype=torch.float64)))
        g = float(F.gelu(torch.tensor(x, dtype=torch.float64), approximate="tanh"))
        assert abs(oracle.silu(x) - s) <= 1e-6 * max(1.0, abs(s))
        assert abs(oracle.gelu_tanh(x) - g) <= 1e-6 * max(1.0, abs(g))


# --------------------------------------------------------- whole model
@pytest.mark.parametrize("gain_std", [0.0, 0.1])
@pytest.mark.parametrize("act,qk_norm", [(0, 1), (1, 0)])
def test_model_matches_float64_library_decoder(gain_std, act, qk_norm):
    cfg = inputs.shrink(inputs.TINY, act=act, qk_norm=qk_norm)
    hw = inputs.host_weights(cfg, seed=3, gain_std=gain_std)
    toks = inputs.prefix_tokens(3, 20, cfg.vocab)
    got = oracle.bruteforce(hw, toks).astype(np.float64)
    ref = torch_ref.logits(hw, toks)
    assert np.max(np.abs(got - ref)) <= 0.03
    top2 = np.sort(ref, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 0.05
    assert np.array_equal(got.argmax(1)[sure], ref.argmax(1)[sure])


def test_gqa_head_mapping_matters():
    """Query head h reads kv head h // group (library convention); a model whose
    two kv heads are swapped must give different logits."""
    cfg = inputs.TINY
    hw = inputs.host_weights(cfg, seed=5)
    toks = inputs.prefix_tokens(5, 8, cfg.vocab)
    base = oracle.bruteforce(hw, toks)
    d, Hq, Hkv = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    w = hw.tensors[("wqkv", 0)].copy()
    k0 = Hq * d
    w[[*range(k0, k0 + d)] + [*range(k0 + d, k0 + 2 * d)]] = \
        w[[*range(k0 + d, k0 + 2 * d)] + [*range(k0, k0 + d)]]
    hw.tensors[("wqkv", 0)] = w
    swapped = oracle.bruteforce(hw, toks)
    ref = torch_ref.logits(hw, toks)
    assert np.max(np.abs(swapped - ref)) <= 0.03
    assert np.max(np.abs(swapped - base)) > 0.03


# --------------------------------------------------------- invariants
@pytest.fixture(scope="module")
def tiny():
    cfg = inputs.TINY
    hw = inputs.host_weights(cfg, seed=0, gain_std=0.1)
    return cfg, hw


def test_cached_decode_equals_bruteforce(tiny):
    cfg, hw = tiny
    toks = inputs.prefix_tokens(0, 40, cfg.vocab)
    bf = oracle.bruteforce(hw, toks)
    m = oracle.OracleModel(hw, 64)
    rows = [m.prefill(toks[:1])[0]] + [m.decode(t)[0] for t in toks[1:]]
    assert np.array_equal(np.stack(rows), bf)


def test_prefill_equals_decode_chain(tiny):
    cfg, hw = tiny
    toks = inputs.prefix_tokens(1, 33, cfg.vocab)
    a = oracle.OracleModel(hw, 64)
    la, na = a.prefill(toks)
    b = oracle.OracleModel(hw, 64)
    for t in toks:
        lb, nb = b.decode(t)
    assert np.array_equal(la, lb) and na == nb == oracle.argmax(la)
    for p in range(len(toks)):
        assert all(np.array_equal(x, y) for x, y in zip(a.kv(1, p), b.kv(1, p)))


def _greedy_chain(hw, prompt, n):
    m = oracle.OracleModel(hw, len(prompt) + n + 8)
    _, t = m.prefill(prompt)
    chain = [t]
    for _ in range(n - 1):
        _, t = m.decode(t)
        chain.append(t)
    return chain


def test_verify_rows_equal_decode_and_accept_longest_prefix(tiny):
    cfg, hw = tiny
    prompt = inputs.prefix_tokens(2, 32, cfg.vocab)
    chain = _greedy_chain(hw, prompt, 24)
    K = 5
    for reject_at in (None, 0, 1, 3):
        toks, n_exp = inputs.window(chain, 0, K, vocab=cfg.vocab, reject_at=reject_at)
        m = oracle.OracleModel(hw, 64)
        m.prefill(prompt)
        lg, am, n, corr = m.verify(toks)
        # acceptance by brute force: largest n with toks[j+1] == argmax_j for j < n
        n_bf = max(j for j in range(K) if all(toks[i + 1] == am[i] for i in range(j)))
        assert n == n_bf == n_exp and corr == am[n] == chain[n + 1]
        assert len(m) == len(prompt) + 1 + n
        # every row equals a decode at the same prefix
        d = oracle.OracleModel(hw, 64)
        d.prefill(prompt)
        for r in range(K):
            lr, _ = d.decode(toks[r])
            assert np.array_equal(lr, lg[r])


def test_row0_ignores_later_rows(tiny):
    cfg, hw = tiny
    prompt = inputs.prefix_tokens(3, 30, cfg.vocab)
    outs = []
    for drafts in ([1, 2, 3], [900, 17, 5], [0, 0, 0]):
        m = oracle.OracleModel(hw, 64)
        _, t0 = m.prefill(prompt)
        lg, am, _, _ = m.verify([t0] + drafts)
        outs.append((lg[0], am[0]))
    assert all(np.array_equal(outs[0][0], o[0]) and outs[0][1] == o[1] for o in outs)


def test_k1_verify_equals_decode(tiny):
    cfg, hw = tiny
    prompt = inputs.prefix_tokens(4, 17, cfg.vocab)
    a, b = oracle.OracleModel(hw, 32), oracle.OracleModel(hw, 32)
    _, t = a.prefill(prompt)
    b.prefill(prompt)
    lg, am, n, c = a.verify([t])
    ld, nd = b.decode(t)
    assert n == 0 and c == nd and np.array_equal(lg[0], ld)


def test_layer_entry_chain_equals_verify(tiny):
    """The per-layer entry (one layer on given rows over a given cache) and the
    head entry, chained over every layer from the embedded rows with the
    model's own cache, reproduce the whole-model verify bit for bit: logits
    and the window's K/V."""
    cfg, hw = tiny
    prompt = inputs.prefix_tokens(4, 21, cfg.vocab)
    m = oracle.OracleModel(hw, 64)
    _, t = m.prefill(prompt)
    chain = [t]
    for _ in range(4):
        chain.append(m.decode(chain[-1])[1])
    m.truncate(len(prompt))
    window = chain[:4]  # the greedy chain: every draft accepted, so its K/V stay committed
    lo, _, n, _ = m.verify(window)
    assert n == 3
    lay = oracle.LayerOracle(hw)
    pos, row = len(prompt), cfg.n_kv_heads * cfg.head_dim
    x = np.stack([hw.get("embed")[tok] for tok in window])
    for l in range(cfg.n_layers):
        kc = np.stack([m.kv(l, p)[0] for p in range(pos)])
        vc = np.stack([m.kv(l, p)[1] for p in range(pos)])
        x, k, v = lay.layer(l, pos, x, kc, vc)
        for r in range(4):
            mk, mv = m.kv(l, pos + r)
            assert np.array_equal(k[r], mk) and np.array_equal(v[r], mv), (l, r)
        assert k.shape == (4, row)
    assert np.array_equal(lay.head(x), lo)


def test_truncate_then_continue_equals_fresh(tiny):
    cfg, hw = tiny
    prompt = inputs.prefix_tokens(5, 30, cfg.vocab)
    chain = _greedy_chain(hw, prompt, 16)
    m = oracle.OracleModel(hw, 80)
    m.prefill(prompt)
    committed = list(prompt)
    i, step = 0, 0
    while i + 4 <= len(chain):
        toks, n_exp = inputs.window(chain, i, 4, seq=5, step=step, p=0.5, vocab=cfg.vocab)
        lg, am, n, corr = m.verify(toks)
        assert n == n_exp
        committed += toks[: n + 1]
        i += n + 1
        step += 1
        # after truncation the state equals a fresh prefill of the committed ids
        fresh = oracle.OracleModel(hw, 80)
        lf, nf = fresh.prefill(committed)
        assert nf == corr == chain[i]
        assert len(fresh) == len(m)
        for p in range(len(committed)):
            assert all(np.array_equal(x, y) for x, y in zip(fresh.kv(0, p), m.kv(0, p)))
    bf = oracle.bruteforce(hw, committed + [chain[i]])
    ld, _ = m.decode(chain[i])
    assert np.array_equal(ld, bf[-1])


def test_generator_is_normal_like():
    hw = inputs.host_weights(inputs.TINY, seed=11)
    w = oracle.bits_to_f32(hw.tensors[("w_gate_up", 0)]).astype(np.float64).ravel()
    assert abs(w.mean()) < 0.02 * 0.01 * 10 and abs(w.std() - 0.02) < 0.02 * 0.01
    assert np.max(np.abs(w)) <= 6 * 0.02 * 1.001
