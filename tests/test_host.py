"""Host-side logic that needs no GPU: the C-ABI library's exported symbols,
the benchmark's counter definitions (pinned to the page's printed counters)
and the replica aggregation across ranks (gloo, world size 2)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _header_functions():
    src = open(os.path.join(ROOT, "include", "sv.h")).read()
    return sorted(set(re.findall(r"^(?:int|void|const char\*)\s+(sv_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol():
    lib_path = os.path.join(ROOT, "greedy_speculative_decode_gb300", "libsv.so")
    if not os.path.exists(lib_path):
        import __graft_entry__
        __graft_entry__.build()
    import ctypes
    lib = ctypes.CDLL(lib_path)
    names = _header_functions()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_loads_and_names_the_same_calls():
    import greedy_speculative_decode_gb300 as sv
    for n in _header_functions():
        assert hasattr(sv.lib(), n)


def test_no_alloc_binding_rejects_host_tensors():
    """The allocation-free call takes device pointers: the binding refuses host
    tensors before calling into the library."""
    import torch
    import greedy_speculative_decode_gb300 as sv
    x = torch.zeros((2, 128), dtype=torch.bfloat16)
    g = torch.ones((128,), dtype=torch.bfloat16)
    w = torch.zeros((256, 128), dtype=torch.bfloat16)
    lg = torch.empty((2, 256), dtype=torch.float32)
    with pytest.raises(ValueError):
        sv.lm_head_noalloc(x, g, w, lg)


def _counters():
    out = {}
    for line in open(os.path.join(GOLDEN, "p2_bench_counters.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = [x.strip() for x in line.split("=")]
            out[k] = float(v)
    return out


def test_counter_definitions_reproduce_the_page():
    import bench
    c = _counters()
    assert c["target_steps"] == c["verify_steps"] + c["commit_decode_steps"] + c["correction_steps"]
    got = bench.counters(c["accepted"], c["proposed"], c["decode_tokens"], c["target_steps"], 1.0)
    assert round(got["acceptance_rate"], 4) == c["acceptance_rate"]
    assert round(got["tokens_per_target_step"], 4) == c["tokens_per_target_step"]
    # tok/s = 1000 / TPOT(ms), and the speedups are ratios of tok/s
    for kind in ("e2e", "decode"):
        base_tps = 1000.0 / c[f"baseline_{kind}_tpot_ms"]
        spec_tps = 1000.0 / c[f"spec_{kind}_tpot_ms"]
        assert abs(base_tps - c[f"baseline_{kind}_tok_s"]) < 5e-3
        assert abs(spec_tps - c[f"spec_{kind}_tok_s"]) < 5e-3
        assert round(spec_tps / base_tps, 4) == c[f"speedup_{kind}"]
    # windows were sometimes shorter than gamma: proposals < 4 per verify step
    assert c["proposed"] < 4 * c["verify_steps"]
    t = bench.counters(10, 30, 25, 10, 0.5)
    assert t["tok_s"] == 50.0 and t["tpot_ms"] == 20.0


def _agg_worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, toks = bench.aggregate(10.0 + 5.0 * rank, 100 + rank, dist)
    q.put((rank, ms, toks))
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_agg_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert all(ms == 15.0 and toks == 201 for _, ms, toks in res)


def test_schedule_follows_acceptance_rule():
    import inputs
    chain = list(range(100, 200))
    sched = inputs.schedule(chain, 4, 30, seq=0, p=0.6, vocab=1000)
    i = 0
    for (ci, toks, n) in sched:
        assert ci == i and toks[0] == chain[i]
        good = [toks[j] == chain[i + j] for j in range(1, 4)]
        assert n == (good.index(False) if False in good else 3)
        i += n + 1
    # forced patterns: all accept / first draft rejected / middle draft rejected
    assert inputs.window(chain, 0, 8, vocab=1000)[1] == 7
    assert inputs.window(chain, 0, 8, vocab=1000, reject_at=0)[1] == 0
    assert inputs.window(chain, 0, 8, vocab=1000, reject_at=4)[1] == 4


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 64, 65, 87, 100, 128, 129, 160, 161, 300, 1024, 4096, 4097])
def test_prefill_block_schedule(n):
    """sv_prefill_blocks (host only): the blocks cover the prompt in order;
    the last holds the 1..32 rows left over; the others hold 32 rows, or up
    to 128 rows (a multiple of 32) with the tcgen05 linears, as large as
    allowed, so a 1024-token prompt streams the weights 9 times, not 32."""
    import greedy_speculative_decode_gb300 as sv
    for use_tc in (False, True):
        sizes = sv.prefill_blocks(n, use_tc=use_tc)
        assert sum(sizes) == n and all(s >= 1 for s in sizes)
        assert sizes[-1] == (n - 1) % sv.MAX_K + 1
        cap = sv.MAX_PREFILL_ROWS if use_tc else sv.MAX_K
        for s in sizes[:-1]:
            assert s % sv.MAX_K == 0 and s <= cap
        # greedy: every block but the last two is full
        assert all(s == cap for s in sizes[:-2])
    assert len(sv.prefill_blocks(1024, use_tc=True)) == 9
    assert len(sv.prefill_blocks(1024, use_tc=False)) == 32


def test_prefill_block_schedule_rejects_bad_calls():
    import ctypes

    import greedy_speculative_decode_gb300 as sv
    L = sv.lib()
    assert L.sv_prefill_blocks(0, 1, None, 0) == sv.SV_E_INVAL
    arr = (ctypes.c_int32 * 2)()
    assert L.sv_prefill_blocks(300, 1, ctypes.cast(arr, ctypes.c_void_p), 2) == sv.SV_E_INVAL


@pytest.mark.parametrize("bad", [-1, 2])
def test_create_rejects_bad_kv_delayed(bad):
    """sv_config.kv_delayed is 0 or 1; anything else is SV_E_INVAL, decided
    before any device work."""
    import ctypes

    import greedy_speculative_decode_gb300 as sv
    c = sv.SvConfig(2, 256, 4, 2, 64, 704, 1024, 1e-6, 1e4, 1, 0, 1, 16, 8, 8, 128, bad)
    w = sv.SvWeights()
    h = ctypes.c_void_p(0)
    assert sv.lib().sv_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == sv.SV_E_INVAL
    assert not h.value


def test_step_buffers_are_checked_before_the_call():
    """The binding refuses a step buffer of the wrong type, layout or size
    (the C call sees only its address); logits must also be device memory.
    No GPU is needed: the checks run before any library call."""
    import torch
    import greedy_speculative_decode_gb300 as sv
    chk = sv._check_buf
    chk(None, "logits", "torch.float32", 10, cuda=True)                 # no buffer: nothing to check
    chk(torch.zeros(4, dtype=torch.int32), "tokens_dev", "torch.int32", 4)  # right type and size
    bad = [
        (torch.zeros(4, dtype=torch.int64), "torch.int32", 4, False),      # type
        (torch.zeros(8, dtype=torch.int32)[::2], "torch.int32", 4, False),  # layout
        (torch.zeros(3, dtype=torch.int32), "torch.int32", 4, False),      # size
        (torch.zeros((4, 10), dtype=torch.float32), "torch.float32", 40, True),  # host logits
    ]
    for t, dtype, n, cuda in bad:
        with pytest.raises(ValueError):
            chk(t, "buf", dtype, n, cuda=cuda)
