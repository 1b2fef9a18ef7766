"""Python binding of libsv.so: argument marshalling over the C-ABI only.

Every step of decode / verify runs in the library's CUDA kernels; this module
passes pointers and sizes. PyTorch provides device memory and streams. If
the compiled library is missing the import fails: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsv.so")

SV_OK, SV_E_INVAL, SV_E_NOMEM, SV_E_CUDA, SV_E_STATE = 0, -1, -2, -3, -4
SV_LIN_O, SV_LIN_GATE_UP, SV_LIN_DOWN, SV_LIN_LM_HEAD = 1, 2, 3, 4
PAGE_SIZE = 16
MAX_K = 32
MAX_PREFILL_ROWS = 128
_ERRNAMES = {SV_E_INVAL: "SV_E_INVAL", SV_E_NOMEM: "SV_E_NOMEM", SV_E_CUDA: "SV_E_CUDA",
             SV_E_STATE: "SV_E_STATE"}

_P = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)
_i32 = ctypes.c_int32


class SvConfig(ctypes.Structure):
    _fields_ = [(n, _i32) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim",
                                   "ffn", "vocab")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + [
        (n, _i32) for n in ("qk_norm", "act", "tie_embeddings", "page_size", "max_pages", "max_k",
                            "max_seq", "kv_delayed")]


LAYER_KEYS = ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate_up", "w_down")


class SvWeights(ctypes.Structure):
    _fields_ = [("embed", _P), ("lm_head", _P), ("final_norm", _P)] + [(k, _PP) for k in LAYER_KEYS]


class SvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRNAMES.get(code, code)}: {msg}")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    L.sv_create.argtypes = [ctypes.POINTER(SvConfig), ctypes.POINTER(SvWeights), _P, ctypes.POINTER(_P)]
    L.sv_destroy.argtypes = [_P]
    L.sv_destroy.restype = None
    L.sv_prefill.argtypes = [_P, _P, _i32, _P, _P]
    L.sv_decode.argtypes = [_P, _i32, _P, _P]
    L.sv_verify.argtypes = [_P, _P, _i32, _P, _P, _P]
    L.sv_verify_async.argtypes = [_P, _P, _i32, _P, _P]
    L.sv_reserve.argtypes = [_P, _i32]
    L.sv_sync.argtypes = [_P]
    L.sv_truncate.argtypes = [_P, _i32]
    L.sv_seq_len.argtypes = [_P]
    L.sv_kv_read.argtypes = [_P, _i32, _i32, _i32, _P, _P]
    L.sv_shuffle_pages.argtypes = [_P, ctypes.c_uint64]
    L.sv_trace_hidden.argtypes = [_P, _P, _i32]
    L.sv_step_kernel_count.argtypes = [_P, _i32, _i32]
    L.sv_prefill_blocks.argtypes = [_i32, _i32, _P, _i32]
    L.sv_spec_generate.argtypes = [_P, _P, _i32, _i32, _i32, _P, _P, _P, _P]
    L.sv_time_linear.argtypes = [_P, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_float),
                                 ctypes.POINTER(ctypes.c_double)]
    L.sv_lm_head_noalloc.argtypes = [_P, _P, _P, _i32, _i32, _i32, ctypes.c_float, _P, _P, _P, _P]
    L.sv_last_error.argtypes = [_P]
    L.sv_last_error.restype = ctypes.c_char_p
    for name in ("sv_create", "sv_prefill", "sv_decode", "sv_verify", "sv_verify_async",
                 "sv_reserve", "sv_sync", "sv_truncate", "sv_seq_len", "sv_kv_read",
                 "sv_shuffle_pages", "sv_trace_hidden", "sv_step_kernel_count", "sv_time_linear",
                 "sv_lm_head_noalloc", "sv_prefill_blocks"):
        getattr(L, name).restype = _i32
    return L


_lib = _load()


def lib():
    return _lib


def _i32_array(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int32 * len(vals))(*vals)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _check_tensor(t, name, dtype, shape):
    """The C call takes raw pointers and cannot check what they point to: a
    wrong dtype, shape, device or layout here would become out-of-bounds
    device accesses there."""
    if t is None:
        return
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name}: must be a CUDA tensor")
    if str(t.dtype) != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _check_buf(t, name, dtype, min_numel, cuda=False):
    """A buffer that a step's kernels read or write whole (tokens, result,
    logits): the C call sees only its address, so a buffer of another type,
    not contiguous or too small would become out-of-bounds accesses there.
    cuda: must also be device memory (the library checks the asynchronous
    call's token and result buffers itself)."""
    if t is None:
        return
    if cuda and not getattr(t, "is_cuda", False):
        raise ValueError(f"{name}: must be a CUDA tensor")
    if str(t.dtype) != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{name}: {t.numel()} elements, at least {min_numel} needed")


def lm_head_noalloc(x, gain, w, logits, argmax=None, status=None, eps=1e-6, stream=None):
    """sv_lm_head_noalloc: logits and greedy tokens of M rows without any
    device allocation by the library (scratch is a fixed array inside it).
    x: bf16 [M, hidden]; gain: bf16 [hidden]; w: bf16 [vocab, hidden];
    logits: fp32 [M, vocab]; argmax: int32 [M] or None; status: int32 [1] or
    None. All CUDA tensors owned by the caller, contiguous. Asynchronous on
    `stream`. Raises ValueError before any device work if a tensor does not
    match these shapes and types."""
    if getattr(x, "dim", lambda: 0)() != 2 or getattr(w, "dim", lambda: 0)() != 2:
        raise ValueError("x and w must be 2-D tensors")
    M, hidden = int(x.shape[0]), int(x.shape[1])
    vocab = int(w.shape[0])
    _check_tensor(x, "x", "torch.bfloat16", (M, hidden))
    _check_tensor(gain, "gain", "torch.bfloat16", (hidden,))
    _check_tensor(w, "w", "torch.bfloat16", (vocab, hidden))
    _check_tensor(logits, "logits", "torch.float32", (M, vocab))
    _check_tensor(argmax, "argmax", "torch.int32", (M,))
    _check_tensor(status, "status", "torch.int32", (1,))
    s = _P(stream.cuda_stream) if stream is not None else _P(0)
    rc = _lib.sv_lm_head_noalloc(_P(_ptr(x)), _P(_ptr(gain)), _P(_ptr(w)), M, hidden, vocab,
                                 float(eps), _P(_ptr(logits)), _P(_ptr(argmax)), _P(_ptr(status)), s)
    if rc != SV_OK:
        raise SvError(rc, "sv_lm_head_noalloc rejected the shapes (scratch limit 8 MiB, "
                          "1 <= M <= 32, hidden % 128 == 0) or a CUDA call failed")


def spec_generate(target: "Context", draft: "Context", pending: int, K: int, n_new: int):
    """sv_spec_generate: greedy speculative generation of at least n_new tokens
    from `pending`, drafted by `draft` and verified by `target` (both holding
    the same tokens).  Returns (tokens committed, next pending token,
    {"verify_steps", "accepted", "proposed"})."""
    out = (ctypes.c_int32 * (n_new + max(K, 1) - 1))()
    n_out, nxt = ctypes.c_int32(0), ctypes.c_int32(0)
    stats = (ctypes.c_int32 * 3)()
    target._check(_lib.sv_spec_generate(target._h, draft._h, int(pending), int(K), int(n_new), out,
                                        ctypes.byref(n_out), ctypes.byref(nxt), stats))
    return (list(out[:n_out.value]), nxt.value,
            {"verify_steps": stats[0], "accepted": stats[1], "proposed": stats[2]})


def prefill_blocks(n: int, use_tc: bool = True) -> list:
    """sv_prefill_blocks: the row blocks sv_prefill cuts n prompt tokens into
    (use_tc: the context runs the tcgen05 linears, the default)."""
    cnt = _lib.sv_prefill_blocks(int(n), 1 if use_tc else 0, None, 0)
    if cnt < 0:
        raise SvError(cnt, f"no prefill of {n} tokens")
    arr = (ctypes.c_int32 * cnt)()
    if _lib.sv_prefill_blocks(int(n), 1 if use_tc else 0, ctypes.cast(arr, _P), cnt) != cnt:
        raise SvError(SV_E_INVAL, "prefill schedule changed size")
    return list(arr)


class Context:
    """One sequence on the GPU.

    cfg: any object with the model-shape fields of sv_config (n_layers,
    hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, rms_eps, rope_theta,
    qk_norm, act, tie_embeddings). weights: mapping (name, layer) -> CUDA
    tensor of bf16 values (layer -1 for embed / lm_head / final_norm), the
    layout of include/sv.h; the tensors must outlive the context.
    kv_delayed: commit a verify window's K/V only after acceptance (sv_config
    kv_delayed = 1) instead of writing it and zeroing the rejected rows.
    """

    def __init__(self, cfg, weights, *, max_k: int, max_seq: int, max_pages: int | None = None,
                 stream=None, kv_delayed: bool = False):
        self.cfg = cfg
        self.max_k, self.max_seq = max_k, max_seq
        pages = max_pages if max_pages is not None else (max_seq + PAGE_SIZE - 1) // PAGE_SIZE
        self._c = SvConfig(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                           cfg.ffn, cfg.vocab, cfg.rms_eps, cfg.rope_theta, cfg.qk_norm, cfg.act,
                           cfg.tie_embeddings, PAGE_SIZE, pages, max_k, max_seq, int(bool(kv_delayed)))
        self._weights = weights  # keep the tensors alive
        w = SvWeights()
        w.embed = _ptr(weights[("embed", -1)])
        lm = weights.get(("lm_head", -1))
        w.lm_head = _ptr(lm) if lm is not None else w.embed
        w.final_norm = _ptr(weights[("final_norm", -1)])
        self._arrays = []
        L = max(cfg.n_layers, 1)
        for k in LAYER_KEYS:
            ptrs = (ctypes.c_void_p * L)(*[_ptr(weights.get((k, l))) for l in range(cfg.n_layers)])
            self._arrays.append(ptrs)
            setattr(w, k, ctypes.cast(ptrs, _PP))
        self._w = w
        self._stream = stream
        h = _P()
        s = _P(stream.cuda_stream) if stream is not None else _P(0)
        rc = _lib.sv_create(ctypes.byref(self._c), ctypes.byref(w), s, ctypes.byref(h))
        if rc != SV_OK:
            raise SvError(rc, "sv_create rejected the configuration or failed to allocate")
        self._h = h

    # ----------------------------------------------------------- plumbing
    def close(self):
        if getattr(self, "_h", None):
            _lib.sv_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def _check(self, rc):
        if rc != SV_OK:
            raise SvError(rc, _lib.sv_last_error(self._h).decode(errors="replace"))

    # ----------------------------------------------------------- the calls
    def prefill(self, tokens, logits=None) -> int:
        _check_buf(logits, "logits", "torch.float32", self.cfg.vocab, cuda=True)
        arr = _i32_array(tokens)
        nxt = ctypes.c_int32(0)
        self._check(_lib.sv_prefill(self._h, arr, len(arr), _P(_ptr(logits)), ctypes.byref(nxt)))
        return nxt.value

    def decode(self, token: int, logits=None) -> int:
        _check_buf(logits, "logits", "torch.float32", self.cfg.vocab, cuda=True)
        nxt = ctypes.c_int32(0)
        self._check(_lib.sv_decode(self._h, int(token), _P(_ptr(logits)), ctypes.byref(nxt)))
        return nxt.value

    def verify(self, tokens, logits=None):
        arr = _i32_array(tokens)
        _check_buf(logits, "logits", "torch.float32", len(arr) * self.cfg.vocab, cuda=True)
        n = ctypes.c_int32(0)
        c = ctypes.c_int32(0)
        self._check(_lib.sv_verify(self._h, arr, len(arr), _P(_ptr(logits)), ctypes.byref(n),
                                   ctypes.byref(c)))
        return n.value, c.value

    def verify_async(self, tokens_dev, K: int, result_dev, logits=None):
        _check_buf(tokens_dev, "tokens_dev", "torch.int32", int(K))
        _check_buf(result_dev, "result_dev", "torch.int32", 4)
        _check_buf(logits, "logits", "torch.float32", int(K) * self.cfg.vocab, cuda=True)
        self._check(_lib.sv_verify_async(self._h, _P(_ptr(tokens_dev)), int(K), _P(_ptr(logits)),
                                         _P(_ptr(result_dev))))

    def reserve(self, length: int):
        self._check(_lib.sv_reserve(self._h, int(length)))

    def sync(self):
        self._check(_lib.sv_sync(self._h))

    def truncate(self, new_len: int):
        self._check(_lib.sv_truncate(self._h, int(new_len)))

    def __len__(self) -> int:
        return int(_lib.sv_seq_len(self._h))

    def kv_read(self, layer: int, first: int, count: int):
        import torch
        c = self.cfg
        k = torch.empty((count, c.n_kv_heads, c.head_dim), dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        self._check(_lib.sv_kv_read(self._h, layer, first, count, _P(k.data_ptr()),
                                    _P(v.data_ptr())))
        return k, v

    def shuffle_pages(self, seed: int):
        self._check(_lib.sv_shuffle_pages(self._h, ctypes.c_uint64(seed)))

    def trace_hidden(self, buf, max_rows: int = 0):
        """Test hook: while ``buf`` (bf16 CUDA [n_layers + 1, rows, hidden]
        for steps of up to ``max_rows`` rows) is set, every step copies its
        residual stream after each layer into it; None turns it off."""
        if buf is not None:
            _check_tensor(buf, "trace", "torch.bfloat16", (self.cfg.n_layers + 1, max_rows, self.cfg.hidden))
        self._check(_lib.sv_trace_hidden(self._h, _P(_ptr(buf)), int(max_rows)))
        self._trace = buf  # keep it alive while the library may write it

    def time_linear(self, which: int, K: int, reps: int = 3):
        """(mean device us per launch, algorithmic bytes per launch) of one
        linear class, timed on the library's stream."""
        us = ctypes.c_float(0.0)
        b = ctypes.c_double(0.0)
        self._check(_lib.sv_time_linear(self._h, int(which), int(K), int(reps), ctypes.byref(us),
                                        ctypes.byref(b)))
        return float(us.value), float(b.value)

    def kernels_per_step(self, K: int, with_head: bool = True) -> int:
        return int(_lib.sv_step_kernel_count(self._h, int(K), 1 if with_head else 0))
