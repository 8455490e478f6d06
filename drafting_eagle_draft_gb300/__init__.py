"""Python binding of the P-EAGLE GB300 draft-pass library (libpeagle.so).

Argument marshalling only: every step of the pass runs in the library's CUDA kernels.
The functions keep the C ABI's names (include/peagle.h); tensors are passed as torch
tensors and handed to the library as raw pointers.  If libpeagle.so has not been built
this module raises on first use instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpeagle.so")

PEAGLE_OK = 0
PEAGLE_ERR_INVALID = -1
PEAGLE_ERR_UNSUPPORTED = -2
PEAGLE_ERR_CAPACITY = -3
PEAGLE_ERR_CUDA = -4
PEAGLE_ERR_DEVICE = -5
PEAGLE_DEV_BAD_TOKEN = 0x1
PEAGLE_DEV_KV_OVERFLOW = 0x2
PEAGLE_DEV_BAD_COMMIT = 0x4
PEAGLE_DEV_BAD_ROW = 0x8
PEAGLE_DEV_TIMEOUT = 0x10
PEAGLE_F32 = 0
PEAGLE_BF16 = 1

# every entry point declared in include/peagle.h
EXPORTS = ("peagle_create", "peagle_draft", "peagle_catch_up", "peagle_verify_greedy",
           "peagle_append_kv",
           "peagle_forward_parallel", "peagle_train_step", "peagle_cod_rows",
           "peagle_sequence_partition",
           "peagle_status",
           "peagle_set_timing", "peagle_read_timing", "peagle_read_pass_trace",
           "peagle_set_wait_limit", "peagle_set_pass_kernel",
           "peagle_decode_attention_static",
           "peagle_device_error_bits", "peagle_strerror", "peagle_destroy")
STAGES = ("fc", "qkv", "attn", "oproj", "gate_up", "down", "lm_head", "norm", "small")

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class PeagleDims(ctypes.Structure):
    _fields_ = [(n, _i32) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "intermediate",
        "draft_vocab", "target_vocab", "max_batch", "max_K", "max_rows", "max_seq",
        "max_positions", "dtype")] + [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                                      ("attn_window", _i32), ("lm_rank", _i32),
                                      ("lm_topk", _i32), ("train", _i32)]


class PeagleWeights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("emb_mask", _vp), ("h_shared", _vp), ("fc", _vp),
                ("input_norm", _vp), ("hidden_norm", _vp), ("qkv", ctypes.POINTER(_vp)),
                ("o", ctypes.POINTER(_vp)), ("attn_norm", ctypes.POINTER(_vp)),
                ("post_norm", ctypes.POINTER(_vp)), ("gate", ctypes.POINTER(_vp)),
                ("up", ctypes.POINTER(_vp)), ("down", ctypes.POINTER(_vp)),
                ("final_norm", _vp), ("lm_head", _vp), ("d2t", _vp), ("lm_proj", _vp),
                ("lm_score", _vp)]


class PeagleGrads(ctypes.Structure):
    _fields_ = [("embed", _vp), ("emb_mask", _vp), ("h_shared", _vp), ("fc", _vp),
                ("input_norm", _vp), ("hidden_norm", _vp), ("qkv", ctypes.POINTER(_vp)),
                ("o", ctypes.POINTER(_vp)), ("attn_norm", ctypes.POINTER(_vp)),
                ("post_norm", ctypes.POINTER(_vp)), ("gate", ctypes.POINTER(_vp)),
                ("up", ctypes.POINTER(_vp)), ("down", ctypes.POINTER(_vp)),
                ("final_norm", _vp), ("lm_head", _vp)]


class PeagleKV(ctypes.Structure):
    _fields_ = [("k", _vp), ("v", _vp), ("capacity", _i32), ("batch", _i32)]


_LIB = None


class PeagleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


def lib():
    """The loaded libpeagle.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with drafting_eagle_draft_gb300.build.build() "
                "(nvcc, sm_103a); there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        L.peagle_create.argtypes = [ctypes.POINTER(PeagleWeights), ctypes.POINTER(PeagleDims),
                                    ctypes.POINTER(_vp)]
        L.peagle_draft.argtypes = [_vp, _i32, ctypes.POINTER(PeagleKV), _vp, _vp, _vp, _i32,
                                   _vp, _vp, _vp]
        L.peagle_catch_up.argtypes = [_vp, _i32, ctypes.POINTER(PeagleKV), _vp, _vp, _vp, _i32,
                                      _vp, _vp, _vp]
        L.peagle_verify_greedy.argtypes = [_i32, _i32, _vp, _vp, _vp, _vp, _vp]
        L.peagle_append_kv.argtypes = [_vp, _i32, ctypes.POINTER(PeagleKV), _vp, _vp, _i32,
                                       _vp, _vp, _i32, _vp]
        L.peagle_forward_parallel.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp,
                                              _vp, _vp]
        L.peagle_train_step.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                        ctypes.POINTER(PeagleGrads), _vp]
        L.peagle_cod_rows.argtypes = [_i32, _i32, ctypes.c_double, _vp, _vp, _vp, _i32]
        L.peagle_sequence_partition.argtypes = [_i32, _vp, _vp, _i32, _vp, _vp]
        L.peagle_status.argtypes = [_vp]
        L.peagle_set_timing.argtypes = [_vp, _i32]
        L.peagle_set_wait_limit.argtypes = [_vp, ctypes.c_uint64, _i32]
        L.peagle_set_pass_kernel.argtypes = [_vp, _i32]
        L.peagle_decode_attention_static.argtypes = [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                                     _i32, _vp, _vp, _vp]
        L.peagle_read_timing.argtypes = [_vp, _vp, _vp]
        L.peagle_read_pass_trace.argtypes = [_vp, _vp, _i32, _vp, _vp]
        L.peagle_read_pass_trace.restype = _i32
        L.peagle_device_error_bits.argtypes = [_vp]
        L.peagle_device_error_bits.restype = _i32
        L.peagle_strerror.argtypes = [ctypes.c_int]
        L.peagle_strerror.restype = ctypes.c_char_p
        L.peagle_destroy.argtypes = [_vp]
        L.peagle_destroy.restype = None
        _LIB = L
    return _LIB


def strerror(code: int) -> str:
    return lib().peagle_strerror(int(code)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _check(code, what):
    if code != PEAGLE_OK:
        raise PeagleError(code, what)


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def make_dims(dims, max_batch, max_K, max_positions, max_rows=0, max_seq=0,
              train=False) -> PeagleDims:
    """C struct from a ``synth.Dims``-like object plus the context's capacity limits
    (``train``: the context also holds the training step's workspaces)."""
    return PeagleDims(hidden=dims.hidden, n_layers=dims.n_layers, n_q_heads=dims.n_q_heads,
                      n_kv_heads=dims.n_kv_heads, head_dim=dims.head_dim,
                      intermediate=dims.intermediate, draft_vocab=dims.draft_vocab,
                      target_vocab=dims.target_vocab, max_batch=max_batch, max_K=max_K,
                      max_rows=max_rows, max_seq=max_seq, max_positions=max_positions,
                      dtype=PEAGLE_F32 if dims.dtype == "f32" else PEAGLE_BF16,
                      rope_theta=dims.rope_theta, rms_eps=dims.rms_eps,
                      attn_window=int(getattr(dims, "attn_window", 0) or 0),
                      lm_rank=int(getattr(dims, "lm_rank", 0) or 0),
                      lm_topk=int(getattr(dims, "lm_topk", 0) or 0), train=int(bool(train)))


class Context:
    """Owns a peagle_ctx (weights + workspaces on the current CUDA device)."""

    def __init__(self, handle, cdims, keep):
        self.handle = handle
        self.cdims = cdims
        self._keep = keep

    def close(self):
        if self.handle:
            lib().peagle_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


def peagle_create(weights: dict, cdims: PeagleDims) -> Context:
    """weights: dict as produced by ``synth.make_weights`` (CPU or CUDA tensors; d2t as a
    numpy int32 array or tensor).  Copies everything into library-owned device memory."""
    import torch

    keep = []

    def p(t):
        if isinstance(t, np.ndarray):
            t = torch.from_numpy(np.ascontiguousarray(t))
        t = t.contiguous()
        keep.append(t)
        return t.data_ptr()

    N = len(weights["layers"])

    def arr(key, allow_none_first=False):
        a = (_vp * N)()
        for i, L in enumerate(weights["layers"]):
            a[i] = None if (allow_none_first and i == 0) else p(L[key])
        keep.append(a)
        return ctypes.cast(a, ctypes.POINTER(_vp))

    w = PeagleWeights(
        embed=p(weights["embed"]), emb_mask=p(weights["emb_mask"]),
        h_shared=p(weights["h_shared"]), fc=p(weights["fc"]),
        input_norm=p(weights["input_norm"]), hidden_norm=p(weights["hidden_norm"]),
        qkv=arr("qkv"), o=arr("o"), attn_norm=arr("attn_norm", True),
        post_norm=arr("post_norm"), gate=arr("gate"), up=arr("up"), down=arr("down"),
        final_norm=p(weights["final_norm"]), lm_head=p(weights["lm_head"]),
        d2t=p(np.asarray(weights["d2t"], np.int32)),
        lm_proj=p(weights["lm_proj"]) if weights.get("lm_proj") is not None else None,
        lm_score=p(weights["lm_score"]) if weights.get("lm_score") is not None else None)
    h = _vp()
    _check(lib().peagle_create(ctypes.byref(w), ctypes.byref(cdims), ctypes.byref(h)),
           "peagle_create")
    return Context(h.value, cdims, None)


def kv_struct(cache_k, cache_v, capacity, batch) -> PeagleKV:
    return PeagleKV(k=_ptr(cache_k), v=_ptr(cache_v), capacity=int(capacity), batch=int(batch))


def peagle_draft(ctx: Context, batch, kv: PeagleKV, seq_lens, target_hidden, new_token, K,
                 out_draft_tokens, out_logits=None, stream=None):
    _check(lib().peagle_draft(ctx.handle, int(batch), ctypes.byref(kv), _ptr(seq_lens),
                              _ptr(target_hidden), _ptr(new_token), int(K),
                              _ptr(out_draft_tokens), _ptr(out_logits), _stream_ptr(stream)),
           "peagle_draft")


def peagle_catch_up(ctx: Context, batch, kv: PeagleKV, seq_lens, hidden, tokens, T,
                    out_tokens=None, out_logits=None, stream=None):
    """Run the accepted tokens through the drafter and write their K/V (include/peagle.h)."""
    _check(lib().peagle_catch_up(ctx.handle, int(batch), ctypes.byref(kv), _ptr(seq_lens),
                                 _ptr(hidden), _ptr(tokens), int(T), _ptr(out_tokens),
                                 _ptr(out_logits), _stream_ptr(stream)),
           "peagle_catch_up")


def peagle_verify_greedy(batch, K, draft_tokens, target_argmax, out_accept_len, out_bonus,
                         stream=None):
    _check(lib().peagle_verify_greedy(int(batch), int(K), _ptr(draft_tokens),
                                      _ptr(target_argmax), _ptr(out_accept_len),
                                      _ptr(out_bonus), _stream_ptr(stream)),
           "peagle_verify_greedy")


def peagle_append_kv(ctx: Context, batch, kv: PeagleKV, seq_lens, n_commit, k_rows=None,
                     v_rows=None, n_max=0, stream=None, n_extra=0):
    _check(lib().peagle_append_kv(ctx.handle, int(batch), ctypes.byref(kv), _ptr(seq_lens),
                                  _ptr(n_commit), int(n_extra), _ptr(k_rows), _ptr(v_rows),
                                  int(n_max), _stream_ptr(stream)),
           "peagle_append_kv")


def peagle_forward_parallel(ctx: Context, n, K, tokens, hidden, row_p, row_d, M, out_argmax,
                            out_logits=None, stream=None):
    _check(lib().peagle_forward_parallel(ctx.handle, int(n), int(K), _ptr(tokens),
                                         _ptr(hidden), _ptr(row_p), _ptr(row_d), int(M),
                                         _ptr(out_argmax), _ptr(out_logits),
                                         _stream_ptr(stream)),
           "peagle_forward_parallel")


def grads_struct(g, n_layers):
    """PeagleGrads over a dict of fp32 device tensors named like the weights (embed and
    attn_norm optional); the per-layer pointer arrays are kept on the struct."""
    def arr(name):
        if name not in g or g[name] is None:
            return None
        a = (_vp * n_layers)(*[_ptr(t) for t in g[name]])
        return a
    st = PeagleGrads()
    for k in ("embed", "emb_mask", "h_shared", "fc", "input_norm", "hidden_norm",
              "final_norm", "lm_head"):
        setattr(st, k, _ptr(g.get(k)))
    st._keep = []
    for k in ("qkv", "o", "attn_norm", "post_norm", "gate", "up", "down"):
        a = arr(k)
        st._keep.append(a)
        setattr(st, k, ctypes.cast(a, ctypes.POINTER(_vp)) if a is not None else None)
    return st


def peagle_train_step(ctx: Context, n, K, tokens, hidden, row_p, row_d, M, labels, out_loss,
                      grads, stream=None):
    """One training step (loss + every parameter gradient); grads: PeagleGrads or a dict
    for grads_struct."""
    st = grads if isinstance(grads, PeagleGrads) else grads_struct(grads, ctx.cdims.n_layers)
    _check(lib().peagle_train_step(ctx.handle, int(n), int(K), _ptr(tokens), _ptr(hidden),
                                   _ptr(row_p), _ptr(row_d), int(M), _ptr(labels),
                                   _ptr(out_loss), ctypes.byref(st), _stream_ptr(stream)),
           "peagle_train_step")


def peagle_cod_rows(n, K, ratio, uniforms):
    """Host-side COD sampling; uniforms float64 [n, K].  Returns (row_p, row_d) int32."""
    u = np.ascontiguousarray(uniforms, np.float64)
    assert u.shape == (n, K)
    cap = n * K
    rp = np.empty(cap, np.int32)
    rd = np.empty(cap, np.int32)
    m = lib().peagle_cod_rows(int(n), int(K), ctypes.c_double(ratio), u.ctypes.data,
                              rp.ctypes.data, rd.ctypes.data, cap)
    if m < 0:
        raise PeagleError(m, "peagle_cod_rows")
    return rp[:m].copy(), rd[:m].copy()


def peagle_sequence_partition(row_p, row_d, boundaries):
    """Chunk index of every retained row (host arrays; see include/peagle.h)."""
    rp = np.ascontiguousarray(row_p, np.int32)
    rd = np.ascontiguousarray(row_d, np.int32)
    bd = np.ascontiguousarray(boundaries, np.int32)
    out = np.empty(len(rp), np.int32)
    _check(lib().peagle_sequence_partition(len(rp), rp.ctypes.data, rd.ctypes.data, len(bd),
                                           bd.ctypes.data, out.ctypes.data),
           "peagle_sequence_partition")
    return out


def peagle_status(ctx: Context) -> int:
    """Synchronises; returns PEAGLE_OK or PEAGLE_ERR_DEVICE (device error bits cleared)."""
    return lib().peagle_status(ctx.handle)


def peagle_set_pass_kernel(ctx: Context, mode: int):
    """-1: the persistent pass kernel up to 16 draft rows (default); 0: never; 1: always."""
    _check(lib().peagle_set_pass_kernel(ctx.handle, int(mode)), "peagle_set_pass_kernel")


def peagle_set_wait_limit(ctx: Context, limit_ns: int, unreachable_step: int = -1):
    """Bounded-wait drill (see include/peagle.h): wait limit in ns (0 = default 2 s) and a
    step of the pass whose waits cannot end (-1 none)."""
    _check(lib().peagle_set_wait_limit(ctx.handle, int(limit_ns), int(unreachable_step)),
           "peagle_set_wait_limit")


def peagle_set_timing(ctx: Context, enable: bool):
    _check(lib().peagle_set_timing(ctx.handle, 1 if enable else 0), "peagle_set_timing")


def peagle_read_timing(ctx: Context) -> dict:
    """{stage: (milliseconds, launches)} since the previous read (synchronises)."""
    ms = np.zeros(len(STAGES), np.float32)
    n = np.zeros(len(STAGES), np.int32)
    _check(lib().peagle_read_timing(ctx.handle, ms.ctypes.data, n.ctypes.data),
           "peagle_read_timing")
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(STAGES)}


def peagle_read_pass_trace(ctx: Context):
    """Per-CTA event times (ns) of every step of the latest pass-kernel call run with
    timing enabled, as an int64 array [phases, ctas, 4] (activations ready, first MMA, last
    accumulator, done; 0 where not applicable); None when none was traced."""
    cap = 512 * 1024
    buf = np.zeros(cap, np.uint64)
    ph = ctypes.c_int32(0)
    ct = ctypes.c_int32(0)
    n = lib().peagle_read_pass_trace(ctx.handle, buf.ctypes.data, cap, ctypes.byref(ph),
                                     ctypes.byref(ct))
    if n < 0:
        _check(n, "peagle_read_pass_trace")
    if n == 0:
        return None
    return buf[:n].astype(np.int64).reshape(ph.value, ct.value, 4)


def peagle_decode_attention_static(batch, K, n_q_heads, n_kv_heads, head_dim, q, k_cache,
                                   v_cache, capacity, seq_lens, out, stream=None):
    """Decode attention with no device allocation (see include/peagle.h)."""
    _check(lib().peagle_decode_attention_static(int(batch), int(K), int(n_q_heads),
                                                int(n_kv_heads), int(head_dim), _ptr(q),
                                                _ptr(k_cache), _ptr(v_cache), int(capacity),
                                                _ptr(seq_lens), _ptr(out), _stream_ptr(stream)),
           "peagle_decode_attention_static")


def peagle_device_error_bits(ctx: Context) -> int:
    return lib().peagle_device_error_bits(ctx.handle)
