"""Seeded synthetic inputs for the P-EAGLE draft pass and its training-style forward.

This module only draws numbers: weights, KV caches, hidden states, token ids and the
uniform variates that COD sampling consumes.  It performs none of the method's
arithmetic, so both the CUDA path and the fp64 oracle can take their inputs from it
without sharing any computation.

All draws use numpy's PCG64 through ``SeedSequence``; large tensors are split into
fixed-size chunks, each with its own spawned seed, so the values depend only on the
seed (not on the thread count or the machine).  bf16 tensors are drawn in fp32 and
rounded to bf16 by torch's CPU conversion (round-to-nearest-even).

Workload shapes follow the pages' workloads:
  * "P-EAGLE: A Technical Deep Dive into Parallel Speculative Decoding", section
    "2. The P-EAGLE Parallel Drafter": one NTP row (emb(new) + h_context) and K-1 MTP
    rows (emb(mask) + h_shared) per request.
  * "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training", A4 (experimental setup):
    4 Llama-3 decoder layers, K_train = 8, COD down-sampling ratio 0.8, sequences of
    up to 8192 tokens; Fig 1 (reasoning traces with median near 4K and P90 above 10K
    tokens) motivates the KV lengths below.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np
import torch

_CHUNK = 1 << 22  # elements per independently seeded chunk


@dataclasses.dataclass(frozen=True)
class Dims:
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    draft_vocab: int
    target_vocab: int
    rope_theta: float
    rms_eps: float
    dtype: str  # "f32" or "bf16"
    d2t: str  # "identity" or "monotone"
    attn_window: int = 0  # drafter attention window in positions (0: the whole context)
    lm_rank: int = 0  # efficient LM head: rank of the scoring projection (0: full head)
    lm_topk: int = 0  # efficient LM head: candidates the full head scores

    @property
    def qkv_out(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    batch: int
    K: int
    seq_lens: tuple  # per-request committed KV length; () when drawn from kv_range
    kv_range: tuple = ()  # (lo, hi) inclusive uniform range for seq_lens
    capacity: int = 0  # KV slots per request (0 = max(seq_lens) + K)
    n_seq: int = 0  # training-style forward: sequence length n
    cod_ratio: float = 0.0
    max_seq: int = 0  # training-style forward: precomputed max-length mask size


DIMS_TINY = Dims(256, 2, 4, 2, 64, 768, 4096, 4096, 10000.0, 1e-5, "f32", "identity")
DIMS_C1 = Dims(2880, 4, 64, 8, 64, 7680, 32000, 201088, 150000.0, 1e-5, "bf16", "monotone")
DIMS_C3 = Dims(4096, 4, 32, 8, 128, 14336, 32000, 32000, 500000.0, 1e-5, "bf16", "identity")

WORKLOADS = {
    # tiny fp32 drafter, B=1, 128 cached positions, K=4
    "tiny_f32": Workload("tiny_f32", DIMS_TINY, 1, 4, (128,)),
    # decode-shaped bf16 drafter (H=2880, 4 layers), B=1, 4096 cached positions, K=8
    "decode_b1": Workload("decode_b1", DIMS_C1, 1, 8, (4096,)),
    # same drafter at concurrency 2, contexts 8192 and 10240, K=8
    "decode_b2": Workload("decode_b2", DIMS_C1, 2, 8, (8192, 10240)),
    # wider drafter (H=4096, hd=128), ragged batch 16 with contexts U[1024, 8192], K=5
    "ragged_b16": Workload("ragged_b16", DIMS_C3, 16, 5, (), kv_range=(1024, 8192)),
    # training-style parallel-prediction forward over n=2048, K=8, COD ratio 0.8
    "train_fwd": Workload("train_fwd", DIMS_C1, 1, 8, (), n_seq=2048, cod_ratio=0.8,
                          max_seq=8192),
}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill_chunks(n: int, seed, fill):
    """Run fill(rng, lo, hi) over fixed-size chunks with per-chunk spawned seeds."""
    nchunk = (n + _CHUNK - 1) // _CHUNK
    root = seed if isinstance(seed, np.random.SeedSequence) else np.random.SeedSequence(seed)
    seeds = root.spawn(max(1, nchunk))

    def job(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        fill(np.random.default_rng(seeds[i]), lo, hi)

    if nchunk <= 1:
        for i in range(nchunk):
            job(i)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(job, range(nchunk)))


def normal(shape, seed, std=1.0, dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) tensor on the CPU, deterministic in ``seed``."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    buf = np.empty(n, np.float32)

    def fill(rng, lo, hi):
        rng.standard_normal(hi - lo, dtype=np.float32, out=buf[lo:hi])
        if std != 1.0:
            buf[lo:hi] *= np.float32(std)

    _fill_chunks(n, seed, fill)
    t = torch.from_numpy(buf).reshape(shape)
    return t if dtype == torch.float32 else t.to(dtype)


def uniform_ints(n, lo, hi, seed) -> np.ndarray:
    """n integers uniform in [lo, hi) as int32."""
    return np.random.default_rng(seed).integers(lo, hi, size=n, dtype=np.int64).astype(np.int32)


def make_d2t(dims: Dims, seed) -> np.ndarray:
    """Draft->target offset table: target id = i + d2t[i].

    "monotone": a sorted random sample of draft_vocab distinct target ids, so
    i + d2t[i] is strictly increasing; "identity": all zeros.
    """
    if dims.d2t == "identity":
        return np.zeros(dims.draft_vocab, np.int32)
    rng = np.random.default_rng(seed)
    ids = np.sort(rng.choice(dims.target_vocab, size=dims.draft_vocab, replace=False))
    return (ids - np.arange(dims.draft_vocab)).astype(np.int32)


def make_weights(dims: Dims, seed: int = 1234, gains: bool = False) -> dict:
    """Random-init drafter weights: linear and embedding weights N(0, 0.02^2),
    emb(mask) and h_shared N(0, 1), RMSNorm gains 1 (the Llama initialisation).

    ``gains=True`` draws every RMSNorm gain as 1 + 0.3 N(0, 1) instead (rounded to the
    storage dtype), each gain vector from its own seed, so that a kernel that drops a
    gain or applies one norm's gain to another shows in its outputs.  The other weights
    are drawn exactly as with unit gains.

    Layout (row-major, PyTorch nn.Linear convention [out, in]):
      embed [Vt, H]; emb_mask [H]; h_shared [3H]; fc [H, 3H];
      per layer: qkv [(nq+2nkv)*hd, 2H (layer 0) or H], o [H, nq*hd],
                 gate [I, H], up [I, H], down [H, I], attn_norm/post_norm [H];
      final_norm [H]; lm_head [Vd, H]; d2t [Vd] int32.
    """
    H, I = dims.hidden, dims.intermediate
    dt = dims.torch_dtype
    ss = np.random.SeedSequence(seed)
    s = iter(ss.spawn(16 + 8 * dims.n_layers))
    w = {
        "embed": normal((dims.target_vocab, H), next(s), 0.02, dt),
        "emb_mask": normal((H,), next(s), 1.0, dt),
        "h_shared": normal((3 * H,), next(s), 1.0, dt),
        "fc": normal((H, 3 * H), next(s), 0.02, dt),
        "input_norm": torch.ones(H, dtype=dt),
        "hidden_norm": torch.ones(H, dtype=dt),
        "final_norm": torch.ones(H, dtype=dt),
        "lm_head": normal((dims.draft_vocab, H), next(s), 0.02, dt),
        "d2t": make_d2t(dims, next(s)),
        "layers": [],
    }
    if dims.lm_rank > 0:
        # rank-r scoring factors (lm_score lm_proj approximates the LM head) and a head
        # that is that product plus N(0, 0.005^2), all in the head's N(0, 0.02^2) scale
        # (own seeds: the other weights are drawn exactly as without the factors)
        r = dims.lm_rank
        s2 = iter(np.random.SeedSequence(seed + 7919).spawn(3))
        std = float(np.sqrt(0.02 / np.sqrt(r)))
        proj = normal((r, H), next(s2), std, torch.float32)
        score = normal((dims.draft_vocab, r), next(s2), std, torch.float32)
        head = score @ proj + normal((dims.draft_vocab, H), next(s2), 0.005, torch.float32)
        w["lm_proj"] = proj.to(dt)
        w["lm_score"] = score.to(dt)
        w["lm_head"] = head.to(dt)
    for layer in range(dims.n_layers):
        din = 2 * H if layer == 0 else H
        w["layers"].append({
            "qkv": normal((dims.qkv_out, din), next(s), 0.02, dt),
            "o": normal((H, dims.n_q_heads * dims.head_dim), next(s), 0.02, dt),
            "gate": normal((I, H), next(s), 0.02, dt),
            "up": normal((I, H), next(s), 0.02, dt),
            "down": normal((H, I), next(s), 0.02, dt),
            "attn_norm": torch.ones(H, dtype=dt),
            "post_norm": torch.ones(H, dtype=dt),
        })
    if gains:
        g = iter(np.random.SeedSequence(seed + 104729).spawn(3 + 2 * dims.n_layers))

        def gain():
            return (1.0 + normal((H,), next(g), 0.3, torch.float32)).to(dt)

        for name in ("input_norm", "hidden_norm", "final_norm"):
            w[name] = gain()
        for L in w["layers"]:
            L["attn_norm"] = gain()
            L["post_norm"] = gain()
    return w


def seq_lens_for(wl: Workload, seed: int = 7) -> np.ndarray:
    if wl.seq_lens:
        return np.asarray(wl.seq_lens, np.int32)
    lo, hi = wl.kv_range
    return uniform_ints(wl.batch, lo, hi + 1, seed)


def make_decode_inputs(wl: Workload, seed: int = 99, capacity: int | None = None) -> dict:
    """Inputs of one draft pass: committed KV cache, seq_lens, target hidden, new token.

    The KV cache holds N(0, 1) entries in the dims' dtype with layout
    [n_layers][batch][n_kv_heads][capacity][head_dim]; cached keys are taken as
    already rotated.  Slots at and beyond seq_lens[b] are filled with random values
    too (the draft pass overwrites slots seq_lens[b] .. seq_lens[b]+K-1).
    """
    d = wl.dims
    ss = iter(np.random.SeedSequence(seed).spawn(8))
    lens = seq_lens_for(wl, next(ss))
    cap = capacity or wl.capacity or int(lens.max()) + wl.K
    shape = (d.n_layers, wl.batch, d.n_kv_heads, cap, d.head_dim)
    return {
        "seq_lens": lens,
        "capacity": cap,
        "K": wl.K,
        "cache_k": normal(shape, next(ss), 1.0, d.torch_dtype),
        "cache_v": normal(shape, next(ss), 1.0, d.torch_dtype),
        "target_hidden": normal((wl.batch, 3 * d.hidden), next(ss), 1.0, d.torch_dtype),
        "new_token": uniform_ints(wl.batch, 0, d.target_vocab, next(ss)),
    }


def uniform_target_argmax(batch: int, K: int, vocab: int, seed: int = 5) -> np.ndarray:
    """Target argmax ids over K+1 positions, uniform over the target vocabulary."""
    return uniform_ints(batch * (K + 1), 0, vocab, seed).reshape(batch, K + 1)


def geometric_prefix_lengths(batch: int, K: int, p_continue: float, seed: int = 6) -> np.ndarray:
    """Agreement lengths m with P(m >= k) = p_continue**k, capped at K."""
    rng = np.random.default_rng(seed)
    m = rng.geometric(1.0 - p_continue, size=batch) - 1  # support 0, 1, 2, ...
    return np.minimum(m, K).astype(np.int32)


def geometric_target_argmax(draft: np.ndarray, vocab: int, p_continue: float = 0.7,
                            seed: int = 6) -> tuple:
    """Target argmax that agrees with ``draft`` [B, K] on a geometric prefix.

    Returns (target_argmax [B, K+1], m [B]): positions i < m copy the draft,
    position m (if m < K) holds a different id, later positions are random.
    """
    B, K = draft.shape
    m = geometric_prefix_lengths(B, K, p_continue, seed)
    rng = np.random.default_rng(seed + 1)
    tgt = rng.integers(0, vocab, size=(B, K + 1)).astype(np.int32)
    for b in range(B):
        tgt[b, : m[b]] = draft[b, : m[b]]
        if m[b] < K and tgt[b, m[b]] == draft[b, m[b]]:
            tgt[b, m[b]] = (draft[b, m[b]] + 1) % vocab
    return tgt, m


def cod_uniforms(n: int, K: int, seed: int = 11) -> np.ndarray:
    """Uniform [0,1) variates u[p, d-1] that COD sampling compares with its ratio
    (column 0, depth 1, is unused: depth 1 is always kept)."""
    return np.random.default_rng(seed).random((n, K))


def make_train_inputs(wl: Workload, seed: int = 21) -> dict:
    """Inputs of the training-style forward: tokens [n], target hidden [n, 3H], COD draws."""
    d = wl.dims
    ss = iter(np.random.SeedSequence(seed).spawn(4))
    return {
        "tokens": uniform_ints(wl.n_seq, 0, d.target_vocab, next(ss)),
        "hidden": normal((wl.n_seq, 3 * d.hidden), next(ss), 1.0, d.torch_dtype),
        "cod_u": cod_uniforms(wl.n_seq, wl.K, next(ss)),
    }


def shrink(dims: Dims, **kw) -> Dims:
    """A copy of ``dims`` with some fields replaced (small test drafters)."""
    return dataclasses.replace(dims, **kw)
