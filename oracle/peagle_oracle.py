"""P-EAGLE oracle: a plain, slow fp64 CPU restatement of the parallel draft pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or executes this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the CUDA
library: inputs come from the seeded generators in ``synth``; everything below is
numpy in float64, written from the pages' statement of the method.

Sources (page title, then section):
  [RH]  "Speeding LLM inference with P-EAGLE in vLLM/Speculators"
        - "COD sampling", "A learnable mask parameter", "Flex-attention mask",
          "Train your own in 4 steps" (the --no-norm-before-residual flag and the
          3-layer hidden-state concatenation), "Example model" (acceptance table).
  [TD]  "P-EAGLE: A Technical Deep Dive into Parallel Speculative Decoding"
        - "2. The P-EAGLE Parallel Drafter" (NTP / MTP inputs, N layers + LM head in
          one execution), "Memory and Training Complexity" (65,536 positions, ~8 GB).
  [E4]  "EAGLE-4" - "EAGLE-4 overview" (greedy acceptance: longest agreeing prefix
        plus one bonus token); "Lossless speculation and floating-point behavior"
        (near-tie policy).
  [PE]  "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training" (arXiv 2602.01469
        notes) - A2 section 2 (architecture), 3.1 (amortized mask construction),
        3.2 (sequence partitioning), A4 (setup: 4 Llama-3 layers, K=8, COD 0.8).

Readings where the pages are silent or ambiguous are listed with the design notes;
the ones this file depends on are repeated at the function that applies them.

Modes of arithmetic (argument ``bf16``):
  * exact (False): every value is widened exactly to float64 and the whole pass is
    evaluated in float64;
  * cast-emulating (a set of point names from CAST_POINTS, or True for all of them):
    values are rounded to the nearest bf16 (ties to even) at the named storage points
    (x0: the 2H first-layer input, xn: normalised projection inputs, q, kv: keys and
    values, o: attention output, act: SwiGLU product, y: LM-head input).  The bf16 GPU
    path rounds keys, values and queries (DRAFT_BF16_CASTS); the default for bf16 dims.
    Accumulations, the residual stream, norms, RoPE and softmax stay float64 here.

Parity status of each function (what pins it, besides this file) is tested in
tests/test_oracle_pins.py.  Logit VALUES of the full pass are not printed anywhere in
the pages; they are pinned only through closed-form degenerate cases and invariants.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# ----------------------------------------------------------------------------------
# scalar helpers
# ----------------------------------------------------------------------------------


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significand bits (7 stored) and fp32's exponent range; the
    smallest subnormal step is 2**-133.  Written from that definition: scale each
    value so its bf16 ulp becomes 1, round half to even with np.rint, scale back.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1  (ulp of bf16 = 2**(e-8))
    shift = np.maximum(e - 8, -133)
    q = np.rint(np.ldexp(x, -shift))
    out = np.ldexp(q, shift)
    out = np.where(np.abs(out) > 3.3895313892515355e38, np.copysign(np.inf, x), out)
    return np.where(x == 0, x, out)


def to64(t):
    """Widen a torch/numpy array (fp32 or bf16) exactly to a float64 numpy array."""
    try:
        import torch

        if isinstance(t, torch.Tensor):
            return t.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def rmsnorm(x, gamma, eps):
    """RMSNorm as in Llama-3 decoder layers ([PE] A2 section 2: Llama-3 layers):
    x / sqrt(mean(x^2) + eps) * gamma, over the last axis."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gamma


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x, pos, theta):
    """Rotary position embedding, rotate-half pairing (i, i + hd/2).

    Reading: the pages only say "Llama-3 with RoPE" ([TD] "2. The P-EAGLE Parallel
    Drafter"; [PE] A2 section 2); this takes the Llama layout with
    inv_freq_i = theta**(-2i/hd), no frequency scaling.
    x: [..., hd]; pos: integer array broadcastable to x.shape[:-1].
    """
    x = np.asarray(x, np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-(2.0 * np.arange(half)) / hd)
    ang = np.asarray(pos, np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attend(q, keys, values, scale):
    """Softmax attention of one query over a set of keys: sum_k softmax(q.k*scale)_k v_k."""
    s = (keys @ q) * scale
    s = s - s.max()
    p = np.exp(s)
    p /= p.sum()
    return p @ values


# ----------------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------------


@dataclass
class Weights64:
    """The drafter's weights widened to float64 (see ``synth.make_weights``)."""

    embed: object  # [Vt, H] kept in its stored dtype; rows are widened on use
    emb_mask: np.ndarray
    h_shared: np.ndarray
    fc: np.ndarray
    input_norm: np.ndarray
    hidden_norm: np.ndarray
    final_norm: np.ndarray
    lm_head: np.ndarray
    d2t: np.ndarray
    layers: list
    lm_proj: object = None   # efficient LM head: [rank, H] projection of the head input
    lm_score: object = None  # efficient LM head: [Vd, rank] scores of the projection

    @staticmethod
    def from_synth(w, lazy=False):
        """``lazy=True`` keeps the per-layer matrices in their stored dtype and widens
        each one when it is used (saves host memory on the large drafters)."""
        conv = (lambda t: t) if lazy else to64
        return Weights64(
            embed=w["embed"],
            emb_mask=to64(w["emb_mask"]),
            h_shared=to64(w["h_shared"]),
            fc=conv(w["fc"]),
            input_norm=to64(w["input_norm"]),
            hidden_norm=to64(w["hidden_norm"]),
            final_norm=to64(w["final_norm"]),
            lm_head=conv(w["lm_head"]),
            d2t=np.asarray(w["d2t"], np.int64),
            layers=[{k: (to64(v) if k.endswith("norm") else conv(v)) for k, v in L.items()}
                    for L in w["layers"]],
            lm_proj=to64(w["lm_proj"]) if "lm_proj" in w else None,
            lm_score=to64(w["lm_score"]) if "lm_score" in w else None,
        )


def _mat(a):
    return a if isinstance(a, np.ndarray) and a.dtype == np.float64 else to64(a)


def linear(x, w):
    """y = x W^T for an nn.Linear weight W [out, in] (x: [rows, in])."""
    return x @ _mat(w).T


# ----------------------------------------------------------------------------------
# the draft pass ([TD] "2. The P-EAGLE Parallel Drafter"; [PE] A2 section 2)
# ----------------------------------------------------------------------------------


@dataclass
class DraftResult:
    logits: np.ndarray  # [B, K, Vd]
    argmax: np.ndarray  # [B, K] draft-vocab index
    tokens: np.ndarray  # [B, K] target-vocab id = argmax + d2t[argmax]
    margin: np.ndarray  # [B, K] top-1 minus top-2 logit
    k_rows: list  # per layer [B, K, nkv, hd] keys written for the draft block (post-RoPE)
    v_rows: list  # per layer [B, K, nkv, hd]
    approx: object = None  # efficient LM head: [B, K, Vd] rank-r scores (else None)


def input_rows(W: Weights64, dims, target_hidden, new_token, K):
    """Per-row drafter inputs for B requests x K positions, row r = b*K + j.

    Row j=0 (NTP): token embedding of the newly generated token and the target's
    concatenated hidden states h_context (3H).  Rows j>=1 (MTP): the learnable mask
    embedding emb(mask) and the learnable shared hidden state h_shared
    ([TD] "2. The P-EAGLE Parallel Drafter").  h_shared is 3H wide, like the target
    hidden it replaces ([RH] "A learnable mask parameter": mask_hidden [1,1,3*hidden]),
    so it goes through fc too.  emb(mask) is a separate H-vector.
    Returns (E [R,H], Hin [R,3H]).
    """
    th = to64(target_hidden)
    B = th.shape[0]
    H = dims.hidden
    E = np.empty((B * K, H))
    Hin = np.empty((B * K, 3 * H))
    for b in range(B):
        for j in range(K):
            r = b * K + j
            if j == 0:
                E[r] = to64(W.embed[int(new_token[b])])
                Hin[r] = th[b]
            else:
                E[r] = W.emb_mask
                Hin[r] = W.h_shared
    return E, Hin


CAST_POINTS = ("x0", "xn", "q", "kv", "o", "act", "y")
# Rounding profile of the bf16 GPU path (draft pass and training-style forward):
# projection inputs travel as bf16 hi + lo pairs (about 16 significant bits), so the bf16
# roundings left are the KV storage format's (keys and values) and the attention
# product's operands (post-RoPE queries; the softmax weights are rounded too, which this
# profile does not model and the logit tolerance absorbs).
DRAFT_BF16_CASTS = frozenset({"kv", "q"})
# The training-style forward rounds at the same points.
FORWARD_BF16_CASTS = DRAFT_BF16_CASTS
# Every storage point rounded to bf16 (a plain all-bf16 pipeline); kept for comparisons.
ALL_BF16_CASTS = frozenset(CAST_POINTS)


def _cast_fn(bf16, point):
    """Rounding applied at a cast point: bf16 is True (every point), False (none) or a
    collection of point names from CAST_POINTS."""
    if bf16 is True:
        return bf16_round
    if not bf16:
        return lambda v: v
    return bf16_round if point in bf16 else (lambda v: v)


def first_layer_input(W: Weights64, dims, E, Hin, bf16):
    """fc projection 3H -> H and the 2H first-layer input.

    f = fc(h); x0 = [RMSNorm_in(e) || RMSNorm_hid(f)]; the residual stream starts at f
    itself, before any norm (reading of the --no-norm-before-residual flag in
    [RH] "Train your own in 4 steps").  Returns (x0 [R,2H], res [R,H]).
    """
    cast = _cast_fn(bf16, "x0")
    f = linear(Hin, W.fc)
    x0 = np.concatenate([rmsnorm(E, W.input_norm, dims.rms_eps),
                         rmsnorm(f, W.hidden_norm, dims.rms_eps)], axis=-1)
    return cast(x0), f


def decoder_layer_decode(L, layer_idx, dims, a, res, pos, cache_k, cache_v, seq_lens, K, bf16):
    """One Llama-3 decoder layer over the K-row draft block of each request.

    a: normalised layer input [R, Din]; res: residual [R, H]; pos: [R] positions
    (row j of request b sits at seq_lens[b] + j).  Attention of row j: the cached
    keys 0..seq_lens[b]-1 plus the draft block's rows 0..j (causal), GQA with
    q head h reading kv head h // (nq/nkv), scale 1/sqrt(hd).
    With dims.attn_window = W > 0 (sliding-window drafter attention, [E4] "EAGLE-4
    overview": the drafter attends to the most recent 4,096 positions; "Long contexts"),
    row j sees only the keys at positions pos - W + 1 .. pos.  Reading: the window counts
    the query's own position.
    Returns (res_out, k_draft [B,K,nkv,hd], v_draft).
    """
    cq, ckv, co = _cast_fn(bf16, "q"), _cast_fn(bf16, "kv"), _cast_fn(bf16, "o")
    cx, ca = _cast_fn(bf16, "xn"), _cast_fn(bf16, "act")
    nq, nkv, hd = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    G = nq // nkv
    R = a.shape[0]
    B = R // K
    qkv = linear(a, L["qkv"])
    q = qkv[:, : nq * hd].reshape(R, nq, hd)
    k = qkv[:, nq * hd: (nq + nkv) * hd].reshape(R, nkv, hd)
    v = qkv[:, (nq + nkv) * hd:].reshape(R, nkv, hd)
    q = cq(rope(q, pos[:, None], dims.rope_theta))
    k = ckv(rope(k, pos[:, None], dims.rope_theta))
    v = ckv(v)
    scale = 1.0 / math.sqrt(hd)
    window = int(getattr(dims, "attn_window", 0) or 0)
    o = np.empty((R, nq, hd))
    kd = k.reshape(B, K, nkv, hd)
    vd = v.reshape(B, K, nkv, hd)
    for b in range(B):
        Lb = int(seq_lens[b])
        for g in range(nkv):
            keys = np.concatenate([to64(cache_k[b, g, :Lb]), kd[b, :, g]], axis=0)
            vals = np.concatenate([to64(cache_v[b, g, :Lb]), vd[b, :, g]], axis=0)
            for j in range(K):
                n_vis = Lb + j + 1  # key index = position
                lo = max(0, n_vis - window) if window > 0 else 0
                for h in range(g * G, (g + 1) * G):
                    o[b * K + j, h] = attend(q[b * K + j, h], keys[lo:n_vis], vals[lo:n_vis],
                                             scale)
    o = co(o.reshape(R, nq * hd))
    res = res + linear(o, L["o"])
    u = cx(rmsnorm(res, L["post_norm"], dims.rms_eps))
    act = ca(silu(linear(u, L["gate"])) * linear(u, L["up"]))
    res = res + linear(act, L["down"])
    return res, kd, vd


def lm_head_argmax(W: Weights64, dims, res, bf16):
    """Final RMSNorm, LM head, greedy argmax (lowest index on ties) and d2t remap.

    d2t is not on the pages; the reading is an offset table (target = i + d2t[i]).
    Returns (logits [R,Vd], argmax [R], tokens [R], margin [R]).
    """
    cast = _cast_fn(bf16, "y")
    y = cast(rmsnorm(res, W.final_norm, dims.rms_eps))
    if getattr(dims, "lm_rank", 0) and W.lm_proj is not None:
        return _efficient_head(W, dims, y)
    logits = linear(y, W.lm_head)
    am = np.argmax(logits, axis=-1)  # first occurrence = lowest index on ties
    top2 = np.partition(logits, -2, axis=-1)[:, -2:]
    margin = top2[:, 1] - top2[:, 0]
    tokens = am + W.d2t[am]
    return logits, am, tokens, margin


def _efficient_head(W: Weights64, dims, y):
    """Efficient LM head ([E4] "EAGLE-4 overview": a rank-128 projection scores the whole
    vocabulary, the full head then scores only the best 128 candidates; "Training with
    TorchSpec": a low-rank approximation selects the top 128 tokens).

    approx = lm_score (lm_proj y); the candidates are the lm_topk largest approx scores
    (ties: lower index first); their exact logits lm_head[c] . y decide (ties: lower
    index).  Returns (logits, argmax, tokens, margin, approx) with logits = the exact
    logits at the candidates and -inf elsewhere, margin = top-1 minus top-2 exact logit
    among the candidates.
    """
    approx = linear(linear(y, W.lm_proj), W.lm_score)
    R, Vd = approx.shape
    k = min(int(dims.lm_topk), Vd)
    logits = np.full((R, Vd), -np.inf)
    am = np.empty(R, np.int64)
    margin = np.empty(R)
    for r in range(R):
        order = np.lexsort((np.arange(Vd), -approx[r]))  # value descending, index ascending
        cand = np.sort(order[:k])
        ex = _mat(W.lm_head)[cand] @ y[r]
        logits[r, cand] = ex
        best = ex.max()
        am[r] = cand[ex == best].min()
        top2 = np.sort(ex)[-2:] if k > 1 else np.array([-np.inf, best])
        margin[r] = top2[1] - top2[0]
    tokens = am + W.d2t[am]
    return logits, am, tokens, margin, approx


def draft_pass(W: Weights64, dims, cache_k, cache_v, seq_lens, target_hidden, new_token, K,
               bf16=None) -> DraftResult:
    """The P-EAGLE parallel draft pass: all K draft tokens of each request in one pass.

    cache_k / cache_v: [n_layers][B][nkv][cap][hd] (torch or numpy), committed entries
    at slots < seq_lens[b], keys already rotated.
    ([TD] "2. The P-EAGLE Parallel Drafter": inputs of the NTP and MTP positions, N
    decoder layers and the LM head in a single execution; [PE] A2 section 2.)
    """
    if bf16 is None:
        bf16 = DRAFT_BF16_CASTS if dims.dtype == "bf16" else False
    E, Hin = input_rows(W, dims, target_hidden, new_token, K)
    return _drafter_block(W, dims, cache_k, cache_v, seq_lens, E, Hin, K, bf16)


def catch_up(W: Weights64, dims, cache_k, cache_v, seq_lens, hidden, tokens, bf16=None):
    """Drafter catch-up: T accepted tokens per request run as depth-1 (NTP) rows.

    Row t of request b takes embed[tokens[b, t]] and fc(hidden[b, t]) (the target's
    hidden states captured for that token), sits at position seq_lens[b] + t, and attends
    to the cached context and to rows 0..t -- the causal depth-1 attention of the
    training mask ("Flex-attention mask": depth-0 positions see each other causally), run
    over the new tokens of a speculative round so that their keys and values enter the
    drafter's cache ([TD] "Technical Architecture", stage 1).
    hidden: [B, T, 3H]; tokens: [B, T].  Returns a DraftResult over the T rows (k_rows /
    v_rows are the keys and values written for slots seq_lens[b] + t).
    """
    if bf16 is None:
        bf16 = DRAFT_BF16_CASTS if dims.dtype == "bf16" else False
    hid = to64(hidden)
    B, T = hid.shape[0], hid.shape[1]
    tokens = np.asarray(tokens)
    E = np.stack([to64(W.embed[int(tokens[b, t])]) for b in range(B) for t in range(T)])
    Hin = hid.reshape(B * T, -1)
    return _drafter_block(W, dims, cache_k, cache_v, seq_lens, E, Hin, T, bf16)


def _drafter_block(W: Weights64, dims, cache_k, cache_v, seq_lens, E, Hin, K, bf16):
    """N decoder layers and the LM head over a K-row block per request (row r = b*K + j at
    position seq_lens[b] + j, causal within the block) given the rows' embeddings E and
    3H hidden inputs Hin."""
    cast = _cast_fn(bf16, "xn")
    seq_lens = np.asarray(seq_lens, np.int64)
    B = len(seq_lens)
    x0, res = first_layer_input(W, dims, E, Hin, bf16)
    pos = np.array([seq_lens[b] + j for b in range(B) for j in range(K)], np.int64)
    k_rows, v_rows = [], []
    for li, L in enumerate(W.layers):
        a = x0 if li == 0 else cast(rmsnorm(res, L["attn_norm"], dims.rms_eps))
        res, kd, vd = decoder_layer_decode(L, li, dims, a, res, pos, cache_k[li], cache_v[li],
                                           seq_lens, K, bf16)
        k_rows.append(kd)
        v_rows.append(vd)
    head = lm_head_argmax(W, dims, res, bf16)
    logits, am, tokens, margin = head[:4]
    Vd = logits.shape[-1]
    approx = head[4].reshape(B, K, Vd) if len(head) > 4 else None
    return DraftResult(logits.reshape(B, K, Vd), am.reshape(B, K), tokens.reshape(B, K),
                       margin.reshape(B, K), k_rows, v_rows, approx)


# ----------------------------------------------------------------------------------
# greedy verification ([E4] "EAGLE-4 overview"; [RH] "What is speculative decoding?")
# ----------------------------------------------------------------------------------


def verify_greedy(draft, target_argmax):
    """Accept the longest prefix of the draft that agrees with the target's argmax,
    plus one bonus token: the target's choice at the first disagreement (or after
    the last draft token when all K agree).

    draft [B, K]; target_argmax [B, K+1].  Returns (accept_len m [B] in 0..K,
    bonus [B] = target_argmax[b, m]).  The emitted length per round is m + 1.
    """
    draft = np.asarray(draft)
    tgt = np.asarray(target_argmax)
    B, K = draft.shape
    acc = np.zeros(B, np.int32)
    bonus = np.zeros(B, np.int32)
    for b in range(B):
        m = 0
        while m < K and draft[b, m] == tgt[b, m]:
            m += 1
        acc[b] = m
        bonus[b] = tgt[b, m]
    return acc, bonus


def acceptance_stats(accept_len, K):
    """Per-position acceptance rates and mean acceptance length.

    Pos-k rate = fraction of rounds whose first k drafts were all accepted; the mean
    acceptance length counts the bonus token: 1 + E[m] = 1 + sum_k Pos-k
    ([RH] "Example model" table).
    """
    m = np.asarray(accept_len)
    rates = np.array([(m >= k).mean() for k in range(1, K + 1)])
    return rates, 1.0 + m.mean()


# ----------------------------------------------------------------------------------
# KV commit
# ----------------------------------------------------------------------------------


def append_kv(cache_k, cache_v, seq_lens, n_commit, k_rows=None, v_rows=None):
    """Commit accepted rows to the drafter's KV cache (returns new arrays).

    With k_rows None the first n_commit[b] draft-block rows already sit at slots
    seq_lens[b] .. seq_lens[b]+n-1 and committing only advances seq_lens.  Otherwise
    k_rows/v_rows [n_layers][B][n_max][nkv][hd] are copied into those slots.
    """
    ck = np.array(cache_k, copy=True)
    cv = np.array(cache_v, copy=True)
    sl = np.array(seq_lens, np.int64, copy=True)
    for b in range(len(sl)):
        n = int(n_commit[b])
        if k_rows is not None:
            for li in range(ck.shape[0]):
                for i in range(n):
                    ck[li, b, :, sl[b] + i] = k_rows[li][b][i]
                    cv[li, b, :, sl[b] + i] = v_rows[li][b][i]
        sl[b] += n
    return ck, cv, sl.astype(np.int32)


# ----------------------------------------------------------------------------------
# training-style forward: COD sampling, mask, amortized mask, partitioning
# ----------------------------------------------------------------------------------


def cod_retained(n, K, ratio, u):
    """Conditional drop-token (COD) sampling of (position, depth) rows.

    Depths are 1-based.  Depth 1 keeps every position.  Row (p, d>=2) exists when
    its anchor p-d+1 >= 0 and is kept with probability ``ratio`` given that its
    dependency (p-1, d-1) was kept, so depth d keeps a ratio**(d-1) share of the
    positions ([RH] "COD sampling": 0.7, 0.49, ... of all positions; [PE] 3.2: n=8192,
    K=8, r=0.8 retains about 34K positions).  No floor (the 0.2 floor is the
    Speculators training option, not the paper's sampler).
    u: uniform variates [n, K]; column d-1 is compared with ratio for depth d.
    Returns the retained rows as an int array [M, 2] of (p, d), p-major order.
    """
    kept = np.zeros((n, K + 1), bool)
    kept[:, 1] = True
    for d in range(2, K + 1):
        for p in range(d - 1, n):
            kept[p, d] = kept[p - 1, d - 1] and (u[p, d - 1] < ratio)
    rows = [(p, d) for p in range(n) for d in range(1, K + 1) if kept[p, d]]
    return np.array(rows, np.int64).reshape(-1, 2)


def cod_expected_rows(n, K, ratio):
    """Expected number of retained rows: sum_d (n - d + 1) * ratio**(d-1)."""
    return sum((n - d + 1) * ratio ** (d - 1) for d in range(1, K + 1))


def mask_allowed(p, d, p2, d2):
    """Whether row (p, d) may attend row (p2, d2) (depths 1-based).

    [RH] "Flex-attention mask": depth-1 rows attend causally to each other; every row
    sees the depth-1 base context up to its anchor a = p-d+1; a deeper row sees its
    own chain (p-j, d-j); never sideways into another rollout, never forward.
    """
    a = p - d + 1
    base = (d2 == 1) and (p2 <= a)
    chain = (p2 - d2 == p - d) and (1 <= d2 <= d)
    return base or chain


def full_mask(n, K):
    """Mask over all n*K rows in p-major order (row index p*K + d-1)."""
    idx = [(p, d) for p in range(n) for d in range(1, K + 1)]
    M = np.zeros((n * K, n * K), bool)
    for i, (p, d) in enumerate(idx):
        for j, (p2, d2) in enumerate(idx):
            M[i, j] = mask_allowed(p, d, p2, d2)
    return M


def amortized_mask(M_max, n, K, rows=None):
    """[PE] 3.1: precompute the max-length mask once, then take the top-left
    (n*K x n*K) sub-matrix for a sequence of length n (a constant-time view), and
    restrict it to the retained rows/columns (p-major indices p*K + d-1)."""
    sub = M_max[: n * K, : n * K]
    if rows is None:
        return sub
    idx = rows[:, 0] * K + (rows[:, 1] - 1)
    return sub[np.ix_(idx, idx)]


def attention_matrix_bytes(n, K, bytes_per_elem=2):
    """Size of a dense (n*K)^2 attention matrix ([TD] "Memory and Training
    Complexity": 8192 tokens x K=8 -> 65,536 positions, about 8 GB in BF16)."""
    return (n * K) ** 2 * bytes_per_elem


def forward_parallel(W: Weights64, dims, tokens, hidden, rows, bf16=None):
    """Training-style parallel-prediction forward over retained rows (p, d).

    Depth-1 rows take the real token embedding and fc(target hidden at p); deeper rows
    take emb(mask) and fc(h_shared) ([PE] A2 section 2).  Row (p, d) sits at RoPE
    position p; attention follows ``mask_allowed``.  ``rows`` may be any subset that is
    closed under the mask's dependencies (e.g. all rows with p < P0).
    Returns (logits [M, Vd], argmax [M], margin [M]).
    """
    if bf16 is None:
        bf16 = FORWARD_BF16_CASTS if dims.dtype == "bf16" else False
    cx0, cxn, cq, ckv = (_cast_fn(bf16, k) for k in ("x0", "xn", "q", "kv"))
    co, cact = _cast_fn(bf16, "o"), _cast_fn(bf16, "act")
    rows = np.asarray(rows, np.int64)
    M = rows.shape[0]
    H = dims.hidden
    nq, nkv, hd = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    G = nq // nkv
    hid = hidden
    E = np.empty((M, H))
    Hin = np.empty((M, 3 * H))
    for i, (p, d) in enumerate(rows):
        if d == 1:
            E[i] = to64(W.embed[int(tokens[p])])
            Hin[i] = to64(hid[p])
        else:
            E[i] = W.emb_mask
            Hin[i] = W.h_shared
    x0, res = first_layer_input(W, dims, E, Hin, bf16)
    pos = rows[:, 0]
    P, D = rows[:, 0], rows[:, 1]
    anchor = P - D + 1
    allowed = ((D[None, :] == 1) & (P[None, :] <= anchor[:, None])) | (
        ((P[None, :] - D[None, :]) == (P - D)[:, None]) & (D[None, :] <= D[:, None]))
    scale = 1.0 / math.sqrt(hd)
    for li, L in enumerate(W.layers):
        a = x0 if li == 0 else cxn(rmsnorm(res, L["attn_norm"], dims.rms_eps))
        qkv = linear(a, L["qkv"])
        q = cq(rope(qkv[:, : nq * hd].reshape(M, nq, hd), pos[:, None], dims.rope_theta))
        k = ckv(rope(qkv[:, nq * hd: (nq + nkv) * hd].reshape(M, nkv, hd), pos[:, None],
                     dims.rope_theta))
        v = ckv(qkv[:, (nq + nkv) * hd:].reshape(M, nkv, hd))
        o = np.empty((M, nq, hd))
        for h in range(nq):
            g = h // G
            s = (q[:, h] @ k[:, g].T) * scale
            s = np.where(allowed, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            pr = np.exp(s)
            pr /= pr.sum(axis=1, keepdims=True)
            o[:, h] = pr @ v[:, g]
        o = co(o.reshape(M, nq * hd))
        res = res + linear(o, L["o"])
        u = cxn(rmsnorm(res, L["post_norm"], dims.rms_eps))
        act = cact(silu(linear(u, L["gate"])) * linear(u, L["up"]))
        res = res + linear(act, L["down"])
    logits, am, _, margin = lm_head_argmax(W, dims, res, bf16)[:4]
    return logits, am, margin


def dependency_closure(rows, targets):
    """Rows that ``targets`` (subset of ``rows``) depend on through the mask, plus the
    targets: every depth-1 row up to the largest anchor and each target's chain."""
    rows = np.asarray(rows, np.int64)
    targets = np.asarray(targets, np.int64).reshape(-1, 2)
    need = set()
    amax = int(max((p - d + 1) for p, d in targets))
    for p, d in rows:
        if d == 1 and p <= amax:
            need.add((int(p), int(d)))
    for p, d in targets:
        for j in range(int(d)):
            need.add((int(p) - j, int(d) - j))
    return np.array(sorted(need), np.int64)


def sequence_partition(rows, boundaries):
    """[PE] 3.2 sequence partitioning of retained rows into S chunks.

    boundaries: increasing chunk start positions b_0 = 0 < b_1 < ... < b_{S-1}.
    Depth-1 and depth-2 rows go to the chunk containing their position index p
    (depths "0 and 1" in the paper's 0-based counting); a row of depth d >= 3 goes to
    the chunk of its dependency (p-1, d-1) (Chunk(p,d) = Chunk(p-1,d-1)).  Each chunk
    additionally carries, as causal context, every depth-1 row whose position is below
    the chunk's end boundary.
    Returns (chunk_of [M] int, context list of arrays of depth-1 positions per chunk).
    """
    rows = np.asarray(rows, np.int64)
    bnd = np.asarray(boundaries, np.int64)
    index = {(int(p), int(d)): i for i, (p, d) in enumerate(rows)}
    chunk = np.full(len(rows), -1, np.int64)
    for i, (p, d) in enumerate(rows):
        if d <= 2:
            chunk[i] = int(np.searchsorted(bnd, p, side="right") - 1)
    for i, (p, d) in enumerate(rows):  # rows are p-major, so parents come first
        if d >= 3:
            chunk[i] = chunk[index[(int(p) - 1, int(d) - 1)]]
    S = len(bnd)
    ends = list(bnd[1:]) + [int(rows[:, 0].max()) + 1 if len(rows) else 0]
    ctx = [np.arange(0, ends[s]) for s in range(S)]
    return chunk, ctx
