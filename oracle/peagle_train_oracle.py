"""P-EAGLE oracle, training step: loss and parameter gradients of the training-style
parallel-prediction forward, in float64 on the CPU.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or executes this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the CUDA
library.

Sources (page title, then section):
  [PE]  "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training" - A2 section 2 (the
        drafter: NTP / MTP inputs, N Llama-3 layers with RoPE, LM head), section 3
        (training over n x K positions with COD-retained rows and the depth mask).
  [RH]  "Speeding LLM inference with P-EAGLE in vLLM/Speculators" - "Flex-attention mask".

The forward is the one of ``peagle_oracle.forward_parallel`` in exact mode (every value
widened to float64, no bf16 rounding), restated here with the intermediates the backward
needs kept.  Reading (the pages name no loss): the training step's loss is the mean over
the retained rows of the cross-entropy of the row's draft-vocabulary logits against a
label per row (synthetic labels are inputs); the step computes the loss and the gradient
of every parameter (no optimizer).  Each gradient below is the chain rule written out by
hand for its forward step; ``tests/test_oracle_pins.py`` pins them against central finite
differences of the loss and the logits against ``forward_parallel``.
"""
from __future__ import annotations

import math

import numpy as np

from .peagle_oracle import Weights64, rope, to64


def _rms_fwd(x, g, eps):
    """RMSNorm y = x r g with r = (mean(x^2) + eps)^-1/2 per row; returns (y, r)."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * g, r


def _rms_bwd(x, r, g, dy):
    """Gradients of y = x r g: dx = r z - r^3 x (z . x) / D with z = dy g (r depends on
    every entry of the row), dg = sum over rows of dy x r."""
    z = dy * g
    D = x.shape[-1]
    dx = r * z - (r ** 3) * x * np.sum(z * x, axis=-1, keepdims=True) / D
    dg = np.sum(dy * x * r, axis=0)
    return dx, dg


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def mask_matrix(rows):
    """allowed[i, j]: row i = (p, d) may attend row j = (p', d') ([RH] "Flex-attention
    mask"): (d' = 1 and p' <= p - d + 1) or (p' - d' = p - d and d' <= d)."""
    rows = np.asarray(rows, np.int64)
    P, D = rows[:, 0], rows[:, 1]
    anchor = P - D + 1
    return ((D[None, :] == 1) & (P[None, :] <= anchor[:, None])) | (
        ((P[None, :] - D[None, :]) == (P - D)[:, None]) & (D[None, :] <= D[:, None]))


def train_step(W: Weights64, dims, tokens, hidden, rows, labels):
    """Loss and gradients of one training step over retained rows (p, d).

    labels: [M] draft-vocabulary ids, one per row.  Returns (loss, logits [M, Vd], grads)
    with grads a dict of float64 arrays shaped like the weights: embed [Vt, H], emb_mask,
    h_shared, fc, input_norm, hidden_norm, final_norm, lm_head and "layers" (per layer:
    qkv, o, gate, up, down, attn_norm, post_norm; layer 0 has no attn_norm use, its
    gradient is zero).
    """
    rows = np.asarray(rows, np.int64)
    labels = np.asarray(labels, np.int64)
    M = rows.shape[0]
    H, eps = dims.hidden, dims.rms_eps
    nq, nkv, hd = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    G = nq // nkv
    scale = 1.0 / math.sqrt(hd)
    layers = [{k: to64(v) for k, v in L.items()} for L in W.layers]
    fc, lm_head = to64(W.fc), to64(W.lm_head)

    # ---- forward ([PE] A2 section 2), keeping the intermediates
    E = np.empty((M, H))
    Hin = np.empty((M, 3 * H))
    mtp = rows[:, 1] != 1
    for i, (p, d) in enumerate(rows):
        if d == 1:
            E[i] = to64(W.embed[int(tokens[p])])
            Hin[i] = to64(hidden[p])
        else:
            E[i] = W.emb_mask
            Hin[i] = W.h_shared
    f = Hin @ fc.T
    n1, r1 = _rms_fwd(E, W.input_norm, eps)
    n2, r2 = _rms_fwd(f, W.hidden_norm, eps)
    x0 = np.concatenate([n1, n2], axis=-1)
    pos = rows[:, 0]
    allowed = mask_matrix(rows)
    res = f
    saved = []
    for li, L in enumerate(layers):
        if li == 0:
            a, ra = x0, None
        else:
            a, ra = _rms_fwd(res, L["attn_norm"], eps)
        qkv = a @ L["qkv"].T
        q = rope(qkv[:, : nq * hd].reshape(M, nq, hd), pos[:, None], dims.rope_theta)
        k = rope(qkv[:, nq * hd: (nq + nkv) * hd].reshape(M, nkv, hd), pos[:, None],
                 dims.rope_theta)
        v = qkv[:, (nq + nkv) * hd:].reshape(M, nkv, hd)
        probs = np.empty((nq, M, M))
        o = np.empty((M, nq, hd))
        for h in range(nq):
            s = np.where(allowed, (q[:, h] @ k[:, h // G].T) * scale, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            pr = np.exp(s)
            pr /= pr.sum(axis=1, keepdims=True)
            probs[h] = pr
            o[:, h] = pr @ v[:, h // G]
        o = o.reshape(M, nq * hd)
        res_mid = res + o @ L["o"].T
        u, ru = _rms_fwd(res_mid, L["post_norm"], eps)
        gt, up = u @ L["gate"].T, u @ L["up"].T
        act = gt * _sigmoid(gt) * up
        saved.append(dict(res_in=res, a=a, ra=ra, q=q, k=k, v=v, probs=probs, o=o,
                          res_mid=res_mid, u=u, ru=ru, gt=gt, up=up, act=act))
        res = res_mid + act @ L["down"].T
    y, ry = _rms_fwd(res, W.final_norm, eps)
    logits = y @ lm_head.T
    mx = logits.max(axis=1, keepdims=True)
    lse = mx[:, 0] + np.log(np.exp(logits - mx).sum(axis=1))
    loss = float(np.mean(lse - logits[np.arange(M), labels]))

    # ---- backward
    g = {"layers": [dict() for _ in layers]}
    dlog = np.exp(logits - lse[:, None])
    dlog[np.arange(M), labels] -= 1.0
    dlog /= M
    g["lm_head"] = dlog.T @ y
    dres, g["final_norm"] = _rms_bwd(res, ry, W.final_norm, dlog @ lm_head)
    dx0 = None
    for li in range(len(layers) - 1, -1, -1):
        L, c, gl = layers[li], saved[li], g["layers"][li]
        # MLP: res_out = res_mid + (silu(gt) * up) down^T
        gl["down"] = dres.T @ c["act"]
        dact = dres @ L["down"]
        sg = _sigmoid(c["gt"])
        dgt = dact * c["up"] * sg * (1.0 + c["gt"] * (1.0 - sg))
        dup = dact * c["gt"] * sg
        gl["gate"] = dgt.T @ c["u"]
        gl["up"] = dup.T @ c["u"]
        du = dgt @ L["gate"] + dup @ L["up"]
        dmid, gl["post_norm"] = _rms_bwd(c["res_mid"], c["ru"], L["post_norm"], du)
        dmid = dmid + dres
        # attention: res_mid = res_in + o W_o^T
        gl["o"] = dmid.T @ c["o"]
        do = (dmid @ L["o"]).reshape(M, nq, hd)
        dq = np.zeros((M, nq, hd))
        dk = np.zeros((M, nkv, hd))
        dv = np.zeros((M, nkv, hd))
        for h in range(nq):
            kv = h // G
            pr = c["probs"][h]
            dv[:, kv] += pr.T @ do[:, h]
            dpr = do[:, h] @ c["v"][:, kv].T
            ds = pr * (dpr - np.sum(dpr * pr, axis=1, keepdims=True))
            dq[:, h] = ds @ c["k"][:, kv] * scale
            dk[:, kv] += ds.T @ c["q"][:, h] * scale
        # RoPE is a rotation per position: its transpose rotates by the opposite angle
        dq = rope(dq, -pos[:, None], dims.rope_theta)
        dk = rope(dk, -pos[:, None], dims.rope_theta)
        dqkv = np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), dv.reshape(M, -1)],
                              axis=1)
        gl["qkv"] = dqkv.T @ c["a"]
        da = dqkv @ L["qkv"]
        if li == 0:
            gl["attn_norm"] = np.zeros_like(L["attn_norm"])
            dx0 = da
            dres = dmid
        else:
            dr, gl["attn_norm"] = _rms_bwd(c["res_in"], c["ra"], L["attn_norm"], da)
            dres = dmid + dr
    # first-layer input: x0 = [rms_in(E) || rms_hid(f)], residual stream starts at f
    dE, g["input_norm"] = _rms_bwd(E, r1, W.input_norm, dx0[:, :H])
    df, g["hidden_norm"] = _rms_bwd(f, r2, W.hidden_norm, dx0[:, H:])
    df = df + dres
    g["fc"] = df.T @ Hin
    dHin = df @ fc
    embed = np.zeros((W.embed.shape[0], H))
    for i, (p, d) in enumerate(rows):
        if d == 1:
            embed[int(tokens[p])] += dE[i]
    g["embed"] = embed
    g["emb_mask"] = dE[mtp].sum(axis=0)
    g["h_shared"] = dHin[mtp].sum(axis=0)
    return loss, logits, g
