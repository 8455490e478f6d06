"""peagle_decode_attention_static: decode attention for callers that may not allocate.

Some users of this library cannot call cudaMalloc where attention runs (their device
memory belongs to their own arena allocator, or they may not make allocating CUDA calls at
that point), so they cannot hold a peagle_ctx.  The static entry point takes only inputs
and outputs and keeps its split-KV partials in an array built into the library.

The check runs the existing entry point, peagle_draft, on a one-layer bf16 drafter chosen
so that its logits show the attention output directly: fc = 0 (the residual starts at 0),
o-proj = identity, MLP = 0, final-norm gain 1 and LM head = identity, so every row's
logits are that row's attention output divided by its RMS.  The static entry point is then
given the same post-RoPE queries and the KV cache peagle_draft just filled (including the
draft block), and its output, RMS-normalised, must match those logits within the bf16
logit tolerance of the other tests.  Two calls in a row on different inputs.
"""
import numpy as np
import pytest
import torch

import synth
from pe_helpers import LOGIT_TOL, make_ctx, pk

pytestmark = pytest.mark.gpu

DIMS = synth.Dims(hidden=256, n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=64,
                  intermediate=64, draft_vocab=256, target_vocab=300, rope_theta=10000.0,
                  rms_eps=1e-5, dtype="bf16", d2t="identity")


def _weights(seed):
    w = synth.make_weights(DIMS, seed)
    H = DIMS.hidden
    eye = torch.eye(H, dtype=torch.bfloat16)
    w["fc"] = torch.zeros_like(w["fc"])
    w["lm_head"] = eye.clone()
    L = w["layers"][0]
    L["o"] = eye.clone()
    L["gate"] = torch.zeros_like(L["gate"])
    L["up"] = torch.zeros_like(L["up"])
    L["down"] = torch.zeros_like(L["down"])
    return w


def _queries(w, inp, K):
    """Post-RoPE queries of the draft rows (float64): x0 = [RMSNorm(e) || 0] since fc = 0."""
    H, nq, hd = DIMS.hidden, DIMS.n_q_heads, DIMS.head_dim
    Wq = w["layers"][0]["qkv"][: nq * hd].double().numpy()
    B = len(inp["seq_lens"])
    q = np.zeros((B * K, nq, hd))
    half = hd // 2
    inv = DIMS.rope_theta ** (-(2.0 * np.arange(half)) / hd)
    for b in range(B):
        for j in range(K):
            e = (w["embed"][int(inp["new_token"][b])] if j == 0 else w["emb_mask"]).double().numpy()
            x = e / np.sqrt(np.mean(e * e) + DIMS.rms_eps)
            x0 = np.concatenate([x, np.zeros(H)])
            qq = (Wq @ x0).reshape(nq, hd)
            ang = (int(inp["seq_lens"][b]) + j) * inv
            c, s = np.cos(ang), np.sin(ang)
            q[b * K + j] = np.concatenate([qq[:, :half] * c - qq[:, half:] * s,
                                           qq[:, half:] * c + qq[:, :half] * s], axis=1)
    return q


def _one_case(lens, K, seed):
    m = pk()
    w = _weights(seed)
    wl = synth.Workload("s", DIMS, len(lens), K, tuple(lens))
    inp = synth.make_decode_inputs(wl, seed + 1)
    cap = inp["capacity"]
    B = len(lens)
    ctx = make_ctx(DIMS, w, B, K, cap)
    ck = inp["cache_k"].cuda()
    cv = inp["cache_v"].cuda()
    sl = torch.from_numpy(inp["seq_lens"]).cuda()
    kv = m.kv_struct(ck, cv, cap, B)
    toks = torch.empty(B, K, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, K, DIMS.draft_vocab, device="cuda")
    m.peagle_draft(ctx, B, kv, sl, inp["target_hidden"].cuda(),
                   torch.from_numpy(inp["new_token"]).cuda(), K, toks, logits)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    ctx.close()
    q = torch.from_numpy(_queries(w, inp, K)).float().cuda().contiguous()
    out = torch.full((B * K, DIMS.n_q_heads, DIMS.head_dim), float("nan"), device="cuda")
    # the cache now holds the draft block written by peagle_draft (layer 0 is the only one)
    m.peagle_decode_attention_static(B, K, DIMS.n_q_heads, DIMS.n_kv_heads, DIMS.head_dim, q,
                                     ck[0], cv[0], cap, sl, out)
    torch.cuda.synchronize()
    o = out.reshape(B * K, -1).double().cpu().numpy()
    normed = o / np.sqrt(np.mean(o * o, axis=1, keepdims=True) + DIMS.rms_eps)
    ref = logits.reshape(B * K, -1).double().cpu().numpy()
    err = float(np.max(np.abs(normed - ref)))
    assert np.isfinite(o).all()
    assert err <= LOGIT_TOL["bf16"], f"static attention vs peagle_draft: {err:.3e}"
    return out


def test_static_attention_matches_draft_pass_two_calls():
    a = _one_case([37, 130], 5, 70)
    b = _one_case([3], 8, 90)
    assert a.shape != b.shape or not torch.equal(a, b)


def test_static_attention_rejects_oversized_batch():
    m = pk()
    # 64 requests x 32 kv heads x 128 rows x 130 floats per chunk exceeds the static array
    q = torch.zeros(1, device="cuda")
    sl = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(m.PeagleError) as ei:
        m.peagle_decode_attention_static(64, 16, 256, 32, 128, q, q, q, 64, sl, q)
    assert ei.value.code == m.PEAGLE_ERR_CAPACITY
