"""peagle_decode_attention_static: decode attention for callers that may not allocate.

Some users of this library cannot call cudaMalloc where attention runs (their device
memory belongs to their own arena allocator, or they may not make allocating CUDA calls at
that point), so they cannot hold a peagle_ctx.  The static entry point takes only inputs
and outputs and keeps its split-KV partials in an array built into the library.

Two checks of its output:
  * against the existing entry point, peagle_draft, on a one-layer bf16 drafter chosen so
    that its logits show the attention output directly: fc = 0 (the residual starts at 0),
    o-proj = identity, MLP = 0, final-norm gain 1 and LM head = identity, so every row's
    logits are that row's attention output divided by its RMS.  The static entry point is
    given the same post-RoPE queries and the KV cache peagle_draft just filled (including
    the draft block); its output, RMS-normalised, must match those logits within the bf16
    logit tolerance of the other tests.  Head dims 64 and 128, two calls in a row.
  * against the fp64 oracle's softmax attention (``attend``) on the same queries (rounded
    to bf16, as the kernel does) and cache, within the same tolerance: the head-dim 64 and
    128 cases above, and a batch whose partials fill the static array so that the call
    runs the reduced plan of fewer, longer chunks.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O
from pe_helpers import LOGIT_TOL, make_ctx, pk

pytestmark = pytest.mark.gpu

DIMS = synth.Dims(hidden=256, n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=64,
                  intermediate=64, draft_vocab=256, target_vocab=300, rope_theta=10000.0,
                  rms_eps=1e-5, dtype="bf16", d2t="identity")
# head_dim 128: n_q_heads * head_dim = hidden keeps the identity o-projection square
DIMS128 = synth.shrink(DIMS, n_q_heads=2, n_kv_heads=1, head_dim=128)
TOL = LOGIT_TOL["bf16"]


def _weights(dims, seed):
    w = synth.make_weights(dims, seed)
    H = dims.hidden
    eye = torch.eye(H, dtype=torch.bfloat16)
    w["fc"] = torch.zeros_like(w["fc"])
    w["lm_head"] = eye.clone()
    L = w["layers"][0]
    L["o"] = eye.clone()
    L["gate"] = torch.zeros_like(L["gate"])
    L["up"] = torch.zeros_like(L["up"])
    L["down"] = torch.zeros_like(L["down"])
    return w


def _queries(dims, w, inp, K):
    """Post-RoPE queries of the draft rows (float64): x0 = [RMSNorm(e) || 0] since fc = 0."""
    H, nq, hd = dims.hidden, dims.n_q_heads, dims.head_dim
    Wq = w["layers"][0]["qkv"][: nq * hd].double().numpy()
    B = len(inp["seq_lens"])
    q = np.zeros((B * K, nq, hd))
    half = hd // 2
    inv = dims.rope_theta ** (-(2.0 * np.arange(half)) / hd)
    for b in range(B):
        for j in range(K):
            e = (w["embed"][int(inp["new_token"][b])] if j == 0 else w["emb_mask"]).double().numpy()
            x = e / np.sqrt(np.mean(e * e) + dims.rms_eps)
            x0 = np.concatenate([x, np.zeros(H)])
            qq = (Wq @ x0).reshape(nq, hd)
            ang = (int(inp["seq_lens"][b]) + j) * inv
            c, s = np.cos(ang), np.sin(ang)
            q[b * K + j] = np.concatenate([qq[:, :half] * c - qq[:, half:] * s,
                                           qq[:, half:] * c + qq[:, :half] * s], axis=1)
    return q


def _oracle_attention(q, ck, cv, lens, K, nq, nkv, cap):
    """fp64 softmax attention of every (row, head): request b's row j sees the slots
    0 .. min(lens[b] + j, cap - 1) of kv head h // (nq / nkv); queries rounded to bf16."""
    B, hd = len(lens), q.shape[-1]
    qr = O.bf16_round(q)
    ck = O.to64(ck)
    cv = O.to64(cv)
    out = np.zeros((B * K, nq, hd))
    for b in range(B):
        for j in range(K):
            n_vis = min(int(lens[b]) + j + 1, cap)
            for h in range(nq):
                g = h // (nq // nkv)
                out[b * K + j, h] = O.attend(qr[b * K + j, h], ck[b, g, :n_vis], cv[b, g, :n_vis],
                                             1.0 / np.sqrt(hd))
    return out


def _static(B, K, nq, nkv, hd, q, ck, cv, cap, sl):
    m = pk()
    out = torch.full((B * K, nq, hd), float("nan"), device="cuda")
    m.peagle_decode_attention_static(B, K, nq, nkv, hd, q, ck, cv, cap, sl, out)
    torch.cuda.synchronize()
    return out


def _one_case(dims, lens, K, seed):
    m = pk()
    w = _weights(dims, seed)
    wl = synth.Workload("s", dims, len(lens), K, tuple(lens))
    inp = synth.make_decode_inputs(wl, seed + 1)
    cap = inp["capacity"]
    B = len(lens)
    ctx = make_ctx(dims, w, B, K, cap)
    ck = inp["cache_k"].cuda()
    cv = inp["cache_v"].cuda()
    sl = torch.from_numpy(inp["seq_lens"]).cuda()
    kv = m.kv_struct(ck, cv, cap, B)
    toks = torch.empty(B, K, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, K, dims.draft_vocab, device="cuda")
    m.peagle_draft(ctx, B, kv, sl, inp["target_hidden"].cuda(),
                   torch.from_numpy(inp["new_token"]).cuda(), K, toks, logits)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    ctx.close()
    q64 = _queries(dims, w, inp, K)
    q = torch.from_numpy(q64).float().cuda().contiguous()
    # the cache now holds the draft block written by peagle_draft (layer 0 is the only one)
    out = _static(B, K, dims.n_q_heads, dims.n_kv_heads, dims.head_dim, q, ck[0], cv[0], cap, sl)
    o = out.reshape(B * K, -1).double().cpu().numpy()
    assert np.isfinite(o).all()
    normed = o / np.sqrt(np.mean(o * o, axis=1, keepdims=True) + dims.rms_eps)
    ref = logits.reshape(B * K, -1).double().cpu().numpy()
    err = float(np.max(np.abs(normed - ref)))
    assert err <= TOL, f"static attention vs peagle_draft: {err:.3e}"
    want = _oracle_attention(q.double().cpu().numpy(), ck[0].cpu(), cv[0].cpu(), lens, K,
                             dims.n_q_heads, dims.n_kv_heads, cap)
    err_o = float(np.max(np.abs(out.double().cpu().numpy() - want)))
    assert err_o <= TOL, f"static attention vs the oracle: {err_o:.3e}"
    return out


@pytest.mark.parametrize("dims", [DIMS, DIMS128], ids=["hd64", "hd128"])
def test_static_attention_matches_draft_pass_two_calls(dims):
    # two calls in a row with the same shapes on different inputs: the second call's
    # output is its own (nothing of the first call's scratch leaks into it)
    a = _one_case(dims, [37, 130], 5, 70)
    b = _one_case(dims, [37, 130], 5, 90)
    assert not torch.equal(a, b)
    _one_case(dims, [3], 8, 110)


def test_static_attention_reduced_chunk_plan():
    """8 requests x 8 kv heads x 128 rows x 130 floats = 4.26 MB of partials per chunk: the
    static array holds one chunk per (request, kv head), fewer than the plan wants, so every
    request's keys run as one long chunk."""
    B, K, nq, nkv, hd = 8, 16, 64, 8, 128
    per_chunk = B * nkv * K * (nq // nkv) * (hd + 2) * 4
    assert (8 << 20) // per_chunk == 1
    lens = [int(x) for x in synth.uniform_ints(B, 0, 280, 5)]
    cap = max(lens) + K
    shape = (B, nkv, cap, hd)
    ck = synth.normal(shape, 6, 1.0, torch.bfloat16).cuda()
    cv = synth.normal(shape, 7, 1.0, torch.bfloat16).cuda()
    q = synth.normal((B * K, nq, hd), 8, 1.0).cuda()
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = _static(B, K, nq, nkv, hd, q, ck, cv, cap, sl)
        want = _oracle_attention(q.double().cpu().numpy(), ck.cpu(), cv.cpu(), lens, K, nq, nkv,
                                 cap)
        err = float(np.max(np.abs(out.double().cpu().numpy() - want)))
        assert err <= TOL, f"reduced chunk plan vs the oracle: {err:.3e}"
        q = -q


def test_static_attention_rejects_oversized_batch():
    m = pk()
    # 64 requests x 32 kv heads x 128 rows x 130 floats per chunk exceeds the static array
    q = torch.zeros(1, device="cuda")
    sl = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(m.PeagleError) as ei:
        m.peagle_decode_attention_static(64, 16, 256, 32, 128, q, q, q, 64, sl, q)
    assert ei.value.code == m.PEAGLE_ERR_CAPACITY
