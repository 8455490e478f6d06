"""GPU parity of the drafter catch-up pass (accepted tokens run as depth-1 rows, their
K/V written to the cache) against the fp64 oracle, through the C ABI; and a round that
chains catch-up, commit and the next draft pass."""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O
from pe_helpers import LOGIT_TOL, MARGIN, compare, make_ctx, oracle_draft, pk, run_draft, to_dev

pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                        intermediate=320, draft_vocab=1000, target_vocab=1500,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")


def _case(dims, lens, T, seed):
    w = synth.make_weights(dims, seed, gains=True)
    wl = synth.Workload("s", dims, len(lens), T, tuple(lens))
    inp = synth.make_decode_inputs(wl, seed + 1, capacity=max(lens) + T + 8)
    hid = synth.normal((len(lens), T, 3 * dims.hidden), seed + 2, 1.0, dims.torch_dtype)
    tok = synth.uniform_ints(len(lens) * T, 0, dims.target_vocab, seed + 3).reshape(len(lens), T)
    return w, inp, hid, tok


def _compare(dims, ref, tokens, logits, what):
    """Logits within the tolerance; ids equal wherever the oracle's margin is clear (the
    few catch-up rows of a random drafter may all be near-ties, so no quota of clear
    rows is required here)."""
    err = float(np.max(np.abs(logits - ref.logits)))
    assert err <= LOGIT_TOL[dims.dtype], f"{what}: logits max abs err {err:.3e}"
    ok = ref.margin > MARGIN
    assert np.array_equal(tokens[ok], ref.tokens[ok]), what


def _run(ctx, dims, inp, hid, tok, T, logits=True, d=None):
    m = pk()
    d = d or to_dev(inp)
    B = d["sl"].shape[0]
    kv = m.kv_struct(d["ck"], d["cv"], d["ck"].shape[3], d["ck"].shape[1])
    out = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    lg = torch.full((B, T, dims.draft_vocab), float("nan"), device="cuda") if logits else None
    m.peagle_catch_up(ctx, B, kv, d["sl"], hid.cuda(), torch.from_numpy(tok).int().cuda(), T,
                      out if logits else None, lg)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    return out.cpu().numpy(), (lg.cpu().numpy() if logits else None), d


@pytest.mark.parametrize("dims,lens,T,pass_kernel", [
    (synth.DIMS_TINY, [20], 4, None),
    (SMALL_BF16, [0, 37, 100], 5, True),
    (SMALL_BF16, [0, 37, 100], 5, False),
    (SMALL_BF16, [64, 3], 1, True),
])
def test_catch_up_matches_oracle(dims, lens, T, pass_kernel):
    w, inp, hid, tok = _case(dims, lens, T, 21 + T)
    ctx = make_ctx(dims, w, len(lens), 8, inp["capacity"], pass_kernel=pass_kernel)
    out, lg, d = _run(ctx, dims, inp, hid, tok, T)
    ctx.close()
    W = O.Weights64.from_synth(w)
    casts = O.DRAFT_BF16_CASTS if dims.dtype == "bf16" else False
    ref = O.catch_up(W, dims, inp["cache_k"], inp["cache_v"], inp["seq_lens"], hid, tok, casts)
    _compare(dims, ref, out, lg, f"catch-up {lens} T={T}")
    # the K/V rows written at seq_lens[b] + t
    for li in range(dims.n_layers):
        for b, L in enumerate(lens):
            got = d["ck"][li, b, :, L:L + T].float().cpu().numpy().transpose(1, 0, 2)
            tol = 3e-2 if dims.dtype == "bf16" else 1e-4
            assert np.max(np.abs(got - ref.k_rows[li][b])) < tol


def test_catch_up_without_outputs_writes_the_same_cache():
    dims = SMALL_BF16
    w, inp, hid, tok = _case(dims, [30, 5], 4, 61)
    ctx = make_ctx(dims, w, 2, 8, inp["capacity"])
    _, _, d1 = _run(ctx, dims, inp, hid, tok, 4, logits=True)
    _, _, d2 = _run(ctx, dims, inp, hid, tok, 4, logits=False)
    ctx.close()
    assert torch.equal(d1["ck"], d2["ck"]) and torch.equal(d1["cv"], d2["cv"])


def test_round_catch_up_commit_then_draft():
    """A speculative round's drafter side: the accepted tokens catch up (K/V into the
    cache), peagle_append_kv commits them, and the next draft pass attends to them."""
    m = pk()
    dims = SMALL_BF16
    lens, T, K = [40, 7], 3, 5
    w, inp, hid, tok = _case(dims, lens, T, 71)
    ctx = make_ctx(dims, w, 2, 8, inp["capacity"])
    d = to_dev(inp)
    _run(ctx, dims, inp, hid, tok, T, logits=False, d=d)
    kv = m.kv_struct(d["ck"], d["cv"], d["ck"].shape[3], 2)
    n = torch.full((2,), T, dtype=torch.int32, device="cuda")
    m.peagle_append_kv(ctx, 2, kv, d["sl"], n, None, None, T)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    assert d["sl"].cpu().tolist() == [L + T for L in lens]
    toks, lg, _ = run_draft(ctx, dims, inp, K, d=d)
    ctx.close()
    # oracle: the same round on the original cache
    W = O.Weights64.from_synth(w)
    cu = O.catch_up(W, dims, inp["cache_k"], inp["cache_v"], inp["seq_lens"], hid, tok)
    ck = inp["cache_k"].clone().float()
    cv = inp["cache_v"].clone().float()
    for li in range(dims.n_layers):
        for b, L in enumerate(lens):
            ck[li, b, :, L:L + T] = torch.from_numpy(cu.k_rows[li][b].transpose(1, 0, 2)).float()
            cv[li, b, :, L:L + T] = torch.from_numpy(cu.v_rows[li][b].transpose(1, 0, 2)).float()
    inp2 = dict(inp)
    inp2["cache_k"], inp2["cache_v"] = ck, cv
    inp2["seq_lens"] = np.array([L + T for L in lens], np.int32)
    ref = oracle_draft(dims, w, inp2, K)
    compare(dims, ref, toks, lg, "round: catch-up + commit + draft")
