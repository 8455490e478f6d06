"""GPU parity of the draft pass, verification and KV commit against the fp64 oracle,
through the C ABI.  Tolerances: logits max-abs 1e-4 (fp32 drafter) / 2e-2 (bf16
drafter); draft ids bit-exact wherever the oracle's top-1 margin exceeds 1e-2 and
always equal to the argmax of the GPU's own logits; accept lengths, bonus tokens and
KV commits bit-exact."""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O
from pe_helpers import (LOGIT_TOL, check_tokens_vs_own_logits, compare, make_ctx, oracle_draft,
                        pk, run_draft, to_dev)

pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                        intermediate=320, draft_vocab=1000, target_vocab=1500,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")
SMALL_HD128 = synth.Dims(hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=128,
                         intermediate=384, draft_vocab=777, target_vocab=777,
                         rope_theta=500000.0, rms_eps=1e-5, dtype="bf16", d2t="identity")
# every projection width a multiple of 256 and 80 draft rows: the shapes the folded GEMM
# form accepts (it is chosen where it pays: the full-size ragged_b16 pass below runs it)
SMALL_FOLD = synth.Dims(hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        intermediate=384, draft_vocab=1024, target_vocab=1536,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")


def _small_case(dims, lens, K, seed, cap=None):
    wl = synth.Workload("s", dims, len(lens), K, tuple(lens))
    w = synth.make_weights(dims, seed, gains=True)
    inp = synth.make_decode_inputs(wl, seed + 1, capacity=cap)
    return w, inp


# ------------------------------------------------------------------ tiny fp32 drafter


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny_f32"]
    w = synth.make_weights(wl.dims, 1234, gains=True)
    inp = synth.make_decode_inputs(wl, 99, capacity=int(wl.seq_lens[0]) + 16)
    ctx = make_ctx(wl.dims, w, wl.batch, 16, inp["capacity"])
    yield wl, w, inp, ctx
    ctx.close()


def test_tiny_f32_draft_parity(tiny):
    wl, w, inp, ctx = tiny
    K = wl.K
    toks, lg, d = run_draft(ctx, wl.dims, inp, K)
    ref = oracle_draft(wl.dims, w, inp, K)
    compare(wl.dims, ref, toks, lg, "tiny_f32")
    check_tokens_vs_own_logits(toks, lg, w["d2t"])
    # the pass wrote the draft block's post-RoPE keys/values into slots L .. L+K-1
    L = int(inp["seq_lens"][0])
    ck = d["ck"].cpu().double().numpy()
    cv = d["cv"].cpu().double().numpy()
    for li in range(wl.dims.n_layers):
        got_k = ck[li, 0, :, L:L + K].transpose(1, 0, 2)
        got_v = cv[li, 0, :, L:L + K].transpose(1, 0, 2)
        assert np.max(np.abs(got_k - ref.k_rows[li][0])) < 1e-4
        assert np.max(np.abs(got_v - ref.v_rows[li][0])) < 1e-4
    # committed slots untouched
    assert torch.equal(d["ck"][:, :, :, :L].cpu(), inp["cache_k"][:, :, :, :L])


@pytest.mark.parametrize("K", [1, 2, 16])
def test_tiny_f32_K_edges(tiny, K):
    wl, w, inp, ctx = tiny
    toks, lg, _ = run_draft(ctx, wl.dims, inp, K)
    ref = oracle_draft(wl.dims, w, inp, K)
    compare(wl.dims, ref, toks, lg, f"tiny K={K}")


def test_tiny_f32_empty_cache():
    dims = synth.DIMS_TINY
    w, inp = _small_case(dims, [0, 3], 4, 40)
    ctx = make_ctx(dims, w, 2, 4, 64)
    toks, lg, _ = run_draft(ctx, dims, inp, 4)
    ref = oracle_draft(dims, w, inp, 4)
    compare(dims, ref, toks, lg, "empty cache")
    ctx.close()


# ------------------------------------------------------------------ small bf16 drafters


@pytest.mark.parametrize("dims,lens,K", [
    (SMALL_BF16, [0, 37, 100], 5),
    (SMALL_BF16, [129], 1),
    (SMALL_BF16, [64, 1, 300, 17], 8),
    (SMALL_HD128, [50, 200], 3),
    (SMALL_HD128, [0], 16),
    (SMALL_HD128, [5, 40, 0, 77, 120, 9, 300, 64], 8),
    (SMALL_FOLD, [3, 50, 0, 17, 90, 200, 8, 64, 33, 1, 120, 77, 9, 45, 150, 260], 5),
])
def test_small_bf16_parity(dims, lens, K):
    w, inp = _small_case(dims, lens, K, 7 + K + len(lens))
    ctx = make_ctx(dims, w, len(lens), K, inp["capacity"] + 1)
    toks, lg, d = run_draft(ctx, dims, inp, K)
    ref = oracle_draft(dims, w, inp, K)
    compare(dims, ref, toks, lg, f"small bf16 {lens} K={K}")
    check_tokens_vs_own_logits(toks, lg, w["d2t"])
    # written draft-block rows (bf16) within one bf16 ulp-ish of the oracle's
    for b, L in enumerate(lens):
        got = d["ck"][0, b, :, L:L + K].float().cpu().numpy().transpose(1, 0, 2)
        assert np.max(np.abs(got - ref.k_rows[0][b])) < 3e-2
    ctx.close()


def test_logits_optional():
    dims = SMALL_BF16
    w, inp = _small_case(dims, [10, 20], 4, 3)
    ctx = make_ctx(dims, w, 2, 4, 64)
    t1, _, _ = run_draft(ctx, dims, inp, 4, logits=False)
    t2, lg, _ = run_draft(ctx, dims, inp, 4, logits=True)
    assert np.array_equal(t1, t2)
    ctx.close()


# ------------------------------------------------------------------ full-size bf16 configs


@pytest.fixture(scope="module")
def c1_drafter():
    dims = synth.DIMS_C1
    w = synth.make_weights(dims, 1234, gains=True)
    ctx = make_ctx(dims, w, 2, 8, 10240 + 8)
    yield dims, w, ctx
    ctx.close()


def test_decode_b1_full(c1_drafter):
    dims, w, ctx = c1_drafter
    wl = synth.WORKLOADS["decode_b1"]
    inp = synth.make_decode_inputs(wl, 99)
    toks, lg, _ = run_draft(ctx, dims, inp, wl.K)
    ref = oracle_draft(dims, w, inp, wl.K)
    err = compare(dims, ref, toks, lg, "decode_b1")
    check_tokens_vs_own_logits(toks, lg, w["d2t"])
    print(f"decode_b1 logits max abs err {err:.3e}")


def test_decode_b2_full_and_verify(c1_drafter):
    dims, w, ctx = c1_drafter
    wl = synth.WORKLOADS["decode_b2"]
    inp = synth.make_decode_inputs(wl, 98)
    toks, lg, _ = run_draft(ctx, dims, inp, wl.K)
    ref = oracle_draft(dims, w, inp, wl.K)
    compare(dims, ref, toks, lg, "decode_b2")
    check_tokens_vs_own_logits(toks, lg, w["d2t"])
    tgt, m = synth.geometric_target_argmax(toks, dims.target_vocab, 0.7, seed=6)
    m_ = pk()
    acc = torch.empty(2, dtype=torch.int32, device="cuda")
    bonus = torch.empty(2, dtype=torch.int32, device="cuda")
    m_.peagle_verify_greedy(2, wl.K, torch.from_numpy(toks).cuda(), torch.from_numpy(tgt).cuda(),
                            acc, bonus)
    racc, rbonus = O.verify_greedy(toks, tgt)
    assert np.array_equal(acc.cpu().numpy(), racc) and np.array_equal(acc.cpu().numpy(), m)
    assert np.array_equal(bonus.cpu().numpy(), rbonus)


def test_ragged_b16_full_sampled():
    wl = synth.WORKLOADS["ragged_b16"]
    dims = wl.dims
    w = synth.make_weights(dims, 4321, gains=True)
    inp = synth.make_decode_inputs(wl, 97)
    ctx = make_ctx(dims, w, wl.batch, wl.K, inp["capacity"])
    toks, lg, _ = run_draft(ctx, dims, inp, wl.K)
    ctx.close()
    idx = [0, int(np.argmax(inp["seq_lens"])), int(np.argmin(inp["seq_lens"])), 15]
    ref = oracle_draft(dims, w, inp, wl.K, idx=idx)
    compare(dims, ref, toks[idx], lg[idx], "ragged_b16 sampled")
    check_tokens_vs_own_logits(toks, lg, w["d2t"])


# ------------------------------------------------------------------ verification / commit


def test_verify_exhaustive_and_random():
    m = pk()
    import itertools
    for K in (1, 2, 3):
        drafts = np.array(list(itertools.product(range(3), repeat=K)), np.int32)
        tgts = np.array(list(itertools.product(range(3), repeat=K + 1)), np.int32)
        D = np.repeat(drafts, len(tgts), axis=0)
        T = np.tile(tgts, (len(drafts), 1))
        B = len(D)
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        bonus = torch.empty(B, dtype=torch.int32, device="cuda")
        m.peagle_verify_greedy(B, K, torch.from_numpy(D).cuda(), torch.from_numpy(T).cuda(), acc,
                               bonus)
        ra, rb = O.verify_greedy(D, T)
        assert np.array_equal(acc.cpu().numpy(), ra) and np.array_equal(bonus.cpu().numpy(), rb)
    rng = np.random.default_rng(0)
    B, K = 5000, 64
    D = rng.integers(0, 2, (B, K)).astype(np.int32)
    T = rng.integers(0, 2, (B, K + 1)).astype(np.int32)
    T[:100, :K] = D[:100]  # full acceptance
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bonus = torch.empty(B, dtype=torch.int32, device="cuda")
    m.peagle_verify_greedy(B, K, torch.from_numpy(D).cuda(), torch.from_numpy(T).cuda(), acc, bonus)
    ra, rb = O.verify_greedy(D, T)
    assert np.array_equal(acc.cpu().numpy(), ra) and np.array_equal(bonus.cpu().numpy(), rb)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_append_kv_modes(dtype):
    m = pk()
    dims = synth.shrink(synth.DIMS_TINY, dtype=dtype)
    w, inp = _small_case(dims, [5, 0, 9], 4, 11, cap=20)
    ctx = make_ctx(dims, w, 3, 4, 64)
    d = to_dev(inp)
    kv = m.kv_struct(d["ck"], d["cv"], 20, 3)
    n_commit = np.array([2, 4, 0], np.int32)
    # copy mode
    n_max = 4
    kr = synth.normal((dims.n_layers, 3, n_max, dims.n_kv_heads, dims.head_dim), 5, 1.0,
                      dims.torch_dtype)
    vr = synth.normal(kr.shape, 6, 1.0, dims.torch_dtype)
    m.peagle_append_kv(ctx, 3, kv, d["sl"], torch.from_numpy(n_commit).cuda(), kr.cuda(),
                       vr.cuda(), n_max)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    ek, ev, esl = O.append_kv(inp["cache_k"].double().numpy(), inp["cache_v"].double().numpy(),
                              inp["seq_lens"], n_commit, kr.double().numpy(), vr.double().numpy())
    assert np.array_equal(d["sl"].cpu().numpy(), esl)
    assert np.array_equal(d["ck"].cpu().double().numpy(), ek)
    assert np.array_equal(d["cv"].cpu().double().numpy(), ev)
    # in-place mode only advances seq_lens
    before = d["ck"].clone()
    m.peagle_append_kv(ctx, 3, kv, d["sl"], torch.from_numpy(n_commit).cuda())
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    assert np.array_equal(d["sl"].cpu().numpy(), esl + n_commit)
    assert torch.equal(before, d["ck"])
    ctx.close()


def test_round_draft_commit_draft():
    """A full round: draft, verify, commit the accepted rows in place, draft again; the
    second pass equals the oracle run on the committed cache."""
    m = pk()
    dims = SMALL_BF16
    K = 4
    w, inp = _small_case(dims, [12, 30], K, 21, cap=48)
    ctx = make_ctx(dims, w, 2, K, 64)
    toks, lg, d = run_draft(ctx, dims, inp, K)
    tgt, mm = synth.geometric_target_argmax(toks, dims.target_vocab, 0.7, seed=3)
    acc = torch.empty(2, dtype=torch.int32, device="cuda")
    bonus = torch.empty(2, dtype=torch.int32, device="cuda")
    m.peagle_verify_greedy(2, K, torch.from_numpy(toks).cuda(), torch.from_numpy(tgt).cuda(), acc,
                           bonus)
    # commit the NTP row plus the accepted drafts' rows (accept_len + 1), as written by
    # the draft pass; a fully accepted block commits all K rows
    acc = torch.clamp(acc, max=K - 1).to(torch.int32)
    kv = m.kv_struct(d["ck"], d["cv"], 48, 2)
    m.peagle_append_kv(ctx, 2, kv, d["sl"], acc, n_extra=1)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    inp2 = dict(inp)
    inp2["cache_k"] = d["ck"].cpu()
    inp2["cache_v"] = d["cv"].cpu()
    inp2["seq_lens"] = d["sl"].cpu().numpy()
    inp2["new_token"] = bonus.cpu().numpy()
    d["nt"] = bonus.clone()
    toks2, lg2, _ = run_draft(ctx, dims, inp2, K, d=d)
    ref2 = oracle_draft(dims, w, inp2, K)
    compare(dims, ref2, toks2, lg2, "second pass")
    ctx.close()


# ------------------------------------------------------------------ device-side checks


def test_device_checks_are_latched_not_fatal():
    m = pk()
    dims = synth.DIMS_TINY
    w, inp = _small_case(dims, [10], 4, 5, cap=16)
    ctx = make_ctx(dims, w, 1, 8, 64)
    d = to_dev(inp)
    kv = m.kv_struct(d["ck"], d["cv"], 16, 1)
    toks = torch.empty(1, 4, dtype=torch.int32, device="cuda")
    bad = torch.tensor([dims.target_vocab + 5], dtype=torch.int32, device="cuda")
    m.peagle_draft(ctx, 1, kv, d["sl"], d["th"], bad, 4, toks)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_BAD_TOKEN
    assert m.peagle_status(ctx) == m.PEAGLE_OK  # cleared
    over = torch.tensor([14], dtype=torch.int32, device="cuda")  # 14 + 4 > 16
    m.peagle_draft(ctx, 1, kv, over, d["th"], d["nt"], 4, toks)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_KV_OVERFLOW
    nc = torch.tensor([9], dtype=torch.int32, device="cuda")
    m.peagle_append_kv(ctx, 1, kv, d["sl"], nc, None, None, 4)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_BAD_COMMIT
    # host-side argument errors return without launching
    with pytest.raises(m.PeagleError):
        m.peagle_draft(ctx, 1, kv, d["sl"], d["th"], d["nt"], 9, toks)  # K > max_K
    with pytest.raises(m.PeagleError):
        m.peagle_draft(ctx, 2, kv, d["sl"], d["th"], d["nt"], 4, toks)  # batch > max_batch
    # the context still works
    toks2, lg, _ = run_draft(ctx, dims, inp, 4)
    ref = oracle_draft(dims, w, inp, 4)
    compare(dims, ref, toks2, lg, "after errors")
    ctx.close()
