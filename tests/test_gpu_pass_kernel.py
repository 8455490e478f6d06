"""The persistent pass kernel (the whole bf16 draft pass as one launch) against the
multi-kernel path and the fp64 oracle, through the C ABI: same logits within the bf16
tolerance, same ids wherever the oracle's margin allows, same KV rows, same device
checks."""
import numpy as np
import pytest
import torch

import synth
from pe_helpers import (LOGIT_TOL, check_tokens_vs_own_logits, compare, make_ctx, oracle_draft,
                        pk, run_draft, to_dev)

pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                        intermediate=320, draft_vocab=1000, target_vocab=1500,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")
SMALL_HD128 = synth.Dims(hidden=256, n_layers=3, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         intermediate=384, draft_vocab=777, target_vocab=777,
                         rope_theta=500000.0, rms_eps=1e-5, dtype="bf16", d2t="identity")


def _both(dims, w, inp, K, cap):
    B = len(inp["seq_lens"])
    out = []
    for flag in (True, False):
        ctx = make_ctx(dims, w, B, K, cap, pass_kernel=flag)
        toks, lg, d = run_draft(ctx, dims, inp, K)
        out.append((toks, lg, d))
        ctx.close()
    return out


@pytest.mark.parametrize("dims,lens,K", [
    (SMALL_BF16, [0, 37, 100], 5),
    (SMALL_BF16, [300, 64], 8),
    (SMALL_BF16, [1, 250, 17, 5], 4),
    (SMALL_HD128, [50, 200], 4),
    (SMALL_HD128, [0], 1),
])
def test_pass_kernel_matches_multi_kernel_and_oracle(dims, lens, K):
    wl = synth.Workload("s", dims, len(lens), K, tuple(lens))
    w = synth.make_weights(dims, 11 + K, gains=True)
    inp = synth.make_decode_inputs(wl, 12 + K)
    (t1, l1, d1), (t2, l2, d2) = _both(dims, w, inp, K, inp["capacity"] + 1)
    assert float(np.max(np.abs(l1 - l2))) <= LOGIT_TOL["bf16"] / 4
    ref = oracle_draft(dims, w, inp, K)
    compare(dims, ref, t1, l1, f"pass kernel {lens} K={K}")
    check_tokens_vs_own_logits(t1, l1, w["d2t"])
    # the draft-block K/V rows written to the cache agree between the two paths
    for b, L in enumerate(lens):
        a = d1["ck"][:, b, :, L:L + K].float()
        c = d2["ck"][:, b, :, L:L + K].float()
        assert float((a - c).abs().max()) < 3e-2


def test_pass_kernel_decode_b1_repeat_deterministic():
    """Two passes on the same inputs give bit-identical logits: the residual stream is
    fixed point and every fix-up adds its partials in a fixed order."""
    wl = synth.WORKLOADS["decode_b1"]
    dims = wl.dims
    w = synth.make_weights(dims, 1234, gains=True)
    inp = synth.make_decode_inputs(wl, 99)
    ctx = make_ctx(dims, w, 1, wl.K, inp["capacity"], pass_kernel=True)
    d = to_dev(inp)
    t1, l1, _ = run_draft(ctx, dims, inp, wl.K, d=d)
    t2, l2, _ = run_draft(ctx, dims, inp, wl.K, d=d)
    ctx.close()
    assert np.array_equal(t1, t2)
    assert np.array_equal(l1, l2)
    ref = oracle_draft(dims, w, inp, wl.K)
    compare(dims, ref, t1, l1, "pass kernel decode_b1")


@pytest.mark.parametrize("use_pass", [True, False])
def test_bf16_device_checks(use_pass):
    """Bad token and KV overflow are latched by the pass kernel and by the bf16 multi-kernel
    path (whose fixed-point q / k,v sums are cleared even for rows without a cache slot);
    a valid pass afterwards matches the oracle."""
    m = pk()
    dims = SMALL_BF16
    wl = synth.Workload("s", dims, 1, 4, (10,))
    w = synth.make_weights(dims, 5, gains=True)
    inp = synth.make_decode_inputs(wl, 6, capacity=16)
    ctx = make_ctx(dims, w, 1, 8, 64, pass_kernel=use_pass)
    d = to_dev(inp)
    kv = m.kv_struct(d["ck"], d["cv"], 16, 1)
    toks = torch.empty(1, 4, dtype=torch.int32, device="cuda")
    bad = torch.tensor([dims.target_vocab + 5], dtype=torch.int32, device="cuda")
    m.peagle_draft(ctx, 1, kv, d["sl"], d["th"], bad, 4, toks)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_BAD_TOKEN
    over = torch.tensor([14], dtype=torch.int32, device="cuda")  # 14 + 4 > 16
    m.peagle_draft(ctx, 1, kv, over, d["th"], d["nt"], 4, toks)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_KV_OVERFLOW
    toks2, lg, _ = run_draft(ctx, dims, inp, 4)
    ref = oracle_draft(dims, w, inp, 4)
    compare(dims, ref, toks2, lg, f"after errors (pass kernel {use_pass})")
    ctx.close()
