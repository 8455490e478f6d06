"""Failure detection of the persistent pass kernel without a GPU fault.

Every wait of the kernel is bounded.  peagle_set_wait_limit shortens the bound to 1 ms and
names one step of the pass whose waits need one completion signal more than the grid can
give, so they run out: the kernel must latch PEAGLE_DEV_TIMEOUT, leave every wait, let its
own loads and tensor-core operations finish, free its tensor memory and return.  The host
sees the bit through peagle_status, which also resets the context's accumulators; the
next normal pass on the same context must match the fp64 oracle again.  Nothing here
faults, traps or hangs the GPU: the wait that runs out is an ordinary bounded spin on a
counter that nothing will raise high enough.
"""
import time

import pytest
import torch

import synth
from pe_helpers import compare, make_ctx, oracle_draft, pk, run_draft, to_dev

pytestmark = pytest.mark.gpu

DIMS = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                  intermediate=320, draft_vocab=1000, target_vocab=1500,
                  rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")
# steps of the two-layer pass: 0 fc, 1 input rows, 2-3 layer-1 QKV halves, 4 attention,
# 5 o-projection, 6 norm, 7 gate/up, 8 down, 9-15 layer 2, 16 final norm, 17 LM head,
# 18 argmax
STEPS = [1, 4, 17]


@pytest.fixture(scope="module")
def case():
    K, lens = 4, [50, 120]
    wl = synth.Workload("f", DIMS, len(lens), K, tuple(lens))
    w = synth.make_weights(DIMS, 77, gains=True)
    inp = synth.make_decode_inputs(wl, 78)
    ctx = make_ctx(DIMS, w, len(lens), K, inp["capacity"] + 1, pass_kernel=True)
    ref = oracle_draft(DIMS, w, inp, K)
    yield ctx, inp, ref, K
    ctx.close()


@pytest.mark.parametrize("step", STEPS)
def test_wait_that_cannot_end_times_out_and_the_context_recovers(case, step):
    ctx, inp, ref, K = case
    m = pk()
    toks, lg, _ = run_draft(ctx, DIMS, inp, K)
    compare(DIMS, ref, toks, lg, f"before the drill (step {step})")
    B = len(inp["seq_lens"])
    d = to_dev(inp)
    kv = m.kv_struct(d["ck"], d["cv"], d["ck"].shape[3], B)
    out = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    m.peagle_set_wait_limit(ctx, 1_000_000, step)
    try:
        t0 = time.perf_counter()
        m.peagle_draft(ctx, B, kv, d["sl"], d["th"], d["nt"], K, out, None)
        rc = m.lib().peagle_status(ctx.handle)
        dt = time.perf_counter() - t0
    finally:
        m.peagle_set_wait_limit(ctx, 0, -1)
    assert rc == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_TIMEOUT
    assert dt < 1.5, f"the drilled pass took {dt:.2f} s"
    # the same context, normal limits: the pass matches the oracle again
    toks, lg, _ = run_draft(ctx, DIMS, inp, K)
    compare(DIMS, ref, toks, lg, f"after the drill (step {step})")
    assert m.peagle_status(ctx) == m.PEAGLE_OK


def test_wait_limit_rejects_a_step_outside_the_pass(case):
    ctx = case[0]
    m = pk()
    with pytest.raises(m.PeagleError) as ei:
        m.peagle_set_wait_limit(ctx, 1000, 10_000)
    assert ei.value.code == m.PEAGLE_ERR_INVALID
