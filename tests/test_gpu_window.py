"""Sliding-window drafter attention ("EAGLE-4", "EAGLE-4 overview": the drafter attends to
the most recent positions only) on the GPU against the fp64 oracle: the fp32 path, the
bf16 pass kernel and the bf16 multi-kernel path, windows shorter than, straddling and
longer than the context."""
import numpy as np
import pytest

import synth
from pe_helpers import compare, make_ctx, oracle_draft, run_draft

pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                        intermediate=320, draft_vocab=1000, target_vocab=1500,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")


def _case(dims, lens, K, seed, cap=None):
    wl = synth.Workload("w", dims, len(lens), K, tuple(lens))
    w = synth.make_weights(dims, seed, gains=True)
    inp = synth.make_decode_inputs(wl, seed + 1, capacity=cap)
    return w, inp


@pytest.mark.parametrize("window", [1, 5, 40, 130])
def test_tiny_f32_window(window):
    dims = synth.shrink(synth.DIMS_TINY, attn_window=window)
    w, inp = _case(dims, [0, 3, 100], 4, 61)
    ctx = make_ctx(dims, w, 3, 4, inp["capacity"] + 1)
    toks, lg, _ = run_draft(ctx, dims, inp, 4)
    ref = oracle_draft(dims, w, inp, 4)
    compare(dims, ref, toks, lg, f"tiny f32 window {window}")
    ctx.close()


@pytest.mark.parametrize("pass_kernel", [True, False])
@pytest.mark.parametrize("window,lens,K", [
    (64, [300, 20, 700], 5),   # windows inside long contexts, one context shorter
    (1, [129, 3], 8),          # each row sees only itself
    (200, [150, 199, 260], 3), # windows straddling the cache / draft-block boundary
])
def test_small_bf16_window(pass_kernel, window, lens, K):
    dims = synth.shrink(SMALL_BF16, attn_window=window)
    w, inp = _case(dims, lens, K, 17 + window + K)
    ctx = make_ctx(dims, w, len(lens), K, inp["capacity"] + 1, pass_kernel=pass_kernel)
    toks, lg, _ = run_draft(ctx, dims, inp, K)
    ref = oracle_draft(dims, w, inp, K)
    compare(dims, ref, toks, lg, f"small bf16 window {window} {lens} K={K} "
                                 f"{'pass' if pass_kernel else 'multi'}")
    ctx.close()


def test_window_longer_than_context_is_full_attention():
    """A window covering every context gives the same logits as no window, bit for bit
    (the items cover the same keys in the same order)."""
    lens, K = [90, 33], 6
    full = SMALL_BF16
    w, inp = _case(full, lens, K, 5)
    out = []
    for dims in (full, synth.shrink(full, attn_window=97)):
        ctx = make_ctx(dims, w, 2, K, inp["capacity"] + 1)
        _, lg, _ = run_draft(ctx, dims, inp, K)
        out.append(lg)
        ctx.close()
    assert np.array_equal(out[0], out[1])


def test_forward_parallel_rejects_a_window():
    import drafting_eagle_draft_gb300 as m
    import torch

    dims = synth.shrink(SMALL_BF16, attn_window=16)
    w = synth.make_weights(dims, 3, gains=True)
    ctx = make_ctx(dims, w, 1, 4, 64, max_rows=64, max_seq=16)
    n, K = 8, 2
    rp, rd = m.peagle_cod_rows(n, K, 1.0, np.zeros((n, K)))
    tok = torch.zeros(n, dtype=torch.int32, device="cuda")
    hid = torch.zeros(n, 3 * dims.hidden, dtype=torch.bfloat16, device="cuda")
    am = torch.empty(len(rp), dtype=torch.int32, device="cuda")
    with pytest.raises(m.PeagleError) as e:
        m.peagle_forward_parallel(ctx, n, K, tok, hid, torch.from_numpy(rp).cuda(),
                                  torch.from_numpy(rd).cuda(), len(rp), am, None)
    assert e.value.code == m.PEAGLE_ERR_UNSUPPORTED
    ctx.close()


def test_decode_b2_full_size_window_4096():
    """The full-size drafter of the decode workloads with a 4096-position window on the
    concurrency-2 contexts (8192 and 10240 cached positions, K = 8): the pass kernel's
    logits and ids against the fp64 oracle's windowed attention."""
    wl = synth.WORKLOADS["decode_b2"]
    dims = synth.shrink(wl.dims, attn_window=4096)
    w = synth.make_weights(dims, 1234, gains=True)
    inp = synth.make_decode_inputs(wl, 98)
    ctx = make_ctx(dims, w, wl.batch, wl.K, inp["capacity"] + 1)
    toks, lg, _ = run_draft(ctx, dims, inp, wl.K)
    ctx.close()
    ref = oracle_draft(dims, w, inp, wl.K)
    compare(dims, ref, toks, lg, "decode_b2 window 4096")
