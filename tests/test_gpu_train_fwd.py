"""GPU parity of the training-style parallel-prediction forward (COD-sampled rows, the
flex-attention mask rules) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O
from pe_helpers import LOGIT_TOL, MARGIN, RECORD, make_ctx, pk

pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                        intermediate=320, draft_vocab=1000, target_vocab=1500,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")
SMALL_HD128 = synth.Dims(hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=128,
                         intermediate=384, draft_vocab=777, target_vocab=777,
                         rope_theta=500000.0, rms_eps=1e-5, dtype="bf16", d2t="identity")


def _run_fwd(ctx, dims, tokens, hidden, rp, rd, n, K, logits=True):
    m = pk()
    M = len(rp)
    am = torch.full((M,), -3, dtype=torch.int32, device="cuda")
    lg = torch.full((M, dims.draft_vocab), float("nan"), device="cuda") if logits else None
    m.peagle_forward_parallel(ctx, n, K, torch.from_numpy(tokens).cuda(), hidden.cuda(),
                              torch.from_numpy(rp).cuda(), torch.from_numpy(rd).cuda(), M, am, lg)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    return am.cpu().numpy(), (lg.cpu().numpy() if logits else None)


def _compare(dims, ref_logits, ref_am, ref_margin, am, lg, what):
    tol = LOGIT_TOL[dims.dtype]
    err = float(np.max(np.abs(lg - ref_logits)))
    assert err <= tol, f"{what}: logits max abs err {err:.3e}"
    ok = ref_margin > MARGIN
    RECORD.append({"case": what, "max_abs_err": err, "tol": tol, "logits": int(lg.size),
                   "id_rows_checked": int(ok.sum()), "id_rows": int(ok.size)})
    assert np.array_equal(am[ok], ref_am[ok]), what
    assert np.array_equal(am, np.argmax(lg, axis=-1)), what
    return err


@pytest.mark.parametrize("dims,n,K,r", [
    (synth.DIMS_TINY, 24, 4, 0.8),
    (SMALL_BF16, 40, 8, 0.8),
    (SMALL_HD128, 30, 3, 0.7),
    (SMALL_BF16, 1, 4, 0.8),
    # every depth kept at K = 16: a block's chain-key window spans several 64-key tiles
    (SMALL_BF16, 120, 16, 1.0),
    # several 64-key tiles of depth-1 keys, head_dim 128
    (SMALL_HD128, 150, 8, 0.9),
])
def test_forward_parallel_small(dims, n, K, r):
    m = pk()
    w = synth.make_weights(dims, 17 + n, gains=True)
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 3)
    hidden = synth.normal((n, 3 * dims.hidden), 4, 1.0, dims.torch_dtype)
    u = synth.cod_uniforms(n, K, seed=5)
    rp, rd = m.peagle_cod_rows(n, K, r, u)
    rows = O.cod_retained(n, K, r, u)
    assert np.array_equal(np.stack([rp, rd], 1), rows)
    ctx = make_ctx(dims, w, 1, K, max(n, 8), max_rows=len(rp), max_seq=n)
    am, lg = _run_fwd(ctx, dims, tokens, hidden, rp, rd, n, K)
    ctx.close()
    W = O.Weights64.from_synth(w)
    casts = O.FORWARD_BF16_CASTS if dims.dtype == "bf16" else False
    ref_logits, ref_am, ref_margin = O.forward_parallel(W, dims, tokens, hidden, rows, bf16=casts)
    _compare(dims, ref_logits, ref_am, ref_margin, am, lg, f"fwd n={n} K={K}")


def test_forward_parallel_rejects_bad_rows():
    m = pk()
    dims = synth.DIMS_TINY
    w = synth.make_weights(dims, 2, gains=True)
    n, K = 8, 4
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 3)
    hidden = synth.normal((n, 3 * dims.hidden), 4)
    rp = np.array([0, 1, 1, 2, 2], np.int32)
    rd = np.array([1, 1, 3, 1, 2], np.int32)  # (1,3): anchor -1, and its parent is absent
    ctx = make_ctx(dims, w, 1, K, 16, max_rows=16, max_seq=n)
    M = len(rp)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    m.peagle_forward_parallel(ctx, n, K, torch.from_numpy(tokens).cuda(), hidden.cuda(),
                              torch.from_numpy(rp).cuda(), torch.from_numpy(rd).cuda(), M, am)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_BAD_ROW
    ctx.close()


def test_forward_parallel_dependency_closure():
    """A closed row set that is not a COD set: the dependency closure of a few deep rows
    (depth-1 rows up to their anchors, their chains), inside a longer sequence whose last
    positions have no depth-1 row at all."""
    dims = SMALL_BF16
    n, K = 160, 8
    w = synth.make_weights(dims, 31, gains=True)
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 7)
    hidden = synth.normal((n, 3 * dims.hidden), 8, 1.0, dims.torch_dtype)
    full = np.array([(p, d) for p in range(n) for d in range(1, K + 1) if p - d + 1 >= 0],
                    np.int64)
    targets = np.array([(150, 8), (151, 5), (99, 4), (152, 2)], np.int64)
    clo = O.dependency_closure(full, targets)
    rp = clo[:, 0].astype(np.int32)
    rd = clo[:, 1].astype(np.int32)
    ctx = make_ctx(dims, w, 1, K, n, max_rows=len(rp), max_seq=n)
    am, lg = _run_fwd(ctx, dims, tokens, hidden, rp, rd, n, K)
    ctx.close()
    W = O.Weights64.from_synth(w)
    rl, ra, rm = O.forward_parallel(W, dims, tokens, hidden, clo, bf16=O.FORWARD_BF16_CASTS)
    _compare(dims, rl, ra, rm, am, lg, "fwd dependency closure")


def test_sequence_partitioned_forward_matches_full():
    """Sequence partitioning (3.2): each chunk's rows, run with every depth-1 row below the
    chunk's end as context (one dependency-closed call), match the fp64 oracle's forward on
    the same rows (bf16 logit tolerance, ids where the margin allows), and give the same
    outputs as the unpartitioned GPU forward over all rows."""
    m = pk()
    dims = SMALL_BF16
    n, K, r = 180, 8, 0.8
    w = synth.make_weights(dims, 41, gains=True)
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 9)
    hidden = synth.normal((n, 3 * dims.hidden), 10, 1.0, dims.torch_dtype)
    rp, rd = m.peagle_cod_rows(n, K, r, synth.cod_uniforms(n, K, seed=12))
    bnd = [0, 50, 110, 150]
    chunk = m.peagle_sequence_partition(rp, rd, bnd)
    ctx = make_ctx(dims, w, 1, K, n, max_rows=len(rp), max_seq=n)
    am, lg = _run_fwd(ctx, dims, tokens, hidden, rp, rd, n, K)
    W = O.Weights64.from_synth(w)
    for c in range(len(bnd)):
        end = bnd[c + 1] if c + 1 < len(bnd) else n
        sel = (chunk == c) | ((rd == 1) & (rp < end))
        own = chunk[sel] == c
        am_c, lg_c = _run_fwd(ctx, dims, tokens, hidden, rp[sel], rd[sel], n, K)
        rows_c = np.stack([rp[sel], rd[sel]], 1).astype(np.int64)
        rl, ra, rm = O.forward_parallel(W, dims, tokens, hidden, rows_c,
                                        bf16=O.FORWARD_BF16_CASTS)
        _compare(dims, rl[own], ra[own], rm[own], am_c[own], lg_c[own], f"chunk {c} vs oracle")
        err = float(np.max(np.abs(lg_c[own] - lg[sel][own])))
        assert err < 2e-3, f"chunk {c}: {err:.3e}"
        ok = np.sort(lg[sel][own], axis=1)
        margin = ok[:, -1] - ok[:, -2]
        assert np.array_equal(am_c[own][margin > 1e-2], am[sel][own][margin > 1e-2])
    ctx.close()


def test_forward_parallel_rejects_missing_depth1_row():
    m = pk()
    dims = SMALL_BF16
    w = synth.make_weights(dims, 3, gains=True)
    n, K = 8, 4
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 3)
    hidden = synth.normal((n, 3 * dims.hidden), 4, 1.0, dims.torch_dtype)
    rp = np.array([0, 2, 3], np.int32)  # (2,1) without (1,1)
    rd = np.array([1, 1, 1], np.int32)
    ctx = make_ctx(dims, w, 1, K, 16, max_rows=16, max_seq=n)
    am = torch.empty(3, dtype=torch.int32, device="cuda")
    m.peagle_forward_parallel(ctx, n, K, torch.from_numpy(tokens).cuda(), hidden.cuda(),
                              torch.from_numpy(rp).cuda(), torch.from_numpy(rd).cuda(), 3, am)
    assert m.peagle_status(ctx) == m.PEAGLE_ERR_DEVICE
    assert m.peagle_device_error_bits(ctx) & m.PEAGLE_DEV_BAD_ROW
    ctx.close()


def test_train_fwd_full_prefix_and_tail():
    """The full n=2048, K=8 forward (about 8.5K rows) on the GPU.  The oracle checks (a)
    every row with p < 96 and (b) the last rows of the sequence through their
    dependency closure (all depth-1 rows up to their anchors plus their chains): the
    mask makes both subsets closed, so the oracle's outputs on them are exact."""
    m = pk()
    wl = synth.WORKLOADS["train_fwd"]
    dims = wl.dims
    w = synth.make_weights(dims, 1234, gains=True)
    ti = synth.make_train_inputs(wl, 21)
    n, K = wl.n_seq, wl.K
    rp, rd = m.peagle_cod_rows(n, K, wl.cod_ratio, ti["cod_u"])
    rows = np.stack([rp, rd], 1).astype(np.int64)
    M = len(rp)
    assert abs(M - O.cod_expected_rows(n, K, wl.cod_ratio)) < 400
    ctx = make_ctx(dims, w, 1, K, n, max_rows=M, max_seq=n)
    am, lg = _run_fwd(ctx, dims, ti["tokens"], ti["hidden"], rp, rd, n, K)
    ctx.close()
    W = O.Weights64.from_synth(w, lazy=True)
    pre = rows[rows[:, 0] < 96]
    rl, ra, rm = O.forward_parallel(W, dims, ti["tokens"], ti["hidden"], pre,
                                    bf16=O.FORWARD_BF16_CASTS)
    _compare(dims, rl, ra, rm, am[: len(pre)], lg[: len(pre)], "train_fwd prefix")
    tail = rows[-3:]
    clo = O.dependency_closure(rows, tail)
    cl, ca, cm = O.forward_parallel(W, dims, ti["tokens"], ti["hidden"], clo,
                                    bf16=O.FORWARD_BF16_CASTS)
    idx = {(int(p), int(d)): i for i, (p, d) in enumerate(clo)}
    sel = [idx[(int(p), int(d))] for p, d in tail]
    _compare(dims, cl[sel], ca[sel], cm[sel], am[-3:], lg[-3:], "train_fwd tail")


def test_sequence_partition_workspace_follows_the_chunk():
    """The memory side of sequence partitioning (3.2): a context sized for one chunk's rows
    allocates less device memory for the training forward than one sized for the whole
    sequence, in proportion to the rows (n = 8192, K = 8, COD 0.8: about 34K rows, four
    chunks).  The dense (nK)^2 mask whose size the pages' memory law counts is never
    allocated: the mask is evaluated from its closed form per (row, key)."""
    m = pk()
    dims = SMALL_BF16
    n, K = 8192, 8
    w = synth.make_weights(dims, 5)
    rp, rd = m.peagle_cod_rows(n, K, 0.8, synth.cod_uniforms(n, K, seed=13))
    chunk = m.peagle_sequence_partition(rp, rd, [0, 2048, 4096, 6144])
    rows_chunk = max(int(((chunk == c) | ((rd == 1) & (rp < e))).sum())
                     for c, e in enumerate([2048, 4096, 6144, n]))

    def alloc(max_rows):
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        ctx = make_ctx(dims, w, 1, K, n, max_rows=max_rows, max_seq=n if max_rows else 0)
        torch.cuda.synchronize()
        used = free0 - torch.cuda.mem_get_info()[0]
        ctx.close()
        return used

    base = alloc(0)
    full = alloc(len(rp)) - base
    part = alloc(rows_chunk) - base
    RECORD.append({"case": "partition workspace", "rows_full": len(rp), "rows_chunk": rows_chunk,
                   "bytes_full": full, "bytes_chunk": part,
                   "dense_mask_bytes_full": O.attention_matrix_bytes(n, K),
                   "dense_mask_bytes_chunk": O.attention_matrix_bytes(n // 4, K)})
    assert 0 < part < full
    # linear in the rows (the per-row buffers dominate), far below the dense mask's bytes
    assert part / full < 1.5 * rows_chunk / len(rp)
    assert full < O.attention_matrix_bytes(n, K) / 10
