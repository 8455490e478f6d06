"""Training step (mean cross-entropy over retained rows, every parameter gradient; "P-EAGLE:
Parallel-Drafting EAGLE with Scalable Training", A2 section 2 and section 3) on the GPU
against the fp64 oracle ``peagle_train_step``'s counterpart in oracle/peagle_train_oracle.

Every gradient is compared element by element: |got - want| <= atol + rtol * |want|, with
atol a fraction of the tensor's largest entry (a gradient entry is a sum of many products,
so its rounding error scales with the tensor's magnitude, not with the entry's own, which
may sit near zero after cancellation).  From the arithmetic: fp32 drafters run every
product in fp32 (unit roundoff 2^-24 = 6e-8 per operation; sums over up to a few
thousand rows): rtol 1e-4, atol 1e-5 of the largest entry.  bf16 drafters' products round
their operands to at most 11 significant bits (TF32; 2^-11 = 4.9e-4 per operand, chained
through the backward's few dependent products): rtol 2e-2, atol 2e-3 of the largest entry,
and 1e-3 on the loss.  A wrong block of entries (one key tile's dK, one chunk's rows)
exceeds these bounds by orders of magnitude."""
import numpy as np
import pytest
import torch

import synth
from oracle import peagle_oracle as O
from oracle import peagle_train_oracle as T
from pe_helpers import make_ctx, pk

pytestmark = pytest.mark.gpu

SMALL_BF16 = synth.Dims(hidden=192, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=64,
                        intermediate=320, draft_vocab=1000, target_vocab=1500,
                        rope_theta=10000.0, rms_eps=1e-5, dtype="bf16", d2t="monotone")


def _weights(dims, seed):
    """Synthetic weights with norm gains, emb(mask) and h_shared away from their initial
    values (a unit gain would hide a missing factor)."""
    w = synth.make_weights(dims, seed)
    g = torch.Generator().manual_seed(seed)
    dt = w["fc"].dtype
    for k in ("input_norm", "hidden_norm", "final_norm"):
        w[k] = (1.0 + 0.3 * torch.randn(dims.hidden, generator=g)).to(dt)
    for L in w["layers"]:
        for k in ("attn_norm", "post_norm"):
            L[k] = (1.0 + 0.3 * torch.randn(dims.hidden, generator=g)).to(dt)
    return w


def _grad_buffers(dims):
    H, I, nq, nkv, hd = (dims.hidden, dims.intermediate, dims.n_q_heads, dims.n_kv_heads,
                         dims.head_dim)
    z = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device="cuda")  # noqa: E731
    q = (nq + 2 * nkv) * hd
    return {"embed": z(dims.target_vocab, H), "emb_mask": z(H), "h_shared": z(3 * H),
            "fc": z(H, 3 * H), "input_norm": z(H), "hidden_norm": z(H), "final_norm": z(H),
            "lm_head": z(dims.draft_vocab, H),
            "qkv": [z(q, 2 * H if l == 0 else H) for l in range(dims.n_layers)],
            "o": [z(H, nq * hd) for _ in range(dims.n_layers)],
            "attn_norm": [z(H) for _ in range(dims.n_layers)],
            "post_norm": [z(H) for _ in range(dims.n_layers)],
            "gate": [z(I, H) for _ in range(dims.n_layers)],
            "up": [z(I, H) for _ in range(dims.n_layers)],
            "down": [z(H, I) for _ in range(dims.n_layers)]}


def _run(dims, seed, n, K, cod):
    w = _weights(dims, seed)
    rng = np.random.default_rng(seed)
    tokens = rng.integers(0, dims.target_vocab, n).astype(np.int32)
    hidden = synth.normal((n, 3 * dims.hidden), np.random.SeedSequence(seed + 1), 1.0,
                          dims.torch_dtype)
    u = rng.random((n, K)) if cod else np.zeros((n, K))
    rp, rd = pk().peagle_cod_rows(n, K, cod if cod else 1.0, u)
    M = len(rp)
    labels = rng.integers(0, dims.draft_vocab, M).astype(np.int32)
    m = pk()
    ctx = make_ctx(dims, w, 1, K, n + 8, max_rows=M, max_seq=n, train=True)
    g = _grad_buffers(dims)
    loss = torch.full((1,), float("nan"), device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    m.peagle_train_step(ctx, n, K, dev(tokens), hidden.cuda(), dev(rp), dev(rd), M, dev(labels),
                        loss, g)
    torch.cuda.synchronize()
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    ctx.close()
    W = O.Weights64.from_synth(w)
    W.embed = O.to64(W.embed)
    rows = np.stack([rp, rd], 1).astype(np.int64)
    ref_loss, _, ref = T.train_step(W, dims, tokens, O.to64(hidden), rows, labels)
    return float(loss.item()), g, ref_loss, ref


def _flat(g, ref, n_layers):
    for k in ("embed", "emb_mask", "h_shared", "fc", "input_norm", "hidden_norm", "final_norm",
              "lm_head"):
        yield k, g[k], ref[k]
    for l in range(n_layers):
        for k in ("qkv", "o", "attn_norm", "post_norm", "gate", "up", "down"):
            yield f"layers.{l}.{k}", g[k][l], ref["layers"][l][k]


GRAD_RECORD = []  # (case, tensor, worst |got - want| / (atol + rtol |want|))


def _compare(dims, out, rtol, atol_frac, loss_tol, case=""):
    loss, g, ref_loss, ref = out
    assert abs(loss - ref_loss) <= loss_tol * abs(ref_loss), (loss, ref_loss)
    for name, got, want in _flat(g, ref, dims.n_layers):
        got = got.cpu().double().numpy()
        assert np.all(np.isfinite(got)), name
        scale = float(np.max(np.abs(want))) if want.size else 0.0
        if scale == 0.0:
            assert np.all(got == 0), name
            continue
        bound = atol_frac * scale + rtol * np.abs(want)
        ratio = np.abs(got - want) / bound
        worst = float(ratio.max())
        GRAD_RECORD.append((case, name, worst))
        bad = np.argwhere(ratio > 1.0)
        assert len(bad) == 0, (f"{case} {name}: {len(bad)} of {ratio.size} entries outside "
                               f"the bound, worst ratio {worst:.2f} at {bad[0].tolist()}")


@pytest.mark.parametrize("n,K,cod", [(24, 4, 0.8), (16, 1, None), (12, 8, None)])
def test_tiny_f32_train_step(n, K, cod):
    dims = synth.DIMS_TINY
    _compare(dims, _run(dims, 3 + K, n, K, cod), 1e-4, 1e-5, 1e-5, f"f32 n={n} K={K}")


# SMALL_BF16 has three q heads per kv head: the TF32 mma.sync prefix-attention kernels.
# (n=40, K=8) and (33, 3) fit one 64-key tile and one 512-row chunk of them; (220, 8, 0.8)
# has four tiles of depth-1 keys and about 900 rows (two chunks of the key-major kernel,
# its double-buffered loop), so every tiling path is compared
@pytest.mark.parametrize("n,K,cod", [(40, 8, 0.8), (33, 3, 0.6), (220, 8, 0.8)])
def test_small_bf16_train_step(n, K, cod):
    dims = SMALL_BF16
    _compare(dims, _run(dims, 7 + K, n, K, cod), 2e-2, 2e-3, 1e-3, f"bf16 n={n} K={K}")


# bf16 drafters whose q heads per kv head (G) take the tcgen05 prefix-attention kernels
# (head_dim 64, G in {1, 2, 4, 8}): 128 MMA rows per CTA = 128 / G query rows x G heads
TC_DIMS = {
    g: synth.Dims(hidden=256, n_layers=2, n_q_heads=2 * g, n_kv_heads=2, head_dim=64,
                  intermediate=384, draft_vocab=1000, target_vocab=1500, rope_theta=10000.0,
                  rms_eps=1e-5, dtype="bf16", d2t="monotone")
    for g in (1, 2, 4, 8)
}


# (220, 8, 0.8): about 900 rows, seven 32-key tiles of depth-1 keys (the last one ragged),
# two 128-key blocks and two 512-row chunks of the key-major backward, row blocks of
# 128 / G rows with a ragged last one; (40, 4, 0.8) fits one key tile
@pytest.mark.parametrize("G,n,K,cod", [(8, 220, 8, 0.8), (4, 220, 8, 0.8), (2, 220, 8, 0.8),
                                       (1, 220, 8, 0.8), (8, 40, 4, 0.8)])
def test_bf16_train_step_tcgen05_attention(G, n, K, cod):
    dims = TC_DIMS[G]
    _compare(dims, _run(dims, 31 + G + K, n, K, cod), 2e-2, 2e-3, 1e-3,
             f"bf16 tcgen05 attention G={G} n={n} K={K}")


def test_train_step_needs_training_workspaces():
    """A windowed drafter cannot hold the training workspaces (UNSUPPORTED at create), and
    a context made without them refuses the step (CAPACITY) instead of allocating."""
    m = pk()
    dims = synth.shrink(SMALL_BF16, attn_window=8)
    w = synth.make_weights(dims, 1)
    with pytest.raises(m.PeagleError) as e:
        make_ctx(dims, w, 1, 2, 32, max_rows=16, max_seq=8, train=True)
    assert e.value.code == m.PEAGLE_ERR_UNSUPPORTED
    dims = SMALL_BF16
    w = synth.make_weights(dims, 1)
    ctx = make_ctx(dims, w, 1, 2, 32, max_rows=16, max_seq=8)
    z = torch.zeros(16, dtype=torch.int32, device="cuda")
    g = _grad_buffers(dims)
    loss = torch.zeros(1, device="cuda")
    with pytest.raises(m.PeagleError) as e:
        m.peagle_train_step(ctx, 8, 2, z, torch.zeros(8, 3 * dims.hidden, device="cuda",
                                                      dtype=torch.bfloat16),
                            z, z, 8, z, loss, g)
    assert e.value.code == m.PEAGLE_ERR_CAPACITY
    ctx.close()


def test_train_step_loss_at_full_size_is_the_forward_cross_entropy():
    """The training workload (decode drafter, n = 2048, K = 8, COD 0.8; 8,407 rows): the
    step's loss equals the mean cross-entropy of the bf16 training forward's logits on the
    same rows (two independent paths: TF32 fp32-activation GEMMs against tcgen05 bf16 hi/lo
    GEMMs), and every gradient is finite."""
    m = pk()
    wl = synth.WORKLOADS["train_fwd"]
    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    ti = synth.make_train_inputs(wl, 21)
    n, K = wl.n_seq, wl.K
    rp, rd = m.peagle_cod_rows(n, K, wl.cod_ratio, ti["cod_u"])
    M = len(rp)
    labels = np.random.default_rng(5).integers(0, dims.draft_vocab, M).astype(np.int32)
    ctx = make_ctx(dims, w, 1, K, n, max_rows=M, max_seq=n, train=True)
    del w
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    tok, hid, rpd, rdd, lab = dev(ti["tokens"]), ti["hidden"].cuda(), dev(rp), dev(rd), dev(labels)
    lg = torch.empty(M, dims.draft_vocab, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    m.peagle_forward_parallel(ctx, n, K, tok, hid, rpd, rdd, M, am, lg)
    ce = (torch.logsumexp(lg.double(), 1) - lg.double()[torch.arange(M), lab.long()]).mean()
    g = _grad_buffers(dims)
    g["embed"] = None
    loss = torch.zeros(1, device="cuda")
    m.peagle_train_step(ctx, n, K, tok, hid, rpd, rdd, M, lab, loss, g)
    torch.cuda.synchronize()
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    ctx.close()
    assert abs(loss.item() - ce.item()) <= 1e-3 * abs(ce.item()), (loss.item(), ce.item())
    for name, t in g.items():
        for x in (t if isinstance(t, list) else [t]):
            if x is not None:
                assert torch.isfinite(x).all(), name


def test_train_step_flags_rows_outside_the_contract():
    """A row set that is not closed under the mask's dependencies (a depth-1 row missing)
    and a label outside the vocabulary are reported through the device error word; the
    calls complete with finite gradients, and a valid call afterwards is clean."""
    m = pk()
    dims = synth.DIMS_TINY
    w = synth.make_weights(dims, 2)
    n, K = 8, 3
    rp, rd = m.peagle_cod_rows(n, K, 1.0, np.zeros((n, K)))
    ctx = make_ctx(dims, w, 1, K, n + 8, max_rows=len(rp), max_seq=n, train=True)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    tok = dev(np.arange(n, dtype=np.int32))
    hid = torch.randn(n, 3 * dims.hidden, device="cuda")

    def run(p, d, labels):
        g = _grad_buffers(dims)
        loss = torch.zeros(1, device="cuda")
        m.peagle_train_step(ctx, n, K, tok, hid, dev(p), dev(d), len(p), dev(labels), loss, g)
        st = m.peagle_status(ctx)
        bits = m.peagle_device_error_bits(ctx)
        assert np.isfinite(loss.item())
        for t in g.values():
            for x in (t if isinstance(t, list) else [t]):
                assert torch.isfinite(x).all()
        return st, bits

    keep = ~((rp == 4) & (rd == 1))  # (5, 1) then misses its dependency (4, 1)
    st, bits = run(rp[keep], rd[keep], np.zeros(int(keep.sum()), np.int32))
    assert st == m.PEAGLE_ERR_DEVICE and bits & m.PEAGLE_DEV_BAD_ROW
    lab = np.zeros(len(rp), np.int32)
    lab[3] = dims.draft_vocab
    st, bits = run(rp, rd, lab)
    assert st == m.PEAGLE_ERR_DEVICE and bits & m.PEAGLE_DEV_BAD_TOKEN
    assert run(rp, rd, np.zeros(len(rp), np.int32))[0] == m.PEAGLE_OK
    ctx.close()
