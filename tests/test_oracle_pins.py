"""Pins of the fp64 oracle against what the pages and mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a value printed on
the pages (tests/golden/*), a closed form, a library routine, an exhaustive
enumeration, or an invariant of the method, chosen so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import synth
from oracle import peagle_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _tiny_dims(**kw):
    base = synth.Dims(hidden=16, n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=8,
                      intermediate=24, draft_vocab=50, target_vocab=60, rope_theta=10000.0,
                      rms_eps=1e-6, dtype="f32", d2t="identity")
    return synth.shrink(base, **kw)


def _tiny_weights(dims, seed=3, d2t=None):
    w = synth.make_weights(dims, seed)
    if d2t is not None:
        w["d2t"] = d2t
    return w


def _tiny_inputs(dims, B, K, L, seed=4):
    wl = synth.Workload("t", dims, B, K, tuple([L] * B))
    return synth.make_decode_inputs(wl, seed)


# ---------------------------------------------------------------- scalar helpers


def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),  # fp32/bf16 subnormals
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0, 65504.0,
                  3.0e38], np.float32),  # exact ties go to even
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 33))
    y = O.rmsnorm(x, np.ones(33), 0.0)
    assert np.allclose(np.sqrt((y * y).mean(-1)), 1.0, atol=1e-12)
    assert np.allclose(O.rmsnorm(7.5 * x, np.ones(33), 0.0), y, atol=1e-12)
    g = rng.standard_normal(33)
    assert np.allclose(O.rmsnorm(x, g, 0.0), y * g, atol=1e-12)


def test_rope_is_complex_rotation():
    """Rotate-half RoPE equals multiplying (x_i + i x_{i+hd/2}) by exp(i pos theta_i)."""
    rng = np.random.default_rng(2)
    hd, theta = 16, 10000.0
    x = rng.standard_normal((6, hd))
    pos = np.array([0, 1, 5, 100, 4097, 10239])
    got = O.rope(x, pos, theta)
    half = hd // 2
    freq = np.array([theta ** (-2.0 * i / hd) for i in range(half)])
    z = (x[:, :half] + 1j * x[:, half:]) * np.exp(1j * pos[:, None] * freq[None, :])
    ref = np.concatenate([z.real, z.imag], axis=1)
    assert np.allclose(got, ref, atol=1e-12)
    assert np.allclose(O.rope(x, np.zeros(6, int), theta), x)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    s1 = O.rope(q, np.array(10), 1e4) @ O.rope(k, np.array(3), 1e4)
    s2 = O.rope(q, np.array(1010), 1e4) @ O.rope(k, np.array(1003), 1e4)
    assert abs(s1 - s2) < 1e-9


def test_attend_closed_forms():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(8)
    v = rng.standard_normal((5, 8))
    k1 = rng.standard_normal((1, 8))
    assert np.allclose(O.attend(q, k1, v[:1], 0.3), v[0])
    keq = np.repeat(k1, 5, axis=0)
    assert np.allclose(O.attend(q, keq, v, 0.3), v.mean(0))
    k2 = rng.standard_normal((2, 8))
    s = 0.35
    p1 = scipy.special.expit((q @ k2[1] - q @ k2[0]) * s)
    assert np.allclose(O.attend(q, k2, v[:2], s), (1 - p1) * v[0] + p1 * v[1])


# ---------------------------------------------------------------- verification


def test_verify_greedy_exhaustive_small_vocab():
    """All (draft, target) pairs over a 3-token vocabulary, K <= 3 (K=4 sampled)."""
    for K in (1, 2, 3):
        for draft in itertools.product(range(3), repeat=K):
            for tgt in itertools.product(range(3), repeat=K + 1):
                acc, bonus = O.verify_greedy(np.array([draft]), np.array([tgt]))
                agree = list(itertools.takewhile(lambda t: t[0] == t[1], zip(draft, tgt)))
                m = len(agree)
                assert acc[0] == m and bonus[0] == tgt[m]
                emitted = list(draft[:m]) + [tgt[m]]
                # the emitted tokens are exactly the target's greedy choices
                assert emitted == list(tgt[: m + 1])
    rng = np.random.default_rng(5)
    d = rng.integers(0, 3, (4000, 4))
    t = rng.integers(0, 3, (4000, 5))
    acc, bonus = O.verify_greedy(d, t)
    for b in range(4000):
        m = next((i for i in range(4) if d[b, i] != t[b, i]), 4)
        assert acc[b] == m and bonus[b] == t[b, m]


def _table():
    rows = []
    with open(os.path.join(GOLD, "acceptance_table.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            rows.append((parts[0], [float(x) / 100 for x in parts[1:8]], float(parts[8])))
    return rows


def test_acceptance_length_counts_bonus_token():
    """Mean acceptance length = 1 + sum of per-position rates (table in "Example model").
    Distributions built from each row's rates must reproduce its printed average."""
    rows = _table()
    assert len(rows) == 10
    for name, rates, avg in rows:
        assert abs(1 + sum(rates) - avg) <= 0.0051, name
        # realise an accept-length sample with exactly these per-position rates
        n = 100000
        counts = np.round(np.array(rates + [0.0]) * n).astype(int)
        m = np.concatenate([np.full(counts[k - 1] - counts[k], k) for k in range(1, 8)]
                           + [np.zeros(n - counts[0], int)])
        got_rates, got_avg = O.acceptance_stats(m, 7)
        assert np.allclose(got_rates, rates, atol=1e-5)
        assert abs(got_avg - avg) <= 0.0051, name


# ---------------------------------------------------------------- COD and mask


def _paper_numbers():
    out = {}
    with open(os.path.join(GOLD, "paper_numbers.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v, tol = line.split()
            out[k] = (float(v), float(tol))
    return out


def test_attention_matrix_closed_form():
    nums = _paper_numbers()
    assert 8192 * 8 == nums["positions_8192_K8"][0]
    b = O.attention_matrix_bytes(8192, 8, 2)
    assert b == 8 * 2 ** 30
    v, tol = nums["attn_matrix_bf16_GB"]
    assert abs(b / 1e9 - v) <= tol + 0.6  # 8 GiB = 8.59 GB, "about 8 GB"


def test_cod_expected_count_matches_paper():
    nums = _paper_numbers()
    e = O.cod_expected_rows(8192, 8, 0.8)
    v, tol = nums["cod_rows_8192_K8_r08"]
    assert abs(e - v) <= tol
    # geometric shares per depth ("COD sampling": 0.7 then 0.49)
    n = 20000
    u = synth.cod_uniforms(n, 3, seed=8)
    rows = O.cod_retained(n, 3, 0.7, u)
    share = [np.mean(rows[:, 1] == d) * 0 + (rows[:, 1] == d).sum() / n for d in (1, 2, 3)]
    assert share[0] == 1.0
    assert abs(share[1] - nums["cod_share_depth2_r07"][0]) < 0.015
    assert abs(share[2] - nums["cod_share_depth3_r07"][0]) < 0.015


def test_cod_seeded_mean_and_closure():
    n, K, r = 2048, 8, 0.8
    counts = []
    for seed in range(12):
        rows = O.cod_retained(n, K, r, synth.cod_uniforms(n, K, seed=100 + seed))
        counts.append(len(rows))
        kept = {(int(p), int(d)) for p, d in rows}
        for p, d in rows:  # dependency closure
            if d >= 2:
                assert (int(p) - 1, int(d) - 1) in kept
        assert all((p, 1) in kept for p in range(n))
        # p-major ordering
        key = rows[:, 0] * (K + 1) + rows[:, 1]
        assert np.all(np.diff(key) > 0)
    e = O.cod_expected_rows(n, K, r)
    # variance bound: each row is Bernoulli, so sd <= sqrt(sum of rows) ; 12 seeds
    sd = math.sqrt(e) / math.sqrt(len(counts))
    assert abs(np.mean(counts) - e) < 4 * sd
    assert abs(e - 8512.1) < 0.1


def test_mask_rules_from_the_page_example():
    """Flex-attention mask example: depth 2 (0-based) at anchor 5 -> 1-based (p=7, d=3)."""
    p, d = 7, 3
    assert O.mask_allowed(p, d, 6, 2)  # depth-1 (0-based) at the same anchor
    assert O.mask_allowed(p, d, 5, 1)  # depth-0 at the same anchor
    assert O.mask_allowed(p, d, p, d)  # itself
    assert not O.mask_allowed(p, d, 4, 2)  # rollout anchored at 3
    assert not O.mask_allowed(p, d, 5, 3)  # rollout anchored at 3
    assert not O.mask_allowed(p, d, 6, 1)  # base context beyond the anchor (forward)
    assert not O.mask_allowed(p, d, 8, 4)  # later depth of the same rollout
    for p2 in range(0, 6):
        assert O.mask_allowed(p, d, p2, 1)  # all base context up to the anchor


def test_mask_depth1_is_causal_and_nothing_sideways():
    n, K = 9, 4
    M = O.full_mask(n, K)
    idx = [(p, d) for p in range(n) for d in range(1, K + 1)]
    d1 = [i for i, (p, d) in enumerate(idx) if d == 1]
    sub = M[np.ix_(d1, d1)]
    assert np.array_equal(sub, np.tril(np.ones((n, n), bool)))
    for i, (p, d) in enumerate(idx):
        assert M[i, i]
        for j, (p2, d2) in enumerate(idx):
            if M[i, j]:
                assert p2 <= p  # never forward
                if d2 >= 2:
                    assert p2 - d2 == p - d  # same rollout (no sideways)


@pytest.mark.parametrize("n", [1, 7, 12])
def test_amortized_mask_is_top_left_slice(n):
    """3.1 amortized mask: the (nK)^2 top-left block of the max-length mask equals
    the mask built directly for length n (p-major order), also after row selection."""
    K, nmax = 4, 16
    Mmax = O.full_mask(nmax, K)
    direct = O.full_mask(n, K)
    assert np.array_equal(O.amortized_mask(Mmax, n, K), direct)
    rows = O.cod_retained(n, K, 0.8, synth.cod_uniforms(n, K, seed=n))
    sel = O.amortized_mask(Mmax, n, K, rows)
    for i, (p, d) in enumerate(rows):
        for j, (p2, d2) in enumerate(rows):
            assert sel[i, j] == O.mask_allowed(p, d, p2, d2)


def test_sequence_partition_keeps_dependencies():
    """3.2: every mask dependency of a row lies in its own chunk or in the chunk's
    depth-1 context, and depth >= 3 rows share their parent's chunk."""
    n, K = 64, 8
    rows = O.cod_retained(n, K, 0.8, synth.cod_uniforms(n, K, seed=9))
    chunk, ctx = O.sequence_partition(rows, [0, 16, 32, 48])
    idx = {(int(p), int(d)): i for i, (p, d) in enumerate(rows)}
    for i, (p, d) in enumerate(rows):
        if d >= 3:
            assert chunk[i] == chunk[idx[(int(p) - 1, int(d) - 1)]]
        c = chunk[i]
        for j, (p2, d2) in enumerate(rows):
            if O.mask_allowed(p, d, p2, d2):
                ok = chunk[j] == c or (d2 == 1 and p2 in set(ctx[c].tolist()))
                assert ok, ((p, d), (p2, d2))
    sizes = np.bincount(chunk)
    assert sizes.min() > 0


def test_sequence_partition_depth2_goes_by_index():
    """3.2: depths 1 and 2 (the paper's depths 0 and 1) are assigned by position index.
    A depth-2 row at a chunk's first position has its parent (p-1, 1) in the previous
    chunk, yet lands in its own position's chunk; the depth-3 row below it follows it
    there, while a depth-3 row at the boundary follows its depth-2 parent back into the
    previous chunk."""
    n, K = 12, 4
    rows = np.array([(p, d) for p in range(n) for d in range(1, K + 1) if p - d + 1 >= 0])
    b = 6
    chunk, ctx = O.sequence_partition(rows, [0, b])
    idx = {(int(p), int(d)): i for i, (p, d) in enumerate(rows)}
    assert chunk[idx[(b - 1, 1)]] == 0 and chunk[idx[(b, 1)]] == 1
    assert chunk[idx[(b, 2)]] == 1          # parent (b-1, 1) is in chunk 0
    assert chunk[idx[(b + 1, 3)]] == 1      # follows its parent (b, 2)
    assert chunk[idx[(b, 3)]] == 0          # follows its parent (b-1, 2)
    assert chunk[idx[(b + 1, 4)]] == 0      # chain (b-1, 2) -> (b, 3) -> (b+1, 4)
    assert chunk[idx[(b - 1, 2)]] == 0
    # chunk 1's context: every depth-1 position below its end
    assert ctx[1].tolist() == list(range(n))
    assert ctx[0].tolist() == list(range(b))


# ---------------------------------------------------------------- the draft pass


def _zero(t):
    return torch.zeros_like(t)


def _run(dims, w, inp, K, bf16=False):
    W = O.Weights64.from_synth(w)
    return O.draft_pass(W, dims, inp["cache_k"], inp["cache_v"], inp["seq_lens"],
                        inp["target_hidden"], inp["new_token"], K, bf16=bf16)


def _rms(x):
    return x / np.sqrt((x * x).mean(-1, keepdims=True))


def test_pass_without_layers_reduces_to_fc_norm_head():
    """With o-proj and down-proj zeroed, the residual stays at f = fc(h): logits are
    lm_head(RMSNorm(fc(h_context))) for the NTP row and lm_head(RMSNorm(fc(h_shared)))
    for the MTP rows; tokens are argmax + d2t."""
    dims = _tiny_dims(n_layers=2, rms_eps=0.0, target_vocab=200, d2t="monotone")
    w = _tiny_weights(dims)
    for L in w["layers"]:
        L["o"] = _zero(L["o"])
        L["down"] = _zero(L["down"])
    B, K = 2, 3
    inp = _tiny_inputs(dims, B, K, 5)
    r = _run(dims, w, inp, K)
    fc = w["fc"].double().numpy()
    lm = w["lm_head"].double().numpy()
    th = inp["target_hidden"].double().numpy()
    hs = w["h_shared"].double().numpy()
    d2t = np.asarray(w["d2t"])
    for b in range(B):
        exp0 = lm @ _rms(fc @ th[b])
        expm = lm @ _rms(fc @ hs)
        assert np.allclose(r.logits[b, 0], exp0, atol=1e-10)
        for j in range(1, K):
            assert np.allclose(r.logits[b, j], expm, atol=1e-10)
        for j in range(K):
            a = int(np.argmax(r.logits[b, j]))
            assert r.tokens[b, j] == a + d2t[a]
    assert np.all(np.diff(np.arange(dims.draft_vocab) + d2t) > 0)


def test_single_key_attention_reduces_to_value_projection():
    """No cache and K=1: the only visible key is the row's own, so attention returns
    its value; with down-proj zeroed the residual is f + W_o(v per q-head's kv head),
    v = W_v x0 and x0 = [RMSNorm(emb(new)) || RMSNorm(f)]."""
    dims = _tiny_dims(rms_eps=0.0)
    w = _tiny_weights(dims)
    w["layers"][0]["down"] = _zero(w["layers"][0]["down"])
    inp = _tiny_inputs(dims, 1, 1, 0)
    r = _run(dims, w, inp, 1)
    H, nq, nkv, hd = dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    e = w["embed"][int(inp["new_token"][0])].double().numpy()
    f = w["fc"].double().numpy() @ inp["target_hidden"][0].double().numpy()
    x0 = np.concatenate([_rms(e), _rms(f)])
    wv = w["layers"][0]["qkv"].double().numpy()[(nq + nkv) * hd:]
    v = (wv @ x0).reshape(nkv, hd)
    o = np.concatenate([v[h // (nq // nkv)] for h in range(nq)])
    res = f + w["layers"][0]["o"].double().numpy() @ o
    exp = w["lm_head"].double().numpy() @ _rms(res)
    assert np.allclose(r.logits[0, 0], exp, atol=1e-10)


def test_uniform_scores_average_visible_values():
    """Zero keys everywhere give uniform softmax: row j averages the values of the L
    cached positions and draft rows 0..j of its kv head (causal draft block)."""
    dims = _tiny_dims(rms_eps=0.0)
    w = _tiny_weights(dims)
    H, nq, nkv, hd = dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    w["layers"][0]["qkv"][nq * hd:(nq + nkv) * hd] = 0
    w["layers"][0]["down"] = _zero(w["layers"][0]["down"])
    B, K, L = 2, 4, 6
    inp = _tiny_inputs(dims, B, K, L)
    inp["cache_k"] = _zero(inp["cache_k"])
    r = _run(dims, w, inp, K)
    cv = inp["cache_v"].double().numpy()[0]
    wv = w["layers"][0]["qkv"].double().numpy()[(nq + nkv) * hd:]
    fc = w["fc"].double().numpy()
    for b in range(B):
        xs = []
        for j in range(K):
            e = (w["embed"][int(inp["new_token"][b])] if j == 0 else w["emb_mask"]).double().numpy()
            f = fc @ (inp["target_hidden"][b] if j == 0 else w["h_shared"]).double().numpy()
            xs.append((f, np.concatenate([_rms(e), _rms(f)])))
        vd = np.stack([(wv @ x0).reshape(nkv, hd) for _, x0 in xs])  # [K, nkv, hd]
        for j in range(K):
            o = []
            for h in range(nq):
                g = h // (nq // nkv)
                vals = np.concatenate([cv[b, g, :L], vd[: j + 1, g]], axis=0)
                o.append(vals.mean(0))
            res = xs[j][0] + w["layers"][0]["o"].double().numpy() @ np.concatenate(o)
            exp = w["lm_head"].double().numpy() @ _rms(res)
            assert np.allclose(r.logits[b, j], exp, atol=1e-10)


def test_two_key_attention_scale_and_rope():
    """One cached key c and a zero draft key: the NTP row's weight on c is
    sigmoid(rope(q, L) . c / sqrt(hd)) (rope via complex rotation)."""
    dims = _tiny_dims(rms_eps=0.0)
    w = _tiny_weights(dims)
    H, nq, nkv, hd = dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    w["layers"][0]["qkv"][nq * hd:(nq + nkv) * hd] = 0
    w["layers"][0]["down"] = _zero(w["layers"][0]["down"])
    L = 1
    inp = _tiny_inputs(dims, 1, 1, L)
    r = _run(dims, w, inp, 1)
    ck = inp["cache_k"].double().numpy()[0, 0]
    cv = inp["cache_v"].double().numpy()[0, 0]
    e = w["embed"][int(inp["new_token"][0])].double().numpy()
    f = w["fc"].double().numpy() @ inp["target_hidden"][0].double().numpy()
    x0 = np.concatenate([_rms(e), _rms(f)])
    Wq = w["layers"][0]["qkv"].double().numpy()[: nq * hd]
    Wv = w["layers"][0]["qkv"].double().numpy()[(nq + nkv) * hd:]
    q = (Wq @ x0).reshape(nq, hd)
    half = hd // 2
    freq = np.array([dims.rope_theta ** (-2.0 * i / hd) for i in range(half)])
    z = (q[:, :half] + 1j * q[:, half:]) * np.exp(1j * L * freq)
    qr = np.concatenate([z.real, z.imag], axis=1)
    vd = (Wv @ x0).reshape(nkv, hd)
    o = []
    for h in range(nq):
        g = h // (nq // nkv)
        pc = scipy.special.expit(qr[h] @ ck[g, 0] / math.sqrt(hd))
        o.append(pc * cv[g, 0] + (1 - pc) * vd[g])
    res = f + w["layers"][0]["o"].double().numpy() @ np.concatenate(o)
    exp = w["lm_head"].double().numpy() @ _rms(res)
    assert np.allclose(r.logits[0, 0], exp, atol=1e-10)


def test_swiglu_mlp_closed_form():
    """Attention output zeroed (o-proj = 0): one layer adds down(silu(gate u) * up u),
    u = RMSNorm(f), with silu(x) = x * sigmoid(x)."""
    dims = _tiny_dims(rms_eps=0.0)
    w = _tiny_weights(dims)
    w["layers"][0]["o"] = _zero(w["layers"][0]["o"])
    inp = _tiny_inputs(dims, 1, 2, 3)
    r = _run(dims, w, inp, 2)
    L0 = {k: v.double().numpy() for k, v in w["layers"][0].items()}
    f = w["fc"].double().numpy() @ inp["target_hidden"][0].double().numpy()
    u = _rms(f)
    g = L0["gate"] @ u
    res = f + L0["down"] @ (g * scipy.special.expit(g) * (L0["up"] @ u))
    exp = w["lm_head"].double().numpy() @ _rms(res)
    assert np.allclose(r.logits[0, 0], exp, atol=1e-10)


def _gains(w):
    g = {k: w[k].double().numpy() for k in ("input_norm", "hidden_norm", "final_norm")}
    g["attn"] = [L["attn_norm"].double().numpy() for L in w["layers"]]
    g["post"] = [L["post_norm"].double().numpy() for L in w["layers"]]
    return g


def test_norm_gains_route_through_attention_path():
    """Distinct random gains, two layers, single visible key (no cache, K=1) and down-proj
    zeroed: layer 1 takes x0 = [rms(e) g_in || rms(f) g_hid], layer 2 takes
    rms(res1) g_attn[2], the head takes rms(res2) g_final; layer 1's attn_norm and every
    post_norm play no part."""
    dims = _tiny_dims(n_layers=2, rms_eps=0.0)
    w = synth.make_weights(dims, 5, gains=True)
    for L in w["layers"]:
        L["down"] = _zero(L["down"])
    inp = _tiny_inputs(dims, 1, 1, 0)
    r = _run(dims, w, inp, 1)
    nq, nkv, hd = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    g = _gains(w)
    for a, b in (("input_norm", "hidden_norm"), ("hidden_norm", "final_norm")):
        assert not np.allclose(g[a], g[b])
    assert not np.allclose(g["attn"][1], g["post"][1])
    e = w["embed"][int(inp["new_token"][0])].double().numpy()
    f = w["fc"].double().numpy() @ inp["target_hidden"][0].double().numpy()
    x = np.concatenate([_rms(e) * g["input_norm"], _rms(f) * g["hidden_norm"]])
    res = f
    for li, L in enumerate(w["layers"]):
        if li > 0:
            x = _rms(res) * g["attn"][li]
        wv = L["qkv"].double().numpy()[(nq + nkv) * hd:]
        v = (wv @ x).reshape(nkv, hd)
        o = np.concatenate([v[h // (nq // nkv)] for h in range(nq)])
        res = res + L["o"].double().numpy() @ o
    exp = w["lm_head"].double().numpy() @ (_rms(res) * g["final_norm"])
    assert np.allclose(r.logits[0, 0], exp, atol=1e-10)
    w2 = dict(w)
    w2["layers"] = [dict(L) for L in w["layers"]]
    w2["layers"][0]["attn_norm"] = w["layers"][0]["attn_norm"] * 3.0
    for L in w2["layers"]:
        L["post_norm"] = -L["post_norm"]
    assert np.allclose(_run(dims, w2, inp, 1).logits, r.logits, atol=1e-12)


def test_norm_gains_route_through_mlp_path():
    """Distinct random gains, two layers, o-proj zeroed (attention adds nothing): layer l
    adds down(silu(gate u) * up u) with u = rms(res) g_post[l]; the head takes
    rms(res) g_final; the NTP row's input gains and every attn_norm play no part."""
    dims = _tiny_dims(n_layers=2, rms_eps=0.0)
    w = synth.make_weights(dims, 6, gains=True)
    for L in w["layers"]:
        L["o"] = _zero(L["o"])
    inp = _tiny_inputs(dims, 1, 2, 3)
    r = _run(dims, w, inp, 2)
    g = _gains(w)
    assert not np.allclose(g["post"][0], g["post"][1])
    f = w["fc"].double().numpy() @ inp["target_hidden"][0].double().numpy()
    res = f
    for li, L in enumerate(w["layers"]):
        Ld = {k: v.double().numpy() for k, v in L.items()}
        u = _rms(res) * g["post"][li]
        gt = Ld["gate"] @ u
        res = res + Ld["down"] @ (gt * scipy.special.expit(gt) * (Ld["up"] @ u))
    exp = w["lm_head"].double().numpy() @ (_rms(res) * g["final_norm"])
    assert np.allclose(r.logits[0, 0], exp, atol=1e-10)
    w2 = dict(w)
    w2["input_norm"] = -w["input_norm"]
    w2["hidden_norm"] = w["hidden_norm"] * 2.0
    w2["layers"] = [dict(L, attn_norm=L["attn_norm"] * 5.0) for L in w["layers"]]
    assert np.allclose(_run(dims, w2, inp, 2).logits, r.logits, atol=1e-12)


def test_draft_rows_are_causal_in_K():
    """Row j never sees rows > j: outputs of rows 0..j do not depend on K (K=1 is the
    single NTP step of EAGLE-3); and row 0 ignores emb(mask) and h_shared."""
    dims = _tiny_dims(n_layers=2)
    w = _tiny_weights(dims)
    inp = _tiny_inputs(dims, 2, 5, 7)
    full = _run(dims, w, inp, 5)
    for K in (1, 2, 3):
        part = _run(dims, w, inp, K)
        assert np.allclose(part.logits, full.logits[:, :K], atol=1e-12)
    w2 = dict(w)
    w2["emb_mask"] = w["emb_mask"] * 3 + 1
    w2["h_shared"] = -w["h_shared"]
    alt = _run(dims, w2, inp, 5)
    assert np.allclose(alt.logits[:, 0], full.logits[:, 0], atol=1e-12)
    assert not np.allclose(alt.logits[:, 1], full.logits[:, 1])


def test_bf16_cast_emulation_is_close_to_exact():
    dims = _tiny_dims(n_layers=2, dtype="bf16")
    w = _tiny_weights(dims)
    inp = _tiny_inputs(dims, 1, 4, 9)
    a = _run(dims, w, inp, 4, bf16=False)
    b = _run(dims, w, inp, 4, bf16=True)
    assert np.max(np.abs(a.logits - b.logits)) < 2e-2
    assert not np.array_equal(a.logits, b.logits)


# ---------------------------------------------------------------- training-style forward


def test_training_mask_reproduces_the_draft_block():
    """The training forward's row (a+j, j+1) equals the draft pass's row j for a request
    whose cache holds the depth-1 rows' keys/values below anchor a, with new token and
    target hidden taken at a: the mask's base-context + chain rule is the inference
    draft block."""
    dims = _tiny_dims(n_layers=2, rms_eps=1e-6)
    w = synth.make_weights(dims, 3, gains=True)
    n, K, a = 10, 4, 6
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 5)
    hidden = synth.normal((n, 3 * dims.hidden), 6)
    rows = np.array([(p, 1) for p in range(n)] + [(a + j, j + 1) for j in range(1, K)])
    rows = rows[np.lexsort((rows[:, 1], rows[:, 0]))]
    W = O.Weights64.from_synth(w)
    logits, _, _ = O.forward_parallel(W, dims, tokens, hidden, rows, bf16=False)
    # depth-1 keys/values per layer, to fill the draft pass's cache
    d1 = np.array([(p, 1) for p in range(n)])
    ks, vs = _depth1_kv(W, dims, tokens, hidden, d1)
    cache_k = np.zeros((dims.n_layers, 1, dims.n_kv_heads, a + K, dims.head_dim))
    cache_v = np.zeros_like(cache_k)
    for li in range(dims.n_layers):
        cache_k[li, 0, :, :a] = ks[li][:a].transpose(1, 0, 2)
        cache_v[li, 0, :, :a] = vs[li][:a].transpose(1, 0, 2)
    r = O.draft_pass(W, dims, cache_k, cache_v, [a], hidden[a:a + 1], tokens[a:a + 1], K,
                     bf16=False)
    idx = {(int(p), int(d)): i for i, (p, d) in enumerate(rows)}
    for j in range(K):
        assert np.allclose(logits[idx[(a + j, j + 1)]], r.logits[0, j], atol=1e-9)


def _depth1_kv(W, dims, tokens, hidden, rows):
    """Keys/values of depth-1 rows per layer, by running the decode pass one position at
    a time with K=1 (the autoregressive NTP step)."""
    n = len(rows)
    nkv, hd = dims.n_kv_heads, dims.head_dim
    ks = [np.zeros((n, nkv, hd)) for _ in range(dims.n_layers)]
    vs = [np.zeros((n, nkv, hd)) for _ in range(dims.n_layers)]
    for p in range(n):
        ck = np.zeros((dims.n_layers, 1, nkv, p + 1, hd))
        cv = np.zeros_like(ck)
        for li in range(dims.n_layers):
            ck[li, 0, :, :p] = ks[li][:p].transpose(1, 0, 2)
            cv[li, 0, :, :p] = vs[li][:p].transpose(1, 0, 2)
        r = O.draft_pass(W, dims, ck, cv, [p], hidden[p:p + 1], tokens[p:p + 1], 1, bf16=False)
        for li in range(dims.n_layers):
            ks[li][p] = r.k_rows[li][0, 0]
            vs[li][p] = r.v_rows[li][0, 0]
    return ks, vs


def test_training_forward_prefix_closure():
    """Rows with p < P0 only depend on rows with p < P0 (position invariance, 3.1): the
    forward over the prefix equals the full forward on those rows."""
    dims = _tiny_dims(n_layers=2)
    w = synth.make_weights(dims, 3, gains=True)
    n, K = 24, 4
    tokens = synth.uniform_ints(n, 0, dims.target_vocab, 7)
    hidden = synth.normal((n, 3 * dims.hidden), 8)
    rows = O.cod_retained(n, K, 0.8, synth.cod_uniforms(n, K, seed=12))
    W = O.Weights64.from_synth(w)
    full, _, _ = O.forward_parallel(W, dims, tokens, hidden, rows, bf16=False)
    pre = rows[rows[:, 0] < 11]
    part, _, _ = O.forward_parallel(W, dims, tokens, hidden, pre, bf16=False)
    assert np.allclose(part, full[: len(pre)], atol=1e-10)
    # dependency closure of a few late rows reproduces them too
    tgt = rows[-3:]
    clo = O.dependency_closure(rows, tgt)
    sub, _, _ = O.forward_parallel(W, dims, tokens, hidden, clo, bf16=False)
    idx = {(int(p), int(d)): i for i, (p, d) in enumerate(clo)}
    for t, (p, d) in enumerate(tgt):
        assert np.allclose(sub[idx[(int(p), int(d))]], full[len(rows) - 3 + t], atol=1e-10)


# ------------------------------------------------------------------ drafter catch-up


def _catch_inputs(dims, T, L, seed):
    w = synth.make_weights(dims, seed)
    wl = synth.Workload("s", dims, 1, 4, (L,))
    inp = synth.make_decode_inputs(wl, seed + 1, capacity=L + T + 4)
    hid = synth.normal((1, T, 3 * dims.hidden), seed + 2, 1.0)
    tok = synth.uniform_ints(T, 0, dims.target_vocab, seed + 3).reshape(1, T)
    return O.Weights64.from_synth(w), inp, hid, tok


def test_catch_up_on_empty_cache_is_the_causal_depth1_forward():
    """With no cached context, the catch-up rows are exactly the depth-1 rows of the
    training-style forward (plain causal attention): two independently written paths."""
    dims = synth.DIMS_TINY
    T = 6
    W, inp, hid, tok = _catch_inputs(dims, T, 0, 31)
    r = O.catch_up(W, dims, inp["cache_k"], inp["cache_v"], [0], hid, tok, bf16=False)
    rows = np.array([(p, 1) for p in range(T)])
    lg, am, _ = O.forward_parallel(W, dims, tok[0], hid[0], rows, bf16=False)
    assert np.max(np.abs(r.logits[0] - lg)) < 1e-12
    assert np.array_equal(r.argmax[0], am)


def test_catch_up_single_row_is_the_ntp_row():
    dims = synth.DIMS_TINY
    W, inp, hid, tok = _catch_inputs(dims, 1, 9, 41)
    r = O.catch_up(W, dims, inp["cache_k"], inp["cache_v"], [9], hid, tok, bf16=False)
    d = O.draft_pass(W, dims, inp["cache_k"], inp["cache_v"], [9], hid[:, 0], tok[:, 0], 1,
                     bf16=False)
    assert np.max(np.abs(r.logits - d.logits)) < 1e-12
    for li in range(dims.n_layers):
        assert np.max(np.abs(r.k_rows[li] - d.k_rows[li])) < 1e-12


def test_catch_up_is_causal():
    dims = synth.DIMS_TINY
    T = 4
    W, inp, hid, tok = _catch_inputs(dims, T, 5, 51)
    a = O.catch_up(W, dims, inp["cache_k"], inp["cache_v"], [5], hid, tok, bf16=False)
    tok2 = tok.copy()
    tok2[0, T - 1] = (tok2[0, T - 1] + 1) % dims.target_vocab
    b = O.catch_up(W, dims, inp["cache_k"], inp["cache_v"], [5], hid, tok2, bf16=False)
    assert np.array_equal(a.logits[0, : T - 1], b.logits[0, : T - 1])
    assert np.max(np.abs(a.logits[0, T - 1] - b.logits[0, T - 1])) > 1e-6


# ---------------------------------------------------------------- sliding-window attention
# ([E4] "EAGLE-4 overview": the drafter attends to the most recent 4,096 positions)


def test_window_covering_the_context_is_full_attention():
    """A window at least as long as the context plus the draft block changes nothing."""
    dims = _tiny_dims(n_layers=2)
    w = _tiny_weights(dims)
    inp = _tiny_inputs(dims, 2, 4, 9)
    full = _run(dims, w, inp, 4)
    for W in (13, 14, 100):
        r = _run(synth.shrink(dims, attn_window=W), w, inp, 4)
        assert np.allclose(r.logits, full.logits, atol=1e-12)
    r = _run(synth.shrink(dims, attn_window=12), w, inp, 4)  # row 3 (position 12) loses key 0
    assert np.allclose(r.logits[:, :3], full.logits[:, :3], atol=1e-12)
    assert not np.allclose(r.logits[:, 3], full.logits[:, 3])


def test_window_of_one_position_is_self_attention():
    """W = 1: every row sees only its own key, whatever the cache holds, so each row is
    the single-key closed form: residual f + W_o(v of its kv heads) (down-proj zeroed),
    v = W_v x0, x0 = [RMSNorm(e) || RMSNorm(f)] with e, f the row's NTP or MTP inputs."""
    dims = _tiny_dims(rms_eps=0.0, attn_window=1)
    w = _tiny_weights(dims)
    w["layers"][0]["down"] = _zero(w["layers"][0]["down"])
    K = 3
    inp = _tiny_inputs(dims, 2, K, 6)
    r = _run(dims, w, inp, K)
    H, nq, nkv, hd = dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    wv = w["layers"][0]["qkv"].double().numpy()[(nq + nkv) * hd:]
    wo = w["layers"][0]["o"].double().numpy()
    fc = w["fc"].double().numpy()
    for b in range(2):
        for j in range(K):
            if j == 0:
                e = w["embed"][int(inp["new_token"][b])].double().numpy()
                f = fc @ inp["target_hidden"][b].double().numpy()
            else:
                e = w["emb_mask"].double().numpy()
                f = fc @ w["h_shared"].double().numpy()
            x0 = np.concatenate([_rms(e), _rms(f)])
            v = (wv @ x0).reshape(nkv, hd)
            o = np.concatenate([v[h // (nq // nkv)] for h in range(nq)])
            exp = w["lm_head"].double().numpy() @ _rms(f + wo @ o)
            assert np.allclose(r.logits[b, j], exp, atol=1e-10)


def test_window_ignores_keys_outside_it():
    """With W = 5, L = 8 and K = 3, row j sees positions 4 + j .. 8 + j: changing cached
    positions 0..3 changes no row; changing position 4 changes row 0 only (one layer, so
    rows meet only through the draft block's own keys)."""
    dims = _tiny_dims(attn_window=5)
    w = _tiny_weights(dims)
    inp = _tiny_inputs(dims, 1, 3, 8)
    base = _run(dims, w, inp, 3)
    far = {k: v for k, v in inp.items()}
    far["cache_k"] = inp["cache_k"].clone()
    far["cache_v"] = inp["cache_v"].clone()
    far["cache_k"][:, :, :, :4] += 1.5
    far["cache_v"][:, :, :, :4] -= 2.0
    assert np.allclose(_run(dims, w, far, 3).logits, base.logits, atol=1e-12)
    edge = {k: v for k, v in inp.items()}
    edge["cache_k"] = inp["cache_k"].clone()
    edge["cache_v"] = inp["cache_v"].clone()
    edge["cache_v"][:, :, :, 4] += 3.0
    r = _run(dims, w, edge, 3)
    assert not np.allclose(r.logits[0, 0], base.logits[0, 0])
    assert np.allclose(r.logits[0, 1:], base.logits[0, 1:], atol=1e-12)


# ---------------------------------------------------------------- efficient LM head
# ([E4] "EAGLE-4 overview": a rank-128 projection scores the vocabulary, the full head
# scores the best 128 candidates)


def _eff_dims(**kw):
    return _tiny_dims(lm_rank=4, lm_topk=6, draft_vocab=50, **kw)


def test_efficient_head_with_every_candidate_is_the_full_head():
    dims = _eff_dims()
    w = _tiny_weights(dims)
    inp = _tiny_inputs(dims, 2, 3, 5)
    full = _run(synth.shrink(dims, lm_rank=0, lm_topk=0), w, inp, 3)
    allc = _run(synth.shrink(dims, lm_topk=dims.draft_vocab), w, inp, 3)
    assert np.array_equal(allc.argmax, full.argmax)
    assert np.array_equal(allc.tokens, full.tokens)
    assert np.allclose(allc.logits, full.logits, atol=1e-12)


def test_efficient_head_on_an_exactly_low_rank_head_is_the_full_argmax():
    """lm_head = lm_score lm_proj: the rank-r scores are the exact logits, so the best
    candidate is the full head's argmax for any candidate count."""
    dims = _eff_dims()
    w = _tiny_weights(dims)
    w["lm_head"] = w["lm_score"].double() @ w["lm_proj"].double()
    inp = _tiny_inputs(dims, 2, 3, 5)
    full = _run(synth.shrink(dims, lm_rank=0, lm_topk=0), w, inp, 3)
    for k in (1, 2, 6):
        r = _run(synth.shrink(dims, lm_topk=k), w, inp, 3)
        assert np.array_equal(r.argmax, full.argmax)
        assert np.allclose(r.approx, full.logits, atol=1e-10)


def test_efficient_head_candidates_and_winner_by_brute_force():
    """The finite logits sit exactly at the lm_topk largest rank-r scores, equal the full
    head's logits there, and the token is the best of them (brute force per row)."""
    dims = _eff_dims()
    w = _tiny_weights(dims)
    inp = _tiny_inputs(dims, 2, 3, 5)
    r = _run(dims, w, inp, 3)
    full = _run(synth.shrink(dims, lm_rank=0, lm_topk=0), w, inp, 3)
    for b in range(2):
        for j in range(3):
            ranked = sorted(range(dims.draft_vocab), key=lambda i: (-r.approx[b, j, i], i))
            cand = set(ranked[:dims.lm_topk])
            assert set(np.nonzero(np.isfinite(r.logits[b, j]))[0].tolist()) == cand
            for c in cand:
                assert abs(r.logits[b, j, c] - full.logits[b, j, c]) < 1e-12
            best = max(cand, key=lambda i: (full.logits[b, j, i], -i))
            assert r.argmax[b, j] == best
            assert r.tokens[b, j] == best + int(w["d2t"][best])


# ---------------------------------------------------------------- training step
from oracle import peagle_train_oracle as T  # noqa: E402


def _train_case(seed=11, n=6, K=3, cod=None):
    """Tiny drafter (two layers, GQA 2:1) with norm gains, emb(mask) and h_shared drawn
    away from their initial values, so that no gradient pin passes on a unit gain."""
    dims = synth.Dims(hidden=8, n_layers=2, n_q_heads=2, n_kv_heads=1, head_dim=4,
                      intermediate=12, draft_vocab=11, target_vocab=13, rope_theta=10000.0,
                      rms_eps=1e-5, dtype="f32", d2t="identity")
    W = O.Weights64.from_synth(synth.make_weights(dims, seed))
    rng = np.random.default_rng(seed)
    W.embed = O.to64(W.embed)
    W.fc, W.lm_head = W.fc * 8.0, W.lm_head * 8.0
    for name in ("input_norm", "hidden_norm", "final_norm"):
        setattr(W, name, 1.0 + 0.3 * rng.standard_normal(dims.hidden))
    for L in W.layers:
        for k in list(L):
            L[k] = (1.0 + 0.3 * rng.standard_normal(L[k].shape)) if k.endswith("norm") \
                else L[k] * 8.0
    tokens = rng.integers(0, dims.target_vocab, n)
    hidden = rng.standard_normal((n, 3 * dims.hidden))
    rows = np.array([(p, d) for p in range(n) for d in range(1, K + 1) if p - d + 1 >= 0])
    if cod is not None:
        rows = O.cod_retained(n, K, cod, rng.random((n, K)))
    labels = rng.integers(0, dims.draft_vocab, len(rows))
    return dims, W, tokens, hidden, rows, labels


def _params(W):
    out = {"embed": W.embed, "emb_mask": W.emb_mask, "h_shared": W.h_shared, "fc": W.fc,
           "input_norm": W.input_norm, "hidden_norm": W.hidden_norm,
           "final_norm": W.final_norm, "lm_head": W.lm_head}
    for li, L in enumerate(W.layers):
        for k, v in L.items():
            out[f"layers.{li}.{k}"] = v
    return out


def _grad(g, name):
    if name.startswith("layers."):
        _, li, k = name.split(".")
        return g["layers"][int(li)][k]
    return g[name]


def test_train_step_forward_is_the_training_forward():
    dims, W, tokens, hidden, rows, labels = _train_case(cod=0.8)
    loss, logits, _ = T.train_step(W, dims, tokens, hidden, rows, labels)
    ref, _, _ = O.forward_parallel(W, dims, tokens, hidden, rows, bf16=False)
    assert np.allclose(logits, ref, rtol=0, atol=1e-12)
    # mean cross-entropy, from scipy's logsumexp
    ce = scipy.special.logsumexp(ref, axis=1) - ref[np.arange(len(rows)), labels]
    assert abs(loss - ce.mean()) < 1e-12


@pytest.mark.parametrize("cod", [None, 0.7])
def test_train_step_gradients_match_finite_differences(cod):
    """Every parameter tensor, several entries each: the hand-written chain rule against
    central differences of the loss (h = 1e-5, fp64)."""
    dims, W, tokens, hidden, rows, labels = _train_case(cod=cod, seed=5 if cod else 11)
    loss, _, g = T.train_step(W, dims, tokens, hidden, rows, labels)
    rng = np.random.default_rng(1)
    used = sorted({int(tokens[p]) for p, d in rows if d == 1})
    h = 1e-5
    for name, arr in _params(W).items():
        if name.endswith("attn_norm") and name.startswith("layers.0."):
            assert not np.any(_grad(g, name))  # layer 1 reads x0, not a norm of res
            continue
        for _ in range(4):
            if name == "embed":
                idx = (used[rng.integers(len(used))], int(rng.integers(arr.shape[1])))
            else:
                idx = tuple(int(rng.integers(s)) for s in arr.shape)
            old = arr[idx]
            arr[idx] = old + h
            lp = T.train_step(W, dims, tokens, hidden, rows, labels)[0]
            arr[idx] = old - h
            lm = T.train_step(W, dims, tokens, hidden, rows, labels)[0]
            arr[idx] = old
            fd = (lp - lm) / (2 * h)
            an = _grad(g, name)[idx]
            assert abs(fd - an) <= 1e-7 + 1e-5 * abs(fd), (name, idx, fd, an)
    # rows of the embedding that no depth-1 row reads get no gradient
    unused = [t for t in range(dims.target_vocab) if t not in used]
    assert not np.any(g["embed"][unused])
