"""Shared helpers of the GPU parity tests: build contexts, run the draft pass through the
C ABI, and compare with the fp64 oracle."""

import numpy as np
import torch

import synth
from oracle import peagle_oracle as O

LOGIT_TOL = {"f32": 1e-4, "bf16": 2e-2}
MARGIN = 1e-2  # draft ids must match the oracle wherever its top-1 margin exceeds this
RECORD = []  # (case, max abs logit error, tolerance, compared logits, rows with clear margin)


def pk():
    from drafting_eagle_draft_gb300 import build

    build.build()
    import drafting_eagle_draft_gb300 as m

    return m


def make_ctx(dims, w, max_batch, max_K, max_positions, max_rows=0, max_seq=0,
             pass_kernel=None, train=False):
    """A context; pass_kernel True / False forces the persistent pass kernel on / off for
    the bf16 draft pass (None: the library default)."""
    m = pk()
    ctx = m.peagle_create(w, m.make_dims(dims, max_batch, max_K, max_positions, max_rows,
                                         max_seq, train))
    if pass_kernel is not None and (dims.dtype == "bf16" or not pass_kernel):
        # fp32 drafters have no persistent pass kernel: they always take separate launches
        m.peagle_set_pass_kernel(ctx, 1 if pass_kernel else 0)
    return ctx


def to_dev(inp, dev="cuda"):
    return {
        "ck": inp["cache_k"].to(dev).contiguous(),
        "cv": inp["cache_v"].to(dev).contiguous(),
        "sl": torch.from_numpy(np.ascontiguousarray(inp["seq_lens"], np.int32)).to(dev),
        "th": inp["target_hidden"].to(dev).contiguous(),
        "nt": torch.from_numpy(np.ascontiguousarray(inp["new_token"], np.int32)).to(dev),
    }


def run_draft(ctx, dims, inp, K, d=None, logits=True):
    """One peagle_draft call; returns (tokens [B,K], logits [B,K,Vd] or None, device dict)."""
    m = pk()
    d = d or to_dev(inp)
    B = d["sl"].shape[0]
    cap = d["ck"].shape[3]
    kv = m.kv_struct(d["ck"], d["cv"], cap, d["ck"].shape[1])
    toks = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    lg = torch.full((B, K, dims.draft_vocab), float("nan"), device="cuda") if logits else None
    m.peagle_draft(ctx, B, kv, d["sl"], d["th"], d["nt"], K, toks, lg)
    assert m.peagle_status(ctx) == m.PEAGLE_OK
    return toks.cpu().numpy(), (lg.cpu().numpy() if logits else None), d


def oracle_draft(dims, w, inp, K, idx=None, W=None):
    """Oracle draft pass with the bf16 path's rounding profile (KV-cache stores only)."""
    W = W or O.Weights64.from_synth(w, lazy=True)
    casts = O.DRAFT_BF16_CASTS if dims.dtype == "bf16" else False
    if idx is None:
        return O.draft_pass(W, dims, inp["cache_k"], inp["cache_v"], inp["seq_lens"],
                            inp["target_hidden"], inp["new_token"], K, bf16=casts)
    idx = list(idx)
    return O.draft_pass(W, dims, inp["cache_k"][:, idx], inp["cache_v"][:, idx],
                        np.asarray(inp["seq_lens"])[idx], inp["target_hidden"][idx],
                        np.asarray(inp["new_token"])[idx], K, bf16=casts)


def check_tokens_vs_own_logits(tokens, logits, d2t):
    """The GPU's ids are the argmax of its own fp32 logits (lowest index on ties) + d2t."""
    am = np.argmax(logits, axis=-1)
    assert np.array_equal(tokens, am + np.asarray(d2t)[am])


def compare(dims, ref, tokens, logits, what=""):
    tol = LOGIT_TOL[dims.dtype]
    err = float(np.max(np.abs(logits - ref.logits)))
    assert err <= tol, f"{what}: logits max abs err {err:.3e} > {tol}"
    ok = ref.margin > MARGIN
    assert ok.mean() > 0.5, f"{what}: too few rows with a clear margin"
    bad = np.argwhere(ok & (tokens != ref.tokens))
    RECORD.append({"case": what, "max_abs_err": err, "tol": tol, "logits": int(logits.size),
                   "id_rows_checked": int(ok.sum()), "id_rows": int(ok.size)})
    assert len(bad) == 0, f"{what}: draft ids differ at {bad[:5].tolist()}"
    return err
