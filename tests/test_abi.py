"""CPU-only checks of the C ABI: the library builds and loads, exports every entry point
that include/peagle.h declares, rejects bad arguments before touching the GPU, and its
host-side COD sampler agrees with the oracle's."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth
from oracle import peagle_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pk():
    from drafting_eagle_draft_gb300 import build

    build.build()
    import drafting_eagle_draft_gb300 as pk

    pk.lib()
    return pk


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(peagle_[a-z_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(pk):
    names = _declared()
    assert {"peagle_create", "peagle_draft", "peagle_append_kv", "peagle_verify_greedy"} <= names
    L = ctypes.CDLL(pk.LIB_PATH)
    for n in sorted(names):
        assert hasattr(L, n), n
    assert set(pk.EXPORTS) == names


def test_struct_layout_matches_header(pk):
    # peagle_dims: 14 int32 + 2 float + attn_window, lm_rank, lm_topk, train;
    # peagle_weights: 18 pointers; peagle_kv: 2 ptr + 2 int
    assert ctypes.sizeof(pk.PeagleDims) == 80
    assert pk.PeagleDims.attn_window.offset == 64
    assert pk.PeagleDims.lm_topk.offset == 72
    assert pk.PeagleDims.train.offset == 76
    assert ctypes.sizeof(pk.PeagleWeights) == 18 * 8
    assert ctypes.sizeof(pk.PeagleKV) == 24
    assert ctypes.sizeof(pk.PeagleGrads) == 15 * 8
    assert pk.PeagleGrads.qkv.offset == 6 * 8 and pk.PeagleGrads.lm_head.offset == 14 * 8


def test_host_argument_errors(pk):
    L = pk.lib()
    assert L.peagle_verify_greedy(0, 4, 1, 1, 1, 1, None) == pk.PEAGLE_ERR_INVALID
    assert L.peagle_verify_greedy(1, 0, 1, 1, 1, 1, None) == pk.PEAGLE_ERR_INVALID
    assert L.peagle_verify_greedy(1, 4, None, 1, 1, 1, None) == pk.PEAGLE_ERR_INVALID
    kv = pk.PeagleKV(1, 1, 16, 1)
    assert L.peagle_draft(None, 1, ctypes.byref(kv), 1, 1, 1, 4, 1, None, None) == pk.PEAGLE_ERR_INVALID
    assert L.peagle_append_kv(None, 1, ctypes.byref(kv), 1, 1, 0, None, None, 0, None) == pk.PEAGLE_ERR_INVALID
    assert L.peagle_set_timing(None, 1) == pk.PEAGLE_ERR_INVALID
    assert L.peagle_forward_parallel(None, 8, 4, 1, 1, 1, 1, 4, 1, None, None) == pk.PEAGLE_ERR_INVALID
    assert L.peagle_status(None) == pk.PEAGLE_ERR_INVALID
    L.peagle_destroy(None)
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(pk.strerror(code), str)


def test_create_rejects_unsupported_dims(pk):
    L = pk.lib()
    base = synth.DIMS_TINY
    h = ctypes.c_void_p()
    w = pk.PeagleWeights()
    cases = [
        (dict(head_dim=96), pk.PEAGLE_ERR_UNSUPPORTED),
        (dict(n_kv_heads=3), pk.PEAGLE_ERR_UNSUPPORTED),
        (dict(hidden=200), pk.PEAGLE_ERR_UNSUPPORTED),
        (dict(hidden=0), pk.PEAGLE_ERR_INVALID),
    ]
    for kw, code in cases:
        d = pk.make_dims(synth.shrink(base, **kw), 1, 4, 256)
        assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == code, kw
        assert not h.value
    d = pk.make_dims(base, 1, 17, 256)
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_CAPACITY
    d = pk.make_dims(base, 64, 8, 256)
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_CAPACITY
    d = pk.make_dims(synth.shrink(base, dtype="f32"), 1, 4, 256)
    d.dtype = 7
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_UNSUPPORTED
    # training workspaces need parallel-forward rows and no window / efficient head
    d = pk.make_dims(base, 1, 4, 256, train=True)
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_INVALID
    d = pk.make_dims(synth.shrink(base, attn_window=8), 1, 4, 256, 64, 16, train=True)
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_UNSUPPORTED
    d = pk.make_dims(base, 1, 4, 256, 64, 16)
    d.train = 2
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_INVALID
    # valid dims but missing weight pointers
    d = pk.make_dims(base, 1, 4, 256)
    assert L.peagle_create(ctypes.byref(w), ctypes.byref(d), ctypes.byref(h)) == pk.PEAGLE_ERR_INVALID


def test_library_needs_no_vendor_blas():
    """Every GEMM of the library (draft pass, training forward, training step) runs on its
    own kernels: the shared object lists no cuBLAS / cuBLASLt dependency."""
    import shutil
    import subprocess

    from drafting_eagle_draft_gb300 import build

    path = build.build()
    tool = shutil.which("readelf")
    if tool is None:
        pytest.skip("readelf not available")
    out = subprocess.run([tool, "-d", path], capture_output=True, text=True, check=True).stdout
    needed = re.findall(r"\(NEEDED\).*\[(.+?)\]", out)
    assert needed, out
    assert not [n for n in needed if "cublas" in n.lower()], needed


@pytest.mark.parametrize("n,K,r", [(1, 4, 0.8), (37, 8, 0.8), (500, 8, 0.7), (64, 16, 0.9)])
def test_cod_rows_matches_oracle(pk, n, K, r):
    u = synth.cod_uniforms(n, K, seed=n + K)
    rp, rd = pk.peagle_cod_rows(n, K, r, u)
    ref = O.cod_retained(n, K, r, u)
    assert np.array_equal(np.stack([rp, rd], 1), ref)


def test_cod_rows_capacity_error(pk):
    L = pk.lib()
    u = np.zeros((10, 4))
    out = np.zeros(5, np.int32)
    rc = L.peagle_cod_rows(10, 4, ctypes.c_double(0.8), u.ctypes.data, out.ctypes.data,
                           out.ctypes.data, 5)
    assert rc == pk.PEAGLE_ERR_CAPACITY


@pytest.mark.parametrize("n,K,r,bnd", [
    (64, 8, 0.8, [0, 16, 32, 48]),
    (500, 8, 0.7, [0, 100, 101, 333]),
    (200, 16, 1.0, [0, 7]),
    (33, 4, 0.8, [0]),
])
def test_sequence_partition_matches_oracle(pk, n, K, r, bnd):
    u = synth.cod_uniforms(n, K, seed=3 * n + K)
    rp, rd = pk.peagle_cod_rows(n, K, r, u)
    got = pk.peagle_sequence_partition(rp, rd, bnd)
    ref, _ = O.sequence_partition(np.stack([rp, rd], 1), bnd)
    assert np.array_equal(got, ref)


def test_sequence_partition_rejects_bad_input(pk):
    rp = np.array([0, 1, 1, 2, 2, 2], np.int32)
    rd = np.array([1, 1, 2, 1, 2, 3], np.int32)
    assert np.array_equal(pk.peagle_sequence_partition(rp, rd, [0, 2]), [0, 0, 0, 1, 1, 0])
    for bnd in ([1, 2], [0, 2, 2], [0, 3, 1]):  # must start at 0 and increase
        with pytest.raises(pk.PeagleError):
            pk.peagle_sequence_partition(rp, rd, bnd)
    with pytest.raises(pk.PeagleError):  # not p-major
        pk.peagle_sequence_partition(rp[::-1], rd[::-1], [0])
    with pytest.raises(pk.PeagleError):  # (2, 3) without (1, 2)
        pk.peagle_sequence_partition(np.array([0, 1, 2, 2], np.int32),
                                     np.array([1, 1, 1, 3], np.int32), [0])
