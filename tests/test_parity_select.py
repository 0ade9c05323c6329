"""GPU parity of the selection kernel: rows whose kept set or top-n the
streaming kernel's candidates cannot settle (large top-p nuclei, large top-k)
go to a second kernel.  For bf16 rows without penalties it selects on bf16
code slots; these cases force its several-valued slots (values near zero, a
catch-all far below the maximum), slots holding thousands of equal values,
boundaries inside them, top-n that reaches -inf, and unaligned rows, each of
which must still give the oracle's result (through the code selection or the
generic radix selection it hands such rows to)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from device_token_sampling_gb300 import workloads as W

from paritylib import compare, custom_workload, device_logits, make_sampler, run_gpu

pytestmark = pytest.mark.gpu

V_FULL = 151_936


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def check(w, expect_handover=True):
    """Both sampling paths against the oracle: the streaming kernel (which must
    hand rows to the selection kernel here) and, for bf16 rows without
    penalties, the flat kernels (which settle most rows themselves)."""
    o = O.sample_workload(w, want_zt=True)
    g = None
    for path in (1, 2):
        s = make_sampler(w)
        try:
            s.set_path(path)
            g = run_gpu(s, w)
            if expect_handover and path == 1:
                assert s.last_handover() > 0, "no row reached the selection kernel"
            compare(g, o, where=f"{w.name} path {path}")
        finally:
            s.close()
    return g, o


def bulk(rng, B, V, sigma=1.5):
    return rng.normal(0, sigma, size=(B, V)).astype(np.float32)


@pytest.mark.parametrize("T", [0.9, 1.5])
def test_large_nucleus_top_p(T):
    rng = np.random.default_rng(101)
    x = W.peaked_rows(rng, 8, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=T,
                        p=[0.5, 0.6, 0.7, 0.8, 0.9, 0.95, 0.99, 0.999], n=20, name=f"nucleus T{T}")
    check(w)


def test_large_top_k():
    rng = np.random.default_rng(102)
    x = bulk(rng, 6, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.2, k=[1500, 2047, 2500, 4000, 9000, 30000],
                        n=8, name="topk large")
    check(w)


def test_top_k_then_top_p_and_min_p():
    rng = np.random.default_rng(103)
    x = bulk(rng, 6, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.3, k=[3000, 6000, 0, 5000, 20000, 0],
                        p=[0.9, 0.5, 0.95, 1.0, 0.8, 0.7], mp=[0.0, 0.0, 0.001, 0.002, 0.0, 0.0005],
                        n=5, name="k+p+minp")
    check(w)


def test_values_near_zero():
    # a fifth of each row exactly zero or below 2^-12 in magnitude: the tiny slot,
    # with several values, above, at and below the boundary
    rng = np.random.default_rng(104)
    B, V = 6, 60_000
    x = bulk(rng, B, V, sigma=0.5)
    for r in range(B):
        idx = rng.choice(V, V // 5, replace=False)
        x[r, idx] = rng.normal(0, 1e-4, size=idx.size).astype(np.float32)
        x[r, idx[::7]] = 0.0
        x[r, idx[1::11]] = -0.0
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=[1.0, 1.5, 2.0, 1.0, 1.5, 3.0],
                        p=[0.9, 0.5, 0.99, 0.7, 0.3, 0.95], n=4, name="near zero")
    check(w)


def test_all_near_zero():
    # the row maximum itself below 2^-12: nearly everything in the tiny slot
    rng = np.random.default_rng(105)
    x = rng.normal(0, 1e-5, size=(4, 40_000)).astype(np.float32)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1e-5, p=[0.5, 0.9, 0.99, 0.7], n=3,
                        name="all tiny")
    check(w, expect_handover=False)


def test_catch_all():
    # a few huge values: the bulk falls more than 4096 codes below the maximum
    rng = np.random.default_rng(106)
    B, V = 6, 50_000
    x = bulk(rng, B, V)
    x[:, :3] = [3.0e4, 2.0e4, 1.0e4]
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=[1e4, 2e4, 5e4, 1e4, 1.0, 3e4],
                        k=[0, 0, 10, 20_000, 0, 0], p=[0.9, 0.99, 1.0, 1.0, 0.9, 0.999], n=5,
                        name="catch-all")
    check(w, expect_handover=False)


def test_dense_equal_values():
    # values on a coarse grid: each bf16 code holds thousands of elements, more
    # than the boundary gather takes, so such rows go to the generic selection
    rng = np.random.default_rng(107)
    x = np.round(bulk(rng, 6, V_FULL, sigma=1.0) * 4.0) / 4.0
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=[1.0, 1.5, 0.8, 1.2, 1.0, 2.0],
                        k=[0, 5000, 0, 0, 30000, 0], p=[0.9, 1.0, 0.5, 0.99, 0.95, 0.7], n=6,
                        name="dense ties")
    check(w)


def test_top_n_reaching_minus_inf():
    # fewer finite values than n on a row whose top-p nucleus is large
    rng = np.random.default_rng(108)
    B, V = 4, 50_000
    x = np.full((B, V), -np.inf, np.float32)
    for r in range(B):
        idx = rng.choice(V, 12, replace=False)
        x[r, idx] = rng.normal(0, 0.01, 12)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.0, p=0.99, n=20, name="few finite")
    check(w, expect_handover=False)


@pytest.mark.parametrize("pad", [1, 3])
def test_unaligned_rows(pad):
    # rows not 16-byte aligned: the generic selection reads them element-wise
    rng = np.random.default_rng(109 + pad)
    x = W.peaked_rows(rng, 4, 70_001)
    w = custom_workload(x, dtype=W.DTYPE_BF16, ld=70_001 + pad, T=1.4, p=[0.9, 0.99, 0.7, 0.95],
                        n=5, name=f"unaligned {pad}")
    check(w)


def test_repeat_calls_reuse_handover_state():
    # the hand-over counters are reset by the selection kernel: a second and third
    # call with the same handle must hand over and sample again
    rng = np.random.default_rng(110)
    x = W.peaked_rows(rng, 8, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.5, p=0.95, n=5, name="repeat")
    s = make_sampler(w)
    try:
        s.set_path(1)
        xd = device_logits(w)
        first = run_gpu(s, w, x=xd)
        for _ in range(2):
            again = run_gpu(s, w, x=xd)
            for k in first:
                np.testing.assert_array_equal(first[k], again[k], err_msg=k)
        assert s.last_handover() > 0
    finally:
        s.close()
