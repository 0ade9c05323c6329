"""GPU parity of the flat kernels (sampling path 2): bf16 batches without
penalties or top-p decay, in six launches over (row, slice) pairs, against the
oracle.  Every row class of the pages [TensorRT-LLM "Sampling": temperature,
top-k, top-p over the survivors renormalised, min-p; the Gumbel-max draw of
vllm.cpp with lowest-index ties; log-probs and top-n of the Tenstorrent
sampling README], the rows the flat kernels hand to the selection kernel (a
top_k above 1024, candidate lists that overflow, fewer finite values than the
candidate threshold needs), non-finite and empty rows, ragged widths, and
seeds that advance over several calls."""
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


def flat_check(w, expect_hand=None, steps=1):
    """Path 2 against the oracle (over `steps` calls, seeds advancing)."""
    s = make_sampler(w)
    try:
        s.set_path(2)
        s.reset_workload(w)
        x = device_logits(w)
        seed = w.seed.copy()
        for step in range(steps):
            g = run_gpu(s, w, x=x, reset=False)
            assert s.last_launches() == 7, "the flat kernels did not run"
            o = O.sample_workload(w, want_zt=True, seed=seed)
            compare(g, o, where=f"{w.name} step {step}")
            seed = np.array([O.next_seed(int(v)) for v in seed], np.uint64)
        if expect_hand is not None:
            handed = s.last_handover()
            assert (handed > 0) == expect_hand, handed
    finally:
        s.close()


def test_b256_workload():
    w = W.b256()
    flat_check(w, expect_hand=False)


@pytest.mark.parametrize("greedy", [False, True])
def test_b32_workload(greedy):
    w = W.b32(greedy=greedy)
    flat_check(w)


@pytest.mark.parametrize("T", [0.3, 0.8, 1.5])
def test_top_p_rows(T):
    rng = np.random.default_rng(int(T * 10) + 1)
    x = W.peaked_rows(rng, 8, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=T,
                        p=[0.3, 0.5, 0.7, 0.8, 0.9, 0.95, 0.99, 0.999], n=20, name=f"top-p T{T}")
    flat_check(w, steps=2)


@pytest.mark.parametrize("k", [2, 20, 300, 1024])
def test_top_k_rows(k):
    rng = np.random.default_rng(k)
    x = W.peaked_rows(rng, 8, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=[0.4, 0.7, 1.0, 1.3] * 2, k=k,
                        p=[1.0] * 4 + [0.5, 0.8, 0.95, 0.99], mp=[0.0, 0.02] * 4, n=8,
                        name=f"top-k {k}")
    flat_check(w, expect_hand=False, steps=2)


@pytest.mark.parametrize("mp", [0.001, 0.05, 0.3])
def test_min_p_and_unfiltered_rows(mp):
    rng = np.random.default_rng(int(mp * 1000))
    x = W.peaked_rows(rng, 8, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=[0.5, 1.0, 1.5, 1.2] * 2,
                        mp=[mp, mp, mp, 0.0] * 2, p=[1.0] * 4 + [0.9] * 4, n=5,
                        name=f"min-p {mp}")
    flat_check(w)


def test_rows_handed_to_the_selection_kernel():
    rng = np.random.default_rng(7)
    x = W.peaked_rows(rng, 8, V_FULL)
    x[2] = 0.0                                    # flat: every element a candidate
    x[3] = np.round(rng.standard_normal(V_FULL))  # few distinct values
    x[4, :] = -np.inf                             # 40 finite values only
    x[4, rng.choice(V_FULL, 40, replace=False)] = rng.standard_normal(40)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.1, k=[2000, 9000, 50, 0, 30, 0, 1024, 0],
                        p=[1.0, 0.9, 1.0, 0.95, 1.0, 0.9, 1.0, 0.5], n=20, name="hand-over")
    flat_check(w, expect_hand=True, steps=2)


def test_invalid_rows():
    rng = np.random.default_rng(8)
    x = W.peaked_rows(rng, 6, 20_000)
    x[0, 5] = np.nan
    x[1, 7] = np.inf
    x[2] = -np.inf
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=[1.0, 0.0, 1.0, 0.7, 0.0, 1.2],
                        k=[0, 0, 40, 10, 0, 0], p=[0.9, 1.0, 1.0, 1.0, 1.0, 0.8], n=4,
                        name="invalid rows")
    flat_check(w)


@pytest.mark.parametrize("V", [1, 7, 16, 17, 100, 1000, 4097, 50_001, 200_003])
def test_vocab_widths(V):
    rng = np.random.default_rng(V)
    x = W.peaked_rows(rng, 8, V) if V >= 16 else rng.standard_normal((8, V)).astype(np.float32)
    ld = (V + 7) // 8 * 8  # the flat kernels take 16-byte aligned rows
    w = custom_workload(x, dtype=W.DTYPE_BF16, ld=ld, T=[0.0, 0.8, 1.0, 1.3] * 2,
                        k=[0, 5, 0, 0, 0, 50, 0, 2], p=[1.0, 1.0, 0.9, 1.0, 0.7, 0.95, 1.0, 1.0],
                        mp=[0.0, 0.0, 0.0, 0.05, 0.0, 0.0, 0.0, 0.0], n=min(4, V),
                        name=f"V={V}")
    flat_check(w)
