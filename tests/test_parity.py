"""GPU parity: the CUDA sampler (through the C ABI) against the CPU oracle,
element by element, on seeded synthetic inputs.  Sizes span several CTAs and
thread-block clusters with ragged tails; the named workloads run at their full
sizes in the launch configuration the benchmark times."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from device_token_sampling_gb300 import workloads as W

from paritylib import check_workload, compare, custom_workload, make_sampler, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def rng_rows(B, V, seed=0, sigma=2.0):
    return np.random.default_rng(seed).normal(0, sigma, size=(B, V)).astype(np.float32)


# --------------------------------------------------------------------------
# the named workloads
# --------------------------------------------------------------------------

def test_tiny():
    check_workload(W.tiny())


@pytest.mark.parametrize("greedy", [False, True])
def test_b32(greedy):
    check_workload(W.b32(greedy=greedy))


def test_b64_penalties():
    check_workload(W.b64())


def test_b256_mixed():
    check_workload(W.b256())


def test_large_sampled_rows():
    w = W.large()
    rows = np.arange(0, w.B, 37)
    check_workload(w, rows=rows)


# --------------------------------------------------------------------------
# shapes: ragged tails, several CTAs per row, padded and unaligned strides
# --------------------------------------------------------------------------

@pytest.mark.parametrize("V", [1, 7, 16, 17, 100, 1000, 4097, 12_289, 50_001, 200_003])
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_vocab_widths(V, dtype):
    B = 6
    x = rng_rows(B, V, seed=V)
    w = custom_workload(x, dtype=dtype, T=[0.0, 0.9, 1.2, 0.7, 1.0, 0.5][:B],
                        k=[0, 0, 5, 0, 40, 3], p=[1.0, 1.0, 1.0, 0.8, 0.9, 1.0],
                        mp=[0.0, 0.0, 0.0, 0.0, 0.0, 0.2], n=min(5, V), name=f"V{V}")
    check_workload(w)


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("pad", [0, 1, 3, 8, 64])
def test_row_stride_padding_and_alignment(dtype, pad):
    V = 30_000 + 5
    x = rng_rows(4, V, seed=pad)
    w = custom_workload(x, dtype=dtype, ld=V + pad, T=[0.0, 1.0, 0.8, 1.1], k=[0, 20, 0, 0],
                        p=[1.0, 0.9, 0.7, 1.0], n=4, name=f"pad{pad}")
    check_workload(w)


# --------------------------------------------------------------------------
# ties, masks and invalid rows
# --------------------------------------------------------------------------

def test_ties_and_masks():
    V = 40_000
    x = rng_rows(8, V, seed=3)
    x[0, :] = 0.5                          # all equal
    x[1, [17, 19_000, 39_999]] = 9.0       # duplicated max across CTAs
    x[2, :] = -np.inf
    x[2, [5, 30_000]] = 1.0                # -inf mask, tie among two
    x[3, ::2] = -np.inf                    # half masked
    x[4, V - 1] = 50.0                     # max at the very end
    x[5, :100] = 3.0                       # 100-way tie at the top
    x[6, :] = np.round(x[6, :], 1)         # many ties everywhere
    x[7, :] = 2.0
    x[7, 12_345] = 2.5
    for T in (0.0, 1.0):
        for k, p in ((0, 1.0), (50, 1.0), (0, 0.6), (3, 0.9)):
            w = custom_workload(x, T=T, k=k, p=p, n=8, name=f"ties T{T} k{k} p{p}")
            check_workload(w)


def test_invalid_rows():
    V = 5000
    x = rng_rows(5, V, seed=4)
    x[0, 77] = np.nan
    x[1, 4000] = np.inf
    x[2, :] = -np.inf
    x[3, 10] = 3e38  # overflows to +inf once multiplied by 1/T
    for T in (0.0, 0.1):
        w = custom_workload(x, T=T, n=3, name=f"invalid T{T}")
        check_workload(w)


def test_fewer_finite_than_logprobs():
    V = 3000
    x = np.full((2, V), -np.inf, np.float32)
    x[0, [3, 2999]] = [1.0, 2.0]
    x[1, 1500] = 0.0
    for T in (0.0, 1.0):
        w = custom_workload(x, T=T, n=6, name="sparse")
        check_workload(w)


# --------------------------------------------------------------------------
# strategies
# --------------------------------------------------------------------------

@pytest.mark.parametrize("trig", [dict(T=0.0, k=50, p=0.3), dict(T=0.7, k=1),
                                  dict(T=1.3, p=0.0), dict(T=0.9, mp=1.0)])
def test_greedy_triggers(trig):
    x = rng_rows(8, 70_000, seed=9)
    w = custom_workload(x, n=5, **trig)
    g, o = check_workload(w)
    assert (o.greedy == 1).all()


@pytest.mark.parametrize("k", [2, 20, 300, 1024, 2047, 3000, 9000])
def test_top_k(k):
    x = W.peaked_rows(np.random.default_rng(k), 8, 151_936)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.0, k=k, n=4, name=f"topk{k}")
    check_workload(w)


@pytest.mark.parametrize("T,p", [(0.3, 0.5), (0.7, 0.9), (1.0, 0.95), (1.5, 0.5), (1.5, 0.99)])
def test_top_p(T, p):
    x = W.peaked_rows(np.random.default_rng(int(T * 100 + p * 1000)), 6, 151_936)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=T, p=p, n=2, name=f"topp T{T} p{p}")
    check_workload(w)


@pytest.mark.parametrize("mp", [0.01, 0.05, 0.3])
@pytest.mark.parametrize("combo", ["minp", "minp+k", "minp+p", "minp+k+p"])
def test_min_p_combos(mp, combo):
    x = W.peaked_rows(np.random.default_rng(5), 6, 100_000)
    kw = dict(mp=mp, T=1.2)
    if "k" in combo:
        kw["k"] = 400
    if "p" in combo:
        kw["p"] = 0.9
    w = custom_workload(x, n=3, name=f"{combo} {mp}", **kw)
    check_workload(w)


def test_unfiltered_draw():
    x = rng_rows(6, 120_000, seed=12, sigma=1.0)
    for kk in (0, 120_000):
        w = custom_workload(x, T=1.0, k=kk, p=1.0, mp=0.0, n=3, name="unfiltered")
        check_workload(w)


# --------------------------------------------------------------------------
# penalties
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_penalties(dtype):
    rng = np.random.default_rng(21)
    B, V = 6, 90_000
    x = rng_rows(B, V, seed=22)
    prompt = [W.zipf_ids(rng, 700, V) for _ in range(B)]
    output = [np.concatenate([W.zipf_ids(rng, 200, V), [0, V - 1, 45_000]]).astype(np.int32)
              for _ in range(B)]
    w = custom_workload(x, dtype=dtype, T=[0.0, 1.0, 0.8, 1.0, 0.6, 1.4], k=[0, 0, 30, 0, 5, 0],
                        p=[1.0, 0.9, 1.0, 1.0, 0.8, 0.95], mp=[0, 0, 0, 0.05, 0, 0],
                        pres=[0.5, 0.0, 1.0, -0.5, 0.3, 0.2], freq=[0.3, 0.2, 0.0, 0.1, 0.0, 0.5],
                        rep=[1.2, 1.0, 0.8, 1.3, 2.0, 1.05], prompt=prompt, output=output, n=5,
                        name="pen")
    check_workload(w)


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_dense_penalties(dtype):
    """Histories that cover most of the row: a slice then holds more penalised
    values than the kernels keep in shared memory (2048), and they go to the
    row's side list in global memory instead; beside them, rows whose
    penalised values fit."""
    rng = np.random.default_rng(23)
    B, V = 4, 150_000
    x = rng_rows(B, V, seed=24)
    # (at most 32,768 ids a row; contiguous id ranges make whole slices dense)
    prompt = [rng.permutation(30_000).astype(np.int32),                # ids 0 .. 29,999
              np.arange(V - 30_000, V, dtype=np.int32),                 # the last 30,000 ids
              W.zipf_ids(rng, 3000, V),
              np.repeat(np.arange(60_000, 76_000, dtype=np.int32), 2)]  # 16,000 ids, twice
    output = [rng.integers(0, V, 50).astype(np.int32) for _ in range(B)]
    w = custom_workload(x, dtype=dtype, T=[1.0, 0.7, 1.2, 0.0], k=[0, 40, 0, 0],
                        p=[0.9, 1.0, 0.95, 1.0], mp=[0.0, 0.0, 0.05, 0.0],
                        pres=[0.4, 0.2, 0.5, 0.3], freq=[0.1, 0.3, 0.2, 0.0],
                        rep=[1.1, 1.3, 0.9, 1.2], prompt=prompt, output=output, n=4,
                        name="dense pen")
    check_workload(w)


def test_counts_table_matches_history():
    rng = np.random.default_rng(31)
    B, V = 5, 20_000
    prompt = [W.zipf_ids(rng, int(rng.integers(0, 900)), V) for _ in range(B)]
    output = [rng.integers(0, V, int(rng.integers(0, 300))).astype(np.int32) for _ in range(B)]
    w = custom_workload(rng_rows(B, V), pres=0.1, prompt=prompt, output=output)
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        torch.cuda.synchronize()
        for r in range(B):
            ids, cnt = s.counts(r)
            u, c = np.unique(np.concatenate([prompt[r], output[r]]), return_counts=True)
            np.testing.assert_array_equal(ids, u)
            np.testing.assert_array_equal(cnt, c)
    finally:
        s.close()


# --------------------------------------------------------------------------
# multi-step decode: seeds advance, counts append, teacher-forced parity
# --------------------------------------------------------------------------

def test_multi_step_teacher_forced():
    rng = np.random.default_rng(41)
    B, V, steps = 8, 60_000, 6
    prompt = [W.zipf_ids(rng, 300, V) for _ in range(B)]
    w = custom_workload(rng_rows(B, V, seed=42), T=0.9, k=[0, 10, 0, 50, 5, 0, 200, 3],
                        p=[0.9, 1.0, 0.8, 0.95, 1.0, 1.0, 0.9, 0.5], mp=0.02, pres=0.4, freq=0.2,
                        rep=1.05, prompt=prompt, n=5, name="decode")
    s = make_sampler(w, max_history=512)
    try:
        s.reset_workload(w)
        seeds = w.seed.copy()
        outputs = [np.zeros(0, np.int32) for _ in range(B)]
        for t in range(steps):
            x = rng_rows(B, V, seed=100 + t)
            wt = custom_workload(x, T=w.temperature, k=w.top_k, p=w.top_p, mp=w.min_p,
                                 pres=w.presence, freq=w.frequency, rep=w.repetition,
                                 prompt=prompt, output=outputs, n=5, name=f"step{t}")
            wt.seed = seeds
            g = run_gpu(s, wt, update_counts=True, reset=False)
            o = O.sample_workload(wt, want_zt=True)
            compare(g, o, where=f"step {t}")
            outputs = [np.concatenate([outputs[r], [g["token"][r]]]).astype(np.int32)
                       for r in range(B)]
            seeds = np.array([O.next_seed(int(v)) for v in seeds], np.uint64)
            np.testing.assert_array_equal(s.seeds(B), seeds)
        for r in range(B):
            ids, cnt = s.counts(r)
            u, c = np.unique(np.concatenate([prompt[r], outputs[r]]), return_counts=True)
            np.testing.assert_array_equal(ids, u)
            np.testing.assert_array_equal(cnt, c)
    finally:
        s.close()


def test_determinism():
    w = W.b256()
    s = make_sampler(w)
    try:
        a = run_gpu(s, w)
        b = run_gpu(s, w)
        for k in a:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    finally:
        s.close()
