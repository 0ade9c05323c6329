"""The GPU draw against the distribution it samples, statistically: one full
row (V = 151,936 bf16, peaked) repeated over 4096 rows with independent seeds,
drawn over many calls (the seeds advance), and the token frequencies compared
with the filtered softmax by a chi-square test [TensorRT-LLM "Sampling":
top-k, top-p over the survivors renormalised; vllm.cpp pull request: a
Gumbel-max draw samples the softmax of the kept logits].  Bit-exact parity with
the oracle pins the formula on unflagged rows; this checks the whole draw path
end to end over many seeds, on both sampling paths and on the vocabulary
split."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
scipy_stats = pytest.importorskip("scipy.stats")

import oracle as O
from device_token_sampling_gb300 import workloads as W

from paritylib import custom_workload, device_logits, make_sampler

pytestmark = pytest.mark.gpu

V = 151_936
ROWS = 4096
CALLS = 25


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def filtered(x, T, k, p):
    o = O.sample_workload(custom_workload(x, dtype=W.DTYPE_BF16, T=T, k=k, p=p, name="one row"),
                          want_zt=True)
    return O.filtered_probs(o.zt[0], int(o.kept_count[0]))


def one_row_case(T, k, p):
    """The repeated workload, its filtered softmax, and the filtered softmax
    at a temperature 10 % higher (a plausible mistake the test must reject)."""
    rng = np.random.default_rng(int(T * 100) + k)
    x = W.peaked_rows(rng, 1, V)
    wb = custom_workload(np.repeat(x, ROWS, axis=0), dtype=W.DTYPE_BF16, T=T, k=k, p=p,
                         seed=int(rng.integers(1 << 30)), name=f"stats T{T} k{k} p{p}")
    return wb, filtered(x, T, k, p), filtered(x, T * 1.1, k, p)


def binned_chi_square(tokens, prob, bins=40):
    """Chi-square of the draws against `prob`, over bins of about equal
    expected mass (tokens in the order of decreasing probability)."""
    kept = np.flatnonzero(prob > 0)
    order = kept[np.argsort(-prob[kept], kind="stable")]
    cum = np.cumsum(prob[order])
    edges = np.searchsorted(cum, np.linspace(0, 1, bins + 1)[1:-1])
    bin_of = np.zeros(len(prob), np.int64)
    bin_of[order] = np.searchsorted(edges, np.arange(len(order)), side="right")
    expected = np.bincount(bin_of[order], weights=prob[order], minlength=bins)
    nz = expected > 0
    assert np.all(prob[tokens] > 0), "a token outside the kept set"
    counts = np.bincount(bin_of[tokens], minlength=bins)
    return scipy_stats.chisquare(counts[nz], len(tokens) * expected[nz] / expected[nz].sum())


def draws(w, path=None, shards=0, K=256):
    s = make_sampler(w)
    toks = []
    try:
        if path:
            s.set_path(path)
        s.reset_workload(w)
        x = device_logits(w)
        edges = np.linspace(0, w.V, shards + 1).astype(int) if shards else None
        for _ in range(CALLS):
            if shards:
                parts = torch.stack([s.shard_partials(x[:, edges[i]:edges[i + 1]], int(edges[i]),
                                                      w.V, K) for i in range(shards)])
                tok = s.shard_merge(parts, w.V, K, 0)[0]
            else:
                tok = s.sample(x, V=w.V, num_logprobs=0, dtype=W.DTYPE_BF16)[0]
            toks.append(tok.cpu().numpy())
        torch.cuda.synchronize()
        s.check_device_errors()
    finally:
        s.close()
    return np.concatenate(toks)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("T,k,p", [(1.0, 50, 1.0), (1.5, 0, 0.9), (0.8, 200, 0.95)])
def test_draw_frequencies_match_the_filtered_softmax(path, T, k, p):
    w, prob, wrong = one_row_case(T, k, p)
    tokens = draws(w, path=path)
    stat, pval = binned_chi_square(tokens, prob)
    assert pval > 1e-4, (stat, pval)
    # the same draws reject the softmax at T * 1.1 (the test has power): by a
    # token outside its kept set, or by the chi-square
    assert not np.all(wrong[tokens] > 0) or binned_chi_square(tokens, wrong)[1] < 1e-6


@pytest.mark.parametrize("T,k,p", [(1.2, 200, 0.9), (1.0, 0, 1.0)])
def test_vocabulary_split_draw_frequencies(T, k, p):
    """Bounded rows draw over the merged records; a row without a filter is
    the best of the shards' own Gumbel winners over every column."""
    w, prob, wrong = one_row_case(T, k, p)
    tokens = draws(w, shards=4)
    stat, pval = binned_chi_square(tokens, prob)
    assert pval > 1e-4, (stat, pval)
    assert not np.all(wrong[tokens] > 0) or binned_chi_square(tokens, wrong)[1] < 1e-6
