"""Pins for the CPU oracle, each against something other than the oracle itself.

Every ``check_*`` function raises AssertionError when the oracle build it is
handed disagrees with what the pages or the mathematics fix.  The normal tests
run them against the real oracle; ``test_planted_mistakes_are_caught`` runs them
against builds with one planted mistake each (the mutation proofs of the
vllm.cpp Gumbel-draw pull request) and requires every one to go red.

What pins what:
  SplitMix64 finaliser       published known-answer outputs (tests/golden)
  greedy + lowest-index ties numpy.argmax (first occurrence) on constructed ties
  greedy triggers            TensorRT-LLM "Sampling": T=0, top_p=0, top_k=1, min_p=1
  penalties                  hand-worked cases (tests/golden/penalty_cases.txt)
  counts over prompt+output  collections.Counter
  log-softmax                scipy.special.logsumexp; sum exp(lp) = 1; numpy.lexsort
  min-p / top-k / top-p      subset enumeration of the page's definitions on V <= 8,
                             closed form on two-value rows
  noise                      KS test of u against U(0,1); -ln u against Exp(1)
  key schedule               independence, not values: the even and odd 24-bit
                             fields of one hash (16x16 contingency tables over
                             every nibble pairing, 1e6 pairs); rows of one seed
                             and consecutive steps of one row (no shared or
                             shifted stream: value-overlap counts against the
                             n^2 / 2^24 of independent streams, and same-column
                             contingency tables)
  draw formula               chi-square of 1e6 draws against the filtered softmax
Which SplitMix64 output feeds which column, and the log-prob convention, are
this implementation's own reading: the pages fix no value for them, so their
values are parity unpinned; the independence checks above pin the properties a
plausible mistake in the schedule would break.
"""
from __future__ import annotations

import collections
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle as O
from device_token_sampling_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def run_rows(x, *, T=1.0, k=0, p=1.0, mp=0.0, pres=0.0, freq=0.0, rep=1.0, seeds=None,
             prompt=None, output=None, n=0, mutant=None, want_zt=False, first_row=0,
             ignore=None, want_probs=False):
    """Oracle on fp32 rows ``x[B, V]`` with scalar or per-row params."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    B, V = x.shape
    full = lambda v, dt: np.broadcast_to(np.asarray(v, dtype=dt), (B,)).copy()
    if seeds is None:
        seeds = np.arange(1, B + 1, dtype=np.uint64) * np.uint64(0x1234567)
    pi, po = W.csr(prompt if prompt is not None else [np.zeros(0, np.int32)] * B)
    oi, oo = W.csr(output if output is not None else [np.zeros(0, np.int32)] * B)
    return O.sample(x, V, W.DTYPE_F32, full(T, np.float32), full(k, np.int32),
                    full(p, np.float32), full(mp, np.float32), full(pres, np.float32),
                    full(freq, np.float32), full(rep, np.float32),
                    np.asarray(seeds, dtype=np.uint64), pi, po, oi, oo, n, want_zt=want_zt,
                    mutant=mutant, first_row=first_row,
                    prompt_ignore=None if ignore is None else full(ignore, np.int32),
                    want_probs=want_probs)


def total_order(z):
    """Indices by (value descending, index ascending), via numpy.lexsort."""
    idx = np.arange(len(z))
    return np.lexsort((idx, -z.astype(np.float64)))


def kept_by_definition(z, k, p, mp):
    """The kept set of one row from the pages' wording, by subset enumeration.

    min-p: p_i >= min_p * p_max.  top-k: the k most probable survivors.
    top-p: among the survivors renormalised, the smallest set of the
    highest-probability tokens whose total probability exceeds top_p.
    Returns the kept indices in the total order.
    """
    order = list(total_order(z))
    prob = np.exp(z.astype(np.float64) - z.max())
    surv = order
    if 0 < mp < 1:
        surv = [i for i in surv if prob[i] >= mp * prob.max()]
    if 1 < k < len(z):
        surv = surv[:k]
    if 0 < p < 1:
        W_ = sum(prob[i] for i in surv)
        best = None
        for size in range(1, len(surv) + 1):
            for sub in itertools.combinations(surv, size):
                if sum(prob[i] for i in sub) > p * W_:
                    if best is None or sum(prob[i] for i in sub) > sum(prob[i] for i in best):
                        best = sub
            if best is not None:
                break
        surv = [i for i in order if i in best]
    return surv


def read_penalty_cases():
    rows = []
    for line in open(os.path.join(GOLDEN, "penalty_cases.txt")):
        line = line.split("#")[0].strip()
        if line:
            x, c, rep, freq, pres, want = line.split()
            rows.append((float(x), int(c), float(rep), float(freq), float(pres), float(want)))
    return rows


# --------------------------------------------------------------------------
# checks (each usable against a planted-mistake build)
# --------------------------------------------------------------------------

def check_splitmix64(mutant=None):
    lines = [l.split() for l in open(os.path.join(GOLDEN, "splitmix64_seed0.txt"))
             if l.strip() and not l.startswith("#")]
    state = 0
    for _, want in lines:
        state = (state + 0x9E3779B97F4A7C15) % 2**64
        got = O.mix64(state, mutant=mutant)
        assert got == int(want, 16), (hex(got), want)
    assert O.mix64(0, mutant=mutant) == 0  # xorshift and multiply both fix zero


def check_greedy_ties(mutant=None):
    V = 16
    rows, want = [], []
    rows.append(np.full(V, 0.25, np.float32)); want.append(0)            # all equal
    r = np.linspace(-1, 1, V).astype(np.float32); r[5] = r[11] = 3.0
    rows.append(r); want.append(5)                                        # duplicated max
    r = np.zeros(V, np.float32); r[V - 1] = 1.0
    rows.append(r); want.append(V - 1)                                    # max at the end
    r = np.full(V, -np.inf, np.float32); r[9] = -7.0; r[12] = -7.0
    rows.append(r); want.append(9)                                        # -inf mask + tie
    x = np.stack(rows)
    for trig in (dict(T=0.0), dict(k=1), dict(p=0.0), dict(mp=1.0)):
        o = run_rows(x, mutant=mutant, **trig)
        assert (o.status == 0).all()
        assert list(o.token) == want, (trig, list(o.token), want)
        # numpy.argmax returns the first occurrence of the maximum
        assert list(o.token) == [int(np.argmax(rr)) for rr in rows]


def check_greedy_triggers(mutant=None):
    rng = np.random.default_rng(11)
    x = rng.normal(0, 2, size=(40, 300)).astype(np.float32)
    x[:, 7] = x.max(axis=1)  # force ties with the maximum at a low index
    base = [int(np.argmax(r)) for r in x]
    for trig in (dict(T=0.0, k=50, p=0.3, mp=0.2), dict(T=0.7, k=1, p=0.9),
                 dict(T=1.3, p=0.0, k=20), dict(T=0.9, mp=1.0, p=0.5)):
        o = run_rows(x, mutant=mutant, **trig)
        assert list(o.token) == base, trig
        assert (o.greedy == 1).all()
        assert (o.kept_count == 1).all()


def check_penalty_cases(mutant=None):
    for x, c, rep, freq, pres, want in read_penalty_cases():
        row = np.array([[x, 0.5, -0.5, 1.0]], np.float32)
        prompt = [np.array([0] * (c - c // 2), np.int32)]
        output = [np.array([0] * (c // 2), np.int32)]  # split the history across both
        o = run_rows(row, T=1.0, rep=rep, freq=freq, pres=pres, prompt=prompt, output=output,
                     want_zt=True, mutant=mutant)
        got = float(o.zt[0, 0])
        assert got == want, (x, c, rep, freq, pres, got, want)
        assert math.copysign(1.0, got) == math.copysign(1.0, want)
        assert list(o.zt[0, 1:]) == [0.5, -0.5, 1.0]  # unseen tokens untouched


def check_prompt_ignore_cases(mutant=None):
    # TensorRT-LLM "Sampling", occurrence penalties: prompt_ignore_length
    rows = []
    for line in open(os.path.join(GOLDEN, "prompt_ignore_cases.txt")):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    assert len(rows) == 8
    for x, npr, nout, N, rep, freq, pres, want in rows:
        row = np.array([[float(x), 0.5, -0.5, 1.0]], np.float32)
        o = run_rows(row, rep=float(rep), freq=float(freq), pres=float(pres),
                     prompt=[np.zeros(int(npr), np.int32)], output=[np.zeros(int(nout), np.int32)],
                     ignore=int(N), want_zt=True, mutant=mutant)
        assert float(o.zt[0, 0]) == float(want), (x, npr, nout, N, float(o.zt[0, 0]), want)
        assert list(o.zt[0, 1:]) == [0.5, -0.5, 1.0]


def check_counts(mutant=None):
    rng = np.random.default_rng(5)
    V = 64
    x = np.round(rng.normal(0, 3, size=(3, V)), 2).astype(np.float32)
    prompts = [rng.integers(0, V, 40).astype(np.int32) for _ in range(3)]
    outputs = [rng.integers(0, 8, 25).astype(np.int32) for _ in range(3)]
    o = run_rows(x, T=1.0, freq=1.0, prompt=prompts, output=outputs, want_zt=True,
                 mutant=mutant)
    for r in range(3):
        cnt = collections.Counter(list(prompts[r]) + list(outputs[r]))
        got = np.round(x[r].astype(np.float64) - o.zt[r]).astype(int)
        assert [int(g) for g in got] == [cnt.get(j, 0) for j in range(V)], r


def check_logsoftmax(mutant=None):
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2.5, size=(6, 777)).astype(np.float32)
    x[2, ::3] = -np.inf
    o = run_rows(x, T=0.8, n=9, want_zt=True, mutant=mutant)
    for r in range(6):
        z = o.zt[r].astype(np.float64)
        lse = scipy.special.logsumexp(z)
        assert abs(o.lse[r] - lse) <= 1e-12 * max(1.0, abs(lse))
        lp = z - o.lse[r]
        assert abs(np.exp(lp).sum() - 1.0) <= 1e-6
        assert (lp <= 0).all()
        order = total_order(o.zt[r])[:9]
        assert list(o.topn_ids[r]) == list(order)
        np.testing.assert_allclose(o.topn_logprobs[r], lp[order], rtol=0, atol=1e-12)
        assert abs(o.logprob[r] - lp[o.token[r]]) <= 1e-12


def check_filters_bruteforce(mutant=None, trials=400):
    rng = np.random.default_rng(17)
    for t in range(trials):
        V = int(rng.integers(2, 9))
        z = rng.normal(0, 1.5, V).astype(np.float32)
        if t % 7 == 0:
            z[rng.integers(0, V)] = z.max()  # ties with the max
        k = int(rng.choice([0, 2, 3, 4, V]))
        p = float(rng.choice([1.0, rng.uniform(0.05, 0.95)]))
        mp = float(rng.choice([0.0, rng.uniform(0.01, 0.6)]))
        o = run_rows(z[None, :], T=1.0, k=k, p=p, mp=mp, mutant=mutant)
        want = kept_by_definition(z, k, p, mp)
        assert o.kept_count[0] == len(want), (z, k, p, mp, o.kept_count[0], want)
        assert o.kth_index[0] == want[-1]
        assert o.token[0] in want


def check_two_value_closed_form(mutant=None):
    for a, b in ((1.0, 0.0), (0.3, -2.0), (4.0, 3.5)):
        p0 = 1.0 / (1.0 + math.exp(b - a))  # probability of the larger logit
        for p in (p0 * 0.5, p0 - 1e-3, p0 + 1e-3, (1 + p0) / 2):
            o = run_rows(np.array([[b, a]], np.float32), T=1.0, p=p, mutant=mutant)
            assert o.kept_count[0] == (1 if p < p0 else 2), (a, b, p, p0)


def chi_square_case(z, k, p, mp, n_draws, mutant=None, batch=100_000):
    V = len(z)
    kept = kept_by_definition(z, k, p, mp)
    prob = np.zeros(V)
    e = np.exp(z.astype(np.float64) - z.max())
    prob[kept] = e[kept] / e[kept].sum()
    counts = np.zeros(V, np.int64)
    rng = np.random.default_rng(1234)
    done = 0
    while done < n_draws:
        b = min(batch, n_draws - done)
        x = np.broadcast_to(z, (b, V))
        o = run_rows(x, T=1.0, k=k, p=p, mp=mp, mutant=mutant,
                     seeds=rng.integers(0, 2**64, b, dtype=np.uint64), first_row=done)
        counts += np.bincount(o.token, minlength=V)
        done += b
    dropped = [j for j in range(V) if j not in kept]
    assert counts[dropped].sum() == 0
    if len(kept) > 1:
        stat, pval = scipy.stats.chisquare(counts[kept], n_draws * prob[kept])
        assert pval >= 1e-3, (k, p, mp, pval)


Z16 = np.array([2.1, 0.3, -0.7, 1.4, 0.0, -2.2, 1.9, 0.8, -0.1, 0.5, -1.3, 1.1, 0.2, -0.4,
                0.9, -3.0], np.float32)


def _contingency_p(a, b, bins=16):
    """p-value of a chi-square independence test of two nibble streams."""
    t = np.zeros((bins, bins), np.int64)
    np.add.at(t, (a.astype(np.int64), b.astype(np.int64)), 1)
    return scipy.stats.chi2_contingency(t)[1]


def check_pair_fields_independent(mutant=None, n_pairs=1_000_000):
    """The even and odd columns of one hash output use disjoint, independent
    bit fields: every nibble of one field against the top nibble of the other."""
    b = O.noise_bits(0x5EED5EED, 11, 0, 2 * n_pairs, mutant=mutant)
    even, odd = b[0::2], b[1::2]
    for s in range(0, 24, 4):
        assert _contingency_p((even >> s) & 15, odd >> 20) >= 1e-4, ("even nibble", s)
        assert _contingency_p((odd >> s) & 15, even >> 20) >= 1e-4, ("odd nibble", s)


def _streams_independent(b1, b2, tag):
    n = len(b1)
    overlap = len(np.intersect1d(b1, b2))
    expect = n * n / 2**24  # distinct values two independent uniform streams share
    assert overlap < expect + 10 * math.sqrt(expect) + 10, (tag, "overlap", overlap, expect)
    assert _contingency_p(b1 >> 20, b2 >> 20) >= 1e-4, (tag, "same-column nibbles")


def check_rows_independent(mutant=None, n=65_536):
    """Rows of one seed draw independent streams, at any row distance."""
    seed = 0xC0FFEE
    for r in (0, 5, 1024):
        b1 = O.noise_bits(seed, r, 0, n, mutant=mutant)
        for d in (1, 2, 3, 64, 1000):
            _streams_independent(b1, O.noise_bits(seed, r + d, 0, n, mutant=mutant), (r, d))


def check_steps_independent(mutant=None, n=65_536):
    """The stream a row draws after its seed advanced once shares nothing with
    this step's streams of the same or a neighbouring row."""
    seed = 0xABCDEF12345
    nxt = O.next_seed(seed)
    for r in (1, 77):
        b1 = O.noise_bits(seed, r, 0, n, mutant=mutant)
        for r2 in (r - 1, r, r + 1):
            _streams_independent(b1, O.noise_bits(nxt, r2, 0, n, mutant=mutant), (r, r2))
            _streams_independent(O.noise_bits(seed, r2, 0, n, mutant=mutant),
                                 O.noise_bits(nxt, r, 0, n, mutant=mutant), (r2, r))


def check_draw_distribution(mutant=None, n_draws=1_000_000):
    for k, p, mp in ((0, 1.0, 0.0), (8, 1.0, 0.0), (0, 0.5, 0.0), (0, 1.0, 0.1)):
        chi_square_case(Z16, k, p, mp, n_draws, mutant=mutant)


# --------------------------------------------------------------------------
# tests
# --------------------------------------------------------------------------

def test_splitmix64_known_answers(oracle_mod):
    check_splitmix64()


def test_uniform_noise_is_uniform(oracle_mod):
    rng = np.random.default_rng(9)
    us = np.array([O.uniform(int(s), int(r), int(j)) for s, r, j in
                   zip(rng.integers(0, 2**63, 200_000), rng.integers(0, 4096, 200_000),
                       rng.integers(0, 300_000, 200_000))])
    assert (us > 0).all() and (us < 1).all()
    b = us * 2**24 - 0.5
    assert np.array_equal(b, np.round(b))  # (b + 1/2) / 2^24 exactly
    assert scipy.stats.kstest(us, "uniform").pvalue >= 1e-3
    assert scipy.stats.kstest(-np.log(us), "expon").pvalue >= 1e-3
    # neighbouring columns share one hash output but are not equal
    pair = [(O.uniform(77, 3, 2 * i), O.uniform(77, 3, 2 * i + 1)) for i in range(2000)]
    assert sum(a == c for a, c in pair) <= 2


def test_noise_bits_match_uniforms(oracle_mod):
    b = O.noise_bits(123, 4, 1000, 64)
    for i in range(64):
        assert O.uniform(123, 4, 1000 + i) == (float(b[i]) + 0.5) / 2**24


def test_pair_fields_independent(oracle_mod):
    check_pair_fields_independent()


def test_rows_of_one_seed_independent(oracle_mod):
    check_rows_independent()


def test_steps_of_one_row_independent(oracle_mod):
    check_steps_independent()


def test_greedy_lowest_index_ties(oracle_mod):
    check_greedy_ties()


def test_greedy_triggers(oracle_mod):
    check_greedy_triggers()


def test_invalid_rows(oracle_mod):
    V = 8
    x = np.zeros((4, V), np.float32)
    x[0, 3] = np.nan
    x[1, 5] = np.inf
    x[2, :] = -np.inf
    x[3, 2] = 1e38  # overflows to +inf once divided by T = 0.1
    for T in (0.0, 1.0):
        o = run_rows(x[:3], T=T, n=3)
        assert list(o.status) == [1, 1, 2]
        assert list(o.token) == [-1, -1, -1]
        assert (o.topn_ids == -1).all()
    o = run_rows(x[3:], T=0.1)
    assert o.status[0] == 1


def test_unfiltered_row_keeps_every_finite_token(oracle_mod):
    rng = np.random.default_rng(4)
    V = 500
    x = rng.normal(0, 1, size=(5, V)).astype(np.float32)
    x[1, ::4] = -np.inf
    x[3, 10:20] = x[3].min()  # ties at the bottom of the order
    g = run_rows(x, T=0.0, n=4)
    for kk in (0, V):
        o = run_rows(x, T=1.0, k=kk, p=1.0, mp=0.0, n=4)
        fin = np.isfinite(x).sum(axis=1)
        assert list(o.kept_count) == list(fin)
        for r in range(5):
            mn = x[r][np.isfinite(x[r])].min()
            assert o.kth_value[r] == mn
            assert o.kth_index[r] == int(np.nonzero(x[r] == mn)[0].max())
        # T = 1 and the greedy route share one distribution: same log-probs
        np.testing.assert_allclose(o.lse, g.lse, rtol=0, atol=0)
        np.testing.assert_array_equal(o.topn_ids, g.topn_ids)


def test_top_k_one_and_temperature_zero_agree(oracle_mod):
    w = W.tiny()
    x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(w.logits))
    a = run_rows(x, T=0.0, n=5)
    b = run_rows(x, T=0.6, k=1, n=5)
    np.testing.assert_array_equal(a.token, b.token)
    np.testing.assert_array_equal(a.topn_ids, b.topn_ids)
    np.testing.assert_allclose(a.topn_logprobs, b.topn_logprobs, rtol=0, atol=0)


def test_penalty_hand_cases(oracle_mod):
    check_penalty_cases()


def test_counts_match_counter(oracle_mod):
    check_counts()


def test_repetition_above_one_pushes_seen_tokens_down(oracle_mod):
    rng = np.random.default_rng(8)
    V = 400
    x = rng.normal(0, 3, size=(2, V)).astype(np.float32)
    hist = [rng.integers(0, V, 100).astype(np.int32) for _ in range(2)]
    o = run_rows(x, T=1.0, rep=1.3, freq=0.1, pres=0.2, prompt=hist, want_zt=True)
    for r in range(2):
        seen = np.zeros(V, bool)
        seen[hist[r]] = True
        assert (o.zt[r][seen] < x[r][seen]).all()
        assert np.array_equal(o.zt[r][~seen], x[r][~seen])


def test_log_softmax(oracle_mod):
    check_logsoftmax()


def test_filters_against_subset_enumeration(oracle_mod):
    check_filters_bruteforce()


def test_top_p_two_value_closed_form(oracle_mod):
    check_two_value_closed_form()


def test_draw_frequencies_chi_square(oracle_mod):
    check_draw_distribution()


def test_temperature_scales_logits(oracle_mod):
    x = np.array([[1.5, -2.0, 0.25, 3.0]], np.float32)
    o = run_rows(x, T=0.5, want_zt=True)
    assert list(o.zt[0]) == [3.0, -4.0, 0.5, 6.0]  # 1.0f/0.5f = 2, exact products


def test_determinism_and_seed_advance(oracle_mod):
    w = W.tiny()
    a = O.sample_workload(w)
    b = O.sample_workload(w)
    np.testing.assert_array_equal(a.token, b.token)
    s = int(w.seed[1])
    assert O.next_seed(s) == (s + 0x9E3779B97F4A7C15) % 2**64
    # the draw depends on the row index as well as the seed
    x = np.broadcast_to(Z16, (64, 16))
    o = run_rows(x, T=1.0, seeds=np.full(64, 99, np.uint64))
    assert len(set(o.token)) > 4


def test_rejects_bad_arguments(oracle_mod):
    x = np.zeros((1, 4), np.float32)
    for bad in (dict(T=-1.0), dict(T=np.nan), dict(k=-1), dict(p=1.5), dict(mp=-0.1),
                dict(rep=0.0), dict(pres=np.inf)):
        with pytest.raises(ValueError):
            run_rows(x, **bad)
    with pytest.raises(ValueError):
        run_rows(x, prompt=[np.array([4], np.int32)])


def test_workload_configs_are_valid_and_sampled(oracle_mod):
    w = W.tiny()
    o = O.sample_workload(w, want_zt=True)
    assert list(o.status) == [0, 0, 0, 0]
    assert list(o.greedy) == [1, 0, 0, 0]
    assert o.kept_count[2] <= 8
    assert o.kept_count[3] >= 1
    # row 3 is penalised; the others are not
    assert np.array_equal(o.zt[0], w.logits[0])
    assert not np.array_equal(o.zt[3], w.logits[3])


MUTANT_CHECKS = {
    "HASH": [check_splitmix64],
    "TIE_HIGH": [check_greedy_ties],
    "PEN_ORDER": [check_penalty_cases],
    "PROMPT_ONLY": [check_counts],
    "TOPP_INCL": [check_filters_bruteforce, check_two_value_closed_form],
    "TOPP_NO_RENORM": [check_filters_bruteforce],
    "SCORE_MUL": [lambda mutant: check_draw_distribution(mutant, n_draws=200_000)],
    "IGNORE_ALL": [check_prompt_ignore_cases],
    "PAIR_OVERLAP": [check_pair_fields_independent],
    "ROW_IGNORED": [check_rows_independent],
    "STEP_IS_ROW": [check_rows_independent, check_steps_independent],
}


@pytest.mark.parametrize("mutant", sorted(MUTANT_CHECKS))
def test_planted_mistakes_are_caught(oracle_mod, mutant):
    O.build(mutant)
    for chk in MUTANT_CHECKS[mutant]:
        with pytest.raises(AssertionError):
            chk(mutant=mutant)


# --------------------------------------------------------------------------
# prompt_ignore_length, the filtered distribution, top-p decay
# --------------------------------------------------------------------------

def test_prompt_ignore_hand_cases(oracle_mod):
    check_prompt_ignore_cases()


def test_prompt_ignore_token_only_in_the_ignored_prefix(oracle_mod):
    # token 1 only in the ignored prefix: repetition alone; token 2 once after
    # it: all three penalties; token 3 unseen
    row = np.array([[0.0, 3.0, 3.0, 3.0]], np.float32)
    o = run_rows(row, rep=2.0, freq=0.5, pres=0.25, prompt=[np.array([1, 1, 2], np.int32)],
                 ignore=2, want_zt=True)
    assert list(o.zt[0]) == [0.0, 1.5, 0.75, 3.0]  # 3/2 ; 3/2 - 0.5 - 0.25 ; untouched


def test_prompt_ignore_zero_matches_no_ignore(oracle_mod):
    rng = np.random.default_rng(31)
    x = rng.normal(0, 2, size=(3, 200)).astype(np.float32)
    pr = [rng.integers(0, 200, 50).astype(np.int32) for _ in range(3)]
    ou = [rng.integers(0, 200, 20).astype(np.int32) for _ in range(3)]
    a = run_rows(x, rep=1.2, freq=0.3, pres=0.4, prompt=pr, output=ou, want_zt=True, n=4)
    b = run_rows(x, rep=1.2, freq=0.3, pres=0.4, prompt=pr, output=ou, want_zt=True, n=4,
                 ignore=[0, -5, 0])
    assert np.array_equal(a.zt, b.zt) and np.array_equal(a.token, b.token)


def check_probs(mutant=None):
    rng = np.random.default_rng(41)
    for trial in range(60):
        V = int(rng.integers(3, 9))
        z = np.round(rng.normal(0, 1.5, size=(1, V)), 1).astype(np.float32)
        k = int(rng.choice([0, 2, V - 1, V]))  # k == 1 is the greedy route, checked apart
        p = float(rng.choice([1.0, 0.3, 0.6, 0.9]))
        mp = float(rng.choice([0.0, 0.1, 0.4]))
        o = run_rows(z, k=k, p=p, mp=mp, want_probs=True, want_zt=True, mutant=mutant)
        if o.topp_near[0]:
            continue
        kept = kept_by_definition(o.zt[0], k, p, mp)
        pr = o.probs[0]
        assert set(np.nonzero(pr)[0]) == set(kept), (trial, kept, pr)
        assert abs(pr.sum() - 1.0) <= 1e-12
        i0 = kept[0]
        for i in kept:  # each kept token's weight relative to the most probable one
            assert abs(pr[i] / pr[i0] - math.exp(float(o.zt[0, i]) - float(o.zt[0, i0]))) <= 1e-12


def test_filtered_distribution_by_definition(oracle_mod):
    # TensorRT-LLM "Sampling", Performance: the sampling probabilities after the
    # top-k / top-p masking, i.e. the kept set renormalised
    check_probs()


def test_filtered_distribution_greedy_and_helper(oracle_mod):
    rng = np.random.default_rng(43)
    z = rng.normal(0, 1, size=(2, 50)).astype(np.float32)
    g = run_rows(z, T=0.0, want_probs=True)
    for r in range(2):
        assert g.probs[r, g.token[r]] == 1.0 and g.probs[r].sum() == 1.0
    o = run_rows(z, T=0.7, k=10, p=0.8, want_probs=True, want_zt=True)
    for r in range(2):
        np.testing.assert_array_equal(O.filtered_probs(o.zt[r], o.kept_count[r]), o.probs[r])
    bad = z.copy()
    bad[0, 3] = np.nan
    b = run_rows(bad, T=1.0, want_probs=True)
    assert np.isnan(b.probs[0]).all() and not np.isnan(b.probs[1]).any()


def test_topp_decay_steps(oracle_mod):
    # TensorRT-LLM "Sampling", Top-P decay: multiplied by the decay after every
    # sampled token, bounded below by top_p_min, reset to the initial top_p
    # when the token top_p_reset_ids is sampled (-1 never matches)
    p, seq = 0.5, []
    for tok in [3, 3, 3, 7, 3]:
        p = O.topp_decay(p, 0.5, 0.5, 0.1, 7, tok)
        seq.append(p)
    assert seq == [0.25, 0.125, float(np.float32(0.1)), 0.5, 0.25]
    assert O.topp_decay(0.3, 0.9, 1.0, 1e-6, -1, 0) == float(np.float32(0.3))
    assert O.topp_decay(0.3, 0.9, 0.5, 1e-6, -1, -1) == float(np.float32(0.9))
