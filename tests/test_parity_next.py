"""GPU parity of the features ranked next on the sampling path (TensorRT-LLM
"Sampling" page): prompt_ignore_length in the occurrence counts, the top-p
decay state, and the filtered distribution on request.  Each compares the
CUDA path through the C ABI with the CPU oracle on seeded inputs."""
from __future__ import annotations

import collections

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from device_token_sampling_gb300 import workloads as W

from paritylib import (check_workload, compare, custom_workload, device_logits, make_sampler,
                       run_gpu)

pytestmark = pytest.mark.gpu

V_FULL = 151_936


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def history(rng, B, V, n_prompt, n_output):
    prompt = [W.zipf_ids(rng, n_prompt, V) for _ in range(B)]
    output = [W.zipf_ids(rng, n_output, V) for _ in range(B)]
    return prompt, output


# --------------------------------------------------------------------------
# prompt_ignore_length
# --------------------------------------------------------------------------

IGNORE = [0, 1, 50, 199, 200, 500, -3, 100]


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_prompt_ignore_length(dtype):
    rng = np.random.default_rng(61)
    B, V = len(IGNORE), 30_011
    x = rng.normal(0, 2.0, size=(B, V)).astype(np.float32)
    prompt, output = history(rng, B, V, 200, 60)
    w = custom_workload(x, dtype=dtype, T=[0.0, 0.8, 1.0, 1.2, 0.9, 1.0, 0.7, 1.1],
                        k=[0, 40, 0, 0, 100, 0, 0, 20], p=[1.0, 0.9, 0.8, 1.0, 0.95, 0.7, 1.0, 0.9],
                        pres=0.6, freq=0.4, rep=1.3, n=5, prompt=prompt, output=output,
                        name="prompt ignore")
    w.prompt_ignore = np.array(IGNORE, np.int32)
    check_workload(w)


def test_prompt_ignore_counts_table():
    rng = np.random.default_rng(62)
    B, V = len(IGNORE), 20_000
    prompt, output = history(rng, B, V, 200, 40)
    w = custom_workload(rng.normal(0, 1, size=(B, V)), pres=0.1, prompt=prompt, output=output)
    w.prompt_ignore = np.array(IGNORE, np.int32)
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        torch.cuda.synchronize()
        for r in range(B):
            ids, cnt = s.counts(r)
            skip = min(max(IGNORE[r], 0), len(prompt[r]))
            counted = collections.Counter(list(prompt[r][skip:]) + list(output[r]))
            seen = np.unique(np.concatenate([prompt[r], output[r]]))
            np.testing.assert_array_equal(ids, seen)  # every seen id, for repetition
            np.testing.assert_array_equal(cnt, [counted.get(int(i), 0) for i in ids])
    finally:
        s.close()


# --------------------------------------------------------------------------
# top-p decay
# --------------------------------------------------------------------------

# per row: T, top_k, initial top_p, decay, top_p_min, reset id (-1: never)
DECAY_ROWS = [
    (1.0, 0, 1.0, 0.9, 1e-6, -1),    # top_p unset: decay alone makes it a top-p row
    (1.2, 0, 0.95, 0.5, 0.3, 17),    # floor reached at step 2, then a reset
    (0.9, 0, 0.9, 0.5, 1e-6, 17),    # toward the floor: nearly greedy
    (1.1, 50, 0.99, 0.7, 0.2, 17),   # top-k then the decayed top-p
    (0.0, 0, 0.9, 0.5, 0.1, -1),     # greedy takes precedence: no decay
    (1.0, 0, 0.8, 1.0, 0.5, 17),     # decay 1: off
    (1.3, 0, 0.7, 0.95, 0.6, -1),    # slow decay, never reset
    (1.0, 1, 0.9, 0.5, 0.1, 17),     # top_k = 1 is greedy: no decay
]
RESET_STEPS = (3, 6)  # steps whose logits make the reset id (17) the clear winner


def decay_step_logits(rng, B, V, step):
    x = W.peaked_rows(rng, B, V)
    if step in RESET_STEPS:
        x[:, 17] = x.max(axis=1) + 12.0
    return x


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_top_p_decay_steps(dtype):
    """Eight calls on one handle: each call samples with the effective top_p the
    state holds, which must follow the oracle's decay rule bit for bit."""
    rng = np.random.default_rng(63)
    B, V, steps = len(DECAY_ROWS), 40_000, 8
    T, k, p0, decay, pmin, reset = (np.array(c) for c in zip(*DECAY_ROWS))
    x0 = decay_step_logits(rng, B, V, 0)
    w = custom_workload(x0, dtype=dtype, T=T, k=k, p=p0, n=4, name="top-p decay")
    s = make_sampler(w)
    try:
        s.reset_params(w.temperature, w.top_k, w.top_p, w.min_p, w.presence, w.frequency,
                       w.repetition, w.seed, top_p_decay=decay.astype(np.float32),
                       top_p_min=pmin.astype(np.float32), top_p_reset_ids=reset.astype(np.int32))
        s.reset_token_counts(w.prompt_ids, w.prompt_offsets, w.output_ids, w.output_offsets)
        active = (decay < 1.0) & (T > 0.0) & (k != 1)
        p_eff = p0.astype(np.float32).copy()
        seed = w.seed.copy()
        resets = 0
        for step in range(steps):
            np.testing.assert_array_equal(s.top_p(B), p_eff, err_msg=f"step {step}")
            x = x0 if step == 0 else decay_step_logits(rng, B, V, step)
            ws = custom_workload(x, dtype=dtype, T=T, k=k, p=p0, n=4, name=f"decay step {step}")
            ws.seed = seed.copy()
            g = run_gpu(s, ws, reset=False)
            o = O.sample_workload(ws, want_zt=True, top_p=p_eff)
            compare(g, o, where=ws.name)
            for r in np.flatnonzero(active):
                if g["status"][r] == 0:
                    resets += int(g["token"][r] == reset[r])
                    p_eff[r] = O.topp_decay(float(p_eff[r]), float(p0[r]), float(decay[r]),
                                            float(pmin[r]), int(reset[r]), int(g["token"][r]))
            seed = np.array([O.next_seed(int(v)) for v in seed], np.uint64)
        np.testing.assert_array_equal(s.top_p(B), p_eff, err_msg="after the last step")
        np.testing.assert_array_equal(s.seeds(B), seed)
        assert resets >= 4, "the reset id was drawn too rarely to test the reset"
        assert p_eff[6] == np.float32(0.6)  # the floor
    finally:
        s.close()


def test_top_p_decay_rejects_out_of_range():
    rng = np.random.default_rng(64)
    w = custom_workload(rng.normal(0, 1, size=(2, 1000)), p=0.9)
    s = make_sampler(w)
    try:
        base = (w.temperature, w.top_k, w.top_p, w.min_p, w.presence, w.frequency, w.repetition,
                w.seed)
        for kw in (dict(top_p_decay=[0.0, 0.9]), dict(top_p_decay=[1.5, 0.9]),
                   dict(top_p_min=[0.0, 0.5]), dict(top_p_min=[0.5, 1.01]),
                   dict(top_p_reset_ids=[-2, 3])):
            with pytest.raises(Exception, match="VT_ERR_INVALID_ARG|out of range|not in|< -1"):
                s.reset_params(*base, **{kk: np.asarray(v) for kk, v in kw.items()})
        # defaults: decay 0.5 alone, floor 1e-6, no reset id
        s.reset_params(*base, top_p_decay=np.array([0.5, 1.0], np.float32))
        np.testing.assert_array_equal(s.top_p(2), np.float32([0.9, 0.9]))
    finally:
        s.close()


# --------------------------------------------------------------------------
# the filtered distribution on request
# --------------------------------------------------------------------------

# fp32 arithmetic against the oracle's double: the exponent argument z_t - m
# is rounded once (relative error |z_t - m| 2^-24, at most about 6e-6 where
# the probability is still a normal fp32 number), expf adds a few ulp, the
# kept set's exp-sum a relative error that grows with the terms a thread
# adds in sequence (about 150 here, 9e-6 at worst); the bound takes 3e-5.
PROBS_RTOL = 3e-5
PROBS_ATOL = 1e-37  # below the smallest normal fp32 number the relative bound stops


def sample_with_probs(s, w, x=None, update_counts=False, ld_probs=None):
    if x is None:
        x = device_logits(w)
    dt = W.DTYPE_BF16 if w.dtype == W.DTYPE_BF16 else W.DTYPE_F32
    ldp = w.V if ld_probs is None else ld_probs
    probs = torch.full((w.B, ldp), -7.0, dtype=torch.float32, device=x.device)
    tok, lp, tid, tlp = s.sample(x, V=w.V, num_logprobs=w.num_logprobs,
                                 update_counts=update_counts, dtype=dt, probs=probs)
    st = s.row_status(w.B)
    kv, ki, kept = s.filter_boundary(w.B)
    torch.cuda.synchronize()
    s.check_device_errors()
    g = dict(token=tok.cpu().numpy(), logprob=lp.cpu().numpy(), topn_ids=tid.cpu().numpy(),
             topn_lp=tlp.cpu().numpy(), status=st.cpu().numpy(), kth_value=kv.cpu().numpy(),
             kth_index=ki.cpu().numpy(), kept=kept.cpu().numpy())
    return g, probs.cpu().numpy()


def check_probs(g, probs, o, where):
    B, V = o.probs.shape
    for r in range(B):
        tag = f"{where} row {r}"
        got = probs[r, :V]
        if o.status[r] != 0:
            assert np.isnan(got).all(), tag
            continue
        if o.greedy[r]:
            want = np.zeros(V)
            want[g["token"][r]] = 1.0
            np.testing.assert_array_equal(got, want, err_msg=tag)
            continue
        kept = int(g["kept"][r])
        want = o.probs[r] if kept == o.kept_count[r] else O.filtered_probs(o.zt[r], kept)
        # the kept set: nothing outside it; inside, fp32 holds every entry that
        # is not below its smallest subnormal
        assert (got[want == 0] == 0).all(), (tag, "outside the kept set")
        assert (got[want >= 1e-44] > 0).all(), (tag, "inside the kept set")
        np.testing.assert_allclose(got, want, rtol=PROBS_RTOL, atol=PROBS_ATOL, err_msg=tag)
        assert abs(float(got.astype(np.float64).sum()) - 1.0) < 1e-4, tag
    if probs.shape[1] > V:
        assert (probs[:, V:] == -7.0).all(), f"{where}: columns beyond V written"


def mixed_probs_workload(rng, dtype, B=12, V=50_003, ld=None, name="probs mixed"):
    x = W.peaked_rows(rng, B, V)
    x[B - 2, 11] = np.nan         # status 1
    x[B - 1, :] = -np.inf         # status 2
    prompt, output = history(rng, B, V, 120, 30)
    return custom_workload(
        x, dtype=dtype, ld=ld, name=name, n=6, prompt=prompt, output=output,
        T=[0.0, 0.7, 1.0, 1.3, 0.9, 2.0, 1.0, 0.8, 1.5, 1.1, 1.0, 1.0][:B],
        k=[0, 0, 50, 0, 300, 0, 1000, 20, 0, 0, 0, 0][:B],
        p=[1.0, 0.9, 1.0, 0.95, 0.8, 1.0, 0.5, 1.0, 0.99, 1.0, 0.9, 0.9][:B],
        mp=[0.0, 0.0, 0.0, 0.05, 0.0, 0.01, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0][:B],
        pres=[0.0, 0.5, 0.0, 0.0, 0.3, 0.0, 0.0, 0.2, 0.0, 0.0, 0.0, 0.0][:B],
        freq=[0.0, 0.2, 0.0, 0.0, 0.1, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0][:B],
        rep=[1.0, 1.2, 1.0, 1.0, 0.9, 1.0, 1.0, 1.1, 1.0, 1.0, 1.0, 1.0][:B])


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_probs_mixed(dtype):
    rng = np.random.default_rng(65)
    w = mixed_probs_workload(rng, dtype)
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        g, probs = sample_with_probs(s, w)
        o = O.sample_workload(w, want_zt=True, want_probs=True)
        compare(g, o, where=w.name)
        check_probs(g, probs, o, w.name)
        assert s.last_launches() in (4, 5)  # the sampling pair, then the two passes
    finally:
        s.close()


@pytest.mark.parametrize("ld_extra", [3, 8])
def test_probs_unaligned_and_padded(ld_extra):
    # odd row strides: element-wise loads and stores; columns past V untouched
    rng = np.random.default_rng(66 + ld_extra)
    V = 30_001
    w = mixed_probs_workload(rng, W.DTYPE_BF16, B=8, V=V, ld=V + ld_extra, name="probs ld")
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        g, probs = sample_with_probs(s, w, ld_probs=V + ld_extra)
        o = O.sample_workload(w, want_zt=True, want_probs=True)
        compare(g, o, where=w.name)
        check_probs(g, probs, o, w.name)
    finally:
        s.close()


def test_probs_with_update_counts():
    """The distribution uses the counts the draw saw; the counts then gain the
    token exactly as a call without the export leaves them."""
    rng = np.random.default_rng(67)
    w = mixed_probs_workload(rng, W.DTYPE_F32, B=10, V=20_000)
    x = device_logits(w)
    a, b = make_sampler(w), make_sampler(w)
    try:
        a.reset_workload(w)
        b.reset_workload(w)
        for step in range(3):
            ga, probs = sample_with_probs(a, w, x=x, update_counts=True)
            gb = run_gpu(b, w, x=x, update_counts=True, reset=False)
            for k in ("token", "status", "kept", "kth_index"):
                np.testing.assert_array_equal(ga[k], gb[k], err_msg=f"step {step} {k}")
            for r in range(w.B):
                np.testing.assert_array_equal(a.counts(r)[0], b.counts(r)[0])
                np.testing.assert_array_equal(a.counts(r)[1], b.counts(r)[1])
            if step == 0:
                o = O.sample_workload(w, want_zt=True, want_probs=True)
                check_probs(ga, probs, o, "update_counts")
    finally:
        a.close()
        b.close()


def test_probs_full_vocab_batch():
    # the b256 mix at full vocabulary, the oracle on a sample of its rows
    w = W.b256(seed=5)
    rows = np.array([0, 1, 2, 63, 64, 127, 128, 191, 200, 255])
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        g, probs = sample_with_probs(s, w)
        o = O.sample_workload(w, want_zt=True, want_probs=True, rows=rows)
        compare(g, o, rows=rows, where="b256")
        check_probs({k: v[rows] for k, v in g.items()}, probs[rows], o, "b256")
    finally:
        s.close()


@pytest.mark.parametrize("V", [1, 7, 17, 100, 4097, 200_003])
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
def test_probs_vocab_widths(V, dtype):
    # ragged tails, one to many CTAs per row, splits of one element to 64 K
    rng = np.random.default_rng(70 + V)
    B = 6
    x = rng.normal(0, 2.0, size=(B, V)).astype(np.float32)
    w = custom_workload(x, dtype=dtype, T=[0.0, 0.9, 1.2, 0.7, 1.0, 0.5],
                        k=[0, 0, 5, 0, 40, 3], p=[1.0, 1.0, 1.0, 0.8, 0.9, 1.0],
                        mp=[0.0, 0.0, 0.0, 0.0, 0.0, 0.2], n=min(5, V), name=f"probs V{V}")
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        g, probs = sample_with_probs(s, w)
        o = O.sample_workload(w, want_zt=True, want_probs=True)
        compare(g, o, where=w.name)
        check_probs(g, probs, o, w.name)
    finally:
        s.close()


def test_probs_single_row_many_splits():
    # one row: the grid spreads it over the most CTAs the plan allows
    rng = np.random.default_rng(77)
    x = W.peaked_rows(rng, 1, V_FULL)
    w = custom_workload(x, dtype=W.DTYPE_BF16, T=1.3, p=0.97, n=3, name="probs B1")
    s = make_sampler(w)
    try:
        s.reset_workload(w)
        g, probs = sample_with_probs(s, w)
        o = O.sample_workload(w, want_zt=True, want_probs=True)
        compare(g, o, where=w.name)
        check_probs(g, probs, o, w.name)
    finally:
        s.close()


def test_features_together_over_steps():
    """prompt_ignore_length, top-p decay, update_counts and the filtered
    distribution in one multi-call run over a bf16 batch whose top-p-only rows
    take the second stream; each call is checked against the oracle with the
    history and effective top_p the previous calls left (teacher forced)."""
    rng = np.random.default_rng(80)
    B, V, steps = 12, 40_000, 3
    T = np.array([0.0, 0.8, 1.1, 0.9, 1.3, 1.0, 0.7, 1.2, 1.0, 0.9, 1.4, 0.6], np.float32)
    k = np.array([0, 30, 0, 0, 0, 100, 0, 0, 1, 0, 0, 0], np.int32)
    p = np.array([1.0, 0.9, 0.8, 0.95, 0.9, 1.0, 0.7, 0.99, 1.0, 1.0, 0.85, 0.9], np.float32)
    pres = np.array([0.3, 0.0, 0.0, 0.5, 0.0, 0.2, 0.0, 0.0, 0.0, 0.4, 0.0, 0.0], np.float32)
    rep = np.array([1.1, 1.0, 1.0, 1.2, 1.0, 1.0, 1.0, 1.0, 1.0, 0.9, 1.0, 1.0], np.float32)
    decay = np.array([1, 1, 1, 0.8, 1, 0.7, 0.9, 1, 1, 1, 1, 1], np.float32)
    pmin = np.full(B, 0.3, np.float32)
    reset = np.full(B, -1, np.int32)
    ignore = np.array([0, 0, 0, 10, 0, 50, 0, 0, 0, 200, 0, 0], np.int32)
    prompt, output = history(rng, B, V, 60, 20)
    output = [list(o) for o in output]
    x0 = W.peaked_rows(rng, B, V)
    w0 = custom_workload(x0, dtype=W.DTYPE_BF16, T=T, k=k, p=p, pres=pres, freq=0.1 * (pres > 0),
                         rep=rep, n=4, prompt=prompt, output=output, name="together")
    w0.prompt_ignore = ignore
    s = make_sampler(w0, max_history=256)
    try:
        s.reset_params(w0.temperature, w0.top_k, w0.top_p, w0.min_p, w0.presence, w0.frequency,
                       w0.repetition, w0.seed, top_p_decay=decay, top_p_min=pmin,
                       top_p_reset_ids=reset)
        s.reset_token_counts(w0.prompt_ids, w0.prompt_offsets, w0.output_ids, w0.output_offsets,
                             prompt_ignore=ignore)
        active = (decay < 1) & (T > 0) & (k != 1)
        p_eff = p.copy()
        seed = w0.seed.copy()
        for step in range(steps):
            x = x0 if step == 0 else W.peaked_rows(rng, B, V)
            ws = custom_workload(x, dtype=W.DTYPE_BF16, T=T, k=k, p=p, pres=pres,
                                 freq=0.1 * (pres > 0), rep=rep, n=4, prompt=prompt,
                                 output=[np.array(o, np.int32) for o in output],
                                 name=f"together step {step}")
            ws.prompt_ignore = ignore
            ws.seed = seed.copy()
            g, probs = sample_with_probs(s, ws, update_counts=True)
            # the split step (3 or 4 launches), the two export passes, the append
            assert s.last_launches() in (6, 7), s.last_launches()
            o = O.sample_workload(ws, want_zt=True, top_p=p_eff, want_probs=True)
            compare(g, o, where=ws.name)
            check_probs(g, probs, o, ws.name)
            for r in range(B):
                if g["status"][r] == 0:
                    output[r].append(int(g["token"][r]))
                    if active[r]:
                        p_eff[r] = O.topp_decay(float(p_eff[r]), float(p[r]), float(decay[r]),
                                                float(pmin[r]), int(reset[r]), int(g["token"][r]))
            seed = np.array([O.next_seed(int(v)) for v in seed], np.uint64)
            np.testing.assert_array_equal(s.top_p(B), p_eff, err_msg=ws.name)
    finally:
        s.close()
