"""Helpers shared by the GPU parity tests: run the CUDA sampler through the C
ABI and compare it with the oracle element by element.

Comparison rules (the tolerances of the sampler's contract):
  * status, greedy tokens, top-n ids, top-k boundaries and kept counts,
    and the count tables: bit-exact;
  * drawn tokens: equal to the oracle's, except where the oracle flags the
    top two Gumbel scores within 1e-6 relative, or a top-p decision next to
    the boundary within 1e-6 of p; then any token in the oracle's acceptable
    set (and a kept count inside its acceptable range) is correct;
  * log-probs: within 1e-5 absolute (fp32 against the oracle's double).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from device_token_sampling_gb300 import sampler as S
from device_token_sampling_gb300 import workloads as W

LP_TOL = 1e-5


def device_logits(w: W.Workload) -> torch.Tensor:
    x = torch.from_numpy(np.ascontiguousarray(w.logits))
    if w.dtype == W.DTYPE_BF16:
        x = x.view(torch.int16)
    return x.cuda()


def make_sampler(w: W.Workload, max_history=None, n=None, **kw) -> S.Sampler:
    if max_history is None:
        h = int(np.max(np.diff(w.prompt_offsets) + np.diff(w.output_offsets))) if w.B else 0
        max_history = max(64, h + 256)
    return S.Sampler(max_batch=w.B, max_vocab=max(w.V, 1), max_logprobs=max(w.num_logprobs, n or 0),
                     max_history=max_history, device=torch.cuda.current_device(), **kw)


def run_gpu(s: S.Sampler, w: W.Workload, x: torch.Tensor | None = None, update_counts=False,
            reset=True):
    """One vt_sample call; returns host numpy copies of every output."""
    if reset:
        s.reset_workload(w)
    if x is None:
        x = device_logits(w)
    dt = W.DTYPE_BF16 if w.dtype == W.DTYPE_BF16 else W.DTYPE_F32
    tok, lp, tid, tlp = s.sample(x, V=w.V, num_logprobs=w.num_logprobs,
                                 update_counts=update_counts, dtype=dt)
    st = s.row_status(w.B)
    kv, ki, kept = s.filter_boundary(w.B)
    torch.cuda.synchronize()
    s.check_device_errors()
    return dict(token=tok.cpu().numpy(), logprob=lp.cpu().numpy(), topn_ids=tid.cpu().numpy(),
                topn_lp=tlp.cpu().numpy(), status=st.cpu().numpy(), kth_value=kv.cpu().numpy(),
                kth_index=ki.cpu().numpy(), kept=kept.cpu().numpy())


def compare(g: dict, o: O.OracleOut, rows=None, zt=None, where=""):
    """Assert the GPU outputs ``g`` match the oracle ``o`` (optionally for a row
    subset: ``rows`` indexes ``g``; ``o`` holds those rows in order)."""
    rows = np.arange(len(o.token)) if rows is None else np.asarray(rows)
    zt = o.zt if zt is None else zt
    for k, r in enumerate(rows):
        tag = f"{where} row {r}"
        assert g["status"][r] == o.status[k], (tag, g["status"][r], o.status[k])
        if o.status[k] != 0:
            assert g["token"][r] == -1, tag
            assert (g["topn_ids"][r] == -1).all(), tag
            continue
        tok = int(g["token"][r])
        kept = int(g["kept"][r])
        if o.greedy[k]:
            assert tok == o.token[k], (tag, "greedy", tok, o.token[k])
            assert kept == 1, tag
        else:
            assert o.kept_lo[k] <= kept <= o.kept_hi[k], (tag, "kept", kept, o.kept_lo[k],
                                                          o.kept_hi[k], o.kept_count[k])
            if kept == o.kept_count[k]:
                assert g["kth_index"][r] == o.kth_index[k], (tag, g["kth_index"][r], o.kth_index[k])
                assert g["kth_value"][r] == o.kth_value[k], (tag, g["kth_value"][r], o.kth_value[k])
            flagged = o.gumbel_near_tie[k] or o.topp_near[k]
            if flagged:
                assert tok in o.alt_tokens[k], (tag, "alt", tok, o.alt_tokens[k])
            else:
                assert tok == o.token[k], (tag, "token", tok, o.token[k], o.best_score[k],
                                           o.second_score[k], o.second_token[k])
        if zt is not None:
            want = float(zt[k, tok]) - o.lse[k]
        else:
            assert tok == o.token[k], tag
            want = o.logprob[k]
        assert abs(g["logprob"][r] - want) <= LP_TOL, (tag, "logprob", g["logprob"][r], want)
        n = o.topn_ids.shape[1]
        if n:
            np.testing.assert_array_equal(g["topn_ids"][r], o.topn_ids[k], err_msg=tag)
            np.testing.assert_allclose(g["topn_lp"][r], o.topn_logprobs[k], rtol=0, atol=LP_TOL,
                                       err_msg=tag)


def check_workload(w: W.Workload, rows=None, s: S.Sampler | None = None, **kw):
    own = s is None
    if own:
        s = make_sampler(w)
    try:
        g = run_gpu(s, w, **kw)
        o = O.sample_workload(w, want_zt=True, rows=rows)
        compare(g, o, rows=rows, where=w.name)
        return g, o
    finally:
        if own:
            s.close()


def custom_workload(x: np.ndarray, *, dtype=W.DTYPE_F32, ld=None, T=1.0, k=0, p=1.0, mp=0.0,
                    pres=0.0, freq=0.0, rep=1.0, n=0, seed=7, prompt=None, output=None,
                    name="custom") -> W.Workload:
    """A workload from explicit fp32 rows and scalar or per-row parameters."""
    x = np.asarray(x, np.float32)
    B, V = x.shape
    ld = V if ld is None else ld
    full = lambda v, dt: np.broadcast_to(np.asarray(v, dtype=dt), (B,)).copy()
    rng = np.random.default_rng(seed)
    pi, po = W.csr(prompt if prompt is not None else [np.zeros(0, np.int32)] * B)
    oi, oo = W.csr(output if output is not None else [np.zeros(0, np.int32)] * B)
    return W.Workload(name, B, V, ld, dtype, W.pad_rows(x, ld, dtype),
                      temperature=full(T, np.float32), top_k=full(k, np.int32),
                      top_p=full(p, np.float32), min_p=full(mp, np.float32),
                      presence=full(pres, np.float32), frequency=full(freq, np.float32),
                      repetition=full(rep, np.float32), seed=W.seeds(rng, B), prompt_ids=pi,
                      prompt_offsets=po, output_ids=oi, output_offsets=oo, num_logprobs=n)
