"""The vocabulary-sharded sampler [Tenstorrent sampling README: TTSampling takes
each device's top-k of its slice of the vocabulary, the candidates are
all-gathered, and LogProbsCalculator combines the devices' maxima and sums of
exponentials; vllm.cpp: the Gumbel draw's ArgReduce runs over true global
indices, so the noise of a column does not depend on which device holds it].

GPU, one device, the shards run one after another: the merged outputs equal
those of the unsharded vt_sample on the same rows and seeds (tokens, kept
counts, filter boundaries, top-n ids bit-exact; log-probs within 1e-5), and
both equal the oracle's.  Degenerate rows too: flat rows and heavy ties (the
exact radix-select path of the partials), masked columns, a shard with no
finite element, NaN, +inf and empty rows, a greedy tie across shards.

CPU, two gloo ranks: the exchange (``gather_partials``) and the composition it
relies on.  Each rank writes the documented records of its own columns from
the oracle's tempered logits; after the all-gather, a plain numpy merge of the
union gives the oracle's unsharded kept set, token, log-prob and top-n on
both ranks.
"""
from __future__ import annotations

import os
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from device_token_sampling_gb300 import sampler as S
from device_token_sampling_gb300 import workloads as W

from paritylib import LP_TOL, compare, custom_workload, device_logits, make_sampler, run_gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEAD_BYTES = 48


def part_bytes(K: int) -> int:
    return HEAD_BYTES + 8 * K


def even_bounds(V: int, n: int):
    b = np.linspace(0, V, n + 1).astype(np.int64)
    return [(int(b[i]), int(b[i + 1])) for i in range(n)]


def ragged_bounds(V: int, n: int, rng):
    cuts = np.sort(rng.choice(np.arange(1, V), n - 1, replace=False))
    b = np.concatenate([[0], cuts, [V]])
    return [(int(b[i]), int(b[i + 1])) for i in range(n)]


def advanced(seeds: np.ndarray, steps: int) -> np.ndarray:
    out = seeds.copy()
    for _ in range(steps):
        out = np.array([O.next_seed(int(v)) for v in out], np.uint64)
    return out


def sampled_workload(rng, B, V, K, dtype, n, name, x=None):
    """Rows the sharded path takes: greedy rows, rows without a filter, and
    sampled rows bounded by a top-k of at most K, some with min-p and some
    with top-p."""
    if x is None:
        x = W.peaked_rows(rng, B, V)
    T = rng.choice(np.array([0.0, 0.6, 1.0, 1.3], np.float32), B)
    k = rng.integers(2, K + 1, B).astype(np.int32)
    p = np.where(rng.random(B) < 0.5, rng.uniform(0.3, 0.99, B), 1.0).astype(np.float32)
    mp_ = np.where(rng.random(B) < 0.3, rng.uniform(0.001, 0.2, B), 0.0).astype(np.float32)
    free = rng.random(B) < 0.2  # no filter: every finite element kept
    k[free], p[free], mp_[free] = 0, 1.0, 0.0
    return custom_workload(x, dtype=dtype, T=T, k=k, p=p, mp=mp_, n=n,
                           seed=int(rng.integers(1 << 30)), name=name)


# --------------------------------------------------------------------------
# GPU: the shards one after another on one device
# --------------------------------------------------------------------------

def run_sharded(s: S.Sampler, w: W.Workload, x: torch.Tensor, K: int, bounds, reset=True):
    """vt_shard_partials on each column range of ``x`` in turn, the records
    stacked as an all-gather would leave them, then vt_shard_merge."""
    if reset:
        s.reset_workload(w)
    parts = [s.shard_partials(x[:, v0:v1], v0, w.V, K) for v0, v1 in bounds]
    tok, lp, tid, tlp = s.shard_merge(torch.stack(parts), w.V, K, w.num_logprobs)
    st = s.row_status(w.B)
    kv, ki, kept = s.filter_boundary(w.B)
    torch.cuda.synchronize()
    s.check_device_errors()
    return dict(token=tok.cpu().numpy(), logprob=lp.cpu().numpy(), topn_ids=tid.cpu().numpy(),
                topn_lp=tlp.cpu().numpy(), status=st.cpu().numpy(), kth_value=kv.cpu().numpy(),
                kth_index=ki.cpu().numpy(), kept=kept.cpu().numpy())


def same_outputs(g: dict, u: dict, where: str):
    """Sharded ``g`` against unsharded ``u``: everything exact but log-probs."""
    for key in ("status", "token", "kept", "kth_index", "topn_ids"):
        np.testing.assert_array_equal(g[key], u[key], err_msg=f"{where}: {key}")
    ok = u["status"] == 0
    np.testing.assert_array_equal(g["kth_value"][ok], u["kth_value"][ok], err_msg=where)
    np.testing.assert_allclose(g["logprob"][ok], u["logprob"][ok], rtol=0, atol=LP_TOL,
                               err_msg=where)
    np.testing.assert_allclose(g["topn_lp"][ok], u["topn_lp"][ok], rtol=0, atol=LP_TOL,
                               err_msg=where)


@pytest.fixture(scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F32])
@pytest.mark.parametrize("n_shards,K,ragged", [(1, 64, False), (2, 64, False), (3, 128, True),
                                               (4, 256, True), (16, 256, False)])
def test_sharded_equals_unsharded_and_oracle(_gpu, dtype, n_shards, K, ragged):
    rng = np.random.default_rng(100 * n_shards + K + dtype)
    B, V = 24, 50_000
    w = sampled_workload(rng, B, V, K, dtype, n=min(K, 6), name=f"sharded S={n_shards} K={K}")
    bounds = ragged_bounds(V, n_shards, rng) if ragged else even_bounds(V, n_shards)
    x = device_logits(w)
    su, ss = make_sampler(w), make_sampler(w)
    try:
        su.reset_workload(w)
        ss.reset_workload(w)
        for step in range(3):  # the seeds advance alike on both paths
            u = run_gpu(su, w, x, reset=False)
            g = run_sharded(ss, w, x, K, bounds, reset=False)
            same_outputs(g, u, f"{w.name} step {step}")
            if step != 1:
                o = O.sample_workload(w, want_zt=True, seed=advanced(w.seed, step))
                compare(g, o, where=f"{w.name} step {step}")
    finally:
        su.close()
        ss.close()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F32])
def test_sharded_full_vocabulary(_gpu, dtype):
    """V = 248,320 over 4 and 8 shards, as a tensor-parallel decode would split it."""
    rng = np.random.default_rng(77 + dtype)
    B, V, K = 8, 248_320, 256
    w = sampled_workload(rng, B, V, K, dtype, n=8, name="sharded full vocabulary")
    x = device_logits(w)
    o = O.sample_workload(w, want_zt=True)
    su = make_sampler(w)
    try:
        u = run_gpu(su, w, x)
        for n_shards in (4, 8):
            g = run_sharded(su, w, x, K, even_bounds(V, n_shards))
            same_outputs(g, u, f"{w.name} S={n_shards}")
            compare(g, o, where=f"{w.name} S={n_shards}")
    finally:
        su.close()


def degenerate_rows(rng, V, bounds):
    """Rows that defeat the partials' quick threshold or the merge's common case."""
    rows, cfg = [], []
    ninf = np.float32(-np.inf)

    def add(x, T=1.0, k=64, p=1.0, mp=0.0):
        rows.append(np.asarray(x, np.float32))
        cfg.append((T, k, p, mp))

    add(np.zeros(V))                                           # flat: every value ties
    add(np.zeros(V), k=60, p=0.5)                              # flat under top-p
    add(np.zeros(V), k=40, mp=0.5)                             # flat under min-p
    add(rng.integers(-3, 4, V), k=64, p=0.9)                   # few distinct values
    add(np.round(rng.standard_normal(V) * 4) / 4, T=0.7, k=50)  # quarter steps
    m = np.full(V, ninf)
    m[rng.choice(np.arange(bounds[1][0], bounds[1][1]), 30, replace=False)] = \
        rng.standard_normal(30)
    add(m, k=40, p=0.95)                                       # 30 finite, in one shard
    m = np.full(V, ninf)
    m[rng.choice(V, 5, replace=False)] = rng.standard_normal(5)
    add(m, k=20)                                               # 5 finite: top-n reaches -inf
    m = rng.standard_normal(V).astype(np.float32)
    m[bounds[0][0]:bounds[0][1]] = ninf
    add(m, T=0.0)                                              # the first shard all -inf
    add(m, T=1.1, k=64, p=0.8)
    m = rng.standard_normal(V).astype(np.float32)
    m[10] = m[bounds[-1][0] + 3] = 9.0
    add(m, T=0.0)                                              # greedy tie across shards
    add(m, T=1.0, k=2)
    m = rng.standard_normal(V).astype(np.float32)
    m[bounds[-1][0] + 7] = np.nan
    add(m, k=10)                                               # NaN: non-finite
    m = rng.standard_normal(V).astype(np.float32)
    m[bounds[1][0]] = np.inf
    add(m, T=0.0)                                              # +inf: non-finite
    add(np.full(V, ninf), k=10)                                # nothing finite: empty
    add(W.peaked_rows(rng, 1, V)[0], k=64, p=0.3)
    T, k, p, mp_ = (np.array(c) for c in zip(*cfg))
    return np.stack(rows), T, k, p, mp_


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F32])
def test_sharded_degenerate_rows(_gpu, dtype):
    rng = np.random.default_rng(31 + dtype)
    V, K = 20_000, 64
    bounds = even_bounds(V, 3)
    x, T, k, p, mp_ = degenerate_rows(rng, V, bounds)
    w = custom_workload(x, dtype=dtype, T=T, k=k, p=p, mp=mp_, n=16, name="sharded degenerate")
    xd = device_logits(w)
    o = O.sample_workload(w, want_zt=True)
    s = make_sampler(w)
    try:
        u = run_gpu(s, w, xd)
        g = run_sharded(s, w, xd, K, bounds)
        same_outputs(g, u, w.name)
        compare(g, o, where=w.name)
        assert list(g["status"][-4:-1]) == [1, 1, 2], g["status"]
    finally:
        s.close()


@pytest.mark.gpu
def test_sharded_rejects_rows_it_cannot_compose(_gpu):
    B, V, K = 4, 5000, 64
    rng = np.random.default_rng(3)
    x = rng.standard_normal((B, V)).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    part = torch.empty((B, part_bytes(K)), dtype=torch.uint8, device="cuda")
    outs = [torch.empty(B, dtype=torch.int32, device="cuda"),
            torch.empty(B, dtype=torch.float32, device="cuda")]
    with S.Sampler(B, V, 4, 64) as s:
        lib = s._lib

        def partials(K_=K, Vs=V, v0=0, B_=B):
            return lib.vt_shard_partials(s.handle, S.P(xd.data_ptr()), W.DTYPE_F32, B_, Vs, V,
                                         v0, V, K_, S.P(part.data_ptr()), None)

        def merge(S_=1, K_=K, n=0):
            return lib.vt_shard_merge(s.handle, S.P(part.data_ptr()), S_, B, V, K_, n,
                                      S.P(outs[0].data_ptr()), S.P(outs[1].data_ptr()), None,
                                      None, None)

        assert partials() == S.VT_ERR_STATE                   # before any reset
        base = custom_workload(x, T=[0.0, 1.0, 0.8, 1.0], k=[0, 10, 64, 2])
        s.reset_workload(base)
        assert partials() == S.VT_OK and merge() == S.VT_OK
        assert partials(K_=0) == S.VT_ERR_INVALID_ARG
        assert partials(K_=257) == S.VT_ERR_INVALID_ARG
        assert partials(Vs=V, v0=1) == S.VT_ERR_INVALID_ARG  # past the row
        assert partials(B_=5) == S.VT_ERR_STATE
        assert merge(S_=65) == S.VT_ERR_INVALID_ARG
        assert merge(S_=64, K_=65) == S.VT_ERR_INVALID_ARG    # S * K above 4096
        assert merge(n=5) == S.VT_ERR_INVALID_ARG             # n > max_logprobs
        for bad in (dict(k=[0, 0, 10, 10], p=[1.0, 0.9, 1.0, 1.0]),  # top-p without top-k
                    dict(k=[0, 65, 10, 10]),                   # top-k above K
                    dict(k=[0, 10, 10, 10], pres=[0, 0.5, 0, 0])):  # penalties
            w = custom_workload(x, T=[0.0, 1.0, 1.0, 1.0], **{"p": 1.0, **bad})  # noqa: PIE800
            s.reset_workload(w)
            assert partials() == S.VT_ERR_INVALID_ARG, bad
            assert b"row 1" in lib.vt_last_error(s.handle)
        s.reset_workload(base)
        assert partials() == S.VT_OK and merge() == S.VT_OK
        torch.cuda.synchronize()
        s.check_device_errors()


# --------------------------------------------------------------------------
# CPU: the exchange over two gloo ranks and the composition of the records
# --------------------------------------------------------------------------

def ord_code(z: np.ndarray) -> np.ndarray:
    """The records' order-preserving code of float32 values (bits 63..32)."""
    u = np.ascontiguousarray(z, np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def code_value(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, np.uint32)
    return np.where(c & 0x80000000, c & 0x7FFFFFFF, ~c).astype(np.uint32).view(np.float32)


def unfiltered(w: W.Workload, r: int) -> bool:
    """A sampled row without top-k, top-p or min-p: every finite element kept."""
    greedy = w.temperature[r] == 0 or w.top_k[r] == 1 or w.top_p[r] == 0 or w.min_p[r] == 1
    topk = 1 < w.top_k[r] < w.V
    return not greedy and not topk and not (0 < w.top_p[r] < 1) and not (0 < w.min_p[r] < 1)


def gumbel_scores(w: W.Workload, r: int, z: np.ndarray, v0: int) -> np.ndarray:
    """z_t - ln(-ln u) in float64 for global columns v0 .. v0 + len(z) - 1."""
    b = O.noise_bits(int(w.seed[r]), r, v0, len(z)).astype(np.float64)
    return z.astype(np.float64) - np.log(-np.log((b + 0.5) * 2.0**-24))


def write_records(zt: np.ndarray, v0: int, K: int, w: W.Workload) -> np.ndarray:
    """One shard's records, in the documented layout, from its tempered logits
    zt [B, Vs] (finite or -inf) holding global columns v0 .. v0 + Vs - 1."""
    B, Vs = zt.shape
    out = np.zeros((B, part_bytes(K)), np.uint8)
    j = np.arange(v0, v0 + Vs, dtype=np.int64)
    f32 = lambda v: np.array([v], np.float32).view(np.uint32)[0]  # noqa: E731
    for r in range(B):
        z = zt[r].astype(np.float32)
        m = np.float32(z.max())
        s = np.float32(np.exp(z.astype(np.float64) - m).sum()) if m > -np.inf else np.float32(0)
        argj = int(j[np.argmax(z)]) if m > -np.inf else 2**31 - 1
        wn = min(K, Vs)
        order = np.lexsort((j, -z))
        top = order[:wn]
        keys = (ord_code(z[top]).astype(np.uint64) << np.uint64(32)) | \
            (~j[top].astype(np.uint32)).astype(np.uint64)
        head = np.zeros(12, np.uint32)
        head[0], head[1], head[2], head[3] = f32(m), f32(s), np.uint32(argj), np.uint32(wn)
        head[4], head[5] = f32(-np.inf), np.uint32(2**31 - 1)
        fin = np.isfinite(z)
        if unfiltered(w, r) and fin.any():
            sc = np.where(fin, gumbel_scores(w, r, z, v0), -np.inf)
            best = int(np.lexsort((j, -sc))[0])
            lastpos = [q for q in order if fin[q]][-1]
            lastkey = (int(ord_code(z[lastpos:lastpos + 1])[0]) << 32) | (~int(j[lastpos]) & 0xFFFFFFFF)
            nk = (~lastkey) & 0xFFFFFFFFFFFFFFFF
            head[4], head[5], head[6] = f32(sc[best]), np.uint32(j[best]), f32(z[best])
            head[7] = np.uint32(fin.sum())
            head[8], head[9] = np.uint32(nk & 0xFFFFFFFF), np.uint32(nk >> 32)
        out[r, :HEAD_BYTES] = head.view(np.uint8)
        out[r, HEAD_BYTES:HEAD_BYTES + 8 * wn] = keys.view(np.uint8)
    return out


def merge_records(parts: np.ndarray, w: W.Workload, K: int):
    """The union of the gathered records [S, B, bytes], composed in float64 by
    the pages' rules: min-p, top-k, top-p over the survivors renormalised,
    then the Gumbel-max draw with the global (row, column) noise."""
    n = w.num_logprobs
    out = dict(token=[], logprob=[], kept=[], topn_ids=[], topn_lp=[])
    for r in range(w.B):
        heads = parts[:, r, :HEAD_BYTES].copy().view(np.uint32)
        ms = heads[:, 0].view(np.float32).astype(np.float64)
        ss = heads[:, 1].view(np.float32).astype(np.float64)
        m = ms.max()
        S_ = sum(s * np.exp(mi - m) for mi, s in zip(ms, ss) if mi > -np.inf)
        lse = m + np.log(S_)
        keys = np.concatenate([parts[sh, r, HEAD_BYTES:HEAD_BYTES + 8 * int(heads[sh, 3])]
                               .copy().view(np.uint64) for sh in range(parts.shape[0])])
        keys = np.sort(keys)[::-1]
        z = code_value((keys >> np.uint64(32)).astype(np.uint32)).astype(np.float64)
        j = (~(keys & np.uint64(0xFFFFFFFF)).astype(np.uint32)).astype(np.int64)
        out["topn_ids"].append(j[:n])
        out["topn_lp"].append(z[:n] - lse)
        if unfiltered(w, r):
            # the best of the shards' Gumbel winners (score, then lower index)
            sc = heads[:, 4].view(np.float32).astype(np.float64)
            wj = heads[:, 5].view(np.int32)
            live = wj != 2**31 - 1
            best = min((-sc[q], wj[q], q) for q in np.flatnonzero(live))[2]
            tok, kept = int(wj[best]), int(heads[:, 7].sum())
            zt_tok = float(heads[best, 6:7].view(np.float32)[0])
            out["token"].append(tok)
            out["kept"].append(kept)
            out["logprob"].append(zt_tok - lse)
            continue
        if w.temperature[r] == 0:
            cand = heads[:, 2].view(np.int32)[ms == m]
            tok, kept = int(cand.min()), 1
        else:
            L = int(np.isfinite(z).sum())
            L1 = L
            if 0 < w.min_p[r] < 1:
                L1 = int((z[:L] - m >= np.log(np.float64(w.min_p[r]))).sum())
            L2 = min(int(w.top_k[r]), L1)
            L3 = L2
            if 0 < w.top_p[r] < 1:
                pre = np.concatenate([[0.0], np.cumsum(np.exp(z[:L2] - m))])
                L3 = max(1, int((pre[:L2] / pre[L2] <= np.float64(w.top_p[r])).sum()))
            bits = np.array([O.noise_bits(int(w.seed[r]), r, int(c), 1)[0] for c in j[:L3]],
                            np.float64)
            u = (bits + 0.5) * 2.0**-24
            score = z[:L3] - np.log(-np.log(u))
            best = max(range(L3), key=lambda i: (score[i], -j[i]))
            tok, kept = int(j[best]), L3
        zt_tok = z[j == tok][0] if (j == tok).any() else m
        out["token"].append(tok)
        out["kept"].append(kept)
        out["logprob"].append(zt_tok - lse)
    return {k: np.array(v) for k, v in out.items()}


def shard_cpu_workload(K: int):
    rng = np.random.default_rng(2718)
    B, V = 12, 6000
    x = W.peaked_rows(rng, B, V)
    x[3, :2500] = -np.inf              # the first rank's columns hold nothing finite
    x[4, 17] = x[4, 4000] = 20.0       # a greedy tie across the ranks
    w = sampled_workload(rng, B, V, K, W.DTYPE_F32, n=5, name="gloo shards", x=x)
    w.temperature[4] = 0.0
    for r in (5, 9):  # rows without a filter: the shards' Gumbel winners compose
        w.temperature[r], w.top_k[r], w.top_p[r], w.min_p[r] = 1.1, 0, 1.0, 0.0
    return w, [(0, 2500), (2500, V)]


def _rank(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        K = 64
        w, bounds = shard_cpu_workload(K)
        o = O.sample_workload(w, want_zt=True)
        v0, v1 = bounds[rank]
        mine = torch.from_numpy(write_records(o.zt[:, v0:v1], v0, K, w))
        gathered = S.gather_partials(mine).numpy()
        assert gathered.shape == (world, w.B, part_bytes(K))
        g = merge_records(gathered, w, K)
        out[rank] = {k: v.tolist() for k, v in g.items()}
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_compose_the_unsharded_result():
    O.build()
    world, K = 2, 64
    port = 31500 + os.getpid() % 2000
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0] == res[1], "every rank merges the same records"
    g = {k: np.array(v) for k, v in res[0].items()}
    w, _ = shard_cpu_workload(K)
    o = O.sample_workload(w, want_zt=True)
    assert (o.status == 0).all()
    np.testing.assert_array_equal(g["topn_ids"], o.topn_ids)
    # the records carry each shard's sum of exponentials in fp32 (relative
    # rounding 2^-24), so the composed log-normaliser is within about 1e-7
    np.testing.assert_allclose(g["topn_lp"], o.topn_logprobs, rtol=0, atol=1e-6)
    for r in range(w.B):
        if not o.topp_near[r]:
            assert g["kept"][r] == o.kept_count[r], (r, g["kept"][r], o.kept_count[r])
        if not (o.topp_near[r] or o.gumbel_near_tie[r]):
            assert g["token"][r] == o.token[r], (r, g["token"][r], o.token[r])
            assert abs(g["logprob"][r] - o.logprob[r]) <= 1e-6
    assert g["token"][4] == 17
    assert (o.kept_count[~o.greedy.astype(bool)] > 1).any()
