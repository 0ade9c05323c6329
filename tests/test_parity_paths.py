"""GPU parity of the paths a single eager vt_sample call does not exercise:
the host-memory entry point, steps captured in a CUDA graph and replayed on
two streams (the benchmark's timed loop), a count table that fills up, fp32
rows of 248,320 elements that reach the selection kernel, and the Large
configuration over 100 consecutive decode steps with the drawn tokens
appended to the counts on the device (teacher-forced: the oracle at step t
uses the tokens the GPU drew before t) [Tenstorrent sampling README,
SeedManager: one seed advance per sampled token; TensorRT-LLM "Sampling",
occurrence penalties over the prompt and everything generated]."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from device_token_sampling_gb300 import sampler as S
from device_token_sampling_gb300 import workloads as W

from paritylib import LP_TOL, compare, custom_workload, device_logits, make_sampler, run_gpu

pytestmark = pytest.mark.gpu
GAMMA = 0x9E3779B97F4A7C15


def advanced(seed, k):
    """Per-row seeds after k calls (each adds GAMMA mod 2^64)."""
    return np.array([(int(v) + k * GAMMA) % 2**64 for v in seed], dtype=np.uint64)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def compare_tokens(tok, lp, tid, tlp, o, where):
    """Tokens, log-probs and top-n of one call against the oracle (no kept-set
    view: that debug output holds only the last call)."""
    for r in range(len(o.token)):
        tag = f"{where} row {r}"
        if o.status[r] != 0:
            assert tok[r] == -1, tag
            continue
        t = int(tok[r])
        if o.greedy[r] or not (o.gumbel_near_tie[r] or o.topp_near[r]):
            assert t == o.token[r], (tag, t, o.token[r])
            assert abs(lp[r] - o.logprob[r]) <= LP_TOL, (tag, lp[r], o.logprob[r])
        else:
            assert t in o.alt_tokens[r], (tag, t, o.alt_tokens[r])
        if o.topn_ids.shape[1]:
            np.testing.assert_array_equal(tid[r], o.topn_ids[r], err_msg=tag)
            np.testing.assert_allclose(tlp[r], o.topn_logprobs[r], rtol=0, atol=LP_TOL,
                                       err_msg=tag)


# --------------------------------------------------------------------------
# vt_sample_host: host logits in, host outputs back
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["b256", "tiny"])
def test_sample_host(name):
    w = W.get(name)
    s = make_sampler(w, host_io=True)
    try:
        s.reset_workload(w)
        dt = W.DTYPE_BF16 if w.dtype == W.DTYPE_BF16 else W.DTYPE_F32
        tok, lp, tid, tlp = s.sample_host(w.logits, w.V, dt, num_logprobs=w.num_logprobs)
        st = s.row_status(w.B)
        kv, ki, kept = s.filter_boundary(w.B)
        torch.cuda.synchronize()
        g = dict(token=tok, logprob=lp, topn_ids=tid, topn_lp=tlp, status=st.cpu().numpy(),
                 kth_value=kv.cpu().numpy(), kth_index=ki.cpu().numpy(), kept=kept.cpu().numpy())
        o = O.sample_workload(w, want_zt=True)
        compare(g, o, where=f"{name} host")
        # the seeds advanced once, as after vt_sample
        np.testing.assert_array_equal(s.seeds(w.B), advanced(w.seed, 1))
    finally:
        s.close()


@pytest.mark.parametrize("path", [1, 2])
def test_sample_host_async_steps(path):
    """Four host steps enqueued back to back (each step's copy-in overlaps the
    previous step's sampling through the two staging slots), waited for once:
    every step equals the oracle on its own logits and advanced seeds."""
    import copy
    w = W.b256()
    rng = np.random.default_rng(5)
    steps = [w.logits] + [w.logits[rng.permutation(w.B)] for _ in range(3)]
    pinned = []
    for x in steps:
        t = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
        pinned.append(t.numpy())
    s = make_sampler(w, host_io=True)
    try:
        s.set_path(path)
        s.reset_workload(w)
        outs = [s.sample_host_async(x, w.V, W.DTYPE_BF16, num_logprobs=w.num_logprobs)
                for x in pinned]
        s.sample_host_wait()
        for k, (x, (tok, lp, tid, tlp)) in enumerate(zip(steps, outs)):
            wk = copy.copy(w)
            wk.logits = x
            o = O.sample_workload(wk, seed=advanced(w.seed, k))
            compare_tokens(tok, lp, tid, tlp, o, where=f"async step {k} path {path}")
        np.testing.assert_array_equal(s.seeds(w.B), advanced(w.seed, len(steps)))
    finally:
        s.close()


# --------------------------------------------------------------------------
# graph-captured steps on two streams, replayed as the benchmark replays them
# --------------------------------------------------------------------------

def test_graph_replay_steps():
    w = W.b256()
    s = make_sampler(w)
    try:
        B, V, n = w.B, w.V, w.num_logprobs
        x0 = device_logits(w)
        gen = torch.Generator(device="cuda")
        bufs = [x0]
        for i in range(1, 3):
            gen.manual_seed(77 + i)
            bufs.append(x0[torch.randperm(B, device="cuda", generator=gen)].contiguous())
        outs = [(torch.empty(B, dtype=torch.int32, device="cuda"),
                 torch.empty(B, dtype=torch.float32, device="cuda"),
                 torch.empty((B, n), dtype=torch.int32, device="cuda"),
                 torch.empty((B, n), dtype=torch.float32, device="cuda")) for _ in bufs]
        stream = torch.cuda.Stream()
        s.reset_workload(w)
        with torch.cuda.stream(stream):  # one eager step first (plans, attributes)
            s.sample(bufs[0], V=V, num_logprobs=n, out=outs[0], stream=stream, dtype=w.dtype)
        stream.synchronize()
        assert s.last_launches() >= 3, "the b256 call is expected to split over two streams"
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(len(bufs)):
                s.sample(bufs[i], V=V, num_logprobs=n, out=outs[i], stream=stream, dtype=w.dtype)
        s.reset_workload(w, stream=stream)  # the replay starts from the initial seeds
        stream.synchronize()
        graph.replay()
        stream.synchronize()
        s.check_device_errors()
        for i, (tok, lp, tid, tlp) in enumerate(outs):
            host = bufs[i].cpu().numpy().view(np.uint16)
            wi = W.Workload(w.name, B, V, V, w.dtype, host, temperature=w.temperature,
                            top_k=w.top_k, top_p=w.top_p, min_p=w.min_p, presence=w.presence,
                            frequency=w.frequency, repetition=w.repetition,
                            seed=advanced(w.seed, i),
                            prompt_ids=w.prompt_ids, prompt_offsets=w.prompt_offsets,
                            output_ids=w.output_ids, output_offsets=w.output_offsets,
                            num_logprobs=n)
            o = O.sample_workload(wi)
            compare_tokens(tok.cpu().numpy(), lp.cpu().numpy(), tid.cpu().numpy(),
                           tlp.cpu().numpy(), o, f"graph step {i}")
        np.testing.assert_array_equal(s.seeds(B), advanced(w.seed, 3))
    finally:
        s.close()


# --------------------------------------------------------------------------
# a count table that fills up
# --------------------------------------------------------------------------

def test_history_full_status():
    rng = np.random.default_rng(31)
    V = 500
    x = rng.normal(0, 1, size=(3, V)).astype(np.float32)
    x[:, 7] = 9.0  # the greedy token of every row
    prompt = [np.array([1, 2, 3, 4], np.int32), np.array([1, 2, 3, 7], np.int32),
              np.array([1, 2], np.int32)]
    w = custom_workload(x, T=0.0, pres=0.1, prompt=prompt, n=2, name="history full")
    s = make_sampler(w, max_history=4)
    try:
        g = run_gpu(s, w, update_counts=True)
        o = O.sample_workload(w, want_zt=True)
        # row 0: a fifth distinct id does not fit; row 1: 7 is there; row 2: room
        assert g["status"].tolist() == [S.ROW_HISTORY_FULL, S.ROW_OK, S.ROW_OK]
        np.testing.assert_array_equal(g["token"], o.token)
        ids0, cnt0 = s.counts(0)
        assert ids0.tolist() == [1, 2, 3, 4] and cnt0.tolist() == [1, 1, 1, 1]
        ids1, cnt1 = s.counts(1)
        assert ids1.tolist() == [1, 2, 3, 7] and cnt1.tolist() == [1, 1, 1, 2]
        ids2, cnt2 = s.counts(2)
        assert ids2.tolist() == [1, 2, 7] and cnt2.tolist() == [1, 1, 1]
    finally:
        s.close()


# --------------------------------------------------------------------------
# fp32 rows of the Large width that the selection kernel finishes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("penalised", [False, True])
def test_fp32_wide_rows_reach_the_selection_kernel(penalised):
    rng = np.random.default_rng(41 + penalised)
    B, V = 6, 248_320
    x = W.peaked_rows(rng, B, V)
    prompt = [W.zipf_ids(rng, 2048, V) for _ in range(B)] if penalised else None
    w = custom_workload(x, T=1.2, p=[0.9, 0.95, 0.99, 0.8, 0.97, 0.93], n=5,
                        pres=0.5 if penalised else 0.0, freq=0.3 if penalised else 0.0,
                        rep=1.1 if penalised else 1.0, prompt=prompt,
                        name=f"fp32 wide pen={penalised}")
    s = make_sampler(w)
    try:
        g = run_gpu(s, w)
        assert s.last_handover() > 0, "no row reached the selection kernel"
        o = O.sample_workload(w, want_zt=True)
        compare(g, o, where=w.name)
    finally:
        s.close()


# --------------------------------------------------------------------------
# Large: 100 decode steps, counts appended on the device, teacher-forced
# --------------------------------------------------------------------------

def large_step_device(step, B, V):
    """The step's logits, made on the device (peaked rows, seed 1000 + step)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + step)
    x = torch.randn(B, V, device="cuda", generator=g) * 1.5
    pos = torch.randint(0, V, (B, 8), device="cuda", generator=g)
    add = torch.rand(B, 8, device="cuda", generator=g) * 4.0 + 8.0
    x.scatter_add_(1, pos, add)
    return x


def test_large_100_decode_steps():
    from oracle_pool import sample_parallel
    w = W.large(with_logits=False)
    B, V, n = w.B, w.V, w.num_logprobs
    steps, checked = 100, (0, 1, 50, 99)
    s = S.Sampler(max_batch=B, max_vocab=V, max_logprobs=n, max_history=4096 + 128,
                  device=torch.cuda.current_device())
    try:
        s.reset_workload(w)
        drawn = []   # host copies of every step's tokens (the teacher-forced history)
        saved = {}
        for t in range(steps):
            x = large_step_device(t, B, V)
            tok, lp, tid, tlp = s.sample(x, V=V, num_logprobs=n, update_counts=True)
            st = s.row_status(B)
            if t in checked:
                torch.cuda.synchronize()
                saved[t] = (x.cpu().numpy(), tok.cpu().numpy(), lp.cpu().numpy(),
                            tid.cpu().numpy(), tlp.cpu().numpy(), st.cpu().numpy())
            drawn.append(tok.cpu().numpy().copy())
        torch.cuda.synchronize()
        s.check_device_errors()
    finally:
        s.close()
    for t in checked:
        xh, tok, lp, tid, tlp, st = saved[t]
        assert (st == S.ROW_OK).all(), t
        # the history: the prompt and every token drawn before step t
        hist = np.stack(drawn[:t], axis=1) if t else np.zeros((B, 0), np.int32)
        oi = hist.reshape(-1).astype(np.int32)
        oo = np.arange(B + 1, dtype=np.int64) * t
        seed = advanced(w.seed, t)
        o = sample_parallel(xh, V, W.DTYPE_F32, w.temperature, w.top_k, w.top_p, w.min_p,
                            w.presence, w.frequency, w.repetition, seed, w.prompt_ids,
                            w.prompt_offsets, oi, oo, n)
        compare_tokens(tok, lp, tid, tlp, o, f"large step {t}")
