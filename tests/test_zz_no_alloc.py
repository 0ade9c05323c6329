"""vt_sample_noalloc, the entry point that allocates nothing, against vt_sample.

Both run the same sampling kernel; the no-allocation call keeps its per-row
state in the library's fixed device scratch array instead of a handle's
buffers, so its outputs must equal the handle's bit for bit.  Two calls in a
row check that what one call leaves in the shared scratch does not leak into
the next.  The file is named to be collected last, and passes alone in a fresh
process as well as after the other tests."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from device_token_sampling_gb300 import _build
from device_token_sampling_gb300 import sampler as S
from device_token_sampling_gb300 import workloads as W


def _case(seed, B, V, dtype, ld, n):
    rng = np.random.default_rng(seed)
    x = W.peaked_rows(rng, B, V)
    if ld > V:
        x = np.concatenate([x, rng.normal(0, 1, (B, ld - V)).astype(np.float32)], axis=1)
    T = rng.choice([0.0, 0.7, 1.0, 1.3], B).astype(np.float32)
    k = rng.choice([0, 0, 1, 20, 300], B).astype(np.int32)
    p = rng.choice([1.0, 1.0, 0.9, 0.5], B).astype(np.float32)
    mp = rng.choice([0.0, 0.0, 0.05], B).astype(np.float32)
    seeds = rng.integers(0, 2**63, B, dtype=np.uint64)
    if dtype == W.DTYPE_BF16:
        dev = torch.from_numpy(W.f32_to_bf16_bits(x).view(np.int16)).cuda()
    else:
        dev = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return dict(x=dev, V=V, dtype=dtype, n=n, T=T, k=k, p=p, mp=mp, seed=seeds)


def _outputs(c):
    B, n = c["x"].shape[0], c["n"]
    dev = c["x"].device
    return dict(token=torch.full((B,), -7, dtype=torch.int32, device=dev),
                logprob=torch.full((B,), 7.0, dtype=torch.float32, device=dev),
                topn_ids=torch.full((B, n), -7, dtype=torch.int32, device=dev),
                topn_lp=torch.full((B, n), 7.0, dtype=torch.float32, device=dev),
                status=torch.full((B,), -7, dtype=torch.int32, device=dev))


def _noalloc(c, out):
    S.sample_noalloc(c["x"], c["T"], c["k"], c["p"], c["mp"], c["seed"], out["token"],
                     V=c["V"], dtype=c["dtype"], num_logprobs=c["n"], out_logprobs=out["logprob"],
                     out_topk_ids=out["topn_ids"] if c["n"] else None,
                     out_topk_logprobs=out["topn_lp"] if c["n"] else None,
                     row_status=out["status"], synchronize=True)


def _handle(c):
    B = c["x"].shape[0]
    with S.Sampler(max_batch=B, max_vocab=c["V"], max_logprobs=c["n"], max_history=0,
                   device=c["x"].device.index) as s:
        s.reset_params(c["T"], c["k"], c["p"], c["mp"], np.zeros(B), np.zeros(B), np.ones(B),
                       c["seed"])
        tok, lp, tid, tlp = s.sample(c["x"], V=c["V"], num_logprobs=c["n"], dtype=c["dtype"])
        st = s.row_status(B)
        torch.cuda.synchronize()
        s.check_device_errors()
        return dict(token=tok.cpu().numpy(), logprob=lp.cpu().numpy(),
                    topn_ids=tid.cpu().numpy(), topn_lp=tlp.cpu().numpy(),
                    status=st.cpu().numpy())


def test_rejects_batch_beyond_limit():
    """Checked before any CUDA call, so this runs without a GPU."""
    lib = ctypes.CDLL(_build.build())
    fn = lib.vt_sample_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = S.SIGNATURES["vt_sample_noalloc"][1]
    err = ctypes.create_string_buffer(256)
    rc = fn(0, None, W.DTYPE_BF16, S.NOALLOC_MAX_BATCH + 1, 1000, 1000, None, None, None, None,
            None, 0, None, None, None, None, None, 1, None, err, len(err))
    assert rc == S.VT_ERR_CAPACITY
    assert b"1024" in err.value and b"1025" in err.value


@pytest.mark.gpu
def test_noalloc_matches_handle_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    cases = [_case(1, 64, 151_936, W.DTYPE_BF16, 151_936, 5),
             _case(2, 200, 32_003, W.DTYPE_F32, 32_008, 0)]
    outs = [_outputs(c) for c in cases]
    torch.cuda.synchronize()
    _noalloc(cases[0], outs[0])
    free_before = torch.cuda.mem_get_info()[0]
    _noalloc(cases[1], outs[1])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "the call changed free device memory"
    for i, (c, o) in enumerate(zip(cases, outs)):
        want = _handle(c)
        got = {k: v.cpu().numpy() for k, v in o.items()}
        if not c["n"]:
            got.pop("topn_ids"), got.pop("topn_lp")
            want.pop("topn_ids"), want.pop("topn_lp")
        for k in want:
            np.testing.assert_array_equal(got[k], want[k], err_msg=f"call {i}: {k}")
        assert (got["status"] == 0).all()
        assert (got["token"] >= 0).all() and (got["token"] < c["V"]).all()
