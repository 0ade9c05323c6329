"""Error paths of the C ABI and host-side failure detection.

The state machine of the Tenstorrent sampling README (a sampler never reads
state that was not reset: reset_sampling_params / reset_prompt_tokens before
sample) and the host-side validation of every parameter and size.  Failures
are made on the host only: out-of-range arguments, capacities the device
cannot hold, and VT_FAULT_INJECT, which makes one allocation of
vt_sampler_create or the parameter upload of vt_reset_params fail as the CUDA
call would.  Nothing here faults the GPU.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from device_token_sampling_gb300 import sampler as S
from device_token_sampling_gb300 import workloads as W

from paritylib import check_workload, custom_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def code(exc_info):
    return exc_info.value.code


def params(B, **over):
    p = dict(temperature=np.ones(B, np.float32), top_k=np.zeros(B, np.int32),
             top_p=np.ones(B, np.float32), min_p=np.zeros(B, np.float32),
             presence=np.zeros(B, np.float32), frequency=np.zeros(B, np.float32),
             repetition=np.ones(B, np.float32), seed=np.arange(B, dtype=np.uint64))
    for k, v in over.items():
        p[k] = np.asarray(v, dtype=p[k].dtype)
    return p


def outputs(B, n=0):
    z = lambda dt, *sh: torch.zeros(*sh, dtype=dt, device="cuda")  # noqa: E731
    return (z(torch.int32, B), z(torch.float32, B), z(torch.int32, B, max(n, 1)),
            z(torch.float32, B, max(n, 1)))


def raw_sample(s, x, B, V, ld=None, n=0, dtype=W.DTYPE_F32, outs=None):
    """vt_sample through the C ABI with explicit arguments (no binding checks)."""
    tok, lp, tid, tlp = outs if outs is not None else outputs(B, n)
    lib = s._lib
    return lib.vt_sample(s.handle, S.P(x.data_ptr()), dtype, B, V, ld if ld is not None else V,
                         n, 0, S.P(tok.data_ptr()), S.P(lp.data_ptr()), S.P(tid.data_ptr()),
                         S.P(tlp.data_ptr()), None)


# --------------------------------------------------------------------------
# the state machine
# --------------------------------------------------------------------------

def test_sample_before_reset_is_a_state_error():
    with S.Sampler(4, 1000, 2, 64) as s:
        x = torch.zeros(4, 1000, device="cuda")
        assert raw_sample(s, x, 4, 1000) == S.VT_ERR_STATE
        assert b"reset" in s._lib.vt_last_error(s.handle)


def test_penalties_without_counts_is_a_state_error():
    with S.Sampler(4, 1000, 2, 64) as s:
        s.reset_params(**params(4, presence=[0, 0.5, 0, 0]))
        x = torch.zeros(4, 1000, device="cuda")
        assert raw_sample(s, x, 4, 1000) == S.VT_ERR_STATE
        # resetting the counts makes the same call valid
        z = np.zeros(5, np.int64)
        s.reset_token_counts(np.zeros(0, np.int32), z, np.zeros(0, np.int32), z)
        assert raw_sample(s, x, 4, 1000) == S.VT_OK
        torch.cuda.synchronize()


def test_more_rows_than_reset_is_a_state_error():
    with S.Sampler(8, 1000, 0, 0) as s:
        s.reset_params(**params(4))
        x = torch.zeros(8, 1000, device="cuda")
        assert raw_sample(s, x, 8, 1000) == S.VT_ERR_STATE


# --------------------------------------------------------------------------
# validation of every argument
# --------------------------------------------------------------------------

@pytest.mark.parametrize("field,value", [
    ("temperature", -1.0), ("temperature", np.inf), ("temperature", np.nan),
    ("temperature", 1e-45),  # 1 / T overflows
    ("top_k", -1), ("top_p", 1.5), ("top_p", -0.1), ("top_p", np.nan), ("min_p", 1.01),
    ("min_p", -0.5), ("repetition", 0.0), ("repetition", -1.0), ("repetition", np.nan),
    ("presence", np.inf), ("frequency", np.nan),
])
def test_reset_params_rejects(field, value):
    with S.Sampler(4, 1000, 0, 0) as s:
        p = params(4)
        p[field][2] = value
        with pytest.raises(S.VtError) as e:
            s.reset_params(**p)
        assert code(e) == S.VT_ERR_INVALID_ARG
        assert b"row 2" in s._lib.vt_last_error(s.handle)


@pytest.mark.parametrize("kw", [dict(top_p_decay=[1.0, 0.0, 1.0, 1.0]),
                                dict(top_p_decay=[1.0, 1.5, 1.0, 1.0]),
                                dict(top_p_min=[0.0, 0.1, 0.1, 0.1]),
                                dict(top_p_reset_ids=[-1, -2, -1, -1])])
def test_reset_params_ex_rejects(kw):
    with S.Sampler(4, 1000, 0, 0) as s:
        with pytest.raises(S.VtError) as e:
            s.reset_params(**params(4), **kw)
        assert code(e) == S.VT_ERR_INVALID_ARG


def test_reset_params_batch_limits():
    with S.Sampler(4, 1000, 0, 0) as s:
        with pytest.raises(S.VtError) as e:
            s.reset_params(**params(5))
        assert code(e) == S.VT_ERR_CAPACITY
        lib = s._lib
        assert lib.vt_reset_params(s.handle, 0, *([None] * 8), None) == S.VT_ERR_INVALID_ARG
        assert lib.vt_reset_params(s.handle, 2, *([None] * 8), None) == S.VT_ERR_INVALID_ARG


def test_reset_token_counts_rejects():
    with S.Sampler(2, 100, 0, 8) as s:
        ids = np.array([1, 2, 100], np.int32)          # 100 is out of range
        with pytest.raises(S.VtError) as e:
            s.reset_token_counts(ids, np.array([0, 2, 3]), np.zeros(0, np.int32),
                                 np.zeros(3, np.int64))
        assert code(e) == S.VT_ERR_INVALID_ARG
        with pytest.raises(S.VtError) as e:               # offsets going backwards
            s.reset_token_counts(np.array([1, 2], np.int32), np.array([0, 2, 1]),
                                 np.zeros(0, np.int32), np.zeros(3, np.int64))
        assert code(e) == S.VT_ERR_INVALID_ARG
        with pytest.raises(S.VtError) as e:               # a row past max_history
            s.reset_token_counts(np.arange(9, dtype=np.int32), np.array([0, 9, 9]),
                                 np.zeros(0, np.int32), np.zeros(3, np.int64))
        assert code(e) == S.VT_ERR_CAPACITY
        with pytest.raises(S.VtError) as e:               # more rows than max_batch
            s.reset_token_counts(np.zeros(0, np.int32), np.zeros(4, np.int64),
                                 np.zeros(0, np.int32), np.zeros(4, np.int64))
        assert code(e) == S.VT_ERR_CAPACITY


def test_sample_rejects():
    with S.Sampler(4, 1000, 2, 0) as s:
        s.reset_params(**params(4))
        x = torch.zeros(4, 1024, device="cuda")
        assert raw_sample(s, x, 4, 1001, ld=1024) == S.VT_ERR_CAPACITY   # V > max_vocab
        assert raw_sample(s, x, 4, 0) == S.VT_ERR_INVALID_ARG            # V < 1
        assert raw_sample(s, x, 4, 1000, ld=999) == S.VT_ERR_INVALID_ARG  # ld < V
        assert raw_sample(s, x, 4, 1000, n=3) == S.VT_ERR_CAPACITY       # n > max_logprobs
        assert raw_sample(s, x, 4, 1000, dtype=7) == S.VT_ERR_INVALID_ARG
        assert raw_sample(s, x, 0, 1000) == S.VT_ERR_INVALID_ARG         # B < 1
        lib = s._lib
        rc = lib.vt_sample(s.handle, S.P(x.data_ptr()), W.DTYPE_F32, 4, 1000, 1024, 2, 0,
                           None, None, None, None, None)                # null outputs
        assert rc == S.VT_ERR_INVALID_ARG
        # after every rejected call the handle still samples
        assert raw_sample(s, x, 4, 1000, ld=1024) == S.VT_OK
        torch.cuda.synchronize()
        s.check_device_errors()


def test_update_counts_needs_history():
    with S.Sampler(2, 100, 0, 0) as s:
        s.reset_params(**params(2))
        x = torch.zeros(2, 100, device="cuda")
        tok, lp, tid, tlp = outputs(2)
        rc = s._lib.vt_sample(s.handle, S.P(x.data_ptr()), W.DTYPE_F32, 2, 100, 100, 0, 1,
                              S.P(tok.data_ptr()), S.P(lp.data_ptr()), None, None, None)
        assert rc == S.VT_ERR_CAPACITY


@pytest.mark.parametrize("cfg", [(0, 1000, 0, 0), (4, 0, 0, 0), (4, 1000, 33, 0),
                                 (4, 1000, 0, 40000), (4, (1 << 20) + 1, 0, 0)])
def test_create_rejects(cfg):
    with pytest.raises(S.VtError) as e:
        S.Sampler(*cfg)
    assert code(e) == S.VT_ERR_INVALID_ARG


# --------------------------------------------------------------------------
# allocation and upload failures (host-side): everything is freed
# --------------------------------------------------------------------------

def free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_create_too_large_for_the_device_frees_everything():
    S.load_library()
    before = free_bytes()
    # the count tables alone would need 2^20 rows x 32768 ids x 8 B = 256 GiB
    with pytest.raises(S.VtError) as e:
        S.Sampler(1 << 20, 1 << 20, 32, 32768)
    assert code(e) == S.VT_ERR_CUDA
    assert abs(free_bytes() - before) <= 4 << 20


def test_injected_allocation_failures_free_everything(monkeypatch):
    S.load_library()
    with S.Sampler(8, 5000, 4, 64) as s:  # the first handle pays the one-time set-up
        pass
    before = free_bytes()
    for n in range(0, 40, 3):
        monkeypatch.setenv("VT_FAULT_INJECT", f"alloc:{n}")
        try:
            s = S.Sampler(8, 5000, 4, 64, host_io=True)
        except S.VtError as e:
            assert e.code == S.VT_ERR_CUDA
        else:  # n is past the handle's last allocation
            s.close()
        assert abs(free_bytes() - before) <= 4 << 20, n
    monkeypatch.delenv("VT_FAULT_INJECT")


def test_injected_upload_failure_invalidates_the_parameters(monkeypatch):
    rng = np.random.default_rng(5)
    x = rng.normal(0, 2, size=(4, 3000)).astype(np.float32)
    w = custom_workload(x, T=[0.0, 0.8, 1.0, 1.2], k=[0, 5, 0, 40], p=[1.0, 1.0, 0.7, 0.9],
                        n=2, name="after upload failure")
    with S.Sampler(4, 3000, 2, 64) as s:
        monkeypatch.setenv("VT_FAULT_INJECT", "upload")
        with pytest.raises(S.VtError) as e:
            s.reset_workload(w)
        assert code(e) == S.VT_ERR_CUDA
        xd = torch.from_numpy(x).cuda()
        assert raw_sample(s, xd, 4, 3000) == S.VT_ERR_STATE
        monkeypatch.delenv("VT_FAULT_INJECT")
        check_workload(w, s=s)  # a clean reset makes the handle sample exactly again


# --------------------------------------------------------------------------
# a device wait that runs out (bounded; nothing faults)
# --------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_the_handle_still_samples():
    w = custom_workload(np.random.default_rng(3).normal(0, 2, size=(4, 3000)).astype(np.float32),
                        T=[0.0, 0.8, 1.0, 1.2], k=[0, 5, 0, 40], p=[1.0, 1.0, 0.7, 0.9], n=2,
                        name="after a timeout")
    with S.Sampler(4, 3000, 2, 64) as s:
        assert s._lib.vt_debug_wait_probe(s.handle, 1_000_000, None) == S.VT_OK  # 1 ms
        with pytest.raises(S.VtError) as e:
            s.check_device_errors()
        assert code(e) == S.VT_ERR_TIMEOUT
        assert b"wait" in s._lib.vt_last_error(s.handle)
        s.check_device_errors()  # the error word was cleared
        check_workload(w, s=s)
