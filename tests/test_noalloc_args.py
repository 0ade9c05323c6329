"""The no-allocation entry point's Python binding rejects short host arrays
and wrong output tensors before the C library reads or writes B rows of them
(a short buffer would otherwise be read or written past its end)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from device_token_sampling_gb300 import sampler as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()


def args(B=4, V=1000, n=2):
    x = torch.zeros(B, V, device="cuda")
    host = dict(temperature=np.ones(B, np.float32), top_k=np.zeros(B, np.int32),
                top_p=np.ones(B, np.float32), min_p=np.zeros(B, np.float32),
                seed=np.arange(B, dtype=np.uint64))
    outs = dict(out_tokens=torch.zeros(B, dtype=torch.int32, device="cuda"),
                out_logprobs=torch.zeros(B, dtype=torch.float32, device="cuda"),
                out_topk_ids=torch.zeros(B, n, dtype=torch.int32, device="cuda"),
                out_topk_logprobs=torch.zeros(B, n, dtype=torch.float32, device="cuda"),
                row_status=torch.zeros(B, dtype=torch.int32, device="cuda"))
    return x, host, outs


def call(x, host, outs, n=2):
    return S.sample_noalloc(x, host["temperature"], host["top_k"], host["top_p"], host["min_p"],
                            host["seed"], num_logprobs=n, **outs)


def test_valid_call_runs():
    x, host, outs = args()
    call(x, host, outs)
    torch.cuda.synchronize()
    assert (outs["row_status"].cpu().numpy() == 0).all()


@pytest.mark.parametrize("name", ["temperature", "top_k", "top_p", "min_p", "seed"])
def test_short_host_array(name):
    x, host, outs = args()
    host[name] = host[name][:3]
    with pytest.raises(ValueError, match=name):
        call(x, host, outs)


@pytest.mark.parametrize("name,bad", [
    ("out_tokens", lambda: torch.zeros(3, dtype=torch.int32, device="cuda")),
    ("out_tokens", lambda: torch.zeros(4, dtype=torch.int64, device="cuda")),
    ("out_tokens", lambda: torch.zeros(4, dtype=torch.int32)),
    ("out_logprobs", lambda: torch.zeros(4, dtype=torch.float16, device="cuda")),
    ("out_topk_ids", lambda: torch.zeros(4, 1, dtype=torch.int32, device="cuda")),
    ("out_topk_logprobs", lambda: torch.zeros(2, 4, dtype=torch.float32, device="cuda").t()),
    ("row_status", lambda: torch.zeros(8, dtype=torch.int32, device="cuda")),
    ("out_topk_ids", lambda: None),
])
def test_bad_output(name, bad):
    x, host, outs = args()
    outs[name] = bad()
    with pytest.raises(ValueError, match=name):
        call(x, host, outs)
