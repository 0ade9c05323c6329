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

from paritylib import check_workload, custom_workload, make_sampler

pytestmark = pytest.mark.gpu


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
