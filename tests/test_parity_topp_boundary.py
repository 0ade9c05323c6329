"""GPU parity at the top-p boundary [TensorRT-LLM "Sampling", top-p: keep the
smallest set of most probable tokens whose probability exceeds top_p].

Rows are built so that one prefix ratio of the sorted, renormalised masses sits
a chosen distance from top_p:
  * 2e-6 away (either side): outside the oracle's 1e-6 tie window, so the GPU's
    kept count, boundary element and token must equal the oracle's exactly --
    the masses the GPU sums are accurate to well inside that window;
  * 5e-7 away: a tie by the oracle's rule; the oracle flags the row and either
    side of the boundary is accepted.
The ratios are read off the oracle's own tempered logits; the expected outputs
come from the oracle run with the chosen top_p.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from device_token_sampling_gb300 import workloads as W

from paritylib import compare, custom_workload, make_sampler, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from device_token_sampling_gb300 import _build
    _build.build()
    O.build()


def prefix_ratios(zt_row, k):
    """Exclusive prefix masses over the top-k survivors (k = 0: all), in the
    total order, divided by their sum."""
    z = zt_row.astype(np.float64)
    idx = np.arange(len(z))
    order = np.lexsort((idx, -z))
    if 1 < k < len(z):
        order = order[:k]
    w = np.exp(z[order] - z.max())
    pre = np.concatenate([[0.0], np.cumsum(w)])
    return pre[:-1] / pre[-1]


def pick_boundaries(R, rng, want, gap=5e-6):
    """Positions i >= 1 whose ratio is isolated by `gap` from both neighbours."""
    ok = [i for i in range(1, len(R) - 1)
          if R[i] - R[i - 1] > gap and R[i + 1] - R[i] > gap and 0.05 < R[i] < 0.995]
    rng.shuffle(ok)
    return ok[:want]


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F32])
@pytest.mark.parametrize("delta", [2e-6, -2e-6, 5e-7, -5e-7])
def test_top_p_near_boundary(dtype, delta):
    rng = np.random.default_rng(2024 + int(delta * 1e8) + 7 * dtype)
    V = 60_000
    base = W.peaked_rows(rng, 8, V)
    T = np.array([1.0, 1.5, 1.2, 0.8, 1.0, 1.5, 1.1, 1.3], np.float32)
    K = np.array([0, 0, 0, 0, 400, 2000, 0, 60], np.int32)
    # the oracle's tempered logits fix the ratios
    probe = custom_workload(base, dtype=dtype, T=T, k=K, p=1.0)
    zt = O.sample_workload(probe, want_zt=True).zt
    rows, P = [], []
    for r in range(8):
        R = prefix_ratios(zt[r], int(K[r]))
        for i in pick_boundaries(R, rng, 2):
            rows.append(r)
            P.append(np.float32(R[i] + delta))
    assert len(rows) >= 8
    x = base[rows]
    w = custom_workload(x, dtype=dtype, T=T[rows], k=K[rows], p=np.array(P, np.float32), n=3,
                        name=f"topp-boundary {delta:+g}")
    s = make_sampler(w)
    try:
        g = run_gpu(s, w)
    finally:
        s.close()
    o = O.sample_workload(w, want_zt=True)
    if abs(delta) > 1e-6:
        # outside the tie window: nothing is flagged, everything is exact
        assert not o.topp_near.any(), o.topp_near
    else:
        assert o.topp_near.all(), o.topp_near
    compare(g, o, where=w.name)
    if abs(delta) > 1e-6:
        np.testing.assert_array_equal(g["kept"], o.kept_count)
        np.testing.assert_array_equal(g["kth_index"], o.kth_index)
