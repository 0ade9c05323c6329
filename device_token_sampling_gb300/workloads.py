"""Seeded synthetic inputs for the batched decode sampler.

This module only makes inputs: logits rows, per-row sampling parameters,
penalty histories and seeds.  It holds none of the sampler's arithmetic, so
both the CUDA path and the CPU oracle can be fed from it without sharing any
sampling code.  It imports numpy only (torch is used by callers to move the
arrays to the device).

The workloads follow the five configurations the sampler is measured on
(the per-step decode sampler of the Tenstorrent sampling README, the vllm.cpp
Gumbel-draw pull request and the TensorRT-LLM "Sampling" page):

* ``tiny``  -- B=4, V=1,000 fp32 logits ~ N(0, 2); one row per strategy.
* ``b32``   -- B=32, V=151,936 bf16 "peaked" logits; T=1, top_k=20, top_p=0.95
               (and a second pass at T=0).
* ``b64``   -- B=64, V=248,320 fp32 peaked logits with presence/frequency/
               repetition penalties over 2,048 prompt + 512 output Zipf ids.
* ``b256``  -- B=256, V=151,936 bf16 peaked logits, mixed per-row strategies,
               20 top log-probs per row.
* ``large`` -- B=1,024, V=248,320 fp32 peaked logits, 4,096-token Zipf
               histories, all filters on, 5 top log-probs, many decode steps.

"Peaked" rows: a N(0, sigma=1.5) base with 8 distinct positions per row raised
by U(8, 12), a stand-in for language-model output (the pages measure on a 27B
checkpoint and real prompts, neither of which is used here).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DTYPE_F32 = 0
DTYPE_BF16 = 1

NAMES = ("tiny", "b32", "b64", "b256", "large")


@dataclass
class Workload:
    """One batch of sampler inputs, all host-side numpy arrays.

    ``logits`` is ``float32[B, ld]`` for fp32 rows or ``uint16[B, ld]`` holding
    bf16 bit patterns for bf16 rows; columns ``[V, ld)`` are padding and hold
    NaN so that a reader of the padding is caught.  Histories are CSR arrays:
    row ``r`` owns ``ids[offsets[r]:offsets[r+1]]``.
    """

    name: str
    B: int
    V: int
    ld: int
    dtype: int
    logits: np.ndarray
    temperature: np.ndarray
    top_k: np.ndarray
    top_p: np.ndarray
    min_p: np.ndarray
    presence: np.ndarray
    frequency: np.ndarray
    repetition: np.ndarray
    seed: np.ndarray
    prompt_ids: np.ndarray
    prompt_offsets: np.ndarray
    output_ids: np.ndarray
    output_offsets: np.ndarray
    num_logprobs: int
    notes: dict = field(default_factory=dict)
    # per row: the first prompt_ignore[r] prompt ids count for the repetition
    # penalty only (None: 0 on every row)
    prompt_ignore: np.ndarray | None = None

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == DTYPE_F32 else 2

    def logits_bytes(self) -> int:
        return self.B * self.V * self.elem_size


# --------------------------------------------------------------------------
# element generators
# --------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns uint16 bits.

    Only finite values and +-inf/NaN are expected; NaN keeps a quiet NaN bit.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    nan = np.isnan(a)
    safe = np.where(nan, np.uint32(0), bits)  # finite and inf values cannot wrap below
    rounded = (safe + (np.uint32(0x7FFF) + ((safe >> 16) & np.uint32(1)))) >> 16
    if nan.any():
        rounded = np.where(nan, (bits >> 16) | np.uint32(0x40), rounded)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def peaked_rows(rng: np.random.Generator, B: int, V: int, sigma: float = 1.5,
                n_peaks: int = 8, lo: float = 8.0, hi: float = 12.0) -> np.ndarray:
    """fp32[B, V]: N(0, sigma) plus ``n_peaks`` distinct positions raised by U(lo, hi)."""
    x = rng.standard_normal(size=(B, V), dtype=np.float32) * np.float32(sigma)
    for r in range(B):
        pos = rng.choice(V, size=n_peaks, replace=False)
        x[r, pos] += rng.uniform(lo, hi, size=n_peaks).astype(np.float32)
    return x


def zipf_ids(rng: np.random.Generator, n: int, V: int, s: float = 1.1) -> np.ndarray:
    """``n`` ids drawn from a finite Zipf(s) law over ranks 1..V (id = rank - 1)."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    ids = np.searchsorted(cdf, rng.random(n), side="right")
    return np.minimum(ids, V - 1).astype(np.int32)


def seeds(rng: np.random.Generator, B: int) -> np.ndarray:
    return rng.integers(0, 2**64, size=B, dtype=np.uint64)


def csr(rows: list[np.ndarray]) -> tuple[np.ndarray, np.ndarray]:
    offs = np.zeros(len(rows) + 1, dtype=np.int64)
    for i, r in enumerate(rows):
        offs[i + 1] = offs[i] + len(r)
    ids = np.concatenate(rows).astype(np.int32) if rows and offs[-1] > 0 else np.zeros(0, np.int32)
    return ids, offs


def pad_rows(x: np.ndarray, ld: int, dtype: int) -> np.ndarray:
    """Store fp32 values ``x[B, V]`` in the requested dtype with row stride ``ld``."""
    B, V = x.shape
    if dtype == DTYPE_F32:
        out = np.full((B, ld), np.nan, dtype=np.float32)
        out[:, :V] = x
    else:
        out = np.full((B, ld), 0x7FC0, dtype=np.uint16)
        out[:, :V] = f32_to_bf16_bits(x)
    return out


def neutral_params(B: int):
    return dict(
        temperature=np.ones(B, np.float32), top_k=np.zeros(B, np.int32),
        top_p=np.ones(B, np.float32), min_p=np.zeros(B, np.float32),
        presence=np.zeros(B, np.float32), frequency=np.zeros(B, np.float32),
        repetition=np.ones(B, np.float32))


def empty_history(B: int):
    z = np.zeros(B + 1, np.int64)
    return dict(prompt_ids=np.zeros(0, np.int32), prompt_offsets=z.copy(),
                output_ids=np.zeros(0, np.int32), output_offsets=z.copy())


# --------------------------------------------------------------------------
# the five configurations
# --------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    """B=4, V=1000 fp32 ~ N(0, 2); one row per strategy, 16+8 history ids per row."""
    rng = np.random.default_rng(seed)
    B, V = 4, 1000
    x = rng.normal(0.0, 2.0, size=(B, V)).astype(np.float32)
    p = neutral_params(B)
    p["temperature"][:] = [0.0, 0.7, 1.0, 1.0]
    p["top_k"][2] = 8
    p["top_p"][2] = 0.5
    p["min_p"][3] = 0.1
    p["presence"][3] = 0.5
    p["frequency"][3] = 0.3
    p["repetition"][3] = 1.2
    pi, po = csr([rng.integers(0, V, 16).astype(np.int32) for _ in range(B)])
    oi, oo = csr([rng.integers(0, V, 8).astype(np.int32) for _ in range(B)])
    return Workload("tiny", B, V, V, DTYPE_F32, pad_rows(x, V, DTYPE_F32), seed=seeds(rng, B),
                    prompt_ids=pi, prompt_offsets=po, output_ids=oi, output_offsets=oo,
                    num_logprobs=5, **p)


def b32(seed: int = 1, greedy: bool = False, B: int = 32, V: int = 151_936) -> Workload:
    """B=32, V=151,936 bf16 peaked rows; T=1, top_k=20, top_p=0.95 (or all greedy)."""
    rng = np.random.default_rng(seed)
    x = peaked_rows(rng, B, V)
    p = neutral_params(B)
    if greedy:
        p["temperature"][:] = 0.0
    else:
        p["top_k"][:] = 20
        p["top_p"][:] = 0.95
    return Workload("b32" + ("_greedy" if greedy else ""), B, V, V, DTYPE_BF16,
                    pad_rows(x, V, DTYPE_BF16), seed=seeds(rng, B), num_logprobs=0,
                    **p, **empty_history(B))


def b64(seed: int = 2, B: int = 64, V: int = 248_320, n_prompt: int = 2048,
        n_output: int = 512) -> Workload:
    """B=64, V=248,320 fp32 peaked rows, penalties over Zipf(1.1) histories."""
    rng = np.random.default_rng(seed)
    x = peaked_rows(rng, B, V)
    p = neutral_params(B)
    p["presence"][:] = 0.5
    p["frequency"][:] = 0.3
    p["repetition"][:] = 1.1
    p["temperature"][:] = 0.8
    p["top_k"][:] = 32
    p["top_p"][:] = 0.9
    pi, po = csr([zipf_ids(rng, n_prompt, V) for _ in range(B)])
    oi, oo = csr([zipf_ids(rng, n_output, V) for _ in range(B)])
    return Workload("b64", B, V, V, DTYPE_F32, pad_rows(x, V, DTYPE_F32), seed=seeds(rng, B),
                    prompt_ids=pi, prompt_offsets=po, output_ids=oi, output_offsets=oo,
                    num_logprobs=0, **p)


def b256_params(rng: np.random.Generator, B: int) -> dict:
    """Mixed strategies by row class r mod 4: greedy / top-k only / top-p only /
    top_k=50 + top_p=0.95 + min_p=0.05; T ~ U[0.3, 1.5] on the sampled rows."""
    p = neutral_params(B)
    for r in range(B):
        cls = r % 4
        if cls == 0:
            p["temperature"][r] = 0.0
            continue
        p["temperature"][r] = rng.uniform(0.3, 1.5)
        if cls == 1:
            p["top_k"][r] = rng.integers(1, 1025)
        elif cls == 2:
            p["top_p"][r] = rng.uniform(0.5, 0.99)
        else:
            p["top_k"][r] = 50
            p["top_p"][r] = 0.95
            p["min_p"][r] = 0.05
    return p


def b256(seed: int = 3, B: int = 256, V: int = 151_936, with_logits: bool = True) -> Workload:
    """B=256, V=151,936 bf16 peaked rows, mixed per-row strategies, 20 top log-probs."""
    rng = np.random.default_rng(seed)
    x = peaked_rows(rng, B, V) if with_logits else np.zeros((B, 0), np.float32)
    p = b256_params(rng, B)
    logits = pad_rows(x, V, DTYPE_BF16) if with_logits else np.zeros((0, V), np.uint16)
    return Workload("b256", B, V, V, DTYPE_BF16, logits, seed=seeds(rng, B), num_logprobs=20,
                    **p, **empty_history(B))


def large_params(rng: np.random.Generator, B: int) -> dict:
    p = neutral_params(B)
    p["presence"][:] = 0.4
    p["frequency"][:] = 0.2
    p["repetition"][:] = 1.05
    p["temperature"][:] = rng.uniform(0.5, 1.2, size=B).astype(np.float32)
    p["top_k"][:] = rng.integers(1, 33, size=B)
    p["top_p"][:] = 0.95
    p["min_p"][:] = 0.02
    return p


def large(seed: int = 4, B: int = 1024, V: int = 248_320, n_prompt: int = 4096,
          with_logits: bool = True) -> Workload:
    """B=1,024 (32 groups x 32 rows flattened), V=248,320 fp32 peaked rows,
    4,096-token Zipf histories; the logits of step t use seed 1000 + t."""
    rng = np.random.default_rng(seed)
    p = large_params(rng, B)
    pi, po = csr([zipf_ids(rng, n_prompt, V) for _ in range(B)])
    x = peaked_rows(np.random.default_rng(1000), B, V) if with_logits else None
    logits = pad_rows(x, V, DTYPE_F32) if with_logits else np.zeros((0, V), np.float32)
    return Workload("large", B, V, V, DTYPE_F32, logits, seed=seeds(rng, B),
                    prompt_ids=pi, prompt_offsets=po,
                    output_ids=np.zeros(0, np.int32), output_offsets=np.zeros(B + 1, np.int64),
                    num_logprobs=5, **p)


def large_step_logits(step: int, B: int = 1024, V: int = 248_320) -> np.ndarray:
    """Host copy of the step-``step`` logits of the large workload (seed 1000+step)."""
    return peaked_rows(np.random.default_rng(1000 + step), B, V)


def get(name: str, **kw) -> Workload:
    return {"tiny": tiny, "b32": b32, "b64": b64, "b256": b256, "large": large}[name](**kw)
