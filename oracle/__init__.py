"""ctypes front end of the CPU oracle: TEST INFRASTRUCTURE ONLY.

The oracle (``oracle.cpp``) is the plain single-threaded definition of the
batched decode sampler that the CUDA path is checked against.  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import this
package; the product package never does.  Parity status of each part (what pins
it) is listed in the test module ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
SRC = os.path.join(HERE, "oracle.cpp")
MAX_ALT = 8

# Planted mistakes the mutation tests compile in, one per variant.
MUTANTS = ("HASH", "TIE_HIGH", "PEN_ORDER", "PROMPT_ONLY", "TOPP_INCL", "TOPP_NO_RENORM",
           "SCORE_MUL", "IGNORE_ALL", "PAIR_OVERLAP", "ROW_IGNORED", "STEP_IS_ROW")


def lib_path(mutant: str | None = None) -> str:
    name = "liboracle.so" if mutant is None else f"liboracle_mut_{mutant.lower()}.so"
    return os.path.join(BUILD_DIR, name)


def build(mutant: str | None = None, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake variant) with g++; returns the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "oracle.h"))):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", SRC, "-o", out + ".tmp"]
    if mutant is not None:
        cmd.insert(1, f"-DORACLE_MUTANT_{mutant}")
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


class RowResult(C.Structure):
    _fields_ = [
        ("status", C.c_int32), ("greedy", C.c_int32), ("token", C.c_int32),
        ("kept_count", C.c_int32), ("kth_value", C.c_float), ("kth_index", C.c_int32),
        ("max_logit", C.c_double), ("lse", C.c_double), ("logprob", C.c_double),
        ("best_score", C.c_double), ("second_score", C.c_double),
        ("second_token", C.c_int32), ("gumbel_near_tie", C.c_int32),
        ("topp_near", C.c_int32), ("kept_lo", C.c_int32), ("kept_hi", C.c_int32),
        ("n_alt", C.c_int32), ("alt_tokens", C.c_int32 * MAX_ALT),
    ]


_libs: dict = {}


def load(mutant: str | None = None) -> C.CDLL:
    key = mutant or ""
    if key in _libs:
        return _libs[key]
    lib = C.CDLL(build(mutant))
    P = C.c_void_p
    lib.oracle_sample.restype = C.c_int
    lib.oracle_sample.argtypes = [C.c_int64, C.c_int, C.c_int, C.c_int64, C.c_int, P, P, P, P, P, P,
                                  P, P,
                                  P, P, P, P, P, C.c_int, P, P, P, P]
    lib.oracle_sample_ex.restype = C.c_int
    lib.oracle_sample_ex.argtypes = [C.c_int64, C.c_int, C.c_int, C.c_int64, C.c_int, P, P, P, P,
                                     P, P, P, P, P, P, P, P, P, P, C.c_int, P, P, P, P, P]
    lib.oracle_topp_decay.restype = C.c_float
    lib.oracle_topp_decay.argtypes = [C.c_float, C.c_float, C.c_float, C.c_float, C.c_int32,
                                      C.c_int32]
    lib.oracle_filtered_probs.restype = C.c_int
    lib.oracle_filtered_probs.argtypes = [P, C.c_int, C.c_int64, P]
    lib.oracle_mix64.restype = C.c_uint64
    lib.oracle_mix64.argtypes = [C.c_uint64]
    lib.oracle_uniform.restype = C.c_double
    lib.oracle_uniform.argtypes = [C.c_uint64, C.c_int64, C.c_int64]
    lib.oracle_next_seed.restype = C.c_uint64
    lib.oracle_next_seed.argtypes = [C.c_uint64]
    lib.oracle_noise_bits.restype = C.c_int
    lib.oracle_noise_bits.argtypes = [C.c_uint64, C.c_int64, C.c_int64, C.c_int64, P]
    _libs[key] = lib
    return lib


@dataclass
class OracleOut:
    status: np.ndarray
    greedy: np.ndarray
    token: np.ndarray
    kept_count: np.ndarray
    kth_value: np.ndarray
    kth_index: np.ndarray
    max_logit: np.ndarray
    lse: np.ndarray
    logprob: np.ndarray
    best_score: np.ndarray
    second_score: np.ndarray
    second_token: np.ndarray
    gumbel_near_tie: np.ndarray
    topp_near: np.ndarray
    kept_lo: np.ndarray
    kept_hi: np.ndarray
    alt_tokens: list
    topn_ids: np.ndarray
    topn_logprobs: np.ndarray
    zt: np.ndarray | None
    probs: np.ndarray | None = None


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def sample(logits, V, dtype, temperature, top_k, top_p, min_p, presence, frequency, repetition,
           seed, prompt_ids, prompt_offsets, output_ids, output_offsets, num_logprobs,
           want_zt=False, mutant=None, rows=None, first_row=0, prompt_ignore=None,
           want_probs=False) -> OracleOut:
    """Run the oracle on host arrays.  ``logits`` is [B, ld] (fp32, or uint16 bf16 bits).

    ``rows`` (optional) restricts the call to a subset of rows; each row keeps its
    batch index as the key of its noise stream.  ``prompt_ignore`` (optional [B])
    is each row's prompt_ignore_length; ``want_probs`` returns the filtered
    distribution of every row in ``probs`` ([B, V] float64)."""
    lib = load(mutant)
    logits = np.ascontiguousarray(logits)
    B, ld = logits.shape
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        outs = [sample(logits[r:r + 1], V, dtype, temperature[r:r + 1], top_k[r:r + 1],
                       top_p[r:r + 1], min_p[r:r + 1], presence[r:r + 1], frequency[r:r + 1],
                       repetition[r:r + 1], seed[r:r + 1],
                       *_row_hist(prompt_ids, prompt_offsets, r),
                       *_row_hist(output_ids, output_offsets, r), num_logprobs,
                       want_zt=want_zt, mutant=mutant, first_row=first_row + int(r),
                       prompt_ignore=None if prompt_ignore is None else prompt_ignore[r:r + 1],
                       want_probs=want_probs)
                for r in rows]
        return _concat(outs)
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    i64 = lambda a: np.ascontiguousarray(a, dtype=np.int64)
    args = dict(t=f32(temperature), k=i32(top_k), p=f32(top_p), mp=f32(min_p), pr=f32(presence),
                fr=f32(frequency), rp=f32(repetition),
                sd=np.ascontiguousarray(seed, dtype=np.uint64), pi=i32(prompt_ids),
                po=i64(prompt_offsets), oi=i32(output_ids), oo=i64(output_offsets))
    res = (RowResult * max(B, 1))()
    n = int(num_logprobs)
    tid = np.zeros((B, n), np.int32)
    tlp = np.zeros((B, n), np.float64)
    zt = np.zeros((B, V), np.float32) if want_zt else None
    probs = np.zeros((B, V), np.float64) if want_probs else None
    ign = None if prompt_ignore is None else i32(prompt_ignore)
    rc = lib.oracle_sample_ex(int(first_row), B, V, ld, dtype, _ptr(logits), _ptr(args["t"]),
                              _ptr(args["k"]), _ptr(args["p"]), _ptr(args["mp"]),
                              _ptr(args["pr"]), _ptr(args["fr"]), _ptr(args["rp"]),
                              _ptr(args["sd"]), _ptr(args["pi"]), _ptr(args["po"]),
                              _ptr(args["oi"]), _ptr(args["oo"]), _ptr(ign), n,
                              C.cast(res, C.c_void_p), _ptr(tid) if n else None,
                              _ptr(tlp) if n else None, _ptr(zt), _ptr(probs))
    if rc != 0:
        raise ValueError("oracle_sample rejected its arguments")
    g = lambda f, dt: np.array([getattr(res[r], f) for r in range(B)], dtype=dt)
    return OracleOut(
        status=g("status", np.int32), greedy=g("greedy", np.int32), token=g("token", np.int32),
        kept_count=g("kept_count", np.int32), kth_value=g("kth_value", np.float32),
        kth_index=g("kth_index", np.int32), max_logit=g("max_logit", np.float64),
        lse=g("lse", np.float64), logprob=g("logprob", np.float64),
        best_score=g("best_score", np.float64), second_score=g("second_score", np.float64),
        second_token=g("second_token", np.int32), gumbel_near_tie=g("gumbel_near_tie", np.int32),
        topp_near=g("topp_near", np.int32), kept_lo=g("kept_lo", np.int32),
        kept_hi=g("kept_hi", np.int32),
        alt_tokens=[list(res[r].alt_tokens[:res[r].n_alt]) for r in range(B)],
        topn_ids=tid, topn_logprobs=tlp, zt=zt, probs=probs)


def _row_hist(ids, offs, r):
    a, b = int(offs[r]), int(offs[r + 1])
    return np.ascontiguousarray(ids[a:b], dtype=np.int32), np.array([0, b - a], np.int64)


def _concat(outs):
    keys = OracleOut.__dataclass_fields__.keys()
    d = {}
    for k in keys:
        vals = [getattr(o, k) for o in outs]
        if k == "alt_tokens":
            d[k] = [x for v in vals for x in v]
        elif vals[0] is None:
            d[k] = None
        else:
            d[k] = np.concatenate(vals)
    return OracleOut(**d)


def sample_workload(w, want_zt=False, rows=None, mutant=None, seed=None, top_p=None,
                    want_probs=False) -> OracleOut:
    """Run the oracle on a ``workloads.Workload`` (optionally on a subset of rows;
    ``top_p`` overrides the rows' top_p, e.g. with a decayed effective one)."""
    return sample(w.logits, w.V, w.dtype, w.temperature, w.top_k,
                  w.top_p if top_p is None else top_p, w.min_p, w.presence,
                  w.frequency, w.repetition, w.seed if seed is None else seed, w.prompt_ids,
                  w.prompt_offsets, w.output_ids, w.output_offsets, w.num_logprobs,
                  want_zt=want_zt, mutant=mutant, rows=rows,
                  prompt_ignore=getattr(w, "prompt_ignore", None), want_probs=want_probs)


def topp_decay(p: float, p_init: float, decay: float, p_min: float, reset_id: int, token: int,
               mutant=None) -> float:
    """One top-p decay step after a sampled token (fp32)."""
    return float(load(mutant).oracle_topp_decay(p, p_init, decay, p_min, reset_id, token))


def filtered_probs(zt_row, kept: int, mutant=None) -> np.ndarray:
    """The filtered distribution of one row of tempered logits whose kept set is
    the first ``kept`` entries of the total order."""
    zt_row = np.ascontiguousarray(zt_row, dtype=np.float32)
    out = np.zeros(zt_row.shape[0], np.float64)
    rc = load(mutant).oracle_filtered_probs(_ptr(zt_row), zt_row.shape[0], int(kept), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_filtered_probs rejected its arguments")
    return out


def mix64(z: int, mutant=None) -> int:
    return int(load(mutant).oracle_mix64(C.c_uint64(z)))


def uniform(seed: int, row: int, j: int, mutant=None) -> float:
    return float(load(mutant).oracle_uniform(C.c_uint64(seed), row, j))


def noise_bits(seed: int, row: int, j0: int, n: int, mutant=None) -> np.ndarray:
    """The 24-bit noise integers b_j of columns j0 .. j0 + n - 1 of ``row``."""
    out = np.zeros(int(n), np.uint32)
    rc = load(mutant).oracle_noise_bits(C.c_uint64(seed % 2**64), int(row), int(j0), int(n),
                                        _ptr(out))
    if rc != 0:
        raise ValueError("oracle_noise_bits rejected its arguments")
    return out


def next_seed(seed: int) -> int:
    return int(load().oracle_next_seed(C.c_uint64(seed)))
