"""The CPU oracle over many rows on all host cores (test infrastructure).

Rows are independent, so a batch splits into chunks of rows, each run by the
plain single-threaded oracle in a process of its own (started with 'spawn',
never forked from a process that holds a GPU context).  Every row keeps its
batch index as the key of its noise stream.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _run(args):
    import oracle as O
    (first, logits, V, dtype, T, K, Pp, MP, pres, freq, rep, seed, pi, po, oi, oo, n) = args
    return O.sample(logits, V, dtype, T, K, Pp, MP, pres, freq, rep, seed, pi, po, oi, oo, n,
                    want_zt=False, first_row=first)


def _rows_csr(ids, offs, a, b):
    lo, hi = int(offs[a]), int(offs[b])
    return np.ascontiguousarray(ids[lo:hi]), (offs[a:b + 1] - offs[a]).astype(np.int64)


def sample_parallel(logits, V, dtype, T, K, Pp, MP, pres, freq, rep, seed, pi, po, oi, oo, n,
                    procs: int | None = None):
    """The oracle's OracleOut for every row, computed over `procs` processes."""
    import oracle as O
    B = logits.shape[0]
    procs = procs or max(1, min(os.cpu_count() or 1, 32))
    bounds = np.linspace(0, B, procs + 1).astype(int)
    jobs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if a == b:
            continue
        pia, poa = _rows_csr(pi, po, a, b)
        oia, ooa = _rows_csr(oi, oo, a, b)
        jobs.append((int(a), np.ascontiguousarray(logits[a:b]), V, dtype, T[a:b], K[a:b],
                     Pp[a:b], MP[a:b], pres[a:b], freq[a:b], rep[a:b], seed[a:b], pia, poa, oia,
                     ooa, n))
    O.build()
    with mp.get_context("spawn").Pool(len(jobs)) as pool:
        outs = pool.map(_run, jobs)
    return O._concat(outs)
