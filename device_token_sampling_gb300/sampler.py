"""Thin ctypes binding of the C ABI in ``include/vt_sampler.h``.

Argument marshalling only: every step of the sampling path runs in the CUDA
kernels of ``libvt_sampler.so``.  PyTorch supplies device memory (output
tensors) and streams.  Importing this module loads the library and raises if it
has not been built (``device_token_sampling_gb300.build()``); there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import _build

DTYPE_F32 = 0
DTYPE_BF16 = 1

VT_OK = 0
VT_ERR_INVALID_ARG = -1
VT_ERR_STATE = -2
VT_ERR_CAPACITY = -3
VT_ERR_CUDA = -4
VT_ERR_TIMEOUT = -5

ROW_OK, ROW_NONFINITE, ROW_EMPTY, ROW_HISTORY_FULL = 0, 1, 2, 3


def library_path() -> str:
    return _build.LIB


class VtError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRNAMES.get(code, code)}: {msg}")
        self.code = code


_ERRNAMES = {VT_ERR_INVALID_ARG: "VT_ERR_INVALID_ARG", VT_ERR_STATE: "VT_ERR_STATE",
             VT_ERR_CAPACITY: "VT_ERR_CAPACITY", VT_ERR_CUDA: "VT_ERR_CUDA",
             VT_ERR_TIMEOUT: "VT_ERR_TIMEOUT"}


class Config(C.Structure):
    _fields_ = [("max_batch", C.c_int32), ("max_vocab", C.c_int32),
                ("max_logprobs", C.c_int32), ("max_history", C.c_int32),
                ("device", C.c_int32), ("host_io", C.c_int32)]


P = C.c_void_p
I32, I64 = C.c_int32, C.c_int64

# entry point -> (restype, argtypes); the single source of the binding's view
# of include/vt_sampler.h
SIGNATURES = {
    "vt_sampler_create": (C.c_int, [C.POINTER(Config), C.POINTER(P)]),
    "vt_sampler_destroy": (None, [P]),
    "vt_reset_params": (C.c_int, [P, I32, P, P, P, P, P, P, P, P, P]),
    "vt_reset_params_ex": (C.c_int, [P, I32, P, P, P, P, P, P, P, P, P, P, P, P]),
    "vt_read_top_p": (C.c_int, [P, P]),
    "vt_debug_probs_plan": (C.c_int, [I32, I32, I32, P, P]),
    "vt_reset_token_counts": (C.c_int, [P, I32, P, P, P, P, P]),
    "vt_reset_token_counts_ex": (C.c_int, [P, I32, P, P, P, P, P, P]),
    "vt_sample": (C.c_int, [P, P, I32, I32, I32, I64, I32, I32, P, P, P, P, P]),
    "vt_sample_ex": (C.c_int, [P, P, I32, I32, I32, I64, I32, I32, P, P, P, P, P, I64, P]),
    "vt_sample_host": (C.c_int, [P, P, I32, I32, I32, I64, I32, I32, P, P, P, P, P]),
    "vt_check_device_errors": (C.c_int, [P]),
    "vt_get_row_status": (C.c_int, [P, P, P]),
    "vt_debug_filter_boundary": (C.c_int, [P, P, P, P, P]),
    "vt_debug_get_counts": (C.c_int, [P, I32, P, P, I32, P]),
    "vt_debug_get_seeds": (C.c_int, [P, P]),
    "vt_debug_set_trace": (C.c_int, [P, P, I64, P]),
    "vt_debug_launch_shape": (C.c_int, [P, I32, I32, P, P, P]),
    "vt_debug_set_phase_event": (C.c_int, [P, P]),
    "vt_debug_last_handover": (C.c_int, [P, P]),
    "vt_debug_last_launches": (C.c_int, [P, P]),
    "vt_debug_set_path": (C.c_int, [P, I32]),
    "vt_sample_host_async": (C.c_int, [P, P, I32, I32, I32, I64, I32, I32, P, P, P, P, P]),
    "vt_sample_host_wait": (C.c_int, [P]),
    "vt_debug_wait_probe": (C.c_int, [P, I64, P]),
    "vt_shard_part_bytes": (I64, [I32]),
    "vt_shard_partials": (C.c_int, [P, P, I32, I32, I32, I64, I32, I32, I32, P, P]),
    "vt_shard_merge": (C.c_int, [P, P, I32, I32, I32, I32, I32, P, P, P, P, P]),
    "vt_sample_noalloc": (C.c_int, [I32, P, I32, I32, I32, I64, P, P, P, P, P, I32, P, P, P, P,
                                    P, I32, P, C.c_char_p, I32]),
    "vt_last_error": (C.c_char_p, [P]),
    "vt_status_string": (C.c_char_p, [C.c_int]),
}

_lib = None


def load_library() -> C.CDLL:
    """Load libvt_sampler.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with device_token_sampling_gb300.build()")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _np_ptr(a):
    return None if a is None else a.ctypes.data_as(P)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return P(stream.cuda_stream)


class Sampler:
    """One sampler handle (``vt_sampler_create``) on one CUDA device."""

    def __init__(self, max_batch: int, max_vocab: int, max_logprobs: int = 0,
                 max_history: int = 0, device: int | None = None, host_io: bool = False):
        import torch
        self._lib = load_library()
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        cfg = Config(max_batch, max_vocab, max_logprobs, max_history, self.device,
                     1 if host_io else 0)
        h = P()
        rc = self._lib.vt_sampler_create(C.byref(cfg), C.byref(h))
        if rc != VT_OK:
            raise VtError(rc, f"vt_sampler_create({max_batch}, {max_vocab}, {max_logprobs}, "
                              f"{max_history}, device={self.device})")
        self._h = h
        self.cfg = cfg

    # -- lifetime ------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            self._lib.vt_sampler_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self):
        return self._h

    def _check(self, rc: int, what: str):
        if rc != VT_OK:
            msg = self._lib.vt_last_error(self._h)
            raise VtError(rc, f"{what}: {msg.decode() if msg else ''}")

    # -- state ---------------------------------------------------------------
    def reset_params(self, temperature, top_k, top_p, min_p, presence, frequency, repetition,
                     seed, stream=None, top_p_decay=None, top_p_min=None, top_p_reset_ids=None):
        """Per-row parameters and seeds; the three top-p decay arrays are
        optional (None: the library's default for every row)."""
        t = np.ascontiguousarray(temperature, np.float32)
        B = t.shape[0]
        arrs = [t, np.ascontiguousarray(top_k, np.int32), np.ascontiguousarray(top_p, np.float32),
                np.ascontiguousarray(min_p, np.float32),
                np.ascontiguousarray(presence, np.float32),
                np.ascontiguousarray(frequency, np.float32),
                np.ascontiguousarray(repetition, np.float32),
                np.ascontiguousarray(seed, np.uint64)]
        for a in arrs:
            if a.shape != (B,):
                raise ValueError("every parameter array must have shape (B,)")
        decay = [None if a is None else np.ascontiguousarray(a, dt)
                 for a, dt in ((top_p_decay, np.float32), (top_p_min, np.float32),
                               (top_p_reset_ids, np.int32))]
        if all(a is None for a in decay):
            rc = self._lib.vt_reset_params(self._h, B, *[_np_ptr(a) for a in arrs],
                                           _stream_ptr(stream))
            self._check(rc, "vt_reset_params")
            return
        for a in decay:
            if a is not None and a.shape != (B,):
                raise ValueError("every top-p decay array must have shape (B,)")
        rc = self._lib.vt_reset_params_ex(self._h, B, *[_np_ptr(a) for a in arrs],
                                          *[_np_ptr(a) for a in decay],
                                          _stream_ptr(stream))
        self._check(rc, "vt_reset_params_ex")

    def reset_token_counts(self, prompt_ids, prompt_offsets, output_ids, output_offsets,
                           stream=None, prompt_ignore=None):
        pi = np.ascontiguousarray(prompt_ids, np.int32)
        po = np.ascontiguousarray(prompt_offsets, np.int64)
        oi = np.ascontiguousarray(output_ids, np.int32)
        oo = np.ascontiguousarray(output_offsets, np.int64)
        B = po.shape[0] - 1
        if oo.shape[0] != B + 1:
            raise ValueError("prompt and output offsets disagree on B")
        if prompt_ignore is None:
            rc = self._lib.vt_reset_token_counts(self._h, B, _np_ptr(pi), _np_ptr(po),
                                                 _np_ptr(oi), _np_ptr(oo), _stream_ptr(stream))
            self._check(rc, "vt_reset_token_counts")
            return
        ig = np.ascontiguousarray(prompt_ignore, np.int32)
        if ig.shape != (B,):
            raise ValueError("prompt_ignore must have shape (B,)")
        rc = self._lib.vt_reset_token_counts_ex(self._h, B, _np_ptr(pi), _np_ptr(po), _np_ptr(oi),
                                                _np_ptr(oo), _np_ptr(ig), _stream_ptr(stream))
        self._check(rc, "vt_reset_token_counts_ex")

    def reset_workload(self, w, stream=None):
        """Reset params, seeds and counts from a ``workloads.Workload``."""
        self.reset_params(w.temperature, w.top_k, w.top_p, w.min_p, w.presence, w.frequency,
                          w.repetition, w.seed, stream=stream)
        if self.cfg.max_history > 0:
            self.reset_token_counts(w.prompt_ids, w.prompt_offsets, w.output_ids,
                                    w.output_offsets, stream=stream,
                                    prompt_ignore=getattr(w, "prompt_ignore", None))

    # -- sampling ------------------------------------------------------------
    def sample(self, logits, V: int | None = None, num_logprobs: int = 0,
               update_counts: bool = False, out=None, stream=None, dtype: int | None = None,
               probs=None):
        """Sample one token per row of a CUDA tensor ``logits`` [B, ld] (float32 or
        bfloat16, or a uint16 tensor of bf16 bits with ``dtype=DTYPE_BF16``).

        Returns ``(tokens, logprobs, topk_ids, topk_logprobs)`` CUDA tensors (the
        last two have shape [B, num_logprobs]).  ``probs`` (a float32 CUDA tensor
        [B, >= V] with contiguous rows) also receives the filtered distribution of
        each row.  Stream-ordered; nothing waits."""
        import torch
        if logits.dim() != 2 or not logits.is_cuda:
            raise ValueError("logits must be a 2-D CUDA tensor")
        if logits.stride(1) != 1:
            raise ValueError("logits rows must be contiguous")
        if dtype is None:
            if logits.dtype == torch.float32:
                dtype = DTYPE_F32
            elif logits.dtype in (torch.bfloat16, torch.uint16, torch.int16):
                dtype = DTYPE_BF16
            else:
                raise ValueError(f"unsupported logits dtype {logits.dtype}")
        B, ld = logits.shape[0], logits.stride(0)
        V = logits.shape[1] if V is None else V
        n = int(num_logprobs)
        dev = logits.device
        if out is None:
            out = (torch.empty(B, dtype=torch.int32, device=dev),
                   torch.empty(B, dtype=torch.float32, device=dev),
                   torch.empty((B, n), dtype=torch.int32, device=dev),
                   torch.empty((B, n), dtype=torch.float32, device=dev))
        tok, lp, tid, tlp = out
        args = (self._h, P(logits.data_ptr()), dtype, B, V, ld, n, 1 if update_counts else 0,
                P(tok.data_ptr()), P(lp.data_ptr()) if lp is not None else None,
                P(tid.data_ptr()) if n else None, P(tlp.data_ptr()) if n else None)
        if probs is None:
            rc = self._lib.vt_sample(*args, _stream_ptr(stream))
            self._check(rc, "vt_sample")
            return out
        if (probs.dim() != 2 or not probs.is_cuda or probs.dtype != torch.float32
                or probs.shape[0] != B or probs.shape[1] < V or probs.stride(1) != 1):
            raise ValueError("probs must be a float32 CUDA tensor [B, >= V] with contiguous rows")
        rc = self._lib.vt_sample_ex(*args, P(probs.data_ptr()), probs.stride(0),
                                    _stream_ptr(stream))
        self._check(rc, "vt_sample_ex")
        return out

    def sample_ptr(self, logits_ptr: int, dtype: int, B: int, V: int, ld: int, num_logprobs: int,
                   update_counts: bool, tokens_ptr: int, logprobs_ptr: int | None,
                   topk_ids_ptr: int | None, topk_lp_ptr: int | None, stream_ptr: int):
        """vt_sample on raw device pointers (no torch involvement)."""
        rc = self._lib.vt_sample(self._h, P(logits_ptr), dtype, B, V, ld, num_logprobs,
                                 1 if update_counts else 0, P(tokens_ptr),
                                 P(logprobs_ptr) if logprobs_ptr else None,
                                 P(topk_ids_ptr) if topk_ids_ptr else None,
                                 P(topk_lp_ptr) if topk_lp_ptr else None, P(stream_ptr))
        self._check(rc, "vt_sample")

    def sample_host(self, logits: np.ndarray, V: int, dtype: int, num_logprobs: int = 0,
                    update_counts: bool = False, stream=None, out=None):
        """vt_sample_host: host logits [B, ld] in, host outputs back; synchronous."""
        x = np.ascontiguousarray(logits)
        B, ld = x.shape
        n = int(num_logprobs)
        if out is None:
            out = (np.empty(B, np.int32), np.empty(B, np.float32), np.empty((B, n), np.int32),
                   np.empty((B, n), np.float32))
        tok, lp, tid, tlp = out
        rc = self._lib.vt_sample_host(self._h, _np_ptr(x), dtype, B, V, ld, n,
                                      1 if update_counts else 0, _np_ptr(tok), _np_ptr(lp),
                                      _np_ptr(tid) if n else None, _np_ptr(tlp) if n else None,
                                      _stream_ptr(stream))
        self._check(rc, "vt_sample_host")
        return out

    def sample_host_async(self, logits: np.ndarray, V: int, dtype: int, num_logprobs: int = 0,
                          update_counts: bool = False, stream=None, out=None):
        """vt_sample_host_async: enqueue one step from host logits [B, ld]
        (pinned for an asynchronous copy); ``out`` is filled once
        ``sample_host_wait`` returns, and both must stay alive until then."""
        # the buffers are read and written after the call returns: no hidden
        # copies, and outputs of the exact dtype and shape
        if logits.ndim != 2 or not logits.flags["C_CONTIGUOUS"]:
            raise ValueError("host logits must be a C-contiguous 2-D array")
        x = logits
        B, ld = x.shape
        n = int(num_logprobs)
        if out is None:
            out = (np.empty(B, np.int32), np.empty(B, np.float32), np.empty((B, n), np.int32),
                   np.empty((B, n), np.float32))
        tok, lp, tid, tlp = out
        for arr, dt, shape in ((tok, np.int32, (B,)), (lp, np.float32, (B,)),
                               (tid, np.int32, (B, n)), (tlp, np.float32, (B, n))):
            if arr.dtype != dt or arr.shape != shape or not arr.flags["C_CONTIGUOUS"]:
                raise ValueError(f"output arrays must be C-contiguous {dt.__name__} {shape}")
        rc = self._lib.vt_sample_host_async(self._h, _np_ptr(x), dtype, B, V, ld, n,
                                            1 if update_counts else 0, _np_ptr(tok), _np_ptr(lp),
                                            _np_ptr(tid) if n else None,
                                            _np_ptr(tlp) if n else None, _stream_ptr(stream))
        self._check(rc, "vt_sample_host_async")
        return out

    def sample_host_wait(self):
        """vt_sample_host_wait: every enqueued host step complete."""
        self._check(self._lib.vt_sample_host_wait(self._h), "vt_sample_host_wait")

    # -- views -----------------------------------------------------------------
    def check_device_errors(self):
        self._check(self._lib.vt_check_device_errors(self._h), "vt_check_device_errors")

    def row_status(self, B: int, stream=None):
        import torch
        st = torch.empty(B, dtype=torch.int32, device=f"cuda:{self.device}")
        self._check(self._lib.vt_get_row_status(self._h, P(st.data_ptr()), _stream_ptr(stream)),
                    "vt_get_row_status")
        return st

    def filter_boundary(self, B: int, stream=None):
        import torch
        d = f"cuda:{self.device}"
        v = torch.empty(B, dtype=torch.float32, device=d)
        i = torch.empty(B, dtype=torch.int32, device=d)
        k = torch.empty(B, dtype=torch.int32, device=d)
        self._check(self._lib.vt_debug_filter_boundary(self._h, P(v.data_ptr()), P(i.data_ptr()),
                                                       P(k.data_ptr()), _stream_ptr(stream)),
                    "vt_debug_filter_boundary")
        return v, i, k

    def counts(self, row: int):
        cap = max(1, self.cfg.max_history)
        ids = np.zeros(cap, np.int32)
        cnt = np.zeros(cap, np.int32)
        n = C.c_int32(0)
        self._check(self._lib.vt_debug_get_counts(self._h, row, _np_ptr(ids), _np_ptr(cnt), cap,
                                                  C.byref(n)), "vt_debug_get_counts")
        return ids[:n.value].copy(), cnt[:n.value].copy()

    def launch_shape(self, dtype: int, V: int):
        c, sl, sm = C.c_int32(), C.c_int32(), C.c_int64()
        self._check(self._lib.vt_debug_launch_shape(self._h, dtype, V, C.byref(c), C.byref(sl),
                                                    C.byref(sm)), "vt_debug_launch_shape")
        return c.value, sl.value, sm.value

    def set_trace(self, buf=None):
        """Enable the per-CTA phase trace into a CUDA int64 tensor [ctas, slots]
        (None disables it).  Returns the slot count."""
        slots = C.c_int32()
        if buf is None:
            self._check(self._lib.vt_debug_set_trace(self._h, None, 0, C.byref(slots)),
                        "vt_debug_set_trace")
        else:
            self._check(self._lib.vt_debug_set_trace(self._h, P(buf.data_ptr()), buf.shape[0],
                                                     C.byref(slots)), "vt_debug_set_trace")
        return slots.value

    def set_phase_event(self, event=None):
        """Record a ``torch.cuda.Event`` between the two launches of every later
        ``sample`` (None turns it off); the caller keeps the event alive."""
        ptr = None if event is None else P(event.cuda_event)
        self._check(self._lib.vt_debug_set_phase_event(self._h, ptr), "vt_debug_set_phase_event")

    def last_handover(self) -> int:
        """Rows the last ``sample`` handed to the selection kernel."""
        v = C.c_int32()
        self._check(self._lib.vt_debug_last_handover(self._h, C.byref(v)), "vt_debug_last_handover")
        return int(v.value)

    def shard_partials(self, logits, v0: int, V: int, K: int, out=None, stream=None,
                       dtype: int | None = None):
        """vt_shard_partials: this shard's records for the columns [v0, v0 + Vs)
        held in ``logits`` [B, ld]; returns a uint8 CUDA tensor [B, part_bytes]."""
        import torch
        if logits.dim() != 2 or not logits.is_cuda or logits.stride(1) != 1:
            raise ValueError("logits must be a 2-D CUDA tensor with contiguous rows")
        if dtype is None:
            dtype = DTYPE_F32 if logits.dtype == torch.float32 else DTYPE_BF16
        B, Vs, ld = logits.shape[0], logits.shape[1], logits.stride(0)
        pb = int(self._lib.vt_shard_part_bytes(K))
        if pb < 0:
            raise ValueError(f"K={K} outside 1..256")
        if out is None:
            out = torch.empty((B, pb), dtype=torch.uint8, device=logits.device)
        elif out.dtype != torch.uint8 or tuple(out.shape) != (B, pb) or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous uint8 tensor of shape {(B, pb)}")
        rc = self._lib.vt_shard_partials(self._h, P(logits.data_ptr()), dtype, B, Vs, ld, v0, V,
                                         K, P(out.data_ptr()), _stream_ptr(stream))
        self._check(rc, "vt_shard_partials")
        return out

    def shard_merge(self, parts, V: int, K: int, num_logprobs: int = 0, stream=None):
        """vt_shard_merge over ``parts`` (uint8 CUDA [S, B, part_bytes], the
        shards' records gathered shard-major); returns (tokens, logprobs,
        topk_ids, topk_logprobs) CUDA tensors."""
        import torch
        if parts.dim() != 3 or parts.dtype != torch.uint8 or not parts.is_contiguous():
            raise ValueError("parts must be a contiguous uint8 tensor [S, B, part_bytes]")
        S_, B = parts.shape[0], parts.shape[1]
        if parts.shape[2] != int(self._lib.vt_shard_part_bytes(K)):
            raise ValueError("parts do not hold records of K elements")
        n = int(num_logprobs)
        dev = parts.device
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        lp = torch.empty(B, dtype=torch.float32, device=dev)
        tid = torch.empty((B, n), dtype=torch.int32, device=dev)
        tlp = torch.empty((B, n), dtype=torch.float32, device=dev)
        rc = self._lib.vt_shard_merge(self._h, P(parts.data_ptr()), S_, B, V, K, n,
                                      P(tok.data_ptr()), P(lp.data_ptr()),
                                      P(tid.data_ptr()) if n else None,
                                      P(tlp.data_ptr()) if n else None, _stream_ptr(stream))
        self._check(rc, "vt_shard_merge")
        return tok, lp, tid, tlp

    def set_path(self, path: int):
        """1 (the default): the streaming kernel for every call; 2: the flat
        kernels for bf16 calls without penalties or top-p decay."""
        self._check(self._lib.vt_debug_set_path(self._h, int(path)), "vt_debug_set_path")

    def last_launches(self) -> int:
        """Kernels the last ``sample`` launched (2, or 3 when its rows were split
        between the two streams)."""
        v = C.c_int32()
        self._check(self._lib.vt_debug_last_launches(self._h, C.byref(v)), "vt_debug_last_launches")
        return int(v.value)

    def top_p(self, B: int):
        """The effective top_p of rows 0..B-1 (decayed on rows with top-p decay)."""
        p = np.zeros(self.cfg.max_batch, np.float32)
        self._check(self._lib.vt_read_top_p(self._h, _np_ptr(p)), "vt_read_top_p")
        return p[:B]

    def seeds(self, B: int):
        s = np.zeros(self.cfg.max_batch, np.uint64)  # the call writes up to max_batch seeds
        self._check(self._lib.vt_debug_get_seeds(self._h, _np_ptr(s)), "vt_debug_get_seeds")
        return s[:B]


NOALLOC_MAX_BATCH = 1024


def sample_noalloc(logits, temperature, top_k, top_p, min_p, seed, out_tokens,
                   V: int | None = None, dtype: int | None = None, num_logprobs: int = 0,
                   out_logprobs=None, out_topk_ids=None, out_topk_logprobs=None,
                   row_status=None, synchronize: bool = True, stream=None):
    """``vt_sample_noalloc``: one sampling step without a handle, in the
    library's fixed device scratch.  All outputs are caller-owned CUDA tensors;
    the parameters are host sequences of length B.  Raises VtError on failure."""
    import torch
    lib = load_library()
    if logits.dim() != 2 or not logits.is_cuda or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D CUDA tensor with contiguous rows")
    if dtype is None:
        if logits.dtype == torch.float32:
            dtype = DTYPE_F32
        elif logits.dtype in (torch.bfloat16, torch.uint16, torch.int16):
            dtype = DTYPE_BF16
        else:
            raise ValueError(f"unsupported logits dtype {logits.dtype}")
    B, ld = logits.shape[0], logits.stride(0)
    V = logits.shape[1] if V is None else V
    n = int(num_logprobs)
    arr = lambda x, t: np.ascontiguousarray(np.asarray(x, dtype=t)).reshape(-1)  # noqa: E731
    T, K, Pp, MP = arr(temperature, np.float32), arr(top_k, np.int32), arr(top_p, np.float32), \
        arr(min_p, np.float32)
    S = arr(seed, np.uint64)
    # the library reads B entries of every host array and writes B rows of
    # every output: check them here, where a short buffer is still an error
    for name, a in (("temperature", T), ("top_k", K), ("top_p", Pp), ("min_p", MP),
                    ("seed", S)):
        if a.shape[0] < B:
            raise ValueError(f"{name} has {a.shape[0]} entries, need {B}")

    def check_out(t, name, dt, cols=None, required=False):
        if t is None:
            if required:
                raise ValueError(f"{name} is required")
            return
        if not t.is_cuda or t.device != logits.device:
            raise ValueError(f"{name} must be a CUDA tensor on {logits.device}")
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}, got {t.dtype}")
        want = (B,) if cols is None else (B, cols)
        if tuple(t.shape) != want or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor of shape {want}")

    check_out(out_tokens, "out_tokens", torch.int32, required=True)
    check_out(out_logprobs, "out_logprobs", torch.float32)
    check_out(row_status, "row_status", torch.int32)
    if n > 0:
        check_out(out_topk_ids, "out_topk_ids", torch.int32, n, required=True)
        check_out(out_topk_logprobs, "out_topk_logprobs", torch.float32, n, required=True)
    tp = lambda t: None if t is None else P(t.data_ptr())  # noqa: E731
    err = C.create_string_buffer(256)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    rc = lib.vt_sample_noalloc(logits.device.index,
                               P(logits.data_ptr()), dtype, B, V, ld, _np_ptr(T), _np_ptr(K),
                               _np_ptr(Pp), _np_ptr(MP), _np_ptr(S), n,
                               tp(out_tokens), tp(out_logprobs), tp(out_topk_ids),
                               tp(out_topk_logprobs), tp(row_status), 1 if synchronize else 0,
                               _stream_ptr(stream), err, len(err))
    if rc != VT_OK:
        raise VtError(rc, err.value.decode(errors="replace"))


def gather_partials(part, group=None):
    """The exchange of the vocabulary-sharded sampler: every rank's records
    ``part`` [B, part_bytes] (uint8) all-gathered over ``group`` into one
    [world, B, part_bytes] tensor, rank-major, as ``vt_shard_merge`` reads them
    (torch.distributed: NCCL for CUDA tensors, gloo for host tensors)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(part.shape), dtype=part.dtype, device=part.device)
    dist.all_gather(list(out.unbind(0)), part.contiguous(), group=group)
    return out


def sharded_sample(sampler: Sampler, logits_shard, v0: int, V: int, K: int,
                   num_logprobs: int = 0, group=None):
    """One step of the vocabulary-sharded sampler on this rank: this rank's
    records (``vt_shard_partials``) for its columns [v0, v0 + Vs), the
    all-gather of every rank's records, then the merge (``vt_shard_merge``).
    Every rank returns the same outputs and advances the same seeds."""
    part = sampler.shard_partials(logits_shard, v0, V, K)
    return sampler.shard_merge(gather_partials(part, group), V, K, num_logprobs)
