"""Scalar CPU oracle for the AttnRes mixture -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library and
never imports it.  The arithmetic lives in ``attn_res_ref.c`` (plain C,
IEEE double); this module only marshals numpy arrays of bf16 bit patterns
(``uint16``) into it.

Pins (tests/test_oracle_*.py) tie it to facts fixed by the pages and by
mathematics: the S=0 closed form (RMSNorm of the current row), identical
sources, weights summing to one, scale invariance of logits, hard selection,
permutation of bank slots, the S=1 sigmoid form, hand-derived tiny cases, a
brute-force float64 restatement at tiny H, and planted mistakes that the pins
must catch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_U16P = ctypes.POINTER(ctypes.c_uint16)
_F64P = ctypes.POINTER(ctypes.c_double)


def _u16(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.uint16
    return a.ctypes.data_as(_U16P)


def _elem_stride(a: np.ndarray, axis: int) -> int:
    s = a.strides[axis]
    assert s % 2 == 0
    return s // 2


class Oracle:
    """One loaded build of the oracle's shared object."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64 = ctypes.c_int64
        lib.attn_res_ref.restype = ctypes.c_int
        lib.attn_res_ref.argtypes = [
            _U16P, _U16P, _U16P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _U16P, _U16P, _U16P, ctypes.c_float, ctypes.c_float, _U16P,
            i64, i64, i64, i64, i64, i64, i64, i64, _F64P, _F64P, ctypes.c_int]
        lib.attn_res_ref_round_bf16.restype = None
        lib.attn_res_ref_round_bf16.argtypes = [_F64P, _U16P, i64]
        lib.attn_res_ref_widen_bf16.restype = None
        lib.attn_res_ref_widen_bf16.argtypes = [_U16P, _F64P, i64]
        self.lib = lib
        self.path = path

    def round_bf16(self, x) -> np.ndarray:
        """float64 array -> bf16 bit patterns, round to nearest even."""
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.attn_res_ref_round_bf16(x.ctypes.data_as(_F64P), _u16(out), x.size)
        return out

    def widen_bf16(self, b) -> np.ndarray:
        """bf16 bit patterns -> float64 (exact)."""
        b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.attn_res_ref_widen_bf16(_u16(b), out.ctypes.data_as(_F64P), b.size)
        return out

    def attn_res(self, prefix: np.ndarray, delta: Optional[np.ndarray],
                 blocks: Optional[np.ndarray], num_blocks: int,
                 block_write_idx: int, res_w: np.ndarray, rms_w: np.ndarray,
                 out_norm_w: Optional[np.ndarray], eps: float, out_eps: float,
                 out: Optional[np.ndarray] = None, n_threads: int = 1,
                 want_weights: bool = False, blocks_group: int = 1):
        """Run the oracle in place on numpy uint16 (bf16-bit) arrays.

        ``prefix``/``delta``/``out`` are [T, >=H] views with unit inner
        stride; ``blocks`` is a [T, capacity, >=H] view with unit inner stride
        (padding columns allowed), or [ceil(T / B), capacity, >=H] with
        ``blocks_group`` = B > 1 token rows per bank row.  ``prefix`` and
        ``blocks`` are modified in place exactly as the library contract says.  Returns ``out`` (and the
        softmax weights and logits, [T, S+1] float64, when ``want_weights``).
        """
        T = prefix.shape[0]
        H = res_w.shape[0]
        assert prefix.shape[1] >= H and prefix.strides[1] == 2
        if out is None:
            out = np.zeros((T, H), dtype=np.uint16)
        if delta is not None:
            assert delta.strides[1] == 2 and delta.shape[0] == T
        cap = bt = bs = 0
        if blocks is not None:
            assert blocks.strides[2] == 2 and blocks.shape[0] == -(-T // blocks_group)
            cap = blocks.shape[1]
            bt = _elem_stride(blocks, 0)
            bs = _elem_stride(blocks, 1)
        N = num_blocks + 1
        w = np.zeros((T, N), dtype=np.float64) if want_weights else None
        lg = np.zeros((T, N), dtype=np.float64) if want_weights else None
        rc = self.lib.attn_res_ref(
            _u16(prefix), _u16(delta), _u16(blocks), num_blocks,
            block_write_idx, cap, _u16(res_w), _u16(rms_w), _u16(out_norm_w),
            eps, out_eps, _u16(out), T, H, _elem_stride(prefix, 0),
            _elem_stride(delta, 0) if delta is not None else 0, bt, bs,
            _elem_stride(out, 0), blocks_group, None if w is None else w.ctypes.data_as(_F64P),
            None if lg is None else lg.ctypes.data_as(_F64P), n_threads)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (status {rc})")
        if want_weights:
            return out, w, lg
        return out


_default: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def round_bf16(x) -> np.ndarray:
    return default().round_bf16(x)


def widen_bf16(b) -> np.ndarray:
    return default().widen_bf16(b)


def attn_res_ref(*args, **kwargs):
    return default().attn_res(*args, **kwargs)


def run_workload(wl, n_threads: int = 1, want_weights: bool = False,
                 tokens=None, oracle: Optional[Oracle] = None):
    """Run the oracle on a workload object (see the package's ``workloads``
    module) on copies of its arrays.  ``tokens`` (an index array) restricts
    the run to those token rows.  Returns a dict with ``out``, the updated
    ``prefix`` and ``bank`` (of the selected rows) and optionally weights."""
    o = oracle or default()
    group = getattr(wl, "group", 1)
    if group > 1 and tokens is not None:
        raise ValueError("token sampling needs one bank row per token (group 1)")
    idx = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    prefix = np.ascontiguousarray(wl.prefix[idx])
    delta = None if wl.delta is None else np.ascontiguousarray(wl.delta[idx])
    bank = np.ascontiguousarray(wl.bank if group > 1 else wl.bank[idx])
    res = o.attn_res(prefix, delta, bank[:, :, : wl.H], wl.num_blocks,
                     wl.block_write_idx, wl.res_w, wl.rms_w, wl.out_norm_w,
                     wl.eps, wl.out_eps, None, n_threads, want_weights,
                     blocks_group=group)
    d = dict(prefix=prefix, bank=bank, tokens=idx)
    if want_weights:
        d["out"], d["weights"], d["logits"] = res
    else:
        d["out"] = res
    return d


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)
