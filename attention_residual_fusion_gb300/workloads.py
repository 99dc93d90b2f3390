"""Seeded synthetic inputs for the AttnRes mixture.

This module only draws random numbers and lays them out; it holds none of the
mixture's arithmetic.  Both the CUDA path (through the tests and the
benchmark) and the CPU oracle consume exactly the bf16 bit patterns made here.

Arrays are numpy ``uint16`` holding bf16 bit patterns:

* ``prefix``  [T, H]           current-layer residual (dense rows)
* ``delta``   [T, H] or None   addend for the current-layer residual
* ``bank``    [T, capacity, slot_stride]  block residual bank; columns
  H..slot_stride-1 are padding and slots >= num_blocks are unused.  Padding,
  unused slots and a write-back target slot that is not a source are filled
  with a NaN canary, so that a stray read poisons the output and a stray
  write is visible.
* ``rms_w``, ``res_w``, ``out_norm_w`` [H]

Recipes (the pages' workloads, restated as distributions):
  activations ~ N(0, 1); optionally each element independently multiplied by
  50 with probability 1% ("outliers"); optionally bank slot i scaled by one
  draw s_i ~ U(lo, hi) shared by all tokens ("per-block scale").  Weights
  rms_w, res_w, out_norm_w ~ 1 + 0.1 N(0, 1); the "mixing" recipe draws
  res_w ~ 0.02 N(0, 1) instead, which spreads the softmax over several
  sources.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

HIDDEN = 7168
CANARY = 0x7FA1  # a NaN bit pattern in bf16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Finite float32 -> bf16 bit patterns, round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    name: str
    T: int
    num_blocks: int
    capacity: int
    has_delta: bool
    has_out_norm: bool
    block_write_idx: int
    prefix: np.ndarray
    delta: Optional[np.ndarray]
    bank: np.ndarray
    rms_w: np.ndarray
    res_w: np.ndarray
    out_norm_w: Optional[np.ndarray]
    eps: float = 1e-6
    out_eps: float = 1e-6
    H: int = HIDDEN
    meta: dict = field(default_factory=dict)
    group: int = 1  # token rows per bank row (bank has ceil(T / group) rows)

    @property
    def slot_stride(self) -> int:
        return self.bank.shape[2]

    @property
    def blocks_view(self) -> np.ndarray:
        """[T, capacity, H] view of the bank without the padding columns."""
        return self.bank[:, :, : self.H]

    def copy(self) -> "Workload":
        return Workload(
            self.name, self.T, self.num_blocks, self.capacity, self.has_delta,
            self.has_out_norm, self.block_write_idx, self.prefix.copy(),
            None if self.delta is None else self.delta.copy(), self.bank.copy(),
            self.rms_w.copy(), self.res_w.copy(),
            None if self.out_norm_w is None else self.out_norm_w.copy(),
            self.eps, self.out_eps, self.H, dict(self.meta), self.group)

    def algorithmic_bytes(self) -> int:
        """Bytes the mixture must move once: source rows read, delta read,
        out / prefix / bank write-backs written, weights read once."""
        R = self.H * 2
        d = 1 if self.has_delta else 0
        w = 1 if self.block_write_idx >= 0 else 0
        o = 1 if self.has_out_norm else 0
        bank_rows = -(-self.T // self.group)
        return (self.T * R * (1 + d + 1 + d) + bank_rows * R * (self.num_blocks + w)
                + R * (2 + o))


def _activations(rng: np.random.Generator, shape: Tuple[int, ...],
                 outliers: bool) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if outliers:
        mask = rng.random(shape, dtype=np.float32) < 0.01
        x[mask] *= np.float32(50.0)
    return x


def make_workload(T: int, num_blocks: int, *, capacity: int = 8,
                  has_delta: bool = True, has_out_norm: bool = True,
                  block_write_idx: int = -1, seed: int = 0, H: int = HIDDEN,
                  slot_stride: Optional[int] = None, outliers: bool = False,
                  slot_scale: Optional[Tuple[float, float]] = None,
                  mixing: bool = False, eps: float = 1e-6,
                  out_eps: float = 1e-6, name: str = "",
                  token_chunk: int = 256, group: int = 1) -> Workload:
    """Draw one workload.  Every tensor has its own child seed, so changing
    one option does not reshuffle the others."""
    if slot_stride is None:
        slot_stride = H
    ss = np.random.SeedSequence(seed)
    (s_prefix, s_delta, s_bank, s_w, s_scale) = ss.spawn(5)

    rng_w = np.random.default_rng(s_w)
    rms_w = f32_to_bf16_bits(1.0 + 0.1 * rng_w.standard_normal(H, dtype=np.float32))
    if mixing:
        res_w = f32_to_bf16_bits(0.02 * rng_w.standard_normal(H, dtype=np.float32))
    else:
        res_w = f32_to_bf16_bits(1.0 + 0.1 * rng_w.standard_normal(H, dtype=np.float32))
    onw = f32_to_bf16_bits(1.0 + 0.1 * rng_w.standard_normal(H, dtype=np.float32))

    scales = np.ones(capacity, dtype=np.float32)
    if slot_scale is not None:
        lo, hi = slot_scale
        scales = np.random.default_rng(s_scale).uniform(lo, hi, capacity).astype(np.float32)

    rng_p = np.random.default_rng(s_prefix)
    rng_d = np.random.default_rng(s_delta)
    rng_b = np.random.default_rng(s_bank)
    prefix = np.empty((T, H), dtype=np.uint16)
    delta = np.empty((T, H), dtype=np.uint16) if has_delta else None
    TB = -(-T // group)  # bank rows
    bank = np.full((TB, capacity, slot_stride), CANARY, dtype=np.uint16)
    for t0 in range(0, T, token_chunk):
        t1 = min(T, t0 + token_chunk)
        prefix[t0:t1] = f32_to_bf16_bits(_activations(rng_p, (t1 - t0, H), outliers))
        if has_delta:
            delta[t0:t1] = f32_to_bf16_bits(_activations(rng_d, (t1 - t0, H), outliers))
    for t0 in range(0, TB, token_chunk):
        t1 = min(TB, t0 + token_chunk)
        if num_blocks > 0:
            x = _activations(rng_b, (t1 - t0, num_blocks, H), outliers)
            x *= scales[None, :num_blocks, None]
            bank[t0:t1, :num_blocks, :H] = f32_to_bf16_bits(x)
    return Workload(name or f"T{T}_S{num_blocks}", T, num_blocks, capacity,
                    has_delta, has_out_norm, block_write_idx, prefix, delta,
                    bank, rms_w, res_w, onw if has_out_norm else None, eps,
                    out_eps, H, dict(seed=seed, outliers=outliers,
                                     slot_scale=slot_scale, mixing=mixing), group)


# ---- the named workloads -------------------------------------------------

def single_token(seed: int = 0) -> Workload:
    """T=1, 4 valid blocks in an 8-slot bank, delta and output norm on,
    no write-back."""
    return make_workload(1, 4, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=-1, seed=seed, name="single_token_T1_S4")


def variant_cell(T: int, S: int, has_delta: bool, has_out_norm: bool,
                 block_write_idx: int, seed: int = 0, capacity: int = 8,
                 mixing: bool = False) -> Workload:
    """One cell of the spec-decode variant matrix, T in {1,4,8}."""
    return make_workload(T, S, capacity=capacity, has_delta=has_delta,
                         has_out_norm=has_out_norm,
                         block_write_idx=block_write_idx, seed=seed,
                         mixing=mixing,
                         name=f"variant_T{T}_S{S}_d{int(has_delta)}_o{int(has_out_norm)}_w{block_write_idx}")


def decode_batch(T: int, seed: int = 0) -> Workload:
    """T in {64, 256}, 8 blocks, delta and output norm on, bank slots scaled
    per block by U(0.5, 20)."""
    return make_workload(T, 8, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=-1, seed=seed, slot_scale=(0.5, 20.0),
                         name=f"decode_T{T}_S8")


def prefill(T: int, S: int, has_out_norm: bool, block_write_idx: int,
            seed: int = 0) -> Workload:
    """T in {1024, 2048}, S in {0,4,8}, delta on, 1% outliers x50."""
    return make_workload(T, S, capacity=8, has_delta=True,
                         has_out_norm=has_out_norm,
                         block_write_idx=block_write_idx, seed=seed,
                         outliers=True,
                         name=f"prefill_T{T}_S{S}_o{int(has_out_norm)}_w{block_write_idx}")


def long_prefill(T: int = 8192, seed: int = 0) -> Workload:
    """T=8192, 8 blocks in a 9-slot bank with padded slot stride 7232,
    delta and output norm on, write-back into slot 8, per-block scales
    U(1, 30)."""
    return make_workload(T, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=seed, slot_stride=7232,
                         slot_scale=(1.0, 30.0), name=f"long_prefill_T{T}_S8_w8")
