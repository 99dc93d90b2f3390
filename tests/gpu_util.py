"""Helpers for the GPU parity tests: guarded device copies of a workload, a
call through the C ABI, and the comparison with the oracle."""
from __future__ import annotations

import numpy as np

import attention_residual_fusion_gb300 as ar
from attention_residual_fusion_gb300 import workloads as W
from tests import restatement as R

GUARD = 4096          # guard elements on each side of every buffer
GUARD_BITS = 0x7FB3   # a NaN pattern, distinct from the bank canary


class Guarded:
    """A device copy of a host uint16 array inside a larger buffer whose
    guard zones must come back untouched."""

    def __init__(self, host: np.ndarray, torch):
        self.shape = host.shape
        flat = np.full(host.size + 2 * GUARD, GUARD_BITS, dtype=np.uint16)
        flat[GUARD:GUARD + host.size] = host.reshape(-1)
        self.dev = torch.from_numpy(flat.view(np.int16)).cuda()
        self.view = self.dev[GUARD:GUARD + host.size].view(torch.bfloat16).view(*host.shape)

    def host(self) -> np.ndarray:
        return self.dev.cpu().numpy().view(np.uint16)[GUARD:-GUARD].reshape(self.shape)

    def guards_intact(self) -> bool:
        a = self.dev.cpu().numpy().view(np.uint16)
        return bool(np.all(a[:GUARD] == GUARD_BITS) and np.all(a[-GUARD:] == GUARD_BITS))


def run_gpu(wl: W.Workload, *, split: int = 0, pdl: bool = False, kernel: int = 0,
            stages: int = 0, vpt: int = 0, prefix_row: int | None = None, out_row: int | None = None):
    """Copy the workload to the device (guarded), call attn_res through the C
    ABI, and return host copies of out, prefix and the bank."""
    import torch

    H = wl.H
    pr = prefix_row or H
    orow = out_row or H
    prefix_h = np.full((wl.T, pr), W.CANARY, dtype=np.uint16)
    prefix_h[:, :H] = wl.prefix
    g_prefix = Guarded(prefix_h, torch)
    g_delta = Guarded(wl.delta, torch) if wl.delta is not None else None
    g_bank = Guarded(wl.bank, torch)
    g_rms = Guarded(wl.rms_w, torch)
    g_res = Guarded(wl.res_w, torch)
    g_onw = Guarded(wl.out_norm_w, torch) if wl.out_norm_w is not None else None
    g_out = Guarded(np.full((wl.T, orow), W.CANARY, dtype=np.uint16), torch)
    out = ar.attn_res(g_prefix.view[:, :H], None if g_delta is None else g_delta.view,
                      g_bank.view[:, :, :H], wl.num_blocks, wl.block_write_idx,
                      g_res.view, g_rms.view, None if g_onw is None else g_onw.view,
                      wl.eps, wl.out_eps, g_out.view[:, :H], pdl=pdl, split=split,
                      kernel=kernel, stages=stages, vpt=vpt, blocks_group=wl.group)
    torch.cuda.synchronize()
    bufs = [g for g in (g_prefix, g_delta, g_bank, g_rms, g_res, g_onw, g_out) if g is not None]
    assert all(g.guards_intact() for g in bufs), "a guard zone was written"
    assert out.data_ptr() == g_out.view.data_ptr()
    res = dict(out_full=g_out.host(), prefix_full=g_prefix.host(), bank=g_bank.host())
    res["out"] = res["out_full"][:, :H]
    res["prefix"] = res["prefix_full"][:, :H]
    # inputs must come back unchanged
    if g_delta is not None:
        assert np.array_equal(g_delta.host(), wl.delta)
    assert np.array_equal(g_rms.host(), wl.rms_w) and np.array_equal(g_res.host(), wl.res_w)
    return res


def tolerance(ref_bits: np.ndarray) -> np.ndarray:
    """Per element: 2 bf16 ulp of the oracle's value, at least 1e-2."""
    r = R.widen(ref_bits)
    return np.maximum(2.0 * R.ulp_bf16(r), 1e-2)


def assert_out_close(gpu_bits: np.ndarray, ref_bits: np.ndarray, tag=""):
    g = R.widen(gpu_bits)
    r = R.widen(ref_bits)
    assert np.all(np.isfinite(g)), f"{tag}: non-finite output"
    err = np.abs(g - r)
    tol = tolerance(ref_bits)
    bad = err > tol
    if np.any(bad):
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(
            f"{tag}: {int(bad.sum())} elements outside tolerance; worst at {i}: "
            f"gpu {g[i]!r} oracle {r[i]!r} tol {tol[i]!r}")


def check_against_oracle(wl: W.Workload, gpu: dict, ref: dict, tokens=None, tag=""):
    """out within tolerance; updated prefix and the whole bank (every slot and
    padding column) bit-exact; padding of prefix/out rows untouched."""
    idx = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    assert_out_close(gpu["out"][idx], ref["out"], tag)
    assert np.array_equal(gpu["prefix"][idx], ref["prefix"][:, :wl.H]), f"{tag}: prefix"
    bank = gpu["bank"] if wl.group > 1 else gpu["bank"][idx]
    assert np.array_equal(bank, ref["bank"]), f"{tag}: bank"
    if gpu["prefix_full"].shape[1] > wl.H:
        assert np.all(gpu["prefix_full"][:, wl.H:] == W.CANARY), f"{tag}: prefix padding"
    if gpu["out_full"].shape[1] > wl.H:
        assert np.all(gpu["out_full"][:, wl.H:] == W.CANARY), f"{tag}: out padding"
