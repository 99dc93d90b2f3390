"""Calls in flight at the same time: several kernel forms on several CUDA
streams at once, and calls made from several host threads at once.  The
library keeps no per-call state (only launch-configuration caches and the
device status word), so every call must match the oracle exactly as when it
runs alone: out within max(2 bf16 ulp, 1e-2), prefix and bank bit-exact."""
import threading

import numpy as np
import pytest

import attention_residual_fusion_gb300 as ar
import oracle
from attention_residual_fusion_gb300 import _build
from attention_residual_fusion_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

NT = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    ar.lib()


# (kernel, T, S, H): the split, stream, staged, row, shared-memory row and
# general forms, and an any-width stream
FORMS = [(ar.KERNEL_SPLIT, 5, 8, 7168), (ar.KERNEL_STREAM, 600, 8, 7168),
         (ar.KERNEL_STAGED, 300, 4, 7168), (ar.KERNEL_ROW, 300, 0, 7168),
         (ar.KERNEL_ROW_SMEM, 200, 6, 7168), (ar.KERNEL_GENERIC, 40, 8, 7168), (0, 400, 8, 4096)]


def _case(i, kernel, T, S, H):
    wl = W.make_workload(T, S, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=500 + i, mixing=True, H=H)
    return wl, oracle.run_workload(wl, n_threads=NT)


def _device(wl, torch):
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return dict(prefix=up(wl.prefix), delta=up(wl.delta), bank=up(wl.bank), res=up(wl.res_w),
                rms=up(wl.rms_w), onw=up(wl.out_norm_w),
                out=torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda"))


def _host(t):
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _call(wl, d, kernel, stream):
    ar.attn_res(d["prefix"], d["delta"], d["bank"][:, :, :wl.H], wl.num_blocks, wl.block_write_idx,
                d["res"], d["rms"], d["onw"], wl.eps, wl.out_eps, d["out"], kernel=kernel,
                stream=stream)


def _check(wl, ref, d, tag):
    G.assert_out_close(_host(d["out"]), ref["out"], tag)
    assert np.array_equal(_host(d["prefix"]), ref["prefix"][:, :wl.H]), f"{tag}: prefix"
    assert np.array_equal(_host(d["bank"]), ref["bank"]), f"{tag}: bank"


def test_kernel_forms_on_concurrent_streams():
    """Every form launched on its own stream, all in flight together, three
    rounds on fresh copies of the inputs."""
    import torch

    cases = [(_case(i, *f), f[0]) for i, f in enumerate(FORMS)]
    streams = [torch.cuda.Stream() for _ in cases]
    for rnd in range(3):
        devs = [_device(wl, torch) for (wl, _), _ in cases]
        torch.cuda.synchronize()
        for ((wl, _), kernel), d, s in zip(cases, devs, streams):
            _call(wl, d, kernel, s)
        torch.cuda.synchronize()
        for ((wl, ref), kernel), d in zip(cases, devs):
            _check(wl, ref, d, f"round {rnd} kernel {kernel} T {wl.T}")
    assert ar.device_status() == 0


def test_calls_from_concurrent_host_threads():
    """Four host threads, each with its own stream and buffers, each making
    ten calls (fresh inputs before every call) while the others do."""
    import torch

    cases = [(_case(10 + i, *f), f[0]) for i, f in enumerate(FORMS[:4])]
    errors = []

    def worker(case, kernel):
        wl, ref = case
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for n in range(10):
                    d = _device(wl, torch)
                    _call(wl, d, kernel, s)
                    s.synchronize()
                    _check(wl, ref, d, f"thread kernel {kernel} call {n}")
        except Exception as e:  # reported on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=c) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert ar.device_status() == 0
