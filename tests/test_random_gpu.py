"""Seeded random configurations against the oracle.

Each case draws a hidden size (7168, another multiple of 1024, or any
multiple of 8: the any-width forms take every width up to 16384), a token count, num_blocks, the bank capacity and its padded
slot stride, delta / output norm / write-back, shared bank rows, PDL, and a
kernel (automatic or forced where the width and bank rows allow it: split,
stream, staged, row and shared-memory row kernels at H = 7168), then checks the CUDA
path against the oracle with the bar of the other parity tests: out within
max(2 bf16 ulp, 1e-2), the updated prefix and every byte of the bank
bit-exact, guard zones untouched."""
import numpy as np
import pytest

import attention_residual_fusion_gb300 as ar
import oracle
from attention_residual_fusion_gb300 import _build
from attention_residual_fusion_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

NT = oracle.default_threads()
CASES = 160


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    ar.lib()


def draw(k: int):
    rng = np.random.default_rng(10_000 + k)
    H = int(rng.choice([7168, 7168, 7168, 1024 * int(rng.integers(1, 17)),
                        8 * int(rng.integers(1, 600))]))
    T = int(rng.choice([1, 2, 3, 5, 8, 17, 64, 79, 80, 81, 130, 257, 600]))
    S = int(rng.integers(0, 9))
    cap = S + int(rng.integers(0, 3)) if S < 8 else 8 + int(rng.integers(0, 2))
    cap = max(cap, 1)
    has_delta = bool(rng.integers(0, 2))
    has_norm = bool(rng.integers(0, 2))
    group = int(rng.choice([1, 1, 1, 2, 3]))
    slots_free = [i for i in range(S, cap)]          # slots that are not sources
    choices = [-1] + slots_free + ([] if group > 1 else list(range(S)))
    widx = int(rng.choice(choices))
    pad = int(rng.choice([0, 0, 8, 64]))
    pdl = bool(rng.integers(0, 2))
    kernels = [0]
    if H == 7168:
        kernels += [ar.KERNEL_SPLIT, ar.KERNEL_STREAM, ar.KERNEL_GENERIC]
        if S <= 2:
            kernels += [ar.KERNEL_ROW]
        if S >= 1:
            kernels += [ar.KERNEL_ROW_SMEM]
        if group == 1 and S <= 5:
            kernels += [ar.KERNEL_STAGED]
    elif H <= 16384 and (S > 0 or has_norm):
        kernels += [ar.KERNEL_STREAM, ar.KERNEL_GENERIC]
        if H <= 8192:
            kernels += [ar.KERNEL_SPLIT]
    else:
        kernels += [ar.KERNEL_GENERIC]
    kernel = int(rng.choice(kernels))
    if kernel in (ar.KERNEL_STREAM, ar.KERNEL_STAGED) and H == 7168 and S == 0 and not has_norm:
        kernel = 0                                   # no exchange: not a stream case
    return dict(H=H, T=T, S=S, cap=cap, has_delta=has_delta, has_norm=has_norm, group=group,
                widx=widx, pad=pad, pdl=pdl, kernel=kernel, seed=20_000 + k)


@pytest.mark.parametrize("k", range(CASES))
def test_random_configuration(k):
    c = draw(k)
    wl = W.make_workload(c["T"], c["S"], capacity=c["cap"], has_delta=c["has_delta"],
                         has_out_norm=c["has_norm"], block_write_idx=c["widx"],
                         seed=c["seed"], H=c["H"], mixing=True,
                         slot_stride=c["H"] + c["pad"], group=c["group"],
                         outliers=bool(k % 2))
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = G.run_gpu(wl, kernel=c["kernel"], pdl=c["pdl"])
    G.check_against_oracle(wl, gpu, ref, tag=str(c))
