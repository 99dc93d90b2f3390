"""Element offsets past 2^31 (byte offsets past 2^32): every kernel form on
token rows that lie far apart in large device allocations.

The row, slot and token strides below place token row t at t x stride
elements, so the last rows start beyond 2^31 elements from the base of
their buffers: any offset formed in 32 bits would wrap there.  Each
allocation is 4.5-5.7 GB (about 21 GB in all); only the rows and a
64-column canary after each row are ever written.  Same bar as the other
parity tests: out within max(2 bf16 ulp, 1e-2), the updated prefix and
every bank slot bit-exact, delta unchanged, canaries untouched."""
import numpy as np
import pytest

import attention_residual_fusion_gb300 as ar
import oracle
from attention_residual_fusion_gb300 import _build
from attention_residual_fusion_gb300 import tp
from attention_residual_fusion_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

NT = oracle.default_threads()
T = 300                    # more tokens than the persistent kernels' clusters
CAP = 9                    # bank slots; slot 8 is the write-back slot
SLOT = (1 << 20) + 64      # elements between the slots of a token's bank row
BTOK = CAP * SLOT + 8      # elements between the tokens' bank rows
ROW = (1 << 23) + 72       # elements between rows of prefix, delta and out
PAD = 64                   # canary columns after every row
assert (T - 1) * BTOK > 2 ** 31 and (T - 1) * ROW > 2 ** 31


def _dev(a: np.ndarray, torch):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _host(t) -> np.ndarray:
    import torch

    # gather the strided rows on the device first: a copy of the view, not
    # of the whole allocation behind it
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def big():
    import torch

    _build.build()
    ar.lib()
    bufs = {"bank": torch.empty(T * BTOK, dtype=torch.bfloat16, device="cuda")}
    for k in ("prefix", "delta", "out"):
        bufs[k] = torch.empty(T * ROW, dtype=torch.bfloat16, device="cuda")
    yield bufs
    del bufs
    torch.cuda.empty_cache()


class Views:
    """Strided views of the large buffers for one workload of width H, its
    data copied in and canaries after every row."""

    def __init__(self, big, wl, torch):
        H = wl.H
        st = torch.as_strided
        self.prefix = st(big["prefix"], (T, H), (ROW, 1))
        self.delta = st(big["delta"], (T, H), (ROW, 1))
        self.out = st(big["out"], (T, H), (ROW, 1))
        self.bank = st(big["bank"], (T, CAP, H), (BTOK, SLOT, 1))
        self.pads = [st(big[k], (T, PAD), (ROW, 1), H) for k in ("prefix", "delta", "out")]
        self.pads.append(st(big["bank"], (T, CAP, PAD), (BTOK, SLOT, 1), H))
        self.prefix.copy_(_dev(wl.prefix, torch))
        self.delta.copy_(_dev(wl.delta, torch))
        self.bank.copy_(_dev(wl.bank[:, :, :H], torch))
        self.out.fill_(0.0)
        for p in self.pads:
            p.view(torch.int16).fill_(W.CANARY)  # the bit pattern, a NaN
        self.res, self.rms, self.onw = (_dev(x, torch) for x in (wl.res_w, wl.rms_w, wl.out_norm_w))

    def check(self, wl, ref, tag):
        import torch

        torch.cuda.synchronize()
        G.assert_out_close(_host(self.out), ref["out"], tag)
        assert np.array_equal(_host(self.prefix), ref["prefix"][:, :wl.H]), f"{tag}: prefix"
        assert np.array_equal(_host(self.bank), ref["bank"][:, :, :wl.H]), f"{tag}: bank"
        assert np.array_equal(_host(self.delta), wl.delta), f"{tag}: delta changed"
        for p in self.pads:
            assert np.all(_host(p) == W.CANARY), f"{tag}: a canary column was written"


# (kernel, bank rows, width): every form the kernel is built for
CASES = [(ar.KERNEL_SPLIT, 8, 7168), (ar.KERNEL_STREAM, 8, 7168), (ar.KERNEL_STAGED, 4, 7168),
         (ar.KERNEL_ROW, 2, 7168), (ar.KERNEL_ROW_SMEM, 8, 7168), (ar.KERNEL_GENERIC, 8, 7168),
         (0, 8, 4096), (ar.KERNEL_SPLIT, 8, 4096), (0, 8, 3000), (ar.KERNEL_GENERIC, 8, 3000)]


@pytest.mark.parametrize("kernel,S,H", CASES, ids=[f"k{k}_S{S}_H{H}" for k, S, H in CASES])
def test_offsets_past_2_31(big, kernel, S, H):
    import torch

    wl = W.make_workload(T, S, capacity=CAP, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=900 + S + H, mixing=True, H=H)
    ref = oracle.run_workload(wl, n_threads=NT)
    v = Views(big, wl, torch)
    out = ar.attn_res(v.prefix, v.delta, v.bank, S, 8, v.res, v.rms, v.onw, wl.eps, wl.out_eps,
                      v.out, kernel=kernel)
    assert out.data_ptr() == v.out.data_ptr()
    v.check(wl, ref, f"k{kernel}_S{S}_H{H}")


# the hidden-sharded kernels on one rank (the shard is the whole row):
# the persistent ring (forced) and one CTA per row, both forms of the sums
TP = [(ar.KERNEL_STREAM, False), (ar.KERNEL_STREAM, True), (ar.KERNEL_GENERIC, False),
      (ar.KERNEL_GENERIC, True)]


@pytest.mark.parametrize("kernel,gram", TP, ids=[f"k{k}_gram{int(g)}" for k, g in TP])
def test_sharded_offsets_past_2_31(big, kernel, gram):
    import torch

    H = 1024
    wl = W.make_workload(T, 8, capacity=CAP, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=950 + int(gram), mixing=True, H=H)
    ref = oracle.run_workload(wl, n_threads=NT)
    v = Views(big, wl, torch)
    tp.attn_res_tp(v.prefix, v.delta, v.bank, 8, 8, v.res, v.rms, v.onw, wl.eps, wl.out_eps,
                   v.out, H=H, all_reduce=lambda t: None, gram=gram, kernel=kernel)
    v.check(wl, ref, f"tp_k{kernel}_gram{int(gram)}")
