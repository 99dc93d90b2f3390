"""A CUDA graph captured around the very first call of a process: each kernel
form's one-time launch set-up (shared-memory attribute, occupancy query)
then runs inside the capture.  Each form runs in a fresh interpreter; the
replayed graph's outputs must equal, bit for bit, those of an ordinary call
on a copy of the same inputs made after it."""
import os
import subprocess
import sys

import pytest

import attention_residual_fusion_gb300 as ar
from attention_residual_fusion_gb300 import _build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np, torch
import attention_residual_fusion_gb300 as ar
from attention_residual_fusion_gb300 import tp, workloads as W
kernel, T, S, H, sharded = (int(a) for a in sys.argv[1:6])
wl = W.make_workload(T, S, capacity=9, has_delta=True, has_out_norm=True, block_write_idx=8,
                     seed=77, mixing=True, H=H)
up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
def fresh():
    return dict(prefix=up(wl.prefix), delta=up(wl.delta), bank=up(wl.bank), res=up(wl.res_w),
                rms=up(wl.rms_w), onw=up(wl.out_norm_w),
                out=torch.empty((T, H), dtype=torch.bfloat16, device="cuda"))
def call(d, s):
    if sharded:
        tp.attn_res_tp(d["prefix"], d["delta"], d["bank"], S, 8, d["res"], d["rms"], d["onw"],
                       wl.eps, wl.out_eps, d["out"], H=H, all_reduce=lambda t: None,
                       gram=bool(sharded - 1), kernel=kernel, stream=s)
    else:
        ar.attn_res(d["prefix"], d["delta"], d["bank"], S, 8, d["res"], d["rms"], d["onw"],
                    wl.eps, wl.out_eps, d["out"], kernel=kernel, stream=s)
s = torch.cuda.Stream()
g_in = fresh()
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    call(g_in, s)
g.replay()
torch.cuda.synchronize()
e_in = fresh()
call(e_in, torch.cuda.current_stream())
torch.cuda.synchronize()
for k in ("out", "prefix", "bank"):
    assert torch.equal(g_in[k].view(torch.int16), e_in[k].view(torch.int16)), k
assert ar.device_status() == 0
print("ok")
"""

# (kernel, T, S, H, sharded: 0 = attn_res, 1 = hidden-sharded two exchanges,
# 2 = hidden-sharded Gram)
FORMS = [(0, 1, 4, 7168, 0), (ar.KERNEL_STREAM, 600, 8, 7168, 0), (ar.KERNEL_STAGED, 300, 4, 7168, 0),
         (ar.KERNEL_ROW, 300, 1, 7168, 0), (ar.KERNEL_ROW_SMEM, 200, 8, 7168, 0),
         (ar.KERNEL_GENERIC, 20, 8, 7168, 0), (0, 400, 8, 3000, 0),
         (ar.KERNEL_STREAM, 300, 8, 1024, 1), (ar.KERNEL_STREAM, 300, 8, 1024, 2),
         (ar.KERNEL_GENERIC, 300, 8, 1024, 2)]


@pytest.mark.parametrize("kernel,T,S,H,sharded", FORMS,
                         ids=[f"k{k}_T{T}_S{S}_H{H}_tp{p}" for k, T, S, H, p in FORMS])
def test_first_call_inside_graph_capture(kernel, T, S, H, sharded):
    _build.build()
    r = subprocess.run([sys.executable, "-c", CHILD, str(kernel), str(T), str(S), str(H),
                        str(sharded)], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-3000:]
