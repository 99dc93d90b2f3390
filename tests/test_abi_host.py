"""The C ABI on the host: the library loads, exports every declared symbol and
rejects bad arguments before touching the device (no GPU needed)."""
import os
import re

import pytest

import attention_residual_fusion_gb300 as ar
from attention_residual_fusion_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_res.h")
H = 7168


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ar.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_res\w*)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "attn_res" in names and len(names) >= 5
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ar.EXPORTS)


def test_constants(lib):
    assert lib.attn_res_hidden_size() == H
    assert lib.attn_res_max_blocks() == 8
    for s in range(6):
        assert ar.status_string(s)
    assert ar.status_string(99) == "unknown status"


def test_launch_shape(lib):
    ls = ar.launch_shape
    assert ls(1, 4, True) == dict(kernel="split", split=7, stages=0, threads=128, ctas=7, cluster=7)
    assert ls(64, 8, False) == dict(kernel="split", split=7, stages=0, threads=128, ctas=448, cluster=7)
    assert ls(8192, 8, True) == dict(kernel="stream", split=7, stages=2, threads=32, ctas=0, cluster=7)
    assert ls(8192, 4, False) == dict(kernel="stream", split=7, stages=2, threads=64, ctas=0, cluster=7)
    assert ls(8192, 0, True)["threads"] == 32
    # no softmax and no output norm: the CTAs of a token never talk
    assert ls(1024, 0, False) == dict(kernel="split", split=7, stages=0, threads=128, ctas=7168, cluster=1)
    assert ls(2, 8, True, ar.FLAG_SPLIT(16)) == dict(kernel="split", split=16, stages=0, threads=64, ctas=32, cluster=16)
    assert ls(2, 8, True, ar.FLAG_SPLIT(4))["threads"] == 224
    assert ls(2, 8, True, ar.FLAG_SPLIT(14))["threads"] == 64
    assert ls(2, 8, True, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(4) | ar.FLAG_VPT(2) | ar.FLAG_STAGES(3))["stages"] == 3
    assert ls(9000, 8, True, ar.FLAG_KERNEL(1))["kernel"] == "split"
    assert ls(10, 8, True, ar.FLAG_KERNEL(3)) == dict(kernel="generic", split=1, stages=0, threads=256, ctas=10, cluster=1)
    assert ls(9000, 8, True, ar.FLAG_SPLIT(7) | ar.FLAG_VPT(2))["threads"] == 64
    assert ls(9000, 8, True, ar.FLAG_SPLIT(7) | ar.FLAG_VPT(1))["threads"] == 128
    for bad in [(-1, 0, 0, 0), (1, 9, 0, 0), (1, -1, 0, 0), (1, 1, 0, ar.FLAG_SPLIT(5)),
                (1, 1, 0, ar.FLAG_KERNEL(4)), (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(16)),
                (1, 1, 0, ar.FLAG_KERNEL(3) | ar.FLAG_SPLIT(7)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_STAGES(4)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(8) | ar.FLAG_VPT(2)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_STAGES(4)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(7) | ar.FLAG_VPT(1) | ar.FLAG_STAGES(3)),
                (1, 1, 0, ar.FLAG_KERNEL(1) | ar.FLAG_VPT(2)),
                (1, 1, 0, ar.FLAG_KERNEL(1) | ar.FLAG_STAGES(2)), (1, 1, 0, 1 << 30)]:
        with pytest.raises(ar.AttnResError):
            ls(*bad)


# Fake, well separated, 16-byte aligned device addresses: validation happens
# before any CUDA call, so these are never dereferenced.
BASE = 1 << 40
GAP = 1 << 34


def addr(i, off=0):
    return BASE + i * GAP + off


def good(T=4, S=4, cap=8, widx=-1, delta=True, onorm=True):
    lay = ar.Layout(prefix_row=H, delta_row=H, blocks_token=cap * H, blocks_slot=H,
                    out_row=H, blocks_capacity=cap, flags=0)
    args = dict(prefix=addr(0), delta=addr(1) if delta else 0, blocks=addr(2),
                num_blocks=S, block_write_idx=widx, res_w=addr(3), rms_w=addr(4),
                out_norm_w=addr(5) if onorm else 0, eps=1e-6, out_eps=1e-6,
                out=addr(6), T=T, layout=lay, stream=0)
    return args


def call(**kw):
    return ar.call_raw(**kw)


def test_valid_arguments_reach_the_device_check(lib):
    # without a CUDA device the first CUDA call fails: EDEVICE (or ECUDA)
    st = call(**good())
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert st in (5, 4)


def test_zero_tokens_is_a_no_op(lib):
    assert call(**good(T=0)) == 0


@pytest.mark.parametrize("change,status", [
    (dict(T=-1), 1),
    (dict(num_blocks=9), 1),
    (dict(num_blocks=-1), 1),
    (dict(block_write_idx=8), 1),       # == capacity
    (dict(block_write_idx=-2), 1),
    (dict(prefix=0), 1),
    (dict(res_w=0), 1),
    (dict(rms_w=0), 1),
    (dict(out=0), 1),
    (dict(blocks=0), 1),                # num_blocks > 0 needs the bank
    (dict(eps=-1.0), 1),
    (dict(eps=float("nan")), 1),
    (dict(out_eps=float("inf")), 1),
    (dict(prefix=addr(0, 8)), 2),
    (dict(delta=addr(1, 2)), 2),
    (dict(blocks=addr(2, 4)), 2),
    (dict(res_w=addr(3, 8)), 2),
    (dict(out_norm_w=addr(5, 2)), 2),
    (dict(out=addr(6, 8)), 2),
    (dict(out=addr(0, 16)), 3),         # out overlaps prefix
    (dict(out=addr(2, 4096 * 2)), 3),   # out inside the bank
    (dict(res_w=addr(6, 1024)), 3),     # a weight inside out
    (dict(delta=addr(0, 4 * 7168 * 2 - 16)), 3),  # delta overlaps the written prefix
])
def test_rejections(lib, change, status):
    kw = good()
    kw.update(change)
    assert call(**kw) == status


def test_num_blocks_above_capacity(lib):
    kw = good(S=4, cap=3)
    assert call(**kw) == 1


def test_append_slot_equal_to_capacity_is_rejected(lib):
    # the 8-slot bank with 8 valid blocks has no slot 8 to append into
    kw = good(S=8, cap=8, widx=8)
    assert call(**kw) == 1


@pytest.mark.parametrize("field,value,status", [
    ("prefix_row", H - 8, 1), ("out_row", 100, 1), ("delta_row", 0, 1),
    ("blocks_slot", H - 8, 1), ("blocks_token", 7 * H, 1),
    ("prefix_row", H + 4, 2), ("blocks_slot", 7232 + 4, 2), ("out_row", H + 1, 2),
    ("blocks_capacity", -1, 1), ("flags", 0x4, 1), ("flags", ar.FLAG_SPLIT(5), 1),
    ("flags", ar.FLAG_KERNEL(7), 1), ("flags", ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(16), 1),
])
def test_layout_rejections(lib, field, value, status):
    kw = good()
    setattr(kw["layout"], field, value)
    if field == "blocks_slot" and value > H:
        kw["layout"].blocks_token = 16 * 7232  # room for the wider slots
    assert call(**kw) == status


def test_optional_pointers(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    kw = good(S=0, widx=-1, delta=False, onorm=False)
    kw["blocks"] = 0
    kw["layout"].blocks_capacity = 0
    assert call(**kw) in (5, 4)  # valid: reaches the device check
    kw["block_write_idx"] = 0
    assert call(**kw) == 1      # a write-back needs a slot


def good_h(H, T=4, S=4, cap=8):
    kw = good(T=T, S=S, cap=cap)
    lay = kw["layout"]
    lay.prefix_row = lay.delta_row = lay.out_row = lay.blocks_slot = H
    lay.blocks_token = cap * H
    return kw


@pytest.mark.parametrize("H,status", [(0, 1), (-8, 1), (4, 1), (12, 1), (7170, 1)])
def test_other_widths_rejected(lib, H, status):
    assert ar.call_raw(**good_h(max(H, 8)), H=H) == status


def test_other_widths_validate_strides(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    kw = good_h(64)
    assert ar.call_raw(**kw, H=64) in (4, 5)        # valid: reaches the device check
    kw["layout"].prefix_row = 56
    assert ar.call_raw(**kw, H=64) == 1             # stride below H
    kw = good_h(64)
    kw["layout"].flags = ar.FLAG_KERNEL(2)
    assert ar.call_raw(**kw, H=64) == 1             # only the general kernel takes other widths
