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
    assert ls(8192, 8, True) == dict(kernel="stream", split=7, stages=2, threads=64, ctas=0, cluster=7)
    # 4 bank rows, output norm, many tokens: the staged form (7,4) at 7 CTAs
    # per SM, two stages of 6 row slices with delta, three of 5 without
    assert ls(8192, 4, True) == dict(kernel="staged", split=7, stages=2, threads=32, ctas=0, cluster=7)
    assert ls(8192, 4, True, has_delta=False)["stages"] == 3
    assert ls(256, 4, True) == dict(kernel="row_smem", split=1, stages=0, threads=128, ctas=256, cluster=1)
    assert ls(256, 4, True, ar.FLAG_KERNEL(2)) == dict(kernel="stream", split=7, stages=2, threads=32, ctas=0, cluster=7)
    assert ls(8192, 4, False) == dict(kernel="stream", split=7, stages=2, threads=32, ctas=0, cluster=7)
    assert ls(256, 4, False)["kernel"] == "row_smem" and ls(256, 7, False)["threads"] == 64
    assert ls(256, 6, True)["kernel"] == "row_smem" and ls(1024, 6, True)["threads"] == 32
    assert ls(2048, 3, True)["kernel"] == "staged" and ls(2048, 5, True)["kernel"] == "staged"
    assert ls(256, 3, False) == dict(kernel="staged", split=4, stages=2, threads=64, ctas=0, cluster=4)
    assert ls(2048, 6, True)["kernel"] == "stream"
    # up to two bank rows: the row kernel, one CTA of 896 / VPT threads per row
    assert ls(8192, 0, True) == dict(kernel="row", split=1, stages=0, threads=128, ctas=8192, cluster=1)
    assert ls(256, 0, True)["threads"] == 224 and ls(256, 1, False)["threads"] == 224
    assert ls(2048, 1, True)["kernel"] == "row_smem" and ls(2048, 2, True)["kernel"] == "row"
    assert ls(4096, 2, True)["kernel"] == "row_smem" and ls(2048, 2, True)["threads"] == 128
    assert ls(2048, 2, False)["kernel"] == "stream" and ls(256, 0, False)["kernel"] == "split"
    assert ls(300, 2, True, ar.FLAG_KERNEL(5) | ar.FLAG_VPT(4))["threads"] == 224
    # shape overrides without a kernel keep the split / stream families
    assert ls(8192, 0, True, ar.FLAG_STAGES(2))["kernel"] == "stream"
    assert ls(8192, 0, True, ar.FLAG_VPT(4)) == dict(kernel="stream", split=2, stages=2, threads=128, ctas=0, cluster=2)
    assert ls(8192, 4, True, ar.FLAG_SPLIT(2))["threads"] == 128      # (2,4,2) with bank rows
    assert ls(8192, 0, True, ar.FLAG_VPT(2))["split"] == 4
    assert ls(8192, 0, True, ar.FLAG_VPT(1))["split"] == 7
    assert ls(8192, 0, True, ar.FLAG_VPT(2) | ar.FLAG_STAGES(3))["split"] == 4
    with pytest.raises(ar.AttnResError):
        ls(8192, 0, True, ar.FLAG_STAGES(3))          # (2,4,3) is not built
    assert ls(9000, 0, True, ar.FLAG_SPLIT(2))["threads"] == 64
    # no softmax and no output norm: the CTAs of a token never talk
    assert ls(256, 0, False) == dict(kernel="split", split=7, stages=0, threads=128, ctas=1792, cluster=1)
    assert ls(2, 8, True, ar.FLAG_SPLIT(16)) == dict(kernel="split", split=16, stages=0, threads=64, ctas=32, cluster=16)
    assert ls(2, 8, True, ar.FLAG_SPLIT(4))["threads"] == 224
    assert ls(2, 8, True, ar.FLAG_SPLIT(14))["threads"] == 64
    assert ls(2, 8, True, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(4) | ar.FLAG_VPT(2) | ar.FLAG_STAGES(3))["stages"] == 3
    assert ls(9000, 8, True, ar.FLAG_KERNEL(1))["kernel"] == "split"
    assert ls(10, 8, True, ar.FLAG_KERNEL(3)) == dict(kernel="generic", split=1, stages=0, threads=256, ctas=10, cluster=1)
    assert ls(9000, 8, True, ar.FLAG_SPLIT(7) | ar.FLAG_VPT(2))["threads"] == 64
    assert ls(9000, 8, True, ar.FLAG_SPLIT(7) | ar.FLAG_VPT(1))["threads"] == 128
    for bad in [(-1, 0, 0, 0), (1, 9, 0, 0), (1, -1, 0, 0), (1, 1, 0, ar.FLAG_SPLIT(5)),
                (1, 1, 0, ar.FLAG_KERNEL(7)), (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(16)),
                (1, 3, 0, ar.FLAG_KERNEL(5)), (1, 0, 0, ar.FLAG_KERNEL(5) | ar.FLAG_VPT(2)),
                (1, 0, 0, ar.FLAG_KERNEL(5) | ar.FLAG_SPLIT(2)),
                (1, 0, 0, ar.FLAG_KERNEL(6)),
                (1, 3, 0, ar.FLAG_KERNEL(6) | ar.FLAG_VPT(1)),
                (1, 8, 0, ar.FLAG_KERNEL(4)),
                (1, 2, 0, ar.FLAG_KERNEL(4) | ar.FLAG_SPLIT(7) | ar.FLAG_VPT(2) | ar.FLAG_STAGES(2)),
                (1, 1, 0, ar.FLAG_KERNEL(3) | ar.FLAG_SPLIT(7)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_STAGES(4)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(8) | ar.FLAG_VPT(2)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(14) | ar.FLAG_VPT(1)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_STAGES(4)),
                (1, 1, 0, ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(7) | ar.FLAG_VPT(1) | ar.FLAG_STAGES(3)),
                (1, 1, 0, ar.FLAG_KERNEL(1) | ar.FLAG_VPT(2)),
                (1, 1, 0, ar.FLAG_KERNEL(1) | ar.FLAG_STAGES(2)), (1, 1, 0, 1 << 30),
                (1, 1, 0, ar.FLAG_TP_GRAM)]:
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
    ("blocks_capacity", -1, 1), ("flags", 0x4, 1), ("flags", ar.FLAG_TP_GRAM, 1), ("flags", ar.FLAG_SPLIT(5), 1),
    ("flags", ar.FLAG_KERNEL(7), 1), ("flags", ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(16), 1),
    ("blocks_group", -1, 1),
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
    kw["layout"].flags = ar.FLAG_KERNEL(2) | ar.FLAG_VPT(4)
    assert ar.call_raw(**kw, H=64) == 1             # no shape overrides at other widths
    kw["layout"].flags = ar.FLAG_KERNEL(1) | ar.FLAG_SPLIT(7)
    assert ar.call_raw(**kw, H=64) == 1


def test_any_width_stream_checks(lib):
    """Widths up to 16384 may take the stream kernel's any-width form
    (ceil(H / 1024) CTAs per row), in its one shape; wider rows and shape
    overrides may not."""
    import torch
    no_gpu = not torch.cuda.is_available()
    for Hh in (64, 1000, 1024, 1536, 4000, 4096, 16376, 16384):
        kw = good_h(Hh, T=200)
        kw["layout"].flags = ar.FLAG_KERNEL(2)
        if no_gpu:
            assert ar.call_raw(**kw, H=Hh) in (4, 5)
        kw["layout"].flags = ar.FLAG_KERNEL(2) | ar.FLAG_VPT(2)
        assert ar.call_raw(**kw, H=Hh) == 1
    for Hh in (17408, 16392):                        # 17 CTAs per row
        kw = good_h(Hh, T=200)
        kw["layout"].flags = ar.FLAG_KERNEL(2)
        assert ar.call_raw(**kw, H=Hh) == 1
        kw["layout"].flags = 0                      # automatic: the general kernel
        if no_gpu:
            assert ar.call_raw(**kw, H=Hh) in (4, 5)
    kw = good_h(4096, T=200, S=0)
    kw["out_norm_w"] = 0
    kw["layout"].flags = ar.FLAG_KERNEL(2)           # no exchange: not a stream case
    assert ar.call_raw(**kw, H=4096) == 1
    # the split kernel's any-width form: up to 8 CTAs per row
    kw = good_h(8192, T=4)
    kw["layout"].flags = ar.FLAG_KERNEL(1)
    if no_gpu:
        assert ar.call_raw(**kw, H=8192) in (4, 5)
    kw["layout"].flags = ar.FLAG_KERNEL(1) | ar.FLAG_SPLIT(8)
    assert ar.call_raw(**kw, H=8192) == 1           # no overrides
    for Hh in (9216, 8200):                          # 9 CTAs per row
        kw = good_h(Hh, T=4)
        kw["layout"].flags = ar.FLAG_KERNEL(1)
        assert ar.call_raw(**kw, H=Hh) == 1
    for Hh in (8, 1000, 8184):                       # 1 .. 8 CTAs, a short last one
        kw = good_h(Hh, T=4)
        kw["layout"].flags = ar.FLAG_KERNEL(1)
        if no_gpu:
            assert ar.call_raw(**kw, H=Hh) in (4, 5)


# ---- hidden-sharded entry points (host checks only) ----

HS = 896  # one rank's shard of 7168 over 8 ranks


def tp_layout(T=4, cap=8, flags=0, W=HS):
    return ar.Layout(prefix_row=W, delta_row=W, blocks_token=cap * W, blocks_slot=W,
                     out_row=W, blocks_capacity=cap, flags=flags)


def tp_call(phase, T=4, S=4, Hs=HS, Hfull=H, sums_row=None, sums=None, sq=None, widx=-1,
            onorm=True, flags=0, **ptrs):
    import ctypes

    L = ar.lib()
    lay = tp_layout(T=T, flags=flags, W=max(Hs, HS))
    p = dict(prefix=addr(0), delta=addr(1), blocks=addr(2), res_w=addr(3), rms_w=addr(4),
             onw=addr(5) if onorm else 0, out=addr(6))
    p.update(ptrs)
    sums = addr(7) if sums is None else sums
    sq = addr(8) if sq is None else sq
    sums_row = 2 * (S + 1) if sums_row is None else sums_row
    n = lambda v: v or None  # noqa: E731
    if phase == 0:
        return L.attn_res_tp_sums(Hs, n(p["prefix"]), n(p["delta"]), n(p["blocks"]), S,
                                  n(p["res_w"]), n(p["rms_w"]), n(sums), sums_row, T,
                                  ctypes.byref(lay), None)
    if phase == 1:
        return L.attn_res_tp_sq(Hs, Hfull, n(p["prefix"]), n(p["delta"]), n(p["blocks"]), S,
                                1e-6, n(sums), sums_row, n(sq), T, ctypes.byref(lay), None)
    return L.attn_res_tp_finish(Hs, Hfull, n(p["prefix"]), n(p["delta"]), n(p["blocks"]), S,
                                widx, n(p["onw"]), 1e-6, 1e-6, n(sums), sums_row, n(sq),
                                n(p["out"]), T, ctypes.byref(lay), None)


@pytest.mark.parametrize("phase", [0, 1, 2])
def test_tp_valid_arguments_reach_the_device_check(lib, phase):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert tp_call(phase) in (4, 5)
    assert tp_call(phase, T=0) == 0


@pytest.mark.parametrize("phase", [0, 1, 2])
@pytest.mark.parametrize("change,status", [
    (dict(Hs=900), 1),                       # not a multiple of 8
    (dict(Hs=0), 1),
    (dict(sums_row=9), 1),                   # < 2N
    (dict(S=9), 1),
    (dict(T=-1), 1),
    (dict(sums=0), 1),
    (dict(sums=addr(7, 2)), 2),              # floats want 4-byte alignment
    (dict(prefix=addr(0, 8)), 2),
    (dict(flags=ar.FLAG_SPLIT(7)), 1),       # no split or vector overrides
    (dict(flags=ar.FLAG_VPT(2)), 1),
    (dict(flags=ar.FLAG_KERNEL(1)), 1),      # forms: ring (2) or one CTA per row (3)
    (dict(flags=ar.FLAG_KERNEL(4)), 1),
    (dict(flags=ar.FLAG_STAGES(1)), 1),      # ring depth 2..4
    (dict(flags=ar.FLAG_STAGES(5)), 1),
    (dict(flags=ar.FLAG_KERNEL(3) | ar.FLAG_STAGES(2)), 1),   # a depth without the ring
    # a forced ring whose stages do not fit in shared memory (2 x 6 rows x 32 KB)
    (dict(flags=ar.FLAG_KERNEL(2), Hs=16384, Hfull=16384), 1),
])
def test_tp_rejections(lib, phase, change, status):
    assert tp_call(phase, **change) == status


@pytest.mark.parametrize("phase", [0, 1, 2])
@pytest.mark.parametrize("flags", [ar.FLAG_KERNEL(2), ar.FLAG_KERNEL(3),
                                   ar.FLAG_KERNEL(2) | ar.FLAG_STAGES(2),
                                   ar.FLAG_KERNEL(2) | ar.FLAG_STAGES(4), ar.FLAG_STAGES(3)])
def test_tp_form_overrides_accepted(lib, phase, flags):
    """Both forms and the ring depths 2..4 pass the host checks (then the
    device check, without a GPU); a depth with the automatic form at few
    rows (one CTA per row) does not apply.  A wide shard falls back to one
    CTA per row unless the ring is forced."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert tp_call(phase, flags=flags) in (4, 5)
    assert tp_call(phase, Hs=16384, Hfull=16384) in (4, 5)


def test_tp_phase_specific_rejections(lib):
    assert tp_call(1, Hfull=HS - 8) == 1                # full width below the shard's
    assert tp_call(2, Hfull=HS - 8) == 1
    assert tp_call(1, sq=0) == 1                         # sq is the output of phase 1
    assert tp_call(2, sq=0) == 1                         # the output norm needs sq
    assert tp_call(1, sq=addr(8, 2)) == 2
    assert tp_call(0, res_w=0) == 1                      # phase 0 reads the weights
    assert tp_call(2, out=0) == 1                        # phase 2 writes out
    assert tp_call(2, onw=addr(5, 8)) == 2
    assert tp_call(0, sums=addr(0, 64)) == 3             # sums written over prefix
    assert tp_call(1, sq=addr(7, 8)) == 3                # sq written over sums
    assert tp_call(2, out=addr(7)) == 3                  # out written over sums
    assert tp_call(2, widx=8) == 1
    import torch
    if not torch.cuda.is_available():
        # reading sums that overlap an input is fine
        assert tp_call(1, sums=addr(1, 64)) in (4, 5)
        assert tp_call(2, sq=0, onorm=False) in (4, 5)   # no output norm: sq unused
        assert tp_call(0, flags=ar.FLAG_PDL) in (4, 5)
        assert tp_call(0, onorm=False, res_w=addr(3), rms_w=addr(4), out=0) in (4, 5)


def test_tp_sums_width(lib):
    assert lib.attn_res_tp_sums_width(8, 0) == 18
    assert lib.attn_res_tp_sums_width(8, 1) == 18 + 36
    assert lib.attn_res_tp_sums_width(0, 1) == 2
    assert lib.attn_res_tp_sums_width(4, 1) == 10 + 10
    assert lib.attn_res_tp_sums_width(9, 0) == -1
    assert lib.attn_res_tp_sums_width(-1, 1) == -1
    from attention_residual_fusion_gb300 import tp
    for S in range(9):
        for g in (0, 1):
            assert tp.sums_width(S, bool(g)) == lib.attn_res_tp_sums_width(S, g)


def test_tp_gram_flag(lib):
    G = ar.FLAG_TP_GRAM
    assert tp_call(1, flags=G) == 1                       # no sq phase in the Gram form
    assert tp_call(0, flags=G) == 1                       # sums_row 10 < 10 + 10
    assert tp_call(2, flags=G) == 1
    import torch
    if not torch.cuda.is_available():
        assert tp_call(0, flags=G, sums_row=20) in (4, 5)
        assert tp_call(2, flags=G | ar.FLAG_PDL, sums_row=20, sq=0) in (4, 5)  # sq unused
        assert tp_call(2, flags=G, sums_row=20, sq=addr(0, 2)) in (4, 5)       # not checked


def test_shared_bank_rows_host_checks(lib):
    import ctypes
    assert ctypes.sizeof(ar.Layout) == 56
    import torch
    no_gpu = not torch.cuda.is_available()
    # a written slot that is also a source is rejected once rows share a bank row
    kw = good(S=4, widx=2)
    kw["layout"].blocks_group = 2
    assert call(**kw) == 1
    kw["layout"].blocks_group = 1
    if no_gpu:
        assert call(**kw) in (4, 5)
    # a slot that is not a source is fine
    kw = good(S=4, widx=6)
    kw["layout"].blocks_group = 2
    if no_gpu:
        assert call(**kw) in (4, 5)
    # T = 4 rows in groups of 4: one bank row, so its token stride is unused
    kw = good(T=4, S=4, widx=6)
    kw["layout"].blocks_group = 4
    kw["layout"].blocks_token = 0
    if no_gpu:
        assert call(**kw) in (4, 5)
    kw["layout"].blocks_group = 2                        # two bank rows: stride checked
    assert call(**kw) == 1
    # the bank extent shrinks with B: an out placed after ceil(T/B) bank rows
    kw = good(T=4, S=4, widx=6)
    kw["layout"].blocks_group = 4
    kw["out"] = addr(2, 8 * H * 2 + 4096)                # past one bank row of 8 slots
    if no_gpu:
        assert call(**kw) in (4, 5)
    kw["layout"].blocks_group = 1                        # four bank rows: overlaps
    assert call(**kw) == 3
    # B > 1: the stream kernel has the one shape (7,2,2)
    kw = good(T=300, S=4, widx=6)
    kw["layout"].blocks_group = 2
    kw["layout"].blocks_token = 8 * H
    kw["layout"].flags = ar.FLAG_KERNEL(2) | ar.FLAG_VPT(4)
    assert call(**kw) == 1
    kw["layout"].flags = ar.FLAG_KERNEL(2) | ar.FLAG_SPLIT(7) | ar.FLAG_VPT(2) | ar.FLAG_STAGES(2)
    if no_gpu:
        assert call(**kw) in (4, 5)


def test_binding_rejects_host_tensors_and_bad_shapes(lib):
    """The binding only marshals device bf16 tensors: host or float tensors,
    and a bank with fewer than ceil(T / blocks_group) token rows, are refused
    before any call (no CPU path)."""
    import torch
    from attention_residual_fusion_gb300 import tp
    T, Hh = 4, 64
    p = torch.zeros((T, Hh), dtype=torch.bfloat16)
    b = torch.zeros((T, 8, Hh), dtype=torch.bfloat16)
    w = torch.ones(Hh, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ar.attn_res(p, None, b, 4, -1, w, w)                      # host tensors
    with pytest.raises(ValueError):
        ar.attn_res(p.float(), None, b, 4, -1, w, w)              # not bf16
    with pytest.raises(ValueError):
        tp.tp_sums(p, None, b, 4, w, w, torch.zeros((T, 10)))     # host tensors
    with pytest.raises(ValueError):
        ar.make_layout(p, None, b[:1], None, 0, blocks_group=2)   # 1 < ceil(4 / 2) bank rows
    lay = ar.make_layout(p, None, b[:2], None, 0, blocks_group=2)
    assert lay.blocks_group == 2 and lay.blocks_token == 8 * Hh and lay.blocks_capacity == 8
    with pytest.raises(ValueError):
        ar.make_layout(p, None, b.transpose(1, 2), None, 0)       # inner stride not 1


def test_extents_that_would_overflow_are_rejected(lib):
    """(rows - 1) x stride far beyond any memory is refused before any
    address arithmetic could wrap."""
    kw = good(T=1 << 30)
    kw["layout"].prefix_row = 1 << 39
    assert call(**kw) == 1
    kw = good(T=1 << 30)
    kw["layout"].blocks_token = 1 << 39
    assert call(**kw) == 1
    assert tp_call(0, T=1 << 30, sums_row=1 << 39) == 1
