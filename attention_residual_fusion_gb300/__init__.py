"""GB300-native Kimi-K3 attention-residual (AttnRes) mixture.

Thin Python binding of the C ABI in ``include/attn_res.h``.  Every step of the
mixture runs in the sm_103a kernels of ``libattn_res.so``; this module only
turns torch tensors into pointers, strides and a stream.  There is no CPU or
PyTorch fallback: if the library is not built, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from ._build import LIB as LIB_PATH

HIDDEN = 7168
MAX_BLOCKS = 8

FLAG_PDL = 0x1
FLAG_TP_GRAM = 0x2
KERNEL_SPLIT = 1
KERNEL_STREAM = 2
KERNEL_GENERIC = 3
KERNEL_STAGED = 4
KERNEL_ROW = 5
KERNEL_ROW_SMEM = 6
KERNEL_NAMES = {KERNEL_SPLIT: "split", KERNEL_STREAM: "stream", KERNEL_GENERIC: "generic",
                KERNEL_STAGED: "staged", KERNEL_ROW: "row",
                KERNEL_ROW_SMEM: "row_smem"}


def FLAG_SPLIT(k: int) -> int:
    return (int(k) & 0xFF) << 8


def FLAG_KERNEL(k: int) -> int:
    return (int(k) & 0xF) << 16


def FLAG_STAGES(n: int) -> int:
    return (int(n) & 0xF) << 20


def FLAG_VPT(n: int) -> int:
    return (int(n) & 0xF) << 24


STATUS = {0: "ATTN_RES_OK", 1: "ATTN_RES_EINVAL", 2: "ATTN_RES_EALIGN",
          3: "ATTN_RES_EALIAS", 4: "ATTN_RES_ECUDA", 5: "ATTN_RES_EDEVICE"}

# Every symbol the header declares.
EXPORTS = ("attn_res", "attn_res_status_string", "attn_res_hidden_size",
           "attn_res_max_blocks", "attn_res_launch_shape", "attn_res_device_status",
           "attn_res_selftest_wait_timeout", "attn_res_h", "attn_res_tp_sums",
           "attn_res_tp_sq", "attn_res_tp_finish", "attn_res_tp_sums_width")


class Layout(ctypes.Structure):
    """attn_res_layout_t"""
    _fields_ = [("prefix_row", ctypes.c_int64), ("delta_row", ctypes.c_int64),
                ("blocks_token", ctypes.c_int64), ("blocks_slot", ctypes.c_int64),
                ("out_row", ctypes.c_int64), ("blocks_capacity", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("blocks_group", ctypes.c_int32)]


class AttnResError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def library_path() -> str:
    return LIB_PATH


def lib():
    """The loaded libattn_res.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "attention_residual_fusion_gb300._build.build() (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp = ctypes.c_void_p
        L.attn_res.restype = ctypes.c_int
        L.attn_res.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                               ctypes.c_float, ctypes.c_float, vp, ctypes.c_int64,
                               ctypes.POINTER(Layout), vp]
        L.attn_res_h.restype = ctypes.c_int
        L.attn_res_h.argtypes = [ctypes.c_int64] + L.attn_res.argtypes
        L.attn_res_status_string.restype = ctypes.c_char_p
        L.attn_res_status_string.argtypes = [ctypes.c_int]
        L.attn_res_hidden_size.restype = ctypes.c_int
        L.attn_res_hidden_size.argtypes = []
        L.attn_res_max_blocks.restype = ctypes.c_int
        L.attn_res_max_blocks.argtypes = []
        L.attn_res_launch_shape.restype = ctypes.c_int
        ip = ctypes.POINTER(ctypes.c_int)
        L.attn_res_launch_shape.argtypes = [
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
            ip, ip, ip, ip, ctypes.POINTER(ctypes.c_int64), ip]
        L.attn_res_device_status.restype = ctypes.c_int
        L.attn_res_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
        L.attn_res_selftest_wait_timeout.restype = ctypes.c_int
        L.attn_res_selftest_wait_timeout.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_uint)]
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lp = ctypes.POINTER(Layout)
        L.attn_res_tp_sums_width.restype = ctypes.c_int
        L.attn_res_tp_sums_width.argtypes = [i32, i32]
        L.attn_res_tp_sums.restype = ctypes.c_int
        L.attn_res_tp_sums.argtypes = [i64, vp, vp, vp, i32, vp, vp, vp, i64, i64, lp, vp]
        L.attn_res_tp_sq.restype = ctypes.c_int
        L.attn_res_tp_sq.argtypes = [i64, i64, vp, vp, vp, i32, f32, vp, i64, vp, i64, lp, vp]
        L.attn_res_tp_finish.restype = ctypes.c_int
        L.attn_res_tp_finish.argtypes = [i64, i64, vp, vp, vp, i32, i32, vp, f32, f32, vp, i64,
                                         vp, vp, i64, lp, vp]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().attn_res_status_string(status).decode()


def launch_shape(T: int, num_blocks: int, has_out_norm: bool, flags: int = 0,
                 has_delta: bool = True) -> dict:
    """Launch attn_res would make: kernel, split, stages, threads per CTA,
    CTAs (0 = persistent grid sized to the device) and cluster size."""
    kern, k, st_, th, cl = (ctypes.c_int() for _ in range(5))
    ctas = ctypes.c_int64()
    st = lib().attn_res_launch_shape(T, num_blocks, int(has_delta), int(has_out_norm), flags,
                                     ctypes.byref(kern), ctypes.byref(k),
                                     ctypes.byref(st_), ctypes.byref(th),
                                     ctypes.byref(ctas), ctypes.byref(cl))
    if st != 0:
        raise AttnResError(st, status_string(st))
    return dict(kernel=KERNEL_NAMES[kern.value], split=k.value,
                stages=st_.value, threads=th.value, ctas=ctas.value, cluster=cl.value)


def device_status(clear: bool = False) -> int:
    """Error bits recorded by the kernels on the current device (0 = none)."""
    bits = ctypes.c_uint()
    st = lib().attn_res_device_status(ctypes.byref(bits), int(clear))
    if st != 0:
        raise AttnResError(st, status_string(st))
    return bits.value


def selftest_wait_timeout(limit_us: int) -> int:
    """Run the bounded-wait self-test; returns the device status word."""
    bits = ctypes.c_uint()
    st = lib().attn_res_selftest_wait_timeout(limit_us, ctypes.byref(bits))
    if st != 0:
        raise AttnResError(st, status_string(st))
    return bits.value


def call_raw(prefix: int, delta: int, blocks: int, num_blocks: int,
             block_write_idx: int, res_w: int, rms_w: int, out_norm_w: int,
             eps: float, out_eps: float, out: int, T: int, layout: Layout,
             stream: int, H: int = HIDDEN) -> int:
    """The C entry point on raw addresses (attn_res, or attn_res_h when H is
    not the built-in width); returns the status code."""
    args = (prefix or None, delta or None, blocks or None, num_blocks,
            block_write_idx, res_w or None, rms_w or None, out_norm_w or None,
            eps, out_eps, out or None, T, ctypes.byref(layout), stream or None)
    if H == HIDDEN:
        return lib().attn_res(*args)
    return lib().attn_res_h(H, *args)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def check_bf16_cuda(**tensors) -> None:
    import torch

    for name, t in tensors.items():
        if t is not None and (t.dtype != torch.bfloat16 or t.device.type != "cuda"):
            raise ValueError(f"{name} must be a CUDA bfloat16 tensor")


def make_layout(prefix, delta, blocks, out, flags: int, blocks_group: int = 1) -> Layout:
    """attn_res_layout_t from the tensors' strides (row tensors [T, W] and
    the bank [ceil(T / blocks_group), capacity, W], all with unit inner
    stride; out may be None)."""
    for name, t in (("prefix", prefix), ("delta", delta), ("out", out)):
        if t is not None and (t.dim() != 2 or t.stride(1) != 1):
            raise ValueError(f"{name} must be a [T, H] tensor with unit inner stride")
    if blocks is not None and (blocks.dim() != 3 or blocks.stride(2) != 1):
        raise ValueError("blocks must be a [T, capacity, H] tensor with unit inner stride")
    if blocks is not None and blocks_group >= 1 and \
            blocks.shape[0] < -(-prefix.shape[0] // blocks_group):
        raise ValueError("blocks has fewer than ceil(T / blocks_group) token rows")
    return Layout(prefix_row=prefix.stride(0),
                  delta_row=delta.stride(0) if delta is not None else 0,
                  blocks_token=blocks.stride(0) if blocks is not None else 0,
                  blocks_slot=blocks.stride(1) if blocks is not None else 0,
                  out_row=out.stride(0) if out is not None else 0,
                  blocks_capacity=blocks.shape[1] if blocks is not None else 0,
                  flags=flags, blocks_group=blocks_group)


def attn_res(prefix, delta, blocks, num_blocks: int, block_write_idx: int,
             res_w, rms_w, out_norm_w=None, eps: float = 1e-6,
             out_eps: float = 1e-6, out=None, *, pdl: bool = False,
             split: int = 0, kernel: int = 0, stages: int = 0, vpt: int = 0,
             blocks_group: int = 1, stream=None):
    """AttnRes mixture on CUDA bf16 tensors (see include/attn_res.h); H is
    the length of ``res_w`` (7168 for the tuned kernels, any multiple of 8).

    prefix [T, H] (updated in place when ``delta`` is given), delta [T, H] or
    None, blocks [T, capacity, H] (any token/slot strides, unit inner stride;
    slot ``block_write_idx`` is overwritten when >= 0), res_w / rms_w /
    out_norm_w [H].  With ``blocks_group`` = B > 1, token row t uses bank row
    t // B (blocks is [ceil(T / B), capacity, H]).  Returns ``out`` [T, H]
    (allocated if not given).
    """
    import torch

    check_bf16_cuda(prefix=prefix, delta=delta, blocks=blocks, res_w=res_w, rms_w=rms_w,
                    out_norm_w=out_norm_w, out=out)
    T = prefix.shape[0]
    H = res_w.shape[0]
    if out is None:
        out = torch.empty((T, H), dtype=prefix.dtype, device=prefix.device)
    lay = make_layout(prefix, delta, blocks, out,
                      (FLAG_PDL if pdl else 0) | FLAG_SPLIT(split) | FLAG_KERNEL(kernel) |
                      FLAG_STAGES(stages) | FLAG_VPT(vpt), blocks_group)
    if stream is None:
        stream = torch.cuda.current_stream(prefix.device)
    st = call_raw(_ptr(prefix), _ptr(delta), _ptr(blocks), num_blocks,
                  block_write_idx, _ptr(res_w), _ptr(rms_w), _ptr(out_norm_w),
                  eps, out_eps, _ptr(out), T, lay, int(stream.cuda_stream), H)
    if st != 0:
        raise AttnResError(st, status_string(st))
    return out
