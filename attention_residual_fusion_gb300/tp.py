"""Hidden-sharded (tensor-parallel) AttnRes mixture.

Each rank holds a contiguous column shard of every row (prefix, delta, bank
rows, weights, output).  The mixture needs two full-row reductions -- the
per-source sums behind the logits, and, with an output norm, the sum of
squares of the mixed row -- so it runs as three kernels with an all-reduce
(sum) of a few floats per token between them:

    sums   [T, 2N] fp32  <- attn_res_tp_sums     (N = num_blocks + 1)
    all-reduce(sums)
    sq     [T] fp32      <- attn_res_tp_sq        (output norm only)
    all-reduce(sq)
    out, write-backs     <- attn_res_tp_finish

With ``gram=True`` the first kernel also writes the Gram entries <x_i, x_j>
(i < j) of the shard and the output norm's sum of squares comes from them
after the single all-reduce: one exchange and two passes over the rows
instead of two and three (exact in real arithmetic; in fp32 it loses relative
accuracy where the weighted rows cancel).

The deployments the prhub summary of vllm PR #54261 evaluates include TP8
(impact section); the arithmetic is that of the unsharded mixture
(implementation walkthrough of vllm-ascend PR #14840), with H the full width.

``attn_res_tp`` is the orchestration; its ``phases`` argument defaults to the
CUDA entry points below and its ``all_reduce`` to torch.distributed's.
"""
from __future__ import annotations

import types

from . import (AttnResError, FLAG_KERNEL, FLAG_PDL, FLAG_STAGES, FLAG_TP_GRAM, _ptr,
               check_bf16_cuda, lib, make_layout, status_string)


def sums_width(num_blocks: int, gram: bool = False) -> int:
    """Floats per token row of the reduced buffer: 2N (+ N(N-1)/2 with gram)."""
    n = num_blocks + 1
    return 2 * n + (n * (n - 1) // 2 if gram else 0)


def _flags(pdl: bool, gram: bool, kernel: int = 0, stages: int = 0) -> int:
    """Layout flags of a sharded call.  ``kernel``: 0 automatic,
    KERNEL_STREAM the persistent ring form, KERNEL_GENERIC one CTA per token
    row; ``stages``: ring depth 2..4 (0 automatic)."""
    return ((FLAG_PDL if pdl else 0) | (FLAG_TP_GRAM if gram else 0) | FLAG_KERNEL(kernel) |
            FLAG_STAGES(stages))


def _stream_handle(stream, device) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _check_f32_cuda(**tensors) -> None:
    import torch

    for name, t in tensors.items():
        if t is not None and (t.dtype != torch.float32 or t.device.type != "cuda"):
            raise ValueError(f"{name} must be a CUDA float32 tensor")


def _raise(st: int) -> None:
    if st != 0:
        raise AttnResError(st, status_string(st))


def tp_sums(prefix, delta, blocks, num_blocks: int, res_w, rms_w, sums, *,
            gram: bool = False, pdl: bool = False, blocks_group: int = 1, kernel: int = 0,
            stages: int = 0, stream=None) -> None:
    """attn_res_tp_sums on the shard: sums[t, :2N] = (sum x_i^2, <x_i, q>),
    then the Gram entries with ``gram``."""
    check_bf16_cuda(prefix=prefix, delta=delta, blocks=blocks, res_w=res_w, rms_w=rms_w)
    _check_f32_cuda(sums=sums)
    lay = make_layout(prefix, delta, blocks, None, _flags(pdl, gram, kernel, stages), blocks_group)
    _raise(lib().attn_res_tp_sums(
        res_w.shape[0], _ptr(prefix) or None, _ptr(delta) or None, _ptr(blocks) or None,
        num_blocks, _ptr(res_w) or None, _ptr(rms_w) or None, _ptr(sums) or None,
        sums.stride(0), prefix.shape[0], lay, _stream_handle(stream, prefix.device)))


def tp_sq(prefix, delta, blocks, num_blocks: int, H: int, eps: float, sums, sq, *,
          pdl: bool = False, blocks_group: int = 1, kernel: int = 0, stages: int = 0,
          stream=None) -> None:
    """attn_res_tp_sq on the shard: sq[t] = sum over the shard of acc^2."""
    check_bf16_cuda(prefix=prefix, delta=delta, blocks=blocks)
    _check_f32_cuda(sums=sums, sq=sq)
    lay = make_layout(prefix, delta, blocks, None, _flags(pdl, False, kernel, stages), blocks_group)
    _raise(lib().attn_res_tp_sq(
        prefix.shape[1], H, _ptr(prefix) or None, _ptr(delta) or None, _ptr(blocks) or None,
        num_blocks, eps, _ptr(sums) or None, sums.stride(0), _ptr(sq) or None,
        prefix.shape[0], lay, _stream_handle(stream, prefix.device)))


def tp_finish(prefix, delta, blocks, num_blocks: int, block_write_idx: int, H: int,
              out_norm_w, eps: float, out_eps: float, sums, sq, out, *,
              gram: bool = False, pdl: bool = False, blocks_group: int = 1, kernel: int = 0,
              stages: int = 0, stream=None) -> None:
    """attn_res_tp_finish on the shard: out and the write-backs of c."""
    check_bf16_cuda(prefix=prefix, delta=delta, blocks=blocks, out_norm_w=out_norm_w, out=out)
    _check_f32_cuda(sums=sums, sq=sq)
    lay = make_layout(prefix, delta, blocks, out, _flags(pdl, gram, kernel, stages), blocks_group)
    _raise(lib().attn_res_tp_finish(
        prefix.shape[1], H, _ptr(prefix) or None, _ptr(delta) or None, _ptr(blocks) or None,
        num_blocks, block_write_idx, _ptr(out_norm_w) or None, eps, out_eps,
        _ptr(sums) or None, sums.stride(0), _ptr(sq) or None, _ptr(out) or None,
        prefix.shape[0], lay, _stream_handle(stream, prefix.device)))


CUDA_PHASES = types.SimpleNamespace(sums=tp_sums, sq=tp_sq, finish=tp_finish)


def attn_res_tp(prefix, delta, blocks, num_blocks: int, block_write_idx: int, res_w, rms_w,
                out_norm_w=None, eps: float = 1e-6, out_eps: float = 1e-6, out=None, *,
                H: int | None = None, group=None, all_reduce=None, phases=None,
                gram: bool = False, pdl: bool = False, blocks_group: int = 1,
                chunk_tokens: int | None = None, kernel: int = 0, stages: int = 0, stream=None):
    """The mixture on this rank's column shard (every row-sized argument is
    the shard, width ``res_w.shape[0]``).  ``H`` is the full width (default:
    shard width x world size of ``group``).  ``all_reduce(tensor)`` sums a
    float32 tensor in place over the ranks and may return a handle with
    ``wait()`` (default: torch.distributed's asynchronous all_reduce on
    ``group``; with no process group initialised the call is local).
    ``gram`` selects the single-exchange form; ``blocks_group`` as for
    attn_res; ``kernel`` and ``stages`` pick the kernels' form (see
    ``_flags``; results do not depend on it beyond fp32 summation order).

    ``chunk_tokens`` runs the token rows in chunks, software-pipelined: the
    first kernel of chunk c+1 is issued while the all-reduce of chunk c is in
    flight, and a chunk's later passes follow its first closely enough to
    find its rows in L2 (a chunk of 1024 rows of an 896-column shard with 8
    bank rows is 18 MB).  It must be a multiple of ``blocks_group``.  Every
    rank must pass the same value: the all-reduces are matched by order.

    With ``stream`` given, the buffers, the kernels and the all-reduces are
    all ordered on that stream.  Returns ``out`` (allocated if not given)."""
    import contextlib

    import torch

    ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
    with ctx:
        return _attn_res_tp(prefix, delta, blocks, num_blocks, block_write_idx, res_w, rms_w,
                            out_norm_w, eps, out_eps, out, H, group, all_reduce, phases, gram,
                            pdl, blocks_group, chunk_tokens, kernel, stages, stream)


def _wait(handle) -> None:
    if handle is not None and hasattr(handle, "wait"):
        handle.wait()


def _attn_res_tp(prefix, delta, blocks, num_blocks, block_write_idx, res_w, rms_w, out_norm_w,
                 eps, out_eps, out, H, group, all_reduce, phases, gram, pdl, blocks_group,
                 chunk_tokens, kernel, stages, stream):
    import torch
    import torch.distributed as dist

    T = prefix.shape[0]
    Hs = res_w.shape[0]
    dist_on = dist.is_available() and dist.is_initialized()
    if H is None:
        H = Hs * (dist.get_world_size(group) if dist_on else 1)
    if all_reduce is None:
        if dist_on:
            def all_reduce(t):
                return dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group, async_op=True)
        else:
            def all_reduce(t):
                return None
    B = max(1, int(blocks_group))
    if chunk_tokens is None or chunk_tokens <= 0 or chunk_tokens >= T:
        chunk = max(T, 1)
    else:
        chunk = int(chunk_tokens)
        if chunk % B:
            raise ValueError("chunk_tokens must be a multiple of blocks_group")
    ph = phases or CUDA_PHASES
    dev = prefix.device
    if out is None:
        out = torch.empty((T, Hs), dtype=prefix.dtype, device=dev)
    gram = bool(gram and out_norm_w is not None)  # the Gram entries serve the output norm only
    two = out_norm_w is not None and not gram     # second exchange (sum of squares)
    sums = torch.empty((T, sums_width(num_blocks, gram)), dtype=torch.float32, device=dev)
    sq = torch.empty((T,), dtype=torch.float32, device=dev) if two else None
    kw = dict(pdl=pdl, stream=stream)
    if B != 1:
        kw["blocks_group"] = B
    if kernel or stages:
        kw.update(kernel=kernel, stages=stages)

    bounds = [(c0, min(T, c0 + chunk)) for c0 in range(0, T, chunk)] or [(0, 0)]

    def rows(c):
        c0, c1 = bounds[c]
        bank = None if blocks is None else blocks[c0 // B:-(-c1 // B)]
        return (prefix[c0:c1], None if delta is None else delta[c0:c1], bank,
                out[c0:c1], sums[c0:c1], None if sq is None else sq[c0:c1])

    def first(c):
        p_, d_, b_, _, s_, _ = rows(c)
        ph.sums(p_, d_, b_, num_blocks, res_w, rms_w, s_, gram=gram, **kw)
        return all_reduce(s_)

    def second(c):
        p_, d_, b_, _, s_, q_ = rows(c)
        ph.sq(p_, d_, b_, num_blocks, H, eps, s_, q_, **kw)
        return all_reduce(q_)

    def last(c):
        p_, d_, b_, o_, s_, q_ = rows(c)
        ph.finish(p_, d_, b_, num_blocks, block_write_idx, H, out_norm_w, eps, out_eps, s_, q_,
                  o_, gram=gram, **kw)

    # software pipeline over the chunks: chunk c+1's first pass overlaps the
    # exchange of chunk c, and the finish of chunk c-1 that of chunk c
    n = len(bounds)
    h1 = {0: first(0)}
    h2 = {}
    for c in range(n):
        if c + 1 < n:
            h1[c + 1] = first(c + 1)
        _wait(h1.pop(c))
        if two:
            h2[c] = second(c)
            if c > 0:
                _wait(h2.pop(c - 1))
                last(c - 1)
        else:
            last(c)
    if two:
        _wait(h2.pop(n - 1))
        last(n - 1)
    return out
