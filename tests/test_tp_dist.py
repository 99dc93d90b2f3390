"""The hidden-sharded orchestration across real processes on CPU: two gloo
ranks each hold a column shard and run attn_res_tp with torch.distributed's
all-reduce.  The device phases are replaced by float64 numpy stand-ins of the
three kernels (per-shard partial sums, per-shard sum of squares, output and
write-backs), so the test checks the orchestration -- the order of the calls,
what is reduced and when, the full width H -- not the kernels.  The composed
rows must match the oracle on the full rows."""
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from attention_residual_fusion_gb300 import workloads as W
from tests import gpu_util as G
from tests import restatement as R


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _set_bits(t, bits: np.ndarray) -> None:
    t.copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16))


def _current_bits(prefix, delta) -> np.ndarray:
    # the sum of two bf16 values, rounded to float32 and then to bf16, is the
    # sum rounded once to bf16: a float32 rounding error can never land on a
    # bf16 halfway point
    if delta is None:
        return _bits(prefix)
    s = (R.widen(_bits(prefix)) + R.widen(_bits(delta))).astype(np.float32)
    return R.bf16_round_via_f32(s)


def _sources(prefix, delta, blocks, S):
    xs = [R.widen(_bits(blocks[:, i, :])) for i in range(S)]
    c = _current_bits(prefix, delta)
    return xs + [R.widen(c)], c


def _weights(sums, S, H, eps):
    N = S + 1
    s = sums.numpy().astype(np.float64)
    logit = s[:, N:2 * N] / np.sqrt(s[:, :N] / H + eps)
    e = np.exp(logit - logit.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _mix(xs, w):
    return sum(w[:, i:i + 1] * x for i, x in enumerate(xs))


def standin_sums(prefix, delta, blocks, S, res_w, rms_w, sums, gram=False, **_):
    xs, _c = _sources(prefix, delta, blocks, S)
    q = R.widen(_bits(rms_w)) * R.widen(_bits(res_w))
    N = S + 1
    for i, x in enumerate(xs):
        sums[:, i] = torch.from_numpy((x * x).sum(axis=1))
        sums[:, N + i] = torch.from_numpy(x @ q)
    if gram:
        g = 2 * N
        for i in range(N):
            for j in range(i + 1, N):
                sums[:, g] = torch.from_numpy((xs[i] * xs[j]).sum(axis=1))
                g += 1


def standin_sq(prefix, delta, blocks, S, H, eps, sums, sq, **_):
    xs, _c = _sources(prefix, delta, blocks, S)
    acc = _mix(xs, _weights(sums, S, H, eps))
    sq.copy_(torch.from_numpy((acc * acc).sum(axis=1)))


def _gram_sq(sums, w):
    """sum acc^2 = sum_i w_i^2 ss_i + 2 sum_{i<j} w_i w_j g_ij."""
    N = w.shape[1]
    s = sums.numpy().astype(np.float64)
    tot = sum(w[:, i] ** 2 * s[:, i] for i in range(N))
    g = 2 * N
    for i in range(N):
        for j in range(i + 1, N):
            tot = tot + 2 * w[:, i] * w[:, j] * s[:, g]
            g += 1
    return tot


def standin_finish(prefix, delta, blocks, S, widx, H, onw, eps, out_eps, sums, sq, out,
                   gram=False, **_):
    xs, c = _sources(prefix, delta, blocks, S)
    w = _weights(sums, S, H, eps)
    acc = _mix(xs, w)
    if onw is not None:
        total = _gram_sq(sums, w) if gram else sq.numpy().astype(np.float64)
        ro = 1.0 / np.sqrt(total / H + out_eps)
        acc = acc * ro[:, None] * R.widen(_bits(onw))
    _set_bits(out, R.bf16_round_via_f32(acc.astype(np.float32)))
    if delta is not None:
        _set_bits(prefix, c)
    if widx >= 0:
        _set_bits(blocks[:, widx, :], c)


STANDIN = types.SimpleNamespace(sums=standin_sums, sq=standin_sq, finish=standin_finish)


def _workload(case):
    S, d, o, w, H = case[:5]
    return W.make_workload(6, S, capacity=9, has_delta=d, has_out_norm=o, block_write_idx=w,
                           seed=31 + S, H=H, mixing=True)


def _tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _chunk(case):
    return case[6] if len(case) > 6 else None


def _rank(rank, world, port, cases, out):
    import torch.distributed as dist
    from attention_residual_fusion_gb300 import tp

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for k, case in enumerate(cases):
            wl = _workload(case)
            Hs = wl.H // world
            a, b = rank * Hs, (rank + 1) * Hs
            prefix = _tensor(wl.prefix[:, a:b])
            delta = None if wl.delta is None else _tensor(wl.delta[:, a:b])
            bank = _tensor(wl.bank[:, :, a:b])
            onw = None if wl.out_norm_w is None else _tensor(wl.out_norm_w[a:b])
            res = tp.attn_res_tp(prefix, delta, bank, wl.num_blocks, wl.block_write_idx,
                                 _tensor(wl.res_w[a:b]), _tensor(wl.rms_w[a:b]), onw,
                                 wl.eps, wl.out_eps, phases=STANDIN,
                                 gram=len(case) > 5 and case[5], chunk_tokens=_chunk(case))
            out[(k, rank)] = (_bits(res), _bits(prefix), _bits(bank))
    finally:
        dist.destroy_process_group()


CASES = [(8, True, True, 8, 256), (4, False, True, 2, 128), (0, True, False, 0, 64),
         (1, False, False, -1, 64), (8, True, False, 3, 512), (8, True, True, 8, 256, True),
         (2, False, True, -1, 64, True), (8, True, True, 8, 256, False, 4),
         (4, True, True, 4, 128, True, 2), (3, False, False, 3, 64, False, 5)]


def test_two_gloo_ranks_compose_to_the_oracle():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, CASES, out), nprocs=world, join=True)
        res = dict(out)
    for k, case in enumerate(CASES):
        wl = _workload(case)
        ref = oracle.run_workload(wl)
        parts = [res[(k, r)] for r in range(world)]
        gpu = dict(out=np.concatenate([p[0] for p in parts], axis=1),
                   prefix=np.concatenate([p[1] for p in parts], axis=1),
                   bank=np.concatenate([p[2] for p in parts], axis=2))
        gpu["prefix_full"], gpu["out_full"] = gpu["prefix"], gpu["out"]
        G.check_against_oracle(wl, gpu, ref, tag=f"gloo_case{k}")


def test_one_rank_without_a_process_group_is_local():
    """No process group: the all-reduce is a no-op and H is the shard width."""
    from attention_residual_fusion_gb300 import tp

    wl = _workload((4, True, True, 4, 128))
    prefix, bank = _tensor(wl.prefix.copy()), _tensor(wl.bank.copy())
    res = tp.attn_res_tp(prefix, _tensor(wl.delta), bank, 4, 4, _tensor(wl.res_w),
                         _tensor(wl.rms_w), _tensor(wl.out_norm_w), wl.eps, wl.out_eps,
                         phases=STANDIN)
    ref = oracle.run_workload(wl)
    gpu = dict(out=_bits(res), prefix=_bits(prefix), bank=_bits(bank))
    gpu["prefix_full"], gpu["out_full"] = gpu["prefix"], gpu["out"]
    G.check_against_oracle(wl, gpu, ref, tag="local")


def test_reductions_are_called_in_order():
    from attention_residual_fusion_gb300 import tp

    seen = []

    def fake_reduce(t):
        seen.append(tuple(t.shape))

    wl = _workload((8, True, True, 8, 64))
    tp.attn_res_tp(_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8, 8,
                   _tensor(wl.res_w), _tensor(wl.rms_w), _tensor(wl.out_norm_w), H=64,
                   all_reduce=fake_reduce, phases=STANDIN)
    assert seen == [(6, 18), (6,)]
    seen.clear()
    tp.attn_res_tp(_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8, 8,
                   _tensor(wl.res_w), _tensor(wl.rms_w), None, H=64,
                   all_reduce=fake_reduce, phases=STANDIN)
    assert seen == [(6, 18)]
    seen.clear()
    tp.attn_res_tp(_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8, 8,
                   _tensor(wl.res_w), _tensor(wl.rms_w), _tensor(wl.out_norm_w), H=64,
                   all_reduce=fake_reduce, phases=STANDIN, gram=True)
    assert seen == [(6, 54)]
    # chunks of 2 rows: chunk c+1's sums are reduced before chunk c's sum of
    # squares, and a finish waits for its own chunk's reduction only
    seen.clear()
    tp.attn_res_tp(_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8, 8,
                   _tensor(wl.res_w), _tensor(wl.rms_w), _tensor(wl.out_norm_w), H=64,
                   all_reduce=fake_reduce, phases=STANDIN, chunk_tokens=2)
    assert seen == [(2, 18), (2, 18), (2,), (2, 18), (2,), (2,)]
    seen.clear()
    tp.attn_res_tp(_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8, 8,
                   _tensor(wl.res_w), _tensor(wl.rms_w), _tensor(wl.out_norm_w), H=64,
                   all_reduce=fake_reduce, phases=STANDIN, chunk_tokens=4, gram=True)
    assert seen == [(4, 54), (2, 54)]
    with pytest.raises(ValueError):
        tp.attn_res_tp(_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8,
                       8, _tensor(wl.res_w), _tensor(wl.rms_w), _tensor(wl.out_norm_w), H=64,
                       all_reduce=fake_reduce, phases=STANDIN, chunk_tokens=3, blocks_group=2)


def test_kernel_form_reaches_every_phase():
    """kernel / stages are passed to every phase call (and nothing extra is
    passed when they are left automatic)."""
    from attention_residual_fusion_gb300 import tp

    calls = []

    def wrap(name, fn):
        def f(*a, **kw):
            calls.append((name, kw.get("kernel"), kw.get("stages")))
            return fn(*a, **kw)
        return f

    spy = types.SimpleNamespace(sums=wrap("sums", standin_sums), sq=wrap("sq", standin_sq),
                                finish=wrap("finish", standin_finish))
    wl = _workload((8, True, True, 8, 64))
    args = (_tensor(wl.prefix.copy()), _tensor(wl.delta), _tensor(wl.bank.copy()), 8, 8,
            _tensor(wl.res_w), _tensor(wl.rms_w), _tensor(wl.out_norm_w))
    tp.attn_res_tp(*args, H=64, all_reduce=lambda t: None, phases=spy, kernel=2, stages=3)
    assert calls == [("sums", 2, 3), ("sq", 2, 3), ("finish", 2, 3)]
    calls.clear()
    tp.attn_res_tp(*args, H=64, all_reduce=lambda t: None, phases=spy)
    assert calls == [("sums", None, None), ("sq", None, None), ("finish", None, None)]
    import attention_residual_fusion_gb300 as ar
    assert tp._flags(True, True, 2, 3) == (ar.FLAG_PDL | ar.FLAG_TP_GRAM | ar.FLAG_KERNEL(2)
                                           | ar.FLAG_STAGES(3))


def test_standins_pin_to_the_oracle_unsharded():
    """The stand-ins themselves, with no sharding, agree with the oracle (so a
    failure above points at the orchestration)."""
    wl = _workload((8, True, True, 8, 256))
    prefix, bank = _tensor(wl.prefix.copy()), _tensor(wl.bank.copy())
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16)
    sums = torch.empty((wl.T, 18), dtype=torch.float32)
    sq = torch.empty((wl.T,), dtype=torch.float32)
    delta, rw, mw, onw = (_tensor(x) for x in (wl.delta, wl.res_w, wl.rms_w, wl.out_norm_w))
    standin_sums(prefix, delta, bank, 8, rw, mw, sums)
    standin_sq(prefix, delta, bank, 8, wl.H, wl.eps, sums, sq)
    standin_finish(prefix, delta, bank, 8, 8, wl.H, onw, wl.eps, wl.out_eps, sums, sq, out)
    ref = oracle.run_workload(wl)
    gpu = dict(out=_bits(out), prefix=_bits(prefix), bank=_bits(bank))
    gpu["prefix_full"], gpu["out_full"] = gpu["prefix"], gpu["out"]
    G.check_against_oracle(wl, gpu, ref, tag="standin")
    with pytest.raises(AssertionError):
        # planted mistake: a dropped source in the mix must fail the bar
        bad = out.clone()
        w = _weights(sums, 8, wl.H, wl.eps)
        xs, _c = _sources(_tensor(wl.prefix), delta, _tensor(wl.bank), 8)
        acc = sum(w[:, i:i + 1] * x for i, x in enumerate(xs) if i != 3)
        ro = 1.0 / np.sqrt(sq.numpy().astype(np.float64) / wl.H + wl.out_eps)
        _set_bits(bad, R.bf16_round_via_f32((acc * ro[:, None] * R.widen(_bits(onw))).astype(np.float32)))
        G.assert_out_close(_bits(bad), ref["out"], "planted")
