"""Hidden-sharded mixture on one GPU vs the CPU oracle.

R ranks are simulated in one process: each rank is a host thread that runs the
orchestration (attn_res_tp) on its column shard of the same device buffers,
and the all-reduce is a host barrier plus a device sum over the ranks'
buffers.  No kernel waits on another.  The composed result must match the
oracle on the full rows with the bar of the unsharded kernels: out within
max(2 bf16 ulp, 1e-2), the updated prefix and every byte of the bank
bit-exact, guard zones untouched."""
import threading

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


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    ar.lib()


class ThreadGroup:
    """All-reduce (sum) among R host threads sharing one device stream."""

    def __init__(self, R: int):
        self.R = R
        self.barrier = threading.Barrier(R, timeout=120)
        self.slots = [None] * R
        self.total = None
        self.calls = [0] * R

    def all_reduce_for(self, r: int):
        def fn(t):
            self.calls[r] += 1
            self.slots[r] = t
            self.barrier.wait()
            if r == 0:
                total = self.slots[0].clone()
                for s in self.slots[1:]:
                    total += s
                self.total = total
            self.barrier.wait()
            t.copy_(self.total)
            self.barrier.wait()
        return fn


def run_tp_ranks(wl: W.Workload, widths, *, pdl=False, out_row=None, gram=False, chunk=None,
                 kernel=0, stages=0):
    """Run attn_res_tp on every column shard (one thread per rank) over guarded
    device copies of the workload; return host copies like gpu_util.run_gpu."""
    import torch

    H = wl.H
    assert sum(widths) == H
    orow = out_row or H
    g_prefix = G.Guarded(wl.prefix, torch)
    g_delta = G.Guarded(wl.delta, torch) if wl.delta is not None else None
    g_bank = G.Guarded(wl.bank, torch)
    g_rms = G.Guarded(wl.rms_w, torch)
    g_res = G.Guarded(wl.res_w, torch)
    g_onw = G.Guarded(wl.out_norm_w, torch) if wl.out_norm_w is not None else None
    g_out = G.Guarded(np.full((wl.T, orow), W.CANARY, dtype=np.uint16), torch)
    bounds = np.concatenate([[0], np.cumsum(widths)])
    group = ThreadGroup(len(widths))
    errors = []
    stream = torch.cuda.current_stream()

    def rank(r):
        a, b = int(bounds[r]), int(bounds[r + 1])
        try:
            with torch.cuda.stream(stream):
                tp.attn_res_tp(
                    g_prefix.view[:, a:b], None if g_delta is None else g_delta.view[:, a:b],
                    g_bank.view[:, :, a:b], wl.num_blocks, wl.block_write_idx,
                    g_res.view[a:b], g_rms.view[a:b],
                    None if g_onw is None else g_onw.view[a:b], wl.eps, wl.out_eps,
                    g_out.view[:, a:b], H=H, all_reduce=group.all_reduce_for(r), gram=gram,
                    pdl=pdl, blocks_group=wl.group, chunk_tokens=chunk, kernel=kernel,
                    stages=stages, stream=stream)
        except BaseException as e:  # noqa: BLE001 - reported below
            errors.append(e)
            group.barrier.abort()

    threads = [threading.Thread(target=rank, args=(r,)) for r in range(len(widths))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]
    torch.cuda.synchronize()
    chunks = -(-wl.T // chunk) if chunk else 1
    expect_calls = (2 if (wl.out_norm_w is not None and not gram) else 1) * max(chunks, 1)
    assert group.calls == [expect_calls] * len(widths)
    bufs = [g for g in (g_prefix, g_delta, g_bank, g_rms, g_res, g_onw, g_out) if g is not None]
    assert all(g.guards_intact() for g in bufs), "a guard zone was written"
    res = dict(out_full=g_out.host(), prefix_full=g_prefix.host(), bank=g_bank.host())
    res["out"] = res["out_full"][:, :H]
    res["prefix"] = res["prefix_full"][:, :H]
    if g_delta is not None:
        assert np.array_equal(g_delta.host(), wl.delta)
    return res


def tp_check(wl, widths, tag, **kw):
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = run_tp_ranks(wl, widths, **kw)
    G.check_against_oracle(wl, gpu, ref, tag=tag)
    return gpu, ref


CASES = [(R, S, d, o, w, g) for R in (1, 2, 8) for S in (0, 1, 4, 8)
         for (d, o, w) in ((True, True, 8), (False, True, -1), (True, False, "S"), (False, False, -1))
         for g in (False, True) if o or not g]

# kernel forms: automatic (the ring from 1024 rows where it fits), one CTA per
# row, the ring
FORMS = {"auto": {}, "rows": dict(kernel=ar.KERNEL_GENERIC), "ring": dict(kernel=ar.KERNEL_STREAM)}


@pytest.mark.parametrize("form", ["ring", "rows"])
@pytest.mark.parametrize("R,S,d,o,w,g", CASES,
                         ids=[f"R{R}_S{S}_d{int(d)}_o{int(o)}_w{w}_g{int(g)}" for R, S, d, o, w, g in CASES])
def test_even_shards(R, S, d, o, w, g, form):
    widx = S if w == "S" else w
    wl = W.make_workload(37, S, capacity=9, has_delta=d, has_out_norm=o, block_write_idx=widx,
                         seed=500 + 10 * R + S, mixing=True)
    widths = [W.HIDDEN // R] * R
    if form == "ring" and not ring_fits(widths[0], S, d, g and o):
        with pytest.raises(ar.AttnResError):   # a forced ring that does not fit is refused
            run_tp_ranks(wl, widths, gram=g, **FORMS[form])
        return
    tp_check(wl, widths, f"tp_R{R}_S{S}_g{int(g)}_{form}", gram=g, **FORMS[form])


def ring_fits(Hs, S, delta, gram, stages=2):
    """Whether every phase's ring of an Hs-wide shard fits the library's 220 KB
    (stages of rows at a 16-byte padded pitch; the Gram sums also hold two
    query rows, 16 bytes and two 16 x 16 fp32 tiles per warp)."""
    rows = S + 1 + int(delta)
    warps = min(-(-Hs // 8 // 32), 128 // 32)
    ring = stages * rows * (Hs * 2 + 16)
    return ring + (4 * Hs + 16 + 2 * warps * 1024 if gram else 0) <= 220 * 1024


@pytest.mark.parametrize("stages", [2, 3, 4])
@pytest.mark.parametrize("gram", [False, True])
def test_ring_wraps(stages, gram):
    """More token rows than resident CTAs: each CTA of the ring form walks
    several tokens and reuses every stage (1500 rows over ~600 CTAs of an
    896-column shard), full oracle comparison, eight shards."""
    wl = W.make_workload(1500, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=900 + stages, mixing=True, outliers=True)
    tp_check(wl, [896] * 8, f"tp_ring{stages}", gram=gram, kernel=ar.KERNEL_STREAM, stages=stages)


@pytest.mark.parametrize("gram", [False, True])
@pytest.mark.parametrize("widths", [[4096, 3072], [8, 7160], [1024] * 7, [2048, 8, 2040, 3072]])
def test_uneven_shards(widths, gram):
    wl = W.make_workload(19, 8, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=3, seed=len(widths), mixing=True, outliers=True)
    tp_check(wl, widths, f"tp_uneven_{len(widths)}", gram=gram)


@pytest.mark.parametrize("form", ["ring", "rows"])
@pytest.mark.parametrize("H,widths", [(64, [8, 56]), (200, [96, 104]), (1024, [256] * 4),
                                     (4096, [2048] * 2), (16384, [4096] * 4), (16384, [16384])])
def test_other_widths(H, widths, form):
    """Any width.  The 16384-wide single shard does not fit a ring (6 rows x
    32 KB x 2 stages > 200 KB): forcing the ring is refused, and at 1100
    rows the automatic form falls back to one CTA per row."""
    wl = W.make_workload(23, 4, capacity=5, has_delta=True, has_out_norm=True,
                         block_write_idx=4, seed=H, H=H, mixing=True, slot_stride=H + 8)
    if form == "ring" and max(widths) == 16384:
        with pytest.raises(ar.AttnResError):
            run_tp_ranks(wl, widths, **FORMS[form])
        wl = W.make_workload(1100, 4, capacity=5, has_delta=True, has_out_norm=True,
                             block_write_idx=4, seed=H, H=H, mixing=True)
        idx = np.sort(np.random.default_rng(5).choice(wl.T, 12, replace=False))
        ref = oracle.run_workload(wl, n_threads=NT, tokens=idx)
        G.check_against_oracle(wl, run_tp_ranks(wl, widths), ref, tokens=idx, tag="tp_wide_auto")
        return
    tp_check(wl, widths, f"tp_H{H}_{form}", **FORMS[form])
    tp_check(wl, widths, f"tp_H{H}_gram_{form}", gram=True, **FORMS[form])


def test_pdl_and_padded_rows():
    wl = W.make_workload(64, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=77, mixing=True, slot_stride=W.HIDDEN + 64)
    gpu, _ = tp_check(wl, [W.HIDDEN // 4] * 4, "tp_pdl_padded", pdl=True, out_row=W.HIDDEN + 16)
    assert np.all(gpu["out_full"][:, W.HIDDEN:] == W.CANARY)


def test_single_rank_matches_unsharded_kernel_bits_for_writebacks():
    """With one rank the three calls and attn_res compute the same c; out may
    differ only by rounding order (within the tolerance of both)."""
    wl = W.make_workload(40, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=9, mixing=True)
    a = run_tp_ranks(wl, [W.HIDDEN])
    b = G.run_gpu(wl)
    assert np.array_equal(a["prefix"], b["prefix"])
    assert np.array_equal(a["bank"], b["bank"])
    G.assert_out_close(a["out"], b["out"], "tp vs unsharded")


def test_zero_tokens():
    import torch

    z = torch.empty((0, 896), dtype=torch.bfloat16, device="cuda")
    bank = torch.empty((0, 8, 896), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(896, dtype=torch.bfloat16, device="cuda")
    out = tp.attn_res_tp(z, z, bank, 8, 2, w, w, w, H=7168, all_reduce=lambda t: None)
    assert out.shape == (0, 896)


@pytest.mark.parametrize("gram", [False, True])
def test_prefill_sharded_sampled(gram):
    """T = 2048, S = 8, eight shards of 896 columns; sampled tokens against the
    oracle."""
    wl = W.prefill(2048, 8, True, 7)
    rng = np.random.default_rng(3)
    idx = np.sort(rng.choice(wl.T, 48, replace=False))
    ref = oracle.run_workload(wl, n_threads=NT, tokens=idx)
    gpu = run_tp_ranks(wl, [896] * 8, gram=gram)
    G.check_against_oracle(wl, gpu, ref, tokens=idx, tag="tp_prefill")


def test_long_prefill_sharded_sampled():
    """The full-size long-prefill workload (T = 8192, 9-slot padded bank,
    write-back into slot 8) over eight shards, single exchange; sampled
    tokens against the oracle."""
    wl = W.long_prefill()
    rng = np.random.default_rng(4)
    idx = np.sort(rng.choice(wl.T, 32, replace=False))
    ref = oracle.run_workload(wl, n_threads=NT, tokens=idx)
    gpu = run_tp_ranks(wl, [896] * 8, gram=True)
    G.check_against_oracle(wl, gpu, ref, tokens=idx, tag="tp_long_prefill")


def test_zero_tokens_gram():
    import torch

    z = torch.empty((0, 896), dtype=torch.bfloat16, device="cuda")
    bank = torch.empty((0, 8, 896), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(896, dtype=torch.bfloat16, device="cuda")
    out = tp.attn_res_tp(z, z, bank, 8, 2, w, w, w, H=7168, all_reduce=lambda t: None, gram=True)
    assert out.shape == (0, 896)


@pytest.mark.parametrize("B,widx,gram", [(2, -1, False), (3, 8, True), (5, 8, False)])
def test_shared_bank_rows(B, widx, gram):
    """B token rows per bank row, over four shards."""
    wl = W.make_workload(23, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=widx, seed=60 + B, mixing=True, group=B)
    tp_check(wl, [W.HIDDEN // 4] * 4, f"tp_group{B}", gram=gram)


@pytest.mark.parametrize("gram,chunk,B", [(False, 16, 1), (True, 16, 1), (False, 12, 3), (True, 7, 1)])
def test_chunked_pipeline(gram, chunk, B):
    """Token chunks, software-pipelined (ragged last chunk), over four shards."""
    wl = W.make_workload(61, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=80 + chunk, mixing=True, group=B)
    tp_check(wl, [W.HIDDEN // 4] * 4, f"tp_chunk{chunk}", gram=gram, chunk=chunk)


def _draw_tp(k: int):
    rng = np.random.default_rng(30_000 + k)
    R = int(rng.choice([1, 2, 3, 4, 8]))
    base = int(rng.choice([8, 64, 896, 1024]))
    widths = [base * int(rng.integers(1, 5)) for _ in range(R)]
    H = sum(widths)
    S = int(rng.integers(0, 9))
    cap = S + int(rng.integers(1, 3)) if S < 8 else 9
    group = int(rng.choice([1, 1, 2]))
    free = list(range(S, cap))
    widx = int(rng.choice([-1] + free + ([] if group > 1 else list(range(S)))))
    T = int(rng.choice([1, 3, 17, 64, 130]))
    chunk = int(rng.choice([0, 0, 2 * group, 8 * group]))
    c = dict(widths=widths, H=H, S=S, cap=cap, group=group, widx=widx, T=T,
             delta=bool(rng.integers(0, 2)), norm=bool(rng.integers(0, 2)),
             gram=bool(rng.integers(0, 2)), pdl=bool(rng.integers(0, 2)),
             chunk=chunk or None, pad=int(rng.choice([0, 8])))
    c["form"] = _draw_form(rng, widths, S, c["delta"])
    return c


def _draw_form(rng, widths, S, delta):
    """Automatic, one CTA per row, or the ring at a depth every shard fits."""
    k = int(rng.integers(0, 4))
    if k == 0:
        return {}
    if k == 1:
        return dict(kernel=ar.KERNEL_GENERIC)
    fit = [st for st in (2, 3, 4) if ring_fits(max(widths), S, delta, True, st)]
    if not fit:
        return dict(kernel=ar.KERNEL_GENERIC)
    return dict(kernel=ar.KERNEL_STREAM, stages=int(rng.choice(fit)))


@pytest.mark.parametrize("k", range(24))
def test_random_sharding(k):
    """Seeded random shardings (rank count, uneven widths, any H), variants,
    shared rows, both exchange forms, PDL and chunking, against the oracle."""
    c = _draw_tp(k)
    wl = W.make_workload(c["T"], c["S"], capacity=c["cap"], has_delta=c["delta"],
                         has_out_norm=c["norm"], block_write_idx=c["widx"], seed=31_000 + k,
                         H=c["H"], mixing=True, slot_stride=c["H"] + c["pad"], group=c["group"])
    tp_check(wl, c["widths"], f"tp_random_{c}", gram=c["gram"], pdl=c["pdl"], chunk=c["chunk"],
             **c["form"])
