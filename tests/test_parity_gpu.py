"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bar: the updated prefix row and every byte of the bank (written slot, other
slots, padding columns) bit-exact; ``out`` within max(2 bf16 ulp of the
oracle's value, 1e-2) per element; guard zones around every buffer and row
padding untouched.  Sizes span several CTAs and clusters, ragged token
counts, every num_blocks / delta / output-norm / write-back combination, every
split override, PDL on and off, and the full-size workloads (sampled tokens
against the oracle, plus properties checked on every token)."""
import numpy as np
import pytest

import attention_residual_fusion_gb300 as ar
import oracle
from attention_residual_fusion_gb300 import _build
from attention_residual_fusion_gb300 import workloads as W
from tests import gpu_util as G
from tests import restatement as R

pytestmark = pytest.mark.gpu

NT = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    ar.lib()


def full_check(wl, tag="", **kw):
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = G.run_gpu(wl, **kw)
    G.check_against_oracle(wl, gpu, ref, tag=tag or wl.name)
    return gpu, ref


def test_single_token_workload():
    full_check(W.single_token())


# the spec-decode variant matrix: T in {1,4,8} x S in {0,1,4,8} x delta x
# output norm x write-back in {-1, S}
MATRIX = [(T, S, d, o, w) for T in (1, 4, 8) for S in (0, 1, 4, 8)
          for d in (False, True) for o in (False, True) for w in (-1, S)]


@pytest.mark.parametrize("T,S,d,o,w", MATRIX,
                         ids=[f"T{T}_S{S}_d{int(d)}_o{int(o)}_w{w}" for T, S, d, o, w in MATRIX])
def test_variant_matrix(T, S, d, o, w):
    if w == 8:
        # slot 8 does not exist in an 8-slot bank: rejected, nothing written
        wl = W.variant_cell(T, S, d, o, w if w < 8 else -1, seed=T * 100 + S)
        wl.block_write_idx = 8
        with pytest.raises(ar.AttnResError) as e:
            G.run_gpu(wl)
        assert e.value.status == 1
        # companion: a 9-slot bank can take the append at slot 8
        wl = W.variant_cell(T, S, d, o, 8, seed=T * 100 + S, capacity=9)
    else:
        wl = W.variant_cell(T, S, d, o, w, seed=T * 100 + S)
    full_check(wl)


@pytest.mark.parametrize("S", range(9))
@pytest.mark.parametrize("split", [4, 7, 8, 14, 16])
def test_every_num_blocks_and_split_mixing(S, split):
    """res_w ~ 0.02 N(0,1): the softmax spreads over several sources, so a
    mixing error cannot hide behind a one-hot weight vector."""
    wl = W.make_workload(5, S, capacity=9, has_delta=True, has_out_norm=(S % 2 == 0),
                         block_write_idx=(S + 3) % 9 if S != 5 else -1, seed=S,
                         mixing=True, name=f"mixing_S{S}")
    full_check(wl, tag=f"mixing_S{S}_k{split}", split=split)


@pytest.mark.parametrize("T", [2, 3, 37, 113, 1000])
def test_ragged_token_counts(T):
    wl = W.make_workload(T, 6, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=2, seed=T, mixing=True)
    full_check(wl)


def test_padded_rows_and_bank():
    wl = W.make_workload(19, 8, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=5, slot_stride=7232,
                         slot_scale=(1.0, 30.0))
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = G.run_gpu(wl, prefix_row=7168 + 64, out_row=7168 + 8)
    G.check_against_oracle(wl, gpu, ref, tag="padded")


# every kernel form with padded prefix / out rows and padded bank slots
# (kernel, bank rows it is built for, token rows)
PADDED = [(ar.KERNEL_SPLIT, 8, 19), (ar.KERNEL_STREAM, 8, 300), (ar.KERNEL_STAGED, 4, 300),
          (ar.KERNEL_ROW, 2, 300), (ar.KERNEL_ROW_SMEM, 5, 300), (ar.KERNEL_GENERIC, 8, 19)]


@pytest.mark.parametrize("kernel,S,T", PADDED, ids=[f"k{k}_S{S}" for k, S, _ in PADDED])
def test_padded_rows_and_bank_every_kernel(kernel, S, T):
    wl = W.make_workload(T, S, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=6 + S, slot_stride=7232, mixing=True,
                         slot_scale=(1.0, 30.0))
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = G.run_gpu(wl, prefix_row=7168 + 64, out_row=7168 + 8, kernel=kernel)
    G.check_against_oracle(wl, gpu, ref, tag=f"padded_k{kernel}")


def test_pdl_launch():
    import torch
    wl = W.make_workload(16, 8, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=7, seed=3, mixing=True)
    full_check(wl, tag="pdl", pdl=True)
    # a producer kernel right before the PDL launch writes delta; the result
    # must reflect the new delta
    ref_wl = wl.copy()
    ref_wl.delta = W.f32_to_bf16_bits(np.full((wl.T, wl.H), 0.25, np.float32))
    ref = oracle.run_workload(ref_wl, n_threads=NT)
    dev = {k: torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)
           for k, v in dict(prefix=wl.prefix, delta=wl.delta, bank=wl.bank, rms=wl.rms_w,
                            res=wl.res_w, onw=wl.out_norm_w).items()}
    out = torch.empty_like(dev["prefix"])
    dev["delta"].fill_(0.25)
    ar.attn_res(dev["prefix"], dev["delta"], dev["bank"], 8, 7, dev["res"], dev["rms"],
                dev["onw"], 1e-6, 1e-6, out, pdl=True)
    torch.cuda.synchronize()
    h = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    G.assert_out_close(h(out), ref["out"], "pdl-producer")
    assert np.array_equal(h(dev["prefix"]), ref["prefix"])
    assert np.array_equal(h(dev["bank"]), ref["bank"])


def test_s0_closed_form_and_identical_sources():
    """Closed forms checked on the GPU directly: S=0 without output norm
    returns c bit for bit; identical sources return the source bit for bit."""
    wl = W.make_workload(9, 0, capacity=1, has_delta=True, has_out_norm=False, seed=4)
    gpu = G.run_gpu(wl)
    c = R.bf16_round_via_f32(R.widen(wl.prefix).astype(np.float32) +
                             R.widen(wl.delta).astype(np.float32))
    assert np.array_equal(gpu["out"], c)
    assert np.array_equal(gpu["prefix"], c)
    wl = W.make_workload(6, 8, capacity=8, has_delta=False, has_out_norm=False, seed=6)
    wl.bank[:, :8, :] = wl.prefix[:, None, :]
    gpu = G.run_gpu(wl)
    assert np.array_equal(gpu["out"], wl.prefix)


def test_zero_tokens():
    import torch
    z = torch.empty((0, 7168), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((0, 8, 7168), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(7168, dtype=torch.bfloat16, device="cuda")
    out = ar.attn_res(z, z.clone(), b, 4, -1, w, w, w)
    assert out.shape == (0, 7168)


@pytest.mark.parametrize("T", [64, 256])
def test_decode_batch(T):
    full_check(W.decode_batch(T))


PREFILL = [(T, S, o, w) for T in (1024, 2048) for S in (0, 4, 8) for o in (False, True)
           for w in (-1, 7)]


@pytest.mark.parametrize("T,S,o,w", PREFILL, ids=[f"T{T}_S{S}_o{int(o)}_w{w}" for T, S, o, w in PREFILL])
def test_prefill(T, S, o, w):
    if w == 7 and S == 0:
        pass  # slot 7 is a pure append target here
    full_check(W.prefill(T, S, o, w))


def test_long_prefill_full_size():
    """T=8192, 9-slot bank with slot stride 7232, write-back into slot 8.
    Sampled tokens against the oracle; on every token: slot 8 == updated
    prefix == bf16(prefix + delta), slots 0..7 and the padding untouched,
    outputs finite."""
    wl = W.long_prefill()
    gpu = G.run_gpu(wl)
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([[0, 1, wl.T - 1], rng.choice(wl.T, 61, replace=False)]))
    ref = oracle.run_workload(wl, n_threads=NT, tokens=tokens)
    G.check_against_oracle(wl, gpu, ref, tokens=tokens, tag="long_prefill")
    c = R.bf16_round_via_f32(R.widen(wl.prefix).astype(np.float32) +
                             R.widen(wl.delta).astype(np.float32))
    assert np.array_equal(gpu["prefix"], c)
    assert np.array_equal(gpu["bank"][:, 8, :wl.H], c)
    assert np.array_equal(gpu["bank"][:, :8], wl.bank[:, :8])
    assert np.all(gpu["bank"][:, 8, wl.H:] == W.CANARY)
    assert np.all(np.isfinite(R.widen(gpu["out"][:: 64])))


def test_repeated_calls_are_deterministic():
    import torch
    wl = W.make_workload(33, 8, capacity=8, has_delta=False, has_out_norm=True,
                         block_write_idx=-1, seed=9, mixing=True)
    a = G.run_gpu(wl)["out"]
    b = G.run_gpu(wl)["out"]
    assert np.array_equal(a, b)


# ---- the persistent stream kernel ------------------------------------------------

SHAPES = [(7, 1, 2), (7, 2, 2), (7, 2, 3), (7, 4, 2), (4, 2, 2), (4, 2, 3), (2, 4, 2), (14, 2, 2),
          (2, 8, 2)]
STREAM = [(S, sh) for S in range(9) for sh in SHAPES]


@pytest.mark.parametrize("S,shape", STREAM, ids=[f"S{S}_k{k}_v{v}_st{st}" for S, (k, v, st) in STREAM])
def test_stream_kernel(S, shape):
    """Every num_blocks x stream shape (split, vectors per thread, ring
    depth); T = 300 gives each persistent cluster several tokens, so every
    stage and mailbox is reused with both parities."""
    k, v, st = shape
    i = S * 8 + SHAPES.index(shape)
    d, o = bool(i & 1), bool(i & 2)
    w = [-1, S, 8][i % 3]
    wl = W.make_workload(300, S, capacity=9, has_delta=d, has_out_norm=o,
                         block_write_idx=w, seed=i, mixing=True,
                         slot_stride=7168 + 8 * (i % 2))
    full_check(wl, tag=f"stream_S{S}_k{k}_v{v}_st{st}_d{int(d)}_o{int(o)}_w{w}",
               kernel=ar.KERNEL_STREAM, split=k, vpt=v, stages=st)


# staged shapes: (split, vectors per thread, CTAs per SM); the ring depth is
# what fits in shared memory for the stage's rows (bank rows, prefix, delta)
STAGED = [(4, 4, 5), (7, 4, 7), (4, 4, 4)]
STAGED_CASES = [(S, sh) for S in range(9) for sh in STAGED]


def staged_depth(S, has_delta, shape):
    """Ring depth of a staged shape: stages of (S + 1 + delta) row slices of
    14336 / split bytes in an SM's 228 KB shared by `ctas_per_sm` CTAs, each
    also holding its mailboxes, 8 stage barrier pairs and 1 KB of system
    reserve, within 227 KB per CTA; at most 8 stages."""
    k, v, cps = shape
    nw = (896 // k // v + 31) // 32
    static = 2 * k * nw * 2 * (S + 1) * 4 + 2 * k * nw * 4 + 32 + 16 * 8
    budget = min(233472 // cps - 1024 - static, 232448 - static)
    return min(8, budget // ((S + (2 if has_delta else 1)) * (14336 // k)))


@pytest.mark.parametrize("S,shape", STAGED_CASES,
                         ids=[f"S{S}_k{k}_v{v}_c{c}" for S, (k, v, c) in STAGED_CASES])
def test_staged_kernel(S, shape):
    """Every num_blocks x staged shape: 2500 tokens, so each CTA reuses
    every stage of even the deepest ring; shapes whose ring cannot hold two
    stages of the rows are refused."""
    k, v, c = shape
    i = S * len(STAGED) + STAGED.index(shape)
    d, o = bool(i & 1), bool(i & 2)
    w = [-1, S, 8][i % 3]
    wl = W.make_workload(2500, S, capacity=9, has_delta=d, has_out_norm=o,
                         block_write_idx=w, seed=100 + i, mixing=True,
                         slot_stride=7168 + 8 * (i % 2))
    if staged_depth(S, d, shape) < 2:
        with pytest.raises(ar.AttnResError) as e:
            G.run_gpu(wl, kernel=ar.KERNEL_STAGED, split=k, vpt=v, stages=c)
        assert e.value.status == 1
        return
    full_check(wl, tag=f"staged_S{S}_k{k}_v{v}_c{c}_d{int(d)}_o{int(o)}_w{w}",
               kernel=ar.KERNEL_STAGED, split=k, vpt=v, stages=c)


# ---- the row kernel (one CTA per token row) ----------------------------------------

ROW_VPTS = (4, 7)
ROW_CASES = [(S, v, d, o) for S in range(3) for v in ROW_VPTS for d in (False, True)
             for o in (False, True)]


@pytest.mark.parametrize("S,vpt,d,o", ROW_CASES,
                         ids=[f"S{S}_v{v}_d{int(d)}_o{int(o)}" for S, v, d, o in ROW_CASES])
def test_row_kernel(S, vpt, d, o):
    """Every num_blocks x vectors per thread x delta x output norm of the row
    kernel, with the write-back slot (a source, the append slot or none) and
    padded bank slots varying by case."""
    i = ROW_CASES.index((S, vpt, d, o))
    w = [-1, S, 8][i % 3]
    wl = W.make_workload(300, S, capacity=9, has_delta=d, has_out_norm=o,
                         block_write_idx=w, seed=200 + i, mixing=True,
                         slot_stride=7168 + 8 * (i % 2))
    full_check(wl, tag=f"row_S{S}_v{vpt}_d{int(d)}_o{int(o)}_w{w}", kernel=ar.KERNEL_ROW, vpt=vpt)


ROW_SMEM_CASES = [(S, v, d, o) for S in range(1, 9) for v in ROW_VPTS for d in (False, True)
                  for o in (False, True)]


@pytest.mark.parametrize("S,vpt,d,o", ROW_SMEM_CASES,
                         ids=[f"S{S}_v{v}_d{int(d)}_o{int(o)}" for S, v, d, o in ROW_SMEM_CASES])
def test_row_smem_kernel(S, vpt, d, o):
    """The row kernel with its rows in shared memory: 1..8 bank rows x
    vectors per thread x delta x output norm, write-back slot and padded
    bank slots varying by case."""
    i = ROW_SMEM_CASES.index((S, vpt, d, o))
    w = [-1, S, 8][i % 3]
    wl = W.make_workload(300, S, capacity=9, has_delta=d, has_out_norm=o,
                         block_write_idx=w, seed=300 + i, mixing=True,
                         slot_stride=7168 + 8 * (i % 2))
    full_check(wl, tag=f"row_smem_S{S}_v{vpt}_d{int(d)}_o{int(o)}_w{w}",
               kernel=ar.KERNEL_ROW_SMEM, vpt=vpt)


@pytest.mark.parametrize("S,vpt", [(3, 7), (8, 4), (0, 2), (1, 1)])
def test_row_kernel_refuses_unbuilt_shapes(S, vpt):
    """The row kernel is built for up to two bank rows and 4 or 7 vectors per
    thread; anything else is refused before a launch."""
    wl = W.make_workload(4, S, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=-1, seed=3)
    with pytest.raises(ar.AttnResError) as e:
        G.run_gpu(wl, kernel=ar.KERNEL_ROW, vpt=vpt)
    assert e.value.status == 1


@pytest.mark.parametrize("T", [1, 2, 7, 1500])
def test_stream_kernel_token_counts(T):
    """Fewer tokens than clusters, and many tokens per cluster."""
    wl = W.make_workload(T, 8, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=3, seed=T, mixing=True)
    full_check(wl, kernel=ar.KERNEL_STREAM)
    full_check(wl, kernel=ar.KERNEL_STREAM, split=7, vpt=1, pdl=True)


def test_split_kernel_at_prefill_size():
    full_check(W.prefill(1024, 8, True, 7), kernel=ar.KERNEL_SPLIT)


def test_zz_device_status_clean():
    """No kernel recorded a stage-wait time-out during the tests above."""
    assert ar.device_status() == 0


@pytest.mark.parametrize("kernel", [ar.KERNEL_SPLIT, ar.KERNEL_STREAM, ar.KERNEL_ROW])
def test_subnormal_current_row_is_correctly_rounded(kernel):
    """c = bf16_rn(prefix + delta) must keep bf16 subnormals (no flush to
    zero) and round ties to even, in both kernels: prefix and delta drawn
    from subnormal and tiny normal bf16 values, S = 0 and no output norm, so
    out == c bit for bit."""
    rng = np.random.default_rng(12)
    T = 130
    wl = W.make_workload(T, 0, capacity=1, has_delta=True, has_out_norm=False,
                         block_write_idx=0, seed=12)
    mag = rng.integers(1, 0x0100, size=(T, wl.H)).astype(np.uint16)  # subnormals and the smallest normals
    sign = (rng.random((T, wl.H)) < 0.5).astype(np.uint16) << 15
    wl.prefix = mag | sign
    mag = rng.integers(1, 0x0100, size=(T, wl.H)).astype(np.uint16)
    sign = (rng.random((T, wl.H)) < 0.5).astype(np.uint16) << 15
    wl.delta = mag | sign
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = G.run_gpu(wl, kernel=kernel)
    assert np.array_equal(gpu["prefix"], ref["prefix"])
    assert np.array_equal(gpu["bank"], ref["bank"])
    assert np.array_equal(gpu["out"], ref["out"])


@pytest.mark.parametrize("T", [1, 300])
def test_pdl_chain_in_graph(T):
    """Three dependent calls captured in a CUDA graph with programmatic
    dependent launch: each call updates prefix in place and the next reads it
    after its grid-dependency wait.  Equal to applying the oracle three
    times."""
    import torch
    wl = W.make_workload(T, 6, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=-1, seed=30 + T, mixing=True)
    ref_wl = wl.copy()
    for _ in range(3):
        r = oracle.run_workload(ref_wl, n_threads=NT)
        ref_wl.prefix = r["prefix"]
    up = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    down = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    d = dict(prefix=up(wl.prefix), delta=up(wl.delta), bank=up(wl.bank), rms=up(wl.rms_w),
             res=up(wl.res_w), onw=up(wl.out_norm_w))
    out = torch.empty_like(d["prefix"])
    s = torch.cuda.Stream()
    args = (d["prefix"], d["delta"], d["bank"], 6, -1, d["res"], d["rms"], d["onw"], 1e-6, 1e-6, out)
    ar.attn_res(*args, pdl=True, stream=s)   # one-time set-up outside capture
    torch.cuda.synchronize()
    d["prefix"].copy_(up(wl.prefix))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            ar.attn_res(*args, pdl=True, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(down(d["prefix"]), r["prefix"])
    G.assert_out_close(down(out), r["out"], "pdl-chain")



@pytest.mark.parametrize("T", [1, 300, 1024])
def test_pdl_chain_with_bank_writes_in_graph(T):
    """A chain captured in a CUDA graph in which one call writes a bank slot
    that a later call reads as a source: call 1 (PDL) appends c to slot 2, a
    plain kernel launched without PDL follows, then call 2 (PDL) mixes slots
    0..2 and the prefix call 1 updated.  Call 2 reads its bank rows before
    its grid-dependency wait, so the plain kernel between them is what the
    PDL contract asks for (no grid that may still be running when a PDL call
    starts writes the rows it reads).  Equal to the oracle applied twice in
    sequence.  Two bank rows then three: the row, shared-memory row and
    staged kernels at 300 and 1024 rows, the split kernel at one."""
    import torch
    wl1 = W.make_workload(T, 2, capacity=8, has_delta=True, has_out_norm=True,
                          block_write_idx=2, seed=50 + T, mixing=True)
    r1 = oracle.run_workload(wl1, n_threads=NT)
    wl2 = wl1.copy()
    wl2.prefix, wl2.bank = r1["prefix"], r1["bank"]
    wl2.num_blocks, wl2.block_write_idx = 3, -1
    wl2.delta = W.make_workload(T, 0, capacity=1, has_delta=True, has_out_norm=False,
                                block_write_idx=-1, seed=90 + T).delta
    r2 = oracle.run_workload(wl2, n_threads=NT)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    down = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    d = dict(prefix=up(wl1.prefix), d1=up(wl1.delta), d2=up(wl2.delta), bank=up(wl1.bank),
             rms=up(wl1.rms_w), res=up(wl1.res_w), onw=up(wl1.out_norm_w))
    out1, out2 = torch.empty_like(d["prefix"]), torch.empty_like(d["prefix"])
    pad = torch.zeros(1 << 16, device="cuda")
    s = torch.cuda.Stream()
    a1 = (d["prefix"], d["d1"], d["bank"], 2, 2, d["res"], d["rms"], d["onw"], 1e-6, 1e-6, out1)
    a2 = (d["prefix"], d["d2"], d["bank"], 3, -1, d["res"], d["rms"], d["onw"], 1e-6, 1e-6, out2)
    ar.attn_res(*a1, pdl=True, stream=s)   # one-time set-up outside capture
    ar.attn_res(*a2, pdl=True, stream=s)
    torch.cuda.synchronize()
    d["prefix"].copy_(up(wl1.prefix))
    d["bank"].copy_(up(wl1.bank))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ar.attn_res(*a1, pdl=True, stream=s)
        pad.add_(1.0)                        # a kernel launched without PDL
        ar.attn_res(*a2, pdl=True, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(down(d["prefix"]), r2["prefix"])
    assert np.array_equal(down(d["bank"]), r2["bank"])
    G.assert_out_close(down(out1), r1["out"], "pdl-write-chain call 1")
    G.assert_out_close(down(out2), r2["out"], "pdl-write-chain call 2")


# ---- the general kernel (any H, multiple of 8) -----------------------------------

GEN = [(H, S) for H in (8, 16, 64, 200, 1024, 4096) for S in (0, 1, 3, 8)]


@pytest.mark.parametrize("H,S", GEN, ids=[f"H{H}_S{S}" for H, S in GEN])
def test_generic_width_against_oracle(H, S):
    """Brute force at small and odd widths: every element against the oracle,
    with delta, output norm and a write-back varying by case."""
    i = H + S
    wl = W.make_workload(37, S, capacity=9, has_delta=bool(i & 1), has_out_norm=bool(i & 2),
                         block_write_idx=[-1, S, 8][i % 3], seed=i, H=H, mixing=True,
                         slot_stride=H + 8 * (i % 2))
    full_check(wl, tag=f"generic_H{H}_S{S}", kernel=ar.KERNEL_GENERIC)
    full_check(wl, tag=f"auto_H{H}_S{S}")


@pytest.mark.parametrize("S", [0, 4, 8])
def test_generic_kernel_forced_at_full_width(S):
    wl = W.make_workload(33, S, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=40 + S, mixing=True)
    full_check(wl, tag=f"generic_forced_S{S}", kernel=ar.KERNEL_GENERIC)


# B token rows per bank row (bank row t // B): every kernel, ragged last
# group, write-back into a slot that is not a source (the group's last row
# writes it), and the rejection of a written source slot.
GROUPED = [(B, T, S, w, k) for B in (2, 3, 8) for (T, S, w) in ((5, 4, -1), (37, 8, 8), (300, 8, 8),
                                                                 (300, 0, 2), (37, 1, 5))
           for k in (ar.KERNEL_SPLIT, ar.KERNEL_STREAM, ar.KERNEL_GENERIC, ar.KERNEL_ROW,
                     ar.KERNEL_ROW_SMEM)
           # the row kernels are built for up to two (registers) and 1..8 bank
           # rows (shared memory)
           if (k != ar.KERNEL_ROW or S <= 2) and (k != ar.KERNEL_ROW_SMEM or S >= 1)]


@pytest.mark.parametrize("B,T,S,w,kernel", GROUPED,
                         ids=[f"B{B}_T{T}_S{S}_w{w}_k{k}" for B, T, S, w, k in GROUPED])
def test_shared_bank_rows(B, T, S, w, kernel):
    wl = W.make_workload(T, S, capacity=9, has_delta=bool(T % 2), has_out_norm=True,
                         block_write_idx=w, seed=70 + B + S, mixing=True, group=B)
    full_check(wl, tag=f"group{B}_T{T}_S{S}", kernel=kernel)


def test_shared_bank_rows_reject_written_source():
    wl = W.make_workload(6, 4, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=2, seed=1, group=2)
    with pytest.raises(ar.AttnResError) as e:
        G.run_gpu(wl)
    assert e.value.status == 1


def _nan_equal(a, b):
    """Bit-equal, except that any NaN pattern matches any NaN pattern."""
    fa, fb = R.widen(a), R.widen(b)
    both_nan = np.isnan(fa) & np.isnan(fb)
    return bool(np.all((a == b) | both_nan))


# (kernel, bank rows it is built for, the two bank slots that get a NaN and an
# infinity)
NONFINITE = [(ar.KERNEL_SPLIT, 8, 2, 5), (ar.KERNEL_STREAM, 8, 2, 5), (ar.KERNEL_GENERIC, 8, 2, 5),
             (ar.KERNEL_ROW, 2, 1, 0), (ar.KERNEL_ROW_SMEM, 5, 2, 4), (ar.KERNEL_STAGED, 4, 2, 3)]


@pytest.mark.parametrize("kernel,S,nan_slot,inf_slot", NONFINITE,
                         ids=[f"k{k}_S{S}" for k, S, _, _ in NONFINITE])
def test_nonfinite_inputs_stay_in_their_token(kernel, S, nan_slot, inf_slot):
    """A NaN or an infinity in one token's rows makes that token's output NaN
    (IEEE arithmetic, as in the oracle) and leaves every other token as the
    oracle computes it; write-backs stay exact (NaN for NaN)."""
    wl = W.make_workload(37, S, capacity=9, has_delta=True, has_out_norm=True,
                         block_write_idx=8, seed=44, mixing=True)
    nan, inf = np.uint16(0x7FC0), np.uint16(0x7F80)
    wl.bank[3, nan_slot, 100] = nan   # a bank row of token 3
    wl.bank[7, inf_slot, 50] = inf    # an infinite bank element of token 7
    wl.delta[11, 4000] = nan          # c of token 11 is NaN in one column
    wl.prefix[20, 7] = inf            # c of token 20 is infinite in one column
    ref = oracle.run_workload(wl, n_threads=NT)
    gpu = G.run_gpu(wl, kernel=kernel)
    bad = [3, 7, 11, 20]
    rest = np.array([t for t in range(wl.T) if t not in bad])
    G.assert_out_close(gpu["out"][rest], ref["out"][rest], "finite tokens")
    for t in bad:
        assert np.all(np.isnan(R.widen(ref["out"][t]))), t
        assert np.all(np.isnan(R.widen(gpu["out"][t]))), t
    assert _nan_equal(gpu["prefix"], ref["prefix"][:, :wl.H])
    assert _nan_equal(gpu["bank"], ref["bank"])



# ---- other widths on the stream kernel (H a multiple of 1024) ---------------------

ANYW = [(H, S) for H in (1024, 2048, 3072, 4096, 8192, 16384) for S in (0, 4, 8)]


@pytest.mark.parametrize("H,S", ANYW, ids=[f"H{H}_S{S}" for H, S in ANYW])
def test_any_width_stream(H, S):
    """H / 1024 CTAs per token row; ragged token count over the clusters,
    padded bank slots, delta / write-back varying by case; automatic choice
    (T >= 80 with bank rows or an output norm streams)."""
    i = H // 1024 + S
    wl = W.make_workload(131, S, capacity=9, has_delta=bool(i & 1), has_out_norm=True,
                         block_write_idx=[-1, S, 8][i % 3],
                         seed=900 + i, H=H, mixing=True, slot_stride=H + 8 * (i % 2))
    full_check(wl, tag=f"anywidth_H{H}_S{S}")


@pytest.mark.parametrize("H", [2048, 12288])
def test_any_width_stream_forced_small_T_and_groups(H):
    """Forced at few tokens (more clusters than tokens), no output norm, and
    with shared bank rows (B = 3)."""
    wl = W.make_workload(5, 8, capacity=9, has_delta=True, has_out_norm=False,
                         block_write_idx=8, seed=H, H=H, mixing=True)
    full_check(wl, tag=f"anywidth_forced_H{H}", kernel=ar.KERNEL_STREAM)
    wl = W.make_workload(200, 6, capacity=8, has_delta=True, has_out_norm=True,
                         block_write_idx=7, seed=H + 1, H=H, mixing=True, group=3)
    full_check(wl, tag=f"anywidth_group_H{H}")



# ---- any-width forms at widths that are not multiples of 1024 ----------------------

RAGGED = [(H, S) for H in (8, 200, 1000, 1032, 3000, 7000, 8200, 15000, 16376) for S in (0, 4, 8)]


@pytest.mark.parametrize("H,S", RAGGED, ids=[f"H{H}_S{S}" for H, S in RAGGED])
def test_ragged_width_fast_kernels(H, S):
    """ceil(H / 1024) CTAs per token row, the last one owning the remainder
    (8 .. 1016 columns; its bank-row copies are that short): the stream form
    at 131 rows (forced and automatic), the split form at 5 rows (up to 8
    CTAs); delta, write-back and padded slots varying by case."""
    i = H + S
    kc = -(-H // 1024)
    wl = W.make_workload(131, S, capacity=9, has_delta=bool(i & 1), has_out_norm=True,
                         block_write_idx=[-1, S, 8][i % 3], seed=7000 + i, H=H, mixing=True,
                         slot_stride=H + 8 * (i % 2), outliers=bool(i & 2))
    full_check(wl, tag=f"ragged_stream_H{H}_S{S}", kernel=ar.KERNEL_STREAM)
    full_check(wl, tag=f"ragged_auto_H{H}_S{S}")
    wl = W.make_workload(5, S, capacity=9, has_delta=not (i & 1), has_out_norm=bool(S % 2) or S == 0,
                         block_write_idx=[8, -1, S][i % 3], seed=7100 + i, H=H, mixing=True)
    full_check(wl, tag=f"ragged_small_auto_H{H}_S{S}")
    if kc <= 8:
        full_check(wl, tag=f"ragged_split_H{H}_S{S}", kernel=ar.KERNEL_SPLIT)


SMALLW = [(H, T, S) for H in (1024, 3072, 8192, 12288) for T in (1, 5, 79) for S in (1, 8)]


@pytest.mark.parametrize("H,T,S", SMALLW, ids=[f"H{H}_T{T}_S{S}" for H, T, S in SMALLW])
def test_any_width_few_tokens(H, T, S):
    """Few tokens at other widths: the split kernel's any-width form (up to 8
    CTAs per row), the stream kernel's above that."""
    wl = W.make_workload(T, S, capacity=9, has_delta=bool(T % 2), has_out_norm=bool(S % 2) or T == 5,
                         block_write_idx=8 if T != 79 else S - 1, seed=H + T + S, H=H, mixing=True)
    full_check(wl, tag=f"anywidth_small_H{H}_T{T}_S{S}")
    if H <= 8192:
        full_check(wl, tag=f"anywidth_small_split_H{H}_T{T}_S{S}", kernel=ar.KERNEL_SPLIT)
