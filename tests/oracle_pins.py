"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` build and raises AssertionError when
the build disagrees with the fact.  ``tests/test_oracle_pins.py`` runs them on
the committed oracle; ``tests/test_oracle_mutants.py`` runs them on builds
with planted mistakes and requires that some pin fails for each.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from attention_residual_fusion_gb300 import workloads as W
from tests import restatement as R

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "handworked.json")


def _hex(a):
    return np.array([[int(v, 16) for v in row] for row in a], dtype=np.uint16)


def _rand_bits(rng, shape, scale=1.0):
    return W.f32_to_bf16_bits(scale * rng.standard_normal(shape, dtype=np.float32))


def _case(rng, T, H, S, cap, has_delta, has_norm, widx, mixing=True):
    prefix = _rand_bits(rng, (T, H))
    delta = _rand_bits(rng, (T, H)) if has_delta else None
    blocks = np.full((T, cap, H), W.CANARY, dtype=np.uint16)
    if S:
        blocks[:, :S] = _rand_bits(rng, (T, S, H))
    rms_w = W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(H, dtype=np.float32))
    res_w = W.f32_to_bf16_bits((0.3 if mixing else 1.0) *
                               rng.standard_normal(H, dtype=np.float32)
                               + (0.0 if mixing else 1.0))
    onw = W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(H, dtype=np.float32)) if has_norm else None
    return prefix, delta, blocks, rms_w, res_w, onw


# ---- bf16 conversions ----------------------------------------------------

def pin_bf16_rounding(o):
    """double -> bf16 is round-to-nearest-even (IEEE 754), checked against an
    exhaustive search over all finite bf16 values in exact rationals."""
    rng = np.random.default_rng(11)
    xs = [0.0, -0.0, 1.0, -1.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135,
          2.0 ** -126, 2.0 ** -126 * (1 - 2.0 ** -9), 3.0e38, 3.3895313892515355e38,
          3.3961775292304e38, 3.4e38, 1e39, float("inf"), -float("inf")]
    # exact midpoints between neighbouring bf16 values, and a hair around them
    for b in [0x3F80, 0x3F81, 0x0001, 0x0002, 0x007F, 0x0080, 0x4B00, 0x7F7E, 0x7F7F, 0xBF80]:
        lo = R.widen(np.array([b], np.uint16))[0]
        hi = R.widen(np.array([b + 1], np.uint16))[0]
        mid = (lo + hi) / 2
        xs += [mid, np.nextafter(mid, -np.inf), np.nextafter(mid, np.inf), lo, hi]
    mags = np.exp2(rng.uniform(-140, 129, 400))
    xs += list(mags * np.where(rng.random(400) < 0.5, -1.0, 1.0))
    xs += list(rng.standard_normal(200))
    xs = np.array(xs, dtype=np.float64)
    got = o.round_bf16(xs)
    for x, g in zip(xs, got):
        want = R.bf16_rne_exact(float(x))
        assert int(g) == want, f"round_bf16({x!r}) = {int(g):#06x}, want {want:#06x}"
    assert (int(o.round_bf16(np.array([np.nan]))[0]) & 0x7FFF) > 0x7F80
    # widening is exact: compare with the float32 view of the bits
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    fin = (bits & 0x7F80) != 0x7F80
    wide = o.widen_bf16(bits)
    ref = R.widen(bits)
    assert np.array_equal(wide[fin], ref[fin])


# ---- hand-derived tiny cases --------------------------------------------

def _golden_symbol(s, env):
    return float(eval(s, {"__builtins__": {}}, env))


def pin_golden_handworked(o):
    """Cases whose outputs were derived by hand (tests/golden)."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    env = {"sigmoid": lambda z: 1.0 / (1.0 + math.exp(-z)),
           "a": 1.0 / (2.0 + math.exp(-2.0)),
           "b": math.exp(-2.0) / (2.0 + math.exp(-2.0))}
    for c in cases:
        prefix = _hex(c["prefix"])
        delta = None if c["delta"] is None else _hex(c["delta"])
        blocks = np.stack([_hex(t) for t in c["blocks"]])
        rms_w = _hex([c["rms_w"]])[0]
        res_w = _hex([c["res_w"]])[0]
        onw = None if c["out_norm_w"] is None else _hex([c["out_norm_w"]])[0]
        out, w, _ = o.attn_res(prefix, delta, blocks, c["num_blocks"],
                               c["block_write_idx"], res_w, rms_w, onw,
                               c["eps"], c["out_eps"], want_weights=True)
        assert np.array_equal(out, _hex(c["expect_out"])), (c["name"], out)
        assert np.array_equal(prefix, _hex(c["expect_prefix"])), (c["name"], prefix)
        assert np.array_equal(blocks, np.stack([_hex(t) for t in c["expect_blocks"]])), c["name"]
        ew = np.array([[_golden_symbol(s, env) for s in row] for row in c["expect_weights"]])
        assert np.allclose(w, ew, rtol=1e-12, atol=0), (c["name"], w, ew)


# ---- closed forms and invariants at the full hidden size ------------------

def pin_s0_is_rmsnorm(o):
    """num_blocks = 0: the single candidate gets weight 1, so without output
    norm out == c bit for bit, and with it out is the textbook RMSNorm of c
    times the weight, correctly rounded."""
    rng = np.random.default_rng(1)
    H = W.HIDDEN
    for has_delta in (False, True):
        prefix, delta, blocks, rms_w, res_w, onw = _case(rng, 3, H, 0, 1, has_delta, True, -1)
        c = R.bf16_round_via_f32(R.widen(prefix).astype(np.float32) +
                                 R.widen(delta).astype(np.float32)) if has_delta else prefix.copy()
        out, w, _ = o.attn_res(prefix.copy(), delta, blocks.copy(), 0, -1, res_w,
                               rms_w, None, 1e-6, 1e-6, want_weights=True)
        assert np.array_equal(out, c)
        assert np.all(w == 1.0)
        out = o.attn_res(prefix.copy(), delta, blocks.copy(), 0, -1, res_w, rms_w,
                         onw, 1e-6, 1e-6)
        cf = R.widen(c)
        eps = float(np.float32(1e-6))
        y = cf / np.sqrt(np.mean(cf ** 2, axis=1, keepdims=True) + eps) * R.widen(onw)
        assert np.all(R.is_nearest_bf16(out, y))


def pin_identical_sources(o):
    """All candidates equal to the same row x: every weight is 1/N and the
    output (no output norm) is x bit for bit."""
    rng = np.random.default_rng(2)
    H = W.HIDDEN
    for S in (1, 3, 8):
        prefix, _, _, rms_w, res_w, _ = _case(rng, 2, H, 0, 1, False, False, -1)
        blocks = np.repeat(prefix[:, None, :], S, axis=1).copy()
        out, w, _ = o.attn_res(prefix.copy(), None, blocks, S, -1, res_w, rms_w,
                               None, 1e-6, 1e-6, want_weights=True)
        assert np.array_equal(out, prefix)
        assert np.allclose(w, 1.0 / (S + 1), rtol=1e-14, atol=0)


def pin_weights_sum_to_one(o):
    rng = np.random.default_rng(3)
    for S in range(9):
        prefix, delta, blocks, rms_w, res_w, onw = _case(rng, 4, 256, S, 8, True, True, -1)
        _, w, _ = o.attn_res(prefix, delta, blocks, S, -1, res_w, rms_w, onw,
                             1e-6, 1e-6, want_weights=True)
        assert w.shape == (4, S + 1)
        assert np.all(w >= 0)
        assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-12


def pin_scale_invariance(o):
    """Scaling a candidate by 2^k leaves its logit unchanged: bit-identical
    with eps = 0; with eps > 0 the relative change is below eps divided by
    the smaller of the two mean squares."""
    rng = np.random.default_rng(4)
    H = 512
    S = 4
    prefix, _, blocks, rms_w, res_w, _ = _case(rng, 3, H, S, S, False, False, -1)
    _, _, l0 = o.attn_res(prefix.copy(), None, blocks.copy(), S, -1, res_w, rms_w,
                          None, 0.0, 0.0, want_weights=True)
    _, _, e0 = o.attn_res(prefix.copy(), None, blocks.copy(), S, -1, res_w, rms_w,
                          None, 1e-6, 0.0, want_weights=True)
    for k in (-3, 1, 4):
        b2 = blocks.copy()
        b2[:, 2] = W.f32_to_bf16_bits(R.widen(blocks[:, 2]).astype(np.float32) * np.float32(2.0 ** k))
        _, _, l1 = o.attn_res(prefix.copy(), None, b2, S, -1, res_w, rms_w,
                              None, 0.0, 0.0, want_weights=True)
        assert np.array_equal(l1, l0), (k, l1 - l0)
        _, _, e1 = o.attn_res(prefix.copy(), None, b2.copy(), S, -1, res_w, rms_w,
                              None, 1e-6, 0.0, want_weights=True)
        ms = np.minimum(np.mean(R.widen(blocks[:, 2]) ** 2, axis=1),
                        np.mean(R.widen(b2[:, 2]) ** 2, axis=1))
        rel = np.abs(e1[:, 2] / e0[:, 2] - 1.0)
        assert np.all(rel <= 1e-6 / ms), (k, rel)
        assert np.array_equal(np.delete(e1, 2, axis=1), np.delete(e0, 2, axis=1))


def pin_hard_selection(o):
    """A candidate aligned with q wins by thousands of logit units: the other
    weights underflow and out (no output norm) equals that candidate."""
    rng = np.random.default_rng(5)
    H = W.HIDDEN
    S = 5
    prefix, delta, blocks, rms_w, res_w, _ = _case(rng, 2, H, S, 8, True, False, -1, mixing=False)
    q = R.widen(rms_w) * R.widen(res_w)
    mag = np.abs(R.widen(blocks[:, 3]))
    blocks[:, 3] = W.f32_to_bf16_bits((np.sign(q)[None, :] * mag).astype(np.float32))
    out, w, _ = o.attn_res(prefix, delta, blocks.copy(), S, -1, res_w, rms_w, None,
                           1e-6, 1e-6, want_weights=True)
    assert np.array_equal(out, blocks[:, 3])
    assert np.all(w[:, 3] == 1.0)


def pin_slot_permutation(o):
    """Permuting the valid bank slots permutes the weights and leaves the
    output unchanged (up to one bf16 step from summation order)."""
    rng = np.random.default_rng(6)
    H = 1024
    S = 6
    prefix, delta, blocks, rms_w, res_w, onw = _case(rng, 3, H, S, 8, True, True, -1)
    out0, w0, _ = o.attn_res(prefix.copy(), delta, blocks.copy(), S, -1, res_w,
                             rms_w, onw, 1e-6, 1e-6, want_weights=True)
    perm = np.array([4, 0, 5, 2, 1, 3])
    b2 = blocks.copy()
    b2[:, :S] = blocks[:, perm]
    out1, w1, _ = o.attn_res(prefix.copy(), delta, b2, S, -1, res_w, rms_w, onw,
                             1e-6, 1e-6, want_weights=True)
    assert np.allclose(w1[:, :S], w0[:, perm], rtol=1e-12, atol=1e-300)
    assert np.allclose(w1[:, S], w0[:, S], rtol=1e-12)
    d = np.abs(R.widen(out1) - R.widen(out0))
    assert np.all(d <= R.ulp_bf16(R.widen(out0)))


def pin_two_sources_sigmoid(o):
    """S = 1: weight of the current row is sigmoid(l_c - l_0); at H = 1 the
    logit is x q / sqrt(x^2 + eps)."""
    rng = np.random.default_rng(7)
    prefix, _, blocks, rms_w, res_w, _ = _case(rng, 8, 64, 1, 1, False, False, -1)
    _, w, lg = o.attn_res(prefix, None, blocks, 1, -1, res_w, rms_w, None,
                          1e-6, 1e-6, want_weights=True)
    sig = 1.0 / (1.0 + np.exp(lg[:, 0] - lg[:, 1]))
    assert np.allclose(w[:, 1], sig, rtol=1e-13, atol=1e-300)
    # H = 1 closed form of the logit
    xs = W.f32_to_bf16_bits(np.array([[0.75], [-2.5], [3e-3], [-40.0]], np.float32))
    bs = W.f32_to_bf16_bits(np.array([[[1.5]], [[0.125]], [[-7.0]], [[2.0]]], np.float32))
    rw = W.f32_to_bf16_bits(np.array([1.25], np.float32))
    qw = W.f32_to_bf16_bits(np.array([-0.5], np.float32))
    _, w, lg = o.attn_res(xs.copy(), None, bs.copy(), 1, -1, qw, rw, None, 1e-6, 0.0,
                          want_weights=True)
    eps = float(np.float32(1e-6))
    q = R.widen(rw)[0] * R.widen(qw)[0]
    for t in range(4):
        for i, x in enumerate((R.widen(bs[t, 0])[0], R.widen(xs[t])[0])):
            assert math.isclose(lg[t, i], x * q / math.sqrt(x * x + eps), rel_tol=1e-14)


def pin_bruteforce_tiny_h(o):
    """Against the independent float64 restatement (numpy/scipy) at tiny H,
    every S, delta, output norm and write-back choice."""
    rng = np.random.default_rng(8)
    for H in (1, 2, 8, 16, 64):
        for S in range(9):
            for has_delta in (False, True):
                for has_norm in (False, True):
                    widx = [-1, S if S < 8 else 7, 0][(H + S) % 3]
                    T = 3
                    prefix, delta, blocks, rms_w, res_w, onw = _case(
                        rng, T, H, S, 9, has_delta, has_norm, widx)
                    p0, b0 = prefix.copy(), blocks.copy()
                    # distinct eps and out_eps, so that swapping them shows
                    out, w, lg = o.attn_res(prefix, delta, blocks, S, widx, res_w,
                                            rms_w, onw, 1e-6, 1e-3,
                                            want_weights=True)
                    c, wr, lr, y = R.restate(p0, delta, b0, S, res_w, rms_w, onw,
                                             1e-6, 1e-3)
                    tag = (H, S, has_delta, has_norm, widx)
                    assert np.allclose(w, wr, rtol=1e-10, atol=1e-15), tag
                    assert np.allclose(lg, lr, rtol=1e-10, atol=1e-12), tag
                    assert np.all(R.is_nearest_bf16(out, y, rel_slack=1e-9)), tag
                    assert np.array_equal(prefix, c if has_delta else p0), tag
                    expect = b0.copy()
                    if widx >= 0:
                        expect[:, widx] = c
                    assert np.array_equal(blocks, expect), tag


def pin_writeback_reads_before_write(o):
    """block_write_idx < num_blocks overwrites a source slot: the weights and
    output are those of the untouched inputs, and the slot ends equal to c."""
    rng = np.random.default_rng(9)
    H = 256
    S = 8
    prefix, delta, blocks, rms_w, res_w, onw = _case(rng, 4, H, S, 8, True, True, 7)
    out_a, w_a, _ = o.attn_res(prefix.copy(), delta, blocks.copy(), S, -1, res_w,
                               rms_w, onw, 1e-6, 1e-6, want_weights=True)
    p, b = prefix.copy(), blocks.copy()
    out_b, w_b, _ = o.attn_res(p, delta, b, S, 7, res_w, rms_w, onw, 1e-6, 1e-6,
                               want_weights=True)
    assert np.array_equal(out_a, out_b)
    assert np.array_equal(w_a, w_b)
    assert np.array_equal(b[:, :7], blocks[:, :7])
    assert np.array_equal(b[:, 7], p)


def pin_threads_agree(o):
    """Splitting tokens across threads changes nothing."""
    rng = np.random.default_rng(10)
    prefix, delta, blocks, rms_w, res_w, onw = _case(rng, 37, 128, 5, 8, True, True, 6)
    res = []
    for n in (1, 4, 16):
        p, b = prefix.copy(), blocks.copy()
        out = o.attn_res(p, delta, b, 5, 6, res_w, rms_w, onw, 1e-6, 1e-6, n_threads=n)
        res.append((out, p, b))
    for r in res[1:]:
        for x, y in zip(r, res[0]):
            assert np.array_equal(x, y)


def pin_grouped_bank(o):
    """B token rows per bank row (the excerpt's row index tb / B): the result
    is the float64 restatement applied to the bank with row t / B repeated
    for every token row t; the written slot of each bank row ends holding c
    of the last row of its group; a written slot that is also a source, and
    B < 1, are rejected."""
    rng = np.random.default_rng(12)
    H, S, cap, T = 64, 4, 8, 7
    for B in (2, 3, 7):
        for widx in (-1, 6):
            prefix, delta, _, rms_w, res_w, onw = _case(rng, T, H, S, cap, True, True, widx)
            TB = -(-T // B)
            bank = np.full((TB, cap, H), W.CANARY, dtype=np.uint16)
            bank[:, :S] = _rand_bits(rng, (TB, S, H))
            p0, b0 = prefix.copy(), bank.copy()
            out, w, _ = o.attn_res(prefix, delta, bank, S, widx, res_w, rms_w, onw, 1e-6,
                                   1e-3, want_weights=True, blocks_group=B)
            expanded = b0[np.arange(T) // B]
            c, wr, _, y = R.restate(p0, delta, expanded, S, res_w, rms_w, onw, 1e-6, 1e-3)
            tag = (B, widx)
            assert np.allclose(w, wr, rtol=1e-10, atol=1e-15), tag
            assert np.all(R.is_nearest_bf16(out, y, rel_slack=1e-9)), tag
            assert np.array_equal(prefix, c), tag
            expect = b0.copy()
            if widx >= 0:
                for g in range(TB):
                    expect[g, widx] = c[min(g * B + B - 1, T - 1)]
            assert np.array_equal(bank, expect), tag
    prefix, delta, _, rms_w, res_w, onw = _case(rng, 4, 16, 2, 4, True, True, 1)
    bank = _rand_bits(rng, (2, 4, 16))
    for B, widx in ((2, 1), (0, -1)):
        try:
            o.attn_res(prefix.copy(), delta, bank.copy() if B else bank[:0], 2, widx, res_w,
                       rms_w, onw, 1e-6, 1e-6, blocks_group=B)
        except (ValueError, AssertionError, ZeroDivisionError):
            continue
        raise AssertionError(f"blocks_group={B}, write slot {widx} accepted")


ALL_PINS = [pin_bf16_rounding, pin_golden_handworked, pin_s0_is_rmsnorm,
            pin_identical_sources, pin_weights_sum_to_one, pin_scale_invariance,
            pin_hard_selection, pin_slot_permutation, pin_two_sources_sigmoid,
            pin_bruteforce_tiny_h, pin_writeback_reads_before_write,
            pin_threads_agree, pin_grouped_bank]
