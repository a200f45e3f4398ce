"""Pins for the layer around the recurrence that the fused decode folds in:
the short causal convolution with its state, the L2 normalisation of q and k,
the output RMSNorm with its sigmoid gate, and their composition with the pool
semantics (``oracle.prefill_fused_pool`` / ``oracle.decode_fused_pool``).

Each part is checked against something other than its own code: numpy's
convolution (a library routine), shift and identity kernels, closed forms of
the norm (a constant row, a saturated gate, scale invariance), a two-element
example worked by hand, and split invariance of the composed prefill (the
convolution state and the matrix state handed over together)."""

import numpy as np
import pytest
import scipy.special
import torch

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ short conv

@pytest.mark.parametrize("W", [2, 3, 4])
def test_conv_matches_numpy_convolve(W):
    """y[t, c] = sum_i w[c, i] xx[t + i, c] is numpy's 'valid' convolution of
    the history-extended input with the reversed taps, channel by channel."""
    rng = _rng(W)
    L, C = 11, 5
    x = rng.standard_normal((L, C))
    prev = rng.standard_normal((W - 1, C))
    w = rng.standard_normal((C, W))
    y, st = oracle.short_conv(x, w, prev)
    xx = np.concatenate([prev, x])
    for c in range(C):
        ref = np.convolve(xx[:, c], w[c, ::-1], mode="valid")
        np.testing.assert_allclose(y[:, c], ref, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(st, xx[-(W - 1):])


def test_conv_current_tap_is_identity_and_oldest_tap_is_a_shift():
    rng = _rng(1)
    L, C, W = 7, 3, 4
    x = rng.standard_normal((L, C))
    prev = rng.standard_normal((W - 1, C))
    cur = np.zeros((C, W)); cur[:, W - 1] = 1.0
    y, _ = oracle.short_conv(x, cur, prev)
    np.testing.assert_array_equal(y, x)
    old = np.zeros((C, W)); old[:, 0] = 1.0
    y, _ = oracle.short_conv(x, old, prev)
    np.testing.assert_array_equal(y[:W - 1], prev)        # the state feeds the first tokens
    np.testing.assert_array_equal(y[W - 1:], x[:L - (W - 1)])


def test_conv_without_state_starts_from_zeros_and_state_of_a_short_segment():
    """No state means zero history; a segment shorter than W - 1 shifts the old
    state by its length (new state = last W-1 of [old state; x])."""
    rng = _rng(2)
    C, W = 4, 4
    x = rng.standard_normal((2, C))
    w = rng.standard_normal((C, W))
    y0, _ = oracle.short_conv(x, w, None)
    y1, _ = oracle.short_conv(x, w, np.zeros((W - 1, C)))
    np.testing.assert_array_equal(y0, y1)
    prev = rng.standard_normal((W - 1, C))
    _, st = oracle.short_conv(x, w, prev)
    np.testing.assert_array_equal(st, np.concatenate([prev[2:], x]))


def test_conv_split_invariance():
    rng = _rng(3)
    C, W = 6, 4
    x = rng.standard_normal((19, C))
    w = rng.standard_normal((C, W))
    prev = rng.standard_normal((W - 1, C))
    y, st = oracle.short_conv(x, w, prev)
    for cut in (1, 2, 3, 8):
        ya, sa = oracle.short_conv(x[:cut], w, prev)
        yb, sb = oracle.short_conv(x[cut:], w, sa)
        np.testing.assert_allclose(np.concatenate([ya, yb]), y, rtol=0, atol=1e-14)
        np.testing.assert_array_equal(sb, st)


def test_conv_silu_is_the_logistic_times_the_linear_output():
    rng = _rng(4)
    x = rng.standard_normal((9, 3))
    w = rng.standard_normal((3, 4))
    lin, _ = oracle.short_conv(x, w, None)
    y, _ = oracle.short_conv(x, w, None, act="silu")
    np.testing.assert_allclose(y, lin * scipy.special.expit(lin), rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------ norms

def test_l2_normalize_unit_rows_same_direction():
    rng = _rng(5)
    x = rng.standard_normal((6, 16)) * 3.0
    y = oracle.l2_normalize(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=1, keepdims=True), x, rtol=1e-14)


def test_rms_norm_gated_hand_worked():
    """o = (3, 4): mean square 12.5, rms 5 / sqrt(2); w = (1, 2);
    gate = (0, ln 3): sigmoid = (1/2, 3/4).  With eps = 0:
    y = (3 sqrt2/5 * 1 * 1/2, 4 sqrt2/5 * 2 * 3/4) = (0.3 sqrt2, 1.2 sqrt2)."""
    y = oracle.rms_norm_gated(np.array([3.0, 4.0]), np.array([1.0, 2.0]),
                              np.array([0.0, np.log(3.0)]), eps=0.0)
    np.testing.assert_allclose(y, [0.3 * np.sqrt(2.0), 1.2 * np.sqrt(2.0)], rtol=1e-14)


def test_rms_norm_gated_closed_forms():
    rng = _rng(6)
    dv = 16
    w = rng.standard_normal(dv)
    gate = rng.standard_normal(dv)
    # a constant row c: RMSNorm gives sign(c)
    for c in (2.5, -0.75):
        y = oracle.rms_norm_gated(np.full(dv, c), w, gate, eps=0.0)
        np.testing.assert_allclose(y, np.sign(c) * w * scipy.special.expit(gate), rtol=1e-14)
    o = rng.standard_normal(dv)
    # a saturated gate: the plain norm (unit mean square once w is divided out)
    y = oracle.rms_norm_gated(o, np.ones(dv), np.full(dv, 60.0), eps=0.0)
    np.testing.assert_allclose(np.mean(y * y), 1.0, rtol=1e-12)
    # a closed gate: nothing passes
    assert np.max(np.abs(oracle.rms_norm_gated(o, w, np.full(dv, -60.0)))) < 1e-20
    # scale invariance without epsilon; epsilon only shrinks
    np.testing.assert_allclose(oracle.rms_norm_gated(7.0 * o, w, gate, eps=0.0),
                               oracle.rms_norm_gated(o, w, gate, eps=0.0), rtol=1e-13)
    assert np.all(np.abs(oracle.rms_norm_gated(o, w, gate)) <=
                  np.abs(oracle.rms_norm_gated(o, w, gate, eps=0.0)) + 1e-15)


# ------------------------------------------------------------------ composition

def _fused_case(seed, lens, H=2, dk=8, dv=8, n_slots=6):
    rng = _rng(seed)
    T = sum(lens)
    C = 2 * dk + dv
    xq = rng.standard_normal((T, H, dk))
    xk = rng.standard_normal((T, H, dk))
    xv = rng.standard_normal((T, H, dv))
    g = -np.exp(rng.standard_normal((T, H, dk)) - 3.0)
    beta = scipy.special.expit(rng.standard_normal((T, H)))
    gate = rng.standard_normal((T, H, dv))
    conv_w = rng.standard_normal((H, C, oracle.CONV_WIDTH)) * 0.5
    norm_w = 1.0 + 0.1 * rng.standard_normal(dv)
    pool = 0.1 * rng.standard_normal((n_slots, H, dk, dv))
    cpool = rng.standard_normal((n_slots, H, C, oracle.CONV_WIDTH - 1))
    return xq, xk, xv, g, beta, gate, conv_w, norm_w, pool, cpool


def test_fused_prefill_inputs_are_unit_keys_and_scaled_queries():
    """After the conv, every key has unit norm and every query norm 1/sqrt(dk):
    the recurrence sees the inputs the rest of the path assumes."""
    xq, xk, xv, g, beta, gate, cw, nw, pool, cpool = _fused_case(7, [9])
    q, k, v, st = oracle.fused_inputs(xq[:, 0], xk[:, 0], xv[:, 0], cw[0], cpool[1, 0])
    np.testing.assert_allclose(np.linalg.norm(k, axis=1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(q, axis=1), 1.0 / np.sqrt(8), rtol=1e-13)
    assert st.shape == (24, 3)


@pytest.mark.parametrize("act", ["none", "silu"])
def test_fused_prefill_split_invariance(act):
    """Prefill of L1 tokens into slot a, then of the next L2 from slot a into
    slot b, equals one prefill of L1 + L2 into slot b: outputs, matrix state
    and convolution state (the two states travel together)."""
    L1, L2 = 5, 7
    xq, xk, xv, g, beta, gate, cw, nw, pool, cpool = _fused_case(8, [L1 + L2])
    args = lambda sl: tuple(a[sl] for a in (xq, xk, xv, g, beta, gate))
    o, p, c, _ = oracle.prefill_fused_pool(*args(slice(None)), cw, nw, [0, L1 + L2],
                                           [[2, 4]], pool, cpool, act=act)
    o1, p1, c1, _ = oracle.prefill_fused_pool(*args(slice(0, L1)), cw, nw, [0, L1],
                                              [[2, 3]], pool, cpool, act=act)
    o2, p2, c2, _ = oracle.prefill_fused_pool(*args(slice(L1, None)), cw, nw, [0, L2],
                                              [[3, 4]], p1, c1, act=act)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(p2[4], p[4], rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(c2[4], c[4])
    np.testing.assert_array_equal(c2[2], cpool[2])      # the source stays as it was


def test_fused_decode_equals_fused_prefill_of_the_same_tokens():
    """n tokens of decode in place on a slot equal a prefill of those tokens
    from that slot into the same slot (both pools)."""
    n = 3
    xq, xk, xv, g, beta, gate, cw, nw, pool, cpool = _fused_case(9, [2 * n])
    slots = [5, 1]
    od, pd, cd = oracle.decode_fused_pool(xq, xk, xv, g, beta, gate, cw, nw, slots, pool,
                                          cpool, n)
    cu = [0, n, 2 * n]
    op, pp, cp, _ = oracle.prefill_fused_pool(xq, xk, xv, g, beta, gate, cw, nw, cu,
                                              [[5, 5], [1, 1]], pool, cpool)
    np.testing.assert_allclose(od, op, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(pd, pp, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(cd, cp)


def test_fused_with_identity_conv_and_open_gate_is_the_plain_recurrence_normed():
    """An identity conv (current tap 1) and a saturated gate reduce the fused
    prefill to the plain prefill of the L2-normalised inputs, RMS-normalised:
    the convolution and gate add nothing of their own."""
    xq, xk, xv, g, beta, gate, cw, nw, pool, cpool = _fused_case(10, [6, 4])
    cw = np.zeros_like(cw); cw[:, :, -1] = 1.0
    gate = np.full_like(gate, 60.0)
    nw = np.ones_like(nw)
    o, p, c, _ = oracle.prefill_fused_pool(xq, xk, xv, g, beta, gate, cw, nw, [0, 6, 10],
                                           [[-1, 0], [3, 2]], pool, cpool)
    q = xq / np.linalg.norm(xq, axis=-1, keepdims=True) / np.sqrt(8)
    k = xk / np.linalg.norm(xk, axis=-1, keepdims=True)
    o_ref, p_ref, _ = oracle.prefill_pool(q, k, xv, g, beta, [0, 6, 10], [[-1, 0], [3, 2]], pool)
    rms = np.sqrt(np.mean(o_ref ** 2, axis=-1, keepdims=True) + oracle.RMS_EPS)
    np.testing.assert_allclose(o, o_ref / rms, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(p, p_ref, rtol=1e-12)


# ------------------------------------------------------------------ operand rounding

def test_round_to_matches_torch_casts_and_bounds():
    """On values that fp32 holds exactly, rounding to bf16 is torch's fp32 ->
    bf16 cast (round to nearest, ties to even); rounding to f32 is numpy's
    cast; both are idempotent, with relative error at most the unit roundoff
    (2^-8 for 8 significant bits)."""
    rng = _rng(11)
    x32 = (rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    x32[:8] = [1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8, 0.0, 3.0, 2.0 ** -9, 7.0]
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to(x32.astype(np.float64), "bf16")
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(oracle.round_to(got, "bf16"), got)
    x = rng.standard_normal(1000)
    np.testing.assert_array_equal(oracle.round_to(x, "f32"), x.astype(np.float32).astype(np.float64))
    r = oracle.round_to(x, "bf16")
    assert np.all(np.abs(r - x) <= 2.0 ** -8 * np.abs(x))   # unit roundoff of 8 bits
    np.testing.assert_array_equal(oracle.round_to(x, None), x)


def test_fused_operand_rounding_is_the_only_difference():
    """With operand_dtype the recurrence sees q, k, v rounded to bf16, and
    nothing else changes: the result equals the plain prefill of the rounded
    exact operands."""
    xq, xk, xv, g, beta, gate, cw, nw, pool, cpool = _fused_case(12, [9, 5])
    cu, slots = [0, 9, 14], [[2, 1], [-1, 3]]
    o, p, c, _ = oracle.prefill_fused_pool(xq, xk, xv, g, beta, gate, cw, nw, cu, slots, pool,
                                           cpool, operand_dtype="bf16")
    H, dk = xq.shape[1], xq.shape[2]
    q, k, v = np.zeros_like(xq), np.zeros_like(xk), np.zeros_like(xv)
    for b, (t0, t1) in enumerate([(0, 9), (9, 14)]):
        src = slots[b][0]
        for h in range(H):
            qb, kb, vb, _ = oracle.fused_inputs(xq[t0:t1, h], xk[t0:t1, h], xv[t0:t1, h], cw[h],
                                                cpool[src, h] if src >= 0 else None)
            q[t0:t1, h] = oracle.round_to(qb, "bf16")
            k[t0:t1, h] = oracle.round_to(kb, "bf16")
            v[t0:t1, h] = oracle.round_to(vb, "bf16")
    o_ref, p_ref, _ = oracle.prefill_pool(q, k, v, g, beta, cu, slots, pool)
    np.testing.assert_allclose(o, oracle.rms_norm_gated(o_ref, nw, gate), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(p, p_ref, rtol=1e-12, atol=1e-14)
