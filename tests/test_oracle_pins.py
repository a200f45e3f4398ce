"""Pins for the fp64 oracle: it is checked against things other than itself.

Each pin is a closed form, an invariant or an exact-arithmetic brute force of
the KDA recurrence (the gated delta rule with per-channel decay described for
Kimi Delta Attention on "Kimi K3 on vLLM: Up to 370 Tokens/sec", section "Kimi
Delta Attention: a hybrid recurrent + full-attention stack").  The pins are
written against a callable with the signature of ``oracle.recurrence`` so that
``test_pins_catch_planted_mistakes`` can run them on deliberately broken copies
and show that every plausible slip fails at least one of them.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, L, dk, dv, unit_k=False, g_scale=1.0):
    q = rng.standard_normal((L, dk))
    k = rng.standard_normal((L, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    g = -np.exp(rng.standard_normal((L, dk)) - 3.0) * g_scale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    S0 = 0.3 * rng.standard_normal((dk, dv))
    return q, k, v, g, beta, S0


# ---------------------------------------------------------------- pin bodies
# Each returns normally when the pin holds and raises AssertionError otherwise.

def pin_hand_worked(rec):
    """tests/golden/hand_worked_2tok.json, derived by hand from the definition."""
    with open(os.path.join(GOLDEN, "hand_worked_2tok.json")) as f:
        gold = json.load(f)
    toks = gold["tokens"]
    q = np.array([t["q"] for t in toks])
    k = np.array([t["k"] for t in toks])
    v = np.array([t["v"] for t in toks])
    g = np.log(np.array([t["exp_g"] for t in toks]))
    beta = np.array([t["beta"] for t in toks])
    o, S, st = rec(q, k, v, g, beta, np.array(gold["S0"]), return_states=True)
    np.testing.assert_allclose(st, np.array(gold["S"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, np.array(gold["o"]), rtol=0, atol=1e-12)


def pin_exact_rational(rec):
    """Brute force in exact rational arithmetic of the operator form
    S_t = (I - b k k^T) Diag(a) S + b k v^T (a = exp g chosen as exact
    binary fractions), on a random 4-token, 3x2 case."""
    rng = np.random.default_rng(7)
    L, dk, dv = 4, 3, 2
    def frac_mat(shape, den):
        return [[Fraction(int(x), den) for x in row]
                for row in rng.integers(-den, den + 1, size=shape)]
    K = frac_mat((L, dk), 8)
    V = frac_mat((L, dv), 8)
    Q = frac_mat((L, dk), 8)
    A = [[Fraction(int(x), 16) for x in row] for row in rng.integers(1, 17, size=(L, dk))]
    Bt = [Fraction(int(x), 8) for x in rng.integers(1, 9, size=L)]
    S = frac_mat((dk, dv), 4)
    S0f = [[float(x) for x in r] for r in S]
    exp_states, exp_out = [], []
    for t in range(L):
        # D = Diag(a) S ; P = I - b k k^T ; S = P D + b k v^T   (exactly)
        D = [[A[t][i] * S[i][j] for j in range(dv)] for i in range(dk)]
        P = [[(1 if i == r else 0) - Bt[t] * K[t][i] * K[t][r] for r in range(dk)]
             for i in range(dk)]
        S = [[sum(P[i][r] * D[r][j] for r in range(dk)) + Bt[t] * K[t][i] * V[t][j]
              for j in range(dv)] for i in range(dk)]
        exp_states.append([[float(x) for x in r] for r in S])
        exp_out.append([float(sum(S[i][j] * Q[t][i] for i in range(dk))) for j in range(dv)])
    f = lambda M: np.array([[float(x) for x in r] for r in M])
    o, Sf, st = rec(f(Q), f(K), f(V), np.log(f(A)), np.array([float(b) for b in Bt]),
                    np.array(S0f), return_states=True)
    np.testing.assert_allclose(st, np.array(exp_states), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, np.array(exp_out), rtol=1e-13, atol=1e-13)


def pin_retrieval(rec):
    """Unit-norm k and beta = 1: the new state maps k_t exactly to v_t,
    S_t^T k_t = v_t, for any decay g (pins the delta correction and that it
    acts on the decayed state); with q_t = k_t the output is then v_t (pins
    that o_t reads the state after token t's update)."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta, S0 = _rand_case(rng, 12, 8, 5, unit_k=True, g_scale=5.0)
    beta[:] = 1.0
    _, _, st = rec(q, k, v, g, beta, S0, return_states=True)
    for t in range(len(k)):
        np.testing.assert_allclose(st[t].T @ k[t], v[t], rtol=0, atol=1e-12)
    o, _ = rec(k, k, v, g, beta, S0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def pin_orthonormal_overwrite(rec):
    """g = 0, beta = 1 and keys forming an orthonormal basis written once each:
    every step replaces the state's component along k_t by v_t, so after all
    dk tokens S = K^T V whatever S0 was (a closed form of the plain delta rule)."""
    rng = np.random.default_rng(2)
    dk, dv = 6, 4
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm.T.copy()                         # rows orthonormal
    v = rng.standard_normal((dk, dv))
    q = rng.standard_normal((dk, dk))
    S0 = rng.standard_normal((dk, dv))
    _, S = rec(q, k, v, np.zeros((dk, dk)), np.ones(dk), S0)
    np.testing.assert_allclose(S, k.T @ v, rtol=0, atol=1e-12)


def pin_beta_zero(rec):
    """beta = 0: nothing is written, the state only decays:
    S_t = Diag(exp(sum_{i<=t} g_i)) S0 and o_t = S_t^T q_t; with g = 0 the
    state stays S0 and o_t = S0^T q_t."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta, S0 = _rand_case(rng, 10, 7, 3)
    beta[:] = 0.0
    o, _, st = rec(q, k, v, g, beta, S0, return_states=True)
    G = np.cumsum(g, axis=0)
    for t in range(len(k)):
        np.testing.assert_allclose(st[t], np.exp(G[t])[:, None] * S0, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(o[t], st[t].T @ q[t], rtol=1e-13, atol=1e-14)
    o0, S = rec(q, k, v, np.zeros_like(g), beta, S0)
    np.testing.assert_allclose(S, S0, rtol=0, atol=0)
    np.testing.assert_allclose(o0, q @ S0, rtol=1e-13, atol=1e-14)


def pin_full_decay(rec):
    """exp(g) = 0 (g = -1e4 underflows to exactly 0): the old state is
    forgotten each step, S_t = b_t k_t v_t^T and o_t = b_t (k_t . q_t) v_t."""
    rng = np.random.default_rng(4)
    q, k, v, g, beta, S0 = _rand_case(rng, 6, 5, 4)
    g[:] = -1e4
    o, _, st = rec(q, k, v, g, beta, S0, return_states=True)
    for t in range(len(k)):
        np.testing.assert_allclose(st[t], beta[t] * np.outer(k[t], v[t]), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(o[t], beta[t] * (k[t] @ q[t]) * v[t], rtol=1e-13, atol=1e-15)


def pin_linear_attention_limit(rec):
    """Without the delta correction (u = v, the oracle's no_delta hook) and with
    g = 0, KDA is plain causal linear attention: S_t = S0 + K[:t]^T V[:t] and
    O = Q S0 + tril(Q K^T) V (the running sum of k v^T).  With a decay it is
    gated linear attention: S_t = Diag(e^{G_t}) S0 + sum_i Diag(e^{G_t-G_i}) k_i v_i^T."""
    rng = np.random.default_rng(5)
    q, k, v, g, beta, S0 = _rand_case(rng, 9, 6, 3)
    o, S, st = rec(q, k, v, np.zeros_like(g), beta, S0, no_delta=True, return_states=True)
    for t in range(len(k)):
        np.testing.assert_allclose(st[t], S0 + k[:t + 1].T @ v[:t + 1], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, q @ S0 + np.tril(q @ k.T) @ v, rtol=1e-13, atol=1e-13)
    _, _, st = rec(q, k, v, g, beta, S0, no_delta=True, return_states=True)
    G = np.cumsum(g, axis=0)
    for t in range(len(k)):
        ref = np.exp(G[t])[:, None] * S0
        for i in range(t + 1):
            ref = ref + np.outer(k[i] * np.exp(G[t] - G[i]), v[i])
        np.testing.assert_allclose(st[t], ref, rtol=1e-13, atol=1e-13)


def pin_linearity(rec):
    """(S0, V) -> (S_T, O) is linear for fixed q, k, g, beta."""
    rng = np.random.default_rng(6)
    q, k, v1, g, beta, S1 = _rand_case(rng, 11, 6, 4)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    a, b = 0.7, -1.3
    o1, F1 = rec(q, k, v1, g, beta, S1)
    o2, F2 = rec(q, k, v2, g, beta, S2)
    o3, F3 = rec(q, k, a * v1 + b * v2, g, beta, a * S1 + b * S2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(F3, a * F1 + b * F2, rtol=1e-12, atol=1e-12)


PINS = [pin_hand_worked, pin_exact_rational, pin_retrieval, pin_orthonormal_overwrite,
        pin_beta_zero, pin_full_decay, pin_linear_attention_limit, pin_linearity]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_numpy_recurrence_pins(pin):
    pin(oracle.recurrence)


def _c_rec(q, k, v, g, beta, S0=None, *, no_delta=False, return_states=False):
    """The C oracle seen through the single-(sequence, head) signature."""
    L = len(k)
    dk, dv = k.shape[1], v.shape[1]
    init = None if S0 is None else np.asarray(S0, dtype=np.float64).reshape(1, 1, dk, dv)
    res = oracle.run(q[:, None], k[:, None], v[:, None], g[:, None], np.asarray(beta)[:, None],
                     [0, L], init, 1 if return_states else 0, no_delta=no_delta, nthreads=2)
    o, S = res.out[:, 0], res.final[0, 0]
    if return_states:
        return o, S, res.snaps[:, 0]
    return o, S


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_c_oracle_pins(pin):
    pin(_c_rec)


# --------------------------------------------------- planted-mistake coverage

def _mutant(kind):
    """A copy of the sequential step with one plausible mistake planted."""
    def rec(q, k, v, g, beta, S0=None, *, no_delta=False, return_states=False):
        L, dk = k.shape
        dv = v.shape[1]
        S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=float)
        o = np.zeros((L, dv))
        st = np.zeros((L, dk, dv))
        for t in range(L):
            a = np.exp(g[t])
            if kind == "decay_after_correction":
                u = beta[t] * (v[t] - S.T @ k[t])
                S = a[:, None] * (S + np.outer(k[t], u))
            else:
                Sd = (a[None, :] * S) if kind == "decay_on_columns" else a[:, None] * S
                if kind == "transposed_read":
                    x = (Sd @ k[t][:Sd.shape[1]]) if dk == dv else Sd.T @ (k[t] * 1.0001)
                else:
                    x = Sd.T @ k[t]
                if kind == "dropped_beta":
                    u = v[t] - x
                elif kind == "sign_flip":
                    u = beta[t] * (v[t] + x)
                elif kind == "beta_on_v_only":
                    u = beta[t] * v[t] - x
                else:
                    u = v[t] if no_delta else beta[t] * (v[t] - x)
                if no_delta and kind not in ("dropped_beta", "sign_flip", "beta_on_v_only"):
                    u = v[t]
                S_prev = S
                S = Sd + np.outer(k[t], u)
                if kind == "output_before_update":
                    o[t] = S_prev.T @ q[t]
                    st[t] = S
                    continue
            o[t] = (S.T @ q[t]) if kind != "output_uses_k" else (S.T @ k[t])
            st[t] = S
        if return_states:
            return o, S, st
        return o, S
    return rec


MUTANTS = ["decay_after_correction", "decay_on_columns", "transposed_read", "dropped_beta",
           "sign_flip", "beta_on_v_only", "output_before_update", "output_uses_k"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistakes(kind):
    rec = _mutant(kind)
    caught = []
    for pin in PINS:
        try:
            pin(rec)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {kind}"


# ------------------------------------------------ chunked form and semantics

@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("L", [1, 17, 64, 129, 256])
def test_chunked_equals_sequential(C, L):
    """The chunked WY/UT evaluation equals the sequential recurrence to fp64
    rounding, for full and ragged last chunks and a nonzero start state."""
    rng = np.random.default_rng(100 + L + C)
    q, k, v, g, beta, S0 = _rand_case(rng, L, 16, 16, unit_k=True)
    o1, S1 = oracle.recurrence(q, k, v, g, beta, S0)
    o2, S2, _ = oracle.chunked(q, k, v, g, beta, S0, C=C)
    assert oracle.rel_l2(o2, o1) < 1e-12
    assert oracle.rel_l2(S2, S1) < 1e-12


def test_chunked_snapshots_match_sequential_states():
    rng = np.random.default_rng(11)
    q, k, v, g, beta, S0 = _rand_case(rng, 200, 8, 8, unit_k=True)
    _, _, st = oracle.recurrence(q, k, v, g, beta, S0, return_states=True)
    _, _, snaps = oracle.chunked(q, k, v, g, beta, S0, C=16, snap_interval=32)
    assert snaps.shape[0] == 200 // 32
    for j in range(snaps.shape[0]):
        assert oracle.rel_l2(snaps[j], st[(j + 1) * 32 - 1]) < 1e-12


def test_split_invariance_and_snapshots():
    """run(L1) then run(L2) from its final state equals run(L1 + L2); snapshot
    j equals the final state of the prefix of length (j+1)*interval."""
    rng = np.random.default_rng(12)
    q, k, v, g, beta, S0 = _rand_case(rng, 96, 8, 6, unit_k=True)
    o, S = oracle.recurrence(q, k, v, g, beta, S0)
    oa, Sa = oracle.recurrence(q[:40], k[:40], v[:40], g[:40], beta[:40], S0)
    ob, Sb = oracle.recurrence(q[40:], k[40:], v[40:], g[40:], beta[40:], Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sb, S, rtol=1e-13, atol=1e-13)
    res = oracle.run(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], [0, 96],
                     S0[None, None], 32, backend="numpy")
    for j in range(3):
        _, Sj = oracle.recurrence(q[:32 * (j + 1)], k[:32 * (j + 1)], v[:32 * (j + 1)],
                                  g[:32 * (j + 1)], beta[:32 * (j + 1)], S0)
        np.testing.assert_allclose(res.snaps[j, 0], Sj, rtol=1e-13, atol=1e-13)


def _varlen_case(rng, lens, H, dk, dv):
    T = sum(lens)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.exp(rng.standard_normal((T, H, dk)) - 3.0)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    cu = np.concatenate([[0], np.cumsum(lens)])
    return q, k, v, g, beta, cu


def test_c_oracle_equals_numpy_oracle_varlen():
    """The C loop and the numpy loop agree on a packed varlen batch with
    initial states, snapshots, a unit sample and a column sample."""
    rng = np.random.default_rng(13)
    lens = [5, 0, 33, 64, 17]
    q, k, v, g, beta, cu = _varlen_case(rng, lens, 3, 16, 16)
    init = rng.standard_normal((len(lens), 3, 16, 16)) * 0.1
    a = oracle.run(q, k, v, g, beta, cu, init, 16, backend="c", nthreads=3)
    b = oracle.run(q, k, v, g, beta, cu, init, 16, backend="numpy")
    for x, y in ((a.out, b.out), (a.final, b.final), (a.snaps, b.snaps)):
        np.testing.assert_allclose(x, y, rtol=1e-14, atol=1e-14)
    units = [(2, 1), (3, 0)]
    c = oracle.run(q, k, v, g, beta, cu, init, 16, units=units, cols=(4, 12), nthreads=2)
    for (bb, hh) in units:
        t0, t1 = cu[bb], cu[bb + 1]
        np.testing.assert_array_equal(c.out[t0:t1, hh, 4:12], a.out[t0:t1, hh, 4:12])
        np.testing.assert_array_equal(c.final[bb, hh][:, 4:12], a.final[bb, hh][:, 4:12])
    assert np.isnan(c.out[cu[0]:cu[1], 0]).all()


def test_pool_semantics():
    """Copy-on-write resume: sources are read, destinations written, other
    slots untouched; src == dst extends in place."""
    rng = np.random.default_rng(14)
    lens = [20, 7, 13]
    q, k, v, g, beta, cu = _varlen_case(rng, lens, 2, 8, 8)
    pool = rng.standard_normal((6, 2, 8, 8))
    slots = np.array([[1, 4], [-1, 5], [2, 2]])
    out, after, _ = oracle.prefill_pool(q, k, v, g, beta, cu, slots, pool)
    np.testing.assert_array_equal(after[[0, 1, 3]], pool[[0, 1, 3]])
    for b, (src, dst) in enumerate(slots):
        S0 = pool[src] if src >= 0 else None
        for h in range(2):
            t0, t1 = cu[b], cu[b + 1]
            o, S = oracle.recurrence(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                                     beta[t0:t1, h], None if S0 is None else S0[h])
            np.testing.assert_allclose(after[dst, h], S, rtol=1e-14, atol=1e-14)
            np.testing.assert_allclose(out[t0:t1, h], o, rtol=1e-14, atol=1e-14)


def test_decode_multi_token_equals_repeated_single():
    """Decoding n tokens at once equals n single-token decodes, and the
    per-token states are the intermediate pool states."""
    rng = np.random.default_rng(15)
    N, n_tok, H, d = 3, 4, 2, 8
    q, k, v, g, beta, _ = _varlen_case(rng, [n_tok] * N, H, d, d)
    pool = rng.standard_normal((5, H, d, d))
    slots = np.array([4, 0, 2])
    out, after, per = oracle.decode_pool(q, k, v, g, beta, slots, pool, n_tok, True)
    cur = pool.copy()
    for j in range(n_tok):
        rows = np.arange(N) * n_tok + j
        o1, cur, _ = oracle.decode_pool(q[rows], k[rows], v[rows], g[rows], beta[rows], slots,
                                        cur, 1)
        np.testing.assert_allclose(out[rows], o1, rtol=1e-13, atol=1e-13)
        for n in range(N):
            np.testing.assert_allclose(per[n, j], cur[slots[n]], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(after, cur, rtol=1e-13, atol=1e-13)
