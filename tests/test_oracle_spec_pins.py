"""Pins for ``oracle.decode_spec_pool``, the speculative verify that commits
the previous step's accepted tokens in the same call.

The protocol is pinned to things other than itself:
* the rollback rule of the per-token-state decode (the slot after a commit of
  a tokens is the state after token a-1 of the previous verify step);
* the delta rule's closed form (a unit key written with beta = 1 is read back
  exactly: S^T k = v), which needs none of the oracle's code;
* the special cases: nothing accepted leaves the pool bit-identical, a
  verify-only call never writes, a commit-only call has no outputs.
The speculator that motivates the protocol is the DSpark verify pass of "Kimi
K3 on vLLM: Up to 370 Tokens/sec" (7 draft tokens; 8 on the vLLM recipe page
for Kimi-K3).
"""

import numpy as np
import pytest

import oracle


def _tokens(rng, T, H, dk, dv, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.exp(rng.standard_normal((T, H, dk)) - 3.0)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def _case(seed, N=4, n_prev=5, n_tok=3, H=2, d=8, n_slots=7):
    rng = np.random.default_rng(seed)
    prev = _tokens(rng, N * n_prev, H, d, d)
    cur = _tokens(rng, N * n_tok, H, d, d)
    pool = 0.3 * rng.standard_normal((n_slots, H, d, d))
    slots = rng.permutation(n_slots)[:N]
    return prev, cur, pool, slots


def test_commit_equals_rollback_of_per_token_states():
    """The committed slot is per_tok_states[n][a-1] of the previous verify
    step (the pool is unchanged where a = 0), and the verify outputs are those
    of a plain decode from the committed state.  n_prev != n_tok, so reading
    the previous step's rows with the current step's stride would fail."""
    N, n_prev, n_tok = 4, 5, 3
    (qp, kp, vp, gp, bp), (q, k, v, g, b), pool, slots = _case(1, N, n_prev, n_tok)
    acc = np.array([0, 1, 3, 5])
    out, after = oracle.decode_spec_pool(q, k, v, g, b, slots, pool, n_tok, kp, vp, gp, bp,
                                         acc, n_prev)
    _, _, per = oracle.decode_pool(qp, kp, vp, gp, bp, slots, pool, n_prev, True)
    expect = pool.copy()
    for n in range(N):
        if acc[n] > 0:
            expect[slots[n]] = per[n, acc[n] - 1]
    np.testing.assert_allclose(after, expect, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(after[slots[0]], pool[slots[0]])
    untouched = np.setdiff1d(np.arange(pool.shape[0]), slots)
    np.testing.assert_array_equal(after[untouched], pool[untouched])
    o_ref, _, _ = oracle.decode_pool(q, k, v, g, b, slots, expect, n_tok)
    np.testing.assert_allclose(out, o_ref, rtol=1e-13, atol=1e-13)


def test_committed_state_reads_back_the_last_accepted_value():
    """Closed form of the delta rule: after a token with unit k and beta = 1,
    S^T k = v exactly, whatever the decay (so the commit applied the last
    accepted token, with its own k and v, last)."""
    N, n_prev, n_tok, H, d = 3, 6, 2, 2, 8
    (qp, kp, vp, gp, bp), (q, k, v, g, b), pool, slots = _case(2, N, n_prev, n_tok, H, d)
    bp = np.ones_like(bp)
    acc = np.array([6, 2, 4])
    _, after = oracle.decode_spec_pool(q, k, v, g, b, slots, pool, n_tok, kp, vp, gp, bp, acc,
                                       n_prev)
    for n in range(N):
        last = n * n_prev + acc[n] - 1
        for h in range(H):
            np.testing.assert_allclose(after[slots[n], h].T @ kp[last, h], vp[last, h],
                                       rtol=0, atol=1e-12)


def test_verify_only_never_writes_and_commit_only_has_no_outputs():
    N, n_prev, n_tok = 3, 4, 4
    (qp, kp, vp, gp, bp), (q, k, v, g, b), pool, slots = _case(3, N, n_prev, n_tok)
    out, after = oracle.decode_spec_pool(q, k, v, g, b, slots, pool, n_tok)
    np.testing.assert_array_equal(after, pool)
    o_ref, _, _ = oracle.decode_pool(q, k, v, g, b, slots, pool, n_tok)
    np.testing.assert_allclose(out, o_ref, rtol=1e-13, atol=1e-13)
    # commit only: the slot advances by all accepted tokens, no outputs
    acc = np.full(N, n_prev)
    out0, after0 = oracle.decode_spec_pool(None, None, None, None, None, slots, pool, 0, kp, vp,
                                           gp, bp, acc, n_prev)
    assert out0.shape[0] == 0
    _, full, _ = oracle.decode_pool(qp, kp, vp, gp, bp, slots, pool, n_prev)
    np.testing.assert_allclose(after0, full, rtol=1e-13, atol=1e-13)


def test_two_step_protocol_equals_sequential_decode():
    """Two verify steps with commits give, for the accepted tokens, the same
    outputs and final slot as decoding only the accepted tokens one by one
    (the state never sees a rejected token)."""
    N, n_tok, H, d = 2, 4, 1, 8
    rng = np.random.default_rng(4)
    steps = [_tokens(rng, N * n_tok, H, d, d) for _ in range(3)]
    pool = 0.3 * rng.standard_normal((3, H, d, d))
    slots = np.array([2, 0])
    accs = [np.array([2, 4]), np.array([1, 3])]
    cur_pool = pool
    outs = []
    for s in range(3):
        q, k, v, g, b = steps[s]
        if s == 0:
            o, cur_pool = oracle.decode_spec_pool(q, k, v, g, b, slots, cur_pool, n_tok)
        else:
            _, kp, vp, gp, bp = steps[s - 1]
            o, cur_pool = oracle.decode_spec_pool(q, k, v, g, b, slots, cur_pool, n_tok, kp, vp,
                                                  gp, bp, accs[s - 1], n_tok)
        outs.append(o)
    for n in range(N):
        S = pool[slots[n], 0]
        for s in range(2):
            q, k, v, g, b = steps[s]
            a = accs[s][n]
            r = slice(n * n_tok, n * n_tok + a)
            o, S = oracle.recurrence(q[r, 0], k[r, 0], v[r, 0], g[r, 0], b[r, 0], S)
            np.testing.assert_allclose(outs[s][n * n_tok:n * n_tok + a, 0], o, rtol=1e-12,
                                       atol=1e-12)
        np.testing.assert_allclose(cur_pool[slots[n], 0], S, rtol=1e-12, atol=1e-12)


def test_accepted_length_out_of_range_is_rejected():
    (qp, kp, vp, gp, bp), (q, k, v, g, b), pool, slots = _case(5, 4, 5, 3)
    with pytest.raises(ValueError):
        oracle.decode_spec_pool(q, k, v, g, b, slots, pool, 3, kp, vp, gp, bp,
                                np.array([0, 6, 1, 1]), 5)


# ---------------------------------------------------------------- retention map

def _varlen(rng, lens, H, d):
    T = sum(lens)
    q, k, v, g, beta = _tokens(rng, T, H, d, d)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return q, k, v, g, beta, cu


def test_retained_snapshot_is_the_prefix_state():
    """A retained snapshot slot holds the state after (j+1) * interval tokens
    of its sequence's segment: the final state of a plain recurrence over that
    prefix from the sequence's start state (split invariance of the
    recurrence); dropped snapshots and slots outside the call are untouched."""
    rng = np.random.default_rng(21)
    lens, H, d, interval = [13, 4, 9], 2, 8, 4
    q, k, v, g, beta, cu = _varlen(rng, lens, H, d)
    pool = 0.3 * rng.standard_normal((12, H, d, d))
    init = np.array([[5, 0], [-1, 1], [2, 3]])
    # snapshots: seq 0 has 3, seq 1 has 1, seq 2 has 2 -> 6 entries
    snap_slots = np.array([7, -1, 9, 10, -1, 11])
    out, after = oracle.prefill_pool_retain(q, k, v, g, beta, cu, init, pool, interval,
                                            snap_slots)
    owners = [(0, 0), (0, 1), (0, 2), (1, 0), (2, 0), (2, 1)]
    for s, (b, j) in enumerate(owners):
        if snap_slots[s] < 0:
            continue
        t0 = cu[b]
        t1 = t0 + (j + 1) * interval
        for h in range(H):
            S0 = pool[init[b, 0], h] if init[b, 0] >= 0 else None
            _, S = oracle.recurrence(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                                     beta[t0:t1, h], S0)
            np.testing.assert_allclose(after[snap_slots[s], h], S, rtol=1e-13, atol=1e-13)
    for slot in (2, 4, 5, 6, 8):  # sources, dropped, outside the call
        np.testing.assert_array_equal(after[slot], pool[slot])
    _, plain, _ = oracle.prefill_pool(q, k, v, g, beta, cu, init, pool, 0)
    np.testing.assert_array_equal(out, oracle.prefill_pool(q, k, v, g, beta, cu, init, pool,
                                                           0)[0])
    for slot in (0, 1, 3):  # destinations: the final states
        np.testing.assert_array_equal(after[slot], plain[slot])


def test_retaining_nothing_equals_no_snapshots():
    rng = np.random.default_rng(22)
    q, k, v, g, beta, cu = _varlen(rng, [10, 7], 1, 8)
    pool = 0.3 * rng.standard_normal((4, 1, 8, 8))
    init = np.array([[-1, 0], [3, 1]])
    out, after = oracle.prefill_pool_retain(q, k, v, g, beta, cu, init, pool, 2,
                                            np.full(8, -1))
    o2, p2, _ = oracle.prefill_pool(q, k, v, g, beta, cu, init, pool, 0)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(after, p2)


# ---------------------------------------------------------------- sequence split

def test_split_recurrence_equals_the_sequential_run():
    """Cutting a sequence into segments (zero-state run plus identity run with
    v = 0 per segment, start states chained, outputs corrected) reproduces the
    token-by-token recurrence, with and without an initial state, for one and
    for several cuts including cuts one token apart."""
    rng = np.random.default_rng(31)
    L, dk, dv = 40, 6, 5
    q, k, v, g, beta = (a[:, 0] for a in _tokens(rng, L, 1, dk, dv))
    S0 = 0.3 * rng.standard_normal((dk, dv))
    o_ref, S_ref = oracle.recurrence(q, k, v, g, beta, S0)
    for splits in ([20], [7, 8, 30], [1, 39], list(range(4, 40, 4))):
        for init in (None, S0):
            o, S = oracle.split_recurrence(q, k, v, g, beta, init, splits)
            o_want, S_want = (o_ref, S_ref) if init is not None else \
                oracle.recurrence(q, k, v, g, beta, None)
            np.testing.assert_allclose(o, o_want, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(S, S_want, rtol=1e-12, atol=1e-12)


def test_identity_run_is_the_product_of_the_token_maps():
    """The identity run with v = 0 is the product of the token maps
    A_t = (I - b_t k_t k_t^T) Diag(exp g_t), written out directly."""
    rng = np.random.default_rng(32)
    L, d = 9, 4
    q, k, v, g, beta = (a[:, 0] for a in _tokens(rng, L, 1, d, d))
    _, Phi = oracle.recurrence(q, k, np.zeros((L, d)), g, beta, np.eye(d))
    P = np.eye(d)
    for t in range(L):
        A = (np.eye(d) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        P = A @ P
    np.testing.assert_allclose(Phi, P, rtol=1e-13, atol=1e-13)
