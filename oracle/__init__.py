"""Plain fp64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` import this package.  The GPU
library never imports, loads or calls it, and this package imports nothing
from the GPU library; the two share no code.  Inputs reach both sides from the
seeded generators in ``hybrid_linear_attention_delta_gb300.inputs``, which hold
none of the method's arithmetic.

What is computed, and where it is stated:

* The recurrence (the gated delta rule with per-channel decay, fp32 state per
  (sequence, head), "a fixed-size matrix-like recurrent state per layer" --
  "Kimi K3 + vLLM: Inside the Day-0 Production Integration", section "Kimi
  Delta Attention: When Prefix Caching Meets Recurrent State"; "Kimi K3 on
  vLLM: Up to 370 Tokens/sec", section "Kimi Delta Attention: a hybrid
  recurrent + full-attention stack")::

      S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T
      o_t = S_t^T q_t

  ``recurrence`` evaluates it token by token; ``kda_oracle.c`` is the same
  sequential loop in C with threads over independent (sequence, head, column
  block) units, used for large cases and for the CPU baseline.

* The chunked evaluation (``chunked``) is the 64-token-chunk WY/UT form that
  the GPU prefill uses, written out in fp64 with library primitives (matmul,
  triangular solve).  It is pinned to the sequential form, not trusted alone.

* Serving semantics of the prefix cache ("Separating Physical Blocks,
  Scheduler Alignment, and Prefix Matching"; "Interval-Based and
  Marconi-Style Retention" of the Day-0 integration page): a sequence resumes
  from a cached state that is copied on write into a private destination slot
  before extension; snapshots are taken every ``snap_interval`` tokens of the
  segment; the final (prompt-boundary) state is always kept.  Decode
  ("a fused CUDA kernel ... for decode", and the speculative-decoding verify
  path) applies the same step to one or several tokens in place on a pool slot
  and can record the state after each token for rollback; ``decode_spec_pool``
  is the speculative verify that commits the previous step's accepted tokens
  before evaluating the new ones.

* ``short_conv``, ``l2_normalize`` and ``rms_norm_gated`` are the layer
  around the recurrence that the pages' fused decode kernel folds into its
  launch (the short causal convolution with its state, the output RMSNorm
  and sigmoid gate); ``prefill_fused_pool`` / ``decode_fused_pool`` compose
  them with the pool semantics above.

* ``split_recurrence`` is the algebra of a sequence-split prefill (segments
  from the zero state plus identity runs with v = 0, start states chained,
  outputs corrected); the GPU library does not implement it yet, and it is
  pinned against the sequential recurrence.

Every function here has pins in ``tests/test_oracle_pins.py`` (closed forms,
invariants, exact-rational brute force, sequential-vs-chunked agreement,
C-vs-numpy agreement).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_SRC = os.path.join(_HERE, "kda_oracle.c")
_lib = None


# ----------------------------------------------------------------------------
# build / load the C oracle
# ----------------------------------------------------------------------------

def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library with the host gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.kda_oracle_run.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P, i32, P, P, P, P,
                                       i32, P, i32, i32, i32]
        lib.kda_oracle_run.restype = ctypes.c_int
        _lib = lib
    return _lib


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    """Exact upcast to a C-contiguous float64 array (bf16/fp32 -> fp64 is exact)."""
    if hasattr(x, "detach"):  # a torch tensor
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------
# one (sequence, head): sequential and chunked fp64 forms
# ----------------------------------------------------------------------------

def recurrence(q, k, v, g, beta, S0=None, *, no_delta=False, return_states=False):
    """Token-by-token fp64 KDA for ONE (sequence, head).

    q, k, g: [L, dk]; v: [L, dv]; beta: [L]; S0: [dk, dv] or None (zero).
    Returns (o [L, dv], S_L [dk, dv]) and, with ``return_states``, also the
    state after every token [L, dk, dv].

    Step t (the operator order of the definition: decay first, then the delta
    correction against the decayed state, then the write; the output reads the
    state after token t's own update):
        S' = Diag(exp g_t) S ;  u = beta_t (v_t - S'^T k_t) ;  S = S' + k_t u^T ;
        o_t = S^T q_t
    ``no_delta`` is a test hook that drops the correction (u = v_t), which
    turns the step into plain gated linear attention.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    beta = _f64(beta).reshape(-1)
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((L, dv))
    states = np.zeros((L, dk, dv)) if return_states else None
    for t in range(L):
        S = np.exp(g[t])[:, None] * S
        u = v[t] if no_delta else beta[t] * (v[t] - S.T @ k[t])
        S = S + np.outer(k[t], u)
        o[t] = S.T @ q[t]
        if return_states:
            states[t] = S
    if return_states:
        return o, S, states
    return o, S


def chunked(q, k, v, g, beta, S0=None, *, C=64, snap_interval=0):
    """Chunked (WY / UT-transform) fp64 KDA for ONE (sequence, head).

    For each chunk of C' <= C tokens with start state S0 and in-chunk
    positions r = 1..C':
        G_r   = sum_{i<=r} g_i                 (per channel)
        K+    = K * exp(G),  K- = K * exp(-G),  Q+ = Q * exp(G)
        A     = Diag(beta) * strict_lower(K+ K-^T)
        T     = (I + A)^{-1} Diag(beta)        (unit lower-triangular solve)
        W     = T K+ ,  U~ = T V ,  U = U~ - W S0
        O     = Q+ S0 + lower_incl(Q+ K-^T) U
        S_end = Diag(exp G_C') S0 + (K * exp(G_C' - G))^T U
    Row r of U is u_r of the sequential form, so O and S_end equal the
    token-by-token result up to rounding.  Returns (o, S_L, snapshots) where
    snapshots are the states after every ``snap_interval`` tokens (which must
    then be a multiple of C).
    """
    import scipy.linalg as sla

    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    beta = _f64(beta).reshape(-1)
    L, dk = k.shape
    dv = v.shape[1]
    if snap_interval and snap_interval % C:
        raise ValueError("snap_interval must be a multiple of the chunk size")
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((L, dv))
    snaps = []
    for c0 in range(0, L, C):
        c1 = min(c0 + C, L)
        n = c1 - c0
        G = np.cumsum(g[c0:c1], axis=0)
        Kp = k[c0:c1] * np.exp(G)
        Km = k[c0:c1] * np.exp(-G)
        Qp = q[c0:c1] * np.exp(G)
        b = beta[c0:c1]
        A = b[:, None] * np.tril(Kp @ Km.T, -1)
        T = sla.solve_triangular(np.eye(n) + A, np.diag(b), lower=True, unit_diagonal=True)
        W = T @ Kp
        U = T @ v[c0:c1] - W @ S
        o[c0:c1] = Qp @ S + np.tril(Qp @ Km.T) @ U
        S = np.exp(G[-1])[:, None] * S + (k[c0:c1] * np.exp(G[-1] - G)).T @ U
        if snap_interval and c1 % snap_interval == 0:
            snaps.append(S.copy())
    return o, S, (np.stack(snaps) if snaps else np.zeros((0, dk, dv)))


# ----------------------------------------------------------------------------
# packed varlen batches (the C oracle, or the numpy loop for tiny cases)
# ----------------------------------------------------------------------------

def snapshot_offsets(cu_seqlens: Sequence[int], snap_interval: int):
    """Snapshot j of sequence b lives at index off[b] + j; off is the exclusive
    scan of floor(L_b / snap_interval).  Returns (off [B], total)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = cu[1:] - cu[:-1]
    if snap_interval <= 0:
        return np.zeros(len(lens), dtype=np.int64), 0
    cnt = lens // snap_interval
    off = np.concatenate([[0], np.cumsum(cnt)[:-1]]).astype(np.int64)
    return off, int(cnt.sum())


@dataclass
class Result:
    out: np.ndarray          # [T, H, dv]
    final: np.ndarray        # [B, H, dk, dv]
    snaps: np.ndarray        # [n_snaps, H, dk, dv]


def run(q, k, v, g, beta, cu_seqlens, init_states=None, snap_interval=0, *, no_delta=False,
        units=None, cols=None, nthreads=None, backend="c") -> Result:
    """KDA over a packed batch.

    q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; cu_seqlens: [B+1];
    init_states: [B, H, dk, dv] or None (zero).  ``units`` optionally restricts
    the work to a set of (b, h) pairs and ``cols`` to a column range (lo, hi) of
    the state -- columns evolve independently, so a sampled column block is an
    exact slice of the full result.  Entries outside the sample are NaN.
    """
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    B = len(cu) - 1
    init = None if init_states is None else _f64(init_states)
    off, n_snaps = snapshot_offsets(cu, snap_interval)
    lo, hi = (0, dv) if cols is None else cols
    mask = None
    if units is not None:
        mask = np.zeros(B * H, dtype=np.int32)
        for (b, h) in units:
            mask[b * H + h] = 1
    out = np.full((T, H, dv), np.nan)
    final = np.full((B, H, dk, dv), np.nan)
    snaps = np.full((n_snaps, H, dk, dv), np.nan)
    if backend == "c":
        lib = _load()
        rc = lib.kda_oracle_run(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu), B, H, dk,
                                dv, _ptr(init), int(snap_interval), _ptr(off), _ptr(out),
                                _ptr(final), _ptr(snaps) if n_snaps else None, int(no_delta),
                                _ptr(mask), int(lo), int(hi),
                                int(nthreads or host_cores()))
        if rc != 0:
            raise ValueError("kda_oracle_run rejected its arguments")
        return Result(out, final, snaps)
    if backend != "numpy":
        raise ValueError(backend)
    for b in range(B):
        for h in range(H):
            if mask is not None and not mask[b * H + h]:
                continue
            t0, t1 = int(cu[b]), int(cu[b + 1])
            S0 = None if init is None else init[b, h][:, lo:hi]
            o, S, st = recurrence(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h, lo:hi], g[t0:t1, h],
                                  beta[t0:t1, h], S0, no_delta=no_delta, return_states=True)
            out[t0:t1, h, lo:hi] = o
            final[b, h][:, lo:hi] = S
            if snap_interval:
                for j in range((t1 - t0) // snap_interval):
                    snaps[off[b] + j, h][:, lo:hi] = st[(j + 1) * snap_interval - 1]
    return Result(out, final, snaps)


# ----------------------------------------------------------------------------
# state-pool semantics of the two library calls
# ----------------------------------------------------------------------------

def prefill_pool(q, k, v, g, beta, cu_seqlens, init_slots, state_pool, snap_interval=0, **kw):
    """What ``kda_prefill_varlen`` must produce.

    init_slots: [B, 2] = (src, dst).  Sequence b starts from pool[src] (zero
    state when src < 0), runs its segment, and its final state is written to
    pool[dst] (copy-on-write: src itself is not modified unless src == dst).
    All sources are read before any destination is written.
    Returns (out [T,H,dv], pool_after [n_slots,H,dk,dv], snaps).
    """
    pool = _f64(state_pool)
    slots = np.asarray(init_slots, dtype=np.int64).reshape(-1, 2)
    B = slots.shape[0]
    H, dk, dv = pool.shape[1:]
    init = np.zeros((B, H, dk, dv))
    for b in range(B):
        if slots[b, 0] >= 0:
            init[b] = pool[slots[b, 0]]
    res = run(q, k, v, g, beta, cu_seqlens, init, snap_interval, **kw)
    after = pool.copy()
    for b in range(B):
        after[slots[b, 1]] = res.final[b]
    return res.out, after, res.snaps


def prefill_pool_retain(q, k, v, g, beta, cu_seqlens, init_slots, state_pool, snap_interval,
                        snap_slots, **kw):
    """What ``kda_prefill_varlen_retain`` must produce.

    The prefill of ``prefill_pool``; snapshot s (numbered as there) is then
    written into pool slot snap_slots[s] when that is >= 0 and dropped when it
    is -1 ("Interval-Based and Marconi-Style Retention" of the Day-0
    integration page: the scheduler keeps only the states it will reuse; the
    prompt-boundary state still goes to dst).  Returns (out, pool_after).
    """
    out, after, snaps = prefill_pool(q, k, v, g, beta, cu_seqlens, init_slots, state_pool,
                                     snap_interval, **kw)
    slots = np.asarray(snap_slots, dtype=np.int64).reshape(-1)
    for s in range(min(len(slots), snaps.shape[0])):
        if slots[s] >= 0:
            after[slots[s]] = snaps[s]
    return out, after


def decode_pool(q, k, v, g, beta, slot_ids, state_pool, n_tok=1, per_tok_states=False, **kw):
    """What ``kda_decode`` must produce.

    Sequence n owns tokens [n*n_tok, (n+1)*n_tok) of the [N*n_tok, H, *] inputs
    and the pool slot slot_ids[n]; the slot is advanced in place to the state
    after all n_tok tokens.  With ``per_tok_states`` the state after token j is
    also returned at [n, j] (the rollback points of speculative verify).
    Returns (out, pool_after, per_tok [N, n_tok, H, dk, dv] or None).
    """
    pool = _f64(state_pool)
    slots = np.asarray(slot_ids, dtype=np.int64).reshape(-1)
    N = len(slots)
    H, dk, dv = pool.shape[1:]
    cu = np.arange(N + 1, dtype=np.int64) * n_tok
    init = np.stack([pool[s] for s in slots]) if N else np.zeros((0, H, dk, dv))
    res = run(q, k, v, g, beta, cu, init, 1 if per_tok_states else 0, **kw)
    after = pool.copy()
    for n in range(N):
        after[slots[n]] = res.final[n]
    per = res.snaps.reshape(N, n_tok, H, dk, dv) if per_tok_states else None
    return res.out, after, per


def decode_spec_pool(q, k, v, g, beta, slot_ids, state_pool, n_tok, k_prev=None, v_prev=None,
                     g_prev=None, beta_prev=None, accepted_prev=None, n_prev=0, **kw):
    """What ``kda_decode_spec`` must produce.

    The speculative-verify protocol (the DSpark speculator's verify pass of
    "Kimi K3 on vLLM: Up to 370 Tokens/sec"; the FLA decode path used under
    speculative decoding, "Kimi K3 + vLLM: Inside the Day-0 Production
    Integration") with the commit of the previous step done in the same call.
    For sequence n with slot s = slot_ids[n] and a = accepted_prev[n]:
      1. S = pool[s]; apply tokens j < a of the previous step (rows
         n*n_prev + j of the *_prev arrays) with the same token step as
         ``recurrence``; if a > 0 the slot becomes that committed state;
      2. from the committed state, tokens j < n_tok of this step (rows
         n*n_tok + j) produce their outputs; the slot keeps the committed
         state.
    Returns (out [N*n_tok, H, dv], pool_after).
    """
    pool = _f64(state_pool)
    slots = np.asarray(slot_ids, dtype=np.int64).reshape(-1)
    N = len(slots)
    H, dk, dv = pool.shape[1:]
    init = np.stack([pool[s] for s in slots]) if N else np.zeros((0, H, dk, dv))
    committed = init.copy()
    after = pool.copy()
    if n_prev > 0:
        acc = np.asarray(accepted_prev, dtype=np.int64).reshape(-1)
        if np.any(acc < 0) or np.any(acc > n_prev):
            raise ValueError("accepted lengths must lie in [0, n_prev]")
        rows = np.concatenate([np.arange(n * n_prev, n * n_prev + acc[n]) for n in range(N)]
                              + [np.zeros(0, dtype=np.int64)]).astype(np.int64)
        if len(rows):
            kp = _f64(k_prev)[rows]
            cu = np.concatenate([[0], np.cumsum(acc)]).astype(np.int64)
            # the replayed tokens have no outputs: any q serves, k is passed
            res = run(kp, kp, _f64(v_prev)[rows], _f64(g_prev)[rows], _f64(beta_prev)[rows], cu,
                      init, 0, **kw)
            for n in range(N):
                if acc[n] > 0:
                    committed[n] = res.final[n]
                    after[slots[n]] = res.final[n]
    if n_tok > 0:
        cu = np.arange(N + 1, dtype=np.int64) * n_tok
        out = run(q, k, v, g, beta, cu, committed, 0, **kw).out
    else:
        out = np.zeros((0, H, dv))
    return out, after


def split_recurrence(q, k, v, g, beta, S0, splits):
    """Sequence-split evaluation of ONE (sequence, head), the algebra of a
    split prefill (a long prompt cut into segments that run in parallel;
    "Kimi K3 on vLLM: Up to 370 Tokens/sec" motivates 1M-token contexts).

    The token step is affine in the state: S_t = A_t S_{t-1} + b_t with
    A_t = (I - beta_t k_t k_t^T) Diag(exp g_t) and b_t = beta_t k_t v_t^T.  So
    a segment [s, e) maps its start state X to Phi X + L, where L is the
    segment run from the zero state and Phi = A_{e-1} ... A_s is the same
    segment run from the identity (a dk x dk state) with v := 0.  Its outputs
    split the same way: o_t = L_t^T q_t + X^T (Phi_t^T q_t), and Phi_t^T q_t is
    the identity run's own output.  Segment start states chain serially
    (X_{i+1} = Phi_i X_i + L_i) and every segment's outputs are then corrected
    independently.  ``splits`` are the cut points (0 < s_1 < ... < L).
    Returns (o [L, dv], S_L), equal to ``recurrence`` up to rounding.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    beta = _f64(beta).reshape(-1)
    L, dk = k.shape
    dv = v.shape[1]
    bounds = [0] + [int(x) for x in splits] + [L]
    X = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((L, dv))
    for s0, s1 in zip(bounds[:-1], bounds[1:]):
        sl = slice(s0, s1)
        o_loc, L_end = recurrence(q[sl], k[sl], v[sl], g[sl], beta[sl], None)
        o_hom, Phi = recurrence(q[sl], k[sl], np.zeros((s1 - s0, dk)), g[sl], beta[sl],
                                np.eye(dk))
        o[sl] = o_loc + o_hom @ X          # row t: L_t^T q_t + X^T Phi_t^T q_t
        X = Phi @ X + L_end
    return o, X


# ----------------------------------------------------------------------------
# the fused layer around the recurrence: short causal convolution before it,
# gated RMSNorm after it
# ----------------------------------------------------------------------------
#
# "Kimi K3 + vLLM: Inside the Day-0 Production Integration": KDA keeps "a
# short causal convolution state" beside its matrix state ("Kimi Delta
# Attention: When Prefix Caching Meets Recurrent State"), both updated at
# every token, and its fused decode kernel "folds causal convolution,
# recurrent state update, gating, and RMSNorm into a single launch"
# ("Separate Prefill/Decode Code Paths"); the vLLM recipe page for Kimi-K3
# fuses "the KDA output RMSNorm and sigmoid gate" into one kernel.  The pages
# fix none of the sizes; the readings taken here (conv width 4, depthwise over
# the raw q, k and v channels, no activation unless asked for SiLU, q and k
# L2-normalised after the conv with q scaled by 1/sqrt(dk), RMSNorm epsilon
# 1e-6 with one weight per value column, the gate through a sigmoid after the
# norm) are the plainest ones consistent with the rest of the path.

CONV_WIDTH = 4
RMS_EPS = 1e-6


def short_conv(x, w, x_prev=None, act="none"):
    """Causal depthwise convolution of ONE sequence over time.

    x: [L, C] raw inputs; w: [C, W] taps (w[c, W-1] multiplies the current
    token, w[c, i] the token W-1-i steps back); x_prev: [W-1, C] the W-1 raw
    inputs before x in time order (the convolution state; zeros when None).
    y[t, c] = act(sum_i w[c, i] * xx[t + i, c]) with xx = [x_prev; x].
    Returns (y [L, C], new state = the last W-1 rows of xx)."""
    x, w = _f64(x), _f64(w)
    L, C = x.shape
    W = w.shape[1]
    prev = np.zeros((W - 1, C)) if x_prev is None else _f64(x_prev).reshape(W - 1, C)
    xx = np.concatenate([prev, x], axis=0)
    y = np.zeros((L, C))
    for i in range(W):
        y += w[:, i][None, :] * xx[i:i + L]
    if act == "silu":
        y = y / (1.0 + np.exp(-y))
    elif act != "none":
        raise ValueError(act)
    return y, xx[L:].copy()


def round_to(x, dtype):
    """Round-to-nearest-even of fp64 values to the significand of `dtype`
    ('bf16': 8 significant bits, 'f32': 24), kept in fp64; None leaves x as it
    is.  (The normal range only: the values here are far from over- and
    underflow.)"""
    x = _f64(x)
    if dtype is None:
        return x
    bits = {"bf16": 8, "f32": 24}[dtype]
    m, e = np.frexp(x)                      # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, bits)), e - bits)   # rint: ties to even


def l2_normalize(x):
    """Each row divided by its L2 norm (rows of zeros stay zero)."""
    x = _f64(x)
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    return x / np.where(n > 0, n, 1.0)


def rms_norm_gated(o, w, gate, eps=RMS_EPS):
    """y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate), over the last axis."""
    o, w, gate = _f64(o), _f64(w), _f64(gate)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o * r * w * (1.0 / (1.0 + np.exp(-gate)))


def fused_inputs(xq, xk, xv, conv_w, conv_state=None, act="none", operand_dtype=None):
    """The recurrence's q, k, v for ONE (sequence, head) from its raw inputs:
    the short conv over the 2 dk + dv channels [q | k | v] (conv_w [2dk+dv, W],
    conv_state [2dk+dv, W-1] channel-major or None), then q and k
    L2-normalised, q scaled by 1/sqrt(dk).  The recurrence takes q, k, v in
    the call's element type, as every call of the library does
    (``operand_dtype`` 'bf16' / 'f32': rounded to it, ties to even; None:
    exact).  Returns (q, k, v, new conv state [2dk+dv, W-1])."""
    xq, xk, xv = _f64(xq), _f64(xk), _f64(xv)
    dk = xq.shape[1]
    x = np.concatenate([xq, xk, xv], axis=1)
    prev = None if conv_state is None else _f64(conv_state).T
    y, st = short_conv(x, conv_w, prev, act)
    q = round_to(l2_normalize(y[:, :dk]) / np.sqrt(dk), operand_dtype)
    k = round_to(l2_normalize(y[:, dk:2 * dk]), operand_dtype)
    return q, k, round_to(y[:, 2 * dk:], operand_dtype), st.T.copy()


def prefill_fused_pool(xq, xk, xv, g, beta, gate, conv_w, norm_w, cu_seqlens, init_slots,
                       state_pool, conv_pool, snap_interval=0, act="none", operand_dtype=None,
                       **kw):
    """What ``kda_prefill_varlen_fused`` must produce: per sequence b and head h,
    the conv starts from conv_pool[src_b, h] (zeros when src_b < 0), its new
    state goes to conv_pool[dst_b, h]; the conv outputs feed ``prefill_pool``
    (matrix states, snapshots, copy-on-write exactly as there); the outputs
    pass through ``rms_norm_gated``.  xq, xk, g: [T, H, dk]; xv, gate:
    [T, H, dv]; conv_w: [H, 2dk+dv, W]; norm_w: [dv]; conv_pool:
    [n_slots, H, 2dk+dv, W-1].  Returns (out, pool_after, conv_after, snaps)."""
    xq, xk, xv = _f64(xq), _f64(xk), _f64(xv)
    cw, cpool = _f64(conv_w), _f64(conv_pool)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    slots = np.asarray(init_slots, dtype=np.int64).reshape(-1, 2)
    T, H, dk = xq.shape
    dv = xv.shape[2]
    q, k, v = np.zeros((T, H, dk)), np.zeros((T, H, dk)), np.zeros((T, H, dv))
    conv_after = cpool.copy()
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        src, dst = int(slots[b, 0]), int(slots[b, 1])
        for h in range(H):
            st0 = cpool[src, h] if src >= 0 else None
            qb, kb, vb, st = fused_inputs(xq[t0:t1, h], xk[t0:t1, h], xv[t0:t1, h], cw[h], st0,
                                          act, operand_dtype)
            q[t0:t1, h], k[t0:t1, h], v[t0:t1, h] = qb, kb, vb
            conv_after[dst, h] = st
    o, after, snaps = prefill_pool(q, k, v, g, beta, cu, slots, state_pool, snap_interval, **kw)
    return rms_norm_gated(o, norm_w, gate), after, conv_after, snaps


def decode_fused_pool(xq, xk, xv, g, beta, gate, conv_w, norm_w, slot_ids, state_pool,
                      conv_pool, n_tok=1, act="none", operand_dtype=None, **kw):
    """What ``kda_decode_fused`` must produce: sequence n owns rows
    [n n_tok, (n+1) n_tok) and slot slot_ids[n] of both pools; its conv runs
    from conv_pool[slot] and the slot's conv state advances in place like the
    matrix state.  Returns (out, pool_after, conv_after)."""
    xq, xk, xv = _f64(xq), _f64(xk), _f64(xv)
    cw, cpool = _f64(conv_w), _f64(conv_pool)
    slots = np.asarray(slot_ids, dtype=np.int64).reshape(-1)
    N = len(slots)
    T, H, dk = xq.shape
    dv = xv.shape[2]
    q, k, v = np.zeros((T, H, dk)), np.zeros((T, H, dk)), np.zeros((T, H, dv))
    conv_after = cpool.copy()
    for n in range(N):
        r0, r1 = n * n_tok, (n + 1) * n_tok
        for h in range(H):
            qb, kb, vb, st = fused_inputs(xq[r0:r1, h], xk[r0:r1, h], xv[r0:r1, h], cw[h],
                                          cpool[slots[n], h], act, operand_dtype)
            q[r0:r1, h], k[r0:r1, h], v[r0:r1, h] = qb, kb, vb
            conv_after[slots[n], h] = st
    o, after, _ = decode_pool(q, k, v, g, beta, slots, state_pool, n_tok, False, **kw)
    return rms_norm_gated(o, norm_w, gate), after, conv_after


def rel_l2(x, ref) -> float:
    """Relative L2 error ||x - ref|| / ||ref|| over the finite entries of ref."""
    x = _f64(x)
    ref = _f64(ref)
    m = np.isfinite(ref)
    num = np.linalg.norm((x - ref)[m])
    den = np.linalg.norm(ref[m])
    return float(num / den) if den > 0 else float(num)
