"""GPU parity of the tcgen05 chunked prefill against the fp64 oracle (through
the C ABI), plus its layout rules: snapshot placement, copy-on-write resume,
untouched slots, split invariance and run-to-run determinism (bit-exact)."""

import numpy as np
import pytest
import torch

import hybrid_linear_attention_delta_gb300 as kda
import oracle
from hybrid_linear_attention_delta_gb300 import inputs
from kda_cases import (TOL, RelL2, assert_untouched, gpu_prefill, oracle_prefill, rel,
                       touched_slots, worst_state, worst_unit)

pytestmark = pytest.mark.gpu
CH = kda.KDA_ALGO_CHUNKED
PER = kda.KDA_ALGO_CHUNKED_PER_STATE
COOP = kda.KDA_ALGO_CHUNKED_COOP
HALVES = kda.KDA_ALGO_CHUNKED_COOP_HALVES
MODES = pytest.mark.parametrize("mode", [PER, COOP, HALVES], ids=["per_state", "coop", "halves"])


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.lib()


def _case(lens, H, n_slots, slots, dv=128, index=92):
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
    tt = inputs.token_tensors(int(cu[-1]), H, 128, dv, torch.bfloat16, index)
    pool = inputs.pool_states(n_slots, H, 128, dv, index)
    return inputs.Batch(cu_seqlens=cu, init_slots=torch.tensor(slots, dtype=torch.int32),
                        pool=pool, **tt)


def _check(b, snap, out, pool, snaps, tol=TOL["bf16"]):
    """Whole tensors within tol, and every (sequence, head) block of the
    outputs, of the touched final states and of the snapshots within 2 tol."""
    ro, rpool, rsn = oracle_prefill(b, snap)
    H = b.q.shape[1]
    e_out = rel(out, ro)
    touched = touched_slots(b)
    e_state = max(rel(pool[s], rpool[s]) for s in touched)
    assert e_out <= tol, f"out rel L2 {e_out:.2e}"
    assert e_state <= tol, f"state rel L2 {e_state:.2e}"
    assert worst_unit(out, ro, b.cu_seqlens.numpy(), H) <= 2 * tol
    assert worst_state(pool[touched], rpool[touched]) <= 2 * tol
    if snap:
        e_sn = rel(snaps, rsn)
        assert e_sn <= tol, f"snapshot rel L2 {e_sn:.2e}"
        if rsn.shape[0]:
            assert worst_state(snaps, rsn) <= 2 * tol
    return e_out, e_state


@MODES
@pytest.mark.parametrize("lens", [[64], [1], [63, 65], [200, 130, 7], [129, 0, 256]])
def test_chunked_ragged_varlen(lens, mode):
    """Ragged tails and empty sequences, in both chunked variants (the
    per-state one with narrow 64-column dv blocks)."""
    B = len(lens)
    slots = [[-1, b] for b in range(B)]
    b = _case(lens, 3, B + 2, slots)
    out, pool, snaps, (st, bits) = gpu_prefill(b, 64, algo=mode)
    assert st == kda.KDA_OK and bits == 0
    _check(b, 64, out, pool, snaps)


def test_chunked_resume_cow_wide_blocks():
    """Copy-on-write resume from cached slots with B*H >= 148 (128-column dv
    blocks): sources stay bit-identical, untouched slots stay bit-identical."""
    lens = [70, 130, 64, 1, 200, 33, 128, 90]
    slots = [[3, 20], [-1, 21], [5, 22], [-1, 23], [7, 24], [9, 9], [-1, 26], [11, 27]]
    b = _case(lens, 20, 30, slots)
    before = b.pool.clone()
    out, pool, snaps, (st, bits) = gpu_prefill(b, 64, algo=CH)
    assert st == kda.KDA_OK and bits == 0
    _check(b, 64, out, pool, snaps)
    assert_untouched(pool, before, touched_slots(b))
    for src in (3, 5, 7, 11):
        assert torch.equal(pool[src].cpu(), before[src])


def test_chunked_dv64_heads():
    lens = [150, 64]
    b = _case(lens, 4, 4, [[1, 2], [-1, 3]], dv=64)
    out, pool, snaps, (st, bits) = gpu_prefill(b, 128, algo=CH)
    assert st == kda.KDA_OK and bits == 0
    _check(b, 128, out, pool, snaps)


@MODES
def test_chunked_matches_recurrent_path(mode):
    lens = [300, 77]
    b = _case(lens, 4, 4, [[0, 2], [-1, 3]])
    o1, p1, s1, _ = gpu_prefill(b, 64, algo=mode)
    o2, p2, s2, _ = gpu_prefill(b, 64, algo=kda.KDA_ALGO_RECURRENT)
    assert rel(o1, o2.float().cpu().numpy()) <= TOL["bf16"]
    assert rel(s1, s2.cpu().numpy()) <= TOL["bf16"]
    assert rel(p1[2:4], p2[2:4].cpu().numpy()) <= TOL["bf16"]


@MODES
def test_chunked_snapshot_equals_prefix_final_state(mode):
    """Snapshot j is bit-identical to the final state of a prefill of the
    first (j+1)*interval tokens (same kernel path, same chunking)."""
    L, I = 320, 64
    b = _case([L], 2, 2, [[-1, 0]])
    _, _, snaps, _ = gpu_prefill(b, I, algo=mode)
    for j in range(L // I):
        n = (j + 1) * I
        bj = inputs.Batch(q=b.q[:n], k=b.k[:n], v=b.v[:n], g=b.g[:n], beta=b.beta[:n],
                          cu_seqlens=torch.tensor([0, n], dtype=torch.int32),
                          init_slots=b.init_slots, pool=b.pool)
        _, pj, _, _ = gpu_prefill(bj, 0, algo=mode)
        assert torch.equal(snaps[j].cpu(), pj[0].cpu()), f"snapshot {j}"


@MODES
def test_chunked_resume_chain_is_exact_on_chunk_boundaries(mode):
    """prefill(L1) -> slot, then prefill(L2) from that slot equals prefill(L1+L2)
    bit for bit when L1 is a multiple of the chunk (the state round-trips
    through the fp32 pool exactly)."""
    L1, L2 = 128, 100
    b = _case([L1 + L2], 2, 3, [[-1, 0]])
    o_all, p_all, _, _ = gpu_prefill(b, 0, algo=mode)
    b1 = inputs.Batch(q=b.q[:L1], k=b.k[:L1], v=b.v[:L1], g=b.g[:L1], beta=b.beta[:L1],
                      cu_seqlens=torch.tensor([0, L1], dtype=torch.int32),
                      init_slots=torch.tensor([[-1, 1]], dtype=torch.int32), pool=b.pool)
    o1, p1, _, _ = gpu_prefill(b1, 0, algo=mode)
    b2 = inputs.Batch(q=b.q[L1:], k=b.k[L1:], v=b.v[L1:], g=b.g[L1:], beta=b.beta[L1:],
                      cu_seqlens=torch.tensor([0, L2], dtype=torch.int32),
                      init_slots=torch.tensor([[1, 2]], dtype=torch.int32),
                      pool=p1.cpu())
    o2, p2, _, _ = gpu_prefill(b2, 0, algo=mode)
    assert torch.equal(torch.cat([o1, o2]).cpu(), o_all.cpu())
    assert torch.equal(p2[2].cpu(), p_all[0].cpu())


@MODES
def test_chunked_deterministic(mode):
    """Bit-identical across runs (the cooperative variant's producers take
    chunks in a different order every run; each package is computed the same)."""
    b = _case([500, 64], 3, 4, [[2, 0], [-1, 1]])
    o1, p1, s1, _ = gpu_prefill(b, 64, algo=mode)
    o2, p2, s2, _ = gpu_prefill(b, 64, algo=mode)
    assert torch.equal(o1.cpu(), o2.cpu()) and torch.equal(p1.cpu(), p2.cpu())
    assert torch.equal(s1.cpu(), s2.cpu())


def test_auto_selects_chunked_for_bf16_128():
    b = _case([100], 2, 1, [[-1, 0]])
    o_auto, _, _, _ = gpu_prefill(b, 0)
    o_ch, _, _, _ = gpu_prefill(b, 0, algo=CH)
    o_coop, _, _, _ = gpu_prefill(b, 0, algo=COOP)
    o_half, _, _, _ = gpu_prefill(b, 0, algo=HALVES)
    assert torch.equal(o_auto.cpu(), o_ch.cpu())
    # few (sequence, head) pairs: cooperative, here with two chain CTAs per pair
    assert torch.equal(o_auto.cpu(), o_half.cpu())
    assert rel(o_half, o_coop.float().cpu().numpy()) <= TOL["bf16"]


def test_coop_and_per_state_agree_with_resume():
    """Both variants of the chunked prefill, on a resumed varlen batch with
    snapshots, agree with each other to the bf16 tolerance (their arithmetic
    differs: the cooperative one expands U = U~ - W S')."""
    lens = [400, 129, 64]
    b = _case(lens, 8, 8, [[5, 0], [-1, 1], [6, 2]])
    o1, p1, s1, st1 = gpu_prefill(b, 128, algo=PER)
    o2, p2, s2, st2 = gpu_prefill(b, 128, algo=COOP)
    o3, p3, s3, st3 = gpu_prefill(b, 128, algo=HALVES)
    assert st1 == (0, 0) and st2 == (0, 0) and st3 == (0, 0)
    for o, p, sn in ((o2, p2, s2), (o3, p3, s3)):
        assert rel(o, o1.float().cpu().numpy()) <= TOL["bf16"]
        assert rel(sn, s1.cpu().numpy()) <= TOL["bf16"]
        assert rel(p[:3], p1[:3].cpu().numpy()) <= TOL["bf16"]
        _check(b, 128, o, p, sn)


def test_coop_refused_for_many_pairs():
    """More than 64 (sequence, head) pairs: the cooperative variant does not
    apply and forcing it is refused up front."""
    b = _case([64] * 5, 16, 6, [[-1, i] for i in range(5)])
    for algo in (COOP, HALVES):
        with pytest.raises(kda.KdaError) as e:
            gpu_prefill(b, 0, algo=algo)
        assert e.value.status == kda.KDA_ERR_UNSUPPORTED


def test_halves_with_most_pairs():
    """64 pairs, the most the cooperative grid serves, with two chain CTAs
    each: 128 chain CTAs and the remaining SMs as producers."""
    b = _case([64, 130, 1, 200], 16, 5, [[-1, 0], [4, 1], [-1, 2], [3, 3]])
    out, pool, snaps, st = gpu_prefill(b, 64, algo=HALVES)
    assert st == (0, 0)
    _check(b, 64, out, pool, snaps)


# ------------------------------------------------------------ full-size workloads

def test_prefill_8k_full():
    """B=1, T=8192, H=32, dk=dv=128, snapshots every 1024: every output, the
    8 snapshots and the final state against the oracle (all heads)."""
    w = inputs.WORKLOADS["prefill_8k"]
    b = inputs.make_batch(w)
    out, pool, snaps, (st, bits) = gpu_prefill(b, w.snap_interval)
    assert st == kda.KDA_OK and bits == 0
    assert snaps.shape[0] == 8
    e_out, e_state = _check(b, w.snap_interval, out, pool, snaps)
    print(f"prefill_8k: out {e_out:.2e} state {e_state:.2e}")


def _check_by_sequence(b, snap, out, pool, snaps, tol=TOL["bf16"]):
    """The checks of _check for a large batch, with the oracle run one
    sequence at a time (all its heads in parallel) so that its fp64 copies stay
    a few GB: whole-tensor errors accumulated over the sequences within tol,
    every (sequence, head) block of outputs, snapshots and final states within
    2 tol.  Returns (out, snapshots, states, worst unit) errors."""
    H = b.q.shape[1]
    cu = b.cu_seqlens.numpy()
    off, n_total = oracle.snapshot_offsets(cu, snap)
    if snap:
        assert snaps.shape[0] == n_total
    e_out, e_snap, e_state = RelL2(), RelL2(), RelL2()
    worst = 0.0
    for s in range(len(cu) - 1):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        sub = {n: getattr(b, n)[t0:t1] for n in ("q", "k", "v", "g", "beta")}
        src, dst = int(b.init_slots[s, 0]), int(b.init_slots[s, 1])
        init = None if src < 0 else b.pool[src][None]
        res = oracle.run(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], [0, t1 - t0],
                         init, snap)
        o = out[t0:t1].float().cpu().numpy()
        e_out.add(o, res.out)
        for h in range(H):
            worst = max(worst, oracle.rel_l2(o[:, h], res.out[:, h]))
        e_state.add(pool[dst].cpu(), res.final[0])
        worst = max(worst, worst_state(pool[dst:dst + 1], res.final))
        n = (t1 - t0) // snap if snap else 0
        if n:
            sn = snaps[off[s]:off[s] + n]
            e_snap.add(sn.cpu(), res.snaps)
            worst = max(worst, worst_state(sn, res.snaps))
    assert e_out.value <= tol and e_state.value <= tol, (e_out.value, e_state.value)
    assert e_snap.value <= tol, e_snap.value
    assert worst <= 2 * tol, worst
    return e_out.value, e_snap.value, e_state.value, worst


def test_varlen_resume_full():
    """16 sequences, L ~ U[512, 32768], 8 resumed from a 1024-slot pool, snapshots
    every 256, all 32 heads: every output, every snapshot and every touched final
    state against the oracle (per sequence; see _check_by_sequence); sources of
    resumed sequences and untouched slots bit-identical."""
    w = inputs.WORKLOADS["varlen_resume"]
    b = inputs.make_batch(w)
    before = b.pool.clone()
    out, pool, snaps, (st, bits) = gpu_prefill(b, w.snap_interval)
    assert st == kda.KDA_OK and bits == 0
    e = _check_by_sequence(b, w.snap_interval, out, pool, snaps)
    print("varlen_resume: out %.2e snaps %.2e states %.2e worst unit %.2e" % e)
    assert_untouched(pool, before, touched_slots(b))
    for s in range(w.B):
        src = int(b.init_slots[s, 0])
        if src >= 0:
            assert torch.equal(pool[src].cpu(), before[src])


def test_prefill_3x32k_full():
    """Three 32768-token sequences at H = 32: 96 (sequence, head) pairs, more
    than the cooperative mode serves and fewer than the SMs, so the per-state
    kernel runs one 128-column CTA per pair.  Every output, snapshot and final
    state against the oracle (per sequence; see _check_by_sequence)."""
    w = inputs.WORKLOADS["prefill_3x32k"]
    b = inputs.make_batch(w)
    out, pool, snaps, (st, bits) = gpu_prefill(b, w.snap_interval)
    assert st == kda.KDA_OK and bits == 0
    e = _check_by_sequence(b, w.snap_interval, out, pool, snaps)
    print("prefill_3x32k: out %.2e snaps %.2e states %.2e worst unit %.2e" % e)


@pytest.mark.slow
def test_prefill_1m_full():
    """B=1, T=2^20, H=16, snapshots every 32768 (inputs drawn on the GPU): every
    output, all 32 snapshots and the final state of every head and column
    against the oracle.  The oracle runs two heads at a time over all 2^20
    tokens (16 independent column blocks, one per host thread); whole-tensor
    errors are accumulated and every head's outputs, snapshots and final state
    are bounded by 2 tol."""
    w = inputs.WORKLOADS["prefill_1m"]
    b = inputs.make_batch(w, device="cuda")
    out, pool, snaps, (st, bits) = gpu_prefill(b, w.snap_interval)
    assert st == kda.KDA_OK and bits == 0
    assert snaps.shape[0] == 32
    tol = TOL["bf16"]
    e_out, e_snap, e_state = RelL2(), RelL2(), RelL2()
    worst = 0.0
    for h0 in range(0, w.H, 2):
        hs = slice(h0, h0 + 2)
        sub = {n: getattr(b, n)[:, hs].cpu() for n in ("q", "k", "v", "g", "beta")}
        res = oracle.run(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], [0, w.T], None,
                         w.snap_interval)
        del sub
        o = out[:, hs].float().cpu().numpy()
        e_out.add(o, res.out)
        sn = snaps[:, hs].cpu().numpy()
        e_snap.add(sn, res.snaps)
        fin = pool[0, hs].cpu().numpy()
        e_state.add(fin, res.final[0])
        for i in range(2):
            worst = max(worst, oracle.rel_l2(o[:, i], res.out[:, i]),
                        oracle.rel_l2(fin[i], res.final[0, i]))
        worst = max(worst, worst_state(sn, res.snaps))
        del o, sn, res
    print(f"prefill_1m: out {e_out.value:.2e} snaps {e_snap.value:.2e} "
          f"state {e_state.value:.2e} worst unit {worst:.2e}")
    assert e_out.value <= tol and e_snap.value <= tol and e_state.value <= tol
    assert worst <= 2 * tol


@MODES
@pytest.mark.parametrize("in_place", [False, True], ids=["cow", "in_place"])
def test_chunked_exact_for_decays_beyond_its_range(mode, in_place):
    """Two g = -60 gates of one channel within 32 tokens (and a g = -1000 gate
    in another sequence) push the chunked algorithm's scaled operands beyond
    fp32 range.  The call still returns the recurrence's result: the chunked
    kernel hands those (sequence, head) units to the exact token-recurrent
    kernel in the same call (status OK, no error bit), including the
    snapshots, a resumed start state and in-place extension (src == dst, whose
    source must survive the chunked pass); the untouched units keep the
    chunked result, bit for bit."""
    lens = [300, 130, 96]
    slots = [[2, 2], [-1, 3], [4, 5]] if in_place else [[2, 0], [-1, 3], [4, 5]]
    b = _case(lens, 3, 6, slots)
    b.g = b.g.clone()
    b.g[10, 0, 5] = -60.0          # sequence 0, head 0: two large decays
    b.g[20, 0, 5] = -60.0
    b.g[300 + 40, 2, 7] = -1000.0  # sequence 1, head 2: e^g = 0 exactly
    out, pool, snaps, (st, bits) = gpu_prefill(b, 64, algo=mode)
    assert st == kda.KDA_OK and bits == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(pool).all()
    assert torch.isfinite(snaps).all()
    _check(b, 64, out, pool, snaps)
    # the units that stayed in range are those of an unmodified batch, bit for bit
    b2 = _case(lens, 3, 6, slots)
    o2, p2, s2, _ = gpu_prefill(b2, 64, algo=mode)
    keep = [(1, 0), (1, 1), (2, 0), (2, 1), (2, 2), (0, 1), (0, 2)]
    cu = b.cu_seqlens.tolist()
    for (s, h) in keep:
        assert torch.equal(out[cu[s]:cu[s + 1], h].cpu(), o2[cu[s]:cu[s + 1], h].cpu()), (s, h)


@MODES
def test_chunked_single_large_gate_is_exact(mode):
    """One g = -60 gate (the state of that channel is wiped at one token) stays
    inside the chunked algorithm's range: no flag, no inf/NaN, oracle parity."""
    b = _case([200], 2, 1, [[-1, 0]])
    b.g = b.g.clone()
    b.g[70, 1, 3] = -60.0
    out, pool, snaps, (st, bits) = gpu_prefill(b, 64, algo=mode)
    assert st == kda.KDA_OK and bits == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(pool).all()
    _check(b, 64, out, pool, snaps)
