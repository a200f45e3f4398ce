"""GPU parity of the layer around the recurrence -- the short causal
convolution with its per-slot state before it and the gated RMSNorm after it
-- against the fp64 oracle (oracle.prefill_fused_pool / decode_fused_pool),
through the C ABI: the fused decode (one launch) and the fused prefill
(convolution, convolution states, prefill, gated RMSNorm), in both chunked
variants and the fp32 path, with copy-on-write resume of both states,
snapshots, in-place extension, and a decode that continues a prefill.

The recurrence takes q, k, v in the call's element type, in the fused layer as
in every other call, so the oracle rounds the convolution's outputs to that
type (its own fp64 arithmetic, ties to even) where the layer hands them on."""

import numpy as np
import pytest
import torch

import hybrid_linear_attention_delta_gb300 as kda
import oracle
from hybrid_linear_attention_delta_gb300 import inputs
from kda_cases import TOL, assert_untouched, rel, worst_state, worst_unit

pytestmark = pytest.mark.gpu
PER = kda.KDA_ALGO_CHUNKED_PER_STATE
COOP = kda.KDA_ALGO_CHUNKED_COOP
HALVES = kda.KDA_ALGO_CHUNKED_COOP_HALVES


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.lib()


def _prefill_case(lens, H, n_slots, slots, dtype="bf16", d=128, index=95):
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
    T = int(cu[-1])
    dt = inputs.torch_dtype(dtype)
    tt = inputs.token_tensors(T, H, d, d, dt, index)
    ft = inputs.fused_tensors(T, H, d, d, dt, index, n_slots)
    pool = inputs.pool_states(n_slots, H, d, d, index)
    return cu, torch.tensor(slots, dtype=torch.int32), tt, ft, pool


def _run_prefill(cu, slots, tt, ft, pool, snap, algo=kda.KDA_ALGO_AUTO, act="none"):
    dev = {n: t.cuda() for n, t in tt.items()}
    f = {n: t.cuda().contiguous() for n, t in ft.items()}
    T, H, d = dev["q"].shape
    dv = dev["v"].shape[2]
    pool_d = pool.cuda()
    out = torch.empty((T, H, dv), dtype=dev["q"].dtype, device="cuda")
    n_snaps = kda.kda_snapshot_count(cu, snap)
    snaps = torch.full((n_snaps, H, d, dv), float("nan"), device="cuda") if snap else None
    ws = kda.workspace_for(len(cu) - 1, H, pool.shape[0])
    kda.kda_prefill_varlen_fused(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], f["gate"],
                                 f["conv_w"], f["norm_w"], cu.cuda(), slots.cuda(), pool_d,
                                 f["conv_pool"], out, snap, snaps, workspace=ws, algo=algo,
                                 conv_act=act)
    st = kda.kda_device_status(ws)
    return out, pool_d, f["conv_pool"], snaps, st


def _dt(t):
    """The element type the recurrence takes its q, k, v in (the call's)."""
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def _oracle_prefill(cu, slots, tt, ft, pool, snap, act="none"):
    return oracle.prefill_fused_pool(tt["q"], tt["k"], tt["v"], tt["g"], tt["beta"], ft["gate"],
                                     ft["conv_w"], ft["norm_w"], cu.numpy(), slots.numpy(), pool,
                                     ft["conv_pool"], snap, act=act, operand_dtype=_dt(tt["q"]))


def _touched(slots):
    return sorted(set(int(s) for s in slots[:, 1].tolist()))


@pytest.mark.parametrize("algo,act", [(PER, "none"), (COOP, "none"), (HALVES, "none"),
                                      (PER, "silu"), (COOP, "silu")],
                         ids=["per_state", "coop", "halves", "per_state_silu", "coop_silu"])
def test_fused_prefill_matches_oracle(algo, act):
    """A varlen batch with ragged tails, a short sequence (shorter than the
    convolution), resumed and fresh sequences, one extended in place: outputs,
    matrix states, snapshots and convolution states against the oracle; the
    convolution states are raw inputs moved, so they match bit for bit."""
    lens = [200, 2, 130, 64]
    slots = [[3, 3], [5, 6], [-1, 7], [1, 0]]
    cu, sl, tt, ft, pool = _prefill_case(lens, 3, 9, slots)
    before, cbefore = pool.clone(), ft["conv_pool"].clone()
    out, p, cp, snaps, (st, bits) = _run_prefill(cu, sl, tt, ft, pool, 64, algo, act)
    assert st == kda.KDA_OK and bits == 0
    ro, rpool, rconv, rsn = _oracle_prefill(cu, sl, tt, ft, pool, 64, act)
    tol = TOL["bf16"]
    touched = _touched(sl)
    assert rel(out, ro) <= tol, rel(out, ro)
    assert worst_unit(out, ro, cu.numpy(), 3) <= 2 * tol
    assert rel(p[touched], rpool[touched]) <= tol
    assert worst_state(p[touched], rpool[touched]) <= 2 * tol
    assert rel(snaps, rsn) <= tol
    got = cp.float().cpu().numpy()
    np.testing.assert_array_equal(got[touched], rconv[touched])
    assert_untouched(p, before, touched)
    assert_untouched(cp, cbefore, touched)


def test_fused_prefill_fp32_path():
    """fp32 inputs take the exact token-recurrent path: 1e-5."""
    lens = [37, 64, 3]
    slots = [[2, 0], [-1, 1], [4, 4]]
    cu, sl, tt, ft, pool = _prefill_case(lens, 2, 6, slots, dtype="f32", d=32)
    out, p, cp, snaps, (st, bits) = _run_prefill(cu, sl, tt, ft, pool, 16)
    assert st == kda.KDA_OK and bits == 0
    ro, rpool, rconv, rsn = _oracle_prefill(cu, sl, tt, ft, pool, 16)
    touched = _touched(sl)
    assert rel(out, ro) <= TOL["f32"]
    assert rel(p[touched], rpool[touched]) <= TOL["f32"]
    assert rel(snaps, rsn) <= TOL["f32"]
    np.testing.assert_array_equal(cp.cpu().numpy()[touched], rconv[touched])


@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (16, "f32")])
def test_fused_prefill_narrow_heads(d, dtype):
    """Heads of 64 and 16 channels: the gated RMSNorm's rows then take two
    elements per lane, or one on half of the lanes."""
    lens = [90, 1, 33]
    slots = [[0, 0], [-1, 1], [2, 3]]
    cu, sl, tt, ft, pool = _prefill_case(lens, 3, 5, slots, dtype=dtype, d=d)
    out, p, cp, snaps, (st, bits) = _run_prefill(cu, sl, tt, ft, pool, 32, act="silu")
    assert st == kda.KDA_OK and bits == 0
    ro, rpool, rconv, rsn = _oracle_prefill(cu, sl, tt, ft, pool, 32, act="silu")
    touched = _touched(sl)
    tol = TOL[dtype]
    assert rel(out, ro) <= tol, rel(out, ro)
    assert worst_unit(out, ro, cu.numpy(), 3) <= 2 * tol
    assert rel(p[touched], rpool[touched]) <= tol
    assert rel(snaps, rsn) <= tol
    np.testing.assert_array_equal(cp.float().cpu().numpy()[touched], rconv[touched])


@pytest.mark.parametrize("n_tok,act,dtype", [(1, "none", "bf16"), (4, "silu", "bf16"),
                                             (3, "none", "f32")])
def test_fused_decode_matches_oracle(n_tok, act, dtype):
    N, H, n_slots = 24, 4, 40
    dt = inputs.torch_dtype(dtype)
    tt = inputs.token_tensors(N * n_tok, H, 128, 128, dt, 96)
    ft = inputs.fused_tensors(N * n_tok, H, 128, 128, dt, 96, n_slots)
    pool = inputs.pool_states(n_slots, H, 128, 128, 96)
    slots = torch.randperm(n_slots, generator=torch.Generator().manual_seed(96))[:N].to(torch.int32)
    dev = {n: t.cuda() for n, t in tt.items()}
    f = {n: t.cuda().contiguous() for n, t in ft.items()}
    pool_d = pool.cuda()
    out = torch.empty_like(dev["v"])
    per = torch.empty((N, n_tok, H, 128, 128), device="cuda")
    ws = kda.workspace_for(N, H, n_slots)
    kda.kda_decode_fused(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], f["gate"],
                         f["conv_w"], f["norm_w"], slots.cuda(), pool_d, f["conv_pool"], out,
                         n_tok, per, workspace=ws, conv_act=act)
    st, bits = kda.kda_device_status(ws)
    assert st == kda.KDA_OK and bits == 0
    ro, rpool, rconv = oracle.decode_fused_pool(tt["q"], tt["k"], tt["v"], tt["g"], tt["beta"],
                                                ft["gate"], ft["conv_w"], ft["norm_w"],
                                                slots.numpy(), pool, ft["conv_pool"], n_tok,
                                                act=act, operand_dtype=_dt(tt["q"]))
    tol = TOL["bf16"] if dtype == "bf16" else TOL["f32"]
    sl = slots.long()
    assert rel(out, ro) <= tol, rel(out, ro)
    assert rel(pool_d[sl], rpool[slots.numpy()]) <= tol
    assert worst_state(pool_d[sl], rpool[slots.numpy()]) <= 2 * tol
    np.testing.assert_array_equal(f["conv_pool"].float().cpu().numpy()[slots.numpy()],
                                  rconv[slots.numpy()])
    assert torch.equal(pool_d[sl].cpu(), per[:, -1].cpu())
    assert_untouched(pool_d, pool, slots.tolist())
    assert_untouched(f["conv_pool"], ft["conv_pool"], slots.tolist())


def test_fused_decode_continues_a_fused_prefill():
    """A fused prefill of L tokens into a slot, then 3 fused decode steps on it,
    gives what the oracle gives for one prefill of L + 3 tokens: the outputs of
    the 3 decoded tokens, the matrix state and the convolution state (both
    states carry over from prefill to decode)."""
    L, H = 150, 2
    cu, sl, tt, ft, pool = _prefill_case([L + 3], H, 4, [[1, 2]], index=97)
    ro, rpool, rconv, _ = _oracle_prefill(cu, sl, tt, ft, pool, 0)
    head = {n: t[:L] for n, t in tt.items()}
    fhead = dict(ft, gate=ft["gate"][:L])
    _, p1, c1, _, st = _run_prefill(torch.tensor([0, L], dtype=torch.int32), sl, head, fhead,
                                    pool, 0)
    assert st == (0, 0)
    ws = kda.workspace_for(1, H, 4)
    slot = torch.tensor([2], dtype=torch.int32, device="cuda")
    cw, nw = ft["conv_w"].cuda(), ft["norm_w"].cuda()
    outs = []
    for j in range(3):
        r = slice(L + j, L + j + 1)
        d = {n: t[r].cuda().contiguous() for n, t in tt.items()}
        o = torch.empty_like(d["v"])
        kda.kda_decode_fused(d["q"], d["k"], d["v"], d["g"], d["beta"],
                             ft["gate"][r].cuda().contiguous(), cw, nw, slot, p1, c1, o, 1,
                             workspace=ws)
        outs.append(o)
    assert kda.kda_device_status(ws) == (0, 0)
    assert rel(torch.cat(outs), ro[L:]) <= TOL["bf16"]
    assert rel(p1[2], rpool[2]) <= TOL["bf16"]
    np.testing.assert_array_equal(c1[2].float().cpu().numpy(), rconv[2])


def test_fused_decode_full_size_256x32():
    """The batched decode workload (256 sequences x 32 heads, 1024-slot pool)
    through the fused decode: every output, state and convolution state."""
    w = inputs.WORKLOADS["decode_256x1"]
    b = inputs.make_batch(w)
    ft = inputs.fused_tensors(w.B, w.H, 128, 128, torch.bfloat16, w.index, w.n_slots)
    dev = {n: getattr(b, n).cuda() for n in ("q", "k", "v", "g", "beta")}
    f = {n: t.cuda().contiguous() for n, t in ft.items()}
    pool_d = b.pool.cuda()
    out = torch.empty_like(dev["v"])
    ws = kda.workspace_for(w.B, w.H, w.n_slots)
    kda.kda_decode_fused(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], f["gate"],
                         f["conv_w"], f["norm_w"], b.slot_ids.cuda(), pool_d, f["conv_pool"], out,
                         1, workspace=ws)
    assert kda.kda_device_status(ws) == (0, 0)
    sub_pool = b.pool[b.slot_ids.long()]
    sub_conv = ft["conv_pool"][b.slot_ids.long()]
    ro, rpool, rconv = oracle.decode_fused_pool(b.q, b.k, b.v, b.g, b.beta, ft["gate"],
                                                ft["conv_w"], ft["norm_w"], list(range(w.B)),
                                                sub_pool, sub_conv, 1, operand_dtype="bf16")
    sl = b.slot_ids.long()
    assert rel(out, ro) <= TOL["bf16"]
    assert rel(pool_d[sl], rpool) <= TOL["bf16"]
    assert worst_state(pool_d[sl], rpool) <= 2 * TOL["bf16"]
    np.testing.assert_array_equal(f["conv_pool"][sl].float().cpu().numpy(), rconv)


@pytest.mark.slow
def test_fused_prefill_8k_full():
    """The 8k-token workload (B=1, T=8192, H=32, snapshots every 1024) through
    the fused prefill, the raw inputs drawn as the workload's q, k, v: every
    output, snapshot and final state against the oracle, and the new
    convolution state bit for bit."""
    w = inputs.WORKLOADS["prefill_8k"]
    b = inputs.make_batch(w)
    T, H = b.q.shape[:2]
    ft = inputs.fused_tensors(T, H, w.dk, w.dv, torch.bfloat16, w.index, b.pool.shape[0])
    tt = {n: getattr(b, n) for n in ("q", "k", "v", "g", "beta")}
    out, p, cp, snaps, (st, bits) = _run_prefill(b.cu_seqlens, b.init_slots, tt, ft, b.pool,
                                                  w.snap_interval)
    assert st == kda.KDA_OK and bits == 0
    ro, rpool, rconv, rsn = _oracle_prefill(b.cu_seqlens, b.init_slots, tt, ft, b.pool,
                                            w.snap_interval)
    touched = _touched(b.init_slots)
    tol = TOL["bf16"]
    e = rel(out, ro)
    print(f"fused prefill 8k: out {e:.2e}")
    assert e <= tol
    assert worst_unit(out, ro, b.cu_seqlens.numpy(), H) <= 2 * tol
    assert rel(p[touched], rpool[touched]) <= tol
    assert worst_state(p[touched], rpool[touched]) <= 2 * tol
    assert rel(snaps, rsn) <= tol
    assert worst_state(snaps, rsn) <= 2 * tol
    np.testing.assert_array_equal(cp.float().cpu().numpy()[touched], rconv[touched])
