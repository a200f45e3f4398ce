"""GPU parity of the token-recurrent prefill kernel and the decode kernels
against the fp64 oracle, through the C ABI, plus the pool/slot layout rules
(bit-exact) and the device-side argument checks."""

import numpy as np
import pytest
import torch

import hybrid_linear_attention_delta_gb300 as kda
from hybrid_linear_attention_delta_gb300 import inputs
from kda_cases import (TOL, assert_untouched, gpu_decode, gpu_prefill, oracle_decode,
                       oracle_prefill, rel, touched_slots, worst_state, worst_unit)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.lib()


def _custom(dtype, dk, dv, H, lens, n_slots, slots, index=90):
    """A scaled case drawn with the standard recipe, explicit lengths and slots."""
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
    tt = inputs.token_tensors(int(cu[-1]), H, dk, dv, inputs.torch_dtype(dtype), index)
    pool = inputs.pool_states(n_slots, H, dk, dv, index)
    return inputs.Batch(cu_seqlens=cu, init_slots=torch.tensor(slots, dtype=torch.int32),
                        pool=pool, **tt)


def test_tiny_fp32_prefill():
    """B=1, T=64, H=2, dk=dv=16, fp32, zero initial state (relative L2 <= 1e-5)."""
    b = inputs.make_batch(inputs.WORKLOADS["tiny_f32"])
    out, pool, _, (st, bits) = gpu_prefill(b)
    ro, rpool, _ = oracle_prefill(b)
    assert st == kda.KDA_OK and bits == 0
    assert rel(out, ro) <= TOL["f32"]
    assert rel(pool, rpool) <= TOL["f32"]
    assert kda.kda_last_launch_count() == 2


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (128, 128), (128, 16)])
def test_fp32_varlen_resume_snapshots(dk, dv):
    lens = [37, 0, 64, 130, 5]
    slots = [[3, 7], [-1, 0], [2, 2], [-1, 9], [5, 4]]
    b = _custom("f32", dk, dv, 3, lens, 12, slots)
    before = b.pool.clone()
    out, pool, snaps, (st, bits) = gpu_prefill(b, snap_interval=16,
                                               algo=kda.KDA_ALGO_RECURRENT)
    ro, rpool, rsn = oracle_prefill(b, 16)
    assert st == kda.KDA_OK and bits == 0
    assert rel(out, ro) <= TOL["f32"]
    for s in touched_slots(b):
        assert rel(pool[s], rpool[s]) <= TOL["f32"]
    assert rel(snaps, rsn) <= TOL["f32"]
    assert_untouched(pool, before, touched_slots(b))
    # copy-on-write: the resumed-from slots that are not destinations are bit-identical
    for src in (3, 5):
        assert torch.equal(pool[src].cpu(), before[src])


def test_bf16_recurrent_prefill_matches_oracle():
    lens = [200, 77, 1]
    slots = [[-1, 0], [4, 1], [-1, 2]]
    b = _custom("bf16", 128, 128, 4, lens, 6, slots)
    out, pool, snaps, (st, bits) = gpu_prefill(b, snap_interval=64, algo=kda.KDA_ALGO_RECURRENT)
    ro, rpool, rsn = oracle_prefill(b, 64)
    assert st == kda.KDA_OK and bits == 0
    assert rel(out, ro) <= TOL["bf16"]
    assert worst_unit(out, ro, b.cu_seqlens.numpy(), 4) <= 2 * TOL["bf16"]
    for s in (0, 1, 2):
        assert rel(pool[s], rpool[s]) <= TOL["bf16"]
    assert rel(snaps, rsn) <= TOL["bf16"]


def _decode_case(N, n_tok, H, n_slots, dtype="bf16", d=128, index=91):
    tt = inputs.token_tensors(N * n_tok, H, d, d, inputs.torch_dtype(dtype), index)
    pool = inputs.pool_states(n_slots, H, d, d, index)
    gen = torch.Generator().manual_seed(index)
    slot_ids = torch.randperm(n_slots, generator=gen)[:N].to(torch.int32)
    cu = torch.arange(N + 1, dtype=torch.int32) * n_tok
    return inputs.Batch(cu_seqlens=cu, slot_ids=slot_ids, pool=pool, **tt)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 128), ("f32", 64), ("bf16", 32)])
def test_decode_single_token(dtype, d):
    b = _decode_case(24, 1, 4, 40, dtype, d)
    before = b.pool.clone()
    out, pool, _, (st, bits) = gpu_decode(b)
    ro, rpool, _ = oracle_decode(b)
    assert st == kda.KDA_OK and bits == 0
    assert rel(out, ro) <= TOL[dtype]
    assert rel(pool[b.slot_ids.long()], rpool[b.slot_ids.numpy()]) <= TOL[dtype]
    assert_untouched(pool, before, touched_slots(b))


@pytest.mark.parametrize("d", [128, 64])
def test_decode_verify_per_token_states(d):
    b = _decode_case(8, 8, 4, 20, "bf16", d)
    out, pool, per, (st, bits) = gpu_decode(b, n_tok=8, per_tok=True)
    ro, rpool, rper = oracle_decode(b, 8, True)
    assert st == kda.KDA_OK and bits == 0
    assert rel(out, ro) <= TOL["bf16"]
    assert rel(per, rper) <= TOL["bf16"]
    assert rel(pool[b.slot_ids.long()], rpool[b.slot_ids.numpy()]) <= TOL["bf16"]
    # the slot holds exactly the state after the last token
    last = per[:, -1].cpu()
    assert torch.equal(pool[b.slot_ids.long()].cpu(), last)


def test_decode_multi_token_equals_repeated_single():
    """n_tok = 8 in one call is bit-identical to 8 single-token calls."""
    b = _decode_case(6, 8, 2, 10, "bf16", 128)
    out8, pool8, _, _ = gpu_decode(b, n_tok=8)
    d = {k: getattr(b, k).cuda() for k in ("q", "k", "v", "g", "beta")}
    pool = b.pool.cuda()
    slots = b.slot_ids.cuda()
    ws = kda.workspace_for(6, 2, 10)
    for j in range(8):
        rows = torch.arange(6) * 8 + j
        o = torch.empty((6, 2, 128), dtype=torch.bfloat16, device="cuda")
        kda.kda_decode(*(d[x][rows.cuda()].contiguous() for x in ("q", "k", "v", "g", "beta")),
                       slots, pool, o, 1, None, workspace=ws)
        assert torch.equal(o.cpu(), out8[rows.cuda()].cpu())
    assert torch.equal(pool.cpu(), pool8.cpu())


def test_decode_full_size_256x32():
    """256 sequences x 32 heads on a 1024-slot pool (the batched decode
    workload), every output and touched state against the oracle."""
    w = inputs.WORKLOADS["decode_256x1"]
    b = inputs.make_batch(w)
    before = b.pool.clone()
    out, pool, _, (st, bits) = gpu_decode(b)
    assert st == kda.KDA_OK and bits == 0
    # the oracle runs on the touched slots only (remapped to 0..N-1)
    sub = inputs.Batch(q=b.q, k=b.k, v=b.v, g=b.g, beta=b.beta, cu_seqlens=b.cu_seqlens,
                       slot_ids=torch.arange(256, dtype=torch.int32),
                       pool=b.pool[b.slot_ids.long()])
    ro, rpool, _ = oracle_decode(sub)
    assert rel(out, ro) <= TOL["bf16"]
    assert rel(pool[b.slot_ids.long()], rpool) <= TOL["bf16"]
    assert_untouched(pool, before, touched_slots(b))


def test_decode_verify_full_size_64x8():
    """64 sequences x 8 tokens x 32 heads with per-token states on a 1024-slot
    pool (the speculative-verify workload, 1 GiB of per-token states): every
    output, every per-token state and every advanced slot against the oracle,
    each (sequence, token, head) state and each (sequence, head) output block
    within 2 tol; the slot holds the last per-token state bit for bit."""
    w = inputs.WORKLOADS["verify_64x8"]
    b = inputs.make_batch(w)
    before = b.pool.clone()
    out, pool, per, (st, bits) = gpu_decode(b, n_tok=w.n_tok, per_tok=True)
    assert st == kda.KDA_OK and bits == 0
    N, n_tok, H = w.B, w.n_tok, w.H
    sub = inputs.Batch(q=b.q, k=b.k, v=b.v, g=b.g, beta=b.beta, cu_seqlens=b.cu_seqlens,
                       slot_ids=torch.arange(N, dtype=torch.int32),
                       pool=b.pool[b.slot_ids.long()])
    ro, rpool, rper = oracle_decode(sub, n_tok, True)
    tol = TOL["bf16"]
    assert rel(out, ro) <= tol
    assert worst_unit(out, ro, b.cu_seqlens.numpy(), H) <= 2 * tol
    per_h = per.cpu()
    assert rel(per_h, rper) <= tol
    assert worst_state(per_h.reshape(N * n_tok, H, 128, 128),
                       rper.reshape(N * n_tok, H, 128, 128)) <= 2 * tol
    slots = b.slot_ids.long()
    assert rel(pool[slots], rpool) <= tol
    assert worst_state(pool[slots], rpool) <= 2 * tol
    assert torch.equal(pool[slots].cpu(), per_h[:, -1])
    assert_untouched(pool, before, touched_slots(b))


def test_decode_device_checks():
    b = _decode_case(4, 1, 2, 8, "bf16", 128)
    b.slot_ids = torch.tensor([3, 3, 6, 1], dtype=torch.int32)   # duplicate
    _, pool, _, (st, bits) = gpu_decode(b)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 2
    b.slot_ids = torch.tensor([3, 1000, 6, -1], dtype=torch.int32)  # out of range
    before = b.pool.clone()
    _, pool, _, (st, bits) = gpu_decode(b)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 1
    assert_untouched(pool, before, [3, 6])
    # a clean call afterwards reports OK (the record was cleared)
    b.slot_ids = torch.tensor([0, 1, 2, 4], dtype=torch.int32)
    _, _, _, (st, bits) = gpu_decode(b)
    assert st == kda.KDA_OK and bits == 0


def test_prefill_device_checks():
    lens = [10, 20]
    b = _custom("bf16", 128, 128, 2, lens, 6, [[-1, 1], [-1, 1]])  # duplicate destination
    _, _, _, (st, bits) = gpu_prefill(b)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 2
    b = _custom("bf16", 128, 128, 2, lens, 6, [[2, 1], [-1, 2]])   # src is another's dst
    _, _, _, (st, bits) = gpu_prefill(b)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 2
    b = _custom("bf16", 128, 128, 2, lens, 6, [[-1, 9], [-1, 2]])  # dst out of range
    before = b.pool.clone()
    _, pool, _, (st, bits) = gpu_prefill(b)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 1
    assert_untouched(pool, before, [2])
    # non-monotone cu_seqlens: nothing is written
    b = _custom("bf16", 128, 128, 2, lens, 6, [[-1, 1], [-1, 2]])
    b.cu_seqlens = torch.tensor([0, 25, 30], dtype=torch.int32)
    before = b.pool.clone()
    b.cu_seqlens[1] = 31
    _, pool, _, (st, bits) = gpu_prefill(b)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 4
    assert torch.equal(pool.cpu(), before)


def test_recurrent_prefill_is_deterministic():
    b = _custom("bf16", 128, 128, 2, [70, 33], 4, [[-1, 0], [3, 1]])
    o1, p1, _, _ = gpu_prefill(b, algo=kda.KDA_ALGO_RECURRENT)
    o2, p2, _, _ = gpu_prefill(b, algo=kda.KDA_ALGO_RECURRENT)
    assert torch.equal(o1.cpu(), o2.cpu()) and torch.equal(p1.cpu(), p2.cpu())
