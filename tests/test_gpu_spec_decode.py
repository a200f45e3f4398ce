"""GPU parity of kda_decode_spec (speculative verify with the commit of the
previous step's accepted tokens) against the fp64 oracle, through the C ABI;
its layout rules bit-exact (a commit equals the per-token-state rollback of
kda_decode, slots outside the call and slots with nothing accepted are
untouched) and its device-side check of the accepted lengths."""

import pytest
import torch

import hybrid_linear_attention_delta_gb300 as kda
import oracle
from hybrid_linear_attention_delta_gb300 import inputs
from kda_cases import TOL, assert_untouched, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.lib()


def _case(N, n_prev, n_tok, H, n_slots, dtype, d, index=93):
    dt = inputs.torch_dtype(dtype)
    prev = inputs.token_tensors(N * n_prev, H, d, d, dt, index)
    cur = inputs.token_tensors(N * n_tok, H, d, d, dt, index + 1)
    pool = inputs.pool_states(n_slots, H, d, d, index)
    gen = torch.Generator().manual_seed(index)
    slots = torch.randperm(n_slots, generator=gen)[:N].to(torch.int32)
    acc = torch.randint(0, n_prev + 1, (N,), generator=gen).to(torch.int32)
    acc[0] = 0
    if N > 1:
        acc[1] = n_prev
    return prev, cur, pool, slots, acc


def _gpu_spec(prev, cur, pool, slots, acc, n_prev, n_tok, out_fill=float("nan")):
    c = {n: t.cuda().contiguous() for n, t in cur.items()}
    p = {n: t.cuda().contiguous() for n, t in prev.items()}
    pool_d = pool.cuda()
    slots_d = slots.cuda()
    N = slots.numel()
    H, d = pool.shape[1], pool.shape[2]
    dt = next(iter(prev.values())).dtype
    out = torch.full((N * n_tok, H, d), out_fill, dtype=dt, device="cuda")
    ws = kda.workspace_for(N, H, pool.shape[0])
    kda.kda_decode_spec(c["q"] if n_tok else None, c["k"] if n_tok else None,
                        c["v"] if n_tok else None, c["g"] if n_tok else None,
                        c["beta"] if n_tok else None, slots_d, pool_d,
                        out if n_tok else None, n_tok,
                        p["k"] if n_prev else None, p["v"] if n_prev else None,
                        p["g"] if n_prev else None, p["beta"] if n_prev else None,
                        acc.cuda() if n_prev else None, n_prev, workspace=ws,
                        H=H, dk=d, dv=d, dtype=kda.KDA_BF16 if dt == torch.bfloat16 else kda.KDA_F32)
    st, bits = kda.kda_device_status(ws)
    return out, pool_d, (st, bits)


def _oracle_spec(prev, cur, pool, slots, acc, n_prev, n_tok):
    return oracle.decode_spec_pool(cur["q"], cur["k"], cur["v"], cur["g"], cur["beta"],
                                   slots.numpy(), pool, n_tok, prev["k"], prev["v"], prev["g"],
                                   prev["beta"], acc.numpy(), n_prev)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 128), ("f32", 64), ("bf16", 32)])
def test_spec_decode_matches_oracle(dtype, d):
    """8 sequences, 8 previous tokens with accepted lengths in [0, 8]
    (including 0 and 8), 8 new tokens; the 128 x 128 kernel and the
    token-recurrent kernel."""
    N, n_prev, n_tok, H, n_slots = 8, 8, 8, 4, 20
    prev, cur, pool, slots, acc = _case(N, n_prev, n_tok, H, n_slots, dtype, d)
    before = pool.clone()
    out, pool_d, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert st == kda.KDA_OK and bits == 0
    assert kda.kda_last_launch_count() == 1
    ro, rpool = _oracle_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert rel(out, ro) <= TOL[dtype]
    committed = [int(s) for s, a in zip(slots.tolist(), acc.tolist()) if a > 0]
    assert rel(pool_d[committed], rpool[committed]) <= TOL[dtype]
    # slots with nothing accepted and slots outside the call: bit-identical
    assert_untouched(pool_d, before, committed)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_spec_previous_and_current_steps_differ_in_length(dtype, d):
    """7 tokens in the previous step (6 drafts + 1), 8 in this one: the
    previous step's rows are read with their own stride."""
    N, n_prev, n_tok, H, n_slots = 6, 7, 8, 2, 16
    prev, cur, pool, slots, acc = _case(N, n_prev, n_tok, H, n_slots, dtype, d, index=103)
    out, pool_d, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert st == kda.KDA_OK and bits == 0
    ro, rpool = _oracle_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert rel(out, ro) <= TOL[dtype]
    committed = [int(s) for s, a in zip(slots.tolist(), acc.tolist()) if a > 0]
    assert rel(pool_d[committed], rpool[committed]) <= TOL[dtype]


@pytest.mark.parametrize("d", [128, 64])
def test_commit_equals_per_token_rollback_bit_exact(d):
    """A commit of a tokens writes exactly the state kda_decode reports after
    token a-1 of the same step (same kernel arithmetic, bit for bit)."""
    N, n_prev, H, n_slots = 6, 8, 2, 12
    prev, cur, pool, slots, acc = _case(N, n_prev, 1, H, n_slots, "bf16", d, index=95)
    p = {n: t.cuda().contiguous() for n, t in prev.items()}
    per = torch.full((N, n_prev, H, d, d), float("nan"), device="cuda")
    pool_a = pool.cuda()
    out_a = torch.empty((N * n_prev, H, d), dtype=torch.bfloat16, device="cuda")
    ws = kda.workspace_for(N, H, n_slots)
    kda.kda_decode(p["q"], p["k"], p["v"], p["g"], p["beta"], slots.cuda(), pool_a, out_a,
                   n_prev, per, workspace=ws)
    _, pool_b, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, n_prev, 0)
    assert st == kda.KDA_OK and bits == 0
    for n in range(N):
        s, a = int(slots[n]), int(acc[n])
        want = per[n, a - 1] if a > 0 else pool[s].cuda()
        assert torch.equal(pool_b[s], want)


def test_verify_only_leaves_pool_bit_identical():
    N, n_tok, H, n_slots = 5, 8, 4, 9
    prev, cur, pool, slots, acc = _case(N, 1, n_tok, H, n_slots, "bf16", 128, index=97)
    out, pool_d, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, 0, n_tok)
    assert st == kda.KDA_OK and bits == 0
    assert torch.equal(pool_d.cpu(), pool)
    ro, _ = _oracle_spec(prev, cur, pool, slots, acc, 0, n_tok)
    assert rel(out, ro) <= TOL["bf16"]


def test_spec_full_size_64x8():
    """64 sequences x 32 heads, 8 previous and 8 new tokens on a 1024-slot
    pool (the verify workload's size); every output and committed state
    against the oracle (run on the touched slots, remapped to 0..N-1)."""
    N, n_prev, n_tok, H, n_slots = 64, 8, 8, 32, 1024
    prev, cur, pool, slots, acc = _case(N, n_prev, n_tok, H, n_slots, "bf16", 128, index=99)
    before = pool.clone()
    out, pool_d, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert st == kda.KDA_OK and bits == 0
    sub = pool[slots.long()]
    ro, rpool = _oracle_spec(prev, cur, sub, torch.arange(N, dtype=torch.int32), acc, n_prev,
                             n_tok)
    assert rel(out, ro) <= TOL["bf16"]
    assert rel(pool_d[slots.long()], rpool) <= TOL["bf16"]
    committed = [int(s) for s, a in zip(slots.tolist(), acc.tolist()) if a > 0]
    assert_untouched(pool_d, before, committed)


def test_accepted_length_out_of_range_is_a_device_check():
    """An accepted length above n_prev (or below 0) is refused on the device:
    bit 64 is reported and that sequence's slot and outputs stay unwritten;
    the other sequences complete."""
    N, n_prev, n_tok, H, n_slots = 4, 4, 2, 2, 8
    prev, cur, pool, slots, acc = _case(N, n_prev, n_tok, H, n_slots, "bf16", 128, index=101)
    acc = torch.tensor([5, 2, -1, 4], dtype=torch.int32)
    out, pool_d, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert st == kda.KDA_ERR_DEVICE_CHECK and bits & 64
    for n in (0, 2):
        assert torch.equal(pool_d[int(slots[n])].cpu(), pool[int(slots[n])])
        assert torch.isnan(out[n * n_tok:(n + 1) * n_tok].float()).all()
    ok = torch.tensor([1, 3])
    ro, rpool = _oracle_spec(prev, cur, pool, slots, torch.tensor([0, 2, 0, 4], dtype=torch.int32),
                             n_prev, n_tok)
    for n in ok.tolist():
        s = int(slots[n])
        assert rel(pool_d[s], rpool[s]) <= TOL["bf16"]
        assert rel(out[n * n_tok:(n + 1) * n_tok], ro[n * n_tok:(n + 1) * n_tok]) <= TOL["bf16"]
    # the record is cleared: a clean call reports OK
    acc = torch.tensor([1, 2, 3, 4], dtype=torch.int32)
    _, _, (st, bits) = _gpu_spec(prev, cur, pool, slots, acc, n_prev, n_tok)
    assert st == kda.KDA_OK and bits == 0
