"""GPU checks of kda_prefill_varlen_retain (snapshots written into pool slots
named by a retention map, or dropped) through the C ABI, on every prefill
kernel: a retained slot is bit-identical to the dense snapshot that
kda_prefill_varlen writes for the same inputs, dropped snapshots write
nothing, outputs and final states do not change, the result matches the
oracle, and bad maps are device-side errors."""

import pytest
import torch

import hybrid_linear_attention_delta_gb300 as kda
import oracle
from hybrid_linear_attention_delta_gb300 import inputs
from kda_cases import TOL, assert_untouched, gpu_prefill, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.lib()


def _case(dtype, d, H, lens, n_slots, slots, index=120):
    """d is dv; dk is 128 on the bf16 (chunked) path and d on the fp32 path."""
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
    dk = 128 if dtype == "bf16" else d
    tt = inputs.token_tensors(int(cu[-1]), H, dk, d, inputs.torch_dtype(dtype), index)
    pool = inputs.pool_states(n_slots, H, dk, d, index)
    return inputs.Batch(cu_seqlens=cu, init_slots=torch.tensor(slots, dtype=torch.int32),
                        pool=pool, **tt)


def _retain_map(n_snaps, free_slots, seed=5):
    """About half the snapshots retained, each into its own free slot."""
    gen = torch.Generator().manual_seed(seed)
    keep = torch.rand(n_snaps, generator=gen) < 0.5
    m = torch.full((n_snaps,), -1, dtype=torch.int32)
    m[keep] = torch.tensor(free_slots[:int(keep.sum())], dtype=torch.int32)
    return m


def _gpu_retain(b, interval, snap_slots, algo):
    d = {n: getattr(b, n).cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    pool = b.pool.cuda()
    T, H, dv = b.v.shape
    out = torch.empty((T, H, dv), dtype=b.q.dtype, device="cuda")
    B = b.cu_seqlens.numel() - 1
    ws = kda.workspace_for(B, H, pool.shape[0])
    kda.kda_prefill_varlen_retain(d["q"], d["k"], d["v"], d["g"], d["beta"], b.cu_seqlens.cuda(),
                                  b.init_slots.cuda(), pool, out, interval, snap_slots.cuda(),
                                  workspace=ws, algo=algo)
    return out, pool, kda.kda_device_status(ws)


CASES = [
    # (algo, dtype, d, H, interval): the token-recurrent kernel (fp32), the
    # per-state chunked kernel and the cooperative chunked kernel (bf16)
    (kda.KDA_ALGO_RECURRENT, "f32", 32, 3, 16),
    (kda.KDA_ALGO_CHUNKED_PER_STATE, "bf16", 128, 2, 64),
    (kda.KDA_ALGO_CHUNKED_COOP, "bf16", 128, 2, 64),
    (kda.KDA_ALGO_CHUNKED_COOP_HALVES, "bf16", 128, 2, 64),
    (kda.KDA_ALGO_CHUNKED_PER_STATE, "bf16", 64, 2, 128),   # dk = 128, dv = 64 below
]


@pytest.mark.parametrize("algo,dtype,d,H,interval", CASES)
def test_retained_slots_equal_dense_snapshots(algo, dtype, d, H, interval):
    lens = [300, 64, 129, 0, 700]
    slots = [[-1, 0], [7, 1], [-1, 2], [-1, 3], [8, 4]]
    n_slots = 60
    b = _case(dtype, d, H, lens, n_slots, slots)
    n_snaps = kda.kda_snapshot_count(b.cu_seqlens, interval)
    free = list(range(10, n_slots))
    smap = _retain_map(n_snaps, free)
    before = b.pool.clone()
    out_d, pool_d, snaps, (st, bits) = gpu_prefill(b, snap_interval=interval, algo=algo)
    assert st == kda.KDA_OK and bits == 0
    out_r, pool_r, (st, bits) = _gpu_retain(b, interval, smap, algo)
    assert st == kda.KDA_OK and bits == 0
    assert torch.equal(out_r, out_d)
    for s in range(n_snaps):
        if smap[s] >= 0:
            assert torch.equal(pool_r[int(smap[s])], snaps[s])
    for dst in range(5):
        assert torch.equal(pool_r[dst], pool_d[dst])
    retained = [int(x) for x in smap.tolist() if x >= 0]
    assert_untouched(pool_r, before, list(range(5)) + retained)
    # and against the oracle
    ro, rpool = oracle.prefill_pool_retain(b.q, b.k, b.v, b.g, b.beta, b.cu_seqlens.numpy(),
                                           b.init_slots.numpy(), b.pool, interval, smap.numpy())
    assert rel(out_r, ro) <= TOL[dtype]
    assert rel(pool_r[retained], rpool[retained]) <= TOL[dtype]


def test_retaining_nothing_writes_only_destinations():
    lens = [256, 100]
    b = _case("bf16", 128, 2, lens, 12, [[-1, 0], [5, 1]], index=121)
    before = b.pool.clone()
    smap = torch.full((kda.kda_snapshot_count(b.cu_seqlens, 64),), -1, dtype=torch.int32)
    _, pool, (st, bits) = _gpu_retain(b, 64, smap, kda.KDA_ALGO_AUTO)
    assert st == kda.KDA_OK and bits == 0
    assert_untouched(pool, before, [0, 1])


def test_bad_retention_maps_are_device_checks():
    """Each bad map refuses the sequence that owns the offending snapshot:
    that sequence writes nothing (destination and retained snapshots stay
    bit-identical), and the error bit names the failed check."""
    lens = [128, 128]
    b = _case("bf16", 128, 2, lens, 10, [[-1, 0], [3, 1]], index=122)
    # interval 64: two snapshots per sequence, entries (seq 0: 0, 1; seq 1: 2, 3)
    before = b.pool.clone()
    cases = [
        # map, error bit, slots the refused sequence would have written
        ([5, 1, 6, 7], 2, [0, 5]),      # seq 0 snapshot on seq 1's destination
        ([5, 6, 3, 7], 2, [1, 3, 7]),   # seq 1 snapshot on its own source
        ([5, 6, 6, -1], 2, []),         # two snapshots on one slot (either may lose)
        ([5, 10, 7, 8], 1, [0, 5]),     # slot out of range
        ([5, 6, -2, 8], 1, [1, 8]),     # below -1
    ]
    for smap, bit, kept in cases:
        _, pool, (st, bits) = _gpu_retain(b, 64, torch.tensor(smap, dtype=torch.int32),
                                          kda.KDA_ALGO_AUTO)
        assert st == kda.KDA_ERR_DEVICE_CHECK and bits & bit, (smap, bits)
        for slot in kept:
            assert torch.equal(pool[slot].cpu(), before[slot]), (smap, slot)
    _, _, (st, bits) = _gpu_retain(b, 64, torch.tensor([5, -1, 6, 7], dtype=torch.int32),
                                   kda.KDA_ALGO_AUTO)
    assert st == kda.KDA_OK and bits == 0
