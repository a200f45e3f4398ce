"""The benchmark's own arithmetic on CPU: the algorithmic byte and flop counts
behind every roofline fraction, checked against figures computed by hand from
the per-unit counts (1282 B per token-head for bf16 at dk = dv = 128, 64 KiB
per fp32 state), and the retention map the `--retain` option builds."""

import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from hybrid_linear_attention_delta_gb300 import inputs  # noqa: E402

STATE = 128 * 128 * 4  # one fp32 state, bytes


def test_prefill_bytes_and_flops_8k():
    """8192 tokens x 32 heads at 1282 B, plus 9 states per head (8 snapshots
    and the final state); flops 180,224 per token-head at chunk 64."""
    w = inputs.WORKLOADS["prefill_8k"]
    nbytes, flops, token_bytes = bench.prefill_algorithmic(w, [8192], 8, 0, 2)
    assert token_bytes == 8192 * 32 * 1282 == 336_068_608
    assert nbytes == 336_068_608 + 32 * 9 * STATE == 354_942_976
    assert flops == 8192 * 32 * 180_224 == 47_244_640_256


def test_prefill_bytes_and_flops_1m():
    """The headline workload: 2^20 tokens x 16 heads at 1282 B, plus 33 states
    per head (32 snapshots and the final state)."""
    w = inputs.WORKLOADS["prefill_1m"]
    nbytes, flops, token_bytes = bench.prefill_algorithmic(w, [1 << 20], 32, 0, 2)
    assert token_bytes == (1 << 20) * 16 * 1282 == 21_508_390_912
    assert nbytes == 21_508_390_912 + 16 * 33 * STATE == 21_542_993_920
    assert flops == (1 << 20) * 16 * 180_224 == 3_023_656_976_384


def test_prefill_bytes_count_resumed_states():
    w = inputs.WORKLOADS["varlen_resume"]
    nbytes, _, _ = bench.prefill_algorithmic(w, [512, 1000], 5, 1, 2)
    assert nbytes == 1512 * 32 * 1282 + 32 * STATE * (2 + 5 + 1)


def test_decode_bytes():
    """256 x 1: 132,354 B per state (read + write + one token's I/O);
    64 x 8 with per-token states: 8 more state writes per state."""
    w1 = inputs.WORKLOADS["decode_256x1"]
    assert bench.decode_algorithmic(w1, 256, 1, False, 2) == 256 * 32 * 132_354 == 1_084_243_968
    w8 = inputs.WORKLOADS["verify_64x8"]
    per_state = 2 * STATE + 8 * 1282 + 8 * STATE
    assert bench.decode_algorithmic(w8, 64, 8, True, 2) == 64 * 32 * per_state == 1_363_181_568


def test_speculative_verify_bytes():
    """One state read per (sequence, head); one write only where something was
    accepted; the replayed tokens carry k, g, v, beta (385 bf16 values), the
    verified ones the full 1282 B."""
    w = inputs.WORKLOADS["spec_verify_64x8"]
    acc = torch.tensor([0, 3, 8, 1], dtype=torch.int32)
    got = bench.spec_algorithmic(w, 4, acc, 2)
    want = 4 * 32 * STATE + 3 * 32 * STATE + 12 * 32 * 385 * 2 + 4 * 8 * 32 * 1282
    assert got == want


def test_retention_map_keeps_every_nth_into_free_slots():
    lens = [300, 64, 129, 1000]
    cu = torch.tensor([0] + list(torch.cumsum(torch.tensor(lens), 0)), dtype=torch.int32)
    slots = torch.tensor([[5, 0], [-1, 1], [2, 2], [-1, 3]], dtype=torch.int32)
    b = inputs.Batch(q=None, k=None, v=None, g=None, beta=None, cu_seqlens=cu,
                     init_slots=slots)
    m = bench.retention_map(b, 64, 2, 40)
    per_seq = [n // 64 for n in lens]
    assert m.numel() == sum(per_seq)
    off = 0
    for cnt in per_seq:
        for j in range(cnt):
            assert (m[off + j] >= 0) == ((j + 1) % 2 == 0)
        off += cnt
    kept = [int(x) for x in m.tolist() if x >= 0]
    assert len(kept) == len(set(kept))                  # distinct
    assert not set(kept) & {0, 1, 2, 3, 5}              # no source or destination
    assert all(0 <= s < 40 for s in kept)


def test_retention_map_refuses_a_pool_without_room():
    import pytest
    cu = torch.tensor([0, 512], dtype=torch.int32)
    slots = torch.tensor([[-1, 0]], dtype=torch.int32)
    b = inputs.Batch(q=None, k=None, v=None, g=None, beta=None, cu_seqlens=cu,
                     init_slots=slots)
    with pytest.raises(ValueError):
        bench.retention_map(b, 64, 2, 1)   # 4 kept snapshots, no free slot
