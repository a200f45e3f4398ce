"""kda_decode_noalloc: the decode entry point for callers that may not
allocate device memory (a framework that owns every device buffer through its
own pool, or a latency path where cudaMalloc, which can synchronise the
device, is not allowed).  It must give what kda_decode gives, call after
call, without the caller's workspace.

This file is named so that pytest collects it last; it passes on its own in
a fresh process (where its first call performs the per-device set-up) and
after the rest of the suite."""

import pytest
import torch

import hybrid_linear_attention_delta_gb300 as kda
from hybrid_linear_attention_delta_gb300 import inputs
from kda_cases import TOL, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.lib()


def _case(N, n_tok, H, n_slots, index=93):
    tt = inputs.token_tensors(N * n_tok, H, 128, 128, torch.bfloat16, index, device="cuda")
    pool = inputs.pool_states(n_slots, H, 128, 128, index, device="cuda")
    gen = torch.Generator().manual_seed(index)
    slots = torch.randperm(n_slots, generator=gen)[:N].to(torch.int32).cuda()
    return tt, pool, slots


@pytest.mark.parametrize("n_tok,per_tok", [(1, False), (4, True)])
def test_noalloc_decode_matches_workspace_decode_twice(n_tok, per_tok):
    N, H, n_slots = 24, 4, 40
    tt, pool, slots = _case(N, n_tok, H, n_slots)
    pool_ref, pool_na = pool.clone(), pool.clone()
    ws = kda.workspace_for(N, H, n_slots)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(2):  # two calls in a row, each continuing from the last state
        o_ref = torch.empty_like(tt["v"])
        o_na = torch.empty_like(tt["v"])
        per_ref = per_na = None
        if per_tok:
            per_ref = torch.empty((N, n_tok, H, 128, 128), device="cuda")
            per_na = torch.empty_like(per_ref)
        kda.kda_decode(tt["q"], tt["k"], tt["v"], tt["g"], tt["beta"], slots, pool_ref, o_ref,
                       n_tok, per_ref, workspace=ws)
        kda.kda_decode_noalloc(tt["q"], tt["k"], tt["v"], tt["g"], tt["beta"], slots, pool_na,
                               o_na, n_tok, per_na, err)
        torch.cuda.synchronize()
        # the same decode kernel runs on the same inputs: identical bits, and
        # the bf16 tolerance the suite uses holds a fortiori
        assert torch.equal(o_na.cpu(), o_ref.cpu()), step
        assert torch.equal(pool_na.cpu(), pool_ref.cpu()), step
        assert rel(o_na, o_ref.float().cpu().numpy()) <= TOL["bf16"], step
        if per_tok:
            assert torch.equal(per_na.cpu(), per_ref.cpu()), step
    assert int(err.item()) == 0
    assert kda.kda_device_status(ws)[0] == kda.KDA_OK


def test_noalloc_reports_duplicate_slots_and_rejects_oversize():
    N, H, n_slots = 4, 2, 8
    tt, pool, _ = _case(N, 1, H, n_slots)
    slots = torch.tensor([1, 1, 5, 6], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(tt["v"])
    kda.kda_decode_noalloc(tt["q"], tt["k"], tt["v"], tt["g"], tt["beta"], slots, pool, out, 1,
                           None, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 2
    # without an err_bits tensor the binding makes one and returns it
    bits = kda.kda_decode_noalloc(tt["q"], tt["k"], tt["v"], tt["g"], tt["beta"], slots, pool,
                                  out, 1)
    assert int(bits.item()) & 2
    # a pool beyond the shared claim table (n_slots * H > 131072) is refused up front
    big = torch.empty((1, 1, 1, 1), device="cuda")
    a = kda.make_args(B=N, T_total=N, H=H, dk=128, dv=128, n_slots=70000,
                      dtype=kda.KDA_BF16)
    st = kda.lib().kda_decode_noalloc(tt["q"].data_ptr(), tt["k"].data_ptr(),
                                      tt["v"].data_ptr(), tt["g"].data_ptr(),
                                      tt["beta"].data_ptr(), slots.data_ptr(), big.data_ptr(),
                                      out.data_ptr(), 1, None, None, kda.ctypes.byref(a))
    assert st == kda.KDA_ERR_INVALID_ARG
