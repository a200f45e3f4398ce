"""Shared helpers of the test suite: run the library on seeded inputs and run
the oracle on the same inputs.  Nothing here computes KDA itself."""

from __future__ import annotations

import numpy as np
import torch

import hybrid_linear_attention_delta_gb300 as kda
import oracle
from hybrid_linear_attention_delta_gb300 import inputs

TOL = {"f32": 1e-5, "bf16": 5e-3}   # relative L2 bars for the two paths


def to_dev(b: inputs.Batch, device="cuda"):
    out = {}
    for name in ("q", "k", "v", "g", "beta", "pool"):
        out[name] = getattr(b, name).to(device).contiguous()
    out["cu"] = b.cu_seqlens.to(device)
    if b.init_slots is not None:
        out["init_slots"] = b.init_slots.to(device).contiguous()
    if b.slot_ids is not None:
        out["slot_ids"] = b.slot_ids.to(device).contiguous()
    return out


def gpu_prefill(b: inputs.Batch, snap_interval=0, algo=kda.KDA_ALGO_AUTO, device="cuda",
                workspace=None, pool=None):
    d = to_dev(b, device)
    if pool is not None:
        d["pool"] = pool
    T, H, _ = d["q"].shape
    dv = d["v"].shape[2]
    dk = d["k"].shape[2]
    out = torch.empty((T, H, dv), dtype=d["q"].dtype, device=device)
    n_snaps = kda.kda_snapshot_count(b.cu_seqlens, snap_interval)
    snaps = (torch.full((n_snaps, H, dk, dv), float("nan"), device=device)
             if snap_interval else None)
    B = b.cu_seqlens.numel() - 1
    ws = workspace if workspace is not None else kda.workspace_for(B, H, d["pool"].shape[0],
                                                                   device)
    kda.kda_prefill_varlen(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"],
                           d["init_slots"], d["pool"], out, snap_interval, snaps, workspace=ws,
                           algo=algo)
    st, bits = kda.kda_device_status(ws)
    return out, d["pool"], snaps, (st, bits)


def oracle_prefill(b: inputs.Batch, snap_interval=0, **kw):
    return oracle.prefill_pool(b.q, b.k, b.v, b.g, b.beta, b.cu_seqlens.numpy(),
                               b.init_slots.numpy(), b.pool, snap_interval, **kw)


def gpu_decode(b: inputs.Batch, n_tok=1, per_tok=False, device="cuda", workspace=None):
    d = to_dev(b, device)
    T, H, _ = d["q"].shape
    dk, dv = d["k"].shape[2], d["v"].shape[2]
    N = d["slot_ids"].numel()
    out = torch.empty((T, H, dv), dtype=d["q"].dtype, device=device)
    pts = (torch.full((N, n_tok, H, dk, dv), float("nan"), device=device) if per_tok else None)
    ws = workspace if workspace is not None else kda.workspace_for(N, H, d["pool"].shape[0],
                                                                   device)
    kda.kda_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["slot_ids"], d["pool"], out,
                   n_tok, pts, workspace=ws)
    st, bits = kda.kda_device_status(ws)
    return out, d["pool"], pts, (st, bits)


def oracle_decode(b: inputs.Batch, n_tok=1, per_tok=False, **kw):
    return oracle.decode_pool(b.q, b.k, b.v, b.g, b.beta, b.slot_ids.numpy(), b.pool, n_tok,
                              per_tok, **kw)


def rel(x, ref) -> float:
    if isinstance(x, torch.Tensor):
        x = x.detach().float().cpu().numpy()
    return oracle.rel_l2(x, ref)


def touched_slots(b: inputs.Batch):
    if b.init_slots is not None:
        return sorted(set(int(s) for s in b.init_slots[:, 1].tolist()))
    return sorted(int(s) for s in b.slot_ids.tolist())


def assert_untouched(pool_after: torch.Tensor, pool_before: torch.Tensor, touched):
    keep = torch.ones(pool_before.shape[0], dtype=torch.bool)
    keep[list(touched)] = False
    idx = torch.nonzero(keep).flatten()
    a = pool_after.detach().cpu()[idx]
    bb = pool_before.detach().cpu()[idx]
    assert torch.equal(a.contiguous().view(torch.uint8), bb.contiguous().view(torch.uint8)), \
        "untouched slots changed"


def worst_unit(x, ref, cu, H):
    """Worst relative L2 over (sequence, head) blocks of a [T, H, d] output."""
    x = np.asarray(x if not isinstance(x, torch.Tensor) else x.float().cpu().numpy())
    worst = 0.0
    for b in range(len(cu) - 1):
        for h in range(H):
            t0, t1 = int(cu[b]), int(cu[b + 1])
            if t1 > t0:
                worst = max(worst, oracle.rel_l2(x[t0:t1, h], ref[t0:t1, h]))
    return worst


def worst_state(x, ref):
    """Worst relative L2 over the (index, head) blocks of [n, H, dk, dv] states
    (final states of touched slots, snapshots or per-token states), so that one
    bad (sequence, head) state is not diluted into a tensor-wide figure."""
    x = np.asarray(x if not isinstance(x, torch.Tensor) else x.detach().float().cpu().numpy())
    ref = np.asarray(ref)
    worst = 0.0
    for i in range(ref.shape[0]):
        for h in range(ref.shape[1]):
            worst = max(worst, oracle.rel_l2(x[i, h], ref[i, h]))
    return worst


class RelL2:
    """Relative L2 accumulated over pieces of one tensor compared piece by
    piece (sum of squared differences over sum of squared references)."""

    def __init__(self):
        self.num = 0.0
        self.den = 0.0

    def add(self, x, ref):
        x = np.asarray(x if not isinstance(x, torch.Tensor) else x.detach().float().cpu().numpy(),
                       dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        self.num += float(np.sum((x - ref) ** 2))
        self.den += float(np.sum(ref ** 2))
        return oracle.rel_l2(x, ref)

    @property
    def value(self):
        return (self.num / self.den) ** 0.5 if self.den > 0 else self.num ** 0.5
