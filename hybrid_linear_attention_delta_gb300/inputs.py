"""Seeded synthetic inputs for the KDA library and its oracle.

This module draws random numbers and lays them out; it holds none of the KDA
arithmetic.  Both the GPU tests/benchmark and the fp64 oracle take their
inputs from here (the oracle only ever sees copies of these tensors).

Recipe (the same for every workload; sizes come from ``WORKLOADS``):

* q, k ~ N(0, 1) per element, then L2-normalised over dk for each (token,
  head); q is further scaled by 1/sqrt(dk).  v ~ N(0, 1).
* g = -exp(N(-3, 1)) per (token, head, channel): a log-decay, used as given.
* beta = sigmoid(N(0, 1)) per (token, head).
* All five are cast to the workload dtype (bf16 or fp32) at the end; the oracle
  reads the cast values back exactly.
* Pool states ~ N(0, 0.1) (standard deviation 0.1), fp32.
* Speculative verify with commit: the previous step's tokens are drawn with
  the same recipe under the workload index + 100, and its accepted lengths
  are integers uniform in [1, n_tok] (the first verified token is always
  kept).
* Each field has its own ``torch.Generator`` seeded with
  ``(20260000 + workload_index) * 100 + field_id`` so fields do not depend on
  the order they are drawn in (a varlen batch needs its lengths before the
  token tensors).
* The layer around the recurrence (short convolution, gated RMSNorm;
  ``fused_tensors``): the raw inputs are q, k, v drawn as above (the
  convolution mixes them, and q and k are normalised again after it), the
  gate logits ~ N(0, 1) per (token, head, value column), the convolution taps
  ~ N(0, 0.5^2) per (head, channel, tap), the RMSNorm weight 1 + N(0, 0.1^2)
  per value column, and the slots' convolution states ~ N(0, 1) raw inputs.
* Large tensors are drawn in token blocks on ``device`` (the CPU by default;
  the benchmark and the full-size tests draw on the GPU for speed).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

F_Q, F_K, F_V, F_G, F_BETA, F_LENS, F_SLOTS, F_POOL, F_RESUME, F_ACCEPT = range(10)
F_GATE, F_CONVW, F_NORMW, F_CONVPOOL = range(10, 14)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    kind: str                     # "prefill" or "decode"
    H: int
    dk: int
    dv: int
    dtype: str                    # "f32" or "bf16"
    B: int = 1
    T: int = 0                    # single-sequence length (prefill, B=1)
    lens_range: Optional[tuple] = None   # varlen: lengths uniform in [lo, hi]
    snap_interval: int = 0
    chunk: int = 64
    n_slots: int = 0              # state pool size (0: one slot per sequence)
    n_resume: int = 0             # how many sequences resume from a cached slot
    n_tok: int = 1                # decode tokens per sequence
    per_tok_states: bool = False
    spec: bool = False            # decode: verify with commit of a previous step
    note: str = ""


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 0, "prefill", H=2, dk=16, dv=16, dtype="f32", B=1, T=64,
                         chunk=16, note="B=1 T=64 H=2 dk=dv=16 fp32, zero initial state"),
    "prefill_8k": Workload("prefill_8k", 1, "prefill", H=32, dk=128, dv=128, dtype="bf16", B=1,
                           T=8192, snap_interval=1024,
                           note="B=1 T=8192 H=32 dk=dv=128 bf16, snapshots every 1024"),
    "varlen_resume": Workload("varlen_resume", 2, "prefill", H=32, dk=128, dv=128, dtype="bf16",
                              B=16, lens_range=(512, 32768), snap_interval=256, n_slots=1024,
                              n_resume=8,
                              note="16 seqs, L~U[512,32768], H=32, 8 resume from a 1024-slot "
                                   "pool (COW), snapshots every 256"),
    "decode_256x1": Workload("decode_256x1", 3, "decode", H=32, dk=128, dv=128, dtype="bf16",
                             B=256, n_slots=1024, n_tok=1,
                             note="256 seqs x 1 token, H=32, 1024-slot pool, in place"),
    "verify_64x8": Workload("verify_64x8", 3, "decode", H=32, dk=128, dv=128, dtype="bf16",
                            B=64, n_slots=1024, n_tok=8, per_tok_states=True,
                            note="64 seqs x 8 tokens (7 draft + 1), per-token states"),
    "spec_verify_64x8": Workload("spec_verify_64x8", 3, "decode", H=32, dk=128, dv=128,
                                 dtype="bf16", B=64, n_slots=1024, n_tok=8, spec=True,
                                 note="64 seqs x 8 tokens verified, commit of the previous "
                                      "step's accepted tokens (1..8) in the same call"),
    "prefill_1m": Workload("prefill_1m", 4, "prefill", H=16, dk=128, dv=128, dtype="bf16", B=1,
                           T=1 << 20, snap_interval=32768,
                           note="B=1 T=2^20 H=16 dk=dv=128 bf16, snapshots every 32768"),
    # between the cooperative mode's 64 pairs and a full GPU of per-state CTAs
    "prefill_3x32k": Workload("prefill_3x32k", 5, "prefill", H=32, dk=128, dv=128, dtype="bf16",
                              B=3, T=32768, snap_interval=1024,
                              note="B=3 x T=32768 H=32 dk=dv=128 bf16 (96 (sequence, head) "
                                   "pairs), snapshots every 1024"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(index: int, fid: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed((20260000 + index) * 100 + fid)
    return gen


@dataclass
class Batch:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor            # int32 [B+1] (host)
    init_slots: Optional[torch.Tensor] = None   # int32 [B, 2] (host)
    slot_ids: Optional[torch.Tensor] = None     # int32 [N] (host)
    pool: Optional[torch.Tensor] = None         # fp32 [n_slots, H, dk, dv]
    extra: dict = field(default_factory=dict)


def token_tensors(T: int, H: int, dk: int, dv: int, dtype: torch.dtype, index: int,
                  device="cpu", block: int = 1 << 15):
    """q, k, v, g, beta for T packed tokens, drawn per the recipe above."""
    dev = torch.device(device)
    out = {}
    shapes = {"q": (T, H, dk), "k": (T, H, dk), "v": (T, H, dv), "g": (T, H, dk),
              "beta": (T, H)}
    fids = {"q": F_Q, "k": F_K, "v": F_V, "g": F_G, "beta": F_BETA}
    for name in ("q", "k", "v", "g", "beta"):
        dst = torch.empty(shapes[name], dtype=dtype, device=dev)
        gen = _gen(index, fids[name], dev)
        for t0 in range(0, T, block):
            t1 = min(T, t0 + block)
            x = torch.randn((t1 - t0,) + shapes[name][1:], generator=gen, device=dev,
                            dtype=torch.float32)
            if name in ("q", "k"):
                x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
                if name == "q":
                    x = x * (1.0 / math.sqrt(dk))
            elif name == "g":
                x = -torch.exp(x - 3.0)
            elif name == "beta":
                x = torch.sigmoid(x)
            dst[t0:t1] = x.to(dtype)
        out[name] = dst
    return out


def pool_states(n_slots: int, H: int, dk: int, dv: int, index: int, device="cpu",
                block: int = 64) -> torch.Tensor:
    dev = torch.device(device)
    pool = torch.empty((n_slots, H, dk, dv), dtype=torch.float32, device=dev)
    gen = _gen(index, F_POOL, dev)
    for s0 in range(0, n_slots, block):
        s1 = min(n_slots, s0 + block)
        pool[s0:s1] = torch.randn((s1 - s0, H, dk, dv), generator=gen, device=dev) * 0.1
    return pool


def seq_lengths(w: Workload) -> List[int]:
    if w.lens_range is None:
        return [w.T] * w.B
    lo, hi = w.lens_range
    gen = _gen(w.index, F_LENS, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (w.B,), generator=gen)]


def make_batch(w: Workload, device="cpu", lengths: Optional[List[int]] = None,
               H: Optional[int] = None) -> Batch:
    """Draw a whole workload.  ``lengths``/``H`` override the sizes (for scaled
    parity cases that keep the recipe)."""
    H = H or w.H
    dt = torch_dtype(w.dtype)
    if w.kind == "prefill":
        lens = lengths if lengths is not None else seq_lengths(w)
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        T = int(cu[-1])
        tt = token_tensors(T, H, w.dk, w.dv, dt, w.index, device)
        B = len(lens)
        if w.n_slots:
            n_slots = w.n_slots
            pool = pool_states(n_slots, H, w.dk, w.dv, w.index, device)
            gen = _gen(w.index, F_SLOTS, "cpu")
            perm = torch.randperm(n_slots, generator=gen)
            src_pool = perm[:B]                 # candidate cached slots
            dst = perm[B:2 * B]                 # fresh, distinct destinations
            rgen = _gen(w.index, F_RESUME, "cpu")
            resume = torch.zeros(B, dtype=torch.bool)
            resume[torch.randperm(B, generator=rgen)[:min(w.n_resume, B)]] = True
            src = torch.where(resume, src_pool, torch.full_like(src_pool, -1))
        else:
            n_slots = B
            pool = torch.zeros((n_slots, H, w.dk, w.dv), dtype=torch.float32, device=device)
            src = torch.full((B,), -1, dtype=torch.int64)
            dst = torch.arange(B)
        slots = torch.stack([src, dst], 1).to(torch.int32)
        return Batch(cu_seqlens=cu, init_slots=slots, pool=pool, **tt)
    # decode
    N = lengths[0] if lengths is not None else w.B
    tt = token_tensors(N * w.n_tok, H, w.dk, w.dv, dt, w.index, device)
    pool = pool_states(w.n_slots, H, w.dk, w.dv, w.index, device)
    gen = _gen(w.index, F_SLOTS, "cpu")
    slot_ids = torch.randperm(w.n_slots, generator=gen)[:N].to(torch.int32)
    cu = torch.arange(N + 1, dtype=torch.int32) * w.n_tok
    extra = {}
    if w.spec:
        extra["prev"] = token_tensors(N * w.n_tok, H, w.dk, w.dv, dt, w.index + 100, device)
        agen = _gen(w.index, F_ACCEPT, "cpu")
        extra["accepted"] = torch.randint(1, w.n_tok + 1, (N,), generator=agen).to(torch.int32)
    return Batch(cu_seqlens=cu, slot_ids=slot_ids, pool=pool, extra=extra, **tt)


def fused_tensors(T: int, H: int, dk: int, dv: int, dtype: torch.dtype, index: int,
                  n_slots: int, device="cpu", conv_width: int = 4):
    """gate [T, H, dv] (dtype), conv_w [H, 2dk+dv, W] fp32, norm_w [dv] fp32,
    conv_pool [n_slots, H, 2dk+dv, W-1] (dtype), per the recipe above."""
    dev = torch.device(device)
    C = 2 * dk + dv
    gate = torch.empty((T, H, dv), dtype=dtype, device=dev)
    gen = _gen(index, F_GATE, dev)
    block = 1 << 15
    for t0 in range(0, T, block):
        t1 = min(T, t0 + block)
        gate[t0:t1] = torch.randn((t1 - t0, H, dv), generator=gen, device=dev).to(dtype)
    conv_w = torch.randn((H, C, conv_width), generator=_gen(index, F_CONVW, dev),
                         device=dev) * 0.5
    norm_w = 1.0 + 0.1 * torch.randn((dv,), generator=_gen(index, F_NORMW, dev), device=dev)
    conv_pool = torch.randn((n_slots, H, C, conv_width - 1),
                            generator=_gen(index, F_CONVPOOL, dev), device=dev).to(dtype)
    return {"gate": gate, "conv_w": conv_w, "norm_w": norm_w, "conv_pool": conv_pool}
