"""CPU-side checks of the boundary: libkda.so builds for sm_103a, loads, and
exports every function include/kda.h declares; host-only entry points and
host-visible argument errors behave as documented (no GPU is touched)."""

import ctypes
import os
import re
import subprocess

import pytest

import hybrid_linear_attention_delta_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(kda_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    kda.build()
    return kda.lib()


def test_library_exports_every_declared_symbol(lib):
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            names += _declared(h)
    assert "kda_prefill_varlen" in names and "kda_decode" in names
    out = subprocess.run(["nm", "-D", "--defined-only", kda.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in names:
        getattr(lib, n)


def test_snapshot_count_and_workspace_bytes(lib):
    assert kda.kda_snapshot_count([0, 8192], 1024) == 8
    assert kda.kda_snapshot_count([0, 100, 100, 612], 256) == 0 + 0 + 2
    with pytest.raises(kda.KdaError):
        kda.kda_snapshot_count([0, 5, 3], 1)
    assert kda.kda_snapshot_count([0, 64], 0) == 0
    n1 = kda.kda_workspace_bytes(1, 32, 1)
    n2 = kda.kda_workspace_bytes(16, 32, 1024)
    assert n1 % 256 == 0 and n2 % 256 == 0
    # few (sequence, head) pairs: room for the cooperative prefill's package
    # ring (6 packages of 73 KiB per pair)
    assert n1 >= 32 * 6 * 74752
    # claims: one word per (slot, head, column block) of the pool; 512 pairs
    # use the per-state prefill, so no ring
    assert 1024 * 32 * 4 * 4 <= n2 < 1024 * 32 * 4 * 4 + 16 * 32 * 64 + 4096


def test_status_strings(lib):
    for code, name in enumerate(["KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED",
                                 "KDA_ERR_CUDA", "KDA_ERR_DEVICE_CHECK", "KDA_ERR_TIMEOUT"]):
        assert kda.status_string(code) == name


def _args(**kw):
    base = dict(B=1, T_total=64, H=2, dk=16, dv=16, n_slots=1, dtype=kda.KDA_F32)
    base.update(kw)
    a = kda.KdaArgs(**base)
    return a


def test_host_visible_errors_return_without_launch(lib):
    V = ctypes.c_void_p
    fake = V(4096)  # never dereferenced: every case below fails a host check first
    # no workspace
    a = _args()
    st = lib.kda_prefill_varlen(fake, fake, fake, fake, fake, fake, fake, fake, fake, 0, None,
                                ctypes.byref(a))
    assert st == kda.KDA_ERR_INVALID_ARG
    # unsupported head dim
    a = _args(dk=48, workspace=V(1 << 20), workspace_bytes=1 << 20)
    st = lib.kda_prefill_varlen(fake, fake, fake, fake, fake, fake, fake, fake, fake, 0, None,
                                ctypes.byref(a))
    assert st == kda.KDA_ERR_UNSUPPORTED
    # workspace too small
    a = _args(workspace=V(1 << 20), workspace_bytes=16)
    st = lib.kda_prefill_varlen(fake, fake, fake, fake, fake, fake, fake, fake, fake, 0, None,
                                ctypes.byref(a))
    assert st == kda.KDA_ERR_INVALID_ARG
    # snap interval with a nonzero capacity but no snapshot buffer
    a = _args(workspace=V(1 << 20), workspace_bytes=1 << 20, snaps_capacity=5)
    st = lib.kda_prefill_varlen(fake, fake, fake, fake, fake, fake, fake, fake, fake, 64, None,
                                ctypes.byref(a))
    assert st == kda.KDA_ERR_INVALID_ARG
    # misaligned token pointer
    st = lib.kda_prefill_varlen(V(4100), fake, fake, fake, fake, fake, fake, fake, fake, 0,
                                None, ctypes.byref(a))
    assert st == kda.KDA_ERR_INVALID_ARG
    # decode: n_tok inconsistent with T_total (the workspace is large enough,
    # so only that check can refuse the call)
    a = _args(B=4, T_total=7, workspace=V(1 << 26), workspace_bytes=1 << 26)
    assert lib.kda_workspace_bytes(ctypes.byref(a)) <= 1 << 26
    st = lib.kda_decode(fake, fake, fake, fake, fake, fake, fake, fake, 2, None, ctypes.byref(a))
    assert st == kda.KDA_ERR_INVALID_ARG
    # speculative decode: negative counts, a previous step without its
    # accepted lengths or tokens, a misaligned previous-step pointer
    a = _args(B=4, T_total=8, workspace=V(1 << 26), workspace_bytes=1 << 26)
    assert lib.kda_workspace_bytes(ctypes.byref(a)) <= 1 << 26
    N = None
    assert lib.kda_decode_spec(fake, fake, fake, fake, fake, fake, fake, fake, -1, N, N, N, N, N,
                               0, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_spec(fake, fake, fake, fake, fake, fake, fake, fake, 2, N, N, N, N, N,
                               -3, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_spec(fake, fake, fake, fake, fake, fake, fake, fake, 2, fake, fake, fake,
                               fake, N, 4, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_spec(fake, fake, fake, fake, fake, fake, fake, fake, 2, fake, N, fake,
                               fake, fake, 4, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_spec(fake, fake, fake, fake, fake, fake, fake, fake, 2, V(4100), fake,
                               fake, fake, fake, 4, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    # n_tok inconsistent with T_total
    assert lib.kda_decode_spec(fake, fake, fake, fake, fake, fake, fake, fake, 3, N, N, N, N, N, 0,
                               ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    # retention map: missing with a nonzero capacity, or given without an interval
    a = _args(workspace=V(1 << 26), workspace_bytes=1 << 26, snaps_capacity=4)
    assert lib.kda_prefill_varlen_retain(fake, fake, fake, fake, fake, fake, fake, fake, fake, 64,
                                         None, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_varlen_retain(fake, fake, fake, fake, fake, fake, fake, fake, fake, 0,
                                         fake, ctypes.byref(a)) == kda.KDA_ERR_INVALID_ARG
    # forcing the chunked algorithm on an fp32 batch is unsupported (with a
    # workspace large enough for the cooperative mode's package ring)
    a = _args(algo=kda.KDA_ALGO_CHUNKED, workspace=V(1 << 26), workspace_bytes=1 << 26)
    st = lib.kda_prefill_varlen(fake, fake, fake, fake, fake, fake, fake, fake, fake, 0, None,
                                ctypes.byref(a))
    assert st == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_last_launch_count() == 0


def test_fused_calls_host_visible_errors_and_scratch_size(lib):
    """The convolution + gated-RMSNorm entry points refuse bad arguments on the
    host before any launch; the prefill's scratch holds q, k, v and o."""
    V = ctypes.c_void_p
    fake = V(4096)
    a = _args(workspace=V(1 << 26), workspace_bytes=1 << 26)
    # T = 64, H = 2, dk = dv = 16, fp32: four 8 KiB regions
    assert lib.kda_fused_scratch_bytes(ctypes.byref(a)) == 4 * 64 * 2 * 16 * 4
    f = kda.KdaFusedArgs(gate=fake, conv_w=fake, norm_w=fake, conv_pool=fake, conv_width=4,
                         conv_act=0, norm_eps=1e-6)
    pre = lambda f_, scratch, n: lib.kda_prefill_varlen_fused(
        fake, fake, fake, fake, fake, fake, fake, fake, fake, 0, None,
        None if f_ is None else ctypes.byref(f_), scratch, n, ctypes.byref(a))
    assert pre(None, fake, 1 << 20) == kda.KDA_ERR_INVALID_ARG
    assert pre(f, fake, 16) == kda.KDA_ERR_INVALID_ARG          # scratch too small
    assert pre(f, None, 1 << 20) == kda.KDA_ERR_INVALID_ARG     # no scratch
    f3 = kda.KdaFusedArgs(gate=fake, conv_w=fake, norm_w=fake, conv_pool=fake, conv_width=3)
    assert pre(f3, fake, 1 << 20) == kda.KDA_ERR_UNSUPPORTED    # only 4 taps
    fa = kda.KdaFusedArgs(gate=fake, conv_w=fake, norm_w=fake, conv_pool=fake, conv_width=4,
                          conv_act=7)
    assert pre(fa, fake, 1 << 20) == kda.KDA_ERR_INVALID_ARG    # unknown activation
    fn = kda.KdaFusedArgs(gate=None, conv_w=fake, norm_w=fake, conv_pool=fake, conv_width=4)
    assert pre(fn, fake, 1 << 20) == kda.KDA_ERR_INVALID_ARG    # no gate
    # the fused decode runs dk = dv = 128 only
    ad = _args(B=4, T_total=4, workspace=V(1 << 26), workspace_bytes=1 << 26)
    assert lib.kda_decode_fused(fake, fake, fake, fake, fake, fake, fake, fake, 1, None,
                                ctypes.byref(f), ctypes.byref(ad)) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_last_launch_count() == 0
