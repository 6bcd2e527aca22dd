"""fa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (for instance while a stream is captured into a CUDA graph, or
inside a host framework whose memory pool they may not touch). It runs on a
device array the library owns instead of a caller-provided workspace.

Checked through the C ABI: two calls in a row (the second finds the first
call's scratch contents) against the fp64 oracle and against fa_decode with a
workspace, within the tolerance of the other GPU tests, for the default split
plan, a forced split count and a key mask; the full long-context decode
shape; the status word; and a problem whose plan cannot fit, which is
rejected before anything is launched.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import _lib
from attention_forward_qk_gb300 import fa as F

pytestmark = pytest.mark.gpu

OUT_MAX = 2e-2
OUT_MEAN = 2e-3
LSE_MAX = 1e-3


def _check(out, lse, ro, rl):
    o = out.float().cpu().double().numpy().reshape(ro.shape)
    lg = lse.cpu().double().numpy().reshape(rl.shape)
    invalid = ~np.isfinite(rl)
    assert np.array_equal(invalid, ~np.isfinite(lg))
    assert np.all(o.reshape(invalid.shape + (-1,))[invalid] == 0.0)
    err = np.abs(o - ro)
    assert err.max() <= OUT_MAX and err.mean() <= OUT_MEAN, (err.max(), err.mean())
    ok = ~invalid
    if ok.any():
        assert np.abs(lg[ok] - rl[ok]).max() <= LSE_MAX


def _noalloc(lib, q, k, v, km, lens, B, S, Hq, Hkv, D, scale, splits, layout):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, 1), float("nan"), dtype=torch.float32, device="cuda")
    lens_arr = (ctypes.c_int64 * B)(*lens)
    st = lib.fa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               km.data_ptr() if km is not None else None, lens_arr, B, S, Hq,
                               Hkv, D, scale, layout, splits, out.data_ptr(), lse.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == _lib.FA_OK, lib.fa_status_string(st)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("splits,masked", [(0, False), (128, False), (0, True)])
def test_noalloc_decode_matches_oracle_twice(cuda_device, splits, masked):
    B, Hq, Hkv, S, D = 4, 16, 4, 2000, 128
    x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=77, len_lo=1, len_hi=S)
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    lens = x["lengths"]
    km_host = None
    if masked:
        g = torch.Generator().manual_seed(78)
        km_host = (torch.rand(B, S, generator=g) < 0.3).to(torch.uint8)
    km = km_host.cuda() if km_host is not None else None
    scale = 1.0 / math.sqrt(D)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], lens, scale=scale, key_mask=km_host)
    ref_out, ref_lse = F.fa_decode(q, k, v, lens, key_mask=km, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    lib = _lib.load()
    for _ in range(2):  # the second call finds the first call's scratch contents
        out, lse = _noalloc(lib, q, k, v, km, lens, B, S, Hq, Hkv, D, scale, splits,
                            _lib.FA_LAYOUT_BNSD)
        _check(out, lse, ro, rl)
        # and the same as fa_decode with a caller workspace
        err = (out.float() - ref_out.float()).abs()
        assert err.max().item() <= OUT_MAX and err.mean().item() <= OUT_MEAN
        assert (lse - ref_lse).abs().max().item() <= LSE_MAX
    assert lib.fa_decode_noalloc_status(None) == _lib.FA_OK


def test_noalloc_long_context_decode(cuda_device):
    """B=1, 32 heads, D=128, 131072 valid keys (BSND): its plan needs a small
    part of the array (the size query's worst-case bound would not fit)."""
    w = workloads.WORKLOADS["long_decode"]
    x = workloads.make(w)
    assert F.fa_decode_workspace_size(w.B, w.S_kv, w.Hq, w.Hkv, w.D, 0) > (8 << 20)
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    lib = _lib.load()
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=w.scale,
                           layout=w.layout)
    for _ in range(2):
        out, lse = _noalloc(lib, q, k, v, None, x["lengths"], w.B, w.S_kv, w.Hq, w.Hkv, w.D,
                            w.scale, 0, _lib.FA_LAYOUT_BSND)
        _check(out, lse, ro, rl)  # one query row: BSND and BNSD are the same memory


def test_noalloc_rejects_a_plan_that_does_not_fit(cuda_device):
    """A forced split of 4096 pieces over 64 heads of D=256 needs about 270 MB
    of partial results: rejected on the host, before any launch (the plan is
    checked here first, so nothing could be launched on the dummy buffers)."""
    lib = _lib.load()
    B, H, D, S, splits = 1, 64, 256, 4096 * 64, 4096
    lens = [S]
    lens_arr = (ctypes.c_int64 * B)(*lens)
    rc, n, mx = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    assert lib.fa_decode_plan(B, S, H, H, D, lens_arr, 152, splits, ctypes.byref(rc),
                              ctypes.byref(n), ctypes.byref(mx)) == _lib.FA_OK
    assert 4 * B * H * mx.value * (D + 1) > 2 * (8 << 20)
    p = torch.empty(64, dtype=torch.bfloat16, device="cuda").data_ptr()
    n0 = lib.fa_kernel_launch_count()
    st = lib.fa_decode_noalloc(p, p, p, None, lens_arr, B, S, H, H, D, 0.1,
                               _lib.FA_LAYOUT_BNSD, splits, p, None, None)
    assert st == _lib.FA_ERR_WORKSPACE_TOO_SMALL
    assert lib.fa_kernel_launch_count() == n0


def test_noalloc_status_reports_a_device_timeout(cuda_device):
    """A device-side timeout of a noalloc call lands in the library-owned
    array's status word, which fa_decode_noalloc_status reads and clears; the
    next call with the default limit matches the oracle again."""
    B, Hq, Hkv, S, D = 2, 8, 2, 3000, 128
    x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=79, len_lo=800, len_hi=S)
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    lib = _lib.load()
    scale = 1.0 / math.sqrt(D)
    assert lib.fa_set_wait_timeout_ns(100) == _lib.FA_OK
    try:
        _noalloc(lib, q, k, v, None, x["lengths"], B, S, Hq, Hkv, D, scale, 0,
                 _lib.FA_LAYOUT_BNSD)
        assert lib.fa_decode_noalloc_status(None) == _lib.FA_ERR_DEVICE_TIMEOUT
        assert lib.fa_decode_noalloc_status(None) == _lib.FA_OK  # read clears it
    finally:
        lib.fa_set_wait_timeout_ns(0)
    out, lse = _noalloc(lib, q, k, v, None, x["lengths"], B, S, Hq, Hkv, D, scale, 0,
                        _lib.FA_LAYOUT_BNSD)
    assert lib.fa_decode_noalloc_status(None) == _lib.FA_OK
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=scale)
    _check(out, lse, ro, rl)
