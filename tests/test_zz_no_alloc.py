"""fa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (for instance while a stream is captured into a CUDA graph, or
inside a host framework whose memory pool they may not touch). It runs on a
device array the library owns instead of a caller-provided workspace; this
checks, through the C ABI, that two calls in a row give the same results as
fa_decode with a workspace, within the tolerance of the other GPU tests."""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads
from attention_forward_qk_gb300 import _lib
from attention_forward_qk_gb300 import fa as F

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode(cuda_device):
    B, Hq, Hkv, S, D = 4, 16, 4, 2000, 128
    x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=77, len_lo=1, len_hi=S)
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    lens = x["lengths"]
    scale = 1.0 / math.sqrt(D)
    ref_out, ref_lse = F.fa_decode(q, k, v, lens, scale=scale)
    torch.cuda.synchronize()
    ref_o = ref_out.float().cpu().numpy()
    ref_l = ref_lse.cpu().numpy()

    lib = _lib.load()
    lens_arr = (ctypes.c_int64 * B)(*lens)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the second call finds the first call's scratch contents
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, 1), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.fa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, lens_arr, B, S,
                                   Hq, Hkv, D, scale, _lib.FA_LAYOUT_BNSD, 0, out.data_ptr(),
                                   lse.data_ptr(), stream)
        assert st == _lib.FA_OK, lib.fa_status_string(st)
        torch.cuda.synchronize()
        err = np.abs(out.float().cpu().numpy() - ref_o)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        assert np.abs(lse.cpu().numpy() - ref_l).max() <= 1e-3


def test_noalloc_rejects_oversized_problems(cuda_device):
    lib = _lib.load()
    p = torch.empty(16, dtype=torch.bfloat16, device="cuda").data_ptr()
    big = 1 << 20  # partial buffers far beyond the scratch array
    lens_arr = (ctypes.c_int64 * 64)(*([big] * 64))
    st = lib.fa_decode_noalloc(p, p, p, None, lens_arr, 64, big, 64, 8, 128, 0.1,
                               _lib.FA_LAYOUT_BNSD, 0, p, None, None)
    assert st == _lib.FA_ERR_WORKSPACE_TOO_SMALL
