"""Failure detection in the real kernels: with the bounded-wait limit set to
0.1 microsecond (fa_set_wait_timeout_ns), the first waits of a real
prefill or decode call run out. The kernel then records FA_ERR_DEVICE_TIMEOUT
in the workspace status word, lets its own copies and tensor-core operations
in flight land, frees TMEM and returns. The next call, with the default limit,
must succeed and match the oracle: the abort left the context usable. Nothing
here faults, traps or hangs a GPU: every wait is bounded."""
import math

import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import _lib
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import compare

pytestmark = pytest.mark.gpu

SHORT_NS = 100


def _prefill(x, ws, D):
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    return F.fa_forward(q, k, v, mask_mode="causal", scale=1 / math.sqrt(D), layout="BSND",
                        workspace=ws)


@pytest.mark.parametrize("D", [128, 256])
def test_prefill_timeout_aborts_and_the_next_call_is_exact(cuda_device, D):
    B, H, S = 1, 4, 1024
    x = workloads.make_prefill(B, H, H, S, S, D, "BSND", seed=31 + D)
    ws = torch.empty(F.fa_forward_workspace_size(B, S, S, H, H, D), dtype=torch.uint8,
                     device="cuda")
    F.fa_set_wait_timeout_ns(SHORT_NS)
    try:
        _prefill(x, ws, D)
        assert F.fa_workspace_status(ws) == _lib.FA_ERR_DEVICE_TIMEOUT
    finally:
        F.fa_set_wait_timeout_ns(0)
    out, lse = _prefill(x, ws, D)
    torch.cuda.synchronize()
    assert F.fa_workspace_status(ws) == _lib.FA_OK
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=1 / math.sqrt(D), layout="BSND",
                              causal=True)
    compare(out, lse, ro, rl, "BSND")


def test_paged_prefill_timeout_aborts_and_the_next_call_is_exact(cuda_device):
    """The paged instantiation: a KV tile lands as several boxes on one
    barrier, all issued after one byte count, so the drain after an abort
    waits for whole tiles as with a contiguous cache."""
    from test_gpu_paged_prefill import _case
    B, H, S, D, bs = 1, 4, 1024, 128, 32
    q, k, v, kp, vp, table = _case(B, H, H, S, S, D, bs, "PA_BBND", seed=33)
    args = (q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, S)
    kw = dict(kv_layout="PA_BBND", mask_mode="causal", scale=1 / math.sqrt(D))
    ws = torch.empty(F.fa_forward_workspace_size(B, S, S, H, H, D), dtype=torch.uint8,
                     device="cuda")
    F.fa_set_wait_timeout_ns(SHORT_NS)
    try:
        F.fa_forward_paged(*args, workspace=ws, **kw)
        assert F.fa_workspace_status(ws) == _lib.FA_ERR_DEVICE_TIMEOUT
    finally:
        F.fa_set_wait_timeout_ns(0)
    out, lse = F.fa_forward_paged(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert F.fa_workspace_status(ws) == _lib.FA_OK
    ro, rl = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=True)
    compare(out, lse, ro, rl, "BNSD")


def test_decode_timeout_aborts_and_the_next_call_is_exact(cuda_device):
    B, Hq, Hkv, S, D = 4, 16, 4, 3000, 128
    x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=41, len_lo=500, len_hi=S)
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    ws = torch.empty(F.fa_decode_workspace_size(B, S, Hq, Hkv, D, 0), dtype=torch.uint8,
                     device="cuda")
    F.fa_set_wait_timeout_ns(SHORT_NS)
    try:
        F.fa_decode(q, k, v, x["lengths"], scale=1 / math.sqrt(D), workspace=ws)
        assert F.fa_workspace_status(ws) == _lib.FA_ERR_DEVICE_TIMEOUT
    finally:
        F.fa_set_wait_timeout_ns(0)
    out, lse = F.fa_decode(q, k, v, x["lengths"], scale=1 / math.sqrt(D), workspace=ws)
    torch.cuda.synchronize()
    assert F.fa_workspace_status(ws) == _lib.FA_OK
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=1 / math.sqrt(D))
    compare(out, lse, ro, rl, "BNSD")


def test_wait_limit_argument_checks(cuda_device):
    lib = _lib.load()
    assert lib.fa_set_wait_timeout_ns(20_000_000_000) == _lib.FA_ERR_PARAM_INVALID
    assert lib.fa_set_wait_timeout_ns(0) == _lib.FA_OK
