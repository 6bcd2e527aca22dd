"""The FA_DEBUG build (libfa_gb300_debug.so): the same kernels with
device-side index checks, which record FA_ERR_DEVICE_CHECK in the workspace
status word and skip the access instead of trapping. On valid inputs no check
may fire and the results must match the oracle as the release build's do:
prefill (padded causal with a key mask, D=256, packed sequences with seqused
and a key mask, a paged cache) and decode (split sequences, forced splits,
paged)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import _lib
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture
def debug_build(cuda_device):
    """Route the binding through the debug library for one test."""
    saved = _lib.load()
    _lib._lib = _lib.load_debug()
    try:
        yield
    finally:
        _lib._lib = saved


def test_debug_prefill_checks_pass_and_match(debug_build):
    for (B, Hq, Hkv, S, D, pad) in [(2, 8, 2, 640, 128, 300), (1, 4, 2, 520, 256, 0)]:
        x = workloads.make_prefill(B, Hq, Hkv, S, S, D, "BNSD", seed=61 + D, max_pad=pad or None)
        ws = torch.empty(F.fa_forward_workspace_size(B, S, S, Hq, Hkv, D), dtype=torch.uint8,
                         device="cuda")
        km = x["key_mask"].cuda() if x["key_mask"] is not None else None
        out, lse = F.fa_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), mask_mode="causal",
                                key_mask=km, scale=1 / math.sqrt(D), workspace=ws)
        assert F.fa_workspace_status(ws) == _lib.FA_OK
        ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=1 / math.sqrt(D), causal=True,
                                  key_mask=x["key_mask"])
        compare(out, lse, ro, rl, "BNSD")


def test_debug_paged_prefill_checks_pass_and_match(debug_build):
    from test_gpu_paged_prefill import _case
    B, Hq, Hkv, S, D, bs = 2, 8, 2, 300, 128, 48
    q, k, v, kp, vp, table = _case(B, Hq, Hkv, S, S, D, bs, "PA_BNBD", seed=63, lens=[300, 211],
                                   table_fill="other")
    ws = torch.empty(F.fa_forward_workspace_size(B, S, S, Hq, Hkv, D), dtype=torch.uint8,
                     device="cuda")
    out, lse = F.fa_forward_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, S,
                                  kv_layout="PA_BNBD", mask_mode="causal",
                                  actual_seq_lengths=[300, 211], scale=1 / math.sqrt(D),
                                  workspace=ws)
    assert F.fa_workspace_status(ws) == _lib.FA_OK
    ro, rl = oracle.attention(q, k, v, scale=1 / math.sqrt(D), causal=True,
                              actual_seq_lengths=[300, 211])
    compare(out, lse, ro, rl, "BNSD")


def test_debug_packed_prefill_checks_pass_and_match(debug_build):
    lq = [300, 129, 700]
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    g = torch.Generator().manual_seed(62)
    T = int(cq[-1])
    q = torch.randn(T, 4, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(T, 2, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(T, 2, 128, generator=g).to(torch.bfloat16)
    km = (torch.rand(T, generator=g) < 0.2).to(torch.uint8)
    uq, ukv = [250, 129, 700], [300, 100, 650]
    ws = torch.empty(F.fa_forward_varlen_workspace_size(3, 700, 700, 4, 2, 128), dtype=torch.uint8,
                     device="cuda")
    out, lse = F.fa_forward_varlen_ex(q.cuda(), k.cuda(), v.cuda(), cq.tolist(), cq.tolist(),
                                      seqused_q=uq, seqused_kv=ukv, key_mask=km.cuda(),
                                      win_left=-1, win_right=0, scale=0.088, workspace=ws)
    assert F.fa_workspace_status(ws) == _lib.FA_OK
    ro, rl = oracle.attention_varlen(q, k, v, cq, cq, scale=0.088, causal=True, seqused_q=uq,
                                     seqused_kv=ukv, key_mask=km)
    o = out.cpu().double().numpy()
    lg = lse.cpu().double().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.abs(o - ro).max() <= 2e-2 and np.abs(lg[fin] - rl[fin]).max() <= 1e-3


@pytest.mark.parametrize("splits", [0, 64])
def test_debug_decode_checks_pass_and_match(debug_build, splits):
    B, Hq, Hkv, S, D = 4, 16, 4, 3000, 128
    x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=63, len_lo=1, len_hi=S)
    ws = torch.empty(F.fa_decode_workspace_size(B, S, Hq, Hkv, D, splits), dtype=torch.uint8,
                     device="cuda")
    out, lse = F.fa_decode(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["lengths"],
                           scale=1 / math.sqrt(D), num_splits=splits, workspace=ws)
    assert F.fa_workspace_status(ws) == _lib.FA_OK
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=1 / math.sqrt(D))
    compare(out, lse, ro, rl, "BNSD")
