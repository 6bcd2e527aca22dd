"""GPU parity of packed variable-length prefill (fa_forward_varlen, TND)
against the fp64 oracle (FlashAttn guide §1.3/§1.4: each sequence is an
independent attention over its own rows). Tolerances as in
test_gpu_parity.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import OUT_MAX, OUT_MEAN, LSE_MAX

pytestmark = pytest.mark.gpu


def _packed(lq, lkv, Hq, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    ckv = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int64)
    q = torch.randn(int(cq[-1]), Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(int(ckv[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(int(ckv[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    return q, k, v, cq, ckv


def _compare(out, lse, ro, rl):
    o = out.detach().cpu().double().numpy()
    lg = lse.detach().cpu().double().numpy()
    invalid = ~np.isfinite(rl)
    assert np.array_equal(invalid, ~np.isfinite(lg))
    assert np.all(lg[invalid] == np.inf) and np.all(o[invalid] == 0)
    err = np.abs(o - ro)
    ok = ~invalid
    assert err.max() <= OUT_MAX, f"max |out err| {err.max():.3e}"
    if ok.any():
        assert err[ok].mean() <= OUT_MEAN
        assert np.abs(lg[ok] - rl[ok]).max() <= LSE_MAX


CASES = [
    # lq, lkv, Hq, Hkv, D, causal
    ([100, 300, 1, 257], [100, 300, 1, 257], 4, 2, 128, True),
    ([128, 0, 640], [128, 0, 640], 8, 8, 64, True),
    ([50, 700, 129], [200, 30, 1000], 4, 1, 128, False),
    ([300, 5], [0, 17], 2, 2, 128, False),
    ([1000], [1000], 8, 2, 128, True),
    ([255, 256, 257, 511, 512, 513], [255, 256, 257, 511, 512, 513], 4, 4, 64, True),
    ([100, 300, 1, 257], [100, 300, 1, 257], 4, 2, 256, True),
    ([50, 700, 129], [200, 30, 1000], 2, 1, 256, False),
]


@pytest.mark.parametrize("lq,lkv,Hq,Hkv,D,causal", CASES)
def test_varlen_matches_oracle(cuda_device, lq, lkv, Hq, Hkv, D, causal):
    q, k, v, cq, ckv = _packed(lq, lkv, Hq, Hkv, D, seed=sum(lq) + D)
    scale = 1.0 / math.sqrt(D)
    out, lse = F.fa_forward_varlen(q.cuda(), k.cuda(), v.cuda(), cq.tolist(), ckv.tolist(),
                                   mask_mode="causal" if causal else None, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_varlen(q, k, v, cq, ckv, scale=scale, causal=causal)
    _compare(out, lse, ro, rl)


WINDOW_CASES = [
    # lens, Hq, Hkv, D, (win_left, win_right)
    ([700, 1, 300, 129], 4, 2, 128, (255, 0)),     # a causal band, shorter than a sequence
    ([1000, 64, 513], 8, 2, 128, (100, 37)),       # both sides, not tile-aligned
    ([600, 0, 90], 4, 4, 64, (-1, 200)),           # unbounded left, bounded right
    ([777, 200], 4, 2, 256, (130, 0)),             # head dim 256 (64-key tiles)
    ([300, 300], 2, 2, 128, (5000, 5000)),         # wider than every sequence: no mask
]


@pytest.mark.parametrize("lens,Hq,Hkv,D,window", WINDOW_CASES)
def test_varlen_window_matches_oracle(cuda_device, lens, Hq, Hkv, D, window):
    q, k, v, cq, ckv = _packed(lens, lens, Hq, Hkv, D, seed=sum(lens) + D + 7)
    scale = 1.0 / math.sqrt(D)
    out, lse = F.fa_forward_varlen_window(q.cuda(), k.cuda(), v.cuda(), cq.tolist(), ckv.tolist(),
                                          window[0], window[1], scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_varlen(q, k, v, cq, ckv, scale=scale, window=window)
    _compare(out, lse, ro, rl)


def test_varlen_window_rejects_unequal_lengths(cuda_device):
    q, k, v, cq, ckv = _packed([100, 50], [100, 60], 2, 2, 128, seed=3)
    with pytest.raises(F.FaError) as e:
        F.fa_forward_varlen_window(q.cuda(), k.cuda(), v.cuda(), cq.tolist(), ckv.tolist(), 10, 0)
    assert e.value.status == 2  # FA_ERR_PARAM_INVALID


def test_varlen_equal_lengths_match_padded_call_bitwise(cuda_device):
    """Equal lengths: the packed call and the BSND batch call compute the same
    tiles in the same order."""
    B, S, Hq, Hkv, D = 3, 600, 8, 2, 128
    g = torch.Generator().manual_seed(4)
    q = torch.randn(B, S, Hq, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16).cuda()
    cu = [i * S for i in range(B + 1)]
    a = F.fa_forward_varlen(q.view(B * S, Hq, D), k.view(B * S, Hkv, D), v.view(B * S, Hkv, D),
                            cu, cu, mask_mode="causal", scale=0.1)
    b = F.fa_forward(q, k, v, mask_mode="causal", scale=0.1, layout="BSND")
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0].view(B * S, Hq, D))
    assert torch.equal(a[1], b[1].permute(0, 2, 1).reshape(B * S, Hq))


def test_varlen_workload_sampled_rows(cuda_device):
    """The bench's packed workload at full size (16 sequences of 512..8192
    tokens): every sequence checked on sampled rows against the oracle."""
    import workloads
    w = workloads.WORKLOADS["varlen_prefill"]
    x = workloads.make(w)
    cu = x["cu_seqlens"]
    out, lse = F.fa_forward_varlen(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), cu, cu,
                                   mask_mode="causal", scale=w.scale)
    torch.cuda.synchronize()
    o = out.cpu()
    l = lse.cpu()
    g = np.random.default_rng(2)
    for b in range(w.B):
        L = cu[b + 1] - cu[b]
        rows = sorted(set([0, L - 1] + g.choice(L, 6, replace=False).tolist()))
        sl = slice(cu[b], cu[b + 1])
        ro, rl = oracle.attention(x["q"][sl][None], x["k"][sl][None], x["v"][sl][None],
                                  scale=w.scale, layout="BSND", causal=True, rows=rows)
        got_o = o[sl][rows].double().numpy()
        got_l = l[sl][rows].double().numpy()
        err = np.abs(got_o - ro[0])
        assert err.max() <= OUT_MAX and err.mean() <= OUT_MEAN
        assert np.abs(got_l - rl[0].T).max() <= LSE_MAX


def _garbage_past_used(q, k, v, cq, ckv, uq, ukv, seed):
    """Random bf16 bit patterns (NaN and Inf included) in the truncated query
    rows and in the keys / values past each used kv length."""
    import workloads
    g = torch.Generator().manual_seed(seed)
    q, k, v = q.clone(), k.clone(), v.clone()
    for b in range(len(uq)):
        for t, c, u in ((q, cq, uq), (k, ckv, ukv), (v, ckv, ukv)):
            lo, hi = int(c[b]) + min(int(u[b]), int(c[b + 1] - c[b])), int(c[b + 1])
            if hi > lo:
                t[lo:hi] = workloads.random_bf16_bits(t[lo:hi].numel(), g).view(t[lo:hi].shape)
    return q, k, v


EX_CASES = [
    # lq, lkv, seqused_q, seqused_kv, masked, window, Hq, Hkv, D
    ([300, 500, 129], [300, 500, 129], [200, 500, 0], [300, 131, 129], False, (-1, 0), 4, 2, 128),
    ([640, 257], [640, 257], [640, 257], [500, 100], True, (-1, 0), 8, 2, 128),
    ([100, 700, 33], [250, 40, 900], [90, 800, 33], [250, 39, 777], True, (-1, -1), 4, 1, 128),
    ([513, 1000], [513, 1000], [400, 999], [513, 1000], True, (100, 17), 4, 4, 64),
    ([300, 520], [300, 520], [290, 520], [255, 400], True, (-1, 0), 2, 2, 256),
    ([0, 128, 1], [0, 128, 1], [5, 128, 1], [0, 0, 1], False, (-1, 0), 2, 1, 128),
]


@pytest.mark.parametrize("lq,lkv,uq,ukv,masked,window,Hq,Hkv,D", EX_CASES)
def test_varlen_seqused_and_key_mask_match_oracle(cuda_device, lq, lkv, uq, ukv, masked, window,
                                                   Hq, Hkv, D):
    """seqused_q / seqused_kv (the shorter of them and the span holds),
    truncated query rows (out 0, lse +inf), garbage past the used lengths and
    a per-packed-key mask, with causal, a window or no mask (FlashAttn guide
    §1.3-§1.5, §1.7)."""
    q, k, v, cq, ckv = _packed(lq, lkv, Hq, Hkv, D, seed=sum(lq) + 3 * D)
    q, k, v = _garbage_past_used(q, k, v, cq, ckv, uq, ukv, seed=sum(lkv))
    km = None
    if masked:
        g = torch.Generator().manual_seed(sum(uq) + 1)
        km = (torch.rand(int(ckv[-1]), generator=g) < 0.2).to(torch.uint8)
    scale = 1.0 / math.sqrt(D)
    out = torch.full_like(q.cuda(), float("nan"))
    lse = torch.full((int(cq[-1]), Hq), float("nan"), dtype=torch.float32, device="cuda")
    F.fa_forward_varlen_ex(q.cuda(), k.cuda(), v.cuda(), cq.tolist(), ckv.tolist(), seqused_q=uq,
                           seqused_kv=ukv, key_mask=km.cuda() if km is not None else None,
                           win_left=window[0], win_right=window[1], scale=scale, out=out, lse=lse)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_varlen(q, k, v, cq, ckv, scale=scale, window=window, seqused_q=uq,
                                     seqused_kv=ukv, key_mask=km)
    _compare(out, lse, ro, rl)


def test_varlen_ex_without_options_equals_varlen(cuda_device):
    """No seqused and no mask: bit-identical to fa_forward_varlen (same kernel,
    same schedule)."""
    q, k, v, cq, ckv = _packed([300, 257, 700], [300, 257, 700], 4, 2, 128, seed=5)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = F.fa_forward_varlen(q, k, v, cq.tolist(), ckv.tolist(), mask_mode="causal",
                                 scale=0.088)
    o2, l2 = F.fa_forward_varlen_ex(q, k, v, cq.tolist(), ckv.tolist(), win_left=-1, win_right=0,
                                    scale=0.088)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
