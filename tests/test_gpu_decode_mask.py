"""Decode with one key mask per query head (aclnnIncreFlashAttention guide
§四, attenMask (B, N, 1, S) and (1, N, 1, S)) through fa_decode_masked,
against the fp64 oracle. Keys masked for every head of a KV group hold NaN
(they must never enter a product); stale cache rows past each length hold
random bits; some heads see no key at all (out 0, lse +inf)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import compare

pytestmark = pytest.mark.gpu


def _per_head_inputs(B, Hq, Hkv, S, D, layout, seed, mask_batches):
    x = workloads.make_decode(B, Hq, Hkv, S, D, layout, seed=seed, len_lo=1, len_hi=S)
    g = torch.Generator().manual_seed(seed + 1)
    km = (torch.rand(mask_batches, Hq, S, generator=g) < 0.3).to(torch.uint8)
    km[0, Hq - 1, :] = 1  # the last head of the first mask batch sees nothing
    # keys masked for every head of KV group 0 hold NaN
    grp = Hq // Hkv
    allm = torch.rand(S, generator=g) < 0.05
    km[:, :grp, allm] = 1
    k, v = x["k"].clone(), x["v"].clone()
    kb = workloads.to_bnsd(k, layout)
    vb = workloads.to_bnsd(v, layout)
    kb[:, 0, allm, :] = float("nan")
    vb[:, 0, allm, :] = float("nan")
    k = workloads.to_bnsd(kb, layout).contiguous()
    v = workloads.to_bnsd(vb, layout).contiguous()
    return x["q"], k, v, x["lengths"], km


CASES = [
    # B, Hq, Hkv, S, D, layout, mask layout, num_splits
    (4, 16, 4, 2000, 128, "BNSD", "BN1S", 0),
    (4, 16, 4, 2000, 128, "BSND", "1N1S", 0),
    (3, 8, 8, 1500, 128, "BNSD", "BN1S", 0),      # one head per KV head
    (2, 32, 4, 1200, 64, "BNSD", "BN1S", 0),      # eight heads per CTA
    (2, 8, 2, 1000, 256, "BSND", "BN1S", 0),
    (2, 16, 4, 3000, 128, "BNSD", "BN1S", 128),   # a forced split count
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,layout,ml,splits", CASES)
def test_per_head_mask_decode_matches_oracle(cuda_device, B, Hq, Hkv, S, D, layout, ml, splits):
    q, k, v, lens, km = _per_head_inputs(B, Hq, Hkv, S, D, layout, seed=B * S + D,
                                         mask_batches=B if ml == "BN1S" else 1)
    km_dev = (km if ml == "BN1S" else km[0]).contiguous().cuda()
    out, lse = F.fa_decode_masked(q.cuda(), k.cuda(), v.cuda(), lens, km_dev, ml,
                                  scale=1 / math.sqrt(D), layout=layout, num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = oracle.decode(q, k, v, lens, scale=1 / math.sqrt(D), layout=layout, key_mask=km)
    compare(out, lse, ro, rl, layout)


def test_shared_layout_is_fa_decode(cuda_device):
    """The (B, 1, 1, S) layout through fa_decode_masked is fa_decode, bit for bit."""
    x = workloads.make_decode(4, 16, 4, 2000, 128, "BNSD", seed=5, len_lo=1, len_hi=2000)
    g = torch.Generator().manual_seed(6)
    km = (torch.rand(4, 2000, generator=g) < 0.3).to(torch.uint8).cuda()
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    o1, l1 = F.fa_decode(q, k, v, x["lengths"], key_mask=km, scale=0.088)
    o2, l2 = F.fa_decode_masked(q, k, v, x["lengths"], km, "B11S", scale=0.088)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
