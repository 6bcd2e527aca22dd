"""GPU parity of the paged-cache decode (fa_decode_paged) against the fp64
oracle. The cache layout is the FlashAttn guide's §1.2 (PagedAttention:
blocks of block_size tokens, a block table per sequence; PA_BBND and
PA_BNBD). The oracle sees the logical, unpaged cache. Tolerances as in
test_gpu_parity.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import compare

pytestmark = pytest.mark.gpu


def _paged_case(B, Hq, Hkv, D, lens, bs, kv_layout, seed, extra_blocks=3):
    """Logical q/k/v (BNSD, cache padded to max_blocks*bs) and the same K/V
    scattered into a shuffled block pool; unused pool rows hold NaN/Inf
    garbage, as do the logical rows past each length."""
    g = torch.Generator().manual_seed(seed)
    max_blocks = max(1, max(math.ceil(L / bs) for L in lens))
    S = max_blocks * bs
    q = torch.randn(B, Hq, 1, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    for b, L in enumerate(lens):
        n = Hkv * (S - L) * D
        k[b, :, L:] = workloads.random_bf16_bits(n, g).view(Hkv, S - L, D)
        v[b, :, L:] = workloads.random_bf16_bits(n, g).view(Hkv, S - L, D)
    used = [math.ceil(L / bs) for L in lens]
    nblk = sum(used) + extra_blocks
    perm = torch.randperm(nblk, generator=g).tolist()
    table = torch.full((B, max_blocks), nblk + 5, dtype=torch.int32)  # unused: out of range
    if kv_layout == "PA_BBND":
        kp = workloads.random_bf16_bits(nblk * bs * Hkv * D, g).view(nblk, bs, Hkv, D)
    else:
        kp = workloads.random_bf16_bits(nblk * Hkv * bs * D, g).view(nblk, Hkv, bs, D)
    vp = workloads.random_bf16_bits(kp.numel(), g).view(kp.shape)
    nxt = 0
    for b in range(B):
        for i in range(used[b]):
            blk = perm[nxt]
            nxt += 1
            table[b, i] = blk
            rows = slice(i * bs, (i + 1) * bs)
            if kv_layout == "PA_BBND":
                kp[blk] = k[b, :, rows].permute(1, 0, 2)
                vp[blk] = v[b, :, rows].permute(1, 0, 2)
            else:
                kp[blk] = k[b, :, rows]
                vp[blk] = v[b, :, rows]
    return q, k, v, kp, vp, table


CASES = [
    # B, Hq, Hkv, D, lens, block_size, kv_layout, splits
    (2, 8, 2, 128, [100, 7], 16, "PA_BBND", 0),
    (3, 32, 8, 128, [1000, 513, 64], 64, "PA_BNBD", 0),
    (2, 4, 4, 64, [333, 1], 128, "PA_BBND", 0),
    (1, 16, 2, 64, [4096], 256, "PA_BBND", 0),
    (4, 8, 1, 128, [0, 200, 17, 1500], 32, "PA_BNBD", 0),
    (2, 8, 2, 128, [3000, 2999], 1024, "PA_BBND", 8),
    (1, 32, 8, 128, [8192], 128, "PA_BNBD", 64),
    # head dim 256: 56-row stages, 8-row boxes
    (3, 16, 4, 256, [777, 16, 2048], 16, "PA_BBND", 0),
    (2, 8, 8, 256, [1500, 90], 48, "PA_BNBD", 3),
    # more units than SMs: shares cut by cost, still on 16-row boundaries
    (40, 32, 8, 128, [(53 * b) % 700 + (b % 3) for b in range(40)], 16, "PA_BBND", 0),
    (24, 16, 16, 64, [(97 * b) % 300 for b in range(24)], 32, "PA_BNBD", 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,bs,kv_layout,splits", CASES)
def test_paged_decode_matches_oracle(cuda_device, B, Hq, Hkv, D, lens, bs, kv_layout, splits):
    q, k, v, kp, vp, table = _paged_case(B, Hq, Hkv, D, lens, bs, kv_layout, seed=3000 + bs + B)
    scale = 1.0 / math.sqrt(D)
    out, lse = F.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, lens,
                                 kv_layout=kv_layout, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = oracle.decode(q, k, v, lens, scale=scale)
    compare(out, lse, ro, rl, "BNSD")


def test_paged_decode_with_key_mask(cuda_device):
    B, Hq, Hkv, D, bs = 2, 8, 2, 128, 64
    lens = [700, 300]
    q, k, v, kp, vp, table = _paged_case(B, Hq, Hkv, D, lens, bs, "PA_BBND", seed=41)
    S = table.shape[1] * bs
    g = torch.Generator().manual_seed(9)
    km = (torch.rand(B, S, generator=g) < 0.3).to(torch.uint8)
    out, lse = F.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, lens,
                                 key_mask=km.cuda(), scale=0.1)
    torch.cuda.synchronize()
    ro, rl = oracle.decode(q, k, v, lens, scale=0.1, key_mask=km)
    compare(out, lse, ro, rl, "BNSD")


def test_paged_equals_contiguous_decode(cuda_device):
    """The same cache paged (any block order) and contiguous gives the same
    result up to the split's rounding; with one piece per unit the two paths
    read the same rows in the same order."""
    B, Hq, Hkv, D, bs = 2, 32, 8, 128, 128
    lens = [4096, 1000]
    q, k, v, kp, vp, table = _paged_case(B, Hq, Hkv, D, lens, bs, "PA_BNBD", seed=8)
    a = F.fa_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, lens,
                          kv_layout="PA_BNBD", scale=0.09)
    b = F.fa_decode(q.cuda(), k.cuda(), v.cuda(), lens, scale=0.09)
    torch.cuda.synchronize()
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2e-2
    assert (a[1] - b[1]).abs().max().item() <= 1e-3


def test_paged_workload_matches_contiguous_run(cuda_device):
    """The bench's paged decode workload: the paged call on the shuffled pool
    against the oracle on the logical cache (full size, every head)."""
    w = workloads.WORKLOADS["paged_decode"]
    x = workloads.make(w)
    lens = x["lengths"]
    bs = w.block_size
    nb = (w.S_kv + bs - 1) // bs
    perm = torch.randperm(w.B * nb, generator=torch.Generator().manual_seed(w.seed))
    table = perm.view(w.B, nb).to(torch.int32)
    kb = workloads.to_bnsd(x["k"], w.layout)
    vb = workloads.to_bnsd(x["v"], w.layout)
    kp = torch.empty(w.B * nb, bs, w.Hkv, w.D, dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    kp[table.view(-1).long()] = kb.reshape(w.B, w.Hkv, nb, bs, w.D).permute(0, 2, 3, 1, 4) \
        .reshape(-1, bs, w.Hkv, w.D)
    vp[table.view(-1).long()] = vb.reshape(w.B, w.Hkv, nb, bs, w.D).permute(0, 2, 3, 1, 4) \
        .reshape(-1, bs, w.Hkv, w.D)
    out, lse = F.fa_decode_paged(x["q"].cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, lens,
                                 scale=w.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], lens, scale=w.scale, layout=w.layout)
    compare(out, lse, ro, rl, w.layout)
