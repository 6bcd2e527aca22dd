"""GPU parity of the paged-cache prefill (fa_forward_paged) against the fp64
oracle: K and V in blocks of block_size rows scattered through a pool, with a
block table per sequence (FlashAttn guide §1.2: layout_kv PA_BBND / PA_BNBD
beside the q layouts BNSD and BSND). The oracle sees the logical, unpaged K/V.
Tolerances as in test_gpu_parity.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import compare

pytestmark = pytest.mark.gpu


def _bsnd(x):
    return x.permute(0, 2, 1, 3).contiguous()


def _case(B, Hq, Hkv, S_q, S_kv, D, bs, kv_layout, seed, lens=None, table_fill="out",
          extra_blocks=3):
    """Logical q, k, v (BNSD; K/V rows past each length hold random bits, NaN
    and Inf included) and the same K/V scattered into a shuffled pool whose
    other rows are random bits. Table entries past the blocks a sequence's
    keys use hold an id outside the pool (table_fill "out") or ids of other
    blocks ("other")."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, S_q, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S_kv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S_kv, D, generator=g).to(torch.bfloat16)
    L = list(lens) if lens is not None else [S_kv] * B
    for b, Lb in enumerate(L):
        n = Hkv * (S_kv - Lb) * D
        k[b, :, Lb:] = workloads.random_bf16_bits(n, g).view(Hkv, S_kv - Lb, D)
        v[b, :, Lb:] = workloads.random_bf16_bits(n, g).view(Hkv, S_kv - Lb, D)
    max_blocks = max(1, math.ceil(S_kv / bs))
    used = [math.ceil(Lb / bs) for Lb in L]
    nblk = sum(used) + extra_blocks
    perm = torch.randperm(nblk, generator=g).tolist()
    if table_fill == "out":
        table = torch.full((B, max_blocks), nblk + 5, dtype=torch.int32)
    else:
        table = torch.randint(0, nblk, (B, max_blocks), generator=g, dtype=torch.int32)
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
            r0, r1 = i * bs, min((i + 1) * bs, S_kv)
            if kv_layout == "PA_BBND":
                kp[blk, :r1 - r0] = k[b, :, r0:r1].permute(1, 0, 2)
                vp[blk, :r1 - r0] = v[b, :, r0:r1].permute(1, 0, 2)
            else:
                kp[blk, :, :r1 - r0] = k[b, :, r0:r1]
                vp[blk, :, :r1 - r0] = v[b, :, r0:r1]
    return q, k, v, kp, vp, table


CASES = [
    # B, Hq, Hkv, S_q, S_kv, D, block_size, kv_layout, q layout, causal, lens, masked, table_fill
    (2, 8, 2, 384, 384, 128, 128, "PA_BBND", "BNSD", True, None, False, "out"),
    (2, 8, 8, 300, 300, 64, 16, "PA_BNBD", "BSND", False, None, False, "out"),   # ragged last tile
    (1, 16, 4, 500, 500, 256, 48, "PA_BBND", "BNSD", True, None, False, "other"),  # 64-key tiles
    (3, 4, 1, 200, 1000, 128, 1024, "PA_BNBD", "BNSD", False, [1000, 517, 1], False, "out"),
    (2, 8, 2, 640, 640, 128, 64, "PA_BBND", "BSND", True, [640, 333], True, "other"),
    (2, 16, 2, 129, 129, 128, 32, "PA_BNBD", "BNSD", True, None, False, "other"),
    (2, 8, 4, 256, 700, 64, 256, "PA_BBND", "BSND", False, [0, 650], False, "out"),  # an empty sequence
]


def _run(case, scale=None):
    B, Hq, Hkv, S_q, S_kv, D, bs, kvl, layout, causal, lens, masked, fill = case
    q, k, v, kp, vp, table = _case(B, Hq, Hkv, S_q, S_kv, D, bs, kvl, seed=4000 + bs + D + B,
                                   lens=lens, table_fill=fill)
    km = None
    if masked:
        g = torch.Generator().manual_seed(B + S_kv)
        km = (torch.rand(B, S_kv, generator=g) < 0.2).to(torch.uint8)
    scale = D ** -0.5 if scale is None else scale
    qx = _bsnd(q) if layout == "BSND" else q
    out, lse = F.fa_forward_paged(qx.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bs, S_kv,
                                  kv_layout=kvl, mask_mode="causal" if causal else None,
                                  key_mask=km.cuda() if km is not None else None,
                                  actual_seq_lengths=lens, scale=scale, layout=layout)
    torch.cuda.synchronize()
    return (q, k, v, km, lens, layout, causal, scale), out, lse


@pytest.mark.parametrize("case", CASES)
def test_paged_prefill_matches_oracle(cuda_device, case):
    (q, k, v, km, lens, layout, causal, scale), out, lse = _run(case)
    cvt = _bsnd if layout == "BSND" else (lambda t: t)
    ro, rl = oracle.attention(cvt(q), cvt(k), cvt(v), scale=scale, layout=layout, causal=causal,
                              key_mask=km, actual_seq_lengths=lens)
    compare(out, lse, ro, rl, layout)


@pytest.mark.parametrize("case", [CASES[0], CASES[4], CASES[2]])
def test_paged_prefill_equals_contiguous(cuda_device, case):
    """The paged call and fa_forward on the logical cache load the same K/V
    tiles and run the same arithmetic: bitwise equal results."""
    (q, k, v, km, lens, layout, causal, scale), out, lse = _run(case)
    cvt = _bsnd if layout == "BSND" else (lambda t: t)
    ref_out, ref_lse = F.fa_forward(cvt(q).cuda(), cvt(k).cuda(), cvt(v).cuda(),
                                    mask_mode="causal" if causal else None,
                                    key_mask=km.cuda() if km is not None else None,
                                    actual_seq_lengths=lens, scale=scale, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


def test_paged_prefill_workload(cuda_device):
    """The bench's paged prefill workload at full size (the causal prefill
    shape with K/V in 128-row blocks in shuffled order): sampled rows of every
    (batch, head) against the oracle on the logical K/V, and the whole output
    bitwise equal to fa_forward on the contiguous K/V."""
    from test_gpu_parity import _sample_rows
    w = workloads.WORKLOADS["paged_prefill"]
    x = workloads.make(w)
    bs = w.block_size
    nb = (w.S_kv + bs - 1) // bs
    perm = torch.randperm(w.B * nb, generator=torch.Generator().manual_seed(w.seed))
    table = perm.view(w.B, nb).to(torch.int32)
    kb = workloads.to_bnsd(x["k"], w.layout)
    vb = workloads.to_bnsd(x["v"], w.layout)
    pool = lambda t: t.reshape(w.B, w.Hkv, nb, bs, w.D).permute(0, 2, 3, 1, 4) \
        .reshape(-1, bs, w.Hkv, w.D)
    kp = torch.empty(w.B * nb, bs, w.Hkv, w.D, dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    kp[table.view(-1).long()] = pool(kb)
    vp[table.view(-1).long()] = pool(vb)
    q = x["q"].cuda()
    out, lse = F.fa_forward_paged(q, kp.cuda(), vp.cuda(), table.cuda(), bs, w.S_kv,
                                  kv_layout="PA_BBND", mask_mode="causal", scale=w.scale,
                                  layout=w.layout)
    ref_out, ref_lse = F.fa_forward(q, x["k"].cuda(), x["v"].cuda(), mask_mode="causal",
                                    scale=w.scale, layout=w.layout)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    rows = _sample_rows(w.S_q, None, w.seed)
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=w.scale, layout=w.layout,
                              causal=True, rows=rows)
    compare(out, lse, ro, rl, w.layout, rows=rows)
