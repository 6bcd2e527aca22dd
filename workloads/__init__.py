"""Seeded synthetic inputs for the fused attention forward.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic. Both the fp64 oracle (``oracle/``) and the CUDA
path (``attention_forward_qk_gb300``) are fed from here, so that the two
sides always see bit-identical bf16 inputs.

Recipe (one ``torch.Generator('cpu')`` per workload, seeded):
  1. Q, K, V drawn with ``randn`` in fp32, in that order, each cast to bf16
     (round to nearest even) -- the pages' cases use iid N(0,1) bf16 data.
  2. Then, from the same generator: per-batch valid KV lengths (decode) or
     the per-batch count of padded keys (prefill with an explicit mask).
  3. Decode caches: every position at or past a batch's valid length is
     overwritten with random bf16 *bit patterns* (NaN and Inf included),
     standing in for a padded KV cache holding stale data.

Shapes follow the pages' layouts: BNSD = [B, N, S, D] and BSND = [B, S, N, D]
(BSH is BSND memory).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "make_prefill",
    "make_decode",
    "make",
    "random_bf16_bits",
    "to_bnsd",
]


@dataclass(frozen=True)
class Workload:
    """One named synthetic workload (sizes, layout, mask recipe, seed)."""

    name: str
    kind: str  # "prefill" or "decode"
    B: int
    Hq: int
    Hkv: int
    S_q: int
    S_kv: int
    D: int
    layout: str  # "BNSD" or "BSND"
    causal: bool = False
    seed: int = 0
    # decode: valid KV length drawn iid uniform in [len_lo, len_hi]
    len_lo: int | None = None
    len_hi: int | None = None
    garbage: bool = False
    # prefill: per-batch count of masked trailing keys, uniform in [0, max_pad]
    max_pad: int | None = None
    # prefill: sliding window (win_left, win_right), -1 = no limit on that side
    window: tuple | None = None
    # paged K/V cache of blocks of this many rows (PA_BBND, shuffled), or None
    block_size: int | None = None
    # prefill: B packed sequences (TND) of lengths drawn uniform in
    # [len_lo, len_hi] (equal q and kv lengths), S_q = S_kv = len_hi
    packed: bool = False
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)


# The five workloads of the pages' problem statement (sizes as given there).
WORKLOADS: dict[str, Workload] = {
    "tiny_prefill": Workload(
        "tiny_prefill", "prefill", B=1, Hq=2, Hkv=2, S_q=128, S_kv=128, D=64,
        layout="BNSD", seed=101,
        note="B=1 N=2 S=128 D=64 BNSD, no mask, LSE out"),
    "gqa_decode": Workload(
        "gqa_decode", "decode", B=8, Hq=32, Hkv=8, S_q=1, S_kv=8192, D=128,
        layout="BNSD", seed=102, len_lo=1024, len_hi=8192, garbage=True,
        note="B=8 Hq=32 Hkv=8 D=128 BNSD, cache padded to 8192, L_b~U[1024,8192]"),
    "long_decode": Workload(
        "long_decode", "decode", B=1, Hq=32, Hkv=32, S_q=1, S_kv=131072, D=128,
        layout="BSND", seed=103, len_lo=131072, len_hi=131072, garbage=False,
        note="B=1 H=32 D=128 BSND, 131072 valid keys, split-KV"),
    "causal_prefill": Workload(
        "causal_prefill", "prefill", B=4, Hq=32, Hkv=32, S_q=4096, S_kv=4096, D=128,
        layout="BSND", causal=True, seed=104,
        note="B=4 H=32 S=4096 D=128 BSND causal"),
    "gqa_masked_prefill": Workload(
        "gqa_masked_prefill", "prefill", B=2, Hq=64, Hkv=8, S_q=8192, S_kv=8192, D=128,
        layout="BNSD", causal=True, seed=105, max_pad=1024,
        note="B=2 Hq=64 Hkv=8 S=8192 D=128 BNSD causal AND key padding p_b~U[0,1024]"),
    # Beyond the five: causal GQA prefill with head dim 256 (FlashAttn guide
    # §3 tiling for D = 256).
    "d256_prefill": Workload(
        "d256_prefill", "prefill", B=4, Hq=16, Hkv=8, S_q=4096, S_kv=4096, D=256,
        layout="BSND", causal=True, seed=110,
        note="B=4 Hq=16 Hkv=8 S=4096 D=256 BSND causal"),
    # Beyond the five: the sliding-window mask (FlashAttn guide §1.5, mode 4)
    # on a long GQA prefill, each query seeing itself and the 1023 keys before.
    "window_prefill": Workload(
        "window_prefill", "prefill", B=2, Hq=32, Hkv=8, S_q=8192, S_kv=8192, D=128,
        layout="BNSD", seed=106, window=(1023, 0),
        note="B=2 Hq=32 Hkv=8 S=8192 D=128 BNSD, window of 1024 keys (1023 before, 0 after)"),
    # Beyond the five: packed variable-length causal prefill (FlashAttn guide
    # §1.3 TND with cu_seqlens), 16 sequences of 512..8192 tokens.
    "varlen_prefill": Workload(
        "varlen_prefill", "prefill", B=16, Hq=32, Hkv=8, S_q=8192, S_kv=8192, D=128,
        layout="TND", causal=True, seed=108, len_lo=512, len_hi=8192, packed=True,
        note="16 packed sequences (TND), lengths ~U[512,8192], Hq=32 Hkv=8 D=128, causal"),
    # Beyond the five: the causal prefill workload with its K/V in a paged
    # cache (FlashAttn guide §1.2, layout_kv PA_BBND beside q in BSND; 128-row
    # blocks in shuffled order).
    "paged_prefill": Workload(
        "paged_prefill", "prefill", B=4, Hq=32, Hkv=32, S_q=4096, S_kv=4096, D=128,
        layout="BSND", causal=True, seed=112, block_size=128,
        note="B=4 H=32 S=4096 D=128 causal, q BSND, K/V paged (PA_BBND, 128-row blocks, "
             "shuffled)"),
    # Beyond the five: the GQA decode workload with head dim 256 (FlashAttn
    # guide §3 tiling for D = 256).
    "d256_decode": Workload(
        "d256_decode", "decode", B=8, Hq=32, Hkv=8, S_q=1, S_kv=8192, D=256,
        layout="BNSD", seed=109, len_lo=1024, len_hi=8192, garbage=True,
        note="B=8 Hq=32 Hkv=8 D=256 BNSD, cache padded to 8192, L_b~U[1024,8192]"),
    # Beyond the five: a serving-size decode batch, 64 sequences of the GQA
    # decode workload's head layout (512 (batch, KV head) units, more than
    # SMs: the split cuts the shares by cost).
    "batch_decode": Workload(
        "batch_decode", "decode", B=64, Hq=32, Hkv=8, S_q=1, S_kv=4096, D=128,
        layout="BNSD", seed=111, len_lo=256, len_hi=4096, garbage=True,
        note="B=64 Hq=32 Hkv=8 D=128 BNSD, cache padded to 4096, L_b~U[256,4096]"),
    # Beyond the five: the GQA decode workload with its cache paged (FlashAttn
    # guide §1.2, PA_BBND, 128-row blocks in shuffled order).
    "paged_decode": Workload(
        "paged_decode", "decode", B=8, Hq=32, Hkv=8, S_q=1, S_kv=8192, D=128,
        layout="BNSD", seed=107, len_lo=1024, len_hi=8192, garbage=True, block_size=128,
        note="B=8 Hq=32 Hkv=8 D=128, paged cache (PA_BBND, 128-row blocks, shuffled), "
             "L_b~U[1024,8192]"),
}


def _shape(layout: str, B: int, H: int, S: int, D: int) -> tuple[int, int, int, int]:
    if layout == "BNSD":
        return (B, H, S, D)
    if layout == "BSND":
        return (B, S, H, D)
    raise ValueError(f"unknown layout {layout!r}")


def random_bf16_bits(n: int, gen: torch.Generator) -> torch.Tensor:
    """``n`` random 16-bit patterns viewed as bf16 (NaN/Inf included)."""
    bits = torch.randint(-32768, 32768, (n,), generator=gen, dtype=torch.int32)
    return bits.to(torch.int16).view(torch.bfloat16)


def to_bnsd(x: torch.Tensor, layout: str) -> torch.Tensor:
    """View a BSND tensor as BNSD (no copy); BNSD is returned as is."""
    if layout == "BNSD":
        return x
    if layout == "BSND":
        return x.permute(0, 2, 1, 3)
    raise ValueError(f"unknown layout {layout!r}")


def make_prefill(B, Hq, Hkv, S_q, S_kv, D, layout="BNSD", seed=0, *,
                 max_pad: int | None = None, lengths: list[int] | None = None):
    """Q, K, V (bf16, CPU) and an optional per-key mask [B, S_kv] (uint8, 1 = masked).

    ``max_pad``: draw p_b ~ U{0..max_pad} per batch after Q, K, V and mask
    the last p_b keys of batch b.
    ``lengths``: explicit per-batch valid KV lengths (returned unchanged).
    """
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(_shape(layout, B, Hq, S_q, D), generator=g).to(torch.bfloat16)
    k = torch.randn(_shape(layout, B, Hkv, S_kv, D), generator=g).to(torch.bfloat16)
    v = torch.randn(_shape(layout, B, Hkv, S_kv, D), generator=g).to(torch.bfloat16)
    key_mask = None
    pads = None
    if max_pad is not None:
        pads = torch.randint(0, max_pad + 1, (B,), generator=g)
        key_mask = torch.zeros((B, S_kv), dtype=torch.uint8)
        for b in range(B):
            p = int(pads[b])
            if p:
                key_mask[b, S_kv - p:] = 1
        pads = [int(p) for p in pads]
    return {"q": q, "k": k, "v": v, "key_mask": key_mask, "pads": pads,
            "lengths": lengths, "layout": layout}


def make_decode(B, Hq, Hkv, S_kv, D, layout="BNSD", seed=0, *,
                len_lo: int = 1, len_hi: int | None = None, garbage: bool = True,
                lengths: list[int] | None = None):
    """Decode inputs: q with S_q = 1, a padded K/V cache of S_kv rows and
    per-batch valid lengths (drawn iid U[len_lo, len_hi] unless given).

    With ``garbage`` every cache row at or past L_b is overwritten with random
    bf16 bit patterns.
    """
    if len_hi is None:
        len_hi = S_kv
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(_shape(layout, B, Hq, 1, D), generator=g).to(torch.bfloat16)
    k = torch.randn(_shape(layout, B, Hkv, S_kv, D), generator=g).to(torch.bfloat16)
    v = torch.randn(_shape(layout, B, Hkv, S_kv, D), generator=g).to(torch.bfloat16)
    if lengths is None:
        if len_lo == len_hi:
            lengths = [int(len_lo)] * B
        else:
            lengths = [int(x) for x in torch.randint(len_lo, len_hi + 1, (B,), generator=g)]
    if garbage:
        kb, vb = to_bnsd(k, layout), to_bnsd(v, layout)
        for b in range(B):
            L = lengths[b]
            if L < S_kv:
                n = Hkv * (S_kv - L) * D
                kb[b, :, L:, :] = random_bf16_bits(n, g).view(Hkv, S_kv - L, D)
                vb[b, :, L:, :] = random_bf16_bits(n, g).view(Hkv, S_kv - L, D)
    return {"q": q, "k": k, "v": v, "key_mask": None, "lengths": lengths,
            "layout": layout}


def make_packed(B, Hq, Hkv, D, seed, *, len_lo, len_hi):
    """Packed (TND) prefill inputs: sequence lengths drawn first, then q, k,
    v [T, H, D] from randn cast to bf16; cu_seqlens (equal for q and kv)."""
    g = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in torch.randint(len_lo, len_hi + 1, (B,), generator=g)]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    T = cu[-1]
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v, "cu_seqlens": cu, "lengths": lens, "layout": "TND",
            "key_mask": None}


def make(w: Workload | str):
    """Inputs of a named workload (see ``WORKLOADS``)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if w.packed:
        return make_packed(w.B, w.Hq, w.Hkv, w.D, w.seed, len_lo=w.len_lo, len_hi=w.len_hi)
    if w.kind == "prefill":
        return make_prefill(w.B, w.Hq, w.Hkv, w.S_q, w.S_kv, w.D, w.layout, w.seed,
                            max_pad=w.max_pad)
    return make_decode(w.B, w.Hq, w.Hkv, w.S_kv, w.D, w.layout, w.seed,
                       len_lo=w.len_lo, len_hi=w.len_hi, garbage=w.garbage)
