"""GPU parity of the sliding-window prefill (fa_forward_window) against the
fp64 oracle. The window reading is FlashAttn guide §1.5 (mask_mode 4): query
i sees keys i - win_left .. i + win_right, -1 = no limit on that side.
Tolerances as in test_gpu_parity.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import fa as F

from test_gpu_parity import compare, _gpu

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, S, D, layout, (win_left, win_right), max_pad, lens
    (1, 2, 2, 300, 64, "BNSD", (0, 0), None, None),
    (2, 4, 2, 640, 128, "BSND", (100, 0), None, None),
    (1, 2, 1, 1000, 128, "BNSD", (200, 200), None, None),
    (2, 8, 2, 512, 128, "BNSD", (-1, 64), 300, None),
    (1, 2, 2, 700, 64, "BSND", (129, 1), None, [650]),
    (1, 4, 4, 384, 128, "BNSD", (1000, 1000), None, None),
    (1, 2, 2, 257, 128, "BNSD", (300, -1), None, None),
    (2, 4, 4, 129, 64, "BSND", (5, 300), 64, None),
    (1, 4, 2, 600, 256, "BNSD", (100, 30), None, None),
    (2, 2, 2, 300, 256, "BSND", (63, 0), 40, None),
]


def _run(x, window, scale, lens=None):
    out, lse = F.fa_forward_window(_gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"]), window[0], window[1],
                                   key_mask=_gpu(x["key_mask"]), actual_seq_lengths=lens,
                                   scale=scale, layout=x["layout"])
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("B,Hq,Hkv,S,D,layout,window,max_pad,lens", CASES)
def test_window_matches_oracle(cuda_device, B, Hq, Hkv, S, D, layout, window, max_pad, lens):
    x = workloads.make_prefill(B, Hq, Hkv, S, S, D, layout, seed=2000 + S + D, max_pad=max_pad)
    scale = 1.0 / math.sqrt(D)
    out, lse = _run(x, window, scale, lens)
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=scale, layout=layout,
                              key_mask=x["key_mask"], actual_seq_lengths=lens, window=window)
    compare(out, lse, ro, rl, layout)


def test_window_left_unbounded_right_zero_equals_causal_bitwise(cuda_device):
    x = workloads.make_prefill(2, 4, 2, 600, 600, 128, "BSND", seed=5, max_pad=200)
    q, k, v, km = _gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"]), _gpu(x["key_mask"])
    a = F.fa_forward(q, k, v, mask_mode="causal", key_mask=km, scale=0.08, layout="BSND")
    b = F.fa_forward_window(q, k, v, -1, 0, key_mask=km, scale=0.08, layout="BSND")
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_window_long_sequence_sampled_rows(cuda_device):
    """8192 keys, a 1024-token look-back window: most KV tiles of every Q tile
    are skipped; checked on a seeded sample of rows that covers all heads."""
    B, H, S, D = 1, 8, 8192, 128
    x = workloads.make_prefill(B, H, H, S, S, D, "BNSD", seed=77)
    window = (1024, 0)
    scale = 1.0 / math.sqrt(D)
    out, lse = _run(x, window, scale)
    g = np.random.default_rng(3)
    rows = sorted(set([0, 1, 127, 128, 1023, 1024, 1025, S - 1] +
                      g.choice(S, 56, replace=False).tolist()))
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=scale, window=window, rows=rows)
    compare(out, lse, ro, rl, "BNSD", rows=rows)


def test_window_workload_sampled_rows(cuda_device):
    """The bench's window workload at full size (B=2, Hq=32, Hkv=8, S=8192,
    window (1023, 0)), on sampled rows of every head."""
    w = workloads.WORKLOADS["window_prefill"]
    x = workloads.make(w)
    out, lse = _run(x, w.window, w.scale)
    g = np.random.default_rng(5)
    rows = sorted(set([0, 1022, 1023, 1024, 1025, 4096, w.S_q - 1] +
                      g.choice(w.S_q, 41, replace=False).tolist()))
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=w.scale, layout=w.layout,
                              window=w.window, rows=rows)
    compare(out, lse, ro, rl, w.layout, rows=rows)
