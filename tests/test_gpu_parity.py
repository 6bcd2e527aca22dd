"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (bf16 output, fp32 LSE): max |out err| <= 2e-2, mean |out err|
<= 2e-3, max |lse err| <= 1e-3. Rows with no valid key must be exactly 0
with lse = +inf (FlashAttn guide §1.7). Small cases are compared element by
element; the full-size workloads on a seeded sample of query rows that
covers every head.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from attention_forward_qk_gb300 import fa as F
from attention_forward_qk_gb300 import _lib

pytestmark = pytest.mark.gpu

OUT_MAX = 2e-2
OUT_MEAN = 2e-3
LSE_MAX = 1e-3


def _gpu(x):
    return x.cuda() if x is not None else None


def compare(out_gpu, lse_gpu, out_ref, lse_ref, layout, rows=None):
    """out_gpu: bf16 tensor in `layout`; out_ref: fp64 array in `layout`;
    lse_*: [B, Hq, rows]. With `rows`, out_gpu/lse_gpu are first sliced."""
    o = workloads.to_bnsd(out_gpu.detach().cpu(), layout).double()
    if rows is not None:
        o = o[:, :, rows, :]
    o = o.numpy()
    r = workloads.to_bnsd(torch.from_numpy(np.ascontiguousarray(out_ref)), layout).numpy()
    lg = lse_gpu.detach().cpu().double().numpy()
    if rows is not None:
        lg = lg[:, :, rows]
    invalid = ~np.isfinite(lse_ref)
    assert np.array_equal(invalid, ~np.isfinite(lg)), "invalid-row pattern differs"
    assert np.all(lg[invalid] == np.inf)
    assert np.all(o[invalid] == 0.0)
    assert np.all(np.isfinite(o))
    err = np.abs(o - r)
    ok = ~invalid
    if ok.any():
        assert err.max() <= OUT_MAX, f"max |out err| {err.max():.3e}"
        assert err[ok].mean() <= OUT_MEAN, f"mean |out err| {err[ok].mean():.3e}"
        lerr = np.abs(lg[ok] - lse_ref[ok])
        assert lerr.max() <= LSE_MAX, f"max |lse err| {lerr.max():.3e}"
    return float(err.max())


def run_prefill(x, *, causal, scale, lens=None):
    q, k, v = _gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"])
    km = _gpu(x["key_mask"])
    out, lse = F.fa_forward(q, k, v, mask_mode="causal" if causal else None, key_mask=km,
                            actual_seq_lengths=lens, scale=scale, layout=x["layout"])
    torch.cuda.synchronize()
    return out, lse


PREFILL_CASES = [
    # B, Hq, Hkv, S_q, S_kv, D, layout, causal, max_pad, lens
    (1, 2, 2, 128, 128, 64, "BNSD", False, None, None),
    (1, 1, 1, 1, 1, 128, "BNSD", False, None, None),
    (2, 4, 2, 300, 300, 128, "BSND", True, None, None),
    (1, 2, 1, 200, 333, 64, "BNSD", False, None, None),
    (2, 8, 2, 640, 640, 128, "BNSD", True, 300, None),
    (3, 2, 2, 257, 257, 64, "BSND", False, None, [257, 100, 0]),
    (2, 8, 1, 512, 512, 128, "BNSD", False, 700, None),
    (1, 4, 4, 1000, 1000, 128, "BSND", True, None, [999]),
    (2, 2, 2, 129, 129, 64, "BSND", True, 128, None),
    # head dim 256: one 128-row Q tile per work item, 64-key KV tiles
    (1, 2, 2, 300, 300, 256, "BNSD", False, None, None),
    (2, 4, 2, 520, 520, 256, "BSND", True, None, None),
    (2, 8, 2, 384, 384, 256, "BNSD", True, 200, None),
    (2, 2, 1, 200, 333, 256, "BSND", False, 100, [333, 64]),
]


@pytest.mark.parametrize("B,Hq,Hkv,S_q,S_kv,D,layout,causal,max_pad,lens", PREFILL_CASES)
def test_prefill_matches_oracle(cuda_device, B, Hq, Hkv, S_q, S_kv, D, layout, causal, max_pad,
                                lens):
    x = workloads.make_prefill(B, Hq, Hkv, S_q, S_kv, D, layout, seed=1000 + S_q + D,
                               max_pad=max_pad)
    if lens is not None:
        # keys past the length hold NaN/Inf garbage: they must not leak
        kb, vb = workloads.to_bnsd(x["k"], layout), workloads.to_bnsd(x["v"], layout)
        g = torch.Generator().manual_seed(7)
        for b, L in enumerate(lens):
            if L < S_kv:
                n = Hkv * (S_kv - L) * D
                kb[b, :, L:] = workloads.random_bf16_bits(n, g).view(Hkv, S_kv - L, D)
                vb[b, :, L:] = workloads.random_bf16_bits(n, g).view(Hkv, S_kv - L, D)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_prefill(x, causal=causal, scale=scale, lens=lens)
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=scale, layout=layout, causal=causal,
                              key_mask=x["key_mask"], actual_seq_lengths=lens)
    compare(out, lse, ro, rl, layout)


def test_prefill_fully_masked_batch_gives_invalid_rows(cuda_device):
    x = workloads.make_prefill(2, 2, 2, 200, 200, 128, "BNSD", seed=3)
    km = torch.zeros(2, 200, dtype=torch.uint8)
    km[1] = 1
    x["key_mask"] = km
    out, lse = run_prefill(x, causal=True, scale=0.09)
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=0.09, causal=True, key_mask=km)
    compare(out, lse, ro, rl, "BNSD")
    assert torch.all(out[1].float() == 0) and torch.all(torch.isinf(lse[1]))


def test_prefill_scale_zero_and_negative(cuda_device):
    x = workloads.make_prefill(1, 2, 2, 256, 256, 64, "BNSD", seed=11)
    for scale in (0.0, -0.2):
        out, lse = run_prefill(x, causal=True, scale=scale)
        ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=scale, causal=True)
        compare(out, lse, ro, rl, "BNSD")


def test_prefill_is_bitwise_deterministic(cuda_device):
    x = workloads.make_prefill(2, 4, 2, 777, 777, 128, "BSND", seed=5, max_pad=100)
    a = run_prefill(x, causal=True, scale=0.1)
    b = run_prefill(x, causal=True, scale=0.1)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def _sample_rows(S, pads, seed, n=24):
    g = np.random.default_rng(seed)
    rows = {0, 1, 2, 127, 128, 129, 255, 256, S // 2, S - 129, S - 128, S - 2, S - 1}
    for p in pads or []:
        for r in (S - p - 1, S - p, S - p + 1):
            if 0 <= r < S:
                rows.add(r)
    while len(rows) < n:
        rows.add(int(g.integers(0, S)))
    return sorted(rows)


@pytest.mark.parametrize("name", ["tiny_prefill", "causal_prefill", "gqa_masked_prefill",
                                  "d256_prefill"])
def test_prefill_workloads(cuda_device, name):
    w = workloads.WORKLOADS[name]
    x = workloads.make(w)
    out, lse = run_prefill(x, causal=w.causal, scale=w.scale)
    rows = None if w.S_q <= 1024 else _sample_rows(w.S_q, x["pads"], w.seed)
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=w.scale, layout=w.layout,
                              causal=w.causal, key_mask=x["key_mask"], rows=rows)
    compare(out, lse, ro, rl, w.layout, rows=rows)


# ------------------------------------------------------------------ decode

def run_decode(x, *, scale, splits=0, key_mask=None):
    q, k, v = _gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"])
    out, lse = F.fa_decode(q, k, v, x["lengths"], key_mask=_gpu(key_mask), scale=scale,
                           layout=x["layout"], num_splits=splits)
    torch.cuda.synchronize()
    return out, lse


DECODE_CASES = [
    # B, Hq, Hkv, S_kv, D, layout, lo, hi, splits, masked
    (4, 8, 2, 1000, 128, "BNSD", 1, 1000, 0, False),
    (3, 16, 2, 700, 64, "BSND", 0, 700, 0, False),
    (2, 64, 8, 2048, 128, "BNSD", 100, 2048, 0, True),
    (5, 6, 3, 333, 128, "BSND", 0, 333, 4, False),
    (1, 4, 4, 4096, 64, "BNSD", 4096, 4096, 7, True),
    (2, 32, 1, 513, 128, "BNSD", 1, 513, 0, False),
    # head dim 256 (decode only): G = 4, 1 and 2 heads per CTA
    (3, 16, 4, 700, 256, "BNSD", 0, 700, 0, False),
    (2, 8, 8, 2500, 256, "BSND", 1, 2500, 5, True),
    (4, 16, 8, 1200, 256, "BNSD", 100, 1200, 0, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,S_kv,D,layout,lo,hi,splits,masked", DECODE_CASES)
def test_decode_matches_oracle(cuda_device, B, Hq, Hkv, S_kv, D, layout, lo, hi, splits, masked):
    x = workloads.make_decode(B, Hq, Hkv, S_kv, D, layout, seed=2000 + S_kv, len_lo=lo,
                              len_hi=hi, garbage=True)
    km = None
    if masked:
        km = (torch.rand(B, S_kv, generator=torch.Generator().manual_seed(3)) < 0.3).to(torch.uint8)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_decode(x, scale=scale, splits=splits, key_mask=km)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=scale, layout=layout,
                           key_mask=km)
    compare(out, lse, ro, rl, layout)


def test_decode_zero_lengths_are_invalid_rows(cuda_device):
    x = workloads.make_decode(3, 4, 2, 256, 128, "BNSD", seed=9, lengths=[0, 256, 0])
    out, lse = run_decode(x, scale=0.1)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=0.1)
    compare(out, lse, ro, rl, "BNSD")


def test_gqa_decode_workload(cuda_device):
    w = workloads.WORKLOADS["gqa_decode"]
    x = workloads.make(w)
    out, lse = run_decode(x, scale=w.scale)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=w.scale, layout=w.layout)
    compare(out, lse, ro, rl, w.layout)
    # repeat: bitwise identical
    out2, lse2 = run_decode(x, scale=w.scale)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)


def test_decode_reuses_a_dirty_workspace(cuda_device):
    # The pieces of a sequence cut across CTAs are counted in the workspace and
    # merged by the CTA that finishes the last one: one workspace, filled with
    # 0xFF bytes first, serves calls whose lengths cut the sequences into
    # different numbers of pieces (and some into none), each exact.
    B, Hq, Hkv, S, D = 4, 32, 8, 4096, 128
    size = F.fa_decode_workspace_size(B, S, Hq, Hkv, D, 0)
    ws = torch.full((size,), 255, dtype=torch.uint8, device="cuda")
    for seed, lo, hi in [(11, 1, 4096), (12, 3000, 4096), (13, 0, 60), (14, 1, 4096)]:
        x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=seed, len_lo=lo, len_hi=hi)
        q, k, v = _gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"])
        out, lse = F.fa_decode(q, k, v, x["lengths"], scale=0.09, workspace=ws)
        torch.cuda.synchronize()
        ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=0.09)
        compare(out, lse, ro, rl, "BNSD")


@pytest.mark.parametrize("name", ["d256_decode", "batch_decode"])
def test_decode_workload(cuda_device, name):
    w = workloads.WORKLOADS[name]
    x = workloads.make(w)
    out, lse = run_decode(x, scale=w.scale)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=w.scale, layout=w.layout)
    compare(out, lse, ro, rl, w.layout)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,layout,masked", [
    # more (batch, KV head, head group) units than SMs: the shares are cut in
    # equal cost, each unit start costing 192 * 128 / D rows (their first rows
    # computed on the host, or, when the launch parameters have no room for
    # them, 871 to 1024 sequences, by the kernel)
    (48, 16, 4, 1500, 256, "BNSD", False),   # G = 4 at D = 256: 192 units
    (8, 32, 32, 3000, 128, "BSND", True),    # G = 1: 256 units, with a key mask
    (32, 64, 8, 1200, 64, "BNSD", False),    # G = 8 at D = 64: 256 units
    (160, 4, 1, 900, 128, "BSND", False),    # one unit per sequence, 160 units
    (900, 8, 2, 300, 128, "BNSD", False),    # G = 4, 1800 units, shares found by the kernel
    (1030, 8, 2, 200, 128, "BSND", True),    # prefix sums in the workspace, shares from the host
])
def test_decode_shares_by_cost(cuda_device, B, Hq, Hkv, S, D, layout, masked):
    x = workloads.make_decode(B, Hq, Hkv, S, D, layout, seed=B + D, len_lo=0, len_hi=S)
    km = None
    if masked:
        g = torch.Generator().manual_seed(B)
        km = (torch.rand(B, S, generator=g) < 0.2).to(torch.uint8)
    out, lse = run_decode(x, scale=D ** -0.5, key_mask=km)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=D ** -0.5,
                           layout=layout, key_mask=km)
    compare(out, lse, ro, rl, layout)


@pytest.mark.parametrize("splits", [128, 1024])
def test_decode_forced_splits_many_shares_per_cta(cuda_device, splits):
    # a forced split count cuts fixed-size shares (64 rows at 1024 splits):
    # 2048 shares for 152 CTAs, each CTA taking its shares in turn
    x = workloads.make_decode(2, 32, 8, 8192, 128, "BNSD", seed=splits, len_lo=5000,
                              len_hi=8192)
    out, lse = run_decode(x, scale=0.088, splits=splits)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=0.088, layout="BNSD")
    compare(out, lse, ro, rl, "BNSD")


def test_decode_forced_splits_more_shares_than_ctas_can_hold(cuda_device):
    # 1024 sequences x 4 heads, 10 shares of 64 rows each: 40 960 shares, more
    # than 152 CTAs x 256 shares, so the grid grows past the SM count; checked
    # on a sample of the sequences (the oracle runs per sequence)
    B, H, S, D = 1024, 4, 640, 64
    lens = [S] * B
    lens[3] = lens[700] = 0
    lens[5], lens[511], lens[1023] = 1, 63, 65
    x = workloads.make_decode(B, H, H, S, D, "BSND", seed=77, lengths=lens, garbage=False)
    out, lse = run_decode(x, scale=0.125, splits=10)
    for b in [0, 3, 5, 6, 200, 511, 700, 701, 1000, 1023]:
        sl = slice(b, b + 1)
        ro, rl = oracle.decode(x["q"][sl], x["k"][sl], x["v"][sl], lens[sl], scale=0.125,
                               layout="BSND")
        compare(out[sl], lse[sl], ro, rl, "BSND")


@pytest.mark.parametrize("B", [257, 1030])
def test_decode_many_sequences(cuda_device, B):
    # the lengths' prefix sums travel in the larger parameter block (B <= 1024)
    # or in the workspace (B > 1024)
    x = workloads.make_decode(B, 4, 2, 64, 64, "BSND", seed=B, len_lo=0, len_hi=64)
    out, lse = run_decode(x, scale=0.125)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=0.125, layout="BSND")
    compare(out, lse, ro, rl, "BSND")


def test_decode_replays_from_a_cuda_graph(cuda_device):
    # One fa_decode call captured into a CUDA graph (the counter clear and the
    # kernel), replayed with new cache contents: every replay is exact, so the
    # per-sequence piece counters start from zero each time.
    B, Hq, Hkv, S, D = 4, 32, 8, 4096, 128
    lens = [4096, 1500, 3333, 77]
    x = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=21, lengths=lens)
    q, k, v = _gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"])
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, 1, dtype=torch.float32, device="cuda")
    ws = torch.empty(F.fa_decode_workspace_size(B, S, Hq, Hkv, D, 0), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        F.fa_decode(q, k, v, lens, scale=0.1, out=out, lse=lse, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        F.fa_decode(q, k, v, lens, scale=0.1, out=out, lse=lse, workspace=ws, stream=s)
    for seed in (22, 23, 24):
        y = workloads.make_decode(B, Hq, Hkv, S, D, "BNSD", seed=seed, lengths=lens)
        q.copy_(_gpu(y["q"]))
        k.copy_(_gpu(y["k"]))
        v.copy_(_gpu(y["v"]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.decode(y["q"], y["k"], y["v"], lens, scale=0.1)
        compare(out, lse, ro, rl, "BNSD")


@pytest.fixture(scope="module")
def long_decode():
    w = workloads.WORKLOADS["long_decode"]
    x = workloads.make(w)
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["lengths"], scale=w.scale, layout=w.layout)
    g = {k: (_gpu(v) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    return w, g, ro, rl


@pytest.mark.parametrize("splits", [0, 128, 256, 512, 1024])
def test_long_decode_workload(cuda_device, long_decode, splits):
    w, x, ro, rl = long_decode
    out, lse = F.fa_decode(x["q"], x["k"], x["v"], x["lengths"], scale=w.scale, layout=w.layout,
                           num_splits=splits)
    torch.cuda.synchronize()
    compare(out, lse, ro, rl, w.layout)


# --------------------------------------------------------------- failures

def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert F.fa_selftest_wait_timeout(ws, 2_000_000) == _lib.FA_OK
    assert F.fa_workspace_status(ws) == _lib.FA_ERR_DEVICE_TIMEOUT
    assert F.fa_workspace_status(ws) == _lib.FA_OK  # read clears it
    # the context is still usable
    x = workloads.make_prefill(1, 2, 2, 128, 128, 64, "BNSD", seed=1)
    out, lse = run_prefill(x, causal=False, scale=0.125)
    ro, rl = oracle.attention(x["q"], x["k"], x["v"], scale=0.125)
    compare(out, lse, ro, rl, "BNSD")


def test_normal_calls_leave_status_clear(cuda_device):
    x = workloads.make_prefill(1, 2, 2, 300, 300, 128, "BNSD", seed=2)
    q, k, v = _gpu(x["q"]), _gpu(x["k"]), _gpu(x["v"])
    ws = torch.empty(F.fa_forward_workspace_size(1, 300, 300, 2, 2, 128), dtype=torch.uint8,
                     device="cuda")
    F.fa_forward(q, k, v, mask_mode="causal", scale=0.1, workspace=ws)
    assert F.fa_workspace_status(ws) == _lib.FA_OK
