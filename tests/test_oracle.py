"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a brute-force restatement, a library
routine (torch's fp64 SDPA), a closed form, a value printed by the pages, or
an invariant of the definition. Sources are cited by page title and section:
  [FA]  "FlashAttn" operator README + developer guide (ops-transformer)
  [IFA] "aclnnIncreFlashAttention usage guide and implementation analysis"
  [FD]  "FlashDecoding" Ascend C tutorial
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(B, Hq, Hkv, S_q, S_kv, D, layout, seed, *, mask=False, lengths=None):
    x = workloads.make_prefill(B, Hq, Hkv, S_q, S_kv, D, layout, seed,
                               max_pad=(S_kv // 2 if mask else None))
    return x["q"], x["k"], x["v"], x["key_mask"], lengths


SMALL = [
    # B, Hq, Hkv, S_q, S_kv, D, layout, causal, mask, lengths
    (1, 1, 1, 5, 7, 4, "BNSD", False, False, None),
    (2, 4, 2, 6, 6, 8, "BNSD", True, False, None),
    (2, 4, 1, 6, 6, 3, "BSND", True, True, None),
    (2, 2, 2, 4, 9, 5, "BSND", False, True, [9, 3]),
    (3, 6, 3, 7, 7, 4, "BNSD", True, False, [7, 0, 4]),
    (1, 3, 3, 1, 11, 6, "BNSD", False, False, [8]),
]


@pytest.mark.parametrize("B,Hq,Hkv,S_q,S_kv,D,layout,causal,mask,lengths", SMALL)
def test_vectorised_matches_bruteforce(B, Hq, Hkv, S_q, S_kv, D, layout, causal, mask, lengths):
    q, k, v, km, lens = _case(B, Hq, Hkv, S_q, S_kv, D, layout, 7 + B + S_kv, mask=mask,
                              lengths=lengths)
    scale = 1.0 / math.sqrt(D)
    o1, l1 = oracle.attention(q, k, v, scale=scale, layout=layout, causal=causal,
                              key_mask=km, actual_seq_lengths=lens)
    o2, l2 = oracle.attention_bruteforce(q, k, v, scale=scale, layout=layout, causal=causal,
                                         key_mask=km, actual_seq_lengths=lens)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    fin = np.isfinite(l2)
    assert np.array_equal(fin, np.isfinite(l1))
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)
    assert np.all(l1[~fin] == np.inf)


@pytest.mark.parametrize("B,Hq,Hkv,S_q,S_kv,D,layout,causal,mask,lengths", SMALL + [
    (2, 8, 2, 33, 33, 16, "BSND", True, True, None),
    (1, 4, 4, 17, 40, 32, "BNSD", False, True, [29]),
])
def test_matches_torch_sdpa_fp64(B, Hq, Hkv, S_q, S_kv, D, layout, causal, mask, lengths):
    """Library special case: torch's SDPA in float64 on CPU (its boolean mask
    is True = attend, the opposite polarity of the pages' mask)."""
    q, k, v, km, lens = _case(B, Hq, Hkv, S_q, S_kv, D, layout, 100 + S_q, mask=mask,
                              lengths=lengths)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.attention(q, k, v, scale=scale, layout=layout, causal=causal,
                                key_mask=km, actual_seq_lengths=lens)
    qt, kt, vt = (workloads.to_bnsd(t, layout).double() for t in (q, k, v))
    g = Hq // Hkv
    kt = kt.repeat_interleave(g, dim=1)
    vt = vt.repeat_interleave(g, dim=1)
    attend = torch.ones(B, 1, S_q, S_kv, dtype=torch.bool)
    for b in range(B):
        L = S_kv if lens is None else lens[b]
        attend[b, :, :, L:] = False
        if km is not None:
            attend[b, :, :, km[b].bool()] = False
    if causal:
        attend &= torch.ones(S_q, S_kv, dtype=torch.bool).tril()
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=attend,
                                                           scale=scale)
    s = scale * qt @ kt.transpose(-1, -2)
    s = s.masked_fill(~attend, float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    out_n = workloads.to_bnsd(torch.from_numpy(out), layout).numpy()
    rows_ok = attend.any(-1).expand(B, Hq, S_q).numpy()
    np.testing.assert_allclose(out_n[rows_ok], ref.numpy()[rows_ok], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[rows_ok], ref_lse.numpy()[rows_ok], rtol=0, atol=1e-12)
    assert np.all(out_n[~rows_ok] == 0) and np.all(lse[~rows_ok] == np.inf)


def test_ifa_worked_example():
    """[IFA] §七: the page's own example call (all-ones fp16 inputs)."""
    with open(os.path.join(GOLDEN, "ifa_example.json")) as f:
        g = json.load(f)
    B, N, Nkv, D, S = g["B"], g["num_heads"], g["num_kv_heads"], g["D"], g["S_kv"]
    q = torch.full((B, N, 1, D), g["fill"], dtype=torch.float16)
    k = torch.full((B, Nkv, S, D), g["fill"], dtype=torch.float16)
    v = torch.full((B, Nkv, S, D), g["fill"], dtype=torch.float16)
    mask = torch.full((B, S), g["mask_value"], dtype=torch.int8)
    out, lse = oracle.decode(q, k, v, g["actual_seq_lengths"], scale=g["scale"],
                             layout=g["layout"], key_mask=mask)
    assert np.all(out == g["expected_out"])
    np.testing.assert_allclose(lse, g["expected_lse"], rtol=0, atol=1e-12)


def test_two_key_closed_form():
    """Hand-worked case: q=(1,0), k1=(1,0), k2=(0,1), scale 1 -> scores (1, 0);
    out = (e*v1 + v2)/(e + 1), lse = ln(e + 1)."""
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    v = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    out, lse = oracle.attention(q, k, v, scale=1.0)
    e = math.e
    np.testing.assert_allclose(out[0, 0, 0], [(e * 1 + 3) / (e + 1), (e * 2 + 4) / (e + 1)],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], math.log(e + 1), rtol=0, atol=1e-15)
    # scale enters the scores: scale 2 -> scores (2, 0)
    out2, lse2 = oracle.attention(q, k, v, scale=2.0)
    e2 = math.e ** 2
    np.testing.assert_allclose(out2[0, 0, 0, 0], (e2 * 1 + 3) / (e2 + 1), atol=1e-15)
    np.testing.assert_allclose(lse2[0, 0, 0], math.log(e2 + 1), atol=1e-15)


def test_single_valid_key_returns_its_value_row():
    q, k, v, _, _ = _case(2, 4, 2, 3, 10, 8, "BNSD", 3)
    lens = [1, 1]
    out, lse = oracle.attention(q, k, v, scale=0.3, actual_seq_lengths=lens)
    for b in range(2):
        for h in range(4):
            np.testing.assert_array_equal(out[b, h], np.broadcast_to(v[b, h // 2, 0].double().numpy(), (3, 8)))
            s = 0.3 * (q[b, h].double() @ k[b, h // 2, 0].double()).numpy()
            np.testing.assert_allclose(lse[b, h], s, atol=1e-12)
    # causal: row 0 sees exactly key 0
    out, lse = oracle.attention(q[:, :, :3], k[:, :, :3], v[:, :, :3], scale=0.3, causal=True)
    np.testing.assert_array_equal(out[:, :, 0], v[:, :, 0].double().numpy().repeat(2, axis=1))


def test_zero_scale_gives_mean_of_valid_rows():
    q, k, v, km, _ = _case(2, 2, 2, 4, 12, 6, "BSND", 11, mask=True)
    lens = [12, 7]
    out, lse = oracle.attention(q, k, v, scale=0.0, layout="BSND", key_mask=km,
                                actual_seq_lengths=lens)
    vn = workloads.to_bnsd(v, "BSND").double().numpy()
    on = workloads.to_bnsd(torch.from_numpy(out), "BSND").numpy()
    for b in range(2):
        sel = [j for j in range(lens[b]) if km[b, j] == 0]
        for h in range(2):
            np.testing.assert_allclose(on[b, h], np.broadcast_to(vn[b, h, sel].mean(0), (4, 6)),
                                       atol=1e-13)
            np.testing.assert_allclose(lse[b, h], math.log(len(sel)), atol=1e-13)


def test_constant_value_rows_give_that_constant():
    q, k, _, _, _ = _case(1, 4, 2, 9, 9, 8, "BNSD", 5)
    v = torch.full((1, 2, 9, 8), -0.75)
    out, _ = oracle.attention(q, k, v, scale=0.5, causal=True)
    np.testing.assert_allclose(out, -0.75, atol=1e-15)


def test_invalid_rows_zero_out_and_infinite_lse():
    """[FA] §1.7: a row with no valid key writes 0 and lse = +inf."""
    q, k, v, _, _ = _case(2, 2, 1, 3, 5, 4, "BNSD", 9)
    km = torch.zeros(2, 5, dtype=torch.uint8)
    km[0, :] = 1  # every key of batch 0 masked
    out, lse = oracle.attention(q, k, v, scale=0.5, key_mask=km, actual_seq_lengths=[5, 0])
    assert np.all(out == 0) and np.all(lse == np.inf)


def test_padding_garbage_has_no_effect():
    """Keys at or past the valid length and masked keys may hold anything,
    NaN and Inf included ([IFA] §1.1: inputs are padded to a fixed length)."""
    x = workloads.make_decode(3, 8, 2, 64, 16, "BNSD", seed=21, len_lo=5, len_hi=60, garbage=True)
    q, k, v, lens = x["q"], x["k"], x["v"], x["lengths"]
    assert not torch.isfinite(k.float()).all()  # the generator did plant NaN/Inf
    out1, lse1 = oracle.decode(q, k, v, lens, scale=0.25)
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate(lens):
        k2[b, :, L:] = 7.0
        v2[b, :, L:] = -3.0
    out2, lse2 = oracle.decode(q, k2, v2, lens, scale=0.25)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)
    assert np.all(np.isfinite(out1))
    # masked keys: content irrelevant
    km = torch.zeros(3, 64, dtype=torch.uint8)
    km[:, 1] = 1
    k3, v3 = k.clone(), v.clone()
    k3[:, :, 1] = float("nan")
    v3[:, :, 1] = float("inf")
    a = oracle.decode(q, k, v, lens, scale=0.25, key_mask=km)
    bb = oracle.decode(q, k3, v3, lens, scale=0.25, key_mask=km)
    np.testing.assert_array_equal(a[0], bb[0])


def test_key_permutation_invariance():
    q, k, v, _, _ = _case(1, 2, 2, 5, 13, 8, "BNSD", 31)
    perm = torch.randperm(13, generator=torch.Generator().manual_seed(1))
    a = oracle.attention(q, k, v, scale=0.4)
    b = oracle.attention(q, k[:, :, perm], v[:, :, perm], scale=0.4)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads():
    """[FA] §1.1: g adjacent query heads share one KV head (h -> h // g)."""
    q, k, v, km, _ = _case(2, 8, 2, 6, 6, 4, "BSND", 41, mask=True)
    a = oracle.attention(q, k, v, scale=0.5, layout="BSND", causal=True, key_mask=km)
    kr = k.repeat_interleave(4, dim=2)
    vr = v.repeat_interleave(4, dim=2)
    b = oracle.attention(q, kr, vr, scale=0.5, layout="BSND", causal=True, key_mask=km)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_common_key_shift_moves_lse_only():
    """Adding one vector w to every key adds scale*q_i.w to every score of
    row i: out is unchanged and lse moves by exactly that amount."""
    q, k, v, _, _ = _case(1, 2, 1, 4, 9, 8, "BNSD", 51)
    w = torch.linspace(-1, 1, 8, dtype=torch.float64)
    a_out, a_lse = oracle.attention(q, k, v, scale=0.3, causal=True)
    b_out, b_lse = oracle.attention(q.double(), k.double() + w, v.double(), scale=0.3, causal=True)
    np.testing.assert_allclose(a_out, b_out, atol=1e-12)
    shift = 0.3 * (q.double() @ w).numpy()
    np.testing.assert_allclose(b_lse - a_lse, shift, atol=1e-12)


@pytest.mark.parametrize("n,nchunks", [(1, 1), (37, 1), (37, 4), (300, 7), (1000, 31)])
def test_split_kv_merges_equal_monolithic(n, nchunks):
    """[FA] §10, [FD] §二/§3.3, [IFA] §8.3: every merge of chunk statistics,
    over any partition of the keys, equals the one-pass softmax."""
    rng = np.random.default_rng(n * 131 + nchunks)
    D = 16
    qv = rng.standard_normal(D)
    kk = rng.standard_normal((n, D))
    vv = rng.standard_normal((n, D))
    s = 0.25 * kk @ qv * 3.0  # widen the score range
    cuts = np.sort(rng.choice(np.arange(1, n), size=nchunks - 1, replace=False)) if nchunks > 1 else []
    bounds = [0, *cuts.tolist(), n] if nchunks > 1 else [0, n]
    ms, ls, os_, lses = oracle.split_partials(s, vv, bounds)
    m = s.max()
    p = np.exp(s - m)
    ref = p @ vv / p.sum()
    ref_lse = m + math.log(p.sum())
    o1, l1 = oracle.merge_max_sum(ms, ls, os_)
    o2, l2 = oracle.merge_sequential(ms, ls, os_)
    o3, l3 = oracle.merge_lse(lses, [oi / li for oi, li in zip(os_, ls)])
    for o, l in ((o1, l1), (o2, l2), (o3, l3)):
        np.testing.assert_allclose(o, ref, atol=1e-12)
        assert abs(l - ref_lse) < 1e-12
    # the chunk statistics themselves: lse_i = m_i + ln l_i is the chunk's own logsumexp
    for (a, e), li_lse in zip(zip(bounds[:-1], bounds[1:]), lses):
        assert abs(li_lse - (np.log(np.sum(np.exp(s[a:e] - 5.0))) + 5.0)) < 1e-12


def test_decode_split_merge_matches_full_decode_row():
    """Split-KV over a padded cache row (stage 1 over chunks of the valid keys,
    stage 2 merge) reproduces the oracle's decode output."""
    x = workloads.make_decode(1, 2, 1, 200, 8, "BNSD", seed=61, len_lo=150, len_hi=150)
    q, k, v, lens = x["q"], x["k"], x["v"], x["lengths"]
    out, lse = oracle.decode(q, k, v, lens, scale=0.35)
    for h in range(2):
        s = 0.35 * (k[0, 0, :150].double() @ q[0, h, 0].double()).numpy()
        vv = v[0, 0, :150].double().numpy()
        ms, ls, os_, lses = oracle.split_partials(s, vv, [0, 64, 128, 150])
        o, l = oracle.merge_lse(lses, [oi / li for oi, li in zip(os_, ls)])
        np.testing.assert_allclose(o, out[0, h, 0], atol=1e-12)
        assert abs(l - lse[0, h, 0]) < 1e-12


def test_row_subset_matches_full():
    q, k, v, km, _ = _case(2, 4, 2, 20, 20, 8, "BSND", 71, mask=True)
    full = oracle.attention(q, k, v, scale=0.3, layout="BSND", causal=True, key_mask=km)
    rows = [19, 0, 7, 13]
    part = oracle.attention(q, k, v, scale=0.3, layout="BSND", causal=True, key_mask=km, rows=rows)
    np.testing.assert_array_equal(part[0], full[0][:, rows])
    np.testing.assert_array_equal(part[1], full[1][:, :, rows])


def test_workload_generator_is_seeded_and_shaped():
    a = workloads.make_prefill(2, 4, 2, 8, 8, 16, "BSND", seed=5, max_pad=4)
    b = workloads.make_prefill(2, 4, 2, 8, 8, 16, "BSND", seed=5, max_pad=4)
    for key in ("q", "k", "v", "key_mask"):
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key])
    assert a["q"].shape == (2, 8, 4, 16) and a["k"].shape == (2, 8, 2, 16)
    assert a["q"].dtype == torch.bfloat16
    for bi, p in enumerate(a["pads"]):
        assert int(a["key_mask"][bi].sum()) == p
        if p:
            assert a["key_mask"][bi, -p:].all()
    d = workloads.make_decode(4, 8, 2, 128, 16, "BNSD", seed=3, len_lo=10, len_hi=100)
    assert all(10 <= L <= 100 for L in d["lengths"])
    assert d["q"].shape == (4, 8, 1, 16)


# ---------------------------------------------------------------- window mask
# [FA] developer guide §1.5: mask_mode 4 is a band of win_left keys before and
# win_right keys after each query (-1 = no limit on that side).

WINDOWS = [(0, 0), (2, 0), (3, 1), (-1, 2), (1, -1), (5, 5)]


@pytest.mark.parametrize("window", WINDOWS)
def test_window_vectorised_matches_bruteforce(window):
    q, k, v, km, _ = _case(2, 4, 2, 9, 9, 6, "BSND", 31, mask=True)
    lens = [9, 6]
    scale = 0.4
    o1, l1 = oracle.attention(q, k, v, scale=scale, layout="BSND", key_mask=km,
                              actual_seq_lengths=lens, window=window)
    o2, l2 = oracle.attention_bruteforce(q, k, v, scale=scale, layout="BSND", key_mask=km,
                                         actual_seq_lengths=lens, window=window)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    fin = np.isfinite(l2)
    assert np.array_equal(fin, np.isfinite(l1))
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", WINDOWS)
def test_window_matches_torch_sdpa_band(window):
    """Library special case: torch's fp64 SDPA with the band built by
    tril/triu (True = attend)."""
    B, Hq, Hkv, S, D = 1, 4, 2, 12, 8
    q, k, v, _, _ = _case(B, Hq, Hkv, S, S, D, "BNSD", 57)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.attention(q, k, v, scale=scale, layout="BNSD", window=window)
    qt, kt, vt = (t.double() for t in (q, k, v))
    kt = kt.repeat_interleave(Hq // Hkv, dim=1)
    vt = vt.repeat_interleave(Hq // Hkv, dim=1)
    band = torch.ones(S, S, dtype=torch.bool)
    wl, wr = window
    if wr >= 0:
        band = band.tril(wr)
    if wl >= 0:
        band = band.triu(-wl)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=band, scale=scale)
    s = (scale * qt @ kt.transpose(-1, -2)).masked_fill(~band, float("-inf"))
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_window_left_unbounded_right_zero_is_causal():
    q, k, v, km, _ = _case(2, 2, 1, 10, 10, 4, "BNSD", 77, mask=True)
    a = oracle.attention(q, k, v, scale=0.3, key_mask=km, causal=True)
    b = oracle.attention(q, k, v, scale=0.3, key_mask=km, window=(-1, 0))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_window_zero_width_returns_own_value_row():
    """Closed form: with window (0, 0) query i sees only key i, so out_i =
    v_i and lse_i = s_ii."""
    q, k, v, _, _ = _case(1, 2, 2, 7, 7, 5, "BNSD", 91)
    scale = 0.7
    out, lse = oracle.attention(q, k, v, scale=scale, window=(0, 0))
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    np.testing.assert_allclose(out, vd, rtol=0, atol=1e-15)
    sii = scale * np.einsum("bhid,bhid->bhi", qd, kd)
    np.testing.assert_allclose(lse, sii, rtol=0, atol=1e-12)


def test_window_wider_than_sequence_is_no_mask():
    q, k, v, _, _ = _case(1, 2, 1, 6, 6, 4, "BSND", 13)
    a = oracle.attention(q, k, v, scale=0.5, layout="BSND")
    b = oracle.attention(q, k, v, scale=0.5, layout="BSND", window=(6, 6))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------- packed sequences
# [FA] developer guide §1.3 (TND) and §1.4 (cu_seqlens).

def test_varlen_equals_per_sequence_bruteforce():
    g = torch.Generator().manual_seed(12)
    lq, lkv = [3, 0, 5, 1], [4, 2, 5, 0]
    cq = np.concatenate([[0], np.cumsum(lq)])
    ckv = np.concatenate([[0], np.cumsum(lkv)])
    Hq, Hkv, D = 4, 2, 6
    q = torch.randn(int(cq[-1]), Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(int(ckv[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(int(ckv[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    out, lse = oracle.attention_varlen(q, k, v, cq, ckv, scale=0.3)
    for b in range(4):
        if lq[b] == 0:
            continue
        qs = q[cq[b]:cq[b + 1]][None]
        ks, vs = k[ckv[b]:ckv[b + 1]][None], v[ckv[b]:ckv[b + 1]][None]
        ro, rl = oracle.attention_bruteforce(qs, ks, vs, scale=0.3, layout="BSND")
        np.testing.assert_allclose(out[cq[b]:cq[b + 1]], ro[0], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isfinite(lse[cq[b]:cq[b + 1]]), np.isfinite(rl[0].T))
        fin = np.isfinite(rl[0].T)
        np.testing.assert_allclose(lse[cq[b]:cq[b + 1]][fin], rl[0].T[fin], rtol=0, atol=1e-12)
    # the sequence with no keys: invalid rows (out 0, lse +inf), [FA] §1.7
    assert np.all(out[cq[3]:cq[4]] == 0) and np.all(lse[cq[3]:cq[4]] == np.inf)


def test_varlen_equal_lengths_match_padded_batch():
    """With equal lengths the packed layout is the BSND batch reshaped."""
    B, S, Hq, Hkv, D = 3, 7, 4, 2, 8
    x = workloads.make_prefill(B, Hq, Hkv, S, S, D, "BSND", 21)
    cu = np.arange(B + 1) * S
    o1, l1 = oracle.attention_varlen(x["q"].reshape(B * S, Hq, D), x["k"].reshape(B * S, Hkv, D),
                                     x["v"].reshape(B * S, Hkv, D), cu, cu, scale=0.2,
                                     causal=True)
    o2, l2 = oracle.attention(x["q"], x["k"], x["v"], scale=0.2, layout="BSND", causal=True)
    np.testing.assert_array_equal(o1, o2.reshape(B * S, Hq, D))
    np.testing.assert_array_equal(l1, l2.transpose(0, 2, 1).reshape(B * S, Hq))


def test_varlen_window_equals_per_sequence_bruteforce():
    """A sliding window inside packed sequences ([FA] §1.5 with §1.3): each
    sequence against the scalar-loop definition with its own window."""
    g = torch.Generator().manual_seed(13)
    lens = [6, 1, 9, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    Hq, Hkv, D = 4, 2, 5
    q = torch.randn(int(cu[-1]), Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(int(cu[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(int(cu[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    for window in [(2, 0), (0, 1), (3, 2), (-1, 1)]:
        out, lse = oracle.attention_varlen(q, k, v, cu, cu, scale=0.4, window=window)
        for b in range(len(lens)):
            sl = slice(cu[b], cu[b + 1])
            ro, rl = oracle.attention_bruteforce(q[sl][None], k[sl][None], v[sl][None], scale=0.4,
                                                 layout="BSND", window=window)
            np.testing.assert_allclose(out[sl], ro[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[sl], rl[0].T, rtol=0, atol=1e-12)
    # (-1, 0) is causal
    o1, l1 = oracle.attention_varlen(q, k, v, cu, cu, scale=0.4, window=(-1, 0))
    o2, l2 = oracle.attention_varlen(q, k, v, cu, cu, scale=0.4, causal=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def _packed_inputs(seed, lq, lkv, Hq=4, Hkv=2, D=5):
    g = torch.Generator().manual_seed(seed)
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    ckv = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int64)
    q = torch.randn(int(cq[-1]), Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(int(ckv[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(int(ckv[-1]), Hkv, D, generator=g).to(torch.bfloat16)
    km = (torch.rand(int(ckv[-1]), generator=g) < 0.3).to(torch.uint8)
    return q, k, v, km, cq, ckv


def test_varlen_seqused_and_key_mask_equal_per_sequence_bruteforce():
    """seqused_q / seqused_kv ([FA] §1.4: the shorter of seqused and the
    cu_seqlens span holds) and a per-packed-key mask: each sequence against
    the scalar-loop definition with its used kv length as the actual length
    and its slice of the mask; query rows past the used q length are
    truncated rows (out 0, lse +inf, [FA] §1.7)."""
    lq, lkv = [5, 3, 7, 4, 2], [5, 6, 7, 4, 3]
    sq, skv = [3, 9, 7, 0, 2], [4, 2, 9, 4, 0]   # shorter and longer than the spans
    q, k, v, km, cq, ckv = _packed_inputs(14, lq, lkv)
    for causal in (False, True):
        out, lse = oracle.attention_varlen(q, k, v, cq, ckv, scale=0.35, causal=causal,
                                           seqused_q=sq, seqused_kv=skv, key_mask=km)
        for b in range(len(lq)):
            uq = min(lq[b], sq[b])
            ukv = min(lkv[b], skv[b])
            qs = q[cq[b]:cq[b] + uq][None]
            ks, vs = k[ckv[b]:ckv[b + 1]][None], v[ckv[b]:ckv[b + 1]][None]
            if uq > 0:
                ro, rl = oracle.attention_bruteforce(qs, ks, vs, scale=0.35, layout="BSND",
                                                     causal=causal, key_mask=km[None, ckv[b]:ckv[b + 1]],
                                                     actual_seq_lengths=[ukv])
                np.testing.assert_allclose(out[cq[b]:cq[b] + uq], ro[0], rtol=0, atol=1e-12)
                lg, lr = lse[cq[b]:cq[b] + uq], rl[0].T
                np.testing.assert_array_equal(np.isfinite(lg), np.isfinite(lr))
                fin = np.isfinite(lr)
                np.testing.assert_allclose(lg[fin], lr[fin], rtol=0, atol=1e-12)
                assert np.all(lg[~fin] == np.inf)
            # truncated rows
            assert np.all(out[cq[b] + uq:cq[b + 1]] == 0)
            assert np.all(lse[cq[b] + uq:cq[b + 1]] == np.inf)
        # the sequence whose used kv length is 0 has only invalid rows
        assert np.all(lse[cq[4]:cq[5]] == np.inf)


def test_varlen_seqused_at_or_past_the_span_changes_nothing():
    """seqused at least the cu_seqlens span (the span is then the shorter),
    and an all-zero key mask, give exactly the plain packed result."""
    lq, lkv = [4, 6, 3], [4, 6, 3]
    q, k, v, _, cq, ckv = _packed_inputs(15, lq, lkv)
    o1, l1 = oracle.attention_varlen(q, k, v, cq, ckv, scale=0.5, causal=True)
    o2, l2 = oracle.attention_varlen(q, k, v, cq, ckv, scale=0.5, causal=True,
                                     seqused_q=[4, 100, 3], seqused_kv=[9, 6, 1 << 20],
                                     key_mask=torch.zeros(int(ckv[-1]), dtype=torch.uint8))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_varlen_truncated_rows_and_keys_have_no_effect():
    """Whatever the truncated query rows and the keys past seqused_kv hold
    (NaN and Inf included), the result is the same; only q rows before the
    used length and keys before it enter the arithmetic."""
    lq, lkv = [6, 5], [7, 5]
    sq, skv = [4, 5], [3, 2]
    q, k, v, km, cq, ckv = _packed_inputs(16, lq, lkv)
    o1, l1 = oracle.attention_varlen(q, k, v, cq, ckv, scale=0.5, seqused_q=sq, seqused_kv=skv,
                                     key_mask=km)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    for b in range(2):
        q2[cq[b] + sq[b]:cq[b + 1]] = float("nan")
        k2[ckv[b] + skv[b]:ckv[b + 1]] = float("inf")
        v2[ckv[b] + skv[b]:ckv[b + 1]] = float("nan")
    o2, l2 = oracle.attention_varlen(q2, k2, v2, cq, ckv, scale=0.5, seqused_q=sq,
                                     seqused_kv=skv, key_mask=km)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def _per_head_case(seed, B=2, Hq=4, Hkv=2, S=9, D=6):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, 1, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("mb", [2, 1])
def test_per_head_mask_equals_bruteforce(mb):
    """attenMask of [IFA] §四 with one mask per query head, (B, N, 1, S) and the
    batch-shared (1, N, 1, S): each head against the scalar-loop definition."""
    q, k, v = _per_head_case(17)
    g = torch.Generator().manual_seed(18)
    km = (torch.rand(mb, 4, 9, generator=g) < 0.4).to(torch.uint8)
    km[0, 1, :] = 1  # head 1 of batch 0 (and, shared, of every batch when mb = 1) sees nothing
    lens = [9, 6]
    o1, l1 = oracle.decode(q, k, v, lens, scale=0.3, key_mask=km)
    o2, l2 = oracle.attention_bruteforce(q, k, v, scale=0.3, key_mask=km, actual_seq_lengths=lens)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isfinite(l1), np.isfinite(l2))
    fin = np.isfinite(l2)
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)
    assert np.all(l1[0, 1] == np.inf) and np.all(o1[0, 1] == 0)


def test_per_head_mask_with_equal_rows_is_the_shared_mask():
    """A per-head mask whose heads all carry the same row is exactly the
    (B, 1, 1, S) key mask."""
    q, k, v = _per_head_case(19)
    g = torch.Generator().manual_seed(20)
    km2 = (torch.rand(2, 9, generator=g) < 0.3).to(torch.uint8)
    km3 = km2[:, None, :].expand(2, 4, 9).contiguous()
    o1, l1 = oracle.decode(q, k, v, [9, 8], scale=0.5, key_mask=km2)
    o2, l2 = oracle.decode(q, k, v, [9, 8], scale=0.5, key_mask=km3)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_per_head_mask_keys_masked_for_a_head_have_no_effect_on_it():
    """Whatever a key holds (NaN included), a head that masks it is not
    changed by it; a head that sees it is (the mask is per head)."""
    q, k, v = _per_head_case(21, B=1)
    km = torch.zeros(1, 4, 9, dtype=torch.uint8)
    km[0, 0, 3] = 1  # head 0 masks key 3; head 1 (same KV head) sees it
    o1, l1 = oracle.decode(q, k, v, [9], scale=0.4, key_mask=km)
    k2, v2 = k.clone(), v.clone()
    k2[0, 0, 3] += 1.0
    v2[0, 0, 3] = float("nan")
    o2, l2 = oracle.decode(q, k2, v2, [9], scale=0.4, key_mask=km)
    np.testing.assert_array_equal(o1[0, 0], o2[0, 0])
    np.testing.assert_array_equal(l1[0, 0], l2[0, 0])
    assert not np.all(np.isfinite(o2[0, 1]))  # head 1 reads the changed key
