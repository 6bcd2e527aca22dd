"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function include/fa.h declares, argument errors come back
before any CUDA call, and the decode split plan behaves as documented."""
import ctypes
import math
import os
import re

import pytest

from attention_forward_qk_gb300 import _lib
from attention_forward_qk_gb300 import fa as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

# 16-byte aligned non-null stand-ins: validation must reject before touching them
P = ctypes.c_void_p(0x10000)
WS = ctypes.c_void_p(0x20000)


@pytest.fixture(scope="module")
def lib():
    from attention_forward_qk_gb300 import build as B
    B.build()
    return _lib.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.fa_abi_version() == 1
    for s in range(8):
        assert lib.fa_status_string(s)
    assert b"unknown" in lib.fa_status_string(99)


def test_workspace_sizes(lib):
    a = lib.fa_forward_workspace_size(2, 8192, 8192, 64, 8, 128)
    assert a >= 256 and a % 256 == 0
    assert lib.fa_forward_workspace_size(-1, 1, 1, 1, 1, 64) == 0
    d0 = lib.fa_decode_workspace_size(8, 8192, 32, 8, 128, 0)
    d128 = lib.fa_decode_workspace_size(8, 8192, 32, 8, 128, 128)
    d2 = lib.fa_decode_workspace_size(8, 8192, 32, 8, 128, 2)
    assert d0 > 0 and d128 > 0 and d2 > 0
    # partial outputs dominate: 8*32*splits*128 fp32
    assert d128 >= 8 * 32 * 128 * 128 * 4
    assert d2 < d128
    assert lib.fa_decode_workspace_size(8, 8192, 32, 8, 128, -1) == 0


def _fwd(lib, **kw):
    args = dict(q=P, k=P, v=P, mask_mode=0, key_mask=None, lens=None, B=1, S_q=128, S_kv=128,
                Hq=2, Hkv=2, D=64, scale=0.125, layout=0, out=P, lse=None, ws=WS,
                ws_bytes=1 << 20, stream=None)
    args.update(kw)
    lens = args["lens"]
    if lens is not None:
        lens = (ctypes.c_int64 * len(lens))(*lens)
    return lib.fa_forward(args["q"], args["k"], args["v"], args["mask_mode"], args["key_mask"],
                          lens, args["B"], args["S_q"], args["S_kv"], args["Hq"], args["Hkv"],
                          args["D"], args["scale"], args["layout"], args["out"], args["lse"],
                          args["ws"], args["ws_bytes"], args["stream"])


def _dec(lib, **kw):
    args = dict(q=P, k=P, v=P, key_mask=None, lens=[100, 7], B=2, S=128, Hq=8, Hkv=2, D=128,
                scale=0.1, layout=0, splits=0, out=P, lse=None, ws=WS, ws_bytes=1 << 22,
                stream=None)
    args.update(kw)
    lens = args["lens"]
    if lens is not None:
        lens = (ctypes.c_int64 * max(len(lens), 1))(*lens)
    return lib.fa_decode(args["q"], args["k"], args["v"], args["key_mask"], lens, args["B"],
                         args["S"], args["Hq"], args["Hkv"], args["D"], args["scale"],
                         args["layout"], args["splits"], args["out"], args["lse"], args["ws"],
                         args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), _lib.FA_ERR_NULLPTR),
    (dict(out=None), _lib.FA_ERR_NULLPTR),
    (dict(ws=None), _lib.FA_ERR_NULLPTR),
    (dict(Hq=3, Hkv=2), _lib.FA_ERR_PARAM_INVALID),
    (dict(D=96), _lib.FA_ERR_UNSUPPORTED),
    (dict(D=512), _lib.FA_ERR_UNSUPPORTED),
    (dict(layout=2), _lib.FA_ERR_PARAM_INVALID),
    (dict(mask_mode=4), _lib.FA_ERR_PARAM_INVALID),
    (dict(mask_mode=3, S_q=64, S_kv=128), _lib.FA_ERR_PARAM_INVALID),
    (dict(B=-1), _lib.FA_ERR_PARAM_INVALID),
    (dict(scale=float("nan")), _lib.FA_ERR_PARAM_INVALID),
    (dict(q=ctypes.c_void_p(0x10008)), _lib.FA_ERR_PARAM_INVALID),
    (dict(ws=ctypes.c_void_p(0x20010)), _lib.FA_ERR_PARAM_INVALID),
    (dict(lens=[129]), _lib.FA_ERR_PARAM_INVALID),
    (dict(lens=[-1]), _lib.FA_ERR_PARAM_INVALID),
    (dict(ws_bytes=16), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
])
def test_forward_rejects_before_any_cuda_call(lib, kw, expect):
    assert _fwd(lib, **kw) == expect


def _fwd_window(lib, wl, wr, **kw):
    args = dict(q=P, k=P, v=P, key_mask=None, lens=None, B=1, S_q=128, S_kv=128, Hq=2, Hkv=2,
                D=64, scale=0.125, layout=0, out=P, lse=None, ws=WS, ws_bytes=1 << 20,
                stream=None)
    args.update(kw)
    return lib.fa_forward_window(args["q"], args["k"], args["v"], wl, wr, args["key_mask"],
                                 None, args["B"], args["S_q"], args["S_kv"], args["Hq"],
                                 args["Hkv"], args["D"], args["scale"], args["layout"],
                                 args["out"], args["lse"], args["ws"], args["ws_bytes"],
                                 args["stream"])


@pytest.mark.parametrize("wl,wr,kw,expect", [
    (-2, 0, {}, _lib.FA_ERR_PARAM_INVALID),
    (0, -5, {}, _lib.FA_ERR_PARAM_INVALID),
    (4, 4, dict(S_q=64, S_kv=128), _lib.FA_ERR_PARAM_INVALID),  # a window needs S_q == S_kv
    (4, 4, dict(q=None), _lib.FA_ERR_NULLPTR),
    (4, 4, dict(D=96), _lib.FA_ERR_UNSUPPORTED),
    (4, 4, dict(ws_bytes=16), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
])
def test_forward_window_rejects_before_any_cuda_call(lib, wl, wr, kw, expect):
    assert _fwd_window(lib, wl, wr, **kw) == expect


def test_forward_window_noop_shapes_return_ok(lib):
    assert _fwd_window(lib, 3, 2, B=0) == _lib.FA_OK
    # no window at all: S_q may differ from S_kv (as for fa_forward without a mask)
    assert _fwd_window(lib, -1, -1, B=0, S_q=5, S_kv=9) == _lib.FA_OK


def test_forward_noop_shapes_return_ok(lib):
    assert _fwd(lib, B=0) == _lib.FA_OK
    assert _fwd(lib, S_q=0, S_kv=5) == _lib.FA_OK


@pytest.mark.parametrize("kw,expect", [
    (dict(lens=None), _lib.FA_ERR_NULLPTR),
    (dict(v=None), _lib.FA_ERR_NULLPTR),
    (dict(Hq=8, Hkv=3), _lib.FA_ERR_PARAM_INVALID),
    (dict(D=32), _lib.FA_ERR_UNSUPPORTED),
    (dict(lens=[129, 1]), _lib.FA_ERR_PARAM_INVALID),
    (dict(splits=-2), _lib.FA_ERR_PARAM_INVALID),
    (dict(ws_bytes=1024), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
    (dict(layout=7), _lib.FA_ERR_PARAM_INVALID),
])
def test_decode_rejects_before_any_cuda_call(lib, kw, expect):
    assert _dec(lib, **kw) == expect


def test_decode_zero_batch_is_noop(lib):
    assert _dec(lib, B=0, lens=[]) == _lib.FA_OK


def test_head_dim_256_is_accepted(lib):
    # D = 256 for decode (the plan and the size query too) and for prefill
    assert _dec(lib, D=256, B=0, lens=[]) == _lib.FA_OK
    assert _dec(lib, D=192, B=0, lens=[]) == _lib.FA_ERR_UNSUPPORTED
    assert F.fa_decode_workspace_size(2, 4096, 16, 4, 256, 0) > 0
    rc, n, mx = _plan([4096, 100], 4096, 16, 4, D=256)
    assert rc >= 224 and n >= 1 and mx >= 1
    assert _fwd(lib, D=256, B=0) == _lib.FA_OK
    assert _fwd(lib, D=192, B=0) == _lib.FA_ERR_UNSUPPORTED


def test_prefill_workspace_counts_work_items_of_the_head_dim():
    # D = 256 items are 128 query rows (one Q tile), others 256: the schedule
    # part of the workspace holds twice as many items
    w128 = F.fa_forward_workspace_size(2, 4096, 4096, 16, 16, 128)
    w256 = F.fa_forward_workspace_size(2, 4096, 4096, 16, 16, 256)
    assert w256 - w128 == 4 * 2 * 16 * (4096 // 128 - 4096 // 256)


def _plan(lens, S, Hq, Hkv, sms=152, splits=0, D=128):
    return F.fa_decode_plan(lens, S, Hq, Hkv, D, sms, splits)


def _heads_per_cta(g, D):
    if D == 64 and g % 8 == 0:
        return 8
    return 4 if g % 4 == 0 else 2 if g % 2 == 0 else 1


def _units(lens, Hq, Hkv, D):
    g = Hq // Hkv
    return Hkv * (g // _heads_per_cta(g, D))


PC128 = 192        # rows a unit start costs at D = 128 when units outnumber SMs
PC128_HEADS = 384  # ... when they do not, and a CTA carries four or more query heads


def _piece_cost(lens, Hq, Hkv, D, sms=152, splits=0):
    """The extra cost of a unit start (scaled by 128 / D): PC128 rows when the
    non-empty units outnumber the SMs, PC128_HEADS when there are fewer (but
    more than one) and a CTA carries four or more query heads, else none."""
    units = _units(lens, Hq, Hkv, D) * sum(1 for L in lens if L)
    if splits or units <= 1:
        return 0
    if units > sms:
        return PC128 * 128 // D
    g = Hq // Hkv
    return PC128_HEADS * 128 // D if _heads_per_cta(g, D) >= 4 else 0


def _pieces(lens, Hq, Hkv, D, rc, pc=0):
    """Brute force: pieces per (batch, KV head, head group) unit when the
    units are laid end to end, row by row, each row costing 1 and the start
    of unit k adding pc * k, and the cost is cut every rc. Returns the
    pieces of every non-empty unit, the total rows and the total cost."""
    KH = _units(lens, Hq, Hkv, D)
    out, pos, k = [], 0, 0
    cost_end = 0
    for L in lens:
        for _ in range(KH):
            if L:
                c0 = pos + pc * k
                out.append(len(range(c0 // rc, (c0 + L - 1) // rc + 1)))
                cost_end = c0 + L
            pos += L
            k += 1
    return out, pos, cost_end


def test_plan_cuts_equal_shares(lib):
    import random
    rng = random.Random(5)
    for _ in range(60):
        B = rng.randint(1, 16)
        S = rng.randint(1, 20000)
        lens = [rng.randint(0, S) for _ in range(B)]
        Hkv = rng.choice([1, 2, 8, 32])
        Hq = Hkv * rng.choice([1, 2, 4, 8])
        D = rng.choice([64, 128])
        rc, n, mx = _plan(lens, S, Hq, Hkv, D=D)
        pc = _piece_cost(lens, Hq, Hkv, D)
        pieces, total, cost = _pieces(lens, Hq, Hkv, D, rc, pc)
        assert rc >= 224 and n == math.ceil(cost / rc) and n <= 152
        assert mx == (max(pieces) if pieces else 0)
        assert mx <= math.ceil(S / 224) + 1  # fits the size query's bound


def test_plan_one_share_per_sm():
    # GQA decode workload shape: 8 batches x 8 KV heads, lengths ~U[1024, 8192];
    # four heads per CTA: the shares are cut by cost
    lens = [1024, 8192, 4000, 6000, 3000, 7777, 2048, 5000]
    rc, n, mx = _plan(lens, 8192, 32, 8)
    cost = 8 * sum(lens) + PC128_HEADS * (8 * 8 - 1)
    assert n == 152 and rc * 152 >= cost > rc * 151
    assert mx == max(_pieces(lens, 32, 8, 128, rc, PC128_HEADS)[0])
    # one query head per KV head and fewer units than SMs: shares of rows
    rc, n, mx = _plan(lens, 8192, 8, 8)
    assert n == 152 and rc * 152 >= 8 * sum(lens) > rc * 151
    # one long sequence, 32 heads: every SM streams an equal share
    rc, n, mx = _plan([131072], 131072, 32, 32)
    assert n == 152 and mx == max(_pieces([131072], 32, 32, 128, rc)[0])
    assert mx <= math.ceil(131072 / rc) + 1


def test_plan_weights_unit_starts():
    # 64 sequences x 8 KV heads = 512 units > 152 SMs: the shares are cut by
    # cost, a row costs 1 and each unit start after the first PC128 rows more
    lens = [(37 * b) % 2000 + 1 for b in range(64)]
    rc, n, mx = _plan(lens, 2048, 32, 8)
    pieces, total, cost = _pieces(lens, 32, 8, 128, rc, PC128)
    assert cost == total + PC128 * (64 * 8 - 1)
    assert rc == math.ceil(cost / 152) and n == 152 and mx == max(pieces)
    # a share that holds unit starts holds fewer rows than one that does not:
    # count the rows of every share by walking the rows with their costs
    rows = [0] * n
    starts = [0] * n
    k = 0
    for L in lens:
        for _ in range(8):
            c0 = sum(rows) + PC128 * k
            for i in range(L):
                rows[(c0 + i) // rc] += 1
            starts[c0 // rc] += 1
            k += 1
    assert sum(rows) == total
    # every share but the last: its cost rc is its rows plus the piece costs
    # in it, one per unit start in it (give or take one straddling a boundary)
    for r, st in zip(rows[:-1], starts[:-1]):
        assert rc - PC128 * (st + 1) <= r <= rc - PC128 * max(st - 1, 0)
    assert max(starts) >= 3 and min(rows[:-1]) < max(rows[:-1]) - PC128
    # D = 64 (eight heads per CTA) charges twice as many rows per unit start
    rc64, n64, _ = _plan(lens, 2048, 64, 8, D=64)
    assert rc64 == math.ceil((8 * sum(lens) + 2 * PC128 * (64 * 8 - 1)) / 152) and n64 == 152
    # forced splits cut rows and charge nothing
    rc2, n2, _ = _plan(lens, 2048, 32, 8, splits=4)
    assert (rc2, n2) == (512, math.ceil(8 * sum(lens) / 512))


def test_plan_with_forced_splits():
    rc, n, mx = _plan([131072], 131072, 32, 32, splits=128)
    assert (rc, n, mx) == (1024, 32 * 128, 128)
    rc, n, mx = _plan([131072], 131072, 32, 32, splits=1024)
    assert (rc, n, mx) == (128, 32 * 1024, 1024)
    rc, n, mx = _plan([1000, 0], 1000, 4, 4, splits=3)
    assert (rc, n) == (384, math.ceil(4000 / 384))
    assert mx == max(_pieces([1000, 0], 4, 4, 128, 384)[0])


def test_plan_zero_lengths():
    rc, n, mx = _plan([0, 0, 0], 4096, 8, 8)
    assert n == 0 and mx == 0


def test_plan_rejects_bad_args(lib):
    with pytest.raises(_lib.FaError):
        _plan([5], 4, 8, 8)          # length above the cache
    with pytest.raises(_lib.FaError):
        _plan([5], 8, 8, 3)          # heads not a multiple
    with pytest.raises(_lib.FaError):
        _plan([5], 8, 8, 8, sms=0)
    with pytest.raises(_lib.FaError):
        _plan([5], 8, 8, 8, D=96)


def _dec_paged(lib, **kw):
    args = dict(q=P, k=P, v=P, kvl=2, bt=P, maxb=4, nblk=16, bs=64, key_mask=None, lens=[100, 7],
                B=2, Hq=8, Hkv=2, D=128, scale=0.1, splits=0, out=P, lse=None, ws=WS,
                ws_bytes=1 << 22, stream=None)
    args.update(kw)
    lens = args["lens"]
    if lens is not None:
        lens = (ctypes.c_int64 * max(len(lens), 1))(*lens)
    return lib.fa_decode_paged(args["q"], args["k"], args["v"], args["kvl"], args["bt"],
                               args["maxb"], args["nblk"], args["bs"], args["key_mask"], lens,
                               args["B"], args["Hq"], args["Hkv"], args["D"], args["scale"],
                               args["splits"], args["out"], args["lse"], args["ws"],
                               args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(bt=None), _lib.FA_ERR_NULLPTR),
    (dict(lens=None), _lib.FA_ERR_NULLPTR),
    (dict(kvl=0), _lib.FA_ERR_PARAM_INVALID),    # a contiguous layout is not a paged one
    (dict(kvl=7), _lib.FA_ERR_PARAM_INVALID),
    (dict(bs=8), _lib.FA_ERR_PARAM_INVALID),     # below 16
    (dict(bs=40), _lib.FA_ERR_PARAM_INVALID),    # not a multiple of 16
    (dict(bs=2048), _lib.FA_ERR_PARAM_INVALID),  # above 1024
    (dict(maxb=-1), _lib.FA_ERR_PARAM_INVALID),
    (dict(lens=[257, 1]), _lib.FA_ERR_PARAM_INVALID),  # past max_blocks * block_size
    (dict(D=96), _lib.FA_ERR_UNSUPPORTED),
    (dict(ws_bytes=16), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_paged_rejects_before_any_cuda_call(lib, kw, expect):
    assert _dec_paged(lib, **kw) == expect


def test_decode_paged_zero_batch_is_noop(lib):
    assert _dec_paged(lib, B=0, lens=[], bt=None) == _lib.FA_OK


def _fwd_paged(lib, **kw):
    args = dict(q=P, k=P, v=P, kvl=2, bt=P, maxb=4, nblk=16, bs=64, mask=0, key_mask=None,
                lens=None, B=2, S_q=256, S_kv=256, Hq=8, Hkv=2, D=128, scale=0.1, layout=0,
                out=P, lse=None, ws=WS, ws_bytes=1 << 22, stream=None)
    args.update(kw)
    lens = args["lens"]
    if lens is not None:
        lens = (ctypes.c_int64 * max(len(lens), 1))(*lens)
    return lib.fa_forward_paged(args["q"], args["k"], args["v"], args["kvl"], args["bt"],
                                args["maxb"], args["nblk"], args["bs"], args["mask"],
                                args["key_mask"], lens, args["B"], args["S_q"], args["S_kv"],
                                args["Hq"], args["Hkv"], args["D"], args["scale"], args["layout"],
                                args["out"], args["lse"], args["ws"], args["ws_bytes"],
                                args["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(bt=None), _lib.FA_ERR_NULLPTR),
    (dict(k=None), _lib.FA_ERR_NULLPTR),
    (dict(kvl=0), _lib.FA_ERR_PARAM_INVALID),     # a contiguous layout is not a paged one
    (dict(kvl=7), _lib.FA_ERR_PARAM_INVALID),
    (dict(layout=2), _lib.FA_ERR_PARAM_INVALID),  # q itself is not paged
    (dict(bs=8), _lib.FA_ERR_PARAM_INVALID),      # below 16
    (dict(bs=40), _lib.FA_ERR_PARAM_INVALID),     # not a multiple of 16
    (dict(bs=2048), _lib.FA_ERR_PARAM_INVALID),   # above 1024
    (dict(maxb=3), _lib.FA_ERR_PARAM_INVALID),    # 3 x 64 rows < S_kv = 256
    (dict(maxb=-1), _lib.FA_ERR_PARAM_INVALID),
    (dict(mask=3, S_q=128), _lib.FA_ERR_PARAM_INVALID),  # causal needs S_q == S_kv
    (dict(mask=4), _lib.FA_ERR_PARAM_INVALID),    # the window has its own entry points
    (dict(lens=[300, 1]), _lib.FA_ERR_PARAM_INVALID),  # past S_kv
    (dict(D=96), _lib.FA_ERR_UNSUPPORTED),
    (dict(ws_bytes=16), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
])
def test_forward_paged_rejects_before_any_cuda_call(lib, kw, expect):
    assert _fwd_paged(lib, **kw) == expect


def test_forward_paged_zero_batch_is_noop(lib):
    assert _fwd_paged(lib, B=0, bt=None) == _lib.FA_OK


def _fwd_varlen(lib, cq, ckv, **kw):
    args = dict(q=P, k=P, v=P, mask=0, Hq=4, Hkv=2, D=128, scale=0.1, out=P, lse=None, ws=WS,
                ws_bytes=1 << 22, stream=None)
    args.update(kw)
    B = len(cq) - 1
    aq = (ctypes.c_int64 * len(cq))(*cq) if cq is not None else None
    akv = (ctypes.c_int64 * len(ckv))(*ckv) if ckv is not None else None
    return lib.fa_forward_varlen(args["q"], args["k"], args["v"], aq, akv, args["mask"],
                                 args.get("B", B), args["Hq"], args["Hkv"], args["D"],
                                 args["scale"], args["out"], args["lse"], args["ws"],
                                 args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("cq,ckv,kw,expect", [
    ([1, 5], [0, 5], {}, _lib.FA_ERR_PARAM_INVALID),          # must start at 0
    ([0, 5, 3], [0, 5, 9], {}, _lib.FA_ERR_PARAM_INVALID),    # decreasing
    ([0, 5, 9], [0, 5, 8], dict(mask=3), _lib.FA_ERR_PARAM_INVALID),  # causal, unequal lengths
    ([0, 5], [0, 5], dict(mask=4), _lib.FA_ERR_PARAM_INVALID),
    ([0, 5], [0, 5], dict(q=None), _lib.FA_ERR_NULLPTR),
    ([0, 5], [0, 5], dict(D=96), _lib.FA_ERR_UNSUPPORTED),
    ([0, 5], [0, 5], dict(ws_bytes=16), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
])
def test_forward_varlen_rejects_before_any_cuda_call(lib, cq, ckv, kw, expect):
    assert _fwd_varlen(lib, cq, ckv, **kw) == expect


def test_forward_varlen_null_offsets(lib):
    assert lib.fa_forward_varlen(P, P, P, None, None, 0, 1, 4, 2, 128, 0.1, P, None, WS,
                                 1 << 22, None) == _lib.FA_ERR_NULLPTR


def _fwd_varlen_window(lib, cq, ckv, wl, wr, **kw):
    args = dict(q=P, Hq=4, Hkv=2, D=128, ws_bytes=1 << 22)
    args.update(kw)
    aq = (ctypes.c_int64 * len(cq))(*cq)
    akv = (ctypes.c_int64 * len(ckv))(*ckv)
    return lib.fa_forward_varlen_window(args["q"], P, P, aq, akv, wl, wr, len(cq) - 1, args["Hq"],
                                        args["Hkv"], args["D"], 0.1, P, None, WS,
                                        args["ws_bytes"], None)


@pytest.mark.parametrize("cq,ckv,wl,wr,kw,expect", [
    ([0, 5, 9], [0, 5, 8], 3, 0, {}, _lib.FA_ERR_PARAM_INVALID),   # a window, unequal lengths
    ([0, 5], [0, 5], -2, 0, {}, _lib.FA_ERR_PARAM_INVALID),         # width below -1
    ([0, 5], [0, 5], 0, -7, {}, _lib.FA_ERR_PARAM_INVALID),
    ([0, 5], [0, 5], 3, 0, dict(q=None), _lib.FA_ERR_NULLPTR),
    ([0, 5], [0, 5], 3, 0, dict(D=80), _lib.FA_ERR_UNSUPPORTED),
    ([0, 5], [0, 5], 3, 0, dict(ws_bytes=16), _lib.FA_ERR_WORKSPACE_TOO_SMALL),
])
def test_forward_varlen_window_rejects_before_any_cuda_call(lib, cq, ckv, wl, wr, kw, expect):
    assert _fwd_varlen_window(lib, cq, ckv, wl, wr, **kw) == expect


def test_forward_varlen_window_null_offsets(lib):
    assert lib.fa_forward_varlen_window(P, P, P, None, None, 3, 0, 1, 4, 2, 128, 0.1, P, None,
                                        WS, 1 << 22, None) == _lib.FA_ERR_NULLPTR


C_CONSUMER = r"""
#include <stdio.h>
#include "fa.h"
int main(void) {
  int64_t lens[2] = {100, 7}, rc = 0, n = 0, mx = 0;
  fa_status st = fa_decode_plan(2, 128, 8, 2, 128, lens, 152, 0, &rc, &n, &mx);
  printf("%d %lld %lld %lld %zu\n", (int)st, (long long)rc, (long long)n, (long long)mx,
         fa_decode_workspace_size(8, 8192, 32, 8, 128, 0));
  printf("%s\n", fa_status_string(FA_ERR_UNSUPPORTED));
  return st == FA_OK ? 0 : 1;
}
"""


def test_header_is_plain_c_and_the_library_links_from_c(lib, tmp_path):
    """include/fa.h compiles as strict C11 and a C program links the library
    and calls its host-side entry points (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_fa.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "use_fa"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.dirname(HEADER), str(src), "-L", libdir, "-lfa_gb300",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    st, rc, n, mx, ws = out[0].split()
    # 4 units (two sequences x two KV heads, four heads per CTA): cut by cost,
    # 214 rows + 3 unit starts x 384 = 1366 over shares of 224, one unit each
    assert (int(st), int(rc), int(n), int(mx)) == (0, 224, 7, 1)
    assert int(ws) == F.fa_decode_workspace_size(8, 8192, 32, 8, 128, 0)
    assert out[1] == lib.fa_status_string(_lib.FA_ERR_UNSUPPORTED).decode()


def test_python_binding_has_every_declared_function():
    """The binding carries the C ABI's names: every function fa.h declares
    has a wrapper of the same name, exported by the package."""
    import attention_forward_qk_gb300 as pkg
    names = set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", open(HEADER).read()))
    assert names and all(hasattr(F, n) for n in names), sorted(n for n in names if not hasattr(F, n))
    assert all(hasattr(pkg, n) for n in names), sorted(n for n in names if not hasattr(pkg, n))
    assert F.fa_forward_varlen_workspace_size(3, 100, 200, 8, 2, 128) == int(
        _lib.load().fa_forward_varlen_workspace_size(3, 100, 200, 8, 2, 128))


def _fwd_varlen_ex(lib, cq, ckv, uq, ukv, wl=-1, wr=0, ws_bytes=1 << 22, km=None):
    B = len(cq) - 1
    aq = (ctypes.c_int64 * len(cq))(*cq)
    akv = (ctypes.c_int64 * len(ckv))(*ckv)
    auq = (ctypes.c_int64 * B)(*uq) if uq is not None else None
    aukv = (ctypes.c_int64 * B)(*ukv) if ukv is not None else None
    return lib.fa_forward_varlen_ex(P, P, P, aq, akv, auq, aukv, km, wl, wr, B, 4, 2, 128, 0.1, P,
                                    None, WS, ws_bytes, None)


@pytest.mark.parametrize("cq,ckv,uq,ukv,wl,wr,expect", [
    ([0, 10, 30], [0, 10, 30], [5, -1], None, -1, 0, _lib.FA_ERR_PARAM_INVALID),
    ([0, 10, 30], [0, 10, 30], None, [-3, 20], -1, 0, _lib.FA_ERR_PARAM_INVALID),
    ([0, 10, 30], [0, 12, 30], [5, 5], [5, 5], -1, 0, _lib.FA_ERR_PARAM_INVALID),  # causal spans
    ([0, 10, 30], [0, 10, 30], [5, 5], [5, 5], -2, 0, _lib.FA_ERR_PARAM_INVALID),
    ([1, 10], [0, 10], None, None, -1, -1, _lib.FA_ERR_PARAM_INVALID),
])
def test_forward_varlen_ex_rejects_before_any_cuda_call(lib, cq, ckv, uq, ukv, wl, wr, expect):
    assert _fwd_varlen_ex(lib, cq, ckv, uq, ukv, wl, wr) == expect


def test_forward_varlen_ex_workspace_and_empty_batch(lib):
    assert _fwd_varlen_ex(lib, [0, 10], [0, 10], [3], [3], ws_bytes=16) == \
        _lib.FA_ERR_WORKSPACE_TOO_SMALL
    assert _fwd_varlen_ex(lib, [0], [0], [], []) == _lib.FA_OK  # B = 0: nothing to do


def test_debug_library_exports_every_declared_function():
    """The FA_DEBUG build (device-side index checks) carries the same C ABI."""
    dbg = _lib.load_debug()
    for n in header_functions():
        assert hasattr(dbg, n), n
    assert dbg.fa_abi_version() == 1
    assert b"FA_ERR_DEVICE_CHECK" in dbg.fa_status_string(_lib.FA_ERR_DEVICE_CHECK)


def test_decode_masked_rejects_an_unknown_mask_layout(lib):
    lens = (ctypes.c_int64 * 1)(10)
    st = lib.fa_decode_masked(P, P, P, P, 3, lens, 1, 16, 4, 4, 128, 0.1, 0, 0, P, None, WS,
                              1 << 22, None)
    assert st == _lib.FA_ERR_PARAM_INVALID
