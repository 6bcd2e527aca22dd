"""Python binding of the C ABI (``include/fa.h``), same names as the C calls.

Argument marshalling only: shapes are read from the tensors, outputs and the
workspace are allocated with torch when not supplied, and every computation
runs in the CUDA library on torch's current stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import FaError, check  # noqa: F401

LAYOUTS = {"BNSD": _lib.FA_LAYOUT_BNSD, "BSND": _lib.FA_LAYOUT_BSND, "BSH": _lib.FA_LAYOUT_BSND}
MASK_MODES = {None: _lib.FA_MASK_NONE, "none": _lib.FA_MASK_NONE, 0: _lib.FA_MASK_NONE,
              "causal": _lib.FA_MASK_CAUSAL, 3: _lib.FA_MASK_CAUSAL}


def _layout_id(layout) -> int:
    if isinstance(layout, int):
        return layout
    return LAYOUTS[layout.upper()]


def _dims(x: torch.Tensor, layout_id: int):
    """(B, N, S, D) of a 4-D tensor in the given layout."""
    if x.dim() != 4:
        raise ValueError("expected a 4-D tensor")
    if layout_id == _lib.FA_LAYOUT_BNSD:
        B, N, S, D = x.shape
    else:
        B, S, N, D = x.shape
    return B, N, S, D


def _check_tensor(x: torch.Tensor, name: str, dtype=torch.bfloat16):
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _lens_array(lens, B):
    if lens is None:
        return None, None
    if isinstance(lens, torch.Tensor):
        lens = lens.detach().cpu().tolist()
    lens = [int(x) for x in lens]
    if len(lens) != B:
        raise ValueError("actual_seq_lengths must have B entries")
    arr = (ctypes.c_int64 * max(B, 1))(*lens)
    return arr, lens


def fa_abi_version() -> int:
    return _lib.load().fa_abi_version()


def fa_status_string(status: int) -> str:
    return _lib.load().fa_status_string(status).decode()


def fa_forward_workspace_size(B, S_q, S_kv, num_heads, num_kv_heads, D) -> int:
    return int(_lib.load().fa_forward_workspace_size(B, S_q, S_kv, num_heads, num_kv_heads, D))


def fa_forward_varlen_workspace_size(B, max_seqlen_q, max_seqlen_kv, num_heads, num_kv_heads,
                                     D) -> int:
    return int(_lib.load().fa_forward_varlen_workspace_size(B, max_seqlen_q, max_seqlen_kv,
                                                            num_heads, num_kv_heads, D))


def fa_decode_workspace_size(B, S_kv_max, num_heads, num_kv_heads, D, num_splits=0) -> int:
    return int(_lib.load().fa_decode_workspace_size(B, S_kv_max, num_heads, num_kv_heads, D,
                                                    num_splits))


def fa_decode_plan(actual_seq_lengths, S_kv_max, num_heads, num_kv_heads, D, num_sms,
                   num_splits=0):
    """(chunk_rows, num_chunks, max_chunks) of the decode split plan (host only)."""
    B = len(actual_seq_lengths)
    arr, _ = _lens_array(actual_seq_lengths, B)
    c, n, m = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    st = _lib.load().fa_decode_plan(B, S_kv_max, num_heads, num_kv_heads, D, arr, num_sms,
                                    num_splits, ctypes.byref(c), ctypes.byref(n), ctypes.byref(m))
    check(st, "fa_decode_plan")
    return c.value, n.value, m.value


def _forward_prep(q, k, v, layout, num_heads, num_kv_heads, out, lse, return_lse, key_mask,
                  workspace, actual_seq_lengths):
    lid = _layout_id(layout)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    B, Hq, S_q, D = _dims(q, lid)
    Bk, Hkv, S_kv, Dk = _dims(k, lid)
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q, k, v shapes disagree")
    if num_heads is not None and num_heads != Hq:
        raise ValueError("num_heads does not match q")
    if num_kv_heads not in (None, 0) and num_kv_heads != Hkv:
        raise ValueError("num_kv_heads does not match k")
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32)
    if key_mask is not None:
        _check_tensor(key_mask, "key_mask", torch.uint8)
    need = fa_forward_workspace_size(B, S_q, S_kv, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lens_arr, _ = _lens_array(actual_seq_lengths, B)
    return lid, (B, S_q, S_kv, Hq, Hkv, D), out, lse, workspace, lens_arr


def fa_forward(q, k, v, *, mask_mode=None, key_mask=None, actual_seq_lengths=None, scale=1.0,
               layout="BNSD", num_heads=None, num_kv_heads=None, out=None, lse=None,
               return_lse=True, workspace=None, stream=None):
    """Prefill attention. Returns (out, lse); lse is None unless requested."""
    lid, (B, S_q, S_kv, Hq, Hkv, D), out, lse, workspace, lens_arr = _forward_prep(
        q, k, v, layout, num_heads, num_kv_heads, out, lse, return_lse, key_mask, workspace,
        actual_seq_lengths)
    st = _lib.load().fa_forward(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), MASK_MODES.get(mask_mode, mask_mode),
        key_mask.data_ptr() if key_mask is not None else None, lens_arr, B, S_q, S_kv, Hq, Hkv,
        D, float(scale), lid, out.data_ptr(), lse.data_ptr() if lse is not None else None,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    check(st, "fa_forward")
    return out, lse


def fa_forward_paged(q, k_cache, v_cache, block_table, block_size, S_kv, *, kv_layout="PA_BBND",
                     mask_mode=None, key_mask=None, actual_seq_lengths=None, scale=1.0,
                     layout="BNSD", num_heads=None, num_kv_heads=None, out=None, lse=None,
                     return_lse=True, workspace=None, stream=None):
    """Prefill attention with K and V in a paged cache: k_cache/v_cache
    [num_blocks, block_size, KV_N, D] (PA_BBND) or [num_blocks, KV_N,
    block_size, D] (PA_BNBD); block_table int32 [B, max_blocks_per_seq] on the
    device; S_kv the keys of each sequence. q and out in `layout`. Returns
    (out, lse)."""
    kvl = {"PA_BBND": _lib.FA_LAYOUT_PA_BBND, "PA_BNBD": _lib.FA_LAYOUT_PA_BNBD}.get(kv_layout)
    if kvl is None:
        raise ValueError("kv_layout must be PA_BBND or PA_BNBD")
    lid = _layout_id(layout)
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_tensor(t, n)
    if block_table.dtype != torch.int32 or not block_table.is_contiguous() or block_table.dim() != 2:
        raise ValueError("block_table must be a contiguous int32 [B, max_blocks_per_seq] tensor")
    B, Hq, S_q, D = _dims(q, lid)
    if kvl == _lib.FA_LAYOUT_PA_BBND:
        nblk, bs, Hkv, Dk = k_cache.shape
    else:
        nblk, Hkv, bs, Dk = k_cache.shape
    if bs != block_size or Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache, v_cache, block_size or D disagree")
    if block_table.shape[0] != B:
        raise ValueError("block_table must have B rows")
    if num_heads is not None and num_heads != Hq:
        raise ValueError("num_heads does not match q")
    if num_kv_heads not in (None, 0) and num_kv_heads != Hkv:
        raise ValueError("num_kv_heads does not match k_cache")
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32)
    if key_mask is not None:
        _check_tensor(key_mask, "key_mask", torch.uint8)
    need = fa_forward_workspace_size(B, S_q, S_kv, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lens_arr, _ = _lens_array(actual_seq_lengths, B)
    st = _lib.load().fa_forward_paged(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), kvl, block_table.data_ptr(),
        block_table.shape[1], nblk, block_size, MASK_MODES.get(mask_mode, mask_mode),
        key_mask.data_ptr() if key_mask is not None else None, lens_arr, B, S_q, int(S_kv), Hq,
        Hkv, D, float(scale), lid, out.data_ptr(), lse.data_ptr() if lse is not None else None,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    check(st, "fa_forward_paged")
    return out, lse


def fa_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, *, mask_mode=None, scale=1.0,
                      num_heads=None, num_kv_heads=None, out=None, lse=None, return_lse=True,
                      workspace=None, stream=None):
    """Prefill attention over packed variable-length sequences (TND): q, out
    [T_q, Hq, D]; k, v [T_kv, Hkv, D]; cu_seqlens_* host sequences of B + 1
    offsets. Returns (out, lse) with lse [T_q, Hq]."""
    return _varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, None, mask_mode, scale, num_heads,
                   out, lse, return_lse, workspace, stream)


def fa_forward_varlen_window(q, k, v, cu_seqlens_q, cu_seqlens_kv, win_left, win_right, *,
                             scale=1.0, num_heads=None, num_kv_heads=None, out=None, lse=None,
                             return_lse=True, workspace=None, stream=None):
    """fa_forward_varlen with a sliding window inside every sequence: row i
    keeps key j iff (win_left < 0 or j >= i - win_left) and (win_right < 0 or
    j <= i + win_right), both counted from the sequence's first token."""
    return _varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, (int(win_left), int(win_right)), None,
                   scale, num_heads, out, lse, return_lse, workspace, stream)


def fa_forward_varlen_ex(q, k, v, cu_seqlens_q, cu_seqlens_kv, *, seqused_q=None,
                         seqused_kv=None, key_mask=None, win_left=-1, win_right=-1, scale=1.0,
                         num_heads=None, num_kv_heads=None, out=None, lse=None, return_lse=True,
                         workspace=None, stream=None):
    """Packed sequences with the used lengths (seqused_q / seqused_kv, host
    sequences of B entries: the shorter of the span and the used length
    holds; truncated query rows read out 0, lse +inf), a per-packed-key mask
    (device uint8 [T_kv], nonzero = excluded) and a window ((-1, 0) causal)."""
    return _varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, (int(win_left), int(win_right)), None,
                   scale, num_heads, out, lse, return_lse, workspace, stream,
                   ex=(seqused_q, seqused_kv, key_mask))


def _varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, window, mask_mode, scale, num_heads, out, lse,
            return_lse, workspace, stream, ex=None):
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    if q.dim() != 3 or k.dim() != 3 or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q, k, v must be [T, H, D] with k and v alike")
    cq = [int(x) for x in cu_seqlens_q]
    ckv = [int(x) for x in cu_seqlens_kv]
    if len(cq) != len(ckv) or len(cq) < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_kv need B + 1 entries each")
    B = len(cq) - 1
    T_q, Hq, D = q.shape
    T_kv, Hkv, Dk = k.shape
    if Dk != D or cq[-1] != T_q or ckv[-1] != T_kv:
        raise ValueError("tensor rows disagree with the offsets")
    if num_heads is not None and num_heads != Hq:
        raise ValueError("num_heads does not match q")
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out")
    if lse is None and return_lse:
        lse = torch.empty((T_q, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32)
    max_q = max([b - a for a, b in zip(cq[:-1], cq[1:])] + [0])
    max_kv = max([b - a for a, b in zip(ckv[:-1], ckv[1:])] + [0])
    need = fa_forward_varlen_workspace_size(B, max_q, max_kv, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    aq = (ctypes.c_int64 * (B + 1))(*cq)
    akv = (ctypes.c_int64 * (B + 1))(*ckv)
    tail = (B, Hq, Hkv, D, float(scale), out.data_ptr(),
            lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if ex is not None:
        used_q, used_kv, km = ex
        uq = (ctypes.c_int64 * B)(*[int(x) for x in used_q]) if used_q is not None else None
        ukv = (ctypes.c_int64 * B)(*[int(x) for x in used_kv]) if used_kv is not None else None
        if (used_q is not None and len(used_q) != B) or (used_kv is not None and len(used_kv) != B):
            raise ValueError("seqused_q / seqused_kv need B entries")
        if km is not None:
            _check_tensor(km, "key_mask", torch.uint8)
            if km.numel() != T_kv:
                raise ValueError("key_mask needs one flag per packed key row")
        st = _lib.load().fa_forward_varlen_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), aq, akv,
                                              uq, ukv, km.data_ptr() if km is not None else None,
                                              window[0], window[1], *tail)
        check(st, "fa_forward_varlen_ex")
    elif window is None:
        st = _lib.load().fa_forward_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), aq, akv,
                                           MASK_MODES.get(mask_mode, mask_mode), *tail)
        check(st, "fa_forward_varlen")
    else:
        st = _lib.load().fa_forward_varlen_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), aq,
                                                  akv, window[0], window[1], *tail)
        check(st, "fa_forward_varlen_window")
    return out, lse


def fa_forward_window(q, k, v, win_left, win_right, *, key_mask=None, actual_seq_lengths=None,
                      scale=1.0, layout="BNSD", num_heads=None, num_kv_heads=None, out=None,
                      lse=None, return_lse=True, workspace=None, stream=None):
    """Prefill attention with a sliding window: query i sees keys i - win_left
    .. i + win_right (-1 = no limit on that side). Returns (out, lse)."""
    lid, (B, S_q, S_kv, Hq, Hkv, D), out, lse, workspace, lens_arr = _forward_prep(
        q, k, v, layout, num_heads, num_kv_heads, out, lse, return_lse, key_mask, workspace,
        actual_seq_lengths)
    st = _lib.load().fa_forward_window(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), int(win_left), int(win_right),
        key_mask.data_ptr() if key_mask is not None else None, lens_arr, B, S_q, S_kv, Hq, Hkv,
        D, float(scale), lid, out.data_ptr(), lse.data_ptr() if lse is not None else None,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    check(st, "fa_forward_window")
    return out, lse


def fa_decode(q, k, v, actual_seq_lengths, *, key_mask=None, scale=1.0, layout="BNSD",
              num_splits=0, num_heads=None, num_kv_heads=None, out=None, lse=None,
              return_lse=True, workspace=None, stream=None):
    """Decode (S_q = 1) attention with Split-KV. Returns (out, lse)."""
    lid = _layout_id(layout)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    B, Hq, S_q, D = _dims(q, lid)
    if S_q != 1:
        raise ValueError("decode takes one query row per batch (S_q = 1)")
    Bk, Hkv, S_kv, Dk = _dims(k, lid)
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q, k, v shapes disagree")
    if num_heads is not None and num_heads != Hq:
        raise ValueError("num_heads does not match q")
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32)
    if key_mask is not None:
        _check_tensor(key_mask, "key_mask", torch.uint8)
    need = fa_decode_workspace_size(B, S_kv, Hq, Hkv, D, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lens_arr, _ = _lens_array(actual_seq_lengths, B)
    if lens_arr is None:
        raise ValueError("actual_seq_lengths is required for decode")
    st = _lib.load().fa_decode(
        q.data_ptr(), k.data_ptr(), v.data_ptr(),
        key_mask.data_ptr() if key_mask is not None else None, lens_arr, B, S_kv, Hq, Hkv, D,
        float(scale), lid, int(num_splits), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    check(st, "fa_decode")
    return out, lse


KEY_MASK_LAYOUTS = {"B11S": 0, "BN1S": 1, "1N1S": 2}


def fa_decode_masked(q, k, v, actual_seq_lengths, key_mask, key_mask_layout, *, scale=1.0,
                     layout="BNSD", num_splits=0, out=None, lse=None, return_lse=True,
                     workspace=None, stream=None):
    """fa_decode with the key mask in a given layout: "B11S" [B, S_kv] (shared
    by the heads), "BN1S" [B, Hq, S_kv] or "1N1S" [Hq, S_kv] (one row per
    query head). Returns (out, lse)."""
    lid = _layout_id(layout)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    _check_tensor(key_mask, "key_mask", torch.uint8)
    B, Hq, S_q, D = _dims(q, lid)
    if S_q != 1:
        raise ValueError("decode takes one query row per batch (S_q = 1)")
    _, Hkv, S_kv, _ = _dims(k, lid)
    ml = KEY_MASK_LAYOUTS[key_mask_layout] if isinstance(key_mask_layout, str) else key_mask_layout
    want = {0: B * S_kv, 1: B * Hq * S_kv, 2: Hq * S_kv}.get(ml)
    if want is not None and key_mask.numel() != want:
        raise ValueError("key_mask size does not match its layout")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(fa_decode_workspace_size(B, S_kv, Hq, Hkv, D, num_splits),
                                dtype=torch.uint8, device=q.device)
    lens_arr, _ = _lens_array(actual_seq_lengths, B)
    st = _lib.load().fa_decode_masked(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), key_mask.data_ptr(), int(ml), lens_arr, B, S_kv,
        Hq, Hkv, D, float(scale), lid, int(num_splits), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    check(st, "fa_decode_masked")
    return out, lse


def fa_decode_paged(q, k_cache, v_cache, block_table, block_size, actual_seq_lengths, *,
                    kv_layout="PA_BBND", key_mask=None, scale=1.0, num_splits=0, num_heads=None,
                    num_kv_heads=None, out=None, lse=None, return_lse=True, workspace=None,
                    stream=None):
    """Decode (S_q = 1) attention against a paged K/V cache. k_cache/v_cache:
    [num_blocks, block_size, KV_N, D] (PA_BBND) or [num_blocks, KV_N,
    block_size, D] (PA_BNBD); block_table: int32 [B, max_blocks_per_seq] on the
    device. Returns (out, lse)."""
    kvl = {"PA_BBND": _lib.FA_LAYOUT_PA_BBND, "PA_BNBD": _lib.FA_LAYOUT_PA_BNBD}.get(kv_layout)
    if kvl is None:
        raise ValueError("kv_layout must be PA_BBND or PA_BNBD")
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_tensor(t, n)
    if block_table.dtype != torch.int32 or not block_table.is_contiguous() or block_table.dim() != 2:
        raise ValueError("block_table must be a contiguous int32 [B, max_blocks_per_seq] tensor")
    B, Hq, S_q, D = _dims(q, 0)
    if S_q != 1:
        raise ValueError("decode takes one query row per batch (S_q = 1)")
    if kvl == _lib.FA_LAYOUT_PA_BBND:
        nblk, bs, Hkv, Dk = k_cache.shape
    else:
        nblk, Hkv, bs, Dk = k_cache.shape
    if bs != block_size or Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache, v_cache, block_size or D disagree")
    if block_table.shape[0] != B:
        raise ValueError("block_table must have B rows")
    if num_heads is not None and num_heads != Hq:
        raise ValueError("num_heads does not match q")
    max_blocks = block_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _check_tensor(out, "out")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor(lse, "lse", torch.float32)
    if key_mask is not None:
        _check_tensor(key_mask, "key_mask", torch.uint8)
    need = fa_decode_workspace_size(B, max_blocks * block_size, Hq, Hkv, D, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lens_arr, _ = _lens_array(actual_seq_lengths, B)
    if lens_arr is None:
        raise ValueError("actual_seq_lengths is required for decode")
    st = _lib.load().fa_decode_paged(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), kvl, block_table.data_ptr(),
        max_blocks, nblk, block_size, key_mask.data_ptr() if key_mask is not None else None,
        lens_arr, B, Hq, Hkv, D, float(scale), int(num_splits), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    check(st, "fa_decode_paged")
    return out, lse


def fa_decode_noalloc(q, k, v, actual_seq_lengths, *, key_mask=None, scale=1.0, layout="BNSD",
                      num_splits=0, out=None, lse=None, return_lse=True, stream=None):
    """fa_decode on the library's own device scratch (no workspace argument):
    for callers that cannot allocate device memory. Returns (out, lse)."""
    lid = _layout_id(layout)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    B, Hq, S_q, D = _dims(q, lid)
    _, Hkv, S_kv, _ = _dims(k, lid)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    lens_arr, _ = _lens_array(actual_seq_lengths, B)
    st = _lib.load().fa_decode_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(),
        key_mask.data_ptr() if key_mask is not None else None, lens_arr, B, S_kv, Hq, Hkv, D,
        float(scale), lid, int(num_splits), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, _stream_ptr(stream))
    check(st, "fa_decode_noalloc")
    return out, lse


def fa_decode_noalloc_status(stream=None) -> int:
    """Synchronise the stream and read/clear the status word of the scratch
    array fa_decode_noalloc uses on the current device."""
    return int(_lib.load().fa_decode_noalloc_status(_stream_ptr(stream)))


def fa_workspace_status(workspace, stream=None) -> int:
    """Synchronise the stream and read/clear the workspace's device status word."""
    return int(_lib.load().fa_workspace_status(workspace.data_ptr(), _stream_ptr(stream)))


def fa_selftest_wait_timeout(workspace, timeout_ns: int, stream=None) -> int:
    return int(_lib.load().fa_selftest_wait_timeout(workspace.data_ptr(), int(timeout_ns),
                                                    _stream_ptr(stream)))


def fa_set_wait_timeout_ns(timeout_ns: int) -> None:
    """Bounded-wait limit of the kernels of later calls from this thread (0 =
    the default, 2 s). A diagnostic for failure-detection tests."""
    check(int(_lib.load().fa_set_wait_timeout_ns(int(timeout_ns))), "fa_set_wait_timeout_ns")


def fa_set_main_kernel_events(before, after) -> None:
    """Record torch.cuda.Event `before`/`after` around the main kernel of every
    later call from this thread (None, None turns it off). Each event must
    have been recorded once by torch so that its handle exists."""
    if before is None or after is None:
        _lib.load().fa_set_main_kernel_events(None, None)
        return
    _lib.load().fa_set_main_kernel_events(ctypes.c_void_p(before.cuda_event),
                                          ctypes.c_void_p(after.cuda_event))


def fa_kernel_launch_count() -> int:
    return int(_lib.load().fa_kernel_launch_count())
