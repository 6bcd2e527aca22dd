"""Plain, slow, fp64 CPU statement of what the attention forward computes.

TEST INFRASTRUCTURE: used only by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; the product path never touches it.

Sources (web pages on the subject, cited by title and section):
  [FA]  "FlashAttn" operator README + developer guide (ops-transformer,
        attention/flash_attn): functional description (formula), developer
        guide §1.1 (MHA/GQA), §1.4 (seqused), §1.5 (mask), §1.6 (LSE),
        §1.7 (row invalid), §10 (FD block merge formula).
  [IFA] "aclnnIncreFlashAttention usage guide and implementation analysis"
        (zskr.cn): §1.2 (formula), §四 (parameters: attenMask, actualSeqLengths,
        numKeyValueHeads), §8.1 (mask select), §8.3 (FlashDecode combine).
  [FD]  "FlashDecoding" Ascend C tutorial (CSDN): §二 (merge formula),
        §3.2 (stage 1), §3.3 (stage 2).

Definition (the method is exact up to rounding, so the oracle is the
definition itself, [FA] functional description; [IFA] §1.2):

    s_ij  = scale * sum_d q[b,h,i,d] * k[b,h//g,j,d]
    valid(i,j) = j < L_b  and  not key_mask[b,j]  and  not (causal and j > i)
                 and  (win_left < 0 or j >= i - win_left)
                 and  (win_right < 0 or j <= i + win_right)
    out_i = sum_{valid j} exp(s_ij - m_i) v_j / l_i,   m_i = max_{valid j} s_ij,
    l_i   = sum_{valid j} exp(s_ij - m_i),             lse_i = m_i + ln l_i
    a row with no valid key: out_i = 0, lse_i = +inf   ([FA] §1.7)

Readings taken where the pages are silent or ambiguous:
  * mask value 1/True means "excluded" ([IFA] §8.1: positions that are true
    in the mask are pushed to a very negative value; [FA] §1.7 "mask all 1"
    gives an invalid row);
  * the explicit mask is one flag per key, [B, S_kv], shared by every head
    and query row (the decode mask of [IFA] §四 has the (B,1,1,S) form);
  * "a very negative value" is read as exact exclusion (-inf);
  * causal means top-left aligned, j <= i ([FA] §1.5 "lower triangular");
  * the window of [FA] §1.5 (mask_mode 4, a band of win_left tokens before
    and win_right tokens after each query) is read as i - win_left <= j <=
    i + win_right, top-left aligned like causal, with -1 meaning "no limit
    on that side" (the value the page gives the two fields when no window
    applies); causal is the window (-1, 0);
  * GQA: query head h reads KV head h // g, g = Hq / Hkv ([FA] §1.1: a group
    of g adjacent query heads shares one KV head);
  * keys at or past actualSeqLengths[b] do not exist ([IFA] §1.1: inputs are
    padded to a fixed length; [FA] §1.4 seqused truncates padding), so their
    contents, NaN included, cannot influence the result; a length of 0 makes
    every row of that batch invalid.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attention",
    "attention_bruteforce",
    "decode",
    "valid_key_matrix",
    "split_partials",
    "merge_max_sum",
    "merge_sequential",
    "merge_lse",
]


def _as_f64(x) -> np.ndarray:
    """Exact widening of a torch tensor / array (bf16 included) to float64."""
    if hasattr(x, "detach"):  # torch tensor; bf16/fp16/fp32 -> fp64 is exact
        return x.detach().cpu().to(dtype=_torch_f64(x)).numpy()
    return np.asarray(x, dtype=np.float64)


def _torch_f64(x):
    import torch  # only reached for torch inputs
    return torch.float64


def _as_np(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy()
    return np.asarray(x)


def _to_bnsd(x: np.ndarray, layout: str) -> np.ndarray:
    if layout == "BNSD":
        return x
    if layout == "BSND":
        return np.transpose(x, (0, 2, 1, 3))
    raise ValueError(f"unknown layout {layout!r}")


def _from_bnsd(x: np.ndarray, layout: str) -> np.ndarray:
    return _to_bnsd(x, layout)  # the permutation is its own inverse


def valid_key_matrix(rows, S_kv: int, L: int, key_mask_row, causal: bool,
                     window=None) -> np.ndarray:
    """valid(i, j) for one batch: boolean [len(rows), S_kv] for query rows ``rows``.

    j < L ([IFA] §四 actualSeqLengths), key_mask_row[j] == 0 ([IFA] §8.1,
    1 = masked), j <= i when causal ([FA] §1.5, lower triangular), and
    i - win_left <= j <= i + win_right for window = (win_left, win_right)
    ([FA] §1.5 mask_mode 4; -1 = no limit on that side).
    """
    rows = np.asarray(rows)
    j = np.arange(S_kv)
    ok = np.broadcast_to(j < L, (len(rows), S_kv)).copy()
    if key_mask_row is not None:
        ok &= (np.asarray(key_mask_row) == 0)[None, :]
    if causal:
        ok &= j[None, :] <= rows[:, None]
    if window is not None:
        wl, wr = window
        if wl >= 0:
            ok &= j[None, :] >= rows[:, None] - wl
        if wr >= 0:
            ok &= j[None, :] <= rows[:, None] + wr
    return ok


def attention(q, k, v, *, scale: float = 1.0, layout: str = "BNSD", causal: bool = False,
              key_mask=None, actual_seq_lengths=None, rows=None, window=None):
    """out (fp64, same layout as q) and lse (fp64, [B, Hq, S_q]).

    q: [B,Hq,S_q,D] (BNSD) or [B,S_q,Hq,D] (BSND); k, v likewise with Hkv heads.
    key_mask: optional [B, S_kv], nonzero = masked, or one mask per query head
    ([IFA] §四 attenMask shapes (B, N, 1, S) and (1, N, 1, S)): [B, Hq, S_kv] or
    [1, Hq, S_kv] (the singleton batch is shared by every batch). actual_seq_lengths:
    optional per-batch valid KV length (default S_kv). rows: optional list of
    query indices; then only those rows are evaluated and the S_q axis of the
    results has len(rows) entries, in that order. window: optional
    (win_left, win_right), see ``valid_key_matrix``.
    """
    qn = _to_bnsd(_as_f64(q), layout)
    kn = _to_bnsd(_as_f64(k), layout)
    vn = _to_bnsd(_as_f64(v), layout)
    km = _as_np(key_mask)
    B, Hq, S_q, D = qn.shape
    _, Hkv, S_kv, _ = kn.shape
    if Hq % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    g = Hq // Hkv
    rows = np.arange(S_q) if rows is None else np.asarray(rows, dtype=np.int64)
    qn = qn[:, :, rows, :]
    R = len(rows)
    lens = [S_kv] * B if actual_seq_lengths is None else [int(x) for x in actual_seq_lengths]
    out = np.zeros((B, Hq, R, D))
    lse = np.full((B, Hq, R), np.inf)
    per_head = km is not None and km.ndim == 3
    for b in range(B):
        L = max(0, min(lens[b], S_kv))
        for h in range(Hq):
            kvh = h // g
            if per_head:
                mrow = km[b if km.shape[0] > 1 else 0, h]
            else:
                mrow = None if km is None else km[b]
            ok = valid_key_matrix(rows, S_kv, L, mrow, causal, window)
            # keys that no row of this head can see (past L or masked) are
            # dropped outright, so whatever they hold (NaN included) never
            # enters a product
            cols = np.nonzero(ok.any(axis=0))[0]
            okc = ok[:, cols]
            has_key = okc.any(axis=1)
            kk = kn[b, kvh][cols]
            vv = vn[b, kvh][cols]
            s = scale * (qn[b, h] @ kk.T)
            s = np.where(okc, s, -np.inf)
            m = np.max(s, axis=1, initial=-np.inf)
            m_safe = np.where(has_key, m, 0.0)
            p = np.where(okc, np.exp(s - m_safe[:, None]), 0.0)
            l = p.sum(axis=1)
            l_safe = np.where(has_key, l, 1.0)
            o = (p @ vv) / l_safe[:, None]
            out[b, h] = np.where(has_key[:, None], o, 0.0)
            lse[b, h] = np.where(has_key, m_safe + np.log(l_safe), np.inf)
    return _from_bnsd(out, layout), lse


def decode(q, k, v, actual_seq_lengths, *, scale: float = 1.0, layout: str = "BNSD",
           key_mask=None):
    """Incremental attention ([IFA] §1.1): S_q = 1 against a padded cache."""
    return attention(q, k, v, scale=scale, layout=layout, causal=False,
                     key_mask=key_mask, actual_seq_lengths=actual_seq_lengths)


def attention_bruteforce(q, k, v, *, scale: float = 1.0, layout: str = "BNSD",
                         causal: bool = False, key_mask=None, actual_seq_lengths=None,
                         window=None):
    """The same definition as scalar Python loops (tiny shapes only).

    Independent of ``attention``: every score, max, exponential and sum is a
    Python float operation over an explicit list of valid keys.
    """
    qn = _to_bnsd(_as_f64(q), layout)
    kn = _to_bnsd(_as_f64(k), layout)
    vn = _to_bnsd(_as_f64(v), layout)
    km = _as_np(key_mask)
    B, Hq, S_q, D = qn.shape
    _, Hkv, S_kv, _ = kn.shape
    g = Hq // Hkv
    out = np.zeros((B, Hq, S_q, D))
    lse = np.full((B, Hq, S_q), np.inf)
    for b in range(B):
        L = S_kv if actual_seq_lengths is None else int(actual_seq_lengths[b])
        for h in range(Hq):
            kvh = h // g
            for i in range(S_q):
                keys = []
                for j in range(min(L, S_kv)):
                    if km is not None and km.ndim == 3 and km[b if km.shape[0] > 1 else 0, h, j]:
                        continue  # one mask per query head
                    if km is not None and km.ndim == 2 and km[b, j]:
                        continue
                    if causal and j > i:
                        continue
                    if window is not None:
                        if window[0] >= 0 and j < i - window[0]:
                            continue
                        if window[1] >= 0 and j > i + window[1]:
                            continue
                    keys.append(j)
                if not keys:
                    continue  # invalid row: out 0, lse +inf
                s = {j: scale * math.fsum(float(qn[b, h, i, d]) * float(kn[b, kvh, j, d])
                                          for d in range(D)) for j in keys}
                m = max(s.values())
                w = {j: math.exp(s[j] - m) for j in keys}
                l = math.fsum(w.values())
                for d in range(D):
                    out[b, h, i, d] = math.fsum(w[j] * float(vn[b, kvh, j, d]) for j in keys) / l
                lse[b, h, i] = m + math.log(l)
    return _from_bnsd(out, layout), lse


# ---------------------------------------------------------------------------
# Split-KV ("FlashDecode") pieces, written in the pages' own notation.
# ---------------------------------------------------------------------------

def split_partials(s: np.ndarray, vv: np.ndarray, bounds):
    """Per-chunk statistics of one query row ([FD] §3.2 stage 1; [FA] §10).

    s: fp64 scores [n] (already scaled, only valid keys), vv: [n, D].
    bounds: chunk edges 0 = e_0 < e_1 < ... < e_K = n.
    Returns lists m_i, l_i = sum exp(s - m_i), o_i = sum exp(s - m_i) v
    (unnormalised) and lse_i = m_i + ln l_i, one entry per chunk.
    """
    ms, ls, os_, lses = [], [], [], []
    for a, e in zip(bounds[:-1], bounds[1:]):
        si = s[a:e]
        m = float(np.max(si))
        w = np.exp(si - m)
        ms.append(m)
        ls.append(float(w.sum()))
        os_.append(w @ vv[a:e])
        lses.append(m + math.log(float(w.sum())))
    return ms, ls, os_, lses


def merge_max_sum(ms, ls, os_):
    """[FA] §10: m = max_i m_i, l = sum_i l_i e^{m_i - m},
    o = sum_i o_i e^{m_i - m} / l. Returns (o, lse)."""
    m = max(ms)
    f = [math.exp(mi - m) for mi in ms]
    l = sum(li * fi for li, fi in zip(ls, f))
    o = sum(oi * fi for oi, fi in zip(os_, f)) / l
    return o, m + math.log(l)


def merge_sequential(ms, ls, os_):
    """[FD] §3.3 stage 2: fold the chunks one at a time into a running
    (m, l, o) with factors e^{m_old - m_new} and e^{m_i - m_new}; divide at the end."""
    gm, gl, go = -math.inf, 0.0, 0.0
    for mi, li, oi in zip(ms, ls, os_):
        nm = max(gm, mi)
        fg = math.exp(gm - nm) if gm != -math.inf else 0.0
        fi = math.exp(mi - nm)
        gl = gl * fg + li * fi
        go = go * fg + oi * fi
        gm = nm
    return go / gl, gm + math.log(gl)


def merge_lse(lses, onorms):
    """[IFA] §8.3 combine: scale_i = exp(lse_i) / sum_j exp(lse_j),
    res = sum_i onorm_i * scale_i, where onorm_i = o_i / l_i is the chunk's
    normalised output. Evaluated with the largest lse factored out (the
    weights are unchanged; exp(lse) itself would overflow). Returns (res, lse)."""
    M = max(lses)
    w = [math.exp(x - M) for x in lses]
    W = sum(w)
    res = sum(oi * (wi / W) for oi, wi in zip(onorms, w))
    return res, M + math.log(W)


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, *, scale: float = 1.0,
                     causal: bool = False, window=None, seqused_q=None, seqused_kv=None,
                     key_mask=None):
    """Packed variable-length sequences ([FA] §1.3 TND layout, §1.4
    cu_seqlens): q [T_q, Hq, D], k/v [T_kv, Hkv, D]; sequence b is q rows
    cu_q[b]..cu_q[b+1]-1 against k/v rows cu_kv[b]..cu_kv[b+1]-1, each an
    independent attention (causal, or the sliding window of [FA] §1.5 given
    as (win_left, win_right), top-left aligned within the sequence).

    seqused_q / seqused_kv ([FA] §1.4, one per sequence) truncate a
    sequence's padding: when given together with cu_seqlens the shorter of
    the two lengths holds. Keys past the used kv length do not exist (as keys
    past actualSeqLengths, whatever they hold); query rows past the used q
    length are truncated rows with no valid key, so they read out 0 and lse
    +inf ([FA] §1.7 names seqused truncation among the causes of an invalid
    row). key_mask: one flag per packed key row, [T_kv], nonzero = excluded
    (the per-key mask of the padded layouts laid out as the keys are).
    Returns out [T_q, Hq, D] and lse [T_q, Hq] (the TND lse shape of [FA] §1.6).
    """
    qn, kn, vn = _as_f64(q), _as_f64(k), _as_f64(v)
    km = _as_np(key_mask)
    T_q, Hq, D = qn.shape
    out = np.zeros((T_q, Hq, D))
    lse = np.full((T_q, Hq), np.inf)
    B = len(cu_seqlens_q) - 1
    for b in range(B):
        q0, q1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        k0, k1 = int(cu_seqlens_kv[b]), int(cu_seqlens_kv[b + 1])
        if seqused_q is not None:
            q1 = min(q1, q0 + int(seqused_q[b]))  # the shorter length holds
        n_kv = k1 - k0
        if seqused_kv is not None:
            n_kv = min(n_kv, int(seqused_kv[b]))
        if q1 <= q0:
            continue
        o, l = attention(qn[None, q0:q1], kn[None, k0:k1], vn[None, k0:k1], scale=scale,
                         layout="BSND", causal=causal, window=window,
                         key_mask=None if km is None else km[None, k0:k1],
                         actual_seq_lengths=[n_kv])
        out[q0:q1] = o[0]
        lse[q0:q1] = l[0].T
    return out, lse
