"""fp64 CPU oracle for paged / causal scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA path.

Every function here is the definition written out in numpy float64. It builds
the full score matrix, subtracts the row maximum, exponentiates, normalises and
multiplies by V. There is no tiling, fusion or reordering beyond that. Sources:

* The attention definition ``Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V``:
  "FlashInfer内核库：利用CUDA Warp-Level Primitives加速级联推理的Attention计算",
  section 1 (背景与挑战). The scale is a parameter; the named workloads pass
  1/sqrt(d).
* Max subtraction for a stable softmax: "TensorRT-LLM深度优化：利用FMHA（Fused
  Multi-Head Attention）内核加速Hopper架构推理", section 2 (Numerical
  Stability).
* Paged K/V: a block table maps each logical block of a sequence to a
  physical page, and the kernel reads K and V through it: "快速注意力内核与算子融合",
  Q&A on paged attention.
* Partial softmax states, combined after the fact: "【FlashAttention-V4，非官方】
  FlashDecoding++", section 1 (FlashDecoding computes each partial separately
  and updates them all at the end).
* The unified maximum value: the same page, sections 1 and 3. Partials are
  computed against one shared preset maximum and need no synchronised update.
* FP8 K/V: "TensorRT-LLM深度优化：利用FMHA（Fused Multi-Head Attention）内核加速
  Hopper架构推理", section 4 (FP8 lowers the memory traffic). The page names no
  format and no scaling.

Readings where the pages are silent (the design document lists them too):

* The LSE is the natural log of ``sum_j exp(scale * q . k_j)``. It is ``-inf``
  for an empty key set, and the output is then 0.
* GQA: query head ``h`` reads KV head ``h // (Hq / Hkv)``.
* Causal: query ``i`` sees keys ``0..i``, and the query length equals the key
  length.
* A split covers a contiguous, page-aligned range of a sequence's blocks.
  Split ``s`` holds blocks ``[s*pps, (s+1)*pps)``.
* The unified-max partial of a chunk is ``(sum exp(s - phi) v, sum exp(s - phi))``
  with a preset ``phi``. Chunks that share ``phi`` merge by plain sums.
* A chunked prefill over a paged cache appends ``C`` new tokens to a sequence
  that already holds ``L0`` tokens: the new tokens' K and V are in the cache at
  positions ``L0 .. L0 + C - 1`` (written before the call), and new token ``i``
  (position ``L0 + i``) sees keys ``0 .. L0 + i``. It joins the paged gather and
  the causal mask; the pages describe both but not their combination.
* FP8 pages hold E4M3 codes (the OCP 8-bit floating-point format), and each
  (page, KV head) tile of K and of V has one float scale: the element's value is
  ``e4m3(code) * scale``. Attention over FP8 pages is the plain attention over
  those values.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attend", "gather_sequence", "decode_paged", "prefill_causal", "merge_states",
    "merge_many", "split_ranges", "decode_split_partials", "cascade_decode",
    "unified_max_partials", "unified_max_combine", "unified_max_needs_fallback",
    "e4m3_to_float", "decode_paged_fp8", "prefill_paged_chunk",
]

NEG_INF = -math.inf


def attend(q_rows, keys, values, scale, keep=None):
    """Softmax attention of ``q_rows[n, D]`` over ``keys[L, D]`` / ``values[L, D]``.

    ``keep`` (bool ``[n, L]``, optional) drops the (row, key) pairs that are False.
    Returns ``out[n, D]`` and ``lse[n]`` (natural log of the softmax denominator
    in scaled-logit units). A row with no key gets ``out = 0`` and ``lse = -inf``.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    n, d = q_rows.shape
    L = keys.shape[0]
    out = np.zeros((n, values.shape[1] if values.ndim == 2 else d), dtype=np.float64)
    lse = np.full((n,), NEG_INF, dtype=np.float64)
    if L == 0:
        return out, lse
    scores = scale * (q_rows @ keys.T)                     # [n, L], the full score matrix
    if keep is not None:
        scores = np.where(keep, scores, NEG_INF)
    m = scores.max(axis=1)                                 # row maximum
    live = np.isfinite(m)
    if not live.any():
        return out, lse
    w = np.exp(scores[live] - m[live, None])               # max-subtracted exponentials
    z = w.sum(axis=1)                                      # softmax denominator
    out[live] = (w @ values) / z[:, None]
    lse[live] = m[live] + np.log(z)
    return out, lse


def gather_sequence(k_pages, v_pages, table_row, kv_len, kv_head):
    """Logical K and V rows ``[kv_len, D]`` of one sequence and one KV head.

    Token ``t`` lives in physical page ``table_row[t // P]`` at slot ``t % P``.
    """
    P = k_pages.shape[2]
    ks, vs = [], []
    for t in range(int(kv_len)):
        page = int(table_row[t // P])
        ks.append(k_pages[page, kv_head, t % P])
        vs.append(v_pages[page, kv_head, t % P])
    d = k_pages.shape[3]
    if not ks:
        return np.zeros((0, d)), np.zeros((0, d))
    return np.asarray(ks, dtype=np.float64), np.asarray(vs, dtype=np.float64)


def _gather_fast(k_pages, v_pages, table_row, kv_len, kv_head):
    """``gather_sequence`` done with one fancy index per tensor (same result, for big cases)."""
    P = k_pages.shape[2]
    t = np.arange(int(kv_len))
    pages = np.asarray(table_row, dtype=np.int64)[t // P]
    return (np.asarray(k_pages[pages, kv_head, t % P], dtype=np.float64),
            np.asarray(v_pages[pages, kv_head, t % P], dtype=np.float64))


def decode_paged(q, k_pages, v_pages, block_table, kv_lens, scale, rows=None):
    """Single-token decode over a paged cache.

    ``q[B, Hq, D]``, pools ``[num_pages, Hkv, P, D]``, ``block_table[B, max_blocks]``,
    ``kv_lens[B]``. Returns ``out[B, Hq, D]`` and ``lse[B, Hq]``. ``rows``, a list
    of ``(b, h)`` pairs, limits the work to those rows (the others stay NaN).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    wanted = None if rows is None else {(int(b), int(h)) for b, h in rows}
    for b in range(B):
        for g in range(Hkv):
            heads = [h for h in range(g * G, (g + 1) * G)
                     if wanted is None or (b, h) in wanted]
            if not heads:
                continue
            K, V = _gather_fast(k_pages, v_pages, block_table[b], kv_lens[b], g)
            o, l = attend(q[b, heads], K, V, scale)
            out[b, heads] = o
            lse[b, heads] = l
    return out, lse


def e4m3_to_float(codes):
    """Values of FP8 E4M3 codes (any integer array of bytes) as float64.

    The OCP 8-bit floating-point E4M3 format: a sign bit s, four exponent bits e with
    bias 7 and three mantissa bits m. e = 0 is subnormal, (-1)^s * 2^-6 * m/8. Otherwise
    the value is (-1)^s * 2^(e-7) * (1 + m/8), except e = 15 with m = 7, which is NaN:
    the format has no infinities, and its largest finite magnitude is 2^8 * 1.75 = 448.
    """
    c = np.asarray(codes).astype(np.int64) & 0xFF
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (c & 7 == 7), np.nan, val)


def decode_paged_fp8(q, k_codes, v_codes, k_scale, v_scale, block_table, kv_lens, scale,
                     rows=None):
    """Single-token decode over a paged cache of FP8 E4M3 codes.

    ``k_codes``/``v_codes`` ``[num_pages, Hkv, P, D]`` (bytes), ``k_scale``/``v_scale``
    ``[num_pages, Hkv]``. Each sequence's tokens are gathered through the block table
    as in ``decode_paged`` and dequantised (code value times its tile's scale) before
    the plain attention. Returns ``out[B, Hq, D]`` and ``lse[B, Hq]``.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_codes.shape[1]
    P = k_codes.shape[2]
    G = Hq // Hkv
    ks = np.asarray(k_scale, dtype=np.float64)
    vs = np.asarray(v_scale, dtype=np.float64)
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    wanted = None if rows is None else {(int(b), int(h)) for b, h in rows}
    for b in range(B):
        t = np.arange(int(kv_lens[b]))
        pages = None
        for g in range(Hkv):
            heads = [h for h in range(g * G, (g + 1) * G)
                     if wanted is None or (b, h) in wanted]
            if not heads:
                continue
            if pages is None:
                pages = np.asarray(block_table[b], dtype=np.int64)[t // P]
            K = e4m3_to_float(k_codes[pages, g, t % P]) * ks[pages, g][:, None]
            V = e4m3_to_float(v_codes[pages, g, t % P]) * vs[pages, g][:, None]
            o, l = attend(q[b, heads], K, V, scale)
            out[b, heads] = o
            lse[b, heads] = l
    return out, lse


def prefill_causal(q, k, v, scale, rows=None):
    """Causal self-attention over ``[B, T, H, D]`` tensors.

    Returns ``out[B, T, Hq, D]`` and ``lse[B, Hq, T]``. Query ``i`` sees keys
    ``0..i``. ``rows``, a list of ``(b, h, i)``, limits the work to those rows
    (the others stay NaN).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, Hq, T), np.nan)
    if rows is None:
        causal = np.tril(np.ones((T, T), dtype=bool))      # keep j <= i
        for b in range(B):
            for h in range(Hq):
                o, l = attend(q[b, :, h], k[b, :, h // G], v[b, :, h // G], scale, keep=causal)
                out[b, :, h] = o
                lse[b, h] = l
        return out, lse
    for b, h, i in rows:
        b, h, i = int(b), int(h), int(i)
        o, l = attend(q[b, i:i + 1, h], k[b, :i + 1, h // G], v[b, :i + 1, h // G], scale)
        out[b, i, h] = o[0]
        lse[b, h, i] = l[0]
    return out, lse


def prefill_paged_chunk(q, k_pages, v_pages, block_table, prefix_lens, scale):
    """Chunked prefill over a paged cache.

    ``q[B, C, Hq, D]`` holds the queries of ``C`` new tokens per sequence; sequence ``b``
    already had ``prefix_lens[b]`` tokens, and its ``prefix_lens[b] + C`` tokens (old and
    new) are in the pools ``[num_pages, Hkv, P, D]`` through ``block_table[b]``. New token
    ``i`` attends to keys ``0 .. prefix_lens[b] + i``. Returns ``out[B, C, Hq, D]`` and
    ``lse[B, Hq, C]``.
    """
    q = np.asarray(q, dtype=np.float64)
    B, C, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    out = np.full((B, C, Hq, D), np.nan)
    lse = np.full((B, Hq, C), np.nan)
    for b in range(B):
        L0 = int(prefix_lens[b])
        L = L0 + C
        keep = np.arange(L)[None, :] <= (L0 + np.arange(C))[:, None]   # [C, L]
        for g in range(Hkv):
            K, V = _gather_fast(k_pages, v_pages, block_table[b], L, g)
            for h in range(g * G, (g + 1) * G):
                o, l = attend(q[b, :, h], K, V, scale, keep=keep)
                out[b, :, h] = o
                lse[b, h] = l
    return out, lse


def merge_states(out_a, lse_a, out_b, lse_b):
    """Combine two partial softmax states over disjoint key sets.

    ``M = max(lse_a, lse_b)``, ``w = exp(lse - M)``,
    ``out = (w_a out_a + w_b out_b) / (w_a + w_b)``, ``lse = M + ln(w_a + w_b)``.
    Two empty sides give ``out = 0`` and ``lse = -inf``.
    """
    return merge_many(np.stack([out_a, out_b]), np.stack([lse_a, lse_b]))


def merge_many(outs, lses):
    """Combine ``S`` partial states: ``outs[S, ..., D]``, ``lses[S, ...]``."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    M = lses.max(axis=0)
    live = np.isfinite(M)
    Msafe = np.where(live, M, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - Msafe[None]), 0.0)   # [S, ...]
    z = w.sum(axis=0)
    num = (w[..., None] * np.where(np.isfinite(lses)[..., None], outs, 0.0)).sum(axis=0)
    out = np.where(live[..., None], num / np.where(live, z, 1.0)[..., None], 0.0)
    lse = np.where(live, Msafe + np.log(np.where(live, z, 1.0)), NEG_INF)
    return out, lse


def split_ranges(n_blocks, pages_per_split):
    """Token-free block ranges ``[lo, hi)`` of the non-empty splits of one sequence."""
    out = []
    lo = 0
    while lo < n_blocks:
        out.append((lo, min(lo + pages_per_split, n_blocks)))
        lo += pages_per_split
    return out


def decode_split_partials(q, k_pages, v_pages, block_table, kv_lens, scale, pages_per_split):
    """Partial ``(out, lse)`` states of each split of each sequence.

    Returns lists indexed ``[b]`` of ``(outs[S_b, Hq, D], lses[S_b, Hq])``. Each
    split is plain attention over its own block range.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    P = k_pages.shape[2]
    result = []
    for b in range(B):
        L = int(kv_lens[b])
        nb = (L + P - 1) // P
        ranges = split_ranges(nb, pages_per_split)
        outs = np.zeros((len(ranges), Hq, D))
        lses = np.full((len(ranges), Hq), NEG_INF)
        for g in range(Hkv):
            K, V = _gather_fast(k_pages, v_pages, block_table[b], L, g)
            for s, (lo, hi) in enumerate(ranges):
                t0, t1 = lo * P, min(hi * P, L)
                o, l = attend(q[b, g * G:(g + 1) * G], K[t0:t1], V[t0:t1], scale)
                outs[s, g * G:(g + 1) * G] = o
                lses[s, g * G:(g + 1) * G] = l
        result.append((outs, lses))
    return result


def cascade_decode(q, k_pages, v_pages, prefix_table, prefix_len, suffix_table, suffix_lens,
                   scale):
    """Decode where every request's sequence is the shared prefix followed by its own suffix.

    This is the definition: plain attention over the concatenated logical
    sequence. How the work is split (prefix once, then merge) is not part of it.
    """
    q = np.asarray(q, dtype=np.float64)
    R, Hq, D = q.shape
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    out = np.zeros((R, Hq, D))
    lse = np.zeros((R, Hq))
    for g in range(Hkv):
        Kp, Vp = _gather_fast(k_pages, v_pages, prefix_table, prefix_len, g)
        for r in range(R):
            Ks, Vs = _gather_fast(k_pages, v_pages, suffix_table[r], suffix_lens[r], g)
            K = np.concatenate([Kp, Ks])
            V = np.concatenate([Vp, Vs])
            o, l = attend(q[r, g * G:(g + 1) * G], K, V, scale)
            out[r, g * G:(g + 1) * G] = o
            lse[r, g * G:(g + 1) * G] = l
    return out, lse


def unified_max_partials(q_rows, keys, values, scale, phi, chunk):
    """Chunked partial sums against a preset unified maximum ``phi``.

    Each chunk of ``chunk`` keys gives ``acc_c = sum_j exp(s_j - phi) v_j`` and
    ``l_c = sum_j exp(s_j - phi)``, with no max taken anywhere. Returns
    ``accs[C, n, D]`` and ``ls[C, n]``.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    L = keys.shape[0]
    n = q_rows.shape[0]
    C = max(1, (L + chunk - 1) // chunk)
    accs = np.zeros((C, n, values.shape[1]))
    ls = np.zeros((C, n))
    for c in range(C):
        s = scale * (q_rows @ keys[c * chunk:(c + 1) * chunk].T)
        e = np.exp(s - phi)
        accs[c] = e @ values[c * chunk:(c + 1) * chunk]
        ls[c] = e.sum(axis=1)
    return accs, ls


def unified_max_combine(accs, ls, phi):
    """Combine unified-max partials that share ``phi``: plain sums, one division."""
    acc = np.asarray(accs).sum(axis=0)
    l = np.asarray(ls).sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(l[:, None] > 0, acc / l[:, None], 0.0)
        lse = np.where(l > 0, phi + np.log(l), NEG_INF)
    return out, lse


def unified_max_needs_fallback(scores, phi, beta_hi, beta_lo):
    """Whether exponentiating against ``phi`` is unsafe for these scaled logits.

    True when a logit sits more than ``beta_hi`` above ``phi`` (its exponential
    risks overflow in fp32) or every logit sits more than ``beta_lo`` below ``phi``
    (every exponential underflows).
    """
    s = np.asarray(scores, dtype=np.float64)
    if s.size == 0:
        return False
    return bool((s > phi + beta_hi).any() or (s < phi - beta_lo).all())
