"""Seeded synthetic inputs for the paged-attention kernels and for the oracle.

This module draws random numbers and lays them out as page pools, block tables
and sequence lengths. It does no attention arithmetic. The CUDA path's tests,
the benchmark and the fp64 oracle all take their inputs from here, so both
sides see exactly the same values.

Layouts (the pages fix none of them; these are this library's readings):

* query            ``q[B, Hq, D]``
* page pools       ``k_pages, v_pages [num_pages, Hkv, page_size, D]``: one
  (page, KV head) tile is ``page_size * D`` contiguous elements.
* block table      ``int32 [B, max_blocks]``: entry ``j`` is the physical page
  that holds logical block ``j`` of a sequence (the block-table mapping in
  "快速注意力内核与算子融合", Q&A on paged attention).
* lengths          ``int32 [B]``.
* prefill tensors  ``[B, T, H, D]`` contiguous.

Pool pages that no sequence uses, and the slots of a last page past the
sequence's length, are filled with NaN when ``poison`` is set, so that a
kernel that reads them shows it in its output. Unused block-table entries are
``-1``.

bf16 cases draw fp32 normals and round them to bf16 (round to nearest even);
the oracle then receives the rounded values widened to fp64.

FP8 cases hold E4M3 codes (bytes) in their page pools and one float32 scale per
(page, KV head) tile of K and of V, ``[num_pages, Hkv]``. A tile's scale is its
largest magnitude over 448, the largest finite E4M3 value, and its codes are the
fp32 normals divided by the scale and rounded to E4M3 (torch's conversion). That
is input preparation; the oracle and the kernel both read the codes and scales.
Poisoned slots hold the NaN code 0x7F.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _normal(g: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


@dataclass
class PagedDecodeCase:
    """One batch of single-token queries against a paged KV cache."""

    q: torch.Tensor
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    block_table: torch.Tensor
    kv_lens: torch.Tensor
    scale: float
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def n_qo_heads(self) -> int:
        return self.q.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_pages.shape[0]

    @property
    def n_kv_heads(self) -> int:
        return self.k_pages.shape[1]

    @property
    def page_size(self) -> int:
        return self.k_pages.shape[2]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.q.dtype == torch.bfloat16 else "f32"

    def kv_bytes(self) -> int:
        """K and V bytes that attention must read once: sum of lengths x Hkv x D x 2 tensors."""
        esize = self.k_pages.element_size()
        return int(self.kv_lens.to(torch.int64).sum()) * self.n_kv_heads * self.head_dim * esize * 2


@dataclass
class PagedDecodeFp8Case:
    q: torch.Tensor            # bf16 [B, Hq, D]
    k_codes: torch.Tensor      # uint8 [num_pages, Hkv, P, D] (E4M3)
    v_codes: torch.Tensor
    k_scale: torch.Tensor      # float32 [num_pages, Hkv]
    v_scale: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_blocks]
    kv_lens: torch.Tensor      # int32 [B]
    scale: float
    name: str = ""

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def n_qo_heads(self) -> int:
        return self.q.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_codes.shape[0]

    @property
    def n_kv_heads(self) -> int:
        return self.k_codes.shape[1]

    @property
    def page_size(self) -> int:
        return self.k_codes.shape[2]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    def kv_bytes(self) -> int:
        """Codes of every token's K and V plus the K and V scales of every page read."""
        toks = int(self.kv_lens.sum())
        pages = int(((self.kv_lens + self.page_size - 1) // self.page_size).sum())
        return toks * self.n_kv_heads * self.head_dim * 2 + pages * self.n_kv_heads * 4 * 2


@dataclass
class PrefillCase:
    """Dense causal self-attention over contiguous ``[B, T, H, D]`` tensors."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    scale: float
    name: str = ""

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def seq_len(self) -> int:
        return self.q.shape[1]

    @property
    def n_qo_heads(self) -> int:
        return self.q.shape[2]

    @property
    def n_kv_heads(self) -> int:
        return self.k.shape[2]

    @property
    def head_dim(self) -> int:
        return self.q.shape[3]

    def causal_flops(self) -> int:
        """4 * B * Hq * D * T(T+1)/2: two products per unmasked (query, key) pair."""
        t = self.seq_len
        return 4 * self.batch * self.n_qo_heads * self.head_dim * t * (t + 1) // 2


@dataclass
class CascadeCase:
    """Requests that share one prefix of pages, each with private suffix pages."""

    q: torch.Tensor
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    prefix_table: torch.Tensor   # int32 [n_prefix_blocks]
    prefix_len: int
    suffix_table: torch.Tensor   # int32 [R, max_suffix_blocks]
    suffix_lens: torch.Tensor    # int32 [R]
    scale: float
    name: str = ""

    @property
    def n_requests(self) -> int:
        return self.q.shape[0]

    @property
    def n_qo_heads(self) -> int:
        return self.q.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def n_kv_heads(self) -> int:
        return self.k_pages.shape[1]

    @property
    def page_size(self) -> int:
        return self.k_pages.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_pages.shape[0]

    def kv_bytes(self) -> int:
        """Prefix K+V counted once plus every suffix's K+V."""
        esize = self.k_pages.element_size()
        per_tok = self.n_kv_heads * self.head_dim * esize * 2
        return (self.prefix_len + int(self.suffix_lens.to(torch.int64).sum())) * per_tok

    def concatenated(self) -> PagedDecodeCase:
        """The same cache seen as plain per-request sequences (prefix blocks, then suffix blocks).

        Only valid when the prefix length is a whole number of pages, which
        every cascade case built here has.
        """
        R = self.n_requests
        n_pre = self.prefix_table.shape[0]
        ms = self.suffix_table.shape[1]
        table = torch.full((R, n_pre + ms), -1, dtype=torch.int32)
        table[:, :n_pre] = self.prefix_table.unsqueeze(0)
        table[:, n_pre:] = self.suffix_table
        lens = (self.suffix_lens + self.prefix_len).to(torch.int32)
        return PagedDecodeCase(self.q, self.k_pages, self.v_pages, table, lens, self.scale,
                               name=self.name + "/concatenated")


def _fill_pages(g, pool_k, pool_v, pages, lens_tokens, page_size, k_std, v_std, poison):
    """Write random K/V into ``pages`` (a list of page ids per sequence) for the given lengths."""
    n_kv, d = pool_k.shape[1], pool_k.shape[3]
    flat = [p for seq in pages for p in seq]
    if flat:
        idx = torch.tensor(flat, dtype=torch.int64)
        shape = (len(flat), n_kv, page_size, d)
        pool_k[idx] = _normal(g, shape, k_std, pool_k.dtype)
        pool_v[idx] = _normal(g, shape, v_std, pool_v.dtype)
    if poison:
        for seq, length in zip(pages, lens_tokens):
            tail = length % page_size
            if seq and tail:
                pool_k[seq[-1], :, tail:, :] = float("nan")
                pool_v[seq[-1], :, tail:, :] = float("nan")


def make_paged_decode(seed: int, batch: int, n_qo_heads: int, n_kv_heads: int, head_dim: int,
                      page_size: int, kv_lens, num_pages: int | None = None,
                      max_blocks: int | None = None, dtype: str = "bf16",
                      q_std: float = 1.0, k_std: float = 1.0, v_std: float = 1.0,
                      scale: float | None = None, poison: bool = True,
                      name: str = "") -> PagedDecodeCase:
    """Build a paged decode batch.

    ``kv_lens`` is a list of lengths or a ``(lo, hi)`` tuple for lengths drawn
    uniformly from ``[lo, hi]``. Pages are drawn without replacement from the
    pool in a seeded random order.
    """
    g = _gen(seed)
    tdt = DTYPES[dtype]
    if isinstance(kv_lens, tuple):
        lo, hi = kv_lens
        lens = torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64).tolist()
    else:
        lens = [int(x) for x in kv_lens]
    assert len(lens) == batch
    nblk = [(l + page_size - 1) // page_size for l in lens]
    if max_blocks is None:
        max_blocks = max(1, max(nblk))
    assert max(nblk) <= max_blocks
    need = sum(nblk)
    if num_pages is None:
        num_pages = max(1, need)
    assert need <= num_pages, "pool too small"
    q = _normal(g, (batch, n_qo_heads, head_dim), q_std, tdt)
    order = torch.randperm(num_pages, generator=g)[:need].tolist()
    pages, pos = [], 0
    for n in nblk:
        pages.append(order[pos:pos + n])
        pos += n
    fill = float("nan") if poison else 0.0
    k_pages = torch.full((num_pages, n_kv_heads, page_size, head_dim), fill, dtype=tdt)
    v_pages = torch.full((num_pages, n_kv_heads, page_size, head_dim), fill, dtype=tdt)
    _fill_pages(g, k_pages, v_pages, pages, lens, page_size, k_std, v_std, poison)
    table = torch.full((batch, max_blocks), -1, dtype=torch.int32)
    for b, seq in enumerate(pages):
        if seq:
            table[b, :len(seq)] = torch.tensor(seq, dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PagedDecodeCase(q, k_pages, v_pages, table, torch.tensor(lens, dtype=torch.int32),
                           float(scale), name=name)


def make_paged_decode_fp8(seed: int, batch: int, n_qo_heads: int, n_kv_heads: int, head_dim: int,
                          page_size: int, kv_lens, num_pages: int | None = None,
                          max_blocks: int | None = None, q_std: float = 1.0, k_std: float = 1.0,
                          v_std: float = 1.0, scale: float | None = None, poison: bool = True,
                          name: str = "") -> PagedDecodeFp8Case:
    """Build a paged decode batch over FP8 E4M3 pages with per-(page, KV head) scales.

    The lengths, page order and query follow ``make_paged_decode`` for the same seed
    (q rounded to bf16); the pages hold E4M3 codes of fp32 normals.
    """
    g = _gen(seed)
    if isinstance(kv_lens, tuple):
        lo, hi = kv_lens
        lens = torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64).tolist()
    else:
        lens = [int(x) for x in kv_lens]
    assert len(lens) == batch
    nblk = [(l + page_size - 1) // page_size for l in lens]
    if max_blocks is None:
        max_blocks = max(1, max(nblk))
    assert max(nblk) <= max_blocks
    need = sum(nblk)
    if num_pages is None:
        num_pages = max(1, need)
    assert need <= num_pages, "pool too small"
    q = _normal(g, (batch, n_qo_heads, head_dim), q_std, torch.bfloat16)
    order = torch.randperm(num_pages, generator=g)[:need].tolist()
    pages, pos = [], 0
    for n in nblk:
        pages.append(order[pos:pos + n])
        pos += n
    shape = (num_pages, n_kv_heads, page_size, head_dim)
    fill = 0x7F if poison else 0
    k_codes = torch.full(shape, fill, dtype=torch.uint8)
    v_codes = torch.full(shape, fill, dtype=torch.uint8)
    k_scale = torch.ones((num_pages, n_kv_heads), dtype=torch.float32)
    v_scale = torch.ones((num_pages, n_kv_heads), dtype=torch.float32)
    flat = [p for seq in pages for p in seq]
    for start in range(0, len(flat), 1024):
        idx = torch.tensor(flat[start:start + 1024], dtype=torch.int64)
        for codes, sc, std in ((k_codes, k_scale, k_std), (v_codes, v_scale, v_std)):
            x = _normal(g, (len(idx), n_kv_heads, page_size, head_dim), std, torch.float32)
            amax = x.abs().amax(dim=(2, 3))
            s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
            y = (x / s[:, :, None, None]).clamp(-448.0, 448.0)
            codes[idx] = y.to(torch.float8_e4m3fn).view(torch.uint8)
            sc[idx] = s
    if poison:
        for seq, length in zip(pages, lens):
            tail = length % page_size
            if seq and tail:
                k_codes[seq[-1], :, tail:, :] = 0x7F
                v_codes[seq[-1], :, tail:, :] = 0x7F
    table = torch.full((batch, max_blocks), -1, dtype=torch.int32)
    for b, seq in enumerate(pages):
        if seq:
            table[b, :len(seq)] = torch.tensor(seq, dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PagedDecodeFp8Case(q, k_codes, v_codes, k_scale, v_scale, table,
                              torch.tensor(lens, dtype=torch.int32), float(scale), name=name)


def make_prefill(seed: int, batch: int, seq_len: int, n_qo_heads: int, n_kv_heads: int,
                 head_dim: int, dtype: str = "bf16", std: float = 1.0,
                 scale: float | None = None, name: str = "") -> PrefillCase:
    g = _gen(seed)
    tdt = DTYPES[dtype]
    q = _normal(g, (batch, seq_len, n_qo_heads, head_dim), std, tdt)
    k = _normal(g, (batch, seq_len, n_kv_heads, head_dim), std, tdt)
    v = _normal(g, (batch, seq_len, n_kv_heads, head_dim), 1.0, tdt)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PrefillCase(q, k, v, float(scale), name=name)


def make_cascade(seed: int, n_requests: int, prefix_len: int, suffix_lens, n_qo_heads: int,
                 n_kv_heads: int, head_dim: int, page_size: int = 16,
                 num_pages: int | None = None, max_suffix_blocks: int | None = None,
                 dtype: str = "bf16", scale: float | None = None, poison: bool = True,
                 name: str = "") -> CascadeCase:
    """Build a shared-prefix batch. ``prefix_len`` must be a multiple of ``page_size``."""
    assert prefix_len % page_size == 0
    g = _gen(seed)
    tdt = DTYPES[dtype]
    if isinstance(suffix_lens, tuple):
        lo, hi = suffix_lens
        lens = torch.randint(lo, hi + 1, (n_requests,), generator=g, dtype=torch.int64).tolist()
    else:
        lens = [int(x) for x in suffix_lens]
    n_pre = prefix_len // page_size
    nblk = [(l + page_size - 1) // page_size for l in lens]
    if max_suffix_blocks is None:
        max_suffix_blocks = max(1, max(nblk))
    need = n_pre + sum(nblk)
    if num_pages is None:
        num_pages = need
    assert need <= num_pages
    q = _normal(g, (n_requests, n_qo_heads, head_dim), 1.0, tdt)
    order = torch.randperm(num_pages, generator=g)[:need].tolist()
    prefix_pages = order[:n_pre]
    pos = n_pre
    suffix_pages = []
    for n in nblk:
        suffix_pages.append(order[pos:pos + n])
        pos += n
    fill = float("nan") if poison else 0.0
    k_pages = torch.full((num_pages, n_kv_heads, page_size, head_dim), fill, dtype=tdt)
    v_pages = torch.full((num_pages, n_kv_heads, page_size, head_dim), fill, dtype=tdt)
    _fill_pages(g, k_pages, v_pages, [prefix_pages] + suffix_pages, [prefix_len] + lens,
                page_size, 1.0, 1.0, poison)
    prefix_table = torch.tensor(prefix_pages, dtype=torch.int32)
    suffix_table = torch.full((n_requests, max_suffix_blocks), -1, dtype=torch.int32)
    for r, seq in enumerate(suffix_pages):
        if seq:
            suffix_table[r, :len(seq)] = torch.tensor(seq, dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return CascadeCase(q, k_pages, v_pages, prefix_table, prefix_len, suffix_table,
                       torch.tensor(lens, dtype=torch.int32), float(scale), name=name)


@dataclass
class FlatGemmCase:
    """The decode-phase flat GEMM: ``x[m, k]`` tokens times the transposed weights ``w[n, k]``."""
    x: torch.Tensor
    w: torch.Tensor
    name: str = ""

    @property
    def m(self) -> int:
        return self.x.shape[0]

    @property
    def n(self) -> int:
        return self.w.shape[0]

    @property
    def k(self) -> int:
        return self.x.shape[1]

    def bytes_moved(self) -> int:
        """Bytes a call must move at least: w and x read once, y written once (bf16)."""
        return 2 * (self.n * self.k + self.m * self.k + self.m * self.n)


def make_flat_gemm(seed: int, m: int, n: int, k: int, name: str = "") -> FlatGemmCase:
    """bf16 ``x ~ N(0, 1)`` and ``w ~ N(0, 1/k)`` (so ``y`` is about N(0, 1)), both rounded to bf16."""
    g = _gen(seed)
    x = _normal(g, (m, k), 1.0, torch.bfloat16)
    w = _normal(g, (n, k), 1.0 / math.sqrt(k), torch.bfloat16)
    return FlatGemmCase(x, w, name=name)


# --------------------------------------------------------------------------------------
# The five named workloads (seed 1000 + workload number).
# --------------------------------------------------------------------------------------

def single_seq_decode_f32() -> PagedDecodeCase:
    """fp32, batch 1, 8 query heads = 8 KV heads, d 64, length 256, page 16, 64-page pool."""
    return make_paged_decode(1001, 1, 8, 8, 64, 16, [256], num_pages=64, dtype="f32",
                             name="single_seq_decode_f32")


def llama7b_batched_decode(poison: bool = True) -> PagedDecodeCase:
    """bf16, batch 16, 32/32 heads, d 128, lengths U[512, 4096], page 16, 8192-page pool."""
    return make_paged_decode(1002, 16, 32, 32, 128, 16, (512, 4096), num_pages=8192,
                             max_blocks=256, dtype="bf16", poison=poison,
                             name="llama7b_batched_decode")


def llama7b_batched_decode_fp8(poison: bool = True) -> PagedDecodeFp8Case:
    """The Llama-7B batch's shape over FP8 E4M3 pages (same lengths and page order)."""
    return make_paged_decode_fp8(1002, 16, 32, 32, 128, 16, (512, 4096), num_pages=8192,
                                 max_blocks=256, poison=poison, name="llama7b_batched_decode_fp8")


def long_context_gqa_decode(poison: bool = True) -> PagedDecodeCase:
    """bf16, batch 4, 32 query heads over 8 KV heads, d 128, length 32768, k ~ 2 N(0,1)."""
    return make_paged_decode(1003, 4, 32, 8, 128, 16, [32768] * 4, num_pages=8192,
                             max_blocks=2048, dtype="bf16", k_std=2.0, poison=poison,
                             name="long_context_gqa_decode")


def long_context_gqa8_decode(poison: bool = True) -> PagedDecodeCase:
    """The long-context batch with 8 query heads per KV head: 64 query heads over 8 KV heads."""
    return make_paged_decode(1013, 4, 64, 8, 128, 16, [32768] * 4, num_pages=8192,
                             max_blocks=2048, dtype="bf16", k_std=2.0, poison=poison,
                             name="long_context_gqa8_decode")


def long_context_gqa8_decode_fp8(poison: bool = True) -> PagedDecodeFp8Case:
    """The same long-context GQA-8 batch over FP8 E4M3 pools with per-(page, KV head) scales."""
    return make_paged_decode_fp8(1014, 4, 64, 8, 128, 16, [32768] * 4, num_pages=8192,
                                 max_blocks=2048, k_std=2.0, poison=poison,
                                 name="long_context_gqa8_decode_fp8")


LONG_CONTEXT_SPLITS = 32


def causal_prefill_llama7b() -> PrefillCase:
    """bf16, batch 8, T 1024, 32/32 heads, d 128, contiguous [B, T, H, D]."""
    return make_prefill(1004, 8, 1024, 32, 32, 128, dtype="bf16", name="causal_prefill_llama7b")


def cascade_shared_prefix_decode(poison: bool = True) -> CascadeCase:
    """bf16, 64 requests, 4096-token shared prefix, suffix U[128, 1024], 32/8 heads, d 128."""
    return make_cascade(1005, 64, 4096, (128, 1024), 32, 8, 128, page_size=16, num_pages=8192,
                        max_suffix_blocks=64, dtype="bf16", poison=poison,
                        name="cascade_shared_prefix_decode")


# The flat GEMMs either side of attention in a Llama-2-7B-shaped decode step (hidden size
# 4096): the fused QKV projection (n = 3 x 4096) and the output projection (n = 4096),
# for m decode tokens. Synthetic weights of that shape (no trained weights are used).
LLAMA7B_HIDDEN = 4096


def llama7b_qkv_projection(m: int) -> FlatGemmCase:
    return make_flat_gemm(1100 + m, m, 3 * LLAMA7B_HIDDEN, LLAMA7B_HIDDEN, name=f"llama7b_qkv_projection_m{m}")


def llama7b_o_projection(m: int) -> FlatGemmCase:
    return make_flat_gemm(1200 + m, m, LLAMA7B_HIDDEN, LLAMA7B_HIDDEN, name=f"llama7b_o_projection_m{m}")
