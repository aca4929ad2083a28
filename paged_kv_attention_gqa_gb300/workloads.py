"""Seeded synthetic workloads for paged GQA attention.

This module only draws inputs: lengths, page assignments, the four index arrays a
caller hands the library, q / new K / new V and the cached prefix.  It holds none of
the attention arithmetic and none of the library's planning, so both the CUDA path
and the oracle can take their inputs from it.

Recipe (all draws from numpy's PCG64 ``default_rng(seed)`` in the order listed, float
data from ``torch.Generator(device).manual_seed(seed)``):

  tiny      4 rows, Hq 8 / Hkv 2, D 64, page 16; L ~ U[17, 100]; a pool of 64 pages,
            shuffled, rows take pages in order; one new token per row.
  batch     128 rows, 32 / 8, D 128, page 16; L ~ U[512, 4096]; pool = ceil(1.1 x pages
            used), shuffled; one new token per row; 32 layers; q scaled by 1/sqrt(128).
  prefill   16 rows, 32 / 8, D 128, page 16; n ~ U[128, 2048]; c ~ U[0, 4096] with
            row 0's c = 0; L = c + n; pool ceil(1.1 x used); causal.
  mixed     100 rows: 4 prompt rows at seeded positions (n ~ U[512, 1024],
            c ~ U[0, 2048]) and 96 one-token rows (L ~ U[256, 8192]); 32 / 8, D 128,
            page 16; pool ceil(1.1 x used) + 1 sink page (the last page of the pool).
  long      8 rows, 64 / 8, D 128, page 16; L ~ U[65536, 131072]; pool ceil(1.1 x used);
            window_left -1 or 4096.

Lengths are post-append: the cache holds L - n tokens before the step, the step
appends n.  q, K and V are N(0, 1) rounded to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

try:  # torch is plumbing here: device memory and RNG for the float inputs
    import torch
except ImportError:  # pragma: no cover - the oracle's CPU tests need numpy only
    torch = None


@dataclass
class PagedBatch:
    """Shapes, lengths and the index arrays of one synthetic step."""
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_lens: np.ndarray            # int64 [B] post-append lengths L_r
    qo_lens: np.ndarray            # int64 [B] new tokens n_r
    page_table: list               # list of int64 arrays, pages of each row in order
    max_pages: int
    num_layers: int = 1
    window_left: int = -1
    causal: bool = True
    sink_page: int = -1
    q_scale: float = 1.0
    max_prefill_rows: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.kv_lens)

    @property
    def num_tokens(self) -> int:
        return int(self.qo_lens.sum())

    @property
    def qo_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.qo_lens)]).astype(np.int32)

    @property
    def kv_indptr(self) -> np.ndarray:
        counts = [len(p) for p in self.page_table]
        return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)

    @property
    def kv_indices(self) -> np.ndarray:
        if not self.page_table:
            return np.zeros(0, dtype=np.int32)
        return np.concatenate([np.asarray(p, dtype=np.int64) for p in self.page_table]).astype(np.int32)

    @property
    def last_page_len(self) -> np.ndarray:
        # the fill count a caller's page table reports for its last page
        return np.array([(int(L) - 1) % self.page_size + 1 if L > 0 else 0 for L in self.kv_lens],
                        dtype=np.int32)

    def index_arrays(self):
        return self.qo_indptr, self.kv_indptr, self.kv_indices, self.last_page_len


def _pages_needed(lengths, page_size):
    return [max(0, math.ceil(int(L) / page_size)) for L in lengths]


def assign_pages(rng, lengths, page_size, pool_pages=None, pool_factor=1.1, reserve_sink=False):
    """Draw each row's pages without replacement from a shuffled pool.

    Returns (page_table, max_pages, sink_page)."""
    need = _pages_needed(lengths, page_size)
    total = sum(need)
    if pool_pages is None:
        pool_pages = max(1, math.ceil(pool_factor * total))
    assert pool_pages >= total
    max_pages = pool_pages + (1 if reserve_sink else 0)
    shuffled = rng.permutation(pool_pages)
    table, at = [], 0
    for k in need:
        table.append(np.asarray(shuffled[at: at + k], dtype=np.int64))
        at += k
    sink = max_pages - 1 if reserve_sink else -1
    return table, max_pages, sink


def _u(rng, lo, hi, size):
    return rng.integers(lo, hi + 1, size=size).astype(np.int64)


def config_tiny(seed: int = 0) -> PagedBatch:
    rng = np.random.default_rng(seed)
    L = _u(rng, 17, 100, 4)
    table, max_pages, _ = assign_pages(rng, L, 16, pool_pages=64)
    return PagedBatch("tiny decode", 8, 2, 64, 16, L, np.ones(4, np.int64), table, max_pages)


def config_batch_decode(seed: int = 0, batch: int = 128, num_layers: int = 32) -> PagedBatch:
    rng = np.random.default_rng(seed)
    L = _u(rng, 512, 4096, batch)
    table, max_pages, _ = assign_pages(rng, L, 16)
    return PagedBatch("batch decode", 32, 8, 128, 16, L, np.ones(batch, np.int64), table, max_pages,
                      num_layers=num_layers, q_scale=1.0 / math.sqrt(128.0))


def config_prefill(seed: int = 0, batch: int = 16, new_range=(128, 2048), prefix_range=(0, 4096)) -> PagedBatch:
    rng = np.random.default_rng(seed)
    n = _u(rng, new_range[0], new_range[1], batch)
    c = _u(rng, prefix_range[0], prefix_range[1], batch)
    c[0] = 0
    L = c + n
    table, max_pages, _ = assign_pages(rng, L, 16)
    return PagedBatch("ragged prefill", 32, 8, 128, 16, L, n, table, max_pages, causal=True,
                      meta={"prefix": c})


def config_mixed(seed: int = 0, decode_rows: int = 96, prompt_rows: int = 4,
                 decode_len=(256, 8192), prompt_new=(512, 1024), prompt_prefix=(0, 2048)) -> PagedBatch:
    rng = np.random.default_rng(seed)
    B = decode_rows + prompt_rows
    where = np.sort(rng.choice(B, size=prompt_rows, replace=False))
    n_prompt = _u(rng, prompt_new[0], prompt_new[1], prompt_rows)
    c_prompt = _u(rng, prompt_prefix[0], prompt_prefix[1], prompt_rows)
    L_dec = _u(rng, decode_len[0], decode_len[1], decode_rows)
    L = np.zeros(B, np.int64)
    n = np.ones(B, np.int64)
    is_prompt = np.zeros(B, bool)
    is_prompt[where] = True
    L[is_prompt] = c_prompt + n_prompt
    n[is_prompt] = n_prompt
    L[~is_prompt] = L_dec
    table, max_pages, sink = assign_pages(rng, L, 16, reserve_sink=True)
    return PagedBatch("mixed", 32, 8, 128, 16, L, n, table, max_pages, causal=True, sink_page=sink,
                      max_prefill_rows=prompt_rows, meta={"prompt_rows": where})


def config_long(seed: int = 0, window_left: int = -1, batch: int = 8,
                length=(65536, 131072)) -> PagedBatch:
    rng = np.random.default_rng(seed)
    L = _u(rng, length[0], length[1], batch)
    table, max_pages, _ = assign_pages(rng, L, 16)
    return PagedBatch("long decode", 64, 8, 128, 16, L, np.ones(batch, np.int64), table, max_pages,
                      window_left=window_left)


def custom(seed: int, kv_lens, qo_lens, *, num_qo_heads, num_kv_heads, head_dim, page_size,
           pool_factor=1.1, pool_pages=None, reserve_sink=False, **kw) -> PagedBatch:
    """Any lengths; used by the parity tests for ragged and edge-case shapes."""
    rng = np.random.default_rng(seed)
    L = np.asarray(kv_lens, np.int64)
    n = np.asarray(qo_lens, np.int64)
    table, max_pages, sink = assign_pages(rng, L, page_size, pool_pages=pool_pages,
                                          pool_factor=pool_factor, reserve_sink=reserve_sink)
    return PagedBatch("custom", num_qo_heads, num_kv_heads, head_dim, page_size, L, n, table, max_pages,
                      sink_page=sink, **kw)


WORKLOADS = {
    "tiny": config_tiny,
    "batch": config_batch_decode,
    "prefill": config_prefill,
    "mixed": config_mixed,
    "long": config_long,
}


# ----------------------------------------------------------------------------------------------
# float inputs (torch is used for memory and its RNG only)

def _flat_slot_rows(pb: PagedBatch, r: int, positions):
    """Row index into a layer slice viewed as [max_pages * 2 * page_size, Hkv, D] of the K
    slot of each position (the V slot is page_size rows further)."""
    pages = pb.page_table[r]
    P = pb.page_size
    pos = np.asarray(positions, np.int64)
    return pages[pos // P] * 2 * P + pos % P


def make_inputs(pb: PagedBatch, *, device="cpu", seed: int = 0, unused: str = "nan",
                layers: int | None = None, prefix: bool = True):
    """q, k_new, v_new and the KV cache for one step.

    unused = "nan":   every slot that holds no token of any row is bf16 NaN (the
                      robustness setting: tails and free pages must never leak in)
    unused = "randn": the whole cache is N(0,1) first (the timed setting)
    The slots of this step's new tokens hold the fill value until the append writes
    them.  Returns dict(q, k_new, v_new, kv_cache[layers, max_pages, 2, P, Hkv, D]).
    """
    assert torch is not None
    layers = pb.num_layers if layers is None else layers
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    bf16 = torch.bfloat16
    T, Hq, Hkv, D, P = pb.num_tokens, pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, pb.page_size
    q = torch.randn(T, Hq, D, generator=g, device=device)
    if pb.q_scale != 1.0:
        q = q * pb.q_scale
    q = q.to(bf16)
    k_new = torch.randn(T, Hkv, D, generator=g, device=device).to(bf16)
    v_new = torch.randn(T, Hkv, D, generator=g, device=device).to(bf16)
    cache = torch.empty(layers, pb.max_pages, 2, P, Hkv, D, dtype=bf16, device=device)
    for l in range(layers):
        if unused == "randn":
            cache[l].normal_(generator=g)
            continue
        cache[l].fill_(float("nan"))
        if not prefix:
            continue
        flat = cache[l].view(pb.max_pages * 2 * P, Hkv, D)
        for r in range(pb.batch):
            c = int(pb.kv_lens[r] - pb.qo_lens[r])
            if c <= 0:
                continue
            kvals = torch.randn(c, Hkv, D, generator=g, device=device).to(bf16)
            vvals = torch.randn(c, Hkv, D, generator=g, device=device).to(bf16)
            rows = torch.as_tensor(_flat_slot_rows(pb, r, range(c)), device=device)
            flat[rows] = kvals
            flat[rows + P] = vvals
    if pb.sink_page >= 0:
        # the reserved sink page holds finite values; the decode pass of a mixed step
        # reads one token of it for every prompt row and drops the result
        cache[:, pb.sink_page].normal_(generator=g)
    return dict(q=q, k_new=k_new, v_new=v_new, kv_cache=cache)


def logical_kv(pb: PagedBatch, kv_layer, r: int, length: int | None = None):
    """K and V of row r as contiguous [L, Hkv, D] tensors, read from a layer slice by the
    page table the generator drew (used by tests to build unpaged inputs)."""
    L = int(pb.kv_lens[r]) if length is None else int(length)
    P = pb.page_size
    flat = kv_layer.reshape(pb.max_pages * 2 * P, pb.num_kv_heads, pb.head_dim)
    rows = torch.as_tensor(_flat_slot_rows(pb, r, range(L)), device=kv_layer.device)
    return flat[rows], flat[rows + P]


def bf16_bits(t) -> np.ndarray:
    """A bf16 tensor's bit patterns as a uint16 numpy array (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
