"""Oracle for the split-KV scheduler: a plain restatement of the split rule.

TEST INFRASTRUCTURE ONLY (see the package header in ``oracle/__init__``).

The pages fix the ingredients and leave the rule open.  MATE's
``msa_interface`` passes ``num_splits`` (0 = choose automatically) and
``page_size`` to ``get_scheduler_metadata`` and counts pages per sequence as
``ceil(kv_len / page_size)`` (``_page_counts``); FlashMLA's ``get_mla_metadata``
(section 2 of its "Tensor Shapes Reference") takes the shapes, the block table
and ``seq_lens`` and returns the metadata the decode kernel consumes.  The
reading used here, written out step by step:

  pages_b   = ceil(max(seq_b, 0) / 64)
  units     = sum_b pages_b * Hk
  cap       = num_sms * ctas_per_sm                      (persistent CTAs)
  chunk     = max(4, ceil(units / (cap * 2)))            (2 items per CTA share)
  n_b       = 1                              if pages_b <= 1
            = min(forced, pages_b, 64)       if forced > 0
            = min(ceil(pages_b / chunk), 64) otherwise
  split s of sequence b covers pages [floor(s P / n), floor((s+1) P / n))
  items     = (b, s, kvh) in (b, s, kvh) order, cost = pages of the split + 1
  grid      = min(#items, cap)
  assignment ("lpt", the host scheduler): items sorted by (cost descending,
            index ascending); each goes to the CTA with the smallest (load, CTA
            index); its load grows by cost.
  assignment ("snake", the device scheduler): the same sorted list dealt in
            rounds of `grid` items, CTA order 0..grid-1 in even rounds and
            grid-1..0 in odd rounds; a CTA's items keep their sorted order.

Packed metadata (int32), the layout the library's scheduler must reproduce
bit for bit:
  [0] 0x50414D31  [1] B  [2] Hk  [3] total_splits  [4] num_items  [5] grid
  [6] chunk  [7] ctas_per_sm
  n_splits[B], split_indptr[B+1], cta_indptr[grid+1],
  items[2 * num_items] as (b, (s << 16) | kvh) in per-CTA assignment order.
"""
from __future__ import annotations

import heapq

MAGIC = 0x50414D31
PAGE = 64
MAX_SPLITS = 64
ITEMS_PER_SHARE = 2
MIN_CHUNK = 4


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def split_counts(seq_lens, num_kv_heads: int, num_sms: int, ctas_per_sm: int,
                 forced_splits: int = 0):
    pages = [_cdiv(max(int(s), 0), PAGE) for s in seq_lens]
    units = sum(pages) * num_kv_heads
    cap = num_sms * ctas_per_sm
    chunk = max(MIN_CHUNK, _cdiv(units, cap * ITEMS_PER_SHARE))
    n = []
    for p in pages:
        if p <= 1:
            n.append(1)
        elif forced_splits > 0:
            n.append(min(forced_splits, p, MAX_SPLITS))
        else:
            n.append(min(_cdiv(p, chunk), MAX_SPLITS))
    return pages, n, chunk


def split_range(pages: int, nsplit: int, s: int):
    return (s * pages) // nsplit, ((s + 1) * pages) // nsplit


def schedule(seq_lens, num_kv_heads: int, num_sms: int, ctas_per_sm: int,
             forced_splits: int = 0, dealing: str = "lpt"):
    """Return the packed metadata as a list of Python ints."""
    B = len(seq_lens)
    pages, n, chunk = split_counts(seq_lens, num_kv_heads, num_sms, ctas_per_sm, forced_splits)
    indptr = [0]
    for x in n:
        indptr.append(indptr[-1] + x)
    items = []  # (cost, index, b, s, kvh)
    for b in range(B):
        for s in range(n[b]):
            lo, hi = split_range(pages[b], n[b], s)
            for kvh in range(num_kv_heads):
                items.append((hi - lo + 1, len(items), b, s, kvh))
    cap = num_sms * ctas_per_sm
    grid = min(len(items), cap)
    order = sorted(items, key=lambda it: (-it[0], it[1]))
    per_cta = [[] for _ in range(grid)]
    if dealing == "lpt":
        heap = [(0, c) for c in range(grid)]
        for cost, _, b, s, kvh in order:
            load, c = heapq.heappop(heap)
            per_cta[c].append((b, s, kvh))
            heapq.heappush(heap, (load + cost, c))
    elif dealing == "snake":
        for r, (cost, _, b, s, kvh) in enumerate(order):
            rnd, pos = divmod(r, grid)
            per_cta[pos if rnd % 2 == 0 else grid - 1 - pos].append((b, s, kvh))
    else:
        raise ValueError(dealing)
    out = [MAGIC, B, num_kv_heads, indptr[-1], len(items), grid, chunk, ctas_per_sm]
    out += n
    out += indptr
    cta_ptr = [0]
    for lst in per_cta:
        cta_ptr.append(cta_ptr[-1] + len(lst))
    out += cta_ptr
    for lst in per_cta:
        for b, s, kvh in lst:
            out += [b, (s << 16) | kvh]
    return out


def unpack(meta):
    """Split packed metadata into its named parts (for tests)."""
    B, hk, total, nitems, grid = meta[1], meta[2], meta[3], meta[4], meta[5]
    o = 8
    n = list(meta[o:o + B]); o += B
    indptr = list(meta[o:o + B + 1]); o += B + 1
    cta_ptr = list(meta[o:o + grid + 1]); o += grid + 1
    raw = list(meta[o:o + 2 * nitems]); o += 2 * nitems
    items = [(raw[2 * i], raw[2 * i + 1] >> 16, raw[2 * i + 1] & 0xFFFF) for i in range(nitems)]
    return dict(batch=B, num_kv_heads=hk, total_splits=total, num_items=nitems, grid=grid,
                chunk=meta[6], ctas_per_sm=meta[7], n_splits=n, split_indptr=indptr,
                cta_indptr=cta_ptr, items=items, length=o)


def static_split_capacity(batch: int, num_kv_heads: int, num_sms: int, ctas_per_sm: int, forced_splits: int = 0):
    """Most splits the rule can produce for `batch` sequences of any lengths:
    sum_b ceil(pages_b / chunk) <= sum_b pages_b / chunk + B <= ITEMS_PER_SHARE * cap / Hk + B."""
    if forced_splits > 0:
        return batch * min(forced_splits, MAX_SPLITS)
    cap = num_sms * ctas_per_sm
    return batch + _cdiv(ITEMS_PER_SHARE * cap, num_kv_heads)


def page_table_from_flat(kv_indices, kv_lens, page_size=64, columns=None):
    """Block table from a flat list of page ids (MATE msa_interface,
    _build_page_table_from_flat_kv_indices, with _page_counts): sequence b owns
    the next ceil(kv_lens[b] / page_size) ids of the list, in order, in the first
    columns of its row; every other entry is 0.  columns defaults to the largest
    page count (the page's table width).  Raises ValueError when the list does
    not hold exactly the implied number of ids, a length is negative, or a row
    does not fit in ``columns``.  Plain loops: test infrastructure only."""
    if page_size <= 0:
        raise ValueError("page_size must be positive")
    counts = []
    for n in kv_lens:
        n = int(n)
        if n < 0:
            raise ValueError("kv_lens must be >= 0")
        counts.append((n + page_size - 1) // page_size)
    if len(kv_indices) != sum(counts):
        raise ValueError("kv_indices does not match the page count implied by kv_lens")
    width = max(counts, default=0) if columns is None else int(columns)
    table = [[0] * width for _ in counts]
    start = 0
    for b, c in enumerate(counts):
        if c > width:
            raise ValueError("a sequence has more pages than the table has columns")
        for j in range(c):
            table[b][j] = int(kv_indices[start + j])
        start += c
    return table
