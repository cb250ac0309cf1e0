"""Query-row partition of one sequence across GPUs (host logic only).

Every query row of the compressed attention is independent once the
compressed pools exist: a query reads its own selected entries and its own
128-token window ("Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X
GPUs with Primus", section "Three attention types, interleaved").  So one
sequence splits across GPUs by query rows, each GPU holding the whole causal
prefix of the key/value side (the compressor is cheap and runs over the
prefix a GPU needs) and computing only its own rows; no collective touches the
data path.

Causal work per row grows with the position (the indexer scores every visible
entry, HCA attends to every visible entry) and saturates for CSA attention
(at most K selected entries), so equal contiguous splits are unbalanced.  The
zig-zag split cuts the sequence into 2*world chunks of equal cost (boundaries
at equal quantiles of the running per-row cost) and gives rank r chunks r and
2*world-1-r, which also evens out what the cost model leaves over.
"""
from __future__ import annotations

import bisect
import itertools

# flop-equivalent of one HBM byte: the bf16 tensor peak over the copy
# bandwidth of the GPU (1932.6 TFLOP/s / 6779 GB/s measured on GB300)
FLOP_PER_BYTE = 285.0


def chunk_bounds(S, n):
    """Boundaries of n near-equal contiguous chunks of [0, S) (sizes differ by at most one)."""
    if S < 1 or n < 1:
        raise ValueError("S and n must be >= 1")
    base, extra = divmod(S, n)
    out, a = [], 0
    for i in range(n):
        b = a + base + (1 if i < extra else 0)
        out.append((a, b))
        a = b
    return out


def cost_bounds(S, n, cost):
    """Boundaries of n contiguous chunks of [0, S) with near-equal total cost:
    chunk i ends at the first position where the running cost reaches
    (i+1)/n of the total.  Chunks may be empty when a few rows carry most of
    the cost."""
    if S < 1 or n < 1:
        raise ValueError("S and n must be >= 1")
    pref = list(itertools.accumulate(float(cost(t)) for t in range(S)))
    total = pref[-1]
    cuts = [0]
    for i in range(1, n):
        cuts.append(max(cuts[-1], bisect.bisect_left(pref, total * i / n) + 1 if total > 0 else S * i // n))
    cuts.append(S)
    return [(cuts[i], cuts[i + 1]) for i in range(n)]


def zigzag_chunks(S, world, rank, cost=None):
    """Query-position ranges [a, b) of `rank` among `world` GPUs.

    world == 1 keeps the sequence whole.  Otherwise rank r takes chunks r and
    2*world-1-r of 2*world chunks, of equal size (cost None) or of equal
    cost (cost: position -> work of that query row); empty chunks are dropped.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if world == 1:
        return [(0, S)]
    ch = chunk_bounds(S, 2 * world) if cost is None else cost_bounds(S, 2 * world, cost)
    picked = [ch[rank], ch[2 * world - 1 - rank]]
    return [(a, b) for a, b in picked if b > a]


def contiguous_chunks(S, world, rank, cost):
    """One contiguous range per rank, boundaries at equal quantiles of the
    per-row cost: one call per layer per rank (the zig-zag split makes two,
    each running the compressor over its own prefix)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    a, b = cost_bounds(S, world, cost)[rank]
    return [(a, b)] if b > a else []


def row_flops(t, ratio, topk, window, heads=64, dim=512, idx_heads=64, idx_dim=128):
    """FLOPs of query position t in one layer: the indexer products over its
    visible entries (CSA) and the attention products over its keys."""
    nv = (t + 1) // ratio if ratio > 0 else 0
    ent = (min(nv, topk) if topk > 0 else nv) if ratio > 0 else 0
    win = t + 1 if window < 0 else min(t + 1, window)
    idx = 2 * idx_heads * idx_dim * nv if (ratio > 0 and topk > 0) else 0
    return idx + 4 * heads * dim * (ent + win)


def row_bytes(ratio, topk, heads=64, dim=512, idx_heads=64, idx_dim=128):
    """HBM bytes of one query row: q read and o written (bf16), and for CSA the
    indexer query, its weights and the selection."""
    b = 2 * heads * dim * 2
    if ratio > 0 and topk > 0:
        b += idx_heads * idx_dim * 2 + idx_heads * 4 + topk * 4
    return b


def row_tile_flops(t, ratio, topk, window, tile=128, heads=64, dim=512, idx_heads=64, idx_dim=128):
    """row_flops with the attention keys rounded up to whole key tiles: the
    tensor-core attention runs a ragged tile (a short selection, a window cut
    by the sequence start) as a full one."""
    nv = (t + 1) // ratio if ratio > 0 else 0
    ent = (min(nv, topk) if topk > 0 else nv) if ratio > 0 else 0
    win = t + 1 if window < 0 else min(t + 1, window)
    idx = 2 * idx_heads * idx_dim * nv if (ratio > 0 and topk > 0) else 0
    tiles = -(-ent // tile) + -(-win // tile)
    return idx + 4 * heads * dim * tile * tiles


def layer_cost(ratio, topk, window, flop_per_byte=FLOP_PER_BYTE, tile=None, **shape):
    """Per-row cost of one layer in flop-equivalents: its FLOPs (attention keys
    rounded to whole tiles when `tile` is given) plus its HBM bytes at the
    machine balance."""
    rb = row_bytes(ratio, topk, **shape) * flop_per_byte
    if tile:
        return lambda t: row_tile_flops(t, ratio, topk, window, tile=tile, **shape) + rb
    return lambda t: row_flops(t, ratio, topk, window, **shape) + rb


def work_of(chunks, cost):
    """Total cost of a list of [a, b) ranges."""
    return sum(cost(t) for a, b in chunks for t in range(a, b))
