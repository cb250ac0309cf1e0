"""Query-row partition of one sequence across GPUs: coverage and balance
(host logic; the per-row independence it relies on is the one of the blog's
section "Three attention types, interleaved": each query reads its own keys)."""
import pytest

from sparse_compressed_attention_gb300 import rows as R

CSA = dict(ratio=4, topk=512, window=128)
HCA = dict(ratio=128, topk=0, window=128)


@pytest.mark.parametrize("S,n", [(1, 1), (7, 3), (16384, 16), (16385, 16), (5, 8)])
def test_chunk_bounds_cover_once_with_near_equal_sizes(S, n):
    ch = R.chunk_bounds(S, n)
    assert ch[0][0] == 0 and ch[-1][1] == S
    assert all(a1 == b0 for (_, b0), (a1, _) in zip(ch, ch[1:]))
    sizes = [b - a for a, b in ch]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("S,world", [(16384, 1), (16384, 2), (16384, 8), (3001, 4), (6, 4), (1, 2)])
def test_zigzag_covers_every_row_exactly_once(S, world):
    seen = []
    for r in range(world):
        for a, b in R.zigzag_chunks(S, world, r, R.layer_cost(**CSA) if world % 2 == 0 else None):
            assert 0 <= a < b <= S
            seen.extend(range(a, b))
    assert sorted(seen) == list(range(S))


def test_zigzag_pairs_chunk_r_with_its_mirror():
    ch = R.chunk_bounds(1600, 8)
    assert R.zigzag_chunks(1600, 4, 1) == [ch[1], ch[6]]
    assert R.zigzag_chunks(1600, 1, 0) == [(0, 1600)]


def test_zigzag_balances_affine_work_exactly():
    S, world = 4096, 4                         # 2 * world divides S
    loads = [sum(3 + 5 * t for a, b in R.zigzag_chunks(S, world, r) for t in range(a, b)) for r in range(world)]
    assert len(set(loads)) == 1


@pytest.mark.parametrize("layer", [CSA, HCA])
@pytest.mark.parametrize("world", [2, 4, 8])
def test_cost_balanced_zigzag_evens_layer_work(layer, world):
    S = 16384
    cost = R.layer_cost(**layer)
    zz = [R.work_of(R.zigzag_chunks(S, world, r, cost), cost) for r in range(world)]
    assert max(zz) / min(zz) - 1 < 0.002
    # equal-size chunks leave CSA's saturating attention work uneven, and a
    # contiguous split leaves the last rank with every long row
    eq = [R.work_of(R.zigzag_chunks(S, world, r), cost) for r in range(world)]
    cont = [R.work_of([c], cost) for c in R.chunk_bounds(S, world)]
    assert max(cont) / min(cont) > max(eq) / min(eq) > max(zz) / min(zz)


def test_cost_bounds_cover_and_split_total_evenly():
    cost = R.layer_cost(**CSA)
    ch = R.cost_bounds(3001, 6, cost)
    assert ch[0][0] == 0 and ch[-1][1] == 3001 and all(a1 == b0 for (_, b0), (a1, _) in zip(ch, ch[1:]))
    parts = [R.work_of([c], cost) for c in ch]
    big = max(cost(t) for t in range(3001))
    assert max(parts) - min(parts) <= 2 * big


def test_row_work_counts_the_pages_keys():
    # CSA at t far past 4 * 512: 512 selected entries + 128 window keys
    t = 8191
    assert R.row_flops(t, 4, 512, 128) == 2 * 64 * 128 * 2048 + 4 * 64 * 512 * 640
    # HCA: every visible entry plus the window, no indexer
    assert R.row_flops(1279, 128, 0, 128) == 4 * 64 * 512 * (10 + 128)
    assert R.row_bytes(128, 0) == 2 * 64 * 512 * 2


@pytest.mark.parametrize("layer", [CSA, HCA])
@pytest.mark.parametrize("world", [1, 2, 8])
def test_contiguous_cost_split_covers_once_and_balances(layer, world):
    S = 16384
    cost = R.layer_cost(**layer)
    parts = [R.contiguous_chunks(S, world, r, cost) for r in range(world)]
    seen = [t for ch in parts for a, b in ch for t in range(a, b)]
    assert seen == list(range(S))                   # in rank order, each row once
    loads = [R.work_of(ch, cost) for ch in parts]
    assert max(loads) / min(loads) - 1 < 0.002


def test_tile_cost_charges_ragged_tiles_in_full():
    # 5 selected entries and a window cut to 21 tokens: two 128-key tiles
    assert R.row_tile_flops(20, 4, 512, 128) == 2 * 64 * 128 * 5 + 4 * 64 * 512 * 128 * 2
    # a full selection and window: the same as the exact count
    assert R.row_tile_flops(8191, 4, 512, 128) == R.row_flops(8191, 4, 512, 128)
    c = R.layer_cost(4, 512, 128, tile=128)
    assert c(20) > R.layer_cost(4, 512, 128)(20)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        R.zigzag_chunks(10, 2, 2)
    with pytest.raises(ValueError):
        R.chunk_bounds(0, 1)
