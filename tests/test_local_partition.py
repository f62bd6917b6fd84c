"""The chunk-local attention kernel's work partition, restated on the CPU: for
every visible-key count and split count, the (split, warp, tile) assignment
covers each 16-key tile of the query's visible keys exactly once, every tile a
warp issues lies inside its split's key range, and the clamped copy key of a
tile's last rows stays below the range end (so a copy never reads past the
visible keys)."""
import pytest

TILE, WARPS = 16, 4


def partition(visible, ns):
    T = (visible + TILE - 1) // TILE
    per = (T + ns - 1) // ns
    tiles = []
    for rank in range(ns):
        tile0 = min(T, rank * per)
        tile1 = min(T, tile0 + per)
        kend = min(visible, tile1 * TILE)
        for warp in range(WARPS):
            n_mine = (tile1 - tile0 - warp + WARPS - 1) // WARPS if tile1 - tile0 > warp else 0
            for n in range(n_mine):
                tile = tile0 + warp + n * WARPS
                key0 = tile * TILE
                assert tile0 <= tile < tile1
                assert key0 < kend                        # at least one visible key in the tile
                assert min(key0 + TILE - 1, kend - 1) < visible
                tiles.append(tile)
    return T, tiles


@pytest.mark.parametrize("ns", [1, 2, 4, 8])
def test_tiles_cover_visible_keys_once(ns):
    for visible in range(0, 700):
        T, tiles = partition(visible, ns)
        assert sorted(tiles) == list(range(T)), (visible, ns)
