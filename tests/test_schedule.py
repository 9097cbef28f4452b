"""The projection GEMMs' work split, read from the library's own host code
(la_gemm_schedule; no GPU needed).  The fused gate/up epilogue relies on
these properties: every (tile, k-unit) is covered exactly once, a tile's
planes are numbered 0 .. np - 1 in CTA order, the work per CTA is even, and
with the whole-tiles-first split a whole tile is one segment (one plane)
and every CTA's split pieces come before its whole tiles, so no CTA waits
for a piece that another CTA has not yet published."""
import numpy as np
import pytest

from helpers import ensure_built

# (tiles, k-units, CTAs): the step gate/up GEMMs of the 7B, 13B and 70B shapes
# (pair tiles of 128 features, 128-column k units), the small test models,
# and plain stream-K shapes (QKV, O, down of the 7B shape).
SHAPES = [(86, 32, 76), (108, 40, 76), (224, 64, 76), (6, 2, 76), (8, 4, 76), (11, 4, 76),
          (48, 32, 76), (16, 32, 76), (16, 86, 76), (250, 32, 76), (1, 1, 1), (3, 7, 5)]


@pytest.fixture(scope="module")
def sched():
    ensure_built()
    from exact_decoding_gb300 import la_gemm_schedule
    return la_gemm_schedule


def check_common(segs, first, planes, tiles, n_kb):
    cover = np.zeros((tiles, n_kb), dtype=np.int32)
    seen = [[] for _ in range(tiles)]
    for t, k0, k1, pl in segs:
        assert 0 <= t < tiles and 0 <= k0 < k1 <= n_kb
        cover[t, k0:k1] += 1
        seen[t].append(pl)
    assert np.all(cover == 1)
    for t in range(tiles):
        assert seen[t] == list(range(planes[t]))          # plane p = the tile's p-th segment in CTA order
    assert first[0] == 0 and first[-1] == len(segs) and np.all(np.diff(first) >= 0)
    work = [int(sum(k1 - k0 for _, k0, k1, _ in segs[first[c]:first[c + 1]])) for c in range(len(first) - 1)]
    assert max(work) - min(work) <= 1                      # even split, +-1 k-unit
    assert sum(work) == tiles * n_kb
    return work


@pytest.mark.parametrize("tiles,n_kb,ctas", SHAPES)
def test_stream_k_split(sched, tiles, n_kb, ctas):
    segs, first, planes = sched(tiles, n_kb, ctas, False)
    check_common(segs, first, planes, tiles, n_kb)
    assert len(first) - 1 == min(ctas, tiles * n_kb)      # never more CTAs than k-units


@pytest.mark.parametrize("tiles,n_kb,ctas", SHAPES)
def test_whole_tiles_first_split(sched, tiles, n_kb, ctas):
    segs, first, planes = sched(tiles, n_kb, ctas, True)
    check_common(segs, first, planes, tiles, n_kb)
    whole = tiles // ctas
    if whole == 0:                                          # fewer tiles than CTAs: plain stream-K
        ref = sched(tiles, n_kb, ctas, False)
        assert all(np.array_equal(a, b) for a, b in zip((segs, first, planes), ref))
        return
    for c in range(ctas):
        run = segs[first[c]:first[c + 1]]
        mine = [t for t, k0, k1, _ in run if k0 == 0 and k1 == n_kb and t < whole * ctas]
        assert mine == list(range(c * whole, (c + 1) * whole))   # its own whole tiles, last in its run
        split = [t for t, *_ in run if t >= whole * ctas]
        kinds = [t >= whole * ctas for t, *_ in run]
        assert kinds == sorted(kinds, reverse=True)       # split pieces before whole tiles
        assert len(split) + len(mine) == len(run)
    assert np.all(planes[:whole * ctas] == 1)


def test_step_gate_up_shapes_mostly_whole(sched):
    """At the 7B shape 76 of the 86 gate/up pair tiles need no partial planes."""
    _, _, planes = sched(86, 32, 76, True)
    assert int(np.sum(planes == 1)) == 76 and int(planes.max()) <= 9


def test_rejects_bad_sizes(sched):
    from exact_decoding_gb300 import LaError
    with pytest.raises(LaError):
        sched(0, 4, 4, False)
