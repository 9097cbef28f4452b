"""The step-row tables the library builds at la_create (positions, the
in-step visibility words, the rows whose logits are read), read through
la_step_tables on the CPU and compared with the oracle.  The library walks
parent pointers; the oracle's mask comes from its closed-form visibility
rule (oracle.lookahead.sees), so the two constructions are independent."""
import numpy as np
import pytest

from helpers import ensure_built
from oracle import lookahead as la

# (N, W, G): the pages' configurations and edge cases (no candidates, one
# column, a single level, the largest step the tables hold)
CONFIGS = [(2, 1, 0), (2, 10, 10), (3, 4, 4), (4, 5, 3), (4, 4, 4), (5, 7, 7), (5, 15, 15), (7, 3, 2),
           (8, 5, 5), (5, 1, 0), (3, 1, 7), (9, 16, 15)]


@pytest.fixture(scope="module")
def tables():
    ensure_built()
    from exact_decoding_gb300 import la_step_tables
    return la_step_tables


def unpack(vis, M):
    return np.array([[(int(vis[r, s // 32]) >> (s % 32)) & 1 for s in range(M)] for r in range(M)], dtype=bool)


@pytest.mark.parametrize("N,W,G", CONFIGS)
def test_tables_match_oracle(tables, N, W, G):
    depth, vis, used = tables(N, W, G)
    M = 1 + (W + G) * (N - 1)
    assert len(depth) == M and vis.shape == (M, 8)
    rows = la.step_rows(N, W, G)
    assert list(depth) == [r.depth for r in rows]
    assert np.array_equal(unpack(vis, M), la.step_mask(N, W, G))
    assert list(used) == la.used_rows(N, W, G)
    for r in range(M):                                   # nothing past the step's rows
        assert all(((int(vis[r, s // 32]) >> (s % 32)) & 1) == 0 for s in range(M, 256))


def test_capacity_and_arguments(tables):
    from exact_decoding_gb300 import LaError
    with pytest.raises(LaError):
        tables(1, 4, 4)                                  # N >= 2
    with pytest.raises(LaError):
        tables(9, 20, 20)                                # 1 + 40 * 8 = 321 rows > 256
