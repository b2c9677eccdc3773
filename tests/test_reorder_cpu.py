"""The library's host row reordering (bsp_reorder_rows) against the
oracle's subset DP (UnionSparse, "Grouped Subset Dynamic Programming"):
the exact solver returns the oracle's permutation and cost; the pairing
heuristic returns a valid permutation whose cost it reports correctly and
that is never worse than the identity grouping.  CPU only."""
import numpy as np
import pytest

import bitmap_encoded_unstructured_gb300 as bsp
from oracle import ie_bme as u


def _tile(H, KL, p, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(-8, 8, size=(H, KL)) * (rng.random((H, KL)) < p)).astype(np.int8)


@pytest.mark.parametrize("H,KL,RA,CA", [(8, 16, 2, 2), (12, 32, 2, 2), (16, 64, 2, 2), (9, 24, 3, 2),
                                        (12, 8, 4, 1), (16, 128, 2, 2)])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_exact_solver_matches_the_oracle(H, KL, RA, CA, seed):
    T = _tile(H, KL, 0.25, 100 * H + seed)
    perm, cost = bsp.bsp_reorder_rows(T, RA, CA, exact=True)
    operm, ocost = u.reorder_rows(T.astype(np.int64), RA, CA)
    assert cost == ocost
    np.testing.assert_array_equal(perm, operm)


@pytest.mark.parametrize("H,KL", [(8, 16), (16, 64)])
@pytest.mark.parametrize("seed", [4, 5, 6])
def test_pairing_heuristic_bounds(H, KL, seed):
    T = _tile(H, KL, 0.3, 10 * H + seed).astype(np.int64)
    perm, cost = bsp.bsp_reorder_rows(T, 2, 2, exact=False)
    assert sorted(perm.tolist()) == list(range(H))
    assert cost == u.union_active(T[perm], 2, 2)
    _, best = u.reorder_rows(T, 2, 2)
    assert best <= cost <= u.union_active(T, 2, 2)


@pytest.mark.parametrize("p", [0.05, 0.2, 0.5])
def test_pairing_heuristic_on_a_64_row_tile(p):
    """The tile size of the union format: a valid permutation, its reported
    cost, never above the identity grouping's."""
    T = _tile(64, 64, p, int(p * 100)).astype(np.int64)
    perm, cost = bsp.bsp_reorder_rows(T, 2, 2, exact=False)
    assert sorted(perm.tolist()) == list(range(64))
    assert cost == u.union_active(T[perm], 2, 2)
    assert cost <= u.union_active(T, 2, 2)


def test_pairing_finds_identical_rows():
    """Rows 2k and 2k + 1 identical, row i and i + 32 disjoint: the identity
    grouping activates the union of two patterns per logical row, the
    pairing of identical rows only one."""
    T = np.zeros((64, 64), dtype=np.int8)
    rng = np.random.default_rng(9)
    for k in range(32):
        pat = rng.random(64) < 0.3
        T[2 * k][pat] = 1
        T[2 * k + 1][pat] = 1
    perm, cost = bsp.bsp_reorder_rows(T, 2, 2, exact=False)
    groups = sorted((int(perm[i]), int(perm[32 + i])) for i in range(32))
    assert groups == [(2 * k, 2 * k + 1) for k in range(32)]
    assert cost < u.union_active(T.astype(np.int64), 2, 2)


def test_argument_errors():
    L = bsp.lib()
    import ctypes
    T = np.zeros((64, 64), dtype=np.int8)
    perm = np.zeros(64, dtype=np.int32)
    c = ctypes.c_int64()
    assert L.bsp_reorder_rows(T.ctypes.data, 64, 64, 2, 2, 1, perm.ctypes.data, ctypes.byref(c)) == 2  # exact, H > 20
    assert L.bsp_reorder_rows(T.ctypes.data, 64, 64, 4, 2, 0, perm.ctypes.data, ctypes.byref(c)) == 2  # heuristic, RA != 2
    assert L.bsp_reorder_rows(T.ctypes.data, 63, 64, 2, 2, 0, perm.ctypes.data, ctypes.byref(c)) == 2  # RA does not divide H
    assert L.bsp_reorder_rows(None, 8, 8, 2, 2, 1, perm.ctypes.data, ctypes.byref(c)) == 1
