"""Pins of the Tiled-CBC oracle (SPDP section 4.1) against facts fixed by
the page and by hand counts, not by the oracle itself.  CPU only."""
import numpy as np
import pytest

from oracle import tiled_cbc as cbc
from bitmap_encoded_unstructured_gb300 import synth


def test_hand_example_one_gtile():
    """One 256 x 64 GTile with nonzeros counted by hand: column 0 holds rows
    3, 64 and 255; column 1 is empty; column 5 holds row 0.  Tile-column
    order gives values [a, b, c, d]; ColInfo packs (start << 16) | nnz:
    column 0 -> (0, 3), column 1 -> (3, 0), columns 2-4 -> (3, 0), column 5
    -> (3, 1), the rest (4, 0); the bitmap words of column 0 are bit 3 of
    word 0, bit 0 of word 1 and bit 63 of word 3."""
    W = np.zeros((256, 64), dtype=np.uint16)
    W[3, 0], W[64, 0], W[255, 0], W[0, 5] = 0x3C00, 0x4000, 0x4200, 0xBC00
    e = cbc.encode(W)
    assert e["NGT"] == 1 and e["NNZ"] == 4
    assert e["values"].tolist() == [0x3C00, 0x4000, 0x4200, 0xBC00]
    assert e["offsets"].tolist() == [0, 4]
    info = e["colinfo"].tolist()
    assert info[0] == (0 << 16) | 3 and info[1] == (3 << 16) | 0 and info[5] == (3 << 16) | 1
    assert all(v == (4 << 16) for v in info[6:])
    words = e["bitmaps"][:4].tolist()
    assert words == [1 << 3, 1 << 0, 0, 1 << 63]
    assert e["bitmaps"][5 * 4:5 * 4 + 4].tolist() == [1, 0, 0, 0]


def test_storage_closed_form_counted_by_hand():
    """Stor = 4 (NGT + 1) + 4 NGT TILE_K + 8 NBM + 2 NNZ: a 512 x 128 fp16
    matrix is 2 x 2 GTiles (NGT = 4), NBM = 512 * 128 / 64 = 1024; with 10
    nonzeros that is 20 + 1024 + 8192 + 20 = 9256 bytes, and the arrays'
    sizes add up to the same."""
    W = np.zeros((512, 128), dtype=np.uint16)
    idx = [(0, 0), (1, 0), (300, 7), (511, 127), (256, 64), (5, 70), (6, 70), (7, 70), (400, 3), (100, 100)]
    for r, c in idx:
        W[r, c] = 0x3C00
    e = cbc.encode(W)
    assert cbc.storage_bytes(e) == 4 * 5 + 4 * 4 * 64 + 8 * 1024 + 2 * 10 == 9256
    assert (e["offsets"].nbytes + e["colinfo"].nbytes + e["bitmaps"].nbytes + e["values"].nbytes) == 9256


@pytest.mark.parametrize("M,K,s", [(256, 64, 0.5), (300, 130, 0.3), (512, 192, 0.7), (256, 128, 0.0)])
def test_round_trip_and_counts(M, K, s):
    W = synth.weights_f16(M, K, s, "uniform" if s else "none", 11 + M + K)
    e = cbc.encode(W)
    np.testing.assert_array_equal(cbc.decode(e), W)
    assert e["NNZ"] == int(np.count_nonzero(W))
    pops = sum(bin(int(w)).count("1") for w in e["bitmaps"])
    assert pops == e["NNZ"] == int(sum(int(v) & 0xFFFF for v in e["colinfo"]))
    # starts are the prefix sums of the column counts inside each GTile
    ci = e["colinfo"].reshape(-1, cbc.TILE_K).astype(np.int64)
    starts, counts = ci >> 16, ci & 0xFFFF
    np.testing.assert_array_equal(starts[:, 1:], np.cumsum(counts, axis=1)[:, :-1])
    assert np.all(starts[:, 0] == 0)


def test_values_of_one_column_are_contiguous_and_top_down():
    """The page's point: a column's nonzeros sit together, so a product that
    skips a column skips one contiguous span.  Column c of GTile t occupies
    [TileOffset[t] + start, + nnz) and lists its rows top to bottom."""
    W = synth.weights_f16(512, 128, 0.5, "uniform", 5)
    e = cbc.encode(W)
    for t in range(e["NGT"]):
        gi, gj = divmod(t, 2)
        for c in (0, 17, 63):
            info = int(e["colinfo"][t * 64 + c])
            base = int(e["offsets"][t]) + (info >> 16)
            col = W[gi * 256:(gi + 1) * 256, gj * 64 + c]
            np.testing.assert_array_equal(e["values"][base:base + (info & 0xFFFF)], col[col != 0])


def test_int8_and_fetch_accounting():
    """int8 stores one byte per value; the column-skipping product fetches
    every GTile's ColInfo and only the active columns' bitmaps and values:
    with every activation zero that is the ColInfo alone, with all active it
    is the whole index but the TileOffset array."""
    W = synth.weights_i8(256, 128, 0.5, 3)
    e = cbc.encode(W)
    assert e["values"].dtype == np.int8 and e["elem_bytes"] == 1
    none = cbc.fetched_bytes(e, np.zeros(128, dtype=bool))
    allb = cbc.fetched_bytes(e, np.ones(128, dtype=bool))
    assert none == 4 * e["NGT"] * 64
    assert allb == cbc.storage_bytes(e) - 4 * (e["NGT"] + 1)


def test_fetch_accounting_partial_activity_by_brute_force():
    """A partial activation pattern on a 2 x 3 grid of GTiles (K = 150, so
    the third GTile column is ragged): the bytes the column-skipping product
    reads, counted from the dense W alone.  Each GTile contributes its 64
    ColInfo words; each active column k of GTile row gi adds its four bitmap
    words and the nonzeros of W[256 gi : 256 (gi + 1), k].  The two GTile
    rows have different densities, so charging a column to the wrong GTile
    (a row-for-column slip in the tiling) changes the total."""
    M, K = 512, 150
    W = synth.weights_f16(M, K, 0.5, "uniform", 11)
    W[256:, :] = np.where(np.arange(K) % 3 == 0, W[256:, :], 0).astype(np.uint16)
    rng = np.random.default_rng(12)
    x_active = rng.random(K) < 0.3
    e = cbc.encode(W)
    assert e["NGT"] == 6
    expect = 4 * 6 * 64
    for gi in range(2):
        for k in range(K):
            if x_active[k]:
                expect += 8 * 4 + 2 * int(np.count_nonzero(W[256 * gi:256 * (gi + 1), k]))
    assert cbc.fetched_bytes(e, x_active) == expect
    # the columns of the zero padding past K never count as active
    act = cbc.active_columns(x_active, e)
    assert act.shape == (6 * 64,)
    assert not act.reshape(2, 3, 64)[:, 2, K - 128:].any()
    assert (act.reshape(2, 3, 64)[0].reshape(-1)[:K] == x_active).all()
    assert (act.reshape(2, 3, 64)[1].reshape(-1)[:K] == x_active).all()
