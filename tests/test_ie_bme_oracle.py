"""Pins of the IE-BME oracle (UnionSparse, "IE-BME" and "LSPD") against
what the page fixes: its worked union words and stream example, its LSPD
segment example, and brute force on small inputs.  CPU only."""
import numpy as np
import pytest

from oracle import ie_bme as u

# UnionSparse, "IE-BME Storage Layout" (Fig. 7): a 2 x 2 partition whose four
# logical mask rows of 16 positions pack, leftmost position in the LSB, to
# these words; each has ten active bits, P_t = 40 and Q * P_t = 160.
FIG7_ROWS = [0x36DB, 0x6DB6, 0x5B6D, 0xB6DA]


def _fig7_weight():
    """An 8 x 32 LT (areas of 4 x 16) whose area 0 is active exactly at the
    Fig. 7 positions (value 1) and whose other areas are zero."""
    W = np.zeros((8, 32), dtype=np.int64)
    for r, word in enumerate(FIG7_ROWS):
        for c in range(16):
            if (word >> c) & 1:
                W[r, c] = 1
    return W


def test_fig7_union_words_counts_and_offset():
    for word in FIG7_ROWS:
        assert bin(word).count("1") == 10
    enc = u.union_encode(_fig7_weight(), 4, lt=(8, 32), areas=(2, 2))
    expect = FIG7_ROWS[0] | FIG7_ROWS[1] << 16 | FIG7_ROWS[2] << 32 | FIG7_ROWS[3] << 48
    assert enc["masks"].tolist() == [expect]
    assert enc["offsets"].tolist() == [0, 160]
    # area 0's stream holds the forty ones; areas 1-3 keep their zeros so that
    # one rank indexes all four streams
    assert enc["values"][:40].tolist() == [1] * 40
    assert enc["values"][40:].tolist() == [0] * 120


def test_group_keeps_area_zero_and_empty_group_emits_nothing():
    """The red-framed group [1, 30, 59, 0]: one active bit, each area appends
    its value at the same rank, the zero included (int8 payloads: 30 and 59
    do not fit int4).  An all-zero group emits nothing."""
    W = np.zeros((8, 32), dtype=np.int64)   # areas 4 x 16: (0,0) (0,16) (4,0) (4,16)
    i, j = 2, 5
    W[i, j], W[i, 16 + j], W[4 + i, j], W[4 + i, 16 + j] = 1, 30, 59, 0
    enc = u.union_encode(W, 8, lt=(8, 32), areas=(2, 2))
    assert enc["masks"].tolist() == [1 << (16 * i + j)]
    assert enc["offsets"].tolist() == [0, 4]
    assert enc["values"].tolist() == [1, 30, 59, 0]
    Z = u.union_encode(np.zeros((8, 32), dtype=np.int64), 8, lt=(8, 32), areas=(2, 2))
    assert Z["masks"].tolist() == [0] and Z["offsets"].tolist() == [0, 0] and Z["values"].size == 0


def test_lspd_segment_example():
    """LSPD, Fig. 9(c): segment 10110100 written leftmost first has active
    positions 0, 2, 3, 5, which take the consecutive indices b..b+3."""
    seg = 0b00101101
    b = 77
    assert u.lspd_indices(seg, 8, b) == [(0, b), (2, b + 1), (3, b + 2), (5, b + 3)]


def test_lspd_matches_the_encoder_ranks():
    """The segment's values sit at consecutive ranks of every stream, after
    the active positions of the preceding segment."""
    W = np.zeros((64, 64), dtype=np.int64)      # default LT, areas of 32 x 32
    W[0, 3] = 5                                  # one active position before the segment
    for p in (0, 2, 3, 5):
        W[0, 8 + p] = 10 + p                     # area 0, row 0, segment 1
        W[32, 8 + p] = -(10 + p)                 # area 2, same positions
    enc = u.union_encode(W, 8)
    P = int(enc["offsets"][1]) // 4
    assert P == 5
    for (p, idx) in u.lspd_indices(0b00101101, 8, 1):
        assert enc["values"][0 * P + idx] == 10 + p
        assert enc["values"][2 * P + idx] == -(10 + p)
        assert enc["values"][1 * P + idx] == 0 and enc["values"][3 * P + idx] == 0


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,s", [(64, 64, 0.5), (130, 200, 0.6), (1, 8, 0.0), (256, 128, 0.9), (64, 192, 1.0)])
def test_round_trip_and_union_property(bits, M, K, s):
    rng = np.random.default_rng(M * 1000 + K + bits)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1))
    W = rng.integers(lo, hi, size=(M, K)) * (rng.random((M, K)) >= s)
    enc = u.union_encode(W, bits)
    np.testing.assert_array_equal(u.union_decode(enc), W)
    # every active position has a nonzero in some area, every inactive none
    Wp = np.zeros((enc["Mp"], enc["Kp"]), dtype=np.int64)
    Wp[:M, :K] = W
    words = enc["masks"].astype("<u8").view(np.uint8)
    bitsarr = np.unpackbits(words, bitorder="little").astype(bool).reshape(-1, 32, 32)
    t = 0
    for ti in range(enc["Mp"] // 64):
        for tj in range(enc["Kp"] // 64):
            tile = Wp[ti * 64:(ti + 1) * 64, tj * 64:(tj + 1) * 64]
            any_nz = (tile[:32, :32] != 0) | (tile[:32, 32:] != 0) | (tile[32:, :32] != 0) | (tile[32:, 32:] != 0)
            np.testing.assert_array_equal(bitsarr[t], any_nz)
            t += 1


@pytest.mark.parametrize("bits", [4, 8])
def test_packed_values_and_storage(bits):
    rng = np.random.default_rng(bits)
    W = rng.integers(-(1 << (bits - 1)), 1 << (bits - 1), size=(128, 320)) * (rng.random((128, 320)) < 0.5)
    enc = u.union_encode(W, bits)
    packed = u.pack_values(enc["values"], bits)
    total = int(enc["offsets"][-1])
    assert packed.size == (total * bits + 7) // 8
    if bits == 4:   # low nibble first, two's complement
        nib = np.stack([packed & 0xF, packed >> 4], axis=1).reshape(-1)[:total].astype(np.int64)
        np.testing.assert_array_equal(np.where(nib >= 8, nib - 16, nib), enc["values"])
    else:
        np.testing.assert_array_equal(packed.view(np.int8), enc["values"])
    nlt = (128 // 64) * (320 // 64)
    assert u.storage_bytes(enc) == 4 * (nlt + 1) + 8 * 16 * nlt + packed.size


def test_product_by_brute_force():
    rng = np.random.default_rng(7)
    W = rng.integers(-8, 8, size=(7, 9)) * (rng.random((7, 9)) < 0.5)
    X = rng.integers(-8, 8, size=(3, 9))
    Y = u.union_spmm(u.union_decode(u.union_encode(W, 4)), X)
    for n in range(3):
        for m in range(7):
            assert Y[n, m] == sum(int(W[m, k]) * int(X[n, k]) for k in range(9))


def test_out_of_range_values_rejected():
    with pytest.raises(ValueError):
        u.union_encode(np.full((64, 64), 8), 4)
    u.union_encode(np.zeros((64, 64)), 4, lt=(64, 64), areas=(4, 4))      # 16 x 16 = 256 bits: whole words
    with pytest.raises(ValueError):
        u.union_encode(np.zeros((8, 8)), 4, lt=(8, 8), areas=(2, 2))        # 4 x 4 = 16 bits: not whole words


# ---------------------------------------------------------------- row reordering

def _all_groupings(rows, RA):
    """Every partition of `rows` into groups of RA (brute force)."""
    from itertools import combinations
    if not rows:
        yield []
        return
    r0, rest = rows[0], rows[1:]
    for others in combinations(rest, RA - 1):
        g = (r0,) + others
        remaining = [r for r in rest if r not in others]
        for tail in _all_groupings(remaining, RA):
            yield [g] + tail


@pytest.mark.parametrize("H,KL,RA,CA,seed", [(6, 8, 2, 2, 1), (8, 8, 2, 1, 2), (8, 16, 2, 2, 3),
                                             (6, 6, 3, 1, 4), (9, 12, 3, 2, 5)])
def test_reorder_dp_is_the_brute_force_optimum(H, KL, RA, CA, seed):
    """The subset DP reaches the minimum of the grouped cost over every
    partition of the rows, and its permutation realizes that cost."""
    rng = np.random.default_rng(seed)
    T = (rng.random((H, KL)) < 0.35).astype(np.int64)
    cost = u.group_costs_table(T, RA, CA)
    best = min(sum(cost[tuple(sorted(g))] for g in part) for part in _all_groupings(list(range(H)), RA))
    perm, c = u.reorder_rows(T, RA, CA)
    assert c == best
    assert sorted(perm.tolist()) == list(range(H))
    assert u.union_active(T[perm], RA, CA) == best
    assert u.union_active(T, RA, CA) >= best


def test_reorder_canonical_form():
    """Rows ascending inside each group, groups in lexicographic order,
    permutation taken partition-wise."""
    rng = np.random.default_rng(11)
    T = (rng.random((8, 8)) < 0.3).astype(np.int64)
    perm, _ = u.reorder_rows(T, 2, 2)
    h = 4
    groups = [(int(perm[i]), int(perm[h + i])) for i in range(h)]
    assert all(a < b for a, b in groups)
    assert groups == sorted(groups)


def test_reorder_pairs_identical_rows():
    """Rows i and i + 4 of an 8-row tile are complementary, rows 2k and
    2k + 1 identical: the identity grouping activates every column, the
    optimum pairs the identical rows (cost = their own activity)."""
    T = np.zeros((8, 8), dtype=np.int64)
    pats = [0b00000011, 0b00001100, 0b00110000, 0b11000000]
    for k in range(4):
        for r in (2 * k, 2 * k + 1):
            for c in range(8):
                T[r, c] = (pats[k] >> c) & 1
    perm, c = u.reorder_rows(T, 2, 1)
    assert c == 4 * 2 and u.union_active(T, 2, 1) > c
    assert perm.tolist() == [0, 2, 4, 6, 1, 3, 5, 7]


@pytest.mark.parametrize("bits", [4, 8])
def test_permuted_encoding_round_trip(bits):
    """An encoding with per-LT row permutations decodes to the original
    matrix, and its union count equals the permuted tiles' activity."""
    rng = np.random.default_rng(bits + 20)
    lo, hi = -(1 << (bits - 1)), 1 << (bits - 1)
    W = rng.integers(lo, hi, size=(128, 192)) * (rng.random((128, 192)) < 0.3)
    perms = [rng.permutation(64) for _ in range(2 * 3)]
    enc = u.union_encode(W, bits, perms=perms)
    np.testing.assert_array_equal(u.union_decode(enc), W)
    t = 0
    for ti in range(2):
        for tj in range(3):
            tile = W[ti * 64:(ti + 1) * 64, tj * 64:(tj + 1) * 64][perms[t]]
            assert int(enc["offsets"][t + 1] - enc["offsets"][t]) == 4 * u.union_active(tile, 2, 2)
            t += 1


def test_pmr_of_the_fig7_example():
    """UnionSparse's PMR for the Fig. 7 LT in W4: 40 nonzeros are 20 payload
    bytes; the LT stores 2 offsets (8 B), one mask word (8 B) and 160 int4
    values (80 B), so the rest is 96 - 20 = 76 bytes."""
    enc = u.union_encode(_fig7_weight(), 4, lt=(8, 32), areas=(2, 2))
    assert enc["nnz"] == 40
    assert u.storage_bytes(enc) == 96
    assert u.payload_to_metadata(enc) == 20 / 76
    # W8: 40 payload bytes of 8 + 8 + 160
    enc8 = u.union_encode(_fig7_weight(), 8, lt=(8, 32), areas=(2, 2))
    assert u.payload_to_metadata(enc8) == 40 / (176 - 40)
