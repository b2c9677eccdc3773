"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test holds one part of the oracle against something it does not
compute itself: a worked example printed on the pages (tests/golden/), a
closed form, a library routine (numpy's fp16 conversion, matmul and
popcount), or a brute-force count.  A plausible mistake in the oracle (a
dropped rank term, a wrong BT order, a transposed operand, a bad fp16
decode) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from bitmap_encoded_unstructured_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f16(vals):
    return np.asarray(vals, dtype=np.float32).astype(np.float16).view(np.uint16)


def _popc_np(a):
    """Independent popcount: unpack bits with numpy and count them."""
    a = np.ascontiguousarray(a, dtype=np.uint64)
    return np.unpackbits(a.view(np.uint8)).reshape(-1, 64).sum(axis=1).astype(np.int64)


# ----------------------------------------------------------- page examples

def test_worked_bitmap_example():
    """SpInfer page, Values-array example: bits 10010110, position 4 -> Values[2]."""
    gold = _golden("spinfer_worked_bitmap.json")
    byte = int(gold["bits_msb_first"], 2)
    assert byte == 0x96
    assert [p for p in range(8) if (byte >> p) & 1] == gold["set_positions"]
    assert oracle.rank(byte, gold["query_position"]) == gold["query_index"]

    # Put the 8 decoded values in row 0, columns 0..7 of a 64x64 W: under the
    # row-major bit reading this is bit p = column of BT 0.
    W = np.zeros((64, 64), dtype=np.uint16)
    W[0, :8] = _f16(gold["decoded_positions_0_to_7"])
    enc = oracle.encode(W)
    assert int(enc["bitmaps"][0]) == byte
    assert enc["NNZ"] == 4
    np.testing.assert_array_equal(enc["values"], _f16(gold["values"]))
    assert enc["values"][oracle.rank(byte, 4)] == _f16([0.05])[0]
    np.testing.assert_array_equal(oracle.decode(enc), W)


def test_lspd_segment_ranks():
    """UnionSparse page, LSPD example: segment 10110100 (LSB first) -> b..b+3."""
    gold = _golden("unionsparse_lspd_segment.json")
    seg = gold["segment_lsb_first"]
    word = sum(1 << i for i, ch in enumerate(seg) if ch == "1")
    active = [p for p in range(8) if (word >> p) & 1]
    assert active == gold["active_positions"]
    assert [oracle.rank(word, p) for p in active] == gold["payload_index_offsets"]


def test_union_words_popcount():
    """UnionSparse page, IE-BME example: four words of 10 active bits, P_t=40, Q*P_t=160."""
    gold = _golden("unionsparse_union_words.json")
    counts = [oracle.popcount64(int(w, 16)) for w in gold["words"]]
    assert counts == [gold["active_bits_per_word"]] * 4
    assert sum(counts) == gold["P_t"]
    assert gold["Q"] * sum(counts) == gold["next_offset"]


def test_layout_table():
    """Hand-computed (r, c) -> (g, p) under the stated tiling reading."""
    gold = _golden("layout_positions.json")
    K = gold["K"]
    for case in gold["cases"]:
        assert oracle.locate(K, case["r"], case["c"]) == (case["g"], case["p"]), case
        assert oracle.position(K, case["g"], case["p"]) == (case["r"], case["c"]), case


def test_locate_is_a_bijection():
    M, K = 128, 192
    seen = set()
    for r in range(M):
        for c in range(K):
            g, p = oracle.locate(K, r, c)
            assert 0 <= g < M * K // 64 and 0 <= p < 64
            assert oracle.position(K, g, p) == (r, c)
            seen.add((g, p))
    assert len(seen) == M * K


# ----------------------------------------------------------- scalar helpers

def test_half_to_double_all_patterns():
    """Every one of the 65536 fp16 bit patterns against numpy's conversion."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # signed zeros and infinities keep their sign
    np.testing.assert_array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_popcount_and_rank():
    g = synth.rng(7)
    words = g.integers(0, 2**63, size=200, dtype=np.int64).astype(np.uint64) * np.uint64(2) \
        + g.integers(0, 2, size=200).astype(np.uint64)
    words = np.concatenate([words, np.array([0, 2**64 - 1, 1, 2**63], dtype=np.uint64)])
    ref = _popc_np(words)
    for w, r in zip(words, ref):
        assert oracle.popcount64(int(w)) == r
        for p in (0, 1, 7, 31, 32, 63, 64):
            want = bin(int(w) & ((1 << p) - 1)).count("1")
            assert oracle.rank(int(w), p) == want


# ----------------------------------------------------------- format invariants

@pytest.mark.parametrize("M,K,s,mask", [(64, 64, 0.5, "bernoulli"),
                                        (128, 320, 0.3, "uniform"),
                                        (256, 256, 0.7, "magnitude"),
                                        (192, 128, 0.0, "none")])
def test_encode_invariants_and_roundtrip(M, K, s, mask):
    W = synth.weights_f16(M, K, s, mask, seed=11)
    enc = oracle.encode(W)
    pc = _popc_np(enc["bitmaps"])
    nnz = int(np.count_nonzero(W))
    assert enc["NNZ"] == nnz == int(pc.sum()) == int(enc["offsets"][-1])
    assert np.all(np.diff(enc["offsets"].astype(np.int64)) >= 0)
    per_gt = pc.reshape(-1, 64).sum(axis=1)
    np.testing.assert_array_equal(np.diff(enc["offsets"].astype(np.int64)), per_gt)
    assert enc["offsets"][0] == 0
    # values are exactly the nonzeros (as a multiset) and decode is bitwise
    np.testing.assert_array_equal(np.sort(enc["values"]), np.sort(W[W != 0]))
    np.testing.assert_array_equal(oracle.decode(enc), W)


def test_roundtrip_special_payloads():
    """-0.0, NaN and Inf have nonzero bits, so they are stored as payload."""
    W = np.zeros((64, 128), dtype=np.uint16)
    specials = _f16([-0.0, np.inf, -np.inf]).tolist() + [0x7E00, 0x7C01, 0x0001, 0x8001]
    for i, v in enumerate(specials):
        W[3 * i, 5 * i + 1] = v
    enc = oracle.encode(W)
    assert enc["NNZ"] == len(specials)
    np.testing.assert_array_equal(oracle.decode(enc), W)


def test_roundtrip_all_zero_and_dense():
    Z = np.zeros((128, 64), dtype=np.uint16)
    enc = oracle.encode(Z)
    assert enc["NNZ"] == 0 and not enc["bitmaps"].any() and not enc["offsets"].any()
    np.testing.assert_array_equal(oracle.decode(enc), Z)
    D = synth.small_int_f16((64, 128), 1, 5, seed=3)
    enc = oracle.encode(D)
    assert enc["NNZ"] == D.size and np.all(enc["bitmaps"] == np.uint64(2**64 - 1))
    np.testing.assert_array_equal(oracle.decode(enc), D)


def test_single_nonzero_every_bt_position():
    for p in range(64):
        for b_r, b_c in ((0, 0), (1, 0), (0, 1), (7, 7)):
            W = np.zeros((64, 64), dtype=np.int8)
            r, c = 8 * b_r + p // 8, 8 * b_c + p % 8
            W[r, c] = -3
            enc = oracle.encode(W)
            g, pp = oracle.locate(64, r, c)
            assert pp == p
            nz = np.flatnonzero(enc["bitmaps"])
            assert nz.tolist() == [g] and int(enc["bitmaps"][g]) == 1 << p
            np.testing.assert_array_equal(oracle.decode(enc), W)


def test_int8_roundtrip():
    W = synth.weights_i8(128, 256, 0.6, seed=5)
    enc = oracle.encode(W)
    assert enc["values"].dtype == np.int8
    assert enc["NNZ"] == int(np.count_nonzero(W))
    np.testing.assert_array_equal(oracle.decode(enc), W)


def test_decode_by_brute_force_python():
    """A second, pure-Python decoder over the oracle's arrays (row-major scan
    of each BT, values consumed in order) must agree with the dense W."""
    W = synth.weights_f16(64, 128, 0.5, "bernoulli", seed=21)
    enc = oracle.encode(W)
    K = 128
    out = np.zeros_like(W)
    k = 0
    for g in range(enc["NBT"]):
        bm = int(enc["bitmaps"][g])
        for p in range(64):
            if (bm >> p) & 1:
                r, c = oracle.position(K, g, p)
                out[r, c] = enc["values"][k]
                k += 1
    assert k == enc["NNZ"]
    np.testing.assert_array_equal(out, W)


# ----------------------------------------------------------- zero-padded edge GroupTiles

@pytest.mark.parametrize("M,K", [(100, 72), (1, 8), (65, 64), (64, 136), (130, 200)])
def test_padded_edges_by_brute_force(M, K):
    """M or K not a multiple of 64: the grid covers W padded with zeros to
    multiples of 64.  Checked position by position against W itself (the
    oracle's own mapping from (row, col) to (BT, bit)), in a pure-Python
    scan: a bit is set exactly for the nonzeros of W, never in the padding,
    and the values come out in BT-then-bit order."""
    W = synth.weights_f16(M, K, 0.5, "bernoulli", seed=M * 1000 + K)
    enc = oracle.encode(W)
    Mp, Kp = -(-M // 64) * 64, -(-K // 64) * 64
    assert (enc["Mp"], enc["Kp"]) == (Mp, Kp)
    assert enc["NGT"] == (Mp // 64) * (Kp // 64) and enc["NBT"] == Mp * Kp // 64
    assert enc["NNZ"] == int(np.count_nonzero(W))
    k = 0
    for g in range(enc["NBT"]):
        bm = int(enc["bitmaps"][g])
        for p in range(64):
            r, c = oracle.position(Kp, g, p)
            inside = r < M and c < K
            want = inside and W[r, c] != 0
            assert ((bm >> p) & 1) == int(want), (g, p, r, c)
            if want:
                assert enc["values"][k] == W[r, c]
                k += 1
    assert k == enc["NNZ"]
    np.testing.assert_array_equal(oracle.decode(enc), W)
    # Stor counts the padded grid's tiles and the true nonzeros only
    assert oracle.storage_bytes(enc) == 4 * (enc["NGT"] + 1) + 8 * enc["NBT"] + 2 * enc["NNZ"]
    # the product ignores the padding: the dense one of the logical W
    X = synth.activations_f16(3, K, seed=5)
    y, _ = oracle.spmm_f16(W, X)
    np.testing.assert_allclose(y, _f64(X) @ _f64(W).T, rtol=1e-12, atol=1e-15)  # [N][M]


# ----------------------------------------------------------- storage accounting

@pytest.mark.parametrize("M,K,s,dt", [(256, 256, 0.5, "f16"), (512, 384, 0.3, "f16"),
                                      (256, 512, 0.6, "i8"), (128, 128, 0.0, "f16")])
def test_storage_closed_form(M, K, s, dt):
    """SpInfer page: Stor = 4B*(NGT+1) + 8B*NBT + 2B*NNZ (B_v = 1 for int8)."""
    W = synth.weights_f16(M, K, s, "uniform", 3) if dt == "f16" else synth.weights_i8(M, K, s, 3)
    enc = oracle.encode(W)
    bv = 2 if dt == "f16" else 1
    NGT, NBT = (M // 64) * (K // 64), M * K // 64
    assert enc["NGT"] == NGT and enc["NBT"] == NBT
    assert oracle.storage_bytes(enc) == 4 * (NGT + 1) + 8 * NBT + bv * enc["NNZ"]


def test_cr_above_one_at_30_percent_and_csr_below():
    """SpInfer page: TCA-BME gives CR > 1 at 30% sparsity; CSR (6 B per
    nonzero for fp16) stays below 1 at low sparsity.  SPDP eq. (1): CR =
    2B*M*K / Stor."""
    W = synth.weights_f16(1024, 1024, 0.3, "uniform", seed=1030)
    enc = oracle.encode(W)
    cr = oracle.compression_ratio(enc)
    assert cr > 1.0
    assert abs(cr - 2 * 1024 * 1024 / oracle.storage_bytes(enc)) < 1e-12
    cr_csr = 2 * W.size / oracle.csr_bytes(W)
    assert cr_csr < 1.0
    W50 = synth.weights_f16(1024, 1024, 0.5, "uniform", seed=1050)
    assert 2 * W50.size / oracle.csr_bytes(W50) < 1.0
    assert oracle.compression_ratio(oracle.encode(W50)) > cr


# ----------------------------------------------------------- products

def _f64(bits):
    return bits.view(np.float16).astype(np.float64)


def test_spmm_f16_matches_library_matmul():
    W = synth.weights_f16(64, 192, 0.5, "bernoulli", seed=31)
    X = synth.activations_f16(5, 192, seed=32)
    Y, S = oracle.spmm_f16(W, X)
    ref = _f64(X) @ _f64(W).T  # [N][M]
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(S, np.abs(_f64(X)) @ np.abs(_f64(W)).T, rtol=1e-12, atol=1e-15)


def test_spmm_f16_small_integers_exact():
    W = synth.small_int_f16((128, 256), -8, 8, seed=41, sparsity=0.5)
    X = synth.small_int_f16((3, 256), -8, 8, seed=42)
    Y, _ = oracle.spmm_f16(W, X)
    ref = X.view(np.float16).astype(np.int64) @ W.view(np.float16).astype(np.int64).T
    np.testing.assert_array_equal(Y, ref.astype(np.float64))


def test_spmm_f16_permutation():
    M = K = 128
    perm = synth.rng(5).permutation(K)
    W = np.zeros((M, K), dtype=np.uint16)
    W[np.arange(M), perm] = _f16([1.0])[0]
    X = synth.activations_f16(4, K, seed=6)
    Y, _ = oracle.spmm_f16(W, X)
    np.testing.assert_array_equal(Y, _f64(X)[:, perm])


def test_spmm_i8_matches_library_matmul():
    W = synth.weights_i8(64, 320, 0.5, seed=51)
    X = synth.activations_i8(7, 320, seed=52)
    Y = oracle.spmm_i8(W, X)
    np.testing.assert_array_equal(Y, X.astype(np.int64) @ W.astype(np.int64).T)


def test_scale_i8_matches_numpy_float32():
    W = synth.weights_i8(128, 256, 0.5, seed=61)
    X = synth.activations_i8(3, 256, seed=62)
    scale = synth.row_scales(128, seed=63)
    acc = oracle.spmm_i8(W, X)
    got = oracle.scale_i8(acc, scale)
    ref = acc.astype(np.float32) * scale[None, :]
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_spmspv_is_n1_product():
    W = synth.weights_f16(128, 256, 0.5, "uniform", seed=71)
    x = synth.activations_relu_f16(256, seed=72)
    y, s = oracle.spmspv_f16(W, x)
    ref = _f64(W) @ _f64(x)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)
    assert np.all(s >= np.abs(y))


# ----------------------------------------------------------- input generators

def test_synth_exact_counts():
    M, K = 256, 512
    for s in (0.3, 0.5, 0.7):
        W = synth.weights_f16(M, K, s, "uniform", seed=1)
        assert np.count_nonzero(W == 0) >= round(s * M * K)
        Wm = synth.weights_f16(M, K, s, "magnitude", seed=2)
        nz = np.count_nonzero(Wm & 0x7FFF)
        assert nz <= M * K - round(s * M * K)
        # magnitude: every kept |w| >= every zeroed original |w|
    Wi = synth.weights_i8(M, K, 0.6, seed=3)
    assert np.count_nonzero(Wi == 0) == round(0.6 * M * K)
    x = synth.activations_relu_f16(20480, seed=4)
    frac = np.count_nonzero(x == 0) / x.size
    assert 0.83 < frac < 0.87


# ----------------------------------------------------------- dynamic pruning (threshold)

def test_prune_activations_worked_values():
    """|x| <= t is pruned: exact fp16 values around t = 0.25; NaN is kept."""
    x = _f16([0.5, -0.25, 0.125, 0.375, -0.75, 0.0, -0.0])
    x = np.concatenate([x, np.array([0x7E00], dtype=np.uint16)])  # NaN
    got = oracle.prune_activations_f16(x, 0.25)
    want = _f16([0.5, 0.0, 0.0, 0.375, -0.75, 0.0, 0.0])
    np.testing.assert_array_equal(got[:7], want)
    assert got[7] == 0x7E00
    # threshold 0 keeps every nonzero value and clears only the two zeros
    np.testing.assert_array_equal(oracle.prune_activations_f16(x, 0.0)[:5], x[:5])


def test_spmspv_threshold_matches_library_on_masked_x():
    W = synth.weights_f16(128, 512, 0.5, "uniform", 81)
    x = synth.activations_f16(1, 512, 82)[0]
    for t in (0.0, 0.3, 1.0, 1e9):
        y, s = oracle.spmspv_threshold_f16(W, x, t)
        xv = x.view(np.float16).astype(np.float64)
        xm = np.where(np.abs(xv) <= np.float64(np.float32(t)), 0.0, xv)
        np.testing.assert_allclose(y, _f64(W) @ xm, rtol=1e-12, atol=1e-15)
    assert np.all(oracle.spmspv_threshold_f16(W, x, 1e9)[0] == 0)


def test_prune_activations_i8():
    x = np.array([-127, -60, -59, 0, 59, 60, 61, 127], dtype=np.int8)
    np.testing.assert_array_equal(oracle.prune_activations_i8(x, 60),
                                  np.array([-127, 0, 0, 0, 0, 0, 61, 127], dtype=np.int8))


# ----------------------------------------------------------- payload-to-metadata ratio

def test_pmr_of_dense_and_half_dense_grouptiles():
    """PMR = value bytes / (bitmap + offset bytes), counted by hand: one
    64 x 64 GroupTile holds 64 bitmaps (512 B) and two offsets (8 B)."""
    dense = _f16(np.full((64, 64), 0.5))
    assert oracle.payload_to_metadata(oracle.encode(dense)) == 8192 / 520
    half = dense.copy()
    half[:, ::2] = 0                       # 2048 values of 2 B
    assert oracle.payload_to_metadata(oracle.encode(half)) == 4096 / 520
    two = np.zeros((64, 128), dtype=np.uint16)
    two[3, 70] = dense[0, 0]               # one value, two GroupTiles: 128 bitmaps + 3 offsets
    assert oracle.payload_to_metadata(oracle.encode(two)) == 2 / (1024 + 12)


def test_csr_bytes_hand_counted():
    """The CSR comparator counted by hand: a 3 x 5 matrix with 4 nonzeros
    holds 4 values (2 B each in fp16, 1 B in int8), 4 column indices of 4 B
    and 3 + 1 row pointers of 4 B: 8 + 16 + 16 = 40 B in fp16, 36 B in int8.
    A dropped row-pointer array, a 2-byte index or an M-entry pointer array
    each changes the count."""
    W16 = np.zeros((3, 5), dtype=np.uint16)
    W16[0, 1] = 0x3C00
    W16[0, 4] = 0xBC00
    W16[2, 0] = 0x4000
    W16[2, 3] = 0x3800
    assert oracle.csr_bytes(W16) == 4 * 2 + 4 * 4 + (3 + 1) * 4 == 40
    W8 = np.zeros((3, 5), dtype=np.int8)
    W8[W16 != 0] = 7
    assert oracle.csr_bytes(W8) == 4 * 1 + 4 * 4 + (3 + 1) * 4 == 36
    assert oracle.csr_bytes(np.zeros((6, 5), dtype=np.uint16)) == (6 + 1) * 4
