"""CPU oracle for the IE-BME low-bit union-bitmap format and its product.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this module; the CUDA library never imports it and
the two share no code.

Source: "UnionSparse" (IE-BME, sections "Area Partitioning", "Shared Union
Mask", "IE-BME Storage Layout"; LSPD, section "Bitmap-Guided Offset
Generation").  Plain numpy, in the order the page describes the steps:

1. A quantized local tile W_t (H_L x K_L) is cut into an R_A x C_A grid of
   areas of h = H_L / R_A rows and w = K_L / C_A columns; Q = R_A * C_A.
   Area a = ra * C_A + ca (row-major over the area grid).
2. Position (i, j) of the h x w logical grid groups the Q values
   W_t[ra * h + i][ca * w + j], one from each area; its union-mask bit is 1
   iff one of them is nonzero.
3. P_t = number of active positions.  The active positions get compact ranks
   in row-major order; every area appends its value at every active
   position (zeros included), so area a's stream of LT t is
   values[o_t + a * P_t + rank].  o_t is the prefix sum of Q * P_t.
4. Union bitmaps: the h x w mask row-major, packed into 64-bit words with
   the leftmost position in the least significant bit.

Readings where the page is silent (its equations were lost in the
extraction): LTs tile the matrix row-major over the grid of H_L x K_L tiles
with M and K zero-padded up to multiples of the tile; h * w must be a
multiple of 64 so that every LT owns whole words; int4 payloads are stored
two per byte, value e of the global stream in byte e // 2, the low nibble
first, in two's complement; the values are integers in the signed b-bit
range, and the product accumulates exactly (int64 here, int32 on the GPU).
"""
from __future__ import annotations

import numpy as np

LT = (64, 64)
AREAS = (2, 2)


def _check(W: np.ndarray, bits: int, lt, areas):
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    H, KL = lt
    RA, CA = areas
    if H % RA or KL % CA:
        raise ValueError("the areas must tile the LT")
    if ((H // RA) * (KL // CA)) % 64:
        raise ValueError("the logical mask of an LT must fill whole 64-bit words")
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    if W.size and (W.min() < lo or W.max() > hi):
        raise ValueError(f"values outside the signed {bits}-bit range")


def union_encode(W: np.ndarray, bits: int, lt=LT, areas=AREAS, perms=None) -> dict:
    """IE-BME arrays of an integer matrix W [M][K] (values in the signed
    `bits`-bit range): masks u64 [NLT * words], offsets u32 [NLT + 1] (value
    counts), values int8 [o_NLT] (one element per value, unpacked).
    perms (optional, [NLT][H_L]): LT t is encoded with its rows reordered,
    row k of the reordered tile being row perms[t][k] of the original."""
    W = np.asarray(W, dtype=np.int64)
    _check(W, bits, lt, areas)
    M, K = W.shape
    H, KL = lt
    RA, CA = areas
    h, w = H // RA, KL // CA
    Q = RA * CA
    Mp, Kp = -(-M // H) * H, -(-K // KL) * KL
    Wp = np.zeros((Mp, Kp), dtype=np.int64)
    Wp[:M, :K] = W
    words_per_lt = h * w // 64
    masks, offsets, values = [], [0], []
    for ti in range(Mp // H):
        for tj in range(Kp // KL):
            tile = Wp[ti * H:(ti + 1) * H, tj * KL:(tj + 1) * KL]
            if perms is not None:
                tile = tile[np.asarray(perms[len(offsets) - 1], dtype=np.int64)]
            area = [tile[ra * h:(ra + 1) * h, ca * w:(ca + 1) * w] for ra in range(RA) for ca in range(CA)]
            B = np.zeros((h, w), dtype=bool)
            for A in area:
                B |= A != 0
            P = int(B.sum())
            for A in area:                       # stream a: A at the active positions, row-major
                values.append(A[B])
            # row-major, position p of the LT in bit p % 64 of word p // 64
            masks.append(np.packbits(B.reshape(-1), bitorder="little").view("<u8"))
            offsets.append(offsets[-1] + Q * P)
    vals = np.concatenate(values).astype(np.int8) if values else np.zeros(0, dtype=np.int8)
    masks = np.concatenate(masks).astype(np.uint64) if masks else np.zeros(0, dtype=np.uint64)
    return {"masks": masks, "offsets": np.array(offsets, dtype=np.uint64).astype(np.uint32),
            "values": vals, "bits": bits, "lt": tuple(lt), "areas": tuple(areas),
            "M": M, "K": K, "Mp": Mp, "Kp": Kp, "nnz": int(np.count_nonzero(W)),
            "perms": None if perms is None else np.asarray(perms, dtype=np.int64)}


def union_decode(enc: dict) -> np.ndarray:
    """W back from the three arrays."""
    H, KL = enc["lt"]
    RA, CA = enc["areas"]
    h, w = H // RA, KL // CA
    Q = RA * CA
    Mp, Kp = enc["Mp"], enc["Kp"]
    words_per_lt = h * w // 64
    W = np.zeros((Mp, Kp), dtype=np.int64)
    t = 0
    for ti in range(Mp // H):
        for tj in range(Kp // KL):
            words = np.ascontiguousarray(enc["masks"][t * words_per_lt:(t + 1) * words_per_lt]).astype("<u8")
            flat = np.unpackbits(words.view(np.uint8), bitorder="little").astype(bool)
            B = flat.reshape(h, w)
            P = int(flat.sum())
            o = int(enc["offsets"][t])
            assert int(enc["offsets"][t + 1]) - o == Q * P
            tile = np.zeros((H, KL), dtype=np.int64)
            for a in range(Q):
                ra, ca = divmod(a, CA)
                A = np.zeros((h, w), dtype=np.int64)
                A[B] = enc["values"][o + a * P:o + (a + 1) * P]
                tile[ra * h:(ra + 1) * h, ca * w:(ca + 1) * w] = A
            if enc.get("perms") is not None:  # undo the LT's row reordering
                orig = np.zeros_like(tile)
                orig[enc["perms"][t]] = tile
                tile = orig
            W[ti * H:(ti + 1) * H, tj * KL:(tj + 1) * KL] = tile
            t += 1
    return W[:enc["M"], :enc["K"]].astype(np.int8)


def pack_values(values: np.ndarray, bits: int) -> np.ndarray:
    """The stored bytes of the value stream: int8 as is; int4 two per byte,
    value e in byte e // 2, low nibble first (two's complement)."""
    v = np.asarray(values, dtype=np.int64)
    if bits == 8:
        return v.astype(np.int8).view(np.uint8)
    nib = (v & 0xF).astype(np.uint8)
    if nib.size % 2:
        nib = np.concatenate([nib, np.zeros(1, dtype=np.uint8)])
    return (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)


def storage_bytes(enc: dict) -> int:
    """Offsets (4 B each) + bitmap words (8 B each) + packed values."""
    total = int(enc["offsets"][-1])
    return 4 * len(enc["offsets"]) + 8 * len(enc["masks"]) + (total * enc["bits"] + 7) // 8


def payload_to_metadata(enc: dict) -> float:
    """UnionSparse's PMR: useful payload bytes (b/8 per nonzero) over every
    other stored byte (offsets, bitmaps, and the zeros kept in active
    groups)."""
    payload = enc["nnz"] * enc["bits"] / 8
    return payload / (storage_bytes(enc) - payload)


def lspd_indices(segment: int, g: int, idx_base: int) -> list:
    """LSPD for one G-bit segment (bit 0 = leftmost position): the active
    positions, in order, with global index idx_base + their rank inside the
    segment."""
    out, r = [], 0
    for p in range(g):
        if (segment >> p) & 1:
            out.append((p, idx_base + r))
            r += 1
    return out


def union_spmm(W: np.ndarray, X: np.ndarray) -> np.ndarray:
    """Y [N][M] = X [N][K] * W^T, exact in int64 (the definition; the format
    does not change the result)."""
    return np.asarray(X, dtype=np.int64) @ np.asarray(W, dtype=np.int64).T


# ---------------------------------------------------------------- row reordering
#
# UnionSparse, "Bitmap-aware row reordering" ("Grouped Cost Formulation",
# "Grouped Subset Dynamic Programming"): the rows of an LT are partitioned
# into groups of R_A rows; a group's cost is the number of logical
# union-mask entries it activates, i.e. over the K_L / C_A grouped columns
# j, whether any of its rows has a nonzero at one of the C_A columns that
# group into j.  A subset DP finds the minimum total cost: F(S) for the set
# S of rows not yet grouped, F(empty) = 0, F(S) = min over the groups g of
# size R_A that contain the smallest row of S of cost(g) + F(S \ g).  The
# result is made canonical (rows ascending inside each group, groups in
# lexicographic order) and turned into a permutation partition-wise: the
# p-th row of every group, group by group, for p = 0 .. R_A - 1.

def group_costs_table(tile: np.ndarray, RA: int, CA: int) -> dict:
    """cost(g) for every group g (a sorted tuple of R_A row indices)."""
    from itertools import combinations
    H, KL = tile.shape
    w = KL // CA
    # grouped activity of each row: column j is active if one of its C_A
    # columns j, w + j, ... holds a nonzero
    act = np.zeros((H, w), dtype=bool)
    for ca in range(CA):
        act |= tile[:, ca * w:(ca + 1) * w] != 0
    return {g: int(np.logical_or.reduce(act[list(g)], axis=0).sum()) for g in combinations(range(H), RA)}


def reorder_rows(tile: np.ndarray, RA: int, CA: int):
    """Optimal grouping of the tile's rows by the subset DP; returns
    (permutation, total cost).  perm[k] = original row placed at row k:
    row i of area row p is the p-th row of group i."""
    from itertools import combinations
    H = tile.shape[0]
    if H % RA:
        raise ValueError("R_A must divide the tile's rows")
    cost = group_costs_table(tile, RA, CA)
    full = (1 << H) - 1
    F = {0: (0, None)}   # state -> (min cost, chosen group)
    # states in order of increasing size (only sizes divisible by R_A occur)
    order = sorted((S for S in range(full + 1) if bin(S).count("1") % RA == 0), key=lambda S: bin(S).count("1"))
    for S in order:
        if S == 0:
            continue
        rows = [r for r in range(H) if (S >> r) & 1]
        r0 = rows[0]
        best = None
        for rest in combinations(rows[1:], RA - 1):   # lexicographic: the first minimum is kept
            g = (r0,) + rest
            T = S
            for r in g:
                T &= ~(1 << r)
            c = cost[g] + F[T][0]
            if best is None or c < best[0]:
                best = (c, g)
        F[S] = best
    groups, S = [], full
    while S:
        g = F[S][1]
        groups.append(tuple(sorted(g)))
        for r in g:
            S &= ~(1 << r)
    groups.sort()
    perm = [g[p] for p in range(RA) for g in groups]
    return np.array(perm, dtype=np.int64), F[full][0]


def union_active(tile: np.ndarray, RA: int, CA: int) -> int:
    """P_t of a tile as it stands (rows grouped i, h + i, 2h + i, ...)."""
    H = tile.shape[0]
    h = H // RA
    cost = 0
    w = tile.shape[1] // CA
    for i in range(h):
        act = np.zeros(w, dtype=bool)
        for ra in range(RA):
            for ca in range(CA):
                act |= tile[ra * h + i, ca * w:(ca + 1) * w] != 0
        cost += int(act.sum())
    return cost
