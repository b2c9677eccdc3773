"""CPU oracle for the Tiled-CBC column-wise bitmap format (the spMspV side
index) and the sparse-vector product that skips inactive columns.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this module; the CUDA library never imports it and
the two share no code.

Source: "Unified Static-Dynamic Pruning for Efficient LLM Inference"
(SPDP), section 4.1 "Tiled-CBC: Unified Compression Format" (Tiling Design,
Storage Structure, the storage equation) and section 4.2 (dynamic pruning:
inactive columns are neither fetched nor multiplied).  Plain numpy loops, in
the page's order:

1. GTiles of TILE_M x TILE_K elements tile W row-major (M and K zero-padded
   up to multiples of the tile); a GTile holds TILE_K column tiles of
   TILE_M x 1 elements, the unit of compression and pruning.
2. Bitmap: TILE_M / 64 uint64 words per column tile; bit (r % 64) of word
   r // 64 is set iff element r of the column is nonzero (raw bits != 0).
3. Values: the nonzeros of a GTile in tile-column order (column 0 top to
   bottom, then column 1, ...); GTiles follow one another in row-major order.
4. TileOffset: uint32 [NGT + 1], value counts before each GTile.
5. ColInfo: one uint32 per column of each GTile, the column's first value
   inside its GTile (TileOffset_Col) in the upper 16 bits and its nonzero
   count (NNZ_Column) in the lower 16.
6. Stor = 4 (NGT + 1) + 4 NGT TILE_K + 8 NBM + B_v NNZ, NBM = M K / 64.

Readings where the page is silent or leaves a choice: TILE_M = 256 as on
the page (four bitmaps per column), TILE_K = 64 (the GroupTile width of the
bitmap format the library's other kernels use; the page does not give its
value); the order of the four bitmap words of a column is by row (rows 0-63
first); "nonzero" means raw bits != 0, as in the row-wise format.
"""
from __future__ import annotations

import numpy as np

TILE_M, TILE_K = 256, 64
WORDS = TILE_M // 64


def _elem_bytes(W: np.ndarray) -> int:
    if W.dtype == np.uint16:
        return 2
    if W.dtype == np.int8:
        return 1
    raise TypeError("W must be uint16 (fp16 bits) or int8")


def encode(W: np.ndarray) -> dict:
    """The five arrays of W [M][K] (fp16 bits or int8)."""
    W = np.ascontiguousarray(W)
    eb = _elem_bytes(W)
    M, K = W.shape
    Mp = -(-M // TILE_M) * TILE_M
    Kp = -(-K // TILE_K) * TILE_K
    Wp = np.zeros((Mp, Kp), dtype=W.dtype)
    Wp[:M, :K] = W
    tr, tc = Mp // TILE_M, Kp // TILE_K
    NGT = tr * tc
    bitmaps = np.zeros(NGT * TILE_K * WORDS, dtype=np.uint64)
    colinfo = np.zeros(NGT * TILE_K, dtype=np.uint32)
    offsets = np.zeros(NGT + 1, dtype=np.uint32)
    values = []
    n = 0
    for gi in range(tr):                      # GTiles row-major
        for gj in range(tc):
            t = gi * tc + gj
            offsets[t] = n
            tile = Wp[gi * TILE_M:(gi + 1) * TILE_M, gj * TILE_K:(gj + 1) * TILE_K]
            start = 0
            for c in range(TILE_K):           # tile-column order
                col = tile[:, c]
                nz = [r for r in range(TILE_M) if col[r] != 0]
                for r in nz:
                    w = (t * TILE_K + c) * WORDS + r // 64
                    bitmaps[w] |= np.uint64(1) << np.uint64(r % 64)
                    values.append(col[r])
                colinfo[t * TILE_K + c] = (start << 16) | len(nz)
                start += len(nz)
            n += start
    offsets[NGT] = n
    vals = np.array(values, dtype=W.dtype) if values else np.zeros(0, dtype=W.dtype)
    return {"M": M, "K": K, "Mp": Mp, "Kp": Kp, "dtype": W.dtype, "elem_bytes": eb,
            "NGT": NGT, "NBM": Mp * Kp // 64, "NNZ": n, "offsets": offsets, "colinfo": colinfo,
            "bitmaps": bitmaps, "values": vals}


def decode(enc: dict) -> np.ndarray:
    """W back from the arrays: element r of column c of GTile t is the value
    at TileOffset[t] + TileOffset_Col + (set bits of the column above r)."""
    Mp, Kp = enc["Mp"], enc["Kp"]
    tc = Kp // TILE_K
    out = np.zeros((Mp, Kp), dtype=enc["dtype"])
    for t in range(enc["NGT"]):
        gi, gj = divmod(t, tc)
        for c in range(TILE_K):
            info = int(enc["colinfo"][t * TILE_K + c])
            base = int(enc["offsets"][t]) + (info >> 16)
            k = 0
            for r in range(TILE_M):
                w = int(enc["bitmaps"][(t * TILE_K + c) * WORDS + r // 64])
                if (w >> (r % 64)) & 1:
                    out[gi * TILE_M + r, gj * TILE_K + c] = enc["values"][base + k]
                    k += 1
            assert k == (info & 0xFFFF)
    return out[:enc["M"], :enc["K"]]


def storage_bytes(enc: dict) -> int:
    """The page's closed form: 4 (NGT + 1) + 4 NGT TILE_K + 8 NBM + B_v NNZ."""
    return 4 * (enc["NGT"] + 1) + 4 * enc["NGT"] * TILE_K + 8 * enc["NBM"] + enc["elem_bytes"] * enc["NNZ"]


def active_columns(x_active: np.ndarray, enc: dict) -> np.ndarray:
    """Per GTile, which of its columns a sparse-vector product touches: column
    c of GTile (gi, gj) is active iff its activation x[gj * TILE_K + c] is."""
    tc = enc["Kp"] // TILE_K
    a = np.zeros(enc["Kp"], dtype=bool)
    a[:x_active.shape[0]] = x_active
    return np.tile(a.reshape(tc, TILE_K), (enc["NGT"] // tc, 1)).reshape(-1)


def fetched_bytes(enc: dict, x_active: np.ndarray) -> int:
    """Bytes a column-skipping spMspV reads from the index: the ColInfo of
    every GTile, and the bitmaps and values of the active columns only (the
    page's step (3): only activation-relevant columns are fetched)."""
    act = active_columns(x_active, enc)
    nnz_act = int(sum(int(enc["colinfo"][i]) & 0xFFFF for i in np.nonzero(act)[0]))
    return 4 * enc["NGT"] * TILE_K + 8 * WORDS * int(act.sum()) + enc["elem_bytes"] * nnz_act
