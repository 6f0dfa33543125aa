"""Which output rows a full-size parity test compares.

At full size the oracle computes a subset of the output rows (rows are
independent, so each is exact). The subset must reach every tile of the
expert GEMMs, so that a fault confined to one tile cannot pass unseen.
Host logic only: the dispatch order it reads is the oracle's.
"""
import numpy as np


TILE_ROWS = 128   # the smallest M tile of the expert GEMMs (a CTA pair's 256-row tile is two)


def tile_stratified_tokens(offsets, src_row, k, T, Fs):
    """Tokens whose output rows reach every M tile of every expert GEMM.

    The expert GEMMs tile each expert's segment of the dispatch order
    (offsets[e] .. offsets[e+1]) into 128-row tiles (a CTA pair's 256-row tile
    is two of them); every output row of a tile spans all N tiles. So the
    token of each tile's first and last row, and the last row of each
    segment, put at least one compared row into every (M tile, N tile) of
    both GEMMs. The shared expert's GEMMs tile the tokens in order: the
    first and last token of each 128-token tile. Taken from the oracle's
    dispatch order, not the CUDA path's."""
    rows = []
    E = offsets.size - 1
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        starts = np.arange(lo, hi, TILE_ROWS)
        rows.append(starts)
        rows.append(np.minimum(starts + TILE_ROWS - 1, hi - 1))
    toks = [np.asarray(src_row, np.int64)[np.concatenate(rows)] // k] if rows else []
    if Fs:
        starts = np.arange(0, T, TILE_ROWS)
        toks += [starts, np.minimum(starts + TILE_ROWS - 1, T - 1)]
    return np.unique(np.concatenate(toks)).astype(np.int64) if toks else np.zeros(0, np.int64)


def tile_coverage(tokens, inv_pos, offsets, k, T, Fs):
    """(M tiles holding at least one compared row, all M tiles), over the
    routed experts' 128-row tiles and, with a shared expert, its token tiles."""
    tokens = np.asarray(tokens, np.int64)
    pos = np.asarray(inv_pos, np.int64).reshape(T, k)[tokens].reshape(-1)
    grp = np.searchsorted(offsets, pos, side="right") - 1
    tile_id = np.asarray([(g, (p - offsets[g]) // TILE_ROWS) for g, p in zip(grp, pos)]).reshape(-1, 2)
    covered = len({(int(a), int(b)) for a, b in tile_id})
    seg = np.diff(offsets.astype(np.int64))
    n_tiles = int(np.sum((seg + TILE_ROWS - 1) // TILE_ROWS))
    if Fs:
        covered += np.unique(tokens // TILE_ROWS).size
        n_tiles += (T + TILE_ROWS - 1) // TILE_ROWS
    return covered, n_tiles
