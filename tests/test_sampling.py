"""The full-size parity tests' row sample reaches every GEMM tile (host logic,
no GPU): checked on the oracle's own dispatch of seeded routings."""
import numpy as np
import pytest

from sampling import TILE_ROWS, tile_coverage, tile_stratified_tokens


def _routing(T, E, k, seed, skew=False):
    rng = np.random.default_rng(seed)
    p = None
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
    idx = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return idx


@pytest.mark.parametrize("T,E,k,Fs,skew", [(5000, 8, 2, 0, False), (3000, 64, 6, 0, False),
                                           (1000, 16, 4, 256, False), (4000, 8, 2, 0, True),
                                           (7, 4, 2, 0, False)])
def test_stratified_sample_covers_every_tile(oracle, T, E, k, Fs, skew):
    idx = _routing(T, E, k, seed=T + E, skew=skew)
    counts, offsets, src_row, inv_pos = oracle.permute(idx, E)
    toks = tile_stratified_tokens(offsets, src_row, k, T, Fs)
    covered, n_tiles = tile_coverage(toks, inv_pos, offsets, k, T, Fs)
    assert covered == n_tiles
    seg = np.diff(offsets.astype(np.int64))
    want = int(np.sum((seg + TILE_ROWS - 1) // TILE_ROWS)) + (((T + TILE_ROWS - 1) // TILE_ROWS) if Fs else 0)
    assert n_tiles == want
    # the sample is far smaller than the batch at full-size ratios
    assert toks.size <= 2 * n_tiles + 2


def test_coverage_notices_a_missing_tile(oracle):
    """Dropping every token of one tile lowers the coverage count."""
    T, E, k = 3000, 8, 2
    idx = _routing(T, E, k, seed=5)
    counts, offsets, src_row, inv_pos = oracle.permute(idx, E)
    toks = tile_stratified_tokens(offsets, src_row, k, T, 0)
    e = 3
    lo = int(offsets[e])
    hi = min(lo + TILE_ROWS, int(offsets[e + 1]))
    gone = set((np.asarray(src_row[lo:hi], np.int64) // k).tolist())
    kept = np.asarray([t for t in toks if t not in gone], np.int64)
    covered, n_tiles = tile_coverage(kept, inv_pos, offsets, k, T, 0)
    assert covered < n_tiles
