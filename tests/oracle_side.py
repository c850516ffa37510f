"""Oracle side of the parity tests: builds the oracle's own cache, quantised
queries and top-k rows from the same seeded FP32 inputs the GPU receives,
and the comparison rules the GPU path must meet."""

from __future__ import annotations

import numpy as np

import oracle as O

SCORE_RTOL = 2e-3   # scores within 2e-3 x the row's max |score|


def oracle_cache(wl, layer: int, with_new: bool = True, fill: int = 0) -> np.ndarray:
    """The oracle's page pool for `layer` (bytes never written hold `fill`):
    cached prefix (+ this step's keys).  Prefix entries sit at entry
    positions 0 .. prefix_entries-1."""
    cache = np.full((wl.num_pages, O.PAGE_BYTES), fill, np.uint8)
    for r in range(wl.R):
        E = int(wl.prefix_entries[r])
        if E:
            slots = O.slot_mapping(np.array([0, E]), np.array([E]), wl.block_table[r:r + 1])
            O.write_k_cache(cache, wl.k_prefix(layer, r), slots)
    if with_new:
        O.write_k_cache(cache, wl.k_new(layer),
                        O.compressed_slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table,
                                                  wl.compress_ratio))
    return cache


def request_keys(wl, layer: int, r: int, k_new=None):
    """Codes/scales of request r by entry position, straight from its FP32
    keys: the prefix entries, then the new tokens that complete an entry."""
    qsl = wl.query_start_loc
    kn = wl.k_new(layer) if k_new is None else k_new
    n = wl.compress_ratio
    parts = []
    if wl.prefix_entries[r]:
        parts.append(wl.k_prefix(layer, r))
    new = kn[qsl[r]:qsl[r + 1]]
    pos = int(wl.prefix_lens[r]) + np.arange(new.shape[0])
    parts.append(new[(pos + 1) % n == 0])
    return O.quantize_blocks(np.concatenate(parts, axis=0))


def oracle_rows(wl, layer: int, rows, q_codes, q_scale, w, k_new=None):
    """{row: float64 scores over its visible keys} for the given query rows."""
    req, pos = O.token_positions(wl.query_start_loc, wl.seq_lens)
    out = {}
    by_req = {}
    for t in rows:
        by_req.setdefault(int(req[t]), []).append(t)
    for r, ts in by_req.items():
        kc, ks = request_keys(wl, layer, r, k_new)
        for t in ts:
            ctx = int(O.visible_entries(pos[t], wl.compress_ratio))
            out[t] = O.index_scores(q_codes[t], q_scale[t], w[t], kc[:ctx], ks[:ctx])
    return out


def check_scores(gpu_row: np.ndarray, ref: np.ndarray, where: str) -> None:
    n = ref.shape[0]
    tol = SCORE_RTOL * max(np.max(np.abs(ref)), 1e-30)
    err = np.abs(gpu_row[:n].astype(np.float64) - ref)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, (f"{where}: {bad.size} scores off by more than {tol:.3g}; "
                           f"first at key {bad[0]}: gpu {gpu_row[bad[0]]} oracle {ref[bad[0]]}")


def check_topk_row(gpu_row: np.ndarray, ref_scores: np.ndarray, k: int, where: str) -> None:
    """GPU row vs oracle: -1 padding and valid count exact; index sets equal up
    to swaps among keys whose oracle score is within the score tolerance of
    the k-th largest."""
    ctx = ref_scores.shape[0]
    n = min(ctx, k)
    assert np.all(gpu_row[n:] == -1), f"{where}: padding is not -1 after {n} entries"
    got = gpu_row[:n]
    assert np.all(got >= 0) and np.all(got < ctx), f"{where}: index outside [0, {ctx})"
    assert np.unique(got).size == n, f"{where}: duplicate indices"
    want = O.topk_row(ref_scores, k)[:n]
    diff = np.setxor1d(got, want)
    if diff.size:
        kth = np.sort(ref_scores)[::-1][n - 1]
        tol = SCORE_RTOL * max(np.max(np.abs(ref_scores)), 1e-30)
        off = np.abs(ref_scores[diff] - kth)
        assert np.all(off <= tol), (f"{where}: {diff.size} differing indices, worst "
                                    f"{off.max():.3g} from the k-th score (tolerance {tol:.3g})")
