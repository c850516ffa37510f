"""Rows long enough to be split across SMs, with heavily tied scores (GPU).

A long decode row is cut into pieces that run on different CTAs and are
merged through their level-1 bin histograms.  Equal scores all fall into one
bin, so these cases drive the merge's exact selection inside the cut bin,
including the streaming path taken when that bin holds more candidates than
a row slot.  Any choice among exactly equal scores is correct; the checks
are the parity rules (valid count, distinct in-range indices, set equal to
the oracle's up to swaps among keys tied with the k-th score).
"""

import numpy as np
import pytest
import torch

import oracle as O
import synth
from conftest import gpu_available
from oracle_side import check_topk_row

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    if not gpu_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_attention_fp8_gb300 import binding, staging
    return binding, staging


def _workload(ctxs, H, k, seed=11):
    ctxs = np.asarray(ctxs, np.int32)
    pages = (ctxs.astype(np.int64) + 63) // 64
    pool = int(pages.sum()) + 2
    perm = np.random.default_rng(seed).permutation(pool).astype(np.int32)
    bt = np.full((len(ctxs), int(pages.max())), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        bt[r, :n] = perm[at:at + n]
        at += int(n)
    q_lens = np.ones(len(ctxs), np.int32)
    return synth.Workload(91, "merge", seed, H=H, index_topk=k, num_layers=1, pattern=None,
                          freq=1, offset=2, q_lens=q_lens, seq_lens=ctxs, block_table=bt,
                          num_pages=pool, max_num_batched_tokens=len(ctxs))


def _run(B, wl, keys, q, w):
    """Write every request's keys (FP32, [ctx, 128] each) and score one query
    row per request (its last position, so it sees all of them)."""
    binding, staging = B
    meta = staging.stage_metadata(wl)
    k_cache = torch.zeros((wl.num_pages, binding.PAGE_BYTES), dtype=torch.uint8, device="cuda")
    ks = np.concatenate(keys, axis=0).astype(np.float32)
    qsl = np.zeros(wl.R + 1, np.int32)
    np.cumsum(wl.seq_lens, out=qsl[1:])
    binding.write_k(torch.from_numpy(ks).cuda(), torch.from_numpy(qsl).cuda(), meta.seq_lens,
                    meta.block_table, k_cache)
    q_fp8, q_scale = binding.quantize_fp8_blocks(torch.from_numpy(q).cuda())
    topk = torch.full((wl.T, wl.index_topk), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
    binding.score_topk(q_fp8, q_scale, torch.from_numpy(w).cuda(), k_cache, meta.query_start_loc,
                       meta.seq_lens, meta.block_table, wl.index_topk, topk, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return topk.cpu().numpy()


def _oracle_scores(keys, q, w, r):
    qc, qs = O.quantize_blocks(q)
    kc, kscale = O.quantize_blocks(keys)
    return O.index_scores(qc[r], qs[r], w[r], kc, kscale)


def _inputs(ctxs, H, seed):
    rng = np.random.default_rng(seed)
    keys = [rng.standard_normal((c, 128)).astype(np.float32) for c in ctxs]
    q = rng.standard_normal((len(ctxs), H, 128)).astype(np.float32)
    w = (rng.standard_normal((len(ctxs), H)) / np.sqrt(H)).astype(np.float32)
    return keys, q, w


def test_all_scores_equal_on_split_rows(B):
    """q = 0: every score is 0.  Row 0 (40,000 keys) is split into many pieces
    and its cut bin holds every candidate, more than a row slot."""
    ctxs, H, k = [40000, 3000, 700], 64, 2048
    wl = _workload(ctxs, H, k)
    keys, q, w = _inputs(ctxs, H, 5)
    q[:] = 0.0
    got = _run(B, wl, keys, q, w)
    for r, c in enumerate(ctxs):
        check_topk_row(got[r], np.zeros(c), k, f"row {r}")


@pytest.mark.parametrize("rank,copies", [(0, 12000), (1500, 3000)])
def test_tied_group_in_split_row(B, rank, copies):
    """One key vector replicated `copies` times into a 40,000-key row: the copies
    score exactly alike.  With the vector of the highest-scoring key the whole
    top-k is drawn from the tie (merge streaming path); with the 1500th the tie
    straddles the k-th score."""
    ctx, H, k = 40000, 64, 2048
    wl = _workload([ctx], H, k, seed=13)
    keys, q, w = _inputs([ctx], H, 17)
    s0 = _oracle_scores(keys[0], q, w, 0)
    src = int(np.argsort(-s0, kind="stable")[rank])
    dst = np.random.default_rng(19).choice(ctx, size=copies, replace=False)
    keys[0][dst] = keys[0][src]
    got = _run(B, wl, keys, q, w)
    check_topk_row(got[0], _oracle_scores(keys[0], q, w, 0), k, "row 0")
