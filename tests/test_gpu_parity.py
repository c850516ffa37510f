"""GPU path vs the CPU oracle, through the C ABI (needs a GB300).

Cache bytes, slot mappings, -1 padding and valid counts must match bit for
bit; scores within 2e-3 x the row's max |score|; top-k index sets equal up to
swaps among keys whose oracle scores lie within that tolerance of the k-th
largest.  Sizes here finish on the oracle in seconds while spanning several
key tiles, split rows, ragged tails and the degenerate cases.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from conftest import gpu_available
from oracle_side import check_scores, check_topk_row, oracle_cache, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    if not gpu_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_attention_fp8_gb300 import binding, staging
    return binding, staging


def _wl(wid, scale=1.0, **over):
    wl = synth.make_workload(wid, seed=0, scale=scale)
    return dataclasses.replace(wl, **over) if over else wl


def _custom(q_lens, seq_lens, H=4, k=32, pool_extra=3, seed=7, wid=9):
    q_lens = np.asarray(q_lens, np.int32)
    seq_lens = np.asarray(seq_lens, np.int32)
    pages = (seq_lens.astype(np.int64) + 63) // 64
    pool = int(pages.sum()) + pool_extra
    perm = np.random.default_rng(seed).permutation(pool).astype(np.int32)
    bt = np.full((len(q_lens), max(1, int(pages.max()))), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        bt[r, :n] = perm[at:at + n]
        at += int(n)
    return synth.Workload(wid, "custom", seed, H=H, index_topk=k, num_layers=1, pattern=None,
                          freq=1, offset=2, q_lens=q_lens, seq_lens=seq_lens, block_table=bt,
                          num_pages=pool, max_num_batched_tokens=int(q_lens.sum()) + 5)


def _run_layer(B, wl, layer=0, scores=True, status=None, topk_fill=-7):
    binding, staging = B
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, layer, meta)
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"],
                    status=status)
    topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), topk_fill, dtype=torch.int32,
                      device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
    sc = None
    if scores:
        sc = torch.full((wl.T, int(wl.seq_lens.max())), float("nan"), dtype=torch.float32,
                        device="cuda")
    binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"], meta.query_start_loc,
                       meta.seq_lens, meta.block_table, wl.index_topk, topk, ws, scores_out=sc,
                       status=status)
    torch.cuda.synchronize()
    return io, topk.cpu().numpy(), (None if sc is None else sc.cpu().numpy())


def _check_layer(wl, io, topk, sc, rows=None, layer=0):
    qc = io["q_fp8"].cpu().numpy()
    qs = io["q_scale"].cpu().numpy()
    oc, os_ = O.quantize_blocks(wl.q(layer))
    assert np.array_equal(qc, oc) and np.array_equal(qs, os_), "query quantisation differs"
    rows = range(wl.T) if rows is None else rows
    ref = oracle_rows(wl, layer, rows, oc, os_, wl.w(layer))
    for t, s in ref.items():
        if sc is not None:
            check_scores(sc[t], s, f"row {t}")
        check_topk_row(topk[t], s, wl.index_topk, f"row {t}")
    assert np.all(topk[wl.T:] == -7), "rows beyond T were touched"


# ----------------------------------------------------------------------------

def test_quantizer_bit_exact(B):
    binding, _ = B
    rng = np.random.default_rng(0)
    x = rng.standard_normal((4096, 128)).astype(np.float32)
    x[:512] *= np.float32(1e-3)
    x[512:1024] *= np.float32(1e4)
    x[1024] = 0.0
    x[1025] = -0.0
    x[1026] = 0.0
    x[1026, 17] = -3.0
    x[1027] *= np.float32(1e-38)                        # subnormal FP32 inputs
    x[1028, :] = np.float32(448.0) * (np.arange(128) / 127.0).astype(np.float32)
    pos = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    x[1029, :126] = ((pos[:-1] + pos[1:]) / 2)[:126].astype(np.float32)  # E4M3 midpoints
    x[1029, 126:] = 448.0                               # scale exactly 1
    codes, scales = binding.quantize_fp8_blocks(torch.from_numpy(x).cuda())
    oc, os_ = O.quantize_blocks(x)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("wid,scale", [(0, 1.0), (1, 0.1), (3, 1 / 32), (2, 1 / 16)])
def test_cache_write_bit_exact(B, wid, scale):
    binding, staging = B
    wl = _wl(wid, scale)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta, cache_fill_byte=0xA5)
    slots = torch.full((wl.T,), -9, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"],
                    slot_mapping=slots, status=st)
    torch.cuda.synchronize()
    ref = np.full((wl.num_pages, O.PAGE_BYTES), 0xA5, np.uint8)
    for r in range(wl.R):
        P = int(wl.prefix_lens[r])
        if P:
            O.write_k_cache(ref, wl.k_prefix(0, r),
                            O.slot_mapping(np.array([0, P]), np.array([P]), wl.block_table[r:r + 1]))
    ref_slots = O.slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table)
    O.write_k_cache(ref, wl.k_new(0), ref_slots)
    assert st.item() == 0
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    got = io["k_cache"].cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} cache bytes differ, first at page/byte {bad[0]}"


@pytest.mark.parametrize("wid,scale,over", [
    (0, 1.0, {}),                                   # tiny prefill, H=4, k=32
    (1, 0.08, {}),                                  # decode, contexts below k: every key returned
    (1, 0.5, {}),                                   # decode, contexts 512..4096 < k=2048 partly
    (1, 0.2, {"index_topk": 100}),                  # decode with selection + compaction
    (3, 1 / 64, {"index_topk": 64}),                # mixed prefill + decode rows
    (2, 1 / 32, {"index_topk": 128}),               # prefix-hit chunked prefill
    (5, 0.25, {}),                                  # MTP decode: 2 rows per request
    (5, 1.0, {"index_topk": 300}),                  # MTP decode, full contexts, selection
])
def test_scores_and_topk(B, wid, scale, over):
    wl = _wl(wid, scale, **over)
    io, topk, sc = _run_layer(B, wl)
    _check_layer(wl, io, topk, sc)
    # the production path (no score dump) selects the same sets
    io2, topk2, _ = _run_layer(B, wl, scores=False)
    _check_layer(wl, io2, topk2, None)


def test_full_decode_config_all_rows(B):
    """64 decode requests, contexts 1024..8192, H=64, k=2048 (all rows)."""
    wl = _wl(1)
    io, topk, sc = _run_layer(B, wl)
    _check_layer(wl, io, topk, sc)


@pytest.mark.parametrize("k", [1, 2, 31, 130])
def test_small_k_and_ties(B, k):
    wl = _custom([3, 1, 40], [700, 129, 300], H=8, k=k)
    io, topk, sc = _run_layer(B, wl)
    _check_layer(wl, io, topk, sc)


def test_degenerate_contexts(B):
    # contexts of 1, 63, 64, 65, 127, 128, 129 keys; a request with no new rows;
    # a request whose rows all see fewer keys than k
    wl = _custom([1, 1, 1, 0, 1, 1, 1, 5], [1, 63, 64, 10, 65, 127, 128, 133], H=16, k=64)
    io, topk, sc = _run_layer(B, wl)
    _check_layer(wl, io, topk, sc)


def test_zero_query_rows_is_a_noop(B):
    binding, staging = B
    wl = _custom([2], [10], H=4, k=8)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    topk = torch.full((4, 8), 5, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(2, 4, 1, 8)
    binding.score_topk(io["q_fp8"][:0], io["q_scale"][:0], io["w"][:0], io["k_cache"],
                       torch.zeros(2, dtype=torch.int32, device="cuda"), meta.seq_lens[:1] * 0,
                       meta.block_table, 8, topk, ws)
    torch.cuda.synchronize()
    assert torch.all(topk == 5)


def test_bad_page_is_reported_not_faulted(B):
    binding, staging = B
    wl = _custom([1, 1], [200, 150], H=4, k=16)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"])
    bt = meta.block_table.clone()
    bt[1, 1] = wl.num_pages + 1000      # out of the pool
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.full((wl.max_num_batched_tokens, 16), -7, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, 16)
    binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"], meta.query_start_loc,
                       meta.seq_lens, bt, 16, topk, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() & binding.STATUS_BAD_PAGE
    got = topk.cpu().numpy()
    # request 0 is unaffected
    ref = oracle_rows(wl, 0, [0], *O.quantize_blocks(wl.q(0)), wl.w(0))
    check_topk_row(got[0], ref[0], 16, "row 0")
    # request 1 returns only keys outside the bad page, all distinct and in range
    row = got[1][got[1] >= 0]
    assert np.unique(row).size == row.size and np.all((row < 64) | (row >= 128))


def test_bad_metadata_is_reported(B):
    binding, staging = B
    wl = _custom([2, 1], [100, 50], H=4, k=8)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"])
    sl = meta.seq_lens.clone()
    sl[0] = 1                           # fewer context tokens than new rows
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.full((wl.max_num_batched_tokens, 8), 3, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, 8)
    binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"], meta.query_start_loc,
                       sl, meta.block_table, 8, topk, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() & binding.STATUS_BAD_METADATA
    got = topk.cpu().numpy()
    assert np.all(got[0:2] == -1)
    ref = oracle_rows(wl, 0, [2], *O.quantize_blocks(wl.q(0)), wl.w(0))
    check_topk_row(got[2], ref[2], 8, "row 2")


def test_page_permutation_invariance(B):
    wl_a = _custom([4, 1], [300, 500], H=8, k=40, seed=1)
    # same data (seed), different page permutation
    wl_b = dataclasses.replace(_custom([4, 1], [300, 500], H=8, k=40, seed=2), seed=wl_a.seed)
    assert not np.array_equal(wl_a.block_table, wl_b.block_table)
    _, ta, sa = _run_layer(B, wl_a)
    _, tb, sb = _run_layer(B, wl_b)
    np.testing.assert_array_equal(sa, sb)
    for t in range(wl_a.T):
        assert set(ta[t].tolist()) == set(tb[t].tolist())
