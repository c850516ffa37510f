"""Compressed indexer cache, one entry per compress_ratio tokens (GPU).

"HBM 索引架构设计" §5.2: a token holds a cache entry only when
(pos + 1) % ratio == 0, at entry pos // ratio; the others get slot -1 and
write nothing.  A row at pos ranks the (pos + 1) // ratio entries completed
at or before it and returns entry numbers; a row that sees none is all -1.
Same bars as the uncompressed parity tests: cache bytes, slots, -1 padding
and valid counts bit-exact; scores within 2e-3 x the row's max |score|;
top-k sets equal up to swaps among keys tied with the k-th score.
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


def _custom(q_lens, seq_lens, ratio, H=16, k=64, seed=3, wid=9):
    """A batch whose block table covers each request's seq_len // ratio entries."""
    q_lens = np.asarray(q_lens, np.int32)
    seq_lens = np.asarray(seq_lens, np.int32)
    pages = np.maximum(1, (seq_lens.astype(np.int64) // ratio + 63) // 64)
    pool = int(pages.sum()) + 2
    perm = np.random.default_rng(seed).permutation(pool).astype(np.int32)
    bt = np.full((len(q_lens), int(pages.max())), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        bt[r, :n] = perm[at:at + n]
        at += int(n)
    return synth.Workload(wid, "custom_compressed", seed, H=H, index_topk=k, num_layers=1,
                          pattern=None, freq=1, offset=2, q_lens=q_lens, seq_lens=seq_lens,
                          block_table=bt, num_pages=pool,
                          max_num_batched_tokens=int(q_lens.sum()) + 3, compress_ratio=ratio)


def _run(B, wl, layer=0, scores=True):
    binding, staging = B
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, layer, meta, cache_fill_byte=0x5A)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.full((wl.T,), -9, dtype=torch.int64, device="cuda")
    binding.write_k_compressed(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table,
                               io["k_cache"], wl.compress_ratio, slot_mapping=slots, status=st)
    topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                      device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
    sc = None
    if scores:
        sc = torch.full((wl.T, max(1, int(wl.entries.max()))), float("nan"), dtype=torch.float32,
                        device="cuda")
    binding.score_topk_compressed(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"],
                                  meta.query_start_loc, meta.seq_lens, meta.block_table,
                                  wl.compress_ratio, wl.index_topk, topk, ws, scores_out=sc,
                                  status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return (io, slots.cpu().numpy(), topk.cpu().numpy(),
            None if sc is None else sc.cpu().numpy())


def _check(wl, io, topk, sc, rows=None, layer=0):
    qc, qs = io["q_fp8"].cpu().numpy(), io["q_scale"].cpu().numpy()
    rows = range(wl.T) if rows is None else rows
    ref = oracle_rows(wl, layer, rows, qc, qs, wl.w(layer))
    for t, s in ref.items():
        if sc is not None and s.size:
            check_scores(sc[t], s, f"row {t}")
        check_topk_row(topk[t], s, wl.index_topk, f"row {t}")
    assert np.all(topk[wl.T:] == -7), "rows beyond T were touched"


@pytest.mark.parametrize("ratio", [4, 128])
def test_compressed_write_bit_exact(B, ratio):
    """Prefill and decode rows of several requests: the cache equals the
    oracle's byte for byte (tokens without an entry leave the 0x5A fill) and
    the slots equal the oracle's compressed mapping."""
    wl = _custom([600, 1, 3, 300], [600, 9000, 140, 2000], ratio)
    io, slots, _, _ = _run(B, wl, scores=False)
    want_slots = O.compressed_slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table, ratio)
    assert np.array_equal(slots, want_slots)
    assert np.count_nonzero(want_slots >= 0) < wl.T
    ref = oracle_cache(wl, 0, fill=0x5A)
    got = io["k_cache"].cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} cache bytes differ, first at page/byte {bad[0]}"


@pytest.mark.parametrize("ratio,k", [(4, 64), (4, 1000), (128, 16), (3, 7)])
def test_compressed_prefill_rows(B, ratio, k):
    """Chunked prefill from position 0 (the first ratio - 1 rows see no entry),
    a prefix-hit chunk, a ragged tail and decode rows; every row checked."""
    wl = _custom([700, 257, 1, 1, 64], [700, 3000, 4 * ratio - 1, 4 * ratio, 6000], ratio, k=k)
    io, _, topk, sc = _run(B, wl)
    _check(wl, io, topk, sc)
    req, pos = O.token_positions(wl.query_start_loc, wl.seq_lens)
    empty = O.visible_entries(pos, ratio) == 0
    assert empty.any() and np.all(topk[:wl.T][empty] == -1)


@pytest.mark.parametrize("scale,k", [(1 / 8, 2048), (1 / 8, 300)])
def test_compressed_decode_rows(B, scale, k):
    """The compressed decode batch (64 requests, one entry per 4 tokens) at
    oracle-friendly contexts: entries 512..4096 against k = 2048 and 300."""
    wl = dataclasses.replace(synth.make_workload(6, scale=scale), index_topk=k)
    io, _, topk, sc = _run(B, wl)
    _check(wl, io, topk, sc)


def test_compressed_decode_full_size_sampled_rows(B):
    """The full compressed decode batch (contexts 16K-128K, entries 4K-32K) in
    the production configuration (no score dump), sampled rows."""
    wl = synth.make_workload(6)
    io, _, topk, _ = _run(B, wl, scores=False)
    rows = sorted({0, wl.T - 1, *np.random.default_rng(6).integers(0, wl.T, 6).tolist()})
    _check(wl, io, topk, None, rows=rows)


def test_compressed_stack_matches_oracle(B):
    """A compressed F/S stack through dsa_layer_stack_run_compressed: F layers
    against the oracle's rows, S layers equal to the last F layer's."""
    binding, staging = B
    wl = dataclasses.replace(synth.make_workload(6, scale=1 / 16), index_topk=256)
    meta = staging.stage_metadata(wl)
    pattern, L = "FSF", 3
    ios = []
    for l in range(L):
        ios.append(staging.stage_layer(wl, l, meta) if pattern[l] == "F" else None)
    topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                      device="cuda")
    per = [torch.full((wl.T, wl.index_topk), -9, dtype=torch.int32, device="cuda")
           for _ in range(L)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
    binding.layer_stack_run_compressed(ios, pattern, 1, 2, wl.H, meta.query_start_loc,
                                       meta.seq_lens, meta.block_table, wl.num_pages,
                                       wl.index_topk, topk, ws, per_layer_out=per, status=st,
                                       compress_ratio=wl.compress_ratio)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = [p.cpu().numpy() for p in per]
    assert np.array_equal(got[1], got[0])
    for l in (0, 2):
        qc, qs = ios[l]["q_fp8"].cpu().numpy(), ios[l]["q_scale"].cpu().numpy()
        ref = oracle_rows(wl, l, range(wl.T), qc, qs, wl.w(l))
        for t, s in ref.items():
            check_topk_row(got[l][t], s, wl.index_topk, f"layer {l} row {t}")


def test_compressed_ratio_one_matches_plain_entry_points(B):
    """compress_ratio 1 runs the plain cache: same slots, cache and top-k as
    dsa_indexer_write_k / dsa_indexer_score_topk."""
    binding, staging = B
    wl = synth.make_workload(3, scale=1 / 64)
    wl = dataclasses.replace(wl, index_topk=64)
    meta = staging.stage_metadata(wl)
    outs = []
    for compressed in (False, True):
        io = staging.stage_layer(wl, 0, meta)
        slots = torch.empty(wl.T, dtype=torch.int64, device="cuda")
        topk = torch.full((wl.max_num_batched_tokens, 64), -7, dtype=torch.int32, device="cuda")
        ws = binding.alloc_workspace(wl.T, wl.H, wl.R, 64)
        if compressed:
            binding.write_k_compressed(io["k"], meta.query_start_loc, meta.seq_lens,
                                       meta.block_table, io["k_cache"], 1, slot_mapping=slots)
            binding.score_topk_compressed(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"],
                                          meta.query_start_loc, meta.seq_lens, meta.block_table,
                                          1, 64, topk, ws)
        else:
            binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table,
                            io["k_cache"], slot_mapping=slots)
            binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"],
                               meta.query_start_loc, meta.seq_lens, meta.block_table, 64, topk, ws)
        torch.cuda.synchronize()
        outs.append((slots.cpu().numpy(), io["k_cache"].cpu().numpy(),
                     np.sort(topk.cpu().numpy(), axis=1)))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_compressed_bad_ratio_is_an_argument_error(B):
    binding, staging = B
    wl = _custom([4], [40], 4)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    with pytest.raises(binding.DsaError):
        binding.write_k_compressed(io["k"], meta.query_start_loc, meta.seq_lens,
                                   meta.block_table, io["k_cache"], 0)
