"""Decode rows scored into the workspace and selected by the row kernel (GPU).

With a workspace sized for max_ctx <= 8192, a decode batch skips the
in-kernel selection: the scoring kernel writes the rows' keys to the
workspace and a second kernel selects each row's top-k.  A batch with a row
beyond the bound keeps the in-kernel path.  Same parity bar as every scoring path: -1 padding and valid counts
exact, sets equal to the oracle's up to swaps among keys tied with the k-th.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from conftest import gpu_available
from oracle_side import check_topk_row, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    if not gpu_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_attention_fp8_gb300 import binding, staging
    return binding, staging


def _run(B, wl, max_ctx, status_expected=0, bt_override=None):
    binding, staging = B
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    binding.write_k_compressed(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table,
                               io["k_cache"], wl.compress_ratio)
    topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                      device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk, max_ctx=max_ctx)
    assert ws.numel() > binding.workspace_bytes(wl.T, wl.H, wl.R, wl.index_topk)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = meta.block_table if bt_override is None else bt_override
    binding.score_topk_compressed(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"],
                                  meta.query_start_loc, meta.seq_lens, bt, wl.compress_ratio,
                                  wl.index_topk, topk, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == status_expected
    return io, topk.cpu().numpy()


def _check(wl, io, topk, rows=None):
    qc, qs = io["q_fp8"].cpu().numpy(), io["q_scale"].cpu().numpy()
    ref = oracle_rows(wl, 0, range(wl.T) if rows is None else rows, qc, qs, wl.w(0))
    for t, s in ref.items():
        check_topk_row(topk[t], s, wl.index_topk, f"row {t}")
    assert np.all(topk[wl.T:] == -7), "rows beyond T were touched"


@pytest.mark.parametrize("scale,k,max_ctx", [
    (0.5, 2048, 8192),      # every row in the workspace; rows of 512..4096 keys vs k = 2048
    (1.0, 300, 8192),       # full contexts, selection of 300
    (1.0, 2048, 4096),      # a row above 4096 keys: the batch keeps the in-kernel path
])
def test_batched_decode_rows(B, scale, k, max_ctx):
    wl = dataclasses.replace(synth.make_workload(1, scale=scale), index_topk=k)
    io, topk = _run(B, wl, max_ctx)
    _check(wl, io, topk)


def test_compressed_decode_rows(B):
    """Compressed entries (one per 4 tokens): 512..4096 entries per row; the
    bound is in entries' terms the caller knows (the largest entry count)."""
    wl = synth.make_workload(6, scale=1 / 8)
    io, topk = _run(B, wl, int(wl.entries.max()))
    _check(wl, io, topk)


def test_full_decode_stack_uses_rows(B):
    """The bench configuration: IndexerStep sizes its workspace for the
    block table's contexts, so the 4-layer batched decode stack runs every
    row through the row kernel; sampled rows of the last layer against the
    oracle."""
    binding, staging = B
    from dsa_sparse_attention_fp8_gb300.step import IndexerStep
    wl = synth.make_workload(1)
    meta = staging.stage_metadata(wl)
    caches, ios = [], []
    for l in range(wl.num_layers):
        io = staging.stage_layer(wl, l, meta)
        caches.append(io["k_cache"])
        ios.append(io)
    step = IndexerStep(num_layers=wl.num_layers, pattern=wl.pattern, freq=wl.freq,
                       offset=wl.offset, H=wl.H, index_topk=wl.index_topk, T=wl.T, R=wl.R,
                       max_blocks=wl.max_blocks, num_pages=wl.num_pages,
                       max_num_batched_tokens=wl.max_num_batched_tokens, k_caches=caches)
    step.set_metadata(meta.query_start_loc, meta.seq_lens, meta.block_table)
    for l, io in enumerate(ios):
        step.set_layer(l, io["k"], io["q_fp8"], io["q_scale"], io["w"])
    step.launch()
    torch.cuda.synchronize()
    assert step.status.item() == 0
    assert step.launches_per_step == 1 + 3 * wl.num_layers   # plan; write, score, rows per layer
    got = step.topk.cpu().numpy()
    last = wl.num_layers - 1
    qc, qs = ios[last]["q_fp8"].cpu().numpy(), ios[last]["q_scale"].cpu().numpy()
    rows = sorted({0, wl.T - 1, *np.random.default_rng(3).integers(0, wl.T, 8).tolist()})
    ref = oracle_rows(wl, last, rows, qc, qs, wl.w(last))
    for t, s in ref.items():
        check_topk_row(got[t], s, wl.index_topk, f"row {t}")


def test_bad_page_on_a_workspace_row(B):
    """A key on a page outside the pool is skipped and reported, as on the
    in-kernel path: the row returns only keys of valid pages."""
    binding, staging = B
    wl = dataclasses.replace(synth.make_workload(1, scale=0.1), index_topk=64)
    meta = staging.stage_metadata(wl)
    r = int(np.argmax(wl.seq_lens))           # a request with at least two pages
    assert wl.seq_lens[r] > 128
    bt = meta.block_table.clone()
    bt[r, 1] = wl.num_pages + 500
    io, topk = _run(B, wl, 1024, status_expected=binding.STATUS_BAD_PAGE, bt_override=bt)
    row = topk[r][topk[r] >= 0]              # decode: row r belongs to request r
    assert row.size > 0 and np.unique(row).size == row.size
    assert np.all((row < 64) | (row >= 128))
    _check(wl, io, topk, rows=[t for t in range(wl.T) if t != r])
