"""The allocation-free scoring entry point (GPU).

dsa_indexer_score_topk_no_alloc serves callers that cannot allocate device
memory when they run the indexer (a server whose device memory belongs to its
own pool, a plugin host that forbids allocation in its enqueue callback).  It
uses a workspace compiled into the library instead of a caller-provided one.
This file runs last so that a failure here leaves every other test already
run; it must also pass on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

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


def _check_same_rows(got, ref, scores, T, k, where):
    """Rows must hold the same number of indices then -1, and the same index
    sets except for swaps among keys whose score is within 2e-3 x the row's
    max |score| of the k-th largest (ties can be broken either way)."""
    for t in range(T):
        g, r = got[t], ref[t]
        n = int((r >= 0).sum())
        assert np.all(r[n:] == -1) and np.all(g[n:] == -1), f"{where} row {t}: padding"
        assert np.all(g[:n] >= 0), f"{where} row {t}: valid count differs"
        diff = np.setxor1d(g[:n], r[:n])
        if diff.size:
            s = scores[t]
            vis = np.isfinite(s)
            kth = np.sort(s[vis])[::-1][n - 1]
            tol = 2e-3 * np.abs(s[vis]).max()
            assert np.all(np.abs(s[diff] - kth) <= tol), f"{where} row {t}: sets differ beyond ties"


@pytest.mark.parametrize("wid,scale,k", [(1, 0.4, 2048), (1, 0.4, 100), (0, 1.0, 32)])
def test_no_alloc_matches_workspace_entry_point(B, wid, scale, k):
    binding, staging = B
    wl = synth.make_workload(wid, scale=scale)
    wl.index_topk = k
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"])

    ref = torch.full((wl.max_num_batched_tokens, k), -7, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, k)
    # the workspace layout grows with the SM count (one scoring CTA per SM)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert ws.numel() <= binding.no_alloc_workspace_bytes(), (
        f"workload {wid} needs {ws.numel()} B of workspace with {n_sm} SMs; the built-in "
        f"workspace holds {binding.no_alloc_workspace_bytes()} B")
    sc = torch.full((wl.T, int(wl.seq_lens.max())), float("nan"), dtype=torch.float32,
                    device="cuda")
    binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"], meta.query_start_loc,
                       meta.seq_lens, meta.block_table, k, ref, ws, scores_out=sc)
    torch.cuda.synchronize()
    want = ref.cpu().numpy()
    scores = sc.cpu().numpy()
    # the FP64 oracle's rows for the same seeded inputs (quantised queries
    # recomputed by the oracle, cache keys straight from the FP32 keys)
    import oracle as O
    oc, os_ = O.quantize_blocks(wl.q(0))
    assert np.array_equal(io["q_fp8"].cpu().numpy(), oc)
    oracle = oracle_rows(wl, 0, range(wl.T), oc, os_, wl.w(0))

    # two calls in a row: the built-in workspace keeps the previous call's contents
    for call in range(2):
        got_buf = torch.full((wl.max_num_batched_tokens, k), -7, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.score_topk_no_alloc(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"],
                                    meta.query_start_loc, meta.seq_lens, meta.block_table, k,
                                    got_buf, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        got = got_buf.cpu().numpy()
        assert np.all(got[wl.T:] == -7), f"call {call}: rows beyond T were touched"
        _check_same_rows(got, want, scores, wl.T, k, f"call {call}")
        for t, ref_scores in oracle.items():
            check_topk_row(got[t], ref_scores, k, f"call {call} row {t} vs oracle")


def test_no_alloc_rejects_batches_beyond_its_workspace(B):
    binding, _ = B
    lib = binding.load()
    need = binding.workspace_bytes(8192, 64, 1, 2048)
    assert need > binding.no_alloc_workspace_bytes()
    fake = ctypes.c_void_p(0x1000)
    rc = lib.dsa_indexer_score_topk_no_alloc(fake, fake, fake, 8192, 64, fake, 16, fake, fake, 1,
                                             fake, 4, 2048, fake, 8192, None, None)
    assert rc == -3
    assert b"built-in workspace" in lib.dsa_last_error()
