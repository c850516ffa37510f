"""The scoring kernel's bounded waits give up cleanly (GPU).

Every wait of one role of the scoring kernel on another (producer, MMA
issuer, epilogue) has an iteration bound; DSA_WAIT_LIMIT lowers it, and 0
makes every such wait give up at once.  The kernel must then report
DSA_STATUS_TIMEOUT through the status word and still leave cleanly -- its own
copies and MMAs drained (those waits keep the full bound), tensor memory freed
-- so that the next call on the same context runs normally and matches the
oracle.  Nothing here faults, traps or hangs the GPU: the failure is a wait
that stops early.
"""

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


@pytest.mark.parametrize("wid,scale", [(0, 1.0), (1, 0.2), (4, 1 / 64)])
def test_waits_time_out_then_the_next_call_is_correct(B, monkeypatch, wid, scale):
    """Tiny prefill (one group per CTA), a decode batch scored into workspace
    rows, and 1M-context rows scaled to 16K keys (rows cut into many pieces
    that share a histogram and merge)."""
    binding, staging = B
    wl = synth.make_workload(wid, scale=scale)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"])
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk, max_ctx=wl.max_blocks * 64)

    def run():
        topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                          device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"],
                           meta.query_start_loc, meta.seq_lens, meta.block_table, wl.index_topk,
                           topk, ws, status=st)
        torch.cuda.synchronize()
        return topk.cpu().numpy(), st.item()

    monkeypatch.setenv("DSA_WAIT_LIMIT", "0")
    _, status = run()
    assert status & binding.STATUS_TIMEOUT, f"status {status}: no wait gave up"
    monkeypatch.delenv("DSA_WAIT_LIMIT")
    got, status = run()
    assert status == 0
    oc, os_ = O.quantize_blocks(wl.q(0))
    ref = oracle_rows(wl, 0, range(wl.T), oc, os_, wl.w(0))
    for t, s in ref.items():
        check_topk_row(got[t], s, wl.index_topk, f"row {t}")
    assert np.all(got[wl.T:] == -7)
