"""Layer stacks and full-size workloads through dsa_layer_stack_run (GPU).

Full-size workloads run in the launch configuration the benchmark uses and
are checked on sampled rows the oracle computes one by one; the layer-stack
tests replay the IndexCache F/S schedules (freq/offset and explicit
patterns) against the oracle at reduced context lengths.
"""

import numpy as np
import pytest
import torch

import oracle as O
import synth
from conftest import gpu_available
from oracle_side import check_scores, check_topk_row, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    if not gpu_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_attention_fp8_gb300 import binding, staging
    return binding, staging


def _run_stack(B, wl, pattern, freq, offset, num_layers):
    binding, staging = B
    meta = staging.stage_metadata(wl)
    full = [O.layer_is_full(l, pattern, freq, offset) for l in range(num_layers)]
    layers = [staging.stage_layer(wl, l, meta) if f else None for l, f in enumerate(full)]
    topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                      device="cuda")
    outs = [torch.full((wl.T, wl.index_topk), -9, dtype=torch.int32, device="cuda")
            for _ in range(num_layers)]
    slots = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
    binding.layer_stack_run(layers, pattern, freq, offset, wl.H, meta.query_start_loc,
                            meta.seq_lens, meta.block_table, wl.num_pages, wl.index_topk, topk, ws,
                            per_layer_out=outs, slot_mapping=slots, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(slots.cpu().numpy(),
                          O.slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table))
    return full, layers, [o.cpu().numpy() for o in outs], topk.cpu().numpy()


def _sample_rows(wl, n, seed=0):
    rng = np.random.default_rng(seed)
    qsl = wl.query_start_loc
    rows = {0, wl.T - 1}
    for r in rng.choice(wl.R, size=min(n, wl.R), replace=False):
        rows.add(int(qsl[r + 1]) - 1)            # last row of the request: longest context
        rows.add(int(rng.integers(qsl[r], qsl[r + 1])))
    return sorted(rows)


def _check_rows(wl, layer, io, got, rows):
    qc, qs = io["q_fp8"].cpu().numpy(), io["q_scale"].cpu().numpy()
    oc, os_ = O.quantize_blocks(wl.q(layer))
    assert np.array_equal(qc, oc) and np.array_equal(qs, os_)
    ref = oracle_rows(wl, layer, rows, oc, os_, wl.w(layer))
    for t, s in ref.items():
        check_topk_row(got[t], s, wl.index_topk, f"layer {layer} row {t}")


def _check_shared(full, outs):
    last = None
    for l, f in enumerate(full):
        if f:
            last = l
        else:
            assert np.array_equal(outs[l], outs[last]), f"S layer {l} != F layer {last}"


# ----------------------------------------------------------------------------
# schedules at reduced size: every F layer against the oracle, S layers equal
# ----------------------------------------------------------------------------

def test_tiny_prefill_stack_fs(B):
    wl = synth.make_workload(0)
    full, layers, outs, buf = _run_stack(B, wl, wl.pattern, wl.freq, wl.offset, wl.num_layers)
    assert full == [True, False]
    _check_rows(wl, 0, layers[0], outs[0], range(wl.T))
    _check_shared(full, outs)
    assert np.array_equal(buf[:wl.T], outs[1])


def test_freq4_offset2_stack_61_layers(B):
    wl = synth.make_workload(3, scale=1 / 64)
    wl.index_topk = 64
    full, layers, outs, _ = _run_stack(B, wl, None, 4, 2, 61)
    assert [l for l, f in enumerate(full) if f] == [0, 1, 5, 9, 13, 17, 21, 25, 29, 33, 37, 41,
                                                     45, 49, 53, 57]
    rows = _sample_rows(wl, 6)
    for l, f in enumerate(full):
        if f and l in (0, 1, 29, 57):
            _check_rows(wl, l, layers[l], outs[l], rows)
    _check_shared(full, outs)


def test_explicit_pattern_stack_78_layers(B):
    wl = synth.make_workload(4, scale=1 / 2048)       # 4 requests x 513 cached tokens
    wl.index_topk = 128
    assert wl.pattern.count("F") == 21 and wl.pattern[:2] == "FF"
    full, layers, outs, _ = _run_stack(B, wl, wl.pattern, wl.freq, wl.offset, wl.num_layers)
    assert full == [c == "F" for c in wl.pattern]
    for l, f in enumerate(full):
        if f:
            _check_rows(wl, l, layers[l], outs[l], range(wl.T))
    _check_shared(full, outs)


def test_pattern_shorter_than_stack(B):
    """Layers beyond the pattern (e.g. MTP layers) run as F."""
    wl = synth.make_workload(1, scale=0.05)
    wl.index_topk = 32
    full, layers, outs, _ = _run_stack(B, wl, "FS", 1, 2, 4)
    assert full == [True, False, True, True]
    for l in (0, 2, 3):
        _check_rows(wl, l, layers[l], outs[l], range(wl.T))
    _check_shared(full, outs)


# ----------------------------------------------------------------------------
# full-size workloads, sampled rows
# ----------------------------------------------------------------------------

def test_full_prefix_hit_chunked_prefill(B):
    wl = synth.make_workload(2)                       # 16384 cached + 8192 new, H=64, k=2048
    full, layers, outs, _ = _run_stack(B, wl, "FS", 1, 2, 2)
    rows = sorted({0, 1, 63, 64, 1000, 4095, 4096, 6001, 8190, 8191}
                  | set(np.random.default_rng(3).integers(0, wl.T, 8).tolist()))
    _check_rows(wl, 0, layers[0], outs[0], rows)
    _check_shared(full, outs)


def test_full_mixed_batch(B):
    """The mixed batch at full size (256 decode rows with contexts up to 65,536
    + 4 prefill chunks of 1024) through its real 61-layer stack, freq 4 and
    offset 2 (16 F layers): sampled rows of the first, a middle and the last F
    layer against the oracle; every S layer equals the F layer before it."""
    wl = synth.make_workload(3)
    full, layers, outs, _ = _run_stack(B, wl, None, wl.freq, wl.offset, wl.num_layers)
    f_layers = [l for l, f in enumerate(full) if f]
    assert len(f_layers) == 16 and f_layers[:3] == [0, 1, 5] and f_layers[-1] == 57
    _check_rows(wl, f_layers[0], layers[f_layers[0]], outs[f_layers[0]], _sample_rows(wl, 8))
    for l in (f_layers[len(f_layers) // 2], f_layers[-1]):
        _check_rows(wl, l, layers[l], outs[l], _sample_rows(wl, 3, seed=l))
    _check_shared(full, outs)


def test_full_mtp_decode_stack(B):
    wl = synth.make_workload(5)                       # 64 requests x 2 rows, ctx 1024..8192
    full, layers, outs, _ = _run_stack(B, wl, None, 1, 2, 2)
    _check_rows(wl, 0, layers[0], outs[0], range(wl.T))
    _check_rows(wl, 1, layers[1], outs[1], _sample_rows(wl, 8))


def test_full_long_context_decode(B):
    """The 1M-context decode batch at full size (4 x (1,048,576 + 1) tokens)
    through its real 78-layer stack with the seeded 21-F pattern: every row of
    the first F layer, one row each of a middle and the last F layer against
    the oracle; every S layer equals the F layer before it."""
    wl = synth.make_workload(4)
    full, layers, outs, _ = _run_stack(B, wl, wl.pattern, wl.freq, wl.offset, wl.num_layers)
    f_layers = [l for l, f in enumerate(full) if f]
    assert len(f_layers) == 21 and f_layers[:2] == [0, 1]
    _check_rows(wl, f_layers[0], layers[f_layers[0]], outs[f_layers[0]], range(wl.T))
    _check_rows(wl, f_layers[10], layers[f_layers[10]], outs[f_layers[10]], [1])
    _check_rows(wl, f_layers[-1], layers[f_layers[-1]], outs[f_layers[-1]], [3])
    _check_shared(full, outs)


def test_full_prefix_hit_scores_on_sampled_rows(B):
    """The prefix-hit chunked prefill at full size (8192 rows x up to 24,576
    keys) through dsa_indexer_score_topk with the debug score dump: every
    visible score of sampled rows within 2e-3 x the row's max |score| of the
    oracle, and the rows' index sets."""
    binding, staging = B
    wl = synth.make_workload(2)
    meta = staging.stage_metadata(wl)
    io = staging.stage_layer(wl, 0, meta)
    binding.write_k(io["k"], meta.query_start_loc, meta.seq_lens, meta.block_table, io["k_cache"])
    topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                      device="cuda")
    ld = int(wl.seq_lens.max())
    sc = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device="cuda")
    ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.score_topk(io["q_fp8"], io["q_scale"], io["w"], io["k_cache"], meta.query_start_loc,
                       meta.seq_lens, meta.block_table, wl.index_topk, topk, ws, scores_out=sc,
                       status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = sorted({0, 1, 127, 128, 2047, 4096, 6001, 8190, 8191}
                  | set(np.random.default_rng(11).integers(0, wl.T, 7).tolist()))
    got = topk.cpu().numpy()
    assert np.all(got[wl.T:] == -7)
    oc, os_ = O.quantize_blocks(wl.q(0))
    ref = oracle_rows(wl, 0, rows, oc, os_, wl.w(0))
    for t, s in ref.items():
        row = sc[t, :s.shape[0]].cpu().numpy()
        check_scores(row, s, f"row {t}")
        check_topk_row(got[t], s, wl.index_topk, f"row {t}")
