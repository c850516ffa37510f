"""BF16 inputs with the query quantisation fused into the cache-write launch (GPU).

BF16 widens to FP32 exactly, so the BF16 path must produce exactly what the
FP32 path produces on the widened values: cache bytes, slots, query codes and
scales bit-exact against the oracle, and the same top-k sets through the layer
stack.
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


@pytest.mark.parametrize("wid,scale", [(1, 0.2), (3, 1 / 32), (5, 0.25)])
def test_write_k_bf16_and_fused_query_quantisation(B, wid, scale):
    binding, staging = B
    wl = synth.make_workload(wid, scale=scale)
    meta = staging.stage_metadata(wl)
    k_cache = torch.full((wl.num_pages, binding.PAGE_BYTES), 0x5A, dtype=torch.uint8,
                         device="cuda")
    k16 = torch.from_numpy(wl.k_new(0)).cuda().bfloat16()
    q16 = torch.from_numpy(wl.q(0)).cuda().bfloat16()
    q_fp8 = torch.full((wl.T, wl.H, 128), 0x77, dtype=torch.uint8, device="cuda")
    q_scale = torch.full((wl.T, wl.H), -1.0, dtype=torch.float32, device="cuda")
    slots = torch.full((wl.T,), -9, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.write_k_bf16(k16, meta.query_start_loc, meta.seq_lens, meta.block_table, k_cache,
                         q=q16, q_fp8=q_fp8, q_scale=q_scale, slot_mapping=slots, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    k_wide = k16.float().cpu().numpy()
    q_wide = q16.float().cpu().numpy()
    ref_slots = O.slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    ref = np.full((wl.num_pages, O.PAGE_BYTES), 0x5A, np.uint8)
    O.write_k_cache(ref, k_wide, ref_slots)
    assert np.array_equal(k_cache.cpu().numpy(), ref)
    oc, os_ = O.quantize_blocks(q_wide)
    assert np.array_equal(q_fp8.cpu().numpy(), oc)
    assert np.array_equal(q_scale.cpu().numpy(), os_)


def test_stack_bf16_matches_oracle_and_fp32_path(B):
    binding, staging = B
    wl = synth.make_workload(5, scale=0.3)          # MTP decode, 2 rows per request
    wl.index_topk = 256
    meta = staging.stage_metadata(wl)
    pattern, L = "FSF", 3
    caches32, caches16, io32, io16, wides = [], [], [], [], []
    for l in range(L):
        if pattern[l] == "S":
            io32.append(None)
            io16.append(None)
            wides.append(None)
            continue
        c32 = torch.zeros((wl.num_pages, binding.PAGE_BYTES), dtype=torch.uint8, device="cuda")
        staging.fill_prefix(wl, l, meta, c32)
        c16 = c32.clone()
        k16 = torch.from_numpy(wl.k_new(l)).cuda().bfloat16()
        q16 = torch.from_numpy(wl.q(l)).cuda().bfloat16()
        w = torch.from_numpy(wl.w(l)).cuda()
        qc, qs = binding.quantize_fp8_blocks(q16.float())
        io32.append({"k": k16.float(), "q_fp8": qc, "q_scale": qs, "w": w, "k_cache": c32})
        io16.append({"k": k16, "q": q16, "w": w, "k_cache": c16,
                     "q_fp8": torch.empty_like(qc), "q_scale": torch.empty_like(qs)})
        wides.append((k16.float().cpu().numpy(), q16.float().cpu().numpy(), wl.w(l)))
    outs = {}
    for name, fn, ios in (("fp32", binding.layer_stack_run, io32),
                          ("bf16", binding.layer_stack_run_bf16, io16)):
        topk = torch.full((wl.max_num_batched_tokens, wl.index_topk), -7, dtype=torch.int32,
                          device="cuda")
        per = [torch.full((wl.T, wl.index_topk), -9, dtype=torch.int32, device="cuda")
               for _ in range(L)]
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = binding.alloc_workspace(wl.T, wl.H, wl.R, wl.index_topk)
        fn(ios, pattern, 1, 2, wl.H, meta.query_start_loc, meta.seq_lens, meta.block_table,
           wl.num_pages, wl.index_topk, topk, ws, per_layer_out=per, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs[name] = [np.sort(p.cpu().numpy(), axis=1) for p in per]
    for l in range(L):
        assert np.array_equal(outs["fp32"][l], outs["bf16"][l]), f"layer {l}: BF16 != FP32 path"
    assert np.array_equal(outs["bf16"][1], outs["bf16"][0])      # S layer reads layer 0's rows
    # the F layers against the oracle on the widened inputs
    req, pos = O.token_positions(wl.query_start_loc, wl.seq_lens)
    for l in (0, 2):
        k_wide, q_wide, w = wides[l]
        qc, qs = O.quantize_blocks(q_wide)
        got = io16[l]["q_fp8"].cpu().numpy()
        assert np.array_equal(got, qc)
        rng = np.random.default_rng(l)
        for t in sorted(set(rng.integers(0, wl.T, 12).tolist()) | {0, wl.T - 1}):
            r = int(req[t])
            P = int(wl.prefix_lens[r])
            keys = np.concatenate([wl.k_prefix(l, r), k_wide[wl.query_start_loc[r]:
                                                              wl.query_start_loc[r + 1]]])
            kc, ks = O.quantize_blocks(keys)
            ctx = int(pos[t]) + 1
            assert ctx <= P + (wl.query_start_loc[r + 1] - wl.query_start_loc[r])
            scores = O.index_scores(qc[t], qs[t], w[t], kc[:ctx], ks[:ctx])
            row = per_layer_row(outs, l, t, io16, wl)
            check_topk_row(row, scores, wl.index_topk, f"layer {l} row {t}")


def per_layer_row(outs, l, t, io16, wl):
    """Row t of layer l as the bf16 stack left it (sorted indices, -1 first):
    back to 'valid indices then -1' order for the parity check."""
    row = outs["bf16"][l][t]
    valid = row[row >= 0]
    return np.concatenate([valid, np.full(wl.index_topk - valid.size, -1, row.dtype)])
