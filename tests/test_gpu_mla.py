"""Sparse MLA attention over the top-k rows, and its record write (GPU).

Record write: cache bytes and slots bit-exact against the oracle.
Attention: the GPU dequantises keys to BF16, multiplies on the tensor cores
with FP32 accumulation, rounds the probabilities to BF16 and writes BF16
outputs, so each of those three roundings (relative 2^-9) enters the result;
the bar, per query row and head, is
    max |out - out_oracle| <= 2e-2 * max |out_oracle| + 2e-3 * max |value|
over the 512 output dimensions (value = the latent of a selected token), and
|lse - lse_oracle| <= 1e-2 (natural-log units).  Rows that select nothing
must give out = 0 and lse = -inf exactly.

At a softmax scale far above the model's (1.0 instead of 1/sqrt(192)) the
top logits of a row lie within the key rounding of one another, and the
rounding decides their weights, like an argmax decided in the kernel's
precision.  That case is compared with the oracle evaluated on keys rounded
as the kernel rounds them (code x scale in FP32, then BF16 round-to-nearest-
even), under the same bar.
"""

import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from conftest import gpu_available

pytestmark = pytest.mark.gpu

OUT_RTOL, OUT_VTOL, LSE_ATOL = 2e-2, 2e-3, 1e-2


@pytest.fixture(scope="module")
def B(lib):
    if not gpu_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_attention_fp8_gb300 import binding, staging
    return binding, staging


def _custom(q_lens, seq_lens, k, seed=5, wid=9):
    q_lens = np.asarray(q_lens, np.int32)
    seq_lens = np.asarray(seq_lens, np.int32)
    pages = (seq_lens.astype(np.int64) + 63) // 64
    pool = int(pages.sum()) + 2
    perm = np.random.default_rng(seed).permutation(pool).astype(np.int32)
    bt = np.full((len(q_lens), int(pages.max())), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        bt[r, :n] = perm[at:at + n]
        at += int(n)
    return synth.Workload(wid, "custom_mla", seed, H=64, index_topk=k, num_layers=1, pattern=None,
                          freq=1, offset=2, q_lens=q_lens, seq_lens=seq_lens, block_table=bt,
                          num_pages=pool, max_num_batched_tokens=int(q_lens.sum()))


def _oracle_cache(wl, layer):
    cache = np.zeros((wl.num_pages, O.MLA_PAGE_BYTES), np.uint8)
    for r in range(wl.R):
        P = int(wl.prefix_lens[r])
        if P:
            O.mla_write_kv_cache(cache, wl.mla_kv_prefix(layer, r),
                                 O.slot_mapping(np.array([0, P]), np.array([P]),
                                                wl.block_table[r:r + 1]))
    O.mla_write_kv_cache(cache, wl.mla_kv_new(layer),
                         O.slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table))
    return cache


def _run(B, wl, heads, scale, topk=None, layer=0):
    binding, staging = B
    meta = staging.stage_metadata(wl)
    io = staging.stage_mla(wl, layer, meta, heads)
    if topk is not None:
        io["topk"] = torch.from_numpy(np.ascontiguousarray(topk, np.int32)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.sparse_mla_attention(io["q"], io["kv_cache"], meta.query_start_loc,
                                            meta.seq_lens, meta.block_table, io["topk"], scale,
                                            status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return io, out.float().cpu().numpy(), lse.cpu().numpy()


def _bf16_keys(codes, scales):
    """Keys as the kernel forms them: FP32 product of code and group scale,
    rounded to BF16 (nearest-even), back in FP64."""
    c = O.e4m3_decode(codes).astype(np.float32).reshape(*codes.shape[:-1], 18, 32)
    k32 = (c * np.asarray(scales, np.float32)[..., :18, None]).reshape(codes.shape)
    return torch.from_numpy(k32).to(torch.bfloat16).double().numpy()


def _check(wl, io, out, lse, scale, rows=None, layer=0, kernel_key_rounding=False):
    cache = io["kv_cache"].cpu().numpy()
    assert np.array_equal(cache, _oracle_cache(wl, layer)), "record bytes differ from the oracle's"
    q = io["q"].float().cpu().numpy().astype(np.float64)
    topk = io["topk"].cpu().numpy()
    ref = O.sparse_mla_attention(q, cache, wl.query_start_loc, wl.seq_lens, wl.block_table, topk,
                                 scale, rows=rows)
    if kernel_key_rounding:
        for t in ref:
            r = int(np.searchsorted(wl.query_start_loc, t, side="right") - 1)
            sel = topk[t][topk[t] >= 0]
            ref[t] = O.sparse_mla_row(q[t], _bf16_keys(*O.mla_read_tokens(cache, wl.block_table[r], sel)),
                                      scale)
    worst = 0.0
    for t, (ro, rl) in ref.items():
        sel = topk[t][topk[t] >= 0]
        if sel.size == 0:
            assert np.all(out[t] == 0) and np.all(np.isneginf(lse[t])), f"row {t}: empty row"
            continue
        r = int(np.searchsorted(wl.query_start_loc, t, side="right") - 1)
        vmax = np.max(np.abs(O.mla_dequant(*O.mla_read_tokens(cache, wl.block_table[r], sel))[:, :512]))
        err = np.max(np.abs(out[t] - ro), axis=1)
        bound = OUT_RTOL * np.max(np.abs(ro), axis=1) + OUT_VTOL * vmax
        assert np.all(err <= bound), (f"row {t}: head {int(np.argmax(err - bound))} off by "
                                      f"{err.max():.3g} (bound {bound.min():.3g})")
        assert np.all(np.abs(lse[t] - rl) <= LSE_ATOL), f"row {t}: lse off by {np.abs(lse[t] - rl).max():.3g}"
        worst = max(worst, float(np.max(err / bound)))
    return worst


def test_record_write_bit_exact(B):
    binding, staging = B
    for wid, scale in ((0, 1.0), (3, 1 / 32)):
        wl = synth.make_workload(wid, scale=scale)
        meta = staging.stage_metadata(wl)
        cache = torch.full((wl.num_pages, binding.MLA_PAGE_BYTES), 0x6B, dtype=torch.uint8,
                           device="cuda")
        slots = torch.full((wl.T,), -9, dtype=torch.int64, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.mla_write_kv(torch.from_numpy(wl.mla_kv_new(0)).cuda(), meta.query_start_loc,
                             meta.seq_lens, meta.block_table, cache, slot_mapping=slots, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        want_slots = O.slot_mapping(wl.query_start_loc, wl.seq_lens, wl.block_table)
        assert np.array_equal(slots.cpu().numpy(), want_slots)
        ref = np.full((wl.num_pages, O.MLA_PAGE_BYTES), 0x6B, np.uint8)
        O.mla_write_kv_cache(ref, wl.mla_kv_new(0), want_slots)
        assert np.array_equal(cache.cpu().numpy(), ref)


@pytest.mark.parametrize("heads", [128, 64, 16, 1])
def test_prefill_and_decode_rows(B, heads):
    """Prefill rows from position 0 (rows selecting 1..k tokens), decode rows,
    a ragged last tile: k = 100 leaves 4 tokens in the last 32-token tile."""
    wl = _custom([40, 1, 1, 3], [40, 700, 129, 3000], k=100)
    scale = 1 / math.sqrt(192)
    io, out, lse = _run(B, wl, heads, scale)
    _check(wl, io, out, lse, scale)


@pytest.mark.parametrize("scale", [1.0, 0.02])
def test_peaky_and_flat_softmax(B, scale):
    """scale 1.0: score spreads of hundreds in log units, so the running
    maximum grows many times and the output is rescaled; 0.02: near-uniform."""
    wl = _custom([1, 1, 2], [5000, 2100, 900], k=2048)
    io, out, lse = _run(B, wl, 128, scale)
    _check(wl, io, out, lse, scale, kernel_key_rounding=scale >= 1.0)


def test_scattered_minus_one_and_empty_rows(B):
    """-1 entries anywhere in a row, a row that selects nothing, repeated rows."""
    wl = _custom([1, 1, 1, 1], [300, 64, 1000, 65], k=96)
    rng = np.random.default_rng(3)
    topk = np.full((4, 96), -1, np.int32)
    topk[0, rng.choice(96, 50, replace=False)] = rng.choice(300, 50, replace=False)
    topk[2] = rng.choice(1000, 96, replace=False)
    topk[3, ::3] = rng.choice(65, 32, replace=False)
    io, out, lse = _run(B, wl, 128, 0.05, topk=topk)
    _check(wl, io, out, lse, 0.05)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_batched_decode_full_size(B):
    """The batched decode batch (64 requests, contexts 1024..8192), 128 heads,
    2048 selected tokens per row, every row."""
    wl = synth.make_workload(1)
    io, out, lse = _run(B, wl, 128, 1 / math.sqrt(192))
    _check(wl, io, out, lse, 1 / math.sqrt(192))


def test_bad_entries_are_reported(B):
    binding, staging = B
    wl = _custom([1], [200], k=8)
    topk = np.array([[3, 250, 7, -1, 199, 0, 1000, 5]], np.int32)   # 250, 1000 >= seq_len
    io, out, lse = None, None, None
    meta = staging.stage_metadata(wl)
    io = staging.stage_mla(wl, 0, meta, 4)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.sparse_mla_attention(io["q"], io["kv_cache"], meta.query_start_loc,
                                            meta.seq_lens, meta.block_table,
                                            torch.from_numpy(topk).cuda(), 0.1, status=st)
    torch.cuda.synchronize()
    assert st.item() & binding.STATUS_BAD_METADATA
    io["topk"] = torch.from_numpy(np.array([[3, 7, 199, 0, 5, -1, -1, -1]], np.int32)).cuda()
    _check(wl, io, out.float().cpu().numpy(), lse.cpu().numpy(), 0.1)
