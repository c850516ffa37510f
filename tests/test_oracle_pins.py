"""Pins of the CPU oracle to facts fixed outside it (CPU only).

Each test checks the oracle against something it does not compute itself:
values the pages print (fixtures under tests/golden/, each citing its page and
section), the OCP E4M3 definition and PyTorch's independent float8_e4m3fn
cast, hand-computed closed forms, invariants, and brute force on tiny inputs.
"""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden


# ----------------------------------------------------------------------------
# byte accounting and page layout
# ----------------------------------------------------------------------------

def test_byte_accounting_matches_page_table():
    g = golden("byte_accounting.json")
    assert O.TOKEN_BYTES == g["bytes_per_token_per_layer"] == g["index_head_dim"] + g["index_head_dim"] // g["quant_block_size"] * 4
    assert O.PAGE_TOKENS == g["page_tokens"]
    assert O.PAGE_BYTES == g["bytes_per_page"]
    L = g["full_indexer_layers"]
    assert O.cache_bytes_per_token(L) == g["bytes_per_token_all_full_layers"]
    assert O.PAGE_BYTES * L == g["bytes_per_page_all_full_layers"]
    n = g["context_tokens_1m"]
    assert n * O.cache_bytes_per_token(L) == g["indexer_bytes_1m_context"]
    assert n // O.PAGE_TOKENS == g["pages_1m_context"]
    assert g["prefill_chunk_tokens"] * O.TOKEN_BYTES == g["prefill_chunk_bytes_per_layer"]
    assert O.cache_bytes_per_token(L) == g["decode_bytes_per_request_step_all_full_layers"]


def test_page_layout_keys_then_scales():
    """One token written at offset o touches exactly its 128 key bytes and its
    4 scale bytes after the page's 64 keys, nothing else."""
    rng = np.random.default_rng(1)
    for off in [0, 1, 31, 63]:
        cache = np.full((3, O.PAGE_BYTES), 0xA5, dtype=np.uint8)
        k = rng.standard_normal((1, 128)).astype(np.float32)
        slot = np.array([2 * 64 + off])
        O.write_k_cache(cache, k, slot)
        codes, scale = O.quantize_blocks(k)
        changed = np.nonzero(cache != 0xA5)
        assert set(changed[0].tolist()) <= {2}
        assert np.array_equal(cache[2, off * 128:(off + 1) * 128], codes[0])
        sb = cache[2, 64 * 128 + off * 4: 64 * 128 + off * 4 + 4]
        assert sb.view("<f4")[0] == scale[0]
        untouched = np.ones(O.PAGE_BYTES, bool)
        untouched[off * 128:(off + 1) * 128] = False
        untouched[8192 + off * 4: 8192 + off * 4 + 4] = False
        assert np.all(cache[2, untouched] == 0xA5)
        assert np.all(cache[[0, 1]] == 0xA5)


def test_full_page_covers_every_byte():
    rng = np.random.default_rng(2)
    cache = np.zeros((1, O.PAGE_BYTES), dtype=np.uint8)
    touched = np.zeros(O.PAGE_BYTES, dtype=np.int64)
    for off in range(64):
        before = np.full((1, O.PAGE_BYTES), 0x5A, np.uint8)
        O.write_k_cache(before, rng.standard_normal((1, 128)).astype(np.float32) + 3.0, np.array([off]))
        touched += (before[0] != 0x5A)
    # every key byte and every scale byte belongs to exactly one token (a few
    # bytes may coincidentally equal the sentinel, so allow rare misses)
    assert touched.max() == 1
    assert touched.sum() >= O.PAGE_BYTES - 64


# ----------------------------------------------------------------------------
# E4M3 codec
# ----------------------------------------------------------------------------

def test_e4m3_decode_reference_values():
    g = golden("e4m3_reference_values.json")
    vals = O.e4m3_decode(np.array(g["codes"], np.uint8))
    for c, v, want in zip(g["codes"], vals, g["values"]):
        assert v == want, (c, v, want)
        assert math.copysign(1.0, v) == math.copysign(1.0, want)
    assert np.all(np.isnan(O.e4m3_decode(np.array(g["nan_codes"], np.uint8))))


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(theirs[~nan]))


def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def test_e4m3_encode_midpoints_round_to_even():
    pos = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact in FP32
    enc = O.e4m3_encode(mids).astype(np.int64)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(enc, want)
    # just off the midpoint goes to the nearer side
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    assert np.array_equal(O.e4m3_encode(up).astype(np.int64), lo + 1)
    assert np.array_equal(O.e4m3_encode(dn).astype(np.int64), lo)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(3)
    y = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 100,
        rng.uniform(-2 ** -5, 2 ** -5, 100000).astype(np.float32),   # subnormal region
        rng.uniform(-448, 448, 100000).astype(np.float32),
        np.array([0.0, -0.0, 2 ** -10, -2 ** -10, 3 * 2 ** -10, 447.9, 448.0], np.float32),
    ])
    y = y[np.abs(y) <= 448]
    ours = O.e4m3_encode(y)
    theirs = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_e4m3_encode_saturates():
    y = np.array([448.001, 449, 463.9, 464, 480, 1e6, 3e38, -449, -1e30], np.float32)
    assert O.e4m3_encode(y).tolist() == [0x7E] * 7 + [0xFE] * 2
    assert O.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_quantize_blocks_properties():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((512, 128)).astype(np.float32)
    x[7] *= 1e-30            # subnormal-scale block
    x[9] = 0.0
    x[10] = -0.0
    x[11, 5] = 3.5           # one non-zero element
    x[11, :5] = 0
    x[11, 6:] = 0
    codes, s = O.quantize_blocks(x)
    amax = np.abs(x).max(axis=1)
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz] / np.float32(448)).astype(np.float32))
    assert s[9] == 1.0 and s[10] == 1.0
    assert np.all(codes[9] == 0) and np.all(codes[10] == 0x80)
    # the element of largest magnitude lands on +-448
    arg = np.abs(x).argmax(axis=1)
    top = codes[np.arange(512), arg][nz]
    assert np.all((top & 0x7F) == 0x7E)
    assert codes[11, 5] == 0x7E
    # dequantised error within half an E4M3 step: relative 2^-4 for normals,
    # absolute 2^-10 * s in the subnormal range
    dq = O.dequant_keys(codes, s)
    err = np.abs(dq - x.astype(np.float64))
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s[:, None].astype(np.float64) * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-6))


# ----------------------------------------------------------------------------
# slot mapping
# ----------------------------------------------------------------------------

def test_slot_mapping_contract_example():
    g = golden("slot_mapping_contract.json")
    row = np.array(g["block_table_row"], np.int32)
    for pos, want in zip(g["positions"], g["slots"]):
        # one request whose context ends at pos: its single new token sits at pos
        got = O.slot_mapping(np.array([0, 1]), np.array([pos + 1]), row[None, :])
        assert got.tolist() == [want]


def test_slot_mapping_brute_force_inverse():
    """Every (request, position) maps to a distinct physical slot, and reading
    the pool page by page recovers (request, position)."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        R = int(rng.integers(1, 5))
        seq = rng.integers(1, 300, size=R)
        ql = np.array([int(rng.integers(0, s + 1)) for s in seq])
        pages = [(s + 63) // 64 for s in seq]
        pool = sum(pages) + int(rng.integers(0, 4))
        perm = rng.permutation(pool)
        bt = np.full((R, max(pages)), -1, np.int32)
        at = 0
        owner = {}
        for r, n in enumerate(pages):
            bt[r, :n] = perm[at:at + n]
            for j in range(n):
                owner[int(perm[at + j])] = (r, j)
            at += n
        qsl = np.concatenate([[0], np.cumsum(ql)])
        slots = O.slot_mapping(qsl, seq, bt)
        req, pos = O.token_positions(qsl, seq)
        assert len(set(slots.tolist())) == len(slots)
        for s, r, p in zip(slots.tolist(), req.tolist(), pos.tolist()):
            rr, j = owner[s // 64]
            assert rr == r and j * 64 + s % 64 == p
            assert seq[r] - ql[r] <= p < seq[r]


# ----------------------------------------------------------------------------
# compressed slot mapping (one cache entry per compress_ratio tokens)
# ----------------------------------------------------------------------------

def test_compressed_slot_mapping_example():
    g = golden("compressed_slot_mapping.json")
    for case in g["cases"]:
        row = np.array(case["block_table_row"], np.int32)[None, :]
        n = int(case["ratio"])
        for pos, want in zip(case["positions"], case["slots"]):
            got = O.compressed_slot_mapping(np.array([0, 1]), np.array([pos + 1]), row, n)
            assert got.tolist() == [want], (n, pos)


def test_compressed_entries_per_256_token_block():
    """A 256-token prefill keeps 64 entries at ratio 4 and 2 at ratio 128, in
    entry order at the front of the request's first indexer page."""
    g = golden("compressed_slot_mapping.json")
    bt = np.array([[9, 4, 6, 1]], np.int32)
    for ratio, want in g["entries_per_256_token_block"].items():
        slots = O.compressed_slot_mapping(np.array([0, 256]), np.array([256]), bt, int(ratio))
        kept = slots[slots >= 0]
        assert kept.size == want
        assert kept.tolist() == [9 * 64 + i for i in range(want)]


def test_compressed_ratio_one_is_the_plain_mapping():
    rng = np.random.default_rng(21)
    seq = np.array([1, 77, 300, 64])
    ql = np.array([1, 5, 300, 0])
    qsl = np.concatenate([[0], np.cumsum(ql)])
    bt = rng.permutation(40).astype(np.int32)[:20].reshape(4, 5)
    assert np.array_equal(O.compressed_slot_mapping(qsl, seq, bt, 1), O.slot_mapping(qsl, seq, bt))
    with pytest.raises(ValueError):
        O.compressed_slot_mapping(qsl, seq, bt, 0)


def test_compressed_write_leaves_unmapped_tokens_out():
    """Rows with slot -1 change no byte; the others land as an uncompressed
    write of just those rows would put them."""
    rng = np.random.default_rng(22)
    k = rng.standard_normal((200, 128)).astype(np.float32)
    bt = np.array([[3, 0]], np.int32)
    slots = O.compressed_slot_mapping(np.array([0, 200]), np.array([200]), bt, 4)
    got = O.write_k_cache(np.full((5, O.PAGE_BYTES), 0x3C, np.uint8), k, slots)
    keep = np.nonzero(slots >= 0)[0]
    assert keep.tolist() == list(range(3, 200, 4))
    want = np.full((5, O.PAGE_BYTES), 0x3C, np.uint8)
    for i in keep:          # one row at a time, at the page offset worked out by hand
        c = i // 4
        O.write_k_cache(want, k[i:i + 1], np.array([3 * 64 + c]))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("ratio", [2, 3, 4, 7])
def test_compressed_rows_brute_force(ratio):
    """Every row against an enumeration of the states its request holds: walk
    the request's tokens in order, let each token that completes a state append
    its key, and rank the states appended by tokens at or before the row."""
    rng = np.random.default_rng(300 + ratio)
    seq = np.array([5 * ratio + 3, ratio - 1, 2 * ratio, 9 * ratio + 1])
    ql = np.array([4 * ratio, ratio - 1, 2, 1])
    R, H, k = len(seq), 4, 5
    tokens = [rng.standard_normal((int(s), 128)).astype(np.float32) for s in seq]
    entries = [int(s) // ratio for s in seq]
    pages = [max(1, (e + 63) // 64) for e in entries]
    pool = sum(pages) + 2
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.full((R, max(pages)), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        bt[r, :n] = perm[at:at + n]
        at += n
    cache = np.zeros((pool, O.PAGE_BYTES), np.uint8)
    for r in range(R):                       # the cached prefix, written by an earlier step
        P = int(seq[r] - ql[r])
        if P:
            sl = O.compressed_slot_mapping(np.array([0, P]), np.array([P]), bt[r:r + 1], ratio)
            O.write_k_cache(cache, tokens[r][:P], sl)
    qsl = np.concatenate([[0], np.cumsum(ql)])
    T = int(qsl[-1])
    k_new = np.concatenate([tokens[r][int(seq[r] - ql[r]):] for r in range(R)])
    qc, qs = O.quantize_blocks(rng.standard_normal((T, H, 128)).astype(np.float32))
    w = rng.standard_normal((T, H)).astype(np.float32)
    buf = np.full((T + 1, k), 7, np.int32)
    O.indexer_layer(cache, k_new, qc, qs, w, qsl, seq, bt, k, buf, compress_ratio=ratio)
    assert np.all(buf[T] == 7)
    for r in range(R):
        for j in range(int(ql[r])):
            t = int(qsl[r]) + j
            pos = int(seq[r] - ql[r]) + j
            states = [tokens[r][p] for p in range(pos + 1) if (p + 1) % ratio == 0]
            if states:
                kc, ks = O.quantize_blocks(np.stack(states))
                s = np.array([sum(float(w[t, h]) * max(float(np.dot(
                    O.e4m3_decode(qc[t, h]) * float(qs[t, h]), O.e4m3_decode(kc[i]) * float(ks[i]))), 0.0)
                    for h in range(H)) for i in range(len(states))])
                want = O.topk_row(s, k)
            else:
                want = np.full(k, -1, np.int32)
            assert np.array_equal(buf[t], want), (ratio, r, j)


# ----------------------------------------------------------------------------
# scores
# ----------------------------------------------------------------------------

def _code(v: float) -> int:
    return int(O.e4m3_encode(np.array([v], np.float32))[0])


def test_scores_closed_form_one_hot():
    """Hand-computed: head 0 sees +1*2 at dim 3, head 1 sees -1*2 (ReLU kills it),
    head 2 sees 1.5*2 + 0.5*(-4) = 1.  With q scales (0.5, 2, 0.25), k scale
    0.125 and w = (3, 7, -2):  3*ReLU(0.5*0.125*2) + 7*ReLU(-...) - 2*ReLU(0.25*0.125*1)
    = 0.375 - 0.0625 = 0.3125."""
    qc = np.zeros((3, 128), np.uint8)
    qc[0, 3] = _code(1.0)
    qc[1, 3] = _code(-1.0)
    qc[2, 3] = _code(1.5)
    qc[2, 9] = _code(0.5)
    kc = np.zeros((2, 128), np.uint8)
    kc[0, 3] = _code(2.0)
    kc[0, 9] = _code(-4.0)
    kc[1, 9] = _code(8.0)        # only head 2 (dim 9) sees key 1: 0.5*8 = 4
    qs = np.array([0.5, 2.0, 0.25], np.float32)
    ks = np.array([0.125, 0.5], np.float32)
    w = np.array([3.0, 7.0, -2.0], np.float32)
    s = O.index_scores(qc, qs, w, kc, ks)
    assert s[0] == 0.3125
    # key 1: head 2 dot = 0.25*0.5*4 = 0.5 -> -2*0.5 = -1
    assert s[1] == -1.0


def test_scores_relu_and_weights():
    rng = np.random.default_rng(6)
    H, n = 5, 40
    qc, qs = O.quantize_blocks(rng.standard_normal((H, 128)).astype(np.float32))
    kc, ks = O.quantize_blocks(rng.standard_normal((n, 128)).astype(np.float32))
    # all-ones weights: score = sum of positive parts of the per-head dots
    s1 = O.index_scores(qc, qs, np.ones(H, np.float32), kc, ks)
    assert np.all(s1 >= 0)
    # negating every query flips which dots are positive: s(q) + s(-q) = sum |dot|
    qneg = qc ^ np.uint8(0x80)
    s2 = O.index_scores(qneg, qs, np.ones(H, np.float32), kc, ks)
    dots = O.dequant_keys(kc, ks) @ O.dequant_keys(qc, qs).T
    assert np.allclose(s1 + s2, np.abs(dots).sum(axis=1), rtol=1e-12, atol=0)
    # permuting heads together with their weights leaves scores unchanged
    w = rng.standard_normal(H).astype(np.float32)
    p = rng.permutation(H)
    a = O.index_scores(qc, qs, w, kc, ks)
    b = O.index_scores(qc[p], qs[p], w[p], kc, ks)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    # doubling a key's scale doubles its score
    ks2 = ks.copy()
    ks2[3] *= 2
    c = O.index_scores(qc, qs, w, kc, ks2)
    assert c[3] == 2 * a[3] and np.array_equal(np.delete(c, 3), np.delete(a, 3))


def test_scores_brute_force_tiny():
    rng = np.random.default_rng(7)
    H, n = 3, 6
    qc, qs = O.quantize_blocks(rng.standard_normal((H, 128)).astype(np.float32))
    kc, ks = O.quantize_blocks(rng.standard_normal((n, 128)).astype(np.float32))
    w = rng.standard_normal(H).astype(np.float32)
    got = O.index_scores(qc, qs, w, kc, ks)
    qv = O.e4m3_decode(qc)
    kv = O.e4m3_decode(kc)
    for s in range(n):
        tot = 0.0
        for h in range(H):
            d = 0.0
            for i in range(128):
                d += float(qv[h, i]) * float(qs[h]) * float(kv[s, i]) * float(ks[s])
            tot += float(w[h]) * max(d, 0.0)
        assert abs(tot - got[s]) <= 1e-9 * max(1.0, abs(tot))


# ----------------------------------------------------------------------------
# top-k
# ----------------------------------------------------------------------------

def test_topk_short_context_returns_every_position():
    rng = np.random.default_rng(8)
    for ctx in [1, 5, 31, 32]:
        out = O.topk_row(rng.standard_normal(ctx), 32)
        assert sorted(out[:ctx].tolist()) == list(range(ctx))
        assert np.all(out[ctx:] == -1)


def test_topk_brute_force_subsets():
    rng = np.random.default_rng(9)
    for _ in range(30):
        n = int(rng.integers(1, 9))
        k = int(rng.integers(1, 6))
        s = rng.standard_normal(n)
        out = O.topk_row(s, k)
        m = min(n, k)
        best = max(itertools.combinations(range(n), m), key=lambda c: sum(s[list(c)]))
        assert sorted(out[:m].tolist()) == sorted(best)
        assert np.all(out[m:] == -1)


def test_topk_ties_prefer_lower_position():
    s = np.array([1.0, 3.0, 2.0, 3.0, 2.0, 2.0])
    assert O.topk_row(s, 4).tolist() == [1, 3, 2, 4]


# ----------------------------------------------------------------------------
# F/S schedule
# ----------------------------------------------------------------------------

def test_schedule_freq4_offset2_61_layers():
    g = golden("freq4_offset2_61.json")
    full = [l for l in range(g["num_layers"]) if O.layer_is_full(l, None, g["freq"], g["offset"])]
    assert full == g["full_layers"]


def test_schedule_pattern_61():
    g = golden("index_topk_pattern_61.json")
    sched = O.layer_schedule(g["num_layers"], g["pattern"])
    assert sum(sched) == g["full_layers"]
    assert len(sched) - sum(sched) == g["shared_layers"]
    assert sched == [c == "F" for c in g["pattern"]]


def test_schedule_defaults_and_rules():
    # freq = 1 (default): every layer is F
    assert all(O.layer_schedule(78, None, 1, 2))
    # layers 0 and 1 are F for any freq under offset 2
    for freq in range(1, 12):
        assert O.layer_is_full(0, None, freq, 2) and O.layer_is_full(1, None, freq, 2)
    # layers past the end of a pattern count as F (MTP layers)
    assert O.layer_is_full(5, "FS", 4, 2) and O.layer_is_full(3, "FSS")
    assert not O.layer_is_full(2, "FSS")
    # a pattern overrides freq
    assert O.layer_schedule(4, "FSFS", 1, 2) == [True, False, True, False]
    with pytest.raises(ValueError):
        O.layer_is_full(1, "FX")
    with pytest.raises(ValueError):
        O.layer_is_full(3, None, 0, 2)


# ----------------------------------------------------------------------------
# whole layer / stack invariants
# ----------------------------------------------------------------------------

def _tiny_case(seed, R=2, H=4, k=8, perm_seed=0):
    rng = np.random.default_rng(seed)
    ql = rng.integers(1, 20, size=R)
    seq = ql + rng.integers(0, 150, size=R)
    pages = (seq + 63) // 64
    pool = int(pages.sum()) + 3
    perm = np.random.default_rng(perm_seed).permutation(pool)
    bt = np.full((R, int(pages.max())), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        bt[r, :n] = perm[at:at + n]
        at += n
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(qsl[-1])
    prefix = [rng.standard_normal((int(seq[r] - ql[r]), 128)).astype(np.float32) for r in range(R)]
    k_new = rng.standard_normal((T, 128)).astype(np.float32)
    qc, qs = O.quantize_blocks(rng.standard_normal((T, H, 128)).astype(np.float32))
    w = rng.standard_normal((T, H)).astype(np.float32)
    return dict(ql=ql, seq=seq, bt=bt, pool=pool, qsl=qsl, T=T, prefix=prefix,
                k_new=k_new, qc=qc, qs=qs, w=w, k=k)


def _run_tiny(c):
    cache = np.zeros((c["pool"], O.PAGE_BYTES), np.uint8)
    R = len(c["seq"])
    for r in range(R):
        n = len(c["prefix"][r])
        if n:
            O.write_k_cache(cache, c["prefix"][r],
                            O.slot_mapping(np.array([0, n]), np.array([n]), c["bt"][r:r + 1]))
    buf = np.full((c["T"] + 2, c["k"]), -1, np.int32)
    O.indexer_layer(cache, c["k_new"], c["qc"], c["qs"], c["w"], c["qsl"], c["seq"], c["bt"],
                    c["k"], buf)
    return buf


def test_page_permutation_invariance():
    for seed in range(4):
        a = _run_tiny(_tiny_case(seed, perm_seed=0))
        b = _run_tiny(_tiny_case(seed, perm_seed=1))
        assert np.array_equal(a, b)


def test_layer_rows_valid_counts_and_padding():
    c = _tiny_case(11, R=3, k=16)
    buf = _run_tiny(c)
    req, pos = O.token_positions(c["qsl"], c["seq"])
    for t in range(c["T"]):
        n = min(int(pos[t]) + 1, c["k"])
        assert np.all(buf[t, :n] >= 0) and np.all(buf[t, :n] <= pos[t])
        assert len(set(buf[t, :n].tolist())) == n
        assert np.all(buf[t, n:] == -1)
    assert np.all(buf[c["T"]:] == -1)          # rows beyond T untouched


def test_stack_shared_layers_read_last_full_layer():
    c = _tiny_case(12, R=2, k=8)
    L = 5
    pattern = "FSFSS"
    caches, inputs = {}, {}
    for l in range(L):
        lr = np.random.default_rng(500 + l)      # different keys/queries per layer, same shapes
        cache = np.zeros((c["pool"], O.PAGE_BYTES), np.uint8)
        for r in range(2):
            pre = lr.standard_normal((int(c["seq"][r] - c["ql"][r]), 128)).astype(np.float32)
            if len(pre):
                O.write_k_cache(cache, pre, O.slot_mapping(np.array([0, len(pre)]), np.array([len(pre)]),
                                                           c["bt"][r:r + 1]))
        caches[l] = cache
        kn = lr.standard_normal((c["T"], 128)).astype(np.float32)
        qc, qs = O.quantize_blocks(lr.standard_normal((c["T"], 4, 128)).astype(np.float32))
        inputs[l] = (kn, qc, qs, lr.standard_normal((c["T"], 4)).astype(np.float32))
    consumed, sched = O.run_layer_stack(L, pattern, 1, 2, inputs, caches, c["qsl"], c["seq"],
                                        c["bt"], 8, c["T"] + 3)
    assert sched == [True, False, True, False, False]
    assert np.array_equal(consumed[1], consumed[0])
    assert np.array_equal(consumed[3], consumed[2]) and np.array_equal(consumed[4], consumed[2])
    assert not np.array_equal(consumed[2], consumed[0])
    with pytest.raises(ValueError):
        O.run_layer_stack(2, "SF", 1, 2, inputs, caches, c["qsl"], c["seq"], c["bt"], 8, c["T"])
