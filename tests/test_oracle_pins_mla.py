"""Pins of the sparse-MLA oracle to facts fixed outside it (CPU only).

The record size and page size against the byte accounting the pages print
(tests/golden/mla_byte_accounting.json), the record layout byte by byte, the
32-element scale groups, the mask equivalence the DeepseekV32 RFC states
(dense attention with a 0 / -inf mask over the top-k equals attention over the
selected tokens), closed forms, and pure-Python brute force.
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle as O
from conftest import golden


def test_record_bytes_match_page_table():
    g = golden("mla_byte_accounting.json")
    assert O.MLA_LATENT == g["latent_dim"] and O.MLA_ROPE == g["rope_dim"]
    assert O.MLA_DIM == g["fp8_bytes"]
    assert O.MLA_SCALE_SLOTS * 4 == g["scale_blocks"] * g["scale_bytes_per_block"]
    assert O.MLA_TOKEN_BYTES == g["bytes_per_token_per_layer"] == O.mla_bytes_per_token()
    L = g["layers"]
    assert O.mla_bytes_per_token(L) == g["bytes_per_token_all_layers"]
    assert O.MLA_PAGE_BYTES == g["bytes_per_page_per_layer"]
    assert O.MLA_PAGE_BYTES * L == g["bytes_per_page_all_layers"]
    assert O.MLA_PAGE_BYTES * L + g["indexer_bytes_per_page_all_full_layers"] == g["bytes_per_block"]
    assert O.mla_bytes_per_token(L) + O.cache_bytes_per_token(21) == g["bytes_per_token_main_plus_indexer"]
    assert round(g["context_tokens_1m"] * O.mla_bytes_per_token(L) / 1e9, 1) == g["main_kv_gb_1m_context"]


def test_record_layout_one_token():
    """A record written at offset o changes exactly its 656 bytes: 576 codes,
    then 20 FP32 scales with the two padding slots zero."""
    rng = np.random.default_rng(2)
    for off in (0, 1, 37, 63):
        cache = np.full((3, O.MLA_PAGE_BYTES), 0xC3, np.uint8)
        kv = rng.standard_normal((1, 576)).astype(np.float32)
        O.mla_write_kv_cache(cache, kv, np.array([64 * 1 + off]))
        changed = np.nonzero(cache != 0xC3)
        assert set(changed[0].tolist()) <= {1}
        lo, hi = off * 656, off * 656 + 656
        assert changed[1].min() >= lo and changed[1].max() < hi
        codes, scales = O.mla_quantize(kv)
        assert np.array_equal(cache[1, lo:lo + 576], codes[0])
        sc = cache[1, lo + 576:hi].copy().view("<f4")
        assert np.array_equal(sc, scales[0])
        assert sc[18] == 0 and sc[19] == 0 and np.all(sc[:18] > 0)
        assert np.all(cache[[0, 2]] == 0xC3)
        c, s = O.mla_read_tokens(cache, np.array([5, 1, 2]), np.array([64 + off]))
        assert np.array_equal(c[0], codes[0]) and np.array_equal(s[0], scales[0])


def test_quantize_scale_groups_are_32_elements():
    """Groups with amax 448 * 2^a get scale exactly 2^a, so every code is the
    E4M3 code of x / 2^a; the largest element of each group is +-448; a
    change in one group leaves the other groups' codes and scales alone."""
    rng = np.random.default_rng(3)
    x = rng.uniform(-1, 1, 576).astype(np.float32)
    exps = np.arange(18) - 9
    for j in range(18):
        g = x[32 * j:32 * j + 32]
        g /= np.max(np.abs(g))
        g *= np.float32(448.0 * 2.0 ** exps[j])
        x[32 * j:32 * j + 32] = g
    codes, scales = O.mla_quantize(x)
    assert np.array_equal(scales[:18], (2.0 ** exps).astype(np.float32))
    for j in range(18):
        g = x[32 * j:32 * j + 32]
        assert np.array_equal(codes[32 * j:32 * j + 32], O.e4m3_encode(g / np.float32(2.0 ** exps[j])))
        assert np.max(np.abs(O.e4m3_decode(codes[32 * j:32 * j + 32]))) == 448.0
    y = x.copy()
    y[40] *= 3.0                        # group 1 only
    c2, s2 = O.mla_quantize(y)
    diff = np.nonzero(c2 != codes)[0]
    assert diff.size and diff.min() >= 32 and diff.max() < 64
    assert np.array_equal(np.nonzero(s2 != scales)[0], [1])
    z = np.zeros(576, np.float32)
    cz, sz = O.mla_quantize(z)
    assert np.all(cz == 0) and np.all(sz[:18] == 1.0)
    # dequantised values within half an E4M3 step: |x/s - y| <= max(|x/s| / 16, 2^-10)
    w = (rng.standard_normal(576) * np.repeat(rng.uniform(0.01, 50, 18), 32)).astype(np.float32)
    cw, sw = O.mla_quantize(w)
    d = O.mla_dequant(cw, sw)
    s_el = np.repeat(sw[:18].astype(np.float64), 32)
    err = np.abs(d - w) / s_el
    assert np.all(err <= np.maximum(np.abs(w) / s_el / 16, 2.0 ** -10) * (1 + 1e-6))


def _tiny_cache(rng, ctx, pages_extra=1):
    n_pages = (ctx + 63) // 64
    pool = n_pages + pages_extra
    bt = rng.permutation(pool)[:n_pages].astype(np.int32)
    cache = np.zeros((pool, O.MLA_PAGE_BYTES), np.uint8)
    kv = rng.standard_normal((ctx, 576)).astype(np.float32)
    slots = bt[np.arange(ctx) // 64].astype(np.int64) * 64 + np.arange(ctx) % 64
    O.mla_write_kv_cache(cache, kv, slots)
    return cache, bt, kv


@pytest.mark.parametrize("scale", [1 / math.sqrt(192), 0.5])
def test_mask_equivalence_dense_vs_sparse(scale):
    """[RFC] §2.1.3: scores over the whole context plus a 0 / -inf mask built
    from the top-k row, softmax over the context, equal the sparse result."""
    rng = np.random.default_rng(4)
    ctx, H, k = 300, 3, 40
    cache, bt, _ = _tiny_cache(rng, ctx)
    q = rng.standard_normal((1, H, 576))
    row = np.full(k + 5, -1, np.int32)
    row[:k] = rng.choice(ctx, k, replace=False)
    rng.shuffle(row)
    res = O.sparse_mla_attention(q, cache, np.array([0, 1]), np.array([ctx]), bt[None, :],
                                 row[None, :], scale)
    out, lse = res[0]
    c, s = O.mla_read_tokens(cache, bt, np.arange(ctx))
    allk = O.mla_dequant(c, s)                                   # every position's key
    z = scale * np.einsum("hd,nd->hn", q[0], allk)
    mask = np.full(ctx, -np.inf)
    mask[row[row >= 0]] = 0.0
    p = softmax(z + mask, axis=1)
    np.testing.assert_allclose(out, p @ allk[:, :512], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, logsumexp(z + mask, axis=1), rtol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(5)
    ctx, H = 130, 4
    cache, bt, _ = _tiny_cache(rng, ctx)
    c, s = O.mla_read_tokens(cache, bt, np.arange(ctx))
    K = O.mla_dequant(c, s)
    q = rng.standard_normal((1, H, 576))
    qsl, seq = np.array([0, 1]), np.array([ctx])
    # one selected token: out is its latent, lse its score
    (out, lse), = O.sparse_mla_attention(q, cache, qsl, seq, bt[None], np.array([[-1, 77, -1]]),
                                         0.3).values()
    np.testing.assert_allclose(out, np.tile(K[77, :512], (H, 1)), rtol=1e-13)
    np.testing.assert_allclose(lse, 0.3 * q[0] @ K[77], rtol=1e-12)
    # q = 0: every selected token weighs the same, lse = ln(n)
    sel = np.array([[3, 9, 127, 64, 65]])
    (out, lse), = O.sparse_mla_attention(np.zeros((1, H, 576)), cache, qsl, seq, bt[None], sel,
                                         1.0).values()
    np.testing.assert_allclose(out, np.tile(K[sel[0], :512].mean(axis=0), (H, 1)), rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(lse, np.log(5.0), rtol=1e-13)
    # two tokens with a known score gap: weights 1 / (1 + e^-d)
    a, b = 10, 20
    d = 0.7 * (q[0] @ K[a] - q[0] @ K[b])
    (out, lse), = O.sparse_mla_attention(q, cache, qsl, seq, bt[None], np.array([[a, b]]),
                                         0.7).values()
    wa = 1.0 / (1.0 + np.exp(-d))
    np.testing.assert_allclose(out, wa[:, None] * K[a, :512] + (1 - wa)[:, None] * K[b, :512],
                               rtol=1e-11, atol=1e-13)
    # nothing selected
    (out, lse), = O.sparse_mla_attention(q, cache, qsl, seq, bt[None], np.array([[-1, -1]]),
                                         0.7).values()
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_brute_force_pure_python():
    """Explicit loops over heads, tokens and elements with math.exp, reading
    each record's bytes straight from the page."""
    rng = np.random.default_rng(6)
    ctx, H, scale = 70, 2, 0.2
    cache, bt, _ = _tiny_cache(rng, ctx)
    q = rng.standard_normal((1, H, 576))
    sel = [5, 69, 0, 33]
    (out, lse), = O.sparse_mla_attention(q, cache, np.array([0, 1]), np.array([ctx]), bt[None],
                                         np.array([sel + [-1]]), scale).values()
    table = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    recs = []
    for p in sel:
        page, off = int(bt[p // 64]), (p % 64) * 656
        raw = cache[page, off:off + 656]
        sc = raw[576:656].copy().view("<f4")
        recs.append([float(table[raw[i]]) * float(sc[i // 32]) for i in range(576)])
    for h in range(H):
        z = [scale * sum(float(q[0, h, i]) * r[i] for i in range(576)) for r in recs]
        m = max(z)
        e = [math.exp(v - m) for v in z]
        tot = sum(e)
        assert lse[h] == pytest.approx(m + math.log(tot), rel=1e-12)
        for dim in (0, 1, 255, 511):
            want = sum(e[j] / tot * recs[j][dim] for j in range(len(sel)))
            assert out[h, dim] == pytest.approx(want, rel=1e-10, abs=1e-12)


def test_order_and_placement_invariance():
    """The order of a top-k row and where its -1 entries sit do not matter;
    nor does the physical page placement of the same records."""
    rng = np.random.default_rng(7)
    ctx, H = 200, 3
    kv = rng.standard_normal((ctx, 576)).astype(np.float32)
    q = rng.standard_normal((1, H, 576))
    sel = rng.choice(ctx, 50, replace=False)
    outs = []
    for seed in (1, 2):
        r2 = np.random.default_rng(seed)
        pool = 6
        bt = r2.permutation(pool)[:4].astype(np.int32)
        cache = np.zeros((pool, O.MLA_PAGE_BYTES), np.uint8)
        slots = bt[np.arange(ctx) // 64].astype(np.int64) * 64 + np.arange(ctx) % 64
        O.mla_write_kv_cache(cache, kv, slots)
        row = np.concatenate([r2.permutation(sel), -np.ones(10, np.int64)])
        r2.shuffle(row)
        outs.append(O.sparse_mla_attention(q, cache, np.array([0, 1]), np.array([ctx]),
                                           bt[None], row[None], 0.1)[0])
    np.testing.assert_allclose(outs[0][0], outs[1][0], rtol=1e-12)
    np.testing.assert_allclose(outs[0][1], outs[1][1], rtol=1e-12)
