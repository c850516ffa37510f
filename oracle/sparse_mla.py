"""Plain, slow CPU definition of sparse MLA attention over the top-k rows, FP64.

TEST INFRASTRUCTURE, under the same rules as ``dsa_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it, and
it shares no code with the CUDA path.

Sources (page title, then section):

* [KV] "GLM-5.3 推理全链路(十二): 主 KV 与索引器缓存的分页预算、前缀命中与驱逐" --
  the byte-accounting table and the list above it: the main KV of one token in
  one layer is an ``fp8_ds_mla`` record of 656 B, packing a 512-d KV latent and
  a 64-d RoPE part (576 one-byte FP8 values) with 16 B of FP32 scales for each
  of five 128-element blocks; 656 x 64 = 41,984 B per page and layer; all 78
  layers write it.  The page-table passage: the indexer cache has no table of
  its own because its slot numbers equal the main KV's.
* [RFC] "RFC: DeepseekV32 模型适配支持" §2.1.3 -- the indexer's top-k enters MLA
  as an additive mask on the q.k scores (0 on the selected tokens, -inf on the
  rest), which is the same as attending over the selected keys only.

Readings where the pages leave a step open:

* Record layout: bytes [0, 576) hold the E4M3 codes of the 576-vector
  [latent (512) | RoPE (64)]; bytes [576, 656) hold 20 FP32 scales, scale j
  for elements [32 j, 32 j + 32) -- four per 128-element block, the fifth
  block holding only the 64 RoPE elements, so scales 18 and 19 are padding
  and stored as 0.  Each 32-element group is quantised with the indexer's
  rule: s = amax / 448 in FP32 (1 for an all-zero group), codes e4m3(x / s).
* A page is 64 records back to back; the record of logical position p is in
  page block_table[r, p // 64] at byte (p % 64) * 656 (the indexer's block
  table and slot numbers).
* MLA in its absorbed decode form (the DeepSeek-V2 and V3 reports, which the
  [KV] series builds on): per query row and head, q is a 576-vector in the
  record's space; a selected token's key is its whole dequantised 576-vector
  and its value the first 512 elements (the latent); score = softmax_scale *
  q . key; out = sum over selected tokens of softmax(score) * value; lse = ln
  sum exp(score).  softmax_scale is an argument.
* Selected tokens are the top-k row's entries >= 0 (logical positions); -1
  selects nothing.  A row that selects nothing has out = 0 and lse = -inf.
"""

from __future__ import annotations

import numpy as np

from .dsa_oracle import E4M3_MAX, PAGE_TOKENS, e4m3_decode, e4m3_encode

MLA_LATENT = 512                    # [KV]: KV latent width
MLA_ROPE = 64                       # [KV]: RoPE part
MLA_DIM = MLA_LATENT + MLA_ROPE     # 576 FP8 bytes per record
MLA_GROUP = 32                      # elements per FP32 scale (four per 128-element block)
MLA_SCALE_SLOTS = 5 * 4             # five 128-element blocks x 4 scales
MLA_TOKEN_BYTES = MLA_DIM + MLA_SCALE_SLOTS * 4     # 656
MLA_PAGE_BYTES = PAGE_TOKENS * MLA_TOKEN_BYTES      # 41,984

__all__ = [
    "MLA_LATENT", "MLA_ROPE", "MLA_DIM", "MLA_GROUP", "MLA_SCALE_SLOTS", "MLA_TOKEN_BYTES",
    "MLA_PAGE_BYTES", "mla_bytes_per_token", "mla_quantize", "mla_dequant",
    "mla_write_kv_cache", "mla_read_tokens", "sparse_mla_row", "sparse_mla_attention",
]


def mla_bytes_per_token(num_layers: int = 1) -> int:
    """[KV] byte-accounting table: 656 B per token per layer."""
    return MLA_TOKEN_BYTES * num_layers


def mla_quantize(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """FP32 [..., 576] -> (E4M3 codes [..., 576], FP32 scales [..., 20]).

    Group j = elements [32 j, 32 j + 32) takes s_j = amax_j / 448 (FP32; 1 for
    an all-zero group) and codes e4m3(x / s_j) with the division in FP32.
    Scale slots 18 and 19 are 0.
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == MLA_DIM
    g = x.reshape(*x.shape[:-1], MLA_DIM // MLA_GROUP, MLA_GROUP)
    amax = np.max(np.abs(g), axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    codes = e4m3_encode((g / s[..., None]).astype(np.float32)).reshape(x.shape)
    scales = np.zeros((*x.shape[:-1], MLA_SCALE_SLOTS), np.float32)
    scales[..., :MLA_DIM // MLA_GROUP] = s
    return codes, scales


def mla_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """FP64 [..., 576]: each code times the scale of its 32-element group."""
    c = e4m3_decode(np.asarray(codes)).reshape(*np.shape(codes)[:-1], MLA_DIM // MLA_GROUP,
                                                MLA_GROUP)
    s = np.asarray(scales, np.float64)[..., :MLA_DIM // MLA_GROUP]
    return (c * s[..., None]).reshape(*np.shape(codes))


def mla_write_kv_cache(cache: np.ndarray, kv: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Store each row of kv [T, 576] as a 656 B record at its slot (page * 64 +
    offset); rows with slot -1 are not written.  ``cache`` is uint8
    [num_pages, 41984]; returns it (modified in place)."""
    slots = np.asarray(slots, np.int64)
    keep = slots >= 0
    codes, scales = mla_quantize(np.asarray(kv)[keep])
    page = (slots[keep] // PAGE_TOKENS)[:, None]
    base = (slots[keep] % PAGE_TOKENS)[:, None] * MLA_TOKEN_BYTES
    cache[page, base + np.arange(MLA_DIM)] = codes
    sb = scales.astype("<f4").view(np.uint8).reshape(-1, MLA_SCALE_SLOTS * 4)
    cache[page, base + MLA_DIM + np.arange(MLA_SCALE_SLOTS * 4)] = sb
    return cache


def mla_read_tokens(cache: np.ndarray, block_table_row: np.ndarray, positions: np.ndarray):
    """(codes [n, 576], scales [n, 20]) of the records of logical positions."""
    pos = np.asarray(positions, np.int64)
    page = np.asarray(block_table_row, np.int64)[pos // PAGE_TOKENS][:, None]
    base = (pos % PAGE_TOKENS)[:, None] * MLA_TOKEN_BYTES
    codes = cache[page, base + np.arange(MLA_DIM)]
    sb = np.ascontiguousarray(cache[page, base + MLA_DIM + np.arange(MLA_SCALE_SLOTS * 4)])
    return codes, sb.view("<f4").reshape(-1, MLA_SCALE_SLOTS).astype(np.float32)


def sparse_mla_row(q: np.ndarray, keys: np.ndarray, softmax_scale: float):
    """One query row over its selected tokens, FP64.

    q [H, 576], keys [n, 576] (dequantised records, values = keys[:, :512]).
    Returns out [H, 512] and lse [H] (natural log).
    """
    q = np.asarray(q, np.float64)
    H = q.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((H, MLA_LATENT)), np.full(H, -np.inf)
    z = float(softmax_scale) * (q @ np.asarray(keys, np.float64).T)       # [H, n]
    zmax = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - zmax)
    denom = np.sum(e, axis=1, keepdims=True)
    out = (e / denom) @ keys[:, :MLA_LATENT]
    lse = (zmax + np.log(denom))[:, 0]
    return out, lse


def sparse_mla_attention(q, cache, query_start_loc, seq_lens, block_table, topk, softmax_scale,
                         rows=None):
    """[RFC] §2.1.3 attention of every query row over the tokens its top-k row
    selects.  q [T, H, 576] (float values), topk [>=T, k] int32.  Returns
    {row: (out [H, 512], lse [H])} for ``rows`` (default all)."""
    qsl = np.asarray(query_start_loc, np.int64)
    T = int(qsl[-1])
    req = np.searchsorted(qsl, np.arange(T), side="right") - 1
    rows = range(T) if rows is None else rows
    res = {}
    for t in rows:
        r = int(req[t])
        sel = np.asarray(topk[t], np.int64)
        sel = sel[sel >= 0]
        codes, scales = mla_read_tokens(cache, block_table[r], sel)
        res[t] = sparse_mla_row(q[t], mla_dequant(codes, scales), softmax_scale)
    return res
