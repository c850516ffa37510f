"""Plain, slow CPU definition of the DSA lightning-indexer step, in FP64.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  It shares no code with the CUDA path and must never be called from it.

Sources (page title, then section):

* [IC] "vLLM IndexCache 实战指南: DeepSeek-V3.2 (DSA) 模型的跨层 Top-k 索引复用与
  配置详解" -- §二 How It Works (F/S layers, shared ``topk_indices_buffer``,
  -1 clear before scatter), §三 配置参数参考 (``index_topk_freq``,
  ``index_topk_pattern``, ``index_skip_topk_offset`` and the skip formula),
  §四 方式二 (pattern example; layers beyond the pattern count as F),
  §六 (pattern overrides freq).
* [KV] "GLM-5.3 推理全链路(十二): 主 KV 与索引器缓存的分页预算、前缀命中与驱逐" --
  the byte-accounting table (132 B per token per layer: 128 FP8 bytes plus one
  FP32 scale), the SGLang ``_buffer_shape`` passage (page row of
  ``64 * (128 + 128 // 128 * 4)`` = 8448 bytes), the ``IndexKeyCache.move``
  comment (each page stores all key bytes, then all scale bytes), the
  ``topk_indices_buffer`` passage (``[max_num_batched_tokens, index_topk]``
  int32) and the write-path section (``store_quantized`` writes the FP8 key and
  its scale at the token's in-page offset).
* [HBM] "HBM 索引架构设计" -- §2.3 物理公式 (slot = block_table[req, pos // bs]
  * bs + pos % bs); §5.1 (a compressed cache stores one entry per
  ``compress_ratio`` tokens: storage block = block size // ratio) and §5.2
  (compressed slot mapping: only a token with (pos + 1) % ratio == 0 gets a
  slot, at entry pos // ratio; every other token gets -1 and is not written).
* [DSA] the DeepSeek-V3.2 report (arXiv:2512.02556), which the [KV] page lists
  among its references for the DSA structure: the lightning-indexer score
  ``I(t, s) = sum_h w[t,h] * ReLU(q[t,h] . k[s])``.  The pages themselves print
  no score formula; this is the reading taken where they are silent.

Readings where the pages leave a step open:

* FP8 format: OCP E4M3 ("e4m3fn": bias 7, 3 mantissa bits, no infinities,
  S.1111.111 is NaN, largest finite 448).  Encoding rounds to nearest, ties to
  even, and saturates to +-448 (finite inputs never become NaN).
* Block scale: one FP32 scale per 128-element block, s = amax / 448 computed in
  FP32; a block of zeros takes s = 1.  Codes are e4m3(x / s) with x / s in FP32.
* q arrives already quantised the same way, one block per (token, head).
* Causality: key s is visible to query token t iff s <= pos(t) (itself
  included); its key is written before scoring.
* Returned indices are logical token positions within the request.
* Compressed indexer (ratio N > 1): the key row of the token that completes a
  state (position (c + 1) * N - 1) is the state's key c -- the compressor that
  produces it runs upstream and is not part of this step.  The indexer page
  still holds 64 entries ([KV] 64-token page section: with ``index_kpool`` = N
  the indexer page stays 64 entries and its numbering is divided by N), so the
  indexer block table maps entry blocks c // 64.  Entry c becomes visible to
  the query at pos once its writer has run (the causality rule above), i.e.
  iff (c + 1) * N - 1 <= pos: a row sees (pos + 1) // N entries, and its
  returned indices are entry numbers c.
* Within a row the order is unspecified; this oracle orders by (score desc,
  position asc) and pads with -1 after min(ctx, k) entries.
"""

from __future__ import annotations

import numpy as np

PAGE_TOKENS = 64          # [KV] 64-token physical pages
HEAD_DIM = 128            # [KV] single-head 128-d indexer key
QUANT_BLOCK = 128         # [KV] one FP32 scale per 128-element block
KEY_BYTES = HEAD_DIM                                  # FP8: one byte per element
SCALE_BYTES = HEAD_DIM // QUANT_BLOCK * 4             # one FP32 per block
TOKEN_BYTES = KEY_BYTES + SCALE_BYTES                 # 132 B per token per layer
PAGE_BYTES = PAGE_TOKENS * TOKEN_BYTES                # 8448 B per page
PAGE_SCALE_OFFSET = PAGE_TOKENS * KEY_BYTES           # scales follow all 64 keys

E4M3_MAX = 448.0

__all__ = [
    "PAGE_TOKENS", "HEAD_DIM", "TOKEN_BYTES", "PAGE_BYTES", "PAGE_SCALE_OFFSET",
    "E4M3_MAX", "e4m3_decode", "e4m3_encode", "quantize_blocks", "token_positions",
    "slot_mapping", "compressed_slot_mapping", "visible_entries", "write_k_cache", "gather_request_keys", "dequant_keys",
    "index_scores", "topk_row", "layer_is_full", "layer_schedule",
    "indexer_layer", "run_layer_stack", "cache_bytes_per_token",
]


# --------------------------------------------------------------------------
# OCP E4M3 codec (FP8 format used for the indexer key and query)
# --------------------------------------------------------------------------

def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each E4M3 code as float64 (NaN for S.1111.111).

    Sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.  Exponent
    field 0 is subnormal: m/8 * 2^-6.  Otherwise (1 + m/8) * 2^(e-7).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0,
                   (m / 8.0) * 2.0 ** -6,
                   (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


# Non-negative finite values, indexed by their code 0x00..0x7E.  Codes of a
# sign-magnitude format with exponent above mantissa are monotone in value.
_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
assert np.all(np.diff(_E4M3_POS) > 0)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Encode FP32 values to E4M3: round to nearest, ties to even, saturate.

    Magnitudes above 448 become 448 (code 0x7E); NaN becomes 0x7F; the sign
    bit of the input (including -0.0) is kept.
    """
    y = np.asarray(y, dtype=np.float32)
    v = np.abs(y).astype(np.float64)
    nan = np.isnan(v)
    v = np.where(nan, 0.0, np.minimum(v, E4M3_MAX))
    hi = np.searchsorted(_E4M3_POS, v, side="left")         # first value >= v
    hi = np.minimum(hi, 0x7E)
    lo = np.where(_E4M3_POS[hi] == v, hi, np.maximum(hi - 1, 0))
    d_lo = v - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(nan, np.uint8(0x7F), code)
    code = code | np.where(np.signbit(y), np.uint8(0x80), np.uint8(0))
    return code.astype(np.uint8)


def quantize_blocks(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantise FP32 rows of 128 to (E4M3 codes, FP32 scale per row).

    s = amax / 448 in FP32 (s = 1 for an all-zero row); codes = e4m3(x / s)
    with the division in FP32.  Works on any leading shape [..., 128].
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == QUANT_BLOCK
    amax = np.max(np.abs(x), axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    y = (x / s[..., None]).astype(np.float32)
    return e4m3_encode(y), s


# --------------------------------------------------------------------------
# Paged indexer-K cache: positions, slots, page bytes
# --------------------------------------------------------------------------

def cache_bytes_per_token(num_full_layers: int = 1) -> int:
    """[KV] byte-accounting table: 132 B per token per F layer."""
    return TOKEN_BYTES * num_full_layers


def token_positions(query_start_loc: np.ndarray, seq_lens: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(request id, position in request) of each new token.

    The step's q_len[r] new tokens are the last ones of the context, so the
    j-th new token of request r sits at seq_len[r] - q_len[r] + j.
    """
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    sl = np.asarray(seq_lens, dtype=np.int64)
    T = int(qsl[-1])
    req = np.empty(T, dtype=np.int64)
    pos = np.empty(T, dtype=np.int64)
    for r in range(sl.shape[0]):
        a, b = int(qsl[r]), int(qsl[r + 1])
        q_len = b - a
        req[a:b] = r
        pos[a:b] = sl[r] - q_len + np.arange(q_len)
    return req, pos


def slot_mapping(query_start_loc, seq_lens, block_table) -> np.ndarray:
    """[HBM] §2.3: slot = block_table[r, pos // 64] * 64 + pos % 64, int64 per token."""
    bt = np.asarray(block_table, dtype=np.int64)
    req, pos = token_positions(query_start_loc, seq_lens)
    page = bt[req, pos // PAGE_TOKENS]
    return page * PAGE_TOKENS + pos % PAGE_TOKENS


def compressed_slot_mapping(query_start_loc, seq_lens, block_table, compress_ratio) -> np.ndarray:
    """[HBM] §5.2: int64 slot per token; -1 unless (pos + 1) % ratio == 0.

    A token that completes a state writes entry c = pos // ratio at
    block_table[r, c // 64] * 64 + c % 64 (64-entry indexer pages).  With
    ratio 1 every token is valid and this is ``slot_mapping``.
    """
    n = int(compress_ratio)
    if n < 1:
        raise ValueError("compress_ratio must be >= 1")
    bt = np.asarray(block_table, dtype=np.int64)
    req, pos = token_positions(query_start_loc, seq_lens)
    slots = np.full(pos.shape[0], -1, dtype=np.int64)
    valid = (pos + 1) % n == 0
    c = pos[valid] // n
    slots[valid] = bt[req[valid], c // PAGE_TOKENS] * PAGE_TOKENS + c % PAGE_TOKENS
    return slots


def visible_entries(pos, compress_ratio: int = 1):
    """Cache entries a query at ``pos`` sees: (pos + 1) // ratio (ratio 1: pos + 1)."""
    return (np.asarray(pos, dtype=np.int64) + 1) // int(compress_ratio)


def write_k_cache(cache: np.ndarray, k: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """[KV] write path: FP8 key bytes and FP32 scale at each token's page offset.

    ``cache`` is uint8 [num_pages, 8448]; page ``p`` holds the 64 keys at
    bytes [off*128, off*128+128) and their scales at 8192 + off*4 ([KV],
    ``IndexKeyCache.move`` comment).  Rows whose slot is -1 are not written
    ([HBM] §5.2).  Returns ``cache`` (modified in place).
    """
    slots = np.asarray(slots, dtype=np.int64)
    keep = slots >= 0
    codes, scales = quantize_blocks(np.asarray(k)[keep])
    slots = slots[keep]
    page = (slots // PAGE_TOKENS)[:, None]
    off = (slots % PAGE_TOKENS)[:, None]
    sbytes = scales.astype("<f4").view(np.uint8).reshape(-1, 4)
    cache[page, off * KEY_BYTES + np.arange(KEY_BYTES)] = codes
    cache[page, PAGE_SCALE_OFFSET + off * 4 + np.arange(4)] = sbytes
    return cache


def gather_request_keys(cache: np.ndarray, block_table_row: np.ndarray, ctx: int):
    """Codes [ctx, 128] and scales [ctx] of one request, by logical position."""
    pos = np.arange(ctx, dtype=np.int64)
    page = np.asarray(block_table_row, dtype=np.int64)[pos // PAGE_TOKENS][:, None]
    off = (pos % PAGE_TOKENS)[:, None]
    codes = cache[page, off * KEY_BYTES + np.arange(KEY_BYTES)]
    sb = np.ascontiguousarray(cache[page, PAGE_SCALE_OFFSET + off * 4 + np.arange(4)])
    return codes, sb.reshape(-1).view("<f4").astype(np.float32)


def dequant_keys(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """FP64 values code * scale, rows of 128."""
    return e4m3_decode(codes) * np.asarray(scales, np.float64)[..., None]


# --------------------------------------------------------------------------
# Lightning-indexer score and top-k
# --------------------------------------------------------------------------

def index_scores(q_codes, q_scale, w, k_codes, k_scales) -> np.ndarray:
    """[DSA] I(s) = sum_h w[h] * ReLU(q[h] . k[s]) for one query token, FP64.

    q[h] = e4m3(q_codes[h]) * q_scale[h]; k[s] = e4m3(k_codes[s]) * k_scales[s].
    Returns float64 [n_keys].
    """
    qd = dequant_keys(np.asarray(q_codes), np.asarray(q_scale))      # [H, 128]
    kd = dequant_keys(np.asarray(k_codes), np.asarray(k_scales))     # [n, 128]
    dots = kd @ qd.T                                                 # [n, H]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def topk_row(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores (ties: lower position first), -1 padded.

    Returns int32 [k]; the first min(len(scores), k) entries are valid.
    """
    n = scores.shape[0]
    order = np.argsort(-np.asarray(scores, np.float64), kind="stable")
    out = np.full(k, -1, dtype=np.int32)
    m = min(n, k)
    out[:m] = order[:m]
    return out


# --------------------------------------------------------------------------
# IndexCache F/S layer schedule
# --------------------------------------------------------------------------

def layer_is_full(layer_id: int, pattern: str | None, freq: int = 1, offset: int = 2) -> bool:
    """[IC] §三/§四: is this DSA layer an F (full indexer) layer?

    With a pattern, 'S' skips and layers beyond its length are F.  Otherwise
    the layer skips iff max(layer_id - offset + 1, 0) % freq != 0.
    """
    if pattern is not None:
        if layer_id >= len(pattern):
            return True
        c = pattern[layer_id]
        if c not in "FS":
            raise ValueError(f"pattern character {c!r} is neither F nor S")
        return c == "F"
    if freq <= 0:
        raise ValueError("index_topk_freq must be positive")
    return max(layer_id - offset + 1, 0) % freq == 0


def layer_schedule(num_layers: int, pattern: str | None, freq: int = 1, offset: int = 2) -> list[bool]:
    return [layer_is_full(i, pattern, freq, offset) for i in range(num_layers)]


# --------------------------------------------------------------------------
# One F layer and a whole stack
# --------------------------------------------------------------------------

def indexer_layer(cache, k_new, q_codes, q_scale, w, query_start_loc, seq_lens,
                  block_table, index_topk, topk_buffer, rows=None, compress_ratio=1):
    """One F layer: write this step's keys, then top-k rows into ``topk_buffer``.

    ``rows`` limits scoring to a subset of query tokens (the whole step's keys
    are still written).  Rows [0, T) of the buffer are rewritten; rows beyond
    T are untouched.  With ``compress_ratio`` N > 1 only the tokens that
    complete a state are written ([HBM] §5.2) and row t ranks the
    (pos + 1) // N entries it sees.  Returns (slot_mapping, {row: scores}).
    """
    slots = compressed_slot_mapping(query_start_loc, seq_lens, block_table, compress_ratio)
    write_k_cache(cache, k_new, slots)
    req, pos = token_positions(query_start_loc, seq_lens)
    T = req.shape[0]
    rows = range(T) if rows is None else rows
    scores_out = {}
    per_req = {}
    for t in rows:
        r, ctx = int(req[t]), int(visible_entries(pos[t], compress_ratio))
        if r not in per_req:
            per_req[r] = gather_request_keys(cache, block_table[r],
                                             int(seq_lens[r]) // int(compress_ratio))
        kc, ks = per_req[r]
        s = index_scores(q_codes[t], q_scale[t], w[t], kc[:ctx], ks[:ctx])
        topk_buffer[t] = topk_row(s, index_topk)
        scores_out[t] = s
    return slots, scores_out


def run_layer_stack(num_layers, pattern, freq, offset, layer_inputs, caches,
                    query_start_loc, seq_lens, block_table, index_topk,
                    max_num_batched_tokens, compress_ratio=1):
    """[IC] §二: F layers write the shared buffer, S layers read what the last F
    layer wrote in this pass.  Returns the buffer contents each layer consumes
    (a copy per layer) and the schedule.

    ``layer_inputs[l]`` = (k_new, q_codes, q_scale, w) for F layers;
    ``caches[l]`` is that layer's page pool.  The buffer starts filled with -1.
    """
    sched = layer_schedule(num_layers, pattern, freq, offset)
    if not sched[0]:
        raise ValueError("the first layer of a pass must be F: nothing has written the buffer yet")
    buf = np.full((max_num_batched_tokens, index_topk), -1, dtype=np.int32)
    consumed = []
    for layer in range(num_layers):
        if sched[layer]:
            k_new, qc, qs, w = layer_inputs[layer]
            indexer_layer(caches[layer], k_new, qc, qs, w, query_start_loc, seq_lens,
                          block_table, index_topk, buf, compress_ratio=compress_ratio)
        consumed.append(buf.copy())
    return consumed, sched
