"""Workload recipes for the DSA lightning-indexer step.

Every random tensor comes from ``numpy.random.default_rng([seed, workload,
layer, tensor_id, ...])`` so any slice can be regenerated on its own (the
oracle regenerates single requests of the long-context workload this way).
Large tensors are drawn in fixed-size chunks, each from its own stream, so
the values do not depend on how many threads generate them.

Shapes follow the serving setups the pages describe:

* 128-d single-head indexer keys, 64-token physical pages ("GLM-5.3 推理全链路
  (十二)", byte-accounting table and the 64-token page section);
* a model-level top-k buffer of ``[max_num_batched_tokens, index_topk]``
  ("GLM-5.3 推理全链路(十二)", top-k / logits workspace section);
* IndexCache F/S stacks given either by ``index_topk_freq`` with offset 2 or
  by an explicit pattern ("vLLM IndexCache 实战指南", parameter table and CLI
  section);
* a compressed indexer cache holding one entry per ``compress_ratio`` tokens
  ("HBM 索引架构设计", §5.1 ratio 4 and §5.3 indexer cache), for contexts of
  16K-128K tokens (the range §5.6 names).

Distributions: q and k ~ N(0, 1) FP32; w ~ N(0, 1) / sqrt(H) FP32; pages of
each request are placed by a random permutation of a pool sized to fit.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128
PAGE_TOKENS = 64

# tensor ids of the random streams
_T_KNEW, _T_Q, _T_W, _T_KPREFIX = 0, 1, 2, 3
_T_CTX, _T_PERM, _T_OUTLIER, _T_PATTERN = 10, 11, 12, 13
_T_MLA_KVNEW, _T_MLA_KVPREFIX, _T_MLA_Q, _T_MLA_SEL = 20, 21, 22, 23

MLA_DIM = 576   # fp8_ds_mla record: 512-d latent + 64-d RoPE

_CHUNK_TOKENS = 16384  # tokens per independent stream chunk (x 128 values)

WORKLOAD_NAMES = {
    0: "tiny_prefill",
    1: "batched_decode",
    2: "prefix_hit_chunked_prefill",
    3: "mixed_batch",
    4: "long_context_decode",
    5: "mtp_decode",
    6: "compressed_decode",
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def _normal_rows(key: tuple, n_rows: int, width: int, threads: int | None = None) -> np.ndarray:
    """FP32 N(0,1) array [n_rows, width], drawn chunk by chunk from streams key+(chunk,)."""
    out = np.empty((n_rows, width), dtype=np.float32)
    n_chunks = (n_rows + _CHUNK_TOKENS - 1) // _CHUNK_TOKENS

    def fill(c: int) -> None:
        lo = c * _CHUNK_TOKENS
        hi = min(n_rows, lo + _CHUNK_TOKENS)
        _rng(*key, c).standard_normal((hi - lo, width), dtype=np.float32, out=out[lo:hi])

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
        return out
    threads = threads or min(n_chunks, max(1, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(n_chunks)))
    return out


@dataclass
class Workload:
    """One batch of the indexer step plus the layer stack it runs through."""

    workload_id: int
    name: str
    seed: int
    H: int                      # indexer heads
    index_topk: int
    num_layers: int
    pattern: str | None         # explicit F/S string, or None to use freq/offset
    freq: int
    offset: int
    q_lens: np.ndarray          # int32 [R] new tokens per request in this step
    seq_lens: np.ndarray        # int32 [R] context length after this step
    block_table: np.ndarray     # int32 [R, max_blocks] physical page ids
    num_pages: int              # pages in the pool (per F layer)
    max_num_batched_tokens: int
    outlier_channels: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))
    outlier_scale: float = 1.0
    compress_ratio: int = 1     # tokens per indexer cache entry

    # ---- derived metadata -------------------------------------------------
    @property
    def R(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.q_lens.sum())

    @property
    def query_start_loc(self) -> np.ndarray:
        out = np.zeros(self.R + 1, dtype=np.int32)
        np.cumsum(self.q_lens, out=out[1:])
        return out

    @property
    def prefix_lens(self) -> np.ndarray:
        """Tokens already in the cache before this step (context minus new tokens)."""
        return (self.seq_lens - self.q_lens).astype(np.int32)

    @property
    def prefix_entries(self) -> np.ndarray:
        """Cache entries written before this step: one per compress_ratio tokens."""
        return (self.prefix_lens // self.compress_ratio).astype(np.int32)

    @property
    def entries(self) -> np.ndarray:
        """Cache entries of each request after this step."""
        return (self.seq_lens // self.compress_ratio).astype(np.int32)

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    # ---- tensors ----------------------------------------------------------
    def _apply_outliers(self, k: np.ndarray) -> np.ndarray:
        if self.outlier_channels.size:
            k[:, self.outlier_channels] *= np.float32(self.outlier_scale)
        return k

    def k_new(self, layer: int) -> np.ndarray:
        """FP32 [T, 128]: the indexer key of every token of this step."""
        k = _normal_rows((self.seed, self.workload_id, layer, _T_KNEW), self.T, HEAD_DIM)
        return self._apply_outliers(k)

    def k_prefix(self, layer: int, request: int) -> np.ndarray:
        """FP32 [prefix_entries, 128]: keys of the cache entries written before
        this step (one per token, or one per compress_ratio tokens)."""
        n = int(self.prefix_entries[request])
        k = _normal_rows((self.seed, self.workload_id, layer, _T_KPREFIX, request), n, HEAD_DIM)
        return self._apply_outliers(k)

    def q(self, layer: int) -> np.ndarray:
        """FP32 [T, H, 128] indexer queries."""
        q = _normal_rows((self.seed, self.workload_id, layer, _T_Q), self.T, self.H * HEAD_DIM)
        return q.reshape(self.T, self.H, HEAD_DIM)

    def w(self, layer: int) -> np.ndarray:
        """FP32 [T, H] per-head weights, N(0,1)/sqrt(H)."""
        w = _rng(self.seed, self.workload_id, layer, _T_W).standard_normal(
            (self.T, self.H), dtype=np.float32)
        return (w / np.float32(math.sqrt(self.H))).astype(np.float32)

    # ---- sparse-MLA inputs (the consumer of the top-k rows) ---------------
    def mla_kv_new(self, layer: int) -> np.ndarray:
        """FP32 [T, 576]: [latent | RoPE] of every token of this step, N(0, 1)."""
        return _normal_rows((self.seed, self.workload_id, layer, _T_MLA_KVNEW), self.T, MLA_DIM)

    def mla_kv_prefix(self, layer: int, request: int) -> np.ndarray:
        """FP32 [prefix_len, 576]: [latent | RoPE] of the cached tokens, N(0, 1)."""
        n = int(self.prefix_lens[request])
        return _normal_rows((self.seed, self.workload_id, layer, _T_MLA_KVPREFIX, request), n,
                            MLA_DIM)

    def mla_q(self, layer: int, heads: int) -> np.ndarray:
        """FP32 [T, heads, 576] absorbed MLA queries, N(0, 1)."""
        q = _normal_rows((self.seed, self.workload_id, layer, _T_MLA_Q, heads), self.T,
                         heads * MLA_DIM)
        return q.reshape(self.T, heads, MLA_DIM)

    def selection_rows(self, layer: int, k: int | None = None) -> np.ndarray:
        """int32 [T, k] stand-in top-k rows: row t holds min(ctx, k) distinct
        positions of [0, ctx) in random order, then -1 (ctx = pos(t) + 1)."""
        k = self.index_topk if k is None else k
        qsl = self.query_start_loc
        out = np.full((self.T, k), -1, np.int32)
        for r in range(self.R):
            pre = int(self.prefix_lens[r])
            for j in range(int(self.q_lens[r])):
                t = int(qsl[r]) + j
                ctx = pre + j + 1
                g = _rng(self.seed, self.workload_id, layer, _T_MLA_SEL, t)
                n = min(ctx, k)
                out[t, :n] = g.choice(ctx, n, replace=False) if n < ctx else g.permutation(ctx)
        return out

    @property
    def pairs_per_full_layer(self) -> int:
        """Sum over query tokens of the keys each one sees (causal, itself
        included; with compress_ratio N, the (pos + 1) // N entries)."""
        pre = self.prefix_lens.astype(np.int64)
        ql = self.q_lens.astype(np.int64)
        if self.compress_ratio == 1:
            # token j (0-based) of request r sees pre[r] + j + 1 keys
            return int(np.sum(ql * pre + ql * (ql + 1) // 2))
        pos = np.repeat(pre, ql) + (np.arange(int(ql.sum())) - np.repeat(np.cumsum(ql) - ql, ql))
        return int(np.sum((pos + 1) // self.compress_ratio))

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "requests": self.R,
            "query_tokens": self.T,
            "heads": self.H,
            "head_dim": HEAD_DIM,
            "index_topk": self.index_topk,
            "layers": self.num_layers,
            "pattern": self.pattern,
            "freq": self.freq,
            "offset": self.offset,
            "max_num_batched_tokens": self.max_num_batched_tokens,
            "pages_per_layer": self.num_pages,
            "compress_ratio": self.compress_ratio,
            "pairs_per_full_layer": self.pairs_per_full_layer,
            "seed": self.seed,
        }


def _pages_for(seq_lens: np.ndarray) -> np.ndarray:
    return (seq_lens.astype(np.int64) + PAGE_TOKENS - 1) // PAGE_TOKENS


def _scatter_pages(seed: int, wid: int, seq_lens: np.ndarray, pool: int,
                   max_blocks: int) -> np.ndarray:
    """Block table whose rows take consecutive slices of a random pool permutation."""
    perm = _rng(seed, wid, 0, _T_PERM).permutation(pool).astype(np.int32)
    need = _pages_for(seq_lens)
    bt = np.full((seq_lens.shape[0], max_blocks), -1, dtype=np.int32)
    at = 0
    for r, n in enumerate(need):
        bt[r, :n] = perm[at:at + n]
        at += int(n)
    assert at <= pool
    return bt


def make_workload(workload_id: int, seed: int = 0, scale: float = 1.0) -> Workload:
    """Build the metadata of one workload; ``scale`` < 1 shrinks context lengths.

    ``scale`` exists so tests can run the same structure at oracle-friendly
    sizes; the published shapes are ``scale=1``.
    """
    wid = int(workload_id)
    name = WORKLOAD_NAMES[wid]
    if wid == 0:
        # 1 request of 256 new tokens, no prefix, H=4, k=32, stack 'FS', 16-page pool
        q_lens = np.array([256], np.int32)
        seq_lens = np.array([256], np.int32)
        pool = 16
        bt = _scatter_pages(seed, wid, seq_lens, pool, 4)
        return Workload(wid, name, seed, H=4, index_topk=32, num_layers=2, pattern="FS",
                        freq=1, offset=2, q_lens=q_lens, seq_lens=seq_lens, block_table=bt,
                        num_pages=pool, max_num_batched_tokens=256)
    if wid == 1:
        # 64 decode requests, context ~ U[1024, 8192], H=64, k=2048, 4 layers all F
        R = 64
        lo, hi = 1024, 8192
        ctx = _rng(seed, wid, 0, _T_CTX).integers(lo, hi, size=R, endpoint=True)
        ctx = np.maximum(2, np.round(ctx * scale)).astype(np.int32)
        q_lens = np.ones(R, np.int32)
        pool = int(_pages_for(ctx).sum())
        bt = _scatter_pages(seed, wid, ctx, pool, int(_pages_for(np.array([max(2, round(hi * scale))]))[0]))
        return Workload(wid, name, seed, H=64, index_topk=2048, num_layers=4, pattern=None,
                        freq=1, offset=2, q_lens=q_lens, seq_lens=ctx, block_table=bt,
                        num_pages=pool, max_num_batched_tokens=R)
    if wid == 2:
        # 1 request: 16384 cached prefix + 8192-token suffix chunk, outlier key channels x20
        prefix = max(1, int(round(16384 * scale)))
        suffix = max(1, int(round(8192 * scale)))
        q_lens = np.array([suffix], np.int32)
        seq_lens = np.array([prefix + suffix], np.int32)
        pool = int(_pages_for(seq_lens).sum())
        bt = _scatter_pages(seed, wid, seq_lens, pool, int(_pages_for(seq_lens)[0]))
        orng = _rng(seed, wid, 0, _T_OUTLIER)
        n_out = int(orng.choice([1, 2]))   # 1 % of 128 channels, rounded either way
        chans = np.sort(orng.choice(HEAD_DIM, n_out, replace=False)).astype(np.int64)
        return Workload(wid, name, seed, H=64, index_topk=2048, num_layers=1, pattern=None,
                        freq=1, offset=2, q_lens=q_lens, seq_lens=seq_lens, block_table=bt,
                        num_pages=pool, max_num_batched_tokens=max(8192, suffix),
                        outlier_channels=chans, outlier_scale=20.0)
    if wid == 3:
        # 256 decode requests (context log-uniform [4096, 65536]) + 4 prefill chunks of
        # 1024 tokens (context U[2048, 8192]); 61 layers, freq 4, offset 2
        crng = _rng(seed, wid, 0, _T_CTX)
        n_dec, n_pre = 256, 4
        chunk = max(1, int(round(1024 * scale)))
        dec_ctx = np.exp(crng.uniform(math.log(4096), math.log(65536), size=n_dec))
        dec_ctx = np.maximum(2, np.round(dec_ctx * scale)).astype(np.int32)
        pre_ctx = crng.integers(2048, 8192, size=n_pre, endpoint=True)
        pre_ctx = np.maximum(chunk, np.round(pre_ctx * scale)).astype(np.int32)
        q_lens = np.concatenate([np.ones(n_dec, np.int32), np.full(n_pre, chunk, np.int32)])
        seq_lens = np.concatenate([dec_ctx, pre_ctx]).astype(np.int32)
        pool = int(_pages_for(seq_lens).sum())
        mb = int(_pages_for(np.array([max(int(seq_lens.max()), 1)]))[0])
        bt = _scatter_pages(seed, wid, seq_lens, pool, mb)
        return Workload(wid, name, seed, H=64, index_topk=2048, num_layers=61, pattern=None,
                        freq=4, offset=2, q_lens=q_lens, seq_lens=seq_lens, block_table=bt,
                        num_pages=pool, max_num_batched_tokens=8192)
    if wid == 4:
        # 4 requests x 1,048,576 cached tokens + 1 new token; 78 layers, 21 F / 57 S pattern
        R = 4
        cached = max(1, int(round(1048576 * scale)))
        q_lens = np.ones(R, np.int32)
        seq_lens = np.full(R, cached + 1, np.int32)
        pool = int(_pages_for(seq_lens).sum())
        bt = _scatter_pages(seed, wid, seq_lens, pool, int(_pages_for(seq_lens)[0]))
        full = _rng(seed, wid, 0, _T_PATTERN).choice(76, 19, replace=False) + 2
        chars = ["S"] * 78
        for i in [0, 1, *full.tolist()]:
            chars[i] = "F"
        return Workload(wid, name, seed, H=64, index_topk=2048, num_layers=78,
                        pattern="".join(chars), freq=1, offset=2, q_lens=q_lens,
                        seq_lens=seq_lens, block_table=bt, num_pages=pool,
                        max_num_batched_tokens=R)
    if wid == 5:
        # 64 decode requests with one speculative (MTP) token each: 2 query rows per
        # request, the second seeing one more key; context ~ U[1024, 8192], H=64,
        # k=2048, 4 layers all F
        R, q = 64, 2
        lo, hi = 1024, 8192
        ctx = _rng(seed, wid, 0, _T_CTX).integers(lo, hi, size=R, endpoint=True)
        ctx = np.maximum(q + 1, np.round(ctx * scale)).astype(np.int32)
        q_lens = np.full(R, q, np.int32)
        pool = int(_pages_for(ctx).sum())
        bt = _scatter_pages(seed, wid, ctx, pool, int(_pages_for(np.array([max(q + 1, round(hi * scale))]))[0]))
        return Workload(wid, name, seed, H=64, index_topk=2048, num_layers=4, pattern=None,
                        freq=1, offset=2, q_lens=q_lens, seq_lens=ctx, block_table=bt,
                        num_pages=pool, max_num_batched_tokens=R * q)
    if wid == 6:
        # 64 decode requests, context log-uniform [16384, 131072], compressed indexer
        # cache (one entry per 4 tokens), H=64, k=2048, 4 layers all F
        R, ratio = 64, 4
        ctx = np.exp(_rng(seed, wid, 0, _T_CTX).uniform(math.log(16384), math.log(131072), size=R))
        ctx = np.maximum(ratio, np.round(ctx * scale)).astype(np.int32)
        q_lens = np.ones(R, np.int32)
        ent = ctx // ratio
        pool = int(_pages_for(ent).sum())
        mb = int(_pages_for(np.array([max(1, round(131072 * scale) // ratio)]))[0])
        bt = _scatter_pages(seed, wid, ent, pool, max(mb, int(_pages_for(ent).max())))
        return Workload(wid, name, seed, H=64, index_topk=2048, num_layers=4, pattern=None,
                        freq=1, offset=2, q_lens=q_lens, seq_lens=ctx, block_table=bt,
                        num_pages=pool, max_num_batched_tokens=R, compress_ratio=ratio)
    raise ValueError(f"unknown workload {workload_id}")
