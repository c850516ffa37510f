"""Host -> device staging of a synthetic workload for the indexer library.

Uploads batch metadata, allocates one page pool per F layer, writes each
request's cached prefix through the library's own cache-write kernel (as the
earlier steps of a serving loop would have), and quantises the step's queries
with the library's block quantiser.  All arithmetic runs in the library.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import binding


@dataclass
class DeviceMeta:
    T: int
    R: int
    H: int
    index_topk: int
    num_pages: int
    max_blocks: int
    max_num_batched_tokens: int
    query_start_loc: torch.Tensor
    seq_lens: torch.Tensor
    block_table: torch.Tensor
    prefix_qsl: torch.Tensor
    prefix_lens: torch.Tensor


def stage_metadata(wl, device="cuda") -> DeviceMeta:
    dev = torch.device(device)
    pre = wl.prefix_lens.astype(np.int32)
    pre_qsl = np.zeros(wl.R + 1, np.int32)
    np.cumsum(pre, out=pre_qsl[1:])
    return DeviceMeta(
        T=wl.T, R=wl.R, H=wl.H, index_topk=wl.index_topk, num_pages=wl.num_pages,
        max_blocks=wl.max_blocks, max_num_batched_tokens=wl.max_num_batched_tokens,
        query_start_loc=torch.from_numpy(wl.query_start_loc).to(dev),
        seq_lens=torch.from_numpy(wl.seq_lens.astype(np.int32)).to(dev),
        block_table=torch.from_numpy(wl.block_table).to(dev),
        prefix_qsl=torch.from_numpy(pre_qsl).to(dev),
        prefix_lens=torch.from_numpy(pre).to(dev),
    )


def fill_prefix(wl, layer: int, meta: DeviceMeta, k_cache: torch.Tensor,
                chunk_tokens: int = 1 << 22) -> None:
    """Write every request's cached-prefix keys of `layer` into `k_cache`.

    Requests are written in batches of at most `chunk_tokens` entries, each
    batch as one cache-write call whose "new tokens" are the prefix entries
    (for a compressed cache, the entries completed before this step, stored
    at entry positions 0 .. prefix_entries-1).
    """
    dev = k_cache.device
    pre = wl.prefix_entries.astype(np.int64)
    r = 0
    while r < wl.R:
        rs, tot = [], 0
        while r < wl.R and (not rs or tot + pre[r] <= chunk_tokens):
            rs.append(r)
            tot += int(pre[r])
            r += 1
        rs = [x for x in rs if pre[x] > 0]
        if not rs:
            continue
        ks = np.concatenate([wl.k_prefix(layer, x) for x in rs], axis=0)
        qsl = np.zeros(len(rs) + 1, np.int32)
        np.cumsum(pre[rs], out=qsl[1:])
        seq = pre[rs].astype(np.int32)
        bt = wl.block_table[rs]
        binding.write_k(torch.from_numpy(ks).to(dev), torch.from_numpy(qsl).to(dev),
                        torch.from_numpy(seq).to(dev), torch.from_numpy(np.ascontiguousarray(bt)).to(dev),
                        k_cache)


def stage_layer(wl, layer: int, meta: DeviceMeta, device="cuda", fill: bool = True,
                cache_fill_byte: int = 0) -> dict:
    """Inputs of one F layer on the device: k, q_fp8, q_scale, w, k_cache."""
    dev = torch.device(device)
    k_cache = torch.full((wl.num_pages, binding.PAGE_BYTES), cache_fill_byte, dtype=torch.uint8,
                         device=dev)
    if fill:
        fill_prefix(wl, layer, meta, k_cache)
    k_new = torch.from_numpy(wl.k_new(layer)).to(dev)
    q = torch.from_numpy(wl.q(layer)).to(dev)
    q_fp8, q_scale = binding.quantize_fp8_blocks(q)
    w = torch.from_numpy(wl.w(layer)).to(dev)
    return {"k": k_new, "q_fp8": q_fp8, "q_scale": q_scale, "w": w, "k_cache": k_cache}


def stage_mla(wl, layer: int, meta: DeviceMeta, heads: int, device="cuda",
              cache_fill_byte: int = 0) -> dict:
    """Sparse-MLA inputs of one layer on the device: the main-KV pool holding
    every cached prefix and this step's records (written by the library's
    record write), BF16 queries and the stand-in top-k rows."""
    dev = torch.device(device)
    cache = torch.full((wl.num_pages, binding.MLA_PAGE_BYTES), cache_fill_byte, dtype=torch.uint8,
                       device=dev)
    pre = wl.prefix_lens.astype(np.int64)
    for r in range(wl.R):
        if pre[r] == 0:
            continue
        qsl = torch.tensor([0, int(pre[r])], dtype=torch.int32, device=dev)
        seq = torch.tensor([int(pre[r])], dtype=torch.int32, device=dev)
        bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[r:r + 1])).to(dev)
        binding.mla_write_kv(torch.from_numpy(wl.mla_kv_prefix(layer, r)).to(dev), qsl, seq, bt,
                             cache)
    binding.mla_write_kv(torch.from_numpy(wl.mla_kv_new(layer)).to(dev), meta.query_start_loc,
                         meta.seq_lens, meta.block_table, cache)
    q = torch.from_numpy(wl.mla_q(layer, heads)).to(dev).bfloat16()
    topk = torch.from_numpy(wl.selection_rows(layer)).to(dev)
    return {"kv_cache": cache, "q": q, "topk": topk}
