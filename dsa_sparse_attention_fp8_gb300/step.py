"""One indexer forward step over an F/S layer stack, with reusable buffers.

`IndexerStep` owns the per-step device buffers (query rows, new keys, batch
metadata, the shared top-k buffer, workspace) and calls
``dsa_layer_stack_run`` on them, eagerly or as a captured CUDA graph.
`run_from_host` is the end-to-end call a serving loop makes: copy this
step's inputs from (pinned) host memory, run the stack, copy the top-k rows
back.  The page pools are device-resident state and are not copied.
"""

from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import binding


class IndexerStep:
    def __init__(self, *, num_layers: int, pattern: Optional[str], freq: int, offset: int,
                 H: int, index_topk: int, T: int, R: int, max_blocks: int, num_pages: int,
                 max_num_batched_tokens: int, k_caches: Sequence[Optional[torch.Tensor]],
                 device="cuda", time_score_kernels: bool = False, bf16: bool = False,
                 compress_ratio: int = 1):
        self.num_layers, self.pattern, self.freq, self.offset = num_layers, pattern, freq, offset
        self.H, self.k, self.T, self.R = H, index_topk, T, R
        self.max_blocks, self.num_pages = max_blocks, num_pages
        self.device = torch.device(device)
        self.bf16 = bf16   # BF16 keys and queries, quantised by the cache-write launch
        self.compress_ratio = compress_ratio  # tokens per cache entry (compressed caches)
        if bf16 and compress_ratio != 1:
            raise ValueError("the BF16 layer stack has no compressed form")
        self.input_keys = ("k", "q", "w") if bf16 else ("k", "q_fp8", "q_scale", "w")
        self.full = [binding.layer_is_full(l, pattern, freq, offset) for l in range(num_layers)]
        dev = self.device
        self.query_start_loc = torch.zeros(R + 1, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros(R, dtype=torch.int32, device=dev)
        self.block_table = torch.zeros((R, max_blocks), dtype=torch.int32, device=dev)
        self.topk = torch.full((max_num_batched_tokens, index_topk), -1, dtype=torch.int32,
                               device=dev)
        # the keys a row sees are bounded by the block table: max_blocks pages of 64
        self.workspace = binding.alloc_workspace(T, H, R, index_topk, device=dev,
                                                 max_ctx=max_blocks * 64)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.layers: list[Optional[dict]] = []
        for l in range(num_layers):
            if not self.full[l]:
                self.layers.append(None)
                continue
            cache = k_caches[l]
            assert cache is not None and cache.shape == (num_pages, binding.PAGE_BYTES)
            io = {
                "k": torch.zeros((T, binding.HEAD_DIM),
                                 dtype=torch.bfloat16 if bf16 else torch.float32, device=dev),
                "q_fp8": torch.zeros((T, H, binding.HEAD_DIM), dtype=torch.uint8, device=dev),
                "q_scale": torch.ones((T, H), dtype=torch.float32, device=dev),
                "w": torch.zeros((T, H), dtype=torch.float32, device=dev),
                "k_cache": cache,
            }
            if bf16:
                io["q"] = torch.zeros((T, H, binding.HEAD_DIM), dtype=torch.bfloat16, device=dev)
            if time_score_kernels:
                io["score_begin"] = torch.cuda.Event(enable_timing=True)
                io["score_end"] = torch.cuda.Event(enable_timing=True)
                # torch creates the CUDA event on first record
                io["score_begin"].record()
                io["score_end"].record()
            self.layers.append(io)
        self.graph: Optional[torch.cuda.CUDAGraph] = None        # with the kernel-timing events
        self.graph_plain: Optional[torch.cuda.CUDAGraph] = None  # without them
        self.launches_per_step = 0

    # -------------------------------------------------------------- inputs
    def set_metadata(self, query_start_loc, seq_lens, block_table, non_blocking=False) -> None:
        self.query_start_loc.copy_(query_start_loc, non_blocking=non_blocking)
        self.seq_lens.copy_(seq_lens, non_blocking=non_blocking)
        self.block_table.copy_(block_table, non_blocking=non_blocking)

    def set_layer(self, layer: int, *inputs, non_blocking=False) -> None:
        """This step's inputs of F layer `layer`: (k, q_fp8, q_scale, w), or
        (k, q, w) in BF16 mode."""
        io = self.layers[layer]
        assert len(inputs) == len(self.input_keys)
        for key, t in zip(self.input_keys, inputs):
            io[key].copy_(t, non_blocking=non_blocking)

    # -------------------------------------------------------------- running
    def launch(self, timed: bool = True) -> None:
        """One step.  timed=False leaves out the scoring kernels' timing events
        (an event between the cache write and the scoring kernel would keep
        the scoring kernel from overlapping the write's tail)."""
        layers = self.layers
        if not timed:
            layers = [None if io is None else {k: v for k, v in io.items()
                                               if k not in ("score_begin", "score_end")}
                      for io in self.layers]
        args = (layers, self.pattern, self.freq, self.offset, self.H, self.query_start_loc,
                self.seq_lens, self.block_table, self.num_pages, self.k, self.topk,
                self.workspace)
        if self.bf16:
            binding.layer_stack_run_bf16(*args, status=self.status, T=self.T)
        else:
            binding.layer_stack_run(*args, status=self.status, T=self.T,
                                    compress_ratio=self.compress_ratio)
        self.launches_per_step = binding.last_launch_count()

    def capture(self) -> None:
        """Record one step as two CUDA graphs, with and without the kernel-timing
        events (after one eager step for warm-up)."""
        self.launch()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.launch(timed=True)
        torch.cuda.synchronize()
        self.graph = g
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.launch(timed=False)
        torch.cuda.synchronize()
        self.graph_plain = g

    def run(self, timed: bool = True) -> None:
        g = self.graph if timed else self.graph_plain
        if g is not None:
            g.replay()
        else:
            self.launch(timed)

    def uses_row_selection(self) -> bool:
        """True when this batch's rows are scored into workspace rows and
        selected by the row kernel (the workspace was sized with room for
        them), False when the scoring kernel selects in place."""
        base = binding.workspace_bytes(self.T, self.H, self.R, self.k)
        return self.workspace.numel() > base

    def score_kernel_ms(self) -> list[float]:
        """Durations of the last step's scoring + selection launches, per F layer
        (needs time_score_kernels)."""
        return [io["score_begin"].elapsed_time(io["score_end"])
                for io in self.layers if io is not None and "score_begin" in io]

    # -------------------------------------------------------------- end to end
    def host_input_bytes(self, host: dict) -> int:
        n = sum(t.numel() * t.element_size() for t in host["meta"])
        for l, io in host["layers"].items():
            n += sum(t.numel() * t.element_size() for t in io)
        return n

    def run_from_host(self, host: dict, out: torch.Tensor) -> None:
        """H2D of this step's inputs, the stack, D2H of rows [0, T) of the top-k buffer.

        ``host["meta"]`` = (query_start_loc, seq_lens, block_table) and
        ``host["layers"][l]`` = the layer's inputs as set_layer takes them, pinned
        CPU tensors;
        ``out`` is a pinned int32 [T, index_topk] CPU tensor.  Asynchronous on
        the current stream.
        """
        self.set_metadata(*host["meta"], non_blocking=True)
        for l, io in host["layers"].items():
            self.set_layer(l, *io, non_blocking=True)
        self.run(timed=False)
        out.copy_(self.topk[: self.T], non_blocking=True)
