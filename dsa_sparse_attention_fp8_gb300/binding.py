"""ctypes binding of libdsa_indexer.so: argument marshalling only.

Every computation happens in the library's CUDA kernels.  There is no CPU
fallback: if the shared library is missing, :func:`load` raises.  Tensors are
PyTorch tensors used as device buffers; the binding checks dtypes, devices,
shapes and contiguity, then passes raw pointers and the current CUDA stream.
"""

from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Optional, Sequence

import torch

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libdsa_indexer.so"

HEAD_DIM = 128
PAGE_TOKENS = 64
PAGE_BYTES = 8448
PAGE_SCALE_OFFSET = 8192
MAX_TOPK = 2048

DSA_OK = 0
ERRORS = {
    -1: "INVALID_ARG",
    -2: "UNSUPPORTED",
    -3: "WORKSPACE_TOO_SMALL",
    -4: "CUDA",
    -5: "TIMEOUT",
}
STATUS_BAD_PAGE = 0x1
STATUS_BAD_METADATA = 0x2
STATUS_TIMEOUT = 0x4

# every symbol declared in include/dsa_indexer.h
EXPORTS = (
    "dsa_abi_version",
    "dsa_last_error",
    "dsa_last_launch_count",
    "dsa_indexer_write_k",
    "dsa_indexer_write_k_bf16",
    "dsa_indexer_write_k_compressed",
    "dsa_quantize_fp8_blocks",
    "dsa_indexer_workspace_bytes",
    "dsa_indexer_score_topk",
    "dsa_indexer_score_topk_no_alloc",
    "dsa_indexer_score_topk_compressed",
    "dsa_indexer_no_alloc_workspace_bytes",
    "dsa_layer_is_full",
    "dsa_layer_stack_run",
    "dsa_layer_stack_run_bf16",
    "dsa_layer_stack_run_compressed",
    "dsa_mla_write_kv",
    "dsa_sparse_mla_attention",
)


class DsaError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


class LayerIO(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("q_fp8", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("score_begin", ctypes.c_void_p),
        ("score_end", ctypes.c_void_p),
    ]


class LayerIOBf16(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("q_fp8", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p),
        ("score_begin", ctypes.c_void_p),
        ("score_end", ctypes.c_void_p),
    ]


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


def _declare(lib: ctypes.CDLL) -> None:
    lib.dsa_abi_version.restype = _I
    lib.dsa_abi_version.argtypes = []
    lib.dsa_last_error.restype = ctypes.c_char_p
    lib.dsa_last_error.argtypes = []
    lib.dsa_last_launch_count.restype = _I
    lib.dsa_last_launch_count.argtypes = []
    lib.dsa_indexer_write_k.restype = _I
    lib.dsa_indexer_write_k.argtypes = [_P, _I, _P, _P, _I, _P, _I, _P, _I64, _P, _P, _P]
    lib.dsa_indexer_write_k_bf16.restype = _I
    lib.dsa_indexer_write_k_bf16.argtypes = [
        _P, _I, _P, _P, _I, _P, _I, _P, _I64, _P, _I, _P, _P, _P, _P, _P]
    lib.dsa_indexer_write_k_compressed.restype = _I
    lib.dsa_indexer_write_k_compressed.argtypes = [
        _P, _I, _P, _P, _I, _P, _I, _P, _I64, _I, _P, _P, _P]
    lib.dsa_quantize_fp8_blocks.restype = _I
    lib.dsa_quantize_fp8_blocks.argtypes = [_P, _I64, _P, _P, _P]
    lib.dsa_indexer_workspace_bytes.restype = _SZ
    lib.dsa_indexer_workspace_bytes.argtypes = [_I, _I, _I, _I64, _I]
    lib.dsa_indexer_score_topk.restype = _I
    lib.dsa_indexer_score_topk.argtypes = [
        _P, _P, _P, _I, _I, _P, _I64, _P, _P, _I, _P, _I, _I, _P, _I, _P, _I64, _P, _SZ, _P, _P]
    lib.dsa_indexer_score_topk_no_alloc.restype = _I
    lib.dsa_indexer_score_topk_no_alloc.argtypes = [
        _P, _P, _P, _I, _I, _P, _I64, _P, _P, _I, _P, _I, _I, _P, _I, _P, _P]
    lib.dsa_indexer_score_topk_compressed.restype = _I
    lib.dsa_indexer_score_topk_compressed.argtypes = [
        _P, _P, _P, _I, _I, _P, _I64, _P, _P, _I, _P, _I, _I, _I, _P, _I, _P, _I64, _P, _SZ, _P,
        _P]
    lib.dsa_indexer_no_alloc_workspace_bytes.restype = _SZ
    lib.dsa_indexer_no_alloc_workspace_bytes.argtypes = []
    lib.dsa_layer_is_full.restype = _I
    lib.dsa_layer_is_full.argtypes = [_I, ctypes.c_char_p, _I, _I]
    lib.dsa_layer_stack_run.restype = _I
    lib.dsa_layer_stack_run.argtypes = [
        _I, ctypes.c_char_p, _I, _I, ctypes.POINTER(LayerIO), _I, _I, _P, _P, _I, _P, _I, _I64,
        _I, _P, _I, ctypes.POINTER(ctypes.c_void_p), _P, _P, _SZ, _P, _P]
    lib.dsa_layer_stack_run_compressed.restype = _I
    lib.dsa_layer_stack_run_compressed.argtypes = [
        _I, ctypes.c_char_p, _I, _I, ctypes.POINTER(LayerIO), _I, _I, _P, _P, _I, _P, _I, _I64,
        _I, _I, _P, _I, ctypes.POINTER(ctypes.c_void_p), _P, _P, _SZ, _P, _P]
    lib.dsa_mla_write_kv.restype = _I
    lib.dsa_mla_write_kv.argtypes = [_P, _I, _P, _P, _I, _P, _I, _P, _I64, _P, _P, _P]
    lib.dsa_sparse_mla_attention.restype = _I
    lib.dsa_sparse_mla_attention.argtypes = [
        _P, _I, _I, _P, _I64, _P, _P, _I, _P, _I, _P, _I, ctypes.c_float, _P, _P, _P, _P]
    lib.dsa_layer_stack_run_bf16.restype = _I
    lib.dsa_layer_stack_run_bf16.argtypes = [
        _I, ctypes.c_char_p, _I, _I, ctypes.POINTER(LayerIOBf16), _I, _I, _P, _P, _I, _P, _I,
        _I64, _I, _P, _I, ctypes.POINTER(ctypes.c_void_p), _P, _P, _SZ, _P, _P]


def load() -> ctypes.CDLL:
    """Load the library (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise ImportError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(there is no CPU fallback for the indexer path)")
        lib = ctypes.CDLL(str(LIB_PATH))
        _declare(lib)
        _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc != DSA_OK:
        msg = load().dsa_last_error().decode(errors="replace")
        raise DsaError(rc, msg)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None:
        for i, (a, b) in enumerate(zip(t.shape, shape)):
            if b is not None and a != b:
                raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
        if len(t.shape) != len(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")


# ----------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------

def abi_version() -> int:
    return load().dsa_abi_version()


def last_launch_count() -> int:
    return load().dsa_last_launch_count()


def layer_is_full(layer_id: int, pattern: Optional[str] = None, freq: int = 1, offset: int = 2) -> bool:
    rc = load().dsa_layer_is_full(layer_id, None if pattern is None else pattern.encode(), freq, offset)
    if rc < 0:
        _check(rc)
    return bool(rc)


def workspace_bytes(T: int, H: int, R: int, index_topk: int, max_ctx: int = 0) -> int:
    n = load().dsa_indexer_workspace_bytes(T, H, R, max_ctx, index_topk)
    if n == 0:
        raise DsaError(-1, f"no workspace size for T={T}, H={H}, R={R}, index_topk={index_topk}")
    return int(n)


def alloc_workspace(T: int, H: int, R: int, index_topk: int, device="cuda",
                    max_ctx: int = 0) -> torch.Tensor:
    """Workspace for score_topk / layer_stack_run.  0 < max_ctx <= 8192 (a bound on
    the keys any row sees) also makes room for decode rows to be scored into the
    workspace and selected by a second kernel (see dsa_indexer_workspace_bytes)."""
    n = workspace_bytes(T, H, R, index_topk, max_ctx)
    return torch.empty(n, dtype=torch.uint8, device=device)


def quantize_fp8_blocks(x: torch.Tensor, codes: Optional[torch.Tensor] = None,
                        scales: Optional[torch.Tensor] = None, stream=None):
    """x [..., 128] FP32 -> (codes uint8 [..., 128], scales FP32 [...])."""
    _need(x, "x", torch.float32)
    if x.shape[-1] != HEAD_DIM:
        raise ValueError("last dimension must be 128")
    nb = x.numel() // HEAD_DIM
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.float32)
    _check(load().dsa_quantize_fp8_blocks(_ptr(x), nb, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def write_k(k: torch.Tensor, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
            block_table: torch.Tensor, k_cache: torch.Tensor,
            slot_mapping: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
            stream=None) -> None:
    _check(load().dsa_indexer_write_k(*_write_k_args(
        k, query_start_loc, seq_lens, block_table, k_cache, slot_mapping, status, stream)))


def write_k_compressed(k: torch.Tensor, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                       block_table: torch.Tensor, k_cache: torch.Tensor, compress_ratio: int,
                       slot_mapping: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Cache write into a compressed cache: only tokens with
    (pos + 1) % compress_ratio == 0 are stored, as entry pos // compress_ratio."""
    a = _write_k_args(k, query_start_loc, seq_lens, block_table, k_cache, slot_mapping, status,
                      stream)
    _check(load().dsa_indexer_write_k_compressed(*a[:9], int(compress_ratio), *a[9:]))


def _write_k_args(k, query_start_loc, seq_lens, block_table, k_cache, slot_mapping, status,
                  stream):
    T = k.shape[0]
    R = seq_lens.shape[0]
    _need(k, "k", torch.float32, (T, HEAD_DIM))
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(k_cache, "k_cache", torch.uint8, (None, PAGE_BYTES))
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", torch.int64, (T,))
    if status is not None:
        _need(status, "status", torch.int32)
    return (_ptr(k), T, _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table),
            block_table.shape[1], _ptr(k_cache), k_cache.shape[0], _ptr(slot_mapping),
            _ptr(status), _stream(stream))


def write_k_bf16(k: torch.Tensor, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                 block_table: torch.Tensor, k_cache: torch.Tensor,
                 q: Optional[torch.Tensor] = None, q_fp8: Optional[torch.Tensor] = None,
                 q_scale: Optional[torch.Tensor] = None,
                 slot_mapping: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Cache write of BF16 keys; with ``q`` [T, H, 128] BF16 the same launch
    quantises the query rows into ``q_fp8`` [T, H, 128] uint8 and ``q_scale``
    [T, H] float32."""
    T = k.shape[0]
    R = seq_lens.shape[0]
    _need(k, "k", torch.bfloat16, (T, HEAD_DIM))
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(k_cache, "k_cache", torch.uint8, (None, PAGE_BYTES))
    H = 0
    if q is not None:
        H = q.shape[1]
        _need(q, "q", torch.bfloat16, (T, H, HEAD_DIM))
        _need(q_fp8, "q_fp8", torch.uint8, (T, H, HEAD_DIM))
        _need(q_scale, "q_scale", torch.float32, (T, H))
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", torch.int64, (T,))
    if status is not None:
        _need(status, "status", torch.int32)
    _check(load().dsa_indexer_write_k_bf16(
        _ptr(k), T, _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table),
        block_table.shape[1], _ptr(k_cache), k_cache.shape[0], _ptr(q), H, _ptr(q_fp8),
        _ptr(q_scale), _ptr(slot_mapping), _ptr(status), _stream(stream)))


def score_topk(q_fp8: torch.Tensor, q_scale: torch.Tensor, w: torch.Tensor,
               k_cache: torch.Tensor, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
               block_table: torch.Tensor, index_topk: int, topk_buffer: torch.Tensor,
               workspace: torch.Tensor, scores_out: Optional[torch.Tensor] = None,
               status: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(load().dsa_indexer_score_topk(*_score_args(
        q_fp8, q_scale, w, k_cache, query_start_loc, seq_lens, block_table, index_topk,
        topk_buffer, workspace, scores_out, status, stream)))


def score_topk_compressed(q_fp8: torch.Tensor, q_scale: torch.Tensor, w: torch.Tensor,
                          k_cache: torch.Tensor, query_start_loc: torch.Tensor,
                          seq_lens: torch.Tensor, block_table: torch.Tensor, compress_ratio: int,
                          index_topk: int, topk_buffer: torch.Tensor, workspace: torch.Tensor,
                          scores_out: Optional[torch.Tensor] = None,
                          status: Optional[torch.Tensor] = None, stream=None) -> None:
    """score_topk over a compressed cache: row t ranks the entries
    c < (pos + 1) // compress_ratio; indices (and scores_out columns) are entries."""
    a = _score_args(q_fp8, q_scale, w, k_cache, query_start_loc, seq_lens, block_table,
                    index_topk, topk_buffer, workspace, scores_out, status, stream)
    _check(load().dsa_indexer_score_topk_compressed(*a[:12], int(compress_ratio), *a[12:]))


def _score_args(q_fp8, q_scale, w, k_cache, query_start_loc, seq_lens, block_table, index_topk,
                topk_buffer, workspace, scores_out, status, stream):
    T, H = q_fp8.shape[0], q_fp8.shape[1]
    R = seq_lens.shape[0]
    _need(q_fp8, "q_fp8", torch.uint8, (T, H, HEAD_DIM))
    _need(q_scale, "q_scale", torch.float32, (T, H))
    _need(w, "w", torch.float32, (T, H))
    _need(k_cache, "k_cache", torch.uint8, (None, PAGE_BYTES))
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(topk_buffer, "topk_buffer", torch.int32, (None, index_topk))
    _need(workspace, "workspace", torch.uint8)
    ld = 0
    if scores_out is not None:
        _need(scores_out, "scores_out", torch.float32, (T, None))
        ld = scores_out.shape[1]
    if status is not None:
        _need(status, "status", torch.int32)
    return (_ptr(q_fp8), _ptr(q_scale), _ptr(w), T, H, _ptr(k_cache), k_cache.shape[0],
            _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table), block_table.shape[1],
            index_topk, _ptr(topk_buffer), topk_buffer.shape[0], _ptr(scores_out), ld,
            _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))


def score_topk_no_alloc(q_fp8: torch.Tensor, q_scale: torch.Tensor, w: torch.Tensor,
                        k_cache: torch.Tensor, query_start_loc: torch.Tensor,
                        seq_lens: torch.Tensor, block_table: torch.Tensor, index_topk: int,
                        topk_buffer: torch.Tensor, status: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """score_topk without a workspace argument: the library's built-in
    workspace is used and nothing is allocated (see include/dsa_indexer.h)."""
    T, H = q_fp8.shape[0], q_fp8.shape[1]
    R = seq_lens.shape[0]
    _need(q_fp8, "q_fp8", torch.uint8, (T, H, HEAD_DIM))
    _need(q_scale, "q_scale", torch.float32, (T, H))
    _need(w, "w", torch.float32, (T, H))
    _need(k_cache, "k_cache", torch.uint8, (None, PAGE_BYTES))
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(topk_buffer, "topk_buffer", torch.int32, (None, index_topk))
    if status is not None:
        _need(status, "status", torch.int32)
    _check(load().dsa_indexer_score_topk_no_alloc(
        _ptr(q_fp8), _ptr(q_scale), _ptr(w), T, H, _ptr(k_cache), k_cache.shape[0],
        _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table), block_table.shape[1],
        index_topk, _ptr(topk_buffer), topk_buffer.shape[0], _ptr(status), _stream(stream)))


def no_alloc_workspace_bytes() -> int:
    return int(load().dsa_indexer_no_alloc_workspace_bytes())


def layer_stack_run(layers: Sequence[Optional[dict]], pattern: Optional[str], freq: int,
                    offset: int, H: int, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                    block_table: torch.Tensor, num_pages: int, index_topk: int,
                    topk_buffer: torch.Tensor, workspace: torch.Tensor,
                    per_layer_out: Optional[Sequence[Optional[torch.Tensor]]] = None,
                    slot_mapping: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, T: Optional[int] = None,
                    stream=None, compress_ratio: int = 1) -> None:
    """Run the F/S layer stack.  ``layers[l]`` is a dict with keys k, q_fp8,
    q_scale, w, k_cache (and optionally score_begin / score_end, torch.cuda.Event
    objects created with enable_timing=True) for F layers, or None for S layers.
    ``compress_ratio`` > 1 runs dsa_layer_stack_run_compressed (compressed
    caches, one entry per compress_ratio tokens)."""
    R = seq_lens.shape[0]
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(topk_buffer, "topk_buffer", torch.int32, (None, index_topk))
    _need(workspace, "workspace", torch.uint8)
    L = len(layers)
    arr = (LayerIO * L)()
    for i, io in enumerate(layers):
        if io is None:
            continue
        if T is None:
            T = io["k"].shape[0]
        _need(io["k"], f"layers[{i}].k", torch.float32, (T, HEAD_DIM))
        _need(io["q_fp8"], f"layers[{i}].q_fp8", torch.uint8, (T, H, HEAD_DIM))
        _need(io["q_scale"], f"layers[{i}].q_scale", torch.float32, (T, H))
        _need(io["w"], f"layers[{i}].w", torch.float32, (T, H))
        _need(io["k_cache"], f"layers[{i}].k_cache", torch.uint8, (num_pages, PAGE_BYTES))
        ev0, ev1 = io.get("score_begin"), io.get("score_end")
        arr[i] = LayerIO(io["k"].data_ptr(), io["q_fp8"].data_ptr(), io["q_scale"].data_ptr(),
                         io["w"].data_ptr(), io["k_cache"].data_ptr(),
                         None if ev0 is None else ev0.cuda_event,
                         None if ev1 is None else ev1.cuda_event)
    if T is None:
        raise ValueError("no F layer given")
    outs = None
    if per_layer_out is not None:
        outs = (ctypes.c_void_p * L)()
        for i, o in enumerate(per_layer_out):
            if o is not None:
                _need(o, f"per_layer_out[{i}]", torch.int32, (T, index_topk))
                outs[i] = o.data_ptr()
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", torch.int64, (T,))
    if status is not None:
        _need(status, "status", torch.int32)
    head = (L, None if pattern is None else pattern.encode(), freq, offset, arr, T, H,
            _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table), block_table.shape[1],
            num_pages)
    tail = (index_topk, _ptr(topk_buffer), topk_buffer.shape[0], outs, _ptr(slot_mapping),
            _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    if compress_ratio == 1:
        _check(load().dsa_layer_stack_run(*head, *tail))
    else:
        _check(load().dsa_layer_stack_run_compressed(*head, int(compress_ratio), *tail))


def layer_stack_run_compressed(*args, compress_ratio: int, **kw) -> None:
    """dsa_layer_stack_run_compressed: layer_stack_run's arguments plus the ratio."""
    layer_stack_run(*args, compress_ratio=compress_ratio, **kw)


def layer_stack_run_bf16(layers: Sequence[Optional[dict]], pattern: Optional[str], freq: int,
                         offset: int, H: int, query_start_loc: torch.Tensor,
                         seq_lens: torch.Tensor, block_table: torch.Tensor, num_pages: int,
                         index_topk: int, topk_buffer: torch.Tensor, workspace: torch.Tensor,
                         per_layer_out: Optional[Sequence[Optional[torch.Tensor]]] = None,
                         slot_mapping: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, T: Optional[int] = None,
                         stream=None) -> None:
    """The F/S layer stack with BF16 inputs.  ``layers[l]`` is a dict with keys
    k [T, 128] and q [T, H, 128] (BF16), w, k_cache, and the scratch q_fp8 /
    q_scale that the cache-write launch fills, for F layers; None for S
    layers."""
    R = seq_lens.shape[0]
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(topk_buffer, "topk_buffer", torch.int32, (None, index_topk))
    _need(workspace, "workspace", torch.uint8)
    L = len(layers)
    arr = (LayerIOBf16 * L)()
    for i, io in enumerate(layers):
        if io is None:
            continue
        if T is None:
            T = io["k"].shape[0]
        _need(io["k"], f"layers[{i}].k", torch.bfloat16, (T, HEAD_DIM))
        _need(io["q"], f"layers[{i}].q", torch.bfloat16, (T, H, HEAD_DIM))
        _need(io["w"], f"layers[{i}].w", torch.float32, (T, H))
        _need(io["k_cache"], f"layers[{i}].k_cache", torch.uint8, (num_pages, PAGE_BYTES))
        _need(io["q_fp8"], f"layers[{i}].q_fp8", torch.uint8, (T, H, HEAD_DIM))
        _need(io["q_scale"], f"layers[{i}].q_scale", torch.float32, (T, H))
        ev0, ev1 = io.get("score_begin"), io.get("score_end")
        arr[i] = LayerIOBf16(io["k"].data_ptr(), io["q"].data_ptr(), io["w"].data_ptr(),
                             io["k_cache"].data_ptr(), io["q_fp8"].data_ptr(),
                             io["q_scale"].data_ptr(),
                             None if ev0 is None else ev0.cuda_event,
                             None if ev1 is None else ev1.cuda_event)
    if T is None:
        raise ValueError("no F layer given")
    outs = None
    if per_layer_out is not None:
        outs = (ctypes.c_void_p * L)()
        for i, o in enumerate(per_layer_out):
            if o is not None:
                _need(o, f"per_layer_out[{i}]", torch.int32, (T, index_topk))
                outs[i] = o.data_ptr()
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", torch.int64, (T,))
    if status is not None:
        _need(status, "status", torch.int32)
    _check(load().dsa_layer_stack_run_bf16(
        L, None if pattern is None else pattern.encode(), freq, offset, arr, T, H,
        _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table), block_table.shape[1],
        num_pages, index_topk, _ptr(topk_buffer), topk_buffer.shape[0], outs, _ptr(slot_mapping),
        _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)))


# ---------------------------------------------------------------- sparse MLA
MLA_DIM = 576
MLA_LATENT = 512
MLA_RECORD_BYTES = 656
MLA_PAGE_BYTES = 41984


def mla_write_kv(kv: torch.Tensor, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                 block_table: torch.Tensor, kv_cache: torch.Tensor,
                 slot_mapping: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Store each new token's [latent | RoPE] (FP32 [T, 576]) as its 656-byte
    record in kv_cache [num_pages, 41984] (dsa_mla_write_kv)."""
    T = kv.shape[0]
    R = seq_lens.shape[0]
    _need(kv, "kv", torch.float32, (T, MLA_DIM))
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(kv_cache, "kv_cache", torch.uint8, (None, MLA_PAGE_BYTES))
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", torch.int64, (T,))
    if status is not None:
        _need(status, "status", torch.int32)
    _check(load().dsa_mla_write_kv(
        _ptr(kv), T, _ptr(query_start_loc), _ptr(seq_lens), R, _ptr(block_table),
        block_table.shape[1], _ptr(kv_cache), kv_cache.shape[0], _ptr(slot_mapping),
        _ptr(status), _stream(stream)))


def sparse_mla_attention(q: torch.Tensor, kv_cache: torch.Tensor, query_start_loc: torch.Tensor,
                         seq_lens: torch.Tensor, block_table: torch.Tensor,
                         topk_indices: torch.Tensor, softmax_scale: float,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None):
    """Attention of each query row (q [T, Hq, 576] BF16) over the tokens its
    top-k row selects (dsa_sparse_mla_attention).  Returns (out [T, Hq, 512]
    BF16, lse [T, Hq] FP32)."""
    T, Hq = q.shape[0], q.shape[1]
    R = seq_lens.shape[0]
    _need(q, "q", torch.bfloat16, (T, Hq, MLA_DIM))
    _need(kv_cache, "kv_cache", torch.uint8, (None, MLA_PAGE_BYTES))
    _need(query_start_loc, "query_start_loc", torch.int32, (R + 1,))
    _need(seq_lens, "seq_lens", torch.int32, (R,))
    _need(block_table, "block_table", torch.int32, (R, None))
    _need(topk_indices, "topk_indices", torch.int32, (None, None))
    if topk_indices.shape[0] < T:
        raise ValueError("topk_indices has fewer rows than q")
    if out is None:
        out = torch.empty((T, Hq, MLA_LATENT), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, (T, Hq, MLA_LATENT))
    _need(lse, "lse", torch.float32, (T, Hq))
    if status is not None:
        _need(status, "status", torch.int32)
    _check(load().dsa_sparse_mla_attention(
        _ptr(q), T, Hq, _ptr(kv_cache), kv_cache.shape[0], _ptr(query_start_loc),
        _ptr(seq_lens), R, _ptr(block_table), block_table.shape[1], _ptr(topk_indices),
        topk_indices.shape[1], float(softmax_scale), _ptr(out), _ptr(lse), _ptr(status),
        _stream(stream)))
    return out, lse
