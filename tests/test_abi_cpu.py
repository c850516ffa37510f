"""The C-ABI library on the host (no GPU): it loads, exports every symbol the
header declares, and its pure-host logic (layer schedule, workspace sizing,
argument checks that fail before any launch) behaves as documented."""

import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle as O
from conftest import ROOT, golden

HEADER = ROOT / "include" / "dsa_indexer.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["dsa_indexer_write_k", "dsa_indexer_score_topk", "dsa_layer_stack_run",
              "dsa_layer_is_full", "dsa_indexer_workspace_bytes", "dsa_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from dsa_sparse_attention_fp8_gb300 import binding
    names = declared_functions()
    assert sorted(binding.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.dsa_abi_version() == 100


def test_layer_is_full_matches_oracle(lib):
    from dsa_sparse_attention_fp8_gb300 import binding
    g = golden("index_topk_pattern_61.json")
    for l in range(70):
        assert binding.layer_is_full(l, g["pattern"]) == O.layer_is_full(l, g["pattern"])
    for freq in range(1, 9):
        for off in range(0, 5):
            for l in range(80):
                assert binding.layer_is_full(l, None, freq, off) == O.layer_is_full(l, None, freq, off)
    g4 = golden("freq4_offset2_61.json")
    full = [l for l in range(61) if binding.layer_is_full(l, None, 4, 2)]
    assert full == g4["full_layers"]


def test_layer_is_full_rejects_bad_input(lib):
    assert lib.dsa_layer_is_full(0, b"FXS", 1, 2) == -1
    assert b"neither" not in lib.dsa_last_error()  # message is the library's own
    assert b"pattern" in lib.dsa_last_error()
    assert lib.dsa_layer_is_full(3, None, 0, 2) == -1
    assert lib.dsa_layer_is_full(-1, None, 1, 2) == -1


def test_workspace_bytes(lib):
    from dsa_sparse_attention_fp8_gb300 import binding
    a = binding.workspace_bytes(64, 64, 64, 2048)
    b = binding.workspace_bytes(8192, 64, 1, 2048)
    assert a > 0 and b > 0 and a % 256 == 0
    assert binding.workspace_bytes(8192, 64, 260, 2048) >= binding.workspace_bytes(4096, 64, 260, 2048)
    assert lib.dsa_indexer_workspace_bytes(64, 12, 64, 0, 2048) == 0     # unsupported H
    assert lib.dsa_indexer_workspace_bytes(64, 64, 64, 0, 4096) == 0     # index_topk too large
    assert lib.dsa_indexer_workspace_bytes(-1, 64, 64, 0, 2048) == 0


def test_argument_checks_fail_before_any_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # null metadata
    rc = lib.dsa_indexer_score_topk(fake, fake, fake, 4, 64, fake, 16, None, None, 1, None, 4,
                                    2048, fake, 4, None, 0, fake, 1 << 30, None, None)
    assert rc == -1
    # unsupported head count
    rc = lib.dsa_indexer_score_topk(fake, fake, fake, 4, 12, fake, 16, fake, fake, 1, fake, 4,
                                    2048, fake, 4, None, 0, fake, 1 << 30, None, None)
    assert rc == -2
    # T above max_num_batched_tokens
    rc = lib.dsa_indexer_score_topk(fake, fake, fake, 9, 64, fake, 16, fake, fake, 1, fake, 4,
                                    2048, fake, 8, None, 0, fake, 1 << 30, None, None)
    assert rc == -1
    # workspace too small
    rc = lib.dsa_indexer_score_topk(fake, fake, fake, 4, 64, fake, 16, fake, fake, 1, fake, 4,
                                    2048, fake, 4, None, 0, fake, 16, None, None)
    assert rc == -3
    # misaligned workspace
    rc = lib.dsa_indexer_score_topk(fake, fake, fake, 4, 64, fake, 16, fake, fake, 1, fake, 4,
                                    2048, fake, 4, None, 0, P(0x1010), 1 << 30, None, None)
    assert rc == -1
    # write: null pointers / bad sizes
    assert lib.dsa_indexer_write_k(None, 4, fake, fake, 1, fake, 4, fake, 16, None, None, None) == -1
    assert lib.dsa_indexer_write_k(fake, 4, fake, fake, 0, fake, 4, fake, 16, None, None, None) == -1
    assert lib.dsa_quantize_fp8_blocks(None, 4, fake, fake, None) == -1


def test_stack_rejects_bad_schedules(lib):
    from dsa_sparse_attention_fp8_gb300.binding import LayerIO
    P = ctypes.c_void_p
    fake = P(0x1000)
    layers = (LayerIO * 3)()
    for i in range(3):
        layers[i] = LayerIO(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, None, None)

    def run(pattern, freq, lay=layers, n=3):
        return lib.dsa_layer_stack_run(n, pattern, freq, 2, lay, 4, 64, fake, fake, 1, fake, 4,
                                       16, 2048, fake, 4, None, None, fake, 1 << 30, None, None)
    assert run(b"SFF", 1) == -1                 # first layer S
    assert run(b"FQF", 1) == -1                 # bad character
    assert run(None, 0) == -1                   # freq 0
    empty = (LayerIO * 3)()
    empty[0] = LayerIO(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, None, None)
    assert run(b"FSF", 1, empty) == -1          # F layer 2 lacks inputs
    assert b"layer 2" in lib.dsa_last_error()
    # T == 0: valid no-op, nothing launched
    assert lib.dsa_layer_stack_run(3, b"FSS", 1, 2, empty, 0, 64, fake, fake, 1, fake, 4, 16,
                                   2048, fake, 4, None, None, fake, 1 << 30, None, None) == 0
    assert lib.dsa_last_launch_count() == 0


def test_workspace_rows_sizing(lib):
    """max_ctx in (0, 8192] adds T rows of max_ctx rounded up to 128 keys (4 B
    each) plus T key counts (rounded to 256 B); beyond 8192, or rows over
    256 MB in all, adds nothing (the batch keeps the in-kernel selection)."""
    from dsa_sparse_attention_fp8_gb300 import binding
    base = binding.workspace_bytes(64, 64, 64, 2048)
    extra = lambda mc, T=64: binding.workspace_bytes(T, 64, T, 2048, max_ctx=mc) - \
        binding.workspace_bytes(T, 64, T, 2048)
    assert extra(0) == 0 and extra(-5) == 0
    for mc, stride in ((1, 128), (128, 128), (129, 256), (1000, 1024), (8192, 8192)):
        assert extra(mc) == 64 * stride * 4 + 256, mc
    assert extra(8193) == 0 and extra(1 << 20) == 0
    assert extra(8192, T=8192) == 8192 * 8192 * 4 + 8192 * 4          # exactly 256 MB of rows
    assert extra(8192, T=8193) == 0                                    # above 256 MB: none
    assert base == binding.workspace_bytes(64, 64, 64, 2048, max_ctx=0)


def test_no_alloc_entry_point_checks_arguments_like_the_workspace_one(lib):
    """The allocation-free scoring call reports a bad argument with the same
    code as dsa_indexer_score_topk (its checks run before its workspace-size
    check), and an oversized batch as WORKSPACE_TOO_SMALL; all before any
    CUDA call."""
    P = ctypes.c_void_p
    fake = P(0x1000)

    def both(T, H, R, k, mnbt=8, meta=fake):
        a = lib.dsa_indexer_score_topk(fake, fake, fake, T, H, fake, 16, meta, meta, R, meta, 4,
                                       k, fake, mnbt, None, 0, fake, 1 << 40, None, None)
        b = lib.dsa_indexer_score_topk_no_alloc(fake, fake, fake, T, H, fake, 16, meta, meta, R,
                                                meta, 4, k, fake, mnbt, None, None)
        return a, b

    assert both(-1, 64, 1, 2048) == (-1, -1)      # T < 0
    assert both(4, 64, 0, 2048) == (-1, -1)       # R < 1
    assert both(4, 12, 1, 2048) == (-2, -2)       # unsupported H
    assert both(4, 64, 1, 4096) == (-2, -2)       # index_topk too large
    assert both(9, 64, 1, 2048) == (-1, -1)       # T > max_num_batched_tokens
    assert both(4, 64, 1, 2048, meta=None) == (-1, -1)   # null metadata
    rc = lib.dsa_indexer_score_topk_no_alloc(fake, fake, fake, 8192, 64, fake, 16, fake, fake, 1,
                                             fake, 4, 2048, fake, 8192, None, None)
    assert rc == -3 and b"built-in workspace" in lib.dsa_last_error()
