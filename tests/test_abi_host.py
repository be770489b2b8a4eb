"""The C ABI library loads and exports every symbol include/attn_varlen.h
declares; argument checks that return before any CUDA call; the binding's
symbol table matches the header.  No GPU needed."""
import ctypes
import os
import re

import pytest

import variable_length_prefill_gb300 as vlp
from variable_length_prefill_gb300 import _binding as B

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "attn_varlen.h")


def _declared():
    names = set()
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b((?:attn_varlen|paged_attn|chunk_delta_rule)_\w+)\s*\(",
                                    src))
    return names


def _codes():
    src = open(HEADER).read()
    return {m.group(1): int(m.group(2))
            for m in re.finditer(r"#define\s+ATTN_VARLEN_(\w+)\s+(-?\d+)", src)}


def test_library_exports_every_declared_symbol():
    lib = vlp.load()
    declared = _declared()
    assert declared == set(B.SYMBOLS), (declared, set(B.SYMBOLS))
    for name in declared:
        assert hasattr(lib, name)


def test_return_codes_match_header():
    codes = _codes()
    assert codes["OK"] == B.OK
    for name in ("INVALID_ARG", "UNSUPPORTED_DIM", "MISALIGNED", "UNSUPPORTED_DEVICE",
                 "CUDA", "OOM", "DEVICE_TIMEOUT", "WORKSPACE_SMALL", "DRIVER", "NOALLOC_LIMIT",
                 "BAD_BLOCK_TABLE"):
        assert codes["ERR_" + name] == getattr(B, "ERR_" + name)
    for name, c in codes.items():
        if name == "NOALLOC_MAX_SEQS":
            assert c == B.NOALLOC_MAX_SEQS
            continue
        assert vlp.strerror(c) != "unknown error code"
    assert vlp.strerror(12345) == "unknown error code"


def test_version_and_workspace_size():
    lib = vlp.load()
    assert lib.attn_varlen_version() >= 100
    assert vlp.workspace_size(-1) == 0
    sizes = [vlp.workspace_size(n) for n in (0, 1, 9, 1000, 100000)]
    assert sizes == sorted(sizes) and all(s % 256 == 0 for s in sizes)
    # 8 tensor maps of 128 B per sequence plus order/prefix arrays
    assert vlp.workspace_size(1000) >= 1000 * 8 * 128 + 2 * 1000 * 4


P = 0x100000  # a fake, 16-byte aligned address; never dereferenced


@pytest.mark.parametrize("args,code", [
    # num_seqs < 0
    ((P, P, P, P, P, -1, 4, 72, P, None), B.ERR_INVALID_ARG),
    # num_heads < 1
    ((P, P, P, P, P, 1, 0, 72, P, None), B.ERR_INVALID_ARG),
    # head_dim not one of 64, 72, 80, 96, 128, 256
    ((P, P, P, P, P, 1, 4, 48, P, None), B.ERR_UNSUPPORTED_DIM),
    ((P, P, P, P, P, 1, 4, 100, P, None), B.ERR_UNSUPPORTED_DIM),
    ((P, P, P, P, P, 1, 4, 192, P, None), B.ERR_UNSUPPORTED_DIM),
    # null pointers
    ((None, P, P, P, P, 1, 4, 72, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, None, 1, 4, 128, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 4, 128, None, None), B.ERR_INVALID_ARG),
    # misaligned bf16 buffers / cu_seqlens
    ((P + 8, P, P, P, P, 1, 4, 72, P, None), B.ERR_MISALIGNED),
    ((P, P, P, P, P, 1, 4, 72, P + 2, None), B.ERR_MISALIGNED),
    ((P, P, P, P + 2, P, 1, 4, 72, P, None), B.ERR_MISALIGNED),
    # num_seqs == 0 is a no-op, even with null pointers
    ((None, None, None, None, None, 0, 4, 72, None, None), B.OK),
])
def test_argument_checks_need_no_gpu(args, code):
    assert vlp.load().attn_varlen_fwd(*args) == code


@pytest.mark.parametrize("args,code", [
    # (q, k, v, cu_q, cu_k, num_seqs, H, head_begin, head_count, D, causal, out, stream)
    ((P, P, P, P, P, 1, 4, -1, 2, 72, 0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 4, 3, 2, 72, 0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 4, 0, -1, 72, 0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 4, 5, 0, 72, 0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 0, 0, 0, 72, 0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 4, 0, 4, 48, 1, P, None), B.ERR_UNSUPPORTED_DIM),
    ((P + 8, P, P, P, P, 1, 4, 0, 4, 72, 0, P, None), B.ERR_MISALIGNED),
    # an empty head range or no sequence is a no-op
    ((P, P, P, P, P, 1, 4, 2, 0, 72, 0, P, None), B.OK),
    ((None, None, None, None, None, 0, 4, 0, 4, 72, 0, None, None), B.OK),
])
def test_head_range_checks_need_no_gpu(args, code):
    assert vlp.load().attn_varlen_fwd_heads(*args) == code


def test_workspace_variant_checks():
    lib = vlp.load()
    need = vlp.workspace_size(2)
    assert lib.attn_varlen_fwd_ws(P, P, P, P, P, 2, 4, 72, P, None, need, None) == B.ERR_INVALID_ARG
    assert lib.attn_varlen_fwd_ws(P, P, P, P, P, 2, 4, 72, P, P + 16, need, None) == B.ERR_MISALIGNED
    assert lib.attn_varlen_fwd_ws(P, P, P, P, P, 2, 4, 72, P, P, need - 1, None) == B.ERR_WORKSPACE_SMALL
    assert lib.attn_varlen_check_ws(None, None) == B.ERR_INVALID_ARG


def test_product_path_has_no_oracle_dependency():
    """The package never imports the CPU oracle."""
    pkg = os.path.dirname(vlp.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_oracle" not in text, f


@pytest.mark.parametrize("args,code", [
    # (query, k, v, tables, lens, n, Hq, Hkv, D, bs, max_blocks, num_blocks, dtype, out)
    ((P, P, P, P, P, -1, 4, 4, 128, 16, 1, 1, 0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 6, 4, 128, 16, 1, 1, 0, P, None), B.ERR_INVALID_ARG),   # Hq % Hkv
    ((P, P, P, P, P, 1, 4, 4, 96, 16, 1, 1, 0, P, None), B.ERR_UNSUPPORTED_DIM),
    ((P, P, P, P, P, 1, 4, 4, 128, 32, 1, 1, 0, P, None), B.ERR_INVALID_ARG),   # block_size
    ((P, P, P, P, P, 1, 4, 4, 128, 16, 1, 1, 2, P, None), B.ERR_INVALID_ARG),   # dtype
    ((P, P, P, P, P, 1, 4, 4, 128, 16, 0, 1, 0, P, None), B.ERR_INVALID_ARG),   # max_blocks
    ((None, P, P, P, P, 1, 4, 4, 128, 16, 1, 1, 0, P, None), B.ERR_INVALID_ARG),
    ((P + 8, P, P, P, P, 1, 4, 4, 128, 16, 1, 1, 0, P, None), B.ERR_MISALIGNED),
    ((P, P, P, P + 2, P, 1, 4, 4, 128, 16, 1, 1, 0, P, None), B.ERR_MISALIGNED),
    ((None, None, None, None, None, 0, 4, 4, 128, 16, 0, 0, 0, None, None), B.OK),
])
def test_paged_argument_checks_need_no_gpu(args, code):
    assert vlp.load().paged_attn_decode(*args) == code


@pytest.mark.parametrize("args,code", [
    # (q, k, v, h, g, B, T, Hq, Hv, K, V, cs, scale, out)
    ((P, P, P, P, P, -1, 64, 2, 4, 128, 128, 64, 0.0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P, P, P, 1, 64, 2, 4, 64, 128, 64, 0.0, P, None), B.ERR_UNSUPPORTED_DIM),
    ((P, P, P, P, P, 1, 64, 2, 4, 128, 128, 32, 0.0, P, None), B.ERR_INVALID_ARG),
    ((None, P, P, P, P, 1, 64, 2, 4, 128, 128, 64, 0.0, P, None), B.ERR_INVALID_ARG),
    ((P, P, P + 8, P, P, 1, 64, 2, 4, 128, 128, 64, 0.0, P, None), B.ERR_MISALIGNED),
    ((P, P, P, P, P + 2, 1, 64, 2, 4, 128, 128, 64, 0.0, P, None), B.ERR_MISALIGNED),
    ((None, None, None, None, None, 1, 0, 2, 4, 128, 128, 64, 0.0, None, None), B.OK),
])
def test_chunk_argument_checks_need_no_gpu(args, code):
    assert vlp.load().chunk_delta_rule_output(*args) == code
