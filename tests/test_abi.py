"""The C ABI library on the host (no GPU): it loads, exports every symbol
include/fa.h declares, and rejects bad arguments before touching a device."""

import ctypes
import os
import re

import pytest

import exact_io_aware_33_gb300 as fa
from conftest import GOLDEN, ROOT


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_33_gb300 import build
    build.build()
    return fa.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names
    for name in names:
        assert hasattr(lib, name), name
        assert name in fa.SIGNATURES, name


def test_header_return_codes_match_binding():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    codes = dict((m[0], int(m[1])) for m in re.findall(r"#define (FA_[A-Z_]+) (-?\d+)", text))
    for name, val in codes.items():
        assert getattr(fa, name) == val, name


def test_strerror_and_version(lib):
    for code in (0, -1, -2, -3, -4, -5, 17):
        s = lib.fa_strerror(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.fa_version() >= 100


def test_workspace_bytes(lib):
    assert lib.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert lib.fa_bwd_workspace_bytes(-1, 1, 1, 64) == 0
    # D and the log2-domain LSE, each fp32 over N rounded up to 128, then the
    # fp32 dQ accumulator over the same padded rows
    B, H, N, d = 2, 3, 100, 64
    n_pad = 128
    assert lib.fa_bwd_workspace_bytes(B, H, N, d) == 2 * B * H * n_pad * 4 + B * H * n_pad * d * 4
    assert lib.fa_bwd_workspace_bytes(1, 1, 256, 128) == 2 * 256 * 4 + 256 * 128 * 4


NULL = ctypes.c_void_p(0)
ALIGNED = ctypes.c_void_p(0x100000)    # never dereferenced: checks fail first
MISALIGNED = ctypes.c_void_p(0x100008)


@pytest.mark.parametrize("args,code", [
    ((1, 1, -1, 64, 0.125), fa.FA_ERR_INVALID),
    ((-2, 1, 8, 64, 0.125), fa.FA_ERR_INVALID),
    ((1, 1, 8, 64, float("nan")), fa.FA_ERR_INVALID),
    ((1, 1, 8, 64, float("inf")), fa.FA_ERR_INVALID),
    ((1, 1, 8, 64, -0.5), fa.FA_ERR_INVALID),
    ((1, 1, 8, 96, 0.125), fa.FA_ERR_UNSUPPORTED),
    ((1, 1, 8, 512, 0.125), fa.FA_ERR_UNSUPPORTED),
    ((1, 1, 8, 32, 0.125), fa.FA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_sizes(lib, args, code):
    B, H, N, d, scale = args
    p = ALIGNED
    assert lib.fa_fwd(p, p, p, p, p, B, H, N, d, 0, scale) == code


def test_fwd_rejects_bad_pointers(lib):
    p = ALIGNED
    assert lib.fa_fwd(NULL, p, p, p, p, 1, 1, 8, 64, 0, 0.125) == fa.FA_ERR_INVALID
    assert lib.fa_fwd(p, p, MISALIGNED, p, p, 1, 1, 8, 64, 0, 0.125) == fa.FA_ERR_INVALID
    assert lib.fa_fwd(p, p, p, p, NULL, 1, 1, 8, 64, 1, 0.125) == fa.FA_ERR_INVALID


def test_empty_problems_are_no_ops(lib):
    assert lib.fa_fwd(NULL, NULL, NULL, NULL, NULL, 0, 4, 128, 64, 0, 0.125) == fa.FA_OK
    assert lib.fa_fwd(NULL, NULL, NULL, NULL, NULL, 2, 4, 0, 128, 1, 0.125) == fa.FA_OK
    n = NULL
    assert lib.fa_bwd(n, n, n, n, n, n, n, n, n, 1, 0, 64, 64, 0, 0.125) == fa.FA_OK


def test_bwd_rejects_bad_arguments(lib):
    p, n = ALIGNED, NULL
    assert lib.fa_bwd(p, p, p, p, p, p, p, p, n, 1, 1, 8, 64, 0, 0.125) == fa.FA_ERR_INVALID
    assert lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 1, 8, 80, 0, 0.125) == fa.FA_ERR_UNSUPPORTED
    # d = 256 is a forward-only head size
    assert lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 1, 8, 256, 0, 0.125) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_stream(p, p, p, p, p, p, p, p, p, 1, 1, 8, 256, 0, 0.125, p, 1 << 20,
                             n) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, 8, 256, 0, 0.125, n) == fa.FA_ERR_UNSUPPORTED
    # the stream form wants a workspace of the advertised size, 256-byte aligned
    ws_need = lib.fa_bwd_workspace_bytes(1, 1, 8, 64)
    assert lib.fa_bwd_stream(p, p, p, p, p, p, p, p, p, 1, 1, 8, 64, 0, 0.125, n, ws_need,
                             n) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_stream(p, p, p, p, p, p, p, p, p, 1, 1, 8, 64, 0, 0.125, p, ws_need - 4,
                             n) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_stream(p, p, p, p, p, p, p, p, p, 1, 1, 8, 64, 0, 0.125,
                             ctypes.c_void_p(0x100010), ws_need, n) == fa.FA_ERR_WORKSPACE


def test_dropout_entry_points_check_arguments_on_the_host(lib):
    p, n = ALIGNED, NULL
    for bad in (-0.1, 1.0, 1.5, float("nan")):
        assert lib.fa_fwd_dropout(p, p, p, p, p, 1, 1, 8, 64, 0, 0.125, bad, 1, 0, n) == fa.FA_ERR_INVALID
        assert lib.fa_bwd_dropout(p, p, p, p, p, p, p, p, p, 1, 1, 8, 64, 0, 0.125, bad, 1, 0, p, 1 << 20,
                                  n) == fa.FA_ERR_INVALID
    # empty problems are no-ops; bad sizes and pointers as without dropout
    assert lib.fa_fwd_dropout(n, n, n, n, n, 0, 4, 128, 64, 0, 0.125, 0.1, 1, 0, n) == fa.FA_OK
    assert lib.fa_fwd_dropout(p, p, p, p, p, 1, 1, 8, 96, 0, 0.125, 0.1, 1, 0, n) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_dropout(n, p, p, p, p, 1, 1, 8, 64, 0, 0.125, 0.1, 1, 0, n) == fa.FA_ERR_INVALID
    ws_need = lib.fa_bwd_workspace_bytes(1, 1, 8, 64)
    assert lib.fa_bwd_dropout(p, p, p, p, p, p, p, p, p, 1, 1, 8, 64, 0, 0.125, 0.1, 1, 0, p, ws_need - 4,
                              n) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_dropout(n, n, n, n, n, n, n, n, n, 1, 0, 64, 64, 0, 0.125, 0.1, 1, 0, n, 0,
                              n) == fa.FA_OK


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_fwd(x, x, x)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_fwd_dropout(x, x, x, 0.1, seed=1)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_bwd_dropout(x, x, x, x, lse, x, 0.1, seed=1)


def test_transfer_ledger_matches_page():
    import json
    g = json.load(open(os.path.join(GOLDEN, "transfer_ledger.json")))
    led = fa.transfer_ledger(g["N"], g["d"], g["d_v"], g["query_block"])
    assert led["reads"] == g["reads"]
    assert led["writes"] == g["writes"]
    assert led["tiled_total"] == g["tiled_total"]
    assert led["dense_total"] == g["dense_total"]


def test_flop_and_byte_counts():
    # 4 B H N^2 d forward, halved when causal; backward 2.5x
    assert fa.flops_fwd(1, 1, 256, 64, False) == 4 * 256 * 256 * 64
    assert fa.flops_fwd(8, 12, 2048, 64, True) == 0.5 * 4 * 8 * 12 * 2048 ** 2 * 64
    assert fa.flops_bwd(8, 12, 2048, 64, True) == 2.5 * fa.flops_fwd(8, 12, 2048, 64, True)
    assert fa.bytes_fwd(1, 16, 8192, 128) == 8 * 16 * 8192 * 128 + 4 * 16 * 8192
    assert fa.bytes_bwd(8, 12, 2048, 64) == 16 * 96 * 2048 * 64 + 8 * 96 * 2048


def test_extended_forward_rejects_bad_arguments_on_the_host(lib):
    p = ctypes.c_void_p(4096)  # never dereferenced: every call below fails its checks first
    z = ctypes.c_void_p(0)
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 64, 64, 0, 4, 0.1, z) == fa.FA_ERR_INVALID  # window, not causal
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 64, 64, 1, -2, 0.1, z) == fa.FA_ERR_INVALID
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 9, 8, 64, 64, 1, 0, 0.1, z) == fa.FA_ERR_INVALID  # Nq > Nk, causal
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 0, 64, 64, 0, 0, 0.1, z) == fa.FA_ERR_INVALID  # no keys
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 96, 64, 0, 0, 0.1, z) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 64, 32, 0, 0, 0.1, z) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_ex(z, z, z, z, z, 0, 1, 8, 8, 64, 64, 0, 0, 0.1, z) == fa.FA_OK  # empty
    assert lib.fa_decode_splitkv(z, z, z, z, z, 1, 1, 0, 8, 64, 64, 0, 0, 0.1, 2, z, 0, z) == fa.FA_OK


def test_decode_split_count_and_workspace(lib):
    # explicit counts: clamped to the key tiles and made free of empty trailing splits
    assert lib.fa_decode_num_splits(1, 1, 1, 300, 64) == 3      # 3 key tiles
    assert lib.fa_decode_num_splits(1, 1, 1, 4096, 5) == 5      # 32 tiles, 7 per split
    assert lib.fa_decode_num_splits(1, 1, 1, 4096, 6) == 6      # 6 per split
    assert lib.fa_decode_num_splits(1, 1, 1, 4096, 11) == 11    # 3 per split -> 11
    assert lib.fa_decode_num_splits(1, 1, 1, 4096, 12) == 11    # 3 per split -> 11
    auto = lib.fa_decode_num_splits(2, 4, 1, 32768, 0)
    assert 1 <= auto <= 128
    s = lib.fa_decode_num_splits(2, 3, 5, 1000, 4)
    assert lib.fa_decode_workspace_bytes(2, 3, 5, 1000, 128, 4) == s * 2 * 3 * 5 * (128 + 1) * 4
    assert lib.fa_decode_workspace_bytes(0, 3, 5, 1000, 128, 4) == 0
