"""Host-side checks of the C ABI: the library loads without a GPU, exports every function that
include/w4a16.h declares, and rejects bad arguments with a status code before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    from int4_w4a16_group_gb300.build import build
    build()
    import int4_w4a16_group_gb300 as w4
    return w4.C


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("w4a16_gemm", "w4a16_gemm_swiglu", "w4a16_gemm_bf16", "w4a16_moe_gemm",
                 "w4a16_moe_workspace_size", "w4a16_quantize", "w4a16_dequantize",
                 "w4a16_load_qw_sc", "w4a16_linear", "w4a16_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.w4a16_abi_version() == 1
    for code in range(9):
        s = lib.w4a16_status_string(code).decode()
        assert s.startswith("W4A16_")
    assert "unknown" in lib.w4a16_status_string(99).decode()


A = 0x10000   # fake, 16-byte aligned addresses: validation must fail before touching them
B = 0x20000
Y = 0x30000


@pytest.mark.parametrize("args,want", [
    # (x, qw, sc, y, M, N, K, group)
    ((A, B, B, Y, 1, 64, 256, 64), 3),       # group != 32 -> UNSUPPORTED
    ((A, B, B, Y, 1, 64, 250, 32), 1),       # K % 32 != 0 -> ARG
    ((A, B, B, Y, 1, 64, 0, 32), 1),         # K == 0 -> ARG
    ((A, B, B, Y, 1, 66, 256, 32), 1),       # N % 4 != 0 -> ARG
    ((A, B, B, Y, -1, 64, 256, 32), 1),      # M < 0 -> ARG
    ((A + 4, B, B, Y, 1, 64, 256, 32), 2),   # misaligned x -> ALIGN
    ((A, B + 8, B, Y, 1, 64, 256, 32), 2),   # misaligned qw -> ALIGN
    ((A, B, B + 4, Y, 1, 64, 256, 32), 2),   # misaligned sc -> ALIGN
    ((A, B, B, Y + 12, 1, 64, 256, 32), 2),  # misaligned y -> ALIGN
    ((0, B, B, Y, 1, 64, 256, 32), 1),       # null x -> ARG
    ((A, 0, B, Y, 1, 64, 256, 32), 1),       # null qw -> ARG
    ((A, B, B, Y, 0, 64, 256, 32), 0),       # M == 0: empty call, no launch
    ((A, B, B, Y, 3, 0, 256, 32), 0),        # N == 0: empty call, no launch
])
def test_gemm_argument_checks(lib, args, want):
    assert lib.w4a16_gemm(*args, None) == want


def test_swiglu_needs_even_halves(lib):
    assert lib.w4a16_gemm_swiglu(A, B, B, Y, 1, 12, 256, 32, None) == 1   # N2 % 8 != 0


def test_bf16_argument_checks(lib):
    assert lib.w4a16_gemm_bf16(A, B, B, Y, 4, 64, 96, 32, None) == 1      # K % 64 != 0
    assert lib.w4a16_gemm_bf16(A, B, B, Y, 4, 60, 128, 32, None) == 1     # N % 8 != 0
    assert lib.w4a16_gemm_bf16(A, B, B, Y, 0, 64, 128, 32, None) == 0     # empty


def test_quantize_argument_checks(lib):
    assert lib.w4a16_quantize(A, 256, 64, 16, B, B, None) == 3
    assert lib.w4a16_quantize(A, 100, 64, 32, B, B, None) == 1
    assert lib.w4a16_quantize(A + 4, 256, 64, 32, B, B, None) == 2
    assert lib.w4a16_dequantize(B, B, 256, 62, 32, A, None) == 1


def test_moe_argument_checks(lib):
    T, topk, E, K, I = 64, 8, 384, 7168, 2048
    need = lib.w4a16_moe_workspace_size(T, topk, E, K, I)
    # the workspace holds at least h [T*topk, I] and the per-pair outputs [T*topk, K]
    assert need >= T * topk * (I + K) * 4
    assert lib.w4a16_moe_workspace_size(2 * T, topk, E, K, I) > need
    args = [A, B, B, T, topk, E, B, B, B, B, Y, K, I, 32]
    assert lib.w4a16_moe_gemm(*args, Y, need - 1, None) == 4        # workspace too small
    assert lib.w4a16_moe_gemm(*args, 0, need, None) == 4            # no workspace
    bad = list(args)
    bad[-1] = 16
    assert lib.w4a16_moe_gemm(*bad, Y, need, None) == 3             # group
    bad = list(args)
    bad[11] = 7000
    assert lib.w4a16_moe_gemm(*bad, Y, need, None) == 1             # K % 32
    bad = list(args)
    bad[1] = B + 4
    assert lib.w4a16_moe_gemm(*bad, Y, need, None) == 2             # misaligned ids
    zero = list(args)
    zero[3] = 0
    assert lib.w4a16_moe_gemm(*zero, 0, 0, None) == 0               # T == 0: empty
    assert lib.w4a16_topk_softmax(A, B, 4, 33, None) == 1
    assert lib.w4a16_topk_softmax(A, B, 0, 8, None) == 0


def test_registry_dispatch_has_no_fallback(lib):
    reg = lib.w4a16_registry_create()
    assert reg
    try:
        K, N = ctypes.c_int(0), ctypes.c_int(0)
        assert lib.w4a16_registry_find(reg, b"mlp.down", ctypes.byref(K), ctypes.byref(N)) == 6
        assert lib.w4a16_linear(reg, b"mlp.down", A, Y, 1, None) == 6       # NOT_FOUND
        assert lib.w4a16_registry_add(reg, b"mlp.down", B, B, 18432, 7168, 32) == 0
        assert lib.w4a16_registry_find(reg, b"mlp.down", ctypes.byref(K), ctypes.byref(N)) == 0
        assert (K.value, N.value) == (18432, 7168)
        assert lib.w4a16_linear(reg, b"mlp.gate_up", A, Y, 1, None) == 6    # other names still miss
        assert lib.w4a16_linear(reg, b"mlp.down", A, Y, 0, None) == 0       # empty call
        assert lib.w4a16_linear(reg, b"mlp.down", A + 4, Y, 1, None) == 2   # checks still apply
        assert lib.w4a16_registry_add(reg, b"bad", B + 4, B, 64, 64, 32) == 2
        assert lib.w4a16_registry_add(reg, b"bad", B, B, 64, 64, 128) == 3
        assert lib.w4a16_registry_add(reg, b"", B, B, 64, 64, 32) == 1
    finally:
        lib.w4a16_registry_destroy(reg)


def test_loader_rejects_missing_and_wrong_size(lib, tmp_path):
    K, N = 64, 8
    qp, sp = tmp_path / "w.qw", tmp_path / "w.sc"
    assert lib.w4a16_load_qw_sc(str(qp).encode(), str(sp).encode(), K, N, 32, B, B) == 7
    np.zeros((K // 8, N), dtype=np.int32).tofile(qp)
    np.zeros((K // 32, N - 1), dtype=np.float32).tofile(sp)          # one column short
    assert lib.w4a16_load_qw_sc(str(qp).encode(), str(sp).encode(), K, N, 32, B, B) == 7
    np.zeros((K // 8, N), dtype=np.int32)[:-1].tofile(qp)            # truncated .qw
    assert lib.w4a16_load_qw_sc(str(qp).encode(), str(sp).encode(), K, N, 32, B, B) == 7


@pytest.mark.parametrize("limit_us", [0, -5, 100001])
def test_selftest_wait_limit_checked_before_any_cuda_call(lib, limit_us):
    assert lib.w4a16_selftest_wait(0, limit_us, None) == 1  # W4A16_ERR_ARG


def test_noalloc_scratch_bound_is_909_pairs(lib):
    # The fixed scratch of w4a16_moe_gemm_noalloc holds the workspace of 909 token-expert pairs
    # at K = 7168, I = 2048 for any expert count up to 4096, and not that of 910.
    limit = 32 << 20
    for E in (1, 64, 384, 4096):
        assert lib.w4a16_moe_workspace_size(909, 1, E, 7168, 2048) <= limit
        assert lib.w4a16_moe_workspace_size(910, 1, E, 7168, 2048) > limit
        assert lib.w4a16_moe_workspace_size(64, 8, E, 7168, 2048) <= limit


@pytest.mark.parametrize("T,topk,E,K,I,group,want", [
    (4096, 8, 384, 7168, 2048, 64, 3),   # a bad group wins over a too-large size: UNSUPPORTED
    (4096, 65, 384, 7168, 2048, 32, 1),  # topk > 64 -> ARG before the size check
    (4096, 8, 5000, 7168, 2048, 32, 1),  # E > 4096 -> ARG
    (4096, 8, 384, 7000, 2048, 32, 1),   # K % 32 != 0 -> ARG
    (0, 8, 384, 7168, 2048, 32, 0),      # T == 0: nothing to do
    (4096, 8, 384, 7168, 2048, 32, 4),   # valid arguments, scratch too small -> WORKSPACE
])
def test_noalloc_checks_arguments_like_the_workspace_entry(lib, T, topk, E, K, I, group, want):
    st = lib.w4a16_moe_gemm_noalloc(A, A, A, T, topk, E, B, B, B, B, Y, K, I, group, None)
    assert st == want
    if want != 4:  # the workspace entry answers the same (with any workspace pointer)
        st2 = lib.w4a16_moe_gemm(A, A, A, T, topk, E, B, B, B, B, Y, K, I, group, Y, 1 << 40, None)
        assert st2 == want
