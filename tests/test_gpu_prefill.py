"""GPU parity of w4a16_gemm_bf16 through the C ABI against the exact float64 product of the oracle:
relative L2 <= 1e-2 (bf16 activations and output). Large M runs the tensor-core contraction, up
to 16 rows the weight-streaming kernels in their bf16 form. Small cases cover one tile, ragged M
and N and several K blocks; the full prefill workload (M=4096, K=7168, N=18432) and the full
M=16 decode shape are checked on sampled rows and columns."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import BF16_TOL, assert_close_rows, dev, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    return lib()


def _bf16_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def _as_f64(t):
    torch.cuda.synchronize()
    return t.float().cpu().numpy().astype(np.float64)


# Tiles of 256 weight columns (128 per CTA of a pair) x up to 256 rows: (130, 264, 128) has a
# second column tile the odd CTA sees only as zero fill, (48, 776, 320) a 48-row tile split 24/24
# between the CTAs, and (2440, 2056, 128) 10 x 9 = 90 tiles, more than one per pair on any GPU,
# with ragged last rows and columns. (40, 8, 64) is a single 8-column tile; (4097, 264, 128) has
# 17 row blocks of 256 whose last holds one row.
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (1, 256, 64), (130, 264, 128),
                                   (300, 520, 192), (512, 1024, 1024), (48, 776, 320),
                                   (17, 264, 64), (2440, 2056, 128), (40, 8, 64),
                                   (4097, 264, 128)])
def test_prefill_small(w4, M, N, K):
    bits = synth.bf16_activations(M, K, seed=M + N)
    W = synth.weights(K, N, seed=K + N)
    qo, so = oracle.quantize_w4a16(W)
    y = w4.w4a16_gemm_bf16(_bf16_dev(bits), dev(qo), dev(so))
    ref = oracle.gemm_bf16(bits, qo, so)
    assert_close_rows(_as_f64(y), ref, BF16_TOL, f"prefill {M}x{N}x{K}")
    assert w4.w4a16_device_error() == 0


def test_prefill_deterministic(w4):
    M, N, K = 384, 768, 512
    bits = synth.bf16_activations(M, K, seed=3)
    qo, so = oracle.quantize_w4a16(synth.weights(K, N, seed=3))
    xd, qd, sd = _bf16_dev(bits), dev(qo), dev(so)
    a = _as_f64(w4.w4a16_gemm_bf16(xd, qd, sd))
    b = _as_f64(w4.w4a16_gemm_bf16(xd, qd, sd))
    np.testing.assert_array_equal(a, b)


def test_prefill_full_size_sampled(w4):
    c = synth.PREFILL
    M, K, N = c["M"], c["K"], c["N"]
    Wd = synth.cuda_weights(K, N, seed=3000)
    qw, sc = w4.w4a16_quantize(Wd)
    xb = synth.cuda_bf16_activations(M, K, seed=3)
    y = w4.w4a16_gemm_bf16(xb, qw, sc)
    torch.cuda.synchronize()
    assert w4.w4a16_device_error() == 0
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([rng.choice(M, 30, replace=False), [0, M - 1]]))
    cols = np.sort(np.concatenate([rng.choice(N, 126, replace=False), [0, N - 1]]))
    cidx = torch.from_numpy(cols).cuda()
    Wc = host(Wd.index_select(1, cidx))
    qo, so = oracle.quantize_w4a16(Wc)
    xbits = xb.index_select(0, torch.from_numpy(rows).cuda()).view(torch.int16).cpu().numpy()
    ref = oracle.gemm_bf16(xbits.view(np.uint16), qo, so)
    got = _as_f64(y)[rows][:, cols]
    assert_close_rows(got, ref, BF16_TOL, "prefill full size")


# ---- bf16 activations at small M (weight-streaming kernels, bf16 form)

@pytest.mark.parametrize("M,N,K", [(1, 264, 128), (3, 1000, 1024), (8, 520, 2048), (9, 256, 192),
                                   (16, 1032, 4096)])
def test_bf16_small_m(w4, M, N, K):
    bits = synth.bf16_activations(M, K, seed=M + 7)
    W = synth.weights(K, N, seed=K + M, outliers=True)
    qo, so = oracle.quantize_w4a16(W)
    y = w4.w4a16_gemm_bf16(_bf16_dev(bits), dev(qo), dev(so))
    ref = oracle.gemm_bf16(bits, qo, so)
    assert_close_rows(_as_f64(y), ref, BF16_TOL, f"bf16 small M={M} N={N} K={K}")
    assert w4.w4a16_device_error() == 0


def test_bf16_small_m_full_size_sampled(w4):
    M, K, N = 16, synth.PREFILL["K"], synth.PREFILL["N"]
    Wd = synth.cuda_weights(K, N, seed=3100)
    qw, sc = w4.w4a16_quantize(Wd)
    xb = synth.cuda_bf16_activations(M, K, seed=31)
    y = w4.w4a16_gemm_bf16(xb, qw, sc)
    torch.cuda.synchronize()
    assert w4.w4a16_device_error() == 0
    rng = np.random.default_rng(1)
    cols = np.sort(np.concatenate([rng.choice(N, 126, replace=False), [0, N - 1]]))
    Wc = host(Wd.index_select(1, torch.from_numpy(cols).cuda()))
    qo, so = oracle.quantize_w4a16(Wc)
    ref = oracle.gemm_bf16(xb.view(torch.int16).cpu().numpy().view(np.uint16), qo, so)
    assert_close_rows(_as_f64(y)[:, cols], ref, BF16_TOL, "bf16 small M full size")


def test_bf16_small_m_deterministic(w4):
    M, N, K = 12, 768, 2048
    bits = synth.bf16_activations(M, K, seed=5)
    qo, so = oracle.quantize_w4a16(synth.weights(K, N, seed=5))
    xd, qd, sd = _bf16_dev(bits), dev(qo), dev(so)
    np.testing.assert_array_equal(_as_f64(w4.w4a16_gemm_bf16(xd, qd, sd)),
                                  _as_f64(w4.w4a16_gemm_bf16(xd, qd, sd)))


def test_prefill_repeatable_under_load(w4):
    """The CTA-pair pipeline hands every stage across SMs through barriers (TMA completion, the
    odd CTA's release relayed to the even CTA, the MMA commit multicast to both): a missed
    ordering would show up as a changed bit somewhere in repeated full-size runs."""
    c = synth.PREFILL
    M, K, N = c["M"], c["K"], c["N"]
    Wd = synth.cuda_weights(K, N, seed=3200)
    qw, sc = w4.w4a16_quantize(Wd)
    del Wd
    xb = synth.cuda_bf16_activations(M, K, seed=32)
    first = w4.w4a16_gemm_bf16(xb, qw, sc)
    y = torch.empty_like(first)
    for _ in range(40):
        w4.w4a16_gemm_bf16(xb, qw, sc, y)
        assert torch.equal(y.view(torch.int16), first.view(torch.int16))
    xs = synth.cuda_bf16_activations(48, K, seed=33)
    first = w4.w4a16_gemm_bf16(xs, qw, sc)
    ys = torch.empty_like(first)
    for _ in range(200):
        w4.w4a16_gemm_bf16(xs, qw, sc, ys)
        assert torch.equal(ys.view(torch.int16), first.view(torch.int16))
    assert w4.w4a16_device_error() == 0
