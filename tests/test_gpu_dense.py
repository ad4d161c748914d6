"""GPU parity of the dense path through the C ABI: quantize/pack (bit-exact), dequantize
(bit-exact), w4a16_gemm and the fused gate/up SwiGLU GEMM (rel-L2 <= 1e-5), linear() dispatch
and the raw-file loader. Small cases span several tiles and a ragged tail; the full-size
workloads are checked on sampled output columns."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import BF16_TOL, FP32_TOL, assert_close_rows, dev, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    return lib()


# ----------------------------------------------------------------------------- format

@pytest.mark.parametrize("K,N,outl", [(32, 4, False), (256, 512, False), (512, 1000, True),
                                      (4096, 388, True)])
def test_quantize_bit_exact(w4, K, N, outl):
    W = synth.weights(K, N, seed=K + N, outliers=outl)
    W[:32, :4] = 0.0                       # an all-zero group
    if K > 32:
        W[32:64, 1] *= np.float32(1e-37)   # a group whose scale and quotients are subnormal
    qo, so = oracle.quantize_w4a16(W)
    qw, sc = w4.w4a16_quantize(dev(W))
    np.testing.assert_array_equal(host(qw), qo)
    np.testing.assert_array_equal(host(sc), so)


def test_dequantize_bit_exact_every_nibble(w4):
    rng = np.random.default_rng(5)
    K, N = 256, 132
    q = rng.integers(-8, 8, size=(K, N))
    q[:8, 0] = -8                          # nibble 0 (never produced by the quantizer)
    qw = oracle.pack_int4(q)
    sc = (rng.random((K // 32, N), dtype=np.float32) * 0.1).astype(np.float32)
    sc[0, 3] = 0.0
    Wg = host(w4.w4a16_dequantize(dev(qw), dev(sc)))
    want = oracle.dequantize(qw, sc).astype(np.float32)   # q*s is exact in f64; one rounding
    np.testing.assert_array_equal(Wg, want)


# ----------------------------------------------------------------------------- GEMM

@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 15, 16, 17, 33, 64, 100, 300])
@pytest.mark.parametrize("K,N", [(512, 1000), (2048, 260)])
def test_gemm_small(w4, M, K, N):
    W = synth.weights(K, N, seed=M + K, outliers=True)
    x = synth.activations(M, K, seed=M)
    qo, so = oracle.quantize_w4a16(W)
    y = w4.w4a16_gemm(dev(x), dev(qo), dev(so))
    assert_close_rows(host(y), oracle.gemm(x, qo, so), FP32_TOL, f"gemm M={M} K={K} N={N}")


def test_gemm_tiny_workload(w4):
    c = synth.TINY
    W = synth.weights(c["K"], c["N"], seed=0)
    x = synth.activations(c["M"], c["K"], seed=0)
    qo, so = oracle.quantize_w4a16(W)
    qw, sc = w4.w4a16_quantize(dev(W))
    y = w4.w4a16_gemm(dev(x), qw, sc)
    assert_close_rows(host(y), oracle.gemm(x, qo, so), FP32_TOL, "tiny")


def test_gemm_handmade_extremes(w4):
    """Nibble 0 (-8) and 15 (+7) everywhere, a zero-scale group, large and tiny scales."""
    K, N, M = 128, 64, 3
    q = np.full((K, N), -8)
    q[:, 1::2] = 7
    qw = oracle.pack_int4(q)
    sc = np.full((K // 32, N), 0.5, dtype=np.float32)
    sc[1, :] = 0.0
    sc[2, :8] = 1e20
    sc[3, 8:16] = 1e-20
    x = synth.activations(M, K, seed=3)
    y = w4.w4a16_gemm(dev(x), dev(qw), dev(sc))
    assert_close_rows(host(y), oracle.gemm(x, qw, sc), FP32_TOL, "extremes")


@pytest.mark.parametrize("M", [3, 8, 16, 20])
def test_gemm_activation_range_along_k(w4, M):
    """Activations whose magnitude jumps by 1e4 up or down along K (and a row that is zero in
    its first half): the kernels' per-row exponents must follow (raised when larger values
    arrive, kept when smaller ones do) without losing the float32 accuracy."""
    K, N = 2048, 520
    W = synth.weights(K, N, seed=31 + M, outliers=True)
    x = synth.activations(M, K, seed=32 + M)
    x[: M // 2, : K // 2] *= 1e-4
    x[M // 2:, K // 2:] *= 1e-4
    x[-1, : K // 2] = 0.0
    qo, so = oracle.quantize_w4a16(W)
    for swiglu in (False, True):
        if swiglu:
            y = w4.w4a16_gemm_swiglu(dev(x), dev(qo), dev(so))
            ref = oracle.swiglu_gemm(x, qo, so)
        else:
            y = w4.w4a16_gemm(dev(x), dev(qo), dev(so))
            ref = oracle.gemm(x, qo, so)
        assert_close_rows(host(y), ref, FP32_TOL, f"range along K, M={M}, swiglu={swiglu}")


def _top_of_binade_rows(M, K, seed):
    """Rows of magnitude <= 1 (one value exactly 1) up to a switch point, then values <= 2 in
    which every block of 64 inputs holds +-(4 - 2^-12): one binade above the start, in its top
    2^-12. The switch points are staggered over the rows, so for any split over K some row
    switches behind an activation-chunk boundary of its rank."""
    x = synth.normal((M, K), 0.3, seed=seed, stream=2)
    np.clip(x, -1.0, 1.0, out=x)
    top = np.float32(4.0 - 2.0 ** -12)
    for m in range(M):
        s = 64 * (1 + 3 * m) % (K - 256) + 128
        x[m, 0] = 1.0
        x[m, s:] *= 2.0
        x[m, s::64] = np.where(np.arange(len(x[m, s::64])) % 2 == 0, top, -top)
    return x


@pytest.mark.parametrize("M", [4, 16])
def test_gemm_activation_top_of_binade(w4, M):
    """A row's exponent may be kept while a later chunk's values are one binade larger; values in
    the top 2^-12 of that binade must still fit the fp16 activation terms (no inf, float32
    accuracy). Wide shapes keep the split over K small, so every rank sees several chunks."""
    K, I = 2048, 18432
    qw, sc = synth.packed_codes(K, 2 * I, seed=40 + M), synth.group_scales(K, 2 * I, seed=41 + M)
    x = _top_of_binade_rows(M, K, seed=42 + M)
    y = host(w4.w4a16_gemm_swiglu(dev(x), dev(qw), dev(sc)))
    assert np.isfinite(y).all(), "non-finite gate/up output"
    cols = np.sort(np.random.default_rng(43 + M).choice(I, 384, replace=False))
    both = np.concatenate([cols, I + cols])
    ref = oracle.swiglu_gemm(x, qw[:, both], sc[:, both])
    assert_close_rows(y[:, cols], ref, FP32_TOL, f"gate/up top of binade, M={M}")
    K, N = 4096, 18432
    qw, sc = synth.packed_codes(K, N, seed=44 + M), synth.group_scales(K, N, seed=45 + M)
    x = _top_of_binade_rows(M, K, seed=46 + M)
    y = host(w4.w4a16_gemm(dev(x), dev(qw), dev(sc)))
    assert np.isfinite(y).all(), "non-finite plain output"
    ref = oracle.gemm(x, qw[:, cols], sc[:, cols])
    assert_close_rows(y[:, cols], ref, FP32_TOL, f"plain top of binade, M={M}")


def test_gemm_activation_magnitude_limits(w4):
    """Rows near the ends of the float32 range: ~2^110, ~2^-95, and one that falls from 2^100 to
    2^-80 along K (the exponent stays at the large part; the small part's contribution is far
    below float32 resolution of the result)."""
    K, N = 2048, 520
    W = synth.weights(K, N, seed=51, outliers=True)
    x = synth.activations(4, K, seed=52)
    x[0] *= np.float32(2.0 ** 110)
    x[1] *= np.float32(2.0 ** -95)
    x[2, : K // 2] *= np.float32(2.0 ** 100)
    x[2, K // 2:] *= np.float32(2.0 ** -80)
    qo, so = oracle.quantize_w4a16(W)
    y = host(w4.w4a16_gemm(dev(x), dev(qo), dev(so)))
    assert np.isfinite(y).all()
    assert_close_rows(y, oracle.gemm(x, qo, so), FP32_TOL, "magnitude limits")


def test_launches_replayed_from_a_cuda_graph(w4):
    """The streaming GEMMs captured in one CUDA graph (as the bench step and a serving loop issue
    them: float32 gate/up at M = 1, 4, 16 and a bf16 call back to back on one stream) and
    replayed twice give the oracle's results."""
    K, I = 2048, 1040
    W = synth.weights(K, 2 * I, seed=61)
    qo, so = oracle.quantize_w4a16(W)
    q, s = dev(qo), dev(so)
    xs = {M: synth.activations(M, K, seed=62 + M) for M in (1, 4, 16)}
    xd = {M: dev(x) for M, x in xs.items()}
    ys = {M: torch.zeros((M, I), dtype=torch.float32, device="cuda") for M in xs}
    bits = synth.bf16_activations(8, K, seed=66)
    xb = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    yb = torch.zeros((8, 2 * I), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for M in (16, 4, 1):
            w4.w4a16_gemm_swiglu(xd[M], q, s, ys[M], stream=cs)
        w4.w4a16_gemm_bf16(xb, q, s, yb, stream=cs)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for M, x in xs.items():
        assert_close_rows(host(ys[M]), oracle.swiglu_gemm(x, qo, so), FP32_TOL, f"graph M={M}")
    yb64 = yb.float().cpu().numpy().astype(np.float64)
    assert_close_rows(yb64, oracle.gemm_bf16(bits, qo, so), BF16_TOL, "graph bf16")
    assert w4.w4a16_device_error() == 0


@pytest.mark.parametrize("M", [1, 8, 16])
def test_gemm_split_over_k_for_every_tile_count(w4, M):
    """1 to 20 wide column tiles at K = 8192: the launch planner splits K over clusters of
    whatever size fills the GPU for each count (1 to 16 CTAs), so the split-K sends, receive
    slots and rank-ordered sums run for most cluster sizes. Sampled columns (first, last and a
    seeded spread) against the oracle."""
    K = 8192
    x = synth.activations(M, K, seed=70 + M)
    for T in range(1, 21):
        N = 512 * T
        qw = synth.packed_codes(K, N, seed=71 + T)
        sc = synth.group_scales(K, N, seed=72 + T)
        y = host(w4.w4a16_gemm(dev(x), dev(qw), dev(sc)))
        rng = np.random.default_rng(73 + T)
        cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 62, replace=False)]))
        assert_close_rows(y[:, cols], oracle.gemm(x, qw[:, cols], sc[:, cols]), FP32_TOL,
                          f"split over K, M={M}, {T} tiles")
    assert w4.w4a16_device_error() == 0


@pytest.mark.parametrize("M", [1, 8, 16])
def test_bf16_split_over_k_for_every_tile_count(w4, M):
    """The bf16 one-term forms over 1 to 20 wide column tiles at K = 8192 (cluster sizes 1 to 16,
    receive slots of their own or in the code ring): sampled columns against the exact product."""
    K = 8192
    bits = synth.bf16_activations(M, K, seed=90 + M)
    xb = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    for T in range(1, 21):
        N = 512 * T
        qw = synth.packed_codes(K, N, seed=91 + T)
        sc = synth.group_scales(K, N, seed=92 + T)
        y = w4.w4a16_gemm_bf16(xb, dev(qw), dev(sc)).float().cpu().numpy().astype(np.float64)
        rng = np.random.default_rng(93 + T)
        cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 62, replace=False)]))
        assert_close_rows(y[:, cols], oracle.gemm_bf16(bits, qw[:, cols], sc[:, cols]), BF16_TOL,
                          f"bf16 split over K, M={M}, {T} tiles")
    assert w4.w4a16_device_error() == 0


def test_gemm_on_two_streams_at_once(w4):
    """Two streams each issue gate/up GEMMs while the other runs: both match the oracle (the
    per-device launch data is shared; nothing else is)."""
    K, I = 2048, 1040
    W = synth.weights(K, 2 * I, seed=81)
    qo, so = oracle.quantize_w4a16(W)
    q, s = dev(qo), dev(so)
    xs = [synth.activations(M, K, seed=82 + M) for M in (4, 16)]
    xd = [dev(x) for x in xs]
    ys = [torch.empty((x.shape[0], I), dtype=torch.float32, device="cuda") for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(8):
        for j in range(2):
            w4.w4a16_gemm_swiglu(xd[j], q, s, ys[j], stream=streams[j])
    torch.cuda.synchronize()
    for j in range(2):
        assert_close_rows(host(ys[j]), oracle.swiglu_gemm(xs[j], qo, so), FP32_TOL,
                          f"stream {j}")
    assert w4.w4a16_device_error() == 0


def test_gemm_zero_weights_and_empty(w4):
    K, N = 256, 128
    qw, sc = oracle.quantize_w4a16(np.zeros((K, N), dtype=np.float32))
    x = synth.activations(4, K, seed=1)
    y = host(w4.w4a16_gemm(dev(x), dev(qw), dev(sc)))
    assert (y == 0).all()
    e = torch.empty((0, K), dtype=torch.float32, device="cuda")
    assert w4.w4a16_gemm(e, dev(qw), dev(sc)).shape == (0, N)


def test_gemm_is_deterministic(w4):
    W = synth.weights(4096, 1024, seed=8)
    x = synth.activations(4, 4096, seed=8)
    qw, sc = w4.w4a16_quantize(dev(W))
    xd = dev(x)
    a = host(w4.w4a16_gemm(xd, qw, sc))
    b = host(w4.w4a16_gemm(xd, qw, sc))
    np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("M", [1, 2, 4, 7, 16, 20, 64, 300])
@pytest.mark.parametrize("K,I", [(1024, 520), (256, 64)])
def test_swiglu_small(w4, M, K, I):
    W = synth.weights(K, 2 * I, seed=M + I)
    x = synth.activations(M, K, seed=M + 1)
    qo, so = oracle.quantize_w4a16(W)
    y = w4.w4a16_gemm_swiglu(dev(x), dev(qo), dev(so))
    assert_close_rows(host(y), oracle.swiglu_gemm(x, qo, so), FP32_TOL, f"swiglu M={M}")


# ----------------------------------------------------------------------------- full size, sampled

def _sampled(w4, K, N, M, cols, outliers, x_std, seed, swiglu):
    """Full-size weights drawn on the device, quantized by the library, GEMM at full size;
    the oracle quantizes only the sampled weight columns (quantization is per column) and
    computes those outputs."""
    Wd = synth.cuda_weights(K, N, seed=seed, outliers=outliers)
    qw, sc = w4.w4a16_quantize(Wd)
    x = synth.activations(M, K, seed=seed + 1, std=x_std)
    if swiglu:
        y = w4.w4a16_gemm_swiglu(dev(x), qw, sc)
        I = N // 2
        wcols = np.concatenate([cols, cols + I])
    else:
        y = w4.w4a16_gemm(dev(x), qw, sc)
        wcols = cols
    idx = torch.from_numpy(wcols).cuda()
    Wc = host(Wd.index_select(1, idx))
    qo, so = oracle.quantize_w4a16(Wc)
    np.testing.assert_array_equal(host(qw.index_select(1, idx)), qo)
    np.testing.assert_array_equal(host(sc.index_select(1, idx)), so)
    ref = oracle.swiglu_gemm(x, qo, so) if swiglu else oracle.gemm(x, qo, so)
    got = host(y)[:, cols]
    del Wd
    return got, ref


@pytest.mark.parametrize("M", [1, 4, 16])
def test_full_size_swiglu_gate_up(w4, M):
    K, I = synth.SWIGLU["K"], synth.SWIGLU["I"]
    rng = np.random.default_rng(M)
    cols = np.sort(np.concatenate([rng.choice(I, 254, replace=False), [0, I - 1]]))
    got, ref = _sampled(w4, K, 2 * I, M, cols, False, 1.0, 100 + M, True)
    assert_close_rows(got, ref, FP32_TOL, f"gate/up M={M}")


@pytest.mark.parametrize("M", [1, 4, 16])
def test_full_size_down(w4, M):
    K, N = synth.DOWN["K"], synth.DOWN["N"]
    rng = np.random.default_rng(M + 7)
    cols = np.sort(np.concatenate([rng.choice(N, 254, replace=False), [0, N - 1]]))
    got, ref = _sampled(w4, K, N, M, cols, True, synth.DOWN_X_STD, 200 + M, False)
    assert_close_rows(got, ref, FP32_TOL, f"down M={M}")


# ----------------------------------------------------------------------------- dispatch + loader

def test_linear_dispatch_and_loader(w4, tmp_path):
    K, N, I = 512, 256, 128
    W = synth.weights(K, N, seed=21)
    Wgu = synth.weights(K, 2 * I, seed=22)
    qo, so = oracle.quantize_w4a16(W)
    qgo, sgo = oracle.quantize_w4a16(Wgu)
    qo.tofile(tmp_path / "down.qw")
    so.tofile(tmp_path / "down.sc")
    qw = torch.empty((K // 8, N), dtype=torch.int32, device="cuda")
    sc = torch.empty((K // 32, N), dtype=torch.float32, device="cuda")
    w4.w4a16_load_qw_sc(str(tmp_path / "down.qw"), str(tmp_path / "down.sc"), K, N, qw, sc)
    np.testing.assert_array_equal(host(qw), qo)
    np.testing.assert_array_equal(host(sc), so)
    reg = w4.Registry()
    reg.add("mlp.down", qw, sc)
    reg.add("mlp.gate_up", dev(qgo), dev(sgo))
    x = synth.activations(3, K, seed=23)
    assert_close_rows(host(reg.linear("mlp.down", dev(x))), oracle.gemm(x, qo, so), FP32_TOL, "linear")
    assert_close_rows(host(reg.linear_swiglu("mlp.gate_up", dev(x))), oracle.swiglu_gemm(x, qgo, sgo),
                      FP32_TOL, "linear_swiglu")
    with pytest.raises(w4.W4A16Error) as ei:
        reg.linear("mlp.up", dev(x))
    assert ei.value.status == 6
    reg.close()
