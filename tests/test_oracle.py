"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes a part of the oracle to something external: a hand-derived fixture, a closed
form, an invariant, a textbook or library routine, or a brute-force restatement on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _word(h):
    return np.array([int(h, 16)], dtype=np.uint32).view(np.int32)[0]


# ----------------------------------------------------------------------------- hand fixtures

def test_hand_quantized_group():
    g = _load("quant_group_k32_n3.json")
    W = np.array(g["W_columns"], dtype=np.float32).T           # [32, 3]
    qw, sc = oracle.quantize_w4a16(W)
    assert qw.dtype == np.int32 and qw.shape == (4, 3)
    assert sc.dtype == np.float32 and sc.shape == (1, 3)
    assert sc[0].tolist() == g["scales"]
    want = np.array([[_word(h) for h in col] for col in g["qw_hex_columns"]], dtype=np.int32).T
    np.testing.assert_array_equal(qw, want)
    np.testing.assert_array_equal(oracle.unpack_int4(qw), np.array(g["q_columns"]).T)
    x = np.zeros((1, 32), dtype=np.float32)
    for k, v in g["x_nonzero"].items():
        x[0, int(k)] = v
    y = oracle.gemm(x, qw, sc)
    assert y[0].tolist() == g["y"]


def test_hand_nibble_decode():
    g = _load("nibble_decode.json")
    for case in g["cases"]:
        qw = np.array([[_word(case["word_hex"])]], dtype=np.int32)
        assert oracle.unpack_int4(qw)[:, 0].tolist() == case["codes"]
        np.testing.assert_array_equal(oracle.pack_int4(np.array(case["codes"])[:, None]), qw)


# ----------------------------------------------------------------------------- format invariants

def test_pack_unpack_roundtrip_all_nibbles():
    rng = np.random.default_rng(1)
    q = rng.integers(-8, 8, size=(64 * 8, 37))
    q[0, 0], q[1, 0], q[2, 5] = -8, 7, -8          # nibbles 0 and 15 present
    qw = oracle.pack_int4(q)
    np.testing.assert_array_equal(oracle.unpack_int4(qw), q)
    u = qw.view(np.uint32)
    # reading of the layout: word i of column n holds k = 8i..8i+7, lowest nibble first
    assert (int(u[0, 0]) & 0xF) == q[0, 0] + 8 and ((int(u[0, 0]) >> 4) & 0xF) == q[1, 0] + 8
    assert ((int(u[0, 5]) >> 8) & 0xF) == q[2, 5] + 8


def test_pack_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.pack_int4(np.full((8, 1), 8))
    with pytest.raises(ValueError):
        oracle.pack_int4(np.full((8, 1), -9))


def test_quantizer_range_and_error_bound():
    W = synth.weights(256, 96, seed=3, outliers=True)
    qw, sc = oracle.quantize_w4a16(W)
    q = oracle.unpack_int4(qw)
    assert q.min() >= -7 and q.max() <= 7            # -8 unreachable under absmax/7
    # every group has a code of magnitude 7 exactly at its absmax entry
    qa = np.abs(q).reshape(8, 32, 96).max(axis=1)
    assert (qa == 7).all()
    # |w - dequant(w)| <= s/2, with one float32 ulp of w/s as slack
    deq = oracle.dequantize(qw, sc)
    s = np.repeat(sc.astype(np.float64), 32, axis=0)
    err = np.abs(W.astype(np.float64) - deq)
    assert (err <= s * (0.5 + 8 * 2.0 ** -24) + 0).all()
    # the bound is attained to within rounding somewhere (the quantizer is not finer than s)
    assert (err / s).max() > 0.45


def test_all_zero_group_and_zero_weights():
    W = np.zeros((64, 8), dtype=np.float32)
    qw, sc = oracle.quantize_w4a16(W)
    assert (sc == 0).all()
    assert (qw.view(np.uint32) == 0x88888888).all()
    x = synth.activations(3, 64, seed=5)
    assert (oracle.gemm(x, qw, sc) == 0).all()


def test_group_direction_is_along_k():
    # one large entry must only change the scale of its own (group, column)
    W = np.full((64, 4), 0.25, dtype=np.float32)
    W[40, 2] = 7.0
    _, sc = oracle.quantize_w4a16(W)
    want = np.full((2, 4), np.float32(0.25) / np.float32(7), dtype=np.float32)
    want[1, 2] = 1.0
    np.testing.assert_array_equal(sc, want)


# ----------------------------------------------------------------------------- grid identity

def test_on_grid_weights_reduce_to_plain_matmul():
    """W = q * 2^e with each group holding a +-7: quantization returns q exactly and the oracle
    equals numpy's float64 matmul of x and W."""
    rng = np.random.default_rng(7)
    K, N, M = 128, 40, 5
    q = rng.integers(-7, 8, size=(K, N))
    for g in range(K // 32):
        q[32 * g + rng.integers(0, 32, size=N), np.arange(N)] = rng.choice([-7, 7], size=N)
    e = rng.integers(-12, 3, size=(K // 32, N))
    s = np.ldexp(1.0, e)
    W = (q * np.repeat(s, 32, axis=0)).astype(np.float32)
    qw, sc = oracle.quantize_w4a16(W)
    np.testing.assert_array_equal(oracle.unpack_int4(qw), q)
    # absmax/7 = 7*2^e/7 = 2^e exactly
    np.testing.assert_array_equal(sc, s.astype(np.float32))
    x = rng.standard_normal((M, K))
    np.testing.assert_array_equal(oracle.gemm(x, qw, sc), x @ W.astype(np.float64))


# ----------------------------------------------------------------------------- brute force

def _brute_quant_gemm(x, W):
    """Scalar restatement on tiny inputs: python max/abs, float32 division via numpy scalars,
    python's round() (half to even), exact sums with math.fsum."""
    K, N = len(W), len(W[0])
    y = [[0.0] * N for _ in x]
    for n in range(N):
        deq = []
        for g in range(K // 32):
            col = [np.float32(W[32 * g + i][n]) for i in range(32)]
            s = np.float32(max(abs(v) for v in col)) / np.float32(7)
            for v in col:
                if s == 0:
                    qv = 0
                else:
                    qv = round(float(np.float32(v) / s))
                    qv = max(-8, min(7, qv))
                deq.append(qv * float(s))
        for m, row in enumerate(x):
            y[m][n] = math.fsum(float(row[k]) * deq[k] for k in range(K))
    return np.array(y)


@pytest.mark.parametrize("M,K,N", [(1, 32, 16), (2, 64, 16), (2, 64, 5)])
def test_brute_force_tiny(M, K, N):
    W = synth.weights(K, N, seed=11 + K + N, outliers=True)
    x = synth.activations(M, K, seed=12 + M)
    qw, sc = oracle.quantize_w4a16(W)
    want = _brute_quant_gemm(x.tolist(), W.tolist())
    got = oracle.gemm(x, qw, sc)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- special cases

def test_one_hot_rows_and_matvec():
    W = synth.weights(96, 24, seed=2)
    qw, sc = oracle.quantize_w4a16(W)
    deq = oracle.dequantize(qw, sc)
    for k in (0, 31, 32, 95):
        x = np.zeros((1, 96))
        x[0, k] = 1.0
        np.testing.assert_array_equal(oracle.gemm(x, qw, sc)[0], deq[k])
    x = synth.activations(1, 96, seed=4)
    np.testing.assert_allclose(oracle.gemm(x, qw, sc)[0], deq.T @ x[0].astype(np.float64),
                               rtol=1e-14, atol=1e-16)


def test_quantization_is_not_a_no_op():
    """INT4 output differs from the unquantized float product by a clearly visible amount (the
    pages check that INT4 and FP32 goldens diverge; here the gap must exceed the kernel tolerance)."""
    W = synth.weights(512, 256, seed=9)
    x = synth.activations(4, 512, seed=10)
    qw, sc = oracle.quantize_w4a16(W)
    d = oracle.rel_l2(oracle.gemm(x, qw, sc), x.astype(np.float64) @ W.astype(np.float64))
    assert 1e-2 < d < 0.5


# ----------------------------------------------------------------------------- SwiGLU

def test_silu_closed_form():
    z = np.array([-30.0, -2.0, -0.5, 0.0, 0.5, 1.0, 3.0, 40.0])
    np.testing.assert_allclose(oracle.silu(z), z * scipy.special.expit(z), rtol=1e-15, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.e ** -1)) < 1e-16


def test_swiglu_gate_up_order():
    """One-hot x picks row k of the dequantized [gate | up] weights; the result must be
    silu(gate) * up, not silu(up) * gate."""
    K, I = 64, 8
    rng = np.random.default_rng(3)
    q = rng.integers(-7, 8, size=(K, 2 * I))
    q[0, :] = 7
    q[32, :] = -7
    W = (q * 0.25).astype(np.float32)
    qw, sc = oracle.quantize_w4a16(W)
    k = 5
    x = np.zeros((1, K))
    x[0, k] = 1.0
    gate, up = W[k, :I].astype(np.float64), W[k, I:].astype(np.float64)
    want = gate * scipy.special.expit(gate) * up
    np.testing.assert_allclose(oracle.swiglu_gemm(x, qw, sc)[0], want, rtol=1e-15)
    assert not np.allclose(want, up * scipy.special.expit(up) * gate)


# ----------------------------------------------------------------------------- MoE

def test_topk_softmax_matches_scipy():
    _, logits = synth.routing(16, 32, 8, seed=1)
    p = oracle.topk_softmax(logits)
    np.testing.assert_allclose(p, scipy.special.softmax(logits.astype(np.float64), axis=1), rtol=1e-14)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-15)


def _tiny_moe(E=6, K=64, I=32, T=5, topk=3, seed=0):
    ids, logits = synth.routing(T, E, topk, seed=seed)
    x = synth.activations(T, K, seed=seed + 1)
    gu, dn = {}, {}
    for e in range(E):
        wg, wd = synth.moe_expert_weights(e, K, I, seed=seed)
        gu[e] = oracle.quantize_w4a16(wg)
        dn[e] = oracle.quantize_w4a16(wd)
    return x, ids, logits, gu, dn


def test_moe_brute_force_per_pair():
    x, ids, logits, gu, dn = _tiny_moe()
    w = oracle.topk_softmax(logits)
    got = oracle.moe_forward(x, ids, w, gu.__getitem__, dn.__getitem__)
    T, topk = ids.shape
    want = np.zeros_like(got)
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            deq_gu = oracle.dequantize(*gu[e])
            deq_dn = oracle.dequantize(*dn[e])
            hh = [math.fsum(float(x[t, k]) * deq_gu[k, n] for k in range(x.shape[1]))
                  for n in range(deq_gu.shape[1])]
            I = len(hh) // 2
            act = [hh[i] / (1.0 + math.exp(-hh[i])) * hh[I + i] for i in range(I)]
            for n in range(deq_dn.shape[1]):
                want[t, n] += w[t, j] * math.fsum(act[i] * deq_dn[i, n] for i in range(I))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_moe_identical_experts_equal_dense_mlp():
    """Router weights sum to one, so with every expert equal the MoE output is that expert's MLP."""
    x, ids, logits, gu, dn = _tiny_moe()
    w = oracle.topk_softmax(logits)
    one_gu, one_dn = gu[0], dn[0]
    got = oracle.moe_forward(x, ids, w, lambda e: one_gu, lambda e: one_dn)
    dense = oracle.gemm(oracle.swiglu_gemm(x, *one_gu), *one_dn)
    np.testing.assert_allclose(got, dense, rtol=1e-12, atol=1e-14)


def test_moe_weights_scale_linearly():
    x, ids, logits, gu, dn = _tiny_moe(seed=4)
    w = oracle.topk_softmax(logits)
    a = oracle.moe_forward(x, ids, w, gu.__getitem__, dn.__getitem__)
    b = oracle.moe_forward(x, ids, 2.0 * w, gu.__getitem__, dn.__getitem__)
    np.testing.assert_allclose(b, 2.0 * a, rtol=1e-14)
    z = oracle.moe_forward(x, ids, np.zeros_like(w), gu.__getitem__, dn.__getitem__)
    assert (z == 0).all()


def _mlp_brute_force(x_row, qgu, qdn):
    """One token through one expert's SwiGLU MLP with scalar exact sums."""
    deq_gu = oracle.dequantize(*qgu)
    deq_dn = oracle.dequantize(*qdn)
    hh = [math.fsum(float(x_row[k]) * deq_gu[k, n] for k in range(len(x_row)))
          for n in range(deq_gu.shape[1])]
    I = len(hh) // 2
    act = [hh[i] / (1.0 + math.exp(-hh[i])) * hh[I + i] for i in range(I)]
    return np.array([math.fsum(act[i] * deq_dn[i, n] for i in range(I))
                     for n in range(deq_dn.shape[1])])


def _shared_expert(K=64, Is=64, seed=9):
    wg, wd = synth.moe_expert_weights(100, K, Is, seed=seed)
    return oracle.quantize_w4a16(wg), oracle.quantize_w4a16(wd)


def test_moe_block_brute_force():
    x, ids, logits, gu, dn = _tiny_moe(seed=2)
    sgu, sdn = _shared_expert()
    w = oracle.topk_softmax(logits)
    got = oracle.moe_block_forward(x, ids, w, gu.__getitem__, dn.__getitem__, sgu, sdn)
    T, topk = ids.shape
    for t in range(T):
        want = _mlp_brute_force(x[t], sgu, sdn)
        for j in range(topk):
            e = int(ids[t, j])
            want = want + w[t, j] * _mlp_brute_force(x[t], gu[e], dn[e])
        np.testing.assert_allclose(got[t], want, rtol=1e-12, atol=1e-14)


def test_moe_block_reduces_to_its_parts():
    """Zero shared weights give the routed block; zero router weights give the shared MLP."""
    x, ids, logits, gu, dn = _tiny_moe(seed=3)
    sgu, sdn = _shared_expert(seed=4)
    w = oracle.topk_softmax(logits)
    zgu = oracle.quantize_w4a16(np.zeros((64, 128), dtype=np.float32))
    zdn = oracle.quantize_w4a16(np.zeros((64, 64), dtype=np.float32))
    routed = oracle.moe_forward(x, ids, w, gu.__getitem__, dn.__getitem__)
    np.testing.assert_array_equal(
        oracle.moe_block_forward(x, ids, w, gu.__getitem__, dn.__getitem__, zgu, zdn), routed)
    only_shared = oracle.moe_block_forward(x, ids, np.zeros_like(w), gu.__getitem__,
                                           dn.__getitem__, sgu, sdn)
    for t in range(x.shape[0]):
        np.testing.assert_allclose(only_shared[t], _mlp_brute_force(x[t], sgu, sdn), rtol=1e-12,
                                   atol=1e-14)


# ----------------------------------------------------------------------------- bf16

def test_bf16_decode_matches_torch():
    import torch
    bits = synth.bf16_activations(4, 64, seed=2)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits), ref)
    special = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x0001], dtype=np.uint16)
    v = oracle.bf16_bits_to_f64(special)
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 0.0 and v[3] == 3.140625
    assert v[4] == 2.0 ** -133


def test_gemm_bf16_is_exact_product():
    bits = synth.bf16_activations(3, 64, seed=6)
    W = synth.weights(64, 16, seed=6)
    qw, sc = oracle.quantize_w4a16(W)
    xv = oracle.bf16_bits_to_f64(bits)
    np.testing.assert_array_equal(oracle.gemm_bf16(bits, qw, sc), xv @ oracle.dequantize(qw, sc))


def test_rel_l2():
    a = np.array([3.0, 4.0])
    assert oracle.rel_l2(a, a) == 0.0
    assert abs(oracle.rel_l2(a + np.array([0.3, 0.4]), a) - 0.1) < 1e-15
