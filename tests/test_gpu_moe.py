"""GPU parity of the routed-expert MoE block (w4a16_moe_gemm) and of the router softmax,
through the C ABI, against the oracle. Small cases cover skewed routing (one expert receiving
more rows than one pass holds), unused experts, ragged widths and top-1; the full-size
tree-verify workload (T=64, E=384, top-8) is checked on sampled tokens, with and without a
shared expert (w4a16_moe_block)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import FP32_TOL, assert_close_rows, dev, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    return lib()


def _experts(w4, E, K, I, seed):
    gu_o, dn_o, gq, gs, dq, ds = [], [], [], [], [], []
    for e in range(E):
        a, b = synth.moe_expert_weights(e, K, I, seed=seed)
        gu_o.append(oracle.quantize_w4a16(a))
        dn_o.append(oracle.quantize_w4a16(b))
        q, s = w4.w4a16_quantize(dev(a))
        gq.append(q)
        gs.append(s)
        q, s = w4.w4a16_quantize(dev(b))
        dq.append(q)
        ds.append(s)
    return gu_o, dn_o, (torch.stack(gq), torch.stack(gs), torch.stack(dq), torch.stack(ds))


def test_topk_softmax(w4):
    _, logits = synth.routing(64, 384, 8, seed=3)
    logits[0] = 0.0
    logits[1, 0] = 50.0
    p = host(w4.w4a16_topk_softmax(dev(logits)))
    ref = oracle.topk_softmax(logits)
    np.testing.assert_allclose(p, ref, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,topk,K,I,skew", [
    (5, 6, 3, 128, 64, False),
    (16, 8, 2, 256, 96, False),      # I not a multiple of the 64-column tile
    (24, 4, 2, 96, 32, True),        # one expert gets > 8 rows (several passes), one gets none
    (7, 5, 1, 64, 64, False),        # top-1
])
def test_moe_small(w4, T, E, topk, K, I, skew):
    seed = T + E
    ids, logits = synth.routing(T, E, topk, seed=seed)
    if skew:
        ids[:, 0] = 0                  # every token picks expert 0 first
        ids[:, 1] = 1 + (np.arange(T) % (E - 2))   # expert E-1 never used
    x = synth.activations(T, K, seed=seed)
    gu_o, dn_o, (gq, gs, dq, ds) = _experts(w4, E, K, I, seed)
    wts = w4.w4a16_topk_softmax(dev(logits))
    out = w4.w4a16_moe_gemm(dev(x), dev(ids), wts, gq, gs, dq, ds)
    ref = oracle.moe_forward(x, ids, oracle.topk_softmax(logits), gu_o.__getitem__, dn_o.__getitem__)
    assert_close_rows(host(out), ref, FP32_TOL, "moe")
    assert w4.w4a16_device_error() == 0


def test_moe_is_deterministic_and_reuses_workspace(w4):
    T, E, topk, K, I = 12, 6, 3, 128, 64
    ids, logits = synth.routing(T, E, topk, seed=9)
    x = synth.activations(T, K, seed=9)
    _, _, (gq, gs, dq, ds) = _experts(w4, E, K, I, 9)
    wts = w4.w4a16_topk_softmax(dev(logits))
    ws = torch.full((w4.w4a16_moe_workspace_size(T, topk, E, K, I),), 0xAB, dtype=torch.uint8,
                    device="cuda")
    a = host(w4.w4a16_moe_gemm(dev(x), dev(ids), wts, gq, gs, dq, ds, workspace=ws))
    b = host(w4.w4a16_moe_gemm(dev(x), dev(ids), wts, gq, gs, dq, ds, workspace=ws))
    np.testing.assert_array_equal(a, b)


def test_moe_bad_expert_id_is_flagged(w4):
    T, E, topk, K, I = 4, 4, 2, 64, 32
    ids, logits = synth.routing(T, E, topk, seed=1)
    ids[2, 1] = E + 3                  # out of range: skipped, flagged on the device
    x = synth.activations(T, K, seed=1)
    gu_o, dn_o, (gq, gs, dq, ds) = _experts(w4, E, K, I, 1)
    w = oracle.topk_softmax(logits)
    out = host(w4.w4a16_moe_gemm(dev(x), dev(ids), dev(w.astype(np.float32)), gq, gs, dq, ds))
    assert w4.w4a16_device_error() == 1
    ids_ok, w_ok = ids.copy(), w.copy()
    ids_ok[2, 1] = 0
    w_ok[2, 1] = 0.0                   # the skipped pair contributes nothing
    ref = oracle.moe_forward(x, ids_ok, w_ok, gu_o.__getitem__, dn_o.__getitem__)
    assert_close_rows(out, ref, FP32_TOL, "moe bad id")
    assert w4.w4a16_device_error() == 0


def test_full_size_tree_verify_moe(w4):
    """T=64 draft-tree rows, 384 experts, top-8: all experts quantized on the device by the
    library, full MoE call; the oracle recomputes two sampled tokens from their experts'
    float32 weights (redrawn from the same per-expert device streams)."""
    c = synth.MOE
    T, E, topk, K, I = c["T"], c["E"], c["topk"], c["K"], c["I"]
    seed = 0
    gq = torch.empty((E, K // 8, 2 * I), dtype=torch.int32, device="cuda")
    gs = torch.empty((E, K // 32, 2 * I), dtype=torch.float32, device="cuda")
    dq = torch.empty((E, I // 8, K), dtype=torch.int32, device="cuda")
    ds = torch.empty((E, I // 32, K), dtype=torch.float32, device="cuda")
    for e in range(E):
        a, b = synth.cuda_moe_expert_weights(e, K, I, seed=seed)
        w4.w4a16_quantize(a, gq[e], gs[e])
        w4.w4a16_quantize(b, dq[e], ds[e])
    del a, b
    ids, logits = synth.routing(T, E, topk, seed=seed)
    x = synth.activations(T, K, seed=seed)
    wts = w4.w4a16_topk_softmax(dev(logits))
    out = host(w4.w4a16_moe_gemm(dev(x), dev(ids), wts, gq, gs, dq, ds))
    assert w4.w4a16_device_error() == 0
    toks = [5, 63]
    need = sorted(set(int(e) for t in toks for e in ids[t]))
    gu_o, dn_o = {}, {}
    for e in need:
        a, b = synth.cuda_moe_expert_weights(e, K, I, seed=seed)
        gu_o[e] = oracle.quantize_w4a16(host(a))
        dn_o[e] = oracle.quantize_w4a16(host(b))
        np.testing.assert_array_equal(host(gq[e]), gu_o[e][0])
        np.testing.assert_array_equal(host(ds[e]), dn_o[e][1])
    ref = oracle.moe_forward(x[toks], ids[toks], oracle.topk_softmax(logits[toks]),
                             gu_o.__getitem__, dn_o.__getitem__)
    assert_close_rows(out[toks], ref, FP32_TOL, "full-size moe")

    # the same block with a shared expert of the routed experts' width
    a, b = synth.cuda_moe_expert_weights(E, K, I, seed=seed + 1)
    sgq, sgs = w4.w4a16_quantize(a)
    sdq, sds = w4.w4a16_quantize(b)
    sgu_o, sdn_o = oracle.quantize_w4a16(host(a)), oracle.quantize_w4a16(host(b))
    del a, b
    blk = host(w4.w4a16_moe_block(dev(x), dev(ids), wts, gq, gs, dq, ds, sgq, sgs, sdq, sds))
    assert w4.w4a16_device_error() == 0
    ref = oracle.moe_block_forward(x[toks], ids[toks], oracle.topk_softmax(logits[toks]),
                                   gu_o.__getitem__, dn_o.__getitem__, sgu_o, sdn_o)
    assert_close_rows(blk[toks], ref, FP32_TOL, "full-size moe block")


@pytest.mark.parametrize("T,E,topk,K,I,Is", [
    (5, 6, 3, 128, 64, 96),
    (20, 8, 2, 256, 96, 64),         # 20 tokens: two 16-row slices of the shared expert
    (7, 5, 1, 64, 64, 32),
])
def test_moe_block_with_shared_expert(w4, T, E, topk, K, I, Is):
    seed = T + E + Is
    ids, logits = synth.routing(T, E, topk, seed=seed)
    x = synth.activations(T, K, seed=seed)
    gu_o, dn_o, (gq, gs, dq, ds) = _experts(w4, E, K, I, seed)
    a, b = synth.moe_expert_weights(99, K, Is, seed=seed)
    sgu_o, sdn_o = oracle.quantize_w4a16(a), oracle.quantize_w4a16(b)
    sgq, sgs = w4.w4a16_quantize(dev(a))
    sdq, sds = w4.w4a16_quantize(dev(b))
    wts = w4.w4a16_topk_softmax(dev(logits))
    out = w4.w4a16_moe_block(dev(x), dev(ids), wts, gq, gs, dq, ds, sgq, sgs, sdq, sds)
    ref = oracle.moe_block_forward(x, ids, oracle.topk_softmax(logits), gu_o.__getitem__,
                                   dn_o.__getitem__, sgu_o, sdn_o)
    assert_close_rows(host(out), ref, FP32_TOL, "moe block")
    assert w4.w4a16_device_error() == 0
