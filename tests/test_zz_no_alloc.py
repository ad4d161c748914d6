"""The MoE entry point for callers that cannot allocate device memory.

w4a16_moe_gemm_noalloc runs the routed-expert MoE block on a fixed scratch array that the
library keeps in device memory, for callers that can only pass inputs and outputs (a plugin or
foreign-function interface with a fixed signature, or a process whose device memory another
runtime has already reserved). These tests call it through the C ABI and compare it with
w4a16_moe_gemm, which takes its scratch from the caller.

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test.
"""
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


def _problem(w4, T, E, topk, K, I, seed):
    """Quantized experts, routing, router weights and activations, all on the device."""
    gq, gs, dq, ds = [], [], [], []
    for e in range(E):
        a, b = synth.moe_expert_weights(e, K, I, seed=seed)
        q, s = w4.w4a16_quantize(torch.from_numpy(a).cuda())
        gq.append(q)
        gs.append(s)
        q, s = w4.w4a16_quantize(torch.from_numpy(b).cuda())
        dq.append(q)
        ds.append(s)
    ids, logits = synth.routing(T, E, topk, seed=seed)
    x = torch.from_numpy(synth.activations(T, K, seed=seed)).cuda()
    wts = w4.w4a16_topk_softmax(torch.from_numpy(logits).cuda())
    return (x, torch.from_numpy(ids).cuda(), wts, torch.stack(gq), torch.stack(gs),
            torch.stack(dq), torch.stack(ds))


def _call_noalloc(w4, prob, out):
    """Raw C-ABI call of w4a16_moe_gemm_noalloc; returns its status."""
    x, ids, wts, gq, gs, dq, ds = prob
    T, K = x.shape
    topk = ids.shape[1]
    E = gq.shape[0]
    I = gq.shape[2] // 2
    return w4.C.w4a16_moe_gemm_noalloc(
        x.data_ptr(), ids.data_ptr(), wts.data_ptr(), T, topk, E, gq.data_ptr(), gs.data_ptr(),
        dq.data_ptr(), ds.data_ptr(), out.data_ptr(), K, I, 32,
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(w4):
    # Two different problems, one call each, back to back: the second call runs on the scratch
    # the first one left behind.
    probs = [_problem(w4, 64, 16, 8, 512, 256, seed=1), _problem(w4, 24, 6, 2, 256, 96, seed=2)]
    refs = [host(w4.w4a16_moe_gemm(*p)) for p in probs]
    outs = [torch.full(tuple(p[0].shape), float("nan"), device="cuda") for p in probs]
    for p, o in zip(probs, outs):
        assert _call_noalloc(w4, p, o) == 0
    for i, (o, r) in enumerate(zip(outs, refs)):
        assert_close_rows(host(o), r, FP32_TOL, f"no-alloc call {i + 1}")
    # and the same problem twice in a row gives the same answer
    again = torch.full(tuple(probs[0][0].shape), float("nan"), device="cuda")
    assert _call_noalloc(w4, probs[0], again) == 0
    assert_close_rows(host(again), refs[0], FP32_TOL, "no-alloc repeat")
    assert w4.w4a16_device_error() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch(w4):
    limit = (32 << 20)
    T, topk, E, K, I = 4096, 8, 384, 7168, 2048
    assert w4.w4a16_moe_workspace_size(T, topk, E, K, I) > limit
    fake = 0x10000  # never touched: the size check comes first
    st = w4.C.w4a16_moe_gemm_noalloc(fake, fake, fake, T, topk, E, fake, fake, fake, fake, fake,
                                     K, I, 32, None)
    assert st == 4  # W4A16_ERR_WORKSPACE
    assert w4.w4a16_moe_workspace_size(64, 8, 384, 7168, 2048) <= limit


def test_noalloc_matches_the_oracle(w4):
    # Experts quantized by the oracle on the host; the no-alloc call against the oracle's MoE
    # forward, every row.
    T, E, topk, K, I, seed = 40, 12, 4, 256, 96, 3
    gu, dn = zip(*[synth.moe_expert_weights(e, K, I, seed=seed) for e in range(E)])
    gu_q = [oracle.quantize_w4a16(a) for a in gu]
    dn_q = [oracle.quantize_w4a16(b) for b in dn]
    ids, logits = synth.routing(T, E, topk, seed=seed)
    x = synth.activations(T, K, seed=seed)
    ref = oracle.moe_forward(x, ids, oracle.topk_softmax(logits), gu_q.__getitem__,
                             dn_q.__getitem__)
    prob = (dev(x), dev(ids), w4.w4a16_topk_softmax(dev(logits)),
            dev(np.stack([q for q, _ in gu_q])), dev(np.stack([s for _, s in gu_q])),
            dev(np.stack([q for q, _ in dn_q])), dev(np.stack([s for _, s in dn_q])))
    out = torch.full((T, K), float("nan"), device="cuda")
    assert _call_noalloc(w4, prob, out) == 0
    assert_close_rows(host(out), ref, FP32_TOL, "no-alloc vs oracle")
    assert w4.w4a16_device_error() == 0


def test_noalloc_at_its_pair_limit(w4):
    # 909 token-expert pairs at K = 7168, I = 2048: the largest problem the fixed scratch holds.
    # Two experts of full size (each streamed once per 8-row pass); the result equals the
    # workspace entry's bit for bit, and three sampled tokens match the oracle, which quantizes
    # their experts from the same float32 weights.
    T, topk, E, K, I, seed = 909, 1, 2, 7168, 2048, 4
    assert w4.w4a16_moe_workspace_size(T, topk, E, K, I) <= 32 << 20
    assert w4.w4a16_moe_workspace_size(T + 1, topk, E, K, I) > 32 << 20
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
    prob = (dev(x), dev(ids), w4.w4a16_topk_softmax(dev(logits)), gq, gs, dq, ds)
    out = torch.full((T, K), float("nan"), device="cuda")
    assert _call_noalloc(w4, prob, out) == 0
    got = host(out)
    np.testing.assert_array_equal(got, host(w4.w4a16_moe_gemm(*prob)))
    assert w4.w4a16_device_error() == 0
    toks = [0, T // 2, T - 1]
    gu_o, dn_o = {}, {}
    for e in sorted(set(int(ids[t, 0]) for t in toks)):
        a, b = synth.cuda_moe_expert_weights(e, K, I, seed=seed)
        gu_o[e] = oracle.quantize_w4a16(host(a))
        dn_o[e] = oracle.quantize_w4a16(host(b))
    ref = oracle.moe_forward(x[toks], ids[toks], oracle.topk_softmax(logits[toks]),
                             gu_o.__getitem__, dn_o.__getitem__)
    assert_close_rows(got[toks], ref, FP32_TOL, "no-alloc at 909 pairs")
