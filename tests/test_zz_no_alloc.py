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

import synth
from gpu_util import FP32_TOL, assert_close_rows, host, lib

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
