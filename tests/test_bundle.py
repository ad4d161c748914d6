"""Multi-tensor weight bundle: the writer and the library's index reader agree on the layout
(host-only checks), malformed files are refused before anything is copied, and on the GPU a
loaded bundle drives linear() with the same results as the tensors passed directly."""
import struct

import numpy as np
import pytest
import torch

import oracle
import synth
from int4_w4a16_group_gb300.bundle import write_bundle


def _tensors():
    out = {}
    for i, (K, N) in enumerate([(64, 96), (256, 40), (32, 4)]):
        out[f"layers.{i}.mlp.w{i}"] = oracle.quantize_w4a16(synth.weights(K, N, seed=70 + i))
    return out


def _align256(v):
    return (v + 255) // 256 * 256


def test_info_reads_the_index(tmp_path):
    from int4_w4a16_group_gb300 import bundle_info
    t = _tensors()
    p = tmp_path / "w.bdl"
    write_bundle(p, t)
    count, nbytes = bundle_info(p)
    assert count == 3
    assert nbytes == sum(_align256(q.nbytes) + _align256(s.nbytes) for q, s in t.values())


@pytest.mark.parametrize("damage", ["magic", "version", "truncated", "bad_k", "dup_name"])
def test_malformed_bundles_are_refused(tmp_path, damage):
    from int4_w4a16_group_gb300 import W4A16Error, bundle_info
    t = _tensors()
    if damage == "dup_name":
        t = [("a", t["layers.0.mlp.w0"]), ("a", t["layers.1.mlp.w1"])]
    p = tmp_path / "w.bdl"
    write_bundle(p, t)
    raw = bytearray(p.read_bytes())
    if damage == "magic":
        raw[0:1] = b"X"
    elif damage == "version":
        raw[8:12] = struct.pack("<I", 2)
    elif damage == "truncated":
        raw = raw[: len(raw) - 100]
    elif damage == "bad_k":
        n = struct.unpack("<I", raw[16:20])[0]
        raw[20 + n:24 + n] = struct.pack("<i", 48)   # K not a multiple of 32
    p.write_bytes(bytes(raw))
    with pytest.raises(W4A16Error) as ei:
        bundle_info(p)
    assert ei.value.status == 7   # W4A16_ERR_IO


def test_missing_file(tmp_path):
    from int4_w4a16_group_gb300 import W4A16Error, bundle_info
    with pytest.raises(W4A16Error):
        bundle_info(tmp_path / "none.bdl")


@pytest.mark.gpu
def test_bundle_drives_linear(tmp_path):
    from gpu_util import FP32_TOL, assert_close_rows, dev, host, lib
    w4 = lib()
    t = _tensors()
    p = tmp_path / "w.bdl"
    write_bundle(p, t)
    reg = w4.Registry()
    reg.load_bundle(p)
    for name, (qo, so) in t.items():
        K, N = reg.find(name)
        assert (K, N) == (qo.shape[0] * 8, qo.shape[1])
        x = synth.activations(3, K, seed=K + N)
        y_reg = host(reg.linear(name, dev(x)))
        y_dir = host(w4.w4a16_gemm(dev(x), dev(qo), dev(so)))
        np.testing.assert_array_equal(y_reg, y_dir)
        assert_close_rows(y_reg, oracle.gemm(x, qo, so), FP32_TOL, name)
    reg.close()
