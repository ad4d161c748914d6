"""Plain, slow, float64 CPU oracle of the INT4 W4A16 symmetric group-quantized GEMM.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``; never by the library. It shares no code with the CUDA path.

Sources (web pages; cited by title and section):

* [Weight of Precision] "The Weight of Precision: Building Native INT4 Quantization for a Custom
  Speculative Decoding Engine" -- sections "The Kernel: w4a16_gemm", "The Reference and Bundle
  Pipeline", "The Engine Dispatch: Model::linear".
* [First Line] "The First Line of Code: Implementing W4A16 Quantization in a Native Speculative
  Decoding Engine" -- section "What the Edit Actually Does".
* [Final Wire] "The Final Wire: How a Single Edit Integrated INT4 Quantization into a Native DDTree
  Inference Engine" -- sections "The Multi-Step Integration Chain", "What the Edit Actually
  Changes", "Input Knowledge Required".

What the pages fix: weights are 4-bit, symmetric, value = nibble - 8 (range [-8, 7]); eight nibbles
per int32 along the input dimension K; one float32 scale per group of 32 input rows per output
column; activations and outputs float32; the reference is a numpy dequantized forward whose
dequantization the kernel must reproduce.

What the pages leave open, and the reading taken here (each is also listed in the design notes):

* scale formula: s = absmax(group) / 7, computed in float32 (the scale file holds float32);
* rounding: q = clamp(rint(w / s), -8, 7), w / s in float32, rint = round half to even (numpy's);
* all-zero group: s = 0 and q = 0 (nibble 8);
* nibble order: k = 8 i + j lives in bits [4 j, 4 j + 3] of word i (lowest nibble = lowest k);
* layout: qw[K/8, N] int32 and sc[K/32, N] float32, both row-major;
* fused gate/up: columns [0, I) are gate, [I, 2I) are up; output silu(gate) * up;
* MoE: out[t] = sum over the token's top-k experts of w[t, slot] * down_e(SwiGLU(gate_up_e(x[t])));
  router weights w = softmax over the token's top-k logits.

Arithmetic: quantization happens in float32 (it decides integers, and both sides decide them in
float32); dequantization and every product and sum after it are float64, where q * s is exact.
"""
from __future__ import annotations

import numpy as np

GROUP = 32          # [Weight of Precision] "The Kernel": group size 32, "matching K2.6"
NIB_PER_WORD = 8    # [Weight of Precision] "The Kernel": 8 nibbles per int32 along the input dim
QMIN, QMAX = -8, 7  # [Weight of Precision] "The Kernel": value = nibble - 8, range [-8, 7]


def _check_kn(K: int, N: int, group: int) -> None:
    if group != GROUP:
        raise ValueError(f"group must be {GROUP}")
    if K % group != 0:
        raise ValueError("K must be a multiple of the group size")


# ------------------------------------------------------------------------------------- format

def pack_int4(q: np.ndarray) -> np.ndarray:
    """Pack integer codes q[K, N] in [-8, 7] into qw[K/8, N] int32.

    nibble = q + 8 ([Weight of Precision] "The Kernel": value = nibble - 8); the eight codes
    k = 8 i .. 8 i + 7 of a column go to word i, code 8 i + j in bits [4 j, 4 j + 3]
    (reading: lowest nibble = lowest k)."""
    q = np.asarray(q)
    K, N = q.shape
    if K % NIB_PER_WORD:
        raise ValueError("K must be a multiple of 8")
    if q.min(initial=0) < QMIN or q.max(initial=0) > QMAX:
        raise ValueError("codes outside [-8, 7]")
    nib = (q.astype(np.int64) + 8).astype(np.uint64).reshape(K // NIB_PER_WORD, NIB_PER_WORD, N)
    word = np.zeros((K // NIB_PER_WORD, N), dtype=np.uint64)
    for j in range(NIB_PER_WORD):
        word |= nib[:, j, :] << np.uint64(4 * j)
    return word.astype(np.uint32).view(np.int32)


def unpack_int4(qw: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_int4`: qw[K/8, N] int32 -> codes q[K, N] int8 = nibble - 8.

    Every nibble 0..15 decodes, including 0 (= -8), which the absmax/7 quantizer never emits
    but the format allows ([Weight of Precision] "The Kernel": range [-8, 7])."""
    u = np.asarray(qw).view(np.uint32).astype(np.uint64)
    K8, N = u.shape
    out = np.empty((K8, NIB_PER_WORD, N), dtype=np.int8)
    for j in range(NIB_PER_WORD):
        out[:, j, :] = ((u >> np.uint64(4 * j)) & np.uint64(0xF)).astype(np.int8) - 8
    return out.reshape(K8 * NIB_PER_WORD, N)


def quantize_w4a16(W: np.ndarray, group: int = GROUP):
    """Symmetric group quantization of float32 weights W[K, N] -> (qw[K/8, N] int32, sc[K/32, N] f32).

    Per group g of 32 consecutive input rows and per output column n
    ([First Line] "What the Edit Actually Does": each group of input rows shares a scale per
    output column; [Final Wire] "Input Knowledge Required": scales shared along the input dim):

        s[g, n] = max_{k in g} |W[k, n]| / 7          (float32; reading: absmax / 7)
        q[k, n] = clamp(rint(W[k, n] / s[g, n]), -8, 7)   (float32 division, half to even)
        s = 0  ->  q = 0

    then :func:`pack_int4`. The scale array is what the ``.sc`` files hold (float32,
    [Weight of Precision] "The Reference and Bundle Pipeline")."""
    W = np.asarray(W, dtype=np.float32)
    K, N = W.shape
    _check_kn(K, N, group)
    Wg = W.reshape(K // group, group, N)
    absmax = np.abs(Wg).max(axis=1)                          # [G, N] float32
    sc = (absmax / np.float32(7.0)).astype(np.float32)       # float32 division
    zero = sc == 0
    denom = np.where(zero, np.float32(1.0), sc).astype(np.float32)
    r = np.rint(Wg / denom[:, None, :])                      # float32 w / s, ties to even
    r = np.where(zero[:, None, :], np.float32(0.0), r)
    q = np.clip(r, QMIN, QMAX).astype(np.int8).reshape(K, N)
    return pack_int4(q), sc


def dequantize(qw: np.ndarray, sc: np.ndarray, group: int = GROUP) -> np.ndarray:
    """float64 weights w[k, n] = (nibble - 8) * s[k // 32, n] (exact in float64).

    [First Line] "What the Edit Actually Does": the dequantization arithmetic is the one the
    kernel must reproduce."""
    q = unpack_int4(qw).astype(np.float64)
    K, N = q.shape
    _check_kn(K, N, group)
    s = np.asarray(sc, dtype=np.float32).astype(np.float64)
    if s.shape != (K // group, N):
        raise ValueError("scale array shape mismatch")
    return q * np.repeat(s, group, axis=0)


# ------------------------------------------------------------------------------------- GEMMs

def gemm(x: np.ndarray, qw: np.ndarray, sc: np.ndarray, group: int = GROUP) -> np.ndarray:
    """y[M, N] = x[M, K] @ dequantize(qw, sc), in float64.

    [Weight of Precision] "The Kernel: w4a16_gemm" and [Final Wire] "The Multi-Step Integration
    Chain" step 1: float32 activations times packed INT4 weights with float32 group scales,
    producing float32 outputs; step 2: the numpy dequantized forward is the spec."""
    x = np.asarray(x, dtype=np.float64)
    return x @ dequantize(qw, sc, group)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)), float64."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_gemm(x: np.ndarray, qw_gu: np.ndarray, sc_gu: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Fused gate/up projection of a SwiGLU MLP: h = x @ W_gu with W_gu = [gate | up] along N,
    output silu(h[:, :I]) * h[:, I:]  ([M, I], float64).

    The SwiGLU MLP (gate, up, down) is the layer the pages route through the INT4 path
    ([Final Wire] "What the Edit Actually Changes"; [Weight of Precision] "The Engine Dispatch")."""
    h = gemm(x, qw_gu, sc_gu, group)
    N2 = h.shape[1]
    if N2 % 2:
        raise ValueError("gate/up width must be even")
    I = N2 // 2
    return silu(h[:, :I]) * h[:, I:]


def topk_softmax(logits: np.ndarray) -> np.ndarray:
    """Router weights over a token's selected experts: softmax of their logits, float64."""
    l = np.asarray(logits, dtype=np.float64)
    e = np.exp(l - l.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def moe_forward(x, topk_ids, topk_w, gate_up, down, group: int = GROUP) -> np.ndarray:
    """Routed-expert MoE block, float64.

    out[t] = sum_{slot} topk_w[t, slot] * down_e(swiglu(gate_up_e(x[t]))),  e = topk_ids[t, slot]

    ``gate_up(e)`` and ``down(e)`` return (qw, sc) of expert e. Experts are visited one at a time
    (each expert's weights are needed once), with all the tokens routed to it.
    [Final Wire] "What the Edit Actually Changes": per token the router selects top-k experts and
    each expert's gate, up and down projections go through the INT4 linear."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids)
    w = np.asarray(topk_w, dtype=np.float64)
    T, topk = ids.shape
    out = np.zeros((T, x.shape[1]), dtype=np.float64)
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        h = swiglu_gemm(x[tok], *gate_up(int(e)), group)
        y = gemm(h, *down(int(e)), group)
        np.add.at(out, tok, w[tok, slot][:, None] * y)
    return out


def moe_block_forward(x, topk_ids, topk_w, gate_up, down, shared_gate_up, shared_down,
                      group: int = GROUP) -> np.ndarray:
    """MoE block with a shared expert, float64: the routed sum of moe_forward plus one expert
    that every token goes through with weight 1,

    out[t] = down_s(swiglu(gate_up_s(x[t]))) + sum_{slot} topk_w[t, slot] * down_e(...)

    ``shared_gate_up`` and ``shared_down`` are (qw, sc) pairs.
    [Weight of Precision] "The Engine Dispatch: Model::linear": the MoE experts, the shared expert
    and the dense MLP layers run through the INT4 path."""
    routed = moe_forward(x, topk_ids, topk_w, gate_up, down, group)
    shared = gemm(swiglu_gemm(x, *shared_gate_up, group), *shared_down, group)
    return routed + shared


# ------------------------------------------------------------------------------------- bf16 prefill

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 numbers given as uint16 bit patterns (bf16 = upper half of a float32)."""
    b = np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def gemm_bf16(x_bits: np.ndarray, qw: np.ndarray, sc: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Large-M contraction with bf16 activations: exact float64 value of x_bf16 @ dequantize(W).

    The CUDA path rounds dequantized weights and its output to bf16; it is compared against this
    exact product with a relative-L2 tolerance."""
    return bf16_bits_to_f64(x_bits) @ dequantize(qw, sc, group)


# ------------------------------------------------------------------------------------- metric

def rel_l2(a: np.ndarray, ref: np.ndarray) -> float:
    """||a - ref||_2 / ||ref||_2 over the whole tensor (0 when both are all-zero)."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((a - ref).ravel())
    if den == 0:
        return 0.0 if num == 0 else float("inf")
    return float(num / den)
