"""CPU oracle of the INT4 W4A16 group-32 path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. It shares no code with the CUDA library and never calls it.

See :mod:`oracle.w4a16_ref` for the definitions and the passages each one follows.
"""
from .w4a16_ref import (  # noqa: F401
    GROUP,
    quantize_w4a16,
    pack_int4,
    unpack_int4,
    dequantize,
    gemm,
    silu,
    swiglu_gemm,
    topk_softmax,
    moe_block_forward,
    moe_forward,
    bf16_bits_to_f64,
    gemm_bf16,
    rel_l2,
)
