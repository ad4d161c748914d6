"""GB300-native INT4 W4A16 group-32 GEMM library (libw4a16.so) and its Python binding.

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI (include/w4a16.h); this
package is a thin ctypes binding over it. The binding loads on first use of any of its names
(so that ``python -m int4_w4a16_group_gb300.build`` can run before the library exists); that
first use raises ImportError when the library has not been built.
"""
_EXPORTS = (
    "C", "GROUP", "LIB_PATH", "Registry", "W4A16Error", "bundle_info", "w4a16_abi_version",
    "w4a16_dequantize",
    "w4a16_device_error", "w4a16_gemm", "w4a16_gemm_bf16", "w4a16_gemm_swiglu",
    "w4a16_load_qw_sc", "w4a16_moe_block", "w4a16_moe_block_workspace_size", "w4a16_moe_gemm",
    "w4a16_moe_gemm_noalloc", "w4a16_moe_workspace_size", "w4a16_quantize", "w4a16_selftest_wait",
    "w4a16_status_string", "w4a16_topk_softmax",
)

__all__ = list(_EXPORTS)


def __getattr__(name):
    if name in _EXPORTS:
        from . import _abi
        return getattr(_abi, name)
    raise AttributeError(name)
