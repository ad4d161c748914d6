"""ctypes binding of libw4a16.so: one Python function per C entry point, same names.

Argument marshalling only: tensors are checked for device, dtype, shape and contiguity, their
device addresses and the current CUDA stream are passed to the C function, and a non-OK status
raises :class:`W4A16Error`. Every step of the computation runs in the library's kernels; there
is no Python or CPU fallback. Importing this module fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("W4A16_LIB", os.path.join(_HERE, "libw4a16.so"))

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libw4a16.so not found at {LIB_PATH}; build it first with "
        "`python -m int4_w4a16_group_gb300.build` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_s = ctypes.c_char_p

# name -> (restype, argtypes)
_SIGS = {
    "w4a16_status_string": (ctypes.c_char_p, [_i]),
    "w4a16_abi_version": (_i, []),
    "w4a16_last_cuda_error": (_i, []),
    "w4a16_quantize": (_i, [_p, _i, _i, _i, _p, _p, _p]),
    "w4a16_dequantize": (_i, [_p, _p, _i, _i, _i, _p, _p]),
    "w4a16_gemm": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _p]),
    "w4a16_gemm_swiglu": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _p]),
    "w4a16_gemm_bf16": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _p]),
    "w4a16_moe_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "w4a16_moe_gemm": (_i, [_p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _i, _i, _i, _p, _sz, _p]),
    "w4a16_moe_gemm_noalloc": (_i, [_p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "w4a16_moe_block_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "w4a16_bundle_info": (_i, [_s, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)]),
    "w4a16_bundle_load": (_i, [_p, _s, _p, _sz]),
    "w4a16_moe_block": (_i, [_p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _i, _p, _i, _i,
                             _i, _p, _sz, _p]),
    "w4a16_topk_softmax": (_i, [_p, _p, _i, _i, _p]),
    "w4a16_load_qw_sc": (_i, [_s, _s, _i, _i, _i, _p, _p]),
    "w4a16_registry_create": (_p, []),
    "w4a16_registry_destroy": (None, [_p]),
    "w4a16_registry_add": (_i, [_p, _s, _p, _p, _i, _i, _i]),
    "w4a16_registry_find": (_i, [_p, _s, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "w4a16_linear": (_i, [_p, _s, _p, _p, _i, _p]),
    "w4a16_linear_swiglu": (_i, [_p, _s, _p, _p, _i, _p]),
    "w4a16_device_error": (_i, [ctypes.POINTER(_i)]),
    "w4a16_selftest_wait": (_i, [_i, _i, _p]),
}

for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)  # AttributeError here = symbol missing from the library
    _f.restype = _res
    _f.argtypes = _args

C = _lib  # raw ctypes handle: the C ABI itself

GROUP = 32
STATUS = {0: "OK", 1: "ERR_ARG", 2: "ERR_ALIGN", 3: "ERR_UNSUPPORTED", 4: "ERR_WORKSPACE",
          5: "ERR_CUDA", 6: "ERR_NOT_FOUND", 7: "ERR_IO", 8: "ERR_TIMEOUT"}


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.w4a16_status_string(status).decode()
        if status == 5:
            msg += f" (cudaError {_lib.w4a16_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != 0:
        raise W4A16Error(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device: a tensor of another GPU would be read from
        # the wrong device's address space
        raise ValueError(f"{name}: on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


# ----------------------------------------------------------------------------- entry points

def w4a16_abi_version() -> int:
    return _lib.w4a16_abi_version()


def w4a16_status_string(status: int) -> str:
    return _lib.w4a16_status_string(status).decode()


def w4a16_quantize(W: torch.Tensor, qw: torch.Tensor | None = None, sc: torch.Tensor | None = None,
                   group: int = GROUP, stream=None):
    """W[K, N] float32 -> (qw[K/8, N] int32, sc[K/32, N] float32)."""
    K, N = W.shape
    if qw is None:
        qw = torch.empty((K // 8, N), dtype=torch.int32, device=W.device)
    if sc is None:
        sc = torch.empty((K // GROUP, N), dtype=torch.float32, device=W.device)
    _check(_lib.w4a16_quantize(_dev(W, torch.float32, "W"), K, N, group,
                               _dev(qw, torch.int32, "qw", (K // 8, N)),
                               _dev(sc, torch.float32, "sc", (K // GROUP, N)), _stream(stream)),
           "w4a16_quantize")
    return qw, sc


def w4a16_dequantize(qw: torch.Tensor, sc: torch.Tensor, W: torch.Tensor | None = None,
                     group: int = GROUP, stream=None):
    K8, N = qw.shape
    K = K8 * 8
    if W is None:
        W = torch.empty((K, N), dtype=torch.float32, device=qw.device)
    _check(_lib.w4a16_dequantize(_dev(qw, torch.int32, "qw"), _dev(sc, torch.float32, "sc", (K // GROUP, N)),
                                 K, N, group, _dev(W, torch.float32, "W", (K, N)), _stream(stream)),
           "w4a16_dequantize")
    return W


def w4a16_gemm(x: torch.Tensor, qw: torch.Tensor, sc: torch.Tensor, y: torch.Tensor | None = None,
               group: int = GROUP, stream=None):
    """y[M, N] = x[M, K] @ dequant(qw, sc)."""
    M, K = x.shape
    N = qw.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(_lib.w4a16_gemm(_dev(x, torch.float32, "x"), _dev(qw, torch.int32, "qw", (K // 8, N)),
                           _dev(sc, torch.float32, "sc", (K // GROUP, N)),
                           _dev(y, torch.float32, "y", (M, N)), M, N, K, group, _stream(stream)),
           "w4a16_gemm")
    return y


def w4a16_gemm_swiglu(x: torch.Tensor, qw_gu: torch.Tensor, sc_gu: torch.Tensor,
                      y: torch.Tensor | None = None, group: int = GROUP, stream=None):
    """y[M, N2/2] = silu(gate) * up, (gate | up) = x @ dequant(qw_gu, sc_gu)."""
    M, K = x.shape
    N2 = qw_gu.shape[1]
    if y is None:
        y = torch.empty((M, N2 // 2), dtype=torch.float32, device=x.device)
    _check(_lib.w4a16_gemm_swiglu(_dev(x, torch.float32, "x"),
                                  _dev(qw_gu, torch.int32, "qw_gu", (K // 8, N2)),
                                  _dev(sc_gu, torch.float32, "sc_gu", (K // GROUP, N2)),
                                  _dev(y, torch.float32, "y", (M, N2 // 2)), M, N2, K, group,
                                  _stream(stream)),
           "w4a16_gemm_swiglu")
    return y


def w4a16_gemm_bf16(x: torch.Tensor, qw: torch.Tensor, sc: torch.Tensor, y: torch.Tensor | None = None,
                    group: int = GROUP, stream=None):
    """y[M, N] bf16 = x[M, K] bf16 @ bf16(dequant(qw, sc)), float32 accumulation."""
    M, K = x.shape
    N = qw.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(_lib.w4a16_gemm_bf16(_dev(x, torch.bfloat16, "x"), _dev(qw, torch.int32, "qw", (K // 8, N)),
                                _dev(sc, torch.float32, "sc", (K // GROUP, N)),
                                _dev(y, torch.bfloat16, "y", (M, N)), M, N, K, group, _stream(stream)),
           "w4a16_gemm_bf16")
    return y


def w4a16_moe_workspace_size(T: int, topk: int, E: int, K: int, I: int) -> int:
    return int(_lib.w4a16_moe_workspace_size(T, topk, E, K, I))


def w4a16_moe_gemm(x, topk_ids, topk_w, qw_gu, sc_gu, qw_dn, sc_dn, out=None, workspace=None,
                   group: int = GROUP, stream=None):
    """Routed-expert MoE block; see w4a16.h. Returns out[T, K]."""
    T, K = x.shape
    topk = topk_ids.shape[1]
    E = qw_gu.shape[0]
    I = qw_gu.shape[2] // 2
    if out is None:
        out = torch.empty((T, K), dtype=torch.float32, device=x.device)
    need = w4a16_moe_workspace_size(T, topk, E, K, I)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(_lib.w4a16_moe_gemm(
        _dev(x, torch.float32, "x"), _dev(topk_ids, torch.int32, "topk_ids", (T, topk)),
        _dev(topk_w, torch.float32, "topk_w", (T, topk)), T, topk, E,
        _dev(qw_gu, torch.int32, "qw_gu", (E, K // 8, 2 * I)),
        _dev(sc_gu, torch.float32, "sc_gu", (E, K // GROUP, 2 * I)),
        _dev(qw_dn, torch.int32, "qw_dn", (E, I // 8, K)),
        _dev(sc_dn, torch.float32, "sc_dn", (E, I // GROUP, K)),
        _dev(out, torch.float32, "out", (T, K)), K, I, group,
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)),
        "w4a16_moe_gemm")
    return out


def w4a16_moe_block_workspace_size(T: int, topk: int, E: int, K: int, I: int, Is: int) -> int:
    return int(_lib.w4a16_moe_block_workspace_size(T, topk, E, K, I, Is))


def w4a16_moe_block(x, topk_ids, topk_w, qw_gu, sc_gu, qw_dn, sc_dn, qs_gu, ss_gu, qs_dn, ss_dn,
                    out=None, workspace=None, group: int = GROUP, stream=None):
    """MoE block with a shared expert; see w4a16.h. Returns out[T, K]."""
    T, K = x.shape
    topk = topk_ids.shape[1]
    E = qw_gu.shape[0]
    I = qw_gu.shape[2] // 2
    Is = qs_gu.shape[1] // 2
    if out is None:
        out = torch.empty((T, K), dtype=torch.float32, device=x.device)
    need = w4a16_moe_block_workspace_size(T, topk, E, K, I, Is)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(_lib.w4a16_moe_block(
        _dev(x, torch.float32, "x"), _dev(topk_ids, torch.int32, "topk_ids", (T, topk)),
        _dev(topk_w, torch.float32, "topk_w", (T, topk)), T, topk, E,
        _dev(qw_gu, torch.int32, "qw_gu", (E, K // 8, 2 * I)),
        _dev(sc_gu, torch.float32, "sc_gu", (E, K // GROUP, 2 * I)),
        _dev(qw_dn, torch.int32, "qw_dn", (E, I // 8, K)),
        _dev(sc_dn, torch.float32, "sc_dn", (E, I // GROUP, K)),
        _dev(qs_gu, torch.int32, "qs_gu", (K // 8, 2 * Is)),
        _dev(ss_gu, torch.float32, "ss_gu", (K // GROUP, 2 * Is)),
        _dev(qs_dn, torch.int32, "qs_dn", (Is // 8, K)),
        _dev(ss_dn, torch.float32, "ss_dn", (Is // GROUP, K)), Is,
        _dev(out, torch.float32, "out", (T, K)), K, I, group,
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)),
        "w4a16_moe_block")
    return out


def w4a16_moe_gemm_noalloc(x, topk_ids, topk_w, qw_gu, sc_gu, qw_dn, sc_dn, out=None,
                           group: int = GROUP, stream=None):
    """MoE block on the library's fixed device scratch (no workspace argument); see w4a16.h."""
    T, K = x.shape
    topk = topk_ids.shape[1]
    E = qw_gu.shape[0]
    I = qw_gu.shape[2] // 2
    if out is None:
        out = torch.empty((T, K), dtype=torch.float32, device=x.device)
    _check(_lib.w4a16_moe_gemm_noalloc(
        _dev(x, torch.float32, "x"), _dev(topk_ids, torch.int32, "topk_ids", (T, topk)),
        _dev(topk_w, torch.float32, "topk_w", (T, topk)), T, topk, E,
        _dev(qw_gu, torch.int32, "qw_gu", (E, K // 8, 2 * I)),
        _dev(sc_gu, torch.float32, "sc_gu", (E, K // GROUP, 2 * I)),
        _dev(qw_dn, torch.int32, "qw_dn", (E, I // 8, K)),
        _dev(sc_dn, torch.float32, "sc_dn", (E, I // GROUP, K)),
        _dev(out, torch.float32, "out", (T, K)), K, I, group, _stream(stream)),
        "w4a16_moe_gemm_noalloc")
    return out


def w4a16_topk_softmax(logits: torch.Tensor, weights: torch.Tensor | None = None, stream=None):
    T, topk = logits.shape
    if weights is None:
        weights = torch.empty_like(logits)
    _check(_lib.w4a16_topk_softmax(_dev(logits, torch.float32, "logits"),
                                   _dev(weights, torch.float32, "weights", (T, topk)), T, topk,
                                   _stream(stream)),
           "w4a16_topk_softmax")
    return weights


def w4a16_load_qw_sc(qw_path: str, sc_path: str, K: int, N: int, qw: torch.Tensor, sc: torch.Tensor,
                     group: int = GROUP):
    _check(_lib.w4a16_load_qw_sc(qw_path.encode(), sc_path.encode(), K, N, group,
                                 _dev(qw, torch.int32, "qw", (K // 8, N)),
                                 _dev(sc, torch.float32, "sc", (K // GROUP, N))),
           "w4a16_load_qw_sc")


def w4a16_device_error() -> int:
    code = ctypes.c_int(0)
    _check(_lib.w4a16_device_error(ctypes.byref(code)), "w4a16_device_error")
    return code.value


def w4a16_selftest_wait(arrive: bool, limit_us: int, stream=None) -> None:
    """Bounded-wait self-test kernel (see w4a16.h); read the result with w4a16_device_error()."""
    _check(_lib.w4a16_selftest_wait(int(bool(arrive)), int(limit_us), _stream(stream)),
           "w4a16_selftest_wait")


def bundle_info(path: str):
    """(number of tensors, device bytes needed) of a weight bundle (w4a16_bundle_info)."""
    count, nbytes = ctypes.c_int(0), ctypes.c_size_t(0)
    _check(_lib.w4a16_bundle_info(str(path).encode(), ctypes.byref(count), ctypes.byref(nbytes)),
           f"w4a16_bundle_info({path})")
    return count.value, nbytes.value


class Registry:
    """Name -> quantized weight map with linear() dispatch (w4a16_registry_* / w4a16_linear*).

    Keeps a reference to each registered tensor so its device memory outlives the entry."""

    def __init__(self):
        self._h = _lib.w4a16_registry_create()
        if not self._h:
            raise MemoryError("w4a16_registry_create failed")
        self._keep = {}

    def close(self):
        if self._h:
            _lib.w4a16_registry_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, name: str, qw: torch.Tensor, sc: torch.Tensor, group: int = GROUP):
        K8, N = qw.shape
        _check(_lib.w4a16_registry_add(self._h, name.encode(), _dev(qw, torch.int32, "qw"),
                                       _dev(sc, torch.float32, "sc", (K8 * 8 // GROUP, N)), K8 * 8, N,
                                       group), f"w4a16_registry_add({name})")
        self._keep[name] = (qw, sc)

    def load_bundle(self, path: str, device="cuda") -> torch.Tensor:
        """Loads every tensor of a weight bundle (w4a16_bundle_load) into one device arena and
        registers its names; returns the arena, which the registry also keeps alive."""
        arena = torch.empty(max(bundle_info(path)[1], 256), dtype=torch.uint8, device=device)
        _check(_lib.w4a16_bundle_load(self._h, str(path).encode(), arena.data_ptr(),
                                      arena.numel()), f"w4a16_bundle_load({path})")
        self._keep[("bundle", str(path))] = arena
        return arena

    def find(self, name: str):
        K, N = ctypes.c_int(0), ctypes.c_int(0)
        _check(_lib.w4a16_registry_find(self._h, name.encode(), ctypes.byref(K), ctypes.byref(N)),
               f"w4a16_registry_find({name})")
        return K.value, N.value

    def linear(self, name: str, x: torch.Tensor, y: torch.Tensor | None = None, stream=None):
        K, N = self.find(name)
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, N), dtype=torch.float32, device=x.device)
        _check(_lib.w4a16_linear(self._h, name.encode(), _dev(x, torch.float32, "x", (M, K)),
                                 _dev(y, torch.float32, "y", (M, N)), M, _stream(stream)),
               f"w4a16_linear({name})")
        return y

    def linear_swiglu(self, name: str, x: torch.Tensor, y: torch.Tensor | None = None, stream=None):
        K, N = self.find(name)
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, N // 2), dtype=torch.float32, device=x.device)
        _check(_lib.w4a16_linear_swiglu(self._h, name.encode(), _dev(x, torch.float32, "x", (M, K)),
                                        _dev(y, torch.float32, "y", (M, N // 2)), M, _stream(stream)),
               f"w4a16_linear_swiglu({name})")
        return y
