"""QMoE layer forward on GB300 (sm_103a): Python binding of the C ABI in include/qmoe.h.

Argument marshalling only. Every step of the forward runs in the CUDA kernels
of libqmoe.so; this module passes device pointers, sizes and the current torch
CUDA stream through ctypes. There is no CPU path: if the library is missing or
was not built for this machine, loading raises.

Functions mirror the C names:

* ``qmoe_workspace_bytes(problem) -> int``
* ``qmoe_forward(problem, x, router_logits, fc1_q, fc1_scales, fc1_zp, fc2_q,
  fc2_scales, fc2_zp, out, workspace, stream=None)``
* ``qmoe_forward_stages(problem, first_stage, last_stage, <qmoe_forward arguments>)``
* ``qmoe_route(problem, router_logits, topk_idx, topk_w, expert_offsets,
  sorted_route, workspace, stream=None)``
* ``qmoe_status_string(status) -> str``
* ``qmoe_workspace_error_offset(problem) -> int``

Tensor arguments may be torch CUDA tensors or raw integer device addresses;
``None`` passes NULL. A non-OK status raises :class:`QMoEError`.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmoe.so")

QMOE_BF16 = 0
QMOE_FP16 = 1

QMOE_OK = 0
QMOE_ERR_INVALID_ARGUMENT = 1
QMOE_ERR_UNSUPPORTED = 2
QMOE_ERR_MISALIGNED = 3
QMOE_ERR_WORKSPACE_TOO_SMALL = 4
QMOE_ERR_CUDA = 5

QMOE_PATH_AUTO = 0
QMOE_PATH_DECODE = 1
QMOE_PATH_GROUPED = 2
QMOE_PATH_GROUPED_ROUTE_TILES = 3
QMOE_PATH_GROUPED_WS = 4
QMOE_FORMAT_INT = 0
QMOE_FORMAT_MXFP4 = 1
QMOE_FORMAT_NVFP4 = 2

# every symbol the header declares
EXPORTED = ("qmoe_workspace_bytes", "qmoe_forward", "qmoe_forward_stages", "qmoe_route",
            "qmoe_status_string", "qmoe_forward_decode_static", "qmoe_forward_ex",
            "qmoe_workspace_error_offset", "qmoe_router_logits")

QMOE_STATIC_WORKSPACE_BYTES = 8 << 20

QMOE_STAGE_ROUTE = 0
QMOE_STAGE_FC1 = 1
QMOE_STAGE_FC2 = 2
QMOE_STAGE_COMBINE = 3


class QMoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {qmoe_status_string(status)} (status {status})")
        self.status = status


class qmoe_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("path", ctypes.c_int32), ("format", ctypes.c_int32)]


class qmoe_options(ctypes.Structure):
    _fields_ = [("full_softmax", ctypes.c_int32), ("fc1_bias", ctypes.c_void_p), ("fc2_bias", ctypes.c_void_p),
                ("decode_layer_kernel", ctypes.c_int32), ("router_weight", ctypes.c_void_p),
                ("fc1_global_scale", ctypes.c_void_p), ("fc2_global_scale", ctypes.c_void_p)]


def problem(T, hidden, inter, num_experts, top_k, bits, block_size, dtype, path=QMOE_PATH_AUTO, fmt=0):
    return qmoe_problem(int(T), int(hidden), int(inter), int(num_experts), int(top_k), int(bits),
                        int(block_size), int(dtype), int(path), int(fmt))


_lib = None


def lib():
    """The loaded libqmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "quantized_mixture_experts_route_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp = ctypes.c_void_p
        P = ctypes.POINTER(qmoe_problem)
        L.qmoe_workspace_bytes.argtypes = [P]
        L.qmoe_workspace_bytes.restype = ctypes.c_size_t
        L.qmoe_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.qmoe_forward.restype = ctypes.c_int
        L.qmoe_forward_stages.argtypes = [P, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp,
                                          vp, vp, vp, ctypes.c_size_t, vp]
        L.qmoe_forward_stages.restype = ctypes.c_int
        L.qmoe_route.argtypes = [P, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.qmoe_route.restype = ctypes.c_int
        L.qmoe_forward_decode_static.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.qmoe_forward_decode_static.restype = ctypes.c_int
        L.qmoe_forward_ex.argtypes = [P, ctypes.POINTER(qmoe_options), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, vp]
        L.qmoe_forward_ex.restype = ctypes.c_int
        L.qmoe_router_logits.argtypes = [P, vp, vp, vp, vp]
        L.qmoe_router_logits.restype = ctypes.c_int
        L.qmoe_workspace_error_offset.argtypes = [P]
        L.qmoe_workspace_error_offset.restype = ctypes.c_size_t
        L.qmoe_status_string.argtypes = [ctypes.c_int]
        L.qmoe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _addr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensors are required (no CPU path)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _nbytes(t):
    if isinstance(t, int):
        raise ValueError("pass the workspace as a tensor, or use the raw entry points of lib()")
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def qmoe_status_string(status: int) -> str:
    return lib().qmoe_status_string(int(status)).decode()


def qmoe_workspace_bytes(p: qmoe_problem) -> int:
    return int(lib().qmoe_workspace_bytes(ctypes.byref(p)))


def qmoe_workspace_error_offset(p: qmoe_problem) -> int:
    """Byte offset of the workspace's int32 failure word (-1 for an invalid problem)."""
    v = int(lib().qmoe_workspace_error_offset(ctypes.byref(p)))
    return -1 if v == (1 << 64) - 1 else v


def qmoe_forward(p: qmoe_problem, x, router_logits, fc1_q, fc1_scales, fc1_zp, fc2_q, fc2_scales,
                 fc2_zp, out, workspace, stream=None) -> None:
    st = lib().qmoe_forward(ctypes.byref(p), _addr(x), _addr(router_logits), _addr(fc1_q),
                            _addr(fc1_scales), _addr(fc1_zp), _addr(fc2_q), _addr(fc2_scales),
                            _addr(fc2_zp), _addr(out), _addr(workspace),
                            _nbytes(workspace) if workspace is not None else 0, _stream(stream))
    if st != QMOE_OK:
        raise QMoEError(st, "qmoe_forward")


def qmoe_forward_ex(p: qmoe_problem, full_softmax: int, fc1_bias, fc2_bias, x, router_logits, fc1_q,
                    fc1_scales, fc1_zp, fc2_q, fc2_scales, fc2_zp, out, workspace, stream=None,
                    decode_layer_kernel: int = 0, router_weight=None, fc1_global_scale=None,
                    fc2_global_scale=None) -> None:
    opt = qmoe_options(int(full_softmax), _addr(fc1_bias), _addr(fc2_bias), int(decode_layer_kernel),
                       _addr(router_weight), _addr(fc1_global_scale), _addr(fc2_global_scale))
    st = lib().qmoe_forward_ex(ctypes.byref(p), ctypes.byref(opt), _addr(x), _addr(router_logits),
                               _addr(fc1_q), _addr(fc1_scales), _addr(fc1_zp), _addr(fc2_q),
                               _addr(fc2_scales), _addr(fc2_zp), _addr(out), _addr(workspace),
                               _nbytes(workspace) if workspace is not None else 0, _stream(stream))
    if st != QMOE_OK:
        raise QMoEError(st, "qmoe_forward_ex")


def qmoe_forward_decode_static(p: qmoe_problem, x, router_logits, fc1_q, fc1_scales, fc1_zp, fc2_q,
                               fc2_scales, fc2_zp, out, stream=None) -> None:
    """qmoe_forward on the decode path with the library's own fixed device workspace."""
    st = lib().qmoe_forward_decode_static(ctypes.byref(p), _addr(x), _addr(router_logits),
                                          _addr(fc1_q), _addr(fc1_scales), _addr(fc1_zp),
                                          _addr(fc2_q), _addr(fc2_scales), _addr(fc2_zp),
                                          _addr(out), _stream(stream))
    if st != QMOE_OK:
        raise QMoEError(st, "qmoe_forward_decode_static")


def qmoe_forward_stages(p: qmoe_problem, first_stage: int, last_stage: int, x, router_logits, fc1_q,
                        fc1_scales, fc1_zp, fc2_q, fc2_scales, fc2_zp, out, workspace,
                        stream=None) -> None:
    st = lib().qmoe_forward_stages(ctypes.byref(p), int(first_stage), int(last_stage), _addr(x),
                                   _addr(router_logits), _addr(fc1_q), _addr(fc1_scales),
                                   _addr(fc1_zp), _addr(fc2_q), _addr(fc2_scales), _addr(fc2_zp),
                                   _addr(out), _addr(workspace),
                                   _nbytes(workspace) if workspace is not None else 0,
                                   _stream(stream))
    if st != QMOE_OK:
        raise QMoEError(st, "qmoe_forward_stages")


def qmoe_router_logits(p: qmoe_problem, x, router_weight, logits, stream=None) -> None:
    """Router logits [T][E] = x [T][H] . router_weight [E][H]^T, rounded once to the dtype."""
    st = lib().qmoe_router_logits(ctypes.byref(p), _addr(x), _addr(router_weight), _addr(logits),
                                  _stream(stream))
    if st != QMOE_OK:
        raise QMoEError(st, "qmoe_router_logits")


def qmoe_route(p: qmoe_problem, router_logits, topk_idx, topk_w, expert_offsets, sorted_route,
               workspace, stream=None) -> None:
    st = lib().qmoe_route(ctypes.byref(p), _addr(router_logits), _addr(topk_idx), _addr(topk_w),
                          _addr(expert_offsets), _addr(sorted_route), _addr(workspace),
                          _nbytes(workspace) if workspace is not None else 0, _stream(stream))
    if st != QMOE_OK:
        raise QMoEError(st, "qmoe_route")
