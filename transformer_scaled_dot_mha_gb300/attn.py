"""Python binding of libattn_gb300.so: the C entry points of include/attn_gb300.h
under the same names, plus tensor-shaped wrappers.

This module only marshals arguments (tensor shapes, data pointers, the current
CUDA stream) and turns status codes into exceptions; every step of the
attention computation runs in the library's kernels. There is no fallback: if
the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_gb300.so")

ATTN_OK, ATTN_ERR_INVALID, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = 0, -1, -2, -3, -4
MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2
BWD_DETERMINISTIC = 1  # attn_bwd flag: the two-kernel schedule, bit-identical on every run

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (loaded once)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp]
        L.attn_fwd.restype = i
        L.attn_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
        L.attn_fwd_host_workspace_size.restype = ctypes.c_size_t
        L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, ctypes.c_size_t, vp]
        L.attn_fwd_host.restype = i
        L.attn_fwd_local.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp]
        L.attn_fwd_local.restype = i
        L.attn_fwd_f32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp]
        L.attn_fwd_f32.restype = i
        L.attn_decode_workspace_size.argtypes = [i, i, i, i, i]
        L.attn_decode_workspace_size.restype = ctypes.c_size_t
        L.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, ctypes.c_size_t, vp]
        L.attn_decode.restype = i
        L.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
        L.attn_decode_noalloc.restype = i
        L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
        L.attn_bwd_workspace_size.restype = ctypes.c_size_t
        L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i, vp,
                               ctypes.c_size_t, vp]
        L.attn_bwd.restype = i
        L.attn_bwd_local.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, i, vp,
                                     ctypes.c_size_t, vp]
        L.attn_bwd_local.restype = i
        L.attn_bwd_host_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.attn_bwd_host_workspace_size.restype = ctypes.c_size_t
        L.attn_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i, vp,
                                    ctypes.c_size_t, vp]
        L.attn_bwd_host.restype = i
        L.attn_weights.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp]
        L.attn_weights.restype = i
        L.attn_linear.argtypes = [vp, vp, vp, vp, i, i, i, vp]
        L.attn_linear.restype = i
        L.attn_mha_workspace_size.argtypes = [i, i, i, i, i, i]
        L.attn_mha_workspace_size.restype = ctypes.c_size_t
        L.attn_mha_fwd.argtypes = [vp] * 11 + [i, i, i, i, i, i, i, f, i, vp, vp, ctypes.c_size_t, vp]
        L.attn_mha_fwd.restype = i
        L.attn_fault_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint32)]
        L.attn_fault_status.restype = i
        L.attn_status_string.argtypes = [i]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_internal_arm_wait_timeout.argtypes = [ctypes.c_ulonglong, i]
        L.attn_internal_arm_wait_timeout.restype = None
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t, name, dtype, ndim=4):
    if t.dtype != dtype or t.dim() != ndim or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D CUDA {dtype} tensor, got {t.dtype} {tuple(t.shape)}")


def _call(fn, q, k, v, out, lse, scale, mask_mode, key_lens, stream, dtype, where):
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check(t, n, dtype)
    B, H, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    if k.shape != (B, H, n_k, d_k) or v.shape != (B, H, n_k, d_v) or out.shape != (B, H, n_q, d_v):
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)} out{tuple(out.shape)}")
    if lse is not None:
        _check(lse, "lse", torch.float32, 3)
        if lse.shape != (B, H, n_q):
            raise ValueError("lse must have shape [B, H, n_q]")
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, 1)
        if key_lens.shape != (B,):
            raise ValueError("key_lens must have shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, n_q, n_k, d_k, d_v, float(scale), int(mask_mode),
            _ptr(key_lens), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, where)
    return out


def attn_fwd(q, k, v, out, lse=None, scale=None, mask_mode=MASK_NONE, key_lens=None, stream=None):
    """bf16 forward into caller-provided ``out`` (and optional fp32 ``lse``)."""
    return _call(lib().attn_fwd, q, k, v, out, lse, scale, mask_mode, key_lens, stream, torch.bfloat16, "attn_fwd")


def attn_fwd_host_workspace_size(B, H, n_q, n_k, d, mask_mode=MASK_NONE) -> int:
    return int(lib().attn_fwd_host_workspace_size(B, H, n_q, n_k, d, int(mask_mode)))


def attn_fwd_host(q, k, v, out, workspace, lse=None, scale=None, mask_mode=MASK_NONE, key_lens=None, stream=None):
    """bf16 forward on HOST tensors (pinned recommended): q, k, v, key_lens are read
    and out, lse written in host memory; the chunked copy/compute pipeline runs on
    the GPU with ``workspace`` (a CUDA uint8 tensor of attn_fwd_host_workspace_size
    bytes) and is asynchronous on ``stream``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 4-D host bf16 tensor, got {t.dtype} {tuple(t.shape)}")
    B, H, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    if k.shape != (B, H, n_k, d_k) or v.shape != (B, H, n_k, d_v) or out.shape != (B, H, n_q, d_v):
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)} out{tuple(out.shape)}")
    if lse is not None and (lse.dtype != torch.float32 or lse.is_cuda or not lse.is_contiguous()
                            or lse.shape != (B, H, n_q)):
        raise ValueError("lse must be a contiguous host float32 tensor of shape [B, H, n_q]")
    if key_lens is not None and (key_lens.dtype != torch.int32 or key_lens.is_cuda or key_lens.shape != (B,)):
        raise ValueError("key_lens must be a host int32 tensor of shape [B]")
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    st = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, n_q, n_k, d_k, d_v,
                             float(scale), int(mask_mode), _ptr(key_lens), _ptr(workspace), workspace.numel(),
                             _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_host")
    return out


def attn_fwd_local(q, k, v, out, window, lse=None, scale=None, mask_mode=MASK_NONE, key_lens=None, stream=None):
    """Local-window (restricted) self-attention, bf16: key j is legal for query i only
    if |i - j| <= window (plus mask_mode)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check(t, n, torch.bfloat16)
    B, H, n, d_k = q.shape
    d_v = v.shape[3]
    if k.shape != (B, H, n, d_k) or v.shape != (B, H, n, d_v) or out.shape != (B, H, n, d_v):
        raise ValueError("local attention is self-attention: q, k, v, out must share B, H, n")
    if lse is not None:
        _check(lse, "lse", torch.float32, 3)
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, 1)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    st = lib().attn_fwd_local(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, n, d_k, d_v, float(scale),
                              int(window), int(mask_mode), _ptr(key_lens), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_local")
    return out


def attn_fwd_f32(q, k, v, out, lse=None, scale=None, mask_mode=MASK_NONE, key_lens=None, stream=None):
    """float32 forward into caller-provided ``out`` (and optional ``lse``)."""
    return _call(lib().attn_fwd_f32, q, k, v, out, lse, scale, mask_mode, key_lens, stream, torch.float32,
                 "attn_fwd_f32")


def attention(q, k, v, scale=None, mask_mode=MASK_NONE, key_lens=None, with_lse=False, stream=None):
    """Allocating convenience wrapper: returns ``out`` (and ``lse``) for bf16 or float32 inputs."""
    B, H, n_q, _ = q.shape
    out = torch.empty((B, H, n_q, v.shape[3]), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device) if with_lse else None
    fn = attn_fwd if q.dtype == torch.bfloat16 else attn_fwd_f32
    fn(q, k, v, out, lse, scale, mask_mode, key_lens, stream)
    return (out, lse) if with_lse else out


def attn_decode_workspace_size(B, H, n_q, n_max, d) -> int:
    return int(lib().attn_decode_workspace_size(B, H, n_q, n_max, d))


def attn_decode(q, k_cache, v_cache, out, cache_lens, workspace, lse=None, scale=None, stream=None):
    """One decoding step: ``q [B,H,n_q,d]`` against caches ``[B,H,n_max,d]`` (bf16),
    ``cache_lens`` int32 ``[B]``, caller-provided ``workspace`` (a CUDA uint8 tensor of
    at least ``attn_decode_workspace_size`` bytes) and ``out`` (and optional ``lse``)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _check(t, n, torch.bfloat16)
    B, H, n_q, d = q.shape
    n_max = k_cache.shape[2]
    if k_cache.shape != (B, H, n_max, d) or v_cache.shape != (B, H, n_max, d) or out.shape != q.shape:
        raise ValueError("shape mismatch between q, caches and out")
    _check(cache_lens, "cache_lens", torch.int32, 1)
    if lse is not None:
        _check(lse, "lse", torch.float32, 3)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, H, n_q, n_max, d,
                           float(scale), _ptr(cache_lens), _ptr(workspace), nbytes, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode")
    return out


NOALLOC_MAX_BYTES = 4 << 20  # ATTN_DECODE_NOALLOC_MAX_BYTES


def attn_decode_noalloc(q, k_cache, v_cache, out, cache_lens, lse=None, scale=None, stream=None):
    """attn_decode without a workspace argument, for callers that cannot allocate
    device memory (e.g. while capturing a CUDA graph): the library uses its own
    static device buffer of NOALLOC_MAX_BYTES, shared by every call on the device,
    so calls must not overlap on the GPU. The first call on a device does a
    one-time set-up and should come before any stream capture."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _check(t, n, torch.bfloat16)
    B, H, n_q, d = q.shape
    n_max = k_cache.shape[2]
    if k_cache.shape != (B, H, n_max, d) or v_cache.shape != (B, H, n_max, d) or out.shape != q.shape:
        raise ValueError("shape mismatch between q, caches and out")
    _check(cache_lens, "cache_lens", torch.int32, 1)
    if lse is not None:
        _check(lse, "lse", torch.float32, 3)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, H, n_q, n_max,
                                   d, float(scale), _ptr(cache_lens), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode_noalloc")
    return out


def attn_bwd_workspace_size(B, H, n_q, d=64, flags=0) -> int:
    return int(lib().attn_bwd_workspace_size(B, H, n_q, d, int(flags)))


def attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, workspace, scale=None, mask_mode=MASK_NONE, key_lens=None,
             stream=None, flags=0):
    """Gradients of attn_fwd into caller-provided ``dq``, ``dk``, ``dv`` (bf16, shaped like
    q, k, v), given ``dout`` and the forward's ``out`` and fp32 ``lse``; ``workspace`` is a
    CUDA tensor of at least ``attn_bwd_workspace_size(B, H, n_q, d, flags)`` bytes;
    ``flags`` = BWD_DETERMINISTIC selects the bit-reproducible schedule."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16)
    B, H, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    if (k.shape != (B, H, n_k, d_k) or v.shape != (B, H, n_k, d_v) or out.shape != (B, H, n_q, d_v)
            or dout.shape != out.shape or dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape):
        raise ValueError("shape mismatch between q, k, v, out, dout and the gradients")
    _check(lse, "lse", torch.float32, 3)
    if lse.shape != (B, H, n_q):
        raise ValueError("lse must have shape [B, H, n_q]")
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, 1)
        if key_lens.shape != (B,):
            raise ValueError("key_lens must have shape [B]")
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, H, n_q, n_k, d_k, d_v, float(scale), int(mask_mode), _ptr(key_lens), int(flags),
                        _ptr(workspace), nbytes, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_local(q, k, v, out, dout, lse, dq, dk, dv, workspace, window, scale=None, mask_mode=MASK_NONE,
                   key_lens=None, stream=None, flags=0):
    """Gradients of attn_fwd_local (key j legal for query i only if |i - j| <= window, plus
    mask_mode); arguments and workspace as in attn_bwd, with n_q = n_k."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16)
    B, H, n, d_k = q.shape
    d_v = v.shape[3]
    if (k.shape != (B, H, n, d_k) or v.shape != (B, H, n, d_v) or out.shape != (B, H, n, d_v)
            or dout.shape != out.shape or dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape):
        raise ValueError("local attention is self-attention: q, k, v, out, dout and the gradients share B, H, n")
    _check(lse, "lse", torch.float32, 3)
    if lse.shape != (B, H, n):
        raise ValueError("lse must have shape [B, H, n]")
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, 1)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib().attn_bwd_local(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                              _ptr(dv), B, H, n, d_k, d_v, float(scale), int(window), int(mask_mode), _ptr(key_lens),
                              int(flags), _ptr(workspace), nbytes, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_local")
    return dq, dk, dv


def attn_bwd_host_workspace_size(B, H, n_q, n_k, d, mask_mode=MASK_NONE, flags=0) -> int:
    return int(lib().attn_bwd_host_workspace_size(B, H, n_q, n_k, d, int(mask_mode), int(flags)))


def attn_bwd_host(q, k, v, out, dout, lse, dq, dk, dv, workspace, scale=None, mask_mode=MASK_NONE, key_lens=None,
                  stream=None, flags=0):
    """attn_bwd on HOST tensors (pinned recommended): q, k, v, out, dout (bf16), lse
    (float32) and key_lens are read and dq, dk, dv written in host memory; the chunked
    copy/compute pipeline runs on the GPU with ``workspace`` (a CUDA uint8 tensor of
    attn_bwd_host_workspace_size bytes) and is asynchronous on ``stream``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 4-D host bf16 tensor, got {t.dtype} {tuple(t.shape)}")
    B, H, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    if (k.shape != (B, H, n_k, d_k) or v.shape != (B, H, n_k, d_v) or out.shape != (B, H, n_q, d_v)
            or dout.shape != out.shape or dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape):
        raise ValueError("shape mismatch between q, k, v, out, dout and the gradients")
    if lse.dtype != torch.float32 or lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, n_q):
        raise ValueError("lse must be a contiguous host float32 tensor of shape [B, H, n_q]")
    if key_lens is not None and (key_lens.dtype != torch.int32 or key_lens.is_cuda or key_lens.shape != (B,)):
        raise ValueError("key_lens must be a host int32 tensor of shape [B]")
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    st = lib().attn_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                             _ptr(dv), B, H, n_q, n_k, d_k, d_v, float(scale), int(mask_mode), _ptr(key_lens),
                             int(flags), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_host")
    return dq, dk, dv


def attn_mha_workspace_size(B, n_q, n_k, d_model, H, d) -> int:
    return int(lib().attn_mha_workspace_size(B, n_q, n_k, d_model, H, d))


def attn_mha_fwd(x_q, x_kv, w_q, w_k, w_v, w_o, out, H, workspace, b_q=None, b_k=None, b_v=None, b_o=None,
                 scale=None, mask_mode=MASK_NONE, key_lens=None, stream=None):
    """Multi-head attention layer into caller-provided ``out [B, n_q, d_model]`` (bf16):
    ``x_q [B,n_q,d_model]``, ``x_kv [B,n_k,d_model]``, ``w_q, w_k, w_v [d_model, H*d]``,
    ``w_o [H*d, d_model]`` (the paper's x W orientation), optional biases, and a CUDA
    ``workspace`` of at least ``attn_mha_workspace_size`` bytes."""
    for t, n in ((x_q, "x_q"), (x_kv, "x_kv"), (out, "out")):
        _check(t, n, torch.bfloat16, 3)
    for t, n in ((w_q, "w_q"), (w_k, "w_k"), (w_v, "w_v"), (w_o, "w_o")):
        _check(t, n, torch.bfloat16, 2)
    for t, n in ((b_q, "b_q"), (b_k, "b_k"), (b_v, "b_v"), (b_o, "b_o")):
        if t is not None:
            _check(t, n, torch.bfloat16, 1)
    B, n_q, d_model = x_q.shape
    n_k = x_kv.shape[1]
    d_k, d_v = w_q.shape[1] // H, w_v.shape[1] // H
    if (x_kv.shape != (B, n_k, d_model) or w_q.shape != (d_model, H * d_k) or w_k.shape != w_q.shape
            or w_v.shape != (d_model, H * d_v) or w_o.shape != (H * d_v, d_model) or out.shape != x_q.shape):
        raise ValueError("inconsistent multi-head attention shapes")
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, 1)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib().attn_mha_fwd(_ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(b_q), _ptr(w_k), _ptr(b_k), _ptr(w_v), _ptr(b_v),
                            _ptr(w_o), _ptr(b_o), _ptr(out), B, n_q, n_k, d_model, H, d_k, d_v, float(scale),
                            int(mask_mode), _ptr(key_lens), _ptr(workspace), nbytes, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_mha_fwd")
    return out


def attn_weights(q, k, lse, w, scale=None, mask_mode=MASK_NONE, key_lens=None, stream=None):
    """The softmax weights ``w [B, H, n_q, n_k]`` (float32, caller-provided) of bf16
    ``q``, ``k`` given the ``lse`` attn_fwd returned for the same inputs and mask."""
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16)
    _check(lse, "lse", torch.float32, 3)
    _check(w, "w", torch.float32)
    B, H, n_q, d = q.shape
    n_k = k.shape[2]
    if k.shape != (B, H, n_k, d) or lse.shape != (B, H, n_q) or w.shape != (B, H, n_q, n_k):
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} lse{tuple(lse.shape)} w{tuple(w.shape)}")
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, 1)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_weights(_ptr(q), _ptr(k), _ptr(lse), _ptr(w), B, H, n_q, n_k, d, float(scale), int(mask_mode),
                            _ptr(key_lens), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_weights")
    return w


def attn_linear(x, w, y, bias=None, stream=None):
    """One projection ``y [M, N] = x [M, K] w [K, N] + bias [N]`` (bf16, row-major,
    caller-provided ``y``)."""
    _check(x, "x", torch.bfloat16, 2)
    _check(w, "w", torch.bfloat16, 2)
    _check(y, "y", torch.bfloat16, 2)
    if bias is not None:
        _check(bias, "bias", torch.bfloat16, 1)
    M, K = x.shape
    N = w.shape[1]
    if w.shape != (K, N) or y.shape != (M, N) or (bias is not None and bias.shape != (N,)):
        raise ValueError(f"shape mismatch: x{tuple(x.shape)} w{tuple(w.shape)} y{tuple(y.shape)}")
    st = lib().attn_linear(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), M, N, K, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_linear")
    return y


def _internal_arm_wait_timeout(wait_ns: int, skip_v_tile: int) -> None:
    """Test hook (not part of the C ABI header): the next plain d = 64 forward launch
    made on this host thread gives up its waits after ``wait_ns`` and never copies the
    V tile of K/V tile ``skip_v_tile``, so it ends through the bounded-wait abort path."""
    lib().attn_internal_arm_wait_timeout(int(wait_ns), int(skip_v_tile))


def attn_fault_status(stream=None, clear=True):
    """(status, raw fault bits) after synchronising ``stream``."""
    code = ctypes.c_uint32(0)
    st = lib().attn_fault_status(_stream_handle(stream), int(clear), ctypes.byref(code))
    return st, code.value
