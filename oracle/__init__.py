"""fp64 CPU oracle for scaled dot-product attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The CUDA library never links, loads or
calls it, and it imports nothing from the CUDA package: the two share no code.

Two formulations of Eq. (1), ``Attention(Q,K,V) = softmax(QK^T/sqrt(d_k)) V``
("Attention Is All You Need", rockcohen.cc, section 5.1; vlmlib.cn summary,
"scaled dot-product attention"):

* ``Oracle.attention`` / ``attention_rows`` / ``attention_weights`` -- the loop
  form in plain C (``attn_oracle.c``), fp64, one query row at a time;
* ``attention_matrix_form`` -- the matrix form in numpy/scipy: the whole score
  matrix, ``-inf`` at illegal entries (rockcohen.cc sections 5.3 and 6.3), a
  library row softmax, then a matmul with V.

The two must agree to 1e-12 (the loop-versus-matrix check of rockcohen.cc
section 10.2, assertion P0a). Inputs may be float64, float32, or bf16 given as
raw uint16 bit patterns; all are widened exactly to float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_DECODE, MASK_WINDOW = 0, 1, 2, 4, 8
_DTYPES = {np.dtype(np.float64): 0, np.dtype(np.float32): 1, np.dtype(np.uint16): 2}
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = SRC, out: str = LIB) -> str:
    """Compile the C oracle into a shared library (gcc, no GPU needed)."""
    cmd = ["gcc", *_CFLAGS, "-I", HERE, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def widen(x) -> np.ndarray:
    """Exact float64 copy of a float64/float32 array or of raw bf16 bits (uint16)."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


class Oracle:
    """ctypes front end of one compiled copy of ``attn_oracle.c``."""

    def __init__(self, path: str = LIB):
        if not os.path.exists(path):
            raise FileNotFoundError(f"oracle library {path} is not built; call oracle.build()")
        self.lib = ctypes.CDLL(path)
        vp, i, d, lp = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_longlong
        self.lib.oracle_attn.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, d, i, vp, i, vp, vp, i]
        self.lib.oracle_attn_rows.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, d, i, vp, i, lp, vp, vp, vp, i]
        self.lib.oracle_attn_weights.argtypes = [vp, vp, i, i, i, i, i, i, d, i, vp, i, vp]
        self.lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, d, i, vp, i, vp, vp, vp, i]
        self.lib.oracle_mha.argtypes = [vp, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, d, i, vp, vp,
                                        i]
        self.lib.oracle_linear.argtypes = [vp, vp, vp, i, i, i, i, vp]
        for f in (self.lib.oracle_attn, self.lib.oracle_attn_rows, self.lib.oracle_attn_weights,
                  self.lib.oracle_attn_bwd, self.lib.oracle_mha, self.lib.oracle_linear):
            f.restype = ctypes.c_int

    @staticmethod
    def _inputs(q, k, v):
        arrs = [np.ascontiguousarray(a) for a in (q, k) + ((v,) if v is not None else ())]
        dt = arrs[0].dtype
        if any(a.dtype != dt for a in arrs) or dt not in _DTYPES:
            raise TypeError(f"q/k/v must share one of float64/float32/uint16(bf16), got {[a.dtype for a in arrs]}")
        if any(a.ndim != 4 for a in arrs):
            raise ValueError("q, k, v must be 4-D [B, H, n, d]")
        return arrs, _DTYPES[dt]

    @staticmethod
    def _lens(mask_mode, key_lens, B):
        if not (mask_mode & (MASK_KEY_PADDING | MASK_DECODE)):
            return None
        kl = np.ascontiguousarray(key_lens, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_lens must have shape [B]")
        return kl

    @staticmethod
    def _threads(n_threads):
        return int(n_threads) if n_threads else (os.cpu_count() or 1)

    def attention(self, q, k, v, scale, mask_mode=MASK_NONE, key_lens=None, n_threads=None, window=0):
        """Full output ``O [B,H,n_q,d_v]`` and ``lse [B,H,n_q]`` in float64."""
        (q, k, v), dt = self._inputs(q, k, v)
        B, H, n_q, d_k = q.shape
        n_k, d_v = k.shape[2], v.shape[3]
        kl = self._lens(mask_mode, key_lens, B)
        out = np.empty((B, H, n_q, d_v), np.float64)
        lse = np.empty((B, H, n_q), np.float64)
        rc = self.lib.oracle_attn(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, B, H, n_q, n_k, d_k, d_v,
                                  float(scale), int(mask_mode), kl.ctypes.data if kl is not None else None,
                                  int(window), out.ctypes.data, lse.ctypes.data, self._threads(n_threads))
        if rc != 0:
            raise ValueError("oracle_attn rejected its arguments")
        return out, lse

    def attention_rows(self, q, k, v, scale, row_ids, mask_mode=MASK_NONE, key_lens=None, n_threads=None, window=0):
        """Output rows for flat row ids ``(b*H + h)*n_q + i``: ``(out [R,d_v], lse [R])``."""
        (q, k, v), dt = self._inputs(q, k, v)
        B, H, n_q, d_k = q.shape
        n_k, d_v = k.shape[2], v.shape[3]
        kl = self._lens(mask_mode, key_lens, B)
        ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        out = np.empty((ids.size, d_v), np.float64)
        lse = np.empty((ids.size,), np.float64)
        rc = self.lib.oracle_attn_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, B, H, n_q, n_k, d_k, d_v,
                                       float(scale), int(mask_mode), kl.ctypes.data if kl is not None else None,
                                       int(window), ids.size, ids.ctypes.data, out.ctypes.data, lse.ctypes.data,
                                       self._threads(n_threads))
        if rc != 0:
            raise ValueError("oracle_attn_rows rejected its arguments")
        return out, lse

    def attention_weights(self, q, k, scale, mask_mode=MASK_NONE, key_lens=None, window=0):
        """The softmax weight matrix ``A [B,H,n_q,n_k]`` (illegal entries exactly 0)."""
        (q, k), dt = self._inputs(q, k, None)
        B, H, n_q, d_k = q.shape
        n_k = k.shape[2]
        kl = self._lens(mask_mode, key_lens, B)
        w = np.empty((B, H, n_q, n_k), np.float64)
        rc = self.lib.oracle_attn_weights(q.ctypes.data, k.ctypes.data, dt, B, H, n_q, n_k, d_k, float(scale),
                                          int(mask_mode), kl.ctypes.data if kl is not None else None, int(window),
                                          w.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_attn_weights rejected its arguments")
        return w


    def attention_bwd(self, q, k, v, dout, scale, mask_mode=MASK_NONE, key_lens=None, window=0, n_threads=None):
        """Gradients ``(dq, dk, dv)`` of ``sum(dout * O)`` in float64."""
        (q, k, v, dout), dt = self._inputs4(q, k, v, dout)
        B, H, n_q, d_k = q.shape
        n_k, d_v = k.shape[2], v.shape[3]
        if dout.shape != (B, H, n_q, d_v):
            raise ValueError("dout must have the output's shape")
        kl = self._lens(mask_mode, key_lens, B)
        dq = np.empty((B, H, n_q, d_k), np.float64)
        dk = np.empty((B, H, n_k, d_k), np.float64)
        dv = np.empty((B, H, n_k, d_v), np.float64)
        rc = self.lib.oracle_attn_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, dt, B, H, n_q,
                                      n_k, d_k, d_v, float(scale), int(mask_mode),
                                      kl.ctypes.data if kl is not None else None, int(window), dq.ctypes.data,
                                      dk.ctypes.data, dv.ctypes.data, self._threads(n_threads))
        if rc != 0:
            raise ValueError("oracle_attn_bwd rejected its arguments")
        return dq, dk, dv

    def mha(self, x_q, x_kv, w_q, w_k, w_v, w_o, H, scale=None, mask_mode=MASK_NONE, key_lens=None,
            b_q=None, b_k=None, b_v=None, b_o=None, n_threads=None):
        """Multi-head attention ``Y [B, n_q, d_model]`` in float64 (``oracle_mha``).

        ``x_q [B,n_q,d_model]``, ``x_kv [B,n_k,d_model]``; ``w_q, w_k [d_model, H*d_k]``,
        ``w_v [d_model, H*d_v]``, ``w_o [H*d_v, d_model]`` (the paper's ``x W``
        orientation); biases optional. All arrays share one dtype. ``scale``
        defaults to 1/sqrt(d_k) rounded to float32, as the CUDA path uses it."""
        arrs = [np.ascontiguousarray(a) for a in (x_q, x_kv, w_q, w_k, w_v, w_o)]
        bias = [None if b is None else np.ascontiguousarray(b) for b in (b_q, b_k, b_v, b_o)]
        dt = arrs[0].dtype
        if any(a.dtype != dt for a in arrs + [b for b in bias if b is not None]) or dt not in _DTYPES:
            raise TypeError("inputs, weights and biases must share one of float64/float32/uint16(bf16)")
        x_q, x_kv, w_q, w_k, w_v, w_o = arrs
        B, n_q, d_model = x_q.shape
        n_k = x_kv.shape[1]
        d_k, d_v = w_q.shape[1] // H, w_v.shape[1] // H
        if (x_kv.shape != (B, n_k, d_model) or w_q.shape != (d_model, H * d_k) or w_k.shape != w_q.shape
                or w_v.shape != (d_model, H * d_v) or w_o.shape != (H * d_v, d_model)):
            raise ValueError("inconsistent multi-head attention shapes")
        for b, n in zip(bias, (H * d_k, H * d_k, H * d_v, d_model)):
            if b is not None and b.shape != (n,):
                raise ValueError("bias shapes must be [H*d_k], [H*d_k], [H*d_v], [d_model]")
        if scale is None:
            scale = float(np.float32(1.0 / np.sqrt(d_k)))
        kl = self._lens(mask_mode, key_lens, B)
        y = np.empty((B, n_q, d_model), np.float64)
        ptr = lambda a: None if a is None else a.ctypes.data
        rc = self.lib.oracle_mha(x_q.ctypes.data, x_kv.ctypes.data, _DTYPES[dt], w_q.ctypes.data, ptr(bias[0]),
                                 w_k.ctypes.data, ptr(bias[1]), w_v.ctypes.data, ptr(bias[2]), w_o.ctypes.data,
                                 ptr(bias[3]), B, n_q, n_k, d_model, H, d_k, d_v, float(scale), int(mask_mode),
                                 ptr(kl), y.ctypes.data, self._threads(n_threads))
        if rc != 0:
            raise ValueError("oracle_mha rejected its arguments")
        return y

    def linear(self, x, w, b=None):
        """One projection ``y [M, N] = x [M, K] w [K, N] + b [N]`` in float64
        (``oracle_linear``); x, w and b share one dtype (float64, float32 or bf16 bits)."""
        x, w = np.ascontiguousarray(x), np.ascontiguousarray(w)
        b = None if b is None else np.ascontiguousarray(b)
        dt = x.dtype
        if w.dtype != dt or (b is not None and b.dtype != dt) or dt not in _DTYPES:
            raise TypeError("x, w and b must share one of float64/float32/uint16(bf16)")
        M, K = x.shape
        N = w.shape[1]
        if w.shape != (K, N) or (b is not None and b.shape != (N,)):
            raise ValueError("shapes must be x [M, K], w [K, N], b [N]")
        y = np.empty((M, N), np.float64)
        rc = self.lib.oracle_linear(x.ctypes.data, w.ctypes.data, None if b is None else b.ctypes.data, _DTYPES[dt],
                                    M, N, K, y.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_linear rejected its arguments")
        return y

    @staticmethod
    def _inputs4(q, k, v, dout):
        (q, k, v), dt = Oracle._inputs(q, k, v)
        dout = np.ascontiguousarray(dout)
        if dout.dtype != q.dtype or dout.ndim != 4:
            raise TypeError("dout must be 4-D with the inputs' dtype")
        return (q, k, v, dout), dt


def legal_mask(B, n_q, n_k, mask_mode, key_lens=None, window=0) -> np.ndarray:
    """Boolean [B,1,n_q,n_k]: True where key j is a legal connection for query i."""
    i = np.arange(n_q)[:, None]
    j = np.arange(n_k)[None, :]
    ok = np.ones((B, 1, n_q, n_k), bool)
    if mask_mode & MASK_CAUSAL:
        ok &= (j <= i)[None, None]
    if mask_mode & MASK_KEY_PADDING:
        ok &= (j[None, None] < np.asarray(key_lens).reshape(B, 1, 1, 1))
    if mask_mode & MASK_DECODE:  # query i sits at position key_len - n_q + i
        pos = np.asarray(key_lens).reshape(B, 1, 1, 1) - n_q + i[None, None]
        ok &= (j[None, None] <= pos)
    if mask_mode & MASK_WINDOW:  # neighbourhood of radius `window`
        ok &= (np.abs(i - j) <= window)[None, None]
    return ok


def attention_matrix_form(q, k, v, scale, mask_mode=MASK_NONE, key_lens=None, window=0):
    """Matrix form of Eq. (1) in float64 with numpy/scipy library steps.

    S = scale * Q K^T; S = -inf where illegal; A = row softmax(S); O = A V;
    lse = row logsumexp(S). Rows with no legal key give O = 0, lse = -inf.
    """
    from scipy.special import logsumexp, softmax

    q, k, v = widen(q), widen(k), widen(v)
    B, H, n_q, _ = q.shape
    n_k = k.shape[2]
    S = scale * (q @ np.swapaxes(k, -1, -2))
    S = np.where(legal_mask(B, n_q, n_k, mask_mode, key_lens, window), S, -np.inf)
    empty = np.all(np.isneginf(S), axis=-1)
    S_safe = np.where(empty[..., None], 0.0, S)
    A = np.where(empty[..., None], 0.0, softmax(S_safe, axis=-1))
    lse = np.where(empty, -np.inf, logsumexp(S_safe, axis=-1))
    return A @ v, lse, A


def attention_bwd_matrix_form(q, k, v, dout, scale, mask_mode=MASK_NONE, key_lens=None, window=0):
    """Matrix form of the gradients of sum(dout * O), float64:
    dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(P * dP)), dQ = scale dS K,
    dK = scale dS^T Q, with P from ``attention_matrix_form``."""
    _, _, P = attention_matrix_form(q, k, v, scale, mask_mode, key_lens, window)
    q, k, v, dout = widen(q), widen(k), widen(v), widen(dout)
    dV = np.swapaxes(P, -1, -2) @ dout
    dP = dout @ np.swapaxes(v, -1, -2)
    dS = P * (dP - np.sum(P * dP, axis=-1, keepdims=True))
    return scale * (dS @ k), scale * (np.swapaxes(dS, -1, -2) @ q), dV
