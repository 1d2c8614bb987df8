"""Seeded synthetic inputs for attention workloads.

This module holds no attention arithmetic: it only names the workload shapes and
draws their inputs, so both the CUDA path and the fp64 oracle are fed from it.

Recipe (the same for every workload):
  * generator: numpy PCG64 seeded with ``20170612 + index`` of the workload;
  * Q, K, V: standard normal float32 draws in that order, times ``input_scale``;
    bf16 workloads round them to bf16 with round-to-nearest-even (bit patterns
    kept as uint16); float32 workloads keep them as drawn;
  * key lengths (key-padding and decode workloads): integers drawn uniformly from
    the inclusive range ``key_len_range`` after V (for decode, the cache length).

Shapes follow the pages' base and big Transformer sizes (d_model 512 with h = 8,
d_model 1024 with h = 16, so d_k = d_v = 64 per head; vlmlib.cn summary,
"multi-head attention"; transformer_lab, section 04) and the three uses of
attention (rockcohen.cc, section 5.3).
"""
from __future__ import annotations

from dataclasses import dataclass
import math

import numpy as np

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_DECODE, MASK_WINDOW = 0, 1, 2, 4, 8
SEED_BASE = 20170612


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n_q: int
    n_k: int
    d_k: int
    d_v: int
    dtype: str  # "f32" or "bf16"
    mask_mode: int
    key_len_range: tuple | None = None
    input_scale: float = 1.0
    index: int = 0
    window: int = -1  # local-window radius (MASK_WINDOW), -1 for none

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def scale(self) -> float:
        """1/sqrt(d_k), computed in double and rounded to float32."""
        return default_scale(self.d_k)

    def legal_pairs(self, key_lens=None) -> int:
        """Number of legal (query, key) pairs over all heads."""
        if self.mask_mode & MASK_WINDOW:
            return legal_pairs_window(self.B, self.H, self.n_q, self.mask_mode, self.window, key_lens)
        return legal_pairs(self.B, self.H, self.n_q, self.n_k, self.mask_mode, key_lens)

    def algorithmic_flops(self, key_lens=None) -> float:
        """2 (d_k + d_v) FLOPs per legal pair: a d_k-long dot product and a d_v-long axpy."""
        return 2.0 * (self.d_k + self.d_v) * self.legal_pairs(key_lens)

    def algorithmic_bwd_flops(self, key_lens=None) -> float:
        """Gradients: 2 (3 d_k + 2 d_v) FLOPs per legal pair -- the five products
        S = Q K^T (d_k), dP = dO V^T (d_v), dV = P^T dO (d_v), dK = dS^T Q and
        dQ = dS K (d_k each)."""
        return 2.0 * (3 * self.d_k + 2 * self.d_v) * self.legal_pairs(key_lens)

    def dense_flops(self) -> float:
        return 2.0 * (self.d_k + self.d_v) * self.B * self.H * self.n_q * self.n_k

    def algorithmic_bytes(self, key_lens=None) -> float:
        """Bytes a perfect kernel moves: Q, the K/V rows some query may use, O (bf16) and
        lse (fp32), each once."""
        rows_kv = 0
        for b in range(self.B):
            lim = self.n_k
            if self.mask_mode & (MASK_KEY_PADDING | MASK_DECODE):
                lim = min(lim, int(key_lens[b]))
            rows_kv += lim
        return float(self.H * (rows_kv * (self.d_k + self.d_v) * 2 +
                               self.B * self.n_q * (self.d_k * 2 + self.d_v * 2 + 4)))


def default_scale(d_k: int) -> float:
    return float(np.float32(1.0 / math.sqrt(d_k)))


def legal_pairs(B, H, n_q, n_k, mask_mode, key_lens=None) -> int:
    total = 0
    for b in range(B):
        lim = n_k
        if mask_mode & MASK_KEY_PADDING:
            lim = min(lim, int(key_lens[b]))
        if mask_mode & MASK_DECODE:
            # query i sits at position len - n_q + i and sees keys 0..position
            L = min(int(key_lens[b]), n_k)
            total += sum(max(0, L - n_q + i + 1) for i in range(n_q))
            continue
        if mask_mode & MASK_WINDOW:
            raise ValueError("use legal_pairs_window for local-window workloads")
        if mask_mode & MASK_CAUSAL:
            # query i sees keys 0..min(i, lim-1)
            full = min(n_q, lim)  # rows whose causal limit i+1 <= lim
            total += full * (full + 1) // 2 + max(0, n_q - full) * lim
        else:
            total += n_q * lim
    return total * H


def legal_pairs_window(B, H, n, mask_mode, window, key_lens=None) -> int:
    """Legal pairs of local-window self-attention (query i sees |i - j| <= window)."""
    total = 0
    for b in range(B):
        lim = min(n, int(key_lens[b])) if mask_mode & MASK_KEY_PADDING else n
        for i in range(n):
            lo = max(0, i - window)
            hi = min(lim, i + 1 if mask_mode & MASK_CAUSAL else i + window + 1)
            total += max(0, hi - lo)
    return total * H


def _wl(index, name, B, H, n_q, n_k, d, dtype, mask, lens=None, scale=1.0, window=-1):
    return Workload(name, B, H, n_q, n_k, d, d, dtype, mask, lens, scale, index, window)


WORKLOADS = {w.name: w for w in [
    _wl(0, "tiny_f32_b1_h1_n16_d8", 1, 1, 16, 16, 8, "f32", MASK_NONE),
    _wl(1, "encoder_self_pad_b32_h8_n128_d64", 32, 8, 128, 128, 64, "bf16", MASK_KEY_PADDING, (64, 128)),
    _wl(2, "decoder_causal_b16_h8_n512_d64", 16, 8, 512, 512, 64, "bf16", MASK_CAUSAL),
    _wl(3, "cross_pad_b16_h16_q256_k512_d64", 16, 16, 256, 512, 64, "bf16", MASK_KEY_PADDING, (384, 512)),
    _wl(4, "long_causal_b2_h16_n8192_d64", 2, 16, 8192, 8192, 64, "bf16", MASK_CAUSAL, None, 0.5),
    _wl(5, "long_none_b2_h16_n8192_d64", 2, 16, 8192, 8192, 64, "bf16", MASK_NONE, None, 0.5),
    _wl(6, "long_causal_b2_h16_n8192_d128", 2, 16, 8192, 8192, 128, "bf16", MASK_CAUSAL, None, 0.5),
    _wl(7, "long_none_b2_h16_n8192_d128", 2, 16, 8192, 8192, 128, "bf16", MASK_NONE, None, 0.5),
    # one autoregressive decoding step (one new query) against a key/value cache
    _wl(8, "decode_b32_h8_q1_k2048_d64", 32, 8, 1, 2048, 64, "bf16", MASK_DECODE, (1024, 2048)),
    _wl(9, "decode_b16_h16_q1_k8192_d64", 16, 16, 1, 8192, 64, "bf16", MASK_DECODE, (4096, 8192)),
    # restricted self-attention: each position attends to a causal neighbourhood of 512
    _wl(10, "local_causal_b2_h16_n8192_d64_w511", 2, 16, 8192, 8192, 64, "bf16", MASK_CAUSAL | MASK_WINDOW, None,
        0.5, 511),
    # encoder-decoder attention at long lengths: 4096 decoder queries against 8192
    # encoder keys/values with right padding (the third use of attention, n_q != n_k)
    _wl(11, "long_cross_pad_b2_h16_q4096_k8192_d64", 2, 16, 4096, 8192, 64, "bf16", MASK_KEY_PADDING, (6144, 8192),
        0.5),
    _wl(12, "long_cross_pad_b2_h16_q4096_k8192_d128", 2, 16, 4096, 8192, 128, "bf16", MASK_KEY_PADDING,
        (6144, 8192), 0.5),
]}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def make_grad_output(w: Workload, seed: int | None = None, **shape) -> np.ndarray:
    """Draw dout, the gradient arriving at the attention output, [B, H, n_q, d_v]:
    standard normal float32 from PCG64 seeded with ``seed + 1`` (default: the
    workload's seed + 1), rounded to bf16 bits for bf16 workloads."""
    B, H = shape.get("B", w.B), shape.get("H", w.H)
    n_q, d_v = shape.get("n_q", w.n_q), shape.get("d_v", w.d_v)
    rng = np.random.Generator(np.random.PCG64((w.seed if seed is None else seed) + 1))
    x = rng.standard_normal((B, H, n_q, d_v), dtype=np.float32)
    return to_bf16_bits(x) if w.dtype == "bf16" else x


def make_mha_inputs(w: Workload, seed: int | None = None, d_model: int | None = None, bias: bool = True, **shape):
    """Draw a multi-head layer's inputs for workload ``w`` (bf16 bits, uint16):
    x_q [B, n_q, d_model] and x_kv [B, n_k, d_model] standard normal; W^Q, W^K, W^V
    [d_model, H*d] and W^O [H*d, d_model] normal with variance 1/(rows) so every
    projection has unit variance; biases normal x 0.1 (None when ``bias`` is False);
    then key lengths as in ``make_inputs``. PCG64 seeded with ``seed + 2`` (default
    the workload's seed + 2); d_model defaults to H*d (the pages' d_model = h d_k)."""
    B, H = shape.get("B", w.B), shape.get("H", w.H)
    n_q, n_k, d = shape.get("n_q", w.n_q), shape.get("n_k", w.n_k), shape.get("d_k", w.d_k)
    d_model = H * d if d_model is None else d_model
    rng = np.random.Generator(np.random.PCG64((w.seed if seed is None else seed) + 2))
    nrm = lambda shp, sc=1.0: to_bf16_bits(rng.standard_normal(shp, dtype=np.float32) * np.float32(sc))
    x_q, x_kv = nrm((B, n_q, d_model)), nrm((B, n_k, d_model))
    w_q, w_k, w_v = (nrm((d_model, H * d), 1 / math.sqrt(d_model)) for _ in range(3))
    w_o = nrm((H * d, d_model), 1 / math.sqrt(H * d))
    biases = [nrm((H * d,), 0.1) for _ in range(3)] + [nrm((d_model,), 0.1)] if bias else [None] * 4
    if w.mask_mode & MASK_KEY_PADDING:
        lo, hi = w.key_len_range
        key_lens = rng.integers(min(lo, n_k), min(hi, n_k), size=B, endpoint=True).astype(np.int32)
    else:
        key_lens = np.full((B,), n_k, np.int32)
    return {"x_q": x_q, "x_kv": x_kv, "w_q": w_q, "w_k": w_k, "w_v": w_v, "w_o": w_o, "b_q": biases[0],
            "b_k": biases[1], "b_v": biases[2], "b_o": biases[3], "key_lens": key_lens, "H": H, "d": d,
            "d_model": d_model}


def make_inputs(w: Workload, seed: int | None = None, **shape):
    """Draw (q, k, v, key_lens) for a workload.

    ``shape`` may override B, H, n_q, n_k, d_k, d_v (for reduced parity cases of
    the same recipe). Returns numpy arrays: uint16 bf16 bits or float32, and an
    int32 ``key_lens`` of shape [B] (all n_k when the workload has no padding).
    """
    B, H = shape.get("B", w.B), shape.get("H", w.H)
    n_q, n_k = shape.get("n_q", w.n_q), shape.get("n_k", w.n_k)
    d_k, d_v = shape.get("d_k", w.d_k), shape.get("d_v", w.d_v)
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    arrs = []
    for shp in ((B, H, n_q, d_k), (B, H, n_k, d_k), (B, H, n_k, d_v)):
        x = rng.standard_normal(shp, dtype=np.float32)
        if w.input_scale != 1.0:
            x *= np.float32(w.input_scale)
        arrs.append(to_bf16_bits(x) if w.dtype == "bf16" else x)
    if w.mask_mode & (MASK_KEY_PADDING | MASK_DECODE):
        lo, hi = w.key_len_range
        lo, hi = min(lo, n_k), min(hi, n_k)
        key_lens = rng.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    else:
        key_lens = np.full((B,), n_k, np.int32)
    return arrs[0], arrs[1], arrs[2], key_lens
