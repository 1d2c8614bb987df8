"""Host-side logic of the input recipe and the FLOP accounting (no GPU)."""
import numpy as np
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import workloads as W


def test_bf16_rounding_matches_torch():
    x = np.random.Generator(np.random.PCG64(5)).standard_normal(100000, dtype=np.float32) * 7
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]  # ties to even
    ours = W.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_inputs_are_deterministic_and_shaped():
    w = W.WORKLOADS["cross_pad_b16_h16_q256_k512_d64"]
    a = W.make_inputs(w, B=2, H=3, n_q=5, n_k=7)
    b = W.make_inputs(w, B=2, H=3, n_q=5, n_k=7)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    q, k, v, kl = a
    assert q.shape == (2, 3, 5, 64) and k.shape == (2, 3, 7, 64) and v.shape == (2, 3, 7, 64)
    assert q.dtype == np.uint16 and kl.dtype == np.int32 and np.all((kl >= 1) & (kl <= 7))
    q, k, v, kl = W.make_inputs(w)
    assert np.all((kl >= 384) & (kl <= 512))
    # N(0,1) draws survive the bf16 rounding
    xs = oracle.widen(q)
    assert abs(xs.mean()) < 0.01 and abs(xs.std() - 1.0) < 0.01


def test_long_inputs_are_scaled_by_half():
    w = W.WORKLOADS["long_causal_b2_h16_n8192_d64"]
    q, _, _, _ = W.make_inputs(w, B=1, H=1, n_q=4096, n_k=8)
    assert abs(oracle.widen(q).std() - 0.5) < 0.01


def test_legal_pairs_brute_force():
    rng = np.random.Generator(np.random.PCG64(9))
    for mode in (0, 1, 2, 3):
        for n_q, n_k in ((7, 7), (5, 9), (9, 5), (16, 16)):
            if mode & 1 and n_q != n_k:
                continue
            kl = rng.integers(0, n_k, size=3, endpoint=True)
            want = int(oracle.legal_mask(3, n_q, n_k, mode, kl).sum()) * 2
            assert W.legal_pairs(3, 2, n_q, n_k, mode, kl) == want


def test_scale_is_float32_of_inverse_sqrt():
    assert W.default_scale(64) == 0.125
    assert W.default_scale(128) == float(np.float32(1 / np.sqrt(128.0)))


def test_decode_legal_pairs_and_bytes():
    w = W.WORKLOADS["decode_b16_h16_q1_k8192_d64"]
    q, k, v, kl = W.make_inputs(w, B=3, H=2)
    assert q.shape == (3, 2, 1, 64) and k.shape == (3, 2, 8192, 64)
    assert np.all((kl >= 4096) & (kl <= 8192))
    want = int(oracle.legal_mask(3, 1, 8192, oracle.MASK_DECODE, kl).sum()) * 2
    assert W.legal_pairs(3, 2, 1, 8192, W.MASK_DECODE, kl) == want
    kl2 = np.array([0, 2, 9], np.int32)
    for n_q in (1, 3, 5):
        want = int(oracle.legal_mask(3, n_q, 9, oracle.MASK_DECODE, kl2).sum())
        assert W.legal_pairs(3, 1, n_q, 9, W.MASK_DECODE, kl2) == want


def test_window_legal_pairs():
    kl = np.array([9, 5], np.int32)
    for mode in (W.MASK_WINDOW, W.MASK_WINDOW | W.MASK_CAUSAL, W.MASK_WINDOW | W.MASK_KEY_PADDING):
        for r in (0, 2, 20):
            want = int(oracle.legal_mask(2, 9, 9, mode, kl, window=r).sum()) * 3
            assert W.legal_pairs_window(2, 3, 9, mode, r, kl) == want
