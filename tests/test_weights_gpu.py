"""attn_weights (the softmax weight matrix of Eq. (1)) against the fp64 oracle's weights,
element by element, on the same bf16 inputs.

Bound: the GPU forms w = exp2(scale*log2(e) * s - lse*log2(e)) with s accumulated in
fp32 and lse taken from attn_fwd, whose lse the forward tests hold to 1e-3 of the
oracle's (natural log). An error e in the exponent's argument moves w by a factor
exp(e), so |w - w_ref| <= (exp(1e-3 + 1e-5) - 1) w_ref, 1e-5 covering the fp32 score,
the scale and exp2.approx (about 2^-22 relative). Illegal weights are exactly 0.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
C, P = W.MASK_CAUSAL, W.MASK_KEY_PADDING
REL = math.expm1(1e-3 + 1e-5)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.lib()
    yield
    st, code = attn.attn_fault_status()
    assert st == attn.ATTN_OK, f"kernel fault record {code:#x}"


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def gpu_weights(q, k, v, kl, scale, mode):
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    kld = torch.from_numpy(kl).cuda() if mode & P else None
    B, H, n_q, _ = q.shape
    n_k = k.shape[2]
    out = torch.empty((B, H, n_q, v.shape[3]), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device="cuda")
    attn.attn_fwd(qd, kd, vd, out, lse, scale, mode, kld)
    w = torch.full((B, H, n_q, n_k), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_weights(qd, kd, lse, w, scale, mode, kld)
    torch.cuda.synchronize()
    return w.cpu().numpy().astype(np.float64)


def check(w, ref):
    assert np.isfinite(w).all()
    illegal = ref == 0.0
    assert np.all(w[illegal] == 0.0), "a masked weight is not exactly 0"
    err = np.abs(w - ref)
    worst = (err[~illegal] / ref[~illegal]).max() if (~illegal).any() else 0.0
    assert worst <= REL, f"max relative error {worst:.3e} > {REL:.3e}"
    rows = ref.sum(axis=-1)
    got = w.sum(axis=-1)
    live = rows > 0
    assert np.all(np.abs(got[live] - 1.0) <= 2 * REL), "a row of weights does not sum to 1"
    assert np.all(got[~live] == 0.0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", [0, C, P, C | P])
def test_weights_self_attention_ragged(orc, d, mode):
    name = "long_none_b2_h16_n8192_d64" if d == 64 else "long_none_b2_h16_n8192_d128"
    w_ = W.WORKLOADS[name]
    q, k, v, kl = W.make_inputs(w_, 5100 + d + mode, B=2, H=2, n_q=300, n_k=300)
    if mode & P:
        kl = np.array([1, 217], np.int32)  # one key, and a length inside a tile
    check(gpu_weights(q, k, v, kl, w_.scale, mode), orc.attention_weights(q, k, w_.scale, mode, kl))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_q,n_k", [(200, 333), (1, 130), (129, 1), (128, 512)])
def test_weights_cross_attention(orc, d, n_q, n_k):
    name = "long_none_b2_h16_n8192_d64" if d == 64 else "long_none_b2_h16_n8192_d128"
    w_ = W.WORKLOADS[name]
    q, k, v, kl = W.make_inputs(w_, 5200 + d + n_q + n_k, B=1, H=3, n_q=n_q, n_k=n_k)
    for mode in (0, P):
        if mode & P:
            kl = np.array([max(1, n_k - 3)], np.int32)
        check(gpu_weights(q, k, v, kl, w_.scale, mode), orc.attention_weights(q, k, w_.scale, mode, kl))


def test_weights_key_length_zero_row(orc):
    """A batch entry with key length 0: every weight of its rows is 0."""
    w_ = W.WORKLOADS["long_none_b2_h16_n8192_d64"]
    q, k, v, _ = W.make_inputs(w_, 5300, B=2, H=1, n_q=140, n_k=140)
    kl = np.array([0, 140], np.int32)
    w = gpu_weights(q, k, v, kl, w_.scale, P)
    assert np.all(w[0] == 0.0)
    check(w, orc.attention_weights(q, k, w_.scale, P, kl))


def test_weights_multi_tile_causal(orc):
    """Several key tiles per row and the zero fill past the diagonal (n = 640)."""
    w_ = W.WORKLOADS["long_causal_b2_h16_n8192_d64"]
    q, k, v, kl = W.make_inputs(w_, 5400, B=1, H=2, n_q=640, n_k=640)
    check(gpu_weights(q, k, v, kl, w_.scale, C), orc.attention_weights(q, k, w_.scale, C))


def test_weights_guard_bands_and_determinism():
    w_ = W.WORKLOADS["long_none_b2_h16_n8192_d64"]
    q, k, v, kl = W.make_inputs(w_, 5500, B=1, H=2, n_q=130, n_k=258)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    out = torch.empty((1, 2, 130, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 2, 130), dtype=torch.float32, device="cuda")
    attn.attn_fwd(qd, kd, vd, out, lse, w_.scale, 0, None)
    n, pad = 2 * 130 * 258, 4096
    outs = []
    for _ in range(2):
        buf = torch.full((n + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
        w = buf[pad:pad + n].view(1, 2, 130, 258)
        attn.attn_weights(qd, kd, lse, w, w_.scale, 0, None)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -7.0) and torch.all(buf[pad + n:] == -7.0)
        outs.append(w.clone())
    assert torch.equal(outs[0], outs[1])


def test_weights_rejects_bad_arguments():
    q = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 16), dtype=torch.float32, device="cuda")
    w = torch.zeros((1, 1, 16, 16), dtype=torch.float32, device="cuda")
    L = attn.lib()
    p = attn._ptr
    assert L.attn_weights(p(q), p(k), None, p(w), 1, 1, 16, 16, 64, 0.125, 0, None, None) == attn.ATTN_ERR_INVALID
    assert L.attn_weights(p(q), p(k), p(lse), p(w), 1, 1, 16, 16, 96, 0.125, 0, None, None) == \
        attn.ATTN_ERR_UNSUPPORTED
    assert L.attn_weights(p(q), p(k), p(lse), p(w), 1, 1, 16, 8, 64, 0.125, C, None, None) == attn.ATTN_ERR_INVALID
    assert L.attn_weights(p(q), p(k), p(lse), p(w) + 4, 1, 1, 16, 16, 64, 0.125, 0, None, None) == \
        attn.ATTN_ERR_INVALID
