"""attn_bwd (dQ, dK, dV on the tensor cores) against the fp64 oracle's gradients,
element by element on the same bf16-rounded inputs.

The forward output and lse the gradients consume come from attn_fwd (as a training
step would use them); dout is a seeded bf16 draw.

Tolerance, derived per element from the arithmetic of the CUDA path (P = the exact
weights, |.| element-wise absolute values, u = 2^-8, twice the one-sided bound of
round-to-nearest bf16):
  * out is the bf16 forward result, off by at most u (P|V|) per element, so
    D_i = dout_i . out_i is off by dD_i <= u A_i with A_i = sum_d |dout_id| (P|V|)_id;
  * P and dS = P (dP - D) are rounded to bf16 before their products:
    |d P| <= u P,  |d dS| <= P dD + u |dS|;
  * each result is rounded to bf16 once: u |g|.
  bound(dV) = u P^T|dout| + u|dV|,  bound(dK) = scale |d dS|^T |Q| + u|dK|,
  bound(dQ) = scale |d dS| |K| + u|dQ|;  the test allows 2 x bound + 1e-6 (fp32
  accumulation and ex2.approx stay far below u).
"""
import numpy as np
import pytest
import torch

from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
U = 2.0 ** -8


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


def bits_to_f64(a):
    return (np.ascontiguousarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def draw(seed, B, H, n_q, n_k, d, mask, lens=None):
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, k, v, _ = W.make_inputs(w, seed=seed, B=B, H=H, n_q=n_q, n_k=n_k, d_k=d, d_v=d)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    dout = W.to_bf16_bits(rng.standard_normal((B, H, n_q, d), dtype=np.float32))
    if lens is None:
        lens = np.full((B,), n_k, np.int32)
    return q, k, v, dout, np.asarray(lens, np.int32)


def run_bwd(q, k, v, dout, scale, mask, lens):
    B, H, n_q, d = q.shape
    qd, kd, vd, gd = dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_bf16(dout)
    kl = torch.from_numpy(lens).cuda() if mask & W.MASK_KEY_PADDING else None
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device="cuda")
    attn.attn_fwd(qd, kd, vd, out, lse, scale, mask, kl)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, n_q), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.full_like(qd, float("nan")), torch.full_like(kd, float("nan")), torch.full_like(vd, float("nan"))
    attn.attn_bwd(qd, kd, vd, out, gd, lse, dq, dk, dv, ws, scale, mask, kl)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f(dq), f(dk), f(dv)


def bounds(orc, q, k, v, dout, scale, mask, lens, ref):
    """Element-wise error bounds of the CUDA path (module docstring)."""
    P = orc.attention_weights(q, k, scale, mask, lens)
    Q, K, V, G = (bits_to_f64(x) for x in (q, k, v, dout))
    dq_r, dk_r, dv_r = ref
    O = P @ V
    A = np.sum(np.abs(G) * (P @ np.abs(V)), axis=-1)
    dS = P * (G @ np.swapaxes(V, -1, -2) - np.sum(G * O, axis=-1)[..., None])
    ddS = P * (U * A)[..., None] + U * np.abs(dS)
    b_dv = U * (np.swapaxes(P, -1, -2) @ np.abs(G)) + U * np.abs(dv_r)
    b_dk = scale * (np.swapaxes(ddS, -1, -2) @ np.abs(Q)) + U * np.abs(dk_r)
    b_dq = scale * (ddS @ np.abs(K)) + U * np.abs(dq_r)
    return b_dq, b_dk, b_dv


def check(got, ref, bnd):
    for name, g, r, b in zip(("dq", "dk", "dv"), got, ref, bnd):
        assert np.isfinite(g).all(), f"{name} has non-finite values"
        err = np.abs(g - r)
        lim = 2.0 * b + 1e-6
        bad = err > lim
        assert not bad.any(), (f"{name}: {bad.sum()} of {bad.size} beyond bound; worst err "
                               f"{err[bad].max():.3e}, max err {err.max():.3e}")


def parity(orc, seed, B, H, n_q, n_k, d, mask, lens=None, scale=None):
    q, k, v, dout, lens = draw(seed, B, H, n_q, n_k, d, mask, lens)
    scale = W.default_scale(d) if scale is None else scale
    got = run_bwd(q, k, v, dout, scale, mask, lens)
    kl = lens if mask & W.MASK_KEY_PADDING else None
    ref = orc.attention_bwd(q, k, v, dout, scale, mask, kl)
    check(got, ref, bounds(orc, q, k, v, dout, scale, mask, kl, ref))
    return got, ref


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [W.MASK_NONE, W.MASK_CAUSAL])
@pytest.mark.parametrize("n", [1, 64, 128, 300, 513])
def test_bwd_self(orc, d, mask, n):
    parity(orc, 7000 + d + n + 3 * mask, 2, 2, n, n, d, mask)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [W.MASK_KEY_PADDING, W.MASK_CAUSAL | W.MASK_KEY_PADDING])
def test_bwd_key_padding(orc, d, mask):
    """Key lengths 0 (no legal key: zero gradients), 1, mid-tile and full."""
    n = 300
    parity(orc, 7100 + d + mask, 4, 2, n, n, d, mask, lens=[0, 1, 190, n])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_q,n_k", [(200, 333), (333, 200), (1, 257), (129, 1)])
def test_bwd_cross(orc, d, n_q, n_k):
    parity(orc, 7200 + d + n_q + n_k, 2, 3, n_q, n_k, d, W.MASK_KEY_PADDING, lens=[n_k, max(1, n_k // 2)])


def test_bwd_sharp_rows(orc):
    """A large scale makes rows nearly one-hot: P rounding and D cancellation at their worst."""
    parity(orc, 7300, 1, 2, 256, 256, 64, W.MASK_CAUSAL, scale=1.0)


def test_bwd_dead_keys_get_zero_gradient(orc):
    """Keys past the key length and keys no causal query sees have dk = dv = 0 exactly."""
    n = 260
    (dq, dk, dv), _ = parity(orc, 7400, 2, 1, n, n, 64, W.MASK_CAUSAL | W.MASK_KEY_PADDING, lens=[100, 0])
    assert np.all(dk[0, :, 100:] == 0) and np.all(dv[0, :, 100:] == 0)
    assert np.all(dk[1] == 0) and np.all(dv[1] == 0) and np.all(dq[1] == 0)


def test_bwd_deterministic():
    """No atomics: two calls give bit-identical gradients."""
    q, k, v, dout, lens = draw(7500, 2, 4, 700, 700, 64, W.MASK_CAUSAL)
    a = run_bwd(q, k, v, dout, W.default_scale(64), W.MASK_CAUSAL, lens)
    b = run_bwd(q, k, v, dout, W.default_scale(64), W.MASK_CAUSAL, lens)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("d,mask", [(64, W.MASK_CAUSAL), (128, W.MASK_NONE)])
def test_bwd_long_sequence(orc, d, mask):
    """n = 4096 (32 tiles each way), the launch shape of the long-sequence workloads."""
    w = W.WORKLOADS["long_causal_b2_h16_n8192_d64"]
    q, k, v, _ = W.make_inputs(w, seed=7600 + d, B=1, H=2, n_q=4096, n_k=4096, d_k=d, d_v=d)
    rng = np.random.Generator(np.random.PCG64(7601 + d))
    dout = W.to_bf16_bits(rng.standard_normal((1, 2, 4096, d), dtype=np.float32))
    lens = np.full((1,), 4096, np.int32)
    got = run_bwd(q, k, v, dout, w.scale, mask, lens)
    ref = orc.attention_bwd(q, k, v, dout, w.scale, mask, None)
    check(got, ref, bounds(orc, q, k, v, dout, w.scale, mask, None, ref))


def test_bwd_rejects_small_workspace():
    q, k, v, dout, lens = draw(7700, 1, 1, 64, 64, 64, W.MASK_NONE)
    qd, kd, vd, gd = dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_bf16(dout)
    lse = torch.zeros((1, 1, 64), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.attn_bwd_workspace_size(1, 1, 64) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_bwd(qd, kd, vd, qd, gd, lse, torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd), ws)
    assert e.value.status == attn.ATTN_ERR_INVALID
