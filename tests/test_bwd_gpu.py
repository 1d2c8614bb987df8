"""attn_bwd (dQ, dK, dV on the tensor cores) against the fp64 oracle's gradients,
element by element on the same bf16-rounded inputs.

The forward output and lse the gradients consume come from attn_fwd (as a training
step would use them); dout is a seeded bf16 draw.

Tolerance, derived from the arithmetic of the CUDA path. P = the exact weights,
u = 2^-8 = bf16's unit roundoff (8 significant bits: one rounding to nearest is off
by at most u of the value), |.| element-wise:
  * D_i = dout_i . out_i is formed from the bf16 forward output; its error dD_i is
    measured (fp64 D from that output minus the exact one, plus the fp32
    accumulation allowance d 2^-23 sum |dout||out|);
  * dS = P (dP - D) is off by -P dD (the same dD along a row) plus its bf16
    rounding e, |e| <= u |dS|; P is rounded to bf16 (u P) before dV;
  * S, dP and D accumulate d products in fp32 (the tensor cores' accumulation is not
    assumed to round to nearest, so one ulp, 2^-23, per addition):
    |S_ij err| <= g (|Q||K|^T)_ij and |dP_ij err| <= eP_ij = g (|dout||V|^T)_ij
    with g = d 2^-23; with the fp32
    exponent arithmetic (scale, log2 e, lse and ex2.approx, 2^-20 (1 + |scale s| +
    |lse|) together) P is off by rP_ij P_ij, rP_ij = scale g (|Q||K|^T)_ij + that;
    so dS also carries x_ij = P_ij eP_ij + rP_ij P_ij |dP_ij - D_i|;
  * dV, dK and dQ accumulate n_q, n_q and n_k products in fp32 (a = n 2^-23 of
    their sums of absolute values) and are rounded to bf16 once (u |g|). The fused
    schedule (d = 64) forms dQ from 128-key partial sums added in fp32 in memory:
    fewer than n_k additions, so the same allowance covers it.
Worst case per element (all rounding errors aligned), checked as |err| <= 1.25
bound (the quarter covers the neglected second-order products of these terms):
  bound(dV) = (u + rP + a_q) P^T|dout| + u|dV|
  bound(dK) = scale (P dD + (u + a_q)|dS| + x)^T |Q| + u|dK|
  bound(dQ) = scale |dD| |P K| + scale ((u + a_k) |dS| + x) |K| + u|dQ|
Typical size (independent roundings add in quadrature), checked over the whole
tensor as ||err||_2 <= ||qbound||_2, where qbound replaces each sum of absolute
values above by the root of the sum of squares and u by u/2, about the RMS of one
rounding's relative error (between u/sqrt(12) and u/sqrt(3) across a binade; the
coherent P dD term of dQ stays as it is). A systematic mistake (a dropped term, a
wrong sign or scale) shows in one or both.
"""
import numpy as np
import pytest
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
U = 2.0 ** -8
RESULTS = []  # (case, ratios) of every parity case run in this session


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


def run_bwd(q, k, v, dout, scale, mask, lens, flags=0, window=None):
    """attn_fwd + attn_bwd, or with a window attn_fwd_local + attn_bwd_local."""
    B, H, n_q, d = q.shape
    qd, kd, vd, gd = dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_bf16(dout)
    kl = torch.from_numpy(lens).cuda() if mask & W.MASK_KEY_PADDING else None
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device="cuda")
    if window is None:
        attn.attn_fwd(qd, kd, vd, out, lse, scale, mask, kl)
    else:
        attn.attn_fwd_local(qd, kd, vd, out, window, lse, scale, mask, kl)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, n_q, d, flags), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.full_like(qd, float("nan")), torch.full_like(kd, float("nan")), torch.full_like(vd, float("nan"))
    if window is None:
        attn.attn_bwd(qd, kd, vd, out, gd, lse, dq, dk, dv, ws, scale, mask, kl, flags=flags)
    else:
        attn.attn_bwd_local(qd, kd, vd, out, gd, lse, dq, dk, dv, ws, window, scale, mask, kl, flags=flags)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return (f(dq), f(dk), f(dv)), f(out)


def bounds(orc, q, k, v, dout, scale, mask, lens, ref, out_dev, P=None, lse=None, window=0):
    """(worst-case bounds, quadrature bounds) of the CUDA path's error, per element
    (module docstring). P and lse, the oracle's weights and log-sum-exp, may be given;
    window as in the oracle (0: none)."""
    if P is None:
        P = orc.attention_weights(q, k, scale, mask, lens, window=window)
    if lse is None:
        _, lse = orc.attention(q, k, v, scale, mask, lens, window=window)
    Q, K, V, G = (bits_to_f64(x) for x in (q, k, v, dout))
    dq_r, dk_r, dv_r = ref
    d, n_q, n_k = Q.shape[-1], Q.shape[-2], K.shape[-2]
    g, a_q, a_k = d * 2.0 ** -23, n_q * 2.0 ** -23, n_k * 2.0 ** -23
    T = lambda x: np.swapaxes(x, -1, -2)
    O = P @ V
    dD = np.abs(np.sum(G * out_dev, -1) - np.sum(G * O, -1)) + g * np.sum(np.abs(G * out_dev), -1)
    dP = G @ T(V)
    dS = P * (dP - np.sum(G * O, axis=-1)[..., None])
    lse_f = np.where(np.isfinite(lse), np.abs(lse), 0.0)[..., None]
    rP = scale * g * (np.abs(Q) @ T(np.abs(K))) + 2.0 ** -20 * (1 + np.abs(scale * (Q @ T(K))) + lse_f)
    x = P * g * (np.abs(G) @ T(np.abs(V))) + rP * np.abs(dS)
    PD = P * dD[..., None]
    worst = (scale * dD[..., None] * np.abs(P @ K) + scale * (((U + a_k) * np.abs(dS) + x) @ np.abs(K))
             + U * np.abs(dq_r),
             scale * (T(PD + (U + a_q) * np.abs(dS) + x) @ np.abs(Q)) + U * np.abs(dk_r),
             (T((U + a_q) * P + rP * P) @ np.abs(G)) + U * np.abs(dv_r))
    h = U / 2
    rss = lambda a, b: np.sqrt(a ** 2 @ b ** 2)
    quad = (scale * dD[..., None] * np.abs(P @ K) + scale * (h * rss(dS, K) + rss(x, K)) + h * np.abs(dq_r),
            scale * (rss(T(PD), Q) + h * rss(T(dS), Q) + rss(T(x), Q)) + h * np.abs(dk_r),
            h * rss(T(P), G) + rss(T(rP * P), G) + h * np.abs(dv_r))
    return worst, quad


def ratios(got, ref, bnd):
    """Per gradient: (max err / worst-case bound, ||err|| / ||quadrature bound||)."""
    worst, quad = bnd
    res = {}
    for name, g, r, b, qb in zip(("dq", "dk", "dv"), got, ref, worst, quad):
        err = np.abs(g - r)
        res[name] = (float(np.max(err / (b + 1e-30))), float(np.linalg.norm(err) / (np.linalg.norm(qb) + 1e-30)))
    return res


def check(got, ref, bnd):
    worst, quad = bnd
    for name, g, r, b, qb in zip(("dq", "dk", "dv"), got, ref, worst, quad):
        assert np.isfinite(g).all(), f"{name} has non-finite values"
        err = np.abs(g - r)
        bad = err > 1.25 * b + 1e-7
        assert not bad.any(), (f"{name}: {bad.sum()} of {bad.size} beyond the worst-case bound; worst err "
                               f"{err[bad].max():.3e}, max err {err.max():.3e}")
        assert np.linalg.norm(err) <= np.linalg.norm(qb) + 1e-7, (
            f"{name}: ||err|| {np.linalg.norm(err):.3e} above the quadrature bound {np.linalg.norm(qb):.3e}")


def parity(orc, seed, B, H, n_q, n_k, d, mask, lens=None, scale=None, flags=0, window=None):
    q, k, v, dout, lens = draw(seed, B, H, n_q, n_k, d, mask, lens)
    scale = W.default_scale(d) if scale is None else scale
    got, out_dev = run_bwd(q, k, v, dout, scale, mask, lens, flags, window)
    kl = lens if mask & W.MASK_KEY_PADDING else None
    # the oracle applies its window under the MASK_WINDOW bit
    omask, ow = (mask, 0) if window is None else (mask | W.MASK_WINDOW, window)
    ref = orc.attention_bwd(q, k, v, dout, scale, omask, kl, window=ow)
    bnd = bounds(orc, q, k, v, dout, scale, omask, kl, ref, out_dev, window=ow)
    RESULTS.append(((B, H, n_q, n_k, d, mask), ratios(got, ref, bnd)))
    check(got, ref, bnd)
    return got, ref


@pytest.mark.parametrize("d,flags", [(64, 0), (64, attn.BWD_DETERMINISTIC), (128, 0)])
@pytest.mark.parametrize("mask", [W.MASK_NONE, W.MASK_CAUSAL])
@pytest.mark.parametrize("n", [1, 64, 128, 300, 513])
def test_bwd_self(orc, d, flags, mask, n):
    parity(orc, 7000 + d + n + 3 * mask, 2, 2, n, n, d, mask, flags=flags)


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


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_deterministic(d):
    """The deterministic schedule (no atomics): two calls give bit-identical gradients."""
    q, k, v, dout, lens = draw(7500, 2, 4, 700, 700, d, W.MASK_CAUSAL)
    a, _ = run_bwd(q, k, v, dout, W.default_scale(d), W.MASK_CAUSAL, lens, attn.BWD_DETERMINISTIC)
    b, _ = run_bwd(q, k, v, dout, W.default_scale(d), W.MASK_CAUSAL, lens, attn.BWD_DETERMINISTIC)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("mask", [W.MASK_CAUSAL, W.MASK_KEY_PADDING])
def test_bwd_fused_matches_deterministic(orc, mask):
    """The fused schedule (d = 64) runs the dK and dV products in the same order as the
    deterministic one, so dk and dv agree bit for bit; dq (reduced in memory, in varying
    order) must meet the derived bounds (checked by parity) and stay within a few bf16
    ulps of the deterministic dq."""
    q, k, v, dout, lens = draw(7550 + mask, 3, 2, 700, 700, 64, mask, lens=[700, 333, 1])
    fused, _ = run_bwd(q, k, v, dout, W.default_scale(64), mask, lens, 0)
    det, _ = run_bwd(q, k, v, dout, W.default_scale(64), mask, lens, attn.BWD_DETERMINISTIC)
    assert np.array_equal(fused[1], det[1]) and np.array_equal(fused[2], det[2])
    diff = np.abs(fused[0] - det[0])
    assert np.all(diff <= 4 * U * np.abs(det[0]) + 1e-6), f"dq differs by up to {diff.max():.3e}"
    parity(orc, 7550 + mask, 3, 2, 700, 700, 64, mask, lens=[700, 333, 1])


@pytest.mark.parametrize("d,mask", [(64, W.MASK_CAUSAL), (128, W.MASK_NONE)])
def test_bwd_long_sequence(orc, d, mask):
    """n = 4096 (32 tiles each way), the launch shape of the long-sequence workloads."""
    w = W.WORKLOADS["long_causal_b2_h16_n8192_d64"]
    q, k, v, _ = W.make_inputs(w, seed=7600 + d, B=1, H=2, n_q=4096, n_k=4096, d_k=d, d_v=d)
    rng = np.random.Generator(np.random.PCG64(7601 + d))
    dout = W.to_bf16_bits(rng.standard_normal((1, 2, 4096, d), dtype=np.float32))
    lens = np.full((1,), 4096, np.int32)
    got, out_dev = run_bwd(q, k, v, dout, w.scale, mask, lens)
    ref = orc.attention_bwd(q, k, v, dout, w.scale, mask, None)
    bnd = bounds(orc, q, k, v, dout, w.scale, mask, None, ref, out_dev)
    RESULTS.append(((1, 2, 4096, 4096, d, mask), ratios(got, ref, bnd)))
    check(got, ref, bnd)


@pytest.mark.parametrize("d,flags", [(64, 0), (64, attn.BWD_DETERMINISTIC), (128, 0)])
@pytest.mark.parametrize("window", [0, 1, 100, 127, 128, 300])
@pytest.mark.parametrize("mask", [W.MASK_NONE, W.MASK_CAUSAL])
def test_bwd_local_window(orc, d, flags, window, mask):
    """attn_bwd_local against the oracle's gradients under its window mask: windows
    inside one tile, at a tile edge and spanning several; n = 460 leaves a ragged tail."""
    parity(orc, 7000 + d + window + mask + flags, 1, 2, 460, 460, d, mask, flags=flags, window=window)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_local_window_key_padding(orc, d):
    """Window and key padding together; one batch entry's keys end inside the window of
    the last rows, the other's at a tile edge."""
    parity(orc, 7100 + d, 2, 2, 400, 400, d, W.MASK_KEY_PADDING | W.MASK_CAUSAL, lens=[300, 256], window=90)
    parity(orc, 7150 + d, 2, 1, 400, 400, d, W.MASK_KEY_PADDING, lens=[37, 400], window=200)


def test_bwd_local_window_covering_everything_equals_attn_bwd():
    """A window at least n - 1 wide is no restriction: attn_bwd_local equals attn_bwd bit
    for bit on dK and dV (the deterministic schedule: dQ too)."""
    q, k, v, dout, lens = draw(7200, 1, 2, 300, 300, 64, W.MASK_CAUSAL)
    scale = W.default_scale(64)
    a, _ = run_bwd(q, k, v, dout, scale, W.MASK_CAUSAL, lens, attn.BWD_DETERMINISTIC)
    for window in (299, 2**31 - 1):  # n - 1, and the widest window an int holds
        b, _ = run_bwd(q, k, v, dout, scale, W.MASK_CAUSAL, lens, attn.BWD_DETERMINISTIC, window=window)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_bwd_rejects_small_workspace():
    q, k, v, dout, lens = draw(7700, 1, 1, 64, 64, 64, W.MASK_NONE)
    qd, kd, vd, gd = dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_bf16(dout)
    lse = torch.zeros((1, 1, 64), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.attn_bwd_workspace_size(1, 1, 64, 64) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_bwd(qd, kd, vd, qd, gd, lse, torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd), ws)
    assert e.value.status == attn.ATTN_ERR_INVALID


@pytest.mark.parametrize("name,heads", [("long_causal_b2_h16_n8192_d64", [(0, 3), (1, 14)]),
                                        ("long_none_b2_h16_n8192_d128", [(1, 7)])])
def test_bwd_full_size_sampled_heads(orc, name, heads):
    """The bench's gradient workloads at full size (B 2, h 16, n 8192), in the launch
    configuration it times: the fused schedule at d = 64, the deterministic one at
    d = 128. Whole heads are sampled and checked element by element against the
    oracle's gradients of that head (its matrix form: one head of n = 8192 is a few
    BLAS products), with the derived bounds."""
    w = W.WORKLOADS[name]
    q, k, v, kl = W.make_inputs(w)
    dout = W.make_grad_output(w)
    got, out_dev = run_bwd(q, k, v, dout, w.scale, w.mask_mode, kl)
    for b, h in heads:
        sl = lambda a: np.ascontiguousarray(a[b:b + 1, h:h + 1])
        hq, hk, hv, hg = sl(q), sl(k), sl(v), sl(dout)
        ref = oracle.attention_bwd_matrix_form(hq, hk, hv, hg, w.scale, w.mask_mode, None)
        _, lse, P = oracle.attention_matrix_form(hq, hk, hv, w.scale, w.mask_mode, None)
        bnd = bounds(orc, hq, hk, hv, hg, w.scale, w.mask_mode, None, ref, sl(out_dev), P=P, lse=lse)
        head_got = tuple(sl(x) for x in got)
        RESULTS.append(((1, 1, w.n_q, w.n_k, w.d_k, w.mask_mode), ratios(head_got, ref, bnd)))
        check(head_got, ref, bnd)
