"""attn_mha_fwd (projections on cuBLASLt + the attention kernel on the heads-
interleaved layout + the output projection) against the fp64 oracle's multi-head
attention on the same bf16 inputs, element by element.

Tolerance, derived from the arithmetic of the CUDA path by first-order error
propagation from the exact intermediates (Q', K', V', P, A, Y of the oracle's
definition; u = 2^-8 = bf16's unit roundoff, the largest relative error of one
rounding to nearest; g_K = K 2^-23 for an fp32 sum of K
products, one ulp per addition since the accumulation is not assumed to round to
nearest; |.| element-wise):
  * projections: |dQ'| <= u|Q'| + g_dmodel (|x||W| + |b|), likewise K', V';
  * scores: |ds_ij| <= scale (|dQ'_i|.|K'_j| + |Q'_i|.|dK'_j|) + scale g_d |Q'_i|.|K'_j|;
  * weights: |dP_ij| <= P_ij (|ds_ij| + sum_j' P_ij' |ds_ij'| + u) (softmax
    sensitivity, plus the kernel's bf16 rounding of P);
  * head outputs: |dA_i| <= sum_j |dP_ij| |V'_j| + P_ij |dV'_j| + u|A_i| + g_nk P|V'|;
  * layer output: |dY| <= |dA| |W^O| + g_hd (|A||W^O| + |b_O|) + u|Y|.
That worst case adds |errors| over every feature of W^O (about 15 |Y| at d_model
1024), so it is checked (twice, for second-order terms) only as a hard ceiling. The
working bound is the quadrature one: the same chain with u/2 (about the RMS of
one rounding's relative error, between u/sqrt(12) and u/sqrt(3) across a binade)
and sums of squares, the root-mean-square of independent roundings. Each element's error is
a sum of many such terms, close to Gaussian with that scale: checked per element as
|err| <= 6 qbound, and over the whole tensor as ||err||_2 <= ||qbound||_2.
"""
import numpy as np
import pytest
import torch

from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
U = 2.0 ** -8
EPS = 2.0 ** -23
RESULTS = []


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.lib()
    yield
    st, code = attn.attn_fault_status()
    assert st == attn.ATTN_OK, f"kernel fault record {code:#x}"


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def wide(a):
    return None if a is None else (np.ascontiguousarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_mha(inp, x_kv, mask, scale):
    xq = dev(inp["x_q"])
    xkv = xq if x_kv is inp["x_q"] else dev(x_kv)
    B, n_q, d_model = inp["x_q"].shape
    n_k = x_kv.shape[1]
    out = torch.full((B, n_q, d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(attn.attn_mha_workspace_size(B, n_q, n_k, d_model, inp["H"], inp["d"]), dtype=torch.uint8,
                     device="cuda")
    kl = torch.from_numpy(inp["key_lens"]).cuda() if mask & W.MASK_KEY_PADDING else None
    attn.attn_mha_fwd(xq, xkv, dev(inp["w_q"]), dev(inp["w_k"]), dev(inp["w_v"]), dev(inp["w_o"]), out, inp["H"], ws,
                      dev(inp["b_q"]), dev(inp["b_k"]), dev(inp["b_v"]), dev(inp["b_o"]), scale, mask, kl)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def heads(x, H):
    """[B, n, H*d] -> [B, H, n, d]."""
    B, n, hd = x.shape
    return np.ascontiguousarray(x.reshape(B, n, H, hd // H).transpose(0, 2, 1, 3))


def bounds(orc, inp, x_kv, mask, scale, y_ref):
    H, d = inp["H"], inp["d"]
    X, XKV = wide(inp["x_q"]), wide(x_kv)
    Wq, Wk, Wv, Wo = (wide(inp[k]) for k in ("w_q", "w_k", "w_v", "w_o"))
    bq, bk, bv, bo = (wide(inp[k]) if inp[k] is not None else 0.0 for k in ("b_q", "b_k", "b_v", "b_o"))
    d_model = X.shape[-1]
    kl = inp["key_lens"] if mask & W.MASK_KEY_PADDING else None
    T = lambda a: np.swapaxes(a, -1, -2)
    proj = lambda x, w, b: (x @ w + b, d_model * EPS * (np.abs(x) @ np.abs(w) + np.abs(b)))
    (Qp, gQ), (Kp, gK), (Vp, gV) = proj(X, Wq, bq), proj(XKV, Wk, bk), proj(XKV, Wv, bv)
    Qh, Kh, Vh = heads(Qp, H), heads(Kp, H), heads(Vp, H)
    eQ, eK, eV = heads(U * np.abs(Qp) + gQ, H), heads(U * np.abs(Kp) + gK, H), heads(U * np.abs(Vp) + gV, H)
    P = orc.attention_weights(Qh, Kh, scale, mask, kl)
    A = P @ Vh
    n_k = Kh.shape[2]
    aQ, aK = np.abs(Qh), np.abs(Kh)
    ds = scale * (eQ @ T(aK) + aQ @ T(eK) + d * EPS * aQ @ T(aK))
    dP = P * (ds + np.sum(P * ds, -1, keepdims=True) + U)
    dA = dP @ np.abs(Vh) + P @ eV + U * np.abs(A) + n_k * EPS * (P @ np.abs(Vh))
    cat = lambda a: a.transpose(0, 2, 1, 3).reshape(a.shape[0], a.shape[2], -1)
    Acat, dAcat = cat(A), cat(dA)
    worst = dAcat @ np.abs(Wo) + H * d * EPS * (np.abs(Acat) @ np.abs(Wo) + np.abs(bo)) + U * np.abs(y_ref)
    # quadrature: u/2 per rounding, sums of squares
    h = U / 2
    qQ, qK, qV = heads(h * np.abs(Qp) + gQ, H), heads(h * np.abs(Kp) + gK, H), heads(h * np.abs(Vp) + gV, H)
    qs = scale * np.sqrt(qQ ** 2 @ T(Kh ** 2) + Qh ** 2 @ T(qK ** 2))
    qP = P * (qs + np.sqrt(np.sum((P * qs) ** 2, -1, keepdims=True)))
    qA = np.sqrt(qP ** 2 @ Vh ** 2 + (h * P) ** 2 @ Vh ** 2 + P ** 2 @ qV ** 2) + h * np.abs(A)
    quad = np.sqrt(cat(qA) ** 2 @ Wo ** 2) + h * np.abs(y_ref)
    return worst, quad


def parity(orc, inp, self_attn, mask, scale=None):
    x_kv = inp["x_q"] if self_attn else inp["x_kv"]
    scale = W.default_scale(inp["d"]) if scale is None else scale
    got = run_mha(inp, x_kv, mask, scale)
    kl = inp["key_lens"] if mask & W.MASK_KEY_PADDING else None
    ref = orc.mha(inp["x_q"], x_kv, inp["w_q"], inp["w_k"], inp["w_v"], inp["w_o"], inp["H"], scale, mask, kl,
                  b_q=inp["b_q"], b_k=inp["b_k"], b_v=inp["b_v"], b_o=inp["b_o"])
    worst, quad = bounds(orc, inp, x_kv, mask, scale, ref)
    err = np.abs(got - ref)
    RESULTS.append(((inp["x_q"].shape, x_kv.shape[1], inp["H"], inp["d"], mask), float(np.max(err / worst)),
                    float(np.max(err / (quad + 1e-30))), float(np.linalg.norm(err) / np.linalg.norm(quad))))
    assert np.isfinite(got).all()
    bad = err > 2 * worst + 1e-6
    assert not bad.any(), f"{bad.sum()} of {bad.size} beyond the worst-case bound; max err {err.max():.3e}"
    bad = err > 6 * quad + 1e-6
    assert not bad.any(), f"{bad.sum()} of {bad.size} beyond 6x the quadrature bound; max err {err.max():.3e}"
    assert np.linalg.norm(err) <= np.linalg.norm(quad), \
        f"||err|| {np.linalg.norm(err):.3e} above the quadrature bound {np.linalg.norm(quad):.3e}"
    return got, ref


ENC = W.WORKLOADS["encoder_self_pad_b32_h8_n128_d64"]
DEC = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
CROSS = W.WORKLOADS["cross_pad_b16_h16_q256_k512_d64"]


@pytest.mark.parametrize("mask", [W.MASK_NONE, W.MASK_KEY_PADDING, W.MASK_CAUSAL, W.MASK_CAUSAL | W.MASK_KEY_PADDING])
def test_mha_self_base_size(orc, mask):
    """d_model 512, h 8, d 64 (the base model), 200 positions: two query blocks, ragged tail."""
    inp = W.make_mha_inputs(ENC, seed=8000 + mask, B=2, H=8, n_q=200, n_k=200)
    inp["key_lens"] = np.array([200, 77], np.int32)
    parity(orc, inp, True, mask)


def test_mha_cross_big_size(orc):
    """Encoder-decoder attention, d_model 1024, h 16: 130 decoder queries, 257 encoder
    keys; key lengths full, partial and 0 (no legal key: the heads give 0, Y = b_O)."""
    inp = W.make_mha_inputs(CROSS, seed=8100, B=3, H=16, n_q=130, n_k=257)
    inp["key_lens"] = np.array([257, 200, 0], np.int32)
    parity(orc, inp, False, W.MASK_KEY_PADDING)


@pytest.mark.parametrize("bias", [True, False])
def test_mha_d128_and_bias(orc, bias):
    inp = W.make_mha_inputs(DEC, seed=8200 + bias, bias=bias, B=1, H=4, n_q=300, n_k=300, d_k=128, d_v=128)
    parity(orc, inp, True, W.MASK_CAUSAL)


def test_mha_d_model_not_h_times_d(orc):
    """d_model need not equal h*d: 256 features, 8 heads of 64."""
    inp = W.make_mha_inputs(DEC, seed=8300, d_model=256, B=2, H=8, n_q=96, n_k=160)
    parity(orc, inp, False, W.MASK_NONE)


@pytest.mark.parametrize("n_q,n_k", [(1, 1), (1, 300), (129, 1)])
def test_mha_edge_lengths(orc, n_q, n_k):
    inp = W.make_mha_inputs(CROSS, seed=8400 + n_q + n_k, B=2, H=4, n_q=n_q, n_k=n_k)
    parity(orc, inp, False, W.MASK_NONE)


def test_mha_longer_sequence(orc):
    """1024 positions (eight query blocks), big size, causal."""
    inp = W.make_mha_inputs(DEC, seed=8500, B=1, H=16, n_q=1024, n_k=1024)
    parity(orc, inp, True, W.MASK_CAUSAL)


@pytest.mark.parametrize("d", [64, 128])
def test_heads_interleaved_attention_equals_split_layout(d):
    """At the long-sequence size (n = 8192, h = 16) the attention kernel on the
    [B, n, h*d] layout gives bit-identical heads to the kernel on [B, h, n, d]: the
    layout only moves addresses. Run through attn_mha_fwd with identity projections
    and no biases (each GEMM then reproduces its input exactly) against attn_fwd on
    the split copy."""
    B, H, n = 1, 16, 8192
    d_model = H * d
    g = torch.Generator(device="cuda").manual_seed(8600 + d)
    x = (torch.randn((B, n, d_model), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    eye = torch.eye(d_model, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(attn.attn_mha_workspace_size(B, n, n, d_model, H, d), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    attn.attn_mha_fwd(x, x, eye, eye, eye, eye, y, H, ws, mask_mode=W.MASK_CAUSAL)
    split = x.view(B, n, H, d).transpose(1, 2).contiguous()
    o = torch.empty_like(split)
    attn.attn_fwd(split, split, split, o, None, None, W.MASK_CAUSAL)
    torch.cuda.synchronize()
    assert torch.equal(y, o.transpose(1, 2).reshape(B, n, d_model))


def test_mha_rejects_bad_arguments():
    inp = W.make_mha_inputs(ENC, seed=8700, B=1, H=2, n_q=8, n_k=8)
    xq = dev(inp["x_q"])
    out = torch.empty_like(xq)
    need = attn.attn_mha_workspace_size(1, 8, 8, 128, 2, 64)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_mha_fwd(xq, xq, dev(inp["w_q"]), dev(inp["w_k"]), dev(inp["w_v"]), dev(inp["w_o"]), out, 2, ws)
    assert e.value.status == attn.ATTN_ERR_INVALID
