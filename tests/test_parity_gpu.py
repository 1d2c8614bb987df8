"""CUDA path against the fp64 oracle, element by element, on the same seeded inputs.

Tolerances (against the oracle run on the very same bf16-rounded inputs):
  bf16 path: max |err| <= 1e-2 and mean |err| <= 1e-3 on the output; |err| <= 1e-3
             on lse (natural log). The kernel rounds the softmax weights to bf16
             before the PV product (relative error <= 2^-8 per weight: bf16 keeps 8
             significant bits, so one rounding to nearest is off by at most 2^-8 of
             the value) and rounds the output to bf16 (<= 2^-8 relative); these
             errors are independent across weights, so for unit-variance V the
             expected max error is a few 1e-3.
  fp32 path: max |err| <= 1e-5 (float32 dot products and sums of at most a few
             hundred terms).
Every call goes through the C ABI (binding in transformer_scaled_dot_mha_gb300.attn).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL, F32_MAX = 1e-2, 1e-3, 1e-3, 1e-5
C, P = W.MASK_CAUSAL, W.MASK_KEY_PADDING


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


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_bf16(q, k, v, kl, scale, mode):
    kl_d = torch.from_numpy(kl).cuda() if mode & P else None
    out, lse = attn.attention(dev_bf16(q), dev_bf16(k), dev_bf16(v), scale, mode, kl_d, with_lse=True)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


def assert_bf16_close(out, lse, ref, ref_lse):
    err = np.abs(out - ref)
    assert np.isfinite(out).all()
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, f"max {err.max():.3e} mean {err.mean():.3e}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(lse[~fin] == -np.inf)
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= LSE_TOL


def gen(name, seed=None, **shape):
    w = W.WORKLOADS[name]
    return w, W.make_inputs(w, seed, **shape)


# ------------------------------------------------------------------ float32 path
def test_f32_two_token_worked_example(orc):
    """attention-paper-guide section 03.2: Q = I, K = [[1,0],[1,1]], V = [[10,0],[0,6]]."""
    q = torch.tensor([[1.0, 0.0], [0.0, 1.0]]).view(1, 1, 2, 2).cuda()
    k = torch.tensor([[1.0, 0.0], [1.0, 1.0]]).view(1, 1, 2, 2).cuda()
    v = torch.tensor([[10.0, 0.0], [0.0, 6.0]]).view(1, 1, 2, 2).cuda()
    out, lse = attn.attention(q, k, v, W.default_scale(2), with_lse=True)
    ref, ref_lse = orc.attention(*(t.cpu().numpy() for t in (q, k, v)), W.default_scale(2))
    assert np.abs(out.cpu().numpy() - ref).max() <= F32_MAX
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= F32_MAX
    assert np.abs(out.cpu().numpy()[0, 0] - [[5, 3], [3.3, 4.0]]).max() <= 0.05


def test_f32_tiny_config(orc):
    w, (q, k, v, _) = gen("tiny_f32_b1_h1_n16_d8")
    out, lse = attn.attention(*(torch.from_numpy(a).cuda() for a in (q, k, v)), w.scale, with_lse=True)
    ref, ref_lse = orc.attention(q, k, v, w.scale)
    assert np.abs(out.cpu().numpy() - ref).max() <= F32_MAX
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= F32_MAX


@pytest.mark.parametrize("mode", [0, C, P, C | P])
@pytest.mark.parametrize("shape", [(2, 3, 37, 37, 5, 7), (1, 2, 19, 70, 8, 3), (2, 1, 40, 40, 256, 256)])
def test_f32_masks_and_shapes(orc, mode, shape):
    B, H, n_q, n_k, d_k, d_v = shape
    if mode & C and n_q != n_k:
        pytest.skip("causal is self-attention only")
    rng = np.random.Generator(np.random.PCG64(hash((mode,) + shape) % (1 << 32)))
    q = rng.standard_normal((B, H, n_q, d_k), dtype=np.float32)
    k = rng.standard_normal((B, H, n_k, d_k), dtype=np.float32)
    v = rng.standard_normal((B, H, n_k, d_v), dtype=np.float32)
    kl = rng.integers(0, n_k, B, endpoint=True).astype(np.int32)
    kl[0] = max(kl[0], 1)
    scale = W.default_scale(d_k)
    kl_d = torch.from_numpy(kl).cuda() if mode & P else None
    out, lse = attn.attention(*(torch.from_numpy(a).cuda() for a in (q, k, v)), scale, mode, kl_d, with_lse=True)
    ref, ref_lse = orc.attention(q, k, v, scale, mode, kl)
    assert np.abs(out.cpu().numpy() - ref).max() <= F32_MAX
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin)
    assert np.abs(lse.cpu().numpy()[fin] - ref_lse[fin]).max() <= F32_MAX


# ------------------------------------------------------------------ bf16 path, reduced sizes
# several 128-key tiles, 256-row query blocks and ragged tails in both n_q and n_k
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", [0, C, P, C | P])
def test_bf16_self_attention_ragged(orc, d, mode):
    w, (q, k, v, kl) = gen("decoder_causal_b16_h8_n512_d64", seed=1000 + d + mode, B=2, H=3, n_q=300, n_k=300,
                           d_k=d, d_v=d)
    kl = np.array([300, 131], np.int32)
    scale = W.default_scale(d)
    out, lse = run_bf16(q, k, v, kl, scale, mode)
    ref, ref_lse = orc.attention(q, k, v, scale, mode, kl)
    assert_bf16_close(out, lse, ref, ref_lse)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", [0, P])
@pytest.mark.parametrize("n_q,n_k", [(200, 333), (513, 129), (1, 1000), (700, 1)])
def test_bf16_cross_attention_ragged(orc, d, mode, n_q, n_k):
    w, (q, k, v, kl) = gen("cross_pad_b16_h16_q256_k512_d64", seed=2000 + n_q + d, B=3, H=2, n_q=n_q, n_k=n_k,
                           d_k=d, d_v=d)
    kl = np.array([n_k, max(1, n_k // 3), 1], np.int32)
    scale = W.default_scale(d)
    out, lse = run_bf16(q, k, v, kl, scale, mode)
    ref, ref_lse = orc.attention(q, k, v, scale, mode, kl)
    assert_bf16_close(out, lse, ref, ref_lse)


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 255, 256, 257, 383, 384, 640])
def test_bf16_tile_boundaries_causal(orc, n):
    w, (q, k, v, kl) = gen("decoder_causal_b16_h8_n512_d64", seed=3000 + n, B=1, H=2, n_q=n, n_k=n)
    out, lse = run_bf16(q, k, v, kl, w.scale, C)
    ref, ref_lse = orc.attention(q, k, v, w.scale, C)
    assert_bf16_close(out, lse, ref, ref_lse)
    # row 0 attends to key 0 alone: the output is V[0] rounded to bf16
    assert np.array_equal(out[:, :, 0], oracle.widen(v)[:, :, 0])


def test_bf16_key_length_zero_and_one(orc):
    w, (q, k, v, _) = gen("encoder_self_pad_b32_h8_n128_d64", seed=4000, B=4, H=2, n_q=150, n_k=150)
    kl = np.array([0, 1, 150, 129], np.int32)
    out, lse = run_bf16(q, k, v, kl, w.scale, P)
    ref, ref_lse = orc.attention(q, k, v, w.scale, P, kl)
    assert_bf16_close(out, lse, ref, ref_lse)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.array_equal(out[1], np.broadcast_to(oracle.widen(v)[1, :, :1], out[1].shape))


def test_bf16_large_scores_rescaling(orc):
    """Scores growing along the key axis force repeated rescaling of the running output."""
    w, (q, k, v, kl) = gen("decoder_causal_b16_h8_n512_d64", seed=4100, B=1, H=2, n_q=256, n_k=1024)
    kf = oracle.widen(k)
    kf *= np.linspace(0.2, 6.0, 1024)[None, None, :, None]  # later keys have much larger norms
    k2 = W.to_bf16_bits(kf.astype(np.float32))
    q2 = W.to_bf16_bits((oracle.widen(q) * 3).astype(np.float32))
    out, lse = run_bf16(q2, k2, v, kl, w.scale, 0)
    ref, ref_lse = orc.attention(q2, k2, v, w.scale, 0)
    # Sharp rows are dominated by a few weights, so the bf16 rounding of P (at most
    # 2^-8 of each weight, and the weights sum to 1) and of the output (2^-8 |o|) no
    # longer average out; together they are bounded by 2 * 2^-8 max|V| = 2^-7 max|V|,
    # which is the bound used here.
    err = np.abs(out - ref)
    assert err.max() <= 2.0 ** -7 * np.abs(oracle.widen(v)).max() and err.mean() <= BF16_MEAN
    assert np.abs(lse - ref_lse).max() <= LSE_TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode", [0, C])
def test_bf16_score_jumps_within_later_tiles(orc, d, mode):
    """Keys whose scores jump well above everything before them, placed in the first
    and the second 64-key half of later 128-key tiles (and in both halves of one tile),
    plus a cluster of keys that raises a half's sum of weights without raising its row
    maximum past the rescaling threshold: every way in which the running maximum of a
    row can be overtaken after the first tile, against the oracle."""
    n = 1024
    name = "long_none_b2_h16_n8192_d64" if d == 64 else "long_none_b2_h16_n8192_d128"
    w, (q, k, v, kl) = gen(name, seed=4150 + d + mode, B=1, H=2, n_q=n, n_k=n)
    rng = np.random.Generator(np.random.PCG64(4160 + d))
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    qf, kf = oracle.widen(q), oracle.widen(k)
    qf += 4.0 * u  # every query leans on u, so a key along u raises every row's score
    # (key, jump of its score in log2 units): after the first tile the reference maximum
    # sits a few units above the typical score, and rescaling starts 8 units above it
    jumps = [(130, 10), (131, 10), (132, 10), (133, 10),  # tile 1, first half: sum only
             (340, 20),                                   # tile 2, second half
             (520, 30), (600, 40),                        # tile 4, both halves
             (800, 26), (1000, 46)]                       # tile 6 below, tile 7 above
    for key, jump in jumps:
        kf[:, :, key, :] += jump * math.log(2.0) / (4.0 * w.scale) * u
    q2, k2 = W.to_bf16_bits(qf.astype(np.float32)), W.to_bf16_bits(kf.astype(np.float32))
    out, lse = run_bf16(q2, k2, v, kl, w.scale, mode)
    ref, ref_lse = orc.attention(q2, k2, v, w.scale, mode)
    # sharp rows: the bound of the rescaling test above (2 * 2^-8 max|V|)
    err = np.abs(out - ref)
    assert np.isfinite(out).all()
    assert err.max() <= 2.0 ** -7 * np.abs(oracle.widen(v)).max() and err.mean() <= BF16_MEAN
    assert np.abs(lse - ref_lse).max() <= LSE_TOL


def test_bf16_guard_bands_and_determinism():
    """Nothing is written outside out / lse, and two calls give identical bits."""
    w, (q, k, v, kl) = gen("cross_pad_b16_h16_q256_k512_d64", seed=4200, B=2, H=2, n_q=257, n_k=300)
    qd, kd, vd, kld = dev_bf16(q), dev_bf16(k), dev_bf16(v), torch.from_numpy(kl).cuda()
    n_out, pad = 2 * 2 * 257 * 64, 4096
    outs = []
    for _ in range(2):
        buf = torch.full((n_out + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
        lbuf = torch.full((2 * 2 * 257 + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
        out = buf[pad:pad + n_out].view(2, 2, 257, 64)
        lse = lbuf[pad:pad + 2 * 2 * 257].view(2, 2, 257)
        attn.attn_fwd(qd, kd, vd, out, lse, w.scale, P, kld)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -7.0) and torch.all(buf[pad + n_out:] == -7.0)
        assert torch.all(lbuf[:pad] == -7.0) and torch.all(lbuf[pad + 2 * 2 * 257:] == -7.0)
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_bf16_runs_on_a_side_stream(orc):
    w, (q, k, v, kl) = gen("decoder_causal_b16_h8_n512_d64", seed=4300, B=1, H=1, n_q=384, n_k=384)
    s = torch.cuda.Stream()
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = torch.empty_like(qd)
        attn.attn_fwd(qd, kd, vd, out, None, w.scale, C, None, stream=s)
    s.synchronize()
    ref, _ = orc.attention(q, k, v, w.scale, C)
    err = np.abs(bf16_to_f64(out) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["encoder_self_pad_b32_h8_n128_d64", "decoder_causal_b16_h8_n512_d64",
                                  "cross_pad_b16_h16_q256_k512_d64"])
def test_bf16_full_size_workloads(orc, name):
    w, (q, k, v, kl) = gen(name)
    out, lse = run_bf16(q, k, v, kl, w.scale, w.mask_mode)
    ref, ref_lse = orc.attention(q, k, v, w.scale, w.mask_mode, kl)
    assert_bf16_close(out, lse, ref, ref_lse)


def _sample_rows(B, H, n):
    heads = [(0, 0), (B - 1, H - 1), (0, H // 2)]
    rows = {0, 1, 2, 127, 128, 129, 255, 256, 257, 511, 512, n // 2 - 1, n // 2, n - 129, n - 128, n - 2, n - 1}
    rows |= set(range(5, n, 97))
    ids = [(b * H + h) * n + i for b, h in heads for i in sorted(rows) if i < n]
    return np.array(ids, np.int64)


@pytest.mark.parametrize("name", ["long_causal_b2_h16_n8192_d64", "long_none_b2_h16_n8192_d64",
                                  "long_causal_b2_h16_n8192_d128", "long_none_b2_h16_n8192_d128",
                                  "long_cross_pad_b2_h16_q4096_k8192_d64",
                                  "long_cross_pad_b2_h16_q4096_k8192_d128"])
def test_bf16_long_sequence_sampled_rows(orc, name):
    """n = 8192 at full size: sampled rows (tile edges, ends, every 97th row of three
    heads) against the oracle, plus properties that hold for every row: each output
    is a convex combination of V rows, and lse is finite and at least the scaled
    score of the key the row attends to first."""
    w, (q, k, v, kl) = gen(name)
    out, lse = run_bf16(q, k, v, kl, w.scale, w.mask_mode)
    ids = _sample_rows(w.B, w.H, w.n_q)
    ref, ref_lse = orc.attention_rows(q, k, v, w.scale, ids, w.mask_mode, kl)
    assert_bf16_close(out.reshape(-1, w.d_v)[ids], lse.reshape(-1)[ids], ref, ref_lse)
    vf = oracle.widen(v)
    vmin, vmax = vf.min(axis=2, keepdims=True), vf.max(axis=2, keepdims=True)
    slack = 1e-2
    assert np.all(out >= vmin - slack) and np.all(out <= vmax + slack)
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens", [(8192, 6145), (6144, 8191), (8064, 8065)])
def test_bf16_long_cross_key_length_edges(orc, d, lens):
    """Encoder-decoder attention at full size (4096 queries x 8192 keys) with key
    lengths on, just past and just before a 128-key tile edge: sampled rows of every
    head class against the oracle."""
    w, (q, k, v, _) = gen(f"long_cross_pad_b2_h16_q4096_k8192_d{d}")
    kl = np.array(lens, np.int32)
    out, lse = run_bf16(q, k, v, kl, w.scale, P)
    ids = _sample_rows(w.B, w.H, w.n_q)
    ref, ref_lse = orc.attention_rows(q, k, v, w.scale, ids, P, kl)
    assert_bf16_close(out.reshape(-1, w.d_v)[ids], lse.reshape(-1)[ids], ref, ref_lse)


@pytest.mark.parametrize("mode,n_q,n_k", [(C | P, 777, 777), (P, 900, 1300), (C, 1025, 1025)])
def test_bf16_multi_wave_grid(orc, mode, n_q, n_k):
    """More than one wave of 128-row Q tiles (here 336-432 CTAs on 2 x 152 slots), with
    key lengths of 0, 1 and a tile edge: CTAs with no K/V tile or a single key run
    beside ordinary ones and in the second wave. Every row against the oracle."""
    B, H = 3, 16
    w, (q, k, v, _) = gen("cross_pad_b16_h16_q256_k512_d64", seed=5000 + n_q + mode, B=B, H=H, n_q=n_q, n_k=n_k)
    kl = np.array([0, 1, min(n_k, 640)], np.int32) if mode & P else np.full(B, n_k, np.int32)
    out, lse = run_bf16(q, k, v, kl, w.scale, mode)
    ref, ref_lse = orc.attention(q, k, v, w.scale, mode, kl)
    assert_bf16_close(out, lse, ref, ref_lse)


def test_bf16_dependent_calls_on_one_stream(orc):
    """Kernels of this library start before the previous kernel on the stream has
    finished (programmatic dependent launch) and wait for it before touching memory.
    Chain them so that each reads what the one before wrote: O1 = Attn(Q, K, V), then
    O2 = Attn(O1, K, V) with no synchronisation in between, several times over. Both
    against the oracle, O2 computed from the oracle's own inputs: the bf16 O1 the GPU
    returned."""
    w, (q, k, v, _) = gen("decoder_causal_b16_h8_n512_d64", seed=5200, B=2, H=4, n_q=640, n_k=640)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    o1, o2 = torch.empty_like(qd), torch.empty_like(qd)
    for _ in range(5):
        o1.fill_(float("nan"))
        o2.fill_(float("nan"))
        attn.attn_fwd(qd, kd, vd, o1, None, w.scale, C, None)
        attn.attn_fwd(o1, kd, vd, o2, None, w.scale, C, None)
    torch.cuda.synchronize()
    o1_bits = o1.view(torch.int16).cpu().numpy().view(np.uint16)
    ref1, _ = orc.attention(q, k, v, w.scale, C)
    ref2, _ = orc.attention(o1_bits, k, v, w.scale, C)
    for out, ref in ((o1, ref1), (o2, ref2)):
        err = np.abs(bf16_to_f64(out) - ref)
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN
