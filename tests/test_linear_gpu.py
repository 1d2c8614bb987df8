"""attn_linear (the multi-head layer's projection kernel) against the fp64 oracle,
element by element, on the same bf16 inputs.

Bound, derived from the kernel's arithmetic (|.| element-wise, u = 2^-8 the unit
roundoff of bf16, the largest relative error of one rounding to nearest even;
2^-23 one fp32 ulp per addition, the tensor cores' accumulation order and rounding
not being assumed):
  |y_gpu - y| <= u |y| + (K + 1) 2^-23 (|x| |W| + |b|)
i.e. one rounding of the result to bf16 plus the fp32 accumulation of K products and
the bias. It is checked per element (no slack factor), and the quadrature version
(u/2 per rounding) over the whole tensor, so that a systematic error cannot hide
under the worst case.
"""
import numpy as np
import pytest
import torch

from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
U, EPS = 2.0 ** -8, 2.0 ** -23


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
    return (np.ascontiguousarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def draw(seed, M, N, K, bias=True):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = W.to_bf16_bits(rng.standard_normal((K, N), dtype=np.float32) * np.float32(1 / np.sqrt(K)))
    b = W.to_bf16_bits(rng.standard_normal(N, dtype=np.float32) * np.float32(0.1)) if bias else None
    return x, w, b


def check(orc, x, w, b, y_gpu, rows=None):
    xs = x if rows is None else x[rows]
    ys = y_gpu if rows is None else y_gpu[rows]
    ref = orc.linear(xs, w, b)
    absb = np.abs(wide(b)) if b is not None else 0.0
    K = x.shape[1]
    bound = U * np.abs(ref) + (K + 1) * EPS * (np.abs(wide(xs)) @ np.abs(wide(w)) + absb)
    err = np.abs(ys - ref)
    assert np.isfinite(ys).all()
    worst = (err / bound).max()
    assert worst <= 1.0, f"max err / bound {worst:.3f}"
    qbound = np.sqrt((U / 2 * ref) ** 2 + ((K + 1) * EPS / 2) ** 2 * ((wide(xs) ** 2) @ (wide(w) ** 2)))
    assert np.linalg.norm(err) <= np.linalg.norm(qbound), "error above its quadrature bound"


def run(x, w, b):
    M, N = x.shape[0], w.shape[1]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    attn.attn_linear(dev(x), dev(w), y, dev(b))
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


# row tails (M not a multiple of 128), a column tail inside a 256-wide block (N = 264),
# a K tail inside a 64-deep step (K = 72), one row, no bias, several waves of tiles
@pytest.mark.parametrize("M,N,K,bias", [(300, 512, 1024, True), (1, 264, 72, True), (513, 1024, 512, False),
                                        (389, 256, 64, True), (128, 8, 8, True), (4000, 768, 1024, True)])
def test_linear_matches_oracle(orc, M, N, K, bias):
    x, w, b = draw(9000 + M + N + K, M, N, K, bias)
    check(orc, x, w, b, run(x, w, b))


def test_linear_cluster_path_odd_row_blocks(orc):
    """A launch of many tiles runs on 2-CTA clusters (row blocks 2u, 2u + 1 together).
    33 row blocks (M = 4103) x 32 column blocks: the last pair's second CTA lies wholly
    past M and must write nothing; sampled rows of every row block edge against the
    oracle, and the rows past M of a guarded buffer untouched."""
    M, N, K = 4103, 8192, 64
    x, w, b = draw(9300, M, N, K)
    pad_rows = 40
    buf = torch.full(((M + pad_rows) * N,), -7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[:M * N].view(M, N)
    attn.attn_linear(dev(x), dev(w), y, dev(b))
    torch.cuda.synchronize()
    assert torch.all(buf[M * N:] == -7.0)
    rows = sorted({0, 1, 127, 128, M // 2, 4095, 4096, M - 2, M - 1} | set(range(5, M, 37)))
    check(orc, x, w, b, y.float().cpu().numpy().astype(np.float64), np.array(rows))


def test_linear_pair_path_tails(orc):
    """A launch of at least 512 tiles runs the 2-SM MMA (two CTAs of a cluster, one
    M256 N256 MMA stream on both SMs). 33 row blocks (M = 4100: the last pair's first
    CTA holds 4 rows, its second none), 17 column blocks (N = 4104: the last holds 8
    columns, so the second CTA's half of that W tile lies wholly past N), K = 200 (a
    K tail inside the fourth 64-deep step): sampled rows against the oracle, all
    columns, and the rows past M of a guarded buffer untouched."""
    M, N, K = 4100, 4104, 200
    x, w, b = draw(9400, M, N, K)
    pad_rows = 40
    buf = torch.full(((M + pad_rows) * N,), -7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[:M * N].view(M, N)
    attn.attn_linear(dev(x), dev(w), y, dev(b))
    torch.cuda.synchronize()
    assert torch.all(buf[M * N:] == -7.0)
    rows = sorted({0, 1, 127, 128, 255, 256, M // 2, 4095, 4096, M - 1} | set(range(7, M, 41)))
    check(orc, x, w, b, y.float().cpu().numpy().astype(np.float64), np.array(rows))


def test_linear_pair_path_split_last_round(orc):
    """When the grid's last round of tiles is partly filled and their halves fit in one
    round, those tiles run as two 128-column halves (M256 N128 on the SM pair). 86 row
    blocks (M = 11000: the last pair's second CTA lies past M) x 6 column blocks (N =
    1288: the last holds 8 columns) = 258 pair tiles; on 76 SM pairs the last 30 run as
    halves. K = 200 ends inside a 64-deep step. Sampled rows, denser over the last five
    row pairs, against the oracle on all columns."""
    M, N, K = 11000, 1288, 200
    x, w, b = draw(9500, M, N, K)
    y = run(x, w, b)
    rows = sorted({0, 1, 255, 256, 9727, 9728, 9729, 10879, 10880, M - 1} | set(range(3, M, 97))
                  | set(range(9728, M, 23)))
    check(orc, x, w, b, y, np.array(rows))


def test_linear_guard_bands_and_determinism():
    """Nothing is written outside y, and two calls give identical bits."""
    x, w, b = draw(9100, 300, 264, 136)
    n, pad = 300 * 264, 4096
    outs = []
    for _ in range(2):
        buf = torch.full((n + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
        y = buf[pad:pad + n].view(300, 264)
        attn.attn_linear(dev(x), dev(w), y, dev(b))
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -7.0) and torch.all(buf[pad + n:] == -7.0)
        outs.append(y.clone())
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("name", ["long_causal_b2_h16_n8192_d64", "long_none_b2_h16_n8192_d128"])
def test_linear_full_size_sampled_rows(orc, name):
    """The layer's projection at full size (x [B*n, d_model], W [d_model, h*d]: 16384
    x 1024 x 1024 at d = 64, 16384 x 2048 x 2048 at d = 128): sampled rows (tile edges,
    the ends, every 61st row) against the oracle."""
    wl = W.WORKLOADS[name]
    inp = W.make_mha_inputs(wl)
    x = inp["x_q"].reshape(-1, inp["d_model"])
    y = run(x, inp["w_q"], inp["b_q"])
    M = x.shape[0]
    rows = sorted({0, 1, 127, 128, 129, 255, 256, M // 2, M - 129, M - 128, M - 1} | set(range(3, M, 61)))
    check(orc, x, inp["w_q"], inp["b_q"], y, np.array(rows))


def test_linear_rejects_bad_arguments():
    x, w, b = draw(9200, 16, 16, 16)
    xd, wd, bd = dev(x), dev(w), dev(b)
    y = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    L = attn.lib()
    assert L.attn_linear(None, attn._ptr(wd), None, attn._ptr(y), 16, 16, 16, None) == attn.ATTN_ERR_INVALID
    assert L.attn_linear(attn._ptr(xd), attn._ptr(wd), None, attn._ptr(y), 0, 16, 16, None) == attn.ATTN_ERR_INVALID
    assert L.attn_linear(attn._ptr(xd), attn._ptr(wd), None, attn._ptr(y), 16, 12, 16, None) == \
        attn.ATTN_ERR_UNSUPPORTED
    assert L.attn_linear(attn._ptr(xd) + 2, attn._ptr(wd), None, attn._ptr(y), 16, 16, 16, None) == \
        attn.ATTN_ERR_INVALID
