"""attn_fwd_local (restricted self-attention, |i - j| <= window) against the oracle's
window mask on the same bf16-rounded inputs; bf16 tolerances as in
test_parity_gpu.py (max |err| <= 1e-2, mean <= 1e-3, lse <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
C, P, WIN = W.MASK_CAUSAL, W.MASK_KEY_PADDING, W.MASK_WINDOW


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


def run_local(q, k, v, kl, scale, window, mode):
    qd = dev_bf16(q)
    out = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    kld = torch.from_numpy(kl).cuda() if mode & P else None
    attn.attn_fwd_local(qd, dev_bf16(k), dev_bf16(v), out, window, lse, scale, mode, kld)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check(out, lse, ref, ref_lse):
    err = np.abs(out - ref)
    assert np.isfinite(out).all()
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, f"max {err.max():.3e} mean {err.mean():.3e}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin) and np.all(lse[~fin] == -np.inf)
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-3


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [0, 1, 63, 127, 128, 200, 1000])
@pytest.mark.parametrize("mode", [0, C, P, C | P])
def test_local_window(orc, d, window, mode):
    w = W.WORKLOADS["local_causal_b2_h16_n8192_d64_w511"]
    q, k, v, _ = W.make_inputs(w, seed=6000 + d + window + mode, B=2, H=2, n_q=700, n_k=700, d_k=d, d_v=d)
    kl = np.array([700, 333], np.int32)
    out, lse = run_local(q, k, v, kl, W.default_scale(d), window, mode)
    ref, ref_lse = orc.attention(q, k, v, W.default_scale(d), mode | WIN, kl, window=window)
    check(out, lse, ref, ref_lse)


def test_local_window_covering_everything_equals_attn_fwd():
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, k, v, kl = W.make_inputs(w, seed=6100, B=1, H=2, n_q=400, n_k=400)
    a, _ = run_local(q, k, v, kl, w.scale, 400, C)
    b = attn.attention(dev_bf16(q), dev_bf16(k), dev_bf16(v), w.scale, C).float().cpu().numpy()
    assert np.array_equal(a, b)
    c, _ = run_local(q, k, v, kl, w.scale, 2**31 - 1, C)  # the widest window an int holds
    assert np.array_equal(a, c)


def test_local_full_size_sampled_rows(orc):
    w = W.WORKLOADS["local_causal_b2_h16_n8192_d64_w511"]
    q, k, v, kl = W.make_inputs(w)
    out, lse = run_local(q, k, v, kl, w.scale, w.window, w.mask_mode & ~WIN)
    rows = sorted({0, 1, 255, 256, 510, 511, 512, 513, 4095, 4096, 8190, 8191} | set(range(7, 8192, 131)))
    ids = np.array([(b * w.H + h) * w.n_q + i for b, h in ((0, 0), (1, 15)) for i in rows], np.int64)
    ref, ref_lse = orc.attention_rows(q, k, v, w.scale, ids, w.mask_mode, kl, window=w.window)
    check(out.reshape(-1, w.d_v)[ids], lse.reshape(-1)[ids], ref, ref_lse)
