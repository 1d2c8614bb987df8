"""attn_decode (one generation step against a key/value cache) against the fp64
oracle's decode mask, element by element on the same bf16-rounded inputs.

Tolerance: max |err| <= 1e-2, mean |err| <= 1e-3, lse |err| <= 1e-3 -- the same
bar as the bf16 forward path (this kernel keeps the weights in fp32, so its only
bf16 rounding is the output's, at most 2^-8 relative).
"""
import numpy as np
import pytest
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu
DEC = W.MASK_DECODE


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


def run_decode(q, k, v, lens, scale, ws_fill=None):
    B, H, n_q, d = q.shape
    n_max = k.shape[2]
    nbytes = attn.attn_decode_workspace_size(B, H, n_q, n_max, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if ws_fill is not None:
        ws.fill_(ws_fill)
    qd = dev_bf16(q)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device="cuda")
    attn.attn_decode(qd, dev_bf16(k), dev_bf16(v), out, torch.from_numpy(lens).cuda(), ws, lse, scale)
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
@pytest.mark.parametrize("n_q", [1, 3, 16])
@pytest.mark.parametrize("n_max", [1, 100, 300, 1000])
def test_decode_ragged(orc, d, n_q, n_max):
    w = W.WORKLOADS["decode_b32_h8_q1_k2048_d64"]
    q, k, v, _ = W.make_inputs(w, seed=5000 + d + n_q + n_max, B=4, H=2, n_q=n_q, n_k=n_max, d_k=d, d_v=d)
    # valid cache lengths only (0 .. n_max), incl. empty and shorter than n_q
    lens = np.minimum(np.array([n_max, max(0, n_q - 1), 1, (n_max * 2) // 3], np.int32), n_max)
    out, lse = run_decode(q, k, v, lens, W.default_scale(d), ws_fill=0xFF)  # NaN-filled workspace
    ref, ref_lse = orc.attention(q, k, v, W.default_scale(d), DEC, lens)
    check(out, lse, ref, ref_lse)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_one_query_chunk_and_tile_edges(orc, d):
    """One query per (b, h) runs one warp per cache chunk: for 8 heads and a 4096-key
    cache that is 32 chunks of 128 keys in 32-key tiles. Cache lengths on and beside
    those boundaries, a length inside the first tile, and the full cache."""
    w = W.WORKLOADS["decode_b32_h8_q1_k2048_d64"]
    q, k, v, _ = W.make_inputs(w, seed=5300 + d, B=8, H=1, n_q=1, n_k=4096, d_k=d, d_v=d)
    lens = np.array([896, 897, 895, 31, 32, 33, 4096, 4095], np.int32)
    out, lse = run_decode(q, k, v, lens, W.default_scale(d), ws_fill=0xFF)  # NaN-filled workspace
    ref, ref_lse = orc.attention(q, k, v, W.default_scale(d), DEC, lens)
    check(out, lse, ref, ref_lse)


def test_decode_equals_last_rows_of_causal_forward(orc):
    """The decode step and the causal forward kernel agree on the newest positions."""
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, k, v, _ = W.make_inputs(w, seed=5100, B=1, H=2, n_q=300, n_k=300)
    n_q = 5
    lens = np.array([300], np.int32)
    dq, dl = run_decode(np.ascontiguousarray(q[:, :, -n_q:]), k, v, lens, w.scale)
    fo, fl = attn.attention(dev_bf16(q), dev_bf16(k), dev_bf16(v), w.scale, W.MASK_CAUSAL, with_lse=True)
    fo = fo.float().cpu().numpy()[:, :, -n_q:]
    assert np.abs(dq - fo).max() <= 1.5e-2
    assert np.abs(dl - fl.cpu().numpy()[:, :, -n_q:]).max() <= 1e-3


def test_decode_repeated_calls_reuse_workspace(orc):
    w = W.WORKLOADS["decode_b32_h8_q1_k2048_d64"]
    q, k, v, lens = W.make_inputs(w, seed=5200, B=2, H=3, n_k=700)
    B, H, n_q, d = q.shape
    ws = torch.empty(attn.attn_decode_workspace_size(B, H, n_q, 700, d), dtype=torch.uint8, device="cuda")
    qd, kd, vd, ld = dev_bf16(q), dev_bf16(k), dev_bf16(v), torch.from_numpy(lens).cuda()
    outs = []
    for _ in range(2):
        out = torch.empty_like(qd)
        attn.attn_decode(qd, kd, vd, out, ld, ws, None, w.scale)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1])
    ref, _ = orc.attention(q, k, v, w.scale, DEC, lens)
    assert np.abs(outs[0].float().cpu().numpy() - ref).max() <= 1e-2


@pytest.mark.parametrize("name", ["decode_b32_h8_q1_k2048_d64", "decode_b16_h16_q1_k8192_d64"])
def test_decode_full_size_workloads(orc, name):
    w = W.WORKLOADS[name]
    q, k, v, lens = W.make_inputs(w)
    out, lse = run_decode(q, k, v, lens, w.scale)
    ref, ref_lse = orc.attention(q, k, v, w.scale, DEC, lens)
    check(out, lse, ref, ref_lse)
