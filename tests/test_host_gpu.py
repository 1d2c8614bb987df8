"""attn_fwd_host -- the forward on operands in host memory -- against attn_fwd.

The host entry point cuts the flattened (b, h) head range into chunks (at least
8 MiB of input each; a ramp up and down by halves when the copies bound the call,
eight equal chunks otherwise) and runs the same attention kernel on each chunk, with the kernel variant chosen for the whole problem, so its output and lse
must equal attn_fwd's on the device copies bit for bit. The cases cover a single
chunk, chunks that start or end inside a batch (one, two and three rectangles per
chunk, each with its batches' key lengths), more chunks than ring slots (slot reuse
inside a call), back-to-back calls with no synchronisation between them (slot reuse
across calls), pageable host memory, and the full-size long-sequence and encoder
workloads. One small case is also checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu

C, P = W.MASK_CAUSAL, W.MASK_KEY_PADDING


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.lib()
    yield
    st, code = attn.attn_fault_status()
    assert st == attn.ATTN_OK, f"kernel fault record {code:#x}"


def host_bf16(a, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def run_both(q, k, v, kl, scale, mode, pin=True):
    B, H, n_q, d = q.shape
    n_k = k.shape[2]
    qh, kh, vh = (host_bf16(a, pin) for a in (q, k, v))
    klh = torch.from_numpy(kl.copy())
    outh = torch.full((B, H, n_q, d), float("nan"), dtype=torch.bfloat16)
    lseh = torch.full((B, H, n_q), float("nan"), dtype=torch.float32)
    if pin:
        klh, outh, lseh = klh.pin_memory(), outh.pin_memory(), lseh.pin_memory()
    ws = torch.empty(attn.attn_fwd_host_workspace_size(B, H, n_q, n_k, d, mode), dtype=torch.uint8, device="cuda")
    attn.attn_fwd_host(qh, kh, vh, outh, ws, lseh, scale, mode, klh if mode & P else None)
    torch.cuda.synchronize()
    kl_d = klh.cuda() if mode & P else None
    out_d, lse_d = attn.attention(qh.cuda(), kh.cuda(), vh.cuda(), scale, mode, kl_d, with_lse=True)
    torch.cuda.synchronize()
    return outh, lseh, out_d.cpu(), lse_d.cpu()


def assert_identical(outh, lseh, out_d, lse_d):
    assert torch.equal(outh.view(torch.int16), out_d.view(torch.int16)), "output differs from attn_fwd"
    assert torch.equal(lseh.view(torch.int32), lse_d.view(torch.int32)), "lse differs from attn_fwd"


CASES = [
    # (B, H, n_q, n_k, d, mask, key length range); input bytes per head 3 * n * d * 2
    (9, 2, 200, 200, 64, P, (64, 200)),          # one chunk
    (10, 5, 2048, 2048, 64, P, (1000, 2048)),    # ramp 11, 20, 19: the 20 is three rectangles
    (7, 4, 2048, 2048, 64, C | P, (1, 2048)),    # ramp 11, 17, split inside batch 2
    (3, 5, 4096, 4096, 128, 0, None),            # ramp 3, 6, 3, 3 at d = 128
    (3, 5, 8192, 8192, 64, P, (4096, 8192)),     # five equal chunks of 3 heads: four slots, reused
    (3, 4, 1000, 3000, 64, P, (1, 3000)),        # cross-attention, n_q != n_k, one chunk
    (2, 3, 300, 300, 64, C | P, (150, 300)),     # ragged rows, one chunk
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}_q{}_k{}_d{}_m{}".format(*c[:6]))
def test_host_forward_equals_device_forward(case):
    B, H, n_q, n_k, d, mode, lens = case
    w = W.WORKLOADS["cross_pad_b16_h16_q256_k512_d64"]
    q, k, v, _ = W.make_inputs(w, B=B, H=H, n_q=n_q, n_k=n_k, d_k=d, d_v=d)
    rng = np.random.Generator(np.random.PCG64(11))
    kl = rng.integers(*lens, size=B, endpoint=True).astype(np.int32) if lens else np.full(B, n_k, np.int32)
    assert_identical(*run_both(q, k, v, kl, d ** -0.5, mode))


def test_host_forward_against_oracle():
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, k, v, kl = W.make_inputs(w, B=5, H=2, n_q=160, n_k=160)
    outh, lseh, _, _ = run_both(q, k, v, kl, w.scale, w.mask_mode)
    ref, ref_lse = oracle.Oracle().attention(q, k, v, w.scale, w.mask_mode)
    err = np.abs(outh.float().numpy().astype(np.float64) - ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, f"max {err.max()} mean {err.mean()}"
    assert np.abs(lseh.numpy() - ref_lse).max() <= 1e-3


def test_pageable_host_memory():
    w = W.WORKLOADS["cross_pad_b16_h16_q256_k512_d64"]
    q, k, v, kl = W.make_inputs(w, B=5, H=3, n_q=64, n_k=200)
    assert_identical(*run_both(q, k, v, kl, w.scale, w.mask_mode, pin=False))


def test_back_to_back_calls_share_the_ring():
    """Two calls queued with no synchronisation reuse the same ring slots: the second
    call's copies in must wait for the first call's copies out."""
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    B, H, n = 2, 8, 512
    ins = [W.make_inputs(w, seed=s, B=B, H=H, n_q=n, n_k=n) for s in (21, 22)]
    ws = torch.empty(attn.attn_fwd_host_workspace_size(B, H, n, n, 64, C), dtype=torch.uint8, device="cuda")
    outs, keep = [], []  # the host buffers must outlive the asynchronous copies
    for q, k, v, _ in ins:
        o = torch.empty((B, H, n, 64), dtype=torch.bfloat16).pin_memory()
        hq, hk, hv = host_bf16(q), host_bf16(k), host_bf16(v)
        attn.attn_fwd_host(hq, hk, hv, o, ws, None, w.scale, C)
        outs.append(o)
        keep += [hq, hk, hv]
    torch.cuda.synchronize()
    for (q, k, v, _), o in zip(ins, outs):
        ref = attn.attention(host_bf16(q).cuda(), host_bf16(k).cuda(), host_bf16(v).cuda(), w.scale, C).cpu()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name", ["long_causal_b2_h16_n8192_d64", "long_none_b2_h16_n8192_d64",
                                  "encoder_self_pad_b32_h8_n128_d64"])
def test_full_size_workloads(name):
    """The bench's end-to-end configurations: the ramp 3, 6, 12, 6, 5 and eight equal
    chunks of 4 heads of n = 8192, and one chunk of 256 heads of n = 128; every chunk
    runs the kernel instantiation the whole problem runs (one Q tile per CTA at d = 64)."""
    w = W.WORKLOADS[name]
    q, k, v, kl = W.make_inputs(w)
    assert_identical(*run_both(q, k, v, kl, w.scale, w.mask_mode))


# ------------------------------------------------------------------ gradients on host operands
BWD_CASES = [
    # (B, H, n, d, mask, flags); plans from 8 MiB minimum chunks and the copy/kernel time ratio
    (7, 4, 2048, 64, C | P, 0),                        # ramp 7, 11, 10: the 11 is three rectangles; fused
    (7, 4, 2048, 64, C | P, attn.BWD_DETERMINISTIC),   # the same, deterministic schedule
    (5, 6, 2048, 128, 0, 0),                           # ramp 4, 8, 9, 5, 4: five chunks, four slots; d = 128
    (2, 3, 300, 64, C | P, 0),                         # ragged rows, one chunk
]


def run_bwd_both(q, k, v, g, kl, scale, mode, flags):
    """attn_bwd_host on pinned host tensors and attn_bwd on device copies, both given the
    device forward's out and lse."""
    B, H, n, d = q.shape
    qh, kh, vh, gh = (host_bf16(a) for a in (q, k, v, g))
    kl_d = torch.from_numpy(kl.copy()).cuda() if mode & P else None
    qd, kd, vd, gd = qh.cuda(), kh.cuda(), vh.cuda(), gh.cuda()
    out_d, lse_d = attn.attention(qd, kd, vd, scale, mode, kl_d, with_lse=True)
    grads_d = [torch.empty_like(t) for t in (qd, kd, vd)]
    ws_d = torch.empty(attn.attn_bwd_workspace_size(B, H, n, d, flags), dtype=torch.uint8, device="cuda")
    attn.attn_bwd(qd, kd, vd, out_d, gd, lse_d, *grads_d, ws_d, scale, mode, kl_d, flags=flags)
    outh, lseh = out_d.cpu().pin_memory(), lse_d.cpu().pin_memory()
    klh = torch.from_numpy(kl.copy()).pin_memory() if mode & P else None
    grads_h = [torch.full(t.shape, float("nan"), dtype=torch.bfloat16).pin_memory() for t in (qd, kd, vd)]
    ws_h = torch.empty(attn.attn_bwd_host_workspace_size(B, H, n, n, d, mode, flags), dtype=torch.uint8,
                       device="cuda")
    attn.attn_bwd_host(qh, kh, vh, outh, gh, lseh, *grads_h, ws_h, scale, mode, klh, flags=flags)
    torch.cuda.synchronize()
    return [t.cpu() for t in grads_d], grads_h


def assert_bwd_match(grads_d, grads_h, bitwise_dq):
    U = 2.0 ** -8
    for name, gd, gh in zip(("dq", "dk", "dv"), grads_d, grads_h):
        if name != "dq" or bitwise_dq:
            assert torch.equal(gd.view(torch.int16), gh.view(torch.int16)), f"{name} differs from attn_bwd"
        else:  # the fused schedule's dq: reduce order varies between the two calls
            a, b = gd.float(), gh.float()
            assert torch.all((a - b).abs() <= 4 * U * a.abs() + 1e-6), f"dq differs by {(a - b).abs().max()}"


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "B{}_H{}_n{}_d{}_m{}_f{}".format(*c))
def test_host_gradients_equal_device_gradients(case):
    B, H, n, d, mode, flags = case
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, k, v, _ = W.make_inputs(w, seed=31, B=B, H=H, n_q=n, n_k=n, d_k=d, d_v=d)
    g = W.make_grad_output(w, seed=31, B=B, H=H, n_q=n, d_v=d)
    rng = np.random.Generator(np.random.PCG64(12))
    kl = rng.integers(1, n, size=B, endpoint=True).astype(np.int32) if mode & P else np.full(B, n, np.int32)
    grads_d, grads_h = run_bwd_both(q, k, v, g, kl, d ** -0.5, mode, flags)
    assert_bwd_match(grads_d, grads_h, bitwise_dq=(d == 128 or flags & attn.BWD_DETERMINISTIC))


def test_host_gradients_full_size():
    """The bench's gradient workload: eight equal chunks of 4 heads of n = 8192, fused."""
    w = W.WORKLOADS["long_causal_b2_h16_n8192_d64"]
    q, k, v, kl = W.make_inputs(w)
    g = W.make_grad_output(w)
    grads_d, grads_h = run_bwd_both(q, k, v, g, kl, w.scale, w.mask_mode, 0)
    assert_bwd_match(grads_d, grads_h, bitwise_dq=False)
