"""The forward kernel's bounded-wait abort path, driven to its limit on the GPU.

Every mbarrier wait in the forward kernel is bounded in time. A wait that runs out
records a fault bit, raises the CTA's abort flag, and every role then stops: the
producer lets its copies in flight land, the MMA issuers wait for their MMAs, TMEM is
freed and the CTA returns, writing nothing. Nothing traps, and the context stays
usable. Here the library's fault-injection instantiation of the d = 64 kernel (waits
shortened to a millisecond; the producer stops before the V copy of one K/V tile and
drains the copies it did issue) makes the PV issuer's wait for that tile run out. The
test checks the reported status and bits, that no output row was written, and that
the next ordinary call on the same stream matches the oracle.
"""
import numpy as np
import pytest
import torch

from transformer_scaled_dot_mha_gb300 import attn, workloads as W

pytestmark = pytest.mark.gpu

FAULT_MMA, FAULT_SOFTMAX = 2, 4


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def test_wait_timeout_aborts_reports_and_recovers(orc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, k, v, _ = W.make_inputs(w, seed=8100, B=1, H=2, n_q=512, n_k=512)
    qd, kd, vd = _dev_bf16(q), _dev_bf16(k), _dev_bf16(v)
    st, code = attn.attn_fault_status(clear=True)
    assert st == attn.ATTN_OK, f"fault record {code:#x} before the test"

    # every CTA visits four K/V tiles; the V copy of tile 1 is never issued
    out = torch.full_like(qd, -7.0)
    lse = torch.full((1, 2, 512), -7.0, device="cuda")
    attn._internal_arm_wait_timeout(1_000_000, 1)
    attn.attn_fwd(qd, kd, vd, out, lse, w.scale, attn.MASK_NONE)
    st, code = attn.attn_fault_status(clear=True)
    assert st == attn.ATTN_ERR_TIMEOUT
    assert code != 0 and code & ~(FAULT_MMA | FAULT_SOFTMAX) == 0, f"fault bits {code:#x}"
    assert torch.all(out == -7.0) and torch.all(lse == -7.0)  # aborted CTAs write nothing
    st, code = attn.attn_fault_status(clear=False)
    assert st == attn.ATTN_OK and code == 0  # the record was cleared

    # the next ordinary call on the same stream runs to completion and matches the oracle
    attn.attn_fwd(qd, kd, vd, out, lse, w.scale, attn.MASK_NONE)
    st, code = attn.attn_fault_status(clear=True)
    assert st == attn.ATTN_OK, f"fault record {code:#x} after recovery"
    ref, ref_lse = orc.attention(q, k, v, w.scale, 0)
    err = np.abs(out.float().cpu().numpy() - ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3
