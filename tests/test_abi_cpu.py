"""The C-ABI library loads, exports every symbol include/*.h declares, and rejects
bad arguments with the documented status codes -- all without a GPU (argument
validation returns before any CUDA call)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from transformer_scaled_dot_mha_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return attn.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    assert {"attn_fwd", "attn_fwd_f32", "attn_fault_status", "attn_status_string"} <= set(declared_functions())


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", attn.LIB_PATH], capture_output=True, text=True, check=True)
    exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_status_strings(L):
    for st in (0, -1, -2, -3, -4):
        assert attn.status_string(st).startswith("ATTN_")
    assert "unknown" in attn.status_string(12345)


VALID = dict(q=16, k=32, v=48, out=64, lse=None, B=1, h=1, n_q=8, n_k=8, d_k=64, d_v=64, scale=0.125,
             mask_mode=0, key_lens=None)


def call(L, fn="attn_fwd", **kw):
    a = dict(VALID, **kw)
    return getattr(L, fn)(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["h"], a["n_q"], a["n_k"], a["d_k"],
                          a["d_v"], a["scale"], a["mask_mode"], a["key_lens"], None)


@pytest.mark.parametrize("fn", ["attn_fwd", "attn_fwd_f32"])
@pytest.mark.parametrize("bad", [
    dict(q=None), dict(k=None), dict(v=None), dict(out=None),
    dict(B=0), dict(h=-1), dict(n_q=0), dict(n_k=0), dict(d_k=0), dict(d_v=0),
    dict(scale=float("inf")), dict(scale=float("nan")),
    dict(mask_mode=4), dict(mask_mode=-1),
    dict(mask_mode=1, n_k=9),                     # causal needs n_q == n_k
    dict(mask_mode=2, key_lens=None),             # key padding needs key_lens
    dict(mask_mode=2, key_lens=2),                # misaligned key_lens
    dict(lse=6),                                  # misaligned lse
    dict(B=1 << 16, h=1 << 16),                   # B*h overflows int32
])
def test_invalid_arguments(L, fn, bad):
    assert call(L, fn, **bad) == attn.ATTN_ERR_INVALID


def test_bf16_alignment_and_unsupported_shapes(L):
    assert call(L, q=8) == attn.ATTN_ERR_INVALID          # bf16 path needs 16-byte alignment
    assert call(L, out=72) == attn.ATTN_ERR_INVALID
    assert call(L, d_k=32, d_v=32) == attn.ATTN_ERR_UNSUPPORTED
    assert call(L, d_k=64, d_v=128) == attn.ATTN_ERR_UNSUPPORTED
    assert call(L, d_k=96, d_v=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call(L, "attn_fwd_f32", d_k=257) == attn.ATTN_ERR_UNSUPPORTED
    assert call(L, "attn_fwd_f32", q=18) == attn.ATTN_ERR_INVALID


def test_library_has_no_oracle_dependency():
    """The product library never links or names the oracle."""
    build.build()
    out = subprocess.run(["nm", "-D", attn.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert "oracle" not in out
    deps = subprocess.run(["readelf", "-d", attn.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert "liboracle" not in deps
    for src in glob.glob(os.path.join(ROOT, "transformer_scaled_dot_mha_gb300", "**", "*.*"), recursive=True):
        if src.endswith((".py", ".cu", ".cuh", ".h")):
            assert "import oracle" not in open(src).read() and "attn_oracle" not in open(src).read(), src


def test_decode_workspace_and_argument_checks(L):
    ws = attn.attn_decode_workspace_size
    assert ws(16, 16, 1, 8192, 64) > 0 and ws(16, 16, 1, 8192, 64) == ws(16, 16, 1, 8192, 64)
    assert ws(1, 1, 17, 100, 64) == 0 and ws(1, 1, 1, 100, 96) == 0 and ws(0, 1, 1, 100, 64) == 0
    # one query: one fp32 partial (d outputs, max, sum) per cache chunk of each (b, h); the
    # chunk count follows the resident warps, not the cache length, so it stays small
    for B, H, n, d in ((16, 16, 8192, 64), (32, 8, 2048, 64), (3, 5, 1000, 128), (1, 1, 1 << 24, 64)):
        nbytes = ws(B, H, 1, n, d)
        assert nbytes > 0 and nbytes % (B * H * (d + 2) * 4) == 0
        assert nbytes <= attn.NOALLOC_MAX_BYTES  # attn_decode_noalloc serves these shapes
    assert ws(1, 1, 1, 1 << 24, 64) < 4096 * 66 * 4
    need = ws(2, 3, 4, 500, 128)
    f = L.attn_decode
    ok = dict(q=16, k=32, v=48, out=64, lse=None, B=2, h=3, n_q=4, n_max=500, d=128, scale=0.088,
              lens=80, ws=96, nbytes=need)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["h"], a["n_q"], a["n_max"], a["d"],
                 a["scale"], a["lens"], a["ws"], a["nbytes"], None)
    assert call(nbytes=need - 1) == attn.ATTN_ERR_INVALID      # workspace too small
    assert call(ws=None) == attn.ATTN_ERR_INVALID
    assert call(lens=None) == attn.ATTN_ERR_INVALID
    assert call(ws=104) == attn.ATTN_ERR_INVALID               # misaligned workspace
    assert call(q=24) == attn.ATTN_ERR_INVALID
    assert call(n_q=0) == attn.ATTN_ERR_INVALID
    assert call(n_q=17) == attn.ATTN_ERR_UNSUPPORTED
    assert call(d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call(scale=float("nan")) == attn.ATTN_ERR_INVALID


def test_bwd_workspace_and_argument_checks(L):
    ws = attn.attn_bwd_workspace_size
    stats = 2 * 3 * 4 * 2 * 128 * 4  # 500 rows -> 4 tiles of 128, two floats per row
    assert ws(2, 3, 500, 64, attn.BWD_DETERMINISTIC) == stats and ws(2, 3, 500, 128, 0) == stats
    assert ws(2, 3, 500, 64, 0) == stats + 2 * 3 * 500 * 64 * 4  # + the fused schedule's fp32 dQ
    assert ws(0, 1, 1) == 0 and ws(1, 1, 0) == 0 and ws(1, 1, 8, 96) == 0 and ws(1, 1, 8, 64, 2) == 0
    need = ws(2, 3, 500, 64, 0)
    f = L.attn_bwd
    ok = dict(q=16, k=32, v=48, out=64, dout=80, lse=96, dq=112, dk=128, dv=144, B=2, h=3, n_q=500, n_k=500,
              d_k=64, d_v=64, scale=0.125, mask=1, lens=None, flags=0, ws=160, nbytes=need)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"], a["h"],
                 a["n_q"], a["n_k"], a["d_k"], a["d_v"], a["scale"], a["mask"], a["lens"], a["flags"], a["ws"],
                 a["nbytes"], None)
    assert call(nbytes=need - 1) == attn.ATTN_ERR_INVALID      # workspace too small
    for name in ("dout", "lse", "dq", "dk", "dv", "ws"):
        assert call(**{name: None}) == attn.ATTN_ERR_INVALID
    assert call(dk=136) == attn.ATTN_ERR_INVALID               # misaligned gradient
    assert call(n_k=400) == attn.ATTN_ERR_INVALID              # causal needs n_q == n_k
    assert call(mask=2) == attn.ATTN_ERR_INVALID               # key padding without key_lens
    assert call(d_k=96, d_v=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call(d_v=128) == attn.ATTN_ERR_UNSUPPORTED
    assert call(scale=float("inf")) == attn.ATTN_ERR_INVALID
    assert call(flags=2) == attn.ATTN_ERR_INVALID              # unknown flag
    # the deterministic schedule's workspace is too small for the fused one (d = 64, flags 0)
    assert call(nbytes=ws(2, 3, 500, 64, attn.BWD_DETERMINISTIC)) == attn.ATTN_ERR_INVALID


def test_host_forward_workspace_and_argument_checks(L):
    ws = attn.attn_fwd_host_workspace_size
    # 32 heads of 28160 input bytes: under the 8 MiB minimum chunk, so one chunk and one
    # slot of q 32*100*64*2, k and v 32*60*64*2, out as q, lse 32*100*4 (each 256-byte
    # aligned), after 16 key lengths padded to 256 bytes
    assert ws(16, 2, 100, 60, 64) == 256 + 409600 + 2 * 245760 + 409600 + 12800
    # 32 heads of n = 8192, 3 MiB of input each (minimum chunk 3 heads). Per head q, k,
    # v, out are 1 MiB each and lse 32 KiB.
    per_head = 4 * 8192 * 64 * 2 + 8192 * 4
    # no mask: a head's kernel (~17 us at 1 PFLOP/s) is over 0.6 of its copies (~21 us
    # at 200 GB/s), so eight equal chunks of 4 heads; four slots of 4 heads
    assert ws(2, 16, 8192, 8192, 64) == 256 + 16 * per_head
    # causal: half the kernel time, transfer-bound, so the ramp 3, 6, 12, 6, 5; the four
    # slots hold chunks {3, 5}, {6}, {12}, {6}
    assert ws(2, 16, 8192, 8192, 64, 1) == 256 + (5 + 6 + 12 + 6) * per_head
    assert ws(1, 1, 8, 8, 64, 4) == 0
    assert ws(1, 1, 1, 1, 96) == 0 and ws(0, 1, 1, 1, 64) == 0 and ws(1, 1, 1, 0, 64) == 0
    need = ws(2, 3, 500, 500, 64, 1)
    ok = dict(q=16, k=32, v=48, out=64, lse=None, B=2, h=3, n_q=500, n_k=500, d_k=64, d_v=64, scale=0.125,
              mask=1, lens=None, ws=256, nbytes=need)

    def call(**kw):
        a = dict(ok, **kw)
        return L.attn_fwd_host(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["h"], a["n_q"], a["n_k"],
                               a["d_k"], a["d_v"], a["scale"], a["mask"], a["lens"], a["ws"], a["nbytes"], None)
    assert call(nbytes=need - 1) == attn.ATTN_ERR_INVALID      # workspace too small
    assert call(ws=None) == attn.ATTN_ERR_INVALID
    assert call(ws=272) == attn.ATTN_ERR_INVALID               # workspace not 256-byte aligned
    for name in ("q", "k", "v", "out"):
        assert call(**{name: None}) == attn.ATTN_ERR_INVALID
    assert call(n_k=400) == attn.ATTN_ERR_INVALID              # causal needs n_q == n_k
    assert call(mask=2) == attn.ATTN_ERR_INVALID               # key padding without key_lens
    assert call(d_k=96, d_v=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call(d_v=128) == attn.ATTN_ERR_UNSUPPORTED
    assert call(scale=float("nan")) == attn.ATTN_ERR_INVALID


def test_host_gradients_workspace_and_argument_checks(L):
    ws = attn.attn_bwd_host_workspace_size
    # 6 heads of n = 300, d = 64: one chunk. One slot of Q, O, dO, dQ and K, V, dK, dV
    # (6*300*64*2 = 230400 bytes each), lse 6*300*4 = 7200 -> 7424, and the gradient
    # workspace of 6 heads: 3 tiles x 1024 bytes of statistics per head, plus the fused
    # schedule's fp32 dQ (300*64*4 per head); after 2 key lengths padded to 256 bytes.
    assert ws(2, 3, 300, 300, 64, 0, 0) == 256 + 8 * 230400 + 7424 + 6 * (3072 + 76800)
    assert ws(2, 3, 300, 300, 64, 0, attn.BWD_DETERMINISTIC) == 256 + 8 * 230400 + 7424 + 6 * 3072
    assert ws(1, 1, 8, 8, 96, 0, 0) == 0 and ws(1, 1, 8, 8, 64, 4, 0) == 0 and ws(1, 1, 8, 8, 64, 0, 2) == 0
    need = ws(2, 3, 300, 300, 64, 1, 0)
    ok = dict(q=16, k=32, v=48, out=64, dout=80, lse=96, dq=112, dk=128, dv=144, B=2, h=3, n_q=300, n_k=300,
              d_k=64, d_v=64, scale=0.125, mask=1, lens=None, flags=0, ws=256, nbytes=need)

    def call(**kw):
        a = dict(ok, **kw)
        return L.attn_bwd_host(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"],
                               a["B"], a["h"], a["n_q"], a["n_k"], a["d_k"], a["d_v"], a["scale"], a["mask"],
                               a["lens"], a["flags"], a["ws"], a["nbytes"], None)
    assert call(nbytes=need - 1) == attn.ATTN_ERR_INVALID      # workspace too small
    assert call(ws=272) == attn.ATTN_ERR_INVALID               # workspace not 256-byte aligned
    for name in ("dout", "lse", "dq", "dk", "dv", "ws"):
        assert call(**{name: None}) == attn.ATTN_ERR_INVALID
    assert call(flags=2) == attn.ATTN_ERR_INVALID
    assert call(n_k=200) == attn.ATTN_ERR_INVALID              # causal needs n_q == n_k
    assert call(mask=2) == attn.ATTN_ERR_INVALID               # key padding without key_lens
    assert call(d_k=96, d_v=96) == attn.ATTN_ERR_UNSUPPORTED


def test_weights_argument_checks(L):
    """attn_weights rejects bad arguments before touching the device (no GPU needed)."""
    ok = dict(q=16, k=32, lse=48, w=64, B=1, h=1, n_q=8, n_k=8, d=64, scale=0.125, mask_mode=0, key_lens=None)

    def cw(**kw):
        a = dict(ok, **kw)
        return L.attn_weights(a["q"], a["k"], a["lse"], a["w"], a["B"], a["h"], a["n_q"], a["n_k"], a["d"],
                              a["scale"], a["mask_mode"], a["key_lens"], None)

    for bad in (dict(q=None), dict(k=None), dict(lse=None), dict(w=None), dict(B=0), dict(n_k=0),
                dict(scale=float("nan")), dict(mask_mode=4), dict(mask_mode=1, n_k=9), dict(mask_mode=2),
                dict(w=72), dict(q=8), dict(lse=50), dict(B=1 << 20, h=1 << 10, n_q=1 << 16, n_k=1 << 16)):
        assert cw(**bad) == attn.ATTN_ERR_INVALID, bad
    assert cw(d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert cw(d=32) == attn.ATTN_ERR_UNSUPPORTED
