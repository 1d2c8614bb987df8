"""Pins that tie the fp64 oracle to something other than itself.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` when the oracle
disagrees with what the pages or the mathematics fix: values the pages print for
their worked examples (``tests/golden``), closed forms, invariants, special cases
that reduce to a library routine, and brute force on tiny inputs. The pins are
chosen so that a plausible slip in the oracle (a dropped scale, a transposed
operand, a flipped or off-by-one mask, a wrong stride, a missing normalisation)
fails at least one of them; ``test_oracle_mutants.py`` plants such slips in a copy
of the oracle's C source and checks that.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
C, P, DEC, WIN = oracle.MASK_CAUSAL, oracle.MASK_KEY_PADDING, oracle.MASK_DECODE, oracle.MASK_WINDOW


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _h(x):
    """[n, d] -> [1, 1, n, d] float64."""
    return np.asarray(x, np.float64)[None, None]


def _rand(seed, B, H, n_q, n_k, d_k, d_v):
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal((B, H, n_q, d_k)), rng.standard_normal((B, H, n_k, d_k)),
            rng.standard_normal((B, H, n_k, d_v)))


# ---------------------------------------------------------------- worked examples
def pin_two_token_printed(orc):
    """attention-paper-guide section 03.2: the page's own printed numbers."""
    g = _golden("two_token_example.json")
    sc = 1.0 / math.sqrt(g["d_k"])
    Q, K, V = _h(g["Q"]), _h(g["K"]), _h(g["V"])
    out, _ = orc.attention(Q, K, V, sc)
    w = orc.attention_weights(Q, K, sc)[0, 0]
    pr, tol = g["printed"], g["tolerance_from_printing"]
    assert np.allclose(np.asarray(g["Q"]) @ np.asarray(g["K"]).T, pr["scores_unscaled"])
    assert np.abs(np.log(w[:, 1] / w[:, 0]) - (np.array(pr["scores_scaled"])[:, 1] - np.array(pr["scores_scaled"])[:, 0])).max() < 2 * tol["scores_scaled"]
    assert np.abs(w - pr["weights"]).max() <= tol["weights"]
    assert np.abs(out[0, 0] - pr["output"]).max() <= tol["output"]
    assert np.abs(out[0, 0, 1] - pr["output_row1_in_text"]).max() <= tol["output_row1_in_text"]


def pin_two_token_closed_form(orc):
    """The same example solved by hand.

    Scaled scores are [c, c] for query 0 and [0, c] for query 1 with c = 1/sqrt(2).
    Query 0 therefore weights both keys 1/2: o_0 = (10/2, 6/2) = (5, 3) and
    lse_0 = c + ln 2. Query 1 weights them 1/(1+e^c) and e^c/(1+e^c):
    o_1 = (10/(1+e^c), 6 e^c/(1+e^c)) and lse_1 = ln(1 + e^c).
    """
    g = _golden("two_token_example.json")
    c = 1.0 / math.sqrt(2.0)
    out, lse = orc.attention(_h(g["Q"]), _h(g["K"]), _h(g["V"]), c)
    e = math.exp(c)
    want = np.array([[5.0, 3.0], [10.0 / (1.0 + e), 6.0 * e / (1.0 + e)]])
    assert np.abs(out[0, 0] - want).max() < 1e-13
    assert abs(lse[0, 0, 0] - (c + math.log(2.0))) < 1e-13
    assert abs(lse[0, 0, 1] - math.log1p(e)) < 1e-13


def pin_running_example_unmasked(orc):
    """rockcohen.cc section 5.1 ledger: S, A and z_0 from the printed Q, K, V."""
    g = _golden("running_example_4token.json")
    sc = 1.0 / math.sqrt(g["d_k"])
    Q, K, V = _h(g["Q"]), _h(g["K"]), _h(g["V"])
    pr, tol = g["printed"], g["tolerance"]
    assert abs(float(np.dot(g["Q"][0], g["K"][1])) - pr["q0_dot_k1_unscaled"]) <= tol["q0_dot_k1_unscaled"]
    # one-key-at-a-time calls expose the scaled score itself: with a single legal
    # key, lse = ln exp(s) = s
    for j in range(4):
        _, lse = orc.attention(Q, K[:, :, j:j + 1], V[:, :, j:j + 1], sc)
        assert np.abs(lse[0, 0] - np.asarray(pr["S_scaled"])[:, j]).max() <= tol["S_scaled"]
    w = orc.attention_weights(Q, K, sc)[0, 0]
    assert np.abs(w - pr["A"]).max() <= tol["A"]
    out, _ = orc.attention(Q, K, V, sc)
    assert np.abs(out[0, 0, 0] - pr["z0"]).max() <= tol["z0"]


def pin_running_example_causal(orc):
    """rockcohen.cc sections 5.3 and 6.3: causal rows, exact zeros above the diagonal."""
    g = _golden("running_example_4token.json")
    sc = 1.0 / math.sqrt(g["d_k"])
    Q, K, V = _h(g["Q"]), _h(g["K"]), _h(g["V"])
    w = orc.attention_weights(Q, K, sc, C)[0, 0]
    pr, tol = g["printed"], g["tolerance"]
    assert np.array_equal(w[0], np.array(pr["causal_A_row0"], np.float64))
    assert np.abs(w[1] - pr["causal_A_row1"]).max() <= tol["causal"]
    assert np.all(w[np.triu_indices(4, 1)] == 0.0)
    out, _ = orc.attention(Q, K, V, sc, C)
    assert np.array_equal(out[0, 0, 0], np.asarray(g["V"], np.float64)[0])


def pin_softmax_example(orc):
    """rockcohen.cc section 3.2: softmax of (3.2, 0.1, -2.5, 0.4)."""
    g = _golden("softmax_example.json")
    q = np.ones((1, 1, 1, 1))
    k = np.asarray(g["scores"], np.float64).reshape(1, 1, 4, 1)
    out, _ = orc.attention(q, k, np.eye(4)[None, None], 1.0)
    assert np.all(np.abs(out[0, 0, 0] - g["printed_weights"]) <= np.asarray(g["tolerance_from_printing"]))


# ---------------------------------------------------------------- invariants
def pin_rows_sum_to_one_and_exact_zeros(orc):
    """rockcohen.cc section 10.2 (P0b, P0c): rows sum to 1; illegal weights are exactly 0.0."""
    q, k, _ = _rand(11, 2, 2, 7, 9, 5, 3)
    kl = np.array([4, 9], np.int32)
    for mode in (0, C, P, C | P):
        n_k = 7 if mode & C else 9
        w = orc.attention_weights(q, k[:, :, :n_k], 0.4, mode, kl)
        assert np.abs(w.sum(-1) - 1.0).max() < 1e-13
        illegal = ~oracle.legal_mask(2, 7, n_k, mode, kl)
        assert np.all(w[np.broadcast_to(illegal, w.shape)] == 0.0)
        assert np.all(w[np.broadcast_to(~illegal, w.shape)] > 0.0)


def pin_permutation_equivariance(orc):
    """rockcohen.cc section 6.2: permuting query rows permutes the output rows; permuting
    key/value rows jointly leaves the output unchanged (no mask)."""
    q, k, v = _rand(12, 1, 2, 6, 8, 4, 5)
    out, lse = orc.attention(q, k, v, 0.5)
    pq = np.random.Generator(np.random.PCG64(1)).permutation(6)
    pk = np.random.Generator(np.random.PCG64(2)).permutation(8)
    out_q, lse_q = orc.attention(q[:, :, pq], k, v, 0.5)
    assert np.abs(out_q - out[:, :, pq]).max() < 1e-13 and np.abs(lse_q - lse[:, :, pq]).max() < 1e-13
    out_k, lse_k = orc.attention(q, k[:, :, pk], v[:, :, pk], 0.5)
    assert np.abs(out_k - out).max() < 1e-13 and np.abs(lse_k - lse).max() < 1e-13


def pin_shift_invariance(orc):
    """rockcohen.cc section 3.2: adding one constant to every score of a row changes
    nothing. K + 1 u^T adds q_i . u to row i, so O is unchanged and lse moves by
    scale * q_i . u."""
    q, k, v = _rand(13, 1, 1, 5, 6, 3, 2)
    u = np.array([0.7, -1.3, 2.1])
    out, lse = orc.attention(q, k, v, 0.6, P, np.array([4], np.int32))
    out2, lse2 = orc.attention(q, k + u, v, 0.6, P, np.array([4], np.int32))
    assert np.abs(out2 - out).max() < 1e-12
    assert np.abs(lse2 - (lse + 0.6 * (q @ u))).max() < 1e-12


def pin_zero_query_is_mean_of_legal_values(orc):
    """Closed form: with Q = 0 every legal score is 0, so o_i is the plain mean of the
    legal V rows (causal: rows 0..i; key padding: rows 0..len-1)."""
    _, k, v = _rand(14, 2, 1, 5, 5, 3, 4)
    q = np.zeros((2, 1, 5, 3))
    kl = np.array([3, 5], np.int32)
    out, lse = orc.attention(q, k, v, 0.5, C | P, kl)
    for b in range(2):
        for i in range(5):
            n = min(i + 1, kl[b])
            assert np.abs(out[b, 0, i] - v[b, 0, :n].mean(0)).max() < 1e-14
            assert abs(lse[b, 0, i] - math.log(n)) < 1e-14


def pin_causal_row_is_prefix_attention(orc):
    """rockcohen.cc section 6.3: causal row i is attention over keys 0..i alone."""
    q, k, v = _rand(15, 1, 1, 6, 6, 4, 3)
    out, lse = orc.attention(q, k, v, 0.5, C)
    for i in range(6):
        o_i, l_i = orc.attention(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], 0.5)
        assert np.abs(out[0, 0, i] - o_i[0, 0, 0]).max() < 1e-13 and abs(lse[0, 0, i] - l_i[0, 0, 0]) < 1e-13


def pin_key_padding_is_truncation(orc):
    """Key padding with length L equals the unpadded call on the first L keys."""
    q, k, v = _rand(16, 3, 2, 4, 9, 3, 5)
    kl = np.array([1, 5, 9], np.int32)
    out, lse = orc.attention(q, k, v, 0.3, P, kl)
    for b, L in enumerate(kl):
        o_b, l_b = orc.attention(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.3)
        assert np.abs(out[b] - o_b[0]).max() < 1e-13 and np.abs(lse[b] - l_b[0]).max() < 1e-13
    # one legal key: the output is that key's value row, exactly
    assert np.array_equal(out[0, :, :, :], np.broadcast_to(v[0, :, :1, :], out[0].shape))


def pin_heads_are_independent(orc):
    """vlmlib.cn summary, multi-head attention: each (b, h) is its own attention call."""
    q, k, v = _rand(17, 2, 3, 5, 7, 4, 6)
    out, lse = orc.attention(q, k, v, 0.5)
    for b in range(2):
        for h in range(3):
            o, l = orc.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], 0.5)
            assert np.array_equal(o[0, 0], out[b, h]) and np.array_equal(l[0, 0], lse[b, h])


def pin_loop_form_equals_matrix_form(orc):
    """rockcohen.cc section 10.2 (P0a): loop form equals matrix form to 1e-12. The
    matrix form uses numpy matmul and scipy's softmax / logsumexp (library steps),
    across self and cross shapes, d_k != d_v, every mask mode and B*H > 1."""
    for seed, (B, H, n_q, n_k, d_k, d_v) in enumerate([(2, 3, 5, 7, 4, 6), (1, 2, 9, 4, 8, 3), (3, 1, 6, 6, 2, 5)]):
        q, k, v = _rand(100 + seed, B, H, n_q, n_k, d_k, d_v)
        kl = np.random.Generator(np.random.PCG64(seed)).integers(1, n_k, B, endpoint=True).astype(np.int32)
        for mode in (0, C, P, C | P):
            if mode & C and n_q != n_k:
                continue
            out, lse = orc.attention(q, k, v, 0.37, mode, kl)
            out_m, lse_m, A = oracle.attention_matrix_form(q, k, v, 0.37, mode, kl)
            assert np.abs(out - out_m).max() < 1e-12 and np.abs(lse - lse_m).max() < 1e-12
            w = orc.attention_weights(q, k, 0.37, mode, kl)
            assert np.abs(w - A).max() < 1e-12


def pin_torch_cpu_reference(orc):
    """Library cross-check: torch float64 on the CPU, softmax(scale QK^T + mask) V."""
    import torch

    q, k, v = _rand(18, 2, 2, 6, 6, 5, 3)
    kl = np.array([6, 3], np.int32)
    for mode in (0, C, P, C | P):
        mask = torch.from_numpy(np.where(oracle.legal_mask(2, 6, 6, mode, kl), 0.0, -np.inf))
        s = 0.45 * torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) + mask
        ref = torch.softmax(s, dim=-1) @ torch.from_numpy(v)
        out, lse = orc.attention(q, k, v, 0.45, mode, kl)
        assert np.abs(out - ref.numpy()).max() < 1e-12
        assert np.abs(lse - torch.logsumexp(s, dim=-1).numpy()).max() < 1e-12


def pin_brute_force_tiny(orc):
    """Pure-Python brute force with math.exp, tiny cross-attention shape with padding."""
    q, k, v = _rand(19, 1, 1, 3, 4, 2, 3)
    L = 3
    out, lse = orc.attention(q, k, v, 0.8, P, np.array([L], np.int32))
    for i in range(3):
        e = [math.exp(0.8 * sum(q[0, 0, i, t] * k[0, 0, j, t] for t in range(2))) for j in range(L)]
        tot = sum(e)
        for t in range(3):
            assert abs(out[0, 0, i, t] - sum(e[j] * v[0, 0, j, t] for j in range(L)) / tot) < 1e-13
        assert abs(lse[0, 0, i] - math.log(tot)) < 1e-13


def pin_empty_row_convention(orc):
    """No legal key (key length 0): the chosen convention o = 0, lse = -inf."""
    q, k, v = _rand(20, 2, 1, 3, 4, 2, 2)
    out, lse = orc.attention(q, k, v, 0.5, P, np.array([0, 2], np.int32))
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def pin_row_subset_matches_full(orc):
    """attention_rows returns exactly the rows of the full call."""
    q, k, v = _rand(21, 2, 2, 5, 6, 3, 4)
    kl = np.array([2, 6], np.int32)
    out, lse = orc.attention(q, k, v, 0.5, P, kl)
    ids = np.array([0, 7, 3, 19, 12])
    o_r, l_r = orc.attention_rows(q, k, v, 0.5, ids, P, kl)
    assert np.array_equal(o_r, out.reshape(-1, 4)[ids]) and np.array_equal(l_r, lse.reshape(-1)[ids])


def pin_input_widening(orc):
    """bf16 bit patterns and float32 inputs are widened exactly: same result as float64
    inputs holding the same values."""
    q, k, v = _rand(22, 1, 2, 4, 5, 3, 3)
    f32 = [a.astype(np.float32) for a in (q, k, v)]
    bits = [(a.view(np.uint32) >> 16).astype(np.uint16) for a in f32]  # truncation: any bf16 values will do
    for arrs in (f32, bits):
        o1, l1 = orc.attention(*arrs, 0.5)
        o2, l2 = orc.attention(*[oracle.widen(a) for a in arrs], 0.5)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # bf16 1.0 is 0x3F80, -2.0 is 0xC000
    assert np.array_equal(oracle.widen(np.array([0x3F80, 0xC000], np.uint16)), [1.0, -2.0])


# ---------------------------------------------------------------- decode (one generation step)
def pin_decode_is_causal_suffix(orc):
    """A decode step of n_q new queries against len keys is exactly the last n_q rows
    of causal self-attention over the first len positions (rockcohen.cc section 6.3:
    each position sees the prefix up to itself; generation adds positions one at a
    time)."""
    rng = np.random.Generator(np.random.PCG64(30))
    B, H, n_q, n_max, dk, dv = 3, 2, 4, 11, 3, 5
    q = rng.standard_normal((B, H, n_q, dk))
    k = rng.standard_normal((B, H, n_max, dk))
    v = rng.standard_normal((B, H, n_max, dv))
    lens = np.array([11, 7, 4], np.int32)
    out, lse = orc.attention(q, k, v, 0.45, DEC, lens)
    for b, L in enumerate(lens):
        qf = np.concatenate([rng.standard_normal((1, H, L - n_q, dk)), q[b:b + 1]], axis=2)
        of, lf = orc.attention(qf, k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.45, C)
        assert np.array_equal(out[b], of[0, :, L - n_q:]) and np.array_equal(lse[b], lf[0, :, L - n_q:])


def pin_decode_single_query_sees_whole_cache(orc):
    """One new query attends to every cached key: the same as key padding with len."""
    q, k, v = _rand(31, 2, 2, 1, 9, 4, 3)
    lens = np.array([9, 5], np.int32)
    o1, l1 = orc.attention(q, k, v, 0.5, DEC, lens)
    o2, l2 = orc.attention(q, k, v, 0.5, P, lens)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_decode_short_cache(orc):
    """Queries whose position is negative (cache shorter than n_q) have no legal key."""
    q, k, v = _rand(32, 1, 1, 3, 6, 2, 2)
    out, lse = orc.attention(q, k, v, 0.5, DEC, np.array([2], np.int32))
    assert np.all(out[0, 0, 0] == 0.0) and np.isneginf(lse[0, 0, 0])
    assert np.all(np.isfinite(lse[0, 0, 1:]))
    o1, _ = orc.attention(q[:, :, 1:2], k[:, :, :1], v[:, :, :1], 0.5)
    assert np.array_equal(out[0, 0, 1], o1[0, 0, 0])


def pin_decode_matrix_form(orc):
    """Loop form equals the matrix form for the decode mask, with the lengths the decode
    workloads use (one and several new queries, ragged caches)."""
    for seed, n_q in ((33, 1), (34, 5)):
        q, k, v = _rand(seed, 3, 2, n_q, 12, 4, 4)
        lens = np.array([12, 6, n_q], np.int32)
        out, lse = orc.attention(q, k, v, 0.3, DEC, lens)
        om, lm, A = oracle.attention_matrix_form(q, k, v, 0.3, DEC, lens)
        assert np.abs(out - om).max() < 1e-12 and np.abs(lse - lm).max() < 1e-12
        w = orc.attention_weights(q, k, 0.3, DEC, lens)
        assert np.abs(w - A).max() < 1e-12


# ---------------------------------------------------------------- local window (restricted self-attention)
def pin_window_is_neighbourhood_attention(orc):
    """Restricted self-attention (csdn blog section 4.3; vlmlib.cn "limitations"): row i
    attends to keys i-r..i+r only, i.e. equals unmasked attention over that slice;
    with the causal mask, to keys i-r..i. Brute force row by row, with key padding."""
    q, k, v = _rand(40, 2, 2, 9, 9, 3, 4)
    kl = np.array([9, 6], np.int32)
    for r in (0, 1, 3, 20):
        for mode in (WIN, WIN | C, WIN | P, WIN | C | P):
            out, lse = orc.attention(q, k, v, 0.4, mode, kl, window=r)
            for b in range(2):
                for i in range(9):
                    lo = max(0, i - r)
                    hi = min(i + r + 1, 9)
                    if mode & C:
                        hi = min(hi, i + 1)
                    if mode & P:
                        hi = min(hi, kl[b])
                    if hi <= lo:
                        assert np.all(out[b, :, i] == 0.0) and np.all(np.isneginf(lse[b, :, i]))
                        continue
                    o1, l1 = orc.attention(q[b:b + 1, :, i:i + 1], k[b:b + 1, :, lo:hi], v[b:b + 1, :, lo:hi], 0.4)
                    assert np.array_equal(out[b, :, i], o1[0, :, 0]) and np.array_equal(lse[b, :, i], l1[0, :, 0])


def pin_window_limits(orc):
    """A window covering the whole sequence changes nothing; radius 0 returns V[i]."""
    q, k, v = _rand(41, 1, 2, 7, 7, 4, 3)
    o_all, l_all = orc.attention(q, k, v, 0.5, C)
    o_w, l_w = orc.attention(q, k, v, 0.5, C | WIN, window=7)
    assert np.array_equal(o_all, o_w) and np.array_equal(l_all, l_w)
    o0, _ = orc.attention(q, k, v, 0.5, WIN, window=0)
    assert np.array_equal(o0, v)


def pin_window_matrix_form(orc):
    q, k, v = _rand(42, 2, 2, 11, 11, 4, 4)
    kl = np.array([11, 8], np.int32)
    for mode, r in ((WIN, 2), (WIN | C, 4), (WIN | P, 3)):
        out, lse = orc.attention(q, k, v, 0.3, mode, kl, window=r)
        om, lm, A = oracle.attention_matrix_form(q, k, v, 0.3, mode, kl, window=r)
        assert np.abs(out - om).max() < 1e-12 and np.abs(lse - lm).max() < 1e-12
        assert np.abs(orc.attention_weights(q, k, 0.3, mode, kl, window=r) - A).max() < 1e-12


# ---------------------------------------------------------------- gradients (training)
def _loss(orc, q, k, v, dout, scale, mode, kl, window=0):
    out, _ = orc.attention(q, k, v, scale, mode, kl, window=window)
    return float(np.sum(out * dout))


def pin_bwd_finite_differences(orc):
    """The gradients of L = sum(dout * O) match central finite differences of the
    (pinned) forward oracle, element by element, for every mask and a cross shape."""
    rng = np.random.Generator(np.random.PCG64(50))
    cases = [(4, 5, 0), (4, 5, P), (5, 5, C), (5, 5, C | P), (5, 5, WIN | C)]
    for n_q, n_k, mode in cases:
        q = rng.standard_normal((1, 2, n_q, 3))
        k = rng.standard_normal((1, 2, n_k, 3))
        v = rng.standard_normal((1, 2, n_k, 2))
        dout = rng.standard_normal((1, 2, n_q, 2))
        kl = np.array([3], np.int32)
        win = 1
        dq, dk, dv = orc.attention_bwd(q, k, v, dout, 0.7, mode, kl, window=win)
        h = 1e-6
        for x, g in ((q, dq), (k, dk), (v, dv)):
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = _loss(orc, q, k, v, dout, 0.7, mode, kl, win)
                x[idx] = old - h
                lm = _loss(orc, q, k, v, dout, 0.7, mode, kl, win)
                x[idx] = old
                assert abs((lp - lm) / (2 * h) - g[idx]) < 1e-7, (mode, idx)


def pin_bwd_torch_autograd(orc):
    """Library cross-check: torch float64 autograd of softmax(scale QK^T + mask) V."""
    import torch

    q, k, v = _rand(51, 2, 2, 6, 6, 4, 3)
    dout = np.random.Generator(np.random.PCG64(52)).standard_normal((2, 2, 6, 3))
    kl = np.array([6, 4], np.int32)
    for mode in (0, C, P, C | P):
        mask = torch.from_numpy(np.where(oracle.legal_mask(2, 6, 6, mode, kl), 0.0, -np.inf))
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        out = torch.softmax(0.45 * tq @ tk.transpose(-1, -2) + mask, dim=-1) @ tv
        (out * torch.from_numpy(dout)).sum().backward()
        dq, dk, dv = orc.attention_bwd(q, k, v, dout, 0.45, mode, kl)
        for a, b in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.abs(a - b.numpy()).max() < 1e-12


def pin_bwd_matrix_form(orc):
    q, k, v = _rand(53, 2, 3, 7, 9, 4, 5)
    dout = np.random.Generator(np.random.PCG64(54)).standard_normal((2, 3, 7, 5))
    kl = np.array([9, 5], np.int32)
    for mode in (0, P):
        g1 = orc.attention_bwd(q, k, v, dout, 0.3, mode, kl)
        g2 = oracle.attention_bwd_matrix_form(q, k, v, dout, 0.3, mode, kl)
        for a, b in zip(g1, g2):
            assert np.abs(a - b).max() < 1e-12


def pin_bwd_shift_invariance_and_dead_keys(orc):
    """Rows of dS sum to zero, so dQ, dK and dV do not change when every key moves by a
    common u (rockcohen.cc section 3.2, score differences only); keys that no query may
    see (padding) get exactly zero dK and dV."""
    q, k, v = _rand(55, 2, 1, 5, 6, 3, 2)
    dout = np.random.Generator(np.random.PCG64(56)).standard_normal((2, 1, 5, 2))
    kl = np.array([6, 4], np.int32)
    g = orc.attention_bwd(q, k, v, dout, 0.6, P, kl)
    g2 = orc.attention_bwd(q, k + np.array([0.5, -1.0, 2.0]), v, dout, 0.6, P, kl)
    for a, b in zip(g, g2):
        assert np.abs(a - b).max() < 1e-12
    assert np.all(g[1][1, :, 4:] == 0.0) and np.all(g[2][1, :, 4:] == 0.0)


# ---------------------------------------------------------------- multi-head attention
def _mha_params(seed, B, n_q, n_k, d_model, H, d, bias=True):
    rng = np.random.Generator(np.random.PCG64(seed))
    x_q = rng.standard_normal((B, n_q, d_model))
    x_kv = rng.standard_normal((B, n_k, d_model))
    w = [rng.standard_normal((d_model, H * d)) / math.sqrt(d_model) for _ in range(3)]
    w_o = rng.standard_normal((H * d, d_model)) / math.sqrt(H * d)
    b = [rng.standard_normal(H * d) for _ in range(3)] + [rng.standard_normal(d_model)] if bias else [None] * 4
    return x_q, x_kv, w, w_o, b


def _mha(orc, x_q, x_kv, w, w_o, b, H, scale, mode=0, kl=None):
    return orc.mha(x_q, x_kv, w[0], w[1], w[2], w_o, H, scale, mode, kl, b_q=b[0], b_k=b[1], b_v=b[2], b_o=b[3])


def pin_mha_single_head_identity(orc):
    """One head with identity projections and no biases is scaled dot-product
    attention itself (vlmlib.cn "multi-head attention" with h = 1, W = I)."""
    rng = np.random.Generator(np.random.PCG64(60))
    x = rng.standard_normal((2, 6, 5))
    eye = np.eye(5)
    kl = np.array([6, 3], np.int32)
    for mode in (0, C, P, C | P):
        y = orc.mha(x, x, eye, eye, eye, eye, 1, 0.4, mode, kl)
        o, _ = orc.attention(x[:, None], x[:, None], x[:, None], 0.4, mode, kl)
        assert np.abs(y - o[:, 0]).max() < 1e-13, mode


def pin_mha_sum_over_heads(orc):
    """Concat(head_1..head_h) W^O equals the sum over heads of head_i W^O_i (the
    block rows of W^O), each head_i = Attention(x_q W_i^Q + b, x_kv W_i^K + b,
    x_kv W_i^V + b) with W_i the i-th block of columns -- restated per head with
    explicit slices and the matrix form of the attention, cross shape and masks."""
    H, d = 3, 4
    x_q, x_kv, w, w_o, b = _mha_params(61, 2, 5, 7, 10, H, d)
    kl = np.array([7, 4], np.int32)
    for mode in (0, P):
        y = _mha(orc, x_q, x_kv, w, w_o, b, H, 0.5, mode, kl)
        ref = np.broadcast_to(b[3], y.shape).copy()
        for h in range(H):
            cols = slice(h * d, (h + 1) * d)
            qh, kh, vh = (src @ wi[:, cols] + bi[cols] for src, wi, bi in
                          ((x_q, w[0], b[0]), (x_kv, w[1], b[1]), (x_kv, w[2], b[2])))
            head = oracle.attention_matrix_form(qh[:, None], kh[:, None], vh[:, None], 0.5, mode, kl)[0]
            ref += head[:, 0] @ w_o[cols, :]
        assert np.abs(y - ref).max() < 1e-12, mode


def pin_mha_torch_module(orc):
    """Library cross-check: torch.nn.MultiheadAttention in float64 with the same
    weights (its projections are x W^T + b, so it takes our W transposed), key
    padding and the causal mask."""
    import torch

    H, d, d_model = 2, 4, 8
    x_q, x_kv, w, w_o, b = _mha_params(62, 2, 6, 6, d_model, H, d)
    kl = np.array([6, 4], np.int32)
    m = torch.nn.MultiheadAttention(d_model, H, bias=True, batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        m.in_proj_weight.copy_(torch.from_numpy(np.concatenate([w[0].T, w[1].T, w[2].T])))
        m.in_proj_bias.copy_(torch.from_numpy(np.concatenate(b[:3])))
        m.out_proj.weight.copy_(torch.from_numpy(w_o.T))
        m.out_proj.bias.copy_(torch.from_numpy(b[3]))
    pad = torch.from_numpy(np.arange(6)[None, :] >= kl[:, None])
    causal = torch.from_numpy(np.triu(np.ones((6, 6), bool), 1))
    for mode, kpm, am in ((0, None, None), (P, pad, None), (C, None, causal), (C | P, pad, causal)):
        with torch.no_grad():
            t, _ = m(torch.from_numpy(x_q), torch.from_numpy(x_kv), torch.from_numpy(x_kv), key_padding_mask=kpm,
                     attn_mask=am, need_weights=False)
        y = _mha(orc, x_q, x_kv, w, w_o, b, H, 1 / math.sqrt(d), mode, kl)
        assert np.abs(y - t.numpy()).max() < 1e-12, mode


def pin_mha_causal_row0_and_head_permutation(orc):
    """With the causal mask, position 0 sees only itself, so every head returns its
    value row: Y_0 = (x_0 W^V + b_V) W^O + b_O (closed form). Renumbering the heads
    (the same permutation of the column blocks of W^Q, W^K, W^V, their biases and
    the row blocks of W^O) leaves Y unchanged (heads are independent and summed)."""
    H, d = 4, 3
    x_q, _, w, w_o, b = _mha_params(63, 2, 5, 5, 9, H, d)
    y = _mha(orc, x_q, x_q, w, w_o, b, H, 0.6, C)
    y0 = (x_q[:, 0] @ w[2] + b[2]) @ w_o + b[3]
    assert np.abs(y[:, 0] - y0).max() < 1e-12
    perm = [2, 0, 3, 1]
    idx = np.concatenate([np.arange(h * d, (h + 1) * d) for h in perm])
    y2 = _mha(orc, x_q, x_q, [wi[:, idx] for wi in w], w_o[idx], [bi[idx] for bi in b[:3]] + [b[3]], H, 0.6, C)
    assert np.abs(y - y2).max() < 1e-12


def pin_mha_bf16_inputs_widen_exactly(orc):
    """bf16 bit patterns are widened exactly: the same values given as float64 give
    bit-identical results."""
    H, d = 2, 4
    x_q, x_kv, w, w_o, b = _mha_params(64, 1, 4, 6, 8, H, d)
    bits = lambda a: ((np.asarray(a, np.float32).view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    wide = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    args16 = [bits(a) for a in (x_q, x_kv, *w, w_o)]
    b16 = [bits(x) for x in b]
    y16 = orc.mha(*args16[:5], args16[5], H, 0.5, P, np.array([5], np.int32),
                  b_q=b16[0], b_k=b16[1], b_v=b16[2], b_o=b16[3])
    y64 = orc.mha(*[wide(a) for a in args16], H, 0.5, P, np.array([5], np.int32),
                  b_q=wide(b16[0]), b_k=wide(b16[1]), b_v=wide(b16[2]), b_o=wide(b16[3]))
    assert np.array_equal(y16, y64)


# ---------------------------------------------------------------- linear projection
def pin_linear_brute_force(orc):
    """y = b + x W entry by entry: an exactly rounded sum (math.fsum) of the products
    x[m, k] W[k, n] and the bias, on small non-square shapes (so a transposed or
    mis-strided operand cannot pass), with and without the bias."""
    rng = np.random.Generator(np.random.PCG64(70))
    M, N, K = 5, 3, 7
    x, w, b = rng.standard_normal((M, K)), rng.standard_normal((K, N)), rng.standard_normal(N)
    for bias in (b, None):
        y = orc.linear(x, w, bias)
        for m in range(M):
            for n in range(N):
                terms = [x[m, k] * w[k, n] for k in range(K)] + ([bias[n]] if bias is not None else [])
                assert abs(y[m, n] - math.fsum(terms)) < 1e-13


def pin_linear_closed_forms(orc):
    """Closed forms: x I = x exactly; a permutation matrix moves columns (x P)[:, j] =
    x[:, p(j)]; a zero input returns the bias in every row; a projection of one row
    with a one-hot weight column picks one input feature."""
    rng = np.random.Generator(np.random.PCG64(71))
    x = rng.standard_normal((4, 6))
    assert np.array_equal(orc.linear(x, np.eye(6)), x)
    perm = np.array([3, 0, 5, 1, 4, 2])
    P = np.zeros((6, 6))
    P[perm, np.arange(6)] = 1.0
    assert np.array_equal(orc.linear(x, P), x[:, perm])
    b = rng.standard_normal(6)
    assert np.array_equal(orc.linear(np.zeros((3, 6)), P, b), np.broadcast_to(b, (3, 6)))
    e = np.zeros((6, 2))
    e[4, 1] = 1.0
    assert np.array_equal(orc.linear(x, e)[:, 1], x[:, 4]) and np.all(orc.linear(x, e)[:, 0] == 0.0)


def pin_linear_matches_mha_projection(orc):
    """The multi-head oracle's projections are this product: with one head of width
    d_model, identity W^K = W^V = W^O, no output bias and causal masking, output
    row 0 is x_0 W^V + b_V (it attends to itself alone) = linear(x, W^V, b_V) row 0."""
    rng = np.random.Generator(np.random.PCG64(72))
    d_model = 6
    x = rng.standard_normal((1, 4, d_model))
    wv, bv = rng.standard_normal((d_model, d_model)), rng.standard_normal(d_model)
    eye = np.eye(d_model)
    y = orc.mha(x, x, eye, eye, wv, eye, 1, 0.3, C, None, b_v=bv)
    assert np.abs(y[0, 0] - orc.linear(x[0], wv, bv)[0]).max() < 1e-13


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
