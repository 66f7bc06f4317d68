"""Pins for the CPU oracle: facts the pages or mathematics fix, checked without
re-using the oracle's own formulas.  CPU only.

Each test names what it pins and where that fact comes from.  Together they
are meant to fail on any plausible slip in the oracle: a decayed current
token, a transposed read-out, a wrong chunk index, a missing causal mask, a
wrong GQA head map, a wrong scale or a wrong rounding.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------- gRet pins

def test_worked_example_2x2():
    """Blog post Section 4: S_prev = 2I, gamma = 0.5, k = [1,0], v = [3,4]
    gives S = [[4,4],[0,1]] and q = [1,0] reads o = [4,4].  Pins the update
    order (decay the old state, add the new outer product undecayed) and the
    read-out o = q S (S q^T would give [4,0])."""
    g = _load("worked_example_2x2.json")
    # gamma = sigmoid(0)^(1/1) = 0.5
    assert abs(oracle.gate(0.0, 1.0) - g["gamma"]) < 1e-16
    q = np.array(g["q"]).reshape(1, 1, 1, 2)
    k = np.array(g["k"]).reshape(1, 1, 1, 2)
    v = np.array(g["v"]).reshape(1, 1, 1, 2)
    S0 = np.array(g["S_prev"]).reshape(1, 1, 2, 2)
    o, S = oracle.gret_recurrent(q, k, v, np.zeros((1, 1, 1)), 1.0, S0=S0)
    np.testing.assert_allclose(S[0, 0], np.array(g["S_expected"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[0, 0, 0], np.array(g["o_expected"]), rtol=0, atol=1e-15)
    # the same step through the chunkwise form (one chunk of one token)
    o2, S2 = oracle.gret_chunkwise(q, k, v, np.zeros((1, 1, 1)), 1.0, 1, S0=S0)
    np.testing.assert_allclose(S2[0, 0], np.array(g["S_expected"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o2[0, 0, 0], np.array(g["o_expected"]), rtol=0, atol=1e-15)


def test_second_state_from_zero():
    """Close-reading notes Section 2.2: from S_0 = 0, S_2 = gamma_2 K_1^T V_1 +
    K_2^T V_2 -- the first token is decayed by the second gate only, the
    current token not at all (D_nn = 1)."""
    k = np.array([[1.0, 2.0, 0.0], [0.0, -1.0, 3.0]]).reshape(1, 2, 1, 3)
    v = np.array([[2.0, 1.0], [-1.0, 4.0]]).reshape(1, 2, 1, 2)
    q = np.zeros((1, 2, 1, 3))
    logits = np.array([1.3, -0.4]).reshape(1, 2, 1)
    tau = 2.0
    g2 = 1.0 / (1.0 + math.exp(0.4))  # sigmoid(-0.4)
    g2 = g2 ** (1.0 / tau)
    expect = np.zeros((3, 2))
    for i in range(3):
        for j in range(2):
            expect[i, j] = g2 * k[0, 0, 0, i] * v[0, 0, 0, j] + k[0, 1, 0, i] * v[0, 1, 0, j]
    _, S = oracle.gret_recurrent(q, k, v, logits, tau)
    np.testing.assert_allclose(S[0, 0], expect, rtol=1e-14, atol=1e-14)


def _int_qkv(rng, B, N, H, dk, dv, lo=-3, hi=4):
    q = rng.integers(lo, hi, size=(B, N, H, dk)).astype(np.float64)
    k = rng.integers(lo, hi, size=(B, N, H, dk)).astype(np.float64)
    v = rng.integers(lo, hi, size=(B, N, H, dv)).astype(np.float64)
    return q, k, v


def test_gamma_one_is_causal_linear_attention():
    """gamma == 1 (logit = +inf, logsigmoid = 0 exactly) removes the decay:
    o_n = q_n sum_{m<=n} k_m^T v_m, causal linear attention.  Integer inputs,
    so every form must be exact."""
    rng = np.random.default_rng(1)
    B, N, H, dk, dv = 2, 37, 3, 5, 4
    q, k, v = _int_qkv(rng, B, N, H, dk, dv)
    logits = np.full((B, N, H), np.inf)
    expect = np.zeros((B, N, H, dv))
    for b in range(B):
        for h in range(H):
            for n in range(N):
                scores = k[b, : n + 1, h, :] @ q[b, n, h, :]       # (q_n . k_m), m <= n
                expect[b, n, h] = scores @ v[b, : n + 1, h, :]
    o_r, _ = oracle.gret_recurrent(q, k, v, logits, 16.0)
    o_p = oracle.gret_parallel(q, k, v, logits, 16.0)
    o_c, _ = oracle.gret_chunkwise(q, k, v, logits, 16.0, 8)
    for o in (o_r, o_p, o_c):
        assert np.array_equal(o, expect)


def test_gamma_zero_keeps_only_current_token():
    """gamma == 0 (logit = -inf) forgets everything before the current token:
    o_n = (q_n . k_n) v_n."""
    rng = np.random.default_rng(2)
    B, N, H, dk, dv = 1, 19, 2, 4, 3
    q, k, v = _int_qkv(rng, B, N, H, dk, dv)
    logits = np.full((B, N, H), -np.inf)
    expect = np.einsum("bnhd,bnhd->bnh", q, k)[..., None] * v
    o_r, _ = oracle.gret_recurrent(q, k, v, logits, 16.0)
    o_p = oracle.gret_parallel(q, k, v, logits, 16.0)
    o_c, _ = oracle.gret_chunkwise(q, k, v, logits, 16.0, 4)
    for o in (o_r, o_p, o_c):
        assert np.array_equal(o, expect)


def test_constant_gate_is_fixed_decay_retention():
    """A constant gate gamma makes D_nm = gamma^(n-m): the fixed-decay
    retention matrix (paper Section 3.1 builds gRet on retention).  Built
    here with matrix powers, not gate products."""
    rng = np.random.default_rng(3)
    B, N, H, dk, dv = 1, 23, 1, 6, 5
    q = rng.standard_normal((B, N, H, dk))
    k = rng.standard_normal((B, N, H, dk))
    v = rng.standard_normal((B, N, H, dv))
    x, tau = 0.7, 3.0
    gam = (1.0 / (1.0 + math.exp(-x))) ** (1.0 / tau)
    logits = np.full((B, N, H), x)
    n = np.arange(N)
    D = np.where(n[:, None] >= n[None, :], gam ** (n[:, None] - n[None, :]).clip(min=0), 0.0)
    A = q[0, :, 0, :] @ k[0, :, 0, :].T
    expect = (A * D) @ v[0, :, 0, :]
    o_r, _ = oracle.gret_recurrent(q, k, v, logits, tau)
    np.testing.assert_allclose(o_r[0, :, 0, :], expect, rtol=1e-12, atol=1e-12)


def test_unrolled_sum_brute_force():
    """Blog post Section 4 unrolled sum: o_t = sum_i (prod_{j=i+1..t} gamma_j)
    (q_t k_i^T) v_i, evaluated with pure-Python loops on a tiny case."""
    rng = np.random.default_rng(4)
    N, dk, dv = 5, 2, 3
    q = rng.standard_normal((N, dk))
    k = rng.standard_normal((N, dk))
    v = rng.standard_normal((N, dv))
    x = rng.standard_normal(N) * 2
    tau = 1.5
    gam = [(1.0 / (1.0 + math.exp(-xi))) ** (1.0 / tau) for xi in x]
    expect = np.zeros((N, dv))
    for t in range(N):
        for i in range(t + 1):
            w = 1.0
            for j in range(i + 1, t + 1):
                w *= gam[j]
            qk = sum(q[t, a] * k[i, a] for a in range(dk))
            for c in range(dv):
                expect[t, c] += w * qk * v[i, c]
    sh = lambda a: a.reshape(1, N, 1, -1)
    lg = x.reshape(1, N, 1)
    for o in (oracle.gret_recurrent(sh(q), sh(k), sh(v), lg, tau)[0],
              oracle.gret_parallel(sh(q), sh(k), sh(v), lg, tau),
              oracle.gret_chunkwise(sh(q), sh(k), sh(v), lg, tau, 2)[0]):
        np.testing.assert_allclose(o[0, :, 0, :], expect, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("C", [1, 2, 3, 16, 64, 256, 200])
def test_three_forms_agree(C):
    """Paper Section 3.1: the parallel, recurrent and chunkwise forms are
    equivalent.  N = 200 is not a multiple of most C (ragged last chunk)."""
    B, N, H, dk, dv = 1, 200, 2, 8, 6
    seed = 11
    q = synth.normal(seed, 1, (B, N, H, dk), "f32") * 0.5
    k = synth.normal(seed, 2, (B, N, H, dk), "f32") * 0.5
    v = synth.normal(seed, 3, (B, N, H, dv), "f32")
    logits = synth.normal(seed, 4, (B, N, H), "f32", mean=1.0, std=2.0)
    tau = 4.0
    o_r, S_r = oracle.gret_recurrent(q, k, v, logits, tau)
    o_c, S_c = oracle.gret_chunkwise(q, k, v, logits, tau, C)
    scale = np.abs(o_r).max()
    np.testing.assert_allclose(o_c, o_r, rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(S_c, S_r, rtol=0, atol=1e-12 * np.abs(S_r).max())
    if C == 16:
        o_p = oracle.gret_parallel(q, k, v, logits, tau)
        np.testing.assert_allclose(o_p, o_r, rtol=0, atol=1e-12 * scale)


def test_state_continuation_equals_one_call():
    """Chunked prefill (blog post Section 6: the prompt is fed in pieces that
    carry the self-decoder state): two calls with the state carried equal one
    call, for both the recurrent and the chunkwise form."""
    B, N, H, d = 2, 150, 2, 4
    q = synth.normal(5, 1, (B, N, H, d), "f32")
    k = synth.normal(5, 2, (B, N, H, d), "f32")
    v = synth.normal(5, 3, (B, N, H, d), "f32")
    lg = synth.normal(5, 4, (B, N, H), "f32")
    o_full, S_full = oracle.gret_recurrent(q, k, v, lg, 16.0)
    n1 = 61
    o1, S1 = oracle.gret_chunkwise(q[:, :n1], k[:, :n1], v[:, :n1], lg[:, :n1], 16.0, 16)
    o2, S2 = oracle.gret_chunkwise(q[:, n1:], k[:, n1:], v[:, n1:], lg[:, n1:], 16.0, 16, S0=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S2, S_full, rtol=0, atol=1e-12)


def test_gate_limits_and_value():
    """gamma = sigmoid(x)^(1/tau): +inf -> 1, -inf -> 0, and a generic value;
    large |x| must not overflow."""
    assert oracle.gate(np.inf, 16.0) == 1.0
    assert oracle.gate(-np.inf, 16.0) == 0.0
    assert abs(oracle.gate(2.0, 16.0) - (1 / (1 + math.exp(-2.0))) ** (1 / 16)) < 1e-15
    assert oracle.gate(800.0, 16.0) == 1.0
    assert 0.0 <= oracle.gate(-800.0, 16.0) < 1e-20


# ---------------------------------------------------------- rounding pins

def test_round_bf16_is_nearest_even():
    """fp64 -> bf16: the result is the nearer of the two bf16 neighbours,
    ties go to the even pattern; checked by brute force on the neighbours
    and against an independent implementation (the input generator's)."""
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                        [1.0, -2.5, 0.0, 3.0e38, 1e-40]])
    bits = oracle.round_bf16(x)
    val = synth.bf16_bits_to_f32(bits).astype(np.float64)
    for xi, vi, bi in zip(x, val, bits):
        bi = int(bi)
        mag = bi & 0x7FFF
        # neighbours of the chosen value on both sides (same sign, magnitude +-1 ulp)
        for s in (-1, 1):
            if 0 <= mag + s < 0x7F80:
                n = float(synth.bf16_bits_to_f32(np.array([(bi & 0x8000) | (mag + s)], dtype=np.uint16))[0])
                assert abs(xi - vi) <= abs(xi - n)
                if abs(xi - vi) == abs(xi - n) and xi != vi:
                    assert mag % 2 == 0
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert oracle.round_bf16(np.array([1.0 + 2 ** -8]))[0] == 0x3F80
    assert oracle.round_bf16(np.array([1.0 + 3 * 2 ** -8]))[0] == 0x3F82
    assert np.array_equal(bits, synth.f64_to_bf16_bits(x))
    assert oracle.round_bf16(np.array([1e39]))[0] == 0x7F80


# ---------------------------------------------------------- shared KV pins

def test_rmsnorm_closed_forms():
    """Eq. 2 with LN = RMSNorm.  A row of +-1 has rms 1, so with eps = 0 the
    projection is M W exactly (dyadic W keeps every sum exact); scaling a row
    by a > 0 leaves the eps = 0 output unchanged; the gain multiplies input
    features."""
    dm, n = 64, 12
    M = synth.signs(9, 1, (5, dm)).astype(np.float64)
    W = synth.dyadic(9, 2, (dm, n)).astype(np.float64)
    expect = np.zeros((5, n))
    for r in range(5):
        for c in range(n):
            expect[r, c] = sum(M[r, i] * W[i, c] for i in range(dm))
    out = oracle.rmsnorm_proj(M, W, 0.0)
    assert np.array_equal(out, expect)
    out2 = oracle.rmsnorm_proj(M * 3.75, W, 0.0)
    assert np.array_equal(out2, expect)
    g = np.zeros(dm)
    g[5] = 2.0
    out3 = oracle.rmsnorm_proj(M, W, 0.0, g=g)
    assert np.array_equal(out3, 2.0 * M[:, 5:6] * W[5:6, :])
    # constant row c: rms = |c| -> r = 1/sqrt(c^2 + eps)
    c, eps = 0.5, 0.75
    out4 = oracle.rmsnorm_proj(np.full((1, dm), c), W, eps)
    np.testing.assert_allclose(out4[0], c / math.sqrt(c * c + eps) * W.sum(axis=0), rtol=1e-14, atol=1e-15)


def test_kv_append_touches_only_new_slots():
    """Section 2.2: the cache gets row t of each new token at slot len + t of
    every kv head (head h takes columns h*d..h*d+d-1); nothing else changes."""
    B, Hkv, cap, d, T, length = 2, 3, 10, 4, 3, 5
    rng = np.random.default_rng(3)
    cache = rng.integers(0, 0xFFFF, size=(B, Hkv, cap, d)).astype(np.uint16)
    # values exactly representable in bf16 that encode (b, t, h, c)
    kv = np.zeros((B, T, Hkv * d))
    for b in range(B):
        for t in range(T):
            for h in range(Hkv):
                for c in range(d):
                    kv[b, t, h * d + c] = 64 * b + 16 * t + 4 * h + c
    new = oracle.kv_append_bf16(cache, kv, length)
    for b in range(B):
        for h in range(Hkv):
            for s in range(cap):
                for c in range(d):
                    if length <= s < length + T:
                        val = synth.bf16_bits_to_f32(np.array([new[b, h, s, c]]))[0]
                        assert val == 64 * b + 16 * (s - length) + 4 * h + c
                    else:
                        assert new[b, h, s, c] == cache[b, h, s, c]


def test_shared_cache_bytes_teaching_numbers():
    """Blog post Sections 2 and 7: 2*B*N*L*H_kv*d_h*b bytes; 26 per-layer
    caches are 13 GiB at 128 Ki tokens, the one shared cache 0.5 GiB -- the
    shared cache does not grow with the number of cross layers."""
    g = _load("shared_cache_bytes.json")
    per_layer = 2 * g["B"] * g["N"] * g["layers"] * g["Hkv"] * g["d"] * g["bytes_per_elem"]
    assert per_layer == g["per_layer_cache_GiB"] * 2 ** 30
    # the append oracle writes one K and one V slot per token regardless of layers
    B, Hkv, d = 1, 2, 4
    cache = np.zeros((B, Hkv, 8, d), dtype=np.uint16)
    touched = (oracle.kv_append_bf16(cache, np.ones((B, 3, Hkv * d)), 0) != 0).sum()
    assert touched == B * 3 * Hkv * d
    shared = 2 * g["B"] * g["N"] * g["Hkv"] * g["d"] * g["bytes_per_elem"]
    assert shared == g["shared_cache_GiB"] * 2 ** 30


# ------------------------------------------------------ attention pins

def test_attention_single_key_and_equal_keys():
    """Softmax over one key returns its value; over equal scores it is the
    mean of the values (Eq. 3)."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, d, cap = 1, 4, 2, 8, 6
    K = rng.standard_normal((B, Hkv, cap, d))
    V = rng.standard_normal((B, Hkv, cap, d))
    Q = rng.standard_normal((B, 1, Hq, d))
    O = oracle.cross_attn(Q, K, V, 0, 0.3)
    for h in range(Hq):
        assert np.array_equal(O[0, 0, h], V[0, h // 2, 0])
    Keq = np.repeat(K[:, :, :1], cap, axis=2)
    O2 = oracle.cross_attn(Q, Keq, V, cap - 1, 0.3)
    for h in range(Hq):
        np.testing.assert_allclose(O2[0, 0, h], V[0, h // 2].mean(axis=0), rtol=1e-14, atol=1e-14)


def test_attention_two_keys_closed_form_and_gqa_map():
    """Two keys: o = v0 + sigmoid(s1 - s0) (v1 - v0) with s = scale q.k.
    Distinct kv heads pin the grouped map kv = h // (Hq / Hkv)."""
    B, Hq, Hkv, d = 1, 6, 3, 4
    rng = np.random.default_rng(6)
    K = rng.standard_normal((B, Hkv, 2, d))
    V = rng.standard_normal((B, Hkv, 2, d))
    Q = rng.standard_normal((B, 1, Hq, d))
    scale = 0.37
    O = oracle.cross_attn(Q, K, V, 1, scale)
    for h in range(Hq):
        g = h // 2
        s0 = scale * float(Q[0, 0, h] @ K[0, g, 0])
        s1 = scale * float(Q[0, 0, h] @ K[0, g, 1])
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(O[0, 0, h], V[0, g, 0] + w1 * (V[0, g, 1] - V[0, g, 0]), rtol=1e-13, atol=1e-14)


def test_attention_causal_mask_and_prefill_rows():
    """Causal mask (Eq. 3; notes Section 2.1: position n reads m <= n): a key
    after the query's position cannot change its output, and prefill row t
    equals a single query at p0 + t."""
    rng = np.random.default_rng(8)
    B, Hq, Hkv, d, cap = 2, 4, 1, 8, 12
    K = rng.standard_normal((B, Hkv, cap, d))
    V = rng.standard_normal((B, Hkv, cap, d))
    Q = rng.standard_normal((B, 5, Hq, d))
    p0 = 4
    O = oracle.cross_attn(Q, K, V, p0, 0.25)
    K2 = K.copy()
    V2 = V.copy()
    K2[:, :, p0 + 5:] = 1e3
    V2[:, :, p0 + 5:] = -7.0
    assert np.array_equal(O, oracle.cross_attn(Q, K2, V2, p0, 0.25))
    for t in range(5):
        Ot = oracle.cross_attn(Q[:, t:t + 1], K, V, p0 + t, 0.25)
        np.testing.assert_allclose(Ot[:, 0], O[:, t], rtol=1e-14, atol=1e-15)


def test_attention_brute_force_pure_python():
    """Naive softmax attention in pure Python (math.exp) on a tiny input."""
    rng = np.random.default_rng(9)
    B, Hq, Hkv, d, cap, T, p0 = 1, 2, 1, 3, 5, 2, 2
    K = rng.standard_normal((B, Hkv, cap, d))
    V = rng.standard_normal((B, Hkv, cap, d))
    Q = rng.standard_normal((B, T, Hq, d))
    scale = 0.5
    O = oracle.cross_attn(Q, K, V, p0, scale)
    for t in range(T):
        for h in range(Hq):
            pos = p0 + t
            e = [math.exp(scale * sum(Q[0, t, h, c] * K[0, 0, m, c] for c in range(d))) for m in range(pos + 1)]
            z = sum(e)
            for c in range(d):
                ref = sum(e[m] / z * V[0, 0, m, c] for m in range(pos + 1))
                assert abs(O[0, t, h, c] - ref) < 1e-13


# ---------------------------------------------- sliding-window attention pins

def test_swa_window_one_returns_own_value():
    """Window C = 1 (Section 3.2, Eq. 8: keys n - C < m <= n): each query sees
    only its own key, so the softmax weight is 1 and o_n = v_n exactly."""
    rng = np.random.default_rng(21)
    B, N, Hq, Hkv, d = 2, 7, 4, 2, 5
    Q = rng.standard_normal((B, N, Hq, d))
    K = rng.standard_normal((B, N, Hkv, d))
    V = rng.standard_normal((B, N, Hkv, d))
    O = oracle.swa_attn(Q, K, V, 1, 0.4)
    for h in range(Hq):
        assert np.array_equal(O[:, :, h], V[:, :, h // 2])


def test_swa_brute_force_pure_python():
    """The window mask written out in pure Python on a tiny input: query n
    weighs keys max(0, n - C + 1) .. n by exp(scale q.k)."""
    rng = np.random.default_rng(22)
    B, N, Hq, Hkv, d, C = 1, 6, 2, 1, 3, 3
    Q = rng.standard_normal((B, N, Hq, d))
    K = rng.standard_normal((B, N, Hkv, d))
    V = rng.standard_normal((B, N, Hkv, d))
    scale = 0.7
    O = oracle.swa_attn(Q, K, V, C, scale)
    for n in range(N):
        keys = [m for m in range(N) if n - C < m <= n]
        for h in range(Hq):
            e = {m: math.exp(scale * sum(Q[0, n, h, c] * K[0, m, 0, c] for c in range(d))) for m in keys}
            z = sum(e.values())
            for c in range(d):
                ref = sum(e[m] / z * V[0, m, 0, c] for m in keys)
                assert abs(O[0, n, h, c] - ref) < 1e-13


def test_swa_wide_window_is_causal_attention():
    """A window at least as long as the sequence masks nothing but the future:
    the result equals the causal attention oracle over the same keys laid out
    as a cache (an independent implementation of Eq. 3)."""
    rng = np.random.default_rng(23)
    B, N, Hq, Hkv, d = 2, 9, 6, 3, 4
    Q = rng.standard_normal((B, N, Hq, d))
    K = rng.standard_normal((B, N, Hkv, d))
    V = rng.standard_normal((B, N, Hkv, d))
    O = oracle.swa_attn(Q, K, V, N + 5, 0.3)
    O_ref = oracle.cross_attn(Q, K.transpose(0, 2, 1, 3), V.transpose(0, 2, 1, 3), 0, 0.3)
    np.testing.assert_allclose(O, O_ref, rtol=1e-13, atol=1e-14)


def test_swa_keys_outside_the_window_change_nothing():
    """Keys older than C positions cannot reach a query: changing them leaves
    its output bit-identical, while changing an in-window key does not."""
    rng = np.random.default_rng(24)
    B, N, Hq, Hkv, d, C = 1, 10, 2, 2, 4, 4
    Q = rng.standard_normal((B, N, Hq, d))
    K = rng.standard_normal((B, N, Hkv, d))
    V = rng.standard_normal((B, N, Hkv, d))
    O = oracle.swa_attn(Q, K, V, C, 0.5)
    K2, V2 = K.copy(), V.copy()
    K2[:, :5] = 50.0
    V2[:, :5] = -3.0
    O2 = oracle.swa_attn(Q, K2, V2, C, 0.5)
    assert np.array_equal(O[:, 8:], O2[:, 8:])   # rows 8, 9 see keys 5..9 only
    assert not np.allclose(O[:, 7], O2[:, 7])    # row 7 sees key 4


# ------------------------------------------ gated retention output (Eq. 7) pins

def test_group_norm_gate_normalises_each_head():
    """Eq. 7, GroupNorm with one group per head: with a gate of swish(g) = g
    sigmoid(g), dividing z by the gate recovers y with mean 0 and variance
    var / (var + eps) over each head's channels, and w, b act per channel."""
    rng = np.random.default_rng(31)
    B, N, H, d, eps = 2, 3, 4, 16, 1e-5
    o = rng.standard_normal((B, N, H, d)) * 3.0 + 1.5
    g = rng.uniform(0.5, 2.0, (B, N, H, d))
    z = oracle.group_norm_gate(o, g, eps)
    y = z / (g / (1.0 + np.exp(-g)))
    var = o.var(axis=-1)
    np.testing.assert_allclose(y.mean(axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=-1), var / (var + eps), rtol=1e-12)
    w = rng.standard_normal(H * d)
    bb = rng.standard_normal(H * d)
    z2 = oracle.group_norm_gate(o, g, eps, w, bb)
    np.testing.assert_allclose(z2, (y * w.reshape(H, d) + bb.reshape(H, d)) * (g / (1.0 + np.exp(-g))),
                               rtol=1e-12, atol=1e-12)


def test_group_norm_gate_special_values():
    """swish(0) = 0 closes the gate; a constant head vector normalises to 0, so
    the output is the gate times the bias."""
    rng = np.random.default_rng(32)
    B, N, H, d = 1, 2, 2, 8
    o = rng.standard_normal((B, N, H, d))
    assert np.array_equal(oracle.group_norm_gate(o, np.zeros_like(o), 1e-6), np.zeros_like(o))
    oc = np.full((B, N, H, d), 4.25)
    g = rng.standard_normal((B, N, H, d))
    bb = rng.standard_normal(H * d)
    z = oracle.group_norm_gate(oc, g, 1e-6, None, bb)
    np.testing.assert_allclose(z, g / (1.0 + np.exp(-g)) * bb.reshape(H, d), rtol=1e-14, atol=1e-15)


def test_group_norm_gate_brute_force():
    """Pure Python on one head vector."""
    rng = np.random.default_rng(33)
    d, eps = 5, 1e-3
    o = rng.standard_normal((1, 1, 1, d))
    g = rng.standard_normal((1, 1, 1, d))
    z = oracle.group_norm_gate(o, g, eps)
    xs = [float(x) for x in o.ravel()]
    mu = sum(xs) / d
    var = sum((x - mu) ** 2 for x in xs) / d
    for c in range(d):
        gc = float(g.ravel()[c])
        ref = (xs[c] - mu) / math.sqrt(var + eps) * gc / (1.0 + math.exp(-gc))
        assert abs(z.ravel()[c] - ref) < 1e-13


# ------------------------------------------------------- rotary encoding pins

def test_rope_position_zero_is_identity_and_pairs_keep_length():
    """Angle 0 at position 0; a rotation keeps the length of every pair."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal((3, 5, 16))
    assert np.array_equal(oracle.rope(x, 0, 10000.0), x)
    pos = rng.integers(0, 10 ** 6, size=(3, 5))
    y = oracle.rope(x, pos, 10000.0)
    np.testing.assert_allclose(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]),
                               rtol=1e-13)


def test_rope_first_pair_turns_by_the_position():
    """Pair 0 has frequency base^0 = 1: (1, 0) at position p becomes (cos p, sin p);
    the last pair of d = 4 turns by p / base^(1/2)."""
    for p in (0, 1, 7, 1000, 123456789):
        y = oracle.rope(np.array([[1.0, 0.0, 0.0, 1.0]]), p, 100.0)
        np.testing.assert_allclose(y[0, :2], [math.cos(p), math.sin(p)], rtol=0, atol=1e-9)
        a = p / 10.0
        np.testing.assert_allclose(y[0, 2:], [-math.sin(a), math.cos(a)], rtol=0, atol=1e-9)


def test_rope_dot_product_depends_on_the_offset_only():
    """q rotated at n and k at m: their dot product is unchanged when both
    positions move by the same amount, and rotations compose additively."""
    rng = np.random.default_rng(42)
    q = rng.standard_normal((1, 32))
    k = rng.standard_normal((1, 32))
    base = 640000.0
    ref = float(oracle.rope(q, 50, base)[0] @ oracle.rope(k, 20, base)[0])
    for shift in (1, 999, 65536):
        got = float(oracle.rope(q, 50 + shift, base)[0] @ oracle.rope(k, 20 + shift, base)[0])
        assert abs(got - ref) < 1e-9 * max(1.0, abs(ref))
    np.testing.assert_allclose(oracle.rope(oracle.rope(q, 300, base), 45, base), oracle.rope(q, 345, base),
                               rtol=1e-12, atol=1e-12)


# ------------------------------------------------ gRet input projection pins

def test_qkvg_project_columns_and_brute_force():
    """The four projections side by side: with W holding unit columns that pick
    input channels, q, k, v and the logits are those channels; and the product
    itself against explicit Python sums on a tiny case."""
    B, N, dm, H, d = 1, 3, 8, 2, 2
    rng = np.random.default_rng(51)
    X = rng.standard_normal((B, N, dm))
    W = np.zeros((dm, 3 * H * d + H))
    for col in range(W.shape[1]):
        W[col % dm, col] = 1.0
    q, k, v, lg = oracle.qkvg_project(X, W, H, d)
    cols = [c % dm for c in range(W.shape[1])]
    np.testing.assert_array_equal(q.reshape(B, N, H * d), X[..., cols[0:4]])
    np.testing.assert_array_equal(k.reshape(B, N, H * d), X[..., cols[4:8]])
    np.testing.assert_array_equal(v.reshape(B, N, H * d), X[..., cols[8:12]])
    np.testing.assert_array_equal(lg, X[..., cols[12:14]])
    W2 = rng.standard_normal(W.shape)
    q2, _, _, lg2 = oracle.qkvg_project(X, W2, H, d)
    for n in range(N):
        for j in range(H * d):
            ref = sum(X[0, n, c] * W2[c, j] for c in range(dm))
            assert abs(q2.reshape(B, N, H * d)[0, n, j] - ref) < 1e-12
        for g in range(H):
            ref = sum(X[0, n, c] * W2[c, 3 * H * d + g] for c in range(dm))
            assert abs(lg2[0, n, g] - ref) < 1e-12
