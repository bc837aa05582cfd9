"""Pins of the float64 oracle against what the mathematics fixes (CPU only).

The pages print no worked values for the gated delta rule, so the oracle is pinned by:
  * hand-evaluated tokens (tests/golden/scalar_delta_rule.txt),
  * closed forms (softplus(0) = ln 2, sigmoid(0) = 1/2, one-hot conv taps, unit l2 norm,
    gated norm with w = 1),
  * special cases that reduce to a textbook result: g = 0, beta = 1 with orthonormal keys is an
    exact associative memory; beta = 0 only decays the state by exp(g),
  * brute force on tiny inputs against an independently written dense form (explicit
    (I - beta k k^T) matrices, the conv as a convolution over the explicitly padded sequence,
    GQA by explicit head duplication),
  * the chunkwise WY/UT form equals the token-by-token recurrence,
  * continuation: prefill(T) then decode(T+1) equals prefill(T+1),
  * invariants: row permutation, untouched slots, padding rows, snapshot compaction,
  * the projections: integer brute force against exact Python arithmetic, permutation
    weights, and the stacked input projection's split checked feature by feature.
"""
import math
import os

import numpy as np
import pytest

import oracle
from gated_deltanet_linear_09_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scalar_delta_rule.txt")


# ----------------------------------------------------------------------------- golden

def _golden():
    scalar, matrix = [], {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "scalar":
                scalar.append([float(x) for x in parts[2:]])
            elif parts[0] == "matrix":
                matrix[parts[1]] = np.array([float(x) for x in parts[2:]])
    return scalar, matrix


def test_golden_scalar_tokens():
    scalar, _ = _golden()
    S = np.zeros((1, 1))
    for g, beta, k, v, q, s_after, o_exp in scalar:
        o = oracle.core_step(S, [k], [v], [q], g, beta)
        assert S[0, 0] == pytest.approx(s_after, abs=1e-15)
        assert o[0] == pytest.approx(o_exp, abs=1e-15)


def test_golden_matrix_token():
    _, m = _golden()
    S = m["S0"].reshape(2, 3).copy()
    o = oracle.core_step(S, m["k"], m["v"], m["q"], m["g"][0], m["beta"][0])
    np.testing.assert_allclose(S, m["S1"].reshape(2, 3), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o, m["o"], rtol=0, atol=1e-15)


# ----------------------------------------------------------------------------- closed forms

def test_scalar_closed_forms():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.silu(0.0) == 0.0
    assert oracle.softplus(50.0) == pytest.approx(50.0, rel=1e-15)
    assert oracle.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert oracle.softplus(800.0) == 800.0          # no overflow
    assert oracle.silu(3.0) == pytest.approx(3.0 / (1.0 + math.exp(-3.0)), rel=1e-15)
    # g = -exp(A_log) * softplus(a + dt_bias): A_log = 0, a = -dt_bias -> g = -ln 2
    g, beta = oracle.gates(0.0, 0.37, -0.37, 0.0)
    assert g == pytest.approx(-math.log(2.0), abs=1e-15)
    assert beta == 0.5
    # exp(A_log) scales linearly: A_log = ln 16 -> 16x the A_log = 0 decay
    g16, _ = oracle.gates(math.log(16.0), 0.2, 0.5, 0.0)
    g1, _ = oracle.gates(0.0, 0.2, 0.5, 0.0)
    assert g16 == pytest.approx(16.0 * g1, rel=1e-14)
    _, b_big = oracle.gates(0.0, 0.0, 0.0, 30.0)
    assert b_big == pytest.approx(1.0, abs=1e-12)


def test_conv_one_hot_taps():
    C, K = 6, 4
    rng = np.random.default_rng(1)
    xs = rng.standard_normal((9, C))
    # tap K-1 (current token) one-hot -> y = SiLU(x_t)
    w = np.zeros((C, K)); w[:, K - 1] = 1.0
    st = np.zeros((K - 1, C))
    for t in range(9):
        y = oracle.conv_step(st, w, xs[t])
        np.testing.assert_allclose(y, xs[t] / (1 + np.exp(-xs[t])), rtol=1e-15, atol=0)
    # the state holds the last K-1 raw inputs, oldest first
    np.testing.assert_array_equal(st, xs[-(K - 1):])
    # tap 0 one-hot -> the input delayed by K-1 (zero before the sequence starts)
    w = np.zeros((C, K)); w[:, 0] = 1.0
    st = np.zeros((K - 1, C))
    for t in range(9):
        y = oracle.conv_step(st, w, xs[t])
        ref = xs[t - (K - 1)] if t >= K - 1 else np.zeros(C)
        np.testing.assert_allclose(y, ref / (1 + np.exp(-ref)), rtol=1e-15, atol=0)
    # per-channel weights: channel c uses row c of w only
    w = np.zeros((C, K)); w[2, 1] = 3.0
    st = np.zeros((K - 1, C))
    for t in range(5):
        y = oracle.conv_step(st, w, xs[t])
    pre = 3.0 * xs[5 - 1 - 2, 2]    # tap 1 of K=4 weights x_{t-2}
    assert y[2] == pytest.approx(pre / (1 + math.exp(-pre)), rel=1e-15)
    assert np.all(y[[0, 1, 3, 4, 5]] == 0.0)


def test_l2norm_and_gated_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(37) * 5
    y = oracle.l2norm(x, 0.0)
    assert np.linalg.norm(y) == pytest.approx(1.0, abs=1e-15)
    np.testing.assert_allclose(y * np.linalg.norm(x), x, rtol=1e-14)
    y2 = oracle.l2norm(x, 0.0, scale=0.25)
    np.testing.assert_allclose(y2, 0.25 * y, rtol=1e-15)
    # eps enters under the root: a tiny vector is not blown up to unit norm
    tiny = np.full(4, 1e-8)
    assert np.linalg.norm(oracle.l2norm(tiny, 1e-6)) < 1e-4
    # gated norm with w = 1, z -> +large: SiLU(z) ~= z, so out / z has unit rms
    o = rng.standard_normal(64) * 3
    z = np.full(64, 40.0)
    out = oracle.gated_rmsnorm(o, z, np.ones(64), 0.0)
    assert math.sqrt(np.mean((out / 40.0) ** 2)) == pytest.approx(1.0, abs=1e-12)
    # z = 0 gates everything off; the norm weight is per channel
    assert np.all(oracle.gated_rmsnorm(o, np.zeros(64), np.ones(64), 1e-6) == 0.0)
    w = rng.standard_normal(64)
    np.testing.assert_allclose(oracle.gated_rmsnorm(o, z, w, 0.0), out * w, rtol=1e-14)


# ----------------------------------------------------------------------------- special cases

def test_associative_memory():
    """g = 0, beta = 1, orthonormal keys: after the writes S^T k_j = v_j exactly."""
    dk, dv, m = 8, 5, 6
    rng = np.random.default_rng(3)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :m].T
    vals = rng.standard_normal((m, dv))
    S = np.zeros((dk, dv))
    for j in range(m):
        o = oracle.core_step(S, keys[j], vals[j], keys[j], 0.0, 1.0)
        np.testing.assert_allclose(o, vals[j], atol=1e-13)
    for j in range(m):
        np.testing.assert_allclose(S.T @ keys[j], vals[j], atol=1e-13)
    # a key orthogonal to all written ones reads zero
    np.testing.assert_allclose(S.T @ Qm[:, m], np.zeros(dv), atol=1e-13)
    # writing the same key again overwrites (delta rule), it does not accumulate
    newv = rng.standard_normal(dv)
    oracle.core_step(S, keys[2], newv, keys[2], 0.0, 1.0)
    np.testing.assert_allclose(S.T @ keys[2], newv, atol=1e-13)
    np.testing.assert_allclose(S.T @ keys[1], vals[1], atol=1e-13)


def test_beta_zero_only_decays():
    dk, dv = 6, 7
    rng = np.random.default_rng(4)
    S = rng.standard_normal((dk, dv))
    for g in (0.0, -0.3, -5.0, -50.0):
        S0 = S.copy()
        q = rng.standard_normal(dk)
        o = oracle.core_step(S, rng.standard_normal(dk), rng.standard_normal(dv), q, g, 0.0)
        np.testing.assert_array_equal(S, S0 * math.exp(g))
        np.testing.assert_allclose(o, (S0 * math.exp(g)).T @ q, rtol=1e-13, atol=1e-300)


def test_partial_beta_interpolates():
    """One token with g = 0: S^T k moves from the old read to v by the fraction beta*|k|^2."""
    dk, dv = 5, 3
    rng = np.random.default_rng(5)
    k = rng.standard_normal(dk); k /= np.linalg.norm(k)
    S = rng.standard_normal((dk, dv))
    old = S.T @ k
    v = rng.standard_normal(dv)
    oracle.core_step(S, k, v, k, 0.0, 0.3)
    np.testing.assert_allclose(S.T @ k, old + 0.3 * (v - old), rtol=1e-13)


# ----------------------------------------------------------------------------- brute force

def _naive_layer(geo, w, rec0, conv0, xs):
    """Independent dense restatement for ONE request over a token sequence.

    The conv is evaluated as a convolution over the explicitly prepended history
    (conv0 rows, then the tokens); GQA by duplicating each K-head r times; the delta rule
    with the explicit matrix (I - beta k k^T).  Returns (outs [T][Hv*dv], S [Hv][dk][dv],
    conv_state [K-1][C])."""
    Hk, Hv, dk, dv, K = geo.Hk, geo.Hv, geo.dk, geo.dv, geo.K
    r = Hv // Hk
    qs = geo.q_scale_eff
    hist = np.concatenate([conv0, xs["qkv"]], axis=0)            # [(K-1)+T][C]
    T = xs["qkv"].shape[0]
    S = rec0.copy()
    outs = np.zeros((T, Hv * dv))
    for t in range(T):
        window = hist[t:t + K]                                    # K rows ending at token t
        pre = np.einsum("jc,cj->c", window, w["conv_w"])
        y = pre / (1.0 + np.exp(-pre))
        q = y[:Hk * dk].reshape(Hk, dk)
        k = y[Hk * dk:2 * Hk * dk].reshape(Hk, dk)
        v = y[2 * Hk * dk:].reshape(Hv, dv)
        q = np.repeat(q, r, axis=0); k = np.repeat(k, r, axis=0)
        for h in range(Hv):
            qh = q[h] / np.sqrt(q[h] @ q[h] + geo.l2_eps) * qs
            kh = k[h] / np.sqrt(k[h] @ k[h] + geo.l2_eps)
            x = xs["a"][t, h] + w["dt_bias"][h]
            sp = np.log1p(np.exp(x)) if x < 30 else x
            g = -np.exp(w["A_log"][h]) * sp
            beta = 1.0 / (1.0 + np.exp(-xs["b"][t, h]))
            M = np.exp(g) * (np.eye(dk) - beta * np.outer(kh, kh))
            S[h] = M @ S[h] + beta * np.outer(kh, v[h])
            o = S[h].T @ qh
            zz = xs["z"][t, h * dv:(h + 1) * dv]
            outs[t, h * dv:(h + 1) * dv] = (o / np.sqrt(np.mean(o * o) + geo.norm_eps)
                                            * w["norm_w"] * zz / (1.0 + np.exp(-zz)))
    return outs, S, hist[-(K - 1):].copy()


def _f64(d):
    return {k: np.asarray(v, np.float64) for k, v in d.items()}


@pytest.mark.parametrize("Hk,Hv,dk,dv", [(2, 4, 3, 2), (1, 3, 4, 5), (2, 2, 2, 2), (1, 1, 1, 1)])
def test_brute_force_decode_and_prefill(Hk, Hv, dk, dv):
    geo = synth.Geometry(Hk, Hv, dk, dv, 4, synth.F32)
    w = _f64(synth.make_weights(geo, 11))
    rec, conv = synth.make_pool(geo, 3, 12, prefilled=True)
    rec = rec.astype(np.float64); conv = conv.astype(np.float64)
    T = 7
    xs = _f64(synth.make_token_inputs(geo, T, 13))
    slot = 1
    ref_out, ref_S, ref_conv = _naive_layer(geo, w, rec[slot], conv[slot], xs)
    # decode: T single-row steps into slot 1
    r2, c2 = rec.copy(), conv.copy()
    for t in range(T):
        rc, out = oracle.decode_step(geo.oracle_dims(), w, r2, c2, [slot],
                                     xs["qkv"][t:t + 1], xs["z"][t:t + 1], xs["a"][t:t + 1],
                                     xs["b"][t:t + 1])
        assert rc == 0
        np.testing.assert_allclose(out[0], ref_out[t], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r2[slot], ref_S, rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(c2[slot], ref_conv)
    np.testing.assert_array_equal(r2[[0, 2]], rec[[0, 2]])
    # prefill continuing from the slot's state gives the same
    r3, c3 = rec.copy(), conv.copy()
    rc, out = oracle.prefill(geo.oracle_dims(), w, r3, c3, [0, T], [slot], [1], xs["qkv"], xs["z"],
                             xs["a"], xs["b"])
    assert rc == 0
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r3[slot], ref_S, rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(c3[slot], ref_conv)


def test_gqa_reduces_to_duplicated_heads():
    """Hv = 2*Hk equals Hk' = Hv with every K-head's q/k channels duplicated in place."""
    g2 = synth.Geometry(1, 2, 4, 3, 4, synth.F32)
    g1 = synth.Geometry(2, 2, 4, 3, 4, synth.F32)
    w2 = _f64(synth.make_weights(g2, 21))
    xs2 = _f64(synth.make_token_inputs(g2, 5, 22))
    dk = 4

    def dup(x):   # [.., q(4) k(4) v(6)] -> [.., q q k k v]
        q, k, v = x[..., :dk], x[..., dk:2 * dk], x[..., 2 * dk:]
        return np.concatenate([q, q, k, k, v], axis=-1)
    w1 = dict(w2); w1["conv_w"] = dup(w2["conv_w"].T).T.copy()
    xs1 = dict(xs2); xs1["qkv"] = dup(xs2["qkv"])
    outs = []
    for geo, w, xs in ((g2, w2, xs2), (g1, w1, xs1)):
        rec = np.zeros((1, 2, 4, 3)); conv = np.zeros((1, 3, geo.cqkv))
        rc, out = oracle.prefill(geo.oracle_dims(), w, rec, conv, [0, 5], [0], [0], xs["qkv"],
                                 xs["z"], xs["a"], xs["b"])
        assert rc == 0
        outs.append((out, rec))
    np.testing.assert_allclose(outs[0][0], outs[1][0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(outs[0][1], outs[1][1], rtol=1e-14, atol=1e-16)


def test_gqa_head_map_is_repeat_interleave():
    """V-head h reads K-head h // r: zeroing K-head 1's q channels changes V-heads 2,3 only."""
    geo = synth.Geometry(2, 4, 4, 2, 4, synth.F32)
    w = _f64(synth.make_weights(geo, 31))
    w["conv_w"][:] = 0.0
    w["conv_w"][:, 3] = 1.0
    xs = _f64(synth.make_token_inputs(geo, 1, 32))
    rec = synth.make_pool(geo, 1, 33, True)[0].astype(np.float64)
    conv = np.zeros((1, 3, geo.cqkv))
    _, o1 = oracle.decode_step(geo.oracle_dims(), w, rec.copy(), conv.copy(), [0], xs["qkv"],
                               xs["z"], xs["a"], xs["b"])
    xs2 = dict(xs); xs2["qkv"] = xs["qkv"].copy(); xs2["qkv"][0, 4:8] *= -1.0   # q of K-head 1
    _, o2 = oracle.decode_step(geo.oracle_dims(), w, rec.copy(), conv.copy(), [0], xs2["qkv"],
                               xs["z"], xs["a"], xs["b"])
    dv = 2
    np.testing.assert_array_equal(o1[0, :2 * dv], o2[0, :2 * dv])
    assert np.all(o1[0, 2 * dv:] != o2[0, 2 * dv:])


# ----------------------------------------------------------------------------- chunkwise

def _prefill_case(geo, lens, seed, has_init, prefilled=True):
    w = _f64(synth.make_weights(geo, seed))
    n = len(lens)
    rec, conv = synth.make_pool(geo, n + 2, seed + 1, prefilled=prefilled)
    cu = synth.cu_seqlens(lens)
    xs = _f64(synth.make_token_inputs(geo, int(cu[-1]), seed + 2))
    slots = np.arange(n, dtype=np.int32)[::-1] + 1
    return w, rec.astype(np.float64), conv.astype(np.float64), cu, slots, np.array(has_init,
                                                                                  np.uint8), xs


@pytest.mark.parametrize("chunk", [1, 2, 3, 16, 64])
def test_chunkwise_equals_sequential(chunk):
    geo = synth.Geometry(2, 4, 16, 8, 4, synth.F32)
    lens = [1, 5, 64, 65, 130, 3]
    w, rec, conv, cu, slots, hi, xs = _prefill_case(geo, lens, 40, [0, 1, 0, 1, 1, 0])
    r1, c1 = rec.copy(), conv.copy()
    rc, o1 = oracle.prefill(geo.oracle_dims(), w, r1, c1, cu, slots, hi, xs["qkv"], xs["z"],
                            xs["a"], xs["b"])
    assert rc == 0
    r2, c2 = rec.copy(), conv.copy()
    rc, o2 = oracle.prefill_chunkwise(geo.oracle_dims(), w, r2, c2, cu, slots, hi, xs["qkv"],
                                      xs["z"], xs["a"], xs["b"], chunk)
    assert rc == 0
    assert np.max(np.abs(o1 - o2)) <= 1e-12 * max(1.0, np.max(np.abs(o1)))
    assert np.linalg.norm(r1 - r2) <= 1e-12 * np.linalg.norm(r1)
    np.testing.assert_array_equal(c1, c2)


def test_chunkwise_survives_extreme_decay():
    """A_log = ln 16 and large a: the within-chunk cumulative decay reaches about -1e3; the chunk
    form never forms exp(+gamma), so it stays finite and equal to the recurrence."""
    geo = synth.Geometry(1, 2, 8, 8, 4, synth.F32)
    w, rec, conv, cu, slots, hi, xs = _prefill_case(geo, [64, 64], 50, [1, 0])
    w["A_log"][:] = math.log(16.0)
    xs["a"][:] = 3.0
    r1, c1 = rec.copy(), conv.copy()
    _, o1 = oracle.prefill(geo.oracle_dims(), w, r1, c1, cu, slots, hi, xs["qkv"], xs["z"],
                           xs["a"], xs["b"])
    r2, c2 = rec.copy(), conv.copy()
    _, o2 = oracle.prefill_chunkwise(geo.oracle_dims(), w, r2, c2, cu, slots, hi, xs["qkv"],
                                     xs["z"], xs["a"], xs["b"], 64)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(r2))
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(r2, r1, rtol=1e-11, atol=1e-300)


# ----------------------------------------------------------------------------- continuation

def test_prefill_then_decode_equals_longer_prefill():
    geo = synth.Geometry(2, 4, 16, 8, 4, synth.F32)
    T = 20
    w, rec, conv, cu, slots, hi, xs = _prefill_case(geo, [T + 1], 60, [0])
    # prefill(T+1) from zero state
    rA, cA = rec.copy(), conv.copy()
    _, oA = oracle.prefill(geo.oracle_dims(), w, rA, cA, [0, T + 1], [1], [0], xs["qkv"], xs["z"],
                           xs["a"], xs["b"])
    # prefill(T) then one decode step of token T
    rB, cB = rec.copy(), conv.copy()
    _, oB = oracle.prefill(geo.oracle_dims(), w, rB, cB, [0, T], [1], [0], xs["qkv"][:T],
                           xs["z"][:T], xs["a"][:T], xs["b"][:T])
    _, od = oracle.decode_step(geo.oracle_dims(), w, rB, cB, [1], xs["qkv"][T:], xs["z"][T:],
                               xs["a"][T:], xs["b"][T:])
    np.testing.assert_allclose(oB, oA[:T], rtol=0, atol=0)
    np.testing.assert_allclose(od[0], oA[T], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(rB, rA, rtol=1e-13, atol=1e-16)
    np.testing.assert_array_equal(cB, cA)
    # and split prefill with has_initial_state = 1 continues exactly (also via the chunk form)
    rC, cC = rec.copy(), conv.copy()
    oracle.prefill_chunkwise(geo.oracle_dims(), w, rC, cC, [0, 7], [1], [0], xs["qkv"][:7],
                             xs["z"][:7], xs["a"][:7], xs["b"][:7], 4)
    _, oC = oracle.prefill_chunkwise(geo.oracle_dims(), w, rC, cC, [0, T + 1 - 7], [1], [1],
                                     xs["qkv"][7:], xs["z"][7:], xs["a"][7:], xs["b"][7:], 4)
    np.testing.assert_allclose(oC, oA[7:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(rC, rA, rtol=1e-12, atol=1e-15)


def test_short_sequence_conv_state_keeps_history():
    """A 1-token continuation keeps the older raw inputs in the conv state (K-1 = 3 rows)."""
    geo = synth.Geometry(1, 1, 2, 2, 4, synth.F32)
    w, rec, conv, cu, slots, hi, xs = _prefill_case(geo, [1], 70, [1])
    c_before = conv[slots[0]].copy()
    oracle.prefill(geo.oracle_dims(), w, rec, conv, [0, 1], slots, [1], xs["qkv"], xs["z"],
                   xs["a"], xs["b"])
    np.testing.assert_array_equal(conv[slots[0]][:2], c_before[1:])
    np.testing.assert_array_equal(conv[slots[0]][2], xs["qkv"][0])
    # and a fresh (has_initial_state = 0) 1-token sequence has zeros before it
    rec2, conv2 = rec.copy(), conv.copy()
    oracle.prefill(geo.oracle_dims(), w, rec2, conv2, [0, 1], slots, [0], xs["qkv"], xs["z"],
                   xs["a"], xs["b"])
    np.testing.assert_array_equal(conv2[slots[0]][:2], np.zeros((2, geo.cqkv)))


# ----------------------------------------------------------------------------- invariants

def test_row_permutation_and_untouched_slots_and_padding():
    geo = synth.Geometry(2, 4, 8, 8, 4, synth.F32)
    w = _f64(synth.make_weights(geo, 80))
    rec, conv = (x.astype(np.float64) for x in synth.make_pool(geo, 6, 81, True))
    xs = _f64(synth.make_token_inputs(geo, 4, 82))
    slots = np.array([4, 1, -1, 3], np.int32)
    r1, c1 = rec.copy(), conv.copy()
    rc, o1 = oracle.decode_step(geo.oracle_dims(), w, r1, c1, slots, xs["qkv"], xs["z"], xs["a"],
                                xs["b"])
    assert rc == 0
    assert np.all(o1[2] == 0.0)                                # padding row: zero output
    for s in (0, 2, 5):                                        # untouched slots
        np.testing.assert_array_equal(r1[s], rec[s])
        np.testing.assert_array_equal(c1[s], conv[s])
    perm = np.array([3, 0, 2, 1])
    r2, c2 = rec.copy(), conv.copy()
    _, o2 = oracle.decode_step(geo.oracle_dims(), w, r2, c2, slots[perm], xs["qkv"][perm],
                               xs["z"][perm], xs["a"][perm], xs["b"][perm])
    np.testing.assert_array_equal(o2, o1[perm])
    np.testing.assert_array_equal(r2, r1)
    np.testing.assert_array_equal(c2, c1)
    # an out-of-range slot is reported and its row skipped
    r3, c3 = rec.copy(), conv.copy()
    rc, o3 = oracle.decode_step(geo.oracle_dims(), w, r3, c3, np.array([9, 1, -1, 3], np.int32),
                                xs["qkv"], xs["z"], xs["a"], xs["b"])
    assert rc == -1 and np.all(o3[0] == 0.0)
    np.testing.assert_array_equal(o3[1], o1[1])


def test_conv1d_update_matches_decode_conv():
    geo = synth.Geometry(2, 4, 8, 8, 4, synth.F32)
    w = _f64(synth.make_weights(geo, 90))
    conv = synth.make_pool(geo, 3, 91, True)[1].astype(np.float64)
    xs = _f64(synth.make_token_inputs(geo, 2, 92))
    c1 = conv.copy()
    rc, y = oracle.conv1d_update(w["conv_w"], c1, [2, 0], xs["qkv"])
    assert rc == 0
    for i, s in enumerate((2, 0)):
        window = np.concatenate([conv[s], xs["qkv"][i:i + 1]], axis=0)
        pre = np.einsum("jc,cj->c", window, w["conv_w"])
        np.testing.assert_allclose(y[i], pre / (1 + np.exp(-pre)), rtol=1e-14, atol=1e-300)
        np.testing.assert_array_equal(c1[s], window[1:])
    np.testing.assert_array_equal(c1[1], conv[1])


def test_compaction_is_snapshot_gather():
    rng = np.random.default_rng(100)
    N = 12
    rec = rng.standard_normal((N, 2, 3, 3))
    conv = rng.standard_normal((N, 3, 5))
    live = np.sort(rng.choice(N, 7, replace=False)).astype(np.int32)
    src = live[::-1].copy()                       # overlapping, reversed order
    dst = np.arange(7, dtype=np.int32)
    r1, c1 = rec.copy(), conv.copy()
    assert oracle.state_compact(r1, c1, src, dst) == 0
    np.testing.assert_array_equal(r1[:7], rec[src])
    np.testing.assert_array_equal(c1[:7], conv[src])
    np.testing.assert_array_equal(r1[7:], rec[7:])
    # a cycle (swap) needs the snapshot semantics
    r2, c2 = rec.copy(), conv.copy()
    oracle.state_compact(r2, c2, np.array([0, 1], np.int32), np.array([1, 0], np.int32))
    np.testing.assert_array_equal(r2[0], rec[1]); np.testing.assert_array_equal(r2[1], rec[0])
    # duplicate destinations are rejected
    assert oracle.state_compact(rec.copy(), conv.copy(), np.array([0, 1], np.int32),
                                np.array([2, 2], np.int32)) == -1


# ----------------------------------------------------------------------------- projections

def test_linear_integer_brute_force():
    """Small integers are exact in float64, so the oracle's y = x w^T must equal Python's exact
    integer sum of x[m][k] * w[n][k] -- with N != K, so a transposed weight index cannot pass."""
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 7
    x = rng.integers(-9, 10, size=(M, K))
    w = rng.integers(-9, 10, size=(N, K))
    y = oracle.linear(x, w)
    assert y.shape == (M, N)
    for m in range(M):
        for n in range(N):
            exact = sum(int(x[m][k]) * int(w[n][k]) for k in range(K))
            assert y[m][n] == exact, (m, n)


def test_linear_permutation_weight_selects_features():
    """A permutation matrix as the weight reorders the input features: y[:, n] = x[:, p[n]]."""
    rng = np.random.default_rng(12)
    K = 9
    p = rng.permutation(K)
    w = np.zeros((K, K))
    w[np.arange(K), p] = 1.0
    x = rng.standard_normal((4, K))
    np.testing.assert_array_equal(oracle.linear(x, w), x[:, p])


def test_in_proj_split_order_and_boundaries():
    """Weight row n = (n + 1) e_0 and x[m][0] = m + 1 make output feature n of row m equal
    (m + 1)(n + 1), so every output says which stacked row produced it: qkv takes rows
    [0, Cqkv), z the next Hv*dv, then b (Hv rows), then a (Hv rows)."""
    dims = dict(Hk=2, Hv=4, dk=8, dv=6)
    cqkv, zd, Hv = 2 * 2 * 8 + 4 * 6, 4 * 6, 4
    n = cqkv + zd + 2 * Hv
    hidden, rows = 5, 3
    w_in = np.zeros((n, hidden))
    w_in[:, 0] = np.arange(1, n + 1)
    x = np.zeros((rows, hidden))
    x[:, 0] = np.arange(1, rows + 1)
    got = oracle.in_proj(dims, x, w_in)
    r = np.arange(1, rows + 1)[:, None]
    np.testing.assert_array_equal(got["qkv"], r * np.arange(1, cqkv + 1))
    np.testing.assert_array_equal(got["z"], r * np.arange(cqkv + 1, cqkv + zd + 1))
    np.testing.assert_array_equal(got["b"], r * np.arange(cqkv + zd + 1, cqkv + zd + Hv + 1))
    np.testing.assert_array_equal(got["a"], r * np.arange(cqkv + zd + Hv + 1, n + 1))


def test_out_proj_shape_and_linearity():
    """out_proj maps [rows][Hv*dv] to [rows][hidden] and is linear in its input."""
    rng = np.random.default_rng(13)
    o1, o2 = rng.standard_normal((2, 3, 12))
    w = rng.standard_normal((7, 12))
    y1, y2, y12 = oracle.out_proj(o1, w), oracle.out_proj(o2, w), oracle.out_proj(2 * o1 - o2, w)
    assert y1.shape == (3, 7)
    np.testing.assert_allclose(y12, 2 * y1 - y2, rtol=0, atol=1e-12)
