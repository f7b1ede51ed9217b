"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Each pin is written so that a plausible mistake in the oracle (a dropped term,
a wrong sign, the decay on the wrong axis, the read before the write, the
wrong operand) fails at least one of them; ``test_planted_mistakes_are_caught``
plants such mistakes in scratch copies of the oracle source and checks that.

Sources:
- "Understanding Kimi K3's Attention": state-update equation (factored form),
  delta form, regression loss and its gradient step, readout equation.
- "Hybrid Attention", section "KDA: don't write the same information twice":
  the worked example (predict 2, target 6, beta 0.5 -> 4).
- "Kimi K3.1 and the Road From Softmax Attention to Kimi Delta Attention",
  section "3. The delta rule": beta = 1 with a unit key reads back v exactly;
  the toy memory experiment and its printed errors.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


def _unit(x, axis=-1):
    return x / np.linalg.norm(x, axis=axis, keepdims=True)


def _rand_case(rng, T, H, dk, dv, unit_keys=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_keys:
        q, k = _unit(q), _unit(k)
    v = rng.standard_normal((T, H, dv))
    g = np.maximum(-5.0, -np.logaddexp(0.0, -(rng.standard_normal((T, H, dk)) + 1.0)))
    beta = rng.uniform(0.0, 1.0, (T, H))
    return q, k, v, g, beta


# ----------------------------------------------------------------------------
# the pins, each a plain function of an oracle object (so that the planted-
# mistake test can run them against a mutated build)
# ----------------------------------------------------------------------------

def pin_worked_example(orc, gold):
    """Hybrid Attention, worked example: prediction 2, target 6, beta 0.5 -> 4
    along a normalised key; untouched key directions keep their content."""
    dk, dv = 4, 3
    key = np.zeros(dk); key[2] = 1.0                       # unit key e_2
    S0 = RNG.standard_normal((1, 1, dk, dv))
    S0[0, 0, 2, :] = gold["prediction"]                    # S0^T k = prediction
    v = np.full((1, 1, dv), gold["target"])
    g = np.full((1, 1, dk), gold["g"])
    beta = np.full((1, 1), gold["beta"])
    out, fin = orc.prefill(key[None, None], key[None, None], v, g, beta, init_state=S0)
    assert np.allclose(fin[0, 0].T @ key, gold["expected_after_write"], atol=1e-15, rtol=0)
    assert np.allclose(out[0, 0], gold["expected_after_write"], atol=1e-15, rtol=0)
    other = [i for i in range(dk) if i != 2]
    assert np.array_equal(fin[0, 0][other], S0[0, 0][other])


def pin_beta_one_reads_back_v(orc):
    """The delta rule, beta = 1, unit key: reading k after the write returns v
    exactly.  With q = k the readout after the write is therefore v_t for any
    decay and any prior state."""
    T, H, dk, dv = 12, 2, 5, 3
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    beta[:] = 1.0
    S0 = RNG.standard_normal((1, H, dk, dv))
    out, _ = orc.prefill(k, k, v, g, beta, init_state=S0)
    assert np.max(np.abs(out - v)) < 1e-12


def pin_beta_zero_closed_form(orc):
    """beta = 0 writes nothing: S_t = Diag(exp(Gamma_t)) S_0 with Gamma_t the
    running sum of g, and o_t = S_t^T q_t."""
    T, H, dk, dv = 9, 2, 4, 6
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    beta[:] = 0.0
    S0 = RNG.standard_normal((1, H, dk, dv))
    out, fin = orc.prefill(q, k, v, g, beta, init_state=S0)
    Gam = np.cumsum(g, axis=0)                            # [T, H, dk]
    for h in range(H):
        for t in range(T):
            St = np.exp(Gam[t, h])[:, None] * S0[0, h]
            assert np.allclose(out[t, h], St.T @ q[t, h], atol=1e-13, rtol=1e-13)
        assert np.allclose(fin[0, h], np.exp(Gam[-1, h])[:, None] * S0[0, h],
                           atol=1e-13, rtol=1e-13)


def pin_toy_memory(orc, gold):
    """The associative-memory experiment of "Kimi K3.1 and the Road From
    Softmax Attention to Kimi Delta Attention", section "3. The delta rule:
    write only the correction", with alpha = 1 (g = 0) and beta = 1.

    Only the draws follow the page (seed, d, pair count, and the order: the
    unit keys, then the values, then the replacement value of key 0), since
    the printed errors depend on them.  The memory of plain linear attention
    is then the closed form K^T V of the written stream, checked without the
    oracle; the delta-rule memory is the oracle's final state, checked against
    the unrolled products of the factored update as well.  The read-out error
    of a key is |S^T key - target| / |target|, compared at two decimals."""
    d, n = int(gold["d"]), int(gold["pairs"])
    rng = np.random.default_rng(int(gold["seed"]))
    keys = _unit(rng.standard_normal((n, d)))     # row by row: the same draws as one at a time
    vals = rng.standard_normal((n, d))
    replacement = rng.standard_normal(d)
    stream_k = np.vstack([keys, keys[0]])         # the n pairs, then key 0 once more
    stream_v = np.vstack([vals, replacement])

    def read_error(S, i, target):
        return float(np.linalg.norm(S.T @ keys[i] - target) / np.linalg.norm(target))

    linear = stream_k.T @ stream_v                # sum over the stream of k v^T
    assert round(read_error(linear, 0, replacement), 2) == gold["linear_attention_key0"]
    assert round(read_error(linear, 5, vals[5]), 2) == gold["linear_attention_key5"]

    T = stream_k.shape[0]
    _, fin = orc.prefill(stream_k[:, None], stream_k[:, None], stream_v[:, None],
                         np.zeros((T, 1, d)), np.ones((T, 1)))
    delta = fin[0, 0]
    _, unrolled = _brute(stream_k, stream_k, stream_v, np.zeros((T, d)), np.ones(T),
                         np.zeros((d, d)))
    np.testing.assert_allclose(delta, unrolled, rtol=0, atol=1e-10)
    assert round(read_error(delta, 0, replacement), 2) == gold["delta_rule_key0"]
    assert round(read_error(delta, 5, vals[5]), 2) == gold["delta_rule_key5"]


def _brute(q, k, v, g, beta, S0):
    """Unrolled products of the factored state-update equation with explicit
    d_k x d_k transition matrices A_s = (I - beta_s k_s k_s^T) Diag(exp g_s):
    S_t = A_t...A_1 S_0 + sum_s A_t...A_{s+1} beta_s k_s v_s^T; o_t = S_t^T q_t."""
    T, dk = k.shape
    A = [(np.eye(dk) - beta[s] * np.outer(k[s], k[s])) @ np.diag(np.exp(g[s])) for s in range(T)]
    outs = []
    for t in range(T):
        P = np.eye(dk)
        S = np.zeros_like(S0)
        for s in range(t, -1, -1):
            S = S + P @ (beta[s] * np.outer(k[s], v[s]))
            P = P @ A[s]
        S = S + P @ S0
        outs.append(S.T @ q[t])
    return np.stack(outs), S


def pin_brute_force(orc):
    """Whole recurrence against brute-force unrolled products (tiny sizes,
    d_k != d_v so that a transposed operand cannot pass, keys not normalised
    so that no unit-norm shortcut hides a mistake)."""
    for (T, dk, dv) in [(1, 3, 2), (5, 3, 4), (8, 4, 4), (7, 2, 5)]:
        H = 2
        q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv, unit_keys=False)
        S0 = RNG.standard_normal((1, H, dk, dv))
        out, fin = orc.prefill(q, k, v, g, beta, init_state=S0)
        for h in range(H):
            o_ref, S_ref = _brute(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], S0[0, h])
            assert np.max(np.abs(out[:, h] - o_ref)) < 1e-12
            assert np.max(np.abs(fin[0, h] - S_ref)) < 1e-12


def pin_gradient_step(orc):
    """One token equals one gradient-descent step of size beta on
    L(S) = 1/2 ||S^T k - v||^2 taken from the decayed state Diag(alpha) S_0.
    The gradient is taken by central finite differences (exact for a
    quadratic up to rounding), not from its closed form."""
    dk, dv = 4, 3
    q, k, v, g, beta = _rand_case(RNG, 1, 1, dk, dv, unit_keys=False)
    S0 = RNG.standard_normal((1, 1, dk, dv))
    M = np.exp(g[0, 0])[:, None] * S0[0, 0]

    def loss(S):
        r = S.T @ k[0, 0] - v[0, 0]
        return 0.5 * r @ r

    h = 1e-3
    grad = np.zeros_like(M)
    for i in range(dk):
        for j in range(dv):
            E = np.zeros_like(M); E[i, j] = h
            grad[i, j] = (loss(M + E) - loss(M - E)) / (2 * h)
    _, fin = orc.prefill(q, k, v, g, beta, init_state=S0)
    assert np.max(np.abs(fin[0, 0] - (M - beta[0, 0] * grad))) < 1e-9


def pin_norm_bound(orc):
    """For unit keys and beta in [0,1], (I - beta k k^T) has spectral norm <= 1
    and alpha <= 1, so ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||."""
    T, H, dk, dv = 40, 1, 8, 8
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    S = RNG.standard_normal((1, H, dk, dv))
    for t in range(T):
        _, S_next = orc.prefill(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                beta[t:t + 1], init_state=S)
        lhs = np.linalg.norm(S_next[0, 0], 2)
        rhs = np.linalg.norm(S[0, 0], 2) + beta[t, 0] * np.linalg.norm(v[t, 0])
        assert lhs <= rhs * (1 + 1e-12)
        S = S_next


def pin_gate_closed_forms(orc):
    """Gate prologue, g = g_min Sigmoid(e^{A_h} z) and beta = Sigmoid(logit)
    ("Understanding Kimi K3's Attention", log-decay bound and symbol table):
    - z = 0 gives g_min / 2 exactly, and a zero logit gives beta = 1/2;
    - with A_h = ln 2 and z = ln(3) / 2, Sigmoid(ln 3) = 3/4, so g = -3.75;
    - g tends to g_min as z grows and to 0 as z falls (alpha -> 1);
    - g(z) + g(-z) = g_min for any A_h;
    - a logit of ln 3 gives beta = 3/4."""
    T, H, dk = 3, 2, 4
    z = np.zeros((T, H, dk))
    z[1, 0, :] = np.log(3.0) / 2
    z[2, 1, 0], z[2, 1, 1] = 60.0, -800.0
    a_log = np.array([np.log(2.0), 0.0])
    bl = np.zeros((T, H))
    bl[1, 1] = np.log(3.0)
    g, beta = orc.gate(z, a_log, bl)
    assert np.all(g[0] == -2.5) and beta[0, 0] == 0.5
    assert abs(g[1, 0, 0] - (-3.75)) < 1e-14
    assert abs(beta[1, 1] - 0.75) < 1e-15
    assert abs(g[2, 1, 0] - (-5.0)) < 1e-14 and g[2, 1, 1] == 0.0
    rng = np.random.default_rng(5)
    zr = rng.normal(0.0, 3.0, (5, H, dk))
    a2 = rng.normal(0.0, 0.5, H)
    gp, _ = orc.gate(zr, a2, np.zeros((5, H)))
    gm, _ = orc.gate(-zr, a2, np.zeros((5, H)))
    assert np.allclose(gp + gm, -5.0, rtol=0, atol=1e-14)
    assert np.all((gp > -5.0) & (gp < 0.0))


def pin_output_gate_closed_forms(orc):
    """Output gate, y = Sigmoid(gate) . RMSNorm(o~) with RMSNorm over one
    head's d_v channels ("Inside Kimi K3", section "Sequence mixing"):
    - a constant row c (any sign) normalises to sign(c); a zero logit halves it;
    - a logit of ln 3 gives Sigmoid = 3/4, and the weight scales channel j;
    - with eps = 3 c^2 a constant row c gives c / sqrt(4 c^2) = sign(c) / 2;
    - each (token, head) row, whatever its scale, leaves with mean square 1
      under an open gate (rows are normalised one head at a time);
    - a zero row stays zero."""
    T, H, dv = 2, 3, 8
    o = np.empty((T, H, dv))
    o[:, 0, :] = 3.0
    o[:, 1, :] = -2.0
    o[:, 2, :] = 0.0
    y = orc.output_gate(o, np.zeros_like(o), eps=1e-30)
    assert np.allclose(y[:, 0], 0.5, rtol=0, atol=1e-15)
    assert np.allclose(y[:, 1], -0.5, rtol=0, atol=1e-15)
    assert np.all(y[:, 2] == 0.0)
    w = np.arange(1.0, dv + 1.0)
    y = orc.output_gate(np.ones((T, H, dv)), np.full((T, H, dv), np.log(3.0)), norm_weight=w,
                        eps=1e-30)
    assert np.allclose(y, 0.75 * w, rtol=1e-15, atol=0)
    y = orc.output_gate(o[:, :2], np.zeros((T, 2, dv)), eps=3.0 * 4.0)   # c = -2: eps = 3 c^2
    assert np.allclose(y[:, 1], -0.25, rtol=0, atol=1e-15)
    rng = np.random.default_rng(11)
    o = rng.standard_normal((4, 3, 16)) * np.array([1e-3, 1.0, 1e3])[None, :, None]
    y = orc.output_gate(o, np.full(o.shape, 40.0), eps=1e-30)
    assert np.allclose((y ** 2).mean(axis=-1), 1.0, rtol=1e-12, atol=0)
    assert np.all(np.sign(y) == np.sign(o))


def pin_scalar_decay_closed_forms(orc, gold):
    """Gated DeltaNet and the delta rule ("Kimi K3.1 and the Road ...",
    sections "3. The delta rule" and "4. Gating"):
    - without a decay (g_head None) the toy memory experiment gives the
      page's delta-rule errors 0.00 (rewritten key) and 0.36 (key 5);
    - beta = 0 writes nothing: S_t = exp(sum of g_head up to t) S_0, one
      factor per head (heads decay at different rates);
    - brute-force unrolled products with the scalar transition
      alpha_s (I - beta_s k_s k_s^T)."""
    d, n = int(gold["d"]), int(gold["pairs"])
    rng = np.random.default_rng(int(gold["seed"]))
    keys = np.stack([_unit(rng.standard_normal(d)) for _ in range(n)])
    vals = np.stack([rng.standard_normal(d) for _ in range(n)])
    new0 = rng.standard_normal(d)
    ks = np.concatenate([keys, keys[:1]])
    vs = np.concatenate([vals, new0[None]])
    _, fin = orc.prefill_scalar_decay(ks[:, None], ks[:, None], vs[:, None], None,
                                      np.ones((ks.shape[0], 1)))
    S = fin[0, 0]
    rel = lambda key, target: np.linalg.norm(S.T @ key - target) / np.linalg.norm(target)
    assert round(rel(keys[0], new0), 2) == gold["delta_rule_key0"]
    assert round(rel(keys[5], vals[5]), 2) == gold["delta_rule_key5"]

    T, H, dk, dv = 9, 2, 4, 6
    q, k, v, _, beta = _rand_case(RNG, T, H, dk, dv)
    gh = -RNG.uniform(0.0, 1.0, (T, H)) * np.array([0.2, 2.0])
    S0 = RNG.standard_normal((1, H, dk, dv))
    out, fin = orc.prefill_scalar_decay(q, k, v, gh, np.zeros((T, H)), init_state=S0)
    for h in range(H):
        for t in range(T):
            St = np.exp(gh[:t + 1, h].sum()) * S0[0, h]
            assert np.allclose(out[t, h], St.T @ q[t, h], atol=1e-13, rtol=1e-13)
        assert np.allclose(fin[0, h], np.exp(gh[:, h].sum()) * S0[0, h], atol=1e-13, rtol=1e-13)

    for (T, dk, dv) in [(5, 3, 4), (8, 4, 2)]:
        q, k, v, _, beta = _rand_case(RNG, T, H, dk, dv, unit_keys=False)
        gh = -RNG.uniform(0.0, 1.5, (T, H))
        S0 = RNG.standard_normal((1, H, dk, dv))
        out, fin = orc.prefill_scalar_decay(q, k, v, gh, beta, init_state=S0)
        for h in range(H):
            g_full = np.repeat(gh[:, h:h + 1], dk, axis=1)
            o_ref, S_ref = _brute(q[:, h], k[:, h], v[:, h], g_full, beta[:, h], S0[0, h])
            assert np.max(np.abs(out[:, h] - o_ref)) < 1e-12
            assert np.max(np.abs(fin[0, h] - S_ref)) < 1e-12


def pin_backward_finite_differences(orc):
    """Gradients of L = sum(d_out . o) + sum(d_final . S_T), reverse mode,
    against central finite differences of the (pinned) forward for every
    entry of q, k, v, g, beta and the initial states; a packed batch with an
    empty sequence, keys not normalised, gates inside the domain."""
    T, H, dk, dv = 6, 2, 3, 4
    rng = np.random.default_rng(21)
    q = rng.standard_normal((T, H, dk))
    k = 0.6 * rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.2, 2.0, (T, H, dk))
    beta = rng.uniform(0.2, 0.8, (T, H))
    cu = np.array([0, 4, 4, 6], np.int32)
    S0 = rng.standard_normal((3, H, dk, dv))
    do = rng.standard_normal((T, H, dv))
    dfin = rng.standard_normal((3, H, dk, dv))
    args = dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)

    def loss(a):
        o, f = orc.prefill(a["q"], a["k"], a["v"], a["g"], a["beta"], init_state=a["S0"],
                           cu_seqlens=cu, num_threads=1)
        return float((o * do).sum() + (f * dfin).sum())

    r = orc.backward(q, k, v, g, beta, do, dfin, init_state=S0, cu_seqlens=cu)
    eps = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("S0", "d_init_state")):
        fd = np.zeros_like(args[name])
        for idx in np.ndindex(fd.shape):
            a = dict(args)
            x = args[name].copy(); x[idx] += eps; a[name] = x; lp = loss(a)
            x = args[name].copy(); x[idx] -= eps; a[name] = x; lm = loss(a)
            fd[idx] = (lp - lm) / (2 * eps)
        assert np.max(np.abs(r[key] - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd))), name


def pin_backward_beta_zero_closed_form(orc):
    """beta = 0 writes nothing: o_t = (Diag(e^{Gamma_t}) S_0)^T q_t and
    S_T = Diag(e^{Gamma_T}) S_0, so dq_t = Diag(e^{Gamma_t}) S_0 do_t, dk = dv = 0,
    dS_0 = sum_t Diag(e^{Gamma_t}) q_t do_t^T + Diag(e^{Gamma_T}) dS_T, and
    dg_t[i] = sum over s >= t of e^{Gamma_s[i]} q_s[i] (S_0 do_s)[i] plus the
    final-state term e^{Gamma_T[i]} (S_0 . dS_T summed over values)[i]."""
    T, H, dk, dv = 7, 2, 4, 3
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    beta[:] = 0.0
    S0 = RNG.standard_normal((1, H, dk, dv))
    do = RNG.standard_normal((T, H, dv))
    dfin = RNG.standard_normal((1, H, dk, dv))
    r = orc.backward(q, k, v, g, beta, do, dfin, init_state=S0)
    Gam = np.cumsum(g, axis=0)
    for h in range(H):
        E = np.exp(Gam[:, h])                            # [T, dk]
        S0h, dfh = S0[0, h], dfin[0, h]
        dq = E * (do[:, h] @ S0h.T)
        assert np.allclose(r["dq"][:, h], dq, atol=1e-12, rtol=1e-12)
        dS0 = (E * q[:, h]).T @ do[:, h] + E[-1][:, None] * dfh
        assert np.allclose(r["d_init_state"][0, h], dS0, atol=1e-12, rtol=1e-12)
        per_s = E * q[:, h] * (do[:, h] @ S0h.T)         # [T, dk]: term of o_s
        dg = np.cumsum(per_s[::-1], axis=0)[::-1] + E[-1] * (S0h * dfh).sum(axis=1)
        assert np.allclose(r["dg"][:, h], dg, atol=1e-12, rtol=1e-12)
    assert np.all(r["dk"] == 0.0) and np.all(r["dv"] == 0.0)


def _conv_ref(x_seq, state, w):
    """Causal width-4 convolution of one channel's inputs by numpy's own
    convolution: the three carried inputs first, then the sequence; tap 3 of
    w multiplies the current token, so the kernel is w reversed."""
    full = np.concatenate([state, x_seq])
    return np.convolve(full, w[::-1])[3:3 + len(x_seq)]


def pin_qkv_prologue_convolution(orc):
    """The short convolution ("Inside Kimi K3", section "Sequence mixing":
    width 4; "Hybrid Attention", section "KDA: don't write the same
    information twice": causal), seen through the value stream.  Since
    Swish(c) - Swish(-c) = c (Sigmoid(c) + Sigmoid(-c) = 1) and the
    convolution is linear, v(x) - v(-x) is the convolution itself:
    - an impulse at token 2 returns the taps newest first, nothing before it;
    - a packed batch (an empty sequence included) matches numpy's
      convolution of each sequence, restarted at each sequence start, with
      the carried conv state in front;
    - the state out is the last three inputs of [state; sequence]."""
    T, H, d = 8, 1, 2
    rng = np.random.default_rng(21)
    w = rng.standard_normal((3, H, d, 4))
    x = np.zeros((T, H, d))
    x[2, 0, 0] = 1.5
    z = np.zeros_like(x)
    v1 = orc.qkv_prologue(z, z, x, w)[2]
    v2 = orc.qkv_prologue(z, z, -x, w)[2]
    c = v1 - v2
    want = np.zeros(T)
    want[2:6] = 1.5 * w[2, 0, 0, ::-1]
    assert np.allclose(c[:, 0, 0], want, rtol=0, atol=1e-14)
    assert np.all(c[:, 0, 1] == 0.0)
    lens = [5, 0, 2, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, d = int(cu[-1]), 2, 3
    x = rng.standard_normal((T, H, d))
    w = rng.standard_normal((3, H, d, 4))
    st = rng.standard_normal((len(lens), 3, 3, H, d))
    z = np.zeros_like(x)
    for state in (None, st):
        v1 = orc.qkv_prologue(z, z, x, w, cu_seqlens=cu, conv_state=state)
        v2 = orc.qkv_prologue(z, z, -x, w, cu_seqlens=cu,
                              conv_state=None if state is None else -state)
        c = v1[2] - v2[2]
        for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
            for h in range(H):
                for j in range(d):
                    s0 = np.zeros(3) if state is None else state[n, 2, :, h, j]
                    assert np.allclose(c[a:b, h, j], _conv_ref(x[a:b, h, j], s0, w[2, h, j]),
                                       rtol=1e-13, atol=1e-13)
                    full = np.concatenate([s0, x[a:b, h, j]])
                    assert np.array_equal(v1[3][n, 2, :, h, j], full[-3:])


def pin_qkv_prologue_swish_norm(orc):
    """Swish and L2Norm ("Understanding Kimi K3's Attention", symbol table:
    q, k = L2Norm(Swish(ShortConv(.))), v = Swish(ShortConv(.))):
    - a current-token tap of 1 and an input of ln 3 give ln 3 Sigmoid(ln 3)
      = 0.75 ln 3 on v; an input of 0 gives 0 on every stream;
    - q is v's row, computed from q's own input and weights, divided by its
      norm over the head's channels (heads of very different scale each end
      with norm 1), and with eps = 3 |v|^2 by 2 |v|; the same for k;
    - v is not normalised."""
    T, H, d = 3, 2, 4
    w = np.zeros((3, H, d, 4))
    w[..., 3] = 1.0
    x = np.full((T, H, d), np.log(3.0))
    z = np.zeros_like(x)
    q, k, v, _ = orc.qkv_prologue(z, z, x, w)
    assert np.allclose(v, 0.75 * np.log(3.0), rtol=1e-15, atol=0)
    assert np.all(q == 0.0) and np.all(k == 0.0)
    rng = np.random.default_rng(22)
    T, H, d = 6, 3, 5
    xs = [rng.standard_normal((T, H, d)) * np.array([1e-3, 1.0, 30.0])[None, :, None]
          for _ in range(3)]
    w = rng.standard_normal((3, H, d, 4))
    q, k, v, _ = orc.qkv_prologue(*xs, w, eps=1e-30)
    assert not np.allclose(np.linalg.norm(v, axis=-1), 1.0)
    for s, got in ((0, q), (1, k)):
        w2 = w.copy()
        w2[2] = w[s]
        ref = orc.qkv_prologue(np.zeros((T, H, d)), xs[1], xs[s], w2, eps=1e-30)[2]
        nrm = np.linalg.norm(ref, axis=-1, keepdims=True)
        assert np.allclose(got, ref / nrm, rtol=1e-12, atol=0)
        big = orc.qkv_prologue(*xs, w, eps=1.0)[s]
        assert np.allclose(big, ref / np.sqrt(nrm ** 2 + 1.0), rtol=1e-12, atol=0)
    one = [xs[0][:, :1], xs[1][:, :1], xs[2][:, :1]]
    vv = orc.qkv_prologue(*one, w[:, :1], eps=1e-30)[2]
    w2 = w[:, :1].copy()
    w2[0] = w2[2]
    e3 = 3.0 * float((vv[0, 0] ** 2).sum())
    qq = orc.qkv_prologue(one[2], one[1], one[2], w2, eps=e3)[0]
    assert np.allclose(qq[0, 0], vv[0, 0] / (2.0 * np.sqrt(e3 / 3.0)), rtol=1e-12, atol=0)


PINS = [pin_worked_example, pin_beta_one_reads_back_v, pin_beta_zero_closed_form,
        pin_toy_memory, pin_brute_force, pin_gradient_step, pin_norm_bound,
        pin_gate_closed_forms, pin_output_gate_closed_forms, pin_scalar_decay_closed_forms,
        pin_backward_finite_differences, pin_backward_beta_zero_closed_form,
        pin_qkv_prologue_convolution, pin_qkv_prologue_swish_norm]


def _run_pin(pin, orc, golden):
    if pin is pin_worked_example:
        pin(orc, golden("worked_delta_example.txt"))
    elif pin is pin_toy_memory or pin is pin_scalar_decay_closed_forms:
        pin(orc, golden("toy_delta_memory.txt"))
    else:
        pin(orc)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, golden):
    _run_pin(pin, oracle._load(), golden)


# ----------------------------------------------------------------------------
# host logic of the oracle (packing, empty sequences, domain, decode)
# ----------------------------------------------------------------------------

def test_packed_equals_separate():
    lens = [5, 0, 11, 1, 7]
    H, dk, dv = 2, 4, 3
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta = _rand_case(RNG, int(cu[-1]), H, dk, dv)
    S0 = RNG.standard_normal((len(lens), H, dk, dv))
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0, cu_seqlens=cu)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        o1, f1 = oracle.prefill(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b],
                                init_state=S0[n:n + 1])
        assert np.array_equal(out[a:b], o1)
        assert np.array_equal(fin[n], f1[0])
    assert np.array_equal(fin[1], S0[1])       # zero-length: final = initial


def test_split_resume():
    """final_state of a prefix is the initial state of the rest."""
    T, H, dk, dv = 23, 2, 4, 5
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    out, fin = oracle.prefill(q, k, v, g, beta)
    o1, f1 = oracle.prefill(q[:9], k[:9], v[:9], g[:9], beta[:9])
    o2, f2 = oracle.prefill(q[9:], k[9:], v[9:], g[9:], beta[9:], init_state=f1)
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(f2, fin)


def test_decode_is_one_token():
    N, H, dk, dv = 3, 2, 4, 4
    q, k, v, g, beta = _rand_case(RNG, N, H, dk, dv)
    S0 = RNG.standard_normal((N, H, dk, dv))
    o_dec, s_dec = oracle.decode(q, k, v, g, beta, S0)
    for n in range(N):
        o1, f1 = oracle.prefill(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1],
                                beta[n:n + 1], init_state=S0[n:n + 1])
        assert np.array_equal(o_dec[n], o1[0])
        assert np.array_equal(s_dec[n], f1[0])


def test_equal_length_default_layout():
    T, N, H, dk, dv = 12, 3, 1, 3, 3
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    cu = np.arange(0, T + 1, T // N, dtype=np.int32)
    a = oracle.prefill(q, k, v, g, beta, cu_seqlens=cu)
    b = oracle.prefill(q, k, v, g, beta, num_seqs=N)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("bad", ["g_low", "g_pos", "beta_high", "cu_bad"])
def test_domain_rejected(bad):
    T, H, dk, dv = 4, 1, 2, 2
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    cu = None
    if bad == "g_low":
        g[1, 0, 0] = -5.5
    elif bad == "g_pos":
        g[2, 0, 1] = 0.1
    elif bad == "beta_high":
        beta[0, 0] = 1.5
    else:
        cu = np.array([0, 3, 2, 4], np.int32)
    with pytest.raises(ValueError):
        oracle.prefill(q, k, v, g, beta, cu_seqlens=cu)


def test_threads_do_not_change_results():
    T, H, dk, dv = 30, 7, 8, 8
    q, k, v, g, beta = _rand_case(RNG, T, H, dk, dv)
    a = oracle.prefill(q, k, v, g, beta, num_threads=1)
    b = oracle.prefill(q, k, v, g, beta, num_threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ----------------------------------------------------------------------------
# planted mistakes (in scratch copies of the oracle, on the CPU)
# ----------------------------------------------------------------------------

MUTANTS = {
    "no_decay": ("alpha[i] = exp(gt[i]);", "alpha[i] = 1.0;"),
    "decay_sign": ("alpha[i] = exp(gt[i]);", "alpha[i] = exp(-gt[i]);"),
    "decay_on_value_axis": ("S[i * dv + j] *= alpha[i];", "S[i * dv + j] *= alpha[j % dk];"),
    "correction_sign": ("u[j] = bt * (vt[j] - p[j]);", "u[j] = bt * (vt[j] + p[j]);"),
    "beta_dropped": ("u[j] = bt * (vt[j] - p[j]);", "u[j] = (vt[j] - p[j]);"),
    "predict_with_q": ("p[j] += S[i * dv + j] * kt[i];", "p[j] += S[i * dv + j] * qt[i];"),
    "read_before_write": ("ot[j] += S[i * dv + j] * qt[i];",
                          "ot[j] += (S[i * dv + j] - kt[i] * u[j]) * qt[i];"),
    "write_with_q": ("S[i * dv + j] += kt[i] * u[j];", "S[i * dv + j] += qt[i] * u[j];"),
    "gate_scale_dropped": ("g[i] = KDA_ORACLE_G_MIN * sigmoid(scale * z[i]);",
                           "g[i] = KDA_ORACLE_G_MIN * sigmoid(z[i]);"),
    "gate_sign": ("g[i] = KDA_ORACLE_G_MIN * sigmoid(scale * z[i]);",
                  "g[i] = KDA_ORACLE_G_MIN * sigmoid(-scale * z[i]);"),
    "gate_beta_raw": ("beta[t * num_heads + h] = sigmoid(beta_logit[t * num_heads + h]);",
                      "beta[t * num_heads + h] = beta_logit[t * num_heads + h];"),
    "scalar_decay_ignored": ("g_head ? g_head[t * num_heads + h] : 0.0;", "0.0;"),
    "scalar_decay_one_head": ("g_head ? g_head[t * num_heads + h] : 0.0;",
                              "g_head ? g_head[t * num_heads] : 0.0;"),
    "bwd_no_prediction_term": ("            dkt[i] += acc;", "            dkt[i] += 0.0 * acc;"),
    "bwd_no_decay": ("for (int64_t j = 0; j < dv; ++j) dS[i * dv + j] = al[i] * dM[i * dv + j];",
                     "for (int64_t j = 0; j < dv; ++j) dS[i * dv + j] = dM[i * dv + j];"),
    "bwd_dbeta_sign": ("db += du[j] * (vt[j] - pp[j]);", "db += du[j] * (vt[j] + pp[j]);"),
    "bwd_dg_no_alpha": ("dgt[i] = al[i] * ga;", "dgt[i] = ga;"),
    "bwd_read_before_write": ("acc += St[i * dv + j] * dot[j];", "acc += Sp[i * dv + j] * dot[j];"),
    "ogate_sum_not_mean": ("const double rinv = 1.0 / sqrt(ss / d_v + eps);",
                           "const double rinv = 1.0 / sqrt(ss + eps);"),
    "ogate_eps_outside_root": ("const double rinv = 1.0 / sqrt(ss / d_v + eps);",
                               "const double rinv = 1.0 / (sqrt(ss / d_v) + eps);"),
    "ogate_gate_sign": ("y[row + j] = sigmoid(gate_logit[row + j]) * o[row + j] * rinv * w;",
                        "y[row + j] = sigmoid(-gate_logit[row + j]) * o[row + j] * rinv * w;"),
    "ogate_weight_dropped": ("const double w = norm_weight ? norm_weight[j] : 1.0;",
                             "const double w = 1.0;"),
    "ogate_norm_over_heads": ("            double ss = 0.0;\n            for (int32_t j = 0; j < d_v; ++j) ss += o[row + j] * o[row + j];",
                              "            double ss = 0.0;\n            for (int32_t j = 0; j < d_v; ++j) ss += o[t * num_heads * (int64_t)d_v + j] * o[t * num_heads * (int64_t)d_v + j];"),
    "conv_taps_reversed": ("c += w[3 - i] * XIN(t - i, h, j);", "c += w[i] * XIN(t - i, h, j);"),
    "conv_not_restarted": ("((u) >= a ? x[", "((u) >= 0 ? x["),
    "conv_state_reversed": ("((u) - a + 3)) * H", "(a - (u) - 1)) * H"),
    "conv_state_out_reversed": ("XIN(b - 3 + p, h, j);", "XIN(b - 1 - p, h, j);"),
    "swish_without_gate": ("row[j] = c * sigmoid(c);", "row[j] = c;"),
    "swish_gate_sign": ("row[j] = c * sigmoid(c);", "row[j] = c * sigmoid(-c);"),
    "l2norm_eps_outside_root": ("const double inv = 1.0 / sqrt(ss + eps);",
                                "const double inv = 1.0 / (sqrt(ss) + eps);"),
    "l2norm_on_v": ("            if (s < 2) {", "            if (s < 3) {"),
    "l2norm_not_on_k": ("            if (s < 2) {", "            if (s < 1) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path, golden):
    src_dir = os.path.dirname(oracle.__file__)
    src = open(os.path.join(src_dir, "kda_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    shutil.copy(os.path.join(src_dir, "kda_oracle.h"), tmp_path / "kda_oracle.h")
    (tmp_path / "m.c").write_text(src.replace(old, new))
    so = tmp_path / f"libmut_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(tmp_path / "m.c"), "-lm"], check=True)
    mutant = oracle.Oracle(str(so))
    failed = []
    for pin in PINS:
        try:
            _run_pin(pin, mutant, golden)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{name}' passed every pin"
