"""Checks that pin the CPU oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:

* numpy's library convolution (the causal conv and its tap order),
* a dense matrix-product statement of the gated delta rule,
  S_T = S_0 P_1 ... P_T + sum_s b_s v_s k_s^T P_{s+1} ... P_T with
  P_t = a_t (I - b_t k_t k_t^T)  (Yang, Kautz & Hatamizadeh, "Gated Delta
  Networks", the gated delta rule written as a product of generalised
  Householder transitions),
* closed forms and special cases (b = 0 is pure decay; a = b = 1 with
  orthonormal keys stores v exactly; key-head sharing),
* the accepted-prefix commit semantics of "Add request-owned eight-way MTP
  serving for Qwen 35B", section 4 (keep = 0 restores the pre-verification
  state; keep = k equals a run over the first k tokens; inactive rows inert),
* an independent fp64 chunked (WY / UT-transform) evaluation of the prompt
  recurrence (the chunked form that "MTP inference: review and commit
  structure", Verification and limits, says differs from the sequential one
  only in rounding),
* a hand-worked example stored under tests/golden/,
* for greedy acceptance: numpy's argmax (the first index of the maximum),
  hand-built drafts whose accepted prefix is known by construction, and the
  defining properties of the accepted prefix,
* for the gated RMSNorm: torch's rms_norm and silu (double precision, CPU),
  and the unit root-mean-square of the normalised vector.

They are plain functions (not tests) so that ``test_oracle_pins.py`` can also
run them against builds of the oracle with planted mistakes and show that each
mistake is caught.
"""
from __future__ import annotations

import json
import os

import numpy as np
from scipy.special import expit

from speculative_decode_gated_gdn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS = 1e-6


# ---------------------------------------------------------------- numpy pieces
def np_conv(hist, x, w, act):
    """Causal conv by numpy.convolve over the explicit history (hist [C][3], x [n][C])."""
    n, C = x.shape
    xt = np.concatenate([hist.T, x], axis=0)
    y = np.empty((n, C))
    for c in range(C):
        y[:, c] = np.convolve(xt[:, c], w[c, ::-1], mode="valid")
    return y * expit(y) if act else y


def np_heads(y, H_k, H_v, d):
    """Split conv output [n][C] into normalised q (scaled), k per value head and v."""
    n = y.shape[0]
    q = y[:, : H_k * d].reshape(n, H_k, d)
    k = y[:, H_k * d: 2 * H_k * d].reshape(n, H_k, d)
    v = y[:, 2 * H_k * d:].reshape(n, H_v, d)
    qn = q / np.linalg.norm(np.concatenate([q, np.full((n, H_k, 1), np.sqrt(EPS))], -1), axis=-1,
                            keepdims=True) / np.sqrt(d)
    kn = k / np.linalg.norm(np.concatenate([k, np.full((n, H_k, 1), np.sqrt(EPS))], -1), axis=-1,
                            keepdims=True)
    rep = H_v // H_k
    return np.repeat(qn, rep, axis=1), np.repeat(kn, rep, axis=1), v


def dense_states(S0, k, v, g, beta):
    """Dense product form for one head: S0 [dv][dk], k/v [T][d], g/beta [T] -> S_t for t=1..T."""
    T, d = k.shape
    P = [np.exp(g[t]) * (np.eye(d) - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    out = []
    for t in range(1, T + 1):
        St = S0.copy()
        for r in range(t):
            St = St @ P[r]
        for s in range(t):
            term = beta[s] * np.outer(v[s], k[s])
            for r in range(s + 1, t):
                term = term @ P[r]
            St = St + term
        out.append(St)
    return out


def chunked_wy(S0, q, k, v, g, beta, chunk):
    """fp64 chunked form for one head (UT transform of the strictly lower block).

    Within a chunk with cumulative log-decay G and gamma = exp(G):
      A[t][s] = beta_t exp(G_t - G_s) k_t.k_s (s < t),  Tm = (I + A)^-1,
      W = Tm diag(beta gamma) K,  U = Tm diag(beta) V,  E = U - W S^T,
      O = diag(gamma) Q S^T + tril(exp(G_t - G_s) q_t.k_s) E,
      S <- gamma_n S + sum_s exp(G_n - G_s) e_s k_s^T.
    """
    S = S0.copy()
    L = len(g)
    out = np.zeros((L, S.shape[0]))
    for c0 in range(0, L, chunk):
        sl = slice(c0, min(c0 + chunk, L))
        K, Q, V, gg, bb = k[sl], q[sl], v[sl], g[sl], beta[sl]
        n = len(gg)
        G = np.cumsum(gg)
        gam = np.exp(G)
        Gam = np.exp(G[:, None] - G[None, :])
        A = np.tril(bb[:, None] * Gam * (K @ K.T), -1)
        Tm = np.linalg.inv(np.eye(n) + A)
        W = Tm @ ((bb * gam)[:, None] * K)
        U = Tm @ (bb[:, None] * V)
        E = U - W @ S.T
        out[sl] = gam[:, None] * (Q @ S.T) + np.tril(Gam * (Q @ K.T)) @ E
        S = gam[-1] * S + (E * np.exp(G[-1] - G)[:, None]).T @ K
    return S, out


def window_after(hist, x, k):
    """Last three raw inputs of hist ++ x[:k] per channel, as [C][3]."""
    seq = np.concatenate([hist.T, x[:k]], axis=0)
    return seq[-3:].T.copy()


def _rand_problem(seed, B, T, H_k, H_v, d):
    geom = synth.Geometry(B=B, T=T, H_k=H_k, H_v=H_v, d=d)
    st = synth.layer_state(geom, seed)
    cy = synth.cycle_inputs(geom, seed, 0)
    C = geom.C
    win = synth.normal(seed, "win", (B, C, 3))
    return dict(
        geom=geom,
        x=synth.bf16_to_f32(cy["x"][0]).astype(np.float64),
        w=synth.bf16_to_f32(st["conv_w"][0]).astype(np.float64),
        win=synth.bf16_to_f32(synth.bf16_bits(win)).astype(np.float64),
        g=cy["g"][0].astype(np.float64),
        beta=cy["beta"][0].astype(np.float64),
        S0=st["state"][0],
    )


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert err <= tol, f"{what}: max abs diff {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------- pins
def pin_conv_numpy(orc):
    rng_hist = synth.normal(11, "h", (7, 3))
    x = synth.normal(11, "x", (5, 7))
    w = synth.normal(11, "w", (7, 4))
    for act in (0, 1):
        _close(orc.causal_conv(rng_hist, x, w, act), np_conv(rng_hist, x, w, act), 1e-13,
               f"conv vs numpy.convolve act={act}")


def pin_conv_taps(orc):
    hist = synth.normal(12, "h", (3, 3))
    x = synth.normal(12, "x", (4, 3))
    e3 = np.tile([0.0, 0.0, 0.0, 1.0], (3, 1))
    assert np.array_equal(orc.causal_conv(hist, x, e3, 0), x), "w = e_3 must be the identity"
    e0 = np.tile([1.0, 0.0, 0.0, 0.0], (3, 1))
    xt = np.concatenate([hist.T, x], axis=0)
    assert np.array_equal(orc.causal_conv(hist, x, e0, 0), xt[:4]), "w = e_0 must delay by three"


def pin_dense_product(orc):
    p = _rand_problem(13, B=1, T=5, H_k=1, H_v=2, d=4)
    act = 1
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], p["beta"], p["S0"], np.ones(1, np.uint8),
                         H_k=1, act=act)
    y = np_conv(p["win"][0], p["x"][0], p["w"], act)
    q, k, v = np_heads(y, 1, 2, 4)
    for h in range(2):
        Sd = dense_states(p["S0"][0, h].astype(np.float64), k[:, h], v[:, h], p["g"][0, :, h],
                          p["beta"][0, :, h])
        for t in range(5):
            _close(Sall[0, t, h], Sd[t], 1e-12, f"state t={t} h={h} vs dense product form")
            _close(o[0, t, h], Sd[t] @ q[t, h], 1e-12, f"output t={t} h={h} vs S_t q_t")


def pin_dense_product_deep(orc):
    """The dense product form at the deep-draft shape the GPU path is checked
    at (T = 8, d = 128), with two value heads sharing one key head."""
    p = _rand_problem(19, B=1, T=8, H_k=1, H_v=2, d=128)
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], p["beta"], p["S0"], np.ones(1, np.uint8), H_k=1)
    q, k, v = np_heads(np_conv(p["win"][0], p["x"][0], p["w"], 1), 1, 2, 128)
    for h in range(2):
        Sd = dense_states(p["S0"][0, h].astype(np.float64), k[:, h], v[:, h], p["g"][0, :, h],
                          p["beta"][0, :, h])
        for t in range(8):
            _close(Sall[0, t, h], Sd[t], 1e-11, f"deep state t={t} h={h} vs dense product form")
            _close(o[0, t, h], Sd[t] @ q[t, h], 1e-11, f"deep output t={t} h={h} vs S_t q_t")


def pin_beta_zero(orc):
    p = _rand_problem(14, B=1, T=3, H_k=1, H_v=1, d=8)
    beta = np.zeros_like(p["beta"])
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], beta, p["S0"], np.ones(1, np.uint8), H_k=1)
    q, _, _ = np_heads(np_conv(p["win"][0], p["x"][0], p["w"], 1), 1, 1, 8)
    G = np.cumsum(p["g"][0, :, 0])
    for t in range(3):
        St = np.exp(G[t]) * p["S0"][0, 0].astype(np.float64)
        _close(Sall[0, t, 0], St, 1e-14, f"beta=0 pure decay t={t}")
        _close(o[0, t, 0], St @ q[t, 0], 1e-14, f"beta=0 output t={t}")


def _identity_problem(T, H_k, H_v, d, keys, queries, values, S0=None):
    """Identity conv (w = e_3, no activation, zero window) so raw inputs reach the rule unchanged."""
    C = 2 * H_k * d + H_v * d
    x = np.zeros((1, T, C))
    for t in range(T):
        x[0, t, : H_k * d] = queries[t].ravel()
        x[0, t, H_k * d: 2 * H_k * d] = keys[t].ravel()
        x[0, t, 2 * H_k * d:] = values[t].ravel()
    w = np.tile([0.0, 0.0, 0.0, 1.0], (C, 1))
    win = np.zeros((1, C, 3))
    if S0 is None:
        S0 = np.zeros((1, H_v, d, d), np.float32)
    return x, w, win, S0


def pin_orthonormal_store(orc):
    """a = b = 1, S0 = 0, orthonormal keys: S k_i = v_i, and q = k_i reads v_i / sqrt(d)."""
    T, d = 4, 8
    big = 1024.0  # raw key length; makes the 1e-6 norm epsilon negligible (1e-12 relative)
    keys = [big * np.eye(d)[t][None, :] for t in range(T)]
    vals = [synth.bf16_to_f32(synth.bf16_bits(synth.normal(15, f"v{t}", (1, d)))).astype(np.float64)
            for t in range(T)]
    x, w, win, S0 = _identity_problem(T, 1, 1, d, keys, keys, vals)
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    o, Sall = orc.verify(x, w, win, g, beta, S0, np.ones(1, np.uint8), H_k=1, act=0)
    for t in range(T):
        for i in range(t + 1):
            _close(Sall[0, t, 0] @ np.eye(d)[i], vals[i][0], 1e-9, f"S_{t} k_{i} = v_{i}")
        _close(o[0, t, 0], vals[t][0] / np.sqrt(d), 1e-9, f"o_{t} = v_{t}/sqrt(d)")


def pin_one_step_store(orc):
    """From any S0, one step with a = b = 1 gives S_1 k = v (the delta rule's defining property)."""
    d = 8
    kraw = synth.normal(16, "k", (1, d)) * 1000.0
    kn = kraw / np.linalg.norm(kraw)
    vals = synth.normal(16, "v", (1, d))
    S0 = synth.normal(16, "S", (1, 1, d, d)).astype(np.float32)
    x, w, win, S0 = _identity_problem(1, 1, 1, d, [kraw], [kraw], [vals], S0)
    o, Sall = orc.verify(x, w, win, np.zeros((1, 1, 1)), np.ones((1, 1, 1)), S0, np.ones(1, np.uint8),
                         H_k=1, act=0)
    _close(Sall[0, 0, 0] @ kn[0], vals[0], 1e-9, "S_1 k = v")


def pin_key_head_sharing(orc):
    """H_k=2, H_v=4: value heads 0,1 read key head 0 and heads 2,3 read key head 1."""
    d, T = 4, 1
    keys = [np.array([[1024.0, 0, 0, 0], [0, 1024.0, 0, 0]])]
    qs = [np.array([[0, 0, 1024.0, 0], [0, 0, 0, 1024.0]])]
    vals = [synth.normal(17, "v", (4, d))]
    x, w, win, S0 = _identity_problem(T, 2, 4, d, keys, qs, vals)
    o, Sall = orc.verify(x, w, win, np.zeros((1, T, 4)), np.ones((1, T, 4)), S0, np.ones(1, np.uint8),
                         H_k=2, act=0)
    for h in range(4):
        hk = h * 2 // 4
        expect = np.outer(vals[0][h], np.eye(d)[hk])
        _close(Sall[0, 0, h], expect, 1e-9, f"head {h} must read key head {hk}")
        _close(o[0, 0, h], np.zeros(d), 1e-9, f"head {h}: q orthogonal to k gives 0")


def pin_commit_prefix(orc):
    """commit(keep=k) equals a run over the first k tokens; offsets advance by k."""
    p = _rand_problem(18, B=2, T=3, H_k=1, H_v=2, d=8)
    act = np.ones(2, np.uint8)
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], p["beta"], p["S0"], act, H_k=1)
    for k in range(0, 4):
        S = p["S0"].copy()
        win = p["win"].copy()
        off = np.array([100, 7], np.int32)
        st = orc.commit(np.array([k, k], np.int32), act, Sall, p["x"], S, win, off)
        assert st == 0
        assert list(off) == [100 + k, 7 + k], f"offsets after keep={k}"
        for b in range(2):
            _close(win[b], window_after(p["win"][b], p["x"][b], k), 0.0, f"window keep={k}")
            if k == 0:
                assert np.array_equal(S[b], p["S0"][b]), "keep=0 must restore exactly"
            else:
                _, Sk = orc.verify(p["x"][b:b + 1, :k], p["w"], p["win"][b:b + 1], p["g"][b:b + 1, :k],
                                   p["beta"][b:b + 1, :k], p["S0"][b:b + 1], act[:1], H_k=1)
                assert np.array_equal(S[b], Sk[0, k - 1].astype(np.float32)), f"keep={k} state"


def pin_restore_and_inert(orc):
    p = _rand_problem(19, B=3, T=2, H_k=1, H_v=2, d=8)
    active = np.array([1, 0, 1], np.uint8)
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], p["beta"], p["S0"], active, H_k=1)
    assert np.all(o[1] == 0), "inactive rows output zeros"
    S = p["S0"].copy()
    win = p["win"].copy()
    off = np.array([5, 6, 7], np.int32)
    st = orc.commit(np.array([0, 2, 5], np.int32), active, Sall, p["x"], S, win, off)
    assert st == 1, "keep=5 > T on an active row must set status bit 0"
    assert np.array_equal(S, p["S0"]), "keep=0, inactive rows and bad keep leave state bytes"
    assert np.array_equal(win, p["win"]) and list(off) == [5, 6, 7]
    st = orc.commit(np.array([-1, 0, 0], np.int32), active, Sall, p["x"], S, win, off)
    assert st == 1 and np.array_equal(S, p["S0"]), "negative keep is treated as 0 and flagged"


def pin_prefill_is_verify_commit(orc):
    p = _rand_problem(20, B=2, T=5, H_k=1, H_v=2, d=8)
    act = np.ones(2, np.uint8)
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], p["beta"], p["S0"], act, H_k=1)
    S1, w1, off1 = p["S0"].copy(), p["win"].copy(), np.array([0, 3], np.int32)
    orc.commit(np.array([5, 5], np.int32), act, Sall, p["x"], S1, w1, off1)
    S2, w2, off2 = p["S0"].copy(), p["win"].copy(), np.array([0, 3], np.int32)
    o2 = orc.prefill(p["x"], p["w"], w2, p["g"], p["beta"], S2, off2, H_k=1)
    assert np.array_equal(S1, S2) and np.array_equal(w1, w2) and np.array_equal(off1, off2)
    _close(o, o2, 0.0, "prefill outputs equal verify outputs")


def pin_chunked_wy(orc):
    """Sequential prompt priming equals an fp64 chunked WY evaluation (chunk 64, ragged tail)."""
    L, d, H_v = 150, 8, 2
    p = _rand_problem(21, B=1, T=L, H_k=1, H_v=H_v, d=d)
    S = p["S0"].copy()
    win = p["win"].copy()
    off = np.zeros(1, np.int32)
    o = orc.prefill(p["x"], p["w"], win, p["g"], p["beta"], S, off, H_k=1)
    q, k, v = np_heads(np_conv(p["win"][0], p["x"][0], p["w"], 1), 1, H_v, d)
    for h in range(H_v):
        Sc, oc = chunked_wy(p["S0"][0, h].astype(np.float64), q[:, h], k[:, h], v[:, h],
                            p["g"][0, :, h], p["beta"][0, :, h], 64)
        _close(S[0, h], Sc, 1e-6 * max(1.0, np.abs(Sc).max()), f"head {h} final state (fp32 store)")
        _close(o[0, :, h], oc, 1e-10 * max(1.0, np.abs(oc).max()), f"head {h} outputs vs chunked WY")
    assert off[0] == L


def pin_golden_hand(orc):
    with open(os.path.join(GOLDEN, "hand_d2_T2.json")) as f:
        gd = json.load(f)
    x = np.array(gd["x"], np.float64)
    C = x.shape[2]
    w = np.tile(gd["conv_w_row"], (C, 1)).astype(np.float64)
    win = np.zeros((1, C, 3))
    g = np.array(gd["g"], np.float64)
    beta = np.array(gd["beta"], np.float64)
    S0 = np.array(gd["S0"], np.float32)
    o, Sall = orc.verify(x, w, win, g, beta, S0, np.ones(1, np.uint8), H_k=1, act=0)
    e = gd["expect"]
    tol = e["tol"]
    _close(Sall[0, 0, 0], e["S1"], tol, "hand S1")
    _close(Sall[0, 1, 0], e["S2"], tol, "hand S2")
    _close(o[0, 0, 0], e["o1"], tol, "hand o1")
    _close(o[0, 1, 0], e["o2"], tol, "hand o2")
    for keep, Sk in ((1, e["S1"]), (2, e["S2"])):
        S = S0.copy()
        wn = win.copy()
        off = np.array([gd["offset0"]], np.int32)
        orc.commit(np.array([keep], np.int32), np.ones(1, np.uint8), Sall, x, S, wn, off)
        _close(S[0, 0], Sk, tol, f"hand commit keep={keep}")
        assert off[0] == gd["offset0"] + keep
        expect_win = np.zeros((C, 3))
        for i in range(keep):
            expect_win[:, 3 - keep + i] = x[0, i]
        assert np.array_equal(wn[0], expect_win), f"hand window keep={keep}"


def pin_row_separable(orc):
    p = _rand_problem(22, B=3, T=2, H_k=2, H_v=4, d=8)
    act = np.ones(3, np.uint8)
    o, Sall = orc.verify(p["x"], p["w"], p["win"], p["g"], p["beta"], p["S0"], act, H_k=2)
    for b in range(3):
        ob, Sb = orc.verify(p["x"][b:b + 1], p["w"], p["win"][b:b + 1], p["g"][b:b + 1],
                            p["beta"][b:b + 1], p["S0"][b:b + 1], act[:1], H_k=2)
        assert np.array_equal(o[b], ob[0]) and np.array_equal(Sall[b], Sb[0]), f"row {b} separable"


def pin_accept_hand(orc):
    """Greedy acceptance on a hand-built case: targets are planted maxima, so
    the accepted prefix is known without running any argmax."""
    B, T, V = 4, 4, 7
    logits = np.zeros((B, T, V))
    targets = np.array([[3, 1, 6, 0], [2, 2, 5, 4], [0, 6, 1, 3], [5, 5, 5, 5]])
    for b in range(B):
        for t in range(T):
            logits[b, t, targets[b, t]] = 2.0 + t
    draft = np.full((B, T), -7, np.int32)
    draft[0, 1:] = [3, 1, 6]      # every draft accepted: keep = T
    draft[1, 1:] = [2, 9, 5]      # second draft rejected: keep = 2
    draft[2, 1:] = [4, 6, 1]      # first draft rejected: keep = 1
    draft[3, 1:] = [5, 5, 5]      # all accepted, but the row is inactive
    active = np.array([1, 1, 1, 0], np.uint8)
    keep, nxt = orc.accept(logits, draft, active)
    assert list(keep) == [4, 2, 1, 0], keep
    assert list(nxt) == [0, 2, 0, -1], nxt


def pin_accept_ties_and_nan(orc):
    """Ties go to the first index; NaN never wins; an all-NaN row gives 0."""
    logits = np.array([[[1.0, 5.0, 5.0, -2.0], [np.nan, 0.5, np.nan, 0.5]],
                       [[np.nan] * 4, [3.0, 3.0, 3.0, 3.0]]])
    draft = np.array([[0, 1], [0, 0]], np.int32)
    keep, nxt = orc.accept(logits, draft, np.ones(2, np.uint8))
    # row 0: target_0 = 1 (first of the tied 5.0s) == draft[0][1] -> keep 2, next = target_1 = 1
    # row 1: target_0 = 0 (all NaN) == draft[1][1] -> keep 2, next = target_1 = 0 (first of ties)
    assert list(keep) == [2, 2] and list(nxt) == [1, 0], (keep, nxt)


def pin_accept_random(orc):
    """Random logits against numpy's argmax and the defining properties of the
    accepted prefix (every accepted draft equals the previous target; the
    first rejected one does not)."""
    rng = np.random.default_rng(7)
    B, T, V = 24, 6, 97
    logits = rng.integers(-20, 20, size=(B, T, V)).astype(np.float64)  # many ties
    tgt = np.argmax(logits, axis=2)
    draft = rng.integers(0, V, size=(B, T)).astype(np.int32)
    for b in range(B):  # plant an accepted prefix of random length
        n = int(rng.integers(0, T))
        draft[b, 1:1 + n] = tgt[b, :n]
    active = (rng.random(B) < 0.8).astype(np.uint8)
    keep, nxt = orc.accept(logits, draft, active)
    for b in range(B):
        if not active[b]:
            assert keep[b] == 0 and nxt[b] == -1
            continue
        k = int(keep[b])
        assert 1 <= k <= T
        assert all(draft[b, t] == tgt[b, t - 1] for t in range(1, k))
        assert k == T or draft[b, k] != tgt[b, k - 1]
        assert nxt[b] == tgt[b, k - 1]


def pin_gated_rmsnorm(orc):
    """Gated RMSNorm against torch's library rms_norm and silu in float64, and
    its defining property: with w = 1 and the gate divided out, the vector has
    unit root mean square (up to eps)."""
    import torch
    rng = np.random.default_rng(11)
    o = rng.normal(size=(5, 3, 64)) * rng.uniform(0.01, 3.0, size=(5, 3, 1))
    z = rng.normal(size=o.shape) * 2.0
    w = rng.normal(size=64)
    eps = 1e-6
    y = orc.gated_rmsnorm(o, z, w, eps)
    to = torch.from_numpy(o)
    ref = torch.nn.functional.rms_norm(to, (64,), weight=torch.from_numpy(w), eps=eps) * \
        torch.nn.functional.silu(torch.from_numpy(z))
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    u = orc.gated_rmsnorm(o, np.full(o.shape, 30.0), np.ones(64), 0.0) / (30.0 / (1.0 + np.exp(-30.0)))
    assert np.allclose(np.sqrt((u ** 2).mean(axis=-1)), 1.0, rtol=1e-12)


ALL_PINS = [pin_conv_numpy, pin_conv_taps, pin_dense_product, pin_dense_product_deep, pin_beta_zero, pin_orthonormal_store,
            pin_one_step_store, pin_key_head_sharing, pin_commit_prefix, pin_restore_and_inert,
            pin_prefill_is_verify_commit, pin_chunked_wy, pin_golden_hand, pin_row_separable,
            pin_accept_hand, pin_accept_ties_and_nan, pin_accept_random, pin_gated_rmsnorm]
