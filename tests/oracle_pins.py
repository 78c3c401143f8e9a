"""Pins for the fp64 CPU oracle: checks against what the mathematics fixes.

None of these re-types the oracle's row loop.  Each check computes the same
quantity by a different route (dense d_k x d_k matrices, exact rationals, a
closed form, a chunked WY/UT evaluation) or checks an invariant the definition
implies.  Every function takes ``mutant`` so the mutation test can run the
whole set against the planted-mistake builds of the oracle; a pin raises
AssertionError when it fails.

The recurrence (page "Optimizing on-device inference for Apple Silicon",
section "Qwen creates three distinct workload shapes", the Gated DeltaNet
paragraph; gate and state fp32 per "Keep the recurrent state on-chip"):
    S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t.
"""
from fractions import Fraction

import numpy as np

import oracle

TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_case(seed, lengths, h_k, h_v, d_k, d_v, unit_k=True, state=True):
    r = _rng(seed)
    T = int(sum(lengths))
    q = r.standard_normal((T, h_k, d_k))
    k = r.standard_normal((T, h_k, d_k))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.standard_normal((T, h_v, d_v))
    g = -np.log1p(np.exp(r.standard_normal((T, h_v))))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, h_v))))
    s0 = r.standard_normal((len(lengths), h_v, d_v, d_k)) * 0.5 if state else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, g, beta, s0, cu


def _brute(q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, scale):
    """Dense evaluation: explicit (I - b k k^T) matrices and matrix products."""
    G = h_v // h_k
    N = len(cu) - 1
    o = np.full((q.shape[0], h_v, d_v), np.nan)
    st = np.zeros((N, h_v, d_v, d_k))
    eye = np.eye(d_k)
    for n in range(N):
        for h in range(h_v):
            S = s0[n, h].copy() if s0 is not None else np.zeros((d_v, d_k))
            for t in range(cu[n], cu[n + 1]):
                kk = k[t, h // G][:, None]          # d_k x 1
                qq = scale * q[t, h // G][:, None]  # d_k x 1
                vv = v[t, h][:, None]               # d_v x 1
                a = np.exp(g[t, h])
                b = beta[t, h]
                S = a * S @ (eye - b * kk @ kk.T) + b * vv @ kk.T
                o[t, h] = (S @ qq)[:, 0]
            st[n, h] = S
    return o, st


def _call(mutant, q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, scale=1.0):
    return oracle.prefill(q, k, v, g, beta, cu, h_k, h_v, d_k, d_v, state_in=s0, scale=scale,
                          threads=4, mutant=mutant)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    m = ~np.isnan(b)
    assert np.array_equal(np.isnan(a), np.isnan(b)), f"{what}: NaN pattern differs"
    err = np.max(np.abs(a[m] - b[m])) if m.any() else 0.0
    scale = max(1.0, float(np.max(np.abs(b[m]))) if m.any() else 1.0)
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol * scale:.3e}"


# --- I1: brute force with dense matrices ----------------------------------------------------
def pin_brute_force(mutant=0):
    """Several heads with shared key heads, d_k != d_v, varlen incl. an empty
    sequence, a random non-symmetric initial state and scale != 1."""
    lengths = [5, 0, 17, 64]
    h_k, h_v, d_k, d_v = 2, 4, 8, 12
    q, k, v, g, beta, s0, cu = _rand_case(11, lengths, h_k, h_v, d_k, d_v, unit_k=False)
    o_ref, st_ref = _brute(q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, 0.7)
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, 0.7)
    _close(o, o_ref, what="o")
    _close(st, st_ref, what="state")


def pin_brute_force_no_state(mutant=0):
    """NULL initial state means zeros; d_k > d_v."""
    lengths = [33]
    h_k, h_v, d_k, d_v = 1, 3, 16, 4
    q, k, v, g, beta, _, cu = _rand_case(12, lengths, h_k, h_v, d_k, d_v, state=False)
    o_ref, st_ref = _brute(q, k, v, g, beta, None, cu, h_k, h_v, d_k, d_v, 1.0)
    o, st = _call(mutant, q, k, v, g, beta, None, cu, h_k, h_v, d_k, d_v)
    _close(o, o_ref, what="o")
    _close(st, st_ref, what="state")


# --- exact rationals: the definition in Fraction arithmetic ----------------------------------
def pin_exact_rational(mutant=0):
    """Two tokens, d_k = 2, d_v = 3, alpha = 1/2 and 1 (g = -ln 2 and 0),
    beta = 1/2 and 1/4, small-integer vectors: the dense definition evaluated
    exactly in rationals, compared with the fp64 oracle."""
    F = Fraction
    k = [[F(1), F(2)], [F(-1), F(1)]]
    q = [[F(3), F(-1)], [F(1), F(1)]]
    v = [[F(1), F(0), F(-2)], [F(2), F(1), F(1)]]
    alpha = [F(1, 2), F(1)]
    beta = [F(1, 2), F(1, 4)]
    S = [[F(1), F(0)], [F(0), F(2)], [F(-1), F(1)]]  # d_v x d_k, not symmetric
    outs = []
    for t in range(2):
        M = [[(F(1) if a == b else F(0)) - beta[t] * k[t][a] * k[t][b] for b in range(2)]
             for a in range(2)]
        S = [[alpha[t] * sum(S[i][c] * M[c][j] for c in range(2)) + beta[t] * v[t][i] * k[t][j]
              for j in range(2)] for i in range(3)]
        outs.append([sum(S[i][j] * q[t][j] for j in range(2)) for i in range(3)])
    f = lambda x: np.array(x, dtype=np.float64)
    qa = f(q)[:, None, :]
    ka = f(k)[:, None, :]
    va = f(v)[:, None, :]
    ga = np.log(f(alpha))[:, None]
    ba = f(beta)[:, None]
    s0 = f([[1, 0], [0, 2], [-1, 1]])[None, None]
    o, st = _call(mutant, qa, ka, va, ga, ba, s0, np.array([0, 2], np.int32), 1, 1, 2, 3)
    _close(o[:, 0, :], f([[float(x) for x in r] for r in outs]), tol=1e-14, what="o")
    _close(st[0, 0], f([[float(x) for x in r] for r in S]), tol=1e-14, what="state")


# --- I2: single token closed form ------------------------------------------------------------
def pin_single_token(mutant=0):
    """S_1 = a S_0 - a b (S_0 k) k^T + b v k^T and o_1 = S_1 q; from S_0 = 0,
    o_1 = b (k.q) v.  Non-symmetric S_0 and d_k != d_v pin the orientation."""
    r = _rng(3)
    d_k, d_v = 5, 7
    q = r.standard_normal((1, 1, d_k))
    k = r.standard_normal((1, 1, d_k))
    v = r.standard_normal((1, 1, d_v))
    g = np.array([[-0.3]])
    b = np.array([[0.6]])
    s0 = r.standard_normal((1, 1, d_v, d_k))
    a = np.exp(-0.3)
    S0 = s0[0, 0]
    kk, qq, vv = k[0, 0], q[0, 0], v[0, 0]
    S1 = a * S0 - a * 0.6 * np.outer(S0 @ kk, kk) + 0.6 * np.outer(vv, kk)
    cu = np.array([0, 1], np.int32)
    o, st = _call(mutant, q, k, v, g, b, s0, cu, 1, 1, d_k, d_v)
    _close(st[0, 0], S1, what="state")
    _close(o[0, 0], S1 @ qq, what="o")
    o, st = _call(mutant, q, k, v, g, b, None, cu, 1, 1, d_k, d_v)
    _close(o[0, 0], 0.6 * float(kk @ qq) * vv, what="o from zero state")


# --- I3 / I6: no write ------------------------------------------------------------------------
def pin_no_write_no_decay(mutant=0):
    """beta = 0 and alpha = 1 leave S unchanged and read o_t = S_0 q_t."""
    lengths = [9]
    q, k, v, g, beta, s0, cu = _rand_case(4, lengths, 1, 2, 6, 5)
    g[:] = 0.0
    beta[:] = 0.0
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, 1, 2, 6, 5, 1.3)
    _close(st, s0, what="state")
    for h in range(2):
        _close(o[:, h, :], (1.3 * q[:, 0, :]) @ s0[0, h].T, what="o")


def pin_pure_decay(mutant=0):
    """beta = 0: S_t = exp(sum_{s<=t} g_s) S_0 and o_t = S_t q_t."""
    lengths = [12]
    q, k, v, g, beta, s0, cu = _rand_case(5, lengths, 1, 1, 4, 6)
    beta[:] = 0.0
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, 1, 1, 4, 6)
    decay = np.exp(np.cumsum(g[:, 0]))
    _close(st[0, 0], decay[-1] * s0[0, 0], what="state")
    _close(o[:, 0, :], decay[:, None] * (q[:, 0, :] @ s0[0, 0].T), what="o")


# --- I4: reset ---------------------------------------------------------------------------------
def pin_reset(mutant=0):
    """alpha = 0 (g = -inf) forgets all history: S_t = b_t v_t k_t^T."""
    lengths = [6]
    q, k, v, g, beta, s0, cu = _rand_case(6, lengths, 1, 1, 4, 3)
    g[3] = -np.inf
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, 1, 1, 4, 3)
    S3 = beta[3, 0] * np.outer(v[3, 0], k[3, 0])
    _close(o[3, 0], S3 @ q[3, 0], what="o at reset")
    # the tail after the reset equals a fresh run from the reset state
    o2, st2 = _call(mutant, q[4:], k[4:], v[4:], g[4:], beta[4:], S3[None, None],
                    np.array([0, 2], np.int32), 1, 1, 4, 3)
    _close(o[4:], o2, what="o after reset")
    _close(st, st2, what="state after reset")


# --- I5: exact write ---------------------------------------------------------------------------
def pin_exact_write(mutant=0):
    """Unit-norm k, alpha = 1, beta = 1: the update stores v_t under key k_t,
    S_t k_t = v_t, whatever S_{t-1} was."""
    lengths = [7]
    q, k, v, g, beta, s0, cu = _rand_case(7, lengths, 1, 1, 8, 5)
    g[:] = 0.0
    beta[:] = 1.0
    for T in range(1, 8):
        _, st = _call(mutant, q[:T], k[:T], v[:T], g[:T], beta[:T], s0,
                      np.array([0, T], np.int32), 1, 1, 8, 5)
        _close(st[0, 0] @ k[T - 1, 0], v[T - 1, 0], what=f"S_t k_t at t={T}")


# --- I7: linearity -----------------------------------------------------------------------------
def pin_linearity(mutant=0):
    """(S_T, o) are jointly linear in (S_0, V) for fixed q, k, g, beta."""
    lengths = [10, 4]
    q, k, v, g, beta, s0, cu = _rand_case(8, lengths, 1, 2, 4, 3)
    r = _rng(9)
    v2 = r.standard_normal(v.shape)
    s2 = r.standard_normal(s0.shape)
    a, b = 0.7, -1.9
    o1, st1 = _call(mutant, q, k, v, g, beta, s0, cu, 1, 2, 4, 3)
    o2, st2 = _call(mutant, q, k, v2, g, beta, s2, cu, 1, 2, 4, 3)
    o3, st3 = _call(mutant, q, k, a * v + b * v2, g, beta, a * s0 + b * s2, cu, 1, 2, 4, 3)
    _close(o3, a * o1 + b * o2, tol=1e-11, what="o")
    _close(st3, a * st1 + b * st2, tol=1e-11, what="state")


# --- I8: chunked WY/UT evaluation --------------------------------------------------------------
def chunked_reference(q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, scale, C):
    """The chunked form, one chunk of C tokens at a time (last chunk partial):
    gamma = in-chunk cumsum of g, A_ri = b_r e^{gamma_r - gamma_i} k_r.k_i (i<r),
    T = (I + A)^{-1}, W = T diag(b Gamma) K, U~ = T diag(b) V, U = U~ - W S^T,
    O = diag(Gamma) Q S^T + (M o Q K^T) U, S' = Gamma_n S + U^T diag(e^{gamma_n - gamma}) K."""
    G = h_v // h_k
    N = len(cu) - 1
    o = np.full((q.shape[0], h_v, d_v), np.nan)
    st = np.zeros((N, h_v, d_v, d_k))
    for nn in range(N):
        for h in range(h_v):
            S = s0[nn, h].copy() if s0 is not None else np.zeros((d_v, d_k))
            for c0 in range(cu[nn], cu[nn + 1], C):
                c1 = min(c0 + C, cu[nn + 1])
                K = k[c0:c1, h // G]
                Q = scale * q[c0:c1, h // G]
                V = v[c0:c1, h]
                b = beta[c0:c1, h]
                gam = np.cumsum(g[c0:c1, h])
                Gam = np.exp(gam)
                diff = gam[:, None] - gam[None, :]
                lower = np.tril(np.ones((c1 - c0, c1 - c0)), -1)
                A = lower * b[:, None] * np.exp(np.where(lower > 0, diff, 0.0)) * (K @ K.T)
                Tm = np.linalg.inv(np.eye(c1 - c0) + A)
                W = Tm @ ((b * Gam)[:, None] * K)
                Ut = Tm @ (b[:, None] * V)
                U = Ut - W @ S.T
                M = np.tril(np.exp(np.where(np.tril(np.ones_like(diff)) > 0, diff, -np.inf)))
                o[c0:c1, h] = Gam[:, None] * (Q @ S.T) + (M * (Q @ K.T)) @ U
                S = Gam[-1] * S + (U * np.exp(gam[-1] - gam)[:, None]).T @ K
            st[nn, h] = S
    return o, st


def pin_chunked_equals_sequential(mutant=0):
    """The chunked WY/UT evaluation equals the oracle, for C = 64 and C = 16,
    with partial last chunks and d_k != d_v."""
    lengths = [150, 64, 1, 0, 65]
    h_k, h_v, d_k, d_v = 1, 2, 16, 24
    q, k, v, g, beta, s0, cu = _rand_case(10, lengths, h_k, h_v, d_k, d_v)
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, 0.9)
    for C in (64, 16):
        o_c, st_c = chunked_reference(q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v, 0.9, C)
        _close(o, o_c, tol=1e-11, what=f"o (C={C})")
        _close(st, st_c, tol=1e-11, what=f"state (C={C})")


# --- I9: row identity (the decode / scan arithmetic) -------------------------------------------
def pin_row_identity(mutant=0):
    """With s = S_{t-1} k and p = S_{t-1} q (read before the update):
    u = b (v - a s), S_t = a S_{t-1} + u k^T, o_t = a p + u (k.q)."""
    lengths = [20]
    h_k, h_v, d_k, d_v = 1, 1, 8, 6
    q, k, v, g, beta, s0, cu = _rand_case(13, lengths, h_k, h_v, d_k, d_v)
    S = s0[0, 0].copy()
    o_ref = np.zeros((20, d_v))
    for t in range(20):
        a, b = np.exp(g[t, 0]), beta[t, 0]
        kk, qq, vv = k[t, 0], q[t, 0], v[t, 0]
        s, p = S @ kk, S @ qq
        u = b * (vv - a * s)
        o_ref[t] = a * p + u * (kk @ qq)
        S = a * S + np.outer(u, kk)
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, h_k, h_v, d_k, d_v)
    _close(o[:, 0], o_ref, what="o")
    _close(st[0, 0], S, what="state")


# --- I10 / I11: split prefill and varlen packing -----------------------------------------------
def pin_split_prefill(mutant=0):
    """prefill(T1) -> state -> prefill(T2) equals prefill(T1 + T2)."""
    lengths = [50]
    q, k, v, g, beta, s0, cu = _rand_case(14, lengths, 1, 2, 4, 4)
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, 1, 2, 4, 4)
    T1 = 23
    oa, sa = _call(mutant, q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], s0,
                   np.array([0, T1], np.int32), 1, 2, 4, 4)
    ob, sb = _call(mutant, q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], sa,
                   np.array([0, 50 - T1], np.int32), 1, 2, 4, 4)
    _close(np.concatenate([oa, ob]), o, tol=1e-13, what="o")
    _close(sb, st, tol=1e-13, what="state")


def pin_varlen_packing(mutant=0):
    """A packed varlen call equals one call per sequence, bit for bit."""
    lengths = [3, 0, 9, 1]
    q, k, v, g, beta, s0, cu = _rand_case(15, lengths, 2, 2, 4, 3)
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, 2, 2, 4, 3)
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        on, sn = _call(mutant, q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], s0[n:n + 1],
                       np.array([0, b - a], np.int32), 2, 2, 4, 3)
        assert np.array_equal(on, o[a:b]), "o differs from the single-sequence call"
        assert np.array_equal(sn, st[n:n + 1]), "state differs from the single-sequence call"


def pin_rows_match_full(mutant=0):
    """The sampled-row entry point returns the same values as the full one."""
    lengths = [7, 12]
    q, k, v, g, beta, s0, cu = _rand_case(16, lengths, 2, 4, 8, 6)
    o, st = _call(mutant, q, k, v, g, beta, s0, cu, 2, 4, 8, 6)
    tasks = [(0, 3, 5), (1, 0, 0), (1, 2, 4)]
    res = oracle.rows(q, k, v, g, beta, cu, 2, 4, 8, 6, tasks, state_in=s0, mutant=mutant)
    for (n, h, i), (on, sn) in zip(tasks, res):
        assert np.array_equal(on, o[cu[n]:cu[n + 1], h, i])
        assert np.array_equal(sn, st[n, h, i])


def pin_qk_l2norm(mutant=0):
    """In-kernel L2 normalisation of q and k (per token and key head, eps 1e-6
    inside the square root): (a) the result does not change when any token's q
    or k is multiplied by a positive number; (b) on unit-norm q and k it equals
    the plain evaluation up to the eps (relative 1e-6); (c) o is still linear in
    `scale` (the scale acts after the normalisation)."""
    lengths = [9, 5]
    h_k, h_v, d_k, d_v = 1, 2, 6, 4
    q, k, v, g, beta, s0, cu = _rand_case(17, lengths, h_k, h_v, d_k, d_v)
    r = _rng(18)
    cq = np.exp(r.uniform(0, 3, (q.shape[0], h_k, 1)))  # norms >= 1: the eps moves < 1e-6
    ck = np.exp(r.uniform(0, 3, (k.shape[0], h_k, 1)))

    def run(qq, kk, scale=1.0, norm=True):
        return oracle.prefill(qq, kk, v, g, beta, cu, h_k, h_v, d_k, d_v, state_in=s0,
                              scale=scale, threads=4, mutant=mutant, qk_l2norm=norm)

    o_n, st_n = run(q, k)
    o_s, st_s = run(q * cq, k * ck)
    _close(o_s, o_n, 1e-5, "o under rescaled q, k")
    _close(st_s, st_n, 1e-5, "state under rescaled q, k")
    o_p, st_p = run(q, k, norm=False)  # q, k of _rand_case have unit norm
    _close(o_n, o_p, 1e-5, "o on unit-norm inputs")
    _close(st_n, st_p, 1e-5, "state on unit-norm inputs")
    o_h, _ = run(q * cq, k * ck, scale=0.5)
    _close(o_h, 0.5 * o_s, TOL, "o linear in scale")


ALL_PINS = [pin_brute_force, pin_brute_force_no_state, pin_exact_rational, pin_single_token,
            pin_no_write_no_decay, pin_pure_decay, pin_reset, pin_exact_write, pin_linearity,
            pin_chunked_equals_sequential, pin_row_identity, pin_split_prefill,
            pin_varlen_packing, pin_rows_match_full, pin_qk_l2norm]
