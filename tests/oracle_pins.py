"""Pins of the CPU oracle to facts outside itself: hand-computed fixtures, closed forms, Monte Carlo of the
white-noise distortion model, brute force on tiny inputs and library routines. Each pin is a plain function
so that tests/test_oracle_mutations.py can run it against an oracle with a planted mistake."""
import itertools
import math

import numpy as np

from conftest import read_golden
from oracle import kvtc_oracle as O
from transform_coded_kv_02_b300 import synth


def _floats(s):
    return np.array([float(x) for x in s.split()], dtype=np.float64)


def _ints(s):
    return np.array([int(x) for x in s.split()], dtype=np.int64)


def _params_from_row(widths, mu, sigma, r_words):
    d = len(widths)
    return O.TensorParams(T=np.eye(d), mu=mu, sigma=sigma, widths=widths, r_words=r_words)


# --- statistics -------------------------------------------------------------------------------------
def pin_statistics_closed_form():
    """mean/centred covariance/un-centred query moment of a 3-token example, solved by hand."""
    k = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 0.0]])
    v = np.array([[0.0, 0.0], [2.0, 2.0], [4.0, -2.0]])
    q = np.array([[1.0, 0.0], [0.0, 2.0]])
    mu_k, s_k, mu_v, s_v, m_q = O.calib_statistics(k, v, q)
    assert np.allclose(mu_k, [3.0, 2.0])
    assert np.allclose(s_k, np.array([[8.0, -4.0], [-4.0, 8.0]]) / 3.0)
    assert np.allclose(mu_v, [2.0, 0.0])
    assert np.allclose(s_v, np.array([[8.0, -4.0], [-4.0, 8.0]]) / 3.0)
    assert np.allclose(m_q, np.array([[0.5, 0.0], [0.0, 2.0]]))


# --- KLT ----------------------------------------------------------------------------------------------
def pin_klt_known_spectrum():
    """Sigma = Q diag(lam) Q^T with a known spectrum: eigenvalues, reconstruction, orthogonality, signs,
    and agreement with numpy.linalg.eigh on the same matrix."""
    rng = np.random.default_rng(7)
    d = 32
    Q = synth.random_orthogonal(d, rng)
    lam = 3.0 * 0.8 ** np.arange(d) + 0.01 * np.arange(d)[::-1]
    sigma = (Q * lam) @ Q.T
    l, u = O.klt(sigma)
    assert np.allclose(l, np.sort(lam)[::-1], rtol=1e-10, atol=1e-12)
    assert np.linalg.norm((u * l) @ u.T - sigma) <= 1e-10 * np.linalg.norm(sigma)
    assert np.linalg.norm(u.T @ u - np.eye(d)) <= 1e-12 * d
    for i in range(d):
        j = int(np.argmax(np.abs(u[:, i])))
        assert u[j, i] > 0
    # each column spans the same line as the generating basis vector of that eigenvalue
    order = np.argsort(-lam)
    for i in range(d):
        assert abs(abs(u[:, i] @ Q[:, order[i]]) - 1.0) < 1e-8
    le, ue = np.linalg.eigh(sigma)
    assert np.allclose(np.sort(le)[::-1], l, rtol=1e-12, atol=1e-13)


def pin_transform_preserves_inner_products():
    """An orthogonal transform keeps q.k: (Tq).(Tk) = q.k (fp64 eigenbasis to 1e-12; fp32 table to 1e-6)."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=64, steps=1)
    pk, _ = O.calibrate(L.calib_k[0], L.calib_v[0], L.calib_q[0], 2.75, 2.75)
    _, s_k, _, _, _ = O.calib_statistics(L.calib_k[0], L.calib_v[0], L.calib_q[0])
    _, u = O.klt(s_k)
    k = synth.as_float(L.k[0, 0])
    q = synth.as_float(L.q[0, 0])
    ref = q @ k.T
    rot = (q @ u) @ (k @ u).T
    assert np.max(np.abs(rot - ref)) <= 1e-12 * np.max(np.abs(ref)) * 128
    t = pk.T.astype(np.float64)
    rot32 = (q @ t.T) @ (k @ t.T).T
    assert np.max(np.abs(rot32 - ref)) <= 1e-6 * np.linalg.norm(q) * np.linalg.norm(k, axis=1).max()


def pin_sixteen_bits_preserve_attention():
    """With every channel at 16 bits the codec is transparent: |q.k - q.k^| <= 1e-3 |q||k| and the decode
    output is within 1e-3 relative L2 of exact attention on the raw keys and values."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=256, steps=1)
    pk, pv = O.calibrate(L.calib_k[0], L.calib_v[0], L.calib_q[0], 2.75, 2.75)
    d = pk.d
    k = synth.as_float(L.k[0, 0])
    v = synth.as_float(L.v[0, 0])
    q = synth.as_float(L.q[0, 0])
    pk16 = O.TensorParams(pk.T, pk.mu, pk.sigma, np.full(d, 16), r_words=1 + 16 * d // 32)
    pv16 = O.TensorParams(pv.T, pv.mu, pv.sigma, np.full(d, 16), r_words=1 + 16 * d // 32)
    rk = O.encode(k, pk16)
    rv = O.encode(v, pv16)
    kh = O.reconstruct(rk, pk16)
    err = np.abs(q @ kh.T - q @ k.T)
    bound = 1e-3 * np.linalg.norm(q, axis=1)[:, None] * np.linalg.norm(k, axis=1)[None, :]
    assert np.all(err <= bound)
    scale = 1.0 / math.sqrt(d)
    o = O.attend_decode(q, rk, rv, pk16, pv16, k.shape[0], scale)
    ex = O.attention(q, k, v, scale)
    assert np.linalg.norm(o - ex) <= 1e-3 * np.linalg.norm(ex)


# --- white-noise distortion model (AATC Key points, 1st bullet) ----------------------------------------
def pin_key_distortion_monte_carlo():
    """E[(q.e)^2] with e = U e^, e^_i ~ N(0, D_i) independent, q drawn from the calibration queries, equals
    sum_i w_i D_i with w_i = u_i^T M_Q u_i (Monte Carlo, within 4 standard errors)."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    ck, cv, cq = L.calib_k[0], L.calib_v[0], L.calib_q[0]
    _, s_k, _, _, m_q = O.calib_statistics(ck, cv, cq)
    lam, u = O.klt(s_k)
    d = u.shape[0]
    D = 1e-2 * (1.0 + (np.arange(d) % 5)) * (1.0 + 10.0 * (np.arange(d) < 8))
    w = O.key_weights(u, m_q)
    predicted = float(w @ D)
    rng = np.random.default_rng(11)
    n = 200_000
    qs = np.asarray(cq, np.float64)[rng.integers(0, cq.shape[0], n)]
    e = (rng.standard_normal((n, d)) * np.sqrt(D)) @ u.T
    x = np.einsum("nd,nd->n", qs, e) ** 2
    se = x.std() / math.sqrt(n)
    assert abs(x.mean() - predicted) <= 4 * se, (x.mean(), predicted, se)


def pin_value_distortion_monte_carlo():
    """E|sum_t p_t e_t|^2 with e_t = U e^_t white = sum_t p_t^2 sum_i D_i (independent of the basis)."""
    rng = np.random.default_rng(12)
    d, n_tok, trials = 128, 16, 20_000
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    _, _, _, s_v, _ = O.calib_statistics(L.calib_k[0], L.calib_v[0], L.calib_q[0])
    _, u = O.klt(s_v)
    D = 1e-2 * (1.0 + (np.arange(d) % 7))
    p = rng.random(n_tok)
    p /= p.sum()
    predicted = float((p ** 2).sum() * D.sum())
    e = (rng.standard_normal((trials, n_tok, d)) * np.sqrt(D)) @ u.T
    x = (np.einsum("t,ntd->nd", p, e) ** 2).sum(axis=1)
    se = x.std() / math.sqrt(trials)
    assert abs(x.mean() - predicted) <= 4 * se
    # the importances the oracle uses for values are the eigenvalues themselves
    assert np.allclose(O.value_importance(np.array([2.0, 1.0, 0.0])), [2.0, 1.0, 0.0])


def pin_additive_key_value_distortion():
    """Small independent white noise on keys and values: the output error energy of both together equals
    the key-only plus the value-only energy (cross terms vanish), to first order."""
    rng = np.random.default_rng(13)
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=32, steps=1)
    k = synth.as_float(L.k[0, 0])
    v = synth.as_float(L.v[0, 0])
    q = synth.as_float(L.q[0, 0])[:1]
    scale = 1.0 / math.sqrt(k.shape[1])
    o = O.attention(q, k, v, scale)
    trials = 4000
    ek = rng.standard_normal((trials,) + k.shape) * 1e-3
    ev = rng.standard_normal((trials,) + v.shape) * 1e-3
    both = np.array([np.sum((O.attention(q, k + ek[i], v + ev[i], scale) - o) ** 2) for i in range(trials)])
    konly = np.array([np.sum((O.attention(q, k + ek[i], v, scale) - o) ** 2) for i in range(trials)])
    vonly = np.array([np.sum((O.attention(q, k, v + ev[i], scale) - o) ** 2) for i in range(trials)])
    diff = both - konly - vonly
    assert abs(diff.mean()) <= 4 * diff.std() / math.sqrt(trials) + 1e-3 * both.mean()


def pin_exchange_rate_monte_carlo():
    """The weight of key against value distortion in the joint allocation. Many tokens, values independent of
    the attention weights, small white key noise in the key basis: the output error energy through exact
    attention, divided by sum_t p_t^2 sum_i w_i D_i (w_i = (u_i.q)^2 for the query used), equals
    rho = alpha^2 tr(Sigma_V) with alpha = 1/sqrt(d) to within the model's approximation (|v_t - o|^2 averages
    to tr(Sigma_V) + |mu_V - o|^2, a few per cent here)."""
    rng = np.random.default_rng(14)
    d, n = 128, 512
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=n, steps=1)
    k = synth.as_float(L.k[0, 0])
    v_basis = synth.random_orthogonal(d, rng)
    lam_v = 0.9 ** np.arange(d)
    v = (rng.standard_normal((n, d)) * np.sqrt(lam_v)) @ v_basis.T
    q = synth.as_float(L.q[0, 0])[:1]
    _, s_k, _, _, _ = O.calib_statistics(k, v, q)
    _, u = O.klt(s_k)
    scale = 1.0 / math.sqrt(d)
    o = O.attention(q, k, v, scale)
    logits = scale * (q @ k.T)[0]
    p = np.exp(logits - logits.max())
    p /= p.sum()
    D = 1e-8 * (1.0 + (np.arange(d) % 3))
    w = (u.T @ q[0]) ** 2
    trials = 3000
    x = np.empty(trials)
    for i in range(trials):
        e = (rng.standard_normal((n, d)) * np.sqrt(D)) @ u.T
        x[i] = np.sum((O.attention(q, k + e, v, scale) - o) ** 2)
    measured = x.mean() / (np.sum(p ** 2) * float(w @ D))
    rho = O.exchange_rate(lam_v, d)
    assert abs(measured / rho - 1) < 0.15, (measured, rho)


def pin_joint_split_by_enumeration():
    """The joint split against an enumeration written here: every word split of the record, each tensor at
    its own integer water-filling, the summed weighted white-noise distortion rho sum lambda_K 4^-b +
    sum lambda_V 4^-b; the chosen split attains the minimum. Limits: keys weighted a million times heavier
    take every word they can use, a million times lighter the fewest; equal importances and weights keep the
    even split (the tie rule)."""
    L = synth.make_layer(synth.WORKLOADS["llama_decode_32k"], T=16, steps=1)
    per_set = []
    for ck, cv, cq in list(zip(L.calib_k, L.calib_v, L.calib_q))[:3]:
        _, s_k, _, s_v, m_q = O.calib_statistics(ck, cv, cq)
        lk, uk = O.klt(s_k)
        lv, _ = O.klt(s_v)
        per_set.append((O.key_importance(lk, uk, m_q), O.value_importance(lv), O.exchange_rate(lv, 128)))
    r_total = 22

    def total(r):
        acc = 0.0
        for ik, iv, rho in per_set:
            bk = O.water_fill_integer(ik, 32 * r - 32, 8)
            bv = O.water_fill_integer(iv, 32 * (r_total - r) - 32, 8)
            acc += rho * float(np.sum(ik * 0.25 ** bk)) + float(np.sum(iv * 0.25 ** bv))
        return acc

    costs = {r: total(r) for r in range(1, r_total)}
    chosen = O.joint_split(per_set, r_total, 11, 8, 128)
    assert costs[chosen] <= min(costs.values()) * (1 + 1e-9)
    heavy = O.joint_split([(ik, iv, rho * 1e6) for ik, iv, rho in per_set], r_total, 11, 8, 128)
    light = O.joint_split([(ik, iv, rho * 1e-6) for ik, iv, rho in per_set], r_total, 11, 8, 128)
    assert heavy > 11 and light < 11 and heavy > light
    same = O.joint_split([(iv, iv, 1.0) for _, iv, _ in per_set], r_total, 11, 8, 128)
    assert same == 11


def pin_aware_basis_commuting():
    """When Sigma_K and M_Q share an eigenbasis (distinct eigenvalues), the KLT already minimises
    prod s_i w_i (Hadamard's inequality for each factor, equality only on the eigenbasis): no rotation is
    taken and the basis comes back unchanged."""
    rng = np.random.default_rng(15)
    d = 16
    q = synth.random_orthogonal(d, rng)
    A = (q * (0.8 ** np.arange(d))) @ q.T
    B = (q * (1.0 + rng.random(d))) @ q.T
    assert np.array_equal(O.attention_aware_key_basis(A, B, q), q)


def pin_aware_basis_two_channels():
    """d = 2: every sweep rotates by a multiple of the grid step pi/96 from the start (2-D rotations compose
    into one), so the result is the best of the 48 lattice angles of the start (enumerated here), and its angle
    lies within one lattice step of the true optimum's (a 20000-point enumeration; the objective has period
    pi/2 in the angle, which swaps the two channels)."""
    rng = np.random.default_rng(16)
    for _ in range(5):
        x = rng.standard_normal((2, 2))
        A = x @ x.T + 0.1 * np.eye(2)
        y = rng.standard_normal((2, 2))
        B = y @ y.T + 0.1 * np.eye(2)
        u0 = np.eye(2)
        u = O.attention_aware_key_basis(A, B, u0)

        def obj(phi):
            c, s = np.cos(phi), np.sin(phi)
            return O.basis_objective(np.array([[c, -s], [s, c]]), A + 1e-12 * np.trace(A) / 2 * np.eye(2),
                                     B + 1e-12 * np.trace(B) / 2 * np.eye(2))

        lattice = min(obj(-np.pi / 4 + k * np.pi / 96) for k in range(48))
        phis = np.linspace(-np.pi / 4, np.pi / 4, 20000, endpoint=False)
        best = phis[int(np.argmin([obj(p) for p in phis]))]
        got = O.basis_objective(u, A + 1e-12 * np.trace(A) / 2 * np.eye(2), B + 1e-12 * np.trace(B) / 2 * np.eye(2))
        assert abs(got - lattice) <= 1e-9, (got, lattice)
        phi = np.arctan2(u[1, 0], u[0, 0])
        gap = abs((phi - best + np.pi / 4) % (np.pi / 2) - np.pi / 4)
        assert gap <= np.pi / 96 + 1e-9, (phi, best)
        assert np.allclose(u.T @ u, np.eye(2), atol=1e-14)


def pin_aware_basis_bounds():
    """On the Llama-shaped layer's statistics the attention-aware basis is orthogonal, its objective lies above
    Hadamard's bound log det Sigma_K + log det M_Q (reached only when one basis diagonalises both) and at
    least 20 nats below the KLT's; the coefficient variances it reports are diag(U^T Sigma_K U)."""
    L = synth.make_layer(synth.WORKLOADS["llama_decode_32k"], T=16, steps=1)
    _, s_k, _, _, m_q = O.calib_statistics(L.calib_k[0], L.calib_v[0], L.calib_q[0])
    lam, u0 = O.klt(s_k)
    var, u = O.key_basis(s_k, m_q, True)
    assert np.abs(u.T @ u - np.eye(128)).max() < 1e-12
    bound = np.linalg.slogdet(s_k)[1] + np.linalg.slogdet(m_q)[1]
    got, klt_obj = O.basis_objective(u, s_k, m_q), O.basis_objective(u0, s_k, m_q)
    assert bound < got < klt_obj - 20.0, (bound, got, klt_obj)
    assert np.allclose(var, np.diag(u.T @ s_k @ u), rtol=1e-12)


def pin_whitened_key_transform():
    """The non-orthogonal key transform: T^-1 T = I; the generalised Parseval relation e^T M_Q e = |T e|^2 / c^2
    for every e (one constant c); uncorrelated coefficients, T Sigma_K T^T diagonal with the returned variances
    on the diagonal; every column of T^-1 of norm at most 1 (one of them exactly 1); and with M_Q = I the rows
    are the KLT's up to sign and one common scale."""
    L = synth.make_layer(synth.WORKLOADS["llama_decode_32k"], T=16, steps=1)
    _, s_k, _, _, m_q = O.calib_statistics(L.calib_k[0], L.calib_v[0], L.calib_q[0])
    var, T, T_inv = O.whitened_key_transform(s_k, m_q)
    d = T.shape[0]
    assert np.abs(T_inv @ T - np.eye(d)).max() < 1e-9
    m = m_q + np.eye(d) * (1e-12 * np.trace(m_q) / d)
    e = np.random.default_rng(17).standard_normal((64, d))
    ratio = np.einsum("nd,dk,nk->n", e, m, e) / np.sum((e @ T.T) ** 2, axis=1)
    assert np.std(ratio) <= 1e-9 * np.mean(ratio)
    c = T @ s_k @ T.T
    assert np.abs(c - np.diag(np.diag(c))).max() <= 1e-9 * np.abs(np.diag(c)).max()
    assert np.allclose(np.diag(c), var, rtol=1e-9, atol=1e-12 * var.max())
    norms = np.linalg.norm(T_inv, axis=0)
    assert norms.max() <= 1 + 1e-12 and abs(norms.max() - 1) < 1e-12
    _, T1, _ = O.whitened_key_transform(s_k, np.eye(d))
    _, u = O.klt(s_k)
    cos = np.abs(np.sum(T1 * u.T, axis=1)) / np.linalg.norm(T1, axis=1)
    assert np.all(cos > 1 - 1e-9)


# --- water-filling -----------------------------------------------------------------------------------
def pin_water_fill_golden():
    for lam, C, bmax, b_real, b_int in read_golden("water_fill_small.txt"):
        lam, C, bmax = _floats(lam), int(C), int(bmax)
        br, _ = O.water_fill_continuous(lam, C, bmax)
        assert np.allclose(br, _floats(b_real), atol=1e-9), (lam, br)
        assert np.array_equal(O.water_fill_integer(lam, C, bmax), _ints(b_int)), lam


def pin_water_fill_kkt():
    """Continuous solution of min sum_i lam_i 2^(-2 b_i) s.t. sum b_i = C, 0 <= b_i <= Bmax: active channels
    share one distortion theta, inactive ones have lam_i <= theta, capped ones lam_i 4^-Bmax >= theta;
    widths are monotone in lam."""
    rng = np.random.default_rng(3)
    for trial in range(20):
        d = int(rng.integers(4, 129))
        lam = np.exp(rng.normal(0, 3, d))
        C = int(rng.integers(1, 8 * d))
        bmax = 8
        b, theta = O.water_fill_continuous(lam, C, bmax)
        assert abs(b.sum() - C) < 1e-6
        assert np.all(b >= 0) and np.all(b <= bmax)
        if theta is None:
            continue
        act = (b > 1e-9) & (b < bmax - 1e-9)
        Dist = lam * 4.0 ** (-b)
        assert np.allclose(Dist[act], theta, rtol=1e-6)
        assert np.all(lam[b <= 1e-9] <= theta * (1 + 1e-6))
        assert np.all(lam[b >= bmax - 1e-9] * 4.0 ** (-bmax) >= theta * (1 - 1e-6))
        order = np.argsort(-lam)
        assert np.all(np.diff(b[order]) <= 1e-9)


def pin_water_fill_integer_properties():
    rng = np.random.default_rng(4)
    for trial in range(30):
        d = int(rng.integers(2, 129))
        lam = np.exp(rng.normal(0, 2, d))
        C = int(rng.integers(0, 8 * d + 1))
        bi = O.water_fill_integer(lam, C, 8)
        br, _ = O.water_fill_continuous(lam, C, 8)
        assert bi.sum() == min(C, 8 * d)
        assert np.all((bi >= 0) & (bi <= 8))
        assert np.all(np.abs(bi - br) < 1.0 + 1e-9)


def brute_force_allocation(lam, C, bmax):
    """Exhaustive integer allocation minimising sum lam_i 4^-b_i with sum b_i = C (tiny d only)."""
    best, arg = math.inf, None
    for b in itertools.product(range(bmax + 1), repeat=len(lam)):
        if sum(b) != C:
            continue
        val = sum(l * 4.0 ** (-x) for l, x in zip(lam, b))
        if val < best:
            best, arg = val, b
    return best, np.array(arg)


def pin_water_fill_vs_brute_force():
    """The rounding rule is within a small factor of the exhaustive integer optimum (reported gap)."""
    rng = np.random.default_rng(5)
    worst = 1.0
    for trial in range(25):
        d = int(rng.integers(2, 6))
        lam = np.exp(rng.normal(0, 2, d))
        C = int(rng.integers(1, 4 * d))
        best, _ = brute_force_allocation(lam, C, 6)
        b = O.water_fill_integer(lam, C, 6)
        val = float(np.sum(lam * 4.0 ** (-b)))
        assert val >= best * (1 - 1e-12)
        worst = max(worst, val / best)
    assert worst < 2.0, worst
    return worst


def pin_compression_accounting():
    for bits, rw, nbytes, ratio, page in read_golden("compression_ratios.txt"):
        r = O.record_words(float(bits), 128)
        assert r == int(rw)
        assert 4 * r == int(nbytes)
        assert abs(16 * 128 / (32 * r) - float(ratio)) < 1e-12
        if page != "none":
            assert abs(16 * 128 / (32 * r) - float(page)) / float(page) < 0.07


# --- quantiser / record ------------------------------------------------------------------------------
def pin_quantize_pack_golden():
    for name, widths, mu, sigma, y, rw, codes, words, yhat in read_golden("quantize_pack_small.txt"):
        p = _params_from_row(_ints(widths), _floats(mu), _floats(sigma), int(rw))
        y32 = _floats(y).astype(np.float32)[None, :]
        z, s, c = O.quantize(y32, p)
        assert np.array_equal(c[0], _ints(codes)), (name, c)
        rec = O.pack(z, s, c, p)
        assert [int(x) for x in rec[0]] == [int(w, 16) for w in words.split()], (name, [hex(x) for x in rec[0]])
        z2, s2, c2 = O.unpack(rec, p)
        assert np.array_equal(c2, c)
        yh = O.dequantize(z2, s2, c2, p)
        assert np.allclose(yh[0], _floats(yhat), atol=1e-12), (name, yh)


def _words_needed(widths, pairing="channels"):
    """Smallest record length whose layout holds the widths (first-fit), for test set-up."""
    lay = O.slot_layout if pairing == "channels" else O.token_slot_layout
    r = 2
    while lay(widths, r) is None:
        r += 1
    return r


def pin_pack_roundtrip():
    """Random widths 0..16 in any order, both layouts: pack then unpack returns the codes, z and s; every
    bit outside the channels' slots is zero; no two channels share a bit."""
    rng = np.random.default_rng(6)
    for trial in range(40):
        pairing = ("channels", "tokens")[trial % 2]
        d = int(rng.integers(1, 130))
        widths = rng.integers(0, 17, d)
        r_words = _words_needed(widths, pairing) + int(rng.integers(0, 2))
        p = O.TensorParams(T=np.eye(d), mu=np.zeros(d), sigma=np.ones(d), widths=widths, r_words=r_words,
                           pairing=pairing)
        n = 7
        codes = np.stack([rng.integers(0, 2 ** int(b), n) if b > 0 else np.zeros(n, np.int64)
                          for b in widths], axis=1)
        z = rng.normal(size=n).astype(np.float16)
        s = np.abs(rng.normal(size=n)).astype(np.float16)
        rec = O.pack(z, s, codes, p)
        assert rec.shape == ((n + p.tokens_per_record - 1) // p.tokens_per_record, p.record_len)
        z2, s2, c2 = O.unpack(rec, p)
        assert np.array_equal(c2[:n], codes)
        assert np.array_equal(z2[:n].view(np.uint16), z.view(np.uint16))
        assert np.array_equal(s2[:n].view(np.uint16), s.view(np.uint16))
        owned = np.zeros(p.record_len, np.uint64)
        for t in range(p.tokens_per_record):
            owned[t] = np.uint64(0xFFFFFFFF)
            for j in range(d):
                b = int(widths[j])
                if b == 0:
                    continue
                if pairing == "channels":
                    k = j // 2
                    w, r0, hi = 1 + int(p.slot_word[k]), int(p.slot_pos[k]), j % 2
                else:
                    w, r0, hi = 2 + int(p.slot_word[j]), int(p.slot_pos[j]), t
                assert r0 + b <= 16
                m = np.uint64(((1 << b) - 1) << (r0 + 16 * hi))
                assert (owned[w] & m) == 0            # no two channels share a bit
                owned[w] |= m
        for w in range(p.tokens_per_record, p.record_len):
            assert np.all((rec[:, w].astype(np.uint64) & ~owned[w] & np.uint64(0xFFFFFFFF)) == 0)


def pin_token_pack_golden():
    """Hand-computed value records in the token-pair layout (tests/golden/quantize_pack_token_pairs.txt)."""
    for name, widths, mu, sigma, ys, rw, codes, recs, yhats in read_golden("quantize_pack_token_pairs.txt"):
        w = _ints(widths)
        p = O.TensorParams(T=np.eye(len(w)), mu=_floats(mu), sigma=_floats(sigma), widths=w, r_words=int(rw),
                           pairing="tokens")
        y32 = np.array([_floats(r) for r in ys.split(";")], np.float32)
        z, s_, c = O.quantize(y32, p)
        assert np.array_equal(c, np.array([_ints(r) for r in codes.split(";")])), (name, c)
        rec = O.pack(z, s_, c, p)
        want = [[int(x, 16) for x in r.split()] for r in recs.split(";")]
        assert rec.astype(np.int64).tolist() == want, (name, [[hex(x) for x in r] for r in rec])
        z2, s2, c2 = O.unpack(rec, p)
        n = y32.shape[0]
        assert np.array_equal(c2[:n], c)
        yh = O.dequantize(z2[:n], s2[:n], c2[:n], p)
        assert np.allclose(yh, np.array([_floats(r) for r in yhats.split(";")]), atol=1e-12), (name, yh)


def pin_token_layout_fit_golden():
    """Hand-solved fits of value widths to the token-pair layout (tests/golden/layout_fit_token_pairs.txt)."""
    for widths, imp, rw, fitted, words, pos in read_golden("layout_fit_token_pairs.txt"):
        f = O.fit_token_layout(_ints(widths), _floats(imp), int(rw))
        assert f.tolist() == _ints(fitted).tolist(), (widths, f)
        lay = O.token_slot_layout(f, int(rw))
        assert lay is not None
        assert lay[0].tolist() == _ints(words).tolist() and lay[1].tolist() == _ints(pos).tolist(), lay


def pin_layout_fit_golden():
    """Hand-solved fits of water-filling widths to the pair layout (tests/golden/layout_fit_small.txt)."""
    for widths, imp, rw, fitted, words, pos in read_golden("layout_fit_small.txt"):
        f = O.fit_layout(_ints(widths), _floats(imp), int(rw))
        assert f.tolist() == _ints(fitted).tolist(), (widths, f)
        lay = O.slot_layout(f, int(rw))
        assert lay is not None
        assert lay[0].tolist() == _ints(words).tolist() and lay[1].tolist() == _ints(pos).tolist(), lay


def pin_layout_fit_properties():
    """On the workloads' calibrations (their own calibration sizes; the batched workload calibrates on a
    sequence's first 1024 tokens): the fitted widths fit the record (key: channel pairs sharing one width no
    larger than the pair's wider water-filling width; value: each channel no wider than its water-filling
    width), and the white-noise distortion sum_j lambda_j 4^-b_j grows by at most 2% over the unconstrained
    integer allocation."""
    worst = 1.0
    for name, bits in (("tiny", 2.75), ("llama_long_128k", 1.33), ("qwen_batched_8k", 2.0),
                       ("qwen_batched_8k", 3.0), ("qwen_batched_8k", 4.0)):
        L = synth.make_layer(synth.WORKLOADS[name], T=1024, B=1, steps=1)
        mu_k, s_k, mu_v, s_v, m_q = O.calib_statistics(L.calib_k[0], L.calib_v[0], L.calib_q[0])
        for lam_u, imp_fn, pairing in ((O.klt(s_k), lambda l, u: O.key_importance(l, u, m_q), "channels"),
                                       (O.klt(s_v), lambda l, u: O.value_importance(l), "tokens")):
            lam, u = lam_u
            imp = imp_fn(lam, u)
            r = O.record_words(bits, 128)
            b = O.water_fill_integer(imp, O.code_bits(r), 8)
            order = O.storage_order(b, imp)
            b, imp = b[order], np.asarray(imp)[order]
            if pairing == "channels":
                f = O.fit_layout(b, imp, r)
                assert O.slot_layout(f, r) is not None
                assert np.array_equal(f[0::2], f[1::2])
                assert np.all(f[0::2] <= np.maximum(b[0::2], b[1::2]))
            else:
                f = O.fit_token_layout(b, imp, r)
                assert O.token_slot_layout(f, r) is not None
                assert np.all(f <= b)
            assert f.sum() <= O.code_bits(r)
            d0 = float(np.sum(imp * 4.0 ** (-b.astype(np.float64))))
            d1 = float(np.sum(imp * 4.0 ** (-f.astype(np.float64))))
            worst = max(worst, d1 / d0)
    assert worst <= 1.02, worst
    return worst


def pin_quantizer_error_bound():
    """Codes lie in [0, 2^b - 1]; normalised reconstruction error <= half a bin (s 2^-b / 2) plus fp32
    rounding for every value inside [z, z + s]."""
    rng = np.random.default_rng(8)
    d = 64
    widths = np.concatenate([np.full(8, 8), np.full(16, 4), np.full(20, 2), np.full(12, 1), np.zeros(8, int)])
    mu = rng.normal(size=d)
    sigma = np.exp(rng.normal(size=d))
    p = _params_from_row(widths, mu, sigma, r_words=1 + int(np.ceil(widths.sum() / 32)))
    y = (rng.normal(size=(500, d)) * sigma + mu).astype(np.float32)
    z, s, c = O.quantize(y, p)
    nz = widths > 0
    assert np.all(c[:, nz] >= 0) and np.all(c[:, nz] <= (2 ** widths[nz]) - 1)
    assert np.all(c[:, ~nz] == 0)
    yp = ((y.astype(np.float64) - p.mu.astype(np.float64)) * p.inv_sigma.astype(np.float64))[:, nz]
    yh = O.dequantize(z, s, c, p)
    yhp = ((yh - p.mu.astype(np.float64)) / p.sigma.astype(np.float64))[:, nz]
    zf = z.astype(np.float64)[:, None]
    sf = s.astype(np.float64)[:, None]
    inside = (yp >= zf) & (yp <= zf + sf)
    half_bin = sf * 2.0 ** (-widths[nz].astype(np.float64)) / 2
    err = np.abs(yp - yhp)
    assert np.all(err[inside] <= (half_bin + 1e-5 * (np.abs(yp) + 1))[inside])


def pin_zero_bit_channels_are_the_mean():
    rng = np.random.default_rng(9)
    d = 16
    widths = np.array([4] * 6 + [0] * 10)
    mu = rng.normal(size=d).astype(np.float32)
    p = _params_from_row(widths, mu, np.ones(d), r_words=2)
    y = rng.normal(size=(20, d)).astype(np.float32)
    yh = O.dequantize(*O.unpack(O.pack(*O.quantize(y, p), p), p), p)
    assert np.array_equal(yh[:, 6:], np.broadcast_to(mu[6:].astype(np.float64), (20, 10)))


def half_rn_sat_bits(x32):
    """Independent fp32 -> saturated fp16 conversion written from the IEEE 754 binary16 definition on the bit
    patterns, with integer arithmetic only: the value of |x| counted in units of the binary16 quantum at its
    exponent (2^(e - 10) for normal results, 2^-24 for subnormal ones), rounded to the nearest integer with ties
    to even, the sign put back; magnitudes >= 65504 give +-65504 (saturation instead of infinity). Returns the
    values as float64."""
    u = np.asarray(x32, np.float32).view(np.uint32).astype(np.int64)
    sign = np.where(u >> 31, -1.0, 1.0)
    ex = (u >> 23) & 0xFF
    frac = u & 0x7FFFFF
    sig = np.where(ex > 0, frac | (1 << 23), frac)            # significand, value = sig 2^(e32 - 150)
    e_unb = np.where(ex > 0, ex - 127, -126)                  # exponent of the leading bit position 23
    lead = np.where(sig > 0, np.floor(np.log2(np.maximum(sig, 1))).astype(np.int64), 0)
    e_val = e_unb + lead - 23                                 # floor(log2 |x|)
    q_exp = np.maximum(e_val, -14) - 10                       # binary16 quantum exponent at that magnitude
    shift = q_exp - (np.where(ex > 0, ex, 1) - 150)           # sig 2^(e32 - 150) / 2^q_exp = sig >> shift
    out = np.empty(u.shape, np.float64)
    for i in range(u.size):
        s_i, sh, sg = int(shift.flat[i]), int(shift.flat[i]), int(sig.flat[i])
        if sh <= 0:
            n = sg << (-sh)
        elif sh >= 62:
            n = 0
        else:
            n, rem, half = sg >> sh, sg & ((1 << sh) - 1), 1 << (sh - 1)
            if rem > half or (rem == half and n & 1):
                n += 1
        mag = float(n) * 2.0 ** int(q_exp.flat[i])
        out.flat[i] = sign.flat[i] * min(mag, 65504.0)
    return out


def pin_half_conversion():
    """fp32 -> fp16 round-to-nearest-even with saturation, per IEEE 754 binary16: hand-picked values; then the
    oracle's converter against half_rn_sat_bits (written from the binary16 definition, integer arithmetic on the
    bit patterns) on every one of the 2^16 binary16 values, every midpoint between neighbouring finite binary16
    values (the ties) with the fp32 values one ulp either side of it, and a sweep of 2^17 fp32 bit patterns
    spread over the whole range."""
    cases = [(1.0 + 2.0 ** -11, 1.0), (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9), (65519.0, 65504.0),
             (65520.0, 65504.0), (1e9, 65504.0), (-1e9, -65504.0), (2.0 ** -25, 0.0),
             (3 * 2.0 ** -26, 2.0 ** -24), (0.1, 0.0999755859375)]
    for x, want in cases:
        assert float(O.half_rn_sat(np.float32(x))) == want, (x, want)
        assert float(half_rn_sat_bits(np.float32(x))) == want, (x, want)
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = h[np.isfinite(h)].astype(np.float64)
    allh = fin.astype(np.float32)                              # exact in fp32
    srt = np.unique(fin)
    mids = ((srt[1:] + srt[:-1]) / 2).astype(np.float32)       # exact in fp32 (one more bit than binary16)
    assert np.array_equal((srt[1:] + srt[:-1]) / 2, mids.astype(np.float64))
    mb = mids.view(np.uint32)
    near = np.concatenate([mb - 1, mb + 1]).view(np.float32)
    sweep = (np.arange(1 << 17, dtype=np.uint64) * 32749 % (1 << 32)).astype(np.uint32).view(np.float32)
    sweep = sweep[np.isfinite(sweep)]
    for xs in (allh, mids, near, sweep):
        want = half_rn_sat_bits(xs)
        got = O.half_rn_sat(xs).astype(np.float64)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (xs[bad[:5]], got[bad[:5]], want[bad[:5]])


# --- decode ------------------------------------------------------------------------------------------
def brute_force_decode(q, rec_k, rec_v, pk, pv, seq_len, scale):
    """Explicit per-element loops: unpack bits, dequantise, rotate back, softmax, weighted sum. Key records
    hold one token with channel pairs sharing slots; value records hold two tokens, one slot per channel."""
    def rec_to_vec(rec, p, t_in=0):
        d = p.d
        two = p.pairing == "tokens"
        word0 = int(rec[t_in])
        z = float(np.array([word0 & 0xFFFF], np.uint16).view(np.float16)[0])
        s = float(np.array([word0 >> 16], np.uint16).view(np.float16)[0])
        first_code = 2 if two else 1
        free = [16] * (len(rec) - first_code)
        where = {}
        if two:      # one slot per channel, first-fit by hand
            for j in range(d):
                b = int(p.widths[j])
                if b == 0:
                    continue
                u = next(i for i in range(len(free)) if free[i] >= b)
                where[j] = (u, 16 - free[u], 16 * t_in)
                free[u] -= b
        else:        # pair k = channels (2k, 2k+1), slot width = the wider one
            for k in range(d // 2):
                sw = max(int(p.widths[2 * k]), int(p.widths[2 * k + 1]))
                if sw == 0:
                    continue
                u = next(i for i in range(len(free)) if free[i] >= sw)
                where[2 * k] = (u, 16 - free[u], 0)
                where[2 * k + 1] = (u, 16 - free[u], 16)
                free[u] -= sw
        y = []
        for j in range(d):
            b = int(p.widths[j])
            if b == 0:
                y.append(float(p.mu[j]))
                continue
            u, r, half = where[j]
            c = (int(rec[first_code + u]) >> (r + half)) & ((1 << b) - 1)
            y.append(float(p.mu[j]) + float(p.sigma[j]) * (z + (c + 0.5) * s / (2 ** b)))
        x = []
        for col in range(d):
            acc = 0.0
            for row in range(d):
                acc += float(p.T[row, col]) * y[row]
            x.append(acc)
        return x

    def token_vec(recs, p, t):
        if p.pairing == "tokens":
            return rec_to_vec(recs[t // 2], p, t % 2)
        return rec_to_vec(recs[t], p)

    ks = [token_vec(rec_k, pk, t) for t in range(seq_len)]
    vs = [token_vec(rec_v, pv, t) for t in range(seq_len)]
    out = []
    for h in range(q.shape[0]):
        logits = [scale * sum(float(q[h, i]) * ks[t][i] for i in range(len(ks[t]))) for t in range(seq_len)]
        mx = max(logits)
        e = [math.exp(l - mx) for l in logits]
        tot = sum(e)
        out.append([sum(e[t] / tot * vs[t][i] for t in range(seq_len)) for i in range(pk.d)])
    return np.array(out)


def pin_decode_brute_force():
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=8, steps=1)
    pk, pv = O.calibrate(L.calib_k[0], L.calib_v[0], L.calib_q[0], 2.75, 2.75)
    k = synth.as_float(L.k[0, 0])
    v = synth.as_float(L.v[0, 0])
    q = synth.as_float(L.q[0, 0])
    rk, rv = O.encode(k, pk), O.encode(v, pv)
    scale = 1.0 / math.sqrt(128)
    for T in (1, 3, 8):
        o = O.attend_decode(q, rk, rv, pk, pv, T, scale)
        ref = brute_force_decode(q, rk, rv, pk, pv, T, scale)
        assert np.allclose(o, ref, rtol=1e-11, atol=1e-11), T


def pin_storage_order():
    """Storage order sorts channels by width (descending), then importance (descending), then eigen-index. The
    value channels of a calibrated set lose no bits to the record layout here, so along storage order their
    widths do not increase, and within each run of equal widths their importances (the variances) do not
    increase either."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    for bits in (1.33, 2.75, 4.0):
        pk, pv = O.calibrate(L.calib_k[0], L.calib_v[0], L.calib_q[0], bits, bits)
        w = np.asarray(pv.widths)
        lam = np.asarray(pv.importance, np.float64)
        assert np.all(np.diff(w) <= 0), bits
        same = np.diff(w) == 0
        assert same.sum() > 10 and np.all(np.diff(lam)[same] <= 0), bits


def pin_calibrate_structure():
    """Calibrated sets: orthogonal T; both channels of a pair share one width; the widths fit the record's
    pair layout and use at most the budget and at least all but one code word of it; mu = T mu_raw,
    sigma^2 = eigenvalues."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=16, steps=1)
    ck, cv, cq = L.calib_k[0], L.calib_v[0], L.calib_q[0]
    pk, pv = O.calibrate(ck, cv, cq, 2.75, 2.75)
    assert pk.pairing == "channels" and pv.pairing == "tokens"
    for p, x in ((pk, ck), (pv, cv)):
        t = p.T.astype(np.float64)
        assert np.linalg.norm(t @ t.T - np.eye(128)) < 1e-5
        if p.pairing == "channels":
            assert np.array_equal(p.widths[0::2], p.widths[1::2])
            assert O.slot_layout(p.widths, 11) is not None
        else:
            assert O.token_slot_layout(p.widths, 11) is not None
        assert O.code_bits(11) - 32 < p.widths.sum() <= O.code_bits(11)
        assert np.allclose(p.mu, t @ np.asarray(x, np.float64).mean(0), atol=1e-5)
        assert np.allclose(p.sigma.astype(np.float64) ** 2, p.eigvals, rtol=1e-5)

# --- rotary embedding of the query ------------------------------------------------------------------
def pin_rotary_embedding():
    """Closed forms where the frequency is exact (channel 0 turns by one radian per position; channel d/4 by
    base^(-1/2), 0.01 rad for base 10000), with cos and sin of 1 and 3 rad as printed in tables; then what any
    rotation by position must satisfy: position 0 is the identity, norms are kept, two embeddings compose, and
    an embedded query and key meet through their position difference only."""
    d = 128
    e = np.eye(d)
    cos1, sin1 = 0.5403023058681398, 0.8414709848078965
    cos3, sin3 = -0.9899924966004454, 0.1411200080598672
    want = np.zeros(d)
    want[0], want[64] = cos3, sin3
    assert np.allclose(O.rotary_embed(e[0], 3, 10000.0), want, rtol=0, atol=1e-15)
    want = np.zeros(d)
    want[0], want[64] = -sin3, cos3
    assert np.allclose(O.rotary_embed(e[64], 3, 10000.0), want, rtol=0, atol=1e-15)
    want = np.zeros(d)
    want[32], want[96] = cos1, sin1
    assert np.allclose(O.rotary_embed(e[32], 100, 10000.0), want, rtol=0, atol=1e-14)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, d))
    k = rng.standard_normal(d)
    assert np.array_equal(O.rotary_embed(x, 0, 500000.0), x)
    for pos in (1, 77, 131071):
        y = O.rotary_embed(x, pos, 500000.0)
        assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    assert np.allclose(O.rotary_embed(O.rotary_embed(x, 1000, 5e5), 234, 5e5), O.rotary_embed(x, 1234, 5e5),
                       atol=1e-12)
    a1 = O.rotary_embed(x, 5000, 5e5) @ O.rotary_embed(k, 4000, 5e5)
    a2 = O.rotary_embed(x, 1000, 5e5) @ k
    assert np.allclose(a1, a2, atol=1e-10)


# --- token-axis allocation --------------------------------------------------------------------------
def pin_token_weights():
    """Closed form: identical keys spread every query evenly, lambda_t = n_q / T^2. Bounds: each query's
    probabilities sum to 1, so n_q / T <= sum_t lambda_t <= n_q. Meaning (Monte Carlo): white noise of variance
    s2 added to token t's value alone moves the outputs by sum_q |delta o_q|^2 = s2 d lambda_t on average."""
    rng = np.random.default_rng(21)
    d, T, nq = 16, 9, 5
    q = rng.standard_normal((nq, d))
    k1 = np.tile(rng.standard_normal(d), (T, 1))
    assert np.allclose(O.token_weights(q, k1, 0.5), nq / T ** 2, rtol=1e-12)
    k = rng.standard_normal((T, d))
    lam = O.token_weights(q, k, 0.7)
    assert nq / T - 1e-12 <= lam.sum() <= nq + 1e-12
    v = rng.standard_normal((T, d))
    base = O.attention(q, k, v, 0.7)
    s2, n = 0.01, 4000
    for t in (0, 4):
        acc = 0.0
        for _ in range(n):
            vp = v.copy()
            vp[t] += np.sqrt(s2) * rng.standard_normal(d)
            acc += np.sum((O.attention(q, k, vp, 0.7) - base) ** 2)
        assert abs(acc / n - s2 * d * lam[t]) <= 0.08 * s2 * d * lam[t], (t, acc / n, s2 * d * lam[t])


def pin_token_keep():
    """Brute force on small token counts: the kept set is the subset of `keep` tokens with the largest total
    weight, ties to the lexicographically earliest; and with one tier the library's reverse water-filling over
    the token axis (widths 0 or 1, `keep` bits in all) keeps the same tokens."""
    rng = np.random.default_rng(22)
    for T in (1, 5, 8):
        lam = rng.choice([1.0, 2.0, 2.0, 5.0, 9.0], size=T)  # repeated values: ties; integer sums are exact
        for keep in range(T + 1):
            best = None
            for sub in itertools.combinations(range(T), keep):
                key = (-sum(lam[list(sub)]), sub)
                if best is None or key < best:
                    best = key
            got = O.token_keep(lam, keep)
            assert tuple(got) == best[1], (T, keep, got, best)
    for _ in range(20):
        lam = rng.gamma(0.5, 1.0, size=40)
        keep = int(rng.integers(1, 40))
        w = O.water_fill_integer(lam, keep, 1)
        assert tuple(np.nonzero(w)[0]) == tuple(O.token_keep(lam, keep))


def pin_compact():
    """Records are per token (keys) or per token half (values), so compacting encoded records equals encoding
    the kept tokens; and decoding the compacted records is attention over the kept tokens alone."""
    L = synth.make_layer(synth.WORKLOADS["tiny"], T=40, steps=1)
    pk, pv = O.calibrate(L.calib_k[0], L.calib_v[0], L.calib_q[0], 2.75, 2.75)
    k = synth.as_float(L.k[0, 0])
    v = synth.as_float(L.v[0, 0])
    for idx in ([0, 3, 4, 9, 20, 39], [1, 2, 5], [7], list(range(0, 40, 3))):
        idx = np.array(idx)
        assert np.array_equal(O.compact(O.encode(k, pk), pk, idx), O.encode(k[idx], pk))
        assert np.array_equal(O.compact(O.encode(v, pv), pv, idx), O.encode(v[idx], pv))
    q = synth.as_float(L.q[0, 0])
    idx = np.array([2, 3, 11, 30])
    rk, rv = O.compact(O.encode(k, pk), pk, idx), O.compact(O.encode(v, pv), pv, idx)
    o = O.attend_decode(q, rk, rv, pk, pv, len(idx), 0.1)
    ref = O.attention(q, O.reconstruct(O.encode(k[idx], pk), pk), O.reconstruct(O.encode(v[idx], pv), pv)[:4], 0.1)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
