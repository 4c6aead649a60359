"""CPU oracle for attention-aware transform coding (AATC) of the KV cache.

TEST INFRASTRUCTURE. Only the tests, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg
import this module. The product library (the C-ABI shared library and its Python binding) neither imports
nor calls it, and this module imports nothing from the product.

What it computes, in the pages' order, written plainly (numpy; fp64 for all statistics, transforms and
attention; IEEE fp32 for the quantiser, whose op sequence is part of the record format):

 1. Calibration statistics per (layer, KV head) [AATC "KV Cache Compression Through the Lens of Transform
    Coding", Key points 2nd bullet: bits are allocated "over a calibration set"; NOVA-KV (third abstract on
    the "SPHERICAL KV" page): transforms "from calibration statistics"]: key/value means, centred
    covariances (divide by n), and the un-centred query second moment M_Q pooled over the g query heads
    that read the KV head.
 2. Transform coding with a KLT [SPECTRA abstract: rotate the cache "into a coordinate system computed
    from its own statistics, removing these correlations"]: Sigma = U Lambda U^T, eigenvalues descending,
    each eigenvector's largest-magnitude component made positive (lowest index on ties).
 3. Attention-aware channel importances [AATC Key points 1st bullet: under white noise the attention
    distortion is additive over keys and values and factors over tokens and channels]:
      keys   lambda_i = sigma_i^2 * w_i,  w_i = u_i^T M_Q u_i  (E[(q.e)^2] = sum_i w_i D_i),
      values lambda_i = sigma_i^2         (E|sum_t p_t e_t|^2 = sum_t p_t^2 sum_i D_i).
 4. Reverse water-filling [AATC Full text; RDKV (first abstract on the "SPHERICAL KV" page): widths "from
    full precision down to zero bits guided by reverse water-filling"]:
      b_i(theta) = min(B_max, max(0, 1/2 log2(lambda_i / theta))), theta by bisection so that
      sum_i b_i = C = 32 R_w - 32, then integer rounding (floors, then one bit each to the largest
      fractional parts compared at 1e-9 resolution; ties to larger lambda, then lower index; never
      above B_max).
 5. Storage order: channels sorted by (width desc, lambda desc, eigen index asc); T = rows of U^T in
    that order; mu_j = rotated mean, sigma_j = sqrt(lambda_j) (fp32), inv_sigma_j = fp32(1/sigma_j).
    Fixed-width layout [NOVA-KV: the allocation has to meet a fixed-width layout]: storage channels
    (2k, 2k+1) form pair k and share one slot, at the same bit position in the low and the high 16-bit
    half of one code word; a pair's slot is as wide as its wider channel. The narrower channel of a pair
    is raised to the slot width (the layout reserves those bits anyway); slots are placed first-fit in
    pair order (lowest code word with room, lowest free bit); while a pair finds no room, the pair with
    the smallest distortion cost 3 (lambda_2k + lambda_2k+1) 4^-w of losing one bit (compared through
    log2 at 1e-9 resolution; ties: the later pair) loses one bit and the placement restarts. That is the
    key layout ("channel pairs"). Values use a "token pairs" layout instead, because decode contracts
    values over tokens: a record holds two consecutive tokens, and each channel j has one slot at the same
    bit of the low half (earlier token) and the high half (later token) of one code word; slots are
    placed first-fit in storage order, and while a channel finds no room the channel with the smallest
    cost 3 lambda_j 4^-b_j (same comparison, ties to the later channel) loses one bit.
 6. Per-token quantiser (fixed fp32 op sequence, no fused multiply-add):
      y'_j = (y_j - mu_j) * inv_sigma_j                 (channels with b_j > 0)
      m, M = min/max of y'_j over b_j > 0;  z = fp16(m), s = fp16(M - z) (round-to-nearest-even, saturated)
      c_j = clamp(floor(((y'_j - z) / s) * 2^b_j), 0, 2^b_j - 1);  all codes 0 when s == 0.
 7. Fixed-width records [NOVA-KV: "a fixed per-token bit count"]. Keys: R_w 32-bit words per token;
    word 0 holds z (bits 0-15) and s (bits 16-31); pair k's codes sit in code word 1 + u_k: channel 2k
    at bits [r_k, r_k + b_2k), channel 2k+1 at bits [16 + r_k, 16 + r_k + b_2k+1). Values: 2 R_w words
    per pair of tokens (2p, 2p+1); words 0 and 1 hold their z/s words, channel j's codes sit in code word
    2 + u_j at bits [r_j, r_j + b_j) (token 2p) and [16 + r_j, 16 + r_j + b_j) (token 2p+1). The budget per
    token is the same. Unused bits are 0.
 8. Decode attention over the records: y^_j = mu_j + sigma_j (z + (c_j + 1/2) s 2^-b_j) for b_j > 0, else
    mu_j; k^ = T^T y^ (and v^); o_h = softmax_t(alpha q_h . k^_t) v^ over t < seq_len, all in fp64.
10. Token-axis allocation [RDKV, first abstract on the "SPHERICAL KV" page: per-token widths "from full precision
    down to zero bits guided by reverse water-filling, applied once after the prefilling stage", each token's
    weight taken from the distortion its compression induces on attention]: a token's weight is
    lambda_t = sum_q p_qt^2 over observation queries q (a white error e on token t's value moves query q's output
    by p_qt e); with one tier above zero bits (the token keeps its record, or is evicted), reverse water-filling
    keeps the `keep` tokens of largest weight (ties: the earlier token); the kept records are compacted, in
    order, into a sequence of their own.
 9. Serving layout [SPECTRA abstract: "longer contexts and larger batches"]: the query may arrive without its
    rotary position embedding, which the decode then applies first: pair (i, i + d/2) of q rotated by the angle
    pos * base^(-2i/d) (the half-split convention of the Llama models, no frequency rescaling), in fp64. Paged
    and multi-layer caches change where records live, not what they hold: the tests gather a sequence's
    records page by page and decode them with 8.

Where the pages are silent this module takes the plainest reading the rest of them supports: the same
bits/element for keys and values, an orthogonal key KLT with the query weighting in the allocation, a
mid-rise quantiser with bin centres, fp16 round-to-nearest-even, a budget that counts the scale/zero word, and
alpha = 1/sqrt(d).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64
HALF_MAX = 65504.0


# ----------------------------------------------------------------------------------------------------
# 1. statistics
# ----------------------------------------------------------------------------------------------------
def calib_statistics(k, v, q):
    """Means and centred covariances (divide by n) of calibration keys/values; un-centred second moment
    of the pooled calibration queries (all g heads' vectors stacked in q)."""
    k = np.asarray(k, F64)
    v = np.asarray(v, F64)
    q = np.asarray(q, F64)
    mu_k = k.mean(axis=0)
    mu_v = v.mean(axis=0)
    ck = k - mu_k
    cv = v - mu_v
    sigma_k = ck.T @ ck / k.shape[0]
    sigma_v = cv.T @ cv / v.shape[0]
    m_q = q.T @ q / q.shape[0]
    return mu_k, sigma_k, mu_v, sigma_v, m_q


# ----------------------------------------------------------------------------------------------------
# 2. KLT
# ----------------------------------------------------------------------------------------------------
def klt(sigma):
    """Eigendecomposition of a symmetric covariance: (eigenvalues descending, U with eigenvectors as
    columns), sign fixed so that each column's largest-|.| entry is positive (first such index)."""
    lam, u = np.linalg.eigh(np.asarray(sigma, F64))
    order = np.argsort(-lam, kind="stable")
    lam = lam[order].copy()
    u = u[:, order].copy()
    for i in range(u.shape[1]):
        j = int(np.argmax(np.abs(u[:, i])))
        if u[j, i] < 0:
            u[:, i] = -u[:, i]
    return lam, u


# ----------------------------------------------------------------------------------------------------
# 3. importances
# ----------------------------------------------------------------------------------------------------
def attention_aware_key_basis(sigma_k, m_q, u0, sweeps: int = 8, grid: int = 48):
    """Orthogonal key basis for the attention-aware distortion. With white quantisation noise of variances
    D_i in basis U the key distortion is sum_i w_i D_i, w_i = u_i^T M_Q u_i, and water-filling against the
    coefficient variances s_i = u_i^T Sigma_K u_i makes it proportional (high-rate model) to
    (prod_i s_i w_i)^(1/d); the KLT minimises prod s_i alone (Hadamard) and ignores w. [NOVA-KV] derives the
    key transform from the attention-aware distortion (its optimum is not orthogonal); this keeps the
    transform orthogonal and minimises sum_i log s_i + log w_i by cyclic Jacobi sweeps from u0 (the KLT):
    pairs (i, j), i < j in row order, each rotated by the angle phi on the grid -pi/4 + k pi/(2 grid),
    k = 0 .. grid-1, that minimises the pair's four log terms (first such k), applied only when it beats
    phi = 0 by more than 1e-10. Sigma_K and M_Q are regularised by 1e-12 tr/d on the diagonal."""
    A = np.array(sigma_k, F64)
    B = np.array(m_q, F64)
    d = A.shape[0]
    A += np.eye(d) * (1e-12 * np.trace(A) / d)
    B += np.eye(d) * (1e-12 * np.trace(B) / d)
    U = np.array(u0, F64)
    a = U.T @ A @ U
    b = U.T @ B @ U
    phis = -np.pi / 4 + np.arange(grid) * (np.pi / 2 / grid)
    c, s = np.cos(phis), np.sin(phis)
    k0 = grid // 2                                            # phi = 0
    for _ in range(sweeps):
        for i in range(d - 1):
            for j in range(i + 1, d):
                f = (np.log(c * c * a[i, i] + 2 * c * s * a[i, j] + s * s * a[j, j]) +
                     np.log(s * s * a[i, i] - 2 * c * s * a[i, j] + c * c * a[j, j]) +
                     np.log(c * c * b[i, i] + 2 * c * s * b[i, j] + s * s * b[j, j]) +
                     np.log(s * s * b[i, i] - 2 * c * s * b[i, j] + c * c * b[j, j]))
                k = int(np.argmin(f))
                if not f[k] < f[k0] - 1e-10:
                    continue
                R = np.array([[c[k], -s[k]], [s[k], c[k]]])    # u_i <- c u_i + s u_j, u_j <- -s u_i + c u_j
                U[:, [i, j]] = U[:, [i, j]] @ R
                for M in (a, b):
                    M[:, [i, j]] = M[:, [i, j]] @ R
                    M[[i, j], :] = R.T @ M[[i, j], :]
    return U


def whitened_key_transform(sigma_k, m_q):
    """[NOVA-KV]'s key transform under the high-resolution model, which is not orthogonal: T = c V^T M_Q^(1/2)
    with V the eigenvectors (KLT) of M_Q^(1/2) Sigma_K M_Q^(1/2). The key distortion E_q[(q.e)^2] = e^T M_Q e
    then equals |T e|^2 / c^2, a mean-squared error in the transform domain (the pages' generalised Parseval
    relation), and the coefficients T k are uncorrelated with variances c^2 x the eigenvalues, so plain
    reverse water-filling on those variances allocates the bits. c is the largest column norm of
    (V^T M_Q^(1/2))^-1, so every column of T^-1 has norm <= 1 and |(T^-T q)_j| <= |q|. M_Q gets 1e-12 tr/d on
    the diagonal. Returns (variances, T with rows = channels, T^-1)."""
    A = np.asarray(sigma_k, F64)
    M = np.array(m_q, F64)
    d = M.shape[0]
    M += np.eye(d) * (1e-12 * np.trace(M) / d)
    lq, Q = np.linalg.eigh(M)
    m_half = (Q * np.sqrt(lq)) @ Q.T
    m_ihalf = (Q / np.sqrt(lq)) @ Q.T
    lam, V = klt(m_half @ A @ m_half)
    T = V.T @ m_half
    T_inv = m_ihalf @ V
    c = float(np.linalg.norm(T_inv, axis=0).max())
    return np.maximum(lam, 0.0) * c * c, T * c, T_inv / c


def basis_objective(u, sigma_k, m_q):
    """sum_i log(u_i^T Sigma_K u_i) + log(u_i^T M_Q u_i): the log of prod_i s_i w_i."""
    u = np.asarray(u, F64)
    return float(np.sum(np.log(np.einsum("ji,jk,ki->i", u, sigma_k, u))) +
                 np.sum(np.log(np.einsum("ji,jk,ki->i", u, m_q, u))))


def key_weights(u, m_q):
    """w_i = u_i^T M_Q u_i for each eigenvector column u_i."""
    u = np.asarray(u, F64)
    return np.einsum("ji,jk,ki->i", u, np.asarray(m_q, F64), u)


def key_importance(lam, u, m_q):
    return np.maximum(lam, 0.0) * key_weights(u, m_q)


def value_importance(lam):
    return np.maximum(np.asarray(lam, F64), 0.0)


# ----------------------------------------------------------------------------------------------------
# 4. reverse water-filling
# ----------------------------------------------------------------------------------------------------
def record_words(bits_per_elem: float, d: int) -> int:
    """R_w = floor(bits * d / 32): the budget counts the 32-bit scale/zero word."""
    return int(np.floor(bits_per_elem * d / 32.0 + 1e-9))


def code_bits(r_words: int) -> int:
    return 32 * r_words - 32


def water_fill_continuous(lam, budget: float, max_bits: int, iters: int = 200):
    """Continuous reverse water-filling: returns (b, theta) with b_i = clip(1/2 log2(lam_i/theta), 0, B).
    theta is found by bisection in log2(theta) over [log2(min lam) - 40, log2(max lam)]."""
    lam = np.asarray(lam, F64)
    d = lam.shape[0]
    pos = lam > 0
    if budget <= 0 or not pos.any():
        return np.zeros(d), None
    if budget >= max_bits * int(pos.sum()):
        return np.where(pos, float(max_bits), 0.0), None
    l2 = np.full(d, -np.inf)
    l2[pos] = np.log2(lam[pos])
    lo = l2[pos].min() - 40.0
    hi = l2[pos].max()

    def b_of(t):
        return np.clip(0.5 * (l2 - t), 0.0, float(max_bits))

    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if b_of(mid).sum() > budget:
            lo = mid
        else:
            hi = mid
    t = 0.5 * (lo + hi)
    return b_of(t), 2.0 ** t


def water_fill_integer(lam, budget: int, max_bits: int):
    """Integer widths: floors of the continuous solution, then the remaining bits one each to the channels
    with the largest fractional part (ties: larger lambda, then lower index), none above max_bits."""
    lam = np.asarray(lam, F64)
    b_real, _ = water_fill_continuous(lam, budget, max_bits)
    b_int = np.floor(b_real).astype(np.int64)
    remaining = int(budget - b_int.sum())
    # fractional parts compared at 1e-9 resolution so that ties in exact arithmetic stay ties after the
    # bisection's rounding noise (about 1e-15)
    frac_key = np.rint((b_real - b_int) * 1e9).astype(np.int64)
    cand = [i for i in range(lam.shape[0]) if b_int[i] < max_bits and lam[i] > 0]
    cand.sort(key=lambda i: (-frac_key[i], -lam[i], i))
    for i in cand[:max(remaining, 0)]:
        b_int[i] += 1
    return b_int


# ----------------------------------------------------------------------------------------------------
# 5. parameter set
# ----------------------------------------------------------------------------------------------------
def storage_order(widths, lam):
    d = len(widths)
    return sorted(range(d), key=lambda i: (-int(widths[i]), -float(lam[i]), i))


HALF = 16   # bits per half of a code word


def slot_layout(widths, r_words: int):
    """First-fit placement of the pair slots: pair k = storage channels (2k, 2k+1), slot width
    max(b_2k, b_2k+1), placed in pair order into the lowest code word (0 .. R_w - 2) whose halves have
    that many free bits, at the lowest free bit. Returns (word [d/2], pos [d/2]) with -1 for empty slots,
    or None when some slot finds no room."""
    w = np.asarray(widths, np.int64)
    if w.shape[0] % 2:
        w = np.concatenate([w, [0]])
    n_words = r_words - 1
    used = [0] * max(n_words, 0)
    word = np.full(w.shape[0] // 2, -1, np.int64)
    pos = np.full(w.shape[0] // 2, -1, np.int64)
    for k in range(w.shape[0] // 2):
        sw = int(max(w[2 * k], w[2 * k + 1]))
        if sw == 0:
            continue
        for u in range(n_words):
            if used[u] + sw <= HALF:
                word[k], pos[k] = u, used[u]
                used[u] += sw
                break
        else:
            return None
    return word, pos


def fit_cost_key(pair_importance: float, width: int) -> int:
    """Integer key ordering the cost 3 (lambda_2k + lambda_2k+1) 4^-w of taking one bit from a pair of
    width w: log2 of the cost (less the common log2 3) at 1e-9 resolution, so that costs equal in exact
    arithmetic compare equal after rounding noise of the statistics."""
    if pair_importance <= 0:
        return -(1 << 62)
    return int(np.rint(np.log2(pair_importance) * 1e9)) - 2_000_000_000 * int(width)


def fit_layout(widths, importance, r_words: int):
    """Widths (storage order) that the pair layout can hold: each pair's narrower channel raised to the
    pair's slot width, then single bits taken from the cheapest pair (smallest cost key; ties to the later
    pair) until first-fit placement succeeds."""
    b = np.asarray(widths, np.int64)
    lam = np.asarray(importance, F64)
    d = b.shape[0]
    assert d % 2 == 0
    w = [int(max(b[2 * k], b[2 * k + 1])) for k in range(d // 2)]
    plam = [float(lam[2 * k] + lam[2 * k + 1]) for k in range(d // 2)]
    while slot_layout(np.repeat(w, 2), r_words) is None:
        _, negk = min((fit_cost_key(plam[k], w[k]), -k) for k in range(d // 2) if w[k] > 0)
        w[-negk] -= 1
    return np.repeat(np.asarray(w, np.int64), 2)


def token_slot_layout(widths, r_words: int):
    """First-fit placement of single channels for the token-pair layout: channel j (width b_j) goes, in
    storage order, to the lowest of the 2 R_w - 2 code words of a two-token record whose 16-bit halves have
    b_j free bits, at the lowest free bit. Returns (word [d], pos [d]) with -1 for zero widths, or None
    when a channel finds no room."""
    w = np.asarray(widths, np.int64)
    n_words = 2 * r_words - 2
    used = [0] * max(n_words, 0)
    word = np.full(w.shape[0], -1, np.int64)
    pos = np.full(w.shape[0], -1, np.int64)
    for j in range(w.shape[0]):
        b = int(w[j])
        if b == 0:
            continue
        for u in range(n_words):
            if used[u] + b <= HALF:
                word[j], pos[j] = u, used[u]
                used[u] += b
                break
        else:
            return None
    return word, pos


def fit_token_layout(widths, importance, r_words: int):
    """Widths (storage order) that the token-pair layout can hold: single bits taken from the cheapest
    channel (smallest cost key of lambda_j, ties to the later channel) until first-fit placement succeeds."""
    w = [int(x) for x in np.asarray(widths, np.int64)]
    lam = [float(x) for x in np.asarray(importance, F64)]
    while token_slot_layout(w, r_words) is None:
        _, negj = min((fit_cost_key(lam[j], w[j]), -j) for j in range(len(w)) if w[j] > 0)
        w[-negj] -= 1
    return np.asarray(w, np.int64)


class TensorParams:
    """One tensor's (K or V) codec parameters in storage order. T: fp32 [d, d] (rows = storage channels);
    mu, sigma, inv_sigma: fp32 [d]; widths: int [d]; r_words: record length in 32-bit words per token;
    pairing: "channels" (key records, one token each, channel pairs share slots) or "tokens" (value
    records, two tokens each, one slot per channel); slot_word / slot_pos: the first-fit placement (per
    channel pair, resp. per channel)."""

    def __init__(self, T, mu, sigma, widths, r_words, eigvals=None, importance=None, pairing="channels",
                 T_inv=None):
        self.T = np.ascontiguousarray(T, F32)
        # inverse of a non-orthogonal transform (fp64; None: T is orthogonal and T^T is its inverse)
        self.T_inv = None if T_inv is None else np.asarray(T_inv, F64)
        self.mu = np.ascontiguousarray(mu, F32)
        self.sigma = np.ascontiguousarray(sigma, F32)
        w = np.asarray(widths, np.int64).copy()
        w[self.sigma == 0] = 0
        self.widths = w
        self.inv_sigma = np.where(self.sigma > 0, (1.0 / np.where(self.sigma > 0, self.sigma, 1)
                                                   .astype(F64)), 0.0).astype(F32)
        self.r_words = int(r_words)
        self.eigvals = eigvals
        self.importance = importance
        if pairing not in ("channels", "tokens"):
            raise ValueError(pairing)
        self.pairing = pairing
        lay = (slot_layout if pairing == "channels" else token_slot_layout)(self.widths, self.r_words)
        if lay is None:
            raise ValueError("widths do not fit the record layout")
        self.slot_word, self.slot_pos = lay

    @property
    def d(self):
        return self.T.shape[0]

    @property
    def tokens_per_record(self):
        return 1 if self.pairing == "channels" else 2

    @property
    def record_len(self):
        """32-bit words per record."""
        return self.r_words * self.tokens_per_record


def build_tensor_params(mu_raw, lam, u, importance, r_words: int, max_bits: int,
                        pairing: str = "channels", u_inv=None) -> TensorParams:
    widths_eig = water_fill_integer(importance, code_bits(r_words), max_bits)
    order = storage_order(widths_eig, importance)
    imp_st = np.asarray(importance)[order]
    if pairing == "channels":
        widths = fit_layout(widths_eig[order], imp_st, r_words)
    else:
        widths = fit_token_layout(widths_eig[order], imp_st, r_words)
    T = u[:, order].T                                   # rows: storage channels
    mu_rot = T @ np.asarray(mu_raw, F64)
    sigma = np.sqrt(np.maximum(lam[order], 0.0))
    # u_inv: the inverse of a non-orthogonal u^T; column i pairs with channel i, so it follows the storage order
    T_inv = None if u_inv is None else np.asarray(u_inv, F64)[:, order]
    return TensorParams(T=T, mu=mu_rot, sigma=sigma, widths=widths, r_words=r_words,
                        eigvals=lam[order], importance=imp_st, pairing=pairing, T_inv=T_inv)


def key_basis(s_k, m_q, attention_aware: bool):
    """(coefficient variances, basis) of the keys: the KLT, or the attention-aware basis started from it."""
    lam_k, u_k = klt(s_k)
    if not attention_aware:
        return lam_k, u_k
    u = attention_aware_key_basis(s_k, m_q, u_k)
    return np.einsum("ji,jk,ki->i", u, np.asarray(s_k, F64), u), u


def calibrate(k, v, q, bits_k: float, bits_v: float, max_bits: int = 8, attention_aware_keys: bool = False,
              whitened_keys: bool = False):
    """Full calibration of one (layer, KV head) set -> (TensorParams K, TensorParams V). whitened_keys: the
    non-orthogonal key transform of whitened_key_transform (the key importances are then the coefficient
    variances: the distortion is already mean-squared in that domain)."""
    d = np.asarray(k).shape[1]
    mu_k, s_k, mu_v, s_v, m_q = calib_statistics(k, v, q)
    if whitened_keys:
        lam_k, t_k, t_inv = whitened_key_transform(s_k, m_q)
        lam_v, u_v = klt(s_v)
        pk = build_tensor_params(mu_k, lam_k, t_k.T, lam_k, record_words(bits_k, d), max_bits, "channels",
                                 u_inv=t_inv)
        pv = build_tensor_params(mu_v, lam_v, u_v, value_importance(lam_v), record_words(bits_v, d), max_bits,
                                 "tokens")
        return pk, pv
    lam_k, u_k = key_basis(s_k, m_q, attention_aware_keys)
    lam_v, u_v = klt(s_v)
    imp_k = key_importance(lam_k, u_k, m_q)
    imp_v = value_importance(lam_v)
    pk = build_tensor_params(mu_k, lam_k, u_k, imp_k, record_words(bits_k, d), max_bits, "channels")
    pv = build_tensor_params(mu_v, lam_v, u_v, imp_v, record_words(bits_v, d), max_bits, "tokens")
    return pk, pv


# ----------------------------------------------------------------------------------------------------
# 5b. joint key/value allocation (one rate trade-off between the two tensors)
# ----------------------------------------------------------------------------------------------------
def exchange_rate(lam_v, d: int) -> float:
    """Weight of key distortion against value distortion in the attention output. To first order a key error
    e_t moves logit t by alpha q.e_t and the output by p_t alpha (q.e_t)(v_t - o); with white noise of
    variances D^K_i (key basis) and D^V_i (value basis), independent across tokens,
        E|do|^2 = sum_t p_t^2 (alpha^2 |v_t - o|^2 sum_i w_i D^K_i + sum_i D^V_i),
    additive in keys and values and factored over tokens and channels ([AATC] Key points, first bullet).
    Taking |v_t - o|^2 at its mean over tokens, tr(Sigma_V), with alpha = 1/sqrt(d) (the softmax scale the
    decode uses by default): rho = tr(Sigma_V) / d multiplies the key importances sigma_i^2 w_i."""
    return float(np.sum(np.maximum(np.asarray(lam_v, F64), 0.0))) / d


def joint_objective(imp_k, imp_v, rho: float, rwk: int, rwv: int, max_bits: int) -> float:
    """sum_i rho imp_k,i 4^-b_i + sum_j imp_v,j 4^-b_j with each tensor's integer water-filling at its own
    budget (the white-noise distortion of a b-bit channel is proportional to sigma^2 4^-b)."""
    bk = water_fill_integer(imp_k, code_bits(rwk), max_bits)
    bv = water_fill_integer(imp_v, code_bits(rwv), max_bits)
    return float(rho * np.sum(np.asarray(imp_k, F64) * 4.0 ** -bk.astype(F64)) +
                 np.sum(np.asarray(imp_v, F64) * 4.0 ** -bv.astype(F64)))


def joint_split(per_set, r_total: int, rwk_sep: int, max_bits: int, d: int) -> int:
    """Key record words R_wK (values get r_total - R_wK) minimising the sum over the parameter sets of
    joint_objective; per_set holds (imp_k, imp_v, rho) of each set. Candidates keep both tensors within
    1 .. 1 + max_bits d / 32 words. Objectives within a relative 1e-9 of the minimum tie; ties go to the split
    nearest rwk_sep (the separate allocation's), then to fewer key words."""
    cands = [r for r in range(1, r_total) if code_bits(r) <= max_bits * d and code_bits(r_total - r) <= max_bits * d]
    J = {r: sum(joint_objective(ik, iv, rho, r, r_total - r, max_bits) for ik, iv, rho in per_set) for r in cands}
    jmin = min(J.values())
    ties = [r for r in cands if J[r] <= jmin * (1.0 + 1e-9)]
    return min(ties, key=lambda r: (abs(r - rwk_sep), r))


def calibrate_joint(sets, bits_k: float, bits_v: float, max_bits: int = 8, attention_aware_keys: bool = False,
                    whitened_keys: bool = False):
    """Calibration of a table of sets [(k, v, q), ...] with the key/value split of the record chosen jointly:
    the table keeps R_wK + R_wV = record_words(bits_k) + record_words(bits_v) words per token, split as
    joint_split decides (one split for the table, since the cache holds one record length per tensor); each
    tensor is then allocated and laid out as in calibrate. Returns [(TensorParams K, TensorParams V), ...]."""
    d = np.asarray(sets[0][0]).shape[1]
    prep = []
    for k, v, q in sets:
        mu_k, s_k, mu_v, s_v, m_q = calib_statistics(k, v, q)
        lam_v, u_v = klt(s_v)
        if whitened_keys:   # importances: the coefficient variances (the distortion is mean-squared there)
            lam_k, t_k, t_inv = whitened_key_transform(s_k, m_q)
            key = (mu_k, lam_k, t_k.T, lam_k, t_inv)
        else:
            lam_k, u_k = key_basis(s_k, m_q, attention_aware_keys)
            key = (mu_k, lam_k, u_k, key_importance(lam_k, u_k, m_q), None)
        prep.append(key + (mu_v, lam_v, u_v, value_importance(lam_v), exchange_rate(lam_v, d)))
    rwk_sep, rwv_sep = record_words(bits_k, d), record_words(bits_v, d)
    rwk = joint_split([(p[3], p[8], p[9]) for p in prep], rwk_sep + rwv_sep, rwk_sep, max_bits, d)
    rwv = rwk_sep + rwv_sep - rwk
    return [(build_tensor_params(p[0], p[1], p[2], p[3], rwk, max_bits, "channels", u_inv=p[4]),
             build_tensor_params(p[5], p[6], p[7], p[8], rwv, max_bits, "tokens")) for p in prep]


# ----------------------------------------------------------------------------------------------------
# 6. quantiser (fp32, fixed op order)
# ----------------------------------------------------------------------------------------------------
def half_rn_sat(x):
    """fp32 -> fp16 round-to-nearest-even with saturation to +-65504 (numpy's conversion is RN-even)."""
    x = np.asarray(x, F32)
    return np.clip(x, F32(-HALF_MAX), F32(HALF_MAX)).astype(np.float16)


def rotate(x, p: TensorParams):
    """y = T x per token (fp64 matmul of the fp32 transform), rounded once to fp32."""
    return (np.asarray(x, F64) @ p.T.astype(F64).T).astype(F32)


def quantize(y32, p: TensorParams):
    """Codes for fp32 rotated coefficients y32 [n, d] -> (z fp16 [n], s fp16 [n], codes int64 [n, d])."""
    y32 = np.asarray(y32, F32)
    n, d = y32.shape
    nz = p.widths > 0
    codes = np.zeros((n, d), np.int64)
    if not nz.any():
        return np.zeros(n, np.float16), np.zeros(n, np.float16), codes
    yp = (y32[:, nz] - p.mu[nz]) * p.inv_sigma[nz]          # fp32 subtract, then fp32 multiply
    m = yp.min(axis=1)
    M = yp.max(axis=1)
    z16 = half_rn_sat(m)
    zf = z16.astype(F32)
    s16 = half_rn_sat(M - zf)
    sf = s16.astype(F32)
    scale = np.ldexp(np.ones(int(nz.sum()), F32), p.widths[nz].astype(np.int32)).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (yp - zf[:, None]) / sf[:, None]                # IEEE fp32 division
        u = t * scale[None, :]                              # exact power-of-two scaling
        c = np.floor(u)
    hi = (2 ** p.widths[nz]) - 1
    c = np.where(np.isfinite(c), c, 0.0)
    c = np.clip(c, 0, hi[None, :]).astype(np.int64)
    c[sf == 0] = 0
    codes[:, nz] = c
    return z16, s16, codes


# ----------------------------------------------------------------------------------------------------
# 7. record packing
# ----------------------------------------------------------------------------------------------------
def _slot_of(p: TensorParams, j: int, t_in_record: int = 0):
    """(word index within the record, bit shift) of storage channel j of the record's token t_in_record."""
    if p.pairing == "channels":
        k = j // 2
        return 1 + int(p.slot_word[k]), int(p.slot_pos[k]) + HALF * (j % 2)
    return 2 + int(p.slot_word[j]), int(p.slot_pos[j]) + HALF * t_in_record


def pack(z16, s16, codes, p: TensorParams):
    """-> uint32 records [n_records, record_len]: one token per record for keys, two for values (a missing
    second token leaves its words 0)."""
    codes = np.asarray(codes, np.int64)
    n, d = codes.shape
    tpr = p.tokens_per_record
    nrec = (n + tpr - 1) // tpr
    rec = np.zeros((nrec, p.record_len), np.uint64)
    zb = np.asarray(z16, np.float16).view(np.uint16).astype(np.uint64)
    sb = np.asarray(s16, np.float16).view(np.uint16).astype(np.uint64)
    for t in range(tpr):
        rows = slice(t, n, tpr)
        m = codes[rows].shape[0]
        rec[:m, t] = zb[rows] | (sb[rows] << np.uint64(16))
        for j in range(d):
            if int(p.widths[j]) == 0:
                continue
            w, sh = _slot_of(p, j, t)
            rec[:m, w] |= codes[rows, j].astype(np.uint64) << np.uint64(sh)
    return rec.astype(np.uint32)


def unpack(rec, p: TensorParams):
    """uint32 records -> (z fp16 [n], s fp16 [n], codes int64 [n, d]) for every token slot of the records
    (n = records x tokens per record)."""
    rec = np.asarray(rec, np.uint32).astype(np.uint64)
    tpr = p.tokens_per_record
    nrec = rec.shape[0]
    n = nrec * tpr
    z16 = np.zeros(n, np.float16)
    s16 = np.zeros(n, np.float16)
    codes = np.zeros((n, p.d), np.int64)
    for t in range(tpr):
        z16[t::tpr] = (rec[:, t] & np.uint64(0xFFFF)).astype(np.uint16).view(np.float16)
        s16[t::tpr] = (rec[:, t] >> np.uint64(16)).astype(np.uint16).view(np.float16)
        for j in range(p.d):
            b = int(p.widths[j])
            if b == 0:
                continue
            w, sh = _slot_of(p, j, t)
            codes[t::tpr, j] = ((rec[:, w] >> np.uint64(sh)) & np.uint64((1 << b) - 1)).astype(np.int64)
    return z16, s16, codes


def records_for(rec, p: TensorParams, n_tokens: int):
    """The leading records that hold the first n_tokens tokens."""
    tpr = p.tokens_per_record
    return np.asarray(rec)[:(n_tokens + tpr - 1) // tpr]


def encode(x, p: TensorParams):
    """Raw vectors x [n, d] -> records (one per token for keys, one per token pair for values)."""
    z, s, c = quantize(rotate(x, p), p)
    return pack(z, s, c, p)


# ----------------------------------------------------------------------------------------------------
# 8. decode attention
# ----------------------------------------------------------------------------------------------------
def dequantize(z16, s16, codes, p: TensorParams):
    """Rotated-domain reconstruction y^ [n, d] in fp64."""
    z = np.asarray(z16, np.float16).astype(F64)[:, None]
    s = np.asarray(s16, np.float16).astype(F64)[:, None]
    mu = p.mu.astype(F64)[None, :]
    sig = p.sigma.astype(F64)[None, :]
    b = p.widths[None, :]
    y = mu + sig * (z + (np.asarray(codes, F64) + 0.5) * s * np.power(2.0, -b.astype(F64)))
    return np.where(b > 0, y, np.broadcast_to(mu, y.shape))


def reconstruct(rec, p: TensorParams):
    """Records -> original-basis vectors x^ = T^-1 y^ [n, d] (fp64; T^-1 = T^T for an orthogonal T), one row per
    token slot."""
    y = dequantize(*unpack(rec, p), p)
    if p.T_inv is not None:
        return y @ p.T_inv.T
    return y @ p.T.astype(F64)


def attention(q, k, v, scale: float):
    """Exact single-query softmax attention in fp64: q [g, d], k/v [n, d] -> [g, d]."""
    q = np.asarray(q, F64)
    logits = scale * (q @ np.asarray(k, F64).T)
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return p @ np.asarray(v, F64)


def attend_decode(q, rec_k, rec_v, pk: TensorParams, pv: TensorParams, seq_len: int, scale: float):
    """Decode attention of the g query heads q [g, d] over the first seq_len tokens of one KV head."""
    kh = reconstruct(records_for(rec_k, pk, seq_len), pk)[:seq_len]
    vh = reconstruct(records_for(rec_v, pv, seq_len), pv)[:seq_len]
    return attention(q, kh, vh, scale)


# ----------------------------------------------------------------------------------------------------
# 9. rotary position embedding of the query
# ----------------------------------------------------------------------------------------------------
def rotary_embed(x, pos: int, base: float):
    """Rotary embedding of x [..., d] at integer position pos (fp64): for i < d/2 the pair (x_i, x_{i+d/2}) is
    turned by the angle pos * base^(-2i/d), x_i' = x_i cos - x_{i+d/2} sin, x_{i+d/2}' = x_i sin + x_{i+d/2} cos."""
    x = np.asarray(x, F64)
    d = x.shape[-1]
    half = d // 2
    freq = np.array([float(base) ** (-2.0 * i / d) for i in range(half)], F64)
    ang = float(pos) * freq
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, lo * s + hi * c], axis=-1)


# ----------------------------------------------------------------------------------------------------
# 10. token-axis allocation
# ----------------------------------------------------------------------------------------------------
def token_weights(q_obs, k, scale: float):
    """Weight of each token of one KV head: lambda_t = sum_q p_qt^2 with p_q = softmax_t(scale q . k_t) over the
    observation queries q_obs [n_q, d] of the head's query heads and the keys k [T, d], in fp64 -> [T]."""
    q = np.asarray(q_obs, F64)
    logits = scale * (q @ np.asarray(k, F64).T)
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return (p * p).sum(axis=0)


def token_keep(lam, keep: int):
    """Reverse water-filling on the token axis with one tier above zero bits: each token keeps its whole record
    or is evicted, and the water level leaves the `keep` tokens of largest weight (ties: the earlier token).
    -> the kept tokens' indices, ascending."""
    lam = np.asarray(lam, F64)
    order = sorted(range(lam.shape[0]), key=lambda t: (-lam[t], t))
    return np.array(sorted(order[:keep]), np.int64)


def compact(rec, p: TensorParams, keep_idx):
    """The records of the kept tokens keep_idx (ascending), in order, as a sequence of their own: one record per
    token for keys, value tokens paired anew two per record."""
    z, s, c = unpack(rec, p)
    idx = np.asarray(keep_idx, np.int64)
    return pack(z[idx], s[idx], c[idx], p)

