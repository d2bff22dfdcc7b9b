"""Checks that pin the float64 oracle to facts fixed outside the oracle itself.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  They are run against the real oracle (test_oracle_pins.py) and against
deliberately broken copies of it (test_oracle_mutants.py), which must each fail at
least one check.

Sources of the pinned facts:
* "FlashAttention: Move Less, Not Compute Less", section "Tiling Is Easy; Softmax
  Couples the Entire Row": the stable-softmax definition (rows of P sum to one,
  the max subtraction) and the online-softmax update (m', l', o'), restated
  blockwise below as an independent second algorithm.
* "FlashAttention-2: Why the Attention Bottleneck Wasn't Where Everyone Was
  Looking", sections "The hook: softmax doesn't tile" (S = QK^T + mask,
  P = softmax(S), O = PV), "FA2 change #1" (deferred division, L = m + log l).
* Course page "10 FlashAttention", section 4 "Tiny example — the algorithm":
  causal rule "query i sees keys 0..i", scale 1/sqrt(d), and the worked check
  that a blockwise computation (blocks of 128, S=2048, d=64) agrees with the
  textbook version to about 1e-15; section "The decode variant: FlashDecoding":
  partial results over disjoint key ranges merge with the same rescaling
  (associativity), which the decode pins use on uneven key splits.
* Library routines used as independent references on tiny inputs:
  ``scipy.special.softmax``/``logsumexp`` and torch float64 autograd.
"""
from __future__ import annotations

import json
import os

import numpy as np
import scipy.special

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _allowed_mask(N, causal):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return (j <= i) if causal else np.ones((N, N), dtype=bool)


def _close(a, b, tol, what):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max-abs error {err:.3e} > {tol:.1e}"
    return err


# ---------------------------------------------------------------- forward pins

def check_rows_of_p_sum_to_one(orc):
    """V = all ones makes O_i = sum_j P_ij, which the definition fixes at 1."""
    r = _rng(1)
    for causal in (False, True):
        q = r.standard_normal((2, 2, 37, 8))
        k = r.standard_normal((2, 2, 37, 8))
        v = np.ones((2, 2, 37, 8))
        o, _ = orc.fwd(q, k, v, causal=causal, scale=0.9, nthreads=2)
        _close(o, np.ones_like(o), 1e-14, f"sum P = 1 (causal={causal})")


def check_identity_v_is_softmax(orc):
    """With N = d and V = I, O is the probability matrix itself; compare with the
    library's softmax/logsumexp of the explicitly masked score matrix."""
    r = _rng(2)
    N = d = 12
    for causal in (False, True):
        q = r.standard_normal((1, 3, N, d))
        k = r.standard_normal((1, 3, N, d))
        v = np.broadcast_to(np.eye(d), (1, 3, N, d)).copy()
        scale = 0.37
        o, lse = orc.fwd(q, k, v, causal=causal, scale=scale, nthreads=1)
        s = scale * np.einsum("bhic,bhjc->bhij", q, k)
        s = np.where(_allowed_mask(N, causal), s, -np.inf)
        _close(o, scipy.special.softmax(s, axis=-1), 1e-14, f"P rows (causal={causal})")
        _close(lse, scipy.special.logsumexp(s, axis=-1), 1e-13, f"L (causal={causal})")


def check_identical_keys(orc):
    """All keys equal: P is uniform over allowed(i), so O_i is the mean of those V
    rows and L_i = scale*q_i.k + ln|allowed(i)|."""
    r = _rng(3)
    B, H, N, d = 1, 2, 50, 16
    q = r.standard_normal((B, H, N, d))
    krow = r.standard_normal((B, H, 1, d))
    k = np.repeat(krow, N, axis=2)
    v = r.standard_normal((B, H, N, d))
    scale = 0.25
    for causal in (False, True):
        o, lse = orc.fwd(q, k, v, causal=causal, scale=scale, nthreads=3)
        counts = np.arange(1, N + 1) if causal else np.full(N, N)
        if causal:
            mean_v = np.cumsum(v, axis=2) / counts[None, None, :, None]
        else:
            mean_v = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        _close(o, mean_v, 1e-13, f"identical keys O (causal={causal})")
        s = scale * np.einsum("bhic,bhc->bhi", q, krow[:, :, 0, :])
        _close(lse, s + np.log(counts)[None, None, :], 1e-12, f"identical keys L (causal={causal})")


def check_causal_row_zero(orc):
    """Causal row 0 sees only key 0: O_0 = V_0 and L_0 = scale*q_0.k_0."""
    r = _rng(4)
    q = r.standard_normal((2, 3, 9, 8))
    k = r.standard_normal((2, 3, 9, 8))
    v = r.standard_normal((2, 3, 9, 8))
    o, lse = orc.fwd(q, k, v, causal=True, scale=0.6, nthreads=2)
    _close(o[:, :, 0, :], v[:, :, 0, :], 0.0, "causal row 0 O")
    _close(lse[:, :, 0], 0.6 * np.sum(q[:, :, 0, :] * k[:, :, 0, :], axis=-1), 1e-14,
           "causal row 0 L")


def check_one_hot_dominant(orc):
    """Q rows = 16 e_0, K_t = 16 e_0, other keys 0, d = 64, scale = 1/8: the score of
    key t exceeds every other by 32, so rows that see t return V_t (within
    (N-1) e^-32); causal rows before t see only zero scores and return the mean."""
    r = _rng(5)
    N, d, t = 40, 64, 17
    q = np.zeros((1, 1, N, d))
    q[..., 0] = 16.0
    k = np.zeros((1, 1, N, d))
    k[0, 0, t, 0] = 16.0
    v = r.standard_normal((1, 1, N, d))
    for causal in (False, True):
        o, lse = orc.fwd(q, k, v, causal=causal, scale=1.0 / 8.0, nthreads=1)
        sees = np.arange(N) >= t if causal else np.ones(N, dtype=bool)
        tol = (N - 1) * np.exp(-32.0) * np.max(np.abs(v)) * 2 + 1e-15
        _close(o[0, 0, sees], np.broadcast_to(v[0, 0, t], (int(sees.sum()), d)), tol,
               f"one-hot O (causal={causal})")
        if causal:
            early = np.arange(t)
            mean_v = np.cumsum(v[0, 0, :t], axis=0) / (early + 1)[:, None]
            _close(o[0, 0, :t], mean_v, 1e-14, "one-hot causal early rows")
            _close(lse[0, 0, :t], np.log(early + 1.0), 1e-14, "one-hot causal early L")
        # L_i = ln(e^32 + (n_i - 1) e^0), n_i = number of keys row i may see
        n_i = (np.arange(N) + 1.0) if causal else np.full(N, float(N))
        l_ref = 32.0 + np.log1p((n_i - 1.0) * np.exp(-32.0))
        _close(lse[0, 0, sees], l_ref[sees], 1e-13, f"one-hot L (causal={causal})")


def check_large_scores_stable(orc):
    """Scores near +-1000 overflow exp() unless the row max is subtracted first
    (the stable form); the result must stay finite and pick the best key."""
    r = _rng(6)
    N, d = 24, 4
    q = np.zeros((1, 1, N, d))
    q[..., 0] = 100.0
    k = np.zeros((1, 1, N, d))
    k[0, 0, :, 0] = np.linspace(-10.0, 10.0, N)
    v = r.standard_normal((1, 1, N, d))
    o, lse = orc.fwd(q, k, v, causal=False, scale=1.0, nthreads=1)
    # the top key's score exceeds the next by 100*20/23 = 87 > 36 nats
    _close(o[0, 0], np.broadcast_to(v[0, 0, N - 1], (N, d)), 1e-14, "large-score O")
    _close(lse[0, 0], np.full(N, 1000.0), 1e-12, "large-score L")


def check_shift_invariance(orc):
    """Adding c to every key leaves P unchanged and shifts L_i by scale*q_i.c."""
    r = _rng(7)
    B, H, N, d = 1, 2, 33, 8
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    c = r.standard_normal(d)
    for causal in (False, True):
        o0, l0 = orc.fwd(q, k, v, causal=causal, scale=0.5, nthreads=2)
        o1, l1 = orc.fwd(q, k + c, v, causal=causal, scale=0.5, nthreads=2)
        _close(o1, o0, 1e-13, f"shift O (causal={causal})")
        _close(l1, l0 + 0.5 * np.einsum("bhic,c->bhi", q, c), 1e-12, f"shift L (causal={causal})")


def check_merge_of_halves(orc):
    """Online softmax is associative: (O, L) over keys [0,n) and [n,2n) combine by the
    rescale rule into (O, L) over all 2n keys."""
    r = _rng(8)
    n, d = 30, 8
    q = r.standard_normal((1, 2, n, d))
    k = r.standard_normal((1, 2, 2 * n, d))
    v = r.standard_normal((1, 2, 2 * n, d))
    oa, la = orc.fwd(q, k[:, :, :n], v[:, :, :n], scale=0.3, nthreads=1)
    ob, lb = orc.fwd(q, k[:, :, n:], v[:, :, n:], scale=0.3, nthreads=1)
    of, lf = orc.fwd(np.concatenate([q, q], axis=2), k, v, scale=0.3, nthreads=1)
    lm = np.logaddexp(la, lb)
    om = np.exp(la - lm)[..., None] * oa + np.exp(lb - lm)[..., None] * ob
    _close(of[:, :, :n], om, 1e-13, "merged O")
    _close(lf[:, :, :n], lm, 1e-13, "merged L")


def check_brute_force(orc):
    """Full score matrix with the library softmax on tiny random inputs."""
    r = _rng(9)
    for (B, H, N, d) in [(1, 1, 1, 4), (2, 3, 7, 5), (1, 2, 33, 16)]:
        q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
        scale = float(r.uniform(0.1, 1.5))
        for causal in (False, True):
            o, lse = orc.fwd(q, k, v, causal=causal, scale=scale, nthreads=2)
            s = scale * np.einsum("bhic,bhjc->bhij", q, k)
            s = np.where(_allowed_mask(N, causal), s, -np.inf)
            p = scipy.special.softmax(s, axis=-1)
            _close(o, p @ v, 1e-13, f"brute force O {B,H,N,d} causal={causal}")
            _close(lse, scipy.special.logsumexp(s, axis=-1), 1e-13, "brute force L")


def blockwise_attention(q, k, v, block_q, block_k, causal, scale):
    """Second, independent algorithm: the online-softmax update of the essay's
    equations applied block by block with the deferred final division.
    q, k, v: [N, d] float64.  Returns (O, L)."""
    N, d = q.shape
    out = np.empty_like(q)
    lse = np.empty(N)
    for i0 in range(0, N, block_q):
        rows = np.arange(i0, min(i0 + block_q, N))
        m = np.full(rows.size, -np.inf)
        ell = np.zeros(rows.size)
        acc = np.zeros((rows.size, d))
        key_end = rows[-1] + 1 if causal else N
        for j0 in range(0, key_end, block_k):
            cols = np.arange(j0, min(j0 + block_k, key_end))
            x = scale * (q[rows] @ k[cols].T)
            if causal:
                x = np.where(cols[None, :] <= rows[:, None], x, -np.inf)
            m_new = np.maximum(m, x.max(axis=1))
            alpha = np.exp(m - m_new)
            pexp = np.exp(x - m_new[:, None])
            ell = alpha * ell + pexp.sum(axis=1)
            acc = alpha[:, None] * acc + pexp @ v[cols]
            m = m_new
        out[rows] = acc / ell[:, None]
        lse[rows] = m + np.log(ell)
    return out, lse


def check_blockwise_equivalence(orc, big=True):
    """The course page's worked check (blocks of 128, S = 2048, d = 64, causal,
    agreement ~1e-15) plus odd block sizes on smaller inputs."""
    with open(os.path.join(GOLDEN, "page_checks.json")) as f:
        spec = json.load(f)["blockwise_vs_textbook"]
    r = _rng(10)
    cases = [(37, 8, 1, 1), (64, 8, 7, 5), (200, 16, 128, 128)]
    if big:
        cases.append((spec["S"], spec["d"], spec["blockQ"], spec["blockK"]))
    for (N, d, bq, bk) in cases:
        q, k, v = (r.standard_normal((1, 1, N, d)) for _ in range(3))
        scale = 1.0 / np.sqrt(d)
        for causal in ((True,) if (N, d) == (spec["S"], spec["d"]) else (False, True)):
            o, lse = orc.fwd(q, k, v, causal=causal, scale=scale)
            ob, lb = blockwise_attention(q[0, 0], k[0, 0], v[0, 0], bq, bk, causal, scale)
            _close(o[0, 0], ob, spec["asserted_max_abs"], f"blockwise O N={N} bq={bq}")
            _close(lse[0, 0], lb, spec["asserted_max_abs"], f"blockwise L N={N} bq={bq}")


def check_rows_subset(orc):
    """fwd_rows returns exactly the selected rows of the full forward."""
    r = _rng(11)
    q, k, v = (r.standard_normal((2, 2, 45, 8)) for _ in range(3))
    rows = np.array([0, 3, 17, 44])
    for causal in (False, True):
        o, lse = orc.fwd(q, k, v, causal=causal, scale=0.4, nthreads=3)
        orows, lrows = orc.fwd_rows(q, k, v, rows, causal=causal, scale=0.4, nthreads=2)
        assert np.array_equal(orows, o[:, :, rows]), "fwd_rows O differs from fwd"
        assert np.array_equal(lrows, lse[:, :, rows]), "fwd_rows L differs from fwd"


def check_thread_count_independent(orc):
    r = _rng(12)
    q, k, v = (r.standard_normal((1, 3, 40, 8)) for _ in range(3))
    a = orc.fwd(q, k, v, causal=True, scale=0.5, nthreads=1)
    b = orc.fwd(q, k, v, causal=True, scale=0.5, nthreads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), "thread count changed O/L"


# --------------------------------------------------------------- backward pins

def _loss(orc, q, k, v, do, causal, scale):
    o, _ = orc.fwd(q, k, v, causal=causal, scale=scale, nthreads=1)
    return float(np.sum(o * do))


def check_bwd_finite_differences(orc):
    """Central differences of f = sum(O * dO) through the oracle's own forward."""
    r = _rng(13)
    B, H, N, d = 1, 2, 6, 4
    h = 1e-5
    for causal in (False, True):
        q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
        scale = 0.7
        dq, dk, dv = orc.bwd(q, k, v, do, causal=causal, scale=scale, nthreads=2)
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.empty_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                fp = _loss(orc, q, k, v, do, causal, scale)
                x[idx] = old - h
                fm = _loss(orc, q, k, v, do, causal, scale)
                x[idx] = old
                num[idx] = (fp - fm) / (2 * h)
            _close(g, num, 1e-8, f"finite differences {name} (causal={causal})")


def check_bwd_torch_autograd(orc):
    """torch float64 autograd of the explicit formula on tiny inputs."""
    import torch
    r = _rng(14)
    for (B, H, N, d) in [(1, 1, 1, 4), (1, 2, 9, 8), (2, 1, 31, 16)]:
        for causal in (False, True):
            q, k, v, do = (r.standard_normal((B, H, N, d)) for _ in range(4))
            scale = 0.45
            tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
            s = scale * tq @ tk.transpose(-1, -2)
            if causal:
                s = s.masked_fill(~torch.tensor(_allowed_mask(N, True)), float("-inf"))
            o = torch.softmax(s, dim=-1) @ tv
            o.backward(torch.tensor(do))
            dq, dk, dv = orc.bwd(q, k, v, do, causal=causal, scale=scale, nthreads=2)
            _close(dq, tq.grad.numpy(), 1e-12, "autograd dQ")
            _close(dk, tk.grad.numpy(), 1e-12, "autograd dK")
            _close(dv, tv.grad.numpy(), 1e-12, "autograd dV")


def check_bwd_invariants(orc):
    """Per head: sum_j dK_j = 0 (each row of dS sums to D_i - D_i) and
    sum_j dV_j = sum_i dO_i (each row of P sums to one)."""
    r = _rng(15)
    q, k, v, do = (r.standard_normal((2, 2, 70, 8)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.bwd(q, k, v, do, causal=causal, scale=0.35, nthreads=4)
        _close(dk.sum(axis=2), np.zeros((2, 2, 8)), 1e-11, f"sum dK (causal={causal})")
        _close(dv.sum(axis=2), do.sum(axis=2), 1e-11, f"sum dV (causal={causal})")


def check_bwd_rows_partition(orc):
    """Backward over a partition of the query rows: the dQ rows are those of the
    full backward and the dK, dV contributions add up to the full dK, dV."""
    r = _rng(16)
    q, k, v, do = (r.standard_normal((1, 2, 41, 8)) for _ in range(4))
    rows_a = np.array([0, 3, 7, 8, 20, 40])
    rows_b = np.setdiff1d(np.arange(41), rows_a)
    for causal in (False, True):
        dq, dk, dv = orc.bwd(q, k, v, do, causal=causal, scale=0.5, nthreads=3)
        qa, ka, va = orc.bwd_rows(q, k, v, do, rows_a, causal=causal, scale=0.5, nthreads=2)
        qb, kb, vb = orc.bwd_rows(q, k, v, do, rows_b, causal=causal, scale=0.5, nthreads=4)
        _close(qa, dq[:, :, rows_a], 1e-14, "bwd_rows dQ (a)")
        _close(qb, dq[:, :, rows_b], 1e-14, "bwd_rows dQ (b)")
        _close(ka + kb, dk, 1e-13, "bwd_rows dK partition")
        _close(va + vb, dv, 1e-13, "bwd_rows dV partition")


# ---------------------------------------------------------------- decode pins

def check_decode_brute_force(orc):
    """Decode shapes (Nq query rows against Nk keys, no mask): full score matrix with
    the library softmax and logsumexp on tiny random inputs."""
    r = _rng(20)
    for (B, H, Nq, Nk, d) in [(1, 1, 1, 1, 4), (1, 2, 1, 40, 8), (2, 3, 5, 17, 16), (1, 1, 9, 3, 6)]:
        q = r.standard_normal((B, H, Nq, d))
        k, v = (r.standard_normal((B, H, Nk, d)) for _ in range(2))
        scale = float(r.uniform(0.1, 1.5))
        o, lse = orc.decode(q, k, v, scale=scale, nthreads=2)
        s = scale * np.einsum("bhic,bhjc->bhij", q, k)
        p = scipy.special.softmax(s, axis=-1)
        _close(o, p @ v, 1e-13, f"decode brute force O {B,H,Nq,Nk,d}")
        _close(lse, scipy.special.logsumexp(s, axis=-1), 1e-13, f"decode brute force L {B,H,Nq,Nk,d}")


def check_decode_identical_keys(orc):
    """All Nk keys equal: every query row averages V, and L = scale*q.k + ln Nk."""
    r = _rng(21)
    B, H, Nq, Nk, d = 2, 2, 3, 77, 8
    q = r.standard_normal((B, H, Nq, d))
    krow = r.standard_normal((B, H, 1, d))
    k = np.repeat(krow, Nk, axis=2)
    v = r.standard_normal((B, H, Nk, d))
    o, lse = orc.decode(q, k, v, scale=0.4, nthreads=3)
    _close(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), 1e-13, "decode identical keys O")
    s = 0.4 * np.einsum("bhic,bhc->bhi", q, krow[:, :, 0, :])
    _close(lse, s + np.log(Nk), 1e-12, "decode identical keys L")


def check_decode_merge_of_splits(orc):
    """The decode variant's key split: (O_s, L_s) over disjoint key ranges merge into
    the result over all keys by L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s
    (the course page's statement that partial results combine with the same
    rescaling).  Uneven splits, one of a single key."""
    r = _rng(22)
    B, H, Nq, Nk, d = 1, 3, 2, 61, 8
    q = r.standard_normal((B, H, Nq, d))
    k, v = (r.standard_normal((B, H, Nk, d)) for _ in range(2))
    full_o, full_l = orc.decode(q, k, v, scale=0.7, nthreads=2)
    cuts = [0, 1, 20, 44, Nk]
    parts = [orc.decode(q, k[:, :, a:b], v[:, :, a:b], scale=0.7, nthreads=1)
             for a, b in zip(cuts[:-1], cuts[1:])]
    ls = np.stack([p[1] for p in parts])
    lm = scipy.special.logsumexp(ls, axis=0)
    om = sum(np.exp(p[1] - lm)[..., None] * p[0] for p in parts)
    _close(om, full_o, 1e-13, "decode merged O")
    _close(lm, full_l, 1e-13, "decode merged L")


def check_decode_is_noncausal_forward(orc):
    """With Nq = Nk the decode rows are the non-causal forward's rows."""
    r = _rng(23)
    q, k, v = (r.standard_normal((2, 2, 13, 8)) for _ in range(3))
    o1, l1 = orc.decode(q, k, v, scale=0.3, nthreads=2)
    o2, l2 = orc.fwd(q, k, v, causal=False, scale=0.3, nthreads=2)
    _close(o1, o2, 0.0, "decode vs forward O")
    _close(l1, l2, 0.0, "decode vs forward L")


FORWARD_CHECKS = [
    check_rows_of_p_sum_to_one,
    check_identity_v_is_softmax,
    check_identical_keys,
    check_causal_row_zero,
    check_one_hot_dominant,
    check_large_scores_stable,
    check_shift_invariance,
    check_merge_of_halves,
    check_brute_force,
    check_blockwise_equivalence,
    check_rows_subset,
    check_thread_count_independent,
    check_decode_brute_force,
    check_decode_identical_keys,
    check_decode_merge_of_splits,
    check_decode_is_noncausal_forward,
]
BACKWARD_CHECKS = [
    check_bwd_finite_differences,
    check_bwd_torch_autograd,
    check_bwd_invariants,
    check_bwd_rows_partition,
]
ALL_CHECKS = FORWARD_CHECKS + BACKWARD_CHECKS
