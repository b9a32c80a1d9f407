"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when it disagrees with what the
pages print or the mathematics fixes. ``test_oracle.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on copies of ``oracle.c`` with one planted mistake each
and requires that every mistake is caught by at least one pin.

Sources (page title, section):
  worked example, merge   -- "11. Fusion, recompute, and flash attention", section 11.6 and the
                             solution of exercise 3 (fixtures in tests/golden/).
  stable softmax          -- ithelp article 10405336, "先回顧 Stable Softmax": subtracting the
                             row max does not change the result.
  late maximum            -- same chapter, "Pitfalls": forgetting to rescale o passes on small
                             scores, so test rows whose maximum arrives late.
  causal                  -- same chapter, exercise "Causal mask": query i sees keys j <= i.
"""
from __future__ import annotations

import itertools
import math
from pathlib import Path

import numpy as np
import scipy.special

GOLDEN = Path(__file__).resolve().parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    ok = np.all(np.isfinite(a)) and np.allclose(a, b, rtol=rtol, atol=atol)
    if not ok:
        err = np.nanmax(np.abs(a - b)) if a.shape == b.shape else "shape"
        raise AssertionError(f"{what}: max |diff| = {err}")


def read_worked_example():
    rows, final = [], None
    for line in (GOLDEN / "online_softmax_worked_example.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "final":
            final = float(f[1])
        else:
            rows.append(dict(zip(("key", "s", "m", "corr", "p", "l", "o"), map(float, f))))
    return rows, final


def read_merge_example():
    parts, final = {}, None
    for line in (GOLDEN / "merge_two_states.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "final":
            final = float(f[1])
        else:
            parts[f[0]] = tuple(map(float, f[1:]))
    return parts, final


WORKED_Q = np.array([[1.0]])
WORKED_K = np.array([[1.0], [3.0], [2.0]])
WORKED_V = np.array([[10.0], [20.0], [30.0]])


# --- values the pages print -------------------------------------------------------------------

def pin_worked_example_states(orc):
    """State (m, l, o) after each key, and the correction and weight of each step."""
    rows, _ = read_worked_example()
    prev_m = -math.inf
    prev_l = 0.0
    for r in rows:
        j = int(r["key"])
        m, l, o = orc.online_state(WORKED_Q[0], WORKED_K, WORKED_V, 0, j + 1, 1.0, block=1)
        _close(m, r["m"], 0, 5e-5, f"m after key {j}")
        _close(l, r["l"], 0, 5e-5, f"l after key {j}")
        _close(o[0], r["o"], 0, 5e-5, f"o after key {j}")
        # The printed corr and p follow from two consecutive states and the score.
        corr = 0.0 if prev_m == -math.inf else math.exp(prev_m - m)
        _close(corr, r["corr"], 0, 5e-5, f"corr at key {j}")
        _close(l - prev_l * corr, r["p"], 0, 5e-5, f"p at key {j}")
        prev_m, prev_l = m, l


def pin_worked_example_final(orc):
    _, final = read_worked_example()
    o = orc.attention(WORKED_Q, WORKED_K, WORKED_V, 1.0)
    _close(o[0, 0], final, 0, 5e-7, "two-pass o/l")
    for block in (1, 2, 3):
        o = orc.attention_online(WORKED_Q, WORKED_K, WORKED_V, 1.0, block=block)
        _close(o[0, 0], final, 0, 5e-7, f"online o/l, block {block}")


def pin_merge_example(orc):
    parts, final = read_merge_example()
    s0 = orc.online_state(WORKED_Q[0], WORKED_K, WORKED_V, 0, 1, 1.0)
    s12 = orc.online_state(WORKED_Q[0], WORKED_K, WORKED_V, 1, 3, 1.0)
    for (m, l, o), key in ((s0, "keys0"), (s12, "keys12")):
        _close([m, l, o[0]], parts[key], 0, 5e-5, f"state {key}")
    m, l, o = orc.merge_state(s0, s12)
    _close([m, l, o[0]], parts["merged"], 0, 5e-5, "merged state")
    _close(o[0] / l, final, 0, 5e-4, "merged o/l")
    m2, l2, o2 = orc.merge_state(s12, s0)  # the merge is symmetric
    _close([m2, l2, o2[0]], [m, l, o[0]], 1e-15, 0, "merge order")


# --- closed forms -----------------------------------------------------------------------------

def pin_equal_scores_give_mean(orc):
    """q = 0 (or scale = 0): every visible key weighs the same, O is the mean of V."""
    rng = _rng(11)
    for causal in (False, True):
        for nq, nk, d in ((5, 7, 3), (9, 9, 4), (4, 13, 2)):
            k = rng.standard_normal((nk, d))
            v = rng.standard_normal((nk, d))
            q = rng.standard_normal((nq, d))
            want = np.stack([v[: (min(i + 1, nk) if causal else nk)].mean(0) for i in range(nq)])
            _close(orc.attention(np.zeros((nq, d)), k, v, 0.7, causal), want, 1e-13, 1e-13,
                   f"q=0 mean, causal={causal}")
            _close(orc.attention(q, k, v, 0.0, causal), want, 1e-13, 1e-13,
                   f"scale=0 mean, causal={causal}")
            _close(orc.attention_online(q, k, v, 0.0, causal, block=3), want, 1e-13, 1e-13,
                   f"online scale=0 mean, causal={causal}")


def pin_single_key_gives_v(orc):
    """Nk = 1: softmax over one key is 1, so every row of O is V[0]; LSE is that one score."""
    rng = _rng(12)
    q = rng.standard_normal((6, 5))
    k = rng.standard_normal((1, 5))
    v = rng.standard_normal((1, 5))
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, 0.3, causal, with_lse=True)
        _close(o, np.repeat(v, 6, 0), 1e-15, 0, "Nk=1")
        _close(lse, 0.3 * (q @ k[0]), 1e-13, 1e-14, "Nk=1 lse")
        _close(orc.attention_online(q, k, v, 0.3, causal), np.repeat(v, 6, 0), 1e-15, 0,
               "online Nk=1")


def pin_causal_first_row_is_v0(orc):
    rng = _rng(13)
    q, k, v = (rng.standard_normal((8, 4)) * 3 for _ in range(3))
    _close(orc.attention(q, k, v, 0.5, True)[0], v[0], 1e-15, 0, "causal row 0")
    _close(orc.attention_online(q, k, v, 0.5, True, block=4)[0], v[0], 1e-15, 0,
           "online causal row 0")


def pin_dominant_key(orc):
    """One key whose score exceeds the rest by more than 800: O is that key's V, exactly in
    fp64, and nothing overflows (the max subtraction of the stable softmax is needed)."""
    d = 4
    k = np.zeros((5, d))
    k[3, 0] = 1.0
    v = np.arange(20, dtype=np.float64).reshape(5, d)
    q = np.zeros((2, d))
    q[:, 0] = [900.0, 1200.0]
    for fn in (lambda: orc.attention(q, k, v, 1.0),
               lambda: orc.attention_online(q, k, v, 1.0, block=2)):
        _close(fn(), np.repeat(v[3:4], 2, 0), 0, 1e-12, "dominant key")


def pin_lse_closed_form(orc):
    """LSE = log sum_j exp(s_j), from scipy's logsumexp over the visible scores."""
    rng = _rng(14)
    q, k, v = rng.standard_normal((7, 6)), rng.standard_normal((9, 6)), rng.standard_normal((9, 6))
    for causal in (False, True):
        s = 0.4 * (q @ k.T)
        want = np.array([scipy.special.logsumexp(s[i, : (i + 1 if causal else 9)])
                         for i in range(7)])
        _, lse = orc.attention(q, k, v, 0.4, causal, with_lse=True)
        _close(lse, want, 1e-13, 1e-13, f"lse causal={causal}")
        _, lse2 = orc.attention_online(q, k, v, 0.4, causal, block=4, with_lse=True)
        _close(lse2, want, 1e-13, 1e-13, f"online lse causal={causal}")


# --- invariants -------------------------------------------------------------------------------

def pin_row_shift_invariance(orc):
    """K' = K + u adds the per-row constant scale*(q_i . u) to every score of row i; O must not
    move, even when the constant is in the thousands (max subtraction keeps exp finite)."""
    rng = _rng(15)
    nq, nk, d = 6, 11, 8
    q, k, v = rng.standard_normal((nq, d)), rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    base = orc.attention(q, k, v, 0.35, False)
    for mag in (1.0, 40.0, 3000.0):
        u = rng.standard_normal(d) * mag
        _close(orc.attention(q, k + u, v, 0.35, False), base, 1e-9, 1e-10, f"shift {mag}")
        _close(orc.attention_online(q, k + u, v, 0.35, False, block=3), base, 1e-9, 1e-10,
               f"online shift {mag}")


def pin_negative_scale_is_negated_keys(orc):
    """A negative scale weights the most negative scores most: attention with -scale equals
    attention with K negated and +scale, exactly (the scores are the same numbers), causal or
    not, with the LSE too; and the weights still form a distribution."""
    rng = _rng(29)
    nq, nk, d = 7, 13, 5
    q, k, v = rng.standard_normal((nq, d)) * 2, rng.standard_normal((nk, d)) * 2, rng.standard_normal((nk, d))
    for causal in (False, True):
        o_neg, l_neg = orc.attention(q, k, v, -0.7, causal, with_lse=True)
        o_ref, l_ref = orc.attention(q, -k, v, 0.7, causal, with_lse=True)
        _close(o_neg, o_ref, 1e-14, 1e-15, f"negative scale causal={causal}")
        _close(l_neg, l_ref, 1e-14, 1e-15, f"negative scale LSE causal={causal}")
        p = orc.softmax(q, k, -0.7, causal)
        _close(p.sum(1), np.ones(nq), 1e-14, 0, f"negative scale rows causal={causal}")
        # The weight goes to the key with the most negative score q . k (row 0, non-causal).
        if not causal:
            s0 = q[0] @ k.T
            if int(np.argmax(p[0])) != int(np.argmin(s0)):
                raise AssertionError("largest weight is not on the most negative score")


def pin_softmax_rows_are_distributions(orc):
    rng = _rng(16)
    q, k = rng.standard_normal((10, 5)) * 2, rng.standard_normal((12, 5)) * 2
    for causal in (False, True):
        p = orc.softmax(q, k, 0.6, causal)
        _close(p.sum(1), np.ones(10), 1e-14, 0, f"row sums causal={causal}")
        if np.any(p < 0):
            raise AssertionError("negative probability")
        if causal and np.any(np.triu(p, 1) != 0):
            raise AssertionError("hidden key has weight")


def pin_key_permutation(orc):
    rng = _rng(17)
    q, k, v = rng.standard_normal((5, 7)), rng.standard_normal((16, 7)), rng.standard_normal((16, 7))
    perm = rng.permutation(16)
    _close(orc.attention(q, k[perm], v[perm], 0.5), orc.attention(q, k, v, 0.5), 1e-13, 1e-14,
           "key permutation")


def pin_query_permutation(orc):
    rng = _rng(18)
    q, k, v = rng.standard_normal((9, 4)), rng.standard_normal((6, 4)), rng.standard_normal((6, 4))
    perm = rng.permutation(9)
    _close(orc.attention(q[perm], k, v, 0.5), orc.attention(q, k, v, 0.5)[perm], 1e-15, 0,
           "query permutation")


def pin_causal_row_is_prefix_attention(orc):
    """Causal row i equals non-causal attention of query i over keys 0..i."""
    rng = _rng(19)
    n, d = 12, 3
    q, k, v = rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d)), rng.standard_normal((n, d))
    oc = orc.attention(q, k, v, 0.8, True)
    for i in range(n):
        _close(oc[i], orc.attention(q[i:i + 1], k[: i + 1], v[: i + 1], 0.8)[0], 1e-14, 1e-15,
               f"causal prefix {i}")


def pin_causal_wide_keys(orc):
    """Causal with Nk > Nq: query i still sees keys 0..i only (top-left alignment)."""
    rng = _rng(20)
    q, k, v = rng.standard_normal((4, 3)), rng.standard_normal((10, 3)), rng.standard_normal((10, 3))
    oc = orc.attention(q, k, v, 1.0, True)
    for i in range(4):
        _close(oc[i], orc.attention(q[i:i + 1], k[: i + 1], v[: i + 1], 1.0)[0], 1e-14, 1e-15,
               f"causal wide {i}")


def pin_batched_slices_independent(orc):
    """Leading (batch, head) slices are independent problems."""
    rng = _rng(21)
    q, k, v = rng.standard_normal((2, 3, 5, 4)), rng.standard_normal((2, 3, 7, 4)), rng.standard_normal((2, 3, 7, 4))
    o = orc.attention(q, k, v, 0.5, True)
    for b in range(2):
        for h in range(3):
            _close(o[b, h], orc.attention(q[b, h], k[b, h], v[b, h], 0.5, True), 0, 0,
                   f"slice {b},{h}")
    rows = orc.attention_rows(q[1, 2, [4, 0, 2]], [4, 0, 2], k[1, 2], v[1, 2], 0.5, True)
    _close(rows, o[1, 2, [4, 0, 2]], 0, 0, "attention_rows")


def pin_late_maximum(orc):
    """Scores that rise along the row move the running max at every key; O must still match the
    definition (the page's pitfall: forgetting to rescale o)."""
    n, d = 40, 2
    k = np.zeros((n, d))
    k[:, 0] = np.linspace(0.0, 6.0, n)  # score grows with the key index
    v = np.stack([np.arange(n, dtype=np.float64), np.ones(n)], 1)
    q = np.array([[1.0, 0.0], [2.5, 0.0]])
    s = q @ k.T
    want = scipy.special.softmax(s, axis=1) @ v
    _close(orc.attention(q, k, v, 1.0), want, 1e-13, 1e-13, "late max, two-pass")
    for block in (1, 3, 7):
        _close(orc.attention_online(q, k, v, 1.0, block=block), want, 1e-13, 1e-13,
               f"late max, online block {block}")


# --- library routine and brute force ----------------------------------------------------------

def pin_matches_scipy_softmax(orc):
    """The P3 chapter's own check: NumPy two-pass attention. Here scipy.special.softmax over the
    masked score matrix, times V."""
    rng = _rng(22)
    for nq, nk, d, causal in ((7, 7, 5, True), (5, 12, 9, False), (16, 16, 8, True), (3, 1, 2, False)):
        q = rng.standard_normal((nq, d)) * 2
        k, v = rng.standard_normal((nk, d)) * 2, rng.standard_normal((nk, d))
        s = 0.45 * (q @ k.T)
        if causal:
            s = np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None], s, -np.inf)
        want = scipy.special.softmax(s, axis=1) @ v
        _close(orc.attention(q, k, v, 0.45, causal), want, 1e-13, 1e-13,
               f"scipy nq={nq} nk={nk} causal={causal}")
        _close(orc.attention_online(q, k, v, 0.45, causal, block=5), want, 1e-13, 1e-13,
               f"scipy online nq={nq} nk={nk} causal={causal}")


def _literal(q, k, v, scale, causal):
    """The formula as written, in plain Python: exp of each score without the max subtraction.
    Safe only for the small scores used here."""
    nq, d = len(q), len(q[0])
    nk = len(k)
    out = []
    for i in range(nq):
        keys = range(min(i + 1, nk)) if causal else range(nk)
        w = [math.exp(scale * sum(q[i][c] * k[j][c] for c in range(d))) for j in keys]
        tot = sum(w)
        out.append([sum(w[t] * v[j][c] for t, j in enumerate(keys)) / tot for c in range(d)])
    return np.array(out)


def pin_brute_force_tiny(orc):
    """Exhaustive small-integer inputs on tiny shapes against the literal formula."""
    # every q, k in {-1, 0, 1}^(1x2), {-1,0,1}^(2x1) keys, D = 1 and 2 keys
    vals = (-1.0, 0.0, 1.0)
    v = [[2.0], [-3.0]]
    for q0, k0, k1 in itertools.product(vals, repeat=3):
        q, k = [[q0]], [[k0], [k1]]
        _close(orc.attention(q, k, v, 0.9), _literal(q, k, v, 0.9, False), 1e-14, 1e-14,
               f"tiny q={q0} k=({k0},{k1})")
    rng = _rng(23)
    for nq in range(1, 10):
        for nk in range(1, 10):
            d = 1 + (nq + nk) % 3
            q = rng.integers(-2, 3, (nq, d)).astype(np.float64)
            k = rng.integers(-2, 3, (nk, d)).astype(np.float64)
            v = rng.integers(-4, 5, (nk, d)).astype(np.float64)
            for causal in (False, True):
                want = _literal(q.tolist(), k.tolist(), v.tolist(), 0.5, causal)
                _close(orc.attention(q, k, v, 0.5, causal), want, 1e-13, 1e-13,
                       f"brute {nq}x{nk}x{d} causal={causal}")
                _close(orc.attention_online(q, k, v, 0.5, causal, block=2), want, 1e-13, 1e-13,
                       f"brute online {nq}x{nk}x{d} causal={causal}")


def pin_two_oracles_agree(orc):
    """Two-pass and online forms agree to 1e-12 (relative) for several block sizes."""
    rng = _rng(24)
    for nq, nk, d, causal, sig in ((33, 301, 16, False, 1.0), (130, 130, 8, True, 3.0),
                                   (64, 37, 64, False, 3.0), (200, 260, 4, True, 1.0)):
        q = rng.standard_normal((2, nq, d)) * sig
        k = rng.standard_normal((2, nk, d)) * sig
        v = rng.standard_normal((2, nk, d))
        o2, l2 = orc.attention(q, k, v, 1 / math.sqrt(d), causal, with_lse=True)
        for block in (1, 37, 128):
            o1, l1 = orc.attention_online(q, k, v, 1 / math.sqrt(d), causal, block=block,
                                          with_lse=True)
            _close(o1, o2, 1e-12, 1e-13, f"online vs two-pass block={block}")
            _close(l1, l2, 1e-12, 1e-13, f"online lse block={block}")


def pin_split_and_merge(orc):
    """Splitting the keys anywhere and merging the two states gives the full state."""
    rng = _rng(25)
    q, k, v = rng.standard_normal(6) * 2, rng.standard_normal((50, 6)) * 2, rng.standard_normal((50, 6))
    m, l, o = orc.online_state(q, k, v, 0, 50, 0.5, block=1)
    for cut in (1, 17, 49):
        a = orc.online_state(q, k, v, 0, cut, 0.5, block=4)
        b = orc.online_state(q, k, v, cut, 50, 0.5, block=3)
        mm, ll, oo = orc.merge_state(a, b)
        _close([mm, ll], [m, l], 1e-13, 0, f"merge at {cut}")
        _close(oo, o, 1e-13, 1e-13, f"merge o at {cut}")
    empty = orc.online_state(q, k, v, 5, 5, 0.5)
    mm, ll, oo = orc.merge_state(empty, (m, l, o))
    _close([mm, ll], [m, l], 0, 0, "merge with empty state")


# --- rotary position embedding ------------------------------------------------------------------

def _angles(rows, half, base=10000.0, offset=0):
    """The usual RoPE angles: position p, pair i -> p * base^(-2i/d)."""
    pos = np.arange(offset, offset + rows, dtype=np.float64)[:, None]
    inv = base ** (-np.arange(half, dtype=np.float64) / half)
    return pos * inv[None, :]


def pin_rope_closed_forms(orc):
    """Zero angle is the identity; a quarter turn sends each pair (a, b) to (-b, a); every
    rotation keeps the length of each pair."""
    rng = _rng(31)
    x = rng.standard_normal((5, 8))
    zeros, ones = np.zeros((5, 4)), np.ones((5, 4))
    for form in (0, 1):
        _close(orc.rope(x, ones, zeros, form), x, 0, 0, f"identity form {form}")
        y = orc.rope(x, zeros, ones, form)
        i0 = np.arange(4) if form == 0 else 2 * np.arange(4)
        i1 = i0 + 4 if form == 0 else i0 + 1
        _close(y[:, i0], -x[:, i1], 0, 0, f"quarter turn a, form {form}")
        _close(y[:, i1], x[:, i0], 0, 0, f"quarter turn b, form {form}")
        th = rng.uniform(-7, 7, (5, 4))
        z = orc.rope(x, np.cos(th), np.sin(th), form)
        _close(z[:, i0] ** 2 + z[:, i1] ** 2, x[:, i0] ** 2 + x[:, i1] ** 2, 1e-13, 1e-13,
               f"pair norms form {form}")


def pin_rope_composes(orc):
    """Rotating by t1 then by t2 is rotating by t1 + t2."""
    rng = _rng(32)
    x = rng.standard_normal((6, 10))
    t1, t2 = rng.uniform(-3, 3, (6, 5)), rng.uniform(-3, 3, (6, 5))
    for form in (0, 1):
        two = orc.rope(orc.rope(x, np.cos(t1), np.sin(t1), form), np.cos(t2), np.sin(t2), form)
        one = orc.rope(x, np.cos(t1 + t2), np.sin(t1 + t2), form)
        _close(two, one, 1e-13, 1e-13, f"composition form {form}")


def pin_rope_relative_position(orc):
    """With position-proportional angles, q_m . k_n depends only on m - n: shifting every
    position by the same amount leaves all scores unchanged."""
    rng = _rng(33)
    q, k = rng.standard_normal((7, 16)), rng.standard_normal((9, 16))
    for form in (0, 1):
        s = []
        for off in (0, 37):
            aq, ak = _angles(7, 8, offset=off), _angles(9, 8, offset=off)
            qr = orc.rope(q, np.cos(aq), np.sin(aq), form)
            kr = orc.rope(k, np.cos(ak), np.sin(ak), form)
            s.append(qr @ kr.T)
        _close(s[0], s[1], 1e-10, 1e-10, f"relative position form {form}")


def pin_rope_forms_are_a_permutation(orc):
    """Interleaved pairs on x equal rotate-half on x with its columns reordered so that pair i
    sits at (i, i + d/2)."""
    rng = _rng(34)
    x = rng.standard_normal((4, 12))
    th = rng.uniform(-2, 2, (4, 6))
    perm = np.concatenate([np.arange(0, 12, 2), np.arange(1, 12, 2)])
    pairs = orc.rope(x, np.cos(th), np.sin(th), 1)
    half = orc.rope(x[:, perm], np.cos(th), np.sin(th), 0)
    _close(pairs[:, perm], half, 0, 0, "forms")


# --- backward ------------------------------------------------------------------------------------

def pin_backward_finite_differences(orc):
    """Each gradient element matches the central difference of L = sum(dO * O) computed by the
    oracle's own forward pass."""
    rng = _rng(41)
    for causal, (nq, nk, d) in ((False, (4, 6, 3)), (True, (5, 5, 2)), (True, (3, 7, 3))):
        q, k, v = (rng.standard_normal((n, d)) for n in (nq, nk, nk))
        do = rng.standard_normal((nq, d))
        dq, dk, dv = orc.attention_backward(q, k, v, do, 0.7, causal)
        h = 1e-6

        def loss(qq, kk, vv):
            return float(np.sum(do * orc.attention(qq, kk, vv, 0.7, causal)))

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = xp, xm
                num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                            loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            _close(g, num, 1e-6, 1e-8, f"d{name} causal={causal}")


def pin_backward_constant_values(orc):
    """When every row of V is the same vector, O does not depend on Q or K: dQ = dK = 0, and
    dV distributes dO by the attention weights (uniform when q = 0)."""
    rng = _rng(42)
    q, k = rng.standard_normal((6, 4)), rng.standard_normal((8, 4))
    v = np.repeat(rng.standard_normal((1, 4)), 8, 0)
    do = rng.standard_normal((6, 4))
    for causal in (False, True):
        dq, dk, dv = orc.attention_backward(q, k, v, do, 0.5, causal)
        _close(dq, np.zeros_like(dq), 0, 1e-13, "dq with constant V")
        _close(dk, np.zeros_like(dk), 0, 1e-13, "dk with constant V")
    _, _, dv = orc.attention_backward(np.zeros((6, 4)), k, rng.standard_normal((8, 4)), do, 0.5)
    _close(dv, np.repeat(do.sum(0, keepdims=True) / 8, 8, 0), 1e-13, 1e-13, "dv uniform")


def pin_backward_key_shift_gradient_sums_to_zero(orc):
    """Moving every key by the same vector leaves O unchanged, so the key gradients sum to 0."""
    rng = _rng(43)
    q, k, v = rng.standard_normal((7, 5)), rng.standard_normal((9, 5)), rng.standard_normal((9, 5))
    do = rng.standard_normal((7, 5))
    for causal in (False, True):
        _, dk, _ = orc.attention_backward(q, k, v, do, 0.9, causal)
        _close(dk.sum(0), np.zeros(5), 0, 1e-12, f"sum dk causal={causal}")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(orc) -> list[str]:
    """Run every pin; return the failures as 'name: message' strings."""
    failures = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception as e:  # noqa: BLE001 -- a crash in a planted mistake counts as caught
            failures.append(f"{pin.__name__}: {type(e).__name__}: {e}")
    return failures
