"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError when the oracle disagrees with:

* central finite differences of its own forward (the backward is the exact
  gradient of L = sum(dO * O)),
* the hand-derived 2x2 worked example in ``tests/golden/worked_2x2.json``,
* closed forms of degenerate inputs (K = 0, V = 0, a single key, a single
  query, causal rows with no visible key),
* invariants (sum_j dS_ij = 0, sum_j P_ij = 1, dV = P^T dO, sum_j dK_j = 0,
  sum_j dV_j = sum_i dO_i),
* an independent library forward (scipy softmax + numpy matmul),
* structural reductions (GQA == MHA with repeated K/V, summed over the group;
  varlen == each sequence run alone),
* the extensions reduced to the plain, already pinned problem on other inputs:
  a local window row by row == the unmasked problem on the keys inside the
  band; causal ALiBi == plain causal attention with one extra head-dimension
  column (q gets slope / scale, k gets the key position); seqused == the
  problem cut to the used rows; a (0, 0) window in closed form; a bias
  constant along the keys shifts only LSE; a bias constant along the queries
  is one more head-dimension column again; a bias equal to the ALiBi terms
  equals ALiBi; dBias = dS is the gradient of L by finite differences;
* dropout: the Philox4x32-10 known-answer vectors, the keep rate, t = 0 equal
  to no dropout, O / dV equal to P o (M s) times V / dO with the mask built
  from the generator here, and the backward as the gradient of the dropout
  forward (fixed seed, finite differences);
* a value head dim Dv different from D: finite differences both ways, the
  problem with zero columns padded onto the narrower side (which has one
  head dim again), and the invariants with the two dims apart.

``tests/test_oracle.py`` runs every pin on the real oracle and also on
mutant builds with a planted mistake, each of which must fail at least one
pin.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_2x2.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    inf_a, inf_b = np.isinf(a), np.isinf(b)
    assert np.array_equal(inf_a, inf_b) and np.array_equal(a[inf_a], b[inf_b]), what + ": inf"
    a = np.where(inf_a, 0.0, a)
    b = np.where(inf_b, 0.0, b)
    denom = max(1.0, float(np.max(np.abs(b)))) if b.size else 1.0
    err = float(np.max(np.abs(a - b))) / denom if a.size else 0.0
    assert err <= rtol, "%s: max err %.3e > %.1e" % (what, err, rtol)


def _dense(rng, B, Sq, Sk, Hq, Hkv, D, scale_in=1.0):
    q = rng.standard_normal((B, Sq, Hq, D)) * scale_in
    k = rng.standard_normal((B, Sk, Hkv, D)) * scale_in
    v = rng.standard_normal((B, Sk, Hkv, D))
    do = rng.standard_normal((B, Sq, Hq, D))
    return q, k, v, do


def _fd_check(orc, q, k, v, do, scale, causal, cu_q=None, cu_k=None, h=1e-6, rtol=2e-7, **ext):
    """Backward (own fp64 forward) == central differences of L = sum(dO * O)."""
    dq, dk, dv = orc.backward(q, k, v, do, scale, causal, cu_q=cu_q, cu_k=cu_k, **ext)

    def loss(qq, kk, vv):
        o, _ = orc.forward(qq, kk, vv, scale, causal, cu_q=cu_q, cu_k=cu_k, nthreads=1, **ext)
        return float(np.sum(do * o))

    for X, G, name in ((q, dq, "dq"), (k, dk, "dk"), (v, dv, "dv")):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp = X.copy()
            Xm = X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            pos = {"dq": 0, "dk": 1, "dv": 2}[name]
            args_p[pos] = Xp
            args_m[pos] = Xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        _close(G, num, rtol, "finite differences " + name)


# ----------------------------------------------------------------- pins

def pin_worked_example(orc):
    g = json.load(open(GOLDEN))
    inp = g["inputs"]
    q = np.array(inp["q"]).reshape(1, 2, 1, 1)
    k = np.array(inp["k"]).reshape(1, 2, 1, 1)
    v = np.array(inp["v"]).reshape(1, 2, 1, 1)
    do = np.array(inp["dout"]).reshape(1, 2, 1, 1)
    for key, causal in (("non_causal", False), ("causal", True)):
        e = g[key]
        o, lse = orc.forward(q, k, v, inp["scale"], causal)
        _close(o.ravel(), e["o"], 1e-14, key + " o")
        _close(lse.ravel(), e["lse"], 1e-14, key + " lse")
        P, dS = orc.head_matrices(q, k, v, do, inp["scale"], causal)
        _close(P, e["P"], 1e-14, key + " P")
        _close(dS, e["dS"], 1e-14, key + " dS")
        for given in (False, True):
            kw = dict(o=o, lse=lse) if given else {}
            dq, dk, dv = orc.backward(q, k, v, do, inp["scale"], causal, **kw)
            _close(dq.ravel(), e["dq"], 1e-14, key + " dq")
            _close(dk.ravel(), e["dk"], 1e-14, key + " dk")
            _close(dv.ravel(), e["dv"], 1e-14, key + " dv")


def pin_fd_dense(orc):
    q, k, v, do = _dense(_rng(1), 2, 6, 6, 2, 2, 4)
    _fd_check(orc, q, k, v, do, 0.7, False)


def pin_fd_causal(orc):
    q, k, v, do = _dense(_rng(2), 1, 9, 9, 1, 1, 3)
    _fd_check(orc, q, k, v, do, 0.5, True)


def pin_fd_causal_rect(orc):
    # Sq < Sk and Sq > Sk (the latter has query rows with no visible key)
    for sq, sk, seed in ((5, 8, 3), (8, 5, 4)):
        q, k, v, do = _dense(_rng(seed), 1, sq, sk, 1, 1, 3)
        _fd_check(orc, q, k, v, do, 0.6, True)


def pin_fd_gqa(orc):
    q, k, v, do = _dense(_rng(5), 1, 5, 5, 4, 2, 3)
    _fd_check(orc, q, k, v, do, 0.8, True)


def pin_fd_varlen(orc):
    rng = _rng(6)
    cu_q = np.array([0, 5, 12], dtype=np.int32)
    cu_k = np.array([0, 7, 11], dtype=np.int32)
    q = rng.standard_normal((12, 2, 3))
    k = rng.standard_normal((11, 2, 3))
    v = rng.standard_normal((11, 2, 3))
    do = rng.standard_normal((12, 2, 3))
    _fd_check(orc, q, k, v, do, 0.9, True, cu_q=cu_q, cu_k=cu_k)


def pin_library_forward(orc):
    """O and LSE against scipy's softmax / logsumexp and numpy matmul."""
    from scipy.special import logsumexp, softmax
    for causal, (sq, sk) in ((False, (7, 7)), (True, (7, 7)), (True, (4, 9)), (True, (9, 4))):
        q, k, v, do = _dense(_rng(7 + sq), 1, sq, sk, 2, 1, 5)
        o, lse = orc.forward(q, k, v, 0.45, causal)
        for h in range(2):
            S = 0.45 * q[0, :, h, :] @ k[0, :, 0, :].T
            if causal:
                i = np.arange(sq)[:, None]
                j = np.arange(sk)[None, :]
                S = np.where(j <= i + (sk - sq), S, -np.inf)
            for r in range(sq):
                if np.all(np.isneginf(S[r])):
                    assert np.isneginf(lse[0, h, r]), "row without keys must have LSE -inf"
                    _close(o[0, r, h], np.zeros(5), 0, "row without keys O")
                    continue
                _close(lse[0, h, r], logsumexp(S[r]), 1e-13, "lse vs logsumexp")
                _close(o[0, r, h], softmax(S[r]) @ v[0, :, 0, :], 1e-13, "O vs softmax@V")


def pin_closed_forms(orc):
    rng = _rng(8)
    B, S, H, D, c = 1, 6, 1, 4, 0.3
    q, k, v, do = _dense(rng, B, S, S, H, H, D)
    # K = 0: P uniform -> dV_j = mean_i... = (1/Sk) sum_i dO_i, dQ = 0
    dq, dk, dv = orc.backward(q, np.zeros_like(k), v, do, c, False)
    _close(dq, np.zeros_like(dq), 1e-15, "K=0 dq")
    for j in range(S):
        _close(dv[0, j, 0], do[0, :, 0].sum(0) / S, 1e-13, "K=0 dv")
    # V = 0: dP = 0 and D = 0 -> dS = 0 -> dQ = dK = 0
    dq, dk, dv = orc.backward(q, k, np.zeros_like(v), do, c, False)
    _close(dq, np.zeros_like(dq), 1e-15, "V=0 dq")
    _close(dk, np.zeros_like(dk), 1e-15, "V=0 dk")
    # one key: P = 1, O_i = v_0, dS = 0, dV_0 = sum_i dO_i
    q1, k1, v1, do1 = _dense(rng, 1, 5, 1, 1, 1, D)
    o, lse = orc.forward(q1, k1, v1, c, False)
    for i in range(5):
        _close(o[0, i, 0], v1[0, 0, 0], 1e-14, "one key O")
        _close(lse[0, 0, i], c * q1[0, i, 0] @ k1[0, 0, 0], 1e-14, "one key LSE")
    dq, dk, dv = orc.backward(q1, k1, v1, do1, c, False)
    _close(dq, np.zeros_like(dq), 1e-14, "one key dq")
    _close(dk, np.zeros_like(dk), 1e-14, "one key dk")
    _close(dv[0, 0, 0], do1[0, :, 0].sum(0), 1e-13, "one key dv")
    # causal, Sq == Sk: query 0 sees key 0 only
    o, lse = orc.forward(q, k, v, c, True)
    _close(o[0, 0, 0], v[0, 0, 0], 1e-14, "causal row 0 O")
    _close(lse[0, 0, 0], c * q[0, 0, 0] @ k[0, 0, 0], 1e-14, "causal row 0 LSE")
    # causal, bottom-right: one query against 3 keys sees all of them
    qa, ka, va, doa = _dense(rng, 1, 1, 3, 1, 1, D)
    oc, lc = orc.forward(qa, ka, va, c, True)
    on, ln = orc.forward(qa, ka, va, c, False)
    _close(oc, on, 1e-15, "bottom-right causal Sq=1 == non-causal")
    _close(lc, ln, 1e-15, "bottom-right causal Sq=1 LSE == non-causal")
    # causal, 3 queries against 1 key: only the last query sees it
    qb, kb, vb, dob = _dense(rng, 1, 3, 1, 1, 1, D)
    ob, lb = orc.forward(qb, kb, vb, c, True)
    assert np.isneginf(lb[0, 0, 0]) and np.isneginf(lb[0, 0, 1]), "rows 0,1 see no key"
    _close(ob[0, :2], np.zeros((2, 1, D)), 0, "rows without keys O")
    _close(ob[0, 2, 0], vb[0, 0, 0], 1e-14, "last row sees the key")
    dq, dk, dv = orc.backward(qb, kb, vb, dob, c, True)
    _close(dq[0, :2], np.zeros((2, 1, D)), 0, "rows without keys dq")
    _close(dv[0, 0, 0], dob[0, 2, 0], 1e-14, "dv from the only visible row")


def pin_invariants(orc):
    for causal, (sq, sk) in ((False, (7, 7)), (True, (7, 7)), (True, (5, 9)), (True, (9, 5))):
        q, k, v, do = _dense(_rng(20 + sq), 1, sq, sk, 2, 1, 4)
        c = 0.55
        dq, dk, dv = orc.backward(q, k, v, do, c, causal)
        dv_sum = np.zeros(4)
        do_sum = np.zeros(4)
        for h in range(2):
            P, dS = orc.head_matrices(q, k, v, do, c, causal, h=h)
            has_key = P.sum(1) > 0
            _close(P.sum(1)[has_key], np.ones(has_key.sum()), 1e-14, "sum_j P = 1")
            _close(dS.sum(1), np.zeros(sq), 1e-14, "sum_j dS = 0")
            _close(dq[0, :, h], c * dS @ k[0, :, 0], 1e-13, "dQ = c dS K")
            dv_sum += do[0, has_key, h].sum(0)
        # GQA group of 2 heads shares kv head 0
        P0, dS0 = orc.head_matrices(q, k, v, do, c, causal, h=0)
        P1, dS1 = orc.head_matrices(q, k, v, do, c, causal, h=1)
        _close(dv[0, :, 0], P0.T @ do[0, :, 0] + P1.T @ do[0, :, 1], 1e-13, "dV = P^T dO")
        _close(dk[0, :, 0], c * (dS0.T @ q[0, :, 0] + dS1.T @ q[0, :, 1]), 1e-13, "dK = c dS^T Q")
        _close(dk[0, :, 0].sum(0), np.zeros(4), 1e-13, "sum_j dK_j = 0")
        _close(dv[0, :, 0].sum(0), dv_sum, 1e-13, "sum_j dV_j = sum_i dO_i")


def pin_gqa_equals_expanded(orc):
    rng = _rng(30)
    q, k, v, do = _dense(rng, 2, 6, 6, 4, 2, 3)
    for causal in (False, True):
        dq, dk, dv = orc.backward(q, k, v, do, 0.6, causal)
        ke = np.repeat(k, 2, axis=2)
        ve = np.repeat(v, 2, axis=2)
        dqe, dke, dve = orc.backward(q, ke, ve, do, 0.6, causal)
        _close(dq, dqe, 1e-14, "GQA dq")
        _close(dk, dke[:, :, 0::2] + dke[:, :, 1::2], 1e-14, "GQA dk = group sum")
        _close(dv, dve[:, :, 0::2] + dve[:, :, 1::2], 1e-14, "GQA dv = group sum")


def pin_varlen_equals_dense(orc):
    rng = _rng(31)
    cu_q = np.array([0, 4, 11, 12], dtype=np.int32)
    cu_k = np.array([0, 6, 9, 13], dtype=np.int32)
    q = rng.standard_normal((12, 2, 3))
    k = rng.standard_normal((13, 1, 3))
    v = rng.standard_normal((13, 1, 3))
    do = rng.standard_normal((12, 2, 3))
    for causal in (False, True):
        o, lse = orc.forward(q, k, v, 0.7, causal, cu_q=cu_q, cu_k=cu_k)
        dq, dk, dv = orc.backward(q, k, v, do, 0.7, causal, cu_q=cu_q, cu_k=cu_k)
        for b in range(3):
            qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            sub = [x[None] for x in (q[qs:qe], k[ks:ke], v[ks:ke], do[qs:qe])]
            ob, lb = orc.forward(*sub[:3], 0.7, causal)
            dqb, dkb, dvb = orc.backward(*sub, 0.7, causal)
            _close(o[qs:qe], ob[0], 1e-15, "varlen o")
            _close(lse[:, qs:qe], lb[0], 1e-15, "varlen lse")
            _close(dq[qs:qe], dqb[0], 1e-15, "varlen dq")
            _close(dk[ks:ke], dkb[0], 1e-15, "varlen dk")
            _close(dv[ks:ke], dvb[0], 1e-15, "varlen dv")


def pin_sampled_equals_full(orc):
    q, k, v, do = _dense(_rng(32), 2, 9, 9, 4, 2, 5)
    dq, dk, dv = orc.backward(q, k, v, do, 0.5, True)
    qrows = [(0, 0, 0), (1, 8, 3), (0, 4, 2), (1, 3, 1)]
    krows = [(0, 0, 0), (1, 8, 1), (0, 5, 1), (1, 2, 0)]
    sq, sk, sv = orc.backward_sampled(q, k, v, do, 0.5, True, qrows=qrows, krows=krows)
    for r, (b, s, h) in enumerate(qrows):
        _close(sq[r], dq[b, s, h], 0, "sampled dq")
    for r, (b, s, hk) in enumerate(krows):
        _close(sk[r], dk[b, s, hk], 0, "sampled dk")
        _close(sv[r], dv[b, s, hk], 0, "sampled dv")


def pin_given_forward_consistent(orc):
    q, k, v, do = _dense(_rng(33), 1, 8, 8, 2, 2, 4)
    o, lse = orc.forward(q, k, v, 0.4, True)
    a = orc.backward(q, k, v, do, 0.4, True)
    b = orc.backward(q, k, v, do, 0.4, True, o=o, lse=lse)
    for x, y, n in zip(a, b, ("dq", "dk", "dv")):
        _close(x, y, 1e-14, "given O/LSE " + n)


def pin_preprocess_identity(orc):
    """Dv_i = <dO_i, O_i> equals sum_j P_ij dP_ij (because O_i = sum_j P_ij v_j),
    and the guarded LSE is the forward's LSE with -inf replaced by 0."""
    for causal, (sq, sk) in ((False, (6, 6)), (True, (6, 6)), (True, (8, 5))):
        q, k, v, do = _dense(_rng(50 + sq + sk), 1, sq, sk, 2, 1, 4)
        dvec, lse_g = orc.preprocess(q, k, v, do, 0.65, causal)
        _, lse = orc.forward(q, k, v, 0.65, causal)
        _close(lse_g, np.where(np.isneginf(lse), 0.0, lse), 0, "guarded LSE")
        for h in range(2):
            P, _ = orc.head_matrices(q, k, v, do, 0.65, causal, h=h)
            dP = do[0, :, h] @ v[0, :, 0].T
            _close(dvec[0, h], (P * dP).sum(1), 1e-13, "Dv = sum_j P dP")
        o, _ = orc.forward(q, k, v, 0.65, causal)
        dvec_given, _ = orc.preprocess(q, k, v, do, 0.65, causal, o=o, lse=lse)
        _close(dvec_given, dvec, 1e-14, "Dv with the given O")


def pin_window_rows_equal_unmasked_band(orc):
    """Row i of a windowed problem == the unmasked problem of query i against
    the keys in [i + diag - left, i + diag + right] (cut from the inputs)."""
    rng = _rng(60)
    for (Sq, Sk, wl, wr, causal) in ((24, 24, 3, 2, False), (10, 20, 2, 1, False),
                                     (20, 12, 4, -1, True), (16, 16, -1, 3, False),
                                     (18, 18, 5, 7, True)):
        q, k, v, do = _dense(rng, 1, Sq, Sk, 2, 1, 4)
        o, lse = orc.forward(q, k, v, 0.6, causal, window=(wl, wr))
        diag = Sk - Sq
        for i in range(Sq):
            lo = 0 if wl < 0 else max(0, i + diag - wl)
            hi = Sk - 1 if wr < 0 else min(Sk - 1, i + diag + wr)
            if causal:
                hi = min(hi, i + diag)
            if hi < lo:
                assert np.all(o[0, i] == 0) and np.all(np.isneginf(lse[0, :, i])), "empty band"
                continue
            o1, l1 = orc.forward(q[:, i:i + 1], k[:, lo:hi + 1], v[:, lo:hi + 1], 0.6, False)
            _close(o[0, i], o1[0, 0], 1e-13, "window row O")
            _close(lse[0, :, i], l1[0, :, 0], 1e-13, "window row LSE")


def pin_window_zero_closed_form(orc):
    """Window (0, 0), Sq == Sk: query i sees key i only: O_i = v_i, LSE_i = s_ii,
    dS = 0 so dQ = dK = 0, and dV_j = sum over the group of dO_j."""
    q, k, v, do = _dense(_rng(61), 1, 9, 9, 4, 2, 5)
    o, lse = orc.forward(q, k, v, 0.8, False, window=(0, 0))
    dq, dk, dv = orc.backward(q, k, v, do, 0.8, False, window=(0, 0))
    for h in range(4):
        _close(o[0, :, h], v[0, :, h // 2], 1e-14, "O = v")
        _close(lse[0, h], 0.8 * np.sum(q[0, :, h] * k[0, :, h // 2], axis=1), 1e-14, "LSE = s_ii")
    _close(dq, np.zeros_like(dq), 1e-14, "dQ = 0")
    _close(dk, np.zeros_like(dk), 1e-14, "dK = 0")
    _close(dv[0, :, 0], do[0, :, 0] + do[0, :, 1], 1e-14, "dV = dO summed")
    _close(dv[0, :, 1], do[0, :, 2] + do[0, :, 3], 1e-14, "dV = dO summed")


def pin_fd_window(orc):
    q, k, v, do = _dense(_rng(62), 1, 7, 9, 2, 1, 3)
    _fd_check(orc, q, k, v, do, 0.7, False, window=(2, 1))
    _fd_check(orc, q, k, v, do, 0.7, True, window=(3, -1))


def _augment(q, k, v, do, slopes, scale):
    """q' = [q, slope_h / scale], k' = [k, j], v' = [v, 0], dO' = [dO, 0]:
    scale * <q', k'> = s + slope_h * j, and the extra column of O' is 0."""
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    sl = np.broadcast_to(np.asarray(slopes, dtype=np.float64), (B, Hq))
    qa = np.concatenate([q, np.broadcast_to((sl / scale)[:, None, :, None], (B, Sq, Hq, 1))], 3)
    pos = np.arange(Sk, dtype=np.float64)[None, :, None, None]
    ka = np.concatenate([k, np.broadcast_to(pos, (B, Sk, Hkv, 1))], 3)
    va = np.concatenate([v, np.zeros((B, Sk, Hkv, 1))], 3)
    da = np.concatenate([do, np.zeros((B, Sq, Hq, 1))], 3)
    return tuple(np.ascontiguousarray(x) for x in (qa, ka, va, da))


def pin_alibi_causal_equals_augmented(orc):
    """Causal ALiBi: every visible key has j <= i + diag, so the bias
    -m (i + diag - j) = m j - m (i + diag): plain causal attention on q', k' of
    one more column (O and the gradients equal; LSE shifts by m (i + diag))."""
    rng = _rng(63)
    for (B, Sq, Sk, Hq, Hkv) in ((2, 11, 11, 4, 2), (1, 7, 13, 2, 2)):
        q, k, v, do = _dense(rng, B, Sq, Sk, Hq, Hkv, 4)
        slopes = rng.uniform(0.05, 0.6, size=(B, Hq))
        sc = 0.55
        o, lse = orc.forward(q, k, v, sc, True, alibi=slopes)
        qa, ka, va, da = _augment(q, k, v, do, slopes, sc)
        oa, la = orc.forward(qa, ka, va, sc, True)
        _close(o, oa[..., :4], 1e-13, "ALiBi O")
        _close(oa[..., 4], np.zeros_like(oa[..., 4]), 0, "augmented O column")
        shift = slopes[:, :, None] * (np.arange(Sq) + (Sk - Sq))[None, None, :]
        fin = np.isfinite(la)
        _close(lse[fin], (la - shift)[fin], 1e-12, "ALiBi LSE")
        dq, dk, dv = orc.backward(q, k, v, do, sc, True, alibi=slopes)
        dqa, dka, dva = orc.backward(qa, ka, va, da, sc, True)
        _close(dq, dqa[..., :4], 1e-12, "ALiBi dQ")
        _close(dk, dka[..., :4], 1e-12, "ALiBi dK")
        _close(dv, dva[..., :4], 1e-12, "ALiBi dV")


def pin_alibi_noncausal(orc):
    """Non-causal ALiBi: a single query at the last position sees every key to
    its left (the augmented problem again); with Sq == Sk, reversing the order
    of queries and keys leaves |i - j| unchanged, so the outputs come back
    reversed; the backward is the gradient of its forward (also Sq != Sk);
    slopes 0 give plain attention."""
    rng = _rng(64)
    q, k, v, do = _dense(rng, 1, 1, 10, 2, 1, 3)
    slopes = np.array([0.3, 0.9])
    o, lse = orc.forward(q, k, v, 0.5, False, alibi=slopes)
    qa, ka, va, _ = _augment(q, k, v, do, slopes, 0.5)
    oa, la = orc.forward(qa, ka, va, 0.5, False)
    _close(o, oa[..., :3], 1e-13, "single-query ALiBi O")
    _close(lse, la - slopes[None, :, None] * 9, 1e-12, "single-query ALiBi LSE")
    q, k, v, do = _dense(rng, 1, 11, 11, 2, 2, 3)
    o, lse = orc.forward(q, k, v, 0.5, False, alibi=slopes)
    dq, dk, dv = orc.backward(q, k, v, do, 0.5, False, alibi=slopes)
    r = lambda x: np.ascontiguousarray(x[:, ::-1])
    o2, lse2 = orc.forward(r(q), r(k), r(v), 0.5, False, alibi=slopes)
    dq2, dk2, dv2 = orc.backward(r(q), r(k), r(v), r(do), 0.5, False, alibi=slopes)
    _close(o2, r(o), 1e-13, "reversed O")
    _close(lse2, np.ascontiguousarray(lse[:, :, ::-1]), 1e-13, "reversed LSE")
    for a, b, n in ((dq2, dq, "dQ"), (dk2, dk, "dK"), (dv2, dv, "dV")):
        _close(a, r(b), 1e-12, "reversed " + n)
    o0, _ = orc.forward(q, k, v, 0.5, False, alibi=np.zeros(2))
    op, _ = orc.forward(q, k, v, 0.5, False)
    _close(o0, op, 0, "zero slopes")
    _fd_check(orc, q[:, :5], k[:, :7], v[:, :7], do[:, :5], 0.5, False, alibi=slopes)


def pin_seqused_equals_cut(orc):
    """seqused == the problem cut to the used rows (dense and varlen); rows past
    the used lengths stay zero."""
    rng = _rng(65)
    q, k, v, do = _dense(rng, 2, 20, 20, 2, 1, 4)
    uq, uk = np.array([12, 20]), np.array([15, 7])
    for causal in (False, True):
        ext = dict(seqused_q=uq, seqused_k=uk, window=(5, -1) if causal else None)
        o, lse = orc.forward(q, k, v, 0.6, causal, **ext)
        dq, dk, dv = orc.backward(q, k, v, do, 0.6, causal, **ext)
        w = dict(window=ext["window"])
        for b in range(2):
            lq, lk = uq[b], uk[b]
            sl = slice(b, b + 1)
            o1, l1 = orc.forward(q[sl, :lq], k[sl, :lk], v[sl, :lk], 0.6, causal, **w)
            d1 = orc.backward(q[sl, :lq], k[sl, :lk], v[sl, :lk], do[sl, :lq], 0.6, causal, **w)
            _close(o[sl, :lq], o1, 1e-14, "seqused O")
            _close(lse[sl, :, :lq], l1, 1e-14, "seqused LSE")
            _close(dq[sl, :lq], d1[0], 1e-14, "seqused dQ")
            _close(dk[sl, :lk], d1[1], 1e-14, "seqused dK")
            _close(dv[sl, :lk], d1[2], 1e-14, "seqused dV")
            for t, n in ((o[sl, lq:], "O"), (dq[sl, lq:], "dQ"), (dk[sl, lk:], "dK"),
                         (dv[sl, lk:], "dV")):
                assert np.all(t == 0), "rows past seqused: " + n
    # varlen: packed sequences with used prefixes
    cu = np.array([0, 9, 21, 30], dtype=np.int32)
    qv = rng.standard_normal((30, 2, 4))
    kv = rng.standard_normal((30, 1, 4))
    vv = rng.standard_normal((30, 1, 4))
    uq, uk = np.array([9, 5, 0]), np.array([4, 12, 6])
    o, lse = orc.forward(qv, kv, vv, 0.6, True, cu_q=cu, cu_k=cu, seqused_q=uq, seqused_k=uk)
    for b in range(3):
        if uq[b] == 0:
            continue
        a, c = cu[b], cu[b]
        o1, l1 = orc.forward(qv[None, a:a + uq[b]], kv[None, c:c + uk[b]], vv[None, c:c + uk[b]],
                             0.6, True)
        _close(o[a:a + uq[b]], o1[0], 1e-14, "varlen seqused O")
        _close(lse[:, a:a + uq[b]], l1[0], 1e-14, "varlen seqused LSE")


def pin_bias_key_column_equals_augmented(orc):
    """bias_ij = u_j (per head): plain attention on q' = [q, 1/scale],
    k' = [k, u_j], v' = [v, 0], dO' = [dO, 0] (G = 1 so k' is per head);
    the column sums of dBias = dS are dK'[:, D] (= sum_i dS_ij)."""
    rng = _rng(70)
    for causal, (Sq, Sk) in ((False, (9, 13)), (True, (12, 12)), (True, (7, 11))):
        B, H, D, sc = 2, 2, 3, 0.45
        q, k, v, do = _dense(rng, B, Sq, Sk, H, H, D)
        u = rng.standard_normal((B, H, Sk))
        bias = np.broadcast_to(u[:, :, None, :], (B, H, Sq, Sk)).copy()
        o, lse = orc.forward(q, k, v, sc, causal, bias=bias)
        dq, dk, dv = orc.backward(q, k, v, do, sc, causal, bias=bias)
        qa = np.concatenate([q, np.full((B, Sq, H, 1), 1.0 / sc)], 3)
        ka = np.concatenate([k, u.transpose(0, 2, 1)[..., None]], 3)
        va = np.concatenate([v, np.zeros((B, Sk, H, 1))], 3)
        da = np.concatenate([do, np.zeros((B, Sq, H, 1))], 3)
        oa, la = orc.forward(qa, ka, va, sc, causal)
        dqa, dka, dva = orc.backward(qa, ka, va, da, sc, causal)
        _close(o, oa[..., :D], 1e-13, "key bias O")
        _close(lse, la, 1e-13, "key bias LSE")
        _close(dq, dqa[..., :D], 1e-12, "key bias dQ")
        _close(dk, dka[..., :D], 1e-12, "key bias dK")
        _close(dv, dva[..., :D], 1e-12, "key bias dV")
        for b in range(B):
            for h in range(H):
                _, dS = orc.head_matrices(q, k, v, do, sc, causal, b=b, h=h, bias=bias)
                _close(dS.sum(0), dka[b, :, h, D], 1e-12, "column sums of dBias")


def pin_bias_query_row_shifts_lse(orc):
    """bias_ij = c_i (constant along the keys) leaves P, O and the gradients
    unchanged and adds c_i to LSE; a [1, Hq, ...] bias broadcasts over the batch."""
    rng = _rng(71)
    q, k, v, do = _dense(rng, 2, 10, 14, 4, 2, 3)
    c = rng.standard_normal((1, 4, 10))
    bias = np.broadcast_to(c[..., None], (1, 4, 10, 14)).copy()
    for causal in (False, True):
        o, lse = orc.forward(q, k, v, 0.6, causal, bias=bias)
        op, lp = orc.forward(q, k, v, 0.6, causal)
        _close(o, op, 1e-13, "row bias O")
        fin = np.isfinite(lp)
        _close(lse[fin], (lp + c)[fin], 1e-13, "row bias LSE")
        g = orc.backward(q, k, v, do, 0.6, causal, bias=bias)
        gp = orc.backward(q, k, v, do, 0.6, causal)
        for a, b_, n in zip(g, gp, ("dQ", "dK", "dV")):
            _close(a, b_, 1e-12, "row bias " + n)


def pin_bias_equals_alibi(orc):
    """A bias holding -slope_h |i + (Lk - Lq) - j| gives what the ALiBi option
    gives (forward and backward), and a [B, Hq] bias stack equals the batch
    broadcast of a [1, Hq] one where the sequences' biases agree."""
    rng = _rng(72)
    for causal, (Sq, Sk) in ((False, (8, 12)), (True, (12, 9))):
        q, k, v, do = _dense(rng, 2, Sq, Sk, 2, 1, 4)
        sl = np.array([0.3, 0.8])
        i = np.arange(Sq)[:, None] + (Sk - Sq)
        j = np.arange(Sk)[None, :]
        bias1 = (-sl[:, None, None] * np.abs(i - j)[None])[None]
        bias2 = np.concatenate([bias1, bias1], 0)
        ref = orc.forward(q, k, v, 0.5, causal, alibi=sl)
        gref = orc.backward(q, k, v, do, 0.5, causal, alibi=sl)
        for bias in (bias1, bias2):
            o, lse = orc.forward(q, k, v, 0.5, causal, bias=bias)
            _close(o, ref[0], 1e-13, "bias == ALiBi O")
            fin = np.isfinite(ref[1])
            _close(lse[fin], ref[1][fin], 1e-13, "bias == ALiBi LSE")
            for a, b_, n in zip(orc.backward(q, k, v, do, 0.5, causal, bias=bias), gref,
                                ("dQ", "dK", "dV")):
                _close(a, b_, 1e-12, "bias == ALiBi " + n)


def pin_fd_bias(orc):
    """dBias = dS (head_matrices) equals central differences of L = sum(dO * O)
    in each bias entry; dQ, dK, dV with a bias are the gradients of its forward."""
    rng = _rng(73)
    q, k, v, do = _dense(rng, 1, 5, 6, 2, 1, 3)
    bias = rng.standard_normal((1, 2, 5, 6))
    for causal in (False, True):
        h = 1e-6
        num = np.zeros_like(bias)
        for idx in np.ndindex(bias.shape):
            bp, bm = bias.copy(), bias.copy()
            bp[idx] += h
            bm[idx] -= h
            lp = np.sum(do * orc.forward(q, k, v, 0.7, causal, nthreads=1, bias=bp)[0])
            lm = np.sum(do * orc.forward(q, k, v, 0.7, causal, nthreads=1, bias=bm)[0])
            num[idx] = (lp - lm) / (2 * h)
        for hh in range(2):
            _, dS = orc.head_matrices(q, k, v, do, 0.7, causal, h=hh, bias=bias)
            _close(dS, num[0, hh], 2e-7, "dBias by finite differences")
        _fd_check(orc, q, k, v, do, 0.7, causal, bias=bias)


# Known-answer vectors of Philox4x32-10 published with the Random123 library
# (Salmon et al., SC 2011): (counter, key) -> output words.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def pin_philox_known_answers(orc):
    for ctr, key, want in PHILOX_KAT:
        assert tuple(orc.philox(ctr, key)) == want, ("philox", ctr, key)


def _mask_here(orc, b, h, Hq, lq, lk, t, seed, off):
    """M * s of one head problem, built from the generator: byte j % 4 of word
    (j / 4) % 4 of Philox(counter (j / 16, i, b Hq + h, off), key (seed))."""
    F = np.zeros((lq, lk))
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for i in range(lq):
        for j0 in range(0, lk, 16):
            out = orc.philox((j0 >> 4, i, b * Hq + h, off), key)
            for j in range(j0, min(lk, j0 + 16)):
                byte = (out[(j >> 2) & 3] >> (8 * (j & 3))) & 0xFF
                F[i, j] = 0.0 if byte < t else 256.0 / (256 - t)
    return F


def pin_dropout_mask_and_rate(orc):
    """The oracle's mask is the generator's (above); the kept fraction is
    1 - t / 256 within 5 standard deviations; t = 0 keeps everything."""
    seed, off = 0x123456789ABCDEF0, 7
    F = orc.dropout_factors(2, 40, 70, 3, 1, 8, b=1, h=2, dropout=(77, seed, off))
    _close(F, _mask_here(orc, 1, 2, 3, 40, 70, 77, seed, off), 0, "dropout mask")
    big = orc.dropout_factors(1, 256, 256, 1, 1, 8, b=0, h=0, dropout=(64, seed, off))
    kept = float(np.mean(big > 0))
    sd = np.sqrt(0.75 * 0.25 / big.size)
    assert abs(kept - 0.75) < 5 * sd, ("keep rate", kept)
    _close(big[big > 0], np.full(int(np.sum(big > 0)), 256.0 / 192), 0, "keep scale")
    none = orc.dropout_factors(1, 16, 16, 1, 1, 8, b=0, h=0, dropout=(0, seed, off))
    _close(none, np.ones_like(none), 0, "t = 0")


def pin_dropout_outputs(orc):
    """O = (P o F) V and dV = (P o F)^T dO with F = M s of the mask built here;
    t = 0 equals no dropout; the backward is the gradient of its forward."""
    rng = _rng(80)
    q, k, v, do = _dense(rng, 2, 9, 11, 2, 1, 3)
    drop = (90, 0xDEADBEEF12345678, 3)
    for causal in (False, True):
        o, lse = orc.forward(q, k, v, 0.6, causal, dropout=drop)
        _, lp = orc.forward(q, k, v, 0.6, causal)
        fin = np.isfinite(lp)
        _close(lse[fin], lp[fin], 0, "dropout leaves LSE")
        dq, dk, dv = orc.backward(q, k, v, do, 0.6, causal, dropout=drop)
        dv_here = np.zeros_like(dv)
        for b in range(2):
            for h in range(2):
                P, _ = orc.head_matrices(q, k, v, do, 0.6, causal, b=b, h=h)
                F = _mask_here(orc, b, h, 2, 9, 11, drop[0], drop[1], drop[2])
                _close(o[b, :, h], (P * F) @ v[b, :, 0], 1e-13, "dropout O")
                dv_here[b, :, 0] += (P * F).T @ do[b, :, h]
        _close(dv, dv_here, 1e-13, "dropout dV")
        z = orc.backward(q, k, v, do, 0.6, causal, dropout=(0, 5, 5))
        for a, b_, n in zip(z, orc.backward(q, k, v, do, 0.6, causal), ("dQ", "dK", "dV")):
            _close(a, b_, 0, "t = 0 " + n)
        _fd_check(orc, q[:1, :5], k[:1, :6], v[:1, :6], do[:1, :5], 0.6, causal, dropout=drop)


def _dense_dv(rng, B, Sq, Sk, Hq, Hkv, D, Dv):
    q = rng.standard_normal((B, Sq, Hq, D))
    k = rng.standard_normal((B, Sk, Hkv, D))
    v = rng.standard_normal((B, Sk, Hkv, Dv))
    do = rng.standard_normal((B, Sq, Hq, Dv))
    return q, k, v, do


def pin_fd_value_dim(orc):
    """A value head dim Dv different from the query / key dim D (both
    directions; causal GQA, rectangular causal, varlen): the backward is the
    gradient of L = sum(dO * O) by central differences."""
    for (D, Dv), causal, shape in (((5, 3), True, (1, 6, 6, 2, 1)), ((3, 5), True, (1, 5, 7, 2, 2)),
                                   ((4, 2), False, (2, 4, 5, 2, 1))):
        q, k, v, do = _dense_dv(_rng(90 + D), *shape, D, Dv)
        _fd_check(orc, q, k, v, do, 0.7, causal)
    rng = _rng(95)
    cu_q = np.array([0, 4, 9], dtype=np.int32)
    cu_k = np.array([0, 6, 9], dtype=np.int32)
    q = rng.standard_normal((9, 2, 4))
    k = rng.standard_normal((9, 1, 4))
    v = rng.standard_normal((9, 1, 2))
    do = rng.standard_normal((9, 2, 2))
    _fd_check(orc, q, k, v, do, 0.8, True, cu_q=cu_q, cu_k=cu_k)


def pin_value_dim_equals_zero_padded(orc):
    """Dv < D: V and dO padded with zero columns to D give the same dQ, dK and
    O, LSE, and a dV whose extra columns are zero.  Dv > D: Q and K padded
    with zero columns to Dv leave every score unchanged, so the padded problem
    gives the same O, LSE, dV and a dQ / dK with zero extra columns.  The
    padded problems have one head dim, pinned by every other pin."""
    for causal in (False, True):
        q, k, v, do = _dense_dv(_rng(97), 2, 7, 9, 4, 2, 6, 3)
        zpad = lambda a, n: np.concatenate([a, np.zeros(a.shape[:-1] + (n,))], axis=-1)
        o, lse = orc.forward(q, k, v, 0.5, causal)
        op, lsep = orc.forward(q, k, zpad(v, 3), 0.5, causal)
        _close(o, op[..., :3], 1e-14, "O, zero-padded V")
        _close(lse, lsep, 1e-14, "LSE, zero-padded V")
        g = orc.backward(q, k, v, do, 0.5, causal)
        gp = orc.backward(q, k, zpad(v, 3), zpad(do, 3), 0.5, causal)
        _close(g[0], gp[0], 1e-13, "dQ, zero-padded V / dO")
        _close(g[1], gp[1], 1e-13, "dK, zero-padded V / dO")
        _close(g[2], gp[2][..., :3], 1e-13, "dV, zero-padded V / dO")
        _close(gp[2][..., 3:], np.zeros_like(gp[2][..., 3:]), 0, "dV padding")
        q2, k2, v2, do2 = _dense_dv(_rng(98), 1, 8, 8, 2, 1, 2, 5)
        o2, lse2 = orc.forward(q2, k2, v2, 0.5, causal)
        o2p, lse2p = orc.forward(zpad(q2, 3), zpad(k2, 3), v2, 0.5, causal)
        _close(o2, o2p, 1e-14, "O, zero-padded Q / K")
        _close(lse2, lse2p, 1e-14, "LSE, zero-padded Q / K")
        h = orc.backward(q2, k2, v2, do2, 0.5, causal)
        hp = orc.backward(zpad(q2, 3), zpad(k2, 3), v2, do2, 0.5, causal)
        _close(h[0], hp[0][..., :2], 1e-13, "dQ, zero-padded Q / K")
        _close(h[1], hp[1][..., :2], 1e-13, "dK, zero-padded Q / K")
        _close(h[2], hp[2], 1e-13, "dV, zero-padded Q / K")
        _close(hp[0][..., 2:], np.zeros_like(hp[0][..., 2:]), 0, "dQ padding")
        _close(hp[1][..., 2:], np.zeros_like(hp[1][..., 2:]), 0, "dK padding")


def pin_value_dim_invariants(orc):
    """dV = P^T dO, dK = c dS^T Q, dQ = c dS K and Dv_i = <dO_i, O_i> with
    Dv != D, against P and dS from the head matrices; the sampled rows equal
    the full backward."""
    c = 0.6
    q, k, v, do = _dense_dv(_rng(99), 1, 9, 9, 2, 1, 5, 3)
    o, lse = orc.forward(q, k, v, c, True)
    dq, dk, dv = orc.backward(q, k, v, do, c, True)
    Ps = [orc.head_matrices(q, k, v, do, c, True, h=h) for h in range(2)]
    _close(dv[0, :, 0], sum(P.T @ do[0, :, h] for h, (P, _) in enumerate(Ps)), 1e-13, "dV = P^T dO")
    _close(dk[0, :, 0], c * sum(dS.T @ q[0, :, h] for h, (_, dS) in enumerate(Ps)), 1e-13,
           "dK = c dS^T Q")
    for h, (P, dS) in enumerate(Ps):
        _close(dq[0, :, h], c * dS @ k[0, :, 0], 1e-13, "dQ = c dS K")
    dvec, _ = orc.preprocess(q, k, v, do, c, True, o=o, lse=lse)
    _close(dvec[0], np.einsum("shd,shd->hs", do[0], o[0]), 1e-13, "Dv = <dO, O>")
    qr = [(0, 3, 1), (0, 8, 0)]
    kr = [(0, 2, 0), (0, 7, 0)]
    sq, sk, sv = orc.backward_sampled(q, k, v, do, c, True, qrows=qr, krows=kr)
    for r, (b, s_, h) in enumerate(qr):
        _close(sq[r], dq[b, s_, h], 0, "sampled dQ")
    for r, (b, s_, hk) in enumerate(kr):
        _close(sk[r], dk[b, s_, hk], 0, "sampled dK")
        _close(sv[r], dv[b, s_, hk], 0, "sampled dV")


ALL_PINS = [pin_fd_value_dim, pin_value_dim_equals_zero_padded, pin_value_dim_invariants,
    pin_preprocess_identity, pin_window_rows_equal_unmasked_band,
    pin_philox_known_answers, pin_dropout_mask_and_rate, pin_dropout_outputs,
    pin_bias_key_column_equals_augmented, pin_bias_query_row_shifts_lse, pin_bias_equals_alibi,
    pin_fd_bias,
    pin_window_zero_closed_form, pin_fd_window, pin_alibi_causal_equals_augmented,
    pin_alibi_noncausal, pin_seqused_equals_cut,
    pin_worked_example, pin_fd_dense, pin_fd_causal, pin_fd_causal_rect, pin_fd_gqa,
    pin_fd_varlen, pin_library_forward, pin_closed_forms, pin_invariants,
    pin_gqa_equals_expanded, pin_varlen_equals_dense, pin_sampled_equals_full,
    pin_given_forward_consistent,
]


def run_all(orc):
    """Runs every pin; returns the names of the pins that failed."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


if __name__ == "__main__":  # used by the mutation test: python oracle_pins.py <libpath>
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import Oracle
    print(json.dumps(run_all(Oracle(sys.argv[1]))))
