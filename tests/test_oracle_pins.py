"""Pins for the CPU oracle: every check here is independent of the oracle's
own code (closed forms, a hand-derived worked example, library routines,
finite differences, identities the pages state), chosen so that a dropped
term, a wrong sign, a wrong index or a transposed operand in the oracle fails
at least one of them.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from online_softmax_05_gb300.inputs import make_inputs, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


# --- online softmax ("Lab 06", section 2) ----------------------------------

@pytest.mark.parametrize("block", [1, 7, 11, 16, 32, 1000, 5000])
def test_online_softmax_matches_logsumexp(block):
    x = rng(1).normal(size=1000) * 5.0
    m, l = oracle.online_softmax_stats(x, block)
    assert m == np.max(x)
    assert abs((m + math.log(l)) - scipy.special.logsumexp(x)) < 1e-12


@pytest.mark.parametrize("block", [1, 3, 7, 16])
def test_online_softmax_growing_max(block):
    # the running max jumps from -40 to 1000 part-way through the row
    x = np.concatenate([np.full(20, -40.0), rng(2).normal(size=13), [1000.0], rng(3).normal(size=9)])
    m, l = oracle.online_softmax_stats(x, block)
    assert np.isfinite(l) and l >= 1.0
    assert m == 1000.0
    assert abs((m + math.log(l)) - scipy.special.logsumexp(x)) < 1e-12


def test_online_softmax_two_pass_equivalence():
    # online (m, l) equals the two-pass result: max first, then sum of exp
    x = rng(4).normal(size=257) * 30.0
    m2 = np.max(x)
    l2 = np.sum(np.exp(x - m2))
    for block in (7, 11, 16, 32):
        m, l = oracle.online_softmax_stats(x, block)
        assert m == m2
        assert abs(l - l2) <= 1e-12 * l2


# --- hand-derived worked example (tests/golden/two_key_closed_form.json) ---

def test_two_key_closed_form():
    with open(os.path.join(GOLDEN, "two_key_closed_form.json")) as f:
        fx = json.load(f)
    for c in fx["cases"]:
        q, k, v, do = (np.array(c[n]) for n in ("q", "k", "v", "do"))
        o, lse = oracle.attn_fwd(q[None], k[None], v[None], c["scale"], c["causal"])
        np.testing.assert_allclose(o[0], c["o"], rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(lse[0], c["lse"], rtol=0, atol=1e-14, err_msg=c["name"])
        dq, dk, dv, dvec = oracle.attn_bwd(q[None], k[None], v[None], do[None], c["scale"], c["causal"])
        np.testing.assert_allclose(dq[0], c["dq"], rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(dk[0], c["dk"], rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(dv[0], c["dv"], rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(dvec[0], c["dvec"], rtol=0, atol=1e-14, err_msg=c["name"])


# --- forward ---------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_probs_rows_sum_to_one_and_mask(causal):
    T, D = 53, 8
    q, k = rng(5).normal(size=(T, D)), rng(6).normal(size=(T, D))
    P = oracle.attn_probs(q, k, 0.7, causal)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()
    if causal:
        assert (P[np.triu_indices(T, 1)] == 0.0).all()
        assert (P[np.tril_indices(T)] > 0.0).all()
    else:
        assert (P > 0).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale", [0.125, 1.0, -0.3])
def test_lse_matches_direct_logsumexp(causal, scale):
    # LSE_i = log sum_j exp(scale q_i.k_j) over visible j, by numpy matmul + scipy logsumexp
    T, D = 41, 16
    q, k, v = (rng(s).normal(size=(2, T, D)) for s in (7, 8, 9))
    o, lse = oracle.attn_fwd(q, k, v, scale, causal)
    for h in range(2):
        S = scale * (q[h] @ k[h].T)
        if causal:
            S = np.where(np.tril(np.ones((T, T), bool)), S, -np.inf)
        np.testing.assert_allclose(lse[h], scipy.special.logsumexp(S, axis=1), rtol=0, atol=1e-12)
        P = scipy.special.softmax(S, axis=1)
        np.testing.assert_allclose(o[h], P @ v[h], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean_of_visible_v(causal):
    # Q = 0: every visible score is 0, so O_i = mean of V over visible keys, LSE_i = log(#visible)
    T, D = 37, 5
    q = np.zeros((T, D))
    k, v = rng(10).normal(size=(T, D)), rng(11).normal(size=(T, D))
    o, lse = oracle.attn_fwd(q[None], k[None], v[None], 0.5, causal)
    for i in range(T):
        n = i + 1 if causal else T
        np.testing.assert_allclose(o[0, i], v[:n].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[0, i] - math.log(n)) < 1e-13


def test_causal_row_zero_returns_v0():
    T, D = 19, 7
    q, k, v = (rng(s).normal(size=(T, D)) * 3 for s in (12, 13, 14))
    o, lse = oracle.attn_fwd(q[None], k[None], v[None], 0.4, True)
    np.testing.assert_array_equal(o[0, 0], v[0])
    assert abs(lse[0, 0] - 0.4 * float(q[0] @ k[0])) < 1e-13


def test_permuting_keys_noncausal_is_invariant():
    # non-causal attention is invariant under a joint permutation of K and V rows
    T, D = 29, 6
    q, k, v = (rng(s).normal(size=(T, D)) for s in (15, 16, 17))
    perm = rng(18).permutation(T)
    o1, l1 = oracle.attn_fwd(q[None], k[None], v[None], 0.9, False)
    o2, l2 = oracle.attn_fwd(q[None], k[perm][None], v[perm][None], 0.9, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("T,bq,bk", [(33, 7, 11), (37, 16, 32), (64, 32, 16), (40, 7, 7), (1, 7, 11), (100, 11, 7)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_recurrence_equals_naive(T, bq, bk, causal):
    # the tiled (m, l, acc) recurrence with block sizes that do not divide T equals the definition
    D = 8
    q, k, v = (rng(s).normal(size=(T, D)) * 2 for s in (19, 20, 21))
    o1, l1 = oracle.attn_fwd(q[None], k[None], v[None], 0.6, causal)
    o2, l2 = oracle.flash_fwd_tiled(q, k, v, 0.6, causal, bq, bk)
    np.testing.assert_allclose(o2, o1[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1[0], rtol=0, atol=1e-12)


def test_tiled_recurrence_large_logits():
    # the max grows by hundreds between key tiles: the rescale must stay exact and finite
    T, D = 48, 4
    q = rng(22).normal(size=(T, D))
    k = rng(23).normal(size=(T, D)) * np.linspace(0.1, 200, T)[:, None]
    v = rng(24).normal(size=(T, D))
    o1, l1 = oracle.attn_fwd(q[None], k[None], v[None], 1.0, False)
    o2, l2 = oracle.flash_fwd_tiled(q, k, v, 1.0, False, 8, 8)
    assert np.isfinite(o2).all() and np.isfinite(l2).all()
    np.testing.assert_allclose(o2, o1[0], rtol=0, atol=1e-11)
    np.testing.assert_allclose(l2, l1[0], rtol=1e-13, atol=0)


def test_rows_variant_matches_full():
    T, D = 70, 8
    q, k, v = (rng(s).normal(size=(T, D)) for s in (25, 26, 27))
    rows = [0, 1, 17, 69]
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q[None], k[None], v[None], 0.3, causal)
        o_r, l_r = oracle.attn_fwd_rows(q, k, v, 0.3, causal, rows)
        np.testing.assert_array_equal(o_r, o[0, rows])
        np.testing.assert_array_equal(l_r, lse[0, rows])


# --- backward ("Lab 06", section 4) ----------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rowsum_identity(causal):
    # D_i = sum_j P_ij dP_ij (oracle, by definition) equals rowsum(dO o O)
    T, D = 45, 12
    q, k, v, do = (rng(s).normal(size=(2, T, D)) for s in (28, 29, 30, 31))
    o, _ = oracle.attn_fwd(q, k, v, 0.25, causal)
    _, _, _, dvec = oracle.attn_bwd(q, k, v, do, 0.25, causal)
    np.testing.assert_allclose(dvec, (do * o).sum(axis=-1), rtol=0, atol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T,D", [(1, 3), (5, 2), (9, 4)])
def test_finite_difference_gradients(causal, T, D):
    # L = sum(dO o O); central differences with h = 1e-6, relative error < 1e-6
    q, k, v, do = (rng(s).normal(size=(1, T, D)) for s in (32, 33, 34, 35))
    scale = 0.8
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]})
                       - loss(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * h)
        denom = max(np.abs(g).max(), 1e-3)
        assert np.abs(fd - g).max() / denom < 1e-6, name


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_float64(causal):
    # the analytic gradients equal autograd through softmax(QK^T scale) V in float64
    T, D = 37, 16
    q, k, v, do = (torch.from_numpy(rng(s).normal(size=(3, T, D))) for s in (36, 37, 38, 39))
    scale = 0.25
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    S = scale * qt @ kt.transpose(-1, -2)
    if causal:
        S = S.masked_fill(~torch.ones(T, T, dtype=torch.bool).tril(), float("-inf"))
    O = torch.softmax(S, dim=-1) @ vt
    O.backward(do)
    dq, dk, dv, _ = oracle.attn_bwd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), scale, causal)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.attn_fwd(q.numpy(), k.numpy(), v.numpy(), scale, causal)[0],
                               O.detach().numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_rows_variant_matches_full(causal):
    T, D = 66, 8
    q, k, v, do = (rng(s).normal(size=(T, D)) for s in (40, 41, 42, 43))
    dq, dk, dv, dvec = oracle.attn_bwd(q[None], k[None], v[None], do[None], 0.35, causal)
    _, lse = oracle.attn_fwd(q[None], k[None], v[None], 0.35, causal)
    rq, rk = [0, 5, 64, 65], [0, 1, 33, 65]
    dq_r, dk_r, dv_r, lse_r, dvec_r = oracle.attn_bwd_rows(q, k, v, do, 0.35, causal, rq, rk)
    np.testing.assert_allclose(dq_r, dq[0, rq], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk_r, dk[0, rk], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv_r, dv[0, rk], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_r, lse[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dvec_r, dvec[0], rtol=0, atol=1e-12)


def test_oracle_on_generated_bf16_inputs_is_finite():
    # the seeded bf16 inputs of the large-logit recipe stay finite through the oracle
    q, k, v, do = make_inputs(1, 2, 64, 16, seed=0, qk_std=4.0, big_row_frac=0.05, big_row_mult=10.0)
    q, k, v, do = (to_f64(t) for t in (q, k, v, do))
    o, lse = oracle.attn_fwd(q, k, v, 0.25, False)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, 0.25, False)
    for a in (o, lse, dq, dk, dv):
        assert np.isfinite(a).all()


# --- queries attending to a longer key sequence (decoding) -------------------

def test_cross_equals_square_when_lengths_match():
    T, D = 31, 8
    q, k, v = (rng(s).normal(size=(2, T, D)) for s in (50, 51, 52))
    o1, l1 = oracle.attn_fwd(q, k, v, 0.4, False)
    o2, l2 = oracle.attn_fwd_cross(q, k, v, 0.4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("Tq,Tk", [(1, 1), (1, 97), (3, 40), (8, 5)])
def test_cross_matches_library_softmax(Tq, Tk):
    D = 6
    q, k, v = rng(53).normal(size=(2, Tq, D)), rng(54).normal(size=(2, Tk, D)), rng(55).normal(size=(2, Tk, D))
    o, lse = oracle.attn_fwd_cross(q, k, v, 0.7)
    for h in range(2):
        S = 0.7 * (q[h] @ k[h].T)
        np.testing.assert_allclose(lse[h], scipy.special.logsumexp(S, axis=1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(o[h], scipy.special.softmax(S, axis=1) @ v[h], rtol=0, atol=1e-12)


def test_cross_uniform_scores_and_single_key():
    # Q = 0: O = mean of all V rows, LSE = log Tk; one key: O = that V row, LSE = its score
    Tq, Tk, D = 2, 50, 4
    k, v = rng(56).normal(size=(1, Tk, D)), rng(57).normal(size=(1, Tk, D))
    o, lse = oracle.attn_fwd_cross(np.zeros((1, Tq, D)), k, v, 1.3)
    np.testing.assert_allclose(o[0], np.broadcast_to(v[0].mean(axis=0), (Tq, D)), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(Tk), rtol=0, atol=1e-13)
    q = rng(58).normal(size=(1, Tq, D))
    o, lse = oracle.attn_fwd_cross(q, k[:, :1], v[:, :1], 1.3)
    np.testing.assert_array_equal(o[0], np.broadcast_to(v[0, 0], (Tq, D)))
    np.testing.assert_allclose(lse[0], 1.3 * (q[0] @ k[0, 0]), rtol=0, atol=1e-13)


# --- grouped-query attention -------------------------------------------------

def test_gqa_group_of_one_is_plain_attention():
    q, k, v, do = (rng(s).normal(size=(1, 3, 17, 4)) for s in (60, 61, 62, 63))
    np.testing.assert_array_equal(oracle.attn_fwd_gqa(q, k, v, 0.5, True)[0], oracle.attn_fwd(q, k, v, 0.5, True)[0])
    for a, b in zip(oracle.attn_bwd_gqa(q, k, v, do, 0.5, True), oracle.attn_bwd(q, k, v, do, 0.5, True)):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_finite_difference_of_shared_keys(causal):
    # L = sum over all query heads of dO o O; dK, dV of a shared head collect every head of its group
    B, Hq, Hkv, T, D = 1, 4, 2, 5, 3
    q, do = rng(64).normal(size=(B, Hq, T, D)), rng(65).normal(size=(B, Hq, T, D))
    k, v = rng(66).normal(size=(B, Hkv, T, D)), rng(67).normal(size=(B, Hkv, T, D))
    scale = 0.9
    _, dk, dv, _ = oracle.attn_bwd_gqa(q, k, v, do, scale, causal)

    def loss(kk, vv):
        return float((oracle.attn_fwd_gqa(q, kk, vv, scale, causal)[0] * do).sum())

    h = 1e-6
    for g, x, is_k in ((dk, k, True), (dv, v, False)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            fd[idx] = ((loss(xp, v) - loss(xm, v)) if is_k else (loss(k, xp) - loss(k, xm))) / (2 * h)
        assert np.abs(fd - g).max() / max(np.abs(g).max(), 1e-3) < 1e-6


# --- packed variable-length sequences ("Triton FlashAttention-2 forward", "Exercises") ---

def test_varlen_single_sequence_is_plain_attention():
    q, k, v = (rng(40 + i).normal(size=(37, 3, 8)) for i in range(3))
    o, lse = oracle.attn_fwd_varlen(q, k, v, [0, 37], 0.6, True)
    o2, l2 = oracle.attn_fwd(q.transpose(1, 0, 2), k.transpose(1, 0, 2), v.transpose(1, 0, 2), 0.6, True)
    np.testing.assert_array_equal(o, o2.transpose(1, 0, 2))
    np.testing.assert_array_equal(lse, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_block_diagonal_softmax(causal):
    # brute force over the whole packed batch: one (total x total) score matrix
    # per head, keys of other sequences (and, causally, later keys of the same
    # sequence, counted from that sequence's start) set to -inf, library softmax
    cu = [0, 5, 5, 17, 18, 40]
    total, H, D, scale = cu[-1], 2, 6, 0.45
    q, k, v = (rng(50 + i).normal(size=(total, H, D)) * 2.0 for i in range(3))
    o, lse = oracle.attn_fwd_varlen(q, k, v, np.array(cu, dtype=np.int32), scale, causal)
    seq = np.zeros(total, dtype=int)
    pos = np.zeros(total, dtype=int)
    for s in range(len(cu) - 1):
        seq[cu[s]:cu[s + 1]] = s
        pos[cu[s]:cu[s + 1]] = np.arange(cu[s + 1] - cu[s])
    allowed = seq[:, None] == seq[None, :]
    if causal:
        allowed &= pos[None, :] <= pos[:, None]
    for h in range(H):
        S = np.where(allowed, scale * q[:, h] @ k[:, h].T, -np.inf)
        np.testing.assert_allclose(o[:, h], scipy.special.softmax(S, axis=1) @ v[:, h], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[h], scipy.special.logsumexp(S, axis=1), rtol=1e-12, atol=1e-12)


def test_varlen_backward_single_sequence_is_plain_backward():
    q, k, v, do = (rng(60 + i).normal(size=(29, 2, 8)) for i in range(4))
    g = oracle.attn_bwd_varlen(q, k, v, do, [0, 29], 0.5, True)
    t = lambda x: x.transpose(1, 0, 2)
    ref = oracle.attn_bwd(t(q), t(k), t(v), t(do), 0.5, True)
    for a, b in zip(g, ref[:3]):
        np.testing.assert_array_equal(a, t(b))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_matches_finite_differences(causal):
    # L = sum(dO * O) over the whole packed batch, O from the (pinned) varlen
    # forward; central differences of L against every input element
    cu = np.array([0, 4, 4, 9, 10], dtype=np.int32)
    total, H, D, scale, h = int(cu[-1]), 1, 3, 0.7, 1e-6
    q, k, v, do = (rng(70 + i).normal(size=(total, H, D)) for i in range(4))
    dq, dk, dv = oracle.attn_bwd_varlen(q, k, v, do, cu, scale, causal)

    def loss(qq, kk, vv):
        return float((oracle.attn_fwd_varlen(qq, kk, vv, cu, scale, causal)[0] * do).sum())

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(grad.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7)
