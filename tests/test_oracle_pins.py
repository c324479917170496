"""Pins of the CPU oracle to facts that do not come from the oracle itself:
the pages' printed compressed lengths, closed forms, textbook reductions that
a library routine computes independently (torch SDPA, numpy sort/matmul,
scipy expit), invariants of the definitions, and brute force on tiny inputs.
Each test is chosen so that a plausible slip in ``oracle.c`` (a dropped term,
a swapped index, a wrong sign, an off-by-one in visibility or the window)
fails it."""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- compressor

def _golden_lengths():
    rows = []
    with open(os.path.join(GOLDEN, "compressed_lengths.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                T, m, n, _ = line.split()
                rows.append((int(T), int(m), int(n)))
    return rows


@pytest.mark.parametrize("T,m,n", _golden_lengths())
def test_compressed_length_matches_pages(T, m, n):
    d = 2 if T > 100000 else 8
    X = np.zeros((T, d))
    G = np.zeros((m, d))
    assert oracle.compress(X, G, m).shape == (n, d)


@pytest.mark.parametrize("T,m", [(1027, 4), (3, 4), (255, 128), (0, 4), (130, 128)])
def test_tail_shorter_than_block_is_dropped(T, m):
    d = 4
    X = RNG.standard_normal((T, d))
    G = RNG.standard_normal((m, d))
    out = oracle.compress(X, G, m)
    assert out.shape == (T // m, d)
    if T // m:
        full = oracle.compress(X[: (T // m) * m], G, m)
        np.testing.assert_array_equal(out, full)


@pytest.mark.parametrize("m", [1, 4, 128])
def test_zero_gates_give_block_mean(m):
    T, d = 4 * m + 3, 16
    X = RNG.standard_normal((T, d))
    out = oracle.compress(X, np.zeros((m, d)), m)
    ref = X[: (T // m) * m].reshape(T // m, m, d).mean(axis=1)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-14)


def test_two_position_gate_is_logistic():
    # m=2: the weight of position 0 is sigmoid(g0 - g1) per channel.
    T, d = 10, 8
    X = RNG.standard_normal((T, d))
    G = RNG.standard_normal((2, d)) * 3
    w0 = expit(G[0] - G[1])
    ref = w0 * X[0::2] + (1 - w0) * X[1::2]
    np.testing.assert_allclose(oracle.compress(X, G, 2), ref, rtol=0, atol=1e-14)


def test_dominant_gate_copies_its_token_per_channel():
    # a +60 logit at a different position in every channel: each output
    # channel copies the token at that channel's own position.
    m, d, T = 4, 8, 12
    X = RNG.standard_normal((T, d))
    G = np.zeros((m, d))
    pick = np.array([0, 1, 2, 3, 3, 2, 1, 0])
    G[pick, np.arange(d)] = 60.0
    out = oracle.compress(X, G, m)
    ref = np.stack([X[j * m + pick, np.arange(d)] for j in range(T // m)])
    # the other weights are below 3*exp(-60); fp64 rounding dominates
    np.testing.assert_allclose(out, ref, rtol=0, atol=4e-16 * np.abs(X).max())


def test_compress_linear_and_position_permutation():
    m, d, T = 4, 6, 20
    X1, X2 = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    G = RNG.standard_normal((m, d))
    a, b = 0.75, -2.5
    np.testing.assert_allclose(oracle.compress(a * X1 + b * X2, G, m),
                               a * oracle.compress(X1, G, m) + b * oracle.compress(X2, G, m),
                               rtol=0, atol=1e-13)
    perm = np.array([2, 0, 3, 1])
    Xp = X1.reshape(T // m, m, d)[:, perm].reshape(T, d)
    np.testing.assert_allclose(oracle.compress(Xp, G[perm], m), oracle.compress(X1, G, m),
                               rtol=0, atol=1e-14)
    # a per-channel shift of the logits changes nothing (softmax), a
    # per-position one does
    np.testing.assert_allclose(oracle.compress(X1, G + RNG.standard_normal(d), m),
                               oracle.compress(X1, G, m), rtol=0, atol=1e-13)
    shifted = G.copy()
    shifted[0] += 1.0
    assert np.abs(oracle.compress(X1, shifted, m) - oracle.compress(X1, G, m)).max() > 1e-3


# -------------------------------------------------------------------- indexer

def test_visibility_boundary():
    # entry j is visible exactly from position (j+1)*m - 1 on
    m, Tc = 4, 5
    for t in range(0, Tc * m):
        nv = int(oracle.n_visible(t, m))
        assert nv == sum(1 for j in range(Tc) if (j + 1) * m - 1 <= t)
    assert oracle.n_visible(2, 4) == 0 and oracle.n_visible(3, 4) == 1
    assert oracle.n_visible(126, 128) == 0 and oracle.n_visible(127, 128) == 1


def test_single_head_unit_weight_is_relu_of_matmul():
    Nq, Tc, dI, m = 24, 6, 16, 4
    q = RNG.standard_normal((Nq, 1, dI))
    k = RNG.standard_normal((Tc, 1, dI))
    t = np.arange(Nq)
    I = oracle.index(q, np.ones((Nq, 1)), k, t, m)
    ref = np.maximum(q[:, 0] @ k[:, 0].T, 0.0)
    for r in range(Nq):
        nv = (r + 1) // m
        np.testing.assert_allclose(I[r, :nv], ref[r, :nv], rtol=0, atol=1e-12)
        assert np.all(np.isneginf(I[r, nv:]))


def test_index_sums_single_head_indexers():
    Nq, Tc, HI, dI, m = 36, 9, 4, 8, 4
    q = RNG.standard_normal((Nq, HI, dI))
    k = RNG.standard_normal((Tc, HI, dI))
    w = RNG.random((Nq, HI))
    t = np.arange(Nq)
    I = oracle.index(q, w, k, t, m)
    parts = sum(oracle.index(q[:, h:h + 1], w[:, h:h + 1], k[:, h:h + 1], t, m) for h in range(HI))
    vis = np.isfinite(I)
    np.testing.assert_array_equal(vis, np.isfinite(parts))
    np.testing.assert_allclose(I[vis], parts[vis], rtol=1e-13, atol=1e-12)
    # positive rescaling of the head weights rescales the score
    np.testing.assert_allclose(oracle.index(q, 3.0 * w, k, t, m)[vis], 3.0 * I[vis], rtol=1e-13)
    # heads whose dot product is negative contribute nothing: flipping the
    # sign of q for a head changes the score by exactly that head's part
    q2 = q.copy()
    q2[:, 1] *= -1
    I2 = oracle.index(q2, w, k, t, m)
    p1 = oracle.index(q[:, 1:2], w[:, 1:2], k[:, 1:2], t, m)
    p1n = oracle.index(q2[:, 1:2], w[:, 1:2], k[:, 1:2], t, m)
    with np.errstate(invalid="ignore"):
        np.testing.assert_allclose(I2[vis], (I - p1 + p1n)[vis], rtol=1e-12, atol=1e-12)
    assert np.all(I[vis] >= 0)


# ---------------------------------------------------------------------- top-k

def _brute_topk(row, nv, k):
    order = sorted(range(nv), key=lambda j: (-row[j], j))[:k]
    return sorted(order) + [-1] * (k - min(k, nv))


def test_topk_hand_worked_ties():
    I = np.array([[1.0, 3.0, 3.0, 0.0, 3.0, 2.0]])
    nv = np.array([6])
    assert oracle.topk(I, nv, 3).tolist() == [[1, 2, 4]]
    assert oracle.topk(I, nv, 2).tolist() == [[1, 2]]
    assert oracle.topk(I, nv, 4).tolist() == [[1, 2, 4, 5]]
    assert oracle.topk(I, nv, 8).tolist() == [[0, 1, 2, 3, 4, 5, -1, -1]]
    # entries beyond the visible count are never read, however large
    I2 = np.array([[1.0, 0.5, 9.0, 9.0]])
    assert oracle.topk(I2, np.array([2]), 1).tolist() == [[0]]
    assert oracle.topk(I2, np.array([0]), 2).tolist() == [[-1, -1]]


def test_topk_signed_zero_ties():
    assert oracle.topk(np.array([[-0.0, 0.0]]), np.array([2]), 1).tolist() == [[0]]
    assert oracle.topk(np.array([[0.0, -0.0]]), np.array([2]), 1).tolist() == [[0]]
    assert oracle.topk(np.array([[-1.0, -0.0, 0.0]]), np.array([3]), 2).tolist() == [[1, 2]]


@pytest.mark.parametrize("levels", [None, 4, 2])
def test_topk_brute_force_and_stable_argsort(levels):
    Nq, ld, k = 64, 50, 7
    if levels is None:
        I = RNG.standard_normal((Nq, ld))
    else:
        I = RNG.integers(0, levels, (Nq, ld)).astype(np.float64)
    nv = RNG.integers(0, ld + 1, Nq)
    got = oracle.topk(I, nv, k)
    for r in range(Nq):
        assert got[r].tolist() == _brute_topk(I[r], int(nv[r]), k)
        sel = np.argsort(-I[r, : nv[r]], kind="stable")[:k]
        keep = min(k, int(nv[r]))
        assert got[r, :keep].tolist() == sorted(sel.tolist())
        assert np.all(got[r, keep:] == -1)


# ------------------------------------------------------------------ attention

def _sdpa(Q, K, V, mask, scale):
    """torch scaled_dot_product_attention in fp64 (a library routine), MQA:
    one K/V shared by every head.  Q [Nq,H,d], K/V [n,d], mask [Nq,n] bool."""
    q = torch.from_numpy(Q).permute(1, 0, 2)  # [H, Nq, d]
    k = torch.from_numpy(K)[None].expand(Q.shape[1], -1, -1)
    v = torch.from_numpy(V)[None].expand(Q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=torch.from_numpy(mask)[None], scale=scale)
    logits = (q @ k.transpose(-1, -2)) * scale
    logits = logits.masked_fill(~torch.from_numpy(mask)[None], -math.inf)
    lse = torch.logsumexp(logits, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


def test_m1_no_window_is_causal_attention():
    T, H, d = 33, 3, 8
    Q = RNG.standard_normal((T, H, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    scale = 1 / math.sqrt(d)
    t = np.arange(T)
    mask = t[None, :] <= t[:, None]
    ref_o, ref_l = _sdpa(Q, K, V, mask, scale)
    # HCA form with m'=1: every past token is an entry
    o, l = oracle.hca_attn(Q, K, V, 1, K[:0], V[:0], 0, t, 0, scale)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)
    # CSA form with m=1 and k >= t+1: select every visible entry
    idx = np.full((T, T), -1, dtype=np.int32)
    for r in range(T):
        idx[r, : r + 1] = np.arange(r + 1)
    o2, l2 = oracle.sparse_attn(Q, K, V, idx, K[:0], V[:0], 0, t, 0, scale)
    np.testing.assert_allclose(o2, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, ref_l, rtol=0, atol=1e-12)


def test_window_only_is_banded_attention():
    # with no compressed entries visible, only the raw window remains
    T, H, d, W = 20, 2, 4, 5
    Q = RNG.standard_normal((T, H, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    t = np.arange(T)
    mask = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - W)
    ref_o, ref_l = _sdpa(Q, K, V, mask, 0.5)
    o, l = oracle.hca_attn(Q, K[:0], V[:0], 1000, K, V, 0, t, W, 0.5)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)
    # W = 1: the output is the token's own value row
    o1, _ = oracle.hca_attn(Q, K[:0], V[:0], 1000, K, V, 0, t, 1, 0.5)
    np.testing.assert_allclose(o1, np.broadcast_to(V[:, None, :], o1.shape), rtol=0, atol=1e-15)


def test_hca_equals_masked_dense_attention_over_entries_and_window():
    m, T, H, d, W = 8, 70, 4, 8, 6
    Q = RNG.standard_normal((T, H, d))
    Kc, Vc = RNG.standard_normal((T // m, d)), RNG.standard_normal((T // m, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    t = np.arange(T)
    j = np.arange(T // m)
    mask_c = (j[None, :] + 1) * m - 1 <= t[:, None]
    mask_r = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - W)
    ref_o, ref_l = _sdpa(Q, np.concatenate([Kc, K]), np.concatenate([Vc, V]),
                         np.concatenate([mask_c, mask_r], axis=1), 0.3)
    o, l = oracle.hca_attn(Q, Kc, Vc, m, K, V, 0, t, W, 0.3)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_sparse_with_all_visible_selected_equals_hca():
    m, T, H, d, W, k = 4, 64, 2, 8, 4, 20
    Q = RNG.standard_normal((T, H, d))
    Kc, Vc = RNG.standard_normal((T // m, d)), RNG.standard_normal((T // m, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    t = np.arange(T)
    nv = oracle.n_visible(t, m)
    assert nv.max() <= k
    idx = oracle.topk(RNG.standard_normal((T, T // m)), nv, k)
    o1, l1 = oracle.sparse_attn(Q, Kc, Vc, idx, K, V, 0, t, W, 0.4)
    o2, l2 = oracle.hca_attn(Q, Kc, Vc, m, K, V, 0, t, W, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_single_key_and_empty_set():
    H, d = 3, 5
    Q = RNG.standard_normal((1, H, d))
    Kc, Vc = RNG.standard_normal((4, d)), RNG.standard_normal((4, d))
    o, l = oracle.sparse_attn(Q, Kc, Vc, np.array([[2, -1, -1]]), Kc[:0], Vc[:0], 0, [11], 0, 0.7)
    np.testing.assert_allclose(o[0], np.broadcast_to(Vc[2], (H, d)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(l[0], 0.7 * Q[0] @ Kc[2], rtol=0, atol=1e-14)
    o, l = oracle.sparse_attn(Q, Kc, Vc, np.array([[-1, -1]]), Kc[:0], Vc[:0], 0, [11], 0, 0.7)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_lse_merge_of_disjoint_key_sets():
    H, d, n = 4, 8, 12
    Q = RNG.standard_normal((1, H, d))
    Kc, Vc = RNG.standard_normal((n, d)), RNG.standard_normal((n, d))
    A, B = [0, 3, 5, 7, 8], [1, 2, 9, 11]
    z = Kc[:0]
    oa, la = oracle.sparse_attn(Q, Kc, Vc, np.array([A]), z, z, 0, [10 ** 6], 0, 0.5)
    ob, lb = oracle.sparse_attn(Q, Kc, Vc, np.array([B]), z, z, 0, [10 ** 6], 0, 0.5)
    ou, lu = oracle.sparse_attn(Q, Kc, Vc, np.array([A + B]), z, z, 0, [10 ** 6], 0, 0.5)
    lm = np.logaddexp(la, lb)
    om = np.exp(la - lm)[..., None] * oa + np.exp(lb - lm)[..., None] * ob
    np.testing.assert_allclose(lu, lm, rtol=0, atol=1e-13)
    np.testing.assert_allclose(ou, om, rtol=0, atol=1e-13)


def test_head_permutation_equivariance_and_window_source_offset():
    m, T, H, d, W = 4, 40, 6, 8, 8
    Q = RNG.standard_normal((T, H, d))
    Kc, Vc = RNG.standard_normal((T // m, d)), RNG.standard_normal((T // m, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    t = np.arange(T)
    idx = oracle.topk(RNG.standard_normal((T, T // m)), oracle.n_visible(t, m), 3)
    o, l = oracle.sparse_attn(Q, Kc, Vc, idx, K, V, 0, t, W, 0.3)
    perm = RNG.permutation(H)
    op, lp = oracle.sparse_attn(Q[:, perm], Kc, Vc, idx, K, V, 0, t, W, 0.3)
    np.testing.assert_allclose(op, o[:, perm], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lp, l[:, perm], rtol=0, atol=1e-14)
    # a raw cache holding only positions 30.. answers the rows t >= 37 alike
    rows = t >= 30 + W - 1
    o2, l2 = oracle.sparse_attn(Q[rows], Kc, Vc, idx[rows], K[30:], V[30:], 30, t[rows], W, 0.3)
    np.testing.assert_allclose(o2, o[rows], rtol=0, atol=1e-14)
    with pytest.raises(ValueError):
        oracle.sparse_attn(Q, Kc, Vc, idx, K[30:], V[30:], 30, t, W, 0.3)


# ------------------------------------------------------ attention sink logit
# The sink is one extra per-head logit in the softmax's denominator with no
# value ("DeepSeek-V4 技术解析…", §1.1, engineering details: a learnable sink
# logit lets a head push its total attention toward zero).


def test_sink_single_key_is_logistic_gate():
    # one key with logit z and a sink s: O = sigmoid(z - s) V, lse = log(e^z + e^s)
    H, d = 3, 5
    Q = RNG.standard_normal((1, H, d))
    Kc, Vc = RNG.standard_normal((4, d)), RNG.standard_normal((4, d))
    sink = np.array([-0.5, 1.25, 3.0])
    o, l = oracle.sparse_attn(Q, Kc, Vc, np.array([[2, -1]]), Kc[:0], Vc[:0], 0, [11], 0, 0.7,
                              sink=sink)
    z = 0.7 * Q[0] @ Kc[2]
    np.testing.assert_allclose(o[0], expit(z - sink)[:, None] * Vc[2][None, :], rtol=0,
                               atol=1e-14)
    np.testing.assert_allclose(l[0], np.logaddexp(z, sink), rtol=0, atol=1e-13)


def test_sink_rescales_the_sinkless_result():
    # O_s = O * e^lse / (e^lse + e^s) and lse_s = logaddexp(lse, s), per head;
    # a sink of -inf is no sink; an empty key set gives O = 0 and lse = s
    m, T, H, d, W = 4, 40, 6, 8, 8
    Q = RNG.standard_normal((T, H, d))
    Kc, Vc = RNG.standard_normal((T // m, d)), RNG.standard_normal((T // m, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    t = np.arange(T)
    sink = np.array([-np.inf, -2.0, 0.0, 0.5, 4.0, 30.0])
    for attn in (lambda s: oracle.hca_attn(Q, Kc, Vc, m, K, V, 0, t, W, 0.3, sink=s),
                 lambda s: oracle.sparse_attn(
                     Q, Kc, Vc, oracle.topk(np.tile(np.arange(T // m, dtype=float), (T, 1)),
                                            oracle.n_visible(t, m), 3),
                     K, V, 0, t, W, 0.3, sink=s)):
        o0, l0 = attn(None)
        o1, l1 = attn(sink)
        gate = np.exp(l0 - np.logaddexp(l0, sink[None, :]))
        np.testing.assert_allclose(o1, o0 * gate[..., None], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l1, np.logaddexp(l0, sink[None, :]), rtol=0, atol=1e-12)
        assert np.array_equal(o1[:, 0], o0[:, 0]) and np.array_equal(l1[:, 0], l0[:, 0])
    o, l = oracle.sparse_attn(Q[:1], Kc, Vc, np.array([[-1, -1]]), Kc[:0], Vc[:0], 0, [11], 0,
                              0.7, sink=sink)
    assert np.all(o == 0) and np.array_equal(l[0], sink)


def test_sink_must_be_a_real_logit_or_minus_inf():
    # NaN and +inf are not logits: the oracle refuses them (the library flags
    # them on the device and treats that head as having no sink)
    rng = np.random.default_rng(9)
    Q = rng.standard_normal((1, 2, 8))
    Kc, Vc = rng.standard_normal((4, 8)), rng.standard_normal((4, 8))
    for bad in (np.nan, np.inf):
        with pytest.raises(ValueError, match="finite or -inf"):
            oracle.hca_attn(Q, Kc, Vc, 1, Kc, Vc, 0, [3], 0, 0.5, sink=np.array([0.0, bad]))


# ------------------------------------------------------ token-gated compressor
# The learned compressor of the pages ("DeepSeek-V4 技术解析…", §1.1, CSA
# paragraph) takes its gates from each token: Z [T, d] holds one gate logit per
# token and channel, softmax-normalised over the m tokens of a block.


def test_token_gates_reduce_to_position_gates():
    # gates that repeat the same [m, d] pattern in every block are the
    # position-gated compressor
    m, d, T = 4, 6, 4 * 9 + 3
    X = RNG.standard_normal((T, d))
    G = RNG.standard_normal((m, d))
    Z = np.tile(G, (T // m + 1, 1))[:T]
    np.testing.assert_allclose(oracle.compress_tok(X, Z, m), oracle.compress(X, G, m),
                               rtol=0, atol=1e-14)


def test_token_gates_closed_forms():
    m, d, T = 8, 5, 8 * 6
    X = RNG.standard_normal((T, d))
    # equal logits within a block (any value per block and channel): block mean
    Z = np.repeat(RNG.standard_normal((T // m, d)) * 30, m, axis=0)
    np.testing.assert_allclose(oracle.compress_tok(X, Z, m),
                               X.reshape(T // m, m, d).mean(axis=1), rtol=0, atol=1e-13)
    # one token of each block 60 above the others, per channel: that token
    pick = RNG.integers(0, m, size=(T // m, d))
    Z = np.zeros((T, d))
    for j in range(T // m):
        for c in range(d):
            Z[j * m + pick[j, c], c] = 60.0
    want = np.array([[X[j * m + pick[j, c], c] for c in range(d)] for j in range(T // m)])
    np.testing.assert_allclose(oracle.compress_tok(X, Z, m), want, rtol=0, atol=1e-24 + 1e-20)
    # m = 2: the first token's weight is expit(z0 - z1)
    Z = RNG.standard_normal((2 * 7, d)) * 3
    X = RNG.standard_normal((2 * 7, d))
    a = expit(Z[0::2] - Z[1::2])
    np.testing.assert_allclose(oracle.compress_tok(X, Z, 2), a * X[0::2] + (1 - a) * X[1::2],
                               rtol=0, atol=1e-14)


def test_token_gates_depend_on_each_token():
    # changing one token's gate changes only its own block, and a logit shift
    # shared by a block's tokens (per channel) changes nothing
    m, d, T = 4, 3, 4 * 5
    X = RNG.standard_normal((T, d))
    Z = RNG.standard_normal((T, d))
    base = oracle.compress_tok(X, Z, m)
    Z2 = Z.copy()
    Z2[9, 1] += 2.0  # block 2, channel 1
    out = oracle.compress_tok(X, Z2, m)
    diff = np.abs(out - base) > 1e-15
    assert diff[2, 1] and diff.sum() == 1
    Z3 = Z + np.repeat(RNG.standard_normal((T // m, d)), m, axis=0) * 10
    np.testing.assert_allclose(oracle.compress_tok(X, Z3, m), base, rtol=0, atol=1e-13)


# ------------------------------------------------------------ partial RoPE
# "DeepSeek-V4 技术解析…", §1.1, engineering details: RoPE acts only on the last
# 64 dimensions; the core-attention output gets the inverse RoPE to restore
# relative positions.  The rotation itself is RoPE as RoFormer defines it
# (pairs as complex numbers multiplied by e^{i p theta_i},
# theta_i = 10000^(-2i/64)).


def _rope_complex(X, pos):
    # independent formulation: complex multiplication of the interleaved pairs
    X = np.asarray(X, dtype=np.float64)
    d = X.shape[-1]
    z = X[..., d - 64::2] + 1j * X[..., d - 64 + 1::2]
    theta = 10000.0 ** (-np.arange(0, 64, 2) / 64.0)
    shape = (len(pos),) + (1,) * (X.ndim - 2) + (32,)
    rot = np.exp(1j * np.asarray(pos, dtype=np.float64).reshape(-1, *([1] * (X.ndim - 1)))
                 * theta).reshape(shape)
    w = z * rot
    Y = X.copy()
    Y[..., d - 64::2] = w.real
    Y[..., d - 64 + 1::2] = w.imag
    return Y


def test_rope_is_roformer_rotation_of_the_last_64_dims():
    X = RNG.standard_normal((7, 3, 128))
    pos = np.array([0, 1, 5, 127, 4095, 1048575, 999983])
    Y = oracle.rope(X, pos)
    np.testing.assert_allclose(Y, _rope_complex(X, pos), rtol=0, atol=1e-9)
    assert np.array_equal(Y[..., :64], X[..., :64])            # first d-64 dims untouched
    np.testing.assert_allclose(Y[0], X[0], rtol=0, atol=0)       # position 0: identity
    # the rotation keeps each pair's norm
    nx = X[..., 64::2] ** 2 + X[..., 65::2] ** 2
    ny = Y[..., 64::2] ** 2 + Y[..., 65::2] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12)
    # the inverse undoes it; d = 64 rotates every dimension
    np.testing.assert_allclose(oracle.rope(Y, pos, inverse=True), X, rtol=0, atol=1e-9)
    X64 = RNG.standard_normal((4, 64))
    p4 = np.array([3, 9, 10, 200])
    np.testing.assert_allclose(oracle.rope(X64, p4), _rope_complex(X64, p4), rtol=0, atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    q, k = RNG.standard_normal((1, 128)), RNG.standard_normal((1, 128))
    for t, s_, delta in ((10, 3, 1000), (500, 499, 123457), (7, 7, 5)):
        a = oracle.rope(q, [t]) @ oracle.rope(k, [s_]).T
        b = oracle.rope(q, [t + delta]) @ oracle.rope(k, [s_ + delta]).T
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-10)


def _rope_case(m, T, W, H=3, d=128, q_from=0):
    Q = RNG.standard_normal((T - q_from, H, d))
    K, V = RNG.standard_normal((T, d)), RNG.standard_normal((T, d))
    G = RNG.standard_normal((m, d))
    return Q, K, V, G


def test_attention_with_rope_is_invariant_to_a_common_shift():
    # the output is rotated back at t, so moving every position (queries,
    # window tokens, entries) by a multiple of m changes nothing; a slip in any
    # rotation (q, k, v, the output, or an entry's position) breaks this
    m, W, T, shift = 4, 6, 64, 4 * 37
    Q, K, V, G = _rope_case(m, T, W)
    rows = np.arange(W - 1, T)          # windows stay inside the stored tokens
    Q = Q[rows]
    Kc, Vc = oracle.compress(K, G, m), oracle.compress(V, G, m)
    idx = np.full((len(rows), T // m), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        nv = (r + 1) // m
        idx[i, :nv] = np.arange(nv)
    o1, l1 = oracle.hca_attn_rope(Q, Kc, Vc, m, K, V, 0, rows, W, 0.3)
    o3, l3 = oracle.sparse_attn_rope(Q, Kc, Vc, idx, K, V, 0, rows, W, 0.3, m)
    np.testing.assert_allclose(o3, o1, rtol=0, atol=1e-12)      # CSA with all selected == HCA
    # the same tokens at positions shift .., after shift/m entries nobody selects
    zc = np.zeros((shift // m, K.shape[1]))
    idx2 = np.where(idx >= 0, idx + shift // m, -1).astype(np.int32)
    o2, l2 = oracle.sparse_attn_rope(Q, np.concatenate([zc, Kc]), np.concatenate([zc, Vc]), idx2,
                                     K, V, shift, rows + shift, W, 0.3, m)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-9)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-9)
    # and RoPE does change the result (the test would be vacuous otherwise)
    o0, _ = oracle.hca_attn(Q, Kc, Vc, m, K, V, 0, rows, W, 0.3)
    assert np.abs(o0 - o1).max() > 1e-2


def test_rope_single_key_at_the_query_position_returns_its_value():
    # one key at the query's own position: q.k is unrotated, v is rotated at t
    # and the output rotated back at t, so O = v exactly
    d, t = 128, 123457
    Q = RNG.standard_normal((1, 2, d))
    K, V = RNG.standard_normal((1, d)), RNG.standard_normal((1, d))
    o, l = oracle.sparse_attn_rope(Q, K[:0], V[:0], np.full((1, 1), -1, np.int32), K, V, t, [t],
                                   1, 0.5, 4)
    np.testing.assert_allclose(o[0], np.repeat(V, 2, axis=0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(l[0], 0.5 * (Q[0] @ K[0]), rtol=0, atol=1e-10)


def test_rope_entry_sits_at_its_last_token():
    # an entry is rotated at the position of its block's last token: a query at
    # exactly that position attending to that entry alone gets its value back
    d, m, j = 128, 4, 5
    t = (j + 1) * m - 1
    Q = RNG.standard_normal((1, 2, d))
    Kc, Vc = RNG.standard_normal((8, d)), RNG.standard_normal((8, d))
    idx = np.array([[j, -1]], dtype=np.int32)
    o, _ = oracle.sparse_attn_rope(Q, Kc, Vc, idx, Kc[:0], Vc[:0], 0, [t], 0, 0.5, m)
    np.testing.assert_allclose(o[0], np.repeat(Vc[j:j + 1], 2, axis=0), rtol=0, atol=1e-12)
    # one position later the value comes back rotated by one step
    o2, _ = oracle.sparse_attn_rope(Q, Kc, Vc, idx, Kc[:0], Vc[:0], 0, [t + 1], 0, 0.5, m)
    np.testing.assert_allclose(o2[0], np.repeat(oracle.rope(Vc[j:j + 1], [-1]), 2, axis=0),
                               rtol=0, atol=1e-12)


# ------------------------------------------------ MX (microscaling) quantizer

def _elem_table(fmt):
    """Every non-negative finite element of the format with its code, listed
    from the format's definition (sign bit clear): E4M3 bias 7, 3 mantissa
    bits, exponent field 15 with mantissa 7 is NaN; E2M1 bias 1, 1 bit."""
    mb, bias, ne = (3, 7, 16) if fmt == oracle.MXFP8 else (1, 1, 4)
    vals = []
    for ef in range(ne):
        for mf in range(1 << mb):
            if fmt == oracle.MXFP8 and ef == 15 and mf == 7:
                continue
            v = (mf / (1 << mb)) * 2.0 ** (1 - bias) if ef == 0 else \
                (1 + mf / (1 << mb)) * 2.0 ** (ef - bias)
            vals.append((v, (ef << mb) | mf))
    return vals


def _nearest_by_search(x, fmt):
    """Brute force: the element nearest to |x|, ties to the even code, the
    largest element for anything beyond it; the sign bit from x."""
    table = _elem_table(fmt)
    a = abs(x)
    best = min(table, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))
    sbit = 0x80 if fmt == oracle.MXFP8 else 0x8
    return (math.copysign(best[0], x), best[1] | (sbit if math.copysign(1, x) < 0 else 0))


def _block_with_unit_scale(vals, fmt):
    """Blocks of 32 whose largest magnitude makes the shared scale 1 (the
    largest element itself), so the codes are those of the raw values."""
    top = 448.0 if fmt == oracle.MXFP8 else 6.0
    vals = list(vals)
    out = []
    for i in range(0, len(vals), 31):
        chunk = vals[i:i + 31]
        out += chunk + [top] * (32 - len(chunk))
    return np.array(out, dtype=np.float64)


@pytest.mark.parametrize("fmt", [8, 4])
def test_mx_elements_are_the_nearest_by_search(fmt):
    table = [v for v, _ in _elem_table(fmt)]
    mids = [(a + b) / 2 for a, b in zip(table[:-1], table[1:])]
    eps = [math.nextafter(v, math.inf) for v in mids] + [math.nextafter(v, 0) for v in mids]
    rnd = list(RNG.uniform(0, table[-1], 600))
    xs = table + mids + eps + rnd
    xs = xs + [-v for v in xs]
    X = _block_with_unit_scale(xs, fmt)
    codes, scales, deq = oracle.mx_quantize(X, fmt)
    assert np.all(scales == 127)
    for x, c, dv in zip(X, codes, deq):
        ev, ec = _nearest_by_search(x, fmt)
        assert dv == ev and c == ec, (x, dv, ev, c, ec)


def test_mxfp8_elements_equal_torch_e4m3():
    # torch's float8_e4m3fn conversion (round to nearest even) on values the
    # unit scale keeps within the finite range
    vals = np.concatenate([RNG.uniform(-448, 448, 3000), RNG.standard_normal(2000) * 4,
                           RNG.uniform(-2.0 ** -6, 2.0 ** -6, 1000)])
    X = _block_with_unit_scale(vals, oracle.MXFP8)
    codes, _, deq = oracle.mx_quantize(X, oracle.MXFP8)
    t = torch.from_numpy(X).float().to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(deq, t.double().numpy())
    np.testing.assert_array_equal(codes, t.view(torch.uint8).numpy())


@pytest.mark.parametrize("fmt,emax", [(8, 8), (4, 2)])
def test_mx_shared_scale_is_floor_log2_amax_minus_emax(fmt, emax):
    amaxes = np.concatenate([2.0 ** RNG.uniform(-60, 60, 400),
                             2.0 ** np.arange(-60, 61, dtype=np.float64)])
    for amax in amaxes:
        X = RNG.uniform(-1, 1, 32) * amax * 0.999
        X[RNG.integers(32)] = -amax if RNG.random() < 0.5 else amax
        _, scales, deq = oracle.mx_quantize(X, fmt)
        e = int(scales[0]) - 127
        # 2^(e + emax) <= amax < 2^(e + emax + 1), by exact comparisons
        assert 2.0 ** (e + emax) <= amax < 2.0 ** (e + emax + 1)
        # every value is within half an element step of its dequantized value,
        # or clamped at the largest element
        top = (448.0 if fmt == 8 else 6.0) * 2.0 ** e
        mb = 3 if fmt == 8 else 1
        emin = -6 if fmt == 8 else 0
        for x, dv in zip(X, deq):
            a = abs(x) / 2.0 ** e
            E = max(math.floor(math.log2(a)) if a > 0 else emin, emin)
            half = 2.0 ** (E - mb - 1) * 2.0 ** e
            assert abs(dv - x) <= half * (1 + 1e-12) or abs(dv) == top


def test_mx_zero_block_and_saturation():
    _, s, d = oracle.mx_quantize(np.zeros(32), oracle.MXFP8)
    assert s[0] == 0 and np.all(d == 0)
    # amax = 500: shared exponent floor(log2 500) - 8 = 0, so 500 clamps to 448
    X = np.zeros(32)
    X[3], X[4] = 500.0, -479.0
    _, s, d = oracle.mx_quantize(X, oracle.MXFP8)
    assert s[0] == 127 and d[3] == 448.0 and d[4] == -448.0
    X[3], X[4] = 7.9, -6.5
    _, s, d = oracle.mx_quantize(X, oracle.MXFP4)
    assert s[0] == 127 and d[3] == 6.0 and d[4] == -6.0


@pytest.mark.parametrize("fmt", [8, 4])
def test_mx_index_is_the_index_of_representable_inputs(fmt):
    # inputs already on the element grid (with the block's own top value so the
    # scale is 1) quantize to themselves: the low-precision score is the exact one
    table = np.array([v for v, _ in _elem_table(fmt)])
    top = table[-1]
    q = RNG.choice(np.concatenate([table, -table]), (3, 2, 64))
    k = RNG.choice(np.concatenate([table, -table]), (9, 2, 64))
    q[..., 0], q[..., 32], k[..., 0], k[..., 32] = top, top, top, top
    w = RNG.uniform(0, 1, (3, 2))
    t = np.array([35, 20, 8])
    np.testing.assert_array_equal(oracle.index_mx(q, w, k, t, 4, fmt),
                                  oracle.index(q, w, k, t, 4))
    # a generic input differs from the exact score by the quantization only
    q2, k2 = RNG.standard_normal((3, 2, 64)), RNG.standard_normal((9, 2, 64))
    I, Iq = oracle.index(q2, w, k2, t, 4), oracle.index_mx(q2, w, k2, t, 4, fmt)
    vis = np.isfinite(I)
    assert np.all(np.isfinite(Iq) == vis) and not np.array_equal(I[vis], Iq[vis])
