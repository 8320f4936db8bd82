"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages or the mathematics fix: a
hand-worked example of the layer formula (L³: Large Lookup Layers, gist.science,
Technical Summary > Core Architecture), special cases with closed forms, invariants,
the block-diagonal masked formulation (Systems-Friendly Design > Batch Sorting),
finite differences and an autograd derivation of the gradient.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_layer(rng, vocab=6, d=5, d_v=4, T=9, n=None, scale=1.0):
    n = np.array(n if n is not None else rng.integers(1, 5, size=vocab))
    offs = np.zeros(len(n) + 1, dtype=np.int64)
    offs[1:] = np.cumsum(n)
    v = int(offs[-1])
    K = rng.standard_normal((v, d)) * scale
    V = rng.standard_normal((v, d_v))
    W_up = rng.standard_normal((d, d_v)) / math.sqrt(d_v)
    W_mix = rng.standard_normal((d, 2 * d)) / math.sqrt(2 * d)
    ids = rng.integers(0, len(n), size=T)
    x = rng.standard_normal((T, d))
    return offs, K, V, W_up, W_mix, ids, x


# ---- hand-worked examples of the layer formula ------------------------------------------

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("hand_worked_layer.json")["cases"], ids=lambda c: c["name"])
def test_hand_worked_layer(case):
    Kt, Vt = np.array(case["K_t"]), np.array(case["V_t"])
    offs = np.array([0, Kt.shape[0]])
    fw = oracle.forward(offs, Kt, Vt, np.array(case["W_up"]), np.array(case["W_mix"]),
                        np.array([0]), np.array([case["x"]]), eps=case["eps"])
    _, _, p, _, _ = oracle.attend(Kt, Vt, np.array(case["x"]))
    np.testing.assert_allclose(p, case["p"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(fw.a[0], case["a"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(fw.u[0], case["u"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(fw.h[0], case["h"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fw.y[0], case["y"], rtol=0, atol=1e-12)


# ---- special cases of the aggregation ------------------------------------------------------

def test_single_row_returns_value_row_exactly():
    rng = np.random.default_rng(1)
    K = rng.standard_normal((1, 7)) * 5
    V = rng.standard_normal((1, 3))
    a, s, p, m, l = oracle.attend(K, V, rng.standard_normal(7))
    assert p.tolist() == [1.0] and l == 1.0
    assert np.array_equal(a, V[0])


def test_zero_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    V = rng.standard_normal((11, 5))
    a, _, p, _, _ = oracle.attend(np.zeros((11, 3)), V, rng.standard_normal(3))
    np.testing.assert_allclose(p, np.full(11, 1 / 11), rtol=1e-15)
    np.testing.assert_allclose(a, V.mean(axis=0), rtol=0, atol=1e-15)


def test_no_temperature_two_rows():
    # p_0 = 1 / (1 + exp(s_1 - s_0)) with s = K_t x unscaled (a 1/sqrt(d) factor fails this)
    K = np.array([[0.7, -0.2, 0.4, 1.1], [0.3, 0.5, -0.6, 0.2]])
    x = np.array([1.5, -0.5, 2.0, 0.25])
    s0, s1 = float(K[0] @ x), float(K[1] @ x)
    V = np.array([[1.0, 0.0], [0.0, 1.0]])
    a, _, p, _, _ = oracle.attend(K, V, x)
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    np.testing.assert_allclose(a, [p0, 1 - p0], rtol=1e-14)


def test_row_permutation_within_range_is_invariant():
    rng = np.random.default_rng(3)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, n=[3, 5, 1, 4])
    y0 = oracle.forward(offs, K, V, W_up, W_mix, ids, x).y
    K2, V2 = K.copy(), V.copy()
    for t in range(4):
        r = oracle.token_rows(offs, t)
        perm = rng.permutation(len(r)) + r.start
        K2[r.start:r.stop], V2[r.start:r.stop] = K[perm], V[perm]
    y1 = oracle.forward(offs, K2, V2, W_up, W_mix, ids, x).y
    np.testing.assert_allclose(y1, y0, rtol=0, atol=1e-13)


def test_dense_masked_attention_equals_gathered():
    rng = np.random.default_rng(4)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, vocab=13, d=8, d_v=6, T=40)
    a = oracle.forward(offs, K, V, W_up, W_mix, ids, x).a
    np.testing.assert_allclose(oracle.attend_dense_masked(offs, K, V, ids, x), a, rtol=0, atol=1e-13)


def test_routing_is_static_rows_of_other_ids_do_not_matter():
    rng = np.random.default_rng(5)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, n=[2, 3, 4, 1, 2, 2])
    ids = np.array([1, 1, 4])
    y0 = oracle.forward(offs, K, V, W_up, W_mix, ids, x[:3]).y
    K2, V2 = K.copy(), V.copy()
    for t in (0, 2, 3, 5):
        r = oracle.token_rows(offs, t)
        K2[r.start:r.stop] = 1e3
        V2[r.start:r.stop] = -7.0
    y1 = oracle.forward(offs, K2, V2, W_up, W_mix, ids, x[:3]).y
    assert np.array_equal(y0, y1)


# ---- LayerNorm and the concatenation --------------------------------------------------------

def test_layer_norm_closed_form_and_invariants():
    u = np.array([1.0, -1.0, 1.0, -1.0])
    h, mu, rstd = oracle.layer_norm(u, eps=0.5)
    assert mu == 0.0 and rstd == 1 / math.sqrt(1.5)
    np.testing.assert_allclose(h, u / math.sqrt(1.5), rtol=1e-15)
    rng = np.random.default_rng(6)
    for eps in (1e-5, 0.1):
        u = rng.standard_normal(64) * 0.03 + 0.2
        h, mu, rstd = oracle.layer_norm(u, eps)
        var = np.var(u)
        assert abs(h.mean()) < 1e-14
        np.testing.assert_allclose(np.mean(h ** 2), var / (var + eps), rtol=1e-12)


def test_concat_order_layer_norm_part_first():
    rng = np.random.default_rng(7)
    d, d_v = 4, 3
    offs, K, V, W_up, _, ids, x = _rand_layer(rng, d=d, d_v=d_v, T=5)
    eye, zero = np.eye(d), np.zeros((d, d))
    fw_x = oracle.forward(offs, K, V, W_up, np.hstack([zero, eye]), ids, x)
    assert np.array_equal(fw_x.y, x)
    fw_h = oracle.forward(offs, K, V, W_up, np.hstack([eye, zero]), ids, x)
    np.testing.assert_allclose(fw_h.y, fw_h.h, rtol=0, atol=1e-15)


def test_w_up_is_out_by_in():
    # W_up is (d x d_v) and u = W_up a: a selection matrix picks components of a
    rng = np.random.default_rng(8)
    d, d_v = 3, 5
    offs, K, V, _, W_mix, ids, x = _rand_layer(rng, d=d, d_v=d_v, T=4)
    W_up = np.zeros((d, d_v))
    W_up[0, 4] = W_up[1, 0] = W_up[2, 2] = 1.0
    fw = oracle.forward(offs, K, V, W_up, W_mix, ids, x)
    np.testing.assert_allclose(fw.u, fw.a[:, [4, 0, 2]], rtol=0, atol=0)


# ---- routing -----------------------------------------------------------------------------------

def test_route_stable_segments():
    ids = np.array([5, 2, 5, 0, 2, 5, 7])
    r = oracle.route(ids)
    assert r.perm.tolist() == [3, 1, 4, 0, 2, 5, 6]
    assert r.seg_start.tolist() == [0, 1, 3, 6, 7]
    assert r.seg_id.tolist() == [0, 2, 5, 7]
    e = oracle.route(np.array([], dtype=np.int64))
    assert e.perm.size == 0 and e.seg_start.tolist() == [0] and e.seg_id.size == 0


# ---- backward ------------------------------------------------------------------------------------

def _loss(offs, K, V, W_up, W_mix, ids, x, dy, eps):
    return float(np.sum(oracle.forward(offs, K, V, W_up, W_mix, ids, x, eps).y * dy))


def test_backward_matches_central_finite_differences():
    rng = np.random.default_rng(9)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, vocab=4, d=4, d_v=3, T=6, n=[3, 1, 2, 4])
    ids = np.array([0, 3, 0, 1, 3, 0])
    dy = rng.standard_normal((6, 4))
    eps = 1e-5
    g = oracle.backward(offs, K, V, W_up, W_mix, ids, x, dy, eps)
    params = {"x": x, "K": K, "V": V, "W_up": W_up, "W_mix": W_mix}
    grads = {"x": g.dx, "K": g.dK, "V": g.dV, "W_up": g.dW_up, "W_mix": g.dW_mix}
    h = 1e-6
    for name, arr in params.items():
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(offs, K, V, W_up, W_mix, ids, x, dy, eps)
            arr[idx] = old - h
            lm = _loss(offs, K, V, W_up, W_mix, ids, x, dy, eps)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        scale = max(1.0, float(np.max(np.abs(num))))
        assert np.max(np.abs(num - grads[name])) <= 1e-6 * scale, name


def test_backward_matches_autograd_fp64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, vocab=7, d=6, d_v=5, T=12)
    dy = rng.standard_normal((12, 6))
    eps = 1e-5
    g = oracle.backward(offs, K, V, W_up, W_mix, ids, x, dy, eps)
    tK, tV, tWu, tWm, tx = (torch.tensor(a, dtype=torch.float64, requires_grad=True)
                            for a in (K, V, W_up, W_mix, x))
    ys = []
    for i, t in enumerate(ids):
        lo, hi = int(offs[t]), int(offs[t + 1])
        p = torch.softmax(tK[lo:hi] @ tx[i], dim=0)
        u = tWu @ (tV[lo:hi].T @ p)
        h = torch.nn.functional.layer_norm(u, (u.shape[0],), eps=eps)
        ys.append(tWm @ torch.cat([h, tx[i]]))
    (torch.stack(ys) * torch.tensor(dy)).sum().backward()
    for ours, t in ((g.dK, tK), (g.dV, tV), (g.dW_up, tWu), (g.dW_mix, tWm), (g.dx, tx)):
        np.testing.assert_allclose(ours, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_gradient_identities():
    # Softmax gradients sum to zero over a token's rows, so the dK rows of a batch of one
    # token sum to (sum_j ds_j) x = 0; rows outside the token's range stay zero.
    rng = np.random.default_rng(11)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, vocab=3, d=4, d_v=3, T=1, n=[2, 5, 3])
    ids = np.array([1])
    dy = rng.standard_normal((1, 4))
    g = oracle.backward(offs, K, V, W_up, W_mix, ids, x, dy)
    r = oracle.token_rows(offs, 1)
    np.testing.assert_allclose(g.dK[r.start:r.stop].sum(axis=0), 0.0, atol=1e-14)
    assert not g.dK[:r.start].any() and not g.dK[r.stop:].any()
    assert not g.dV[:r.start].any() and not g.dV[r.stop:].any()


def test_row_gradients_keep_only_touched_rows_and_match_the_dense_form():
    # the sparse form stores the same sums: the touched ids' rows of dense dK/dV, every
    # other row of the dense form zero, dx and dW unchanged; subsets of tokens and ids
    # select rows of the same results
    rng = np.random.default_rng(12)
    offs, K, V, W_up, W_mix, ids, x = _rand_layer(rng, vocab=7, d=5, d_v=4, T=11)
    dy = rng.standard_normal((11, 5))
    dense = oracle.backward(offs, K, V, W_up, W_mix, ids, x, dy)
    sp = oracle.backward_rows(offs, K, V, W_up, W_mix, ids, x, dy)
    assert sorted(sp.rows) == sorted(set(ids.tolist()))
    touched = np.zeros(int(offs[-1]), bool)
    for t, (gK, gV) in sp.rows.items():
        r = oracle.token_rows(offs, t)
        touched[r.start:r.stop] = True
        np.testing.assert_allclose(gK, dense.dK[r.start:r.stop], rtol=0, atol=1e-13)
        np.testing.assert_allclose(gV, dense.dV[r.start:r.stop], rtol=0, atol=1e-13)
    assert not dense.dK[~touched].any() and not dense.dV[~touched].any()
    np.testing.assert_allclose(sp.dx, dense.dx, atol=1e-13)
    np.testing.assert_allclose(sp.dW_up, dense.dW_up, atol=1e-13)
    np.testing.assert_allclose(sp.dW_mix, dense.dW_mix, atol=1e-13)
    some = [8, 2]
    t0 = int(ids[5])
    sub = oracle.backward_rows(offs, K, V, W_up, W_mix, ids, x, dy, tokens=some, row_ids=[t0],
                               weights=False)
    assert sub.dW_up is None and list(sub.rows) == [t0]
    np.testing.assert_allclose(sub.dx, dense.dx[some], atol=1e-13)
    r = oracle.token_rows(offs, t0)
    np.testing.assert_allclose(sub.rows[t0][0], dense.dK[r.start:r.stop], atol=1e-13)
