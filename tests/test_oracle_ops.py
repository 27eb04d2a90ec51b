"""Pins of the oracle's operations (CPU only): closed forms, invariants, special
cases and pure-Python brute force on tiny inputs."""
import math

import numpy as np

from oracle import ops


def _loops_gemv(W, a):
    return [sum(W[i][j] * a[j] for j in range(len(a))) for i in range(len(W))]


def test_gemv_brute_force_integer_exact():
    rng = np.random.default_rng(0)
    for (n, k) in [(1, 1), (3, 7), (17, 33), (8, 129)]:
        W = rng.integers(-8, 9, (n, k)).astype(np.float64)
        a = rng.integers(-8, 9, k).astype(np.float64)
        assert ops.gemv(W, a).tolist() == _loops_gemv(W.tolist(), a.tolist())


def test_gemv_orientation():
    # [out, in] layout: row i of W produces output i
    W = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 2.0]])
    assert ops.gemv(W, np.array([3.0, 5.0, 7.0])).tolist() == [3.0, 14.0]
    W = np.array([[1.0, 2.0], [3.0, 4.0]])
    assert ops.gemv(W, np.array([1.0, 0.0])).tolist() == [1.0, 3.0]


def test_rmsnorm_closed_forms():
    x = np.array([3.0, 4.0])
    y = ops.rmsnorm(x, np.ones(2), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(y, [3 / r, 4 / r], rtol=1e-15)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(257)
    y = ops.rmsnorm(x, np.ones(257), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1) < 1e-14          # unit RMS with g = 1
    assert np.allclose(ops.rmsnorm(7.5 * x, np.ones(257), 0.0), y, rtol=1e-14)  # scale invariance
    g = rng.standard_normal(257)
    assert np.allclose(ops.rmsnorm(x, g, 0.0), y * g, rtol=1e-14)  # gain multiplies elementwise
    # eps enters under the root: x = 0 -> 0, and a tiny x is damped
    eps = 1e-6
    small = np.full(4, 1e-3)
    assert np.allclose(ops.rmsnorm(small, np.ones(4), eps), small / math.sqrt(1e-6 + eps), rtol=1e-14)


def test_rope_pos0_identity_and_rotation_form():
    rng = np.random.default_rng(2)
    u = rng.standard_normal((3, 128))
    assert np.array_equal(ops.rope(u, 0, 1e4), u)
    # basis vector e_i (i < 64) rotates into the (i, i+64) plane by theta_i = pos * base^(-2i/d)
    for i in (0, 1, 31, 63):
        e = np.zeros((1, 128))
        e[0, i] = 1.0
        pos = 37
        th = pos * 1e4 ** (-2 * i / 128)
        r = ops.rope(e, pos, 1e4)[0]
        want = np.zeros(128)
        want[i], want[i + 64] = math.cos(th), math.sin(th)
        assert np.allclose(r, want, atol=1e-15)
        e2 = np.zeros((1, 128))
        e2[0, i + 64] = 1.0
        r2 = ops.rope(e2, pos, 1e4)[0]
        want2 = np.zeros(128)
        want2[i], want2[i + 64] = -math.sin(th), math.cos(th)
        assert np.allclose(r2, want2, atol=1e-15)


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    for p in (1, 100, 4097):
        assert abs(np.linalg.norm(ops.rope(q, p, 1e4)) - np.linalg.norm(q)) < 1e-12
    d1 = float(ops.rope(q, 10, 1e4)[0] @ ops.rope(k, 3, 1e4)[0])
    d2 = float(ops.rope(q, 1010, 1e4)[0] @ ops.rope(k, 1003, 1e4)[0])
    assert abs(d1 - d2) < 1e-10
    # the first pair turns by exactly pos radians (theta_0 = pos)
    e = np.zeros((1, 128))
    e[0, 0] = 1
    assert abs(ops.rope(e, 2, 1e4)[0, 0] - math.cos(2.0)) < 1e-15


def test_softmax_sums_to_one_and_brute_force():
    rng = np.random.default_rng(4)
    s = rng.standard_normal(50) * 10
    p = ops.softmax(s)
    assert abs(p.sum() - 1) < 1e-15
    m = max(s)
    z = [math.exp(v - m) for v in s]
    assert np.allclose(p, [v / sum(z) for v in z], rtol=1e-14)
    assert np.allclose(ops.softmax(s + 1000.0), p, rtol=1e-13)


def _loops_attention(q, K, V):
    n_q, d = len(q), len(q[0])
    n_kv = len(K)
    grp = n_q // n_kv
    out = []
    for h in range(n_q):
        g = h // grp
        sc = [sum(q[h][i] * K[g][j][i] for i in range(d)) / math.sqrt(d) for j in range(len(K[g]))]
        m = max(sc)
        z = [math.exp(v - m) for v in sc]
        t = sum(z)
        out.append([sum(z[j] / t * V[g][j][i] for j in range(len(z))) for i in range(d)])
    return out


def test_attention_brute_force_gqa():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((6, 8))
    K = rng.standard_normal((2, 5, 8))
    V = rng.standard_normal((2, 5, 8))
    got = ops.attention(q, K, V)
    want = _loops_attention(q.tolist(), K.tolist(), V.tolist())
    assert np.allclose(got, want, rtol=1e-13, atol=1e-14)
    # GQA grouping: heads 0-2 share kv head 0, heads 3-5 kv head 1
    assert [ops.kv_group(h, 6, 2) for h in range(6)] == [0, 0, 0, 1, 1, 1]


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 16))
    V = rng.standard_normal((2, 1, 16))
    K = rng.standard_normal((2, 1, 16))
    o = ops.attention(q, K, V)                          # one position: output is V exactly
    assert np.array_equal(o[0], V[0, 0]) and np.array_equal(o[3], V[1, 0])
    K = np.tile(rng.standard_normal((1, 1, 16)), (2, 7, 1))   # all keys equal: mean of V
    V = rng.standard_normal((2, 7, 16))
    o = ops.attention(q, K, V)
    assert np.allclose(o[0], V[0].mean(0), rtol=1e-13) and np.allclose(o[2], V[1].mean(0), rtol=1e-13)
    K = np.zeros((2, 7, 16))                            # one key far ahead: its V
    K[:, 4] = q[0] * 1e3
    o = ops.attention(q[:1].repeat(2, 0), K, V)
    assert np.allclose(o[0], V[0, 4], atol=1e-12)
    # n_kv == n_q is plain multi-head attention
    K = rng.standard_normal((4, 9, 16))
    V = rng.standard_normal((4, 9, 16))
    o = ops.attention(q, K, V)
    for h in range(4):
        p = ops.softmax(K[h] @ q[h] / 4.0)
        assert np.allclose(o[h], p @ V[h], rtol=1e-13)


def test_silu_and_swiglu():
    assert ops.silu(0.0) == 0.0
    assert abs(ops.silu(1.0) - 1 / (1 + math.exp(-1))) < 1e-16
    assert abs(ops.silu(40.0) - 40.0) < 1e-12 and abs(ops.silu(-40.0)) < 1e-15
    Wg = np.array([[1.0, 0.0], [0.0, 1.0]])
    Wu = np.array([[2.0, 0.0], [0.0, 3.0]])
    Wd = np.array([[1.0, 1.0]])
    b = np.array([1.0, -2.0])
    want = ops.silu(1.0) * 2.0 + ops.silu(-2.0) * (-6.0)
    assert abs(ops.swiglu_ffn(b, Wg, Wu, Wd)[0] - want) < 1e-15


def test_topk_brute_force_and_ties():
    rng = np.random.default_rng(7)
    for _ in range(20):
        r = rng.integers(-5, 5, 64).astype(np.float64)     # many ties
        k = 8
        want = sorted(range(64), key=lambda i: (-r[i], i))[:k]
        assert ops.topk_desc(r, k).tolist() == want
    S, pi = ops.route(np.array([0.0, 3.0, 1.0, 3.0]), 2)
    assert S.tolist() == [1, 3] and np.allclose(pi, [0.5, 0.5])


def test_route_equals_renormalised_full_softmax():
    rng = np.random.default_rng(8)
    r = rng.standard_normal(512)
    S, pi = ops.route(r, 8)
    full = ops.softmax(r)
    assert np.allclose(pi, full[S] / full[S].sum(), rtol=1e-13)
    assert abs(pi.sum() - 1) < 1e-15 and np.all(np.diff(pi) <= 0)


def test_moe_special_cases():
    rng = np.random.default_rng(9)
    H, I, E = 12, 6, 10
    Wg, Wu, Wd = rng.standard_normal((I, H)), rng.standard_normal((I, H)), rng.standard_normal((H, I))
    zero = (np.zeros((I, H)), np.zeros((I, H)), np.zeros((H, I)))
    b = rng.standard_normal(H)
    Wr = rng.standard_normal((E, H))
    # identical routed experts, zero shared: output equals one expert (weights sum to 1)
    y, S, pi = ops.moe_ffn(b, Wr, lambda e: zero if e == E else (Wg, Wu, Wd), 4, [E], fp32_router_logits=False)
    assert np.allclose(y, ops.swiglu_ffn(b, Wg, Wu, Wd), rtol=1e-13)
    # k = 1: only the argmax expert, weight 1
    experts = [(rng.standard_normal((I, H)), rng.standard_normal((I, H)), rng.standard_normal((H, I))) for _ in range(E)]
    y, S, pi = ops.moe_ffn(b, Wr, lambda e: zero if e == E else experts[e], 1, [E], fp32_router_logits=False)
    top = int(np.argmax(Wr @ b))
    assert S.tolist() == [top] and pi.tolist() == [1.0]
    assert np.allclose(y, ops.swiglu_ffn(b, *experts[top]), rtol=1e-13)
    # shared expert added with weight 1 on top of the routed ones
    y2, _, _ = ops.moe_ffn(b, Wr, lambda e: (Wg, Wu, Wd) if e == E else experts[e], 1, [E], fp32_router_logits=False)
    assert np.allclose(y2 - y, ops.swiglu_ffn(b, Wg, Wu, Wd), rtol=1e-12, atol=1e-12)


def test_argmax_and_acceptance():
    assert ops.argmax_first(np.array([1.0, 5.0, 5.0, 2.0])) == 1
    assert ops.accepted_prefix([7, 1, 2, 3], [1, 2, 3, 9]) == 4
    assert ops.accepted_prefix([7, 1, 2, 3], [1, 5, 3, 9]) == 2
    assert ops.accepted_prefix([7, 1, 2, 3], [4, 2, 3, 9]) == 1
    assert ops.accepted_prefix([7], [4]) == 1
