"""The decode step's operations, one function each, in fp64.

Test infrastructure only (see the package docstring). Arrays are numpy fp64;
matrices are [out_features, in_features]. Conventions the pages leave open
are stated where they are taken (readings R1-R21 of the design notes).
"""
from __future__ import annotations

import numpy as np


def gemv(W: np.ndarray, a: np.ndarray) -> np.ndarray:
    """y = W a: the matrix-vector product that dominates batch-1 decode (Kog, "3k tokens/s
    per request", section "what limits decode speed on GPUs")."""
    return W @ a


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm: y_i = x_i / sqrt(mean_j x_j^2 + eps) * g_i (pre-norm placement, reading R1)."""
    return x / np.sqrt(np.mean(x * x) + eps) * g


def rope(u: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotary embedding of every head row of ``u`` [n_heads, d] at position ``pos``.

    Rotate-half pairing (reading R3): for i < d/2, theta_i = pos * base^(-2i/d) and
    (u_i, u_{i+d/2}) -> (u_i cos - u_{i+d/2} sin, u_i sin + u_{i+d/2} cos).
    """
    d = u.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    theta = pos * base ** (-2.0 * i / d)
    c, s = np.cos(theta), np.sin(theta)
    u1, u2 = u[..., :half], u[..., half:]
    return np.concatenate([u1 * c - u2 * s, u1 * s + u2 * c], axis=-1)


def softmax(s: np.ndarray) -> np.ndarray:
    """exp(s - max s) / sum exp(s - max s)."""
    z = np.exp(s - np.max(s))
    return z / np.sum(z)


def kv_group(h: int, n_q: int, n_kv: int) -> int:
    """kv head of query head h: consecutive groups of n_q/n_kv query heads share one (reading R7)."""
    return h // (n_q // n_kv)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """GQA decode attention of one token: o_h = softmax(q_h K_g^T / sqrt(d)) V_g.

    q [n_q, d]; K, V [n_kv, S, d] (every cached position the token may see, its own
    included). Returns o [n_q, d]. No soft-capping (reading R21).
    """
    n_q, d = q.shape
    n_kv = K.shape[0]
    o = np.empty_like(q)
    for h in range(n_q):
        g = kv_group(h, n_q, n_kv)
        p = softmax(K[g] @ q[h] / np.sqrt(d))
        o[h] = p @ V[g]
    return o


def silu(z):
    """silu(z) = z / (1 + e^-z)."""
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(b, Wg, Wu, Wd):
    """SwiGLU feed-forward: W_d (silu(W_g b) * (W_u b)) (reading R8: gate is the silu branch)."""
    return Wd @ (silu(Wg @ b) * (Wu @ b))


def topk_desc(r: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries, largest first; equal values -> lower index first (R9)."""
    order = np.lexsort((np.arange(len(r)), -r))
    return order[:k]


def route(r: np.ndarray, k: int):
    """Router: top-k experts of the logits r and their weights softmax(r_S) over the selected
    set only, which equals the full softmax renormalised over S (reading R10)."""
    S = topk_desc(r, k)
    return S, softmax(r[S])


def moe_ffn(b, W_router, expert, k, shared_ids, fp32_router_logits=True):
    """MoE feed-forward of one token (Ling-3.0-flash: 8 of 512 routed experts + 1 shared).

    r = W_router b, rounded to fp32 when the router's logits are fp32 (the top-k decision
    is taken at the precision the logits are kept in); S, pi = route(r, k);
    y = sum_{shared s} E_s(b) + sum_{i in S} pi_i E_i(b)  (shared weight 1, no bias, R11).
    ``expert(e)`` returns the fp64 (W_gate, W_up, W_down) of expert e.
    Returns (y, S, pi).
    """
    r = W_router @ b
    if fp32_router_logits:
        r = r.astype(np.float32).astype(np.float64)
    S, pi = route(r, k)
    y = np.zeros(b.shape[0])
    for s in shared_ids:
        y = y + swiglu_ffn(b, *expert(s))
    for e, p in zip(S, pi):
        y = y + p * swiglu_ffn(b, *expert(int(e)))
    return y, S, pi


def argmax_first(logits: np.ndarray) -> int:
    """Greedy token: index of the largest logit, the lowest index among equals (R12)."""
    return int(np.flatnonzero(logits == np.max(logits))[0])


def accepted_prefix(tokens, argmax) -> int:
    """Verify window acceptance (reading R19): tokens[0] is the token fed at pos and tokens[i]
    the draft for pos+i; argmax[i] is the model's choice after position pos+i. Accept the
    longest j with tokens[i+1] == argmax[i] for all i < j, plus the model's bonus token:
    n_accepted = j + 1."""
    j = 0
    while j + 1 < len(tokens) and tokens[j + 1] == argmax[j]:
        j += 1
    return j + 1
