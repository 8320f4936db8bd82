"""CPU fp64 oracle for the Large Lookup Layer (L³) — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline and
reference legs) may import this module. The CUDA library never calls it, and it shares no
code with the library: no kernels, headers, helpers or constants.

Sources (pages on arXiv:2601.21461, "L³: Large Lookup Layers", Tseng & De Sa):

* [gist] the gist.science explainer of the paper (English page; the German and Dutch pages
  translate it), section "Technical Summary":
  - "Core Architecture": inputs are a hidden state x and a token id t; static routing
    fixes t's subset of a large embedding table; attention of x over the keys K_t and
    values V_t; the layer output is W_mix [LayerNorm(W_up(V_tᵀ Softmax(K_t x))); x].
  - "Information-Theoretic Embedding Allocation": a budget of v embeddings is spread over
    the vocabulary, every token gets at least 1 and at most k rows, and the result is
    heavy-tailed (frequent tokens get many rows).
  - "Systems-Friendly Design": sorting a batch by token id makes the layer's attention
    mask block-diagonal.
* [abs] the arXiv abstract (aiqbench.com and fugumt.com pages): static token-based
  routing aggregates a set of learned embeddings per token in a context-dependent way.

Readings where the pages are silent (each is listed in the design notes):

* no softmax temperature (the formula shows a bare Softmax(K_t x));
* LayerNorm over the d features, biased variance, eps passed in (1e-5), no affine;
* no biases, no residual; W matrices are (out x in); the concatenation puts the LayerNorm
  part first and x second, as the formula stacks them;
* the row allocation replaces the corpus-driven Algorithm 1 (not on the pages) by a
  frequency rule: weights freq^power, water-filled into [n_min, n_max] so that they sum
  to v, rounded by largest remainder (ties to the lower id).

Every function computes in fp64 with plain per-token loops; a library primitive (matrix
product, sort) serves only as one step of the definition. Tables may be fp32 arrays or
any object whose ``[r0:r1]`` slice gives those rows as numbers.
"""
from __future__ import annotations

import math
from typing import NamedTuple

import numpy as np


# --------------------------------------------------------------------------------------
# Allocation: how many rows each token id owns ([gist] "Information-Theoretic Embedding
# Allocation": 1 <= n_t <= k, sum n_t = v, heavy-tailed by frequency).
# --------------------------------------------------------------------------------------

class Allocation(NamedTuple):
    n: np.ndarray        # [vocab] int64, rows per id
    offs: np.ndarray     # [vocab+1] int64, CSR offsets (exclusive prefix sum of n)
    target: np.ndarray   # [vocab] fp64, real-valued water-filled targets r_i


def _fill_level(w: np.ndarray, c: float, n_min: float, n_max: float) -> float:
    """sum_i clamp(c*w_i, n_min, n_max), summed left to right in id order."""
    return float(np.cumsum(np.minimum(np.maximum(c * w, n_min), n_max))[-1])


def allocate(freq, v: int, n_min: int, n_max: int, power: float) -> Allocation:
    """Rows per token id, proportional to freq^power and clamped to [n_min, n_max].

    1. w_i = pow(freq_i, power) (C library pow).
    2. Water level c with sum_i clamp(c w_i, n_min, n_max) = v: 200 bisection steps on
       [0, 2 n_max / min w] locate the clamped sets H (c w_i >= n_max) and L
       (c w_i <= n_min); then c* = (v - n_max|H| - n_min|L|) / sum_{free} w_i exactly
       for that active set, the free sum taken in increasing id order.
    3. r_i = n_max on H, n_min on L, clamp(c* w_i) otherwise.
    4. n_i = floor(r_i); the D = v - sum floor(r_i) ids with the largest r_i - floor(r_i)
       among those with floor(r_i) < n_max get one more row (ties go to the lower id).
    """
    freq = np.asarray(freq, dtype=np.float64)
    N = freq.shape[0]
    if N < 1 or n_min < 1 or n_max < n_min:
        raise ValueError("bad allocation arguments")
    if not (N * n_min <= v <= N * n_max):
        raise ValueError("infeasible: need vocab*n_min <= v <= vocab*n_max")
    if np.any(~np.isfinite(freq)) or np.any(freq <= 0):
        raise ValueError("frequencies must be positive and finite")
    w = np.array([math.pow(float(f), float(power)) for f in freq], dtype=np.float64)
    lo_c, hi_c = 0.0, 2.0 * n_max / float(w.min())
    for _ in range(200):
        mid = 0.5 * (lo_c + hi_c)
        if _fill_level(w, mid, float(n_min), float(n_max)) < v:
            lo_c = mid
        else:
            hi_c = mid
    cw = hi_c * w
    in_h = cw >= n_max
    in_l = (cw <= n_min) & ~in_h
    free = ~(in_h | in_l)
    r = np.where(in_h, float(n_max), float(n_min)).astype(np.float64)
    if free.any():
        s_free = float(np.cumsum(w[free])[-1])
        c_star = (float(v) - float(n_max) * int(in_h.sum()) - float(n_min) * int(in_l.sum())) / s_free
        r[free] = np.minimum(np.maximum(c_star * w[free], float(n_min)), float(n_max))
    f = np.floor(r).astype(np.int64)
    D = int(v - int(f.sum()))
    eligible = [i for i in range(N) if f[i] < n_max]
    if D < 0 or D > len(eligible):
        raise ValueError("apportionment failed")
    rem = r - f
    order = sorted(eligible, key=lambda i: (-rem[i], i))
    n = f.copy()
    for i in order[:D]:
        n[i] += 1
    offs = np.zeros(N + 1, dtype=np.int64)
    offs[1:] = np.cumsum(n)
    return Allocation(n, offs, r)


# --------------------------------------------------------------------------------------
# Frequencies from a token stream ([gist] "Information-Theoretic Embedding Allocation":
# the allocation follows how often each token occurs; a stream of token ids stands in
# for the training corpus, whose corpus-driven Algorithm 1 is not on the pages).
# --------------------------------------------------------------------------------------

def count_ids(ids, vocab: int) -> np.ndarray:
    """Occurrences of each id 0..vocab-1 in the stream (int64). Ids outside [0, vocab)
    are an error."""
    ids = np.asarray(ids, dtype=np.int64)
    if ids.size and (ids.min() < 0 or ids.max() >= vocab):
        raise ValueError("token id outside [0, vocab)")
    return np.bincount(ids, minlength=vocab).astype(np.int64)


def allocate_from_counts(counts, v: int, n_min: int, n_max: int, power: float,
                         smoothing: float) -> Allocation:
    """The frequency allocation with freq_t = count_t + smoothing (add-smoothing keeps an
    id that never occurred at a positive frequency; the clamp gives it n_min rows)."""
    freq = np.asarray(counts, dtype=np.int64).astype(np.float64) + float(smoothing)
    return allocate(freq, v, n_min, n_max, power)


# --------------------------------------------------------------------------------------
# Routing ([gist] "Core Architecture": static routing, t alone selects rows;
# "Systems-Friendly Design": sorting the batch by token id).
# --------------------------------------------------------------------------------------

class Route(NamedTuple):
    perm: np.ndarray       # [T] int64: sorted position -> original token index (stable)
    seg_start: np.ndarray  # [S+1] int64: segment s holds sorted positions seg_start[s]..seg_start[s+1]-1
    seg_id: np.ndarray     # [S] int64: token id of segment s (increasing)


def route(ids) -> Route:
    """Stable sort of token ids; one segment per distinct id, in increasing id order."""
    ids = np.asarray(ids, dtype=np.int64)
    perm = np.argsort(ids, kind="stable")
    starts, seg_id = [], []
    for q in range(len(perm)):
        if q == 0 or ids[perm[q]] != ids[perm[q - 1]]:
            starts.append(q)
            seg_id.append(int(ids[perm[q]]))
    starts.append(len(perm))
    return Route(perm.astype(np.int64), np.array(starts, dtype=np.int64), np.array(seg_id, dtype=np.int64))


def token_rows(offs, t: int) -> range:
    """Row ids owned by token id t: offs[t] .. offs[t+1]-1 (a contiguous CSR range)."""
    return range(int(offs[t]), int(offs[t + 1]))


# --------------------------------------------------------------------------------------
# Forward ([gist] "Core Architecture", the layer formula), one token at a time.
# --------------------------------------------------------------------------------------

def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def attend(Kt, Vt, x):
    """Context-dependent aggregation of one token's rows.

    s = K_t x; p = softmax(s) (no temperature); a = V_tᵀ p.
    Returns (a, s, p, m, l) with m = max s and l = sum exp(s - m).
    """
    Kt, Vt, x = _f64(Kt), _f64(Vt), _f64(x)
    s = Kt @ x
    m = float(np.max(s))
    e = np.exp(s - m)
    l = float(np.sum(e))
    p = e / l
    a = Vt.T @ p
    return a, s, p, m, l


def layer_norm(u, eps: float):
    """LayerNorm without affine: h = (u - mean u) / sqrt(mean((u - mean u)^2) + eps)."""
    u = _f64(u)
    mu = float(np.mean(u))
    var = float(np.mean((u - mu) ** 2))
    rstd = 1.0 / math.sqrt(var + eps)
    return (u - mu) * rstd, mu, rstd


class Forward(NamedTuple):
    y: np.ndarray     # [T, d]
    a: np.ndarray     # [T, d_v]  V_tᵀ p
    u: np.ndarray     # [T, d]    W_up a
    h: np.ndarray     # [T, d]    LayerNorm(u)
    mu: np.ndarray    # [T]
    rstd: np.ndarray  # [T]
    m: np.ndarray     # [T] max score
    l: np.ndarray     # [T] softmax denominator, relative to m


def forward_token(offs, K, V, W_up, W_mix, t: int, x, eps: float):
    """y = W_mix [LayerNorm(W_up(V_tᵀ Softmax(K_t x))); x] for one token."""
    rows = token_rows(offs, t)
    Kt = _f64(K[rows.start:rows.stop])
    Vt = _f64(V[rows.start:rows.stop])
    a, _, _, m, l = attend(Kt, Vt, x)
    u = _f64(W_up) @ a
    h, mu, rstd = layer_norm(u, eps)
    c = np.concatenate([h, _f64(x)])
    y = _f64(W_mix) @ c
    return y, a, u, h, mu, rstd, m, l


def forward(offs, K, V, W_up, W_mix, ids, x, eps: float = 1e-5, tokens=None) -> Forward:
    """The layer over a batch, each token independently (``tokens`` picks a subset)."""
    ids = np.asarray(ids)
    x = np.asarray(x)
    sel = range(len(ids)) if tokens is None else list(tokens)
    d = np.asarray(W_mix).shape[0]
    d_v = np.asarray(W_up).shape[1]
    n = len(sel)
    out = Forward(np.zeros((n, d)), np.zeros((n, d_v)), np.zeros((n, d)), np.zeros((n, d)),
                  np.zeros(n), np.zeros(n), np.zeros(n), np.zeros(n))
    for j, i in enumerate(sel):
        y, a, u, h, mu, rstd, m, l = forward_token(offs, K, V, W_up, W_mix, int(ids[i]), x[i], eps)
        out.y[j], out.a[j], out.u[j], out.h[j] = y, a, u, h
        out.mu[j], out.rstd[j], out.m[j], out.l[j] = mu, rstd, m, l
    return out


def attend_dense_masked(offs, K, V, ids, x):
    """The aggregation written as attention over ALL v rows with a block mask.

    Token i may attend only to rows offs[t_i]..offs[t_i+1]-1 (score -inf elsewhere); this
    is the masked form that sorting by id makes block-diagonal ([gist] "Systems-Friendly
    Design"). Returns a [T, d_v].
    """
    K, V = _f64(K), _f64(V)
    ids = np.asarray(ids)
    out = np.zeros((len(ids), V.shape[1]))
    for i in range(len(ids)):
        s = K @ _f64(x[i])
        mask = np.full(K.shape[0], -np.inf)
        r = token_rows(offs, int(ids[i]))
        mask[r.start:r.stop] = 0.0
        s = s + mask
        e = np.exp(s - np.max(s))
        out[i] = V.T @ (e / e.sum())
    return out


# --------------------------------------------------------------------------------------
# Backward: the chain rule of the layer formula, one token at a time.
# --------------------------------------------------------------------------------------

class Backward(NamedTuple):
    dx: np.ndarray      # [T, d]
    dK: np.ndarray      # [v, d]
    dV: np.ndarray      # [v, d_v]
    dW_up: np.ndarray   # [d, d_v]
    dW_mix: np.ndarray  # [d, 2d]


def backward_token(offs, K, V, W_up, W_mix, t: int, x, g, eps: float):
    """The chain rule of the layer formula for one token (id t, input x, upstream dy = g).

    Forward values s, p, a, u, h, mu, rstd of the token, then:
      dW_mix term: g cᵀ with c = [h; x];  dc = W_mixᵀ g;  dh = dc[:d];  dx = dc[d:]
      du = rstd (dh - mean(dh) - h mean(dh h))          (LayerNorm, no affine)
      dW_up term: du aᵀ;  da = W_upᵀ du
      dp_j = V_j . da;  ds_j = p_j (dp_j - sum_k p_k dp_k)   (softmax)
      dx += K_Rᵀ ds;  dK[R] term: ds xᵀ;  dV[R] term: p daᵀ
    Returns (dx, dK_rows, dV_rows, dW_up term, dW_mix term) for the rows R of id t.
    """
    W_up, W_mix = _f64(W_up), _f64(W_mix)
    d = W_up.shape[0]
    rows = token_rows(offs, t)
    Kt = _f64(K[rows.start:rows.stop])
    Vt = _f64(V[rows.start:rows.stop])
    xi = _f64(x)
    g = _f64(g)
    a, _, p, _, _ = attend(Kt, Vt, xi)
    u = W_up @ a
    h, _, rstd = layer_norm(u, eps)
    c = np.concatenate([h, xi])
    dc = W_mix.T @ g
    dh = dc[:d]
    du = rstd * (dh - np.mean(dh) - h * np.mean(dh * h))
    da = W_up.T @ du
    dp = Vt @ da
    ds = p * (dp - np.dot(p, dp))
    dx = dc[d:] + Kt.T @ ds
    return dx, np.outer(ds, xi), np.outer(p, da), np.outer(du, a), np.outer(g, c)


def backward(offs, K, V, W_up, W_mix, ids, x, dy, eps: float = 1e-5) -> Backward:
    """Gradients of sum(dy * y) for the layer formula, in fp64, dense dK and dV
    (``backward_token`` per token, summed)."""
    W_up, W_mix = _f64(W_up), _f64(W_mix)
    ids = np.asarray(ids)
    d, d_v = W_up.shape
    v = int(offs[-1])
    dx = np.zeros((len(ids), d))
    dK = np.zeros((v, d))
    dV = np.zeros((v, d_v))
    dW_up = np.zeros((d, d_v))
    dW_mix = np.zeros((d, 2 * d))
    for i in range(len(ids)):
        t = int(ids[i])
        rows = token_rows(offs, t)
        dx[i], gK, gV, gu, gm = backward_token(offs, K, V, W_up, W_mix, t, x[i], dy[i], eps)
        dK[rows.start:rows.stop] += gK
        dV[rows.start:rows.stop] += gV
        dW_up += gu
        dW_mix += gm
    return Backward(dx, dK, dV, dW_up, dW_mix)


class SparseBackward(NamedTuple):
    dx: np.ndarray      # [len(tokens), d] for the requested tokens
    rows: dict          # id t -> (dK rows [n_t, d], dV rows [n_t, d_v]), summed over t's tokens
    dW_up: object       # [d, d_v], or None when not requested
    dW_mix: object      # [d, 2d], or None


def backward_rows(offs, K, V, W_up, W_mix, ids, x, dy, eps: float = 1e-5, tokens=None,
                  row_ids=None, weights: bool = True) -> SparseBackward:
    """The same gradients with dK and dV kept only for the rows the batch touches.

    ``tokens``: the tokens whose dx is returned (default all). ``row_ids``: the ids whose
    row gradients are returned (default every id in the batch); each sums over all of
    that id's tokens in the batch. ``weights``: also sum dW_up and dW_mix over all tokens.
    Only the tokens these outputs need are visited.
    """
    ids = np.asarray(ids)
    W_up, W_mix = _f64(W_up), _f64(W_mix)
    d, d_v = W_up.shape
    tok = list(range(len(ids))) if tokens is None else [int(i) for i in tokens]
    want = set(int(t) for t in (np.unique(ids) if row_ids is None else row_ids))
    visit = range(len(ids)) if weights else sorted(set(tok) | {i for i in range(len(ids))
                                                                  if int(ids[i]) in want})
    pos = {i: j for j, i in enumerate(tok)}
    dx = np.zeros((len(tok), d))
    rows = {t: (np.zeros((len(token_rows(offs, t)), d)), np.zeros((len(token_rows(offs, t)), d_v)))
            for t in want}
    dW_up = np.zeros((d, d_v)) if weights else None
    dW_mix = np.zeros((d, 2 * d)) if weights else None
    for i in visit:
        t = int(ids[i])
        gx, gK, gV, gu, gm = backward_token(offs, K, V, W_up, W_mix, t, x[i], dy[i], eps)
        if i in pos:
            dx[pos[i]] = gx
        if t in rows:
            rows[t][0][:] += gK
            rows[t][1][:] += gV
        if weights:
            dW_up += gu
            dW_mix += gm
    return SparseBackward(dx, rows, dW_up, dW_mix)
