"""Builds GPU cases for the parity tests: inputs from l3_workloads, the library's own
offsets (checked bit for bit against the oracle's), device tensors, workspaces, and host
views of the table rows the oracle needs."""
from __future__ import annotations

import numpy as np
import torch

import l3_workloads as W
import oracle
import static_token_routed_csr_b300 as l3

FP32_RTOL = 1e-5      # normwise: max|g - r| / max|r|
BF16_ATOL = 2e-2      # max|g - r| <= 2e-2 * max(1, max|r|)
# Gradients of the fwd+bwd preset: its inputs are bf16 values but every step of the
# backward runs in fp32 (reading "fwd+bwd preset"), so each gradient also meets an
# fp32-level normwise bound; 1e-4 leaves room for fp32 sums of up to 2d terms scaled by
# rstd (up to ~300 here).
GRAD_FP32_RTOL = 1e-4
BF16_U = 2.0 ** -8    # unit roundoff of bf16 (8-bit significand, round to nearest even)


class RowTable:
    """Host copy of only the table rows owned by a set of ids; sliced like the table."""

    def __init__(self, table_dev, offs: np.ndarray, ids):
        ranges = sorted({(int(offs[t]), int(offs[t + 1])) for t in set(int(i) for i in ids)})
        rows = np.concatenate([np.arange(a, b) for a, b in ranges]) if ranges else np.zeros(0, np.int64)
        self.host = W.table_rows_to_numpy(table_dev, rows)
        self._pos = {}
        k = 0
        for a, b in ranges:
            self._pos[(a, b)] = k
            k += b - a

    def __getitem__(self, sl):
        k = self._pos[(sl.start, sl.stop)]
        return self.host[k:k + sl.stop - sl.start]


class Case:
    def __init__(self, cid: int, T=None, shard: int = 0, with_dy=None, ids=None, device="cuda"):
        self.wl = W.make(cid, T=(len(ids) if ids is not None else T), shard=shard, with_dy=with_dy)
        if ids is not None:
            self.wl.ids = np.asarray(ids, dtype=np.int32)
        p = self.p = self.wl.p
        self.T = self.wl.T
        self.offs_np = l3.l3_alloc_offsets(self.wl.freq, p.v, 1, p.k_max, p.power)
        ref = oracle.allocate(self.wl.freq, p.v, 1, p.k_max, p.power)
        assert np.array_equal(self.offs_np.astype(np.int64), ref.offs)
        dt = W.torch_dtype(p)
        self.dt = dt
        self.K, self.V = W.tables(self.wl, device)
        self.offs = torch.as_tensor(self.offs_np, device=device)
        self.W_up = torch.as_tensor(self.wl.W_up, device=device).to(dt).contiguous()
        self.W_mix = torch.as_tensor(self.wl.W_mix, device=device).to(dt).contiguous()
        self.ids = torch.as_tensor(self.wl.ids, device=device)
        self.x = torch.as_tensor(self.wl.x, device=device).to(dt).contiguous()
        self.dy = None if self.wl.dy is None else torch.as_tensor(self.wl.dy, device=device).to(dt).contiguous()
        self.layer = l3.make_layer(self.offs, self.K, self.V, self.W_up, self.W_mix, p.k_max)
        self.ws = torch.empty(max(1, l3.l3_workspace_size(self.layer, self.T, l3.L3_PASS_FORWARD)),
                              dtype=torch.uint8, device=device)

    def forward(self, y_dtype=None, saved=False):
        y = torch.empty((self.T, self.p.d), dtype=y_dtype or self.dt, device=self.x.device)
        sv = None
        if saved:
            sv = torch.empty(max(1, l3.l3_saved_size(self.layer, self.T)), dtype=torch.uint8,
                             device=self.x.device)
        l3.l3_forward(self.layer, self.ids, self.x, y, self.ws, saved=sv)
        return y, sv

    def saved_views(self, sv):
        """(a [T,d_v], ml [T,2], mu [T], rstd [T]) views of a saved-state buffer."""
        T, dv = self.T, self.p.d_v
        f = sv.view(torch.float32)
        al = lambda n: (n * 4 + 255) // 256 * 256 // 4  # noqa: E731  (256-byte aligned carve)
        o = 0
        a = f[o:o + T * dv].view(T, dv)
        o += al(T * dv)
        ml = f[o:o + 2 * T].view(T, 2)
        o += al(2 * T)
        mu = f[o:o + T]
        o += al(T)
        rstd = f[o:o + T]
        return a, ml, mu, rstd

    def host_tables(self, ids=None):
        ids = self.wl.ids if ids is None else ids
        return RowTable(self.K, self.offs_np, ids), RowTable(self.V, self.offs_np, ids)

    def oracle_forward(self, tokens=None):
        sel = range(self.T) if tokens is None else list(tokens)
        Kh, Vh = self.host_tables(self.wl.ids[list(sel)])
        return oracle.forward(self.offs_np, Kh, Vh, self.wl.W_up, self.wl.W_mix, self.wl.ids,
                              self.wl.x, eps=1e-5, tokens=sel)

    def oracle_weights(self, tokens):
        """Per token: (p, V_t rows, a, l) of the oracle's aggregation."""
        Kh, Vh = self.host_tables(self.wl.ids[list(tokens)])
        out = []
        for i in tokens:
            t = int(self.wl.ids[i])
            r0, r1 = int(self.offs_np[t]), int(self.offs_np[t + 1])
            a, _, p, _, l = oracle.attend(Kh[r0:r1], Vh[r0:r1], self.wl.x[i])
            out.append((p, np.asarray(Vh[r0:r1], np.float64), a, l))
        return out

    def long_segment_tokens(self) -> np.ndarray:
        """Mask of the tokens the tensor-core attend takes: in a bf16 batch of at least 1024
        tokens, those whose id has at least 8 tokens in the batch."""
        ids = self.wl.ids
        if self.p.dtype != "bf16" or self.T < 1024:
            return np.zeros(self.T, bool)
        cnt = np.bincount(ids, minlength=self.p.vocab)
        return cnt[ids] >= 8


class RouteOnly:
    """A layer of ``vocab`` ids with one row each, for routing tests only. With the default
    2^20 ids, (id, position) no longer packs into 32-bit sort keys, so routing takes its
    64-bit key path."""

    def __init__(self, T: int, seed: int = 0, vocab: int = 1 << 20, device="cuda"):
        rng = np.random.default_rng([seed, 11])
        pool = rng.integers(0, vocab, 500)
        ids = np.where(rng.random(T) < 0.7, pool[rng.integers(0, 500, T)], rng.integers(0, vocab, T))
        if T >= 2:
            ids[0], ids[-1] = vocab - 1, 0
        self.ids_np = ids.astype(np.int32)
        self.T = T
        bf = torch.bfloat16
        self.offs = torch.arange(vocab + 1, dtype=torch.int32, device=device)
        self.K = torch.zeros((vocab, 64), dtype=bf, device=device)
        self.V = torch.zeros((vocab, 64), dtype=bf, device=device)
        self.W_up = torch.zeros((64, 64), dtype=bf, device=device)
        self.W_mix = torch.zeros((64, 128), dtype=bf, device=device)
        self.layer = l3.make_layer(self.offs, self.K, self.V, self.W_up, self.W_mix, 1)
        self.ids = torch.as_tensor(self.ids_np, device=device)
        self.ws = torch.empty(max(1, l3.l3_workspace_size(self.layer, T, l3.L3_PASS_FORWARD)),
                              dtype=torch.uint8, device=device)


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_fp32_close(g, r, what="", rtol=None):
    rtol = FP32_RTOL if rtol is None else rtol
    g, r = np.asarray(g, np.float64), np.asarray(r, np.float64)
    scale = max(np.max(np.abs(r)), 1e-30)
    err = np.max(np.abs(g - r)) / scale if r.size else 0.0
    assert err <= rtol, f"{what}: normwise relative error {err:.3e} > {rtol}"
    return err


def assert_bf16_close(g, r, what=""):
    g, r = np.asarray(g, np.float64), np.asarray(r, np.float64)
    if r.size == 0:
        return 0.0
    tol = BF16_ATOL * max(1.0, float(np.max(np.abs(r))))
    err = float(np.max(np.abs(g - r)))
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.3e}"
    return err


def assert_rounded_weight_bound(a_gpu, l_gpu, ref_tokens, what=""):
    """Bound of the tensor-core attend, whose MMA takes the softmax weights as bf16.

    Reading "tensor-core attend weights": each weight e_j = exp(s_j - m) is rounded to
    bf16, e_j (1 + d_j) with |d_j| <= u = 2^-8, and a is normalised by the sum of the
    rounded weights. Then a is a convex combination of the value rows whose weights are
    p_j (1 + d_j) / (1 + D) with D = sum_k p_k d_k, so p'_j - p_j = p_j (d_j - D) / (1 + D),
    and because sum_j (p'_j - p_j) = 0:
        |a_c - a_ref,c| <= 2u / (1 - u) * sum_j p_j |V_jc - a_ref,c|
    per token and value column; the saved denominator is within relative u of l. fp32
    accumulation adds a term far below these (1e-6 of max|a| is allowed for it).
    ``ref_tokens``: per token (p, Vt, a_ref, l_ref) from the oracle's aggregation.
    """
    u = BF16_U
    a_gpu = np.asarray(a_gpu, np.float64)
    scale = max(max(float(np.abs(r[2]).max()) for r in ref_tokens), 1e-30)
    for k, (p, Vt, a_ref, l_ref) in enumerate(ref_tokens):
        bound = 2 * u / (1 - u) * (p[:, None] * np.abs(Vt - a_ref[None, :])).sum(0) + 1e-6 * scale
        err = np.abs(a_gpu[k] - a_ref)
        assert np.all(err <= bound), f"{what}: token {k} a off by {err.max():.3e} (bound {bound[err.argmax()]:.3e})"
        assert abs(float(l_gpu[k]) - l_ref) <= (u + 1e-6) * l_ref, f"{what}: token {k} l"


def assert_close(p, g, r, what=""):
    return assert_fp32_close(g, r, what) if p.dtype == "f32" else assert_bf16_close(g, r, what)
