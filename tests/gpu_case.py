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


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_fp32_close(g, r, what=""):
    g, r = np.asarray(g, np.float64), np.asarray(r, np.float64)
    scale = max(np.max(np.abs(r)), 1e-30)
    err = np.max(np.abs(g - r)) / scale if r.size else 0.0
    assert err <= FP32_RTOL, f"{what}: normwise relative error {err:.3e} > {FP32_RTOL}"
    return err


def assert_bf16_close(g, r, what=""):
    g, r = np.asarray(g, np.float64), np.asarray(r, np.float64)
    if r.size == 0:
        return 0.0
    tol = BF16_ATOL * max(1.0, float(np.max(np.abs(r))))
    err = float(np.max(np.abs(g - r)))
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.3e}"
    return err


def assert_close(p, g, r, what=""):
    return assert_fp32_close(g, r, what) if p.dtype == "f32" else assert_bf16_close(g, r, what)
