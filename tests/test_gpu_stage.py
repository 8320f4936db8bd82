"""Staging a batch's rows from host-resident tables (l3_stage_rows): the staged layer gives
the forward the same outputs, bit for bit, as the full tables in device memory; the staged
ids, offsets and rows are the batch's distinct ids in increasing order ("Systems-Friendly
Design", gist.science explainer: tables in CPU memory, the rows a batch needs fetched
ahead because routing is static)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import static_token_routed_csr_b300 as l3  # noqa: E402
from gpu_case import Case, assert_close, to_np  # noqa: E402


def _stage(c, K_h, V_h, max_rows):
    L_h = l3.make_layer(c.offs, K_h, V_h, c.W_up, c.W_mix, c.p.k_max)
    T, dev = c.T, "cuda"
    K_s = torch.empty((max_rows, c.p.d), dtype=c.dt, device=dev)
    V_s = torch.empty((max_rows, c.p.d_v), dtype=c.dt, device=dev)
    offs_s = torch.full((T + 1,), -1, dtype=torch.int32, device=dev)
    ids_s = torch.full((T,), -1, dtype=torch.int32, device=dev)
    n_rows = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(l3.l3_workspace_size(L_h, T, l3.L3_PASS_STAGE), dtype=torch.uint8, device=dev)
    staged = l3.l3_stage_rows(L_h, c.ids, K_s, V_s, offs_s, ids_s, n_rows, ws)
    torch.cuda.synchronize()
    return staged, K_s, V_s, offs_s, ids_s, n_rows, ws


@pytest.mark.parametrize("cid,T", [(2, 1000), (3, 64), (5, None)])
def test_staged_forward_equals_device_forward(cid, T):
    c = Case(cid, T=T)
    y_dev, _ = c.forward()
    K_h, V_h = c.K.cpu().pin_memory(), c.V.cpu().pin_memory()
    uniq = np.unique(c.wl.ids)
    n = np.diff(c.offs_np.astype(np.int64))[uniq]
    U = int(n.sum())
    staged, K_s, V_s, offs_s, ids_s, n_rows, ws = _stage(c, K_h, V_h, U + c.T)
    assert l3.l3_get_error(ws) == 0
    assert int(n_rows.item()) == U
    S = len(uniq)
    r = oracle.route(c.wl.ids)
    assert np.array_equal(r.seg_id, uniq)
    seg_of = np.searchsorted(uniq, c.wl.ids)
    assert np.array_equal(ids_s.cpu().numpy(), seg_of)
    assert np.array_equal(offs_s.cpu().numpy()[:S + 1], np.concatenate([[0], np.cumsum(n)]))
    rows = np.concatenate([np.arange(c.offs_np[t], c.offs_np[t + 1]) for t in uniq])
    assert torch.equal(K_s[:U].cpu(), K_h[torch.as_tensor(rows)])
    assert torch.equal(V_s[:U].cpu(), V_h[torch.as_tensor(rows)])
    y_st = torch.empty_like(y_dev)
    ws_f = torch.empty(l3.l3_workspace_size(staged, c.T, l3.L3_PASS_FORWARD), dtype=torch.uint8,
                       device="cuda")
    l3.l3_forward(staged, ids_s, c.x, y_st, ws_f)
    torch.cuda.synchronize()
    assert l3.l3_get_error(ws_f) == 0
    assert torch.equal(y_st, y_dev)
    toks = list(range(0, c.T, max(1, c.T // 16)))
    assert_close(c.p, to_np(y_st)[toks], c.oracle_forward(tokens=toks).y, "staged y")


def test_stage_reports_short_capacity_and_rejects_pageable_tables():
    c = Case(5)
    K_h, V_h = c.K.cpu().pin_memory(), c.V.cpu().pin_memory()
    *_, ws = _stage(c, K_h, V_h, c.T)  # far fewer rows than the batch touches
    assert l3.l3_status_string(l3.l3_get_error(ws)) == "L3_ERR_WORKSPACE"
    with pytest.raises(l3.L3Error) as e:
        _stage(c, c.K.cpu(), c.V.cpu(), 4 * c.T)
    assert e.value.status == 1
