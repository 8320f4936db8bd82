"""GPU parity of the row-gradient backward (l3_backward_rows) against the oracle's
row form of the backward (oracle.backward_rows): dx, the touched rows' dK and dV with
their table indices, dW_up and dW_mix.

Bars: the row indices and their count bit for bit; every gradient within the bf16 bar
max|g - r| <= 2e-2 max(1, max|r|) (this path takes h, x and dy as bf16 operands of the
weight gradients; u, du, da, p and ds reach fp32 accuracy through bf16 hi + lo pairs). Full-size batches compare sampled tokens and ids the
oracle computes one by one, plus the exact row count and the ordering of the row indices.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import l3_workloads as W  # noqa: E402
import static_token_routed_csr_b300 as l3  # noqa: E402
from gpu_case import Case, RowTable, assert_bf16_close, to_np  # noqa: E402


def _touched(case):
    ids = np.unique(case.wl.ids)
    rows = np.concatenate([np.arange(case.offs_np[t], case.offs_np[t + 1]) for t in ids])
    return ids, rows


def _run(case, max_rows=None):
    p, T, dev = case.p, case.T, "cuda"
    _, sv = case.forward(saved=True)
    _, rows = _touched(case)
    cap = len(rows) if max_rows is None else max_rows
    alloc = cap + 16  # rows past the capacity must stay untouched
    out = dict(dx=torch.empty((T, p.d), device=dev),
               row_index=torch.full((alloc,), -1, dtype=torch.int32, device=dev),
               dK=torch.full((alloc, p.d), float("nan"), device=dev),
               dV=torch.full((alloc, p.d_v), float("nan"), device=dev),
               n_rows=torch.zeros(1, dtype=torch.int32, device=dev),
               dW_up=torch.empty((p.d, p.d_v), device=dev), dW_mix=torch.empty((p.d, 2 * p.d), device=dev))
    ws = torch.empty(l3.l3_workspace_size(case.layer, T, l3.L3_PASS_BACKWARD_ROWS), dtype=torch.uint8,
                     device=dev)
    ri = out["row_index"][:cap]
    l3.l3_backward_rows(case.layer, case.ids, case.x, case.dy, sv, out["dx"], ri, out["dK"], out["dV"],
                        out["n_rows"], out["dW_up"], out["dW_mix"], ws)
    torch.cuda.synchronize()
    return out, l3.l3_get_error(ws)


def _check_rows(case, out, ref_rows, ids_checked):
    ri = out["row_index"].cpu().numpy()
    pos = {int(r): k for k, r in enumerate(ri[:int(out["n_rows"].item())])}
    dK, dV = out["dK"], out["dV"]
    for t in ids_checked:
        r0, r1 = int(case.offs_np[t]), int(case.offs_np[t + 1])
        k0 = pos[r0]
        assert [pos[r] for r in range(r0, r1)] == list(range(k0, k0 + r1 - r0))
        gK = to_np(dK[k0:k0 + r1 - r0])
        gV = to_np(dV[k0:k0 + r1 - r0])
        assert_bf16_close(gK, ref_rows[t][0], f"dK rows of id {t}")
        assert_bf16_close(gV, ref_rows[t][1], f"dV rows of id {t}")


def _check_structure(case, out):
    _, rows = _touched(case)
    n = int(out["n_rows"].item())
    assert n == len(rows)
    assert np.array_equal(out["row_index"].cpu().numpy()[:n], rows)  # ascending, exact


@pytest.mark.parametrize("cid,T", [(5, None), (5, 37), (6, None), (2, 600)])
def test_backward_rows_all_outputs(cid, T):
    c = Case(cid, T=T, with_dy=True)
    out, err = _run(c)
    assert err == 0
    _check_structure(c, out)
    Kh, Vh = c.host_tables()
    ref = oracle.backward_rows(c.offs_np, Kh, Vh, c.wl.W_up, c.wl.W_mix, c.wl.ids, c.wl.x, c.wl.dy)
    assert_bf16_close(to_np(out["dx"]), ref.dx, "dx")
    assert_bf16_close(to_np(out["dW_up"]), ref.dW_up, "dW_up")
    assert_bf16_close(to_np(out["dW_mix"]), ref.dW_mix, "dW_mix")
    _check_rows(c, out, ref.rows, sorted(ref.rows))


def test_backward_rows_full_size_large_prefill_sampled():
    c = Case(4, with_dy=True)
    out, err = _run(c)
    assert err == 0
    _check_structure(c, out)
    ids = c.wl.ids
    cnt = np.bincount(ids, minlength=c.p.vocab)
    rng = np.random.default_rng(3)
    toks = np.unique(np.concatenate([rng.choice(c.T, 24, replace=False), [0, c.T - 1]]))
    few = np.nonzero((cnt >= 1) & (cnt <= 12))[0]
    row_ids = np.unique(np.concatenate([rng.choice(few, 6, replace=False), [few.max()]]))
    need = np.unique(np.concatenate([ids[toks], row_ids]))
    Kh, Vh = RowTable(c.K, c.offs_np, need), RowTable(c.V, c.offs_np, need)
    ref = oracle.backward_rows(c.offs_np, Kh, Vh, c.wl.W_up, c.wl.W_mix, ids, c.wl.x, c.wl.dy,
                               tokens=toks, row_ids=row_ids, weights=False)
    assert_bf16_close(to_np(out["dx"][torch.as_tensor(toks, device="cuda")]), ref.dx, "dx sampled")
    _check_rows(c, out, ref.rows, list(row_ids))
    del c, out
    torch.cuda.empty_cache()


def test_backward_rows_is_deterministic():
    c = Case(2, T=2048, with_dy=True)
    o1, _ = _run(c)
    o2, _ = _run(c)
    n = int(o1["n_rows"].item())
    for k in ("dx", "dW_up", "dW_mix"):
        assert torch.equal(o1[k], o2[k]), k
    assert torch.equal(o1["dK"][:n], o2["dK"][:n]) and torch.equal(o1["dV"][:n], o2["dV"][:n])


def test_backward_rows_reports_a_short_row_output():
    c = Case(5, with_dy=True)
    _, rows = _touched(c)
    out, err = _run(c, max_rows=len(rows) - 5)
    assert l3.l3_status_string(err) == "L3_ERR_WORKSPACE"
    assert int(out["n_rows"].item()) == len(rows)
    # nothing was written past the capacity
    cap = len(rows) - 5
    assert torch.isnan(out["dK"][cap:]).all() and torch.isnan(out["dV"][cap:]).all()
    assert (out["row_index"][cap:] == -1).all()
