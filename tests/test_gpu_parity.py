"""GPU parity: the CUDA library (through the C ABI) against the CPU fp64 oracle.

Bars: routing and offsets bit-exact; fp32 layers normwise relative error <= 1e-5; bf16
layers max abs error <= 2e-2 * max(1, max|ref|). Full-size presets run in the launch
configuration the benchmark times and compare sampled tokens, which the oracle computes
one by one.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a CUDA device", allow_module_level=True)

import l3_workloads as W  # noqa: E402
import static_token_routed_csr_b300 as l3  # noqa: E402
from gpu_case import (BF16_U, GRAD_FP32_RTOL, Case, assert_close, assert_fp32_close,  # noqa: E402
                      RouteOnly, assert_rounded_weight_bound, to_np)


def _route(case):
    T = case.T
    dev = case.ids.device
    perm = torch.full((max(T, 1),), -7, dtype=torch.int32, device=dev)
    seg_start = torch.full((T + 1,), -7, dtype=torch.int32, device=dev)
    seg_id = torch.full((max(T, 1),), -7, dtype=torch.int32, device=dev)
    n_seg = torch.full((1,), -7, dtype=torch.int32, device=dev)
    l3.l3_route(case.layer, case.ids, case.ws, perm, seg_start, seg_id, n_seg)
    torch.cuda.synchronize()
    S = int(n_seg.item())
    return perm.cpu().numpy()[:T], seg_start.cpu().numpy()[:S + 1], seg_id.cpu().numpy()[:S], S


# ---- routing ---------------------------------------------------------------------------------

@pytest.mark.parametrize("cid,T", [(1, None), (2, None), (3, None), (1, 1), (2, 4096), (2, 4097),
                                   (2, 12289), (4, None)])
def test_route_bit_exact(cid, T):
    c = Case(cid, T=T)
    perm, seg_start, seg_id, S = _route(c)
    ref = oracle.route(c.wl.ids)
    assert S == len(ref.seg_id)
    assert np.array_equal(perm, ref.perm)
    assert np.array_equal(seg_start, ref.seg_start)
    assert np.array_equal(seg_id, ref.seg_id)
    assert l3.l3_get_error(c.ws) == 0


@pytest.mark.parametrize("T", [3000, 40000])  # one CTA sort; sorted runs of 4096 and 4 merge passes
def test_route_wide_vocab_bit_exact(T):
    c = RouteOnly(T)
    perm, seg_start, seg_id, S = _route(c)
    ref = oracle.route(c.ids_np)
    assert S == len(ref.seg_id)
    assert np.array_equal(perm, ref.perm)
    assert np.array_equal(seg_start, ref.seg_start)
    assert np.array_equal(seg_id, ref.seg_id)
    assert l3.l3_get_error(c.ws) == 0


def test_route_all_equal_ids_and_reverse_order():
    ids = np.full(9000, 3, dtype=np.int32)
    c = Case(1, ids=ids)
    perm, seg_start, seg_id, S = _route(c)
    assert S == 1 and np.array_equal(perm, np.arange(9000)) and seg_id.tolist() == [3]
    ids = np.arange(255, -1, -1, dtype=np.int32).repeat(20)
    c = Case(1, ids=ids)
    perm, seg_start, seg_id, S = _route(c)
    ref = oracle.route(ids)
    assert np.array_equal(perm, ref.perm) and np.array_equal(seg_start, ref.seg_start)


def test_token_id_out_of_range_is_reported_not_trapped():
    ids = np.array([0, 5, 256, 7, -1], dtype=np.int32)  # vocab is 256
    c = Case(1, ids=ids)
    y, _ = c.forward()
    assert l3.l3_get_error(c.ws) == 5
    # the valid tokens are still right
    fw = c.oracle_forward(tokens=[0, 1, 3])
    assert_fp32_close(to_np(y)[[0, 1, 3]], fw.y, "valid rows")
    assert l3.l3_get_error(c.ws) == 0  # cleared


def test_check_layer():
    c = Case(1)
    l3.l3_check_layer(c.layer, c.ws)
    bad = c.offs.clone()
    bad[10] = bad[11]  # empty range
    L = l3.make_layer(bad, c.K, c.V, c.W_up, c.W_mix, c.p.k_max)
    with pytest.raises(l3.L3Error) as e:
        l3.l3_check_layer(L, c.ws)
    assert e.value.status == 7
    long = c.offs.clone()
    long[1] = 0
    long[2] = 17  # a 17-row range with k_max = 16
    L = l3.make_layer(long, c.K, c.V, c.W_up, c.W_mix, c.p.k_max)
    with pytest.raises(l3.L3Error):
        l3.l3_check_layer(L, c.ws)


# ---- forward ---------------------------------------------------------------------------------

def test_forward_fp32_tiny_all_tokens_and_intermediates():
    c = Case(1)
    y, sv = c.forward(saved=True)
    torch.cuda.synchronize()
    fw = c.oracle_forward()
    assert_fp32_close(to_np(y), fw.y, "y")
    a, ml, mu, rstd = c.saved_views(sv)
    assert_fp32_close(to_np(a), fw.a, "a")
    assert_fp32_close(to_np(ml[:, 0]), fw.m, "max score")
    np.testing.assert_allclose(to_np(ml[:, 1]), fw.l, rtol=1e-5)
    np.testing.assert_allclose(to_np(mu), fw.mu, rtol=1e-4, atol=1e-6 * np.abs(fw.mu).max())
    np.testing.assert_allclose(to_np(rstd), fw.rstd, rtol=1e-5)
    assert l3.l3_get_error(c.ws) == 0


def test_single_row_tokens_return_value_row_exactly_fp32():
    c = Case(1)
    n = np.diff(c.offs_np)
    ones = np.nonzero(n == 1)[0][:40].astype(np.int32)
    c2 = Case(1, ids=ones)
    _, sv = c2.forward(saved=True)
    a = c2.saved_views(sv)[0].cpu().numpy()
    V = W.table_rows_to_numpy(c2.V, c2.offs_np[ones])
    assert np.array_equal(a, V)


# (T <= 64 takes the transposed GEMMs: 37 tokens on d = 320 ends the last feature tile at 64
# rows, 64 tokens on d = 64 has a single partial tile)
@pytest.mark.parametrize("cid,T", [(5, None), (1, 1), (1, 129), (5, 300), (2, 1024), (2, 333),
                                   (6, 37), (5, 64), (2, 50), (3, 1)])
def test_forward_small_all_tokens(cid, T):
    c = Case(cid, T=T)
    y, _ = c.forward()
    fw = c.oracle_forward()
    assert_close(c.p, to_np(y), fw.y, "y")
    assert l3.l3_get_error(c.ws) == 0


def test_forward_ragged_tile_shapes_all_tokens():
    # d = 320: odd column-tile counts in both GEMMs (5 tiles of 64, a 256-wide tile and a
    # ragged one); 1100 tokens: odd row-tile count, long segments on tensor cores, short
    # ones split
    c = Case(6)
    y, _ = c.forward()
    fw = c.oracle_forward()
    assert_close(c.p, to_np(y), fw.y, "y")
    assert l3.l3_get_error(c.ws) == 0


def test_forward_many_cta_plan_all_tokens():
    # 9000 tokens (above the 8192 that one CTA sorts and plans): the many-CTA segment and
    # plan pass, on the ragged shape (short segments split, long ones on tensor cores); all
    # tokens against the oracle, the saved (max, denominator) too
    c = Case(6, T=9000)
    y, sv = c.forward(saved=True)
    fw = c.oracle_forward()
    assert_close(c.p, to_np(y), fw.y, "y")
    a, ml, _, _ = c.saved_views(sv)
    assert_fp32_close(to_np(ml[:, 0]), fw.m, "max score", rtol=1e-5)
    assert l3.l3_get_error(c.ws) == 0


def test_forward_bf16_fp32_output():
    c = Case(2, T=512)
    y, _ = c.forward(y_dtype=torch.float32)
    fw = c.oracle_forward()
    assert_close(c.p, to_np(y), fw.y, "y fp32 out")


def _sample_tokens(c, k, seed=0):
    rng = np.random.default_rng(seed)
    ids = c.wl.ids
    top = np.nonzero(ids == np.bincount(ids).argmax())[0][:4]
    rare = np.argsort(np.diff(c.offs_np)[ids], kind="stable")[:4]
    return np.unique(np.concatenate([rng.choice(c.T, size=k, replace=False), top, rare, [0, c.T - 1]]))


@pytest.mark.parametrize("cid,k", [(2, 48), (3, 64), (4, 40)])
def test_forward_full_size_sampled(cid, k):
    c = Case(cid)
    y, _ = c.forward()
    toks = _sample_tokens(c, min(k, c.T))
    fw = c.oracle_forward(tokens=toks)
    assert_close(c.p, to_np(y[torch.as_tensor(toks, device=y.device)]), fw.y, f"config {cid} y")
    assert l3.l3_get_error(c.ws) == 0
    del c
    torch.cuda.empty_cache()


def test_all_tokens_same_id_largest_range():
    ids = np.zeros(700, dtype=np.int32)  # id 0 owns k = 512 rows
    c = Case(2, ids=ids)
    y, _ = c.forward()
    fw = c.oracle_forward(tokens=range(0, 700, 7))
    assert_close(c.p, to_np(y)[::7], fw.y, "same id")


def test_forward_host_buffers_equal_device_path():
    c = Case(2, T=777)
    y_dev, _ = c.forward()
    ws_h = torch.empty(l3.l3_workspace_size(c.layer, c.T, l3.L3_PASS_FORWARD_HOST),
                       dtype=torch.uint8, device="cuda")
    ids_h = c.ids.cpu().pin_memory()
    x_h = c.x.cpu().pin_memory()
    y_h = torch.empty((c.T, c.p.d), dtype=c.dt).pin_memory()
    l3.l3_forward_host(c.layer, ids_h, x_h, y_h, ws_h)
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_dev.cpu())


def test_forward_is_deterministic():
    c = Case(2, T=2048)
    y1, _ = c.forward()
    y2, _ = c.forward()
    assert torch.equal(y1, y2)


def test_forward_timed_events():
    c = Case(5)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(l3.L3_FWD_STAGES + 1)]
    for e in evs:
        e.record()
    y = torch.empty((c.T, c.p.d), dtype=c.dt, device="cuda")
    l3.l3_forward_timed(c.layer, c.ids, c.x, y, c.ws, evs)
    torch.cuda.synchronize()
    times = [evs[k].elapsed_time(evs[k + 1]) for k in range(l3.L3_FWD_STAGES)]
    assert all(t >= 0 for t in times)
    y2, _ = c.forward()
    assert torch.equal(y, y2)


# ---- backward --------------------------------------------------------------------------------

def _backward(c):
    y, sv = c.forward(saved=True)
    p = c.p
    dev = "cuda"
    out = dict(dx=torch.empty((c.T, p.d), device=dev), dK=torch.empty((p.v, p.d), device=dev),
               dV=torch.empty((p.v, p.d_v), device=dev), dW_up=torch.empty((p.d, p.d_v), device=dev),
               dW_mix=torch.empty((p.d, 2 * p.d), device=dev))
    wsb = torch.empty(l3.l3_workspace_size(c.layer, c.T, l3.L3_PASS_BACKWARD), dtype=torch.uint8,
                      device=dev)
    l3.l3_backward(c.layer, c.ids, c.x, c.dy, sv, out["dx"], out["dK"], out["dV"], out["dW_up"],
                   out["dW_mix"], wsb)
    torch.cuda.synchronize()
    assert l3.l3_get_error(wsb) == 0
    return out


@pytest.mark.parametrize("cid,T", [(5, None), (5, 37), (1, None)])
def test_backward_parity(cid, T):
    c = Case(cid, T=T, with_dy=True)
    g = _backward(c)
    K = W.table_rows_to_numpy(c.K)
    V = W.table_rows_to_numpy(c.V)
    ref = oracle.backward(c.offs_np, K, V, c.wl.W_up, c.wl.W_mix, c.wl.ids, c.wl.x, c.wl.dy)
    for name in ("dx", "dK", "dV", "dW_up", "dW_mix"):
        assert_close(c.p, to_np(g[name]), getattr(ref, name), name)
        # every step of the backward is fp32: an fp32-level normwise bound as well
        assert_fp32_close(to_np(g[name]), getattr(ref, name), name + " (fp32 level)",
                          rtol=GRAD_FP32_RTOL if c.p.dtype == "bf16" else None)


def test_backward_deterministic_and_untouched_rows_zero():
    c = Case(5, with_dy=True)
    g1 = _backward(c)
    g2 = _backward(c)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k
    present = np.zeros(c.p.v, dtype=bool)
    for t in np.unique(c.wl.ids):
        present[c.offs_np[t]:c.offs_np[t + 1]] = True
    dK = g1["dK"].cpu().numpy()
    assert not dK[~present].any()


@pytest.mark.parametrize("T", [1000, 1500])  # CUDA-core attend below 1024 tokens, tensor cores above
def test_forward_bf16_saved_state_and_layernorm_statistics(T):
    c = Case(2, T=T)
    y, sv = c.forward(saved=True)
    torch.cuda.synchronize()
    fw = c.oracle_forward()
    a, ml, mu, rstd = c.saved_views(sv)
    a, ml = to_np(a), to_np(ml)
    long = c.long_segment_tokens()
    assert (T < 1024) == (not long.any())
    # split-row tokens: fp32 arithmetic on the bf16 inputs (weights as bf16 hi + lo)
    assert_fp32_close(a[~long], fw.a[~long], "a (fp32 copy), split-row tokens")
    np.testing.assert_allclose(ml[~long, 1], fw.l[~long], rtol=1e-5)
    if long.any():
        # tensor-core tokens: the derived bound of bf16-rounded weights
        toks = np.nonzero(long)[0]
        assert_rounded_weight_bound(a[toks], ml[toks, 1], c.oracle_weights(toks), "a, tensor-core tokens")
    np.testing.assert_allclose(ml[:, 0], fw.m, rtol=0, atol=1e-3 * np.abs(fw.m).max() + 1e-4)
    # A and U enter the GEMMs rounded to bf16 (reading "bf16 storage"). Rounding u_n to
    # u_n (1 + d_n), |d_n| <= u, moves the mean by at most u max|u| and the variance by a
    # relative 2u (rstd by u); the rounding of a only adds errors uncorrelated with u_n,
    # smaller by about 1/sqrt(d). Bound: 2u for both.
    np.testing.assert_allclose(to_np(rstd), fw.rstd, rtol=2 * BF16_U)
    np.testing.assert_allclose(to_np(mu), fw.mu, rtol=0, atol=2 * BF16_U * np.abs(fw.u).max())
    assert_close(c.p, to_np(y), fw.y, "y")
    assert l3.l3_get_error(c.ws) == 0


def test_tile_gemms_as_cta_pairs_every_token_and_column():
    # 37900 tokens of the ragged-tile shapes (d = 320): 297 row tiles x 2 column tiles of
    # 128 x 256 make four waves on 148 SMs, so GEMM-up and GEMM-mix run as CTA pairs. The
    # last pair's second CTA holds no rows at all, and in the second column tile the second
    # CTA's half of the weight rows lies wholly past d. Reference: the oracle's LayerNorm and
    # fp64 products on the GPU's own a rounded to bf16 (the GEMMs' input), with U rounded to
    # bf16 before the LayerNorm (reading "bf16 storage"), for every token and column.
    c = Case(6, T=37900)
    y, sv = c.forward(saved=True)
    y32, _ = c.forward(y_dtype=torch.float32)
    torch.cuda.synchronize()
    a, _, mu, rstd = c.saved_views(sv)
    a16 = to_np(a.to(torch.bfloat16))
    u16 = to_np(torch.as_tensor(a16 @ to_np(c.W_up).T).to(torch.bfloat16))
    ln = [oracle.layer_norm(u16[i], 1e-5) for i in range(c.T)]
    h = np.stack([r[0] for r in ln])
    y_ref = np.concatenate([h, to_np(c.x)], axis=1) @ to_np(c.W_mix).T
    np.testing.assert_allclose(to_np(rstd), [r[2] for r in ln], rtol=2 * BF16_U)
    np.testing.assert_allclose(to_np(mu), [r[1] for r in ln], rtol=0,
                               atol=2 * BF16_U * np.abs(u16).max())
    g, g32 = to_np(y), to_np(y32)
    assert_close(c.p, g, y_ref, "y")
    # bf16 output: each element rounded once (relative u); fp32 output: fp32 sums only
    assert np.linalg.norm(g - y_ref) <= 2 * BF16_U * np.linalg.norm(y_ref)
    assert np.linalg.norm(g32 - y_ref) <= 1e-3 * np.linalg.norm(y_ref)
    assert l3.l3_get_error(c.ws) == 0


def test_tensor_core_attend_one_long_segment_and_mixed_ranges():
    # 1400 tokens: 1100 of id 0 (512 rows: 4 row chunks, 18 token chunks) and ids with
    # few rows (partial 16-row boxes, single-token items)
    rng = np.random.default_rng(7)
    ids = np.concatenate([np.zeros(1100, np.int32), rng.integers(20000, 32768, 300).astype(np.int32)])
    rng.shuffle(ids)
    c = Case(2, ids=ids)
    y, sv = c.forward(saved=True)
    toks = np.unique(np.concatenate([np.nonzero(ids == 0)[0][::37], np.nonzero(ids != 0)[0][::5]]))
    fw = c.oracle_forward(tokens=toks)
    assert_close(c.p, to_np(y)[toks], fw.y, "y")
    a, ml, _, _ = c.saved_views(sv)
    long = c.long_segment_tokens()[toks]
    assert long.any() and (~long).any()
    assert_rounded_weight_bound(to_np(a)[toks[long]], to_np(ml)[toks[long], 1],
                                c.oracle_weights(toks[long]), "a, id 0")
    assert_fp32_close(to_np(a)[toks[~long]], fw.a[~long], "a, short ids")
    assert l3.l3_get_error(c.ws) == 0


def test_split_attend_one_token_spread_over_many_ctas_and_long_segments():
    # decode shapes: one token of the id with the most rows (512 rows = 64 chunks, one per
    # CTA, merged by the last CTA), then a batch where one id fills several 8-token groups
    for ids in (np.array([0], np.int32),
                np.concatenate([np.zeros(19, np.int32), np.arange(1, 46, dtype=np.int32)])):
        c = Case(3, ids=ids)
        y, sv = c.forward(saved=True)
        fw = c.oracle_forward()
        assert_close(c.p, to_np(y), fw.y, "y")
        a, ml, _, _ = c.saved_views(sv)
        assert_fp32_close(to_np(a), fw.a, "a (fp32 copy)")
        np.testing.assert_allclose(to_np(ml[:, 0]), fw.m, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(to_np(ml[:, 1]), fw.l, rtol=1e-5)
        assert l3.l3_get_error(c.ws) == 0
        del c
        torch.cuda.empty_cache()


def test_single_row_tokens_return_value_row_exactly_bf16():
    # bf16 storage: p = exp(0) / 1 = 1 exactly, and the weights enter the tensor-core
    # product as bf16 hi + lo terms (1 and 0), so a is the value row bit for bit
    c = Case(5)
    n = np.diff(c.offs_np)
    ones = np.nonzero(n == 1)[0][:40].astype(np.int32)
    c2 = Case(5, ids=ones)
    _, sv = c2.forward(saved=True)
    a = c2.saved_views(sv)[0].cpu().numpy()
    V = W.table_rows_to_numpy(c2.V, c2.offs_np[ones])
    assert np.array_equal(a, V)


def test_bounded_wait_runs_out_and_reports_timeout_without_a_fault():
    # a wait that nothing completes gives up after its limit (20 ms), records the timeout,
    # and the device stays usable: a forward afterwards is clean
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    l3.l3_selftest_wait_timeout(ws, 20_000_000)
    assert l3.l3_status_string(l3.l3_get_error(ws)) == "L3_ERR_TIMEOUT"
    assert l3.l3_get_error(ws) == 0  # read-and-clear
    c = Case(5)
    y, _ = c.forward()
    assert l3.l3_get_error(c.ws) == 0
    assert_close(c.p, to_np(y), c.oracle_forward().y, "y after the timeout")
