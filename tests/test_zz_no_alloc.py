"""l3_route_noalloc: the batch sort for callers that cannot allocate device memory.

Such callers (a plugin whose host program owns all device allocations, a latency-critical
loop that must not enter an allocator) cannot hand the library a workspace. This entry
point keeps its scratch in a fixed array the library declares in device memory. The test
calls it through the C ABI twice in a row, on different batches, and checks both results
against l3_route and against the oracle's stable sort (bit for bit: the outputs are
integers), then covers the largest batch the fixed array holds (65536 tokens, on both sort
paths), an empty batch, the size limit and the bad-id report. This file is collected last
so that a run stopping at the first failure has run every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import static_token_routed_csr_b300 as l3  # noqa: E402
from gpu_case import Case, RouteOnly  # noqa: E402


def _outs(T, dev="cuda"):
    return (torch.full((max(T, 1),), -7, dtype=torch.int32, device=dev),
            torch.full((T + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((max(T, 1),), -7, dtype=torch.int32, device=dev),
            torch.full((1,), -7, dtype=torch.int32, device=dev))


def _with_workspace(case):
    perm, start, sid, n = _outs(case.T)
    l3.l3_route(case.layer, case.ids, case.ws, perm, start, sid, n)
    return perm, start, sid, n


def _no_alloc(case):
    perm, start, sid, n = _outs(case.T)
    rc = l3.lib().l3_route_noalloc(ctypes.byref(case.layer), case.ids.data_ptr(), case.T,
                                   perm.data_ptr(), start.data_ptr(), sid.data_ptr(),
                                   n.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, l3.l3_status_string(rc)
    return perm, start, sid, n


def _same(a, b):
    pa, sa, ia, na = (t.cpu().numpy() for t in a)
    pb, sb, ib, nb = (t.cpu().numpy() for t in b)
    S = int(na[0])
    assert S == int(nb[0]) and S > 0
    T = len(pa) if len(pa) == len(sa) - 1 else len(sa) - 1
    assert np.array_equal(pa[:T], pb[:T])
    assert np.array_equal(sa[:S + 1], sb[:S + 1])
    assert np.array_equal(ia[:S], ib[:S])


def _matches_oracle(got, ids_np):
    perm, start, sid, n = (t.cpu().numpy() for t in got)
    ref = oracle.route(ids_np)
    S = int(n[0])
    assert S == len(ref.seg_id)
    T = len(ids_np)
    assert np.array_equal(perm[:T], ref.perm)
    assert np.array_equal(start[:S + 1], ref.seg_start)
    assert np.array_equal(sid[:S], ref.seg_id)


def test_no_alloc_route_matches_workspace_route_twice():
    first = Case(2, T=12289)   # several sort runs and merge passes
    second = Case(1)           # small batch: one CTA sort, leftovers of the first call remain
    for case in (first, second):
        ref = _with_workspace(case)
        got = _no_alloc(case)
        torch.cuda.synchronize()
        _same(got, ref)
        _matches_oracle(got, case.wl.ids)


@pytest.mark.parametrize("vocab,T", [(128256, 65536),    # 32-bit keys: 8 runs, 3 merge passes
                                     (1 << 20, 65536),   # 64-bit keys: 16 runs, 4 merge passes
                                     (1 << 20, 3000)])   # 64-bit keys, one CTA
def test_no_alloc_route_full_array_and_wide_ids(vocab, T):
    case = RouteOnly(T, seed=vocab % 97, vocab=vocab)
    got = _no_alloc(case)
    torch.cuda.synchronize()
    _matches_oracle(got, case.ids_np)
    _same(got, _with_workspace(case))


def test_no_alloc_route_empty_batch():
    case = Case(1)
    n = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    start = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    rc = l3.lib().l3_route_noalloc(ctypes.byref(case.layer), None, 0, None, start.data_ptr(), None,
                                   n.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, l3.l3_status_string(rc)
    torch.cuda.synchronize()
    assert int(n.item()) == 0 and int(start.item()) == 0


def test_no_alloc_limits_and_bad_ids():
    case = Case(1)
    big = torch.zeros(65537, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = l3.lib().l3_route_noalloc(ctypes.byref(case.layer), big.data_ptr(), 65537, None, None,
                                   None, n.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert l3.l3_status_string(rc) == "L3_ERR_WORKSPACE"
    rc = l3.lib().l3_route_noalloc(ctypes.byref(case.layer), big.data_ptr(), 16, None, None,
                                   None, None, torch.cuda.current_stream().cuda_stream)
    assert l3.l3_status_string(rc) == "L3_ERR_INVALID_ARG"
    bad = Case(1, ids=np.array([3, 300, 3], dtype=np.int32))  # vocab is 256
    got = _no_alloc(bad)
    torch.cuda.synchronize()
    assert int(got[3].item()) == -1
    # the next call starts from clean status words
    again = _no_alloc(case)
    torch.cuda.synchronize()
    _same(again, _with_workspace(case))
