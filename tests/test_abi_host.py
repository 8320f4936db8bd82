"""The C-ABI library on the host (CPU only, no GPU calls).

Checks that libl3.so loads and exports every function include/l3.h declares, that the
host-only allocation matches the oracle bit for bit, and that argument errors are
returned before any device work.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import l3_workloads as W
import oracle

l3 = pytest.importorskip("static_token_routed_csr_b300")

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "l3.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return sorted(set(re.findall(r"\b(l3_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    try:
        return l3.lib()
    except ImportError as e:
        pytest.fail(str(e))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert l3.l3_abi_version() == 2
    assert l3.l3_status_string(5) == "L3_ERR_TOKEN_RANGE"


@pytest.mark.parametrize("cid", sorted(W.PRESETS))
def test_alloc_offsets_bit_exact_vs_oracle(lib, cid):
    p = W.PRESETS[cid]
    f = W.zipf_freq(p.vocab)
    ours = l3.l3_alloc_offsets(f, p.v, 1, p.k_max, p.power)
    ref = oracle.allocate(f, p.v, 1, p.k_max, p.power)
    assert np.array_equal(ours.astype(np.int64), ref.offs)


@pytest.mark.parametrize("seed", range(60))
def test_alloc_offsets_random_small_bit_exact(lib, seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 300))
    lo = int(rng.integers(1, 4))
    hi = int(rng.integers(lo, 40))
    v = int(rng.integers(N * lo, N * hi + 1))
    f = rng.uniform(1e-3, 1.0, size=N) ** 3
    power = float(rng.choice([0.3, 0.7, 1.0, 1.5]))
    ours = l3.l3_alloc_offsets(f, v, lo, hi, power)
    ref = oracle.allocate(f, v, lo, hi, power)
    assert np.array_equal(ours.astype(np.int64), ref.offs)


def test_alloc_offsets_errors(lib):
    f = np.ones(4)
    out = np.zeros(5, dtype=np.int32)
    assert lib.l3_alloc_offsets(None, 4, 8, 1, 4, 1.0, out.ctypes.data) == 1
    assert lib.l3_alloc_offsets(f.ctypes.data, 4, 8, 1, 4, 1.0, None) == 1
    assert lib.l3_alloc_offsets(f.ctypes.data, 4, 17, 1, 4, 1.0, out.ctypes.data) == 2
    assert lib.l3_alloc_offsets(f.ctypes.data, 4, 3, 1, 4, 1.0, out.ctypes.data) == 2
    bad = np.array([1.0, 0.0, 1.0, 1.0])
    assert lib.l3_alloc_offsets(bad.ctypes.data, 4, 8, 1, 4, 1.0, out.ctypes.data) == 1
    nan = np.array([1.0, np.nan, 1.0, 1.0])
    assert lib.l3_alloc_offsets(nan.ctypes.data, 4, 8, 1, 4, 1.0, out.ctypes.data) == 1


def _fake_layer(**kw):
    # Host-side validation never dereferences these pointers.
    base = dict(vocab=256, v=1024, d=64, d_v=64, k_max=16, dtype=1, ln_eps=1e-5, reserved=0,
                offs=0x1000, K=0x2000, V=0x3000, W_up=0x4000, W_mix=0x5000)
    base.update(kw)
    return l3.L3Layer(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(d=48), 3), (dict(d=4096), 3), (dict(d_v=1024), 3), (dict(k_max=513), 3),
    (dict(dtype=7), 1), (dict(ln_eps=0.0), 1), (dict(reserved=1), 1), (dict(offs=None), 1),
    (dict(K=None), 1), (dict(v=100), 1), (dict(v=256 * 16 + 1), 1),
])
def test_layer_validation_before_device_work(lib, kw, status):
    L = _fake_layer(**kw)
    assert lib.l3_workspace_size(ctypes.byref(L), 128, 0) == 0
    rc = lib.l3_forward(ctypes.byref(L), 0x10, 128, 0x20, 0x30, 0, None, 0x40, 1 << 30, None)
    assert rc == status


def test_forward_argument_errors(lib):
    L = _fake_layer()
    ws = lib.l3_workspace_size(ctypes.byref(L), 128, 0)
    assert ws > 0 and lib.l3_workspace_size(ctypes.byref(L), 128, 1) > 0
    assert lib.l3_workspace_size(ctypes.byref(L), 128, 9) == 0
    assert lib.l3_saved_size(ctypes.byref(L), 128) >= 128 * (64 + 4) * 4
    # too little workspace
    assert lib.l3_forward(ctypes.byref(L), 0x10, 128, 0x20, 0x30, 1, None, 0x40, ws - 1, None) == 4
    # y dtype neither fp32 nor the layer's
    L32 = _fake_layer(dtype=0)
    assert lib.l3_forward(ctypes.byref(L32), 0x10, 128, 0x20, 0x30, 1, None, 0x40, 1 << 30, None) == 1
    # null x / ids / y with T > 0
    assert lib.l3_forward(ctypes.byref(L), None, 128, 0x20, 0x30, 1, None, 0x40, 1 << 30, None) == 1
    assert lib.l3_forward(ctypes.byref(L), 0x10, 128, None, 0x30, 1, None, 0x40, 1 << 30, None) == 1
    assert lib.l3_forward(ctypes.byref(L), 0x10, -1, 0x20, 0x30, 1, None, 0x40, 1 << 30, None) == 1
    # x or y not 16-byte aligned (their rows move by TMA tensor copies)
    assert lib.l3_forward(ctypes.byref(L), 0x10, 128, 0x28, 0x30, 1, None, 0x40, 1 << 30, None) == 1
    assert lib.l3_forward(ctypes.byref(L), 0x10, 128, 0x20, 0x34, 1, None, 0x40, 1 << 30, None) == 1
    # T = 0 is a no-op
    assert lib.l3_forward(ctypes.byref(L), None, 0, None, None, 1, None, None, 1 << 30, None) == 0
    # backward needs saved state and outputs
    wsb = lib.l3_workspace_size(ctypes.byref(L), 128, 1)
    assert lib.l3_backward(ctypes.byref(L), 0x10, 128, 0x20, 0x30, None, 0x50, 0x60, 0x70,
                           0x80, 0x90, 0x40, wsb, None) == 1
    assert lib.l3_backward(ctypes.byref(L), 0x10, 128, 0x20, 0x30, 0x35, 0x50, 0x60, 0x70,
                           0x80, 0x90, 0x40, wsb - 1, None) == 4
    assert lib.l3_get_error(None, None) == 1
    assert lib.l3_forward_timed(ctypes.byref(L), 0x10, 128, 0x20, 0x30, 1, None, 0x40, ws, None, None) == 1


def test_launch_counter_is_monotone(lib):
    a = l3.l3_launch_count()
    assert l3.l3_launch_count() >= a >= 0


def test_wait_selftest_argument_errors(lib):
    # rejected on the host, before any device work
    assert lib.l3_selftest_wait_timeout(None, 1 << 20, 10_000_000, None) == 1
    assert lib.l3_selftest_wait_timeout(0x40, 255, 10_000_000, None) == 1
    assert lib.l3_selftest_wait_timeout(0x40, 1 << 20, 999, None) == 1
    assert lib.l3_selftest_wait_timeout(0x40, 1 << 20, 10_000_000_001, None) == 1


def test_stage_names_follow_the_header_enum():
    src = open(HEADER).read()
    stages = dict((name.lower(), int(v)) for name, v in
                  re.findall(r"L3_STAGE_([A-Z_]+)\s*=\s*(\d+)", src))
    n = int(re.search(r"L3_FWD_STAGES\s*=\s*(\d+)", src).group(1))
    assert l3.L3_FWD_STAGES == n == len(l3.STAGE_NAMES)
    assert [stages[s] for s in l3.STAGE_NAMES] == list(range(n))


def test_workspace_grows_with_the_batch_and_covers_decode_scratch(lib):
    # bf16 layer of the decode shape (d 2048, d_v 512): batches of at most 64 tokens carry
    # the small-batch GEMMs' scratch (both halves' fp32 accumulators, d x 64 x 2) whatever
    # their size; larger batches need more of everything
    L = _fake_layer(d=2048, d_v=512, k_max=512, vocab=1024, v=1024 * 256)
    sizes = [lib.l3_workspace_size(ctypes.byref(L), T, 0) for T in (1, 64, 512, 8192, 65536)]
    assert all(s > 0 for s in sizes)
    assert sizes[-1] > sizes[-2] > sizes[1] >= sizes[0]
    assert sizes[0] > 2048 * 64 * 2 * 4


@pytest.mark.parametrize("seed", range(4))
def test_alloc_offsets_from_counts_bit_exact_vs_oracle(seed):
    rng = np.random.default_rng([seed, 21])
    vocab = int(rng.integers(50, 3000))
    ids = W.sample_ids(vocab, int(rng.integers(0, 50000)), rng)
    counts = oracle.count_ids(ids, vocab)
    v = int(vocab * rng.integers(2, 30))
    smoothing = [1.0, 0.5, 1e-3, 2.0][seed]
    got = l3.l3_alloc_offsets_counts(counts, v, 1, 64, 0.7, smoothing)
    want = oracle.allocate_from_counts(counts, v, 1, 64, 0.7, smoothing).offs
    assert np.array_equal(got.astype(np.int64), want)


def test_alloc_offsets_from_counts_errors():
    counts = np.array([3, 0, 5], dtype=np.int64)
    with pytest.raises(l3.L3Error) as e:
        l3.l3_alloc_offsets_counts(counts, 6, 1, 4, 1.0, 0.0)  # an unseen id, no smoothing
    assert e.value.status == 1
    with pytest.raises(l3.L3Error):
        l3.l3_alloc_offsets_counts(np.array([3, -1], dtype=np.int64), 4, 1, 4, 1.0, 1.0)
    with pytest.raises(l3.L3Error):
        l3.l3_alloc_offsets_counts(counts, 6, 1, 4, 1.0, float("nan"))
    with pytest.raises(l3.L3Error) as e:
        l3.l3_alloc_offsets_counts(counts, 100, 1, 4, 1.0, 1.0)  # 100 > 3 * 4 rows
    assert e.value.status == 2


def test_count_ids_argument_errors(lib):
    ws = np.zeros(256, np.uint8)
    counts = np.zeros(4, np.int64)
    assert lib.l3_count_ids(None, 5, 4, counts.ctypes.data, ws.ctypes.data, 256, None) == 1
    assert lib.l3_count_ids(None, 0, 0, counts.ctypes.data, ws.ctypes.data, 256, None) == 1
    assert lib.l3_count_ids(None, 0, 4, None, ws.ctypes.data, 256, None) == 1
    assert lib.l3_count_ids(None, 0, 4, counts.ctypes.data, ws.ctypes.data, 8, None) == 4
