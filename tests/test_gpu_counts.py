"""Token-stream counts on the GPU against the oracle (bit for bit: integers), and the
allocation taken from them ("Information-Theoretic Embedding Allocation", gist.science
explainer: rows follow token frequency)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import l3_workloads as W  # noqa: E402
import static_token_routed_csr_b300 as l3  # noqa: E402


def _count(ids_np, vocab, offset=0):
    base = torch.zeros(len(ids_np) + 4, dtype=torch.int32, device="cuda")
    ids = base[offset:offset + len(ids_np)]  # offset 1..3: not 16-byte aligned
    ids.copy_(torch.as_tensor(np.asarray(ids_np, np.int32)))
    counts = torch.full((vocab,), -5, dtype=torch.int64, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    l3.l3_count_ids(ids, vocab, counts, ws)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), l3.l3_get_error(ws)


@pytest.mark.parametrize("vocab,n,offset", [(256, 0, 0), (256, 1, 1), (256, 3, 3),
                                            (300, 4_000_001, 2),        # all ids in shared memory
                                            (128256, 1_000_003, 1),    # Zipf head and tail
                                            (1 << 20, 777_777, 0)])    # mostly global atomics
def test_counts_bit_exact(vocab, n, offset):
    rng = np.random.default_rng([vocab, n])
    ids = W.sample_ids(vocab, n, rng) if vocab < (1 << 20) else rng.integers(0, vocab, n).astype(np.int32)
    got, err = _count(ids, vocab, offset)
    assert err == 0
    assert np.array_equal(got, oracle.count_ids(ids, vocab))


def test_ids_out_of_range_are_reported_and_skipped():
    ids = np.array([1, 7, -3, 1, 9, 2, 1 << 30], np.int32)
    got, err = _count(ids, 8)
    assert l3.l3_status_string(err) == "L3_ERR_TOKEN_RANGE"
    assert np.array_equal(got, oracle.count_ids(ids[(ids >= 0) & (ids < 8)], 8))


def test_allocation_from_stream_counts_matches_oracle():
    vocab, v = 32768, 262144
    ids = W.sample_ids(vocab, 2_000_000, np.random.default_rng(5))
    got, err = _count(ids, vocab)
    assert err == 0
    offs = l3.l3_alloc_offsets_counts(got, v, 1, 512, 0.7, 1.0)
    want = oracle.allocate_from_counts(oracle.count_ids(ids, vocab), v, 1, 512, 0.7, 1.0)
    assert np.array_equal(offs.astype(np.int64), want.offs)
