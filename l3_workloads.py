"""Seeded synthetic inputs for the Large Lookup Layer (L³) workloads.

This module is shared by the tests, the benchmark and the smoke check. It only draws
random numbers and rounds them to the storage type; it holds none of the layer's
arithmetic (no routing, no allocation, no softmax, no GEMM). The CPU oracle and the CUDA
library each compute the row allocation from ``freq`` on their own.

Workloads (five named presets, shapes as the benchmark specification gives them):

====  =======================  ======  =======  ====  ====  =====  =====  =====  ========
 id    name                    vocab    v        d     d_v   T      k      power  dtype
====  =======================  ======  =======  ====  ====  =====  =====  =====  ========
 1    tiny-fp32-fwd             256     1024     64    64    128    16     1.0    f32
 2    prefill-bf16              32768   262144   1024  256   8192   512    0.7    bf16
 3    decode-bf16               128256  1048576  2048  512   64     512    0.7    bf16
 4    large-prefill-bf16        128256  4194304  2048  512   65536  512    0.7    bf16
 5    fwd-bwd-bf16 (1's shape)  256     1024     64    64    128    16     1.0    bf16
====  =======================  ======  =======  ====  ====  =====  =====  =====  ========

Distributions: token id i has Zipf(1.1) rank i+1 (id 0 most frequent), truncated to the
vocabulary; ``freq[i] = (i+1)^-1.1`` is the allocation's frequency input. x ~ N(0,1);
K, V ~ N(0, 0.02^2) (std 0.02); W_up ~ N(0, 1/d_v), W_mix ~ N(0, 1/(2d)) (variance
1/fan_in); dy ~ N(0,1). Values are drawn in fp64/fp32 and rounded to the storage type
with round-to-nearest-even, so the oracle sees exactly the values the GPU sees.

Seeds: config c uses numpy ``default_rng([c, j])`` with j = 1 ids, 2 x, 5 W_up, 6 W_mix,
7 dy, and a torch generator seeded ``1000*c + j`` with j = 3 (K), 4 (V) on the device that
holds the tables (tables up to 17 GB are drawn where they live). ``shard`` > 0 (one
independent batch per rank) offsets the token-side seeds only.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

ZIPF_S = 1.1
TABLE_STD = 0.02


@dataclasses.dataclass(frozen=True)
class Preset:
    cid: int
    name: str
    vocab: int
    v: int
    d: int
    d_v: int
    T: int
    k_max: int
    power: float
    dtype: str  # "f32" or "bf16"
    backward: bool


PRESETS = {
    1: Preset(1, "tiny-fp32-fwd", 256, 1024, 64, 64, 128, 16, 1.0, "f32", False),
    2: Preset(2, "prefill-bf16", 32768, 262144, 1024, 256, 8192, 512, 0.7, "bf16", False),
    3: Preset(3, "decode-bf16", 128256, 1048576, 2048, 512, 64, 512, 0.7, "bf16", False),
    4: Preset(4, "large-prefill-bf16", 128256, 4194304, 2048, 512, 65536, 512, 0.7, "bf16", False),
    5: Preset(5, "fwd-bwd-bf16", 256, 1024, 64, 64, 128, 16, 1.0, "bf16", True),
    # parity-only shape whose GEMM tiles and attend chunks all end ragged (d = 5 x 64)
    6: Preset(6, "ragged-tiles-bf16", 4096, 65536, 320, 128, 1100, 64, 0.7, "bf16", False),
}


def zipf_freq(vocab: int) -> np.ndarray:
    """Unnormalised Zipf(1.1) frequencies by id: freq[i] = (i+1)^-1.1 (fp64)."""
    return np.arange(1, vocab + 1, dtype=np.float64) ** (-ZIPF_S)


def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even. Inputs are finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the exact fp32 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round an array to the storage type; returns fp32 values representable in it."""
    a = np.asarray(a, dtype=np.float32)
    if dtype == "f32":
        return a
    return bf16_bits_to_f32(round_to_bf16_bits(a)).reshape(a.shape)


def sample_ids(vocab: int, T: int, rng: np.random.Generator) -> np.ndarray:
    """T token ids drawn from the truncated Zipf(1.1) law (id i has rank i+1)."""
    f = zipf_freq(vocab)
    return rng.choice(vocab, size=T, p=f / f.sum()).astype(np.int32)


@dataclasses.dataclass
class Workload:
    preset: Preset
    T: int
    freq: np.ndarray          # [vocab] fp64, allocation input
    ids: np.ndarray           # [T] int32
    x: np.ndarray             # [T, d] fp32, storage-representable
    W_up: np.ndarray          # [d, d_v] fp32, storage-representable (out x in)
    W_mix: np.ndarray         # [d, 2d] fp32, storage-representable (out x in)
    dy: Optional[np.ndarray]  # [T, d] fp32, storage-representable
    table_seed: int

    @property
    def p(self) -> Preset:
        return self.preset


def make(cid: int, T: Optional[int] = None, shard: int = 0, with_dy: Optional[bool] = None,
         vocab: Optional[int] = None, v: Optional[int] = None) -> Workload:
    """Token-side inputs and weights of preset ``cid`` (tables are drawn by ``tables``).

    ``T`` overrides the token count (parity cases at reduced size); ``shard`` selects an
    independent batch (one per rank); ``vocab`` and ``v`` shrink the vocabulary and the
    table (tests of tiny variants, profiler captures of a preset's shapes on smaller tables).
    """
    p = PRESETS[cid]
    if vocab is not None:
        p = dataclasses.replace(p, vocab=vocab)
    if v is not None:
        p = dataclasses.replace(p, v=v)
    T = p.T if T is None else int(T)
    c = cid + 100 * shard
    ids = sample_ids(p.vocab, T, np.random.default_rng([c, 1]))
    x = to_storage(np.random.default_rng([c, 2]).standard_normal((T, p.d), dtype=np.float32), p.dtype)
    W_up = to_storage(np.random.default_rng([cid, 5]).standard_normal((p.d, p.d_v)) / np.sqrt(p.d_v), p.dtype)
    W_mix = to_storage(np.random.default_rng([cid, 6]).standard_normal((p.d, 2 * p.d)) / np.sqrt(2 * p.d), p.dtype)
    want_dy = p.backward if with_dy is None else with_dy
    dy = None
    if want_dy:
        dy = to_storage(np.random.default_rng([c, 7]).standard_normal((T, p.d), dtype=np.float32), p.dtype)
    return Workload(p, T, zipf_freq(p.vocab), ids, x, W_up, W_mix, dy, table_seed=1000 * cid)


def tables(wl: Workload, device="cpu", chunk_rows: int = 1 << 18):
    """Draw the key and value tables K[v,d], V[v,d_v] (torch tensors on ``device``)."""
    import torch

    p = wl.p
    tdt = torch.float32 if p.dtype == "f32" else torch.bfloat16
    out = []
    for j, cols in ((3, p.d), (4, p.d_v)):
        g = torch.Generator(device=device)
        g.manual_seed(wl.table_seed + j)
        t = torch.empty((p.v, cols), dtype=tdt, device=device)
        for r0 in range(0, p.v, chunk_rows):
            r1 = min(p.v, r0 + chunk_rows)
            z = torch.randn((r1 - r0, cols), generator=g, device=device, dtype=torch.float32)
            t[r0:r1] = (z * TABLE_STD).to(tdt)
        out.append(t)
    return out[0], out[1]


def torch_dtype(p: Preset):
    import torch

    return torch.float32 if p.dtype == "f32" else torch.bfloat16


def table_rows_to_numpy(t, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Host copy of a table (or of the listed rows) as exact fp32 values."""
    import torch

    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=t.device)
        t = t.index_select(0, idx)
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f32(t.view(torch.int16).numpy().view(np.uint16)).reshape(tuple(t.shape))
    return t.float().numpy()
