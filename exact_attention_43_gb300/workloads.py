"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module draws inputs only: it holds none of the attention arithmetic, so
both the CUDA path and the float64 oracle can take their inputs from it.

The five workloads are the ones the attention pages work at (head_dim 128,
32 heads, sequences up to 32768, a GQA group of 4 and a flash-decoding batch):

* ``tiny``   B1 H4 S256 D64 fp16, non-causal and causal, scale 1/8;
* ``mha``    B4 H32 S2048 D128 bf16 causal, scale 1/sqrt(128);
* ``gqa``    B2 Hq32 Hkv8 S8192 D128 bf16 causal, Q ~ N(0, 3^2), K, V ~ N(0, 1);
* ``long``   B1 H32 S32768 D128 bf16 causal (checked on sampled rows);
* ``decode`` B64 Hq32 Hkv8 D128 bf16, cache [64, 8, 32768, 128], seq_lens
  uniform in [512, 32768], chunk 512 (64 splits).

Values are drawn in float32 from a ``torch.Generator`` seeded with
0x43 + workload index and rounded once to the workload's dtype; the same
rounded tensors go to the GPU and to the oracle.  Large workloads are drawn on
the GPU (the CUDA generator is seeded the same way) and the oracle receives
copies of the drawn tensors.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SEED_BASE = 0x43


@dataclass(frozen=True)
class FwdWorkload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    dtype: torch.dtype
    causal: bool
    q_std: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self, causal: bool | None = None) -> float:
        """Algorithmic flops: 4*D per visible (query, key) pair."""
        causal = self.causal if causal is None else causal
        return 4.0 * self.D * self.B * self.Hq * visible_pairs(self.Sq, self.Skv, causal)

    def io_bytes(self) -> int:
        """Bytes every exact implementation must move at least once: Q, K, V, O, LSE."""
        el = 2
        return (2 * self.B * self.Hq * self.Sq * self.D * el
                + 2 * self.B * self.Hkv * self.Skv * self.D * el
                + 4 * self.B * self.Hq * self.Sq)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    max_S: int
    D: int
    dtype: torch.dtype
    len_lo: int
    len_hi: int
    num_splits: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def chunk(self) -> int:
        return -(-self.max_S // self.num_splits)

    def kv_bytes(self, seq_lens) -> int:
        """K and V bytes of the valid prefixes: sum_b L_b * Hkv * D * 2 B * 2."""
        total = int(torch.as_tensor(seq_lens).to(torch.int64).sum())
        return total * self.Hkv * self.D * 2 * 2

    def io_bytes(self, seq_lens) -> int:
        """Algorithmic bytes: valid K/V prefixes plus q and O."""
        return self.kv_bytes(seq_lens) + 2 * self.B * self.Hq * self.D * 2

    def flops(self, seq_lens) -> float:
        total = int(torch.as_tensor(seq_lens).to(torch.int64).sum())
        return 4.0 * self.D * self.Hq * total


def visible_pairs(Sq: int, Skv: int, causal: bool) -> int:
    """Number of (query, key) pairs with key j <= i + (Skv - Sq) (or all, non-causal)."""
    if not causal:
        return Sq * Skv
    per_row = torch.clamp(torch.arange(Sq, dtype=torch.int64) + (Skv - Sq) + 1, 0, Skv)
    return int(per_row.sum())


TINY = FwdWorkload("tiny", 0, 1, 4, 4, 256, 256, 64, torch.float16, False)
MHA = FwdWorkload("mha", 1, 4, 32, 32, 2048, 2048, 128, torch.bfloat16, True)
GQA = FwdWorkload("gqa", 2, 2, 32, 8, 8192, 8192, 128, torch.bfloat16, True, q_std=3.0)
LONG = FwdWorkload("long", 3, 1, 32, 32, 32768, 32768, 128, torch.bfloat16, True)
DECODE = DecodeWorkload("decode", 4, 64, 32, 8, 32768, 128, torch.bfloat16, 512, 32768, 64)

FWD_WORKLOADS = {w.name: w for w in (TINY, MHA, GQA, LONG)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, *, seed: int, std: float = 1.0, dtype=torch.bfloat16, device="cpu"):
    """N(0, std^2) drawn in float32 from a seeded generator, rounded once to dtype."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def fwd_inputs(B, Hq, Hkv, Sq, Skv, D, *, dtype=torch.bfloat16, seed=SEED_BASE,
               q_std=1.0, kv_std=1.0, device="cpu"):
    """q [B,Hq,Sq,D], k and v [B,Hkv,Skv,D], contiguous, drawn with seeds seed, seed+1, seed+2."""
    q = normal((B, Hq, Sq, D), seed=seed, std=q_std, dtype=dtype, device=device)
    k = normal((B, Hkv, Skv, D), seed=seed + 1, std=kv_std, dtype=dtype, device=device)
    v = normal((B, Hkv, Skv, D), seed=seed + 2, std=kv_std, dtype=dtype, device=device)
    return q, k, v


def workload_fwd_inputs(w: FwdWorkload, device="cpu"):
    return fwd_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, dtype=w.dtype,
                      seed=SEED_BASE + w.index, q_std=w.q_std, device=device)


def seq_lens(B, lo, hi, *, seed):
    """B sequence lengths, i.i.d. uniform integers in [lo, hi], int32 on the CPU."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def decode_inputs(B, Hq, Hkv, max_S, D, lens, *, dtype=torch.bfloat16, seed=SEED_BASE,
                  device="cpu"):
    """q [B,Hq,D], k_cache and v_cache [B,Hkv,max_S,D] (the whole cache is drawn)."""
    q = normal((B, Hq, D), seed=seed + 10, dtype=dtype, device=device)
    k = normal((B, Hkv, max_S, D), seed=seed + 11, dtype=dtype, device=device)
    v = normal((B, Hkv, max_S, D), seed=seed + 12, dtype=dtype, device=device)
    return q, k, v, torch.as_tensor(lens, dtype=torch.int32)


def workload_decode_inputs(w: DecodeWorkload, device="cpu"):
    lens = seq_lens(w.B, w.len_lo, w.len_hi, seed=SEED_BASE + w.index)
    return decode_inputs(w.B, w.Hq, w.Hkv, w.max_S, w.D, lens, dtype=w.dtype,
                         seed=SEED_BASE + w.index, device=device)


def paged_cache(k, v, lens, page_size: int, *, seed: int, spare_pages: int = 3):
    """Scatter contiguous caches [B, Hkv, max_S, D] into a page pool.

    Returns k_pages, v_pages [num_pages, Hkv, page_size, D] and block_table
    [B, ceil(max_S / page_size)] int32.  Each sequence gets ceil(len / page_size)
    pages at seeded random places in the pool; `spare_pages` pages belong to no
    sequence, and block-table entries past a sequence's pages are -1 (never
    read).  Positions past max_S inside a last page are zero.
    """
    k, v = k.cpu(), v.cpu()
    B, Hkv, max_S, D = k.shape
    max_pages = -(-max_S // page_size)
    need = [-(-int(n) // page_size) for n in lens]
    num_pages = sum(need) + spare_pages
    g = _gen(seed, "cpu")
    phys = torch.randperm(num_pages, generator=g)
    k_pages = torch.zeros((num_pages, Hkv, page_size, D), dtype=k.dtype)
    v_pages = torch.zeros_like(k_pages)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for pg in range(need[b]):
            pid = int(phys[nxt])
            nxt += 1
            table[b, pg] = pid
            lo, hi = pg * page_size, min((pg + 1) * page_size, max_S)
            k_pages[pid, :, : hi - lo] = k[b, :, lo:hi]
            v_pages[pid, :, : hi - lo] = v[b, :, lo:hi]
    return k_pages, v_pages, table


def varlen_inputs(lens_q, lens_k, Hq, Hkv, D, *, dtype=torch.bfloat16, seed=SEED_BASE,
                  pad_q: int = 0, device="cpu"):
    """Packed variable-length batch: q [total_q, Hq, D], k and v [total_k, Hkv, D] and the
    offsets cu_q, cu_k ([B + 1] int32, on the CPU).  Sequence b owns query rows
    cu_q[b]..cu_q[b+1]-1 and key rows cu_k[b]..cu_k[b+1]-1; `pad_q` extra query rows
    at the end belong to no sequence."""
    cu_q = torch.zeros(len(lens_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(lens_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.as_tensor(lens_q, dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.as_tensor(lens_k, dtype=torch.int64), 0).to(torch.int32)
    total_q, total_k = int(cu_q[-1]) + pad_q, int(cu_k[-1])
    q = normal((total_q, Hq, D), seed=seed + 20, dtype=dtype, device=device)
    k = normal((total_k, Hkv, D), seed=seed + 21, dtype=dtype, device=device)
    v = normal((total_k, Hkv, D), seed=seed + 22, dtype=dtype, device=device)
    return q, k, v, cu_q, cu_k


def sample_rows(S: int, n: int, *, seed: int):
    """n distinct query rows drawn uniformly from [0, S) without replacement, sorted."""
    g = _gen(seed, "cpu")
    n = min(n, S)
    return torch.randperm(S, generator=g)[:n].sort().values
