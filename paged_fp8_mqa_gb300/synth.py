"""Seeded synthetic inputs for the paged FP8 indexer.

This module only draws random numbers and packs them into the byte layouts the indexer reads;
it holds none of the indexer's arithmetic.  Both the CUDA path's tests/benchmark and the CPU
oracle take their inputs from here.

Layouts follow "flashinfer.attn_scores", fp8_paged_mqa_logits, Parameters:
  * q        e4m3 [batch, next_n, num_heads, head_dim]
  * kv_fused uint8 [num_blocks, block_size*(head_dim+4)]: per block, all e4m3 values
             token-major, then block_size little-endian float32 per-token scales (the pages'
             Example builds it with one torch.cat of the two regions; so does this module).
  * weights  float32 [batch*next_n, num_heads]
  * block_tables int32 [batch, ceil(max_seq_len/block_size)]
  * seq_lens int32 [batch]

Draw order, all from one CPU ``torch.Generator`` seeded with the workload's seed:
seq_lens, (zero-length request choice), page permutation, q, k, (outlier-row mask), kv scales,
weights, and later threshold noise and (forced-repair row choice), or the MXFP4 q and k.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEADS = 64
HEAD_DIM = 128
BLOCK = 64


@dataclass
class Workload:
    """One seeded problem instance, on the CPU."""
    name: str
    seed: int
    batch: int
    next_n: int
    num_heads: int
    head_dim: int
    block_size: int
    max_seq_len: int
    seq_lens: torch.Tensor          # int32 [batch]
    block_tables: torch.Tensor      # int32 [batch, width]
    kv_fused: torch.Tensor          # uint8 [num_blocks, block_size*(head_dim+4)]
    q: torch.Tensor                 # uint8 view of e4m3 [batch, next_n, H, D]
    weights: torch.Tensor           # float32 [batch*next_n, H]
    top_k: int | None = None
    capacity: int | None = None
    gen: torch.Generator | None = field(default=None, repr=False)
    spec: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.batch * self.next_n

    @property
    def num_blocks(self) -> int:
        return self.kv_fused.shape[0]

    def row_ends(self) -> torch.Tensor:
        """int32 [rows]: max(0, seq_lens[b] - next_n + t + 1), the per-slot extents."""
        n = self.next_n
        t = torch.arange(n, dtype=torch.int64)
        re = self.seq_lens.to(torch.int64)[:, None] - n + t[None, :] + 1
        return re.clamp_min(0).reshape(-1).to(torch.int32)

    def valid_scores(self) -> int:
        """Number of (query row, KV position) pairs inside the extents."""
        return int(self.row_ends().to(torch.int64).sum())

    def kv_bytes(self) -> int:
        """Bytes of K values and scales the extents touch, page-granular (132 B per token)."""
        pages = (self.seq_lens.to(torch.int64) + self.block_size - 1) // self.block_size
        return int(pages.sum()) * self.block_size * (self.head_dim + 4)


def _draw_seq_lens(g: torch.Generator, spec: dict) -> torch.Tensor:
    B = spec["batch"]
    kind = spec["lens"]
    if kind == "fixed":
        lens = torch.tensor(spec["values"], dtype=torch.int64)
    elif kind == "uniform":
        lo, hi = spec["range"]
        lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    elif kind == "loguniform":
        lo, hi = spec["range"]
        u = torch.rand(B, generator=g, dtype=torch.float64)
        lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).floor().to(torch.int64)
        lens = lens.clamp(lo, hi)
        zeros = spec.get("zeros", 0)
        if zeros:
            lens[torch.randperm(B, generator=g)[:zeros]] = 0
    else:
        raise ValueError(kind)
    return lens.to(torch.int32)


def make_workload(name: str, seed: int, batch: int, next_n: int, max_seq_len: int, lens: str,
                  *, values=None, len_range=None, zeros: int = 0, pool_pages: int | None = None,
                  scale_range=(0.5, 2.0), outlier_frac: float = 0.0, outlier_mult: float = 8.0,
                  unused_entries: str = "zero", top_k: int | None = None,
                  capacity: int | None = None, num_heads: int = HEADS,
                  head_dim: int = HEAD_DIM, block_size: int = BLOCK) -> Workload:
    """Draw one instance.  ``unused_entries`` fills block-table entries past a request's own
    page count: "zero" (page 0, safe for any reader) or "poison" (0x7fffffff, for readers that
    must never touch them)."""
    spec = dict(batch=batch, lens=lens, values=values, range=len_range, zeros=zeros)
    g = torch.Generator().manual_seed(seed)
    seq_lens = _draw_seq_lens(g, spec)
    pages = (seq_lens.to(torch.int64) + block_size - 1) // block_size
    need = int(pages.sum())
    pool = pool_pages if pool_pages is not None else max(need, 1)
    if pool < need:
        raise ValueError(f"pool of {pool} pages is smaller than the {need} needed")
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    width = max(1, -(-max_seq_len // block_size))
    fill = 0 if unused_entries == "zero" else 0x7FFFFFFF
    block_tables = torch.full((batch, width), fill, dtype=torch.int32)
    cursor = 0
    for b in range(batch):
        k = int(pages[b])
        block_tables[b, :k] = perm[cursor:cursor + k]
        cursor += k

    q = torch.randn(batch, next_n, num_heads, head_dim, generator=g)
    q8 = q.to(torch.float8_e4m3fn).view(torch.uint8)
    k = torch.randn(pool, block_size, head_dim, generator=g)
    if outlier_frac > 0:
        mask = torch.rand(pool, block_size, generator=g) < outlier_frac
        k[mask] *= outlier_mult
    k8 = k.to(torch.float8_e4m3fn)
    del k
    lo, hi = scale_range
    scales = torch.rand(pool, block_size, generator=g) * (hi - lo) + lo
    kv_fused = torch.cat([k8.view(torch.uint8).flatten(1), scales.view(torch.uint8).flatten(1)],
                         dim=1)
    weights = torch.rand(batch * next_n, num_heads, generator=g) * 2.0 - 1.0
    return Workload(name=name, seed=seed, batch=batch, next_n=next_n, num_heads=num_heads,
                    head_dim=head_dim, block_size=block_size, max_seq_len=max_seq_len,
                    seq_lens=seq_lens, block_tables=block_tables, kv_fused=kv_fused,
                    q=q8.contiguous(), weights=weights.contiguous(), top_k=top_k,
                    capacity=capacity, gen=g, spec=dict(spec, seed=seed))


# ---- MXFP4 inputs ("flashinfer.attn_scores", fp4_paged_mqa_logits, Parameters q, q_sf,
# kv_fused) -----------------------------------------------------------------------------------

# The E2M1 magnitudes by code 0..7 (OCP Microscaling Formats, FP4 E2M1); code | 8 negates.
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_mxfp4(x: torch.Tensor):
    """Packs float32 rows [..., D] (D a multiple of 32) as MXFP4: per 32 consecutive elements a
    UE8M0 scale byte e (the group's values are x / 2^(e - 127)), the smallest power of two for
    which the group's largest magnitude is at most 6, and per element the E2M1 code of the
    nearest magnitude (ties to the smaller), packed two per byte, element 2j in the low nibble of
    byte j.  Returns (values uint8 [..., D/2], scales uint8 [..., D/32])."""
    *lead, D = x.shape
    g = x.reshape(*lead, D // 32, 32).to(torch.float64)
    amax = g.abs().amax(-1)
    e = torch.ceil(torch.log2(torch.clamp(amax, min=2.0 ** -127) / 6.0)).clamp(-127, 127)
    y = g / torch.exp2(e)[..., None]
    mags = torch.tensor(E2M1_MAGNITUDES, dtype=torch.float64)
    code = (y.abs()[..., None] - mags).abs().argmin(-1)  # first (smaller) on ties
    code = code | ((y < 0) & (code > 0)).to(torch.int64) << 3
    code = code.reshape(*lead, D).to(torch.uint8)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), (e + 127).to(torch.uint8).contiguous()


@dataclass
class Mxfp4Inputs:
    q: torch.Tensor          # uint8 [batch, next_n, H, D/2]: packed E2M1
    q_sf: torch.Tensor       # uint8 [batch, next_n, H, D/32]: UE8M0
    kv_fused: torch.Tensor   # uint8 [num_blocks, block_size*(D/2 + D/32)]


def make_mxfp4(w: Workload, *, spread_tokens: int = 0) -> Mxfp4Inputs:
    """MXFP4 q and KV pool for workload ``w`` (same lengths, pages, weights), drawn next from its
    generator: N(0,1) values, quantized.  ``spread_tokens`` KV tokens get one group scaled by
    2^-12 (their block scales then span more than 8 binades)."""
    g = w.gen
    B, n, H, D, BS = w.batch, w.next_n, w.num_heads, w.head_dim, w.block_size
    pool = w.num_blocks
    q = torch.randn(B, n, H, D, generator=g)
    k = torch.randn(pool, BS, D, generator=g)
    if spread_tokens:
        idx = torch.randperm(pool * BS, generator=g)[:spread_tokens]
        k.view(pool * BS, D)[idx, :32] *= 2.0 ** -12
    qv, qs = quantize_mxfp4(q)
    kv, ks = quantize_mxfp4(k)
    kv_fused = torch.cat([kv.flatten(1), ks.flatten(1)], dim=1).contiguous()
    return Mxfp4Inputs(q=qv, q_sf=qs, kv_fused=kv_fused)


# The five workloads of the indexer, by what they are.
def tiny(unused_entries: str = "zero") -> Workload:
    """B=2, next_n=1, seq_lens [300, 1000], a 24-page pool, max_seq_len 1024."""
    return make_workload("tiny", 0, 2, 1, 1024, "fixed", values=[300, 1000], pool_pages=24,
                         unused_entries=unused_entries)


def decode(batch: int = 64, unused_entries: str = "zero") -> Workload:
    """Decode batch: B=64, next_n=1, seq_lens U[1024, 32768], max 32768."""
    return make_workload("decode", 1, batch, 1, 32768, "uniform", len_range=(1024, 32768),
                         unused_entries=unused_entries)


def mtp(batch: int = 32, unused_entries: str = "zero") -> Workload:
    """MTP/speculative: B=32, next_n=4, seq_lens U[4096, 65536], 1% outlier keys x8,
    kv scales U[0.25, 4]."""
    return make_workload("mtp", 2, batch, 4, 65536, "uniform", len_range=(4096, 65536),
                         scale_range=(0.25, 4.0), outlier_frac=0.01, outlier_mult=8.0,
                         unused_entries=unused_entries)


def long_select(batch: int = 8, seq_len: int = 131072,
                unused_entries: str = "zero") -> Workload:
    """Long context with selection: B=8, next_n=2, seq_lens 131072, top_k 2048, capacity 4096."""
    return make_workload("long_select", 3, batch, 2, seq_len, "fixed", values=[seq_len] * batch,
                         top_k=2048, capacity=4096, unused_entries=unused_entries)


def serving(batch: int = 128, unused_entries: str = "zero") -> Workload:
    """Serving mix: B=128, next_n=1, seq_lens log-uniform [64, 65536] with 3 zero-length
    requests, top_k 2048, capacity 2047."""
    return make_workload("serving", 4, batch, 1, 65536, "loguniform", len_range=(64, 65536),
                         zeros=min(3, batch), top_k=2048, capacity=2047,
                         unused_entries=unused_entries)


WORKLOADS = {"tiny": tiny, "decode": decode, "mtp": mtp, "long_select": long_select,
             "serving": serving}


def thresholds_below_kth(w: Workload, kth: torch.Tensor, forced: int = 10,
                         noise: float = 0.05) -> torch.Tensor:
    """Long-context thresholds: each row's K'-th largest logit minus U[0, noise]*|value|, then
    ``forced`` randomly chosen rows set to +inf (those cannot fit and must be repaired)."""
    kth = kth.to(torch.float32)
    u = torch.rand(kth.shape[0], generator=w.gen)
    thr = kth - u * noise * kth.abs()
    if forced:
        thr[torch.randperm(kth.shape[0], generator=w.gen)[:forced]] = float("inf")
    return thr.contiguous()


def thresholds_scaled_kth(w: Workload, kth: torch.Tensor, lo: float = 0.9,
                          hi: float = 1.1) -> torch.Tensor:
    """Serving thresholds: the previous step's estimate, K'-th largest logit x U[lo, hi];
    rows with no keys (kth NaN) get 0."""
    kth = kth.to(torch.float32)
    u = torch.rand(kth.shape[0], generator=w.gen) * (hi - lo) + lo
    thr = kth * u
    thr[torch.isnan(kth)] = 0.0
    return thr.contiguous()
