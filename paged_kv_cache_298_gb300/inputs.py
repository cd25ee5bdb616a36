"""Seeded synthetic inputs for paged decode attention and the fp8 sliding-window variant.

This module only draws random numbers and places them in memory; it holds none of the
attention arithmetic.  Both the CUDA path and the CPU oracle consume what it produces,
and it imports neither of them.

Recipe (values are drawn with torch's seeded generators, on CPU for small cases and on the
target device for large ones; the same tensors are copied to whichever side needs them):

* q, k, v: float32 N(0, 1) rounded to bf16 (round to nearest even).
* Paged pool: ``num_pages = ceil(pool_factor * pages_needed)`` physical pages of
  ``[page_size, Hkv, D]``; a seeded permutation of the pool (seed + 100) assigns pages
  to sequences in order; unused entries of the block table point at one unused page.
  With ``poison=True`` every unused page, and every in-page row past the end of its
  sequence, holds NaN, so any read outside the attended rows shows up as NaN in the
  output instead of a plausible number.
* fp8 latent cache: float32 N(0, 1) converted to float8_e4m3fn by torch (RNE; |x| < 448
  so saturation never applies), stored as uint8; per-slot inverse scales U[0.5, 2)
  rounded to bf16; per-token window lengths U{1..W}; the first len slots of a token are
  distinct uniform slots of the cache, the rest -1.
* e4m3 GQA cache: the paged pool and table above; K and V codes float32 N(0, 1) converted
  to float8_e4m3fn by torch; per-(page, kv head, slot) factors U[0.5, 2) rounded to bf16;
  poisoning writes the NaN code 0x7F and NaN factors.
* Multi-token decode: the paged pool above holding every new token already; q packed
  [sum(q_lens), Hq, D], N(0, 1) bf16 (seed + 200).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN_BITS = 0x7FC0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class PagedCase:
    """One paged decode problem.  Shapes: q [B,Hq,D]; k_cache/v_cache [P,ps,Hkv,D];
    block_table [B,max_pages] int32; seq_lens [B] int32."""
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    page_size: int
    scale: float
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        return self.k_cache.shape[2]

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def max_pages(self):
        return self.block_table.shape[1]

    @property
    def max_kv_len(self):
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def total_kv(self):
        return int(self.seq_lens.to(torch.int64).sum().item())

    def kv_bytes(self) -> int:
        """bf16 K and V bytes of the attended rows."""
        return self.total_kv * self.Hkv * self.D * 2 * 2

    def to(self, device) -> "PagedCase":
        return PagedCase(self.q.to(device), self.k_cache.to(device), self.v_cache.to(device),
                         self.block_table.to(device), self.seq_lens.to(device), self.page_size,
                         self.scale, self.name, dict(self.extra))


def make_paged_case(B, Hq, Hkv, D, page_size, seq_lens, seed, *, pool_factor=2.0,
                    num_pages=None, max_pages=None, device="cpu", poison=True,
                    name="") -> PagedCase:
    seq_lens = [int(x) for x in seq_lens]
    assert len(seq_lens) == B and Hq % Hkv == 0
    need = [(L + page_size - 1) // page_size for L in seq_lens]
    total = sum(need)
    if num_pages is None:
        num_pages = max(total + 1, int(math.ceil(pool_factor * total)))
    assert num_pages >= total + 1, "the pool keeps one unused page for padding entries"
    if max_pages is None:
        max_pages = max(1, max(need) if need else 1)
    g = _gen(seed, device)
    q = randn_bf16((B, Hq, D), g, device)
    k_cache = randn_bf16((num_pages, page_size, Hkv, D), g, device)
    v_cache = randn_bf16((num_pages, page_size, Hkv, D), g, device)
    perm = torch.randperm(num_pages, generator=_gen(seed + 100, "cpu")).to(torch.int32)
    pad_page = int(perm[total])
    table = torch.full((B, max_pages), pad_page, dtype=torch.int32)
    pos = 0
    for b in range(B):
        table[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    if poison:
        used = torch.zeros(num_pages, dtype=torch.bool)
        used[perm[:total].long()] = True
        nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
        unused = (~used).nonzero().flatten().to(device)
        k_cache[unused] = nan
        v_cache[unused] = nan
        for b in range(B):
            tail = seq_lens[b] % page_size
            if need[b] and tail:
                last = int(table[b, need[b] - 1])
                k_cache[last, tail:] = nan
                v_cache[last, tail:] = nan
    return PagedCase(q, k_cache, v_cache, table.to(device),
                     torch.tensor(seq_lens, dtype=torch.int32, device=device), page_size,
                     1.0 / math.sqrt(D), name)


@dataclass
class MultiCase:
    """A multi-token decode problem: the paged caches of a PagedCase (already holding the
    new tokens' K/V, so seq_lens counts them) and q packed [total_q, Hq, D], sequence b's
    q_lens[b] rows back to back."""
    q: torch.Tensor
    kv: PagedCase
    q_lens: list

    @property
    def total_q(self):
        return self.q.shape[0]

    def to(self, device) -> "MultiCase":
        return MultiCase(self.q.to(device), self.kv.to(device), list(self.q_lens))


def make_multi_case(B, Hq, Hkv, D, page_size, seq_lens, q_lens, seed, *, device="cpu", poison=True,
                    name="") -> MultiCase:
    """Caches as make_paged_case (same seed), q [sum(q_lens), Hq, D] N(0,1) bf16 from seed + 200."""
    assert len(q_lens) == B and all(x >= 0 for x in q_lens)
    kv = make_paged_case(B, Hq, Hkv, D, page_size, seq_lens, seed, device=device, poison=poison, name=name)
    q = randn_bf16((int(sum(q_lens)), Hq, D), _gen(seed + 200, device), device)
    return MultiCase(q, kv, [int(x) for x in q_lens])


@dataclass
class Fp8KvCase:
    """A paged GQA decode problem over an e4m3 cache.  q [B,Hq,D] bf16; k_codes / v_codes
    [P,ps,Hkv,D] uint8 (OCP e4m3 codes); k_scale / v_scale [P,Hkv,ps] bf16 dequantisation
    factors; block_table [B,max_pages] int32; seq_lens [B] int32."""
    q: torch.Tensor
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    page_size: int
    scale: float
    name: str = ""

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        return self.k_codes.shape[2]

    @property
    def max_kv_len(self):
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def total_kv(self):
        return int(self.seq_lens.to(torch.int64).sum().item())

    def to(self, device) -> "Fp8KvCase":
        return Fp8KvCase(self.q.to(device), self.k_codes.to(device), self.v_codes.to(device),
                         self.k_scale.to(device), self.v_scale.to(device), self.block_table.to(device),
                         self.seq_lens.to(device), self.page_size, self.scale, self.name)


E4M3_NAN_CODE = 0x7F


def make_fp8kv_case(B, Hq, Hkv, D, page_size, seq_lens, seed, *, device="cpu", poison=True,
                    name="") -> Fp8KvCase:
    """Block table, pool and q as make_paged_case (same seed); codes are float32 N(0,1)
    converted to float8_e4m3fn by torch (RNE, no saturation at these values), factors
    U[0.5, 2) rounded to bf16 (seed + 300).  With poison=True unused pages and in-page
    rows past a sequence's end hold the NaN code 0x7F and NaN factors."""
    base = make_paged_case(B, Hq, Hkv, D, page_size, seq_lens, seed, device=device, poison=False, name=name)
    P = base.num_pages
    g = _gen(seed + 300, device)
    def codes():
        x = torch.randn((P, page_size, Hkv, D), generator=g, device=device, dtype=torch.float32)
        return x.to(torch.float8_e4m3fn).view(torch.uint8)
    def factors():
        u = torch.rand((P, Hkv, page_size), generator=g, device=device, dtype=torch.float32)
        return (0.5 + 1.5 * u).to(torch.bfloat16)
    kc, vc = codes(), codes()
    ks, vs = factors(), factors()
    if poison:
        lens = [int(x) for x in seq_lens]
        need = [(L + page_size - 1) // page_size for L in lens]
        table = base.block_table.cpu()
        used = torch.zeros(P, dtype=torch.bool)
        for b in range(B):
            used[table[b, :need[b]].long()] = True
        nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
        unused = (~used).nonzero().flatten().to(device)
        for c in (kc, vc):
            c[unused] = E4M3_NAN_CODE
        for f in (ks, vs):
            f[unused] = nan
        for b in range(B):
            tail = lens[b] % page_size
            if need[b] and tail:
                last = int(table[b, need[b] - 1])
                for c in (kc, vc):
                    c[last, tail:] = E4M3_NAN_CODE
                for f in (ks, vs):
                    f[last, :, tail:] = nan
    return Fp8KvCase(base.q, kc, vc, ks, vs, base.block_table, base.seq_lens, page_size, base.scale, name)


def logical_kv(case: PagedCase, max_len=None):
    """The contiguous [B, max_len, Hkv, D] copies of K and V that the paged pool holds
    (rows past a sequence's length are zero).  A data move, used to build the contiguous
    layout from the same values."""
    B, ps = case.B, case.page_size
    if max_len is None:
        max_len = max(1, case.max_kv_len)
    dev = case.k_cache.device
    k = torch.zeros((B, max_len, case.Hkv, case.D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    table = case.block_table.cpu()
    lens = case.seq_lens.cpu()
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        t = torch.arange(L)
        pages = table[b, (t // ps)].long().to(dev)
        slots = (t % ps).to(dev)
        k[b, :L] = case.k_cache[pages, slots]
        v[b, :L] = case.v_cache[pages, slots]
    return k, v


def uniform_lengths(B, lo, hi, seed) -> list[int]:
    """B lengths drawn uniformly from {lo..hi}."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


@dataclass
class Fp8Case:
    """One fp8 sliding-window latent decode problem.  q [T,NH,HD] bf16; kv_cache
    [NB,bs,HD] uint8 (e4m3 codes); inv_scale [NB*bs,1] bf16; indices [T,W] int64;
    lens [T] int64."""
    q: torch.Tensor
    kv_cache: torch.Tensor
    inv_scale: torch.Tensor
    indices: torch.Tensor
    lens: torch.Tensor
    block_size: int
    scale: float
    name: str = ""

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def NH(self):
        return self.q.shape[1]

    @property
    def HD(self):
        return self.q.shape[2]

    @property
    def W(self):
        return self.indices.shape[1]

    @property
    def num_blocks(self):
        return self.kv_cache.shape[0]

    def to(self, device) -> "Fp8Case":
        return Fp8Case(self.q.to(device), self.kv_cache.to(device), self.inv_scale.to(device),
                       self.indices.to(device), self.lens.to(device), self.block_size,
                       self.scale, self.name)


def make_fp8_case(T, NH, HD, num_blocks, block_size, W, seed, *, lens=None, device="cpu",
                  name="") -> Fp8Case:
    g = _gen(seed, "cpu")
    slots = num_blocks * block_size
    q = randn_bf16((T, NH, HD), g, "cpu")
    cache = torch.randn((num_blocks, block_size, HD), generator=g, dtype=torch.float32)
    cache = cache.to(torch.float8_e4m3fn).view(torch.uint8)
    inv = (torch.rand((slots, 1), generator=g, dtype=torch.float32) * 1.5 + 0.5).to(torch.bfloat16)
    if lens is None:
        lens = torch.randint(1, W + 1, (T,), generator=g, dtype=torch.int64)
    else:
        lens = torch.as_tensor(lens, dtype=torch.int64)
    idx = torch.full((T, W), -1, dtype=torch.int64)
    for t in range(T):
        n = int(min(int(lens[t]), W))
        if n > 0:
            idx[t, :n] = torch.randperm(slots, generator=g)[:n]
    case = Fp8Case(q, cache, inv, idx, lens, block_size, 1.0 / math.sqrt(HD), name)
    return case.to(device) if str(device) != "cpu" else case


# ---- the workloads, named by what they are -------------------------------------------

def tiny_paged(device="cpu") -> PagedCase:
    """B=2, Hq=4, Hkv=2, D=64, page_size=16, seq_lens {37,100}, a 16-page pool assigned
    by a seeded permutation."""
    return make_paged_case(2, 4, 2, 64, 16, [37, 100], 298001, num_pages=16, device=device,
                           name="tiny paged GQA decode B=2 Hq=4 Hkv=2 D=64 ps=16 L={37,100}")


def llama_paged(device="cpu") -> PagedCase:
    """B=16, Hq=32, Hkv=8, D=128, every kv_len 2048, page_size 16, 2x pool."""
    return make_paged_case(16, 32, 8, 128, 16, [2048] * 16, 298002, device=device,
                           name="Llama GQA decode B=16 Hq=32 Hkv=8 D=128 ps=16 L=2048")


def ragged_paged(device="cpu", B=128) -> PagedCase:
    """B=128, Hq=32, Hkv=8, D=128, kv_len U{256..4096}, page_size 16, 2x pool."""
    lens = uniform_lengths(B, 256, 4096, 298003)
    return make_paged_case(B, 32, 8, 128, 16, lens, 298003, device=device,
                           name=f"ragged GQA decode B={B} Hq=32 Hkv=8 D=128 ps=16 "
                                f"L~U[256,4096]")


def long_paged(B=1, device="cpu") -> PagedCase:
    """B in {1,4}, Hq=64, Hkv=8, D=128, kv_len 32768, page_size 64, 2x pool."""
    return make_paged_case(B, 64, 8, 128, 64, [32768] * B, 298004, device=device,
                           name=f"long-context GQA decode B={B} Hq=64 Hkv=8 D=128 ps=64 "
                                f"L=32768")


def spec_verify_paged(device="cpu", B=128, q_len=4, Hq=32) -> MultiCase:
    """Speculative-decoding verification: the ragged decode batch (B=128, Hq=32 or 64,
    Hkv=8, D=128, page_size 16, kv_len U{256..4096}) with q_len new tokens per sequence
    attending causally."""
    lens = uniform_lengths(B, 256, 4096, 298003)
    return make_multi_case(B, Hq, 8, 128, 16, lens, [q_len] * B, 298006, device=device,
                           name=f"multi-token GQA decode B={B} q_len={q_len} Hq={Hq} Hkv=8 D=128 ps=16 "
                                f"L~U[256,4096]")


def ragged_fp8kv(device="cpu", B=128) -> Fp8KvCase:
    """The ragged decode batch (B=128, Hq=32, Hkv=8, D=128, page 16, kv_len U{256..4096})
    with an e4m3 K/V cache and per-(slot, kv head) bf16 factors."""
    lens = uniform_lengths(B, 256, 4096, 298003)
    return make_fp8kv_case(B, 32, 8, 128, 16, lens, 298007, device=device,
                           name=f"ragged GQA decode, e4m3 KV, B={B} Hq=32 Hkv=8 D=128 ps=16 L~U[256,4096]")


def fp8_swa(device="cpu") -> Fp8Case:
    """T=64 tokens, NH=128 heads, HD=512, 64 blocks of 256 slots, window 128."""
    return make_fp8_case(64, 128, 512, 64, 256, 128, 298005, device=device,
                         name="fp8 sliding-window latent decode T=64 NH=128 HD=512 W=128")
