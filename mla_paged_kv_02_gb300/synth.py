"""Seeded synthetic inputs for MLA paged-KV decode.

This module only draws random tensors and lays them out as a paged cache; it
holds none of the decode arithmetic.  Both the CUDA path (through the C-ABI
binding) and the CPU oracle consume what it returns.

Recipe (one ``torch.Generator`` seeded per case; draws in this order):
  1. kv_lens per request (fixed, uniform integer, or clipped lognormal);
  2. the page permutation: ``randperm`` of a pool of exactly
     sum_b ceil(L_b / page_size) pages (plus spare pages when requested);
  3. the latent cache, fp32 ~ N(0, 0.1^2) rounded to bf16 (RNE), or quantised to
     FP8-E4M3 with one per-tensor scale amax/448;
  4. q_nope ~ N(0, 1) -> bf16 (or, for an FP8 query, E4M3 with one scale
     amax/448 shared with q_pe);
  5. q_pe ~ N(0, 1) -> bf16 (or E4M3).
The block table is ``[B, ceil(max_L / page_size)]`` int32, padded with -1.

Workload shapes follow the vLLM MLA decode microbenchmarks the TokenSpeed MLA
summary quotes (num_heads=32, bs=64, kv_len=80k with MTP-3 / MTP-7) and the
DeepSeek-R1 latent dims (kv_lora_rank 512, qk_rope 64).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

KV_LORA_RANK = 512
QK_ROPE_DIM = 64
KV_ROW = KV_LORA_RANK + QK_ROPE_DIM
PAGE_SIZE = 64
SOFTMAX_SCALE = 1.0 / math.sqrt(128 + 64)  # 1/sqrt(qk_nope + qk_rope)
E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    """One decode workload: shapes plus how kv_lens are drawn."""

    name: str
    batch: int
    num_heads: int
    q_len: int
    kv: object  # int (all equal), list[int], ("uniform", lo, hi) or ("lognormal", median, sigma, lo, hi)
    kv_fp8: bool = False
    out_fp32: bool = False
    page_size: int = PAGE_SIZE

    @property
    def rows_per_request(self) -> int:
        return self.num_heads * self.q_len


# The five decode workloads (plus the MTP-7 variant of the MTP shape).
WORKLOADS = {
    "tiny": Workload("tiny", 4, 16, 1, [1, 17, 64, 200], out_fp32=True),
    "plain": Workload("plain", 64, 128, 1, 4096),
    "mtp3": Workload("mtp3", 64, 32, 4, 81920),
    "mtp7": Workload("mtp7", 64, 32, 8, 81920),
    "fp8": Workload("fp8", 128, 128, 2, ("lognormal", 4096, 1.0, 1024, 32768), kv_fp8=True),
    "hetero": Workload("hetero", 256, 16, 1, ("uniform", 1, 131072)),
}


@dataclasses.dataclass
class Inputs:
    """Decode inputs.  Tensors live on ``device``; the cache is bf16 or uint8 (e4m3 bits)."""

    batch: int
    num_heads: int
    q_len: int
    page_size: int
    q_nope: torch.Tensor  # [B, q_len, H, 512] bf16
    q_pe: torch.Tensor  # [B, q_len, H, 64] bf16
    kv_cache: torch.Tensor  # [num_pages, page_size, 576] bf16, or uint8 holding e4m3 codes
    kv_fp8: bool
    kv_scale: float  # dequant scale (x = e4m3 * scale); 1.0 for bf16
    block_table: torch.Tensor  # [B, max_pages] int32, -1 padded
    seq_lens: torch.Tensor  # [B] int32
    softmax_scale: float = SOFTMAX_SCALE
    out_fp32: bool = False
    q_fp8: bool = False  # q_nope / q_pe hold e4m3 codes (uint8); query = code * q_scale
    q_scale: float = 1.0

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.batch else 0

    def to(self, device) -> "Inputs":
        d = dataclasses.replace(self)
        for f in ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens"):
            setattr(d, f, getattr(self, f).to(device))
        return d


def draw_kv_lens(wl: Workload, gen: torch.Generator) -> list:
    kv = wl.kv
    if isinstance(kv, int):
        return [kv] * wl.batch
    if isinstance(kv, list):
        assert len(kv) == wl.batch
        return list(kv)
    if kv[0] == "uniform":
        _, lo, hi = kv
        return torch.randint(lo, hi + 1, (wl.batch,), generator=gen).tolist()
    if kv[0] == "lognormal":
        _, median, sigma, lo, hi = kv
        z = torch.randn(wl.batch, generator=gen, dtype=torch.float64)
        vals = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
        return [int(v) for v in vals.tolist()]
    raise ValueError(f"unknown kv_len spec {kv!r}")


def _randn_chunked(shape, gen, device, std, out_dtype, chunk_rows=1 << 14):
    """randn(shape) * std cast to ``out_dtype``, drawn in row chunks to bound memory."""
    out = torch.empty(shape, dtype=out_dtype, device=device)
    flat = out.view(shape[0], -1)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        x = torch.randn((e - s, flat.shape[1]), generator=gen, device=device, dtype=torch.float32)
        flat[s:e] = (x * std).to(out_dtype)
    return out


def make_inputs(
    wl: Workload | str,
    seed: int = 0,
    device: str | torch.device = "cpu",
    kv_lens: Optional[list] = None,
    q_len: Optional[int] = None,
    sharp: float = 1.0,
    page_offset: float = 0.0,
    needle: bool = False,
    nan_tail: bool = False,
    spare_pages: int = 0,
    kv_fp8: Optional[bool] = None,
    batch: Optional[int] = None,
    num_heads: Optional[int] = None,
    q_fp8: bool = False,
) -> Inputs:
    """Build one seeded decode problem.

    Structural variants (used to make wrong pages, masks or dropped tiles visible):
      sharp       -- multiply Q by this factor (peaked softmax);
      page_offset -- add +/-page_offset (sign drawn per physical page) to c_kv;
      needle      -- each request's query rows share a component 8*u_b and one
                     visible token carries c_kv = 32*u_b, so it dominates;
      nan_tail    -- fill slots past L in last pages and all spare pages with NaN;
      spare_pages -- extra pool pages that no request references.
    q_fp8 quantises the query (q_nope and q_pe together) to FP8-E4M3 with one
    per-tensor scale amax/448, after the same draws.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    wl = dataclasses.replace(
        wl,
        q_len=q_len if q_len is not None else wl.q_len,
        kv_fp8=wl.kv_fp8 if kv_fp8 is None else kv_fp8,
        batch=batch if batch is not None else wl.batch,
        num_heads=num_heads if num_heads is not None else wl.num_heads,
    )
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    cpu_gen = torch.Generator()
    cpu_gen.manual_seed(seed)

    lens = list(kv_lens) if kv_lens is not None else draw_kv_lens(wl, cpu_gen)
    B, H, q, ps = len(lens), wl.num_heads, wl.q_len, wl.page_size
    pages_per = [(L + ps - 1) // ps for L in lens]
    used = sum(pages_per)
    pool = used + spare_pages
    perm = torch.randperm(pool, generator=cpu_gen).to(torch.int32) if pool else torch.zeros(0, dtype=torch.int32)
    max_pages = max(pages_per) if pages_per else 0
    bt = torch.full((B, max(max_pages, 1)), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off : off + n]
        off += n

    # Latent cache (fp32 draw, then bf16 or e4m3).
    if wl.kv_fp8:
        x = _randn_chunked((pool, ps, KV_ROW), gen, dev, 0.1, torch.float32)
        if page_offset:
            sgn = torch.randint(0, 2, (pool,), generator=gen, device=dev).to(torch.float32) * 2 - 1
            x[:, :, :KV_LORA_RANK] += (page_offset * sgn)[:, None, None]
        amax = float(x.abs().max().item()) if x.numel() else 1.0
        scale = amax / E4M3_MAX if amax > 0 else 1.0
        kv = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
        del x
    else:
        scale = 1.0
        kv = _randn_chunked((pool, ps, KV_ROW), gen, dev, 0.1, torch.bfloat16)
        if page_offset:
            sgn = torch.randint(0, 2, (pool,), generator=gen, device=dev).to(torch.float32) * 2 - 1
            kv[:, :, :KV_LORA_RANK] += (page_offset * sgn).to(torch.bfloat16)[:, None, None]

    qn32 = torch.randn((B, q, H, KV_LORA_RANK), generator=gen, device=dev) * sharp
    qp32 = torch.randn((B, q, H, QK_ROPE_DIM), generator=gen, device=dev) * sharp
    q_nope = qn32.to(torch.bfloat16)
    q_pe = qp32.to(torch.bfloat16)

    bt_dev = bt.to(dev)
    if needle:
        for b, L in enumerate(lens):
            vis = L - q + 1  # every row of request b sees tokens [0, vis)
            t = int(torch.randint(0, vis, (1,), generator=cpu_gen).item())
            u = torch.randn(KV_LORA_RANK, generator=cpu_gen, dtype=torch.float32)
            u = (u / u.norm()).to(dev)
            q_nope[b] = (q_nope[b].float() + 8.0 * u).to(torch.bfloat16)
            qn32[b] += 8.0 * u
            page, slot = int(bt[b, t // ps]), t % ps
            row = 32.0 * u
            if wl.kv_fp8:
                kv[page, slot, :KV_LORA_RANK] = (row / scale).clamp(-E4M3_MAX, E4M3_MAX).to(
                    torch.float8_e4m3fn).view(torch.uint8)
            else:
                kv[page, slot, :KV_LORA_RANK] = row.to(torch.bfloat16)

    if nan_tail:
        nan_code = 0x7F if wl.kv_fp8 else None
        for b, L in enumerate(lens):
            r = L % ps
            if r:
                page = int(bt[b, L // ps])
                if wl.kv_fp8:
                    kv[page, r:, :] = nan_code
                else:
                    kv[page, r:, :] = float("nan")
        if spare_pages:
            spare = perm[used:].to(torch.int64).to(dev)
            if wl.kv_fp8:
                kv[spare] = 0x7F
            else:
                kv[spare] = float("nan")

    q_scale = 1.0
    if q_fp8:
        amax = max(float(qn32.abs().max().item()), float(qp32.abs().max().item())) if qn32.numel() else 1.0
        q_scale = amax / E4M3_MAX if amax > 0 else 1.0
        q_nope = (qn32 / q_scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
        q_pe = (qp32 / q_scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    del qn32, qp32

    return Inputs(
        batch=B,
        num_heads=H,
        q_len=q,
        page_size=ps,
        q_nope=q_nope,
        q_pe=q_pe,
        kv_cache=kv,
        kv_fp8=wl.kv_fp8,
        kv_scale=float(scale),
        block_table=bt_dev,
        seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev),
        out_fp32=wl.out_fp32,
        q_fp8=q_fp8,
        q_scale=float(q_scale),
    )


def permute_pages(inp: Inputs, seed: int) -> Inputs:
    """Same logical problem with the physical pages shuffled and the block table remapped."""
    g = torch.Generator()
    g.manual_seed(seed)
    P = inp.num_pages
    perm = torch.randperm(P, generator=g)  # new physical slot of old page p is perm[p]
    kv = torch.empty_like(inp.kv_cache)
    kv[perm.to(inp.kv_cache.device)] = inp.kv_cache
    bt = inp.block_table.clone()
    valid = bt >= 0
    bt_cpu = bt.cpu()
    bt_cpu[valid.cpu()] = perm[bt_cpu[valid.cpu()].long()].to(torch.int32)
    d = dataclasses.replace(inp)
    d.kv_cache = kv
    d.block_table = bt_cpu.to(inp.block_table.device)
    return d


def subset(inp: Inputs, reqs) -> Inputs:
    """Host copy of the listed requests only: their pages gathered into a compact cache
    with a remapped block table (pure data movement, for evaluating a sample)."""
    pages, bt_rows, lens = [], [], []
    nxt = 0
    for b in reqs:
        L = int(inp.seq_lens[b])
        n = (L + inp.page_size - 1) // inp.page_size
        pages.append(inp.block_table[b, :n].long())
        bt_rows.append(torch.arange(nxt, nxt + n, dtype=torch.int32))
        nxt += n
        lens.append(L)
    kv = inp.kv_cache[torch.cat(pages)].cpu()
    width = max(len(r) for r in bt_rows)
    bt = torch.full((len(reqs), width), -1, dtype=torch.int32)
    for k, r in enumerate(bt_rows):
        bt[k, : len(r)] = r
    idx = torch.tensor(list(reqs), device=inp.q_nope.device)
    return Inputs(batch=len(reqs), num_heads=inp.num_heads, q_len=inp.q_len,
                  page_size=inp.page_size, q_nope=inp.q_nope[idx].cpu(), q_pe=inp.q_pe[idx].cpu(),
                  kv_cache=kv, kv_fp8=inp.kv_fp8, kv_scale=inp.kv_scale, block_table=bt,
                  seq_lens=torch.tensor(lens, dtype=torch.int32), softmax_scale=inp.softmax_scale,
                  out_fp32=inp.out_fp32, q_fp8=inp.q_fp8, q_scale=inp.q_scale)
