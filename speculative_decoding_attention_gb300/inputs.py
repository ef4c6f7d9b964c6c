"""Seeded synthetic inputs for the decode-attention workloads.

Shared by the CUDA path's tests and bench and by the oracle's tests; it holds
none of the method's arithmetic -- only random numbers laid out in the
library's documented layouts.

Layouts (all bf16 unless stated):
  contiguous store  k, v: [B, Hkv, n_cap, D], n_cap = max context + max depth
  paged store       k, v: [n_pages, Hkv, page_size, D]; block_table [B, max_pages] int32,
                    unused entries -1; pool order randomly permuted
  seq_lens          [B] int64: context N_b; the verify tokens' own K/V are the
                    last T entries below N_b
  q_draft           [d, B, Hq, D]: query of draft step j at position N_b + j
  k_new, v_new      [d, B, Hkv, D]: the entry draft step j appends (position N_b + j);
                    the same values are stored in the store at that position so
                    the store doubles as the draft's history by position
  q_verify          [B, T, Hq, D]: query i at position N_b - T + i
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from .workloads import Workload

_CHUNK = 1 << 26  # elements generated per randn call


def _normal_into(dst: torch.Tensor, gen: torch.Generator, std: float = 1.0) -> None:
    """Fill a bf16 tensor with N(0, std^2) values rounded to bf16, in chunks."""
    flat = dst.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        e = min(flat.numel(), s + _CHUNK)
        x = torch.randn(e - s, generator=gen, device=dst.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e].copy_(x)


def _normal(shape, gen, device, std=1.0) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.bfloat16, device=device)
    _normal_into(t, gen, std)
    return t


@dataclass
class Inputs:
    workload: Workload
    depth: int
    seq_lens: torch.Tensor          # [B] int64, on device
    seq_lens_host: list[int]
    k: torch.Tensor                 # store (contiguous or paged pool)
    v: torch.Tensor
    block_table: torch.Tensor | None
    q_draft: torch.Tensor           # [d, B, Hq, D]
    k_new: torch.Tensor             # [d, B, Hkv, D]
    v_new: torch.Tensor
    q_verify: torch.Tensor          # [B, T, Hq, D]

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    @property
    def n_verify(self) -> int:
        return self.q_verify.shape[1]

    def position_rows(self, pos_per_seq: list[int]) -> tuple[torch.Tensor, torch.Tensor]:
        """K and V rows [B, Hkv, D] stored at the given position of each sequence."""
        ks, vs = [], []
        for b, p in enumerate(pos_per_seq):
            if self.block_table is None:
                ks.append(self.k[b, :, p, :])
                vs.append(self.v[b, :, p, :])
            else:
                ps = self.k.shape[2]
                page = int(self.block_table[b, p // ps])
                ks.append(self.k[page, :, p % ps, :])
                vs.append(self.v[page, :, p % ps, :])
        return torch.stack(ks), torch.stack(vs)


def make_inputs(w: Workload, depth: int | None = None, device="cpu", context: int | None = None,
                seed_offset: int = 0) -> Inputs:
    """Seeded inputs of workload ``w`` at draft depth ``depth`` (verify T = depth + 1).

    ``context`` overrides the context length (same recipe, smaller sizes) for
    cases the oracle evaluates in full.
    """
    d = w.max_depth if depth is None else depth
    T = d + 1
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + 7919 * seed_offset)
    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim

    if w.ragged and context is None:
        lo, hi = w.ragged
        lens = torch.randint(lo, hi + 1, (B,), generator=gen, device=device).tolist()
    elif w.ragged:
        lens = torch.randint(max(T, context // 16), context + 1, (B,), generator=gen,
                             device=device).tolist()
    else:
        lens = [context if context is not None else w.context] * B
    lens = [int(n) for n in lens]
    cap = max(lens) + d

    block_table = None
    if w.page_size:
        ps = w.page_size
        n_pages_b = [-(-(n + d) // ps) for n in lens]
        n_pages = sum(n_pages_b)
        max_pages = max(n_pages_b)
        k = _normal((n_pages, Hkv, ps, D), gen, device)
        v = _normal((n_pages, Hkv, ps, D), gen, device)
        perm = torch.randperm(n_pages, generator=gen, device=device).to(torch.int32)
        block_table = torch.full((B, max_pages), -1, dtype=torch.int32, device=device)
        off = 0
        for b, nb in enumerate(n_pages_b):
            block_table[b, :nb] = perm[off:off + nb]
            off += nb
    else:
        k = torch.empty((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
        v = torch.empty((B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
        if w.peaked_frac > 0:
            # K rounded to bf16 after the selected positions are scaled.
            for b in range(B):
                n_peak = int(round(w.peaked_frac * lens[b]))
                idx = torch.randperm(lens[b], generator=gen, device=device)[:n_peak]
                for h in range(Hkv):
                    x = torch.randn((cap, D), generator=gen, device=device, dtype=torch.float32)
                    x[idx] *= w.peaked_gain
                    k[b, h].copy_(x)
                    del x
        else:
            _normal_into(k, gen)
        _normal_into(v, gen)

    seq_lens = torch.tensor(lens, dtype=torch.int64, device=device)
    q_draft = _normal((d, B, Hq, D), gen, device, w.q_std)
    q_verify = _normal((B, T, Hq, D), gen, device, w.q_std)
    inp = Inputs(w, d, seq_lens, lens, k, v, block_table, q_draft,
                 torch.empty(0), torch.empty(0), q_verify)
    kn, vn = [], []
    for j in range(d):
        kj, vj = inp.position_rows([n + j for n in lens])
        kn.append(kj)
        vn.append(vj)
    inp.k_new = torch.stack(kn).contiguous()
    inp.v_new = torch.stack(vn).contiguous()
    return inp
