"""Seeded random shapes through the C ABI against the fp64 oracle.

Each case draws a head dim, KV heads, GQA group, verify positions (up to 64
rows per KV head), batch, ragged lengths (some empty), a contiguous or paged
store (page sizes 64-256 keys, pool permuted) and a split count; the draft
cases draw sink and window sizes and append past several ring wraps.  The
draws are fixed by the seed, so a failure names a reproducible case.
"""
import math
import random

import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


def rand_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device).to(torch.bfloat16)


def verify_case(seed: int):
    rng = random.Random(seed)
    D = rng.choice([64, 128, 256])
    Hkv = rng.choice([1, 2, 4])
    G = rng.choice([1, 2, 4, 8, 16])
    T = rng.randint(1, max(1, 64 // G))
    B = rng.randint(1, 4)
    cap = rng.choice([200, 900, 2600])
    lens = [rng.choice([0, rng.randint(1, T), rng.randint(1, cap)]) for _ in range(B)]
    lens[rng.randrange(B)] = cap
    page = rng.choice([0, 64, 128, 192, 256])
    n_split = rng.choice([0, 0, 1, rng.randint(2, 9)])
    return D, Hkv, G, T, B, cap, lens, page, n_split


@pytest.mark.parametrize("seed", range(24))
def test_random_verify_matches_oracle(seed):
    dev = gpu()
    D, Hkv, G, T, B, cap, lens, page, n_split = verify_case(seed)
    gen = torch.Generator(device=dev).manual_seed(7000 + seed)
    q = rand_bf16((B, T, Hkv * G, D), gen, dev)
    if page:
        max_pages = (cap + page - 1) // page
        n_pages = B * max_pages + 1
        perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(7100 + seed))
        block_table = perm[: B * max_pages].view(B, max_pages).to(torch.int32).to(dev)
        k = rand_bf16((n_pages, Hkv, page, D), gen, dev)
        v = rand_bf16((n_pages, Hkv, page, D), gen, dev)
    else:
        block_table = None
        k = rand_bf16((B, Hkv, cap, D), gen, dev)
        v = rand_bf16((B, Hkv, cap, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev), block_table)
    scale = 1 / math.sqrt(D)
    out, lse = wm.verify_attn(kv, q, scale, n_split=n_split)
    ref, ref_lse = oracle.verify(oracle_kv(k, v, block_table), q.cpu(), lens, scale)
    assert_close(f"seed {seed}: D={D} Hkv={Hkv} G={G} T={T} B={B} lens={lens} page={page} ns={n_split}",
                 out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("seed", range(12))
def test_random_draft_steps_match_oracle(seed):
    """Fused draft steps (append + attention) after a bulk fill, at random
    sink / window sizes, checked against the oracle at every step."""
    dev = gpu()
    rng = random.Random(8000 + seed)
    D = rng.choice([64, 128, 256])
    Hkv = rng.choice([1, 2, 4])
    G = rng.choice([1, 4, 8, 16])
    B = rng.randint(1, 3)
    S = rng.choice([0, 1, 4, 16])
    W = rng.choice([1, 17, 64, 300])
    steps = rng.randint(1, 4)
    lens = [rng.randint(1, 3 * (S + W) + 5) for _ in range(B)]
    n_split = rng.choice([0, 0, 1, rng.randint(2, 6)])
    gen = torch.Generator(device=dev).manual_seed(8100 + seed)
    n = max(lens) + steps
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor(lens, device=dev)))
    ws = wm.step_workspace(ring, Hkv * G, n_split)
    hist = oracle_kv(hk, hv)
    scale = 1 / math.sqrt(D)
    for j in range(steps):
        q = rand_bf16((B, Hkv * G, D), gen, dev)
        kn = torch.stack([hk[b, :, L + j] for b, L in enumerate(lens)]).contiguous()
        vn = torch.stack([hv[b, :, L + j] for b, L in enumerate(lens)]).contiguous()
        out, lse = wm.draft_step(ring, kn, vn, q, scale, ws, n_split=n_split)
        ref, ref_lse = oracle.draft(hist, q.cpu(), [L + j for L in lens], S, W, scale)
        assert_close(f"seed {seed}: D={D} Hkv={Hkv} G={G} B={B} S={S} W={W} lens={lens} step {j} ns={n_split}",
                     out, lse, ref, ref_lse)
    assert ring.n_seen.tolist() == [L + steps for L in lens]
    assert wm.get_device_error() == 0
