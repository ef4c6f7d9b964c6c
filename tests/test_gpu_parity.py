"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Sizes are small enough for the oracle to evaluate every row in seconds but
span several 64-key tiles and splits, with ragged tails.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import inputs, wm, workloads

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


def rand_bf16(shape, gen, device, std=1.0):
    return (torch.randn(shape, generator=gen, device=device) * std).to(torch.bfloat16)


def run_step(w, context, depth, dev, n_split=0, check_verify=True):
    """Ring fill + d draft steps + verify through the library; compare each with the oracle."""
    inp = inputs.make_inputs(w, depth=depth, device=dev, context=context)
    kv = wm.KVCache(inp.k, inp.v, inp.seq_lens, inp.block_table)
    ring = wm.Ring.create(w.batch, w.n_kv_heads, w.head_dim, w.sink, w.window, dev)
    wm.ring_fill(ring, kv)
    hist = oracle_kv(inp.k, inp.v, inp.block_table)
    for j in range(depth):
        wm.ring_append(ring, inp.k_new[j], inp.v_new[j])
        out, lse = wm.draft_attn(ring, inp.q_draft[j], w.scale, n_split=n_split)
        pos = [n + j for n in inp.seq_lens_host]
        ref, ref_lse = oracle.draft(hist, inp.q_draft[j].cpu(), pos, w.sink, w.window, w.scale)
        assert_close(f"{w.name} draft step {j}", out, lse, ref, ref_lse)
    if check_verify:
        out, lse = wm.verify_attn(kv, inp.q_verify, w.scale, n_split=n_split)
        ref, ref_lse = oracle.verify(hist, inp.q_verify.cpu(), inp.seq_lens_host, w.scale)
        assert_close(f"{w.name} verify", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("name,context", [
    ("tiny_4k", 4096), ("gqa8_128k", 3000), ("hybrid_1m_d256", 5000),
    ("paged_ragged_b8", 1500), ("nope_1m_b2", 9000)])
def test_workloads_reduced_context(name, context):
    run_step(workloads.get(name), context, workloads.get(name).max_depth, gpu())


@pytest.mark.parametrize("n_split", [1, 3, 64])
def test_forced_split_counts(n_split):
    run_step(workloads.get("tiny_4k"), 4096, 1, gpu(), n_split=n_split)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G,T", [(1, 1), (4, 3), (8, 2), (16, 4)])
def test_verify_shapes(D, G, T):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(100 + D + 7 * G + T)
    B, Hkv = 2, 2
    Hq = G * Hkv
    lens = [1000 + 37 * D // 64, 613]
    cap = 1200
    k = rand_bf16((B, Hkv, cap, D), gen, dev)
    v = rand_bf16((B, Hkv, cap, D), gen, dev)
    q = rand_bf16((B, T, Hq, D), gen, dev, 1.0)
    seq = torch.tensor(lens, dtype=torch.int64, device=dev)
    kv = wm.KVCache(k, v, seq)
    s = 1 / math.sqrt(D)
    for ns in (0, 1, 5):
        out, lse = wm.verify_attn(kv, q, s, n_split=ns)
        ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), lens, s)
        assert_close(f"verify D={D} G={G} T={T} ns={ns}", out, lse, ref, ref_lse)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("scale", [-0.21, 0.0, 1e-3])
def test_negative_zero_and_tiny_softmax_scales(D, scale):
    """The scale is any finite float: a negative one flips which keys dominate,
    zero gives uniform weights (lse = ln of the key count).  Verify and draft."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(150 + D)
    B, Hkv, G, T, cap = 2, 2, 4, 3, 900
    lens = [850, 333]
    k, v = rand_bf16((B, Hkv, cap, D), gen, dev), rand_bf16((B, Hkv, cap, D), gen, dev)
    q = rand_bf16((B, T, Hkv * G, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev))
    out, lse = wm.verify_attn(kv, q, scale)
    ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), lens, scale)
    assert_close(f"verify D={D} scale={scale}", out, lse, ref, ref_lse)
    ring = wm.Ring.create(B, Hkv, D, 4, 300, dev)
    wm.ring_fill(ring, kv)
    qd = rand_bf16((B, Hkv * G, D), gen, dev)
    out, lse = wm.draft_attn(ring, qd, scale)
    ref, ref_lse = oracle.draft(oracle_kv(k, v), qd.cpu(), [n - 1 for n in lens], 4, 300, scale)
    assert_close(f"draft D={D} scale={scale}", out, lse, ref, ref_lse)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S,W", [(0, 1), (0, 100), (4, 60), (16, 200), (3, 1)])
def test_draft_ring_wraps(D, S, W):
    """Appends past several wraps of a small window; every step checked."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(200 + D + S + W)
    B, Hkv, G = 2, 2, 4
    n_pos = 3 * (S + W) + 7
    hk = rand_bf16((B, Hkv, n_pos, D), gen, dev)
    hv = rand_bf16((B, Hkv, n_pos, D), gen, dev)
    hist = oracle_kv(hk, hv)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    q = rand_bf16((n_pos, B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    check_at = sorted({0, 1, S, S + W - 1, S + W, S + W + 1, n_pos // 2, n_pos - 1} & set(range(n_pos)))
    for p in range(n_pos):
        wm.ring_append(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous())
        if p in check_at:
            out, lse = wm.draft_attn(ring, q[p], 1.0)
            ref, ref_lse = oracle.draft(hist, q[p].cpu(), [p] * B, S, W, 1.0)
            assert_close(f"draft D={D} S={S} W={W} p={p}", out, lse, ref, ref_lse)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S,W,n_split", [(4, 1020, 1), (4, 1021, 1), (16, 1500, 1), (16, 2100, 2), (0, 3000, 3)])
def test_draft_long_splits(D, S, W, n_split):
    """Splits around and above 1024 ring keys, where a CTA stops staging the
    split's tags with Q and reads them from global memory a tile ahead; plain
    and fused-step, with the window part-filled and wrapped."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(250 + D + S + W + n_split)
    B, Hkv, G = 2, 2, 4
    n_pos = 2 * (S + W) + 5
    hk = rand_bf16((B, Hkv, n_pos, D), gen, dev)
    hv = rand_bf16((B, Hkv, n_pos, D), gen, dev)
    hist = oracle_kv(hk, hv)
    scale = 1 / math.sqrt(D)
    for start in (S + W // 2, n_pos - 3):  # ring part-filled; ring wrapped
        ring = wm.Ring.create(B, Hkv, D, S, W, dev)
        wm.ring_fill(ring, wm.KVCache(hk, hv, torch.full((B,), start, dtype=torch.int64, device=dev)))
        ws = wm.step_workspace(ring, Hkv * G, n_split)
        for j in range(2):
            p = start + j
            q = rand_bf16((B, Hkv * G, D), gen, dev)
            if j == 0:
                wm.ring_append(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous())
                out, lse = wm.draft_attn(ring, q, scale, n_split=n_split)
            else:
                out, lse = wm.draft_step(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous(), q, scale, ws,
                                         n_split=n_split)
            ref, ref_lse = oracle.draft(hist, q.cpu(), [p] * B, S, W, scale)
            assert_close(f"draft D={D} S={S} W={W} ns={n_split} p={p}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


def test_draft_with_window_covering_everything_equals_verify():
    """S + W >= p + 1: windowed draft equals full causal attention (single query)."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(300)
    B, Hkv, D, G = 1, 2, 128, 8
    n = 700
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, 4, 1000, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor([n], device=dev)))
    q = rand_bf16((B, Hkv * G, D), gen, dev, 0.1)
    d_out, d_lse = wm.draft_attn(ring, q, 1.0)
    v_out, v_lse = wm.verify_attn(wm.KVCache(hk, hv, torch.tensor([n], device=dev)), q[:, None], 1.0)
    ref, ref_lse = oracle.verify(oracle_kv(hk, hv), q[:, None].cpu(), [n], 1.0)
    assert_close("draft==full", d_out, d_lse, ref, ref_lse)
    assert_close("verify T=1", v_out, v_lse, ref, ref_lse)


def test_ring_slot_rotation_invariance():
    """Permuting ring slots together with their tags leaves the draft output unchanged."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(301)
    B, Hkv, D, G, S, W = 2, 2, 128, 4, 4, 300
    n = 1000
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.full((B,), n, dtype=torch.int64, device=dev)))
    q = rand_bf16((B, Hkv * G, D), gen, dev, 0.1)
    a_out, a_lse = wm.draft_attn(ring, q, 1.0)
    perm = torch.randperm(S + W, generator=gen, device=dev)
    rot = wm.Ring(ring.k[:, :, perm].contiguous(), ring.v[:, :, perm].contiguous(),
                  ring.pos_tag[:, perm].contiguous(), ring.n_seen.clone(), S, W)
    b_out, b_lse = wm.draft_attn(rot, q, 1.0)
    ref, ref_lse = oracle.draft(oracle_kv(hk, hv), q.cpu(), [n - 1] * B, S, W, 1.0)
    assert_close("ring", a_out, a_lse, ref, ref_lse)
    assert_close("rotated ring", b_out, b_lse, ref, ref_lse)


def test_empty_and_degenerate_cases():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(302)
    B, Hkv, D, G, T = 3, 1, 64, 2, 3
    cap = 200
    k, v = rand_bf16((B, Hkv, cap, D), gen, dev), rand_bf16((B, Hkv, cap, D), gen, dev)
    # seq_len 0 (no keys at all), seq_len 2 < T (first query has no key), seq_len 1
    lens = [0, 2, 1]
    q = rand_bf16((B, T, Hkv * G, D), gen, dev)
    out, lse = wm.verify_attn(wm.KVCache(k, v, torch.tensor(lens, device=dev)), q, 0.3, n_split=2)
    ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), lens, 0.3)
    assert_close("degenerate verify", out, lse, ref, ref_lse)
    # empty ring (nothing appended): no key, out 0 / lse -inf
    ring = wm.Ring.create(1, 1, D, 4, 16, dev)
    q1 = rand_bf16((1, G, D), gen, dev)
    out, lse = wm.draft_attn(ring, q1, 1.0)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_stale_bytes_beyond_length_never_leak():
    """NaN/Inf bit patterns in cache rows past seq_len and in never-written ring
    slots must not reach the output (masked keys get zero weight and zeroed V)."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(303)
    B, Hkv, D, G, T = 1, 2, 128, 4, 2
    cap, n = 640, 517
    k, v = rand_bf16((B, Hkv, cap, D), gen, dev), rand_bf16((B, Hkv, cap, D), gen, dev)
    k[:, :, n:] = float("nan")
    v[:, :, n:] = float("inf")
    q = rand_bf16((B, T, Hkv * G, D), gen, dev, 0.1)
    out, lse = wm.verify_attn(wm.KVCache(k, v, torch.tensor([n], device=dev)), q, 1.0)
    ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), [n], 1.0)
    assert_close("verify with NaN tail", out, lse, ref, ref_lse)
    ring = wm.Ring.create(B, Hkv, D, 4, 200, dev)
    ring.k.fill_(float("nan"))
    ring.v.fill_(float("nan"))
    for p in range(50):
        wm.ring_append(ring, k[:, :, p].contiguous(), v[:, :, p].contiguous())
    q1 = rand_bf16((B, Hkv * G, D), gen, dev, 0.1)
    out, lse = wm.draft_attn(ring, q1, 1.0)
    ref, ref_lse = oracle.draft(oracle_kv(k, v), q1.cpu(), [49], 4, 200, 1.0)
    assert_close("draft over partly written ring", out, lse, ref, ref_lse)


def test_paged_verify_matches_contiguous_oracle():
    dev = gpu()
    w = workloads.get("paged_ragged_b8")
    inp = inputs.make_inputs(w, depth=2, device=dev, context=3000, seed_offset=3)
    kv = wm.KVCache(inp.k, inp.v, inp.seq_lens, inp.block_table)
    for ns in (0, 1, 7):
        out, lse = wm.verify_attn(kv, inp.q_verify, w.scale, n_split=ns)
        ref, ref_lse = oracle.verify(oracle_kv(inp.k, inp.v, inp.block_table), inp.q_verify.cpu(),
                                     inp.seq_lens_host, w.scale)
        assert_close(f"paged ns={ns}", out, lse, ref, ref_lse)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("page", [64, 128, 192, 256])
def test_paged_page_sizes_and_short_sequences(D, page):
    """Paged verify over a permuted page pool at several page sizes (128-key
    boxes when the page holds whole 128-key tiles; at 192 keys a split may
    start mid-page), with an empty sequence and one shorter than the verify
    window (its early queries see no key)."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(400 + D + page)
    B, Hkv, G, T = 4, 2, 4, 3
    lens = [0, 2, 70, 3 * page + 17]
    max_pages = (max(lens) + page - 1) // page + 1
    n_pages = B * max_pages + 3
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(7 + page))
    block_table = perm[: B * max_pages].view(B, max_pages).to(torch.int32).to(dev)
    k = rand_bf16((n_pages, Hkv, page, D), gen, dev)
    v = rand_bf16((n_pages, Hkv, page, D), gen, dev)
    q = rand_bf16((B, T, Hkv * G, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev), block_table)
    ref, ref_lse = oracle.verify(oracle_kv(k, v, block_table), q.cpu(), lens, D ** -0.5)
    for ns in (0, 1, 3, 5):  # 5: 256-key splits, which start mid-page at 192-key pages
        out, lse = wm.verify_attn(kv, q, D ** -0.5, n_split=ns)
        assert_close(f"paged D={D} page={page} ns={ns}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("G,T", [(8, 6), (16, 3), (8, 5), (16, 4), (8, 7)])
@pytest.mark.parametrize("page", [0, 64, 192, 256])
def test_verify_head_dim_256_many_rows(G, T, page):
    """head_dim 256 with 33-64 rows per KV head (the largest tensor-core row
    tiles, where only two K/V staging slots fit): a split of ~10 tiles cycles
    the slots many times; one and several splits, contiguous and paged, with
    ragged ends whose masked keys have their V rows zeroed."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(500 + 3 * G + T + page)
    B, Hkv, D = 2, 2, 256
    lens = [1290, 5 + T // 2]
    q = rand_bf16((B, T, Hkv * G, D), gen, dev)
    if page:
        max_pages = (max(lens) + page - 1) // page + 1
        n_pages = B * max_pages + 2
        perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(11 + page))
        block_table = perm[: B * max_pages].view(B, max_pages).to(torch.int32).to(dev)
        k = rand_bf16((n_pages, Hkv, page, D), gen, dev)
        v = rand_bf16((n_pages, Hkv, page, D), gen, dev)
    else:
        block_table = None
        k = rand_bf16((B, Hkv, 1400, D), gen, dev)
        v = rand_bf16((B, Hkv, 1400, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev), block_table)
    hist = oracle_kv(k, v, block_table)
    ref, ref_lse = oracle.verify(hist, q.cpu(), lens, D ** -0.5)
    for ns in (0, 1, 4, 12):  # 12: one 128-key tile per split, starting mid-page at 192-key pages
        out, lse = wm.verify_attn(kv, q, D ** -0.5, n_split=ns)
        assert_close(f"verify D=256 G={G} T={T} page={page} ns={ns}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


def test_lse_merge_kernel_matches_oracle():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(304)
    rows, parts, D = 37, 11, 256
    o = torch.randn((rows, parts, D), generator=gen, device=dev)
    ls = torch.randn((rows, parts), generator=gen, device=dev) * 5
    ls[3, :] = -float("inf")           # a row with only empty parts
    ls[5, ::2] = -float("inf")         # some empty parts
    out, lse = wm.lse_merge(o, ls)
    ref, ref_lse = oracle.lse_merge(o.double().cpu().numpy(), ls.double().cpu().numpy())
    assert_close("lse_merge", out, lse, ref, ref_lse)


def test_split_plan_fills_waves():
    """Default plans: one wave of resident CTAs for a single sequence; for a
    batch on the split plan, the per-split K+V cap rounded up to fill its last
    wave."""
    gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # hybrid verify: 2 KV heads, 32 rows at head_dim 256 (one CTA per SM), 1M keys
    assert wm.plan_splits(wm.WM_OP_VERIFY, 1, 2, 16, 4, 256, 1 << 20, 0) == sms // 2
    # two 1M sequences x 8 KV heads, 40 rows at head_dim 256 (V in half tiles,
    # so the split plan rather than the persistent grid; one CTA per SM): the
    # 8 MB cap asks for ceil(1M / 8192) = 128 splits, 2048 CTAs; the count is
    # raised to the most splits that still fit in ceil(2048 / sms) waves
    ns = wm.plan_splits(wm.WM_OP_VERIFY, 2, 8, 64, 5, 256, 1 << 20, 0)
    units, waves = 16, -(-16 * 128 // sms)
    assert ns >= 128 and units * ns <= waves * sms < units * (ns + 1)


@pytest.mark.parametrize("B,cap,paged", [(3, 20000, False), (16, 6000, True), (17, 3000, False)])
def test_ragged_batch_split_sizes(B, cap, paged):
    """Ragged batches with the planned split count: a few long sequences and
    many short or empty ones, so that most planned splits are empty."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(600 + B)
    Hkv, G, T, D = 2, 4, 2, 128
    cpu_gen = torch.Generator().manual_seed(601 + B)
    lens = torch.randint(0, cap + 1, (B,), generator=cpu_gen).tolist()
    lens[0], lens[-1] = cap, 1
    q = rand_bf16((B, T, Hkv * G, D), gen, dev)
    if paged:
        page = 64
        max_pages = (cap + page - 1) // page
        n_pages = B * max_pages
        perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(602 + B))
        block_table = perm.view(B, max_pages).to(torch.int32).to(dev)
        k = rand_bf16((n_pages, Hkv, page, D), gen, dev)
        v = rand_bf16((n_pages, Hkv, page, D), gen, dev)
    else:
        block_table = None
        k = rand_bf16((B, Hkv, cap, D), gen, dev)
        v = rand_bf16((B, Hkv, cap, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev), block_table)
    out, lse = wm.verify_attn(kv, q, D ** -0.5)
    ref, ref_lse = oracle.verify(oracle_kv(k, v, block_table), q.cpu(), lens, D ** -0.5)
    assert_close(f"ragged B={B} paged={paged}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


def test_reused_buffers_and_shapes():
    """Calls that reuse an address with another shape, or a shape at another
    address, each get their own tensor map: every result matches the oracle."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(777)
    D, Hkv, G, T = 128, 2, 4, 3
    store = rand_bf16((2 * Hkv * 1024 * D,), gen, dev)
    vstore = rand_bf16((2 * Hkv * 1024 * D,), gen, dev)
    other_k = rand_bf16((1, Hkv, 1024, D), gen, dev)
    other_v = rand_bf16((1, Hkv, 1024, D), gen, dev)
    cases = [  # (k, v, lens): the same storage as [2, Hkv, 1024, D] and as [1, Hkv, 2048, D]
        (store.view(2, Hkv, 1024, D), vstore.view(2, Hkv, 1024, D), [1000, 700]),
        (store.view(1, Hkv, 2048, D), vstore.view(1, Hkv, 2048, D), [1900]),
        (other_k, other_v, [1024]),
        (store.view(2, Hkv, 1024, D), vstore.view(2, Hkv, 1024, D), [1000, 700]),
    ]
    for i, (k, v, lens) in enumerate(cases):
        q = rand_bf16((len(lens), T, Hkv * G, D), gen, dev)
        out, lse = wm.verify_attn(wm.KVCache(k, v, torch.tensor(lens, device=dev)), q, D ** -0.5)
        ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), lens, D ** -0.5)
        assert_close(f"case {i}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0
