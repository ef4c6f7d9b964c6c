"""The persistent verify for batches of several sequences (device-side
schedule): every resident CTA takes an equal run of the batch's key tiles laid
end to end, the run is cut into one segment per (sequence, KV head) it
touches, and the segment partials are merged.  Checked against the fp64
oracle on length mixes that make runs cross many units, hold empty and
one-tile sequences, end on and off tile edges, and leave CTAs without work."""
import math

import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu

WM_DEVERR_TIMEOUT = 3


def rand_bf16(shape, gen, device, std=1.0):
    return (torch.randn(shape, generator=gen, device=device) * std).to(torch.bfloat16)


def make_cache(lens, Hkv, D, gen, dev, paged, page=64, seed=0):
    cap = max(1, max(lens))
    B = len(lens)
    if paged:
        max_pages = -(-cap // page)
        n_pages = B * max_pages
        perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
        bt = perm.view(B, max_pages).to(torch.int32).to(dev)
        k = rand_bf16((n_pages, Hkv, page, D), gen, dev)
        v = rand_bf16((n_pages, Hkv, page, D), gen, dev)
    else:
        bt = None
        k = rand_bf16((B, Hkv, cap, D), gen, dev)
        v = rand_bf16((B, Hkv, cap, D), gen, dev)
    return k, v, bt


def check(name, lens, Hkv, G, T, D, paged, seed, n_split=0):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(seed)
    k, v, bt = make_cache(lens, Hkv, D, gen, dev, paged, seed=seed + 1)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev), bt)
    q = rand_bf16((len(lens), T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    out, lse = wm.verify_attn(kv, q, 1.0, n_split=n_split)
    ref, ref_lse = oracle.verify(oracle_kv(k, v, bt), q.cpu(), lens, 1.0)
    assert_close(name, out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0
    return kv, q, out, lse


MIX = [4000, 0, 130, 128, 1, 2500, 777, 3, 256, 1900]


@pytest.mark.parametrize("D,G,T", [(128, 4, 3), (128, 8, 4), (128, 8, 5), (128, 8, 8), (256, 4, 3), (256, 8, 4)])
@pytest.mark.parametrize("paged", [False, True])
def test_every_persistent_configuration(D, G, T, paged):
    """16, 32, 48 and 64 rows per KV head at head_dim 128, 16 and 32 at 256;
    contiguous and paged caches."""
    check(f"D={D} rows={G * T} paged={paged}", MIX, 2, G, T, D, paged, 1100 + D + 10 * G + T + paged)


@pytest.mark.parametrize("paged", [False, True])
def test_many_short_sequences(paged):
    """More (sequence, KV head) units than CTAs: each run crosses many units,
    and most units hold one or two tiles."""
    lens = torch.randint(0, 400, (300,), generator=torch.Generator().manual_seed(1200)).tolist()
    check(f"300 short sequences paged={paged}", lens, 2, 4, 2, 128, paged, 1201 + paged)


def test_batch_beyond_the_shared_memory_prefix():
    """More sequences than the schedule keeps in shared memory (2048): its
    searches read the tile prefix back from global memory."""
    g = torch.Generator().manual_seed(1250)
    lens = torch.randint(0, 300, (2100,), generator=g).tolist()
    check("2100 sequences", lens, 1, 4, 1, 128, False, 1251)


def test_one_long_sequence_among_tiny_ones():
    """The first runs cross dozens of tiny units before reaching the long one,
    whose tiles are shared by most of the grid."""
    g = torch.Generator().manual_seed(1300)
    lens = [40000] + torch.randint(0, 70, (63,), generator=g).tolist()
    check("one long, 63 tiny", lens, 2, 8, 4, 128, False, 1301)


def test_equal_lengths_and_tile_edges():
    """Equal lengths (the tiles split evenly between the units) and lengths on
    and one past a tile edge."""
    check("equal 3 x 9000", [9000, 9000, 9000], 4, 8, 5, 128, False, 1400)
    check("tile edges", [128, 129, 256, 255, 1024, 1025], 2, 4, 3, 128, True, 1401)


def test_sequences_shorter_than_their_queries_and_all_empty():
    """Lengths below n_q give rows that see no key (out = 0, lse = -inf); a
    batch with no key at all leaves every CTA without work."""
    check("short", [2, 0, 1, 5], 2, 4, 3, 128, False, 1500)
    check("all empty", [0, 0, 0], 2, 4, 3, 128, False, 1501)


def test_explicit_split_count_keeps_the_split_plan():
    """n_split > 0 runs the split plan; both agree with the oracle."""
    check("explicit n_split=5", MIX, 2, 4, 3, 128, True, 1600, n_split=5)


def test_repeated_calls_are_bit_identical():
    kv, q, out, lse = check("first call", MIX, 2, 8, 4, 128, False, 1700)
    for _ in range(3):
        out2, lse2 = wm.verify_attn(kv, q, 1.0)
        assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_graph_replay_reads_lengths_on_the_device():
    """The schedule is made on the device at every launch: a captured graph
    replayed after the lengths changed in place follows the new lengths."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(1800)
    D, Hkv, G, T = 128, 2, 4, 3
    lens_a, lens_b = [3000, 100, 0, 2000], [50, 3100, 1500, 7]
    cap = max(lens_a + lens_b)
    k, v = rand_bf16((4, Hkv, cap, D), gen, dev), rand_bf16((4, Hkv, cap, D), gen, dev)
    seq_lens = torch.tensor(lens_a, dtype=torch.int64, device=dev)
    kv = wm.KVCache(k, v, seq_lens)
    q = rand_bf16((4, T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    need = wm.workspace_size(wm.WM_OP_VERIFY, 4, Hkv, Hkv * G, T, D, kv.capacity)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = torch.full((4, T, Hkv * G, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((4, T, Hkv * G), float("nan"), dtype=torch.float32, device=dev)
    wm.verify_attn(kv, q, 1.0, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    graph, s = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=s):
        wm.verify_attn(kv, q, 1.0, out=out, lse=lse, workspace=ws)
    hist = oracle_kv(k, v)
    for lens in (lens_b, lens_a):
        seq_lens.copy_(torch.tensor(lens, dtype=torch.int64))
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref, ref_lse = oracle.verify(hist, q.cpu(), lens, 1.0)
        assert_close(f"graph replay lens={lens}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


def test_plan_and_workspace():
    """wm_plan_splits answers the persistent grid's CTA count for a batch left
    to the library; the call refuses a workspace one byte short."""
    dev = gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n16 = wm.plan_splits(wm.WM_OP_VERIFY, 4, 2, 8, 3, 128, 4096, 0)
    n48 = wm.plan_splits(wm.WM_OP_VERIFY, 2, 8, 64, 5, 128, 1 << 20, 0)
    # one CTA per SM: a kernel that allocates tensor memory is resident once per SM
    assert n16 == sms and n48 == sms
    # head_dim 256 with more than 32 rows (V in half tiles) stays on the split plan
    assert wm.plan_splits(wm.WM_OP_VERIFY, 2, 2, 16, 5, 256, 1 << 16, 0) != sms
    gen = torch.Generator(device=dev).manual_seed(1900)
    lens = [700, 50, 300, 0]
    k, v = rand_bf16((4, 2, 700, 128), gen, dev), rand_bf16((4, 2, 700, 128), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, device=dev))
    q = rand_bf16((4, 3, 8, 128), gen, dev)
    need = wm.workspace_size(wm.WM_OP_VERIFY, 4, 2, 8, 3, 128, kv.capacity)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    with pytest.raises(wm.WmError):
        wm.verify_attn(kv, q, 1.0, workspace=ws[: need - 1])
    wm.verify_attn(kv, q, 1.0, workspace=ws)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("D,G,T", [(128, 4, 3), (128, 8, 5), (256, 8, 4)])
@pytest.mark.parametrize("stall_unit", [0, 1, 3, 6])
def test_persistent_wait_times_out_then_next_call_is_clean(D, G, T, stall_unit):
    """The test hook stops every CTA's producer at the given copy unit of its
    run: the waits give up, the kernel returns, and the next call is clean."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(2000 + D + G + T + stall_unit)
    lens = [150000, 60000]  # ~3300 tiles: every CTA's run holds well over 6 copy units
    Hkv = 2
    k, v = rand_bf16((2, Hkv, max(lens), D), gen, dev), rand_bf16((2, Hkv, max(lens), D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor(lens, device=dev))
    q = rand_bf16((2, T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    wm.set_test_stall(stall_unit, 4000)
    try:
        wm.verify_attn(kv, q, 1.0)
        torch.cuda.synchronize()
    finally:
        wm.set_test_stall(-1)
    assert wm.get_device_error() == WM_DEVERR_TIMEOUT
    out, lse = wm.verify_attn(kv, q, 1.0)
    ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), lens, 1.0)
    assert_close(f"persistent verify after the timeout D={D} G={G} T={T}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("D,G,T,paged", [(128, 4, 3, True), (128, 8, 5, False), (256, 8, 4, False)])
def test_many_graph_replays_are_bit_identical(D, G, T, paged):
    """300 replays of a captured persistent verify over a mix whose runs cross
    several units (segment boundaries, query restaging, partial slots): every
    replay gives the first replay's bits, and the first matches the oracle --
    a race on a barrier phase or a buffer would show as a differing replay."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(2100 + D + G + T)
    lens = [3000, 17, 2500, 0, 129, 4100, 640, 1]
    Hkv = 2
    k, v, bt = make_cache(lens, Hkv, D, gen, dev, paged, seed=2101)
    kv = wm.KVCache(k, v, torch.tensor(lens, dtype=torch.int64, device=dev), bt)
    q = rand_bf16((len(lens), T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    need = wm.workspace_size(wm.WM_OP_VERIFY, len(lens), Hkv, Hkv * G, T, D, kv.capacity)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = torch.empty((len(lens), T, Hkv * G, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((len(lens), T, Hkv * G), dtype=torch.float32, device=dev)
    wm.verify_attn(kv, q, 1.0, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    graph, s = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=s):
        wm.verify_attn(kv, q, 1.0, out=out, lse=lse, workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    ref, r_lse = oracle.verify(oracle_kv(k, v, bt), q.cpu(), lens, 1.0)
    assert_close(f"persistent D={D} rows={G * T}", ref_out, ref_lse, ref, r_lse)
    outs = torch.empty((300,) + out.shape, dtype=out.dtype, device=dev)
    lses = torch.empty((300,) + lse.shape, dtype=lse.dtype, device=dev)
    for i in range(300):
        out.fill_(float("nan"))
        graph.replay()
        outs[i].copy_(out)
        lses[i].copy_(lse)
    torch.cuda.synchronize()
    same = [(torch.equal(outs[i], ref_out) and torch.equal(lses[i], ref_lse)) for i in range(300)]
    assert all(same), f"{same.count(False)} of 300 replays differ from the first"
    assert wm.get_device_error() == 0
