"""Pins of the fp64 oracle to facts it does not compute itself.

Each pin checks the oracle against something other than its own formula:
closed forms of softmax attention, PyTorch's own scaled-dot-product attention
(its causal mask and its GQA head mapping), a textbook sink-list + deque model
of a StreamingLLM cache, the paged/contiguous equivalence, and the split-merge
identity.  ``test_planted_mistakes_are_caught`` rebuilds the oracle with one
deliberate mistake at a time and checks that some pin fails for each.

Pages: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
Context" (Abstract) -- draft attention over a sliding window plus attention
sinks, full-attention verification intact; "Strong Drafts Need Compact
Memories: Long-Context Speculative Decoding with Compressed KV Cache" (4.1,
Appendix C) -- the draft's working memory adds compressed memory slots to the
sinks and the window.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.ring_model import StreamingCache

TIGHT = 1e-12


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float64).to(torch.bfloat16)


def f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def rand_bf16(shape, gen, std=1.0):
    return (torch.randn(shape, generator=gen, dtype=torch.float64) * std).to(torch.bfloat16)


def close(a, b, tol=TIGHT):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return a.shape == b.shape and np.allclose(a, b, rtol=tol, atol=tol, equal_nan=False)


# ---------------------------------------------------------------- closed forms

def test_one_key_returns_its_value():
    g = torch.Generator().manual_seed(1)
    q, k, v = rand_bf16((64,), g), rand_bf16((1, 64), g), rand_bf16((1, 64), g)
    out, lse = oracle.attend_subset(q, k, v, [True], scale=0.37)
    assert np.array_equal(out, f64(v[0]).numpy())
    assert lse == pytest.approx(0.37 * float(f64(q) @ f64(k[0])), rel=1e-14, abs=1e-14)


def test_identical_keys_give_mean_value_and_log_count():
    g = torch.Generator().manual_seed(2)
    n, D = 9, 32
    q = rand_bf16((D,), g)
    k = rand_bf16((1, D), g).repeat(n, 1)
    v = rand_bf16((n, D), g)
    out, lse = oracle.attend_subset(q, k, v, [True] * n, scale=0.5)
    assert close(out, f64(v).mean(0).numpy())
    logit = 0.5 * float(f64(q) @ f64(k[0]))
    assert lse == pytest.approx(logit + math.log(n), rel=1e-13)


def test_zero_query_averages_the_member_values():
    g = torch.Generator().manual_seed(3)
    n, D = 40, 16
    q = torch.zeros(D, dtype=torch.bfloat16)
    k, v = rand_bf16((n, D), g), rand_bf16((n, D), g)
    member = (torch.rand(n, generator=g) < 0.4).numpy()
    out, lse = oracle.attend_subset(q, k, v, member, scale=1.0)
    assert close(out, f64(v)[torch.from_numpy(member)].mean(0).numpy())
    assert lse == pytest.approx(math.log(member.sum()), rel=1e-14)


def test_constant_values_pass_through():
    g = torch.Generator().manual_seed(4)
    n, D = 33, 64
    c = rand_bf16((D,), g)
    out, _ = oracle.attend_subset(rand_bf16((D,), g), rand_bf16((n, D), g, 3.0), c.repeat(n, 1),
                                  [True] * n, scale=1.0)
    assert close(out, f64(c).numpy())


def test_two_keys_follow_logistic_weights():
    # logits are chosen as exact bf16 products: q = e0, k_i = a_i e0.
    D = 8
    q = bf16([1.0] + [0.0] * (D - 1))
    k = bf16([[1.5] + [0.0] * (D - 1), [-0.25] + [0.0] * (D - 1)])
    v = bf16([[1.0, 2.0, 0, 0, 0, 0, 0, 4.0], [-3.0, 0.5, 0, 0, 0, 0, 1.0, 0]])
    out, lse = oracle.attend_subset(q, k, v, [True, True], scale=2.0)
    a, b = 3.0, -0.5
    w1 = 1.0 / (1.0 + math.exp(b - a))
    assert close(out, (w1 * f64(v[0]) + (1 - w1) * f64(v[1])).numpy())
    assert lse == pytest.approx(float(np.logaddexp(a, b)), rel=1e-15)


def test_empty_key_set():
    g = torch.Generator().manual_seed(5)
    out, lse = oracle.attend_subset(rand_bf16((8,), g), rand_bf16((4, 8), g), rand_bf16((4, 8), g),
                                    [False] * 4, scale=1.0)
    assert np.all(out == 0) and lse == -math.inf


# ------------------------------------------------------------ library routes

def test_subset_matches_dense_torch_softmax():
    g = torch.Generator().manual_seed(6)
    for n, D in [(1, 64), (17, 128), (300, 256)]:
        q, k, v = rand_bf16((D,), g), rand_bf16((n, D), g), rand_bf16((n, D), g)
        member = torch.rand(n, generator=g) < 0.6
        member[0] = True
        s = 1 / math.sqrt(D)
        logits = (f64(k)[member] @ f64(q)) * s
        ref = torch.softmax(logits, 0) @ f64(v)[member]
        out, lse = oracle.attend_subset(q, k, v, member.numpy(), scale=s)
        assert close(out, ref.numpy())
        assert lse == pytest.approx(float(torch.logsumexp(logits, 0)), rel=1e-13)


def _verify_case(plant=0, T=3, N=150, Hq=8, Hkv=2, D=32, B=2, seed=7):
    """Oracle verify vs PyTorch SDPA (its causal mask, its GQA mapping) in fp64."""
    g = torch.Generator().manual_seed(seed)
    k = rand_bf16((B, Hkv, N + 5, D), g)
    v = rand_bf16((B, Hkv, N + 5, D), g)
    lens = [N, N - 37][:B]
    q = rand_bf16((B, T, Hq, D), g, 0.3)
    s = 0.7
    out, lse = oracle.verify(oracle.KV(k, v), q, lens, s, plant=plant)
    out = out.reshape(B, T, Hq, D)
    lse = lse.reshape(B, T, Hq)
    ok = True
    for b in range(B):
        n = lens[b]
        # A full square causal self-attention whose last T query rows are ours.
        qf = rand_bf16((Hq, n, D), g, 0.3)
        qf[:, n - T:, :] = q[b].transpose(0, 1)
        kb, vb = f64(k[b, :, :n]), f64(v[b, :, :n])
        ref = torch.nn.functional.scaled_dot_product_attention(
            f64(qf)[None], kb[None], vb[None], is_causal=True, scale=s, enable_gqa=True)[0]
        ok &= close(out[b].transpose(1, 0, 2), ref[:, n - T:, :].numpy(), 1e-11)
        # lse from the library's logsumexp over the causal logits
        G = Hq // Hkv
        for h in range(Hq):
            for i in range(T):
                P = n - T + i
                logit = (kb[h // G, :P + 1] @ f64(q[b, i, h])) * s
                ok &= abs(float(torch.logsumexp(logit, 0)) - lse[b, i, h]) < 1e-11
    return ok


def test_verify_matches_torch_sdpa_causal_gqa():
    assert _verify_case()


def test_verify_single_position_is_full_attention():
    g = torch.Generator().manual_seed(8)
    N, D = 64, 16
    k, v = rand_bf16((1, 1, N, D), g), rand_bf16((1, 1, N, D), g)
    q = rand_bf16((1, 1, 1, D), g)
    out, lse = oracle.verify(oracle.KV(k, v), q, [N], 0.25)
    ref, ref_lse = oracle.attend_subset(q.reshape(-1), k[0, 0], v[0, 0], [True] * N, 0.25)
    assert np.array_equal(out[0], ref) and lse[0] == ref_lse


def test_gqa_contiguous_groups_closed_form():
    # KV head g holds a constant value c_g, so query head h must return c_{h // G}.
    Hq, Hkv, D, N = 8, 2, 16, 20
    g = torch.Generator().manual_seed(9)
    k = rand_bf16((1, Hkv, N, D), g)
    v = torch.empty((1, Hkv, N, D), dtype=torch.bfloat16)
    consts = [0.5, -2.0]
    for h in range(Hkv):
        v[0, h] = consts[h]
    q = rand_bf16((1, 1, Hq, D), g)
    out, _ = oracle.verify(oracle.KV(k, v), q, [N], 1.0)
    for h in range(Hq):
        assert np.all(out[h] == consts[h // (Hq // Hkv)])


def _paged_case(plant=0, seed=10):
    """Paged store == contiguous store of the same logical cache (bit-identical)."""
    g = torch.Generator().manual_seed(seed)
    B, Hkv, D, ps, T, Hq = 3, 2, 16, 8, 2, 4
    lens = [45, 17, 64]
    cap = 64
    k = rand_bf16((B, Hkv, cap, D), g)
    v = rand_bf16((B, Hkv, cap, D), g)
    n_pages_b = [-(-n // ps) for n in lens]
    P = sum(n_pages_b)
    perm = torch.randperm(P, generator=g)
    bt = torch.full((B, max(n_pages_b)), -1, dtype=torch.int32)
    kp = torch.zeros((P, Hkv, ps, D), dtype=torch.bfloat16)
    vp = torch.zeros((P, Hkv, ps, D), dtype=torch.bfloat16)
    off = 0
    for b in range(B):
        for i in range(n_pages_b[b]):
            page = int(perm[off + i])
            bt[b, i] = page
            kp[page] = k[b, :, i * ps:(i + 1) * ps]
            vp[page] = v[b, :, i * ps:(i + 1) * ps]
        off += n_pages_b[b]
    q = rand_bf16((B, T, Hq, D), g)
    a = oracle.verify(oracle.KV(k, v), q, lens, 0.3, plant=plant)
    p = oracle.verify(oracle.KV(kp, vp, bt), q, lens, 0.3, plant=plant)
    return np.array_equal(a[0], p[0]) and np.array_equal(a[1], p[1])


def test_paged_equals_contiguous():
    assert _paged_case()


# ----------------------------------------------------- draft key set (window)

def _draft_bruteforce(plant=0, n_tok=16, D=16):
    """Every S in 0..16, W in 1..16, p in 0..15: the oracle's sink+window draft
    equals dense fp64 attention over exactly the positions a sink-list +
    deque(maxlen=W) cache holds after appending positions 0..p."""
    g = torch.Generator().manual_seed(11)
    k = rand_bf16((1, 1, n_tok, D), g)
    v = rand_bf16((1, 1, n_tok, D), g)
    kv = oracle.KV(k, v)
    q = rand_bf16((1, 2, D), g)  # two query heads sharing the one KV head
    kd, vd = f64(k[0, 0]), f64(v[0, 0])
    for S in range(0, n_tok + 1):
        for W in range(1, n_tok + 1):
            cache = StreamingCache(S, W)
            for p in range(n_tok):
                cache.append(p)
                held = torch.tensor(cache.held())
                out, lse = oracle.draft(kv, q, [p], S, W, 0.5, plant=plant)
                for h in range(2):
                    logit = (kd[held] @ f64(q[0, h])) * 0.5
                    ref = torch.softmax(logit, 0) @ vd[held]
                    if not (close(out[h], ref.numpy(), 1e-12)
                            and abs(lse[h] - float(torch.logsumexp(logit, 0))) < 1e-12):
                        return False
    return True


def test_draft_keyset_bruteforce_16_tokens():
    assert _draft_bruteforce()


def test_window_covering_the_prefix_equals_full_attention():
    g = torch.Generator().manual_seed(12)
    N, D, Hq = 300, 32, 4
    k, v = rand_bf16((1, 2, N, D), g), rand_bf16((1, 2, N, D), g)
    kv = oracle.KV(k, v)
    q = rand_bf16((1, Hq, D), g)
    for p, S, W in [(0, 0, 1), (99, 4, 96), (99, 0, 100), (299, 16, 284), (299, 300, 5)]:
        d_out, d_lse = oracle.draft(kv, q, [p], S, W, 0.2)
        f_out, f_lse = oracle.verify(kv, q[:, None], [p + 1], 0.2)
        assert np.array_equal(d_out, f_out) and np.array_equal(d_lse, f_lse)


def test_pure_sliding_window_is_a_contiguous_slice():
    # S = 0 reduces to plain sliding-window attention over positions p-W+1..p.
    g = torch.Generator().manual_seed(13)
    N, D, W = 500, 64, 37
    k, v = rand_bf16((1, 1, N, D), g), rand_bf16((1, 1, N, D), g)
    q = rand_bf16((1, 1, D), g)
    out, lse = oracle.draft(oracle.KV(k, v), q, [411], 0, W, 0.125)
    kd, vd = f64(k[0, 0, 411 - W + 1:412]), f64(v[0, 0, 411 - W + 1:412])
    logit = (kd @ f64(q[0, 0])) * 0.125
    assert close(out[0], (torch.softmax(logit, 0) @ vd).numpy())
    assert lse[0] == pytest.approx(float(torch.logsumexp(logit, 0)), rel=1e-13)


def test_window_of_one_without_sinks_returns_the_current_value():
    g = torch.Generator().manual_seed(14)
    k, v = rand_bf16((1, 1, 50, 16), g), rand_bf16((1, 1, 50, 16), g)
    out, _ = oracle.draft(oracle.KV(k, v), rand_bf16((1, 1, 16), g), [23], 0, 1, 1.0)
    assert np.array_equal(out[0], f64(v[0, 0, 23]).numpy())


def test_held_count_is_min_of_prefix_and_slots():
    for S, W in [(0, 1), (4, 256), (16, 50)]:
        c = StreamingCache(S, W)
        for p in range(400):
            c.append(p)
            assert len(c.held()) == min(p + 1, S + W)


# --------------------------------------------------------- merge / invariance

def test_merge_of_parts_equals_single_pass():
    g = torch.Generator().manual_seed(15)
    n, D = 200, 64
    q, k, v = rand_bf16((D,), g, 2.0), rand_bf16((n, D), g), rand_bf16((n, D), g)
    full, full_lse = oracle.attend_subset(q, k, v, [True] * n, 0.3)
    for n_parts in (1, 2, 7, 30):
        owner = torch.randint(0, n_parts + 1, (n,), generator=g)  # part n_parts stays empty
        owner[owner == n_parts] = 0
        o_parts = np.zeros((1, n_parts + 1, D))
        l_parts = np.zeros((1, n_parts + 1))
        for s in range(n_parts + 1):
            o_parts[0, s], l_parts[0, s] = oracle.attend_subset(q, k, v, (owner == s).numpy(), 0.3)
        assert l_parts[0, n_parts] == -math.inf
        out, lse = oracle.lse_merge(o_parts, l_parts)
        assert close(out[0], full) and lse[0] == pytest.approx(full_lse, rel=1e-13)


def test_merge_of_only_empty_parts():
    out, lse = oracle.lse_merge(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_key_order_does_not_matter():
    g = torch.Generator().manual_seed(16)
    n, D = 120, 32
    q, k, v = rand_bf16((D,), g), rand_bf16((n, D), g), rand_bf16((n, D), g)
    member = (torch.rand(n, generator=g) < 0.5).numpy()
    a = oracle.attend_subset(q, k, v, member, 0.4)
    perm = torch.randperm(n, generator=g)
    b = oracle.attend_subset(q, k[perm], v[perm], member[perm.numpy()], 0.4)
    assert close(a[0], b[0]) and a[1] == pytest.approx(b[1], rel=1e-13)


# ------------------------------------------------------------ memory slots

def _draft_mem_case(plant=0, seed=21):
    """Memory-augmented draft: for several (S, W, p, slot count) the oracle
    equals dense fp64 softmax attention (torch) over the keys a sink-list +
    deque cache holds after positions 0..p, concatenated with the first
    `count` memory slots -- per sequence, with two query heads per KV head."""
    g = torch.Generator().manual_seed(seed)
    B, Hkv, G, N, cap, D = 2, 2, 2, 60, 9, 16
    k, v = rand_bf16((B, Hkv, N, D), g), rand_bf16((B, Hkv, N, D), g)
    mk, mv = rand_bf16((B, Hkv, cap, D), g), rand_bf16((B, Hkv, cap, D), g)
    hist, mem = oracle.KV(k, v), oracle.KV(mk, mv)
    for S, W, pos, counts in [(4, 8, [59, 30], [9, 3]), (0, 5, [10, 59], [1, 0]), (2, 60, [59, 0], [4, 9]),
                              (1, 1, [0, 1], [9, 9])]:
        q = rand_bf16((B, Hkv * G, D), g)
        out, lse = oracle.draft_mem(hist, mem, counts, q, pos, S, W, 0.4, plant=plant)
        for b in range(B):
            cache = StreamingCache(S, W)
            for p in range(pos[b] + 1):
                cache.append(p)
            held = torch.tensor(cache.held(), dtype=torch.long)
            for h in range(Hkv * G):
                kvh = h // G
                keys = torch.cat([f64(k[b, kvh])[held], f64(mk[b, kvh, :counts[b]])])
                vals = torch.cat([f64(v[b, kvh])[held], f64(mv[b, kvh, :counts[b]])])
                logit = (keys @ f64(q[b, h])) * 0.4
                ref = torch.softmax(logit, 0) @ vals
                r = b * Hkv * G + h
                if not (close(out[r], ref.numpy()) and abs(lse[r] - float(torch.logsumexp(logit, 0))) < 1e-12):
                    return False
    return True


def test_draft_with_memory_slots_matches_dense_softmax_over_the_union():
    assert _draft_mem_case()


def test_no_memory_slot_reduces_to_the_windowed_draft():
    g = torch.Generator().manual_seed(22)
    B, Hkv, N, D = 2, 2, 80, 32
    k, v = rand_bf16((B, Hkv, N, D), g), rand_bf16((B, Hkv, N, D), g)
    mk, mv = rand_bf16((B, Hkv, 5, D), g), rand_bf16((B, Hkv, 5, D), g)
    q = rand_bf16((B, 4, D), g)
    a = oracle.draft(oracle.KV(k, v), q, [79, 40], 4, 16, 0.3)
    m = oracle.draft_mem(oracle.KV(k, v), oracle.KV(mk, mv), [0, 0], q, [79, 40], 4, 16, 0.3)
    assert np.array_equal(a[0], m[0]) and np.array_equal(a[1], m[1])


def test_memory_slot_equal_to_a_window_key_counts_twice():
    # A slot holding a copy of the query's own key and value: exactly the
    # two-key closed form when the window holds only that key.
    g = torch.Generator().manual_seed(23)
    D = 16
    k, v = rand_bf16((1, 1, 3, D), g), rand_bf16((1, 1, 3, D), g)
    mk, mv = k[:, :, 2:3].clone(), v[:, :, 2:3].clone()
    q = rand_bf16((1, 1, D), g)
    out, lse = oracle.draft_mem(oracle.KV(k, v), oracle.KV(mk, mv), [1], q, [2], 0, 1, 0.5)
    l2 = 0.5 * float(f64(k[0, 0, 2]) @ f64(q[0, 0]))
    assert close(out[0], f64(v[0, 0, 2]).numpy())
    assert lse[0] == pytest.approx(l2 + math.log(2.0), rel=1e-13, abs=1e-13)


# ------------------------------------------------------------ planted mistakes

PLANTS = {
    1: "window excludes the query's own position",
    2: "window one position too wide",
    3: "attention sinks dropped",
    4: "softmax scale ignored",
    5: "GQA heads interleaved instead of grouped",
    6: "verify query drops its own key",
    7: "log-sum-exp loses its max term",
    8: "block table row of sequence 0 used for every sequence",
    9: "newest memory slot dropped",
}


def _passes(pin, plant):
    try:
        return pin(plant=plant)
    except ValueError:  # the oracle rejected its own reads: also a caught mistake
        return False


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_planted_mistakes_are_caught(plant):
    caught = (not _passes(_verify_case, plant) or not _passes(_paged_case, plant)
              or not _passes(lambda plant: _draft_bruteforce(plant=plant, n_tok=12), plant)
              or not _passes(_draft_mem_case, plant))
    assert caught, f"no pin caught the planted mistake: {PLANTS[plant]}"


def test_unplanted_oracle_passes_the_planted_suite():
    assert _verify_case() and _paged_case() and _draft_bruteforce(n_tok=12) and _draft_mem_case()
