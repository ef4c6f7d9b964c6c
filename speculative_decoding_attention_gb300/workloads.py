"""The five decode-attention workloads: shapes, window sizes and value recipes.

Each workload is one speculative-decoding step of the Windowed-MTP setting
("Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
Context", Abstract): d sequential draft steps, each appending one entry to the
draft's sink + window ring buffer and attending over it, then verification of
T = d + 1 proposed positions over the full bf16 KV cache.

This module holds shapes and recipes only -- none of the method's arithmetic.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    context: int                 # N (ignored when ``ragged`` is set)
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    sink: int                    # S
    window: int                  # W
    depths: tuple[int, ...]      # draft depths d; verify uses T = d + 1
    q_std: float                 # q entries ~ N(0, q_std^2)
    scale: float                 # softmax scale handed to the kernels
    seed: int
    ragged: tuple[int, int] | None = None  # contexts ~ U[lo, hi] per sequence
    page_size: int = 0           # 0: contiguous cache; else paged with this page size
    peaked_frac: float = 0.0     # fraction of key positions whose K is scaled ...
    peaked_gain: float = 1.0     # ... by this gain (before bf16 rounding)
    ring_appends: int = 0        # trailing context positions appended one by one

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def slots(self) -> int:
        return self.sink + self.window

    @property
    def max_depth(self) -> int:
        return max(self.depths)

    def describe(self) -> str:
        ctx = f"{self.ragged[0]}-{self.ragged[1]} ragged" if self.ragged else str(self.context)
        kv = f"paged{self.page_size}" if self.page_size else "contiguous"
        return (f"{self.name}: B={self.batch} N={ctx} Hq={self.n_q_heads} Hkv={self.n_kv_heads} "
                f"D={self.head_dim} S={self.sink} W={self.window} depths={self.depths} {kv}")


WORKLOADS: dict[str, Workload] = {
    # 1 sequence, 4K context, GQA 4, D=128; S=4, W=256 (260-slot ring); 1 draft step, verify 2.
    "tiny_4k": Workload("tiny_4k", batch=1, context=4096, n_q_heads=8, n_kv_heads=2, head_dim=128,
                        sink=4, window=256, depths=(1,), q_std=1 / math.sqrt(128), scale=1.0,
                        seed=1001),
    # 1 sequence, 128K context, GQA 8, D=128, RoPE already applied to cached K; 3 draft steps, verify 4.
    "gqa8_128k": Workload("gqa8_128k", batch=1, context=131072, n_q_heads=32, n_kv_heads=4,
                          head_dim=128, sink=4, window=2048, depths=(3,), q_std=1.0,
                          scale=1 / math.sqrt(128), seed=1002),
    # 1 sequence, 1M context, full-attention layer of a hybrid linear/full target: GQA 8, D=256;
    # S=4, W=4096; draft depths 1, 3, 5; 1% of keys scaled x8 (peaked softmax).
    "hybrid_1m_d256": Workload("hybrid_1m_d256", batch=1, context=1048576, n_q_heads=16,
                               n_kv_heads=2, head_dim=256, sink=4, window=4096, depths=(1, 3, 5),
                               q_std=1.0, scale=1 / math.sqrt(256), seed=1003, peaked_frac=0.01,
                               peaked_gain=8.0),
    # 8 sequences, ragged contexts U[32K, 512K], paged KV (64-token pages, permuted pool);
    # GQA 4, D=128; S=4, W=1024; 2 draft steps, verify 3.
    "paged_ragged_b8": Workload("paged_ragged_b8", batch=8, context=524288, n_q_heads=32,
                                n_kv_heads=8, head_dim=128, sink=4, window=1024, depths=(2,),
                                q_std=1.0, scale=1 / math.sqrt(128), seed=1004,
                                ragged=(32768, 524288), page_size=64),
    # NoPE attention at 1M context, batch 2, GQA 8, D=128; S=16, W=8192 ring that wraps over the
    # last 20,000 positions appended one at a time; draft depth 4, verify 5.
    "nope_1m_b2": Workload("nope_1m_b2", batch=2, context=1048576, n_q_heads=64, n_kv_heads=8,
                           head_dim=128, sink=16, window=8192, depths=(4,),
                           q_std=1 / math.sqrt(128), scale=1.0, seed=1005, ring_appends=20000),
}

# The single-GPU workload the benchmark times by default (1M context).
BENCH_WORKLOAD = "hybrid_1m_d256"
BENCH_DEPTH = 3


def get(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None
