"""Helpers shared by the GPU parity tests: tolerances and oracle calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

# Tolerance on bf16 outputs: |gpu - ref| <= ATOL + RTOL * |ref| elementwise
# (max |err| 2e-3, relative 1e-2); lse: |gpu - ref| <= LSE_TOL.
ATOL, RTOL, LSE_TOL = 2e-3, 1e-2, 2e-3


def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_attention_gb300 import build as wm_build
    wm_build.build()
    return torch.device("cuda:0")


def assert_close(name: str, got: torch.Tensor, got_lse: torch.Tensor, ref: np.ndarray,
                 ref_lse: np.ndarray) -> None:
    g = got.float().cpu().numpy().reshape(ref.shape)
    gl = got_lse.float().cpu().numpy().reshape(ref_lse.shape)
    err = np.abs(g - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{name}: {int(bad.sum())}/{bad.size} outputs outside tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(gl)), f"{name}: lse finiteness differs"
    if fin.any():
        le = np.abs(gl[fin] - ref_lse[fin])
        assert le.max() <= LSE_TOL, f"{name}: lse max err {le.max():.3e}"
    if (~fin).any():
        assert np.all(gl[~fin] == -np.inf) and np.all(g.reshape(len(gl.reshape(-1)), -1)[~fin.reshape(-1)]
                                                      == 0), f"{name}: empty rows must be 0 / -inf"


def oracle_kv(k: torch.Tensor, v: torch.Tensor, block_table: torch.Tensor | None = None):
    return oracle.KV(k.cpu(), v.cpu(), None if block_table is None else block_table.cpu())
