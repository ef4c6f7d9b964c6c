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
    """Elementwise check of (out, lse) against the oracle.  Every comparison is
    written so that a NaN or an infinity on the GPU side fails it (a
    comparison with NaN is False, so the checks test for being inside the
    tolerance, never for being outside it)."""
    g = got.float().cpu().numpy().reshape(ref.shape)
    gl = got_lse.float().cpu().numpy().reshape(ref_lse.shape)
    assert np.isfinite(ref).all(), f"{name}: the oracle's outputs must be finite"
    n_bad_vals = int((~np.isfinite(g)).sum())
    assert n_bad_vals == 0, f"{name}: {n_bad_vals}/{g.size} outputs are NaN or infinite"
    err = np.abs(g - ref)
    ok = err <= ATOL + RTOL * np.abs(ref)
    assert ok.all(), (f"{name}: {int((~ok).sum())}/{ok.size} outputs outside tolerance; "
                      f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    fin = np.isfinite(ref_lse)
    assert not np.isnan(ref_lse).any() and not (ref_lse == np.inf).any(), f"{name}: oracle lse must be finite or -inf"
    assert np.array_equal(fin, np.isfinite(gl)), f"{name}: lse finiteness differs (NaN or inf on the GPU side?)"
    if fin.any():
        le = np.abs(gl[fin] - ref_lse[fin])
        assert (le <= LSE_TOL).all(), f"{name}: lse max err {le.max():.3e}"
    if (~fin).any():
        rows = g.reshape(gl.size, -1)[~fin.reshape(-1)]
        assert (gl[~fin] == -np.inf).all() and (rows == 0).all(), f"{name}: empty rows must be 0 / -inf"


def nan_like(t: torch.Tensor) -> torch.Tensor:
    """An output buffer pre-filled with NaN, so that a row a kernel never
    writes cannot pass as a result."""
    return torch.full_like(t, float("nan"))


def oracle_kv(k: torch.Tensor, v: torch.Tensor, block_table: torch.Tensor | None = None):
    return oracle.KV(k.cpu(), v.cpu(), None if block_table is None else block_table.cpu())
