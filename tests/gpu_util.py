"""Helpers for the GPU parity tests: moving generator arrays to the device and
comparing results with the tolerances the tests use."""

import numpy as np
import pytest

# Tolerances: fp32 inputs max-abs 1e-5; bf16 inputs (fp32 accumulation)
# max-abs 2e-2 or relative 1e-2 (an element passes if either holds).
TOL_F32 = 1e-5
TOL_BF16_ABS = 2e-2
TOL_BF16_REL = 1e-2


def lib():
    import __graft_entry__
    __graft_entry__.build()
    import tree_speculative_decoding_spec_gb300 as st
    return st


def to_dev(a, dev="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:     # bf16 bit patterns
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    if dtype == "f32":
        bad = err > TOL_F32
    else:
        bad = (err > TOL_BF16_ABS) & (err > TOL_BF16_REL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max():.3e}"
    return float(err.max())
