"""Helpers for the GPU parity tests: move generator bits to the device, call the
library through its C ABI binding, compare with the fp64 oracle.

Tolerances (from the workload definition): O, dQ, dK, dV within 2e-2 of the oracle
in max-abs error normalised by the oracle's max magnitude; LSE within 1e-3
absolute; every output finite. The normaliser has a floor of 1e-2: where every
softmax row has a single allowed key (S = 1, window = 1) the exact dQ is zero and
the GPU returns fp32 rounding residue, which is then compared in absolute terms.
"""
import numpy as np
import torch

TOL_REL = 2e-2
TOL_LSE = 1e-3
NORM_FLOOR = 1e-2


def to_dev(bits, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16).to(dev)


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_err(got, ref):
    ref = np.asarray(ref, np.float64)
    den = max(float(np.max(np.abs(ref))), NORM_FLOOR)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref))) / den


def check(name, got, ref):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite output"
    e = rel_err(got, ref)
    assert e <= TOL_REL, f"{name}: normalised max error {e:.3e} > {TOL_REL}"
    return e


def check_lse(name, got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: finiteness differs"
    assert np.array_equal(got[~fin], ref[~fin]), f"{name}: non-finite values differ"
    e = float(np.max(np.abs(got[fin] - ref[fin]))) if fin.any() else 0.0
    assert e <= TOL_LSE, f"{name}: max abs error {e:.3e} > {TOL_LSE}"
    return e
