"""Helpers shared by the GPU parity tests: run the block through the C ABI and
through the oracle on the same seeded inputs, and measure the error."""
from __future__ import annotations

import numpy as np
import torch

import workloads
from oracle import block as ob
from oracle.bf16 import round_bf16, identity
from tests.parity_log import record_parity  # noqa: F401  (re-exported for the tests)

BF16_TOL = 2e-2
F32_TOL = 1e-4
ULPS = 2      # output-format rounding steps allowed per element (see check_bf16_output)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |err| / rms(ref), the parity metric."""
    return float(np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2)))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (normal range)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def check_bf16_output(got: np.ndarray, exact: np.ndarray, tol: float = BF16_TOL, what: str = "y",
                      assert_: bool = True):
    """Parity of a bf16 output with the oracle.

    ref = the oracle's output (its value rounded to bf16 at the same point);
    rms = rms(ref).  Asserted, per element:
        max(0, |got - ref| - ULPS * ulp(ref)) <= tol * rms
    i.e. the stated bound max|err|/rms(ref) <= tol once rounding steps of the
    output format are allowed: a value next to a bf16 rounding boundary may
    round the other way after last-bit differences upstream (fp32 vs fp64
    accumulation, carried through the block's bf16 rounding points).  The
    output y = R(h + R(branch)) has two rounded inputs, each of which can
    carry such a flip, hence ULPS = 2.  Also asserted: the rms error stays
    below tol / 4 of rms (no systematic drift).  Printed: the raw
    max|err|/rms and the share of elements that differ.
    Returns (raw metric, fraction differing, error beyond the ulps, rms error),
    all relative to rms(ref); ``assert_=False`` only measures."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ref = round_bf16(exact)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    diff = np.abs(got - ref)
    raw = float(np.max(diff)) / rms
    beyond = float(np.max(np.maximum(diff - ULPS * bf16_ulp(ref), 0.0))) / rms
    rms_err = float(np.sqrt(np.mean(diff ** 2))) / rms
    frac = float(np.count_nonzero(diff)) / diff.size
    record_parity(f"[parity] {what}: max|err|/rms = {raw:.3e}, beyond {ULPS} ulps = {beyond:.3e}, "
                  f"rms err = {rms_err:.2e}, differing {100 * frac:.2f}%")
    if assert_:
        assert beyond <= tol, f"{what}: error beyond {ULPS} bf16 ulps = {beyond:.4e} x rms > {tol}"
        assert rms_err <= tol / 4, f"{what}: rms error {rms_err:.3e} > {tol / 4}"
    return raw, frac, beyond, rms_err


def rnd_for(dtype):
    return round_bf16 if dtype == torch.bfloat16 else identity


def oracle_weights(inp: workloads.BlockInputs):
    to64 = workloads.to_numpy64
    return {k: to64(v) for k, v in inp.weights.items()}, {k: to64(v) for k, v in inp.gains.items()}


def gpu_block(inp: workloads.BlockInputs, max_seq: int, device="cuda:0"):
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dev = torch.device(device)
    w = {k: v.to(dev) for k, v in inp.weights.items()}
    g = {k: v.to(dev) for k, v in inp.gains.items()}
    return ddb.LlamaBlock(inp.dims, w, g, max_seq), ddb


def run_prefill(blk, ddb, x_dev, kc_dev, vc_dev):
    kv = ddb.KVCache(kc_dev, vc_dev)
    B, T = x_dev.shape[:2]
    ws = blk.workspace(B, T)
    y = torch.empty_like(x_dev)
    blk.prefill(x_dev, kv, y, ws)
    return y


def run_decode(blk, ddb, x_dev, kc_dev, vc_dev, pos):
    kv = ddb.KVCache(kc_dev, vc_dev)
    ws = blk.workspace(x_dev.shape[0], 1)
    y = torch.empty_like(x_dev)
    blk.decode(x_dev, kv, pos, y, ws)
    return y
