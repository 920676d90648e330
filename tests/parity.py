"""Comparison of the CUDA path against the fp64 oracle.

Tolerances (the parity bar this path is held to, fixed up front, not derived here):
    max |O_gpu - O_ref|              <= 2e-2
    ||O_gpu - O_ref||_2 / ||O_ref||_2 <= 5e-3
    max |LSE_gpu - LSE_ref|          <= 1e-3
O_gpu is bf16, LSE_gpu fp32; the oracle is fp64 on the same bf16 inputs.
"""
from __future__ import annotations

import json
import os

import numpy as np

O_MAX_ABS = 2e-2
O_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3


def metrics(o_gpu, o_ref, lse_gpu, lse_ref):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    lse_gpu = np.asarray(lse_gpu, np.float64)
    lse_ref = np.asarray(lse_ref, np.float64)
    err = np.abs(o_gpu - o_ref)
    denom = np.linalg.norm(o_ref.ravel())
    rel = np.linalg.norm((o_gpu - o_ref).ravel()) / denom if denom > 0 else float(err.max(initial=0))
    lerr = np.abs(lse_gpu - lse_ref)
    return {
        "o_max_abs": float(err.max(initial=0.0)),
        "o_rel_rms": float(rel),
        "lse_max_abs": float(lerr.max(initial=0.0)),
        "finite": bool(np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu))),
        "o_argmax": int(np.argmax(err)) if err.size else -1,
        "lse_argmax": int(np.argmax(lerr)) if lerr.size else -1,
    }


def within(m) -> bool:
    return (m["finite"] and m["o_max_abs"] <= O_MAX_ABS and m["o_rel_rms"] <= O_REL_RMS
            and m["lse_max_abs"] <= LSE_MAX_ABS)


def describe(m) -> str:
    return (f"o_max_abs={m['o_max_abs']:.3e} (<= {O_MAX_ABS}) o_rel_rms={m['o_rel_rms']:.3e} "
            f"(<= {O_REL_RMS}) lse_max_abs={m['lse_max_abs']:.3e} (<= {LSE_MAX_ABS}) "
            f"finite={m['finite']} o_argmax={m['o_argmax']} lse_argmax={m['lse_argmax']}")


def record(label: str, m) -> None:
    """Append the metrics of one case to $PARITY_LOG (JSON lines), if set."""
    path = os.environ.get("PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": label, **m}) + "\n")
