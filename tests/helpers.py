"""Test-side helpers written from the format and layout definitions.

Nothing here is shared with the CUDA path or with the oracle's arithmetic:
the decode tables are built from torch's float8_e4m3fn dtype (a library
routine) and the E2M1 closed form, and the packed-layout unpacking follows
the layout description in include/moe_nvfp4.h.
"""
import math
import os

import numpy as np
import torch

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], np.float64)


def e4m3_table_torch():
    """E4M3(fn) code -> value, decoded by torch (library routine)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant_np(q, s):
    """Canonical NVFP4 [..., rows, k/2] + [..., rows, k/16] -> float64 [..., rows, k]."""
    lo = q & 15
    hi = q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    vals = E2M1_VALUES[codes]
    sc = e4m3_table_torch()[s]
    return vals * np.repeat(sc, 16, axis=-1)


def parse_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def num(tok):
    """Parse decimal, hex-integer or hex-float tokens."""
    t = tok.lower()
    if t in ("nan", "-nan"):
        return float("nan")
    if "p" in t:
        return float.fromhex(t)
    if t.startswith("0x") or t.startswith("-0x"):
        return int(t, 16)
    return float(t)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))
