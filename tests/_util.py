"""Helpers shared by the tests (no arithmetic of the path: conversions,
library build-on-demand, tolerance checks)."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsakv.h")

# SFA tolerance: |delta| <= 1.5e-2 absolute and sum|delta| / sum|ref| <= 2e-3,
# delta measured between the bf16 output and the float64 oracle rounded to
# bf16.
SFA_ABS_TOL = 1.5e-2
SFA_MEAN_REL_TOL = 2e-3


def ensure_library():
    from decode_dsa_kv_gb300 import build
    return build.build()


def header_functions(path=HEADER):
    """Names of the functions declared in a C header."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "while", "defined")]


def bits_to_f64(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sfa_errors(gpu_bits: np.ndarray, ref_bits: np.ndarray):
    g = bits_to_f64(gpu_bits)
    r = bits_to_f64(ref_bits)
    d = np.abs(g - r)
    return float(d.max()), float(d.sum() / max(np.abs(r).sum(), 1e-300))
