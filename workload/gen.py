"""Seeded generators for the inputs of the decode-step KV path.

Both the CUDA path and the CPU oracle are fed from here; this module holds none
of the path's arithmetic (no top-k, no plan, no gather, no attention).

* Latent KV rows and queries: standard-normal bf16 values from the
  counter-based generator in `_gen.c` (SplitMix64 + Box-Muller), keyed by
  (seed, domain, a, b, row), so that any single row can be regenerated.
* Indexer scores: float32, one array [B][ctx_stride] per decode step, from
  numpy's PCG64 streams, one per request. Positions at or beyond a request's
  context length hold NaN, so a reader that strays past the context notices.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile
import threading

import numpy as np

from .configs import D, Workload

DOMAIN_KV = 1
DOMAIN_Q = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "_gen.c")
_SO = os.path.join(_HERE, "_gen.so")
_lock = threading.Lock()
_lib = None


def build_native(force: bool = False) -> str:
    """Compile `_gen.c` into `_gen.so` beside it (gcc, host architecture)."""
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _SO


def _native():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_native())
            lib.gen_normal_bf16.restype = ctypes.c_int
            lib.gen_normal_bf16.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(n_rows: int, dim: int, seed: int, domain: int, a: int, b: int,
                row0: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """Rows row0 .. row0+n_rows-1 of `dim` N(0,1) bf16 values (uint16 bits)."""
    if out is None:
        out = np.empty((n_rows, dim), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.ndim == 2 and out.shape == (n_rows, dim)
    assert out.strides[1] == 2
    if n_rows == 0:
        return out
    _native().gen_normal_bf16(out.ctypes.data, out.strides[0] // 2, dim,
                              seed, domain, a, b, row0, n_rows, _threads())
    return out


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values (exact)."""
    return (x.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Context lengths, latent KV rows, queries
# --------------------------------------------------------------------------

def ctx_lens(w: Workload, first_request: int = 0) -> np.ndarray:
    """Context length of requests first_request .. first_request+B-1 (int32 [B])."""
    if w.ctx_lo == w.ctx:
        return np.full(w.B, w.ctx, dtype=np.int32)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 11])))
    return rng.integers(w.ctx_lo, w.ctx + 1,
                        size=first_request + w.B)[first_request:].astype(np.int32)


def fill_host_kv(w: Workload, out: np.ndarray, layers=None, requests=None,
                 first_request: int = 0) -> None:
    """Write the latent rows of every (layer, request) into `out`
    ([layers][B][ctx_stride][576] uint16); rows past a request's context are
    left as they are. Request b of `out` is request first_request + b of the
    workload."""
    assert out.shape == (w.layers, w.B, w.ctx_stride, D) and out.dtype == np.uint16
    lens = ctx_lens(w, first_request)
    for l in (range(w.layers) if layers is None else layers):
        for b in (range(w.B) if requests is None else requests):
            n = int(lens[b])
            normal_bf16(n, D, w.seed, DOMAIN_KV, l, first_request + b, 0, out[l, b, :n])


def host_kv_rows(w: Workload, layer: int, b: int, rows) -> np.ndarray:
    """Regenerate chosen latent rows of one (layer, request): uint16 [n][576]."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, D), dtype=np.uint16)
    for i, t in enumerate(rows):
        normal_bf16(1, D, w.seed, DOMAIN_KV, layer, b, int(t), out[i:i + 1])
    return out


def queries(w: Workload, step: int, out: np.ndarray | None = None,
            first_request: int = 0) -> np.ndarray:
    """Queries of one decode step: uint16 [layers][B][H][576]."""
    if out is None:
        out = np.empty((w.layers, w.B, w.H, D), dtype=np.uint16)
    for l in range(w.layers):
        for b in range(w.B):
            normal_bf16(w.H, D, w.seed, DOMAIN_Q, step, (l << 32) | (first_request + b), 0,
                        out[l, b])
    return out


# --------------------------------------------------------------------------
# Indexer scores
# --------------------------------------------------------------------------

def _upper_tail(x: float) -> float:
    return 0.5 * math.erfc(x / math.sqrt(2.0))


def _both_above(a: float, rho: float) -> float:
    """P(X > a, Y > a) for a standard bivariate normal with correlation rho."""
    from scipy.stats import multivariate_normal
    if rho >= 1.0:
        return _upper_tail(a)
    cov = [[1.0, rho], [rho, 1.0]]
    # P(X>a, Y>a) = P(-X < -a, -Y < -a) = Phi2(-a, -a; rho)
    return float(multivariate_normal(mean=[0.0, 0.0], cov=cov).cdf([-a, -a]))


def calibrate_rho(frac: float, overlap: float, hot_frac: float = 0.0,
                  hot_offset: float = 0.0) -> float:
    """Correlation of consecutive steps' scores for which the expected top-k
    overlap of adjacent steps is `overlap`, when a fraction `frac` of the
    positions is selected and a fraction `hot_frac` of the positions sits
    `hot_offset` sigma higher (large-context limit, closed form through the
    bivariate normal orthant probability)."""
    from scipy.optimize import brentq

    def sel(t):
        return (1 - hot_frac) * _upper_tail(t) + hot_frac * _upper_tail(t - hot_offset)

    t = brentq(lambda x: sel(x) - frac, -20.0, 20.0, xtol=1e-12)

    def ov(rho):
        both = (1 - hot_frac) * _both_above(t, rho)
        if hot_frac:
            both += hot_frac * _both_above(t - hot_offset, rho)
        return both / frac

    if ov(0.0) >= overlap:
        return 0.0
    return float(brentq(lambda r: ov(r) - overlap, 0.0, 0.999999, xtol=1e-7))


class ScoreStream:
    """Indexer scores, one decode step at a time: `next()` returns float32
    [B][ctx_stride]. The process per workload:

    * 'walk'     : step 0 U(0,1); then previous + N(0, walk_sigma).
    * 'ar1'      : s_t = rho s_{t-1} + sqrt(1-rho^2) e_t, e ~ N(0,1), rho
                   calibrated per request for the target overlap.
    * 'ar1_hot'  : 'ar1' plus hot_offset on a hot set of hot_frac of the
                   positions; each step hot_drift of the members are replaced
                   by random non-members.
    * 'iid_ties' : independent N(0,1) each step; a fresh tie_frac of the
                   positions rounded to the tie_grid; request overflow_request
                   gets overflow_boost on overflow_count fresh positions of set
                   overflow_set (position mod S) each step.
    """

    def __init__(self, w: Workload, first_request: int = 0):
        self.w = w
        self.lens = ctx_lens(w, first_request)
        self.step = 0
        self.rngs = [np.random.Generator(np.random.PCG64(
            np.random.SeedSequence([w.seed, 7, first_request + b]))) for b in range(w.B)]
        self.state = [None] * w.B
        self.hot = [None] * w.B
        self.rho = [0.0] * w.B
        if w.scores in ("ar1", "ar1_hot"):
            cache = {}
            for b in range(w.B):
                n = int(self.lens[b])
                key = n
                if key not in cache:
                    cache[key] = calibrate_rho(w.k / n, w.overlap, w.hot_frac, w.hot_offset)
                self.rho[b] = cache[key]

    def _one(self, b: int) -> np.ndarray:
        w, rng, n = self.w, self.rngs[b], int(self.lens[b])
        if w.scores == "walk":
            if self.state[b] is None:
                s = rng.random(n)
            else:
                s = self.state[b] + rng.normal(0.0, w.walk_sigma, n)
            self.state[b] = s
            return s.astype(np.float32)
        if w.scores in ("ar1", "ar1_hot"):
            e = rng.standard_normal(n)
            if self.state[b] is None:
                s = e
            else:
                r = self.rho[b]
                s = r * self.state[b] + math.sqrt(1.0 - r * r) * e
            self.state[b] = s
            if w.scores == "ar1":
                return s.astype(np.float32)
            if self.hot[b] is None:
                self.hot[b] = rng.permutation(n)[: int(round(w.hot_frac * n))]
            else:
                hot = self.hot[b]
                m = int(round(w.hot_drift * hot.size))
                if m:
                    mask = np.zeros(n, dtype=bool)
                    mask[hot] = True
                    out_i = rng.choice(hot.size, size=m, replace=False)
                    cand = np.flatnonzero(~mask)
                    new = cand[rng.choice(cand.size, size=m, replace=False)]
                    hot = hot.copy()
                    hot[out_i] = new
                    self.hot[b] = hot
            s = s.copy()
            s[self.hot[b]] += w.hot_offset
            return s.astype(np.float32)
        if w.scores == "iid_ties":
            s = rng.standard_normal(n)
            q = rng.choice(n, size=int(round(w.tie_frac * n)), replace=False)
            s[q] = np.round(s[q] / w.tie_grid) * w.tie_grid
            if b == w.overflow_request:
                members = np.arange(w.overflow_set, n, w.S)
                pick = rng.choice(members.size, size=w.overflow_count, replace=False)
                s[members[pick]] += w.overflow_boost
            return s.astype(np.float32)
        raise ValueError(w.scores)

    def next(self) -> np.ndarray:
        w = self.w
        out = np.full((w.B, w.ctx_stride), np.nan, dtype=np.float32)
        for b in range(w.B):
            out[b, : int(self.lens[b])] = self._one(b)
        self.step += 1
        return out
