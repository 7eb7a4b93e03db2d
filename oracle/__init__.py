"""fp64 CPU oracle for Parallax (PLX) attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product path (the CUDA library and its Python binding) never imports, links
or runs it, and the two share no code: the arithmetic lives in
``plx_oracle.c`` (plain C, double precision), compiled by ``oracle/build.py``
with gcc and called here through ctypes.

Forms (see ``plx_oracle.c`` for the formulas and their sources in
"Parallax: Parameterized Local Linear Attention for Language Modeling"):

* ``SA``       -- textbook softmax attention, o^SA = softmax(q K^T * scale) V
* ``EXPLICIT`` -- o = o^SA - Sigma_KV rho with the d x d weighted covariance
                  built explicitly (ground truth)
* ``STREAM``   -- o = (1 + c) vbar - u, c = sum w (rho.k), u = sum w (rho.k) v
* ``NOINT``    -- the family's no-intercept member, o = -(sum w v k^T) rho with
                  the raw second moment built explicitly (linear attention
                  with probe -rho at uniform weights)

Every function here takes arrays of values (float32 or float64) and widens
them to float64 before calling the C code; nothing here does arithmetic of
the method.  Row lists are split over host threads (ctypes releases the GIL
during each C call).

Pinning: every form is checked, in ``tests/test_oracle_pins.py``, against
closed forms, a weighted least-squares fit solved by numpy, the uniform-weight
(linear-attention) limit, invariants and a high-precision brute force.
"""
from __future__ import annotations

import ctypes
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

SA, EXPLICIT, STREAM, NOINT = 0, 1, 2, 3
FORMS = {"sa": SA, "explicit": EXPLICIT, "stream": STREAM, "noint": NOINT}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libplx_oracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _form(form) -> int:
    return FORMS[form] if isinstance(form, str) else int(form)


def n_threads() -> int:
    return max(1, os.cpu_count() or 1)


class OracleLib:
    """ctypes view of one compiled copy of ``plx_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.plx_oracle_query.argtypes = [ctypes.c_int, _dp, _dp, _dp, _dp, ctypes.c_long,
                                         ctypes.c_int, ctypes.c_double, _dp, _dp]
        lib.plx_oracle_query.restype = ctypes.c_int
        lib.plx_oracle_prefill_rows.argtypes = [ctypes.c_int, _dp, _dp, _dp, _dp, ctypes.c_long,
                                                ctypes.c_int, ctypes.c_double, _lp, ctypes.c_long,
                                                _dp, _dp]
        lib.plx_oracle_prefill_rows.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def query(self, form, q, rho, K, V, scale: float):
        """One query q (probe rho) over keys K[n, d] and values V[n, d].

        Returns ``(out[d], lse)`` in float64."""
        q, K, V = _f64(q), _f64(K), _f64(V)
        d = q.shape[-1]
        rho = _f64(rho) if rho is not None else np.zeros(d)
        n = K.shape[0] if K.ndim == 2 else 0
        if n == 0:
            K = np.zeros((1, d))
            V = np.zeros((1, d))
        out = np.empty(d)
        lse = np.empty(1)
        rc = self.lib.plx_oracle_query(_form(form), _ptr(q), _ptr(rho), _ptr(K), _ptr(V), n, d,
                                       float(scale), _ptr(out), _ptr(lse))
        if rc:
            raise RuntimeError(f"oracle query failed: {rc}")
        return out, float(lse[0])

    def prefill_head(self, form, Q, K, V, RHO, scale: float, rows=None):
        """Causal prefill for one head: Q, K, V, RHO are [N, d]; row i
        attends to keys 0..i.  ``rows`` selects rows (default: all)."""
        Q, K, V, RHO = _f64(Q), _f64(K), _f64(V), _f64(RHO)
        N, d = Q.shape
        rows = (np.arange(N, dtype=np.int64) if rows is None
                else np.ascontiguousarray(rows, np.int64))
        out = np.empty((len(rows), d))
        lse = np.empty(len(rows))
        if len(rows):
            rc = self.lib.plx_oracle_prefill_rows(
                _form(form), _ptr(Q), _ptr(K), _ptr(V), _ptr(RHO), N, d, float(scale),
                rows.ctypes.data_as(_lp), len(rows), _ptr(out), _ptr(lse))
            if rc:
                raise RuntimeError(f"oracle prefill failed: {rc}")
        return out, lse


def default() -> OracleLib:
    """The oracle built from ``plx_oracle.c`` (rebuilt when the source is newer)."""
    global _default
    with _lock:
        if _default is None:
            src = os.path.join(_HERE, "plx_oracle.c")
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src)):
                from . import build
                build.build()
            _default = OracleLib(_LIB_PATH)
        return _default


def query(form, q, rho, K, V, scale: float):
    """One query against n keys with the default oracle; see ``OracleLib.query``."""
    return default().query(form, q, rho, K, V, scale)


def prefill_head(form, Q, K, V, RHO, scale: float, rows=None):
    """Causal prefill rows of one head with the default oracle."""
    return default().prefill_head(form, Q, K, V, RHO, scale, rows)


def prefill(form, q, k, v, rho, scale: float, heads=None, rows=None, threads=None):
    """Causal prefill over [B, H, N, d] inputs.

    ``heads``: list of (b, h) pairs (default: all).  ``rows``: row indices per
    head (default: all), either one array for every head or a dict keyed by
    (b, h).  Returns ``{(b, h): (out[len(rows), d], lse[len(rows)], rows)}``."""
    B, H, N, d = q.shape
    nt = threads or n_threads()
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    jobs = []
    for (b, h) in heads:
        r = rows.get((b, h)) if isinstance(rows, dict) else rows
        r = np.arange(N, dtype=np.int64) if r is None else np.asarray(r, np.int64)
        # split long row lists so that every host thread gets work
        nchunk = max(1, min(len(r), -(-4 * nt // max(1, len(heads)))))
        for chunk in np.array_split(r, nchunk):
            if len(chunk):
                jobs.append((b, h, chunk))
    head_cache = {(b, h): (_f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]), _f64(rho[b, h]))
                  for (b, h) in heads}
    lib = default()

    def run(job):
        b, h, chunk = job
        Q, K, V, R = head_cache[(b, h)]
        o, l = lib.prefill_head(form, Q, K, V, R, scale, chunk)
        return b, h, chunk, o, l

    results = {}
    with ThreadPoolExecutor(max_workers=nt) as ex:
        for b, h, chunk, o, l in ex.map(run, jobs):
            results.setdefault((b, h), []).append((chunk, o, l))
    out = {}
    for key, parts in results.items():
        rr = np.concatenate([p[0] for p in parts])
        oo = np.concatenate([p[1] for p in parts])
        ll = np.concatenate([p[2] for p in parts])
        order = np.argsort(rr, kind="stable")
        out[key] = (oo[order], ll[order], rr[order])
    return out


def decode(form, q, rho, k_cache, v_cache, seqlens, scale: float, heads=None, threads=None):
    """One-token decode: for each (b, h) the query q[b, h] (probe rho[b, h])
    attends to cache positions 0..seqlens[b]-1 (the cache already holds the
    current token at seqlens[b]-1).  Lengths above the cache capacity are
    clamped to it; lengths <= 0 give o = 0, lse = -inf.

    Returns ``{(b, h): (out[d], lse)}``."""
    B, H, S_cap, d = k_cache.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    lib = default()

    def run(bh):
        b, h = bh
        L = int(min(max(int(seqlens[b]), 0), S_cap))
        o, l = lib.query(form, q[b, h], rho[b, h] if rho is not None else None,
                         k_cache[b, h, :L], v_cache[b, h, :L], scale)
        return bh, o, l

    out = {}
    with ThreadPoolExecutor(max_workers=threads or n_threads()) as ex:
        for bh, o, l in ex.map(run, heads):
            out[bh] = (o, l)
    return out
