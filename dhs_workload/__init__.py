"""Seeded synthetic inputs for the hierarchical sparse KV resolve + gather path.

This package holds none of the method's arithmetic: it only draws the inputs
that both the CUDA library and the CPU oracle consume (row payloads, top-k
selections, resident page sets, append counts).  The arithmetic lives in
``gen.c`` (splitmix64, Box-Muller, Zipf inverse CDF, Fisher-Yates); this
module compiles it with gcc and wraps it with ctypes.

The pages ("Adaptive DHiSparse", Evidence section) measure on real
GLM-5.3 / DeepSeek-V4.1-Flash decode traffic that is not available; the
configurations in :mod:`dhs_workload.configs` stand in for it with the
shapes the pages name (32K-500K histories, concurrency 8-128, verify blocks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libdhsw.so")
_lib = None
_lock = threading.Lock()

SEED = 0


def build(force: bool = False) -> str:
    """Compile gen.c into libdhsw.so next to it (gcc, no CUDA)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared",
                           "-fno-math-errno", "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            u64, u32, i64, i32 = (ctypes.c_uint64, ctypes.c_uint32,
                                  ctypes.c_int64, ctypes.c_int32)
            vp, dbl = ctypes.c_void_p, ctypes.c_double
            L.dhsw_key.restype = u64
            L.dhsw_key.argtypes = [u64, u64, u64, u64, u64]
            L.dhsw_f32_to_bf16.restype = ctypes.c_uint16
            L.dhsw_f32_to_bf16.argtypes = [ctypes.c_float]
            L.dhsw_payload_row.restype = None
            L.dhsw_payload_row.argtypes = [u64, u32, u32, u32, i64, i32, vp]
            L.dhsw_payload_pairs.restype = ctypes.c_int
            L.dhsw_payload_pairs.argtypes = [u64, u32, i32, vp, vp, i64, i64,
                                             i32, vp, i64, i32]
            L.dhsw_zipf_cdf.restype = ctypes.c_int
            L.dhsw_zipf_cdf.argtypes = [i64, dbl, vp]
            L.dhsw_permutation.restype = ctypes.c_int
            L.dhsw_permutation.argtypes = [u64, u32, u32, u32, i64, vp]
            L.dhsw_select.restype = ctypes.c_int
            L.dhsw_select.argtypes = [u64, u32, u32, u32, u64, u64, i64, i64,
                                      i32, i64, dbl, vp, vp, vp, i32, dbl, vp,
                                      i32, vp, vp, vp]
            L.dhsw_residency.restype = ctypes.c_int
            L.dhsw_residency.argtypes = [u64, u32, u32, u32, i64, i64, vp]
            L.dhsw_append_counts.restype = ctypes.c_int
            L.dhsw_append_counts.argtypes = [u64, u32, u32, i32, i32, i32, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """bf16 bits (round-to-nearest-even) of float32 values, via gen.c."""
    L = lib()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([L.dhsw_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def payload_row(cfg: int, src: int, req: int, row: int, elems: int,
                seed: int = SEED) -> np.ndarray:
    out = np.empty(elems, dtype=np.uint16)
    lib().dhsw_payload_row(seed, cfg, src, req, row, elems, _ptr(out))
    return out


def payload_pairs_into(out_ptr: int, pair_stride_rows: int, cfg: int,
                       pairs, row0: int, nrows: int, elems: int,
                       seed: int = SEED, nthreads: int | None = None) -> None:
    """Write rows [row0, row0+nrows) of each (src, req) pair to raw memory.

    Pair p's row r lands at ``out_ptr + ((p*pair_stride_rows) + r - row0)
    * elems * 2`` bytes.  ``out_ptr`` may be any host address (numpy array or
    a pinned buffer).
    """
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    srcs = np.ascontiguousarray([p[0] for p in pairs], dtype=np.uint32)
    reqs = np.ascontiguousarray([p[1] for p in pairs], dtype=np.uint32)
    rc = lib().dhsw_payload_pairs(seed, cfg, len(pairs), _ptr(srcs), _ptr(reqs),
                                  row0, nrows, elems, out_ptr,
                                  pair_stride_rows, nthreads)
    if rc != 0:
        raise ValueError(f"dhsw_payload_pairs failed ({rc})")


def payload_rows(cfg: int, src: int, req: int, row0: int, nrows: int,
                 elems: int, seed: int = SEED) -> np.ndarray:
    out = np.empty((nrows, elems), dtype=np.uint16)
    payload_pairs_into(_ptr(out), nrows, cfg, [(src, req)], row0, nrows,
                       elems, seed)
    return out


def zipf_cdf(n: int, s: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if lib().dhsw_zipf_cdf(n, s, _ptr(out)) != 0:
        raise ValueError("zipf_cdf")
    return out


def permutation(cfg: int, src: int, req: int, n: int,
                seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if lib().dhsw_permutation(seed, cfg, src, req, n, _ptr(out)) != 0:
        raise ValueError("permutation")
    return out


def select(cfg: int, src: int, req: int, stream_a: int, stream_b: int,
           L: int, N: int, k: int, window: int, frac_recent: float,
           cdf: np.ndarray, perm: np.ndarray, prev_z: np.ndarray | None,
           rho: float, exclude: np.ndarray | None = None,
           seed: int = SEED):
    """One sorted top-k selection; returns (rows, zipf_rows)."""
    out = np.empty(max(k, 1), dtype=np.int32)
    out_z = np.empty(max(k, 1), dtype=np.int32)
    nz = ctypes.c_int32(0)
    if prev_z is None:
        prev_z = np.empty(0, dtype=np.int32)
    if exclude is None:
        exclude = np.empty(0, dtype=np.int32)
    prev_z = np.ascontiguousarray(prev_z, dtype=np.int32)
    exclude = np.ascontiguousarray(exclude, dtype=np.int32)
    rc = lib().dhsw_select(seed, cfg, src, req, stream_a, stream_b, L, N, k,
                           window, frac_recent, _ptr(cdf), _ptr(perm),
                           _ptr(prev_z), len(prev_z), rho, _ptr(exclude),
                           len(exclude), _ptr(out), _ptr(out_z),
                           ctypes.byref(nz))
    if rc != 0:
        raise ValueError(f"dhsw_select failed ({rc}) L={L} N={N} k={k}")
    return out[:k].copy(), out_z[: nz.value].copy()


def residency(cfg: int, src: int, req: int, pages: int, count: int,
              seed: int = SEED) -> np.ndarray:
    out = np.empty(max(pages, 1), dtype=np.uint8)
    if lib().dhsw_residency(seed, cfg, src, req, pages, count, _ptr(out)) != 0:
        raise ValueError("residency")
    return out[:pages].copy()


def append_counts(cfg: int, req: int, steps: int, lo: int, hi: int,
                  seed: int = SEED) -> np.ndarray:
    out = np.empty(max(steps, 1), dtype=np.int32)
    if lib().dhsw_append_counts(seed, cfg, req, steps, lo, hi, _ptr(out)) != 0:
        raise ValueError("append_counts")
    return out[:steps].copy()
