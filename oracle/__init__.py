"""Plain fp64 CPU oracle for neighborhood attention (NA) forward and backward.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's CPU
baseline may import this package; the library itself never does.  The arithmetic lives in
``na_oracle.c`` (double precision, OpenMP over rows); this module compiles it on first use and
marshals numpy arrays through ctypes.  It shares no code with the CUDA library.

Every function follows the definitions stated in the header of ``na_oracle.c``: the neighbourhood
of NATTEN issue #161 ("Backward pass is very slow towards much tokens and large kernels", the
user's na2d/na3d benchmark script), read as a per-axis residue-class window that shifts at the
borders, softmax(scale * q.k) over it, and the analytic backward with the Delta = <dO, O> prologue
that the maintainer's fused-kernel profile lists as ComputeDelta.

Parity pins: every exported function is checked in tests/test_oracle.py against dense masked
attention built from an independent characterisation of the window, full self-attention,
finite differences, and closed-form special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "na_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libna_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile na_oracle.c into a shared library (gcc, -O2, OpenMP, strict IEEE)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    global _lib
    with _lock:
        if True:
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            IP = ctypes.POINTER(ctypes.c_int)
            lib.na_oracle_fwd.argtypes = [P, P, P, I, I, I, IP, I, I, IP, IP, ctypes.c_double,
                                          P, I64, P, P, I]
            lib.na_oracle_fwd.restype = I
            lib.na_oracle_bwd.argtypes = [P, P, P, P, I, I, I, IP, I, I, IP, IP, ctypes.c_double,
                                          P, I64, P, P, I64, P, P, I]
            lib.na_oracle_bwd.restype = I
            lib.na_oracle_first_neighbour.argtypes = [I, I, I, I]
            lib.na_oracle_first_neighbour.restype = I
            lib.na_oracle_max_threads.argtypes = []
            lib.na_oracle_max_threads.restype = I
            _lib = lib
    return lib


def _load():
    with _lock:
        lib = _lib
    if lib is None:
        lib = _bind(ctypes.CDLL(build()))
    return lib


class library:
    """Context manager that points this module at another build of the oracle.

    Used by the mutation tests, which compile copies of na_oracle.c with a planted mistake and
    check that the pins reject them.
    """

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self.saved = _lib
            _lib = None
        _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def max_threads() -> int:
    return int(_load().na_oracle_max_threads())


def _ints(vals):
    arr = (ctypes.c_int * len(vals))(*[int(x) for x in vals])
    return arr


def _prep(x):
    """Accept float32, bfloat16 bit patterns (uint16) or float64; returns (array, kind code)."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, 0
    if x.dtype == np.uint16:
        return x, 1
    if x.dtype == np.float64:
        return x, 2
    raise TypeError(f"unsupported input dtype {x.dtype}")


def _rows(rows):
    if rows is None:
        return None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    return r


def first_neighbour(i: int, L: int, k: int, d: int) -> int:
    """Spatial index of the first neighbour of index i along one axis (-1 on invalid input)."""
    return int(_load().na_oracle_first_neighbour(int(i), int(L), int(k), int(d)))


def _shape(q):
    B = q.shape[0]
    spatial = tuple(int(s) for s in q.shape[1:-2])
    heads, D = int(q.shape[-2]), int(q.shape[-1])
    return B, spatial, heads, D


def na_fwd(q, k, v, kernel, dilation, scale, rows=None, nthreads=None):
    """Oracle forward.  q, k, v: [B, L1..Ln, heads, D] float32, float64 or bf16 bits (uint16).

    Returns (O, LSE) in float64: with rows=None, O is [B, L.., heads, D] and LSE [B, L.., heads];
    with rows (flat indices ((b*N + token)*heads + head)), O is [len(rows), D] and LSE [len(rows)].
    """
    q, bq = _prep(q)
    k, bk = _prep(k)
    v, bv = _prep(v)
    if not (bq == bk == bv) or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share shape and dtype")
    B, spatial, heads, D = _shape(q)
    ndim = len(spatial)
    total = B * int(np.prod(spatial)) * heads
    r = _rows(rows)
    n = total if r is None else int(r.size)
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    nt = nthreads or max_threads()
    rc = _load().na_oracle_fwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, bq, B, ndim, _ints(spatial), heads, D,
        _ints(kernel), _ints(dilation), float(scale),
        None if r is None else r.ctypes.data, n, o.ctypes.data, lse.ctypes.data, int(nt))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    if r is None:
        return o.reshape(q.shape), lse.reshape(q.shape[:-1])
    return o, lse


def na_bwd(q, k, v, dO, kernel, dilation, scale, qrows=None, krows=None, nthreads=None,
           want_dq=True, want_dkdv=True):
    """Oracle backward.  Returns (dQ, dK, dV) in float64.

    With qrows/krows None the full tensors are returned ([B, L.., heads, D]); otherwise dQ has
    one row per entry of qrows and dK/dV one per entry of krows.  The oracle recomputes O and
    LSE itself from q, k, v.
    """
    q, bq = _prep(q)
    k, bk = _prep(k)
    v, bv = _prep(v)
    dO, bd = _prep(dO)
    if not (bq == bk == bv == bd) or not (q.shape == k.shape == v.shape == dO.shape):
        raise ValueError("q, k, v, dO must share shape and dtype")
    B, spatial, heads, D = _shape(q)
    ndim = len(spatial)
    total = B * int(np.prod(spatial)) * heads
    qr = _rows(qrows)
    kr = _rows(krows)
    nq = 0 if not want_dq else (total if qr is None else int(qr.size))
    nk = 0 if not want_dkdv else (total if kr is None else int(kr.size))
    dq = np.zeros((max(nq, 1), D), dtype=np.float64)
    dk = np.zeros((max(nk, 1), D), dtype=np.float64)
    dv = np.zeros((max(nk, 1), D), dtype=np.float64)
    nt = nthreads or max_threads()
    rc = _load().na_oracle_bwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dO.ctypes.data, bq, B, ndim, _ints(spatial),
        heads, D, _ints(kernel), _ints(dilation), float(scale),
        None if (qr is None or not want_dq) else qr.ctypes.data, nq, dq.ctypes.data,
        None if (kr is None or not want_dkdv) else kr.ctypes.data, nk, dk.ctypes.data, dv.ctypes.data,
        int(nt))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    dq, dk, dv = dq[:nq], dk[:nk], dv[:nk]
    if qr is None and want_dq:
        dq = dq.reshape(q.shape)
    if kr is None and want_dkdv:
        dk = dk.reshape(q.shape)
        dv = dv.reshape(q.shape)
    return dq, dk, dv
