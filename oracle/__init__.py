"""Oracle for paged-KV grouped-query attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import, call, link or execute anything in this package.
The product library (``paged_kv_gqa_nx_gb300``) never imports it, and it
never imports the product library: the two share no code.

Contents
--------
``attend``            dense offset-causal GQA attention over a contiguous
                      K/V history (C core in ``attention.c``, double
                      accumulation, rounded once to f32; ``set_threads``
                      spreads its (query, head) pairs over host cores).
``ContiguousCache``   the contiguous per-layer K/V history a sequence would
                      have, with append / advance / truncate / fork
                      (``contiguous_cache.py``).
``PoolModel``         the pool / page-table / refcount metadata model
                      (``pool_model.py``).
``rope_neox``         rotary position embedding, NeoX pairing, float64
                      (``rope.py``).
``round_bf16``        the bf16 pool's rounding of stored rows (nearest,
                      ties to even; ``kv_format.py``).
``round_e4m3``        the fp8 pool's stored-and-read value (e4m3 of x/scale,
                      nearest, ties to even, saturating; ``kv_format.py``).

Every function cites the passage of the pages it follows; the pages are the
source listings "nx_f32_attn_paged.nx source", "nx_f32_gqa_attention.nx
source", "nx_f32_llama_v4b.nx source" and "nx_paged_kv_gate.nx source".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_BAD_DIM = 1
ERR_BAD_GQA = 2


def build(force: bool = False) -> str:
    """Compile ``attention.c`` into ``liboracle.so`` with gcc when it is
    missing or stale: -O3, OpenMP over (query, head) pairs, no fast-math, no
    contraction into fused multiply-adds, no host-specific flags.  Without
    OpenMP support the same source builds single-threaded."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    base = ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC]
    try:
        subprocess.check_call(base + ["-fopenmp", "-lm"], stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.check_call(base + ["-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            fp = ctypes.POINTER(ctypes.c_float)
            lib.oracle_attend.argtypes = [fp, fp, fp, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_float, fp]
            lib.oracle_attend.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = ctypes.c_int
            lib.oracle_set_threads(0)
            _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Threads for ``attend`` from now on (n < 1: every core the host offers;
    the default).  Returns the count in effect (1 when the C core was built
    without OpenMP).  The result does not depend on it."""
    return int(_load().oracle_set_threads(int(n)))


def _padded(a: np.ndarray, n: int) -> np.ndarray:
    if a.size >= n:
        return a
    return np.concatenate([a, np.zeros(n - a.size, dtype=np.float32)])


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def attend(Q, K, V, n_q: int, total_k: int, n_heads: int, n_kv_heads: int,
           head_dim: int, causal: int, scale: float):
    """Offset-causal GQA attention over a contiguous history.

    Follows "nx_f32_attn_paged.nx source" (header comment: same math as the
    contiguous path, q_pos = total_k - n_q + i; step 3: q head h reads kv head
    h / group) and "nx_f32_gqa_attention.nx source" (GQA wrapper, layouts).

    Q: [n_q, n_heads*head_dim]; K, V: [>= total_k, n_kv_heads*head_dim] (only
    the first total_k rows are read).  Returns ``(rc, out)``; ``out`` is
    [n_q, n_heads*head_dim] float32, or None when rc != 0.
    """
    kv_dim = n_kv_heads * head_dim if n_kv_heads > 0 and head_dim > 0 else 0
    q_dim = n_heads * head_dim if n_heads > 0 and head_dim > 0 else 0
    Qa = np.ascontiguousarray(np.asarray(Q, dtype=np.float32).reshape(-1))
    Ka = np.ascontiguousarray(np.asarray(K, dtype=np.float32).reshape(-1))
    Va = np.ascontiguousarray(np.asarray(V, dtype=np.float32).reshape(-1))
    # The C core validates sizes and grouping before it reads anything; arrays
    # shorter than the stated sizes (as in a rejected call) are zero-padded so
    # the core never reads past them.
    Qa = _padded(Qa, max(n_q, 0) * q_dim)
    Ka = _padded(Ka, max(total_k, 0) * kv_dim)
    Va = _padded(Va, max(total_k, 0) * kv_dim)
    out = np.zeros(max(n_q, 0) * max(q_dim, 0) or 1, dtype=np.float32)
    rc = _load().oracle_attend(_fptr(Qa), _fptr(Ka), _fptr(Va), int(n_q), int(total_k),
                               int(n_heads), int(n_kv_heads), int(head_dim), int(causal),
                               float(np.float32(scale)), _fptr(out))
    if rc != OK:
        return rc, None
    return rc, out[: n_q * q_dim].reshape(n_q, q_dim)


from .contiguous_cache import ContiguousCache  # noqa: E402
from .pool_model import PoolModel, SeqModel  # noqa: E402
from . import pool_model  # noqa: E402
from .rope import rope_neox, rope_neox_f32  # noqa: E402
from .kv_format import round_bf16, round_e4m3  # noqa: E402

__all__ = ["attend", "build", "set_threads", "ContiguousCache", "PoolModel", "SeqModel", "pool_model",
           "OK", "ERR_BAD_DIM", "ERR_BAD_GQA"]
