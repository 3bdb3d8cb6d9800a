"""fp64 CPU oracle for the multi-LoRA delta, the LRU slot table and the
adapter byte count.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it. The product library never imports, loads
or calls anything here, and nothing here imports the product.

* ``lora_apply_ref``  -- the per-token delta in double precision (C source
  ``lora_oracle.c``, compiled with gcc, OpenMP over tokens).
* ``LruSlotSim``      -- an independent simulator of the GPU slot table.
* ``adapter_bytes``   -- the capacity formula.
* ``belady``          -- an offline replay that evicts the adapter used
  farthest in the future: the yardstick for the eviction policies.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .lru_sim import LruSlotSim, NO_SLOT, RANK_ERR  # noqa: F401
from .adapter_bytes import adapter_bytes  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-std=c11", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)
            lib.oracle_lora_apply.argtypes = [i32, i64p, i32, i32, i32, i32, i32,
                                              vp, vp, vp, vp, vp, vp, vp, i32, vp]
            lib.oracle_lora_apply.restype = i32
            lib.oracle_threads.restype = i32
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_set_threads.restype = None
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    """OpenMP threads for the calls that follow (timing only)."""
    _load().oracle_set_threads(int(n))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def lora_apply_ref(x, y_in, A_pool, B_pool, rank, alpha, token_slot_idx,
                   tokens=None, dtype=BF16, loop_padded=False) -> np.ndarray:
    """Per-token LoRA delta in fp64 for one layer.

    x [T, d_in], y_in [T, d_out], A_pool [S, R, d_in], B_pool [S, d_out, R]
    (uint16 bf16 bits when dtype == BF16, float32 when dtype == F32);
    rank int32 [S]; alpha float64 [S]; token_slot_idx int32 [T].
    Returns float64 [len(tokens), d_out] (all tokens when ``tokens`` is None).
    """
    lib = _load()
    et = np.uint16 if dtype == BF16 else np.float32
    x = np.ascontiguousarray(x, dtype=et)
    y_in = np.ascontiguousarray(y_in, dtype=et)
    A_pool = np.ascontiguousarray(A_pool, dtype=et)
    B_pool = np.ascontiguousarray(B_pool, dtype=et)
    rank = np.ascontiguousarray(rank, dtype=np.int32)
    alpha = np.ascontiguousarray(alpha, dtype=np.float64)
    idx = np.ascontiguousarray(token_slot_idx, dtype=np.int32)
    T, d_in = x.shape
    S, R, d_in2 = A_pool.shape
    d_out = B_pool.shape[1]
    if d_in2 != d_in or B_pool.shape != (S, d_out, R) or y_in.shape != (T, d_out):
        raise ValueError("shape mismatch")
    if idx.shape != (T,) or rank.shape != (S,) or alpha.shape != (S,):
        raise ValueError("shape mismatch (idx/rank/alpha)")
    tok = (np.arange(T, dtype=np.int64) if tokens is None
           else np.ascontiguousarray(tokens, dtype=np.int64))
    if tok.size and (tok.min() < 0 or tok.max() >= T):
        raise ValueError("token index out of range")
    out = np.empty((tok.shape[0], d_out), dtype=np.float64)
    rc = lib.oracle_lora_apply(int(tok.shape[0]), tok.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                               d_in, d_out, S, R, int(dtype), _ptr(x), _ptr(y_in),
                               _ptr(A_pool), _ptr(B_pool), _ptr(rank), _ptr(alpha), _ptr(idx),
                               1 if loop_padded else 0, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_lora_apply failed")
    return out
