"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This module holds none of the method's arithmetic: it draws the random
numbers that stand in for checkpoint weights, latent tokens and conditioning
vectors, and names the five benchmark workloads. Both sides of every parity
check take their inputs from here, bit for bit.

Recipe (see ``gen.c`` for the generator's definition):
  * every weight ~ N(0, 0.02), drawn in fp32 and rounded to bf16 (RNE);
    stream id = (block << 8) | param_index, params in the block's fixed order;
  * latent tokens x ~ N(0, 1) fp32, shape [R, T, hidden], stream id TOKENS_ID;
  * conditioning c ~ N(0, 1) fp32, shape [R, cond_dim], stream id COND_ID.

The C generator is compiled on first use with the host C compiler (OpenMP
when available) into ``synthetic/_build``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import CONFIGS, WorkloadConfig, get_config  # noqa: F401

TOKENS_ID = 0xF0000001
COND_ID = 0xF0000002
WEIGHT_STD = 0.02

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library; returns its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64 = ctypes.c_uint64, ctypes.c_int64
            lib.syn_raw_u64.argtypes = [u64, u64, i64, ctypes.c_void_p]
            lib.syn_normal_f32.argtypes = [u64, u64, i64, ctypes.c_double, ctypes.c_void_p]
            lib.syn_normal_bf16.argtypes = [u64, u64, i64, ctypes.c_double, ctypes.c_void_p]
            lib.syn_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def raw_u64(seed: int, tensor_id: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().syn_raw_u64(seed, tensor_id, n, out.ctypes.data)
    return out


def normal_f32(seed: int, tensor_id: int, shape, std: float = 1.0, out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().syn_normal_f32(seed, tensor_id, n, std, out.ctypes.data)
    return out


def normal_bf16_bits(seed: int, tensor_id: int, shape, std: float, out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().syn_normal_bf16(seed, tensor_id, n, std, out.ctypes.data)
    return out


def weight_bits(seed: int, block: int, param: int, shape, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits of one parameter of one block, ~N(0, 0.02)."""
    return normal_bf16_bits(seed, (block << 8) | param, shape, WEIGHT_STD, out)


def tokens(seed: int, R: int, T: int, hidden: int) -> np.ndarray:
    return normal_f32(seed, TOKENS_ID, (R, T, hidden), 1.0)


def cond(seed: int, R: int, cond_dim: int) -> np.ndarray:
    return normal_f32(seed, COND_ID, (R, cond_dim), 1.0)


def threads() -> int:
    return int(_load().syn_max_threads())
