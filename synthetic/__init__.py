"""Seeded synthetic inputs for the Ulysses attention block.

Shared by the CPU oracle's tests, the GPU parity tests and the benchmark.  This module
holds none of the block's arithmetic: only the counter-based normal generator (defined
in ``gen.c``), bf16 storage helpers and the choice of sampled rows.

Recipe (the same for every consumer):
  * X ~ N(0, 1)            seed 0, tensor id 0, shape [S][hidden]
  * W_qkv ~ N(0, 0.02^2)   seed 0, tensor id 1, shape [(H + 2G) * D][hidden]
  * dO ~ N(0, 1)           seed 1, tensor id 0, shape of O
  * Q, K, V drawn directly in head layout (attention-stage tests): seed 0, ids 2, 3, 4
  * a raw [S][H + 2G][D] activation for permute tests: seed 0, id 5
Values are rounded to float32 and then to bf16 (round to nearest even) and kept as
uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None

TENSOR_X, TENSOR_W, TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_QKV = 0, 1, 2, 3, 4, 5
TENSOR_WO = 6          # output projection weight (seed 0); with seed 1, the gradient dy
SEED_FWD, SEED_DO, SEED_SAMPLE = 0, 1, 2


def build() -> str:
    """Compile gen.c into libsynth.so beside it (plain C, any host architecture)."""
    src = os.path.join(_HERE, "gen.c")
    if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal.restype = ctypes.c_int
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def normal_bf16(seed: int, tensor_id: int, shape, std: float = 1.0, mean: float = 0.0,
                offset: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, std^2) draws [offset, offset + prod(shape))."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    n = out.size
    if n:
        _load().synth_normal(seed, tensor_id, offset, n, mean, std,
                             out.ctypes.data, None, _threads())
    return out


def normal_f64(seed: int, tensor_id: int, shape, std: float = 1.0, mean: float = 0.0,
               offset: int = 0) -> np.ndarray:
    """The same draws before any rounding, as float64."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.float64)
    if out.size:
        _load().synth_normal(seed, tensor_id, offset, out.size, mean, std,
                             None, out.ctypes.data, _threads())
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def sample_rows(S: int, P: int, n: int, seed: int = SEED_SAMPLE, stream: int = 0) -> np.ndarray:
    """Sorted query rows: n drawn uniformly without replacement, plus the shard edges.

    The edges 0, 1, S/P - 1, S/P and S - 1 are always included."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    n = min(n, S)
    picked = rng.choice(S, size=n, replace=False) if n else np.zeros(0, np.int64)
    edges = [0, 1, S // P - 1, S // P, S - 1] if S else []
    rows = np.unique(np.concatenate([picked.astype(np.int64),
                                     np.array([e for e in edges if 0 <= e < S], np.int64)]))
    return rows


def to_torch_bf16(bits: np.ndarray):
    """Wrap bf16 bit patterns as a CPU torch.bfloat16 tensor (no copy)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def torch_bf16_to_bits(t) -> np.ndarray:
    """bf16 torch tensor (any device) -> uint16 bit patterns on the host."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
