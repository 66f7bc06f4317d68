"""Seeded synthetic inputs, shared by the tests, the bench and the smoke check.

This module holds none of the method's arithmetic: it only turns
(seed, stream, element index) into numbers.  The same generator is
implemented for the device in ``synth_dev.cu`` (libsynth.so) so that a
full-size input can be made in HBM while the oracle regenerates exactly the
slice it needs on the host.

Definition (counter based, every element independent):
  * splitmix64(x): x += 0x9E3779B97F4A7C15;
                   x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9;
                   x = (x ^ (x >> 27)) * 0x94D049BB133111EB;
                   return x ^ (x >> 31)        (all mod 2^64)
  * stream key:    key = splitmix64(splitmix64(seed) ^ stream)
  * element i:     a = splitmix64(key + 2 i), b = splitmix64(key + 2 i + 1)
                   u1 = ((a >> 11) + 1) * 2^-53      in (0, 1]
                   u2 =  (b >> 11)      * 2^-53      in [0, 1)
  * normal:        z = sqrt(-2 ln u1) * cos(2pi * u2)     (Box-Muller, fp64)
                   value = mean + std * z, rounded ONCE to the target type
  * sign:          +1 if (a >> 63) == 0 else -1           (exact)
  * dyadic:        0 with probability 1/4, else sign * 2^-(4 + (a >> 40) % 5)

Rounding fp64 -> bf16 is round-to-nearest-even done as: fp64 -> fp32 with
round-to-odd (truncate toward zero, set the last bit if inexact), then fp32 ->
bf16 nearest-even on the bit pattern; the 16 extra bits make the two steps
round exactly once.

Stream ids name the tensor: ``stream_id(config, layer, tensor, step)``.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
_GOLD = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
TWO_PI = 6.283185307179586  # 2*pi rounded to fp64 (0x401921FB54442D18)
DEFAULT_SEED = 20240509

# tensor tags used in stream ids
T_Q, T_K, T_V, T_LOGIT, T_M, T_WK, T_WV, T_CACHE_K, T_CACHE_V, T_QX, T_S0, T_RMSW = range(1, 13)


def stream_id(config: int, layer: int, tensor: int, step: int = 0) -> int:
    """Pack (config, layer, tensor, step) into one 64-bit stream tag."""
    return ((config & 0xFF) << 56) | ((layer & 0xFFFF) << 40) | ((tensor & 0xFF) << 32) | (step & 0xFFFFFFFF)


def splitmix64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GOLD
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    k0 = splitmix64(np.uint64(seed & MASK64))
    return splitmix64(np.uint64(k0) ^ np.uint64(stream & MASK64))


def _counters(seed, stream, start, count):
    key = stream_key(seed, stream)
    i = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        a = splitmix64(key + np.uint64(2) * i)
        b = splitmix64(key + np.uint64(2) * i + np.uint64(1))
    return a, b


def normal_at(seed: int, stream: int, idx, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """fp64 normals of the stream at arbitrary element indices (any shape)."""
    idx = np.asarray(idx, dtype=np.uint64)
    key = stream_key(seed, stream)
    with np.errstate(over="ignore"):
        a = splitmix64(key + np.uint64(2) * idx)
        b = splitmix64(key + np.uint64(2) * idx + np.uint64(1))
    u1 = ((a >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
    u2 = (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return mean + std * (np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2))


def normal_f64(seed: int, stream: int, count: int, mean: float = 0.0, std: float = 1.0,
               start: int = 0) -> np.ndarray:
    """Elements start..start+count-1 of the stream as fp64 normals (before rounding)."""
    a, b = _counters(seed, stream, start, count)
    u1 = ((a >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
    u2 = (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)
    return mean + std * z


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, nearest-even, via fp32 round-to-odd."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)                       # nearest-even
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    f = np.where(over, np.nextafter(f, np.float32(0)), f)  # -> truncation toward zero
    inexact = f.astype(np.float64) != x
    bits = f.view(np.uint32).copy()
    bits |= inexact.astype(np.uint32)             # round to odd
    bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        out = ((bits + bias) >> np.uint32(16)).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(seed: int, stream: int, shape, dtype: str, mean: float = 0.0, std: float = 1.0,
           start: int = 0) -> np.ndarray:
    """Seeded normals of `shape`, rounded once.  dtype 'bf16' returns uint16 bit
    patterns, 'f32' returns float32 values."""
    n = int(np.prod(shape))
    x = normal_f64(seed, stream, n, mean, std, start)
    if dtype == "bf16":
        return f64_to_bf16_bits(x).reshape(shape)
    if dtype == "f32":
        return x.astype(np.float32).reshape(shape)
    raise ValueError(dtype)


def signs(seed: int, stream: int, shape, start: int = 0) -> np.ndarray:
    """Exact +-1 values (float32)."""
    n = int(np.prod(shape))
    a, _ = _counters(seed, stream, start, n)
    return np.where((a >> np.uint64(63)) == 0, 1.0, -1.0).astype(np.float32).reshape(shape)


def dyadic(seed: int, stream: int, shape, start: int = 0) -> np.ndarray:
    """Exact values in {0, +-2^-4 .. +-2^-8} (float32); about a quarter are 0."""
    n = int(np.prod(shape))
    a, _ = _counters(seed, stream, start, n)
    sgn = np.where((a >> np.uint64(63)) == 0, 1.0, -1.0)
    e = 4 + ((a >> np.uint64(40)) % np.uint64(5)).astype(np.int64)
    zero = ((a >> np.uint64(20)) & np.uint64(3)) == 0
    v = np.where(zero, 0.0, sgn * np.ldexp(1.0, -e))
    return v.astype(np.float32).reshape(shape)


# ----------------------------------------------------------- device copy

_dev_lib = None


def _device_lib():
    global _dev_lib
    if _dev_lib is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libsynth.so")
        if not os.path.exists(path):
            raise ImportError(f"{path} missing; run synth/build.py (nvcc)")
        L = ctypes.CDLL(path)
        for name in ("synth_normal_bf16", "synth_normal_f32"):
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                           ctypes.c_double, ctypes.c_int64, ctypes.c_void_p]
        _dev_lib = L
    return _dev_lib


def fill_normal_(t, seed: int, stream: int, mean: float = 0.0, std: float = 1.0, start: int = 0):
    """Fill a contiguous CUDA tensor (bfloat16 or float32) in place with elements
    start..start+numel-1 of the stream -- the same values normal() returns."""
    import ctypes
    import torch
    assert t.is_cuda and t.is_contiguous()
    L = _device_lib()
    fn = L.synth_normal_bf16 if t.dtype == torch.bfloat16 else L.synth_normal_f32
    if t.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(t.dtype)
    st = torch.cuda.current_stream().cuda_stream
    rc = fn(ctypes.c_void_p(t.data_ptr()), t.numel(), seed & MASK64, stream & MASK64, float(mean), float(std),
            int(start), ctypes.c_void_p(st))
    if rc != 0:
        raise RuntimeError(f"synth device generator failed with CUDA error {rc}")
    return t
