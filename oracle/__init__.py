"""CPU oracle for the YOCO token-mixing path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline arm of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation); this module
only marshals numpy arrays to it.  Every function widens its inputs to fp64
exactly (bf16 bit patterns and fp32 values are representable in fp64), so the
oracle sees the same numbers the GPU path consumes.

Citations (paper: "You Only Cache Once: Decoder-Decoder Architectures for
Language Models", arXiv:2405.05254v2):
  * gret_recurrent  -- Section 3.1, Eq. 5; Appendix F RecurrentRetention
  * gret_parallel   -- Section 3.1, Eq. 4
  * gret_chunkwise  -- Eq. 6 with consistent indices (close-reading notes
                       Section 2.3; slides backup "chunkwise recurrence with
                       consistent indices"); Appendix F ChunkwiseRetention
  * rmsnorm_proj    -- Section 2.2, Eq. 2 (LN = RMSNorm)
  * kv_append_bf16  -- Section 2.2 (one cache, written once, shared by layers)
  * cross_attn      -- Section 2.2, Eq. 3 (causal, grouped-query softmax)
  * swa_attn        -- Section 3.2, Eq. 8 (sliding-window attention, window
                       mask n - C < m <= n)
  * group_norm_gate -- Section 3.1, Eq. 7 (GroupNorm per head, swish gate)
  * rope            -- Section 3.1 (Q (.) Theta, K (.) conj(Theta)); the notes'
                       cross-decoder walk-through (K^ rotated in the shared
                       projection, each layer's Q rotated)
  * qkvg_project    -- Section 3.1 (Q = X W_Q (.) Theta, K = X W_K (.) conj(Theta),
                       V = X W_V, gamma from X W_gamma): one product with the
                       four weight matrices side by side

Parity status: every function here is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def lib():
    """Load the compiled oracle, building it first if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            from . import build as _b
            _b.build()
        L = ctypes.CDLL(_LIB_PATH)
        i, d, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
        L.oracle_set_threads.argtypes = [i]
        L.oracle_set_threads.restype = None
        L.oracle_gate.argtypes = [d, d]
        L.oracle_gate.restype = d
        L.oracle_gret_recurrent.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, d, _dp, _dp, _dp]
        L.oracle_gret_parallel.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, d, _dp]
        L.oracle_gret_chunkwise.argtypes = [i, i, i, i, i, i, _dp, _dp, _dp, _dp, d, _dp, _dp, _dp]
        L.oracle_rmsnorm_proj.argtypes = [i, i, i, _dp, _dp, d, _dp, _dp]
        L.oracle_round_bf16.argtypes = [d]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        L.oracle_kv_append_bf16.argtypes = [i, i, i, i, i64, i64, _dp, _u16p]
        L.oracle_cross_attn.argtypes = [i, i, i, i, i, i64, _dp, _dp, _dp, i64, d, _dp]
        L.oracle_swa_attn.argtypes = [i, i, i, i, i, i64, _dp, _dp, _dp, d, _dp]
        L.oracle_group_norm_gate.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, d, _dp]
        L.oracle_rope.argtypes = [i64, i, ctypes.POINTER(ctypes.c_int64), d, _dp]
        for name in ("oracle_gret_recurrent", "oracle_gret_parallel", "oracle_gret_chunkwise",
                     "oracle_rmsnorm_proj", "oracle_kv_append_bf16", "oracle_cross_attn"):
            getattr(L, name).restype = None
        _lib = L
    return _lib



def set_threads(n):
    """Threads the oracle's OpenMP loops use from now on (n > 0)."""
    lib().oracle_set_threads(int(n))

def _f64(a) -> np.ndarray:
    """Widen to a contiguous fp64 array (exact for bf16 bits given as float32 and fp32)."""
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gate(logit: float, tau: float) -> float:
    """gamma = sigmoid(logit)^(1/tau), through logsigmoid (Section 3.1 Eq. 4; Appendix F)."""
    return lib().oracle_gate(float(logit), float(tau))


def gret_recurrent(q, k, v, logits, tau, S0=None):
    """Recurrent gRet (Eq. 5).  q,k [B,N,H,dk], v [B,N,H,dv], logits [B,N,H].
    Returns (o [B,N,H,dv], S_final [B,H,dk,dv]) in fp64."""
    q, k, v, lg = _f64(q), _f64(k), _f64(v), _f64(logits)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    S0 = None if S0 is None else _f64(S0)
    o = np.zeros((B, N, H, dv))
    S = np.zeros((B, H, dk, dv))
    lib().oracle_gret_recurrent(B, N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(lg), float(tau),
                                _ptr(S0), _ptr(o), _ptr(S))
    return o, S


def gret_parallel(q, k, v, logits, tau):
    """Parallel gRet (Eq. 4), zero initial state.  O(N^2): small N only."""
    q, k, v, lg = _f64(q), _f64(k), _f64(v), _f64(logits)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, N, H, dv))
    lib().oracle_gret_parallel(B, N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(lg), float(tau), _ptr(o))
    return o


def gret_chunkwise(q, k, v, logits, tau, chunk, S0=None):
    """Chunkwise gRet (corrected Eq. 6).  Returns (o, S_final) in fp64."""
    q, k, v, lg = _f64(q), _f64(k), _f64(v), _f64(logits)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    S0 = None if S0 is None else _f64(S0)
    o = np.zeros((B, N, H, dv))
    S = np.zeros((B, H, dk, dv))
    lib().oracle_gret_chunkwise(B, N, H, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v), _ptr(lg),
                                float(tau), _ptr(S0), _ptr(o), _ptr(S))
    return o, S


def rmsnorm_proj(M, W, eps, g=None):
    """RMSNorm(M) @ W (Eq. 2).  M [..., dm], W [dm, n] -> fp64 [..., n]."""
    M, W = _f64(M), _f64(W)
    lead = M.shape[:-1]
    dm = M.shape[-1]
    n = W.shape[1]
    R = int(np.prod(lead)) if lead else 1
    g = None if g is None else _f64(g)
    out = np.zeros((R, n))
    lib().oracle_rmsnorm_proj(R, dm, n, _ptr(M.reshape(R, dm)), _ptr(g), float(eps), _ptr(W), _ptr(out))
    return out.reshape(*lead, n)


def round_bf16(x) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest, ties to even (elementwise)."""
    x = _f64(x)
    f = lib().oracle_round_bf16
    return np.array([f(float(t)) for t in x.ravel()], dtype=np.uint16).reshape(x.shape)


def kv_append_bf16(cache_bits, kv_new, length):
    """Expected cache after appending kv_new [B,T,Hkv*d] at slot `length`.
    cache_bits [B,Hkv,cap,d] uint16 (bf16 bits) is copied, not modified."""
    c = np.ascontiguousarray(np.array(cache_bits, dtype=np.uint16, copy=True))
    B, Hkv, cap, d = c.shape
    kv = _f64(kv_new)
    T = kv.shape[1]
    lib().oracle_kv_append_bf16(B, T, Hkv, d, cap, int(length), _ptr(kv), c.ctypes.data_as(_u16p))
    return c


def cross_attn(Q, Kc, Vc, p0, scale):
    """Causal GQA softmax attention (Eq. 3).  Q [B,T,Hq,d]; Kc, Vc [B,Hkv,cap,d].
    Row t sits at position p0 + t and reads slots 0..p0+t.  Returns fp64 O."""
    Q, Kc, Vc = _f64(Q), _f64(Kc), _f64(Vc)
    B, T, Hq, d = Q.shape
    Hkv, cap = Kc.shape[1], Kc.shape[2]
    O = np.zeros((B, T, Hq, d))
    lib().oracle_cross_attn(B, T, Hq, Hkv, d, cap, _ptr(Q), _ptr(Kc), _ptr(Vc), int(p0), float(scale), _ptr(O))
    return O


def swa_attn(Q, K, V, window, scale):
    """Sliding-window attention (Section 3.2, Eq. 8): the query at position n sees
    keys n - window < m <= n.  Q [B,N,Hq,d]; K, V [B,N,Hkv,d].  Returns fp64 O."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, N, Hq, d = Q.shape
    Hkv = K.shape[2]
    O = np.zeros((B, N, Hq, d))
    lib().oracle_swa_attn(B, N, Hq, Hkv, d, int(window), _ptr(Q), _ptr(K), _ptr(V), float(scale), _ptr(O))
    return O


def group_norm_gate(o, gpre, eps, w=None, b=None):
    """Eq. 7: swish(gpre) * GroupNorm_h(o) with one group per head.  o, gpre
    [B,N,H,d]; w, b [H*d] or None (1 and 0).  Returns fp64 z."""
    o, gpre = _f64(o), _f64(gpre)
    B, N, H, d = o.shape
    z = np.zeros_like(o)
    wp = None if w is None else _f64(np.asarray(w, dtype=np.float64).reshape(H * d))
    bp = None if b is None else _f64(np.asarray(b, dtype=np.float64).reshape(H * d))
    lib().oracle_group_norm_gate(B, N, H, d, _ptr(o), _ptr(gpre), None if wp is None else _ptr(wp),
                                 None if bp is None else _ptr(bp), float(eps), _ptr(z))
    return z


def rope(x, pos, base):
    """Rotary encoding of channel pairs (2i, 2i+1) by pos * base^(-2i/d).  x [..., d]
    (fp64 copy returned); pos broadcastable to x.shape[:-1] (integer positions)."""
    x = np.array(_f64(x), dtype=np.float64, copy=True)
    d = x.shape[-1]
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int64), x.shape[:-1]).reshape(-1))
    flat = np.ascontiguousarray(x.reshape(-1, d))
    lib().oracle_rope(flat.shape[0], d, p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), float(base), _ptr(flat))
    return flat.reshape(x.shape)


def qkvg_project(X, W, H, d, pos0=0, rope_base=0.0):
    """Section 3.1's projections of a gRet layer: Y = X W with W = [W_Q | W_K | W_V | W_gamma]
    (an fp64 matrix product), split into q, k, v [B, N, H, d] and the gate logits
    [B, N, H]; with rope_base > 0, q and k turned by position pos0 + n."""
    X, W = _f64(X), _f64(W)
    B, N, dm = X.shape
    Hd = H * d
    Y = X.reshape(B * N, dm) @ W
    q = Y[:, :Hd].reshape(B, N, H, d)
    k = Y[:, Hd:2 * Hd].reshape(B, N, H, d)
    v = Y[:, 2 * Hd:3 * Hd].reshape(B, N, H, d)
    logits = Y[:, 3 * Hd:3 * Hd + H].reshape(B, N, H)
    if rope_base > 0:
        pos = (pos0 + np.arange(N))[None, :, None]
        q = rope(q, pos, rope_base)
        k = rope(k, pos, rope_base)
    return q, k, v, logits
