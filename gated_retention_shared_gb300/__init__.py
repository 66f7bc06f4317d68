"""Python binding of libyoco (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: it reads shapes and device pointers off torch
tensors, passes them with the current CUDA stream through ctypes, and raises
on a non-OK status.  All computation runs in the CUDA kernels of
``_build/libyoco.so``; there is no fallback.  If the library is missing the
import fails with a message saying how to build it.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# YOCO_LIB_PATH selects another build of the same library (the debug-checks build
# in _build_debug/, for its tests); the default is the release build
LIB_PATH = os.environ.get("YOCO_LIB_PATH") or os.path.join(_HERE, "_build", "libyoco.so")

YOCO_OK, YOCO_ERR_INVALID_ARG, YOCO_ERR_UNSUPPORTED, YOCO_ERR_CAPACITY, YOCO_ERR_CUDA, YOCO_ERR_TIMEOUT, \
    YOCO_ERR_WORKSPACE = range(7)
YOCO_F32, YOCO_BF16 = 0, 1


class YocoError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status} ({detail})")
        self.status = status


class _KVCacheC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len_dev", ctypes.c_void_p),
                ("len_host", ctypes.c_int64), ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("capacity", ctypes.c_int64), ("dtype", ctypes.c_int),
                ("rope_base", ctypes.c_float)]


class _SwaRingC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("window", ctypes.c_int32), ("pos", ctypes.c_int64), ("dtype", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libyoco.so not found at {LIB_PATH}; build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_int64
    cp = ctypes.POINTER(_KVCacheC)
    rp = ctypes.POINTER(_SwaRingC)
    sigs = {
        "yoco_gret_prefill_chunkwise": (i, [vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, i, i, i, vp, sz, vp]),
        "yoco_gret_prefill_workspace_size": (sz, [i, i, i, i, i, i, i]),
        "yoco_gret_decode_step": (i, [vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, i, vp]),
        "yoco_shared_kv_project_append": (i, [vp, vp, f, vp, vp, i, i, cp, vp, sz, vp]),
        "yoco_shared_kv_workspace_size": (sz, [i, i, i, cp]),
        "yoco_cross_attn_prefill": (i, [vp, i, i, i64, cp, f, vp, vp, sz, vp]),
        "yoco_cross_attn_decode": (i, [vp, i, cp, f, i, vp, vp, sz, vp]),
        "yoco_cross_attn_workspace_size": (sz, [i, i, i, cp, i]),
        "yoco_cross_attn_decode_noalloc": (i, [vp, i, cp, f, i, vp, vp]),
        "yoco_status_string": (ctypes.c_char_p, [i]),
        "yoco_last_error": (ctypes.c_char_p, []),
        "yoco_version": (i, []),
        "yoco_launch_count": (ctypes.c_uint64, []),
        "yoco_workspace_status": (i, [vp, i, vp]),
        "yoco_selftest_wait_timeout": (i, [vp, ctypes.c_uint64, vp]),
        "yoco_swa_prefill": (i, [vp, vp, vp, i, i, f, vp, rp, vp, sz, vp]),
        "yoco_swa_decode": (i, [vp, vp, vp, i, f, vp, rp, vp, sz, vp]),
        "yoco_swa_workspace_size": (sz, [i, i, rp]),
        "yoco_gret_group_norm_gate": (i, [vp, vp, vp, vp, f, vp, i, i, i, i, i, vp]),
        "yoco_gret_decode_step_gn_gate": (i, [vp, vp, vp, vp, f, vp, vp, vp, vp, f, vp, i, i, i, i, i, vp]),
        "yoco_rope_apply": (i, [vp, i, i, i, i, i64, f, i, vp]),
        "yoco_gret_qkvg_project": (i, [vp, vp, i, i, i, i, i, i64, f, vp, vp, vp, vp, vp, sz, vp]),
        "yoco_gret_qkvg_workspace_size": (sz, [i, i, i, i, f]),
        "yoco_cross_attn_decode_noalloc_status": (i, [i, vp]),
        "yoco_test_hook": (i, [i, i64]),
        "yoco_gret_prefill_chunkwise_gn_gate": (i, [vp, vp, vp, vp, f, vp, vp, vp, f, vp, vp, i, i, i, i, i, i, vp, sz,
                                                    vp]),
        "yoco_selftest_occupy_sms": (i, [i, ctypes.c_uint64, vp]),
        "yoco_debug_checks": (i, [i, ctypes.POINTER(ctypes.c_uint32)]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


lib = _load()
EXPORTED = ("yoco_gret_prefill_chunkwise", "yoco_gret_prefill_workspace_size", "yoco_gret_decode_step",
            "yoco_shared_kv_project_append", "yoco_shared_kv_workspace_size", "yoco_cross_attn_prefill",
            "yoco_cross_attn_decode", "yoco_cross_attn_workspace_size", "yoco_status_string",
            "yoco_last_error", "yoco_version", "yoco_launch_count",
            "yoco_workspace_status", "yoco_cross_attn_decode_noalloc", "yoco_selftest_wait_timeout",
            "yoco_swa_prefill", "yoco_swa_decode", "yoco_swa_workspace_size", "yoco_gret_group_norm_gate",
            "yoco_rope_apply", "yoco_gret_qkvg_project", "yoco_gret_qkvg_workspace_size",
            "yoco_gret_decode_step_gn_gate", "yoco_cross_attn_decode_noalloc_status", "yoco_test_hook",
            "yoco_selftest_occupy_sms", "yoco_gret_prefill_chunkwise_gn_gate", "yoco_debug_checks")
YOCO_HOOK_FAIL_NEXT_CALLS, YOCO_HOOK_GRET_SEG0_DELAY_NS, YOCO_HOOK_GRET_SEGMENTS = 1, 2, 3


def _check(status: int, where: str):
    if status != YOCO_OK:
        detail = lib.yoco_last_error().decode() or lib.yoco_status_string(status).decode()
        raise YocoError(status, where, detail)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return YOCO_F32
    if t.dtype == torch.bfloat16:
        return YOCO_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return workspace
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace


# ------------------------------------------------------------------ gRet

def yoco_gret_prefill_workspace_size(B, N, H, dk, dv, chunk, dtype) -> int:
    return lib.yoco_gret_prefill_workspace_size(B, N, H, dk, dv, chunk, dtype)


def yoco_gret_prefill_chunkwise(q, k, v, gate_logits, tau, o, state, chunk=0, workspace=None, stream=None):
    """q, k [B,N,H,dk]; v, o [B,N,H,dv]; gate_logits [B,N,H] fp32; state [B,H,dk,dv] fp32 (in/out)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate_logits, "gate_logits"), (o, "o"), (state, "state")):
        _need(t, n)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dt(q)
    ws_n = lib.yoco_gret_prefill_workspace_size(B, N, H, dk, dv, chunk, dt)
    ws = _workspace(ws_n, q.device, workspace)
    st = lib.yoco_gret_prefill_chunkwise(_ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), float(tau), _ptr(o),
                                         _ptr(state), B, N, H, dk, dv, chunk, dt, _dt(o), _ptr(ws),
                                         0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_gret_prefill_chunkwise")


def yoco_gret_prefill_chunkwise_gn_gate(q, k, v, gate_logits, tau, gate, z, state, eps=1e-5, gn_weight=None,
                                        gn_bias=None, workspace=None, stream=None):
    """z = swish(gate) * GroupNorm_h(chunkwise gRet output); q, k, v, gate, z [B,N,H,d];
    gate_logits [B,N,H] fp32; state [B,H,d,d] fp32 (in/out); gn_weight, gn_bias fp32 [H*d] or None."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate_logits, "gate_logits"), (gate, "gate"), (z, "z"),
                 (state, "state")):
        _need(t, n)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dt(q)
    for t, n in ((gn_weight, "gn_weight"), (gn_bias, "gn_bias")):
        if t is not None and (t.dtype != torch.float32 or t.numel() != H * dv):
            raise ValueError(f"{n} must be fp32 with H * d elements")
    ws_n = lib.yoco_gret_prefill_workspace_size(B, N, H, dk, dv, 0, dt)
    ws = _workspace(ws_n, q.device, workspace)
    st = lib.yoco_gret_prefill_chunkwise_gn_gate(_ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), float(tau), _ptr(gate),
                                                 _ptr(gn_weight), _ptr(gn_bias), float(eps), _ptr(z), _ptr(state), B, N,
                                                 H, dk, dv, dt, _ptr(ws),
                                                 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_gret_prefill_chunkwise_gn_gate")


def yoco_workspace_status(workspace, clear=True, stream=None):
    """Wait for the stream and raise YocoError(YOCO_ERR_TIMEOUT) if a kernel
    that used `workspace` gave up a bounded on-device wait."""
    _check(lib.yoco_workspace_status(_ptr(workspace), int(clear), _stream(stream)), "yoco_workspace_status")


def yoco_gret_decode_step(q, k, v, gate_logits, tau, state, o, stream=None):
    """q, k [B,H,dk]; v, o [B,H,dv]; gate_logits [B,H] fp32; state [B,H,dk,dv] fp32 (in/out)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate_logits, "gate_logits"), (o, "o"), (state, "state")):
        _need(t, n)
    B, H, dk = q.shape
    dv = v.shape[-1]
    st = lib.yoco_gret_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), float(tau), _ptr(state),
                                   _ptr(o), B, H, dk, dv, _dt(q), _dt(o), _stream(stream))
    _check(st, "yoco_gret_decode_step")


def yoco_gret_decode_step_gn_gate(q, k, v, gate_logits, tau, state, gate, z, eps=1e-5, gn_weight=None, gn_bias=None,
                                  stream=None):
    """One recurrent step and, fused, z = swish(gate) * GroupNorm_h(o) for that token.
    q, k [B,H,dk]; v, gate, z [B,H,dv] (one dtype); gate_logits [B,H] fp32; state
    [B,H,dk,dv] fp32 (in/out); gn_weight, gn_bias fp32 [H * dv] or None."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate_logits, "gate_logits"), (state, "state"), (gate, "gate"),
                 (z, "z")):
        _need(t, n)
    B, H, dk = q.shape
    dv = v.shape[-1]
    for t, n in ((gn_weight, "gn_weight"), (gn_bias, "gn_bias")):
        if t is not None and (t.dtype != torch.float32 or t.numel() != H * dv):
            raise ValueError(f"{n} must be fp32 with H * dv elements")
    st = lib.yoco_gret_decode_step_gn_gate(_ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), float(tau), _ptr(state),
                                           _ptr(gate), _ptr(gn_weight), _ptr(gn_bias), float(eps), _ptr(z), B, H, dk,
                                           dv, _dt(q), _stream(stream))
    _check(st, "yoco_gret_decode_step_gn_gate")


# ------------------------------------------------------------- shared KV

class KVCache:
    """Caller-side holder of the shared K^/V^ cache: two [B, Hkv, capacity, d]
    tensors, the device length pair and the C descriptor that points at them."""

    def __init__(self, B, Hkv, d, capacity, dtype=torch.bfloat16, device="cuda", k=None, v=None, rope_base=0.0):
        self.k = k if k is not None else torch.zeros(B, Hkv, capacity, d, dtype=dtype, device=device)
        self.v = v if v is not None else torch.zeros(B, Hkv, capacity, d, dtype=dtype, device=device)
        self.len_dev = torch.zeros(2, dtype=torch.int32, device=self.k.device)
        self.c = _KVCacheC(self.k.data_ptr(), self.v.data_ptr(), self.len_dev.data_ptr(), 0, B, Hkv, d,
                           capacity, _dt(self.k), float(rope_base))

    @property
    def length(self) -> int:
        return int(self.c.len_host)

    def set_length(self, n: int):
        """Declare the first n slots filled (e.g. after writing k/v directly)."""
        self.c.len_host = n
        self.len_dev[0] = n

    @staticmethod
    def nbytes(B, Hkv, d, capacity, elem_bytes=2) -> int:
        return 2 * B * Hkv * capacity * d * elem_bytes


def yoco_shared_kv_project_append(M, Wk, Wv, cache: KVCache, eps=1e-6, rms_w=None, workspace=None, stream=None):
    """M [B, T, dm]; Wk, Wv [dm, Hkv*d]; appends T slots to `cache`."""
    for t, n in ((M, "M"), (Wk, "Wk"), (Wv, "Wv")):
        _need(t, n)
    B, T, dm = M.shape
    ws_n = lib.yoco_shared_kv_workspace_size(B, T, dm, ctypes.byref(cache.c))
    ws = _workspace(ws_n, M.device, workspace)
    st = lib.yoco_shared_kv_project_append(_ptr(M), _ptr(rms_w), float(eps), _ptr(Wk), _ptr(Wv), T, dm,
                                           ctypes.byref(cache.c), _ptr(ws),
                                           0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_shared_kv_project_append")


# -------------------------------------------------------- cross attention

def yoco_cross_attn_decode_noalloc(Q, cache: KVCache, O, scale=None, num_splits=0, stream=None):
    """Decode attention without a workspace: the split partials go to scratch
    built into the library, for callers that cannot allocate device memory.
    Calls on one device share that scratch, so do not overlap them."""
    _need(Q, "Q")
    _need(O, "O")
    B, Hq, d = Q.shape
    scale = d ** -0.5 if scale is None else scale
    st = lib.yoco_cross_attn_decode_noalloc(_ptr(Q), Hq, ctypes.byref(cache.c), float(scale), num_splits, _ptr(O),
                                            _stream(stream))
    _check(st, "yoco_cross_attn_decode_noalloc")


def yoco_cross_attn_workspace_size(B, Hq, T, cache: KVCache, num_splits=0) -> int:
    return lib.yoco_cross_attn_workspace_size(B, Hq, T, ctypes.byref(cache.c), num_splits)


def yoco_cross_attn_prefill(Q, cache: KVCache, p0, O, scale=None, workspace=None, stream=None):
    """Q, O [B, T, Hq, d]; rows at positions p0..p0+T-1."""
    _need(Q, "Q")
    _need(O, "O")
    B, T, Hq, d = Q.shape
    scale = d ** -0.5 if scale is None else scale
    ws_n = lib.yoco_cross_attn_workspace_size(B, Hq, T, ctypes.byref(cache.c), 0)
    ws = _workspace(ws_n, Q.device, workspace)
    st = lib.yoco_cross_attn_prefill(_ptr(Q), Hq, T, int(p0), ctypes.byref(cache.c), float(scale), _ptr(O), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_cross_attn_prefill")


def yoco_cross_attn_decode(Q, cache: KVCache, O, scale=None, num_splits=0, workspace=None, stream=None):
    """Q, O [B, Hq, d]; the query sits at position len - 1."""
    _need(Q, "Q")
    _need(O, "O")
    B, Hq, d = Q.shape
    scale = d ** -0.5 if scale is None else scale
    ws_n = lib.yoco_cross_attn_workspace_size(B, Hq, 1, ctypes.byref(cache.c), num_splits)
    ws = _workspace(ws_n, Q.device, workspace)
    st = lib.yoco_cross_attn_decode(_ptr(Q), Hq, ctypes.byref(cache.c), float(scale), num_splits, _ptr(O), _ptr(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_cross_attn_decode")


# ----------------------------------------------- sliding-window self-decoder

class SwaRing:
    """Caller-side ring cache of one sliding-window layer: k, v [B, Hkv, window, d]
    (token at position p in slot p % window) and the C descriptor; `pos` counts
    the tokens seen."""

    def __init__(self, B, Hkv, d, window, dtype=torch.bfloat16, device="cuda"):
        self.k = torch.zeros(B, Hkv, window, d, dtype=dtype, device=device)
        self.v = torch.zeros(B, Hkv, window, d, dtype=dtype, device=device)
        self.c = _SwaRingC(self.k.data_ptr(), self.v.data_ptr(), B, Hkv, d, window, 0, _dt(self.k))

    @property
    def pos(self) -> int:
        return int(self.c.pos)


def yoco_swa_prefill(q, k, v, ring: SwaRing, o, scale=None, workspace=None, stream=None):
    """q, o [B, N, Hq, d]; k, v [B, N, Hkv, d]; starts the sequence held in `ring`."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, n)
    B, N, Hq, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    ws = _workspace(max(256, lib.yoco_swa_workspace_size(B, Hq, ctypes.byref(ring.c))), q.device, workspace)
    st = lib.yoco_swa_prefill(_ptr(q), _ptr(k), _ptr(v), Hq, N, float(scale), _ptr(o), ctypes.byref(ring.c),
                              _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_swa_prefill")


def yoco_swa_decode(q, k, v, ring: SwaRing, o, scale=None, workspace=None, stream=None):
    """q, o [B, Hq, d]; k, v [B, Hkv, d] of the new token."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, n)
    B, Hq, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    ws = _workspace(max(256, lib.yoco_swa_workspace_size(B, Hq, ctypes.byref(ring.c))), q.device, workspace)
    st = lib.yoco_swa_decode(_ptr(q), _ptr(k), _ptr(v), Hq, float(scale), _ptr(o), ctypes.byref(ring.c), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "yoco_swa_decode")


def yoco_gret_group_norm_gate(o, gate, z, eps=1e-5, gn_weight=None, gn_bias=None, stream=None):
    """z = swish(gate) * GroupNorm_h(o); o, gate, z [B, N, H, d] (or [B, H, d] for a decode step);
    gn_weight, gn_bias fp32 [H * d] or None.  z may be o."""
    for t, n in ((o, "o"), (gate, "gate"), (z, "z")):
        _need(t, n)
    if o.dim() == 3:
        B, H, d = o.shape
        N = 1
    else:
        B, N, H, d = o.shape
    for t, n in ((gn_weight, "gn_weight"), (gn_bias, "gn_bias")):
        if t is not None and (t.dtype != torch.float32 or t.numel() != H * d):
            raise ValueError(f"{n} must be fp32 with H * d elements")
    st = lib.yoco_gret_group_norm_gate(_ptr(o), _ptr(gate), _ptr(gn_weight), _ptr(gn_bias), float(eps), _ptr(z), B, N,
                                       H, d, _dt(o), _stream(stream))
    _check(st, "yoco_gret_group_norm_gate")


# ------------------------------------------------- rotary position encoding

def yoco_rope_apply(x, base, pos0=0, stream=None):
    """Rotary encoding of x [B, N, H, d] (token-major q or k) in place: row n at position pos0 + n."""
    _need(x, "x")
    B, N, H, d = x.shape
    st = lib.yoco_rope_apply(_ptr(x), B, N, H, d, int(pos0), float(base), _dt(x), _stream(stream))
    _check(st, "yoco_rope_apply")


def yoco_gret_qkvg_project(X, W, H, q, k, v, gate_logits, rope_base=0.0, pos0=0, workspace=None, stream=None):
    """X [B, N, dm] bf16; W [dm, 3 H d + H] bf16 (W_Q | W_K | W_V | W_gamma); writes q, k, v
    [B, N, H, d] bf16 and gate_logits [B, N, H] fp32."""
    for t, n in ((X, "X"), (W, "W"), (q, "q"), (k, "k"), (v, "v"), (gate_logits, "gate_logits")):
        _need(t, n)
    B, N, dm = X.shape
    d = q.shape[-1]
    ws_n = lib.yoco_gret_qkvg_workspace_size(B, N, H, d, float(rope_base))
    ws = _workspace(ws_n, X.device, workspace)
    st = lib.yoco_gret_qkvg_project(_ptr(X), _ptr(W), B, N, dm, H, d, int(pos0), float(rope_base), _ptr(q), _ptr(k),
                                    _ptr(v), _ptr(gate_logits), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream))
    _check(st, "yoco_gret_qkvg_project")
