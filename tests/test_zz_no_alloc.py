"""The allocation-free decode entry point (collected last on purpose).

yoco_cross_attn_decode_noalloc serves callers that cannot allocate device
memory while they decode; it keeps its split partials in scratch built into
the library instead of a caller workspace.  At the split
count it runs with, its output must equal yoco_cross_attn_decode's bit for bit
on consecutive calls (the scratch keeps the previous call's contents), and
both must match the oracle; an automatic split count whose partials would not
fit is lowered, and an explicit one is refused before anything runs.
"""
import ctypes

import pytest

import oracle
import synth
from _util import gen, host_bits, host_f64, max_abs, rel_l2

pytestmark = pytest.mark.gpu

BF16_REL_L2 = 1e-2
FP32_MAX_ABS = 1e-4
SCRATCH_BYTES = 4 << 20  # the built-in scratch's documented size
SEED = synth.DEFAULT_SEED


def _auto_splits(Y, cache, Hq):
    """The workspace call's automatic split count, read back from its workspace
    size (partials of B * Hq * splits * (d + 2) fp32 after a 256-byte status word)."""
    ws = Y.lib.yoco_cross_attn_workspace_size(cache.c.B, Hq, 1, ctypes.byref(cache.c), 0)
    per_split = cache.c.B * Hq * (cache.c.d + 2) * 4
    return max(1, (ws - 256) // per_split)


@pytest.fixture(scope="module")
def Y():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import gated_retention_shared_gb300 as Y
    return Y


def _cache(Y, B, Hkv, d, length, dtype="bf16"):
    Kh, Kd = gen(SEED, synth.stream_id(40, 0, synth.T_CACHE_K), (B, Hkv, length, d), dtype)
    Vh, Vd = gen(SEED, synth.stream_id(40, 0, synth.T_CACHE_V), (B, Hkv, length, d), dtype)
    cache = Y.KVCache(B, Hkv, d, length, dtype=Kd.dtype, k=Kd, v=Vd)
    cache.set_length(length)
    return cache, Kh, Vh


def _noalloc(Y, Qd, Hq, cache, d, num_splits, O):
    import torch
    return Y.lib.yoco_cross_attn_decode_noalloc(ctypes.c_void_p(Qd.data_ptr()), Hq, ctypes.byref(cache.c), d ** -0.5,
                                                num_splits, ctypes.c_void_p(O.data_ptr()),
                                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _splits_that_fit(B, Hq, d, auto):
    """The split count the no-workspace call runs with: the automatic one, lowered
    until the partials fit the 4 MiB scratch."""
    s = auto
    while s > 1 and 256 + B * Hq * s * (d + 2) * 4 > SCRATCH_BYTES:
        s -= 1
    return s


@pytest.mark.parametrize("B,Hq,Hkv,d,length,dtype", [
    (2, 24, 8, 128, 3001, "bf16"),    # the tensor-core decode kernel
    (3, 8, 2, 64, 2500, "f32"),       # the CUDA-core kernel (fp32, d = 64)
    (64, 64, 8, 128, 3001, "bf16"),   # automatic splits (2) need 4.26 MB of partials: lowered to fit
])
def test_noalloc_decode_matches_workspace_decode_and_oracle(Y, B, Hq, Hkv, d, length, dtype):
    """Two calls in a row, different queries.  At the split count the no-workspace
    call runs with, the workspace call runs the same kernels and must give the
    same bits; both are held to the oracle's naive softmax attention."""
    import torch
    cache, Kh, Vh = _cache(Y, B, Hkv, d, length, dtype)
    G = Hq // Hkv
    for call in range(2):
        Qh, Qd = gen(SEED, synth.stream_id(40, 1, synth.T_QX, call), (B, Hq, d), dtype)
        O = torch.full_like(Qd, float("nan"))
        st = _noalloc(Y, Qd, Hq, cache, d, 0, O)
        assert st == Y.YOCO_OK, Y.lib.yoco_last_error()
        torch.cuda.synchronize()
        splits = _splits_that_fit(B, Hq, d, _auto_splits(Y, cache, Hq))
        O_ws = torch.empty_like(Qd)
        Y.yoco_cross_attn_decode(Qd, cache, O_ws, num_splits=splits)
        torch.cuda.synchronize()
        if dtype == "bf16":
            assert bool((host_bits(O) == host_bits(O_ws)).all())
        else:
            assert bool((O.cpu() == O_ws.cpu()).all())
        for b, hk in {(0, 0), (B - 1, Hkv - 1)}:
            O_ref = oracle.cross_attn(Qh[b, hk * G:(hk + 1) * G][None, None], Kh[b, hk][None, None],
                                      Vh[b, hk][None, None], length - 1, d ** -0.5)[0, 0]
            got = host_f64(O[b, hk * G:(hk + 1) * G])
            if dtype == "bf16":
                assert rel_l2(got, O_ref) <= BF16_REL_L2
            else:
                assert max_abs(got, O_ref) <= FP32_MAX_ABS
    assert Y.lib.yoco_cross_attn_decode_noalloc_status(0, None) == Y.YOCO_OK, Y.lib.yoco_last_error()


def test_noalloc_decode_explicit_splits_bit_identical(Y):
    """An explicit split count that fits: the same kernels as the workspace call,
    so the same bits."""
    import torch
    B, Hq, Hkv, d, length = 2, 24, 8, 128, 3001
    cache, _, _ = _cache(Y, B, Hkv, d, length)
    for call in range(2):
        _, Qd = gen(SEED, synth.stream_id(40, 2, synth.T_QX, call), (B, Hq, d), "bf16")
        O_ref = torch.empty_like(Qd)
        Y.yoco_cross_attn_decode(Qd, cache, O_ref, num_splits=5)
        O = torch.full_like(Qd, float("nan"))
        assert _noalloc(Y, Qd, Hq, cache, d, 5, O) == Y.YOCO_OK, Y.lib.yoco_last_error()
        torch.cuda.synchronize()
        assert bool((host_bits(O) == host_bits(O_ref)).all())


def test_noalloc_decode_refuses_oversized_split_count(Y):
    import torch
    B, Hq, Hkv, d, length = 2, 24, 8, 128, 3001
    cache, _, _ = _cache(Y, B, Hkv, d, length)
    Qd = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros_like(Qd)
    st = Y.lib.yoco_cross_attn_decode_noalloc(ctypes.c_void_p(Qd.data_ptr()), Hq, ctypes.byref(cache.c), 0.1,
                                              4096, ctypes.c_void_p(O.data_ptr()), None)
    assert st == Y.YOCO_ERR_UNSUPPORTED
    assert b"scratch" in Y.lib.yoco_last_error()
    torch.cuda.synchronize()
    assert bool((O == 0).all())


def test_noalloc_decode_refuses_more_than_4096_splits(Y):
    """The merge holds one factor per split, at most 4096; a count above that
    is refused even when its partials would fit the scratch."""
    import torch
    B, Hq, Hkv, d, length = 1, 1, 1, 64, 3001
    cache, _, _ = _cache(Y, B, Hkv, d, length)
    Qd = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros_like(Qd)
    st = Y.lib.yoco_cross_attn_decode_noalloc(ctypes.c_void_p(Qd.data_ptr()), Hq, ctypes.byref(cache.c), 0.1,
                                              5000, ctypes.c_void_p(O.data_ptr()), None)
    assert st == Y.YOCO_ERR_UNSUPPORTED
    assert b"4096" in Y.lib.yoco_last_error()
    torch.cuda.synchronize()
    assert bool((O == 0).all())
