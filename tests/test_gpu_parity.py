"""GPU parity: every libyoco call against the CPU oracle on the same seeded
inputs, through the C ABI (the Python binding only marshals arguments).

Tolerances: fp32 paths max-abs <= 1e-4; bf16-input / fp32-accumulate paths
relative L2 <= 1e-2 per output tensor; the cache append bit-exact where the
inputs make every sum exact.  Sizes span several chunks / tiles / splits and
end on ragged tails.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from _util import dev_bf16, dev_f32, gen, host_bits, host_f64, max_abs, rel_l2, worst_block_rel_l2

pytestmark = pytest.mark.gpu

FP32_MAX_ABS = 1e-4
BF16_REL_L2 = 1e-2
BLOCK_REL_L2 = 3e-2  # worst 128-row block: bf16 rounding of one block, with room (a wrong block is ~1)
SEED = synth.DEFAULT_SEED


@pytest.fixture(scope="module")
def Y():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import gated_retention_shared_gb300 as Y
    return Y


def sid(cfg, layer, tensor, step=0):
    return synth.stream_id(cfg, layer, tensor, step)


def gret_inputs(cfg, B, N, H, d, dtype, logit_mean=0.0, qk_std=None):
    qk_std = d ** -0.5 if qk_std is None else qk_std
    q, qd = gen(SEED, sid(cfg, 0, synth.T_Q), (B, N, H, d), dtype, std=qk_std)
    k, kd = gen(SEED, sid(cfg, 0, synth.T_K), (B, N, H, d), dtype, std=qk_std)
    v, vd = gen(SEED, sid(cfg, 0, synth.T_V), (B, N, H, d), dtype)
    lg = synth.normal(SEED, sid(cfg, 0, synth.T_LOGIT), (B, N, H), "f32", mean=logit_mean)
    return (q, k, v, lg.astype(np.float64)), (qd, kd, vd, dev_f32(lg))


def run_prefill(Y, dev_in, B, N, H, d, dtype, S0=None, chunk=0):
    import torch
    qd, kd, vd, lgd = dev_in
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    o = torch.empty(B, N, H, d, dtype=tdt, device="cuda")
    S = torch.zeros(B, H, d, d, dtype=torch.float32, device="cuda") if S0 is None else dev_f32(S0)
    Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, S, chunk=chunk)
    torch.cuda.synchronize()
    return host_f64(o), S.cpu().numpy().astype(np.float64)


# --------------------------------------------------------------- gRet prefill

def test_gret_prefill_fp32_tiny_config(Y):
    """B=1, N=256, 2 heads x 64, q,k,v ~ N(0,1)/8, logits ~ N(0,1), tau 16, chunk 64."""
    B, N, H, d = 1, 256, 2, 64
    host, dev = gret_inputs(1, B, N, H, d, "f32", qk_std=1 / 8)
    o, S = run_prefill(Y, dev, B, N, H, d, "f32", chunk=64)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0)
    assert max_abs(o, o_ref) <= FP32_MAX_ABS
    assert max_abs(S, S_ref) <= FP32_MAX_ABS


@pytest.mark.parametrize("N", [1, 63, 200, 2049])
def test_gret_prefill_fp32_ragged_with_state(Y, N):
    """Ragged lengths, B=2, d=128, a non-zero initial state; N=2049 runs the
    sequence-split path (segment states + scan)."""
    B, H, d = 2, 3, 128
    host, dev = gret_inputs(10 + N % 7, B, N, H, d, "f32", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(11, 0, synth.T_S0), (B, H, d, d), "f32", std=0.1).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "f32", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert max_abs(o, o_ref) <= FP32_MAX_ABS
    assert max_abs(S, S_ref) <= FP32_MAX_ABS


def test_gret_prefill_fp32_many_segments(Y):
    """One head, long sequence: the kernel splits it into many segments."""
    B, N, H, d = 1, 5000, 1, 64
    host, dev = gret_inputs(12, B, N, H, d, "f32", logit_mean=3.0)
    o, S = run_prefill(Y, dev, B, N, H, d, "f32")
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0)
    assert max_abs(o, o_ref) <= FP32_MAX_ABS
    assert max_abs(S, S_ref) <= FP32_MAX_ABS


@pytest.mark.parametrize("chunk", [0, 64, 128])
@pytest.mark.parametrize("N", [130, 1500])
def test_gret_prefill_bf16(Y, N, chunk):
    B, H, d = 1, 4, 128
    host, dev = gret_inputs(2, B, N, H, d, "bf16", logit_mean=2.0)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", chunk=chunk)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    assert rel_l2(S, S_ref) <= BF16_REL_L2


@pytest.mark.parametrize("B,N,H,with_state", [(1, 8192 + 77, 24, True), (2, 300, 80, True), (1, 128, 3, False),
                                              (3, 1, 2, True)])
def test_gret_prefill_bf16_tensor_core_shapes(Y, B, N, H, with_state):
    """Tensor-core path: many chunks per segment (N=8269 over 24 heads), one
    segment per sequence (B*H >= 152), exactly one chunk, a single token."""
    import torch
    d = 128
    host, dev = gret_inputs(7, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = None
    if with_state:
        S0 = synth.normal(SEED, sid(7, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    assert rel_l2(S, S_ref) <= BF16_REL_L2
    ws = torch.empty(max(256, Y.yoco_gret_prefill_workspace_size(B, N, H, d, d, 0, Y.YOCO_BF16)),
                     dtype=torch.uint8, device="cuda")
    qd, kd, vd, lgd = dev
    o2 = torch.empty_like(vd)
    S2 = torch.zeros(B, H, d, d, device="cuda")
    Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o2, S2, workspace=ws)
    Y.yoco_workspace_status(ws)  # no bounded wait gave up


@pytest.mark.parametrize("B,N,H", [(1, 10000, 5), (3, 3100, 7), (1, 6403, 9)])
def test_gret_prefill_bf16_uneven_head_counts(Y, B, N, H):
    """Head counts that do not divide the SM count (5, 3 x 7 and 9 heads: 27,
    7 and 13 segments of 3, 4 and 4 chunks, the last one shorter and ragged),
    from an initial state: every head's output, worst 128-row block and final
    state against the oracle."""
    d = 128
    host, dev = gret_inputs(48, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(48, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    for b in range(B):
        for h in range(H):
            assert worst_block_rel_l2(o[b, :, h], o_ref[b, :, h], 128) <= BLOCK_REL_L2, (b, h)
            assert rel_l2(S[b, h], S_ref[b, h]) <= BF16_REL_L2, (b, h)


@pytest.mark.parametrize("B,N,H", [(1, 128 * 100 + 33, 1), (2, 300, 38)])
def test_gret_prefill_bf16_segment_prefix_extremes(Y, B, N, H):
    """Each output CTA folds the earlier segments' end states into its own
    initial state: one head over 101 chunks (101 one-chunk segments; a chunk
    decays by about e^-1.4 here, so the later CTAs fold the last ~28 states and
    leave the older ones out) and 76 heads (two segments), both from an initial
    state."""
    d = 128
    host, dev = gret_inputs(37, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(37, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    assert rel_l2(S, S_ref) <= BF16_REL_L2


def test_gret_prefill_bf16_many_segments_state_and_strong_decay(Y):
    """Many segments per head with an initial state and a stretch of near-zero
    gates inside a segment (B=2, N=7600, 4 heads: 15 segments of 4
    chunks; chunk 15 has total decay far below the factoring limit)."""
    B, N, H, d = 2, 7600, 4, 128
    host, dev = gret_inputs(31, B, N, H, d, "bf16", logit_mean=1.0)
    lg = host[3].copy()
    lg[:, 2000:2010] = -2000.0
    dev = dev[:3] + (dev_f32(lg),)
    S0 = synth.normal(SEED, sid(31, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(host[0], host[1], host[2], lg, 16.0, S0=S0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    assert rel_l2(S, S_ref) <= BF16_REL_L2


def test_gret_prefill_bf16_no_decay_many_segments(Y):
    """gamma = 1 everywhere (logits +inf): no state contribution is small, so the
    segment-state walk covers every chunk and every output CTA folds all earlier
    segments and the initial state (41 one-chunk segments of one head)."""
    B, N, H, d = 1, 128 * 40 + 17, 2, 128
    host, dev = gret_inputs(41, B, N, H, d, "bf16")
    lg = np.full_like(host[3], np.inf)
    dev = dev[:3] + (dev_f32(lg),)
    S0 = synth.normal(SEED, sid(41, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(host[0], host[1], host[2], lg, 16.0, S0=S0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    assert rel_l2(S, S_ref) <= BF16_REL_L2


def test_gret_prefill_bf16_mixed_decay_across_segments(Y):
    """Segments that decay strongly (the backward walk stops after a couple of
    chunks and later segments leave the older states out) next to segments
    with no decay at all (the walk and the fold reach back through them), from
    an initial state: 24 heads, 6 segments of 11 chunks."""
    B, N, H, d = 1, 128 * 60 + 50, 24, 128
    host, dev = gret_inputs(42, B, N, H, d, "bf16", logit_mean=2.0)
    lg = host[3].copy()
    seg = 11 * 128
    lg[:, 0:seg] = np.inf                    # segment 0: gamma = 1
    lg[:, seg:2 * seg] -= 5.0                # segment 1: about e^-0.3 per token
    lg[:, 2 * seg:3 * seg] = np.inf          # segment 2: gamma = 1
    lg[:, 4 * seg + 300:4 * seg + 420] = -8  # a strongly decaying stretch inside segment 4
    lg[:, :, ::2] = np.inf                   # every other head never decays
    dev = dev[:3] + (dev_f32(lg),)
    S0 = synth.normal(SEED, sid(42, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    o_ref, S_ref = oracle.gret_recurrent(host[0], host[1], host[2], lg, 16.0, S0=S0)
    for h in range(H):
        assert rel_l2(o[:, :, h], o_ref[:, :, h]) <= BF16_REL_L2, h
        assert worst_block_rel_l2(o[0, :, h], o_ref[0, :, h], 128) <= BLOCK_REL_L2, h
        assert rel_l2(S[:, h], S_ref[:, h]) <= BF16_REL_L2, h


@pytest.mark.parametrize("B,N,H", [(1, 4000, 8), (1, 10000, 5)])
def test_gret_prefill_final_state_parked_hand_off(Y, B, N, H):
    """With segment 0 made to take the caller's state 20 ms late (test hook), the
    last segment of every head finishes first, parks the final state in the
    workspace, and segment 0 copies it to `state` after reading the initial one
    (8 heads of 16 segments; 5 heads of 27).  Two calls in a row on one
    workspace; results as without the delay."""
    import torch
    d = 128
    host, dev = gret_inputs(43, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(43, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    ws = torch.empty(max(256, Y.yoco_gret_prefill_workspace_size(B, N, H, d, d, 0, Y.YOCO_BF16)),
                     dtype=torch.uint8, device="cuda")
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_GRET_SEG0_DELAY_NS, 20_000_000) == Y.YOCO_OK
    try:
        qd, kd, vd, lgd = dev
        for _ in range(2):
            S = dev_f32(S0)
            o = torch.empty_like(vd)
            Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, S, workspace=ws)
            torch.cuda.synchronize()
            Y.yoco_workspace_status(ws)
            o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
            assert rel_l2(host_f64(o), o_ref) <= BF16_REL_L2
            assert rel_l2(S.cpu().numpy().astype(np.float64), S_ref) <= BF16_REL_L2
    finally:
        assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_GRET_SEG0_DELAY_NS, 0) == Y.YOCO_OK


def test_injected_launch_failure_writes_nothing(Y):
    """A launch failure injected in the status layer (test hook): the gRet
    prefill and the decode attention return YOCO_ERR_CUDA with the outputs and
    the state untouched, and the next calls run normally."""
    import torch
    B, N, H, d = 1, 300, 2, 128
    host, dev = gret_inputs(44, B, N, H, d, "bf16", logit_mean=2.0)
    qd, kd, vd, lgd = dev
    o = torch.full_like(vd, 7.0)
    S = torch.full((B, H, d, d), 3.0, device="cuda")
    ws = torch.empty(max(256, Y.yoco_gret_prefill_workspace_size(B, N, H, d, d, 0, Y.YOCO_BF16)),
                     dtype=torch.uint8, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_FAIL_NEXT_CALLS, 2) == Y.YOCO_OK
    n0 = Y.lib.yoco_launch_count()
    st = Y.lib.yoco_gret_prefill_chunkwise(P(qd), P(kd), P(vd), P(lgd), 16.0, P(o), P(S), B, N, H, d, d, 0, 1, 1,
                                           P(ws), ws.numel(), stream)
    assert st == Y.YOCO_ERR_CUDA and b"launch failure" in Y.lib.yoco_last_error()
    Kc, Vc = torch.randn(1, 2, 64, d, device="cuda").bfloat16(), torch.randn(1, 2, 64, d, device="cuda").bfloat16()
    cache = Y.KVCache(1, 2, d, 64, k=Kc, v=Vc)
    cache.set_length(64)
    Qd = torch.randn(1, 6, d, device="cuda").bfloat16()
    Od = torch.full_like(Qd, 5.0)
    wsa = torch.empty(max(256, Y.lib.yoco_cross_attn_workspace_size(1, 6, 1, ctypes.byref(cache.c), 0)),
                      dtype=torch.uint8, device="cuda")
    st = Y.lib.yoco_cross_attn_decode(P(Qd), 6, ctypes.byref(cache.c), 0.1, 0, P(Od), P(wsa), wsa.numel(), stream)
    assert st == Y.YOCO_ERR_CUDA
    assert Y.lib.yoco_launch_count() == n0  # nothing was enqueued
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((S == 3.0).all()) and bool((Od == 5.0).all())
    # the hook is spent: the same calls now run and match the oracle
    S.zero_()
    Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, S, workspace=ws)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0)
    assert rel_l2(host_f64(o), o_ref) <= BF16_REL_L2
    Y.yoco_cross_attn_decode(Qd, cache, Od)
    torch.cuda.synchronize()
    assert np.isfinite(host_f64(Od)).all()


def test_gret_prefill_bf16_strong_decay(Y):
    """Gates near 0 inside chunks (b_C < -80) take the direct-exponent branch."""
    B, N, H, d = 1, 1000, 4, 128
    host, dev = gret_inputs(8, B, N, H, d, "bf16", logit_mean=-6.0)
    lg = host[3].copy()
    lg[:, 500:530] = -2000.0
    dev = dev[:3] + (dev_f32(lg),)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16")
    o_ref, S_ref = oracle.gret_recurrent(host[0], host[1], host[2], lg, 16.0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    assert rel_l2(S, S_ref) <= BF16_REL_L2


def test_gret_prefill_state_continuation(Y):
    """Two calls with the state carried equal one oracle pass (chunked prefill)."""
    B, N, H, d = 1, 1500, 2, 128
    host, dev = gret_inputs(3, B, N, H, d, "bf16", logit_mean=2.0)
    import torch
    n1 = 700
    parts = [tuple(t[:, :n1].contiguous() for t in dev), tuple(t[:, n1:].contiguous() for t in dev)]
    S = torch.zeros(B, H, d, d, dtype=torch.float32, device="cuda")
    outs = []
    for (qd, kd, vd, lgd) in parts:
        o = torch.empty_like(vd)
        Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, S)
        outs.append(host_f64(o))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0)
    assert rel_l2(np.concatenate(outs, axis=1), o_ref) <= BF16_REL_L2
    assert rel_l2(S.cpu().numpy(), S_ref) <= BF16_REL_L2


def test_gret_prefill_two_calls_on_one_dirty_workspace(Y):
    """Two chained calls (the second continues the first's final state) on one
    workspace that starts as int32 ones (status word aside): segment 0 of each
    (b, h) starts from the caller's state while the first pass runs, and the
    final state replaces it only after segment 0 has its copy (the hand-off word
    is cleared by each call; 16 segments per head here, with a nonzero initial
    state)."""
    import torch
    B, N, H, d = 1, 4000, 8, 128
    host, dev = gret_inputs(37, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(37, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    n1 = 2048
    nbytes = max(256, Y.yoco_gret_prefill_workspace_size(B, max(n1, N - n1), H, d, d, 0, Y.YOCO_BF16))
    ws = torch.ones((nbytes + 3) // 4, dtype=torch.int32, device="cuda").view(torch.uint8)[:nbytes]
    ws[:256] = 0
    S = dev_f32(S0)
    outs = []
    for sl in (slice(0, n1), slice(n1, N)):
        qd, kd, vd, lgd = (t[:, sl].contiguous() for t in dev)
        o = torch.empty_like(vd)
        Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, S, workspace=ws)
        outs.append(o)
    torch.cuda.synchronize()
    Y.yoco_workspace_status(ws)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert rel_l2(np.concatenate([host_f64(o) for o in outs], axis=1), o_ref) <= BF16_REL_L2
    assert rel_l2(S.cpu().numpy().astype(np.float64), S_ref) <= BF16_REL_L2


def test_gret_prefill_gate_limits(Y):
    """Logits of +inf (gamma = 1) and -inf (gamma = 0) mixed in."""
    B, N, H, d = 1, 300, 2, 64
    host, dev = gret_inputs(4, B, N, H, d, "f32")
    lg = host[3].copy()
    lg[:, ::7] = np.inf
    lg[:, 3::11] = -np.inf
    dev = dev[:3] + (dev_f32(lg),)
    o, S = run_prefill(Y, dev, B, N, H, d, "f32")
    o_ref, S_ref = oracle.gret_recurrent(host[0], host[1], host[2], lg, 16.0)
    assert max_abs(o, o_ref) <= FP32_MAX_ABS
    assert max_abs(S, S_ref) <= FP32_MAX_ABS


def test_gret_prefill_empty_sequence(Y):
    import torch
    S = torch.full((1, 2, 64, 64), 0.5, device="cuda")
    z = torch.empty(1, 0, 2, 64, device="cuda")
    lg = torch.empty(1, 0, 2, device="cuda")
    Y.yoco_gret_prefill_chunkwise(z, z, z, lg, 16.0, z, S)
    torch.cuda.synchronize()
    assert bool((S == 0.5).all())


# ---------------------------------------------------------------- gRet decode

@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_gret_decode_steps(Y, dtype, d):
    """Several recurrent steps from a random state match the oracle."""
    import torch
    B, H, steps = 2, 3, 5
    host, dev = gret_inputs(5, B, steps, H, d, dtype, logit_mean=1.0)
    S0 = synth.normal(SEED, sid(5, 0, synth.T_S0), (B, H, d, d), "f32", std=0.2).astype(np.float64)
    S = dev_f32(S0)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    outs = []
    for t in range(steps):
        o = torch.empty(B, H, d, dtype=tdt, device="cuda")
        Y.yoco_gret_decode_step(*(x[:, t].contiguous() for x in dev), 16.0, S, o)
        outs.append(host_f64(o))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    o_gpu = np.stack(outs, axis=1)
    if dtype == "f32":
        assert max_abs(o_gpu, o_ref) <= FP32_MAX_ABS
        assert max_abs(S.cpu().numpy(), S_ref) <= FP32_MAX_ABS
    else:
        assert rel_l2(o_gpu, o_ref) <= BF16_REL_L2
        assert rel_l2(S.cpu().numpy(), S_ref) <= BF16_REL_L2


# ------------------------------------------------------------- shared KV

def test_kv_append_bit_exact(Y):
    """+-1 rows (rms 1), eps 0 and dyadic weights make every sum exact: the
    cache must equal the oracle's bit for bit, and only the new slots change."""
    import torch
    B, dm, Hkv, d, cap = 2, 256, 2, 64, 16
    rng_bits = np.random.default_rng(0).integers(0, 0x7F7F, size=(B, Hkv, cap, d)).astype(np.uint16)
    cache = Y.KVCache(B, Hkv, d, cap, k=dev_bf16(rng_bits), v=dev_bf16(rng_bits[::-1].copy()))
    cache.set_length(3)
    kref, vref = rng_bits.copy(), rng_bits[::-1].copy()
    Wk = synth.dyadic(SEED, sid(20, 0, synth.T_WK), (dm, Hkv * d))
    Wv = synth.dyadic(SEED, sid(20, 0, synth.T_WV), (dm, Hkv * d))
    Wkd, Wvd = dev_bf16(synth.f64_to_bf16_bits(Wk)), dev_bf16(synth.f64_to_bf16_bits(Wv))
    length = 3
    for step, T in enumerate((5, 4)):
        M = synth.signs(SEED, sid(20, 0, synth.T_M, step), (B, T, dm))
        Y.yoco_shared_kv_project_append(dev_bf16(synth.f64_to_bf16_bits(M)), Wkd, Wvd, cache, eps=0.0)
        kref = oracle.kv_append_bf16(kref, oracle.rmsnorm_proj(M, Wk, 0.0), length)
        vref = oracle.kv_append_bf16(vref, oracle.rmsnorm_proj(M, Wv, 0.0), length)
        length += T
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(cache.k), kref)
        assert np.array_equal(host_bits(cache.v), vref)
        assert cache.length == length and int(cache.len_dev[0]) == length and int(cache.len_dev[1]) == 0


@pytest.mark.parametrize("B,T,dm,Hkv,d,gain", [(1, 1, 3072, 8, 128, False), (2, 2, 3072, 8, 128, True),
                                                (3, 1, 3072, 8, 128, False), (1, 3, 256, 1, 64, False),
                                                (4, 1, 1000, 2, 128, True)])
def test_kv_append_decode_rows_bit_exact(Y, B, T, dm, Hkv, d, gain):
    """The few-row (decode) projection: at most four input rows, each CTA one
    16-column strip of [W_K | W_V] over all of d_model.  +-1 rows, eps 0, dyadic
    weights (and a gain of powers of two) make every sum exact, so the slots
    must equal the oracle's bit for bit, twice in a row, and nothing else in the
    cache may change."""
    import torch
    cap = 2 * T + 3
    rng_bits = np.random.default_rng(1).integers(0, 0x7F7F, size=(B, Hkv, cap, d)).astype(np.uint16)
    cache = Y.KVCache(B, Hkv, d, cap, k=dev_bf16(rng_bits), v=dev_bf16(rng_bits[::-1].copy()))
    cache.set_length(1)
    kref, vref = rng_bits.copy(), rng_bits[::-1].copy()
    Wk = synth.dyadic(SEED, sid(21, 0, synth.T_WK), (dm, Hkv * d))
    Wv = synth.dyadic(SEED, sid(21, 0, synth.T_WV), (dm, Hkv * d))
    Wkd, Wvd = dev_bf16(synth.f64_to_bf16_bits(Wk)), dev_bf16(synth.f64_to_bf16_bits(Wv))
    g = None
    if gain:
        g = 2.0 ** (np.arange(dm) % 3 - 1)  # 0.5, 1, 2, ...
    length = 1
    for step in range(2):
        M = synth.signs(SEED, sid(21, 0, synth.T_M, step), (B, T, dm))
        gd = None if g is None else dev_bf16(synth.f64_to_bf16_bits(g))
        Y.yoco_shared_kv_project_append(dev_bf16(synth.f64_to_bf16_bits(M)), Wkd, Wvd, cache, eps=0.0, rms_w=gd)
        kref = oracle.kv_append_bf16(kref, oracle.rmsnorm_proj(M, Wk, 0.0, g=g), length)
        vref = oracle.kv_append_bf16(vref, oracle.rmsnorm_proj(M, Wv, 0.0, g=g), length)
        length += T
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(cache.k), kref)
        assert np.array_equal(host_bits(cache.v), vref)
        assert cache.length == length and int(cache.len_dev[0]) == length and int(cache.len_dev[1]) == 0


def test_kv_append_tensor_core_bit_exact(Y):
    """The tensor-core projection (>= 128 rows, Hkv*d a multiple of 256): exact
    inputs give a bit-identical cache, appended after existing slots."""
    import torch
    B, T, dm, Hkv, d, cap, length = 2, 150, 512, 8, 128, 170, 7
    rng_bits = np.random.default_rng(1).integers(0, 0x7F7F, size=(B, Hkv, cap, d)).astype(np.uint16)
    cache = Y.KVCache(B, Hkv, d, cap, k=dev_bf16(rng_bits), v=dev_bf16(rng_bits.copy()))
    cache.set_length(length)
    Wk = synth.dyadic(SEED, sid(21, 0, synth.T_WK), (dm, Hkv * d))
    Wv = synth.dyadic(SEED, sid(21, 0, synth.T_WV), (dm, Hkv * d))
    M = synth.signs(SEED, sid(21, 0, synth.T_M), (B, T, dm))
    Y.yoco_shared_kv_project_append(dev_bf16(synth.f64_to_bf16_bits(M)), dev_bf16(synth.f64_to_bf16_bits(Wk)),
                                    dev_bf16(synth.f64_to_bf16_bits(Wv)), cache, eps=0.0)
    torch.cuda.synchronize()
    kref = oracle.kv_append_bf16(rng_bits, oracle.rmsnorm_proj(M, Wk, 0.0), length)
    vref = oracle.kv_append_bf16(rng_bits, oracle.rmsnorm_proj(M, Wv, 0.0), length)
    assert np.array_equal(host_bits(cache.k), kref)
    assert np.array_equal(host_bits(cache.v), vref)
    assert cache.length == length + T and int(cache.len_dev[0]) == length + T and int(cache.len_dev[1]) == 0


def test_kv_append_tensor_core_3b_width(Y):
    """d_model 3072 -> 8 x 128 (the 3B shape) on random data, ragged row count."""
    import torch
    B, T, dm, Hkv, d = 2, 150, 3072, 8, 128
    M, Md = gen(SEED, sid(22, 0, synth.T_M), (B, T, dm), "bf16")
    Wk, Wkd = gen(SEED, sid(22, 0, synth.T_WK), (dm, Hkv * d), "bf16", std=0.02)
    Wv, Wvd = gen(SEED, sid(22, 0, synth.T_WV), (dm, Hkv * d), "bf16", std=0.02)
    cache = Y.KVCache(B, Hkv, d, T)
    ws = torch.empty(Y.lib.yoco_shared_kv_workspace_size(B, T, dm, __import__("ctypes").byref(cache.c)),
                     dtype=torch.uint8, device="cuda")
    Y.yoco_shared_kv_project_append(Md, Wkd, Wvd, cache, eps=1e-6, workspace=ws)
    Y.yoco_workspace_status(ws)
    kref = oracle.rmsnorm_proj(M, Wk, 1e-6).reshape(B, T, Hkv, d).transpose(0, 2, 1, 3)
    vref = oracle.rmsnorm_proj(M, Wv, 1e-6).reshape(B, T, Hkv, d).transpose(0, 2, 1, 3)
    assert rel_l2(host_f64(cache.k), kref) <= BF16_REL_L2
    assert rel_l2(host_f64(cache.v), vref) <= BF16_REL_L2


def test_kv_append_tensor_core_many_tiles_per_pair(Y):
    """12040 rows at the 3B width: 48 row blocks x 8 column tiles, so each CTA pair
    runs about five tiles and both factor buffers of the in-GEMM row norm, and
    both parities of their barriers, are used several times; the last row block
    holds 8 rows (its odd CTA none).  Against the oracle on every 7th row and the
    last 40 (both CTAs of every row block), per tensor and per row block of each
    kv head."""
    import torch
    B, T, dm, Hkv, d = 1, 12040, 3072, 8, 128
    M, Md = gen(SEED, sid(23, 0, synth.T_M), (B, T, dm), "bf16")
    Wk, Wkd = gen(SEED, sid(23, 0, synth.T_WK), (dm, Hkv * d), "bf16", std=0.02)
    Wv, Wvd = gen(SEED, sid(23, 0, synth.T_WV), (dm, Hkv * d), "bf16", std=0.02)
    cache = Y.KVCache(B, Hkv, d, T)
    ws = torch.empty(Y.lib.yoco_shared_kv_workspace_size(B, T, dm, ctypes.byref(cache.c)), dtype=torch.uint8,
                     device="cuda")
    Y.yoco_shared_kv_project_append(Md, Wkd, Wvd, cache, eps=1e-6, workspace=ws)
    Y.yoco_workspace_status(ws)
    assert cache.length == T and int(cache.len_dev[0]) == T and int(cache.len_dev[1]) == 0
    rows = np.array(sorted(set(range(0, T, 7)) | set(range(T - 40, T))))
    blocks = rows // 256
    for W, got in ((Wk, cache.k), (Wv, cache.v)):
        ref = oracle.rmsnorm_proj(M[0, rows], W, 1e-6).reshape(len(rows), Hkv, d)
        g = host_f64(got)[0][:, rows].transpose(1, 0, 2)  # [rows, Hkv, d]
        assert rel_l2(g, ref) <= BF16_REL_L2
        for blk in np.unique(blocks):
            sel = blocks == blk
            for h in range(Hkv):
                assert rel_l2(g[sel, h], ref[sel, h]) <= BLOCK_REL_L2, (blk, h)


def test_kv_append_fp32_and_gain(Y):
    """fp32 cache (tiny config: dm 128 -> one 64-wide head), with an RMSNorm gain."""
    import torch
    B, T, dm, Hkv, d = 1, 256, 128, 1, 64
    M, Md = gen(SEED, sid(1, 0, synth.T_M), (B, T, dm), "f32")
    Wk, Wkd = gen(SEED, sid(1, 0, synth.T_WK), (dm, Hkv * d), "f32", std=0.02)
    Wv, Wvd = gen(SEED, sid(1, 0, synth.T_WV), (dm, Hkv * d), "f32", std=0.02)
    g, gd = gen(SEED, sid(1, 0, synth.T_RMSW), (dm,), "f32", mean=1.0, std=0.1)
    cache = Y.KVCache(B, Hkv, d, T + 4, dtype=torch.float32)
    Y.yoco_shared_kv_project_append(Md, Wkd, Wvd, cache, eps=1e-6, rms_w=gd)
    torch.cuda.synchronize()
    kref = oracle.rmsnorm_proj(M, Wk, 1e-6, g=g).reshape(B, T, Hkv, d).transpose(0, 2, 1, 3)
    vref = oracle.rmsnorm_proj(M, Wv, 1e-6, g=g).reshape(B, T, Hkv, d).transpose(0, 2, 1, 3)
    assert max_abs(host_f64(cache.k)[:, :, :T], kref) <= FP32_MAX_ABS
    assert max_abs(host_f64(cache.v)[:, :, :T], vref) <= FP32_MAX_ABS
    assert bool((cache.k[:, :, T:] == 0).all())


def test_kv_append_capacity_error_writes_nothing(Y):
    import torch
    B, dm, Hkv, d, cap = 1, 64, 1, 64, 12
    cache = Y.KVCache(B, Hkv, d, cap)
    cache.set_length(10)
    before = cache.k.clone()
    M = torch.ones(B, 3, dm, dtype=torch.bfloat16, device="cuda")
    W = torch.ones(dm, Hkv * d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Y.YocoError) as e:
        Y.yoco_shared_kv_project_append(M, W, W, cache)
    assert e.value.status == Y.YOCO_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.equal(before, cache.k) and cache.length == 10 and int(cache.len_dev[0]) == 10


# ----------------------------------------------------------- cross attention

def fill_cache(Y, B, Hkv, d, cap, length, dtype, cfg):
    import torch
    K, Kd = gen(SEED, sid(cfg, 0, synth.T_CACHE_K), (B, Hkv, cap, d), dtype)
    V, Vd = gen(SEED, sid(cfg, 0, synth.T_CACHE_V), (B, Hkv, cap, d), dtype)
    cache = Y.KVCache(B, Hkv, d, cap, dtype=Kd.dtype, k=Kd, v=Vd)
    cache.set_length(length)
    return K, V, cache


def test_cross_attn_prefill_fp32_full_causal(Y):
    """Tiny config: 256 causal rows, 2 query heads on one 64-wide kv head."""
    import torch
    B, Hq, Hkv, d, N = 1, 2, 1, 64, 256
    K, V, cache = fill_cache(Y, B, Hkv, d, N, N, "f32", 1)
    Q, Qd = gen(SEED, sid(1, 0, synth.T_QX), (B, N, Hq, d), "f32")
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd, cache, 0, O)
    torch.cuda.synchronize()
    O_ref = oracle.cross_attn(Q, K, V, 0, d ** -0.5)
    assert max_abs(host_f64(O), O_ref) <= FP32_MAX_ABS


@pytest.mark.parametrize("T,p0", [(1, 999), (37, 100), (130, 0)])
def test_cross_attn_prefill_bf16_gqa(Y, T, p0):
    import torch
    B, Hq, Hkv, d = 2, 24, 8, 128
    length = p0 + T + 5
    K, V, cache = fill_cache(Y, B, Hkv, d, length + 3, length, "bf16", 3)
    Q, Qd = gen(SEED, sid(3, 1, synth.T_QX), (B, T, Hq, d), "bf16")
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd, cache, p0, O)
    torch.cuda.synchronize()
    O_ref = oracle.cross_attn(Q, K, V, p0, d ** -0.5)
    assert rel_l2(host_f64(O), O_ref) <= BF16_REL_L2


@pytest.mark.parametrize("B,T,p0", [(2, 300, 77), (1, 64, 0), (1, 2048, 0), (1, 257, 4000)])
def test_cross_attn_prefill_many_rows(Y, B, T, p0):
    """Many-row prefill (128-row query tiles): ragged last tile, a diagonal that
    does not start on a tile boundary, a block of exactly 64 rows, 2048 causal
    rows, rows far into a long cache."""
    import torch
    Hq, Hkv, d = 24, 8, 128
    length = p0 + T
    K, V, cache = fill_cache(Y, B, Hkv, d, length + 129, length, "bf16", 34)
    Q, Qd = gen(SEED, sid(34, 1, synth.T_QX), (B, T, Hq, d), "bf16")
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd, cache, p0, O)
    torch.cuda.synchronize()
    O_ref = oracle.cross_attn(Q, K, V, p0, d ** -0.5)
    assert rel_l2(host_f64(O), O_ref) <= BF16_REL_L2


def test_cross_attn_prefill_growing_scores(Y):
    """Keys whose scale grows along the sequence (x1 .. x8) push each row's
    running maximum up tile after tile, so the output is rescaled many times."""
    import torch
    B, T, Hq, Hkv, d = 1, 1024, 24, 8, 128
    Kb = synth.normal_f64(SEED, sid(35, 0, synth.T_CACHE_K), B * Hkv * T * d).reshape(B, Hkv, T, d)
    Kb *= (1.0 + 7.0 * np.arange(T) / T)[None, None, :, None]
    kbits = synth.f64_to_bf16_bits(Kb)
    K = synth.bf16_bits_to_f32(kbits).astype(np.float64)
    V, Vd = gen(SEED, sid(35, 0, synth.T_CACHE_V), (B, Hkv, T, d), "bf16")
    cache = Y.KVCache(B, Hkv, d, T, dtype=Vd.dtype, k=dev_bf16(kbits), v=Vd)
    cache.set_length(T)
    Q, Qd = gen(SEED, sid(35, 1, synth.T_QX), (B, T, Hq, d), "bf16", std=2.0)
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd, cache, 0, O)
    torch.cuda.synchronize()
    O_ref = oracle.cross_attn(Q, K, V, 0, d ** -0.5)
    assert rel_l2(host_f64(O), O_ref) <= BF16_REL_L2


def test_cross_attn_decode_split_invariance(Y):
    """The decode result does not depend on the number of key splits."""
    import torch
    B, Hq, Hkv, d, length = 2, 24, 8, 128, 3001
    K, V, cache = fill_cache(Y, B, Hkv, d, length, length, "bf16", 5)
    Q, Qd = gen(SEED, sid(5, 2, synth.T_QX), (B, Hq, d), "bf16")
    O_ref = oracle.cross_attn(Q[:, None], K, V, length - 1, d ** -0.5)[:, 0]
    results = []
    for splits in (1, 2, 7, 0):
        O = torch.empty_like(Qd)
        Y.yoco_cross_attn_decode(Qd, cache, O, num_splits=splits)
        torch.cuda.synchronize()
        results.append(host_f64(O))
        assert rel_l2(results[-1], O_ref) <= BF16_REL_L2
    for r in results[1:]:
        assert rel_l2(r, results[0]) <= 1e-2


@pytest.mark.parametrize("dtype,d,length,splits", [("bf16", 128, 40000, 300), ("f32", 64, 9000, 100)])
def test_cross_attn_decode_more_splits_than_merge_threads(Y, dtype, d, length, splits):
    """The log-sum-exp merge runs d threads per query row; with more splits than
    threads each thread gathers several splits' maxima and sums (tensor-core and
    CUDA-core split kernels)."""
    import torch
    B, Hq, Hkv = 1, 6, 2
    K, V, cache = fill_cache(Y, B, Hkv, d, length, length, dtype, 36)
    Q, Qd = gen(SEED, sid(36, 2, synth.T_QX), (B, Hq, d), dtype)
    O_ref = oracle.cross_attn(Q[:, None], K, V, length - 1, d ** -0.5)[:, 0]
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_decode(Qd, cache, O, num_splits=splits)
    torch.cuda.synchronize()
    if dtype == "bf16":
        assert rel_l2(host_f64(O), O_ref) <= BF16_REL_L2
    else:
        assert max_abs(host_f64(O), O_ref) <= FP32_MAX_ABS


def test_cross_attn_decode_garbage_workspace_twice(Y):
    """Decode needs no clean workspace: one full of arbitrary bytes (status
    word aside) gives the oracle's result, and so does a second call on it."""
    import torch
    B, Hq, Hkv, d, length = 1, 24, 8, 128, 5000
    K, V, cache = fill_cache(Y, B, Hkv, d, length, length, "bf16", 32)
    Q, Qd = gen(SEED, sid(32, 2, synth.T_QX), (B, Hq, d), "bf16")
    O_ref = oracle.cross_attn(Q[:, None], K, V, length - 1, d ** -0.5)[:, 0]
    for splits in (0, 5):
        n = Y.yoco_cross_attn_workspace_size(B, Hq, 1, cache, splits)
        ws = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
        ws[:256] = 0  # the status word of a fresh workspace
        for _ in range(2):
            O = torch.empty_like(Qd)
            Y.yoco_cross_attn_decode(Qd, cache, O, num_splits=splits, workspace=ws)
            torch.cuda.synchronize()
            assert rel_l2(host_f64(O), O_ref) <= BF16_REL_L2
        Y.yoco_workspace_status(ws)


def test_early_exit_matches_full_prefill_last_row(Y):
    """Early exit (paper Fig. 3): the last prompt row computed alone equals the
    last row of the full causal prefill."""
    import torch
    B, Hq, Hkv, d, N = 1, 6, 2, 64, 300
    K, V, cache = fill_cache(Y, B, Hkv, d, N, N, "f32", 6)
    Q, Qd = gen(SEED, sid(6, 0, synth.T_QX), (B, N, Hq, d), "f32")
    O_full = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd, cache, 0, O_full)
    O_last = torch.empty(B, 1, Hq, d, device="cuda")
    Y.yoco_cross_attn_prefill(Qd[:, -1:].contiguous(), cache, N - 1, O_last)
    torch.cuda.synchronize()
    assert max_abs(host_f64(O_last)[:, 0], host_f64(O_full)[:, -1]) <= FP32_MAX_ABS


# --------------------------------------------------- tiny config end to end

def test_tiny_config_pipeline_fp32(Y):
    """The whole tiny fp32 configuration: gRet prefill (2 heads x 64, N=256),
    shared KV from a 128-wide M, 2 cross layers x 2 query heads over all 256
    rows, then 16 decode steps (recurrent step, append, 2 cross layers)."""
    import torch
    B, N, H, d, dm, Hkv, Hq, L, steps = 1, 256, 2, 64, 128, 1, 2, 2, 16
    host, dev = gret_inputs(1, B, N, H, d, "f32", qk_std=1 / 8)
    o, S = run_prefill(Y, dev, B, N, H, d, "f32", chunk=64)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0)
    assert max_abs(o, o_ref) <= FP32_MAX_ABS
    M, Md = gen(SEED, sid(1, 0, synth.T_M), (B, N + steps, dm), "f32")
    Wk, Wkd = gen(SEED, sid(1, 0, synth.T_WK), (dm, d), "f32", std=0.02)
    Wv, Wvd = gen(SEED, sid(1, 0, synth.T_WV), (dm, d), "f32", std=0.02)
    cache = Y.KVCache(B, Hkv, d, N + steps, dtype=torch.float32)
    Y.yoco_shared_kv_project_append(Md[:, :N].contiguous(), Wkd, Wvd, cache, eps=1e-6)
    Kall = oracle.rmsnorm_proj(M, Wk, 1e-6).reshape(B, N + steps, Hkv, d).transpose(0, 2, 1, 3)
    Vall = oracle.rmsnorm_proj(M, Wv, 1e-6).reshape(B, N + steps, Hkv, d).transpose(0, 2, 1, 3)
    for layer in range(L):
        Q, Qd = gen(SEED, sid(1, layer, synth.T_QX), (B, N, Hq, d), "f32")
        O = torch.empty_like(Qd)
        Y.yoco_cross_attn_prefill(Qd, cache, 0, O)
        torch.cuda.synchronize()
        assert max_abs(host_f64(O), oracle.cross_attn(Q, Kall, Vall, 0, d ** -0.5)) <= FP32_MAX_ABS
    Sd = dev_f32(S)
    S_host = S_ref
    for t in range(steps):
        xs, xd = gret_inputs(100 + t, B, 1, H, d, "f32", qk_std=1 / 8)
        od = torch.empty(B, H, d, device="cuda")
        Y.yoco_gret_decode_step(*(x[:, 0].contiguous() for x in xd), 16.0, Sd, od)
        o1, S_host = oracle.gret_recurrent(*xs, 16.0, S0=S_host)
        Y.yoco_shared_kv_project_append(Md[:, N + t:N + t + 1].contiguous(), Wkd, Wvd, cache, eps=1e-6)
        torch.cuda.synchronize()
        assert max_abs(host_f64(od), o1[:, 0]) <= FP32_MAX_ABS
        for layer in range(L):
            Q, Qd = gen(SEED, sid(1, layer, synth.T_QX, 1 + t), (B, Hq, d), "f32")
            O = torch.empty_like(Qd)
            Y.yoco_cross_attn_decode(Qd, cache, O)
            torch.cuda.synchronize()
            O_ref = oracle.cross_attn(Q[:, None], Kall, Vall, N + t, d ** -0.5)[:, 0]
            assert max_abs(host_f64(O), O_ref) <= FP32_MAX_ABS
    assert max_abs(Sd.cpu().numpy(), S_host) <= FP32_MAX_ABS


def test_device_generator_matches_host(Y):
    """The device copy of the input generator reproduces the host one."""
    import torch
    t = torch.empty(100003, dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(t, SEED, sid(2, 3, synth.T_Q), std=0.25, start=17)
    host = synth.normal(SEED, sid(2, 3, synth.T_Q), (100003,), "bf16", std=0.25, start=17)
    assert np.mean(host_bits(t) != host) < 1e-4
    f = torch.empty(5000, dtype=torch.float32, device="cuda")
    synth.fill_normal_(f, SEED, 99, mean=2.0)
    assert np.max(np.abs(f.cpu().numpy() - synth.normal(SEED, 99, (5000,), "f32", mean=2.0))) <= 1e-6


# ------------------------------------------------ sliding-window self-decoder

def swa_inputs(cfg, B, N, Hq, Hkv, d):
    q, qd = gen(SEED, sid(cfg, 0, synth.T_Q), (B, N, Hq, d), "bf16")
    k, kd = gen(SEED, sid(cfg, 0, synth.T_K), (B, N, Hkv, d), "bf16")
    v, vd = gen(SEED, sid(cfg, 0, synth.T_V), (B, N, Hkv, d), "bf16")
    return (q, k, v), (qd, kd, vd)


@pytest.mark.parametrize("B,N,Hq,Hkv,window", [(1, 3000, 8, 8, 1024), (2, 777, 24, 8, 200), (1, 500, 4, 2, 4096),
                                                (1, 130, 6, 3, 1)])
def test_swa_prefill(Y, B, N, Hq, Hkv, window):
    """Sliding-window prefill against the window-mask oracle: multi-head and
    grouped heads, windows shorter than the sequence (a multiple of the key
    tile and not), longer than it, and a window of one key."""
    import torch
    d = 128
    (q, k, v), (qd, kd, vd) = swa_inputs(40, B, N, Hq, Hkv, d)
    ring = Y.SwaRing(B, Hkv, d, window)
    o = torch.empty_like(qd)
    Y.yoco_swa_prefill(qd, kd, vd, ring, o)
    torch.cuda.synchronize()
    o_ref = oracle.swa_attn(q, k, v, window, d ** -0.5)
    assert rel_l2(host_f64(o), o_ref) <= BF16_REL_L2
    assert ring.pos == N
    # the ring holds the last min(N, window) tokens at slot position % window
    for p in range(max(0, N - window), N, max(1, min(N, window) // 7)):
        assert np.array_equal(host_bits(ring.k[:, :, p % window]), host_bits(kd[:, p]))
        assert np.array_equal(host_bits(ring.v[:, :, p % window]), host_bits(vd[:, p]))


@pytest.mark.parametrize("window", [256, 100])
def test_swa_decode_continues_prefill(Y, window):
    """Prefill 300 tokens, then 40 decode steps through the ring (window 100
    wraps it several times): every generated token's output equals the oracle
    over the whole sequence with the window mask."""
    import torch
    B, Hq, Hkv, d, N0, steps = 2, 6, 2, 128, 300, 40
    N = N0 + steps
    (q, k, v), (qd, kd, vd) = swa_inputs(41, B, N, Hq, Hkv, d)
    ring = Y.SwaRing(B, Hkv, d, window)
    o = torch.empty_like(qd)
    Y.yoco_swa_prefill(qd[:, :N0].contiguous(), kd[:, :N0].contiguous(), vd[:, :N0].contiguous(), ring,
                       o[:, :N0].contiguous())
    outs = []
    for t in range(N0, N):
        ot = torch.empty(B, Hq, d, dtype=qd.dtype, device="cuda")
        Y.yoco_swa_decode(qd[:, t].contiguous(), kd[:, t].contiguous(), vd[:, t].contiguous(), ring, ot)
        outs.append(ot)
    torch.cuda.synchronize()
    assert ring.pos == N
    o_ref = oracle.swa_attn(q, k, v, window, d ** -0.5)
    got = np.stack([host_f64(x) for x in outs], axis=1)
    assert rel_l2(got, o_ref[:, N0:]) <= BF16_REL_L2


def test_swa_decode_fp32_from_empty_ring(Y):
    """fp32, head size 64: decode from the first token on (no prefill)."""
    import torch
    B, Hq, Hkv, d, N, window = 1, 4, 4, 64, 50, 16
    q, qd = gen(SEED, sid(42, 0, synth.T_Q), (B, N, Hq, d), "f32")
    k, kd = gen(SEED, sid(42, 0, synth.T_K), (B, N, Hkv, d), "f32")
    v, vd = gen(SEED, sid(42, 0, synth.T_V), (B, N, Hkv, d), "f32")
    ring = Y.SwaRing(B, Hkv, d, window, dtype=torch.float32)
    outs = []
    for t in range(N):
        ot = torch.empty(B, Hq, d, device="cuda")
        Y.yoco_swa_decode(qd[:, t].contiguous(), kd[:, t].contiguous(), vd[:, t].contiguous(), ring, ot)
        outs.append(ot)
    torch.cuda.synchronize()
    got = np.stack([host_f64(x) for x in outs], axis=1)
    assert max_abs(got, oracle.swa_attn(q, k, v, window, d ** -0.5)) <= FP32_MAX_ABS


# --------------------------------------------- gated retention output (Eq. 7)

@pytest.mark.parametrize("dtype,d,affine,inplace", [("bf16", 128, True, False), ("f32", 64, False, True),
                                                    ("bf16", 64, False, True), ("f32", 128, True, False)])
def test_group_norm_gate(Y, dtype, d, affine, inplace):
    """swish(gate) * GroupNorm_h(o) over 777 tokens x 6 heads: bf16 within the
    relative-L2 bound, fp32 within the max-abs bound; with and without the
    per-channel affine; in place (z = o)."""
    import torch
    B, N, H = 2, 777, 6
    o, od = gen(SEED, sid(50, 0, synth.T_V), (B, N, H, d), dtype, mean=0.3, std=2.0)
    g, gd = gen(SEED, sid(50, 0, synth.T_Q), (B, N, H, d), dtype)
    w = b = wd = bd = None
    if affine:
        w = synth.normal(SEED, sid(50, 1, synth.T_K), (H * d,), "f32", mean=1.0, std=0.2)
        b = synth.normal(SEED, sid(50, 2, synth.T_K), (H * d,), "f32", std=0.2)
        wd, bd = dev_f32(w), dev_f32(b)
    z = od if inplace else torch.empty_like(od)
    Y.yoco_gret_group_norm_gate(od, gd, z, eps=1e-5, gn_weight=wd, gn_bias=bd)
    torch.cuda.synchronize()
    z_ref = oracle.group_norm_gate(o, g, 1e-5, w, b)
    if dtype == "f32":
        assert max_abs(host_f64(z), z_ref) <= FP32_MAX_ABS
    else:
        assert rel_l2(host_f64(z), z_ref) <= BF16_REL_L2


@pytest.mark.parametrize("B,N,H,d,dtype,affine,with_state", [
    (1, 8192 + 77, 24, 128, "bf16", True, True),    # tensor cores, 6 segments per head
    (1, 6403, 9, 128, "bf16", True, True),           # tensor cores, 13 segments per head
    (2, 300, 8, 128, "bf16", False, False),          # tensor cores, 3 one-chunk segments
    (3, 200, 80, 128, "bf16", True, False),          # tensor cores, one segment (B*H >= SMs)
    (1, 1000, 3, 64, "f32", True, True),             # CUDA cores, then Eq. 7 in place
])
def test_gret_prefill_gn_gate_fused(Y, B, N, H, d, dtype, affine, with_state):
    """The chunkwise prefill with Eq. 7's output fused (z = swish(gate) (.)
    GroupNorm_h(o)) against the oracle's recurrent form followed by its
    group_norm_gate, and the final state; the bf16 result also against the two
    separate calls."""
    import torch
    host, dev = gret_inputs(46, B, N, H, d, dtype, logit_mean=2.0)
    gh, gd = gen(SEED, sid(46, 1, synth.T_QX), (B, N, H, d), dtype)
    w = b = wd = bd = None
    if affine:
        w = 1.0 + 0.25 * synth.normal(SEED, sid(46, 2, synth.T_QX), (H * d,), "f32").astype(np.float64)
        b = 0.1 * synth.normal(SEED, sid(46, 3, synth.T_QX), (H * d,), "f32").astype(np.float64)
        wd, bd = dev_f32(w), dev_f32(b)
    S0 = None
    if with_state:
        S0 = synth.normal(SEED, sid(46, 4, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    qd, kd, vd, lgd = dev
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    z = torch.full((B, N, H, d), float("nan"), dtype=tdt, device="cuda")
    S = torch.zeros(B, H, d, d, device="cuda") if S0 is None else dev_f32(S0)
    Y.yoco_gret_prefill_chunkwise_gn_gate(qd, kd, vd, lgd, 16.0, gd, z, S, eps=1e-5, gn_weight=wd, gn_bias=bd)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    z_ref = oracle.group_norm_gate(o_ref, gh, 1e-5, w, b)
    zg = host_f64(z)
    if dtype == "f32":
        assert max_abs(zg, z_ref) <= FP32_MAX_ABS
        assert max_abs(S.cpu().numpy(), S_ref) <= FP32_MAX_ABS
        return
    assert rel_l2(zg, z_ref) <= BF16_REL_L2
    for bb in range(B):
        for h in range(H):
            assert worst_block_rel_l2(zg[bb, :, h], z_ref[bb, :, h], 128) <= BLOCK_REL_L2, (bb, h)
    assert rel_l2(S.cpu().numpy(), S_ref) <= BF16_REL_L2
    # the two separate calls (o rounded to bf16 between them) agree to bf16 rounding
    o2 = torch.empty_like(vd)
    S2 = torch.zeros(B, H, d, d, device="cuda") if S0 is None else dev_f32(S0)
    Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o2, S2)
    z2 = torch.empty_like(o2)
    Y.yoco_gret_group_norm_gate(o2, gd, z2, eps=1e-5, gn_weight=wd, gn_bias=bd)
    torch.cuda.synchronize()
    assert rel_l2(zg, host_f64(z2)) <= BF16_REL_L2


def test_group_norm_gate_decode_row(Y):
    """A decode step's output [B, H, d] goes through the same call (N = 1)."""
    import torch
    B, H, d = 3, 24, 128
    o, od = gen(SEED, sid(51, 0, synth.T_V), (B, H, d), "bf16")
    g, gd = gen(SEED, sid(51, 0, synth.T_Q), (B, H, d), "bf16")
    z = torch.empty_like(od)
    Y.yoco_gret_group_norm_gate(od, gd, z)
    torch.cuda.synchronize()
    z_ref = oracle.group_norm_gate(o[:, None], g[:, None], 1e-5)[:, 0]
    assert rel_l2(host_f64(z), z_ref) <= BF16_REL_L2


@pytest.mark.parametrize("dtype,d,affine", [("bf16", 128, False), ("bf16", 128, True), ("f32", 64, True),
                                            ("f32", 128, False)])
def test_gret_decode_step_gn_gate_fused(Y, dtype, d, affine):
    """Three recurrent steps with GroupNorm_h + swish gate fused (the dv/32 CTAs of a
    head as one cluster): each step's z equals the oracle's step output passed
    through the oracle's group_norm_gate, and the carried state the oracle's."""
    import torch
    B, H, steps = 2, 24, 3
    host, dev = gret_inputs(52, B, steps, H, d, dtype, logit_mean=1.0)
    S0 = synth.normal(SEED, sid(52, 0, synth.T_S0), (B, H, d, d), "f32", std=0.2).astype(np.float64)
    S = dev_f32(S0)
    g, gd = gen(SEED, sid(52, 1, synth.T_Q), (B, steps, H, d), dtype)
    w = b = wd = bd = None
    if affine:
        w = synth.normal(SEED, sid(52, 1, synth.T_K), (H * d,), "f32", mean=1.0, std=0.2)
        b = synth.normal(SEED, sid(52, 2, synth.T_K), (H * d,), "f32", std=0.2)
        wd, bd = dev_f32(w), dev_f32(b)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    zs = []
    for t in range(steps):
        z = torch.empty(B, H, d, dtype=tdt, device="cuda")
        Y.yoco_gret_decode_step_gn_gate(*(x[:, t].contiguous() for x in dev), 16.0, S, gd[:, t].contiguous(), z,
                                        eps=1e-5, gn_weight=wd, gn_bias=bd)
        zs.append(host_f64(z))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    z_ref = oracle.group_norm_gate(o_ref, g, 1e-5, w, b)
    z_gpu = np.stack(zs, axis=1)
    if dtype == "f32":
        assert max_abs(z_gpu, z_ref) <= FP32_MAX_ABS
        assert max_abs(S.cpu().numpy(), S_ref) <= FP32_MAX_ABS
    else:
        assert rel_l2(z_gpu, z_ref) <= BF16_REL_L2
        assert rel_l2(S.cpu().numpy(), S_ref) <= BF16_REL_L2


def test_gret_decode_step_gn_gate_matches_the_two_calls(Y):
    """The fused call equals the plain step followed by yoco_gret_group_norm_gate
    on its fp32 output (fp32 throughout, so only the variance formula differs)."""
    import torch
    B, H, d = 1, 8, 128
    host, dev = gret_inputs(53, B, 1, H, d, "f32", logit_mean=1.0)
    S0 = synth.normal(SEED, sid(53, 0, synth.T_S0), (B, H, d, d), "f32", std=0.2)
    g, gd = gen(SEED, sid(53, 1, synth.T_Q), (B, H, d), "f32")
    q, k, v, lg = (x[:, 0].contiguous() for x in dev)
    S1, S2 = dev_f32(S0), dev_f32(S0)
    z1 = torch.empty(B, H, d, device="cuda")
    Y.yoco_gret_decode_step_gn_gate(q, k, v, lg, 16.0, S1, gd, z1)
    o = torch.empty(B, H, d, device="cuda")
    Y.yoco_gret_decode_step(q, k, v, lg, 16.0, S2, o)
    z2 = torch.empty_like(o)
    Y.yoco_gret_group_norm_gate(o, gd, z2)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2)
    assert max_abs(host_f64(z1), host_f64(z2)) <= FP32_MAX_ABS


# ------------------------------------------------- rotary position encoding

@pytest.mark.parametrize("dtype,d,pos0,base", [("bf16", 128, 0, 10000.0), ("bf16", 128, 1000000, 8e7),
                                               ("f32", 64, 77, 10000.0), ("f32", 128, 262000, 5e6)])
def test_rope_apply(Y, dtype, d, pos0, base):
    """In-place rotation of token-major q/k against the oracle, at positions up
    to one million with the 1M-context base: bf16 within the relative-L2 bound,
    fp32 within the max-abs bound."""
    import torch
    B, N, H = 2, 300, 3
    x, xd = gen(SEED, sid(60, 0, synth.T_Q), (B, N, H, d), dtype)
    Y.yoco_rope_apply(xd, base, pos0=pos0)
    torch.cuda.synchronize()
    ref = oracle.rope(x, (pos0 + np.arange(N))[None, :, None], base)
    if dtype == "f32":
        assert max_abs(host_f64(xd), ref) <= FP32_MAX_ABS
    else:
        assert rel_l2(host_f64(xd), ref) <= BF16_REL_L2


@pytest.mark.parametrize("T,dtype,d,Hkv", [(1, "bf16", 128, 8), (256, "bf16", 128, 8), (20, "f32", 64, 2)])
def test_kv_append_rotates_keys(Y, T, dtype, d, Hkv):
    """With rope_base set, the append turns K^ at its slot positions (GEMV for a
    decode token, tensor-core GEMM for 256 rows, CUDA cores for fp32) and leaves
    V as without it."""
    import torch
    B, dm, length, base = 1, 256, 4000, 640000.0
    M, Md = gen(SEED, sid(61, 0, synth.T_M), (B, T, dm), dtype)
    Wk, Wkd = gen(SEED, sid(61, 0, synth.T_WK), (dm, Hkv * d), dtype, std=0.05)
    Wv, Wvd = gen(SEED, sid(61, 0, synth.T_WV), (dm, Hkv * d), dtype, std=0.05)
    cache = Y.KVCache(B, Hkv, d, length + T + 3, dtype=Md.dtype, rope_base=base)
    cache.set_length(length)
    Y.yoco_shared_kv_project_append(Md, Wkd, Wvd, cache, eps=1e-6)
    torch.cuda.synchronize()
    kref = oracle.rmsnorm_proj(M, Wk, 1e-6).reshape(B, T, Hkv, d)
    vref = oracle.rmsnorm_proj(M, Wv, 1e-6).reshape(B, T, Hkv, d)
    kref = oracle.rope(kref, (length + np.arange(T))[None, :, None], base)
    kgot = host_f64(cache.k[:, :, length:length + T]).transpose(0, 2, 1, 3)
    vgot = host_f64(cache.v[:, :, length:length + T]).transpose(0, 2, 1, 3)
    if dtype == "f32":
        assert max_abs(kgot, kref) <= FP32_MAX_ABS and max_abs(vgot, vref) <= FP32_MAX_ABS
    else:
        assert rel_l2(kgot, kref) <= BF16_REL_L2 and rel_l2(vgot, vref) <= BF16_REL_L2


def rope_cache(Y, B, Hkv, d, length, dtype, cfg, base):
    """A cache whose keys are already rotated at their slots (as appends leave
    them), built from oracle values only."""
    import torch
    K = synth.normal_f64(SEED, sid(cfg, 0, synth.T_CACHE_K), B * Hkv * length * d).reshape(B, Hkv, length, d)
    Krot = oracle.rope(K, np.arange(length)[None, None, :], base)
    if dtype == "bf16":
        bits = synth.f64_to_bf16_bits(Krot)
        Kh, Kd = synth.bf16_bits_to_f32(bits).astype(np.float64), dev_bf16(bits)
    else:
        Kh = Krot.astype(np.float32).astype(np.float64)
        Kd = dev_f32(Kh)
    V, Vd = gen(SEED, sid(cfg, 0, synth.T_CACHE_V), (B, Hkv, length, d), dtype)
    cache = Y.KVCache(B, Hkv, d, length, dtype=Vd.dtype, k=Kd, v=Vd, rope_base=base)
    cache.set_length(length)
    return Kh, V, cache


@pytest.mark.parametrize("kind", ["decode", "early_exit", "many_rows", "noalloc"])
def test_cross_attn_rotates_queries(Y, kind):
    """With rope_base set every attention path turns each query row by its
    position before the scores: decode (tensor cores), the early-exit row,
    many prefill rows (128-row tiles) and decode without a workspace."""
    import torch
    B, Hq, Hkv, d, length, base = 1, 24, 8, 128, 3000, 5e6
    K, V, cache = rope_cache(Y, B, Hkv, d, length, "bf16", 62, base)
    T, p0 = {"decode": (1, length - 1), "early_exit": (1, length - 1), "many_rows": (300, 1500),
             "noalloc": (1, length - 1)}[kind]
    Q, Qd = gen(SEED, sid(62, 1, synth.T_QX), (B, T, Hq, d), "bf16")
    if kind in ("decode", "noalloc"):
        O = torch.empty(B, Hq, d, dtype=Qd.dtype, device="cuda")
        if kind == "decode":
            Y.yoco_cross_attn_decode(Qd[:, 0].contiguous(), cache, O)
        else:
            Y.yoco_cross_attn_decode_noalloc(Qd[:, 0].contiguous(), cache, O)
        O = O[:, None]
    else:
        O = torch.empty_like(Qd)
        Y.yoco_cross_attn_prefill(Qd, cache, p0, O)
    torch.cuda.synchronize()
    Qrot = oracle.rope(Q, (p0 + np.arange(T))[None, :, None], base)
    O_ref = oracle.cross_attn(Qrot, K, V, p0, d ** -0.5)
    assert rel_l2(host_f64(O), O_ref) <= BF16_REL_L2


def test_cross_attn_rotates_queries_fp32(Y):
    """The CUDA-core path (fp32, head size 64) turns its query rows too."""
    import torch
    B, Hq, Hkv, d, length, base = 1, 4, 2, 64, 400, 10000.0
    K, V, cache = rope_cache(Y, B, Hkv, d, length, "f32", 63, base)
    T, p0 = 40, 300
    Q, Qd = gen(SEED, sid(63, 1, synth.T_QX), (B, T, Hq, d), "f32")
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd, cache, p0, O)
    torch.cuda.synchronize()
    Qrot = oracle.rope(Q, (p0 + np.arange(T))[None, :, None], base)
    assert max_abs(host_f64(O), oracle.cross_attn(Qrot, K, V, p0, d ** -0.5)) <= FP32_MAX_ABS


# ------------------------------------------- gRet input projections (one GEMM)

def qkvg_run(Y, cfg, B, N, dm, H, d, pos0=0, rope_base=0.0):
    import torch
    X, Xd = gen(SEED, sid(cfg, 0, synth.T_M), (B, N, dm), "bf16")
    W, Wd = gen(SEED, sid(cfg, 0, synth.T_WK), (dm, 3 * H * d + H), "bf16", std=dm ** -0.5)
    q = torch.empty(B, N, H, d, dtype=torch.bfloat16, device="cuda")
    k, v = torch.empty_like(q), torch.empty_like(q)
    lg = torch.empty(B, N, H, device="cuda")
    Y.yoco_gret_qkvg_project(Xd, Wd, H, q, k, v, lg, rope_base=rope_base, pos0=pos0)
    torch.cuda.synchronize()
    return (X, W), (q, k, v, lg)


@pytest.mark.parametrize("B,N,dm,H,d,pos0,rope_base", [(2, 300, 256, 8, 128, 0, 0.0), (2, 300, 256, 8, 128, 1000, 5e6),
                                                       (1, 200, 128, 16, 64, 7, 10000.0),
                                                       (1, 100, 192, 8, 64, 0, 0.0)])
def test_qkvg_project(Y, B, N, dm, H, d, pos0, rope_base):
    """q, k, v (bf16, [B, N, H, d]) and the fp32 gate logits of one GEMM over
    [W_Q | W_K | W_V | W_gamma], with and without rotary encoding; ragged rows
    (at 100 rows the second 128-row half of the 256-row tile lies wholly past X)
    and a last column tile that is mostly past the matrix."""
    (X, W), (q, k, v, lg) = qkvg_run(Y, 70, B, N, dm, H, d, pos0, rope_base)
    rq, rk, rv, rlg = oracle.qkvg_project(X, W, H, d, pos0, rope_base)
    for got, ref in ((q, rq), (k, rk), (v, rv)):
        assert rel_l2(host_f64(got), ref) <= BF16_REL_L2
    assert rel_l2(host_f64(lg), rlg) <= 1e-4


def test_qkvg_project_3b_width_sampled_rows(Y):
    """The 3B layer's width (d_model 3072, 24 heads x 128: 9240 columns) over
    4096 tokens; 64 sampled rows against the oracle."""
    B, N, dm, H, d = 1, 4096, 3072, 24, 128
    (X, W), (q, k, v, lg) = qkvg_run(Y, 71, B, N, dm, H, d, 0, 8e7)
    rows = np.linspace(0, N - 1, 64).astype(int)
    # the oracle on the sampled rows only (positions kept: rotate by the row's own position)
    Yr = X[0, rows] @ W
    Hd = H * d
    rq = oracle.rope(Yr[:, :Hd].reshape(-1, H, d), rows[:, None], 8e7)
    rk = oracle.rope(Yr[:, Hd:2 * Hd].reshape(-1, H, d), rows[:, None], 8e7)
    assert rel_l2(host_f64(q[0, rows]), rq) <= BF16_REL_L2
    assert rel_l2(host_f64(k[0, rows]), rk) <= BF16_REL_L2
    assert rel_l2(host_f64(v[0, rows]), Yr[:, 2 * Hd:3 * Hd].reshape(-1, H, d)) <= BF16_REL_L2
    assert rel_l2(host_f64(lg[0, rows]), Yr[:, 3 * Hd:]) <= 1e-4


def test_qkvg_feeds_the_chunk_kernel(Y):
    """The projections' outputs go straight into the chunkwise gRet call: the
    layer (projections + retention) matches the oracle's projections followed
    by the recurrent form on their bf16-rounded values."""
    import torch
    B, N, dm, H, d = 1, 600, 256, 8, 128
    (X, W), (q, k, v, lg) = qkvg_run(Y, 72, B, N, dm, H, d)
    o = torch.empty_like(v)
    S = torch.zeros(B, H, d, d, device="cuda")
    Y.yoco_gret_prefill_chunkwise(q, k, v, lg, 16.0, o, S)
    torch.cuda.synchronize()
    rq, rk, rv, rlg = oracle.qkvg_project(X, W, H, d)
    rnd = lambda a: synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(a)).astype(np.float64)  # noqa: E731
    o_ref, _ = oracle.gret_recurrent(rnd(rq), rnd(rk), rnd(rv), rlg.astype(np.float32).astype(np.float64), 16.0)
    assert rel_l2(host_f64(o), o_ref) <= BF16_REL_L2


# ------------------------------------------------------------- CUDA graphs

def test_gret_decode_steps_replayed_from_a_cuda_graph(Y):
    """The recurrent step launches nothing that a stream capture forbids: 13
    layers' steps captured once and replayed three times give bit for bit what
    three eager passes give (the state carries from replay to replay)."""
    import torch
    B, H, d, layers = 1, 24, 128, 13
    ins = []
    for l in range(layers):
        q, qd = gen(SEED, sid(33, l, synth.T_Q), (B, H, d), "bf16", std=d ** -0.5)
        k, kd = gen(SEED, sid(33, l, synth.T_K), (B, H, d), "bf16", std=d ** -0.5)
        v, vd = gen(SEED, sid(33, l, synth.T_V), (B, H, d), "bf16")
        lg = synth.normal(SEED, sid(33, l, synth.T_LOGIT), (B, H), "f32", mean=2.0)
        ins.append((qd, kd, vd, dev_f32(lg)))
    S0 = dev_f32(synth.normal(SEED, sid(33, 99, synth.T_S0), (layers, B, H, d, d), "f32", std=0.05))

    def run(S, outs, stream=None):
        for l in range(layers):
            qd, kd, vd, lgd = ins[l]
            Y.yoco_gret_decode_step(qd, kd, vd, lgd, 16.0, S[l], outs[l], stream=stream)

    S_e, o_e = S0.clone(), [torch.empty_like(ins[0][2]) for _ in range(layers)]
    for _ in range(3):
        run(S_e, o_e)
    S_g, o_g = S0.clone(), [torch.empty_like(ins[0][2]) for _ in range(layers)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        run(S_g, o_g)
    S_g.copy_(S0)  # capture recorded the launches without running them; start from S0
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(S_g, S_e)
    for a, b in zip(o_g, o_e):
        assert torch.equal(a, b)


# ------------------------------------------------------------- failure path

def test_bounded_wait_times_out_and_context_survives(Y):
    """A device wait that nothing completes gives up after its limit, the
    timeout shows up through yoco_workspace_status, and the GPU keeps
    working (a gRet call right after matches the oracle)."""
    import ctypes
    import time
    import torch
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    st = Y.lib.yoco_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 50_000_000,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == Y.YOCO_OK
    with pytest.raises(Y.YocoError) as e:
        Y.yoco_workspace_status(ws)
    assert e.value.status == Y.YOCO_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    Y.yoco_workspace_status(ws)  # cleared by the previous read
    B, N, H, d = 1, 300, 2, 128
    host, dev = gret_inputs(30, B, N, H, d, "bf16", logit_mean=2.0)
    o, S = run_prefill(Y, dev, B, N, H, d, "bf16")
    o_ref, _ = oracle.gret_recurrent(*host, 16.0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2


def test_calls_make_progress_with_most_sms_taken(Y):
    """A self-test kernel holds all but 30 SMs (one CTA on each, most of its shared
    memory) for 300 ms on another stream.  Meanwhile a segmented gRet prefill
    (24 heads x 6 segments: 264 CTAs of its two kernels, one per SM, far more than
    the free SMs hold at once) and a split-KV decode run on this stream: both
    finish while the other kernel still runs, record no timeout, and match the
    oracle."""
    import torch
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    B, N, H, d = 1, 8192 + 77, 24, 128
    host, dev = gret_inputs(45, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(45, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    qd, kd, vd, lgd = dev
    o = torch.empty_like(vd)
    S = dev_f32(S0)
    ws = torch.zeros(max(256, Y.yoco_gret_prefill_workspace_size(B, N, H, d, d, 0, Y.YOCO_BF16)),
                     dtype=torch.uint8, device="cuda")
    Kh, Kd = gen(SEED, sid(45, 2, synth.T_CACHE_K), (1, 2, 5000, d), "bf16")
    Vh, Vd = gen(SEED, sid(45, 2, synth.T_CACHE_V), (1, 2, 5000, d), "bf16")
    cache = Y.KVCache(1, 2, d, 5000, k=Kd, v=Vd)
    cache.set_length(5000)
    Qh, Qd = gen(SEED, sid(45, 3, synth.T_QX), (1, 6, d), "bf16")
    Od = torch.empty_like(Qd)
    wsa = torch.zeros(max(256, Y.lib.yoco_cross_attn_workspace_size(1, 6, 1, ctypes.byref(cache.c), 0)),
                      dtype=torch.uint8, device="cuda")
    # The same calls once beforehand: with CUDA's lazy module loading, the first launch
    # of a kernel in a process waits for work already running on the device (here the
    # occupying kernel), which is not what this test is about.
    Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, dev_f32(S0), workspace=ws)
    Y.yoco_cross_attn_decode(Qd, cache, Od, workspace=wsa)
    torch.cuda.synchronize()
    other = torch.cuda.Stream()
    assert Y.lib.yoco_selftest_occupy_sms(n_sm - 30, 300_000_000, ctypes.c_void_p(other.cuda_stream)) == Y.YOCO_OK
    Y.yoco_gret_prefill_chunkwise(qd, kd, vd, lgd, 16.0, o, S, workspace=ws)
    Y.yoco_cross_attn_decode(Qd, cache, Od, workspace=wsa)
    done = torch.cuda.Event()
    done.record()
    done.synchronize()
    assert not other.query(), "the occupying kernel ended before the calls did"
    torch.cuda.synchronize()
    Y.yoco_workspace_status(ws)
    Y.yoco_workspace_status(wsa)
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert rel_l2(host_f64(o), o_ref) <= BF16_REL_L2
    assert rel_l2(S.cpu().numpy().astype(np.float64), S_ref) <= BF16_REL_L2
    O_ref = oracle.cross_attn(Qh[:, None], Kh, Vh, 4999, d ** -0.5)[:, 0]
    assert rel_l2(host_f64(Od), O_ref) <= BF16_REL_L2


@pytest.mark.parametrize("segments", [1, 3, 40])
def test_gret_prefill_forced_segment_counts(Y, segments):
    """The tensor-core prefill with its sequence split forced (test hook) to one
    segment per head, three, or 40 (one per chunk here): the same result, for
    every head."""
    import torch
    B, N, H, d = 1, 128 * 40 - 5, 4, 128
    host, dev = gret_inputs(47, B, N, H, d, "bf16", logit_mean=2.0)
    S0 = synth.normal(SEED, sid(47, 1, synth.T_S0), (B, H, d, d), "f32", std=0.05).astype(np.float64)
    assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_GRET_SEGMENTS, segments) == Y.YOCO_OK
    try:
        o, S = run_prefill(Y, dev, B, N, H, d, "bf16", S0=S0)
    finally:
        assert Y.lib.yoco_test_hook(Y.YOCO_HOOK_GRET_SEGMENTS, 0) == Y.YOCO_OK
    o_ref, S_ref = oracle.gret_recurrent(*host, 16.0, S0=S0)
    assert rel_l2(o, o_ref) <= BF16_REL_L2
    for h in range(H):
        assert worst_block_rel_l2(o[0, :, h], o_ref[0, :, h], 128) <= BLOCK_REL_L2, h
        assert rel_l2(S[0, h], S_ref[0, h]) <= BF16_REL_L2, h
