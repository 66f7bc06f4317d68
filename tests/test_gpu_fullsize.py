"""Parity at the full workload sizes, in the launch configuration the bench
times, on outputs the oracle can compute one by one: whole heads of the 32K
gRet layer, a head of the 512K gRet layer, decode attention over 128K- and
1M-token shared caches for sampled (sequence, kv head) groups, and the
appended cache slots.

Inputs are made on the device by the seeded generator's device copy; the
oracle regenerates exactly the elements it needs on the host (same
counter-based definition), never from a libyoco result.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import dev_f32, host_bits, host_f64, rel_l2, worst_block_rel_l2

pytestmark = pytest.mark.gpu

BF16_REL_L2 = 1e-2
BLOCK_REL_L2 = 3e-2  # worst 128-row block (or row group): bf16 rounding of one block, with room
SEED = synth.DEFAULT_SEED
SID = synth.stream_id


@pytest.fixture(scope="module")
def Y():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import gated_retention_shared_gb300 as Y
    return Y


def dev_normal(shape, dtype, stream, mean=0.0, std=1.0):
    import torch
    t = torch.empty(shape, dtype=dtype, device="cuda")
    return synth.fill_normal_(t, SEED, stream, mean, std)


def host_head(stream, B, N, H, D, b, h, n0, n1, mean=0.0, std=1.0, bf16=True):
    """Elements [b, n0:n1, h, :] of a [B, N, H, D] tensor of the stream, as the
    bf16 (or fp32) values the device holds, widened to fp64."""
    n = np.arange(n0, n1, dtype=np.uint64)[:, None]
    c = np.arange(D, dtype=np.uint64)[None, :]
    idx = ((np.uint64(b) * np.uint64(N) + n) * np.uint64(H) + np.uint64(h)) * np.uint64(D) + c
    x = synth.normal_at(SEED, stream, idx, mean, std)
    if bf16:
        return synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(x)).astype(np.float64)
    return x.astype(np.float32).astype(np.float64)


def host_logits(stream, B, N, H, b, h, n0, n1, mean):
    n = np.arange(n0, n1, dtype=np.uint64)
    idx = (np.uint64(b) * np.uint64(N) + n) * np.uint64(H) + np.uint64(h)
    return synth.normal_at(SEED, stream, idx, mean, 1.0).astype(np.float32).astype(np.float64)


def _gret_layer(Y, cfg, B, N, H, D, heads):
    import torch
    q = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_Q), std=D ** -0.5)
    k = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_K), std=D ** -0.5)
    v = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_V))
    lg = dev_normal((B, N, H), torch.float32, SID(cfg, 0, synth.T_LOGIT), mean=2.0)
    o = torch.empty_like(v)
    S = torch.zeros(B, H, D, D, device="cuda")
    ws = torch.empty(max(256, Y.yoco_gret_prefill_workspace_size(B, N, H, D, D, 0, Y.YOCO_BF16)),
                     dtype=torch.uint8, device="cuda")
    Y.yoco_gret_prefill_chunkwise(q, k, v, lg, 16.0, o, S, workspace=ws)
    Y.yoco_workspace_status(ws)
    for h in heads:
        hq = host_head(SID(cfg, 0, synth.T_Q), B, N, H, D, 0, h, 0, N, std=D ** -0.5)
        hk = host_head(SID(cfg, 0, synth.T_K), B, N, H, D, 0, h, 0, N, std=D ** -0.5)
        hv = host_head(SID(cfg, 0, synth.T_V), B, N, H, D, 0, h, 0, N)
        hl = host_logits(SID(cfg, 0, synth.T_LOGIT), B, N, H, 0, h, 0, N, 2.0)
        o_ref, S_ref = oracle.gret_recurrent(hq[None, :, None], hk[None, :, None], hv[None, :, None],
                                             hl[None, :, None], 16.0)
        o_gpu = host_f64(o[0, :, h])
        assert rel_l2(o_gpu, o_ref[0, :, 0]) <= BF16_REL_L2, (h, rel_l2(o_gpu, o_ref[0, :, 0]))
        # every 128-token chunk on its own, so one wrong chunk or segment boundary shows
        worst = worst_block_rel_l2(o_gpu, o_ref[0, :, 0], 128)
        assert worst <= BLOCK_REL_L2, (h, worst)
        assert rel_l2(S[0, h].cpu().numpy(), S_ref[0, 0]) <= BF16_REL_L2


def test_gret_layer_32k_x24_whole_heads(Y):
    """The 32K-token, 24 x 128 gRet layer (the bench's layer shape): three whole
    heads, every output and the final state."""
    _gret_layer(Y, 2, 1, 32768, 24, 128, heads=(0, 13, 23))


def test_gret_gn_gate_fused_32k_x24_heads(Y):
    """The 32K-token, 24 x 128 gRet layer with Eq. 7's output fused (GroupNorm per
    head and the swish gate as rows leave the kernel): three whole heads of z,
    chunk by chunk, against the oracle's recurrent form followed by its
    group_norm_gate, and their final states."""
    import torch
    B, N, H, D, cfg = 1, 32768, 24, 128, 2
    q = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_Q), std=D ** -0.5)
    k = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_K), std=D ** -0.5)
    v = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_V))
    lg = dev_normal((B, N, H), torch.float32, SID(cfg, 0, synth.T_LOGIT), mean=2.0)
    g = dev_normal((B, N, H, D), torch.bfloat16, SID(cfg, 0, synth.T_QX))
    z = torch.empty_like(v)
    S = torch.zeros(B, H, D, D, device="cuda")
    ws = torch.empty(max(256, Y.yoco_gret_prefill_workspace_size(B, N, H, D, D, 0, Y.YOCO_BF16)),
                     dtype=torch.uint8, device="cuda")
    Y.yoco_gret_prefill_chunkwise_gn_gate(q, k, v, lg, 16.0, g, z, S, eps=1e-5, workspace=ws)
    Y.yoco_workspace_status(ws)
    for h in (0, 13, 23):
        hq = host_head(SID(cfg, 0, synth.T_Q), B, N, H, D, 0, h, 0, N, std=D ** -0.5)
        hk = host_head(SID(cfg, 0, synth.T_K), B, N, H, D, 0, h, 0, N, std=D ** -0.5)
        hv = host_head(SID(cfg, 0, synth.T_V), B, N, H, D, 0, h, 0, N)
        hl = host_logits(SID(cfg, 0, synth.T_LOGIT), B, N, H, 0, h, 0, N, 2.0)
        hg = host_head(SID(cfg, 0, synth.T_QX), B, N, H, D, 0, h, 0, N)
        o_ref, S_ref = oracle.gret_recurrent(hq[None, :, None], hk[None, :, None], hv[None, :, None],
                                             hl[None, :, None], 16.0)
        z_ref = oracle.group_norm_gate(o_ref, hg[None, :, None], 1e-5)[0, :, 0]
        z_gpu = host_f64(z[0, :, h])
        assert rel_l2(z_gpu, z_ref) <= BF16_REL_L2, (h, rel_l2(z_gpu, z_ref))
        worst = worst_block_rel_l2(z_gpu, z_ref, 128)
        assert worst <= BLOCK_REL_L2, (h, worst)
        assert rel_l2(S[0, h].cpu().numpy(), S_ref[0, 0]) <= BF16_REL_L2


def test_gret_layer_512k_x24_whole_head(Y):
    """One gRet layer of the 512K-token prefill (six segments of 87424 tokens):
    all 524288 outputs of head 7, chunk by chunk, and its final state."""
    _gret_layer(Y, 4, 1, 524288, 24, 128, heads=(7,))


def _decode_cache(Y, cfg, B, Hkv, D, length, extra):
    import torch
    K = dev_normal((B, Hkv, length + extra, D), torch.bfloat16, SID(cfg, 0, synth.T_CACHE_K))
    V = dev_normal((B, Hkv, length + extra, D), torch.bfloat16, SID(cfg, 0, synth.T_CACHE_V))
    cache = Y.KVCache(B, Hkv, D, length + extra, k=K, v=V)
    cache.set_length(length)
    return cache


def _host_cache_rows(cfg, tensor, B, Hkv, cap, D, b, hk, n1, block=65536):
    out = np.empty((n1, D))
    c = np.arange(D, dtype=np.uint64)[None, :]
    base = (np.uint64(b) * np.uint64(Hkv) + np.uint64(hk)) * np.uint64(cap)
    for r0 in range(0, n1, block):
        n = np.arange(r0, min(n1, r0 + block), dtype=np.uint64)[:, None]
        x = synth.normal_at(SEED, SID(cfg, 0, tensor), (base + n) * np.uint64(D) + c)
        out[r0:r0 + len(n)] = synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(x))
    return out


@pytest.mark.parametrize("B", [1, 8, 32])
def test_decode_step_131072_cache(Y, B):
    """Shared-KV decode at 131072 cached tokens, 8 kv heads x 128, 24 query
    heads: append one projected token per sequence, then one cross layer.
    Sampled (sequence, kv head) groups are checked against the oracle,
    including the appended slot."""
    import torch
    Hkv, Hq, D, N, DM = 8, 24, 128, 131072, 3072
    cfg = 3
    cache = _decode_cache(Y, cfg, B, Hkv, D, N, 1024)
    M = dev_normal((B, 1, DM), torch.bfloat16, SID(cfg, 0, synth.T_M, 1))
    Wk = dev_normal((DM, Hkv * D), torch.bfloat16, SID(cfg, 0, synth.T_WK), std=0.02)
    Wv = dev_normal((DM, Hkv * D), torch.bfloat16, SID(cfg, 0, synth.T_WV), std=0.02)
    Y.yoco_shared_kv_project_append(M, Wk, Wv, cache, eps=1e-6)
    Q = dev_normal((B, Hq, D), torch.bfloat16, SID(cfg, 0, synth.T_QX, 1))
    O = torch.empty_like(Q)
    Y.yoco_cross_attn_decode(Q, cache, O)
    torch.cuda.synchronize()
    cap = N + 1024
    hM = synth.bf16_bits_to_f32(synth.normal(SEED, SID(cfg, 0, synth.T_M, 1), (B, 1, DM), "bf16")).astype(np.float64)
    hWk = synth.bf16_bits_to_f32(synth.normal(SEED, SID(cfg, 0, synth.T_WK), (DM, Hkv * D), "bf16", std=0.02))
    hWv = synth.bf16_bits_to_f32(synth.normal(SEED, SID(cfg, 0, synth.T_WV), (DM, Hkv * D), "bf16", std=0.02))
    for b, hk in {(0, 0), (B - 1, Hkv - 1), (B // 2, 3)}:
        newk = oracle.rmsnorm_proj(hM[b], hWk, 1e-6)[0, hk * D:(hk + 1) * D]
        newv = oracle.rmsnorm_proj(hM[b], hWv, 1e-6)[0, hk * D:(hk + 1) * D]
        got_k = host_f64(cache.k[b, hk, N])
        assert rel_l2(got_k, newk) <= BF16_REL_L2
        assert rel_l2(host_f64(cache.v[b, hk, N]), newv) <= BF16_REL_L2
        Kh = _host_cache_rows(cfg, synth.T_CACHE_K, B, Hkv, cap, D, b, hk, N)
        Vh = _host_cache_rows(cfg, synth.T_CACHE_V, B, Hkv, cap, D, b, hk, N)
        # the appended slot as the oracle rounds it
        Kh = np.concatenate([Kh, synth.bf16_bits_to_f32(oracle.round_bf16(newk))[None].astype(np.float64)], axis=0)
        Vh = np.concatenate([Vh, synth.bf16_bits_to_f32(oracle.round_bf16(newv))[None].astype(np.float64)], axis=0)
        G = Hq // Hkv
        hQ = synth.bf16_bits_to_f32(synth.normal(SEED, SID(cfg, 0, synth.T_QX, 1), (B, Hq, D), "bf16"))
        Qg = hQ[b, hk * G:(hk + 1) * G].astype(np.float64)[None, None]
        O_ref = oracle.cross_attn(Qg, Kh[None, None], Vh[None, None], N, D ** -0.5)[0, 0]
        assert rel_l2(host_f64(O[b, hk * G:(hk + 1) * G]), O_ref) <= BF16_REL_L2
        # each query head on its own
        assert worst_block_rel_l2(host_f64(O[b, hk * G:(hk + 1) * G]), O_ref, 1) <= BLOCK_REL_L2
    assert cache.length == N + 1


def test_cross_attn_full_prefill_32k(Y):
    """Causal cross-attention prefill of all 32768 rows over a 32768-token cache
    (24 query heads on 8 kv heads): sampled rows of two kv groups, from the
    first and last query tiles and between, against the oracle row by row."""
    import torch
    B, Hkv, Hq, D, N = 1, 8, 24, 128, 32768
    cfg = 36
    K = dev_normal((B, Hkv, N, D), torch.bfloat16, SID(cfg, 0, synth.T_CACHE_K))
    V = dev_normal((B, Hkv, N, D), torch.bfloat16, SID(cfg, 0, synth.T_CACHE_V))
    cache = Y.KVCache(B, Hkv, D, N, k=K, v=V)
    cache.set_length(N)
    Q = dev_normal((B, N, Hq, D), torch.bfloat16, SID(cfg, 1, synth.T_QX))
    O = torch.empty_like(Q)
    Y.yoco_cross_attn_prefill(Q, cache, 0, O)
    torch.cuda.synchronize()
    G = Hq // Hkv
    for hk in (0, Hkv - 1):
        Kh = _host_cache_rows(cfg, synth.T_CACHE_K, B, Hkv, N, D, 0, hk, N)
        Vh = _host_cache_rows(cfg, synth.T_CACHE_V, B, Hkv, N, D, 0, hk, N)
        for row in (0, 127, 128, 5000, 16383, N - 1):
            Qg = np.stack([host_head(SID(cfg, 1, synth.T_QX), B, N, Hq, D, 0, h, row, row + 1)[0]
                           for h in range(hk * G, (hk + 1) * G)])
            O_ref = oracle.cross_attn(Qg[None, None], Kh[None, None, :row + 1], Vh[None, None, :row + 1], row,
                                      D ** -0.5)[0, 0]
            got = host_f64(O[0, row, hk * G:(hk + 1) * G])
            assert rel_l2(got, O_ref) <= BF16_REL_L2, (hk, row, rel_l2(got, O_ref))
            assert worst_block_rel_l2(got, O_ref, 1) <= BLOCK_REL_L2, (hk, row)


def test_decode_1m_cache_and_state_step(Y):
    """1M-token decode: one recurrent gRet step on 24 x 128 x 128 states and a
    cross layer over 1048576 cached tokens (kv head 0's group checked)."""
    import torch
    Hkv, Hq, D, N, H = 8, 24, 128, 1048576, 24
    cfg = 5
    cache = _decode_cache(Y, cfg, 1, Hkv, D, N, 256)
    Q = dev_normal((1, Hq, D), torch.bfloat16, SID(cfg, 0, synth.T_QX, 1))
    O = torch.empty_like(Q)
    Y.yoco_cross_attn_decode(Q, cache, O)
    S0_host = synth.normal(SEED, SID(cfg, 0, synth.T_S0), (1, H, D, D), "f32", std=0.05).astype(np.float64)
    S0 = dev_f32(S0_host)
    q1 = dev_normal((1, H, D), torch.bfloat16, SID(cfg, 0, synth.T_Q, 1), std=D ** -0.5)
    k1 = dev_normal((1, H, D), torch.bfloat16, SID(cfg, 0, synth.T_K, 1), std=D ** -0.5)
    v1 = dev_normal((1, H, D), torch.bfloat16, SID(cfg, 0, synth.T_V, 1))
    lg1 = dev_normal((1, H), torch.float32, SID(cfg, 0, synth.T_LOGIT, 1), mean=2.0)
    o1 = torch.empty_like(v1)
    Y.yoco_gret_decode_step(q1, k1, v1, lg1, 16.0, S0, o1)
    torch.cuda.synchronize()
    cap = N + 256
    Kh = _host_cache_rows(cfg, synth.T_CACHE_K, 1, Hkv, cap, D, 0, 0, N)
    Vh = _host_cache_rows(cfg, synth.T_CACHE_V, 1, Hkv, cap, D, 0, 0, N)
    hQ = synth.bf16_bits_to_f32(synth.normal(SEED, SID(cfg, 0, synth.T_QX, 1), (1, Hq, D), "bf16"))
    O_ref = oracle.cross_attn(hQ[0, 0:3].astype(np.float64)[None, None], Kh[None, None], Vh[None, None], N - 1,
                              D ** -0.5)[0, 0]
    assert rel_l2(host_f64(O[0, 0:3]), O_ref) <= BF16_REL_L2
    assert worst_block_rel_l2(host_f64(O[0, 0:3]), O_ref, 1) <= BLOCK_REL_L2
    f = lambda t, **kw: synth.bf16_bits_to_f32(synth.normal(SEED, t, (1, 1, H, D), "bf16", **kw))  # noqa: E731
    hq = f(SID(cfg, 0, synth.T_Q, 1), std=D ** -0.5)
    hk = f(SID(cfg, 0, synth.T_K, 1), std=D ** -0.5)
    hv = f(SID(cfg, 0, synth.T_V, 1))
    hl = synth.normal(SEED, SID(cfg, 0, synth.T_LOGIT, 1), (1, 1, H), "f32", mean=2.0)
    o_ref, S_ref = oracle.gret_recurrent(hq, hk, hv, hl, 16.0, S0=S0_host)
    assert rel_l2(host_f64(o1), o_ref[:, 0]) <= BF16_REL_L2
    assert rel_l2(S0.cpu().numpy(), S_ref) <= BF16_REL_L2
