"""Small valid cases of every libyoco call, run against whichever build of the
library YOCO_LIB_PATH names (the debug-checks build, from
tests/test_gpu_debug_build.py).  Each result is checked against the oracle,
then the build's index checks must all have passed (debug word 0).  Prints
"debug cases ok" on success; any failure raises."""
import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import gated_retention_shared_gb300 as Y  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from _util import dev_f32, gen, host_f64, rel_l2  # noqa: E402

SEED = synth.DEFAULT_SEED
sid = synth.stream_id


def debug_word():
    w = ctypes.c_uint32(0xFFFFFFFF)
    st = Y.lib.yoco_debug_checks(1, ctypes.byref(w))
    assert st == Y.YOCO_OK, Y.lib.yoco_last_error()
    return w.value


def check(name, got, ref, tol=1e-2):
    err = rel_l2(got, ref)
    assert err <= tol, (name, err)
    w = debug_word()
    assert w == 0, (name, hex(w))


def main():
    assert os.environ.get("YOCO_LIB_PATH"), "run with YOCO_LIB_PATH set to the debug build"
    d = 128
    # gRet prefill: tensor cores (6 segments per head), CUDA cores (fp32, d = 64), fused Eq. 7
    for (B, N, H, dt, dd) in ((1, 2000, 24, "bf16", 128), (1, 300, 2, "f32", 64)):
        q, qd = gen(SEED, sid(50, 0, synth.T_Q), (B, N, H, dd), dt, std=dd ** -0.5)
        k, kd = gen(SEED, sid(50, 0, synth.T_K), (B, N, H, dd), dt, std=dd ** -0.5)
        v, vd = gen(SEED, sid(50, 0, synth.T_V), (B, N, H, dd), dt)
        lg = synth.normal(SEED, sid(50, 0, synth.T_LOGIT), (B, N, H), "f32", mean=2.0).astype(np.float64)
        o = torch.empty_like(vd)
        S = torch.zeros(B, H, dd, dd, device="cuda")
        Y.yoco_gret_prefill_chunkwise(qd, kd, vd, dev_f32(lg), 16.0, o, S)
        o_ref, S_ref = oracle.gret_recurrent(q, k, v, lg, 16.0)
        check(f"gret prefill {dt}", host_f64(o), o_ref)
        g, gd = gen(SEED, sid(50, 1, synth.T_QX), (B, N, H, dd), dt)
        z = torch.empty_like(vd)
        S.zero_()
        Y.yoco_gret_prefill_chunkwise_gn_gate(qd, kd, vd, dev_f32(lg), 16.0, gd, z, S)
        check(f"gret prefill + Eq. 7 {dt}", host_f64(z), oracle.group_norm_gate(o_ref, g, 1e-5))
        # one recurrent step from the final state
        o1 = torch.empty(B, H, dd, dtype=vd.dtype, device="cuda")
        S1 = dev_f32(S_ref)
        Y.yoco_gret_decode_step(qd[:, -1].contiguous(), kd[:, -1].contiguous(), vd[:, -1].contiguous(),
                                dev_f32(lg[:, -1]), 16.0, S1, o1)
        o1_ref, _ = oracle.gret_recurrent(q[:, -1:], k[:, -1:], v[:, -1:], lg[:, -1:], 16.0, S0=S_ref)
        check(f"gret step {dt}", host_f64(o1), o1_ref[:, 0])
    # shared K^/V^ append: strip GEMV (1 row), split-K GEMV (6 rows), tensor cores (300 rows)
    Hkv, Hq, dm = 2, 6, 256
    W, Wd = gen(SEED, sid(50, 2, synth.T_WK), (dm, 2 * Hkv * d), "bf16", std=0.05)
    Wkd, Wvd = Wd[:, :Hkv * d].contiguous(), Wd[:, Hkv * d:].contiguous()
    cache = Y.KVCache(1, Hkv, d, 400, device="cuda")
    rows_seen = []
    for T in (300, 6, 1):
        M, Md = gen(SEED, sid(50, 3 + T, synth.T_M), (1, T, dm), "bf16")
        Y.yoco_shared_kv_project_append(Md, Wkd, Wvd, cache, eps=1e-6)
        rows_seen.append(M[0])
        kv = oracle.rmsnorm_proj(M[0], W, 1e-6)
        n0 = cache.length - T
        got = host_f64(cache.k[0, :, n0:n0 + T]).transpose(1, 0, 2).reshape(T, Hkv * d)
        check(f"append {T}", got, kv[:, :Hkv * d])
    Kc, Vc = host_f64(cache.k), host_f64(cache.v)
    L = cache.length
    # cross attention: the early-exit row (tensor cores), many rows (flash kernel), decode (split-KV)
    Q, Qd = gen(SEED, sid(50, 4, synth.T_QX), (1, 100, Hq, d), "bf16")
    O = torch.empty_like(Qd)
    Y.yoco_cross_attn_prefill(Qd[:, :1].contiguous(), cache, L - 1, O[:, :1])
    check("cross early exit", host_f64(O[:, :1]), oracle.cross_attn(Q[:, :1], Kc, Vc, L - 1, d ** -0.5))
    Y.yoco_cross_attn_prefill(Qd, cache, L - 100, O)
    check("cross many rows", host_f64(O), oracle.cross_attn(Q, Kc, Vc, L - 100, d ** -0.5))
    Od = torch.empty(1, Hq, d, dtype=torch.bfloat16, device="cuda")
    Y.yoco_cross_attn_decode(Qd[:, 0].contiguous(), cache, Od, num_splits=3)
    check("cross decode", host_f64(Od), oracle.cross_attn(Q[:, :1], Kc, Vc, L - 1, d ** -0.5)[:, 0])
    # sliding-window self-decoder, rotary encoding, the projections in one GEMM
    ring = Y.SwaRing(1, Hkv, d, 64, device="cuda")
    ks, ksd = gen(SEED, sid(50, 5, synth.T_K), (1, 200, Hkv, d), "bf16")
    vs, vsd = gen(SEED, sid(50, 5, synth.T_V), (1, 200, Hkv, d), "bf16")
    qs, qsd = gen(SEED, sid(50, 5, synth.T_Q), (1, 200, Hq, d), "bf16")
    os_ = torch.empty_like(qsd)
    Y.yoco_swa_prefill(qsd, ksd, vsd, ring, os_)
    check("swa prefill", host_f64(os_), oracle.swa_attn(qs, ks, vs, 64, d ** -0.5))
    xr, xrd = gen(SEED, sid(50, 6, synth.T_Q), (1, 50, 4, d), "bf16")
    Y.yoco_rope_apply(xrd, 1e4, pos0=1000)
    pos = 1000 + np.arange(50)
    check("rope", host_f64(xrd), oracle.rope(xr, pos[None, :, None], 1e4))
    X, Xd = gen(SEED, sid(50, 7, synth.T_M), (1, 130, dm), "bf16")
    Wg, Wgd = gen(SEED, sid(50, 7, synth.T_WK), (dm, 3 * 8 * d + 8), "bf16", std=dm ** -0.5)
    qg = torch.empty(1, 130, 8, d, dtype=torch.bfloat16, device="cuda")
    kg, vg = torch.empty_like(qg), torch.empty_like(qg)
    lgg = torch.empty(1, 130, 8, device="cuda")
    Y.yoco_gret_qkvg_project(Xd, Wgd, 8, qg, kg, vg, lgg)
    rq, _, _, _ = oracle.qkvg_project(X, Wg, 8, d)
    check("qkvg", host_f64(qg), rq)
    print("debug cases ok", flush=True)


if __name__ == "__main__":
    main()
