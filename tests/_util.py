"""Helpers shared by the tests: host <-> device marshalling and error measures."""
import numpy as np

import synth


def dev_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(device)


def dev_f32(x, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def host_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def host_bits(t):
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def worst_block_rel_l2(x, ref, block):
    """Largest relative L2 error over consecutive blocks of `block` rows (axis 0):
    a single wrong chunk or segment boundary shows here even where the
    whole-tensor figure would absorb it."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    worst = 0.0
    for r0 in range(0, x.shape[0], block):
        worst = max(worst, rel_l2(x[r0:r0 + block], ref[r0:r0 + block]))
    return worst


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def gen(seed, stream, shape, dtype, mean=0.0, std=1.0):
    """(host values as fp64, device tensor) for one seeded input."""
    if dtype == "bf16":
        bits = synth.normal(seed, stream, shape, "bf16", mean=mean, std=std)
        return synth.bf16_bits_to_f32(bits).astype(np.float64), dev_bf16(bits)
    x = synth.normal(seed, stream, shape, "f32", mean=mean, std=std)
    return x.astype(np.float64), dev_f32(x)
