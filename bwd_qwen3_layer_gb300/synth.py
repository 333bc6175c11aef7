"""Seeded synthetic inputs shared by the CUDA path's tests and the CPU oracle.

This module draws numbers and nothing else: it holds none of the layer's
arithmetic. Every tensor of a workload is addressed by (seed, name) and drawn
from its own counter-based stream, so a tensor's values do not depend on which
other tensors were drawn or in what order.

Generator (published definitions, written here from them):

* splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state advances by the golden-ratio increment
  0x9E3779B97F4A7C15 and each output is the state passed through the
  variant-13 64-bit finaliser. Element i of a stream is the finaliser applied
  to key + (i + 1) * increment, so any element can be drawn on its own.
* stream key = finaliser(seed XOR finaliser(FNV-1a-64(name))).
* uniform in (0, 1): ((z >> 11) + 0.5) * 2^-53 (never 0 or 1).
* normal: Box-Muller on consecutive uniform pairs (u1, u2):
  sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2).
* integers in [0, n): floor(n * u) (bias below n / 2^53).

Workload recipe (the layer's parameter names follow the decoder-layer
description of the "KYNETRA FOUNDRY" page, pre-normalisation paragraph, and
the capability list of "From-scratch GPU LLM training"):

* projection weights ~ N(0, 0.02), stored [out, in] row-major;
* RMSNorm gains ~ 1 + N(0, 0.02) (not all ones, so a missing gain multiply
  cannot hide);
* hidden states X ~ N(0, 1); upstream gradient dY ~ N(0, 1);
* lm-head weight ~ N(0, 0.02); targets uniform over the vocabulary.

For bf16 runs each drawn value is rounded to bf16 (round to nearest even)
before either side sees it; both sides then consume identical values.

Full-size benchmark tensors (hundreds of millions of elements) are drawn on
the device with torch's seeded Philox generator instead (``device_normal``):
the same distribution and seeding discipline, at device speed. Tests that need
the oracle to see the exact same values read them back from the device.
"""
from __future__ import annotations

import numpy as np

_MASK = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _mix_int(z: int) -> int:
    """splitmix64 finaliser on a Python int (wrapping 64-bit arithmetic)."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def _mix_arr(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (numpy wraps silently)."""
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def fnv1a64(name: str) -> int:
    """FNV-1a 64-bit hash of the UTF-8 bytes of ``name``."""
    h = 0xCBF29CE484222325
    for b in name.encode("utf-8"):
        h ^= b
        h = (h * 0x100000001B3) & _MASK
    return h


def stream_key(seed: int, name: str) -> int:
    return _mix_int((seed & _MASK) ^ _mix_int(fnv1a64(name)))


def raw_u64(seed: int, name: str, count: int, start: int = 0) -> np.ndarray:
    """Elements start .. start+count-1 of the (seed, name) stream."""
    key = np.uint64(stream_key(seed, name))
    out = np.empty(count, dtype=np.uint64)
    chunk = 1 << 22
    for c0 in range(0, count, chunk):
        c1 = min(count, c0 + chunk)
        idx = np.arange(start + c0 + 1, start + c1 + 1, dtype=np.uint64)
        out[c0:c1] = _mix_arr(key + idx * np.uint64(_GOLDEN))
    return out


def uniform(seed: int, name: str, count: int, start: int = 0) -> np.ndarray:
    z = raw_u64(seed, name, count, start)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """fp64 array of the given shape, N(mean, std^2), Box-Muller pairs."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    npairs = (n + 1) // 2
    u = uniform(seed, name, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * npairs, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return (mean + std * z[:n]).reshape(shape)


def randint(seed: int, name: str, shape, high: int) -> np.ndarray:
    """int64 array, uniform over [0, high)."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    u = uniform(seed, name, n)
    return np.minimum(np.floor(u * high).astype(np.int64), high - 1).reshape(shape)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even); returned as fp64.

    Storage rounding of inputs only. Goes through fp32 first, which is exact
    for the rounding decision except for values within one fp32 ulp of a bf16
    tie, where it can pick the other neighbour; both sides see the result, so
    this only changes which inputs are drawn, never parity.
    """
    f = np.ascontiguousarray(a, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    b = (b + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return b.astype(np.uint32).view(np.float32).astype(np.float64).reshape(np.shape(a))


# ----------------------------------------------------------------------------
# Workload recipe
# ----------------------------------------------------------------------------

LAYER_WEIGHT_NAMES = ("gamma1", "Wq", "Wk", "Wv", "Wo", "gamma2", "Wg", "Wu", "Wd")


def layer_weight_shapes(H: int, Hq: int, Hkv: int, d: int, I: int) -> dict:
    return {
        "gamma1": (H,),
        "Wq": (Hq * d, H),
        "Wk": (Hkv * d, H),
        "Wv": (Hkv * d, H),
        "Wo": (H, Hq * d),
        "gamma2": (H,),
        "Wg": (I, H),
        "Wu": (I, H),
        "Wd": (H, I),
    }


def layer_weights(seed: int, H: int, Hq: int, Hkv: int, d: int, I: int,
                  bf16: bool = False, prefix: str = "layer0", qk_norm: bool = False) -> dict:
    """Projection weights N(0, 0.02) [out, in]; norm gains 1 + N(0, 0.02);
    with qk_norm also the per-head q/k gains gamma_q, gamma_k of length d."""
    out = {}
    shapes = layer_weight_shapes(H, Hq, Hkv, d, I)
    if qk_norm:
        shapes = dict(shapes, gamma_q=(d,), gamma_k=(d,))
    for name, shape in shapes.items():
        if name.startswith("gamma"):
            w = normal(seed, f"{prefix}.{name}", shape, std=0.02, mean=1.0)
        else:
            w = normal(seed, f"{prefix}.{name}", shape, std=0.02)
        out[name] = round_bf16(w) if bf16 else w
    return out


def layer_inputs(seed: int, T: int, H: int, bf16: bool = False) -> dict:
    X = normal(seed, "X", (T, H))
    dY = normal(seed, "dY", (T, H))
    if bf16:
        X, dY = round_bf16(X), round_bf16(dY)
    return {"X": X, "dY": dY}


def lmhead_inputs(seed: int, N: int, H: int, V: int, bf16: bool = False) -> dict:
    X = normal(seed, "lm.X", (N, H))
    W = normal(seed, "lm.W", (V, H), std=0.02)
    if bf16:
        X, W = round_bf16(X), round_bf16(W)
    tgt = randint(seed, "lm.targets", (N,), V)
    return {"X": X, "W": W, "targets": tgt}


def device_normal(shape, std: float, mean: float, seed: int, name: str, dtype, device):
    """Large seeded N(mean, std^2) tensor drawn on the device (torch Philox)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((stream_key(seed, name) >> 1) & 0x7FFFFFFFFFFFFFFF)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(mean=mean, std=std, generator=g)
    return t.to(dtype)


def device_randint(shape, high: int, seed: int, name: str, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((stream_key(seed, name) >> 1) & 0x7FFFFFFFFFFFFFFF)
    return torch.randint(0, high, shape, generator=g, device=device, dtype=torch.int32)
