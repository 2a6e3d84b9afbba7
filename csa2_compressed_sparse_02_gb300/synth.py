"""Seeded synthetic inputs for the CSA2 path (host side, numpy).

Counter-based, so any element can be produced on its own: the value of stream
``key`` at counter ``i`` is ``mix(key + (i + 1) * GAMMA)``, where ``mix`` is the
SplitMix64 output function (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; constants as published by Vigna). The GPU
twin in ``csrc/synth/synth.cu`` implements the same definitions, so the host
(oracle side) and the device (product side) see bit-identical inputs without
copying hundreds of GB through the host.

This module holds input distributions only — none of the method's arithmetic.
Distributions (the shapes of the workloads' latents, codes, scales and weights):

* ``normal``: unit-variance, zero-mean Irwin-Hall sum of eight 16-bit uniforms
  (two 64-bit draws per value), scaled by one fp32 constant, so both sides
  compute it exactly (integer sum, one IEEE fp32 multiply).
* ``e2m1_bytes``: two E2M1 codes per byte, each uniform over the 15 distinct
  E2M1 values (-6..6; code 0x8, i.e. -0, is never drawn).
* ``scale_pow2_bytes``: E4M3 bytes of 1.0 or 2.0 (power-of-two group scales).
* ``w_pow2``: 2^u with u uniform in {-2, -1, 0, 1}.
"""
from __future__ import annotations

import numpy as np

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
C1 = 0xBF58476D1CE4E5B9
C2 = 0x94D049BB133111EB

# stream kinds
KV, GATE, Q, SINK, IDX_Q, IDX_Q_SCALE, IDX_W, IDX_K, IDX_K_SCALE, PLANT = range(1, 11)

# E2M1 codes of the 15 distinct values, ascending: -6 -4 -3 -2 -1.5 -1 -0.5 0 0.5 ... 6
E2M1_CODES15 = np.array([0xF, 0xE, 0xD, 0xC, 0xB, 0xA, 0x9, 0x0,
                         0x1, 0x2, 0x3, 0x4, 0x5, 0x6, 0x7], np.uint8)
E4M3_ONE, E4M3_TWO, E4M3_FOUR = 0x38, 0x40, 0x48

# 1/sqrt(32*(65536^2-1)/12) rounded to fp32; unit variance of (2*sum8 - 8*65535)
NORMAL_SCALE_BITS = 0x371CC471
NORMAL_SCALE = np.array([NORMAL_SCALE_BITS], np.uint32).view(np.float32)[0]


def _mix_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * C1) & M64
    z = ((z ^ (z >> 27)) * C2) & M64
    return z ^ (z >> 31)


def stream_key(seed: int, kind: int, a: int = 0, b: int = 0) -> int:
    """64-bit key of the stream (kind, a, b) under `seed` (a: layer, b: sequence)."""
    sid = ((kind & 0xFF) << 56) | ((a & 0xFFFFFF) << 32) | (b & 0xFFFFFFFF)
    return _mix_int((seed & M64) ^ _mix_int(sid))


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=False)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(C1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(C2)
    return z ^ (z >> np.uint64(31))


def u64(key: int, counters: np.ndarray) -> np.ndarray:
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (c + np.uint64(1)) * np.uint64(GAMMA)
    return _mix(z)


def normal(key: int, counters: np.ndarray) -> np.ndarray:
    """fp32 unit-variance values at the given element counters."""
    c = np.asarray(counters, dtype=np.uint64)
    a = u64(key, c * np.uint64(2))
    b = u64(key, c * np.uint64(2) + np.uint64(1))
    s = np.zeros(c.shape, np.int64)
    for x in (a, b):
        for sh in (0, 16, 32, 48):
            s += ((x >> np.uint64(sh)) & np.uint64(0xFFFF)).astype(np.int64)
    n = (2 * s - 8 * 65535).astype(np.float32)  # exact: |n| < 2^20
    return (n * NORMAL_SCALE).astype(np.float32)


def normal_range(key: int, start: int, count: int) -> np.ndarray:
    return normal(key, np.arange(start, start + count, dtype=np.uint64))


def e2m1_bytes(key: int, counters: np.ndarray) -> np.ndarray:
    x = u64(key, counters)
    lo = ((x & np.uint64(0xFFFF)) * np.uint64(15)) >> np.uint64(16)
    hi = (((x >> np.uint64(16)) & np.uint64(0xFFFF)) * np.uint64(15)) >> np.uint64(16)
    return (E2M1_CODES15[lo.astype(np.int64)] | (E2M1_CODES15[hi.astype(np.int64)] << 4)
            ).astype(np.uint8)


def scale_pow2_bytes(key: int, counters: np.ndarray) -> np.ndarray:
    x = u64(key, counters)
    return np.where((x & np.uint64(1)) == 0, E4M3_ONE, E4M3_TWO).astype(np.uint8)


def w_pow2(key: int, counters: np.ndarray) -> np.ndarray:
    x = u64(key, counters)
    u = (x & np.uint64(3)).astype(np.int32) - 2
    return np.ldexp(np.float32(1.0), u).astype(np.float32)


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def uniform_int(key: int, counters: np.ndarray, n: int) -> np.ndarray:
    """Integers uniform-ish in [0, n) (multiply-shift on the top 32 bits)."""
    x = u64(key, counters)
    return (((x >> np.uint64(32)) * np.uint64(n)) >> np.uint64(32)).astype(np.int64)


# ----------------------------------------------------------------------------- plants
def plant_positions(seed: int, group: int, seq: int, n_c: int, count: int = 16) -> np.ndarray:
    """Distinct compressed positions that carry a planted index key (sorted)."""
    key = stream_key(seed, PLANT, group, seq)
    out, i = [], 0
    while len(out) < min(count, n_c):
        p = int(uniform_int(key, np.array([i], np.uint64), n_c)[0])
        if p not in out:
            out.append(p)
        i += 1
    return np.array(sorted(out), np.int64)


def plant_row(q_vals: np.ndarray, w: np.ndarray):
    """Planted index key: the E2M1 codes of the index-query head with the largest
    weight (first such head), with group scale 4 (E4M3 0x48) on every group."""
    h = int(np.argmax(w))
    return q_vals[h].copy(), np.full(q_vals.shape[1] // 8, E4M3_FOUR, np.uint8)


# ----------------------------------------------------------------------------- device twin
G_NORMAL_F32, G_NORMAL_BF16, G_E2M1_BYTES, G_SCALE_POW2_BYTES, G_W_POW2_F32 = range(5)


def gpu_fill(kind: int, keys, counter0: int, n_per_stream: int, out, stride: int | None = None,
             stream=None):
    """Fill out[s * stride + i] = value(keys[s], counter0 + i) on the device with the
    same definitions as the host functions above (libcsa2synth.so)."""
    import ctypes

    import torch

    from ._lib import synth_lib
    keys = [int(k) & M64 for k in keys]
    for s0 in range(0, len(keys), 64):
        chunk = keys[s0:s0 + 64]
        arr = (ctypes.c_uint64 * len(chunk))(*chunk)
        st = n_per_stream if stride is None else stride
        base = out.data_ptr() + s0 * st * out.element_size()
        s = (torch.cuda.current_stream() if stream is None else stream).cuda_stream
        rc = synth_lib().csa2synth_fill(kind, arr, len(chunk), counter0, n_per_stream, base, st, s)
        if rc != 0:
            raise RuntimeError("csa2synth_fill failed (%d)" % rc)
