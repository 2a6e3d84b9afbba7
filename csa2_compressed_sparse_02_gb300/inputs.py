"""Input recipe of the CSA2 decode configurations (host side, numpy only).

Everything a configuration feeds the path is a function of (seed, stream,
counter) through ``synth``, so any one sequence's inputs can be regenerated on
the host for the oracle while the device builds the full batch with the GPU
twin of the generator. No arithmetic of the method lives here.

Shapes follow the pages' serving setup ("DeepSeek-V4.1-Flash-NVFP4" §六:
max-model-len 1,048,576, max-num-seqs 32; §四: KV-source layers shared by the
layers in between; §3.3: index results published by one layer and reused).
A *group* is one KV-source layer and the layers that read its compressed
cache (the source included): per decode step it runs one Compressor append
on the source, a window append on every reader, one Indexer scan, one
two-level selection and one sparse attention per layer, with shared indices
and each layer's own query and window.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import synth

SEED_BASE = 0xC5A20000
LEN = 11  # stream kind for ragged context lengths


@dataclass(frozen=True)
class DecodeConfig:
    number: int
    workload: str
    B: int
    groups: int         # KV-source groups per step
    readers: int        # layers per group that attend (source included)
    steps: int          # consecutive decode steps per run
    quant: bool         # NVFP4 cache / E4M3 window / bf16 query, else all fp32
    plants: int         # planted index keys per sequence
    kscale_pow2: bool   # index-key group scales drawn from {1, 2} (else 1)
    T: int = 0          # context length (incl. the step's token) at step 0; 0 = ragged
    T_range: tuple = (4096, 1048576)
    ratio: int = 2      # raw tokens per compressed position: 2 (pooled) or 1 (1:1 layers)
    rope: bool = False  # the Compressor rotates the last ROPE_DIM dims of each compressed row

    @property
    def seed(self) -> int:
        return SEED_BASE + self.number

    def first_lengths(self) -> list:
        """Raw context length of every sequence at its first decode step."""
        if self.T:
            return [self.T] * self.B
        lo, hi = math.log(self.T_range[0]), math.log(self.T_range[1])
        out = []
        for s in range(self.B):
            x = int(synth.u64(synth.stream_key(self.seed, LEN, 0, s), np.array([0], np.uint64))[0])
            u = (x >> 11) * 2.0 ** -53
            out.append(2 * int(round(math.exp(lo + u * (hi - lo)) / 2)))
        return out

    def layer(self, g: int, r: int) -> int:
        return g * self.readers + r


CONFIGS = {
    1: DecodeConfig(1, "decode B=1 T=4096 unquantised (fp32)", B=1, groups=1, readers=1,
                    steps=1, quant=False, plants=0, kscale_pow2=False, T=4096),
    2: DecodeConfig(2, "decode B=8 T=65536 NVFP4", B=8, groups=1, readers=1, steps=1,
                    quant=True, plants=16, kscale_pow2=True, T=65536),
    3: DecodeConfig(3, "decode B=32 T=1048576 NVFP4, 4 KV-source groups x 10 layers", B=32,
                    groups=4, readers=10, steps=1, quant=True, plants=16, kscale_pow2=True,
                    T=1048576),
    # a profiling size of the decode step: index keys (151 MB) still larger than L2
    6: DecodeConfig(6, "decode B=32 T=131072 NVFP4, 1 group x 2 layers (profiling size)", B=32,
                    groups=1, readers=2, steps=1, quant=True, plants=16, kscale_pow2=True,
                    T=131072),
    # the 8-index-source reading of the step: 8 scans + 8 selections + 40 attention
    # calls (each index source published to 5 layers), against configuration 3's 4
    8: DecodeConfig(8, "decode B=32 T=1048576 NVFP4, 8 index sources x 5 layers", B=32,
                    groups=8, readers=5, steps=1, quant=True, plants=16, kscale_pow2=True,
                    T=1048576),
    # the uncompressed 1:1 layers: n_c = T, pooling skipped (two layers share the cache)
    7: DecodeConfig(7, "decode B=8 T=32768 1:1 layers (n_c = T) NVFP4, 1 group x 2 layers", B=8,
                    groups=1, readers=2, steps=1, quant=True, plants=16, kscale_pow2=True,
                    T=32768, ratio=1),
    # the compressed KV rotated by the Compressor (YaRN, base 160000, factor 16, last 64 dims)
    9: DecodeConfig(9, "decode B=8 T=65536 NVFP4, compressed-KV RoPE (YaRN x16, base 160000, "
                       "last 64 dims)", B=8, groups=1, readers=1, steps=1, quant=True, plants=16,
                    kscale_pow2=True, T=65536, rope=True),
    5: DecodeConfig(5, "decode B=32 ragged T in [4096, 1048576], 1 index source + 5 readers, "
                       "16 steps", B=32, groups=1, readers=6, steps=16, quant=True, plants=16,
                    kscale_pow2=True),
}



@dataclass(frozen=True)
class PrefillConfig:
    """A prefill chunk appended to a prior context of one sequence: query i sits
    at raw position T0 + i, so its context (itself included) is T0 + i + 1 tokens
    and it sees compressed positions j with 2j + 1 <= T0 + i (n_c = (T0+i+1)//2).
    Per-query inputs use the decode recipe with the query index as the step."""
    number: int
    workload: str
    T0: int
    chunk: int
    quant: bool = True
    plants: int = 16
    kscale_pow2: bool = True
    B: int = 1
    ratio: int = 2      # the prefill chunk runs on a pooled (2:1) layer
    groups: int = 1
    readers: int = 1

    @property
    def seed(self) -> int:
        return SEED_BASE + self.number

    def first_lengths(self) -> list:
        return [self.T0 + 1]

    def layer(self, g: int, r: int) -> int:
        return g * self.readers + r


PREFILL = PrefillConfig(4, "prefill chunk of 8192 queries on a 262,144-token context, NVFP4",
                        T0=262144, chunk=8192)

D, H, HI, DI, W = 512, 64, 32, 128, 128
ROPE_DIM = 64  # rotated width of the compressed KV (a reading; the pages give only the base)


# =============================================================================== host side
def host_kv(cfg: DecodeConfig, layer: int, s: int, t0: int, t1: int, kind=synth.KV) -> np.ndarray:
    key = synth.stream_key(cfg.seed, kind, layer, s)
    return synth.normal_range(key, t0 * D, (t1 - t0) * D).reshape(t1 - t0, D)


def host_gate(cfg, layer, s, t0, t1):
    return host_kv(cfg, layer, s, t0, t1, kind=synth.GATE)


def host_q(cfg, layer: int, s: int, step: int) -> np.ndarray:
    """Attention query [H, D] as the kernels see it (fp64 of the bf16 / fp32 value)."""
    key = synth.stream_key(cfg.seed, synth.Q, layer, s)
    x = synth.normal_range(key, step * H * D, H * D).reshape(H, D)
    if cfg.quant:
        return synth.bf16_to_f64(synth.bf16_bits_rne(x))
    return x.astype(np.float64)


def host_sink(cfg, layer: int) -> np.ndarray:
    return synth.normal_range(synth.stream_key(cfg.seed, synth.SINK, layer, 0), 0, H)


def host_index_q(cfg, g: int, s: int, step: int):
    kq = synth.stream_key(cfg.seed, synth.IDX_Q, g, s)
    vals = synth.e2m1_bytes(kq, np.arange(step * HI * DI // 2, (step + 1) * HI * DI // 2,
                                          dtype=np.uint64)).reshape(HI, DI // 2)
    scales = np.full((HI, DI // 16), synth.E4M3_ONE, np.uint8)
    kw = synth.stream_key(cfg.seed, synth.IDX_W, g, s)
    w = synth.w_pow2(kw, np.arange(step * HI, (step + 1) * HI, dtype=np.uint64))
    return vals, scales, w


def plants(cfg, g: int, s: int):
    """(positions, values row, scales row) of the planted index keys of one sequence."""
    if not cfg.plants:
        return np.zeros(0, np.int64), None, None
    n_c0 = cfg.first_lengths()[s] // cfg.ratio
    pos = synth.plant_positions(cfg.seed, g, s, n_c0, cfg.plants)
    qv, _, w = host_index_q(cfg, g, s, 0)
    rv, rs = synth.plant_row(qv, w)
    return pos, rv, rs


def host_index_keys(cfg, g: int, s: int, n: int):
    """Index keys [n, 64] + scales [n, 8] of one sequence, plants included."""
    kk = synth.stream_key(cfg.seed, synth.IDX_K, g, s)
    vals = synth.e2m1_bytes(kk, np.arange(n * DI // 2, dtype=np.uint64)).reshape(n, DI // 2)
    if cfg.kscale_pow2:
        ks = synth.stream_key(cfg.seed, synth.IDX_K_SCALE, g, s)
        scales = synth.scale_pow2_bytes(ks, np.arange(n * DI // 16, dtype=np.uint64)
                                        ).reshape(n, DI // 16)
    else:
        scales = np.full((n, DI // 16), synth.E4M3_ONE, np.uint8)
    pos, rv, rs = plants(cfg, g, s)
    for p in pos:
        if p < n:
            vals[p], scales[p] = rv, rs
    return vals, scales
