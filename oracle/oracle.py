"""CSA2 CPU oracle, Python side — TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper around ``oracle.c`` (plain C, fp64). Only the tests, the
smoke check and the bench's CPU-baseline leg import this module; the product
path never does. ``build()`` compiles the C library with gcc (no CUDA, no code
shared with the product).

Sources are cited per function in ``oracle.h``: the "DeepSeek-V4.1-Flash-NVFP4"
walkthrough (lpnh.cn) §三, §3.1-§3.4, §四 and the "CSA2稀疏注意力、384专家MoE与1M上下文"
config walkthrough (nxmr.cn) §2.1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile liboracle.so (gcc, -O2, no FP contraction so x86 and Arm agree)."""
    stale = (not os.path.exists(_SO)) or any(
        os.path.getmtime(p) > os.path.getmtime(_SO) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.orc_e2m1_value.restype = ctypes.c_double
            L.orc_e2m1_value.argtypes = [ctypes.c_int]
            L.orc_e4m3_value.restype = ctypes.c_double
            L.orc_e4m3_value.argtypes = [ctypes.c_int]
            L.orc_e4m3_encode.restype = ctypes.c_int
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_e2m1_encode.restype = ctypes.c_int
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]
            L.orc_nvfp4_quantize.restype = None
            L.orc_nvfp4_quantize.argtypes = [_f32p, ctypes.c_int64, _u8p, _u8p]
            L.orc_nvfp4_value.restype = ctypes.c_double
            L.orc_nvfp4_value.argtypes = [_u8p, _u8p, ctypes.c_int64]
            L.orc_pool.restype = ctypes.c_float
            L.orc_pool.argtypes = [ctypes.c_float] * 4
            L.orc_compress_append.restype = ctypes.c_int64
            L.orc_compress_append.argtypes = [
                ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p, _f32p,
                _f32p, _f32p, _u8p, _u8p, _f32p, _u8p, _f32p]
            L.orc_compress_append_ratio.restype = ctypes.c_int64
            L.orc_compress_append_ratio.argtypes = [
                ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p,
                _f32p, _f32p, _f32p, _u8p, _u8p, _f32p, _u8p, _f32p]
            L.orc_rope_freqs.restype = None
            L.orc_rope_freqs.argtypes = [ctypes.POINTER(Rope), _f64p]
            L.orc_rope_rotate.restype = None
            L.orc_rope_rotate.argtypes = [_f32p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.POINTER(Rope)]
            L.orc_compress_row.restype = None
            L.orc_compress_row.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int64, _f32p, _f32p, _f32p, _f32p,
                ctypes.POINTER(Rope), _u8p, _u8p, _f32p]
            L.orc_compress_append_rope.restype = ctypes.c_int64
            L.orc_compress_append_rope.argtypes = [
                ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(Rope), _f32p, _f32p, _f32p, _f32p, _u8p, _u8p, _f32p, _u8p, _f32p]
            L.orc_index_scores.restype = ctypes.c_int64
            L.orc_index_scores.argtypes = [
                ctypes.c_int, ctypes.c_int, _u8p, _u8p, _f32p, ctypes.c_int64, _u8p, _u8p, _f32p]
            L.orc_block_max.restype = None
            L.orc_block_max.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int, _f32p]
            L.orc_select.restype = ctypes.c_int
            L.orc_select.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _i32p]
            L.orc_sparse_attn.restype = ctypes.c_int
            L.orc_sparse_attn.argtypes = [
                ctypes.c_int, ctypes.c_int, _f64p, _f64p, ctypes.c_double, ctypes.c_int64,
                ctypes.c_int, _u8p, _f32p, _u8p, _u8p, _f32p, _i32p, ctypes.c_int, _f64p]
            L.orc_nvfp4_payload_bytes.restype = ctypes.c_int64
            L.orc_nvfp4_payload_bytes.argtypes = [ctypes.c_int64, ctypes.c_int]
            L.orc_nvfp4_scale_bytes.restype = ctypes.c_int64
            L.orc_nvfp4_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int]
            _lib = L
    return _lib


class Rope(ctypes.Structure):
    """orc_rope: the compressed KV's rotary embedding (oracle.h)."""
    _fields_ = [("dim", ctypes.c_int), ("base", ctypes.c_double), ("factor", ctypes.c_double),
                ("orig_len", ctypes.c_double), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double)]


def rope_config(dim=64, base=160000.0, factor=16.0, orig_len=65536.0, beta_fast=32.0,
                beta_slow=1.0) -> Rope:
    """The pages' compressed-KV rotary setting ("CSA2稀疏注意力、384专家MoE与1M上下文" §2.2
    compress_rope_theta, §四 rope_scaling; "DeepSeek-V4.1-Flash-NVFP4" §3.2), with the
    rotated width as a reading (default: the last 64 dims)."""
    return Rope(dim, base, factor, orig_len, beta_fast, beta_slow)


def _rp(rope):
    return ctypes.byref(rope) if rope is not None else ctypes.cast(None, ctypes.POINTER(Rope))


def _p(a, typ):
    if a is None:
        return ctypes.cast(None, typ)
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(typ)


# --------------------------------------------------------------------------- formats
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e4m3_encode(x: float) -> int:
    return lib().orc_e4m3_encode(float(x))


def e2m1_encode(x: float) -> int:
    return lib().orc_e2m1_encode(float(x))


def nvfp4_quantize(x: np.ndarray):
    """fp32 [..., 16k] -> (values uint8 [..., 8k], scales uint8 [..., k])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape[-1] % 16 == 0
    g = x.size // 16
    vals = np.zeros(x.shape[:-1] + (x.shape[-1] // 2,), np.uint8)
    scales = np.zeros(x.shape[:-1] + (x.shape[-1] // 16,), np.uint8)
    lib().orc_nvfp4_quantize(_p(x, _f32p), g, _p(vals, _u8p), _p(scales, _u8p))
    return vals, scales


def nvfp4_dequant(vals: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """NVFP4 rows -> fp64 values (element by element through the oracle)."""
    vals = np.ascontiguousarray(vals, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    n_el = vals.shape[-1] * 2
    rows = vals.reshape(-1, vals.shape[-1])
    srows = scales.reshape(-1, scales.shape[-1])
    out = np.empty((rows.shape[0], n_el), np.float64)
    L = lib()
    for r in range(rows.shape[0]):
        vr = np.ascontiguousarray(rows[r])
        sr = np.ascontiguousarray(srows[r])
        for i in range(n_el):
            out[r, i] = L.orc_nvfp4_value(_p(vr, _u8p), _p(sr, _u8p), i)
    return out.reshape(vals.shape[:-1] + (n_el,))


def pool(kv0: float, kv1: float, g0: float, g1: float) -> float:
    return lib().orc_pool(float(kv0), float(kv1), float(g0), float(g1))


# --------------------------------------------------------------------------- rotary
def rope_freqs(rope: Rope) -> np.ndarray:
    th = np.zeros(rope.dim // 2, np.float64)
    lib().orc_rope_freqs(ctypes.byref(rope), _p(th, _f64p))
    return th


def rope_rotate(x: np.ndarray, pos: int, rope: Rope) -> np.ndarray:
    """Rotated copy of the fp32 row(s) x [..., D] at raw position pos."""
    x = np.array(x, dtype=np.float32, copy=True).reshape(-1, np.shape(x)[-1])
    for r in range(x.shape[0]):
        row = np.ascontiguousarray(x[r])
        lib().orc_rope_rotate(_p(row, _f32p), row.size, int(pos), ctypes.byref(rope))
        x[r] = row
    return x.reshape(np.shape(x)) if x.shape[0] > 1 else x[0]


def compress_row(j: int, kv, g=None, ratio: int = 2, rope: Rope | None = None, f32=False):
    """Compressed row j from its raw tokens kv [ratio, D] (and gates g [2, D] at
    ratio 2): -> fp32 [D] when f32, else (vals [D/2], scales [D/16])."""
    kv = np.ascontiguousarray(kv, np.float32).reshape(ratio, -1)
    D = kv.shape[1]
    if ratio == 2:
        g = np.ascontiguousarray(g, np.float32).reshape(2, D)
        k0, k1, g0, g1 = (np.ascontiguousarray(a) for a in (kv[0], kv[1], g[0], g[1]))
    else:
        k0, k1, g0, g1 = np.ascontiguousarray(kv[0]), None, None, None
    vals = None if f32 else np.zeros(D // 2, np.uint8)
    scales = None if f32 else np.zeros(D // 16, np.uint8)
    out = np.zeros(D, np.float32) if f32 else None
    lib().orc_compress_row(D, ratio, int(j), _p(k0, _f32p), _p(k1, _f32p), _p(g0, _f32p),
                           _p(g1, _f32p), _rp(rope), _p(vals, _u8p), _p(scales, _u8p),
                           _p(out, _f32p))
    return out if f32 else (vals, scales)


# --------------------------------------------------------------------------- compressor
class SeqState:
    """One sequence's cache for one layer, as the oracle keeps it (host arrays)."""

    def __init__(self, cap_comp: int, D: int = 512, W: int = 128,
                 comp_f32: bool = False, win_f32: bool = False, has_comp: bool = True,
                 ratio: int = 2, rope: Rope | None = None):
        """ratio 2: the 2:1 pooled layers; ratio 1: the 1:1 layers (pooling skipped);
        rope: rotate each compressed row at its raw position (None: rows unrotated)."""
        assert ratio in (1, 2)
        self.D, self.W, self.T, self.ratio, self.rope = D, W, 0, ratio, rope
        self.pend_kv = np.zeros(D, np.float32)
        self.pend_g = np.zeros(D, np.float32)
        self.comp_f32 = np.zeros((cap_comp, D), np.float32) if (has_comp and comp_f32) else None
        self.comp_vals = (np.zeros((cap_comp, D // 2), np.uint8)
                          if (has_comp and not comp_f32) else None)
        self.comp_scales = (np.zeros((cap_comp, D // 16), np.uint8)
                            if (has_comp and not comp_f32) else None)
        self.win_f32 = np.zeros((W, D), np.float32) if win_f32 else None
        self.win_u8 = None if win_f32 else np.zeros((W, D), np.uint8)

    def append(self, kv: np.ndarray, g: np.ndarray | None):
        kv = np.ascontiguousarray(kv, dtype=np.float32).reshape(-1, self.D)
        if g is not None:
            g = np.ascontiguousarray(g, dtype=np.float32).reshape(-1, self.D)
        self.T = lib().orc_compress_append_rope(
            self.T, kv.shape[0], self.D, self.W, self.ratio, _rp(self.rope), _p(kv, _f32p),
            _p(g, _f32p),
            _p(self.pend_kv, _f32p), _p(self.pend_g, _f32p), _p(self.comp_vals, _u8p),
            _p(self.comp_scales, _u8p), _p(self.comp_f32, _f32p), _p(self.win_u8, _u8p),
            _p(self.win_f32, _f32p))

    @property
    def n_comp(self) -> int:
        return self.T // self.ratio


# --------------------------------------------------------------------------- indexer
def index_scores(q_vals, q_scales, w, k_vals, k_scales):
    """-> (scores fp32 [n_c], number of scores not guaranteed exact in fp32)."""
    q_vals = np.ascontiguousarray(q_vals, np.uint8)
    q_scales = np.ascontiguousarray(q_scales, np.uint8)
    w = np.ascontiguousarray(w, np.float32)
    k_vals = np.ascontiguousarray(k_vals, np.uint8)
    k_scales = np.ascontiguousarray(k_scales, np.uint8)
    Hi, Di = q_vals.shape[0], q_vals.shape[1] * 2
    n_c = k_vals.shape[0]
    scores = np.zeros(n_c, np.float32)
    inexact = lib().orc_index_scores(Hi, Di, _p(q_vals, _u8p), _p(q_scales, _u8p), _p(w, _f32p),
                                     n_c, _p(k_vals, _u8p), _p(k_scales, _u8p),
                                     _p(scores, _f32p))
    return scores, int(inexact)


def block_max(scores, blk: int = 8):
    scores = np.ascontiguousarray(scores, np.float32)
    n_b = (scores.size + blk - 1) // blk
    out = np.zeros(n_b, np.float32)
    lib().orc_block_max(_p(scores, _f32p), scores.size, blk, _p(out, _f32p))
    return out


def select(scores, blk: int = 8, Kb: int = 2048, Kp: int = 512):
    """-> (idx int32 [Kp] ascending, -1 padded; number valid)."""
    scores = np.ascontiguousarray(scores, np.float32)
    idx = np.full(Kp, -1, np.int32)
    n = lib().orc_select(_p(scores, _f32p), scores.size, blk, Kb, Kp, _p(idx, _i32p))
    return idx, int(n)


# --------------------------------------------------------------------------- attention
def sparse_attn(q, sink, scale, T, W, win_u8=None, win_f32=None, comp_vals=None,
                comp_scales=None, comp_f32=None, idx=None):
    """q fp64-convertible [H, D] -> (out fp64 [H, D], number of attended positions)."""
    q = np.ascontiguousarray(q, np.float64)
    sink = np.ascontiguousarray(sink, np.float64)
    H, D = q.shape
    idx = np.ascontiguousarray(idx if idx is not None else np.zeros(0, np.int32), np.int32)
    out = np.zeros((H, D), np.float64)
    conv = lambda a, t: None if a is None else np.ascontiguousarray(a, t)
    win_u8, win_f32 = conv(win_u8, np.uint8), conv(win_f32, np.float32)
    comp_vals, comp_scales = conv(comp_vals, np.uint8), conv(comp_scales, np.uint8)
    comp_f32 = conv(comp_f32, np.float32)
    n = lib().orc_sparse_attn(H, D, _p(q, _f64p), _p(sink, _f64p), float(scale), int(T), W,
                              _p(win_u8, _u8p), _p(win_f32, _f32p), _p(comp_vals, _u8p),
                              _p(comp_scales, _u8p), _p(comp_f32, _f32p), _p(idx, _i32p),
                              idx.size, _p(out, _f64p))
    return out, int(n)


def nvfp4_payload_bytes(n: int, D: int = 512) -> int:
    return lib().orc_nvfp4_payload_bytes(n, D)


def nvfp4_scale_bytes(n: int, D: int = 512) -> int:
    return lib().orc_nvfp4_scale_bytes(n, D)
