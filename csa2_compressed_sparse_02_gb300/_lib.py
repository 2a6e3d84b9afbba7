"""ctypes loader for ``libcsa2.so`` (the CUDA kernels). There is no fallback: if
the library is missing or does not load, every call raises."""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libcsa2.so")
SYNTH_PATH = os.path.join(PKG, "libcsa2synth.so")
HEADER = os.path.join(ROOT, "include", "csa2.h")

_lock = threading.Lock()
_lib = None
_synth = None

P = ctypes.c_void_p
I32 = ctypes.c_int
I64 = ctypes.c_int64
SZ = ctypes.c_size_t


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "heads", "head_dim", "index_heads", "index_dim", "window", "block_size", "topk_blocks",
        "topk_pos", "compress_ratio", "kv_format", "win_format", "q_format")] + [
        ("softmax_scale", ctypes.c_float), ("win_layout", ctypes.c_int), ("max_ctas", ctypes.c_int),
        ("rope_dim", ctypes.c_int), ("rope_theta", ctypes.c_float), ("rope_factor", ctypes.c_float),
        ("rope_orig_len", ctypes.c_float), ("rope_beta_fast", ctypes.c_float),
        ("rope_beta_slow", ctypes.c_float)]


PP = ctypes.POINTER(Params)

SIGNATURES = {
    "csa2_default_params": (None, [PP]),
    "csa2_version": (I32, []),
    "csa2_trace_attach": (I32, [P]),
    "csa2_last_error": (ctypes.c_char_p, []),
    "csa2_compress_append": (I32, [PP, I32, I32, P, P, P, P, P, P, P, P, P, P, P]),
    "csa2_nvfp4_quantize": (I32, [P, I64, I32, P, P, P]),
    "csa2_window_linear": (I32, [PP, I32, I32, P, P, P, P, P]),
    "csa2_index_keys_write": (I32, [PP, I32, I64, P, P, P, P, P, P, P]),
    "csa2_index_scores": (I32, [PP, I32, I64, P, P, P, P, P, P, P, P, P]),
    "csa2_index_scores_cuda_cores": (I32, [PP, I32, I64, P, P, P, P, P, P, P, P, P]),
    "csa2_index_scores_shared": (I32, [PP, I32, I64, P, P, P, P, P, P, P, P, P]),
    "csa2_select_topk": (I32, [PP, I32, I64, P, P, P, P, P, P, P]),
    "csa2_sparse_attn_workspace_size": (SZ, [PP, I32]),
    "csa2_sparse_attn": (I32, [PP, I32, P, P, P, P, P, P, P, P, P, SZ, P, P]),
    "csa2_sparse_attn_mma": (I32, [PP, I32, P, P, P, P, P, P, P, P, P, SZ, P, P]),
    "csa2_sparse_attn_noalloc": (I32, [PP, I32, P, P, P, P, P, P, P, P, P, P]),
    "csa2_sparse_attn_layers": (I32, [PP, I32, I32, P, P, P, P, P, P, P, P, P, P]),
    "csa2_sparse_attn_layers_mma": (I32, [PP, I32, I32, P, P, P, P, P, P, P, P, P, P]),
    "csa2_sparse_attn_layers_part": (I32, [PP, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P]),
    "csa2_sparse_attn_layers_split": (I32, [PP, I32, I32, P, P, P, P, P, P, P, P, P, SZ, P, P]),
    "csa2_sparse_attn_layers_split_workspace_size": (SZ, [PP, I32, I32]),
    "csa2_fp4_mma_peak": (I32, [I32, I32, P, P]),
}


class Csa2Error(RuntimeError):
    pass


def header_symbols(path: str = HEADER) -> list[str]:
    """Names of the functions a header declares (for the export check)."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text)))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise Csa2Error("libcsa2.so is not built (run __graft_entry__.build()); "
                                "there is no non-CUDA fallback")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def synth_lib():
    global _synth
    with _lock:
        if _synth is None:
            if not os.path.exists(SYNTH_PATH):
                raise Csa2Error("libcsa2synth.so is not built (run __graft_entry__.build())")
            L = ctypes.CDLL(SYNTH_PATH)
            L.csa2synth_fill.restype = I32
            L.csa2synth_fill.argtypes = [I32, P, I32, ctypes.c_uint64, I64, P, I64, P]
            _synth = L
    return _synth


def check(rc: int, what: str):
    if rc != 0:
        msg = lib().csa2_last_error().decode(errors="replace")
        raise Csa2Error("%s failed (status %d): %s" % (what, rc, msg))
