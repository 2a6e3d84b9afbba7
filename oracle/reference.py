"""Oracle results for one sequence of one decode step — TEST INFRASTRUCTURE ONLY.

Composes the pinned oracle functions (oracle.py) in the order of the path —
Compressor, Indexer, two-level selection, sparse attention ("DeepSeek-V4.1-
Flash-NVFP4" §3.2-§3.4) — on inputs regenerated on the host from the seeded
recipe (csa2_compressed_sparse_02_gb300.inputs, numpy only; no CUDA path).

Only what the step's outputs depend on is recomputed: the compressed rows of
the selected positions (pooling is per pair, so a pair lands in a compact row
of its own; at ratio 1 a position is one raw token) and the window's last W raw
tokens of every attending layer.
"""
from __future__ import annotations

import math
import time
from types import SimpleNamespace

import numpy as np

from csa2_compressed_sparse_02_gb300 import inputs as I

from . import oracle as orc


def index_and_select(cfg, g: int, s: int, step: int):
    """Indexer scores, block maxima and selection of sequence s after `step`."""
    T = cfg.first_lengths()[s] + step
    n_c = T // cfg.ratio
    qv, qs, w = I.host_index_q(cfg, g, s, step)
    kv, ks = I.host_index_keys(cfg, g, s, n_c)
    t0 = time.perf_counter()
    scores, inexact = orc.index_scores(qv, qs, w, kv, ks)
    bm = orc.block_max(scores, 8)
    idx, n_sel = orc.select(scores, 8, 2048, 512)
    return dict(T=T, n_c=n_c, scores=scores, block_max=bm, idx=idx, n_sel=n_sel,
                inexact=inexact, seconds=time.perf_counter() - t0)


def compressed_rows(cfg, layer: int, s: int, positions):
    """Compact cache whose row i is compressed position positions[i] of `layer`:
    each row recomputed from its raw tokens (pooled at ratio 2, rotated at raw
    position ratio*j when the configuration rotates the compressed KV)."""
    rt = cfg.ratio
    rope = orc.rope_config(dim=I.ROPE_DIM) if getattr(cfg, "rope", False) else None
    n = max(1, len(positions))
    st = SimpleNamespace(comp_f32=None, comp_vals=None, comp_scales=None)
    if cfg.quant:
        st.comp_vals = np.zeros((n, I.D // 2), np.uint8)
        st.comp_scales = np.zeros((n, I.D // 16), np.uint8)
    else:
        st.comp_f32 = np.zeros((n, I.D), np.float32)
    for i, j in enumerate(positions):  # position j is raw tokens rt*j .. rt*j + rt - 1
        kv = I.host_kv(cfg, layer, s, rt * j, rt * j + rt)
        g = I.host_gate(cfg, layer, s, rt * j, rt * j + rt) if rt == 2 else None
        row = orc.compress_row(j, kv, g, ratio=rt, rope=rope, f32=not cfg.quant)
        if cfg.quant:
            st.comp_vals[i], st.comp_scales[i] = row
        else:
            st.comp_f32[i] = row
    return st


def window_state(cfg, layer: int, s: int, T: int):
    """Window ring of `layer` holding raw tokens max(0, T-W)..T-1."""
    st = orc.SeqState(cap_comp=1, D=I.D, W=I.W, has_comp=False, win_f32=not cfg.quant)
    t0 = max(0, T - I.W)
    st.T = t0
    if T > t0:
        st.append(I.host_kv(cfg, layer, s, t0, T), None)
    return st


def attention(cfg, g: int, r: int, s: int, step: int, sel, comp_state):
    """Sparse attention of layer (g, r) for sequence s; sel = selected positions."""
    T = cfg.first_lengths()[s] + step
    layer = cfg.layer(g, r)
    win = window_state(cfg, layer, s, T)
    q = I.host_q(cfg, layer, s, step)
    sink = I.host_sink(cfg, layer).astype(np.float64)
    compact = np.arange(len(sel), dtype=np.int32)
    out, n = orc.sparse_attn(q, sink, 1.0 / math.sqrt(I.D), T, I.W, win_u8=win.win_u8,
                             win_f32=win.win_f32, comp_vals=comp_state.comp_vals,
                             comp_scales=comp_state.comp_scales, comp_f32=comp_state.comp_f32,
                             idx=compact)
    return out, n


def decode_step(cfg, g: int, s: int, step: int, readers=None):
    """Everything one decode step produces for sequence s of group g."""
    res = index_and_select(cfg, g, s, step)
    sel = [int(j) for j in res["idx"][:res["n_sel"]]]
    t0 = time.perf_counter()
    comp = compressed_rows(cfg, cfg.layer(g, 0), s, sel)
    res["out"] = {}
    for r in (range(cfg.readers) if readers is None else readers):
        res["out"][r], res["attended"] = attention(cfg, g, r, s, step, sel, comp)
    res["seconds"] += time.perf_counter() - t0
    return res
