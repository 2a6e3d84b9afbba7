"""Python binding of the CSA2 C ABI (``include/csa2.h``): argument marshalling only.

Every function has the ABI call's name without the ``csa2_`` prefix, takes
torch CUDA tensors, passes their device pointers and the current CUDA stream,
and raises ``Csa2Error`` on a non-zero status. All arithmetic runs in the CUDA
kernels of ``libcsa2.so``; nothing here computes on the data.

``LayerCache`` and ``IndexKeyCache`` allocate one layer's per-sequence buffers
with PyTorch (device memory is PyTorch's job) and build the device arrays of
per-sequence base pointers the ABI takes.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from ._lib import Csa2Error, Params, check, lib  # noqa: F401

F32, NVFP4, E4M3, BF16 = 0, 1, 2, 3
WIN_RING, WIN_LINEAR = 0, 1
D, H, HI, DI, W, BLK, KB, KP = 512, 64, 32, 128, 128, 8, 2048, 512
KEY_TILE, KEY_TILE_BYTES = 128, 9216


def default_params(**over) -> Params:
    p = Params()
    lib().csa2_default_params(ctypes.byref(p))
    for k, v in over.items():
        setattr(p, k, v)
    return p


def version() -> int:
    return lib().csa2_version()


TRACE_KERNELS = {0: "none", 1: "compress_append", 2: "index_scores", 3: "select_topk",
                 4: "sparse_attn_layers"}


def trace_attach():
    """Attach a zeroed pinned record to the library's launch trace (csa2_trace_attach)
    and return it; read it with trace_read() after an error."""
    rec = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    check(lib().csa2_trace_attach(ctypes.c_void_p(rec.data_ptr())), "trace_attach")
    return rec


def trace_read(rec) -> str:
    """The trace record as text: the last launch that started and the last whose
    first CTA finished."""
    v = [int(x) for x in rec.tolist()]
    return "last launch started: %s #%d; last first-CTA finish: %s #%d" % (
        TRACE_KERNELS.get(v[0], str(v[0])), v[1], TRACE_KERNELS.get(v[2], str(v[2])), v[3])


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise Csa2Error("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def ptr_array(tensors, device=None) -> torch.Tensor:
    """Device int64 array of the base addresses of `tensors` (one per sequence)."""
    addrs = [t.data_ptr() for t in tensors]
    dev = device or tensors[0].device
    return torch.tensor(addrs, dtype=torch.int64, device=dev)


# --------------------------------------------------------------------------- calls
def compress_append(params, kv_new, gate_new, pend_kv, pend_gate, comp_ptrs, comp_scale_ptrs,
                    comp_cap, win_ptrs, n_tokens, dev_status=None, stream=None):
    B = n_tokens.numel()
    n_new = kv_new.shape[1] if kv_new.dim() == 3 else 0
    check(lib().csa2_compress_append(
        ctypes.byref(params), B, n_new, _ptr(kv_new), _ptr(gate_new), _ptr(pend_kv),
        _ptr(pend_gate), _ptr(comp_ptrs), _ptr(comp_scale_ptrs), _ptr(comp_cap), _ptr(win_ptrs),
        _ptr(n_tokens), _ptr(dev_status), _stream(stream)), "compress_append")


def window_linear(params, kv_new, win_ptrs, n_tokens, out, stream=None):
    """Linear FP8 windows of a prefill chunk (before its append): out [B, W-1+n_new, D]."""
    B, n_new = n_tokens.numel(), kv_new.shape[1]
    check(lib().csa2_window_linear(ctypes.byref(params), B, n_new, _ptr(kv_new), _ptr(win_ptrs),
                                   _ptr(n_tokens), _ptr(out), _stream(stream)), "window_linear")


def nvfp4_quantize(x, vals, scales, stream=None):
    check(lib().csa2_nvfp4_quantize(_ptr(x), x.numel() // x.shape[-1], x.shape[-1], _ptr(vals),
                                    _ptr(scales), _stream(stream)), "nvfp4_quantize")


def index_keys_write(params, vals, scales, pos0, dst_ptrs, cap, dev_status=None, stream=None):
    """Plain NVFP4 index keys vals [B, n, 64] / scales [B, n, 8] -> tiled caches."""
    B, n = vals.shape[0], vals.shape[1]
    check(lib().csa2_index_keys_write(
        ctypes.byref(params), B, n, _ptr(vals), _ptr(scales), _ptr(pos0), _ptr(dst_ptrs),
        _ptr(cap), _ptr(dev_status), _stream(stream)), "index_keys_write")


def index_scores(params, max_ncomp, q_vals, q_scales, w, key_cache_ptrs, n_tokens, scores,
                 block_max, dev_status=None, stream=None, cuda_cores=False):
    B = n_tokens.numel()
    f = lib().csa2_index_scores_cuda_cores if cuda_cores else lib().csa2_index_scores
    check(f(ctypes.byref(params), B, max_ncomp, _ptr(q_vals), _ptr(q_scales), _ptr(w),
            _ptr(key_cache_ptrs), _ptr(n_tokens), _ptr(scores), _ptr(block_max), _ptr(dev_status),
            _stream(stream)), "index_scores")


def index_scores_shared(params, max_ncomp, q_vals, q_scales, w, key_cache, n_tokens, scores,
                        block_max, dev_status=None, stream=None):
    """Q queries against ONE tiled key cache (a uint8 device tensor): the prefill
    Indexer. q_vals [Q,32,64], q_scales [Q,32,8], w [Q,32], n_tokens [Q]."""
    Q = n_tokens.numel()
    check(lib().csa2_index_scores_shared(
        ctypes.byref(params), Q, max_ncomp, _ptr(q_vals), _ptr(q_scales), _ptr(w), _ptr(key_cache),
        _ptr(n_tokens), _ptr(scores), _ptr(block_max), _ptr(dev_status), _stream(stream)),
        "index_scores_shared")


def select_topk(params, max_ncomp, scores, block_max, n_tokens, idx, n_sel=None, dev_status=None,
                stream=None):
    B = n_tokens.numel()
    check(lib().csa2_select_topk(
        ctypes.byref(params), B, max_ncomp, _ptr(scores), _ptr(block_max), _ptr(n_tokens),
        _ptr(idx), _ptr(n_sel), _ptr(dev_status), _stream(stream)), "select_topk")


def sparse_attn_workspace_size(params, B) -> int:
    return lib().csa2_sparse_attn_workspace_size(ctypes.byref(params), B)


def sparse_attn(params, q, sink, win_ptrs, n_tokens, comp_ptrs, comp_scale_ptrs, idx, out,
                workspace, dev_status=None, stream=None, mma_sync=False):
    """One layer (csa2_sparse_attn: tcgen05 for the quantised formats); mma_sync=True
    runs the legacy mma.sync split-KV implementation (csa2_sparse_attn_mma)."""
    B = n_tokens.numel()
    fn = lib().csa2_sparse_attn_mma if mma_sync else lib().csa2_sparse_attn
    check(fn(
        ctypes.byref(params), B, _ptr(q), _ptr(sink), _ptr(win_ptrs), _ptr(n_tokens),
        _ptr(comp_ptrs), _ptr(comp_scale_ptrs), _ptr(idx), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)),
        "sparse_attn_mma" if mma_sync else "sparse_attn")


def sparse_attn_layers_split_workspace(params, L, B, device="cuda"):
    """Zero-filled workspace for sparse_attn_layers(..., workspace=...) on the
    current device (one partial-result slot per CTA boundary + the counts)."""
    n = lib().csa2_sparse_attn_layers_split_workspace_size(ctypes.byref(params), L, B)
    return torch.zeros(max(int(n), 256), dtype=torch.uint8, device=device)


def sparse_attn_layers(params, q, sink, win_ptrs, n_tokens, comp_ptrs, comp_scale_ptrs, idx, out,
                       dev_status=None, stream=None, mma_sync=False, workspace=None):
    """L layers sharing one compressed cache and selection: q/out [L, B, H, D] bf16,
    sink [L, H], win_ptrs [L*B] (layer-major), n_tokens [B]. mma_sync=True runs
    the legacy warp-level tensor-core implementation of the same contract. With a
    workspace (sparse_attn_layers_split_workspace) the tcgen05 path spreads the
    (unit, tile) work evenly over the CTAs (csa2_sparse_attn_layers_split)."""
    L, B = q.shape[0], q.shape[1]
    if workspace is not None and not mma_sync:
        check(lib().csa2_sparse_attn_layers_split(
            ctypes.byref(params), L, B, _ptr(q), _ptr(sink), _ptr(win_ptrs), _ptr(n_tokens),
            _ptr(comp_ptrs), _ptr(comp_scale_ptrs), _ptr(idx), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)),
            "sparse_attn_layers_split")
        return
    fn = lib().csa2_sparse_attn_layers_mma if mma_sync else lib().csa2_sparse_attn_layers
    check(fn(
        ctypes.byref(params), L, B, _ptr(q), _ptr(sink), _ptr(win_ptrs), _ptr(n_tokens),
        _ptr(comp_ptrs), _ptr(comp_scale_ptrs), _ptr(idx), _ptr(out), _ptr(dev_status),
        _stream(stream)), "sparse_attn_layers_mma" if mma_sync else "sparse_attn_layers")


def sparse_attn_layers_part(params, b0, nb, q, sink, win_ptrs, n_tokens, comp_ptrs, comp_scale_ptrs,
                            idx, out, dev_status=None, stream=None):
    """sparse_attn_layers for the sequences [b0, b0 + nb) only; every array keeps
    its full-batch shape (q/out [L, B, H, D], win_ptrs [L*B], n_tokens [B], ...)."""
    L, B = q.shape[0], q.shape[1]
    check(lib().csa2_sparse_attn_layers_part(
        ctypes.byref(params), L, B, b0, nb, _ptr(q), _ptr(sink), _ptr(win_ptrs), _ptr(n_tokens),
        _ptr(comp_ptrs), _ptr(comp_scale_ptrs), _ptr(idx), _ptr(out), _ptr(dev_status),
        _stream(stream)), "sparse_attn_layers_part")


def sparse_attn_noalloc(params, q, sink, win_ptrs, n_tokens, comp_ptrs, comp_scale_ptrs, idx, out,
                        dev_status=None, stream=None):
    """csa2_sparse_attn without a workspace: for callers that cannot allocate device
    memory (their HBM already belongs to an engine's pool, or an allocation would
    synchronise a latency-critical path). At most 32 sequences per call; calls that
    overlap on the GPU share the library's one scratch array and must be ordered."""
    B = n_tokens.numel()
    check(lib().csa2_sparse_attn_noalloc(
        ctypes.byref(params), B, _ptr(q), _ptr(sink), _ptr(win_ptrs), _ptr(n_tokens),
        _ptr(comp_ptrs), _ptr(comp_scale_ptrs), _ptr(idx), _ptr(out), _ptr(dev_status),
        _stream(stream)), "sparse_attn_noalloc")


def fp4_mma_peak(ctas, iters, dev_status=None, stream=None):
    """Enqueue the FP4 tensor-core rate measurement (csa2_fp4_mma_peak): ctas x iters
    MMA pairs of 2 x 128 x 128 x 128 flop each. The caller times it."""
    check(lib().csa2_fp4_mma_peak(int(ctas), int(iters), _ptr(dev_status), _stream(stream)),
          "fp4_mma_peak")


# --------------------------------------------------------------------------- buffers
@dataclass
class LayerCache:
    """One layer's per-sequence state: compressed cache (NVFP4 or fp32, absent
    for window-only layers), ring window, pending half-pair, token counts."""
    B: int
    caps: list
    params: Params
    has_comp: bool = True
    device: str = "cuda"

    def __post_init__(self):
        dev, B, p = self.device, self.B, self.params
        nv = p.kv_format == NVFP4
        self.comp, self.comp_scales = [], []
        if self.has_comp:
            for cap in self.caps:
                cap = max(1, int(cap))
                if nv:
                    self.comp.append(torch.zeros(cap, D // 2, dtype=torch.uint8, device=dev))
                    self.comp_scales.append(torch.zeros(cap, D // 16, dtype=torch.uint8, device=dev))
                else:
                    self.comp.append(torch.zeros(cap, D, dtype=torch.float32, device=dev))
        wdt = torch.uint8 if p.win_format == E4M3 else torch.float32
        self.win = torch.zeros(B, W, D, dtype=wdt, device=dev)
        self.pend_kv = torch.zeros(B, D, dtype=torch.float32, device=dev)
        self.pend_gate = torch.zeros(B, D, dtype=torch.float32, device=dev)
        self.n_tokens = torch.zeros(B, dtype=torch.int32, device=dev)
        self.comp_cap = torch.tensor([max(1, int(c)) for c in self.caps], dtype=torch.int64,
                                     device=dev)
        self.comp_ptrs = ptr_array(self.comp) if self.has_comp else None
        self.comp_scale_ptrs = ptr_array(self.comp_scales) if (self.has_comp and nv) else None
        self.win_ptrs = ptr_array(list(self.win.unbind(0)))

    def append(self, kv_new, gate_new=None, dev_status=None, stream=None):
        compress_append(self.params, kv_new, gate_new if self.has_comp else None,
                        self.pend_kv if self.has_comp else None,
                        self.pend_gate if self.has_comp else None,
                        self.comp_ptrs, self.comp_scale_ptrs,
                        self.comp_cap if self.has_comp else None, self.win_ptrs, self.n_tokens,
                        dev_status, stream)

    def shares_compressed_cache_of(self, other: "LayerCache"):
        """Point this (window-only) layer's compressed-cache arrays at `other`'s."""
        self.comp_ptrs, self.comp_scale_ptrs = other.comp_ptrs, other.comp_scale_ptrs


@dataclass
class IndexKeyCache:
    """Per-sequence tiled FP4 index-key caches (include/csa2.h layout): ceil(cap/128)
    tiles of 9216 bytes each."""
    caps: list
    device: str = "cuda"

    def __post_init__(self):
        self.tiles = [max(1, -(-int(c) // KEY_TILE)) for c in self.caps]
        self.buf = [torch.zeros(t * KEY_TILE_BYTES, dtype=torch.uint8, device=self.device)
                    for t in self.tiles]
        self.ptrs = ptr_array(self.buf)
        self.cap = torch.tensor([t * KEY_TILE for t in self.tiles], dtype=torch.int64,
                                device=self.device)

    def write(self, params, vals, scales, pos0, dev_status=None, stream=None):
        """Write plain rows vals [B, n, 64], scales [B, n, 8] at positions pos0[b]..."""
        index_keys_write(params, vals, scales, pos0, self.ptrs, self.cap, dev_status, stream)

    def write_seq(self, params, b, vals, scales, pos0=0, dev_status=None, stream=None):
        """Write plain rows [n, 64] / [n, 8] of one sequence starting at pos0."""
        p0 = torch.tensor([pos0], dtype=torch.int64, device=self.device)
        index_keys_write(params, vals[None], scales[None], p0, self.ptrs[b:b + 1],
                         self.cap[b:b + 1], dev_status, stream)


def n_blocks(n: int) -> int:
    return math.ceil(n / BLK)
