"""C ABI checks that need no GPU: the library loads, exports every function
include/*.h declares, and rejects bad arguments on the host before touching
CUDA (no compute call is made here)."""
import ctypes
import glob
import os

import pytest

from csa2_compressed_sparse_02_gb300 import _lib, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return _lib.lib()


def test_every_declared_symbol_is_exported(L):
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names += _lib.header_symbols(h)
    assert names, "no declarations found"
    raw = ctypes.CDLL(_lib.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    assert set(names) >= set(_lib.SIGNATURES)


def test_defaults_are_the_pages_sizes(L):
    p = api.default_params()
    assert (p.heads, p.head_dim, p.index_heads, p.index_dim, p.window, p.block_size,
            p.topk_blocks, p.topk_pos, p.compress_ratio) == (64, 512, 32, 128, 128, 8, 2048, 512, 2)
    assert abs(p.softmax_scale - 512 ** -0.5) < 1e-8
    assert (p.kv_format, p.win_format, p.q_format) == (api.NVFP4, api.E4M3, api.BF16)
    # compressed-KV rotary setting: config walkthrough §2.2 (compress_rope_theta) and §四
    # (YaRN factor 16 over 65536, beta_fast 32, beta_slow 1); off by default
    assert (p.rope_dim, p.rope_theta, p.rope_factor, p.rope_orig_len, p.rope_beta_fast,
            p.rope_beta_slow) == (0, 160000.0, 16.0, 65536.0, 32.0, 1.0)


def test_workspace_size_covers_split_partials(L):
    p = api.default_params()
    assert api.sparse_attn_workspace_size(p, 0) == 0
    assert api.sparse_attn_workspace_size(p, 32) >= 32 * 5 * 64 * 512 * 4


def test_host_side_rejections_without_launching(L):
    p = api.default_params()
    pp = ctypes.byref(p)
    assert L.csa2_compress_append(pp, -1, 1, *([None] * 11)) == 1
    assert L.csa2_compress_append(None, 1, 1, *([None] * 11)) == 1
    assert "params" in L.csa2_last_error().decode()
    assert L.csa2_index_scores(pp, 1, 10, *([None] * 9)) == 1  # NULL buffers
    assert L.csa2_index_scores_cuda_cores(pp, 1, 10, *([None] * 9)) == 1
    bad = api.default_params(index_heads=16)
    assert L.csa2_index_scores(ctypes.byref(bad), 1, 10, *([None] * 9)) == 4
    # more sequences than one launch takes (grid.y of the CUDA-core build): rejected
    # before anything is enqueued; the buffers are host memory, never dereferenced
    buf = (ctypes.c_uint8 * 64)()
    base = ctypes.addressof(buf)
    al = ctypes.c_void_p((base + 15) & ~15)
    for fn in (L.csa2_index_scores, L.csa2_index_scores_cuda_cores):
        assert fn(pp, 65536, 10, al, al, al, al, al, al, al, None, None) == 4
        assert "65535" in L.csa2_last_error().decode()
    bad_dim = api.default_params(index_dim=64)
    assert L.csa2_index_keys_write(ctypes.byref(bad_dim), 1, 4, *([None] * 7)) == 4
    assert L.csa2_index_keys_write(pp, 1, 4, *([None] * 7)) == 1
    bad = api.default_params(topk_pos=256)
    assert L.csa2_select_topk(ctypes.byref(bad), 1, 10, *([None] * 7)) == 4
    assert L.csa2_sparse_attn(pp, 1, *([None] * 8), None, 0, None, None) == 1
    assert L.csa2_nvfp4_quantize(None, 4, 24, None, None, None) == 2  # row_len % 16
    assert L.csa2_sparse_attn_layers(pp, 2, 4, *([None] * 10)) == 1  # NULL buffers
    assert L.csa2_sparse_attn_layers_part(pp, 2, 4, 3, 2, *([None] * 10)) == 1  # range past B
    assert L.csa2_sparse_attn_layers_part(pp, 2, 4, -1, 1, *([None] * 10)) == 1
    assert L.csa2_sparse_attn_layers_part(pp, 2, 4, 1, 0, *([None] * 10)) == 0  # empty range
    bad_ratio = api.default_params(compress_ratio=3)
    assert L.csa2_compress_append(ctypes.byref(bad_ratio), 1, 1, *([None] * 11)) == 4
    # rotary settings the Compressor is not built for, rejected before any launch
    # (the buffers are host memory, never dereferenced)
    for over, code in ((dict(rope_dim=62), 4), (dict(rope_dim=1024), 4), (dict(rope_dim=-4), 4),
                       (dict(rope_dim=64, rope_beta_fast=0.5), 1),
                       (dict(rope_dim=64, rope_theta=0.0), 1)):
        bp = api.default_params(**over)
        assert L.csa2_compress_append(ctypes.byref(bp), 1, 1, al, None, None, None, None, None,
                                      None, al, al, None, None) == code, over
    # the FP4 MMA rate measurement rejects empty or oversized launches on the host
    assert L.csa2_fp4_mma_peak(0, 10, None, None) == 1
    assert L.csa2_fp4_mma_peak(4, 0, None, None) == 1
    assert L.csa2_fp4_mma_peak(4, (1 << 22) + 1, None, None) == 1
    # nothing to do is not an error
    assert L.csa2_compress_append(pp, 0, 1, *([None] * 11)) == 0
