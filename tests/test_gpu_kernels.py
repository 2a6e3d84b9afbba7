"""GPU parity of each C ABI call against the CPU oracle, element by element, at
sizes that span several tiles and ragged tails, plus edge cases.

Bars: NVFP4 bytes, FP8 window bytes, index scores, block maxima and selected
indices bit-exact; bf16 attention within max|d| <= 1.5e-2 and relative
Frobenius error <= 4e-3 of the fp64 oracle; the fp32 (unquantised) attention
within 1e-4 / 1e-5 (fp32 rounding of 512-term dot products)."""
import math

import numpy as np
import pytest
import torch

from csa2_compressed_sparse_02_gb300 import api, synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
DEV = "cuda"


def t(x, dtype=None):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV) if dtype is None else \
        torch.from_numpy(np.ascontiguousarray(x)).to(DEV, dtype)


def close_bf16(o, e):
    err = np.abs(o - e).max()
    rel = np.linalg.norm(o - e) / max(np.linalg.norm(e), 1e-30)
    return err <= 1.5e-2 and rel <= 4e-3, (err, rel)


# --------------------------------------------------------------------------- quantiser
def test_nvfp4_quantize_bit_exact_on_identical_fp32():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((700, 512)) * rng.choice([1e-4, 1e-2, 1, 100, 3e4], (700, 1))
    grid = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7])
    mid = np.tile(np.concatenate([grid, -grid]), 16)[:512] * 0.375  # ties after scaling
    special = np.stack([np.zeros(512), mid, mid * 3, np.full(512, 1e30), np.full(512, 1e-30),
                        -np.zeros(512), np.nextafter(mid, 10), np.nextafter(mid, -10)])
    x = np.concatenate([x, special]).astype(np.float32)
    vals = torch.empty(x.shape[0], 256, dtype=torch.uint8, device=DEV)
    scales = torch.empty(x.shape[0], 32, dtype=torch.uint8, device=DEV)
    api.nvfp4_quantize(t(x), vals, scales)
    torch.cuda.synchronize()
    rv, rs = orc.nvfp4_quantize(x)
    assert np.array_equal(scales.cpu().numpy(), rs)
    gv = vals.cpu().numpy()
    bad = np.argwhere(gv != rv)
    assert bad.size == 0, (bad[:4], gv[tuple(bad[0])] if bad.size else None)


# --------------------------------------------------------------------------- compressor
def _oracle_states(kv_chunks, g_chunks, B, caps, f32):
    st = [orc.SeqState(cap_comp=caps[b], D=512, W=128, comp_f32=f32, win_f32=f32) for b in range(B)]
    for kv, g in zip(kv_chunks, g_chunks):
        for b in range(B):
            st[b].append(kv[b], g[b])
    return st


def _pool_error_bound(kv0, kv1):
    """fp32 pooling error bound: 8 ulp of the larger term (expf, product, sum and
    divide roundings) (the pooled value
    itself can be far smaller when the two tokens cancel)."""
    m = np.maximum(np.abs(kv0), np.abs(kv1)).astype(np.float32)
    return 8 * np.spacing(m)


def _near_boundary_flip_ok(c_ref_group, bound, gpu_vals8, gpu_scale):
    """The GPU's bytes equal the oracle's after moving one element by at most its
    fp32 pooling error bound."""
    for i in range(16):
        for f in np.linspace(-1.0, 1.0, 41):
            y = c_ref_group.copy()
            y[i] = np.float32(y[i] + f * bound[i])
            v, s = orc.nvfp4_quantize(y)
            if s[0] == gpu_scale and np.array_equal(v, gpu_vals8):
                return True
    return False


@pytest.mark.parametrize("f32", [False, True])
def test_compress_append_matches_oracle(f32):
    rng = np.random.default_rng(1 if f32 else 2)
    B = 3
    n_news = [1, 1, 2, 7, 300, 1, 129, 34]  # ends on an odd count: a half pair is pending
    total = sum(n_news)
    caps = [total // 2 + 1] * B
    p = api.default_params() if not f32 else api.default_params(
        kv_format=api.F32, win_format=api.F32, q_format=api.F32)
    cache = api.LayerCache(B, caps, p)
    kvs, gs = [], []
    for n in n_news:
        kv = (rng.standard_normal((B, n, 512)) * 2).astype(np.float32)
        g = (rng.standard_normal((B, n, 512)) * 3).astype(np.float32)
        kvs.append(kv)
        gs.append(g)
        cache.append(t(kv), t(g), dev_status=None)
    torch.cuda.synchronize()
    st = _oracle_states(kvs, gs, B, caps, f32)
    assert cache.n_tokens.cpu().tolist() == [total] * B
    n_c = total // 2
    assert total % 2 == 1
    for b in range(B):  # the pending half pair (meaningful only for odd T)
        assert np.array_equal(cache.pend_kv[b].cpu().numpy(), st[b].pend_kv)
        assert np.array_equal(cache.pend_gate[b].cpu().numpy(), st[b].pend_g)
        kv_all = np.concatenate([k[b] for k in kvs])
        g_all = np.concatenate([g[b] for g in gs])
        bound = _pool_error_bound(kv_all[0:2 * n_c:2], kv_all[1:2 * n_c:2])
        if f32:
            got = cache.comp[b][:n_c].cpu().numpy()
            ref = st[b].comp_f32[:n_c]
            err = np.abs(got.astype(np.float64) - ref)
            assert np.all(err <= bound), (err / bound).max()
            assert np.array_equal(cache.win[b].cpu().numpy(), st[b].win_f32)
        else:
            assert np.array_equal(cache.win[b].cpu().numpy(), st[b].win_u8)  # E4M3 of identical fp32
            gv = cache.comp[b][:n_c].cpu().numpy()
            gsc = cache.comp_scales[b][:n_c].cpu().numpy()
            rv, rsc = st[b].comp_vals[:n_c], st[b].comp_scales[:n_c]
            bad_groups = set(map(tuple, np.argwhere(gsc != rsc)))
            bad_groups |= set((int(j), int(c) // 8) for j, c in np.argwhere(gv != rv))
            assert len(bad_groups) <= max(2, n_c * 32 // 2000)
            for j, gi in bad_groups:
                # the oracle's pooled fp32 value of this group, for the nudge test
                c = np.array([orc.pool(kv_all[2 * j, d], kv_all[2 * j + 1, d], g_all[2 * j, d],
                                       g_all[2 * j + 1, d]) for d in range(16 * gi, 16 * gi + 16)],
                             np.float32)
                assert _near_boundary_flip_ok(c, bound[j, 16 * gi:16 * gi + 16],
                                              gv[j, 8 * gi:8 * gi + 8], gsc[j, gi]), (j, gi)


@pytest.mark.parametrize("ratio,T0,f32", [(2, 0, False), (2, 1046528, False), (1, 1046528, False),
                                          (2, 1046528, True)])
def test_compress_append_rope_matches_oracle(ratio, T0, f32):
    """Compressed-KV rotary embedding ("CSA2稀疏注意力、384专家MoE与1M上下文" §2.2, §四;
    "DeepSeek-V4.1-Flash-NVFP4" §3.2): YaRN rotation of the last 64 dims of row j at
    raw position ratio*j, after pooling and before quantising, near 0 and near 1M.
    At ratio 1 the rotation sees identical fp32 inputs; the rotated value may differ
    from the oracle's by one fp32 rounding (both fp64, rounded once), plus the fp32
    pooling error of both pair members at ratio 2; a code may flip only where moving
    the oracle's value by that bound crosses a rounding boundary."""
    rng = np.random.default_rng(30 + ratio + (T0 > 0))
    B = 2
    rope = orc.rope_config(dim=64)
    n_news = [1, 2, 7, 150, 1, 33] if ratio == 2 else [1, 2, 7, 150, 3]
    total = sum(n_news)
    cap = (T0 + total) // ratio + 1
    over = dict(rope_dim=64, compress_ratio=ratio)
    if f32:
        over.update(kv_format=api.F32, win_format=api.F32, q_format=api.F32)
    p = api.default_params(**over)
    cache = api.LayerCache(B, [cap] * B, p)
    cache.n_tokens.fill_(T0)
    kvs, gs = [], []
    for n in n_news:
        kv = (rng.standard_normal((B, n, 512)) * 2).astype(np.float32)
        g = (rng.standard_normal((B, n, 512)) * 3).astype(np.float32)
        kvs.append(kv)
        gs.append(g)
        cache.append(t(kv), t(g) if ratio == 2 else None, dev_status=None)
    torch.cuda.synchronize()
    assert cache.n_tokens.cpu().tolist() == [T0 + total] * B
    j_lo, j_hi = T0 // ratio, (T0 + total) // ratio
    for b in range(B):
        kv_all = np.concatenate([k[b] for k in kvs])
        g_all = np.concatenate([g[b] for g in gs])
        got_f = cache.comp[b][j_lo:j_hi].cpu().numpy() if f32 else None
        gv = None if f32 else cache.comp[b][j_lo:j_hi].cpu().numpy()
        gsc = None if f32 else cache.comp_scales[b][j_lo:j_hi].cpu().numpy()
        flips = 0
        for j in range(j_lo, j_hi):
            t0 = ratio * j - T0
            kvp = kv_all[t0:t0 + ratio]
            gp = g_all[t0:t0 + 2] if ratio == 2 else None
            ref = orc.compress_row(j, kvp, gp, ratio=ratio, rope=rope, f32=True)
            if ratio == 2:
                bound = _pool_error_bound(kvp[0], kvp[1]).astype(np.float64)
            else:
                bound = np.zeros(512)
            tail = slice(512 - 64, 512)
            pair_b = bound[tail].reshape(-1, 2).sum(1).repeat(2)  # both members feed each output
            bound[tail] = pair_b + np.spacing(np.abs(ref[tail]).astype(np.float32) + np.float32(1e-30))
            if f32:
                err = np.abs(got_f[j - j_lo].astype(np.float64) - ref)
                assert np.all(err <= bound), (b, j, (err / np.maximum(bound, 1e-30)).max())
                continue
            rv, rs = orc.nvfp4_quantize(ref)
            for gi in range(32):
                if rs[gi] == gsc[j - j_lo, gi] and np.array_equal(rv[8 * gi:8 * gi + 8],
                                                                  gv[j - j_lo, 8 * gi:8 * gi + 8]):
                    continue
                flips += 1
                assert _near_boundary_flip_ok(ref[16 * gi:16 * gi + 16], bound[16 * gi:16 * gi + 16],
                                              gv[j - j_lo, 8 * gi:8 * gi + 8], gsc[j - j_lo, gi]), (b, j, gi)
        assert flips <= max(2, (j_hi - j_lo) * 32 // 1000)
    # the rotation is active: rows differ from the unrotated Compressor's
    p0 = api.default_params(**dict(over, rope_dim=0))
    flat = api.LayerCache(1, [cap], p0)
    flat.n_tokens.fill_(T0)
    for kv, g in zip(kvs, gs):
        flat.append(t(kv[:1]), t(g[:1]) if ratio == 2 else None)
    torch.cuda.synchronize()
    a, z = cache.comp[0][j_lo + 1:j_hi].cpu().numpy(), flat.comp[0][j_lo + 1:j_hi].cpu().numpy()
    head = slice(0, 448) if f32 else slice(0, 224)
    assert np.array_equal(a[:, head], z[:, head]) and not np.array_equal(a, z)


def test_compress_append_rope_rejects_bad_settings():
    cache = api.LayerCache(1, [4], api.default_params())
    kv = torch.zeros(1, 2, 512, device=DEV)
    for over in (dict(rope_dim=62), dict(rope_dim=516), dict(rope_dim=64, rope_beta_fast=1.0)):
        p = api.default_params(**over)
        with pytest.raises(api.Csa2Error):
            api.compress_append(p, kv, kv, cache.pend_kv, cache.pend_gate, cache.comp_ptrs,
                                cache.comp_scale_ptrs, cache.comp_cap, cache.win_ptrs,
                                cache.n_tokens)
    torch.cuda.synchronize()
    assert cache.n_tokens.item() == 0  # nothing was enqueued


def test_compress_capacity_overflow_sets_status_and_writes_nothing_past_cap():
    p = api.default_params()
    cache = api.LayerCache(1, [2], p)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv = torch.randn(1, 8, 512, device=DEV)
    cache.append(kv, kv, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 2
    assert cache.n_tokens.item() == 8


# --------------------------------------------------------------------------- indexer
def _index_case(seed, n_cs, pow2=True):
    rng = np.random.default_rng(seed)
    B = len(n_cs)
    key = synth.stream_key(seed, synth.IDX_K)
    qv = synth.e2m1_bytes(key, np.arange(B * 32 * 64, dtype=np.uint64)).reshape(B, 32, 64)
    qs = np.full((B, 32, 8), 0x38, np.uint8)
    w = synth.w_pow2(key ^ 7, np.arange(B * 32, dtype=np.uint64)).reshape(B, 32)
    kvs, kss = [], []
    for b, n in enumerate(n_cs):
        kv = synth.e2m1_bytes(key ^ (b + 11), np.arange(max(n, 1) * 64, dtype=np.uint64)).reshape(-1, 64)
        ks = (synth.scale_pow2_bytes(key ^ (b + 99), np.arange(max(n, 1) * 8, dtype=np.uint64))
              if pow2 else np.full(max(n, 1) * 8, 0x38, np.uint8)).reshape(-1, 8)
        if n > 10:  # a planted key: q head copy with scale 4
            kv[n // 3], ks[n // 3] = qv[b, int(np.argmax(w[b]))], 0x48
        kvs.append(kv)
        kss.append(ks)
    return qv, qs, w, kvs, kss, rng


def _tiled_caches(p, kvs, kss):
    """Index-key caches written through csa2_index_keys_write from plain rows."""
    cache = api.IndexKeyCache([max(len(k), 1) for k in kvs])
    for b, (kv, ks) in enumerate(zip(kvs, kss)):
        cache.write_seq(p, b, t(kv), t(ks))
    return cache


def test_index_keys_write_produces_the_documented_tile_image():
    rng = np.random.default_rng(12)
    n = 300  # 3 tiles, the last partial
    kv = rng.integers(0, 256, (n, 64), dtype=np.uint8)
    ks = rng.integers(0, 256, (n, 8), dtype=np.uint8)
    p = api.default_params()
    cache = _tiled_caches(p, [kv], [ks])
    torch.cuda.synchronize()
    img = cache.buf[0].cpu().numpy()
    assert img.size == 3 * 9216
    for t_ in range(n):  # formulas of include/csa2.h, written out independently here
        tile, m = divmod(t_, 128)
        base = tile * 9216
        for c in range(4):
            off = base + m * 64 + ((c ^ ((m >> 1) & 3)) << 4)
            assert np.array_equal(img[off:off + 16], kv[t_, 16 * c:16 * c + 16])
        for g in range(8):
            off = base + 8192 + (g >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (g & 3)
            assert img[off] == ks[t_, g]


# (cuda_cores, max_ctas). With the full grid this batch gives every CTA less than
# one chunk of super-tiles (the tensor-core build's contiguous tail ranges only);
# 3 CTAs take several round-robin chunks each, cross sequence boundaries inside a
# chunk and wrap the stage ring many times.
INDEX_MODES = {"tcgen05": (False, 0), "tcgen05_3ctas": (False, 3), "cuda_cores": (True, 0)}


@pytest.mark.parametrize("mode", list(INDEX_MODES))
def test_index_scores_bit_exact_ragged(mode):
    cuda_cores, max_ctas = INDEX_MODES[mode]
    n_cs = [1, 7, 8, 9, 127, 128, 129, 255, 256, 257, 1000, 5003, 0, 70000]
    qv, qs, w, kvs, kss, _ = _index_case(3, n_cs)
    B = len(n_cs)
    max_nc = max(n_cs)
    p = api.default_params()
    p.max_ctas = max_ctas
    cache = _tiled_caches(p, kvs, kss)
    n_tok = t(np.array([2 * n for n in n_cs], np.int32))
    scores = torch.full((B, max_nc), -7.0, device=DEV)
    bmax = torch.full((B, math.ceil(max_nc / 8)), -7.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.index_scores(p, max_nc, t(qv), t(qs), t(w), cache.ptrs, n_tok, scores, bmax, st,
                     cuda_cores=cuda_cores)
    torch.cuda.synchronize()
    assert st.item() == 0
    gs, gb = scores.cpu().numpy(), bmax.cpu().numpy()
    for b, n in enumerate(n_cs):
        ref, inexact = orc.index_scores(qv[b], qs[b], w[b], kvs[b][:n], kss[b][:n])
        assert inexact == 0
        bad = np.nonzero(gs[b, :n] != ref)[0]
        assert bad.size == 0, (b, n, bad[:5], gs[b, bad[:5]], ref[bad[:5]])
        assert np.all(gs[b, n:] == -7.0)  # untouched past n_c
        nb = math.ceil(n / 8)
        assert np.array_equal(gb[b, :nb], orc.block_max(ref, 8)), b


@pytest.mark.parametrize("pow2", [True, False])
def test_index_scores_shared_key_stream_bit_exact(pow2):
    """Many queries against one key stream (the prefill Indexer): ragged causal
    lengths (0, partial blocks and tiles, the full stream, past max_ncomp -> clipped
    and flagged), a query count that is not a multiple of 16."""
    n = 5003
    qv, qs, w, kvs, kss, rng = _index_case(8, [n], pow2=pow2)
    Q = 37
    key = synth.stream_key(17, synth.IDX_Q)
    qv = synth.e2m1_bytes(key, np.arange(Q * 32 * 64, dtype=np.uint64)).reshape(Q, 32, 64)
    qs = np.full((Q, 32, 8), 0x38, np.uint8)
    w = synth.w_pow2(key ^ 5, np.arange(Q * 32, dtype=np.uint64)).reshape(Q, 32)
    lens = np.array([0, 1, 7, 8, 9, 127, 128, 129, 511, 512, 513, 2048, 4999, n, n + 40] +
                    [int(x) for x in rng.integers(0, n + 1, Q - 15)], np.int64)
    p = api.default_params()
    cache = _tiled_caches(p, [kvs[0]], [kss[0]])
    n_tok = t((2 * lens).astype(np.int32))
    scores = torch.full((Q, n), -7.0, device=DEV)
    bmax = torch.full((Q, math.ceil(n / 8)), -7.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.index_scores_shared(p, n, t(qv), t(qs), t(w), cache.buf[0], n_tok, scores, bmax, st)
    torch.cuda.synchronize()
    assert st.item() == 2  # the query past max_ncomp is clipped and flagged
    gs, gb = scores.cpu().numpy(), bmax.cpu().numpy()
    for i in range(Q):
        m = int(min(lens[i], n))
        ref, inexact = orc.index_scores(qv[i], qs[i], w[i], kvs[0][:m], kss[0][:m])
        if pow2:
            assert inexact == 0
            bad = np.nonzero(gs[i, :m] != ref)[0]
            assert bad.size == 0, (i, m, bad[:5], gs[i, bad[:5]], ref[bad[:5]])
        else:
            assert np.all(gs[i, :m] == ref) or np.abs(gs[i, :m] - ref).max() <= 1e-5 * max(1, np.abs(ref).max())
        assert np.all(gs[i, m:] == -7.0)
        nb = math.ceil(m / 8)
        assert np.array_equal(gb[i, :nb], orc.block_max(gs[i, :m], 8)), i
        assert np.all(gb[i, nb:] == -7.0)


def test_index_scores_general_e4m3_scales_match_cuda_cores():
    """Non-power-of-two E4M3 scales (mantissa bits): the tensor-core and CUDA-core
    builds must agree with the oracle to fp32 rounding."""
    rng = np.random.default_rng(21)
    n_cs = [4000, 333]
    qv, qs, w, kvs, kss, _ = _index_case(5, n_cs)
    qs = rng.integers(0x28, 0x40, qs.shape, dtype=np.uint8)        # 0.125 .. 1.875
    kss = [rng.integers(0x28, 0x48, k.shape, dtype=np.uint8) for k in kss]
    p = api.default_params()
    cache = _tiled_caches(p, kvs, kss)
    n_tok = t(np.array([2 * n for n in n_cs], np.int32))
    outs = []
    for cc in (False, True):
        scores = torch.zeros(2, max(n_cs), device=DEV)
        bmax = torch.zeros(2, math.ceil(max(n_cs) / 8), device=DEV)
        api.index_scores(p, max(n_cs), t(qv), t(qs), t(w), cache.ptrs, n_tok, scores, bmax,
                         cuda_cores=cc)
        torch.cuda.synchronize()
        outs.append(scores.cpu().numpy())
    for b, n in enumerate(n_cs):
        ref, _ = orc.index_scores(qv[b], qs[b], w[b], kvs[b][:n], kss[b][:n])
        for o in outs:
            err = np.abs(o[b, :n].astype(np.float64) - ref) / np.maximum(np.abs(ref), 1.0)
            assert err.max() < 1e-5, err.max()


def test_index_scores_clip_and_status_when_length_exceeds_max():
    qv, qs, w, kvs, kss, _ = _index_case(4, [100])
    p = api.default_params()
    cache = _tiled_caches(p, kvs, kss)
    for cc in (False, True):
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        scores = torch.zeros(1, 50, device=DEV)
        bmax = torch.zeros(1, 7, device=DEV)
        api.index_scores(p, 50, t(qv), t(qs), t(w), cache.ptrs, t(np.array([200], np.int32)),
                         scores, bmax, st, cuda_cores=cc)
        torch.cuda.synchronize()
        assert st.item() & 2
        ref, _ = orc.index_scores(qv[0], qs[0], w[0], kvs[0][:50], kss[0][:50])
        assert np.array_equal(scores[0].cpu().numpy(), ref)


# --------------------------------------------------------------------------- selection
@pytest.mark.parametrize("cluster", [True, False], ids=["cluster4", "one_cta"])
@pytest.mark.parametrize("levels,pad", [(1, 0), (3, 0), (50, 0), (0, 0), (0, 4)])
def test_select_topk_exact_with_ties(levels, pad, cluster):
    """pad = 0: every row 16-byte aligned (vector loads where a sequence has at most
    65,536 blocks); pad = 4: odd rows misaligned (scalar loads). cluster: each
    sequence on a cluster of 4 CTAs (the small-batch launch), else on one CTA
    (max_ctas below 4 B forces it). Paths: up to 2,048 candidate blocks go flat
    (positions at or above the level-1 threshold, one exact select); with 1 level
    8,000 positions put all 1,000 blocks and 8,000 positions at the threshold, and
    with 3 levels 16,384 positions about 1,970 blocks and 5,500 positions: more than
    the flat pass's 4,096, so the 512 best blocks are selected first, as they are
    for 20,000..40,000 positions (2,400..4,800 candidate blocks). 70,001 and more
    with few levels put over 8,192 blocks there: the exact select over every block."""
    rng = np.random.default_rng(levels + 5)
    n_cs = [0, 1, 5, 511, 512, 513, 4095, 8000, 16384, 16385, 20000, 40000, 70001, 524288, 600000]
    B, max_nc = len(n_cs), max(n_cs) + pad
    scores = np.zeros((B, max_nc), np.float32)
    for b, n in enumerate(n_cs):
        if levels:
            scores[b, :n] = rng.integers(0, levels, n).astype(np.float32) * 0.25
        else:
            scores[b, :n] = rng.standard_normal(n).astype(np.float32)
        if n > 100:
            scores[b, rng.choice(n, 16, replace=False)] = 1e4
    nb = math.ceil(max_nc / 8)
    bm = np.full((B, nb), -np.inf, np.float32)
    for b, n in enumerate(n_cs):
        pad = np.full(math.ceil(n / 8) * 8, -np.inf, np.float32)
        pad[:n] = scores[b, :n]
        bm[b, :len(pad) // 8] = pad.reshape(-1, 8).max(1) if n else bm[b, :0]
    p = api.default_params(max_ctas=0 if cluster else B)
    idx = torch.full((B, 512), 123, dtype=torch.int32, device=DEV)
    n_sel = torch.zeros(B, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):  # twice: the launch leaves nothing behind that the next one reads
        api.select_topk(p, max_nc, t(scores), t(bm), t(np.array([2 * n for n in n_cs], np.int32)),
                        idx, n_sel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    gi, gn = idx.cpu().numpy(), n_sel.cpu().numpy()
    for b, n in enumerate(n_cs):
        ref, m = orc.select(scores[b, :n], 8, 2048, 512)
        assert gn[b] == m, (b, n)
        assert np.array_equal(gi[b], ref), (b, n, np.nonzero(gi[b] != ref)[0][:5])


@pytest.mark.parametrize("levels", [3, 0], ids=["ties", "continuous"])
def test_select_topk_many_sequences_half_build(levels):
    """More sequences than SMs (one CTA each, the 512-thread build with two CTAs per
    SM): every sequence exact, over ragged lengths from empty to 70,001 positions,
    with tied and continuous scores and planted maxima."""
    rng = np.random.default_rng(31 + levels)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    base = [0, 1, 5, 511, 512, 513, 4095, 8000, 16384, 16385, 20000, 40000, 70001]
    B = sms + 48
    n_cs = base + [int(x) for x in rng.integers(0, 30000, B - len(base))]
    max_nc = max(n_cs)
    scores = np.zeros((B, max_nc), np.float32)
    for b, n in enumerate(n_cs):
        if levels:
            scores[b, :n] = rng.integers(0, levels, n).astype(np.float32) * 0.25
        else:
            scores[b, :n] = rng.standard_normal(n).astype(np.float32)
        if n > 100:
            scores[b, rng.choice(n, 16, replace=False)] = 1e4
    nb = math.ceil(max_nc / 8)
    bm = np.full((B, nb), -np.inf, np.float32)
    for b, n in enumerate(n_cs):
        padded = np.full(math.ceil(n / 8) * 8, -np.inf, np.float32)
        padded[:n] = scores[b, :n]
        bm[b, :len(padded) // 8] = padded.reshape(-1, 8).max(1) if n else bm[b, :0]
    p = api.default_params()
    idx = torch.full((B, 512), 123, dtype=torch.int32, device=DEV)
    n_sel = torch.zeros(B, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.select_topk(p, max_nc, t(scores), t(bm), t(np.array([2 * n for n in n_cs], np.int32)),
                    idx, n_sel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    gi, gn = idx.cpu().numpy(), n_sel.cpu().numpy()
    for b, n in enumerate(n_cs):
        ref, m = orc.select(scores[b, :n], 8, 2048, 512)
        assert gn[b] == m, (b, n)
        assert np.array_equal(gi[b], ref), (b, n, np.nonzero(gi[b] != ref)[0][:5])


# --------------------------------------------------------------------------- attention
def _attn_case(rng, Ts, f32, n_idx_valid):
    B = len(Ts)
    p = api.default_params() if not f32 else api.default_params(
        kv_format=api.F32, win_format=api.F32, q_format=api.F32)
    caps = [max(1, T // 2) for T in Ts]
    cache = api.LayerCache(B, caps, p)
    st = []
    for b, T in enumerate(Ts):
        kv = rng.standard_normal((T, 512)).astype(np.float32)
        g = rng.standard_normal((T, 512)).astype(np.float32)
        s = orc.SeqState(cap_comp=caps[b], D=512, W=128, comp_f32=f32, win_f32=f32)
        s.append(kv, g)
        st.append(s)
        # the device cache gets the oracle's bytes (this test isolates attention)
        if f32:
            cache.comp[b].copy_(t(s.comp_f32))
            cache.win[b].copy_(t(s.win_f32))
        else:
            cache.comp[b].copy_(t(s.comp_vals))
            cache.comp_scales[b].copy_(t(s.comp_scales))
            cache.win[b].copy_(t(s.win_u8))
    cache.n_tokens.copy_(t(np.array(Ts, np.int32)))
    idx = np.full((B, 512), -1, np.int32)
    for b, T in enumerate(Ts):
        n_c = T // 2
        k = min(n_idx_valid, n_c)
        if k:
            sel = np.sort(rng.choice(n_c, k, replace=False))
            slots = rng.choice(512, k, replace=False)  # holes anywhere
            idx[b, slots] = sel
    q = rng.standard_normal((B, 64, 512)).astype(np.float32)
    if not f32:
        qb = synth.bf16_bits_rne(q)
        q_dev = torch.from_numpy(qb.view(np.int16)).to(DEV).view(torch.bfloat16)
        q64 = synth.bf16_to_f64(qb)
    else:
        q_dev, q64 = t(q), q.astype(np.float64)
    sink = rng.standard_normal(64).astype(np.float32)
    return p, cache, st, idx, q_dev, q64, sink


# csa2_sparse_attn's paths: (fp32 formats, mma_sync ablation entry, max_ctas). The
# quantised formats run on tcgen05; with 3 CTAs the even split cuts 2 of the 8
# units, whose pieces merge by log-sum-exp through the workspace.
SINGLE_MODES = {
    "tcgen05": (False, False, 0),
    "tcgen05_3ctas": (False, False, 3),
    "mma_sync": (False, True, 0),
    "f32": (True, False, 0),
}


@pytest.mark.parametrize("mode", list(SINGLE_MODES))
def test_sparse_attn_matches_oracle(mode):
    f32, mma_sync, max_ctas = SINGLE_MODES[mode]
    rng = np.random.default_rng(7 if f32 else 8)
    Ts = [1, 50, 127, 128, 129, 1000, 4096, 1025]
    valid = [512, 512, 512, 100, 512, 512, 512, 0]
    p, cache, st, idx, q_dev, q64, sink = _attn_case(rng, Ts, f32, 512)
    p.max_ctas = max_ctas
    for b, v in enumerate(valid):
        if v < 512:
            idx[b, rng.choice(512, 512 - v, replace=False)] = -1
    B = len(Ts)
    out = torch.empty(B, 64, 512, dtype=torch.float32 if f32 else torch.bfloat16, device=DEV)
    # garbage in the workspace: the call must not depend on its contents
    ws = torch.full((api.sparse_attn_workspace_size(p, B),), 0x5A, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):  # twice: the cut units' counts are left clean for the next call
        api.sparse_attn(p, q_dev, t(sink), cache.win_ptrs, cache.n_tokens, cache.comp_ptrs,
                        cache.comp_scale_ptrs, t(idx), out, ws, status, mma_sync=mma_sync)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    for b, T in enumerate(Ts):
        s = st[b]
        ref, n = orc.sparse_attn(q64[b], sink.astype(np.float64), 1 / math.sqrt(512), T, 128,
                                 win_u8=s.win_u8, win_f32=s.win_f32, comp_vals=s.comp_vals,
                                 comp_scales=s.comp_scales, comp_f32=s.comp_f32, idx=idx[b])
        if f32:
            err = np.abs(got[b] - ref).max()
            rel = np.linalg.norm(got[b] - ref) / np.linalg.norm(ref)
            assert err <= 1e-4 and rel <= 1e-5, (b, err, rel)
        else:
            ok, e = close_bf16(got[b], ref)
            assert ok, (b, T, e)


def test_sparse_attn_out_of_range_index_is_skipped_and_flagged():
    rng = np.random.default_rng(9)
    p, cache, st, idx, q_dev, q64, sink = _attn_case(rng, [600], False, 200)
    idx[0, 5] = 10_000  # beyond n_c = 300
    out = torch.empty(1, 64, 512, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(api.sparse_attn_workspace_size(p, 1), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.sparse_attn(p, q_dev, t(sink), cache.win_ptrs, cache.n_tokens, cache.comp_ptrs,
                    cache.comp_scale_ptrs, t(idx), out, ws, status)
    torch.cuda.synchronize()
    assert status.item() & 1
    keep = idx[0].copy()
    keep[5] = -1
    s = st[0]
    ref, _ = orc.sparse_attn(q64[0], sink.astype(np.float64), 1 / math.sqrt(512), 600, 128,
                             win_u8=s.win_u8, comp_vals=s.comp_vals, comp_scales=s.comp_scales,
                             idx=keep)
    ok, e = close_bf16(out[0].float().cpu().numpy().astype(np.float64), ref)
    assert ok, e


# How the fused reader attention is launched: (mma_sync, split, max_ctas). The
# split modes cut the (unit, tile) work into equal ranges per CTA; max_ctas caps
# the grid so that ranges cut units at many different tiles. With 13 CTAs both
# tests below have ranges that open on a one-tile piece (the window tile alone)
# followed by more pieces (boundaries at 24 and 64 of 105 items, 369 of 960).
LAYER_MODES = {
    "tcgen05": (False, False, 0),
    "tcgen05_split": (False, True, 0),
    "tcgen05_split_4ctas": (False, True, 4),
    "tcgen05_split_13ctas": (False, True, 13),
    "mma_sync": (True, False, 0),
}


def _run_layers(mode, p, L, B, *args, repeat=1):
    mma_sync, split, max_ctas = LAYER_MODES[mode]
    p.max_ctas = max_ctas
    ws = api.sparse_attn_layers_split_workspace(p, L, B) if split else None
    for _ in range(repeat):
        api.sparse_attn_layers(p, *args, mma_sync=mma_sync, workspace=ws)
    return ws


@pytest.mark.parametrize("sinks", ["normal", "extreme"])
@pytest.mark.parametrize("mode", list(LAYER_MODES))
def test_sparse_attn_layers_matches_oracle_per_layer(mode, sinks):
    """L layers share one compressed cache and one selection; each has its own
    window ring, query and sink (the KV-sharing readers of a source layer).
    sinks = "extreme": per head +30 (the sink outweighs every position, output near
    0), -30, -inf (a plain softmax), 0 and 5, across the running maximum, the sink
    term of the denominator and, in the split modes, the merge of cut units."""
    rng = np.random.default_rng(31)
    L = 3
    Ts = [1, 70, 128, 129, 900, 4096, 2001]
    B = len(Ts)
    p = api.default_params()
    src = api.LayerCache(B, [max(1, T // 2) for T in Ts], p)
    wins = [api.LayerCache(B, [1] * B, p, has_comp=False) for _ in range(L - 1)]
    st_src, st_win = [], [[] for _ in range(L - 1)]
    for b, T in enumerate(Ts):
        kv = rng.standard_normal((T, 512)).astype(np.float32)
        g = rng.standard_normal((T, 512)).astype(np.float32)
        s = orc.SeqState(cap_comp=max(1, T // 2), D=512, W=128)
        s.append(kv, g)
        st_src.append(s)
        src.comp[b].copy_(t(s.comp_vals))
        src.comp_scales[b].copy_(t(s.comp_scales))
        src.win[b].copy_(t(s.win_u8))
        for l in range(L - 1):
            w = orc.SeqState(cap_comp=1, D=512, W=128, has_comp=False)
            w.append(rng.standard_normal((T, 512)).astype(np.float32), None)
            st_win[l].append(w)
            wins[l].win[b].copy_(t(w.win_u8))
    src.n_tokens.copy_(t(np.array(Ts, np.int32)))
    idx = np.full((B, 512), -1, np.int32)
    for b, T in enumerate(Ts):
        n_c = T // 2
        k = min(int(rng.integers(0, 513)), n_c) if b % 2 else min(512, n_c)
        if k:
            idx[b, np.sort(rng.choice(512, k, replace=False))] = np.sort(rng.choice(n_c, k, replace=False))
    idx[5, 7] = 10 ** 6  # out of range: skipped, flagged
    q = rng.standard_normal((L, B, 64, 512)).astype(np.float32)
    qb = synth.bf16_bits_rne(q)
    q_dev = torch.from_numpy(qb.view(np.int16)).to(DEV).view(torch.bfloat16)
    sink = rng.standard_normal((L, 64)).astype(np.float32)
    if sinks == "extreme":
        prof = np.array([30.0, -30.0, -np.inf, 0.0, 5.0], np.float32)
        sink = prof[(np.arange(L)[:, None] + np.arange(64)[None, :]) % len(prof)]
    win_all = torch.cat([src.win_ptrs] + [w.win_ptrs for w in wins])
    out = torch.empty(L, B, 64, 512, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = _run_layers(mode, p, L, B, q_dev, t(sink), win_all, src.n_tokens, src.comp_ptrs,
                     src.comp_scale_ptrs, t(idx), out, status)
    torch.cuda.synchronize()
    assert status.item() == 1
    if ws is not None:  # every boundary count is back at zero for the next launch
        n_slots = max(0, min(L * B, p.max_ctas or 10 ** 9, torch.cuda.get_device_properties(0).multi_processor_count) - 1)
        assert int(ws[: 4 * n_slots].view(torch.int32).abs().sum().item()) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    q64 = synth.bf16_to_f64(qb)
    for l in range(L):
        for b, T in enumerate(Ts):
            keep = idx[b].copy()
            keep[keep >= T // 2] = -1
            win = st_src[b].win_u8 if l == 0 else st_win[l - 1][b].win_u8
            s = st_src[b]
            ref, _ = orc.sparse_attn(q64[l, b], sink[l].astype(np.float64), 1 / math.sqrt(512), T,
                                     128, win_u8=win, comp_vals=s.comp_vals,
                                     comp_scales=s.comp_scales, idx=keep)
            ok, e = close_bf16(got[l, b], ref)
            assert ok, (l, b, T, e)


def _e4m3_small_bytes(rng, shape):
    """E4M3 bytes of magnitude < 4 (exponent field <= 8), random sign."""
    e = rng.integers(0, 9, shape)
    m = rng.integers(0, 8, shape)
    sgn = rng.integers(0, 2, shape)
    return ((sgn << 7) | (e << 3) | m).astype(np.uint8)


@pytest.mark.parametrize("mode", list(LAYER_MODES))
def test_sparse_attn_layers_rescale_and_many_units(mode):
    """192 (layer, sequence) units (more than one per SM), partial windows, empty
    and out-of-range selections, NaN bytes in window slots that are not yet
    valid, and planted compressed rows aligned with a query head whose logits
    jump far above the window's in tiles 2 and 4, so the running maximum moves
    in the middle of the stream (the output must not depend on where)."""
    rng = np.random.default_rng(77)
    L, B = 4, 48
    Ts = [int(x) for x in rng.choice([40, 127, 128, 300, 1000, 2049, 5000], B)]
    p = api.default_params()
    n_cs = [T // 2 for T in Ts]
    src = api.LayerCache(B, [max(1, n) for n in n_cs], p)
    wins = [api.LayerCache(B, [1] * B, p, has_comp=False) for _ in range(L - 1)]
    q = rng.standard_normal((L, B, 64, 512)).astype(np.float32)
    qb = synth.bf16_bits_rne(q)
    q64 = synth.bf16_to_f64(qb)
    idx = np.full((B, 512), -1, np.int32)
    comp_v, comp_s, win_b = [], [], [[None] * B for _ in range(L)]
    for b, T in enumerate(Ts):
        n_c = n_cs[b]
        rows = rng.standard_normal((max(1, n_c), 512)).astype(np.float32)
        k = min(512, n_c)
        if k:
            idx[b, :k] = np.sort(rng.choice(n_c, k, replace=False))
        if n_c >= 512 and b % 3 != 2:  # plant: head h0 of layer 0 aligned with two selected rows
            h0 = b % 64
            sign = np.where(q64[0, b, h0] >= 0, 1.0, -1.0).astype(np.float32)
            rows[idx[b, 200]] = sign
            rows[idx[b, 450]] = 3 * sign
        if b % 5 == 4 and k:
            idx[b, k // 2:] = -1  # a short selection
        if b == 7 and k:
            idx[b, 3] = n_c + 5  # out of range: skipped, flagged
        v, sc = orc.nvfp4_quantize(rows)
        comp_v.append(v)
        comp_s.append(sc)
        src.comp[b][: v.shape[0]].copy_(t(v))
        src.comp_scales[b][: sc.shape[0]].copy_(t(sc))
        for l in range(L):
            w = _e4m3_small_bytes(rng, (128, 512))
            if T < 128:
                w[T:] = 0x7F  # E4M3 NaN in slots that hold no token yet
            win_b[l][b] = w
            (src.win[b] if l == 0 else wins[l - 1].win[b]).copy_(t(w))
    src.n_tokens.copy_(t(np.array(Ts, np.int32)))
    q_dev = torch.from_numpy(qb.view(np.int16)).to(DEV).view(torch.bfloat16)
    sink = rng.standard_normal((L, 64)).astype(np.float32)
    win_all = torch.cat([src.win_ptrs] + [w.win_ptrs for w in wins])
    out = torch.empty(L, B, 64, 512, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _run_layers(mode, p, L, B, q_dev, t(sink), win_all, src.n_tokens, src.comp_ptrs,
                src.comp_scale_ptrs, t(idx), out, status)
    torch.cuda.synchronize()
    assert status.item() == 1  # the planted out-of-range index only
    if LAYER_MODES[mode][1]:  # a second launch on the same workspace gives the same bytes
        out2 = torch.empty_like(out)
        _run_layers(mode, p, L, B, q_dev, t(sink), win_all, src.n_tokens, src.comp_ptrs,
                    src.comp_scale_ptrs, t(idx), out2, status, repeat=2)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    for l in range(L):
        for b, T in enumerate(Ts):
            keep = idx[b].copy()
            keep[keep >= n_cs[b]] = -1
            ref, _ = orc.sparse_attn(q64[l, b], sink[l].astype(np.float64), 1 / math.sqrt(512), T,
                                     128, win_u8=win_b[l][b], comp_vals=comp_v[b],
                                     comp_scales=comp_s[b], idx=keep)
            ok, e = close_bf16(got[l, b], ref)
            assert ok, (l, b, T, e)


def test_fp4_mma_peak_completes_with_a_clean_status():
    """The FP4 tensor-core rate measurement (the prefill Indexer's MMA issued back to
    back) completes, twice, more CTAs than SMs included."""
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    api.fp4_mma_peak(3, 50, st)
    api.fp4_mma_peak(2 * sms + 1, 200, st)
    torch.cuda.synchronize()
    assert st.item() == 0


def test_launch_trace_names_the_last_launch():
    """csa2_trace_attach: after a selection launch the host-mapped record names it
    (started and first-CTA-finished), without a synchronising read of device
    memory; detaching stops the stores."""
    p = api.default_params()
    B, n_c = 2, 300
    rng = np.random.default_rng(5)
    scores = t(rng.standard_normal((B, 320)).astype(np.float32))
    bmax = torch.full((B, 40), -1.0, device=DEV)
    bmax[:, :38] = t(rng.standard_normal((B, 38)).astype(np.float32))
    n_tok = t(np.full(B, 2 * n_c, np.int32))
    idx = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rec = api.trace_attach()
    try:
        api.select_topk(p, 320, scores, bmax, n_tok, idx)
        torch.cuda.synchronize()
        v = [int(x) for x in rec.tolist()]
        assert v[0] == 3 and v[2] == 3 and v[1] >= 1 and v[3] == v[1], v
        assert "select_topk" in api.trace_read(rec)
    finally:
        api.check(api.lib().csa2_trace_attach(None), "trace detach")
    before = [int(x) for x in rec.tolist()]
    api.select_topk(p, 320, scores, bmax, n_tok, idx)
    torch.cuda.synchronize()
    assert [int(x) for x in rec.tolist()] == before
