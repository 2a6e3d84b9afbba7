"""Pins of the oracle's Indexer ("DeepSeek-V4.1-Flash-NVFP4" §3.3: 32 FP4 index
query heads score the shared index key, ReLU, per-head weights; config
walkthrough §2.1: index_n_heads 32, index_head_dim 128) against a numpy matmul
of independently decoded values, and of its exactness check."""
import numpy as np
import torch

from csa2_compressed_sparse_02_gb300 import synth
from oracle import oracle as orc

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                 -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def decode_nvfp4_np(vals, scales):
    v = np.asarray(vals, np.uint8)
    codes = np.empty(v.shape[:-1] + (v.shape[-1] * 2,), np.int64)
    codes[..., 0::2] = v & 15
    codes[..., 1::2] = v >> 4
    s = torch.tensor(np.asarray(scales, np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    return E2M1[codes] * np.repeat(s, 16, axis=-1)


def make_case(seed, n_c, Hi=32, Di=128, kscale="pow2"):
    kq = synth.stream_key(seed, synth.IDX_Q)
    kk = synth.stream_key(seed, synth.IDX_K)
    kw = synth.stream_key(seed, synth.IDX_W)
    q_vals = synth.e2m1_bytes(kq, np.arange(Hi * Di // 2, dtype=np.uint64)).reshape(Hi, Di // 2)
    q_scales = np.full((Hi, Di // 16), synth.E4M3_ONE, np.uint8)
    w = synth.w_pow2(kw, np.arange(Hi, dtype=np.uint64))
    k_vals = synth.e2m1_bytes(kk, np.arange(n_c * Di // 2, dtype=np.uint64)).reshape(n_c, Di // 2)
    if kscale == "pow2":
        k_scales = synth.scale_pow2_bytes(kk ^ 1, np.arange(n_c * Di // 16, dtype=np.uint64)
                                          ).reshape(n_c, Di // 16)
    else:
        k_scales = np.full((n_c, Di // 16), synth.E4M3_ONE, np.uint8)
    return q_vals, q_scales, w, k_vals, k_scales


def numpy_scores(q_vals, q_scales, w, k_vals, k_scales):
    Q = decode_nvfp4_np(q_vals, q_scales)  # [Hi, Di]
    K = decode_nvfp4_np(k_vals, k_scales)  # [n_c, Di]
    dots = K @ Q.T                          # [n_c, Hi]
    return (np.maximum(dots, 0.0) * w[None, :].astype(np.float64)).sum(axis=1)


def test_scores_match_numpy_matmul_bitwise():
    for seed, kscale in ((1, "one"), (2, "pow2"), (3, "pow2")):
        case = make_case(seed, 300, kscale=kscale)
        got, inexact = orc.index_scores(*case)
        ref = numpy_scores(*case)
        assert inexact == 0
        assert np.array_equal(got, ref.astype(np.float32))
        assert np.all(ref == ref.astype(np.float32))  # exact by construction


def test_relu_and_weights_matter():
    q_vals, q_scales, w, k_vals, k_scales = make_case(4, 64)
    got, _ = orc.index_scores(q_vals, q_scales, w, k_vals, k_scales)
    # flipping the sign of every key turns ReLU'd positive dots into zeros and vice versa
    neg_vals = k_vals ^ np.uint8(0x88)
    got_neg, _ = orc.index_scores(q_vals, q_scales, w, neg_vals, k_scales)
    Q = decode_nvfp4_np(q_vals, q_scales)
    K = decode_nvfp4_np(k_vals, k_scales)
    ref_neg = (np.maximum(-(K @ Q.T), 0) * w).sum(1)
    assert np.array_equal(got_neg, ref_neg.astype(np.float32))
    assert not np.array_equal(got, got_neg)
    w2 = w.copy()
    w2[0] *= 2
    got_w2, _ = orc.index_scores(q_vals, q_scales, w2, k_vals, k_scales)
    ref_w2 = numpy_scores(q_vals, q_scales, w2, k_vals, k_scales)
    assert np.array_equal(got_w2, ref_w2.astype(np.float32))


def test_exactness_flag_catches_non_power_of_two_weights():
    q_vals, q_scales, w, k_vals, k_scales = make_case(5, 200)
    w = np.full(32, np.float32(1.0 / 3.0))
    k_scales = np.full_like(k_scales, 0x3F)  # 1.875: adds mantissa bits
    _, inexact = orc.index_scores(q_vals, q_scales, w, k_vals, k_scales)
    assert inexact > 0


def test_block_max_matches_numpy():
    rng = np.random.default_rng(6)
    for n in (1, 7, 8, 9, 64, 1001):
        s = rng.standard_normal(n).astype(np.float32)
        pad = np.full(-(-n // 8) * 8, -np.inf, np.float32)
        pad[:n] = s
        assert np.array_equal(orc.block_max(s, 8), pad.reshape(-1, 8).max(1))
