"""Pins of the oracle's Compressor ("DeepSeek-V4.1-Flash-NVFP4" §3.2: per-channel
softmax-gated pooling of 2 consecutive tokens, a pending half-pair kept in
state during decode, NVFP4 output) and ring window (§3.1: 128 slots, one write
per token, FP8)."""
import numpy as np
import scipy.special
import torch

from oracle import oracle as orc


def test_pool_equal_gates_is_the_mean():
    rng = np.random.default_rng(0)
    for _ in range(500):
        a, b, g = rng.standard_normal(3).astype(np.float32)
        assert orc.pool(a, b, g, g) == np.float32((np.float64(a) + np.float64(b)) / 2)


def test_pool_saturated_gate_selects_one_token():
    assert orc.pool(1.25, -7.0, 200.0, 0.0) == np.float32(1.25)
    assert orc.pool(1.25, -7.0, 0.0, 200.0) == np.float32(-7.0)


def test_pool_matches_logistic_closed_form():
    # softmax over a pair: alpha_0 = sigmoid(g0 - g1) (scipy's expit is the library routine)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2000, 4)).astype(np.float32) * np.float32(3)
    for kv0, kv1, g0, g1 in x:
        a0 = scipy.special.expit(np.float64(g0) - np.float64(g1))
        ref = a0 * np.float64(kv0) + (1 - a0) * np.float64(kv1)
        got = orc.pool(kv0, kv1, g0, g1)
        assert abs(got - ref) <= 2 * np.spacing(np.float32(abs(ref)) + np.float32(1e-30))


def _state(comp_f32=False):
    return orc.SeqState(cap_comp=64, D=32, W=8, comp_f32=comp_f32, win_f32=comp_f32)


def test_append_token_by_token_equals_one_chunk():
    rng = np.random.default_rng(2)
    kv = rng.standard_normal((37, 32)).astype(np.float32)
    g = rng.standard_normal((37, 32)).astype(np.float32)
    for f32 in (False, True):
        a, b = _state(f32), _state(f32)
        a.append(kv, g)
        for i in range(37):
            b.append(kv[i:i + 1], g[i:i + 1])
        assert a.T == b.T == 37 and a.n_comp == 18
        for x, y in ((a.comp_vals, b.comp_vals), (a.comp_scales, b.comp_scales),
                     (a.comp_f32, b.comp_f32), (a.win_u8, b.win_u8), (a.win_f32, b.win_f32)):
            if x is not None:
                assert np.array_equal(x, y)
        assert np.array_equal(a.pend_kv, kv[36]) and np.array_equal(b.pend_kv, kv[36])


def test_compressed_rows_are_pooled_pairs():
    rng = np.random.default_rng(3)
    kv = rng.standard_normal((20, 32)).astype(np.float32)
    g = rng.standard_normal((20, 32)).astype(np.float32)
    s = _state(True)
    s.append(kv, g)
    for j in range(10):
        for d in range(32):
            assert s.comp_f32[j, d] == orc.pool(kv[2 * j, d], kv[2 * j + 1, d], g[2 * j, d],
                                                g[2 * j + 1, d])
    q = _state(False)
    q.append(kv, g)
    v, sc = orc.nvfp4_quantize(s.comp_f32[:10])
    assert np.array_equal(q.comp_vals[:10], v) and np.array_equal(q.comp_scales[:10], sc)
    assert not q.comp_vals[10:].any()


def test_window_ring_holds_the_newest_tokens_as_e4m3():
    rng = np.random.default_rng(4)
    kv = rng.standard_normal((21, 32)).astype(np.float32)
    s = _state(False)
    s.append(kv, kv)
    ref = torch.tensor(kv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for p in range(21 - 8, 21):
        assert np.array_equal(s.win_u8[p % 8], ref[p])


def test_window_only_layer_keeps_no_compressed_state():
    s = orc.SeqState(cap_comp=4, D=32, W=8, has_comp=False)
    kv = np.ones((5, 32), np.float32)
    s.append(kv, None)
    assert s.T == 5 and s.comp_vals is None and s.win_u8.any()
