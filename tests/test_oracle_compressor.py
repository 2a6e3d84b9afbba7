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


# --------------------------------------------------------------------------- 1:1 layers
def test_ratio_one_rows_are_the_quantised_raw_tokens():
    """1:1 layers ("CSA2稀疏注意力、384专家MoE与1M上下文" §2.2, "DeepSeek-V4.1-Flash-NVFP4"
    §3.2): no pooling, so compressed row p is the NVFP4 encoding of raw token p, and
    there are T compressed positions (not T/2). Checked against the quantiser, which
    is pinned on its own (test_oracle_codecs)."""
    rng = np.random.default_rng(11)
    kv = (rng.standard_normal((37, 32)) * rng.choice([1e-3, 1, 50], (37, 1))).astype(np.float32)
    st = orc.SeqState(cap_comp=64, D=32, W=8, ratio=1)
    for a, b in [(0, 1), (1, 6), (6, 7), (7, 37)]:  # odd and even chunk boundaries
        st.append(kv[a:b], None)
    assert st.T == 37 and st.n_comp == 37
    v, s = orc.nvfp4_quantize(kv)
    assert np.array_equal(st.comp_vals[:37], v) and np.array_equal(st.comp_scales[:37], s)
    assert not st.comp_vals[37:].any()


def test_ratio_one_fp32_rows_and_window_match_the_raw_tokens():
    rng = np.random.default_rng(12)
    kv = rng.standard_normal((21, 32)).astype(np.float32)
    st = orc.SeqState(cap_comp=32, D=32, W=8, ratio=1, comp_f32=True, win_f32=True)
    st.append(kv, None)
    assert np.array_equal(st.comp_f32[:21], kv)
    for p in range(21 - 8, 21):  # ring slot p mod W holds the newest token with that slot
        assert np.array_equal(st.win_f32[p % 8], kv[p])


def test_ratio_two_is_unchanged_by_the_ratio_argument():
    rng = np.random.default_rng(13)
    kv = rng.standard_normal((19, 32)).astype(np.float32)
    g = rng.standard_normal((19, 32)).astype(np.float32)
    a = orc.SeqState(cap_comp=16, D=32, W=8)
    b = orc.SeqState(cap_comp=16, D=32, W=8, ratio=2)
    a.append(kv, g)
    b.append(kv[:4], g[:4])
    b.append(kv[4:], g[4:])
    assert a.n_comp == 9 == b.n_comp
    assert np.array_equal(a.comp_vals, b.comp_vals) and np.array_equal(a.comp_scales, b.comp_scales)
    # row j is the pooled pair (2j, 2j+1): pin one against the pooling definition
    row = np.array([orc.pool(kv[6, d], kv[7, d], g[6, d], g[7, d]) for d in range(32)], np.float32)
    v, s = orc.nvfp4_quantize(row[None])
    assert np.array_equal(a.comp_vals[3], v[0]) and np.array_equal(a.comp_scales[3], s[0])
