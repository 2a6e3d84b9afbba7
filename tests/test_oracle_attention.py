"""Pins of the oracle's sparse attention ("DeepSeek-V4.1-Flash-NVFP4" §3.4: gather
by index, softmax with a learnable attn_sink, no n x n matrix; §三: each query
attends to 128 window + 512 selected = 640 positions; §3.1 window; §一: one KV
head of dim 512 shared by the query heads, K = V = the latent).

Independent references: scipy's softmax over the concatenated logits, torch's
E4M3 decode, and the pages' own statement that the sparse path is dense
attention over the attended set."""
import numpy as np
import scipy.special
import torch

from oracle import oracle as orc

H, D, W = 8, 64, 16


def e4m3_np(u8):
    return torch.tensor(np.asarray(u8, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def dense_reference(q, keys, sink, scale):
    """softmax([sink, scale*q.k_j]) over every key, weights applied to the keys."""
    out = np.zeros((q.shape[0], keys.shape[1]))
    for h in range(q.shape[0]):
        z = np.concatenate([[sink[h]], scale * keys @ q[h]])
        p = scipy.special.softmax(z)
        out[h] = p[1:] @ keys
    return out


def make_state(T, seed):
    rng = np.random.default_rng(seed)
    s = orc.SeqState(cap_comp=T // 2 + 1, D=D, W=W)
    s.append(rng.standard_normal((T, D)).astype(np.float32),
             rng.standard_normal((T, D)).astype(np.float32))
    q = rng.standard_normal((H, D))
    sink = rng.standard_normal(H)
    return s, q, sink


def gathered_rows(s, idx):
    T = s.T
    win = [e4m3_np(s.win_u8[p % W]) for p in range(max(0, T - W), T)]
    comp = [orc.nvfp4_dequant(s.comp_vals[j], s.comp_scales[j]) for j in idx if j >= 0]
    return np.array(win + comp)


def test_sparse_equals_dense_when_everything_is_selected():
    # context small enough that window + all compressed positions are attended
    s, q, sink = make_state(T=40, seed=0)
    idx = np.arange(s.n_comp, dtype=np.int32)
    out, n = orc.sparse_attn(q, sink, 1 / np.sqrt(D), s.T, W, win_u8=s.win_u8,
                             comp_vals=s.comp_vals, comp_scales=s.comp_scales, idx=idx)
    assert n == W + s.n_comp
    ref = dense_reference(q, gathered_rows(s, idx), sink, 1 / np.sqrt(D))
    assert np.max(np.abs(out - ref)) < 1e-12


def test_sink_to_minus_infinity_is_plain_softmax_and_plus_infinity_is_zero():
    s, q, _ = make_state(T=30, seed=1)
    idx = np.array([3, -1, 7, 11], np.int32)
    rows = gathered_rows(s, idx)
    out, _ = orc.sparse_attn(q, np.full(H, -np.inf), 0.125, s.T, W, win_u8=s.win_u8,
                             comp_vals=s.comp_vals, comp_scales=s.comp_scales, idx=idx)
    for h in range(H):
        p = scipy.special.softmax(0.125 * rows @ q[h])
        assert np.max(np.abs(out[h] - p @ rows)) < 1e-12
    out, _ = orc.sparse_attn(q, np.full(H, 1e4), 0.125, s.T, W, win_u8=s.win_u8,
                             comp_vals=s.comp_vals, comp_scales=s.comp_scales, idx=idx)
    assert np.max(np.abs(out)) == 0.0


def test_order_of_selected_indices_does_not_matter():
    s, q, sink = make_state(T=60, seed=2)
    idx = np.array([1, 5, 9, 13, 17, 21, 25, -1], np.int32)
    a, _ = orc.sparse_attn(q, sink, 0.1, s.T, W, win_u8=s.win_u8, comp_vals=s.comp_vals,
                           comp_scales=s.comp_scales, idx=idx)
    b, _ = orc.sparse_attn(q, sink, 0.1, s.T, W, win_u8=s.win_u8, comp_vals=s.comp_vals,
                           comp_scales=s.comp_scales, idx=idx[::-1].copy())
    assert np.max(np.abs(a - b)) < 1e-12


def test_one_hot_logits_reproduce_the_value_row():
    s, _, _ = make_state(T=50, seed=3)
    idx = np.array([4, 9], np.int32)
    rows = gathered_rows(s, idx)
    target = rows[-1]
    q = np.tile(target * 1e3, (H, 1))  # this key's logit dominates every other by far
    out, _ = orc.sparse_attn(q, np.full(H, -np.inf), 1.0, s.T, W, win_u8=s.win_u8,
                             comp_vals=s.comp_vals, comp_scales=s.comp_scales, idx=idx)
    assert np.max(np.abs(out - target)) < 1e-9


def test_window_covers_min_T_W_newest_tokens_and_fp32_path():
    rng = np.random.default_rng(4)
    for T in (0, 1, 5, W, W + 3, 3 * W):
        s = orc.SeqState(cap_comp=T // 2 + 1, D=D, W=W, comp_f32=True, win_f32=True)
        kv = rng.standard_normal((T, D)).astype(np.float32)
        if T:
            s.append(kv, kv)
        q = rng.standard_normal((H, D))
        sink = rng.standard_normal(H)
        out, n = orc.sparse_attn(q, sink, 0.2, s.T, W, win_f32=s.win_f32, comp_f32=s.comp_f32,
                                 idx=np.zeros(0, np.int32))
        assert n == min(T, W)
        if T:
            ref = dense_reference(q, kv[max(0, T - W):].astype(np.float64), sink, 0.2)
            assert np.max(np.abs(out - ref)) < 1e-12
        else:
            assert not out.any()
