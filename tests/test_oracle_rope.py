"""Pins of the oracle's rotary embedding of the compressed KV (config walkthrough
"CSA2稀疏注意力、384专家MoE与1M上下文" §2.2 compress_rope_theta 160000, §四 rope_scaling
yarn / factor 16 / original 65536 / beta_fast 32 / beta_slow 1;
"DeepSeek-V4.1-Flash-NVFP4" §3.2), checked against things other than the oracle's
own formula:
  * with factor 1 YaRN is plain RoPE, which rotates each pair like the complex
    number a + ib multiplied by exp(i pos theta_i) (RoFormer's complex form,
    evaluated with Python's cmath);
  * a rotation keeps each pair's length and leaves the unrotated dims alone;
  * the dot product of a rotated query and a rotated key depends only on the
    distance of their positions (the property RoPE exists for);
  * YaRN keeps the fast pairs, interpolates the slow ones by exactly 1/factor
    (rotating at 16 m equals plain RoPE at m), and blends monotonically in
    between, with the boundaries derived by hand in tests/golden/rope_yarn_ramp.txt;
  * the Compressor rotates a row at the raw position of its pair's first token,
    after pooling and before quantising."""
import cmath

import numpy as np
import pytest

from conftest import read_golden
from oracle import oracle as orc

FIG = {k: float(v) for k, v in read_golden("pages_figures.txt")}
RAMP = {r[0]: (int(r[1]), int(r[2])) for r in read_golden("rope_yarn_ramp.txt")}
D = 512


def pages_rope(**over):
    kw = dict(dim=64, base=FIG["compress_rope_theta"], factor=FIG["yarn_factor"],
              orig_len=FIG["yarn_original_length"], beta_fast=FIG["yarn_beta_fast"],
              beta_slow=FIG["yarn_beta_slow"])
    kw.update(over)
    return orc.rope_config(**kw)


def effective_angles(rope, pos):
    """Angle each pair of the oracle's rotation turns (1, 0) by at position pos."""
    x = np.zeros(D, np.float32)
    x[D - rope.dim::2] = 1.0
    y = orc.rope_rotate(x, pos, rope).astype(np.float64)
    tail = y[D - rope.dim:]
    return np.arctan2(tail[1::2], tail[0::2])


@pytest.mark.parametrize("pos", [0, 1, 7, 1000, 65535, 1048575])
def test_factor_one_is_roformer_complex_rotation(pos):
    rope = pages_rope(factor=1.0)
    rng = np.random.default_rng(pos)
    x = rng.standard_normal(D).astype(np.float32) * 3
    y = orc.rope_rotate(x, pos, rope)
    base, dim = FIG["compress_rope_theta"], 64
    for i in range(dim // 2):
        a, b = float(x[D - dim + 2 * i]), float(x[D - dim + 2 * i + 1])
        z = complex(a, b) * cmath.exp(1j * pos * base ** (-2.0 * i / dim))
        ya, yb = y[D - dim + 2 * i], y[D - dim + 2 * i + 1]
        # both are fp64 results rounded once to fp32: equal up to that rounding
        assert abs(ya - z.real) <= np.spacing(np.float32(abs(z.real)) + np.float32(1e-30)) + 1e-9
        assert abs(yb - z.imag) <= np.spacing(np.float32(abs(z.imag)) + np.float32(1e-30)) + 1e-9
    if pos == 0:
        assert np.array_equal(y, x)


def test_rotation_keeps_pair_lengths_and_the_unrotated_dims():
    rope = pages_rope()
    rng = np.random.default_rng(1)
    for pos in (3, 4097, 524288, 1048574):
        x = rng.standard_normal(D).astype(np.float32)
        y = orc.rope_rotate(x, pos, rope)
        assert np.array_equal(y[:D - 64], x[:D - 64])
        n0 = np.hypot(x[D - 64::2].astype(np.float64), x[D - 63::2].astype(np.float64))
        n1 = np.hypot(y[D - 64::2].astype(np.float64), y[D - 63::2].astype(np.float64))
        assert np.allclose(n0, n1, rtol=3e-7, atol=0)


def test_rotated_dot_depends_only_on_the_position_distance():
    rope = pages_rope()
    rng = np.random.default_rng(2)
    q = rng.standard_normal(D).astype(np.float32)
    k = rng.standard_normal(D).astype(np.float32)
    for m, n, c in ((10, 4, 1000), (65536, 2, 262144), (1048000, 0, 500), (7, 7, 999999)):
        d0 = np.dot(orc.rope_rotate(q, m, rope)[D - 64:].astype(np.float64),
                    orc.rope_rotate(k, n, rope)[D - 64:].astype(np.float64))
        d1 = np.dot(orc.rope_rotate(q, m + c, rope)[D - 64:].astype(np.float64),
                    orc.rope_rotate(k, n + c, rope)[D - 64:].astype(np.float64))
        scale = np.abs(q[D - 64:]).sum() * np.abs(k[D - 64:]).max()
        assert abs(d0 - d1) <= 1e-6 * scale, (m, n, c, d0, d1)
    # and it does change with the distance
    d_near = np.dot(orc.rope_rotate(q, 5, rope)[D - 64:], orc.rope_rotate(k, 5, rope)[D - 64:])
    d_far = np.dot(orc.rope_rotate(q, 5, rope)[D - 64:], orc.rope_rotate(k, 6, rope)[D - 64:])
    assert d_near != d_far


def test_yarn_keeps_fast_pairs_and_interpolates_slow_pairs_by_the_factor():
    yarn, plain = pages_rope(), pages_rope(factor=1.0)
    keep0, keep1 = RAMP["keep"]
    blend0, blend1 = RAMP["blend"]
    int0, int1 = RAMP["interpolate"]
    # fast pairs: the same rotation as plain RoPE at every position
    for pos in (1, 3, 100, 123457):
        a = orc.rope_rotate(np.ones(D, np.float32), pos, yarn)
        b = orc.rope_rotate(np.ones(D, np.float32), pos, plain)
        sl = slice(D - 64 + 2 * keep0, D - 64 + 2 * keep1 + 2)
        assert np.array_equal(a[sl], b[sl]), pos
    # slow pairs: YaRN at 16 m turns exactly as far as plain RoPE at m (position
    # interpolation); compared on the measured angles (small, no wrap)
    s = int(FIG["yarn_factor"])
    for m in (1, 2, 5):
        ay = effective_angles(yarn, s * m)[int0:int1 + 1]
        ap = effective_angles(plain, m)[int0:int1 + 1]
        assert np.allclose(ay, ap, rtol=1e-6, atol=1e-12), m
    # the blend: the frequency ratio YaRN/plain at position 1 lies strictly between
    # 1/16 and 1 inside the ramp, is 1 before it and 1/16 after it, and falls with i
    ratio = effective_angles(yarn, 1) / effective_angles(plain, 1)
    assert np.allclose(ratio[keep0:keep1 + 1], 1.0, rtol=1e-6)
    assert np.allclose(ratio[int0:int1 + 1], 1.0 / s, rtol=1e-5)
    mid = ratio[blend0:blend1 + 1]
    assert np.all(mid < 1.0 - 1e-4) and np.all(mid > 1.0 / s + 1e-4)
    assert np.all(np.diff(ratio) <= 1e-7)
    assert np.all(np.diff(mid) < 0)


def test_freqs_table_agrees_with_the_measured_rotation():
    yarn = pages_rope()
    th = orc.rope_freqs(yarn)
    assert th.shape == (32,)
    assert np.allclose(effective_angles(yarn, 1), th, rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("ratio", [1, 2])
def test_compressor_rotates_each_row_at_its_first_raw_position(ratio):
    rope = pages_rope()
    rng = np.random.default_rng(10 + ratio)
    T = 41 * ratio + 1  # ratio 2: ends on a pending half pair
    kv = rng.standard_normal((T, D)).astype(np.float32)
    g = rng.standard_normal((T, D)).astype(np.float32)
    gg = g if ratio == 2 else None
    for f32 in (True, False):
        rot = orc.SeqState(cap_comp=T, D=D, W=16, comp_f32=f32, win_f32=f32, ratio=ratio, rope=rope)
        flat = orc.SeqState(cap_comp=T, D=D, W=16, comp_f32=f32, win_f32=f32, ratio=ratio)
        # token by token through the decode path, and in one chunk
        chunk = orc.SeqState(cap_comp=T, D=D, W=16, comp_f32=f32, win_f32=f32, ratio=ratio,
                             rope=rope)
        for t in range(T):
            rot.append(kv[t:t + 1], None if gg is None else gg[t:t + 1])
        flat.append(kv, gg)
        chunk.append(kv, gg)
        n = T // ratio
        for j in range(n):
            if f32:
                # rotation of the unrotated (pooled) fp32 row at raw position ratio * j
                want = orc.rope_rotate(flat.comp_f32[j], ratio * j, rope)
                assert np.array_equal(rot.comp_f32[j], want), j
            else:
                fr = orc.compress_row(j, kv[ratio * j:ratio * j + ratio],
                                      None if gg is None else gg[ratio * j:ratio * j + 2],
                                      ratio=ratio, rope=None, f32=True)
                v, sc = orc.nvfp4_quantize(orc.rope_rotate(fr, ratio * j, rope))
                assert np.array_equal(rot.comp_vals[j], v) and np.array_equal(rot.comp_scales[j], sc)
        for a, b in ((rot.comp_f32, chunk.comp_f32), (rot.comp_vals, chunk.comp_vals),
                     (rot.comp_scales, chunk.comp_scales), (rot.win_u8, flat.win_u8),
                     (rot.win_f32, flat.win_f32)):
            if a is not None:
                assert np.array_equal(a, b)  # the window is not rotated
        # the leading 448 dims are untouched by the rotation
        if f32:
            assert np.array_equal(rot.comp_f32[:n, :D - 64], flat.comp_f32[:n, :D - 64])
        assert not np.array_equal((rot.comp_f32 if f32 else rot.comp_vals)[1:n],
                                  (flat.comp_f32 if f32 else flat.comp_vals)[1:n])


def test_zero_width_rotation_is_the_unrotated_compressor():
    rng = np.random.default_rng(5)
    kv = rng.standard_normal((20, D)).astype(np.float32)
    g = rng.standard_normal((20, D)).astype(np.float32)
    a = orc.SeqState(cap_comp=10, D=D, W=8, rope=pages_rope(dim=0))
    b = orc.SeqState(cap_comp=10, D=D, W=8)
    a.append(kv, g)
    b.append(kv, g)
    assert np.array_equal(a.comp_vals, b.comp_vals) and np.array_equal(a.comp_scales, b.comp_scales)
    # row 0 sits at position 0: the rotation is the identity there
    c = orc.SeqState(cap_comp=10, D=D, W=8, rope=pages_rope())
    c.append(kv, g)
    assert np.array_equal(c.comp_vals[0], b.comp_vals[0])
