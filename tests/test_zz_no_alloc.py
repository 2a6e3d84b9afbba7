"""csa2_sparse_attn_noalloc — the variant for callers that cannot allocate device
memory (an engine whose pool already owns the free HBM, or a latency-critical
path where an allocation would synchronise the device). It keeps its scratch (the
partial results of the attention's schedules: the tcgen05 kernel's cut units for
the quantised formats, the split-KV passes for fp32) in a fixed array inside the
library instead of a caller workspace.

Checked through the C ABI against csa2_sparse_attn with a workspace, on two
calls in a row with different inputs (the shared array keeps the previous
call's contents, which must not leak into the next result), plus the batch
limit. Self-contained, so it passes alone in a fresh process or after the rest.
"""
import numpy as np
import pytest
import torch

from csa2_compressed_sparse_02_gb300 import api, synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, B, T, f32=False):
    rng = np.random.default_rng(seed)
    p = api.default_params(**(dict(kv_format=api.F32, win_format=api.F32, q_format=api.F32)
                              if f32 else {}))
    cache = api.LayerCache(B, [T // 2] * B, p)
    for b in range(B):
        s = orc.SeqState(cap_comp=T // 2, D=512, W=128, comp_f32=f32, win_f32=f32)
        s.append(rng.standard_normal((T, 512)).astype(np.float32),
                 rng.standard_normal((T, 512)).astype(np.float32))
        if f32:
            cache.comp[b].copy_(torch.from_numpy(s.comp_f32))
            cache.win[b].copy_(torch.from_numpy(s.win_f32))
        else:
            cache.comp[b].copy_(torch.from_numpy(s.comp_vals))
            cache.comp_scales[b].copy_(torch.from_numpy(s.comp_scales))
            cache.win[b].copy_(torch.from_numpy(s.win_u8))
    cache.n_tokens.fill_(T)
    idx = np.full((B, 512), -1, np.int32)
    for b in range(B):
        k = int(rng.integers(1, 513))
        idx[b, :k] = np.sort(rng.choice(T // 2, k, replace=False))
    qf = rng.standard_normal((B, 64, 512)).astype(np.float32)
    if f32:
        q_dev = torch.from_numpy(qf).to(DEV)
    else:
        q = synth.bf16_bits_rne(qf)
        q_dev = torch.from_numpy(q.view(np.int16)).to(DEV).view(torch.bfloat16)
    sink = torch.from_numpy(rng.standard_normal(64).astype(np.float32)).to(DEV)
    return p, cache, torch.from_numpy(idx).to(DEV), q_dev, sink


@pytest.mark.parametrize("f32", [False, True], ids=["nvfp4", "fp32"])
def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(f32):
    odt = torch.float32 if f32 else torch.bfloat16
    for call, (seed, B, T) in enumerate(((1, 32, 3000), (2, 5, 1400))):
        p, cache, idx, q, sink = _case(seed + 10 * f32, B, T, f32)
        ref = torch.empty(B, 64, 512, dtype=odt, device=DEV)
        ws = torch.empty(api.sparse_attn_workspace_size(p, B), dtype=torch.uint8, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        api.sparse_attn(p, q, sink, cache.win_ptrs, cache.n_tokens, cache.comp_ptrs,
                        cache.comp_scale_ptrs, idx, ref, ws, st)
        got = torch.full((B, 64, 512), float("nan"), dtype=odt, device=DEV)
        api.sparse_attn_noalloc(p, q, sink, cache.win_ptrs, cache.n_tokens, cache.comp_ptrs,
                                cache.comp_scale_ptrs, idx, got, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        o = got.float().cpu().numpy().astype(np.float64)
        e = ref.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(o).all(), call
        err = np.abs(o - e).max()
        rel = np.linalg.norm(o - e) / np.linalg.norm(e)
        if f32:
            assert err <= 1e-4 and rel <= 1e-5, (call, err, rel)
        else:
            assert err <= 1.5e-2 and rel <= 4e-3, (call, err, rel)


def test_noalloc_rejects_batches_beyond_its_scratch():
    p, cache, idx, q, sink = _case(3, 1, 600)
    big = 33
    n_tok = torch.full((big,), 600, dtype=torch.int32, device=DEV)
    out = torch.empty(big, 64, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(api.Csa2Error, match="at most 32"):
        api.sparse_attn_noalloc(p, q, sink, cache.win_ptrs, n_tok, cache.comp_ptrs,
                                cache.comp_scale_ptrs, idx, out)
