"""The oracle's sizes against the figures the pages print (tests/golden/
pages_figures.txt, each line cited): 128 + 512 = 640 attended positions, the
memory ledger of "DeepSeek-V4.1-Flash-NVFP4" §四, the FP8 window of §3.1 and the
≈1/1560 work ratio of §三."""
import numpy as np

from conftest import read_golden
from oracle import oracle as orc

FIG = {k: float(v) for k, v in read_golden("pages_figures.txt")}


def test_attended_set_is_640_at_full_context():
    W, D, H = int(FIG["window_tokens"]), 32, 2
    T = 3000
    s = orc.SeqState(cap_comp=T // 2, D=D, W=W)
    rng = np.random.default_rng(0)
    s.append(rng.standard_normal((T, D)).astype(np.float32),
             rng.standard_normal((T, D)).astype(np.float32))
    scores = rng.standard_normal(s.n_comp).astype(np.float32)
    idx, m = orc.select(scores, int(FIG["candidate_block_size"]), int(FIG["candidate_topk_blocks"]),
                        int(FIG["selected_positions"]))
    _, n = orc.sparse_attn(rng.standard_normal((H, D)), np.zeros(H), 0.1, s.T, W,
                           win_u8=s.win_u8, comp_vals=s.comp_vals, comp_scales=s.comp_scales,
                           idx=idx)
    assert n == FIG["attended_per_query"] == FIG["window_tokens"] + FIG["selected_positions"]


def test_memory_ledger():
    n = int(FIG["compressed_positions_1M"])
    assert n == FIG["context_tokens"] // FIG["compress_ratio"]
    D = int(FIG["kv_head_dim"])
    payload = orc.nvfp4_payload_bytes(n, D)
    assert payload == 134_217_728                 # 524,288 x 512 x 0.5 B
    assert round(payload / 1e6) == FIG["source_layer_payload_approx_MiB"]  # the page's "134" is MB
    assert 4 * payload == FIG["four_source_layers_approx_GiB"] * 2 ** 30  # exactly 0.5 GiB
    assert orc.nvfp4_scale_bytes(n, D) == n * D // int(FIG["nvfp4_group"]) == 16_777_216
    dense = FIG["context_tokens"] * D * 2
    assert dense == FIG["dense_bf16_1M_approx_GiB"] * 2 ** 30


def test_window_bytes_per_layer():
    s = orc.SeqState(cap_comp=1, D=int(FIG["kv_head_dim"]), W=int(FIG["window_tokens"]))
    assert s.win_u8.nbytes == 65_536 and s.win_u8.nbytes // 1024 == FIG["window_layer_approx_KB"]


def test_work_ratio():
    r = FIG["attended_per_query"] / 1e6
    assert abs(1 / r - FIG["dense_ratio_approx"]) / FIG["dense_ratio_approx"] < 0.005  # 1/1562.5
    assert FIG["context_tokens"] / FIG["attended_per_query"] == 1638.4
