"""End-to-end parity of whole decode steps for the decode configurations, in the
launch configuration the bench times (DecodeRun.step through the C ABI).

Configurations 1, 2, 7 and 9 are checked on every sequence. Configurations 3
(32 x 1,048,576 tokens, 4 KV-source groups x 10 layers), 8 (8 index sources x 5
layers), 4 (the prefill chunk: 36 queries around block, tile and super-tile
boundaries) and 5 (ragged, 16 steps: every sequence's Indexer and selection at
step 0) are checked on samples, recomputed by the oracle from the
host-regenerated inputs on every host core; the device must also report a clean
status word for the whole batch."""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from csa2_compressed_sparse_02_gb300 import inputs, workloads
from oracle import reference

pytestmark = pytest.mark.gpu


def _check(run, g, s, step, readers=None, ref=None):
    cfg = run.cfg
    ref = ref if ref is not None else reference.decode_step(cfg, g, s, step, readers)
    grp = run.groups[g]
    n_c = ref["n_c"]
    assert ref["inexact"] == 0, "index inputs not exact in fp32"
    assert int(grp["src"].n_tokens[s].item()) == ref["T"]
    got = grp["scores"][s, :n_c].cpu().numpy()
    assert np.array_equal(got, ref["scores"]), (g, s, np.nonzero(got != ref["scores"])[0][:5])
    nb = math.ceil(n_c / 8)
    assert np.array_equal(grp["bmax"][s, :nb].cpu().numpy(), ref["block_max"])
    assert int(grp["n_sel"][s].item()) == ref["n_sel"]
    assert np.array_equal(grp["idx"][s].cpu().numpy(), ref["idx"])
    for r, e in ref["out"].items():
        o = grp["out"][r][s].float().cpu().numpy().astype(np.float64)
        err = np.abs(o - e).max()
        rel = np.linalg.norm(o - e) / np.linalg.norm(e)
        if cfg.quant:
            assert err <= 1.5e-2 and rel <= 4e-3, (g, r, s, err, rel)
        else:
            assert err <= 1e-4 and rel <= 1e-5, (g, r, s, err, rel)
    return ref


def test_config1_full():
    cfg = inputs.CONFIGS[1]
    run = workloads.DecodeRun(cfg, n_steps=1)
    run.step()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    ref = _check(run, 0, 0, 0)
    assert ref["n_c"] == 2048 and ref["n_sel"] == 512 and ref["attended"] == 640


def test_config2_full():
    cfg = inputs.CONFIGS[2]
    run = workloads.DecodeRun(cfg, n_steps=1)
    run.step()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    for s in range(cfg.B):
        ref = _check(run, 0, s, 0)
        # planted keys sit far above the rest and are always selected
        pos, _, _ = inputs.plants(cfg, 0, s)
        assert set(pos.tolist()) <= set(ref["idx"].tolist())
        sc = ref["scores"]
        unpl = np.delete(sc, pos)
        assert sc[pos].min() >= unpl.mean() + 8 * unpl.std()


def test_config7_ratio_one_full():
    """1:1 layers: n_c = T compressed positions, each one raw token quantised."""
    cfg = inputs.CONFIGS[7]
    run = workloads.DecodeRun(cfg, n_steps=1)
    run.step()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    for s in range(cfg.B):
        ref = _check(run, 0, s, 0)
        assert ref["n_c"] == cfg.T and ref["n_sel"] == 512
        pos, _, _ = inputs.plants(cfg, 0, s)
        assert set(pos.tolist()) <= set(ref["idx"].tolist())


def test_config9_compressed_kv_rope_full():
    """Configuration 2 with the compressed KV rotated by the Compressor (YaRN, base
    160000, factor 16, last 64 dims): every sequence's whole decode step."""
    cfg = inputs.CONFIGS[9]
    run = workloads.DecodeRun(cfg, n_steps=1)
    assert run.params.rope_dim == inputs.ROPE_DIM
    run.step()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    for s in range(cfg.B):
        ref = _check(run, 0, s, 0)
        assert ref["n_sel"] == 512 and ref["attended"] == 640


def test_config3_sampled():
    cfg = inputs.CONFIGS[3]
    run = workloads.DecodeRun(cfg, n_steps=1)
    run.step()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    for g, s in ((0, 0), (3, 31)):
        _check(run, g, s, 0, readers=[0, 9])
    # every sequence of every group selected 512 positions, ascending
    for grp in run.groups:
        assert torch.all(grp["n_sel"] == 512)
        idx = grp["idx"].cpu().numpy()
        assert np.all(np.diff(idx, axis=1) > 0)


def test_config5_sampled_over_16_steps():
    """Ragged batch over 16 steps: at step 0 every sequence's Indexer scores, block
    maxima and selection (and the shortest one's attention); after the last step
    the attention of the shortest, the longest and one more sequence."""
    cfg = inputs.CONFIGS[5]
    run = workloads.DecodeRun(cfg, n_steps=cfg.steps)
    T0 = cfg.first_lengths()
    for k in range(cfg.steps):
        run.step()
        if k == 0:
            torch.cuda.synchronize()
            grp = run.groups[0]
            scores, bmax = grp["scores"].cpu().numpy(), grp["bmax"].cpu().numpy()
            idx, n_sel = grp["idx"].cpu().numpy(), grp["n_sel"].cpu().numpy()
            sel = _oracle_map(lambda s: reference.index_and_select(cfg, 0, s, 0), list(range(cfg.B)))
            for s, ref in enumerate(sel):
                n_c = ref["n_c"]
                assert ref["inexact"] == 0 and n_c == T0[s] // cfg.ratio
                assert np.array_equal(scores[s, :n_c], ref["scores"]), s
                assert np.array_equal(bmax[s, :math.ceil(n_c / 8)], ref["block_max"]), s
                assert n_sel[s] == ref["n_sel"] and np.array_equal(idx[s], ref["idx"]), s
            _check(run, 0, int(np.argmin(T0)), 0, readers=[0, 5])
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    picks = (int(np.argmin(T0)), int(np.argmax(T0)), 7)
    refs = _oracle_map(lambda s: reference.decode_step(cfg, 0, s, cfg.steps - 1, [0, 3, 5]), picks)
    for s, ref in zip(picks, refs):
        _check(run, 0, s, cfg.steps - 1, ref=ref)


def test_config8_eight_index_sources_sampled():
    """The 8-index-source step (8 scans, 8 selections, 5 layers each): 2 sequences
    of 2 index sources, whole steps."""
    cfg = inputs.CONFIGS[8]
    run = workloads.DecodeRun(cfg, n_steps=1)
    run.step()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    units = [(0, 0), (0, 31), (7, 5), (7, 31)]
    refs = _oracle_map(lambda gs: reference.decode_step(cfg, gs[0], gs[1], 0, [0, 4]), units)
    for (g, s), ref in zip(units, refs):
        _check(run, g, s, 0, ref=ref)
    for grp in run.groups:
        assert torch.all(grp["n_sel"] == 512)


def _oracle_map(fn, items):
    """fn over items on every host core (the oracle's C calls release the GIL)."""
    with ThreadPoolExecutor(max_workers=max(1, min(len(items), os.cpu_count() or 1))) as ex:
        return list(ex.map(fn, items))


# Prefill queries checked: the first and last of several 16-query blocks of the
# shared-key Indexer, and queries around the causal lengths that cross a 128-position
# key tile (n_c = 131,072 + (i + 1) // 2 reaches 131,200 at i = 255) and a
# 512-position super-tile (i = 1023) boundary, then the chunk's end.
PREFILL_QUERIES = (0, 1, 2, 3, 14, 15, 16, 17, 31, 32, 254, 255, 256, 257, 510, 511, 512, 1022,
                   1023, 1024, 1025, 2047, 2048, 2049, 3071, 3072, 4095, 4096, 4097, 6143, 6144,
                   8175, 8176, 8177, 8190, 8191)


def test_config4_prefill_sampled_queries():
    """Prefill chunk: 8,192 queries on a 262,144-token context (135,168 compressed
    positions visible at the end), per-query causal Indexer, selection and
    attention with a causal 128-token window."""
    cfg = inputs.PREFILL
    run = workloads.PrefillRun(cfg)
    run.run()
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    assert int(run.src.n_tokens.item()) == cfg.T0 + cfg.chunk
    assert int(run.n_sel.min().item()) == 512
    refs = _oracle_map(lambda i: reference.decode_step(cfg, 0, 0, i, readers=[0]), PREFILL_QUERIES)
    for i, ref in zip(PREFILL_QUERIES, refs):
        n_c = ref["n_c"]
        assert n_c == (cfg.T0 + i + 1) // 2 and ref["inexact"] == 0
        got = run.scores[i, :n_c].cpu().numpy()
        assert np.array_equal(got, ref["scores"]), (i, np.nonzero(got != ref["scores"])[0][:5])
        nb = math.ceil(n_c / 8)
        assert np.array_equal(run.bmax[i, :nb].cpu().numpy(), ref["block_max"]), i
        assert np.array_equal(run.idx[i].cpu().numpy(), ref["idx"]), i
        o = run.out[0, i].float().cpu().numpy().astype(np.float64)
        e = ref["out"][0]
        err = np.abs(o - e).max()
        rel = np.linalg.norm(o - e) / np.linalg.norm(e)
        assert err <= 1.5e-2 and rel <= 4e-3, (i, err, rel)


def test_pipelined_steps_overlapped_copies_config1():
    """The end-to-end loop the bench times: per-step inputs sent from pinned host
    memory and outputs read back on side streams, overlapped with the neighbouring
    steps (double-buffered outputs). Each step's host outputs match the oracle."""
    cfg = inputs.CONFIGS[1]
    K = 5
    run = workloads.DecodeRun(cfg, n_steps=K + 1, out_slots=2)
    assert run.n_prep % 2 == 0
    assert run.capture()
    host_in = {k: run.host_input_pairs(k) for k in range(run.n_prep)}
    # scramble the device slots: the step must use what was sent from the host
    for grp in run.groups:
        for name in ("kv", "gate", "kv_rd", "q", "iq", "iw"):
            if name in grp:
                grp[name].zero_()
    outs = [torch.empty(run.outputs_of_slot(0).shape, dtype=run.outputs_of_slot(0).dtype,
                        pin_memory=True) for _ in range(K)]
    stream = torch.cuda.current_stream()
    run.pipelined_steps(K, host_in, lambda i: outs[i], stream)
    torch.cuda.synchronize()
    assert run.dev_status.item() == 0
    for k in (0, 1, K - 1):
        ref = reference.decode_step(cfg, 0, 0, k)
        for r, e in ref["out"].items():
            o = outs[k][0][r][0].float().numpy().astype(np.float64)
            err = np.abs(o - e).max()
            rel = np.linalg.norm(o - e) / np.linalg.norm(e)
            assert err <= 1.5e-2 and rel <= 4e-3, (k, r, err, rel)
