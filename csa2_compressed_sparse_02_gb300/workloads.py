"""Device side of the CSA2 decode configurations: builds a configuration's
caches and per-step inputs on the GPU from the seeded generator (the recipe is
in ``inputs.py``) and enqueues decode steps through the C ABI (``api.py``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import synth
from .inputs import CONFIGS, D, DI, H, HI, ROPE_DIM, W, DecodeConfig, plants  # noqa: F401

# =============================================================================== device side
@dataclass
class DecodeRun:
    """Device state of one decode configuration, ready to run `n_steps` steps.

    Per-step inputs (new tokens, queries, index queries) are generated for
    min(n_steps, max_prepared) steps and reused cyclically beyond that; the
    caches always advance by one token per step."""
    cfg: DecodeConfig
    n_steps: int
    device: str = "cuda"
    max_prepared: int = 64
    cuda_core_indexer: bool = False
    fused_attention: bool = True
    # fused attention with the (unit, tile) work cut evenly over the CTAs
    split_attention: bool = True
    # attention outputs per input slot parity (2: a step's outputs can be read back
    # while the next step writes its own; the prepared slot count is then even)
    out_slots: int = 1
    step_done: int = 0
    groups: list = field(default_factory=list)

    def __post_init__(self):
        import torch

        from . import api
        self.torch, self.api = torch, api
        cfg, dev = self.cfg, self.device
        self.T0 = cfg.first_lengths()
        self.B = cfg.B
        self.n_prep = max(1, min(self.n_steps, self.max_prepared))
        assert self.out_slots in (1, 2)
        if self.out_slots == 2:
            self.n_prep = max(2, self.n_prep - self.n_prep % 2)
        rope = dict(rope_dim=ROPE_DIM) if cfg.rope else {}
        if cfg.quant:
            self.params = api.default_params(compress_ratio=cfg.ratio, **rope)
        else:
            self.params = api.default_params(kv_format=api.F32, win_format=api.F32,
                                             q_format=api.F32, compress_ratio=cfg.ratio, **rope)
        last = [T + self.n_steps - 1 for T in self.T0]          # T after the last step
        rt = cfg.ratio
        self.comp_caps = [t // rt + 1 for t in last]
        self.n_c_max = max(t // rt for t in last)
        self.key_rows = [max(1, t // rt) for t in last]
        # rows of the score and block-max arrays 16-byte aligned: vector loads in the selection
        self.max_ncomp = -(-self.n_c_max // 32) * 32
        self.n_b_max = math.ceil(self.max_ncomp / 8)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = api.sparse_attn_workspace_size(self.params, self.B)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.attn_ws = None
        if cfg.quant and self.fused_attention and self.split_attention:
            # sized for the full grid (max_ctas 0), so it also serves capped grids
            self.attn_ws = api.sparse_attn_layers_split_workspace(self.params, cfg.readers, self.B,
                                                                  device=dev)
        qdt = torch.bfloat16 if cfg.quant else torch.float32
        # Per-step inputs of every group live in one contiguous slot per prepared
        # step (in_buf[k]) and the attention outputs of every group in one buffer per
        # output slot (out_buf_all[k % out_slots]): a caller sends a step's inputs
        # with one copy and reads its outputs back with one.
        R, G, Bn = cfg.readers, cfg.groups, self.B
        shapes = [("kv", (Bn, 1, D), torch.float32), ("gate", (Bn, 1, D), torch.float32)]
        if R > 1:
            shapes.append(("kv_rd", (Bn * (R - 1), 1, D), torch.float32))
        shapes += [("q", (R, Bn, H, D), qdt), ("iq", (Bn, HI, DI // 2), torch.uint8),
                   ("iw", (Bn, HI), torch.float32)]
        layout, off = [], 0
        for g in range(G):
            for name, shp, dt in shapes:
                nbytes = math.prod(shp) * torch.empty((), dtype=dt).element_size()
                layout.append((g, name, shp, dt, off))
                off += -(-nbytes // 256) * 256
        self.slot_bytes = off
        self.in_buf = torch.empty(self.n_prep, off, dtype=torch.uint8, device=dev)
        self.out_buf_all = torch.empty(self.out_slots, G, R, Bn, H, D, dtype=qdt, device=dev)
        for g in range(cfg.groups):
            grp = {}
            grp["src"] = api.LayerCache(self.B, self.comp_caps, self.params, device=dev)
            if cfg.readers > 1:
                grp["rd"] = api.LayerCache(self.B * (cfg.readers - 1), [1] * (self.B * (cfg.readers - 1)),
                                           self.params, has_comp=False, device=dev)
            grp["keys"] = api.IndexKeyCache(self.key_rows, device=dev)
            if cfg.readers > 1:
                grp["win_all"] = torch.cat([grp["src"].win_ptrs, grp["rd"].win_ptrs])
            else:
                grp["win_all"] = grp["src"].win_ptrs
            grp["scores"] = torch.empty(self.B, self.max_ncomp, dtype=torch.float32, device=dev)
            grp["bmax"] = torch.empty(self.B, self.n_b_max, dtype=torch.float32, device=dev)
            grp["idx"] = torch.empty(self.B, 512, dtype=torch.int32, device=dev)
            grp["n_sel"] = torch.empty(self.B, dtype=torch.int32, device=dev)
            grp["out_buf"] = self.out_buf_all[:, g]
            grp["out_all"] = grp["out_buf"][0]
            grp["out"] = list(grp["out_all"].unbind(0))
            grp["sink_all"] = torch.empty(cfg.readers, H, dtype=torch.float32, device=dev)
            grp["sink"] = list(grp["sink_all"].unbind(0))
            # per-step inputs, resident before timing: [n_prep, ...] views into in_buf
            for gg, name, shp, dt, o in layout:
                if gg != g:
                    continue
                es = torch.empty((), dtype=dt).element_size()
                inner = [1]
                for n in reversed(shp[1:]):
                    inner.insert(0, inner[0] * n)
                grp[name] = self.in_buf.view(dt).as_strided(
                    (self.n_prep,) + shp, (off // es,) + tuple(inner), o // es)
            grp["iqs"] = torch.full((self.n_prep, self.B, HI, DI // 16), synth.E4M3_ONE,
                                    dtype=torch.uint8, device=dev)
            self.groups.append(grp)
        self._fill()

    # ------------------------------------------------------------------ setup
    def _keys(self, kind, layer):
        return [synth.stream_key(self.cfg.seed, kind, layer, s) for s in range(self.B)]

    def _prefill_source(self, g, grp, chunk=8192):
        """Compressor over raw tokens [0, T0-1) of every sequence of the group's source."""
        torch, cfg, src = self.torch, self.cfg, grp["src"]
        lay = cfg.layer(g, 0)
        for seqs in self._seq_sets():
            n_pre = self.T0[seqs[0]] - 1
            nb = len(seqs)
            sl = slice(seqs[0], seqs[0] + nb)
            view = _CacheView(src, sl)
            kvk = [synth.stream_key(cfg.seed, synth.KV, lay, s) for s in seqs]
            gk = [synth.stream_key(cfg.seed, synth.GATE, lay, s) for s in seqs]
            ch = max(1, min(chunk, (1 << 29) // (nb * D * 8)))
            kv = torch.empty(nb, ch, D, dtype=torch.float32, device=self.device)
            gt = torch.empty_like(kv)
            for t0 in range(0, n_pre, ch):
                n = min(ch, n_pre - t0)
                synth.gpu_fill(synth.G_NORMAL_F32, kvk, t0 * D, n * D, kv, stride=n * D)
                synth.gpu_fill(synth.G_NORMAL_F32, gk, t0 * D, n * D, gt, stride=n * D)
                self.api.compress_append(self.params, kv.view(-1)[:nb * n * D].view(nb, n, D),
                                         gt.view(-1)[:nb * n * D].view(nb, n, D), view.pend_kv,
                                         view.pend_gate, view.comp_ptrs, view.comp_scale_ptrs,
                                         view.comp_cap, view.win_ptrs, view.n_tokens,
                                         self.dev_status)

    def _seq_sets(self):
        """Sequences grouped by first length (all of them at once when uniform)."""
        if len(set(self.T0)) == 1:
            return [list(range(self.B))]
        return [[s] for s in range(self.B)]

    def _prefill_readers(self, g, grp):
        """Windows of the readers: raw tokens [T0-W, T0-1) of each reader layer."""
        torch, cfg, rd = self.torch, self.cfg, grp["rd"]
        for r in range(1, cfg.readers):
            lay = cfg.layer(g, r)
            for seqs in self._seq_sets():
                T0 = self.T0[seqs[0]]
                t_start = max(0, T0 - W)
                n = T0 - 1 - t_start
                i0 = (r - 1) * self.B + seqs[0]
                view = _CacheView(rd, slice(i0, i0 + len(seqs)))
                view.n_tokens.fill_(t_start)
                if n <= 0:
                    continue
                kv = torch.empty(len(seqs), n, D, dtype=torch.float32, device=self.device)
                synth.gpu_fill(synth.G_NORMAL_F32,
                               [synth.stream_key(cfg.seed, synth.KV, lay, s) for s in seqs],
                               t_start * D, n * D, kv)
                self.api.compress_append(self.params, kv, None, None, None, None, None, None,
                                         view.win_ptrs, view.n_tokens, self.dev_status)

    def _fill(self):
        torch, cfg = self.torch, self.cfg
        for g, grp in enumerate(self.groups):
            self._prefill_source(g, grp)
            if cfg.readers > 1:
                self._prefill_readers(g, grp)
            keys = grp["keys"]
            for s in range(self.B):
                n = self.key_rows[s]
                kv = torch.empty(n, DI // 2, dtype=torch.uint8, device=self.device)
                ks = torch.empty(n, DI // 16, dtype=torch.uint8, device=self.device)
                synth.gpu_fill(synth.G_E2M1_BYTES, [synth.stream_key(cfg.seed, synth.IDX_K, g, s)],
                               0, n * DI // 2, kv)
                if cfg.kscale_pow2:
                    synth.gpu_fill(synth.G_SCALE_POW2_BYTES,
                                   [synth.stream_key(cfg.seed, synth.IDX_K_SCALE, g, s)], 0,
                                   n * DI // 16, ks)
                else:
                    ks.fill_(synth.E4M3_ONE)
                pos, rv, rs = plants(cfg, g, s)
                pos = pos[pos < n]
                if pos.size:
                    pi = torch.from_numpy(pos).to(self.device)
                    kv[pi] = torch.from_numpy(np.tile(rv, (pos.size, 1))).to(self.device)
                    ks[pi] = torch.from_numpy(np.tile(rs, (pos.size, 1))).to(self.device)
                keys.write_seq(self.params, s, kv, ks, 0, self.dev_status)
            for r in range(cfg.readers):
                lay = cfg.layer(g, r)
                synth.gpu_fill(synth.G_NORMAL_F32, [synth.stream_key(cfg.seed, synth.SINK, lay, 0)],
                               0, H, grp["sink"][r])
            qkind = synth.G_NORMAL_BF16 if cfg.quant else synth.G_NORMAL_F32
            for k in range(self.n_prep):
                for seqs in self._seq_sets():
                    tok = self.T0[seqs[0]] - 1 + k  # raw position of this step's token
                    s0, nb = seqs[0], len(seqs)
                    for r in range(cfg.readers):
                        lay = cfg.layer(g, r)
                        kk = [synth.stream_key(cfg.seed, synth.KV, lay, s) for s in seqs]
                        if r == 0:
                            gk = [synth.stream_key(cfg.seed, synth.GATE, lay, s) for s in seqs]
                            synth.gpu_fill(synth.G_NORMAL_F32, kk, tok * D, D,
                                           grp["kv"][k, s0:s0 + nb], stride=D)
                            synth.gpu_fill(synth.G_NORMAL_F32, gk, tok * D, D,
                                           grp["gate"][k, s0:s0 + nb], stride=D)
                        else:
                            i0 = (r - 1) * self.B + s0
                            synth.gpu_fill(synth.G_NORMAL_F32, kk, tok * D, D,
                                           grp["kv_rd"][k, i0:i0 + nb], stride=D)
                for r in range(cfg.readers):
                    synth.gpu_fill(qkind, self._keys(synth.Q, cfg.layer(g, r)), k * H * D, H * D,
                                   grp["q"][k, r])
                synth.gpu_fill(synth.G_E2M1_BYTES, [synth.stream_key(cfg.seed, synth.IDX_Q, g, s)
                                                    for s in range(self.B)],
                               k * HI * DI // 2, HI * DI // 2, grp["iq"][k])
                synth.gpu_fill(synth.G_W_POW2_F32, [synth.stream_key(cfg.seed, synth.IDX_W, g, s)
                                                    for s in range(self.B)], k * HI, HI, grp["iw"][k])
        torch.cuda.synchronize()

    # ------------------------------------------------------------------ one step
    def _timed(self, timers, cat, st, fn, *args):
        """Run fn(st, *args) (which enqueues on stream st), bracketed by timing
        events on st when timers is a dict."""
        if timers is None:
            fn(st, *args)
            return
        torch = self.torch
        kw = {"enable_timing": True}
        if getattr(self, "_external_events", False):
            kw["external"] = True
        e0, e1 = torch.cuda.Event(**kw), torch.cuda.Event(**kw)
        e0.record(st)
        fn(st, *args)
        e1.record(st)
        timers.setdefault(cat, []).append((e0, e1))

    # the four calls of a group's step, each enqueued on stream s
    def _compress(self, s, grp, k):
        src, cfg = grp["src"], self.cfg
        src.append(grp["kv"][k], grp["gate"][k], self.dev_status, s)
        if cfg.readers > 1:
            grp["rd"].append(grp["kv_rd"][k], None, self.dev_status, s)

    def _index(self, s, grp, k, params):
        self.api.index_scores(params, self.max_ncomp, grp["iq"][k], grp["iqs"][k], grp["iw"][k],
                              grp["keys"].ptrs, grp["src"].n_tokens, grp["scores"], grp["bmax"],
                              self.dev_status, s, cuda_cores=self.cuda_core_indexer)

    def _select(self, s, grp, k):
        self.api.select_topk(self.params, self.max_ncomp, grp["scores"], grp["bmax"],
                             grp["src"].n_tokens, grp["idx"], grp["n_sel"], self.dev_status, s)

    def out_of_slot(self, grp, k):
        """Attention outputs [readers, B, H, D] written by the step of input slot k."""
        return grp["out_buf"][k % self.out_slots]

    def outputs_of_slot(self, k):
        """Attention outputs of every group [groups, readers, B, H, D] (contiguous)
        written by the step of input slot k."""
        return self.out_buf_all[k % self.out_slots]

    def _attn(self, s, grp, k, params):
        api, cfg, src = self.api, self.cfg, grp["src"]
        out_all = self.out_of_slot(grp, k)
        if cfg.quant and self.fused_attention:
            api.sparse_attn_layers(params, grp["q"][k], grp["sink_all"], grp["win_all"],
                                   src.n_tokens, src.comp_ptrs, src.comp_scale_ptrs, grp["idx"],
                                   out_all, self.dev_status, s, workspace=self.attn_ws)
            return
        for r in range(cfg.readers):
            if r == 0:
                win_ptrs, n_tok = src.win_ptrs, src.n_tokens
            else:
                sl = slice((r - 1) * self.B, r * self.B)
                win_ptrs, n_tok = grp["rd"].win_ptrs[sl], grp["rd"].n_tokens[sl]
            api.sparse_attn(self.params, grp["q"][k, r], grp["sink"][r], win_ptrs, n_tok,
                            src.comp_ptrs, src.comp_scale_ptrs, grp["idx"], out_all[r],
                            self.workspace, self.dev_status, s)

    def _enqueue(self, k, stream=None, timers=None, timer_cats=None, timer_groups=None):
        """Enqueue one decode step (every group, every layer) using input slot k.
        timers: optional dict receiving (start, end) CUDA events per call category
        ("compress", "index", "select", "attn"), recorded on the launching stream;
        timer_cats / timer_groups restrict the events to those categories / group
        indices (None: all). Groups run in layer order: group g+1's index query
        comes from the hidden state after group g's layers, so its scan cannot
        start earlier."""
        st = self.torch.cuda.current_stream() if stream is None else stream

        def tm(cat, g):
            keep = timers is not None and (timer_cats is None or cat in timer_cats) and (
                timer_groups is None or g in timer_groups)
            return timers if keep else None

        for g, grp in enumerate(self.groups):
            self._timed(tm("compress", g), "compress", st, self._compress, grp, k)
            self._timed(tm("index", g), "index", st, self._index, grp, k, self.params)
            self._timed(tm("select", g), "select", st, self._select, grp, k)
            self._timed(tm("attn", g), "attn", st, self._attn, grp, k, self.params)

    def step(self, stream=None, timers=None):
        """Enqueue the next decode step eagerly (one launch per kernel)."""
        assert self.step_done < self.n_steps, "more steps than the caches were sized for"
        self._enqueue(self.step_done % self.n_prep, stream, timers)
        self.step_done += 1

    def capture(self, with_timers=False, timer_cats=None, timer_groups=None):
        """Capture one CUDA graph per prepared input slot (a whole step each) as the
        graphs step_graph() replays. Timing events (with_timers; restricted by
        timer_cats / timer_groups as in _enqueue) are recorded inside the graphs:
        each one orders the kernels around it fully, so they cost step time.
        Returns False if the timers were requested but this torch cannot record
        events inside a graph."""
        got = self.capture_set(with_timers, timer_cats, timer_groups)
        if got is None:
            return False
        self.graphs, self.graph_timers = got
        return True

    def capture_set(self, with_timers=False, timer_cats=None, timer_groups=None):
        """Capture a set of per-slot step graphs without installing it: returns
        (graphs, timers per graph), or None if events cannot be recorded in a graph."""
        torch = self.torch
        self._external_events = False
        if with_timers:
            try:
                torch.cuda.Event(enable_timing=True, external=True)
                self._external_events = True
            except TypeError:
                return None
        graphs, graph_timers = [], []
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        for k in range(self.n_prep):
            g = torch.cuda.CUDAGraph()
            tm = {} if with_timers else None
            with torch.cuda.graph(g, stream=cs):
                self._enqueue(k, None, tm, timer_cats, timer_groups)
            graphs.append(g)
            graph_timers.append(tm)
        torch.cuda.current_stream().wait_stream(cs)
        return graphs, graph_timers

    def step_graph(self):
        """Replay the captured step of the next input slot on the current stream."""
        assert self.step_done < self.n_steps, "more steps than the caches were sized for"
        self.graphs[self.step_done % self.n_prep].replay()
        self.step_done += 1

    def host_input_pairs(self, k):
        """(pinned host copy, device slot) pairs of the per-step inputs of slot k: one
        pair, the whole contiguous slot in_buf[k] of every group's inputs, the host
        copy filled from the device slot (the data a caller would send)."""
        torch = self.torch
        d = self.in_buf[k]
        h = torch.empty(d.shape, dtype=d.dtype, pin_memory=True)
        h.copy_(d)
        return [(h, d)]

    def pipelined_steps(self, K, host_in, host_out_of, stream):
        """K steps with every step's inputs sent from pinned host memory and its
        attention outputs read back, the copies overlapped with the neighbouring
        steps' compute: step i+1's inputs travel on one side stream into their own
        prepared slot while step i computes on `stream`, and step i's outputs
        (double-buffered by slot parity; needs out_slots=2) travel back on another
        while step i+1 computes (captured graphs when capture() ran, else eager).
        host_in: slot -> list of (host, device) pairs (host_input_pairs);
        host_out_of(i): the pinned host tensor shaped like outputs_of_slot(k) that
        receives step i's outputs (one copy). Everything is enqueued; on return
        `stream` waits for every copy."""
        torch = self.torch
        assert self.out_slots == 2, "needs out_slots=2"
        graphs = bool(getattr(self, "graphs", None))
        n_prep, slot0 = self.n_prep, self.step_done
        slot = lambda i: (slot0 + i) % n_prep
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in range(K)]
        comp_done = [torch.cuda.Event() for _ in range(K)]
        out_done = [torch.cuda.Event() for _ in range(K)]
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)

        def send(i):
            if i - n_prep >= 0:  # the slot was last read by step i - n_prep
                s_in.wait_event(comp_done[i - n_prep])
            with torch.cuda.stream(s_in):
                for h, d in host_in[slot(i)]:
                    d.copy_(h, non_blocking=True)
            in_done[i].record(s_in)

        if K > 0:
            send(0)
        with torch.cuda.stream(stream):
            for i in range(K):
                stream.wait_event(in_done[i])
                if i >= 2:  # the output buffer of this slot parity was read back
                    stream.wait_event(out_done[i - 2])
                if graphs:
                    self.step_graph()
                else:
                    self.step(stream)
                comp_done[i].record(stream)
                if i + 1 < K:
                    send(i + 1)
                s_out.wait_event(comp_done[i])
                with torch.cuda.stream(s_out):
                    host_out_of(i).copy_(self.outputs_of_slot(slot(i)), non_blocking=True)
                out_done[i].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    def tokens_after(self, s: int) -> int:
        return self.T0[s] - 1 + self.step_done

    def launches_per_step(self) -> int:
        """Kernels of this library one step launches (see step())."""
        n = 0
        for _ in self.groups:
            n += 1 + (1 if self.cfg.readers > 1 else 0)   # compress / window appends
            n += 1 + 1                                    # Indexer, selection
            if self.cfg.quant and self.fused_attention:
                n += 1                                    # fused multi-layer attention
            else:
                n += 2 * self.cfg.readers                  # attention split pass + merge
        return n

    def scan_bytes(self) -> float:
        """Algorithmic bytes of one Indexer launch at the current step: 72 B of
        key read + 4 B score + 0.5 B block max written per position."""
        return sum((T - 1 + self.step_done) // self.cfg.ratio for T in self.T0) * 76.5

    def attn_bytes_per_call(self) -> float:
        """Algorithmic bytes of one sparse-attention call: per sequence the
        window (128 x 512 B), the selected rows (512 x 288 B), q and out
        (64 x 512 x 2 B each) and idx (512 x 4 B)."""
        per = 128 * 512 + 512 * 288 + 2 * 64 * 512 * 2 + 512 * 4
        if not self.cfg.quant:
            per = 128 * 2048 + 512 * 2048 + 2 * 64 * 512 * 4 + 512 * 4
        return per * self.B


class _CacheView:
    """A contiguous slice of a LayerCache's sequences, addressable on its own."""

    def __init__(self, cache, sl: slice):
        self.pend_kv = cache.pend_kv[sl]
        self.pend_gate = cache.pend_gate[sl]
        self.n_tokens = cache.n_tokens[sl]
        self.comp_ptrs = cache.comp_ptrs[sl] if cache.comp_ptrs is not None else None
        self.comp_scale_ptrs = cache.comp_scale_ptrs[sl] if cache.comp_scale_ptrs is not None else None
        self.comp_cap = cache.comp_cap[sl]
        self.win_ptrs = cache.win_ptrs[sl]


class PrefillRun:
    """Device state of a prefill chunk (inputs.PrefillConfig): the prior context is
    compressed into the cache, then run() appends the chunk and computes, for
    every query of the chunk, its Indexer scores over the compressed positions it
    sees, its two-level selection and its sparse attention (window rows from a
    linear buffer built before the append)."""

    def __init__(self, cfg, device="cuda", index_batch=1024, shared_indexer=True):
        import torch

        from . import api
        self.torch, self.api, self.cfg, self.device = torch, api, cfg, device
        self.index_batch = index_batch
        # shared_indexer: every query of the chunk against the one key stream as an FP4
        # GEMM (csa2_index_scores_shared); else the decode Indexer with one "sequence"
        # per query (csa2_index_scores, index_batch queries per call)
        self.shared_indexer = shared_indexer
        T0, n = cfg.T0, cfg.chunk
        self.n_c_final = (T0 + n) // 2
        self.params = api.default_params()
        self.params_lin = api.default_params(win_layout=api.WIN_LINEAR)
        dev = device
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.src = api.LayerCache(1, [self.n_c_final + 1], self.params, device=dev)
        # prior context through the Compressor
        kvk = [synth.stream_key(cfg.seed, synth.KV, 0, 0)]
        gk = [synth.stream_key(cfg.seed, synth.GATE, 0, 0)]
        ch = 65536
        kv = torch.empty(1, ch, D, dtype=torch.float32, device=dev)
        gt = torch.empty_like(kv)
        for t0 in range(0, T0, ch):
            m = min(ch, T0 - t0)
            synth.gpu_fill(synth.G_NORMAL_F32, kvk, t0 * D, m * D, kv)
            synth.gpu_fill(synth.G_NORMAL_F32, gk, t0 * D, m * D, gt)
            self.src.append(kv[:, :m], gt[:, :m], self.dev_status)
        # the chunk's raw tokens
        self.kv = torch.empty(1, n, D, dtype=torch.float32, device=dev)
        self.gate = torch.empty_like(self.kv)
        synth.gpu_fill(synth.G_NORMAL_F32, kvk, T0 * D, n * D, self.kv)
        synth.gpu_fill(synth.G_NORMAL_F32, gk, T0 * D, n * D, self.gate)
        # index keys of every compressed position the chunk will expose
        self.keys = api.IndexKeyCache([self.n_c_final], device=dev)
        nk = self.n_c_final
        kv8 = torch.empty(nk, DI // 2, dtype=torch.uint8, device=dev)
        ks8 = torch.empty(nk, DI // 16, dtype=torch.uint8, device=dev)
        synth.gpu_fill(synth.G_E2M1_BYTES, [synth.stream_key(cfg.seed, synth.IDX_K, 0, 0)], 0,
                       nk * DI // 2, kv8)
        synth.gpu_fill(synth.G_SCALE_POW2_BYTES, [synth.stream_key(cfg.seed, synth.IDX_K_SCALE, 0, 0)],
                       0, nk * DI // 16, ks8)
        pos, rv, rs = plants(cfg, 0, 0)
        if pos.size:
            pi = torch.from_numpy(pos).to(dev)
            kv8[pi] = torch.from_numpy(np.tile(rv, (pos.size, 1))).to(dev)
            ks8[pi] = torch.from_numpy(np.tile(rs, (pos.size, 1))).to(dev)
        self.keys.write_seq(self.params, 0, kv8, ks8, 0, self.dev_status)
        del kv8, ks8
        # per-query inputs (query i = step i of the recipe)
        self.iq = torch.empty(n, HI, DI // 2, dtype=torch.uint8, device=dev)
        synth.gpu_fill(synth.G_E2M1_BYTES, [synth.stream_key(cfg.seed, synth.IDX_Q, 0, 0)], 0,
                       n * HI * DI // 2, self.iq)
        self.iqs = torch.full((n, HI, DI // 16), synth.E4M3_ONE, dtype=torch.uint8, device=dev)
        self.iw = torch.empty(n, HI, dtype=torch.float32, device=dev)
        synth.gpu_fill(synth.G_W_POW2_F32, [synth.stream_key(cfg.seed, synth.IDX_W, 0, 0)], 0,
                       n * HI, self.iw)
        self.q = torch.empty(1, n, H, D, dtype=torch.bfloat16, device=dev)
        synth.gpu_fill(synth.G_NORMAL_BF16, [synth.stream_key(cfg.seed, synth.Q, 0, 0)], 0,
                       n * H * D, self.q)
        self.sink = torch.empty(1, H, dtype=torch.float32, device=dev)
        synth.gpu_fill(synth.G_NORMAL_F32, [synth.stream_key(cfg.seed, synth.SINK, 0, 0)], 0, H,
                       self.sink)
        # per-query views of the one sequence
        self.n_tok_q = torch.arange(T0 + 1, T0 + 1 + n, dtype=torch.int32, device=dev)
        self.key_ptrs = self.keys.ptrs[:1].repeat(n)
        self.comp_ptrs = self.src.comp_ptrs[:1].repeat(n)
        self.comp_scale_ptrs = self.src.comp_scale_ptrs[:1].repeat(n)
        self.winbuf = torch.empty(1, W - 1 + n, D, dtype=torch.uint8, device=dev)
        self.win_q = (self.winbuf.data_ptr() +
                      torch.arange(n, dtype=torch.int64, device=dev) * D)
        self.scores = torch.empty(n, self.n_c_final, dtype=torch.float32, device=dev)
        self.bmax = torch.empty(n, math.ceil(self.n_c_final / 8), dtype=torch.float32, device=dev)
        self.idx = torch.empty(n, 512, dtype=torch.int32, device=dev)
        self.n_sel = torch.empty(n, dtype=torch.int32, device=dev)
        self.out = torch.empty(1, n, H, D, dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()

    def reset(self):
        """Back to the state before run() (the chunk's rows are then rewritten with
        the same values), so the chunk can be timed repeatedly."""
        self.src.n_tokens.fill_(self.cfg.T0)

    def run(self, timers=None):
        """The chunk on the current stream. timers: optional dict receiving
        (start, end) CUDA events per call category ("append", "index", "select",
        "attn")."""
        api, n, ds, torch = self.api, self.cfg.chunk, self.dev_status, self.torch
        st = torch.cuda.current_stream()

        def timed(cat, fn):
            if timers is None:
                fn()
                return
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            timers.setdefault(cat, []).append((e0, e1))

        def append():
            api.window_linear(self.params, self.kv, self.src.win_ptrs, self.src.n_tokens, self.winbuf)
            self.src.append(self.kv, self.gate, ds)

        def index():
            if self.shared_indexer:
                api.index_scores_shared(self.params, self.n_c_final, self.iq, self.iqs, self.iw,
                                        self.keys.buf[0], self.n_tok_q, self.scores, self.bmax, ds)
                return
            for s0 in range(0, n, self.index_batch):
                s1 = min(n, s0 + self.index_batch)
                api.index_scores(self.params, self.n_c_final, self.iq[s0:s1], self.iqs[s0:s1],
                                 self.iw[s0:s1], self.key_ptrs[s0:s1], self.n_tok_q[s0:s1],
                                 self.scores[s0:s1], self.bmax[s0:s1], ds)

        timed("append", append)
        timed("index", index)
        timed("select", lambda: api.select_topk(self.params, self.n_c_final, self.scores, self.bmax,
                                                self.n_tok_q, self.idx, self.n_sel, ds))
        timed("attn", lambda: api.sparse_attn_layers(self.params_lin, self.q, self.sink, self.win_q,
                                                     self.n_tok_q, self.comp_ptrs,
                                                     self.comp_scale_ptrs, self.idx, self.out, ds))
