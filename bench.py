#!/usr/bin/env python
"""Decode benchmark: one decode step of B=4 sequences through an interleaved
8-layer CSA/HCA stack at a context of 2**20 tokens (stack_1m), on one B300.

A step, for every layer in order: append the new token of each sequence to the
layer's cache (dsv4_compress_append), then CSA layers (even) run
dsv4_index_topk + dsv4_csa_decode and HCA layers (odd) run dsv4_hca_decode.
Each step's launch sequence is captured once as a CUDA graph and replayed; the
caches (2.8 GB) and every step's inputs are resident in HBM before timing. A
step moves 393.5 MB of algorithmic bytes, more than the 126 MB L2, so no L2
flush is needed between steps.

The same JSON line also carries, measured in the same run: `layers`, one CSA
and one HCA layer of the stack timed on their own (per-layer decode tokens/s),
and `compress_1m`, the compressor streaming 2**20 tokens of 512 dims in
4096-token chunks into a ratio-4 CSA cache (with FP4 indexer keys) and a
ratio-128 HCA cache (cache GB/s read and written). `--workload` makes one of
these, or the batched CSA configuration (csa_b32_128k), the headline instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0). Under torchrun every rank runs its own four
sequences (weak scaling, no data-path collective); `value` is the tokens/s of
all ranks. `--impl reference` times the float64 CPU oracle on a bounded sample
of the same workload instead.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from compressed_sparse_kv_05_b300 import accounting, synth  # noqa: E402
from compressed_sparse_kv_05_b300 import workloads as W  # noqa: E402

METRIC = "decode tokens/s per CSA/HCA layer at 128K-1M ctx; achieved HBM GB/s vs roofline"
# workload name -> layers of one decode step. stack_1m is the headline line; the
# others are single layers of it (per-layer figures, small profiling cases) and
# the batched CSA configuration.
WORKLOADS = {
    "stack_1m": W.STACK_1M,
    "stack_1m_csa": (W.STACK_CSA,),
    "stack_1m_hca": (W.STACK_HCA,),
    "csa_b32_128k": (W.CSA_B32_128K,),
    "compress_1m": (W.COMPRESS_1M_CSA, W.COMPRESS_1M_HCA),
    "project_1m": (W.COMPRESS_1M_CSA,),
}
PROJECT_METRIC = ("projection TFLOP/s (2^20 hidden states of 4096 dims to the x, z, u, zu streams of a ratio-4 "
                  "layer with 128-dim indexer keys, RoPE on the rotated dims, 4096-token calls)")
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1400.0
DTYPE = ("fp8-e4m3 / bf16 / fp4-e2m1 storage; attention on f16 tensor-core operands with fp32 accumulation, "
         "indexer on block-scaled fp4 tensor-core operands with fp32 accumulation, pooling and softmax in fp32")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-compress", action="store_true", help="skip the compressor sub-measurement")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="stack_1m")
    ap.add_argument("--compress-tokens", type=int, default=None,
                    help="tokens of the compressor workload (a multiple of 4096; default 2^20): smaller cases "
                         "for profiling, named in the line's config")
    args = ap.parse_args()
    if args.compress_tokens:
        if args.compress_tokens % W.COMPRESS_1M_CHUNK:
            ap.error("--compress-tokens must be a multiple of the 4096-token chunk")
        W.COMPRESS_1M_TOKENS = args.compress_tokens
    return args


# ----------------------------------------------------------------------------- graphs


def upload_graphs(graphs, stream):
    """Uploads each instantiated graph to the device ahead of its first launch
    (otherwise the first launch does it, inside whatever is being timed)."""
    try:
        from cuda.bindings import runtime as rt
        st = rt.cudaStream_t(init_value=stream.cuda_stream)
        for g in graphs:
            err, = rt.cudaGraphUpload(rt.cudaGraphExec_t(init_value=g.raw_cuda_graph_exec()), st)
            if err != rt.cudaError_t.cudaSuccess:
                return False
        stream.synchronize()
        return True
    except Exception:
        return False


# ----------------------------------------------------------------------------- peaks, clocks


def tensor_peak():
    """The measured sustained dense bf16 peak (a kernel timed inside a long loop), TFLOP/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback (sustained)"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- device workload


class Stack:
    """The eight layers' caches, biases and per-step inputs, all on the device."""

    def __init__(self, dsv4, layers, steps_total, seed, extra_tokens=None):
        self.dsv4 = dsv4
        self.layers = layers
        self.steps_total = steps_total
        extra_tokens = steps_total if extra_tokens is None else extra_tokens
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        self.g = g
        self.descs, self.caches, self.bias, self.bias_u = [], [], [], []
        for li, L in enumerate(layers):
            cap = L.capacity(extra_tokens)
            desc = dsv4.layer_desc(L, cap)
            cache = dsv4.Cache(desc)
            self._fill(L, desc, cache)
            self.descs.append(desc)
            self.caches.append(cache)
            self.bias.append(0.1 * torch.randn((L.ratio, L.dim), generator=g, device="cuda"))
            self.bias_u.append(0.1 * torch.randn((L.ratio, L.idx_dim), generator=g, device="cuda")
                               if L.kind == "csa" else None)
        ws_bytes = max(dsv4.dsv4_workspace_size(d, L.heads, L.idx_heads, L.topk) for d, L in zip(self.descs, layers))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        self.topk = [torch.zeros((L.batch, max(L.topk, 1)), dtype=torch.int32, device="cuda") for L in layers]
        # per-step inputs: one contiguous buffer per step (for one H2D copy in the end-to-end run)
        self.in_specs = []
        for li, L in enumerate(layers):
            spec = [("k", (L.batch, 1, L.dim), torch.int16), ("z", (L.batch, 1, L.dim), torch.int16),
                    ("q", (L.batch, L.heads, L.dim), torch.int16)]
            if L.kind == "csa":
                spec += [("u", (L.batch, 1, L.idx_dim), torch.int16), ("zu", (L.batch, 1, L.idx_dim), torch.int16),
                         ("q_idx", (L.batch, L.idx_heads, L.idx_dim), torch.int16),
                         ("w", (L.batch, L.idx_heads), torch.float32)]
            self.in_specs.append(spec)
        self.in_bytes = 0
        self.offsets = []
        for spec in self.in_specs:
            offs = {}
            for name, shape, dt in spec:
                self.in_bytes = (self.in_bytes + 255) // 256 * 256
                offs[name] = (self.in_bytes, shape, dt)
                self.in_bytes += int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
            self.offsets.append(offs)
        self.in_bytes = (self.in_bytes + 255) // 256 * 256
        self.inbuf = torch.empty((steps_total, self.in_bytes), dtype=torch.uint8, device="cuda")
        for s in range(steps_total):
            for li, L in enumerate(layers):
                for name, (off, shape, dt) in self.offsets[li].items():
                    t = self.view(s, li, name)
                    if dt == torch.float32:
                        t.copy_(torch.rand(shape, generator=g, device="cuda"))
                    else:
                        t.copy_(torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16).view(torch.int16))
        self.plant_keys()
        H_max = max(L.heads for L in layers)
        D_max = max(L.dim for L in layers)
        B = layers[0].batch
        # one output slot per step slot, so that a step's read-back can overlap the next step
        slots = self.inbuf.shape[0]
        self.out = torch.zeros((slots, len(layers), B, H_max, D_max), dtype=torch.float32, device="cuda")
        self.lse = torch.zeros((slots, len(layers), B, H_max), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()

    def view(self, step, li, name):
        off, shape, dt = self.offsets[li][name]
        n = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
        return self.inbuf[step, off:off + n].view(dt).view(shape)

    def _fill(self, L, desc, cache):
        """Cache contents drawn directly: pooled rows ~N(0,1) quantised by the
        library's own quantisers, window tokens ~N(0,1) bf16, n_tokens = context."""
        d = self.dsv4
        g = self.g
        n_c = L.n_comp
        for b in range(L.batch):
            for r0 in range(0, n_c, 65536):
                r1 = min(n_c, r0 + 65536)
                y = torch.randn((r1 - r0, L.dim), generator=g, device="cuda")
                d.dsv4_quantize_kv_rows(y, r1 - r0, L.d_nope, L.d_rope, cache.k_nope[b, r0:r1], cache.k_scale[b, r0:r1],
                                        cache.k_rope[b, r0:r1])
                if L.kind == "csa":
                    yi = torch.randn((r1 - r0, L.idx_dim), generator=g, device="cuda")
                    d.dsv4_quantize_fp4_rows(yi, r1 - r0, L.idx_dim, cache.idx_codes[b, r0:r1],
                                             cache.idx_scales[b, r0:r1])
            cache.win_k[b].copy_(torch.randn((L.window, L.dim), generator=g, device="cuda")
                                 .to(torch.bfloat16).view(torch.int16))
        cache.n_tokens.fill_(L.n_tokens)

    def plant_keys(self):
        """1% of each CSA cache's blocks get a key aligned with the step-0 indexer
        query (4 * qbar / rms(qbar), qbar = sum_h w_h q_h), quantised to FP4."""
        d = self.dsv4
        for li, L in enumerate(self.layers):
            if L.kind != "csa" or L.planted_frac <= 0:
                continue
            cache = self.caches[li]
            cnt = max(1, math.ceil(L.planted_frac * L.n_comp))
            qi = self.view(0, li, "q_idx").view(torch.bfloat16).float()
            w = self.view(0, li, "w")
            for b in range(L.batch):
                qbar = (w[b][:, None] * qi[b]).sum(0)
                key = 4.0 * qbar / qbar.pow(2).mean().sqrt()
                idx = torch.randperm(L.n_comp, generator=self.g, device="cuda")[:cnt].sort().values
                rows = key[None].expand(cnt, -1).contiguous()
                codes = torch.empty((cnt, L.idx_dim // 2), dtype=torch.uint8, device="cuda")
                scales = torch.empty((cnt, L.idx_dim // 16), dtype=torch.uint8, device="cuda")
                d.dsv4_quantize_fp4_rows(rows, cnt, L.idx_dim, codes, scales)
                cache.idx_codes[b, idx] = codes
                cache.idx_scales[b, idx] = scales

    def step(self, s, events=None, only=None):
        """Launch one decode step (inputs of step slot s). events: dict call -> list of (start, end).
        only: run that one layer instead of the whole stack."""
        d = self.dsv4
        for li, L in enumerate(self.layers):
            if only is not None and li != only:
                continue
            desc, cache = self.descs[li], self.caches[li]
            v = lambda n: self.view(s, li, n)  # noqa: E731
            H = L.heads
            out = self.out[s, li, :, :H, :L.dim]
            lse = self.lse[s, li, :, :H]

            def timed(call, fn):
                if events is None:
                    fn()
                    return
                e0 = torch.cuda.Event(enable_timing=True, external=True)
                e1 = torch.cuda.Event(enable_timing=True, external=True)
                e0.record()
                fn()
                e1.record()
                events.setdefault(call, []).append((e0, e1))

            if L.kind == "csa":
                timed("append", lambda: d.dsv4_compress_append(desc, cache, 1, v("k"), None, v("z"), self.bias[li],
                                                               v("u"), v("zu"), self.bias_u[li]))
                timed("index_topk", lambda: d.dsv4_index_topk(desc, cache, L.idx_heads, v("q_idx"), v("w"), L.topk,
                                                              self.topk[li], None, self.ws))
                timed("csa_decode", lambda: d.dsv4_csa_decode(desc, cache, H, v("q"), L.sm_scale, self.topk[li],
                                                              L.topk, out, lse, self.ws))
            else:
                timed("append", lambda: d.dsv4_compress_append(desc, cache, 1, v("k"), None, v("z"), self.bias[li],
                                                               None, None, None))
                timed("hca_decode", lambda: d.dsv4_hca_decode(desc, cache, H, v("q"), L.sm_scale, out, lse, self.ws))


class Compress:
    """The compressor workload: one sequence of 2**20 tokens (512 dims, ~N(0,1))
    streamed in 4096-token chunks into a ratio-4 CSA cache (with 128-dim FP4
    indexer keys) and a ratio-128 HCA cache, each compressor with its own gate
    logits ~N(0,1) and position bias ~N(0,0.1). A step appends the whole stream
    to empty caches (n_tokens reset at its start), chunk by chunk. The two
    caches are independent, so their calls run on two streams (the CSA cache's
    on the caller's stream, the HCA cache's on a second stream forked from it
    and joined at the end of the step); each cache's chunks stay in order."""

    def __init__(self, dsv4, seed):
        self.dsv4 = dsv4
        self.csa, self.hca = W.COMPRESS_1M_CSA, W.COMPRESS_1M_HCA
        n, C = W.COMPRESS_1M_TOKENS, W.COMPRESS_1M_CHUNK
        self.n, self.chunk = n, C
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)

        def bf16(shape):
            t = torch.empty(shape, dtype=torch.int16, device="cuda")
            for r0 in range(0, shape[0], 1 << 18):
                r1 = min(shape[0], r0 + (1 << 18))
                t[r0:r1].copy_(torch.randn((r1 - r0,) + shape[1:], generator=g, device="cuda")
                               .to(torch.bfloat16).view(torch.int16))
            return t

        D, Di = self.csa.dim, self.csa.idx_dim
        self.x = bf16((n, D))
        self.z_csa = bf16((n, D))
        self.z_hca = bf16((n, D))
        self.u = bf16((n, Di))
        self.zu = bf16((n, Di))
        self.b_csa = 0.1 * torch.randn((self.csa.ratio, D), generator=g, device="cuda")
        self.b_hca = 0.1 * torch.randn((self.hca.ratio, D), generator=g, device="cuda")
        self.bu = 0.1 * torch.randn((self.csa.ratio, Di), generator=g, device="cuda")
        self.d_csa = dsv4.layer_desc(self.csa, n // self.csa.ratio + 1)
        self.d_hca = dsv4.layer_desc(self.hca, n // self.hca.ratio + 1)
        self.c_csa = dsv4.Cache(self.d_csa)
        self.c_hca = dsv4.Cache(self.d_hca)
        self.side = torch.cuda.Stream()
        torch.cuda.synchronize()

    def input_bytes(self):
        return sum(t.numel() * t.element_size() for t in (self.x, self.z_csa, self.z_hca, self.u, self.zu))

    def step(self):
        d = self.dsv4
        main, side = torch.cuda.current_stream(), self.side
        side.wait_stream(main)
        self.c_csa.n_tokens.zero_()
        with torch.cuda.stream(side):
            self.c_hca.n_tokens.zero_()
        for t0 in range(0, self.n, self.chunk):
            t1 = t0 + self.chunk
            d.dsv4_compress_append(self.d_csa, self.c_csa, self.chunk, self.x[t0:t1], None, self.z_csa[t0:t1],
                                   self.b_csa, self.u[t0:t1], self.zu[t0:t1], self.bu, stream=main)
            d.dsv4_compress_append(self.d_hca, self.c_hca, self.chunk, self.x[t0:t1], None, self.z_hca[t0:t1],
                                   self.b_hca, stream=side)
        main.wait_stream(side)


def compress_bytes():
    """Algorithmic bytes of one pass of the compressor workload: the token
    stream read once (x shared by both compressors, each compressor's gate
    logits, the indexer-key stream and its gates), the caches' entries and keys
    written once."""
    csa, hca = W.COMPRESS_1M_CSA, W.COMPRESS_1M_HCA
    n = W.COMPRESS_1M_TOKENS
    read = n * (csa.dim * 2 * 3 + csa.idx_dim * 2 * 2)
    written = (n // csa.ratio) * (accounting.entry_bytes(csa) + accounting.idx_key_bytes(csa)) + \
        (n // hca.ratio) * accounting.entry_bytes(hca)
    return read, written


def _graph_time(fn, K, Wm, stream):
    """ms per call of fn() captured in one CUDA graph, K timed replays after Wm."""
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    upload_graphs([g], stream)
    for _ in range(Wm):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        with torch.cuda.stream(stream):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / K


def time_next_rows(dsv4, st, K, Wm, seed):
    """The decode-side rows beyond single-token decode, on the stack's first CSA
    and HCA layers (their caches as the stack step left them):
      multi_token  T = 4 queries per sequence after their tokens were appended
                   (speculative or chunked decode): causal top-k, CSA and HCA
                   attention with the window rows from a span of the last
                   T + W - 1 raw tokens; tokens/s = B * T / (time of one CSA and
                   one HCA layer's calls);
      window_only  the window-only layer (k = 0) at the CSA layer's shape;
      ratio1       selection over the raw tokens (ratio 1) at a 128K context:
                   index_topk then csa_decode, B = 4, the stack's dims."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    stream = torch.cuda.Stream()
    Lc, Lh = st.layers[0], st.layers[1]
    dc, cc, dh, ch = st.descs[0], st.caches[0], st.descs[1], st.caches[1]
    B, H, D, Hi, Di, k = Lc.batch, Lc.heads, Lc.dim, Lc.idx_heads, Lc.idx_dim, Lc.topk

    def bf16(shape):
        return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)

    out = {}
    T = 4
    q, qh = bf16((B, T, H, D)), bf16((B, T, Lh.heads, Lh.dim))
    qi = bf16((B, T, Hi, Di))
    w = torch.rand((B, T, Hi), generator=g, device="cuda")
    span_c, span_h = bf16((B, T + Lc.window - 1, D)), bf16((B, T + Lh.window - 1, Lh.dim))
    ws_c = dsv4.workspace_multi(dc, T, H, Hi, k)
    ws_h = dsv4.workspace_multi(dh, T, Lh.heads)
    topk = torch.zeros((B, T, k), dtype=torch.int32, device="cuda")
    o_c = torch.empty((B, T, H, D), device="cuda")
    l_c = torch.empty((B, T, H), device="cuda")
    o_h = torch.empty((B, T, Lh.heads, Lh.dim), device="cuda")
    l_h = torch.empty((B, T, Lh.heads), device="cuda")

    def multi():
        dsv4.dsv4_index_topk_multi(dc, cc, T, Hi, qi, w, k, topk, None, ws_c)
        dsv4.dsv4_csa_decode_multi(dc, cc, T, H, q, Lc.sm_scale, topk, k, span_c, None, o_c, l_c, ws_c)
        dsv4.dsv4_hca_decode_multi(dh, ch, T, Lh.heads, qh, Lh.sm_scale, span_h, None, o_h, l_h, ws_h)

    ms = _graph_time(multi, K, Wm, stream)
    out["multi_token"] = {"queries_per_sequence": T, "ms_per_step": round(ms, 4),
                          "tokens_per_s": round(B * T / (ms * 1e-3), 1),
                          "layers": "one CSA + one HCA layer of stack_1m (appends not included)"}
    del ws_c, ws_h

    ws = dsv4.workspace(dc, H, Hi, k)
    q1 = bf16((B, H, D))
    o1 = torch.empty((B, H, D), device="cuda")
    l1 = torch.empty((B, H), device="cuda")
    ms = _graph_time(lambda: dsv4.dsv4_csa_decode(dc, cc, H, q1, Lc.sm_scale, None, 0, o1, l1, ws), K, Wm, stream)
    out["window_only"] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
                          "layer": f"window {Lc.window}, {H} heads, {Lc.d_nope}+{Lc.d_rope} dims, B = {B}"}
    del ws

    # ratio 1 at a 128K context: a cache of raw tokens (entries and FP4 keys drawn directly)
    n = 1 << 17
    L1 = W.scaled(Lc, ratio=1, n_tokens=n, planted_frac=0.0)
    d1 = dsv4.layer_desc(L1, n + 64)
    c1 = dsv4.Cache(d1)
    for b in range(B):
        for r0 in range(0, n, 1 << 16):
            r1 = min(n, r0 + (1 << 16))
            y = torch.randn((r1 - r0, D), generator=g, device="cuda")
            dsv4.dsv4_quantize_kv_rows(y, r1 - r0, L1.d_nope, L1.d_rope, c1.k_nope[b, r0:r1], c1.k_scale[b, r0:r1],
                                       c1.k_rope[b, r0:r1])
            yi = torch.randn((r1 - r0, Di), generator=g, device="cuda")
            dsv4.dsv4_quantize_fp4_rows(yi, r1 - r0, Di, c1.idx_codes[b, r0:r1], c1.idx_scales[b, r0:r1])
        c1.win_k[b].copy_(bf16((L1.window, D)).view(torch.int16))
    c1.n_tokens.fill_(n)
    ws = dsv4.workspace(d1, H, Hi, k)
    qi1 = bf16((B, Hi, Di))
    w1 = torch.rand((B, Hi), generator=g, device="cuda")
    tk = torch.zeros((B, k), dtype=torch.int32, device="cuda")

    def ratio1():
        dsv4.dsv4_index_topk(d1, c1, Hi, qi1, w1, k, tk, None, ws)
        dsv4.dsv4_csa_decode(d1, c1, H, q1, L1.sm_scale, tk, k, o1, l1, ws)

    ms = _graph_time(ratio1, K, Wm, stream)
    out["ratio1"] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
                     "layer": f"ratio 1 over {n} raw tokens, top-{k}, window {L1.window}, B = {B}"}
    del c1, ws
    return out


def time_project(dsv4, K, Wm, seed, e2e=False):
    """Times K passes of the projection workload: the x, z, u and zu streams of
    a ratio-4 layer with 128-dim indexer keys (1280 output columns) projected
    from 2^20 hidden states of 4096 dims (~N(0,1) bf16, weights ~N(0, 1/4096))
    in 4096-token calls, RoPE on the rotated dims; one CUDA graph per pass.
    Tensor-core bound: FLOPs = 2 x tokens x 4096 x 1280."""
    L = W.COMPRESS_1M_CSA
    n, C, dm = W.COMPRESS_1M_TOKENS, W.COMPRESS_1M_CHUNK, W.PROJECT_D_MODEL
    D, Di = L.dim, L.idx_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    hidden = torch.empty((n, dm), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, n, 1 << 16):
        hidden[r0:r0 + (1 << 16)] = torch.randn((min(1 << 16, n - r0), dm), generator=g, device="cuda")
    weight = (torch.randn((2 * D + 2 * Di, dm), generator=g, device="cuda") / dm ** 0.5).to(torch.bfloat16)
    desc = dsv4.layer_desc(L, 64)
    cache = dsv4.Cache(desc)
    x = torch.empty((C, D), dtype=torch.bfloat16, device="cuda")
    z = torch.empty_like(x)
    u = torch.empty((C, Di), dtype=torch.bfloat16, device="cuda")
    zu = torch.empty_like(u)
    stream = torch.cuda.Stream()

    def one_pass():
        for c0 in range(0, n, C):
            dsv4.dsv4_project_streams(desc, cache, C, dm, hidden[c0:c0 + C], weight, 10000.0, x, z, u, zu,
                                      stream.cuda_stream)

    with torch.cuda.stream(stream):
        one_pass()
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        one_pass()
    for _ in range(Wm):
        with torch.cuda.stream(stream):
            gr.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        with torch.cuda.stream(stream):
            gr.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    flops = 2.0 * n * dm * (2 * D + 2 * Di)
    tf = flops / (ms * 1e-3) / 1e12
    peak, kind = tensor_peak()
    out = {"workload": "project_1m", "ms_per_pass": round(ms, 4), "tokens_per_s": round(n / (ms * 1e-3), 1),
           "TFLOP/s": round(tf, 1),
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(tf / peak, 4), "peak_kind": kind},
           "shape": f"{n} tokens x {dm} hidden -> {2 * D + 2 * Di} columns (x, z, u, zu), {C}-token calls",
           "launches_per_pass": n // C}
    if e2e:
        # end to end: every pass copies the hidden states from pinned host
        # memory and reads the last chunk's streams back
        host = torch.empty(hidden.shape, dtype=hidden.dtype, pin_memory=True)
        host.copy_(hidden.cpu())
        back = torch.empty((C, D), dtype=torch.bfloat16, pin_memory=True)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(K):
                hidden.copy_(host, non_blocking=True)
                gr.replay()
                back.copy_(x, non_blocking=True)
        stream.synchronize()
        ms_e2e = (time.perf_counter() - w0) * 1e3 / K
        out["e2e"] = {"unit": "TFLOP/s", "ms_per_pass": ms_e2e, "h2d_bytes_per_step": int(hidden.numel() * 2),
                      "d2h_bytes_per_step": int(back.numel() * 2)}
        del host
    del gr, hidden
    return out


def time_compress(dsv4, K, Wm, seed, peak, e2e=False):
    """Times K passes of the compressor workload (one CUDA graph per pass) after
    Wm warm-up passes; returns a dict of the figures (and the end-to-end pass
    with the token stream copied from pinned host memory when e2e)."""
    cp = Compress(dsv4, seed)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        cp.step()                                 # eager pass: kernel attributes set outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cp.step()
    probe = torch.cuda.CUDAGraph(keep_graph=True)      # captured only to count its kernel nodes
    with torch.cuda.graph(probe, stream=stream):
        cp.step()
    kernels = count_kernel_nodes(probe)
    del probe
    for _ in range(Wm):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        with torch.cuda.stream(stream):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    read, written = compress_bytes()
    gbs = (read + written) / (ms * 1e-3) / 1e9
    out = {"workload": "compress_1m", "ms_per_pass": round(ms, 4), "tokens_per_s": round(cp.n / (ms * 1e-3), 1),
           "GB/s": round(gbs, 1), "roofline_frac": round(gbs / peak, 4), "bytes_read": int(read),
           "bytes_written": int(written),
           "note": ("algorithmic bytes count the shared token stream x once; the two compressors are separate "
                    "calls, so x is read twice (the bytes the kernels move exceed the algorithmic bytes by "
                    f"{cp.x.numel() * 2 / 1e9:.2f} GB)"),
           "kernel_nodes_per_pass": kernels,
           "kernel_nodes_note": "library launches (two per append call) plus the two n_tokens resets"}
    if e2e:
        host = {n_: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for n_, t in (("x", cp.x), ("z_csa", cp.z_csa), ("z_hca", cp.z_hca), ("u", cp.u), ("zu", cp.zu))}
        for n_, t in host.items():
            t.copy_(getattr(cp, n_).cpu())
        res = torch.empty(2, dtype=torch.int64, pin_memory=True)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(K):
                for n_, t in host.items():
                    getattr(cp, n_).copy_(t, non_blocking=True)
                g.replay()
                res[0:1].copy_(cp.c_csa.n_tokens, non_blocking=True)
                res[1:2].copy_(cp.c_hca.n_tokens, non_blocking=True)
        stream.synchronize()
        ms_e2e = (time.perf_counter() - w0) * 1e3 / K
        out["e2e"] = {"value": round(cp.n / (ms_e2e * 1e-3), 1), "unit": "tokens/s", "ms_per_pass": ms_e2e,
                      "h2d_bytes_per_step": int(cp.input_bytes()), "d2h_bytes_per_step": 16}
    del g, cp
    torch.cuda.synchronize()
    return out


def workload_config(name, layers, world, step_bytes):
    kinds = [L.kind for L in layers]
    c = {"workload": name, "layers": len(layers) if len(layers) > 1 else kinds[0],
         "batch_per_gpu": layers[0].batch, "context": layers[0].n_tokens, "heads": layers[0].heads,
         "kv_dim": f"{layers[0].d_nope} fp8 + {layers[0].d_rope} bf16"}
    if len(layers) > 1:
        c["order"] = "CSA even, HCA odd"
    for L in layers:
        if L.kind == "csa" and "csa" not in c:
            c["csa"] = (f"ratio {L.ratio}, {L.n_comp} entries, indexer {L.idx_heads}x{L.idx_dim} fp4, "
                        f"top-{L.topk}, window {L.window}")
        if L.kind == "hca" and "hca" not in c:
            c["hca"] = f"ratio {L.ratio}, dense over {L.n_comp} entries, window {L.window}"
    c["l2"] = (f"inputs {step_bytes / 1e6:.1f} MB per step > 126 MB L2 (no flush)" if step_bytes > 126e6 else
               f"inputs {step_bytes / 1e6:.1f} MB per step < 126 MB L2: steps rotate over "
               f"distinct input slots but the caches stay L2-resident (upper bound)")
    c["parallelism"] = f"replicas x{world}"
    return c


def count_kernel_nodes(graph):
    """Kernel nodes in a captured graph (None when the graph handle is not reachable)."""
    try:
        from cuda.bindings import runtime as rt
        h = graph.raw_cuda_graph()
        err, _, n = rt.cudaGraphGetNodes(h, 0)
        err, nodes, n = rt.cudaGraphGetNodes(h, n)
        kernels = 0
        for node in nodes:
            e, t = rt.cudaGraphNodeGetType(node)
            if t == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                kernels += 1
        return kernels
    except Exception:
        return None


def traffic_for(call):
    """DRAM bytes per launch from a committed ncu capture, when the kernel source
    has not changed since (profiles/traffic.json records the source hash)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(call)
        if not rec:
            return None
        for src, sha in rec["sources"].items():
            h = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
            if h != sha:
                return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


def max_over_ranks(x, world, device):
    """The largest x over the ranks (the slowest rank's time); x itself on one rank."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, batch, ms_per_step):
    """Whole-job throughput: every rank decodes its own `batch` sequences (weak
    scaling), one token each per step, in the slowest rank's step time."""
    return world * batch * 1000.0 / ms_per_step


def run_ours(args, rank, world):
    from compressed_sparse_kv_05_b300 import dsv4
    layers = WORKLOADS[args.workload]
    B = layers[0].batch
    K, Wm = args.steps, args.warmup
    total = K + Wm
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    # input slots: [0, total) timed run, [total, total + K) per-call event run and
    # end-to-end run, then one eager warm-up step and one probe capture
    # appends: eager warm-up, W + K timed, K per-call, K end-to-end steps, and
    # W + K steps of each layer timed on its own
    st = Stack(dsv4, layers, total + K + 2, seed=1234 + rank, extra_tokens=2 * total + 2 * K + 4)
    stream = torch.cuda.Stream()
    # eager warm-up of every call (kernel attributes are set outside capture)
    with torch.cuda.stream(stream):
        st.step(total + K)
    stream.synchronize()
    # timed graphs hold only the library's launches, so consecutive kernels keep
    # their programmatic (overlapping) launch edges; a second set with an event
    # pair around every call gives the per-call durations
    graphs, ev_graphs, events = [], [], []
    for s in range(total):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            st.step(s)
        graphs.append(g)
    for i in range(K):
        g = torch.cuda.CUDAGraph()
        ev = {}
        with torch.cuda.graph(g, stream=stream):
            st.step(total + i, ev)
        ev_graphs.append(g)
        events.append(ev)
    probe = torch.cuda.CUDAGraph(keep_graph=True)       # captured only to count its kernel nodes
    with torch.cuda.graph(probe, stream=stream):
        st.step(total + K + 1)
    kernels_per_step = count_kernel_nodes(probe)
    uploaded = upload_graphs(graphs + ev_graphs, stream)
    for s in range(Wm):
        graphs[s].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(Wm, total):
        with torch.cuda.stream(stream):
            graphs[s].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), world, "cuda")
    ms_step = ms / K
    value = job_tokens_per_s(world, B, ms_step)

    # per-call durations: K more steps through the graphs with events
    for g in ev_graphs:
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    per_call = {}
    for ev in events:
        for call, pairs in ev.items():
            per_call.setdefault(call, []).extend(a.elapsed_time(b) for a, b in pairs)
    call_layer = {"append": layers[0]}
    for L in layers:
        call_layer.setdefault("index_topk" if L.kind == "csa" else "hca_decode", L)
        if L.kind == "csa":
            call_layer.setdefault("csa_decode", L)
    share = {c: sum(v) for c, v in per_call.items()}
    dominant = max(share, key=share.get)
    mean_ms = statistics.mean(per_call[dominant])
    alg = accounting.call_bytes(call_layer[dominant], dominant)
    peak, peak_kind = hbm_peak()
    achieved = alg / (mean_ms * 1e-3) / 1e9
    calls = {c: {"mean_us": round(statistics.mean(v) * 1e3, 2), "launches": len(v),
                 "GB/s": round(accounting.call_bytes(call_layer[c], c) / (statistics.mean(v) * 1e-3) / 1e9, 1)}
             for c, v in per_call.items()}
    step_bytes = sum(accounting.decode_step_bytes(L) + accounting.call_bytes(L, "append") for L in layers)

    # end to end: per step, H2D of that step's inputs from pinned host memory,
    # the step, and a D2H read of every layer's output; the copies run on their
    # own streams, so step i's read-back and step i + 1's inputs overlap the
    # steps around them (each step waits for its inputs, each read-back for its step)
    in_host = torch.empty((K, st.in_bytes), dtype=torch.uint8, pin_memory=True)
    in_host.copy_(st.inbuf[Wm:total].cpu())
    out_host = torch.empty((K,) + tuple(st.out.shape[1:]), dtype=torch.float32, pin_memory=True)
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    inputs_in = [torch.cuda.Event() for _ in range(K)]
    step_done = [torch.cuda.Event() for _ in range(K)]
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    h2d.wait_event(e0)
    for i in range(K):
        with torch.cuda.stream(h2d):
            st.inbuf[Wm + i].copy_(in_host[i], non_blocking=True)
            inputs_in[i].record(h2d)
    for i in range(K):
        s = Wm + i
        stream.wait_event(inputs_in[i])
        with torch.cuda.stream(stream):
            graphs[s].replay()
            step_done[i].record(stream)
        d2h.wait_event(step_done[i])
        with torch.cuda.stream(d2h):
            out_host[i].copy_(st.out[s], non_blocking=True)
    reads_done = torch.cuda.Event()
    reads_done.record(d2h)
    stream.wait_event(reads_done)
    e1.record(stream)
    stream.synchronize()
    wall = (time.perf_counter() - w0) * 1e3
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), wall), world, "cuda")
    e2e = {"value": round(job_tokens_per_s(world, B, e2e_ms / K), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": int(st.in_bytes), "d2h_bytes_per_step": int(st.out[0].numel() * 4),
           "copies": "own streams, overlapping the neighbouring steps"}

    # per-layer decode: the first CSA and the first HCA layer of the stack, each
    # replayed on its own (append + its attention calls), W + K graphs
    per_layer = {}
    if len(layers) > 1:
        for li in (0, 1):
            L = layers[li]
            gs = []
            for s in range(total):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st.step(s, only=li)
                gs.append(g)
            upload_graphs(gs, stream)
            for s in range(Wm):
                with torch.cuda.stream(stream):
                    gs[s].replay()
            torch.cuda.synchronize()
            e0.record(stream)
            for s in range(Wm, total):
                with torch.cuda.stream(stream):
                    gs[s].replay()
            e1.record(stream)
            torch.cuda.synchronize()
            lms = max_over_ranks(e0.elapsed_time(e1), world, "cuda") / K
            lbytes = accounting.decode_step_bytes(L) + accounting.call_bytes(L, "append")
            per_layer[f"{args.workload}_{L.kind}"] = {
                "layer": li, "kind": L.kind, "tokens_per_s": round(job_tokens_per_s(world, L.batch, lms), 1),
                "ms_per_step": round(lms, 4), "bytes_per_step": int(lbytes),
                "GB/s": round(lbytes / (lms * 1e-3) / 1e9, 1),
                "roofline_frac": round(lbytes / (lms * 1e-3) / 1e9 / peak, 4)}
            del gs

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE, "data": "synthetic",
        "config": workload_config(args.workload, layers, world, step_bytes),
        "step_bytes": int(step_bytes),
        "step_GBps": round(step_bytes / (ms_step * 1e-3) / 1e9, 1),
        "step_roofline_frac": round(step_bytes / (ms_step * 1e-3) / 1e9 / peak, 4),
        "calls": calls,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic_for(dominant), "algorithmic_bytes_per_launch": int(alg)},
        "e2e": e2e,
        "gpu_launches": (kernels_per_step * K) if kernels_per_step is not None else None,
        "clocks": clk,
    }
    line["config"]["graphs_uploaded_before_timing"] = uploaded
    if per_layer:
        line["layers"] = per_layer
    if args.workload == "stack_1m":
        line["next_rows"] = time_next_rows(dsv4, st, min(K, 10), 3, 2468 + rank)
    if args.workload == "stack_1m" and not args.no_compress:
        del graphs, ev_graphs, probe
        line["compress_1m"] = time_compress(dsv4, min(K, 10), 3, 4321 + rank, peak)
        line["project_1m"] = time_project(dsv4, min(K, 5), 2, 8765 + rank)
    return line


def project_config(world):
    L = W.COMPRESS_1M_CSA
    return {"workload": "project_1m", "tokens": W.COMPRESS_1M_TOKENS, "chunk": W.COMPRESS_1M_CHUNK,
            "d_model": W.PROJECT_D_MODEL, "columns": 2 * L.dim + 2 * L.idx_dim,
            "streams": "x 448+64 (RoPE on the last 64), z 512, u 128 (RoPE on the last 64), zu 128",
            "l2": "hidden states 8.6 GB per pass > 126 MB L2 (no flush)", "parallelism": f"replicas x{world}"}


def run_project(args, rank, world):
    """The projection workload as the headline: TFLOP/s on the tensor cores."""
    from compressed_sparse_kv_05_b300 import dsv4
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    r = time_project(dsv4, args.steps, args.warmup, 8765 + rank, e2e=True)
    clk = clocks.stop()
    ms = max_over_ranks(r["ms_per_pass"], world, "cuda")
    flops = project_flops(W.COMPRESS_1M_TOKENS)
    tf = world * flops / (ms * 1e-3) / 1e12
    e2e = r.pop("e2e")
    e2e_ms = max_over_ranks(e2e.pop("ms_per_pass"), world, "cuda")
    e2e["value"] = round(world * flops / (e2e_ms * 1e-3) / 1e12, 1)
    roof = dict(r["roofline"])
    roof.update({"achieved": round(tf / world, 1), "frac": round(tf / world / roof["peak"], 4), "kernel": "project",
                 "traffic": None, "algorithmic_flops_per_launch": project_flops(W.COMPRESS_1M_CHUNK)})
    return {"metric": PROJECT_METRIC, "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 operands, fp32 accumulate, bf16 out",
            "data": "synthetic", "config": project_config(world), "roofline": roof, "detail": r, "e2e": e2e,
            "gpu_launches": r["launches_per_pass"] * args.steps, "clocks": clk}


def run_compress(args, rank, world):
    """The compressor workload as the headline: cache GB/s read and written."""
    from compressed_sparse_kv_05_b300 import dsv4
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    peak, peak_kind = hbm_peak()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    r = time_compress(dsv4, args.steps, args.warmup, 4321 + rank, peak, e2e=True)
    clk = clocks.stop()
    ms = max_over_ranks(r["ms_per_pass"], world, "cuda")
    read, written = compress_bytes()
    gbs = world * (read + written) / (ms * 1e-3) / 1e9
    e2e = r.pop("e2e")
    e2e_ms = max_over_ranks(e2e.pop("ms_per_pass"), world, "cuda")
    e2e["value"] = round(world * (read + written) / (e2e_ms * 1e-3) / 1e9, 1)
    e2e["unit"] = "GB/s"
    return {"metric": "compressor cache GB/s read + written (2^20 tokens of 512 dims in 4096-token chunks into "
                      "a ratio-4 CSA and a ratio-128 HCA cache)",
            "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE, "data": "synthetic",
            "config": {"workload": "compress_1m", "tokens": W.COMPRESS_1M_TOKENS, "chunk": W.COMPRESS_1M_CHUNK,
                       "kv_dim": "448 fp8 + 64 bf16", "csa": "ratio 4, FP4 indexer keys 128 dims",
                       "hca": "ratio 128", "l2": f"inputs {(read / 1e9):.2f} GB per pass > 126 MB L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "compress_append", "achieved": round(gbs / world, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / world / peak, 4), "peak_kind": peak_kind,
                         "traffic": None, "algorithmic_bytes_per_launch": int(read + written)},
            "detail": r, "e2e": e2e,
            "gpu_launches": (r["kernel_nodes_per_pass"] - 2) * args.steps if r["kernel_nodes_per_pass"] else None,
            "clocks": clk}


# ----------------------------------------------------------------------------- the oracle on the host


def oracle_sample_setup(layers):
    """One sequence of one layer of each kind in the workload (full context),
    caches quantised by the oracle from the seeded rows."""
    import oracle as O
    tag = "bench"
    out = []
    seen = set()
    for li, L in enumerate(layers):
        if L.kind in seen:
            continue
        seen.add(L.kind)
        rows = synth.direct_rows(tag, li, L, 0)
        p = {}
        p["k_nope"], p["k_scale"], p["k_rope"] = O.quantize_kv_rows(rows["kv"], L.d_nope)
        if L.kind == "csa":
            p["idx_codes"], p["idx_scales"] = O.quantize_fp4_rows(rows["idx"])
        win = synth.window_tokens(tag, li, L, 0)["k"]
        ring = np.zeros((L.window, L.dim), np.uint16)
        pos = np.arange(L.n_tokens - L.window, L.n_tokens)
        ring[pos % L.window] = win
        p["ring"] = ring
        p["dec"] = synth.decode_inputs(tag, li, L)
        out.append((L, p))
    return out


def sample_scale(layers):
    """Sequences-times-layers of one step per sample step (one sequence of each kind)."""
    n_csa = sum(L.kind == "csa" for L in layers)
    n_hca = len(layers) - n_csa
    return max(n_csa, n_hca)


def oracle_sample_step(sample):
    import oracle as O
    for L, p in sample:
        dec = p["dec"]
        if L.kind == "csa":
            sc = O.index_scores(p["idx_codes"], p["idx_scales"], dec["q_idx"][0], dec["w"][0])
            sel = O.topk_blocks(sc, L.topk)
            O.csa_attend(dec["q"][0], np.float32(L.sm_scale), sel, L.n_tokens, L.ratio, L.window,
                         p["k_nope"], p["k_scale"], p["k_rope"], p["ring"])
        else:
            O.hca_attend(dec["q"][0], np.float32(L.sm_scale), L.n_tokens, L.ratio, L.window,
                         p["k_nope"], p["k_scale"], p["k_rope"], p["ring"])


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def sample_desc(name, layers):
    if name == "project_1m":
        return (f"{PROJECT_SAMPLE_TOKENS} tokens of the projection (float64 matmul and RoPE) per sample step; "
                f"TFLOP/s = the sample's FLOPs / sample-step time")
    if name == "compress_1m":
        return (f"the first {COMPRESS_SAMPLE_TOKENS} tokens of the compressor stream pooled and quantised into both "
                f"caches per sample step; GB/s = algorithmic bytes of those tokens / sample-step time")
    kinds = sorted({L.kind.upper() for L in layers})
    return (f"one sequence x (one {' + one '.join(kinds)} layer) of {name} at the full context per sample step; "
            f"tokens/s = 1 / (sample-step time x {sample_scale(layers)})")


COMPRESS_SAMPLE_TOKENS = 8192


def oracle_compress_setup():
    tag = "bench"
    n = COMPRESS_SAMPLE_TOKENS
    csa, hca = W.COMPRESS_1M_CSA, W.COMPRESS_1M_HCA
    t = synth.token_stream(tag, 0, csa, 1, 0, n)
    zh = synth.token_stream(tag, 1, hca, 1, 0, n)["z"]
    return {"k": t["k"][0], "z": t["z"][0], "u": t["u"][0], "zu": t["zu"][0], "zh": zh[0],
            "b": synth.position_bias(tag, 0, csa, "b"), "bu": synth.position_bias(tag, 0, csa, "bu"),
            "bh": synth.position_bias(tag, 1, hca, "b")}


def oracle_compress_step(p):
    import oracle as O
    csa, hca = W.COMPRESS_1M_CSA, W.COMPRESS_1M_HCA
    O.build_cache(p["k"], p["z"], p["b"], csa.ratio, csa.d_nope, csa.window, None, p["u"], p["zu"], p["bu"])
    O.build_cache(p["k"], p["zh"], p["bh"], hca.ratio, hca.d_nope, hca.window)


PROJECT_SAMPLE_TOKENS = 256


def oracle_project_setup():
    L = W.COMPRESS_1M_CSA
    D, Di, dm = L.dim, L.idx_dim, W.PROJECT_D_MODEL
    h = synth.bf16_bits(synth.normal(("bench", "project", "h"), (PROJECT_SAMPLE_TOKENS, dm)))
    w = synth.bf16_bits(synth.normal(("bench", "project", "w"), (2 * D + 2 * Di, dm)) / np.sqrt(dm))
    return {"h": h, "w": w}


def oracle_project_step(p):
    import oracle as O
    L = W.COMPRESS_1M_CSA
    O.project_streams(p["h"], p["w"], L.d_nope, L.d_rope, L.idx_dim, np.arange(PROJECT_SAMPLE_TOKENS), 10000.0)


def project_flops(tokens):
    L = W.COMPRESS_1M_CSA
    return 2.0 * tokens * W.PROJECT_D_MODEL * (2 * L.dim + 2 * L.idx_dim)


def oracle_sample(name, layers):
    """(sample inputs, step function) of the oracle for a workload."""
    if name == "compress_1m":
        return oracle_compress_setup(), oracle_compress_step
    if name == "project_1m":
        return oracle_project_setup(), oracle_project_step
    return oracle_sample_setup(layers), oracle_sample_step


BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                    "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def oracle_child(name, steps, warmup):
    """Runs in a child process whose BLAS pool was sized by the environment
    before numpy loaded: seconds per sample step of the oracle."""
    sample, fn = oracle_sample(name, WORKLOADS[name])
    for _ in range(warmup):
        fn(sample)
    t = time.perf_counter()
    for _ in range(steps):
        fn(sample)
    return {"dt": (time.perf_counter() - t) / steps}


def time_oracle(name, steps, warmup, threads):
    """Seconds per sample step of the oracle with its BLAS threads pinned to
    `threads`: timed in a child process started with every BLAS thread-count
    variable set, so the pin holds whichever BLAS numpy carries."""
    env = dict(os.environ)
    for v in BLAS_THREAD_VARS:
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import json, bench; "
            f"print('ORACLE ' + json.dumps(bench.oracle_child({name!r}, {int(steps)}, {int(warmup)})))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    for line in r.stdout.splitlines():
        if line.startswith("ORACLE "):
            return json.loads(line[7:])["dt"]
    raise RuntimeError("oracle timing failed:\n" + r.stdout[-2000:] + r.stderr[-2000:])


def oracle_rate(name, layers, dt):
    """(value, unit) of the oracle from its sample-step time."""
    if name == "project_1m":
        return project_flops(PROJECT_SAMPLE_TOKENS) / dt / 1e12, "TFLOP/s"
    if name == "compress_1m":
        read, written = compress_bytes()
        frac = COMPRESS_SAMPLE_TOKENS / W.COMPRESS_1M_TOKENS
        return (read + written) * frac / dt / 1e9, "GB/s"
    return 1.0 / (sample_scale(layers) * dt), "tokens/s"


def cpu_baseline(name, layers, steps=2):
    """The oracle as it stands (numpy; BLAS threads pinned explicitly) on a
    bounded sample of the workload: with one BLAS thread per host core and with
    one thread."""
    n = os.cpu_count() or 1
    dt_all = time_oracle(name, steps, 1, n)
    dt_one = time_oracle(name, steps, 1, 1)
    v_all, unit = oracle_rate(name, layers, dt_all)
    v_one, _ = oracle_rate(name, layers, dt_one)
    return {"value": round(v_all, 4), "unit": unit, "cores": n, "kind": "oracle", "sample": sample_desc(name, layers),
            "s_per_sample_step": round(dt_all, 3), "cpu_model": cpu_model(),
            "one_thread": {"value": round(v_one, 4), "cores": 1, "s_per_sample_step": round(dt_one, 3)}}


def run_reference(args):
    """The reference arm: the float64 oracle, as it stands, on the host cores,
    on a bounded sample of the same workload (each step one sample step)."""
    layers = WORKLOADS[args.workload]
    n = os.cpu_count() or 1
    dt = time_oracle(args.workload, args.steps, args.warmup, n)
    value, unit = oracle_rate(args.workload, layers, dt)
    desc = sample_desc(args.workload, layers)
    cb = {"value": round(value, 4), "unit": unit, "cores": n, "kind": "oracle", "sample": desc,
          "cpu_model": cpu_model()}
    if args.workload == "compress_1m":
        metric = ("compressor cache GB/s read + written (2^20 tokens of 512 dims in 4096-token chunks into "
                  "a ratio-4 CSA and a ratio-128 HCA cache)")
        config = {"workload": "compress_1m", "tokens": W.COMPRESS_1M_TOKENS, "chunk": W.COMPRESS_1M_CHUNK}
        projected = None
    elif args.workload == "project_1m":
        metric = PROJECT_METRIC
        config = project_config(1)
        projected = None
    else:
        metric = METRIC
        step_bytes = sum(accounting.decode_step_bytes(L) + accounting.call_bytes(L, "append") for L in layers)
        config = workload_config(args.workload, layers, 1, step_bytes)
        projected = round(dt * sample_scale(layers) * layers[0].batch * 1e3, 2)
    return {"impl": "reference", "metric": metric, "value": round(value, 4), "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
            "sample_step": "each timed step is one sample step of the oracle (see cpu_baseline.sample)",
            "projected_ms_per_full_step": projected,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config, "cpu_baseline": cb,
            "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    if args.workload == "compress_1m":
        line = run_compress(args, rank, world)
    elif args.workload == "project_1m":
        line = run_project(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, WORKLOADS[args.workload])
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
