#!/usr/bin/env python3
"""Benchmark of the DSA decode hot path on one GB300 (or N replicas).

Headline step (the 128K-context MTP decode workload): 32 requests x 131072
cached tokens, next_n = 2 (64 query rows), 64 index heads x 128 FP8 keys in
64-token pages behind a shuffled block table, then
  1. dsa_indexer_logits   (Eq. (1) over all 8.4 M (row, key) pairs)
  2. dsa_topk             (exact top-2048 per row; cutoff path)
  3. dsa_sparse_mla_decode (128 heads x 576-d bf16 latents of the selected tokens)
The candidate-block path (64 x 196608 ctx, 512 candidate blocks, MXFP4 keys,
one expansion + 4 consumer layers of candidate logits + top-k) is timed in the
same run and reported under "candidate_path".

value = indexer keys scored (row, key pairs) per second of the whole step.
All inputs are seeded synthetic data generated on the device; the key cache
(553.6 MB) and the latent cache (4.8 GB) are larger than L2, so no flush is
needed between steps.

The tiny decode (1 x 8192 tokens) and the batched varlen full path (64
requests, L ~ U[16K, 64K], indexer + top-2048 + sparse MLA) are timed in the
same run ("configs"), and the chunked prefill's launches are broken down with
their tensor-pipe fractions.  The fp64 CPU oracle is timed on the host cores on
every workload ("cpu_baseline").

--impl reference times the fp64 CPU oracle (the reference arm) on the
headline workload's 64 rows per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# DRAM bytes (read + write) of one dsa_indexer_logits launch per cached token,
# measured by ncu on this workload at 16 requests x 131072 tokens, next_n = 2
# (`bench.py --requests 16 --no-candidate --no-layers --no-prefill --no-configs
# --no-cpu-baseline --steps 1 --warmup 3`, fourth indexer launch, the current
# kernel): 277.30 MB read + 6.76 MB written (the rest of the logits leave L2
# after the kernel).
INDEXER_DRAM_BYTES_PER_TOKEN = (277.30e6 + 6.76e6) / (16 * 131072)
METRIC = "indexer keys scored/s + HBM GB/s at 128K decode; top-k rows/s; sparse-attn tok/s"
WORKLOAD = ("128K MTP decode: 32 requests x 131072 ctx, next_n=2 (64 rows), FP8 indexer "
            "64x128 over 64-token shuffled pages, exact top-2048, sparse MLA 128 heads x "
            "576-d bf16 latents")
TOPK = 2048


def peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source): the copy bandwidth and the
    cuBLAS bf16 rate measured on this machine; each kernel here is timed alone
    (one launch between two events), so its tensor peak is the burst figure.
    FP8 kind::f8f6f4 contractions take twice the bf16 figure (the nominal
    dense ratio, 4.5 / 2.25 PFLOP/s)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Targets the method's statement sets for one GB300: the 128K decode indexer at
# >= 70 % of the HBM roofline, the top-k and the sparse MLA >= 50 % of theirs.
TARGETS = {"indexer_hbm_frac": 0.70, "topk_frac": 0.50, "sparse_mla_frac": 0.50}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        try:
            rows = [l.strip().split(", ") for l in open(self.path) if l.strip()]
        except Exception:
            return out
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except Exception:
                continue
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                   "reasons": sorted(reasons), "samples": len(sm)}
        return out


# ------------------------------------------------------------------ our arm --

def build_decode(device, seed=0, requests=32):
    import torch
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case = W.make_indexer_case([131072] * requests, next_n=2, seed=seed, device=device)
    R = case.rows
    L = W.row_lengths(case.layout.ctx_len, 2).to(torch.int32)
    ld = 131072
    mla = W.make_mla_case(R, case.layout.num_pages, seed=seed, device=device)
    st = dict(case=case, R=R, L=L, ld=ld, mla=mla)
    st["logits"] = torch.empty((R, ld), device=device)
    st["idx"] = torch.empty((R, TOPK), dtype=torch.int32, device=device)
    st["out"] = torch.empty((R, W.MLA_HEADS, W.MLA_DV), dtype=torch.bfloat16, device=device)
    st["lse"] = torch.empty((R, W.MLA_HEADS), device=device)
    from deepseek_sparse_attention_02_gb300 import dsa
    wsb = dsa.dsa_sparse_mla_workspace_size(R, TOPK)
    st["ws"] = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)
    st["wsb"] = wsb
    return st


def decode_kernels(st):
    """The three launches of one decode step, as callables."""
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case, R, ld = st["case"], st["R"], st["ld"]
    c = case.cache
    lay = case.layout

    def indexer():
        dsa.dsa_indexer_logits(case.q, case.q_scale, case.w, c, W.FP8_PAGE_BYTES,
                               c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES, lay.num_pages,
                               lay.block_table, lay.ctx_len, len(lay.ctx_len), 2, st["logits"], ld)

    def topk():
        dsa.dsa_topk(st["logits"], ld, st["L"], R, TOPK, st["idx"])

    def mla():
        m = st["mla"]
        dsa.dsa_sparse_mla_decode(m.q, m.kv, 64 * 576 * 2, lay.num_pages, lay.block_table,
                                  len(lay.ctx_len), 2, st["idx"], TOPK, m.scale, st["out"],
                                  st["lse"], st["ws"], st["wsb"])

    return [("indexer", indexer), ("topk", topk), ("sparse_mla", mla)]


def build_dense_config(device, cfg):
    """The tiny decode (cfg 0: 1 request x 8192 tokens, contiguous cache,
    indexer + top-2048) or the batched varlen full path (cfg 1: 64 requests,
    L ~ U[16K, 64K], shuffled pages, indexer + top-2048 + sparse MLA)."""
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    spec = W.config_ctx(cfg)
    case = W.make_indexer_case(spec["ctx"], next_n=spec["next_n"], seed=cfg, device=device,
                               shuffle=spec["shuffle"])
    R = case.rows
    L = W.row_lengths(case.layout.ctx_len, spec["next_n"]).to(torch.int32)
    ld = (int(L.max()) + 3) // 4 * 4
    st = dict(cfg=cfg, case=case, R=R, L=L, ld=ld, next_n=spec["next_n"],
              logits=torch.empty((R, ld), device=device),
              idx=torch.empty((R, TOPK), dtype=torch.int32, device=device), mla=None)
    if cfg == 1:
        st["mla"] = W.make_mla_case(R, case.layout.num_pages, seed=cfg, device=device)
        st["out"] = torch.empty((R, W.MLA_HEADS, W.MLA_DV), dtype=torch.bfloat16, device=device)
        st["lse"] = torch.empty((R, W.MLA_HEADS), device=device)
        st["wsb"] = dsa.dsa_sparse_mla_workspace_size(R, TOPK)
        st["ws"] = torch.empty(max(st["wsb"], 16), dtype=torch.uint8, device=device)
    return st


def dense_config_kernels(st):
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case, R, ld, nn = st["case"], st["R"], st["ld"], st["next_n"]
    c, lay = case.cache, case.layout

    def indexer():
        dsa.dsa_indexer_logits(case.q, case.q_scale, case.w, c, W.FP8_PAGE_BYTES,
                               c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES, lay.num_pages,
                               lay.block_table, lay.ctx_len, len(lay.ctx_len), nn, st["logits"], ld)

    def topk():
        dsa.dsa_topk(st["logits"], ld, st["L"], R, TOPK, st["idx"])
    ks = [("indexer", indexer), ("topk", topk)]
    if st["mla"] is not None:
        def mla():
            m = st["mla"]
            dsa.dsa_sparse_mla_decode(m.q, m.kv, 64 * 576 * 2, lay.num_pages, lay.block_table,
                                      len(lay.ctx_len), nn, st["idx"], TOPK, m.scale, st["out"],
                                      st["lse"], st["ws"], st["wsb"])
        ks.append(("sparse_mla", mla))
    return ks


def dense_metrics(st, total_ms, per, steps, hbm, bf16_tf):
    """Throughput and per-kernel roofline fractions of a dense decode leg."""
    R = st["R"]
    keys = float(st["L"].sum().item())
    tokens = float(st["case"].layout.ctx_len.sum().item())
    ms = total_ms / steps
    idx_bytes = tokens * 132 + keys * 4
    out = {"ms_per_step": round(ms, 4),
           "breakdown_ms": {k: round(v, 4) for k, v in per.items()},
           "keys_per_s": keys / (ms * 1e-3),
           "indexer_keys_per_s": keys / (per["indexer"] * 1e-3),
           "indexer_hbm_frac": round(idx_bytes / (per["indexer"] * 1e-3) / 1e9 / hbm, 4),
           "topk_rows_per_s": R / (per["topk"] * 1e-3),
           "topk_frac": round(kernel_roofline(keys * 4 + R * TOPK * 4, 0.0, per["topk"], hbm,
                                              bf16_tf)["frac"], 4)}
    if "sparse_mla" in per:
        mla_bytes = R * TOPK * 1152 + R * 128 * 576 * 2 + R * 128 * 512 * 2
        mla_flops = R * 2 * 128 * TOPK * (576 + 512)
        out["attended_tok_per_s"] = R * TOPK / (per["sparse_mla"] * 1e-3)
        out["sparse_mla_frac"] = round(kernel_roofline(mla_bytes, mla_flops, per["sparse_mla"],
                                                       hbm, bf16_tf)["frac"], 4)
    return out


def build_candidate(device, seed=3, requests=64):
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    ctx = [196608] * requests
    layers = [W.make_indexer_case(ctx, next_n=1, seed=seed + i, device=device, fmt="mxfp4")
              for i in range(4)]
    cand = W.make_candidates(ctx, 1, 64, 512, seed=seed, device=device)
    R, nb = cand.shape
    nbytes = dsa.dsa_candidate_schedule_size(R)
    st = dict(layers=layers, cand=cand, R=R, nb=nb, sched_bytes=nbytes,
              si=torch.empty_like(cand), end=torch.empty(R, dtype=torch.int32, device=device),
              sched=torch.zeros(nbytes // 4, dtype=torch.int32, device=device),
              logits=torch.empty((R, nb * 64), device=device),
              logits16=torch.empty((R, nb * 64), dtype=torch.bfloat16, device=device),
              idx=torch.empty((4, R, TOPK), dtype=torch.int32, device=device))
    return st


def candidate_kernels(st, bf16=False):
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    R, nb = st["R"], st["nb"]
    ld = nb * 64
    lay0 = st["layers"][0].layout
    ks = [("expand", lambda: dsa.dsa_candidate_expand(st["cand"], R, nb, 64, lay0.ctx_len, 1,
                                                      st["si"], st["end"], st["sched"],
                                                      st["sched_bytes"]))]
    cl = dsa.dsa_candidate_logits_bf16 if bf16 else dsa.dsa_candidate_logits
    tk = dsa.dsa_topk_bf16 if bf16 else dsa.dsa_topk
    buf = st["logits16"] if bf16 else st["logits"]
    for i, case in enumerate(st["layers"]):
        def logits(case=case):
            c = case.cache
            cl(case.q, case.q_scale, case.w, c, W.FP4_PAGE_BYTES, c.data_ptr() + W.FP4_KEY_BYTES,
               W.FP4_PAGE_BYTES, case.layout.num_pages, case.layout.block_table, R, 1, st["si"],
               nb, 64, st["end"], st["sched"], st["sched_bytes"], buf, ld)

        def topk(i=i):
            tk(buf, ld, st["end"], R, TOPK, st["idx"][i], col_blocks=st["si"], nb=nb,
               block_size=64)
        ks.append((f"cand_logits_{i}", logits))
        ks.append((f"cand_topk_{i}", topk))
    return ks


LAYER_SCHEDULES = [(1, False), (1, True), (2, False), (2, True), (4, False), (4, True)]


def build_layers(st, n_layers=8):
    """A decode step over n_layers DSA layers for the IndexCache / Multi-layer
    Indexer schedules: every layer has its own indexer and attention queries;
    all read the headline workload's key and latent caches (each far larger
    than L2, so sharing them changes no traffic)."""
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case, R, dev = st["case"], st["R"], st["L"].device
    c = case.cache
    layers = []
    for l in range(n_layers):
        qc, qs, w = W.make_index_queries(R, seed=100 + l, device=dev)
        layers.append(dict(q_fp8=qc, q_scale=qs, weights=w, k_cache=c,
                           k_scale=c.data_ptr() + W.FP8_KEY_BYTES,
                           q=W.make_mla_queries(R, seed=200 + l, device=dev), kv_cache=st["mla"].kv,
                           out=torch.empty((R, W.MLA_HEADS, W.MLA_DV), dtype=torch.bfloat16,
                                           device=dev),
                           lse=torch.empty((R, W.MLA_HEADS), device=dev)))
    wsb = dsa.dsa_decode_layers_workspace_size(R, st["ld"], TOPK)
    return dict(layers=layers, wsb=wsb, ws=torch.zeros(wsb, dtype=torch.uint8, device=dev),
                side=torch.cuda.Stream(device=dev))


def time_layers(st, lst, steps, warmup, stream):
    """ms per multi-layer step for each (retention 1/r, MLI) schedule."""
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    lay = st["case"].layout
    n = len(lst["layers"])
    res, launches = {}, 0
    for r, mli in LAYER_SCHEDULES:
        keep = [l % r == 0 for l in range(n)]

        def step():
            dsa.dsa_decode_layers(lst["layers"], keep, mli, 8448, 8448, 64 * 576 * 2,
                                  lay.num_pages, lay.block_table, lay.ctx_len, st["L"],
                                  len(lay.ctx_len), 2, TOPK, st["mla"].scale, st["ld"],
                                  lst["ws"], lst["wsb"], stream=stream, side_stream=lst["side"])
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        res[f"r{r}_{'mli' if mli else 'seq'}"] = a.elapsed_time(b) / steps
        launches += steps * (2 * sum(keep) + n * (1 + (1 if st["wsb"] > 0 else 0)))
    return res, launches


def build_prefill(device, ctx=65536, nq=4096, budget=256 << 20):
    """The chunked-prefill workload: one request with a 65536-token FP8 key cache
    and latent cache, its last 4096 positions as query rows (each sees the
    tokens up to itself), top-2048 and the sparse attention per row; run in the
    chunks the plan gives for a 256 MiB logits budget, and in one chunk."""
    import numpy as np
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case = W.make_indexer_case([ctx], next_n=nq, seed=4, device=device)
    mla = W.make_mla_case(nq, case.layout.num_pages, seed=4, device=device)
    plans = {}
    for name, b in (("chunked", budget), ("one_chunk", None)):
        pieces = dsa.dsa_prefill_chunk_plan([nq], [ctx], b or (nq + 1) * ctx * 4)
        chunks = []
        for ch in sorted({p[0] for p in pieces}):
            ps = [p for p in pieces if p[0] == ch]
            j0, j1 = ps[0][2], ps[-1][3]
            n = j1 - j0
            ld = (ctx + 3) // 4 * 4
            chunks.append(dict(
                j0=j0, n=n, ld=ld,
                cu=torch.tensor([0, n], dtype=torch.int32, device=device),
                ctx=torch.tensor([ctx - (nq - j1)], dtype=torch.int32, device=device),
                btr=torch.zeros(1, dtype=torch.int32, device=device),
                row_bt=torch.zeros(n, dtype=torch.int32, device=device)))
        nmax = max(c["n"] for c in chunks)
        wsb = dsa.dsa_sparse_mla_workspace_size(nmax, TOPK)
        plans[name] = dict(chunks=chunks,
                           logits=torch.empty((nmax, chunks[0]["ld"]), device=device),
                           row_len=torch.empty(nmax, dtype=torch.int32, device=device),
                           sel=torch.empty((nmax, TOPK), dtype=torch.int32, device=device),
                           ws=torch.empty(max(wsb, 16), dtype=torch.uint8, device=device),
                           wsb=wsb)
    out = torch.empty((nq, W.MLA_HEADS, W.MLA_DV), dtype=torch.bfloat16, device=device)
    lse = torch.empty((nq, W.MLA_HEADS), device=device)
    return dict(case=case, mla=mla, plans=plans, out=out, lse=lse, nq=nq, ctx=ctx, budget=budget)


def prefill_step(pst, plan):
    """One chunked prefill through the public API; returns the launches made."""
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case, mla = pst["case"], pst["mla"]
    lay, c = case.layout, case.cache
    P = pst["plans"][plan]
    launches = 0
    for ch in P["chunks"]:
        j0, n, ld = ch["j0"], ch["n"], ch["ld"]
        logits = P["logits"][:n]
        dsa.dsa_indexer_logits_varlen(case.q[j0:j0 + n], case.q_scale[j0:j0 + n],
                                      case.w[j0:j0 + n], c, W.FP8_PAGE_BYTES,
                                      c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES,
                                      lay.num_pages, lay.block_table, ch["btr"], ch["ctx"],
                                      ch["cu"], 1, n, n, logits, ld)
        dsa.dsa_varlen_row_lengths(ch["ctx"], ch["cu"], 1, n, P["row_len"])
        dsa.dsa_topk(logits, ld, P["row_len"], n, TOPK, P["sel"])
        wsb = dsa.dsa_sparse_mla_workspace_size(n, TOPK)
        dsa.dsa_sparse_mla_decode_varlen(mla.q[j0:j0 + n], mla.kv, 64 * 576 * 2, lay.num_pages,
                                         lay.block_table, ch["row_bt"], n, P["sel"][:n], TOPK,
                                         mla.scale, pst["out"][j0:j0 + n], pst["lse"][j0:j0 + n],
                                         P["ws"], P["wsb"])
        launches += 5 + (1 if wsb > 0 else 0)
    return launches


def prefill_kernel_ms(pst, plan, reps, stream):
    """Mean ms per step of the prefill's indexer, top-k and sparse MLA launches
    (events around each launch of every chunk, summed over the chunks)."""
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case, mla = pst["case"], pst["mla"]
    lay, c = case.layout, case.cache
    P = pst["plans"][plan]
    acc = {"indexer": 0.0, "topk": 0.0, "sparse_mla": 0.0}
    for _ in range(reps):
        evs = []
        for ch in P["chunks"]:
            j0, n, ld = ch["j0"], ch["n"], ch["ld"]
            logits = P["logits"][:n]
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            dsa.dsa_indexer_logits_varlen(case.q[j0:j0 + n], case.q_scale[j0:j0 + n],
                                          case.w[j0:j0 + n], c, W.FP8_PAGE_BYTES,
                                          c.data_ptr() + W.FP8_KEY_BYTES, W.FP8_PAGE_BYTES,
                                          lay.num_pages, lay.block_table, ch["btr"], ch["ctx"],
                                          ch["cu"], 1, n, n, logits, ld)
            e[1].record(stream)
            dsa.dsa_varlen_row_lengths(ch["ctx"], ch["cu"], 1, n, P["row_len"])
            dsa.dsa_topk(logits, ld, P["row_len"], n, TOPK, P["sel"])
            e[2].record(stream)
            dsa.dsa_sparse_mla_decode_varlen(mla.q[j0:j0 + n], mla.kv, 64 * 576 * 2,
                                             lay.num_pages, lay.block_table, ch["row_bt"], n,
                                             P["sel"][:n], TOPK, mla.scale,
                                             pst["out"][j0:j0 + n], pst["lse"][j0:j0 + n],
                                             P["ws"], P["wsb"])
            e[3].record(stream)
            evs.append(e)
        torch.cuda.synchronize()
        for e in evs:
            acc["indexer"] += e[0].elapsed_time(e[1])
            acc["topk"] += e[1].elapsed_time(e[2])
            acc["sparse_mla"] += e[2].elapsed_time(e[3])
    return {k: v / reps for k, v in acc.items()}


def time_prefill(pst, steps, warmup, stream):
    import torch
    res, launches = {}, 0
    for plan in ("chunked", "one_chunk"):
        for _ in range(warmup):
            prefill_step(pst, plan)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            launches += prefill_step(pst, plan)
        b.record(stream)
        torch.cuda.synchronize()
        res[plan] = a.elapsed_time(b) / steps
    return res, launches


def kernel_roofline(alg_bytes, flops, ms, hbm_gbs, bf16_tflops):
    """A kernel against its own roofline: the least time its algorithmic bytes
    (at the measured copy bandwidth) and flops (at the bf16 tensor peak) allow,
    divided by its measured time."""
    t_mem = alg_bytes / (hbm_gbs * 1e9)
    t_math = flops / (bf16_tflops * 1e12)
    bound = t_mem if t_mem >= t_math else t_math
    return {"bound": "hbm" if t_mem >= t_math else "tensor", "roofline_us": bound * 1e6,
            "measured_us": ms * 1e3, "frac": bound / (ms * 1e-3)}


def time_kernels(kernels, steps, warmup, stream):
    """Runs `steps` timed passes of the launches back to back (the step's time)
    and `steps` passes with an event after every launch (the per-kernel
    breakdown; events between kernels add time of their own and keep a kernel
    from being scheduled while the previous one finishes).  Returns (total ms
    of the plain passes, {name: mean ms per launch})."""
    import torch
    for _ in range(warmup):
        for _, fn in kernels:
            fn()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        for _, fn in kernels:
            fn()
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    n = len(kernels)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    for s in range(steps):
        ev[s][0].record(stream)
        for j, (_, fn) in enumerate(kernels):
            fn()
            ev[s][j + 1].record(stream)
    torch.cuda.synchronize()
    per = {}
    for j, (name, _) in enumerate(kernels):
        per[name] = sum(ev[s][j].elapsed_time(ev[s][j + 1]) for s in range(steps)) / steps
    return total, per


def e2e_decode_pipelined(st, steps, warmup, stream):
    """The same step through the public API with the per-step host inputs
    (pinned) copied in and the step's outputs copied out, as a server runs it:
    two device sets of per-step inputs and outputs; step i's input copy runs on
    a copy stream while step i-1's kernels run, and its output copy on another
    while step i+1's kernels run.  Every step copies all its inputs in and all
    its outputs out; the timed region ends when the last output has landed."""
    import torch
    from deepseek_sparse_attention_02_gb300 import dsa
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case, mla, R, ld = st["case"], st["mla"], st["R"], st["ld"]
    c, lay = case.cache, case.layout
    host_in = [t.cpu().pin_memory() for t in (case.q, case.q_scale, case.w, lay.block_table,
                                               lay.ctx_len, st["L"], mla.q)]
    sets = []
    for _ in range(2):
        ins = [torch.empty_like(t, device=st["out"].device) for t in host_in]
        outs = [torch.empty_like(st["out"]), torch.empty_like(st["lse"]), torch.empty_like(st["idx"])]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        sets.append(dict(ins=ins, outs=outs, host_out=host_out,
                         in_ready=torch.cuda.Event(), in_free=torch.cuda.Event(),
                         out_free=torch.cuda.Event()))
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def kernels(io):
        q, qs, w, bt, ctx, rl, mq = io["ins"]
        out, lse, idx = io["outs"]
        dsa.dsa_indexer_logits(q, qs, w, c, W.FP8_PAGE_BYTES, c.data_ptr() + W.FP8_KEY_BYTES,
                               W.FP8_PAGE_BYTES, lay.num_pages, bt, ctx, len(lay.ctx_len), 2,
                               st["logits"], ld)
        dsa.dsa_topk(st["logits"], ld, rl, R, TOPK, idx)
        dsa.dsa_sparse_mla_decode(mq, mla.kv, 64 * 576 * 2, lay.num_pages, bt, len(lay.ctx_len),
                                  2, idx, TOPK, mla.scale, out, lse, st["ws"], st["wsb"])

    def step(i, first):
        io = sets[i % 2]
        with torch.cuda.stream(h2d_s):
            if not first[i % 2]:
                h2d_s.wait_event(io["in_free"])  # step i-2's kernels are done with these inputs
            for h, d in zip(host_in, io["ins"]):
                d.copy_(h, non_blocking=True)
            io["in_ready"].record(h2d_s)
        stream.wait_event(io["in_ready"])
        if not first[i % 2]:
            stream.wait_event(io["out_free"])  # step i-2's outputs have been read back
        with torch.cuda.stream(stream):
            kernels(io)
            io["in_free"].record(stream)
        d2h_s.wait_event(io["in_free"])
        with torch.cuda.stream(d2h_s):
            for h, d in zip(io["host_out"], io["outs"]):
                h.copy_(d, non_blocking=True)
            io["out_free"].record(d2h_s)
        first[i % 2] = False

    first = [True, True]
    for i in range(warmup):
        step(i, first)
    torch.cuda.synchronize()
    first = [True, True]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    h2d_s.wait_event(a)
    for i in range(steps):
        step(i, first)
    for io in sets:
        stream.wait_event(io["out_free"])
    b.record(stream)
    torch.cuda.synchronize()
    # the read-back outputs are the step's results
    assert torch.equal(sets[(steps - 1) % 2]["host_out"][2], sets[(steps - 1) % 2]["outs"][2].cpu())
    return a.elapsed_time(b) / steps


def e2e_decode(st, steps, warmup, stream):
    """Same step through the public API with per-step host inputs (pinned) copied in
    and the step's outputs copied out inside the timed region."""
    import torch
    case, mla = st["case"], st["mla"]
    dev_inputs = [case.q, case.q_scale, case.w, case.layout.block_table, case.layout.ctx_len,
                  st["L"], mla.q]
    host_inputs = [t.cpu().pin_memory() for t in dev_inputs]
    dev_outputs = [st["out"], st["lse"], st["idx"]]
    host_outputs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_outputs]
    kernels = decode_kernels(st)

    def step():
        for h, d in zip(host_inputs, dev_inputs):
            d.copy_(h, non_blocking=True)
        for _, fn in kernels:
            fn()
        for h, d in zip(host_outputs, dev_outputs):
            h.copy_(d, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(t.numel() * t.element_size() for t in host_inputs)
    d2h = sum(t.numel() * t.element_size() for t in host_outputs)
    return ms, h2d, d2h


# ---------------------------------------------------------- oracle timings --
# The fp64 CPU oracle (test infrastructure) timed on this host's cores as the
# reported baseline of each workload, on the very inputs the GPU legs ran
# (copied to the host), with the samples the benchmark spec plans: the tiny decode,
# the batched varlen path and the candidate path in full, all 64 rows of the
# 128K step, and 64 of the 4096 prefill rows (extrapolated by their (row,
# key) pairs).

def _np(t):
    return t.detach().cpu().numpy()


def _bits(t):
    import numpy as np
    from deepseek_sparse_attention_02_gb300 import workloads as W
    return W.bf16_bits(t).cpu().numpy().view(np.uint16)


def oracle_dense_path(case, next_n, mla, th, rows=None):
    """Indexer + full-sort top-2048 (+ sparse MLA over the oracle's own
    selection when `mla` is given) of `rows` (all by default) of a dense
    workload.  Returns (seconds, (row, key) pairs, rows)."""
    import numpy as np
    import oracle
    from deepseek_sparse_attention_02_gb300 import workloads as W
    sel = np.arange(case.rows, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    ctx = _np(case.layout.ctx_len)
    L = oracle.row_lengths(ctx, next_n)[sel]
    cache = _np(case.cache).reshape(-1)
    bt = _np(case.layout.block_table)
    q, qs, w = _np(case.q), _np(case.q_scale), _np(case.w)
    if mla is not None:
        q_bits, kv_bits = _bits(mla.q), _bits(mla.kv)
    t0 = time.perf_counter()
    ref, _ = oracle.indexer_logits(q, qs, w, cache, W.FP8_PAGE_BYTES, cache[W.FP8_KEY_BYTES:],
                                   W.FP8_PAGE_BYTES, 64, bt, ctx, next_n, rows=sel, nthreads=th)
    idx = oracle.topk(ref, L, TOPK, nthreads=th)
    if mla is not None:
        idx_full = np.full((case.rows, TOPK), -1, np.int32)
        idx_full[sel] = idx
        oracle.sparse_mla(q_bits, kv_bits, 64 * 576, 64, bt, next_n, idx_full, mla.scale, rows=sel,
                          nthreads=th)
    return time.perf_counter() - t0, float(L.sum()), len(sel)


def oracle_candidate_path(cst, th):
    """The candidate path in full: one expansion, then the 4 consumer layers'
    MXFP4 candidate logits and the top-2048 over them.  Returns (seconds,
    candidate (row, column) pairs scored)."""
    import oracle
    from deepseek_sparse_attention_02_gb300 import workloads as W
    cand = _np(cst["cand"])
    ctx = _np(cst["layers"][0].layout.ctx_len)
    layers = [(_np(c.q), _np(c.q_scale), _np(c.w), _np(c.cache).reshape(-1),
               _np(c.layout.block_table)) for c in cst["layers"]]
    t0 = time.perf_counter()
    si, end = oracle.candidate_expand(cand, 64, ctx, 1)
    for q, qs, w, cache, bt in layers:
        lg, _ = oracle.candidate_logits(q, qs, w, cache, W.FP4_PAGE_BYTES, cache[W.FP4_KEY_BYTES:],
                                        W.FP4_PAGE_BYTES, 64, bt, 1, si, 64, end, nthreads=th)
        oracle.topk(lg, end, TOPK, col_blocks=si, bs=64, nthreads=th)
    return time.perf_counter() - t0, float(end.sum()) * len(layers)


def oracle_baselines(th, st, dense, cst, pst):
    """Every workload's oracle time on this host (the plan above), on the
    inputs of the GPU legs that ran."""
    import numpy as np
    out = {}
    for d in dense:
        name = "tiny_decode" if d["cfg"] == 0 else "batched_varlen"
        dt, keys, n = oracle_dense_path(d["case"], d["next_n"], d["mla"], th)
        out[name] = {"seconds": round(dt, 3), "keys_per_s": keys / dt,
                     "sample": f"all {n} rows (full workload)"}
    dt, keys, n = oracle_dense_path(st["case"], 2, st["mla"], th)
    out["mtp_128k"] = {"seconds": round(dt, 3), "keys_per_s": keys / dt,
                       "sample": f"all {n} rows (full workload)"}
    if cst is not None:
        dt, keys = oracle_candidate_path(cst, th)
        out["candidate"] = {"seconds": round(dt, 3), "keys_per_s": keys / dt,
                            "sample": "full workload (1 expansion + 4 layers)"}
    if pst is not None:
        nq, ctx = pst["nq"], pst["ctx"]
        rng = np.random.default_rng(4)
        rows = np.unique(np.concatenate([[0, nq - 1], rng.choice(nq, 62, replace=False)]))[:64]
        dt, keys, n = oracle_dense_path(pst["case"], nq, pst["mla"], th, rows=rows)
        total = sum(ctx - (nq - 1 - j) for j in range(nq))
        out["prefill"] = {"seconds_sample": round(dt, 3), "keys_per_s": keys / dt,
                          "seconds_full_extrapolated": round(dt * total / keys, 1),
                          "sample": f"{n} of the {nq} query rows (first, last, seeded middle); "
                                    "full time extrapolated by (row, key) pairs"}
    return out


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def aggregate_value(world: int, units_per_rank: float, ms_max: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's step."""
    return world * units_per_rank / (ms_max * 1e-3)


def reduce_max(pg, value: float, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg, device):
    if pg is not None:
        if device.type == "cuda":
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def run_ours(args):
    import torch
    world, rank, local, pg = dist_setup()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import __graft_entry__ as g
    g.build()
    from deepseek_sparse_attention_02_gb300 import dsa
    stream = torch.cuda.current_stream()
    st = build_decode(device, requests=args.requests)
    kernels = decode_kernels(st)
    cst = None if args.no_candidate else build_candidate(device, requests=args.candidate_requests)
    ckernels = [] if cst is None else candidate_kernels(cst)
    ckernels16 = [] if cst is None else candidate_kernels(cst, bf16=True)
    lst = None if args.no_layers else build_layers(st)
    pst = None if args.no_prefill else build_prefill(device)
    dense = [] if args.no_configs else [build_dense_config(device, cfg) for cfg in (0, 1)]
    torch.cuda.synchronize()

    barrier(pg, device)
    with ClockSampler(local) as clocks:
        total_ms, per = time_kernels(kernels, args.steps, args.warmup, stream)
        dense_res = [time_kernels(dense_config_kernels(d), args.steps, args.warmup, stream)
                     for d in dense]
        if ckernels:
            c_total_ms, c_per = time_kernels(ckernels, args.steps, args.warmup, stream)
            c16_total_ms, c16_per = time_kernels(ckernels16, args.steps, args.warmup, stream)
        if lst is not None:
            lay_ms, lay_launches = time_layers(st, lst, args.steps, args.warmup, stream)
        if pst is not None:
            pre_ms, pre_launches = time_prefill(pst, args.steps, args.warmup, stream)
            pre_kms = prefill_kernel_ms(pst, "one_chunk", max(1, args.steps // 4), stream)
    barrier(pg, device)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0, "device error word set during the benchmark"
    ms_step = total_ms / args.steps
    ms_step_max = reduce_max(pg, ms_step, device)

    keys_per_step = float(st["L"].sum().item())
    value = aggregate_value(world, keys_per_step, ms_step_max)
    hbm, bf16_tf, peak_src = peaks()
    dense_out = {}
    for d, (tms, dper) in zip(dense, dense_res):
        name = "tiny_decode" if d["cfg"] == 0 else "batched_varlen"
        dense_out[name] = dense_metrics(d, tms, dper, args.steps, hbm, bf16_tf)
    # dominant kernel: the indexer (HBM-bound): 128 B key + 4 B scale per cached
    # token read, 4 B logit per (row, key) written
    tokens = args.requests * 131072
    alg_bytes = tokens * 132 + keys_per_step * 4
    # measured DRAM traffic of the indexer, scaled by the cached tokens (the
    # traffic grows in proportion to them)
    traffic = INDEXER_DRAM_BYTES_PER_TOKEN * tokens
    t_idx = per["indexer"] * 1e-3
    achieved = alg_bytes / t_idx / 1e9
    R = st["R"]
    # top-k: 4 B per valid logit read + the indices written; sparse MLA: the
    # selected latents (1152 B each) + Q read + O written, and its flops
    topk_bytes = keys_per_step * 4 + R * TOPK * 4
    mla_bytes = R * TOPK * 1152 + R * 128 * 576 * 2 + R * 128 * 512 * 2
    mla_flops = R * 2 * 128 * TOPK * (576 + 512)
    e2e_serial_ms, h2d, d2h = e2e_decode(st, args.steps, args.warmup, stream)
    e2e_serial_ms = reduce_max(pg, e2e_serial_ms, device)
    e2e_ms = e2e_decode_pipelined(st, args.steps, args.warmup, stream)
    e2e_ms = reduce_max(pg, e2e_ms, device)
    # candidate path numbers
    cand = None
    if cst is not None:
        cand_keys = float(cst["end"].sum().item()) * 4
        c_ms = c_total_ms / args.steps
        c_log = statistics.mean(c_per[f"cand_logits_{i}"] for i in range(4))
        c_bytes = float(cst["end"].sum().item()) * 68 + float(cst["end"].sum().item()) * 4
        ctk = statistics.mean(c_per[f"cand_topk_{i}"] for i in range(4))
        cand = {"workload": f"{cst['R']} requests x 196608 ctx, 512 candidate blocks of 64, "
                            "MXFP4 keys, 1 expansion + 4 consumer layers (logits + top-2048)",
                "ms_per_step": c_ms,
                "breakdown_ms": {k: round(v, 4) for k, v in c_per.items()},
                "candidate_keys_per_s": cand_keys / (c_ms * 1e-3),
                "logits_hbm_gbs": c_bytes / (c_log * 1e-3) / 1e9,
                # 64 B packed key + 4 B UE8M0 scales read + 4 B logit written per column
                "logits_hbm_frac": round(c_bytes / (c_log * 1e-3) / 1e9 / hbm, 4),
                "topk_rows_per_s": cst["R"] / (ctk * 1e-3),
                "topk_frac": round(kernel_roofline(float(cst["end"].sum().item()) * 4 +
                                                   cst["R"] * TOPK * 4, 0.0, ctk, hbm,
                                                   bf16_tf)["frac"], 4),
                "bf16_logits": {
                    "ms_per_step": c16_total_ms / args.steps,
                    "breakdown_ms": {k: round(v, 4) for k, v in c16_per.items()},
                    "candidate_keys_per_s": cand_keys / (c16_total_ms / args.steps * 1e-3)}}

    layers = None
    if lst is not None:
        base = lay_ms["r1_seq"]
        layers = {"workload": f"{len(lst['layers'])} DSA layers of the headline step (own "
                              "indexer and attention queries per layer, shared caches); "
                              "retention 1/r keeps the indexer of layers l % r == 0; "
                              "mli = each layer attends the previous indexer layer's "
                              "selection, its own indexer on a second stream",
                  "ms_per_step": {k: round(v, 4) for k, v in lay_ms.items()},
                  "speedup_vs_r1_seq": {k: round(base / v, 3) for k, v in lay_ms.items()}}

    prefill = None
    if pst is not None:
        nrows, ctxn = pst["nq"], pst["ctx"]
        nchunks = len(pst["plans"]["chunked"]["chunks"])
        pairs = sum(ctxn - (nrows - 1 - j) for j in range(nrows))
        prefill = {"workload": f"1 request, {ctxn}-token cache, its last {nrows} positions as "
                               f"query rows: indexer, top-{TOPK}, sparse MLA per row",
                   "chunked": {"budget_bytes": pst["budget"], "chunks": nchunks,
                               "ms": round(pre_ms["chunked"], 4),
                               "keys_per_s": pairs / (pre_ms["chunked"] * 1e-3)},
                   "one_chunk": {"logits_bytes": nrows * ctxn * 4,
                                 "ms": round(pre_ms["one_chunk"], 4),
                                 "keys_per_s": pairs / (pre_ms["one_chunk"] * 1e-3),
                                 "breakdown_ms": {k: round(v, 4) for k, v in pre_kms.items()}}}
        # tensor-pipe fractions of the one-chunk launches: the indexer's FP8
        # contraction (2 * 64 * 128 flops per (row, key)) against twice the
        # measured bf16 burst (the nominal FP8 : bf16 dense ratio), the
        # attention's bf16 contractions (2 * 128 * k * (576 + 512) per row)
        # against the bf16 burst
        idx_flops = pairs * 2 * 64 * 128
        mla_flops_p = nrows * 2 * 128 * TOPK * (576 + 512)
        prefill["one_chunk"]["indexer_tensor_frac"] = round(
            idx_flops / (pre_kms["indexer"] * 1e-3) / 1e12 / (2 * bf16_tf), 4)
        prefill["one_chunk"]["sparse_mla_tensor_frac"] = round(
            mla_flops_p / (pre_kms["sparse_mla"] * 1e-3) / 1e12 / bf16_tf, 4)
        prefill["one_chunk"]["attended_tok_per_s"] = nrows * TOPK / (pre_kms["sparse_mla"] * 1e-3)

    topk_rf = kernel_roofline(topk_bytes, 0.0, per["topk"], hbm, bf16_tf)
    mla_rf = kernel_roofline(mla_bytes, mla_flops, per["sparse_mla"], hbm, bf16_tf)
    kernels_rf = {"topk": {"frac": round(topk_rf["frac"], 4), "bound": "hbm",
                           "measured_us": round(topk_rf["measured_us"], 2),
                           "roofline_us": round(topk_rf["roofline_us"], 2)},
                  "sparse_mla": {"frac": round(mla_rf["frac"], 4), "bound": mla_rf["bound"],
                                 "measured_us": round(mla_rf["measured_us"], 2),
                                 "roofline_us": round(mla_rf["roofline_us"], 2)}}
    if cand is not None:
        kernels_rf["candidate_logits"] = {"frac": cand["logits_hbm_frac"], "bound": "hbm"}
        kernels_rf["candidate_topk"] = {"frac": cand["topk_frac"], "bound": "hbm"}
    if prefill is not None:
        kernels_rf["prefill_indexer"] = {"frac": prefill["one_chunk"]["indexer_tensor_frac"],
                                         "bound": "tensor (fp8 = 2 x bf16 burst)"}
        kernels_rf["prefill_sparse_mla"] = {
            "frac": prefill["one_chunk"]["sparse_mla_tensor_frac"], "bound": "tensor (bf16 burst)"}
    for name, d in dense_out.items():
        kernels_rf[f"{name}_indexer"] = {"frac": d["indexer_hbm_frac"], "bound": "hbm"}
        kernels_rf[f"{name}_topk"] = {"frac": d["topk_frac"], "bound": "hbm"}
        if "sparse_mla_frac" in d:
            kernels_rf[f"{name}_sparse_mla"] = {"frac": d["sparse_mla_frac"], "bound": "max"}
    fr = {"indexer_hbm_frac": achieved / hbm, "topk_frac": topk_rf["frac"],
          "sparse_mla_frac": mla_rf["frac"]}
    targets = {f"{k} >= {v:.2f}": {"value": round(fr[k], 4), "pass": bool(fr[k] >= v)}
               for k, v in TARGETS.items()}
    n_dense = sum(2 * args.steps * len(dense_config_kernels(d)) for d in dense)
    n_pre = 0
    if pst is not None:
        P1 = pst["plans"]["one_chunk"]
        n_pre = max(1, args.steps // 4) * len(P1["chunks"]) * (4 + (1 if P1["wsb"] > 0 else 0))
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "keys/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8-e4m3 indexer (f32 accumulate), f32 top-k, bf16 MLA (f32 accumulate)",
        "data": "synthetic (seeded, generated on device)",
        "config": {"workload": WORKLOAD if args.requests == 32 else
                   WORKLOAD.replace("32 requests", f"{args.requests} requests").replace(
                       "(64 rows)", f"({2 * args.requests} rows)"),
                   "global_batch": 2 * args.requests * world, "seq_len": 131072,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({tokens * 132 / 1e6:.1f} MB key cache, "
                         f"{tokens * 1152 / 1e9:.1f} GB latent cache); no flush"},
        "candidate_path": cand,
        "layer_schedules": layers,
        "prefill_chunks": prefill,
        "indexer": {"keys_per_s": keys_per_step / t_idx, "hbm_gbs": achieved,
                    "unique_keys_per_s": tokens / t_idx},
        "topk": {"rows_per_s": R / (per["topk"] * 1e-3),
                 "logit_gbs": keys_per_step * 4 / (per["topk"] * 1e-3) / 1e9,
                 "roofline": topk_rf},
        "sparse_mla": {"attended_tok_per_s": R * TOPK / (per["sparse_mla"] * 1e-3),
                       "gather_gbs": R * TOPK * 1152 / (per["sparse_mla"] * 1e-3) / 1e9,
                       "tflops": mla_flops / (per["sparse_mla"] * 1e-3) / 1e12,
                       "roofline": mla_rf},
        # time_kernels times the plain passes and the event-instrumented ones
        "gpu_launches": 2 * args.steps * (len(kernels) + (1 if st["wsb"] > 0 else 0)) +
                        2 * (args.steps * (len(ckernels) + 1) if ckernels else 0) * 2 +
                        (lay_launches if lst is not None else 0) +
                        (pre_launches if pst is not None else 0) + n_dense + n_pre,
        "e2e": {"value": world * keys_per_step / (e2e_ms * 1e-3), "unit": "keys/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "pinned host; step i+1's inputs and step i-1's outputs copied while "
                          "step i's kernels run (two buffer sets, two copy streams)",
                "serial": {"value": world * keys_per_step / (e2e_serial_ms * 1e-3),
                           "ms_per_step": e2e_serial_ms}},
        "clocks": clocks.summary(),
        # the per-workload figures last (the end of the line is what a reader
        # of a truncated log sees)
        "configs": dense_out,
        "breakdown_ms": {k: round(v, 4) for k, v in per.items()},
        "roofline": {"kernel": "dsa_indexer_logits", "bound": "hbm", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                     "peak_source": peak_src, "alg_bytes_per_launch": alg_bytes,
                     "kernels": kernels_rf, "targets": targets},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        th = _oracle_threads()
        ob = oracle_baselines(th, st, dense, cst, pst)
        line["cpu_baseline"] = {"value": ob["mtp_128k"]["keys_per_s"], "unit": "keys/s",
                                "cores": th, "kind": "oracle",
                                "sample": "the 128K MTP step's 64 rows in full (oracle indexer, "
                                          "full-sort top-2048, sparse MLA); keys/s = (row, key) "
                                          "pairs / time",
                                "seconds": ob["mtp_128k"]["seconds"], "workloads": ob}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def _oracle_threads():
    import oracle
    return oracle.hardware_threads()


def run_reference(args):
    """The oracle (the reference arm of this build) on the headline workload:
    each step is the 128K MTP step's 64 rows in full on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    th = _oracle_threads()
    vals, dts = [], []
    from deepseek_sparse_attention_02_gb300 import workloads as W
    case = W.make_indexer_case([131072] * 32, next_n=2, seed=0, device="cpu")
    mla = W.make_mla_case(case.rows, case.layout.num_pages, seed=0, device="cpu")
    for _ in range(args.warmup):
        oracle_dense_path(case, 2, mla, th)
    for _ in range(args.steps):
        dt, keys, n = oracle_dense_path(case, 2, mla, th)
        vals.append(keys / dt)
        dts.append(dt)
    value = statistics.mean(vals)
    tokens = 32 * 131072
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(dts),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "global_batch": 64, "seq_len": 131072,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({tokens * 132 / 1e6:.1f} MB key cache, "
                         f"{tokens * 1152 / 1e9:.1f} GB latent cache); no flush"},
        "cpu_baseline": {"value": value, "unit": "keys/s", "cores": th, "kind": "oracle",
                         "sample": "the 128K MTP step's 64 rows in full per step (oracle indexer, "
                                   "full-sort top-2048, sparse MLA)"},
        "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--requests", type=int, default=32,
                    help="decode requests (32 = the 128K workload; fewer for profiling)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the chunked-prefill measurement")
    ap.add_argument("--no-layers", action="store_true",
                    help="skip the multi-layer IndexCache / MLI schedule measurement")
    ap.add_argument("--no-candidate", action="store_true",
                    help="skip the candidate-path leg (profiling)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the tiny-decode and batched-varlen legs (profiling)")
    ap.add_argument("--candidate-requests", type=int, default=64,
                    help="candidate-path requests (64 = the candidate workload; fewer for profiling)")
    return ap


def main():
    args = build_parser().parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
