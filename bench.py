#!/usr/bin/env python3
"""Benchmark of the VQ KV-cache decode step on GB300.

One step = the whole hot path over one batch: the new token's K and V rows
are quantised into the cache (vqkv_encode, keys smoothed + rotated), then
decode attention runs over the packed cache (vqkv_decode_attn).  The
workload is the Llama-3.1-8B-shaped 2-bit decode at 196,608 cached tokens
(batch 1, 32 query heads over 8 KV heads, head_dim 128); its cache is
produced by the library's own GPU encoder from seeded synthetic K/V.

Prints one JSON line: the contract's keys (metric, value, unit, n_gpus,
steps, warmup, ms_per_step, config, ...) plus "roofline" (the decode
kernel's algorithmic bytes per launch over its back-to-back launch time,
against the measured HBM copy bandwidth), "cpu_baseline" (the CPU oracle on
a bounded sample), "e2e" (through the public binding with host buffers),
"near_ties" (near-tie counts of the encodes the run made) and
"fp16_kv_decode" (the fp16-KV comparison kernel on the same shape).
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from vector_quantized_bit_gb300 import calib, synth  # noqa: E402

METRIC = "decode-attn KV tokens/s and HBM GB/s vs GB300 peak (2-bit, Llama-8B shape, 196k)"
WORKLOAD_ID = 1
GRAPH_STEPS = 100           # steps captured per CUDA graph
SOAK_S = 0.5                # untimed load on each side of the timed region for clock sampling
PROFILE_JSON = os.path.join(ROOT, "profiles", "decode_vq2_llama8b_196k.json")
BITS = {0: 2, 1: 1.5, 2: 4, 3: 3, 4: 1.25}   # bits per element of each code mode


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=[1, 2, 3, 4],
                    help="1: Llama-3.1-8B 196k 2-bit (default); 2: ragged batch of 32; "
                         "3: Qwen2.5-14B 1.5-bit; 4: Mistral-7B encode + decode")
    ap.add_argument("--mode", type=int, default=None, choices=[0, 1, 2, 3, 4],
                    help="override the workload's bit-width (0: 2-bit, 1: 1.5-bit, 2: 4-bit)")
    ap.add_argument("--queries", type=int, default=1,
                    help="queries per sequence (multi-query decode, e.g. speculative decoding): a step encodes "
                         "that many new K/V rows per sequence and runs vqkv_decode_attn_multi")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK_TOKENS",
                    help="keep the cache in a pool of blocks of this many tokens behind a shuffled block table "
                         "(vqkv_encode_paged / vqkv_decode_attn_paged)")
    ap.add_argument("--unfused", action="store_true",
                    help="2-bit: run a step as vqkv_encode (K) + vqkv_encode (V) + vqkv_decode_attn instead of "
                         "the fused vqkv_decode_append")
    ap.add_argument("--profile-fp16", type=int, default=0,
                    help="run this many fp16-KV comparison decodes of the workload (eager) and exit: the "
                         "command the fp16 kernel's ncu summary is taken with")
    ap.add_argument("--calib", action="store_true",
                    help="time the offline calibration stage (smoothing, key transform, K-Means training) instead")
    ap.add_argument("--ablation", action="store_true",
                    help="codebook utilisation and reconstruction error of the five key transforms instead")
    ap.add_argument("--profile-encode", type=int, default=-1, choices=[-1, 0, 1, 3, 4],
                    help="time the key prefill encode of 4 of the Mistral-shaped workload's sequences (4 x 8 x "
                         "16,384 rows) in this code mode (0: 2-bit, 1: 1.5-bit, 3: 3-bit, 4: 1.25-bit), 3 calls, "
                         "and exit: the command the encode ncu summaries are taken with")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="set up the workload, run this many plain (eager) steps and exit: "
                         "the command the ncu summaries under profiles/ are taken with")
    return ap.parse_args()


# ------------------------------------------------------------- workload

def _gen_head(args):
    w, b, kvh = args
    return synth.keys(w, b, kvh, 0, w.seq_len), synth.values(w, b, kvh, 0, w.seq_len)


def _cal_head(args):
    w, kvh = args
    return calib.calibrate_head(w, kvh)


def _cal_head_small(args):
    w, kvh = args
    return calib.calibrate_head(w, kvh, sample_tokens=2048, iters=2 if w.mode else 10)


def host_calibration(w):
    """Codebooks and s only (no full K/V on the host)."""
    import concurrent.futures
    import multiprocessing
    n = min(w.Hkv, os.cpu_count() or 1)
    with concurrent.futures.ProcessPoolExecutor(n, mp_context=multiprocessing.get_context("spawn")) as ex:
        cal = list(ex.map(_cal_head_small, [(w, h) for h in range(w.Hkv)]))
    return np.stack([c[0] for c in cal]), np.stack([c[1] for c in cal]), np.stack([c[2] for c in cal])


def host_workload(w):
    """Calibration and synthetic K/V on host worker processes (spawned before
    any CUDA call)."""
    import concurrent.futures
    import multiprocessing
    n = min(w.Hkv, os.cpu_count() or 1)
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(n, mp_context=ctx) as ex:
        cal = list(ex.map(_cal_head, [(w, h) for h in range(w.Hkv)]))
        kv = list(ex.map(_gen_head, [(w, 0, h) for h in range(w.Hkv)]))
    s = np.stack([c[0] for c in cal])
    kcb = np.stack([c[1] for c in cal])
    vcb = np.stack([c[2] for c in cal])
    return s, kcb, vcb, kv


def algorithmic_bytes(w, lens):
    """Packed indices + codebooks + q + O per decode call."""
    E, dsub = synth.MODE_GEOMETRY[w.mode]
    code_bits = int(math.log2(E))
    th = int(np.sum(lens)) * w.Hkv
    idx = 2 * th * (128 // dsub) * code_bits // 8
    cbs = 2 * w.Hkv * E * dsub * 2
    qo = 2 * w.B * w.Hq * 128 * 2
    return idx + cbs + qo


# ------------------------------------------------------------- clocks

class ClockSampler:
    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="vqkv_clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- cpu baseline (the oracle)

_ORACLE_INPUTS = {}


def _oracle_setup(max_tokens):
    """Inputs of the oracle runs (built once per worker, not timed): every KV
    head's codebooks and s (a small calibration), the queries, and seeded
    uniform codes of the first max_tokens tokens of each KV head."""
    w = synth.WORKLOADS[WORKLOAD_ID]
    cal = [calib.calibrate_head(w, h, sample_tokens=512, iters=2) for h in range(w.Hkv)]
    _ORACLE_INPUTS.update(
        s=np.stack([c[0] for c in cal]), kcb=np.stack([c[1] for c in cal]), vcb=np.stack([c[2] for c in cal]),
        q=synth.queries(w),
        kc=[[synth.uniform_codes(w, 0, h, 0, max_tokens) for h in range(w.Hkv)]],
        vc=[[synth.uniform_codes(w, 0, h, 1, max_tokens) for h in range(w.Hkv)]])
    return True


def _oracle_decode_step(n_tokens):
    """Seconds the oracle takes for one decode step of the workload cut to its
    first n_tokens tokens: all 32 query heads over all 8 KV heads."""
    import oracle
    d = _ORACLE_INPUTS
    t0 = time.perf_counter()
    oracle.decode_attention(d["q"], d["kc"], d["vc"], d["kcb"], d["vcb"], d["s"], np.array([n_tokens]))
    return time.perf_counter() - t0


def _oracle_worker(max_tokens):
    import concurrent.futures
    import multiprocessing
    cores = os.cpu_count() or 1
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = str(cores)
    ex = concurrent.futures.ProcessPoolExecutor(1, mp_context=multiprocessing.get_context("spawn"),
                                                initializer=_oracle_setup, initargs=(max_tokens,))
    return ex, cores


def _size_step(ex, seconds, lo=16, hi=196608):
    """Tokens per oracle step so that one step takes about `seconds`."""
    t = ex.submit(_oracle_decode_step, 1024).result()
    n = int(min(hi, max(lo, 1024 * seconds / max(t, 1e-4))))
    return max(16, n // 16 * 16)


def cpu_baseline(budget_s=15.0):
    """The oracle as it stands (fp64 numpy, the plain original-domain path) on
    a bounded sample of the same workload: whole decode steps (all 32 query
    heads over the 8 KV heads) over the first n tokens, n sized so the run
    takes about budget_s of host work."""
    ex, cores = _oracle_worker(196608)
    with ex:
        n = _size_step(ex, budget_s / 3)
        ex.submit(_oracle_decode_step, n).result()   # warm-up
        times = [ex.submit(_oracle_decode_step, n).result() for _ in range(2)]
    t = sum(times) / len(times)
    return {"value": n / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"2 timed decode steps (all 32 query heads, 8 KV heads) over the first {n} of 196608 "
                      f"tokens, {t:.2f} s each; tokens/s = {n} / step seconds"}


# ------------------------------------------------------------- reference arm

def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores.  Each step
    is one decode step of the workload (all 32 query heads over the 8 KV
    heads) over the first n tokens of the cache, n = all 196,608 when the
    whole run fits in about two minutes, else fewer; ms_per_step is the
    measured time of that step and value = n / step seconds."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synth.WORKLOADS[WORKLOAD_ID]
    total = args.steps + args.warmup
    per_step = 120.0 / max(total, 1)
    ex, cores = _oracle_worker(196608)
    with ex:
        n = _size_step(ex, per_step)
        times = []
        for i in range(total):
            dt = ex.submit(_oracle_decode_step, n).result()
            if i >= args.warmup:
                times.append(dt)
    step_s = sum(times) / len(times)
    value = n / step_s
    sample = ("the whole step" if n == w.seq_len else f"the first {n} of {w.seq_len} tokens") + \
        " of all 32 query heads over the 8 KV heads per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": sample, "tokens_per_step": n,
                   "timing": "wall clock around each oracle step on the host"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------- our arm

def max_over_ranks(x, world, device):
    """The largest x over all ranks (the slowest replica sets the job's time)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_replica, ms_per_step, world):
    """Whole-job KV tokens/s of `world` independent replicas (weak scaling:
    every rank decodes its own copy of the workload; no data-path collective)."""
    return world * tokens_per_replica / (ms_per_step * 1e-3)


KERNEL_SOURCES = ("decode.cu", "decode_common.cuh", "encode_common.cuh", "common.cuh", "internal.h")


def kernel_sources_sha256():
    """Hash of the sources the 2-bit decode kernel is compiled from; a stored
    ncu traffic figure is used only while it matches."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "vector_quantized_bit_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def profile_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    try:
        prof = json.load(open(PROFILE_JSON))
    except (OSError, ValueError):
        return None, None
    if prof.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None, prof.get("kernel")
    return prof.get("dram_bytes_per_launch"), prof.get("kernel")


def run_ours(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.WORKLOADS[args.workload]
    if args.mode is not None:
        w = w.with_mode(args.mode)
    headline = args.workload == WORKLOAD_ID and w.mode == synth.MODE_VQ2 and args.queries == 1 and not args.paged
    lens = synth.seq_lens(w)
    if headline:
        s_h, kcb_h, vcb_h, kv = host_workload(w)
    else:
        s_h, kcb_h, vcb_h = host_calibration(w)
        kv = None
    cpu = None
    if headline and rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile_steps:
        cpu = cpu_baseline()

    import torch
    from vector_quantized_bit_gb300 import _build, _lib
    _build.build()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    mode, cap = w.mode, w.cap_len
    sb = _lib.vqkv_code_bytes(mode, cap)
    s = torch.from_numpy(s_h).to(dev)
    kcb = torch.from_numpy(kcb_h).to(dev)
    vcb = torch.from_numpy(vcb_h).to(dev)
    BT = args.paged
    if BT:
        if args.queries != 1 or cap % BT:
            raise SystemExit("--paged needs one query per sequence and a capacity that is a multiple of the block")
        max_blocks = cap // BT
        num_blocks = w.B * max_blocks
        table = torch.from_numpy(np.random.default_rng([w.seed, w.config_id, 77]).permutation(num_blocks)
                                 .reshape(w.B, max_blocks).astype(np.int32)).to(dev)
        kcodes = torch.zeros((num_blocks, w.Hkv, _lib.vqkv_code_bytes(mode, BT)), dtype=torch.uint8, device=dev)
    else:
        kcodes = torch.zeros((w.B, w.Hkv, sb), dtype=torch.uint8, device=dev)
    vcodes = torch.zeros_like(kcodes)

    def encode(role, x, pos_, codes):
        cb = kcb if role == 0 else vcb
        if BT:
            _lib.vqkv_encode_paged(mode, role, x, pos_, s if role == 0 else None, cb, codes, cap, table, BT,
                                   num_blocks)
        else:
            _lib.vqkv_encode(mode, role, x, pos_, s if role == 0 else None, cb, codes, cap)

    zeros = torch.zeros(w.B, dtype=torch.int32, device=dev)
    near_ties = None
    if kv is not None:
        # encode the whole cache (all KV heads, all positions) in one call per K / V,
        # counting near-ties (best two fp32 distances within 1e-6 relative)
        cnt = torch.zeros(2, dtype=torch.int64, device=dev)
        for role, codes in ((0, kcodes), (1, vcodes)):
            x = torch.from_numpy(np.stack([kv[h][role] for h in range(w.Hkv)])[None]).to(dev)
            _lib.vqkv_encode(mode, role, x, zeros, s if role == 0 else None, kcb if role == 0 else vcb, codes, cap,
                             near_tie_count=cnt[role:role + 1])
            del x
        n_codes = w.B * w.Hkv * w.seq_len * (128 // w.d_sub)
        near_ties = {"cache_encode": {"K": int(cnt[0].item()), "V": int(cnt[1].item()), "codes_per_role": n_codes}}
    else:
        # other workloads: seeded uniform codes (decode cost does not depend on code values)
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed * 1000 + w.config_id)
        kcodes.random_(0, 256, generator=gen)
        vcodes.random_(0, 256, generator=gen)
    kv_fp16 = None if args.profile_steps else kv   # kept for the fp16-KV comparison
    del kv
    torch.cuda.synchronize()

    # rotating copies of the cache so each step reads from HBM, not L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cache_bytes = 2 * kcodes.numel()
    n_copies = max(2, math.ceil(3 * l2 / cache_bytes) + 1)
    copies = [(kcodes, vcodes)] + [(kcodes.clone(), vcodes.clone()) for _ in range(n_copies - 1)]

    M = args.queries
    if M == 1:
        q = torch.from_numpy(synth.queries(w)).to(dev)
    else:   # M seeded query sets of the same distribution
        q = torch.from_numpy(np.stack([synth.queries(w.scaled(seed=w.seed + 101 * m)) for m in range(M)], 1)).to(dev)
    new_k = torch.from_numpy(np.stack([np.stack([synth.appended_keys(w, b, h, M) for h in range(w.Hkv)])
                                       for b in range(w.B)])).to(dev)
    new_v = torch.from_numpy(np.stack([np.stack([synth.values(w, b, h, int(lens[b]) - M, M) for h in range(w.Hkv)])
                                       for b in range(w.B)])).to(dev)
    pos = torch.from_numpy((lens - M).astype(np.int32)).to(dev)
    seq = torch.from_numpy(lens.astype(np.int32)).to(dev)
    out = torch.empty(q.shape, dtype=torch.float16, device=dev)
    max_len = int(lens.max())
    ws = _lib.decode_workspace(mode, w.B, w.Hq, w.Hkv, cap, max_len, device=dev, n_queries=M)
    dargs = _lib.decode_args(mode, q.view(w.B, M * w.Hq, 128), kcodes, vcodes, seq, kcb, vcb, s, out, ws, cap,
                             max_len)
    dargs.Hq = w.Hq
    n_splits = _lib.vqkv_decode_num_splits(dargs)
    dec_kernels = _lib.vqkv_decode_kernel_count(dargs)

    fused = mode in (synth.MODE_VQ2, synth.MODE_VQ4) and not args.unfused and M == 1 and not BT

    def decode_only(kc, vc):
        if BT:
            _lib.vqkv_decode_attn_paged(mode, q, kc, vc, seq, kcb, vcb, s, out, ws, cap, max_len, table, BT,
                                        num_blocks)
        elif M == 1:
            _lib.vqkv_decode_attn(mode, q, kc, vc, seq, kcb, vcb, s, out, ws, cap, max_len)
        else:
            _lib.vqkv_decode_attn_multi(mode, q, kc, vc, seq, kcb, vcb, s, out, ws, cap, max_len)

    def step_unfused(i, ev=None):
        kc, vc = copies[i % n_copies]
        encode(0, new_k, pos, kc)
        encode(1, new_v, pos, vc)
        if ev is not None:
            ev[0].record()
        decode_only(kc, vc)
        if ev is not None:
            ev[1].record()

    def decode_call(i):
        kc, vc = copies[i % n_copies]
        if fused:
            _lib.vqkv_decode_append(mode, q, kc, vc, seq, kcb, vcb, s, out, ws, cap, max_len, new_k, new_v)
        else:
            decode_only(kc, vc)

    def step(i, ev=None):
        if not fused:
            return step_unfused(i, ev)
        if ev is not None:
            ev[0].record()
        decode_call(i)
        if ev is not None:
            ev[1].record()

    if fused and near_ties is not None:
        # the step's own encode of the new rows, counted once outside the timed region
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        kc0, vc0 = copies[0]
        _lib.vqkv_decode_append(mode, q, kc0, vc0, seq, kcb, vcb, s, out, ws, cap, max_len, new_k, new_v,
                                near_tie_count=cnt)
        near_ties["append_step"] = {"near_ties": int(cnt.item()), "codes": 2 * w.B * w.Hkv * (128 // w.d_sub)}
    if args.profile_fp16:
        fp16_profile_run(w, lens, dev, args.profile_fp16)
        return
    if args.profile_steps:
        for i in range(args.profile_steps):
            step(i)
        torch.cuda.synchronize()
        print(f"profile run: {args.profile_steps} steps of {w.name}, {n_splits} splits per KV head", flush=True)
        return

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        g_steps = GRAPH_STEPS - GRAPH_STEPS % n_copies if GRAPH_STEPS >= n_copies else n_copies
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(g_steps):
                step(i)
        # the timed region is exactly args.steps steps: whole graphs of g_steps
        # steps, then one graph of the remaining steps (back to back, each
        # step's kernels chained to the previous step's by programmatic
        # dependent launch inside a graph)
        rest_steps = args.steps % g_steps
        graph_rest = None
        if rest_steps:
            graph_rest = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_rest, stream=stream):
                for i in range(rest_steps):
                    step(i)
        # instrumented graph: events around every decode launch
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(g_steps)]
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, stream=stream):
            for i in range(g_steps):
                step(i, evs[i])
        graph.replay()
        torch.cuda.synchronize()

        def run_steps(k):
            for _ in range(k // g_steps):
                graph.replay()
            if k % g_steps:
                assert graph_rest is not None and k % g_steps == rest_steps
                graph_rest.replay()

        # time one replay to size the soak
        t0 = time.perf_counter()
        graph.replay()
        torch.cuda.synchronize()
        per_step = (time.perf_counter() - t0) / g_steps
        soak = max(1, int(SOAK_S / per_step)) // g_steps * g_steps or g_steps

        clocks = ClockSampler(local)
        clocks.start()
        run_steps(soak)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ms_total = e0.elapsed_time(e1)
        run_steps(soak)
        torch.cuda.synchronize()
        clk = clocks.stop()
        # dominant kernel: decode launch durations from the instrumented graph
        graph_ev.replay()
        torch.cuda.synchronize()
        dec_ms = [a.elapsed_time(b) for a, b in evs]
        dec_step_ms = sum(dec_ms) / len(dec_ms)
        # dominant kernel on its own: a graph of back-to-back decode launches
        # over the rotating copies, CUDA events around its replays
        graph_dec = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_dec, stream=stream):
            for i in range(g_steps):
                decode_call(i)
        graph_dec.replay()
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(1, int(0.5 / max(dec_step_ms * 1e-3 * g_steps, 1e-6)))
        d0.record(stream)
        for _ in range(reps):
            graph_dec.replay()
        d1.record(stream)
        torch.cuda.synchronize()
        dec_avg_ms = d0.elapsed_time(d1) / (reps * g_steps)
        unfused_ms = None
        if fused:
            # the same step as three calls (two encodes, then the decode), for comparison
            graph_unf = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_unf, stream=stream):
                for i in range(g_steps):
                    step_unfused(i)
            graph_unf.replay()
            torch.cuda.synchronize()
            d0.record(stream)
            for _ in range(reps):
                graph_unf.replay()
            d1.record(stream)
            torch.cuda.synchronize()
            unfused_ms = d0.elapsed_time(d1) / (reps * g_steps)

    ms_total = max_over_ranks(ms_total, world, dev)

    # end to end through the public API: pinned host buffers, copies inside the timed region
    q_host = q.cpu().pin_memory()
    nk_host = new_k.cpu().pin_memory()
    nv_host = new_v.cpu().pin_memory()
    o_host = torch.empty(tuple(out.shape), dtype=torch.float16).pin_memory()
    fp16 = None if args.profile_steps or M > 1 or BT else fp16_baseline(w, kv_fp16, lens, dev, stream)
    del kv_fp16
    e2e_steps = max(20, min(args.steps, 2000))
    with torch.cuda.stream(stream):
        def e2e_step(i):
            kc, vc = copies[i % n_copies]
            q.copy_(q_host, non_blocking=True)
            new_k.copy_(nk_host, non_blocking=True)
            new_v.copy_(nv_host, non_blocking=True)
            if fused:
                _lib.vqkv_decode_append(mode, q, kc, vc, seq, kcb, vcb, s, out, ws, cap, max_len, new_k, new_v)
            else:
                encode(0, new_k, pos, kc)
                encode(1, new_v, pos, vc)
                decode_only(kc, vc)
            o_host.copy_(out, non_blocking=True)
            stream.synchronize()
        for i in range(10):
            e2e_step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        e2e_s = (time.perf_counter() - t0) / e2e_steps

    tokens = int(lens.sum())
    ms_step = ms_total / args.steps
    value = replica_throughput(tokens, ms_step, world)
    alg = algorithmic_bytes(w, lens) + (M - 1) * 2 * w.B * w.Hq * 128 * 2   # q and O of every query
    if fused:
        alg += 2 * w.B * w.Hkv * (128 * 2 + 128 // 4)   # the new rows read, their codes written
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    achieved = alg / (dec_avg_ms * 1e-3) / 1e9
    traffic = profile_traffic()[0] if headline else None
    line = {
        "metric": METRIC if headline else f"decode-attn KV tokens/s and HBM GB/s ({w.name}, "
                                                 f"{BITS[w.mode]}-bit"
                                                 f"{f', {M} queries per sequence' if M > 1 else ''}"
                                                 f"{f', paged cache ({BT}-token blocks)' if BT else ''})",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 operands, f32 accumulate (u8 codes)", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "seq_len": int(lens[0]),
                   "bits": BITS[w.mode], "splits_per_kv_head": n_splits, "queries_per_sequence": M,
                   "paged_block_tokens": BT or None,
                   "step": ("vqkv_decode_append: 1 new K row + 1 new V row per sequence encoded into the cache "
                            "and attended in the same kernel" if fused else
                            "vqkv_encode (1 new K row per sequence), vqkv_encode (V), vqkv_decode_attn"),
                   "cache": ("encoded on the GPU by vqkv_encode from seeded synthetic K/V" if headline
                             else "seeded uniform codes (decode cost does not depend on code values)"),
                   "l2": f"{n_copies} rotating cache copies ({n_copies * cache_bytes / 1e6:.0f} MB > "
                         f"{l2 / 1e6:.0f} MB L2)",
                   "timing": (f"timed region = exactly {args.steps} steps: {args.steps // g_steps} replays of a "
                              f"CUDA graph of {g_steps} back-to-back steps"
                              + (f" + one graph of {args.steps % g_steps} steps" if args.steps % g_steps else "")
                              + "; CUDA events on the launch stream"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": "decode_vq15_kernel" if w.mode == synth.MODE_VQ15 else "decode_vq2_kernel",
                     "launch_ms": dec_avg_ms, "algorithmic_bytes": alg,
                     "how": f"graph of {g_steps} back-to-back {'vqkv_decode_append' if fused else 'vqkv_decode_attn'} "
                            f"calls ({dec_kernels} kernel(s) each) over the rotating cache copies, CUDA events on "
                            "the launch stream",
                     "in_step_launch_ms": dec_step_ms},
        "clocks": clk,
        "e2e": {"value": world * tokens / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": q.numel() * 2 + new_k.numel() * 2 + new_v.numel() * 2,
                "d2h_bytes_per_step": out.numel() * 2,
                "how": "public binding per step: H2D q and new K/V rows, "
                       + ("vqkv_decode_append" if fused else "2 encodes, decode") + ", D2H O, sync"},
        "gpu_launches": (dec_kernels if fused else 2 + dec_kernels) * args.steps,
    }
    if near_ties is not None:
        line["near_ties"] = near_ties
    if unfused_ms is not None:
        line["unfused_step_ms"] = unfused_ms
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if fp16 is not None:
        fp16["vq_decode_speedup"] = fp16["launch_us"] / (dec_avg_ms * 1e3)
        line["fp16_kv_decode"] = fp16
    if args.workload == 4 and not args.profile_steps:
        line["encode_prefill"] = encode_prefill_bench(w, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def encode_prefill_bench(w, dev, reps=3):
    """vqkv_encode of the whole prefill (B x Hkv x prefill rows) for K and V in
    both bit-widths; keys are Gaussian with the workload's outlier channels,
    made on the GPU; codebooks calibrated on the host."""
    import torch
    from vector_quantized_bit_gb300 import _lib
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + w.config_id + 31)
    res = {}
    for mode in (synth.MODE_VQ2, synth.MODE_VQ15):
        wm = w.with_mode(mode)
        s_h, kcb_h, vcb_h = host_calibration(wm)
        s, kcb, vcb = (torch.from_numpy(a).to(dev) for a in (s_h, kcb_h, vcb_h))
        codes = torch.zeros((w.B, w.Hkv, _lib.vqkv_code_bytes(mode, w.cap_len)), dtype=torch.uint8, device=dev)
        pos = torch.zeros(w.B, dtype=torch.int32, device=dev)
        out = {}
        for role in (0, 1):
            x = torch.randn((w.B, w.Hkv, w.prefill, 128), generator=gen, device=dev)
            if role == 0:
                for h in range(w.Hkv):
                    ch, sc = synth.outlier_channels(w, h)
                    x[:, h, :, torch.from_numpy(ch).to(dev)] *= torch.from_numpy(sc).to(dev)
            x = x.half()
            call = lambda: _lib.vqkv_encode(mode, role, x, pos, s if role == 0 else None,  # noqa: E731
                                            kcb if role == 0 else vcb, codes, w.cap_len)
            cnt = torch.zeros(1, dtype=torch.int64, device=dev)
            _lib.vqkv_encode(mode, role, x, pos, s if role == 0 else None, kcb if role == 0 else vcb, codes,
                             w.cap_len, near_tie_count=cnt)   # untimed: the near-tie count of this encode
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            out["K" if role == 0 else "V"] = {"ms": ms, "rows_per_s": w.B * w.Hkv * w.prefill / (ms * 1e-3),
                                              "near_ties": int(cnt.item()),
                                              "codes": w.B * w.Hkv * w.prefill * (128 // wm.d_sub)}
            del x
        if mode == synth.MODE_VQ15:
            # ALU floor: one fp32 compare per (subvector, candidate) on every lane;
            # tensor floor: the screening MMAs (K = 16 per candidate) at the measured bf16/fp16 rate
            props = torch.cuda.get_device_properties(dev)
            try:
                peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
            except (OSError, ValueError):
                peaks = {}
            mhz = peaks.get("sm_max_mhz") or 2070.0
            cand = w.B * w.Hkv * w.prefill * (128 // wm.d_sub) * wm.entries
            alu_peak = props.multi_processor_count * 128 * mhz * 1e6
            tflops = peaks.get("bf16_tflops") or 1900.0
            best_ms = min(out["K"]["ms"], out["V"]["ms"])
            out["roofline"] = {"bound": "alu", "unit": "candidates/s", "achieved": cand / (best_ms * 1e-3),
                               "peak": alu_peak, "frac": cand / (best_ms * 1e-3) / alu_peak,
                               "peak_source": f"{props.multi_processor_count} SMs x 128 fp32 lanes x {mhz:.0f} MHz, "
                                              "one compare per candidate",
                               "tensor_floor_ms": 2 * cand * 16 / (tflops * 1e12) * 1e3,
                               "alu_floor_ms": cand / alu_peak * 1e3}
        res["2-bit" if mode == 0 else "1.5-bit"] = out
    return res


def encode_profile_run(mode, B=4, calls=3):
    """calls x vqkv_encode of the key prefill of B sequences of the
    Mistral-shaped workload (B x 8 KV heads x 16,384 rows, 134 MB of fp16
    rows at B = 4, more than L2), keys made on the GPU as in
    encode_prefill_bench; prints the mean call time (CUDA events)."""
    import torch
    from vector_quantized_bit_gb300 import _build, _lib
    _build.build()
    dev = torch.device("cuda")
    w = synth.WORKLOADS[4].with_mode(mode).scaled(B=B)
    s_h, kcb_h, _ = host_calibration(w)
    s, kcb = torch.from_numpy(s_h).to(dev), torch.from_numpy(kcb_h).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + w.config_id + 31)
    x = torch.randn((w.B, w.Hkv, w.prefill, 128), generator=gen, device=dev)
    for h in range(w.Hkv):
        ch, sc = synth.outlier_channels(w, h)
        x[:, h, :, torch.from_numpy(ch).to(dev)] *= torch.from_numpy(sc).to(dev)
    x = x.half()
    codes = torch.zeros((w.B, w.Hkv, _lib.vqkv_code_bytes(mode, w.cap_len)), dtype=torch.uint8, device=dev)
    pos = torch.zeros(w.B, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    _lib.vqkv_encode(mode, 0, x, pos, s, kcb, codes, w.cap_len)   # warm-up (module load, attributes)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls):
        _lib.vqkv_encode(mode, 0, x, pos, s, kcb, codes, w.cap_len, near_tie_count=cnt)
    e1.record()
    torch.cuda.synchronize()
    rows = w.B * w.Hkv * w.prefill
    ms = e0.elapsed_time(e1) / calls
    print(json.dumps({"encode_profile": {"mode": mode, "rows": rows, "calls": calls, "ms_per_call": ms,
                                         "rows_per_s": rows / (ms * 1e-3), "near_ties_all_calls": int(cnt.item())}}),
          flush=True)


def fp16_profile_run(w, lens, dev, n):
    """n eager vqkv_decode_attn_fp16 calls over seeded Gaussian fp16 K/V."""
    import torch
    from vector_quantized_bit_gb300 import _lib
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + w.config_id + 17)
    k = torch.randn((w.B, w.Hkv, w.cap_len, 128), generator=gen, device=dev, dtype=torch.float16)
    v = torch.randn((w.B, w.Hkv, w.cap_len, 128), generator=gen, device=dev, dtype=torch.float16)
    q = torch.from_numpy(synth.queries(w)).to(dev)
    seq = torch.from_numpy(lens.astype(np.int32)).to(dev)
    out = torch.empty((w.B, w.Hq, 128), dtype=torch.float16, device=dev)
    max_len = int(lens.max())
    ws = _lib.fp16_decode_workspace(w.B, w.Hq, w.Hkv, w.cap_len, max_len, device=dev)
    for _ in range(n):
        _lib.vqkv_decode_attn_fp16(q, k, v, seq, out, ws, max_len)
    torch.cuda.synchronize()
    print(f"fp16 profile run: {n} decodes of {w.name}", flush=True)


def fp16_baseline(w, kv, lens, dev, stream, launches=60, reps=5):
    """The same decode over a plain fp16 K/V cache (vqkv_decode_attn_fp16):
    average launch time from CUDA events around a graph of launches.  The fp16
    cache is larger than L2, so consecutive launches stream from HBM.  kv:
    the workload's host K/V rows, or None for seeded Gaussian rows made on the
    GPU."""
    import torch
    from vector_quantized_bit_gb300 import _lib
    if kv is not None:
        k = torch.from_numpy(np.stack([kv[h][0] for h in range(w.Hkv)])[None]).to(dev)
        v = torch.from_numpy(np.stack([kv[h][1] for h in range(w.Hkv)])[None]).to(dev)
    else:
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed * 1000 + w.config_id + 17)
        k = torch.randn((w.B, w.Hkv, w.cap_len, 128), generator=gen, device=dev, dtype=torch.float16)
        v = torch.randn((w.B, w.Hkv, w.cap_len, 128), generator=gen, device=dev, dtype=torch.float16)
    q = torch.from_numpy(synth.queries(w)).to(dev)
    seq = torch.from_numpy(lens.astype(np.int32)).to(dev)
    out = torch.empty((w.B, w.Hq, 128), dtype=torch.float16, device=dev)
    max_len = int(lens.max())
    ws = _lib.fp16_decode_workspace(w.B, w.Hq, w.Hkv, w.cap_len, max_len, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(5):
            _lib.vqkv_decode_attn_fp16(q, k, v, seq, out, ws, max_len)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(launches):
                _lib.vqkv_decode_attn_fp16(q, k, v, seq, out, ws, max_len)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (launches * reps)
    tokens = int(lens.sum())
    nbytes = tokens * w.Hkv * 2 * 128 * 2 + 2 * q.numel() * 2   # K and V rows read, q read, O written
    return {"launch_us": us, "tokens_per_s": tokens / (us * 1e-6), "GB_per_s": nbytes / us / 1e3,
            "algorithmic_bytes": nbytes, "kernel": "decode_fp16_kernel",
            "how": "graph of 60 launches x 5 replays, CUDA events; fp16 K/V of the same synthetic cache"}


# ------------------------------------------------------------- calibration stage

CALIB_POINTS = 65536          # sampled subvectors a codebook is trained on
CALIB_ITERS = 20              # Lloyd steps after k-means++
CALIB_SHAPES = ((256, 4), (4096, 8))


def _calib_rows(w, kvh=0):
    """Key rows (fp16 [L][128]) of one KV head of the workload, as generated for its cache."""
    return synth.keys(w, 0, kvh, 0, w.seq_len)


def _time_cuda(fn, reps, warm=2):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _sample_points(xt, dim, n_points, rng):
    """n_points subvectors of dim channels from randomly chosen rows of xt (fp32 [L][128], device)."""
    import torch
    rows = n_points * dim // 128
    idx = np.sort(rng.choice(xt.shape[0], size=rows, replace=False))
    return xt[torch.from_numpy(idx).to(xt.device)].reshape(-1, dim).contiguous()


def run_calibration(args):
    """The offline stage on one KV head of the Llama-shaped workload: key
    smoothing over its 196,608 rows, the smooth + rotate transform, and
    K-Means training (k-means++ then 20 Lloyd steps) of a 256 x 4 and a
    4096 x 8 codebook from 65,536 sampled subvectors.  Headline: the Lloyd
    assignment rate of the 4096 x 8 codebook (distance evaluations per second)
    against the fp32 ALU roofline."""
    import torch
    from vector_quantized_bit_gb300 import _lib
    w = synth.WORKLOADS[1]
    dev = torch.device("cuda")
    rows = torch.from_numpy(_calib_rows(w)).to(dev)
    L = rows.shape[0]
    s = torch.empty(128, dtype=torch.float32, device=dev)
    xt = torch.empty((L, 128), dtype=torch.float32, device=dev)
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    t_smooth = _time_cuda(lambda: _lib.vqkv_smoothing(rows, s), 20)
    t_xf = _time_cuda(lambda: _lib.vqkv_calib_transform(rows, xt, s_pre=s, rotate=True), 20)
    rng = np.random.default_rng(0)
    shapes = {}
    for k, dim in CALIB_SHAPES:
        pts = _sample_points(xt, dim, CALIB_POINTS, rng)
        u = torch.from_numpy(rng.random(k).astype(np.float32)).to(dev)
        cent = torch.empty((k, dim), dtype=torch.float32, device=dev)
        cent2 = torch.empty_like(cent)
        seeds = torch.empty(k, dtype=torch.int32, device=dev)
        idx = torch.empty(CALIB_POINTS, dtype=torch.int32, device=dev)
        ws = _lib.kmeans_workspace(CALIB_POINTS, dim, k)
        t_seed = _time_cuda(lambda: _lib.vqkv_kmeans_seed(pts, u, cent, seeds, workspace=ws), 3, 1)
        t_assign = _time_cuda(lambda: _lib.vqkv_kmeans_assign(pts, cent, idx), 50)
        t_update = _time_cuda(lambda: _lib.vqkv_kmeans_update(pts, idx, cent, cent2), 50)
        t_train = _time_cuda(lambda: _lib.vqkv_kmeans(pts, u, cent, CALIB_ITERS, workspace=ws), 3, 1)
        evals = CALIB_POINTS * k
        shapes[f"{k}x{dim}"] = {"seed_ms": t_seed, "assign_us": t_assign * 1e3, "update_us": t_update * 1e3,
                                "train_ms": t_train, "assign_evals_per_s": evals / (t_assign * 1e-3)}
    clocks = clk.stop()
    props = torch.cuda.get_device_properties(dev)
    mhz = clocks.get("sm_max_mhz") or 2070.0
    ops = 2 * 8 + 3   # per evaluation at dim 8: 8 sub, 1 mul, 7 fma, compare + 2 selects
    peak = props.multi_processor_count * 128 * mhz * 1e6 / ops
    head = shapes["4096x8"]
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import kmeans_oracle as ko
        p_np = _sample_points(xt, 8, CALIB_POINTS, np.random.default_rng(1)).cpu().numpy()[:1024]
        c_np = p_np[:512].copy()
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            ko.assign(p_np, c_np)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps * 1024 * 512 / dt, "unit": "distance evals/s", "cores": 1, "kind": "oracle",
               "sample": f"oracle assignment of 1024 points x 512 centroids (dim 8), {reps} passes, {dt:.1f} s"}
    print(json.dumps({
        "metric": "K-Means Lloyd assignment distance evaluations/s (4096 x 8 codebook, 65,536 subvectors)",
        "value": head["assign_evals_per_s"], "unit": "evals/s", "higher_is_better": True, "n_gpus": 1,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "calibration_llama8b_kvh0_l196608", "rows": L, "points": CALIB_POINTS,
                   "iters": CALIB_ITERS, "l2": "points (2 MB) stay in L2: the assignment is ALU-bound"},
        "roofline": {"bound": "alu", "achieved": head["assign_evals_per_s"] / 1e12, "peak": peak / 1e12,
                     "unit": "T evals/s", "frac": head["assign_evals_per_s"] / peak, "traffic": None,
                     "peak_source": f"{props.multi_processor_count} SMs x 128 fp32 lanes x {mhz:.0f} MHz / "
                                    f"{ops} ops per evaluation"},
        "stages": {"smoothing_us": t_smooth * 1e3, "smoothing_GB_per_s": L * 256 / (t_smooth * 1e-3) / 1e9,
                   "transform_us": t_xf * 1e3, "transform_GB_per_s": L * (256 + 512) / (t_xf * 1e-3) / 1e9,
                   **{f"kmeans_{key}": val for key, val in shapes.items()}},
        "cpu_baseline": cpu, "clocks": clocks}))


ABLATION_VARIANTS = ("none", "smooth", "hadamard", "smooth_hadamard", "hadamard_smooth")


def run_ablation(args):
    """Codebook utilisation and key reconstruction error of the five key
    transforms, for the 256 x 4 and 4096 x 8 codebooks, on one KV head of the
    Llama-shaped outlier keys (196,608 rows).  On the GPU: smoothing, the
    transform, k-means++ + 20 Lloyd steps on 65,536 sampled subvectors, and
    the assignment of every subvector of every row.  On the host (measurement
    only): the reconstruction from the codes, its relative error against the
    original keys, and the relative error of q.k scores for 16 random
    queries."""
    import scipy.linalg
    import torch
    from vector_quantized_bit_gb300 import _lib
    w = synth.WORKLOADS[1]
    dev = torch.device("cuda")
    k_np = _calib_rows(w)
    rows = torch.from_numpy(k_np).to(dev)
    L = rows.shape[0]
    k64 = k_np.astype(np.float64)
    hn = scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128.0)
    q = np.random.default_rng(5).standard_normal((16, 128))
    scores = k64 @ q.T
    out = {}
    for variant in ABLATION_VARIANTS:
        xt = torch.empty((L, 128), dtype=torch.float32, device=dev)
        s = torch.empty(128, dtype=torch.float32, device=dev)
        if variant == "none":
            _lib.vqkv_calib_transform(rows, xt)
        elif variant in ("smooth", "smooth_hadamard"):
            _lib.vqkv_smoothing(rows, s)
            _lib.vqkv_calib_transform(rows, xt, s_pre=s, rotate=variant == "smooth_hadamard")
        elif variant == "hadamard":
            _lib.vqkv_calib_transform(rows, xt, rotate=True)
        else:
            rot = torch.empty_like(xt)
            _lib.vqkv_calib_transform(rows, rot, rotate=True)
            _lib.vqkv_smoothing(rot, s)
            _lib.vqkv_calib_transform(rot, xt, s_post=s)
        s_np = s.cpu().numpy().astype(np.float64)
        res = {}
        for k, dim in CALIB_SHAPES:
            rng = np.random.default_rng(k)
            pts = _sample_points(xt, dim, CALIB_POINTS, rng)
            u = torch.from_numpy(rng.random(k).astype(np.float32)).to(dev)
            cent = torch.empty((k, dim), dtype=torch.float32, device=dev)
            cb = torch.empty((k, dim), dtype=torch.float16, device=dev)
            _lib.vqkv_kmeans(pts, u, cent, CALIB_ITERS, codebook=cb)
            allp = xt.reshape(-1, dim)
            codes = torch.empty(allp.shape[0], dtype=torch.int32, device=dev)
            _lib.vqkv_kmeans_assign(allp, cb.float().contiguous(), codes)
            c = codes.cpu().numpy()
            rec = cb.float().cpu().numpy().astype(np.float64)[c].reshape(L, 128)
            if variant == "smooth":
                rec = rec * s_np
            elif variant == "hadamard":
                rec = rec @ hn.T
            elif variant == "smooth_hadamard":
                rec = (rec @ hn.T) * s_np
            elif variant == "hadamard_smooth":
                rec = (rec * s_np) @ hn.T
            err = rec - k64
            counts = np.bincount(c, minlength=k).astype(np.float64)
            pr = counts[counts > 0] / counts.sum()
            res[f"{k}x{dim}"] = {
                "key_rel_mse": float((err * err).sum() / (k64 * k64).sum()),
                "score_rel_err": float(np.linalg.norm(rec @ q.T - scores) / np.linalg.norm(scores)),
                "used_fraction": float((counts > 0).mean()), "code_entropy_bits": float(-(pr * np.log2(pr)).sum())}
        out[variant] = res
    print(json.dumps({"metric": "key transform ablation: codebook utilisation and reconstruction error",
                      "data": "synthetic", "config": {"workload": "llama8b_kvh0_l196608_outlier_keys", "rows": L,
                                                      "points": CALIB_POINTS, "iters": CALIB_ITERS},
                      "ablation": out}))


def main():
    args = parse()
    if args.profile_encode >= 0:
        encode_profile_run(args.profile_encode)
    elif args.impl == "reference":
        run_reference(args)
    elif args.calib:
        run_calibration(args)
    elif args.ablation:
        run_ablation(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
