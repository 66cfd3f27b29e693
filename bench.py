#!/usr/bin/env python3
"""Bench: paged GQA decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload cfg2]
                    [--impl ours|reference]

A step is one pass of the hot path over one batch: for every layer, the append
of the new token's key/value and the decode attention over the paged cache
(plus verify and greedy acceptance for the speculative workload); by default
the append runs inside the attention launch (gqa_append_decode_attention),
with --unfused as separate kv_append launches.
The default workload is the one the bandwidth target (>= 75 % of peak HBM on the
long-context batches) is stated for: the ragged batch of B=256 sequences,
N=32, K=8, H=128, bf16, log-normal contexts (median 2048, clipped to
[1, 32768]), shuffled block tables, append of one token then decode attention.
The other workloads (--workload cfg1|cfg2|cfg3|cfg5) are measured the same way.  The step's
library calls are captured once into CUDA graphs and replayed, so launch overhead does not hide the kernels; the attention graph is
bracketed by its own events, which gives the attention kernel's average launch
duration live inside the timed region.

Multi-GPU: every rank runs its own replica of the workload (the path has no
exchange step); value = all ranks' bytes / the slowest rank's time.  Ranks come
from torchrun, or, with --gpus N and no torchrun environment, from N processes
this script spawns itself.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention achieved HBM GB/s (% of GB300 peak) and attention tokens/sec"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    # Default: the workload the metric's bandwidth target is quoted on -- the
    # long-context ragged batch (B=256, log-normal contexts, 3.5 GB per step).
    ap.add_argument("--workload", default="cfg4",
                    choices=["cfg1", "cfg2", "cfg3", "cfg4", "cfg5", "hybrid", "tree"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=None,
                    help="a batch of B sequences drawn by the same workload recipe, for "
                         "small profiling captures")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the oracle CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the oracle check of the timed step's outputs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--accept", default="greedy", choices=["greedy", "sampled"],
                    help="acceptance step of a verify workload: greedy longest prefix over "
                         "logits, or stochastic acceptance (speculative sampling) over "
                         "probabilities")
    ap.add_argument("--kv", default="same", choices=["same", "int8", "e4m3"],
                    help="KV cache element type: q's dtype, or one-byte int8 / e4m3 codes with "
                         "a per-row fp32 scale (quantized append + attention, H = 128)")
    ap.add_argument("--engine", default="auto", choices=["auto", "warp", "direct", "tmem"],
                    help="attention kernel: picked by shape (auto), the persistent warp-level "
                         "mma.sync kernel, the direct one (one CTA per sequence and KV head), "
                         "or the tensor-memory (tcgen05) kernel")
    ap.add_argument("--unfused", action="store_true",
                    help="separate kv_append launches instead of the append fused into "
                         "the attention launch")
    args = ap.parse_args(argv)
    if args.workload == "tree" and args.accept == "sampled":
        ap.error("stochastic acceptance over a draft tree is not built (--accept greedy)")
    return args


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---- accounting ------------------------------------------------------------------
def step_bytes(w, kv="same"):
    from gqa_decode_attention_02_gb300 import analytic as A

    e = 2
    q8 = {} if kv == "same" else {"kv_elem_bytes": 1, "row_scale_bytes": 4}
    ctx = w.context_lens.cpu().numpy()
    # mean over the layers (they differ only in their local-attention window)
    attn = sum(A.attention_algorithmic_bytes(ctx, w.T, w.N, w.K, w.H, e, window=w.window(l), **q8)
               for l in range(w.layers)) // w.layers
    if not w.appended:
        app = 0
    elif kv == "same":
        app = A.kv_append_bytes(w.B, w.T, w.K, w.H, e)
    else:
        app = A.kv_append_quant_bytes(w.B, w.T, w.K, w.H, e)
    acc = A.accept_bytes(w.B, w.T, w.logits.shape[-1]) if w.logits is not None else 0
    return attn, app, acc


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def kernel_source_hash(engine="warp"):
    """Hash of a kernel's source code with comments and whitespace removed, so
    that a comment edit does not invalidate counters taken on the same code."""
    import re

    h = hashlib.sha256()
    files = ("attention.cu", "ptx.cuh") if engine in ("warp", "direct") else (
        "attention_tc.cu", "tcgen05.cuh", "ptx.cuh")
    for f in files:
        src = open(os.path.join(ROOT, "gqa_decode_attention_02_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, engine="warp"):
    """dram bytes per attention launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    name = {"warp": f"attention_{workload}", "direct": f"direct_attention_{workload}"}.get(
        engine, f"tc_attention_{workload}")
    p = os.path.join(ROOT, "profiles", f"{name}_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != kernel_source_hash(engine):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def combine_ranks(step_ms: float, bytes_step: int, world: int, device):
    """Whole-job figure over replicas: every rank processed `bytes_step` per
    step; the job's step time is the slowest rank's.  Returns (max step ms,
    GB/s of all ranks' bytes).  Uses the default process group when world > 1."""
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([step_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    return step_ms, world * bytes_step / (step_ms * 1e-3) / 1e9


# ---- clocks ------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", index, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        import statistics

        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_index_for_smi(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[local_rank].strip()
    return str(local_rank)


# ---- CPU oracle timing --------------------------------------------------------------
def _oracle_layer_inputs(w, layer, quant=None):
    """CPU copies of one layer's inputs with the new tokens already appended by
    the oracle (untimed: the timed part is the oracle's attention).  quant =
    (kv, k codes, v codes, k scales, v scales) per layer (CPU): a one-byte
    cache, returned as (q, codes_k, codes_v, scales_k, scales_v)."""
    import numpy as np
    import torch

    import oracle

    q = w.q[layer].cpu()
    if quant is not None:
        kv, ck, cv, sk, sv = quant
        out = oracle.kv_append_quant(w.k_new[layer].cpu(), w.v_new[layer].cpu(), ck[layer],
                                     cv[layer], sk[layer], sv[layer], w.block_tables.cpu(),
                                     w.context_lens.cpu(), w.dtype, kv)
        return (q,) + tuple(out[:4])
    kc, vc = w.k_cache[layer].cpu(), w.v_cache[layer].cpu()
    if w.appended:
        kb, vb, _ = oracle.kv_append(w.k_new[layer].cpu(), w.v_new[layer].cpu(), kc, vc,
                                     w.block_tables.cpu(), w.context_lens.cpu())
        kc = torch.from_numpy(kb.view(np.int16)).view(w.torch_dtype)
        vc = torch.from_numpy(vb.view(np.int16)).view(w.torch_dtype)
    return q, kc, vc


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                name = line.split(":", 1)[1].strip()
                if name and not name.isdigit():
                    vendor = [l.split(":", 1)[1].strip() for l in out.splitlines()
                              if l.startswith("Vendor ID")]
                    return f"{vendor[0]} {name}" if vendor else name
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform

    return platform.processor() or platform.machine()


def oracle_sample(w, budget_s, quant=None, nthreads=0, inputs=None):
    """Time the oracle's attention (as it stands; nthreads=0: all host threads)
    on a bounded sample of the workload: (layer, 8-sequence chunk) units in
    order until the budget is spent.  `inputs` caches each layer's oracle
    inputs across calls.  Returns (GB/s of algorithmic attention bytes,
    seconds, description, threads)."""
    import numpy as np

    import oracle
    from gqa_decode_attention_02_gb300 import analytic as A

    oracle.build()
    ctx = w.context_lens.cpu().numpy()
    tables, lens = w.block_tables.cpu(), w.context_lens.cpu()
    done_bytes, spent, units, seqs = 0, 0.0, 0, 0
    q8 = {} if quant is None else {"kv_elem_bytes": 1, "row_scale_bytes": 4}
    inputs = {} if inputs is None else inputs
    for layer in range(w.layers):
        if layer not in inputs:
            inputs.clear()
            inputs[layer] = _oracle_layer_inputs(w, layer, quant)
        ins = inputs[layer]
        q, kc, vc = ins[:3]
        qa = {} if quant is None else {"kv": quant[0], "k_scale": ins[3], "v_scale": ins[4]}
        for s0 in range(0, w.B, 8):
            bl = np.arange(s0, min(w.B, s0 + 8), dtype=np.int32)
            t0 = time.perf_counter()
            oracle.attention(q, kc, vc, tables, lens, w.dtype, b_list=bl, window=w.window(layer),
                             tree_mask=w.tree_mask(), nthreads=nthreads, **qa)
            spent += time.perf_counter() - t0
            done_bytes += A.attention_algorithmic_bytes(ctx[bl], w.T, w.N, w.K, w.H, 2,
                                                        window=w.window(layer), **q8)
            units += 1
            seqs += len(bl)
            if spent >= budget_s:
                break
        if spent >= budget_s:
            break
    thr = nthreads if nthreads > 0 else oracle.num_threads()
    desc = (f"oracle attention over {seqs} of the {w.layers * w.B} (layer, sequence) pairs "
            f"({units} chunks of <= 8 sequences); fp64 C, {thr} thread(s)")
    return done_bytes / spent / 1e9, spent, desc, thr


def parity_sample(w, outs, quant=None, inputs=None, n_seq=8, seed=1234):
    """Check the timed step's attention outputs against the oracle on a seeded
    sample of sequences (the shortest and the longest always included) of the
    first and last layer, outside the timed region.  Returns the record."""
    import numpy as np

    import oracle

    ctx = w.context_lens.cpu().numpy()
    rng = np.random.default_rng(seed)
    pick = {int(np.argmin(ctx)), int(np.argmax(ctx))}
    rest = [b for b in range(w.B) if b not in pick]
    pick |= set(int(b) for b in rng.choice(rest, size=min(len(rest), n_seq - len(pick)),
                                            replace=False)) if rest else set()
    bl = np.array(sorted(pick), np.int32)
    tol = {"f16": 2e-3, "bf16": 1e-2}[w.dtype]
    mant = 10 if w.dtype == "f16" else 7
    worst, ok = 0.0, True
    inputs = {} if inputs is None else inputs
    layers = sorted({0, w.layers - 1})
    for layer in layers:
        if layer not in inputs:
            inputs.clear()
            inputs[layer] = _oracle_layer_inputs(w, layer, quant)
        ins = inputs[layer]
        qa = {} if quant is None else {"kv": quant[0], "k_scale": ins[3], "v_scale": ins[4]}
        ref, err = oracle.attention(ins[0], ins[1], ins[2], w.block_tables.cpu(),
                                    w.context_lens.cpu(), w.dtype, b_list=bl,
                                    window=w.window(layer), tree_mask=w.tree_mask(), **qa)
        got = outs[layer][torch_index(bl, outs[layer].device)].double().cpu().numpy()
        d = np.abs(got - ref)
        a = np.abs(ref)
        one_ulp = np.exp2(np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))),
                                     -14 if w.dtype == "f16" else -126) - mant)
        ok &= bool(np.isfinite(got).all() and (d <= np.maximum(tol, one_ulp)).all()
                   and (err == 0).all())
        worst = max(worst, float(d.max()) if d.size else 0.0)
    return {"max_abs_err": worst, "parity_pass": ok, "tol": tol,
            "rule": "|gpu - oracle| <= max(tol, one ulp of the oracle value in the dtype)",
            "sample": f"sequences {bl.tolist()} (shortest and longest included) of layers "
                      f"{layers}, the timed step's outputs vs the fp64 oracle"}


def torch_index(bl, device):
    import torch

    return torch.as_tensor(bl, dtype=torch.long, device=device)


def hold_gpu(steps: int) -> None:
    """Keep the GPU busy (a spin kernel, before the first step's events) while
    the host enqueues the timed steps, so that every step's events measure
    GPU time only: a short step (tens of microseconds) would otherwise also
    count the host's launch latency whenever the host falls behind."""
    import torch

    torch.cuda._sleep(int(2.0e9 * max(2e-3, steps * 3e-4)))  # ~cycles at ~2 GHz


# ---- our arm -----------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import gqa_decode_attention_02_gb300 as gq
    from gqa_decode_attention_02_gb300 import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    w = workloads.make(args.workload, device=dev, B=args.batch)
    L = w.layers
    attn_fn = gq.decode_attention if w.T == 1 else gq.verify_attention
    fused_fn = gq.append_decode_attention if w.T == 1 else gq.append_verify_attention
    q8 = args.kv != "same"
    fused = w.appended and not args.unfused and not q8  # no fused one-byte append
    if q8:
        # Input preparation (outside the timed region): the cached part of each
        # layer's cache as one-byte codes with per-row scales, quantized here
        # with plain torch ops (absmax rule); the step's own append writes the
        # new tokens with the library.
        qk, qv, sk, sv = [], [], [], []
        for l in range(L):
            for src, codes, scales in ((w.k_cache[l], qk, sk), (w.v_cache[l], qv, sv)):
                x = torch.nan_to_num(src.float(), nan=0.0)
                amax = x.abs().amax(-1)  # [NB, 16, K]
                sc = amax / (127.0 if args.kv == "int8" else 448.0)
                y = x / sc.clamp_min(1e-30)[..., None]
                if args.kv == "int8":
                    c = y.round().clamp(-128, 127).to(torch.int8).view(torch.uint8)
                else:
                    c = y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
                codes.append(c.contiguous())
                scales.append(sc.permute(0, 2, 1).contiguous())
                del x, y
            w.k_cache[l] = w.v_cache[l] = None  # the 2-byte caches are not used
        torch.cuda.empty_cache()
        quant_cpu = None  # CPU copies for the oracle: parity and the CPU baseline
        if rank == 0 and (not args.no_parity or (world == 1 and not args.no_cpu_baseline)):
            quant_cpu = (args.kv, [c.cpu() for c in qk], [c.cpu() for c in qv],
                         [c.cpu() for c in sk], [c.cpu() for c in sv])
        attn_q8 = gq.decode_attention_quant if w.T == 1 else gq.verify_attention_quant
    ws_bytes = gq.attention_workspace_size(w.q[0], qk[0] if q8 else w.k_cache[0],
                                           w.block_tables)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    outs = [torch.empty_like(q) for q in w.q]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    has_acc = w.logits is not None
    sampled = has_acc and args.accept == "sampled"
    if has_acc:
        ctx_scratch = w.context_lens.clone()
        acc_ws = torch.zeros(gq._lib.lib().gqa_accept_workspace_size(w.B, w.T),
                             dtype=torch.uint8, device=dev)
        acc_out = torch.empty(w.B, dtype=torch.int32, device=dev)
        nxt_out = torch.empty(w.B, dtype=torch.int32, device=dev)
        V = w.logits.shape[-1]
    if sampled:
        sin = workloads.sampling_inputs(w.B, w.T, V, seed=workloads.SPECS[args.workload]["seed"]
                                        + 1000, device=dev)

    tm = w.tree_mask()
    tree_t = None if tm is None else torch.from_numpy(tm.view(np.int64)).to(dev)
    extra = {} if tree_t is None else {"tree_mask": tree_t}
    # a draft tree: acceptance walks the tree and the kept branch's cache rows
    # are compacted behind its root (every layer's caches)
    tree_acc = has_acc and not sampled and tree_t is not None
    if tree_acc:
        parents_d = torch.as_tensor(w.parents()).to(dev)
        path_out = torch.empty((w.B, w.T - 1), dtype=torch.int32, device=dev)

    def do_append():
        if w.appended and not fused:
            for l in range(L):
                if q8:
                    gq.kv_append_quant(w.k_new[l], w.v_new[l], qk[l], qv[l], sk[l], sv[l],
                                       w.block_tables, w.context_lens, kv=args.kv, status=st,
                                       pdl=True)
                else:
                    gq.kv_append(w.k_new[l], w.v_new[l], w.k_cache[l], w.v_cache[l],
                                 w.block_tables, w.context_lens, status=st, pdl=True)

    def do_attn():
        for l in range(L):
            # early_kv: the previous kernel here is the previous layer's attention
            # (or, across the graph boundary, fully ordered), which writes neither
            # the tables, the lengths nor any cache position below ctx - T.
            if q8:
                attn_q8(w.q[l], qk[l], qv[l], sk[l], sv[l], w.block_tables, w.context_lens,
                        kv=args.kv, out=outs[l], workspace=ws, status=st, pdl=True,
                        early_kv=True, window=w.window(l), **extra)
            elif fused:
                fused_fn(w.q[l], w.k_new[l], w.v_new[l], w.k_cache[l], w.v_cache[l],
                         w.block_tables, w.context_lens, out=outs[l], workspace=ws, status=st,
                         pdl=True, early_kv=True, window=w.window(l), engine=args.engine,
                         **extra)
            else:
                attn_fn(w.q[l], w.k_cache[l], w.v_cache[l], w.block_tables, w.context_lens,
                        out=outs[l], workspace=ws, status=st, pdl=True, early_kv=True,
                        window=w.window(l), engine=args.engine, **extra)

    def do_acc():
        if sampled:
            gq.accept_sampled(sin.q, sin.p, sin.draft, sin.uniforms, ctx_scratch,
                              accepted=acc_out, next_token=nxt_out, status=st)
        elif tree_acc:
            gq.accept_tree(w.logits, w.draft, parents_d, ctx_scratch, accepted=acc_out,
                           next_token=nxt_out, path=path_out, status=st, workspace=acc_ws)
            for l in range(L):
                if q8:
                    gq.kv_compact(qk[l], qv[l], w.block_tables, ctx_scratch, path_out, acc_out,
                                  k_scale=sk[l], v_scale=sv[l], kv=args.kv, status=st, pdl=True)
                else:
                    gq.kv_compact(w.k_cache[l], w.v_cache[l], w.block_tables, ctx_scratch,
                                  path_out, acc_out, status=st, pdl=True)
        elif has_acc:
            gq.accept_prefix(w.logits, w.draft, ctx_scratch, accepted=acc_out,
                             next_token=nxt_out, status=st, workspace=acc_ws)

    # eager warm-up (also builds the launch plans), then capture
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        do_append(), do_attn(), do_acc()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    class _NoGraph:
        def replay(self):
            pass

    graphs = {}
    for name, fn, used in (("append", do_append, w.appended and not fused), ("attn", do_attn, True),
                           ("acc", do_acc, has_acc)):
        if not used:
            graphs[name] = _NoGraph()
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def refresh():
        # Evict L2 (126 MB) between steps by READING a 256 MiB buffer: the lines
        # it leaves are clean, so no write-back lands in the next timed step.
        flush.max()
        if has_acc:
            ctx_scratch.copy_(w.context_lens)

    for _ in range(args.warmup):
        refresh()
        graphs["append"].replay()
        graphs["attn"].replay()
        graphs["acc"].replay()
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())} during warm-up")

    K = args.steps
    # events bracket the phases that have work only: an event pair around
    # nothing costs ~2 us of the GPU timeline
    phases = [n for n in ("append", "attn", "acc") if not isinstance(graphs[n], _NoGraph)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
           for _ in range(K)]
    clocks = ClockSampler(gpu_index_for_smi(local)) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    hold_gpu(K)
    for i in range(K):
        refresh()
        e = evs[i]
        e[0].record()
        for j, name in enumerate(phases):
            graphs[name].replay()
            e[j + 1].record()
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if clocks else None
    step_ms = sum(e[0].elapsed_time(e[-1]) for e in evs) / K
    span = {name: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / K
            for j, name in enumerate(phases)}
    attn_ms = span["attn"]
    app_ms = span.get("append", 0.0)
    acc_ms = span.get("acc", 0.0)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())} in the timed region")

    # Parity of the timed step's outputs (outside the timed region, before any
    # other launch writes `outs`): attention on a seeded sample of sequences,
    # acceptance on the whole batch.
    oracle_inputs = {}
    parity = None
    if rank == 0 and not args.no_parity:
        import oracle

        oracle.build()
        parity = parity_sample(w, outs, quant_cpu if q8 else None, oracle_inputs)
        if has_acc:
            ctx0 = w.context_lens.cpu().numpy()
            rp = None
            if sampled:
                ra, rn, rc, _ = oracle.accept_sampled(
                    sin.q.cpu().numpy(), sin.p.cpu().numpy(), sin.draft.cpu().numpy(),
                    sin.uniforms.cpu().numpy(), ctx0)
            elif tree_acc:
                ra, rn, rp, rc, _ = oracle.accept_tree(w.logits.cpu(), w.draft.cpu(), w.parents(),
                                                       ctx0)
            else:
                ra, rn, rc = oracle.accept_prefix(w.logits.cpu(), w.draft.cpu(), ctx0)
            acc_ok = (np.array_equal(acc_out.cpu().numpy(), ra)
                      and np.array_equal(nxt_out.cpu().numpy(), rn)
                      and np.array_equal(ctx_scratch.cpu().numpy(), rc))
            if rp is not None:
                acc_ok = acc_ok and np.array_equal(path_out.cpu().numpy(), rp)
                # the compacted rows: after the step's append node i's rows are
                # k_new / v_new[b, i] (one-byte caches: the oracle's codes and
                # scale of that row); the oracle's branch says which node each
                # position base+1+j must now hold (every layer)
                comp_ok = True
                bt_h = w.block_tables.cpu().numpy()
                for l in range(L):
                    news = (w.k_new[l].cpu(), w.v_new[l].cpu())
                    if q8:
                        caches = (qk[l].cpu(), qv[l].cpu())
                        scales = (sk[l].cpu(), sv[l].cpu())
                    else:
                        caches = (w.k_cache[l].cpu(), w.v_cache[l].cpu())
                    for b in range(w.B):
                        base = int(rc[b]) - 1 - int(ra[b])
                        for j in range(int(ra[b])):
                            pos = base + 1 + j
                            blk, row = int(bt_h[b, pos // 16]), pos % 16
                            node = int(rp[b, j])
                            for c, cache in enumerate(caches):
                                src = news[c][b, node]  # [K, H]
                                if not q8:
                                    comp_ok &= torch.equal(cache[blk, row].view(torch.int16),
                                                           src.view(torch.int16))
                                    continue
                                for kh in range(w.K):
                                    codes, scale = oracle.quantize_row(src[kh], w.dtype, args.kv)
                                    comp_ok &= bool(np.array_equal(
                                        cache[blk, row, kh].numpy(), codes)
                                        and float(scales[c][blk, kh, row]) == scale)
                parity["compaction_bit_exact"] = bool(comp_ok)
                acc_ok = acc_ok and comp_ok
            parity["accept_bit_exact"] = bool(acc_ok)
            parity["parity_pass"] = bool(parity["parity_pass"] and acc_ok)

    # Tree verification: the same launches with the plain chain mask, for the
    # cost of the custom mask (the speculation blog reports up to 50 % for a
    # mask over the whole sequence).
    tree_rec = None
    if tree_t is not None:
        g_chain = torch.cuda.CUDAGraph()
        saved = dict(extra)
        extra.clear()
        with torch.cuda.graph(g_chain):
            do_attn()
        extra.update(saved)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for _ in range(args.warmup):
            refresh()
            g_chain.replay()
        hold_gpu(K)
        for i in range(K):
            refresh()
            ev[i][0].record()
            g_chain.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        chain_ms = sum(a.elapsed_time(b) for a, b in ev) / K
        tree_rec = {"nodes": w.T, "parents": list(w.tree), "tree_attention_us": round(
            attn_ms * 1e3 / L, 3), "chain_attention_us": round(chain_ms * 1e3 / L, 3),
            "tree_over_chain": round(attn_ms / chain_ms, 4)}

    attn_b, app_b, acc_b = step_bytes(w, args.kv)
    if sampled:
        from gqa_decode_attention_02_gb300 import analytic as A

        acc_b = A.accept_sampled_bytes(acc_out.cpu().numpy(), w.T, V)
    elif tree_acc:
        from gqa_decode_attention_02_gb300 import analytic as A

        acc_b = (A.accept_tree_bytes(w.B, w.T, V)
                 + L * A.kv_compact_bytes(acc_out.cpu().numpy(), w.K, w.H, 1 if q8 else 2, w.T,
                                          scale_bytes=4 if q8 else 0))
    bytes_step = L * (attn_b + app_b) + acc_b
    step_ms_max, value = combine_ranks(step_ms, bytes_step, world, dev)
    peak, peak_src = measured_peak()
    attn_launch_ms = attn_ms / L
    kernel_b = attn_b + (app_b if fused else 0)  # the fused launch also does the append
    achieved = kernel_b / (attn_launch_ms * 1e-3) / 1e9
    # which kernel served the attention calls (the library's own choice; the
    # one-byte cache always runs on the warp-level kernel)
    if q8:
        engine = "warp"
    else:
        picks = {gq.attention_engine(w.q[l], w.k_cache[l], w.block_tables, window=w.window(l),
                                     engine=args.engine) for l in range(L)}
        engine = picks.pop() if len(picks) == 1 else "mixed"
    traffic = profiled_traffic(args.workload if not q8 else f"{args.workload}_{args.kv}", engine)

    # e2e: host buffers -> device, the captured API calls, results -> host
    e2e = None
    e2e_eager = None
    if not args.no_e2e:
        h_in = [t.cpu().pin_memory() for t in (w.q + (w.k_new + w.v_new if w.appended else []))]
        d_in = w.q + (w.k_new + w.v_new if w.appended else [])
        h_meta = [w.block_tables.cpu().pin_memory(), w.context_lens.cpu().pin_memory()]
        d_meta = [w.block_tables, w.context_lens]
        h_out = [torch.empty_like(o, device="cpu").pin_memory() for o in outs]
        if sampled:
            for t in (sin.q, sin.p, sin.draft, sin.uniforms):
                h_in.append(t.cpu().pin_memory())
                d_in.append(t)
        elif has_acc:
            for t in (w.logits, w.draft) + ((parents_d,) if tree_acc else ()):
                h_in.append(t.cpu().pin_memory())
                d_in.append(t)
        if has_acc:
            h_acc = [torch.empty(w.B, dtype=torch.int32).pin_memory() for _ in range(2)]
            if tree_acc:
                h_acc.append(torch.empty_like(path_out, device="cpu").pin_memory())
        h2d = sum(t.numel() * t.element_size() for t in h_in + h_meta)
        d2h = (sum(t.numel() * t.element_size() for t in h_out)
               + (sum(t.numel() * t.element_size() for t in h_acc) if has_acc else 0))

        def e2e_step(use_graph):
            for d, h in zip(d_in + d_meta, h_in + h_meta):
                d.copy_(h, non_blocking=True)
            if use_graph:
                graphs["append"].replay()
                graphs["attn"].replay()
                graphs["acc"].replay()
            else:
                do_append(), do_attn(), do_acc()
            for h, o in zip(h_out, outs):
                h.copy_(o, non_blocking=True)
            if has_acc:
                h_acc[0].copy_(acc_out, non_blocking=True)
                h_acc[1].copy_(nxt_out, non_blocking=True)
                if tree_acc:
                    h_acc[2].copy_(path_out, non_blocking=True)

        for use_graph in (True, False):
            for _ in range(2):
                refresh()
                e2e_step(use_graph)
            torch.cuda.synchronize()
            tot = 0.0
            for _ in range(K):
                refresh()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                e2e_step(use_graph)
                torch.cuda.synchronize()
                tot += time.perf_counter() - t0
            ms = tot / K * 1e3
            rec = {"value": world * bytes_step / (ms * 1e-3) / 1e9, "unit": "GB/s",
                   "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
            if use_graph:
                rec["how"] = ("pinned host inputs copied in, the step's library calls "
                              "replayed from their CUDA-graph capture, outputs copied out; "
                              "host wall clock around each step")
                e2e = rec
            else:
                rec["how"] = "as e2e but every library call made from Python each step"
                e2e_eager = rec

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, spent, desc, thr = oracle_sample(w, args.cpu_seconds, quant_cpu if q8 else None,
                                            inputs=oracle_inputs)
        v1, spent1, desc1, _ = oracle_sample(w, args.cpu_seconds / 3,
                                             quant_cpu if q8 else None, nthreads=1,
                                             inputs=oracle_inputs)
        cpu = {"value": v, "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2), "cpu_model": cpu_model(),
               "single_thread": {"value": v1, "unit": "GB/s", "cores": 1, "sample": desc1,
                                 "seconds": round(spent1, 2)}}

    ctx = w.context_lens.cpu().numpy()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) values rounded to the dtype, paged cache with "
                "NaN sentinels in unused slots, shuffled block tables",
        "config": {
            "workload": f"{w.name}: {w.desc}",
            "B": w.B, "T": w.T, "N": w.N, "K": w.K, "H": w.H, "layers": L,
            "block_size": w.block_size, "sum_context_tokens": int(ctx.sum()),
            "l2": "flushed between steps (256 MiB read outside the step events)",
            "accept": ("none" if not has_acc else
                       "stochastic (speculative sampling) over fp32 probabilities [B,T,V] and "
                       "[B,T-1,V], seeded Dirichlet rows" if sampled else
                       "greedy over the draft tree (fp32 logits [B,T,V]), then compaction of "
                       "the kept branch's cache rows" if tree_acc else
                       "greedy longest prefix over fp32 logits [B,T,V]"),
            "append": ("fused into the attention launch" if fused else
                       "separate kv_append launches" if w.appended else "none"),
            "parallelism": f"replicas x{world}",
            "engine": engine,
            "windows": list(w.windows) if w.windows else None,
            "kv_cache": ("dtype of q" if not q8 else
                         f"{args.kv} codes + fp32 scale per cached row (quantized append, "
                         f"then attention)"),
        },
        "pct_of_peak": round(100 * value / world / peak, 2),
        "attention_tokens_per_s": round(world * w.B * w.T * L / (step_ms_max * 1e-3), 1),
        "context_tokens_per_s": round(world * int(ctx.sum()) * L / (step_ms_max * 1e-3), 1),
        "breakdown_ms": {"append": round(app_ms, 5), "attention": round(attn_ms, 5),
                         "accept": round(acc_ms, 5)},
        "roofline": {"bound": "hbm",
                     "kernel": {"warp": "attention_kernel", "direct": "direct_kernel"}.get(
                                    engine, "tc_attention_kernel (tcgen05)") + (
                                    "" if not fused else " (kv_append fused)"
                                    if engine in ("warp", "direct")
                                    else " (with the kv_append launch of the same call)") + (
                         f" (one-byte {args.kv} cache)" if q8 else ""),
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": kernel_b,
                     "avg_launch_us": round(attn_launch_ms * 1e3, 3)},
        "tree_verify": tree_rec,
        "parity": parity,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_eager": e2e_eager,
        # the tensor-memory kernel's fused form is a kv_append launch + the attention launch
        "gpu_launches": K * ((L if w.appended and (not fused or engine == "tmem") else 0) + L
                             + (1 if has_acc else 0) + (L if tree_acc else 0)),
        "clocks": clk,
        "wall_s_timed": round(wall, 4),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ---- reference arm: the oracle on the host cores ----------------------------------------
def run_reference(args, world, rank, local):
    """The reference arm: the fp64 oracle on the host cores, same workload, same
    metric.  One step = the oracle's attention over one (layer, 8-sequence)
    chunk, cycling through the batch."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from gqa_decode_attention_02_gb300 import analytic as A
    from gqa_decode_attention_02_gb300 import workloads

    oracle.build()
    w = workloads.make(args.workload, B=args.batch)  # CPU tensors
    ctx = w.context_lens.numpy()
    chunk = 8
    units = [(l, s) for l in range(w.layers) for s in range(0, w.B, chunk)]
    K, W = args.steps, args.warmup
    times, nbytes, cache = [], [], {}
    quant = None
    if args.kv != "same":  # the oracle's own one-byte caches
        codes = [oracle.quantize_cache(c, w.dtype, args.kv) for c in w.k_cache]
        vcodes = [oracle.quantize_cache(c, w.dtype, args.kv) for c in w.v_cache]
        quant = (args.kv, [c for c, _ in codes], [c for c, _ in vcodes],
                 [s_ for _, s_ in codes], [s_ for _, s_ in vcodes])
    q8 = {} if quant is None else {"kv_elem_bytes": 1, "row_scale_bytes": 4}
    for i in range(W + K):
        l, s0 = units[i % len(units)]
        if l not in cache:
            cache.clear()
            cache[l] = _oracle_layer_inputs(w, l, quant)
        q, kc, vc = cache[l][:3]
        qa = {} if quant is None else {"kv": args.kv, "k_scale": cache[l][3],
                                       "v_scale": cache[l][4]}
        bl = np.arange(s0, min(w.B, s0 + chunk), dtype=np.int32)
        t0 = time.perf_counter()
        oracle.attention(q, kc, vc, w.block_tables, w.context_lens, w.dtype, b_list=bl,
                         window=w.window(l), tree_mask=w.tree_mask(), **qa)
        dt = time.perf_counter() - t0
        if i >= W:
            times.append(dt)
            nbytes.append(A.attention_algorithmic_bytes(ctx[bl], w.T, w.N, w.K, w.H, 2,
                                                        window=w.window(l), **q8))
    value = sum(nbytes) / sum(times) / 1e9
    ms = 1e3 * sum(times) / K
    desc = (f"each step: the fp64 oracle's attention over one layer x {chunk} sequences of "
            f"{w.name}, cycling through {w.layers} layers x {w.B} sequences")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
        "data": "synthetic (same seeded recipe as our arm)",
        "config": {"workload": f"{w.name}: {w.desc}", "B": w.B, "T": w.T, "N": w.N,
                   "K": w.K, "H": w.H, "layers": w.layers, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _free_port() -> int:
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _replica(local, n, port, fn, argv):
    """Child process of launch_replicas: the environment torchrun would give
    rank `local` of `n` on this node, then fn(argv)."""
    os.environ.update(RANK=str(local), LOCAL_RANK=str(local), WORLD_SIZE=str(n),
                      LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    fn(argv)


def launch_replicas(n: int, fn, argv) -> None:
    """Run fn(argv) in n spawned processes, one rank each (RANK / LOCAL_RANK /
    WORLD_SIZE / MASTER_ADDR=127.0.0.1 / MASTER_PORT set as torchrun sets
    them); raises if any rank fails."""
    import torch.multiprocessing as mp

    mp.start_processes(_replica, args=(n, _free_port(), fn, argv), nprocs=n, join=True,
                       start_method="spawn")


def main(argv=None):
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # launched directly with --gpus N: start the N ranks here
        launch_replicas(args.gpus, main, sys.argv[1:] if argv is None else argv)
        return
    world, rank, local = dist_env()  # a launcher's world size wins over --gpus
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
