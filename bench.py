"""Benchmark of one Ulysses attention block training pass on GB300.

One step = the whole hot path over one batch of synthetic input, all through the C ABI
on one stream:
  QKV projection -> seq->head (+RoPE) -> causal GQA attention forward (+lse) ->
  head->seq of O -> seq->head of dO -> attention backward (dQ, dK, dV) ->
  head->seq of dQ, dK, dV.
Workload (default): the Llama-3.1-8B-shaped attention block at S=131072, P=8 virtual
ranks, hidden 4096, 32 query / 8 KV heads, head_dim 128, RoPE theta 500000, bf16.
Metric: causal attention fwd+bwd TFLOPS (algorithmic FLOPs: fwd 2*S^2*D*H, bwd 2.5x fwd)
over the whole step time; the permute GB/s (read + write bytes) is reported beside it.

With N > 1 GPUs (torchrun, one process per GPU) the step is the block as the pages run it
across GPUs: P = N ranks, each holding S/N tokens, with the two all-to-alls as NCCL
exchanges through the library (ulysses_a2a_exchange); the sequence length stays S, so the
job's work is fixed ("strong" scaling).  --sharded runs that same path at N = 1.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--seq S]    (S other than 131072 is for quick checks only)
       [--sharded]  (the multi-GPU code path, also at N = 1)
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

WORKLOAD = dict(name="llama3.1-8b-attention-block-fwd-bwd", S=131072, P=8, hidden=4096, H=32,
                G=8, D=128, theta=500000.0)
METRIC = "causal attn fwd+bwd TFLOPS at S=128K (whole step incl. projection and all-to-all permutes)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_config(S, P, parallelism):
    """The workload a line measures (the same dict for both arms at one N)."""
    w = WORKLOAD
    return {"workload": w["name"], "seq_len": S, "P": P, "hidden": w["hidden"],
            "n_q_heads": w["H"], "n_kv_heads": w["G"], "head_dim": w["D"],
            "rope_theta": w["theta"], "global_batch": 1, "parallelism": parallelism,
            "l2": "inputs larger than L2 (no flush)"}


def parallelism_of(world, P):
    return "ulysses-sp%d" % P if world > 1 else "single GPU, P=%d virtual ranks" % P


def attn_flops(S, H, D):
    fwd = 2.0 * S * S * D * H          # causal: half of the dense 4 S^2 D H
    return fwd, 2.5 * fwd


# DRAM bytes of one ulysses_attn_bwd call at the bench workload (S=131072), summed over its six
# kernels (dram__bytes_read.sum + dram__bytes_write.sum, one pass each, --clock-control none):
# attn_bwd_kernel and bwd_dq_kernel each from a capture of that kernel alone at S=131072
# (17.57 GB read + 8.84 GB written; 2.148 + 1.045 GB); the other four streaming kernels
# (largest magnitudes, pre-pass, two fp16 copies), whose bytes are a fixed number per element,
# from a capture of one call at S=32768 scaled by 4.  Valid only for the kernel source it was
# taken on: the figure is dropped (null) as soon as the hash of that source changes.
BWD_TRAFFIC = {"bytes": (17.569 + 8.838) * 1e9 + (2.148 + 1.045) * 1e9
                        + 4 * (0.673954 + 2.102759 + 0.081413 + 0.081357) * 1e9,
               "seq_len": 131072,
               "source_sha256": "dbe1906bf75f3a355795b09b5bf401a6346b3d5a72e4498ed604357326d48348"}


def bwd_traffic(seq_len):
    import hashlib
    h = hashlib.sha256()
    for f in ("attn_bwd.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "long_context_sequence_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != BWD_TRAFFIC["source_sha256"] or seq_len != BWD_TRAFFIC["seq_len"]:
        return None
    return BWD_TRAFFIC["bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        peaks = {k: float(d[k]) for k in FALLBACK_PEAKS}
        # the median SM clock under load while the sustained GEMM peak was measured
        clk = (d.get("clocks_under_load") or {}).get("sm_mhz_median")
        peaks["sustained_sm_mhz"] = float(clk) if clk else None
        return peaks, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS, sustained_sm_mhz=None), "fallback"


def reduce_max_ms(ms, world, dist=None, device=None):
    """Step time of the whole job: the maximum over ranks (every rank's own events)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step, world, ms_per_step):
    """Whole-job throughput: the work of all ranks divided by the slowest rank's time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------- CPU oracle leg
def oracle_sample(S, H, D, n_rows, seed_stream=0):
    """Times the oracle on a bounded sample of the workload: n_rows seed-sampled query rows
    of one head (causal forward over the full prefix, then dq of those rows).  Returns
    (algorithmic FLOPs of the sample, seconds, description)."""
    import numpy as np

    import oracle as O
    import synthetic
    rows = np.sort(synthetic.sample_rows(S, 8, n_rows, stream=seed_stream))[-n_rows:]
    jmax = int(rows.max()) + 1
    k = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_K, (jmax, 1, D), std=1.28))
    v = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_V, (jmax, 1, D), std=1.28))
    q = np.zeros((jmax, 1, D))
    q[rows] = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_Q, (rows.size, 1, D), std=1.28))
    do = np.zeros((jmax, 1, D))
    do[rows] = synthetic.bf16_to_f64(synthetic.normal_bf16(1, 0, (rows.size, 1, D)))
    t0 = time.perf_counter()
    O.causal_attention_bwd_rows(q, k, v, do, rows, jmax)   # forward of the rows + their dq
    dt = time.perf_counter() - t0
    flops = 3.5 * float(np.sum(4.0 * (rows + 1) * D))      # fwd + 2.5x bwd, causal prefix
    desc = ("%d seed-sampled query rows of one head at S=%d (fwd over the causal prefix + "
            "dq of those rows), D=%d" % (rows.size, S, D))
    return flops, dt, desc


def run_reference(args):
    """The oracle arm: each step is one bounded sample of the workload on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOAD
    S = args.seq or w["S"]
    rows = 1024
    for _ in range(args.warmup):
        oracle_sample(S, w["H"], w["D"], rows)
    flops = secs = 0.0
    desc = ""
    for i in range(args.steps):
        f, s, desc = oracle_sample(S, w["H"], w["D"], rows, seed_stream=i + 1)
        flops += f
        secs += s
    value = flops / secs / 1e12
    cores = host_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(S, w["P"] if args.gpus <= 1 else args.gpus,
                                      parallelism_of(args.gpus, w["P"] if args.gpus <= 1 else args.gpus)),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# --------------------------------------------------------------------------- GPU leg
class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx = float(f[2])
                except ValueError:
                    continue
                for name, val in zip(("hw_slowdown", "hw_thermal_slowdown",
                                      "sw_thermal_slowdown", "sw_power_cap"), f[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def run_sharded(args, U, world, rank, local, dev, dist):
    """One rank of a P = world GPU group: the shard's projection, the seq->head exchange of
    q, k, v, attention of the rank's head group, the head->seq exchange of o, then the
    backward: dO's exchange, the attention backward, and the gradients' exchange back with
    the RoPE backward in the unpack.  Every exchange is one NCCL group (the library's)."""
    import torch
    w = WORKLOAD
    S, hidden, H, G, D, theta = (args.seq or w["S"]), w["hidden"], w["H"], w["G"], w["D"], w["theta"]
    P = world
    cfg = U.make_config(S, P, hidden, H, G, D, rope_theta=theta)
    plan = U.ulysses_plan_rank(cfg, rank)
    sh = plan.shapes()
    n = S // P
    uid = [U.ulysses_nccl_unique_id() if rank == 0 else None]
    if world > 1:
        dist.broadcast_object_list(uid, src=0)
    comm = U.ulysses_nccl_comm_init(world, rank, uid[0])
    bf = torch.bfloat16
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    x = torch.randn(sh["x"], generator=gen, device=dev).to(bf)
    gen2 = torch.Generator(device=dev)
    gen2.manual_seed(999)                       # the weight is the same on every rank
    wq = (torch.randn(sh["w"], generator=gen2, device=dev) * 0.02).to(bf)
    do_loc = torch.randn(sh["o_seq"], generator=gen, device=dev).to(bf)
    e = lambda name, dt=bf: torch.empty(sh[name], dtype=dt, device=dev)   # noqa: E731
    qkv_loc = e("qkv")
    sq, sk, sv, rq, rk, rv = e("q"), e("k"), e("v"), e("q"), e("k"), e("v")
    o, o_lo, ro = e("o"), e("o"), e("o")
    lse = e("lse", torch.float32)
    o_loc = e("o_seq")
    sdo, rdo = e("o"), e("o")
    dq, dk, dv, xq, xk, xv = e("q"), e("k"), e("v"), e("q"), e("k"), e("v")
    dqkv_loc = e("qkv")
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sid = stream.cuda_stream
    names = ["qkv_proj", "pack_qkv", "exchange_qkv", "attn_fwd", "exchange_o", "unpack_o",
             "pack_do", "exchange_do", "attn_bwd", "exchange_grads", "unpack_grads"]
    launches_per_step = 1 + 1 + 1 + 1 + 1 + 6 + 1   # the library's kernels (NCCL's not counted)

    def step(ev=None, io=None):
        xs, dos, os_, dqs = io if io is not None else (x, do_loc, o_loc, dqkv_loc)

        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        U.ulysses_qkv_proj(plan, xs, wq, qkv_loc, sid)
        mark(1)
        U.ulysses_a2a_pack_qkv(plan, qkv_loc, sq, sk, sv, apply_rope=True, stream=sid)
        mark(2)
        U.ulysses_a2a_exchange(plan, comm, [sq, sk, sv], [rq, rk, rv], sid)
        mark(3)
        U.ulysses_attn_fwd(plan, rq, rk, rv, o, lse, sid, o_lo=o_lo)
        mark(4)
        U.ulysses_a2a_exchange(plan, comm, [o], [ro], sid)
        mark(5)
        U.ulysses_a2a_unpack_heads(plan, ro, H, os_, sid)
        mark(6)
        U.ulysses_a2a_pack_heads(plan, dos, H, sdo, sid)
        mark(7)
        U.ulysses_a2a_exchange(plan, comm, [sdo], [rdo], sid)
        mark(8)
        U.ulysses_attn_bwd(plan, rq, rk, rv, o, lse, rdo, dq, dk, dv, ws, sid, o_lo=o_lo)
        mark(9)
        U.ulysses_a2a_exchange(plan, comm, [dq, dk, dv], [xq, xk, xv], sid)
        mark(10)
        U.ulysses_a2a_unpack_qkv(plan, xq, xk, xv, dqs, apply_rope=True, stream=sid)
        mark(11)

    for _ in range(args.warmup):
        step()
    st = U.ulysses_sync_status(plan, sid)
    if st != U.ULY_OK:
        raise RuntimeError("device status %d during warm-up: %s" % (st, U.ulysses_last_error()))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(12)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    st = U.ulysses_sync_status(plan, sid)
    if st != U.ULY_OK:
        raise RuntimeError("device status %d: %s" % (st, U.ulysses_last_error()))
    ms_step = reduce_max_ms(t0.elapsed_time(t1) / args.steps, world, dist, dev)
    avg = {nm: sum(e_[i].elapsed_time(e_[i + 1]) for e_ in evs) / len(evs)
           for i, nm in enumerate(names)}
    fwd_f, bwd_f = attn_flops(S, H, D)
    value = job_tflops((fwd_f + bwd_f) / world, world, ms_step)

    # end to end through the same calls: x and dO of the shard uploaded from pinned host
    # memory and o and dqkv of the shard read back, every step, inside the timed region
    hx = torch.empty(sh["x"], dtype=bf, pin_memory=True)
    hdo = torch.empty(sh["o_seq"], dtype=bf, pin_memory=True)
    hx.copy_(x)
    hdo.copy_(do_loc)
    ho = torch.empty(sh["o_seq"], dtype=bf, pin_memory=True)
    hg = torch.empty(sh["qkv"], dtype=bf, pin_memory=True)
    xs, dos = torch.empty_like(x), torch.empty_like(do_loc)

    def e2e_step():
        xs.copy_(hx, non_blocking=True)
        dos.copy_(hdo, non_blocking=True)
        step(io=(xs, dos, o_loc, dqkv_loc))
        ho.copy_(o_loc, non_blocking=True)
        hg.copy_(dqkv_loc, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(args.steps, 5)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ems = reduce_max_ms(e0.elapsed_time(e1) / e2e_steps, world, dist, dev)
    if not torch.equal(hg, dqkv_loc.cpu()):
        raise RuntimeError("e2e read-back differs from the device result")
    e2e = {"value": job_tflops((fwd_f + bwd_f) / world, world, ems), "unit": "TFLOPS",
           "h2d_bytes_per_step": world * (hx.numel() + hdo.numel()) * 2,
           "d2h_bytes_per_step": world * (ho.numel() + hg.numel()) * 2, "ms_per_step": ems,
           "copies": "on the compute stream, not overlapped", "steps": e2e_steps}
    s2h, h2s = U.ulysses_a2a_volume(cfg)
    if rank == 0:
        peaks, peak_kind = load_peaks()
        bwd_tf = bwd_f / world / (avg["attn_bwd"] * 1e-3) / 1e12
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (device torch.randn, seeded; X~N(0,1), W~N(0,0.02^2), dO~N(0,1))",
            "config": workload_config(S, P, "ulysses-sp%d" % P),
            "roofline": {"kernel": "ulysses_attn_bwd", "bound": "tensor", "achieved": bwd_tf,
                         "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                         "frac": bwd_tf / peaks["bf16_tflops_sustained"], "traffic": None,
                         "peak_source": "%s bf16_tflops_sustained" % peak_kind},
            "kernels_ms": avg, "exchange_bytes_per_rank": s2h + h2s,
            "gpu_launches": launches_per_step * args.steps, "clocks": clk.summary(),
            "e2e": e2e, "cpu_baseline": None,
        }
        print(json.dumps(line))
    U.ulysses_nccl_comm_destroy(comm)
    plan.close()


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import long_context_sequence_gb300 as U

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 or args.sharded:
        run_sharded(args, U, world, rank, local, dev, dist)
        if world > 1:
            dist.destroy_process_group()
        return
    w = WORKLOAD
    S, P, hidden, H, G, D, theta = (args.seq or w["S"]), w["P"], w["hidden"], w["H"], w["G"], w["D"], w["theta"]
    plan = U.ulysses_plan(U.make_config(S, P, hidden, H, G, D, rope_theta=theta))
    sh = plan.shapes()
    bf = torch.bfloat16
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    x = torch.randn(sh["x"], generator=gen, device=dev).to(bf)
    wq = (torch.randn(sh["w"], generator=gen, device=dev) * 0.02).to(bf)
    do_seq = torch.randn(sh["o_seq"], generator=gen, device=dev).to(bf)
    qkv = torch.empty(sh["qkv"], dtype=bf, device=dev)
    q, k, v = (torch.empty(sh[n], dtype=bf, device=dev) for n in ("q", "k", "v"))
    o = torch.empty(sh["o"], dtype=bf, device=dev)
    o_lo = torch.empty(sh["o"], dtype=bf, device=dev)
    lse = torch.empty(sh["lse"], dtype=torch.float32, device=dev)
    o_seq = torch.empty(sh["o_seq"], dtype=bf, device=dev)
    do = torch.empty(sh["o"], dtype=bf, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dqkv_seq = torch.empty(sh["qkv"], dtype=bf, device=dev)
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sid = stream.cuda_stream
    names = ["qkv_proj", "seq_to_head", "attn_fwd", "head_to_seq_o", "seq_to_head_do",
             "attn_bwd", "head_to_seq_grads"]
    # qkv_proj, seq_to_head, attn_fwd, head_to_seq (O), seq_to_head (dO), attn_bwd (largest
    # magnitudes, pre, two fp16 copies, main, dQ conversion), head_to_seq of the gradients
    launches_per_step = 1 + 1 + 1 + 1 + 1 + 6 + 1

    def step(ev=None, io=None, sync=None):
        # io: the step's input and output buffers (x, dO_seq, o_seq, dqkv_seq)
        # sync (end-to-end runs): events the step waits for before it first reads x and dO,
        # and records once o_seq is final
        xs, dos, os_, dqs = io if io is not None else (x, do_seq, o_seq, dqkv_seq)

        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        if sync is not None:
            stream.wait_event(sync["x"])
        U.ulysses_qkv_proj(plan, xs, wq, qkv, sid)
        mark(1)
        U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=True, stream=sid)
        mark(2)
        U.ulysses_attn_fwd(plan, q, k, v, o, lse, sid, o_lo=o_lo)
        mark(3)
        U.ulysses_head_to_seq(plan, o, H, os_, sid)
        if sync is not None:
            sync["o"].record(stream)
        mark(4)
        if sync is not None:
            stream.wait_event(sync["do"])
        U.ulysses_seq_to_head_heads(plan, dos, H, do, sid)
        mark(5)
        U.ulysses_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws, sid, o_lo=o_lo)
        mark(6)
        U.ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqs, apply_rope=True, stream=sid)
        mark(7)

    for _ in range(args.warmup):
        step()
    st = U.ulysses_sync_status(plan, sid)
    if st != U.ULY_OK:
        raise RuntimeError("device status %d during warm-up: %s" % (st, U.ulysses_last_error()))

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    st = U.ulysses_sync_status(plan, sid)
    if st != U.ULY_OK:
        raise RuntimeError("device status %d: %s" % (st, U.ulysses_last_error()))
    total_ms = t_start.elapsed_time(t_end)
    per = {n: [] for n in names}
    for e in evs:
        for i, n in enumerate(names):
            per[n].append(e[i].elapsed_time(e[i + 1]))
    avg = {n: sum(vs) / len(vs) for n, vs in per.items()}
    total_ms = reduce_max_ms(total_ms, world, dist, dev)
    ms_step = total_ms / args.steps
    fwd_f, bwd_f = attn_flops(S, H, D)
    value = job_tflops(fwd_f + bwd_f, world, ms_step)

    # permute traffic per step (read + write bytes)
    C = (H + 2 * G) * D
    perm_bytes = {"seq_to_head": S * C * 2 * 2, "head_to_seq_o": S * H * D * 2 * 2,
                  "seq_to_head_do": S * H * D * 2 * 2,
                  "head_to_seq_grads": S * (H + 2 * G) * D * 2 * 2}
    perm_ms = sum(avg[n] for n in perm_bytes)
    perm_gbs = sum(perm_bytes.values()) / (perm_ms * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    bwd_tflops = bwd_f / (avg["attn_bwd"] * 1e-3) / 1e12
    fwd_tflops = fwd_f / (avg["attn_fwd"] * 1e-3) / 1e12
    qkv_tflops = 2.0 * S * hidden * C / (avg["qkv_proj"] * 1e-3) / 1e12
    s2h_gbs = perm_bytes["seq_to_head"] / (avg["seq_to_head"] * 1e-3) / 1e9

    # End to end through the same calls: every step copies its inputs (x, dO) from pinned
    # host memory and reads its outputs (o_seq, dqkv_seq) back, all inside the timed region.
    # The copies run on two copy streams (up, down) with two buffer sets, so step i's read-back and
    # step i+1's upload overlap the compute of the steps next to them, as a training loop
    # that streams its activations would run.
    e2e = None
    if not args.no_e2e:
        hx = torch.empty(sh["x"], dtype=bf, pin_memory=True)
        hdo = torch.empty(sh["o_seq"], dtype=bf, pin_memory=True)
        hx.copy_(x)
        hdo.copy_(do_seq)
        sets = [(x, do_seq, o_seq, dqkv_seq),
                (torch.empty_like(x), torch.empty_like(do_seq), torch.empty_like(o_seq),
                 torch.empty_like(dqkv_seq))]
        houts = [[torch.empty(t.shape, dtype=bf, pin_memory=True) for t in (o_seq, dqkv_seq)]
                 for _ in range(2)]
        h2d = hx.numel() * 2 + hdo.numel() * 2
        d2h = o_seq.numel() * 2 + dqkv_seq.numel() * 2
        up = torch.cuda.Stream(dev)      # host -> device
        down = torch.cuda.Stream(dev)    # device -> host
        ev = lambda: torch.cuda.Event()   # noqa: E731
        x_up = [ev(), ev()]         # x of set b is on the device
        do_up = [ev(), ev()]        # dO of set b is on the device
        o_ready = [ev(), ev()]      # o_seq of set b is final
        computed = [ev(), ev()]     # the step on set b is done (inputs free, outputs ready)
        read_back = [ev(), ev()]    # outputs of set b are on the host

        # x is uploaded first and dO after it: the step reads dO only at its backward half,
        # and o_seq goes back to the host as soon as it is final, so only the first step's x
        # and the last step's dqkv_seq cannot overlap compute.
        def e2e_run(n):
            for i in range(n):
                b = i % 2
                xs, dos, os_, dqs = sets[b]
                with torch.cuda.stream(up):
                    if i >= 2:
                        up.wait_event(computed[b])
                    xs.copy_(hx, non_blocking=True)
                    x_up[b].record(up)
                    dos.copy_(hdo, non_blocking=True)
                    do_up[b].record(up)
                if i >= 2:
                    stream.wait_event(read_back[b])
                step(io=sets[b], sync={"x": x_up[b], "do": do_up[b], "o": o_ready[b]})
                computed[b].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(o_ready[b])
                    houts[b][0].copy_(os_, non_blocking=True)
                    down.wait_event(computed[b])
                    houts[b][1].copy_(dqs, non_blocking=True)
                    read_back[b].record(down)
            for b in range(min(n, 2)):
                stream.wait_event(read_back[b])

        e2e_run(2)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        # at least 10 steps, so that the first upload and the last read-back (which nothing
        # can overlap) weigh as little as in a training loop
        e2e_steps = max(args.steps, 10)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        e2e_run(e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = reduce_max_ms(e0.elapsed_time(e1) / e2e_steps, world, dist, dev)
        # the last step's outputs arrived on the host intact
        last = (e2e_steps - 1) % 2
        if not (torch.equal(houts[last][0], sets[last][2].cpu()) and
                torch.equal(houts[last][1], sets[last][3].cpu())):
            raise RuntimeError("e2e read-back differs from the device result")
        e2e = {"value": job_tflops(fwd_f + bwd_f, world, ems), "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "copies": "H2D and D2H streams, double-buffered, overlapped with compute",
               "steps": e2e_steps}

    # The whole attention layer's training step, timed on its own after the hot-path step:
    # projection, seq->head (RoPE), attention forward, output projection read straight from
    # the head layout, its backward written straight into the head layout, attention
    # backward, gradient head->seq (RoPE backward), projection backward.
    layer = None
    if not args.no_layer:
        wo = (torch.randn((hidden, H * D), generator=gen, device=dev) * 0.02).to(bf)
        dy = torch.randn((S, hidden), generator=gen, device=dev).to(bf)
        y = torch.empty((S, hidden), dtype=bf, device=dev)
        dx = torch.empty(sh["x"], dtype=bf, device=dev)
        dw = torch.empty(sh["w"], dtype=torch.float32, device=dev)
        dwo = torch.empty((hidden, H * D), dtype=torch.float32, device=dev)
        lnames = ["qkv_proj", "seq_to_head", "attn_fwd", "o_proj", "o_proj_bwd", "attn_bwd",
                  "head_to_seq_grads", "qkv_proj_bwd"]

        def layer_step(ev=None):
            def mark(i):
                if ev is not None:
                    ev[i].record(stream)
            mark(0)
            U.ulysses_qkv_proj(plan, x, wq, qkv, sid)
            mark(1)
            U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=True, stream=sid)
            mark(2)
            U.ulysses_attn_fwd(plan, q, k, v, o, lse, sid, o_lo=o_lo)
            mark(3)
            U.ulysses_o_proj(plan, o, wo, y, sid)
            mark(4)
            U.ulysses_o_proj_bwd(plan, o, wo, dy, do, dwo, sid)
            mark(5)
            U.ulysses_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws, sid, o_lo=o_lo)
            mark(6)
            U.ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqkv_seq, apply_rope=True, stream=sid)
            mark(7)
            U.ulysses_qkv_proj_bwd(plan, x, wq, dqkv_seq, dx, dw, sid)
            mark(8)

        for _ in range(args.warmup):
            layer_step()
        lev = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for e in lev:
            layer_step(e)
        torch.cuda.synchronize()
        st = U.ulysses_sync_status(plan, sid)
        if st != U.ULY_OK:
            raise RuntimeError("device status %d: %s" % (st, U.ulysses_last_error()))
        lper = {n: sum(e[i].elapsed_time(e[i + 1]) for e in lev) / len(lev)
                for i, n in enumerate(lnames)}
        lms = sum(e[0].elapsed_time(e[8]) for e in lev) / len(lev)
        proj_f = 2.0 * S * hidden * C          # each of the three QKV GEMMs
        oproj_f = 2.0 * S * hidden * H * D     # each of the three output-projection GEMMs
        layer_f = fwd_f + bwd_f + 3 * proj_f + 3 * oproj_f
        layer = {"ms_per_step": lms, "tflops": layer_f / (lms * 1e-3) / 1e12,
                 "flops_per_step": layer_f, "kernels_ms": lper,
                 "o_proj_tflops": oproj_f / (lper["o_proj"] * 1e-3) / 1e12,
                 "o_proj_bwd_tflops": 2 * oproj_f / (lper["o_proj_bwd"] * 1e-3) / 1e12,
                 "qkv_proj_bwd_tflops": 2 * proj_f / (lper["qkv_proj_bwd"] * 1e-3) / 1e12,
                 "launches_per_step": 1 + 1 + 1 + 1 + 2 + 6 + 1 + 2}

    # Ring attention (what "Snowflake's Ulysses trick ..." para 3 compares Ulysses with) on
    # the same virtual ranks and tokens: its forward with the K/V exchange, beside the
    # Ulysses forward path (seq->head, attention, head->seq of O), and the per-rank volumes
    # of the two exchanges.
    ring = None
    if not args.no_ring:
        n = S // P
        q_s = torch.randn((P, n, H, D), generator=gen, device=dev).mul_(1.28).to(bf)
        k_s = torch.randn((P, n, G, D), generator=gen, device=dev).mul_(1.28).to(bf)
        v_s = torch.randn((P, n, G, D), generator=gen, device=dev).mul_(1.28).to(bf)
        o_s = torch.empty((P, n, H, D), dtype=bf, device=dev)
        lse_s = torch.empty((P, H, n), dtype=torch.float32, device=dev)
        rws = torch.empty(U.ulysses_ring_workspace_bytes(plan), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            U.ulysses_ring_attn_fwd(plan, q_s, k_s, v_s, o_s, lse_s, rws, sid)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        b0 = U.ulysses_bytes_moved(plan)
        r0.record(stream)
        for _ in range(args.steps):
            U.ulysses_ring_attn_fwd(plan, q_s, k_s, v_s, o_s, lse_s, rws, sid)
        r1.record(stream)
        torch.cuda.synchronize()
        st = U.ulysses_sync_status(plan, sid)
        if st != U.ULY_OK:
            raise RuntimeError("device status %d: %s" % (st, U.ulysses_last_error()))
        rms = r0.elapsed_time(r1) / args.steps
        cfg = U.make_config(S, P, hidden, H, G, D, rope_theta=theta)
        rv = U.ulysses_ring_volume(cfg)
        uv = sum(U.ulysses_a2a_volume(cfg))
        uly_fwd_ms = avg["seq_to_head"] + avg["attn_fwd"] + avg["head_to_seq_o"]
        ring = {"ms": rms, "tflops": fwd_f / (rms * 1e-3) / 1e12,
                "exchange_bytes_moved_per_call": (U.ulysses_bytes_moved(plan) - b0) // args.steps,
                "volume_per_rank_bytes": rv, "ulysses_volume_per_rank_bytes": uv,
                "volume_ratio_ring_over_ulysses": rv / uv,
                "ulysses_fwd_path_ms": uly_fwd_ms, "launches_per_call": 2 * P - 1}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        f, s, desc = oracle_sample(S, H, D, 6144)
        cpu = {"value": f / s / 1e12, "unit": "TFLOPS", "cores": host_cores(), "kind": "oracle",
               "sample": desc, "seconds": s}

    clocks = clk.summary()

    def fractions(tflops):
        # against the sustained peak (for a kernel inside a long step), the burst peak, and
        # the sustained peak with the kernel's time taken at the clock the peak was measured
        # at (time x bench SM MHz / peak SM MHz), so that a faster clock here flatters nothing
        f = {"frac_sustained": tflops / peaks["bf16_tflops_sustained"],
             "frac_burst": tflops / peaks["bf16_tflops"]}
        if clocks.get("sm_mhz") and peaks.get("sustained_sm_mhz"):
            f["frac_sustained_at_peak_clock"] = (tflops * peaks["sustained_sm_mhz"] / clocks["sm_mhz"]
                                                 / peaks["bf16_tflops_sustained"])
        return f

    if rank == 0:
        peak = peaks["bf16_tflops_sustained"]
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (device torch.randn, seeded; X~N(0,1), W~N(0,0.02^2), dO~N(0,1))",
            "config": workload_config(S, P, parallelism_of(world, P)),
            "roofline": dict({"kernel": "ulysses_attn_bwd", "bound": "tensor",
                              "achieved": bwd_tflops, "peak": peak, "unit": "TFLOP/s",
                              "frac": bwd_tflops / peak, "traffic": bwd_traffic(S),
                              "peak_source": "%s bf16_tflops_sustained" % peak_kind,
                              "peak_burst": peaks["bf16_tflops"],
                              "sm_mhz": clocks.get("sm_mhz"),
                              "peak_sustained_sm_mhz": peaks.get("sustained_sm_mhz")},
                             **fractions(bwd_tflops)),
            "kernels_ms": avg,
            "attn_fwd_tflops": fwd_tflops, "attn_bwd_tflops": bwd_tflops,
            "attn_fwd_frac": fwd_tflops / peak, "attn_fwd_fractions": fractions(fwd_tflops),
            "qkv_proj_tflops": qkv_tflops,
            "permute_gbs": perm_gbs, "permute_frac_hbm": perm_gbs / peaks["hbm_gbs"],
            "seq_to_head_gbs": s2h_gbs, "peaks": peaks, "peaks_source": peak_kind,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
            "layer_train_step": layer, "ring_attention": ring,
        }
        print(json.dumps(line))
    plan.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seq", type=int, default=0, help="override S (quick checks only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-layer", action="store_true")
    ap.add_argument("--no-ring", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sharded", action="store_true",
                    help="run the multi-GPU (real-rank, NCCL exchange) path, also at N = 1")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.seq:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
