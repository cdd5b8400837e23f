"""Benchmark of the paged GQA attention hot path on GB300.

One step = one pass of the whole path over one batch: for every layer, kv_append_paged of the
step's new tokens, attn_prefill_chunk of the prompt chunk, attn_decode_paged (split-KV + merge)
of the decoding sequences. The default workload is the 28-layer mixed scheduler step
(one 4,096-query chunk at offset 32,768 plus 31 decodes of 5,000..90,000 keys, each layer with
its own K/V pools: about 173 GB of HBM), so every step reads far more than L2 holds.

Reported (one JSON line from rank 0):
  value      decode KV-read GB/s = sum of decode KV bytes / device time of the decode calls
  prefill    chunked-prefill TFLOP/s = 4*D*Hq*(visible pairs) / device time of the prefill calls
  roofline   the dominant kernel against the measured (else fallback) HBM / tensor peak
  e2e        the same metrics through the public calls with pinned host buffers, per-step
             host->device copies of the step's inputs and device->host copies of the results
             inside the timed region
  cpu_baseline  the fp64 oracle timed on a bounded sample on the host cores

``--impl reference`` times the oracle itself (the only reference that exists for this path) on
the same workload, one bounded sample per step.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s HBM3e figure decode is quoted against
BUCKETS = (1, 2, 4, 8, 16, 32)


# ----------------------------------------------------------------------------------------------
# work accounting
# ----------------------------------------------------------------------------------------------
def decode_kv_bytes(seq_lens) -> int:
    """Bytes the method must read: every cached key and value of every decoding sequence."""
    return int(np.sum(seq_lens)) * W.kv_bytes_per_token()


def prefill_pairs(seq_len: int, q_len: int) -> int:
    """Visible (query, key) pairs of one chunk under bottom-right causal alignment."""
    off = seq_len - q_len
    return q_len * off + q_len * (q_len + 1) // 2


def prefill_flops(pairs: int) -> float:
    return 4.0 * W.HEAD_DIM * W.HQ * pairs  # QK^T and PV, 2 flops per MAC


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained", bf)
            if hbm and bf:
                return float(hbm), float(bf), float(bfs), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "long_context_paged_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel_file: str, src_hash: str, algorithmic_bytes: float):
    """DRAM bytes per launch, scaled from a committed ncu summary of a small case of the same
    kernel: the summary records DRAM bytes (read + write) per algorithmic byte of that case,
    and traffic grows with the bytes the launch must move. None if the summary is missing or
    was taken on another source."""
    path = os.path.join(ROOT, "profiles", kernel_file)
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != src_hash:
        return None
    try:
        return round(float(vals["dram_bytes_per_algorithmic_byte"]) * algorithmic_bytes)
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, out_path=None):
        self.proc = None
        self.path = out_path or os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, uuid=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if uuid and uuid not in parts[1]:
                continue
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def device_uuid():
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# ----------------------------------------------------------------------------------------------
# the timed step
# ----------------------------------------------------------------------------------------------
class Step:
    """Owns the workload on the device and runs/times one pass of the hot path."""

    def __init__(self, pa, name, device):
        self.pa = pa
        self.name = name
        self.inp = W.make_workload(name, device=device)
        self.dev = device
        inp = self.inp
        L, ql = inp.host_seq_lens, inp.host_q_lens
        self.is_chunk = ql > 1
        self.chunk_idx = np.nonzero(self.is_chunk)[0]
        self.dec_idx = np.nonzero(~self.is_chunk)[0]
        assert len(self.chunk_idx) <= 1 and (len(self.chunk_idx) == 0 or self.chunk_idx[0] == 0), \
            "the prompt chunk is the first sequence"
        self.n_chunk_rows = int(ql[self.chunk_idx].sum()) if len(self.chunk_idx) else 0
        self.layers = inp.layers
        self.max_s = int(L.max())
        self.append = name == "mixed_28l"
        self.dec_bytes = decode_kv_bytes(L[self.dec_idx]) if len(self.dec_idx) else 0
        self.pairs = sum(prefill_pairs(int(L[i]), int(ql[i])) for i in self.chunk_idx)
        self.pf_flops = prefill_flops(self.pairs)
        # bytes the prefill launch must move: the chunk's queries, its sequence's K/V, outputs
        self.pf_bytes = sum(int(ql[i]) * W.HQ * W.HEAD_DIM * 2 * 2 + int(ql[i]) * W.HQ * 4
                            + int(L[i]) * W.kv_bytes_per_token() for i in self.chunk_idx)
        B = inp.batch
        nd = len(self.dec_idx)
        if nd:
            d0 = int(self.dec_idx[0])
            self.dec_bt = inp.block_table[d0:].contiguous()
            self.dec_sl = inp.seq_lens[d0:].contiguous()
            ws = pa.decode_workspace_size(nd, self.max_s)
            self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
            self.dec_out = torch.empty(nd, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=device)
            self.dec_lse = torch.empty(nd, W.HQ, dtype=torch.float32, device=device)
        if self.n_chunk_rows:
            self.pf_cu = inp.cu_q_lens[:2].contiguous()
            self.pf_bt = inp.block_table[:1].contiguous()
            self.pf_sl = inp.seq_lens[:1].contiguous()
            self.pf_out = torch.empty(self.n_chunk_rows, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16,
                                      device=device)
            self.pf_lse = torch.empty(self.n_chunk_rows, W.HQ, dtype=torch.float32, device=device)
            self.pf_ws = torch.empty(max(256, pa.prefill_workspace_size(1, self.n_chunk_rows, self.max_s)),
                                     dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # kernels per call: append 1; prefill 2 (the chunk kernel and its merge); decode 1 or 2
        self.dec_kernels = pa.decode_kernels_per_call(nd, self.max_s) if nd else 0
        self.launches_per_step = self.layers * ((1 if self.append else 0) + (2 if self.n_chunk_rows else 0)
                                                + self.dec_kernels)

    def run(self, events=None, q_src=None, parts=("append", "prefill", "decode"), split=None):
        """One pass over the layers. split = (prefill CTAs, decode CTAs): after each layer's append,
        the decode runs on a second stream beside the prefill, each call's persistent grid capped
        at its share of the SMs, and the first stream waits for it before the next layer."""
        pa, inp = self.pa, self.inp
        stream = torch.cuda.current_stream()
        both = split is not None and self.n_chunk_rows and len(self.dec_idx) \
            and "prefill" in parts and "decode" in parts
        if both and not hasattr(self, "side"):
            self.side = torch.cuda.Stream(device=self.dev)
        for layer in range(self.layers):
            q = inp.q[layer] if q_src is None else q_src[layer]
            if self.append and "append" in parts:
                pa.kv_append_paged(inp.k_new[layer], inp.v_new[layer], inp.cu_q_lens, inp.start_pos,
                                   inp.block_table, inp.k_pools[layer], inp.v_pools[layer],
                                   status=self.status, stream=stream)
            if both:
                self.side.wait_stream(stream)
                pa.attn_prefill_chunk(q[:self.n_chunk_rows], self.pf_cu, inp.k_pools[layer],
                                      inp.v_pools[layer], self.pf_bt, self.pf_sl, self.n_chunk_rows,
                                      self.max_s, inp.scale, out=self.pf_out, lse=self.pf_lse,
                                      workspace=self.pf_ws, status=self.status, stream=stream,
                                      max_ctas=split[0])
                pa.attn_decode_paged(q[self.n_chunk_rows:], inp.k_pools[layer], inp.v_pools[layer],
                                     self.dec_bt, self.dec_sl, self.max_s, inp.scale,
                                     out=self.dec_out, lse=self.dec_lse, workspace=self.ws,
                                     status=self.status, stream=self.side, max_ctas=split[1])
                stream.wait_stream(self.side)
                continue
            if self.n_chunk_rows and "prefill" in parts:
                if events is not None:
                    events["pf"][layer][0].record(stream)
                pa.attn_prefill_chunk(q[:self.n_chunk_rows], self.pf_cu, inp.k_pools[layer],
                                      inp.v_pools[layer], self.pf_bt, self.pf_sl, self.n_chunk_rows,
                                      self.max_s, inp.scale, out=self.pf_out, lse=self.pf_lse,
                                      workspace=self.pf_ws, status=self.status, stream=stream)
                if events is not None:
                    events["pf"][layer][1].record(stream)
            if len(self.dec_idx) and "decode" in parts:
                if events is not None:
                    events["dec"][layer][0].record(stream)
                pa.attn_decode_paged(q[self.n_chunk_rows:], inp.k_pools[layer], inp.v_pools[layer],
                                     self.dec_bt, self.dec_sl, self.max_s, inp.scale,
                                     out=self.dec_out, lse=self.dec_lse, workspace=self.ws,
                                     status=self.status, stream=stream)
                if events is not None:
                    events["dec"][layer][1].record(stream)


def make_events(layers):
    mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(layers)]
    return {"pf": mk(), "dec": mk()}


def elapsed(evs):
    return sum(a.elapsed_time(b) for a, b in evs) / 1e3  # seconds


# ----------------------------------------------------------------------------------------------
# end-to-end through the public calls with host buffers
# ----------------------------------------------------------------------------------------------
def e2e_run(step: Step, steps: int):
    """Per step and layer: H2D of q, k_new, v_new (pinned), the four calls, D2H of every output.

    Decode e2e time per layer spans its q H2D, the decode call and the D2H of its output; the
    prefill phase likewise. Returns (decode GB/s, prefill TFLOP/s, h2d bytes, d2h bytes)."""
    inp = step.inp
    L = step.layers
    host_q = [inp.q[l].cpu().pin_memory() for l in range(L)]
    host_k = [inp.k_new[l].cpu().pin_memory() for l in range(L)] if step.append else None
    host_v = [inp.v_new[l].cpu().pin_memory() for l in range(L)] if step.append else None
    dev_q = torch.empty_like(inp.q[0])
    dev_k = torch.empty_like(inp.k_new[0]) if step.append else None
    dev_v = torch.empty_like(inp.v_new[0]) if step.append else None
    out_pf = torch.empty((max(step.n_chunk_rows, 1), W.HQ, W.HEAD_DIM), dtype=torch.bfloat16).pin_memory()
    lse_pf = torch.empty((max(step.n_chunk_rows, 1), W.HQ), dtype=torch.float32).pin_memory()
    nd = len(step.dec_idx)
    out_dec = torch.empty((max(nd, 1), W.HQ, W.HEAD_DIM), dtype=torch.bfloat16).pin_memory()
    lse_dec = torch.empty((max(nd, 1), W.HQ), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    pa = step.pa
    h2d = d2h = 0
    t_dec = t_pf = 0.0
    torch.cuda.synchronize()
    meta_host = [t.cpu().pin_memory() for t in (inp.cu_q_lens, inp.start_pos, inp.seq_lens)]
    meta_dev = [inp.cu_q_lens, inp.start_pos, inp.seq_lens]
    for s in range(steps):
        ev = make_events(L)
        for hsrc, ddst in zip(meta_host, meta_dev):   # the step's lengths and positions
            ddst.copy_(hsrc, non_blocking=True)
            if s == 0:
                h2d += hsrc.numel() * 4
        for layer in range(L):
            if step.append:
                dev_k.copy_(host_k[layer], non_blocking=True)
                dev_v.copy_(host_v[layer], non_blocking=True)
                pa.kv_append_paged(dev_k, dev_v, inp.cu_q_lens, inp.start_pos, inp.block_table,
                                   inp.k_pools[layer], inp.v_pools[layer], stream=stream)
                if s == 0:
                    h2d += 2 * dev_k.numel() * 2
            if step.n_chunk_rows:
                ev["pf"][layer][0].record(stream)
                n = step.n_chunk_rows
                dev_q[:n].copy_(host_q[layer][:n], non_blocking=True)
                pa.attn_prefill_chunk(dev_q[:n], step.pf_cu, inp.k_pools[layer], inp.v_pools[layer],
                                      step.pf_bt, step.pf_sl, n, step.max_s, inp.scale,
                                      out=step.pf_out, lse=step.pf_lse, workspace=step.pf_ws,
                                      stream=stream)
                out_pf.copy_(step.pf_out, non_blocking=True)
                lse_pf.copy_(step.pf_lse, non_blocking=True)
                ev["pf"][layer][1].record(stream)
                if s == 0:
                    h2d += n * W.HQ * W.HEAD_DIM * 2
                    d2h += out_pf.numel() * 2 + lse_pf.numel() * 4
            if nd:
                ev["dec"][layer][0].record(stream)
                n0 = step.n_chunk_rows
                dev_q[n0:n0 + nd].copy_(host_q[layer][n0:n0 + nd], non_blocking=True)
                pa.attn_decode_paged(dev_q[n0:n0 + nd], inp.k_pools[layer], inp.v_pools[layer],
                                     step.dec_bt, step.dec_sl, step.max_s, inp.scale,
                                     out=step.dec_out, lse=step.dec_lse, workspace=step.ws,
                                     stream=stream)
                out_dec.copy_(step.dec_out, non_blocking=True)
                lse_dec.copy_(step.dec_lse, non_blocking=True)
                ev["dec"][layer][1].record(stream)
                if s == 0:
                    h2d += nd * W.HQ * W.HEAD_DIM * 2
                    d2h += out_dec.numel() * 2 + lse_dec.numel() * 4
        torch.cuda.synchronize()
        if nd:
            t_dec += elapsed(ev["dec"])
        if step.n_chunk_rows:
            t_pf += elapsed(ev["pf"])
    dec = step.dec_bytes * L * steps / t_dec / 1e9 if nd else None
    pf = step.pf_flops * L * steps / t_pf / 1e12 if step.n_chunk_rows else None
    return dec, pf, h2d, d2h


# ----------------------------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ----------------------------------------------------------------------------------------------
def cpu_baseline(step: Step, budget_s: float = 10.0, prefill_budget_s: float = 4.0,
                 full_pass: bool = True):
    """The oracle on the host cores over a bounded sample of the step's layer 0: its decode
    sequences, cycled until ``budget_s`` has passed (and at least once each if ``full_pass``),
    and 64-row groups of its prefill chunk (from the last rows back, at least one group) until
    ``prefill_budget_s`` has passed."""
    import oracle
    inp = step.inp
    cores = len(os.sched_getaffinity(0))
    kp = inp.k_pools[0].view(torch.int16).cpu().numpy()
    vp = inp.v_pools[0].view(torch.int16).cpu().numpy()
    q = inp.q[0].view(torch.int16).cpu().numpy()
    res = {}
    if len(step.dec_idx):
        n0 = step.n_chunk_rows
        bt = inp.host_block_table[len(step.chunk_idx):]
        sl = inp.host_seq_lens[len(step.chunk_idx):]
        t0 = time.perf_counter()
        done = 0
        calls = 0
        need = len(sl) if full_pass else 1
        while True:
            b = calls % len(sl)
            oracle.decode(q[n0:], kp, vp, bt, sl, inp.scale, seqs=[b], threads=cores)
            done += int(sl[b])
            calls += 1
            if calls >= need and time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        res["decode"] = {"value": done * W.kv_bytes_per_token() / dt / 1e9, "unit": "GB/s",
                         "sample": f"oracle decode of the {len(sl)} sequence(s) of layer 0, "
                                   f"{calls / len(sl):.2f} passes ({done} cached tokens), {dt:.1f} s"}
    if step.n_chunk_rows:
        n = step.n_chunk_rows
        L0 = int(inp.host_seq_lens[0])
        t0 = time.perf_counter()
        pairs = 0
        done_rows = 0
        while done_rows < n and (done_rows == 0 or time.perf_counter() - t0 < prefill_budget_s):
            rows = list(range(max(0, n - done_rows - 64), n - done_rows))
            oracle.prefill(q[:n], [0, n], kp, vp, inp.host_block_table[:1], inp.host_seq_lens[:1],
                           inp.scale, rows=rows, threads=cores)
            pairs += sum(L0 - n + r + 1 for r in rows)
            done_rows += len(rows)
        dt = time.perf_counter() - t0
        res["prefill"] = {"value": prefill_flops(pairs) / dt / 1e12, "unit": "TFLOP/s",
                          "sample": f"oracle prefill of the last {done_rows} chunk rows x 16 heads "
                                    f"of layer 0, {dt:.1f} s"}
    return res, cores


# ----------------------------------------------------------------------------------------------
# CUDA-graph replay: the C-ABI calls are capture-safe (grids from host bounds, no host sync),
# so each timed phase is captured once and replayed; the device time then has no host gaps.
# ----------------------------------------------------------------------------------------------
def capture(step: Step, parts, split=None):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run(parts=parts, split=split)
    return g


def max_over_ranks(dist, values, device):
    """Element-wise maximum of per-rank timings (every rank gets the result)."""
    if dist is None:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def weak_scaling_rate(units_per_rank, n_ranks, seconds):
    """Whole-job throughput: every rank processed units_per_rank in at most `seconds`."""
    return units_per_rank * n_ranks / seconds


def timed_replays(graph, steps, warmup, dist):
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return a.elapsed_time(b) / 1e3


# ----------------------------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="mixed_28l",
                    choices=sorted(W.CONFIG_SEED) + ["adaptor_90min", "decode_graph_buckets",
                                                     "prefill_ragged_mix"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-buckets", action="store_true",
                    help="skip the decode batch-bucket latencies added to the default line")
    ap.add_argument("--clocks-out", default=None)
    ap.add_argument("--decode-ctas", type=int, default=-1,
                    help="whole-step graph: CTAs of each layer's decode, run on a second stream "
                         "beside the prefill on the other SMs (-1: 43.5%% of the SMs; 0: one after "
                         "the other)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import long_context_paged_gb300 as pa
    pa.load()
    dev = f"cuda:{local}"
    if args.workload == "adaptor_90min":
        return run_adaptor(pa, args, dev, dist, world, rank)
    if args.workload == "decode_graph_buckets":
        return run_decode_buckets(pa, args, dev, dist, world, rank)
    if args.workload == "prefill_ragged_mix":
        return run_prefill_ragged(pa, args, dev, dist, world, rank)
    step = Step(pa, args.workload, dev)
    hbm, bf16, bf16s, peak_src = peaks()

    step.run()                      # first eager pass: per-device one-time set-up
    torch.cuda.synchronize()
    flags = pa.read_device_status(step.status)
    if flags:
        raise RuntimeError(f"device status flagged errors in the first pass: {flags}")
    has_dec, has_pf = len(step.dec_idx) > 0, step.n_chunk_rows > 0
    # The whole step: after each layer's append, the chunk's prefill (tensor-bound) and the
    # decode batch (HBM-bound) run side by side on disjoint SMs; the per-mode graphs below keep
    # each call alone on the whole GPU (that is where the decode and prefill rates come from).
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    step_split = None
    if has_dec and has_pf and args.decode_ctas != 0:
        nd = round(0.435 * sms) if args.decode_ctas < 0 else min(args.decode_ctas, sms - 1)
        step_split = (sms - nd, nd)
    g_step = capture(step, ("append", "prefill", "decode"), split=step_split)
    g_dec = capture(step, ("decode",)) if has_dec else None
    g_pf = capture(step, ("prefill",)) if has_pf and has_dec else None

    sampler = ClockSampler(args.clocks_out)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    W_, K_ = max(args.warmup, 0), args.steps
    total_s = timed_replays(g_step, K_, W_, dist)
    t_dec = timed_replays(g_dec, K_, W_, dist) if g_dec is not None else 0.0
    t_pf = timed_replays(g_pf, K_, W_, dist) if g_pf is not None else 0.0
    if has_pf and not has_dec:
        t_pf = total_s
    if has_dec and not has_pf and not step.append:
        t_dec = total_s
    clocks = sampler.stop(device_uuid()) if rank == 0 else None
    total_s, t_dec, t_pf = max_over_ranks(dist, [total_s, t_dec, t_pf], dev)
    n = world
    launches = K_ * (step.launches_per_step + (step.dec_kernels * step.layers if g_dec is not None else 0)
                     + (2 * step.layers if g_pf is not None else 0))
    dec_gbs = weak_scaling_rate(step.dec_bytes * step.layers * K_, n, t_dec) / 1e9 if t_dec else None
    pf_tflops = weak_scaling_rate(step.pf_flops * step.layers * K_, n, t_pf) / 1e12 if t_pf else None

    if pa.read_device_status(step.status):
        raise RuntimeError("device status flagged errors in the timed region")

    buckets = None
    if args.workload == "mixed_28l" and not args.no_buckets:
        buckets = bucket_latencies(pa, dev, dist, args.warmup)

    e2e = None
    if not args.no_e2e:
        e_dec, e_pf, h2d, d2h = e2e_run(step, max(1, min(args.steps, 3)))
        e2e = {"value": None if e_dec is None else round(e_dec * n, 1), "unit": "GB/s",
               "prefill_value": None if e_pf is None else round(e_pf * n, 2),
               "prefill_unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        res, cores = cpu_baseline(step)
        main_key = "decode" if "decode" in res else "prefill"
        cpu = {"value": round(res[main_key]["value"], 4), "unit": res[main_key]["unit"],
               "cores": cores, "kind": "oracle", "sample": res[main_key]["sample"]}
        if main_key == "decode" and "prefill" in res:
            cpu["prefill"] = {"value": round(res["prefill"]["value"], 5), "unit": "TFLOP/s",
                              "sample": res["prefill"]["sample"]}

    # roofline of the dominant kernel (by device time), the other one alongside
    dec_src = source_hash("decode.cu", "pa_common.cuh", "cluster_common.cuh")
    pf_src = source_hash("prefill_tc.cu", "tc_common.cuh", "pa_common.cuh")
    roofs = []
    if t_dec:
        per_launch_s = t_dec / (step.layers * K_)
        ach = step.dec_bytes / per_launch_s / 1e9
        split = step.dec_kernels == 2   # else the single-launch short-batch path
        roofs.append((t_dec, {"kernel": "attn_decode_paged (" + ("decode_splitkv + merge" if split else
                                                                  "decode_cluster, one launch") + ")",
                              "bound": "hbm",
                              "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                              "frac": round(ach / hbm, 4), "peak_source": f"{peak_src} hbm_gbs (a read+write copy)",
                              "frac_of_nominal_8tbs": round(ach / NOMINAL_HBM_GBS, 4),
                              "traffic": traffic_from_profile("decode_splitkv_decode_b16_l27k.md", dec_src,
                                                              step.dec_bytes) if split else None,
                              "traffic_source": "ncu dram bytes of decode_b16_l27k per algorithmic byte x "
                                                "this launch's algorithmic bytes",
                              "algorithmic_bytes_per_launch": step.dec_bytes}))
    if t_pf:
        per_launch_s = t_pf / (step.layers * K_)
        ach = step.pf_flops / per_launch_s / 1e12
        pk = bf16s if step.layers > 1 else bf16
        roofs.append((t_pf, {"kernel": "attn_prefill_chunk", "bound": "tensor",
                             "achieved": round(ach, 2), "peak": pk, "unit": "TFLOP/s",
                             "frac": round(ach / pk, 4),
                             "peak_source": f"{peak_src} bf16_tflops" + ("_sustained" if step.layers > 1 else ""),
                             "traffic": traffic_from_profile("prefill_tc_prefill_4096_at_32768.md", pf_src,
                                                             step.pf_bytes),
                             "traffic_source": "ncu dram bytes of prefill_4096_at_32768 (the mixed step's "
                                               "prefill launch alone) per algorithmic byte x this launch's",
                             "algorithmic_flops_per_launch": step.pf_flops,
                             "algorithmic_bytes_per_launch": step.pf_bytes}))
    roofs.sort(key=lambda x: -x[0])

    L = step.inp.host_seq_lens
    value = dec_gbs if dec_gbs is not None else pf_tflops
    unit = "GB/s" if dec_gbs is not None else "TFLOP/s"
    line = {
        "metric": "paged GQA attn: decode KV-read GB/s (% HBM peak); prefill-chunk TFLOP/s (% peak)",
        "value": round(value, 2), "unit": unit, "n_gpus": n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_s * 1e3 / K_, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, paged 16, scattered pages)",
        "config": {"workload": args.workload, "layers": step.layers,
                   "decode_seqs": int(len(step.dec_idx)),
                   "decode_kv_tokens": int(L[step.dec_idx].sum()) if len(step.dec_idx) else 0,
                   "prefill_chunk": step.n_chunk_rows,
                   "prefill_offset": int(L[0] - step.n_chunk_rows) if step.n_chunk_rows else None,
                   "heads": "16q/8kv", "head_dim": 128, "page_size": 16,
                   "parallelism": f"replicas x{n}",
                   "l2": "inputs larger than L2 (each step reads every layer's pools)",
                   "timing": "CUDA events around K CUDA-graph replays each of: the whole step "
                             "(ms_per_step), its decode calls only (decode GB/s), its prefill "
                             "calls only (prefill TFLOP/s)",
                   "step_overlap": None if step_split is None else
                   {"prefill_ctas": step_split[0], "decode_ctas": step_split[1],
                    "how": "per layer, after kv_append: prefill and decode on two streams, "
                           "each call's persistent grid capped at its share of the SMs"}},
        "phase_ms_per_step": {"step": round(total_s * 1e3 / K_, 3),
                              "decode": round(t_dec * 1e3 / K_, 3) if t_dec else None,
                              "prefill": round(t_pf * 1e3 / K_, 3) if t_pf else None},
        "decode": None if dec_gbs is None else {"value": round(dec_gbs, 1), "unit": "GB/s",
                                                 "frac_of_hbm_peak": round(dec_gbs / hbm, 4),
                                                 "frac_of_nominal_8tbs": round(dec_gbs / NOMINAL_HBM_GBS, 4)},
        "prefill": None if pf_tflops is None else {"value": round(pf_tflops, 2), "unit": "TFLOP/s",
                                                    "frac_of_bf16_peak": round(pf_tflops / (bf16s if step.layers > 1 else bf16), 4)},
        "roofline": roofs[0][1] if roofs else None,
        "roofline_other": [r[1] for r in roofs[1:]],
        "decode_buckets": buckets,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16s,
                  "source": peak_src},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_adaptor(pa, args, dev, dist, world, rank):
    """4x temporal merge + adaptor MLP for 90 minutes of audio (270,000 frames -> 67,500
    embeddings): two tcgen05 GEMMs (4096 -> 1024 with SiLU, 1024 -> 1024) and a LayerNorm."""
    n_frames = 270_000
    inp = W.make_adaptor(W.ADAPTOR_SEED, n_frames, device=dev)
    T = n_frames // 4
    out = torch.empty(T, 1024, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pa.adaptor_workspace_size(n_frames), dtype=torch.uint8, device=dev)
    call = lambda: pa.adaptor_mlp_merge4(inp.frames, inp.w1, inp.b1, inp.w2, inp.b2, inp.gamma,
                                         inp.beta, inp.eps, out=out, workspace=ws)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    sampler = ClockSampler(args.clocks_out)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    t = timed_replays(g, args.steps, max(args.warmup, 0), dist)
    clocks = sampler.stop(device_uuid()) if rank == 0 else None
    (t,) = max_over_ranks(dist, [t], dev)
    flops = 2.0 * T * 1024 * (4096 + 1024)
    tflops = weak_scaling_rate(flops * args.steps, world, t) / 1e12
    hbm, bf16, bf16s, peak_src = peaks()
    if rank == 0:
        print(json.dumps({
            "metric": "adaptor (4x merge + Linear-SiLU-Linear-LayerNorm) TFLOP/s", "value": round(tflops, 1),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "adaptor_90min", "frames": n_frames, "tokens": T,
                       "timing": "CUDA events around CUDA-graph replays of the call"},
            "roofline": {"kernel": "gemm_bias_act (two GEMMs) + layernorm", "bound": "tensor",
                         "achieved": round(tflops, 1), "peak": bf16, "unit": "TFLOP/s",
                         "frac": round(tflops / bf16, 4), "peak_source": f"{peak_src} bf16_tflops",
                         "traffic": None, "algorithmic_flops_per_launch": flops},
            "gpu_launches": 3 * args.steps, "clocks": clocks}), flush=True)


def run_prefill_ragged(pa, args, dev, dist, world, rank):
    """Several requests' prompt chunks coalesced into one attn_prefill_chunk call: chunks of
    4,096 / 2,048 / 1,024 / 512 queries at offsets 28,672 / 61,440 / 10,000 / 0 (a new request),
    plus a 1-token and a 2-token extend, as a scheduler packs a prefill step."""
    inp = W.make_ragged_prefill(device=dev)
    q_lens, seq_lens = inp.host_q_lens, inp.host_seq_lens
    rows = int(q_lens.sum())
    max_s = int(seq_lens.max())
    out = torch.empty(rows, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, W.HQ, dtype=torch.float32, device=dev)
    ws = torch.empty(pa.prefill_workspace_size(len(q_lens), int(q_lens.max()), max_s),
                     dtype=torch.uint8, device=dev)
    call = lambda: pa.attn_prefill_chunk(inp.q[0], inp.cu_q_lens, inp.k_pools[0], inp.v_pools[0],
                                         inp.block_table, inp.seq_lens, int(q_lens.max()), max_s,
                                         inp.scale, out=out, lse=lse, workspace=ws)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    sampler = ClockSampler(args.clocks_out)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    (t,) = max_over_ranks(dist, [timed_replays(g, args.steps, max(args.warmup, 0), dist)], dev)
    clocks = sampler.stop(device_uuid()) if rank == 0 else None
    flops = prefill_flops(sum(prefill_pairs(int(L), int(q)) for L, q in zip(seq_lens, q_lens)))
    tflops = weak_scaling_rate(flops * args.steps, world, t) / 1e12
    hbm, bf16, bf16s, peak_src = peaks()
    if rank == 0:
        print(json.dumps({
            "metric": "paged GQA attn: prefill-chunk TFLOP/s, ragged multi-request call",
            "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V, paged 16, scattered pages)",
            "config": {"workload": "prefill_ragged_mix", "chunks": [list(x) for x in W.RAGGED_PREFILL_MIX],
                       "query_rows": rows, "timing": "CUDA events around CUDA-graph replays of the call"},
            "roofline": {"kernel": "attn_prefill_chunk", "bound": "tensor", "achieved": round(tflops, 2),
                         "peak": bf16, "unit": "TFLOP/s", "frac": round(tflops / bf16, 4),
                         "peak_source": f"{peak_src} bf16_tflops", "traffic": None,
                         "algorithmic_flops_per_launch": flops},
            "gpu_launches": 2 * args.steps, "clocks": clocks}), flush=True)


def bucket_latencies(pa, dev, dist, warmup, layers=28, seq_len=1000):
    """Decode latency by batch bucket, the way a serving engine replays CUDA graphs: B = 1, 2,
    4, 8, 16, 32 sequences of ``seq_len`` cached tokens (80 s of audio each), each layer with
    its own pools. Two figures per bucket: microseconds per decode call inside one graph of
    ``layers`` calls (one per layer, as in a decoder step's graph), and microseconds per replay
    of a graph holding a single call (which adds the graph launch itself)."""
    per_call, single, gbs, kernels = {}, {}, {}, {}
    for B in BUCKETS:
        kernels[str(B)] = pa.decode_kernels_per_call(B, seq_len)
        seed = W.CONFIG_SEED["decode_b1_l1000"] + B
        inp = W.make_paged(seed, np.full(B, seq_len), np.ones(B, np.int64), layers=layers,
                           device=dev, with_new_kv=False)
        out = torch.empty(B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, W.HQ, dtype=torch.float32, device=dev)
        ws = torch.empty(pa.decode_workspace_size(B, seq_len), dtype=torch.uint8, device=dev)
        call = lambda l: pa.attn_decode_paged(inp.q[l], inp.k_pools[l], inp.v_pools[l],
                                              inp.block_table, inp.seq_lens, seq_len, inp.scale,
                                              out=out, lse=lse, workspace=ws)
        call(0)
        torch.cuda.synchronize()
        g_all, g_one = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all):
            for l in range(layers):
                call(l)
        with torch.cuda.graph(g_one):
            call(0)
        reps = 200
        (t_all,) = max_over_ranks(dist, [timed_replays(g_all, reps, max(warmup, 3) * 5, dist)], dev)
        (t_one,) = max_over_ranks(dist, [timed_replays(g_one, reps * 10, max(warmup, 3) * 50, dist)], dev)
        per_call[str(B)] = round(t_all / (reps * layers) * 1e6, 2)
        single[str(B)] = round(t_one / (reps * 10) * 1e6, 2)
        gbs[str(B)] = round(B * seq_len * W.kv_bytes_per_token() / (t_all / (reps * layers)) / 1e9, 1)
        del g_all, g_one, inp
        torch.cuda.empty_cache()
    return {"seq_len": seq_len, "us_per_call_in_layer_graph": per_call,
            "us_per_single_call_graph_replay": single, "kv_read_gbs_in_layer_graph": gbs,
            "kernels_per_call": kernels, "layers_per_graph": layers}


def run_decode_buckets(pa, args, dev, dist, world, rank):
    """Decode-step latency by batch bucket (see bucket_latencies). The one-sequence bucket is
    the single-stream decode configuration."""
    sampler = ClockSampler(args.clocks_out)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    res = bucket_latencies(pa, dev, dist, args.warmup)
    clocks = sampler.stop(device_uuid()) if rank == 0 else None
    hbm, bf16, bf16s, peak_src = peaks()
    lat = res["us_per_call_in_layer_graph"]
    g32 = res["kv_read_gbs_in_layer_graph"]["32"]
    if rank == 0:
        print(json.dumps({
            "metric": "decode latency by batch bucket (CUDA-graph replay), us per call", "value": lat["1"],
            "unit": "us", "n_gpus": world, "steps": 200, "warmup": max(args.warmup, 3) * 5,
            "ms_per_step": round(lat["1"] / 1e3, 5), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode_graph_buckets", "seq_len": res["seq_len"], "buckets": list(BUCKETS),
                       "timing": "CUDA events around back-to-back replays of a 28-call graph (one call per "
                                 "layer) and of a one-call graph, per bucket"},
            "buckets": res,
            "roofline": {"kernel": "attn_decode_paged (decode_splitkv + merge at 32 sequences)",
                         "bound": "hbm", "achieved": g32, "peak": hbm, "unit": "GB/s",
                         "frac": round(g32 / hbm, 4), "peak_source": f"{peak_src} hbm_gbs",
                         "traffic": None, "note": "at the 32-sequence bucket; small buckets are latency-bound"},
            "gpu_launches": 200 * (28 + 10) * sum(res["kernels_per_call"].values()),
            "clocks": clocks}), flush=True)


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle  # noqa: F401
    name = args.workload
    L, ql = W.lengths_for(name)
    # only the data the sampled work touches is generated (on the host)
    cores = len(os.sched_getaffinity(0))
    inp = W.make_workload(name, device="cpu", layers=1) if name != "mixed_28l" else \
        W.make_paged(W.CONFIG_SEED[name], L, ql, pool_factor=1.0, extra_pages=16, layers=1)
    step = type("S", (), {})()
    step.inp = inp
    is_chunk = inp.host_q_lens > 1
    step.chunk_idx = np.nonzero(is_chunk)[0]
    step.dec_idx = np.nonzero(~is_chunk)[0]
    step.n_chunk_rows = int(inp.host_q_lens[step.chunk_idx].sum()) if len(step.chunk_idx) else 0
    budget = max(2.0, 20.0 / max(1, args.steps + args.warmup))
    vals, pvals = [], []
    sample = None
    for i in range(args.warmup + args.steps):
        res, _ = cpu_baseline(step, budget_s=budget, prefill_budget_s=0.0, full_pass=False)
        if i >= args.warmup:
            k = "decode" if "decode" in res else "prefill"
            vals.append(res[k]["value"])
            sample = res[k]["sample"]
            unit = res[k]["unit"]
            if "prefill" in res and k == "decode":
                pvals.append(res["prefill"]["value"])
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": "paged GQA attn: decode KV-read GB/s (% HBM peak); prefill-chunk TFLOP/s (% peak)",
            "value": round(v, 4), "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": {"workload": name},
            "cpu_baseline": {"value": round(v, 4), "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "prefill": {"value": round(statistics.median(pvals), 5), "unit": "TFLOP/s"} if pvals else None,
            "e2e": {"value": round(v, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
