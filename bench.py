#!/usr/bin/env python
"""DSA decode benchmark (one GPU per process; torchrun for N > 1).

A step is one pass of the whole hot path over one batch: write the batch's new tokens
into the paged caches (MXFP8 indexer keys, FP8 latent rows), run the fused Lightning
Indexer + Top-K over the paged MXFP8 K-cache, then Sparse Flash Attention over the
selected latent rows.  The workload is the decode batch of 32 sequences x 32768 tokens
(indexer 64 heads x 128, Top-K 2048, SFA 128 heads x 576, page size 64, shuffled pages),
synthetic and seeded.  Prints one JSON line (rank 0).

Timing: W warm-up steps, then K steps timed with CUDA events on the launching stream,
an L2 flush (a 256 MB write, outside the events) before every step, max over ranks.

--impl reference times the CPU oracle (float64 numpy) on a bounded sample of the same
workload instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA decode tokens/sec (indexer+TopK+SFA) and achieved HBM GB/s vs 8 TB/s"
K_BYTES_PER_TOKEN = 132     # 128 E4M3 codes + 4 E8M0 scales per cached indexer key
KV_BYTES_PER_ENTRY = 596    # 576 E4M3 codes + 5 fp32 tile scales per gathered latent row


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode_b32_ctx32k")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="approximate CPU time budget of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


# ---- clocks sampled during the timed region -------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, f in enumerate(fl) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---- the GPU arm ------------------------------------------------------------------------

def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "dsa_sparse_attention_topk_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel, sha):
    """dram bytes per launch from the committed ncu summary, if it was taken on this
    exact kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel)
    if not d or d.get("source_sha") != sha:
        return None
    return d.get("dram_bytes_per_launch")


def max_over_ranks(values, device):
    """The element-wise maximum of `values` over every rank (one all-reduce): the slowest
    rank's times are the job's."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def rows_per_second(rows_per_rank, world, ms_per_step):
    """Whole-job throughput: every rank's query rows per step over the (slowest) step time."""
    return rows_per_rank * world / (ms_per_step * 1e-3)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import dsa_sparse_attention_topk_gb300 as dsa
    from dsa_sparse_attention_topk_gb300 import workloads as W
    from dsa_sparse_attention_topk_gb300.layer import DsaDecodeLayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    dsa.lib()

    wl = W.make(args.workload)
    layer = DsaDecodeLayer(wl.num_pages, wl.h_i, wl.h_s, wl.topk, wl.sm_scale, dev)
    q_idx_cpu, w_cpu = wl.q_index(), wl.weights()
    q_sfa_cpu = wl.q_sfa()
    k_new, kv_new, s_new = [], [], []
    for b in range(wl.B):
        k, kv = wl.k_seq(b, q_idx_cpu, w_cpu), wl.kv_seq(b)
        slots = wl.slot_mapping(b)
        layer.write(k.to(dev), kv.to(dev), torch.from_numpy(slots).to(dev))
        pos = wl.q_pos[wl.q_seq == b]
        k_new.append(k[pos]); kv_new.append(kv[pos]); s_new.append(torch.from_numpy(slots[pos]))
    host = {
        "k_new": torch.cat(k_new), "kv_new": torch.cat(kv_new), "s_new": torch.cat(s_new),
        "q_idx": q_idx_cpu, "w": w_cpu, "q_sfa": q_sfa_cpu,
        "page_table": torch.from_numpy(wl.page_table), "seq_lens": torch.from_numpy(wl.seq_lens),
        "q_seq": torch.from_numpy(wl.q_seq), "q_pos": torch.from_numpy(wl.q_pos),
    }
    d = {k: v.to(dev) for k, v in host.items()}
    torch.cuda.synchronize()
    assert dsa.device_status() == 0

    n_q = wl.n_q
    idx = torch.empty(n_q, wl.topk, dtype=torch.int32, device=dev)
    out = torch.empty(n_q, wl.h_s, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(n_q, wl.h_s, dtype=torch.float32, device=dev)
    ws_n = dsa.sparse_attn_workspace_size(n_q, wl.h_s, wl.topk)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev) if ws_n else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(inner=False):
        if not inner:
            # a decode step as DsaDecodeLayer.step issues it: one library call
            dsa.decode_step(d["k_new"], d["kv_new"], d["s_new"], layer.k_cache, layer.kv_cache, d["q_idx"],
                            d["w"], d["q_sfa"], d["page_table"], d["seq_lens"], d["q_seq"], d["q_pos"], wl.topk,
                            wl.max_ctx, wl.sm_scale, q_group=wl.q_group, out_idx=idx, out=out, out_lse=lse,
                            workspace=ws)
            return
        # the per-kernel breakdown: the same three stages as separate calls, events between
        dsa.quant_kv(d["k_new"], d["kv_new"], d["s_new"], layer.k_cache, layer.kv_cache)
        ev[1].record()
        dsa.indexer_topk(d["q_idx"], d["w"], layer.k_cache, d["page_table"], d["seq_lens"], d["q_seq"],
                         d["q_pos"], wl.topk, wl.max_ctx, q_group=wl.q_group, out_idx=idx)
        ev[2].record()
        dsa.sparse_attn(d["q_sfa"], layer.kv_cache, d["page_table"], d["seq_lens"], d["q_seq"], idx,
                        wl.sm_scale, out=out, out_lse=lse, workspace=ws)

    # the step writes its new tokens inside the indexer (one per query row), then SFA and,
    # with several splits, the split merge
    fused = d["k_new"].shape[0] == n_q
    launches_per_step = (0 if fused else 1) + 2 + (1 if ws_n else 0)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        ev[0].record(); step(); ev[3].record()
    torch.cuda.synchronize()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device())
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.05)
    for i in range(K):
        flush.zero_()
        ev = evs[i]
        ev[0].record(); step(); ev[3].record()
    torch.cuda.synchronize()
    time.sleep(0.05)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    t_step = sum(e[0].elapsed_time(e[3]) for e in evs) / K   # ms
    # per-kernel breakdown from a second pass with events between the kernels (they can
    # keep consecutive kernels from overlapping, so the headline comes from the pass above)
    Kb = min(K, 100)
    for i in range(Kb):
        flush.zero_()
        ev = evs[i]
        ev[0].record(); step(inner=True); ev[3].record()
    torch.cuda.synchronize()
    t_write = sum(e[0].elapsed_time(e[1]) for e in evs[:Kb]) / Kb
    t_idx = sum(e[1].elapsed_time(e[2]) for e in evs[:Kb]) / Kb
    t_sfa = sum(e[2].elapsed_time(e[3]) for e in evs[:Kb]) / Kb
    assert dsa.device_status() == 0

    # ---- end to end through the public API, host buffers, copies inside the region ----
    # every input of a step lives in one pinned staging buffer (256-byte aligned slices), so
    # a step's inputs go to the device in one copy, as a serving loop would stage them
    offs, nbytes = {}, 0
    for k, v in host.items():
        offs[k] = nbytes
        nbytes = (nbytes + v.numel() * v.element_size() + 255) // 256 * 256

    def slices(buf):
        return {k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                for k, v in host.items()}

    pin_buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for k, v in slices(pin_buf).items():
        v.copy_(host[k])
    dd = slices(dev_buf)
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = nbytes
    d2h = out_host.numel() * out_host.element_size()

    def e2e_eager():
        dev_buf.copy_(pin_buf, non_blocking=True)
        o, _, _ = layer.step(dd["k_new"], dd["kv_new"], dd["s_new"], dd["q_idx"], dd["w"], dd["q_sfa"],
                             dd["page_table"], dd["seq_lens"], dd["q_seq"], dd["q_pos"], wl.max_ctx,
                             wl.q_group)
        out_host.copy_(o, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # the same step recorded once as a CUDA graph (copy in, decode step, copy out) through
    # DsaDecodeLayer.capture_step, as a serving loop would replay it; the eager calls if the
    # capture is refused
    e2e_graph = False
    e2e_step = e2e_eager
    try:
        replay = layer.capture_step(
            dict(k_new=dd["k_new"], kv_new=dd["kv_new"], slots_new=dd["s_new"], q_idx=dd["q_idx"], w=dd["w"],
                 q_sfa=dd["q_sfa"], page_table=dd["page_table"], seq_lens=dd["seq_lens"], q_seq=dd["q_seq"],
                 q_pos=dd["q_pos"]),
            wl.max_ctx, wl.q_group, stage=(pin_buf, dev_buf), result=out_host)

        def e2e_step():
            replay()
            torch.cuda.current_stream().synchronize()
        e2e_graph = True
    except RuntimeError as exc:
        print(f"e2e: graph capture refused ({exc}); timing the eager calls", file=sys.stderr)

    for _ in range(3):
        flush.zero_(); torch.cuda.synchronize(); e2e_step()
    e2e_times = []
    for _ in range(args.e2e_steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    t_e2e = sum(e2e_times) / len(e2e_times)

    if world > 1:
        t_step, t_idx, t_sfa, t_write, t_e2e = max_over_ranks([t_step, t_idx, t_sfa, t_write, t_e2e], dev)

    peaks, peaks_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    n_max = np.array([min(int(wl.q_pos[r]) + 1, int(wl.seq_lens[wl.q_seq[r]])) for r in range(n_q)])
    groups = n_max.reshape(-1, wl.q_group).max(1)
    idx_bytes = int(groups.sum()) * K_BYTES_PER_TOKEN
    sel = np.minimum(n_max, wl.topk)
    kv_bytes = int(sel.sum()) * KV_BYTES_PER_ENTRY
    sfa_flops = float(sel.sum()) * wl.h_s * (576 + 512) * 2
    idx_flops = float(groups.sum()) * wl.q_group * wl.h_i * 128 * 2  # q . k over every scanned position
    step_bytes = idx_bytes + kv_bytes

    # dominant kernel by time share
    if t_idx >= t_sfa:
        dom, t_dom = "indexer", t_idx
        sha = source_sha("indexer_tc.cu", "topk_cluster.cuh", "tc_utils.cuh", "dsa_common.cuh", "quant_tok.cuh")
        ach = idx_bytes / (t_dom * 1e-3) / 1e9
        roof = {"kernel": "indexer_topk", "bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(ach / hbm, 4), "peak_source": peaks_src,
                "algorithmic_bytes_per_launch": idx_bytes}
    else:
        dom, t_dom = "sfa", t_sfa
        sha = source_sha("sfa_tc.cu", "tc_utils.cuh", "dsa_common.cuh")
        # bf16 tensor-core path; the kernel is timed alone, so the burst peak applies
        bf16 = peaks.get("bf16_tflops", 1900.0)
        ach = sfa_flops / (t_dom * 1e-3) / 1e12
        roof = {"kernel": "sparse_attn", "bound": "tensor", "achieved": round(ach, 1), "peak": bf16,
                "unit": "TFLOP/s", "frac": round(ach / bf16, 4), "peak_source": peaks_src,
                "algorithmic_flops_per_launch": sfa_flops}
    roof["traffic"] = traffic_for(dom, sha)
    roof["source_sha"] = sha

    value = rows_per_second(n_q, world, t_step)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(t_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "seq_len": wl.max_ctx, "query_rows": n_q,
                   "indexer_heads": wl.h_i, "topk": wl.topk, "sfa_heads": wl.h_s, "page_size": 64,
                   "l2": "flushed (256 MB write) before every step", "parallelism": f"replicas x{world}"},
        "path_roofline": {"algorithmic_bytes": step_bytes, "indexer_bytes": idx_bytes, "gathered_kv_bytes": kv_bytes,
                          "achieved_gbs": round(step_bytes / (t_step * 1e-3) / 1e9, 1), "peak_gbs": hbm,
                          "frac": round(step_bytes / (t_step * 1e-3) / 1e9 / hbm, 4), "peak_source": peaks_src},
        "kernels_ms": {"cache_write": round(t_write, 5), "indexer_topk": round(t_idx, 5),
                       "sparse_attn": round(t_sfa, 5)},
        "roofline": roof,
        # both kernels against their own bounds (the dominant one is "roofline" above): the
        # indexer against HBM and the FP8 tensor peak (nominally twice bf16's), SFA against
        # the bf16 tensor peak
        "kernel_rooflines": {
            "indexer_topk": {"bound": "hbm", "achieved_gbs": round(idx_bytes / (t_idx * 1e-3) / 1e9, 1),
                             "frac_hbm": round(idx_bytes / (t_idx * 1e-3) / 1e9 / hbm, 4),
                             "fp8_tflops": round(idx_flops / (t_idx * 1e-3) / 1e12, 1),
                             "frac_fp8": round(idx_flops / (t_idx * 1e-3) / 1e12 / (2 * peaks.get("bf16_tflops", 1900.0)), 4)},
            "sparse_attn": {"bound": "tensor", "bf16_tflops": round(sfa_flops / (t_sfa * 1e-3) / 1e12, 1),
                            "frac_bf16": round(sfa_flops / (t_sfa * 1e-3) / 1e12 / peaks.get("bf16_tflops", 1900.0), 4),
                            "achieved_gbs": round(kv_bytes / (t_sfa * 1e-3) / 1e9, 1)},
        },
        "e2e": {"value": round(rows_per_second(n_q, world, t_e2e * 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(t_e2e * 1e3, 4), "cuda_graph": e2e_graph},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---- the CPU oracle ----------------------------------------------------------------------

def _oracle_inputs(wl, rows):
    q_idx = wl.q_index().double().numpy()
    w = wl.weights().double().numpy()
    q_sfa = wl.q_sfa(rows).double().numpy()
    seqs = {}
    for r in rows:
        b = int(wl.q_seq[r])
        if b not in seqs:
            seqs[b] = (wl.k_seq(b).double().numpy(), wl.kv_seq(b).double().numpy())
    return q_idx, w, q_sfa, seqs


def _oracle_rows(wl, rows, inputs):
    import oracle
    q_idx, w, q_sfa, seqs = inputs
    oracle.decode_rows(range(len(rows)), [q_idx[r] for r in rows], [w[r] for r in rows],
                       [seqs[int(wl.q_seq[r])][0] for r in rows], list(q_sfa),
                       [seqs[int(wl.q_seq[r])][1] for r in rows], [int(wl.q_pos[r]) for r in rows],
                       [int(wl.seq_lens[wl.q_seq[r]]) for r in rows], wl.topk, wl.sm_scale)


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, budget_s):
    """The oracle, as it stands, on the first rows of the workload until ~budget_s."""
    rows_done, t_total = 0, 0.0
    r = 0
    while t_total < budget_s and r < wl.n_q:
        inputs = _oracle_inputs(wl, [r])
        t0 = time.perf_counter()
        _oracle_rows(wl, [r], inputs)
        t_total += time.perf_counter() - t0
        rows_done += 1
        r += 1
    return {"value": round(rows_done / t_total, 4), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{rows_done} of {wl.n_q} query rows of {wl.name} (whole path per row: quantise the "
                      f"row's k and selected kv, fp64 scores, Top-{wl.topk}, fp64 SFA); BLAS may use every "
                      f"core, elementwise numpy runs on one", "seconds": round(t_total, 2)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from dsa_sparse_attention_topk_gb300 import workloads as W
    wl = W.make(args.workload)
    W_ = max(3, args.warmup)
    times = []
    cache = {}
    for i in range(W_ + args.steps):
        r = i % wl.n_q
        if r not in cache:
            cache = {r: _oracle_inputs(wl, [r])}
        t0 = time.perf_counter()
        _oracle_rows(wl, [r], cache[r])
        dt = time.perf_counter() - t0
        if i >= W_:
            times.append(dt)
    t = sum(times) / len(times)
    value = 1.0 / t
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": W_, "ms_per_step": round(t * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.B, "seq_len": wl.max_ctx, "query_rows": wl.n_q,
                       "step": "one query row of the batch per step (bounded sample)"},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                             "sample": "one query row per step, rotating through the batch"},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
