"""Benchmark of one MLA decode step on B300: append + decode over a paged latent cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole hot path over one batch: mla_append of the
newest token of every sequence (latent RMSNorm, decoupled RoPE, paged row
write) followed by mla_decode (W_UK absorption, attention over every cached
token of every sequence, split combine and W_UV). The default workload is
DeepSeek-V2-shaped decode at the 128K context of the report's long-context
extension (128 heads, 512 + 64 latent row, bf16, batch 4, 131072 cached
tokens per sequence, 64-token pages shuffled in the pool); --workload picks
the others (dsv2_b16: batch 16 x 4096, ragged_b64, fp8_b32, yarn_b4).

Metric: cached tokens attended per second = sum_b L_b / step time. The cache
and weights are resident in HBM; L2 is flushed between timed steps, outside
the timed events: a 512 MiB memset (write) followed by a read of another
512 MiB buffer, so that the memset's dirty lines are written back before the
step starts rather than inside it. Under torchrun every rank runs its own
replica (weak scaling, no collective on the data path); rank 0 prints one
JSON line.

--impl reference times the fp64 CPU oracle (the slow, plain statement of the
method) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_synth as S  # noqa: E402

METRIC = "MLA decode cached-tokens attended/s on 1 B300; % of HBM/tensor roofline"
UNIT = "tokens/s"
FLOP_PER_HEAD_TOKEN = 2 * (576 + 512)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_b4", choices=sorted(S.SHAPES))
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget per measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--q-len", type=int, default=1,
                    help="new tokens decoded per sequence per step (multi-token prediction drafts); 1 = plain decode")
    ap.add_argument("--hidden", type=int, default=0,
                    help="take the decode output to this hidden size with W_UV folded into W_O (mla_decode_hidden)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int):
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens_per_rank: int, steps: int, slowest_seconds: float) -> float:
    """Whole-job throughput: every rank decodes its own replica of the workload (weak scaling),
    so the job attends world * tokens_per_rank cached tokens per step, timed by the slowest rank."""
    return world * tokens_per_rank * steps / slowest_seconds


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4) if r[3 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- the GPU arm

# the sources a kernel is built from (paths relative to the repository root); a committed ncu
# figure is used only while these files are unchanged
_CSRC = "head_latent_attention_22_b300/csrc/"
KERNEL_SOURCES = {
    "attend_tc": [_CSRC + "attend_pair.cuh", _CSRC + "decode_tc.cuh", _CSRC + "tc.cuh", _CSRC + "common.cuh"],
    "prefill_attn": [_CSRC + "prefill.cuh", _CSRC + "decode_tc.cuh", _CSRC + "tc.cuh", _CSRC + "common.cuh"],
    "kv_up": [_CSRC + "prefill.cuh", _CSRC + "decode_tc.cuh", _CSRC + "tc.cuh", _CSRC + "common.cuh"],
}


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summary, if it was
    captured on the kernel's present sources (same digest); None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path)).get(kernel, {}).get(workload)
        files = KERNEL_SOURCES[kernel]
    except (OSError, ValueError, AttributeError, KeyError):
        return None
    if not rec or rec.get("source_digest") != source_digest(files):
        return None
    return rec.get("dram_bytes_per_launch")


def out_groups_guess(hidden: int) -> int:
    """Contraction slices of the folded output GEMM (as the library picks them for this GPU); each
    writes one fp32 partial of [batch, hidden]."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    m_tiles = hidden // 128
    return max(1, min(64, (4 * sms + m_tiles - 1) // m_tiles))


def peaks():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, 1800.0, 1400.0, "fallback"


def run_gpu(args, rank, world, local):
    import head_latent_attention_22_b300 as M
    from head_latent_attention_22_b300 import build as B
    B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world)
    shape = S.SHAPES[args.workload]
    inp = S.make_inputs(shape)
    cfg = M.MLAConfig.from_shape(shape)
    B_, H = shape.batch, shape.n_heads
    q = args.q_len
    cache_tokens = int(inp.lengths.sum())
    # tokens attended per step: new token k of sequence b sees its first L_b - (q - 1 - k) rows
    tokens = int(sum(max(0, int(L) - (q - 1 - k)) for L in inp.lengths for k in range(q)))
    max_len = int(inp.lengths.max())

    # resident state: weights, page table, pool filled with every token
    pool = M.new_pool(cfg, inp.num_pages, dev)
    bt = torch.from_numpy(inp.block_table).to(dev)
    seq_lens = torch.from_numpy(inp.lengths.astype(np.int32)).to(dev)
    w_uk, w_uv = inp.w_uk.to(dev), inp.w_uv.to(dev)
    pos_all = torch.from_numpy(inp.positions())
    seq_all = torch.from_numpy(inp.seq_index())
    chunk = 1 << 20
    for s in range(0, cache_tokens, chunk):
        e = min(cache_tokens, s + chunk)
        M.append(cfg, inp.c_kv_raw[s:e].to(dev), inp.k_rope_raw[s:e].to(dev), pos_all[s:e].to(dev), pool, bt,
                 seq_idx=seq_all[s:e].to(dev))
    torch.cuda.synchronize()
    del pos_all, seq_all

    # the step's new tokens are each sequence's last q rows (rewritten by the step's append)
    new_pos = torch.from_numpy(np.array([int(L) - q + k for L in inp.lengths for k in range(q)], np.int32)).to(dev)
    new_seq = torch.from_numpy(np.repeat(np.arange(B_, dtype=np.int32), q)).to(dev)
    hid = args.hidden
    if hid:
        if q != 1:
            raise SystemExit("--hidden runs the single-token decode")
        w_ouv = M.fold_output_weight(cfg, w_uv, S.draw_w_o(shape, hid).to(dev))
        out = torch.empty((B_, hid), dtype=torch.float32, device=dev)
        ws = torch.empty(max(256, M.decode_hidden_workspace_size(cfg, B_, max_len, hid)), dtype=torch.uint8,
                         device=dev)
    elif q == 1:
        out = torch.empty((B_, H, shape.d_head), dtype=torch.float32, device=dev)
        ws = torch.empty(max(256, M.workspace_size(cfg, B_, max_len)), dtype=torch.uint8, device=dev)
    else:
        out = torch.empty((B_, q, H, shape.d_head), dtype=torch.float32, device=dev)
        ws = torch.empty(max(256, M.workspace_size_multi(cfg, B_, q, bt.shape[1], max_len)), dtype=torch.uint8,
                         device=dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.int64, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()
    n_steps = args.warmup + args.steps
    steps = [S.draw_step(inp, k) if q == 1 else S.draw_step_multi(inp, k, q) for k in range(min(n_steps, 8))]
    dsteps = [tuple(t.to(dev) for t in (st.q_nope, st.q_rope, st.c_new, st.k_new)) for st in steps]
    stream = torch.cuda.current_stream()

    def step(k, tensors=None):
        qn, qr, cn, kn = dsteps[k % len(dsteps)] if tensors is None else tensors
        M.append(cfg, cn, kn, new_pos, pool, bt, seq_idx=new_seq)
        if hid:
            M.decode_hidden(cfg, qn, qr, w_uk, w_ouv, pool, bt, seq_lens, max_len, out=out, workspace=ws)
        elif q == 1:
            M.decode(cfg, qn, qr, w_uk, w_uv, pool, bt, seq_lens, max_len, out=out, workspace=ws)
        else:
            M.decode_multi(cfg, qn, qr, w_uk, w_uv, pool, bt, seq_lens, max_len, out=out, workspace=ws)

    names = M.decode_stage_names(cfg)
    if hid:
        names = names[:3] + ["out_tc", "out_reduce"]
    launches_per_step = 1 + (q > 1) + len(names)
    for k in range(args.warmup):
        step(k)
        flush_l2()
    torch.cuda.synchronize()
    M.check_device_errors()

    # timed region: K steps, each bracketed by its own events; L2 flushed between steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            flush_l2()
            torch.cuda._sleep(2_000_000)   # the step's launches are all queued before its first event fires
            ev[k][0].record(stream)
            step(args.warmup + k)
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    M.check_device_errors()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(world, tokens, args.steps, total_ms / 1e3)

    # the decode alone (no append in the step), same timing rules
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for k in range(args.steps):
        qn, qr, _, _ = dsteps[(args.warmup + k) % len(dsteps)]
        flush_l2()
        torch.cuda._sleep(2_000_000)
        dev_ev[k][0].record(stream)
        if hid:
            M.decode_hidden(cfg, qn, qr, w_uk, w_ouv, pool, bt, seq_lens, max_len, out=out, workspace=ws)
        elif q == 1:
            M.decode(cfg, qn, qr, w_uk, w_uv, pool, bt, seq_lens, max_len, out=out, workspace=ws)
        else:
            M.decode_multi(cfg, qn, qr, w_uk, w_uv, pool, bt, seq_lens, max_len, out=out, workspace=ws)
        dev_ev[k][1].record(stream)
    torch.cuda.synchronize()
    dec_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in dev_ev), world, dev) / args.steps
    decode_only = {"ms_per_step": round(dec_ms, 5), "value": job_value(world, tokens, 1, dec_ms / 1e3),
                   "unit": UNIT}

    # per-kernel durations (separate pass, same steps, events between the kernels). A GPU-side
    # sleep ahead of each step lets the host enqueue all of the step's launches and events before
    # the first event fires, so an interval holds its kernel's GPU time and no host enqueue gap.
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush_l2()
        torch.cuda._sleep(2_000_000)
        M.set_stage_events(kev[k])
        step(args.warmup + k)
    M.set_stage_events(None)
    torch.cuda.synchronize()
    per_kernel = {n: statistics.mean(kev[k][i].elapsed_time(kev[k][i + 1]) for k in range(args.steps))
                  for i, n in enumerate(names)}
    dom = max(per_kernel, key=per_kernel.get)
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    row = M.cache_row_bytes(cfg)
    # the cache is read once per step (the q new tokens of a sequence share its pages), the queries
    # of every new token once
    attend_bytes = cache_tokens * row + B_ * q * H * (shape.d_c + shape.d_rope) * 2
    attend_flop = tokens * H * FLOP_PER_HEAD_TOKEN
    weight_bytes = 2 * H * shape.d_head * shape.d_c * (2 if shape.io_dtype == "bf16" else 4)
    if dom.startswith("attend"):
        alg_bytes, alg_flop = attend_bytes, attend_flop
    elif dom == "out_tc":
        alg_bytes = hid * H * shape.d_c * 2 + 2 * B_ * H * shape.d_c * 2 + 4 * B_ * hid * out_groups_guess(hid)
        alg_flop = 2 * 2 * B_ * hid * H * shape.d_c
    else:
        alg_bytes, alg_flop = weight_bytes / 2, 2 * B_ * H * shape.d_head * shape.d_c
    t = per_kernel[dom] / 1e3
    ach_gbs = alg_bytes / t / 1e9
    ach_tf = alg_flop / t / 1e12
    # the kernel's bound is whichever of its bytes over HBM and its FLOPs over the tensor peak takes longer
    tensor_bound = alg_flop / (tf_burst * 1e12) > alg_bytes / (hbm * 1e9)
    roofline = {"bound": "tensor" if tensor_bound else "hbm",
                "achieved": round(ach_tf if tensor_bound else ach_gbs, 1),
                "peak": tf_burst if tensor_bound else hbm, "unit": "TFLOP/s" if tensor_bound else "GB/s",
                "frac": round(ach_tf / tf_burst if tensor_bound else ach_gbs / hbm, 4),
                "traffic": committed_traffic(dom, shape.name + (f"_q{q}" if q > 1 else "")), "kernel": dom,
                "kernel_ms": round(per_kernel[dom], 5), "algorithmic_bytes": alg_bytes, "algorithmic_flop": alg_flop,
                "hbm_gbs": round(ach_gbs, 1), "hbm_peak": hbm, "tensor_tflops": round(ach_tf, 1),
                "tensor_peak": tf_burst,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json)" if peak_kind == "measured" else peak_kind,
                "per_kernel_ms": {k: round(v, 5) for k, v in per_kernel.items()}}
    # whole-step roofline: the slower of all bytes over HBM and all FLOPs over the tensor peak
    step_bytes = attend_bytes + weight_bytes + B_ * q * row
    step_flop = attend_flop + 4 * B_ * q * H * shape.d_head * shape.d_c
    if hid:   # W_UV's bytes and FLOPs replaced by the folded weight's (hi and lo operands of o_lat)
        step_bytes += hid * H * shape.d_c * 2 - weight_bytes / 2
        step_flop += 2 * 2 * B_ * hid * H * shape.d_c - 2 * B_ * H * shape.d_head * shape.d_c
    t_roof = max(step_bytes / (hbm * 1e9), step_flop / (tf_burst * 1e12))
    roofline["step_frac"] = round(t_roof / (ms_per_step / 1e3), 4)

    # end to end through the public API with host buffers (pinned), copies inside the timed region:
    # each step's inputs (q_nope, q_rope and the new tokens' raw latent and rope key) travel as one
    # pinned block, the step runs as a captured CUDA graph (M.StepGraph: mla_append + mla_decode),
    # and the outputs come back to pinned memory before the step counts as done
    srcs = [(st.q_nope, st.q_rope, st.c_new, st.k_new) for st in steps]
    nbytes = [t.numel() * t.element_size() for t in srcs[0]]
    offs, total = [], 0
    for n in nbytes:
        offs.append(total)
        total += (n + 255) // 256 * 256
    host = []
    for tensors in srcs:
        blk = torch.empty(total, dtype=torch.uint8).pin_memory()
        for t, o, n in zip(tensors, offs, nbytes):
            blk[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        host.append(blk)
    dblk = torch.empty(total, dtype=torch.uint8, device=dev)
    dv = [dblk[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(srcs[0], offs, nbytes)]
    dv_q_nope, dv_q_rope, dv_c_new, dv_k_new = dv
    dblk.copy_(host[0])
    if q == 1 and not hid:
        graph = M.StepGraph(cfg, c_new=dv_c_new, k_new=dv_k_new, positions=new_pos, seq_idx=new_seq,
                            q_nope=dv_q_nope, q_rope=dv_q_rope, w_uk=w_uk, w_uv=w_uv, pool=pool, block_table=bt,
                            seq_lens=seq_lens, max_seq_len=max_len, out=out, workspace=ws)
        run_step = graph.replay
        e2e_path = "M.StepGraph replay (CUDA graph of mla_append + mla_decode); inputs in one pinned block"
    else:
        def run_step():
            step(0, (dv_q_nope, dv_q_rope, dv_c_new, dv_k_new))
        e2e_path = "eager M.append + M.decode_multi calls; inputs in one pinned block"
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(nbytes)
    d2h = out_host.numel() * out_host.element_size()
    e2e_s = 0.0
    for k in range(args.warmup + args.steps):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dblk.copy_(host[k % len(host)], non_blocking=True)
        run_step()
        out_host.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if k >= args.warmup:
            e2e_s += time.perf_counter() - t0
    M.check_device_errors()
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e = {"value": job_value(world, tokens, args.steps, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * e2e_s / args.steps, 4),
           "path": e2e_path}

    res = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": shape.io_dtype if shape.cache_dtype != "fp8_e4m3_b128"
           else "bf16+fp8cache", "data": "synthetic (seeded; random-init weights)",
           "config": {"workload": shape.name, "batch": B_, "seq_len": max_len, "cached_tokens": cache_tokens,
                      "attended_tokens_per_step": tokens,
                      "n_heads": H, "d_c": shape.d_c, "d_rope": shape.d_rope, "d_head": shape.d_head,
                      "page_size": shape.page_size, "cache_dtype": shape.cache_dtype, "q_len": q,
                      "output": f"hidden {hid} (W_UV folded into W_O)" if hid else "per-head [B, H, d_head]",
                      "parallelism": f"replicas x{world}", "l2": "flushed between steps (512 MiB memset + 512 MiB read)",
                      "decode_path": "tcgen05" if M.decode_path(cfg) else "cuda-core"},
           "roofline": roofline, "e2e": e2e, "decode_only": decode_only,
           "gpu_launches": launches_per_step * args.steps,
           "pages_context": {"kv_cache_reduction_vs_67b": "93.3%",
                             "max_generation_throughput_vs_67b": "5.76x (end-to-end serving, 8x H800 node)",
                             "note": "the pages give no number for the decode kernel itself"},
           "clocks": clocks.summary()}
    return res, inp


PREFILL_METRIC = "MLA prefill prompt tokens/s on 1 B300 (non-absorbed form, causal); % of tensor roofline"


def prefill_flop(lengths, n_new, H=128, d_c=512, d_h=128, d_r=64) -> tuple:
    """Algorithmic FLOPs of one prefill: the K/V up-projection of every cached row (2 d_c x 2 H d_h
    per row) and, per head, the causal scores (d_h + d_r) and weighted values (d_h) of every new
    token against the rows up to its position."""
    up = sum(int(L) for L in lengths) * 2 * d_c * 2 * H * d_h
    pairs = sum(sum(int(L) - int(n) + k + 1 for k in range(int(n))) for L, n in zip(lengths, n_new))
    att = pairs * H * 2 * (d_h + d_r + d_h)
    return up, att


def run_prefill(args, rank, world, local):
    """One step = mla_prefill of every prompt of the workload (the prompts already in the cache)."""
    import head_latent_attention_22_b300 as M
    from head_latent_attention_22_b300 import build as B
    B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world)
    shape = S.SHAPES[args.workload]
    inp = S.make_inputs(shape)
    cfg = M.MLAConfig.from_shape(shape)
    pool = M.new_pool(cfg, inp.num_pages, dev)
    bt = torch.from_numpy(inp.block_table).to(dev)
    seq_lens = torch.from_numpy(inp.lengths.astype(np.int32)).to(dev)
    w_uk, w_uv = inp.w_uk.to(dev), inp.w_uv.to(dev)
    M.append(cfg, inp.c_kv_raw.to(dev), inp.k_rope_raw.to(dev), torch.from_numpy(inp.positions()).to(dev), pool, bt,
             seq_idx=torch.from_numpy(inp.seq_index()).to(dev))
    torch.cuda.synchronize()
    pfs = [S.draw_prefill(inp, step=k) for k in range(2)]
    dq = [(p.q_nope.to(dev), p.q_rope.to(dev)) for p in pfs]
    q_start = torch.from_numpy(pfs[0].q_start.astype(np.int32)).to(dev)
    T = int(pfs[0].q_start[-1])
    max_len = int(inp.lengths.max())
    out = torch.empty((T, shape.n_heads, shape.d_head), dtype=torch.float32, device=dev)
    ws = torch.empty(M.prefill_workspace_size(cfg, shape.batch, max_len), dtype=torch.uint8, device=dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.int64, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()

    def step(k, tensors=None):
        qn, qr = dq[k % len(dq)] if tensors is None else tensors
        M.prefill(cfg, qn, qr, w_uk, w_uv, pool, bt, seq_lens, q_start, max_len, out=out, workspace=ws)

    for k in range(args.warmup):
        step(k)
        flush_l2()
    torch.cuda.synchronize()
    M.check_device_errors()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            flush_l2()
            torch.cuda._sleep(2_000_000)
            ev[k][0].record(stream)
            step(args.warmup + k)
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    M.check_device_errors()
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(world, T, args.steps, total_ms / 1e3)
    # per-kernel times: events between the two kernels (programmatic dependent launch off)
    names = ["kv_up", "prefill_attn"]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush_l2()
        torch.cuda._sleep(2_000_000)
        M.set_stage_events(kev[k])
        step(args.warmup + k)
    M.set_stage_events(None)
    torch.cuda.synchronize()
    per_kernel = {n: statistics.mean(kev[k][i].elapsed_time(kev[k][i + 1]) for k in range(args.steps))
                  for i, n in enumerate(names)}
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    up, att = prefill_flop(inp.lengths, pfs[0].n_new)
    flop = {"kv_up": up, "prefill_attn": att}
    dom = max(per_kernel, key=per_kernel.get)
    ach = flop[dom] / (per_kernel[dom] / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(ach, 1), "peak": tf_burst, "unit": "TFLOP/s",
                "frac": round(ach / tf_burst, 4), "traffic": committed_traffic(dom, shape.name), "kernel": dom,
                "kernel_ms": round(per_kernel[dom], 5), "algorithmic_flop": flop[dom],
                "peak_source": peak_kind + " (MEASURED_PEAKS.json)" if peak_kind == "measured" else peak_kind,
                "per_kernel_ms": {k: round(v, 5) for k, v in per_kernel.items()},
                "per_kernel_tflops": {k: round(flop[k] / (per_kernel[k] / 1e3) / 1e12, 1) for k in names},
                "step_frac": round((up + att) / (tf_burst * 1e12) / (ms_per_step / 1e3), 4)}
    # end to end: queries from pinned host memory, outputs back to pinned host memory, every step
    hq = [(p.q_nope.pin_memory(), p.q_rope.pin_memory()) for p in pfs]
    dqn, dqr = torch.empty_like(dq[0][0]), torch.empty_like(dq[0][1])
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_s = 0.0
    for k in range(args.warmup + args.steps):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dqn.copy_(hq[k % 2][0], non_blocking=True)
        dqr.copy_(hq[k % 2][1], non_blocking=True)
        step(0, (dqn, dqr))
        out_host.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if k >= args.warmup:
            e2e_s += time.perf_counter() - t0
    M.check_device_errors()
    e2e_s = max_over_ranks(e2e_s, world, dev)
    h2d = dqn.numel() * 2 + dqr.numel() * 2
    e2e = {"value": job_value(world, T, args.steps, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": out_host.numel() * 4, "ms_per_step": round(1e3 * e2e_s / args.steps, 4),
           "path": "eager M.prefill; queries copied from pinned memory, fp32 outputs copied back"}
    res = {"metric": PREFILL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; random-init weights)",
           "config": {"workload": shape.name, "batch": shape.batch, "prompt_len": max_len, "prompt_tokens": T,
                      "n_heads": shape.n_heads, "d_c": shape.d_c, "d_rope": shape.d_rope, "d_head": shape.d_head,
                      "page_size": shape.page_size, "cache_dtype": shape.cache_dtype,
                      "parallelism": f"replicas x{world}",
                      "l2": "flushed between steps (512 MiB memset + 512 MiB read)"},
           "roofline": roofline, "e2e": e2e, "gpu_launches": 2 * args.steps,
           "pages_context": {"prefill_throughput": "above 100K tokens/s (whole model, 8x H800 node)"},
           "clocks": clocks.summary()}
    return res, inp


# ----------------------------------------------------------------------------- the oracle arm

def _sample_order(batch: int, n_heads: int, step: int):
    rng = np.random.default_rng(step)
    return [(int(b), int(i)) for b, i in zip(rng.integers(0, batch, 1 << 16), rng.integers(0, n_heads, 1 << 16))]


def oracle_prep(inp):
    """What timed oracle samples start from (not timed: it is resident state, the same for every
    step): the weights in fp64 and the cache content of up to 64 sequences the samples may touch."""
    from oracle import mla_oracle as O
    s = inp.shape
    inv_freq = O.yarn_inv_freq(s.d_rope, s.rope_theta, s.yarn_factor, s.yarn_alpha, s.yarn_beta, s.yarn_orig_len)
    cache = {}
    for b in sorted({b for b, _ in _sample_order(s.batch, s.n_heads, 0)[:64]}):
        o0, o1 = int(inp.token_offsets[b]), int(inp.token_offsets[b + 1]) - 1
        c, kr, _ = O.append_rows(inp.c_kv_raw[o0:o1].double().numpy(), inp.k_rope_raw[o0:o1].double().numpy(),
                                 np.arange(o1 - o0), cache_dtype=s.cache_dtype, eps=s.eps, theta=s.rope_theta,
                                 inv_freq=inv_freq)
        cache[b] = (c, kr)
    return {"cache": cache, "inv_freq": inv_freq, "w_uk": inp.w_uk.double().numpy(),
            "w_uv": inp.w_uv.double().numpy(), "scale": s.scale * O.yarn_logit_factor(s.yarn_factor, s.yarn_mscale)}


def oracle_sample(inp, seconds: float, step: int = 0, form: str = "absorbed", prep=None):
    """Time the fp64 oracle on a bounded sample of one step: the append of every
    sequence's newest token, then (sequence, head) decodes until the budget is used,
    in the absorbed form (W_UK folded into the query, the latent as the value) or the
    explicit one (per-head keys and values up-projected from the latent first)."""
    from oracle import mla_oracle as O
    s = inp.shape
    p = oracle_prep(inp) if prep is None else prep
    cache, inv_freq, scale, w_uk, w_uv = p["cache"], p["inv_freq"], p["scale"], p["w_uk"], p["w_uv"]
    st = S.draw_step(inp, step)   # the step's queries and new tokens
    qn, qr = st.q_nope.double().numpy(), st.q_rope.double().numpy()
    head = {"absorbed": O.head_absorbed, "explicit": O.head_explicit}[form]
    t0 = time.perf_counter()
    c_new, k_new, _ = O.append_rows(st.c_new.double().numpy(), st.k_new.double().numpy(), inp.lengths - 1,
                                    cache_dtype=s.cache_dtype, eps=s.eps, theta=s.rope_theta, inv_freq=inv_freq)
    done, tok = 0, 0
    for b, i in _sample_order(s.batch, s.n_heads, step):
        if b not in cache:
            continue
        c = np.concatenate([cache[b][0], c_new[b:b + 1]])
        kr = np.concatenate([cache[b][1], k_new[b:b + 1]])
        head(qn[b, i], qr[b, i], w_uk[i], w_uv[i], c, kr, scale)
        done += 1
        tok += len(c)
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    # a token attended = one cached token for all heads of its sequence
    return tok / s.n_heads / dt, done, dt


def blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max([x.get("num_threads", 1) for x in info] or [1])
    except Exception:
        return os.cpu_count() or 1


def host_cores():
    return os.cpu_count() or 1


def cpu_baseline(inp, seconds):
    """The fp64 oracle's absorbed form (the headline CPU number), and beside it the explicit form
    with half the time budget."""
    prep = oracle_prep(inp)
    v, done, dt = oracle_sample(inp, seconds, prep=prep)
    ve, done_e, dt_e = oracle_sample(inp, seconds / 2, form="explicit", prep=prep)
    return {"value": v, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": f"{done} (sequence, head) decodes of {inp.shape.name} in the fp64 absorbed form "
                      f"({dt:.1f} s), plus the append of the step's new tokens; tokens/s = cached tokens "
                      f"visited / n_heads / time; numpy's BLAS pool had {blas_threads()} threads",
            "explicit": {"value": ve, "unit": UNIT,
                         "sample": f"{done_e} (sequence, head) decodes in the fp64 explicit form (per-head keys "
                                   f"and values up-projected from the latent; {dt_e:.1f} s), same accounting"}}


def oracle_prefill_sample(inp, seconds: float, step: int = 0):
    """Time the fp64 oracle's prefill (explicit form) on a bounded sample of one prefill step:
    (sequence, head) pairs, all new tokens of each, until the budget is used. Returns prompt tokens
    per second (query rows per second over all heads / n_heads), the pairs done and the time."""
    from oracle import mla_oracle as O
    s = inp.shape
    pf = S.draw_prefill(inp, step=step)
    rng = np.random.default_rng(step)
    w_uk, w_uv = inp.w_uk.double().numpy(), inp.w_uv.double().numpy()
    qn, qr = pf.q_nope.double().numpy(), pf.q_rope.double().numpy()
    inv_freq = O.yarn_inv_freq(s.d_rope, s.rope_theta, s.yarn_factor, s.yarn_alpha, s.yarn_beta, s.yarn_orig_len)
    b = int(rng.integers(0, s.batch))
    o0, o1 = int(inp.token_offsets[b]), int(inp.token_offsets[b + 1])
    c, kr, _ = O.append_rows(inp.c_kv_raw[o0:o1].double().numpy(), inp.k_rope_raw[o0:o1].double().numpy(),
                             np.arange(o1 - o0), cache_dtype=s.cache_dtype, eps=s.eps, theta=s.rope_theta,
                             inv_freq=inv_freq)
    n = int(pf.n_new[b])
    rows = list(range(int(pf.q_start[b]), int(pf.q_start[b]) + n))
    cs = [c if k == b else np.zeros((0, s.d_c)) for k in range(s.batch)]
    ks = [kr if k == b else np.zeros((0, s.d_rope)) for k in range(s.batch)]
    n_new = [n if k == b else 0 for k in range(s.batch)]
    sl = slice(int(pf.q_start[b]), int(pf.q_start[b]) + n)
    t0 = time.perf_counter()
    done = 0
    for i in rng.permutation(s.n_heads):
        O.prefill(qn[sl], qr[sl], w_uk, w_uv, cs, ks, n_new, s.scale * O.yarn_logit_factor(s.yarn_factor, s.yarn_mscale),
                  heads=[int(i)])
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    return n * done / s.n_heads / dt, done, dt


def run_reference(args, rank, world):
    if rank != 0:
        return None
    shape = S.SHAPES[args.workload]
    inp = S.make_inputs(shape)
    if args.workload in S.PREFILL_SHAPES:
        vals, secs = [], 0.0
        per_step = max(0.5, args.cpu_seconds / max(1, args.steps))
        for k in range(args.warmup):
            oracle_prefill_sample(inp, min(1.0, args.cpu_seconds / 10), k)
        for k in range(args.steps):
            v, done, dt = oracle_prefill_sample(inp, per_step, args.warmup + k)
            vals.append(v)
            secs += dt
        value = float(np.mean(vals))
        return {"impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded; random-init weights)",
                "config": {"workload": shape.name, "batch": shape.batch, "prompt_len": int(inp.lengths.max()),
                           "n_heads": shape.n_heads, "cache_dtype": shape.cache_dtype, "parallelism": "host cores"},
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                                 "sample": f"each step: {per_step:.1f} s of single-head fp64 explicit-form prefills "
                                           f"of one {shape.name} prompt; numpy's BLAS pool had {blas_threads()} threads"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    prep = oracle_prep(inp)   # the resident cache, built once
    for k in range(args.warmup):
        oracle_sample(inp, min(1.0, args.cpu_seconds / 10), k, prep=prep)
    vals, secs = [], 0.0
    per_step = max(0.5, args.cpu_seconds / max(1, args.steps))
    for k in range(args.steps):
        v, done, dt = oracle_sample(inp, per_step, args.warmup + k, prep=prep)
        vals.append(v)
        secs += dt
    value = float(np.mean(vals))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": shape.name, "batch": shape.batch, "seq_len": int(inp.lengths.max()),
                       "cached_tokens": int(inp.lengths.sum()), "n_heads": shape.n_heads,
                       "cache_dtype": shape.cache_dtype, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": f"each step: {per_step:.1f} s of (sequence, head) fp64 absorbed-form "
                                       f"decodes of {shape.name}; numpy's BLAS pool had {blas_threads()} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.workload in S.PREFILL_SHAPES:
        res, inp = run_prefill(args, rank, world, local)
    else:
        res, inp = run_gpu(args, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline:
        if args.workload in S.PREFILL_SHAPES:
            v, done, dt = oracle_prefill_sample(inp, args.cpu_seconds)
            res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                                   "sample": f"{done} single-head fp64 explicit-form prefills of one {inp.shape.name} "
                                             f"prompt ({dt:.1f} s); tokens/s = prompt tokens x heads done / n_heads "
                                             f"/ time; numpy's BLAS pool had {blas_threads()} threads"}
        else:
            res["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
