"""Benchmark of the speculative-decoding verify step on GB300.

One step = one pass of the whole verify path over one batch of synthetic
inputs already resident in HBM: paged verify attention (one attention layer),
acceptance (rejection sampling at the workload's temperature, or greedy), and,
for workloads with gated-delta-net layers, the recurrent-state commit.

Metric: verified tokens/s = sum_b (accept_len_b + 1) / step time.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle instead
(on the host cores, a bounded sample of the same workload, scaled to the same
metric).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_verification_paged_gb300 import workloads as wl  # noqa: E402

METRIC = "verified tokens/s per verify step (1 GB300); verify-attn & accept HBM GB/s vs peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "hybrid_gdn"
L2_FLUSH_BYTES = 512 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
# The device code of each kernel: a recorded ncu traffic figure stays valid while
# these files hash to the recorded value (host launch code may change).
_CSRC = "speculative_decoding_verification_paged_gb300/csrc/"
KERNEL_SOURCES = {
    "attention/mma": [_CSRC + "common.cuh", _CSRC + "attention_device.cuh", _CSRC + "attention_mma.cuh"],
    "attention/tc": [_CSRC + "common.cuh", _CSRC + "attention_device.cuh", _CSRC + "attention_tc.cuh"],
    "accept": [_CSRC + "common.cuh", _CSRC + "accept.cu"],
    "commit": [_CSRC + "common.cuh", _CSRC + "commit.cu"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--mode", default=None, choices=[None, "sample", "greedy", "mixed"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--commit", default="copy", choices=["copy", "select"],
                    help="recurrent-state commit: copy the kept checkpoint into the live state, or select it "
                         "in place by exchanging state-pool row indices (zero-copy)")
    ap.add_argument("--gdn-verify", action="store_true",
                    help="add one gated-delta-net layer's recurrence over the verify chain to the step "
                         "(workloads with recurrent state; pooled when --commit select)")
    ap.add_argument("--seed", type=int, default=None,
                    help="draw the synthetic inputs from this seed instead of the workload's own")
    ap.add_argument("--gdn-layers", type=int, default=None,
                    help="override the workload's recurrent-state layer count (small profiler captures); "
                         "the line's config reports the count used")
    return ap.parse_args()


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; each rank verifies its own batch)
# --------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------
# algorithmic bytes
# --------------------------------------------------------------------------
def attention_bytes(w, ctx_lens):
    ctx = [int(c) for c in ctx_lens]
    kv = sum(ctx) * w.num_kv_heads * w.head_dim * 2 * 2
    qo = w.batch * w.rows * w.num_q_heads * w.head_dim * (2 + 4)
    table = sum(-(-c // w.block_size) for c in ctx) * 4 + w.batch * 4
    return kv + qo + table


def accept_bytes(w, modes, accept_len):
    V, k = w.vocab, w.k_draft
    total = 0
    for md, m in zip(modes, accept_len):
        m = int(m)
        if m < 0:
            continue
        total += (m + 1) * 4 * V
        if md == 1:
            total += (4 * V if m < k else 0) + 32 * m
    total += w.batch * (k * 4 + 4 + 4 + (k + 1) * 4 + 4)  # drafts, mode, temperature, out_tokens, accept_len
    return total


def acceptance_rate(alen, k):
    """Per-position acceptance rate: accepted drafts over decided drafts (a row that
    stops at m < k decided m + 1 drafts, a fully accepted row k)."""
    alen = np.asarray(alen, dtype=np.int64)
    decided = np.where(alen < k, alen + 1, k).sum()
    return float(alen.sum() / decided) if decided else None


def commit_bytes(w, commit="copy"):
    if not w.gdn_layers:
        return 0
    if commit == "select":  # per (layer, row): accept_len, live_row and one window index read, two written
        return w.gdn_layers * w.batch * 5 * 4
    return 2 * w.gdn_layers * w.batch * w.state_elems * 4


def gdn_verify_bytes(w):
    """One layer: read each (row, head) state once, write R checkpoints; q, k, v, out; g, beta."""
    states = w.batch * w.gdn_heads
    state_bytes = w.gdn_dv * w.gdn_dk * 4
    return (states * state_bytes * (1 + w.rows) + w.batch * w.rows * w.gdn_heads * (2 * w.gdn_dk + 2 * w.gdn_dv) * 4
            + w.batch * w.rows * w.gdn_heads * 8)


def select_tables(w, dev):
    """State-pool index tables for the zero-copy commit: (layer, row) unit u owns pool
    rows u*(W+1) (live) and u*(W+1)+1 .. u*(W+1)+W (its checkpoint window, W = k+1)."""
    W = w.rows
    units = torch.arange(w.gdn_layers * w.batch, dtype=torch.int32, device=dev) * (W + 1)
    live_row = units.view(w.gdn_layers, w.batch).clone()
    ckpt_rows = (units.view(-1, 1) + 1 + torch.arange(W, dtype=torch.int32, device=dev)).view(
        w.gdn_layers, w.batch, W).contiguous()
    return live_row, ckpt_rows


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def live_ceilings(dev):
    """Same-run context for the roofline: a 1 GiB device-to-device copy (read + write
    bytes) and a 2 GiB read-only reduction, best of 5, CUDA events; taken after the
    timed region."""
    src = torch.ones(1 << 28, dtype=torch.float32, device=dev)
    dst = torch.empty_like(src)
    big = torch.ones(1 << 29, dtype=torch.float32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def best(fn, nbytes):
        fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(5):
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        return nbytes / (min(t) / 1e3) / 1e9

    out = {"copy_gbs": best(lambda: dst.copy_(src), 2 * src.numel() * 4),
           "read_gbs": best(lambda: big.sum(), big.numel() * 4),
           "how": "1 GiB copy_ (read+write bytes) and a 2 GiB sum, best of 5, after the timed region"}
    del src, dst, big
    torch.cuda.empty_cache()
    return out


def workload_for(args):
    w = wl.WORKLOADS[args.config]
    if args.seed is not None:
        w = w.replace(seed=args.seed)
    if args.gdn_layers is not None:
        if not w.gdn_layers or args.gdn_layers < 1:
            raise SystemExit(f"--gdn-layers needs a workload with recurrent state and a count >= 1 ({w.name})")
        w = w.replace(gdn_layers=args.gdn_layers)
    return w


def kernel_sources_sha256(paths):
    """sha256 over the repo-relative path and the bytes of each file, in order."""
    h = hashlib.sha256()
    for rel in paths:
        h.update(rel.encode() + b"\0")
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_key(kernel, plan=None):
    """The source set a kernel's traffic record is keyed to."""
    return f"attention/{plan['kernel']}" if kernel == "attention" else kernel


def recorded_traffic(kernel, workload, plan=None, units=None):
    """DRAM bytes per call of `kernel` on `workload` from an ncu capture, if the capture ran the
    instance the library launches now (attention: the plan spec_verify_attention_plan reports) and
    the kernel's device sources are unchanged since. A record taken on a smaller case of the same
    kernel (fewer recurrent-state layers) is scaled to the call by its unit count, since the
    commit's traffic grows in proportion to the states it moves."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        entry = json.load(f).get(kernel, {}).get(workload)
    if not entry:
        return None
    if kernel == "attention" and entry.get("plan") != plan:
        return None
    if entry.get("kernel_sources_sha256") != kernel_sources_sha256(KERNEL_SOURCES[traffic_key(kernel, plan)]):
        return None
    per_unit = entry.get("dram_bytes_per_unit")
    if per_unit is not None:
        return per_unit * units if units else None
    return entry.get("dram_bytes_per_call")


def dominant_traffic(kernel, workload, plan, w, select):
    """Recorded DRAM bytes per call of the step's dominant kernel, or None."""
    if kernel == "attention":
        return recorded_traffic("attention", workload, plan)
    if kernel == "commit" and not select:
        return recorded_traffic("commit", workload, units=w.gdn_layers * w.batch)
    return None


# --------------------------------------------------------------------------
# native arm
# --------------------------------------------------------------------------
def run_native(args, world, rank, local):
    import speculative_decoding_verification_paged_gb300 as sv

    sv.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_for(args)
    mode = args.mode or w.mode
    a = wl.make_attention_inputs(w, device=dev, seed=w.seed + 1000 * rank)
    acc_in = wl.make_accept_inputs(w, device=dev, seed=w.seed + 1000 * rank, mode=mode)
    select = bool(w.gdn_layers) and args.commit == "select"
    g = wl.make_gdn_inputs(w, device=dev, seed=w.seed + 1000 * rank) if w.gdn_layers and not select else None
    tables = select_tables(w, dev) if select else None
    gv = None
    if args.gdn_verify and w.gdn_layers:
        gv = wl.make_gdn_verify_inputs(w, device=dev, seed=w.seed + 1000 * rank, layers=1)
        gv = {n: (t[0] if torch.is_tensor(t) else t) for n, t in gv.items()}
        gv["out"] = torch.empty((w.batch, w.rows, w.gdn_heads, w.gdn_dv), device=dev)
        if select:  # layer 0's rows of the pool: unit b owns rows b*(W+1) .. b*(W+1)+W
            gv["pool"] = torch.zeros((w.batch * (w.rows + 1), w.state_elems), device=dev)
            gv["pool"][tables[0][0].long()] = gv["state"].view(w.batch, -1)
    B, R = w.batch, w.rows
    out = torch.empty((B, R, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)
    ws = sv.new_attention_workspace(
        sv.spec_verify_attention_workspace(a["q"], a["k_cache"], a["block_table"], w.k_draft), dev)
    toks = torch.empty((B, R), dtype=torch.int32, device=dev)
    alen = torch.empty((B,), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def attention():
        sv.spec_verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["ctx_lens"], w.k_draft, out,
                                 workspace=ws, dev_err=err)

    def accept():
        sv.spec_accept(acc_in["target_logits"], acc_in["draft_tokens"], acc_in["draft_probs"],
                       acc_in["philox_seed"], acc_in["mode"], acc_in["temperature"], toks, alen, dev_err=err)

    def commit():
        if tables is not None:
            sv.spec_commit_select(alen, tables[0], tables[1], w.rows, sv.ALIGN_TOKEN, dev_err=err)
        elif g is not None:
            sv.spec_commit_state(g["snapshots"], alen, g["live_state"], dev_err=err)

    def gdn_verify():
        qkv = [gv[n] for n in ("q", "k", "v", "g", "beta")]
        if tables is not None:
            sv.spec_gdn_verify_pooled(*qkv, gv["pool"], tables[0][0], tables[1][0], gv["out"], gv["scale"],
                                      dev_err=err)
        else:
            sv.spec_gdn_verify(*qkv, g["live_state"][0].view(w.batch, w.gdn_heads, w.gdn_dv, w.gdn_dk),
                               g["snapshots"][0].view(w.batch, w.rows, w.gdn_heads, w.gdn_dv, w.gdn_dk),
                               gv["out"], gv["scale"], dev_err=err)

    def step():
        attention()
        if gv is not None:
            gdn_verify()
        accept()
        commit()

    launches_per_step = 1 + 1 + (1 if w.gdn_layers else 0) + (1 if gv is not None else 0)
    nvtx = torch.cuda.nvtx  # phase markers for timeline profilers
    nvtx.range_push("warm-up")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    nvtx.range_pop()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    # The step (and each call alone) is captured once into a CUDA graph and
    # replayed, so the device timeline carries no host launch gaps.
    graphs = {}
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for name, fn in (("step", step), ("attention", attention), ("accept", accept), ("commit", commit),
                         ("gdn_verify", gdn_verify)):
            if name == "commit" and not w.gdn_layers:
                continue
            if name == "gdn_verify" and gv is None:
                continue
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                fn()
            graphs[name] = graph
    stream.wait_stream(side)
    torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def l2_flush():
        # write a buffer larger than L2, then read another one so the dirty lines
        # are written back here and not inside the next timed region
        flush.zero_()
        flush_read.sum()

    def timed(graph, n):
        times = []
        for _ in range(n):
            l2_flush()  # between timed replays, outside the events
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return times

    for _ in range(2):
        graphs["step"].replay()
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start
    nvtx.range_push("timed steps")
    per_step = timed(graphs["step"], args.steps)
    torch.cuda.synchronize()
    nvtx.range_pop()
    barrier(world)
    clk = clocks.stop()
    nvtx.range_push("per-kernel timing")
    t_attn = timed(graphs["attention"], args.steps)
    t_acc = timed(graphs["accept"], args.steps)
    t_cmt = timed(graphs["commit"], args.steps) if "commit" in graphs else [0.0]
    t_gdn = timed(graphs["gdn_verify"], args.steps) if "gdn_verify" in graphs else None
    nvtx.range_pop()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    ms = statistics.mean(per_step)
    alen_h = alen.cpu().numpy()
    tokens = float(np.sum(alen_h + 1))
    ms_max = reduce_max(ms, world)
    tokens_all = reduce_sum(tokens, world)
    value = tokens_all / (ms_max / 1e3)

    peak, peak_kind = measured_peaks()
    ctx = a["ctx_lens"].cpu().numpy()
    ab = attention_bytes(w, ctx)
    cb = accept_bytes(w, acc_in["mode"].cpu().numpy(), alen_h)
    mb = commit_bytes(w, "select" if select else "copy")
    ta, tc, tm = statistics.mean(t_attn), statistics.mean(t_acc), statistics.mean(t_cmt)
    plan = sv.spec_verify_attention_plan(a["q"], a["k_cache"], a["block_table"], w.k_draft)
    # every position of every row read (logits, and the draft rows of the sampling rows): the
    # bytes an acceptance without early exit would move, reported beside the early-exit basis
    full_read = w.batch * 4 * w.vocab * (R + w.k_draft)
    kernels = {
        "attention": {"ms": ta, "bytes": ab, "GBps": ab / ta / 1e6, "frac": ab / ta / 1e6 / peak, "plan": plan},
        "accept": {"ms": tc, "bytes": cb, "GBps": cb / tc / 1e6, "frac": cb / tc / 1e6 / peak,
                   "full_read_bytes": full_read, "frac_full_read": full_read / tc / 1e6 / peak},
    }
    if w.gdn_layers:
        kernels["commit"] = {"ms": tm, "bytes": mb, "GBps": mb / tm / 1e6, "frac": mb / tm / 1e6 / peak,
                             "kind": "select" if select else "copy"}
    if t_gdn is not None:
        tg, gb = statistics.mean(t_gdn), gdn_verify_bytes(w)
        kernels["gdn_verify"] = {"ms": tg, "bytes": gb, "GBps": gb / tg / 1e6, "frac": gb / tg / 1e6 / peak,
                                 "layers": 1}
    dominant = max(kernels, key=lambda k: kernels[k]["ms"])
    dk = kernels[dominant]
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": dk["GBps"], "peak": peak, "unit": "GB/s",
                "frac": dk["frac"], "peak_source": peak_kind,
                "traffic": dominant_traffic(dominant, args.config, plan, w, select),
                "same_run_ceilings": live_ceilings(dev)}

    e2e = None
    if not args.no_e2e:
        nvtx.range_push("end to end")
        e2e = run_e2e(sv, w, a, acc_in, commit, out, ws, toks, alen, err, dev, args, flush, gv, gdn_verify)
        nvtx.range_pop()

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch_per_gpu": w.batch, "k_draft": w.k_draft, "mode": mode, "seed": w.seed,
                   "ctx": list(w.ctx_range) if w.ctx_range else sorted(set(w.ctx_lens)),
                   "block_size": w.block_size, "heads": [w.num_q_heads, w.num_kv_heads], "head_dim": w.head_dim,
                   "vocab": w.vocab, "gdn_layers": w.gdn_layers, "parallelism": f"replicas x{world}",
                   **({"commit": "select (zero-copy: pool-row index exchange)" if select else "copy"}
                      if w.gdn_layers else {}),
                   **({"gdn_verify": f"one layer: {w.gdn_heads} heads, {w.gdn_dv}x{w.gdn_dk} fp32 state, "
                                     f"{w.rows} tokens"} if gv is not None else {}),
                   "l2": "flushed between timed steps (512 MiB write, then 512 MiB read)",
                   "timing": "CUDA-graph replay of the step, CUDA events on the launching stream"},
        "verified_tokens_per_step": tokens_all, "mean_accept_len": float(np.mean(alen_h)),
        "acceptance_rate": acceptance_rate(alen_h, w.k_draft),
        "kernels": kernels, "roofline": roofline, "clocks": clk, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
    }
    return result


def run_e2e(sv, w, a, acc_in, commit, out, ws, toks, alen, err, dev, args, flush, gv=None, gdn_verify=None):
    """Same metric through the public API with the step's inputs in pinned host memory. The
    serving state stays resident in HBM, as it does in an engine: the paged KV cache, the
    recurrent state and its checkpoints. The step's activations and scheduling data are copied
    in every step: q, the block table and context lengths, the target logits, the draft tokens
    and draft probabilities, per-row mode and temperature (and, with --gdn-verify, the
    recurrence's q, k, v and gates). The outputs are read back. Within a step the acceptance
    inputs are copied on a second stream while the attention call runs, as an engine would
    overlap them."""
    host = {n: a[n].cpu().pin_memory() for n in ("q", "block_table", "ctx_lens")}
    for n in ["target_logits", "draft_tokens", "draft_probs", "mode", "temperature"]:
        host[n] = acc_in[n].cpu().pin_memory()
    gdn_host = {}
    if gv is not None:
        gdn_host = {n: gv[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    devbuf = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    attn_inputs = ("q", "block_table", "ctx_lens")
    side = torch.cuda.Stream(device=dev)  # the acceptance inputs arrive while attention runs
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    toks_h = torch.empty(toks.shape, dtype=toks.dtype).pin_memory()
    alen_h = torch.empty(alen.shape, dtype=alen.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + list(gdn_host.values()))
    d2h = out_h.numel() * 4 + toks_h.numel() * 4 + alen_h.numel() * 4
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step():
        side.wait_stream(stream)  # the previous step is done with the buffers
        with torch.cuda.stream(side):
            for n, t in host.items():
                if n not in attn_inputs:
                    devbuf[n].copy_(t, non_blocking=True)
        for n in attn_inputs:
            devbuf[n].copy_(host[n], non_blocking=True)
        sv.spec_verify_attention(devbuf["q"], a["k_cache"], a["v_cache"], devbuf["block_table"],
                                 devbuf["ctx_lens"], w.k_draft, out, workspace=ws, dev_err=err)
        if gv is not None:
            for n, t in gdn_host.items():  # the step's activations into the buffers the recurrence reads
                gv[n].copy_(t, non_blocking=True)
            gdn_verify()
        stream.wait_stream(side)
        sv.spec_accept(devbuf["target_logits"], devbuf["draft_tokens"], devbuf["draft_probs"],
                       acc_in["philox_seed"], devbuf["mode"], devbuf["temperature"], toks, alen, dev_err=err)
        commit()
        out_h.copy_(out, non_blocking=True)
        toks_h.copy_(toks, non_blocking=True)
        alen_h.copy_(alen, non_blocking=True)

    n = max(3, min(args.steps, 10))
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(n):
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.mean(times)
    tokens = float((alen_h.numpy() + 1).sum())
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n}


# --------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# --------------------------------------------------------------------------
class OracleStep:
    """The CPU oracle over one step of a workload, timed on a bounded sample (inputs drawn once)."""

    def __init__(self, w, mode, seed_offset=0, commit="copy", gdn_verify=False):
        import oracle
        oracle.build()
        self.oracle, self.w, self.commit = oracle, w, commit
        a = wl.make_attention_inputs(w, device="cpu", seed=w.seed + seed_offset)
        self.acc_in = wl.make_accept_inputs(w, device="cpu", seed=w.seed + seed_offset, mode=mode)
        self.q = a["q"].view(torch.int16).numpy().view(np.uint16)
        self.kc = a["k_cache"].view(torch.int16).numpy().view(np.uint16)
        self.vc = a["v_cache"].view(torch.int16).numpy().view(np.uint16)
        self.table, self.ctx = a["block_table"].numpy(), a["ctx_lens"].numpy()
        self.threads = oracle.max_threads()
        self.g = None
        if w.gdn_layers and commit != "select":
            self.g = wl.make_gdn_inputs(w.replace(gdn_layers=1), device="cpu", seed=w.seed + seed_offset)
        self.gdn = None
        if gdn_verify and w.gdn_layers:  # one layer; a few rows (all heads), scaled to the batch
            rows = min(4, w.batch)
            x = wl.make_gdn_verify_inputs(w.replace(batch=rows), device="cpu", seed=w.seed + seed_offset)
            self.gdn = ([x[n][0].numpy() for n in ("q", "k", "v", "g", "beta")], x["state"][0].numpy(),
                        x["scale"], rows)

    def run(self, budget_s):
        """Seconds per full step (sampled parts scaled), verified tokens, the sample, threads."""
        o, w, acc_in = self.oracle, self.w, self.acc_in
        # attention: whole sequences, a few at a time so that every thread has a (sequence,
        # kv head) unit, until the budget is spent; scaled by context tokens
        per_call = max(1, -(-self.threads // w.num_kv_heads))
        t0 = time.perf_counter()
        done_ctx, done = 0, 0
        while done < w.batch and time.perf_counter() - t0 < budget_s * 0.7:
            seqs = np.arange(done, min(w.batch, done + per_call), dtype=np.int32)
            o.verify_attention(self.q, self.kc, self.vc, self.table, self.ctx, seqs=seqs)
            done_ctx += int(self.ctx[seqs].sum())
            done += len(seqs)
        t_attn = (time.perf_counter() - t0) * float(self.ctx.sum()) / max(done_ctx, 1)
        t1 = time.perf_counter()
        tok, alen, _, _, _ = o.accept(acc_in["target_logits"].numpy(), acc_in["draft_tokens"].numpy(),
                                      acc_in["draft_probs"].numpy(), acc_in["philox_seed"],
                                      acc_in["mode"].numpy(), acc_in["temperature"].numpy())
        t_acc = time.perf_counter() - t1
        t_cmt = 0.0
        if w.gdn_layers and self.commit == "select":
            live_row, ckpt_rows = (t.numpy() for t in select_tables(w, "cpu"))
            t2 = time.perf_counter()
            o.commit_select(alen, live_row, ckpt_rows, w.rows, 0)
            t_cmt = time.perf_counter() - t2
        elif self.g is not None:
            live = self.g["live_state"].numpy()
            t2 = time.perf_counter()
            o.commit_state(self.g["snapshots"].numpy(), alen, live)
            t_cmt = (time.perf_counter() - t2) * w.gdn_layers
        t_gdn, gdn_rows = 0.0, 0
        if self.gdn is not None:
            arrays, state, scale, gdn_rows = self.gdn
            t3 = time.perf_counter()
            o.gdn_verify(*arrays, state, scale=scale)
            t_gdn = (time.perf_counter() - t3) * w.batch / gdn_rows
        tokens = float(np.sum(alen + 1))
        sample = (f"attention over {done}/{w.batch} sequences ({done_ctx} of {int(self.ctx.sum())} context tokens, "
                  f"scaled by tokens) + acceptance of all {w.batch} rows"
                  + ((" + zero-copy commit of all layers" if self.commit == "select" else
                      f" + commit of 1/{w.gdn_layers} layers (scaled)") if w.gdn_layers else "")
                  + (f" + one gated-delta-net layer over {gdn_rows}/{w.batch} rows (scaled)" if gdn_rows else ""))
        return t_attn + t_acc + t_cmt + t_gdn, tokens, sample, self.threads


def run_reference(args, world, rank):
    w = workload_for(args)
    mode = args.mode or w.mode
    per_step_budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    step = OracleStep(w, mode, commit=args.commit, gdn_verify=args.gdn_verify)
    times, tokens, sample, threads = [], 0.0, "", 1
    for i in range(args.warmup + args.steps):
        s, tokens, sample, threads = step.run(per_step_budget)
        if i >= args.warmup:
            times.append(s)
    ms = statistics.mean(times) * 1e3
    value = tokens / (ms / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch_per_gpu": w.batch, "k_draft": w.k_draft, "mode": mode, "seed": w.seed,
                   "parallelism": "host cores (OpenMP)", **({"commit": args.commit} if w.gdn_layers else {})},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    result = run_native(args, world, rank, local)
    if rank == 0:
        if args.no_cpu_baseline or world > 1:  # the oracle baseline is an N = 1 measurement
            result["cpu_baseline"] = None
        else:
            w = workload_for(args)
            s, tokens, sample, threads = OracleStep(w, args.mode or w.mode, commit=args.commit,
                                                    gdn_verify=args.gdn_verify).run(args.cpu_seconds)
            result["cpu_baseline"] = {"value": tokens / s, "unit": UNIT, "cores": threads, "kind": "oracle",
                                      "sample": sample}
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
