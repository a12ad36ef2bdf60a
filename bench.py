"""Benchmark of the LM-head logprob path: rows/s and each dominant kernel's roofline.

One step = one pass of the whole hot path over one batch: lmh_select_rows on
the batch's cu_seqlens, then lmh_project_logprobs on the selected rows (row
gather, tcgen05 head GEMM with the fused lse / selected-logprob / top-k
epilogue, partial merge); for the prompt-scoring chunk, one
lmh_logprobs_from_logits call.  A pure-decode batch (every sequence one
decode row) passes no row indices, as the pages' pure-decode case does: the
selection is the identity and the head reads the hidden rows in place.

The headline workload is the mixed serving step (Llama-3-8B head shape: H
4096, V 128256; 64 decode rows, 4 prefill segments of 512 and one
1024-position scoring segment: 1092 selected rows), the largest selective
configuration.  The same JSON line carries a "workloads" object with the
other configurations (decode batch K 5 and K 1, selective prefill, the
16384-row full projection arm, the 256 x 248320 logits chunk), each with its
own value, roofline, CPU baseline and id check.  Inputs are seeded synthetic
tensors (workloads.py) resident in HBM; every head is larger than L2, so each
step streams it from HBM, and the chunk rotates four copies.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixed_batch]
    python bench.py --impl reference ...   # the CPU oracle on the same workload

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its
own batch (rows are independent: weak scaling, no collective on the data
path); the value is all ranks' rows over the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "logprob rows/sec (head+lse+top-K) and % of HBM / bf16 tensor roofline"
UNIT = "rows/s"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "dram_traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


HEADLINE = "mixed_batch"
SUB_WORKLOADS = ("decode_batch", "decode_batch_k1", "prefill_batch", "prefill_full", "logits_chunk")
WORKLOADS = (HEADLINE,) + SUB_WORKLOADS
SUB_TIMED_S = 1.0  # about this much device time per extra workload's timed region


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE, choices=list(WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sub", action="store_true", help="only the headline workload (profiling runs)")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    p.add_argument("--k", type=int, default=None,
                   help="override the workload's K (-1: the full-vocabulary output, every id's logprob)")
    p.add_argument("--logit-scale", type=float, default=1.0,
                   help="head transform: every logit scaled by this factor (head workloads)")
    p.add_argument("--w-hv", action="store_true",
                   help="the head weight stored [H x V] (vocabulary contiguous) instead of lm_head.weight's [V x H]")
    p.add_argument("--sample", action="store_true",
                   help="device-side Gumbel-max sampling of every row at temperature 1 (head workloads)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def make_workload(name, rank=0):
    import workloads
    seed_shift = 1000 * rank  # every rank gets its own batch
    if name in ("decode_batch", "decode_batch_k1"):
        b = workloads.decode_batch(seed=1 + seed_shift, k=1 if name.endswith("k1") else 5)
    elif name in ("prefill_batch", "prefill_full"):
        b = workloads.prefill_batch(seed=2 + seed_shift)
        if name == "prefill_full":  # every packed row through the head (the materializing 'before' arm)
            b = dict(b, name="prefill_full", num_decode=0, all_rows_mask=None,
                     full=True, n_sel=b["hidden"].shape[0], sel=b["sel_all"])
    elif name == "mixed_batch":
        b = workloads.mixed_batch(seed=4 + seed_shift)
    else:
        b = workloads.logits_chunk("normal", seed=3 + seed_shift)
        b["k"] = 20
    return b


def apply_options(b, args):
    """--k and --logit-scale on a workload (K -1: every id's logprob; per-row K is then unused)."""
    if getattr(args, "k", None) is not None:
        b = dict(b, k=args.k, row_k=None if args.k < 0 else b.get("row_k"))
    if getattr(args, "logit_scale", 1.0) != 1.0:
        b = dict(b, logit_scale=args.logit_scale)
    if getattr(args, "sample", False) and b["name"] != "logits_chunk":
        b = dict(b, sample=True)
    if getattr(args, "w_hv", False) and b["name"] != "logits_chunk":
        b = dict(b, w_hv=True)
    return b


def workload_config(b):
    if b["name"] == "logits_chunk":
        return {"workload": "logits_chunk", "rows": b["rows"], "V": b["V"], "k": b["k"], "dtype_in": "bf16",
                "l2": "inputs larger than L2 (a 127 MB chunk; 4 chunks rotated)"}
    cfg = {"workload": b["name"], "rows": int(b["n_sel"]), "tokens": int(b["hidden"].shape[0]),
           "H": int(b["H"]), "V": int(b["V"]), "k": int(b["k"]),
           "l2": "inputs larger than L2 (the %.0f MB head is streamed from HBM every step)"
                 % (b["V"] * b["H"] * 2 / 1e6)}
    if b.get("logit_scale", 1.0) != 1.0:
        cfg["logit_scale"] = b["logit_scale"]
    if b.get("sample"):
        cfg["sampling"] = "Gumbel-max, temperature 1, every row"
    if b.get("w_hv"):
        cfg["w_layout"] = "[H x V] (vocabulary contiguous)"
    return cfg


def pure_decode(b):
    """Every sequence is one decode row: the selection is the identity and no indices are passed."""
    return b["name"] != "logits_chunk" and not b.get("full") and int(b["num_decode"]) == b["cu_seqlens"].numel() - 1 \
        and int(b["n_sel"]) == int(b["hidden"].shape[0])


def algorithmic(b):
    """(bound, per-launch algorithmic amount, unit) of the dominant kernel (dominant_kernel(b))."""
    if b["name"] == "logits_chunk":
        if b["k"] < 0:  # the full-vocabulary pass: read the logits, write every fp32 logprob
            return "hbm", b["rows"] * b["V"] * (2 + 4), "GB/s"
        return "hbm", b["rows"] * b["V"] * 2 + b["rows"] * (2 + 2 * b["k"]) * 4, "GB/s"
    rows, H, V = int(b["n_sel"]), int(b["H"]), int(b["V"])
    if rows >= 256:  # the projection is tensor-bound from a few hundred rows on
        return "tensor", 2.0 * rows * H * V, "TFLOP/s"
    return "hbm", V * H * 2 + rows * H * 2, "GB/s"


def dominant_kernel(b):
    if b["name"] == "logits_chunk":
        return "full_logprobs" if b["k"] < 0 else "logits_reduce"
    return "head_logprobs"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons, power = [], None, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def rejected(clocks):
    if not clocks:
        return False
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clocks["reasons"]):
        return True
    return clocks["sm_max_mhz"] and clocks["sm_mhz"] < 0.5 * clocks["sm_max_mhz"] and not clocks["reasons"]


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def packed(tensors, device, pinned=False):
    """One byte buffer holding a copy of each named tensor at 256-byte aligned offsets.

    Returns (buffer, {name: view}); with one buffer a step moves its inputs (or its
    results) in a single copy, as a serving loop packs them.
    """
    import torch
    layout, off = {}, 0
    for name, t in tensors.items():
        nbytes = t.numel() * t.element_size()
        layout[name] = (off, nbytes, t.shape, t.dtype)
        off = (off + nbytes + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = {name: buf[o:o + nb].view(dt).view(shape) for name, (o, nb, shape, dt) in layout.items()}
    return buf, views


def step_outputs(rows, k, V, with_sel, device):
    """Preallocated outputs of one call (K -1: [rows, V] logprobs, no ids)."""
    import torch
    return {"lse": torch.empty(rows, dtype=torch.float32, device=device),
            "sel_logprob": torch.empty(rows, dtype=torch.float32, device=device) if with_sel else None,
            "topk_ids": None if k < 0 else torch.empty((rows, k), dtype=torch.int32, device=device),
            "topk_logprobs": torch.empty((rows, V if k < 0 else k), dtype=torch.float32, device=device)}


class Step:
    """Device-resident inputs, preallocated outputs/workspace and one step of the path."""

    def __init__(self, lmh, b, device):
        import torch
        self.lmh, self.b, self.dev = lmh, b, device
        self.chunk = b["name"] == "logits_chunk"
        if self.chunk:
            # rotate 4 copies so consecutive steps do not hit in L2 (a chunk is about the size of L2)
            self.logits = [b["logits"].to(device) for _ in range(4)]
            self.sel = b["sel"].to(device)
            self.k = b["k"]
            self.rows = b["rows"]
            self.ws = torch.empty(lmh.workspace_bytes(self.rows, 0, b["V"], self.k, lmh.PATH_FROM_LOGITS),
                                  dtype=torch.uint8, device=device)
            self.out = self._outputs(self.rows, self.k, True)
            self.i = 0
            return
        self.full = b.get("full", False)
        self.scale = b.get("logit_scale", 1.0)
        self.sampling = None
        if b.get("sample"):
            self.sampling = {"temperature": torch.ones(int(b["n_sel"]), dtype=torch.float32, device=device),
                             "seed": 1234, "offsets": torch.arange(int(b["n_sel"]), dtype=torch.int64, device=device)}
        self.hidden = b["hidden"].to(device)
        self.w_layout = lmh.W_HV if b.get("w_hv") else lmh.W_VH
        self.W = (b["W"].t().contiguous() if b.get("w_hv") else b["W"]).to(device)
        self.cu = b["cu_seqlens"].to(device)
        self.mask = None if b["all_rows_mask"] is None else b["all_rows_mask"].to(device)
        self.sel = b["sel"].to(device)
        self.row_k = None if b["row_k"] is None else b["row_k"].to(device)
        self.k = int(b["k"])
        self.rows = int(b["n_sel"])
        self.pure = pure_decode(b)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = torch.empty(lmh.workspace_bytes(self.rows, b["H"], b["V"], self.k, lmh.PATH_PROJECT),
                              dtype=torch.uint8, device=device)
        self.out = self._outputs(self.rows, self.k, True)

    def _outputs(self, rows, k, with_sel):
        return step_outputs(rows, k, int(self.b["V"]), with_sel, self.dev)

    def run(self):
        lmh = self.lmh
        if self.chunk:
            x = self.logits[self.i & 3]
            self.i += 1
            return lmh.logprobs_from_logits(x, sel=self.sel, k_max=self.k, workspace=self.ws, out=self.out)
        if self.full or self.pure:
            return lmh.project_logprobs(self.hidden, self.W, sel=self.sel, row_k=self.row_k, k_max=self.k,
                                        workspace=self.ws, out=self.out, dev_status=self.status,
                                        logit_scale=self.scale, sampling=self.sampling, w_layout=self.w_layout)
        ri, _ = lmh.select_rows(self.cu, self.b["num_decode"], self.mask, max_out_rows=self.rows,
                                dev_status=self.status)
        return lmh.project_logprobs(self.hidden, self.W, row_idx=ri, sel=self.sel, row_k=self.row_k,
                                    k_max=self.k, workspace=self.ws, out=self.out, dev_status=self.status,
                                    logit_scale=self.scale, sampling=self.sampling, w_layout=self.w_layout)


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (all ranks get it); `ms` unchanged on one process."""
    import torch
    if not dist:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(rows_per_step, steps, world, ms):
    """Whole-job rows/s: the rows every rank processed over the slowest rank's time."""
    return rows_per_step * steps * world / (ms / 1e3)


def timed_region(step, steps, dist, world):
    import torch
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step.run()
    stop.record()
    torch.cuda.synchronize()
    return max_over_ranks(start.elapsed_time(stop), dist, "cuda")


def e2e_leg(lmh, b, device, steps):
    """Same metric through the public API with inputs in pinned host memory.

    Every step copies its inputs host->device (hidden rows, cu_seqlens,
    selected ids; the head weight stays resident like model weights), runs
    the path, copies the compact result device->host and reads it on the
    host.  As a serving loop would, each step's calls and its copy out are
    captured once in a CUDA graph and replayed every step (if capture fails
    the calls run eagerly), two buffer sets alternate, and step i+1 is issued
    before the host waits for step i's result.

    The value is the loop as a serving engine runs it: the copies in go on a
    copy stream, so step i+1's inputs cross while step i computes, and every
    step's GPU work runs on one compute stream, after the previous step's.
    Two more loops are reported as context: "serial" (copy in and compute on
    one stream, nothing overlaps) and "pipelined" (one stream per buffer set:
    two independent batches in flight, whose heads share W's reads in L2).
    """
    import torch
    chunk = b["name"] == "logits_chunk"
    pure = pure_decode(b)
    src = {"logits": b["logits"], "sel": b["sel"]} if chunk else \
        {"hidden": b["hidden"], "cu": b["cu_seqlens"], "sel": b["sel"]}
    h_in_buf, h_in = packed(src, "cpu", pinned=True)  # the step's inputs, packed in pinned host memory
    for key, v in src.items():
        h_in[key].copy_(v)
    if not chunk:
        w_layout = lmh.W_HV if b.get("w_hv") else lmh.W_VH
        W = (b["W"].t().contiguous() if b.get("w_hv") else b["W"]).to(device)
        mask = None if b["all_rows_mask"] is None else b["all_rows_mask"].to(device)
        row_k = None if b["row_k"] is None else b["row_k"].to(device)
    rows = b["rows"] if chunk else int(b["n_sel"])
    k = int(b["k"])
    if chunk:
        ws_bytes = lmh.workspace_bytes(rows, 0, b["V"], k, lmh.PATH_FROM_LOGITS)
    else:
        ws_bytes = lmh.workspace_bytes(rows, int(b["H"]), int(b["V"]), k, lmh.PATH_PROJECT)
    copy_stream, compute_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def buffers():
        d_in_buf, d_in = packed(h_in, device)
        shapes = {key: v for key, v in step_outputs(rows, k, int(b["V"]), True, "meta").items() if v is not None}
        d_out_buf, out = packed(shapes, device)
        h_out_buf, h_out = packed(shapes, "cpu", pinned=True)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        return {"d_in_buf": d_in_buf, "d_in": d_in, "d_out_buf": d_out_buf, "out": out, "h_out_buf": h_out_buf,
                "h_out": h_out, "ws": ws, "ev": torch.cuda.Event(), "in_ev": torch.cuda.Event(),
                "stream": torch.cuda.Stream()}

    bufs = [buffers(), buffers()]
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in bufs[0]["h_out"].values())

    def copy_in(bf):
        bf["d_in_buf"].copy_(h_in_buf, non_blocking=True)  # one copy in

    def compute_ops(bf):
        d_in = bf["d_in"]
        if chunk:
            o = lmh.logprobs_from_logits(d_in["logits"], sel=d_in["sel"], k_max=k, workspace=bf["ws"],
                                         out=bf["out"])
        else:
            ri = None
            if not pure:
                ri, _ = lmh.select_rows(d_in["cu"], b["num_decode"], mask, max_out_rows=rows)
            o = lmh.project_logprobs(d_in["hidden"], W, row_idx=ri, sel=d_in["sel"], row_k=row_k, k_max=k,
                                     workspace=bf["ws"], out=bf["out"], logit_scale=b.get("logit_scale", 1.0),
                                     w_layout=w_layout)
        assert all(o[key].data_ptr() == bf["out"][key].data_ptr() for key in bf["out"])
        bf["h_out_buf"].copy_(bf["d_out_buf"], non_blocking=True)  # one copy out

    def run_compute(bf):
        if "graph" in bf:
            bf["graph"].replay()
        else:
            compute_ops(bf)

    def issue(bf, mode):
        if mode == "overlap":  # copy in on the copy stream, compute on the compute stream
            copy_stream.wait_event(bf["ev"])  # the buffer set's previous step has finished with it
            with torch.cuda.stream(copy_stream):
                copy_in(bf)
                bf["in_ev"].record()
            compute_stream.wait_event(bf["in_ev"])
            with torch.cuda.stream(compute_stream):
                run_compute(bf)
                bf["ev"].record()
        else:
            st = compute_stream if mode == "serial" else bf["stream"]
            with torch.cuda.stream(st):
                copy_in(bf)
                run_compute(bf)
                bf["ev"].record()

    def read(bf):  # the host waits for, and touches, the step's result
        bf["ev"].synchronize()
        return float(bf["h_out"]["lse"][0])

    torch.cuda.synchronize()  # the weights and inputs above were placed on the default stream
    for s in range(5):
        issue(bufs[s % 2], "serial")
        read(bufs[s % 2])
    graph_note = "each step's calls and copy out replayed from a CUDA graph"
    try:
        for bf in bufs:
            copy_in(bf)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                compute_ops(bf)
            bf["graph"] = g
        for s in range(4):
            issue(bufs[s % 2], "serial")
            read(bufs[s % 2])
    except Exception as e:  # capture is an optimisation of the loop, not a requirement
        for bf in bufs:
            bf.pop("graph", None)
        graph_note = "eager calls (graph capture failed: %s)" % str(e).splitlines()[0][:80]
        torch.cuda.synchronize()

    def timed(n, mode):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(n):
            issue(bufs[s % 2], mode)
            if s > 0:
                read(bufs[(s - 1) % 2])
        read(bufs[(n - 1) % 2])
        return time.perf_counter() - t0

    dt = timed(steps, "overlap")
    dt_serial = timed(steps, "serial")
    dt_pipe = timed(steps, "pipelined")
    return {"value": rows * steps / dt, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": 1e3 * dt / steps,
            "mode": "copies in on a copy stream overlap the previous step's compute; every step's GPU work on "
                    "one compute stream; " + graph_note,
            "serial": {"value": rows * steps / dt_serial, "ms_per_step": 1e3 * dt_serial / steps,
                       "note": "copy in, compute and copy out on one stream: nothing overlaps"},
            "pipelined": {"value": rows * steps / dt_pipe, "ms_per_step": 1e3 * dt_pipe / steps,
                          "note": "one stream per buffer set: two independent batches in flight, whose heads "
                                  "share W's reads in L2 (context only)"}}


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash(kernel):
    src = {"head_logprobs": ("head_kernel.cuh", "head_gemm.cu"), "logits_reduce": ("logits_reduce.cu",)}[kernel]
    h = hashlib.sha256()
    for name in src + ("device_common.cuh",):
        with open(os.path.join(ROOT, "top_reduction_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu capture, if the kernel is unchanged since."""
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    r = rec.get("%s/%s" % (kernel, workload))
    if not r or r.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return r.get("dram_bytes_per_launch")


class OracleStep:
    """One step of the oracle, as it stands, on the same workload.

    A step is one batch of selected rows (as many as the oracle has threads,
    so they are all busy): row selection, f64 projection and the
    full-vocabulary f64 log-softmax + full sort.  Rows cycle through the
    workload's selected rows.  The last step's rows and results are kept for
    the id check against the GPU's output.
    """

    def __init__(self, b, threads=0):
        import numpy as np
        import oracle
        import workloads
        self.oracle, self.b = oracle, b
        self.req_threads = int(threads)
        self.cores = oracle.cores()
        if b["name"] == "logits_chunk":
            self.x = workloads.bits(b["logits"])
            self.n = b["rows"]
        else:
            mask = None if b["all_rows_mask"] is None else b["all_rows_mask"].numpy()
            self.ri, _ = oracle.select_rows(b["cu_seqlens"].numpy(), b["num_decode"], mask)
            if b.get("full"):
                self.ri = np.arange(b["hidden"].shape[0], dtype=np.int32)
            self.hid, self.W = workloads.bits(b["hidden"]), workloads.bits(b["W"])
            self.n = len(self.ri)
        self.per = max(1, min(self.n, self.req_threads or self.cores))
        self.pos = 0
        self.threads = self.req_threads or self.cores
        self.last = None

    def run(self):
        import numpy as np
        b, o = self.b, self.oracle
        idx = (self.pos + np.arange(self.per)) % self.n
        self.pos = (self.pos + self.per) % self.n
        sel = b["sel"].numpy()[idx]
        k = max(int(b["k"]), 0)
        if b["name"] == "logits_chunk":
            r = o.logprobs(self.x[idx], dtype=o.BF16, sel=sel, k_max=k, threads=self.req_threads,
                           return_threads=True)
            self.threads = r["threads"]
            self.last = (idx, r, None)
        else:
            rk = None if b["row_k"] is None else b["row_k"].numpy()[idx]
            z, self.threads = o.project(self.hid, self.W, row_idx=self.ri[idx], threads=self.req_threads,
                                        return_threads=True)
            r = o.logprobs(z, sel=sel, row_k=rk, k_max=k, threads=self.req_threads)
            self.last = (idx, r, z)
        return self.per

    def describe(self):
        what = ("rows of the logits chunk (full-vocabulary f64 log-softmax + full sort)"
                if self.b["name"] == "logits_chunk" else
                "selected rows (row selection + f64 projection + full-vocabulary f64 log-softmax + full sort)")
        return "%d %s of %s per step" % (self.per, what, self.b["name"])


class IdCheck:
    """The GPU's top-k ids against the oracle's on the rows the oracle scored.

    From given logits the ids must be identical (the logits widen exactly).
    For the fused head a differing rank counts as a certified near-tie swap
    only when the oracle's values at the two ids differ by at most 2 * delta,
    delta = gamma_H * sum_h |A_h * W_hv| (the fp32 dot-product bound, gamma_H
    = H u / (1 - H u), u = 2^-24); anything else is an uncertified mismatch.
    The named workloads expect 0 of both.
    """

    def __init__(self, b, gpu_ids):
        self.b, self.ids = b, gpu_ids
        self.rows = self.ranks = self.mismatched = self.certified = 0
        self.max_gap = 0.0  # the largest oracle gap |z_gpu_id - z_oracle_id| among certified swaps

    def add(self, st):
        import numpy as np
        if self.ids is None or st.last is None:
            return
        idx, orc, z = st.last
        b = self.b
        k_max = max(int(b["k"]), 0)
        if k_max == 0:
            return
        ks = np.full(len(idx), k_max) if b.get("row_k") is None else np.clip(b["row_k"].numpy()[idx], 0, k_max)
        for j, r in enumerate(idx):
            k = int(ks[j])
            g, o = self.ids[r, :k], orc["topk_ids"][j, :k]
            self.rows += 1
            self.ranks += k
            for q in np.nonzero(g != o)[0]:
                self.mismatched += 1
                if z is None or g[q] < 0:
                    continue
                H = int(b["H"])
                u = 2.0 ** -24
                gamma = H * u / (1 - H * u)
                a = b["hidden"][int(st.ri[r])].float().double().numpy()
                Wc = b["W"][[int(g[q]), int(o[q])]].float().double().numpy()
                delta = b.get("logit_scale", 1.0) * gamma * np.abs(Wc * a[None, :]).sum(axis=1).max()
                gap = abs(z[j, g[q]] - z[j, o[q]])
                if gap <= 2 * delta:
                    self.certified += 1
                    self.max_gap = max(self.max_gap, float(gap))

    def summary(self):
        return {"rows_checked": self.rows, "ranks_checked": self.ranks, "certified_swaps": self.certified,
                "max_certified_gap": self.max_gap, "uncertified_mismatches": self.mismatched - self.certified}


def cpu_baseline(b, budget_s=12.0, single_s=4.0, gpu_ids=None):
    """The oracle on a bounded sample of the workload: about budget_s seconds on every
    host core, then about single_s seconds on one thread.  The rows it scores also
    check the GPU's ids (IdCheck)."""
    chk = IdCheck(b, gpu_ids)

    def timed(st, budget):
        t0 = time.perf_counter()
        rows, steps = 0, 0
        while steps == 0 or time.perf_counter() - t0 < budget:
            rows += st.run()
            steps += 1
            chk.add(st)
        return rows, steps, time.perf_counter() - t0

    st = OracleStep(b)
    rows, steps, dt = timed(st, budget_s)
    one = OracleStep(b, threads=1)
    rows1, steps1, dt1 = timed(one, single_s)
    return {"value": rows / dt, "unit": UNIT, "cores": int(st.threads), "kind": "oracle",
            "sample": "%d steps of %s (%.1f s)" % (steps, st.describe(), dt),
            "single_thread": {"value": rows1 / dt1, "unit": UNIT, "cores": 1,
                              "sample": "%d steps of %s (%.1f s)" % (steps1, one.describe(), dt1)},
            "id_check": chk.summary()}


def roofline(b, per_kernel, ms_per_step, peaks, peak_src):
    """The dominant kernel's roofline record: algorithmic amount over its traced launch time
    (for the logits chunk the whole call, stream and select kernels, over the step's event
    time)."""
    bound, amount, unit = algorithmic(b)
    kernel = dominant_kernel(b)
    if b["name"] == "logits_chunk" and b["k"] >= 0:
        us = 1e3 * ms_per_step
        kernel_label = "logits_reduce whole call (logits_stream_tma + logits_select)"
    else:
        us = per_kernel.get(kernel, {}).get("avg_us")
        kernel_label = kernel
    if bound == "hbm":
        peak = peaks["hbm_gbs"]
        achieved = amount / (us * 1e-6) / 1e9 if us else None
    else:
        peak = peaks["bf16_tflops"]
        achieved = amount / (us * 1e-6) / 1e12 if us else None
    roof = {"kernel": kernel_label, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": (achieved / peak) if achieved else None, "peak_source": peak_src + " (burst)",
            "algorithmic_per_launch": amount, "avg_launch_us": us,
            "traffic": recorded_traffic(kernel, b["name"])}
    if bound == "tensor" and achieved:
        roof["frac_of_sustained"] = achieved / peaks.get("bf16_tflops_sustained", peak)
    return roof


def measure(lmh, b, device, steps, warmup, dist, world, local, retry_clocks):
    """Warm-up, the timed region (the value), then the same steps traced per kernel."""
    import torch
    step = Step(lmh, b, device)
    for _ in range(max(warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    if steps is None:  # size the region to about SUB_TIMED_S of device time
        t = timed_region(step, 10, dist, world) / 10
        steps = int(min(20000, max(20, SUB_TIMED_S * 1e3 / max(t, 1e-3))))
    # Region 1 (the value): plain launches, no per-kernel events, so consecutive kernels of a
    # call can overlap their launch through programmatic dependent launch.
    # Region 2 (the roofline): the same steps with an event pair recorded around every launch
    # on the launching stream; its per-kernel averages give each kernel's duration.
    result = None
    for attempt in range(2 if retry_clocks else 1):
        with ClockSampler(local) as cs:
            ms = timed_region(step, steps, dist, world)
        clocks = cs.summary()
        result = (ms, clocks)
        if not rejected(clocks):
            break
    ms, clocks = result
    lmh.trace_reset()
    lmh.trace_enable(True)
    ms_traced = timed_region(step, steps, dist, world)
    lmh.trace_enable(False)
    launches = 0
    per_kernel = {}
    for kname in lmh.lmh.TRACE_KERNELS:
        n, t = lmh.trace_read(kname)
        launches += n
        if n:
            per_kernel[kname] = {"launches": n, "avg_us": 1e3 * t / n}
    status = int(step.status.item()) if hasattr(step, "status") else 0
    if status:
        raise RuntimeError("device status %#x during the benchmark of %s" % (status, b["name"]))
    out = step.out
    gpu_ids = None if out.get("topk_ids") is None else out["topk_ids"].cpu().numpy()
    return {"step": step, "steps": steps, "ms": ms, "ms_traced": ms_traced, "clocks": clocks,
            "per_kernel": per_kernel, "launches": launches, "gpu_ids": gpu_ids}


_SHARED = {"decode_batch_k1": "decode_batch", "prefill_full": "prefill_batch"}


def run_ours(args):
    import torch
    import top_reduction_gb300 as lmh
    from top_reduction_gb300 import _build
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    _build.build()
    peaks, peak_src = load_peaks()

    b = apply_options(make_workload(args.workload, rank), args)
    m = measure(lmh, b, device, args.steps, args.warmup, dist, world, local, retry_clocks=True)
    value = job_value(m["step"].rows, args.steps, world, m["ms"])
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": m["ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(b),
            "roofline": roofline(b, m["per_kernel"], m["ms"] / args.steps, peaks, peak_src),
            "kernels": m["per_kernel"], "traced_ms_per_step": m["ms_traced"] / args.steps,
            # launches counted by the event trace over the second region, which runs the same steps
            "gpu_launches": m["launches"], "clocks": m["clocks"]}
    if rank == 0 and not args.no_e2e:
        line["e2e"] = e2e_leg(lmh, b, device, args.e2e_steps or max(200, min(args.steps, 2000)))
    head_ids = m["gpu_ids"]
    del m
    torch.cuda.empty_cache()

    # the other configurations, one at a time, each on its own inputs
    subs = {}
    cache = {}
    for name in ([] if args.no_sub else [w for w in WORKLOADS if w != args.workload]):
        base = _SHARED.get(name, name)
        if base not in cache:
            cache.clear()
            cache[base] = make_workload(base, rank)
        src = cache[base]
        if name == base:
            sb = src
        elif name == "decode_batch_k1":  # the decode batch's tensors at K 1
            sb = dict(src, name=name, k=1)
        else:  # the prefill batch's tensors, every packed row through the head
            sb = dict(src, name="prefill_full", num_decode=0, all_rows_mask=None, full=True,
                      n_sel=src["hidden"].shape[0], sel=src["sel_all"])
        sm = measure(lmh, sb, device, None, 10, dist, world, local, retry_clocks=False)
        rec = {"value": job_value(sm["step"].rows, sm["steps"], world, sm["ms"]), "unit": UNIT,
               "steps": sm["steps"], "ms_per_step": sm["ms"] / sm["steps"], "config": workload_config(sb),
               "roofline": roofline(sb, sm["per_kernel"], sm["ms"] / sm["steps"], peaks, peak_src),
               "kernels": sm["per_kernel"], "gpu_launches": sm["launches"], "clocks": sm["clocks"]}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            rec["cpu_baseline"] = cpu_baseline(sb, budget_s=4.0, single_s=2.0, gpu_ids=sm["gpu_ids"])
            rec["certified_swaps"] = rec["cpu_baseline"]["id_check"]["certified_swaps"]
        subs[name] = rec
        del sm
        torch.cuda.empty_cache()
    if subs:
        line["workloads"] = subs
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(b, gpu_ids=head_ids)
            line["certified_swaps"] = line["cpu_baseline"]["id_check"]["certified_swaps"]
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle, as it stands, on our arm's workload and metric, on the host cores.

    W warm-up steps (fewer if they would take more than a warm-up budget), then up to
    K timed steps; the run stops early once its time budget is spent (the line says
    how many steps ran).
    """
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    b = apply_options(make_workload(args.workload), args)
    st = OracleStep(b)
    budget, warm_budget = 150.0, 30.0
    tw = time.perf_counter()
    warm = 0
    while warm < args.warmup and (warm == 0 or time.perf_counter() - tw < warm_budget):
        st.run()
        warm += 1
    t0 = time.perf_counter()
    rows, steps = 0, 0
    while steps < args.steps and (steps == 0 or time.perf_counter() - t0 < budget):
        rows += st.run()
        steps += 1
    dt = time.perf_counter() - t0
    value = rows / dt
    sample = "%d of %d requested steps within a %.0f s budget; %s" % (steps, args.steps, budget, st.describe())
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * dt / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(b),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(st.threads), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
