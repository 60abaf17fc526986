"""Throughput of the drafter-sampling hot path on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

One step is one pass of every hot-path row over one batch of synthetic input,
at the batched-verify workload's sizes (B=16 sequences, gamma=6, V=128256,
K=32768, fp32 target logits, head hidden size 2048):

  calibrate   vt_calibrate_topk over 50M Zipf(1.1) token ids -> counts, Top-K
  trim        vt_trim_head: W [128256, 2048] bf16 -> W_trim [32768, 2048]
  draft x6    vt_draft_step: hidden [16, 2048] bf16 -> q[:, j, :], tokens[:, j]
  verify      vt_verify: logits [16, 7, 128256] fp32, q, tokens -> tokens, n

The metric is verified draft positions per second: B*gamma = 96 positions per
step divided by the step time.  Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "verified draft positions/sec (B=16, γ=6, V=128256, K=32768) + % of HBM BW"
UNIT = "positions/s"
L2_BYTES = 129 * 1000 * 1000
B, GAMMA, V, K, H = 16, 6, 128256, 32768, 2048
N_CAL = 50_000_000
T = 1.0
ROWS = ["calibrate", "trim", "draft", "verify"]


# ---------------------------------------------------------------- helpers
def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def peak_tensor_tflops():
    """Dense bf16 tensor peak for a kernel timed alone (the burst figure)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def max_over_ranks(torch, x: float, dist, dev) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(steps: int, world: int, total_ms: float) -> float:
    """Verified positions per second over all ranks: each rank verifies
    B * GAMMA positions per step."""
    return B * GAMMA * steps * world / (total_ms / 1e3)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def algorithmic_bytes():
    """Bytes each call must move at least once (decimal), per call."""
    return {
        # ids read, counts written, counts read by the selection, Top-K written
        "calibrate": N_CAL * 4 + V * 4 + V * 4 + K * 4,
        # selected rows read and written, ids in/out, inverse map written
        "trim": 2 * K * H * 2 + K * 4 * 2 + V * 4,
        # trimmed head read once, hidden read, q written, tokens/uniforms
        "draft": K * H * 2 + B * H * 2 + B * K * 4 + B * 4 * 2,
        # logits once, one q row per sequence, inv_map, the drafted ids and
        # their q, uniforms, outputs
        "verify": (B * (GAMMA + 1) * V * 4 + B * K * 4 + V * 4 + B * GAMMA * 4 * 3
                   + B * (GAMMA + 1) * 4 + B * (GAMMA + 1) * 4 + B * 4 + B * GAMMA * 4),
    }


CALLS_PER_STEP = {"calibrate": 1, "trim": 1, "draft": GAMMA, "verify": 1}
# kernels of this library launched per call (memsets issued by the driver
# are not counted)
# kernels launched per call: calibrate = zero, sample, hot select, main
# histogram, digit counts, and one radix pass per <= 10 bits of the largest
# possible count (N_CAL); trim = index mapper + gather; draft = projection +
# finalize; verify = stats + finish
_SORT_PASSES = -(-max(1, int(N_CAL).bit_length()) // 10)
KERNELS_PER_CALL = {"calibrate": 5 + _SORT_PASSES, "trim": 2, "draft": 2, "verify": 2}

KERNEL_SOURCES = {
    "calibrate": ["drafter_sampling_gb300/csrc/vt_calib.cu"],
    "trim": ["drafter_sampling_gb300/csrc/vt_calib.cu"],
    "draft": ["drafter_sampling_gb300/csrc/vt_draft.cu", "drafter_sampling_gb300/csrc/vt_umma.cuh"],
    "verify": ["drafter_sampling_gb300/csrc/vt_verify.cu"],
}


def _code_only(text: str) -> str:
    """C/CUDA source without its comments and blank space, so that a change
    to a comment does not count as a change to the kernels."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths + ["drafter_sampling_gb300/csrc/vt_common.cuh"]:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(row: str):
    """DRAM bytes per call from the committed ncu summary, if it was captured
    on the current source of that call's kernels; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        e = d[row]
        if e.get("source_digest") != source_digest(KERNEL_SOURCES[row]):
            return None
        return float(e["dram_bytes_per_call"])
    except Exception:
        return None


# ----------------------------------------------------------------- inputs
class HostInputs:
    """Seeded synthetic inputs of one step (numpy, host)."""

    def __init__(self):
        perm = synthetic.rank_permutation(V)
        self.ids = synthetic.zipf_ids(N_CAL, V, s=1.1, seed=synthetic.SEED_CALIB, perm=perm)
        self.W = synthetic.head_weights(V, H, seed=synthetic.SEED_CALIB)
        self.hidden = synthetic.hidden_states((GAMMA, B, H), seed=synthetic.SEED_VERIFY)
        self.u_draft = synthetic.uniforms(synthetic.SEED_VERIFY, 6, (GAMMA, B))
        vi = synthetic.verify_inputs(B=B, gamma=GAMMA, V=V, K=K, seed=synthetic.SEED_VERIFY)
        self.logits = vi["logits"]
        self.u_accept = vi["u_accept"]
        self.u_resample = vi["u_resample"]
        # the workload's own drafter distributions and drafts (correlated
        # with the logits), for the verify-only line and tau
        self.q_verify = vi["q"]
        self.draft_verify = vi["draft"]
        self.inv_map_verify = vi["inv_map"]

    def step_inputs(self):
        """What a step consumes from the host: the calibration ids, the
        drafter's hidden states and uniforms, the target's logits and the
        verification uniforms.  The drafter head's weights W are model state,
        resident on the device like any model's weights."""
        return dict(ids=self.ids, hidden=self.hidden, u_draft=self.u_draft,
                    logits=self.logits, u_accept=self.u_accept, u_resample=self.u_resample)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = []
        for t, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append((t, parts))
        inwin = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1] or rows
        if not inwin:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for _, p in inwin if num(p[0]) is not None]
        smax = [num(p[1]) for _, p in inwin if num(p[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in inwin:
            for name, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inwin)}


# -------------------------------------------------------------- GPU step
class GpuStep:
    """Device buffers, outputs and workspaces of one step."""

    def __init__(self, torch, vt, dev, host: HostInputs, nsets: int):
        self.torch, self.vt, self.dev = torch, vt, dev
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.ids = t(host.ids)
        self.W = t(host.W.view(np.int16))
        self.hidden = t(host.hidden.view(np.int16))
        self.u_draft = t(host.u_draft)
        base = dict(logits=t(host.logits), u_acc=t(host.u_accept), u_res=t(host.u_resample))
        self.vsets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
        i32 = torch.int32
        self.counts = torch.empty(V, dtype=i32, device=dev)
        self.topk = torch.empty(K, dtype=i32, device=dev)
        self.W_trim = torch.empty((K, H), dtype=torch.int16, device=dev)
        self.trim_ids = torch.empty(K, dtype=i32, device=dev)
        self.inv_map = torch.empty(V, dtype=i32, device=dev)
        self.q = torch.empty((B, GAMMA, K), dtype=torch.float32, device=dev)
        self.tokens = torch.empty((B, GAMMA), dtype=i32, device=dev)
        self.out_tokens = torch.empty((B, GAMMA + 1), dtype=i32, device=dev)
        self.out_n = torch.empty(B, dtype=i32, device=dev)
        self.out_acc = torch.empty((B, GAMMA), dtype=torch.float32, device=dev)
        self.status = torch.zeros(4, dtype=i32, device=dev)
        # the per-position views a decoder holds for its drafting steps
        # (hidden states, uniforms, q column, token column), made once
        self.draft_views = [(self.hidden[j], self.u_draft[j], self.q[:, j, :], self.tokens[:, j])
                            for j in range(GAMMA)]
        self.status_views = [self.status[i:i + 1] for i in range(4)]
        u8 = torch.uint8
        self.ws_cal = torch.empty(vt.workspace_bytes("calibrate", n=N_CAL, V=V, K=K), dtype=u8,
                                  device=dev)
        self.ws_trim = torch.empty(vt.workspace_bytes("trim", V=V, K=K), dtype=u8, device=dev)
        self.ws_draft = torch.empty(vt.workspace_bytes("draft", B=B, H=H, K=K), dtype=u8,
                                    device=dev)
        self.ws_ver = torch.empty(vt.workspace_bytes("verify", B=B, gamma=GAMMA, V=V, K=K),
                                  dtype=u8, device=dev)
        self.nsets = nsets

    def run(self, k: int, events=None, group=None):
        """One step.  `events` maps row -> list of (start, end) events around
        every call of the row; `group` = (row, start, end) records one pair of
        events around all calls of one row (the other calls stay back to back,
        so their programmatic-dependent-launch overlap is kept)."""
        vt = self.vt
        s = self.vsets[k % self.nsets]
        ncalls = {"calibrate": 1, "trim": 1, "draft": GAMMA, "verify": 1}

        def mark(row, i):
            if events is not None:
                events[row][i].record()
            if group is not None and group[0] == row:
                if i == 0:
                    group[1].record()
                elif i == 2 * ncalls[row] - 1:
                    group[2].record()

        sv = self.status_views
        mark("calibrate", 0)
        vt.vt_calibrate_topk(self.ids, V, K, counts=self.counts, topk_ids=self.topk,
                             dev_status=sv[0], workspace=self.ws_cal)
        mark("calibrate", 1)
        mark("trim", 0)
        vt.vt_trim_head(self.W, self.topk, W_trim=self.W_trim, trim_ids=self.trim_ids,
                        inv_map=self.inv_map, dev_status=sv[1], workspace=self.ws_trim)
        mark("trim", 1)
        for j in range(GAMMA):
            hj, uj, qj, tj = self.draft_views[j]
            mark("draft", 2 * j)
            vt.vt_draft_step(hj, self.W_trim, self.trim_ids, uj, T, q=qj, tokens=tj,
                             dev_status=sv[2], workspace=self.ws_draft)
            mark("draft", 2 * j + 1)
        mark("verify", 0)
        vt.vt_verify(s["logits"], self.q, self.inv_map, self.tokens, s["u_acc"], s["u_res"], T,
                     out_tokens=self.out_tokens, out_num_accepted=self.out_n,
                     out_accept_prob=self.out_acc, dev_status=sv[3], workspace=self.ws_ver)
        mark("verify", 1)


# ------------------------------------------------- the oracle on the host
def oracle_step(x, draft_steps: int = GAMMA):
    """One step of the hot path on the CPU oracle, on the step's own inputs:
    the 50M-id histogram and Top-K, the trim, `draft_steps` drafting steps of
    B = 16 rows over the full trimmed head, and the verification of all 16
    sequences.  Returns seconds per row."""
    import oracle
    t = {}
    t0 = time.perf_counter()
    topk = oracle.top_k(oracle.token_histogram(x["ids"], V), K)
    t1 = time.perf_counter()
    W_trim, trim_ids, inv_map = oracle.trim_head(x["W"], topk)
    t2 = time.perf_counter()
    q = np.zeros((B, GAMMA, K))
    tokens = np.zeros((B, GAMMA), dtype=np.int32)
    for j in range(GAMMA):
        if j < draft_steps:
            d = oracle.draft_step(x["hidden"][j], W_trim, trim_ids, x["u_draft"][j], T)
            q[:, j, :], tokens[:, j] = d["q"], d["tokens"]
        else:  # the remaining positions reuse the first drafted q and tokens
            q[:, j, :], tokens[:, j] = q[:, 0, :], tokens[:, 0]
    t3 = time.perf_counter()
    oracle.verify(x["logits"], q, inv_map, tokens, x["u_accept"], x["u_resample"], T)
    t4 = time.perf_counter()
    return {"calibrate": t1 - t0, "trim": t2 - t1, "draft": (t3 - t2) / draft_steps,
            "verify": t4 - t3}


def oracle_child(path: str, mode: str, runs: int) -> int:
    """Entry of the spawned process that times the oracle on the step's
    inputs (saved by the parent as .npy files in `path`); prints one JSON
    line with the per-run row seconds."""
    x = {n: np.load(os.path.join(path, n + ".npy"), mmap_mode="r")
         for n in ("ids", "W", "hidden", "u_draft", "logits", "u_accept", "u_resample")}
    x = {n: np.ascontiguousarray(v) for n, v in x.items()}
    steps = GAMMA if mode == "all" else 1
    oracle_step(x, steps)  # warm-up
    out = [oracle_step(x, steps) for _ in range(runs)]
    print(json.dumps({"runs": out, "cpu_count": os.cpu_count()}))
    return 0


ORACLE_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
                      "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")


def cpu_baseline_measure(host: HostInputs, runs: int = 5):
    """The oracle as it stands, timed on whole rows of the step's own inputs
    in child processes: once with every host core available (numpy's BLAS
    threads; the histogram and the verification loop are single-threaded
    numpy) and once pinned to one thread.  Medians of `runs` runs."""
    import tempfile
    inp = host.step_inputs()
    inp["W"] = host.W
    res = {}
    with tempfile.TemporaryDirectory() as d:
        for n, v in inp.items():
            np.save(os.path.join(d, n + ".npy"), np.ascontiguousarray(v))
        for mode in ("all", "one"):
            env = {k: v for k, v in os.environ.items() if k not in ORACLE_THREAD_VARS}
            if mode == "one":
                env.update({k: "1" for k in ORACLE_THREAD_VARS})
            r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-child", d,
                                "--oracle-mode", mode, "--oracle-runs", str(runs)],
                               capture_output=True, text=True, env=env, timeout=900)
            if r.returncode != 0:
                raise RuntimeError(f"oracle timing failed: {r.stderr[-2000:]}")
            res[mode] = json.loads(r.stdout.strip().splitlines()[-1])
    out = {}
    for mode, d in res.items():
        rows = {r: statistics.median([x[r] for x in d["runs"]]) for r in ROWS}
        per_step = rows["calibrate"] + rows["trim"] + GAMMA * rows["draft"] + rows["verify"]
        out[mode] = {"rows_s": rows, "s_per_step": per_step, "cpu_count": d["cpu_count"],
                     "runs": len(d["runs"])}
    return out


def config_dict(world: int):
    """The workload of one step, identical in both arms' lines."""
    return {"workload": workload_text(), "global_batch": B * world, "seq_len": GAMMA + 1,
            "parallelism": f"replicas x{world}",
            "l2": "each step streams >1.3 GB (>4x L2) of distinct inputs; logits rotate over "
                  "2 buffers"}


def run_reference(args):
    """The oracle as the reference arm: every step is one full step of the
    hot path on the CPU oracle (no sampling, no extrapolation), on every host
    core numpy's BLAS uses; rank 0 alone runs it."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    host = HostInputs()
    x = dict(host.step_inputs(), W=host.W)
    for _ in range(args.warmup):
        oracle_step(x)
    t0 = time.perf_counter()
    per = [oracle_step(x) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    value = whole_job_value(args.steps, 1, wall * 1e3)
    rows = {r: statistics.median([p[r] for p in per]) for r in ROWS}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{args.steps} full steps of the workload timed back to "
                                       "back (50M-id histogram and Top-K, trim, 6 drafting "
                                       "steps of 16 rows, verification of 16 sequences), numpy "
                                       "fp64, BLAS on all cores",
                             "median_row_s": rows},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_text():
    return ("speculative block with VocabTrim calibration: calibrate 50M Zipf(1.1) ids -> "
            "Top-32768 of V=128256, trim W[128256,2048] bf16, 6 drafter steps B=16, "
            "verify B=16 gamma=6 fp32 logits N(0,2)+3 ln Zipf_1.1 rank bias, T=1")


def run_row(torch, vt, dev, host, args):
    """Profiling mode: one full step (it fills W_trim, q, the drafts and the
    inverse map), then only `args.row`'s calls for warmup + steps iterations,
    in a process that holds one set of the step's buffers (~1.6 GB).  Made for
    ncu captures of one kernel (-k, -s 1 skips the set-up step's launch)."""
    step = GpuStep(torch, vt, dev, host, nsets=1)
    step.run(0)
    torch.cuda.synchronize()
    s = step.vsets[0]
    calls = {
        "calibrate": lambda: vt.vt_calibrate_topk(step.ids, V, K, counts=step.counts,
                                                  topk_ids=step.topk,
                                                  dev_status=step.status[0:1],
                                                  workspace=step.ws_cal),
        "trim": lambda: vt.vt_trim_head(step.W, step.topk, W_trim=step.W_trim,
                                        trim_ids=step.trim_ids, inv_map=step.inv_map,
                                        dev_status=step.status[1:2], workspace=step.ws_trim),
        "draft": lambda: [vt.vt_draft_step(step.hidden[j], step.W_trim, step.trim_ids,
                                           step.u_draft[j], T, q=step.q[:, j, :],
                                           tokens=step.tokens[:, j],
                                           dev_status=step.status[2:3],
                                           workspace=step.ws_draft) for j in range(GAMMA)],
        # the drafter's top-8 candidates (the expansion step of a draft tree)
        "topk": lambda: vt.vt_draft_topk(step.hidden[0], step.W_trim, step.trim_ids, 8, T),
        "verify": lambda: vt.vt_verify(s["logits"], step.q, step.inv_map, step.tokens,
                                       s["u_acc"], s["u_res"], T, out_tokens=step.out_tokens,
                                       out_num_accepted=step.out_n,
                                       out_accept_prob=step.out_acc,
                                       dev_status=step.status[3:4], workspace=step.ws_ver),
    }
    fn = calls[args.row]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ncalls = args.steps * CALLS_PER_STEP.get(args.row, 1)
    per_call = e0.elapsed_time(e1) * 1e3 / ncalls
    print(json.dumps({"row": args.row, "calls": ncalls,
                      "us_per_call": per_call,
                      "dev_status": [int(v) for v in step.status.cpu().tolist()]}))
    return 0


def run_row_large(torch, vt, dev, args):
    """Profiling mode for the large-batch drafting step (B = 256, H = 4096,
    K = 38016 trimmed rows, T = 0.7: the tcgen05 tiles of 256 batch columns,
    two 128-row tiles per CTA): random inputs of those shapes built on the
    device (about 0.4 GB), then warmup + steps calls."""
    B4, H4, K4, T4 = 256, 4096, 38016, 0.7
    gen = torch.Generator(device=dev)
    gen.manual_seed(21)
    hidden = torch.randn((B4, H4), generator=gen, device=dev).to(torch.bfloat16)
    W_trim = (torch.randn((K4, H4), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    trim_ids = torch.arange(K4, dtype=torch.int32, device=dev)
    u = torch.rand(B4, generator=gen, device=dev)
    q = torch.empty((B4, K4), dtype=torch.float32, device=dev)
    tok = torch.empty(B4, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(vt.workspace_bytes("draft", B=B4, H=H4, K=K4), dtype=torch.uint8, device=dev)

    def fn():
        vt.vt_draft_step(hidden, W_trim, trim_ids, u, T4, q=q, tokens=tok, dev_status=st,
                         workspace=ws)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"row": args.row, "calls": args.steps,
                      "us_per_call": e0.elapsed_time(e1) * 1e3 / max(1, args.steps),
                      "dev_status": int(st.item())}))
    return 0


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--row", default=None, choices=ROWS + ["topk", "draft_large"],
                    help="profiling mode: after one full step, run only this row's calls for "
                         "warmup + steps iterations (prints a short summary, not the bench line)")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-mode", default="all", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-runs", type=int, default=5, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        return oracle_child(args.oracle_child, args.oracle_mode, args.oracle_runs)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    import drafter_sampling_gb300 as vt

    if args.row == "draft_large":
        return run_row_large(torch, vt, dev, args)
    host = HostInputs()
    if args.row:
        return run_row(torch, vt, dev, host, args)
    # every step streams ~1.3 GB (ids, W, W_trim, logits), far more than L2,
    # so no input is L2-resident when the next step reads it; the logits also
    # rotate between two buffers
    step = GpuStep(torch, vt, dev, host, nsets=2)
    stream = torch.cuda.current_stream()
    for k in range(max(3, args.warmup)):
        step.run(k)
    torch.cuda.synchronize()

    # per-row call times from a short profiling pass with events around every
    # call (events between calls serialise the launch overlap of consecutive
    # kernels, so this pass is not the timed one)
    peak, peak_kind = peaks()
    peak_tf = peak_tensor_tflops()
    alg = algorithmic_bytes()
    nev = {"calibrate": 2, "trim": 2, "draft": 2 * GAMMA, "verify": 2}
    nprof = 5
    events = [{r: [torch.cuda.Event(enable_timing=True) for _ in range(nev[r])] for r in ROWS}
              for _ in range(nprof)]
    for k in range(nprof):
        step.run(k, events[k])
    torch.cuda.synchronize()
    call_us = {r: [] for r in ROWS}
    for ev in events:
        for r in ROWS:
            e = ev[r]
            for i in range(0, len(e), 2):
                call_us[r].append(e[i].elapsed_time(e[i + 1]) * 1e3)
    rows = {}
    for r in ROWS:
        avg = float(np.mean(call_us[r]))
        ach = alg[r] / (avg * 1e-6) / 1e9
        rows[r] = {"calls_per_step": CALLS_PER_STEP[r], "avg_call_us_isolated": avg,
                   "algorithmic_bytes": alg[r], "achieved_gbs_isolated": ach,
                   "frac_isolated": ach / peak, "traffic": traffic_for(r),
                   "kernels_per_call": KERNELS_PER_CALL[r]}
    dominant = max(ROWS, key=lambda r: rows[r]["avg_call_us_isolated"] * CALLS_PER_STEP[r])

    # the timed region: K steps back to back; one pair of events per step
    # around the calls of the dominant row gives its live per-call time
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    clocks = ClockSampler(int(vis) if vis.isdigit() else local)
    clocks.start()
    time.sleep(0.3)
    # every eighth step (at least one) carries the event pair, so the rest of
    # the timed region runs without any event between its kernels
    sampled = set(range(min(4, args.steps - 1), args.steps, 8))
    groups = [(dominant, torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              if k in sampled else None for k in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(args.steps):
        step.run(k, group=groups[k])
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist is not None:
        dist.barrier()
    clocks.stop()
    total_ms = max_over_ranks(torch, start.elapsed_time(end), dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_value(args.steps, world, total_ms)
    status = [int(x) for x in step.status.cpu().tolist()]
    live_us = float(np.mean([g[1].elapsed_time(g[2]) * 1e3 for g in groups if g is not None])) \
        / CALLS_PER_STEP[dominant]
    dom = dict(rows[dominant])
    dom["avg_call_us"] = live_us
    dom["achieved_gbs"] = alg[dominant] / (live_us * 1e-6) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": config_dict(world),
        "roofline": {"bound": "hbm", "kernel": f"vt_{dominant} (dominant row)",
                     "achieved": dom["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": dom["achieved_gbs"] / peak, "traffic": dom["traffic"],
                     "algorithmic_bytes": dom["algorithmic_bytes"],
                     "avg_launch_us": dom["avg_call_us"],
                     "timing": "events around the row's calls in every timed step, "
                               "averaged per call",
                     "peak_source": f"{peak_kind} hbm_gbs (copy, of measured)"},
        "rows": rows,
        "verify_only": {"value": B * GAMMA / (rows["verify"]["avg_call_us_isolated"] * 1e-6),
                        "unit": UNIT,
                        "timing": "one event pair around each call of a short profiling pass"},
        "gpu_launches": sum(KERNELS_PER_CALL[r] * CALLS_PER_STEP[r] for r in ROWS) * args.steps,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "dev_status": status,
        "next_rows": {"greedy_block": run_greedy_block(torch, vt, step),
                      **run_selection(torch, vt, step),
                      "block_graph": run_block_graph(torch, vt, step),
                      "verify_batched": run_verify_batched(torch, vt, step, host),
                      "toy_chain": run_toy_chain(torch, vt),
                      **run_tree(torch, vt, step)},
    }
    if not args.no_configs:
        line["configs_measured"] = {
            "note": "the head, calibration and large-batch configurations, each timed as one "
                    "CUDA graph of calls (no host overhead); not part of the step",
            "trimmed_vs_full_head": run_head_batches(torch, vt, step, peak),
            "calibration_H3072": run_calibration_h3072(torch, vt, step, peak),
            "large_batch_B256": run_large_batch(torch, vt, step, peak, peak_tf)}

    line["timing_distribution"] = run_timing_distribution(torch, vt, step, host)
    # B * gamma / t(vt_verify) with t from graphs of back-to-back calls (no
    # event between calls), beside the event-pair figure above
    tv = line["timing_distribution"]["verify"]["graph_per_call"]["median_us"]
    line["verify_only"]["graph_value"] = B * GAMMA / (tv * 1e-6)
    line["verify_only"]["graph_us_per_call"] = tv
    line["verify_only"]["graph_frac_of_measured_hbm"] = \
        alg["verify"] / (tv * 1e-6) / 1e9 / peak
    if not args.no_e2e:
        line["e2e"] = run_e2e(torch, step, host, stream, args, dist, dev, world)
        line["e2e_online_block"] = run_e2e_block(torch, step, host, stream, args, dist, dev,
                                                 world)
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline_measure(host)
        line["cpu_baseline"] = {
            "value": B * GAMMA / cb["all"]["s_per_step"], "unit": UNIT,
            "cores": cb["all"]["cpu_count"], "kind": "oracle",
            "sample": "whole rows of the step's own inputs, median of 5 runs each: the 50M-id "
                      "histogram and Top-K, the trim, 6 drafting steps of 16 rows over the full "
                      "trimmed head, the verification of 16 sequences; numpy fp64 with its "
                      "BLAS on every host core (histogram and verification loops on one core)",
            "median_row_s": cb["all"]["rows_s"],
            "single_thread": {"value": B * GAMMA / cb["one"]["s_per_step"], "unit": UNIT,
                              "cores": 1, "median_row_s": cb["one"]["rows_s"],
                              "sample": "the same rows with one BLAS thread; one drafting "
                                        "step timed per run, counted 6 times per step"}}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


def run_greedy_block(torch, vt, step, nblocks: int = 100):
    """Greedy (temperature 0) block on the step's tensors: six greedy draft
    steps (argmax through the trimmed head, one-hot q) and greedy
    verification (argmax of every target row).  Timed back to back with one
    event pair around all blocks; the drafts reuse the calibrated W_trim."""
    s = step.vsets[0]

    def block():
        for j in range(GAMMA):
            vt.vt_draft_step(step.hidden[j], step.W_trim, step.trim_ids, None, 0.0,
                             q=step.q[:, j, :], tokens=step.tokens[:, j],
                             dev_status=step.status[2:3], workspace=step.ws_draft)
        vt.vt_verify(s["logits"], None, None, step.tokens, None, None, 0.0,
                     out_tokens=step.out_tokens, out_num_accepted=step.out_n,
                     out_accept_prob=step.out_acc, dev_status=step.status[3:4],
                     workspace=step.ws_ver)

    for _ in range(3):
        block()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(nblocks):
        block()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / nblocks
    alg = algorithmic_bytes()
    # greedy verify reads the logits once (no q, no residual row)
    bytes_block = GAMMA * alg["draft"] + B * (GAMMA + 1) * V * 4
    status = [int(x) for x in step.status[2:4].cpu().tolist()]
    return {"value": B * GAMMA / (us * 1e-6), "unit": UNIT, "us_per_block": us,
            "algorithmic_bytes_per_block": bytes_block,
            "achieved_gbs": bytes_block / (us * 1e-6) / 1e9,
            "mean_accepted": float(step.out_n.float().mean().item()), "dev_status": status,
            "note": "temperature 0: greedy drafting and verification, calibrate/trim excluded"}


def run_tree(torch, vt, step, ncalls: int = 100):
    """Draft trees of the pages' size (32 nodes) for the step's batch:
    vt_verify_tree over [B, 33, V] fp32 logits (seeded normal values, one
    shared random tree shape) and vt_draft_topk (k = 8) through the
    calibrated trimmed head."""
    N, k = 32, 8
    gen = torch.Generator(device=step.dev)
    gen.manual_seed(5)
    logits = torch.randn((B, N + 1, V), generator=gen, device=step.dev, dtype=torch.float32)
    g = np.random.default_rng(5)
    parent = torch.tensor([-1] + [int(g.integers(-1, i)) for i in range(1, N)],
                          dtype=torch.int32, device=step.dev)
    tokens = torch.randint(0, V, (B, N), generator=gen, device=step.dev, dtype=torch.int32)
    out = torch.empty((B, N + 1), dtype=torch.int32, device=step.dev)
    n = torch.empty(B, dtype=torch.int32, device=step.dev)
    path = torch.empty((B, N), dtype=torch.int32, device=step.dev)
    ws_t = torch.empty(vt.lib().vt_verify_tree_workspace_bytes(B, N, V), dtype=torch.uint8,
                       device=step.dev)
    ids = torch.empty((B, k), dtype=torch.int32, device=step.dev)
    logq = torch.empty((B, k), dtype=torch.float32, device=step.dev)
    ws_k = torch.empty(vt.lib().vt_draft_topk_workspace_bytes(B, H, K, k), dtype=torch.uint8,
                       device=step.dev)
    calls = {
        "tree_verify_32": (lambda: vt.vt_verify_tree(
            logits, parent, tokens, out_tokens=out, out_num_accepted=n, out_path=path,
            dev_status=step.status[3:4], workspace=ws_t), B * (N + 1) * V * 4),
        "draft_topk_8": (lambda: vt.vt_draft_topk(
            step.hidden[0], step.W_trim, step.trim_ids, k, T, out_ids=ids, out_logq=logq,
            dev_status=step.status[2:3], workspace=ws_k), K * H * 2 + 2 * B * K * 4),
    }
    res = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(ncalls):
            fn()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / ncalls
        res[name] = {"us_per_call": us, "algorithmic_bytes": nbytes,
                     "achieved_gbs": nbytes / (us * 1e-6) / 1e9}
    res["tree_verify_32"]["mean_accepted"] = float(n.float().mean().item())
    del logits
    return res


def run_verify_batched(torch, vt, step, host, ncalls: int = 200):
    """vt_verify alone on the batched-verify workload's own q and drafts
    (q = softmax over the trimmed ids of logit + N(0,1), drafts drawn from
    q): verified positions/s of the verify call and tau = mean tokens per
    block (accepted + 1)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(step.dev)
    q, draft, inv_map = t(host.q_verify), t(host.draft_verify), t(host.inv_map_verify)

    def call(k):
        s = step.vsets[k % step.nsets]
        vt.vt_verify(s["logits"], q, inv_map, draft, s["u_acc"], s["u_res"], T,
                     out_tokens=step.out_tokens, out_num_accepted=step.out_n,
                     out_accept_prob=step.out_acc, dev_status=step.status[3:4],
                     workspace=step.ws_ver)

    call(0)
    torch.cuda.synchronize()
    tau = float((step.out_n.float() + 1).mean().item())
    status = int(step.status[3].item())
    for k in range(3):
        call(k)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(ncalls):
        call(k)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / ncalls
    return {"value": B * GAMMA / (us * 1e-6), "unit": UNIT, "us_per_call": us,
            "achieved_gbs": algorithmic_bytes()["verify"] / (us * 1e-6) / 1e9, "tau": tau,
            "dev_status": status,
            "note": "verify only, logits rotating over 2 buffers; tau from the first call"}


def run_block_graph(torch, vt, step, nblocks: int = 100):
    """The speculative block (six drafting steps + verification, T = 1) as
    one CUDA graph replayed back to back, beside the same calls launched
    one by one; tau = mean tokens emitted per block (accepted + 1)."""
    s = step.vsets[0]
    g = vt.BlockGraph(step.hidden, step.W_trim, step.trim_ids, step.inv_map, s["logits"],
                      u_draft=step.u_draft, u_accept=s["u_acc"], u_resample=s["u_res"],
                      temperature=T)

    def direct():
        for j in range(GAMMA):
            vt.vt_draft_step(step.hidden[j], step.W_trim, step.trim_ids, step.u_draft[j], T,
                             q=step.q[:, j, :], tokens=step.tokens[:, j],
                             dev_status=step.status[2:3], workspace=step.ws_draft)
        vt.vt_verify(s["logits"], step.q, step.inv_map, step.tokens, s["u_acc"], s["u_res"], T,
                     out_tokens=step.out_tokens, out_num_accepted=step.out_n,
                     out_accept_prob=step.out_acc, dev_status=step.status[3:4],
                     workspace=step.ws_ver)

    res = {}
    for name, fn in (("graph", g.launch), ("direct", direct)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(nblocks):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) * 1e3 / nblocks
    tau = float((g.out_num_accepted.float() + 1).mean().item())
    status = [int(x) for x in g.dev_status.cpu().tolist()]
    g.close()
    # Overlap of block k+1's W_trim stream with block k's verification: the
    # first projection of a block requests its W_trim stages before its
    # dependency wait, while the verification's finish (which releases its
    # dependents early) still runs.  Measured two ways:
    #  - graphs of 20 consecutive blocks against graphs of one block (no
    #    kernel of the previous replay to overlap);
    #  - direct blocks back to back against the same with an event recorded
    #    between blocks (an event between kernels cuts the overlap).
    sep = torch.cuda.Event()

    def direct_cut():
        direct()
        sep.record()

    for name, fn in (("direct_cut", direct_cut),):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(nblocks):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) * 1e3 / nblocks
    res["graph_of_1"] = graph_us(torch, direct, 1, reps=20)
    res["graph_of_20"] = graph_us(torch, direct, 20, reps=5)
    return {"value": B * GAMMA / (res["graph"] * 1e-6), "unit": UNIT,
            "us_per_block_graph": res["graph"], "us_per_block_direct": res["direct"],
            "tau": tau, "dev_status": status,
            "w_trim_overlap": {
                "us_per_block_graph_of_1": res["graph_of_1"],
                "us_per_block_graph_of_20": res["graph_of_20"],
                "us_per_block_direct_cut": res["direct_cut"],
                "us_per_block_direct": res["direct"],
                "gain_graph_us": res["graph_of_1"] - res["graph_of_20"],
                "note": "block k+1's first projection streams W_trim during block k's "
                        "verification; 'cut': an event between blocks removes the overlap"},
            "note": "drafting steps + verification as one CUDA graph (calibrate/trim excluded); "
                    "tau = mean tokens per block on the synthetic (unaligned) drafter; tau on "
                    "the toy workload is next_rows.toy_chain"}


def run_selection(torch, vt, step, ncalls: int = 20):
    """Top-P (P = 0.95) and minimum-frequency (f = 64) selection on the
    step's 50M calibration ids: histogram, full ranking and K per call."""
    out = {}
    ws = torch.empty(vt.workspace_bytes("select", n=N_CAL, V=V), dtype=torch.uint8,
                     device=step.ids.device)
    ranked = torch.empty(V, dtype=torch.int32, device=step.ids.device)
    k_out = torch.empty(1, dtype=torch.int32, device=step.ids.device)
    calls = {"top_p_0.95": lambda: vt.vt_calibrate_top_p(
                 step.ids, V, 0.95, counts=step.counts, ranked_ids=ranked, k_out=k_out,
                 dev_status=step.status[0:1], workspace=ws),
             "min_count_64": lambda: vt.vt_calibrate_min_count(
                 step.ids, V, 64, counts=step.counts, ranked_ids=ranked, k_out=k_out,
                 dev_status=step.status[0:1], workspace=ws)}
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(ncalls):
            fn()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / ncalls
        out["calibrate_" + name] = {"us_per_call": us, "K": int(k_out.item()),
                                    "achieved_gbs": algorithmic_bytes()["calibrate"] / (us * 1e-6) / 1e9,
                                    "dev_status": int(step.status[0].item())}
    return out


def graph_us(torch, fn, ncalls: int, reps: int = 3):
    """Median per-call time of `fn` captured ncalls times in one CUDA graph
    (host overhead excluded), after two warm replays."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(ncalls):
                fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ts = []
    for r in range(reps + 2):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        if r >= 2:
            ts.append(e0.elapsed_time(e1) * 1e3 / ncalls)
    del g
    return float(np.median(ts))


def run_head_batches(torch, vt, step, peak, ncalls: int = 24):
    """The head configuration: one drafting step (projection, softmax,
    draw) through the trimmed head (K = 32768) and through the full head
    (K = V = 128256) at B in {1, 8, 16, 64}, H = 2048, T = 1.  Two W_trim
    copies alternate so that consecutive calls never find theirs in L2 (the
    full head, 525 MB, exceeds L2 alone)."""
    dev = step.dev
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    Wt = [step.W_trim, step.W_trim.clone()]
    full_ids = torch.arange(V, dtype=torch.int32, device=dev)
    out = {}
    for Bx in (1, 8, 16, 64):
        hid = (torch.randn((Bx, H), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
        u = torch.rand(Bx, generator=gen, device=dev)
        row = {}
        for name, Ws, ids, Kx in (("trimmed", Wt, step.trim_ids, K), ("full", [step.W], full_ids, V)):
            q = torch.empty((Bx, Kx), dtype=torch.float32, device=dev)
            tok = torch.empty(Bx, dtype=torch.int32, device=dev)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            ws = torch.empty(vt.lib().vt_draft_workspace_bytes(Bx, H, Kx), dtype=torch.uint8,
                             device=dev)
            it = [0]

            def fn(Ws=Ws, ids=ids, q=q, tok=tok, st=st, ws=ws):
                it[0] += 1
                vt.vt_draft_step(hid, Ws[it[0] % len(Ws)], ids, u, 1.0, q=q, tokens=tok,
                                 dev_status=st, workspace=ws)
            us = graph_us(torch, fn, ncalls)
            nbytes = Kx * H * 2 + Bx * H * 2 + Bx * Kx * 4
            row[name] = {"us_per_step": us, "algorithmic_bytes": nbytes,
                         "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
                         "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                         "dev_status": int(st.item())}
            del q, ws
        row["speedup_full_over_trimmed"] = row["full"]["us_per_step"] / row["trimmed"]["us_per_step"]
        row["ideal_speedup_bytes"] = (V * H * 2 + Bx * V * 4) / (K * H * 2 + Bx * K * 4)
        out[f"B{Bx}"] = row
    del Wt
    return out


def run_calibration_h3072(torch, vt, step, peak):
    """The calibration configuration: the step's 50M Zipf(1.1) ids
    -> Top-K for K in {8192, 16384, 32768, 65536}, and the row gather of
    W [128256, 3072] bf16 N(0, 0.02) into W_trim (timed apart: one graph of
    calls each)."""
    dev = step.dev
    H3 = 3072
    gen = torch.Generator(device=dev)
    gen.manual_seed(12)
    W3 = (torch.randn((V, H3), generator=gen, device=dev) * 0.02).to(torch.bfloat16) \
        .view(torch.int16)
    out = {}
    for Kc in (8192, 16384, 32768, 65536):
        counts = torch.empty(V, dtype=torch.int32, device=dev)
        topk = torch.empty(Kc, dtype=torch.int32, device=dev)
        st = torch.zeros(2, dtype=torch.int32, device=dev)
        wsc = torch.empty(vt.lib().vt_calibrate_topk_workspace_bytes(N_CAL, V, Kc),
                          dtype=torch.uint8, device=dev)
        Wt = torch.empty((Kc, H3), dtype=torch.int16, device=dev)
        ti = torch.empty(Kc, dtype=torch.int32, device=dev)
        im = torch.empty(V, dtype=torch.int32, device=dev)
        wst = torch.empty(vt.lib().vt_trim_head_workspace_bytes(V, Kc), dtype=torch.uint8,
                          device=dev)

        def cal():
            vt.vt_calibrate_topk(step.ids, V, Kc, counts=counts, topk_ids=topk,
                                 dev_status=st[0:1], workspace=wsc)

        def trim():
            vt.vt_trim_head(W3, topk, W_trim=Wt, trim_ids=ti, inv_map=im, dev_status=st[1:2],
                            workspace=wst)
        us_c = graph_us(torch, cal, 8)
        us_t = graph_us(torch, trim, 8)
        bc = N_CAL * 4 + 2 * V * 4 + Kc * 4
        bt = 2 * Kc * H3 * 2 + Kc * 4 * 2 + V * 4
        out[f"K{Kc}"] = {"calibrate_us": us_c, "calibrate_gbs": bc / (us_c * 1e-6) / 1e9,
                         "calibrate_frac": bc / (us_c * 1e-6) / 1e9 / peak,
                         "trim_us": us_t, "trim_gbs": bt / (us_t * 1e-6) / 1e9,
                         "trim_frac": bt / (us_t * 1e-6) / 1e9 / peak,
                         "dev_status": [int(x) for x in st.cpu().tolist()]}
        del counts, topk, wsc, Wt, ti, im, wst
    del W3
    return out


def run_large_batch(torch, vt, step, peak, peak_tf):
    """The large-batch configuration: B=256, gamma=8, V=152064,
    H=4096, K=38016 trimmed ids, T=0.7.  One drafting step (tcgen05 tiles of
    256 batch columns) and one verification over bf16 logits; inputs built on
    the device with the recipe's shape: logits N(0,2) + 3 ln Zipf_1.1(rank),
    q = softmax over the trimmed ids of (logit + N(0,1)) / T, drafts drawn
    from q."""
    dev = step.dev
    B4, G4, V4, H4, K4, T4 = 256, 8, 152064, 4096, 38016, 0.7
    gen = torch.Generator(device=dev)
    gen.manual_seed(13)
    perm = torch.randperm(V4, generator=gen, device=dev)
    trim_ids = torch.sort(perm[:K4]).values.to(torch.int32)   # the K4 best ranks, ascending ids
    inv_map = torch.full((V4,), -1, dtype=torch.int32, device=dev)
    inv_map[trim_ids.long()] = torch.arange(K4, dtype=torch.int32, device=dev)
    rank_of = torch.empty(V4, dtype=torch.float64, device=dev)
    rank_of[perm] = torch.arange(1, V4 + 1, dtype=torch.float64, device=dev)
    bias = (3.0 * (-1.1 * torch.log(rank_of))).to(torch.float32)
    logits = (torch.randn((B4, G4 + 1, V4), generator=gen, device=dev) * 2.0 + bias) \
        .to(torch.bfloat16)
    x = logits[:, :G4, :].float()[:, :, trim_ids.long()] + \
        torch.randn((B4, G4, K4), generator=gen, device=dev)
    q = torch.softmax(x / T4, dim=-1).contiguous()
    del x
    draft = trim_ids[torch.multinomial(q.view(-1, K4), 1, generator=gen).view(B4, G4)].contiguous()
    u_acc = torch.rand((B4, G4), generator=gen, device=dev)
    u_res = torch.rand((B4, G4 + 1), generator=gen, device=dev)
    out_tok = torch.empty((B4, G4 + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty(B4, dtype=torch.int32, device=dev)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    wsv = torch.empty(vt.lib().vt_verify_workspace_bytes(B4, G4, V4, K4), dtype=torch.uint8,
                      device=dev)

    def ver():
        vt.vt_verify(logits, q, inv_map, draft, u_acc, u_res, T4, out_tokens=out_tok,
                     out_num_accepted=out_n, dev_status=st[0:1], workspace=wsv)
    us_v = graph_us(torch, ver, 10)
    bv = B4 * (G4 + 1) * V4 * 2 + B4 * K4 * 4 + V4 * 4
    res = {"verify_us": us_v, "verify_algorithmic_bytes": bv,
           "verify_gbs": bv / (us_v * 1e-6) / 1e9, "verify_frac": bv / (us_v * 1e-6) / 1e9 / peak,
           "mean_accepted": float(out_n.float().mean().item())}
    del logits, q, wsv
    Wt = [(torch.randn((K4, H4), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
          .view(torch.int16) for _ in range(2)]
    hid = torch.randn((B4, H4), generator=gen, device=dev).to(torch.bfloat16).view(torch.int16)
    u = torch.rand(B4, generator=gen, device=dev)
    qd = torch.empty((B4, K4), dtype=torch.float32, device=dev)
    tok = torch.empty(B4, dtype=torch.int32, device=dev)
    wsd = torch.empty(vt.lib().vt_draft_workspace_bytes(B4, H4, K4), dtype=torch.uint8,
                      device=dev)
    it = [0]

    def drf():
        it[0] += 1
        vt.vt_draft_step(hid, Wt[it[0] % 2], trim_ids, u, T4, q=qd, tokens=tok,
                         dev_status=st[1:2], workspace=wsd)
    us_d = graph_us(torch, drf, 12)
    bd = K4 * H4 * 2 + B4 * H4 * 2 + B4 * K4 * 4
    fl = 2.0 * B4 * K4 * H4
    res.update({"draft_us": us_d, "draft_algorithmic_bytes": bd,
                "draft_gbs": bd / (us_d * 1e-6) / 1e9, "draft_frac_hbm": bd / (us_d * 1e-6) / 1e9 / peak,
                "draft_tflops": fl / (us_d * 1e-6) / 1e12,
                "draft_frac_tensor": fl / (us_d * 1e-6) / 1e12 / peak_tf,
                "dev_status": [int(x) for x in st.cpu().tolist()]})
    del Wt, qd, wsd
    return res


def _pcts(xs):
    xs = np.asarray(xs, dtype=np.float64)
    return {"median_us": float(np.median(xs)), "p10_us": float(np.percentile(xs, 10)),
            "p90_us": float(np.percentile(xs, 90)), "n": int(xs.size)}


def run_timing_distribution(torch, vt, step, host, ncalls: int = 240):
    """Per-call time distributions of the two rows the metric and the
    roofline rest on, over >= 200 launches each.
    verify: `ncalls` calls on the batched-verify workload, logits rotating
      over three buffers (172 MB, more than L2), (a) one event pair around
      every call and (b) CUDA graphs of 20 calls replayed back to back (per
      call time of each replay);
    draft: the six drafting calls of a block as in the step, (a) with an
      event pair around each call, (b) graphs of 20 blocks replayed (per call)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(step.dev)
    q, draft, inv_map = t(host.q_verify), t(host.draft_verify), t(host.inv_map_verify)
    logits = [step.vsets[0]["logits"], step.vsets[1]["logits"], step.vsets[0]["logits"].clone()]
    s0 = step.vsets[0]
    Ev = lambda: torch.cuda.Event(enable_timing=True)

    def ver(k):
        vt.vt_verify(logits[k % 3], q, inv_map, draft, s0["u_acc"], s0["u_res"], T,
                     out_tokens=step.out_tokens, out_num_accepted=step.out_n,
                     out_accept_prob=step.out_acc, dev_status=step.status[3:4],
                     workspace=step.ws_ver)

    def drf(j):
        vt.vt_draft_step(step.hidden[j], step.W_trim, step.trim_ids, step.u_draft[j], T,
                         q=step.q[:, j, :], tokens=step.tokens[:, j],
                         dev_status=step.status[2:3], workspace=step.ws_draft)

    out = {}
    for name, fn, per in (("verify", ver, 1), ("draft", drf, GAMMA)):
        for k in range(6):
            fn(k % per if per > 1 else k)
        torch.cuda.synchronize()
        ev = [(Ev(), Ev()) for _ in range(ncalls)]
        for k in range(ncalls):
            ev[k][0].record()
            fn(k % per if per > 1 else k)
            ev[k][1].record()
        torch.cuda.synchronize()
        each = [a.elapsed_time(b) * 1e3 for a, b in ev]
        # graphs of 20 calls (verify) or 20 blocks of six calls (draft)
        gcalls = 20 * per
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for k in range(gcalls):
                    fn(k % per if per > 1 else k)
        torch.cuda.synchronize()
        reps = max(12, -(-ncalls // gcalls))
        per_call = []
        for r in range(reps + 2):
            a, b = Ev(), Ev()
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            if r >= 2:
                per_call.append(a.elapsed_time(b) * 1e3 / gcalls)
        del g
        alg = algorithmic_bytes()[name]
        pk, _ = peaks()
        e, gr = _pcts(each), _pcts(per_call)
        out[name] = {"event_pair_per_call": e, "graph_per_call": gr,
                     "graph_launches": reps * gcalls,
                     "frac_of_measured_hbm_at_graph_median":
                         alg / (gr["median_us"] * 1e-6) / 1e9 / pk}
    out["verify"]["positions_per_s_at_graph_median"] = \
        B * GAMMA / (out["verify"]["graph_per_call"]["median_us"] * 1e-6)
    out["note"] = ("event_pair_per_call: one pair of events around each call (the pair itself "
                   "costs the launch overlap between calls); graph_per_call: replays of a graph "
                   "of calls, time per call of each replay")
    return out


def toy_expectations(p_tab, q_tab, gamma: int):
    """Exact per-context expectations of the toy workload's blocks
    ("A rejection rule keeps speculative decoding's output exact", section
    "What draft accuracy buys"; "Speculative decoding" glossary, "Why a
    rejection needs a special draw").  A drafted x ~ q(.|c) is accepted with
    probability min(1, p(x|c)/q(x|c)), so a position with context c is
    accepted with probability beta(c) = sum_x min(p, q)(x|c), and the
    accepted token is x with probability min(p, q)(x|c) / beta(c); the next
    position's context is x + 1 (contexts: 0 = BOS, t + 1 after token t).
    Returns beta [C] and E[tokens per block | block starts at c] [C] (the
    accepted drafts plus the one drawn token)."""
    mn = np.minimum(np.asarray(p_tab, np.float64), np.asarray(q_tab, np.float64))
    beta = mn.sum(axis=1)
    acc = np.zeros(mn.shape[0])           # expected accepted drafts, 0 positions left
    for _ in range(gamma):
        acc = beta + mn @ acc[1:]         # the next context after token x is x + 1
    return beta, 1.0 + acc


def run_toy_chain(torch, vt, nblocks: int = 50_000, gamma: int = 4, seed: int = 31):
    """The toy workload (V = 18, 19 contexts, q_w = (p + q0)/2, gamma = 4) as
    a chain of blocks through vt_verify on the GPU, the drafts drawn on the
    host from q_w: tau (tokens per block) and the empirical acceptance rate
    alpha against their exact expectations over the visited contexts."""
    p_tab, _, q_tab = synthetic.toy_tables()
    Vt = p_tab.shape[1]
    beta, etok = toy_expectations(p_tab, q_tab, gamma)
    logp = torch.from_numpy(np.log(p_tab).astype(np.float32)).cuda()
    qd = torch.from_numpy(q_tab.astype(np.float32)).cuda()
    g = synthetic.rng(seed, 0)
    ua = torch.from_numpy(synthetic.uniforms(seed, 1, (nblocks, gamma))).cuda()
    ur = torch.from_numpy(synthetic.uniforms(seed, 2, (nblocks, gamma + 1))).cuda()
    inv_map = torch.arange(Vt, dtype=torch.int32, device="cuda")
    logits = torch.empty((1, gamma + 1, Vt), dtype=torch.float32, device="cuda")
    q = torch.empty((1, gamma, Vt), dtype=torch.float32, device="cuda")
    dr = torch.empty((1, gamma), dtype=torch.int32, device="cuda")
    ws = torch.empty(vt.workspace_bytes("verify", B=1, gamma=gamma, V=Vt, K=Vt),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((1, gamma + 1), dtype=torch.int32, device="cuda")
    n_t = torch.empty(1, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    ctx = 0
    status = 0
    ns = np.empty(nblocks, np.int64)
    e_tok = np.empty(nblocks)
    b_sum = b_var = 0.0
    tested = 0
    t0 = time.perf_counter()
    for k in range(nblocks):
        draft = synthetic.toy_drafts(g, q_tab, ctx, gamma)
        ctxs = [ctx] + [int(x) + 1 for x in draft]
        ci = torch.tensor(ctxs, device="cuda")
        logits[0].copy_(logp[ci])
        q[0].copy_(qd[ci[:gamma]])
        dr[0].copy_(torch.from_numpy(draft))
        vt.vt_verify(logits, q, inv_map, dr, ua[k:k + 1], ur[k:k + 1], 1.0, out_tokens=out,
                     out_num_accepted=n_t, dev_status=st, workspace=ws,
                     want_accept_prob=False)
        res = torch.cat([out[0], n_t, st]).cpu().numpy()
        n = int(res[gamma + 1])
        status |= int(res[gamma + 2])
        ns[k] = n
        e_tok[k] = etok[ctx]
        t = min(n + 1, gamma)                 # positions tested in this block
        bb = beta[np.array(ctxs[:t])]
        b_sum += float(bb.sum())
        b_var += float((bb * (1 - bb)).sum())
        tested += t
        ctx = int(res[n]) + 1                 # the block's last emitted token
    wall = time.perf_counter() - t0
    tau = float((ns + 1).mean())
    tau_exact = float(e_tok.mean())
    tau_sigma = float(np.std(ns + 1 - e_tok) / np.sqrt(nblocks))
    alpha = float(ns.sum() / tested)
    alpha_exact = b_sum / tested
    alpha_sigma = float(np.sqrt(b_var) / tested)
    return {"blocks": nblocks, "gamma": gamma, "dev_status": status,
            "tau": tau, "tau_exact": tau_exact, "tau_sigma": tau_sigma,
            "tau_within_4_sigma": abs(tau - tau_exact) <= 4 * tau_sigma,
            "alpha": alpha, "alpha_exact_mean_beta": alpha_exact, "alpha_sigma": alpha_sigma,
            "alpha_within_4_sigma": abs(alpha - alpha_exact) <= 4 * alpha_sigma,
            "tokens_per_block": tau, "wall_s": wall,
            "note": "drafts from the toy q_w on the host, one vt_verify call per block on "
                    "the GPU; exact values: per-context expectations of the rule averaged "
                    "over the visited contexts"}


def run_e2e_block(torch, step, host, stream, args, dist, dev, world):
    """The online block end to end through the public API: per block the host
    ships only what a decoder produces per block (the drafter's hidden states
    and uniforms, the target's logits, the verification uniforms, ~58 MB) and
    reads the verified tokens back; calibration and trim are offline
    (VocabTrim section 3) and done once before the timed region, like the
    trimmed head's weights.  Copies of block k+1 overlap block k."""
    vt = step.vt
    inp = host.step_inputs()
    names = ("hidden", "u_draft", "logits", "u_accept", "u_resample")
    pinned = {n: torch.from_numpy(np.ascontiguousarray(
        inp[n].view(np.int16) if inp[n].dtype == np.uint16 else inp[n])).pin_memory()
        for n in names}
    sets = [{n: torch.empty(pinned[n].shape, dtype=pinned[n].dtype, device=dev) for n in names}
            for _ in range(2)]
    out_host = torch.empty(B * (GAMMA + 1) + B, dtype=torch.int32).pin_memory()
    nblocks = max(1, min(args.steps, 50))
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(k):
        x = k % 2
        copy_stream.wait_event(done[x])
        with torch.cuda.stream(copy_stream):
            for n in names:
                sets[x][n].copy_(pinned[n], non_blocking=True)
            ready[x].record(copy_stream)

    def run_block(k):
        x = k % 2
        d = sets[x]
        stream.wait_event(ready[x])
        for j in range(GAMMA):
            vt.vt_draft_step(d["hidden"][j], step.W_trim, step.trim_ids, d["u_draft"][j], T,
                             q=step.q[:, j, :], tokens=step.tokens[:, j],
                             dev_status=step.status[2:3], workspace=step.ws_draft)
        vt.vt_verify(d["logits"], step.q, step.inv_map, step.tokens, d["u_accept"],
                     d["u_resample"], T, out_tokens=step.out_tokens,
                     out_num_accepted=step.out_n, out_accept_prob=step.out_acc,
                     dev_status=step.status[3:4], workspace=step.ws_ver)
        done[x].record(stream)
        out_host[: B * (GAMMA + 1)].copy_(step.out_tokens.view(-1), non_blocking=True)
        out_host[B * (GAMMA + 1):].copy_(step.out_n, non_blocking=True)

    def pipeline(n):
        copy_stream.wait_stream(stream)
        issue_copy(0)
        for k in range(n):
            if k + 1 < n:
                issue_copy(k + 1)
            run_block(k)

    pipeline(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipeline(nblocks)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(torch, e0.elapsed_time(e1), dist, dev)
    # the same blocks with the inputs already on the device (GPU-only time)
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for k in range(nblocks):
        run_block_dev = sets[k % 2]
        for j in range(GAMMA):
            vt.vt_draft_step(run_block_dev["hidden"][j], step.W_trim, step.trim_ids,
                             run_block_dev["u_draft"][j], T, q=step.q[:, j, :],
                             tokens=step.tokens[:, j], dev_status=step.status[2:3],
                             workspace=step.ws_draft)
        vt.vt_verify(run_block_dev["logits"], step.q, step.inv_map, step.tokens,
                     run_block_dev["u_accept"], run_block_dev["u_resample"], T,
                     out_tokens=step.out_tokens, out_num_accepted=step.out_n,
                     out_accept_prob=step.out_acc, dev_status=step.status[3:4],
                     workspace=step.ws_ver)
    e3.record(stream)
    torch.cuda.synchronize()
    ms_dev = max_over_ranks(torch, e2.elapsed_time(e3), dist, dev)
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    return {"value": whole_job_value(nblocks, world, ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_host.numel() * 4,
            "blocks": nblocks, "ms_per_block": ms / nblocks,
            "link_gbs": h2d / (ms / nblocks * 1e-3) / 1e9,
            "gpu_only": {"value": whole_job_value(nblocks, world, ms_dev), "unit": UNIT,
                         "ms_per_block": ms_dev / nblocks},
            "block": "6 drafting steps (B=16) and the verification; calibration and trim "
                     "offline, W_trim resident",
            "overlap": "copies of block k+1 on a second stream during block k"}


def run_e2e(torch, step, host, stream, args, dist, dev, world):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads the verified tokens back.
    The copies of step k + 1 run on a second stream into a second set of
    device buffers while step k computes (every copy and every read-back is
    inside the timed region; the CPU-GPU link, not the kernels, bounds it)."""
    inp = host.step_inputs()
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in inp.items()}
    # the model's weights are loaded once, before the timed region
    step.W.copy_(torch.from_numpy(np.ascontiguousarray(host.W.view(np.int16))).pin_memory(),
                 non_blocking=True)
    names = ("ids", "hidden", "u_draft")
    sets = [{n: getattr(step, n) for n in names},
            {n: torch.empty_like(getattr(step, n)) for n in names}]
    out_host = torch.empty(B * (GAMMA + 1) + B, dtype=torch.int32).pin_memory()
    nsteps = max(1, min(args.steps, 50))
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    assert step.nsets == 2  # the logits sets follow k % 2 as well

    def issue_copy(k):
        x = k % 2
        copy_stream.wait_event(done[x])  # step k - 2 no longer reads set x
        with torch.cuda.stream(copy_stream):
            for n, d in sets[x].items():
                src = pinned[n]
                d.copy_(src.view(d.dtype) if src.dtype != d.dtype else src, non_blocking=True)
            vs = step.vsets[x]
            vs["logits"].copy_(pinned["logits"], non_blocking=True)
            vs["u_acc"].copy_(pinned["u_accept"], non_blocking=True)
            vs["u_res"].copy_(pinned["u_resample"], non_blocking=True)
            ready[x].record(copy_stream)

    def run_step(k):
        x = k % 2
        stream.wait_event(ready[x])
        for n in names:
            setattr(step, n, sets[x][n])
        step.run(k)
        done[x].record(stream)
        out_host[: B * (GAMMA + 1)].copy_(step.out_tokens.view(-1), non_blocking=True)
        out_host[B * (GAMMA + 1):].copy_(step.out_n, non_blocking=True)

    def pipeline(n):
        copy_stream.wait_stream(stream)
        issue_copy(0)
        for k in range(n):
            if k + 1 < n:
                issue_copy(k + 1)
            run_step(k)

    pipeline(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipeline(nsteps)
    e1.record(stream)
    torch.cuda.synchronize()
    for n in names:
        setattr(step, n, sets[0][n])
    ms = max_over_ranks(torch, e0.elapsed_time(e1), dist, dev)
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    return {"value": whole_job_value(nsteps, world, ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_host.numel() * 4,
            "steps": nsteps, "ms_per_step": ms / nsteps,
            "link_gbs": h2d / (ms / nsteps * 1e-3) / 1e9,
            "overlap": "copies of step k+1 on a second stream during step k",
            "resident": "W, the drafter head's weights (model state), loaded once before "
                        "the timed region"}

if __name__ == "__main__":
    sys.exit(main())
