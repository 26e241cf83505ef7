"""Benchmark of the owner-local Muon optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]
    python bench.py --case soap|shampoo [--steps K] ...     (one second-order case, one line)

A step is one pass of the whole hot path over one batch of synthetic input resident in HBM:
W-way gradient deposit + Nesterov momentum + Frobenius norm, Newton–Schulz (5 quintic
iterations) of every owned matrix, the scaled update with decoupled weight decay, and AdamW on
the packed tail.  The default workload is the Llama-3-70B owner share (24 MLP matrices of
28672x8192 / 8192x28672 and 16 of 8192x8192, W = 2 bf16 contributions, about 131 GB resident),
the largest of the five workloads on one GPU; the GPT-2-small owner set (48 matrices of hidden
768, W = 8) is measured beside it under ``gpt2_small``.  The same contribution batch is reused
every step; momentum, weights and AdamW state evolve.  Inputs exceed the 129 MB L2, so no
flush is inserted.

Prints ONE JSON line (rank 0).  ``value`` is owner-step milliseconds (lower is better); the
Newton–Schulz TFLOP/s count 4 m^2 n + 2 m^3 FLOPs per iteration (m <= n).  ``--impl reference``
times the CPU float64 oracle on the machine's host cores instead, on a bounded per-step sample,
extrapolated to the whole owned set.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import get_config, synth  # noqa: E402

METRIC = "owner Muon step ms; Newton–Schulz TFLOP/s and % of GB300 bf16 dense peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# DRAM traffic of the Newton–Schulz kernels: dram__bytes_read.sum + dram__bytes_write.sum per
# launch, averaged over the launches of one step, from one ncu capture of the named workload.
# Each entry holds the SHA-256 of the sources that decide those launches (kernel, launch
# planner, shared definitions) at capture time; once they change, the figure no longer
# describes the kernel and the line reports null.  The capture commands and per-launch
# figures are in profiles/.
NS_TRAFFIC_SOURCES = ("matrix_optimizer_owner_gb300/csrc/ns_gemm.cu",
                      "matrix_optimizer_owner_gb300/csrc/api.cpp",
                      "matrix_optimizer_owner_gb300/csrc/mfsdp_internal.h")
NS_TRAFFIC = {
    # config index: (sources sha256, bytes per launch, profile summary)
    1: ("37d8b0068cdbb9c6d0c975d47beecdac27dc53780c59d966e0f94750898c9ef9", 207298184,
        "profiles/owner_step_gpt2_small_launch_list.md"),
    4: ("37d8b0068cdbb9c6d0c975d47beecdac27dc53780c59d966e0f94750898c9ef9", 71944308701,
        "profiles/owner_step_llama3_70b_launch_list.md"),
}


def ns_sources_sha():
    """SHA-256 of the kernel sources with comments and blank lines removed (a comment edit
    does not change the kernel)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in NS_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        lines = [ln.rstrip() for ln in src.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()


def ns_traffic_per_launch(cfg):
    if cfg is None or cfg not in NS_TRAFFIC:
        return None
    sha, nbytes, _ = NS_TRAFFIC[cfg]
    return nbytes if sha == ns_sources_sha() else None


# ----------------------------------------------------------------------------- workload
def shapes_workload(spec: str):
    """A custom owned set for profiling: "RxC,RxC,..." matrices, W = 8 bf16 contributions of
    std 1e-3, no tail, the step's usual hyperparameters."""
    from workloads.configs import ParamSpec, Workload as Wl
    params = []
    for i, tok in enumerate(spec.split(",")):
        r, c = (int(v) for v in tok.lower().split("x"))
        params.append(ParamSpec(f"m{i}", r, c, i, True))
    return Wl(9, f"custom owned set {spec}, W=8 bf16", tuple(params), world_size=1, rank=0, W=8,
              contrib_dtype="bf16", grad_std=1e-3)


class Workload:
    """Owned set of one rank, its buffers, and seeded inputs drawn on the device."""

    def __init__(self, cfg: int, owner_rank_shift: int, device, shapes=None):
        from matrix_optimizer_owner_gb300 import owner_step
        self.wl = wl = get_config(cfg) if not shapes else shapes_workload(shapes)
        self.rank = (wl.rank + owner_rank_shift) % wl.world_size
        params = [(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
        self.lay = lay = owner_step.owned_layout(params, wl.world_size, self.rank)
        self.shapes = [(wl.params[i].rows, wl.params[i].cols) for i in lay.matrices]
        self.runner = owner_step.OwnerStep(self.shapes, lay.matrix_offsets, lay.n_tail,
                                           device=device)
        self.dev = device
        r = self.runner
        dt = synth.torch_dtype(wl.contrib_dtype)
        for pi, off, (rr, cc) in zip(lay.matrices, lay.matrix_offsets, self.shapes):
            r.weights[off:off + rr * cc] = synth.weight(wl, pi, device)
        for pi, off in zip(lay.tails, lay.tail_offsets):
            n = wl.params[pi].numel
            r.tail_p[off:off + n] = synth.weight(wl, pi, device)
        self.contrib = []
        for w in range(wl.W):
            buf = torch.empty(r.n, dtype=dt, device=device)
            for pi, off, (rr, cc) in zip(lay.matrices, lay.matrix_offsets, self.shapes):
                buf[off:off + rr * cc] = synth.contribution(wl, 0, pi, w, device)
            self.contrib.append(buf)
        self.tail_contrib = []
        for w in range(wl.W if lay.n_tail else 0):
            buf = torch.empty(lay.n_tail, dtype=dt, device=device)
            for pi, off in zip(lay.tails, lay.tail_offsets):
                n = wl.params[pi].numel
                buf[off:off + n] = synth.contribution(wl, 0, pi, w, device)
            self.tail_contrib.append(buf)
        self.elem_bytes = 2 if dt == torch.bfloat16 else 4

    # algorithmic work per step ------------------------------------------------------------
    def ns_flops(self):
        s = self.wl.hyper.ns_steps
        nominal = executed = 0
        for rr, cc in self.shapes:
            m, n = min(rr, cc), max(rr, cc)
            nominal += s * (4 * m * m * n + 2 * m ** 3)
            executed += s * (m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n)
        return nominal, executed

    def stream_bytes(self):
        N = sum(r * c for r, c in self.shapes)
        W, e = self.wl.W, self.elem_bytes
        return {"reduce_momentum_norm": N * (W * e + 10), "apply_update": N * 10,
                "adamw_tail": self.lay.n_tail * (W * e + 24)}

    def ns_groups(self):
        """(split-precision matrices present, bf16 CTA-pair matrices present)."""
        n_split = self.runner.oset.split_count()
        return n_split > 0, n_split < len(self.shapes)

    def ns_launches_per_step(self):
        return 3 * self.wl.hyper.ns_steps * sum(self.ns_groups())

    def ns_kernel_name(self):
        split, pair = self.ns_groups()
        names = (["ns_gemm_pair_kernel"] if pair else []) + \
            (["ns_gemm_kernel<split>"] if split else [])
        return " + ".join(names) + " (every Newton–Schulz launch of a step)"

    def launches_per_step(self):
        r = self.runner
        n_split = r.oset.split_count()
        groups = (1 if n_split else 0) + (1 if n_split < len(self.shapes) else 0)
        unaligned = sum(1 for (rr, cc), o in zip(self.shapes, self.lay.matrix_offsets)
                        if o % 8 or cc % 8)
        return 2 + 3 * self.wl.hyper.ns_steps * groups + 2 * unaligned + 1 + \
            (1 if self.lay.n_tail else 0)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, flags in rows for k, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "reasons": reasons}


# ----------------------------------------------------------------------------- CPU oracle
# The fp64 oracle runs one owned matrix's whole Muon step when it costs at most this many
# nominal Newton–Schulz FLOPs (a few seconds on the host cores); above it a sample runs the
# step with one Newton–Schulz iteration in place of five (every iteration costs the same).
ORACLE_SAMPLE_MAX_FLOPS = 4e12


def _ns_nominal(rows, cols, steps):
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4 * m * m * n + 2 * m ** 3)


def oracle_muon_sample(wl, shapes, inputs_of, budget_s, max_mats=None):
    """Time the oracle's owner Muon step on a bounded sample of an owned set (host cores).

    shapes: the owned (rows, cols) in set order; inputs_of(k) -> (W0, contributions) of owned
    matrix k as fp64 arrays.  Matrices are taken smallest first (nominal Newton–Schulz FLOPs)
    until ``budget_s`` is spent or ``max_mats`` are done.  A matrix whose full step exceeds
    ORACLE_SAMPLE_MAX_FLOPS runs with one Newton–Schulz iteration (and only that one matrix).
    Returns (seconds, nominal NS FLOPs covered, description)."""
    from oracle import step as ostep
    hp = wl.hyper
    order = sorted(range(len(shapes)), key=lambda k: (_ns_nominal(*shapes[k], 1), k))
    spent = flops = 0.0
    taken, iters = 0, hp.ns_steps
    for k in order:
        if spent >= budget_s or (max_mats is not None and taken >= max_mats):
            break
        rr, cc = shapes[k]
        if taken == 0 and _ns_nominal(rr, cc, hp.ns_steps) > ORACLE_SAMPLE_MAX_FLOPS:
            iters = 1
        W0, cs = inputs_of(k)
        t0 = time.perf_counter()
        ostep.muon_matrix_step(W0, np.zeros_like(W0), cs, momentum=hp.momentum,
                               nesterov=hp.nesterov, grad_scale=hp.grad_scale,
                               ns_steps=iters, a=hp.ns_a, b=hp.ns_b, c=hp.ns_c,
                               eps=hp.ns_eps, lr=hp.lr, weight_decay=hp.weight_decay,
                               lr_adjust=hp.lr_adjust)
        spent += time.perf_counter() - t0
        flops += _ns_nominal(rr, cc, iters)
        taken += 1
        if iters != hp.ns_steps:
            break
    if iters != hp.ns_steps:
        r, c = shapes[order[0]]
        what = (f"one {r}x{c} owned matrix: deposit, momentum, norm, 1 of the "
                f"{hp.ns_steps} Newton–Schulz iterations, update")
    else:
        what = f"{taken} of {len(shapes)} owned matrices, one whole step each"
    return spent, flops, what


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def set_nominal_ns_flops(wl, shapes):
    return sum(_ns_nominal(r, c, wl.hyper.ns_steps) for r, c in shapes)


# ----------------------------------------------------------------------------- runs
def time_steps(wb, steps, warmup, stream, clock_window_s=0.0):
    """Warm up, keep stepping (untimed) for ``clock_window_s`` so the clock sampler, already
    running, sees the GPU under this load, then time exactly ``steps`` steps."""
    hp = wb.wl.hyper
    r = wb.runner
    for _ in range(warmup):
        r.step(wb.contrib, wb.tail_contrib, hp)
    torch.cuda.synchronize()
    t_end = time.perf_counter() + clock_window_s
    while time.perf_counter() < t_end:
        for _ in range(4):
            r.step(wb.contrib, wb.tail_contrib, hp)
        torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        e = ev[k]
        r.t += 1
        e[0].record(stream)
        r.reduce_momentum(wb.contrib, hp)
        e[1].record(stream)
        r.newton_schulz(hp)
        e[2].record(stream)
        r.apply_update(hp)
        e[3].record(stream)
        r.adamw_tail(wb.tail_contrib, hp, r.t)
        e[4].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    phases = {name: sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(steps))
              for i, name in enumerate(["reduce_momentum_norm", "newton_schulz", "apply_update",
                                        "adamw_tail"])}
    return total, phases


def time_graph(wb, steps, warmup):
    """The same step with deposit, Newton–Schulz and update replayed from one CUDA graph
    (AdamW tail launched after it); returns (ms per step over the timed region, the K
    per-step times)."""
    hp = wb.wl.hyper
    r = wb.runner
    g = r.capture(wb.contrib, hp)
    for _ in range(warmup):
        r.graph_step(g, wb.tail_contrib, hp)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for k in range(steps):
        r.graph_step(g, wb.tail_contrib, hp)
        ev[k + 1].record()
    torch.cuda.synchronize()
    per_step = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    return ev[0].elapsed_time(ev[steps]) / steps, per_step


def time_e2e(wb, steps, stream, n_copy_streams=2):
    """Same step through the C ABI with host buffers: every step copies its contributions
    host->device from pinned memory, runs, and reads the per-matrix update norms back.  The
    copies of step k+1 run on copy streams into a second set of device buffers while step k
    computes (each waits until the step that last used its buffers has finished)."""
    hp = wb.wl.hyper
    r = wb.runner
    host = []
    for c in wb.contrib + wb.tail_contrib:   # pinned host copies, written straight from HBM
        h = torch.empty(c.shape, dtype=c.dtype, pin_memory=True)
        h.copy_(c)
        host.append(h)
    n_c = len(wb.contrib)
    sets = [wb.contrib + wb.tail_contrib,
            [torch.empty_like(c) for c in wb.contrib + wb.tail_contrib]]
    norm_h = torch.empty(r.norm.numel(), dtype=torch.float32).pin_memory()
    copy_streams = [torch.cuda.Stream() for _ in range(n_copy_streams)]
    done = [torch.cuda.Event() for _ in range(2)]
    copied = [[torch.cuda.Event() for _ in copy_streams] for _ in range(2)]

    def issue_copies(b):
        for k, cs in enumerate(copy_streams):
            cs.wait_event(done[b])
            with torch.cuda.stream(cs):
                for d, h in list(zip(sets[b], host))[k::n_copy_streams]:
                    d.copy_(h, non_blocking=True)
            copied[b][k].record(cs)

    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    issue_copies(0)
    for i in range(steps):
        b = i & 1
        for ev in copied[b]:
            stream.wait_event(ev)
        if i + 1 < steps:
            issue_copies(b ^ 1)
        r.step(sets[b][:n_c], sets[b][n_c:], hp)
        done[b].record(stream)
        norm_h.copy_(r.norm, non_blocking=True)
    e.record(stream)
    torch.cuda.synchronize()
    h2d = sum(c.numel() * c.element_size() for c in host)
    return s.elapsed_time(e) / steps, h2d, norm_h.numel() * 4


def time_repack(wb, reps, stream, world=8):
    """Owner-segment repacking of the workload's whole parameter list (2-byte elements): pack
    the canonical buffer into the owner shards of a RoleGreedy plan over ``world`` ranks, all
    held on this GPU.  HBM traffic = read + write of every parameter byte."""
    from matrix_optimizer_owner_gb300 import mfsdp
    params = [(p.rows, p.cols, p.block, p.is_matrix) for p in wb.wl.params]
    segs, table, _ = mfsdp.mfsdp_plan_owner_set(params, world, mfsdp.POLICY_ROLE_GREEDY)
    sizes = [sum(row[r] for row in table) for r in range(world)]
    total = sum(sizes)
    canon = torch.empty(total, dtype=torch.bfloat16, device=stream.device)
    canon.view(torch.int16).random_()
    shards = [torch.empty(n, dtype=torch.bfloat16, device=stream.device) for n in sizes]
    ws = torch.empty(mfsdp.mfsdp_repack_workspace_bytes(len(params)), dtype=torch.uint8,
                     device=stream.device)
    plan = mfsdp.RepackPlan(params, segs, world)
    for _ in range(3):
        plan.pack(canon, shards, ws, stream)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        plan.pack(canon, shards, ws, stream)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / reps
    return ms, 2 * total * 2, len(params)


FFMA_PEAK_NOTE = "152 SMs x 128 fp32 lanes x 2 FLOP x the sampled SM clock"
TF32_PER_BF16 = 1.1 / 2.25   # nominal dense tensor rates of GB300, PFLOP/s


def _upper_tiles(d, tile=256):
    """Output tiles of a d x d symmetric product that reach the upper triangle."""
    nt = -(-d // tile)
    return nt * (nt + 1) // 2


def time_shampoo(device, reps=2, root_iters=30, precision=0):
    """Owner Shampoo step on one GPT-2-small layer's matrices (2304x768, 768x768, 3072x768,
    768x3072): statistics, 30 coupled-Newton steps for every inverse fourth root, the
    preconditioned update; precision 0 = fp32 products (3xTF32 tensor cores), 1 = the root
    iteration and P on the tensor cores with split-bf16 operands.  Returns (ms per step,
    nominal FLOPs per step, tensor-core FLOPs executed per step)."""
    from matrix_optimizer_owner_gb300 import mfsdp
    shapes = [(2304, 768), (768, 768), (3072, 768), (768, 3072)]
    offs, o = [], 0
    for r, c in shapes:
        offs.append(o)
        o += r * c
    sset = mfsdp.ShampooSet([(r, c, off) for (r, c), off in zip(shapes, offs)])
    ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=device)
    l = torch.empty(sset.l_numel, dtype=torch.float32, device=device)
    r_ = torch.empty(sset.r_numel, dtype=torch.float32, device=device)
    sset.init_state(1e-6, l, r_, ws)
    g = torch.randn(o, device=device) * 1e-3
    w = torch.randn(o, device=device) * 0.02
    sset.step(g, l, r_, w, 0.02, 0.01, root_iters, ws, precision=precision)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        sset.step(g, l, r_, w, 0.02, 0.01, root_iters, ws, precision=precision)
    e.record()
    torch.cuda.synchronize()
    flops = tensor = 0
    for r, c in shapes:
        flops += 2 * r * r * c + 2 * r * c * c          # statistics
        flops += root_iters * 4 * 2 * (r ** 3 + c ** 3)  # roots
        flops += 2 * r * r * c + 2 * r * c * c          # P
        # tensor path: a symmetric side product runs the 256x256 output tiles that reach the
        # upper triangle, the last iteration forms X only, three MMAs per split product
        sym = sum(_upper_tiles(d) * 256 * 256 * 2 * (64 * -(-d // 64)) for d in (r, c))
        tensor += 3 * ((4 * (root_iters - 1) + 1) * sym + 2 * r * r * c + 2 * r * c * c)
    sset.close()
    return s.elapsed_time(e) / reps, flops, tensor


def time_soap(device, warm=3, reps=2, max_sweeps=20):
    """Owner SOAP step on one GPT-2-small layer's matrices (2304x768, 768x768, 3072x768,
    768x3072), eigenbases exact every step: `warm` untimed steps (the first starts the Jacobi
    solves from Q = I, later ones from the previous basis), then `reps` timed steps on fresh
    gradients.  Returns (ms per step, sweeps per side of the last step, SGEMM FLOPs per step,
    Jacobi FLOPs of the last step counting every block of every rotating sweep)."""
    from matrix_optimizer_owner_gb300 import mfsdp
    shapes = [(2304, 768), (768, 768), (3072, 768), (768, 3072)]
    offs, o = [], 0
    for r, c in shapes:
        offs.append(o)
        o += r * c
    sset = mfsdp.SoapSet([(r, c, off) for (r, c), off in zip(shapes, offs)])
    ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=device)
    st = {k: torch.empty(n, dtype=torch.float32, device=device)
          for k, n in sset.state_sizes(o).items()}
    sset.init_state(st, ws)
    gen = torch.Generator(device=device)
    gen.manual_seed(11)
    w = torch.randn(o, generator=gen, device=device) * 0.02
    grads = [torch.randn(o, generator=gen, device=device) * 1e-3 for _ in range(warm + reps)]
    info = torch.zeros(2 * len(shapes), dtype=torch.int32, device=device)
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.95, beta_stats=0.95, eps=1e-8, weight_decay=1e-2,
                 max_sweeps=max_sweeps)
    for t in range(1, warm + 1):
        sset.step(grads[t - 1], w, st, t, workspace=ws, info=info, **hyper)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for t in range(warm + 1, warm + reps + 1):
        sset.step(grads[t - 1], w, st, t, workspace=ws, info=info, **hyper)
    e.record()
    torch.cuda.synchronize()
    sweeps = [int(x) for x in info.cpu().tolist()]
    # a step that keeps the eigenbases (SOAP refreshes them every f steps)
    s2 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event(enable_timing=True)
    s2.record()
    sset.step(grads[-1], w, st, warm + reps + 1, workspace=ws, refresh=False, **hyper)
    e2.record()
    torch.cuda.synchronize()
    keep_ms = s2.elapsed_time(e2)
    sides = [r for r, _ in shapes] + [c for _, c in shapes]
    gemm = 0
    for r, c in shapes:
        gemm += 2 * r * r * c + 2 * r * c * c            # statistics
        gemm += 2 * (2 * r ** 3 + 2 * c ** 3)            # Q^T L Q
        gemm += 2 * r ** 3 + 2 * c ** 3                  # Rayleigh quotients
        gemm += 2 * (2 * r ** 3 + 2 * c ** 3)            # polar step: Z^T Z, then T Z^T
        gemm += 2 * (2 * r * r * c + 2 * r * c * c)      # G', M' into the eigenbasis
        gemm += 2 * r * r * c + 2 * r * c * c            # N back out
    jac = 0
    for d, sw in zip(sides, sweeps):
        dp = (d + 63) // 64 * 64
        jac += 8 * dp ** 3 * max(abs(sw) - 1, 0)         # the last sweep only checks
    sset.close()
    return s.elapsed_time(e) / reps, sweeps, gemm, jac, keep_ms


def config_of(wl, cfg, rank, shapes, n_tail):
    """The workload block of the JSON line (the same for both arms)."""
    return {"workload": wl.name, "config_index": cfg, "owner_rank": rank,
            "matrices": len(shapes), "owned_elements": int(sum(r * c for r, c in shapes)),
            "tail_elements": int(n_tail), "W": wl.W, "contrib_dtype": wl.contrib_dtype,
            "ns_steps": wl.hyper.ns_steps, "l2": "inputs > 129 MB L2, no flush",
            "parallelism": "owner replicas, no collective"}


def config_block(wb, cfg):
    return config_of(wb.wl, cfg, wb.rank, wb.shapes, wb.lay.n_tail)


def measure_step(wb, cfg, args, stream, peaks, peak_src, world, dev, local_rank):
    """Owner-step time of one resident workload (call by call with per-phase events, then as a
    CUDA graph), with the clock record of both timed regions and the Newton–Schulz roofline."""
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        total_ms, phases = time_steps(wb, args.steps, max(args.warmup, 3), stream,
                                      args.clock_window_s)
        # the product's launch path: deposit, Newton–Schulz and update replayed from one
        # CUDA graph, the AdamW tail launched after it
        graph_ms, graph_steps = (None, None) if args.no_graph else \
            time_graph(wb, args.steps, max(args.warmup, 3))
    clocks = clk.summary()
    if clocks is not None:
        clocks["window"] = (f"{args.clock_window_s:.1f} s of untimed steps + the timed "
                            "regions (call by call, then graph replay)")
    eager_ms = total_ms / args.steps
    step_ms = graph_ms if graph_ms is not None else eager_ms
    if world > 1:
        t = torch.tensor([step_ms, eager_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        step_ms, eager_ms = float(t[0].item()), float(t[1].item())
    nominal, executed = wb.ns_flops()
    ns_ms = phases["newton_schulz"] / args.steps
    ns_tf_nominal = nominal / (ns_ms * 1e-3) / 1e12
    ns_tf_exec = executed / (ns_ms * 1e-3) / 1e12
    # burst peak for a timed region short enough to stay under the power cap, the sustained
    # (seconds-long, power-capped) one otherwise
    sustained = total_ms > 1000.0 and "bf16_tflops_sustained" in peaks
    peak_tf = float(peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    ns_launches = wb.ns_launches_per_step()
    sb = wb.stream_bytes()
    gbs = {k: (sb[k] / (phases[k] / args.steps * 1e-3) / 1e9 if phases[k] > 0 else None)
           for k in sb}
    hbm = float(peaks["hbm_gbs"])
    return {
        "ms_per_step": step_ms, "eager_ms_per_step": round(eager_ms, 4),
        "launch": ("CUDA graph (deposit, Newton–Schulz, update) + AdamW tail"
                   if graph_ms is not None else "call by call"),
        "step_ms_median": round(statistics.median(graph_steps), 4) if graph_steps else None,
        "step_ms_max": round(max(graph_steps), 4) if graph_steps else None,
        "ns_ms_per_step": round(ns_ms, 4),
        "ns_tflops": round(ns_tf_nominal, 1), "ns_tflops_executed": round(ns_tf_exec, 1),
        "ns_frac_of_peak": round(ns_tf_exec / peak_tf, 4),
        "phases_ms_per_step": {k: round(v / args.steps, 4) for k, v in phases.items()},
        "streaming_gbs": {k: (round(v, 1) if v else None) for k, v in gbs.items()},
        "streaming_frac_of_hbm": {k: (round(v / hbm, 4) if v else None) for k, v in gbs.items()},
        "roofline": {"kernel": wb.ns_kernel_name(), "bound": "tensor",
                     "achieved": round(ns_tf_exec, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(ns_tf_exec / peak_tf, 4),
                     "traffic": ns_traffic_per_launch(cfg),
                     "peak_source": f"{peak_src} bf16 {'sustained' if sustained else 'burst'}",
                     "launches_per_step": ns_launches,
                     "avg_launch_us": round(1e3 * ns_ms / ns_launches, 2),
                     "flops_per_launch": round(executed / ns_launches),
                     "flops_counted": "executed: upper 256-tiles of the symmetric Gram and "
                                      "polynomial products, m(m+1)n + m^2(m+1) + 2m^2n per "
                                      "iteration"},
        "gpu_launches": wb.launches_per_step() * args.steps,
        "clocks": clocks,
    }


def cpu_baseline_of(wb, budget_s):
    """The oracle on the host cores, on a bounded sample of the resident workload's own
    (device-drawn) inputs, extrapolated to the whole owned set by nominal Newton–Schulz FLOP
    share."""
    r, lay = wb.runner, wb.lay

    def inputs_of(k):
        rr, cc = wb.shapes[k]
        off = lay.matrix_offsets[k]
        W0 = r.weights[off:off + rr * cc].double().cpu().numpy().reshape(rr, cc)
        cs = [c[off:off + rr * cc].double().cpu().numpy().reshape(rr, cc) for c in wb.contrib]
        return W0, cs

    spent, flops, what = oracle_muon_sample(wb.wl, wb.shapes, inputs_of, budget_s)
    total = set_nominal_ns_flops(wb.wl, wb.shapes)
    return {"value": round(1e3 * spent * total / flops, 1), "unit": "ms",
            "cores": blas_threads(), "kind": "oracle",
            "sample": f"{what} ({spent:.1f} s), extrapolated to the whole owned set by "
                      "nominal Newton–Schulz FLOP share",
            "timed_s": round(spent, 2), "extrapolated": flops < total,
            "sampled_flop_fraction": round(flops / total, 6)}


def free_workload(wb):
    wb.runner.close()
    wb.contrib.clear()
    wb.tail_contrib.clear()
    del wb.runner
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def run_ours(args, rank, world, local_rank):
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wb = Workload(args.config, rank, dev, args.shapes)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    m = measure_step(wb, None if args.shapes else args.config, args, stream, peaks, peak_src,
                     world, dev, local_rank)
    status = mfsdp.mfsdp_query_status()
    ms = m.pop("ms_per_step")
    clocks = m.pop("clocks")
    launches = m.pop("gpu_launches")
    roofline = m.pop("roofline")

    e2e_steps = max(3, args.steps)  # the same K as the device timing
    e2e_ms, h2d, d2h = time_e2e(wb, e2e_steps, stream) if not args.no_e2e else (None, 0, 0)
    if world > 1 and e2e_ms is not None:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())

    line = {
        "metric": METRIC, "value": round(ms, 4), "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, device-drawn)",
        "config": config_block(wb, args.config if not args.shapes else None),
        **m,
        "roofline": roofline,
        "e2e": {"value": round(e2e_ms, 4) if e2e_ms is not None else None, "unit": "ms",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "steps": e2e_steps if e2e_ms is not None else 0},
        "gpu_launches": launches,
        "clocks": clocks, "device_status": status,
    }
    if not args.no_repack:
        rms, rbytes, nparams = time_repack(wb, 10, stream)
        line["repack"] = {
            "kernel": "segment_copy_kernel", "what": f"pack {nparams} parameters (2-byte "
            f"elements) of the {wb.wl.name.split(':')[0]} list from the canonical axis into "
            "8-rank RoleGreedy owner shards",
            "ms": round(rms, 4), "bytes": rbytes, "bound": "hbm",
            "achieved_gbs": round(rbytes / (rms * 1e-3) / 1e9, 1), "peak_gbs": peaks["hbm_gbs"],
            "frac": round(rbytes / (rms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 4)}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_of(wb, args.cpu_seconds)
    free_workload(wb)
    del wb

    # The GPT-2-small owner set (48 matrices of hidden 768): the small-matrix regime of the
    # same step, reported beside the headline workload.
    if not args.shapes and args.config != 1 and not args.no_gpt2_small:
        wb1 = Workload(1, rank, dev)
        m1 = measure_step(wb1, 1, args, stream, peaks, peak_src, world, dev, local_rank)
        m1["ms_per_step"] = round(m1["ms_per_step"], 4)
        line["gpt2_small"] = {"config": config_block(wb1, 1), **m1,
                              "device_status": mfsdp.mfsdp_query_status()}
        if rank == 0 and not args.no_cpu_baseline:
            line["gpt2_small"]["cpu_baseline"] = cpu_baseline_of(wb1, args.cpu_seconds)
        free_workload(wb1)
        del wb1

    if not args.no_shampoo and rank == 0:
        what = ("one owner Shampoo step of one GPT-2-small layer (2304x768, 768x768, "
                "3072x768, 768x3072), 30 coupled-Newton steps per inverse fourth root")
        sms_, sflops, _ = time_shampoo(dev)
        tf32_peak = float(peaks["bf16_tflops"]) * TF32_PER_BF16
        line["shampoo"] = {
            "kernel": "tf32x3_gemm_kernel (tcgen05 kind::tf32, three split products per "
                      "multiply) + root and update kernels",
            "what": what, "precision": "fp32 (3xTF32)",
            "ms": round(sms_, 3), "flops": sflops, "bound": "tensor",
            "tensor_flops_executed": 3 * sflops,
            "achieved_tflops": round(3 * sflops / (sms_ * 1e-3) / 1e12, 1),
            "peak_tflops": round(tf32_peak, 1),
            "peak_source": f"{peak_src} bf16 burst x {TF32_PER_BF16:.4f} (nominal dense TF32 / "
                           "bf16 rate, 1.1 / 2.25 PFLOP/s)",
            "frac": round(3 * sflops / (sms_ * 1e-3) / 1e12 / tf32_peak, 4),
            "frac_note": "three TF32 products per fp32 multiply over the whole step time "
                         "(norms and elementwise kernels included)"}
        tms, tflops, texec = time_shampoo(dev, precision=1)
        line["shampoo_tc"] = {
            "kernel": "ns_gemm_pair_kernel<split> (tcgen05 CTA pairs, split-bf16) for the "
                      "roots and P; tf32x3_gemm_kernel (tcgen05 3xTF32) for the statistics",
            "what": what, "precision": "split_bf16",
            "ms": round(tms, 3), "flops": tflops, "bound": "tensor",
            "tensor_flops_executed": texec,
            "achieved_tflops": round(texec / (tms * 1e-3) / 1e12, 1),
            "peak_tflops": float(peaks["bf16_tflops"]),
            "peak_source": f"{peak_src} bf16 burst",
            "frac": round(texec / (tms * 1e-3) / 1e12 / float(peaks["bf16_tflops"]), 4),
            "frac_note": "executed tensor FLOPs over the whole step time (statistics, norms "
                         "and elementwise kernels included)"}
    if not args.no_soap and rank == 0:
        sms_, sweeps, gemm, jac, keep_ms = time_soap(dev)
        sm_mhz = (clocks or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
        ffma_peak = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12
        ach = (gemm + jac) / (sms_ * 1e-3) / 1e12
        line["soap"] = {
            "kernel": "jacobi_solve_kernel + jacobi_apply_kernel (block Jacobi subproblems and "
                      "A's rotations, fp32 CUDA cores) + jacobi_zrot_tc_kernel (Z^T's "
                      "rotations) + tf32x3_gemm_kernel (statistics, Q^T L Q, polar step, "
                      "Rayleigh quotients, rotations into and out of the eigenbasis) (tcgen05 "
                      "3xTF32)",
            "what": "one owner SOAP step of one GPT-2-small layer (2304x768, 768x768, 3072x768, "
                    "768x3072), exact eigenbases every step, warm-started",
            "ms": round(sms_, 3), "sweeps_per_side": sweeps, "bound": "alu",
            "ms_without_refresh": round(keep_ms, 3),
            "ms_amortised_refresh_every_10": round((sms_ + 9 * keep_ms) / 10, 3),
            "flops": gemm + jac, "achieved_tflops": round(ach, 2),
            "peak_tflops": round(ffma_peak, 1), "peak_source": FFMA_PEAK_NOTE,
            "frac": round(ach / ffma_peak, 4),
            "flops_counted": "SGEMMs + 8 dp^3 per side per rotating sweep (every 64x64 block "
                             "product of the rotations): an upper bound, since pairs whose "
                             "rotation is the identity skip their blocks; half of the "
                             "rotation FLOPs (Z^T's) run on the tensor cores, so the fraction "
                             "of the FFMA peak is a mixed figure"}
    return line


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: ownership from the oracle's planner, the workload's
    seeded inputs drawn on the host (torch's CPU generator: the same distributions as the
    device draws, other values), and each step times the oracle's Muon step on a bounded
    sample of the owned set (the same sample rule as our arm's cpu_baseline), extrapolated to
    the whole owned set by nominal Newton–Schulz FLOP share, plus the whole AdamW tail.  No
    library code and no GPU work on this path."""
    if rank != 0:
        return None
    from oracle import adamw as oadamw
    from oracle import plan as oplan
    wl = get_config(args.config)
    hp = wl.hyper
    ps = [oplan.Param(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
    mats, tails = oplan.owned(ps, oplan.plan(ps, wl.world_size), wl.rank)
    shapes = [(ps[i].rows, ps[i].cols) for i in mats]
    total_flops = set_nominal_ns_flops(wl, shapes)
    cache = {}

    def inputs_of(k):          # drawn once (outside the timed region), reused every step
        if k not in cache:
            i = mats[k]
            r, c = shapes[k]
            cache[k] = (synth.weight(wl, i).double().numpy().reshape(r, c),
                        [synth.contribution(wl, 0, i, w).double().numpy().reshape(r, c)
                         for w in range(wl.W)])
        return cache[k]

    tail_in = None
    if tails:
        p0 = np.concatenate([synth.weight(wl, i).double().numpy() for i in tails])
        g = sum(np.concatenate([synth.contribution(wl, 0, i, w).double().numpy()
                                for i in tails]) for w in range(wl.W)) * hp.grad_scale
        tail_in = (p0, g)
    per_step, timed, what, frac = [], 0.0, "", 1.0
    for k in range(max(args.warmup, 0) + args.steps):
        spent, flops, what = oracle_muon_sample(wl, shapes, inputs_of, args.ref_seconds,
                                                max_mats=args.ref_mats)
        frac = flops / total_flops if total_flops else 1.0
        step_s = spent / frac if flops else 0.0
        if tail_in is not None:  # the AdamW tail, whole
            b1, b2 = hp.adam_betas
            t0 = time.perf_counter()
            oadamw.adamw_step(tail_in[0], np.zeros_like(tail_in[0]), np.zeros_like(tail_in[0]),
                              tail_in[1], 1, hp.adam_lr, b1, b2, hp.adam_eps, hp.adam_wd)
            dt = time.perf_counter() - t0
            step_s += dt
            spent += dt
        if k >= args.warmup:
            per_step.append(1e3 * step_s)
            timed += spent
    v = statistics.mean(per_step)
    n_tail = sum(ps[i].numel for i in tails)
    return {
        "metric": METRIC, "value": round(v, 1), "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v, 1),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, host-drawn)",
        "config": config_of(wl, args.config, wl.rank, shapes, n_tail), "impl": "reference",
        "cpu_baseline": {"value": round(v, 1), "unit": "ms", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"each step: {what}, extrapolated to the whole owned set by "
                                   "nominal Newton–Schulz FLOP share"
                                   + (", plus the whole AdamW tail" if tails else ""),
                         "timed_s": round(timed, 2), "extrapolated": frac < 1.0,
                         "sampled_flop_fraction": round(frac, 6)},
        "e2e": {"value": round(v, 1), "unit": "ms", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- cases
GPT2_LAYER = [(2304, 768), (768, 768), (3072, 768), (768, 3072)]


def run_case(args):
    """One second-order case for timing and profiling: ``args.steps`` owner steps of one
    GPT-2-small layer's matrices on cuda:0 from seeded synthetic gradients; prints the time of
    the last step and, for SOAP, the Jacobi sweeps each side took."""
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    offs, numel = [], 0
    for r, c in GPT2_LAYER:
        offs.append(numel)
        numel += r * c
    mats = [(r, c, off) for (r, c), off in zip(GPT2_LAYER, offs)]
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    w = torch.randn(numel, generator=gen, device=dev) * 0.02
    if args.case == "soap":
        sset = mfsdp.SoapSet(mats)
        ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=dev)
        st = {k: torch.empty(n, dtype=torch.float32, device=dev)
              for k, n in sset.state_sizes(numel).items()}
        sset.init_state(st, ws)
        info = torch.zeros(2 * len(GPT2_LAYER), dtype=torch.int32, device=dev)
    else:
        sset = mfsdp.ShampooSet(mats)
        ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=dev)
        lst = torch.empty(sset.l_numel, dtype=torch.float32, device=dev)
        rst = torch.empty(sset.r_numel, dtype=torch.float32, device=dev)
        sset.init_state(1e-6, lst, rst, ws)
    ms = 0.0
    for t in range(1, args.steps + 1):
        g = torch.randn(numel, generator=gen, device=dev) * 1e-3
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        if args.case == "soap":
            sset.step(g, w, st, t, lr=1e-3, beta1=0.9, beta2=0.95, beta_stats=0.95, eps=1e-8,
                      weight_decay=1e-2, max_sweeps=args.max_sweeps, workspace=ws, info=info)
        else:
            sset.step(g, lst, rst, w, 0.02, 0.01, args.root_iters, ws, precision=args.precision)
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e)
    extra = f" sweeps={info.cpu().tolist()}" if args.case == "soap" else \
        f" precision={args.precision}"
    print(f"{args.case} steps={args.steps} last_ms={ms:.2f}{extra} "
          f"status={mfsdp.mfsdp_query_status()}", flush=True)
    sset.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--shapes", default=None,
                    help='custom owned set for profiling, e.g. "4096x14336,1024x4096"')
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=5.0,
                    help="reference arm: oracle seconds per step (at least one sample unit)")
    ap.add_argument("--ref-mats", type=int, default=None,
                    help="reference arm: owned matrices per step (default: as many as the "
                         "--cpu-seconds budget allows)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-repack", action="store_true",
                    help="skip the owner-shard repacking measurement")
    ap.add_argument("--no-soap", action="store_true",
                    help="skip the owner SOAP measurement (one GPT-2-small layer)")
    ap.add_argument("--no-shampoo", action="store_true",
                    help="skip the owner Shampoo measurement")
    ap.add_argument("--no-gpt2-small", action="store_true",
                    help="skip the GPT-2-small owner set measured beside another workload")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step call by call only (no CUDA-graph replay)")
    ap.add_argument("--clock-window-s", type=float, default=1.0)
    ap.add_argument("--case", choices=["soap", "shampoo"], default=None,
                    help="run one second-order case of a GPT-2-small layer and print one line")
    ap.add_argument("--max-sweeps", type=int, default=20, help="--case soap: Jacobi sweep limit")
    ap.add_argument("--precision", type=int, default=0,
                    help="--case shampoo: 0 fp32, 1 split-bf16 tensor cores")
    ap.add_argument("--root-iters", type=int, default=30, help="--case shampoo: Newton steps")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl")
    try:
        line = run_ours(args, rank, world, local_rank)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
