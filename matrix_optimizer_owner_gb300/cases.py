"""Runnable cases of the second-order owner optimizers, for timing and profiling.

    python -m matrix_optimizer_owner_gb300.cases soap --steps 2 --max-sweeps 4
    python -m matrix_optimizer_owner_gb300.cases shampoo --steps 1 --precision 1

Each case runs owner steps of one GPT-2-small layer's matrices (2304x768, 768x768, 3072x768,
768x3072) on cuda:0 from seeded synthetic gradients and prints one line with the time of the
last step and, for SOAP, the Jacobi sweeps each side took.
"""

from __future__ import annotations

import argparse

import torch

from . import mfsdp

GPT2_LAYER = [(2304, 768), (768, 768), (3072, 768), (768, 3072)]


def _layout(shapes):
    offs, o = [], 0
    for r, c in shapes:
        offs.append(o)
        o += r * c
    return offs, o


def run_soap(steps: int, max_sweeps: int) -> None:
    dev = torch.device("cuda", 0)
    offs, numel = _layout(GPT2_LAYER)
    sset = mfsdp.SoapSet([(r, c, off) for (r, c), off in zip(GPT2_LAYER, offs)])
    ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=dev)
    st = {k: torch.empty(n, dtype=torch.float32, device=dev)
          for k, n in sset.state_sizes(numel).items()}
    sset.init_state(st, ws)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    w = torch.randn(numel, generator=gen, device=dev) * 0.02
    info = torch.zeros(2 * len(GPT2_LAYER), dtype=torch.int32, device=dev)
    ms = 0.0
    for t in range(1, steps + 1):
        g = torch.randn(numel, generator=gen, device=dev) * 1e-3
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        sset.step(g, w, st, t, lr=1e-3, beta1=0.9, beta2=0.95, beta_stats=0.95, eps=1e-8,
                  weight_decay=1e-2, max_sweeps=max_sweeps, workspace=ws, info=info)
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e)
    print(f"soap steps={steps} last_ms={ms:.2f} sweeps={info.cpu().tolist()} "
          f"status={mfsdp.mfsdp_query_status()}")
    sset.close()


def run_shampoo(steps: int, precision: int, root_iters: int) -> None:
    dev = torch.device("cuda", 0)
    offs, numel = _layout(GPT2_LAYER)
    sset = mfsdp.ShampooSet([(r, c, off) for (r, c), off in zip(GPT2_LAYER, offs)])
    ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=dev)
    l = torch.empty(sset.l_numel, dtype=torch.float32, device=dev)
    r = torch.empty(sset.r_numel, dtype=torch.float32, device=dev)
    sset.init_state(1e-6, l, r, ws)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    w = torch.randn(numel, generator=gen, device=dev) * 0.02
    ms = 0.0
    for _ in range(steps):
        g = torch.randn(numel, generator=gen, device=dev) * 1e-3
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        sset.step(g, l, r, w, 0.02, 0.01, root_iters, ws, precision=precision)
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e)
    print(f"shampoo steps={steps} precision={precision} last_ms={ms:.2f} "
          f"status={mfsdp.mfsdp_query_status()}")
    sset.close()


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("case", choices=["soap", "shampoo"])
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--max-sweeps", type=int, default=20)
    ap.add_argument("--precision", type=int, default=0)
    ap.add_argument("--root-iters", type=int, default=30)
    a = ap.parse_args()
    torch.cuda.set_device(0)
    if a.case == "soap":
        run_soap(a.steps, a.max_sweeps)
    else:
        run_shampoo(a.steps, a.precision, a.root_iters)


if __name__ == "__main__":
    main()
