"""Run one attention shape through the public API a few times, for profilers.

    python -m attention_tiled_fwd_gb300.run_case B H N D [--causal] [--backward]
        [--reps R] [--dtype bf16|f32] [--std S]

Each repetition runs fa_forward and, with --backward, fa_backward_dq and
fa_backward_dkdv, on seeded synthetic inputs (seed 4242, the benchmark's
generator).  A profiler pointed at one kernel with a launch skip of 1 sees the
second, warm launch.  Exits non-zero if the device status word reports a
failed wait.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("B", type=int)
    ap.add_argument("H", type=int)
    ap.add_argument("N", type=int)
    ap.add_argument("D", type=int)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--backward", action="store_true")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--dtype", choices=("bf16", "f32"), default="bf16")
    ap.add_argument("--std", type=float, default=1.0)
    a = ap.parse_args(argv)

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import attention_tiled_fwd_gb300 as fa
    from synthetic_inputs import make_qkv

    dev = torch.device("cuda:0")
    h = make_qkv(a.B, a.H, a.N, a.D, 4242, a.dtype, a.std, with_dO=a.backward)
    q, k, v = (h[n].to(dev) for n in ("q", "k", "v"))
    dO = h["dO"].to(dev) if a.backward else None
    for _ in range(a.reps):
        o, lse = fa.fa_forward(q, k, v, causal=a.causal)
        if a.backward:
            dq, delta = fa.fa_backward_dq(q, k, v, o, dO, lse, causal=a.causal, grad_dtype=torch.bfloat16)
            fa.fa_backward_dkdv(q, k, v, dO, lse, delta, causal=a.causal, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    st = fa.fa_device_status()
    if st != 0:
        print(f"device status {st}", file=sys.stderr)
        return 1
    print("ok", a.B, a.H, a.N, a.D, "causal" if a.causal else "non-causal",
          "fwd+bwd" if a.backward else "fwd", a.dtype)
    return 0


if __name__ == "__main__":
    sys.exit(main())
