"""Seeded synthetic inputs for the tiled-attention path.

This module holds shapes, seeds and value distributions only: none of the
attention arithmetic.  Both sides of every comparison (the CUDA path and the
float64 CPU oracle under ``oracle/``) draw their inputs from here, so the two
share nothing else.

Recipe (the same for every workload):

* a CPU ``torch.Generator`` seeded with the workload's seed;
* ``torch.randn`` in float32, drawn in the order Q, K, V, dO, each of shape
  ``[B, H, N, D]`` (contiguous), multiplied by the workload's ``std``;
* cast to the run dtype (float32 or bfloat16, round-to-nearest-even).

The oracle reads the *cast* tensors upcast exactly to float64, so both sides
see bit-identical input values.

The workloads are the shapes the attention pages benchmark or discuss: the
(B,H,S,D) = (2,4,2048,128) Apple-M1 benchmark of "Learning Metal with
FlashAttention" ("Benchmark" section) is shape-compatible with
``fwd_bf16_b4h16n2048d128`` (same N and D); the 32K-context case of the
metalworking "Flash Attention" page is ``fwdbwd_bf16_b1h32n32768d64_causal``;
the large-head-dimension (D=256) register-pressure case of the
metal-flash-attention page is ``fwd_bf16_b1h8n8192d256`` (forward) and
``fwdbwd_bf16_b1h8n8192d256`` (forward and backward).  No public dataset
is involved: attention inputs are i.i.d. Gaussian.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str                  # "f32" or "bf16"
    causal: Tuple[bool, ...]    # causal modes the workload is run in
    passes: Tuple[str, ...]     # "fwd", "bwd"
    seed: int
    std: float = 1.0
    grad_dtypes: Tuple[str, ...] = ()

    @property
    def scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("fwd_f32_b1h1n256d64", 1, 1, 256, 64, "f32", (False,), ("fwd",), 1001),
        Workload("fwd_bf16_b4h16n2048d128", 4, 16, 2048, 128, "bf16", (False, True), ("fwd",), 1002),
        Workload("fwd_bf16_b1h8n8192d256", 1, 8, 8192, 256, "bf16", (False,), ("fwd",), 1003, std=0.5),
        Workload("bwd_bf16_b2h16n4096d128_causal", 2, 16, 4096, 128, "bf16", (True,), ("fwd", "bwd"), 1004,
                 grad_dtypes=("f32", "bf16")),
        Workload("fwdbwd_bf16_b1h32n32768d64_causal", 1, 32, 32768, 64, "bf16", (True,), ("fwd", "bwd"), 1005,
                 grad_dtypes=("bf16",)),
        # the D = 256 shape above with a backward as well (the wide-head backward kernels)
        Workload("fwdbwd_bf16_b1h8n8192d256", 1, 8, 8192, 256, "bf16", (False,), ("fwd", "bwd"), 1006, std=0.5,
                 grad_dtypes=("bf16",)),
    )
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_qkv(B: int, H: int, N: int, D: int, seed: int, dtype: str = "bf16", std: float = 1.0,
             with_dO: bool = False) -> Dict[str, torch.Tensor]:
    """Draw Q, K, V (and dO) on the CPU in the run dtype, per the recipe above."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    names = ("q", "k", "v", "dO") if with_dO else ("q", "k", "v")
    out = {}
    for n in names:
        t = torch.randn((B, H, N, D), generator=g, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        out[n] = t.to(TORCH_DTYPE[dtype]).contiguous()
    return out


def workload_inputs(w: Workload, with_dO: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    if with_dO is None:
        with_dO = "bwd" in w.passes
    return make_qkv(w.B, w.H, w.N, w.D, w.seed, w.dtype, w.std, with_dO)


def sample_rows(B: int, H: int, N: int, count: int, seed: int, include_edges: bool = True):
    """Seeded (b, h, i) triples to check at sizes the oracle cannot finish in full.

    Edges (row 0, row N-1, the rows around the first tile boundary) are always
    included so that causal row 0, the ragged tail and the diagonal tile are
    covered.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 77)
    rows = set()
    if include_edges:
        for b in {0, B - 1}:
            for h in {0, H - 1}:
                for i in {0, 1, min(127, N - 1), min(128, N - 1), N - 1}:
                    rows.add((b, h, i))
    while len(rows) < count:
        b = int(torch.randint(0, B, (1,), generator=g))
        h = int(torch.randint(0, H, (1,), generator=g))
        i = int(torch.randint(0, N, (1,), generator=g))
        rows.add((b, h, i))
    return sorted(rows)
