"""CPU oracle for the step between the gate/up and down projections of a
decoder layer — test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA library.

What it computes (plain fp64 definitions, no blocking):

  silu(z)         = z / (1 + exp(-z))
  silu_mul(g, u)  = silu(g) * u, element by element

The pages never name the activation between the projections.  The gate/up/down
shapes of the Qwen2.5-7B decoder linears that the measurements use are its
gated MLP, whose hidden state is h = SiLU(gate(x)) * up(x), fed to down(h);
that is the reading taken here.  Fusing this elementwise step into the matmul
that produces g and u follows "Why LLM Decoding Is Slow, and Why Batching Is
(Almost) Free" (§3 "The Real Constraint: Two Ceilings": the measured step time
sits above the weight-streaming estimate, and the author's suspect is the
overhead of layernorm, attention and many small ops around the matmuls).

silu_mul_bound(g, u, bg, bu) is the per-element tolerance of an h computed in
fp32 from a gate output within bg of g and an up output within bu of u (the
matmul bound of each): silu is 1.1-Lipschitz (its derivative lies in
[-0.0998, 1.0998]), so

  |h' - h| <= 1.1 bg (|u| + bu) + |silu(g)| bu + rounding,

with the fp32 evaluation of silu and the product allowed 16 units in the last
place (2^-20 of the magnitude) on top.
"""
from __future__ import annotations

import numpy as np

SILU_LIPSCHITZ = 1.1
ROUNDING = 2.0 ** -20


def silu(z):
    """z / (1 + exp(-z)) in fp64."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def silu_mul(g, u):
    """h = silu(g) * u in fp64 (g, u: the gate and up projections' outputs)."""
    return silu(g) * np.asarray(u, dtype=np.float64)


def silu_mul_bound(g, u, bg, bu):
    """Tolerance of an fp32 h computed from outputs within bg of g and bu of u."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    bg = np.asarray(bg, dtype=np.float64)
    bu = np.asarray(bu, dtype=np.float64)
    s = np.abs(silu(g))
    prop = SILU_LIPSCHITZ * bg * (np.abs(u) + bu) + s * bu
    return prop + ROUNDING * (s * np.abs(u) + prop) + 1e-30
