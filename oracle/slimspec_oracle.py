"""CPU oracle of the SlimSpec low-rank draft LM head.

TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
benchmark's CPU-baseline leg are the only code that may import or run this
module. It shares no code with the CUDA library and imports nothing from it;
the product path never calls it.

Pages cited, by title:

  [SlimSpec]   "SlimSpec: Low-Rank Draft LM-Head for Accelerated Speculative
               Decoding" (gist.science, paper 2605.10453); section
               "방법론: SlimSpec", "아키텍처": the draft's full-rank head
               z = W_full h (W_full of V x d) is replaced by the factored
               z = W_up (W_down h), W_down of r x d compressing the hidden state,
               W_up of V x r projecting it back to the whole vocabulary, r a
               hyperparameter such as d/8, which cuts the head's work from
               O(Vd) to O(rd + Vr).
  [SD-anatomy] "LLM 투기적 디코딩(Speculative Decoding) 해부 ..." (blog.huny.dev),
               §3: the draft proposes from its full-vocabulary distribution
               q = softmax(z).

Readings taken where the pages are silent (each is also listed in the design
notes):
  * h, W_down and W_up arrive as bf16 values; everything here is exact fp64
    arithmetic on them, and the intermediate u = W_down h is NOT rounded (a
    kernel that rounds it is held to a rounding bound by the tests);
  * the head's outputs are the logits z, and per row the maximum, the natural
    log-sum-exp lse = log sum_v exp(z_v) (so q_v = exp(z_v - lse)) and the
    first index of the maximum (the greedy draft token; lowest index on ties);
  * a batch is M rows of h, each projected independently.
"""
from __future__ import annotations

import numpy as np

from .ssd_oracle import bf16_to_f64


def lowrank_project(h: np.ndarray, w_down: np.ndarray, w_up: np.ndarray):
    """[SlimSpec "아키텍처"] u = W_down h, z = W_up u for each row of h.

    h [M][d], w_down [r][d], w_up [V][r] as fp64 values; returns (u [M][r], z [M][V]).
    Row m of the batch is the column vector h of the page: u[m] = W_down h[m],
    z[m] = W_up u[m].
    """
    h = np.asarray(h, np.float64)
    w_down = np.asarray(w_down, np.float64)
    w_up = np.asarray(w_up, np.float64)
    if h.ndim != 2 or w_down.ndim != 2 or w_up.ndim != 2:
        raise ValueError("h, W_down and W_up are matrices")
    if w_down.shape[1] != h.shape[1] or w_up.shape[1] != w_down.shape[0]:
        raise ValueError("shapes: h [M][d], W_down [r][d], W_up [V][r]")
    u = h @ w_down.T            # u[m, j] = sum_k W_down[j, k] h[m, k]
    z = u @ w_up.T              # z[m, v] = sum_j W_up[v, j] u[m, j]
    return u, z


def head_stats(z: np.ndarray):
    """[SD-anatomy §3: q = softmax(z)] per row: max, natural log-sum-exp, first argmax.

    lse is written as max + log(sum exp(z - max)), which equals log(sum exp z)
    and does not overflow.
    """
    z = np.asarray(z, np.float64)
    zmax = z.max(axis=-1)
    lse = zmax + np.log(np.exp(z - zmax[..., None]).sum(axis=-1))
    arg = np.argmax(z, axis=-1)          # numpy returns the first maximum
    return zmax, lse, arg


def slimspec_head(h_bits: np.ndarray, w_down_bits: np.ndarray, w_up_bits: np.ndarray) -> dict:
    """The head on bf16 inputs (uint16 bit patterns): u, z, row max, lse, argmax."""
    u, z = lowrank_project(bf16_to_f64(h_bits), bf16_to_f64(w_down_bits), bf16_to_f64(w_up_bits))
    zmax, lse, arg = head_stats(z)
    return {"u": u, "z": z, "row_max": zmax, "lse": lse, "argmax": arg.astype(np.int64)}


def fullrank_head(h_bits: np.ndarray, w_full_bits: np.ndarray) -> dict:
    """[SlimSpec "아키텍처"] the head SlimSpec replaces: z = W_full h, W_full of V x d."""
    h = bf16_to_f64(h_bits)
    w = bf16_to_f64(w_full_bits)
    z = h @ w.T
    zmax, lse, arg = head_stats(z)
    return {"z": z, "row_max": zmax, "lse": lse, "argmax": arg.astype(np.int64)}


def mac_counts(d: int, r: int, V: int) -> dict:
    """[SlimSpec "아키텍처"] multiply-adds per row: full rank V*d, factored r*d + V*r."""
    return {"full": V * d, "lowrank": r * d + V * r}
