"""Seeded synthetic inputs for the speculate-and-verify step.

This module only draws random numbers and lays them out; it contains none of
the step's arithmetic (no matching, no attention, no softmax, no acceptance).
Both the CPU oracle tests and the CUDA path are fed from here, byte for byte.

Shapes follow the workloads the SwitchSD page describes ("어떻게 쓰나",
experiments on Llama-3.1-8B, Llama-3.3-70B and Qwen3-8B): a token context with
verbatim repeats, a mid-layer hidden state for the probe, a GQA KV cache, the
candidate tokens' Q/K/V, and target/draft logits over the full vocabulary.

Conventions
-----------
* ``N(0, x)`` in a workload description means variance ``x``.
* bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
  from an fp32 draw); fp32 tensors as ``float32``.
* Uniforms are multiples of 2^-24 in [0, 1) so they are exact in fp32.
* Layouts (row-major):
    ctx      [B][ctx_stride] int32 (padding -1), ctx_len [B] int32
    h        [B][d]   (f32 or bf16 bits),  w [d] f32
    q        [B][NT][Hq][dh]           (NT = NB * Dmax candidate slots)
    k_cache  [B][Hkv][P_max][dh],  v_cache likewise
    k_cand   [B][NT][Hkv][dh],     v_cand likewise
    tgt      [B][1 + NT][V]   target logits (row 0 = current position)
    drf      [B][K][V]        draft logits of the chain block (if K > 0)
    chain_tok[B][K] int32     draft tokens, drawn from softmax(drf) (Gumbel-max)
    u_acc    [B][NB][Dmax] f32, u_fin [B] f32
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 0x55D0


# ---------------------------------------------------------------------------
# workload descriptions
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    ctx_len: tuple            # (lo, hi) inclusive; lo == hi for a fixed length
    V: int
    zipf_s: float             # 0 -> uniform token ids
    repeat_density: tuple     # (lo, hi) fraction of tokens inside planted repeats
    span_len: tuple           # (lo, hi) planted span lengths
    n_spans: int              # > 0: plant exactly this many spans (ignores density)
    kappa: int
    W: int
    D: int
    K: int                    # chain draft length (0 = no chain block)
    chain_policy: int         # 0 none, 1 chain block when the gate is off, 2 always
    d_probe: int
    h_dtype: str              # 'f32' | 'bf16'
    tau: float
    Hq: int
    Hkv: int
    dh: int
    kv_dtype: str             # 'f32' | 'bf16'
    logit_dtype: str          # 'f32' | 'bf16'
    logit_var: float
    gate_on_frac: float       # fraction of sequences whose probe score is set high
    mode: str = "sample"      # 'sample' | 'greedy'
    description: str = ""

    @property
    def NB(self) -> int:
        return self.W + (1 if self.chain_policy else 0)

    @property
    def Dmax(self) -> int:
        return max(self.D, self.K) if self.chain_policy else self.D

    @property
    def NT(self) -> int:
        return self.NB * self.Dmax

    @property
    def NR(self) -> int:
        return 1 + self.NT

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        name="tiny", B=1, ctx_len=(512, 512), V=1000, zipf_s=0.0,
        repeat_density=(0.0, 0.0), span_len=(8, 40), n_spans=4,
        kappa=5, W=2, D=8, K=8, chain_policy=1,
        d_probe=64, h_dtype="f32", tau=0.4,
        Hq=4, Hkv=2, dh=64, kv_dtype="f32", logit_dtype="f32", logit_var=2.0,
        gate_on_frac=1.0,
        description="1 seq, ctx 512 uniform over V=1000, 4 planted repeats, "
                    "W=2 D=8, fp32 4q/2kv dh64, fp32 logits N(0,2)"),
    "llama8b": Workload(
        name="llama8b", B=1, ctx_len=(4096, 4096), V=128256, zipf_s=1.1,
        repeat_density=(0.3, 0.3), span_len=(20, 200), n_spans=0,
        kappa=5, W=4, D=20, K=0, chain_policy=0,
        d_probe=4096, h_dtype="bf16", tau=0.4,
        Hq=32, Hkv=8, dh=128, kv_dtype="bf16", logit_dtype="f32", logit_var=3.0,
        gate_on_frac=1.0,
        description="Llama-3.1-8B-shaped verify: B=1, prefix 4096, GQA 32/8 dh128 "
                    "bf16 KV, W=4 D=20, fp32 logits V=128256"),
    "batched": Workload(
        name="batched", B=32, ctx_len=(1024, 16384), V=128256, zipf_s=1.1,
        repeat_density=(0.0, 0.6), span_len=(20, 200), n_spans=0,
        kappa=5, W=8, D=16, K=7, chain_policy=1,
        d_probe=4096, h_dtype="bf16", tau=0.4,
        Hq=32, Hkv=8, dh=128, kv_dtype="bf16", logit_dtype="f32", logit_var=3.0,
        gate_on_frac=0.5,
        description="batched serving: B=32, prefix 1k-16k, W=8 D=16, half gated "
                    "off -> chain K=7"),
    "llama70b": Workload(
        name="llama70b", B=4, ctx_len=(32768, 32768), V=128256, zipf_s=1.1,
        repeat_density=(0.3, 0.3), span_len=(20, 200), n_spans=0,
        kappa=5, W=4, D=20, K=5, chain_policy=2,
        d_probe=8192, h_dtype="bf16", tau=0.4,
        Hq=64, Hkv=8, dh=128, kv_dtype="bf16", logit_dtype="f32", logit_var=3.0,
        gate_on_frac=1.0,
        description="Llama-3.3-70B-shaped verify: B=4, prefix 32768, GQA 64/8, "
                    "W=4 D=20 plus a K=5 chain block"),
    "qwen8b_mixed": Workload(
        name="qwen8b_mixed", B=64, ctx_len=(2048, 8192), V=151936, zipf_s=1.1,
        repeat_density=(0.0, 0.6), span_len=(20, 200), n_spans=0,
        kappa=5, W=4, D=20, K=5, chain_policy=1,
        d_probe=4096, h_dtype="bf16", tau=0.4,
        Hq=32, Hkv=8, dh=128, kv_dtype="bf16", logit_dtype="bf16", logit_var=3.0,
        gate_on_frac=0.5,
        description="Qwen3-8B-shaped mixed batch: B=64, prefix 2k-8k, copy (W=4 "
                    "D=20) or chain (K=5) per sequence, bf16 logits V=151936"),
}

# the Qwen3-8B-shaped batch at the copy-mode activation rate the SwitchSD page reports for
# Qwen3-8B ("어떻게 쓰나": copying fires on 8.6% of steps): 6 of 64 sequences in copy mode
WORKLOADS["qwen8b_mixed_act086"] = WORKLOADS["qwen8b_mixed"].replace(
    name="qwen8b_mixed_act086", gate_on_frac=0.086,
    description="Qwen3-8B-shaped mixed batch at 8.6% copy activation: B=64, prefix 2k-8k, copy (W=4 "
                "D=20) for 6 sequences, chain (K=5) for the rest, bf16 logits V=151936")

# order of the five workloads (small case first); variants take the seeds after them
WORKLOAD_ORDER = ["tiny", "llama8b", "batched", "llama70b", "qwen8b_mixed"]
VARIANT_ORDER = ["qwen8b_mixed_act086"]


def default_seed(name: str) -> int:
    """The seed a workload's inputs are drawn with unless one is given."""
    if name in WORKLOAD_ORDER:
        return SEED_BASE + WORKLOAD_ORDER.index(name)
    if name in VARIANT_ORDER:
        return SEED_BASE + len(WORKLOAD_ORDER) + VARIANT_ORDER.index(name)
    return SEED_BASE

# the speculation-tax experiment: every sequence ends in a repeated kappa-gram, half of
# them copy-intended (probe high, target follows the copy), half accidental (probe low,
# target unrelated to the copy)
TAX_WORKLOAD = Workload(
    name="tax64", B=64, ctx_len=(1024, 1024), V=32000, zipf_s=1.1,
    repeat_density=(0.1, 0.1), span_len=(20, 60), n_spans=0,
    kappa=5, W=4, D=8, K=0, chain_policy=0,
    d_probe=1024, h_dtype="bf16", tau=0.4,
    Hq=8, Hkv=2, dh=128, kv_dtype="bf16", logit_dtype="f32", logit_var=3.0,
    gate_on_frac=1.0,
    description="speculation tax: B=64, ctx 1024, every sequence ends in a repeated 5-gram, "
                "half copy-intended, half accidental; W=4 D=8, fp32 logits V=32000")


# ---------------------------------------------------------------------------
# helpers (sampling and bit layout only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)   # no overflow for finite x
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def uniforms24(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniforms k * 2^-24, k uniform on [0, 2^24): exact in fp32."""
    k = rng.integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (k.astype(np.float64) * 2.0 ** -24).astype(np.float32)


def _zipf_ids(rng: np.random.Generator, n: int, V: int, s: float, perm: np.ndarray) -> np.ndarray:
    """Truncated Zipf(s) over V ranks by inverse CDF, mapped through a fixed id permutation."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    r = np.searchsorted(cdf, rng.random(n), side="right")
    r = np.minimum(r, V - 1)
    return perm[r].astype(np.int32)


def _plant_spans(rng, row: np.ndarray, n: int, span_len, density: float, n_spans: int):
    """Copy verbatim spans from earlier positions to later ones (forward copies)."""
    lo, hi = span_len
    covered, planted = 0, 0
    target = density * n
    guard = 0
    while (planted < n_spans) if n_spans > 0 else (covered < target):
        guard += 1
        if guard > 100000:
            break
        L = int(rng.integers(lo, hi + 1))
        if 2 * L + 1 > n:
            L = max(1, (n - 1) // 2)
        dst = int(rng.integers(L, n - L + 1))
        src = int(rng.integers(0, dst - L + 1))
        row[dst:dst + L] = row[src:src + L].copy()
        covered += L
        planted += 1


def _plant_copy_tail(rng, row: np.ndarray, n: int, kappa: int, D: int, reps: int):
    """Make the context end inside a repeat: the last m >= kappa tokens equal an
    earlier span whose next D tokens exist, and plant `reps` more copies of that
    span (with its continuation) at distinct earlier positions."""
    m = int(rng.integers(kappa, 2 * kappa + 1))
    span = m + D
    need = (reps + 1) * (span + 1) + m + 1
    if need > n:
        reps = max(0, (n - m - 1) // (span + 1) - 1)
    tail0 = n - m
    # source of the tail: somewhere early, with room for its continuation
    slots = (tail0 - 1) // (span + 1)
    if slots < 1:
        return
    chosen = np.sort(rng.choice(slots, size=min(slots, reps + 1), replace=False))
    starts = [int(c) * (span + 1) + int(rng.integers(0, 2)) for c in chosen]
    starts = [s for s in starts if s + span < tail0]
    if not starts:
        return
    src = starts[0]
    seg = row[src:src + span].copy()
    for s in starts[1:]:
        row[s:s + span] = seg
    row[tail0:n] = seg[:m]


def _probe_pair(rng, d: int, alphas: np.ndarray, h_dtype: str):
    """w ~ N(0, 1/d); h_b = alpha_b * w/|w|^2 + noise orthogonal to w, so w.h_b = alpha_b
    before the cast to the storage dtype."""
    w64 = rng.standard_normal(d) / math.sqrt(d)
    w32 = w64.astype(np.float32)
    w = w32.astype(np.float64)
    ww = float(w @ w)
    B = len(alphas)
    noise = rng.standard_normal((B, d))
    noise -= np.outer(noise @ w / ww, w)
    h = alphas[:, None] * w[None, :] / ww + noise
    return _cast(h.astype(np.float32), h_dtype), w32


def logit_of(p: float) -> float:
    return math.log(p / (1.0 - p))


# ---------------------------------------------------------------------------
# main entry
# ---------------------------------------------------------------------------
def make_inputs(wl: Workload, seed: int | None = None, *, full_width: bool = True,
                with_attention: bool = True, with_logits: bool = True,
                ctx_lens=None, gate_on=None, q_scale: float = 1.0, probe_on=None) -> dict:
    """Draw one batch of inputs for workload `wl`.

    full_width: gate-on sequences get W extra copies of the tail's source span, so
        retrieval finds >= W candidates of full length D (measurement runs).
        False draws the number of extra copies from U{0..2W-1} (correctness runs).
    ctx_lens / gate_on: optional per-sequence overrides (gate_on plants the copy tail and,
        unless probe_on is given, sets the probe score high).
    probe_on: optional per-sequence probe target (score 0.9 or 0.1) independent of the tail.
    q_scale: multiplies Q (sharper attention for tests).
    """
    if seed is None:
        seed = default_seed(wl.name)
    rng = np.random.Generator(np.random.PCG64(seed))
    B = wl.B
    lo, hi = wl.ctx_len
    if ctx_lens is None:
        ctx_lens = rng.integers(lo, hi + 1, size=B) if hi > lo else np.full(B, lo)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    if gate_on is None:
        n_on = int(round(wl.gate_on_frac * B))
        gate_on = np.zeros(B, dtype=bool)
        gate_on[rng.permutation(B)[:n_on]] = True
    gate_on = np.asarray(gate_on, dtype=bool)

    stride = max(1, int(ctx_lens.max()))
    ctx = np.full((B, stride), -1, dtype=np.int32)
    perm = rng.permutation(wl.V).astype(np.int32) if wl.zipf_s > 0 else None
    dens_lo, dens_hi = wl.repeat_density
    for b in range(B):
        n = int(ctx_lens[b])
        if n == 0:
            continue
        if wl.zipf_s > 0:
            row = _zipf_ids(rng, n, wl.V, wl.zipf_s, perm)
        else:
            row = rng.integers(0, wl.V, size=n, dtype=np.int32)
        dens = float(rng.uniform(dens_lo, dens_hi)) if dens_hi > dens_lo else dens_lo
        _plant_spans(rng, row, n, wl.span_len, dens, wl.n_spans)
        if gate_on[b] and wl.W > 0:
            reps = wl.W if full_width else int(rng.integers(0, 2 * wl.W))
            _plant_copy_tail(rng, row, n, wl.kappa, wl.D, reps)
        ctx[b, :n] = row

    probe_on = gate_on if probe_on is None else np.asarray(probe_on, dtype=bool)
    alphas = np.where(probe_on, logit_of(0.9), logit_of(0.1))
    h, w = _probe_pair(rng, wl.d_probe, alphas, wl.h_dtype)

    out = dict(ctx=ctx, ctx_len=ctx_lens, h=h, w=w, gate_on_target=gate_on)

    NB, Dmax, NT = wl.NB, wl.Dmax, wl.NT
    if with_attention:
        P_max = stride
        f = np.float32
        q = rng.standard_normal((B, NT, wl.Hq, wl.dh), dtype=f)
        if q_scale != 1.0:
            q *= f(q_scale)
        out["q"] = _cast(q, wl.kv_dtype)
        del q
        out["k_cache"] = _cast(rng.standard_normal((B, wl.Hkv, P_max, wl.dh), dtype=f), wl.kv_dtype)
        out["v_cache"] = _cast(rng.standard_normal((B, wl.Hkv, P_max, wl.dh), dtype=f), wl.kv_dtype)
        out["k_cand"] = _cast(rng.standard_normal((B, NT, wl.Hkv, wl.dh), dtype=f), wl.kv_dtype)
        out["v_cand"] = _cast(rng.standard_normal((B, NT, wl.Hkv, wl.dh), dtype=f), wl.kv_dtype)
        out["prefix_len"] = ctx_lens.copy()

    if with_logits:
        sd = np.float32(math.sqrt(wl.logit_var))
        tgt = rng.standard_normal((B, wl.NR, wl.V), dtype=np.float32)
        tgt *= sd
        out["tgt"] = _cast(tgt, wl.logit_dtype)
        del tgt
        if wl.K > 0:
            drf = rng.standard_normal((B, wl.K, wl.V), dtype=np.float32)
            drf *= sd
            # draft tokens ~ softmax(drf) by the Gumbel-max construction; the
            # logits are taken in the precision they are stored in
            drf_stored = _cast(drf, wl.logit_dtype)
            drf_vals = drf if wl.logit_dtype == "f32" else bf16_bits_to_f32(drf_stored)
            g = -np.log(-np.log(rng.random((B, wl.K, wl.V)) * (1 - 1e-12) + 1e-300))
            out["chain_tok"] = np.argmax(drf_vals.astype(np.float64) + g, axis=2).astype(np.int32)
            out["drf"] = drf_stored
            del drf, g
        else:
            out["chain_tok"] = np.zeros((B, 0), dtype=np.int32)
            out["drf"] = None
    if not with_logits:
        out["chain_tok"] = rng.integers(0, wl.V, size=(B, wl.K)).astype(np.int32)
    out["u_acc"] = uniforms24(rng, (B, NB, Dmax))
    out["u_fin"] = uniforms24(rng, (B,))
    return out


def make_inputs_device(wl: Workload, seed: int | None, device, *, full_width: bool = True) -> dict:
    """The recipe of make_inputs with the large tensors drawn on `device` by torch's seeded
    generator: Q, the prefix K/V cache and the candidate K/V ~ N(0, 1) and the target and
    draft logits ~ N(0, logit_var), stored as bf16 (torch.bfloat16 viewed as int16) or fp32,
    and the chain tokens drawn from softmax(draft logits) by the Gumbel-max construction.
    The context, probe and uniforms come from make_inputs on the host. Host-side drawing of
    the multi-GB batches takes minutes; the values differ from make_inputs' but follow the
    same distributions (timing runs only: no oracle sees them)."""
    import torch
    if seed is None:
        seed = default_seed(wl.name)
    out = make_inputs(wl, seed, full_width=full_width, with_attention=False, with_logits=False)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) + 0x7E57)
    B, NT = wl.B, wl.NT
    P_max = int(out["ctx"].shape[1])

    def draw(shape, dtype, std=1.0):
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16).view(torch.int16) if dtype == "bf16" else x

    out["q"] = draw((B, NT, wl.Hq, wl.dh), wl.kv_dtype)
    out["k_cache"] = draw((B, wl.Hkv, P_max, wl.dh), wl.kv_dtype)
    out["v_cache"] = draw((B, wl.Hkv, P_max, wl.dh), wl.kv_dtype)
    out["k_cand"] = draw((B, NT, wl.Hkv, wl.dh), wl.kv_dtype)
    out["v_cand"] = draw((B, NT, wl.Hkv, wl.dh), wl.kv_dtype)
    out["prefix_len"] = out["ctx_len"].copy()
    sd = math.sqrt(wl.logit_var)
    out["tgt"] = draw((B, wl.NR, wl.V), wl.logit_dtype, sd)
    if wl.K > 0:
        drf = draw((B, wl.K, wl.V), wl.logit_dtype, sd)
        vals = drf.view(torch.bfloat16).float() if wl.logit_dtype == "bf16" else drf
        u = torch.rand((B, wl.K, wl.V), generator=gen, device=device, dtype=torch.float64)
        g = -torch.log(-torch.log(u * (1 - 1e-12) + 1e-300))
        out["chain_tok"] = torch.argmax(vals.double() + g, dim=2).to(torch.int32).cpu().numpy()
        out["drf"] = drf
        del u, g, vals
    else:
        out["chain_tok"] = np.zeros((B, 0), dtype=np.int32)
        out["drf"] = None
    return out


def boost_accepts(tgt: np.ndarray, logit_dtype: str, row_tok: dict, boost: float = 20.0) -> np.ndarray:
    """Return a copy of target logits with `boost` added at (b, row, tok) for every
    entry of row_tok {(b, row): tok}; used to make long accepted runs likely."""
    t = tgt.copy()
    for (b, r), tok in row_tok.items():
        if logit_dtype == "f32":
            t[b, r, tok] = np.float32(t[b, r, tok] + boost)
        else:
            v = bf16_bits_to_f32(t[b, r, tok:tok + 1])[0] + np.float32(boost)
            t[b, r, tok] = f32_to_bf16_bits(np.array([v], dtype=np.float32))[0]
    return t


def algorithmic_bytes(wl: Workload, prefix_len: np.ndarray, blk_len: np.ndarray) -> dict:
    """Bytes one step must move at minimum: the prefix KV once per kv head, the
    candidate Q/K/V/O, every needed target/draft logit row once, the context, h and w.
    blk_len [B][NB] gives the verified tokens per block."""
    kv_es = 4 if wl.kv_dtype == "f32" else 2
    lg_es = 4 if wl.logit_dtype == "f32" else 2
    h_es = 4 if wl.h_dtype == "f32" else 2
    T = int(blk_len.sum())
    kv = int(prefix_len.sum()) * wl.Hkv * wl.dh * kv_es * 2
    qo = T * wl.Hq * wl.dh * kv_es * 2
    kvc = T * wl.Hkv * wl.dh * kv_es * 2
    n_rows = 0
    n_drf = 0
    for b in range(blk_len.shape[0]):
        n_rows += 1 + int(blk_len[b].sum())
        if wl.chain_policy:
            n_drf += int(blk_len[b, wl.W])
    logits = (n_rows + n_drf) * wl.V * lg_es
    other = int(prefix_len.sum()) * 4 + blk_len.shape[0] * wl.d_probe * h_es + wl.d_probe * 4
    return dict(kv=kv, q_o=qo, kv_cand=kvc, logits=logits, other=other,
                attn=kv + qo + kvc, total=kv + qo + kvc + logits + other, tokens=T)


# ---------------------------------------------------------------------------
# the SlimSpec low-rank draft head (a second workload; SlimSpec page,
# "방법론: SlimSpec" / "아키텍처": r = d/8, evaluated on Llama-3.1-8B drafters at
# batch 1 and 64)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class HeadWorkload:
    name: str
    M: int                    # rows of h (draft positions of a batch)
    d: int                    # hidden size
    r: int                    # rank
    V: int                    # vocabulary
    z_std: float              # standard deviation of the logits the weights produce
    description: str = ""


HEAD_WORKLOADS = {
    # small: several 128-row vocabulary tiles and a ragged tail (V % 128 != 0), a
    # rank that is not a multiple of 64, a batch that is not a multiple of 16
    "head_small": HeadWorkload("head_small", M=5, d=512, r=72, V=1000, z_std=3.0,
                               description="low-rank head d=512 r=72 V=1000, 5 rows"),
    "head_llama8b_b1": HeadWorkload("head_llama8b_b1", M=1, d=4096, r=512, V=128256, z_std=3.0,
                                    description="low-rank head d=4096 r=512 V=128256, batch 1"),
    "head_llama8b_b64": HeadWorkload("head_llama8b_b64", M=64, d=4096, r=512, V=128256, z_std=3.0,
                                     description="low-rank head d=4096 r=512 V=128256, batch 64"),
}


def make_head_inputs(hw: HeadWorkload, seed: int | None = None) -> dict:
    """bf16 bit patterns: h [M][d] ~ N(0, 1), W_down [r][d] ~ N(0, 1/d),
    W_up [V][r] ~ N(0, z_std^2 / r), so that W_down h has unit-variance entries
    and the logits have standard deviation about z_std."""
    if seed is None:
        seed = SEED_BASE + 0x5E
    rng = np.random.Generator(np.random.PCG64(seed))
    h = rng.standard_normal((hw.M, hw.d), dtype=np.float32)
    w_down = rng.standard_normal((hw.r, hw.d), dtype=np.float32) * np.float32(1.0 / math.sqrt(hw.d))
    w_up = rng.standard_normal((hw.V, hw.r), dtype=np.float32) * np.float32(hw.z_std / math.sqrt(hw.r))
    return {"h": f32_to_bf16_bits(h), "w_down": f32_to_bf16_bits(w_down), "w_up": f32_to_bf16_bits(w_up)}
