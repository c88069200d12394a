"""Shared by the full-size GPU tests: seeded inputs of each workload (drawn once per
process), the oracle's attention on a list of slots in threads, the step in the
benchmark's configuration, and target/draft rows boosted into long accepted runs and
given as fp32 probabilities (the oracle's softmax)."""
import concurrent.futures as cf
import os

import numpy as np

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import VerifyStep, default_early_rows

TOL = 1e-2
CACHE = {}


def inputs(name):
    if name not in CACHE:
        wl = WL.WORKLOADS[name]
        CACHE[name] = (wl, WL.make_inputs(wl, WL.default_seed(name) + 300, full_width=False))
    return CACHE[name]


def oracle_attention(inp, wl, bl, slots, threads=None):
    threads = threads or min(16, os.cpu_count() or 1)
    chunks = [slots[i::threads] for i in range(threads) if slots[i::threads]]
    out = {}
    with cf.ThreadPoolExecutor(len(chunks)) as ex:
        for part in ex.map(lambda ch: O.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"],
                                                         inp["v_cand"], inp["prefix_len"], bl, wl.Dmax, wl.kv_dtype,
                                                         ch), chunks):
            out.update(part)
    return out


def bench_step(wl, inp, **kw):
    st = VerifyStep(wl, inp, early_rows=default_early_rows(wl), **kw)
    st.run()
    return st, st.results()


def max_err(got_attn, ref, dtype):
    with np.errstate(invalid="ignore"):
        g = O.to_f64(got_attn, dtype)
    return max(float(np.max(np.abs(g[b, t] - o))) for (b, t), o in ref.items())


def boosted_probs(wl, inp, seed):
    """Target and draft rows as fp32 probabilities (the oracle's softmax), the target rows
    boosted so that each block accepts a random number of leading tokens."""
    kind = "logits_bf16" if wl.logit_dtype == "bf16" else "logits_f32"
    _, _, gate, _ = O.gate_match(inp["ctx"], inp["ctx_len"], inp["h"], wl.h_dtype, inp["w"], wl.tau, wl.kappa)
    bt, bl, _ = O.retrieve(inp["ctx"], inp["ctx_len"], gate, wl.kappa, wl.W, wl.D, wl.K, wl.chain_policy,
                           inp["chain_tok"])
    rng = np.random.default_rng(seed)
    rows = {}
    for b in range(wl.B):
        for k in range(wl.NB):
            # every third block accepts all of its tokens (bonus draws), the others a random run
            a = int(bl[b, k]) if (b + k) % 3 == 0 else int(rng.integers(0, int(bl[b, k]) + 1))
            for d in range(a):
                rows[(b, 0 if d == 0 else 1 + k * wl.Dmax + d - 1)] = int(bt[b, k, d])
    tgt = WL.boost_accepts(inp["tgt"], wl.logit_dtype, rows)
    out = dict(inp)
    out["tgt"] = np.stack([O.row_probs(tgt[b], kind) for b in range(wl.B)])
    if inp.get("drf") is not None:
        out["drf"] = np.stack([O.row_probs(inp["drf"][b], kind) for b in range(wl.B)])
    return out


