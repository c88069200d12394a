"""GPU vocabulary rows, acceptance and final draw against the oracle.

Given identical fp32 probabilities and uniforms (SSD_PROBS_F32) every decision
is bit-exact. From logits, p is within 1e-5 relative and decisions agree
except where the oracle's own margin is below that precision. The sampler's
output distribution passes a chi-square test (>= 1e6 trials)."""
import numpy as np
import pytest
import scipy.stats
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import VerifyStep, arena_bytes, to_device

pytestmark = pytest.mark.gpu

KIND = {"probs_f32": S.SSD_PROBS_F32, "logits_f32": S.SSD_LOGITS_F32, "logits_bf16": S.SSD_LOGITS_BF16}
MODE = {"sample": S.SSD_SAMPLE, "greedy": S.SSD_GREEDY}


def _blocks(rng, B, W, Dmax, K, V, chain_policy):
    NB = W + (1 if chain_policy else 0)
    blk_len = rng.integers(0, Dmax + 1, size=(B, NB)).astype(np.int32)
    if chain_policy:
        blk_len[:, W] = np.where(rng.random(B) < 0.5, K, 0)
    blk_len[rng.random(B) < 0.1] = 0                              # some sequences without any block
    blk_tok = rng.integers(0, V, size=(B, NB, Dmax)).astype(np.int32)
    for b in range(B):
        for k in range(NB):
            blk_tok[b, k, blk_len[b, k]:] = -1
    return blk_tok, blk_len


def _rows_probs(rng, shape, conc=0.3):
    p = rng.gamma(conc, size=shape)
    return (p / p.sum(axis=-1, keepdims=True)).astype(np.float32)


def _boost_probs(tgt, blk_tok, blk_len, Dmax, rng):
    """Put most of a row's mass on the token it verifies for a random leading run."""
    t = tgt.copy()
    B, NB, _ = blk_tok.shape
    for b in range(B):
        for k in range(NB):
            a = int(rng.integers(0, blk_len[b, k] + 1))
            for d in range(a):
                r = 0 if d == 0 else 1 + k * Dmax + d - 1
                t[b, r] *= 0.05
                t[b, r, blk_tok[b, k, d]] += 0.95
    return t


def _gpu_accept(mode, kind, tgt, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin, probs=False, early=False):
    dev = "cuda"
    T = lambda a: to_device(np.asarray(a), dev) if a is not None else None
    tt = T(tgt)
    po = torch.empty(tgt.shape, dtype=torch.float32, device=dev) if probs else None
    r = S.ssd_accept(tt, T(drf), T(blk_tok), T(blk_len), T(u_acc), T(u_fin), mode=MODE[mode], kind=KIND[kind], K=K,
                     chain_blk=chain_blk, probs_out=po, early_rows=early)
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in r.items()}
    if probs:
        out["probs"] = po.cpu().numpy()
    return out


def _oracle(mode, kind, tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin):
    return O.verify_step_accept(mode, kind, tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin)


def _assert_same(got, ref):
    for k in ("acc_len", "best_blk", "n_out", "out_tok"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


@pytest.mark.parametrize("mode", ["sample", "greedy"])
@pytest.mark.parametrize("V,B,W,Dmax,K,policy", [(17, 64, 3, 6, 4, 1), (1000, 40, 4, 20, 5, 2),
                                                  (4099, 16, 8, 16, 7, 1), (128256, 3, 4, 20, 0, 0)])
def test_accept_probs_bit_exact(mode, V, B, W, Dmax, K, policy):
    rng = np.random.default_rng(V + B)
    blk_tok, blk_len = _blocks(rng, B, W, Dmax, K, V, policy)
    NB = blk_tok.shape[1]
    tgt = _boost_probs(_rows_probs(rng, (B, 1 + NB * Dmax, V)), blk_tok, blk_len, Dmax, rng)
    drf = _rows_probs(rng, (B, K, V)) if policy else None
    if policy:
        # chain tokens drawn where q has mass, so q(x) > 0
        for b in range(B):
            for d in range(blk_len[b, W]):
                blk_tok[b, W, d] = int(np.argmax(drf[b, d] * rng.random(V)))
    u_acc = WL.uniforms24(rng, (B, NB, Dmax))
    u_fin = WL.uniforms24(rng, (B,))
    chain_blk = W if policy else -1
    got = _gpu_accept(mode, "probs_f32", tgt, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin)
    ref = _oracle(mode, "probs_f32", tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin)
    _assert_same(got, ref)
    assert ref["acc_len"].max() > 0          # the boost produced accepted runs


@pytest.mark.parametrize("early", [True, False])
@pytest.mark.parametrize("V,B,W,Dmax,K,policy,kind", [(1000, 40, 4, 20, 5, 2, "probs_f32"),
                                                       (128256, 3, 4, 20, 5, 1, "probs_f32"),
                                                       (151936, 4, 4, 20, 5, 1, "logits_bf16")])
def test_accept_row_pass_full_vocabularies(early, V, B, W, Dmax, K, policy, kind):
    """The row pass on full vocabularies in both modes: decisions bit-exact against the oracle
    where probabilities are given; p of every needed row within 1e-5 relative from bf16
    logits."""
    rng = np.random.default_rng(V + B + 5)
    blk_tok, blk_len = _blocks(rng, B, W, Dmax, K, V, policy)
    NB = blk_tok.shape[1]
    if kind == "probs_f32":
        tgt = _boost_probs(_rows_probs(rng, (B, 1 + NB * Dmax, V)), blk_tok, blk_len, Dmax, rng)
        drf = _rows_probs(rng, (B, K, V))
    else:
        lg = (rng.standard_normal((B, 1 + NB * Dmax, V)) * np.sqrt(3)).astype(np.float32)
        tgt = WL.f32_to_bf16_bits(lg)
        drf = WL.f32_to_bf16_bits((rng.standard_normal((B, K, V)) * np.sqrt(3)).astype(np.float32))
    for b in range(B):
        for d in range(blk_len[b, W]):
            q = drf[b, d] if kind == "probs_f32" else np.exp(WL.bf16_bits_to_f32(drf[b, d]) - 10)
            blk_tok[b, W, d] = int(np.argmax(q * rng.random(V)))
    u_acc = WL.uniforms24(rng, (B, NB, Dmax))
    u_fin = WL.uniforms24(rng, (B,))
    got = _gpu_accept("sample", kind, tgt, drf, blk_tok, blk_len, K, W, u_acc, u_fin, probs=True, early=early)
    ref = _oracle("sample", kind, tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin)
    if kind == "probs_f32":
        _assert_same(got, ref)
    else:
        for b in range(B):
            rows = [0] + [1 + k * Dmax + d for k in range(NB) for d in range(int(blk_len[b, k]))]
            np.testing.assert_allclose(got["probs"][b, rows], O.softmax_f64(O.row_values(tgt[b, rows], kind)),
                                       rtol=1e-5, atol=1e-30)
            same = all(np.array_equal(got[k][b], ref[k][b]) for k in ("acc_len", "best_blk", "n_out", "out_tok"))
            if not same:
                assert _margins_explain(kind, tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin, got, ref, b)


@pytest.mark.parametrize("mode", ["sample", "greedy"])
@pytest.mark.parametrize("V,B,W,Dmax,K,policy", [(17, 64, 3, 6, 4, 1), (4099, 16, 8, 16, 7, 1),
                                                  (128256, 3, 4, 20, 0, 0)])
def test_accept_early_rows(mode, V, B, W, Dmax, K, policy):
    """The early row pass reads every row, rows of absent tokens included: filled with
    NaN here, they must change nothing. Bit-exact against the oracle and against the
    row pass that reads only the needed rows."""
    rng = np.random.default_rng(3 * V + B)
    blk_tok, blk_len = _blocks(rng, B, W, Dmax, K, V, policy)
    NB = blk_tok.shape[1]
    tgt = _boost_probs(_rows_probs(rng, (B, 1 + NB * Dmax, V)), blk_tok, blk_len, Dmax, rng)
    drf = _rows_probs(rng, (B, K, V)) if policy else None
    if policy:
        for b in range(B):
            for d in range(blk_len[b, W]):
                blk_tok[b, W, d] = int(np.argmax(drf[b, d] * rng.random(V)))
    u_acc = WL.uniforms24(rng, (B, NB, Dmax))
    u_fin = WL.uniforms24(rng, (B,))
    chain_blk = W if policy else -1
    ref = _oracle(mode, "probs_f32", tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin)
    poisoned = tgt.copy()
    for b in range(B):
        for k in range(NB):
            poisoned[b, 1 + k * Dmax + blk_len[b, k]:1 + (k + 1) * Dmax] = np.nan   # rows no token reads
    if policy:
        drf = drf.copy()
        for b in range(B):
            drf[b, blk_len[b, W]:] = np.nan
    early = _gpu_accept(mode, "probs_f32", poisoned, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin, early=True)
    late = _gpu_accept(mode, "probs_f32", poisoned, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin, early=False)
    _assert_same(early, ref)
    _assert_same(late, ref)


@pytest.mark.parametrize("max_ctas", [1, 7, 52])
def test_accept_row_pass_on_capped_grid(max_ctas):
    """The row pass on at most max_ctas SMs (one 16-warp CTA each) gives the same statistics:
    decisions bit-exact against the oracle given probabilities, early mode and not."""
    rng = np.random.default_rng(900 + max_ctas)
    V, B, W, Dmax, K, policy = 4000, 6, 4, 20, 5, 1
    blk_tok, blk_len = _blocks(rng, B, W, Dmax, K, V, policy)
    NB = blk_tok.shape[1]
    tgt = _boost_probs(_rows_probs(rng, (B, 1 + NB * Dmax, V)), blk_tok, blk_len, Dmax, rng)
    drf = _rows_probs(rng, (B, K, V))
    for b in range(B):
        for d in range(blk_len[b, W]):
            blk_tok[b, W, d] = int(np.argmax(drf[b, d] * rng.random(V)))
    u_acc = WL.uniforms24(rng, (B, NB, Dmax))
    u_fin = WL.uniforms24(rng, (B,))
    ref = _oracle("sample", "probs_f32", tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin)
    dev = "cuda"
    T = lambda a: to_device(np.asarray(a), dev)
    for early in (True, False):
        r = S.ssd_accept(T(tgt), T(drf), T(blk_tok), T(blk_len), T(u_acc), T(u_fin), mode=S.SSD_SAMPLE,
                         kind=S.SSD_PROBS_F32, K=K, chain_blk=W, early_rows=early, max_ctas=max_ctas)
        torch.cuda.synchronize()
        _assert_same({k: v.cpu().numpy() for k, v in r.items()}, ref)


@pytest.mark.parametrize("early", [True, False])
def test_accept_back_to_back_calls_share_a_workspace(early):
    """Calls issued one after another on one stream may share a workspace: each call's
    row pass writes the workspace only after the previous call's finish kernel (which
    reads it) has completed, in the early mode too. Pairs of calls with different rows
    on one workspace, each pair's results bit-exact against the oracle."""
    rng = np.random.default_rng(808 + early)
    V, B, W, Dmax, K, policy = 128256, 3, 4, 20, 5, 2
    dev = "cuda"
    T = lambda a: to_device(np.asarray(a), dev) if a is not None else None
    calls = []
    for _ in range(2):
        blk_tok, blk_len = _blocks(rng, B, W, Dmax, K, V, policy)
        NB = blk_tok.shape[1]
        tgt = _boost_probs(_rows_probs(rng, (B, 1 + NB * Dmax, V)), blk_tok, blk_len, Dmax, rng)
        drf = _rows_probs(rng, (B, K, V))
        for b in range(B):
            for d in range(blk_len[b, W]):
                blk_tok[b, W, d] = int(np.argmax(drf[b, d] * rng.random(V)))
        u_acc = WL.uniforms24(rng, (B, NB, Dmax))
        u_fin = WL.uniforms24(rng, (B,))
        calls.append((tgt, drf, blk_tok, blk_len, u_acc, u_fin))
    dv = [tuple(T(a) for a in c) for c in calls]
    args = S.accept_args(S.SSD_SAMPLE, S.SSD_PROBS_F32, *dv[0][:4], K, W, *dv[0][4:],
                         S.alloc_accept_outputs(B, W + 1, Dmax, dev))
    ws = torch.zeros(S.ssd_accept_workspace_size(args), dtype=torch.uint8, device=dev)
    refs = [_oracle("sample", "probs_f32", *c[:4], W, policy, *c[4:]) for c in calls]
    for rep in range(20):
        outs = []
        for c in dv:
            outs.append(S.ssd_accept(c[0], c[1], c[2], c[3], c[4], c[5], mode=S.SSD_SAMPLE, kind=S.SSD_PROBS_F32,
                                     K=K, chain_blk=W, ws=ws, early_rows=early))
        torch.cuda.synchronize()
        for ref, o in zip(refs, outs):
            _assert_same({k: v.cpu().numpy() for k, v in o.items()}, ref)
    assert S.ssd_read_device_error(ws) == S.SSD_OK


def _margins_explain(kind, tgt, drf, blk_tok, blk_len, W, policy, u_acc, u_fin, got, ref, b):
    """True if sequence b's disagreement sits within fp32 precision of one of the
    oracle's decision boundaries: an acceptance test u*q vs p, or the inverse-CDF
    threshold against a prefix sum of the final draw (both measured with the
    oracle's own quantities)."""
    B, NB, Dmax = blk_tok.shape
    for k in range(NB):
        for d in range(1, int(blk_len[b, k]) + 1):
            x = int(blk_tok[b, k, d - 1])
            r = 0 if d == 1 else 1 + k * Dmax + d - 2
            p = O.row_probs(tgt[b, r], kind)[x]
            q = O.row_probs(drf[b, d - 1], kind)[x] if (policy and k == W) else 1.0
            if abs(float(u_acc[b, k, d - 1]) * float(q) - float(p)) <= 1e-5 * max(float(p), 1e-30):
                return True
    n = int(ref["n_out"][b])
    if not (got["n_out"][b] == n and np.array_equal(got["out_tok"][b, :n - 1], ref["out_tok"][b, :n - 1])):
        return False
    ks = int(ref["best_blk"][b])
    a = n - 1
    L = int(blk_len[b, ks]) if ks >= 0 else 0
    r_stop = 0 if a == 0 else 1 + ks * Dmax + a - 1
    P = O.prob_weights(O.row_probs(tgt[b, r_stop], kind))
    Wt = P
    if a < L:
        if policy and ks == W:
            Q = O.prob_weights(O.row_probs(drf[b, a], kind))
        else:
            Q = np.zeros_like(P)
            Q[int(blk_tok[b, ks, a])] = 1 << O.FIX_PROB
        Wt = O.residual_weights(P, Q)
        if Wt.sum() == 0:
            Wt = P
    S_ = int(Wt.sum())
    T = (int(np.float32(u_fin[b]) * np.float32(2 ** 24)) * S_) >> 24
    C = np.cumsum(Wt)
    return float(np.min(np.abs(C - T))) <= 1e-5 * S_


@pytest.mark.parametrize("kind", ["logits_f32", "logits_bf16"])
@pytest.mark.parametrize("V", [1000, 151936])
def test_accept_logits_probs_and_decisions(kind, V):
    rng = np.random.default_rng(V + len(kind))
    B, W, Dmax, K, policy = 6, 4, 20, 5, 1
    blk_tok, blk_len = _blocks(rng, B, W, Dmax, K, V, policy)
    NB = blk_tok.shape[1]
    lg = (rng.standard_normal((B, 1 + NB * Dmax, V)) * np.sqrt(3)).astype(np.float32)
    dl = (rng.standard_normal((B, K, V)) * np.sqrt(3)).astype(np.float32)
    # long accepted runs: +20 on the logit of the verified token at leading positions
    for b in range(B):
        for k in range(NB):
            for d in range(int(rng.integers(0, blk_len[b, k] + 1))):
                r = 0 if d == 0 else 1 + k * Dmax + d - 1
                lg[b, r, blk_tok[b, k, d]] += 20.0
    if kind == "logits_bf16":
        lg, dl = WL.f32_to_bf16_bits(lg), WL.f32_to_bf16_bits(dl)
    u_acc = WL.uniforms24(rng, (B, NB, Dmax))
    u_fin = WL.uniforms24(rng, (B,))
    got = _gpu_accept("sample", kind, lg, dl, blk_tok, blk_len, K, W, u_acc, u_fin, probs=True)
    # p of every needed row within 1e-5 relative of the fp64 softmax
    for b in range(B):
        rows = [0] + [1 + k * Dmax + d for k in range(NB) for d in range(int(blk_len[b, k]))]
        ref_p = O.softmax_f64(O.row_values(lg[b, rows], kind))
        np.testing.assert_allclose(got["probs"][b, rows], ref_p, rtol=1e-5, atol=1e-30)
    ref = _oracle("sample", kind, lg, dl, blk_tok, blk_len, W, policy, u_acc, u_fin)
    for b in range(B):
        same = all(np.array_equal(got[k][b], ref[k][b]) for k in ("acc_len", "best_blk", "n_out", "out_tok"))
        if not same:
            assert _margins_explain(kind, lg, dl, blk_tok, blk_len, W, policy, u_acc, u_fin, got, ref, b)
    # greedy from logits: argmax comparisons are exact
    gg = _gpu_accept("greedy", kind, lg, dl, blk_tok, blk_len, K, W, u_acc, u_fin)
    _assert_same(gg, _oracle("greedy", kind, lg, dl, blk_tok, blk_len, W, policy, u_acc, u_fin))


@pytest.mark.parametrize("name,order", [(n, "two_streams") for n in WL.WORKLOAD_ORDER] +
                         [("tiny", "rows_first"), ("llama8b", "rows_first"), ("batched", "rows_first"),
                          ("tiny", "attn_first"), ("llama8b", "attn_first"),
                          ("tiny", "bench"), ("llama8b", "bench"), ("tiny", "split"), ("llama8b", "split"),
                          ("batched", "split")])
def test_whole_step_workloads(name, order):
    """gate -> retrieve -> accept and attention through the step's own launch path (one
    stream in either order, or attention on a second stream), compared with the oracle
    step on the same inputs (sampled rows for attention). One-stream steps run twice back
    to back on the same buffers; the second run's results are the ones checked."""
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl, 77 + len(name), full_width=False)
    two = order == "two_streams"
    split = order == "split"
    # "bench": the launch configuration the benchmark times (one stream, early row pass); "split":
    # the attention on a second stream (every row) beside the acceptance chain on capped grids
    st = VerifyStep(wl, inp, with_attention=(name in ("tiny", "llama8b")),
                    order=order if (order.endswith("_first") or split) else "rows_first",
                    early_rows=order == "bench" or (split and name != "batched"),
                    attn_ctas=96 if split else 0, rows_ctas=52 if split else 0)
    for _ in range(1 if two else 2):
        st.run(aux=torch.cuda.Stream() if (two or split) else None)
    got = st.results()
    ref = O.verify_step(inp, wl, attention_slots=None)
    for k in ("gate", "last_match_end", "blk_tok", "blk_len", "n_cand"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    kind = "logits_bf16" if wl.logit_dtype == "bf16" else "logits_f32"
    for b in range(wl.B):
        same = all(np.array_equal(got[k][b], ref[k][b]) for k in ("acc_len", "best_blk", "n_out", "out_tok"))
        if not same:
            assert _margins_explain(kind, inp["tgt"], inp.get("drf"), ref["blk_tok"], ref["blk_len"], wl.W,
                                    wl.chain_policy, inp["u_acc"], inp["u_fin"], got, ref, b)
    if st.with_attention:
        bl = ref["blk_len"]
        slots = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(bl[b, k])][:40]
        ra = O.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"], inp["v_cand"],
                                inp["prefix_len"], bl, wl.Dmax, wl.kv_dtype, slots)
        with np.errstate(invalid="ignore"):
            g = O.to_f64(got["attn"], wl.kv_dtype)
        assert max(float(np.max(np.abs(g[b, t] - o))) for (b, t), o in ra.items()) <= 1e-2


@pytest.mark.parametrize("V", [16, 64])
def test_gpu_sampler_chi_square(V):
    """One chain token per trial, q far from p: the first emitted token follows p."""
    rng = np.random.default_rng(500 + V)
    p = _rows_probs(rng, (V,), 0.7)
    q = _rows_probs(rng, (V,), 0.7)
    B = 250_000
    reps = 4
    dev = "cuda"
    tgt = torch.from_numpy(np.broadcast_to(np.stack([p, p])[None], (B, 2, V)).copy()).to(dev)
    drf = torch.from_numpy(np.broadcast_to(q[None, None], (B, 1, V)).copy()).to(dev)
    blk_len = torch.ones((B, 1), dtype=torch.int32, device=dev)
    counts = np.zeros(V, np.int64)
    for rep in range(reps):
        qd = q.astype(np.float64)
        x = rng.choice(V, size=B, p=qd / qd.sum()).astype(np.int32)
        u_acc = WL.uniforms24(rng, (B, 1, 1))
        u_fin = WL.uniforms24(rng, (B,))
        r = S.ssd_accept(tgt, drf, torch.from_numpy(x.reshape(B, 1, 1)).to(dev), blk_len,
                         torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_fin).to(dev), mode=S.SSD_SAMPLE,
                         kind=S.SSD_PROBS_F32, K=1, chain_blk=0)
        first = r["out_tok"][:, 0].cpu().numpy()
        counts += np.bincount(first, minlength=V)
        if rep == 0:
            # the same trials through the oracle: bit-exact on a subset
            n = 2000
            ref = O.verify_step_accept("sample", "probs_f32", np.broadcast_to(np.stack([p, p])[None], (n, 2, V)),
                                       np.broadcast_to(q[None, None], (n, 1, V)), x[:n].reshape(n, 1, 1),
                                       np.ones((n, 1), np.int32), 0, 2, u_acc[:n], u_fin[:n])
            np.testing.assert_array_equal(first[:n], ref["out_tok"][:, 0])
    N = B * reps
    pd = p.astype(np.float64)
    chi2, pval = scipy.stats.chisquare(counts, pd / pd.sum() * N)
    assert pval > 0.01, (chi2, pval)


@pytest.mark.parametrize("name", ["tiny", "llama8b"])
def test_steps_back_to_back_with_new_inputs(name):
    """Steps issued back to back on one stream and one set of buffers, the inputs replaced
    in place between them (ordinary copies on the same stream): the kernels of a step may
    start while the previous step's kernels still run, and each step's results must be
    those of its own inputs."""
    wl = WL.WORKLOADS[name]
    inps = [WL.make_inputs(wl, 300 + k, full_width=False) for k in range(3)]
    st = VerifyStep(wl, inps[0], early_rows=True)
    main = torch.cuda.Stream()
    got = []
    with torch.cuda.stream(main):
        for k, inp in enumerate(inps):
            if k > 0:
                for key, t in st.x.items():
                    t.copy_(to_device(inp[key], t.device).view(t.dtype).view(t.shape), non_blocking=False)
            st.run(main)
            got.append({key: v.clone() for key, v in {**st.ret_out, **st.acc_out}.items()})
            if st.with_attention:
                got[-1]["attn"] = st.attn_out.clone()
    torch.cuda.synchronize()
    for inp, g in zip(inps, got):
        ref = O.verify_step(inp, wl, attention_slots=None)
        for key in ("blk_tok", "blk_len", "n_cand"):
            np.testing.assert_array_equal(g[key].cpu().numpy(), ref[key], err_msg=key)
        kind = "logits_bf16" if wl.logit_dtype == "bf16" else "logits_f32"
        res = {key: g[key].cpu().numpy() for key in ("acc_len", "best_blk", "n_out", "out_tok")}
        for b in range(wl.B):
            same = all(np.array_equal(res[key][b], ref[key][b]) for key in res)
            if not same:
                assert _margins_explain(kind, inp["tgt"], inp.get("drf"), ref["blk_tok"], ref["blk_len"], wl.W,
                                        wl.chain_policy, inp["u_acc"], inp["u_fin"], res, ref, b)
        if "attn" in g:
            bl = ref["blk_len"]
            slots = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(bl[b, k])][:24]
            ra = O.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"], inp["v_cand"],
                                    inp["prefix_len"], bl, wl.Dmax, wl.kv_dtype, slots)
            ga = g["attn"].cpu()
            ga = ga.numpy() if wl.kv_dtype == "f32" else ga.view(torch.int16).numpy().view(np.uint16)
            with np.errstate(invalid="ignore"):
                ga = O.to_f64(ga, wl.kv_dtype)
            assert max(float(np.max(np.abs(ga[b, t] - o))) for (b, t), o in ra.items()) <= 1e-2


def test_step_from_one_input_arena_matches_separate_inputs():
    """The inputs placed in one arena (refreshed by a single host-to-device copy) give
    the same step results as separately allocated inputs."""
    wl = WL.WORKLOADS["llama8b"]
    inp = WL.make_inputs(wl, 91, full_width=False)
    a = VerifyStep(wl, inp, order="attn_first")
    b = VerifyStep(wl, inp, order="attn_first",
                   arena=torch.empty(arena_bytes(inp), dtype=torch.uint8, device="cuda"))
    a.run()
    b.run()
    ra, rb = a.results(), b.results()
    for k in ra:
        if k != "attn":
            np.testing.assert_array_equal(ra[k], rb[k], err_msg=k)
    bl = ra["blk_len"]
    for bb in range(wl.B):
        for k in range(wl.NB):
            sl = slice(k * wl.Dmax, k * wl.Dmax + int(bl[bb, k]))
            np.testing.assert_array_equal(ra["attn"][bb, sl], rb["attn"][bb, sl])
