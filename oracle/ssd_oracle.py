"""CPU oracle for the SwitchSD speculate-and-verify step.

TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
benchmark's CPU-baseline / reference leg are the only code that may import or
run this module. It shares no code with the CUDA library and imports nothing
from it; the product path never calls it.

It is a plain, slow, readable restatement of what the pages define, in fp64
where floating point is involved. Pages cited below, by title:

  [SwitchSD]   "SwitchSD는 LLM 내부 표현으로 추측 디코딩의 복사 모드를 판별한다"
               (onedev.kr, papers/87); sections "어떻게 동작하나" (probe),
               "무엇과 다른가" (inference procedure: gate, retrieval,
               block-triangular mask, longest verified continuation).
  [SD-anatomy] "LLM 투기적 디코딩(Speculative Decoding) 해부: 작은 드래프트 모델의
               선행 추측과 리젝션 샘플링(Rejection Sampling) 무손실 병렬 검증 원리"
               (blog.huny.dev); §2 Phase 2-3 (parallel verify, sequential
               accept, bonus token), §3.1 acceptance rule alpha = min(1, p/q),
               §3.2 residual p' = max(0, p-q)/sum, §3.3 lossless identity.
  [SD-lossless] "추측 디코딩은 왜 빨라지면서 답은 바뀌지 않나" (jl917.github.io);
               "2단계 · 일괄 검증(Verify)" (match -> accept, first mismatch ->
               truncate, the target generates from there).

Readings taken where the pages are silent or garbled (each is also listed in
the design notes):
  * the probe fires when sigma(w.h) >= tau ("τ 이상" = at least tau);
  * w.h is summed exactly in fixed point: each product h_i*w_i is exact in fp64,
    truncated toward zero at 2^-32 and summed as an integer; the decision is
    S >= ceil(logit(tau) * 2^32), which equals sigma(S*2^-32) >= tau;
  * an earlier occurrence of the kappa-gram may overlap the current one; its end
    j ranges over kappa-1 <= j <= n-2; retrieval ranks by j, largest first, and
    truncates a continuation at the current token: len = min(D, n-1-j);
  * token d of a block is checked against the target row that predicts it:
    row 0 (the current position, shared by every block) for d = 1, else the row
    at the block's token d-1; the bonus / stop row after a tokens is the row at
    token a of the block (row 0 when a = 0);
  * copy candidates are deterministic drafts: q is one-hot on the candidate;
  * the accept test is the exact real comparison u*q(x) < p(x) (both fp32,
    compared as fp64 products, which are exact);
  * the final draw uses integer weights P_i = floor(p_i 2^40) (and Q_i likewise,
    one-hot Q = 2^40), residual weight max(0, P_i - Q_i), bonus weight P_i,
    threshold T = floor(floor(u 2^24) * S / 2^24), token = smallest i whose
    prefix sum exceeds T; if the residual sums to 0 the bonus weights are used;
  * the longest accepted run wins; ties go to the lowest block index (the most
    recent copy candidate; the chain block is last); with no block at all the
    step emits one token drawn from row 0 (an ordinary decode step);
  * temperature 1, no top-k/top-p; greedy mode takes the argmax of the row as
    given (lowest index on ties).
"""
from __future__ import annotations

import math

import numpy as np

FIX_SCORE = 32          # probe products are fixed point at 2^-32
FIX_PROB = 40           # probability weights are fixed point at 2^-40
U_BITS = 24             # uniforms are quantised to 2^-24


# ---------------------------------------------------------------------------
# dtype helpers
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an fp32 word: widen exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_to_f64(x)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# a1: probe gate  [SwitchSD "어떻게 동작하나": p(j) = sigma(w^T H_j);
#                  "무엇과 다른가": copy path needs score >= tau]
# ---------------------------------------------------------------------------
def probe_threshold_fixed(tau: float):
    """Integer threshold T with  S >= T  <=>  sigma(S * 2^-32) >= tau.

    Returns None when the probe always fires (tau <= 0) and the string 'never'
    when it never fires (tau >= 1)."""
    t = float(np.float32(tau))
    if t <= 0.0:
        return None
    if t >= 1.0:
        return "never"
    return math.ceil(math.log(t / (1.0 - t)) * 2.0 ** FIX_SCORE)


def probe_fixed_sum(h: np.ndarray, h_dtype: str, w: np.ndarray) -> np.ndarray:
    """S_b = sum_i trunc(h_bi * w_i * 2^32) as int64; every product is exact in fp64."""
    h64 = to_f64(h, h_dtype)
    w64 = np.asarray(w, dtype=np.float32).astype(np.float64)
    prod = h64 * w64[None, :]
    fixed = np.trunc(prod * 2.0 ** FIX_SCORE).astype(np.int64)
    return fixed.sum(axis=1, dtype=np.int64)


def probe_gate(h, h_dtype, w, tau):
    """Returns (score, probe_on, S): score = sigma(S 2^-32), probe_on = score >= tau."""
    S = probe_fixed_sum(h, h_dtype, w)
    s = S.astype(np.float64) * 2.0 ** -FIX_SCORE
    score = 1.0 / (1.0 + np.exp(-s))
    T = probe_threshold_fixed(tau)
    if T is None:
        on = np.ones(len(S), dtype=bool)
    elif T == "never":
        on = np.zeros(len(S), dtype=bool)
    else:
        on = np.array([int(v) >= T for v in S], dtype=bool)
    return score, on, S


# ---------------------------------------------------------------------------
# a2: kappa-gram structural check  [SwitchSD "무엇과 다른가": the kappa-gram
#     (kappa = 5) ending at the current token must occur earlier in the context]
# ---------------------------------------------------------------------------
def kgram_match_ends(row: np.ndarray, n: int, kappa: int) -> np.ndarray:
    """All j with kappa-1 <= j <= n-2 and row[j-kappa+1 .. j] == row[n-kappa .. n-1],
    largest j first."""
    if kappa < 1 or n < kappa + 1:
        return np.zeros(0, dtype=np.int64)
    row = np.asarray(row[:n])
    g = row[n - kappa:n]
    j = np.arange(kappa - 1, n - 1)
    eq = np.ones(len(j), dtype=bool)
    for i in range(kappa):
        eq &= row[j - (kappa - 1) + i] == g[i]
    return j[eq][::-1].astype(np.int64)


def gate_match(ctx, ctx_len, h, h_dtype, w, tau, kappa):
    """gate_b = probe_on_b AND (the kappa-gram has an earlier occurrence).
    last_match_end_b = the largest such j, or -1 (reported whether or not the probe fires)."""
    score, probe_on, _ = probe_gate(h, h_dtype, w, tau)
    B = len(ctx_len)
    last = np.full(B, -1, dtype=np.int32)
    for b in range(B):
        js = kgram_match_ends(ctx[b], int(ctx_len[b]), kappa)
        if len(js):
            last[b] = js[0]
    gate = probe_on & (last >= 0)
    return score, probe_on, gate.astype(np.int32), last


# ---------------------------------------------------------------------------
# a3: retrieval  [SwitchSD "무엇과 다른가": up to W continuations of length D,
#     most recent first]; a9 chain block [SwitchSD: otherwise delegate to the
#     draft model; SD-anatomy §2 Phase 1: the draft proposes K tokens]
# ---------------------------------------------------------------------------
def num_blocks(W: int, chain_policy: int) -> int:
    return W + (1 if chain_policy else 0)


def retrieve(ctx, ctx_len, gate, kappa, W, D, K, chain_policy, chain_tok):
    """Candidate blocks per sequence.

    Blocks 0..W-1 are copy candidates (recency order); block W, present when
    chain_policy != 0, holds the K draft tokens: when the gate is off
    (chain_policy 1) or always (chain_policy 2).
    Returns blk_tok [B][NB][Dmax] (-1 padded), blk_len [B][NB], n_cand [B]."""
    B = len(ctx_len)
    NB = num_blocks(W, chain_policy)
    Dmax = max(D, K) if chain_policy else D
    blk_tok = np.full((B, NB, Dmax), -1, dtype=np.int32)
    blk_len = np.zeros((B, NB), dtype=np.int32)
    n_cand = np.zeros(B, dtype=np.int32)
    for b in range(B):
        n = int(ctx_len[b])
        if gate[b]:
            js = kgram_match_ends(ctx[b], n, kappa)[:W]
            for k, j in enumerate(js):
                L = min(D, n - 1 - int(j))
                blk_tok[b, k, :L] = ctx[b, j + 1:j + 1 + L]
                blk_len[b, k] = L
            n_cand[b] = len(js)
        if chain_policy == 2 or (chain_policy == 1 and not gate[b]):
            blk_tok[b, W, :K] = chain_tok[b, :K]
            blk_len[b, W] = K
    return blk_tok, blk_len, n_cand


# ---------------------------------------------------------------------------
# a4 + a5: verification attention  [SwitchSD "무엇과 다른가": one target pass
#     for all candidates under a block-triangular mask: a candidate token sees
#     the whole prefix and the earlier tokens of its own candidate, never
#     another candidate; SD-anatomy §2 Phase 2: causal mask for a chain]
# ---------------------------------------------------------------------------
def allowed_keys(P: int, k: int, d: int, Dmax: int):
    """Key set of token d (1-based) of block k: prefix 0..P-1 and the block's own
    slots k*Dmax + 0 .. k*Dmax + d-1 (itself included)."""
    return np.arange(P), np.arange(k * Dmax, k * Dmax + d)


def verify_attention(q, k_cache, v_cache, k_cand, v_cand, prefix_len, blk_len,
                     Dmax, dtype, slots=None):
    """o = sum_j softmax_j(q.k_j / sqrt(dh)) v_j over each token's allowed keys, fp64.

    q [B][NT][Hq][dh]; k_cache/v_cache [B][Hkv][P_max][dh]; k_cand/v_cand
    [B][NT][Hkv][dh]. q-head h reads kv-head h // (Hq/Hkv).
    slots: optional list of (b, t) to evaluate; default: every present token.
    Returns {(b, t): array [Hq][dh]} in fp64."""
    B, NT, Hq, dh = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(dh)
    if slots is None:
        slots = [(b, k * Dmax + d - 1)
                 for b in range(B) for k in range(blk_len.shape[1])
                 for d in range(1, int(blk_len[b, k]) + 1)]
    out = {}
    for (b, t) in slots:
        k, d = t // Dmax, t % Dmax + 1
        assert d <= blk_len[b, k], "slot is not a present token"
        P = int(prefix_len[b])
        pre, own = allowed_keys(P, k, d, Dmax)
        o = np.empty((Hq, dh))
        for kvh in range(Hkv):
            keys = np.concatenate([to_f64(k_cache[b, kvh, pre], dtype),
                                   to_f64(k_cand[b, own, kvh], dtype)], axis=0)
            vals = np.concatenate([to_f64(v_cache[b, kvh, pre], dtype),
                                   to_f64(v_cand[b, own, kvh], dtype)], axis=0)
            qh = to_f64(q[b, t, kvh * G:(kvh + 1) * G], dtype)      # [G][dh]
            s = qh @ keys.T * scale                                  # [G][nkeys]
            s -= s.max(axis=1, keepdims=True)
            e = np.exp(s)
            o[kvh * G:(kvh + 1) * G] = (e / e.sum(axis=1, keepdims=True)) @ vals
        out[(b, t)] = o
    return out


PAGE = 128              # tokens per page of a paged prefix cache


def gather_pages(pages, block_table, P_max):
    """The contiguous cache [B][Hkv][P_max][dh] that a paged one stands for: key
    position p of sequence b is row p % PAGE of page block_table[b][p // PAGE]
    (pages [num_pages][Hkv][PAGE][dh]; SD-anatomy §6 names a PagedAttention pool)."""
    B = block_table.shape[0]
    num_pages, Hkv, page, dh = pages.shape
    assert page == PAGE
    out = np.zeros((B, Hkv, P_max, dh), dtype=pages.dtype)
    for b in range(B):
        for p in range(P_max):
            pg = int(block_table[b, p // PAGE])
            if 0 <= pg < num_pages:
                out[b, :, p, :] = pages[pg, :, p % PAGE, :]
    return out


def verify_attention_paged(q, k_pages, v_pages, block_table, k_cand, v_cand, prefix_len, blk_len,
                           Dmax, dtype, slots=None):
    """verify_attention over a paged prefix cache (see gather_pages)."""
    P_max = PAGE * block_table.shape[1]
    return verify_attention(q, gather_pages(k_pages, block_table, P_max), gather_pages(v_pages, block_table, P_max),
                            k_cand, v_cand, prefix_len, blk_len, Dmax, dtype, slots)


# ---------------------------------------------------------------------------
# a6: vocabulary rows  [SD-anatomy §2 Phase 2: the target yields a next-token
#     distribution at every verified position; §3: p and q are full-vocab
#     distributions]
# ---------------------------------------------------------------------------
def softmax_f64(logits: np.ndarray) -> np.ndarray:
    """p_i = exp(l_i - max l) / sum_j exp(l_j - max l), fp64, along the last axis."""
    x = np.asarray(logits, dtype=np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def row_probs(rows: np.ndarray, kind: str) -> np.ndarray:
    """fp32 probabilities of rows given as 'logits_f32', 'logits_bf16' or 'probs_f32'."""
    if kind == "probs_f32":
        return np.asarray(rows, dtype=np.float32)
    vals = bf16_to_f64(rows) if kind == "logits_bf16" else np.asarray(rows, np.float32).astype(np.float64)
    return softmax_f64(vals).astype(np.float32)


def row_values(rows: np.ndarray, kind: str) -> np.ndarray:
    """The row as given, widened to fp64 (what greedy takes the argmax of)."""
    if kind == "logits_bf16":
        return bf16_to_f64(rows)
    return np.asarray(rows, dtype=np.float32).astype(np.float64)


def first_argmax(x: np.ndarray) -> np.ndarray:
    """Index of the maximum along the last axis, lowest index on ties."""
    return np.argmax(x, axis=-1)


# ---------------------------------------------------------------------------
# a7: acceptance test  [SD-anatomy §3.1: alpha(x) = min(1, p(x)/q(x)); p >= q
#     accepts outright, else accept with probability p/q; read as u*q < p]
# ---------------------------------------------------------------------------
def accept_test(u, q_x, p_x):
    """Exact real comparison u*q(x) < p(x); fp32*fp32 is exact in fp64."""
    u = np.asarray(u, np.float32).astype(np.float64)
    return u * np.asarray(q_x, np.float32).astype(np.float64) < np.asarray(p_x, np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# a8: final token  [SD-anatomy §3.2 residual max(0, p - q) normalised;
#     §2 Phase 3 bonus token drawn from the next target distribution when all
#     drafts are accepted; §3.3 lossless identity]
# ---------------------------------------------------------------------------
def prob_weights(p32: np.ndarray) -> np.ndarray:
    """P_i = floor(p_i * 2^40), exact in int64 for fp32 p in [0, 1]."""
    return np.floor(np.asarray(p32, np.float32).astype(np.float64) * 2.0 ** FIX_PROB).astype(np.int64)


def residual_weights(P: np.ndarray, Q: np.ndarray) -> np.ndarray:
    """max(0, P_i - Q_i): the un-normalised residual of §3.2 in integer weights."""
    return np.maximum(0, P - Q)


def draw_index(weights: np.ndarray, u: float) -> int:
    """Inverse CDF on integer weights: T = floor(floor(u 2^24) * S / 2^24);
    return the smallest i with sum_{j<=i} W_j > T."""
    S = int(np.sum(weights, dtype=np.int64))
    assert S > 0
    U = int(math.floor(float(np.float32(u)) * 2.0 ** U_BITS))
    T = (U * S) >> U_BITS
    C = np.cumsum(weights, dtype=np.int64)
    return int(np.searchsorted(C, T, side="right"))


def verify_step_accept(mode, kind, tgt, drf, blk_tok, blk_len, W, chain_policy,
                       u_acc, u_fin):
    """Acceptance and selection for every sequence.

    tgt [B][1+NB*Dmax][V] target rows (logits or probabilities per `kind`);
    drf [B][K][V] draft rows of the chain block (same kind) or None;
    blk_tok [B][NB][Dmax], blk_len [B][NB]; u_acc [B][NB][Dmax]; u_fin [B].
    Returns dict(acc_len [B][NB], best_blk [B], n_out [B], out_tok [B][Dmax+1])."""
    B, NB, Dmax = blk_tok.shape
    acc_len = np.zeros((B, NB), dtype=np.int32)
    best = np.full(B, -1, dtype=np.int32)
    n_out = np.zeros(B, dtype=np.int32)
    out_tok = np.full((B, Dmax + 1), -1, dtype=np.int32)
    chain_blk = W if chain_policy else -1

    def trow(k, d):                      # target row that predicts token d+1 of block k
        return 0 if d == 0 else 1 + k * Dmax + (d - 1)

    for b in range(B):
        cache_p, cache_q = {}, {}

        def p_row(r):
            if r not in cache_p:
                cache_p[r] = row_probs(tgt[b, r], kind)
            return cache_p[r]

        def q_row(i):
            if i not in cache_q:
                cache_q[i] = row_probs(drf[b, i], kind)
            return cache_q[i]

        # a7: per block, the leading run of accepted tokens
        for k in range(NB):
            L = int(blk_len[b, k])
            a = 0
            for d in range(1, L + 1):
                x = int(blk_tok[b, k, d - 1])
                r = trow(k, d - 1)
                if mode == "greedy":
                    ok = x == int(first_argmax(row_values(tgt[b, r], kind)))
                else:
                    qx = q_row(d - 1)[x] if k == chain_blk else np.float32(1.0)
                    ok = bool(accept_test(u_acc[b, k, d - 1], qx, p_row(r)[x]))
                if not ok:
                    break
                a += 1
            acc_len[b, k] = a

        # a8: longest accepted run; ties -> lowest block index
        present = [k for k in range(NB) if blk_len[b, k] > 0]
        if present:
            ks = max(present, key=lambda k: (int(acc_len[b, k]), -k))
            a, L = int(acc_len[b, ks]), int(blk_len[b, ks])
        else:
            ks, a, L = -1, 0, 0
        best[b] = ks
        if a:
            out_tok[b, :a] = blk_tok[b, ks, :a]
        r_stop = trow(ks, a)
        if mode == "greedy":
            fin = int(first_argmax(row_values(tgt[b, r_stop], kind)))
        else:
            P = prob_weights(p_row(r_stop))
            if a < L:                    # rejected at token a+1: residual
                x_rej = int(blk_tok[b, ks, a])
                if ks == chain_blk:
                    Q = prob_weights(q_row(a))
                else:
                    Q = np.zeros_like(P)
                    Q[x_rej] = 1 << FIX_PROB
                Wt = residual_weights(P, Q)
                if int(Wt.sum(dtype=np.int64)) == 0:
                    Wt = P
            else:                        # all accepted: bonus from the stop row
                Wt = P
            fin = draw_index(Wt, u_fin[b])
        out_tok[b, a] = fin
        n_out[b] = a + 1
    return dict(acc_len=acc_len, best_blk=best, n_out=n_out, out_tok=out_tok)


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------
def verify_step(inp: dict, wl, mode=None, kind=None, attention_slots="all"):
    """Gate -> retrieval -> verification attention -> acceptance, on one batch.

    inp: arrays as produced by the workload generator; wl: its workload
    description (only sizes and flags are read). attention_slots: 'all', None
    (skip attention) or an explicit list of (b, t)."""
    mode = mode or wl.mode
    if kind is None:
        kind = "logits_bf16" if wl.logit_dtype == "bf16" else "logits_f32"
    score, probe_on, gate, last = gate_match(inp["ctx"], inp["ctx_len"], inp["h"], wl.h_dtype,
                                             inp["w"], wl.tau, wl.kappa)
    blk_tok, blk_len, n_cand = retrieve(inp["ctx"], inp["ctx_len"], gate, wl.kappa, wl.W, wl.D,
                                        wl.K, wl.chain_policy, inp["chain_tok"])
    res = dict(score=score, probe_on=probe_on, gate=gate, last_match_end=last,
               blk_tok=blk_tok, blk_len=blk_len, n_cand=n_cand)
    if attention_slots is not None and "q" in inp:
        res["attn"] = verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"],
                                       inp["v_cand"], inp["prefix_len"], blk_len, wl.Dmax,
                                       wl.kv_dtype,
                                       None if attention_slots == "all" else attention_slots)
    if "tgt" in inp:
        res.update(verify_step_accept(mode, kind, inp["tgt"], inp.get("drf"), blk_tok, blk_len,
                                      wl.W, wl.chain_policy, inp["u_acc"], inp["u_fin"]))
    return res


# ---------------------------------------------------------------------------
# after the step: committing the accepted candidates' keys and values
#     [SD-anatomy §6, "KV 캐시 롤백(Rollback) 및 페이징 메모리 오버헤드 관리": the
#     target holds the candidates' K/V to verify them, and what follows the first
#     rejection must be released.] Here the candidates' K/V sit beside the cache, so
#     the accepted ones are appended to it and the rejected ones never enter it.
# ---------------------------------------------------------------------------
def commit_kv(k_cache, v_cache, k_cand, v_cand, prefix_len, best_blk, n_out, Dmax):
    """Append the accepted tokens' keys and values to the prefix cache.

    For sequence b with chosen block k = best_blk[b] >= 0, the a = n_out[b] - 1
    accepted tokens (the emitted tokens minus the final one, whose K/V the next
    step computes) occupy candidate slots k*Dmax .. k*Dmax + a - 1; their rows of
    every kv head become cache rows P_b .. P_b + a - 1 and prefix_len[b] grows by a.
    A sequence whose cache has no room (P_b + a > P_max) is left unchanged and
    flagged. Layouts as in verify_attention. Returns (k_cache', v_cache',
    prefix_len', ok[B])."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    pl = np.array(prefix_len, dtype=np.int32, copy=True)
    B, Hkv, P_max = kc.shape[:3]
    ok = np.ones(B, dtype=bool)
    for b in range(B):
        k = int(best_blk[b])
        a = int(n_out[b]) - 1 if k >= 0 else 0
        if a <= 0:
            continue
        P = int(pl[b])
        if P + a > P_max:
            ok[b] = False
            continue
        for i in range(a):
            slot = k * Dmax + i
            kc[b, :, P + i, :] = k_cand[b, slot, :, :]
            vc[b, :, P + i, :] = v_cand[b, slot, :, :]
        pl[b] = P + a
    return kc, vc, pl, ok


# ---------------------------------------------------------------------------
# speculation tax  [SwitchSD "무엇인가": a copy draft opened by an accidental surface
#     repetition is verified and accepted for 0 tokens, so the step pays the
#     verification for nothing; "어떻게 쓰나" reports how often copying fires and the
#     accepted length it gets]
# ---------------------------------------------------------------------------
def copy_stats(gate, n_cand, acc_len, W):
    """Counts over a batch: copy attempts (gate on and at least one copy candidate), taxed
    attempts (no copy block accepted a token), accepted copy tokens (over attempts, the
    longest accepted run among the W copy blocks), sequences. Returns int64 [4]."""
    attempts = taxed = tokens = 0
    for b in range(len(gate)):
        if not (int(gate[b]) != 0 and int(n_cand[b]) > 0):
            continue
        run = int(np.max(acc_len[b, :W])) if W > 0 else 0
        attempts += 1
        taxed += 1 if run == 0 else 0
        tokens += run
    return np.array([attempts, taxed, tokens, len(gate)], dtype=np.int64)
