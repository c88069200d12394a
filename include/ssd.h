/*
 * ssd.h — C ABI of the GB300 speculate-and-verify step (SwitchSD copy mode +
 * chain drafts), implemented by libssd.so (hand-written CUDA for sm_103a).
 *
 * The step, per sequence of a batch:
 *   ssd_gate_match   probe score sigma(w.h) >= tau AND an earlier occurrence of
 *                    the kappa-gram ending at the current token
 *                    [SwitchSD page, "어떻게 동작하나" (probe p = sigma(w^T H)) and
 *                     "무엇과 다른가" (copy path needs both conditions)]
 *   ssd_retrieve     up to W continuations of length D, most recent first,
 *                    plus an optional chain-draft block of K tokens
 *                    [SwitchSD page, "무엇과 다른가"]
 *   ssd_verify_attn  one attention pass for every candidate token under the
 *                    block-triangular mask: the whole prefix plus the earlier
 *                    tokens of its own block, never another block
 *                    [SwitchSD page, "무엇과 다른가"; Speculative Decoding 해부
 *                     page, §2 Phase 2 (one parallel target pass)]
 *   ssd_accept       full-vocabulary rows, greedy or rejection-sampling
 *                    acceptance (accept if u*q(x) < p(x)), residual
 *                    max(0, p-q) or bonus draw, longest accepted block wins
 *                    [Speculative Decoding 해부 page, §2 Phase 3, §3.1, §3.2;
 *                     SwitchSD page, "무엇과 다른가" (longest verified
 *                     continuation); 추측 디코딩은 왜… page, "2단계 · 일괄 검증"]
 *
 * Around the step: ssd_gate_retrieve (gate and retrieval in one launch),
 * ssd_commit_kv (append the accepted candidates' keys and values to the cache),
 * ssd_copy_stats (copy attempts and speculation tax), ssd_lowrank_head (the
 * SlimSpec low-rank draft LM head), ssd_accept_static (ssd_accept without a
 * caller workspace) with ssd_read_static_error, and the diagnostics
 * ssd_read_device_error, ssd_status_string, ssd_version, ssd_launch_count,
 * ssd_profile_kernel, ssd_selftest_wait, and the measurement tool ssd_read_probe.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless a comment says otherwise. The caller
 *     owns every buffer; the library allocates nothing and keeps no state
 *     between calls beyond per-process caches filled on first use (kernel
 *     attributes, occupancy queries), the launch counter and profiling hook,
 *     and the fixed scratch array of ssd_accept_static (described there).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Every call is
 *     asynchronous on that stream and never synchronises, except
 *     ssd_read_device_error and ssd_read_static_error, which are documented
 *     as synchronous.
 *   - Return value: SSD_OK or a negative ssd_status. Arguments are validated on
 *     the host before any launch; on an error nothing is launched and no output
 *     is written. SSD_ERR_CUDA means a launch failed (cudaGetLastError).
 *   - Layouts are dense row-major with the shapes given below.
 *     NB = number of blocks, Dmax = slots per block, NT = NB * Dmax.
 *   - Calls are safe from several host threads on distinct streams with
 *     distinct output and workspace buffers.
 *   - Stream order: most kernels are launched with programmatic dependent
 *     launch, so such a kernel may start before the kernel issued before it on
 *     the same stream has completed. It completes
 *     only after that kernel, it writes nothing that kernel may still read or
 *     write, and results are those of strictly ordered calls. It may read the
 *     caller's inputs early (the logits in ssd_accept's early_rows mode; with
 *     all_rows, everything ssd_verify_attn reads). The retrieval kernels
 *     (ssd_gate_match, ssd_retrieve, ssd_gate_retrieve) are ordinary launches:
 *     they start only after everything before them on the stream, so a step
 *     that begins with them sees every earlier write.
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
enum {
  SSD_OK = 0,
  SSD_ERR_INVALID = -1,      /* bad pointer, size or enum value               */
  SSD_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. head dim 96)  */
  SSD_ERR_CUDA = -3,         /* a CUDA launch or query failed                 */
  SSD_ERR_WORKSPACE = -4,    /* workspace NULL, misaligned or too small       */
  SSD_ERR_TIMEOUT = -5,      /* a device-side wait gave up (device error word) */
  SSD_ERR_DEVICE = -6        /* a device-side check failed (device error word) */
};

/* element types */
enum { SSD_F32 = 0, SSD_BF16 = 1 };
/* what the vocabulary rows hold */
enum { SSD_LOGITS_F32 = 0, SSD_LOGITS_BF16 = 1, SSD_PROBS_F32 = 2 };
/* acceptance rule */
enum { SSD_GREEDY = 0, SSD_SAMPLE = 1 };
/* when the chain-draft block is present */
enum { SSD_CHAIN_NONE = 0, SSD_CHAIN_WHEN_GATE_OFF = 1, SSD_CHAIN_ALWAYS = 2 };

/* Human-readable name of a status code (static string, never NULL). */
const char* ssd_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int ssd_version(void);

/* Number of kernels this process has launched through the library (host
 * counter, all threads). Kernels replayed from a captured CUDA graph are not
 * counted again. */
uint64_t ssd_launch_count(void);

/*
 * ssd_selftest_wait — exercise the device-side failure detection.
 *
 * The pages have no counterpart; this tests the library's bounded waits without
 * faulting or hanging the GPU. One CTA initialises an mbarrier in shared memory
 * and waits on it with the same bounded wait the kernels use. With arrive != 0
 * it arrives first and the wait completes; with arrive == 0 nothing arrives, so
 * the wait gives up after limit_clocks SM clocks, records SSD_ERR_TIMEOUT in the
 * header of `ws` (read back by ssd_read_device_error) and the kernel returns
 * normally, leaving the context usable.
 *   ws: device workspace of at least 256 bytes, 256-byte aligned (its header
 *       must hold SSD_OK beforehand for the error to be recorded);
 *   1 <= limit_clocks <= 2^32.
 * Errors: SSD_ERR_INVALID, SSD_ERR_WORKSPACE, SSD_ERR_CUDA (launch failure).
 */
int ssd_selftest_wait(void* ws, int arrive, uint64_t limit_clocks, void* stream);

/*
 * ssd_gate_match — probe gate and kappa-gram check.
 *
 * For each sequence b (n = ctx_len[b], the current token is ctx[b][n-1]):
 *   S_b        = sum_i trunc(h[b][i] * w[i] * 2^32)  (each product exact in
 *                fp64, summed as int64, so the result does not depend on the
 *                summation order)
 *   score[b]   = sigma(S_b * 2^-32)                   (fp32, informative)
 *   probe_on   = S_b >= ceil(logit(tau) * 2^32), i.e. sigma >= tau; always on
 *                for tau <= 0, never on for tau >= 1
 *   last_match_end[b] = the largest j with kappa-1 <= j <= n-2 and
 *                ctx[b][j-kappa+1 .. j] == ctx[b][n-kappa .. n-1], else -1
 *                (reported whether or not the probe fires)
 *   gate[b]    = probe_on AND last_match_end[b] >= 0
 * Arguments
 *   ctx [B][ctx_stride] int32, ctx_len [B] int32 (0 <= ctx_len <= ctx_stride)
 *   h   [B][h_stride] elements of h_dtype (SSD_F32 or SSD_BF16), first d used
 *   w   [d] fp32
 *   1 <= kappa <= 64;  B >= 0 (B == 0 launches nothing);  d >= 1
 *   score [B] fp32, gate [B] int32, last_match_end [B] int32: outputs;
 *   probe_on [B] int32: optional output (may be NULL)
 * Requires |h_i * w_i| < 2^31 and |S_b| < 2^63 (not checked).
 */
int ssd_gate_match(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                   const void* h, int h_dtype, int64_t h_stride, const float* w, int d,
                   float tau, int kappa,
                   float* score, int32_t* gate, int32_t* last_match_end, int32_t* probe_on,
                   void* stream);

/*
 * ssd_retrieve — copy candidates, most recent first, plus the chain block.
 *
 * Block layout per sequence: NB = W + (chain_policy != SSD_CHAIN_NONE),
 * Dmax = chain_policy ? max(D, K) : D. Blocks 0..W-1 are copy candidates:
 * if gate[b], the k-th largest match end j_k (same definition as
 * ssd_gate_match) gives blk_tok[b][k][0..len-1] = ctx[b][j_k+1 ..] with
 * len = min(D, n-1-j_k); up to W of them (n_cand[b] <= W). Block W (if
 * present) is the chain draft chain_tok[b][0..K-1], present when the gate is
 * off (SSD_CHAIN_WHEN_GATE_OFF) or always (SSD_CHAIN_ALWAYS). Absent blocks
 * and unused slots have length 0 and tokens -1.
 * Arguments
 *   ctx, ctx_stride, ctx_len, B, kappa: as for ssd_gate_match
 *   gate [B] int32 (from ssd_gate_match)
 *   last_match_end [B] int32 or NULL: accepted for symmetry with
 *     ssd_gate_match and not read (the scan starts at the current token; the
 *     most recent matches lie in its first staged chunk)
 *   1 <= W <= 64, 1 <= D <= 256, 0 <= K <= 256 (K >= 1 if chain_policy != 0)
 *   chain_tok [B][K] int32, may be NULL when chain_policy == SSD_CHAIN_NONE
 *   blk_tok [B][NB][Dmax], blk_len [B][NB], n_cand [B]: int32 outputs
 */
int ssd_retrieve(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                 const int32_t* gate, const int32_t* last_match_end,
                 int kappa, int W, int D, int K, int chain_policy, const int32_t* chain_tok,
                 int32_t* blk_tok, int32_t* blk_len, int32_t* n_cand, void* stream);

/*
 * ssd_gate_retrieve — ssd_gate_match and ssd_retrieve fused into one launch
 * (one pass over the context per sequence); same definitions, arguments and
 * outputs as the two calls made in sequence. probe_on may be NULL.
 */
int ssd_gate_retrieve(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                      const void* h, int h_dtype, int64_t h_stride, const float* w, int d,
                      float tau, int kappa, int W, int D, int K, int chain_policy,
                      const int32_t* chain_tok,
                      float* score, int32_t* gate, int32_t* last_match_end, int32_t* probe_on,
                      int32_t* blk_tok, int32_t* blk_len, int32_t* n_cand, void* stream);

/*
 * ssd_verify_attn — attention of every candidate token over its allowed keys.
 *
 * Token d (1-based) of block k of sequence b sits in slot t = k*Dmax + d-1 and
 * is present iff d <= blk_len[b][k]. For each present token and q-head h
 * (kv-head h / (Hq/Hkv)):
 *   out = sum_j softmax_j(scale * q.k_j) v_j over the keys
 *         {k_cache[b][kvh][0 .. prefix_len[b]-1]} U {k_cand[b][k*Dmax + 0 .. t][kvh]}
 * Rows of absent tokens are not written.
 * Layouts (elements of `dtype`; out has the same dtype):
 *   q, out          [B][NT][Hq][dh]
 *   k_cache,v_cache [B][Hkv][P_max][dh]      (prefix_len[b] <= P_max)
 *   k_cand,v_cand   [B][NT][Hkv][dh]
 *   prefix_len [B] int32, blk_len [B][NB] int32
 * Supported: dh in {64, 128}; Hq % Hkv == 0; 1 <= Dmax <= 256.
 * scale == 0 selects 1/sqrt(dh). Accumulation is fp32 whatever `dtype`.
 * out_dtype is `dtype` or SSD_F32 (an fp32 output for bf16 inputs).
 * Paged prefix cache (block_table != NULL; bf16, dh 128 only, else
 * SSD_ERR_UNSUPPORTED): the Speculative Decoding 해부 page's §6 names a
 * PagedAttention pool for the cache. k_cache, v_cache are then pages of 128
 * tokens, [num_pages][Hkv][128][dh], and key position p of sequence b is row
 * p % 128 of page block_table[b][p / 128] (block_table [B][pages_per_seq] int32,
 * prefix_len[b] <= 128 * pages_per_seq; pages may be shared by sequences). A page
 * index outside [0, num_pages) records SSD_ERR_DEVICE and reads page 0. P_max is
 * then unused.
 * skip_absent (0, 1 or 2; tensor-core path only, ignored by the fp32 /
 * head-dim-64 pass): 1 makes every CTA first wait for the kernel before it on
 * the stream (the one whose outputs include blk_len, or a later one) and then
 * skip a tile of 128 packed rows in which no token is present, e.g. the
 * copy-block rows of a sequence whose gate is off. Outputs are identical; the
 * attention then no longer overlaps the tail of that preceding kernel, so it
 * pays off only when many candidate slots are empty. 2 skips the same tiles
 * without that wait: the caller guarantees that blk_len is complete when the
 * call's kernel launches, i.e. the kernel that wrote it has completed before
 * the kernel issued just before this call lets its dependents launch (true
 * after ssd_accept, whose finish kernel launches only once the retrieval has
 * completed, or after an event wait); the attention then runs beside the
 * kernel before it and waits for it only before its grid ends. 0: every tile
 * is computed, blk_len is read only before the merge.
 * all_rows (0 or 1): 1 writes the row of every slot t, present or not, as the
 * attention of its q over the prefix and the slots k*Dmax .. t of its block
 * (what the row of a present token holds), and never reads blk_len (it may be
 * NULL), so the call depends on no earlier kernel's output and may run on
 * another stream beside the retrieval. On its own stream it still completes
 * after the kernel issued before it (it waits for that kernel only after its
 * rows are written). Requires skip_absent == 0.
 * max_ctas (>= 0): 0 lets the call use the whole GPU; n > 0 sizes the
 * tensor-core grid to at most max(n, clusters of one CTA) CTAs, one per SM, so
 * that a kernel on another stream can hold the remaining SMs at the same time.
 * Workspace: ssd_verify_attn_workspace_size(a) bytes, 256-byte aligned: 256
 * bytes where the tensor-core path applies (bf16, dh 128, 16-byte aligned
 * tensors, a GPU of compute capability 10.3), else room for every split's
 * partial rows; the size is that of the path the same arguments (pointers
 * included) take on the current device. Its
 * contents need no initialisation for the results. Device-side errors are recorded
 * in its first word, which keeps whatever it held before: zero the header (its first
 * 256 bytes) once after allocating it, or read it once with ssd_read_device_error,
 * before relying on that word.
 */
typedef struct {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_cand;
  const void* v_cand;
  void* out;
  const int32_t* prefix_len;
  const int32_t* blk_len;
  int dtype;
  int B, NB, Dmax, Hq, Hkv, dh;
  int64_t P_max;
  float scale;
  int out_dtype;
  const int32_t* block_table;
  int pages_per_seq;
  int64_t num_pages;
  int skip_absent;
  int all_rows;
  int max_ctas;
} ssd_attn_args;

size_t ssd_verify_attn_workspace_size(const ssd_attn_args* a);
int ssd_verify_attn(const ssd_attn_args* a, void* ws, size_t ws_bytes, void* stream);

/*
 * ssd_accept — vocabulary rows, acceptance, choice of block, final token.
 *
 * Target row 0 is the current position (it predicts token 1 of every block);
 * row 1 + k*Dmax + (d-1) is the position of token d of block k (it predicts
 * token d+1, or the bonus after d tokens). Draft row i of drf is the draft
 * distribution of chain token i+1.
 *   p = softmax(row) in fp32 (rows given as logits) or the row itself
 *       (SSD_PROBS_F32); q of a copy block is one-hot on its token; q of the
 *       chain block is softmax(drf row).
 *   greedy: token d is accepted iff it equals the argmax of its target row
 *           (lowest index on ties);
 *   sample: accepted iff u_acc[b][k][d-1] * q(x) < p(x), compared exactly.
 *   acc_len[b][k] = leading accepted tokens of block k;
 *   best_blk[b]   = the present block with the largest acc_len, lowest index
 *                   on ties (-1 if no block is present);
 *   out_tok[b][0..a-1] = its accepted tokens; out_tok[b][a] = the final token:
 *     greedy: argmax of the stop row; sample: an inverse-CDF draw with
 *     threshold floor(floor(u_fin 2^24) * S / 2^24) over integer weights
 *     P_i = floor(p_i 2^40): residual max(0, P_i - Q_i) after a rejection (Q
 *     one-hot 2^40 for a copy block), P_i for the bonus when all tokens of the
 *     block were accepted, P_i again if the residual is all zero;
 *   n_out[b] = a + 1; out_tok[b][n_out..Dmax] = -1.
 * Layouts:
 *   tgt [B][1 + NB*Dmax][V], drf [B][K][V] (NULL iff chain_blk < 0), of `kind`
 *   blk_tok [B][NB][Dmax], blk_len [B][NB] (from ssd_retrieve)
 *   u_acc [B][NB][Dmax] fp32, u_fin [B] fp32, uniforms in [0, 1)
 *   acc_len [B][NB], best_blk [B], n_out [B], out_tok [B][Dmax+1]: int32 outputs
 *   probs_out: optional fp32 [B][1 + NB*Dmax][V]; when given, p of every
 *     needed target row is written there (diagnostics; costs a full write)
 *   early_rows: 0 — the row pass waits for the kernel before it on the stream
 *     (the retrieval that wrote blk_len) and reads only the rows a present
 *     token needs; 1 — it starts at once and reads every target row a block
 *     length can reach (all but the chain block's rows at positions K and
 *     beyond) and every draft row when chain_blk >= 0, so that it overlaps the kernel
 *     launched just before it (the retrieval, or an attention launched after
 *     the retrieval); blk_tok and blk_len are read only after that kernel has
 *     completed, and the call's last kernel starts only then. Results are
 *     identical; early_rows = 1 reads rows of absent tokens too (their
 *     contents are never used). With early_rows = 1 the caller guarantees
 *     that tgt and drf are complete before the call is issued (they are read
 *     while the kernel before it on the stream may still run); only blk_tok
 *     and blk_len may come from that kernel. In both modes the workspace is
 *     written only after the kernel before the call on the stream has
 *     completed, so consecutive calls on one stream may share a workspace.
 *   max_ctas (>= 0): 0 sizes the row pass to the whole GPU; n > 0 runs it as at
 *     most n CTAs of one SM each, so that a kernel on another stream can hold
 *     the remaining SMs at the same time.
 * 2 <= V < 2^31; NB*Dmax < 4096;
 * Dmax <= 256; 0 <= chain_blk < NB or chain_blk == -1.
 * Workspace: ssd_accept_workspace_size(a) bytes, 256-byte aligned; its
 * contents need no initialisation for the results (the error word in its first
 * bytes: as for ssd_verify_attn). Calls issued one after another on one
 * stream may share it; calls that overlap on the GPU (other streams) may not.
 */
typedef struct {
  int mode;
  int kind;
  const void* tgt;
  const void* drf;
  int64_t V;
  const int32_t* blk_tok;
  const int32_t* blk_len;
  int B, NB, Dmax, K;
  int chain_blk;
  const float* u_acc;
  const float* u_fin;
  int32_t* acc_len;
  int32_t* best_blk;
  int32_t* n_out;
  int32_t* out_tok;
  float* probs_out;
  int early_rows;
  int max_ctas;
} ssd_accept_args;

size_t ssd_accept_workspace_size(const ssd_accept_args* a);
int ssd_accept(const ssd_accept_args* a, void* ws, size_t ws_bytes, void* stream);

/*
 * ssd_commit_kv — append the accepted tokens' keys and values to the prefix cache.
 *
 * Speculative Decoding 해부 page, §6 "KV 캐시 롤백(Rollback) 및 페이징 메모리
 * 오버헤드 관리": the target holds the candidates' K/V to verify them and what
 * follows the first rejection must be released. Here the candidates' K/V sit
 * beside the cache (k_cand, v_cand), so after ssd_accept the accepted ones are
 * appended and the rejected ones never enter it. For sequence b with chosen block
 * k = best_blk[b] >= 0, the a = n_out[b] - 1 accepted tokens (all emitted tokens
 * but the final one, whose K/V the next step computes) occupy candidate slots
 * k*Dmax .. k*Dmax + a - 1; their rows of every kv head become cache rows
 * prefix_len[b] .. prefix_len[b] + a - 1 and prefix_len[b] grows by a.
 * Layouts (elements of `dtype`, SSD_F32 or SSD_BF16):
 *   k_cache, v_cache [B][Hkv][P_max][dh]   (updated in place)
 *   k_cand, v_cand   [B][NB*Dmax][Hkv][dh]
 *   prefix_len [B] int32 (updated in place); best_blk [B], n_out [B] int32 (from
 *   ssd_accept; read after the kernel before this one on the stream completes)
 * A sequence whose cache has no room (prefix_len + a > P_max) is left unchanged and
 * SSD_ERR_DEVICE is recorded in the workspace header. The regions must not overlap.
 * Workspace: at least 256 bytes, 256-byte aligned (the status header).
 */
typedef struct {
  void* k_cache;
  void* v_cache;
  const void* k_cand;
  const void* v_cand;
  int32_t* prefix_len;
  const int32_t* best_blk;
  const int32_t* n_out;
  int dtype;
  int B, NB, Dmax, Hkv, dh;
  int64_t P_max;
} ssd_commit_args;

int ssd_commit_kv(const ssd_commit_args* a, void* ws, size_t ws_bytes, void* stream);

/*
 * ssd_copy_stats — count copy attempts and the speculation tax over a batch.
 *
 * SwitchSD page, "무엇인가": a copy draft opened by an accidental surface repetition
 * is verified and accepted for 0 tokens, so the step pays the verification for
 * nothing (the speculation tax); "어떻게 쓰나" reports how often copying fires and
 * the accepted length it gets. Adds to counts[4] (int64, device memory, running
 * totals across calls):
 *   counts[0] += sequences with gate[b] != 0 and n_cand[b] > 0 (copy attempts)
 *   counts[1] += those whose W copy blocks all accepted 0 tokens (taxed attempts)
 *   counts[2] += over attempts, the longest accepted run among the copy blocks
 *   counts[3] += B
 * gate, n_cand [B] int32 (from ssd_gate_retrieve / ssd_retrieve); acc_len [B][NB]
 * int32 (from ssd_accept; copy blocks are 0 .. W-1, NB >= W). Read after the
 * kernel before this one on the stream completes. B == 0 launches nothing.
 * Errors: SSD_ERR_INVALID (NULL pointer, W < 0 or NB < W).
 */
int ssd_copy_stats(const int32_t* gate, const int32_t* n_cand, const int32_t* acc_len, int B, int NB, int W,
                   int64_t* counts, void* stream);

/*
 * ssd_lowrank_head — the SlimSpec low-rank draft LM head with its softmax statistics.
 *
 * SlimSpec page ("SlimSpec: Low-Rank Draft LM-Head for Accelerated Speculative
 * Decoding"), "방법론: SlimSpec" / "아키텍처": the drafter's logits are
 * z = W_up (W_down h), W_down [r][d] compressing the hidden state to rank r (such
 * as d/8) and W_up [V][r] projecting it to the whole vocabulary, in place of the
 * full-rank z = W_full h. The draft distribution is q = softmax(z) (Speculative
 * Decoding 해부 page, §3). For each of the M rows of h:
 *   u = W_down h       fp32 accumulation, rounded to bf16 (the operand of the
 *                      second product)
 *   z = W_up u         fp32 accumulation
 *   row_max[m] = max_v z_v;  lse[m] = log sum_v exp(z_v) (natural log), so that
 *   q_v = exp(z_v - lse[m]);  argmax[m] = the lowest v with z_v = row_max[m]
 *   (the greedy draft token);  logits [M][V] (when not NULL) receive z as fp32
 *   (logits_dtype SSD_F32) or bf16 rounded to nearest even (SSD_BF16).
 * Layouts: h [M][d], w_down [r][d], w_up [V][r], bf16, dense row-major, 16-byte
 * aligned. row_max, lse [M] fp32; argmax [M] int32.
 * Limits: 1 <= M <= 64 (larger batches: several calls), d and r multiples of 8,
 * 8 <= r <= 1024, 1 <= V < 2^31 - 128; SSD_ERR_UNSUPPORTED otherwise (or off sm_103).
 * Workspace: ssd_lowrank_head_workspace_size(a) bytes (0 for invalid arguments),
 * 256-byte aligned: the status header, u, and per-CTA partial statistics. Three
 * kernels run on `stream` (down projection, up projection with the statistics,
 * per-row merge); outputs are complete when the last one finishes. A device-side
 * wait that gives up records SSD_ERR_TIMEOUT in the header (ssd_read_device_error).
 */
typedef struct {
  const void* h;
  const void* w_down;
  const void* w_up;
  void* logits;           /* optional [M][V] */
  int logits_dtype;       /* SSD_F32 or SSD_BF16 */
  float* row_max;
  float* lse;
  int32_t* argmax;
  int M, d, r, V;
} ssd_head_args;

size_t ssd_lowrank_head_workspace_size(const ssd_head_args* a);
int ssd_lowrank_head(const ssd_head_args* a, void* ws, size_t ws_bytes, void* stream);

/*
 * ssd_accept_static — ssd_accept without a caller-provided workspace.
 *
 * The pages have no counterpart for this call; it exists for callers that
 * cannot allocate device memory at the point where they run the step: code
 * that runs inside a stream capture or a real-time serving loop where every
 * allocation is forbidden, hosts whose device memory is owned by a separate
 * pool the library cannot draw from, or bindings with no allocator at all.
 * Arguments, outputs and results are those of ssd_accept.
 * Scratch: a fixed 4 MiB array inside the library's device code, present on
 * every GPU that loads the library and held until the process exits. A call
 * whose scratch need (ssd_accept_workspace_size) exceeds 4 MiB returns
 * SSD_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address (and loads
 * the library's device code there); make that first call before any stream
 * capture. The call allocates nothing: no cudaMalloc, cudaFree or other
 * allocating routine.
 * Every call on a device shares the one array and it keeps the previous call's
 * contents (nothing in it needs to start at zero), so calls that overlap on
 * the GPU — on different streams or from different threads — race; serialise
 * them. Calls issued one after another on one stream are serialised (in both
 * early_rows modes). Device-side errors (a candidate token outside [0, V), a
 * block longer than its slots) are recorded in the array's header; read and
 * clear them with ssd_read_static_error.
 */
int ssd_accept_static(const ssd_accept_args* a, void* stream);

/*
 * ssd_read_static_error — SYNCHRONOUS: waits for `stream`, then reads and
 * clears the device error word of ssd_accept_static's fixed scratch on the
 * current device. *out receives SSD_OK or the first error recorded since the
 * last read (SSD_ERR_DEVICE, SSD_ERR_TIMEOUT). Like ssd_accept_static it
 * allocates nothing (one small copy to the host, one to the device when the
 * word was set) and has no counterpart on the pages. `out` is a host pointer.
 * Errors: SSD_ERR_INVALID (out NULL), SSD_ERR_CUDA.
 */
int ssd_read_static_error(void* stream, int32_t* out);

/*
 * ssd_checked_build — 1 for the checked build of the library (libssd_checked.so,
 * compiled with -DSSD_CHECKS=1), 0 for the normal one. The checked build tests every
 * guarded device index (token ids, block lengths, prefix lengths, output offsets,
 * workspace offsets) against the extent it must stay within before the access; a
 * failed test records SSD_ERR_DEVICE in the call's workspace header, when the call has
 * one, and in a check word of the library, and the access is skipped. No counterpart
 * on the pages: a debugging aid for callers and tests.
 */
int ssd_checked_build(void);

/*
 * ssd_read_check_error — SYNCHRONOUS: waits for `stream`, then reads and clears the
 * library's check words (checked build; always SSD_OK in the normal build). *out gets
 * SSD_OK or SSD_ERR_DEVICE. `out` is a host pointer. Errors: SSD_ERR_INVALID, SSD_ERR_CUDA.
 */
int ssd_read_check_error(void* stream, int32_t* out);

/*
 * ssd_read_probe — measurement tool (no counterpart on the pages): reads `bytes`
 * bytes of device memory at `buf` once with plain 16-byte loads (eight in flight
 * per thread, a grid of ctas_per_sm x 256-thread CTAs per SM) and discards them,
 * so that CUDA events around it give the device's read bandwidth for a burst of
 * that size. Writes at most 16 bytes at `sink` (and in practice nothing).
 *   buf, sink: device pointers, 16-byte aligned; bytes a multiple of 16, >= 16;
 *   1 <= ctas_per_sm <= 8.
 * Errors: SSD_ERR_INVALID, SSD_ERR_CUDA.
 */
int ssd_read_probe(const void* buf, size_t bytes, int ctas_per_sm, void* sink, void* stream);

/*
 * ssd_read_device_error — SYNCHRONOUS: waits for `stream`, then reads and
 * clears the device error word at the head of a workspace used by
 * ssd_verify_attn or ssd_accept. *out receives SSD_OK, SSD_ERR_TIMEOUT or
 * SSD_ERR_DEVICE. `ws` is a device pointer; `out` a host pointer.
 */
int ssd_read_device_error(void* ws, void* stream, int32_t* out);

/*
 * ssd_profile_kernel — measurement hook (no counterpart on the pages).
 * From now on every launch of kernel `kernel_id` (SSD_KERNEL_*) is bracketed
 * by cudaEventRecord(start_event) / cudaEventRecord(end_event) on the stream
 * the kernel is launched on (as external event nodes while that stream is
 * being captured into a CUDA graph). Each kernel id has its own pair; calling
 * again replaces it. kernel_id 0 (events ignored) switches every hook off.
 * The events are cudaEvent_t handles owned by the caller and must stay valid
 * while hooked. Process-wide; not thread-safe against concurrent launches.
 */
enum {
  SSD_KERNEL_NONE = 0,
  SSD_KERNEL_VOCAB_STATS = 1,
  SSD_KERNEL_VERIFY_ATTN = 2,        /* the tensor-core attention kernel, or the SIMT prefix pass */
  SSD_KERNEL_ATTN_COMBINE = 3,
  SSD_KERNEL_ACCEPT_FINISH = 4,      /* merge, acceptance, choice and final draw */
  SSD_KERNEL_RESERVED_5 = 5,         /* unused */
  SSD_KERNEL_GATE_MATCH = 6,
  SSD_KERNEL_RETRIEVE = 7,
  SSD_KERNEL_HEAD_DOWN = 8,          /* ssd_lowrank_head: u = W_down h */
  SSD_KERNEL_HEAD_UP = 9,            /* ssd_lowrank_head: z = W_up u and its statistics */
  SSD_KERNEL_HEAD_COMBINE = 10       /* ssd_lowrank_head: per-row merge */
};
int ssd_profile_kernel(int kernel_id, void* start_event, void* end_event);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H */
