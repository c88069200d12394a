"""ctypes binding of libssd.so: argument marshalling only.

Every function takes CUDA torch tensors (torch is used for device memory and
streams only), checks shapes and dtypes, allocates missing outputs with torch
and calls the C entry point of the same name on the current (or given) stream.
All arithmetic happens in the library's kernels. If the library has not been
built, every call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64, c_void_p

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libssd.so")
CHECKED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libssd_checked.so")

SSD_OK, SSD_ERR_INVALID, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_WORKSPACE, SSD_ERR_TIMEOUT, SSD_ERR_DEVICE = (
    0, -1, -2, -3, -4, -5, -6)
SSD_F32, SSD_BF16 = 0, 1
SSD_LOGITS_F32, SSD_LOGITS_BF16, SSD_PROBS_F32 = 0, 1, 2
SSD_GREEDY, SSD_SAMPLE = 0, 1
SSD_CHAIN_NONE, SSD_CHAIN_WHEN_GATE_OFF, SSD_CHAIN_ALWAYS = 0, 1, 2

EXPORTED = ["ssd_status_string", "ssd_version", "ssd_launch_count", "ssd_gate_match", "ssd_retrieve",
            "ssd_verify_attn_workspace_size", "ssd_verify_attn", "ssd_accept_workspace_size", "ssd_accept",
            "ssd_read_device_error", "ssd_profile_kernel", "ssd_accept_static", "ssd_gate_retrieve",
            "ssd_selftest_wait", "ssd_commit_kv",
            "ssd_copy_stats", "ssd_lowrank_head_workspace_size", "ssd_lowrank_head", "ssd_read_static_error",
            "ssd_read_probe", "ssd_checked_build", "ssd_read_check_error"]
SSD_KERNEL = dict(vocab_stats=1, verify_attn=2, attn_combine=3, accept_finish=4, gate_match=6,
                  retrieve=7, head_down=8, head_up=9, head_combine=10)


class SsdError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} ({status})")
        self.status = status


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k_cache", c_void_p), ("v_cache", c_void_p), ("k_cand", c_void_p),
                ("v_cand", c_void_p), ("out", c_void_p), ("prefix_len", c_void_p), ("blk_len", c_void_p),
                ("dtype", c_int), ("B", c_int), ("NB", c_int), ("Dmax", c_int), ("Hq", c_int), ("Hkv", c_int),
                ("dh", c_int), ("P_max", c_int64), ("scale", c_float), ("out_dtype", c_int),
                ("block_table", c_void_p), ("pages_per_seq", c_int), ("num_pages", c_int64),
                ("skip_absent", c_int), ("all_rows", c_int), ("max_ctas", c_int)]


class CommitArgs(ctypes.Structure):
    _fields_ = [("k_cache", c_void_p), ("v_cache", c_void_p), ("k_cand", c_void_p), ("v_cand", c_void_p),
                ("prefix_len", c_void_p), ("best_blk", c_void_p), ("n_out", c_void_p), ("dtype", c_int),
                ("B", c_int), ("NB", c_int), ("Dmax", c_int), ("Hkv", c_int), ("dh", c_int), ("P_max", c_int64)]


class HeadArgs(ctypes.Structure):
    _fields_ = [("h", c_void_p), ("w_down", c_void_p), ("w_up", c_void_p), ("logits", c_void_p),
                ("logits_dtype", c_int), ("row_max", c_void_p), ("lse", c_void_p), ("argmax", c_void_p),
                ("M", c_int), ("d", c_int), ("r", c_int), ("V", c_int)]


class AcceptArgs(ctypes.Structure):
    _fields_ = [("mode", c_int), ("kind", c_int), ("tgt", c_void_p), ("drf", c_void_p), ("V", c_int64),
                ("blk_tok", c_void_p), ("blk_len", c_void_p), ("B", c_int), ("NB", c_int), ("Dmax", c_int),
                ("K", c_int), ("chain_blk", c_int), ("u_acc", c_void_p), ("u_fin", c_void_p),
                ("acc_len", c_void_p), ("best_blk", c_void_p), ("n_out", c_void_p), ("out_tok", c_void_p),
                ("probs_out", c_void_p), ("early_rows", c_int), ("max_ctas", c_int)]


_lib = None
_loaded = {}


def lib() -> ctypes.CDLL:
    """The library every call goes through: libssd.so unless use_library() selected another
    build. Raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


class use_library:
    """Context manager: calls inside go through the library at `path` (e.g. the checked build)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.prev = _lib
        _lib = load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def load(path) -> ctypes.CDLL:
    """Load one build of the library (once per path) with every entry point's signature."""
    if path not in _loaded:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with speculative_decoding_copy_gb300.build.build_all()")
        L = ctypes.CDLL(path)
        L.ssd_status_string.restype = ctypes.c_char_p
        L.ssd_status_string.argtypes = [c_int]
        L.ssd_version.restype = c_int
        L.ssd_launch_count.restype = c_uint64
        L.ssd_selftest_wait.restype = c_int
        L.ssd_selftest_wait.argtypes = [c_void_p, c_int, ctypes.c_uint64, c_void_p]
        L.ssd_commit_kv.restype = c_int
        L.ssd_commit_kv.argtypes = [c_void_p, c_void_p, ctypes.c_size_t, c_void_p]
        L.ssd_copy_stats.restype = c_int
        L.ssd_copy_stats.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]
        L.ssd_lowrank_head_workspace_size.restype = c_size_t
        L.ssd_lowrank_head_workspace_size.argtypes = [POINTER(HeadArgs)]
        L.ssd_lowrank_head.restype = c_int
        L.ssd_lowrank_head.argtypes = [POINTER(HeadArgs), c_void_p, c_size_t, c_void_p]
        L.ssd_gate_match.restype = c_int
        L.ssd_gate_match.argtypes = [c_void_p, c_int64, c_void_p, c_int, c_void_p, c_int, c_int64, c_void_p, c_int,
                                     c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
        L.ssd_retrieve.restype = c_int
        L.ssd_retrieve.argtypes = [c_void_p, c_int64, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                   c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
        L.ssd_gate_retrieve.restype = c_int
        L.ssd_gate_retrieve.argtypes = [c_void_p, c_int64, c_void_p, c_int, c_void_p, c_int, c_int64, c_void_p,
                                        c_int, c_float, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
        L.ssd_verify_attn_workspace_size.restype = c_size_t
        L.ssd_verify_attn_workspace_size.argtypes = [POINTER(AttnArgs)]
        L.ssd_verify_attn.restype = c_int
        L.ssd_verify_attn.argtypes = [POINTER(AttnArgs), c_void_p, c_size_t, c_void_p]
        L.ssd_accept_workspace_size.restype = c_size_t
        L.ssd_accept_workspace_size.argtypes = [POINTER(AcceptArgs)]
        L.ssd_accept.restype = c_int
        L.ssd_accept.argtypes = [POINTER(AcceptArgs), c_void_p, c_size_t, c_void_p]
        L.ssd_read_device_error.restype = c_int
        L.ssd_read_device_error.argtypes = [c_void_p, c_void_p, POINTER(c_int32)]
        L.ssd_accept_static.restype = c_int
        L.ssd_accept_static.argtypes = [POINTER(AcceptArgs), c_void_p]
        L.ssd_read_probe.restype = c_int
        L.ssd_read_probe.argtypes = [c_void_p, c_size_t, c_int, c_void_p, c_void_p]
        L.ssd_read_static_error.restype = c_int
        L.ssd_read_static_error.argtypes = [c_void_p, POINTER(c_int32)]
        L.ssd_profile_kernel.restype = c_int
        L.ssd_profile_kernel.argtypes = [c_int, c_void_p, c_void_p]
        L.ssd_checked_build.restype = c_int
        L.ssd_read_check_error.restype = c_int
        L.ssd_read_check_error.argtypes = [c_void_p, POINTER(c_int32)]
        _loaded[path] = L
    return _loaded[path]


def status_string(status: int) -> str:
    return lib().ssd_status_string(int(status)).decode()


def launch_count() -> int:
    return int(lib().ssd_launch_count())


def _check(fn: str, rc: int):
    if rc != SSD_OK:
        raise SsdError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtypes, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


_HALF = (torch.bfloat16, torch.int16)


def _elem_type(t) -> int:
    return SSD_F32 if t.dtype == torch.float32 else SSD_BF16


def _empty_like_dtype(shape, like, dtype=None):
    return torch.empty(shape, dtype=dtype or like.dtype, device=like.device)


# ---------------------------------------------------------------------------
def ssd_gate_match(ctx, ctx_len, h, w, tau, kappa, *, out=None, stream=None):
    """Probe gate and kappa-gram check; returns dict(score, gate, last_match_end, probe_on)."""
    _need(ctx, "ctx", (torch.int32,), 2)
    _need(ctx_len, "ctx_len", (torch.int32,), 1)
    _need(h, "h", (torch.float32,) + _HALF, 2)
    _need(w, "w", (torch.float32,), 1)
    B = ctx.shape[0]
    d = w.shape[0]
    o = out or {}
    score = o.get("score") if o.get("score") is not None else _empty_like_dtype((B,), ctx, torch.float32)
    gate = o.get("gate") if o.get("gate") is not None else _empty_like_dtype((B,), ctx)
    last = o.get("last_match_end") if o.get("last_match_end") is not None else _empty_like_dtype((B,), ctx)
    on = o.get("probe_on") if o.get("probe_on") is not None else _empty_like_dtype((B,), ctx)
    rc = lib().ssd_gate_match(_ptr(ctx), ctx.shape[1], _ptr(ctx_len), B, _ptr(h), _elem_type(h), h.shape[1],
                              _ptr(w), d, float(tau), int(kappa), _ptr(score), _ptr(gate), _ptr(last), _ptr(on),
                              _stream(stream))
    _check("ssd_gate_match", rc)
    return dict(score=score, gate=gate, last_match_end=last, probe_on=on)


def ssd_retrieve(ctx, ctx_len, gate, last_match_end, kappa, W, D, K, chain_policy, chain_tok=None, *,
                 out=None, stream=None):
    """Copy candidates (most recent first) and the chain block; returns dict(blk_tok, blk_len, n_cand)."""
    _need(ctx, "ctx", (torch.int32,), 2)
    _need(gate, "gate", (torch.int32,), 1)
    B = ctx.shape[0]
    NB = W + (1 if chain_policy else 0)
    Dmax = max(D, K) if chain_policy else D
    o = out or {}
    blk_tok = o.get("blk_tok") if o.get("blk_tok") is not None else _empty_like_dtype((B, NB, Dmax), ctx)
    blk_len = o.get("blk_len") if o.get("blk_len") is not None else _empty_like_dtype((B, NB), ctx)
    n_cand = o.get("n_cand") if o.get("n_cand") is not None else _empty_like_dtype((B,), ctx)
    if chain_tok is not None:
        _need(chain_tok, "chain_tok", (torch.int32,), 2)
    rc = lib().ssd_retrieve(_ptr(ctx), ctx.shape[1], _ptr(ctx_len), B, _ptr(gate), _ptr(last_match_end),
                            int(kappa), int(W), int(D), int(K), int(chain_policy), _ptr(chain_tok), _ptr(blk_tok),
                            _ptr(blk_len), _ptr(n_cand), _stream(stream))
    _check("ssd_retrieve", rc)
    return dict(blk_tok=blk_tok, blk_len=blk_len, n_cand=n_cand)


def ssd_gate_retrieve(ctx, ctx_len, h, w, tau, kappa, W, D, K, chain_policy, chain_tok=None, *, out=None,
                      stream=None):
    """Gate and retrieval in one launch; returns the outputs of both calls."""
    _need(ctx, "ctx", (torch.int32,), 2)
    _need(ctx_len, "ctx_len", (torch.int32,), 1)
    _need(h, "h", (torch.float32,) + _HALF, 2)
    _need(w, "w", (torch.float32,), 1)
    B = ctx.shape[0]
    NB = W + (1 if chain_policy else 0)
    Dmax = max(D, K) if chain_policy else D
    o = dict(out or {})
    need = dict(score=((B,), torch.float32), gate=((B,), torch.int32), last_match_end=((B,), torch.int32),
                probe_on=((B,), torch.int32), blk_tok=((B, NB, Dmax), torch.int32), blk_len=((B, NB), torch.int32),
                n_cand=((B,), torch.int32))
    for k, (shape, dt) in need.items():
        if o.get(k) is None:
            o[k] = torch.empty(shape, dtype=dt, device=ctx.device)
    if chain_tok is not None:
        _need(chain_tok, "chain_tok", (torch.int32,), 2)
    rc = lib().ssd_gate_retrieve(_ptr(ctx), ctx.shape[1], _ptr(ctx_len), B, _ptr(h), _elem_type(h), h.shape[1],
                                 _ptr(w), w.shape[0], float(tau), int(kappa), int(W), int(D), int(K),
                                 int(chain_policy), _ptr(chain_tok), _ptr(o["score"]), _ptr(o["gate"]),
                                 _ptr(o["last_match_end"]), _ptr(o["probe_on"]), _ptr(o["blk_tok"]),
                                 _ptr(o["blk_len"]), _ptr(o["n_cand"]), _stream(stream))
    _check("ssd_gate_retrieve", rc)
    return o


def attn_args(q, k_cache, v_cache, k_cand, v_cand, prefix_len, blk_len, Dmax, out, scale=0.0,
              block_table=None, skip_absent=False, all_rows=False, max_ctas=0, NB=None) -> AttnArgs:
    """k_cache/v_cache: [B][Hkv][P_max][dh], or with block_table [B][pages_per_seq] pages of 128
    tokens [num_pages][Hkv][128][dh]. blk_len may be None with all_rows (NB then given)."""
    B, NT, Hq, dh = q.shape
    Hkv = k_cache.shape[1]
    NB = blk_len.shape[1] if blk_len is not None else (NB if NB is not None else NT // int(Dmax))
    tail = (int(skip_absent), int(bool(all_rows)), int(max_ctas))
    if block_table is None:
        return AttnArgs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_cand), _ptr(v_cand), _ptr(out),
                        _ptr(prefix_len), _ptr(blk_len), _elem_type(q), B, NB, int(Dmax), Hq, Hkv, dh,
                        k_cache.shape[2], float(scale), _elem_type(out), None, 0, 0, *tail)
    pps = block_table.shape[1]
    return AttnArgs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_cand), _ptr(v_cand), _ptr(out),
                    _ptr(prefix_len), _ptr(blk_len), _elem_type(q), B, NB, int(Dmax), Hq, Hkv, dh,
                    128 * pps, float(scale), _elem_type(out), _ptr(block_table), pps, k_cache.shape[0], *tail)


def ssd_verify_attn_workspace_size(args: AttnArgs) -> int:
    return int(lib().ssd_verify_attn_workspace_size(ctypes.byref(args)))


def ssd_verify_attn(q, k_cache, v_cache, k_cand, v_cand, prefix_len, blk_len, Dmax, *, out=None, ws=None,
                    scale=0.0, stream=None, out_f32=False, block_table=None, skip_absent=False, all_rows=False,
                    max_ctas=0, NB=None):
    """Block-triangular verification attention; returns the output tensor [B][NT][Hq][dh]
    (the inputs' dtype, or fp32 with out_f32). With block_table [B][pages_per_seq] int32 the
    caches are pages of 128 tokens [num_pages][Hkv][128][dh]. all_rows: every slot's row is
    written and blk_len is not read (it may be None, NB then given)."""
    types = (torch.float32,) + _HALF
    for n, t in [("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("k_cand", k_cand), ("v_cand", v_cand)]:
        _need(t, n, types, 4)
        if _elem_type(t) != _elem_type(q):
            raise ValueError("all attention tensors must share one dtype")
    _need(prefix_len, "prefix_len", (torch.int32,), 1)
    if blk_len is not None or not all_rows:
        _need(blk_len, "blk_len", (torch.int32,), 2)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out_f32 else torch.empty_like(q)
    if block_table is not None:
        _need(block_table, "block_table", (torch.int32,), 2)
    args = attn_args(q, k_cache, v_cache, k_cand, v_cand, prefix_len, blk_len, Dmax, out, scale, block_table,
                     skip_absent, all_rows, max_ctas, NB)
    need = ssd_verify_attn_workspace_size(args)
    if ws is None:
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib().ssd_verify_attn(ctypes.byref(args), _ptr(ws), ws.numel(), _stream(stream))
    _check("ssd_verify_attn", rc)
    return out


def accept_args(mode, kind, tgt, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin, outs, probs_out=None,
                early_rows=False, max_ctas=0):
    B, NR, V = tgt.shape
    _, NB, Dmax = blk_tok.shape
    return AcceptArgs(int(mode), int(kind), _ptr(tgt), _ptr(drf), V, _ptr(blk_tok), _ptr(blk_len), B, NB, Dmax,
                      int(K), int(chain_blk), _ptr(u_acc), _ptr(u_fin), _ptr(outs["acc_len"]),
                      _ptr(outs["best_blk"]), _ptr(outs["n_out"]), _ptr(outs["out_tok"]), _ptr(probs_out),
                      int(bool(early_rows)), int(max_ctas))


def ssd_accept_workspace_size(args: AcceptArgs) -> int:
    return int(lib().ssd_accept_workspace_size(ctypes.byref(args)))


def alloc_accept_outputs(B, NB, Dmax, device):
    z = lambda *s: torch.empty(s, dtype=torch.int32, device=device)
    return dict(acc_len=z(B, NB), best_blk=z(B), n_out=z(B), out_tok=z(B, Dmax + 1))


def ssd_accept(tgt, drf, blk_tok, blk_len, u_acc, u_fin, *, mode, kind, K=0, chain_blk=-1, out=None, ws=None,
               probs_out=None, stream=None, early_rows=False, max_ctas=0):
    """Acceptance, choice of block and final token; returns dict(acc_len, best_blk, n_out, out_tok).
    early_rows: the row pass reads every row without first waiting for the kernel before it."""
    _need(tgt, "tgt", (torch.float32,) + _HALF, 3)
    if drf is not None:
        _need(drf, "drf", (tgt.dtype,), 3)
    _need(blk_tok, "blk_tok", (torch.int32,), 3)
    _need(blk_len, "blk_len", (torch.int32,), 2)
    B, NR, V = tgt.shape
    _, NB, Dmax = blk_tok.shape
    outs = out or alloc_accept_outputs(B, NB, Dmax, tgt.device)
    args = accept_args(mode, kind, tgt, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin, outs, probs_out,
                       early_rows, max_ctas)
    need = ssd_accept_workspace_size(args)
    if ws is None:
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=tgt.device)
    rc = lib().ssd_accept(ctypes.byref(args), _ptr(ws), ws.numel(), _stream(stream))
    _check("ssd_accept", rc)
    return outs


def ssd_selftest_wait(ws, arrive, limit_clocks, stream=None):
    """One CTA waits on an mbarrier with the library's bounded wait (arrived on, or never)."""
    _check("ssd_selftest_wait", lib().ssd_selftest_wait(_ptr(ws), int(arrive), int(limit_clocks), _stream(stream)))


def ssd_commit_kv(k_cache, v_cache, k_cand, v_cand, prefix_len, best_blk, n_out, Dmax, ws=None, stream=None):
    """Append the accepted tokens' K/V rows (from ssd_accept's best_blk, n_out) to the prefix
    cache in place and advance prefix_len. Returns the workspace (its header holds any
    device-side error)."""
    _need(k_cache, "k_cache", (torch.float32,) + _HALF, 4)
    B, Hkv, P_max, dh = k_cache.shape
    NT = k_cand.shape[1]
    dt = SSD_F32 if k_cache.dtype == torch.float32 else SSD_BF16
    args = CommitArgs(_ptr(k_cache), _ptr(v_cache), _ptr(k_cand), _ptr(v_cand), _ptr(prefix_len), _ptr(best_blk),
                      _ptr(n_out), dt, B, NT // Dmax, Dmax, Hkv, dh, P_max)
    if ws is None:
        ws = torch.zeros(256, dtype=torch.uint8, device=k_cache.device)
    _check("ssd_commit_kv", lib().ssd_commit_kv(ctypes.byref(args), _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def ssd_copy_stats(gate, n_cand, acc_len, W, counts, stream=None):
    """Add this batch's copy attempts, taxed attempts, accepted copy tokens and sequences
    to counts (int64 [4] on the device)."""
    _need(acc_len, "acc_len", (torch.int32,), 2)
    B, NB = acc_len.shape
    if counts.dtype != torch.int64 or counts.numel() < 4 or not counts.is_cuda:
        raise ValueError("counts: int64 device tensor of 4")
    _check("ssd_copy_stats", lib().ssd_copy_stats(_ptr(gate), _ptr(n_cand), _ptr(acc_len), B, NB, int(W), _ptr(counts),
                                                  _stream(stream)))
    return counts


def head_args(h, w_down, w_up, row_max, lse, argmax, logits=None) -> HeadArgs:
    """Marshal the low-rank head's arguments (shapes and dtypes checked)."""
    _need(h, "h", (torch.bfloat16,), 2)
    _need(w_down, "w_down", (torch.bfloat16,), 2)
    _need(w_up, "w_up", (torch.bfloat16,), 2)
    M, d = h.shape
    r, V = w_down.shape[0], w_up.shape[0]
    if w_down.shape[1] != d or w_up.shape[1] != r:
        raise ValueError("shapes: h [M][d], w_down [r][d], w_up [V][r]")
    for t, n, dt in ((row_max, "row_max", torch.float32), (lse, "lse", torch.float32), (argmax, "argmax", torch.int32)):
        _need(t, n, (dt,), 1)
        if t.numel() != M:
            raise ValueError(f"{n} must hold M = {M} values")
    ldt = SSD_F32
    if logits is not None:
        _need(logits, "logits", (torch.float32, torch.bfloat16), 2)
        if tuple(logits.shape) != (M, V):
            raise ValueError(f"logits must be [{M}][{V}]")
        ldt = SSD_F32 if logits.dtype == torch.float32 else SSD_BF16
    return HeadArgs(_ptr(h), _ptr(w_down), _ptr(w_up), _ptr(logits), ldt, _ptr(row_max), _ptr(lse), _ptr(argmax),
                    M, d, r, V)


def ssd_lowrank_head_workspace_size(args: HeadArgs) -> int:
    return int(lib().ssd_lowrank_head_workspace_size(ctypes.byref(args)))


def ssd_lowrank_head(h, w_down, w_up, logits=None, logits_dtype=None, out=None, ws=None, stream=None):
    """The low-rank draft head z = W_up (W_down h) with per-row max, log-sum-exp and first
    argmax. h [M][d], w_down [r][d], w_up [V][r] bf16 on the device. logits_dtype
    (torch.float32 / torch.bfloat16) asks for the logits [M][V]; out = (row_max, lse,
    argmax[, logits]) reuses buffers. Returns (row_max, lse, argmax, logits or None, ws)."""
    M, V = h.shape[0], w_up.shape[0]
    dev = h.device
    if out is not None:
        row_max, lse, argmax = out[:3]
        logits = out[3] if len(out) > 3 else None
    else:
        row_max = torch.empty(M, dtype=torch.float32, device=dev)
        lse = torch.empty(M, dtype=torch.float32, device=dev)
        argmax = torch.empty(M, dtype=torch.int32, device=dev)
        logits = torch.empty(M, V, dtype=logits_dtype, device=dev) if logits_dtype is not None else None
    args = head_args(h, w_down, w_up, row_max, lse, argmax, logits)
    need = ssd_lowrank_head_workspace_size(args)
    if need == 0:   # invalid or unsupported arguments: the call itself reports which
        _check("ssd_lowrank_head", lib().ssd_lowrank_head(ctypes.byref(args), None, 0, _stream(stream)))
        raise SsdError("ssd_lowrank_head_workspace_size", SSD_ERR_INVALID)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    _check("ssd_lowrank_head", lib().ssd_lowrank_head(ctypes.byref(args), _ptr(ws), ws.numel(), _stream(stream)))
    return row_max, lse, argmax, logits, ws


def ssd_read_probe(buf, nbytes, sink, ctas_per_sm=2, stream=None):
    """Read `nbytes` of the device tensor `buf` once (measurement tool for read bandwidth)."""
    if not buf.is_cuda or not sink.is_cuda or sink.numel() * sink.element_size() < 16:
        raise ValueError("buf and sink (>= 16 bytes) must be CUDA tensors")
    if nbytes > buf.numel() * buf.element_size():
        raise ValueError("nbytes exceeds the buffer")
    _check("ssd_read_probe", lib().ssd_read_probe(_ptr(buf), int(nbytes), int(ctas_per_sm), _ptr(sink),
                                                  _stream(stream)))


def ssd_read_check_error(stream=None) -> int:
    """Read and clear the check words of the checked build (SSD_OK in the normal build)."""
    v = c_int32(0)
    _check("ssd_read_check_error", lib().ssd_read_check_error(_stream(stream), ctypes.byref(v)))
    return int(v.value)


def ssd_read_device_error(ws, stream=None) -> int:
    v = c_int32(0)
    rc = lib().ssd_read_device_error(_ptr(ws), _stream(stream), ctypes.byref(v))
    _check("ssd_read_device_error", rc)
    return int(v.value)


def ssd_profile_kernel(kernel: str | None, start=None, end=None):
    """Bracket every later launch of `kernel` with the given torch.cuda.Events
    (created with enable_timing=True); None switches the hook off."""
    if kernel is None:
        _check("ssd_profile_kernel", lib().ssd_profile_kernel(0, None, None))
        return
    for ev in (start, end):
        if ev.cuda_event == 0:     # torch creates the CUDA event lazily
            ev.record()
    rc = lib().ssd_profile_kernel(SSD_KERNEL[kernel], ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(end.cuda_event))
    _check("ssd_profile_kernel", rc)


def ssd_accept_static(tgt, drf, blk_tok, blk_len, u_acc, u_fin, *, mode, kind, K=0, chain_blk=-1, out=None,
                      stream=None, early_rows=False):
    """ssd_accept with the library's fixed internal scratch instead of a workspace
    (for callers that cannot allocate); calls must not overlap on the GPU."""
    _need(tgt, "tgt", (torch.float32,) + _HALF, 3)
    _need(blk_tok, "blk_tok", (torch.int32,), 3)
    _need(blk_len, "blk_len", (torch.int32,), 2)
    B, NR, V = tgt.shape
    _, NB, Dmax = blk_tok.shape
    outs = out or alloc_accept_outputs(B, NB, Dmax, tgt.device)
    args = accept_args(mode, kind, tgt, drf, blk_tok, blk_len, K, chain_blk, u_acc, u_fin, outs, None, early_rows)
    rc = lib().ssd_accept_static(ctypes.byref(args), _stream(stream))
    _check("ssd_accept_static", rc)
    return outs


def ssd_read_static_error(stream=None) -> int:
    """Read and clear the device error word of ssd_accept_static's fixed scratch on the
    current device (synchronises the stream)."""
    v = c_int32(0)
    _check("ssd_read_static_error", lib().ssd_read_static_error(_stream(stream), ctypes.byref(v)))
    return int(v.value)
