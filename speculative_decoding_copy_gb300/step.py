"""One speculate-and-verify step on the GPU: device buffers for a batch and the
launch order of the C-ABI calls.

    gate_retrieve -> accept (row pass, finish) -> verify_attn     (one stream, "rows_first")
    gate_retrieve -> verify_attn -> accept (early rows)            (one stream, "attn_first")
    gate_retrieve -> { verify_attn (aux stream) || accept }       (two streams)
    { gate_retrieve -> accept (early rows, part of the SMs) }
      || verify_attn (every row, aux stream, the other SMs)       ("split")

Verification attention and acceptance both depend only on the retrieval output.
On one stream the kernels are chained by programmatic dependent launch: the row
pass streams the needed logit rows right after the retrieval, and the attention's
main loop (which needs nothing from the acceptance) runs on the SMs the
latency-bound finish kernel leaves free; it waits for its predecessors only before
writing.

early_rows=True lets the row pass stream every row while the retrieval still runs;
all its CTAs but the last let the finish kernel launch at once, and the last waits
for the retrieval first, so the finish (and the attention after it) are launched as
soon as the retrieval is done. Where every row is needed anyway (default_early_rows)
this is the faster mode. skip_absent makes the attention skip 128-row tiles without a
present token, at the price of waiting for its predecessor first; it pays off in
batches whose gate sends sequences to the chain draft. In the "attn_first" order the
attention's main loop starts while the retrieval still runs and the row pass, in its
early mode, streams beside it (measured slower; kept as an option).

Unless skip_absent is on, the attention writes every slot's row (all_rows): it reads
nothing that the step's earlier kernels write, so on one stream its merge does not
wait for the finish kernel to complete (it waits only before the grid ends, after its
rows are written). In the "split" order it therefore starts on an auxiliary stream
together with the retrieval, on at most attn_ctas SMs, while the retrieval, the row
pass (early mode, at most rows_ctas SMs of one CTA each) and the finish kernel run on
the main stream.

Inputs may sit in one device arena (arena_bytes), so that a caller refreshes all of
them with a single host-to-device copy. The step issues only library calls; it
computes nothing itself.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as ssd


def to_device(a: np.ndarray, device) -> torch.Tensor:
    """numpy -> CUDA tensor; bf16 bit patterns (uint16) become int16 tensors."""
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


INPUT_KEYS = ["ctx", "ctx_len", "h", "w", "q", "k_cache", "v_cache", "k_cand", "v_cand", "prefix_len", "tgt", "drf",
              "chain_tok", "u_acc", "u_fin"]
ATTN_KEYS = ("q", "k_cache", "v_cache", "k_cand", "v_cand")
ARENA_ALIGN = 256


def _step_inputs(inp: dict, with_attention: bool):
    """(key, contiguous numpy array or device tensor) for every input a step reads, in
    INPUT_KEYS order."""
    out = []
    for k in INPUT_KEYS:
        v = inp.get(k)
        if v is None or (not with_attention and k in ATTN_KEYS):
            continue
        if isinstance(v, torch.Tensor):
            out.append((k, v))
            continue
        a = np.ascontiguousarray(v)
        out.append((k, a.view(np.int16) if a.dtype == np.uint16 else a))
    return out


def arena_bytes(inp: dict, with_attention=True) -> int:
    """Bytes of one arena that holds every input of a step, each at a 256-byte boundary."""
    n = 0
    for _, a in _step_inputs(inp, with_attention):
        n = -(-n // ARENA_ALIGN) * ARENA_ALIGN + a.nbytes
    return max(n, ARENA_ALIGN)


def default_early_rows(wl) -> bool:
    """The row-pass mode measured faster for a workload: early (every row streamed while the
    retrieval runs) unless the gate can send sequences to the chain draft, whose unused
    copy-block rows the early mode would read as well."""
    return wl.chain_policy != 1


class VerifyStep:
    """Holds the inputs, outputs and workspaces of one batch of workload `wl`."""

    def __init__(self, wl, inp: dict, device="cuda", mode=None, kind=None, with_attention=True,
                 with_probs=False, early_rows=False, order="rows_first", arena: torch.Tensor | None = None,
                 skip_absent=None, attn_ctas=0, rows_ctas=0):
        """`arena`: optional uint8 device tensor of at least arena_bytes(inp, with_attention)
        bytes; the inputs are then placed in it (256-byte aligned views), so that a caller
        can refresh all of them with one host-to-device copy of a same-layout host buffer.
        `skip_absent`: the attention skips 128-row tiles without a present token (after
        waiting for its predecessor); None turns it on for batches whose gate can send
        sequences to the chain draft, where the copy-block rows of those sequences are empty."""
        if order not in ("rows_first", "attn_first", "split"):
            raise ValueError(f"unknown step order {order!r}")
        self.wl = wl
        self.early_rows = early_rows
        self.order = order
        self.attn_ctas, self.rows_ctas = int(attn_ctas), int(rows_ctas)
        self.skip_absent = (wl.chain_policy == 1 and wl.B > 1) if skip_absent is None else bool(skip_absent)
        if order == "split":
            self.skip_absent = False          # the attention reads nothing from the retrieval
        # without skip_absent the attention writes every slot's row: it then reads nothing the
        # step's earlier kernels write and waits for them only after its last row is written
        self.all_rows = not self.skip_absent
        self.mode = ssd.SSD_SAMPLE if (mode or wl.mode) == "sample" else ssd.SSD_GREEDY
        if kind is None:
            kind = ssd.SSD_LOGITS_BF16 if wl.logit_dtype == "bf16" else ssd.SSD_LOGITS_F32
        self.kind = kind
        self.device = torch.device(device)
        self.x = {}
        self.arena = arena
        if arena is not None:
            same_dev = arena.device.type == self.device.type and (self.device.index is None or
                                                                  arena.device.index == self.device.index)
            if arena.dtype != torch.uint8 or not same_dev or arena.numel() < arena_bytes(inp, with_attention):
                raise ValueError("arena must be a uint8 tensor on the step's device of at least arena_bytes() bytes")
            off = 0
            for k, a in _step_inputs(inp, with_attention):
                off = -(-off // ARENA_ALIGN) * ARENA_ALIGN
                t = arena[off:off + a.nbytes].view(torch.from_numpy(a[:0].reshape(-1)).dtype).view(a.shape)
                t.copy_(torch.from_numpy(a))
                self.x[k] = t
                off += a.nbytes
        else:
            for k, a in _step_inputs(inp, with_attention):
                # device tensors (inputs drawn on the GPU) are used in place
                self.x[k] = a.contiguous() if isinstance(a, torch.Tensor) else to_device(a, self.device)
        B = wl.B
        self.with_attention = with_attention and "q" in self.x
        i32 = lambda *s: torch.empty(s, dtype=torch.int32, device=self.device)
        self.gate_out = dict(score=torch.empty(B, dtype=torch.float32, device=self.device), gate=i32(B),
                             last_match_end=i32(B), probe_on=i32(B))
        self.ret_out = dict(blk_tok=i32(B, wl.NB, wl.Dmax), blk_len=i32(B, wl.NB), n_cand=i32(B))
        self.acc_out = ssd.alloc_accept_outputs(B, wl.NB, wl.Dmax, self.device)
        self.chain_blk = wl.W if wl.chain_policy else -1
        self.with_accept = "tgt" in self.x
        self.probs = (torch.empty((B, wl.NR, wl.V), dtype=torch.float32, device=self.device)
                      if (with_probs and self.with_accept) else None)
        if self.with_accept:
            a = ssd.accept_args(self.mode, self.kind, self.x["tgt"], self.x.get("drf"), self.ret_out["blk_tok"],
                                self.ret_out["blk_len"], wl.K, self.chain_blk, self.x["u_acc"], self.x["u_fin"],
                                self.acc_out, self.probs)
            self.acc_ws = torch.zeros(max(256, ssd.ssd_accept_workspace_size(a)), dtype=torch.uint8,
                                      device=self.device)
        if self.with_attention:
            self.attn_out = torch.empty_like(self.x["q"])
            a = ssd.attn_args(self.x["q"], self.x["k_cache"], self.x["v_cache"], self.x["k_cand"],
                              self.x["v_cand"], self.x["prefix_len"], self.ret_out["blk_len"], wl.Dmax,
                              self.attn_out, skip_absent=self.skip_absent, all_rows=self.all_rows,
                              max_ctas=self.attn_ctas)
            self.attn_ws = torch.zeros(max(256, ssd.ssd_verify_attn_workspace_size(a)), dtype=torch.uint8,
                                       device=self.device)

    # -------------------------------------------------------------------
    def gate(self, stream=None):
        wl, x = self.wl, self.x
        return ssd.ssd_gate_match(x["ctx"], x["ctx_len"], x["h"], x["w"], wl.tau, wl.kappa, out=self.gate_out,
                                  stream=stream)

    def retrieve(self, stream=None):
        wl, x = self.wl, self.x
        ct = x.get("chain_tok") if wl.chain_policy else None
        return ssd.ssd_retrieve(x["ctx"], x["ctx_len"], self.gate_out["gate"], self.gate_out["last_match_end"],
                                wl.kappa, wl.W, wl.D, wl.K, wl.chain_policy, ct, out=self.ret_out, stream=stream)

    def gate_retrieve(self, stream=None):
        """Gate and retrieval fused into one launch (same outputs as gate() then retrieve())."""
        wl, x = self.wl, self.x
        ct = x.get("chain_tok") if wl.chain_policy else None
        return ssd.ssd_gate_retrieve(x["ctx"], x["ctx_len"], x["h"], x["w"], wl.tau, wl.kappa, wl.W, wl.D, wl.K,
                                     wl.chain_policy, ct, out={**self.gate_out, **self.ret_out}, stream=stream)

    def attention(self, stream=None, blk_len_ready=False):
        """blk_len_ready: the retrieval has completed before this launch (the acceptance chain
        or an event sits between them), so the attention skips empty tiles without waiting for
        the kernel before it (skip_absent mode 2)."""
        x = self.x
        skip = (2 if blk_len_ready else 1) if self.skip_absent else 0
        return ssd.ssd_verify_attn(x["q"], x["k_cache"], x["v_cache"], x["k_cand"], x["v_cand"], x["prefix_len"],
                                   self.ret_out["blk_len"], self.wl.Dmax, out=self.attn_out, ws=self.attn_ws,
                                   stream=stream, skip_absent=skip, all_rows=self.all_rows,
                                   max_ctas=self.attn_ctas)

    def accept(self, stream=None, early_rows=None):
        wl, x = self.wl, self.x
        early = self.early_rows if early_rows is None else early_rows
        return ssd.ssd_accept(x["tgt"], x.get("drf") if wl.chain_policy else None, self.ret_out["blk_tok"],
                              self.ret_out["blk_len"], x["u_acc"], x["u_fin"], mode=self.mode, kind=self.kind,
                              K=wl.K, chain_blk=self.chain_blk, out=self.acc_out, ws=self.acc_ws,
                              probs_out=self.probs, stream=stream, early_rows=early,
                              max_ctas=self.rows_ctas if self.order == "split" else 0)

    def run(self, stream=None, aux: torch.cuda.Stream | None = None):
        """Issue the whole step on `stream` (default: current), attention on `aux` if given
        (the "split" order needs `aux`)."""
        main = stream or torch.cuda.current_stream()
        if self.order == "split" and self.with_attention:
            if aux is None:
                raise ValueError("the split order runs the attention on an auxiliary stream")
            ev = torch.cuda.Event()
            ev.record(main)
            aux.wait_event(ev)
            self.attention(aux)
            self.gate_retrieve(main)
            if self.with_accept:
                self.accept(main)
            ev2 = torch.cuda.Event()
            ev2.record(aux)
            main.wait_event(ev2)
            return
        self.gate_retrieve(main)
        if self.with_attention and aux is not None:
            ev = torch.cuda.Event()
            ev.record(main)
            aux.wait_event(ev)
            self.attention(aux, blk_len_ready=True)
            if self.with_accept:
                self.accept(main)
            ev2 = torch.cuda.Event()
            ev2.record(aux)
            main.wait_event(ev2)
        elif self.order == "attn_first" and self.with_attention:
            # one stream: the attention right behind the retrieval, then the row pass in its
            # early mode beside the attention, then the finish kernel
            self.attention(main)
            if self.with_accept:
                self.accept(main, early_rows=True)
        else:
            # one stream: the acceptance chain first (it needs only the retrieval's output),
            # then the attention, whose main loop overlaps the latency-bound finish kernel
            if self.with_accept:
                self.accept(main)
            if self.with_attention:
                # after the acceptance chain: its finish kernel launches only once the
                # retrieval has completed (in either row-pass mode)
                self.attention(main, blk_len_ready=self.with_accept)

    def results(self) -> dict:
        """Copy every output to host numpy arrays (synchronises)."""
        torch.cuda.synchronize()
        outs = {**self.gate_out, **self.ret_out, **(self.acc_out if self.with_accept else {})}
        r = {k: v.cpu().numpy() for k, v in outs.items()}
        if self.with_attention:
            o = self.attn_out
            # fp32 output as float32; bf16 output as its uint16 bit patterns
            r["attn"] = o.cpu().numpy() if o.dtype == torch.float32 else o.view(torch.int16).cpu().numpy().view(np.uint16)
        if self.probs is not None:
            r["probs"] = self.probs.cpu().numpy()
        return r
