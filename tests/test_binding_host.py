"""The Python binding refuses to compute anywhere but on the GPU (no GPU needed): host
tensors are rejected before any call into the library, and a missing library raises
instead of falling back to anything else."""
import numpy as np
import pytest
import torch

from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL


def _host(inp, k):
    a = np.ascontiguousarray(inp[k])
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)


def test_host_tensors_are_rejected():
    wl = WL.WORKLOADS["tiny"]
    inp = WL.make_inputs(wl, 4)
    t = {k: _host(inp, k) for k in ("ctx", "ctx_len", "h", "w", "q", "k_cache", "v_cache", "k_cand", "v_cand",
                                      "prefix_len", "tgt", "drf", "u_acc", "u_fin", "chain_tok")}
    blk_len = torch.zeros((wl.B, wl.NB), dtype=torch.int32)
    blk_tok = torch.full((wl.B, wl.NB, wl.Dmax), -1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        S.ssd_gate_retrieve(t["ctx"], t["ctx_len"], t["h"], t["w"], wl.tau, wl.kappa, wl.W, wl.D, wl.K,
                            wl.chain_policy, t["chain_tok"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        S.ssd_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_cand"], t["v_cand"], t["prefix_len"], blk_len,
                          wl.Dmax)
    with pytest.raises(ValueError, match="CUDA tensor"):
        S.ssd_accept(t["tgt"], t["drf"], blk_tok, blk_len, t["u_acc"], t["u_fin"], mode=S.SSD_SAMPLE,
                     kind=S.SSD_LOGITS_F32, K=wl.K, chain_blk=wl.W)
    h = torch.zeros((2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        S.ssd_lowrank_head(h, torch.zeros((8, 64), dtype=torch.bfloat16), torch.zeros((100, 8), dtype=torch.bfloat16))


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(S, "_lib", None)
    monkeypatch.setattr(S, "LIB_PATH", str(tmp_path / "libssd.so"))
    with pytest.raises(RuntimeError, match="missing"):
        S.lib()
