"""GPU verification attention against the fp64 oracle: max-abs error <= 1e-2
(bf16 inputs, fp32 accumulation), on every present token for small shapes
spanning several tiles with ragged tails, and on sampled tokens at the full
workload sizes."""
import numpy as np
import pytest
import torch

from oracle import ssd_oracle as O
from speculative_decoding_copy_gb300 import _binding as S
from speculative_decoding_copy_gb300 import workloads as WL
from speculative_decoding_copy_gb300.step import VerifyStep, to_device

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _as_f64(x, dtype):
    # rows of absent tokens are never written and may hold any bit pattern
    with np.errstate(invalid="ignore"):
        return O.to_f64(x, dtype)


def _run_attn(case, blk_len, Dmax, dtype, out_f32=False, max_ctas=0):
    dev = "cuda"
    t = {k: to_device(np.asarray(v), dev) for k, v in case.items()}
    bl = to_device(blk_len, dev)
    out = S.ssd_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_cand"], t["v_cand"], t["prefix_len"], bl, Dmax,
                            out_f32=out_f32, max_ctas=max_ctas)
    torch.cuda.synchronize()
    o = out.cpu()
    return o.numpy() if (dtype == "f32" or out_f32) else o.view(torch.int16).numpy().view(np.uint16)


def _case(rng, B, NB, Dmax, Hq, Hkv, dh, prefix, dtype, q_scale=1.0):
    P_max = max(1, max(prefix))
    NT = NB * Dmax
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    cast = (lambda x: x) if dtype == "f32" else WL.f32_to_bf16_bits
    return dict(q=cast(f(B, NT, Hq, dh) * np.float32(q_scale)), k_cache=cast(f(B, Hkv, P_max, dh)),
                v_cache=cast(f(B, Hkv, P_max, dh)), k_cand=cast(f(B, NT, Hkv, dh)), v_cand=cast(f(B, NT, Hkv, dh)),
                prefix_len=np.asarray(prefix, np.int32))


def _check_all(case, blk_len, Dmax, dtype, slots=None, out_f32=False, max_ctas=0):
    got = _run_attn(case, blk_len, Dmax, dtype, out_f32, max_ctas)
    ref = O.verify_attention(case["q"], case["k_cache"], case["v_cache"], case["k_cand"], case["v_cand"],
                             case["prefix_len"], blk_len, Dmax, dtype, slots)
    g = _as_f64(got, "f32" if out_f32 else dtype)
    err = 0.0
    for (b, t), o in ref.items():
        err = max(err, float(np.max(np.abs(g[b, t] - o))))
    assert err <= TOL, err
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dh", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_attention_small_shapes(dtype, dh, G):
    rng = np.random.default_rng(dh + G + (7 if dtype == "bf16" else 0))
    Hkv = 2
    B, NB, Dmax = 3, 3, 5
    prefix = [0, 37, 300]             # empty prefix, ragged tails, several key tiles
    case = _case(rng, B, NB, Dmax, Hkv * G, Hkv, dh, prefix, dtype, q_scale=2.0)
    blk_len = np.array([[5, 0, 3], [1, 5, 5], [2, 4, 0]], np.int32)
    # sharpened scores give outputs up to |o| ~ 4, where rounding the output itself to
    # bf16 costs up to 0.008: the bound is checked on an fp32 output
    _check_all(case, blk_len, Dmax, dtype, out_f32=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_attention_sharp_and_long(dtype):
    # sharper scores (q scaled) and a prefix spanning many splits
    rng = np.random.default_rng(31)
    case = _case(rng, 2, 2, 8, 8, 2, 128, [2049, 4100], dtype, q_scale=4.0)
    blk_len = np.array([[8, 3], [6, 8]], np.int32)
    _check_all(case, blk_len, 8, dtype, out_f32=True)


@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("max_ctas", [0, 2])
def test_attention_reference_jumps(G, max_ctas):
    """Planted keys whose scores jump far above every earlier key of their row (by about
    20, 40 and 65 in log2 units), each in the second half of its 128-key tile and in
    ever later tiles (0, 4 and 10), so that the running reference max moves several
    times and the sum so far is rescaled each time. With max_ctas = 2 each kv head's row
    tile is one CTA that walks the whole prefix (no split), so every jump happens inside
    one running sum."""
    rng = np.random.default_rng(70 + G)
    Hkv, B, NB, Dmax = 2, 1, 2, 4
    Hq, dh, P = Hkv * G, 128, 1500
    NT = NB * Dmax
    u = rng.standard_normal(dh)
    u /= np.linalg.norm(u)
    q = 0.3 * rng.standard_normal((B, NT, Hq, dh)) + 3.0 * u
    k = 0.3 * rng.standard_normal((B, Hkv, P, dh))
    for pos, beta in ((100, 52.0), (600, 110.0), (1350, 170.0)):   # columns 100, 88, 70 of tiles 0, 4, 10
        k[:, :, pos, :] = beta * u
    cast = WL.f32_to_bf16_bits
    case = dict(q=cast(q.astype(np.float32)), k_cache=cast(k.astype(np.float32)),
                v_cache=cast(rng.standard_normal((B, Hkv, P, dh)).astype(np.float32)),
                k_cand=cast(rng.standard_normal((B, NT, Hkv, dh)).astype(np.float32)),
                v_cand=cast(rng.standard_normal((B, NT, Hkv, dh)).astype(np.float32)),
                prefix_len=np.array([P], np.int32))
    blk_len = np.array([[4, 2]], np.int32)
    _check_all(case, blk_len, Dmax, "bf16", out_f32=True, max_ctas=max_ctas)


def test_attention_tiny_workload():
    wl = WL.WORKLOADS["tiny"]
    inp = WL.make_inputs(wl)
    keys = ("q", "k_cache", "v_cache", "k_cand", "v_cand", "prefix_len")
    blk_len = np.array([[wl.D, wl.D, 0]], np.int32)
    _check_all({k: inp[k] for k in keys}, blk_len, wl.Dmax, wl.kv_dtype)


@pytest.mark.parametrize("name", ["llama8b", "llama70b", "batched", "qwen8b_mixed"])
def test_attention_full_size_sampled(name):
    """Full workload size, the step's own launch path; 24 sampled tokens against the oracle."""
    wl = WL.WORKLOADS[name]
    inp = WL.make_inputs(wl, with_logits=False)
    st = VerifyStep(wl, inp)
    st.gate()
    st.retrieve()
    st.attention()
    r = st.results()
    bl = r["blk_len"]
    present = [(b, k * wl.Dmax + d) for b in range(wl.B) for k in range(wl.NB) for d in range(bl[b, k])]
    rng = np.random.default_rng(3)
    pick = [present[i] for i in rng.choice(len(present), size=min(24, len(present)), replace=False)]
    ref = O.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_cand"], inp["v_cand"],
                             inp["prefix_len"], bl, wl.Dmax, wl.kv_dtype, pick)
    g = _as_f64(r["attn"], wl.kv_dtype)
    err = max(float(np.max(np.abs(g[b, t] - o))) for (b, t), o in ref.items())
    assert err <= TOL, err


@pytest.mark.parametrize("prefix", [[1, 127, 128, 129], [4096, 4100, 300, 1000]])
@pytest.mark.parametrize("G", [4, 8])
def test_attention_tcgen05_and_simt_paths(prefix, G, monkeypatch):
    """bf16, head dim 128: the tcgen05 prefix pass and the SIMT prefix pass both
    match the oracle (ragged prefixes around the 128-key tile edge, several M tiles)."""
    rng = np.random.default_rng(G * 1000 + prefix[0])
    B, NB, Dmax, Hkv = len(prefix), 5, 20, 2
    case = _case(rng, B, NB, Dmax, Hkv * G, Hkv, 128, prefix, "bf16", q_scale=2.0)
    blk_len = rng.integers(0, Dmax + 1, size=(B, NB)).astype(np.int32)
    blk_len[:, 0] = Dmax
    errs = {}
    for path in ("tc", "simt"):
        if path == "simt":
            monkeypatch.setenv("SSD_ATTN_KERNEL", "simt")
        else:
            monkeypatch.delenv("SSD_ATTN_KERNEL", raising=False)
        errs[path] = _check_all(case, blk_len, Dmax, "bf16", out_f32=True)
    assert errs["tc"] <= TOL and errs["simt"] <= TOL


def _paged(rng, cache_bits, spare=5):
    """A contiguous cache [B][Hkv][P_max][dh] (bf16 bits) scattered into 128-token pages in
    a random order, with unused pages of noise; returns (pages, block_table)."""
    B, Hkv, P_max, dh = cache_bits.shape
    pps = -(-P_max // 128)
    n = B * pps + spare
    order = rng.permutation(n)
    pages = WL.f32_to_bf16_bits(rng.standard_normal((n, Hkv, 128, dh)).astype(np.float32))
    table = np.zeros((B, pps), np.int32)
    for b in range(B):
        for j in range(pps):
            pg = int(order[b * pps + j])
            table[b, j] = pg
            rows = cache_bits[b, :, j * 128:min(P_max, (j + 1) * 128)]
            pages[pg, :, :rows.shape[1]] = rows
    return pages, table


@pytest.mark.parametrize("G,prefix", [(4, [0, 37, 300]), (1, [129, 256, 500]), (8, [4096, 1000, 2049])])
def test_attention_paged_cache(G, prefix):
    """The tensor-core pass reading its prefix through a block table of 128-token pages
    (random page order, pages shared by two sequences) against the oracle."""
    rng = np.random.default_rng(G + len(prefix) + prefix[0])
    Hkv, B, NB, Dmax = 2, 3, 3, 5
    case = _case(rng, B, NB, Dmax, Hkv * G, Hkv, 128, prefix, "bf16", q_scale=2.0)
    blk_len = np.array([[5, 0, 3], [1, 5, 5], [2, 4, 0]], np.int32)
    kp, table = _paged(rng, case["k_cache"])
    vp = np.zeros_like(kp)
    for b in range(B):
        for j in range(table.shape[1]):
            rows = case["v_cache"][b, :, j * 128:min(case["v_cache"].shape[2], (j + 1) * 128)]
            vp[table[b, j], :, :rows.shape[1]] = rows
    table[2, 0] = table[0, 0]                          # sequence 2 reads sequence 0's first page (a shared prompt)
    dev = "cuda"
    t = {k: to_device(np.asarray(v), dev) for k, v in case.items()}
    out = S.ssd_verify_attn(t["q"], to_device(kp, dev), to_device(vp, dev), t["k_cand"], t["v_cand"], t["prefix_len"],
                            to_device(blk_len, dev), Dmax, out_f32=True, block_table=to_device(table, dev))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = O.verify_attention_paged(case["q"], kp, vp, table, case["k_cand"], case["v_cand"], case["prefix_len"],
                                   blk_len, Dmax, "bf16")
    err = max(float(np.max(np.abs(got[b, t_] - o))) for (b, t_), o in ref.items())
    assert err <= TOL, err


def test_attention_paged_bad_page_is_reported():
    rng = np.random.default_rng(77)
    case = _case(rng, 1, 1, 4, 4, 1, 128, [300], "bf16")
    kp, table = _paged(rng, case["k_cache"])
    vp = kp.copy()
    table[0, 1] = kp.shape[0] + 3                      # a page that does not exist
    dev = "cuda"
    t = {k: to_device(np.asarray(v), dev) for k, v in case.items()}
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    S.ssd_verify_attn(t["q"], to_device(kp, dev), to_device(vp, dev), t["k_cand"], t["v_cand"], t["prefix_len"],
                      to_device(np.array([[4]], np.int32), dev), 4, ws=ws, block_table=to_device(table, dev))
    assert S.ssd_read_device_error(ws) == S.SSD_ERR_DEVICE


@pytest.mark.parametrize("G", [4, 8])
def test_attention_skip_absent_tiles(G):
    """skip_absent (both modes): 128-row tiles in which no token is present are skipped.
    Present rows equal the full computation bit for bit and the oracle within the bound;
    absent rows are written by none of the three calls."""
    rng = np.random.default_rng(50 + G)
    Hkv, B, NB, Dmax = 2, 4, 3, 20
    prefix = [300, 0, 4100, 129]
    case = _case(rng, B, NB, Dmax, Hkv * G, Hkv, 128, prefix, "bf16", q_scale=2.0)
    # tile 0 empty / tile 1 empty / everything empty / everything present
    blk_len = np.array([[0, 0, 5], [3, 0, 0], [0, 0, 0], [20, 20, 20]], np.int32)
    dev = "cuda"
    t = {k: to_device(np.asarray(v), dev) for k, v in case.items()}
    bl = to_device(blk_len, dev)
    outs = []
    # 0: every tile; 1: skip after waiting for the kernel before; 2: skip, blk_len complete at
    # launch (a host copy wrote it), no wait before the grid's end
    for skip in (0, 1, 2):
        out = torch.full(t["q"].shape, 7.0, dtype=torch.float32, device=dev)
        S.ssd_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_cand"], t["v_cand"], t["prefix_len"], bl, Dmax,
                          out=out, skip_absent=skip)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    present = np.zeros((B, NB * Dmax), bool)
    for b in range(B):
        for k in range(NB):
            present[b, k * Dmax:k * Dmax + blk_len[b, k]] = True
    for mode in (1, 2):
        np.testing.assert_array_equal(outs[mode][present], outs[0][present])
        assert np.all(outs[mode][~present] == 7.0)
    assert np.all(outs[0][~present] == 7.0)
    ref = O.verify_attention(case["q"], case["k_cache"], case["v_cache"], case["k_cand"], case["v_cand"],
                             case["prefix_len"], blk_len, Dmax, "bf16", None)
    err = max(float(np.max(np.abs(outs[1][b, t_] - o))) for (b, t_), o in ref.items())
    assert err <= TOL, err


@pytest.mark.parametrize("dtype,dh,G,max_ctas", [("bf16", 128, 4, 0), ("bf16", 128, 4, 5), ("bf16", 128, 8, 30),
                                                 ("bf16", 128, 1, 2), ("f32", 64, 4, 0)])
def test_attention_all_rows(dtype, dh, G, max_ctas):
    """all_rows: every slot's row is written (blk_len not given) as the attention of its q over
    the prefix and its block's slots up to it, which is the oracle's result for that slot when
    the slot is present; with the grid capped to max_ctas CTAs as well."""
    rng = np.random.default_rng(70 + G + dh + max_ctas)
    Hkv, B, NB, Dmax = 2, 3, 3, 20
    prefix = [300, 0, 4100]
    case = _case(rng, B, NB, Dmax, Hkv * G, Hkv, dh, prefix, dtype, q_scale=2.0)
    dev = "cuda"
    t = {k: to_device(np.asarray(v), dev) for k, v in case.items()}
    out = S.ssd_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_cand"], t["v_cand"], t["prefix_len"], None, Dmax,
                            out_f32=True, all_rows=True, max_ctas=max_ctas, NB=NB)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    full = np.full((B, NB), Dmax, np.int32)
    ref = O.verify_attention(case["q"], case["k_cache"], case["v_cache"], case["k_cand"], case["v_cand"],
                             case["prefix_len"], full, Dmax, dtype, None)
    assert len(ref) == B * NB * Dmax
    err = max(float(np.max(np.abs(got[b, t_] - o))) for (b, t_), o in ref.items())
    assert err <= TOL, err


def test_attention_all_rows_rejects_skip_absent():
    rng = np.random.default_rng(5)
    case = _case(rng, 1, 1, 4, 4, 1, 128, [128], "bf16")
    dev = "cuda"
    t = {k: to_device(np.asarray(v), dev) for k, v in case.items()}
    with pytest.raises(S.SsdError):
        S.ssd_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_cand"], t["v_cand"], t["prefix_len"],
                          to_device(np.array([[4]], np.int32), dev), 4, all_rows=True, skip_absent=True)
