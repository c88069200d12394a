"""Pins of the paged prefix cache in the oracle: scattering a contiguous cache into
pages (any page order, pages shared between sequences) and reading it back through
the block table changes nothing."""
import numpy as np

from oracle import ssd_oracle as O


def _scatter(cache, rng, spare=3):
    """Contiguous [B][Hkv][P_max][dh] -> pages [num_pages][Hkv][128][dh] in a random order
    (plus unused pages of noise) and the block table that reads them back."""
    B, Hkv, P_max, dh = cache.shape
    pps = -(-P_max // O.PAGE)
    n = B * pps + spare
    order = rng.permutation(n)
    pages = rng.standard_normal((n, Hkv, O.PAGE, dh)).astype(cache.dtype)
    table = np.zeros((B, pps), np.int32)
    for b in range(B):
        for j in range(pps):
            pg = int(order[b * pps + j])
            table[b, j] = pg
            rows = cache[b, :, j * O.PAGE:min(P_max, (j + 1) * O.PAGE)]
            pages[pg, :, :rows.shape[1]] = rows
    return pages, table


def test_gather_inverts_the_scatter():
    rng = np.random.default_rng(21)
    cache = rng.standard_normal((3, 2, 300, 8)).astype(np.float32)
    pages, table = _scatter(cache, rng)
    back = O.gather_pages(pages, table, 300)
    np.testing.assert_array_equal(back, cache)


def test_paged_attention_equals_contiguous():
    rng = np.random.default_rng(22)
    B, NB, Dmax, Hq, Hkv, dh = 2, 2, 3, 4, 2, 16
    P_max = 260
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, kc, vc = f(B, NB * Dmax, Hq, dh), f(B, Hkv, P_max, dh), f(B, Hkv, P_max, dh)
    kd, vd = f(B, NB * Dmax, Hkv, dh), f(B, NB * Dmax, Hkv, dh)
    prefix = np.array([260, 131], np.int32)
    blk_len = np.array([[3, 1], [2, 3]], np.int32)
    kp, table = _scatter(kc, rng)
    vp = np.zeros_like(kp)
    for b in range(B):
        for j in range(table.shape[1]):
            rows = vc[b, :, j * O.PAGE:min(P_max, (j + 1) * O.PAGE)]
            vp[table[b, j], :, :rows.shape[1]] = rows
    ref = O.verify_attention(q, kc, vc, kd, vd, prefix, blk_len, Dmax, "f32")
    got = O.verify_attention_paged(q, kp, vp, table, kd, vd, prefix, blk_len, Dmax, "f32")
    for key in ref:
        np.testing.assert_array_equal(got[key], ref[key])


def test_shared_pages_give_equal_rows():
    """Two sequences whose tables name the same pages (a shared prompt) and whose queries
    and candidates are equal get equal outputs; a different page changes them."""
    rng = np.random.default_rng(23)
    Hq, Hkv, dh, Dmax = 2, 1, 8, 2
    pages = rng.standard_normal((4, Hkv, O.PAGE, dh)).astype(np.float32)
    vpages = rng.standard_normal((4, Hkv, O.PAGE, dh)).astype(np.float32)
    q1 = rng.standard_normal((1, Dmax, Hq, dh)).astype(np.float32)
    kd1 = rng.standard_normal((1, Dmax, Hkv, dh)).astype(np.float32)
    q, kd = np.concatenate([q1, q1]), np.concatenate([kd1, kd1])
    prefix = np.array([200, 200], np.int32)
    blk_len = np.array([[2], [2]], np.int32)
    same = O.verify_attention_paged(q, pages, vpages, np.array([[2, 0], [2, 0]], np.int32), kd, kd, prefix, blk_len,
                                    Dmax, "f32")
    for t in range(Dmax):
        np.testing.assert_array_equal(same[(0, t)], same[(1, t)])
    diff = O.verify_attention_paged(q, pages, vpages, np.array([[2, 0], [2, 3]], np.int32), kd, kd, prefix, blk_len,
                                    Dmax, "f32")
    assert not np.allclose(diff[(0, 0)], diff[(1, 0)])
