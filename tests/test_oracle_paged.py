"""Pins for the paged decode-step oracle: against the pinned contiguous path (quantize every row,
attend over the contiguous cache), invariance to which physical pages hold the tokens, and the
appended rows landing in their page slots and nowhere else."""
import numpy as np

import oracle
from oracle import paged, rng
from oracle.codebook import sphere_codebook


def _setup(d=16, seed=3):
    Pi, S = rng.method_matrices(seed, d, d)
    Pv, _ = rng.method_matrices(seed + 1, d, 1)
    return Pi, S, sphere_codebook(d, 2), Pv, sphere_codebook(d, 3)


def _fill(kpool, vpool, table, lens, ps, K, V, Pi, S, cbk, Pv, cbv):
    """Write tokens 0 .. lens[b] - 1 of K, V [B, Hkv, N, d] into their pages."""
    for b in range(len(lens)):
        for i in range(lens[b]):
            page, slot = table[b][i // ps], i % ps
            for h in range(K.shape[1]):
                zk = oracle.quantize(K[b, h, i][None], Pi, cbk, S)
                zv = oracle.quantize(V[b, h, i][None], Pv, cbv)
                kpool.idx[page, h, slot], kpool.norm16[page, h, slot] = zk.idx[0], zk.norm16[0]
                kpool.signs[page, h, slot], kpool.rnorm16[page, h, slot] = zk.signs[0], zk.rnorm16[0]
                vpool.idx[page, h, slot], vpool.norm16[page, h, slot] = zv.idx[0], zv.norm16[0]


def test_paged_step_equals_the_contiguous_path():
    d, B, Hkv, G, ps, npages = 16, 2, 2, 4, 8, 12
    Pi, S, cbk, Pv, cbv = _setup(d)
    lens = np.array([13, 0])
    K = rng.gaussian_stream(10, B * Hkv * 14 * d).reshape(B, Hkv, 14, d)
    V = rng.gaussian_stream(11, B * Hkv * 14 * d).reshape(B, Hkv, 14, d)
    q = rng.gaussian_stream(12, B * Hkv * G * d).reshape(B, Hkv * G, d)
    table = np.array([[7, 2, 9, -1], [4, -1, -1, -1]])
    kpool, vpool = paged.alloc_pool(npages, Hkv, ps, d, d), paged.alloc_pool(npages, Hkv, ps, d)
    _fill(kpool, vpool, table, lens, ps, K, V, Pi, S, cbk, Pv, cbv)
    out, new = paged.paged_decode_step(q, K[:, :, 13], V[:, :, 13], kpool, vpool, table, lens, ps,
                                       Pi, S, cbk, Pv, cbv, 0.25)
    assert np.array_equal(new, [14, 1])
    # contiguous reference: sequence 0 holds K[0, :, :14]; sequence 1 holds only its new token,
    # which the step took from K[1, :, 13]
    Kc = K.copy()
    Kc[1, :, 0], Vc = K[1, :, 13], V.copy()
    Vc[1, :, 0] = V[1, :, 13]
    flat_k = oracle.quantize(Kc.reshape(-1, d), Pi, cbk, S)
    flat_v = oracle.quantize(Vc.reshape(-1, d), Pv, cbv)
    kz = oracle.Quantized(idx=flat_k.idx.reshape(B, Hkv, 14, d), norm16=flat_k.norm16.reshape(B, Hkv, 14),
                          signs=flat_k.signs.reshape(B, Hkv, 14, d), rnorm16=flat_k.rnorm16.reshape(B, Hkv, 14))
    vz = oracle.Quantized(idx=flat_v.idx.reshape(B, Hkv, 14, d), norm16=flat_v.norm16.reshape(B, Hkv, 14))
    ref = oracle.attention_output(q, kz, new, Pi, S, cbk, 0.25, values=vz, Pi_v=Pv, cb_v=cbv)
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


def test_output_does_not_depend_on_which_pages_hold_the_tokens():
    d, B, Hkv, G, ps = 16, 1, 1, 4, 4
    Pi, S, cbk, Pv, cbv = _setup(d, seed=5)
    lens = np.array([9])
    K = rng.gaussian_stream(20, 10 * d).reshape(1, 1, 10, d)
    V = rng.gaussian_stream(21, 10 * d).reshape(1, 1, 10, d)
    q = rng.gaussian_stream(22, G * d).reshape(1, G, d)
    outs = []
    for table in (np.array([[0, 1, 2]]), np.array([[5, 3, 1]])):
        kpool, vpool = paged.alloc_pool(6, Hkv, ps, d, d), paged.alloc_pool(6, Hkv, ps, d)
        _fill(kpool, vpool, table, lens, ps, K, V, Pi, S, cbk, Pv, cbv)
        out, _ = paged.paged_decode_step(q, K[:, :, 9], V[:, :, 9], kpool, vpool, table, lens, ps,
                                         Pi, S, cbk, Pv, cbv, 0.5)
        outs.append(out)
    assert np.array_equal(outs[0], outs[1])


def test_appended_rows_land_in_their_slots_only():
    d, B, Hkv, ps = 16, 2, 2, 4
    Pi, S, cbk, Pv, cbv = _setup(d, seed=7)
    lens = np.array([5, 3])
    table = np.array([[2, 0], [1, 3]])
    kpool, vpool = paged.alloc_pool(4, Hkv, ps, d, d), paged.alloc_pool(4, Hkv, ps, d)
    kn = rng.gaussian_stream(30, B * Hkv * d).reshape(B, Hkv, d)
    vn = rng.gaussian_stream(31, B * Hkv * d).reshape(B, Hkv, d)
    q = rng.gaussian_stream(32, B * 4 * d).reshape(B, 4, d)
    before = kpool.idx.copy()
    paged.paged_decode_step(q, kn, vn, kpool, vpool, table, lens, ps, Pi, S, cbk, Pv, cbv, 1.0)
    for b, (pg, slot) in ((0, (table[0][5 // ps], 5 % ps)), (1, (table[1][3 // ps], 3 % ps))):
        for h in range(Hkv):
            z = oracle.quantize(kn[b, h][None], Pi, cbk, S)
            assert np.array_equal(kpool.idx[pg, h, slot], z.idx[0]) and kpool.norm16[pg, h, slot] == z.norm16[0]
            assert np.array_equal(kpool.signs[pg, h, slot], z.signs[0])
            zv = oracle.quantize(vn[b, h][None], Pv, cbv)
            assert np.array_equal(vpool.idx[pg, h, slot], zv.idx[0])
    changed = np.argwhere((kpool.idx != before).any(axis=-1))
    assert {tuple(x) for x in changed} <= {(0, 0, 1), (0, 1, 1), (1, 0, 3), (1, 1, 3)}
