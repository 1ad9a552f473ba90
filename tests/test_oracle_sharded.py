"""Pins for the oracle's sharded attention and search: each is pinned to the unsharded oracle
step it reassembles (attention_values, search_topk), over uneven blocks, empty blocks and
sequences, and ties that straddle two blocks."""
from math import sqrt

import numpy as np
import pytest

import oracle
from oracle import rng, sharded
from oracle.codebook import sphere_codebook


def _coded_case(B, Hkv, G, N, d, seed):
    Pi, S = rng.method_matrices(seed, d, d)
    Piv, _ = rng.method_matrices(seed + 1, d, 1)
    cbk, cbv = sphere_codebook(d, 2), sphere_codebook(d, 3)
    X = rng.gaussian_stream(seed + 2, B * Hkv * N * d).reshape(B, Hkv, N, d)
    V = rng.gaussian_stream(seed + 3, B * Hkv * N * d).reshape(B, Hkv, N, d)
    q = rng.gaussian_stream(seed + 4, B * Hkv * G * d).reshape(B, Hkv * G, d)
    kz = oracle.quantize(X, Pi, cbk, S)
    vz = oracle.quantize(V, Piv, cbv)
    return Pi, S, Piv, cbk, cbv, V, q, kz, vz


def _slice(z, lo, hi):
    return oracle.Quantized(idx=z.idx[:, :, lo:hi], norm16=z.norm16[:, :, lo:hi])


def test_shard_bounds_cover_every_row_once():
    for n in (0, 1, 7, 100, 131073):
        for world in (1, 2, 3, 8):
            b = [sharded.shard_bounds(n, world, r) for r in range(world)]
            assert b[0][0] == 0 and b[-1][1] == n
            assert all(b[r][1] == b[r + 1][0] for r in range(world - 1))
            sizes = [hi - lo for lo, hi in b]
            assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("world", [1, 2, 3, 5])
@pytest.mark.parametrize("coded", [True, False])
def test_merged_partials_equal_the_unsharded_values(world, coded):
    B, Hkv, G, N, d = 3, 2, 4, 37, 16
    Pi, S, Piv, cbk, cbv, V, q, kz, vz = _coded_case(B, Hkv, G, N, d, seed=5)
    lens = np.array([37, 11, 0])                       # full, short (some blocks empty), empty sequence
    logits = oracle.attention_logits(q, kz, lens, Pi, S, cbk, 1.0 / sqrt(d))
    logits = np.nan_to_num(logits, nan=0.0)
    if coded:
        ref = oracle.attention_values(logits, lens, Hkv, values=vz, Pi_v=Piv, cb_v=cbv)
    else:
        ref = oracle.attention_values(logits, lens, Hkv, values_dense=V)
    parts = []
    for r in range(world):
        lo, hi = sharded.shard_bounds(N, world, r)
        ll = np.clip(lens - lo, 0, hi - lo)
        if coded:
            parts.append(sharded.attention_partial(logits[:, :, lo:hi], ll, Hkv, values=_slice(vz, lo, hi), cb_v=cbv))
        else:
            parts.append(sharded.attention_partial(logits[:, :, lo:hi], ll, Hkv, values_dense=V[:, :, lo:hi]))
    got = sharded.merge_partials(parts, Piv if coded else None)
    assert np.max(np.abs(got - ref)) < 1e-12
    assert np.all(got[2] == 0.0)                       # the empty sequence stays zero


def test_one_dominant_logit_selects_its_value_across_blocks():
    d, N = 8, 10
    V = rng.gaussian_stream(1, N * d).reshape(1, 1, N, d)
    logits = np.zeros((1, 1, N))
    logits[0, 0, 7] = 80.0                             # in the second of two blocks
    parts = [sharded.attention_partial(logits[:, :, lo:hi], np.array([hi - lo]), 1, values_dense=V[:, :, lo:hi])
             for lo, hi in ((0, 5), (5, 10))]
    got = sharded.merge_partials(parts)
    assert np.max(np.abs(got[0, 0] - V[0, 0, 7])) < 1e-12


@pytest.mark.parametrize("world,k", [(2, 10), (3, 7), (4, 30)])
def test_merged_topk_equals_the_unsharded_search(world, k):
    # The oracle's float64 scores of one vector can differ in the last bits between a whole-
    # database and a block matrix product, so rows may trade places only where their scores are
    # within 1e-12 (relative) of each other; everything else is identical.
    d, n, nq = 16, 90, 6
    Pi, S = rng.method_matrices(9, d, d)
    cb = sphere_codebook(d, 2)
    X = rng.gaussian_stream(10, n * d).reshape(n, d)
    X[70] = X[3]                                       # near-equal scores in different blocks
    X[44] = X[3]
    Q = np.concatenate([X[3:4], rng.gaussian_stream(11, (nq - 1) * d).reshape(nq - 1, d)])
    z = oracle.quantize(X, Pi, cb, S)
    ref_s, ref_i = oracle.search_topk(Q, z, Pi, cb, S, k)
    all_s = oracle.estimate_all(Q, z, Pi, cb, S)
    lists = []
    for r in range(world):
        lo, hi = sharded.shard_bounds(n, world, r)
        zr = oracle.Quantized(idx=z.idx[lo:hi], norm16=z.norm16[lo:hi], signs=z.signs[lo:hi], rnorm16=z.rnorm16[lo:hi])
        s, i = oracle.search_topk(Q, zr, Pi, cb, S, k)   # k may exceed a block: it returns all of it
        lists.append((s, i + lo))
    got_s, got_i = sharded.merge_topk(lists, k)
    assert got_s.shape == ref_s.shape
    assert np.max(np.abs(got_s - ref_s)) < 1e-12 * np.max(np.abs(ref_s))
    for r in range(nq):
        for a, b in zip(got_i[r], ref_i[r]):
            if a != b:
                assert abs(all_s[r, a] - all_s[r, b]) < 1e-12 * abs(all_s[r, b])
    assert set(got_i[0][:3]) == {3, 44, 70}


def test_merge_topk_orders_exact_ties_by_global_row():
    lists = [(np.array([[5.0, 3.0, 3.0]]), np.array([[0, 2, 7]])),
             (np.array([[5.0, 3.0]]), np.array([[10, 1]])),
             (np.array([[9.0]]), np.array([[40]]))]
    s, i = sharded.merge_topk(lists, 5)
    assert i.tolist() == [[40, 0, 10, 1, 2]]
    assert s.tolist() == [[9.0, 5.0, 5.0, 3.0, 3.0]]
