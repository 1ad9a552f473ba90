"""Pins for attention over compressed keys and for top-k search."""
from math import pi, sqrt

import numpy as np

import oracle
from oracle import rng
from oracle.codebook import sphere_codebook


def _setup(B=2, Hkv=2, G=2, N=20, d=16, seed=0):
    Pi, S = rng.method_matrices(seed, d, d)
    Piv, _ = rng.method_matrices(seed + 1, d, 1)
    cbk = sphere_codebook(d, 2)
    cbv = sphere_codebook(d, 3)
    K = rng.gaussian_stream(seed + 2, B * Hkv * N * d).reshape(B, Hkv, N, d)
    V = rng.gaussian_stream(seed + 3, B * Hkv * N * d).reshape(B, Hkv, N, d)
    q = rng.gaussian_stream(seed + 4, B * Hkv * G * d).reshape(B, Hkv * G, d)
    kz = oracle.quantize(K, Pi, cbk, S)
    vz = oracle.quantize(V, Piv, cbv)
    return dict(Pi=Pi, S=S, Piv=Piv, cbk=cbk, cbv=cbv, K=K, V=V, q=q, kz=kz, vz=vz)


def test_logits_by_scalar_loops():
    s = _setup()
    lens = np.array([20, 7])
    scale = 0.25
    L = oracle.attention_logits(s["q"], s["kz"], lens, s["Pi"], s["S"], s["cbk"], scale)
    c = s["cbk"].centroids
    for b in range(2):
        for h in range(4):
            g = h // 2
            qr = s["Pi"] @ s["q"][b, h]
            u = s["S"] @ s["q"][b, h]
            for i in range(20):
                if i >= lens[b]:
                    assert np.isnan(L[b, h, i])
                    continue
                mse = sum(qr[j] * c[s["kz"].idx[b, g, i, j]] for j in range(16))
                qj = sum(u[j] * (1.0 if s["kz"].signs[b, g, i, j] else -1.0) for j in range(16))
                est = s["kz"].norm16[b, g, i] * mse + s["kz"].rnorm16[b, g, i] * sqrt(pi / 2) / 16 * qj
                assert abs(L[b, h, i] - scale * est) < 1e-12 * max(1.0, abs(est))


def test_output_by_scalar_loops_and_softmax():
    s = _setup()
    lens = np.array([20, 7])
    scale = 0.3
    O = oracle.attention_output(s["q"], s["kz"], lens, s["Pi"], s["S"], s["cbk"], scale,
                                values=s["vz"], Pi_v=s["Piv"], cb_v=s["cbv"])
    L = oracle.attention_logits(s["q"], s["kz"], lens, s["Pi"], s["S"], s["cbk"], scale)
    for b in range(2):
        for h in range(4):
            n = lens[b]
            w = np.exp(L[b, h, :n] - L[b, h, :n].max())
            p = w / w.sum()
            assert abs(p.sum() - 1.0) < 1e-12
            vhat = oracle.dequantize(s["vz"].idx[b, h // 2, :n], s["vz"].norm16[b, h // 2, :n], s["Piv"], s["cbv"])
            ref = sum(p[i] * vhat[i] for i in range(n))
            assert np.allclose(O[b, h], ref, rtol=1e-12, atol=1e-12)


def test_equal_keys_give_mean_and_dominant_key_gives_its_value():
    s = _setup(B=1, Hkv=1, G=1, N=6)
    kz = s["kz"]
    same = oracle.Quantized(idx=np.repeat(kz.idx[:, :, :1], 6, axis=2), norm16=np.repeat(kz.norm16[:, :, :1], 6, axis=2),
                            signs=np.repeat(kz.signs[:, :, :1], 6, axis=2), rnorm16=np.repeat(kz.rnorm16[:, :, :1], 6, axis=2))
    O = oracle.attention_output(s["q"], same, np.array([6]), s["Pi"], s["S"], s["cbk"], 1.0, values_dense=s["V"])
    assert np.allclose(O[0, 0], s["V"][0, 0].mean(axis=0), rtol=1e-12, atol=1e-12)
    # key 3 made dominant by scaling its norm: the output tends to v_3
    big = oracle.Quantized(idx=kz.idx.copy(), norm16=kz.norm16.copy(), signs=kz.signs.copy(), rnorm16=kz.rnorm16.copy())
    L = oracle.attention_logits(s["q"], kz, np.array([6]), s["Pi"], s["S"], s["cbk"], 1.0)[0, 0]
    i = int(np.argmax(L))
    big.norm16[0, 0, i] *= 1e3
    big.rnorm16[0, 0, i] *= 1e3
    O = oracle.attention_output(s["q"], big, np.array([6]), s["Pi"], s["S"], s["cbk"], 1.0, values_dense=s["V"])
    assert np.allclose(O[0, 0], s["V"][0, 0, i], atol=1e-9)


def test_gqa_group_mapping_and_empty_sequence():
    s = _setup(B=1, Hkv=2, G=3, N=5)
    O = oracle.attention_output(s["q"], s["kz"], np.array([0]), s["Pi"], s["S"], s["cbk"], 1.0, values_dense=s["V"])
    assert np.all(O == 0)
    L = oracle.attention_logits(s["q"], s["kz"], np.array([5]), s["Pi"], s["S"], s["cbk"], 1.0)
    for h in range(6):
        z = oracle.Quantized(idx=s["kz"].idx[0, h // 3], norm16=s["kz"].norm16[0, h // 3],
                             signs=s["kz"].signs[0, h // 3], rnorm16=s["kz"].rnorm16[0, h // 3])
        assert np.allclose(L[0, h], oracle.estimate(s["q"][0, h], z, s["Pi"], s["cbk"], s["S"]), rtol=1e-13)


def _db(n, d, seed):
    Pi, S = rng.method_matrices(seed, d, d)
    cb = sphere_codebook(d, 2)
    X = rng.gaussian_stream(seed + 1, n * d).reshape(n, d)
    X /= np.linalg.norm(X, axis=1, keepdims=True)
    return Pi, S, cb, X, oracle.quantize(X, Pi, cb, S)


def test_topk_brute_force():
    d, n = 24, 300
    Pi, S, cb, X, z = _db(n, d, 30)
    Q = rng.gaussian_stream(99, 7 * d).reshape(7, d)
    top_s, top_i = oracle.search_topk(Q, z, Pi, cb, S, 10)
    for r in range(7):
        sc = [oracle.estimate(Q[r], z, Pi, cb, S)[i] for i in range(n)]
        order = sorted(range(n), key=lambda i: (-sc[i], i))[:10]
        assert list(top_i[r]) == order
        assert np.array_equal(top_s[r], np.array(sc)[order])


def test_topk_k_equals_n_ties_and_recall():
    d, n = 16, 50
    Pi, S, cb, X, z = _db(n, d, 40)
    # duplicate vector 3 at position 10: identical codes, identical scores; lower index first
    for f in ("idx", "signs"):
        getattr(z, f)[10] = getattr(z, f)[3]
    z.norm16[10], z.rnorm16[10] = z.norm16[3], z.rnorm16[3]
    Q = X[[3, 5]]
    top_s, top_i = oracle.search_topk(Q, z, Pi, cb, S, n)
    for r in range(2):
        assert sorted(top_i[r]) == list(range(n))
        assert np.all(np.diff(top_s[r]) <= 0)
        p3, p10 = list(top_i[r]).index(3), list(top_i[r]).index(10)
        assert p3 < p10
    true_top1 = np.argmax(Q @ X.T, axis=1)
    assert oracle.recall_at_1(top_i, true_top1) == 1.0       # recall@1@N = 1
