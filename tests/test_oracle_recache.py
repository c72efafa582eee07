"""Pins for the recache oracle: projection, RMSNorm, 3D RoPE (CPU only)."""

import math

import numpy as np

from oracle import recache as orc


def test_projection_against_loops():
    rng = np.random.default_rng(0)
    hid = rng.standard_normal((5, 6))
    w = rng.standard_normal((6, 12))
    k, v = orc.project(hid, w)
    for i in range(5):
        for j in range(6):
            assert abs(k[i, j] - sum(hid[i, t] * w[t, j] for t in range(6))) < 1e-12
            assert abs(v[i, j] - sum(hid[i, t] * w[t, 6 + j] for t in range(6))) < 1e-12


def test_rmsnorm_unit_rms_and_gain():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 96)) * 3.0
    y = orc.rmsnorm(x, None, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-14)
    g = rng.standard_normal(96)
    assert np.allclose(orc.rmsnorm(x, g, eps=0.0), y * g, atol=1e-14)
    # eps enters under the root: a zero row stays zero, a tiny row is damped
    assert np.all(orc.rmsnorm(np.zeros((1, 8)), None, 1e-6) == 0)


def test_rope_bands():
    assert orc.rope_bands(128) == (22, 21, 21)
    assert orc.rope_bands(64) == (12, 10, 10)
    assert orc.rope_bands(6) == (1, 1, 1)


def test_rope_worked_examples():
    # D = 6: one pair per axis, every band has b = 2 dims so omega_0 = 1
    x = np.array([[[1.0, 0.0, 1.0, 0.0, 0.0, 2.0]]])
    y = orc.rope3d(x, [1], [2], [0], theta=10000.0)
    want = [math.cos(1), math.sin(1), math.cos(2), math.sin(2), 0.0, 2.0]
    assert np.allclose(y[0, 0], want, atol=1e-15)
    # D = 12: two pairs per band (b = 4): omega = 1, theta^(-1/2)
    x = np.zeros((1, 1, 12))
    x[0, 0, 2] = 1.0  # second pair of the frame band
    y = orc.rope3d(x, [3], [0], [0], theta=10000.0)
    ang = 3 * 10000.0 ** -0.5
    assert np.allclose(y[0, 0, 2:4], [math.cos(ang), math.sin(ang)], atol=1e-15)
    assert np.allclose(np.delete(y[0, 0], [2, 3]), 0)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(2)
    T, H, D = 11, 2, 128
    q = rng.standard_normal((T, H, D))
    k = rng.standard_normal((T, H, D))
    zero = np.zeros(T, int)
    assert np.allclose(orc.rope3d(q, zero, zero, zero), q, atol=0)
    pf, ph, pw = rng.integers(0, 900, T), rng.integers(0, 30, T), rng.integers(0, 52, T)
    rq = orc.rope3d(q, pf, ph, pw)
    pn = lambda x: np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
    assert np.allclose(pn(rq), pn(q), atol=1e-12)
    # <R(m) q, R(n) k> depends only on m - n on every axis
    sf, sh, sw = 37, 5, 11
    a = np.einsum("thd,thd->th", orc.rope3d(q, pf, ph, pw), orc.rope3d(k, pf[::-1], ph[::-1], pw[::-1]))
    b = np.einsum("thd,thd->th", orc.rope3d(q, pf + sf, ph + sh, pw + sw),
                  orc.rope3d(k, pf[::-1] + sf, ph[::-1] + sh, pw[::-1] + sw))
    assert np.allclose(a, b, atol=1e-9)


def test_token_positions():
    f, h, w = orc.token_positions(2, 4680, 1560, 3, 52)
    assert f[0] == 6 and f[-1] == 8 and f[1560] == 7
    assert h[0] == 0 and w[0] == 0 and h[51] == 0 and w[51] == 51 and h[52] == 1
    assert h[1559] == 29 and w[1559] == 51


def test_recache_composition():
    rng = np.random.default_rng(3)
    H, D, tpf, cf, gw = 2, 64, 16, 2, 4
    Tc = tpf * cf
    ids = [0, 4, 5]
    hid = rng.standard_normal((len(ids) * Tc, H * D))
    w = rng.standard_normal((H * D, 2 * H * D)) * 0.05
    gamma = rng.uniform(0.5, 1.5, H * D)
    k, v = orc.recache(hid, w, gamma, ids, H, D, tpf, cf, gw)
    kv = hid @ w
    assert np.allclose(v.reshape(-1, H * D), kv[:, H * D:], atol=1e-12)
    kn = kv[:, :H * D] / np.sqrt(np.mean(kv[:, :H * D] ** 2, axis=1, keepdims=True) + 1e-6) * gamma
    # chunk 4 tokens: RoPE at frames 8, 9
    f, hh, ww = orc.token_positions(4, Tc, tpf, cf, gw)
    want = orc.rope3d(kn[Tc:2 * Tc].reshape(Tc, H, D), f, hh, ww)
    assert np.allclose(k[Tc:2 * Tc], want, atol=1e-12)
    # the norm is taken before the rotation: rotation keeps the row RMS
    assert np.allclose(np.sqrt(np.mean(k.reshape(-1, H * D) ** 2, axis=1)),
                       np.sqrt(np.mean(kn ** 2, axis=1)), atol=1e-12)


def test_recache_equals_appended_chunk_projections():
    """Recache => append consistency: project each chunk's hidden states as it
    arrives (project_chunk, K and V appended to the cache model), stream past
    evictions, then recache the present chunks from the same hidden states:
    every cached row comes out the same.  The present chunks {0, 5, 6} sit at
    non-adjacent frame positions, so a wrong position offset or chunk order in
    either path shows."""
    from oracle.cache_model import CacheModel
    rng = np.random.default_rng(5)
    H, D, tpf, cf, gw, W = 2, 64, 16, 2, 4, 2
    Tc, HD = tpf * cf, H * D
    w_qkv = rng.standard_normal((HD, 3 * HD)) * 0.05
    gq, gk = rng.uniform(0.5, 1.5, HD), rng.uniform(0.5, 1.5, HD)
    m = CacheModel(H, D, Tc, W)
    hid = {}
    for c in range(7):
        hid[c] = rng.standard_normal((Tc, HD))
        if c > W:
            m.evict(c - W)
        q, k, v = orc.project_chunk(hid[c], w_qkv, gq, gk, c, H, D, tpf, cf, gw)
        assert q.shape == k.shape == v.shape == (Tc, H, D)
        m.append(c, k, v)
    ids = m.present_chunks()
    assert ids == [0, 5, 6]
    K0, V0 = m.physical()
    k, v = orc.recache(np.concatenate([hid[c] for c in ids]), w_qkv[:, HD:], gk, ids, H, D, tpf,
                       cf, gw)
    m.recache(ids, k, v)
    K1, V1 = m.physical()
    assert np.allclose(K1, K0, rtol=0, atol=1e-12) and np.allclose(V1, V0, rtol=0, atol=1e-12)
    # and Q is the K rule applied to the Q columns with Q's gain
    q, _, _ = orc.project_chunk(hid[6], w_qkv, gq, gk, 6, H, D, tpf, cf, gw)
    qq, _ = orc.recache(hid[6], np.concatenate([w_qkv[:, :HD], w_qkv[:, :HD]], axis=1), gq, [6],
                        H, D, tpf, cf, gw)
    assert np.allclose(q, qq, rtol=0, atol=1e-12)


def test_recache_with_shot_offsets_equals_appended_projections():
    """Multi-shot positions: chunks projected at frame0 = c*cf + shot*offset
    and appended (a shot boundary at chunk 5) are reproduced by a recache that
    takes each region's frame0 from the cache model."""
    from oracle.cache_model import CacheModel
    rng = np.random.default_rng(6)
    H, D, tpf, cf, gw, W, off = 2, 64, 16, 2, 4, 2, 11
    Tc, HD = tpf * cf, H * D
    w_qkv = rng.standard_normal((HD, 3 * HD)) * 0.05
    gk = rng.uniform(0.5, 1.5, HD)
    m = CacheModel(H, D, Tc, W, chunk_frames=cf, rope_offset_frames=off)
    hid = {}
    for c in range(7):
        hid[c] = rng.standard_normal((Tc, HD))
        if (c - W) in m.window_chunks():
            m.evict(c - W)
        shot = c == 5
        f0 = c * cf + (m.shot + (1 if shot else 0)) * off
        _, k, v = orc.project_chunk(hid[c], w_qkv, None, gk, c, H, D, tpf, cf, gw, frame0=f0)
        (m.append_shot if shot else m.append)(c, k, v)
        assert m.frame0[c] == f0
    ids = m.present_chunks()
    assert ids == [5, 6] and m.chunk_of_region == [5, -1, 6]
    K0, V0 = m.physical(fill=0.0)
    k, v = orc.recache(np.concatenate([hid[c] for c in ids]), w_qkv[:, HD:], gk, ids, H, D, tpf,
                       cf, gw, frame0=[m.frame0[c] for c in ids])
    m.recache(ids, k, v)
    K1, V1 = m.physical(fill=0.0)
    assert np.allclose(K1, K0, rtol=0, atol=1e-12) and np.allclose(V1, V0, rtol=0, atol=1e-12)
    # the offset matters: absolute positions give different keys
    k_abs, _ = orc.recache(np.concatenate([hid[c] for c in ids]), w_qkv[:, HD:], gk, ids, H, D,
                           tpf, cf, gw)
    assert np.max(np.abs(k_abs - k)) > 1e-3
