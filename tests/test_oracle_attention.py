"""Pins for the attention oracle and the cache model (CPU only).

Brute-force pure-Python loops on the small case, a full block-causal masked
softmax over the whole sequence (a different formulation) when the window
covers every chunk, closed forms (one key, Q = 0), and the invariants the
frame-sink / short-window description fixes.
"""

import math

import numpy as np
import pytest

from oracle import attention as oatt
from oracle.cache_model import (CacheModel, CacheStateError, region_of_chunk,
                                visible_chunks_of_step)
from synth import TINY, LAYER_1P3B, bf16_to_f64, chunk_qkv


def _brute_attention(q, k, v, scale):
    """Pure-Python loops: q [Tq][H][D], k, v [L][H][D] nested lists/arrays."""
    Tq, H, D = len(q), len(q[0]), len(q[0][0])
    L = len(k)
    out = [[[0.0] * D for _ in range(H)] for _ in range(Tq)]
    for h in range(H):
        for i in range(Tq):
            logits = []
            for j in range(L):
                acc = 0.0
                for d in range(D):
                    acc += float(q[i][h][d]) * float(k[j][h][d])
                logits.append(acc * scale)
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            for d in range(D):
                acc = 0.0
                for j in range(L):
                    acc += w[j] * float(v[j][h][d])
                out[i][h][d] = acc / z
    return np.array(out)


def _stream_tiny(n_chunks=6, W=TINY.window_chunks, dist="rms1"):
    sh = TINY
    m = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, W)
    steps = []
    for c in range(n_chunks):
        q, k, v = chunk_qkv(sh, 0, 0, c, dist)
        if c > W:
            m.evict(c - W)
        m.append(c, bf16_to_f64(k), bf16_to_f64(v))
        steps.append((c, bf16_to_f64(q), m.present_chunks(), *m.visible_kv()))
    return steps


def test_brute_force_tiny_stream():
    scale = 1.0 / math.sqrt(TINY.head_dim)
    sh = TINY
    m = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks)
    for c in range(6):
        q, k, v = (bf16_to_f64(t) for t in chunk_qkv(sh, 0, 0, c, "rms1"))
        if c > sh.window_chunks:
            m.evict(c - sh.window_chunks)
        m.append(c, k, v)
        got = oatt.sinkwin_attention(m, q, scale)
        kk, vv = m.visible_kv()
        rows = [0, 7, 31] if c != 3 else list(range(32))
        want = _brute_attention(q[rows], kk, vv, scale)
        assert np.allclose(got[rows], want, rtol=0, atol=1e-12)


def _block_causal_full(q_all, k_all, v_all, Tc, scale):
    """Masked softmax over the whole concatenated sequence: query token i may see
    key token j iff chunk(j) <= chunk(i)."""
    T, H, D = q_all.shape
    ci = np.arange(T) // Tc
    mask = ci[None, :] <= ci[:, None]
    out = np.empty_like(q_all)
    for h in range(H):
        s = (q_all[:, h, :] @ k_all[:, h, :].T) * scale
        s = np.where(mask, s, -np.inf)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v_all[:, h, :]
    return out


def test_window_covering_all_chunks_equals_block_causal():
    n = 5
    sh = TINY
    scale = 1.0 / math.sqrt(sh.head_dim)
    m = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, window_chunks=n)  # W >= all
    qs, ks, vs, outs = [], [], [], []
    for c in range(n):
        q, k, v = (bf16_to_f64(t) for t in chunk_qkv(sh, 0, 0, c, "rms1"))
        m.append(c, k, v)
        qs.append(q), ks.append(k), vs.append(v)
        outs.append(oatt.sinkwin_attention(m, q, scale))
    full = _block_causal_full(np.concatenate(qs), np.concatenate(ks), np.concatenate(vs),
                              sh.chunk_tokens, scale)
    assert np.allclose(np.concatenate(outs), full, rtol=0, atol=1e-12)


def test_probabilities_sum_to_one():
    for c, q, _, k, v in _stream_tiny():
        p = oatt.attention_probs(q, k, 0.125)
        assert np.allclose(p.sum(axis=2), 1.0, atol=1e-12)
        assert np.all(p >= 0)


def test_single_key_returns_v_and_zero_query_returns_mean():
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, 2, 16))
    v = rng.standard_normal((1, 2, 16))
    q = rng.standard_normal((5, 2, 16))
    assert np.allclose(oatt.attention(q, k, v, 0.3), np.broadcast_to(v, (5, 2, 16)), atol=0)
    k = rng.standard_normal((40, 2, 16))
    v = rng.standard_normal((40, 2, 16))
    o = oatt.attention(np.zeros((3, 2, 16)), k, v, 0.3)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=0), (3, 2, 16)), atol=1e-14)


def test_key_permutation_invariance():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((9, 3, 32))
    k = rng.standard_normal((50, 3, 32))
    v = rng.standard_normal((50, 3, 32))
    perm = rng.permutation(50)
    a = oatt.attention(q, k, v, 0.2)
    b = oatt.attention(q, k[perm], v[perm], 0.2)
    assert np.allclose(a, b, atol=1e-13)


def test_evicted_chunk_has_no_influence_and_sink_always_does():
    sh = TINY
    W = sh.window_chunks
    scale = 0.125
    base = _stream_tiny()
    for c, q, present, k, v in base:
        assert present[0] == 0  # the sink is always there
        assert present == visible_chunks_of_step(c, W)
    # perturb an evicted chunk (chunk 1 is gone from step W+1 on): outputs identical
    m1 = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, W)
    m2 = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, W)
    m3 = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, W)
    for c in range(6):
        q, k, v = (bf16_to_f64(t) for t in chunk_qkv(sh, 0, 0, c, "rms1"))
        if c > W:
            for mm in (m1, m2, m3):
                mm.evict(c - W)
        k2, v2 = (k + 3.0, v - 2.0) if c == 1 else (k, v)
        k3, v3 = (k * 0.5 + 1.0, v + 1.0) if c == 0 else (k, v)
        m1.append(c, k, v), m2.append(c, k2, v2), m3.append(c, k3, v3)
        o1 = oatt.sinkwin_attention(m1, q, scale)
        o2 = oatt.sinkwin_attention(m2, q, scale)
        o3 = oatt.sinkwin_attention(m3, q, scale)
        if 1 not in m1.present_chunks():
            assert np.array_equal(o1, o2)  # bit-identical
        else:
            assert not np.allclose(o1, o2)
        assert np.max(np.abs(o1 - o3)) > 1e-3  # the sink changes every step


@pytest.mark.parametrize("sh,want", [
    (TINY, [32, 64, 96, 96, 96, 96]),
    (LAYER_1P3B, [4680, 9360, 14040, 18720, 18720, 18720]),
])
def test_kv_length_table(sh, want):
    m = CacheModel(1, 16, sh.chunk_tokens, sh.window_chunks)
    got = []
    z = np.zeros((sh.chunk_tokens, 1, 16))
    for c in range(6):
        if c > sh.window_chunks:
            m.evict(c - sh.window_chunks)
        m.append(c, z, z)
        got.append(m.kv_length())
    assert got == want


def test_slot_rule_and_physical_layout():
    W, Tc = 3, 4
    assert [region_of_chunk(c, W) for c in range(9)] == [0, 1, 2, 3, 1, 2, 3, 1, 2]
    m = CacheModel(1, 16, Tc, W)
    for c in range(7):
        if c > W:
            m.evict(c - W)
        m.append(c, np.full((Tc, 1, 16), float(c)), np.full((Tc, 1, 16), -float(c)))
    assert m.chunk_of_region == [0, 4, 5, 6]
    K, V = m.physical()
    assert np.array_equal(K[:, 0, 0], np.repeat([0.0, 4.0, 5.0, 6.0], Tc))
    assert np.array_equal(V[:, 0, 0], -np.repeat([0.0, 4.0, 5.0, 6.0], Tc))


def test_state_errors():
    m = CacheModel(1, 16, 2, 2)
    z = np.zeros((2, 1, 16))
    with pytest.raises(CacheStateError):
        m.append(1, z, z)  # sink first
    m.append(0, z, z)
    m.append(0, z, z)  # re-append newest: overwrite
    with pytest.raises(CacheStateError):
        m.append(2, z, z)  # skips chunk 1
    m.append(1, z, z)
    m.append(2, z, z)
    with pytest.raises(CacheStateError):
        m.append(3, z, z)  # slot of chunk 1 still occupied
    with pytest.raises(CacheStateError):
        m.evict(0)  # sink
    with pytest.raises(CacheStateError):
        m.evict(2)  # not the oldest
    m.evict(1)
    with pytest.raises(CacheStateError):
        m.evict(1)
    m.append(3, z, z)
    with pytest.raises(CacheStateError):
        m.recache([0, 3, 2], np.zeros((6, 1, 16)), np.zeros((6, 1, 16)))
    m.recache([0, 2, 3], np.ones((6, 1, 16)), np.ones((6, 1, 16)))
    assert m.k[3][0, 0, 0] == 1.0


def test_window_of_one_chunk_streams():
    """W = 1: the window holds only the current chunk; evicting it empties the
    window and the next chunk still follows the last one appended."""
    m = CacheModel(1, 16, 2, 1)
    z = np.zeros((2, 1, 16))
    m.append(0, z, z)
    for c in range(1, 6):
        if c > 1:
            with pytest.raises(CacheStateError):
                m.append(c, z, z)  # slot still holds c - 1
            m.evict(c - 1)
            with pytest.raises(CacheStateError):
                m.append(c - 1, z, z)  # evicted: cannot come back
        m.append(c, z, z)
        m.append(c, z, z)  # overwrite while cached
        assert m.chunk_of_region == [0, c]
        assert m.present_chunks() == visible_chunks_of_step(c, 1)


def test_attention_rows_against_brute_force_and_full_attention():
    """attention_rows (the expected value of every sampled full-size parity
    test) against pure-Python loops on a small case, and against the full
    attention() for random row and head subsets, including heads=None."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal((9, 3, 8))
    k = rng.standard_normal((13, 3, 8))
    v = rng.standard_normal((13, 3, 8))
    rows, heads = [8, 0, 5], [2, 0]
    got = oatt.attention_rows(q, k, v, 0.4, rows, heads)
    brute = _brute_attention(q, k, v, 0.4)
    assert got.shape == (3, 2, 8)
    assert np.allclose(got, brute[rows][:, heads], rtol=0, atol=1e-13)
    sh = LAYER_1P3B
    q, k, v = (bf16_to_f64(t) for t in chunk_qkv(sh, 1, 0, 0, "rms1", q_rows=300))
    full = oatt.attention(q, k, v, 1.0 / math.sqrt(sh.head_dim))
    for trial in range(3):
        rows = rng.choice(300, size=17, replace=False)
        heads = None if trial == 0 else list(rng.choice(sh.heads, size=5, replace=False))
        got = oatt.attention_rows(q, k, v, 1.0 / math.sqrt(sh.head_dim), rows, heads)
        want = full[rows] if heads is None else full[rows][:, heads]
        assert np.allclose(got, want, rtol=0, atol=1e-13)


def test_pool_matches_single_process():
    """oracle.pool spreads attention_rows over spawned processes; the result
    equals one call up to the library matmul's summation order."""
    from oracle.pool import attention_rows_parallel
    rng = np.random.default_rng(12)
    q = rng.standard_normal((50, 3, 16))
    k = rng.standard_normal((70, 3, 16))
    v = rng.standard_normal((70, 3, 16))
    rows = [49, 3, 17, 0, 25]
    got = attention_rows_parallel(q, k, v, 0.3, rows, workers=2, rows_per_unit=2)
    assert np.allclose(got, oatt.attention_rows(q, k, v, 0.3, rows), rtol=0, atol=1e-14)


def _shot_stream(m, n_chunks, shots, k_of, v_of):
    """Stream chunks 0..n_chunks-1 through a CacheModel; chunks in `shots` open
    a new shot.  Step c evicts c - W when it is in the window."""
    for c in range(n_chunks):
        if (c - m.W) in m.window_chunks():
            m.evict(c - m.W)
        (m.append_shot if c in shots else m.append)(c, k_of(c), v_of(c))
        yield c


def test_multi_shot_sink_state_and_positions():
    """Multi-shot sink: the first chunk of a new shot becomes the sink and the
    old sink leaves; the window keeps the previous shot's recent chunks; the
    new sink's own ring slot stays unused; positions shift by the RoPE offset
    at every boundary after chunk 0."""
    W, Tc, cf, off = 2, 2, 3, 7
    m = CacheModel(1, 16, Tc, W, chunk_frames=cf, rope_offset_frames=off)
    z = lambda c: np.full((Tc, 1, 16), float(c))
    seen = {}
    for c in _shot_stream(m, 9, {0, 5}, z, z):
        seen[c] = (list(m.chunk_of_region), m.present_chunks(), m.frame0_of_region())
    assert seen[4][0] == [0, 3, 4]
    assert seen[5][0] == [5, -1, 4]           # 3 evicted, 5 is the sink, 0 gone
    assert seen[5][1] == [5, 4]
    assert seen[6][0] == [5, -1, 6]           # 4 evicted; 6 in slot (6-1) % 2
    assert seen[7][0] == [5, 7, 6]            # 5 is the sink, not evicted; 7 in 5's old slot
    assert seen[8][0] == [5, 7, 8]
    assert seen[4][2] == [0, 9, 12]           # frame0 = c*cf before the boundary
    assert seen[8][2] == [5 * cf + off, 7 * cf + off, 8 * cf + off]
    with pytest.raises(CacheStateError):
        m.evict(5)                            # the shot's sink is never evicted
    with pytest.raises(CacheStateError):
        m.append_shot(7, z(7), z(7))          # a shot starts at the next chunk only
    m.append_shot(9, z(9), z(9))
    assert m.chunk_of_region[0] == 9 and m.shot == 2 and m.frame0[9] == 9 * cf + 2 * off
    m.append_shot(9, z(9), z(9))              # overwrite of the shot's own sink
    assert m.shot == 2
    m.append(9, z(9), z(9))                   # the same through the plain append
    assert m.chunk_of_region[0] == 9


def _masked_full(q_all, k_all, v_all, Tc, visible, scale):
    """Masked softmax over the whole sequence: query chunk i sees key chunk j iff
    visible(i, j)."""
    T, H, D = q_all.shape
    ci = np.arange(T) // Tc
    n = T // Tc
    vis = np.array([[visible(i, j) for j in range(n)] for i in range(n)])
    mask = vis[ci][:, ci]
    out = np.empty_like(q_all)
    for h in range(H):
        s = (q_all[:, h, :] @ k_all[:, h, :].T) * scale
        s = np.where(mask, s, -np.inf)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v_all[:, h, :]
    return out


def test_multi_shot_window_covering_all_equals_masked_full_attention():
    """With a window wider than the stream, a multi-shot cache shows query
    chunk i every key chunk j <= i except the sinks of earlier shots: the
    oracle's step outputs equal one masked softmax over the whole sequence."""
    sh = TINY
    n, shots = 7, {0, 3, 5}
    scale = 1.0 / math.sqrt(sh.head_dim)
    m = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, window_chunks=n)
    data = {c: tuple(bf16_to_f64(t) for t in chunk_qkv(sh, 0, 0, c, "rms1")) for c in range(n)}
    outs = []
    for c in _shot_stream(m, n, shots, lambda c: data[c][1], lambda c: data[c][2]):
        outs.append(oatt.sinkwin_attention(m, data[c][0], scale))
    starts = sorted(shots)

    def visible(i, j):
        cur = max(s for s in starts if s <= i)
        return j <= i and (j not in starts or j == cur)

    full = _masked_full(*(np.concatenate([data[c][t] for c in range(n)]) for t in range(3)),
                        sh.chunk_tokens, visible, scale)
    assert np.allclose(np.concatenate(outs), full, rtol=0, atol=1e-12)


def test_multi_shot_old_sink_has_no_influence_new_sink_always_does():
    sh = TINY
    scale = 0.125
    W = sh.window_chunks
    rng = np.random.default_rng(21)
    data = {c: tuple(bf16_to_f64(t) for t in chunk_qkv(sh, 0, 1, c, "rms1")) for c in range(8)}
    bump = lambda c, which, d: data[c][which] + (d if c == which_chunk[0] else 0.0)
    outs = {}
    for variant, which_chunk in (("base", [-1]), ("old", [0]), ("new", [4])):
        m = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, W)
        res = []
        for c in _shot_stream(m, 8, {0, 4}, lambda c: bump(c, 1, 3.0), lambda c: bump(c, 2, -2.0)):
            res.append(oatt.sinkwin_attention(m, data[c][0], scale))
        outs[variant] = res
    for c in range(4, 8):
        assert np.array_equal(outs["base"][c], outs["old"][c])  # old sink gone: bit-identical
        assert np.max(np.abs(outs["base"][c] - outs["new"][c])) > 1e-3  # new sink counts
    assert np.max(np.abs(outs["base"][2] - outs["old"][2])) > 1e-3
    del rng
