"""Pins of the fp64 CPU oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a closed form,
an invariant, a hand-worked case, a brute-force scalar loop on a tiny input, or a
number printed on one of the pages (tests/golden/page_figures.json).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")
rng = np.random.default_rng(12345)


def bf16_round(x):
    """Round float64 values to bf16 (RNE) so test inputs are representable."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return O.bf16_bits_to_f64(u.astype(np.uint16))


# ----------------------------------------------------------------------------- bf16

def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x0001, 0x3FC0, 0x4049], np.uint16)
    v = O.bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 0.0
    assert math.copysign(1.0, v[3]) == -1.0 and v[3] == 0.0
    assert math.isinf(v[4]) and v[4] > 0
    assert v[5] == 2.0 ** -133          # smallest bf16 subnormal
    assert v[6] == 1.5
    assert v[7] == 3.140625


# ----------------------------------------------------------------------------- LSE

def test_lse_two_key_closed_form():
    # x = [q.k0, q.k1] / sqrt(4) = [1, 0]  ->  LSE = ln(e + 1); a 1/d scale would give 0.5.
    q = np.zeros((1, 1, 1, 4)); q[0, 0, 0, 0] = 2.0
    k = np.zeros((1, 1, 2, 4)); k[0, 0, 0, 0] = 1.0
    out = O.lse(q, k, None)
    assert abs(out[0, 0, 0] - math.log(math.e + 1.0)) < 1e-15


def test_lse_zero_queries_count_visible_keys():
    # q = 0: every visible logit is 0, so LSE_j = ln(#visible) = ln(off + j + 1).
    L, Hq, Hkv, d, T, nt, nq = 2, 4, 2, 8, 7, 5, 4
    q = np.zeros((L, Hq, nq, d))
    kc = rng.normal(size=(L, Hkv, T, d)); kt = rng.normal(size=(L, Hkv, nt, d))
    out = O.lse(q, kc, kt)
    off = T + nt - nq
    want = np.log(off + np.arange(nq) + 1.0)
    assert np.allclose(out, np.broadcast_to(want, out.shape), atol=1e-14, rtol=0)


def test_lse_first_query_sees_one_key():
    # Self-attention (n_q == n_k): query 0 sees key 0 only, so LSE_0 = q_0.k_0/sqrt(d).
    d = 16
    q = rng.normal(size=(1, 1, 3, d)); k = rng.normal(size=(1, 1, 3, d))
    out = O.lse(q, k, None)
    assert abs(out[0, 0, 0] - float(q[0, 0, 0] @ k[0, 0, 0]) / 4.0) < 1e-13


def test_lse_rows_sum_to_one_bruteforce():
    # Sum over visible keys of exp(x_ji - LSE_j) with scalar loops equals 1.
    L, Hq, Hkv, d, T, nt, nq = 1, 2, 1, 8, 6, 4, 5
    q = rng.normal(size=(L, Hq, nq, d)) * 2
    kc = rng.normal(size=(L, Hkv, T, d)); kt = rng.normal(size=(L, Hkv, nt, d))
    out = O.lse(q, kc, kt)
    keys = np.concatenate([kc, kt], 2)[0, 0]
    off = T + nt - nq
    for h in range(Hq):
        for j in range(nq):
            s = 0.0
            for i in range(off + j + 1):
                dot = sum(q[0, h, j, c] * keys[i, c] for c in range(d))
                s += math.exp(dot / math.sqrt(d) - out[0, h, j])
            assert abs(s - 1.0) < 1e-12


def test_lse_gqa_group_mapping():
    # KV head 1 has all-zero keys: query heads 2 and 3 (group of KV head 1 under
    # contiguous grouping) get ln(#visible); heads 0 and 1 do not.
    L, Hq, Hkv, d, T, nq = 1, 4, 2, 8, 6, 6
    q = rng.normal(size=(L, Hq, nq, d)) * 3
    k = rng.normal(size=(L, Hkv, T, d)) * 3
    k[:, 1] = 0.0
    out = O.lse(q, k, None)
    want = np.log(np.arange(nq) + 1.0)
    assert np.allclose(out[0, 2], want) and np.allclose(out[0, 3], want)
    assert not np.allclose(out[0, 0], want) and not np.allclose(out[0, 1], want)


def test_lse_large_logits_stable():
    # All keys equal: LSE = c + ln(#visible) even when c is huge.
    d = 4
    q = np.full((1, 1, 3, d), 40.0); k = np.full((1, 1, 5, d), 30.0)
    out = O.lse(q, k, None)
    c = 40.0 * 30.0 * d / 2.0
    assert np.allclose(out[0, 0], c + np.log(np.arange(3) + 3.0), rtol=1e-15, atol=1e-9)


# ----------------------------------------------------------------------------- KVzip / KVzip+

def test_kvzip_zero_queries_closed_form():
    # q = 0: a_ji = 1/(off+j+1) for every visible key; the max over j is at j = 0.
    L, Hq, Hkv, d, T, nt, nq = 1, 4, 2, 8, 9, 6, 5
    q = np.zeros((L, Hq, nq, d))
    kc = rng.normal(size=(L, Hkv, T, d)); kt = rng.normal(size=(L, Hkv, nt, d))
    s = O.kvzip_score(q, kc, kt)
    off = T + nt - nq
    assert np.allclose(s, -math.log(off + 1.0), atol=1e-14)


def test_kvzip_plus_factors_closed_form():
    # q = 0 with varying ||W_O v_i|| and ||h_j||:
    # s+_i = vn_i * max_j 1 / ((off + j + 1) * ||h_j||)   (a product, not a ratio inverted).
    L, Hq, Hkv, d, T, nt, nq, Dh = 1, 2, 1, 4, 5, 3, 3, 6
    q = np.zeros((L, Hq, nq, d))
    kc = rng.normal(size=(L, Hkv, T, d)); kt = rng.normal(size=(L, Hkv, nt, d))
    vn = rng.uniform(0.5, 3.0, size=(L, Hq, T))
    h = rng.normal(size=(L, nq, Dh)) * rng.uniform(0.2, 5.0, size=(1, nq, 1))
    s = O.kvzip_score(q, kc, kt, vnorm=vn, h=h)
    off = T + nt - nq
    hn = [math.sqrt(sum(x * x for x in h[0, j])) for j in range(nq)]
    best_j = max(1.0 / ((off + j + 1) * hn[j]) for j in range(nq))
    for i in range(T):
        want = math.log(max(vn[0, 0, i], vn[0, 1, i]) * best_j)
        assert abs(s[0, 0, i] - want) < 1e-13


def test_kvzip_one_hot_copy_orthogonal_keys():
    # Orthonormal basis keys; query j of head h points at key pi_h(j) with logit c.
    # Visible count n_j = off + j + 1; the pointed key gets e^c/(e^c + n_j - 1), the
    # others 1/(e^c + n_j - 1).  Score = max over j and over the group's heads.
    d = 16; T = 6; nt = 4; nq = 3; Hq = 2
    keys = np.eye(d)[: T + nt]
    kc = keys[:T][None, None]; kt = keys[T:][None, None]
    beta = 8.0
    c = beta / math.sqrt(d)
    pis = [[0, 3, 3], [5, 1, 0]]
    q = np.zeros((1, Hq, nq, d))
    for h in range(Hq):
        for j in range(nq):
            q[0, h, j, pis[h][j]] = beta
    s = O.kvzip_score(q, kc, kt, log=False)
    off = T + nt - nq
    for i in range(T):
        best = 0.0
        for h in range(Hq):
            for j in range(nq):
                n = off + j + 1
                a = (math.exp(c) if pis[h][j] == i else 1.0) / (math.exp(c) + n - 1)
                best = max(best, a)
        assert abs(s[0, 0, i] - best) < 1e-14
    assert s.max() < 1.0 and s.min() > 0.0


def test_kvzip_score_in_unit_interval_and_attains_max():
    L, Hq, Hkv, d, T, nt, nq = 2, 4, 2, 16, 20, 9, 7
    q = rng.normal(size=(L, Hq, nq, d)) * 2
    kc = rng.normal(size=(L, Hkv, T, d)) * 2; kt = rng.normal(size=(L, Hkv, nt, d))
    s = O.kvzip_score(q, kc, kt, log=False)
    assert (s > 0).all() and (s <= 1).all()
    # brute force on one (layer, kv head): scalar-loop softmax rows, max over j and heads
    keys = np.concatenate([kc, kt], 2)
    off = T + nt - nq
    l, hk = 1, 1
    for i in range(0, T, 3):
        best = 0.0
        for hq in (2, 3):
            for j in range(nq):
                xs = [float(q[l, hq, j] @ keys[l, hk, t]) / 4.0 for t in range(off + j + 1)]
                m = max(xs)
                den = sum(math.exp(x - m) for x in xs)
                best = max(best, math.exp(xs[i] - m) / den)
        assert abs(s[l, hk, i] - best) < 1e-14


def test_kvzip_chunked_is_max_over_chunks():
    L, Hq, Hkv, d, T = 1, 2, 1, 8, 10
    kc = rng.normal(size=(L, Hkv, T, d))
    qs = [rng.normal(size=(L, Hq, 4, d)) for _ in range(3)]
    tails = [rng.normal(size=(L, Hkv, n, d)) for n in (6, 9, 9)]
    sc = O.kvzip_score_chunked(qs, kc, tails)
    per = np.stack([O.kvzip_score(qs[c], kc, tails[c]) for c in range(3)])
    assert np.array_equal(sc, per.max(axis=0))


def test_kvzip_chunked_zero_queries_closed_form():
    """q = 0: every visible key gets 1 / (number of keys the query sees).  Chunk c's
    query j sees the T context keys, the chunk's tail before its block and the block up
    to j: T + (tail_c - n) + j + 1 keys, so the score of a context key is the max over
    chunks of 1 / (T + tail_c - n + 1): the chunk with the shortest tail decides.  With
    constant value norms vn and hidden norms hn the KVzip+ score is that times vn / hn."""
    L, Hq, Hkv, d, T, n = 1, 4, 2, 8, 13, 5
    kc = rng.normal(size=(L, Hkv, T, d))
    tails_len = (n + 3, n + 7, n + 2)          # prefix + carry + block; chunk 2 is shortest
    qs = [np.zeros((L, Hq, n, d)) for _ in tails_len]
    tails = [rng.normal(size=(L, Hkv, m, d)) for m in tails_len]
    s = O.kvzip_score_chunked(qs, kc, tails, log=False)
    assert np.allclose(s, 1.0 / (T + min(tails_len) - n + 1), rtol=0, atol=1e-14)
    vn = np.full((L, Hq, T), 3.0)
    hs = [np.full((L, n, 16), 0.5) for _ in tails_len]   # ||h_j|| = 0.5 * 4 = 2
    s_plus = O.kvzip_score_chunked(qs, kc, tails, vnorm=vn, h_chunks=hs, log=False)
    assert np.allclose(s_plus, s * 3.0 / 2.0, rtol=1e-13, atol=0)


def test_kvzip_chunked_copy_in_one_chunk():
    """A query of chunk 1 (one head of the group) that copies context key i with a large
    gain gives s_i -> 1, whichever chunk it sits in; the other keys stay far below it."""
    L, Hq, Hkv, d, T, n = 1, 2, 1, 16, 12, 4
    kc = np.eye(d)[None, None, :T] * 1.0             # orthonormal context keys
    tails = [np.zeros((L, Hkv, n + 2, d)) for _ in range(3)]
    qs = [np.zeros((L, Hq, n, d)) for _ in range(3)]
    qs[1][0, 1, 2] = 60.0 * np.sqrt(d) * kc[0, 0, 7]  # chunk 1, head 1, query 2 copies key 7
    s = O.kvzip_score_chunked(qs, kc, tails, log=False)
    assert s[0, 0, 7] > 1 - 1e-12
    others = np.delete(s[0, 0], 7)
    assert (others < 0.1).all()


# ----------------------------------------------------------------------------- future mass

def test_future_mass_zero_queries_harmonic():
    # q = 0, causal: a_ji = 1/(j+1); f_i = g * sum_{j=i+w}^{n-1} 1/(j+1).
    L, Hq, Hkv, d, n, w = 1, 4, 2, 8, 12, 3
    q = np.zeros((L, Hq, n, d)); k = rng.normal(size=(L, Hkv, n, d))
    f = O.future_attention_mass(q, k, w)
    g = Hq // Hkv
    for i in range(n):
        want = g * sum(1.0 / (j + 1) for j in range(i + w, n))
        assert abs(f[0, 0, i] - want) < 1e-13 and abs(f[0, 1, i] - want) < 1e-13


def test_future_mass_w0_rows_sum_to_one():
    L, Hq, Hkv, d, n = 2, 4, 2, 16, 17
    q = rng.normal(size=(L, Hq, n, d)) * 2; k = rng.normal(size=(L, Hkv, n, d)) * 2
    f = O.future_attention_mass(q, k, 0, row_block=5)
    g = Hq // Hkv
    assert np.allclose(f.sum(axis=-1), g * n, rtol=1e-13)


def test_future_mass_window_limits():
    L, Hq, Hkv, d, n = 1, 2, 1, 8, 9
    q = rng.normal(size=(L, Hq, n, d)); k = rng.normal(size=(L, Hkv, n, d))
    assert np.all(O.future_attention_mass(q, k, n) == 0.0)
    assert np.all(O.future_attention_mass(q, k, n + 5) == 0.0)
    f2 = O.future_attention_mass(q, k, 2)
    assert np.all(f2[..., n - 2:] == 0.0) and np.all(f2[..., : n - 2] > 0.0)


def test_future_mass_one_hot_orthogonal():
    # Orthonormal keys, query j points at key p_j <= j with logit c: row j puts
    # e^c/(e^c + j) on p_j and 1/(e^c + j) on every other key i <= j.
    n, d, w = 7, 8, 2
    k = np.eye(d)[:n][None, None]
    beta = 6.0; c = beta / math.sqrt(d)
    p = [0, 0, 1, 0, 2, 4, 4]
    q = np.zeros((1, 1, n, d))
    for j in range(n):
        q[0, 0, j, p[j]] = beta
    f = O.future_attention_mass(q, k, w)
    for i in range(n):
        want = 0.0
        for j in range(i + w, n):
            want += (math.exp(c) if p[j] == i else 1.0) / (math.exp(c) + j)
        assert abs(f[0, 0, i] - want) < 1e-14


# ----------------------------------------------------------------------------- norms

def test_value_norm_orthonormal_columns_and_head_slices():
    # W_O^{(h)} = c_h * (orthonormal columns)  =>  ||W_O^{(h)} v|| = c_h ||v||, with
    # query head h reading KV head h // g.
    L, Hkv, Hq, T, d, Dh = 1, 2, 4, 5, 4, 12
    v = rng.normal(size=(L, Hkv, T, d)) * np.array([1.0, 3.0])[None, :, None, None]
    w_o = np.zeros((L, Dh, Hq * d))
    cs = [0.5, 1.0, 2.0, 4.0]
    for h in range(Hq):
        Qm, _ = np.linalg.qr(rng.normal(size=(Dh, d)))
        w_o[0, :, h * d:(h + 1) * d] = cs[h] * Qm
    vn = O.value_norm(v, w_o, Hq)
    for h in range(Hq):
        for i in range(T):
            want = cs[h] * math.sqrt(sum(x * x for x in v[0, h // 2, i]))
            assert abs(vn[0, h, i] - want) < 1e-12 * max(1.0, want)


def test_value_norm_gram_identity():
    # ||W v||^2 = v^T (W^T W) v  -- an independent route through the Gram matrix.
    L, Hkv, Hq, T, d, Dh = 2, 1, 3, 6, 8, 20
    v = rng.normal(size=(L, Hkv, T, d)); w_o = rng.normal(size=(L, Dh, Hq * d))
    vn = O.value_norm(v, w_o, Hq)
    for l in range(L):
        for h in range(Hq):
            Wh = w_o[l][:, h * d:(h + 1) * d]
            G = Wh.T @ Wh
            for i in range(T):
                quad = float(v[l, 0, i] @ G @ v[l, 0, i])
                assert abs(vn[l, h, i] ** 2 - quad) < 1e-10 * quad


def test_hidden_norm_pythagoras():
    h = np.array([[[3.0, 4.0, 0.0], [5.0, 12.0, 0.0], [0.0, 0.0, 0.0]]])
    assert np.array_equal(O.hidden_norm(h), np.array([[5.0, 13.0, 0.0]]))


# ----------------------------------------------------------------------------- surrogate

def test_surrogate_zero_weight_gives_bias_head_major():
    L, T, Dh, H = 2, 5, 6, 3
    h = rng.normal(size=(L, T, Dh)); W = np.zeros((L, Dh, H)); b = rng.normal(size=(L, H))
    z = O.linear_surrogate(h, W, b)
    assert z.shape == (L, H, T)
    assert np.array_equal(z, np.broadcast_to(b[:, :, None], (L, H, T)))


def test_surrogate_one_hot_weight_selects_channel():
    L, T, Dh, H = 1, 4, 7, 3
    h = rng.normal(size=(L, T, Dh)); b = np.array([[1.0, -2.0, 0.5]])
    W = np.zeros((L, Dh, H)); chan = [6, 0, 3]
    for hh in range(H):
        W[0, chan[hh], hh] = 1.0
    z = O.linear_surrogate(h, W, b)
    for hh in range(H):
        for t in range(T):
            assert z[0, hh, t] == h[0, t, chan[hh]] + b[0, hh]


def test_surrogate_small_integers_exact():
    L, T, Dh, H = 1, 6, 9, 4
    hi = rng.integers(-8, 9, size=(L, T, Dh)); Wi = rng.integers(-8, 9, size=(L, Dh, H))
    bi = rng.integers(-50, 50, size=(L, H))
    z = O.linear_surrogate(hi.astype(float), Wi.astype(float), bi.astype(float))
    for hh in range(H):
        for t in range(T):
            want = sum(int(hi[0, t, c]) * int(Wi[0, c, hh]) for c in range(Dh)) + int(bi[0, hh])
            assert z[0, hh, t] == want


# ------------------------------------------------------------------ attention forward

def test_attention_forward_uniform_rows_give_causal_means():
    # q = 0: every visible key gets weight 1/(off+j+1), so o_j is the mean of the
    # values it sees (bottom-right causal)
    L, Hkv, g, d, T, nt, nq = 1, 2, 2, 4, 5, 3, 4
    v_ctx = rng.normal(size=(L, Hkv, T, d)); v_tail = rng.normal(size=(L, Hkv, nt, d))
    k_ctx = rng.normal(size=(L, Hkv, T, d)); k_tail = rng.normal(size=(L, Hkv, nt, d))
    q = np.zeros((L, Hkv * g, nq, d))
    o, l_ = O.attention_forward(q, k_ctx, k_tail, v_ctx, v_tail)
    off = T + nt - nq
    vals = np.concatenate([v_ctx, v_tail], 2)
    for hq in range(Hkv * g):
        for j in range(nq):
            want = vals[0, hq // g, : off + j + 1].mean(axis=0)
            assert np.allclose(o[0, hq, j], want, rtol=0, atol=1e-13)
            assert abs(l_[0, hq, j] - math.log(off + j + 1)) < 1e-13


def test_attention_forward_constant_values_pass_through():
    L, Hkv, Hq, d, T, nt, nq = 2, 1, 3, 8, 9, 4, 6
    c = rng.normal(size=d)
    q = rng.normal(size=(L, Hq, nq, d)) * 2
    k_ctx = rng.normal(size=(L, Hkv, T, d)); k_tail = rng.normal(size=(L, Hkv, nt, d))
    v_ctx = np.broadcast_to(c, (L, Hkv, T, d)).copy(); v_tail = np.broadcast_to(c, (L, Hkv, nt, d)).copy()
    o, _ = O.attention_forward(q, k_ctx, k_tail, v_ctx, v_tail)
    assert np.allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


def test_attention_forward_one_hot_keys_copy_values():
    # orthonormal keys scaled by alpha and q_j = alpha * e_pi(j): the visible key pi(j)
    # takes essentially all the weight, so o_j = v_pi(j)
    d, n, alpha = 8, 8, 40.0
    keys = np.eye(n, d)[None, None] * alpha
    vals = rng.normal(size=(1, 1, n, d))
    pi = [0, 1, 0, 3, 2, 5, 4, 7]                       # pi(j) <= j: visible causally
    q = np.stack([np.eye(n, d)[p] * alpha for p in pi])[None, None]
    o, _ = O.attention_forward(q, keys, None, vals, None)
    for j, p in enumerate(pi):
        assert np.allclose(o[0, 0, j], vals[0, 0, p], rtol=0, atol=1e-9)


def test_attention_forward_brute_force_loops():
    L, Hkv, g, d, T, nt, nq = 1, 2, 2, 3, 4, 2, 3
    q = rng.normal(size=(L, Hkv * g, nq, d))
    k_ctx = rng.normal(size=(L, Hkv, T, d)); k_tail = rng.normal(size=(L, Hkv, nt, d))
    v_ctx = rng.normal(size=(L, Hkv, T, d)); v_tail = rng.normal(size=(L, Hkv, nt, d))
    o, l_ = O.attention_forward(q, k_ctx, k_tail, v_ctx, v_tail)
    nk = T + nt
    for hq in range(Hkv * g):
        kv = hq // g
        for j in range(nq):
            ws, vs = [], []
            for i in range(nk):
                if i > nk - nq + j:
                    continue
                k = k_ctx[0, kv, i] if i < T else k_tail[0, kv, i - T]
                v = v_ctx[0, kv, i] if i < T else v_tail[0, kv, i - T]
                ws.append(math.exp(sum(q[0, hq, j, c] * k[c] for c in range(d)) / math.sqrt(d)))
                vs.append(v)
            z = sum(ws)
            assert abs(l_[0, hq, j] - math.log(z)) < 1e-12
            for c in range(d):
                assert abs(o[0, hq, j, c] - sum(w * v[c] for w, v in zip(ws, vs)) / z) < 1e-12


# ------------------------------------------------------------------ value refit

def _refit_case(seed, T=12, n_q=7, g=2, d=4, keep=5):
    r = np.random.default_rng(seed)
    q = r.normal(size=(1, g, n_q, d)); k = r.normal(size=(1, 1, T, d)); v = r.normal(size=(1, 1, T, d))
    mask = np.zeros((1, 1, T), dtype=np.uint8)
    mask[0, 0, r.choice(T, keep, replace=False)] = 1
    return q, k, v, mask


def test_value_refit_keeping_everything_at_small_lambda_recovers_values():
    # with every key kept, A_S is the full softmax and V itself fits exactly; as lam -> 0
    # the ridge solution tends to V wherever A_S has full column rank (n >= T rows)
    q, k, v, _ = _refit_case(1, T=6, n_q=8, g=2)
    mask = np.ones((1, 1, 6), dtype=np.uint8)
    vv, _ = O.value_refit(q * 3, k, v, mask, 1e-12)
    assert np.allclose(vv[0][0], v[0, 0], rtol=0, atol=1e-4)


def test_value_refit_normal_equations_and_optimality():
    # the refit satisfies A^T (A V' - O) + lam V' = 0, and any perturbation raises the
    # ridge objective (it is strictly convex)
    q, k, v, mask = _refit_case(2)
    lam = 0.05
    vv, parts = O.value_refit(q, k, v, mask, lam)
    A, Ot = parts[0][0]
    Vp = vv[0][0]
    grad = A.T @ (A @ Vp - Ot) + lam * Vp
    assert np.abs(grad).max() < 1e-12
    f = lambda X: ((A @ X - Ot) ** 2).sum() + lam * (X ** 2).sum()
    r = np.random.default_rng(3)
    for _ in range(5):
        assert f(Vp + 1e-3 * r.normal(size=Vp.shape)) > f(Vp)


def test_value_refit_single_kept_key_closed_form():
    # one kept key: A_S is the all-ones column, so V' = sum_j O_j / (n + lam)
    q, k, v, _ = _refit_case(4, T=9, n_q=5, g=3)
    mask = np.zeros((1, 1, 9), dtype=np.uint8); mask[0, 0, 4] = 1
    lam = 0.3
    vv, _ = O.value_refit(q, k, v, mask, lam)
    x = (q[0].reshape(15, -1) @ k[0, 0].T) / 2.0
    a = np.exp(x - x.max(1, keepdims=True)); a /= a.sum(1, keepdims=True)
    Ot = a @ v[0, 0]
    assert np.allclose(vv[0][0][0], Ot.sum(0) / (15 + lam), rtol=0, atol=1e-12)


def test_value_refit_gqa_rows_and_kept_order():
    # the g query heads of a group are stacked as training rows; kept keys in position order
    L, Hkv, g, n_q, d, T = 1, 2, 2, 3, 4, 7
    r = np.random.default_rng(5)
    q = r.normal(size=(L, Hkv * g, n_q, d)); k = r.normal(size=(L, Hkv, T, d)); v = r.normal(size=(L, Hkv, T, d))
    mask = np.zeros((L, Hkv, T), dtype=np.uint8); mask[0, 0, [1, 4, 6]] = 1; mask[0, 1, [0, 2]] = 1
    vv, parts = O.value_refit(q, k, v, mask, 0.1)
    assert vv[0][0].shape == (3, d) and vv[0][1].shape == (2, d)
    A, Ot = parts[0][1]
    assert A.shape == (g * n_q, 2)
    x = (q[0, 2] @ k[0, 1, [0, 2]].T) / 2.0          # head 2 is the first of group 1
    a = np.exp(x - x.max(1, keepdims=True)); a /= a.sum(1, keepdims=True)
    assert np.allclose(A[:n_q], a, rtol=0, atol=1e-14)


# ------------------------------------------------------------------ decode-time pruning

def test_decode_prune_hand_example():
    kept, window = O.decode_prune(np.array([[0.0, 5.0, -1.0, 3.0, 7.0]]), 2.0, 2)
    assert kept == [[1]] and window == [[3, 4]]
    kept, window = O.decode_prune(np.array([[0.0, 5.0, -1.0, 3.0, 7.0]]), 2.0, 0)
    assert kept == [[1, 3, 4]] and window == [[]]


def test_decode_prune_equals_prefill_threshold():
    # phase-agnostic: deciding each token as it leaves the window keeps exactly what the
    # prefill threshold rule keeps (kept tokens plus the final window)
    for w in (0, 1, 5, 40, 100):
        r = np.random.default_rng(w)
        T = 60
        s = np.round(r.normal(size=(4, T)) * 2) / 2
        s[r.random(s.shape) < 0.05] = np.nan
        tau = 0.5
        kept, window = O.decode_prune(s, tau, w)
        mask, keep = O.prune_threshold(s, tau, w)
        for row in range(4):
            assert kept[row] == sorted(kept[row])
            assert window[row] == list(range(max(0, T - w), T))
            got = np.zeros(T, dtype=np.uint8)
            got[kept[row] + window[row]] = 1
            assert np.array_equal(got, mask[row])
            assert len(kept[row]) + len(window[row]) == keep[row]


# ------------------------------------------------------------------ MLP surrogate (GELU)

# standard normal CDF at 1, -1, 2 (normal-table values)
PHI_1 = 0.8413447460685429
PHI_M1 = 0.15865525393145707
PHI_2 = 0.9772498680518208


def test_gelu_normal_table_values():
    g = O.gelu(np.array([0.0, 1.0, -1.0, 2.0, 40.0, -40.0]))
    assert g[0] == 0.0
    assert abs(g[1] - PHI_1) < 1e-15 and abs(g[2] + PHI_M1) < 1e-15
    assert abs(g[3] - 2 * PHI_2) < 1e-15
    assert g[4] == 40.0 and abs(g[5]) < 1e-300


def test_gelu_odd_part_is_identity():
    # Phi(x) + Phi(-x) = 1  =>  GELU(x) - GELU(-x) = x
    x = rng.normal(size=50) * 3
    assert np.allclose(O.gelu(x) - O.gelu(-x), x, rtol=0, atol=1e-14)


def _mlp_weights(L, Dh, Dm, H, b1_shift=0.0):
    W1 = rng.normal(size=(L, Dm, Dh)) / math.sqrt(Dh)
    b1 = rng.normal(size=(L, Dm)) * 0.5 + b1_shift
    W2 = rng.normal(size=(L, H, Dm)) / math.sqrt(Dm)
    b2 = rng.normal(size=(L, H)) - 4.0
    return W1, b1, W2, b2


def test_mlp_in_linear_regime_equals_composed_linear_surrogate():
    # all pre-activations >> 0: GELU is the identity, so the MLP is the linear
    # surrogate with W = W1^T W2^T and b = W2 b1 + b2
    L, T, Dh, Dm, H = 2, 7, 16, 4, 3
    h = rng.normal(size=(L, T, Dh))
    W1, b1, W2, b2 = _mlp_weights(L, Dh, Dm, H, b1_shift=60.0)
    z = O.mlp_surrogate(h, W1, b1, W2, b2)
    W = np.stack([W1[l].T @ W2[l].T for l in range(L)])
    b = np.stack([W2[l] @ b1[l] + b2[l] for l in range(L)])
    assert z.shape == (L, H, T)
    assert np.allclose(z, O.linear_surrogate(h, W, b), rtol=1e-12, atol=1e-10)


def test_mlp_with_dead_hidden_units_gives_output_bias():
    L, T, Dh, Dm, H = 2, 5, 8, 4, 3
    h = rng.normal(size=(L, T, Dh))
    W1, b1, W2, b2 = _mlp_weights(L, Dh, Dm, H, b1_shift=-60.0)
    z = O.mlp_surrogate(h, W1, b1, W2, b2)
    assert np.allclose(z, np.broadcast_to(b2[:, :, None], (L, H, T)), rtol=0, atol=1e-12)


def test_mlp_brute_force_loops():
    L, T, Dh, Dm, H = 2, 3, 5, 4, 2
    h = rng.normal(size=(L, T, Dh))
    W1, b1, W2, b2 = _mlp_weights(L, Dh, Dm, H)
    z = O.mlp_surrogate(h, W1, b1, W2, b2)
    for l in range(L):
        for t in range(T):
            hidden = []
            for m in range(Dm):
                u = b1[l, m] + sum(W1[l, m, c] * h[l, t, c] for c in range(Dh))
                hidden.append(u * 0.5 * math.erfc(-u / math.sqrt(2.0)))
            for hh in range(H):
                want = b2[l, hh] + sum(W2[l, hh, m] * hidden[m] for m in range(Dm))
                assert abs(z[l, hh, t] - want) < 1e-12


# ----------------------------------------------------------------------------- pruning

def test_threshold_hand_example():
    s = np.array([-1.0, 0.5, np.nan, 0.49, -10.0, np.nan])
    mask, keep = O.prune_threshold(s, 0.5, 2)
    assert mask.tolist() == [0, 1, 0, 0, 1, 1] and int(keep) == 3


def test_threshold_limits_and_monotone():
    s = rng.normal(size=(3, 40)); w = 5
    m_lo, _ = O.prune_threshold(s, -np.inf, w)
    m_hi, k_hi = O.prune_threshold(s, np.inf, w)
    assert m_lo.all()
    assert (k_hi == w).all() and m_hi[:, -w:].all()
    prev = None
    for tau in np.linspace(-3, 3, 13):
        _, k = O.prune_threshold(s, tau, w)
        if prev is not None:
            assert (k <= prev).all()
        prev = k


def test_topk_hand_example_ties_and_nan():
    s = np.array([5.0, 1.0, 5.0, np.nan, 3.0, 5.0, 0.0, 0.0])
    want = {3: [1, 0, 1, 0, 0, 1, 1, 1], 4: [1, 0, 1, 0, 1, 1, 1, 1],
            5: [1, 1, 1, 0, 1, 1, 1, 1], 6: [1, 1, 1, 1, 1, 1, 1, 1],
            2: [1, 0, 1, 0, 0, 0, 1, 1], 0: [0, 0, 0, 0, 0, 0, 1, 1]}
    for k, m in want.items():
        mask, keep = O.prune_topk(s, k, 2)
        assert mask.tolist() == m, k
        assert int(keep) == sum(m)


def test_topk_budget_and_limits():
    s = rng.normal(size=(2, 3, 50))
    for k in (0, 1, 10, 44, 45, 46, 60):
        for w in (0, 5, 50, 70):
            mask, keep = O.prune_topk(s, k, w)
            assert (keep == min(50, k + min(w, 50))).all()
            assert mask[..., 50 - min(w, 50):].all()
    # all-equal scores: the earliest positions win
    mask, _ = O.prune_topk(np.zeros(10), 3, 2)
    assert mask.tolist() == [1, 1, 1, 0, 0, 0, 0, 0, 1, 1]


def test_topk_selects_largest():
    s = rng.permutation(30).astype(float)
    mask, _ = O.prune_topk(s, 7, 0)
    assert sorted(np.nonzero(mask)[0].tolist()) == sorted(np.argsort(-s)[:7].tolist())


# ----------------------------------------------------------------------------- compaction

def test_compaction_hand_example():
    k = np.zeros((1, 2, 5, 1), dtype=np.int64)
    for h in range(2):
        for t in range(5):
            k[0, h, t, 0] = t + 10 * h + 1
    v = -k
    mask = np.array([[[1, 0, 1, 1, 0], [0, 1, 0, 0, 0]]], dtype=np.uint8)
    kp, vp, bt, sl, tot = O.compact_paged(k, v, mask, page_size=2)
    assert tot == 3
    assert kp[:, :, 0].tolist() == [[1, 3], [4, 0], [12, 0]]
    assert vp[:, :, 0].tolist() == [[-1, -3], [-4, 0], [-12, 0]]
    assert bt.tolist() == [[[0, 1, -1], [2, -1, -1]]]
    assert sl.tolist() == [[3, 1]]


def test_compaction_all_kept_reproduces_input():
    L, H, T, d, ps = 2, 3, 37, 4, 16
    k = rng.normal(size=(L, H, T, d)); v = rng.normal(size=(L, H, T, d))
    kp, vp, bt, sl, tot = O.compact_paged(k, v, np.ones((L, H, T), np.uint8), ps)
    assert tot == L * H * 3 and (sl == T).all()
    for l in range(L):
        for h in range(H):
            rows = np.concatenate([kp[p] for p in bt[l, h] if p >= 0])
            assert np.array_equal(rows[:T], k[l, h]) and not rows[T:].any()


def test_compaction_counts_match_mask():
    L, H, T, d = 2, 2, 50, 2
    k = rng.normal(size=(L, H, T, d)); v = rng.normal(size=(L, H, T, d))
    mask = (rng.random((L, H, T)) < 0.4).astype(np.uint8)
    kp, vp, bt, sl, tot = O.compact_paged(k, v, mask, 16)
    assert int(sl.sum()) == int(mask.sum())
    assert tot == int(sum(-(-int(n) // 16) for n in sl.ravel()))


# ----------------------------------------------------------------------------- page numbers

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_kv_memory_formula_reproduces_pages():
    g = _golden()["kv_memory"]
    a = g[0]
    assert O.kv_cache_bytes(a["L"], a["T"], a["H_kv"], a["d"], a["bytes_per_elem"]) == a["bytes"]
    b = g[1]
    gb = O.kv_cache_bytes(b["L"], b["T"], b["H_kv"], b["d"], b["bytes_per_elem"]) / 1e9
    assert math.floor(gb) == b["gigabytes_printed"]


def test_overhead_formulas_reproduce_appendix_b():
    for r in _golden()["overhead_percent"]:
        C = O.layer_linear_flops(r["D_h"], r["H_q"], r["H_kv"], r["D"], r["D_int"])
        mlp = 100 * O.kvzap_mlp_flops(r["D_h"], r["H_kv"]) / C
        lin = 100 * O.kvzap_linear_flops(r["D_h"], r["H_kv"]) / C
        assert round(mlp, 2) == r["mlp"], (r["cite"], mlp)
        assert round(lin, 2) == r["linear"], (r["cite"], lin)


def test_surrogate_param_counts_match_table():
    for r in _golden()["surrogate_params_millions"]:
        f = O.kvzap_mlp_params if r["kind"] == "mlp" else O.kvzap_linear_params
        m = f(r["L"], r["D_h"], r["H_kv"]) / 1e6
        tol = 0.5 if r["millions"] >= 10 else 0.06   # the table rounds to the shown digit
        assert abs(m - r["millions"]) < tol, (r, m)


def test_compression_factor_table2():
    for r in _golden()["compression"]:
        f = O.compression_factor(r["ratio"])
        assert math.floor(f * 10) / 10 == r["factor_printed"]


def test_quantile_lower_nearest_rank():
    assert O.quantile_lower([3, 1, 2, 4], 0.25) == 1
    assert O.quantile_lower([3, 1, 2, 4], 0.5) == 2
    assert O.quantile_lower(np.arange(101), 0.25) == 25
    assert O.quantile_lower([5.0, 0.0, 1.0], 0.0) == 0.0 and O.quantile_lower([5.0, 0.0, 1.0], 1.0) == 5.0
    # NaN below every number: [nan, nan, -1, 2, 7] by rank
    v = [2.0, np.nan, 7.0, -1.0, np.nan]
    assert np.isnan(O.quantile_lower(v, 0.25))        # rank floor(0.25 * 4) = 1
    assert O.quantile_lower(v, 0.5) == -1.0           # rank 2
    assert O.quantile_lower(v, 0.8) == 2.0            # rank 3


def test_quantile_rank_brute_force():
    """The nearest-rank property by counting: with r = floor(q (N - 1)), at most r values
    lie below tau and more than r lie at or below it; tau is one of the values."""
    rng = np.random.default_rng(7)
    for N, levels in [(1, None), (10, None), (999, None), (1000, 4), (257, 2)]:
        v = rng.normal(size=N)
        if levels:
            v = np.round(v * levels) / levels
        for q in (0.0, 0.1, 0.25, 0.5, 0.999, 1.0):
            tau = O.quantile_lower(v, q)
            r = int(math.floor(q * (N - 1)))
            assert (v < tau).sum() <= r < (v <= tau).sum()
            assert tau in v


def test_prune_quantile_per_layer():
    """Per layer: tau from that layer's non-window scores of every head (window scores,
    however small, never move it); the mask is the threshold rule with that tau; the
    keep count is at least (1 - q) of the candidates plus the window."""
    rng = np.random.default_rng(3)
    L, H, T, w, q = 3, 4, 50, 7, 0.25
    s = rng.normal(size=(L, H, T))
    s[1] += 10.0                      # a shifted layer gets its own tau
    s[:, :, T - w:] = -100.0          # window scores are excluded from the quantile
    m, k, tau = O.prune_quantile(s, q, w)
    for l in range(L):
        cand = s[l, :, : T - w].ravel()
        assert tau[l] == np.sort(cand)[int(math.floor(q * (cand.size - 1)))]
        m_ref, k_ref = O.prune_threshold(s[l], tau[l], w)
        assert np.array_equal(m[l], m_ref) and np.array_equal(k[l], k_ref)
        assert k[l].sum() >= math.ceil((1 - q) * cand.size) + H * w
    assert tau[1] > tau[0] + 5 and tau[1] > tau[2] + 5
    # everything in the window: no candidate, tau = +inf, only the window kept
    m, k, tau = O.prune_quantile(s, q, T)
    assert np.isinf(tau).all() and (k == T).all()
    m, k, tau = O.prune_quantile(s, q, 0)
    assert (k.sum(axis=1) >= math.ceil((1 - q) * H * T)).all()
