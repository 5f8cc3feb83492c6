"""Per-entry-point parity of the CUDA path against the fp64 oracle, element by element,
at sizes that span several tiles with ragged tails, plus the degenerate cases."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_util import (LOG_SCORE_ATOL, LSE_ATOL, MASK_BAND, SCORE_RTOL, assert_close_abs,
                            assert_close_rel, assert_masks_match_near, cuda, f64, need_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    need_gpu()
    from kv_cache_eviction_lse_gb300 import build
    build.build()
    from kv_cache_eviction_lse_gb300 import capi
    return capi


def _inputs(L, Hkv, Hq, d, T, n_tail, n_q, seed, scale=1.0, D_h=0):
    from kv_cache_eviction_lse_gb300.workloads import random_kv_inputs
    return random_kv_inputs(L, Hkv, Hq, d, T, n_tail, n_q, seed, scale=scale, D_h=D_h)


LSE_SHAPES = [
    # L, Hkv, Hq, d, T, n_tail, n_q
    (2, 2, 6, 128, 150, 79, 70),
    (1, 1, 2, 64, 256, 264, 256),
    (2, 2, 4, 128, 200, 0, 200),     # causal self-attention
    (1, 3, 3, 64, 1, 0, 1),          # single key
    (1, 1, 4, 128, 0, 97, 97),       # no context keys
    (3, 1, 2, 128, 333, 5, 1),       # one query
]


@pytest.mark.parametrize("shape", LSE_SHAPES, ids=[str(s) for s in LSE_SHAPES])
@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_lse(C, shape, scale):
    L, Hkv, Hq, d, T, nt, nq = shape
    x = _inputs(*shape, seed=11 + T + nq, scale=scale)
    g = cuda(x)
    out = torch.full((L, Hq, nq), float("nan"), device="cuda")
    C.kvs_lse(C.dims(L, Hq, Hkv, d), g["q"], nq, g["k_ctx"] if T else None, T,
              g["k_tail"] if nt else None, nt, out)
    torch.cuda.synchronize()
    want = O.lse(f64(x["q"]), f64(x["k_ctx"]), f64(x["k_tail"]))
    assert_close_abs(out.cpu().numpy(), want, LSE_ATOL, "lse")


FWD_SHAPES = [
    # L, Hkv, Hq, d, T, n_tail, n_q
    (2, 2, 6, 128, 150, 79, 70),
    (1, 1, 2, 64, 256, 264, 256),
    (2, 2, 4, 128, 300, 0, 300),     # causal self-attention, ragged tiles
    (1, 3, 3, 64, 1, 0, 1),          # single key
    (1, 1, 4, 128, 0, 97, 97),       # no context keys
    (3, 1, 2, 128, 333, 5, 1),       # one query
    (1, 2, 4, 128, 700, 20, 400),    # several key tiles per query tile, two query tiles
    # more 128-query units than SMs: the persistent grid's CTAs carry TMEM, rings and
    # barrier phases from one unit to the next (causal units of different lengths)
    (2, 4, 32, 64, 300, 40, 300),
    (1, 8, 64, 128, 260, 200, 450),
]


def _fwd_inputs(shape, seed, scale):
    L, Hkv, Hq, d, T, nt, nq = shape
    x = _inputs(*shape, seed=seed, scale=scale)
    gen = torch.Generator().manual_seed(seed + 1)
    x["v_tail"] = torch.randn(L, Hkv, nt, d, generator=gen).to(torch.bfloat16)
    return x


def _o_tolerance(o_ref, v_ctx, v_tail, g):
    """Bound on |o_gpu - o_ref|: the softmax weights are rounded to bf16 (relative
    2^-9 each, so at most 2^-9 max|v| on any output) and o is stored as bf16 (2^-9
    |o|); the fp32 accumulation and ex2.approx add far less.  Twice that bound."""
    vals = np.concatenate([v_ctx, v_tail], 2) if v_tail.shape[2] else v_ctx
    vmax = np.abs(vals).max(axis=(2, 3)) if vals.shape[2] else np.zeros(vals.shape[:2])
    vmax = np.repeat(vmax, g, axis=1)[:, :, None, None]
    return 2.0 ** -8 * (np.abs(o_ref) + vmax)


@pytest.mark.parametrize("shape", FWD_SHAPES, ids=[str(s) for s in FWD_SHAPES])
@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_attn_fwd(C, shape, scale):
    L, Hkv, Hq, d, T, nt, nq = shape
    x = _fwd_inputs(shape, seed=23 + T + nq, scale=scale)
    g = cuda(x)
    o = torch.full((L, Hq, nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((L, Hq, nq), float("nan"), device="cuda")
    C.kvs_attn_fwd(C.dims(L, Hq, Hkv, d), g["q"], nq, g["k_ctx"] if T else None,
                   g["v_ctx"] if T else None, T, g["k_tail"] if nt else None,
                   g["v_tail"] if nt else None, nt, o, lse)
    lse_only = torch.empty_like(lse)
    C.kvs_lse(C.dims(L, Hq, Hkv, d), g["q"], nq, g["k_ctx"] if T else None, T,
              g["k_tail"] if nt else None, nt, lse_only)
    torch.cuda.synchronize()
    vc, vt = f64(x["v_ctx"]), f64(x["v_tail"])
    o_ref, lse_ref = O.attention_forward(f64(x["q"]), f64(x["k_ctx"]), f64(x["k_tail"]), vc, vt)
    assert_close_abs(lse.cpu().numpy(), lse_ref, LSE_ATOL, "forward lse")
    assert_close_abs(lse.cpu().numpy(), lse_only.cpu().numpy(), LSE_ATOL, "forward lse vs kvs_lse")
    err = np.abs(f64(o) - o_ref)
    tol = _o_tolerance(o_ref, vc, vt, Hq // Hkv)
    assert (err <= tol).all(), f"forward o: {(err > tol).sum()} beyond bound; max err {err.max()}"


def test_attn_fwd_growing_logits_rescale(C):
    # keys grow along the sequence, so the row max keeps rising across key tiles and O
    # is rescaled in TMEM many times
    L, Hkv, Hq, d, T = 1, 1, 2, 128, 1024
    gen = torch.Generator().manual_seed(5)
    ramp = torch.linspace(0.2, 3.0, T)[None, None, :, None]
    k = (torch.randn(L, Hkv, T, d, generator=gen) * ramp).to(torch.bfloat16)
    v = torch.randn(L, Hkv, T, d, generator=gen).to(torch.bfloat16)
    q = (torch.randn(L, Hq, T, d, generator=gen) * 2).to(torch.bfloat16)
    o = torch.empty(L, Hq, T, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(L, Hq, T, device="cuda")
    C.kvs_attn_fwd(C.dims(L, Hq, Hkv, d), q.cuda(), T, k.cuda(), v.cuda(), T, None, None, 0, o, lse)
    torch.cuda.synchronize()
    o_ref, lse_ref = O.attention_forward(f64(q), f64(k), None, f64(v), None)
    assert_close_abs(lse.cpu().numpy(), lse_ref, LSE_ATOL, "forward lse (growing logits)")
    err = np.abs(f64(o) - o_ref)
    tol = _o_tolerance(o_ref, f64(v), f64(v)[:, :, :0], Hq // Hkv)
    assert (err <= tol).all(), f"forward o: {(err > tol).sum()} beyond bound; max err {err.max()}"


SCORE_SHAPES = [
    (2, 2, 6, 128, 150, 79, 70, 192),
    (1, 1, 2, 64, 256, 264, 256, 0),
    (2, 4, 8, 128, 77, 40, 33, 128),
    (1, 2, 2, 64, 1, 3, 2, 64),
]


@pytest.mark.parametrize("shape", SCORE_SHAPES, ids=[str(s) for s in SCORE_SHAPES])
def test_vnorm_lse_score_max(C, shape):
    L, Hkv, Hq, d, T, nt, nq, Dh = shape
    x = _inputs(L, Hkv, Hq, d, T, nt, nq, seed=5 + T, scale=1.5, D_h=Dh)
    g = cuda(x)
    dm = C.dims(L, Hq, Hkv, d, Dh)
    lse = torch.empty((L, Hq, nq), device="cuda")
    C.kvs_lse(dm, g["q"], nq, g["k_ctx"], T, g["k_tail"], nt, lse)
    score = torch.empty((L, Hkv, T), device="cuda")
    vn = None
    if Dh:
        vn = torch.empty((L, Hq, T), device="cuda")
        ws = torch.empty(C.kvs_vnorm_workspace_size(dm), dtype=torch.uint8, device="cuda")
        C.kvs_vnorm(dm, g["v_ctx"], T, g["w_o"], vn, ws, ws.numel())
        sws = torch.empty(C.kvs_score_max_workspace_size(dm, nq, 1), dtype=torch.uint8, device="cuda")
        C.kvs_score_max(dm, g["q"], nq, g["k_ctx"], T, lse, vn, g["h"], 0, score, sws, sws.numel())
    else:
        sws = torch.empty(max(16, C.kvs_score_max_workspace_size(dm, nq, 0)), dtype=torch.uint8,
                          device="cuda")
        C.kvs_score_max(dm, g["q"], nq, g["k_ctx"], T, lse, None, None, 0, score, sws, sws.numel())
    torch.cuda.synchronize()
    q, kc, kt = f64(x["q"]), f64(x["k_ctx"]), f64(x["k_tail"])
    vref = O.value_norm(f64(x["v_ctx"]), f64(x["w_o"]), Hq) if Dh else None
    if Dh:
        assert_close_rel(vn.cpu().numpy(), vref, 1e-4, "vnorm")
    want = O.kvzip_score(q, kc, kt, vnorm=vref, h=f64(x["h"]) if Dh else None)
    assert_close_abs(score.cpu().numpy(), want, LOG_SCORE_ATOL, "log score")


def test_score_max_accumulate(C):
    L, Hkv, Hq, d, T, nt, nq = 1, 2, 4, 128, 100, 50, 40
    xa = _inputs(L, Hkv, Hq, d, T, nt, nq, seed=1)
    xb = _inputs(L, Hkv, Hq, d, T, nt, nq, seed=2)
    xb["k_ctx"] = xa["k_ctx"]
    dm = C.dims(L, Hq, Hkv, d)
    score = torch.empty((L, Hkv, T), device="cuda")
    for i, x in enumerate((xa, xb)):
        g = cuda(x)
        lse = torch.empty((L, Hq, nq), device="cuda")
        C.kvs_lse(dm, g["q"], nq, g["k_ctx"], T, g["k_tail"], nt, lse)
        sws = torch.empty(C.kvs_score_max_workspace_size(dm, nq, 0), dtype=torch.uint8,
                          device="cuda")
        C.kvs_score_max(dm, g["q"], nq, g["k_ctx"], T, lse, None, None, i, score, sws, sws.numel())
    torch.cuda.synchronize()
    want = O.kvzip_score_chunked([f64(xa["q"]), f64(xb["q"])], f64(xa["k_ctx"]),
                                 [f64(xa["k_tail"]), f64(xb["k_tail"])])
    assert_close_abs(score.cpu().numpy(), want, LOG_SCORE_ATOL, "accumulated log score")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T,w", [(333, 0), (333, 17), (333, 128), (333, 400), (64, 1), (1, 0)])
def test_future_sum(C, d, T, w):
    L, Hkv, Hq = 2, 2, 4
    x = _inputs(L, Hkv, Hq, d, T, 0, T, seed=T + w + d, scale=1.5)
    g = cuda(x)
    dm = C.dims(L, Hq, Hkv, d)
    lse = torch.empty((L, Hq, T), device="cuda")
    C.kvs_lse(dm, g["q"], T, g["k_ctx"], T, None, 0, lse)
    f = torch.full((L, Hkv, T), float("nan"), device="cuda")
    fws = torch.empty(C.kvs_score_future_sum_workspace_size(dm, T), dtype=torch.uint8, device="cuda")
    C.kvs_score_future_sum(dm, g["q"], g["k_ctx"], T, lse, w, f, fws, fws.numel())
    torch.cuda.synchronize()
    want = O.future_attention_mass(f64(x["q"]), f64(x["k_ctx"]), w)
    got = f.cpu().numpy()
    assert_close_rel(got, want, SCORE_RTOL, "future mass")
    assert (got[..., max(0, T - w):] == 0).all()


@pytest.mark.parametrize("Hkv", [8, 3, 12])
@pytest.mark.parametrize("T", [40000, 1000, 16, 1])  # 40000: whole tiles per warp; else split
def test_surrogate(C, Hkv, T):
    L, Dh, w, tau = 2, 256, 7, -4.5
    gen = torch.Generator().manual_seed(Hkv * 1000 + T)
    h = torch.randn(L, T, Dh, generator=gen).to(torch.bfloat16)
    W = (torch.randn(L, Dh, Hkv, generator=gen) / 16).to(torch.bfloat16)
    b = torch.randn(L, Hkv, generator=gen) - 4.0
    dm = C.dims(L, Hkv, Hkv, 128, Dh)
    z = torch.empty(L, Hkv, T, device="cuda")
    mask = torch.empty(L, Hkv, T, dtype=torch.uint8, device="cuda")
    keep = torch.full((L, Hkv), -7, dtype=torch.int32, device="cuda")
    C.kvs_surrogate(dm, h.cuda(), T, W.cuda(), b.cuda(), z, tau, w, mask, keep)
    z2 = torch.empty_like(z)
    C.kvs_surrogate(dm, h.cuda(), T, W.cuda(), b.cuda(), z2)  # unfused
    torch.cuda.synchronize()
    want = O.linear_surrogate(f64(h), f64(W), b.double().numpy())
    zg = z.cpu().numpy()
    assert_close_abs(zg, want, LOG_SCORE_ATOL, "surrogate")
    assert np.array_equal(zg, z2.cpu().numpy())
    # the fused decision matches the threshold rule applied to the kernel's own fp32 scores
    m_same, k_same = O.prune_threshold(zg.astype(np.float64), np.float32(tau), w)
    assert np.array_equal(mask.cpu().numpy(), m_same)
    assert np.array_equal(keep.cpu().numpy(), k_same)
    # and the oracle's decision except next to tau
    m_ref, _ = O.prune_threshold(want, tau, w)
    assert_masks_match_near(mask.cpu().numpy(), m_ref, want, np.full(want.shape[:-1], tau),
                            MASK_BAND, "surrogate mask", log_domain=True)


MLP_SHAPES = [
    # L, T, D_h, D_mid, H_kv   (parts P of D_mid: <= 256 columns, multiples of 32)
    (2, 300, 256, 64, 8),      # P=1, N=64, ragged last token tile
    (2, 1000, 512, 512, 4),    # P=2, N=256
    (1, 257, 1024, 640, 2),    # P=4, N=160
    (1, 130, 128, 128, 16),    # 16 heads
    (3, 1, 64, 32, 1),         # one token, one k-block
    (1, 384, 4096, 512, 8),    # the Qwen3-8B shape (64 k-blocks), three full tiles
]


def _mlp_parts(Dm):
    """Column parts of D_mid as kvs.h documents them: the fewest parts of at most 256
    columns, each a multiple of 32."""
    P = -(-Dm // 256)
    while Dm % P or (Dm // P) % 32:
        P += 1
    return P


def _mlp_inputs(L, T, Dh, Dm, H, seed):
    gen = torch.Generator().manual_seed(seed)
    h = torch.randn(L, T, Dh, generator=gen).to(torch.bfloat16)
    W1 = (torch.randn(L, Dm, Dh, generator=gen) / math.sqrt(Dh)).to(torch.bfloat16)
    b1 = torch.randn(L, Dm, generator=gen) * 0.5
    W2 = (torch.randn(L, H, Dm, generator=gen) / math.sqrt(Dm)).to(torch.bfloat16)
    b2 = torch.randn(L, H, generator=gen) - 4.0
    return h, W1, b1, W2, b2


@pytest.mark.parametrize("shape", MLP_SHAPES, ids=[str(s) for s in MLP_SHAPES])
def test_surrogate_mlp(C, shape):
    L, T, Dh, Dm, H = shape
    w, tau = 5, -4.0
    h, W1, b1, W2, b2 = _mlp_inputs(L, T, Dh, Dm, H, seed=T * 7 + Dm)
    dm = C.dims(L, H, H, 128, Dh)
    args = [t.cuda() for t in (h, W1, b1, W2, b2)]
    z = torch.full((L, H, T), float("nan"), device="cuda")
    mask = torch.empty(L, H, T, dtype=torch.uint8, device="cuda")
    keep = torch.full((L, H), -7, dtype=torch.int32, device="cuda")
    C.kvs_surrogate_mlp(dm, args[0], T, Dm, *args[1:], z, tau, w, mask, keep)
    z2 = torch.empty_like(z)
    C.kvs_surrogate_mlp(dm, args[0], T, Dm, *args[1:], z2)  # unfused
    torch.cuda.synchronize()
    want = O.mlp_surrogate(f64(h), f64(W1), b1.double().numpy(), f64(W2), b2.double().numpy())
    zg = z.cpu().numpy()
    assert_close_abs(zg, want, LOG_SCORE_ATOL, "mlp surrogate")
    if _mlp_parts(Dm) <= 2:  # at most two partial sums per score: order-independent
        assert np.array_equal(zg, z2.cpu().numpy())
    m_same, k_same = O.prune_threshold(zg.astype(np.float64), np.float32(tau), w)
    assert np.array_equal(mask.cpu().numpy(), m_same)
    assert np.array_equal(keep.cpu().numpy(), k_same)
    m_ref, _ = O.prune_threshold(want, tau, w)
    assert_masks_match_near(mask.cpu().numpy(), m_ref, want, np.full(want.shape[:-1], tau),
                            MASK_BAND, "mlp surrogate mask", log_domain=True)


def test_surrogate_mlp_empty_and_unsupported(C):
    h, W1, b1, W2, b2 = (t.cuda() for t in _mlp_inputs(1, 4, 64, 32, 2, seed=3))
    z = torch.full((1, 2, 4), 5.0, device="cuda")
    C.kvs_surrogate_mlp(C.dims(1, 2, 2, 128, 64), h, 0, 32, W1, b1, W2, b2, z)  # T = 0: no-op
    torch.cuda.synchronize()
    assert (z == 5.0).all()
    with pytest.raises(C.KvsError) as e:
        C.kvs_surrogate_mlp(C.dims(1, 3, 3, 128, 64), h, 4, 32, W1, b1, W2, b2, z)
    assert e.value.status == C.KVS_ERR_UNSUPPORTED
    with pytest.raises(C.KvsError) as e:
        C.kvs_surrogate_mlp(C.dims(1, 2, 2, 128, 64), h, 4, 48, W1, b1, W2, b2, z)
    assert e.value.status == C.KVS_ERR_UNSUPPORTED


def _scores_with_ties(shape, seed, levels=None, nan_frac=0.0):
    r = np.random.default_rng(seed)
    s = r.normal(size=shape).astype(np.float32)
    if levels:
        s = np.round(s * levels).astype(np.float32) / levels
    if nan_frac:
        s[r.random(shape) < nan_frac] = np.nan
    return s


@pytest.mark.parametrize("T", [1, 7, 300, 2048, 5000])
@pytest.mark.parametrize("levels,nan_frac", [(None, 0.0), (3, 0.0), (4, 0.05)])
def test_prune_threshold_exact(C, T, levels, nan_frac):
    L, H = 2, 3
    s = _scores_with_ties((L, H, T), T, levels, nan_frac)
    for tau, w in [(0.0, 0), (0.25, 5), (-np.inf, 0), (np.inf, 3), (0.5, T), (0.0, T + 4)]:
        mask = torch.empty(L, H, T, dtype=torch.uint8, device="cuda")
        keep = torch.empty(L, H, dtype=torch.int32, device="cuda")
        C.kvs_prune_mask(C.dims(L, H, H, 128), torch.from_numpy(s).cuda(), T, C.KVS_THRESHOLD,
                         tau, 0, w, mask, keep)
        torch.cuda.synchronize()
        m_ref, k_ref = O.prune_threshold(s.astype(np.float64), tau, w)
        assert np.array_equal(mask.cpu().numpy(), m_ref), (tau, w)
        assert np.array_equal(keep.cpu().numpy(), k_ref), (tau, w)


# row lengths on both sides of every register-resident width (1, 2, 4, 8, 16 tokens per
# thread, with and without 16-byte rows) and past it (rows re-read from global memory)
@pytest.mark.parametrize("T", [1, 7, 300, 1024, 1025, 2048, 3001, 4096, 6002, 8192, 16383,
                               16384, 20000])
@pytest.mark.parametrize("levels,nan_frac", [(None, 0.0), (3, 0.0), (4, 0.05)])
def test_prune_topk_exact(C, T, levels, nan_frac):
    L, H = 2, 3
    s = _scores_with_ties((L, H, T), T + 1, levels, nan_frac)
    for k, w in [(0, 0), (1, 0), (T // 4, 0), (T // 4, 16), (T // 2, T // 3), (T, 0), (T - 5, 5),
                 (T + 3, 2), (3, T), (2, T + 9)]:
        if k < 0:
            continue
        mask = torch.empty(L, H, T, dtype=torch.uint8, device="cuda")
        keep = torch.empty(L, H, dtype=torch.int32, device="cuda")
        C.kvs_prune_mask(C.dims(L, H, H, 128), torch.from_numpy(s).cuda(), T, C.KVS_TOPK, 0.0, k,
                         w, mask, keep)
        torch.cuda.synchronize()
        m_ref, k_ref = O.prune_topk(s.astype(np.float64), k, w)
        assert np.array_equal(mask.cpu().numpy(), m_ref), (k, w)
        assert np.array_equal(keep.cpu().numpy(), k_ref), (k, w)


@pytest.mark.parametrize("T,page", [(1, 16), (100, 16), (4096, 16), (5000, 16), (9000, 7),
                                    (333, 1), (17, 4096), (48, 16), (2048, 16), (6144, 8),
                                    (8192, 16), (45056, 16)])
@pytest.mark.parametrize("d", [64, 128])
def test_compact_exact(C, T, page, d):
    L, H = 2, 3
    r = np.random.default_rng(T + page + d)
    p_keep = r.uniform(0.0, 1.0, size=(L, H, 1))
    mask = (r.random((L, H, T)) < p_keep).astype(np.uint8)
    mask[0, 0] = 1
    mask[1, 2] = 0
    gen = torch.Generator().manual_seed(T)
    k = torch.randn(L, H, T, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(L, H, T, d, generator=gen).to(torch.bfloat16)
    from kv_cache_eviction_lse_gb300.pipeline import Pages, compact_into
    dm = C.dims(L, H, H, d)
    pages = Pages(L, H, T, d, page, "cuda")
    pages.k_pages.fill_(7.0)
    pages.v_pages.fill_(7.0)
    ws = torch.empty(C.kvs_compact_workspace_size(dm, T), dtype=torch.uint8, device="cuda")
    compact_into(dm, k.cuda(), v.cuda(), T, torch.from_numpy(mask).cuda(), pages, ws)
    torch.cuda.synchronize()
    kb = k.view(torch.int16).numpy()
    vb = v.view(torch.int16).numpy()
    kp, vp, bt, sl, tot = O.compact_paged(kb, vb, mask, page, pages.max_pages)
    assert int(pages.needed.item()) == tot
    assert np.array_equal(pages.seq_lens.cpu().numpy(), sl)
    assert np.array_equal(pages.block_table.cpu().numpy(), bt)
    assert np.array_equal(pages.k_pages[:tot].cpu().view(torch.int16).numpy(), kp)
    assert np.array_equal(pages.v_pages[:tot].cpu().view(torch.int16).numpy(), vp)
    # pages past the total are untouched
    if tot < pages.capacity:
        assert bool((pages.k_pages[tot:] == 7.0).all())


@pytest.mark.parametrize("L,H,T,w", [(1, 1, 1, 0), (2, 3, 300, 16), (3, 8, 2048, 128),
                                     (2, 2, 5000, 5000), (1, 4, 20001, 7), (2, 8, 9000, 128),
                                     (1, 3, 70001, 0), (2, 20, 4200, 100)])
@pytest.mark.parametrize("levels,nan_frac", [(None, 0.0), (3, 0.0), (4, 0.05)])
def test_prune_quantile_exact(C, L, H, T, w, levels, nan_frac):
    """The per-layer tau is exactly the oracle's order statistic of the same fp32 scores
    (NaN lowest) and the masks and counts are the threshold rule with it.  Layers of at
    least 65536 non-window scores in rows of at least 4096 (the last three shapes, and
    20001 x 4) take the many-blocks-per-layer select."""
    s = _scores_with_ties((L, H, T), L * T + H, levels, nan_frac)
    s[-1] += 3.0  # the last layer's scores sit higher: its own tau
    for q in (0.25, 0.0, 1.0, 0.5):
        tau = torch.full((L,), 123.0, device="cuda")
        mask = torch.full((L, H, T), 9, dtype=torch.uint8, device="cuda")
        keep = torch.full((L, H), -1, dtype=torch.int32, device="cuda")
        C.kvs_prune_quantile(C.dims(L, H, H, 128), torch.from_numpy(s).cuda(), T, q, w, tau, mask,
                             keep)
        torch.cuda.synchronize()
        m_ref, k_ref, t_ref = O.prune_quantile(s.astype(np.float64), q, w)
        tg = tau.cpu().double().numpy()
        assert np.array_equal(np.isnan(tg), np.isnan(t_ref)), (q, tg, t_ref)
        ok = ~np.isnan(t_ref)
        assert np.array_equal(tg[ok], t_ref[ok]), (q, tg, t_ref)
        assert np.array_equal(mask.cpu().numpy(), m_ref), q
        assert np.array_equal(keep.cpu().numpy(), k_ref), q


def test_prune_quantile_rejects_bad_q(C):
    t = torch.empty(64, device="cuda")
    m = torch.empty(64, dtype=torch.uint8, device="cuda")
    kp = torch.empty(16, dtype=torch.int32, device="cuda")
    for q in (-0.1, 1.5, float("nan")):
        with pytest.raises(C.KvsError) as e:
            C.kvs_prune_quantile(C.dims(1, 1, 1, 128), t, 8, q, 0, t, m, kp)
        assert e.value.status == C.KVS_ERR_ARG


# several budgets in one launch: row lengths on both sides of the shared-memory staging
# limit (16384), ties crossing the k-th value, NaN, windows, k = 0 and k >= T - w
@pytest.mark.parametrize("T", [1, 7, 300, 2048, 4097, 16384, 20000])
@pytest.mark.parametrize("levels,nan_frac", [(None, 0.0), (3, 0.0), (4, 0.05)])
def test_prune_topk_multi_exact(C, T, levels, nan_frac):
    L, H = 2, 3
    s = _scores_with_ties((L, H, T), T + 7, levels, nan_frac)
    for w, ks in [(0, [T // 4, T // 2, 0, T]), (16, [1, T // 3, T + 3]), (T // 3, [T // 2]),
                  (T, [5, 0]), (0, [3, 3, 3, 3, 3, 3, 3, 3])]:
        nb = len(ks)
        masks = torch.full((nb, L, H, T), 9, dtype=torch.uint8, device="cuda")
        keeps = torch.full((nb, L, H), -1, dtype=torch.int32, device="cuda")
        C.kvs_prune_topk_multi(C.dims(L, H, H, 128), torch.from_numpy(s).cuda(), T, ks, w, masks,
                               keeps)
        torch.cuda.synchronize()
        for b, k in enumerate(ks):
            m_ref, k_ref = O.prune_topk(s.astype(np.float64), k, w)
            assert np.array_equal(masks[b].cpu().numpy(), m_ref), (w, ks, b)
            assert np.array_equal(keeps[b].cpu().numpy(), k_ref), (w, ks, b)


def test_prune_topk_signed_zero_ties(C):
    """-0 and +0 are equal scores: a tie between them goes to the earlier position, in
    both the single-budget and the multi-budget selection."""
    T = 9
    s = np.array([[[-0.0, 0.0, 1.0, -0.0, 2.0, 0.0, -1.0, 0.0, -0.0]]], dtype=np.float32)
    for k in range(T + 1):
        m_ref, _ = O.prune_topk(s.astype(np.float64), k, 0)
        mask = torch.empty(1, 1, T, dtype=torch.uint8, device="cuda")
        keep = torch.empty(1, 1, dtype=torch.int32, device="cuda")
        C.kvs_prune_mask(C.dims(1, 1, 1, 128), torch.from_numpy(s).cuda(), T, C.KVS_TOPK, 0.0, k, 0,
                         mask, keep)
        masks = torch.empty(2, 1, 1, T, dtype=torch.uint8, device="cuda")
        keeps = torch.empty(2, 1, 1, dtype=torch.int32, device="cuda")
        C.kvs_prune_topk_multi(C.dims(1, 1, 1, 128), torch.from_numpy(s).cuda(), T, [k, k], 0,
                               masks, keeps)
        torch.cuda.synchronize()
        assert np.array_equal(mask.cpu().numpy(), m_ref), k
        assert np.array_equal(masks[1].cpu().numpy(), m_ref), k


def test_prune_topk_multi_rejects_bad_budgets(C):
    t = torch.empty(64, device="cuda")
    m = torch.empty(64, dtype=torch.uint8, device="cuda")
    kp = torch.empty(16, dtype=torch.int32, device="cuda")
    for ks, st in [([], C.KVS_ERR_UNSUPPORTED), ([1] * 9, C.KVS_ERR_UNSUPPORTED),
                   ([2, -1], C.KVS_ERR_ARG)]:
        with pytest.raises(C.KvsError) as e:
            C.kvs_prune_topk_multi(C.dims(1, 1, 1, 128), t, 8, ks, 0, m, kp)
        assert e.value.status == st


@pytest.mark.parametrize("T,page,n_masks", [(1, 16, 2), (300, 16, 3), (2048, 16, 3),
                                            (5000, 7, 2), (16384, 16, 2), (100, 4096, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_compact_multi_exact(C, T, page, n_masks, d):
    """n masks over the same K/V in one call: equal to the oracle's compaction of the
    masks stacked as n L layers over K/V repeated n times (pages mask-major)."""
    L, H = 2, 3
    r = np.random.default_rng(T + page + d + n_masks)
    p_keep = r.uniform(0.0, 1.0, size=(n_masks, L, H, 1))
    masks = (r.random((n_masks, L, H, T)) < p_keep).astype(np.uint8)
    masks[0, 0, 0] = 1
    masks[-1, 1, 2] = 0
    gen = torch.Generator().manual_seed(T + d)
    k = torch.randn(L, H, T, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(L, H, T, d, generator=gen).to(torch.bfloat16)
    dm = C.dims(L, H, H, d)
    max_pages = -(-T // page)
    cap = n_masks * L * H * max_pages
    kp = torch.full((cap, page, d), 7.0, dtype=torch.bfloat16, device="cuda")
    vp = torch.full((cap, page, d), 7.0, dtype=torch.bfloat16, device="cuda")
    bt = torch.empty((n_masks, L, H, max_pages), dtype=torch.int32, device="cuda")
    sl = torch.empty((n_masks, L, H), dtype=torch.int32, device="cuda")
    need = torch.empty(4, dtype=torch.int32, device="cuda")
    nws = C.kvs_compact_multi_workspace_size(dm, T, n_masks)
    assert nws >= C.kvs_compact_workspace_size(dm, T)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    C.kvs_compact_paged_multi(dm, k.cuda(), v.cuda(), T, n_masks, torch.from_numpy(masks).cuda(),
                              page, kp, vp, cap, bt, max_pages, sl, need, ws, nws)
    torch.cuda.synchronize()
    kb = np.concatenate([k.view(torch.int16).numpy()] * n_masks)
    vb = np.concatenate([v.view(torch.int16).numpy()] * n_masks)
    kr, vr, btr, slr, tot = O.compact_paged(kb, vb, masks.reshape(n_masks * L, H, T), page,
                                            max_pages)
    assert int(need[0].item()) == tot
    assert np.array_equal(sl.cpu().numpy().reshape(n_masks * L, H), slr)
    assert np.array_equal(bt.cpu().numpy().reshape(n_masks * L, H, max_pages), btr)
    assert np.array_equal(kp[:tot].cpu().view(torch.int16).numpy(), kr)
    assert np.array_equal(vp[:tot].cpu().view(torch.int16).numpy(), vr)
    if tot < cap:
        assert bool((kp[tot:] == 7.0).all())


def test_compact_capacity_overflow(C):
    L, H, T, d, page = 1, 2, 100, 128, 16
    mask = torch.ones(L, H, T, dtype=torch.uint8)
    k = torch.randn(L, H, T, d).to(torch.bfloat16).cuda()
    from kv_cache_eviction_lse_gb300.pipeline import Pages, compact_into
    dm = C.dims(L, H, H, d)
    pages = Pages(L, H, T, d, page, "cuda", capacity=5)
    pages.k_pages.fill_(3.0)
    ws = torch.empty(C.kvs_compact_workspace_size(dm, T), dtype=torch.uint8, device="cuda")
    compact_into(dm, k, k, T, mask.cuda(), pages, ws)
    torch.cuda.synchronize()
    assert int(pages.needed.item()) == 14
    assert bool((pages.block_table == -1).all())
    assert pages.seq_lens.cpu().tolist() == [[100, 100]]
    assert bool((pages.k_pages == 3.0).all())


# ----------------------------------------------------------------------------- decode

def _decode_run(C, L, H, B, d, T, w, page, tau, scores, k, v, capacity, max_pages):
    """Feed T tokens of every row one decode step at a time (graph-free)."""
    rows = L * H * B
    dev = "cuda"
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    ring_s = torch.full((L, H, B, max(w, 1)), float("nan"), device=dev)
    ring_k = torch.zeros(L, H, B, max(w, 1), d, dtype=torch.bfloat16, device=dev)
    ring_v = torch.zeros_like(ring_k)
    kp = torch.full((capacity, page, d), 7, dtype=torch.bfloat16, device=dev)
    vp = torch.full_like(kp, 7)
    nxt = torch.zeros(1, dtype=torch.int32, device=dev)
    bt = torch.full((L, H, B, max_pages), -1, dtype=torch.int32, device=dev)
    sl = torch.zeros(L, H, B, dtype=torch.int32, device=dev)
    sc, kc, vc = scores.cuda(), k.cuda(), v.cuda()
    dm = C.dims(L, H, H, d)
    for t in range(T):
        C.kvs_decode_step(dm, B, w, pos, sc[..., t].contiguous(), kc[..., t, :].contiguous(),
                          vc[..., t, :].contiguous(), ring_s if w else None,
                          ring_k if w else None, ring_v if w else None, tau, page, kp, vp,
                          capacity, nxt, bt, max_pages, sl)
    torch.cuda.synchronize()
    return dict(pos=pos, ring_s=ring_s, ring_k=ring_k, kp=kp, vp=vp, nxt=nxt, bt=bt, sl=sl)


@pytest.mark.parametrize("w,page,d", [(16, 16, 128), (0, 16, 128), (5, 1, 64), (40, 16, 64)])
def test_decode_step_matches_oracle(C, w, page, d):
    L, H, B, T, tau = 2, 3, 4, 150, 0.25
    gen = torch.Generator().manual_seed(w * 100 + page + d)
    scores = torch.round(torch.randn(L, H, B, T, generator=gen) * 2) / 2
    scores[torch.rand(L, H, B, T, generator=gen) < 0.03] = float("nan")
    k = torch.randn(L, H, B, T, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(L, H, B, T, d, generator=gen).to(torch.bfloat16)
    max_pages = -(-T // page)
    capacity = L * H * B * max_pages
    st = _decode_run(C, L, H, B, d, T, w, page, tau, scores, k, v, capacity, max_pages)
    assert (st["pos"].cpu() == T).all()
    kept, window = O.decode_prune(scores.reshape(-1, T).double().numpy(), tau, w)
    sl = st["sl"].cpu().reshape(-1).numpy()
    bt = st["bt"].cpu().reshape(-1, max_pages).numpy()
    kp, vp = st["kp"].cpu(), st["vp"].cpu()
    kr, vr = k.reshape(-1, T, d), v.reshape(-1, T, d)
    used = []
    for r in range(L * H * B):
        n = len(kept[r])
        assert sl[r] == n
        npg = -(-n // page)
        ids = bt[r]
        assert (ids[:npg] >= 0).all() and (ids[npg:] == -1).all()
        used += list(ids[:npg])
        got_k = kp[ids[:npg]].reshape(-1, d)
        got_v = vp[ids[:npg]].reshape(-1, d)
        assert torch.equal(got_k[:n].view(torch.int16), kr[r, kept[r]].view(torch.int16))
        assert torch.equal(got_v[:n].view(torch.int16), vr[r, kept[r]].view(torch.int16))
        assert (got_k[n:].float() == 0).all() and (got_v[n:].float() == 0).all()
        if w:
            rk = st["ring_k"].cpu().reshape(-1, w, d)[r]
            for t in window[r]:
                assert torch.equal(rk[t % w].view(torch.int16), kr[r, t].view(torch.int16))
    assert sorted(used) == list(range(int(st["nxt"].item())))  # each page handed out once
    code = C.kvs_device_error(clear=True)
    assert code == 0


def test_decode_step_pool_exhaustion_is_reported(C):
    L, H, B, d, T, w, page, tau = 1, 2, 2, 128, 40, 4, 4, -100.0   # keeps everything
    gen = torch.Generator().manual_seed(9)
    scores = torch.zeros(L, H, B, T)
    k = torch.randn(L, H, B, T, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(L, H, B, T, d, generator=gen).to(torch.bfloat16)
    capacity = 5   # far fewer pages than the 4 rows need
    st = _decode_run(C, L, H, B, d, T, w, page, tau, scores, k, v, capacity, max_pages=16)
    assert int(st["nxt"].item()) >= capacity
    sl = st["sl"].cpu().reshape(-1)
    assert int(sl.sum()) <= capacity * page
    assert C.kvs_device_error(clear=True) == 4
    # what was appended is still right: each row's first tokens in order
    bt = st["bt"].cpu().reshape(-1, 16).numpy()
    kr = k.reshape(-1, T, d)
    for r in range(L * H * B):
        n = int(sl[r])
        ids = bt[r][: -(-n // page)]
        assert (ids < capacity).all()
        got = st["kp"].cpu()[ids].reshape(-1, d)[:n]
        assert torch.equal(got.view(torch.int16), kr[r, :n].view(torch.int16))


# ----------------------------------------------------------------------------- value refit

REFIT_SHAPES = [
    # L, Hkv, Hq, d, T, n_q, k
    (1, 2, 4, 128, 300, 200, 100),
    (2, 1, 2, 64, 130, 70, 77),       # k not a multiple of 64, d = 64
    (1, 1, 3, 128, 520, 257, 1),      # a single kept key
    (1, 2, 2, 128, 700, 300, 333),    # several 128-row tiles of the Gram matrix
    (1, 1, 2, 128, 1600, 300, 1500),  # 24 Cholesky panels, more kept keys than rows
    (1, 1, 2, 64, 2100, 150, 2048),   # 32 panels
    (1, 2, 4, 128, 4400, 160, 4224),  # c4's 25 % budget plus its window (66 panels)
    # many problems: on 152 SMs the triangular solves take right-hand-side blocks of 32,
    # then 64 columns (16 above)
    (2, 40, 40, 64, 200, 70, 150),
    (3, 100, 100, 64, 200, 70, 150),
]


def _refit_objective(A, Ot, lam, V):
    return float(((A @ V - Ot) ** 2).sum() + lam * (V ** 2).sum())


@pytest.mark.parametrize("shape", REFIT_SHAPES, ids=[str(s) for s in REFIT_SHAPES])
def test_value_refit(C, shape):
    """The refit reaches the oracle's ridge optimum: the objective of the GPU solution,
    evaluated in fp64 with the oracle's A_S, O and lam, exceeds the optimum by at most
    2^-16 ||O||^2.  The GPU keeps O and A_S in fp16 (relative 2^-12 each, so ||dO||^2 <=
    2^-22 ||O||^2, and a least-squares solution moves the objective by at most ||dO||^2;
    the rounding of A_S moves it by the same order), and the fp32 Cholesky adds far less:
    the bound leaves a factor of 64."""
    L, Hkv, Hq, d, T, nq, k = shape
    lam_rel = 1e-3
    x = _inputs(L, Hkv, Hq, d, T, 0, nq, seed=T + k)
    gen = torch.Generator().manual_seed(k)
    mask = torch.zeros(L, Hkv, T, dtype=torch.uint8)
    for l in range(L):
        for h in range(Hkv):
            mask[l, h, torch.randperm(T, generator=gen)[:k]] = 1
    idx = [[torch.nonzero(mask[l, h]).flatten() for h in range(Hkv)] for l in range(L)]
    k_kept = torch.stack([torch.stack([x["k_ctx"][l, h, idx[l][h]] for h in range(Hkv)])
                          for l in range(L)]).contiguous()
    g = cuda(dict(q=x["q"], k_ctx=x["k_ctx"], v_ctx=x["v_ctx"], k_kept=k_kept))
    dm = C.dims(L, Hq, Hkv, d)
    nbytes = C.kvs_value_refit_workspace_size(dm, nq, k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    vfit = torch.full((L, Hkv, k, d), float("nan"), device="cuda")
    C.kvs_value_refit(dm, g["q"], nq, g["k_ctx"], g["v_ctx"], T, g["k_kept"], k, lam_rel, vfit,
                      ws, nbytes)
    torch.cuda.synchronize()
    assert C.kvs_device_error(clear=True) == 0
    q64, k64, v64 = f64(x["q"]), f64(x["k_ctx"]), f64(x["v_ctx"])
    _, parts = O.value_refit(q64, k64, v64, mask.numpy(), 1.0)  # A_S and O only
    vg = vfit.cpu().double().numpy()
    for l in range(L):
        for h in range(Hkv):
            A, Ot = parts[l][h]
            lam = lam_rel * float((A * A).sum()) / k
            vv, _ = O.value_refit(q64[l:l + 1, h * (Hq // Hkv):(h + 1) * (Hq // Hkv)],
                                  k64[l:l + 1, h:h + 1], v64[l:l + 1, h:h + 1],
                                  mask[l:l + 1, h:h + 1].numpy(), lam)
            best = _refit_objective(A, Ot, lam, vv[0][0])
            got = _refit_objective(A, Ot, lam, vg[l, h])
            assert np.isfinite(vg[l, h]).all()
            assert got - best <= 2.0 ** -16 * float((Ot ** 2).sum()), (l, h, got, best)
