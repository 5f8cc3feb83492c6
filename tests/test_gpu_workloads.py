"""Parity of the whole path on the workloads at their full sizes, in the launch
configuration the benchmark times (every layer in one call).  The oracle checks sampled
outputs it can afford: all of c1; the first and last layers of c2 (and of its value
refit); (layer 0, KV head 0) and (last layer, last KV head) of c3 and c4; the first and
last layers of c5; sampled tokens of c6's first and last layers; sampled rows of c4's
attention forward; whole decode steps of c7.  Compaction is checked bit-exactly given the
kernel's mask."""
import gc

import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_util import (LOG_SCORE_ATOL, LSE_ATOL, MASK_BAND, SCORE_RTOL, assert_close_abs,
                            assert_close_rel, assert_masks_match_near, cuda, f64, kth_value,
                            need_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    need_gpu()
    from kv_cache_eviction_lse_gb300 import build
    build.build()
    from kv_cache_eviction_lse_gb300 import pipeline, workloads
    return pipeline, workloads


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _check_pages(pages, l, h, k, v, mask_lh):
    """Compaction of one (layer, head) row is bit-exact given the kernel's mask."""
    kb = k.contiguous().view(torch.int16).numpy()[None, None]
    vb = v.contiguous().view(torch.int16).numpy()[None, None]
    kp, vp, bt, sl, tot = O.compact_paged(kb, vb, mask_lh[None, None], pages.page_size,
                                          pages.max_pages)
    assert int(pages.seq_lens[l, h].item()) == int(sl[0, 0])
    ids = pages.block_table[l, h].cpu().numpy()
    n = int((ids >= 0).sum())
    assert n == tot and (ids[n:] == -1).all()
    assert (np.diff(ids[:n]) == 1).all() if n > 1 else True
    got_k = pages.k_pages[ids[:n]].cpu().view(torch.int16).numpy()
    got_v = pages.v_pages[ids[:n]].cpu().view(torch.int16).numpy()
    assert np.array_equal(got_k, kp) and np.array_equal(got_v, vp)


def test_c1_full(mods):
    pipeline, W = mods
    wl = W.WORKLOADS["c1"]
    x = W.generate(wl)
    p = pipeline.make_pipeline(wl, cuda(x))
    p.step()
    torch.cuda.synchronize()
    q, kc, kt = f64(x["q"]), f64(x["k_ctx"]), f64(x["k_tail"])
    lse = O.lse(q, kc, kt)
    assert_close_abs(p.lse.cpu().numpy(), lse, LSE_ATOL, "c1 lse")
    s = O.kvzip_score(q, kc, kt, lse_=lse)
    assert_close_abs(p.score.cpu().numpy(), s, LOG_SCORE_ATOL, "c1 log score")
    k = wl.topk_budget(0.25)
    m_ref, k_ref = O.prune_topk(s, k, wl.w)
    assert (p.keeps[0].cpu().numpy() == k + wl.w).all() and (k_ref == k + wl.w).all()
    assert_masks_match_near(p.masks[0].cpu().numpy(), m_ref, s, kth_value(s, k, wl.w), MASK_BAND,
                            "c1 mask", log_domain=True)
    _check_pages(p.pages[0], 0, 0, x["k_ctx"][0, 0], x["v_ctx"][0, 0], p.masks[0][0, 0].cpu().numpy())


def test_c2_full(mods):
    pipeline, W = mods
    wl = W.WORKLOADS["c2"]
    x = W.generate(wl)
    p = pipeline.make_pipeline(wl, cuda(x))
    p.step()
    torch.cuda.synchronize()
    for l in (0, wl.L - 1):
        sl = slice(l, l + 1)
        q, kc, kt = f64(x["q"][sl]), f64(x["k_ctx"][sl]), f64(x["k_tail"][sl])
        lse = O.lse(q, kc, kt)
        assert_close_abs(p.lse[sl].cpu().numpy(), lse, LSE_ATOL, f"c2 lse layer {l}")
        vn = O.value_norm(f64(x["v_ctx"][sl]), f64(x["w_o"][sl]), wl.H_q)
        assert_close_rel(p.vnorm[sl].cpu().numpy(), vn, 1e-4, f"c2 vnorm layer {l}")
        s = O.kvzip_score(q, kc, kt, lse_=lse, vnorm=vn, h=f64(x["h"][sl]))
        assert_close_abs(p.score[sl].cpu().numpy(), s, LOG_SCORE_ATOL, f"c2 log score layer {l}")
        for r, m, kp, pg in zip(p.ratios, p.masks, p.keeps, p.pages):
            k = wl.topk_budget(r)
            m_ref, k_ref = O.prune_topk(s, k, wl.w)
            assert np.array_equal(kp[sl].cpu().numpy(), k_ref)
            assert_masks_match_near(m[sl].cpu().numpy(), m_ref, s, kth_value(s, k, wl.w),
                                    MASK_BAND, f"c2 mask r={r} layer {l}", log_domain=True)
            for h in range(wl.H_kv):
                _check_pages(pg, l, h, x["k_ctx"][l, h], x["v_ctx"][l, h], m[l, h].cpu().numpy())


def _layer_tau(score_l, T, w, qtl):
    """Reading of the c3 threshold: the lower nearest-rank quantile qtl of the layer's
    non-window scores over all its KV heads, sorted[floor(qtl (N - 1))], taken from the
    kernel's fp32 scores (a workload parameter, then used by both sides)."""
    flat = score_l[:, : T - w].flatten()
    k = int(np.floor(qtl * (flat.numel() - 1))) + 1
    return float(torch.kthvalue(flat.float().cpu(), k).values)


def _c3_oracle_row(x, wl, l, hk, keys=None):
    """The oracle's chunked KVzip+ log score of KV head hk of layer l, on the context keys
    `keys` (all when None).  Each chunk's LSE runs over every key its queries see (the
    full context and the chunk's tail); the score of a key needs only its own column of
    the attention rows, so the context passed to the score holds just the sampled keys
    (every context key is visible to every scoring query, so their visibility and the
    tail's causal offsets are unchanged)."""
    g, d = wl.g, wl.d
    hs = slice(hk * g, (hk + 1) * g)
    sl = slice(l, l + 1)
    kc = f64(x["k_ctx"][sl, hk:hk + 1])
    ks = kc if keys is None else kc[:, :, keys]
    v = f64(x["v_ctx"][sl, hk:hk + 1])
    vn = O.value_norm(v if keys is None else v[:, :, keys],
                      f64(x["w_o"][sl, :, hk * g * d:(hk + 1) * g * d]), g)
    best = None
    for c in range(wl.n_chunks):
        q = f64(x["q"][c][sl, hs])
        tail = f64(x["k_tail"][c][sl, hk:hk + 1])
        lse_c = O.lse(q, kc, tail)
        s = O.kvzip_score(q, ks, tail, lse_=lse_c, vnorm=vn, h=f64(x["h"][c][sl]), log=False)
        best = s if best is None else np.maximum(best, s)
    with np.errstate(divide="ignore"):
        return vn, np.log(best)


def test_c3_full_corners(mods):
    """c3 at full size: (layer 0, KV head 0) on every context key, and the far corner
    (last layer, last KV head) on its first and last 2048 keys, against the oracle;
    the per-layer threshold at the 25th percentile of the layer's non-window scores
    over all 8 KV heads (selected on the GPU in the step, checked against the same
    order statistic of the kernel's scores), then the masks and pages of both rows."""
    pipeline, W = mods
    wl = W.WORKLOADS["c3"]
    x = W.generate(wl, device="cuda")
    p = pipeline.make_pipeline(wl, x)
    p.step()
    torch.cuda.synchronize()
    g, T, w = wl.g, wl.T, wl.w
    # the step selects tau on the GPU: exactly the quantile of the kernel's own scores
    tau_gpu = p.tau_dev[: wl.L].cpu().tolist()
    assert tau_gpu == [_layer_tau(p.score[l], T, w, wl.tau_quantile) for l in range(wl.L)]
    keys_far = np.r_[0:2048, T - 2048:T]
    for l, hk, keys in ((0, 0, None), (wl.L - 1, wl.H_kv - 1, keys_far)):
        vn, s = _c3_oracle_row(x, wl, l, hk, keys)
        cols = slice(None) if keys is None else keys
        vg = p.vnorm[l:l + 1, hk * g:(hk + 1) * g].cpu().numpy()[..., cols]
        assert_close_rel(vg, vn, 1e-4, f"c3 vnorm (layer {l}, head {hk})")
        got = p.score[l:l + 1, hk:hk + 1].cpu().numpy()[..., cols]
        assert_close_abs(got, s, LOG_SCORE_ATOL, f"c3 log score (layer {l}, head {hk})")
        tau = tau_gpu[l]
        m_ref, _ = O.prune_threshold(s, tau, 0)
        pos = np.arange(T)[cols]
        m_ref[..., pos >= T - w] = 1  # the window (positions of the sampled keys)
        mg = p.mask[l:l + 1, hk:hk + 1].cpu().numpy()
        assert_masks_match_near(mg[..., cols], m_ref, s, np.full((1, 1), tau), MASK_BAND,
                                f"c3 mask (layer {l}, head {hk})", log_domain=True)
        # the whole row's mask is the threshold rule on the kernel's own fp32 scores
        m_same, _ = O.prune_threshold(p.score[l:l + 1, hk:hk + 1].cpu().numpy().astype(np.float64),
                                      np.float32(tau), w)
        assert np.array_equal(mg, m_same)
        _check_pages(p.pages, l, hk, x["k_ctx"][l, hk].cpu(), x["v_ctx"][l, hk].cpu(), mg[0, 0])


def test_c4_full_corners(mods):
    """c4 at full size: LSE, future mass, top-k masks and pages of (layer 0, KV head 0)
    and of the far corner (last layer, last KV head) against the oracle."""
    pipeline, W = mods
    wl = W.WORKLOADS["c4"]
    x = W.generate(wl, device="cuda")
    p = pipeline.make_pipeline(wl, x)
    p.step()
    torch.cuda.synchronize()
    g = wl.g
    for l, hk in ((0, 0), (wl.L - 1, wl.H_kv - 1)):
        sl, hs = slice(l, l + 1), slice(hk * g, (hk + 1) * g)
        q = f64(x["q"][sl, hs])
        k = f64(x["k"][sl, hk:hk + 1])
        lse = O.lse(q, k, None)
        assert_close_abs(p.lse[sl, hs].cpu().numpy(), lse, LSE_ATOL, f"c4 lse (layer {l}, head {hk})")
        f = O.future_attention_mass(q, k, wl.w, lse_=lse)
        assert_close_rel(p.score[sl, hk:hk + 1].cpu().numpy(), f, SCORE_RTOL,
                         f"c4 future mass (layer {l}, head {hk})")
        for r, m, kp, pg in zip(p.ratios, p.masks, p.keeps, p.pages):
            kk = wl.topk_budget(r)
            m_ref, k_ref = O.prune_topk(f, kk, wl.w)
            assert int(kp[l, hk].item()) == int(k_ref[0, 0]) == kk + wl.w
            assert_masks_match_near(m[sl, hk:hk + 1].cpu().numpy(), m_ref, f,
                                    kth_value(f, kk, wl.w), MASK_BAND,
                                    f"c4 mask r={r} (layer {l}, head {hk})", log_domain=False)
            _check_pages(pg, l, hk, x["k"][l, hk].cpu(), x["v"][l, hk].cpu(), m[l, hk].cpu().numpy())


def test_c5_full_first_and_last_layer(mods):
    pipeline, W = mods
    wl = W.WORKLOADS["c5"]
    x = W.generate(wl, device="cuda")
    p = pipeline.make_pipeline(wl, x)
    p.step()
    torch.cuda.synchronize()
    for l in (0, wl.L - 1):
        sl = slice(l, l + 1)
        z = O.linear_surrogate(f64(x["h"][sl]), f64(x["W"][sl]), x["b"][sl].double().cpu().numpy())
        zg = p.score[sl].cpu().numpy()
        assert_close_abs(zg, z, LOG_SCORE_ATOL, f"c5 surrogate (layer {l})")
        m_ref, _ = O.prune_threshold(z, wl.tau, wl.w)
        mg = p.mask[sl].cpu().numpy()
        assert_masks_match_near(mg, m_ref, z, np.full(z.shape[:-1], wl.tau), MASK_BAND,
                                f"c5 mask (layer {l})", log_domain=True)
        assert np.array_equal(p.keep[sl].cpu().numpy(), mg.sum(-1))
        for h in range(wl.H_kv):
            _check_pages(p.pages, l, h, x["k"][l, h].cpu(), x["v"][l, h].cpu(), mg[0, h])
    # the page plan covers every layer: offsets are the prefix sum of ceil(keep/16)
    sl = p.pages.seq_lens.cpu().numpy().ravel()
    first = p.pages.block_table[:, :, 0].cpu().numpy().ravel()
    npg = -(-sl // wl.page_size)
    assert np.array_equal(first[npg > 0], (np.cumsum(npg) - npg)[npg > 0])
    assert int(p.pages.needed.item()) == int(npg.sum())


def test_c6_full_sampled(mods):
    """c6: the MLP surrogate of layers 0 and 35 on their first and last 4096 tokens
    against the oracle; each layer's whole mask against the threshold rule applied to the
    kernel's own scores; pages bit-exact."""
    pipeline, W = mods
    wl = W.WORKLOADS["c6"]
    x = W.generate(wl, device="cuda")
    p = pipeline.make_pipeline(wl, x)
    p.step()
    torch.cuda.synchronize()
    rows = np.r_[0:4096, wl.T - 4096:wl.T]
    for l in (0, wl.L - 1):
        sl = slice(l, l + 1)
        z = O.mlp_surrogate(f64(x["h"][sl, rows]), f64(x["W1"][sl]), x["b1"][sl].double().cpu().numpy(),
                            f64(x["W2"][sl]), x["b2"][sl].double().cpu().numpy())
        zg = p.score[sl].cpu().numpy()
        assert_close_abs(zg[..., rows], z, LOG_SCORE_ATOL,
                         f"c6 MLP surrogate (layer {l}, sampled tokens)")
        mg = p.mask[sl].cpu().numpy()
        # the threshold rule applied to the kernel's own fp32 scores, over the whole layer
        m_same, _ = O.prune_threshold(zg.astype(np.float64), np.float32(wl.tau), wl.w)
        assert np.array_equal(mg, m_same)
        # and the oracle's decision on the sampled tokens, except next to tau
        m_ref, _ = O.prune_threshold(z, wl.tau, 0)
        m_ref[..., rows >= wl.T - wl.w] = 1
        assert_masks_match_near(mg[..., rows], m_ref, z, np.full(z.shape[:-1], wl.tau), MASK_BAND,
                                f"c6 mask (layer {l}, sampled tokens)", log_domain=True)
        assert np.array_equal(p.keep[sl].cpu().numpy(), mg.sum(-1))
        for h in range(wl.H_kv):
            _check_pages(p.pages, l, h, x["k"][l, h].cpu(), x["v"][l, h].cpu(), mg[0, h])


def test_c4_attention_forward_sampled_rows(mods):
    """The attention forward (output + LSE) as pass 1 of the c4 step: the first and the
    last 256 queries of layer 0, KV-head group 0, against the oracle, and its LSE
    against the LSE-only pass 1 everywhere."""
    pipeline, W = mods
    wl = W.WORKLOADS["c4"]
    x = W.generate(wl, device="cuda")
    p = pipeline.make_pipeline(wl, x, attn_forward=True)
    p.step()
    ref = pipeline.make_pipeline(wl, x)
    ref.score_step()
    torch.cuda.synchronize()
    assert_close_abs(p.lse.cpu().numpy(), ref.lse.cpu().numpy(), LSE_ATOL, "c4 forward lse vs kvs_lse")
    g, T, n = wl.g, wl.T, 256
    for lo in (0, T - n):
        q = f64(x["q"][0:1, 0:g, lo:lo + n])
        k = f64(x["k"][0:1, 0:1, : lo + n])
        v = f64(x["v"][0:1, 0:1, : lo + n])
        o_ref, lse_ref = O.attention_forward(q, k, None, v, None)
        assert_close_abs(p.lse[0:1, 0:g, lo:lo + n].cpu().numpy(), lse_ref, LSE_ATOL, "c4 forward lse")
        err = np.abs(f64(p.o[0:1, 0:g, lo:lo + n]) - o_ref)
        vmax = np.abs(v).max()
        tol = 2.0 ** -8 * (np.abs(o_ref) + vmax)
        assert (err <= tol).all(), f"c4 forward o rows {lo}: max err {err.max()}"


def test_c7_decode_steps_full_size(mods):
    """c7 at full size (32 layers x 8 KV heads x 64 sequences): the surrogate score of
    the arriving tokens against the oracle, then 2w + 37 decode steps.  The synthetic
    step repeats the same arriving token, so a row keeps every token that leaves its
    window (steps - w of them) iff its score passes tau; pages hold copies of that
    token's K and V."""
    pipeline, W = mods
    wl = W.WORKLOADS["c7"]
    x = W.generate(wl, device="cuda")
    p = pipeline.make_pipeline(wl, x, max_steps=512)
    steps = 2 * wl.w + 37
    for _ in range(steps):
        p.step()
    torch.cuda.synchronize()
    z = O.linear_surrogate(f64(x["h"]), f64(x["W"]), x["b"].double().cpu().numpy())
    zg = p.score.cpu().numpy()
    assert_close_abs(zg, z, LOG_SCORE_ATOL, "c7 surrogate of the arriving tokens")
    assert (p.pos.cpu() == steps).all()
    keep_row = (zg.astype(np.float64) >= np.float32(wl.tau))
    sl = p.seq_lens.cpu().numpy()
    assert np.array_equal(sl, np.where(keep_row, steps - wl.w, 0))
    kept, window = O.decode_prune(np.repeat(zg.reshape(-1, 1).astype(np.float64), steps, 1),
                                  np.float32(wl.tau), wl.w)
    assert [len(k) for k in kept] == list(sl.reshape(-1))
    bt = p.block_table.cpu().numpy()
    kpages = p.k_pages
    for l in (0, wl.L - 1):
        for h in range(wl.H_kv):
            for b in (0, wl.batch - 1):
                n = int(sl[l, h, b])
                ids = bt[l, h, b, : -(-n // wl.page_size)]
                got = kpages[torch.as_tensor(ids, device="cuda").long()].reshape(-1, wl.d)[:n]
                want = x["k"][l, h, b][None].expand(n, wl.d)
                assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert C_error_clear() == 0


def C_error_clear():
    from kv_cache_eviction_lse_gb300 import capi
    return capi.kvs_device_error(clear=True)


def test_c2_value_refit_first_and_last_layer(mods):
    """Select+Fit at c2 size: the r = 0.3 top-k keys (614 per head) of every layer and
    head, refitted; the first and last layers' KV heads reach the fp64 ridge optimum within
    the bound of the per-op test (objective excess <= 2^-16 ||O||^2)."""
    pipeline, W = mods
    wl = W.WORKLOADS["c2"]
    x = W.generate(wl)
    p = pipeline.make_pipeline(wl, cuda(x), refit=True)
    p.step()
    torch.cuda.synchronize()
    from kv_cache_eviction_lse_gb300 import capi
    assert capi.kvs_device_error(clear=True) == 0
    k = p.k_fit
    g = wl.g
    for l in (0, wl.L - 1):
        mask = p.masks[0][l:l + 1].cpu().numpy()
        assert (mask.sum(-1) == k).all()
        q64, k64, v64 = f64(x["q"][l:l + 1]), f64(x["k_ctx"][l:l + 1]), f64(x["v_ctx"][l:l + 1])
        # the dense gather is the kept keys in position order
        for h in range(wl.H_kv):
            idx = np.nonzero(mask[0, h])[0]
            assert np.array_equal(p.k_kept()[l, h].cpu().view(torch.int16).numpy(),
                                  x["k_ctx"][l, h][idx].view(torch.int16).numpy())
        _, parts = O.value_refit(q64, k64, v64, mask, 1.0)
        vg = p.v_fit[l].cpu().double().numpy()
        for h in range(wl.H_kv):
            A, Ot = parts[0][h]
            lam = p.REFIT_LAMBDA_REL * float((A * A).sum()) / k
            vv, _ = O.value_refit(q64[:, h * g:(h + 1) * g], k64[:, h:h + 1], v64[:, h:h + 1],
                                  mask[:, h:h + 1], lam)
            f = lambda V: float(((A @ V - Ot) ** 2).sum() + lam * (V ** 2).sum())
            assert f(vg[h]) - f(vv[0][0]) <= 2.0 ** -16 * float((Ot ** 2).sum()), (l, h)
