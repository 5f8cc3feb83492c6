"""Host orchestration of the scoring -> pruning -> compaction path, one class per workload.

Each pipeline allocates its outputs and scratch once (torch, on the inputs' device) and
``step()`` enqueues the library calls on the current stream: no arithmetic of the
method happens here, only call sequencing and buffer management.

  KVzip / KVzip+ (c1, c2)   [vnorm] -> lse -> score_max -> top-k per budget -> compact
  chunked KVzip+  (c3)      vnorm -> per chunk (lse -> score_max, max-accumulated)
                            -> threshold at the layer's score quantile -> compact
  KVpop target    (c4)      lse (causal self-attention) -> future_sum -> top-k per budget
                            -> compact
  KVzap           (c5)      surrogate (+ fused threshold) -> compact
"""
from __future__ import annotations

import types

import torch

from . import capi as C
from .workloads import Workload


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


class Pages:
    """Paged cache buffers for one compaction of a [L][H][T][d] K/V pair."""

    def __init__(self, L, H, T, d, page_size, device, capacity=None):
        self.page_size = page_size
        self.max_pages = -(-T // page_size)
        self.capacity = capacity if capacity is not None else L * H * self.max_pages
        self.k_pages = _empty((self.capacity, page_size, d), torch.bfloat16, device)
        self.v_pages = _empty((self.capacity, page_size, d), torch.bfloat16, device)
        self.block_table = _empty((L, H, self.max_pages), torch.int32, device)
        self.seq_lens = _empty((L, H), torch.int32, device)
        self.needed = _empty((1,), torch.int32, device)

    def bytes_written(self):
        """Algorithmic bytes a compaction writes: kept K and V rows."""
        d = self.k_pages.shape[-1]
        return int(self.seq_lens.sum().item()) * 2 * d * 2


class PagePool:
    """One paged cache for n masks over the same [L][H][T][d] K/V pair: the pages of mask
    b follow those of masks 0 .. b-1 in one pool; ``view(b)`` exposes mask b's block
    table and lengths (absolute page ids into the shared pool)."""

    def __init__(self, n, L, H, T, d, page_size, device):
        self.n = n
        self.page_size = page_size
        self.max_pages = -(-T // page_size)
        self.capacity = n * L * H * self.max_pages
        self.k_pages = _empty((self.capacity, page_size, d), torch.bfloat16, device)
        self.v_pages = _empty((self.capacity, page_size, d), torch.bfloat16, device)
        self.block_table = _empty((n, L, H, self.max_pages), torch.int32, device)
        self.seq_lens = _empty((n, L, H), torch.int32, device)
        self.needed = _empty((1,), torch.int32, device)

    def view(self, b):
        return types.SimpleNamespace(page_size=self.page_size, max_pages=self.max_pages,
                                     capacity=self.capacity, k_pages=self.k_pages,
                                     v_pages=self.v_pages, block_table=self.block_table[b],
                                     seq_lens=self.seq_lens[b], needed=self.needed)


def compact_multi_into(dm, k, v, T, masks, pool: PagePool, ws):
    C.kvs_compact_paged_multi(dm, k, v, T, pool.n, masks, pool.page_size, pool.k_pages,
                              pool.v_pages, pool.capacity, pool.block_table, pool.max_pages,
                              pool.seq_lens, pool.needed, ws, ws.numel())


def compact_into(dm, k, v, T, mask, pages: Pages, ws):
    C.kvs_compact_paged(dm, k, v, T, mask, pages.page_size, pages.k_pages, pages.v_pages,
                        pages.capacity, pages.block_table, pages.max_pages, pages.seq_lens,
                        pages.needed, ws, ws.numel())


class _Budgets:
    """Top-k budgets over one score tensor: all masks in one [n][L][H_kv][T] tensor, all
    pages in one pool, each selected and compacted by one library call."""

    def _budgets(self, wl, L, dev, ratios):
        self.ratios = tuple(ratios if ratios is not None else wl.keep_ratios)
        n = len(self.ratios)
        self.mask_all = _empty((n, L, wl.H_kv, wl.T), torch.uint8, dev)
        self.keep_all = _empty((n, L, wl.H_kv), torch.int32, dev)
        self.masks = [self.mask_all[b] for b in range(n)]
        self.keeps = [self.keep_all[b] for b in range(n)]
        self.pool = PagePool(n, L, wl.H_kv, wl.T, wl.d, wl.page_size, dev)
        self.pages = [self.pool.view(b) for b in range(n)]
        self.cws = _empty((C.kvs_compact_multi_workspace_size(self.dm, wl.T, n),), torch.uint8, dev)


def _prune_budgets(p):
    wl = p.wl
    C.kvs_prune_topk_multi(p.dm, p.score, wl.T, [wl.topk_budget(r) for r in p.ratios], wl.w,
                           p.mask_all, p.keep_all)


class KVzipPipeline(_Budgets):
    """c1 / c2: KVzip (plain) or KVzip+ scoring of the context, then top-k budgets."""

    # ridge weight of the value refit relative to the mean diagonal of A_S^T A_S (reading:
    # the pages name ridge regression but no weight)
    REFIT_LAMBDA_REL = 1e-3

    def __init__(self, wl: Workload, x: dict, ratios=None, refit=False):
        self.wl, self.x = wl, x
        dev = x["q"].device
        L = x["q"].shape[0]
        self.L = L
        self.plus = "w_o" in x
        self.dm = C.dims(L, wl.H_q, wl.H_kv, wl.d, wl.D_h if self.plus else 0)
        self.n_q, self.n_tail = x["q"].shape[2], x["k_tail"].shape[2]
        self.lse = _empty((L, wl.H_q, self.n_q), torch.float32, dev)
        self.score = _empty((L, wl.H_kv, wl.T), torch.float32, dev)
        self.vnorm = None
        if self.plus:
            self.vnorm = _empty((L, wl.H_q, wl.T), torch.float32, dev)
            self.vws = _empty((C.kvs_vnorm_workspace_size(self.dm),), torch.uint8, dev)
        self.sws = _empty((max(16, C.kvs_score_max_workspace_size(self.dm, self.n_q, self.plus)),),
                          torch.uint8, dev)
        self._budgets(wl, L, dev, ratios)
        # refit: Select+Fit on the first budget -- the kept keys gathered densely (one
        # page of exactly k rows per head), then their values refitted in closed form
        self.refit = refit
        if refit:
            self.k_fit = wl.topk_budget(self.ratios[0]) + wl.w
            self.dense = Pages(L, wl.H_kv, wl.T, wl.d, self.k_fit, dev)
            self.v_fit = _empty((L, wl.H_kv, self.k_fit, wl.d), torch.float32, dev)
            n = C.kvs_value_refit_workspace_size(self.dm, self.n_q, self.k_fit)
            self.rws = _empty((n,), torch.uint8, dev)

    def k_kept(self):
        """The kept keys of the first budget as [L][H_kv][k][d] (refit only)."""
        wl = self.wl
        return self.dense.k_pages[: self.L * wl.H_kv].view(self.L, wl.H_kv, self.k_fit, wl.d)

    def _refit(self):
        wl, x, dm = self.wl, self.x, self.dm
        compact_into(dm, x["k_ctx"], x["v_ctx"], wl.T, self.masks[0], self.dense, self.cws)
        C.kvs_value_refit(dm, x["q"], self.n_q, x["k_ctx"], x["v_ctx"], wl.T, self.k_kept(),
                          self.k_fit, self.REFIT_LAMBDA_REL, self.v_fit, self.rws,
                          self.rws.numel())

    def score_step(self):
        if self.plus:
            self._vnorm()
        self._lse()
        self._score()

    def prune_step(self):
        self._prune()
        self._compact()

    def _vnorm(self):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_vnorm(dm, x["v_ctx"], wl.T, x["w_o"], self.vnorm, self.vws, self.vws.numel())

    def _lse(self):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_lse(dm, x["q"], self.n_q, x["k_ctx"], wl.T, x["k_tail"], self.n_tail, self.lse)

    def _score(self):
        wl, x, dm = self.wl, self.x, self.dm
        if self.plus:
            C.kvs_score_max(dm, x["q"], self.n_q, x["k_ctx"], wl.T, self.lse, self.vnorm, x["h"], 0,
                            self.score, self.sws, self.sws.numel())
        else:
            C.kvs_score_max(dm, x["q"], self.n_q, x["k_ctx"], wl.T, self.lse, None, None, 0,
                            self.score, self.sws, self.sws.numel())

    def _prune(self):
        _prune_budgets(self)

    def _compact(self):
        x = self.x
        compact_multi_into(self.dm, x["k_ctx"], x["v_ctx"], self.wl.T, self.mask_all, self.pool,
                           self.cws)

    def stages(self):
        """(name, callable) per library entry point, in step order."""
        st = [("kvs_vnorm", self._vnorm)] if self.plus else []
        st += [("kvs_lse", self._lse), ("kvs_score_max", self._score),
               ("kvs_prune_topk_multi", self._prune), ("kvs_compact_paged_multi", self._compact)]
        return st + ([("kvs_value_refit", self._refit)] if self.refit else [])

    def step(self):
        for _, fn in self.stages():
            fn()


class ChunkedKVzipPipeline:
    """c3: chunked KVzip+ reconstruction, per-layer threshold tau, window w."""

    def __init__(self, wl: Workload, x: dict, tau=None):
        self.wl, self.x = wl, x
        dev = x["k_ctx"].device
        L = x["k_ctx"].shape[0]
        self.L = L
        self.dm = C.dims(L, wl.H_q, wl.H_kv, wl.d, wl.D_h)
        self.dm1 = C.dims(1, wl.H_q, wl.H_kv, wl.d, wl.D_h)
        self.lse = _empty((L, wl.H_q, wl.n_rep), torch.float32, dev)
        self.score = _empty((L, wl.H_kv, wl.T), torch.float32, dev)
        self.vnorm = _empty((L, wl.H_q, wl.T), torch.float32, dev)
        self.vws = _empty((C.kvs_vnorm_workspace_size(self.dm),), torch.uint8, dev)
        self.sws = _empty((max(16, C.kvs_score_max_workspace_size(self.dm, wl.n_rep, 1)),),
                          torch.uint8, dev)
        # per-layer threshold: the tau_quantile of the layer's non-window scores, set on
        # the device by kvs_prune_quantile in every step; a caller may instead fix it
        # (a list of floats, one per layer), as a model-specific tau would be
        self.tau = tau
        self.tau_dev = _empty((max(L, 4),), torch.float32, dev)
        self.mask = _empty((L, wl.H_kv, wl.T), torch.uint8, dev)
        self.keep = _empty((L, wl.H_kv), torch.int32, dev)
        self.pages = Pages(L, wl.H_kv, wl.T, wl.d, wl.page_size, dev)
        self.cws = _empty((C.kvs_compact_workspace_size(self.dm, wl.T),), torch.uint8, dev)

    def _vnorm(self):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_vnorm(dm, x["v_ctx"], wl.T, x["w_o"], self.vnorm, self.vws, self.vws.numel())

    def _lse(self, c):
        wl, x, dm = self.wl, self.x, self.dm
        nt = x["k_tail"][c].shape[2]
        C.kvs_lse(dm, x["q"][c], wl.n_rep, x["k_ctx"], wl.T, x["k_tail"][c], nt, self.lse)

    def _score(self, c):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_score_max(dm, x["q"][c], wl.n_rep, x["k_ctx"], wl.T, self.lse, self.vnorm, x["h"][c],
                        int(c > 0), self.score, self.sws, self.sws.numel())

    def score_step(self):
        self._vnorm()
        for c in range(self.wl.n_chunks):
            self._lse(c)
            self._score(c)

    def _prune(self):
        wl = self.wl
        if self.tau is None:
            C.kvs_prune_quantile(self.dm, self.score, wl.T, wl.tau_quantile, wl.w, self.tau_dev,
                                 self.mask, self.keep)
            return
        for l in range(self.L):
            C.kvs_prune_mask(self.dm1, self.score[l], wl.T, C.KVS_THRESHOLD, float(self.tau[l]), 0,
                             wl.w, self.mask[l], self.keep[l])

    def _compact(self):
        wl, x = self.wl, self.x
        compact_into(self.dm, x["k_ctx"], x["v_ctx"], wl.T, self.mask, self.pages, self.cws)

    def prune_step(self):
        self._prune()
        self._compact()

    def stages(self):
        """(name, callable) per library entry point; lse and score_max cover all chunks
        (the chunks alternate lse -> score_max, so they are timed as pairs per chunk)."""
        def lse_all():
            for c in range(self.wl.n_chunks):
                self._lse(c)

        def score_all():
            for c in range(self.wl.n_chunks):
                self._score(c)
        prune = "kvs_prune_quantile" if self.tau is None else "kvs_prune_mask"
        return [("kvs_vnorm", self._vnorm), ("kvs_lse", lse_all), ("kvs_score_max", score_all),
                (prune, self._prune), ("kvs_compact_paged", self._compact)]

    def step(self):
        self.score_step()
        self.prune_step()


class FuturePipeline(_Budgets):
    """c4: KVpop future-attention target, then top-k budgets plus the window."""

    def __init__(self, wl: Workload, x: dict, ratios=None, attn_forward=False):
        self.wl, self.x = wl, x
        dev = x["q"].device
        L = x["q"].shape[0]
        self.L = L
        self.dm = C.dims(L, wl.H_q, wl.H_kv, wl.d, 0)
        self.lse = _empty((L, wl.H_q, wl.T), torch.float32, dev)
        # attn_forward: pass 1 is the attention forward itself (output + LSE), as in a
        # model that runs attention anyway and hands its LSE to the transposed pass
        self.attn_forward = attn_forward
        self.o = _empty((L, wl.H_q, wl.T, wl.d), torch.bfloat16, dev) if attn_forward else None
        self.score = _empty((L, wl.H_kv, wl.T), torch.float32, dev)
        self.fws = _empty((C.kvs_score_future_sum_workspace_size(self.dm, wl.T),), torch.uint8, dev)
        self._budgets(wl, L, dev, ratios)

    def _lse(self):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_lse(dm, x["q"], wl.T, x["k"], wl.T, None, 0, self.lse)

    def _forward(self):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_attn_fwd(dm, x["q"], wl.T, x["k"], x["v"], wl.T, None, None, 0, self.o, self.lse)

    def _future(self):
        wl, x, dm = self.wl, self.x, self.dm
        C.kvs_score_future_sum(dm, x["q"], x["k"], wl.T, self.lse, wl.w, self.score, self.fws,
                               self.fws.numel())

    def _prune(self):
        _prune_budgets(self)

    def _compact(self):
        x = self.x
        compact_multi_into(self.dm, x["k"], x["v"], self.wl.T, self.mask_all, self.pool, self.cws)

    def _pass1(self):
        return ("kvs_attn_fwd", self._forward) if self.attn_forward else ("kvs_lse", self._lse)

    def score_step(self):
        self._pass1()[1]()
        self._future()

    def prune_step(self):
        self._prune()
        self._compact()

    def stages(self):
        return [self._pass1(), ("kvs_score_future_sum", self._future),
                ("kvs_prune_topk_multi", self._prune), ("kvs_compact_paged_multi", self._compact)]

    def step(self):
        for _, fn in self.stages():
            fn()


class KVzapPipeline:
    """c5: KVzap-Linear surrogate with fused threshold + window, then compaction."""

    def __init__(self, wl: Workload, x: dict):
        self.wl, self.x = wl, x
        dev = x["h"].device
        L = x["h"].shape[0]
        self.L = L
        self.dm = C.dims(L, wl.H_q, wl.H_kv, wl.d, wl.D_h)
        self.score = _empty((L, wl.H_kv, wl.T), torch.float32, dev)
        self.mask = _empty((L, wl.H_kv, wl.T), torch.uint8, dev)
        self.keep = _empty((L, wl.H_kv), torch.int32, dev)
        self.pages = Pages(L, wl.H_kv, wl.T, wl.d, wl.page_size, dev)
        self.cws = _empty((C.kvs_compact_workspace_size(self.dm, wl.T),), torch.uint8, dev)

    def score_step(self):
        wl, x = self.wl, self.x
        C.kvs_surrogate(self.dm, x["h"], wl.T, x["W"], x["b"], self.score, wl.tau, wl.w, self.mask,
                        self.keep)

    def prune_step(self):
        wl, x = self.wl, self.x
        compact_into(self.dm, x["k"], x["v"], wl.T, self.mask, self.pages, self.cws)

    def stages(self):
        return [("kvs_surrogate", self.score_step), ("kvs_compact_paged", self.prune_step)]

    def step(self):
        self.score_step()
        self.prune_step()


class KVzapMLPPipeline(KVzapPipeline):
    """c6: KVzap-MLP surrogate (D_h -> D_h/8 -> H_kv) with the threshold + window rule,
    then compaction."""

    def score_step(self):
        wl, x = self.wl, self.x
        C.kvs_surrogate_mlp(self.dm, x["h"], wl.T, wl.D_mid, x["W1"], x["b1"], x["W2"], x["b2"],
                            self.score, wl.tau, wl.w, self.mask, self.keep)

    def stages(self):
        return [("kvs_surrogate_mlp", self.score_step), ("kvs_compact_paged", self.prune_step)]


class DecodePipeline:
    """c7: one decode step of `batch` sequences per call: the KVzap-Linear score of the
    arriving token (the surrogate over the batch's hidden states), then the window-
    boundary decision and append (kvs_decode_step).  State (ring, pages, positions)
    lives on the device and advances with every step; `reset` starts over."""

    def __init__(self, wl: Workload, x: dict, max_steps=4096):
        self.wl, self.x = wl, x
        dev = x["h"].device
        L, H, B, d, w = x["h"].shape[0], wl.H_kv, wl.batch, wl.d, wl.w
        self.L, self.B = L, B
        self.dm = C.dims(L, wl.H_q, H, d, wl.D_h)
        self.rows = L * H * B
        self.max_pages = -(-max_steps // wl.page_size) + 1
        self.capacity = self.rows * self.max_pages
        self.score = _empty((L, H, B), torch.float32, dev)
        self.pos = torch.zeros(B, dtype=torch.int32, device=dev)
        self.ring_score = _empty((L, H, B, w), torch.float32, dev)
        self.ring_k = _empty((L, H, B, w, d), torch.bfloat16, dev)
        self.ring_v = _empty((L, H, B, w, d), torch.bfloat16, dev)
        self.k_pages = _empty((self.capacity, wl.page_size, d), torch.bfloat16, dev)
        self.v_pages = _empty((self.capacity, wl.page_size, d), torch.bfloat16, dev)
        self.next_page = torch.zeros(1, dtype=torch.int32, device=dev)
        self.block_table = torch.full((L, H, B, self.max_pages), -1, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros((L, H, B), dtype=torch.int32, device=dev)
        self.reset()

    def reset(self):
        self.pos.zero_()
        self.next_page.zero_()
        self.seq_lens.zero_()
        self.block_table.fill_(-1)
        self.ring_score.fill_(float("nan"))

    def _score(self):
        wl, x = self.wl, self.x
        C.kvs_surrogate(self.dm, x["h"], self.B, x["W"], x["b"], self.score)

    def _decide(self):
        wl, x = self.wl, self.x
        C.kvs_decode_step(self.dm, self.B, wl.w, self.pos, self.score, x["k"], x["v"],
                          self.ring_score, self.ring_k, self.ring_v, wl.tau, wl.page_size,
                          self.k_pages, self.v_pages, self.capacity, self.next_page,
                          self.block_table, self.max_pages, self.seq_lens)

    def stages(self):
        return [("kvs_surrogate", self._score), ("kvs_decode_step", self._decide)]

    def step(self):
        self._score()
        self._decide()


def make_pipeline(wl: Workload, x: dict, **kw):
    if wl.kind in ("kvzip", "kvzip_plus"):
        return KVzipPipeline(wl, x, **kw)
    if wl.kind == "kvzip_plus_chunked":
        return ChunkedKVzipPipeline(wl, x, **kw)
    if wl.kind == "future":
        return FuturePipeline(wl, x, **kw)
    if wl.kind == "kvzap":
        return KVzapPipeline(wl, x, **kw)
    if wl.kind == "kvzap_mlp":
        return KVzapMLPPipeline(wl, x, **kw)
    if wl.kind == "decode":
        return DecodePipeline(wl, x, **kw)
    raise ValueError(wl.kind)
