"""Plain fp64 CPU oracle for KV-cache importance scoring and pruning.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  The product path (the CUDA
library and its Python binding) never calls it and shares no code with it.

Every function here is the plain definition written out: dense attention rows are
formed explicitly with numpy in float64, then reduced exactly as the pages state.
Sources (page title, then section / equation):

  [KVzap]  "KVzap: Fast, Adaptive, and Faithful KV Cache Pruning" (Jump2Paper review):
           background (KV cache shape), 3.1 KVzip (Eq. 1), 3.2 KVzip+ (Eq. 2, Eq. 3),
           3.3 KVzap (surrogate h_t -> R^H), training setup table (MLP width D_h/8),
           thresholding with a sliding window,
           Algorithm 1 (compress), Appendix B (compute overhead), Table 2.
  [KVpop]  "[Paper review] KVpop -- Key-Value Cache Compression with Predictive Online
           Pruning": 1. Key Terms (future-attention target, transposed-attention pass,
           LSE normaliser), 3. Method (per-head top-k within a fixed budget).
  [KVzip]  KVzip review (seokmin-hardstudy): Background-optional (KV memory formula),
           Methods (teacher-forced repeat), Methods: technical details (chunking).

Where the pages leave a step open the plainest reading is taken; each such reading
is named in the docstring of the function that takes it.

Inputs are float64 arrays (use ``bf16_bits_to_f64`` on raw bf16 bit patterns; the
conversion is exact).  Shapes follow the library's layouts:
  q [L][H_q][n_q][d], keys [L][H_kv][n][d], w_o [L][D_h][H_q*d], h [L][n][D_h].
Query head ``hq`` reads KV head ``hq // g`` with ``g = H_q / H_kv`` (contiguous
GQA groups).

Parity status: every function below is pinned by closed forms, invariants or
brute force in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------- inputs

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64: the bf16 value is
    the top half of an IEEE binary32, so shifting left by 16 gives the float32."""
    b = np.ascontiguousarray(bits).view(np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _group(H_q: int, H_kv: int) -> int:
    if H_kv <= 0 or H_q % H_kv:
        raise ValueError("H_q must be a positive multiple of H_kv")
    return H_q // H_kv


# ----------------------------------------------------------------------------- pass 1

def attention_logits(q_row_block: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """x_ji = q_j . k_i / sqrt(d) for a block of queries against all given keys."""
    d = keys.shape[-1]
    return (q_row_block @ keys.T) / math.sqrt(d)


def causal_visible(n_q: int, n_k: int) -> np.ndarray:
    """Bottom-right causal visibility: query j (0-based among the last n_q positions
    of an n_k-token sequence) sees keys i <= (n_k - n_q) + j.  The scoring queries
    are the last positions of the sequence: the repeated block [KVzap 3.1;
    KVzip Methods, teacher forcing], or the whole sequence when n_q == n_k [KVpop]."""
    off = n_k - n_q
    return np.arange(n_k)[None, :] <= (off + np.arange(n_q))[:, None]


def lse(q: np.ndarray, k_ctx: np.ndarray, k_tail: np.ndarray | None = None) -> np.ndarray:
    """Per-query log-sum-exp normaliser [KVpop 1. Key Terms, LSE normaliser].

    LSE^h_j = ln sum_{i visible to j} exp(q^h_j . k_i / sqrt(d)), natural log, over
    the concatenated keys [context | tail] of the query head's KV head.  Formed as
    m + ln sum exp(x - m) with m the row maximum.  Returns [L][H_q][n_q]."""
    L, H_q, n_q, d = q.shape
    H_kv = k_ctx.shape[1]
    g = _group(H_q, H_kv)
    keys = k_ctx if k_tail is None or k_tail.shape[2] == 0 else np.concatenate([k_ctx, k_tail], 2)
    n_k = keys.shape[2]
    if n_q > n_k:
        raise ValueError("more scoring queries than keys")
    vis = causal_visible(n_q, n_k)
    out = np.empty((L, H_q, n_q))
    for l in range(L):
        for hq in range(H_q):
            x = attention_logits(q[l, hq], keys[l, hq // g])
            x = np.where(vis, x, -np.inf)
            m = x.max(axis=1)
            out[l, hq] = m + np.log(np.exp(x - m[:, None]).sum(axis=1))
    return out


def attention_rows(q: np.ndarray, keys: np.ndarray, lse_rows: np.ndarray) -> np.ndarray:
    """Dense softmax rows a_ji = exp(x_ji - LSE_j) of one query head over the keys
    it sees, zero where not visible.  q [n_q][d], keys [n_k][d], lse_rows [n_q]."""
    n_q, n_k = q.shape[0], keys.shape[0]
    x = attention_logits(q, keys)
    a = np.exp(x - lse_rows[:, None])
    return np.where(causal_visible(n_q, n_k), a, 0.0)


def attention_forward(q, k_ctx, k_tail, v_ctx, v_tail):
    """Attention forward of every query head with its LSE normaliser.  The output of
    head h at query j is o^h_j = sum_i a_ji v_i, the term that W_O then maps into the
    residual stream [KVzap 3.2, Eq. 2]; the LSE is the normaliser an attention kernel
    returns and the transposed pass reuses [KVpop 1. Key Terms].  Keys and values are
    the concatenated [context | tail] of the head's KV head, bottom-right causal.
    q [L][H_q][n_q][d], k_*/v_* [L][H_kv][n][d] (tail may be None or empty).
    Returns (o [L][H_q][n_q][d], lse [L][H_q][n_q])."""
    L, H_q, n_q, d = q.shape
    g = _group(H_q, k_ctx.shape[1])
    has_tail = k_tail is not None and k_tail.shape[2] > 0
    keys = np.concatenate([k_ctx, k_tail], 2) if has_tail else k_ctx
    vals = np.concatenate([v_ctx, v_tail], 2) if has_tail else v_ctx
    lse_ = lse(q, k_ctx, k_tail if has_tail else None)
    o = np.empty((L, H_q, n_q, d))
    for l in range(L):
        for hq in range(H_q):
            a = attention_rows(q[l, hq], keys[l, hq // g], lse_[l, hq])
            o[l, hq] = a @ vals[l, hq // g]
    return o, lse_


# ----------------------------------------------------------------------------- norms

def value_norm(v: np.ndarray, w_o: np.ndarray, H_q: int) -> np.ndarray:
    """||W_O^{(h)} v_i||_2 for every query head h and context token i [KVzap 3.2,
    Eq. 2/Eq. 3: the residual contribution of token i through head h is
    a_ji W_O v_i].  W_O^{(h)} is the d columns h*d..h*d+d-1 of o_proj.weight
    [D_h][H_q*d] (reading: per-head slice of the output projection).  Computed
    directly as a D_h x d mat-vec per token.  Returns [L][H_q][T]."""
    L, H_kv, T, d = v.shape
    g = _group(H_q, H_kv)
    out = np.empty((L, H_q, T))
    for l in range(L):
        for hq in range(H_q):
            Wh = w_o[l][:, hq * d:(hq + 1) * d]          # [D_h][d]
            y = v[l, hq // g] @ Wh.T                      # [T][D_h]
            out[l, hq] = np.sqrt((y * y).sum(axis=1))
    return out


def hidden_norm(h: np.ndarray) -> np.ndarray:
    """||h_j||_2 of the residual-stream input at each query position [KVzap 3.2,
    Eq. 3 denominator].  Reading: plain L2 norm of the given row.  h [L][n][D_h]."""
    return np.sqrt((h * h).sum(axis=-1))


# ----------------------------------------------------------------------------- pass 2

def kvzip_score(q, k_ctx, k_tail, lse_=None, vnorm=None, h=None, log=True):
    """KVzip / KVzip+ importance of each context key [KVzap 3.1 Eq. 1, 3.2 Eq. 3].

    s_i  = max_{j in repeated block} a_ji                         (Eq. 1)
    s+_i = max_{j in repeated block} a_ji ||W_O v_i|| / ||h_j||    (Eq. 3)
    Under GQA the max also runs over every query head of the KV head's group
    [KVzap 3.1, Eq. 1 notes].  a_ji are the dense attention rows of the scoring
    queries over [context | tail]; only context keys i < T are scored.  ``vnorm``
    [L][H_q][T] and ``h`` [L][n_q][D_h] are optional (KVzip when both are None).
    ``lse_`` may be passed (computed by ``lse``); otherwise it is computed here.
    Returns ln s (natural log) when ``log`` is true, else s; shape [L][H_kv][T]."""
    L, H_q, n_q, d = q.shape
    H_kv, T = k_ctx.shape[1], k_ctx.shape[2]
    g = _group(H_q, H_kv)
    if lse_ is None:
        lse_ = lse(q, k_ctx, k_tail)
    keys = k_ctx if k_tail is None or k_tail.shape[2] == 0 else np.concatenate([k_ctx, k_tail], 2)
    hn = hidden_norm(h) if h is not None else None
    out = np.full((L, H_kv, T), -np.inf)
    for l in range(L):
        for hk in range(H_kv):
            best = np.zeros(T)
            for hq in range(hk * g, (hk + 1) * g):
                a = attention_rows(q[l, hq], keys[l, hk], lse_[l, hq])[:, :T]   # [n_q][T]
                if vnorm is not None:
                    a = a * vnorm[l, hq][None, :]
                if hn is not None:
                    a = a / hn[l][:, None]
                best = np.maximum(best, a.max(axis=0))
            out[l, hk] = best
    if log:
        with np.errstate(divide="ignore"):
            return np.log(out)
    return out


def kvzip_score_chunked(q_chunks, k_ctx, tail_chunks, vnorm=None, h_chunks=None, log=True):
    """Chunked reconstruction [KVzip Methods: technical details]: the repeat runs
    chunk by chunk; each chunk's queries see the full context plus that chunk's tail
    (prefix, carried keys of the previous chunk, the chunk itself, causally).  Each
    chunk has its own LSE; the score of a context key is the max over chunks (the
    max of Eq. 1/Eq. 3 taken over all repeated positions)."""
    best = None
    for c in range(len(q_chunks)):
        s = kvzip_score(q_chunks[c], k_ctx, tail_chunks[c], None, vnorm,
                        None if h_chunks is None else h_chunks[c], log=False)
        best = s if best is None else np.maximum(best, s)
    if log:
        with np.errstate(divide="ignore"):
            return np.log(best)
    return best


def future_attention_mass(q, k, w, lse_=None, row_block=1024):
    """KVpop future-attention target [KVpop 1. Key Terms]: the attention mass key i
    receives from queries after it has left the protected window of w tokens,
    f_i = sum_{h in group} sum_{j >= i + w, j < n} a^h_ji, over causal
    self-attention (n_q == n_k, query j sees keys i <= j).  Reading: summed over the
    g query heads of the KV head's group, no normalisation by the query count.
    Rows of A are formed explicitly, ``row_block`` query rows at a time (to bound
    memory).  q [L][H_q][n][d], k [L][H_kv][n][d] -> [L][H_kv][n]."""
    L, H_q, n, d = q.shape
    H_kv = k.shape[1]
    g = _group(H_q, H_kv)
    if lse_ is None:
        lse_ = lse(q, k, None)
    out = np.zeros((L, H_kv, n))
    cols = np.arange(n)
    for l in range(L):
        for hq in range(H_q):
            hk = hq // g
            for j0 in range(0, n, row_block):
                j1 = min(n, j0 + row_block)
                rows = np.arange(j0, j1)
                x = attention_logits(q[l, hq, j0:j1], k[l, hk])
                a = np.exp(x - lse_[l, hq, j0:j1, None])
                band = rows[:, None] >= cols[None, :] + w          # j >= i + w (implies causal)
                out[l, hk] += np.where(band, a, 0.0).sum(axis=0)
    return out


# ----------------------------------------------------------------------------- surrogate

def linear_surrogate(h, W, b):
    """KVzap-Linear [KVzap 3.3]: at each position t the hidden state h_t in R^{D_h}
    maps to H_kv scores, z_t = h_t W + b (a predicted ln s+).  h [L][T][D_h],
    W [L][D_h][H_kv], b [L][H_kv] -> z [L][H_kv][T] (head-major)."""
    L = h.shape[0]
    return np.stack([(h[l] @ W[l] + b[l][None, :]).T for l in range(L)], 0)


def _erf(x):
    try:
        from scipy.special import erf
        return erf(x)
    except ImportError:  # plain per-element fallback
        return np.vectorize(math.erf, otypes=[np.float64])(x)


def gelu(x):
    """GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2, Phi the standard normal CDF.
    Reading: the pages do not name the MLP surrogate's activation; the exact (erf)
    form of GELU is taken."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def mlp_surrogate(h, W1, b1, W2, b2):
    """KVzap-MLP [KVzap 3.3; training setup table]: per layer a two-layer MLP
    D_h -> D_h/8 -> H_kv applied independently at every position,
    z_t = W2 GELU(W1 h_t + b1) + b2 (a predicted ln s+ per KV head).
    Weights in the (out, in) layout of a linear layer: W1 [L][D_mid][D_h],
    b1 [L][D_mid], W2 [L][H_kv][D_mid], b2 [L][H_kv].  h [L][T][D_h] ->
    z [L][H_kv][T] (head-major, like the linear surrogate)."""
    L = h.shape[0]
    out = []
    for l in range(L):
        u = h[l] @ W1[l].T + b1[l][None, :]
        out.append((gelu(u) @ W2[l].T + b2[l][None, :]).T)
    return np.stack(out, 0)


# ----------------------------------------------------------------------------- pruning

def prune_threshold(score, tau, w):
    """KVzap threshold rule with a sliding window [KVzap, thresholding; Algorithm 1]:
    keep token t of head h  <=>  score_{t,h} >= tau  or  t >= T - w.
    Algorithm 1 sets the last ``window`` scores to +inf and keeps ``scores >=
    threshold``; NaN compares false, so a NaN score is dropped unless in the
    window.  score [..][T] -> (mask uint8 [..][T], keep int32 [..])."""
    score = np.asarray(score, dtype=np.float64)
    T = score.shape[-1]
    t = np.arange(T)
    with np.errstate(invalid="ignore"):
        keep = (score >= tau) | (t >= T - w)
    mask = keep.astype(np.uint8)
    return mask, mask.sum(axis=-1).astype(np.int32)


def topk_order(row):
    """Ranking used by per-head top-k: score descending, then position ascending;
    NaN ranks below every number (reading: ties go to the earlier token)."""
    row = np.asarray(row, dtype=np.float64)
    pos = np.arange(row.shape[0])
    nan = np.isnan(row)
    key = np.where(nan, 0.0, -row)
    return np.lexsort((pos, key, nan))


def prune_topk(score, k, w):
    """Per-head top-k within a fixed budget plus the protected recent window
    [KVpop 3. Method: top-k per head; KVzap 3.1: KVzip keeps a fixed ratio; sliding
    window of w recent tokens].  Keep = {t >= T - w} U top-k of the other T - w
    tokens (all of them if k >= T - w).  score [..][T] -> (mask, keep)."""
    score = np.asarray(score, dtype=np.float64)
    shp = score.shape
    T = shp[-1]
    flat = score.reshape(-1, T)
    mask = np.zeros(flat.shape, dtype=np.uint8)
    wn = min(max(w, 0), T)
    for r in range(flat.shape[0]):
        mask[r, T - wn:] = 1
        cand = flat[r, :T - wn]
        kk = min(max(k, 0), T - wn)
        order = topk_order(cand)[:kk]
        mask[r, order] = 1
    mask = mask.reshape(shp)
    return mask, mask.sum(axis=-1).astype(np.int32)


# ----------------------------------------------------------------------------- compaction

def compact_paged(k, v, mask, page_size=16, max_pages=None):
    """Gather of the kept keys/values [KVzap Algorithm 1: keys[indices],
    values[indices]] into a per-head variable-length paged cache (the pages call
    for PagedAttention-like storage because each head keeps a different number of
    tokens [KVzap, trade-offs and limitation 3]).

    Reading of the layout: each (layer, head) gets ceil(keep/page_size) consecutive
    pages, allocated layer-major then head; its first page id is the exclusive prefix
    sum of the page counts before it.  Kept tokens are stored in ascending position;
    unused rows of a head's last page are zero.  ``block_table[l][h][p]`` is the
    absolute page id of the head's p-th page, -1 past the end.  K and V share page ids.

    k, v [L][H][T][d] (any dtype, copied verbatim), mask [L][H][T].
    Returns k_pages, v_pages [P][page_size][d], block_table [L][H][max_pages] int32,
    seq_lens [L][H] int32, total pages P."""
    L, H, T, d = k.shape
    if max_pages is None:
        max_pages = -(-T // page_size)
    keep = mask.astype(bool).sum(axis=-1)
    pages = -(-keep // page_size)
    total = int(pages.sum())
    k_pages = np.zeros((total, page_size, d), dtype=k.dtype)
    v_pages = np.zeros((total, page_size, d), dtype=v.dtype)
    block_table = np.full((L, H, max_pages), -1, dtype=np.int32)
    seq_lens = keep.astype(np.int32)
    first = 0
    for l in range(L):
        for hh in range(H):
            idx = np.nonzero(mask[l, hh])[0]             # ascending positions
            for n, t in enumerate(idx):
                p, r = divmod(n, page_size)
                k_pages[first + p, r] = k[l, hh, t]
                v_pages[first + p, r] = v[l, hh, t]
            for p in range(pages[l, hh]):
                block_table[l, hh, p] = first + p
            first += int(pages[l, hh])
    return k_pages, v_pages, block_table, seq_lens, total


def value_refit(q, k_ctx, v_ctx, mask, lam):
    """Closed-form value refit on the kept keys [KVSculpt summary, 2. Method: with the
    keys fixed, the attention weights they induce are fixed and the values follow in
    closed form by least squares with ridge regularisation; Select+Fit is attention-score
    selection plus this value fit].

    Readings: the training queries are the scoring queries q of the KV head's g query
    heads, stacked (n = g n_q rows); each sees every context key (the repeat block
    follows the whole context).  The target is the attention output over the full
    context, O = softmax(q K^T / sqrt d) V; the kept keys K_S (mask != 0, in position
    order) induce A_S = softmax(q K_S^T / sqrt d) over the kept keys alone; the ridge
    penalty is lam ||V'||^2:
        V' = argmin ||A_S V' - O||_F^2 + lam ||V'||_F^2 = (A_S^T A_S + lam I)^-1 A_S^T O.
    q [L][H_q][n_q][d], k_ctx, v_ctx [L][H_kv][T][d], mask [L][H_kv][T], lam > 0.
    Returns per (l, hk) the refitted values [k][d] (a list of lists) and the pieces
    (A_S, O) of the least-squares problem for checking."""
    L, H_q, n_q, d = q.shape
    H_kv, T = k_ctx.shape[1], k_ctx.shape[2]
    g = _group(H_q, H_kv)
    out, parts = [], []
    for l in range(L):
        row_v, row_p = [], []
        for hk in range(H_kv):
            Q = q[l, hk * g:(hk + 1) * g].reshape(g * n_q, d)
            K, V = k_ctx[l, hk], v_ctx[l, hk]
            idx = np.nonzero(mask[l, hk])[0]
            x = attention_logits(Q, K)
            a_full = np.exp(x - x.max(axis=1, keepdims=True))
            a_full /= a_full.sum(axis=1, keepdims=True)
            O_t = a_full @ V
            xs = x[:, idx]
            a_s = np.exp(xs - xs.max(axis=1, keepdims=True))
            a_s /= a_s.sum(axis=1, keepdims=True)
            M = a_s.T @ a_s + lam * np.eye(len(idx))
            row_v.append(np.linalg.solve(M, a_s.T @ O_t))
            row_p.append((a_s, O_t))
        out.append(row_v)
        parts.append(row_p)
    return out, parts


def decode_prune(score, tau, w):
    """Decode-time pruning at the window boundary [KVzap: the criterion is
    phase-agnostic and works while decoding; KVpop 1. Key Terms: a token's fate is
    decided when it leaves the protected window].  Tokens arrive one per step; when
    token t arrives, token t - w leaves the window and is appended to its row's cache
    iff its score >= tau (a NaN score is dropped).  With w = 0 a token is decided on
    arrival.  Every row (a (layer, KV head, sequence) stream) is independent.
    score [R][T] -> (kept: per row the appended positions in append order,
    window: per row the positions still in the window after the last step)."""
    score = np.asarray(score, dtype=np.float64)
    R, T = score.shape
    kept = [[] for _ in range(R)]
    window = [[] for _ in range(R)]
    for t in range(T):
        for r in range(R):
            window[r].append(t)
            if len(window[r]) > w:
                leaving = window[r].pop(0)
                if score[r, leaving] >= tau:
                    kept[r].append(leaving)
    return kept, window


# ----------------------------------------------------------------------------- formulas

def kv_cache_bytes(L, T, H_kv, d, bytes_per_elem):
    """KV cache size 2 * layers * tokens * kv heads * head dim * bytes
    [KVzip Background-optional; KVzap background, cache shape (2, L, H, T, D)]."""
    return 2 * L * T * H_kv * d * bytes_per_elem


def layer_linear_flops(D_h, H_q, H_kv, D, D_int):
    """Per-token linear-projection cost of a transformer layer [KVzap Appendix B]:
    C = 4 D_h (H_Q D + H D) + 6 D_h D_int."""
    return 4 * D_h * (H_q * D + H_kv * D) + 6 * D_h * D_int


def kvzap_mlp_flops(D_h, H_kv):
    """KVzap-MLP cost per token [KVzap Appendix B]: (D_h / 4)(D_h + H)."""
    return D_h / 4 * (D_h + H_kv)


def kvzap_linear_flops(D_h, H_kv):
    """KVzap-Linear cost per token [KVzap Appendix B]: 2 D_h H."""
    return 2 * D_h * H_kv


def kvzap_linear_params(L, D_h, H_kv, bias=True):
    """Parameters of per-layer linear surrogates D_h -> H_kv [KVzap Table 2]."""
    return L * (D_h * H_kv + (H_kv if bias else 0))


def kvzap_mlp_params(L, D_h, H_kv, bias=True):
    """Parameters of per-layer 2-layer MLP surrogates D_h -> D_h/8 -> H_kv
    [KVzap training setup table]."""
    hid = D_h // 8
    return L * (D_h * hid + hid * H_kv + ((hid + H_kv) if bias else 0))


def compression_factor(ratio_removed):
    """A compression ratio (fraction of KV pairs removed) as a size-reduction factor
    1 / (1 - ratio) [KVzap Table 2: 0.72 is written 3.5x]."""
    return 1.0 / (1.0 - ratio_removed)


def quantile_lower(values, qtl):
    """Lower nearest-rank quantile sorted[floor(qtl * (N - 1))] (reading for the
    threshold set at the 25th percentile of the scores of a layer).  NaN ranks below
    every number, as in the top-k ranking."""
    v = np.asarray(values, dtype=np.float64).ravel()
    nan = np.isnan(v)
    s = np.concatenate([v[nan], np.sort(v[~nan])])
    return float(s[int(math.floor(qtl * (s.size - 1)))])


def prune_quantile(score, qtl, w):
    """Threshold pruning with tau set per layer at a quantile of the layer's scores
    [KVzip Methods: ratio-based threshold; reading: tau_l is the lower nearest-rank
    quantile ``qtl`` of the non-window scores of all KV heads of layer l], then the
    KVzap threshold rule with the window [KVzap, thresholding; Algorithm 1].
    score [L][H_kv][T] -> (mask, keep, tau [L]); with no candidate (w >= T) tau is +inf
    and only the window is kept."""
    score = np.asarray(score, dtype=np.float64)
    L, H, T = score.shape
    wn = min(max(w, 0), T)
    tau = np.full(L, np.inf)
    for l in range(L):
        if T - wn > 0:
            tau[l] = quantile_lower(score[l, :, : T - wn], qtl)
    masks, keeps = zip(*[prune_threshold(score[l], tau[l], w) for l in range(L)])
    return np.stack(masks), np.stack(keeps), tau
