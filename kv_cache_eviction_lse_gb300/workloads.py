"""Seeded synthetic inputs for the KV-cache scoring and pruning path.

This module only draws random numbers and lays them out in the tensor layouts that
the library (and its CPU checker) take.  It holds none of the method's arithmetic:
no attention, no norms, no scoring, no selection.

Five workloads are defined, shaped like the models the pages evaluate:

  c1  tiny KVzip max-score (1 layer, 1 KV head, 2 query heads, d=64, two sink keys)
  c2  Qwen2.5-1.5B-shaped KVzip+ scoring (28 layers, 2 KV / 12 query heads, d=128)
  c3  Qwen3-8B-shaped chunked KVzip+ scoring (36 layers, 8 / 32 heads, T=32768)
  c4  Qwen3-4B-shaped future-attention target (36 layers, 8 / 32 heads, T=16384)
  c5  Llama-3-8B-shaped KVzap linear-surrogate pruning (32 layers, 8 KV heads, T=131072)
  c6  Qwen3-8B-shaped KVzap MLP-surrogate pruning (36 layers, 8 KV heads, 4096 -> 512 -> 8)
  c7  Llama-3-8B-shaped decode-time pruning: 64 sequences, one token per step, KVzap-Linear
      score of the arriving token, window w=128 ring, threshold at the window boundary

Every layer is drawn from its own generator seeded with
``20261202 + 1000 * workload_index + layer``, so any subset of layers can be
regenerated without drawing the others.  Values are drawn in fp32 and rounded to
bf16 with round-to-nearest-even (``Tensor.to(torch.bfloat16)``).

Layouts (row-major, innermost last):
  q        [L][H_q][n_q][d]        bf16   scoring queries
  k_ctx    [L][H_kv][T][d]         bf16   context keys being scored
  v_ctx    [L][H_kv][T][d]         bf16
  k_tail   [L][H_kv][n_tail][d]    bf16   keys after the context (prefix, carry, block)
  w_o      [L][D_h][H_q*d]         bf16   attention output projection (o_proj.weight)
  h        [L][n_q][D_h]           bf16   residual-stream input at the scoring queries
  W        [L][D_h][H_kv]          bf16   linear surrogate weight
  b        [L][H_kv]               fp32   linear surrogate bias
  W1       [L][D_h/8][D_h]         bf16   MLP surrogate first layer (out, in)
  b1       [L][D_h/8]              fp32
  W2       [L][H_kv][D_h/8]        bf16   MLP surrogate second layer (out, in)
  b2       [L][H_kv]               fp32
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    """Shapes and distribution parameters of one synthetic workload."""

    name: str
    index: int
    title: str
    L: int
    H_kv: int
    H_q: int
    d: int
    D_h: int
    T: int                    # context keys scored per (layer, KV head)
    kind: str                 # kvzip | kvzip_plus | kvzip_plus_chunked | future | kvzap | kvzap_mlp | decode
    batch: int = 0            # decode: sequences advanced together, one token each per step
    prefix: int = 0           # repeat-prompt tokens between context and repeated block
    n_rep: int = 0            # scoring queries per call (repeated block, or one chunk)
    n_chunks: int = 1
    carry: int = 0            # keys of the previous chunk repeated before each chunk
    w: int = 0                # protected recent window
    keep_ratios: tuple = ()   # per-head top-k budgets as a fraction of T
    tau: float | None = None  # fixed threshold (log-score space)
    tau_quantile: float | None = None  # threshold set at this quantile of the scores
    page_size: int = 16
    sinks: int = 0            # leading context keys scaled by sink_scale
    sink_scale: float = 8.0
    channel_scales: bool = False
    low_rank: int = 0

    @property
    def g(self) -> int:
        return self.H_q // self.H_kv

    @property
    def D_mid(self) -> int:
        """Hidden width of the MLP surrogate: D_h / 8."""
        return self.D_h // 8

    def seed(self, layer: int) -> int:
        return BASE_SEED + 1000 * self.index + layer

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (smaller test sizes)."""
        return dataclasses.replace(self, **kw)

    def tail_len(self, chunk: int = 0) -> int:
        """Keys after the context that the scoring queries of ``chunk`` see."""
        if self.kind == "kvzip_plus_chunked":
            return self.prefix + (self.carry if chunk > 0 else 0) + self.n_rep
        if self.kind in ("kvzip", "kvzip_plus"):
            return self.prefix + self.n_rep
        return 0

    def topk_budget(self, ratio: float) -> int:
        """k = floor(r*T + 0.5) tokens kept by per-head top-k besides the window."""
        return int(math.floor(ratio * self.T + 0.5))


WORKLOADS = {
    "c1": Workload(
        name="c1", index=1,
        title="tiny KVzip max-score, 1 layer, 1 KV head, 2 query heads, d=64, "
              "ctx 256 + prefix 8 + repeated 256, top-25% + w=16",
        L=1, H_kv=1, H_q=2, d=64, D_h=0, T=256, kind="kvzip",
        prefix=8, n_rep=256, w=16, keep_ratios=(0.25,), sinks=2),
    "c2": Workload(
        name="c2", index=2,
        title="Qwen2.5-1.5B-shaped KVzip+ scoring, 28 layers, 2 KV / 12 query heads, "
              "d=128, hidden 1536, ctx 2048 + prefix 16 + repeated 2048",
        L=28, H_kv=2, H_q=12, d=128, D_h=1536, T=2048, kind="kvzip_plus",
        prefix=16, n_rep=2048, w=0, keep_ratios=(0.3, 0.5, 0.7), channel_scales=True),
    "c3": Workload(
        name="c3", index=3,
        title="Qwen3-8B-shaped chunked KVzip+ scoring, 36 layers, 8 KV / 32 query heads, "
              "d=128, hidden 4096, ctx 32768 in 16 chunks of 2048 (prefix 16, carry 8), "
              "tau = 25th percentile, w=128",
        L=36, H_kv=8, H_q=32, d=128, D_h=4096, T=32768, kind="kvzip_plus_chunked",
        prefix=16, n_rep=2048, n_chunks=16, carry=8, w=128, tau_quantile=0.25,
        channel_scales=True),
    "c4": Workload(
        name="c4", index=4,
        title="Qwen3-4B-shaped future-attention target, 36 layers, 8 KV / 32 query heads, "
              "d=128, causal T=16384 + rank-8 shared component, w=128, top-25%/12.5%",
        L=36, H_kv=8, H_q=32, d=128, D_h=0, T=16384, kind="future",
        w=128, keep_ratios=(0.25, 0.125), low_rank=8),
    "c5": Workload(
        name="c5", index=5,
        title="Llama-3-8B-shaped KVzap linear-surrogate pruning, 32 layers, 8 KV heads, "
              "d=128, hidden 4096, T=131072, tau=-5, w=128",
        L=32, H_kv=8, H_q=32, d=128, D_h=4096, T=131072, kind="kvzap",
        w=128, tau=-5.0),
    "c6": Workload(
        name="c6", index=6,
        title="Qwen3-8B-shaped KVzap MLP-surrogate pruning, 36 layers, 8 KV heads, "
              "d=128, hidden 4096 -> 512 -> 8 (GELU), T=131072, tau=-4, w=128",
        L=36, H_kv=8, H_q=32, d=128, D_h=4096, T=131072, kind="kvzap_mlp",
        w=128, tau=-4.0),
    "c7": Workload(
        name="c7", index=7,
        title="Llama-3-8B-shaped decode-time pruning, 32 layers, 8 KV heads, d=128, "
              "hidden 4096, 64 sequences x 1 token per step, KVzap-Linear score, w=128 "
              "ring, tau=-5 at the window boundary, pages of 16",
        L=32, H_kv=8, H_q=32, d=128, D_h=4096, T=1, kind="decode", batch=64,
        w=128, tau=-5.0),
}


# --------------------------------------------------------------------------- helpers

def _gen(wl: Workload, layer: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed(layer))
    return g


def _randn(gen, shape, device, std=1.0, mean=0.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _log_uniform(gen, shape, device, lo=0.5, hi=4.0):
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    return torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _layers(wl: Workload, layers):
    return list(range(wl.L)) if layers is None else list(layers)


# --------------------------------------------------------------------------- per kind

def _kvzip_layer(wl: Workload, layer: int, device):
    """One layer of the (unchunked) KVzip / KVzip+ workloads (c1, c2)."""
    gen = _gen(wl, layer, device)
    d, Hq, Hkv = wl.d, wl.H_q, wl.H_kv
    if wl.channel_scales:
        sq = _log_uniform(gen, (Hq, 1, d), device)
        sk = _log_uniform(gen, (Hkv, 1, d), device)
        sv = _log_uniform(gen, (Hkv, 1, d), device)
    k_ctx = _randn(gen, (Hkv, wl.T, d), device)
    v_ctx = _randn(gen, (Hkv, wl.T, d), device)
    k_tail = _randn(gen, (Hkv, wl.prefix + wl.n_rep, d), device)
    q = _randn(gen, (Hq, wl.n_rep, d), device)
    if wl.channel_scales:
        k_ctx.mul_(sk); v_ctx.mul_(sv); k_tail.mul_(sk); q.mul_(sq)
    if wl.sinks:
        k_ctx[:, : wl.sinks, :].mul_(wl.sink_scale)
    out = dict(q=_bf16(q), k_ctx=_bf16(k_ctx), v_ctx=_bf16(v_ctx), k_tail=_bf16(k_tail))
    if wl.kind == "kvzip_plus":
        out["w_o"] = _bf16(_randn(gen, (wl.D_h, Hq * d), device, std=1.0 / math.sqrt(wl.D_h)))
        out["h"] = _bf16(_randn(gen, (wl.n_rep, wl.D_h), device, std=math.sqrt(wl.D_h)))
    return out


def _stack(parts, key):
    return torch.stack([p[key] for p in parts], 0).contiguous()


def generate(wl: Workload, layers=None, device="cpu") -> dict:
    """Draw the inputs of ``wl`` for the given layers (all by default).

    Returns a dict of tensors on ``device``.  For the chunked workload the
    per-chunk tensors are lists indexed by chunk: ``q``, ``k_tail`` and ``h``.
    """
    layers = _layers(wl, layers)
    if wl.kind in ("kvzip", "kvzip_plus"):
        parts = [_kvzip_layer(wl, l, device) for l in layers]
        return {k: _stack(parts, k) for k in parts[0]}
    if wl.kind == "kvzip_plus_chunked":
        return _generate_chunked(wl, layers, device)
    if wl.kind == "future":
        return _generate_future(wl, layers, device)
    if wl.kind == "kvzap":
        return _generate_kvzap(wl, layers, device)
    if wl.kind == "kvzap_mlp":
        return _generate_kvzap_mlp(wl, layers, device)
    if wl.kind == "decode":
        return _generate_decode(wl, layers, device)
    raise ValueError(wl.kind)


def _generate_chunked(wl: Workload, layers, device):
    """c3: context, one repeat prefix per layer, and a repeated block of T tokens
    processed in ``n_chunks`` chunks of ``n_rep``.  Chunk c>0 is preceded by the
    last ``carry`` keys of chunk c-1 (the same vectors)."""
    nL, d, Hq, Hkv, T = len(layers), wl.d, wl.H_q, wl.H_kv, wl.T
    assert wl.n_chunks * wl.n_rep == T
    bf = torch.bfloat16
    k_ctx = torch.empty((nL, Hkv, T, d), dtype=bf, device=device)
    v_ctx = torch.empty_like(k_ctx)
    w_o = torch.empty((nL, wl.D_h, Hq * d), dtype=bf, device=device)
    q = [torch.empty((nL, Hq, wl.n_rep, d), dtype=bf, device=device) for _ in range(wl.n_chunks)]
    h = [torch.empty((nL, wl.n_rep, wl.D_h), dtype=bf, device=device) for _ in range(wl.n_chunks)]
    k_tail = [torch.empty((nL, Hkv, wl.tail_len(c), d), dtype=bf, device=device)
              for c in range(wl.n_chunks)]
    for i, l in enumerate(layers):
        gen = _gen(wl, l, device)
        sq = _log_uniform(gen, (Hq, 1, d), device)
        sk = _log_uniform(gen, (Hkv, 1, d), device)
        sv = _log_uniform(gen, (Hkv, 1, d), device)
        k_ctx[i] = _bf16(_randn(gen, (Hkv, T, d), device).mul_(sk))
        v_ctx[i] = _bf16(_randn(gen, (Hkv, T, d), device).mul_(sv))
        w_o[i] = _bf16(_randn(gen, (wl.D_h, Hq * d), device, std=1.0 / math.sqrt(wl.D_h)))
        prefix = _bf16(_randn(gen, (Hkv, wl.prefix, d), device).mul_(sk))
        rep_k = _bf16(_randn(gen, (Hkv, T, d), device).mul_(sk))
        rep_q = _bf16(_randn(gen, (Hq, T, d), device).mul_(sq))
        rep_h = _bf16(_randn(gen, (T, wl.D_h), device, std=math.sqrt(wl.D_h)))
        for c in range(wl.n_chunks):
            s = c * wl.n_rep
            q[c][i] = rep_q[:, s:s + wl.n_rep]
            h[c][i] = rep_h[s:s + wl.n_rep]
            pieces = [prefix]
            if c > 0 and wl.carry:
                pieces.append(rep_k[:, s - wl.carry:s])
            pieces.append(rep_k[:, s:s + wl.n_rep])
            k_tail[c][i] = torch.cat(pieces, 1)
        del rep_k, rep_q, rep_h
    return dict(k_ctx=k_ctx, v_ctx=v_ctx, w_o=w_o, q=q, h=h, k_tail=k_tail)


def _generate_future(wl: Workload, layers, device):
    """c4: causal self-attention inputs, N(0,1) plus a rank-r component shared by
    q (all heads of the group), k and v of each KV head."""
    nL, d, Hq, Hkv, T, r = len(layers), wl.d, wl.H_q, wl.H_kv, wl.T, wl.low_rank
    bf = torch.bfloat16
    q = torch.empty((nL, Hq, T, d), dtype=bf, device=device)
    k = torch.empty((nL, Hkv, T, d), dtype=bf, device=device)
    v = torch.empty_like(k)
    for i, l in enumerate(layers):
        gen = _gen(wl, l, device)
        low = None
        if r:
            basis = _randn(gen, (Hkv, r, d), device, std=1.0 / math.sqrt(r))
            coef = _randn(gen, (Hkv, T, r), device)
            low = torch.bmm(coef, basis)                      # [Hkv][T][d]
        kk = _randn(gen, (Hkv, T, d), device)
        vv = _randn(gen, (Hkv, T, d), device)
        qq = _randn(gen, (Hq, T, d), device)
        if low is not None:
            kk.add_(low); vv.add_(low)
            qq.add_(low.repeat_interleave(wl.g, 0))
        k[i] = _bf16(kk); v[i] = _bf16(vv); q[i] = _bf16(qq)
    return dict(q=q, k=k, v=v)


def _generate_kvzap(wl: Workload, layers, device):
    """c5: hidden states, linear surrogate weights and the K/V to compact."""
    nL, d, Hkv, T, Dh = len(layers), wl.d, wl.H_kv, wl.T, wl.D_h
    bf = torch.bfloat16
    h = torch.empty((nL, T, Dh), dtype=bf, device=device)
    W = torch.empty((nL, Dh, Hkv), dtype=bf, device=device)
    b = torch.empty((nL, Hkv), dtype=torch.float32, device=device)
    k = torch.empty((nL, Hkv, T, d), dtype=bf, device=device)
    v = torch.empty_like(k)
    for i, l in enumerate(layers):
        gen = _gen(wl, l, device)
        W[i] = _bf16(_randn(gen, (Dh, Hkv), device, std=1.0 / 64.0))
        b[i] = _randn(gen, (Hkv,), device, mean=-4.0)
        h[i] = _bf16(_randn(gen, (T, Dh), device))
        k[i] = _bf16(_randn(gen, (Hkv, T, d), device))
        v[i] = _bf16(_randn(gen, (Hkv, T, d), device))
    return dict(h=h, W=W, b=b, k=k, v=v)


def _generate_kvzap_mlp(wl: Workload, layers, device):
    """c6: hidden states, MLP surrogate weights (W1 std 1/sqrt(D_h), b1 std 1/2,
    W2 std 1/sqrt(D_h/8), b2 ~ N(-4, 1)) and the K/V to compact."""
    nL, d, Hkv, T, Dh, Dm = len(layers), wl.d, wl.H_kv, wl.T, wl.D_h, wl.D_mid
    bf = torch.bfloat16
    h = torch.empty((nL, T, Dh), dtype=bf, device=device)
    W1 = torch.empty((nL, Dm, Dh), dtype=bf, device=device)
    b1 = torch.empty((nL, Dm), dtype=torch.float32, device=device)
    W2 = torch.empty((nL, Hkv, Dm), dtype=bf, device=device)
    b2 = torch.empty((nL, Hkv), dtype=torch.float32, device=device)
    k = torch.empty((nL, Hkv, T, d), dtype=bf, device=device)
    v = torch.empty_like(k)
    for i, l in enumerate(layers):
        gen = _gen(wl, l, device)
        W1[i] = _bf16(_randn(gen, (Dm, Dh), device, std=1.0 / math.sqrt(Dh)))
        b1[i] = _randn(gen, (Dm,), device, std=0.5)
        W2[i] = _bf16(_randn(gen, (Hkv, Dm), device, std=1.0 / math.sqrt(Dm)))
        b2[i] = _randn(gen, (Hkv,), device, mean=-4.0)
        h[i] = _bf16(_randn(gen, (T, Dh), device))
        k[i] = _bf16(_randn(gen, (Hkv, T, d), device))
        v[i] = _bf16(_randn(gen, (Hkv, T, d), device))
    return dict(h=h, W1=W1, b1=b1, W2=W2, b2=b2, k=k, v=v)


def _generate_decode(wl: Workload, layers, device):
    """c7: the linear surrogate of c5 and the inputs of one decode step: the arriving
    token's hidden state per sequence and its K/V per (layer, KV head, sequence)."""
    nL, d, Hkv, Dh, B = len(layers), wl.d, wl.H_kv, wl.D_h, wl.batch
    bf = torch.bfloat16
    h = torch.empty((nL, B, Dh), dtype=bf, device=device)
    W = torch.empty((nL, Dh, Hkv), dtype=bf, device=device)
    b = torch.empty((nL, Hkv), dtype=torch.float32, device=device)
    k = torch.empty((nL, Hkv, B, d), dtype=bf, device=device)
    v = torch.empty_like(k)
    for i, l in enumerate(layers):
        gen = _gen(wl, l, device)
        W[i] = _bf16(_randn(gen, (Dh, Hkv), device, std=1.0 / 64.0))
        b[i] = _randn(gen, (Hkv,), device, mean=-4.0)
        h[i] = _bf16(_randn(gen, (B, Dh), device))
        k[i] = _bf16(_randn(gen, (Hkv, B, d), device))
        v[i] = _bf16(_randn(gen, (Hkv, B, d), device))
    return dict(h=h, W=W, b=b, k=k, v=v)


def random_kv_inputs(L, H_kv, H_q, d, T, n_tail, n_q, seed, device="cpu", scale=1.0,
                     D_h=0):
    """Generic seeded inputs of arbitrary (ragged) shape for edge-case tests."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = dict(
        q=_bf16(_randn(gen, (L, H_q, n_q, d), device, std=scale)),
        k_ctx=_bf16(_randn(gen, (L, H_kv, T, d), device, std=scale)),
        v_ctx=_bf16(_randn(gen, (L, H_kv, T, d), device)),
        k_tail=_bf16(_randn(gen, (L, H_kv, n_tail, d), device, std=scale)),
    )
    if D_h:
        out["w_o"] = _bf16(_randn(gen, (L, D_h, H_q * d), device, std=1.0 / math.sqrt(D_h)))
        out["h"] = _bf16(_randn(gen, (L, n_q, D_h), device, std=math.sqrt(D_h)))
    return out
