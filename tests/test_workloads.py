"""Seeded generators: determinism, per-layer independence, shapes and stated recipes."""
import math

import numpy as np
import torch

import oracle as O
from kv_cache_eviction_lse_gb300 import workloads as W


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_layer_subset_matches_full_generation():
    wl = W.WORKLOADS["c2"].scaled(L=3, T=64, n_rep=64, prefix=4, D_h=32)
    full = W.generate(wl)
    sub = W.generate(wl, layers=[2])
    for k in full:
        assert torch.equal(full[k][2:3], sub[k]), k


def test_c1_shapes_and_sinks():
    wl = W.WORKLOADS["c1"]
    x = W.generate(wl)
    assert x["q"].shape == (1, 2, 256, 64) and x["k_ctx"].shape == (1, 1, 256, 64)
    assert x["k_tail"].shape == (1, 1, 264, 64)
    k = x["k_ctx"].float()
    # the two sink keys are 8x larger in norm than the rest on average
    n = k[0, 0].norm(dim=-1)
    assert n[:2].min() > 4 * n[2:].mean()


def test_chunked_carry_repeats_previous_chunk_keys():
    wl = W.WORKLOADS["c3"].scaled(L=1, T=48, n_rep=16, n_chunks=3, D_h=32, prefix=4, carry=8)
    x = W.generate(wl)
    assert [t.shape[2] for t in x["k_tail"]] == [20, 28, 28]
    for c in (1, 2):
        carry = x["k_tail"][c][:, :, 4:12]
        prev_chunk_end = x["k_tail"][c - 1][:, :, -8:]
        assert torch.equal(carry, prev_chunk_end)
        assert torch.equal(x["k_tail"][c][:, :, :4], x["k_tail"][0][:, :, :4])   # shared prefix


def test_kvzap_keep_fraction_statistics():
    # z = h W + b with h ~ N(0,1), W ~ N(0, 1/64^2): given W, z_h ~ N(b_h, ||W_h||^2);
    # threshold -5 keeps about Phi((b_h + 5) / ||W_h||) of the tokens of head h.
    wl = W.WORKLOADS["c5"].scaled(L=2, T=4096, D_h=4096)
    x = W.generate(wl)
    h = O.bf16_bits_to_f64(_bits(x["h"]))
    Wt = O.bf16_bits_to_f64(_bits(x["W"]))
    b = x["b"].double().numpy()
    z = O.linear_surrogate(h, Wt, b)
    mask, keep = O.prune_threshold(z, -5.0, 0)
    for l in range(2):
        for hh in range(8):
            sig = math.sqrt((Wt[l, :, hh] ** 2).sum())
            p = 0.5 * math.erfc(-((b[l, hh] + 5.0) / sig) / math.sqrt(2))
            tol = 5 * math.sqrt(max(p * (1 - p), 1e-4) / 4096) + 1e-3
            assert abs(keep[l, hh] / 4096 - p) < tol


def test_kvzap_mlp_shapes_and_recipe():
    wl = W.WORKLOADS["c6"].scaled(L=2, T=256, D_h=512)
    x = W.generate(wl)
    assert wl.D_mid == 64
    assert x["h"].shape == (2, 256, 512) and x["W1"].shape == (2, 64, 512)
    assert x["b1"].shape == (2, 64) and x["W2"].shape == (2, 8, 64) and x["b2"].shape == (2, 8)
    assert x["W1"].dtype == torch.bfloat16 and x["b1"].dtype == torch.float32
    w1 = x["W1"].double()
    assert abs(w1.std().item() * math.sqrt(512) - 1.0) < 0.05
    assert abs(x["b2"].mean().item() + 4.0) < 1.5
    sub = W.generate(wl, layers=[1])
    for k in x:
        assert torch.equal(x[k][1:2], sub[k]), k


def test_kvzip_plus_recipe():
    """c2: W_O std 1/sqrt(D_h), h std sqrt(D_h), per-channel log-uniform [0.5, 4] scales of
    q, k and v (the channel spreads of the generated rows cover that range)."""
    wl = W.WORKLOADS["c2"]
    x = W.generate(wl, layers=[0])
    w_o, h = x["w_o"].double(), x["h"].double()
    assert abs(w_o.std().item() * math.sqrt(wl.D_h) - 1.0) < 0.02
    assert abs(h.std().item() / math.sqrt(wl.D_h) - 1.0) < 0.02
    for key in ("q", "k_ctx", "v_ctx"):
        ch = x[key].double()[0].std(dim=1)  # [heads][d]: per-channel std over tokens
        assert 0.45 < ch.min().item() < 0.6 and 3.4 < ch.max().item() < 4.4, key
        # log-uniform: the median channel scale sits near sqrt(0.5 * 4)
        assert abs(math.log(ch.median().item()) - math.log(math.sqrt(2.0))) < 0.2, key


def test_future_low_rank_component_is_shared():
    """c4: q, k and v of a KV head share one rank-8 component of unit variance per element
    (q through every head of the group); the other KV heads' components are independent."""
    wl = W.WORKLOADS["c4"].scaled(L=1, T=4096)
    x = W.generate(wl)
    q, k, v = (x[n].double()[0] for n in ("q", "k", "v"))
    assert abs(k.var().item() - 2.0) < 0.1 and abs(v.var().item() - 2.0) < 0.1

    def corr(a, b):
        a, b = a.flatten() - a.mean(), b.flatten() - b.mean()
        return float((a * b).sum() / (a.norm() * b.norm()))

    g = wl.g
    assert abs(corr(k[0], v[0]) - 0.5) < 0.05
    assert abs(corr(q[g - 1], k[0]) - 0.5) < 0.05        # last head of group 0
    assert abs(corr(q[g], k[0])) < 0.05                  # first head of group 1
    assert abs(corr(k[0], k[1])) < 0.05
