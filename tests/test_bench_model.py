"""The benchmark's algorithmic work model (the numerator of every roofline figure) against
independent counts: visible query-key pairs counted element by element from the oracle's
causal mask and band rule on small copies of the workloads, and the pages' per-token
surrogate costs [KVzap Appendix B] as the oracle states them.  CPU only."""
import types

import numpy as np
import pytest

import bench
import oracle as O
from kv_cache_eviction_lse_gb300 import workloads as W


def _p(wl, **kw):
    return types.SimpleNamespace(L=wl.L, **kw)


@pytest.mark.parametrize("name,scale", [
    ("c1", {}),
    ("c2", dict(L=2, T=300, n_rep=200, prefix=16)),
    ("c3", dict(L=1, H_kv=2, H_q=4, T=500, n_rep=128, n_chunks=3, prefix=16, carry=8)),
])
def test_scoring_pairs_match_the_causal_mask(name, scale):
    wl = W.WORKLOADS[name].scaled(**scale)
    work = bench.algorithmic_work(wl, _p(wl))
    chunks = wl.n_chunks if wl.kind == "kvzip_plus_chunked" else 1
    visible = sum(int(O.causal_visible(wl.n_rep, wl.T + wl.tail_len(c)).sum())
                  for c in range(chunks))
    assert work["kvs_lse"] == ("tensor", 2 * wl.d * wl.L * wl.H_q * visible, "flop")
    # pass 2 scores every context key against every scoring query of every chunk
    assert work["kvs_score_max"][1] == 2 * wl.d * wl.L * wl.H_q * wl.n_rep * wl.T * chunks
    if wl.kind != "kvzip":
        # the Gram form: G = W_h^T W_h (2 D_h d^2) and v^T G v per key (2 d^2)
        assert work["kvs_vnorm"][1] == wl.L * wl.H_q * (2 * wl.D_h * wl.d ** 2
                                                         + 2 * wl.T * wl.d ** 2)


@pytest.mark.parametrize("T,w", [(300, 0), (300, 17), (256, 128), (64, 64), (64, 100)])
def test_future_mass_pairs_match_the_band(T, w):
    wl = W.WORKLOADS["c4"].scaled(L=1, H_kv=2, H_q=4, T=T, w=w)
    work = bench.algorithmic_work(wl, _p(wl))
    j = np.arange(T)[:, None]   # query (row) position
    i = np.arange(T)[None, :]   # key position
    causal = int((i <= j).sum())
    band = int((j >= i + w).sum())
    assert work["kvs_lse"][1] == 2 * wl.d * wl.H_q * causal
    assert work["kvs_attn_fwd"][1] == 4 * wl.d * wl.H_q * causal
    assert work["kvs_score_future_sum"][1] == 2 * wl.d * wl.H_q * band


def test_surrogate_costs_follow_appendix_b():
    wl = W.WORKLOADS["c6"].scaled(L=2, T=1000)
    work = bench.algorithmic_work(wl, _p(wl))
    assert work["kvs_surrogate_mlp"][1] == pytest.approx(
        wl.L * wl.T * O.kvzap_mlp_flops(wl.D_h, wl.H_kv))
    wl = W.WORKLOADS["c5"].scaled(L=2, T=1000)
    work = bench.algorithmic_work(wl, _p(wl))
    # bytes: the hidden rows and the weights are read once, scores (fp32) and mask written
    assert work["kvs_surrogate"] == ("hbm", wl.L * wl.T * wl.D_h * 2 + wl.L * wl.D_h * wl.H_kv * 2
                                     + wl.L * wl.H_kv * wl.T * 5, "byte")


def test_units_are_context_tokens_per_layer():
    wl = W.WORKLOADS["c2"]
    assert bench.units_per_step(wl, _p(wl)) == wl.T * wl.L
    assert bench.whole_job_value(1000, 4, 2.0) == pytest.approx(4 * 1000 / 2e-3)


def test_reference_arm_reports_what_it_timed():
    """The reference arm's steps x ms_per_step is time it really spent (it fits inside
    the wall time of the call), and its config is the one the GPU arm prints."""
    import time
    args = types.SimpleNamespace(workload="c1", layers=None, steps=2, warmup=3,
                                 attn_forward=False, refit=False)
    t0 = time.perf_counter()
    res = bench.run_reference(args, 0, 1)
    wall_ms = 1e3 * (time.perf_counter() - t0)
    assert res["steps"] == 2 and res["warmup"] == 3
    assert res["steps"] * res["ms_per_step"] <= wall_ms
    assert res["extrapolation"]["measured_ms_per_step"] == res["ms_per_step"]
    wl = W.WORKLOADS["c1"]
    ex = res["extrapolation"]
    assert res["value"] == pytest.approx(ex["tokens_per_layer"] / (ex["layer_equivalent_ms"] / 1e3),
                                         rel=1e-3)
    assert res["config"] == bench.run_config(wl, args, 1, wl.L)
    assert res["cpu_baseline"]["value"] == res["value"]
