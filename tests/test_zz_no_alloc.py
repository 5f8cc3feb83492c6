"""kvs_vnorm_noalloc: the value norm for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns every device allocation, or a serving
loop that forbids allocation after warm-up) cannot provide kvs_vnorm's workspace; this
entry point uses a scratch array built into the library instead.  The test calls it
through the C ABI twice in a row, with different shapes, and checks each result against
kvs_vnorm (caller workspace) within the value-norm tolerance of the other GPU tests.
It runs last (file name) so that a stop-at-first-failure run has run everything else;
it must also pass on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import assert_close_rel, need_gpu

pytestmark = pytest.mark.gpu

VNORM_RTOL = 1e-4


@pytest.fixture(scope="module")
def C():
    need_gpu()
    from kv_cache_eviction_lse_gb300 import build
    build.build()
    from kv_cache_eviction_lse_gb300 import capi
    return capi


def _inputs(L, Hkv, Hq, d, T, Dh, seed):
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(L, Hkv, T, d, generator=g).to(torch.bfloat16).cuda()
    w_o = (torch.randn(L, Dh, Hq * d, generator=g) / Dh ** 0.5).to(torch.bfloat16).cuda()
    return v, w_o


def test_vnorm_noalloc_matches_workspace_version_twice(C):
    shapes = [(3, 2, 6, 128, 300, 192, 1), (2, 4, 32, 128, 1000, 512, 2)]
    _compare(C, shapes)


def test_vnorm_noalloc_at_the_capacity_limit_and_small_shapes(C):
    """One layer that fills the built-in scratch exactly (H_q d d 4 bytes = 8 MiB at
    H_q = 128, d = 128), a head dimension of 64, and a single layer."""
    shapes = [(1, 8, 128, 128, 260, 256, 3), (2, 2, 8, 64, 777, 320, 4), (1, 1, 4, 64, 129, 64, 5)]
    assert 128 * 128 * 128 * 4 == 8 << 20  # the documented size of the built-in scratch
    _compare(C, shapes)


def test_vnorm_noalloc_empty_context_writes_nothing(C):
    """T = 0: the call succeeds and leaves the output as it was."""
    dm = C.dims(2, 8, 2, 128, 256)
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    out = torch.full((64,), 7.0, device="cuda")
    C.kvs_vnorm_noalloc(dm, t, 0, t, out)
    torch.cuda.synchronize()
    assert (out.cpu() == 7.0).all()


def _compare(C, shapes):
    for L, Hkv, Hq, d, T, Dh, seed in shapes:
        v, w_o = _inputs(L, Hkv, Hq, d, T, Dh, seed)
        dm = C.dims(L, Hq, Hkv, d, Dh)
        ws = torch.empty(C.kvs_vnorm_workspace_size(dm), dtype=torch.uint8, device="cuda")
        want = torch.empty(L, Hq, T, device="cuda")
        C.kvs_vnorm(dm, v, T, w_o, want, ws, ws.numel())
        got = torch.full((L, Hq, T), float("nan"), device="cuda")
        C.kvs_vnorm_noalloc(dm, v, T, w_o, got)
        torch.cuda.synchronize()
        assert_close_rel(got.cpu().numpy(), want.cpu().numpy(), VNORM_RTOL, "vnorm no-alloc")
        assert np.isfinite(got.cpu().numpy()).all()


def test_vnorm_noalloc_rejects_oversized_layers(C):
    dm = C.dims(1, 256, 8, 128, 512)  # 256 * 128 * 128 * 4 B = 16 MiB per layer
    t = torch.empty(16, device="cuda")
    with pytest.raises(C.KvsError) as ei:
        C.kvs_vnorm_noalloc(dm, t, 4, t, t)
    assert ei.value.status == C.KVS_ERR_CAPACITY
    assert "built-in scratch" in str(ei.value)
