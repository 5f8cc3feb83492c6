"""The C-ABI library builds, loads and exports every symbol include/kvs.h declares; its
host-side validation rejects bad arguments with the documented status codes.  No GPU:
every call here fails validation, or is an empty call, before anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvs.h")


@pytest.fixture(scope="module")
def capi():
    from kv_cache_eviction_lse_gb300 import build
    build.build()
    from kv_cache_eviction_lse_gb300 import capi as C
    return C


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvs_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(capi):
    syms = declared_symbols()
    assert len(syms) >= 14
    lib = ctypes.CDLL(capi.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(capi.EXPORTED)


def test_validation_of_multi_budget_and_quantile_calls(capi):
    """kvs_prune_topk_multi, kvs_prune_quantile and kvs_compact_paged_multi reject bad
    arguments before anything is enqueued, and their empty calls succeed."""
    C = capi
    lib = C._lib
    by = ctypes.byref
    dm = C.dims(2, 4, 2, 128, 0)
    fake = 1 << 20
    ks = (ctypes.c_int32 * 9)(*([5] * 9))
    # top-k of several budgets: count outside 1..8, a negative budget, null k, misaligned
    assert lib.kvs_prune_topk_multi(by(dm), fake, 10, 0, ks, 0, fake, fake, None) == C.KVS_ERR_UNSUPPORTED
    assert lib.kvs_prune_topk_multi(by(dm), fake, 10, 9, ks, 0, fake, fake, None) == C.KVS_ERR_UNSUPPORTED
    neg = (ctypes.c_int32 * 2)(3, -1)
    assert lib.kvs_prune_topk_multi(by(dm), fake, 10, 2, neg, 0, fake, fake, None) == C.KVS_ERR_ARG
    assert lib.kvs_prune_topk_multi(by(dm), fake, 10, 2, None, 0, fake, fake, None) == C.KVS_ERR_ARG
    assert lib.kvs_prune_topk_multi(by(dm), fake, 10, 2, ks, -1, fake, fake, None) == C.KVS_ERR_ARG
    assert lib.kvs_prune_topk_multi(by(dm), fake + 4, 10, 2, ks, 0, fake, fake, None) == C.KVS_ERR_ALIGN
    assert lib.kvs_prune_topk_multi(by(dm), fake, 10, 2, ks, 0, None, fake, None) == C.KVS_ERR_ARG
    # quantile threshold: q outside [0, 1] (NaN included), null tau, negative window
    f = ctypes.c_float
    for q in (-0.5, 1.5, float("nan")):
        assert lib.kvs_prune_quantile(by(dm), fake, 10, f(q), 0, fake, fake, fake, None) == C.KVS_ERR_ARG
    assert lib.kvs_prune_quantile(by(dm), fake, 10, f(0.25), 0, None, fake, fake, None) == C.KVS_ERR_ARG
    assert lib.kvs_prune_quantile(by(dm), fake, 10, f(0.25), -3, fake, fake, fake, None) == C.KVS_ERR_ARG
    # compaction of several masks: no mask, workspace of one mask only, bad page size
    need1 = lib.kvs_compact_workspace_size(by(dm), 100)
    need3 = lib.kvs_compact_multi_workspace_size(by(dm), 100, 3)
    assert need3 > need1 and lib.kvs_compact_multi_workspace_size(by(dm), 100, 0) == 0
    args = lambda n, ws: (by(dm), fake, fake, 100, n, fake, 16, fake, fake, 1000, fake, 7, fake,
                          fake, fake, ws, None)
    assert lib.kvs_compact_paged_multi(*args(0, need3)) == C.KVS_ERR_ARG
    assert lib.kvs_compact_paged_multi(*args(3, need1)) == C.KVS_ERR_CAPACITY
    assert "workspace" in C.kvs_last_error()
    st = lib.kvs_compact_paged_multi(by(dm), fake, fake, 100, 3, fake, 5000, fake, fake, 1000,
                                     fake, 7, fake, fake, fake, need3, None)
    assert st == C.KVS_ERR_UNSUPPORTED


def test_version_string(capi):
    assert "sm_103a" in capi.kvs_version()


def _raw(capi):
    return ctypes.CDLL(capi.LIB_PATH)


def test_validation_codes(capi):
    C = capi
    lib = C._lib
    dm = C.dims(1, 4, 2, 128, 0)
    fake = 1 << 20  # never dereferenced: validation fails first
    # n_q larger than keys
    st = lib.kvs_lse(ctypes.byref(dm), fake, 100, fake, 10, fake, 5, fake, None)
    assert st == C.KVS_ERR_SHAPE and "exceeds" in C.kvs_last_error()
    # unsupported head dim
    bad = C.dims(1, 4, 2, 96, 0)
    st = lib.kvs_lse(ctypes.byref(bad), fake, 4, fake, 10, None, 0, fake, None)
    assert st == C.KVS_ERR_UNSUPPORTED
    # H_q not a multiple of H_kv
    bad = C.dims(1, 5, 2, 128, 0)
    assert lib.kvs_lse(ctypes.byref(bad), fake, 4, fake, 10, None, 0, fake, None) == C.KVS_ERR_SHAPE
    # null output
    assert lib.kvs_lse(ctypes.byref(dm), fake, 4, fake, 10, None, 0, None, None) == C.KVS_ERR_ARG
    # misaligned pointer
    assert lib.kvs_lse(ctypes.byref(dm), fake + 2, 4, fake, 10, None, 0, fake, None) == C.KVS_ERR_ALIGN
    # null dims
    assert lib.kvs_lse(None, fake, 4, fake, 10, None, 0, fake, None) == C.KVS_ERR_ARG
    # bad prune mode / negative k
    assert lib.kvs_prune_mask(ctypes.byref(dm), fake, 10, 7, 0.0, 1, 0, fake, fake, None) == C.KVS_ERR_ARG
    assert lib.kvs_prune_mask(ctypes.byref(dm), fake, 10, 1, 0.0, -1, 0, fake, fake, None) == C.KVS_ERR_ARG
    # workspace too small
    dmh = C.dims(1, 4, 2, 128, 64)
    need = lib.kvs_vnorm_workspace_size(ctypes.byref(dmh))
    assert need == 4 * 128 * 128 * 4
    st = lib.kvs_vnorm(ctypes.byref(dmh), fake, 10, fake, fake, fake, need - 16, None)
    assert st == C.KVS_ERR_CAPACITY
    # surrogate limits
    big = C.dims(1, 32, 32, 128, 4096)
    assert lib.kvs_surrogate(ctypes.byref(big), fake, 10, fake, fake, fake, 0.0, 0, None, None,
                             None) == C.KVS_ERR_UNSUPPORTED
    odd = C.dims(1, 8, 8, 128, 100)
    assert lib.kvs_surrogate(ctypes.byref(odd), fake, 10, fake, fake, fake, 0.0, 0, None, None,
                             None) == C.KVS_ERR_UNSUPPORTED
    # MLP surrogate limits: H_kv not a power of two up to 16, D_mid not a multiple of 32,
    # D_h not a multiple of 64, misaligned hidden states
    for H, Dh, Dm in ((3, 256, 64), (32, 256, 64), (8, 256, 48), (8, 96, 64)):
        bad = C.dims(1, H, H, 128, Dh)
        assert lib.kvs_surrogate_mlp(ctypes.byref(bad), fake, 10, Dm, fake, fake, fake, fake, fake,
                                     0.0, 0, None, None, None) == C.KVS_ERR_UNSUPPORTED
    okd = C.dims(1, 8, 8, 128, 256)
    assert lib.kvs_surrogate_mlp(ctypes.byref(okd), fake + 2, 10, 64, fake, fake, fake, fake, fake,
                                 0.0, 0, None, None, None) == C.KVS_ERR_ALIGN
    assert lib.kvs_surrogate_mlp(ctypes.byref(okd), fake, 10, 64, fake, fake, fake, fake, fake,
                                 0.0, 0, fake, None, None) == C.KVS_ERR_ARG
    # compaction: max_pages too small, bad page size
    st = lib.kvs_compact_paged(ctypes.byref(dm), fake, fake, 100, fake, 16, fake, fake, 10, fake, 6,
                               fake, fake, fake, 1 << 20, None)
    assert st == C.KVS_ERR_SHAPE
    st = lib.kvs_compact_paged(ctypes.byref(dm), fake, fake, 100, fake, 0, fake, fake, 10, fake, 7,
                               fake, fake, fake, 1 << 20, None)
    assert st == C.KVS_ERR_UNSUPPORTED


def test_validation_codes_next_rows(capi):
    """The attention forward, pass-2 reductions, value refit and decode step."""
    C = capi
    lib = C._lib
    by = ctypes.byref
    dm = C.dims(1, 4, 2, 128, 0)
    fake = 1 << 20  # never dereferenced
    # attention forward: more queries than keys, missing output, missing tail, empty call
    assert lib.kvs_attn_fwd(by(dm), fake, 20, fake, fake, 10, fake, fake, 5, fake, fake,
                            None) == C.KVS_ERR_SHAPE
    assert lib.kvs_attn_fwd(by(dm), fake, 4, fake, fake, 10, None, None, 0, None, fake,
                            None) == C.KVS_ERR_ARG
    assert lib.kvs_attn_fwd(by(dm), fake, 4, fake, fake, 10, None, None, 2, fake, fake,
                            None) == C.KVS_ERR_ARG
    assert lib.kvs_attn_fwd(by(dm), None, 0, None, None, 10, None, None, 0, None, None,
                            None) == C.KVS_OK
    # KVzip(+) maximum: hidden states without D_h, short workspace, empty call
    assert lib.kvs_score_max(by(dm), fake, 4, fake, 10, fake, None, fake, 0, fake, fake, 1 << 30,
                             None) == C.KVS_ERR_SHAPE
    need = lib.kvs_score_max_workspace_size(by(dm), 4, 0)
    assert lib.kvs_score_max(by(dm), fake, 4, fake, 10, fake, None, None, 0, fake, fake, need - 1,
                             None) == C.KVS_ERR_CAPACITY
    assert lib.kvs_score_max(by(dm), None, 4, None, 0, None, None, None, 0, None, None, 0,
                             None) == C.KVS_OK
    # future mass: negative window, short workspace
    assert lib.kvs_score_future_sum(by(dm), fake, fake, 10, fake, -1, fake, fake, 1 << 30,
                                    None) == C.KVS_ERR_ARG
    need = lib.kvs_score_future_sum_workspace_size(by(dm), 10)
    assert need > 0
    assert lib.kvs_score_future_sum(by(dm), fake, fake, 10, fake, 0, fake, fake, need - 1,
                                    None) == C.KVS_ERR_CAPACITY
    # value refit: more kept keys than keys, negative ridge, k past the largest
    # factorisation, short workspace, empty call
    assert lib.kvs_value_refit(by(dm), fake, 10, fake, fake, 10, fake, 11, 1e-3, fake, fake,
                               1 << 30, None) == C.KVS_ERR_SHAPE
    assert lib.kvs_value_refit(by(dm), fake, 10, fake, fake, 100, fake, 50, -1.0, fake, fake,
                               1 << 30, None) == C.KVS_ERR_ARG
    assert lib.kvs_value_refit(by(dm), fake, 10, fake, fake, 9000, fake, 8193, 1e-3, fake, fake,
                               1 << 30, None) == C.KVS_ERR_UNSUPPORTED
    need = lib.kvs_value_refit_workspace_size(by(dm), 10, 100)
    # O fp16 [40][128], lse fp32 [40], A_S fp16 [40][128], Gram fp32 [2][128][128],
    # right-hand sides fp32 [2][128][128], each rounded up to 256 bytes
    assert need == 10240 + 256 + 10240 + 131072 + 131072
    assert lib.kvs_value_refit(by(dm), fake, 10, fake, fake, 200, fake, 100, 1e-3, fake, fake,
                               need - 1, None) == C.KVS_ERR_CAPACITY
    assert lib.kvs_value_refit(by(dm), None, 0, None, None, 200, None, 100, 1e-3, None, None, 0,
                               None) == C.KVS_OK
    # decode step: head dim, page size, block-table width, negative batch, empty call
    dd = C.dims(1, 2, 2, 128, 0)
    args = lambda B, page, maxp, d=dd: (by(d), B, 4, fake, fake, fake, fake, fake, fake, fake,
                                        0.0, page, fake, fake, 8, fake, fake, maxp, fake, 1, None)
    assert lib.kvs_decode_step(*args(2, 16, 4, C.dims(1, 2, 2, 96, 0))) == C.KVS_ERR_UNSUPPORTED
    assert lib.kvs_decode_step(*args(2, 0, 4)) == C.KVS_ERR_UNSUPPORTED
    assert lib.kvs_decode_step(*args(2, 16, 0)) == C.KVS_ERR_SHAPE
    assert lib.kvs_decode_step(*args(-1, 16, 4)) == C.KVS_ERR_ARG
    assert lib.kvs_decode_step(*args(0, 16, 4)) == C.KVS_OK


def test_workspace_sizes(capi):
    C = capi
    dm = C.dims(36, 32, 8, 128, 4096)
    assert C.kvs_vnorm_workspace_size(dm) == 36 * 32 * 128 * 128 * 4
    # ln||h|| [L][n_q] (256-byte aligned), constants [L][H_q][n_q rounded to 256][16] bf16,
    # a 128 x 16 bf16 ones tile
    assert C.kvs_score_max_workspace_size(dm, 2048, 1) == 36 * 32 * 2048 * 32 + 4096
    assert C.kvs_score_max_workspace_size(dm, 2048, 0) == 36 * 32 * 2048 * 32 + 4096
    assert C.kvs_score_max_workspace_size(dm, 100, 0) == 36 * 32 * 256 * 32 + 4096
    assert C.kvs_compact_workspace_size(dm, 32768) >= 36 * 8 * (8 + 1) * 4


def test_binding_rejects_host_tensors(capi):
    import torch
    C = capi
    dm = C.dims(1, 2, 1, 64, 0)
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        C.kvs_lse(dm, q, 4, q, 4, None, 0, q, stream=0)


def _prototypes():
    """name -> (return type, [parameter types]) of every function declared in kvs.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w ]*?[\s\*]+)(kvs_[a-z_]+)\s*\(([^;{]*?)\)\s*;",
                                        text):
        plist = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        # drop the parameter name: what remains is the type
        out[name] = (ret.strip(), [re.sub(r"\s*\b\w+$", "", p).strip() if not p.endswith("*")
                                   else p for p in plist])
    return out


def _kind(ctype_or_c):
    """Coarse kind of a C type string or a ctypes type: ptr, f32, i32, u64, str."""
    if isinstance(ctype_or_c, str):
        t = ctype_or_c.replace("const", "").strip()
        if "char" in t and "*" in t:
            return "str"
        if "*" in t:
            return "ptr"
        # size_t and uint64_t are the same 64-bit unsigned type on LP64 (and in ctypes)
        return {"float": "f32", "int32_t": "i32", "int": "i32", "size_t": "u64",
                "uint64_t": "u64", "kvs_status": "i32"}[t]
    c = ctype_or_c
    if c is ctypes.c_char_p:
        return "str"
    if c in (ctypes.c_void_p,) or (isinstance(c, type) and issubclass(c, ctypes._Pointer)):
        return "ptr"
    if c is ctypes.c_float:
        return "f32"
    if c in (ctypes.c_int32, ctypes.c_int):
        return "i32"
    if c in (ctypes.c_size_t, ctypes.c_uint64):
        return "u64"
    raise AssertionError(c)


def test_binding_signatures_match_the_header(capi):
    protos = _prototypes()
    assert set(protos) == set(capi._SIGS), set(protos) ^ set(capi._SIGS)
    for name, (ret, params) in protos.items():
        args, res = capi._SIGS[name]
        assert [_kind(p) for p in params] == [_kind(a) for a in args], name
        assert _kind(ret) == _kind(res), name
