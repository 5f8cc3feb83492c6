"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Every mutation below is a one-line slip (a dropped term, a wrong sign, index or
comparison, a transposed operand).  The mutated source is compiled into a fresh
module on the CPU; the pin tests of ``test_oracle_pins`` run against it and at
least one of them must fail.
"""
import inspect
import os
import types

import pytest

import oracle.kvs_oracle as real
from tests import test_oracle_pins as pins

SRC = inspect.getsource(real)

MUTATIONS = [
    ("logit scale 1/d", "return (q_row_block @ keys.T) / math.sqrt(d)",
     "return (q_row_block @ keys.T) / d"),
    ("causal off by one", "<= (off + np.arange(n_q))[:, None]", "< (off + np.arange(n_q))[:, None]"),
    ("top-left causal alignment", "off = n_k - n_q\n    return", "off = 0\n    return"),
    ("lse drops the max", "out[l, hq] = m + np.log(", "out[l, hq] = np.log("),
    ("gqa modulo mapping", "x = attention_logits(q[l, hq], keys[l, hq // g])",
     "x = attention_logits(q[l, hq], keys[l, hq % H_kv])"),
    ("kvzip+ multiplies by ||h||", "a = a / hn[l][:, None]", "a = a * hn[l][:, None]"),
    ("kvzip+ divides by vn", "a = a * vnorm[l, hq][None, :]", "a = a / vnorm[l, hq][None, :]"),
    ("kvzip sum instead of max", "best = np.maximum(best, a.max(axis=0))",
     "best = np.maximum(best, a.sum(axis=0))"),
    ("kvzip first head only", "for hq in range(hk * g, (hk + 1) * g):\n                a = attention_rows",
     "for hq in range(hk * g, hk * g + 1):\n                a = attention_rows"),
    ("vnorm uses the kv head's slice", "Wh = w_o[l][:, hq * d:(hq + 1) * d]",
     "Wh = w_o[l][:, (hq // g) * d:(hq // g + 1) * d]"),
    ("vnorm transposed weight", "y = v[l, hq // g] @ Wh.T", "y = v[l, hq // g] @ Wh[:d].T"),
    ("hidden norm squared", "return np.sqrt((h * h).sum(axis=-1))", "return (h * h).sum(axis=-1)"),
    ("future band strict", "band = rows[:, None] >= cols[None, :] + w",
     "band = rows[:, None] > cols[None, :] + w"),
    ("future band reversed", "band = rows[:, None] >= cols[None, :] + w",
     "band = cols[None, :] >= rows[:, None] + w"),
    ("future uses wrong lse rows", "a = np.exp(x - lse_[l, hq, j0:j1, None])",
     "a = np.exp(x - lse_[l, hq, :j1 - j0, None])"),
    ("surrogate drops bias", "(h[l] @ W[l] + b[l][None, :]).T", "(h[l] @ W[l]).T"),
    ("surrogate token-major", "(h[l] @ W[l] + b[l][None, :]).T for l", "(h[l] @ W[l] + b[l][None, :]) for l"),
    ("threshold strict", "keep = (score >= tau) | (t >= T - w)", "keep = (score > tau) | (t >= T - w)"),
    ("window off by one", "keep = (score >= tau) | (t >= T - w)", "keep = (score >= tau) | (t > T - w)"),
    ("topk ties to later tokens", "return np.lexsort((pos, key, nan))", "return np.lexsort((-pos, key, nan))"),
    ("topk nan ranks high", "key = np.where(nan, 0.0, -row)", "key = np.where(nan, -np.inf, -row)\n    nan = nan & False"),
    ("topk ignores window", "mask[r, T - wn:] = 1", "mask[r, T - wn:] = 0"),
    ("chunked sum over chunks", "best = s if best is None else np.maximum(best, s)",
     "best = s if best is None else best + s"),
    ("chunked first chunk only", "best = s if best is None else np.maximum(best, s)",
     "best = s if best is None else best"),
    ("chunked last chunk only", "best = s if best is None else np.maximum(best, s)",
     "best = s"),
    ("quantile upper rank", "s[int(math.floor(qtl * (s.size - 1)))]", "s[int(math.ceil(qtl * (s.size - 1)))]"),
    ("quantile nan ranks high", "s = np.concatenate([v[nan], np.sort(v[~nan])])", "s = np.sort(v)"),
    ("quantile over the window too", "tau[l] = quantile_lower(score[l, :, : T - wn], qtl)",
     "tau[l] = quantile_lower(score[l], qtl)"),
    ("quantile per head 0 only", "tau[l] = quantile_lower(score[l, :, : T - wn], qtl)",
     "tau[l] = quantile_lower(score[l, 0, : T - wn], qtl)"),
    ("compaction descending", "idx = np.nonzero(mask[l, hh])[0]", "idx = np.nonzero(mask[l, hh])[0][::-1]"),
    ("compaction head-major pages", "block_table[l, hh, p] = first + p", "block_table[l, hh, p] = first + p + 1"),
    ("kv bytes without K and V", "return 2 * L * T * H_kv * d * bytes_per_elem",
     "return L * T * H_kv * d * bytes_per_elem"),
    ("mlp cost over 8", "return D_h / 4 * (D_h + H_kv)", "return D_h / 8 * (D_h + H_kv)"),
    ("bf16 shift 15", "<< np.uint32(16)", "<< np.uint32(15)"),
    ("forward uses modulo kv head for values", "o[l, hq] = a @ vals[l, hq // g]",
     "o[l, hq] = a @ vals[l, hq % vals.shape[1]]"),
    ("forward drops tail values", "vals = np.concatenate([v_ctx, v_tail], 2) if has_tail else v_ctx",
     "vals = np.concatenate([v_ctx, 0 * v_tail], 2) if has_tail else v_ctx"),
    ("forward transposes the weights", "o[l, hq] = a @ vals[l, hq // g]",
     "o[l, hq] = (a[:, ::-1] @ vals[l, hq // g][::-1])[::-1]"),
    ("refit uses kv-head rows only", "Q = q[l, hk * g:(hk + 1) * g].reshape(g * n_q, d)",
     "Q = np.concatenate([q[l, hk * g]] * g).reshape(g * n_q, d)"),
    ("refit normalises over all keys", "a_s /= a_s.sum(axis=1, keepdims=True)",
     "a_s /= np.exp(x - xs.max(axis=1, keepdims=True)).sum(axis=1, keepdims=True)"),
    ("refit drops the ridge", "M = a_s.T @ a_s + lam * np.eye(len(idx))", "M = a_s.T @ a_s + 1e-14 * np.eye(len(idx))"),
    ("refit solves a scaled system", "row_v.append(np.linalg.solve(M, a_s.T @ O_t))",
     "row_v.append(np.linalg.solve(M.T * 1.01, a_s.T @ O_t))"),
    ("decode strict threshold", "if score[r, leaving] >= tau:", "if score[r, leaving] > tau:"),
    ("decode evicts the newest", "leaving = window[r].pop(0)", "leaving = window[r].pop()"),
    ("decode window one short", "if len(window[r]) > w:", "if len(window[r]) >= w:"),
    ("gelu without 1/sqrt2", "_erf(x / math.sqrt(2.0))", "_erf(x)"),
    ("gelu tanh form", "return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))",
     "return 0.5 * x * (1.0 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))"),
    ("mlp relu", "out.append((gelu(u) @ W2[l].T", "out.append((np.maximum(u, 0) @ W2[l].T"),
    ("mlp drops hidden bias", "u = h[l] @ W1[l].T + b1[l][None, :]", "u = h[l] @ W1[l].T"),
    ("mlp drops output bias", "@ W2[l].T + b2[l][None, :]).T)", "@ W2[l].T).T)"),
    ("mlp token-major", "@ W2[l].T + b2[l][None, :]).T)", "@ W2[l].T + b2[l][None, :]))"),
]


def _pin_tests():
    return [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _mutant(src):
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = real.__file__
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


# a planted slip may produce NaN or inf along the way (e.g. -inf - -inf); that is expected
@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new, monkeypatch):
    assert SRC.count(old) >= 1, f"mutation anchor not found: {name}"
    mutant = _mutant(SRC.replace(old, new, 1))
    monkeypatch.setattr(pins, "O", mutant)
    failures = 0
    for t in _pin_tests():
        try:
            t()
        except Exception:
            failures += 1
    assert failures > 0, f"no pin catches: {name}"


def test_unmutated_oracle_passes_all_pins(monkeypatch):
    monkeypatch.setattr(pins, "O", _mutant(SRC))
    for t in _pin_tests():
        t()
