"""The seeded input generators the tests and the benchmark share: determinism and the
properties the read-side measurements and parity cases rely on."""
import numpy as np
import pytest

import rkv_workload as wl

C = wl.CONFIGS


@pytest.mark.parametrize("name", ["long-131k-fp8ref", "llama3.1-8b-kv"])
def test_gather_selection(name):
    cfg = C[name]
    s0 = wl.gather_selection(cfg, 0)
    assert s0.dtype == np.int32
    assert np.all(np.diff(s0) > 0)                           # sorted, unique
    assert s0[0] >= 0 and s0[-1] == cfg.T - 1
    tail = np.arange(cfg.T - cfg.gather_tail, cfg.T)
    assert np.isin(tail, s0).all()                           # the last tokens always
    n = int(np.floor(cfg.gather_frac * cfg.T))
    assert n <= s0.size <= n + cfg.gather_tail
    assert np.array_equal(s0, wl.gather_selection(cfg, 0))   # deterministic per step
    assert not np.array_equal(s0, wl.gather_selection(cfg, 1))


def test_layer_kv_is_deterministic_and_layers_differ():
    cfg = C["llama3.1-8b-kv"].replace(T=512)
    a = wl.layer_kv(cfg, 0)
    assert a.shape == (cfg.B, cfg.T, cfg.W) and a.dtype == np.uint16
    assert np.array_equal(a, wl.layer_kv(cfg, 0))
    assert not np.array_equal(a, wl.layer_kv(cfg, 1))


@pytest.mark.parametrize("name", ["llama3.1-8b-kv", "long-131k-fp8ref", "multimodal-8x4096-int2"])
def test_synthetic_records_are_well_formed(name):
    cfg = C[name].replace(T=700)
    n_ref = 50
    q, zmin, delta, idx, refs = wl.synthetic_records(cfg, n_ref, 3)
    assert q.shape == (cfg.T, cfg.d_c) and q.max() < (1 << cfg.bits)
    assert np.all(delta[:, ::7] == 0) and np.all(delta >= 0)
    cnt = (idx >= 0).sum(axis=1)
    assert cnt.min() >= 1 and cnt.max() <= cfg.k
    for t in range(cfg.T):                                   # ascending, -1 padded, distinct
        v = idx[t, :cnt[t]]
        assert np.all(np.diff(v) > 0) and np.all(idx[t, cnt[t]:] == -1)
        assert v.min() >= 0 and v.max() < n_ref
    if cfg.ref_dtype == "fp8":
        assert refs.dtype == np.uint8 and not np.isin(refs, [0x7F, 0xFF]).any()


def test_synthetic_reference_sets_follow_their_definition():
    # each row's set is its first cnt draws of Floyd's sampling of k distinct slots, sorted
    cfg = C["llama3.1-8b-kv"].replace(T=300)
    n_ref = 40
    _, _, _, idx, _ = wl.synthetic_records(cfg, n_ref, 0)
    key = lambda part: wl.stream_key(cfg.seed, wl.TAG_REC, 0, part)
    cnt = 1 + np.minimum(np.floor(wl.uniform(key(3), cfg.T) * cfg.k), cfg.k - 1).astype(np.int64)
    u = wl.uniform(key(4), cfg.T * cfg.k).reshape(cfg.T, cfg.k)
    for t in range(cfg.T):
        taken = []
        for i in range(cfg.k):
            j = n_ref - cfg.k + i
            r = min(int(np.floor(u[t, i] * (j + 1))), j)
            taken.append(j if r in taken else r)
        assert len(set(taken)) == cfg.k
        want = np.full(cfg.k, -1)
        want[:cnt[t]] = np.sort(taken[:cnt[t]])
        assert np.array_equal(idx[t], want)
