"""The benchmark's roofline arithmetic against closed forms derived by hand.

With a fixed stride s and references at positions 0, s, 2s, ..., the s - 1 tokens after
reference q see q + 1 earlier references, so the causal (token, reference) pairs of one
layer-sequence sum to (s - 1) * n_ref * (n_ref + 1) / 2.  The algorithmic FLOPs are then
the distances (2W per pair), the first compressor layer once per non-reference token and
once per reference (4 W d_ff), and W_c3 once per non-reference token (2 d_ff d_c).
"""
import pytest

import bench
import rkv_workload as wl

C = wl.CONFIGS


def _pairs_closed_form(T, s):
    n_ref = T // s
    return (s - 1) * n_ref * (n_ref + 1) // 2


@pytest.mark.parametrize("name,pairs_per_seq", [
    ("llama3.1-8b-kv", 3_673_600),          # 7 * 1024 * 1025 / 2
    ("qwen2.5-7b-kv", 58_734_592),          # 7 * 4096 * 4097 / 2
    ("long-131k-fp8ref", 503_377_920),      # 15 * 8192 * 8193 / 2
    ("multimodal-8x4096-int2", 919_296),    # 7 * 512 * 513 / 2
])
def test_causal_pool_pairs(name, pairs_per_seq):
    cfg = C[name]
    assert _pairs_closed_form(cfg.T, cfg.stride) == pairs_per_seq
    fl, n_ref, n_non, pairs = bench.algorithmic(cfg)
    assert pairs == pairs_per_seq
    assert n_ref == cfg.T // cfg.stride and n_non == cfg.T - n_ref


@pytest.mark.parametrize("name", ["llama3.1-8b-kv", "qwen2.5-7b-kv", "long-131k-fp8ref",
                                  "multimodal-8x4096-int2"])
def test_algorithmic_flops_per_step(name):
    cfg = C[name]
    W, F, Dc = cfg.W, cfg.d_ff, cfg.d_c
    n_ref = cfg.T // cfg.stride
    n_non = cfg.T - n_ref
    per_seq = (_pairs_closed_form(cfg.T, cfg.stride) * 2 * W + n_non * (4 * W * F + 2 * F * Dc)
               + n_ref * 4 * W * F)
    fl, _, _, _ = bench.algorithmic(cfg)
    assert sum(fl.values()) == pytest.approx(cfg.L * cfg.B * per_seq, rel=1e-12)


def test_llama_step_is_2_92_tflop():
    fl, _, _, _ = bench.algorithmic(C["llama3.1-8b-kv"])
    assert round(sum(fl.values()) / 1e12, 2) == 2.92


def test_read_bytes_per_token():
    # codes 256 + extremes 128 + slots 16 + index 4, then the outputs in bf16
    cfg = C["long-131k-fp8ref"]
    assert bench.gather_bytes_per_token(cfg) == 256 + 128 + 16 + 4 + 512 * 2 + 2048 * 2 == 5524
    assert bench.restore_bytes_per_token(cfg) == 256 + 128 + 16 + 4 + 2048 * 2 == 4500
