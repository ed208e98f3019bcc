"""GPU parity of sparse attention over the restored set: the CUDA path through the C ABI
against the fp64 oracle on the same generator inputs, alone and after the restore."""
import math

import numpy as np
import pytest
import torch

import oracle
import rkv_workload as wl
from reference_residual_kv_gb300 import rkv

from _gpu_common import GUARD, assert_guards, ensure_lib, out_buffer, to_device
from test_gpu_restore import load_records, refs_f64

pytestmark = pytest.mark.gpu

C = wl.CONFIGS


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _attend(cfg, q_bits, k_bits, v_bits, sel):
    ensure_lib()
    p = rkv.params_from_config(cfg)
    LB = cfg.L * cfg.B
    out = out_buffer((LB, cfg.H, cfg.D), torch.float32)
    n_sel = sel.shape[1]
    ws = out_buffer((max(rkv.rkv_attention_workspace(p, cfg.H, n_sel), 256),), torch.uint8)
    rkv.rkv_sparse_attention(p, cfg.H, _bf16(q_bits), _bf16(k_bits), _bf16(v_bits),
                             torch.from_numpy(sel.astype(np.int32)).cuda(), n_sel, out, ws, ws.numel())
    torch.cuda.synchronize()
    assert_guards()
    return out.cpu().numpy()


@pytest.mark.parametrize("name,n_sel,shape", [
    ("llama3.1-8b-kv", 1200, {}),                      # 32 query heads on 8 KV heads; ragged batches
    ("qwen2.5-7b-kv", 700, {}),                        # 28 query heads on 4 KV heads (groups of 7)
    ("llama3.1-8b-kv", 333, dict(N=16, D=64)),         # D = 64, groups of 2
    ("llama3.1-8b-kv", 517, dict(N=4, D=64)),          # D = 64, groups of 8
    ("llama3.1-8b-kv", 901, dict(N=4, D=256, H=16)),   # D = 256, groups of 4
    # D = 128 takes the tensor-core pass: one query head per KV head, groups of 2 and 8,
    # and selections one row short of, one row past and just under whole 128-row tiles
    ("llama3.1-8b-kv", 127, dict(H=8)),
    ("llama3.1-8b-kv", 129, dict(H=16)),
    ("llama3.1-8b-kv", 255, dict(H=64)),
])
def test_attention_matches_oracle(name, n_sel, shape):
    cfg = C[name].replace(L=2, T=4096, **shape)
    dk = cfg.N * cfg.D
    kv = [wl.layer_kv(cfg, l)[0] for l in range(cfg.L)]           # rows stand in for K^ | V^
    rng = np.random.default_rng(n_sel)
    sel = np.stack([rng.choice(cfg.T, n_sel, replace=False) for _ in range(cfg.L)]).astype(np.int32)
    sel[:, 5] = -1                                                 # padding
    sel[1, 9] = cfg.T + 7                                          # outside [0, T): left out
    K = np.stack([kv[l][sel[l].clip(0, cfg.T - 1), :dk] for l in range(cfg.L)])
    V = np.stack([kv[l][sel[l].clip(0, cfg.T - 1), dk:] for l in range(cfg.L)])
    q = np.stack([wl.decode_queries(cfg, l, 0)[0] for l in range(cfg.L)])
    got = _attend(cfg, q, K, V, sel)
    for l in range(cfg.L):
        valid = ((sel[l] >= 0) & (sel[l] < cfg.T)).astype(np.int32)
        want = oracle.attention(wl.stored_to_f64(q[l], "bf16"), wl.stored_to_f64(K[l], "bf16"),
                                wl.stored_to_f64(V[l], "bf16"), cfg.N, valid)
        scale = np.abs(want).max()
        assert np.abs(got[l] - want).max() <= 1e-4 * scale, np.abs(got[l] - want).max() / scale


def test_attention_with_no_selected_row_is_zero():
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=256)
    dk = cfg.N * cfg.D
    sel = np.full((1, 40), -1, np.int32)
    z = np.zeros((1, 40, dk), np.uint16)
    got = _attend(cfg, wl.decode_queries(cfg, 0, 0), z, z, sel)
    assert not got.any()


def test_restore_then_attention_matches_the_oracle_chain():
    # generator records -> GPU restore -> GPU attention, against the fp64 restore and
    # attention of the oracle.  The bf16 rounding of K^ and V^ moves each score by about
    # 2^-9 |q||k| / sqrt(D); with N(0, 1) pool vectors the scores are O(1), the softmax is
    # smooth, and the outputs agree to about 1e-2 of their scale.  (Uniform FP8 bytes reach
    # +-448: scores in the hundreds make the softmax nearly one-hot and any rounding of
    # K^ decisive, so that pool is left to the restore's own parity test.)
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=8192)
    ensure_lib()
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p, guard=GUARD)
    rec = wl.synthetic_records(cfg, bufs.n_ref, 0)
    load_records(cfg, bufs, [rec])
    Wd = wl.decoder_weights(cfg, 0)
    sel = np.sort(np.random.default_rng(3).choice(cfg.T, 2000, replace=False)).astype(np.int32)[None]
    dk = cfg.N * cfg.D
    sel_d = torch.from_numpy(sel).cuda()
    out_k = out_buffer((1, sel.shape[1], dk), torch.bfloat16)
    out_v = out_buffer(out_k.shape, out_k.dtype)
    bufs.restore(to_device(Wd[None], cfg.kv_dtype), sel_d, out_k, out_v, cfg.rope_base)
    q = wl.decode_queries(cfg, 0, 0)
    out = out_buffer((1, cfg.H, cfg.D), torch.float32)
    bufs.attend(cfg.H, _bf16(q), out_k, out_v, sel_d, out)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    assert_guards(bufs)
    q_, zmin, delta, idx, refs = rec
    K, V = oracle.restore(cfg, refs_f64(cfg, refs), q_, zmin, delta, idx,
                          wl.stored_to_f64(Wd, cfg.kv_dtype), sel[0])
    want = oracle.attention(wl.stored_to_f64(q[0], "bf16"), K, V, cfg.N)
    got = out.cpu().numpy()[0]
    assert np.abs(got - want).max() <= 1e-2 * np.abs(want).max()


def test_attention_full_size():
    # as the benchmark runs it: 32 query heads on 8 KV heads over one long-context decode
    # step's whole selection (~39.7 k rows), one call
    cfg = C["long-131k-fp8ref"]
    sel = wl.gather_selection(cfg, 0).astype(np.int32)[None]
    n = sel.shape[1]
    dk = cfg.N * cfg.D
    rng = np.random.default_rng(5)
    K = wl.store(rng.normal(size=(1, n, dk)), "bf16")
    V = wl.store(rng.normal(size=(1, n, dk)), "bf16")
    q = wl.decode_queries(cfg, 0, 0)
    got = _attend(cfg, q, K, V, sel)
    want = oracle.attention(wl.stored_to_f64(q[0], "bf16"), wl.stored_to_f64(K[0], "bf16"),
                            wl.stored_to_f64(V[0], "bf16"), cfg.N)
    scale = np.abs(want).max()
    assert np.abs(got[0] - want).max() <= 1e-4 * scale, np.abs(got[0] - want).max() / scale
