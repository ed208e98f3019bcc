"""GPU parity of the restore step (linear decoder + reference mean + RoPE on keys):
the CUDA path through the C ABI against the fp64 oracle on the same records.

Records come from the seeded generator (arbitrary well-formed codes, extremes,
reference relations and pools), not from the CUDA write path, so the oracle sees only
generator values.  A second test restores reference tokens of a cache the GPU wrote
and checks the properties that must hold whatever the codes are."""
import math

import numpy as np
import pytest
import torch

import oracle
import rkv_workload as wl
from reference_residual_kv_gb300 import rkv

from _gpu_common import GUARD, assert_guards, ensure_lib, gen_inputs, out_buffer, run_gpu, to_device

pytestmark = pytest.mark.gpu

C = wl.CONFIGS

# bf16 decoder input (2^-9 relative per element), fp32 accumulation and one bf16
# rounding of the output (2^-9 relative): an element may be off by a few units of
# 2^-9 of its row's largest magnitude; the row's RMS error is held tighter.
TOL_MAX = 8e-3
TOL_RMS = 3e-3


def pack_codes(q: np.ndarray, bits: int) -> np.ndarray:
    """[..][d_c] codes -> stored bytes: INT4 coordinate 2j in the low nibble of byte j,
    INT2 coordinate 4j+i in bits 2i..2i+1 of byte j."""
    q = q.astype(np.uint8)
    if bits == 4:
        return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return (q[..., 0::4] | (q[..., 1::4] << 2) | (q[..., 2::4] << 4) | (q[..., 3::4] << 6)).astype(np.uint8)


def refs_f64(cfg, refs):
    if cfg.ref_dtype == "fp8":
        return oracle.fp8_decode(refs.reshape(-1)).reshape(refs.shape)
    return wl.stored_to_f64(refs, cfg.ref_dtype)


def load_records(cfg, bufs, recs):
    """Copy generator records [(codes, zmin, delta, ref_idx, refs)] per lb into the
    GPU pool and cache buffers."""
    for lb, (q, zmin, delta, idx, refs) in enumerate(recs):
        bufs.codes[lb].copy_(torch.from_numpy(pack_codes(q, cfg.bits)))
        bufs.hdr[lb].copy_(torch.from_numpy(np.stack([zmin, delta], axis=-1).astype(np.float32)))
        bufs.ref_idx[lb].copy_(torch.from_numpy(idx))
        if cfg.ref_dtype == "fp8":
            bufs.ref_vec[lb].copy_(torch.from_numpy(refs))
        else:
            bufs.ref_vec[lb].copy_(torch.from_numpy(refs.view(np.int16)).view(torch.bfloat16))


def compare_rows(got, want, what):
    err = np.abs(got - want)
    rmax = np.abs(want).max(axis=1, keepdims=True)
    bad = err > TOL_MAX * rmax + 1e-6
    assert not bad.any(), "%s: %d elements off; worst %.3g of row max %.3g" % (
        what, bad.sum(), err.max(), rmax.max())
    rms = np.sqrt((err ** 2).mean(axis=1)) / np.maximum(np.sqrt((want ** 2).mean(axis=1)), 1e-30)
    assert rms.max() <= TOL_RMS, "%s: row RMS error %.3g" % (what, rms.max())


def _restore_case(cfg, n_sel, seed):
    ensure_lib()
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p, guard=GUARD)
    n_ref = bufs.n_ref
    recs = [wl.synthetic_records(cfg, n_ref, lb) for lb in range(cfg.L * cfg.B)]
    load_records(cfg, bufs, recs)
    Wd = [wl.decoder_weights(cfg, l) for l in range(cfg.L)]
    Wd_d = to_device(np.stack(Wd), cfg.kv_dtype)
    rng = np.random.default_rng(seed)
    sel = np.stack([np.sort(rng.choice(cfg.T, n_sel, replace=False)) for _ in range(cfg.L * cfg.B)])
    sel[:, -1] = cfg.T - 1                         # the largest position (widest RoPE angles)
    sel_d = torch.from_numpy(sel.astype(np.int32)).cuda()
    dk = cfg.N * cfg.D
    out_k = out_buffer((cfg.L * cfg.B, n_sel, dk), torch.bfloat16)
    out_v = out_buffer(out_k.shape, out_k.dtype)
    bufs.restore(Wd_d, sel_d, out_k, out_v, cfg.rope_base)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    assert_guards(bufs)
    gk = out_k.float().cpu().numpy()
    gv = out_v.float().cpu().numpy()
    for lb, (q, zmin, delta, idx, refs) in enumerate(recs):
        l = lb // cfg.B
        K, V = oracle.restore(cfg, refs_f64(cfg, refs), q, zmin, delta, idx,
                              wl.stored_to_f64(Wd[l], cfg.kv_dtype), sel[lb])
        compare_rows(gk[lb], K, "%s lb %d keys" % (cfg.name, lb))
        compare_rows(gv[lb], V, "%s lb %d values" % (cfg.name, lb))


@pytest.mark.parametrize("name,T,n_sel", [
    ("llama3.1-8b-kv", 1000, 300),          # bf16 pool, INT4; 300 = one full and one ragged pair tile
    ("long-131k-fp8ref", 131072, 260),      # FP8 pool, positions up to 131071
    ("multimodal-8x4096-int2", 4096, 200),  # INT2, 8 sequences
])
def test_restore_matches_oracle_on_generator_records(name, T, n_sel):
    cfg = C[name].replace(L=min(C[name].L, 2), T=T)
    _restore_case(cfg, n_sel, seed=T)


def test_restore_of_reference_tokens_in_a_written_cache():
    # a reference token's record is z = 0 with its own slot: V^ is the stored reference
    # bit for bit (one fp32 add, times 1, rounded to bf16), K^ its rotation per head
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=1000)
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w, want_z=False)
    s = cfg.stride
    sel = np.arange(0, cfg.T, s, dtype=np.int32)[:100]
    Wd_d = to_device(wl.decoder_weights(cfg, 0)[None], cfg.kv_dtype)
    dk = cfg.N * cfg.D
    out_k = out_buffer((1, sel.size, dk), torch.bfloat16)
    out_v = out_buffer(out_k.shape, out_k.dtype)
    bufs.restore(Wd_d, torch.from_numpy(sel[None]).cuda(), out_k, out_v, cfg.rope_base)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    assert_guards(bufs)
    x = kv[0][0][sel]                                    # bf16 bits [n][W]
    assert np.array_equal(out_v[0].cpu().view(torch.int16).numpy().view(np.uint16), x[:, dk:])
    xk = wl.stored_to_f64(x[:, :dk], "bf16")
    i = np.arange(cfg.D // 2)
    theta = cfg.rope_base ** (-2.0 * i / cfg.D)
    got = out_k[0].float().cpu().numpy()
    for n, t in enumerate(sel):
        a = t * theta
        for h in range(cfg.N):
            v = xk[n, h * cfg.D:(h + 1) * cfg.D]
            want = np.empty_like(v)
            want[0::2] = v[0::2] * np.cos(a) - v[1::2] * np.sin(a)
            want[1::2] = v[0::2] * np.sin(a) + v[1::2] * np.cos(a)
            g = got[n, h * cfg.D:(h + 1) * cfg.D]
            assert np.abs(g - want).max() <= 2 ** -8 * np.abs(want).max() + 1e-6, (t, h)


def test_restore_padding_and_out_of_range_indices():
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=600)
    ensure_lib()
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p)
    load_records(cfg, bufs, [wl.synthetic_records(cfg, bufs.n_ref, 0)])
    Wd_d = to_device(wl.decoder_weights(cfg, 0)[None], cfg.kv_dtype)
    sel = np.array([[5, -1, 17, cfg.T + 3, 40]], np.int32)
    dk = cfg.N * cfg.D
    out_k = torch.full((1, 5, dk), 7.0, dtype=torch.bfloat16, device="cuda")
    out_v = torch.full_like(out_k, 7.0)
    bufs.restore(Wd_d, torch.from_numpy(sel).cuda(), out_k, out_v, cfg.rope_base)
    torch.cuda.synchronize()
    assert bufs.device_status() == rkv.RKV_ERR_INDEX
    k = out_k.float().cpu().numpy()[0]
    v = out_v.float().cpu().numpy()[0]
    for j in (1, 3):                                    # padding and the bad index: zero rows
        assert not k[j].any() and not v[j].any()
    for j in (0, 2, 4):                                 # the others are restored
        assert np.abs(v[j]).max() > 0


def test_restore_full_size_sampled():
    # the long-context workload as the benchmark restores it: one decode step's whole
    # selection (30 % of 131,072 positions plus the last 512) in one call, FP8 pool;
    # sampled rows against the oracle
    cfg = C["long-131k-fp8ref"]
    ensure_lib()
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p, guard=GUARD)
    rec = wl.synthetic_records(cfg, bufs.n_ref, 0)
    load_records(cfg, bufs, [rec])
    Wd = wl.decoder_weights(cfg, 0)
    sel = wl.gather_selection(cfg, 0).astype(np.int32)[None]
    n = sel.shape[1]
    dk = cfg.N * cfg.D
    out_k = out_buffer((1, n, dk), torch.bfloat16)
    out_v = out_buffer(out_k.shape, out_k.dtype)
    bufs.restore(to_device(Wd[None], cfg.kv_dtype), torch.from_numpy(sel).cuda(), out_k, out_v,
                 cfg.rope_base)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    assert_guards(bufs)
    pick = np.sort(np.random.default_rng(11).choice(n, 64, replace=False))
    pick[-1] = n - 1                                     # the last position
    q, zmin, delta, idx, refs = rec
    K, V = oracle.restore(cfg, refs_f64(cfg, refs), q, zmin, delta, idx,
                          wl.stored_to_f64(Wd, cfg.kv_dtype), sel[0][pick])
    idx_t = torch.from_numpy(pick).cuda()
    compare_rows(out_k[0].index_select(0, idx_t).float().cpu().numpy(), K, "full-size keys")
    compare_rows(out_v[0].index_select(0, idx_t).float().cpu().numpy(), V, "full-size values")
