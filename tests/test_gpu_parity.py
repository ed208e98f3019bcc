"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs.  Small cases check every token's reference set and a sample of
tokens' codes; full-size configs (launched as the benchmark launches them: all layers
in one call) check sampled tokens of several layers.  Read-path tests check the
gather against the records it reads and against the oracle's means, that it never
reads an unselected token, and that bad indices are reported, not faulted on."""
import math

import numpy as np
import pytest
import torch

import oracle
import rkv_workload as wl
from reference_residual_kv_gb300 import rkv

from _gpu_common import (CODE_BUDGET, assert_guards, check_all_indices, check_tokens, gen_inputs,
                         host_records, out_buffer, run_gpu, sample_tokens, to_device)

pytestmark = pytest.mark.gpu

C = wl.CONFIGS


def _parity(cfg, n_sample=120, layers_checked=None, all_idx=True, seed=0):
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w)
    assert bufs.device_status() == 0
    gpu = host_records(cfg, bufs)
    report = {}
    layers_checked = range(cfg.L) if layers_checked is None else layers_checked
    for l in layers_checked:
        for b in range(cfg.B):
            lb = l * cfg.B + b
            if all_idx:
                check_all_indices(cfg, kv[l][b], gpu["idx"][lb], report=report)
            toks = sample_tokens(cfg, n_sample, seed + lb)
            if not all_idx:
                check_all_indices(cfg, kv[l][b], gpu["idx"][lb], tokens=toks, report=report)
            check_tokens(cfg, kv[l][b], w[l], gpu, lb, toks, report=report)
    assert report["flips"] <= CODE_BUDGET * report["coords"], report
    print(cfg.name, report)
    return bufs, kv, w, gpu, report


# ------------------------------------------------------------------ write path
def test_tiny_fp32_every_token():
    cfg = C["tiny-fp32"]
    bufs, kv, w, gpu, rep = _parity(cfg, n_sample=cfg.T)
    assert rep["tokens"] == cfg.T and rep["max_rel_z"] < 1e-4


SMALL = {
    "llama-2x1000": C["llama3.1-8b-kv"].replace(L=2, T=1000),
    "qwen-1x777": C["qwen2.5-7b-kv"].replace(L=1, T=777),
    "long-fp8-1x1500": C["long-131k-fp8ref"].replace(T=1500),
    "mm-int2-2x4096": C["multimodal-8x4096-int2"].replace(B=2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_bf16_small_ragged(name):
    cfg = SMALL[name]
    _parity(cfg, n_sample=100, all_idx=True)


@pytest.mark.parametrize("name,layers", [
    ("llama3.1-8b-kv", [0, 17, 31]),
    ("qwen2.5-7b-kv", [0, 27]),
    ("long-131k-fp8ref", [0]),
    ("multimodal-8x4096-int2", [0]),
])
def test_full_size_sampled(name, layers):
    cfg = C[name]
    n = 60 if cfg.T > 10000 else 80
    _parity(cfg, n_sample=n, layers_checked=layers, all_idx=False)


def test_gate_weight_placement_gives_identical_records():
    # W_c2 after W_c1 at a 16-byte multiple is loaded with one TMA box per stage, the
    # other order with two; both must give bit-identical records
    cfg = SMALL["llama-2x1000"]
    kv, w = gen_inputs(cfg)
    kv_d = to_device(np.stack(kv), cfg.kv_dtype)
    W1 = np.stack([x[0] for x in w])
    W2 = np.stack([x[1] for x in w])
    W3 = to_device(np.stack([x[2] for x in w]), cfg.kv_dtype)
    after = to_device(np.stack([W1, W2]), cfg.kv_dtype)       # [W_c1 | W_c2]
    before = to_device(np.stack([W2, W1]), cfg.kv_dtype)      # [W_c2 | W_c1]
    recs = []
    for w1, w2 in ((after[0], after[1]), (before[1], before[0])):
        bufs = rkv.Buffers(rkv.params_from_config(cfg), want_z=True)
        bufs.build_ref_pool(kv_d)
        bufs.compress(kv_d, w1, w2, W3)
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        recs.append(host_records(cfg, bufs))
    for key in ("idx", "q", "hdr", "z"):
        assert np.array_equal(recs[0][key], recs[1][key]), key


def test_edge_cases_small_T_first_offset_k():
    base = C["llama3.1-8b-kv"].replace(L=1, N=2, D=64, d_ff=256, d_c=64)
    # T % 8 == 0 with a stride dividing 8 from position 0 takes the layout that leaves
    # the reference rows out of the first compressor layer: one group, a ragged tile,
    # references at every 4th and every 2nd position
    for cfg in (base.replace(T=1), base.replace(T=9), base.replace(T=130),
                base.replace(T=300, first=5), base.replace(T=300, k=1),
                base.replace(T=300, k=2, bits=2), base.replace(T=8), base.replace(T=136),
                base.replace(T=512, stride=4), base.replace(T=264, stride=2)):
        bufs, kv, w, gpu, rep = _parity(cfg, n_sample=cfg.T)
        if cfg.first > 0:
            # tokens before the first reference have an empty pool: no refs, z = f_c(kv)
            assert np.all(gpu["idx"][0][: cfg.first] == -1)


def test_dynamic_schedule_matches_oracle_and_table6():
    # the device schedule (recurrence on one thread, pools by binary search) equals the
    # oracle's, and reproduces Table VI's reference counts under the stated reading
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "table6_ref_counts.json")))
    for alpha, n in zip(g["alpha"][1:], g["n_ref"][1:]):
        cfg = wl.CONFIGS["tiny-fp32"].replace(T=g["T"], N=1, D=4, d_ff=32, d_c=32, stride=g["s0"],
                                             alpha=alpha, n_sink=g["n_sink"])
        p = rkv.params_from_config(cfg)
        bufs = rkv.Buffers(p)
        kv = torch.zeros((1, cfg.T, cfg.W), dtype=torch.float32, device="cuda")
        bufs.build_ref_pool(kv)
        torch.cuda.synchronize()
        ref_pos = oracle.schedule(cfg)
        assert bufs.n_ref == n == ref_pos.size
        assert np.array_equal(bufs.ref_pos.cpu().numpy()[:n], ref_pos)
        ps = bufs.pool_size.cpu().numpy()
        assert np.array_equal(ps, np.searchsorted(ref_pos, np.arange(cfg.T), side="left"))
        slot = bufs.ref_slot.cpu().numpy()
        assert np.array_equal(np.nonzero(slot >= 0)[0], ref_pos) and np.array_equal(slot[ref_pos], np.arange(n))


def test_dynamic_schedule_write_path_parity():
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=3000, stride=10, alpha=0.05, n_sink=4)
    _parity(cfg, n_sample=120, all_idx=True)
    cfg = C["long-131k-fp8ref"].replace(T=5000, stride=12, alpha=0.02)
    _parity(cfg, n_sample=80, all_idx=True)


def test_constant_group_and_ties():
    # token 3 is a copy of reference 0 (its only pool member): z = 0 exactly and
    # every group is constant; references 5, 6, 7 duplicate reference 4, so the
    # lower slots win the ties.
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=512, N=2, D=64, d_ff=256, d_c=64)
    kv, w = gen_inputs(cfg)
    kv[0] = kv[0].copy()
    kv[0][0, 3] = kv[0][0, 0]
    for s in (5, 6, 7):
        kv[0][0, 8 * s] = kv[0][0, 32]
    kv[0][0, 300] = kv[0][0, 32]
    bufs, _ = run_gpu(cfg, kv, w)
    gpu = host_records(cfg, bufs)
    assert np.all(gpu["z"][0, 3] == 0) and np.all(gpu["hdr"][0, 3] == 0) and np.all(gpu["q"][0, 3] == 0)
    assert gpu["idx"][0, 300].tolist() == [4, 5, 6, 7]
    check_all_indices(cfg, kv[0][0], gpu["idx"][0])
    check_tokens(cfg, kv[0][0], w[0], gpu, 0, np.array([3, 300, 301]))


def test_many_tied_references_take_the_block_scan():
    # references 4..15 are identical and token 300 sits on them: all eight expansion
    # candidates tie, so the top-k is settled by the exact block scan (lowest slots win)
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=640, N=2, D=64, d_ff=256, d_c=64)
    kv, w = gen_inputs(cfg)
    kv[0] = kv[0].copy()
    for s in range(5, 16):
        kv[0][0, 8 * s] = kv[0][0, 32]
    kv[0][0, 300] = kv[0][0, 32]
    kv[0][0, 301] = kv[0][0, 32] ^ np.uint16(1)        # one bit away from the cluster
    bufs, _ = run_gpu(cfg, kv, w)
    gpu = host_records(cfg, bufs)
    assert gpu["idx"][0, 300].tolist() == [4, 5, 6, 7]
    check_all_indices(cfg, kv[0][0], gpu["idx"][0])
    check_tokens(cfg, kv[0][0], w[0], gpu, 0, np.array([300, 301, 302, 639]))


def test_records_requantise_bit_exactly_from_gpu_z():
    # the kernels' own quantisation decision, repeated on the host in fp32 with the
    # same operations, reproduces every code and group header bit for bit
    cfg = SMALL["llama-2x1000"]
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w)
    gpu = host_records(cfg, bufs)
    z = gpu["z"].reshape(-1, cfg.d_c // 32, 32).astype(np.float32)
    lo, hi = z.min(-1), z.max(-1)
    qmax = np.float32((1 << cfg.bits) - 1)
    with np.errstate(divide="ignore", invalid="ignore"):
        dl = (hi - lo) / qmax
        u = (z - lo[..., None]) / dl[..., None] + np.float32(0.5)
    q = np.clip(np.floor(u), 0, qmax)
    q = np.where((hi == lo)[..., None], 0, q).astype(np.uint8)
    dl = np.where(hi == lo, np.float32(0), dl)
    assert np.array_equal(q.reshape(gpu["q"].shape), gpu["q"])
    hdr = gpu["hdr"].reshape(-1, cfg.d_c // 32, 2)
    assert np.array_equal(hdr[..., 0], lo) and np.array_equal(hdr[..., 1], dl)


# ------------------------------------------------------------------ read path
def _oracle_read(cfg, kv_seq, gpu, lb, sel):
    """The oracle's read [RKV §2.7] over the GPU's own records of one (layer,
    sequence): dequantised codes and reference means of the tokens in `sel`."""
    refs64, _ = oracle.stored_refs(cfg, kv_seq, oracle.schedule(cfg))
    G = cfg.d_c // 32
    return oracle.gather(cfg, refs64, gpu["q"][lb], gpu["hdr"][lb][..., 0].reshape(-1, G),
                         gpu["hdr"][lb][..., 1].reshape(-1, G), gpu["idx"][lb], sel), refs64


def _check_read(cfg, kv_seq, gpu, lb, sel, gz, gm, out):
    """GPU read outputs against the oracle's read of the same records, element by
    element: one rounding to the output type (z~ = q*delta + z_min is one fused
    multiply-add in fp32; the mean is an fp32 sum of at most k stored references,
    off the exact sum by at most k * 2^-24 * max |r|)."""
    (zq, mn), refs64 = _oracle_read(cfg, kv_seq, gpu, lb, sel)
    ulp = 2.0 ** -23 if out == "f32" else 2.0 ** -8
    np.testing.assert_allclose(gz, zq, rtol=ulp, atol=1e-30)
    atol = cfg.k * 2.0 ** -24 * float(np.abs(refs64).max(initial=1.0))
    np.testing.assert_allclose(gm, mn, rtol=ulp, atol=atol)


@pytest.mark.parametrize("name,out", [("tiny-fp32", "f32"), ("llama-2x1000", "bf16"),
                                      ("long-fp8-1x1500", "bf16"), ("mm-int2-2x4096", "bf16")])
def test_gather_matches_oracle_read(name, out):
    cfg = C[name] if name in C else SMALL[name]
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w)
    gpu = host_records(cfg, bufs)
    LB = cfg.L * cfg.B
    sels = [np.sort(np.random.default_rng(lb).choice(cfg.T, size=min(300, cfg.T), replace=False))
            for lb in range(LB)]
    n_sel = len(sels[0])
    sel = torch.tensor(np.stack(sels), dtype=torch.int32, device="cuda")
    odt = torch.float32 if out == "f32" else torch.bfloat16
    out_z = out_buffer((LB, n_sel, cfg.d_c), odt)
    out_m = out_buffer((LB, n_sel, cfg.W), odt)
    bufs.gather(sel, out_z, out_m)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    assert_guards(bufs)
    gz = out_z.float().cpu().numpy()
    gm = out_m.float().cpu().numpy()
    for lb in range(LB):
        l, b = divmod(lb, cfg.B)
        _check_read(cfg, kv[l][b], gpu, lb, sels[lb], gz[lb], gm[lb], out)
        # and the records' means are the oracle write path's means wherever the
        # reference sets agree (they differ only inside the tie band, checked above)
        toks = sels[lb][:80]
        o = oracle.compress_tokens(cfg, kv[l][b], w[l], toks, want_mean=True)
        same = np.all(gpu["idx"][lb][toks][:, : cfg.k] == o["idx"], axis=1)
        np.testing.assert_allclose(gm[lb][:80][same], o["mean"][same], rtol=2.0 ** -8 if out != "f32" else 2.0 ** -23,
                                   atol=1e-6)


@pytest.mark.parametrize("name", ["long-fp8-1x1500", "llama-2x1000", "tiny-fp32"])
def test_pool_bytes_and_norms_match_oracle(name):
    # the stored pool is the oracle's storage round trip bit for bit (FP8 E4M3 codes
    # from the oracle's own RNE encoder [RKV §2.4 = Sec. V-A]; bf16 / fp32 rows
    # copied), and ||r||^2 is the squared norm of the stored reference to fp32
    # accumulation error (a dropped coordinate would be ~1/W off)
    cfg = C[name] if name in C else SMALL[name]
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w, want_z=False)
    ref_pos = oracle.schedule(cfg)
    n = ref_pos.size
    assert bufs.n_ref == n
    assert np.array_equal(bufs.ref_pos.cpu().numpy()[:n], ref_pos)
    vec = bufs.ref_vec.cpu()
    if cfg.ref_dtype == "fp8":
        got = vec.view(torch.uint8).numpy()
    elif cfg.kv_dtype == "bf16":
        got = vec.view(torch.int16).numpy().view(np.uint16)
    else:
        got = vec.numpy()
    got = got.reshape(cfg.L * cfg.B, -1, cfg.W)
    sq = bufs.ref_sqnorm.cpu().numpy().reshape(cfg.L * cfg.B, -1)
    for l in range(cfg.L):
        for b in range(cfg.B):
            lb = l * cfg.B + b
            refs64, stored = oracle.stored_refs(cfg, kv[l][b], ref_pos)
            exp = np.asarray(stored)
            if cfg.ref_dtype != "fp8" and cfg.kv_dtype == "bf16":
                exp = exp.view(np.uint16)
            assert np.array_equal(got[lb][:n], exp.reshape(n, cfg.W)), "stored reference bytes differ"
            norm = np.sum(refs64 * refs64, axis=1)
            np.testing.assert_allclose(sq[lb][:n], norm, rtol=64 * 2.0 ** -24, atol=0)


def test_gather_standalone_padding_and_isolation():
    cfg = SMALL["long-fp8-1x1500"]
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w)
    T = cfg.T
    # standalone mode (every token) equals the union of sparse reads
    allsel = torch.arange(T, dtype=torch.int32, device="cuda").view(1, T)
    za = out_buffer((1, T, cfg.d_c), torch.bfloat16)
    ma = out_buffer((1, T, cfg.W), torch.bfloat16)
    bufs.gather(allsel, za, ma)
    sel_np = wl.gather_selection(cfg, 0)
    sel = torch.tensor(np.concatenate([sel_np, [-1, -1, -1]]), dtype=torch.int32, device="cuda").view(1, -1)
    zs = out_buffer((1, sel.shape[1], cfg.d_c), torch.bfloat16)
    ms = out_buffer((1, sel.shape[1], cfg.W), torch.bfloat16)
    bufs.gather(sel, zs, ms)
    torch.cuda.synchronize()
    idx = torch.tensor(sel_np, device="cuda", dtype=torch.long)
    assert torch.equal(zs[0, : len(sel_np)], za[0, idx]) and torch.equal(ms[0, : len(sel_np)], ma[0, idx])
    assert torch.all(zs[0, len(sel_np):] == 0) and torch.all(ms[0, len(sel_np):] == 0)
    # poison every record the selection does not name: the read must not change
    other = torch.ones(T, dtype=torch.bool, device="cuda")
    other[idx] = False
    bufs.codes[0, other] = 0xFF
    bufs.hdr[0, other] = float("nan")
    bufs.ref_idx[0, other] = 1 << 30
    zp, mp = out_buffer(zs.shape, zs.dtype), out_buffer(ms.shape, ms.dtype)
    bufs.gather(sel, zp, mp)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    assert torch.equal(zp, zs) and torch.equal(mp, ms)
    assert_guards(bufs)


@pytest.mark.parametrize("name", ["tiny-fp32", "long-fp8-1x1500"])
def test_gather_out_of_range_index_is_reported_not_faulted(name):
    cfg = C[name] if name in C else SMALL[name]
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w)
    sel = torch.tensor([[0, 5, cfg.T, 7]], dtype=torch.int32, device="cuda")
    oz = torch.full((1, 4, cfg.d_c), 9.0, device="cuda")
    om = torch.full((1, 4, cfg.W), 9.0, device="cuda")
    bufs.gather(sel, oz, om)
    torch.cuda.synchronize()
    assert bufs.device_status() == rkv.RKV_ERR_INDEX
    assert torch.all(oz[0, 2] == 0) and torch.all(om[0, 2] == 0)
    assert torch.all(om[0, 0] != 9.0)
    # an empty selection launches nothing
    bufs.status.zero_()
    rkv.rkv_gather_dequant(bufs.p, bufs.pool, bufs.cache, None, 0, None, None, rkv.RKV_F32, None)


def test_long_context_decode_steps():
    # the long-context workload's read side: several decode steps of 30% random
    # tokens plus the last 512, element by element against the oracle's read of the
    # GPU's records on sampled selected tokens
    cfg = C["long-131k-fp8ref"]
    kv, w = gen_inputs(cfg)
    bufs, _ = run_gpu(cfg, kv, w, want_z=False)
    gpu = host_records(cfg, bufs)
    for step in range(3):
        s = wl.gather_selection(cfg, step)
        sel = torch.tensor(s, dtype=torch.int32, device="cuda").view(1, -1)
        oz = out_buffer((1, s.size, cfg.d_c), torch.bfloat16)
        om = out_buffer((1, s.size, cfg.W), torch.bfloat16)
        bufs.gather(sel, oz, om)
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        assert_guards(bufs)
        pick = np.sort(np.concatenate([np.random.default_rng(step).choice(s.size - 512, 40, replace=False),
                                       s.size - 1 - np.arange(8)]))
        _check_read(cfg, kv[0][0], gpu, 0, s[pick], oz[0, pick].float().cpu().numpy(),
                    om[0, pick].float().cpu().numpy(), "bf16")
