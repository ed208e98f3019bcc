"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs, unpack its records, and compare them with the fp64 oracle under the
tolerances of the write path:
  * reference indices bit-exact, except tokens whose oracle k-th and (k+1)-th
    distances lie within 1e-5 relative (then the GPU set must still be a valid
    nearest set within that band);
  * z within 2e-2 of the token's max |z| (floored at 1e-3 of the largest |z| among
    the checked tokens), all scales taken from the oracle's z;
  * group minima within the same per-token tolerance, group steps within
    2 * 2e-2 * scale / (2^b - 1);
  * codes equal except +-1 on at most 0.1% of coordinates, and only where the
    oracle's (z - z_min)/delta lies within the z discrepancy of a rounding boundary.
"""
from __future__ import annotations

import concurrent.futures as cf
import math

import numpy as np
import torch

import oracle
import rkv_workload as wl
from reference_residual_kv_gb300 import build, rkv

TIE_BAND = 1e-5
Z_TOL = 2e-2
CODE_BUDGET = 1e-3


def ensure_lib():
    build.build()
    rkv.lib()


def gen_inputs(cfg: wl.Config, layers=None):
    """Stored kv [L][B][T][W] and weights (lists per layer), generated in threads."""
    layers = list(range(cfg.L)) if layers is None else layers
    with cf.ThreadPoolExecutor(max_workers=min(16, len(layers))) as ex:
        kv = list(ex.map(lambda l: wl.layer_kv(cfg, l), layers))
        w = list(ex.map(lambda l: wl.layer_weights(cfg, l), layers))
    return kv, w


def to_device(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


# Guard bytes after every device buffer the GPU tests hand to the library: a write past a
# buffer's end changes them (checked by assert_guards and Buffers.guard_violations).
GUARD = 4096
_guarded = []


def out_buffer(shape, dtype):
    """An uninitialised device output tensor followed by GUARD guard bytes."""
    t, raw = rkv.guarded_empty(tuple(shape), dtype, "cuda", GUARD)
    _guarded.append((t, raw))
    return t


def assert_guards(*bufs):
    """Every out_buffer since the last call, and every given Buffers, still has intact
    guard bytes."""
    torch.cuda.synchronize()
    bad = [i for i, (t, raw) in enumerate(_guarded) if not rkv.guard_intact(t, raw)]
    _guarded.clear()
    assert not bad, "writes past the end of output buffers %s" % bad
    for b in bufs:
        v = b.guard_violations()
        assert not v, "writes past the end of %s" % v


def run_gpu(cfg: wl.Config, kv, w, want_z=True):
    """Build pool + compress through the C ABI; returns (Buffers, device inputs)."""
    ensure_lib()
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p, want_z=want_z, guard=GUARD)
    kv_d = to_device(np.stack(kv), cfg.kv_dtype)
    W1 = to_device(np.stack([x[0] for x in w]), cfg.kv_dtype)
    W2 = to_device(np.stack([x[1] for x in w]), cfg.kv_dtype)
    W3 = to_device(np.stack([x[2] for x in w]), cfg.kv_dtype)
    bufs.build_ref_pool(kv_d)
    bufs.compress(kv_d, W1, W2, W3)
    torch.cuda.synchronize()
    assert_guards(bufs)
    return bufs, (kv_d, W1, W2, W3)


def unpack_codes(codes: np.ndarray, bits: int, d_c: int) -> np.ndarray:
    c = codes.astype(np.uint8)
    if bits == 4:
        q = np.stack([c & 15, c >> 4], axis=-1)
    else:
        q = np.stack([(c >> (2 * i)) & 3 for i in range(4)], axis=-1)
    return q.reshape(*codes.shape[:-1], d_c)


def host_records(cfg, bufs):
    """GPU records as numpy: ref_idx [LB][T][4], q [LB][T][d_c], hdr [LB][T][G][2], z."""
    out = dict(idx=bufs.ref_idx.cpu().numpy(), hdr=bufs.hdr.cpu().numpy(),
               q=unpack_codes(bufs.codes.cpu().numpy(), cfg.bits, cfg.d_c))
    if bufs.z is not None:
        out["z"] = bufs.z.cpu().numpy()
    return out


def check_tokens(cfg, kv_seq, w_layer, gpu, lb, tokens, report=None):
    """Compare one (layer, sequence)'s GPU records for `tokens` with the oracle.

    Every tolerance input comes from the oracle: a token's z scale is the oracle's
    max |z| of that token, floored at 1e-3 of the largest oracle |z| among the checked
    tokens.  Per token: z within Z_TOL of its scale; each group's z_min within the
    same; each group's step within 2 Z_TOL scale / (2^b - 1) (max and min each move by
    at most the z tolerance).  Tokens whose GPU reference set differs inside the
    1e-5 tie band are compared with the oracle run on the GPU's set (forced-index
    mode), so no token leaves the check."""
    tokens = np.asarray(tokens, dtype=np.int32)
    o = oracle.compress_tokens(cfg, kv_seq, w_layer, tokens)
    ref_pos = oracle.schedule(cfg)
    gidx = gpu["idx"][lb][tokens][:, : cfg.k]
    exempt = np.zeros(tokens.size, bool)
    mism = np.nonzero(np.any(gidx != o["idx"], axis=1))[0]
    refs64 = None
    for n in mism:
        dk, dk1 = o["dk"][n]
        assert dk1 - dk <= TIE_BAND * max(dk, 1e-300), (
            "token %d: GPU refs %s, oracle %s, gap %.3g (d_k %.6g)" % (tokens[n], gidx[n], o["idx"][n], dk1 - dk, dk))
        if refs64 is None:
            refs64, _ = oracle.stored_refs(cfg, kv_seq, ref_pos)
        x = wl.stored_to_f64(kv_seq[tokens[n]], cfg.kv_dtype)
        for s in gidx[n][gidx[n] >= 0]:
            assert oracle.sqdist(x, refs64[s]) <= dk * (1 + TIE_BAND) + 1e-300
        exempt[n] = True
    if exempt.any():
        # the GPU's equally near set, encoded by the oracle
        f = oracle.compress_tokens(cfg, kv_seq, w_layer, tokens[exempt], forced_idx=gidx[exempt])
        for key in ("z", "q", "zmin", "delta"):
            o[key][exempt] = f[key]
    zo = o["z"]
    zg = gpu["z"][lb][tokens] if "z" in gpu else None
    zabs = np.abs(zo).max(axis=1, initial=0.0)
    zscale = np.maximum(zabs, 1e-3 * zabs.max(initial=0.0))
    tol = Z_TOL * zscale
    if zg is not None:
        err = np.abs(zg - zo).max(axis=1, initial=0.0)
        bad = err > tol
        assert not bad.any(), "z mismatch at tokens %s: err %s scale %s" % (
            tokens[bad][:5], err[bad][:5], zscale[bad][:5])
    # group headers {z_min, step}, per token
    qmax = (1 << cfg.bits) - 1
    hdr = gpu["hdr"][lb][tokens]
    dmin = np.abs(hdr[..., 0] - o["zmin"])
    ddl = np.abs(hdr[..., 1] - o["delta"])
    bad = np.any(dmin > tol[:, None], axis=1)
    assert not bad.any(), "z_min mismatch at tokens %s: %s > %s" % (
        tokens[bad][:5], dmin[bad].max(axis=1)[:5], tol[bad][:5])
    bad = np.any(ddl > 2.0 * tol[:, None] / qmax, axis=1)
    assert not bad.any(), "group step mismatch at tokens %s: %s > %s" % (
        tokens[bad][:5], ddl[bad].max(axis=1)[:5], 2.0 * tol[bad][:5] / qmax)
    # codes: +-1 only near a rounding boundary
    qg = gpu["q"][lb][tokens].astype(int)
    qo = o["q"].astype(int)
    diff = qg != qo
    n_diff = int(diff.sum())
    if n_diff:
        assert np.all(np.abs(qg - qo)[diff] == 1), "code differs by more than 1"
        rows, cols = np.nonzero(diff)
        g = cols // 32
        dl_o = o["delta"][rows, g]
        mn_o = o["zmin"][rows, g]
        u = (zo[rows, cols] - mn_o) / dl_o
        frac = u - np.floor(u)
        if zg is not None:
            dz = np.abs(zg[rows, cols] - zo[rows, cols])
        else:
            dz = tol[rows]
        slack = (dz + dmin[rows, g] + qo[rows, cols] * ddl[rows, g]) / dl_o + 1e-6
        assert np.all(np.abs(frac - 0.5) <= slack), "code flip away from a rounding boundary"
    if report is not None:
        report["coords"] = report.get("coords", 0) + int(qo.size)
        report["flips"] = report.get("flips", 0) + n_diff
        report["exempt"] = report.get("exempt", 0) + int(exempt.sum())
        report["tokens"] = report.get("tokens", 0) + int(tokens.size)
        if zg is not None and zo.size:
            rel = (np.abs(zg - zo).max(axis=1) / np.maximum(zscale, 1e-30)).max()
            report["max_rel_z"] = max(report.get("max_rel_z", 0.0), float(rel))
    return o


def check_all_indices(cfg, kv_seq, gpu_idx_seq, tokens=None, report=None):
    """Reference sets of `tokens` (default: every token) against the oracle's retrieval."""
    tokens = np.arange(cfg.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    idx, ki, dk = oracle.retrieve_tokens(cfg, kv_seq, tokens)
    g = gpu_idx_seq[tokens][:, : cfg.k]
    assert np.all(gpu_idx_seq[tokens][:, cfg.k:] == -1)
    bad = np.nonzero(np.any(g != idx, axis=1))[0]
    for n in bad:
        assert dk[n, 1] - dk[n, 0] <= TIE_BAND * max(dk[n, 0], 1e-300), (
            "token %d: GPU %s oracle %s (d_k %.8g, d_k+1 %.8g)" % (tokens[n], g[n], idx[n], dk[n, 0], dk[n, 1]))
    if report is not None:
        report["idx_exempt"] = report.get("idx_exempt", 0) + int(bad.size)
        report["idx_tokens"] = report.get("idx_tokens", 0) + int(tokens.size)
    return int(bad.size)


def sample_tokens(cfg, n, seed):
    """Edge tokens (first few, tile boundaries, last ones) plus a random sample."""
    T = cfg.T
    edge = [t for t in (1, 2, 3, 7, 9, 15, 17, 31, 33, 63, 127, 129, 255, 257, T - 2, T - 1) if 0 <= t < T]
    rng = np.random.default_rng(seed)
    rest = rng.choice(T, size=min(n, T), replace=False)
    return np.unique(np.concatenate([edge, rest])).astype(np.int32)
