"""fp64 oracle of the ResidualKV write and read path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (the C-ABI library and its binding) never
loads it.  The arithmetic lives in ``rkv_oracle.c`` (plain C, fp64, single thread);
this file compiles it with gcc, decodes stored inputs (fp32 / bf16 bit patterns) to
float64 exactly, and marshals arrays through ctypes.

Every function is pinned by tests in ``tests/test_oracle_*.py`` (brute force, closed
forms, library routines, the paper's identities and worked numbers).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

import rkv_workload as wl

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rkv_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "librkv_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_up = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, no fast-math) into oracle/_lib."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        # RKV_ORACLE_LIB lets the mutation test load a deliberately broken copy
        alt = os.environ.get("RKV_ORACLE_LIB")
        _lib = ctypes.CDLL(alt if alt else build())
        L = _lib
        L.rkvo_fixed_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip]
        L.rkvo_fixed_schedule.restype = ctypes.c_int
        L.rkvo_dynamic_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                            ctypes.c_int, _ip, ctypes.c_int]
        L.rkvo_dynamic_schedule.restype = ctypes.c_int
        L.rkvo_fp8_decode.argtypes = [ctypes.c_uint8]
        L.rkvo_fp8_decode.restype = ctypes.c_double
        L.rkvo_fp8_encode.argtypes = [ctypes.c_double]
        L.rkvo_fp8_encode.restype = ctypes.c_uint8
        L.rkvo_sqdist.argtypes = [_dp, _dp, ctypes.c_int]
        L.rkvo_sqdist.restype = ctypes.c_double
        L.rkvo_retrieve.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, _dp]
        L.rkvo_retrieve.restype = ctypes.c_int
        L.rkvo_mean.argtypes = [_dp, _ip, ctypes.c_int, ctypes.c_int, _dp]
        L.rkvo_mean.restype = None
        L.rkvo_swish.argtypes = [ctypes.c_double]
        L.rkvo_swish.restype = ctypes.c_double
        L.rkvo_fc.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp]
        L.rkvo_fc.restype = None
        L.rkvo_quantize.argtypes = [_dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _up, _dp, _dp]
        L.rkvo_quantize.restype = None
        L.rkvo_dequantize.argtypes = [_up, _dp, _dp, ctypes.c_int, ctypes.c_int, _dp]
        L.rkvo_dequantize.restype = None
        L.rkvo_compress_tokens.argtypes = (
            [ctypes.c_int] * 7 + [_dp, _dp, _ip, ctypes.c_int, _dp, _dp, _dp, _ip, ctypes.c_int, _ip,
                                  _ip, _ip, _dp, _dp, _up, _dp, _dp, _dp])
        L.rkvo_compress_tokens.restype = None
        L.rkvo_retrieve_tokens.argtypes = ([ctypes.c_int] * 2 + [_dp, _dp, _ip, ctypes.c_int, _ip,
                                                                ctypes.c_int, _ip, _ip, _dp])
        L.rkvo_retrieve_tokens.restype = None
        L.rkvo_gather.argtypes = ([ctypes.c_int] * 4 + [_dp, _up, _dp, _dp, _ip, _ip, ctypes.c_int, _dp, _dp])
        L.rkvo_gather.restype = None
    return _lib


def _d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(_dp)


def _i(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_ip)


def _u(a):
    a = np.ascontiguousarray(a, dtype=np.uint8)
    return a, a.ctypes.data_as(_up)


def _null(t):
    return ctypes.cast(None, t)


# --- single functions -------------------------------------------------------------
def fixed_schedule(T: int, stride: int, first: int = 0) -> np.ndarray:
    out = np.zeros(max(T, 1), dtype=np.int32)
    n = lib().rkvo_fixed_schedule(T, stride, first, out.ctypes.data_as(_ip))
    return out[:n].copy()


def dynamic_schedule(T: int, s0: int, alpha: float, n_sink: int = 0, first: int = 0) -> np.ndarray:
    out = np.zeros(max(T, 1), dtype=np.int32)
    n = lib().rkvo_dynamic_schedule(T, s0, float(alpha), n_sink, first, out.ctypes.data_as(_ip), T)
    return out[:n].copy()


def fp8_decode(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    f = lib().rkvo_fp8_decode
    return np.array([f(int(v)) for v in b.ravel()], dtype=np.float64).reshape(b.shape)


def fp8_encode(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    f = lib().rkvo_fp8_encode
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def sqdist(x, r) -> float:
    x, px = _d(x)
    r, pr = _d(r)
    return lib().rkvo_sqdist(px, pr, x.size)


def retrieve(x, refs, k: int):
    """Returns (idx[k] ascending, -1 padded, k_i, (d_k, d_{k+1}))."""
    x, px = _d(x)
    refs, pr = _d(np.asarray(refs).reshape(-1, x.size) if np.size(refs) else np.zeros((0, x.size)))
    idx = np.zeros(k, dtype=np.int32)
    dk = np.zeros(2)
    ki = lib().rkvo_retrieve(px, pr, refs.shape[0], x.size, k, idx.ctypes.data_as(_ip),
                             dk.ctypes.data_as(_dp))
    return idx, ki, (dk[0], dk[1])


def mean(refs, idx) -> np.ndarray:
    refs, pr = _d(refs)
    idx = np.asarray(idx, dtype=np.int32)
    ki = int((idx >= 0).sum())
    idx, pi = _i(idx)
    out = np.zeros(refs.shape[1])
    lib().rkvo_mean(pr, pi, ki, refs.shape[1], out.ctypes.data_as(_dp))
    return out


def swish(u: float) -> float:
    return lib().rkvo_swish(float(u))


def fc(x, W1t, W2t, W3t, return_h: bool = False):
    x, px = _d(x)
    W1t, p1 = _d(W1t)
    W2t, p2 = _d(W2t)
    W3t, p3 = _d(W3t)
    d_ff, W = W1t.shape
    d_c = W3t.shape[0]
    out = np.zeros(d_c)
    h = np.zeros(d_ff)
    lib().rkvo_fc(px, p1, p2, p3, W, d_ff, d_c, out.ctypes.data_as(_dp), h.ctypes.data_as(_dp))
    return (out, h) if return_h else out


def quantize(z, group: int, bits: int):
    z, pz = _d(z)
    d_c = z.size
    ng = (d_c + group - 1) // group
    q = np.zeros(d_c, dtype=np.uint8)
    zmin = np.zeros(ng)
    delta = np.zeros(ng)
    lib().rkvo_quantize(pz, d_c, group, bits, q.ctypes.data_as(_up), zmin.ctypes.data_as(_dp),
                        delta.ctypes.data_as(_dp))
    return q, zmin, delta


def dequantize(q, zmin, delta, group: int) -> np.ndarray:
    q, pq = _u(q)
    zmin, pm = _d(zmin)
    delta, pd = _d(delta)
    out = np.zeros(q.size)
    lib().rkvo_dequantize(pq, pm, pd, q.size, group, out.ctypes.data_as(_dp))
    return out


# --- per-sequence drivers -----------------------------------------------------------
def schedule(cfg: wl.Config) -> np.ndarray:
    if getattr(cfg, "alpha", 0.0) > 0.0:
        return dynamic_schedule(cfg.T, cfg.stride, cfg.alpha, cfg.n_sink, cfg.first)
    return fixed_schedule(cfg.T, cfg.stride, cfg.first)


def stored_refs(cfg: wl.Config, kv_seq: np.ndarray, ref_pos: np.ndarray):
    """Reference vectors after the storage round trip, as float64 [n_ref][W], plus the
    stored bytes (FP8 codes for ref_dtype 'fp8', else the kv storage itself)."""
    rows = np.asarray(kv_seq)[ref_pos]
    v = wl.stored_to_f64(rows, cfg.kv_dtype)
    if cfg.ref_dtype == "fp8":
        codes = fp8_encode(v)
        return fp8_decode(codes), codes
    return v, rows


def weights_f64(cfg: wl.Config, w):
    return tuple(wl.stored_to_f64(a, cfg.kv_dtype) for a in w)


def compress_tokens(cfg: wl.Config, kv_seq, weights, tokens, forced_idx=None, want_mean=False,
                    kv64=None, refs64=None, ref_pos=None):
    """Write path for `tokens` of one (layer, sequence).  kv_seq: stored [T][W];
    weights: stored (W1t, W2t, W3t).  Returns a dict of numpy arrays."""
    if ref_pos is None:
        ref_pos = schedule(cfg)
    if kv64 is None:
        kv64 = wl.stored_to_f64(kv_seq, cfg.kv_dtype)
    if refs64 is None:
        refs64, _ = stored_refs(cfg, kv_seq, ref_pos)
    W1, W2, W3 = weights if weights[0].dtype == np.float64 else weights_f64(cfg, weights)
    tokens = np.asarray(tokens, dtype=np.int32)
    n, k, d_c, W = tokens.size, cfg.k, cfg.d_c, cfg.W
    ng = (d_c + cfg.group - 1) // cfg.group
    kv64, pkv = _d(kv64)
    refs64, prf = _d(refs64 if refs64.size else np.zeros((1, W)))
    ref_pos, ppos = _i(ref_pos)
    W1, p1 = _d(W1)
    W2, p2 = _d(W2)
    W3, p3 = _d(W3)
    tokens, ptok = _i(tokens)
    fi = _null(_ip)
    if forced_idx is not None:
        forced_idx, fi = _i(forced_idx)
    out = dict(idx=np.zeros((n, k), np.int32), ki=np.zeros(n, np.int32), dk=np.zeros((n, 2)),
               z=np.zeros((n, d_c)), q=np.zeros((n, d_c), np.uint8), zmin=np.zeros((n, ng)),
               delta=np.zeros((n, ng)))
    pm = _null(_dp)
    if want_mean:
        out["mean"] = np.zeros((n, W))
        pm = out["mean"].ctypes.data_as(_dp)
    lib().rkvo_compress_tokens(
        cfg.T, W, cfg.d_ff, d_c, k, cfg.group, cfg.bits, pkv, prf, ppos, ref_pos.size, p1, p2, p3,
        ptok, n, fi, out["idx"].ctypes.data_as(_ip), out["ki"].ctypes.data_as(_ip),
        out["dk"].ctypes.data_as(_dp), out["z"].ctypes.data_as(_dp), out["q"].ctypes.data_as(_up),
        out["zmin"].ctypes.data_as(_dp), out["delta"].ctypes.data_as(_dp), pm)
    return out


def gather(cfg: wl.Config, refs64, q, zmin, delta, idx, sel):
    """Read path over records [T][...] of one sequence for the index list `sel`."""
    refs64, prf = _d(refs64)
    q, pq = _u(q)
    zmin, pmn = _d(zmin)
    delta, pdl = _d(delta)
    idx, pidx = _i(idx)
    sel, psel = _i(sel)
    n = sel.size
    zq = np.zeros((n, cfg.d_c))
    mn = np.zeros((n, cfg.W))
    lib().rkvo_gather(cfg.W, cfg.d_c, cfg.group, cfg.k, prf, pq, pmn, pdl, pidx, psel, n,
                      zq.ctypes.data_as(_dp), mn.ctypes.data_as(_dp))
    return zq, mn


def retrieve_tokens(cfg: wl.Config, kv_seq, tokens, kv64=None, refs64=None, ref_pos=None):
    """Reference sets of `tokens` of one (layer, sequence): (idx [n][k], k_i [n], dk [n][2])."""
    if ref_pos is None:
        ref_pos = schedule(cfg)
    if kv64 is None:
        kv64 = wl.stored_to_f64(kv_seq, cfg.kv_dtype)
    if refs64 is None:
        refs64, _ = stored_refs(cfg, kv_seq, ref_pos)
    tokens = np.asarray(tokens, dtype=np.int32)
    n = tokens.size
    kv64, pkv = _d(kv64)
    refs64, prf = _d(refs64 if refs64.size else np.zeros((1, cfg.W)))
    ref_pos, ppos = _i(ref_pos)
    tokens, ptok = _i(tokens)
    idx = np.zeros((n, cfg.k), np.int32)
    ki = np.zeros(n, np.int32)
    dk = np.zeros((n, 2))
    lib().rkvo_retrieve_tokens(cfg.W, cfg.k, pkv, prf, ppos, ref_pos.size, ptok, n,
                               idx.ctypes.data_as(_ip), ki.ctypes.data_as(_ip), dk.ctypes.data_as(_dp))
    return idx, ki, dk


def rope(x, pos: float, base: float) -> np.ndarray:
    """Rotary embedding of one head vector x [D] at position pos (consecutive pairs)."""
    x = np.array(x, dtype=np.float64)
    lib().rkvo_rope(x.ctypes.data_as(_dp), x.size, ctypes.c_double(pos), ctypes.c_double(base))
    return x


def decode(z, Wd) -> np.ndarray:
    """Linear decoder f_d(z) = z W_d with Wd stored out-major [W][d_c]."""
    z, pz = _d(z)
    Wd, pw = _d(Wd)
    out = np.zeros(Wd.shape[0])
    lib().rkvo_decode(pz, pw, z.size, Wd.shape[0], out.ctypes.data_as(_dp))
    return out


def restore(cfg: wl.Config, refs64, q, zmin, delta, idx, Wd64, sel):
    """Restored K^, V^ [n_sel][N*D] of the selected tokens of one sequence (K^ rotated at
    each token's position), from records [T][...] and the decoder weights [W][d_c]."""
    refs64, prf = _d(refs64)
    q, pq = _u(q)
    zmin, pmn = _d(zmin)
    delta, pdl = _d(delta)
    idx, pidx = _i(idx)
    Wd64, pw = _d(Wd64)
    sel, psel = _i(sel)
    n = sel.size
    ko = np.zeros((n, cfg.N * cfg.D))
    vo = np.zeros((n, cfg.N * cfg.D))
    lib().rkvo_restore(cfg.N, cfg.D, cfg.d_c, cfg.group, cfg.k, ctypes.c_double(cfg.rope_base),
                       prf, pq, pmn, pdl, pidx, pw, psel, n, ko.ctypes.data_as(_dp),
                       vo.ctypes.data_as(_dp))
    return ko, vo


def attention(q, K, V, N: int, valid=None) -> np.ndarray:
    """Sparse attention of one decode step: q [H][D], K/V [n][N*D] -> o [H][D]."""
    q, pq = _d(q)
    K, pk = _d(K)
    V, pv = _d(V)
    H, D = q.shape
    n = K.shape[0]
    if valid is None:
        valid = np.ones(n, np.int32)
    valid, pva = _i(np.asarray(valid, np.int32))
    o = np.zeros((H, D))
    lib().rkvo_attention(H, N, D, pq, pk, pv, pva, n, o.ctypes.data_as(_dp))
    return o
