"""Python binding of librkv: the same entry points as include/rkv.h, argument
marshalling only.  Every step of the path runs in the library's CUDA kernels; torch
only allocates device memory and supplies streams.  There is no fallback: if
librkv.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "librkv.so")
_lib = None

RKV_F32, RKV_BF16, RKV_FP8_E4M3 = 0, 1, 2
RKV_OK, RKV_ERR_INVALID_ARG, RKV_ERR_UNSUPPORTED, RKV_ERR_ALIGNMENT = 0, 1, 2, 3
RKV_ERR_CUDA, RKV_ERR_INDEX, RKV_ERR_DEVICE_TIMEOUT, RKV_ERR_WORKSPACE = 4, 5, 6, 7
EXPORTED = ("rkv_n_ref", "rkv_query_sizes", "rkv_build_ref_pool", "rkv_compress",
            "rkv_gather_dequant", "rkv_restore_kv", "rkv_attention_workspace", "rkv_sparse_attention",
            "rkv_append_token", "rkv_compress_noalloc", "rkv_profile_enable", "rkv_profile_collect",
            "rkv_debug_wait_fault", "rkv_status_string")
_DTYPES = {"f32": RKV_F32, "bf16": RKV_BF16, "fp8": RKV_FP8_E4M3}


class rkv_params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "L", "B", "T", "N", "D", "d_ff", "d_c", "k", "group", "bits", "kv_dtype", "ref_dtype",
        "stride", "first")] + [("alpha", ctypes.c_double), ("n_sink", ctypes.c_int32),
                               ("reserved", ctypes.c_int32)]


class rkv_ref_pool(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("ref_pos", "ref_slot", "pool_size", "ref_vec",
                                               "ref_sqnorm")]


class rkv_cache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("codes", "hdr", "ref_idx")]


class RkvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, rkv_status_string(code), code))


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load librkv.so (raises if it is absent: there is no other implementation)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("librkv.so is not built (%s); run "
                               "reference_residual_kv_gb300.build.build()" % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        P, V, I32 = ctypes.POINTER(rkv_params), ctypes.c_void_p, ctypes.c_int32
        sz = ctypes.POINTER(ctypes.c_size_t)
        L.rkv_n_ref.argtypes = [P]
        L.rkv_n_ref.restype = I32
        L.rkv_query_sizes.argtypes = [P, sz, sz, sz]
        L.rkv_query_sizes.restype = I32
        L.rkv_build_ref_pool.argtypes = [P, V, ctypes.POINTER(rkv_ref_pool), V]
        L.rkv_build_ref_pool.restype = I32
        L.rkv_compress.argtypes = [P, V, ctypes.POINTER(rkv_ref_pool), V, V, V,
                                   ctypes.POINTER(rkv_cache), V, ctypes.c_size_t, V, V, V]
        L.rkv_compress.restype = I32
        L.rkv_compress_noalloc.argtypes = [P, V, ctypes.POINTER(rkv_ref_pool), V, V, V,
                                           ctypes.POINTER(rkv_cache), V, V, V]
        L.rkv_compress_noalloc.restype = I32
        L.rkv_gather_dequant.argtypes = [P, ctypes.POINTER(rkv_ref_pool), ctypes.POINTER(rkv_cache),
                                         V, I32, V, V, I32, V, V]
        L.rkv_gather_dequant.restype = I32
        L.rkv_restore_kv.argtypes = [P, ctypes.POINTER(rkv_ref_pool), ctypes.POINTER(rkv_cache),
                                     V, V, I32, ctypes.c_double, V, V, V, V]
        L.rkv_restore_kv.restype = I32
        L.rkv_append_token.argtypes = [P, V, I32, ctypes.POINTER(rkv_ref_pool), V, V, V,
                                       ctypes.POINTER(rkv_cache), V, ctypes.c_size_t, V, V]
        L.rkv_append_token.restype = I32
        L.rkv_attention_workspace.argtypes = [P, I32, I32, sz]
        L.rkv_attention_workspace.restype = I32
        L.rkv_sparse_attention.argtypes = [P, I32, V, V, V, V, I32, V, V, ctypes.c_size_t, V]
        L.rkv_sparse_attention.restype = I32
        L.rkv_profile_enable.argtypes = [I32]
        L.rkv_profile_enable.restype = I32
        L.rkv_profile_collect.argtypes = [ctypes.c_char_p, I32, ctypes.POINTER(ctypes.c_float),
                                          ctypes.POINTER(I32), I32]
        L.rkv_profile_collect.restype = I32
        L.rkv_debug_wait_fault.argtypes = [ctypes.c_int64, I32]
        L.rkv_debug_wait_fault.restype = I32
        L.rkv_status_string.argtypes = [I32]
        L.rkv_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_params(L, B, T, N, D, d_ff, d_c, k=4, group=32, bits=4, kv_dtype="bf16",
                ref_dtype=None, stride=8, first=0, alpha=0.0, n_sink=0) -> rkv_params:
    kd = _DTYPES[kv_dtype] if isinstance(kv_dtype, str) else kv_dtype
    rd = kd if ref_dtype is None else (_DTYPES[ref_dtype] if isinstance(ref_dtype, str) else ref_dtype)
    return rkv_params(L, B, T, N, D, d_ff, d_c, k, group, bits, kd, rd, stride, first, float(alpha),
                      n_sink, 0)


def params_from_config(cfg) -> rkv_params:
    """rkv_params from a workload description with the same field names."""
    return make_params(cfg.L, cfg.B, cfg.T, cfg.N, cfg.D, cfg.d_ff, cfg.d_c, cfg.k, cfg.group,
                       cfg.bits, cfg.kv_dtype, cfg.ref_dtype, cfg.stride, cfg.first,
                       getattr(cfg, "alpha", 0.0), getattr(cfg, "n_sink", 0))


# ---- entry points (same names as the C ABI) -------------------------------------------
def rkv_status_string(code: int) -> str:
    return lib().rkv_status_string(int(code)).decode()


def rkv_n_ref(p: rkv_params) -> int:
    return lib().rkv_n_ref(ctypes.byref(p))


def rkv_query_sizes(p: rkv_params):
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    st = lib().rkv_query_sizes(ctypes.byref(p), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    if st:
        raise RkvError(st, "rkv_query_sizes")
    return a.value, b.value, c.value


def rkv_build_ref_pool(p: rkv_params, kv, pool: rkv_ref_pool, stream=None) -> None:
    st = lib().rkv_build_ref_pool(ctypes.byref(p), _ptr(kv), ctypes.byref(pool), _stream(stream))
    if st:
        raise RkvError(st, "rkv_build_ref_pool")


def rkv_compress(p: rkv_params, kv, pool: rkv_ref_pool, W1t, W2t, W3t, cache: rkv_cache,
                 workspace, workspace_bytes: int, z_out, dev_status, stream=None) -> None:
    st = lib().rkv_compress(ctypes.byref(p), _ptr(kv), ctypes.byref(pool), _ptr(W1t), _ptr(W2t),
                            _ptr(W3t), ctypes.byref(cache), _ptr(workspace), int(workspace_bytes),
                            _ptr(z_out), _ptr(dev_status), _stream(stream))
    if st:
        raise RkvError(st, "rkv_compress")


def rkv_compress_noalloc(p: rkv_params, kv, pool: rkv_ref_pool, W1t, W2t, W3t, cache: rkv_cache,
                         z_out, dev_status, stream=None) -> None:
    """rkv_compress with the library's built-in 64 MiB scratch instead of a workspace
    (for callers that cannot allocate device memory at the call)."""
    st = lib().rkv_compress_noalloc(ctypes.byref(p), _ptr(kv), ctypes.byref(pool), _ptr(W1t),
                                    _ptr(W2t), _ptr(W3t), ctypes.byref(cache), _ptr(z_out),
                                    _ptr(dev_status), _stream(stream))
    if st:
        raise RkvError(st, "rkv_compress_noalloc")


def rkv_gather_dequant(p: rkv_params, pool: rkv_ref_pool, cache: rkv_cache, sel, n_sel: int,
                       out_z, out_mean, out_dtype: int, dev_status, stream=None) -> None:
    st = lib().rkv_gather_dequant(ctypes.byref(p), ctypes.byref(pool), ctypes.byref(cache),
                                  _ptr(sel), int(n_sel), _ptr(out_z), _ptr(out_mean),
                                  int(out_dtype), _ptr(dev_status), _stream(stream))
    if st:
        raise RkvError(st, "rkv_gather_dequant")


def rkv_restore_kv(p: rkv_params, pool: rkv_ref_pool, cache: rkv_cache, Wd, sel, n_sel: int,
                   rope_base: float, out_k, out_v, dev_status, stream=None) -> None:
    st = lib().rkv_restore_kv(ctypes.byref(p), ctypes.byref(pool), ctypes.byref(cache), _ptr(Wd),
                              _ptr(sel), int(n_sel), float(rope_base), _ptr(out_k), _ptr(out_v),
                              _ptr(dev_status), _stream(stream))
    if st:
        raise RkvError(st, "rkv_restore_kv")


def rkv_append_token(p: rkv_params, kv_new, t: int, pool: rkv_ref_pool, W1t, W2t, W3t,
                     cache: rkv_cache, workspace, workspace_bytes: int, dev_status, stream=None) -> None:
    st = lib().rkv_append_token(ctypes.byref(p), _ptr(kv_new), int(t), ctypes.byref(pool), _ptr(W1t),
                                _ptr(W2t), _ptr(W3t), ctypes.byref(cache), _ptr(workspace),
                                int(workspace_bytes), _ptr(dev_status), _stream(stream))
    if st:
        raise RkvError(st, "rkv_append_token")


def rkv_attention_workspace(p: rkv_params, H: int, n_sel: int) -> int:
    b = ctypes.c_size_t()
    st = lib().rkv_attention_workspace(ctypes.byref(p), int(H), int(n_sel), ctypes.byref(b))
    if st:
        raise RkvError(st, "rkv_attention_workspace")
    return b.value


def rkv_sparse_attention(p: rkv_params, H: int, q, k_hat, v_hat, sel, n_sel: int, out, workspace,
                         workspace_bytes: int, stream=None) -> None:
    st = lib().rkv_sparse_attention(ctypes.byref(p), int(H), _ptr(q), _ptr(k_hat), _ptr(v_hat),
                                    _ptr(sel), int(n_sel), _ptr(out), _ptr(workspace),
                                    int(workspace_bytes), _stream(stream))
    if st:
        raise RkvError(st, "rkv_sparse_attention")


def rkv_debug_wait_fault(wait_cycles: int, skip_use: int) -> None:
    st = lib().rkv_debug_wait_fault(int(wait_cycles), int(skip_use))
    if st:
        raise RkvError(st, "rkv_debug_wait_fault")


def rkv_profile_enable(on: bool) -> None:
    lib().rkv_profile_enable(1 if on else 0)


def rkv_profile_collect(max_entries: int = 64, name_len: int = 48):
    """{kernel name: (total ms, launches)} since the last rkv_profile_enable(True)."""
    names = ctypes.create_string_buffer(max_entries * name_len)
    ms = (ctypes.c_float * max_entries)()
    cnt = (ctypes.c_int32 * max_entries)()
    n = lib().rkv_profile_collect(names, name_len, ms, cnt, max_entries)
    if n < 0:
        raise RkvError(RKV_ERR_CUDA, "rkv_profile_collect")
    raw = names.raw
    out = {}
    for i in range(n):
        nm = raw[i * name_len:(i + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (float(ms[i]), int(cnt[i]))
    return out


# ---- device buffers ----------------------------------------------------------------
_TORCH_REF = {RKV_F32: torch.float32, RKV_BF16: torch.bfloat16, RKV_FP8_E4M3: torch.uint8}


GUARD_BYTE = 0xA5


def guarded_empty(shape, dtype, device, guard: int, fill=None):
    """(tensor, raw): an uninitialised tensor of `shape` that is the head of a byte
    allocation followed by `guard` bytes of GUARD_BYTE (guard = 0: a plain allocation,
    raw is None).  A write past the tensor's end changes the tail (see guard_intact)."""
    if guard <= 0:
        t = torch.empty(shape, dtype=dtype, device=device)
        if fill is not None:
            t.fill_(fill)
        return t, None
    n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
    raw = torch.empty(n + guard, dtype=torch.uint8, device=device)
    raw[n:].fill_(GUARD_BYTE)
    t = raw[:n].view(dtype).view(shape)
    if fill is not None:
        t.fill_(fill)
    return t, raw


def guard_intact(t, raw) -> bool:
    if raw is None:
        return True
    n = t.numel() * t.element_size()
    return bool((raw[n:] == GUARD_BYTE).all().item())


class Buffers:
    """Caller-owned device buffers for one rkv_params: pool, cache, workspace, status.
    guard > 0 puts that many guard bytes after every buffer (test support: the tails are
    checked by guard_violations())."""

    def __init__(self, p: rkv_params, device="cuda", want_z: bool = False, guard: int = 0):
        self.p = p
        LB, T, W = p.L * p.B, p.T, 2 * p.N * p.D
        R = rkv_n_ref(p)
        if R < 0:
            raise RkvError(RKV_ERR_INVALID_ARG, "Buffers")
        self.n_ref = R
        _, _, ws = rkv_query_sizes(p)
        self.guard = guard
        self._raw = {}

        def alloc(name, shape, dtype, fill=None):
            t, raw = guarded_empty(shape, dtype, device, guard, fill)
            self._raw[name] = raw
            return t

        i32 = torch.int32
        self.ref_pos = alloc("ref_pos", (max(R, 1),), i32)
        self.ref_slot = alloc("ref_slot", (T,), i32)
        self.pool_size = alloc("pool_size", (T,), i32)
        self.ref_vec = alloc("ref_vec", (LB, max(R, 1), W), _TORCH_REF[p.ref_dtype])
        self.ref_sqnorm = alloc("ref_sqnorm", (LB, max(R, 1)), torch.float32)
        self.codes = alloc("codes", (LB, T, p.d_c * p.bits // 8), torch.uint8)
        self.hdr = alloc("hdr", (LB, T, p.d_c // 32, 2), torch.float32)
        self.ref_idx = alloc("ref_idx", (LB, T, 4), i32)
        self.workspace_bytes = ws
        self.workspace = alloc("workspace", (max(ws, 256),), torch.uint8)
        self.status = alloc("status", (4,), i32, fill=0)
        self.z = alloc("z", (LB, T, p.d_c), torch.float32) if want_z else None
        self.pool = rkv_ref_pool(_ptr(self.ref_pos), _ptr(self.ref_slot), _ptr(self.pool_size),
                                 _ptr(self.ref_vec), _ptr(self.ref_sqnorm))
        self.cache = rkv_cache(_ptr(self.codes), _ptr(self.hdr), _ptr(self.ref_idx))

    def build_ref_pool(self, kv, stream=None):
        rkv_build_ref_pool(self.p, kv, self.pool, stream)

    def compress(self, kv, W1t, W2t, W3t, stream=None):
        rkv_compress(self.p, kv, self.pool, W1t, W2t, W3t, self.cache, self.workspace,
                     self.workspace_bytes, self.z, self.status, stream)

    def gather(self, sel, out_z, out_mean, out_dtype=None, stream=None):
        n_sel = sel.shape[-1]
        if out_dtype is None:
            out_dtype = RKV_F32 if out_z.dtype == torch.float32 else RKV_BF16
        rkv_gather_dequant(self.p, self.pool, self.cache, sel, n_sel, out_z, out_mean, out_dtype,
                           self.status, stream)

    def restore(self, Wd, sel, out_k, out_v, rope_base: float, stream=None):
        rkv_restore_kv(self.p, self.pool, self.cache, Wd, sel, sel.shape[-1], rope_base, out_k,
                       out_v, self.status, stream)

    def append(self, kv_new, t: int, W1t, W2t, W3t, stream=None):
        rkv_append_token(self.p, kv_new, t, self.pool, W1t, W2t, W3t, self.cache, self.workspace,
                         self.workspace_bytes, self.status, stream)

    def attend(self, H: int, q, k_hat, v_hat, sel, out, stream=None):
        n_sel = sel.shape[-1]
        need = rkv_attention_workspace(self.p, H, n_sel)
        if getattr(self, "_attn_ws", None) is None or self._attn_ws.numel() < need:
            self._attn_ws, self._raw["attention_workspace"] = guarded_empty(
                (max(need, 256),), torch.uint8, self.status.device, self.guard)
        rkv_sparse_attention(self.p, H, q, k_hat, v_hat, sel, n_sel, out, self._attn_ws,
                             self._attn_ws.numel(), stream)

    def device_status(self) -> int:
        return int(self.status[0].item())

    def guard_violations(self):
        """Names of the buffers whose guard bytes changed (empty without guards)."""
        bad = []
        for name, raw in self._raw.items():
            t = self._attn_ws if name == "attention_workspace" else getattr(self, name)
            if raw is not None and t is not None and not guard_intact(t, raw):
                bad.append(name)
        return bad
