"""Seeded synthetic workloads for the ResidualKV cache-write and sparse-read path.

This module draws random numbers and rounds them to a storage format; it holds no
step of the method itself (no distance, mean, compressor or quantizer).  Both the
CUDA path and the fp64 oracle are fed from here, so that they see the same bytes.

Random numbers come from a counter-based generator: splitmix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) applied to
``key + (i + 1) * 0x9E3779B97F4A7C15`` for draw ``i`` of a stream, where ``key``
is derived from the config seed and a tuple of integer tags.  Normal draws use
Box-Muller on two consecutive uniforms.  Every operation is plain uint64 / float64
numpy arithmetic, so the draws do not depend on the numpy version.

The value recipes (shapes, centroid counts, noise scales, copy rule, image
segments, reference strides) stand in for the real-model KV caches that the
ResidualKV experiments use; the tokens are synthetic.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLD = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream tags (purpose of a random stream)
TAG_CENT, TAG_CID, TAG_NOISE, TAG_COPYFLAG, TAG_COPYSRC = 1, 2, 3, 4, 5
TAG_PATCH, TAG_W1, TAG_W2, TAG_W3, TAG_SEL, TAG_USER = 6, 7, 8, 9, 10, 11
TAG_WD, TAG_REC, TAG_QUERY = 12, 13, 14


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser, in place on a uint64 array."""
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, *tags: int) -> int:
    """64-bit key of the stream named by (seed, tags)."""
    with np.errstate(over="ignore"):
        h = _mix(np.array([seed], dtype=np.uint64) + _GOLD)
        for t in tags:
            h = _mix(h ^ (np.array([t], dtype=np.uint64) * _GOLD + np.uint64(0x632BE59BD9B4E019)))
    return int(h[0])


def uniform(key: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws offset..offset+n-1 of stream `key` as float64 in [0, 1) (53 bits)."""
    with np.errstate(over="ignore"):
        z = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z *= _GOLD
        z += np.uint64(key)
        _mix(z)
    z >>= np.uint64(11)
    # 53-bit integers are exact in int64 and float64
    out = z.view(np.int64).astype(np.float64)
    out *= 1.0 / 9007199254740992.0
    return out


def normal(key: int, n: int, offset: int = 0) -> np.ndarray:
    """Normal draws offset..offset+n-1 of stream `key` (Box-Muller on uniform pairs)."""
    u = uniform(key, 2 * n, 2 * offset).reshape(n, 2)
    r = np.log1p(-u[:, 0])
    r *= -2.0
    np.sqrt(r, out=r)
    c = u[:, 1] * (2.0 * math.pi)
    np.cos(c, out=c)
    r *= c
    return r


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype ('f32' -> float32, 'bf16' -> uint16 bits)."""
    x32 = x.astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def stored_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    raise ValueError(dtype)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    seed: int
    L: int
    B: int
    T: int
    N: int
    D: int
    d_ff: int
    d_c: int
    k: int = 4
    group: int = 32
    bits: int = 4
    stride: int = 8             # fixed stride, or s0 of the dynamic schedule
    first: int = 0
    alpha: float = 0.0          # dynamic-stride growth (0: fixed stride)
    n_sink: int = 0
    kv_dtype: str = "bf16"      # 'f32' or 'bf16' (kv and compressor weights)
    ref_dtype: str = "bf16"     # same as kv_dtype, or 'fp8' (OCP E4M3)
    recipe: str = "text"        # 'centroids' | 'text' | 'multimodal'
    n_cent: int = 256
    noise: float = 0.3
    copy_p: float = 0.4
    copy_gap: int = 17          # a copy source j satisfies j <= i - copy_gap
    copy_noise: float = 0.05
    n_patch: int = 64
    patch_noise: float = 0.2
    seg_len: int = 576
    n_seg: int = 4
    gather_frac: float = 0.3
    gather_tail: int = 512
    gather_steps: int = 0
    rope_base: float = 10000.0  # base of the rotary embedding applied to restored keys
    H: int = 32                 # query heads of the attention that reads the cache

    @property
    def W(self) -> int:
        return 2 * self.N * self.D

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# The five workloads.  Model shapes: Llama-3.1-8B (8 KV heads x 128) and Qwen2.5-7B
# (4 KV heads x 128), ResidualKV paper Table I.
CONFIGS = {
    "tiny-fp32": Config("tiny-fp32", seed=0, L=1, B=1, T=256, N=2, D=64, d_ff=256, d_c=64,
                        stride=8, kv_dtype="f32", ref_dtype="f32", recipe="centroids", n_cent=16),
    "llama3.1-8b-kv": Config("llama3.1-8b-kv", seed=1, L=32, B=1, T=8192, N=8, D=128,
                             d_ff=1024, d_c=512, stride=8),
    "qwen2.5-7b-kv": Config("qwen2.5-7b-kv", seed=2, L=28, B=1, T=32768, N=4, D=128,
                            d_ff=512, d_c=256, stride=8, H=28),
    "long-131k-fp8ref": Config("long-131k-fp8ref", seed=3, L=1, B=1, T=131072, N=8, D=128,
                               d_ff=1024, d_c=512, stride=16, ref_dtype="fp8", gather_steps=256),
    "multimodal-8x4096-int2": Config("multimodal-8x4096-int2", seed=4, L=1, B=8, T=4096, N=8,
                                     D=128, d_ff=1024, d_c=512, bits=2, stride=8,
                                     recipe="multimodal"),
}
CONFIG_ORDER = ["tiny-fp32", "llama3.1-8b-kv", "qwen2.5-7b-kv", "long-131k-fp8ref",
                "multimodal-8x4096-int2"]


def _text_mask(cfg: Config) -> np.ndarray:
    m = np.ones(cfg.T, dtype=bool)
    if cfg.recipe == "multimodal":
        for s0, s1 in image_segments(cfg):
            m[s0:s1] = False
    return m


def image_segments(cfg: Config):
    """[start, end) of each image segment: n_seg segments of seg_len tokens with equal
    text gaps before and between them; the remainder is trailing text."""
    gap = (cfg.T - cfg.n_seg * cfg.seg_len) // (cfg.n_seg + 1)
    return [(gap + m * (gap + cfg.seg_len), gap + m * (gap + cfg.seg_len) + cfg.seg_len)
            for m in range(cfg.n_seg)]


def _normal_rows(key: int, T: int, W: int, threads: int = 0) -> np.ndarray:
    """normal(key, T*W) as [T][W], drawn in row blocks on several threads (the stream is
    counter-based, so the values do not depend on the blocking)."""
    if threads <= 1 or T * W < (1 << 24):
        return normal(key, T * W).reshape(T, W)
    import concurrent.futures as cf
    out = np.empty((T, W), dtype=np.float64)
    step = max(1, T // (4 * threads))

    def fill(r0):
        r1 = min(T, r0 + step)
        out[r0:r1] = normal(key, (r1 - r0) * W, r0 * W).reshape(r1 - r0, W)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(0, T, step)))
    return out


GEN_THREADS = 16


def sequence_kv64(cfg: Config, layer: int, seq: int) -> np.ndarray:
    """Unrounded float64 kv rows [T][W] of one (layer, sequence)."""
    T, W = cfg.T, cfg.W
    s = cfg.seed
    kv = np.empty((T, W), dtype=np.float64)
    threads = GEN_THREADS if cfg.L * cfg.B == 1 else 0
    noise = _normal_rows(stream_key(s, TAG_NOISE, layer, seq), T, W, threads)
    if cfg.recipe == "centroids":
        cent = normal(stream_key(s, TAG_CENT, layer, seq), cfg.n_cent * W).reshape(cfg.n_cent, W)
        cid = np.minimum((uniform(stream_key(s, TAG_CID, layer, seq), T) * cfg.n_cent).astype(np.int64),
                         cfg.n_cent - 1)
        return cent[cid] + cfg.noise * noise

    text = _text_mask(cfg)
    tpos = np.nonzero(text)[0]
    cent = normal(stream_key(s, TAG_CENT, layer, seq), cfg.n_cent * W).reshape(cfg.n_cent, W)
    u_cid = uniform(stream_key(s, TAG_CID, layer, seq), T)
    cid = np.minimum((u_cid * cfg.n_cent).astype(np.int64), cfg.n_cent - 1)
    kv[:] = cent[cid] + cfg.noise * noise
    if cfg.recipe == "multimodal":
        pid = np.minimum((u_cid * cfg.n_patch).astype(np.int64), cfg.n_patch - 1)
        for m, (s0, s1) in enumerate(image_segments(cfg)):
            pc = normal(stream_key(s, TAG_PATCH, layer, seq, m), cfg.n_patch * W).reshape(cfg.n_patch, W)
            kv[s0:s1] = pc[pid[s0:s1]] + cfg.patch_noise * noise[s0:s1]

    # copy rule (text tokens only): with probability copy_p, token i repeats an earlier
    # text token j <= i - copy_gap (itself possibly a copy) plus copy_noise * N(0,1).
    u_flag = uniform(stream_key(s, TAG_COPYFLAG, layer, seq), T)
    u_src = uniform(stream_key(s, TAG_COPYSRC, layer, seq), T)
    n_avail = np.searchsorted(tpos, np.arange(T) - cfg.copy_gap, side="right")
    is_copy = text & (u_flag < cfg.copy_p) & (n_avail > 0)
    src = np.where(is_copy, tpos[np.minimum((u_src * n_avail).astype(np.int64),
                                            np.maximum(n_avail - 1, 0))], -1)
    rows = np.nonzero(is_copy)[0]
    # a copy's source lies >= copy_gap rows back, so blocks of copy_gap-1 rows are
    # independent and can be filled together in increasing order
    blk = max(cfg.copy_gap - 1, 1)
    if rows.size:
        bid = rows // blk
        cuts = np.nonzero(np.diff(bid))[0] + 1
        for grp in np.split(rows, cuts):
            kv[grp] = kv[src[grp]] + cfg.copy_noise * noise[grp]
    return kv


def layer_kv(cfg: Config, layer: int) -> np.ndarray:
    """Stored kv of one layer, [B][T][W] (float32, or uint16 bf16 bit patterns)."""
    out = np.empty((cfg.B, cfg.T, cfg.W), dtype=np.float32 if cfg.kv_dtype == "f32" else np.uint16)
    for b in range(cfg.B):
        out[b] = store(sequence_kv64(cfg, layer, b), cfg.kv_dtype)
    return out


def layer_weights(cfg: Config, layer: int):
    """Stored compressor weights of one layer, out-major (as a linear layer keeps them):
    W1t, W2t: [d_ff][W]  (W1t[f][c] = W_c1[c][f]),  W3t: [d_c][d_ff]  (W3t[j][f] = W_c3[f][j]).
    Entries ~ N(0, 1/fan_in)."""
    W, F, C, s = cfg.W, cfg.d_ff, cfg.d_c, cfg.seed
    w1 = normal(stream_key(s, TAG_W1, layer), F * W).reshape(F, W) * math.sqrt(1.0 / W)
    w2 = normal(stream_key(s, TAG_W2, layer), F * W).reshape(F, W) * math.sqrt(1.0 / W)
    w3 = normal(stream_key(s, TAG_W3, layer), C * F).reshape(C, F) * math.sqrt(1.0 / F)
    return store(w1, cfg.kv_dtype), store(w2, cfg.kv_dtype), store(w3, cfg.kv_dtype)


def decoder_weights(cfg: Config, layer: int):
    """Stored linear-decoder weights of one layer, out-major: Wd [W][d_c]
    (Wd[c][j] = W_d[j][c]), entries ~ N(0, 1/d_c)."""
    w = normal(stream_key(cfg.seed, TAG_WD, layer), cfg.W * cfg.d_c).reshape(cfg.W, cfg.d_c)
    return store(w * math.sqrt(1.0 / cfg.d_c), cfg.kv_dtype)


def decode_queries(cfg: Config, layer: int, step: int) -> np.ndarray:
    """Query vectors of one decode step of one layer, [B][H][D] ~ N(0, 1), stored in the
    kv dtype (the model that would produce them is not part of this workload)."""
    q = normal(stream_key(cfg.seed, TAG_QUERY, layer, step), cfg.B * cfg.H * cfg.D)
    return store(q.reshape(cfg.B, cfg.H, cfg.D), cfg.kv_dtype)


def synthetic_records(cfg: Config, n_ref: int, lb: int = 0):
    """Arbitrary well-formed cache records of one (layer, sequence), for testing the read
    side on its own: codes [T][d_c] uniform in [0, 2^bits), group minima ~ N(0, 0.1^2),
    steps ~ U(0, 0.05) with every 7th group constant (step 0), reference relations of
    1..k distinct slots in [0, n_ref) (the first ones of a Floyd sample of k distinct
    slots), ascending, -1 padded; and n_ref pool vectors
    ~ N(0, 1) stored in ref_dtype (FP8: uniform non-NaN bytes).
    Returns (codes, zmin, delta, ref_idx, refs)."""
    T, C, G, k = cfg.T, cfg.d_c, cfg.d_c // cfg.group, cfg.k
    key = lambda part: stream_key(cfg.seed, TAG_REC, lb, part)
    codes = np.minimum(np.floor(uniform(key(0), T * C) * (1 << cfg.bits)),
                       (1 << cfg.bits) - 1).astype(np.uint8).reshape(T, C)
    zmin = (normal(key(1), T * G) * 0.1).reshape(T, G)
    delta = (uniform(key(2), T * G) * 0.05).reshape(T, G)
    delta[:, ::7] = 0.0
    cnt = 1 + np.minimum(np.floor(uniform(key(3), T) * k), k - 1).astype(np.int64)
    # Floyd's sampling of k distinct slots per row: draw i picks r in [0, j], j = n_ref - k + i,
    # and takes j instead when r was already taken
    assert n_ref >= k
    u = uniform(key(4), T * k).reshape(T, k)
    first = np.empty((T, k), np.int64)
    for i in range(k):
        j = n_ref - k + i
        r = np.minimum(np.floor(u[:, i] * (j + 1)), j).astype(np.int64)
        dup = (first[:, :i] == r[:, None]).any(axis=1)
        first[:, i] = np.where(dup, j, r)
    # row t: its first cnt[t] sampled slots in ascending order, then -1
    used = np.arange(k)[None, :] < cnt[:, None]
    first = np.sort(np.where(used, first, np.iinfo(np.int64).max), axis=1)
    ref_idx = np.where(first == np.iinfo(np.int64).max, -1, first).astype(np.int32)
    if cfg.ref_dtype == "fp8":
        # stored FP8 bytes drawn directly: any byte but the two NaN codes 0x7f, 0xff
        b = np.floor(uniform(key(5), n_ref * cfg.W) * 254).astype(np.int64)
        refs = (b + (b >= 0x7f)).astype(np.uint8).reshape(n_ref, cfg.W)
    else:
        refs = store(normal(key(5), n_ref * cfg.W).reshape(n_ref, cfg.W), cfg.ref_dtype)
    return codes, zmin.astype(np.float32), delta.astype(np.float32), ref_idx, refs


def gather_selection(cfg: Config, step: int, seq: int = 0) -> np.ndarray:
    """Decode-step index set: a uniform random floor(gather_frac*T)-subset of [0, T)
    (without replacement) united with the last gather_tail tokens; sorted, unique."""
    T = cfg.T
    n = int(math.floor(cfg.gather_frac * T))
    keys = uniform(stream_key(cfg.seed, TAG_SEL, step, seq), T)
    pick = np.argsort(keys, kind="stable")[:n]
    tail = np.arange(max(0, T - cfg.gather_tail), T)
    return np.unique(np.concatenate([pick, tail])).astype(np.int32)
