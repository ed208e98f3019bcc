// rkv_api.cu -- the extern "C" boundary of librkv: argument validation, size
// queries, workspace carve-up and dispatch to the kernels.  No entry point
// allocates device memory.
#include "rkv_internal.cuh"

#include <limits.h>
#include <math.h>

namespace rkv {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Reference count of the schedule p_{m+1} = p_m + stride + floor(alpha (p_m - n_sink)),
// computed with the same double arithmetic as the device schedule kernel.
static int schedule_count(const rkv_params *p)
{
    if (p->T <= p->first) return 0;
    if (p->alpha == 0.0) return (p->T - p->first + p->stride - 1) / p->stride;
    long long pos = p->first;
    int n = 0;
    while (pos < p->T) {
        ++n;
        pos = pos + p->stride + (long long)floor(p->alpha * (double)(pos - p->n_sink));
    }
    return n;
}

Geometry make_geometry(const rkv_params *p)
{
    Geometry g;
    g.L = p->L;
    g.B = p->B;
    g.LB = p->L * p->B;
    g.T = p->T;
    g.N = p->N;
    g.D = p->D;
    g.W = 2 * p->N * p->D;
    g.d_ff = p->d_ff;
    g.d_c = p->d_c;
    g.k = p->k;
    g.bits = p->bits;
    g.n_ref = schedule_count(p);
    g.n_groups = p->d_c / 32;
    g.code_pitch = p->d_c * p->bits / 8;
    g.kv_dtype = p->kv_dtype;
    g.ref_dtype = p->ref_dtype;
    g.stride = p->stride;
    g.first = p->first;
    g.alpha = p->alpha;
    g.n_sink = p->n_sink;
    g.n_mtiles = (p->T + kTileM - 1) / kTileM;
    int max_nt = (g.n_ref + kBN - 1) / kBN;
    g.max_chunks = max_nt == 0 ? 1 : (max_nt + kDistChunk - 1) / kDistChunk;
    return g;
}

Workspace workspace_layout(const Geometry &g)
{
    Workspace w{};
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += align256(bytes); return o; };
    const size_t LB = (size_t)g.LB, T = (size_t)g.T, R = (size_t)g.n_ref;
    const bool tc = g.kv_dtype == RKV_BF16;
    w.ref_mma = take(g.ref_dtype == RKV_FP8_E4M3 ? LB * R * g.W * 2 : 0);
    // one extra all-zero row after the last reference's row (padding for unused slots);
    // the tensor-core path keeps both projections interleaved in P1 ({P1[f], P2[f]})
    w.P1 = take((LB * R + 1) * g.d_ff * (tc ? 8 : 4));
    w.P2 = take(tc ? 0 : (LB * R + 1) * g.d_ff * 4);
    w.rn_max = take(LB * 4);
    w.cand = take(tc ? LB * T * g.max_chunks * kCand * 8 : 0);
    w.copy_flag = take(LB * T);
    w.xnorm = take(tc ? LB * T * 4 : 0);
    w.scan_list = take(tc ? (LB * T + 1) * 4 : 0);     // list, then its count
    w.rr_list = take(tc ? LB * T * 8 + 8 : 0);         // list, then its count
    w.dh_hi = take(tc ? LB * T * g.d_ff * 2 : 0);
    w.dh_lo = take(tc ? LB * T * g.d_ff * 2 : 0);
    w.dh32 = take(tc ? 0 : LB * T * g.d_ff * 4);
    w.z32 = take(tc ? 0 : LB * T * g.d_c * 4);
    w.total = off;
    return w;
}

static rkv_status check_params(const rkv_params *p)
{
    if (!p) return RKV_ERR_INVALID_ARG;
    if (p->L < 1 || p->B < 1 || p->T < 1 || p->N < 1 || p->D < 1 || p->d_ff < 1 || p->d_c < 1)
        return RKV_ERR_INVALID_ARG;
    if (p->stride < 1 || p->first < 0 || p->k < 1 || p->group < 1)
        return RKV_ERR_INVALID_ARG;
    if (!(p->alpha >= 0.0) || p->alpha > 1e6 || p->n_sink < 0) return RKV_ERR_INVALID_ARG;
    // the schedule's steps grow with the position; the first one must advance
    if (p->stride + (long long)floor(p->alpha * (double)(p->first - p->n_sink)) < 1)
        return RKV_ERR_INVALID_ARG;
    if (p->bits != 2 && p->bits != 4) return RKV_ERR_INVALID_ARG;
    if (p->kv_dtype != RKV_F32 && p->kv_dtype != RKV_BF16) return RKV_ERR_INVALID_ARG;
    if (p->ref_dtype != p->kv_dtype && !(p->ref_dtype == RKV_FP8_E4M3 && p->kv_dtype == RKV_BF16))
        return RKV_ERR_INVALID_ARG;
    // sizes that are legal for the method but not handled here
    if (p->k > kMaxK || p->group != 32 || p->d_c % 32 != 0) return RKV_ERR_UNSUPPORTED;
    long long W = 2LL * p->N * p->D;
    if (W % 8 != 0 || p->d_ff % 8 != 0) return RKV_ERR_UNSUPPORTED;
    if (W > (1 << 20) || p->d_ff > (1 << 16) || p->d_c > (1 << 14)) return RKV_ERR_UNSUPPORTED;
    if ((long long)p->L * p->B > (1 << 20)) return RKV_ERR_UNSUPPORTED;
    if ((long long)p->L * p->B * p->T > (long long)INT_MAX) return RKV_ERR_UNSUPPORTED;
    return RKV_OK;
}

static bool aligned16(const void *q) { return ((uintptr_t)q & 15u) == 0; }

static size_t elem_bytes(int dt) { return dt == RKV_F32 ? 4 : (dt == RKV_BF16 ? 2 : 1); }

static rkv_status check_pool(const rkv_ref_pool *pool, int n_ref)
{
    if (!pool || !pool->ref_slot || !pool->pool_size) return RKV_ERR_INVALID_ARG;
    // the reference arrays are empty (and may be NULL) when no reference exists
    if (n_ref > 0 && (!pool->ref_pos || !pool->ref_vec || !pool->ref_sqnorm))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(pool->ref_pos) || !aligned16(pool->ref_slot) || !aligned16(pool->pool_size) ||
        !aligned16(pool->ref_vec) || !aligned16(pool->ref_sqnorm))
        return RKV_ERR_ALIGNMENT;
    return RKV_OK;
}

static rkv_status check_cache(const rkv_cache *c)
{
    if (!c || !c->codes || !c->hdr || !c->ref_idx) return RKV_ERR_INVALID_ARG;
    if (!aligned16(c->codes) || !aligned16(c->hdr) || !aligned16(c->ref_idx))
        return RKV_ERR_ALIGNMENT;
    return RKV_OK;
}

int current_device()
{
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

int device_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n;
}

}  // namespace rkv

using namespace rkv;

extern "C" {

const char *rkv_status_string(rkv_status s)
{
    switch (s) {
    case RKV_OK: return "ok";
    case RKV_ERR_INVALID_ARG: return "invalid argument";
    case RKV_ERR_UNSUPPORTED: return "unsupported size or type";
    case RKV_ERR_ALIGNMENT: return "buffer not 16-byte aligned";
    case RKV_ERR_CUDA: return "CUDA runtime error";
    case RKV_ERR_INDEX: return "index out of range (device)";
    case RKV_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case RKV_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

int32_t rkv_n_ref(const rkv_params *p)
{
    if (check_params(p) == RKV_ERR_INVALID_ARG) return -1;
    return make_geometry(p).n_ref;
}

rkv_status rkv_query_sizes(const rkv_params *p, size_t *pool_bytes, size_t *cache_bytes,
                           size_t *workspace_bytes)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    Geometry g = make_geometry(p);
    const size_t LB = (size_t)g.LB, T = (size_t)g.T, R = (size_t)g.n_ref;
    if (pool_bytes)
        *pool_bytes = R * 4 + 2 * T * 4 + LB * R * g.W * elem_bytes(g.ref_dtype) + LB * R * 4;
    if (cache_bytes)
        *cache_bytes = LB * T * ((size_t)g.code_pitch + (size_t)g.n_groups * 8 + 16);
    if (workspace_bytes) *workspace_bytes = workspace_layout(g).total;
    return RKV_OK;
}

rkv_status rkv_build_ref_pool(const rkv_params *p, const void *kv, const rkv_ref_pool *pool,
                              void *stream)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    if (!kv) return RKV_ERR_INVALID_ARG;
    if ((st = check_pool(pool, make_geometry(p).n_ref)) != RKV_OK) return st;
    if (!aligned16(kv)) return RKV_ERR_ALIGNMENT;
    Geometry g = make_geometry(p);
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_build_schedule(g, pool, s) != cudaSuccess) return RKV_ERR_CUDA;
    if (g.n_ref > 0 && launch_build_refs(g, kv, pool, s) != cudaSuccess) return RKV_ERR_CUDA;
    return RKV_OK;
}

rkv_status rkv_compress(const rkv_params *p, const void *kv, const rkv_ref_pool *pool,
                        const void *W1t, const void *W2t, const void *W3t,
                        const rkv_cache *cache, void *workspace, size_t workspace_bytes,
                        float *z_out, int32_t *dev_status, void *stream)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    if (!kv || !W1t || !W2t || !W3t || !dev_status) return RKV_ERR_INVALID_ARG;
    if ((st = check_pool(pool, make_geometry(p).n_ref)) != RKV_OK) return st;
    if ((st = check_cache(cache)) != RKV_OK) return st;
    if (!aligned16(kv) || !aligned16(W1t) || !aligned16(W2t) || !aligned16(W3t) ||
        !aligned16(dev_status) || (z_out && !aligned16(z_out)))
        return RKV_ERR_ALIGNMENT;
    Geometry g = make_geometry(p);
    // tensor-core path: epilogues work on 32-column slices of d_ff
    if (g.kv_dtype == RKV_BF16 && g.d_ff % 32 != 0) return RKV_ERR_UNSUPPORTED;
    // projection-row offsets are 32-bit in the encoder
    if (((long long)g.LB * g.n_ref + 1) * g.d_ff >= (1LL << 31)) return RKV_ERR_UNSUPPORTED;
    Workspace wl = workspace_layout(g);
    if (wl.total > 0 && (!workspace || workspace_bytes < wl.total)) return RKV_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return RKV_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (g.kv_dtype == RKV_BF16)
        e = launch_umma_compress(g, kv, pool, W1t, W2t, W3t, cache, (uint8_t *)workspace, wl,
                                 z_out, dev_status, s);
    else
        e = launch_simt_compress(g, kv, pool, W1t, W2t, W3t, cache, (uint8_t *)workspace, wl,
                                 z_out, dev_status, s);
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

rkv_status rkv_gather_dequant(const rkv_params *p, const rkv_ref_pool *pool,
                              const rkv_cache *cache, const int32_t *sel, int32_t n_sel,
                              void *out_z, void *out_mean, int32_t out_dtype,
                              int32_t *dev_status, void *stream)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    if (n_sel < 0) return RKV_ERR_INVALID_ARG;
    if (out_dtype != RKV_F32 && out_dtype != RKV_BF16) return RKV_ERR_INVALID_ARG;
    if ((st = check_pool(pool, make_geometry(p).n_ref)) != RKV_OK) return st;
    if ((st = check_cache(cache)) != RKV_OK) return st;
    if (n_sel == 0) return RKV_OK;
    if (!sel || !out_z || !out_mean || !dev_status) return RKV_ERR_INVALID_ARG;
    if (!aligned16(sel) || !aligned16(out_z) || !aligned16(out_mean) || !aligned16(dev_status))
        return RKV_ERR_ALIGNMENT;
    Geometry g = make_geometry(p);
    if ((long long)g.LB * n_sel > (long long)INT_MAX) return RKV_ERR_UNSUPPORTED;
    cudaError_t e = launch_gather(g, pool, cache, sel, n_sel, out_z, out_mean, out_dtype,
                                  dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

rkv_status rkv_restore_kv(const rkv_params *p, const rkv_ref_pool *pool, const rkv_cache *cache,
                          const void *Wd, const int32_t *sel, int32_t n_sel, double rope_base,
                          void *out_k, void *out_v, int32_t *dev_status, void *stream)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    if (n_sel < 0 || !(rope_base > 0.0) || !isfinite(rope_base)) return RKV_ERR_INVALID_ARG;
    if (p->kv_dtype != RKV_BF16) return RKV_ERR_UNSUPPORTED;
    if ((p->d_c != 256 && p->d_c != 512) || (2 * p->N * p->D) % 256 != 0 || p->D % 32 != 0 ||
        p->D > 256)
        return RKV_ERR_UNSUPPORTED;
    if ((st = check_pool(pool, make_geometry(p).n_ref)) != RKV_OK) return st;
    if ((st = check_cache(cache)) != RKV_OK) return st;
    if (n_sel == 0) return RKV_OK;
    if (!Wd || !sel || !out_k || !out_v || !dev_status) return RKV_ERR_INVALID_ARG;
    if (!aligned16(Wd) || !aligned16(sel) || !aligned16(out_k) || !aligned16(out_v) ||
        !aligned16(dev_status))
        return RKV_ERR_ALIGNMENT;
    Geometry g = make_geometry(p);
    if ((long long)g.LB * n_sel * g.W > (long long)INT_MAX * 64) return RKV_ERR_UNSUPPORTED;
    cudaError_t e = launch_restore(g, pool, cache, Wd, sel, n_sel, rope_base, out_k, out_v,
                                   dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

rkv_status rkv_append_token(const rkv_params *p, const void *kv_new, int32_t t,
                            const rkv_ref_pool *pool, const void *W1t, const void *W2t,
                            const void *W3t, const rkv_cache *cache, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    if (t < 0 || t >= p->T) return RKV_ERR_INVALID_ARG;
    Geometry g = make_geometry(p);
    if ((st = check_pool(pool, g.n_ref)) != RKV_OK) return st;
    if ((st = check_cache(cache)) != RKV_OK) return st;
    if (!kv_new || !W1t || !W2t || !W3t || !dev_status) return RKV_ERR_INVALID_ARG;
    if (!aligned16(kv_new) || !aligned16(W1t) || !aligned16(W2t) || !aligned16(W3t) ||
        !aligned16(dev_status))
        return RKV_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < append_workspace_bytes(g)) return RKV_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255) != 0) return RKV_ERR_ALIGNMENT;
    cudaError_t e = launch_append(g, kv_new, t, pool, W1t, W2t, W3t, cache, workspace, dev_status,
                                  (cudaStream_t)stream);
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

static rkv_status check_attention(const rkv_params *p, int32_t H, int32_t n_sel)
{
    rkv_status st = check_params(p);
    if (st != RKV_OK) return st;
    if (n_sel < 0 || H <= 0) return RKV_ERR_INVALID_ARG;
    if (p->kv_dtype != RKV_BF16) return RKV_ERR_UNSUPPORTED;
    if ((p->D != 64 && p->D != 128 && p->D != 256) || H % p->N != 0 || H / p->N > 8 ||
        (p->D == 256 && H / p->N > 4))
        return RKV_ERR_UNSUPPORTED;
    return RKV_OK;
}

rkv_status rkv_attention_workspace(const rkv_params *p, int32_t H, int32_t n_sel, size_t *bytes)
{
    rkv_status st = check_attention(p, H, n_sel);
    if (st != RKV_OK) return st;
    if (!bytes) return RKV_ERR_INVALID_ARG;
    *bytes = attention_workspace_bytes(make_geometry(p), H, n_sel);
    return RKV_OK;
}

rkv_status rkv_sparse_attention(const rkv_params *p, int32_t H, const void *q, const void *k_hat,
                                const void *v_hat, const int32_t *sel, int32_t n_sel, float *out,
                                void *workspace, size_t workspace_bytes, void *stream)
{
    rkv_status st = check_attention(p, H, n_sel);
    if (st != RKV_OK) return st;
    Geometry g = make_geometry(p);
    if (!q || !out) return RKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return RKV_ERR_ALIGNMENT;
    if (n_sel == 0) {
        cudaError_t e = cudaMemsetAsync(out, 0, (size_t)g.LB * H * g.D * sizeof(float), (cudaStream_t)stream);
        return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
    }
    if (!k_hat || !v_hat || !sel) return RKV_ERR_INVALID_ARG;
    if (!aligned16(k_hat) || !aligned16(v_hat) || !aligned16(sel)) return RKV_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < attention_workspace_bytes(g, H, n_sel)) return RKV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return RKV_ERR_ALIGNMENT;
    cudaError_t e = launch_attention(g, H, q, k_hat, v_hat, sel, n_sel, out, workspace, (cudaStream_t)stream);
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

}  // extern "C"
