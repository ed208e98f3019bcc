// rkv_topk.cu -- final reference choice per token [RKV §2.2 = Sec. IV-A]:
//   R_t = the k_t = min(k, pool_size[t]) references with pos < t nearest to kv_t in
//   squared L2, ties to the lower slot, stored in ascending slot order.
//
// The tensor-core pass ranks references by the expansion ||r||^2 - 2 x.r (the
// ||x||^2 term is common to a row) and keeps each work item's best kCand.  Here one
// warp per token merges those candidates and decides:
//   * if the k-th/(k+1)-th expansion gap exceeds twice the expansion error bound
//     E = kTau (rmax + 2 sqrt(||x||^2 rmax)), rmax = max ||r||^2 of the sequence,
//     the expansion's top-k is the exact top-k;
//   * else, if every possible member of the exact top-k is among the candidates
//     (all of the pool fits, or the 8th candidate is more than 2E behind the k-th),
//     the candidates are re-ranked by exact distances;
//   * else every reference of the pool is scanned with exact distances.
// It also flags tokens that are bit-identical to every chosen reference: their mean
// equals the token exactly, so z = 0 exactly [RKV §2.3], which the encoder then
// writes directly (the tensor cores need not round the token's and the
// references' projections identically, since they sit in different tile rows).
// Exact distances sum (x - r)^2 in fp32: for bf16 data x - r is exact, each group of
// 8 squares is added as a tree, and the warp adds its lanes as a tree.
// Without candidates (the fp32 path) every token takes the full scan.
#include "rkv_internal.cuh"

namespace rkv {

template <typename T> struct Vec8;
template <> struct Vec8<float> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[8])
    {
        float4 a = *(const float4 *)p, b = *(const float4 *)(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};
template <> struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[8])
    {
        uint4 raw = *(const uint4 *)p;
        const __nv_bfloat16 *h = (const __nv_bfloat16 *)&raw;
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __bfloat162float(h[j]);
    }
};

__device__ __forceinline__ float warp_tree_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__device__ __forceinline__ float warp_sqdist(const T *x, const T *r, int W, int lane)
{
    float acc = 0.0f;
    for (int c = lane * 8; c < W; c += 256) {
        float a[8], b[8];
        Vec8<T>::load(x + c, a);
        Vec8<T>::load(r + c, b);
        float s[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float d = a[j] - b[j];
            s[j] = d * d;
        }
        float s8 = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
        acc += s8;
    }
    return warp_tree_sum(acc);
}

template <typename T>
__device__ __forceinline__ float warp_sqnorm(const T *x, int W, int lane)
{
    // four independent 8-element loads in flight per lane
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int c = lane * 8;
    for (; c + 3 * 256 < W; c += 4 * 256) {
        float a[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) Vec8<T>::load(x + c + u * 256, a[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[u] = fmaf(a[u][j], a[u][j], acc[u]);
    }
    for (; c < W; c += 256) {
        float a[8];
        Vec8<T>::load(x + c, a);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[0] = fmaf(a[j], a[j], acc[0]);
    }
    return warp_tree_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
}

__device__ __forceinline__ bool key_less(float ea, int sa, float eb, int sb)
{
    return ea < eb || (ea == eb && (unsigned)sa < (unsigned)sb);
}

// Insert (e, s) into an ascending list of n entries (registers, uniform per lane).
template <int N>
__device__ __forceinline__ void list_insert(float (&le)[N], int (&ls)[N], float e, int s)
{
#pragma unroll
    for (int q = 0; q < N; ++q) {
        bool lt = key_less(e, s, le[q], ls[q]);
        float te = lt ? le[q] : e;
        int ts = lt ? ls[q] : s;
        if (lt) { le[q] = e; ls[q] = s; }
        e = te;
        s = ts;
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
k_topk_finalize(const T *__restrict__ kv, const T *__restrict__ refs,
                const int32_t *__restrict__ ref_slot, const int32_t *__restrict__ pool_size,
                const float2 *__restrict__ cand, const float *__restrict__ rn_max, int LB, int T_,
                int W, int n_ref, int k, int max_chunks, int4 *__restrict__ ref_idx,
                uint8_t *__restrict__ copy_flag)
{
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (gw >= (long long)LB * T_) return;
    const int lb = (int)(gw / T_), t = (int)(gw % T_);

    int out[4] = {-1, -1, -1, -1};
    int same = 0;
    const int own = ref_slot[t];
    const int pool = pool_size[t];
    const T *x = kv + ((size_t)lb * T_ + t) * W;
    const T *rb = refs + (size_t)lb * n_ref * W;
    if (own >= 0) {
        out[0] = own;
    } else if (pool <= k) {
        same = pool > 0;
        for (int j = 0; j < pool; ++j) {
            out[j] = j;
            same &= warp_sqdist(x, rb + (size_t)j * W, W, lane) == 0.0f;
        }
    } else {
        float be[kMaxK];
        int bs[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) { be[j] = INFINITY; bs[j] = 0x7fffffff; }
        bool full_scan = (cand == nullptr);
        if (!full_scan) {
            // merge the work items' candidate lists: per-lane top-kCand, then 8 warp argmins
            const int m = t / kBM;
            const int nt = dist_ntiles(pool_size, T_, m);
            const int nch = (nt + kDistChunk - 1) / kDistChunk;
            const float2 *cp = cand + ((size_t)lb * T_ + t) * max_chunks * kCand;
            float le[kCand];
            int ls[kCand];
#pragma unroll
            for (int q = 0; q < kCand; ++q) { le[q] = INFINITY; ls[q] = 0x7fffffff; }
            for (int u = lane; u < nch * kCand; u += 32) {
                float2 c = cp[u];
                int s = __float_as_int(c.y);
                if (s >= 0 && c.x < INFINITY) list_insert<kCand>(le, ls, c.x, s);
            }
            float ce[kCand];
            int cs[kCand];
            int head = 0;
#pragma unroll
            for (int r = 0; r < kCand; ++r) {
                float e = INFINITY;
                int s = 0x7fffffff;
#pragma unroll
                for (int q = 0; q < kCand; ++q)
                    if (q == head) { e = le[q]; s = ls[q]; }
                float we = e;
                int ws = s, wl = lane;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    float oe = __shfl_xor_sync(0xffffffffu, we, o);
                    int os = __shfl_xor_sync(0xffffffffu, ws, o);
                    int ol = __shfl_xor_sync(0xffffffffu, wl, o);
                    if (key_less(oe, os, we, ws)) { we = oe; ws = os; wl = ol; }
                }
                ce[r] = we;
                cs[r] = ws;
                if (wl == lane && we < INFINITY) ++head;
            }
            const int nvalid = pool < kCand ? pool : kCand;
            const float xn = warp_sqnorm(x, W, lane);
            const float rm = rn_max[lb];
            const float E = kTau * (rm + 2.0f * sqrtf(xn * rm));
            if (nvalid > k && ce[k] - ce[k - 1] > 2.0f * E) {
                for (int j = 0; j < k; ++j) { be[j] = ce[j]; bs[j] = cs[j]; }
                // possibly an exact copy of all k: confirm with exact distances
                if (xn + ce[k - 1] <= 2.0f * E) {
                    for (int j = 0; j < k; ++j) be[j] = warp_sqdist(x, rb + (size_t)bs[j] * W, W, lane);
                } else {
                    be[0] = 1.0f;   // not a copy
                }
            } else if (pool <= kCand || ce[kCand - 1] - ce[k - 1] > 2.0f * E) {
                for (int r = 0; r < nvalid; ++r) {
                    float d = warp_sqdist(x, rb + (size_t)cs[r] * W, W, lane);
                    list_insert<kMaxK>(be, bs, d, cs[r]);
                }
            } else {
                full_scan = true;
            }
        }
        if (full_scan) {
            for (int s = 0; s < pool; ++s) {
                float d = warp_sqdist(x, rb + (size_t)s * W, W, lane);
                list_insert<kMaxK>(be, bs, d, s);
            }
        }
        same = 1;
        for (int j = 0; j < k; ++j) same &= be[j] == 0.0f;
        // chosen slots in ascending order
        int ch[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) ch[j] = j < k ? bs[j] : 0x7fffffff;
#pragma unroll
        for (int a = 0; a < kMaxK; ++a)
#pragma unroll
            for (int b = 0; b + 1 < kMaxK - a; ++b)
                if (ch[b] > ch[b + 1]) { int tmp = ch[b]; ch[b] = ch[b + 1]; ch[b + 1] = tmp; }
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) out[j] = j < k ? ch[j] : -1;
    }
    if (lane == 0) {
        ref_idx[(size_t)lb * T_ + t] = make_int4(out[0], out[1], out[2], out[3]);
        copy_flag[(size_t)lb * T_ + t] = (uint8_t)same;
    }
}

cudaError_t launch_topk_finalize(const Geometry &g, const void *kv, const void *ref_exact,
                                 int ref_exact_is_f32, const rkv_ref_pool *pool,
                                 const float2 *cand, const float *rn_max, int32_t *ref_idx,
                                 uint8_t *copy_flag, int32_t *status, cudaStream_t s)
{
    (void)status;
    long long warps = (long long)g.LB * g.T;
    unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    ProfScope prof("topk_finalize", s);
    if (ref_exact_is_f32)
        k_topk_finalize<float><<<blocks, 256, 0, s>>>(
            (const float *)kv, (const float *)ref_exact, pool->ref_slot, pool->pool_size, cand,
            rn_max, g.LB, g.T, g.W, g.n_ref, g.k, g.max_chunks, (int4 *)ref_idx, copy_flag);
    else
        k_topk_finalize<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16 *)kv, (const __nv_bfloat16 *)ref_exact, pool->ref_slot,
            pool->pool_size, cand, rn_max, g.LB, g.T, g.W, g.n_ref, g.k, g.max_chunks,
            (int4 *)ref_idx, copy_flag);
    return cudaGetLastError();
}

}  // namespace rkv
