// rkv_topk.cu -- final reference choice per token [RKV §2.2 = Sec. IV-A]:
//   R_t = the k_t = min(k, pool_size[t]) references with pos < t nearest to kv_t in
//   squared L2, ties to the lower slot, stored in ascending slot order.
//
// The tensor-core pass ranks references by the expansion ||r||^2 - 2 x.r (the
// ||x||^2 term is common to a row); every work item leaves two sorted lists of its
// kList best per token.  Here one thread per token merges those lists and decides
// (k_topk_select):
//   * if the k-th/(k+1)-th expansion gap exceeds twice the expansion error bound
//     E = kTau (rmax + 2 sqrt(||x||^2 rmax)), rmax = max ||r||^2 of the sequence,
//     the expansion's top-k is the exact top-k;
//   * else, if every possible member of the exact top-k is among the entries (no
//     full list ends inside the band e <= e_k + 2E), the entries inside the band are
//     re-ranked by exact distances: the token goes on a queue that k_topk_rerank serves
//     with one warp per token (two distances in flight), so that warps holding many such
//     tokens do not serialise the pass;
//   * else every reference of the pool is scanned with exact distances.
// It also flags tokens that are bit-identical to every chosen reference (checked with
// exact distances on the same queue, only where the expansion allows it): their mean
// equals the token exactly, so z = 0 exactly [RKV §2.3], which the encoder then
// writes directly (the tensor cores need not round the token's and the
// references' projections identically, since they sit in different tile rows).
// Exact distances sum (x - r)^2 in fp32: for bf16 data x - r is exact, each group of
// 8 squares is added as a tree, a lane keeps four partial sums over its groups, and the
// warp adds its lanes as a tree.
// Without candidates (the fp32 path) every token takes the full scan, one warp per
// token.  On the tensor-core path the (rare) full scans are deferred to
// k_topk_fullscan: the token is appended to a list and a whole block scans its pool,
// eight warps in parallel (near-tied clusters of FP8-rounded references otherwise
// leave single warps scanning thousands of references one after another).
#include "rkv_internal.cuh"
#include "rkv_exact.cuh"

namespace rkv {

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

constexpr int kNoSlot = 0x7fffffff;

// Writes a token's choice: the chosen slots in ascending order, -1 for unused places.
__device__ __forceinline__ void store_choice(int4 *ref_idx, uint8_t *copy_flag, long long g,
                                             const int (&c)[kMaxK], int same)
{
    int a[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) a[j] = c[j];
#pragma unroll
    for (int i = 0; i < kMaxK; ++i)
#pragma unroll
        for (int j = 0; j + 1 < kMaxK - i; ++j)
            if (a[j] > a[j + 1]) { const int tmp = a[j]; a[j] = a[j + 1]; a[j + 1] = tmp; }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) a[j] = a[j] == kNoSlot ? -1 : a[j];
    ref_idx[g] = make_int4(a[0], a[1], a[2], a[3]);
    copy_flag[g] = (uint8_t)same;
}

// fp32 path: one warp per token scans its whole pool with exact distances.
template <typename T>
__global__ void __launch_bounds__(256)
k_topk_scan_warp(const T *__restrict__ kv, const T *__restrict__ refs,
                 const int32_t *__restrict__ ref_slot, const int32_t *__restrict__ pool_size,
                 int LB, int T_, int W, int n_ref, int k, int4 *__restrict__ ref_idx,
                 uint8_t *__restrict__ copy_flag)
{
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (gw >= (long long)LB * T_) return;
    const int lb = (int)(gw / T_), t = (int)(gw % T_);
    const int own = ref_slot[t];
    const int pool = pool_size[t];
    const T *x = kv + (size_t)gw * W;
    const T *rb = refs + (size_t)lb * n_ref * W;
    float be[kMaxK];
    int bs[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) { be[j] = INFINITY; bs[j] = kNoSlot; }
    int same = 0;
    if (own >= 0) {
        bs[0] = own;
    } else {
        for (int s = 0; s < pool; ++s) {
            const float d = warp_sqdist(x, rb + (size_t)s * W, W, lane);
            list_insert<kMaxK>(be, bs, d, s);
        }
        same = pool > 0;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) same &= (j >= pool) || be[j] == 0.0f;
            else bs[j] = kNoSlot;
        }
    }
    if (lane == 0) store_choice(ref_idx, copy_flag, gw, bs, same);
}

// Tensor-core path.  One thread per token makes the decision from its work items'
// sorted lists (a merge of list heads with early exit, so it reads only the entries that
// can enter the top k + 1); the few tokens that need exact distances (a re-rank inside
// the band, or the confirmation of an exact copy) are then served one after another by
// the whole warp; tokens whose candidates may be incomplete go to the full-scan list.
template <typename T>
__global__ void __launch_bounds__(256)
k_topk_select(const T *__restrict__ kv, const T *__restrict__ refs,
              const int32_t *__restrict__ ref_slot, const int32_t *__restrict__ pool_size,
              const float2 *__restrict__ cand, const float *__restrict__ xnorm,
              const float *__restrict__ rn_max, int LB, int T_, int W, int n_ref, int k,
              int max_chunks, int4 *__restrict__ ref_idx, uint8_t *__restrict__ copy_flag,
              int32_t *__restrict__ scan_list, int32_t *__restrict__ scan_count,
              int2 *__restrict__ rr_list, int32_t *__restrict__ rr_count)
{
    enum { kNone = 0, kDone, kRerank, kCopyCheck, kFull };
    const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    int state = kNone, lb = 0, nlists = 0;
    int ch[kMaxK] = {kNoSlot, kNoSlot, kNoSlot, kNoSlot};
    float band = 0.0f;
    if (gt < (long long)LB * T_) {
        lb = (int)(gt / T_);
        const int t = (int)(gt % T_);
        const int own = ref_slot[t];
        const int pool = pool_size[t];
        if (own >= 0) {
            ch[0] = own;
            state = kDone;
        } else if (pool <= k) {
            // every reference of the pool is chosen; the token can equal all of them only
            // if the expansion puts each within the error bound of distance 0 (the lists
            // hold every pool member, pool <= k < kList)
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) ch[j] = j < pool ? j : kNoSlot;
            state = kDone;
            if (pool > 0) {
                const float4 *cp = (const float4 *)(cand + (size_t)gt * max_chunks * kCand);
                float e_max = -INFINITY;
                int seen = 0;
#pragma unroll
                for (int j = 0; j < kCand / 2; ++j) {
                    const float4 c = cp[j];
                    if (__float_as_int(c.y) >= 0 && __float_as_int(c.y) < pool) { e_max = fmaxf(e_max, c.x); ++seen; }
                    if (__float_as_int(c.w) >= 0 && __float_as_int(c.w) < pool) { e_max = fmaxf(e_max, c.z); ++seen; }
                }
                const float xn = xnorm[gt];
                const float rm = rn_max[lb];
                const float E = kTau * (rm + 2.0f * sqrtf(xn * rm));
                if (seen != pool || xn + e_max <= 2.0f * E) state = kCopyCheck;
            }
        } else {
            const int nch = (dist_ntiles(pool_size, T_, t / kTileM) + kDistChunk - 1) / kDistChunk;
            nlists = 2 * nch;
            const float4 *cp = (const float4 *)(cand + (size_t)gt * max_chunks * kCand);
            float te[kMaxK + 1];
            int ts[kMaxK + 1];
#pragma unroll
            for (int j = 0; j <= kMaxK; ++j) { te[j] = INFINITY; ts[j] = kNoSlot; }
            float e_last = INFINITY;   // smallest last entry of a full list
            for (int item = 0; item < nch; ++item) {
                // the work item's two sorted lists, all their float4 loads in flight at once
                float4 e4[kCand / 2];
#pragma unroll
                for (int j = 0; j < kCand / 2; ++j) e4[j] = cp[item * (kCand / 2) + j];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 tail = e4[h * (kList / 2) + kList / 2 - 1];
                    if (__float_as_int(tail.w) >= 0) e_last = fminf(e_last, tail.z);
#pragma unroll
                    for (int j = 0; j < kList / 2; ++j) {
                        const float4 c = e4[h * (kList / 2) + j];
                        const int s0 = __float_as_int(c.y), s1 = __float_as_int(c.w);
                        if (s0 < 0 || !key_less(c.x, s0, te[kMaxK], ts[kMaxK])) break;
                        list_insert<kMaxK + 1>(te, ts, c.x, s0);
                        if (s1 < 0 || !key_less(c.z, s1, te[kMaxK], ts[kMaxK])) break;
                        list_insert<kMaxK + 1>(te, ts, c.z, s1);
                    }
                }
            }
            const float xn = xnorm[gt];
            const float rm = rn_max[lb];
            const float E = kTau * (rm + 2.0f * sqrtf(xn * rm));
            float e_k = te[0], e_k1 = te[1];   // k-th and (k+1)-th expansion values
#pragma unroll
            for (int j = 1; j < kMaxK; ++j)
                if (j == k - 1) { e_k = te[j]; e_k1 = te[j + 1]; }
            if (e_k1 - e_k > 2.0f * E) {
                // the expansion's top-k is the exact top-k; an exact copy of all k is
                // possible only if the distance estimate is within the error bound
#pragma unroll
                for (int j = 0; j < kMaxK; ++j) ch[j] = j < k ? ts[j] : kNoSlot;
                state = xn + e_k <= 2.0f * E ? kCopyCheck : kDone;
            } else {
                // every reference that can reach the exact top-k has expansion <= band;
                // a full list whose last entry is inside the band may have dropped some
                band = e_k + 2.0f * E;
                state = e_last <= band ? kFull : kRerank;
            }
        }
        if (state == kDone) store_choice(ref_idx, copy_flag, gt, ch, 0);
        if (state == kFull) scan_list[atomicAdd(scan_count, 1)] = (int32_t)gt;
        if (state == kCopyCheck) {
            // the choice is final; k_topk_rerank confirms or clears the copy flag
            store_choice(ref_idx, copy_flag, gt, ch, 0);
            rr_list[atomicAdd(rr_count, 1)] = make_int2((int)((uint32_t)gt | 0x80000000u), 0);
        }
        if (state == kRerank) rr_list[atomicAdd(rr_count, 1)] = make_int2((int)gt, __float_as_int(band));
    }
}

// The queued tokens of k_topk_select, one warp each: a copy check computes the exact
// distances to the chosen references (the copy flag is set only if all are 0); a
// re-rank computes the exact distances of the list entries inside the band, two at a
// time, and keeps the k nearest (ties to the lower slot).
template <typename T>
__global__ void __launch_bounds__(256)
k_topk_rerank(const T *__restrict__ kv, const T *__restrict__ refs,
              const int32_t *__restrict__ pool_size, const float2 *__restrict__ cand, int T_, int W,
              int n_ref, int k, int max_chunks, const int2 *__restrict__ rr_list,
              const int32_t *__restrict__ rr_count, int4 *__restrict__ ref_idx,
              uint8_t *__restrict__ copy_flag)
{
    const int lane = threadIdx.x & 31;
    const int nw = (int)((gridDim.x * blockDim.x) >> 5);
    const int n = *rr_count;
    for (int e = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); e < n; e += nw) {
        const int2 ent = rr_list[e];
        const bool copy = ent.x < 0;
        const long long g = (long long)((uint32_t)ent.x & 0x7fffffffu);
        const int glb = (int)(g / T_), t = (int)(g % T_);
        const T *x = kv + (size_t)g * W;
        const T *rb = refs + (size_t)glb * n_ref * W;
        int cs[kMaxK];
        int same = 1;
        if (copy) {
            const int4 c4 = ref_idx[g];
            const int cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int j = 0; j < kMaxK; ++j)
                if (cc[j] >= 0) same &= warp_sqdist(x, rb + (size_t)cc[j] * W, W, lane) == 0.0f;
            if (lane == 0) copy_flag[g] = (uint8_t)same;
            continue;
        }
        const float bd = __int_as_float(ent.y);
        const int nch = (dist_ntiles(pool_size, T_, t / kTileM) + kDistChunk - 1) / kDistChunk;
        const int nent = 2 * nch * kList;
        const float2 *cp = cand + (size_t)g * max_chunks * kCand;
        float be[kMaxK];
        int bs[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) { be[j] = INFINITY; bs[j] = kNoSlot; }
        for (int b = 0; b < nent; b += 32) {
            float ev = INFINITY;
            int sl = -1;
            if (b + lane < nent) {
                const float2 c = cp[b + lane];
                ev = c.x;
                sl = __float_as_int(c.y);
            }
            unsigned in = __ballot_sync(0xffffffffu, sl >= 0 && ev <= bd);
            while (in) {
                const int q0 = __ffs(in) - 1;
                in &= in - 1;
                const int s0 = __shfl_sync(0xffffffffu, sl, q0);
                if (in) {
                    const int q1 = __ffs(in) - 1;
                    in &= in - 1;
                    const int s1 = __shfl_sync(0xffffffffu, sl, q1);
                    float d0, d1;
                    warp_sqdist2(x, rb + (size_t)s0 * W, rb + (size_t)s1 * W, W, lane, d0, d1);
                    list_insert<kMaxK>(be, bs, d0, s0);
                    list_insert<kMaxK>(be, bs, d1, s1);
                } else {
                    list_insert<kMaxK>(be, bs, warp_sqdist(x, rb + (size_t)s0 * W, W, lane), s0);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            cs[j] = j < k ? bs[j] : kNoSlot;
            if (j < k) same &= be[j] == 0.0f;
        }
        if (lane == 0) store_choice(ref_idx, copy_flag, g, cs, same);
    }
}

// One block per listed token: its eight warps scan slots w, w+8, ... of the pool with
// exact distances, each keeping a top-k; warp 0 merges the eight lists.
template <typename T>
__global__ void __launch_bounds__(256)
k_topk_fullscan(const T *__restrict__ kv, const T *__restrict__ refs,
                const int32_t *__restrict__ pool_size, int T_, int W, int n_ref, int k,
                const int32_t *__restrict__ scan_list, const int32_t *__restrict__ scan_count,
                int4 *__restrict__ ref_idx, uint8_t *__restrict__ copy_flag)
{
    __shared__ float sd[8][kMaxK];
    __shared__ int ss[8][kMaxK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = *scan_count;
    for (int e = blockIdx.x; e < n; e += gridDim.x) {
        const int flat = scan_list[e];
        const int lb = flat / T_, t = flat % T_;
        const int pool = pool_size[t];
        const T *x = kv + (size_t)flat * W;
        const T *rb = refs + (size_t)lb * n_ref * W;
        float be[kMaxK];
        int bs[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) { be[j] = INFINITY; bs[j] = 0x7fffffff; }
        for (int s = warp; s < pool; s += 8) {
            const float d = warp_sqdist(x, rb + (size_t)s * W, W, lane);
            list_insert<kMaxK>(be, bs, d, s);
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) { sd[warp][j] = be[j]; ss[warp][j] = bs[j]; }
        }
        __syncthreads();
        if (warp == 0) {
            float d = sd[lane >> 2][lane & 3];
            int sl = ss[lane >> 2][lane & 3];
            float cd[kMaxK];
            int cs[kMaxK];
#pragma unroll
            for (int r = 0; r < kMaxK; ++r) {
                float wd = d;
                int ws = sl;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float od = __shfl_xor_sync(0xffffffffu, wd, o);
                    const int os = __shfl_xor_sync(0xffffffffu, ws, o);
                    if (key_less(od, os, wd, ws)) { wd = od; ws = os; }
                }
                cd[r] = wd;
                cs[r] = ws;
                if (sl == ws && d == wd) { d = INFINITY; sl = 0x7fffffff; }
            }
            int same = 1, ch[kMaxK];
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) {
                ch[j] = j < k ? cs[j] : 0x7fffffff;
                if (j < k) same &= cd[j] == 0.0f;
            }
#pragma unroll
            for (int a = 0; a < kMaxK; ++a)
#pragma unroll
                for (int b = 0; b + 1 < kMaxK - a; ++b)
                    if (ch[b] > ch[b + 1]) { int tmp = ch[b]; ch[b] = ch[b + 1]; ch[b + 1] = tmp; }
            if (lane == 0) {
                ref_idx[flat] = make_int4(ch[0], k > 1 ? ch[1] : -1, k > 2 ? ch[2] : -1,
                                          k > 3 ? ch[3] : -1);
                copy_flag[flat] = (uint8_t)same;
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_topk_finalize(const Geometry &g, const void *kv, const void *ref_exact,
                                 int ref_exact_is_f32, const rkv_ref_pool *pool,
                                 const float2 *cand, const float *xnorm, const float *rn_max,
                                 int32_t *ref_idx, uint8_t *copy_flag, int32_t *scan_list,
                                 int32_t *scan_count, int2 *rr_list, int32_t *rr_count,
                                 int32_t *status, cudaStream_t s)
{
    (void)status;
    long long warps = (long long)g.LB * g.T;
    unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    cudaError_t e;
    if (scan_list && (e = cudaMemsetAsync(scan_count, 0, sizeof(int32_t), s)) != cudaSuccess)
        return e;
    if (rr_list && (e = cudaMemsetAsync(rr_count, 0, sizeof(int32_t), s)) != cudaSuccess)
        return e;
    {
        ProfScope prof("topk_finalize", s);
        if (cand) {
            const unsigned tb = (unsigned)(((long long)g.LB * g.T + 255) / 256);
            k_topk_select<__nv_bfloat16><<<tb, 256, 0, s>>>(
                (const __nv_bfloat16 *)kv, (const __nv_bfloat16 *)ref_exact, pool->ref_slot,
                pool->pool_size, cand, xnorm, rn_max, g.LB, g.T, g.W, g.n_ref, g.k,
                g.max_chunks, (int4 *)ref_idx, copy_flag, scan_list, scan_count, rr_list, rr_count);
        } else if (ref_exact_is_f32) {
            k_topk_scan_warp<float><<<blocks, 256, 0, s>>>(
                (const float *)kv, (const float *)ref_exact, pool->ref_slot, pool->pool_size,
                g.LB, g.T, g.W, g.n_ref, g.k, (int4 *)ref_idx, copy_flag);
        } else {
            k_topk_scan_warp<__nv_bfloat16><<<blocks, 256, 0, s>>>(
                (const __nv_bfloat16 *)kv, (const __nv_bfloat16 *)ref_exact, pool->ref_slot,
                pool->pool_size, g.LB, g.T, g.W, g.n_ref, g.k, (int4 *)ref_idx, copy_flag);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (cand && rr_list) {
        ProfScope prof("topk_rerank", s);
        k_topk_rerank<__nv_bfloat16><<<4 * device_sm_count(), 256, 0, s>>>(
            (const __nv_bfloat16 *)kv, (const __nv_bfloat16 *)ref_exact, pool->pool_size, cand, g.T,
            g.W, g.n_ref, g.k, g.max_chunks, rr_list, rr_count, (int4 *)ref_idx, copy_flag);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (scan_list) {
        ProfScope prof("topk_fullscan", s);
        const int grid = 2 * device_sm_count();
        if (ref_exact_is_f32)
            k_topk_fullscan<float><<<grid, 256, 0, s>>>(
                (const float *)kv, (const float *)ref_exact, pool->pool_size, g.T, g.W, g.n_ref,
                g.k, scan_list, scan_count, (int4 *)ref_idx, copy_flag);
        else
            k_topk_fullscan<__nv_bfloat16><<<grid, 256, 0, s>>>(
                (const __nv_bfloat16 *)kv, (const __nv_bfloat16 *)ref_exact, pool->pool_size, g.T,
                g.W, g.n_ref, g.k, scan_list, scan_count, (int4 *)ref_idx, copy_flag);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace rkv
