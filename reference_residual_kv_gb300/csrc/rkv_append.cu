// rkv_append.cu -- decode-time write of one new token per (layer, sequence)
// [RKV §2.7 = Sec. IV-C, step 4 of a decode step: the new token's state enters the
// cache, directly at a reference position, otherwise encoded]:
//   reference position: its row joins the pool (rkv_pool.cu) and its record is the
//     reference record (own slot, z = 0);
//   otherwise the write path of one token [RKV §2.2-§2.4]: the k_t nearest references
//     with pos < t by exact squared distance (ties to the lower slot), their mean in KV
//     space, z = f_c(kv) - f_c(mean), group quantisation.
// With one token per layer-sequence the compressor is a set of matrix-vector products
// whose cost is reading W_c1, W_c2, W_c3 once; they run on CUDA cores in fp32:
//   k_app_dist    (pool slices x lb): exact distances, a top-k per slice
//   k_app_select  (lb): merge the slices, write ref_idx, form the mean (fp32)
//   k_app_h       (d_ff / 8 x lb): dh_f = Swish(x W1_f) (x W2_f) - Swish(m W1_f) (m W2_f)
//   k_app_z       (d_c / 8 x lb):  z_j = dh . W3_j
//   k_app_quant   (lb): group min/max quantisation and packing, as the batch path.
#include "rkv_internal.cuh"
#include "rkv_exact.cuh"

namespace rkv {
namespace {

constexpr int kSlice = 32;        // pool slots per distance CTA
constexpr int kNoSlot = 0x7fffffff;

struct AppWs {                    // workspace carve-up (floats / ints)
    float2 *part;                 // [LB][slices][kMaxK] {d, slot}
    float *mean;                  // [LB][W]
    int *state;                   // [LB] bit 0: reference token, bit 1: exact copy
    float *dh;                    // [LB][d_ff]
    float *z;                     // [LB][d_c]
};

int slices_of(const Geometry &g) { return g.n_ref > 0 ? (g.n_ref + kSlice - 1) / kSlice : 1; }

AppWs carve(const Geometry &g, void *ws)
{
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    uint8_t *b = (uint8_t *)ws;
    AppWs w;
    size_t o = 0;
    w.part = (float2 *)(b + o); o += up((size_t)g.LB * slices_of(g) * kMaxK * sizeof(float2));
    w.mean = (float *)(b + o); o += up((size_t)g.LB * g.W * sizeof(float));
    w.state = (int *)(b + o); o += up((size_t)g.LB * sizeof(int));
    w.dh = (float *)(b + o); o += up((size_t)g.LB * g.d_ff * sizeof(float));
    w.z = (float *)(b + o);
    return w;
}

template <typename TX, typename TR>
__global__ void __launch_bounds__(256)
k_app_dist(const TX *__restrict__ kv_new, int t, const int32_t *__restrict__ ref_slot,
           const int32_t *__restrict__ pool_size, const TR *__restrict__ ref_vec, int W, int n_ref,
           int slices, float2 *__restrict__ part)
{
    __shared__ float sd[8][kMaxK];
    __shared__ int ss[8][kMaxK];
    const int s = blockIdx.x, lb = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pool = ref_slot[t] >= 0 ? 0 : pool_size[t];
    const int m0 = s * kSlice, m1 = min(pool, m0 + kSlice);
    const TX *x = kv_new + (size_t)lb * W;
    const TR *rb = ref_vec + (size_t)lb * n_ref * W;
    float be[kMaxK];
    int bs[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) { be[j] = INFINITY; bs[j] = kNoSlot; }
    // two of the warp's references at a time (their loads in flight together)
    for (int m = m0 + warp; m < m1; m += 16) {
        if (m + 8 < m1) {
            float d0, d1;
            warp_sqdist2(x, rb + (size_t)m * W, rb + (size_t)(m + 8) * W, W, lane, d0, d1);
            list_insert<kMaxK>(be, bs, d0, m);
            list_insert<kMaxK>(be, bs, d1, m + 8);
        } else {
            list_insert<kMaxK>(be, bs, warp_sqdist(x, rb + (size_t)m * W, W, lane), m);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) { sd[warp][j] = be[j]; ss[warp][j] = bs[j]; }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float fe[kMaxK];
        int fs[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) { fe[j] = INFINITY; fs[j] = kNoSlot; }
        for (int w = 0; w < 8; ++w)
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) list_insert<kMaxK>(fe, fs, sd[w][j], ss[w][j]);
        float2 *dst = part + ((size_t)lb * slices + s) * kMaxK;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) dst[j] = make_float2(fe[j], __int_as_float(fs[j]));
    }
}

template <typename TR>
__device__ __forceinline__ float ref_value(const TR *p);
template <> __device__ __forceinline__ float ref_value<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ref_value<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}
template <> __device__ __forceinline__ float ref_value<uint8_t>(const uint8_t *p)
{
    __nv_fp8_e4m3 q;
    q.__x = *p;
    return (float)q;
}

template <typename TR>
__global__ void __launch_bounds__(256)
k_app_select(int t, int k, const int32_t *__restrict__ ref_slot, const int32_t *__restrict__ pool_size,
             const TR *__restrict__ ref_vec, int W, int n_ref, int T, int slices,
             const float2 *__restrict__ part, int4 *__restrict__ ref_idx, float *__restrict__ mean,
             int *__restrict__ state)
{
    __shared__ int ch[kMaxK];
    __shared__ int info[2];       // k_t, state
    const int lb = blockIdx.x;
    const int own = ref_slot[t];
    float fe[kMaxK];
    int fs[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) { fe[j] = INFINITY; fs[j] = kNoSlot; }
    if (own < 0 && threadIdx.x < 32) {
        // the slices' candidates, merged by the first warp: lane l keeps the k best of
        // entries l, l + 32, ..., then five butterfly rounds merge the lanes' lists
        // ((distance, slot) is a total order, so the k best are those of a serial merge)
        const int lane = threadIdx.x;
        const int total = ((pool_size[t] + kSlice - 1) / kSlice) * kMaxK;
        const float2 *src = part + (size_t)lb * slices * kMaxK;
        for (int i = lane; i < total; i += 32) {
            const float2 e = src[i];
            list_insert<kMaxK>(fe, fs, e.x, __float_as_int(e.y));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float pe[kMaxK];
            int ps[kMaxK];
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) {
                pe[j] = __shfl_xor_sync(0xffffffffu, fe[j], o);
                ps[j] = __shfl_xor_sync(0xffffffffu, fs[j], o);
            }
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) list_insert<kMaxK>(fe, fs, pe[j], ps[j]);
        }
    }
    if (threadIdx.x == 0) {
        int c[kMaxK] = {kNoSlot, kNoSlot, kNoSlot, kNoSlot};
        int kt = 0, st = 0;
        if (own >= 0) {
            c[0] = own;
            st = 1;
        } else {
            const int pool = pool_size[t];
            kt = min(k, pool);
            bool same = kt > 0;
#pragma unroll
            for (int j = 0; j < kMaxK; ++j)
                if (j < kt) { c[j] = fs[j]; same &= fe[j] == 0.0f; }
            st = same ? 2 : 0;           // every chosen reference equals the token: z = 0
        }
        // ascending slots, -1 padded
#pragma unroll
        for (int i = 0; i < kMaxK; ++i)
#pragma unroll
            for (int j = 0; j + 1 < kMaxK - i; ++j)
                if (c[j] > c[j + 1]) { const int tmp = c[j]; c[j] = c[j + 1]; c[j + 1] = tmp; }
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) { if (c[j] == kNoSlot) c[j] = -1; ch[j] = c[j]; }
        ref_idx[(size_t)lb * T + t] = make_int4(c[0], c[1], c[2], c[3]);
        info[0] = kt;
        info[1] = st;
        state[lb] = st;
    }
    __syncthreads();
    // the mean of the chosen references in KV space: fp32 sum in ascending slot order,
    // times 1/k_t (reference tokens and exact copies do not need it)
    const int kt = info[0];
    if (info[1] != 0) return;
    const float inv = kt > 0 ? 1.0f / (float)kt : 0.0f;
    const TR *rb = ref_vec + (size_t)lb * n_ref * W;
#pragma unroll 4
    for (int c = threadIdx.x; c < W; c += blockDim.x) {
        float v[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) v[j] = j < kt ? ref_value(rb + (size_t)ch[j] * W + c) : 0.0f;
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
            if (j < kt) acc += v[j];
        mean[(size_t)lb * W + c] = acc * inv;
    }
}

__device__ __forceinline__ float swish(float u) { return u / (1.0f + expf(-u)); }

// One warp per d_ff column f: the four dot products of length W.
template <typename TX>
__global__ void __launch_bounds__(256)
k_app_h(const TX *__restrict__ kv_new, const TX *__restrict__ W1t, const TX *__restrict__ W2t,
        int W, int d_ff, int B, const float *__restrict__ mean, const int *__restrict__ state,
        float *__restrict__ dh)
{
    const int lane = threadIdx.x & 31;
    const int f = blockIdx.x * 8 + (threadIdx.x >> 5), lb = blockIdx.y;
    if (f >= d_ff) return;
    float *out = dh + (size_t)lb * d_ff + f;
    if (state[lb] != 0) {                     // reference token or exact copy: z = 0
        if (lane == 0) *out = 0.0f;
        return;
    }
    const TX *x = kv_new + (size_t)lb * W;
    const float *m = mean + (size_t)lb * W;
    const size_t wrow = ((size_t)(lb / B) * d_ff + f) * W;
    float a1 = 0.0f, a2 = 0.0f, b1 = 0.0f, b2 = 0.0f;
    // 8 consecutive coordinates per lane and step (16-byte loads of bf16 rows); four
    // steps' loads in flight at once
#pragma unroll 4
    for (int c = lane * 8; c < W; c += 256) {
        float w1[8], w2[8], xv[8], mv[8];
        Vec8<TX>::load(W1t + wrow + c, w1);
        Vec8<TX>::load(W2t + wrow + c, w2);
        Vec8<TX>::load(x + c, xv);
        Vec8<float>::load(m + c, mv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            a1 = fmaf(xv[j], w1[j], a1);
            a2 = fmaf(xv[j], w2[j], a2);
            b1 = fmaf(mv[j], w1[j], b1);
            b2 = fmaf(mv[j], w2[j], b2);
        }
    }
    a1 = warp_tree_sum(a1);
    a2 = warp_tree_sum(a2);
    b1 = warp_tree_sum(b1);
    b2 = warp_tree_sum(b2);
    if (lane == 0) *out = swish(a1) * a2 - swish(b1) * b2;
}

// One warp per output j of W_c3.
template <typename TX>
__global__ void __launch_bounds__(256)
k_app_z(const TX *__restrict__ W3t, int d_ff, int d_c, int B, const float *__restrict__ dh,
        float *__restrict__ z)
{
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5), lb = blockIdx.y;
    if (j >= d_c) return;
    const float *h = dh + (size_t)lb * d_ff;
    const TX *w = W3t + ((size_t)(lb / B) * d_c + j) * d_ff;
    float acc = 0.0f;
#pragma unroll 4
    for (int f = lane * 8; f < d_ff; f += 256) {
        float hv[8], wv[8];
        Vec8<float>::load(h + f, hv);
        Vec8<TX>::load(w + f, wv);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = fmaf(hv[j], wv[j], acc);
    }
    acc = warp_tree_sum(acc);
    if (lane == 0) z[(size_t)lb * d_c + j] = acc;
}

// One thread per group of 32 coordinates.
__global__ void k_app_quant(int t, int T, int d_c, int bits, const float *__restrict__ z,
                            uint8_t *__restrict__ codes, float2 *__restrict__ hdr, float *__restrict__ z_out)
{
    const int lb = blockIdx.x, g = threadIdx.x;
    if (g >= d_c / 32) return;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = z[(size_t)lb * d_c + g * 32 + j];
    uint32_t wq[4];
    float zmin, delta;
    quant_group32(v, bits, wq, zmin, delta);
    const size_t rec = (size_t)lb * T + t;
    uint8_t *dst = codes + rec * (size_t)(d_c * bits / 8) + g * (bits * 4);
    if (bits == 4) *(uint4 *)dst = make_uint4(wq[0], wq[1], wq[2], wq[3]);
    else *(uint2 *)dst = make_uint2(wq[0], wq[1]);
    hdr[rec * (d_c / 32) + g] = make_float2(zmin, delta);
    if (z_out) {
#pragma unroll
        for (int j = 0; j < 32; ++j) z_out[rec * d_c + g * 32 + j] = v[j];
    }
}

template <typename TX, typename TR>
cudaError_t run_append(const Geometry &g, const TX *kv_new, int t, const rkv_ref_pool *pool,
                       const TX *W1t, const TX *W2t, const TX *W3t, const rkv_cache *cache, void *ws,
                       cudaStream_t s)
{
    AppWs w = carve(g, ws);
    const int slices = slices_of(g);
    const TR *rv = (const TR *)pool->ref_vec;
    cudaError_t e;
    {
        ProfScope prof("append_distance", s);
        k_app_dist<TX, TR><<<dim3(slices, g.LB), 256, 0, s>>>(kv_new, t, pool->ref_slot, pool->pool_size,
                                                              rv, g.W, g.n_ref, slices, w.part);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        ProfScope prof("append_select", s);
        k_app_select<TR><<<g.LB, 256, 0, s>>>(t, g.k, pool->ref_slot, pool->pool_size, rv, g.W, g.n_ref,
                                              g.T, slices, w.part, (int4 *)cache->ref_idx, w.mean, w.state);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        ProfScope prof("append_swiglu", s);
        k_app_h<TX><<<dim3((g.d_ff + 7) / 8, g.LB), 256, 0, s>>>(kv_new, W1t, W2t, g.W, g.d_ff, g.B,
                                                                w.mean, w.state, w.dh);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        ProfScope prof("append_z", s);
        k_app_z<TX><<<dim3((g.d_c + 7) / 8, g.LB), 256, 0, s>>>(W3t, g.d_ff, g.d_c, g.B, w.dh, w.z);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ProfScope prof("append_quant", s);
    k_app_quant<<<g.LB, 32 * ((g.d_c / 32 + 31) / 32), 0, s>>>(t, g.T, g.d_c, g.bits, w.z, cache->codes,
                                                               (float2 *)cache->hdr, nullptr);
    return cudaGetLastError();
}

}  // namespace

size_t append_workspace_bytes(const Geometry &g)
{
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    return up((size_t)g.LB * slices_of(g) * kMaxK * sizeof(float2)) + up((size_t)g.LB * g.W * sizeof(float)) +
           up((size_t)g.LB * sizeof(int)) + up((size_t)g.LB * g.d_ff * sizeof(float)) +
           up((size_t)g.LB * g.d_c * sizeof(float));
}

cudaError_t launch_append(const Geometry &g, const void *kv_new, int t, const rkv_ref_pool *pool,
                          const void *W1t, const void *W2t, const void *W3t, const rkv_cache *cache,
                          void *ws, int32_t *status, cudaStream_t s)
{
    (void)status;
    cudaError_t e = launch_append_ref(g, kv_new, t, pool, s);
    if (e != cudaSuccess) return e;
    if (g.kv_dtype == RKV_F32)
        return run_append<float, float>(g, (const float *)kv_new, t, pool, (const float *)W1t,
                                        (const float *)W2t, (const float *)W3t, cache, ws, s);
    if (g.ref_dtype == RKV_FP8_E4M3)
        return run_append<__nv_bfloat16, uint8_t>(g, (const __nv_bfloat16 *)kv_new, t, pool,
                                                  (const __nv_bfloat16 *)W1t, (const __nv_bfloat16 *)W2t,
                                                  (const __nv_bfloat16 *)W3t, cache, ws, s);
    return run_append<__nv_bfloat16, __nv_bfloat16>(g, (const __nv_bfloat16 *)kv_new, t, pool,
                                                    (const __nv_bfloat16 *)W1t, (const __nv_bfloat16 *)W2t,
                                                    (const __nv_bfloat16 *)W3t, cache, ws, s);
}

}  // namespace rkv
