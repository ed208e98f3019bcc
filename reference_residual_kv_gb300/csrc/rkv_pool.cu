// rkv_pool.cu -- reference schedule and stored references
// [RKV §2.6 = Sec. IV-A fixed stride; §2.4 / §2.5 = Sec. IV-A, IV-B, V-A: references
// are kept uncompressed or as FP8, and every later step uses the stored values].
#include "rkv_internal.cuh"

namespace rkv {

// ref_slot[t], pool_size[t] for t < T and ref_pos[m] for m < n_ref.
__global__ void k_schedule(int T, int stride, int first, int n_ref, int32_t *ref_pos,
                           int32_t *ref_slot, int32_t *pool_size)
{
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < T) {
        int rel = t - first;
        ref_slot[t] = (rel >= 0 && rel % stride == 0) ? rel / stride : -1;
        // references at first + m*stride < t
        pool_size[t] = rel <= 0 ? 0 : (rel + stride - 1) / stride;
    }
    if (t < n_ref) ref_pos[t] = first + t * stride;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp stores one reference row: copy (or FP8-encode) the token's row into pool row
// `row` and take the squared norm of the stored values in fp32.
template <typename TIn, int OUT_FP8>
__device__ __forceinline__ void store_ref_row(const TIn *__restrict__ src, void *ref_vec,
                                              float *__restrict__ ref_sqnorm, size_t row, int W,
                                              int lane)
{
    float acc = 0.0f;
    if constexpr (sizeof(TIn) == 4) {
        float *dst = (float *)ref_vec + row * W;
        for (int c = lane * 4; c < W; c += 128) {
            float4 v = *(const float4 *)(src + c);
            *(float4 *)(dst + c) = v;
            acc += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
    } else {
        for (int c = lane * 8; c < W; c += 256) {
            uint4 raw = *(const uint4 *)(src + c);
            const __nv_bfloat16 *h = (const __nv_bfloat16 *)&raw;
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __bfloat162float(h[j]);
            if constexpr (OUT_FP8) {
                uint8_t b[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    b[j] = (uint8_t)__nv_cvt_float_to_fp8(f[j], __NV_SATFINITE, __NV_E4M3);
                    __nv_fp8_e4m3 q;
                    q.__x = b[j];
                    f[j] = (float)q;
                }
                uint8_t *dst = (uint8_t *)ref_vec + row * W;
                *(uint2 *)(dst + c) = *(const uint2 *)b;
            } else {
                __nv_bfloat16 *dst = (__nv_bfloat16 *)ref_vec + row * W;
                *(uint4 *)(dst + c) = raw;
            }
            float s = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) s += f[j] * f[j];
            acc += s;
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) ref_sqnorm[row] = acc;
}

// One warp per (lb, reference slot).
template <typename TIn, int OUT_FP8>
__global__ void k_build_refs(const TIn *__restrict__ kv, const int32_t *__restrict__ ref_pos,
                             void *ref_vec, float *__restrict__ ref_sqnorm, int LB, int T, int W,
                             int n_ref)
{
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (gw >= (long long)LB * n_ref) return;
    const int lb = (int)(gw / n_ref), m = (int)(gw % n_ref);
    store_ref_row<TIn, OUT_FP8>(kv + ((size_t)lb * T + ref_pos[m]) * W, ref_vec, ref_sqnorm,
                                (size_t)lb * n_ref + m, W, lane);
}

// Single-token write: one warp per lb stores the new token's row if position t is a
// reference position (the schedule is the same for every sequence).
template <typename TIn, int OUT_FP8>
__global__ void k_append_ref(const TIn *__restrict__ kv_new, int t, const int32_t *__restrict__ ref_slot,
                             void *ref_vec, float *__restrict__ ref_sqnorm, int LB, int W, int n_ref)
{
    const int lane = threadIdx.x & 31;
    const int lb = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (lb >= LB) return;
    const int slot = ref_slot[t];
    if (slot < 0) return;
    store_ref_row<TIn, OUT_FP8>(kv_new + (size_t)lb * W, ref_vec, ref_sqnorm, (size_t)lb * n_ref + slot,
                                W, lane);
}

cudaError_t launch_append_ref(const Geometry &g, const void *kv_new, int t, const rkv_ref_pool *pool,
                              cudaStream_t s)
{
    if (g.n_ref == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((g.LB * 32 + 255) / 256);
    ProfScope prof("append_ref", s);
    if (g.kv_dtype == RKV_F32)
        k_append_ref<float, 0><<<blocks, 256, 0, s>>>((const float *)kv_new, t, pool->ref_slot,
                                                      pool->ref_vec, pool->ref_sqnorm, g.LB, g.W, g.n_ref);
    else if (g.ref_dtype == RKV_FP8_E4M3)
        k_append_ref<__nv_bfloat16, 1><<<blocks, 256, 0, s>>>((const __nv_bfloat16 *)kv_new, t, pool->ref_slot,
                                                              pool->ref_vec, pool->ref_sqnorm, g.LB, g.W, g.n_ref);
    else
        k_append_ref<__nv_bfloat16, 0><<<blocks, 256, 0, s>>>((const __nv_bfloat16 *)kv_new, t, pool->ref_slot,
                                                              pool->ref_vec, pool->ref_sqnorm, g.LB, g.W, g.n_ref);
    return cudaGetLastError();
}

// Dynamic stride: the positions follow a recurrence, so one thread writes them in
// order (their number grows like log T for alpha > 0) ...
__global__ void k_schedule_dynamic_pos(int T, int stride, int first, double alpha, int n_sink,
                                       int n_ref, int32_t *ref_pos)
{
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    long long p = first;
    for (int m = 0; m < n_ref && p < T; ++m) {
        ref_pos[m] = (int32_t)p;
        p = p + stride + (long long)floor(alpha * (double)(p - n_sink));
    }
}

// ... and every token finds its pool by binary search: pool_size[t] = #{m: p_m < t}.
__global__ void k_schedule_dynamic_tok(int T, int n_ref, const int32_t *__restrict__ ref_pos,
                                       int32_t *ref_slot, int32_t *pool_size)
{
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    int lo = 0, hi = n_ref;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (ref_pos[mid] < t) lo = mid + 1;
        else hi = mid;
    }
    pool_size[t] = lo;
    ref_slot[t] = (lo < n_ref && ref_pos[lo] == t) ? lo : -1;
}

cudaError_t launch_build_schedule(const Geometry &g, const rkv_ref_pool *pool, cudaStream_t s)
{
    ProfScope prof("build_schedule", s);
    if (g.alpha == 0.0) {
        int n = g.T > g.n_ref ? g.T : g.n_ref;
        k_schedule<<<(n + 255) / 256, 256, 0, s>>>(g.T, g.stride, g.first, g.n_ref, pool->ref_pos,
                                                   pool->ref_slot, pool->pool_size);
    } else {
        k_schedule_dynamic_pos<<<1, 32, 0, s>>>(g.T, g.stride, g.first, g.alpha, g.n_sink, g.n_ref,
                                                pool->ref_pos);
        k_schedule_dynamic_tok<<<(g.T + 255) / 256, 256, 0, s>>>(g.T, g.n_ref, pool->ref_pos,
                                                                pool->ref_slot, pool->pool_size);
    }
    return cudaGetLastError();
}

cudaError_t launch_build_refs(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                              cudaStream_t s)
{
    long long warps = (long long)g.LB * g.n_ref;
    unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    ProfScope prof("build_refs", s);
    if (g.kv_dtype == RKV_F32)
        k_build_refs<float, 0><<<blocks, 256, 0, s>>>((const float *)kv, pool->ref_pos,
                                                      pool->ref_vec, pool->ref_sqnorm, g.LB, g.T,
                                                      g.W, g.n_ref);
    else if (g.ref_dtype == RKV_FP8_E4M3)
        k_build_refs<__nv_bfloat16, 1><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16 *)kv, pool->ref_pos, pool->ref_vec, pool->ref_sqnorm, g.LB, g.T,
            g.W, g.n_ref);
    else
        k_build_refs<__nv_bfloat16, 0><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16 *)kv, pool->ref_pos, pool->ref_vec, pool->ref_sqnorm, g.LB, g.T,
            g.W, g.n_ref);
    return cudaGetLastError();
}

// ---- compress-time preparation -------------------------------------------------
// FP8 references decoded to bf16 (exact: every E4M3 value is a bf16 value) so that
// the tensor cores can read them next to bf16 tokens.
__global__ void k_decode_fp8_refs(const uint8_t *__restrict__ src, __nv_bfloat16 *__restrict__ dst,
                                  long long n8)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (long long)gridDim.x * blockDim.x) {
        uint2 raw = ((const uint2 *)src)[i];
        const uint8_t *b = (const uint8_t *)&raw;
        __align__(16) __nv_bfloat16 o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            __nv_fp8_e4m3 q;
            q.__x = b[j];
            o[j] = __float2bfloat16_rn((float)q);
        }
        ((uint4 *)dst)[i] = *(const uint4 *)o;
    }
}

// rn_max[lb] = max_m ref_sqnorm[lb][m]  (scale of the distance-expansion error bound);
// block 0 also clears the all-zero projection rows (if given)
__global__ void k_rn_max(const float *__restrict__ rn, float *__restrict__ out, int n_ref,
                         float *__restrict__ z1, float *__restrict__ z2, int d_ff)
{
    __shared__ float sm[32];
    const int lb = blockIdx.x;
    if (lb == 0 && z1) {
        for (int i = threadIdx.x; i < d_ff; i += blockDim.x) { z1[i] = 0.0f; z2[i] = 0.0f; }
    }
    float v = 0.0f;
    for (int m = threadIdx.x; m < n_ref; m += blockDim.x) v = fmaxf(v, rn[(size_t)lb * n_ref + m]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < (blockDim.x >> 5) ? sm[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (threadIdx.x == 0) out[lb] = v;
    }
}

cudaError_t launch_prep_refs(const Geometry &g, const rkv_ref_pool *pool, void *ref_mma,
                             float *rn_max, float *zero_row1, float *zero_row2, cudaStream_t s)
{
    if (g.n_ref == 0) {
        cudaError_t e = cudaMemsetAsync(rn_max, 0, sizeof(float) * g.LB, s);
        if (e == cudaSuccess && zero_row1) e = cudaMemsetAsync(zero_row1, 0, sizeof(float) * g.d_ff, s);
        if (e == cudaSuccess && zero_row2) e = cudaMemsetAsync(zero_row2, 0, sizeof(float) * g.d_ff, s);
        return e;
    }
    if (g.ref_dtype == RKV_FP8_E4M3) {
        long long n8 = (long long)g.LB * g.n_ref * g.W / 8;
        int blocks = (int)((n8 + 255) / 256);
        if (blocks > 4 * 1024) blocks = 4 * 1024;
        ProfScope prof("decode_fp8_refs", s);
        k_decode_fp8_refs<<<blocks, 256, 0, s>>>((const uint8_t *)pool->ref_vec,
                                                 (__nv_bfloat16 *)ref_mma, n8);
    }
    ProfScope prof("ref_norm_max", s);
    k_rn_max<<<g.LB, 256, 0, s>>>(pool->ref_sqnorm, rn_max, g.n_ref, zero_row1, zero_row2, g.d_ff);
    return cudaGetLastError();
}

}  // namespace rkv
