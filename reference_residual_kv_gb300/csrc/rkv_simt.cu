// rkv_simt.cu -- the write path for fp32 kv and weights on the CUDA cores.
//
// bf16 inputs take the tensor-core path (rkv_umma.cu).  fp32 inputs keep full fp32
// precision here: every dot product is a chain of fp32 FMAs.  Steps:
//   1. P1 = R W_c1, P2 = R W_c2 for every stored reference R (once per reference);
//   2. top-k by exact distances (rkv_topk.cu, full scan);
//   3. dh_t = Swish(x_t W_c1) ⊙ x_t W_c2 - Swish(p1) ⊙ p2 with p = mean of the chosen
//      references' P rows -- by linearity of x -> x W this is the first layer of
//      f_c evaluated at the KV-space mean [RKV §2.2, §2.3 = Sec. IV-A];
//   4. z_t = dh_t W_c3 = f_c(kv_t) - f_c(mean_t);
//   5. group quantisation [RKV §2.4].
#include "rkv_internal.cuh"

namespace rkv {

template <typename T> __device__ __forceinline__ float ld1(const T *p, size_t i);
template <> __device__ __forceinline__ float ld1<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i)
{
    return __bfloat162float(p[i]);
}

// Gated projection tile: rows [m0, m0+64) of A (lda = W) against d_ff columns
// [f0, f0+32) of W1t and W2t.  MODE 0 writes P1/P2; MODE 1 writes dh.
template <typename T, int MODE>
__global__ void __launch_bounds__(256)
k_simt_gate(const T *__restrict__ A, int rows, int W, int d_ff, int B_,
            const T *__restrict__ W1t, const T *__restrict__ W2t, float *__restrict__ P1,
            float *__restrict__ P2, int n_ref, const int32_t *__restrict__ ref_slot,
            const int4 *__restrict__ ref_idx, const uint8_t *__restrict__ copy_flag,
            float *__restrict__ dh)
{
    constexpr int BM = 64, BN = 32, BK = 32;
    __shared__ float As[BK][BM + 1];
    __shared__ float B1s[BK][BN + 1];
    __shared__ float B2s[BK][BN + 1];
    const int lb = blockIdx.z, layer = lb / B_;
    const int m0 = blockIdx.y * BM, f0 = blockIdx.x * BN;
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const T *Ab = A + (size_t)lb * rows * W;
    const T *W1b = W1t + (size_t)layer * d_ff * W;
    const T *W2b = W2t + (size_t)layer * d_ff * W;
    float a1[4][2] = {}, a2[4][2] = {};
    for (int k0 = 0; k0 < W; k0 += BK) {
        for (int i = tid; i < BM * BK; i += 256) {
            int r = i / BK, c = i % BK;
            int gr = m0 + r, gc = k0 + c;
            As[c][r] = (gr < rows && gc < W) ? ld1(Ab, (size_t)gr * W + gc) : 0.0f;
        }
        for (int i = tid; i < BN * BK; i += 256) {
            int r = i / BK, c = i % BK;
            int gf = f0 + r, gc = k0 + c;
            bool ok = gf < d_ff && gc < W;
            B1s[c][r] = ok ? ld1(W1b, (size_t)gf * W + gc) : 0.0f;
            B2s[c][r] = ok ? ld1(W2b, (size_t)gf * W + gc) : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float av[4], b1[2], b2[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 2; ++j) { b1[j] = B1s[kk][tx * 2 + j]; b2[j] = B2s[kk][tx * 2 + j]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    a1[i][j] = fmaf(av[i], b1[j], a1[i][j]);
                    a2[i][j] = fmaf(av[i], b2[j], a2[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = m0 + ty * 4 + i;
        if (r >= rows) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int f = f0 + tx * 2 + j;
            if (f >= d_ff) continue;
            if (MODE == 0) {
                P1[((size_t)lb * n_ref + r) * d_ff + f] = a1[i][j];
                P2[((size_t)lb * n_ref + r) * d_ff + f] = a2[i][j];
            } else {
                float v = 0.0f;
                if (ref_slot[r] < 0 && !copy_flag[(size_t)lb * rows + r]) {
                    int4 ix = ref_idx[(size_t)lb * rows + r];
                    int sl[4] = {ix.x, ix.y, ix.z, ix.w};
                    float p1 = 0.0f, p2 = 0.0f;
                    int k = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (sl[q] >= 0) {
                            p1 += P1[((size_t)lb * n_ref + sl[q]) * d_ff + f];
                            p2 += P2[((size_t)lb * n_ref + sl[q]) * d_ff + f];
                            ++k;
                        }
                    if (k > 0) { p1 = __fdiv_rn(p1, (float)k); p2 = __fdiv_rn(p2, (float)k); }
                    v = silu(a1[i][j]) * a2[i][j] - silu(p1) * p2;
                }
                dh[((size_t)lb * rows + r) * d_ff + f] = v;
            }
        }
    }
}

// z = dh W_c3 (dh fp32 [LB][T][d_ff], W3t [L][d_c][d_ff]); 64x64 tiles.
template <typename T>
__global__ void __launch_bounds__(256)
k_simt_z(const float *__restrict__ dh, const T *__restrict__ W3t, float *__restrict__ z, int T_,
         int d_ff, int d_c, int B_)
{
    constexpr int BM = 64, BN = 64, BK = 32;
    __shared__ float As[BK][BM + 1];
    __shared__ float Bs[BK][BN + 1];
    const int lb = blockIdx.z, layer = lb / B_;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const float *Ab = dh + (size_t)lb * T_ * d_ff;
    const T *Bb = W3t + (size_t)layer * d_c * d_ff;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d_ff; k0 += BK) {
        for (int i = tid; i < BM * BK; i += 256) {
            int r = i / BK, c = i % BK;
            int gr = m0 + r, gc = k0 + c;
            As[c][r] = (gr < T_ && gc < d_ff) ? Ab[(size_t)gr * d_ff + gc] : 0.0f;
        }
        for (int i = tid; i < BN * BK; i += 256) {
            int r = i / BK, c = i % BK;
            int gn = n0 + r, gc = k0 + c;
            Bs[c][r] = (gn < d_c && gc < d_ff) ? ld1(Bb, (size_t)gn * d_ff + gc) : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { av[i] = As[kk][ty * 4 + i]; bv[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = m0 + ty * 4 + i;
        if (r >= T_) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = n0 + tx * 4 + j;
            if (c < d_c) z[((size_t)lb * T_ + r) * d_c + c] = acc[i][j];
        }
    }
}

// One thread per (lb, token, group of 32): quantise, pack, store the record.
__global__ void k_quant_rows(const float *__restrict__ z, const int32_t *__restrict__ ref_slot,
                             int LB, int T_, int d_c, int bits, uint8_t *__restrict__ codes,
                             float2 *__restrict__ hdr, float *__restrict__ z_out)
{
    const int ng = d_c / 32;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)LB * T_ * ng) return;
    const int g = (int)(i % ng);
    const long long rec = i / ng;
    const int t = (int)(rec % T_);
    const bool is_ref = ref_slot[t] >= 0;
    float v[32];
    const float *src = z + rec * d_c + g * 32;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = is_ref ? 0.0f : src[j];
    uint32_t w[4];
    float zmin, delta;
    quant_group32(v, bits, w, zmin, delta);
    const int pitch = d_c * bits / 8;
    uint8_t *dst = codes + rec * pitch + g * (bits * 4);
    if (bits == 4) *(uint4 *)dst = make_uint4(w[0], w[1], w[2], w[3]);
    else *(uint2 *)dst = make_uint2(w[0], w[1]);
    hdr[rec * ng + g] = make_float2(zmin, delta);
    if (z_out) {
#pragma unroll
        for (int j = 0; j < 32; ++j) z_out[rec * d_c + g * 32 + j] = v[j];
    }
}

cudaError_t launch_simt_compress(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                                 const void *W1t, const void *W2t, const void *W3t,
                                 const rkv_cache *cache, uint8_t *ws, const Workspace &wl,
                                 float *z_out, int32_t *status, cudaStream_t s)
{
    cudaError_t e;
    float *P1 = (float *)(ws + wl.P1), *P2 = (float *)(ws + wl.P2);
    float *rn_max = (float *)(ws + wl.rn_max);
    float *dh = (float *)(ws + wl.dh32), *z = (float *)(ws + wl.z32);
    if ((e = launch_prep_refs(g, pool, nullptr, rn_max, nullptr, nullptr, s)) != cudaSuccess) return e;
    const float *X = (const float *)kv;
    if (g.n_ref > 0) {
        dim3 grid((g.d_ff + 31) / 32, (g.n_ref + 63) / 64, g.LB);
        ProfScope prof("simt_ref_proj", s);
        k_simt_gate<float, 0><<<grid, 256, 0, s>>>((const float *)pool->ref_vec, g.n_ref, g.W,
                                                   g.d_ff, g.B, (const float *)W1t,
                                                   (const float *)W2t, P1, P2, g.n_ref, nullptr,
                                                   nullptr, nullptr, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    uint8_t *copy_flag = ws + wl.copy_flag;
    if ((e = launch_topk_finalize(g, kv, pool->ref_vec, 1, pool, nullptr, nullptr, rn_max,
                                  cache->ref_idx, copy_flag, nullptr, nullptr, nullptr, nullptr,
                                  status, s)) != cudaSuccess)
        return e;
    {
        dim3 grid((g.d_ff + 31) / 32, (g.T + 63) / 64, g.LB);
        ProfScope prof("simt_swiglu_diff", s);
        k_simt_gate<float, 1><<<grid, 256, 0, s>>>(X, g.T, g.W, g.d_ff, g.B, (const float *)W1t,
                                                   (const float *)W2t, P1, P2, g.n_ref,
                                                   pool->ref_slot, (const int4 *)cache->ref_idx,
                                                   copy_flag, dh);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        dim3 grid((g.d_c + 63) / 64, (g.T + 63) / 64, g.LB);
        ProfScope prof("simt_z", s);
        k_simt_z<float><<<grid, 256, 0, s>>>(dh, (const float *)W3t, z, g.T, g.d_ff, g.d_c, g.B);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    long long n = (long long)g.LB * g.T * g.n_groups;
    ProfScope prof("quant_rows", s);
    k_quant_rows<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(z, pool->ref_slot, g.LB, g.T, g.d_c,
                                                            g.bits, cache->codes,
                                                            (float2 *)cache->hdr, z_out);
    return cudaGetLastError();
}

}  // namespace rkv
