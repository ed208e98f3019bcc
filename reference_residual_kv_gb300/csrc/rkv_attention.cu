// rkv_attention.cu -- sparse attention of one decode step over the restored set
// [RKV §2.7 = Sec. IV-C]:
//   o_j = softmax( q_j K^_I^T / sqrt(D) ) V^_I   for each query head j,
// query head j reading key/value head floor(j / (H/N)); I = the selected rows that
// are not padding.  Reading the restored K^ and V^ dominates (2 N D bf16 per token),
// so the pass is bound by HBM and runs on CUDA cores in fp32:
//   k_attn_split    one CTA per (split of the selected rows, KV head, layer-sequence):
//                   each warp keeps an online softmax (running max, sum and weighted
//                   value sum) per query head of the group over its rows, four rows'
//                   loads at a time, D/32 coordinates per lane; the 8 warps merge in shared
//                   memory and write the split's partial (max, sum, D sums).
//   k_attn_combine  one block per (layer-sequence, query head): merges the splits.
#include "rkv_internal.cuh"

#include <math.h>

namespace rkv {
namespace {

constexpr int kMaxG = 8;          // query heads per key/value head
constexpr int kWarps = 8;
constexpr int kRows = 4;          // rows a warp loads at once

template <int EPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *p, float (&x)[EPL])
{
    if constexpr (EPL == 8) {
        const uint4 u = __ldg((const uint4 *)p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[2 * j] = __uint_as_float(w[j] << 16);
            x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
    } else if constexpr (EPL == 4) {
        const uint2 u = __ldg((const uint2 *)p);
        x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const uint32_t u = __ldg((const uint32_t *)p);
        x[0] = __uint_as_float(u << 16); x[1] = __uint_as_float(u & 0xffff0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Partials: [LB][N][splits][G][D + 2] floats = {D weighted sums, max, sum}.
template <int EPL, int GM>
__global__ void __launch_bounds__(32 * kWarps, 2)
k_attn_split(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kh,
             const __nv_bfloat16 *__restrict__ vh, const int32_t *__restrict__ sel, int n_sel,
             int T, int H, int N, int chunk, int splits, float scale, float *__restrict__ part)
{
    constexpr int D = 32 * EPL;
    __shared__ float sm[kWarps][GM][D + 2];
    const int s = blockIdx.x, n = blockIdx.y, lb = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = H / N;
    float qr[GM][EPL], o[GM][EPL], m[GM], l[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) { o[g][e] = 0.0f; qr[g][e] = 0.0f; }
        if (g < G) {
            load_row<EPL>(q + ((size_t)lb * H + n * G + g) * D + lane * EPL, qr[g]);
#pragma unroll
            for (int e = 0; e < EPL; ++e) qr[g][e] *= scale;     // 1/sqrt(D), a power of 2 for D = 64, 256
        }
    }
    const int r0 = s * chunk, r1 = min(n_sel, r0 + chunk);
    const size_t rs = (size_t)N * D;                          // row stride of K^, V^
    // kRows rows per warp and iteration: all their loads are issued before the first
    // score is formed
    for (int rb = r0 + warp * kRows; rb < r1; rb += kWarps * kRows) {
        int t_l = -1;
        if (lane < kRows && rb + lane < r1) t_l = __ldg(sel + (size_t)lb * n_sel + rb + lane);
        float kx[kRows][EPL], vx[kRows][EPL];
        bool ok[kRows];
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int t = __shfl_sync(0xffffffffu, t_l, u);
            ok[u] = t >= 0 && t < T;                          // padding: uniform per warp
            if (ok[u]) {
                const size_t off = ((size_t)lb * n_sel + rb + u) * rs + (size_t)n * D + lane * EPL;
                load_row<EPL>(kh + off, kx[u]);
                load_row<EPL>(vh + off, vx[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            if (!ok[u]) continue;
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g >= G) break;
                float d = 0.0f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d = fmaf(qr[g][e], kx[u][e], d);
                const float sc = warp_sum(d);
                const float mn = fmaxf(m[g], sc);
                const float a = __expf(m[g] - mn), b = __expf(sc - mn);
                l[g] = fmaf(l[g], a, b);
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[g][e] = fmaf(o[g][e], a, b * vx[u][e]);
                m[g] = mn;
            }
        }
    }
    // merge the warps
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g >= G) break;
#pragma unroll
        for (int e = 0; e < EPL; ++e) sm[warp][g][lane * EPL + e] = o[g][e];
        if (lane == 0) { sm[warp][g][D] = m[g]; sm[warp][g][D + 1] = l[g]; }
    }
    __syncthreads();
    for (int g = warp; g < G; g += kWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm[w][g][D]);
        float L = 0.0f, acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.0f;
        for (int w = 0; w < kWarps; ++w) {
            const float f = M == -INFINITY ? 0.0f : __expf(sm[w][g][D] - M);
            L = fmaf(sm[w][g][D + 1], f, L);
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(sm[w][g][lane * EPL + e], f, acc[e]);
        }
        float *dst = part + ((((size_t)lb * N + n) * splits + s) * G + g) * (D + 2);
#pragma unroll
        for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = acc[e];
        if (lane == 0) { dst[D] = M; dst[D + 1] = L; }
    }
}

// One block per (layer-sequence, query head): the maximum over the splits, then each
// warp accumulates a strided subset of the splits, merged in shared memory.
template <int EPL>
__global__ void __launch_bounds__(32 * kWarps)
k_attn_combine(const float *__restrict__ part, int H, int N, int splits, float *__restrict__ out)
{
    constexpr int D = 32 * EPL;
    __shared__ float red[kWarps];
    __shared__ float acc_s[kWarps][D + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lb = blockIdx.x / H, j = blockIdx.x % H;
    const int G = H / N, n = j / G, g = j % G;
    const float *base = part + (((size_t)lb * N + n) * splits) * G * (D + 2) + (size_t)g * (D + 2);
    const size_t ss = (size_t)G * (D + 2);                   // split stride
    float M = -INFINITY;
    for (int s = threadIdx.x; s < splits; s += blockDim.x) M = fmaxf(M, base[s * ss + D]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w]);
    float L = 0.0f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.0f;
    for (int s = warp; s < splits; s += kWarps) {
        const float f = M == -INFINITY ? 0.0f : __expf(base[s * ss + D] - M);
        L = fmaf(base[s * ss + D + 1], f, L);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(base[s * ss + lane * EPL + e], f, acc[e]);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc_s[warp][lane * EPL + e] = acc[e];
    if (lane == 0) acc_s[warp][D] = L;
    __syncthreads();
    if (warp == 0) {
        float Lt = 0.0f, a[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) a[e] = 0.0f;
        for (int w = 0; w < kWarps; ++w) {
            Lt += acc_s[w][D];
#pragma unroll
            for (int e = 0; e < EPL; ++e) a[e] += acc_s[w][lane * EPL + e];
        }
        const float inv = Lt > 0.0f ? 1.0f / Lt : 0.0f;
        float *dst = out + ((size_t)lb * H + j) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dst[e] = a[e] * inv;
    }
}

constexpr int kChunk = 256;       // selected rows per split

template <int EPL>
cudaError_t run_attn(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                     const int32_t *sel, int n_sel, float *out, float *part, cudaStream_t s)
{
    const int splits = (n_sel + kChunk - 1) / kChunk;
    const float scale = (float)(1.0 / sqrt((double)g.D));
    {
        ProfScope prof("attention_split", s);
        if (H / g.N <= 4)
            k_attn_split<EPL, 4><<<dim3(splits, g.N, g.LB), 32 * kWarps, 0, s>>>(
                (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kh, (const __nv_bfloat16 *)vh, sel, n_sel,
                g.T, H, g.N, kChunk, splits, scale, part);
        else if constexpr (EPL < 8)
            k_attn_split<EPL, kMaxG><<<dim3(splits, g.N, g.LB), 32 * kWarps, 0, s>>>(
                (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kh, (const __nv_bfloat16 *)vh, sel, n_sel,
                g.T, H, g.N, kChunk, splits, scale, part);
        else
            return cudaErrorInvalidValue;                     // D = 256 takes groups of <= 4
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    ProfScope prof("attention_combine", s);
    k_attn_combine<EPL><<<(unsigned)(g.LB * H), 32 * kWarps, 0, s>>>(part, H, g.N, splits, out);
    return cudaGetLastError();
}

}  // namespace

size_t attention_workspace_bytes(const Geometry &g, int H, int n_sel)
{
    const size_t splits = (size_t)((n_sel + kChunk - 1) / kChunk);
    return (size_t)g.LB * H * splits * (g.D + 2) * sizeof(float);
}

cudaError_t launch_attention(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                             const int32_t *sel, int n_sel, float *out, void *workspace, cudaStream_t s)
{
    float *part = (float *)workspace;
    switch (g.D) {
    case 64: return run_attn<2>(g, H, q, kh, vh, sel, n_sel, out, part, s);
    case 128: return run_attn<4>(g, H, q, kh, vh, sel, n_sel, out, part, s);
    case 256: return run_attn<8>(g, H, q, kh, vh, sel, n_sel, out, part, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rkv
