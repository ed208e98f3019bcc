// rkv_exact.cuh -- exact squared distances and small sorted lists, shared by the
// top-k finalisation (rkv_topk.cu) and the single-token write (rkv_append.cu) so that
// both rank references by the same fp32 values.
//
// Exact distances sum (x - r)^2 in fp32.  For bf16 tokens and bf16 or FP8 references
// x - r is exact in fp32 (both operands decode exactly); each group of 8 squares is
// added as a tree, a lane keeps four partial sums over its groups, and the warp adds
// its lanes as a tree.
#pragma once

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
template <> struct Vec8<uint8_t> {      // FP8 E4M3 bytes, decoded exactly
    static __device__ __forceinline__ void load(const uint8_t *p, float (&v)[8])
    {
        const uint2 raw = *(const uint2 *)p;
        const uint8_t *b = (const uint8_t *)&raw;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            __nv_fp8_e4m3 q;
            q.__x = b[j];
            v[j] = (float)q;
        }
    }
};

__device__ __forceinline__ float warp_tree_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Adds the squares of the eight bf16 values of one 16-byte word to acc, in element order.
__device__ __forceinline__ float bf16x8_sqsum(const uint4 &v, float acc)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xffff0000u);
        acc = fmaf(a, a, acc);
        acc = fmaf(b, b, acc);
    }
    return acc;
}

template <typename TX, typename TR>
__device__ __forceinline__ float sq8(const TX *x, const TR *r)
{
    float a[8], b[8], s[8];
    Vec8<TX>::load(x, a);
    Vec8<TR>::load(r, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float d = a[j] - b[j];
        s[j] = d * d;
    }
    return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// Exact squared distance of two rows, summed by the whole warp (four 8-element groups
// of a lane in flight at once).
template <typename TX, typename TR = TX>
__device__ __forceinline__ float warp_sqdist(const TX *x, const TR *r, int W, int lane)
{
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int c = lane * 8;
    for (; c + 3 * 256 < W; c += 4 * 256) {
        float p[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) p[u] = sq8(x + c + u * 256, r + c + u * 256);
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] += p[u];
    }
    for (; c < W; c += 256) acc[0] += sq8(x + c, r + c);
    return warp_tree_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
}

// warp_sqdist of two rows against the same x, their loads interleaved; each result is
// formed exactly as warp_sqdist forms it.
template <typename TX, typename TR = TX>
__device__ __forceinline__ void warp_sqdist2(const TX *x, const TR *r0, const TR *r1, int W, int lane,
                                             float &d0, float &d1)
{
    float a0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int c = lane * 8;
    for (; c + 3 * 256 < W; c += 4 * 256) {
        float p0[4], p1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            p0[u] = sq8(x + c + u * 256, r0 + c + u * 256);
            p1[u] = sq8(x + c + u * 256, r1 + c + u * 256);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) { a0[u] += p0[u]; a1[u] += p1[u]; }
    }
    for (; c < W; c += 256) {
        a0[0] += sq8(x + c, r0 + c);
        a1[0] += sq8(x + c, r1 + c);
    }
    d0 = warp_tree_sum((a0[0] + a0[1]) + (a0[2] + a0[3]));
    d1 = warp_tree_sum((a1[0] + a1[1]) + (a1[2] + a1[3]));
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

}  // namespace rkv
