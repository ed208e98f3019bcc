// rkv_gather.cu -- the sparse read [RKV §2.7 = Sec. IV-C]: a sparse-attention step
// names the tokens it needs; for each, read only that token's record (codes, group
// extremes, reference slots) and its stored references, and return the dequantised
// code z~ = q*delta + z_min [RKV §2.4] and the reference mean in KV space [RKV §2.2].
// Groups never span tokens [RKV §2.4], so no unselected neighbour is touched.
//
// Warps take one selected token at a time, persistent for bf16 and fp32 references
// with the next token's record loaded ahead.  Records are read with 8/16-byte loads, references with 8/16-byte loads
// (L2-resident: one sequence's pool is a few MB), outputs are written with 16-byte
// stores.
#include "rkv_internal.cuh"

#include <cuda_fp16.h>

namespace rkv {

// Adds 8 consecutive reference values into 8 fp32 accumulators: one IEEE add per
// element of its exact widening, in the same order as scalar code (bf16 and fp16
// operands go straight into the fp32 add).
__device__ __forceinline__ void add_bf16x2(uint32_t w, float &a0, float &a1)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w));
}
__device__ __forceinline__ void add_f16x2(uint32_t w, float &a0, float &a1)
{
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w));
}

template <typename T> struct RefLoad;
template <> struct RefLoad<float> {
    static __device__ __forceinline__ void add(const float *p, float (&a)[8])
    {
        const float4 u = *(const float4 *)p, v = *(const float4 *)(p + 4);
        const float x[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const float2 r = __fadd2_rn(make_float2(a[j], a[j + 1]), make_float2(x[j], x[j + 1]));
            a[j] = r.x;
            a[j + 1] = r.y;
        }
    }
};
template <> struct RefLoad<__nv_bfloat16> {
    static __device__ __forceinline__ void add(const __nv_bfloat16 *p, float (&a)[8])
    {
        const uint4 raw = *(const uint4 *)p;
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) add_bf16x2(w[j], a[2 * j], a[2 * j + 1]);
    }
};
template <> struct RefLoad<uint8_t> {     // FP8 E4M3: exact in fp16, two per conversion
    static __device__ __forceinline__ void add(const uint8_t *p, float (&a)[8])
    {
        const uint2 raw = *(const uint2 *)p;
        const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            // a word's four bytes: its two 16-bit halves converted to fp16 pairs, then four
            // widening adds
            float *aj = a + 4 * j;
            asm("{\n\t.reg .b16 b0, b1;\n\t.reg .b32 p0, p1;\n\t.reg .f16 f0, f1, f2, f3;\n\t"
                "mov.b32 {b0, b1}, %4;\n\t"
                "cvt.rn.f16x2.e4m3x2 p0, b0;\n\tcvt.rn.f16x2.e4m3x2 p1, b1;\n\t"
                "mov.b32 {f0, f1}, p0;\n\tmov.b32 {f2, f3}, p1;\n\t"
                "add.rn.f32.f16 %0, f0, %0;\n\tadd.rn.f32.f16 %1, f1, %1;\n\t"
                "add.rn.f32.f16 %2, f2, %2;\n\tadd.rn.f32.f16 %3, f3, %3;\n\t}"
                : "+f"(aj[0]), "+f"(aj[1]), "+f"(aj[2]), "+f"(aj[3])
                : "r"(w[j]));
        }
    }
};

// Launch shape by reference dtype (measured): bf16 and fp32 references run persistent
// warps, 3 blocks per SM, each warp walking several tokens with the next token's record
// loaded ahead; FP8 references (half the bytes per reference, more conversions) run one
// warp per token at 4 blocks per SM (64 registers) with four mean steps' loads in flight
// (a sweep of 2..8 blocks and 2..8 steps: 4 and 4 fastest, 4 % ahead of 5 and 4).
template <typename RefT> constexpr bool kPersistent = sizeof(RefT) != 1;
template <typename RefT> constexpr int kGatherBlocks = kPersistent<RefT> ? 3 : 4;

template <typename OutT>
__device__ __forceinline__ void store8(OutT *dst, const float (&v)[8]);
template <> __device__ __forceinline__ void store8<float>(float *dst, const float (&v)[8])
{
    *(float4 *)dst = make_float4(v[0], v[1], v[2], v[3]);
    *(float4 *)(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&v)[8])
{
    __align__(16) __nv_bfloat162 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __float22bfloat162_rn(make_float2(v[2 * j], v[2 * j + 1]));
    *(uint4 *)dst = *(const uint4 *)o;
}

// A selected token's record as a warp holds it: reference slots, and this lane's first
// two code words and group extremes (d_c <= 512 needs no more).
struct GRec {
    int4 ix;
    uint32_t w[2];
    float2 h[2];
};

__device__ __forceinline__ GRec load_rec(int lane, int t, bool ok, size_t rec, int d_c, int bits,
                                         const uint8_t *__restrict__ codes, const float2 *__restrict__ hdr,
                                         const int4 *__restrict__ ref_idx)
{
    GRec r;
    r.ix = make_int4(-1, -1, -1, -1);
    r.w[0] = r.w[1] = 0u;
    r.h[0] = r.h[1] = make_float2(0.0f, 0.0f);
    if (!ok) return r;
    r.ix = __ldg(ref_idx + rec);
    const uint8_t *crow = codes + rec * (size_t)(d_c * bits / 8);
    const float2 *hrow = hdr + rec * (size_t)(d_c / 32);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c = lane * 8 + u * 256;
        if (c < d_c) {
            r.h[u] = __ldg(hrow + (c >> 5));
            r.w[u] = bits == 4 ? __ldg((const uint32_t *)(crow + (c >> 1)))
                               : (uint32_t)__ldg((const uint16_t *)(crow + (c >> 2)));
        }
    }
    return r;
}

// Persistent: each warp takes the selected tokens gw, gw + nw, ... in turn, and loads the
// next token's record and the position of the one after it before it decodes the
// current one, so that the chain position -> record -> reference rows overlaps the work.
template <typename RefT, typename OutT>
__global__ void __launch_bounds__(256, kGatherBlocks<RefT>)
k_gather(const int32_t *__restrict__ sel, int n_sel, int T, int W, int d_c, int bits,
         int n_ref, const RefT *__restrict__ ref_vec, const uint8_t *__restrict__ codes,
         const float2 *__restrict__ hdr, const int4 *__restrict__ ref_idx, OutT *__restrict__ out_z,
         OutT *__restrict__ out_mean, long long total, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
    long long tok = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (tok >= total) return;
    const float zero8[8] = {0, 0, 0, 0, 0, 0, 0, 0};

    int t = __ldg(sel + tok);
    GRec rc = load_rec(lane, t, t >= 0 && t < T, (size_t)(tok / n_sel) * T + t, d_c, bits, codes, hdr, ref_idx);
    long long tn = tok + nw;
    int t_n = -1;
    if constexpr (kPersistent<RefT>) t_n = tn < total ? __ldg(sel + tn) : -1;
    while (tok < total) {
        // ahead: the next token's record and the position of the token after it
        long long tnn = tn + nw;
        int t_nn = -1;
        GRec rn = rc;
        if constexpr (kPersistent<RefT>) {
            t_nn = tnn < total ? __ldg(sel + tnn) : -1;
            rn = load_rec(lane, t_n, tn < total && t_n >= 0 && t_n < T,
                          (size_t)(tn < total ? tn / n_sel : 0) * T + t_n, d_c, bits, codes, hdr, ref_idx);
            asm volatile("" ::: "memory");
        } else {
            tn = total;                                 // one token per warp
        }

        // ---- the current token
        const int lb = (int)(tok / n_sel);
        OutT *oz = out_z + (size_t)tok * d_c;
        OutT *om = out_mean + (size_t)tok * W;
        bool ok = t >= 0 && t < T;
        if (t >= T) set_status(status, RKV_ERR_INDEX);
        const int slots[4] = {rc.ix.x, rc.ix.y, rc.ix.z, rc.ix.w};
        int k = 0;
        if (ok) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (slots[j] >= n_ref) { ok = false; set_status(status, RKV_ERR_INDEX); }
                if (slots[j] >= 0) ++k;
            }
        }
        if (!ok) {
            for (int c = lane * 8; c < d_c; c += 256) store8(oz + c, zero8);
            for (int c = lane * 8; c < W; c += 256) store8(om + c, zero8);
        } else {
            // z~: each lane decodes 8 coordinates per step
            const size_t rec = (size_t)lb * T + t;
            int u = 0;
            for (int c = lane * 8; c < d_c; c += 256, ++u) {
                float2 h;
                uint32_t word;
                if (u < 2) {
                    h = u == 0 ? rc.h[0] : rc.h[1];
                    word = u == 0 ? rc.w[0] : rc.w[1];
                } else {
                    const uint8_t *crow = codes + rec * (size_t)(d_c * bits / 8);
                    h = __ldg(hdr + rec * (size_t)(d_c / 32) + (c >> 5));
                    word = bits == 4 ? __ldg((const uint32_t *)(crow + (c >> 1)))
                                     : (uint32_t)__ldg((const uint16_t *)(crow + (c >> 2)));
                }
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t q = bits == 4 ? (word >> (4 * j)) & 15u : (word >> (2 * j)) & 3u;
                    v[j] = fmaf((float)q, h.y, h.x);
                }
                store8(oz + c, v);
            }

            // mean of the stored references, summed in ascending slot order, times 1/k
            const RefT *rbase = ref_vec + (size_t)lb * n_ref * W;
            const float inv_k = k > 0 ? 1.0f / (float)k : 0.0f;
            const float2 ik2 = make_float2(inv_k, inv_k);
#pragma unroll (kPersistent<RefT> ? 2 : 4)
            for (int c = lane * 8; c < W; c += 256) {
                float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (slots[j] >= 0) RefLoad<RefT>::add(rbase + (size_t)slots[j] * W + c, a);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 m = __fmul2_rn(make_float2(a[2 * j], a[2 * j + 1]), ik2);
                    a[2 * j] = m.x;
                    a[2 * j + 1] = m.y;
                }
                store8(om + c, a);
            }
        }
        tok = tn;
        t = t_n;
        rc = rn;
        tn = tnn;
        t_n = t_nn;
    }
}

template <typename RefT>
static void gather_out(const Geometry &g, const rkv_ref_pool *pool, const rkv_cache *cache,
                       const int32_t *sel, int n_sel, void *out_z, void *out_mean, int out_dtype,
                       int32_t *status, cudaStream_t s)
{
    long long total = (long long)g.LB * n_sel;
    // 8-warp blocks: one warp per token, or at most the resident blocks (persistent warps)
    const long long need = (total + 7) / 8, cap = (long long)kGatherBlocks<RefT> * device_sm_count();
    unsigned blocks = (unsigned)(kPersistent<RefT> && need > cap ? cap : need);
    ProfScope prof("gather_dequant", s);
    if (out_dtype == RKV_BF16)
        k_gather<RefT, __nv_bfloat16><<<blocks, 256, 0, s>>>(
            sel, n_sel, g.T, g.W, g.d_c, g.bits, g.n_ref, (const RefT *)pool->ref_vec, cache->codes,
            (const float2 *)cache->hdr, (const int4 *)cache->ref_idx, (__nv_bfloat16 *)out_z,
            (__nv_bfloat16 *)out_mean, total, status);
    else
        k_gather<RefT, float><<<blocks, 256, 0, s>>>(
            sel, n_sel, g.T, g.W, g.d_c, g.bits, g.n_ref, (const RefT *)pool->ref_vec, cache->codes,
            (const float2 *)cache->hdr, (const int4 *)cache->ref_idx, (float *)out_z,
            (float *)out_mean, total, status);
}

cudaError_t launch_gather(const Geometry &g, const rkv_ref_pool *pool, const rkv_cache *cache,
                          const int32_t *sel, int n_sel, void *out_z, void *out_mean,
                          int out_dtype, int32_t *status, cudaStream_t s)
{
    if (g.ref_dtype == RKV_F32)
        gather_out<float>(g, pool, cache, sel, n_sel, out_z, out_mean, out_dtype, status, s);
    else if (g.ref_dtype == RKV_BF16)
        gather_out<__nv_bfloat16>(g, pool, cache, sel, n_sel, out_z, out_mean, out_dtype, status, s);
    else
        gather_out<uint8_t>(g, pool, cache, sel, n_sel, out_z, out_mean, out_dtype, status, s);
    return cudaGetLastError();
}

}  // namespace rkv
