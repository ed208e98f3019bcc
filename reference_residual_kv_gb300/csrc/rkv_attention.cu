// rkv_attention.cu -- sparse attention of one decode step over the restored set
// [RKV §2.7 = Sec. IV-C]:
//   o_j = softmax( q_j K^_I^T / sqrt(D) ) V^_I   for each query head j,
// query head j reading key/value head floor(j / (H/N)); I = the selected rows that
// are not padding.  Reading the restored K^ and V^ dominates (2 N D bf16 per token),
// so the pass is bound by HBM and runs on CUDA cores in fp32:
//   k_attn_split    one CTA per (split of the selected rows, KV head, layer-sequence),
//                   about one CTA per SM.  A warp takes 8 rows at a time, 16 lanes per
//                   row (D/16 coordinates per lane, 16-byte loads), and issues the next
//                   8 rows' loads before it scores the current ones (where registers
//                   allow); the row loads do not wait for the selection entries.  The 16-lane partial
//                   dot products of 4 rows x G heads are summed by one transposing
//                   butterfly (each lane ends with whole scores), the online softmax
//                   (running max, sum) is updated once per 8 rows and head, and the
//                   probabilities go through shared memory to the lanes that hold V.
//                   The 8 warps merge in shared memory and write the split's partial
//                   (max, sum, D weighted sums).
//   k_attn_combine  one block per (layer-sequence, query head): merges the splits.
#include "rkv_internal.cuh"

#include <math.h>

namespace rkv {
namespace {

constexpr int kMaxG = 8;          // query heads per key/value head
constexpr int kWarps = 8;
constexpr int kLPR = 16;          // lanes per row
constexpr int kU = 4;             // rows per 16-lane group and batch
constexpr int kRB = 2 * kU;       // rows per warp and batch
constexpr int kMinRows = 64;      // fewest rows a split is given
constexpr int kMaxCtas = 1024;    // CTAs the workspace is sized for

// EPL bf16 values of one row: EPL / 2 packed words
template <int EPL> struct Raw { uint32_t w[EPL / 2]; };

template <int EPL>
__device__ __forceinline__ void load_raw(const __nv_bfloat16 *p, Raw<EPL> &r)
{
    if constexpr (EPL == 4) {
        const uint2 u = __ldg((const uint2 *)p);
        r.w[0] = u.x; r.w[1] = u.y;
    } else {
#pragma unroll
        for (int c = 0; c < EPL / 8; ++c) {
            const uint4 u = __ldg((const uint4 *)p + c);
            r.w[4 * c] = u.x; r.w[4 * c + 1] = u.y; r.w[4 * c + 2] = u.z; r.w[4 * c + 3] = u.w;
        }
    }
}

template <int EPL>
__device__ __forceinline__ void unpack(const Raw<EPL> &r, float (&x)[EPL])
{
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) {
        x[2 * i] = __uint_as_float(r.w[i] << 16);
        x[2 * i + 1] = __uint_as_float(r.w[i] & 0xffff0000u);
    }
}

// One butterfly step over lane bit O: a lane keeps the half of its N values that its
// bit selects and adds the partner's copy of that half.
template <int N, int O>
__device__ __forceinline__ void fold(const float (&a)[N], float (&b)[N / 2], int lane)
{
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = up ? a[i] : a[i + N / 2];
        const float keep = up ? a[i + N / 2] : a[i];
        b[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
}

__device__ __forceinline__ float max_over_groups(float v)
{
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float sum_over_groups(float v)
{
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

// The 8 rows of batch rb: row rb + 2u + h is loaded by 16-lane group h (rows past r1
// are not, and read as zero); lane i < 8 loads the selection entry of row rb + i.  The
// row loads do not wait for the selection entries: padding rows are read like the
// others and masked when scored.
template <int EPL>
__device__ __forceinline__ void load_batch(const __nv_bfloat16 *kb, const __nv_bfloat16 *vb,
                                           const int32_t *sb, size_t rs, int rb, int r1, int lane,
                                           Raw<EPL> (&kx)[kU], Raw<EPL> (&vx)[kU], int &t)
{
    t = -1;
    if (lane < kRB && rb + lane < r1) t = __ldg(sb + rb + lane);
    const int h = lane >> 4;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        if (rb + 2 * u + h < r1) {
            const size_t off = (size_t)(rb + 2 * u + h) * rs;
            load_raw<EPL>(kb + off, kx[u]);
            load_raw<EPL>(vb + off, vx[u]);
        } else {
#pragma unroll
            for (int i = 0; i < EPL / 2; ++i) { kx[u].w[i] = 0u; vx[u].w[i] = 0u; }
        }
    }
}

// Partials: [LB][N][splits][G][D + 2] floats = {D weighted sums, max, sum}.
template <int EPL, int GM>
__global__ void __launch_bounds__(32 * kWarps, 1)
k_attn_split(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kh,
             const __nv_bfloat16 *__restrict__ vh, const int32_t *__restrict__ sel, int n_sel,
             int T, int H, int N, int chunk, int splits, float scale, float *__restrict__ part)
{
    constexpr int D = kLPR * EPL;
    constexpr int V = kU * GM;             // partial scores per lane and batch: (row u, head g)
    constexpr int E = V / kLPR;            // whole scores per lane after the butterfly
    // batches whose loads are in flight ahead of the one being scored (registers allow)
    constexpr int kAhead = EPL * GM <= 32 ? 1 : 0;
    __shared__ float sm[kWarps][GM][D + 2];
    __shared__ __align__(16) float pbuf[kWarps][2][V];
    __shared__ __align__(16) float abuf[kWarps][GM];
    const int s = blockIdx.x, n = blockIdx.y, lb = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = lane >> 4, j = lane & 15;
    const int G = H / N;

    float qr[GM][EPL], o[GM][EPL];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) { o[g][e] = 0.0f; qr[g][e] = 0.0f; }
        if (g < G) {
            Raw<EPL> r;
            load_raw<EPL>(q + ((size_t)lb * H + n * G + g) * D + j * EPL, r);
            unpack<EPL>(r, qr[g]);
#pragma unroll
            for (int e = 0; e < EPL; ++e) qr[g][e] *= scale;   // 1/sqrt(D): a power of 2 for D = 64, 256
        }
    }
    // lane's score entries v = j E + e: row u = v / GM of its group, head g = v % GM
    float m_s[E], l_s[E];
#pragma unroll
    for (int e = 0; e < E; ++e) { m_s[e] = -INFINITY; l_s[e] = 0.0f; }

    const int r0 = s * chunk, r1 = min(n_sel, r0 + chunk);
    const size_t rs = (size_t)N * D;                          // row stride of K^, V^
    const __nv_bfloat16 *kb = kh + (size_t)lb * n_sel * rs + (size_t)n * D + j * EPL;
    const __nv_bfloat16 *vb = vh + (size_t)lb * n_sel * rs + (size_t)n * D + j * EPL;
    const int32_t *sb = sel + (size_t)lb * n_sel;

    constexpr int kStep = kWarps * kRB;
    Raw<EPL> kc[kU], vc[kU], kn[kU], vn[kU];
    int tc = -1, tn = -1;
    int rb = r0 + warp * kRB;
    if (rb < r1) load_batch<EPL>(kb, vb, sb, rs, rb, r1, lane, kc, vc, tc);
    if constexpr (kAhead == 2) {
        if (rb + kStep < r1) load_batch<EPL>(kb, vb, sb, rs, rb + kStep, r1, lane, kn, vn, tn);
    }
    while (rb < r1) {
        const int ra = rb + kAhead * kStep;
        Raw<EPL> ka[kU], va[kU];
        int ta = -1;
        if constexpr (kAhead > 0) {
            if (ra < r1) load_batch<EPL>(kb, vb, sb, rs, ra, r1, lane, ka, va, ta);
            asm volatile("" ::: "memory");   // the later batches' loads stay ahead of this batch's work
        }
        // bit i: row rb + i is selected, not padding, and inside [0, T)
        const uint32_t vm = __ballot_sync(0xffffffffu, lane < kRB && tc >= 0 && tc < T);
        // partial scores of this lane's coordinates, then whole scores by the butterfly
        float a[V];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            float kf[EPL];
            unpack<EPL>(kc[u], kf);
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float d = 0.0f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d = fmaf(qr[g][e], kf[e], d);
                a[u * GM + g] = d;
            }
        }
        float b8[V / 2], b4[V / 4], b2[V / 8], sc[E];
        fold<V, 8>(a, b8, lane);
        fold<V / 2, 4>(b8, b4, lane);
        fold<V / 4, 2>(b4, b2, lane);
        fold<V / 8, 1>(b2, sc, lane);
        // online softmax, once per batch and head
        __syncwarp();
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int v = j * E + e, u = v / GM, g = v % GM;
            const bool live = ((vm >> (2 * u + h)) & 1u) && g < G;
            const float x = live ? sc[e] : -INFINITY;
            const float mn = fmaxf(m_s[e], max_over_groups(x));
            const float mu = mn == -INFINITY ? 0.0f : mn;
            const float alpha = __expf(m_s[e] - mu);
            const float pr = __expf(x - mu);
            l_s[e] = fmaf(l_s[e], alpha, sum_over_groups(pr));
            m_s[e] = mn;
            pbuf[warp][h][v] = pr;
            if (h == 0 && v < GM) abuf[warp][v] = alpha;
        }
        __syncwarp();
        float pw[V], al[GM];
#pragma unroll
        for (int i = 0; i < V / 4; ++i) {
            const float4 t4 = *(const float4 *)&pbuf[warp][h][4 * i];
            pw[4 * i] = t4.x; pw[4 * i + 1] = t4.y; pw[4 * i + 2] = t4.z; pw[4 * i + 3] = t4.w;
        }
#pragma unroll
        for (int i = 0; i < GM / 4; ++i) {
            const float4 t4 = *(const float4 *)&abuf[warp][4 * i];
            al[4 * i] = t4.x; al[4 * i + 1] = t4.y; al[4 * i + 2] = t4.z; al[4 * i + 3] = t4.w;
        }
        float vf[kU][EPL];
#pragma unroll
        for (int u = 0; u < kU; ++u) unpack<EPL>(vc[u], vf[u]);
#pragma unroll
        for (int g = 0; g < GM; ++g) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float acc = o[g][e] * al[g];
#pragma unroll
                for (int u = 0; u < kU; ++u) acc = fmaf(pw[u * GM + g], vf[u][e], acc);
                o[g][e] = acc;
            }
        }
        rb += kStep;
        if constexpr (kAhead == 2) {
#pragma unroll
            for (int u = 0; u < kU; ++u) { kc[u] = kn[u]; vc[u] = vn[u]; kn[u] = ka[u]; vn[u] = va[u]; }
            tc = tn;
            tn = ta;
        } else if constexpr (kAhead == 1) {
#pragma unroll
            for (int u = 0; u < kU; ++u) { kc[u] = ka[u]; vc[u] = va[u]; }
            tc = ta;
        } else {
            if (rb < r1) load_batch<EPL>(kb, vb, sb, rs, rb, r1, lane, kc, vc, tc);
        }
    }
    // the two 16-lane groups summed different rows under the same running maxima
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
    if (h == 0) {
#pragma unroll
        for (int g = 0; g < GM; ++g)
#pragma unroll
            for (int e = 0; e < EPL; ++e) sm[warp][g][j * EPL + e] = o[g][e];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int v = j * E + e;
            if (v < GM) { sm[warp][v][D] = m_s[e]; sm[warp][v][D + 1] = l_s[e]; }
        }
    }
    __syncthreads();
    // merge the warps: one warp per query head
    for (int g = warp; g < G; g += kWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm[w][g][D]);
        float f[kWarps], L = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            f[w] = M == -INFINITY ? 0.0f : __expf(sm[w][g][D] - M);
            L = fmaf(sm[w][g][D + 1], f[w], L);
        }
        float *dst = part + ((((size_t)lb * N + n) * splits + s) * G + g) * (D + 2);
        for (int d = lane; d < D; d += 32) {
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc = fmaf(sm[w][g][d], f[w], acc);
            dst[d] = acc;
        }
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

// Splits of the selected rows per (KV head, layer-sequence): enough CTAs for `ctas`,
// each with at least kMinRows rows.
int attn_splits(const Geometry &g, int n_sel, int ctas)
{
    const int heads = g.N * g.LB;
    int sp = (ctas + heads - 1) / heads;
    sp = min(sp, (n_sel + kMinRows - 1) / kMinRows);
    return max(sp, 1);
}

template <int EPL>
cudaError_t run_attn(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                     const int32_t *sel, int n_sel, float *out, float *part, cudaStream_t s)
{
    const int splits = attn_splits(g, n_sel, min(device_sm_count(), kMaxCtas));
    const int chunk = ((n_sel + splits - 1) / splits + kRB - 1) / kRB * kRB;
    const float scale = (float)(1.0 / sqrt((double)g.D));
    const dim3 grid(splits, g.N, g.LB);
    {
        ProfScope prof("attention_split", s);
        if (H / g.N <= 4)
            k_attn_split<EPL, 4><<<grid, 32 * kWarps, 0, s>>>(
                (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kh, (const __nv_bfloat16 *)vh, sel, n_sel,
                g.T, H, g.N, chunk, splits, scale, part);
        else if constexpr (EPL < 16)
            k_attn_split<EPL, kMaxG><<<grid, 32 * kWarps, 0, s>>>(
                (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kh, (const __nv_bfloat16 *)vh, sel, n_sel,
                g.T, H, g.N, chunk, splits, scale, part);
        else
            return cudaErrorInvalidValue;                     // D = 256 takes groups of <= 4
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    ProfScope prof("attention_combine", s);
    k_attn_combine<EPL / 2><<<(unsigned)(g.LB * H), 32 * kWarps, 0, s>>>(part, H, g.N, splits, out);
    return cudaGetLastError();
}

}  // namespace

size_t attention_workspace_bytes(const Geometry &g, int H, int n_sel)
{
    const size_t splits = (size_t)attn_splits(g, n_sel, kMaxCtas);
    return (size_t)g.LB * H * splits * (g.D + 2) * sizeof(float);
}

cudaError_t launch_attention(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                             const int32_t *sel, int n_sel, float *out, void *workspace, cudaStream_t s)
{
    float *part = (float *)workspace;
    switch (g.D) {
    case 64: return run_attn<4>(g, H, q, kh, vh, sel, n_sel, out, part, s);
    case 128: return run_attn<8>(g, H, q, kh, vh, sel, n_sel, out, part, s);
    case 256: return run_attn<16>(g, H, q, kh, vh, sel, n_sel, out, part, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rkv
