// rkv_attention.cu -- sparse attention of one decode step over the restored set
// [RKV §2.7 = Sec. IV-C]:
//   o_j = softmax( q_j K^_I^T / sqrt(D) ) V^_I   for each query head j,
// query head j reading key/value head floor(j / (H/N)); I = the selected rows that
// are not padding.  Reading the restored K^ and V^ dominates (2 N D bf16 per token), so
// the pass is bound by HBM.  Two implementations of the same partials:
//   k_attn_tc       D = 128 (the long-context and Qwen shapes): scores and weighted sums
//                   on the tensor cores (tcgen05, TMA-fed rings of K^ and V^ tiles),
//                   softmax on 4 warps; described above the kernel
//   k_attn_split    other D: CUDA cores in fp32.  One CTA per (split of the selected
//                   rows, KV head, layer-sequence), about one CTA per SM.  A warp takes 8
//                   rows at a time, 16 lanes per row (D/16 coordinates per lane, 16-byte
//                   loads), and issues the next 8 rows' loads before it scores the current
//                   ones (where registers allow); the row loads do not wait for the
//                   selection entries.  The 16-lane partial dot products of 4 rows x G
//                   heads are summed by one transposing butterfly (each lane ends with
//                   whole scores), the online softmax (running max, sum) is updated once
//                   per 8 rows and head, and the probabilities go through shared memory to
//                   the lanes that hold V.  The 8 warps merge in shared memory and write
//                   the split's partial (max, sum, D weighted sums).
//   k_attn_combine  one block per (layer-sequence, query head): merges the splits.
#include "rkv_internal.cuh"
#include "umma.cuh"

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
    // launched as a programmatic dependent of the split pass: wait for that grid to
    // complete and its partials to be visible (no effect after an ordinary launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

// ---------------------------------------------------------------- tensor-core pass, D = 128
// k_attn_tc: the same partials from the 5th-generation tensor cores.  One CTA per (split
// of the selected rows, KV head, layer-sequence); the split is walked in tiles of 128
// rows.
//   warp 0     TMA producer: the tile's K^ and V^ rows of this head (2 boxes of 64
//              coordinates each) into two rings of 3 x 32 KB: a K^ slot is free once
//              the scores have read it, a V^ slot once the output product has.  The
//              producer and the MMA thread issue whatever is ready (no fixed order), so
//              a late copy holds up only the work that reads it
//   warp 1     TMEM allocation (64 columns); MMA issue, one thread:
//                S = K^_tile q^T      M = 128 rows, N = 16 (the G <= 8 query heads of
//                                     this KV head, zero-padded), K = D
//                O^T = V^_tile^T P    M = D = 128, N = 16, K = 128 rows; V^ is read in
//                                     place as an MN-major operand, and P holds the
//                                     probabilities as bf16 hi (columns 0..7) + lo (8..15)
//              S and O^T each have two TMEM buffers, so the scores of tile i + 1 are
//              computed while tile i's probabilities are written
//   warps 2..5 thread t: row t of the tile for the softmax, coordinate d = t of the output.
//              Online softmax in base 2: the tile's maximum per head over the 128 rows
//              (warp shuffles, then the 4 warps through shared memory), p = 2^(s - m),
//              P written to shared memory; then the previous tile's O^T is read back and
//              folded into registers, o = o * 2^(m_prev - m) + O (the accumulator is never
//              rescaled in TMEM).
// Every wait is bounded; a CTA whose wait runs out writes NaN into its partial, so the
// merged outputs of that head read NaN.
namespace tc {
constexpr int kRows = 128;                     // selected rows per tile
constexpr int kD = 128;
constexpr int kStages = 3;                     // per ring (K^, V^)
constexpr int kTileBytes = kRows * kD * 2;     // 32 KB: one of K^, V^
constexpr int kStageBytes = 2 * kTileBytes;    // a K^ slot and a V^ slot
constexpr int kQBytes = 16 * kD * 2;           // 16 rows (query heads, zero-padded) x D
constexpr int kPBytes = 16 * kRows * 2;        // 16 rows (P hi, P lo) x 128 tile rows
constexpr int kBarBytes = 256;
constexpr int kSmem = kStages * kStageBytes + kQBytes + 2 * kPBytes + kBarBytes + 1024;
constexpr int kThreads = 64 + 128;
constexpr int kTmemCols = 64;                  // S: 2 x 16, O^T: 2 x 16
static_assert(kSmem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
}  // namespace tc

// 16-byte unit u of row n of a K-major, 128-byte-swizzled 16-row block
__device__ __forceinline__ uint32_t sw128_unit(int n, int u)
{
    return (uint32_t)(n * 128 + ((u ^ (n & 7)) << 4));
}

__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int GM>
__global__ void __launch_bounds__(tc::kThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
          const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ sel, int n_sel, int T,
          int H, int N, int chunk, int splits, float scale_log2, float *__restrict__ part)
{
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    static_assert(GM == 4 || GM == 8, "query heads per KV head: up to 4, or up to 8");
    __shared__ float red[2][4][GM];
    __shared__ float lred[4][GM];
    uint8_t *stg = smem_raw + ((1024u - (um::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *qs = stg + kStages * kStageBytes;
    uint8_t *ps = qs + kQBytes;
    uint8_t *kring = stg, *vring = stg + kStages * kTileBytes;
    uint64_t *fullK = (uint64_t *)(ps + 2 * kPBytes);
    uint64_t *emptyK = fullK + kStages, *fullV = emptyK + kStages, *emptyV = fullV + kStages;
    uint64_t *s_full = emptyV + kStages, *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2, *o_full = p_full + 2, *o_empty = o_full + 2;
    uint64_t *drain = o_empty + 2;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int s = blockIdx.x, n = blockIdx.y, lb = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = H / N;
    const int r0 = s * chunk, r1 = min(n_sel, r0 + chunk);
    const int nt = r1 > r0 ? (r1 - r0 + kRows - 1) / kRows : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            um::mbar_init(&fullK[i], 1);
            um::mbar_init(&emptyK[i], 1);
            um::mbar_init(&fullV[i], 1);
            um::mbar_init(&emptyV[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            um::mbar_init(&s_full[b], 1);
            um::mbar_init(&s_empty[b], 4);
            um::mbar_init(&p_full[b], 4);
            um::mbar_init(&o_full[b], 1);
            um::mbar_init(&o_empty[b], 4);
        }
        um::mbar_init(drain, 1);
        *abort_flag = 0;
        um::fence_mbar_init();
    }
    // the producer: the first slots' copies go out before the rest of the setup
    auto issue = [&](const CUtensorMap *m, uint8_t *ring, uint64_t *full, int i) {
        const int st = i % kStages;
        uint8_t *b = ring + st * kTileBytes;
        um::mbar_arrive_expect_tx(&full[st], kTileBytes);
        const int y = r0 + i * kRows, x = n * kD;
        um::tma_load_3d(b, m, &full[st], x, y, lb);
        um::tma_load_3d(b + kTileBytes / 2, m, &full[st], x + 64, y, lb);
    };
    const int first = min(nt, kStages);
    if (threadIdx.x == 0) {
        um::prefetch_tmap(&tmK);
        um::prefetch_tmap(&tmV);
        for (int i = 0; i < first; ++i) {
            issue(&tmK, kring, fullK, i);
            issue(&tmV, vring, fullV, i);
        }
        // the merge kernel may be scheduled now; it waits for this grid's completion
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == 1) {
        um::tmem_alloc(tmem_slot, kTmemCols);
        um::tmem_relinquish();
    }
    // the query heads of this KV head (rows >= G zero) and both P buffers (zero: their
    // rows for heads >= G are never written), in the swizzled K-major layout
    for (int u = threadIdx.x - 32; u >= 0 && u < 16 * (kD / 8); u += blockDim.x - 32) {
        const int row = u / (kD / 8), uu = u % (kD / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < G) v = __ldg((const uint4 *)(q + ((size_t)lb * H + n * G + row) * kD) + uu);
        *(uint4 *)(qs + (uu >> 3) * (16 * 128) + sw128_unit(row, uu & 7)) = v;
    }
    for (int u = threadIdx.x - 32; u >= 0 && u < 2 * kPBytes / 16; u += blockDim.x - 32)
        *(uint4 *)(ps + u * 16) = make_uint4(0u, 0u, 0u, 0u);
    um::fence_proxy_async_smem();
    um::tc_fence_before();
    __syncthreads();
    um::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // slot i % 3 of a ring is free once tile i - 3's reader has finished
            auto free_slot = [&](uint64_t *empty, int i) {
                return um::mbar_try_wait(&empty[i % kStages], (((uint32_t)(i / kStages)) & 1u) ^ 1u);
            };
            int ik = first, iv = first;
            bool ok = true;
            long long t0 = clock64();
            while ((ik < nt || iv < nt) && ok) {
                bool did = false;
                if (ik < nt && free_slot(emptyK, ik)) { issue(&tmK, kring, fullK, ik++); did = true; }
                if (iv < nt && free_slot(emptyV, iv)) { issue(&tmV, vring, fullV, iv++); did = true; }
                if (did) t0 = clock64();
                else if (*abort_flag || clock64() - t0 > kWaitCycles) ok = false;
            }
            if (!ok) *abort_flag = 1;
            // no copy is in flight when the CTA leaves
            for (int i = max(0, ik - kStages); i < ik; ++i)
                um::mbar_wait(&fullK[i % kStages], (uint32_t)(i / kStages) & 1u, kWaitCycles);
            for (int i = max(0, iv - kStages); i < iv; ++i)
                um::mbar_wait(&fullV[i % kStages], (uint32_t)(i / kStages) & 1u, kWaitCycles);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = um::idesc_bf16_f32(kRows, 16);
            const uint32_t id_o = um::idesc_bf16_f32(kD, 16) | (1u << 15);   // A (V^) MN-major
            const uint32_t qb = um::smem_u32(qs), pb = um::smem_u32(ps);
            const uint32_t kb0 = um::smem_u32(kring), vb0 = um::smem_u32(vring);
            // the scores of tile i: its K^ slot has landed and the softmax has read S(i - 2)
            auto qk_ready = [&](int i) {
                return um::mbar_try_wait(&fullK[i % kStages], ((uint32_t)(i / kStages)) & 1u) &&
                       um::mbar_try_wait(&s_empty[i & 1], (((uint32_t)i >> 1) & 1u) ^ 1u);
            };
            // the output product of tile i: P(i) is written, O(i - 2) folded, V^ landed
            auto pv_ready = [&](int i) {
                const uint32_t ph = ((uint32_t)i >> 1) & 1u;
                return um::mbar_try_wait(&p_full[i & 1], ph) && um::mbar_try_wait(&o_empty[i & 1], ph ^ 1u) &&
                       um::mbar_try_wait(&fullV[i % kStages], ((uint32_t)(i / kStages)) & 1u);
            };
            int iq = 0, ip = 0;
            bool ok = true;
            long long t0 = clock64();
            while (ip < nt && ok) {
                bool did = false;
                if (iq < nt && qk_ready(iq)) {
                    um::tc_fence_after();
                    const uint32_t kb = kb0 + (iq % kStages) * kTileBytes;
#pragma unroll
                    for (int kc = 0; kc < kD / 64; ++kc) {
                        const uint64_t ad = um::sdesc_sw128(kb + kc * (kTileBytes / 2));
                        const uint64_t bd = um::sdesc_sw128(qb + kc * (16 * 128));
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            um::mma_bf16(tmem + (iq & 1) * 16, ad + 2 * k, bd + 2 * k, id_s, (kc | k) != 0);
                    }
                    um::mma_commit(&s_full[iq & 1]);
                    um::mma_commit(&emptyK[iq % kStages]);
                    ++iq;
                    did = true;
                }
                if (ip < iq && pv_ready(ip)) {
                    um::tc_fence_after();
                    const uint32_t vb = vb0 + (ip % kStages) * kTileBytes;
                    const uint32_t pbi = pb + (ip & 1) * kPBytes;
#pragma unroll
                    for (int k = 0; k < kRows / 16; ++k) {
                        // 16 tile rows: V^ rows 16k.. (two 8-row groups 1024 B apart; the
                        // second 64 coordinates 16 KB on) against P's K chunk k / 4
                        const uint64_t ad = um::sdesc_sw128_mn(vb + k * 2048, kTileBytes / 2, 1024);
                        const uint64_t bd = um::sdesc_sw128(pbi + (k >> 2) * (16 * 128)) + 2 * (k & 3);
                        um::mma_bf16(tmem + 32 + (ip & 1) * 16, ad, bd, id_o, k != 0);
                    }
                    um::mma_commit(&emptyV[ip % kStages]);
                    um::mma_commit(&o_full[ip & 1]);
                    ++ip;
                    did = true;
                }
                if (did) t0 = clock64();
                else if (*abort_flag || clock64() - t0 > kWaitCycles) ok = false;
            }
            if (!ok) *abort_flag = 1;
            // every issued MMA completes before TMEM is released
            um::mma_commit(drain);
            um::mbar_wait(drain, 0, kWaitCycles);
        }
    } else {
        // ------------------------------------------------------------ softmax and output
        const int qq = warp & 3;
        const int t = qq * 32 + lane;                    // tile row; output coordinate
        const uint32_t tl = tmem + ((uint32_t)(qq * 32) << 16);
        float m_run[GM], l_t[GM], o_acc[GM], al_prev[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) { m_run[g] = -INFINITY; l_t[g] = 0.0f; o_acc[g] = 0.0f; al_prev[g] = 1.0f; }
        bool ok = true;
        // fold tile j's O^T (scale of its own maximum) into o_acc
        auto fold = [&](int j, const float (&al)[GM]) -> bool {
            bool w = !*abort_flag && um::mbar_wait(&o_full[j & 1], ((uint32_t)j >> 1) & 1u, kWaitCycles);
            if (!__all_sync(0xffffffffu, w)) return false;
            um::tc_fence_after();
            float hi[8], lo[8];
            um::tmem_ld8(tl + 32 + (j & 1) * 16, hi);
            um::tmem_ld8(tl + 32 + (j & 1) * 16 + 8, lo);
            um::tc_fence_before();
            __syncwarp();
            if (lane == 0) um::mbar_arrive(&o_empty[j & 1]);
#pragma unroll
            for (int g = 0; g < GM; ++g) o_acc[g] = fmaf(o_acc[g], al[g], hi[g] + lo[g]);
            return true;
        };
        const int32_t *sb = sel + (size_t)lb * n_sel;
        for (int i = 0; i < nt; ++i) {
            const int r = r0 + i * kRows + t;
            bool valid = false;
            if (r < r1) {
                const int ts = __ldg(sb + r);
                valid = ts >= 0 && ts < T;
            }
            bool w = !*abort_flag && um::mbar_wait(&s_full[i & 1], ((uint32_t)i >> 1) & 1u, kWaitCycles);
            w = __all_sync(0xffffffffu, w);
            float x[GM];
            if (w) {
                um::tc_fence_after();
                float sv[8];
                um::tmem_ld8(tl + (i & 1) * 16, sv);
                um::tc_fence_before();
                __syncwarp();
                if (lane == 0) um::mbar_arrive(&s_empty[i & 1]);
#pragma unroll
                for (int g = 0; g < GM; ++g) x[g] = valid && g < G ? sv[g] * scale_log2 : -INFINITY;
            } else {
#pragma unroll
                for (int g = 0; g < GM; ++g) x[g] = -INFINITY;
            }
            // the tile's maximum per head: this warp's 32 rows, then the 4 warps
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float v = x[g];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                if (lane == 0) red[i & 1][qq][g] = v;
            }
            // every softmax warp reaches this barrier each tile: a wait that ran out in
            // one of them ends the loop in all four
            if (!um::bar_and(1, 128, w)) { ok = false; break; }
            float al[GM], p[GM];
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                const float mt = fmaxf(fmaxf(red[i & 1][0][g], red[i & 1][1][g]),
                                       fmaxf(red[i & 1][2][g], red[i & 1][3][g]));
                const float mn = fmaxf(m_run[g], mt);
                const float mu = mn == -INFINITY ? 0.0f : mn;
                al[g] = ex2_fast(m_run[g] - mu);
                p[g] = ex2_fast(x[g] - mu);
                l_t[g] = fmaf(l_t[g], al[g], p[g]);
                m_run[g] = mn;
            }
            // P of tile i: row t of the K-major block, hi in rows 0..7, lo in rows 8..15
            uint8_t *pbuf = ps + (i & 1) * kPBytes + (t >> 6) * (16 * 128);
            const int u = (t & 63) >> 3, e = (t & 7) * 2;
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g < G) {
                    const __nv_bfloat16 hb = __float2bfloat16_rn(p[g]);
                    const __nv_bfloat16 lbv = __float2bfloat16_rn(p[g] - __bfloat162float(hb));
                    *(__nv_bfloat16 *)(pbuf + sw128_unit(g, u) + e) = hb;
                    *(__nv_bfloat16 *)(pbuf + sw128_unit(8 + g, u) + e) = lbv;
                }
            }
            um::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) um::mbar_arrive(&p_full[i & 1]);
            if (i > 0 && !fold(i - 1, al_prev)) { ok = false; }
            if (!um::bar_and(2, 128, ok)) { ok = false; break; }
#pragma unroll
            for (int g = 0; g < GM; ++g) al_prev[g] = al[g];
        }
        if (ok && nt > 0 && !um::bar_and(2, 128, fold(nt - 1, al_prev))) ok = false;
        // the sum of p over the split's rows, per head
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            float v = l_t[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) lred[qq][g] = v;
        }
        um::bar_sync(1, 128);
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (g >= G) break;
            float *dst = part + ((((size_t)lb * N + n) * splits + s) * G + g) * (kD + 2);
            dst[t] = ok ? o_acc[g] : NAN;
            if (t == 0) {
                const float L = (lred[0][g] + lred[1][g]) + (lred[2][g] + lred[3][g]);
                // the partial's maximum in natural-log units: e^(m ln 2) = 2^m
                dst[kD] = ok ? (m_run[g] == -INFINITY ? -INFINITY : m_run[g] * 0.69314718055994531f) : NAN;
                dst[kD + 1] = ok ? L : NAN;
            }
        }
    }

    um::tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        um::tc_fence_after();
        um::tmem_dealloc(tmem, kTmemCols);
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

// The tensor-core pass (D = 128, G <= 8, 16-byte-aligned operands); false when the
// shape or the operands do not fit it or the driver rejects its tensor maps.
static bool run_attn_tc(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                        const int32_t *sel, int n_sel, float *out, float *part, cudaStream_t s,
                        cudaError_t &err)
{
    const int G = H / g.N;
    if (g.D != tc::kD || G > 8 || ((uintptr_t)q | (uintptr_t)kh | (uintptr_t)vh) % 16 != 0) return false;
    CUtensorMap mK, mV;
    const int rows = max(n_sel, 1);
    if (!make_map(&mK, kh, (uint64_t)g.N * g.D, rows, g.LB, tc::kRows) ||
        !make_map(&mV, vh, (uint64_t)g.N * g.D, rows, g.LB, tc::kRows))
        return false;
    static PerDevice<int> setup;
    int unused = 0;
    err = per_device(setup, unused, [](int &) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_tc<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_attn_tc<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmem);
        return e;
    });
    if (err != cudaSuccess) return true;
    // splits of whole 128-row tiles, about one CTA per SM
    int splits = attn_splits(g, n_sel, min(device_sm_count(), kMaxCtas));
    int chunk = n_sel > 0 ? ((n_sel + splits - 1) / splits + tc::kRows - 1) / tc::kRows * tc::kRows : tc::kRows;
    splits = n_sel > 0 ? (n_sel + chunk - 1) / chunk : 1;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.D));
    {
        ProfScope prof("attention_split", s);
        auto kern = G <= 4 ? k_attn_tc<4> : k_attn_tc<8>;
        kern<<<dim3(splits, g.N, g.LB), tc::kThreads, tc::kSmem, s>>>(
            mK, mV, (const __nv_bfloat16 *)q, sel, n_sel, g.T, H, g.N, chunk, splits, scale_log2, part);
        err = cudaGetLastError();
        if (err != cudaSuccess) return true;
    }
    // the merge launches as a programmatic dependent: its blocks are scheduled while the
    // split pass drains and wait on the device for its completion
    ProfScope prof("attention_combine", s);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(g.LB * H), 1, 1);
    cfg.blockDim = dim3(32 * kWarps, 1, 1);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, k_attn_combine<tc::kD / 32>, (const float *)part, H, g.N, splits, out);
    if (err == cudaSuccess) err = cudaGetLastError();
    return true;
}

template <int EPL>
cudaError_t run_attn(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                     const int32_t *sel, int n_sel, float *out, float *part, cudaStream_t s)
{
    cudaError_t tce = cudaSuccess;
    if (run_attn_tc(g, H, q, kh, vh, sel, n_sel, out, part, s, tce)) return tce;
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
