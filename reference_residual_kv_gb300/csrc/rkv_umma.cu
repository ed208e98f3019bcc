// rkv_umma.cu -- the write path for bf16 kv on the 5th-generation tensor cores.
//
// All four dense contractions of the path run through one persistent,
// warp-specialised kernel (one CTA per SM):
//   warp 0      TMA producer: 128x64 A tile + 256x64 B tile per stage, 4 stages
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma 128x256x16, bf16 -> fp32,
//               into one of two 256-column TMEM accumulators
//   warps 2..9  epilogue: one accumulator row (= one token or reference) per
//               thread and half of the columns per warp, read with tcgen05.ld
//               while the next tile accumulates
// The epilogue is what differs between the four uses:
//   M_P    P1 | P2 = R [W_c1 | W_c2] for each stored reference (fp32 out)
//   M_DIST ||r||^2 - 2 x.r for the causal pool of each token, best kList per row
//          and column half
//          [RKV §2.2 = Sec. IV-A; ||x||^2 is common to a row and left out]
//   M_S1   dh = Swish(x W_c1) ⊙ x W_c2 - Swish(p1) ⊙ p2, p = mean of the chosen
//          references' P rows, i.e. the first layer of f_c at the KV-space mean
//          by linearity [RKV §2.2, §2.3 = Sec. IV-A]; stored as bf16 hi + lo
//   M_S2   z = dh_hi W_c3 + dh_lo W_c3 = f_c(kv) - f_c(mean), then per-token
//          group min/max quantisation and packing [RKV §2.4]
// Every mbarrier wait is bounded; on expiry the kernel reports
// RKV_ERR_DEVICE_TIMEOUT, lets its copies and MMAs land, frees TMEM and returns.
#include "rkv_internal.cuh"
#include "umma.cuh"

#include <cudaTypedefs.h>

namespace rkv {

enum { M_P = 0, M_DIST = 1, M_S1 = 2, M_S2 = 3 };

constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kInfoBytes = kEpiWarps * 64 * 32; // S1: 64 tokens x 32 B per epilogue warp
constexpr int kS1Round = 8;                     // S1: tokens whose gathers are in flight at once
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256 + kInfoBytes;
constexpr uint32_t kIdesc = um::idesc_bf16_f32(kBM, kBN);
// projections run transposed: D[f][t] = W[f][:] . X[t][:], two 128x128 MMAs per step
constexpr uint32_t kIdescT = um::idesc_bf16_f32(kBM, kBN / 2);

// M_P and M_S1 put the weights on the MMA's M side (TMEM lane = d_ff column f) and
// the tokens (or references) on N (TMEM column = token), so that the epilogue's
// per-token gathers of reference projections and its stores are coalesced across
// the 32 lanes of a warp (consecutive f).
template <int MODE> struct Transposed { static constexpr bool value = MODE == M_P || MODE == M_S1; };

struct UmmaArgs {
    int LB, B, T, rows;   // rows: A-operand rows per lb (T, or n_ref for M_P)
    int n_mtiles, n_ntiles, k_chunks, a_sources, b_split, b_per_layer, max_chunks;
    int W, d_ff, d_c, n_ref, bits;
    float *P1, *P2;
    const float *ref_sqnorm;
    const int32_t *pool_size, *ref_slot;
    float2 *cand;
    const int4 *ref_idx;
    const uint8_t *copy_flag;
    __nv_bfloat16 *dh_hi, *dh_lo;
    uint8_t *codes;
    float2 *hdr;
    float *z_out;
    int32_t *status;
};

struct Item { int lb, m, n0, n1, chunk; };

// A cluster of C CTAs works on C consecutive token tiles against the same B tiles
// (weights or references), each CTA loading 1/C of every B tile and multicasting it
// to all C.
template <int C>
__device__ __forceinline__ int n_groups(const UmmaArgs &a) { return (a.n_mtiles + C - 1) / C; }

template <int MODE, int C>
__device__ __forceinline__ int item_count(const UmmaArgs &a)
{
    return a.LB * n_groups<C>(a) * (MODE == M_DIST ? a.max_chunks : a.n_ntiles);
}

// Work item i -> (lb, this CTA's token tile, N-tile range), identical N range and K
// loop for all CTAs of the cluster.  The (layer, sequence) index is the slowest, so
// the CTAs in flight share one layer's weights, references and projections in L2;
// the N tile is the fastest, so neighbouring CTAs reuse the same token rows.
// Distance items visit the late (largest-pool) token tiles first; a group's N range
// is that of its last tile.
template <int MODE, int C>
__device__ __forceinline__ bool item_get(const UmmaArgs &a, int i, int rank, Item &it)
{
    const int ng = n_groups<C>(a);
    if (MODE == M_DIST) {
        const int chunk = i % a.max_chunks, r = i / a.max_chunks;
        const int g = ng - 1 - r % ng, lb = r / ng;
        const int last = min(a.n_mtiles - 1, g * C + C - 1);
        const int nt = dist_ntiles(a.pool_size, a.T, last);
        it.lb = lb; it.m = g * C + rank; it.chunk = chunk;
        it.n0 = chunk * kDistChunk;
        it.n1 = min(nt, it.n0 + kDistChunk);
        return it.n0 < it.n1;
    }
    const int n = i % a.n_ntiles, r = i / a.n_ntiles;
    it.m = (r % ng) * C + rank; it.lb = r / ng; it.chunk = 0;
    it.n0 = n; it.n1 = n + 1;
    return true;
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16 *dst, const float (&v)[8])
{
    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __float2bfloat16_rn(v[j]);
    *(uint4 *)dst = *(const uint4 *)o;
}

// Swish with a fast division (relative error ~1e-7, far inside the z tolerance)
__device__ __forceinline__ float silu_fast(float u)
{
    return __fdividef(u, 1.0f + __expf(-u));
}

template <int MODE, int C>
__global__ void __launch_bounds__(kThreads, 1)
k_umma(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
       const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
       const UmmaArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = smem_raw + ((1024u - (um::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = (uint64_t *)(tiles + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    int4 *info_buf = (int4 *)(tiles + kStages * kStageBytes + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            um::mbar_init(&full[s], 1);
            um::mbar_init(&empty[s], C);          // one commit from every CTA of the cluster
        }
        for (int b = 0; b < 2; ++b) {
            um::mbar_init(&tfull[b], 1);
            um::mbar_init(&tempty[b], 32 * kEpiWarps);
        }
        um::mbar_init(drain, 1);
        *abort_flag = 0;
        um::fence_mbar_init();
    }
    if (warp == 1) {
        um::tmem_alloc(tmem_slot, 512);
        um::tmem_relinquish();
    }
    um::tc_fence_before();
    if (C > 1) um::cluster_sync();   // peers multicast into our stages only after our init
    else __syncthreads();
    um::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = item_count<MODE, C>(a);
    const int rank = C > 1 ? (int)um::cluster_rank() : 0;
    const int cid = blockIdx.x / C, ncl = gridDim.x / C;
    constexpr uint16_t kMask = (uint16_t)((1u << C) - 1u);
    constexpr int kSlice = kBN / C;                // B rows each CTA loads
    const int k_iters = a.k_chunks * a.a_sources;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            um::prefetch_tmap(&tmA0);
            um::prefetch_tmap(&tmA1);
            um::prefetch_tmap(&tmB0);
            um::prefetch_tmap(&tmB1);
            int stage = 0;
            uint32_t ph = 0;
            uint32_t last_ph[kStages];
            bool used[kStages];
            for (int s = 0; s < kStages; ++s) { used[s] = false; last_ph[s] = 0; }
            bool ok = true;
            for (int i = cid; i < n_items && ok; i += ncl) {
                Item it;
                if (!item_get<MODE, C>(a, i, rank, it)) continue;
                const int bz = a.b_per_layer ? it.lb / a.B : it.lb;
                for (int n = it.n0; n < it.n1 && ok; ++n) {
                    for (int kc = 0; kc < k_iters; ++kc) {
                        if (*abort_flag || !um::mbar_wait(&empty[stage], ph ^ 1u, kWaitCycles)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = tiles + stage * kStageBytes;
                        uint8_t *sb = sa + kABytes;
                        um::mbar_arrive_expect_tx(&full[stage], kStageBytes);
                        const int src = kc / a.k_chunks;
                        const int kx = (kc - src * a.k_chunks) * kBK;
                        um::tma_load_3d(sa, src ? &tmA1 : &tmA0, &full[stage], kx, it.m * kBM, it.lb);
                        if (C == 1) {
                            if (a.b_split) {
                                um::tma_load_3d(sb, &tmB0, &full[stage], kx, n * (kBN / 2), bz);
                                um::tma_load_3d(sb + kBBytes / 2, &tmB1, &full[stage], kx, n * (kBN / 2), bz);
                            } else {
                                um::tma_load_3d(sb, &tmB0, &full[stage], kx, n * kBN, bz);
                            }
                        } else {
                            // this CTA's slice of the B tile, into every CTA of the cluster;
                            // split B: slices [0, C/2) from tmB0, [C/2, C) from tmB1
                            uint8_t *dst = sb + rank * kSlice * (kBK * 2);
                            if (a.b_split) {
                                const int hs = C / 2;
                                const int yrow = n * (kBN / 2) + (rank % hs) * kSlice;
                                um::tma_load_3d_mc(dst, rank < hs ? &tmB0 : &tmB1, &full[stage], kx, yrow, bz, kMask);
                            } else {
                                um::tma_load_3d_mc(dst, &tmB0, &full[stage], kx, n * kBN + rank * kSlice, bz, kMask);
                            }
                        }
                        used[stage] = true;
                        last_ph[stage] = ph;
                        if (++stage == kStages) { stage = 0; ph ^= 1u; }
                    }
                }
            }
            if (!ok) {
                set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            // every issued copy must land before the CTA may exit
            for (int s = 0; s < kStages; ++s)
                if (used[s]) um::mbar_wait(&full[s], last_ph[s], kWaitCycles);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0, cnt = 0;
            bool ok = true;
            for (int i = cid; i < n_items && ok; i += ncl) {
                Item it;
                if (!item_get<MODE, C>(a, i, rank, it)) continue;
                for (int n = it.n0; n < it.n1 && ok; ++n) {
                    const uint32_t buf = cnt & 1u, tph = (cnt >> 1) & 1u;
                    if (*abort_flag || !um::mbar_wait(&tempty[buf], tph ^ 1u, kWaitCycles)) {
                        ok = false;
                        break;
                    }
                    um::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * kBN;
                    // distance tiles: only the references this CTA's token rows can see
                    // (causal pool of its last row), N rounded up to 16; none -> no MMA
                    uint32_t idesc = kIdesc;
                    bool issue = true;
                    if (MODE == M_DIST) {
                        const int own = a.pool_size[min(a.T, (it.m + 1) * kBM) - 1] - n * kBN;
                        const int cols = own < kBN ? own : kBN;
                        issue = it.m < a.n_mtiles && cols > 0;
                        if (issue) idesc = um::idesc_bf16_f32(kBM, (cols + 15) & ~15);
                    }
                    for (int kc = 0; kc < k_iters; ++kc) {
                        if (*abort_flag || !um::mbar_wait(&full[stage], ph, kWaitCycles)) {
                            ok = false;
                            break;
                        }
                        um::tc_fence_after();
                        const uint32_t sa = um::smem_u32(tiles + stage * kStageBytes);
                        const uint64_t ad = um::sdesc_sw128(sa);
                        const uint64_t bd = um::sdesc_sw128(sa + kABytes);
                        if (Transposed<MODE>::value) {
                            // stage = [token tile | W1 tile | W2 tile]: D1 = W1 X^T, D2 = W2 X^T
                            const uint64_t w1 = bd, w2 = um::sdesc_sw128(sa + kABytes + kBBytes / 2);
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k) {
                                um::mma_bf16(d_tmem, w1 + 2 * k, ad + 2 * k, kIdescT, (kc | k) != 0);
                                um::mma_bf16(d_tmem + kBN / 2, w2 + 2 * k, ad + 2 * k, kIdescT, (kc | k) != 0);
                            }
                        } else if (issue) {
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k)
                                um::mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kc | k) != 0);
                        }
                        if (C > 1) um::mma_commit_mc(&empty[stage], kMask);
                        else um::mma_commit(&empty[stage]);
                        if (++stage == kStages) { stage = 0; ph ^= 1u; }
                    }
                    if (!ok) break;
                    um::mma_commit(&tfull[buf]);
                    ++cnt;
                }
            }
            if (!ok) {
                set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            // all issued MMAs complete before TMEM can be released
            um::mma_commit(drain);
            um::mbar_wait(drain, 0, kWaitCycles);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // 8 warps: warp w reads TMEM lanes [32q, 32q+32), q = w % 4 (hardware rule),
        // and half h of the tile's columns.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
        uint32_t cnt = 0;
        bool ok = true;
        for (int i = cid; i < n_items; i += ncl) {
            Item it;
            if (!item_get<MODE, C>(a, i, rank, it)) continue;
            const int r = it.m * kBM + row;
            const bool in = r < a.rows;

            float be[kList];
            int bs[kList];
            int pool = 0, tile_pool = 0;
            if (MODE == M_DIST) {
#pragma unroll
                for (int j = 0; j < kList; ++j) { be[j] = INFINITY; bs[j] = -1; }
                pool = in ? a.pool_size[r] : 0;
                tile_pool = a.pool_size[min(a.T, (it.m + 1) * kBM) - 1];
            }
            bool is_ref = true;
            if (MODE == M_S2) is_ref = in ? (a.ref_slot[r] >= 0) : true;
            if (MODE == M_S1) {
                // this warp's 64 tokens: row offsets of the chosen references' projection
                // rows (unused places point at the all-zero row), 1/k and a live flag,
                // prepared in shared memory while the accumulator fills
                int4 *info = info_buf + (warp - 2) * 128;
                const int zoff = a.LB * a.n_ref * a.d_ff;
                const int lboff = it.lb * a.n_ref;
                __syncwarp();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int tj = it.m * kBM + h * 64 + cc * 32 + lane;
                    int rs = 0, cf = 1;
                    int4 ix = make_int4(-1, -1, -1, -1);
                    if (tj < a.rows) {
                        rs = a.ref_slot[tj];
                        cf = a.copy_flag[(size_t)it.lb * a.T + tj];
                        ix = a.ref_idx[(size_t)it.lb * a.T + tj];
                    }
                    int4 o = make_int4(zoff, zoff, zoff, zoff);
                    float inv_k = 0.0f, live = 0.0f;
                    if (rs < 0 && !cf) {
                        int kk = 0;
                        if (ix.x >= 0) { o.x = (lboff + ix.x) * a.d_ff; ++kk; }
                        if (ix.y >= 0) { o.y = (lboff + ix.y) * a.d_ff; ++kk; }
                        if (ix.z >= 0) { o.z = (lboff + ix.z) * a.d_ff; ++kk; }
                        if (ix.w >= 0) { o.w = (lboff + ix.w) * a.d_ff; ++kk; }
                        inv_k = kk > 0 ? 1.0f / (float)kk : 0.0f;
                        live = 1.0f;
                    }
                    info[2 * (cc * 32 + lane)] = o;
                    info[2 * (cc * 32 + lane) + 1] = make_int4(__float_as_int(inv_k), __float_as_int(live), 0, 0);
                }
                __syncwarp();
            }

            for (int n = it.n0; n < it.n1; ++n) {
                const uint32_t buf = cnt & 1u, tph = (cnt >> 1) & 1u;
                bool w = !*abort_flag && um::mbar_wait(&tfull[buf], tph, kWaitCycles);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                um::tc_fence_after();
                const uint32_t tb = tl + buf * kBN;

                if (MODE == M_P) {
                    // lane = d_ff column f, TMEM column = reference slot
                    const int f = n * (kBN / 2) + q * 32 + lane;
#pragma unroll 1
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c0 = h * 64 + cc * 32;
                        float v1[32], v2[32];
                        um::tmem_ld32(tb + c0, v1);
                        um::tmem_ld32(tb + kBN / 2 + c0, v2);
                        const int r0 = it.m * kBM + c0;
                        if (f < a.d_ff) {
                            float *p1 = a.P1 + ((size_t)it.lb * a.n_ref + r0) * a.d_ff + f;
                            float *p2 = a.P2 + ((size_t)it.lb * a.n_ref + r0) * a.d_ff + f;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                if (r0 + j < a.rows) {
                                    p1[(size_t)j * a.d_ff] = v1[j];
                                    p2[(size_t)j * a.d_ff] = v2[j];
                                }
                            }
                        }
                    }
                } else if (MODE == M_DIST) {
                    const float *rn = a.ref_sqnorm + (size_t)it.lb * a.n_ref;
#pragma unroll 1
                    for (int c0 = h * (kBN / 2); c0 < (h + 1) * (kBN / 2); c0 += 32) {
                        const int s0 = n * kBN + c0;
                        if (s0 >= tile_pool) break;          // uniform over the warp
                        float v[32];
                        um::tmem_ld32(tb + c0, v);
                        const float rn_l = (s0 + lane < a.n_ref) ? rn[s0 + lane] : 0.0f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float rj = __shfl_sync(0xffffffffu, rn_l, j);
                            const float e = fmaf(-2.0f, v[j], rj);
                            if (s0 + j < pool && e < be[kList - 1]) {
                                // this warp's slots arrive in increasing order: strict <
                                // keeps the lower slot ahead of an equal later one
                                float ce = e;
                                int cs = s0 + j;
#pragma unroll
                                for (int qq = 0; qq < kList; ++qq) {
                                    const bool lt = ce < be[qq];
                                    const float te = lt ? be[qq] : ce;
                                    const int ts = lt ? bs[qq] : cs;
                                    if (lt) { be[qq] = ce; bs[qq] = cs; }
                                    ce = te;
                                    cs = ts;
                                }
                            }
                        }
                    }
                } else if (MODE == M_S1) {
                    // lane = d_ff column f, TMEM column = token.  For each token the
                    // warp reads its references' projection rows as 128-byte lines,
                    // kS1Round tokens (8 loads each) in flight per round.
                    const int f = n * (kBN / 2) + q * 32 + lane;
                    const bool fok = f < a.d_ff;
                    const float *P1f = a.P1 + (fok ? f : 0);
                    const float *P2f = a.P2 + (fok ? f : 0);
                    const int4 *info = info_buf + (warp - 2) * 128;
#pragma unroll 1
                    for (int c = 0; c < 64; c += kS1Round) {
                        const int t0 = it.m * kBM + h * 64 + c;
                        float x1[kS1Round][4], x2[kS1Round][4], ik[kS1Round], lv[kS1Round];
#pragma unroll
                        for (int u = 0; u < kS1Round; ++u) {
                            const int4 o = info[2 * (c + u)];
                            const int4 b = info[2 * (c + u) + 1];
                            ik[u] = __int_as_float(b.x);
                            lv[u] = __int_as_float(b.y);
                            x1[u][0] = __ldg(P1f + o.x); x2[u][0] = __ldg(P2f + o.x);
                            x1[u][1] = __ldg(P1f + o.y); x2[u][1] = __ldg(P2f + o.y);
                            x1[u][2] = __ldg(P1f + o.z); x2[u][2] = __ldg(P2f + o.z);
                            x1[u][3] = __ldg(P1f + o.w); x2[u][3] = __ldg(P2f + o.w);
                        }
                        float v1[kS1Round], v2[kS1Round];
#pragma unroll
                        for (int p8 = 0; p8 < kS1Round; p8 += 8) {
                            um::tmem_ld8(tb + h * 64 + c + p8, v1 + p8);
                            um::tmem_ld8(tb + kBN / 2 + h * 64 + c + p8, v2 + p8);
                        }
                        __nv_bfloat16 *hi = a.dh_hi + ((size_t)it.lb * a.T + t0) * a.d_ff + f;
                        __nv_bfloat16 *lo = a.dh_lo + ((size_t)it.lb * a.T + t0) * a.d_ff + f;
#pragma unroll
                        for (int u = 0; u < kS1Round; ++u) {
                            const float m1 = ((x1[u][0] + x1[u][1]) + (x1[u][2] + x1[u][3])) * ik[u];
                            const float m2 = ((x2[u][0] + x2[u][1]) + (x2[u][2] + x2[u][3])) * ik[u];
                            // reference token or exact copy: lv = 0, z = 0
                            const float dh = (silu_fast(v1[u]) * v2[u] - silu_fast(m1) * m2) * lv[u];
                            const __nv_bfloat16 hb = __float2bfloat16_rn(dh);
                            if (fok && t0 + u < a.rows) {
                                hi[(size_t)u * a.d_ff] = hb;
                                lo[(size_t)u * a.d_ff] = __float2bfloat16_rn(dh - __bfloat162float(hb));
                            }
                        }
                    }
                } else {  // M_S2
#pragma unroll 1
                    for (int g8 = h * 4; g8 < h * 4 + 4; ++g8) {
                        const int c0 = n * kBN + g8 * 32;
                        if (c0 >= a.d_c) break;              // uniform
                        float v[32];
                        um::tmem_ld32(tb + g8 * 32, v);
                        if (!in) continue;
                        if (is_ref) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                        }
                        uint32_t wq[4];
                        float zmin, delta;
                        quant_group32(v, a.bits, wq, zmin, delta);
                        const size_t rec = (size_t)it.lb * a.T + r;
                        const int g = c0 >> 5;
                        uint8_t *dst = a.codes + rec * (size_t)(a.d_c * a.bits / 8) + g * (a.bits * 4);
                        if (a.bits == 4) *(uint4 *)dst = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                        else *(uint2 *)dst = make_uint2(wq[0], wq[1]);
                        a.hdr[rec * (a.d_c / 32) + g] = make_float2(zmin, delta);
                        if (a.z_out) {
                            float4 *zo = (float4 *)(a.z_out + rec * a.d_c + c0);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                zo[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        }
                    }
                }
                um::tc_fence_before();
                um::mbar_arrive(&tempty[buf]);
                ++cnt;
            }
            if (MODE == M_DIST && ok && in) {
                // this warp's sorted list (its half of the columns) as is; the two
                // halves' lists stay separate: [chunk][h * kList + j]
                float4 *cp = (float4 *)(a.cand + (((size_t)it.lb * a.T + r) * a.max_chunks + it.chunk) * kCand +
                                        h * kList);
#pragma unroll
                for (int j = 0; j < kList / 2; ++j)
                    cp[j] = make_float4(be[2 * j], __int_as_float(bs[2 * j]), be[2 * j + 1],
                                        __int_as_float(bs[2 * j + 1]));
            }
            if (!ok) break;
        }
        if (!ok) {
            set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    }

    um::tc_fence_before();
    // no CTA leaves while a peer may still multicast into it or signal its barriers
    if (C > 1) um::cluster_sync();
    else __syncthreads();
    if (warp == 1) {
        um::tc_fence_after();
        um::tmem_dealloc(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// bf16 [batch][rows][inner] row-major, box = 64 (inner) x box_rows, 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                     uint64_t batch, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {inner * 2, inner * 2 * rows};
    cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Clusters of kCluster CTAs share every B tile through TMA multicast.
constexpr int kCluster = 2;

template <int MODE>
static cudaError_t run(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b0,
                       const CUtensorMap &b1, const UmmaArgs &args, cudaStream_t s)
{
    constexpr int C = kCluster;
    auto kern = k_umma<MODE, C>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const long long groups = (args.n_mtiles + C - 1) / C;
    const long long items = (long long)args.LB * groups * (MODE == M_DIST ? args.max_chunks : args.n_ntiles);
    if (items <= 0) return cudaSuccess;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    static int max_clusters = 0;
    if (max_clusters == 0) {
        cfg.gridDim = dim3(C * 64, 1, 1);
        cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, (void *)kern, &cfg);
        if (e != cudaSuccess || max_clusters <= 0) max_clusters = device_sm_count() / C;
    }
    const long long nc = items < max_clusters ? items : max_clusters;
    cfg.gridDim = dim3((unsigned)(nc * C), 1, 1);
    static const char *names[4] = {"umma_ref_proj", "umma_distance_topk", "umma_swiglu_diff",
                                   "umma_z_quant"};
    ProfScope prof(names[MODE], s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_umma_compress(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                                 const void *W1t, const void *W2t, const void *W3t,
                                 const rkv_cache *cache, uint8_t *ws, const Workspace &wl,
                                 float *z_out, int32_t *status, cudaStream_t s)
{
    cudaError_t e;
    float *P1 = (float *)(ws + wl.P1), *P2 = (float *)(ws + wl.P2);
    float *rn_max = (float *)(ws + wl.rn_max);
    float2 *cand = (float2 *)(ws + wl.cand);
    __nv_bfloat16 *dh_hi = (__nv_bfloat16 *)(ws + wl.dh_hi);
    __nv_bfloat16 *dh_lo = (__nv_bfloat16 *)(ws + wl.dh_lo);
    const bool fp8 = g.ref_dtype == RKV_FP8_E4M3;
    void *ref_mma = fp8 ? (void *)(ws + wl.ref_mma) : pool->ref_vec;
    const size_t zrow = (size_t)g.LB * g.n_ref * g.d_ff;     // the all-zero projection row
    if ((e = launch_prep_refs(g, pool, ref_mma, rn_max, P1 + zrow, P2 + zrow, s)) != cudaSuccess)
        return e;

    UmmaArgs a{};
    a.LB = g.LB; a.B = g.B; a.T = g.T; a.W = g.W; a.d_ff = g.d_ff; a.d_c = g.d_c;
    a.n_ref = g.n_ref; a.bits = g.bits; a.max_chunks = g.max_chunks;
    a.P1 = P1; a.P2 = P2; a.ref_sqnorm = pool->ref_sqnorm; a.pool_size = pool->pool_size;
    a.ref_slot = pool->ref_slot; a.cand = cand; a.ref_idx = (const int4 *)cache->ref_idx;
    uint8_t *copy_flag = ws + wl.copy_flag;
    a.copy_flag = copy_flag;
    a.dh_hi = dh_hi; a.dh_lo = dh_lo; a.codes = cache->codes; a.hdr = (float2 *)cache->hdr;
    a.z_out = z_out; a.status = status;
    const int kw = (g.W + kBK - 1) / kBK;

    CUtensorMap mX, mW1, mW2, mW3, mHi, mLo, mRa, mRb;
    // B maps load one cluster slice per box: kBN / kCluster rows
    constexpr int kSliceRows = kBN / kCluster;
    static_assert(kCluster == 1 || kCluster == 2 || kCluster == 4, "cluster of 1, 2 or 4");
    const int split_rows = kCluster == 1 ? kBN / 2 : kSliceRows;
    if (!make_map(&mX, kv, g.W, g.T, g.LB, kBM) || !make_map(&mW1, W1t, g.W, g.d_ff, g.L, split_rows) ||
        !make_map(&mW2, W2t, g.W, g.d_ff, g.L, split_rows) ||
        !make_map(&mW3, W3t, g.d_ff, g.d_c, g.L, kSliceRows) ||
        !make_map(&mHi, dh_hi, g.d_ff, g.T, g.LB, kBM) ||
        !make_map(&mLo, dh_lo, g.d_ff, g.T, g.LB, kBM))
        return cudaErrorInvalidValue;

    if (g.n_ref > 0) {
        if (!make_map(&mRa, ref_mma, g.W, g.n_ref, g.LB, kBM) ||
            !make_map(&mRb, ref_mma, g.W, g.n_ref, g.LB, kSliceRows))
            return cudaErrorInvalidValue;
        // P1 | P2 for every reference
        UmmaArgs p = a;
        p.rows = g.n_ref; p.n_mtiles = (g.n_ref + kBM - 1) / kBM; p.n_ntiles = (g.d_ff + 127) / 128;
        p.k_chunks = kw; p.a_sources = 1; p.b_split = 1; p.b_per_layer = 1;
        if ((e = run<M_P>(mRa, mRa, mW1, mW2, p, s)) != cudaSuccess) return e;
        // distance expansion and per-item candidates
        UmmaArgs d = a;
        d.rows = g.T; d.n_mtiles = g.n_mtiles; d.n_ntiles = 1;
        d.k_chunks = kw; d.a_sources = 1; d.b_split = 0; d.b_per_layer = 0;
        if ((e = run<M_DIST>(mX, mX, mRb, mRb, d, s)) != cudaSuccess) return e;
    }
    int32_t *scan_list = (int32_t *)(ws + wl.scan_list);
    float *xnorm = (float *)(ws + wl.xnorm);
    if (g.n_ref > 0 && (e = launch_token_norms(g, kv, xnorm, s)) != cudaSuccess) return e;
    if ((e = launch_topk_finalize(g, kv, ref_mma, 0, pool, cand, xnorm, rn_max, cache->ref_idx,
                                  copy_flag, scan_list, scan_list + (size_t)g.LB * g.T, status,
                                  s)) != cudaSuccess)
        return e;
    {
        UmmaArgs p = a;
        p.rows = g.T; p.n_mtiles = g.n_mtiles; p.n_ntiles = (g.d_ff + 127) / 128;
        p.k_chunks = kw; p.a_sources = 1; p.b_split = 1; p.b_per_layer = 1;
        if ((e = run<M_S1>(mX, mX, mW1, mW2, p, s)) != cudaSuccess) return e;
    }
    {
        UmmaArgs p = a;
        p.rows = g.T; p.n_mtiles = g.n_mtiles; p.n_ntiles = (g.d_c + kBN - 1) / kBN;
        p.k_chunks = (g.d_ff + kBK - 1) / kBK; p.a_sources = 2; p.b_split = 0; p.b_per_layer = 1;
        if ((e = run<M_S2>(mHi, mLo, mW3, mW3, p, s)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace rkv
