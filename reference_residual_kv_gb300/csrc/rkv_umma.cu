// rkv_umma.cu -- the write path for bf16 kv on the 5th-generation tensor cores.
//
// All four dense contractions of the path run through one persistent,
// warp-specialised kernel launched as CTA pairs (clusters of 2) that issue 2-SM
// MMAs: tcgen05.mma.cta_group::2, 256 x 256 x 16, bf16 in, fp32 in TMEM.  Each CTA
// of a pair holds 128 rows of A and half (128 rows) of B in its own shared memory;
// the leader (rank 0) issues the MMAs and each CTA's TMEM receives its own 128 rows
// of the 256 x 256 product, so each SM reads 8 KB of operands per 1 MFLOP step
// (a single-SM 128 x 128 step reads the same 8 KB for half the work).
//   warp 0      TMA producer (both CTAs): this CTA's A rows and B half per stage
//   warp 1      TMEM allocation (both CTAs, 512 columns = two 256-column
//               accumulators); MMA issue (leader only)
//   warps 2..9  epilogue: TMEM lane quarter q = warp % 4, column half h
//   warps 10, 11, 14, 15 (M_DIST only) ||x||^2 of every token row, read from the token
//               tiles in shared memory on each token tile's first N tile while the
//               MMA works; a stage is free once the MMA and these warps are done
//               with it (the top-k finalisation's distance bound needs the norms)
// The epilogue is what differs between the four uses:
//   M_P    P1 | P2 = R W_c1^T | R W_c2^T for each stored reference (fp32 out,
//          interleaved per column: {P1[f], P2[f]})
//   M_DIST ||r||^2 - 2 x.r for the causal pool of each token, best kList per row
//          and column half
//          [RKV §2.2 = Sec. IV-A; ||x||^2 is common to a row and left out]
//   M_S1   dh = Swish(x W_c1) ⊙ x W_c2 - Swish(p1) ⊙ p2, p = mean of the chosen
//          references' P rows, i.e. the first layer of f_c at the KV-space mean
//          by linearity [RKV §2.2, §2.3 = Sec. IV-A]; stored as bf16 hi + lo
//   M_S2   z = dh_hi W_c3 + dh_lo W_c3 = f_c(kv) - f_c(mean), then per-token
//          group min/max quantisation and packing [RKV §2.4]
// M_P and M_S1 run transposed (weights on the MMA's M side, tokens on N), each CTA's 128
// A rows covering 64 d_ff columns of W_c1 and W_c2.  In M_S1 they are 64 rows of W_c1
// and the same 64 rows of W_c2, so TMEM lane l < 64 holds x.W_c1[f] and lane 64 + l
// holds x.W_c2[f] of one column f, and a warp's 32 lanes are 32 consecutive f: the
// epilogue's per-token gathers of reference projections and its stores are contiguous
// runs.  In M_P each 32-row lane quarter is 16 rows of W_c1 and then the same 16 rows of
// W_c2, so lanes l and l + 16 write the two halves of one {P1[f], P2[f]} pair and a
// warp's stores are contiguous 128-byte runs.
// Every mbarrier wait is bounded; on expiry the kernel reports
// RKV_ERR_DEVICE_TIMEOUT, lets its copies and MMAs land, frees TMEM and returns.
#include "rkv_exact.cuh"
#include "rkv_internal.cuh"
#include "umma.cuh"

#include <cudaTypedefs.h>

#include <atomic>

namespace rkv {

enum { M_P = 0, M_DIST = 1, M_S1 = 2, M_S2 = 3 };

constexpr int kHalfN = kBN / 2;                  // B rows each CTA of a pair holds
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kBBytes = kHalfN * kBK * 2;        // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;   // per CTA
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kNormWarps = 4;                    // M_DIST: token-norm warps per CTA
// M_DIST launches warps 10..15 and runs the norm warps as 10, 11, 14 and 15 (schedulers 2
// and 3): warps 12 and 13 would share schedulers 0 and 1 with the single producer and MMA
// threads, so they stay idle
template <int MODE> constexpr int threads_of() { return kThreads + (MODE == M_DIST ? 32 * (kNormWarps + 2) : 0); }
constexpr int kInfoBytes = kEpiWarps * 64 * 32;  // S1: 64 tokens x 32 B per epilogue warp
constexpr int kS1Round = 4;                      // S1: tokens per round of gathers (one round ahead)
constexpr int kXTok = 8;                         // S1: tokens per exchange between warp pairs
constexpr int kXBytes = 2 * kEpiWarps * kXTok * 32 * 4;   // double-buffered exchange
constexpr int kGateRows = 16;                    // M_P: W_c1 rows, then the same W_c2 rows, per lane quarter
constexpr int kDistVBytes = kEpiWarps * 32 * 32 * 4;   // M_DIST: each epilogue lane's 32 expansion values
constexpr uint16_t kPairMask = 3;

template <int MODE> struct Cfg {
    static constexpr bool kT = MODE == M_P || MODE == M_S1;   // transposed
    static constexpr int kStages = MODE == M_S1 || MODE == M_DIST ? 6 : 7;
    static constexpr int kExtra = MODE == M_S1 ? kInfoBytes + kXBytes : (MODE == M_DIST ? kDistVBytes : 0);
    static constexpr int kSmem = kStages * kStageBytes + 1024 + 256 + kExtra;
    static_assert(kSmem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
    static_assert((3 * kStages + 5) * 8 + 8 <= 256, "barriers overflow their 256-byte block");
};

struct UmmaArgs {
    int LB, B, T, rows;   // rows: token (reference for M_P) rows per lb
    int tiles_t;          // ceil(rows / 256): pair tiles of tokens (references)
    int tiles_n;          // M_P/M_S1: 128-column d_ff slices; M_S2: 256-column d_c tiles;
                          // M_DIST: distance chunks (max_chunks)
    int k_chunks, a_sources;
    int fused_gate;       // M_P/M_S1: tmA0 maps W_c1 and W_c2 together (one box per stage)
    int W, d_ff, d_c, n_ref, bits;
    int dh_rows;          // rows of dh per lb: T, or the non-reference count when compacted
    float *P12;           // [LB * n_ref + 1][d_ff] of {x.W_c1[f], x.W_c2[f]} per reference
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
    const __nv_bfloat16 *xrows;   // M_DIST: the token rows (bf16, [LB*T][W]) ...
    float *xnorm;                 // ... and their ||x||^2, written by the norm warps
    long long wait_cycles;        // limit of every barrier wait (a.wait_cycles)
    int skip_use;                 // test hook: the pair peer skips its loads for this
                                  // stage use (-1: never)
};

// One work item of a pair: (lb, token tile t of 256 rows, N range [n0, n1)).
struct Item { int lb, t, n0, n1, chunk; };

__device__ __forceinline__ int item_count(const UmmaArgs &a)
{
    return a.LB * a.tiles_t * a.tiles_n;
}

// Work item of pair `pid` in round r.  A round takes the next npairs items of the
// order; odd rounds hand them out in reverse (boustrophedon), so that where item
// costs fall along the order (distance items: late token tiles first, and a tile's
// later reference chunks are shorter) every pair's total evens out.  Dealing items
// out with a fixed stride instead gave each pair the same chunk index of every tile
// whenever the number of pairs is a multiple of the chunk count.
__device__ __forceinline__ int item_at(int r, int pid, int npairs)
{
    return r * npairs + ((r & 1) ? npairs - 1 - pid : pid);
}

// The (layer, sequence) index is the slowest, so the pairs in flight share one layer's
// weights, references and projections in L2; the N index is the fastest, so
// neighbouring pairs reuse the same token rows.  Distance items visit the late
// (largest-pool) token tiles first.
template <int MODE>
__device__ __forceinline__ bool item_get(const UmmaArgs &a, int i, Item &it)
{
    const int n = i % a.tiles_n, r = i / a.tiles_n;
    it.lb = r / a.tiles_t;
    it.t = r % a.tiles_t;
    it.chunk = 0;
    if (MODE == M_DIST) {
        it.t = a.tiles_t - 1 - it.t;
        const int nt = dist_ntiles(a.pool_size, a.T, it.t);
        it.chunk = n;
        it.n0 = n * kDistChunk;
        it.n1 = min(nt, it.n0 + kDistChunk);
        return it.n0 < it.n1;
    }
    it.n0 = n;
    it.n1 = n + 1;
    return true;
}

// M_DIST: MMA N of N-tile n of pair tile t: the references the tile's last row can see,
// rounded up to 32 (so that each CTA's half is a multiple of 16 rows); CTA r of the pair
// supplies references [n*256 + r*N/2, n*256 + (r+1)*N/2).
__device__ __forceinline__ int dist_cols(const UmmaArgs &a, int t, int n)
{
    const int own = a.pool_size[min(a.T, (t + 1) * kTileM) - 1] - n * kBN;
    return own >= kBN ? kBN : ((own + 31) & ~31);
}

// S1: offset, from the warp's first token, of the token in its j-th own accumulator
// column; with reference rows skipped (kG > 0) a column group of kG - 1 covers kG tokens
template <int kG>
__host__ __device__ constexpr int s1_token(int j)
{
    return kG > 0 ? (j / (kG - 1)) * kG + j % (kG - 1) + 1 : j;
}

// 2^x and 1/x by the approximate hardware instructions (relative error ~2^-22)
__device__ __forceinline__ float exp2f_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_fast(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// kG > 0: every position that is 0 mod kG is a reference (fixed stride dividing kG,
// first reference at 0), where dh = 0 and the record is all zero.
//   S1: those token rows are not loaded: tmB is then a [LB][T/kG][kG][W] view, each CTA's
//       B half holds rows 1..kG-1 of its 128/kG groups (kBRows rows), and the MMA's N is
//       2 kBRows.  TMEM column j of half h is token h*128 + (j / (kG-1)) kG + j % (kG-1)
//       + 1 of the tile.  dh is stored compacted: row c of [LB][T (kG-1)/kG][d_ff] is the
//       c-th non-reference position, so a warp's tokens are consecutive rows.
//   S2: runs over the compacted rows (a.rows of them); row c is token
//       (c / (kG-1)) kG + c % (kG-1) + 1, and the row that opens a group also writes the
//       all-zero record of the group's reference token.
template <int MODE, int kG>
__global__ void __launch_bounds__(threads_of<MODE>(), 1)
k_umma(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
       const __grid_constant__ CUtensorMap tmB, const UmmaArgs a)
{
    using C = Cfg<MODE>;
    constexpr int S = C::kStages;
    constexpr bool kSkip = MODE == M_S1 && kG > 0;
    constexpr bool kCompact = MODE == M_S2 && kG > 0;
    constexpr int kBRows = kSkip ? kHalfN * (kG - 1) / kG : kHalfN;
    static_assert(!kSkip || (kHalfN % (kSkip ? kG : 1) == 0 && (kBRows / 2) % kXTok == 0 && kBRows % 8 == 0),
                  "skip layout: whole groups per CTA, whole exchanges per warp");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = smem_raw + ((1024u - (um::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = (uint64_t *)(tiles + S * kStageBytes);   // leader's: both CTAs' bytes
    uint64_t *empty = full + S;                                  // freed by the pair's MMA
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;                                // leader's: both epilogues
    uint64_t *drain = tempty + 2;
    uint64_t *landed = drain + 1;                                // M_DIST, peer: stage landed
    uint32_t *tmem_slot = (uint32_t *)(landed + S);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    int4 *info_buf = (int4 *)(tiles + S * kStageBytes + 256);
    float *xbuf = (float *)(tiles + S * kStageBytes + 256 + kInfoBytes);
    float *dvbuf = (float *)(tiles + S * kStageBytes + 256);   // M_DIST

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = um::cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            um::mbar_init(&full[s], 1);
            // M_DIST: the MMA's commit and one arrival per norm warp
            um::mbar_init(&empty[s], MODE == M_DIST ? 1 + kNormWarps : 1);
        }
        for (int b = 0; b < 2; ++b) {
            um::mbar_init(&tfull[b], 1);
            um::mbar_init(&tempty[b], 2 * kEpiWarps);
        }
        um::mbar_init(drain, 1);
        if (MODE == M_DIST)
            for (int s = 0; s < S; ++s) um::mbar_init(&landed[s], 1);
        *abort_flag = 0;
        um::fence_mbar_init();
    }
    if (warp == 1) {
        um::tmem_alloc2(tmem_slot, 512);
        um::tmem_relinquish2();
    }
    um::tc_fence_before();
    um::cluster_sync();   // the peer signals our barriers only after our init
    um::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = item_count(a);
    const int pid = blockIdx.x / 2, npairs = gridDim.x / 2;
    const int k_iters = a.k_chunks * a.a_sources;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            um::prefetch_tmap(&tmA0);
            um::prefetch_tmap(&tmA1);
            um::prefetch_tmap(&tmB);
            // The stage loop is kept short (no divisions, no memory reads): this one
            // thread shares its scheduler with epilogue warps, and every cycle it loses
            // delays a refill the MMA waits for.
            int stage = 0;
            uint32_t ph = 0;
            uint32_t used_mask = 0, ph_mask = 0;   // per stage: used, parity of its last use
            bool ok = true;
            int use = 0;
            const int kx_end = a.k_chunks * kBK;
            for (int rnd = 0; rnd * npairs < n_items && ok; ++rnd) {
                const int i = item_at(rnd, pid, npairs);
                if (i >= n_items) continue;
                Item it;
                if (!item_get<MODE>(a, i, it)) continue;
                const int lz = it.lb / a.B;                          // layer of the weights
                const int own_rows = it.t * 2 * kBM + (int)rank * kBM;
                for (int n = it.n0; n < it.n1 && ok; ++n) {
                    if (*abort_flag) { ok = false; break; }
                    // coordinates that stay fixed along K: A (y, z), B (y, z)
                    int ay, az, by, bz;
                    if (C::kT) {
                        // A: 64 d_ff columns of W_c1 and W_c2 (M_P: in 16-row groups);
                        // B: 128 tokens or references
                        const int f0 = n * kBM + (int)rank * (kBM / 2);
                        ay = a.fused_gate ? (MODE == M_P ? (lz * a.d_ff + f0) / kGateRows : lz * a.d_ff + f0) : f0;
                        az = a.fused_gate ? 0 : lz;
                        by = own_rows;
                        bz = it.lb;
                    } else {
                        // A: 128 token rows (M_S2: dh_hi, then dh_lo); B: half of N tile n
                        ay = own_rows;
                        az = it.lb;
                        const int half = MODE == M_DIST ? dist_cols(a, it.t, n) / 2 : kHalfN;
                        by = n * kBN + (int)rank * half;
                        bz = MODE == M_S2 ? lz : it.lb;
                    }
                    for (int src = 0; src < a.a_sources && ok; ++src) {
                        const CUtensorMap *mA = src ? &tmA1 : &tmA0;
                        for (int kx = 0; kx < kx_end; kx += kBK) {
                            if (!um::mbar_wait(&empty[stage], ph ^ 1u, a.wait_cycles)) {
                                ok = false;
                                break;
                            }
                            used_mask |= 1u << stage;
                            ph_mask = (ph_mask & ~(1u << stage)) | (ph << stage);
                            // test hook of the timeout path: the peer leaves one stage
                            // short, so the leader's full barrier never completes
                            if (!leader && use++ == a.skip_use) {
                                if (++stage == S) { stage = 0; ph ^= 1u; }
                                continue;
                            }
                            uint8_t *sa = tiles + stage * kStageBytes;
                            const uint32_t fb = um::smem_u32(&full[stage]);
                            // the leader's full barrier counts both CTAs' bytes
                            if (leader) um::mbar_arrive_expect_tx(&full[stage], 2 * (kABytes + kBRows * 128));
                            const uint32_t bar = leader ? fb : um::mapa(fb, 0);
                            if (MODE == M_P && a.fused_gate) {
                                // [4 groups][W_c1, W_c2][16 rows] in one box
                                um::tma_load_4d_pair(sa, &tmA0, bar, kx, 0, 0, ay);
                            } else if (MODE == M_P) {
                                // the same order from two separate matrices, 16 rows a box
#pragma unroll
                                for (int g = 0; g < kBM / (2 * kGateRows); ++g) {
                                    uint8_t *dg = sa + g * 2 * kGateRows * 128;
                                    um::tma_load_3d_pair(dg, &tmA0, bar, kx, ay + g * kGateRows, az);
                                    um::tma_load_3d_pair(dg + kGateRows * 128, &tmA1, bar, kx,
                                                         ay + g * kGateRows, az);
                                }
                            } else if (C::kT && !a.fused_gate) {
                                um::tma_load_3d_pair(sa, &tmA0, bar, kx, ay, az);
                                um::tma_load_3d_pair(sa + kABytes / 2, &tmA1, bar, kx, ay, az);
                            } else {
                                um::tma_load_3d_pair(sa, mA, bar, kx, ay, az);
                            }
                            if (kSkip) um::tma_load_4d_pair(sa + kABytes, &tmB, bar, kx, 1, by / (kSkip ? kG : 1), bz);
                            else um::tma_load_3d_pair(sa + kABytes, &tmB, bar, kx, by, bz);
                            if (++stage == S) { stage = 0; ph ^= 1u; }
                        }
                    }
                }
            }
            if (!ok) {
                set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            // a stage's copies have landed once the pair's MMA has freed it
            for (int s = 0; s < S; ++s)
                if ((used_mask >> s) & 1u) um::mbar_wait(&empty[s], (ph_mask >> s) & 1u, a.wait_cycles);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t ph = 0, cnt = 0;
            bool ok = true;
            for (int rnd = 0; rnd * npairs < n_items && ok; ++rnd) {
                const int i = item_at(rnd, pid, npairs);
                if (i >= n_items) continue;
                Item it;
                if (!item_get<MODE>(a, i, it)) continue;
                for (int n = it.n0; n < it.n1 && ok; ++n) {
                    const uint32_t buf = cnt & 1u, tph = (cnt >> 1) & 1u;
                    if (*abort_flag || !um::mbar_wait(&tempty[buf], tph ^ 1u, a.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    um::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * kBN;
                    // distance tiles: only the references the tile's rows can see
                    const uint32_t id = MODE == M_DIST ? um::idesc_bf16_f32(2 * kBM, dist_cols(a, it.t, n))
                                                       : um::idesc_bf16_f32(2 * kBM, 2 * kBRows);
                    for (int kc = 0; kc < k_iters; ++kc) {
                        if (!um::mbar_wait(&full[stage], ph, a.wait_cycles)) {
                            ok = false;
                            break;
                        }
                        um::tc_fence_after();
                        const uint32_t sa = um::smem_u32(tiles + stage * kStageBytes);
                        const uint64_t ad = um::sdesc_sw128(sa);
                        const uint64_t bd = um::sdesc_sw128(sa + kABytes);
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k)
                            um::mma2_bf16(d_tmem, ad + 2 * k, bd + 2 * k, id, (kc | k) != 0);
                        um::mma2_commit_mc(&empty[stage], kPairMask);
                        if (++stage == S) { stage = 0; ph ^= 1u; }
                    }
                    if (!ok) break;
                    um::mma2_commit_mc(&tfull[buf], kPairMask);
                    ++cnt;
                }
            }
            if (!ok) {
                set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            // all issued MMAs complete before TMEM can be released
            um::mma2_commit_mc(drain, 1);
            um::mbar_wait(drain, 0, a.wait_cycles);
        }
    } else if (MODE == M_DIST && warp >= 2 + kEpiWarps && (warp & 3) < 2) {
        // idle (see threads_of)
    } else if (MODE == M_DIST && warp >= 2 + kEpiWarps) {
        // ------------------------------------------------------------ token norms
        // Every stage use, in the producer's order: wait until its copies have landed
        // (the leader: its full barrier, which counts both CTAs' bytes; the peer: the
        // leader's forward of it), read it if it is part of a token tile's first N
        // tile, then add this warp's arrival to the stage's release.  Lane l of norm
        // warp w owns token row 32w + l of this CTA's 128 A rows; a stage holds 64 of
        // its values (one 128-byte row, 16-byte chunk c at position c ^ (row % 8), the
        // 128-byte swizzle).  ||x||^2 is a sum over stages of per-stage sums of squares.
        const int nrow = (warp < 12 ? warp - 10 : warp - 12) * 32 + lane;
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int rnd = 0; rnd * npairs < n_items && ok; ++rnd) {
            const int i = item_at(rnd, pid, npairs);
            if (i >= n_items) continue;
            Item it;
            if (!item_get<MODE>(a, i, it)) continue;
            for (int n = it.n0; n < it.n1 && ok; ++n) {
                const bool need = it.chunk == 0 && n == 0;
                float acc = 0.0f;
                for (int kc = 0; kc < k_iters; ++kc) {
                    const bool w = um::mbar_wait(leader ? &full[stage] : &landed[stage], ph, a.wait_cycles);
                    if (*abort_flag || !w) {
                        ok = false;
                        break;
                    }
                    if (leader && warp == 2 + kEpiWarps && lane == 0)
                        um::mbar_arrive_cluster_relaxed(um::mapa(um::smem_u32(&landed[stage]), 1));
                    if (need) {
                        const uint8_t *rowp = tiles + stage * kStageBytes + nrow * 128;
                        float part[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            part[c] = bf16x8_sqsum(*(const uint4 *)(rowp + ((c ^ (nrow & 7)) << 4)), 0.0f);
                        acc += ((part[0] + part[1]) + (part[2] + part[3])) +
                               ((part[4] + part[5]) + (part[6] + part[7]));
                    }
                    __syncwarp();
                    if (lane == 0) um::mbar_arrive(&empty[stage]);
                    if (++stage == S) { stage = 0; ph ^= 1u; }
                }
                const int r = it.t * 2 * kBM + (int)rank * kBM + nrow;
                if (need && ok && r < a.rows) a.xnorm[(size_t)it.lb * a.T + r] = acc;
            }
        }
        if (!ok) {
            set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // 8 warps: warp w reads TMEM lanes [32q, 32q+32), q = w % 4 (hardware rule),
        // and half h of the tile's columns.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
        // M_S1: warps (q, h) and (q ^ 2, h) hold the two gate halves of the same
        // 32 d_ff columns and trade accumulator columns through shared memory
        const int pair_id = 1 + (q & 1) + 2 * h;
        uint32_t cnt = 0, xcnt = 0;
        bool ok = true;
        for (int rnd = 0; rnd * npairs < n_items; ++rnd) {
            const int i = item_at(rnd, pid, npairs);
            if (i >= n_items) continue;
            Item it;
            if (!item_get<MODE>(a, i, it)) continue;
            const int r = it.t * 2 * kBM + (int)rank * kBM + row;   // token row (M_DIST, M_S2)
            const bool in = r < a.rows;
            // M_S2 over compacted rows: the token of row r
            const int tokr = kCompact ? (r / (kCompact ? kG - 1 : 1)) * kG + r % (kCompact ? kG - 1 : 1) + 1 : r;

            float be[kList];
            int bs[kList];
            int pool = 0, tile_pool = 0;
            if (MODE == M_DIST) {
#pragma unroll
                for (int j = 0; j < kList; ++j) { be[j] = INFINITY; bs[j] = -1; }
                pool = in ? a.pool_size[r] : 0;
                tile_pool = a.pool_size[min(a.T, (it.t + 1) * 2 * kBM) - 1];
            }
            bool is_ref = true;
            // a reference token or an exact copy of its references has z = 0 (S1 leaves
            // its dh rows as they come)
            if (MODE == M_S2)
                is_ref = in ? (a.ref_slot[tokr] >= 0 || a.copy_flag[(size_t)it.lb * a.T + tokr] != 0) : true;
            if (MODE == M_S1) {
                // this warp's 64 tokens: row offsets of the chosen references' projection
                // rows (unused places point at the all-zero row) and 1/k, prepared in
                // shared memory while the accumulator fills
                int4 *info = info_buf + (warp - 2) * 128;
                const int tok0 = it.t * 2 * kBM + h * kHalfN + (q < 2 ? 0 : 64);
                const int zoff = a.LB * a.n_ref * a.d_ff;
                const int lboff = it.lb * a.n_ref;
                __syncwarp();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int j = cc * 32 + lane;
                    if (j >= kBRows / 2) continue;         // a skip layout has fewer than 64
                    const int tj = tok0 + s1_token<kSkip ? kG : 0>(j);
                    int rs = 0, cf = 1;
                    int4 ix = make_int4(-1, -1, -1, -1);
                    if (tj < a.rows) {
                        rs = a.ref_slot[tj];
                        cf = a.copy_flag[(size_t)it.lb * a.T + tj];
                        ix = a.ref_idx[(size_t)it.lb * a.T + tj];
                    }
                    int4 o = make_int4(zoff, zoff, zoff, zoff);
                    float inv_k = 0.0f;
                    if (rs < 0 && !cf) {
                        int kk = 0;
                        if (ix.x >= 0) { o.x = (lboff + ix.x) * a.d_ff; ++kk; }
                        if (ix.y >= 0) { o.y = (lboff + ix.y) * a.d_ff; ++kk; }
                        if (ix.z >= 0) { o.z = (lboff + ix.z) * a.d_ff; ++kk; }
                        if (ix.w >= 0) { o.w = (lboff + ix.w) * a.d_ff; ++kk; }
                        inv_k = kk > 0 ? 1.0f / (float)kk : 0.0f;
                    }
                    info[2 * j] = o;
                    // 1/k (0 when the pool is empty, and for a reference token or an exact
                    // copy, whose z the W_c3 pass sets to 0)
                    info[2 * j + 1] = make_int4(__float_as_int(inv_k), 0, 0, 0);
                }
                __syncwarp();
            }

            for (int n = it.n0; n < it.n1; ++n) {
                const uint32_t buf = cnt & 1u, tph = (cnt >> 1) & 1u;
                bool w = !*abort_flag && um::mbar_wait(&tfull[buf], tph, a.wait_cycles);
                w = __all_sync(0xffffffffu, w);
                if (MODE == M_S1) w = um::bar_and(pair_id, 64, w);   // the pair leaves together
                if (!w) { ok = false; break; }
                um::tc_fence_after();
                const uint32_t tb = tl + buf * kBN;

                if (MODE == M_P) {
                    // lane l: d_ff column f of W_c1 (l < 16) or W_c2 (l >= 16); TMEM column =
                    // reference
                    const int f = n * kBM + (int)rank * (kBM / 2) + q * kGateRows + (lane & 15);
                    float *P = a.P12 + ((size_t)it.lb * a.n_ref * a.d_ff + f) * 2 + (lane >> 4);
#pragma unroll 1
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c0 = h * kHalfN + cc * 32;
                        float v[32];
                        um::tmem_ld32(tb + c0, v);
                        const int r0 = it.t * 2 * kBM + c0;
                        if (f < a.d_ff) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (r0 + j < a.rows) P[(size_t)(r0 + j) * a.d_ff * 2] = v[j];
                        }
                    }
                } else if (MODE == M_DIST) {
                    // ||r||^2 of this half's 128 columns, loaded before the accumulator
                    // reads (lane l holds column 32 cc + l of chunk cc)
                    const float *rn = a.ref_sqnorm + (size_t)it.lb * a.n_ref;
                    float rnv[kHalfN / 32];
#pragma unroll
                    for (int cc = 0; cc < kHalfN / 32; ++cc) {
                        const int sl = n * kBN + h * kHalfN + cc * 32 + lane;
                        rnv[cc] = sl < tile_pool ? __ldg(rn + sl) : 0.0f;
                    }
#pragma unroll
                    for (int cc = 0; cc < kHalfN / 32; ++cc) {
                        const int c0 = h * kHalfN + cc * 32;
                        const int s0 = n * kBN + c0;
                        if (s0 >= tile_pool) break;          // uniform over the warp
                        float v[32];
                        um::tmem_ld32(tb + c0, v);
                        // the columns whose expansion is below this row's current last
                        // entry (a superset of those that will enter: the bound only falls),
                        // collected in four independent partial masks
                        float thr = be[kList - 1];
                        const int lim = pool - s0;           // columns j < lim are in the pool
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float rj = __shfl_sync(0xffffffffu, rnv[cc], j);
                            v[j] = fmaf(-2.0f, v[j], rj);
                        }
                        // a row's first full chunk (empty list): instead of +inf, the largest
                        // of the eight 4-column minima, which is at or above the chunk's 8th
                        // smallest value (eight values lie at or below it), so no column that
                        // belongs in the list is left out and about half the columns are
                        const bool seed = thr == INFINITY && lim >= 32;
                        if (__any_sync(0xffffffffu, seed)) {
                            float mx = -INFINITY;
#pragma unroll
                            for (int g = 0; g < 8; ++g)
                                mx = fmaxf(mx, fminf(fminf(v[4 * g], v[4 * g + 1]), fminf(v[4 * g + 2], v[4 * g + 3])));
                            if (seed) thr = nextafterf(mx, INFINITY);
                        }
                        uint32_t hm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                        for (int j = 0; j < 32; ++j) hm[j & 3] |= (uint32_t)(j < lim && v[j] < thr) << j;
                        uint32_t hit = (hm[0] | hm[1]) | (hm[2] | hm[3]);
                        // each lane inserts only its own hits, in increasing column order
                        // (strict < keeps the lower slot ahead of an equal later one).  The
                        // warp runs max-popcount rounds, all lanes together and without
                        // branches: a lane out of hits inserts +inf, which never enters, and
                        // a hit that no longer beats the last entry passes through
                        // unchanged.
                        const int rounds = (int)__reduce_max_sync(0xffffffffu, (unsigned)__popc(hit));
                        // the chunk's values go to this lane's row of shared memory (16-byte
                        // unit u of lane l at u ^ (l % 8)), so that a round reads its
                        // candidate with one indexed load
                        float *vrow = dvbuf + ((warp - 2) * 32 + lane) * 32;
                        if (rounds > 0) {
                            __syncwarp();                    // the previous chunk's reads are done
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                *(float4 *)(vrow + ((u ^ (lane & 7)) << 2)) =
                                    make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                            __syncwarp();
                        }
                        for (int rd = 0; rd < rounds; ++rd) {
                            const int j = __ffs(hit) - 1;
                            float ce = hit ? vrow[(((j >> 2) ^ (lane & 7)) << 2) | (j & 3)] : INFINITY;
                            hit &= hit - 1u;
                            int cs = s0 + j;
#pragma unroll
                            for (int qq = 0; qq < kList; ++qq) {
                                const bool lt = ce < be[qq];
                                const float te = lt ? be[qq] : ce;
                                const int ts = lt ? bs[qq] : cs;
                                be[qq] = lt ? ce : be[qq];
                                bs[qq] = lt ? cs : bs[qq];
                                ce = te;
                                cs = ts;
                            }
                        }
                    }
                } else if (MODE == M_S1) {
                    // lane = d_ff column f; this warp holds x.W_c1[f] (q < 2) or x.W_c2[f]
                    // for all 256 tokens of the tile, finishes 64 of them and hands the
                    // other gate half of its partner's 64 over
                    const bool gate = q < 2;
                    const int f = n * kBM + (int)rank * (kBM / 2) + (q & 1) * 32 + lane;
                    const bool fok = f < a.d_ff;
                    const float2 *P12f = (const float2 *)a.P12 + (fok ? f : 0);
                    // this warp's own accumulator columns and those it hands over; both
                    // warps of the pair hold kBRows / 2 tokens
                    constexpr int kOwn = kBRows / 2;
                    const int own0 = h * kBRows + (gate ? 0 : kOwn);
                    const int give0 = h * kBRows + (gate ? kOwn : 0);
                    const int tok0 = it.t * 2 * kBM + h * kHalfN + (gate ? 0 : 64);
                    // dh row of this warp's first token (compacted when reference rows are
                    // left out: the warp's tokens are then consecutive rows)
                    const int drow0 = kSkip ? it.t * 2 * kBRows + own0 : tok0;
                    const int4 *info = info_buf + (warp - 2) * 128;
                    const int gb = 2 + 4 * h;                     // first warp of this half
                    const int me = warp - 2, partner = gb + ((warp - gb) ^ 2) - 2;
                    // the chosen references' projection pairs of 4 tokens per round, two
                    // rounds ahead of the arithmetic (a ring of three register buffers; the
                    // loop below is unrolled so that every buffer index is static)
                    float2 pr3[3][kS1Round][4];
                    float sc3[3][kS1Round];                // 1/k of each token
                    auto gather = [&](int c, float2 (&pr)[kS1Round][4], float (&sc)[kS1Round]) {
#pragma unroll
                        for (int u = 0; u < kS1Round; ++u) {
                            const int4 o = info[2 * (c + u)];
                            sc[u] = __int_as_float(info[2 * (c + u) + 1].x);
                            pr[u][0] = __ldg(P12f + o.x);
                            pr[u][1] = __ldg(P12f + o.y);
                            pr[u][2] = __ldg(P12f + o.z);
                            pr[u][3] = __ldg(P12f + o.w);
                        }
                    };
                    // dh = Swish(g1) g2 - Swish(m1) m2 for 4 tokens, with Swish(u) =
                    // u / (1 + e^-u) over one reciprocal of both denominators:
                    //   dh = (g1 g2 (1 + e_m) - m1 m2 (1 + e_g)) / ((1 + e_g)(1 + e_m));
                    // e^-u is clamped at 2^63 (u < -43.6: Swish is below 1e-17 there) so
                    // the denominator stays finite.  The dh of a reference token or an
                    // exact copy is not used: the W_c3 pass sets its z to 0.
                    auto finish = [&](int c, const float (&v)[kXTok], int v0, const float *xr,
                                      const float2 (&pr)[kS1Round][4], const float (&sc)[kS1Round]) {
                        __nv_bfloat16 *hi = a.dh_hi + ((size_t)it.lb * a.dh_rows + drow0) * a.d_ff + f;
                        __nv_bfloat16 *lo = a.dh_lo + ((size_t)it.lb * a.dh_rows + drow0) * a.d_ff + f;
#pragma unroll
                        for (int u = 0; u < kS1Round; ++u) {
                            const float pv = xr[(v0 + u) * 32 + lane];
                            const float g1 = gate ? v[v0 + u] : pv, g2 = gate ? pv : v[v0 + u];
                            const float2 s01 = __fadd2_rn(pr[u][0], pr[u][1]);
                            const float2 s23 = __fadd2_rn(pr[u][2], pr[u][3]);
                            const float2 m = __fmul2_rn(__fadd2_rn(s01, s23), make_float2(sc[u], sc[u]));
                            const float2 t = __fmul2_rn(make_float2(g1, m.x),
                                                        make_float2(-1.4426950408889634f, -1.4426950408889634f));
                            const float eg = exp2f_fast(fminf(t.x, 63.0f));
                            const float em = exp2f_fast(fminf(t.y, 63.0f));
                            const float2 d = __fadd2_rn(make_float2(eg, em), make_float2(1.0f, 1.0f));
                            const float2 pq = __fmul2_rn(make_float2(g1, m.x), make_float2(g2, m.y));
                            const float num = fmaf(pq.x, d.y, -(pq.y * d.x));
                            const float dh = num * rcp_fast(d.x * d.y);
                            const __nv_bfloat16 hb = __float2bfloat16_rn(dh);
                            if (fok && drow0 + c + u < a.dh_rows) {
                                hi[(size_t)(c + u) * a.d_ff] = hb;
                                lo[(size_t)(c + u) * a.d_ff] = __float2bfloat16_rn(dh - __bfloat162float(hb));
                            }
                        }
                    };
                    gather(0, pr3[0], sc3[0]);
                    gather(kS1Round, pr3[1], sc3[1]);
#pragma unroll
                    for (int c = 0; c < kOwn; c += kXTok) {
                        // double-buffered: a buffer is rewritten only after the next
                        // exchange barrier, which the partner reaches after reading it
                        float *xw = xbuf + (size_t)(((xcnt & 1u) * kEpiWarps + me) * kXTok) * 32;
                        const float *xr = xbuf + (size_t)(((xcnt & 1u) * kEpiWarps + partner) * kXTok) * 32;
                        ++xcnt;
                        {
                            float g[kXTok];
                            um::tmem_ld8(tb + give0 + c, g);
#pragma unroll
                            for (int j = 0; j < kXTok; ++j) xw[j * 32 + lane] = g[j];
                        }
                        um::bar_sync(pair_id, 64);
                        float v[kXTok];
                        um::tmem_ld8(tb + own0 + c, v);
                        const int r0 = c / kS1Round;       // rounds r0 and r0 + 1 of this exchange
                        if (c + 2 * kS1Round < kOwn) gather(c + 2 * kS1Round, pr3[(r0 + 2) % 3], sc3[(r0 + 2) % 3]);
                        finish(c, v, 0, xr, pr3[r0 % 3], sc3[r0 % 3]);
                        if (c + 3 * kS1Round < kOwn) gather(c + 3 * kS1Round, pr3[(r0 + 3) % 3], sc3[(r0 + 3) % 3]);
                        finish(c + kS1Round, v, kS1Round, xr, pr3[(r0 + 1) % 3], sc3[(r0 + 1) % 3]);
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
                        const size_t rec = (size_t)it.lb * a.T + tokr;
                        const int g = c0 >> 5;
                        const size_t cpitch = (size_t)(a.d_c * a.bits / 8);
                        uint8_t *dst = a.codes + rec * cpitch + g * (a.bits * 4);
                        if (a.bits == 4) *(uint4 *)dst = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                        else *(uint2 *)dst = make_uint2(wq[0], wq[1]);
                        a.hdr[rec * (a.d_c / 32) + g] = make_float2(zmin, delta);
                        if (a.z_out) {
                            float4 *zo = (float4 *)(a.z_out + rec * a.d_c + c0);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                zo[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        }
                        if (kCompact && r % (kCompact ? kG - 1 : 1) == 0) {
                            // the group's reference token, just before this one: zero record
                            uint8_t *dr = dst - cpitch;
                            if (a.bits == 4) *(uint4 *)dr = make_uint4(0u, 0u, 0u, 0u);
                            else *(uint2 *)dr = make_uint2(0u, 0u);
                            a.hdr[(rec - 1) * (a.d_c / 32) + g] = make_float2(0.0f, 0.0f);
                            if (a.z_out) {
                                float4 *zo = (float4 *)(a.z_out + (rec - 1) * a.d_c + c0);
#pragma unroll
                                for (int j = 0; j < 8; ++j) zo[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            }
                        }
                    }
                }
                // this warp is done with the accumulator (every tcgen05.ld has been
                // waited for): one relaxed arrival on the leader's barrier, which counts
                // both CTAs' epilogue warps; the warp's stores need no ordering with it
                um::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader) um::mbar_arrive_relaxed(&tempty[buf]);
                    else um::mbar_arrive_cluster_relaxed(um::mapa(um::smem_u32(&tempty[buf]), 0));
                }
                ++cnt;
            }
            if (MODE == M_DIST && ok && in) {
                // this warp's sorted list (its half of the columns) as is; the two
                // halves' lists stay separate: [chunk][h * kList + j]
                float4 *cp = (float4 *)(a.cand + (((size_t)it.lb * a.T + r) * a.tiles_n + it.chunk) * kCand +
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
    // no CTA leaves while its peer may still read its shared memory or signal its
    // barriers
    um::cluster_sync();
    if (warp == 1) {
        um::tc_fence_after();
        um::tmem_dealloc2(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------- host
// One-shot fault of the timeout path, armed by rkv_debug_wait_fault and taken by the
// next W_c3 launch of the write path.
static std::atomic<long long> g_fault_cycles{0};
static std::atomic<int> g_fault_skip{-1};

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
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
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

// A bf16 [batch][rows][inner] output tensor for TMA stores of box_inner x box_rows tiles
// from 64-byte-swizzled shared memory (box_inner * 2 bytes = 64).
bool make_map_store(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t batch,
                    uint32_t box_inner, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {inner * 2, inner * 2 * rows};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 token rows [batch][rows][inner] as [batch][rows / g][g][inner] (rows % g == 0):
// box = 64 (inner) x rows 1..g-1 of a group x 128 / g groups, 128-byte swizzle; the box
// lands as 128 (g - 1) / g consecutive 128-byte rows.
static bool make_map_skip(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                          uint64_t batch, int g)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {inner, (cuuint64_t)g, rows / g, batch};
    cuuint64_t strides[3] = {inner * 2, inner * 2 * g, inner * 2 * rows};
    cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)(g - 1), (cuuint32_t)(kHalfN / g), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// W_c1 and W_c2 ([L][d_ff][W] each, i.e. [L*d_ff][W]) seen as one [2][L*d_ff][W] tensor
// whose matrix stride is the distance between them: box = 64 (inner) x 64 rows x both
// matrices, i.e. 64 rows of W_c1 followed by the same 64 rows of W_c2.
static bool make_map_gates(CUtensorMap *m, const void *W1, long long gate_off, uint64_t inner,
                           uint64_t rows, uint64_t layers)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows * layers, 2};
    cuuint64_t strides[2] = {inner * 2, (cuuint64_t)gate_off};
    cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)(kBM / 2), 2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(W1), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same two matrices as a 4-D tensor [L*d_ff/16 groups][2 matrices][16 rows][W]:
// box = 64 (inner) x 16 rows x both matrices x 4 groups, i.e. per 32-row quarter 16 rows
// of W_c1 followed by the same 16 rows of W_c2 (the reference-projection layout).
static bool make_map_gates16(CUtensorMap *m, const void *W1, long long gate_off, uint64_t inner,
                             uint64_t rows, uint64_t layers)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {inner, (cuuint64_t)kGateRows, 2, rows * layers / kGateRows};
    cuuint64_t strides[3] = {inner * 2, (cuuint64_t)gate_off, inner * 2 * kGateRows};
    cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)kGateRows, 2, (cuuint32_t)(kBM / (2 * kGateRows))};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(W1), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE, int kG = 0>
static cudaError_t run(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b,
                       const UmmaArgs &args, cudaStream_t s)
{
    auto kern = k_umma<MODE, kG>;
    constexpr int smem = Cfg<MODE>::kSmem;
    const long long items = (long long)args.LB * args.tiles_t * args.tiles_n;
    if (items <= 0) return cudaSuccess;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(threads_of<MODE>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // per device: the raised shared-memory limit, then the pairs that fit at once
    static PerDevice<int> setup;
    int max_pairs = 0;
    cudaError_t se = per_device(setup, max_pairs, [&](int &mp) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = cfg;
        q.gridDim = dim3(2 * 64, 1, 1);
        mp = 0;
        e = cudaOccupancyMaxActiveClusters(&mp, (void *)kern, &q);
        if (e != cudaSuccess || mp <= 0) {
            (void)cudaGetLastError();
            mp = device_sm_count() / 2;
        }
        return cudaSuccess;
    });
    if (se != cudaSuccess) return se;
    const long long np = items < max_pairs ? items : max_pairs;
    cfg.gridDim = dim3((unsigned)(2 * np), 1, 1);
    static const char *names[4] = {"umma_ref_proj", "umma_distance_topk", "umma_swiglu_diff",
                                   "umma_z_quant"};
    ProfScope prof(names[MODE], s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a0, a1, b, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_umma_compress(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                                 const void *W1t, const void *W2t, const void *W3t,
                                 const rkv_cache *cache, uint8_t *ws, const Workspace &wl,
                                 float *z_out, int32_t *status, cudaStream_t s)
{
    cudaError_t e;
    float *P12 = (float *)(ws + wl.P1);                        // interleaved {P1, P2}
    float *rn_max = (float *)(ws + wl.rn_max);
    float2 *cand = (float2 *)(ws + wl.cand);
    __nv_bfloat16 *dh_hi = (__nv_bfloat16 *)(ws + wl.dh_hi);
    __nv_bfloat16 *dh_lo = (__nv_bfloat16 *)(ws + wl.dh_lo);
    const bool fp8 = g.ref_dtype == RKV_FP8_E4M3;
    void *ref_mma = fp8 ? (void *)(ws + wl.ref_mma) : pool->ref_vec;
    const size_t zrow = (size_t)g.LB * g.n_ref * g.d_ff * 2; // the all-zero projection row
    float *xnorm = (float *)(ws + wl.xnorm);
    if ((e = launch_prep_refs(g, pool, ref_mma, rn_max, P12 + zrow, P12 + zrow + g.d_ff, s)) != cudaSuccess)
        return e;

    UmmaArgs a{};
    a.wait_cycles = kWaitCycles;
    a.skip_use = -1;
    a.LB = g.LB; a.B = g.B; a.T = g.T; a.W = g.W; a.d_ff = g.d_ff; a.d_c = g.d_c;
    a.n_ref = g.n_ref; a.bits = g.bits;
    a.P12 = P12; a.ref_sqnorm = pool->ref_sqnorm; a.pool_size = pool->pool_size;
    a.ref_slot = pool->ref_slot; a.cand = cand; a.ref_idx = (const int4 *)cache->ref_idx;
    uint8_t *copy_flag = ws + wl.copy_flag;
    a.copy_flag = copy_flag;
    a.dh_hi = dh_hi; a.dh_lo = dh_lo; a.codes = cache->codes; a.hdr = (float2 *)cache->hdr;
    a.z_out = z_out; a.status = status;
    a.dh_rows = g.T;
    const int kw = (g.W + kBK - 1) / kBK;
    const int ff_slices = (g.d_ff + kBM - 1) / kBM;
    // W_c2 at a 16-byte multiple after W_c1 (e.g. both in one allocation): the two gate
    // halves of a stage come in one TMA box
    const long long gate_off = (long long)((const char *)W2t - (const char *)W1t);
    const bool fused = gate_off > 0 && gate_off % 16 == 0 && gate_off < (1ll << 40);

    // token and reference rows: 128 per CTA; W_c1 / W_c2: 64 rows each per CTA;
    // W_c3: 128 rows (one CTA's half of a 256-column d_c tile)
    CUtensorMap mX, mW1, mW2, mW3, mHi, mLo, mR;
    if (!make_map(&mX, kv, g.W, g.T, g.LB, kBM) || !make_map(&mW1, W1t, g.W, g.d_ff, g.L, kBM / 2) ||
        !make_map(&mW2, W2t, g.W, g.d_ff, g.L, kBM / 2) ||
        !make_map(&mW3, W3t, g.d_ff, g.d_c, g.L, kHalfN) ||
        !make_map(&mHi, dh_hi, g.d_ff, g.T, g.LB, kBM) ||
        !make_map(&mLo, dh_lo, g.d_ff, g.T, g.LB, kBM))
        return cudaErrorInvalidValue;

    CUtensorMap mG1 = mW1;
    if (fused) {
        if (!make_map_gates(&mG1, W1t, gate_off, g.W, g.d_ff, g.L)) return cudaErrorInvalidValue;
        a.fused_gate = 1;
    }
    // the reference projections take the 16-row-group layout: one 4-D box per stage
    // when the gates are fused and d_ff is a multiple of 16, else 16-row boxes
    const bool fused16 = fused && g.d_ff % kGateRows == 0;
    CUtensorMap mP1, mP2;
    if (fused16) {
        if (!make_map_gates16(&mP1, W1t, gate_off, g.W, g.d_ff, g.L)) return cudaErrorInvalidValue;
        mP2 = mP1;
    } else if (!make_map(&mP1, W1t, g.W, g.d_ff, g.L, kGateRows) ||
               !make_map(&mP2, W2t, g.W, g.d_ff, g.L, kGateRows)) {
        return cudaErrorInvalidValue;
    }
    if (g.n_ref > 0) {
        if (!make_map(&mR, ref_mma, g.W, g.n_ref, g.LB, kHalfN)) return cudaErrorInvalidValue;
        // P1 | P2 for every reference
        UmmaArgs p = a;
        p.rows = g.n_ref; p.tiles_t = (g.n_ref + kTileM - 1) / kTileM; p.tiles_n = ff_slices;
        p.k_chunks = kw; p.a_sources = 1;
        p.fused_gate = fused16 ? 1 : 0;
        if ((e = run<M_P>(mP1, mP2, mR, p, s)) != cudaSuccess) return e;
        // distance expansion and per-item candidates
        UmmaArgs d = a;
        d.rows = g.T; d.tiles_t = g.n_mtiles; d.tiles_n = g.max_chunks;
        d.k_chunks = kw; d.a_sources = 1;
        d.xrows = (const __nv_bfloat16 *)kv; d.xnorm = xnorm;
        if ((e = run<M_DIST>(mX, mX, mR, d, s)) != cudaSuccess) return e;
    }
    int32_t *scan_list = (int32_t *)(ws + wl.scan_list);
    int2 *rr_list = (int2 *)(ws + wl.rr_list);
    if ((e = launch_topk_finalize(g, kv, ref_mma, 0, pool, cand, xnorm, rn_max, cache->ref_idx,
                                  copy_flag, scan_list, scan_list + (size_t)g.LB * g.T, rr_list,
                                  (int32_t *)(rr_list + (size_t)g.LB * g.T), status, s)) != cudaSuccess)
        return e;
    // a fixed schedule from position 0 whose stride divides 8 makes every position 0 mod 8
    // a reference: those rows are left out of S1's MMA, and dh holds only the other 7 of
    // every 8 positions, which S2 then runs over
    const bool skip8 = g.alpha == 0.0 && g.first == 0 && g.stride >= 1 && 8 % g.stride == 0 &&
                       g.T % 8 == 0;
    CUtensorMap mXs, mHc, mLc;
    const int Tc = g.T / 8 * 7;
    const bool compact = skip8 && make_map_skip(&mXs, kv, g.W, g.T, g.LB, 8) &&
                         make_map(&mHc, dh_hi, g.d_ff, Tc, g.LB, kBM) && make_map(&mLc, dh_lo, g.d_ff, Tc, g.LB, kBM);
    {
        UmmaArgs p = a;
        p.rows = g.T; p.tiles_t = g.n_mtiles; p.tiles_n = ff_slices;
        p.k_chunks = kw; p.a_sources = 1;
        if (compact) {
            p.dh_rows = Tc;
            if ((e = run<M_S1, 8>(mG1, mW2, mXs, p, s)) != cudaSuccess) return e;
        } else if ((e = run<M_S1>(mG1, mW2, mX, p, s)) != cudaSuccess) {
            return e;
        }
    }
    {
        UmmaArgs p = a;
        p.rows = compact ? Tc : g.T;
        p.tiles_t = (p.rows + kTileM - 1) / kTileM;
        p.tiles_n = (g.d_c + kBN - 1) / kBN;
        p.k_chunks = (g.d_ff + kBK - 1) / kBK; p.a_sources = 2;
        const long long fc = g_fault_cycles.exchange(0);
        const int fs = g_fault_skip.exchange(-1);
        if (fc > 0 && fs >= 0) {
            p.wait_cycles = fc;
            p.skip_use = fs;
        }
        if (compact) {
            if ((e = run<M_S2, 8>(mHc, mLc, mW3, p, s)) != cudaSuccess) return e;
        } else if ((e = run<M_S2>(mHi, mLo, mW3, p, s)) != cudaSuccess) {
            return e;
        }
    }
    return cudaSuccess;
}

}  // namespace rkv

using namespace rkv;

extern "C" rkv_status rkv_debug_wait_fault(int64_t wait_cycles, int32_t skip_use)
{
    if (wait_cycles < 10000 || wait_cycles > kWaitCycles || skip_use < 0) return RKV_ERR_INVALID_ARG;
    g_fault_skip.store(skip_use);
    g_fault_cycles.store(wait_cycles);
    return RKV_OK;
}
