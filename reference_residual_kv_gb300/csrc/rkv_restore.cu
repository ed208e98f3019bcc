// rkv_restore.cu -- restore K and V of the tokens a decode step selects
// [RKV §2.5 = Sec. IV-B, §2.7 = Sec. IV-C]:
//   KV^_t = z~_t W_d + mean_t,  K^ = KV^[0, N D), V^ = KV^[N D, 2 N D),
// z~_t = q delta + z_min (the token's own codes), mean_t = the mean of its stored
// references, and each key head rotated at the token's own position t (the restored
// key is pre-RoPE [RKV §2.1]): consecutive pairs (2i, 2i+1) by t * base^(-2i/D).
//
// One persistent kernel on CTA pairs issuing 2-SM MMAs (tcgen05.mma.cta_group::2,
// M = 256 selected tokens x N = 256 output columns x K = 16, bf16 in, fp32 in TMEM):
//   warp 0      TMA producer (both CTAs): this CTA's 128 rows of W_d (out-major) per
//               64-wide K chunk; both CTAs' copies complete on the leader's barrier
//   warp 1      TMEM allocation (both CTAs); MMA issue (leader)
//   warps 2..9  per item (256 selected tokens of one layer-sequence and a group of
//               consecutive N tiles): first write the CTA's 128 rows of z~ (dequantised
//               codes, bf16) into shared memory in the 128-byte-swizzled K-major layout
//               the MMA reads, resident for the group's N tiles; then, per N tile, read
//               the accumulator, add the reference mean, rotate key pairs and store bf16.
// Items split the N tiles into groups when that evens out the rounds of the pairs.
// Every mbarrier wait is bounded; on expiry the kernel reports RKV_ERR_DEVICE_TIMEOUT.
#include "rkv_internal.cuh"
#include "umma.cuh"

#include <cuda_fp16.h>
#include <math.h>
#include <string.h>

namespace rkv {
namespace {

constexpr int kEpi = 8;
constexpr int kThr = 64 + 32 * kEpi;
constexpr int kMaxDc = 512;                    // resident z~ tile: 128 rows x d_c bf16
constexpr int kZBytes = kBM * kMaxDc * 2;      // 128 KB
constexpr int kWBytes = (kBN / 2) * kBK * 2;   // 16 KB: this CTA's 128 W_d rows x 64
constexpr int kStages = 4;
// output staging: per epilogue warp two 32-row x 32-column bf16 tiles (64-byte swizzle),
// each written back by one TMA store
constexpr int kOutTile = 32 * 32 * 2;
constexpr int kOutBytes = kEpi * 2 * kOutTile;
constexpr int kSmem = kZBytes + kStages * kWBytes + kOutBytes + 1024 + 256;
static_assert(kSmem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
constexpr int kMaxPairs = 128;                 // D <= 256

struct RestoreArgs {
    int LB, B, T, n_sel, W, dk, D, d_c, bits, n_ref, ref_fp8;
    int tiles_t, n_tiles, k_chunks;
    int n_groups, group_tiles;                 // an item: one token tile x group_tiles N tiles
    int wide;                                  // the pool is 32-byte aligned: 32-byte loads
    const int32_t *sel;
    const uint8_t *codes;
    const float2 *hdr;
    const int4 *ref_idx;
    const void *ref_vec;
    __nv_bfloat16 *out_k, *out_v;
    int32_t *status;
    uint32_t turns[kMaxPairs];                 // theta_i / (2 pi) as a 0.32 fixed-point fraction
};

// cos and sin of pos * theta_i.  theta_i / (2 pi) is held as a 32-bit fixed-point
// fraction f_i (theta_i < 2 pi, so no integer part); pos * f_i mod 2^32, one integer
// multiply, is the angle's fraction of a turn, exact for that f_i.  Read as a signed
// 32-bit value it lies in [-1/2, 1/2) turns, so the sine and cosine are evaluated on
// [-pi, pi).  Rounding f_i to 32 bits moves the angle by at most pos * 2^-33 turns
// (1e-4 rad at pos = 2^17), far below the bf16 rounding of the output.
__device__ __forceinline__ void rope_cs(uint32_t pos, uint32_t f, float &c, float &s)
{
    const int32_t frac = (int32_t)(pos * f);
    __sincosf((float)frac * 1.4629180792671596e-09f, &s, &c);   // 2 pi / 2^32
}

// One lane's share of a token row of z~: coordinates [lane*cpl, (lane+1)*cpl),
// cpl = d_c/32 (8 or 16): its code words and its group's {z_min, delta}.
struct RowCodes {
    uint32_t w0, w1;
    float2 gh;
};

__device__ __forceinline__ RowCodes load_row(int lane, int d_c, int bits, const uint8_t *crow,
                                             const float2 *hrow, bool ok)
{
    RowCodes rc = {0u, 0u, make_float2(0.0f, 0.0f)};
    if (ok) {
        const int cpl = d_c >> 5;
        const int c0 = lane * cpl;
        rc.gh = __ldg(hrow + (c0 >> 5));
        const int nbytes = cpl * bits / 8;      // 2, 4 or 8
        const uint8_t *p = crow + c0 * bits / 8;
        if (nbytes == 8) { const uint2 u = __ldg((const uint2 *)p); rc.w0 = u.x; rc.w1 = u.y; }
        else if (nbytes == 4) rc.w0 = __ldg((const uint32_t *)p);
        else rc.w0 = __ldg((const unsigned short *)p);
    }
    return rc;
}

// Dequantise a lane's share (z~ = q delta + z_min, one fma) and write it as bf16 into
// the z~ tile, row r.  Layout: K chunk kc (64 coordinates) is a 128-row x 128-byte block
// at kc * 16 KB; the 16-byte unit j (8 coordinates) of row r sits at unit j ^ (r & 7).
// Rows that are not restored (padding, bad index) are written as zeros.
__device__ __forceinline__ void write_row(uint8_t *zt, int r, int lane, int d_c, int bits,
                                          const RowCodes &rc, bool ok)
{
    const int cpl = d_c >> 5;
    const int c0 = lane * cpl;
    const uint32_t w[2] = {rc.w0, rc.w1};
#pragma unroll
    for (int u8 = 0; u8 < 2; ++u8) {
        if (u8 * 8 >= cpl) break;
        __align__(16) __nv_bfloat162 o[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int c = u8 * 8 + e;            // coordinate within the lane
            int q0, q1;
            if (bits == 4) {
                q0 = (w[c >> 3] >> (4 * (c & 7))) & 15;
                q1 = (w[(c + 1) >> 3] >> (4 * ((c + 1) & 7))) & 15;
            } else {
                q0 = (w[c >> 4] >> (2 * (c & 15))) & 3;
                q1 = (w[(c + 1) >> 4] >> (2 * ((c + 1) & 15))) & 3;
            }
            const float z0 = ok ? fmaf((float)q0, rc.gh.y, rc.gh.x) : 0.0f;
            const float z1 = ok ? fmaf((float)q1, rc.gh.y, rc.gh.x) : 0.0f;
            o[e >> 1] = __float22bfloat162_rn(make_float2(z0, z1));
        }
        const int cc = c0 + u8 * 8;              // first coordinate of this unit
        const int kc = cc >> 6, j = (cc & 63) >> 3;
        *(uint4 *)(zt + kc * (kBM * 128) + r * 128 + ((j ^ (r & 7)) << 4)) = *(const uint4 *)o;
    }
}

// The stored bytes of the k references' values at 32 consecutive coordinates of one
// token (FP8: 32 bytes, bf16: 64 bytes per reference), loaded ahead of their use.
template <bool FP8> struct RefChunk {
    static constexpr int kU = FP8 ? 2 : 4;      // uint4 per reference
    uint4 u[4][kU];

    __device__ __forceinline__ void load(const RestoreArgs &a, const int (&slot)[4], int lb, int c0)
    {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (slot[q] < 0) continue;
            const size_t row = ((size_t)lb * a.n_ref + slot[q]) * a.W + c0;
            const uint4 *p = FP8 ? (const uint4 *)((const uint8_t *)a.ref_vec + row)
                                 : (const uint4 *)((const __nv_bfloat16 *)a.ref_vec + row);
            if (a.wide) {
                // 32 bytes per load (one L1 wavefront per row for two 16-byte units)
#pragma unroll
                for (int v = 0; v < kU; v += 2)
                    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                                 : "=r"(u[q][v].x), "=r"(u[q][v].y), "=r"(u[q][v].z), "=r"(u[q][v].w),
                                   "=r"(u[q][v + 1].x), "=r"(u[q][v + 1].y), "=r"(u[q][v + 1].z),
                                   "=r"(u[q][v + 1].w)
                                 : "l"(p + v));
            } else {
#pragma unroll
                for (int v = 0; v < kU; ++v) u[q][v] = __ldg(p + v);
            }
        }
    }

    // fp32 sum in ascending slot order: each value enters as one add of its exact
    // widening (FP8 E4M3 through fp16, bf16 directly) to the fp32 accumulator
    __device__ __forceinline__ void sum(const int (&slot)[4], float (&m)[32]) const
    {
#pragma unroll
        for (int j = 0; j < 32; ++j) m[j] = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (slot[q] < 0) continue;
#pragma unroll
            for (int v = 0; v < kU; ++v) {
                const uint32_t wv[4] = {u[q][v].x, u[q][v].y, u[q][v].z, u[q][v].w};
                if (FP8) {
                    // a word's four E4M3 bytes: its two 16-bit halves converted to fp16
                    // pairs, then four widening adds (byte i into accumulator i)
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        float *mm = m + v * 16 + 4 * w4;
                        asm("{\n\t.reg .b16 b0, b1;\n\t.reg .b32 p0, p1;\n\t.reg .f16 f0, f1, f2, f3;\n\t"
                            "mov.b32 {b0, b1}, %4;\n\t"
                            "cvt.rn.f16x2.e4m3x2 p0, b0;\n\tcvt.rn.f16x2.e4m3x2 p1, b1;\n\t"
                            "mov.b32 {f0, f1}, p0;\n\tmov.b32 {f2, f3}, p1;\n\t"
                            "add.rn.f32.f16 %0, f0, %0;\n\tadd.rn.f32.f16 %1, f1, %1;\n\t"
                            "add.rn.f32.f16 %2, f2, %2;\n\tadd.rn.f32.f16 %3, f3, %3;\n\t}"
                            : "+f"(mm[0]), "+f"(mm[1]), "+f"(mm[2]), "+f"(mm[3])
                            : "r"(wv[w4]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
                            "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
                            : "+f"(m[v * 8 + 2 * e]), "+f"(m[v * 8 + 2 * e + 1])
                            : "r"(wv[e]));
                }
            }
        }
    }
};

template <bool FP8>
__global__ void __launch_bounds__(kThr, 1)
k_restore(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmK,
          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ RestoreArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *zt = smem_raw + ((1024u - (um::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *wst = zt + kZBytes;                                  // W_d stages
    uint8_t *ostg = wst + kStages * kWBytes;                      // output tiles
    uint64_t *full = (uint64_t *)(ostg + kOutBytes);              // leader's: both CTAs' bytes
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 2;                                  // leader's: both epilogues
    uint64_t *zready = tempty + 2;                                 // leader's: both z~ tiles
    uint64_t *drain = zready + 1;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = um::cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            um::mbar_init(&full[s], 1);
            um::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            um::mbar_init(&tfull[b], 1);
            um::mbar_init(&tempty[b], 2 * kEpi);
        }
        um::mbar_init(zready, 2 * kEpi);
        um::mbar_init(drain, 1);
        *abort_flag = 0;
        um::fence_mbar_init();
    }
    if (warp == 1) {
        um::tmem_alloc2(tmem_slot, 512);
        um::tmem_relinquish2();
    }
    um::tc_fence_before();
    um::cluster_sync();
    um::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = a.LB * a.tiles_t * a.n_groups;
    const int pid = blockIdx.x / 2, npairs = gridDim.x / 2;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            um::prefetch_tmap(&tmW);
            int stage = 0;
            uint32_t ph = 0;
            uint32_t last_ph[kStages];
            bool used[kStages];
            for (int s = 0; s < kStages; ++s) { used[s] = false; last_ph[s] = 0; }
            bool ok = true;
            for (int i = pid; i < n_items && ok; i += npairs) {
                const int lz = (i / a.n_groups / a.tiles_t) / a.B;
                const int nb = (i % a.n_groups) * a.group_tiles;
                for (int n = nb; n < nb + a.group_tiles && ok; ++n) {
                    for (int kc = 0; kc < a.k_chunks; ++kc) {
                        const bool w = um::mbar_wait(&empty[stage], ph ^ 1u, kWaitCycles);
                        if (*abort_flag || !w) { ok = false; break; }
                        const uint32_t fb = um::smem_u32(&full[stage]);
                        if (leader) um::mbar_arrive_expect_tx(&full[stage], 2 * kWBytes);
                        um::tma_load_3d_pair(wst + stage * kWBytes, &tmW, leader ? fb : um::mapa(fb, 0),
                                             kc * kBK, n * kBN + (int)rank * (kBN / 2), lz);
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
            for (int s = 0; s < kStages; ++s)
                if (used[s]) um::mbar_wait(&empty[s], last_ph[s], kWaitCycles);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t ph = 0, cnt = 0, ic = 0;
            bool ok = true;
            const uint32_t idesc = um::idesc_bf16_f32(2 * kBM, kBN);
            const uint32_t zbase = um::smem_u32(zt);
            for (int i = pid; i < n_items && ok; i += npairs, ++ic) {
                // both CTAs' z~ tiles of this item are written
                const bool wz = um::mbar_wait(zready, ic & 1u, kWaitCycles);
                if (*abort_flag || !wz) { ok = false; break; }
                um::tc_fence_after();
                for (int n = 0; n < a.group_tiles && ok; ++n) {
                    const uint32_t buf = cnt & 1u, tph = (cnt >> 1) & 1u;
                    const bool w = um::mbar_wait(&tempty[buf], tph ^ 1u, kWaitCycles);
                    if (*abort_flag || !w) { ok = false; break; }
                    um::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * kBN;
                    for (int kc = 0; kc < a.k_chunks; ++kc) {
                        const bool wf = um::mbar_wait(&full[stage], ph, kWaitCycles);
                        if (*abort_flag || !wf) { ok = false; break; }
                        um::tc_fence_after();
                        const uint64_t ad = um::sdesc_sw128(zbase + kc * (kBM * 128));
                        const uint64_t bd = um::sdesc_sw128(um::smem_u32(wst + stage * kWBytes));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k)
                            um::mma2_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kc | k) != 0);
                        um::mma2_commit_mc(&empty[stage], 3);
                        if (++stage == kStages) { stage = 0; ph ^= 1u; }
                    }
                    if (!ok) break;
                    um::mma2_commit_mc(&tfull[buf], 3);
                    ++cnt;
                }
            }
            if (!ok) {
                set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            um::mma2_commit_mc(drain, 1);
            um::mbar_wait(drain, 0, kWaitCycles);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int row = q * 32 + lane;                      // TMEM lane = z~ row
        const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t zready_l = um::smem_u32(zready);
        uint32_t cnt = 0, sb = 0;
        bool ok = true;
        for (int i = pid; i < n_items; i += npairs) {
            const int lb = i / a.n_groups / a.tiles_t, t = (i / a.n_groups) % a.tiles_t;
            const int nb = (i % a.n_groups) * a.group_tiles, ne = nb + a.group_tiles;
            const int e0 = t * 2 * kBM + (int)rank * kBM;   // this CTA's first selected entry
            // (1) this warp's 16 rows of the CTA's z~ tile: every load first (the rows'
            // positions, then their codes and extremes), then dequantise and write
            constexpr int kRows = kBM / kEpi;
            const int rbase = (warp - 2) * kRows;
            int tsel = -1;
            if (lane < kRows && e0 + rbase + lane < a.n_sel)
                tsel = __ldg(a.sel + (size_t)lb * a.n_sel + e0 + rbase + lane);
            RowCodes rcs[kRows];
            bool okr[kRows];
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                const int tok = __shfl_sync(0xffffffffu, tsel, rr);
                okr[rr] = tok >= 0 && tok < a.T;
                const size_t rec = (size_t)lb * a.T + (okr[rr] ? tok : 0);
                rcs[rr] = load_row(lane, a.d_c, a.bits, a.codes + rec * (size_t)(a.d_c * a.bits / 8),
                                   a.hdr + rec * (a.d_c / 32), okr[rr]);
            }
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr)
                write_row(zt, rbase + rr, lane, a.d_c, a.bits, rcs[rr], okr[rr]);
            um::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (leader) um::mbar_arrive(zready);
                else um::mbar_arrive_cluster(um::mapa(zready_l, 0));
            }
            // (2) this thread's token: position, reference slots, 1/k
            const int e = e0 + row;
            int tok = e < a.n_sel ? __ldg(a.sel + (size_t)lb * a.n_sel + e) : -1;
            if (tok >= a.T) set_status(a.status, RKV_ERR_INDEX);
            bool okt = tok >= 0 && tok < a.T;
            int slot[4] = {-1, -1, -1, -1};
            int kk = 0;
            if (okt) {
                const int4 ix = __ldg(a.ref_idx + (size_t)lb * a.T + tok);
                slot[0] = ix.x; slot[1] = ix.y; slot[2] = ix.z; slot[3] = ix.w;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (slot[j] >= a.n_ref) { okt = false; set_status(a.status, RKV_ERR_INDEX); }
                    if (slot[j] >= 0) ++kk;
                }
            }
            const float inv_k = kk > 0 ? 1.0f / (float)kk : 0.0f;
            const uint32_t pos = (uint32_t)(okt ? tok : 0);
            // (3) the N tiles' accumulators; the next chunk's reference values are
            // loaded while this chunk is rotated and stored
            RefChunk<FP8> rch;
            if (okt) rch.load(a, slot, lb, nb * kBN + h * (kBN / 2));
            for (int n = nb; n < ne; ++n) {
                const uint32_t buf = cnt & 1u, tph = (cnt >> 1) & 1u;
                bool w = !*abort_flag && um::mbar_wait(&tfull[buf], tph, kWaitCycles);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                um::tc_fence_after();
                const uint32_t tb = tl + buf * kBN;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    const int col = h * (kBN / 2) + cc * 32;          // column within the tile
                    const int c0 = n * kBN + col;                     // output coordinate
                    float o[32];
                    um::tmem_ld32(tb + col, o);
                    if (okt) {
                        // KV^ = f_d(z~) + (sum of the references) * 1/k
                        float m[32];
                        rch.sum(slot, m);
                        const float2 ik2 = make_float2(inv_k, inv_k);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float2 r = __ffma2_rn(make_float2(m[2 * j], m[2 * j + 1]), ik2,
                                                        make_float2(o[2 * j], o[2 * j + 1]));
                            o[2 * j] = r.x;
                            o[2 * j + 1] = r.y;
                        }
                    }
                    const int g1 = n * 4 + cc + 1;
                    if (okt && g1 < ne * 4)
                        rch.load(a, slot, lb, (g1 >> 2) * kBN + h * (kBN / 2) + (g1 & 3) * 32);
                    const bool is_k = c0 < a.dk;
                    if (okt) {
                        if (is_k) {
                            const int p0 = (c0 % a.D) >> 1;           // first pair index
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                float cs, sn;
                                rope_cs(pos, a.turns[p0 + j], cs, sn);
                                const float x0 = o[2 * j], x1 = o[2 * j + 1];
                                // (x0 cs - x1 sn, x1 cs + x0 sn)
                                const float2 r = __ffma2_rn(make_float2(-x1, x0), make_float2(sn, sn),
                                                            __fmul2_rn(make_float2(x0, x1), make_float2(cs, cs)));
                                o[2 * j] = r.x;
                                o[2 * j + 1] = r.y;
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = 0.0f;
                    }
                    // the warp's 32 rows x 32 columns go through shared memory to one TMA
                    // store (rows past the selection are clipped by the tensor map); a
                    // staging buffer is rewritten once the store before the last has read it
                    uint8_t *stg = ostg + ((warp - 2) * 2 + sb) * kOutTile;
                    if (lane == 0) um::bulk_wait_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __align__(16) __nv_bfloat162 pk[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            pk[j] = __float22bfloat162_rn(make_float2(o[8 * u + 2 * j], o[8 * u + 2 * j + 1]));
                        // 64-byte swizzle: 16-byte unit u of row r at u ^ ((r / 2) % 4)
                        *(uint4 *)(stg + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) = *(const uint4 *)pk;
                    }
                    um::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        um::tma_store_3d(is_k ? &tmK : &tmV, stg, is_k ? c0 : c0 - a.dk, e0 + q * 32, lb);
                        um::bulk_commit();
                    }
                    sb ^= 1u;
                }
                um::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader) um::mbar_arrive_relaxed(&tempty[buf]);
                    else um::mbar_arrive_cluster_relaxed(um::mapa(um::smem_u32(&tempty[buf]), 0));
                }
                ++cnt;
            }
            if (!ok) break;
        }
        // the warp's stores complete before the CTA leaves
        if (lane == 0) um::bulk_wait_all();
        __syncwarp();
        if (!ok) {
            set_status(a.status, RKV_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    }

    um::tc_fence_before();
    um::cluster_sync();
    if (warp == 1) {
        um::tc_fence_after();
        um::tmem_dealloc2(tmem_base, 512);
    }
}

}  // namespace

cudaError_t launch_restore(const Geometry &g, const rkv_ref_pool *pool, const rkv_cache *cache,
                           const void *Wd, const int32_t *sel, int n_sel, double rope_base,
                           void *out_k, void *out_v, int32_t *status, cudaStream_t s)
{
    RestoreArgs a;
    memset((void *)&a, 0, sizeof(a));
    a.LB = g.LB; a.B = g.B; a.T = g.T; a.n_sel = n_sel; a.W = g.W; a.dk = g.W / 2;
    a.D = g.D; a.d_c = g.d_c; a.bits = g.bits; a.n_ref = g.n_ref;
    a.ref_fp8 = g.ref_dtype == RKV_FP8_E4M3;
    a.tiles_t = (n_sel + kTileM - 1) / kTileM;
    a.n_tiles = g.W / kBN;
    // rows and 32-column chunks then start on 32-byte boundaries as well
    a.wide = ((uintptr_t)pool->ref_vec & 31u) == 0 && ((size_t)g.W * (a.ref_fp8 ? 1 : 2)) % 32 == 0;
    a.n_groups = 1;
    a.group_tiles = a.n_tiles;
    a.k_chunks = g.d_c / kBK;
    a.sel = sel; a.codes = cache->codes; a.hdr = (const float2 *)cache->hdr;
    a.ref_idx = (const int4 *)cache->ref_idx; a.ref_vec = pool->ref_vec;
    a.out_k = (__nv_bfloat16 *)out_k; a.out_v = (__nv_bfloat16 *)out_v; a.status = status;
    for (int i = 0; i < a.D / 2; ++i) {
        // the fraction of a turn of theta_i (whole turns do not move the angle)
        const double th = pow(rope_base, -2.0 * (double)i / (double)a.D);
        double f = th / (2.0 * 3.14159265358979323846);
        f -= floor(f);
        a.turns[i] = (uint32_t)(llrint(f * 4294967296.0) & 0xffffffffLL);
    }

    auto kern = a.ref_fp8 ? k_restore<true> : k_restore<false>;
    if ((long long)g.LB * a.tiles_t <= 0) return cudaSuccess;
    CUtensorMap mW, mK, mV;
    if (!make_map(&mW, Wd, g.d_c, g.W, g.L, kBN / 2) ||
        !make_map_store(&mK, out_k, a.dk, n_sel, g.LB, 32, 32) ||
        !make_map_store(&mV, out_v, a.dk, n_sel, g.LB, 32, 32))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThr, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // per device and reference type: the raised shared-memory limit, then the pairs
    // that fit at once
    static PerDevice<int> setup[2];
    int max_pairs = 0;
    cudaError_t se = per_device(setup[a.ref_fp8 ? 1 : 0], max_pairs, [&](int &mp) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
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
    // N-tile groups: the split whose rounds of items over the pairs, each costing its
    // tiles plus about half a tile for writing the z~ tile, finish first
    {
        const long long base = (long long)g.LB * a.tiles_t;
        double best = 0.0;
        for (int ng = 1; ng <= a.n_tiles; ng *= 2) {
            if (a.n_tiles % ng) continue;
            const long long rounds = (base * ng + max_pairs - 1) / max_pairs;
            const double cost = (double)rounds * ((double)(a.n_tiles / ng) + 0.5);
            if (ng == 1 || cost < best) { best = cost; a.n_groups = ng; }
        }
        a.group_tiles = a.n_tiles / a.n_groups;
    }
    const long long items = (long long)g.LB * a.tiles_t * a.n_groups;
    const long long np = items < max_pairs ? items : max_pairs;
    cfg.gridDim = dim3((unsigned)(2 * np), 1, 1);
    ProfScope prof("restore_kv", s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mW, mK, mV, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace rkv
