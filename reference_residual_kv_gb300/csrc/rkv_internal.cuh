// rkv_internal.cuh -- declarations shared by the librkv translation units.
//
// Citations: [RKV §x = paper y] names a section of the reading-notes page
// "ResidualKV：基于参考向量与残差的 KV Cache 压缩" (arXiv 2602.08005v2) and the
// paper section it summarises.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda.h>
#include <stdint.h>
#include <stddef.h>

#include <mutex>

#include "../../include/rkv.h"

namespace rkv {

// Retrieval: number of expansion candidates kept per token and chunk, and the
// relative error budget of the tensor-core distance expansion.  A token's top-k
// is accepted from the expansion only if its k-th/(k+1)-th gap exceeds twice
// kTau * (max ||r||^2 + 2 ||x|| max ||r||); otherwise it is re-ranked with exact
// differences.
constexpr int kList = 8;                  // sorted list kept per row and column half (>= k + 1)
constexpr int kCand = 2 * kList;          // candidate entries per row and work item
constexpr float kTau = 1.0f / 32768.0f;   // 2^-15
constexpr int kMaxK = 4;                  // ref_idx rows are int4
static_assert(kList >= kMaxK + 1 && kList % 2 == 0,
              "a list must hold the (k+1)-th entry; entries go out as float4 pairs");

// tcgen05 GEMM tiling: 128 token rows x 256 columns, K chunks of 64 bf16.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kTileM = 2 * kBM;          // token rows of a CTA-pair tile (2-SM MMA, M = 256)
constexpr int kDistChunk = 16;            // N-tiles (4096 references) per distance work item

// Bounded waits: ~1 s at 2 GHz.
constexpr long long kWaitCycles = 2000000000LL;

struct Geometry {
    int L, B, LB, T, N, D, W, d_ff, d_c, k, bits, n_ref, n_groups, code_pitch;
    int kv_dtype, ref_dtype;
    int stride, first, n_sink;
    double alpha;
    int n_mtiles;        // ceil(T / kTileM): CTA-pair token tiles
    int max_chunks;      // distance work items per token tile
};

Geometry make_geometry(const rkv_params *p);

// Workspace carve-up (offsets in bytes from the workspace base, 256-aligned).
struct Workspace {
    size_t ref_mma;      // bf16 [LB][n_ref][W]   decoded FP8 references (FP8 only)
    size_t P1, P2;       // f32  [LB][n_ref][d_ff] (tensor-core path: P1 holds float2 {P1, P2})
    size_t rn_max;       // f32  [LB]
    size_t cand;         // f32x2 [LB][T][max_chunks][kCand]  (tensor-core path)
    size_t copy_flag;    // u8   [LB][T]  1: every chosen reference equals the token
    size_t xnorm;        // f32  [LB][T]  ||x||^2 of every token (tensor-core path)
    size_t scan_list;    // i32  [LB*T] tokens whose top-k needs a full exact scan, + count
    size_t rr_list;      // i32x2 [LB*T] tokens to re-rank or copy-check exactly, + count
    size_t dh_hi, dh_lo; // bf16 [LB][T][d_ff]   (tensor-core path)
    size_t dh32;         // f32  [LB][T][d_ff]   (fp32 path)
    size_t z32;          // f32  [LB][T][d_c]    (fp32 path)
    size_t total;
};
Workspace workspace_layout(const Geometry &g);

// ---- launchers (each returns cudaGetLastError()) ----------------------------
cudaError_t launch_build_schedule(const Geometry &g, const rkv_ref_pool *pool, cudaStream_t s);
cudaError_t launch_build_refs(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                              cudaStream_t s);
cudaError_t launch_prep_refs(const Geometry &g, const rkv_ref_pool *pool, void *ref_mma,
                             float *rn_max, float *zero_row1, float *zero_row2, cudaStream_t s);
cudaError_t launch_gather(const Geometry &g, const rkv_ref_pool *pool, const rkv_cache *cache,
                          const int32_t *sel, int n_sel, void *out_z, void *out_mean,
                          int out_dtype, int32_t *status, cudaStream_t s);

// fp32 path (CUDA cores): projections, top-k by exact distances, z, quantisation
cudaError_t launch_simt_compress(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                                 const void *W1t, const void *W2t, const void *W3t,
                                 const rkv_cache *cache, uint8_t *ws, const Workspace &wl,
                                 float *z_out, int32_t *status, cudaStream_t s);

// bf16 path (tcgen05 + TMA)
cudaError_t launch_umma_compress(const Geometry &g, const void *kv, const rkv_ref_pool *pool,
                                 const void *W1t, const void *W2t, const void *W3t,
                                 const rkv_cache *cache, uint8_t *ws, const Workspace &wl,
                                 float *z_out, int32_t *status, cudaStream_t s);

// top-k finalisation shared by both paths: exact re-rank / full scan
cudaError_t launch_topk_finalize(const Geometry &g, const void *kv, const void *ref_exact,
                                 int ref_exact_is_f32, const rkv_ref_pool *pool,
                                 const float2 *cand, const float *xnorm, const float *rn_max,
                                 int32_t *ref_idx, uint8_t *copy_flag, int32_t *scan_list,
                                 int32_t *scan_count, int2 *rr_list, int32_t *rr_count,
                                 int32_t *status, cudaStream_t s);

int device_sm_count();

// ---- per-device host state ----------------------------------------------------
// Launch facts that belong to a device (a kernel's raised shared-memory limit, its
// cluster occupancy, the address of a __device__ array) are set up once per device,
// on the first call that reaches it, under std::call_once: several host threads and
// several devices in one process each get their own.
constexpr int kMaxDevices = 64;
int current_device();   // the calling thread's current device; -1 on error

template <class T>
struct PerDevice {
    std::once_flag once[kMaxDevices];
    cudaError_t err[kMaxDevices];
    T value[kMaxDevices];
};

// Runs setup(value&) once for the current device; returns its error and the value.
template <class T, class F>
cudaError_t per_device(PerDevice<T> &pd, T &value, F setup)
{
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(pd.once[dev], [&] { pd.err[dev] = setup(pd.value[dev]); });
    value = pd.value[dev];
    return pd.err[dev];
}

// bf16 [batch][rows][inner] tensor map, box = 64 (inner) x box_rows, 128-byte swizzle
// (rkv_umma.cu); false if the driver rejects it.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
              uint64_t batch, uint32_t box_rows);
bool make_map_store(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t batch,
                    uint32_t box_inner, uint32_t box_rows);

// single-token write (rkv_pool.cu: the pool entry; rkv_append.cu: the record)
cudaError_t launch_append_ref(const Geometry &g, const void *kv_new, int t, const rkv_ref_pool *pool,
                              cudaStream_t s);
size_t append_workspace_bytes(const Geometry &g);
cudaError_t launch_append(const Geometry &g, const void *kv_new, int t, const rkv_ref_pool *pool,
                          const void *W1t, const void *W2t, const void *W3t, const rkv_cache *cache,
                          void *ws, int32_t *status, cudaStream_t s);

// sparse attention over the restored set (rkv_attention.cu)
size_t attention_workspace_bytes(const Geometry &g, int H, int n_sel);
cudaError_t launch_attention(const Geometry &g, int H, const void *q, const void *kh, const void *vh,
                             const int32_t *sel, int n_sel, float *out, void *workspace, cudaStream_t s);

// restore of K and V for selected tokens (rkv_restore.cu)
cudaError_t launch_restore(const Geometry &g, const rkv_ref_pool *pool, const rkv_cache *cache,
                           const void *Wd, const int32_t *sel, int n_sel, double rope_base,
                           void *out_k, void *out_v, int32_t *status, cudaStream_t s);

// per-kernel event timing (rkv_prof.cu); no-ops unless rkv_profile_enable(1)
void prof_begin(const char *name, cudaStream_t s);
void prof_end(cudaStream_t s);
struct ProfScope {
    cudaStream_t s;
    ProfScope(const char *name, cudaStream_t st) : s(st) { prof_begin(name, st); }
    ~ProfScope() { prof_end(s); }
};

// ---- device helpers ---------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t *st, int code)
{
    if (st) atomicCAS(st, 0, code);
}

// Number of N-tiles (256 references) the 256-token pair tile m needs: its last row's pool.
__device__ __forceinline__ int dist_ntiles(const int32_t *pool_size, int T, int m)
{
    int last = min(T, (m + 1) * kTileM) - 1;
    int pool = pool_size[last];
    return (pool + kBN - 1) / kBN;
}

__device__ __forceinline__ float silu(float u)
{
    return u / (1.0f + __expf(-u));
}

// [RKV §2.4 = Sec. IV-A] min/max quantisation of one group of 32 latent values.
// delta = (max - min)/(2^b - 1) (IEEE division), q = floor((z - min)/delta + 1/2)
// clamped to [0, 2^b - 1]; max == min stores the constant with delta = 0, q = 0.
// Packs INT4 as 4 words (coordinate 2j low nibble of byte j) and INT2 as 2 words
// (coordinate 4j+i in bits 2i..2i+1 of byte j).
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c)
{
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// max of three that returns NaN if any input is NaN
__device__ __forceinline__ float max3f_nan(float a, float b, float c)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// bits [0, len) of a inserted into b at bit pos
__device__ __forceinline__ uint32_t bfi32(uint32_t a, uint32_t b, int pos, int len)
{
    uint32_t r;
    asm("bfi.b32 %0, %1, %2, %3, %4;" : "=r"(r) : "r"(a), "r"(b), "r"(pos), "r"(len));
    return r;
}
__device__ __forceinline__ void quant_group32(const float (&v)[32], int bits, uint32_t (&w)[4],
                                              float &zmin, float &delta)
{
    // extremes by three-input min/max: a chain of 15 steps per extreme
    float lo = fminf(v[0], v[1]), hi = fmaxf(v[0], v[1]);
#pragma unroll
    for (int j = 2; j < 32; j += 2) {
        lo = min3f(lo, v[j], v[j + 1]);
        hi = max3f(hi, v[j], v[j + 1]);
    }
    const int qmax = (1 << bits) - 1;
    zmin = lo;
    w[0] = w[1] = w[2] = w[3] = 0u;
    if (hi == lo) {
        delta = 0.0f;
        return;
    }
    const float dl = __fdiv_rn(__fsub_rn(hi, lo), (float)qmax);
    delta = dl;
    // q = floor(RN(RN(d/delta) + 1/2)) with d = v - lo in [0, hi - lo].  It is first
    // estimated from x = d RN(1/delta), rounded to the nearest integer inside the same
    // FMA (adding 1.5 2^23 leaves round(x) in the low mantissa bits), and r = x - round(x)
    // from one more FMA.  x lies within 2^-19 of RN(d/delta) (RN(1/delta) is within
    // 2^-24 relative and the quotient is at most 15, within 2^-20 of its rounding); so
    // where |r| is at least 2^-17 short of 1/2, RN(d/delta) is more than 2^-18 away from
    // the half-integer where floor(. + 1/2) changes, the rounding of RN(d/delta) + 1/2
    // (at most 2^-20) cannot cross it, and q = round(x) (in [0, 2^b - 1]: 0 <= x <=
    // (2^b - 1)(1 + 2^-22)).  If any coordinate of the group is nearer than that (or delta
    // is too small for a finite reciprocal) the correctly rounded division decides them all.
    const float rdl = __frcp_rn(dl);
    constexpr float kMagic = 12582912.0f;     // 1.5 * 2^23
    // fast path, two coordinates per packed operation: t = x + 1.5 2^23 rounded, whose low
    // mantissa bits are round(x); r = x - round(x) = x + (1.5 2^23 - t); the group takes
    // this path when every |r| is at least 2^-17 short of 1/2
    const float2 nlo = make_float2(-lo, -lo), rdl2 = make_float2(rdl, rdl);
    const float2 mg = make_float2(kMagic, kMagic);
    float rmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 d = __fadd2_rn(make_float2(v[j], v[j + 1]), nlo);
        const float2 t = __ffma2_rn(d, rdl2, mg);
        const float2 nq = __fadd2_rn(mg, make_float2(-t.x, -t.y));
        const float2 r = __ffma2_rn(d, rdl2, nq);
        rmax = max3f_nan(rmax, fabsf(r.x), fabsf(r.y));   // a NaN input takes the exact path
        const uint32_t q0 = __float_as_uint(t.x), q1 = __float_as_uint(t.y);   // code in the low bits
        if (bits == 4) {
            w[j >> 3] = bfi32(q0, w[j >> 3], 4 * (j & 7), 4);
            w[j >> 3] = bfi32(q1, w[j >> 3], 4 * ((j + 1) & 7), 4);
        } else {
            w[j >> 4] = bfi32(q0, w[j >> 4], 2 * (j & 15), 2);
            w[j >> 4] = bfi32(q1, w[j >> 4], 2 * ((j + 1) & 15), 2);
        }
    }
    if (dl >= 0x1p-100f && rmax <= 0.5f - 0x1p-17f) return;
    // near a tie somewhere in the group (or delta too small for a finite reciprocal): the
    // correctly rounded division for every coordinate
    w[0] = w[1] = w[2] = w[3] = 0u;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float u = __fadd_rn(__fdiv_rn(__fsub_rn(v[j], lo), dl), 0.5f);
        int q = (int)floorf(u);
        q = q < 0 ? 0 : (q > qmax ? qmax : q);
        if (bits == 4)
            w[j >> 3] |= (uint32_t)q << (4 * (j & 7));
        else
            w[j >> 4] |= (uint32_t)q << (2 * (j & 15));
    }
}

}  // namespace rkv
