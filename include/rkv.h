/*
 * rkv.h -- C ABI of librkv: the ResidualKV cache-write path and its sparse read
 * path on one GB300 GPU (sm_103a).
 *
 * Citations name sections of the reading-notes page "ResidualKV：基于参考向量与
 * 残差的 KV Cache 压缩" (on "ResidualKV: Residual-Based KV Cache Compression for
 * Efficient Long-Context Inference", arXiv 2602.08005v2), written [RKV §x = paper y].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All array arguments are DEVICE pointers owned by the caller (for instance
 *   torch allocations); the library keeps no pointer after a call returns and
 *   allocates no device memory of its own.  Scratch comes from a caller-provided
 *   workspace whose size rkv_query_sizes() reports.
 * - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *   default stream) and runs asynchronously; outputs are valid once the stream
 *   has been synchronised.
 * - Every device buffer must start on a 16-byte boundary.
 * - Host-side validation runs before anything is enqueued: on an error nothing is
 *   launched and the function returns the error.  A launch failure returns
 *   RKV_ERR_CUDA.  Errors found on the device (an out-of-range index, a wait
 *   that timed out) are written to *dev_status (an int32 in device memory that
 *   the caller sets to RKV_OK before the call; the first error wins) and the
 *   kernel skips the offending work instead of faulting.  Nothing traps, exits
 *   or prints.
 *
 * Shapes (per rkv_params):  L layers, B sequences per layer, T tokens per
 * sequence, W = 2*N*D (K of all heads concatenated with V of all heads, pre-RoPE,
 * [RKV §2.1 = Sec. IV-A]), n_ref references per sequence (rkv_n_ref()).
 * Per-(layer, sequence) arrays are stacked with the layer index outermost:
 * index lb = layer*B + b.
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rkv_status {
    RKV_OK = 0,
    RKV_ERR_INVALID_ARG = 1,     /* null pointer, bad size or inconsistent params   */
    RKV_ERR_UNSUPPORTED = 2,     /* valid for the method, not handled by this library */
    RKV_ERR_ALIGNMENT = 3,       /* a buffer is not 16-byte aligned                  */
    RKV_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed             */
    RKV_ERR_INDEX = 5,           /* device-detected: index out of range              */
    RKV_ERR_DEVICE_TIMEOUT = 6,  /* device-detected: a bounded wait expired          */
    RKV_ERR_WORKSPACE = 7        /* workspace smaller than rkv_query_sizes() asks    */
} rkv_status;

typedef enum rkv_dtype {
    RKV_F32 = 0,
    RKV_BF16 = 1,
    RKV_FP8_E4M3 = 2             /* OCP OFP8 E4M3: round to nearest even, saturating */
} rkv_dtype;

typedef struct rkv_params {
    int32_t L;          /* layers; each has its own compressor weights               */
    int32_t B;          /* sequences per layer (same T, same reference schedule)     */
    int32_t T;          /* tokens per sequence, >= 1                                  */
    int32_t N, D;       /* KV heads and head dim: W = 2*N*D, W % 8 == 0               */
    int32_t d_ff;       /* compressor hidden width   [RKV §2.3 = Sec. IV-A]           */
    int32_t d_c;        /* latent code width, d_c % group == 0                        */
    int32_t k;          /* references per token, 1..4 (paper default 4) [RKV §2.2]    */
    int32_t group;      /* quantisation group, 32 [RKV §2.4]                          */
    int32_t bits;       /* 2 or 4 [RKV §2.4]                                          */
    int32_t kv_dtype;   /* RKV_F32 or RKV_BF16: kv and compressor weights             */
    int32_t ref_dtype;  /* kv_dtype, or RKV_FP8_E4M3 (bf16 kv only) [RKV §2.4 = V-A]  */
    int32_t stride;     /* reference stride s (s0 of the dynamic schedule), >= 1      */
    int32_t first;      /* position of the first reference, 0 <= first               */
    double  alpha;      /* stride growth; 0 = fixed stride [RKV §2.6 = Sec. IV-A]     */
    int32_t n_sink;     /* sink tokens of the dynamic schedule, >= 0                  */
    int32_t reserved;   /* set to 0                                                   */
} rkv_params;

/* Reference pool [RKV §2.2, §2.6 = Sec. IV-A]; filled by rkv_build_ref_pool.
 * References are stored uncompressed (or FP8) and are the values every later
 * step uses (encoder and decoder share them [RKV §2.5 = Sec. IV-B]).            */
typedef struct rkv_ref_pool {
    int32_t *ref_pos;     /* [n_ref]  position of reference slot m, ascending       */
    int32_t *ref_slot;    /* [T]      slot of token t if it is a reference, else -1 */
    int32_t *pool_size;   /* [T]      number of references at positions < t         */
    void    *ref_vec;     /* [L*B][n_ref][W] in ref_dtype                            */
    float   *ref_sqnorm;  /* [L*B][n_ref] squared L2 norm of the stored reference   */
} rkv_ref_pool;

/* Compressed per-token records [RKV §2.4]: each token owns its codes, its group
 * extremes and its reference relation, so one token can be read alone.
 *  codes:   [L*B][T][d_c*bits/8] bytes; INT4: coordinate 2j in the low nibble of
 *           byte j, 2j+1 in the high nibble; INT2: coordinate 4j+i in bits 2i..2i+1.
 *  hdr:     [L*B][T][d_c/group][2] float {z_min, delta}; z~ = q*delta + z_min.
 *  ref_idx: [L*B][T][4] int32 reference slots, ascending, -1 padded (k_t = number
 *           of entries >= 0).  A reference token stores {own slot,-1,-1,-1}, zero
 *           codes and zero extremes, so that a read returns the reference itself. */
typedef struct rkv_cache {
    uint8_t *codes;
    float   *hdr;
    int32_t *ref_idx;
} rkv_cache;

/* Reference schedule [RKV §2.6 = Sec. IV-A]: p_0 = first and
 *   p_{m+1} = p_m + stride + floor(alpha * (p_m - n_sink)),
 * every p_m < T; alpha = 0 is the fixed stride.  The first step must be >= 1
 * (stride + floor(alpha (first - n_sink)) >= 1), otherwise the params are invalid.
 * Returns the number of references per sequence, or -1 on invalid params.        */
int32_t rkv_n_ref(const rkv_params *p);

/* Host-only: bytes the caller must provide.  Any output pointer may be NULL.
 *  pool_bytes:      ref_vec + ref_sqnorm + the three int32 schedule arrays
 *  cache_bytes:     codes + hdr + ref_idx
 *  workspace_bytes: scratch for rkv_compress                                     */
rkv_status rkv_query_sizes(const rkv_params *p, size_t *pool_bytes, size_t *cache_bytes,
                           size_t *workspace_bytes);

/* Step 0 of the write path: the reference schedule [RKV §2.6 = Sec. IV-A] and
 * the stored references.  kv: [L*B][T][W] in kv_dtype.  Writes every field of
 * *pool; with ref_dtype = RKV_FP8_E4M3 each reference is rounded to E4M3
 * (nearest even, saturating) and ref_sqnorm is taken over the rounded values.    */
rkv_status rkv_build_ref_pool(const rkv_params *p, const void *kv, const rkv_ref_pool *pool,
                              void *stream);

/* The write path [RKV §2.2-§2.4 = Sec. IV-A] for every token of every (layer,
 * sequence), given the pool from rkv_build_ref_pool:
 *  1. retrieval: for a non-reference token t, the k_t = min(k, pool_size[t])
 *     references with pos < t nearest in squared L2 (ties -> lower slot);
 *  2. mean of those references in KV space;
 *  3. z_t = f_c(kv_t) - f_c(mean_t),  f_c(x) = (Swish(x W_c1) ⊙ x W_c2) W_c3;
 *  4. per-token groups of `group` coordinates quantised with min/max scaling to
 *     `bits` bits (a constant group is stored exactly: delta = 0).
 * Weights are stored out-major, one set per layer, in kv_dtype:
 *  W1t, W2t: [L][d_ff][W] with W1t[f][c] = W_c1[c][f];  W3t: [L][d_c][d_ff].
 *  (bf16 path: if W2t lies at a positive multiple of 16 bytes after W1t, e.g. both in
 *  one allocation, the two gate halves load as one tile per pipeline stage, which is
 *  faster; any other placement is equally correct.)
 * workspace: >= workspace_bytes from rkv_query_sizes, 256-byte aligned.
 * z_out (nullable): [L*B][T][d_c] fp32 unquantised z (0 for reference tokens and for
 * tokens equal to all their chosen references).
 * dev_status: device int32, set to RKV_OK by the caller.                         */
rkv_status rkv_compress(const rkv_params *p, const void *kv, const rkv_ref_pool *pool,
                        const void *W1t, const void *W2t, const void *W3t,
                        const rkv_cache *cache, void *workspace, size_t workspace_bytes,
                        float *z_out, int32_t *dev_status, void *stream);

/* The sparse read [RKV §2.7 = Sec. IV-C]: for each selected token read only its
 * own record and its references, and return
 *   out_z[lb][i]    = dequantised z~ of token sel[lb][i]        ([L*B][n_sel][d_c])
 *   out_mean[lb][i] = mean of its stored references in KV space ([L*B][n_sel][W])
 * in out_dtype (RKV_F32 or RKV_BF16): z~ by one fp32 fma per coordinate, the mean
 * as fp32 sums in ascending slot order times 1/k, each rounded once to out_dtype.
 * sel: [L*B][n_sel] int32 token positions; an entry of -1 is padding and yields
 * zero rows; an entry >= T sets RKV_ERR_INDEX and yields zero rows.  Unselected
 * tokens' records are never read.  With n_sel = T and sel = 0..T-1 this is the
 * paper's standalone mode (every code restored).                                 */
rkv_status rkv_gather_dequant(const rkv_params *p, const rkv_ref_pool *pool,
                              const rkv_cache *cache, const int32_t *sel, int32_t n_sel,
                              void *out_z, void *out_mean, int32_t out_dtype,
                              int32_t *dev_status, void *stream);

/* Restore K and V of the selected tokens [RKV §2.5 = Sec. IV-B; §2.7 = Sec. IV-C]:
 *   KV^_t = z~_t W_d + mean_t   (z~_t, mean_t as returned by rkv_gather_dequant),
 *   K^_t = KV^_t[0, N D),  V^_t = KV^_t[N D, 2 N D),  head h = [h D, (h+1) D);
 * every key head is rotated at the token's own position t (its index in the
 * sequence; the restored key is pre-RoPE [RKV §2.1]): coordinate pairs (2i, 2i+1)
 * by the angle t * rope_base^(-2i/D).  The page does not fix the RoPE variant; this
 * is the rotary embedding as first defined, with consecutive pairs.  The angle is
 * formed in turns, t * (theta_i / 2 pi) mod 1, with theta_i / 2 pi rounded to 32
 * fractional bits on the host (an angle error below t * 2^-33 turns, 1e-4 rad at
 * t = 2^17), then evaluated on [-pi, pi).
 * Wd: [L][2 N D][d_c] out-major (Wd[c][j] = W_d[j][c]), bf16.
 * sel: [L*B][n_sel] int32 token positions (-1: padding, zero rows; >= T or a stored
 * slot >= n_ref: RKV_ERR_INDEX in dev_status and zero rows).
 * out_k, out_v: bf16 [L*B][n_sel][N D], 16-byte aligned (written by TMA tile stores).
 * The decoder runs on the tensor cores with z~ rounded to bf16 and fp32 accumulation;
 * the mean is an fp32 sum in ascending slot order times 1/k.
 * Requires kv_dtype bf16, d_c in {256, 512}, 2 N D a multiple of 256, D a multiple
 * of 32 and at most 256, rope_base > 0 (else RKV_ERR_UNSUPPORTED / _INVALID_ARG).    */
rkv_status rkv_restore_kv(const rkv_params *p, const rkv_ref_pool *pool, const rkv_cache *cache,
                          const void *Wd, const int32_t *sel, int32_t n_sel, double rope_base,
                          void *out_k, void *out_v, int32_t *dev_status, void *stream);

/* Sparse attention of one decode step over the restored set [RKV §2.7 = Sec. IV-C]:
 *   out[lb][j] = softmax( q[lb][j] K^_I^T / sqrt(D) ) V^_I   for each query head j < H,
 * query head j reading key/value head floor(j / (H/N)) (grouped heads; the page writes
 * the formula per head).  I = the rows n < n_sel of k_hat/v_hat whose sel[lb][n] is a
 * position in [0, T) (padding and out-of-range entries, zero rows of rkv_restore_kv,
 * are left out); an empty I gives zeros.  Softmax and sums in fp32; for D = 128 the
 * scores and the weighted sums of V^ run on the tensor cores (bf16 q, K^, V^ with fp32
 * accumulation; the probabilities enter as a bf16 hi + lo pair, relative error about
 * 2^-16), other D on CUDA cores in fp32.  On the tensor-core path a device wait that runs
 * out (about a second) leaves NaN in the affected head's outputs.
 * q: bf16 [L*B][H][D]; k_hat, v_hat: bf16 [L*B][n_sel][N D] (rkv_restore_kv's
 * outputs); sel: as given to rkv_restore_kv; out: fp32 [L*B][H][D].
 * workspace: >= the bytes rkv_attention_workspace reports (per-split partials).
 * Requires kv_dtype bf16, D in {64, 128, 256}, H a multiple of N with H/N <= 8
 * (H/N <= 4 for D = 256).                                                          */
rkv_status rkv_attention_workspace(const rkv_params *p, int32_t H, int32_t n_sel, size_t *bytes);
rkv_status rkv_sparse_attention(const rkv_params *p, int32_t H, const void *q, const void *k_hat,
                                const void *v_hat, const int32_t *sel, int32_t n_sel, float *out,
                                void *workspace, size_t workspace_bytes, void *stream);

/* Decode-time write of one new token per (layer, sequence) [RKV §2.7 = Sec. IV-C,
 * step 4 of a decode step]: the token at position t (the same t for every sequence)
 * joins the cache.  At a reference position of the schedule its row is stored in the
 * pool (copy or FP8 encode, squared norm) and its record is the reference record;
 * otherwise it is encoded like rkv_compress encodes it: the k_t nearest references
 * with pos < t by exact squared distance (ties to the lower slot), their mean in KV
 * space, z = f_c(kv) - f_c(mean) (fp32 on CUDA cores), group quantisation.
 * p->T is the capacity (0 <= t < T); tokens 0..t-1 must already be written (by
 * rkv_compress, or by earlier calls) into `pool` and `cache`, whose schedule
 * (rkv_build_ref_pool for capacity T) is fixed in advance.
 * kv_new: [L*B][W] in kv_dtype; weights as for rkv_compress.
 * workspace: >= workspace_bytes of rkv_query_sizes, 256-byte aligned.               */
rkv_status rkv_append_token(const rkv_params *p, const void *kv_new, int32_t t,
                            const rkv_ref_pool *pool, const void *W1t, const void *W2t,
                            const void *W3t, const rkv_cache *cache, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, void *stream);

/* rkv_compress without a workspace argument: for callers that cannot allocate
 * device memory at the call site -- code running while a CUDA graph is captured
 * (cudaMalloc is not allowed there), runtimes whose device memory belongs to an
 * arena the caller cannot reach, serving loops that must not allocate after
 * start-up.  The paper has no counterpart; this is an interface convenience.
 * Same arguments, semantics and results as rkv_compress, except that the scratch
 * is a fixed 64 MiB array inside the library's device image (a device holds it
 * until the process exits; with lazy module loading it is reserved when this entry
 * point is first used on that device).  Problems whose rkv_query_sizes()
 * workspace exceeds 64 MiB return RKV_ERR_WORKSPACE and launch nothing (one
 * Llama-3.1-8B-shape layer of 8192 tokens fits).  It calls no cudaMalloc/cudaFree
 * and no allocating library routine.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  All calls share the one array and nothing in it needs to
 * start at zero (every byte read is written earlier in the same call), but calls
 * that overlap on the GPU -- on different streams, or from several host threads --
 * race on it: serialise them.                                                      */
rkv_status rkv_compress_noalloc(const rkv_params *p, const void *kv, const rkv_ref_pool *pool,
                                const void *W1t, const void *W2t, const void *W3t,
                                const rkv_cache *cache, float *z_out, int32_t *dev_status,
                                void *stream);

/* Diagnostics: per-kernel device time.  rkv_profile_enable(1) clears the record
 * and brackets every later kernel launch of the library with two CUDA events on
 * the launch stream; rkv_profile_enable(0) stops recording.  rkv_profile_collect
 * waits for the recorded events and writes, per kernel name, the summed elapsed
 * milliseconds and the launch count: names is a caller buffer of max_entries rows
 * of name_len chars.  Returns the number of rows written, or -1 on error.  Not
 * thread-safe; meant for benchmarks.                                             */
rkv_status rkv_profile_enable(int32_t on);
int32_t rkv_profile_collect(char *names, int32_t name_len, float *total_ms, int32_t *launches,
                            int32_t max_entries);

/* Test hook of the device-side timeout path (failure handling; the paper has no
 * counterpart).  Arms a one-shot fault that the next rkv_compress call with bf16 kv,
 * from any host thread, takes in its W_c3 kernel: every barrier wait of that kernel
 * gives up after wait_cycles SM clock cycles instead of about 2e9, and the second CTA
 * of every CTA pair skips its tile loads for its stage use number skip_use, so that a
 * wait runs out.  The kernel then sets RKV_ERR_DEVICE_TIMEOUT in *dev_status, lets the
 * copies and MMAs it issued finish, frees its tensor memory and returns: nothing
 * traps, and the context stays usable for later calls.  The records of that call are
 * incomplete.  For tests of the error path only.  Returns RKV_ERR_INVALID_ARG unless
 * 1e4 <= wait_cycles <= 2e9 and skip_use >= 0.                                      */
rkv_status rkv_debug_wait_fault(int64_t wait_cycles, int32_t skip_use);

/* Static description of a status code. */
const char *rkv_status_string(rkv_status s);

#ifdef __cplusplus
}
#endif
#endif /* RKV_H */
