/*
 * mhc_seam.h -- C ABI of libmhcseam, the GB300 (sm_103a) delayed mHC seam.
 *
 * The seam is the hyper-connection work between two sub-layers of a model
 * whose residual is n = 4 bf16 streams of width H ("[FlyDSL] Single-launch
 * Mega-mHC on gfx950", Motivation; "[Triton/Gluon] [gfx950] [dsv4.1-flash] mHC
 * fused kernel", the five unfused mHC kernels it replaces).  One call, in this
 * order (the same page, Kernel Architecture, "Order"):
 *
 *   post-mix     R'[t,i,h] = sum_j comb_prev[t,i,j] R[t,j,h] + post_prev[t,i] Y[t,h]
 *                (stored bf16, round to nearest even)
 *   projection   s_R = sum R'^2 and d[k] = sum_{i,h} R'[t,i,h] fn[i*H+h, k], k < 24,
 *                over K = 4H, split over CTAs and reduced across the split
 *   rstd         rstd_R = 1 / sqrt(s_R / 4H + eps)
 *   gates        l[k] = alpha[g(k)] rstd_R d[k] + bias[k];  g = 0 (k<4), 1 (k<8), 2
 *                pre = sigmoid(l[0:4]), post = 2 sigmoid(l[4:8]),
 *                comb = Sinkhorn(exp(l[8:24]) as 4x4 row-major), 20 rounds of
 *                (row normalise, column normalise)
 *   layer input  x[t,h] = sum_i pre_prev[t,i] R'[t,i,h]  (the CARRIED pre)
 *   norm         norm[t,h] = bf16(x * rstd_x * gamma[h]),  rstd_x = 1/sqrt(mean x^2 + eps)
 *   mxfp8        optional: per 32 contiguous h, e = smallest integer with
 *                amax <= 448 * 2^e (amax floored at amax_floor), clamped to
 *                [-127, 127]; code = e4m3fn(norm * 2^-e) rounded to nearest even
 *                and saturating; scale byte = e + 127 (e8m0)  (Kernel
 *                Architecture, "out_dtype"; Limitations, ue8m0 notes)
 *
 * The stored bf16 R' feeds the sums, the projection and x.  The gates written
 * here are the next seam's carried gates ("delayed", single pass).
 *
 * Identity form (comb_prev, Y and post_prev all NULL): the first block's seam,
 * with nothing to mix in, R' = R bit for bit; residual_out is not written.
 * The page compares a "first block" form beside post and no_post ("[FlyDSL]
 * Single-launch Mega-mHC on gfx950", Correctness) without defining it; this
 * is the plainest reading.
 *
 * Conventions for every entry point:
 *  - Device pointers are caller-owned, dense, row-major and on the current
 *    device.  The library never allocates device memory.
 *  - Every call is asynchronous on `stream` (cudaStream_t passed as void*;
 *    NULL = legacy default stream) and returns a status: 0 on success, a
 *    negative mhc_status on a rejected call (nothing was launched), and
 *    MHC_ERR_CUDA when a CUDA call failed (mhc_last_error_string() says which).
 *  - T == 0 is valid and launches nothing.  Offsets are 64-bit.
 *  - Thread safety: calls may come from several host threads; a workspace
 *    must not be shared by calls that can overlap on the GPU.
 */
#ifndef MHC_SEAM_H
#define MHC_SEAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHC_OUT_BF16 = 0,     /* norm only */
    MHC_OUT_MXFP8 = 1,    /* norm + e4m3 codes + e8m0 scales, one per 32 elements */
    MHC_OUT_FP8_GRID = 2  /* norm + the bf16 grid: the same per-32 ue8m0 quantisation
                             dequantised, bf16(e4m3 value * 2^e) per element ("[FlyDSL]
                             Single-launch Mega-mHC on gfx950", Kernel Architecture,
                             out_dtype fp8_grid); streaming path only */
} mhc_out_mode;

typedef enum {
    MHC_OK = 0,
    MHC_ERR_NULL = -1,            /* a required pointer is NULL */
    MHC_ERR_SHAPE = -2,           /* T < 0, H <= 0, H % 8 != 0, or H % 32 != 0 for mxfp8 */
    MHC_ERR_ALIGN = -3,           /* a pointer breaks its alignment rule */
    MHC_ERR_INCOMPLETE_POST = -4, /* exactly one of Y, post_prev is NULL, or Y without comb_prev */
    MHC_ERR_WORKSPACE = -5,       /* workspace NULL or smaller than mhc_workspace_bytes() */
    MHC_ERR_CAPTURE = -6,         /* first call on a device made during stream capture */
    MHC_ERR_TIMEOUT = -7,         /* a bounded device wait gave up (see mhc_check_status) */
    MHC_ERR_CUDA = -8,            /* a CUDA runtime/driver call failed */
    MHC_ERR_ALIAS = -9,           /* an output overlaps an input (other than R' == R exactly) */
    MHC_ERR_CONFIG = -10          /* a config field is out of range */
} mhc_status;

/* Launch choices.  Zero in any field means "the policy decides". */
typedef struct {
    int path;            /* 0 auto: 2 from 1024 tokens; below that 3 when H >= 1024 and
                            fn_packed is given, else 1; 1 whenever the streaming path
                            cannot take H or block_m / cols_per_cta is set; 1 split path (H spread
                            over many small CTAs, CUDA-core projection, global split-K
                            with a last-arriving-CTA finish); 2 streaming path (TMA-staged
                            streams, tensor-core projection, split-K over a cluster of 4
                            CTAs: bandwidth-tuned); 3 streaming path over clusters of 16
                            CTAs (a quarter of the columns per CTA: latency-tuned for
                            small T; tcgen05 projection only) */
    int block_m;         /* tokens per CTA: path 1: 1, 2, 4, 8, 16 or 32; 0 = policy */
    int cols_per_cta;    /* path 1: columns of H per CTA, a multiple of 32; 0 = policy */
    int sinkhorn_iters;  /* Sinkhorn rounds; 0 = 20 */
    float amax_floor;    /* ue8m0 amax floor; 0 = 1e-10 */
    long long spin_limit;/* limit of every device-side wait, in units of about 100 ns; 0 = default
                            (10^7: about 1 s).  Split path: a wait past it gives up (status
                            bit 0).  Streaming paths: a wait past it is reported (status
                            bit 1) and goes on; a wait one second past it abandons the call
                            (the kernel stops issuing work, waits for its copies and MMAs in
                            flight, frees tensor memory and returns; the workspace's
                            counters may then be left set: run mhc_workspace_init() on it
                            before its next call).  Either way mhc_check_status() then
                            returns MHC_ERR_TIMEOUT */
    int projection;      /* streaming path's gate projection: 0 = policy (2 when H <= 5120, else 1);
                            1 = warp-level tensor-core MMA (m16n8k16) in the compute warps;
                            2 = tcgen05 MMA issued by one thread into tensor memory (H <= 5120) */
    int wave_split;      /* streaming paths: column parts per token block of the last, partial
                            round of blocks ("[FlyDSL] Single-launch Mega-mHC on gfx950", Kernel
                            Architecture: the split-K fallback at the wave edge).  When the
                            blocks left for that round are fewer than the clusters that fit,
                            each is cut into k column parts on k clusters, whose partial
                            sums meet in the workspace (cooperative launch: every cluster is
                            resident).  0 = the policy: no split (a part's fixed cost, measured
                            at about 24 chunk steps, exceeds what it saves at H = 5120), 1 = never
                            split, k >= 2 = at most k parts where they fit (H a multiple of 64 x
                            cluster size) */
} mhc_config;

/* Bytes of the per-stream workspace for a call of T tokens of width H with
 * `cfg` (NULL = defaults): a status word plus, on the split path, the
 * per-CTA partial sums and the arrival counters of every token group, and on
 * the streaming paths the partial sums and counters of the split last round
 * and the item scheduler's ticket counter (776 KiB + 128 bytes).  Where the
 * policy's path depends on whether fn_packed is given, the size covers both.
 * One workspace per stream whose calls can overlap on the GPU; it needs
 * mhc_workspace_init() once, after which the counters reset themselves and any
 * call (T' <= T, same H and cfg) may follow any other. */
size_t mhc_workspace_bytes(int64_t T, int H, const mhc_config* cfg);

/* The same for mhc_seam_unshifted() (the split path needs more shared memory
 * there, so a cfg may be refused by one and not the other). */
size_t mhc_workspace_bytes_unshifted(int64_t T, int H, const mhc_config* cfg);

/* Zero a workspace on `stream` (async).  Returns MHC_ERR_WORKSPACE when
 * `ws` is NULL or `bytes` is smaller than the status word. */
int mhc_workspace_init(void* ws, size_t bytes, void* stream);

/* Read and clear the device status word of `ws` (synchronises `stream`).
 * Returns MHC_OK, or MHC_ERR_TIMEOUT when a device wait of an earlier call on
 * this workspace ran past cfg->spin_limit (that call's outputs are then
 * unspecified). */
int mhc_check_status(void* ws, void* stream);

/* Bytes of the packed gate weight for width H: fn transposed to [48, 4H]
 * bf16, rows 0..23 the bf16 rounding ("hi") of fn[:, k], rows 24..47 the bf16
 * rounding of the remainder fn - hi ("lo").  hi + lo carries 16 significant
 * bits of each fp32 weight, enough for the 1e-3 gate tolerance.  The pages
 * pre-pack fn the same way ("fn pre-packed as bf16 hi/lo", Kernel
 * Architecture; "fn pre-pack cache", Files Changed). */
size_t mhc_packed_fn_bytes(int H);

/* Pack fn [4H, 24] fp32 (device) into fn_packed (device, 16-byte aligned,
 * mhc_packed_fn_bytes(H) bytes).  Call it once per weight update, before any
 * graph capture.  Returns MHC_ERR_NULL / MHC_ERR_SHAPE / MHC_ERR_ALIGN /
 * MHC_ERR_CUDA. */
int mhc_pack_fn(const float* fn, void* fn_packed, int H, void* stream);

/* One seam call.
 *   R           [T,4,H] bf16, 16-byte aligned
 *   Y           [T,H]   bf16, 16-byte aligned, or NULL (no_post form: R' = comb . R)
 *   post_prev   [T,4]   fp32, NULL exactly when Y is NULL
 *   comb_prev   [T,4,4] fp32, row i mixes into output stream i; NULL selects the
 *               identity form (then Y and post_prev must be NULL too, else
 *               MHC_ERR_INCOMPLETE_POST)
 *   pre_prev    [T,4]   fp32, the carried pre used for x
 *   fn          [4H,24] fp32, row i*H + h; 16-byte aligned
 *   fn_packed   mhc_pack_fn(fn) output, or NULL; required by paths 2 and 3
 *   bias [24], alpha [3] fp32;  gamma [H] bf16 (16-byte aligned)
 *   eps         added to both mean squares
 *   residual_out[T,4,H] bf16 (R'), 16-byte aligned; may be R itself (in place)
 *                but must not partly overlap any input; ignored (not written,
 *                may be NULL) in the identity form
 *   norm        [T,H] bf16, 16-byte aligned
 *   fp8_codes   [T,H] u8 e4m3fn, 16-byte aligned;  e8m0_scales [T,H/32] u8;
 *               both required for MHC_OUT_MXFP8, ignored otherwise;
 *               MHC_OUT_FP8_GRID writes the bf16 grid [T,H] through
 *               fp8_codes (2 bytes per element, 16-byte aligned) and
 *               ignores e8m0_scales
 *   pre_out, post_out [T,4], comb_out [T,4,4] fp32: the gates for the next seam
 *   workspace   from mhc_workspace_bytes()/mhc_workspace_init(), per stream
 *   cfg         NULL = all defaults
 * Every pointer except bias, alpha and e8m0_scales must be 16-byte aligned.
 * Outputs must not overlap inputs or each other.  The first call on a device
 * sets kernel attributes and must not be made during stream capture
 * (MHC_ERR_CAPTURE); later calls may be captured into a CUDA graph. */
int mhc_seam(const void* R, const void* Y, const float* post_prev, const float* comb_prev,
             const float* pre_prev, const float* fn, const void* fn_packed, const float* bias,
             const float* alpha, const void* gamma, float eps, int64_t T, int H,
             mhc_out_mode out_mode, void* residual_out, void* norm, uint8_t* fp8_codes,
             uint8_t* e8m0_scales, float* pre_out, float* post_out, float* comb_out,
             void* workspace, size_t ws_bytes, const mhc_config* cfg, void* stream);

/* The unshifted ordering of the seam ("[FlyDSL] Single-launch Mega-mHC on
 * gfx950", the table of seam implementations: the HIP mhc_fused_post_pre
 * kernel uses the unshifted ordering and has no RMSNorm).  The post-mix and the
 * gates are those of mhc_seam(); the layer input then uses the FRESH pre just
 * computed instead of a carried one, and is not normalised:
 *   x[t,h] = bf16( sum_i pre[t,i] R'[t,i,h] ),  pre = sigmoid(l[0:4]) of this call
 * Arguments as in mhc_seam(), without pre_prev, gamma, out_mode and the
 * quantised outputs:
 *   x_out      [T,H] bf16, 16-byte aligned (the layer input)
 *   pre_out    the fresh pre used for x; post_out and comb_out are the gates
 *              of the next seam's post-mix
 *   workspace  mhc_workspace_bytes_unshifted(T, H, cfg) bytes
 * comb_prev NULL (with Y and post_prev NULL) is the identity form.  The path
 * policy is mhc_seam()'s.  On the streaming paths (2, 3) the call is two
 * launches: the seam kernel writes R' and the gates, then a second kernel reads
 * R' back and forms x (8 H more bytes per token than the ordering needs).  On
 * the split path each CTA keeps its R' in shared memory and x is formed in the
 * same launch; a cfg->block_m * cfg->cols_per_cta whose R' tile (8 bytes per
 * element) does not fit is refused (MHC_ERR_CONFIG).  Errors as in
 * mhc_seam(). */
int mhc_seam_unshifted(const void* R, const void* Y, const float* post_prev, const float* comb_prev,
                       const float* fn, const void* fn_packed, const float* bias, const float* alpha, float eps,
                       int64_t T, int H, void* residual_out, void* x_out, float* pre_out, float* post_out,
                       float* comb_out, void* workspace, size_t ws_bytes, const mhc_config* cfg, void* stream);

/* Standalone per-32 ue8m0 quantiser of bf16 rows x [rows,H] (the same rule as
 * the seam's mxfp8 output; used to test the quantiser on crafted groups).
 * codes [rows,H] u8, scales [rows,H/32] u8.  H % 32 == 0; x and codes
 * 16-byte aligned.  amax_floor <= 0 means 1e-10. */
int mhc_quant_ue8m0(const void* x, int64_t rows, int H, float amax_floor, uint8_t* codes,
                    uint8_t* scales, void* stream);

/* Device-to-device copy of `bytes` bytes with this library's vectorised
 * streaming kernel (16-byte aligned pointers, bytes % 16 == 0).  It measures
 * the copy ceiling the seam is compared with (a copy whose read + write bytes
 * equal the seam's). */
int mhc_copy(const void* src, void* dst, size_t bytes, void* stream);

/* mhc_seam() on the split path (cfg->path 0 or 1; paths 2 and 3 are refused) for
 * callers that cannot allocate device memory: a plug-in inside a host program
 * that owns every device allocation, code running inside an allocator
 * callback, or a loop that must never block in the allocator.  The method's
 * pages describe no such entry point; it exists only for such callers.
 * Arguments are those of mhc_seam() without fn_packed, workspace and ws_bytes.
 * The scratch (partial sums, arrival counters, status word) lives in a fixed
 * 1 MiB static device array in the library, held by every GPU that loads it
 * until the process exits; a call whose mhc_workspace_bytes(T, H, cfg with
 * path 1) exceeds 1 MiB is refused with MHC_ERR_WORKSPACE (at H = 5120 and
 * the default policy: T above 480).  It calls no cudaMalloc/cudaFree or
 * allocating routine.  The first call on a device resolves the array's
 * address (cudaGetSymbolAddress) and should be made before any stream
 * capture.  Every call first clears the partial sums and arrival counters it
 * uses (cudaMemsetAsync on `stream`); all calls share the array, so calls that
 * can overlap on the GPU race on it and must be serialised by the caller.  The
 * array's status word is not cleared by a call: mhc_noalloc_check_status()
 * reports a bounded wait that ran out in any earlier call. */
int mhc_seam_noalloc(const void* R, const void* Y, const float* post_prev, const float* comb_prev,
                     const float* pre_prev, const float* fn, const float* bias, const float* alpha,
                     const void* gamma, float eps, int64_t T, int H, mhc_out_mode out_mode, void* residual_out,
                     void* norm, uint8_t* fp8_codes, uint8_t* e8m0_scales, float* pre_out, float* post_out,
                     float* comb_out, const mhc_config* cfg, void* stream);

/* mhc_check_status() for the static scratch of mhc_seam_noalloc() on the
 * current device: reads and clears its status word (synchronises `stream`).
 * Returns MHC_OK, or MHC_ERR_TIMEOUT when a bounded device wait of an earlier
 * mhc_seam_noalloc() call ran out (that call's outputs are unspecified).  Like
 * the entry point it serves, it has no counterpart in the method's pages and
 * allocates nothing. */
int mhc_noalloc_check_status(void* stream);

/* Number of kernel launches the last successful mhc_seam() on this host
 * thread issued (1 for every non-empty call). */
int mhc_last_launch_count(void);

/* Column parts per block of the partial last round in the last successful
 * mhc_seam() or mhc_seam_unshifted() on this host thread (cfg->wave_split):
 * 1 when that round was not split (or the call took the split path). */
int mhc_last_wave_parts(void);

/* Human-readable text of the last error on this host thread ("" if none). */
const char* mhc_last_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* MHC_SEAM_H */
