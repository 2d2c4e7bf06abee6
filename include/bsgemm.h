/*
 * bsgemm.h -- C ABI of the block-scaled GEMM + Amax library (libbsgemm.so).
 *
 * Operation ("GEMM + Amax (SM100)", section "Equations"):
 *
 *     Ahat[m,k,l] = dec(A[m,k,l]) * sf(SFA[m, k/sf_vec_size, l])
 *     Bhat[n,k,l] = dec(B[n,k,l]) * sf(SFB[n, k/sf_vec_size, l])
 *     C[m,n,l]    = sum_k Ahat[m,k,l] * Bhat[n,k,l]      (fp32 accumulation)
 *     Amax        = max_{m,n,l} |C[m,n,l]|               (of the stored C)
 *
 * sf(byte) is 2^(byte - 127) for E8M0 scale bytes and the float8_e4m3fn
 * value of the byte for E4M3 scales (the NVFP4 form, "Dtypes").  E4M3 scale
 * bytes must have the sign bit clear (the tensor cores read them as
 * unsigned E4M3); a byte with it set gives unspecified results.
 *
 * C is stored rounded to its type, to nearest with ties to even.  For the
 * low-precision C types (E4M3, E5M2, packed E2M1; "Support surface and
 * constraints", "Dtypes") the rounding saturates to the largest finite
 * value, a NaN stays NaN in FP8 and becomes +0 in E2M1 (which has no NaN),
 * and Amax is the largest stored magnitude decoded back to fp32.
 *
 * Tensors ("Parameters", "Input/Output tensors"; all device memory of one
 * GPU, "Environment": all tensors on the same device):
 *
 *   A    (M, K, L), k-major: strides (K, 1, M*K) in elements.  FP8 codes one
 *        per byte; packed FP4 (E2M1) two per byte, element 2i in the low
 *        nibble, so a row holds K/2 bytes ("Layouts and strides").  FP8 A
 *        may instead be m-major: strides (1, M, M*K) ("Parameters").
 *   B    (N, K, L), k-major (or, FP8, n-major), same element rules as A.
 *   SFA  E8M0 (or E4M3) bytes, physical C-contiguous (L, ceil(M/128),
 *        ceil(K/(4*sfv)), 32, 4, 4), which is the page's logical (32, 4, ceil(M/128), 4,
 *        ceil(K/(4*sfv)), L) view permuted ("Using JAX arrays").  Row
 *        m = 128*mt + 32*m1 + m0 and K-block kb = 4*kt + kin sit at byte
 *        ((l*T_m + mt)*T_k + kt)*512 + m0*16 + m1*4 + kin.
 *   SFB  the same for the N rows of B.
 *   C    (M, N, L), fp32 / fp16 / bf16 / E4M3 / E5M2, n-major strides
 *        (N, 1, M*N) or m-major strides (1, M, M*N); packed E2M1 only
 *        n-major, two per byte (element 2i of a row in the low nibble).
 *   Amax one fp32 (shape (1,1,1)); overwritten by every run, not accumulated.
 *
 * Padding entries of SFA/SFB (rows past M or N, K-blocks past
 * ceil(K/sfv)) multiply zero codes or rows that are never stored; they must
 * hold a finite scale (any byte but 0xFF for E8M0; any byte but 0x7F and
 * 0xFF for E4M3) so that 0 * scale stays 0.
 *
 * Support ("Support surface and constraints"): A/B k-major, or m-major A /
 * n-major B for FP8 (M, N a multiple of 16; an n-major B runs on CTA pairs
 * or 128-wide tiles, not on one 256-wide CTA); A/B both FP8
 * (E4M3/E5M2, each on its own) with sf_vec_size 32 and E8M0 scales, or both
 * E2M1 with sf_vec_size 32 and E8M0 scales or sf_vec_size 16 and E8M0 or
 * E4M3 scales; C fp32/fp16/bf16 always, E4M3/E5M2/E2M1 with E2M1 operands
 * only.  Rows of A, B and C must be 16-byte aligned along their contiguous
 * dimension (K bytes of a k-major operand, M or N bytes of an MN-major one,
 * an E2M1 C row of N/2 bytes with N even), every pointer 16-byte aligned.
 * M, N, K and L are at least 1 (an empty problem is BSG_ERR_INVALID_ARG)
 * and below 2^31.  Everything else returns BSG_ERR_UNSUPPORTED or
 * BSG_ERR_INVALID_ARG before any launch (errors are reported before launch,
 * as "Grouped GEMM (SM100 BF16)", "Scheduling, caching, and errors", does).
 *
 * Ownership: the caller owns every device buffer (A, B, SFA, SFB, C, Amax,
 * workspace).  A plan owns host memory only.  No entry point allocates
 * device memory.  bsg_run is asynchronous on the given stream and never
 * synchronises.  No exception or abort crosses this boundary.
 */
#ifndef BSGEMM_H
#define BSGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSG_OK = 0,
    BSG_ERR_INVALID_ARG = 1,    /* null pointer, non-positive size, bad enum, bad hint */
    BSG_ERR_UNSUPPORTED = 2,    /* a combination outside the support surface */
    BSG_ERR_ALIGNMENT = 3,      /* a pointer or a contiguous row not 16-byte aligned */
    BSG_ERR_ARCH = 4,           /* device is not compute capability 10.3 (sm_103a) */
    BSG_ERR_WORKSPACE = 5,      /* workspace missing or smaller than required */
    BSG_ERR_CUDA = 6,           /* a CUDA runtime/driver call failed */
    BSG_ERR_DEVICE_TIMEOUT = 7  /* a pipeline wait in the kernel ran out of time */
} bsg_status;

typedef enum {
    BSG_E4M3 = 0,   /* float8_e4m3fn codes (A/B/C) or scale bytes (SFA/SFB) */
    BSG_E5M2 = 1,   /* float8_e5m2 codes (A/B/C) */
    BSG_E2M1 = 2,   /* float4_e2m1fn, packed two per byte (A/B/C) */
    BSG_UE8M0 = 3,  /* float8_e8m0fnu scale bytes (SFA/SFB) */
    BSG_F32 = 4,    /* C */
    BSG_F16 = 5,    /* C */
    BSG_BF16 = 6    /* C */
} bsg_dtype;

/* Problem statement, after the page's constructor arguments ("Common
 * parameters", "Class-specific parameters": mma_tiler_mn, cluster_shape_mn).
 * tile_* and cluster_* are hints only: 0 lets the library choose; otherwise
 * tile_m must be 128, tile_n 128, 224 or 256 (224: FP8 operands and M > 128
 * only, else BSG_ERR_UNSUPPORTED), cluster_m 1 or 2 (2 is a pair of CTAs
 * running 256-row MMAs, the default for tile_n 224 and 256) and cluster_n 1.
 * cluster_m 4 and cluster_n 2 or 4 (shapes whose CTAs would share a tile by
 * multicast) are accepted values that this library does not build:
 * BSG_ERR_UNSUPPORTED; any other value is BSG_ERR_INVALID_ARG. */
typedef struct {
    int64_t M, N, K, L;
    int32_t a_dtype, b_dtype;   /* bsg_dtype */
    int32_t sf_dtype;           /* BSG_UE8M0, or BSG_E4M3 (E2M1 A/B, sfv 16) */
    int32_t c_dtype;            /* BSG_F32, BSG_F16, BSG_BF16, BSG_E4M3, BSG_E5M2, BSG_E2M1 */
    char a_major, b_major;      /* 'k'; or 'm' (A) / 'n' (B) for FP8 operands */
    char c_major;               /* 'n' or 'm' */
    char reserved0;
    int32_t sf_vec_size;        /* 16 or 32 */
    int32_t tile_m, tile_n;
    int32_t cluster_m, cluster_n;
} bsg_problem;

typedef struct bsg_plan bsg_plan;

/* What a plan chose (for logging and the benchmark). */
typedef struct {
    int32_t tile_m, tile_n, tile_k_bytes;  /* CTA tile; K bytes per pipeline stage */
    int32_t stages;                        /* shared-memory pipeline depth */
    int32_t grid;                          /* persistent CTAs per launch */
    int32_t threads;                       /* threads per CTA */
    int32_t smem_bytes;                    /* dynamic shared memory per CTA */
    int32_t num_tiles;                     /* output tiles per launch */
    int32_t mma_kind;                      /* 0 mxf8f6f4 1X, 1 mxf4nvf4 4X, 2 mxf4nvf4 2X */
    int32_t cluster_m;                     /* 1: CTAs alone; 2: cta_group::2 pairs */
    char kernel_name[64];
    int32_t half_tiles;                    /* tiles of the last wave run as two 256 x 128
                                              half-width units (0: none), when the
                                              K halves below are not run */
    int32_t k_split_tiles;                 /* tiles past the whole waves run as two K
                                              halves at full width, with the plan's full
                                              workspace (0: none) */
} bsg_plan_info;

/* Host-only validation of a problem against the support surface; touches
 * no device.  Returns BSG_OK or the first violated rule. */
bsg_status bsg_problem_check(const bsg_problem *problem);

/* Validate, pick the kernel, tile and pipeline for `device`, and record
 * them in a new plan (the analogue of check_support() + compile() of the
 * page's class API, "Class API").  Fails with BSG_ERR_ARCH unless the device
 * is sm_103.  *out is set only on BSG_OK. */
bsg_status bsg_plan_create(const bsg_problem *problem, int device, bsg_plan **out);

/* Bytes of device workspace for the plan's fastest form.  256 bytes hold
 * a cross-CTA amax slot, an arrival counter and an error word; a plan that
 * runs its leftover tiles as two K halves (bsg_plan_info.k_split_tiles > 0:
 * FP8 256-wide pairs with at least two whole waves of tiles and at least 40
 * K stages of 128 bytes; the environment variable BSG_KSPLIT_MIN_STAGES,
 * read by bsg_plan_create, moves that threshold) adds two words per split
 * tile and CTA and, per split tile, four 128 x 256 fp32
 * partial sums (512 KiB).  bsg_run accepts any workspace of at least 256
 * bytes and runs the K halves only when it is at least this size; a smaller
 * one runs the half-width split of the last wave instead (same inputs, C
 * within the same tolerance, not bit-identical).
 * The workspace lives in the caller's allocator, as the workspaces of
 * "Grouped GEMM (SM100 BF16)", section "Using JAX arrays", do. */
bsg_status bsg_plan_workspace_size(const bsg_plan *plan, size_t *bytes);

/* Zero a workspace on `stream` (cudaMemsetAsync).  Must be called once
 * before a workspace is first used, with the size later runs pass; every
 * run leaves it zeroed again, an abandoned one too, but for the error word
 * that bsg_check_device_status reads and clears (caller-allocator
 * workspaces: "Grouped GEMM (SM100 BF16)", "Using JAX arrays"). */
bsg_status bsg_workspace_init(const bsg_plan *plan, void *workspace, size_t ws_bytes,
                              void *stream);

/* One launch of the GEMM + Amax on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) -- the analogue of execute() ("Class API").
 * A, B, SFA, SFB, C, amax and workspace are device pointers of the plan's
 * device, which must be the calling thread's current device
 * (BSG_ERR_INVALID_ARG otherwise).  Checks pointers, alignment and the
 * workspace size, then launches exactly one kernel.  Allocates nothing, never
 * synchronises.  Runs sharing one workspace must not overlap on the device. */
bsg_status bsg_run(const bsg_plan *plan, const void *A, const void *B, const void *SFA,
                   const void *SFB, void *C, float *amax, void *workspace, size_t ws_bytes,
                   void *stream);

/* bsg_run without a caller workspace, for callers that cannot allocate
 * device memory (no allocator to draw from, or code running where
 * cudaMalloc is not permitted).  The pages have no counterpart: it is a
 * convenience of this library.  The workspace comes from a fixed array
 * inside the library (4096 bytes on every GPU that loads it, kept until the
 * process exits; zero when the library is loaded); a plan whose fastest form
 * needs more runs the form a small workspace gets (see
 * bsg_plan_workspace_size).  The arguments are checked first, exactly as
 * bsg_run checks them, so a bad pointer or the wrong current device returns
 * its status before anything is enqueued.  The first call on a device then
 * looks up the array's device address (cudaGetSymbolAddress, host side
 * only), so make that first call before any stream capture.  Each call
 * clears the array's first 16 bytes with cudaMemsetAsync on `stream`, then
 * launches exactly as bsg_run.  All
 * calls share the one array: calls that overlap on the device race and
 * give wrong results.  A device-side wait timeout is not reported here (use
 * bsg_run with a workspace and bsg_check_device_status for that).  Nothing
 * is allocated. */
bsg_status bsg_run_noalloc(const bsg_plan *plan, const void *A, const void *B, const void *SFA,
                           const void *SFB, void *C, float *amax, void *stream);

/* Device buffers for bsg_run_host: caller-allocated, sized for the plan. */
typedef struct {
    void *A, *B, *SFA, *SFB, *C;
    float *amax;
    void *workspace;
    size_t ws_bytes;
} bsg_device_buffers;

/* End-to-end form of bsg_run over HOST buffers (preferably pinned).  The
 * pages have no counterpart; it is this library's own, the form the
 * end-to-end measurement uses.  It copies
 * hA, hB, hSFA, hSFB to the device buffers, runs, and copies C and Amax back
 * to hC and h_amax, all enqueued on `stream` (one cudaMemcpyAsync per
 * tensor).  Asynchronous like bsg_run: synchronise the stream before reading
 * hC or *h_amax. */
bsg_status bsg_run_host(const bsg_plan *plan, const void *hA, const void *hB, const void *hSFA,
                        const void *hSFB, void *hC, float *h_amax,
                        const bsg_device_buffers *dev, void *stream);

/* Synchronise `stream`, then read and clear the workspace's device error
 * word (the read and the clear are enqueued on `stream` and waited for, so
 * the clear is ordered before later launches on it).  Returns
 * BSG_ERR_DEVICE_TIMEOUT if a kernel of an earlier run gave
 * up on a pipeline wait (its outputs are then invalid), else BSG_OK.  The
 * pages have no counterpart: the bounded waits and their error word are
 * this library's own. */
bsg_status bsg_check_device_status(const bsg_plan *plan, void *workspace, void *stream);

/* Fill *info with the plan's choices (this library's own; no page
 * counterpart). */
bsg_status bsg_plan_describe(const bsg_plan *plan, bsg_plan_info *info);

/* Free a plan (host memory only).  NULL is ignored.  The class API's
 * object lifetime ("Class API") in C form. */
void bsg_plan_destroy(bsg_plan *plan);

/* Static text for a status code (this library's own). */
const char *bsg_status_string(bsg_status status);

#ifdef __cplusplus
}
#endif

#endif /* BSGEMM_H */
