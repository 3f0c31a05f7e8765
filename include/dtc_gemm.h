/*
 * dtc_gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * The operation (all entry points):  C[M,N] = A[M,K] . Bop[K,N], accumulated in fp32 in Tensor
 * Memory and rounded once to the output format (round to nearest even).
 *   - "NT": B is stored row-major [N,K] and Bop = B^T. This is the product of TileLang SM100
 *     Support (Preview), "Code Example" (A is (M, K), B is (N, K), the gemm uses trans_B=True,
 *     accumulator T.alloc_tmem(..., "float")) and "Compilation and Usage"
 *     (ref_c = (a.float() @ b.T.float()).to(torch.bfloat16)).
 *   - "NN": B is stored row-major [K,N] and Bop = B. This is the product of tilelang (velog),
 *     section 1.1 Front-End DSL (A is (M, K), B is (K, N), accum_dtype "float").
 *   - "TN", "TT": as "NN", "NT" with A stored row-major [K,M] (Aop = A^T). The first letter is
 *     A's transpose flag, the second B's: the trans_A / trans_B arguments of T.gemm in TileLang
 *     SM100 Support (Preview), "Current Limitations" and "Code Example". 16-bit products only.
 *   In NT and NN, A is row-major [M,K]. C is always row-major [M,N]. With the plain entry points
 *   every row is dense (row stride = number of columns), as the generated host code of tilelang
 *   (velog) section 1.3 also assumes; gemm_ex takes leading dimensions (lda, ldb, ldc in
 *   gemm_options) for operands and results that are rows of larger row-major arrays.
 *
 * Pointers: A, B, C (and sfA, sfB, and a stream-K workspace) are DEVICE pointers of the current
 * CUDA device (or managed memory), owned by the caller; the library keeps no reference after the
 * call returns. A pointer into host memory or into another GPU's memory is refused with
 * GEMM_ERR_INVALID_ARG before anything is launched. C must not overlap A, B or the scales. All
 * pointers must be 16-byte aligned (the tensor-memory-access unit's global address rule), and
 * every row must start on a 16-byte boundary (see each function).
 *
 * Asynchrony: every GEMM call only enqueues work on `stream` (0 = the legacy default stream) and
 * returns; the status it returns covers argument checks and the launch. A device-side wait that
 * gave up (see GEMM_ERR_TIMEOUT) is reported by gemm_stream_status().
 *
 * Errors: a non-zero status leaves a one-line message for the calling thread in
 * gemm_last_error(). No call ever aborts the process or traps on the device.
 *
 * Degenerate sizes: M == 0 or N == 0 does nothing and returns GEMM_OK. K == 0 writes C = +0 (the
 * empty sum) with an asynchronous memset on `stream`.
 */
#ifndef DTC_GEMM_H
#define DTC_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA's stream handle, without including the CUDA headers. */
typedef struct CUstream_st* dtc_stream_t;

typedef enum {
    GEMM_LAYOUT_NT = 0, /* A is [M,K], B is [N,K] row-major: C = A . B^T   */
    GEMM_LAYOUT_NN = 1, /* A is [M,K], B is [K,N] row-major: C = A . B     */
    GEMM_LAYOUT_TN = 2, /* A is [K,M], B is [K,N] row-major: C = A^T . B   */
    GEMM_LAYOUT_TT = 3  /* A is [K,M], B is [N,K] row-major: C = A^T . B^T */
} gemm_layout;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* rejected before any launch: see the rules per function (all but
                                 the device-memory check need no CUDA call) */
    GEMM_ERR_UNSUPPORTED = 2, /* the current device is not an sm_103 GPU, or a variant that the
                                 requested shape or layout does not allow was forced */
    GEMM_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed; the message names it */
    GEMM_ERR_TIMEOUT = 4      /* a device-side wait gave up (reported by gemm_stream_status) */
} gemm_status;

/* Kernel variants (gemm_options.variant). AUTO picks per shape. */
typedef enum {
    GEMM_VARIANT_AUTO = 0,
    GEMM_VARIANT_1CTA = 1,   /* persistent 128 x 256 or 128 x 224 tiles, one CTA per tile */
    GEMM_VARIANT_2CTA = 2,   /* persistent 256 x 256 or 256 x 224 tiles on a CTA pair
                                (cluster 2x1, tcgen05 cta_group::2); for the block-scaled
                                product 256 x 224 tiles with 256-deep stages, for 128-element
                                scale blocks, K % 128 == 0 and a workspace that receives the
                                repacked scales (see gemm_workspace_size) */
    GEMM_VARIANT_SPLITK = 3  /* 128 x 128 tiles with K split over a cluster of 2 or 4 CTAs, or
                                128 x 256 tiles split over 2; each CTA copies the partial sums
                                of the rows another CTA owns into that CTA's shared memory, and
                                the owner reduces and stores them (few-tile products, such as
                                the skinny memory-bound M = 128 case); or, unsplit, one CTA per
                                128 x 64 tile with the whole K (few tiles with a short K) */
} gemm_variant;

typedef struct {
    int variant;          /* a gemm_variant; GEMM_VARIANT_AUTO (0) chooses per shape */
    int split_k;          /* SPLITK only: number of K-slices (2 or 4), or 1: one CTA per
                             128 x 64 tile with the whole K (no exchange; K % 64 == 0); 0 =
                             choose */
    uint64_t timeout_ns;  /* limit of every device-side wait; 0 = the default (2 s) */
    int fault_inject;     /* test hook, 0 in normal use. 1 = the load producer skips its first
                             stage, so the consumer's bounded wait runs out and the call reports
                             GEMM_ERR_TIMEOUT through gemm_stream_status. */
    int tile_n;           /* force the N-tile: 256, 224 (not SPLITK; one-CTA tiles need B stored
                             [N,K]; block-scaled: 224 only), 128 (SPLITK and 2CTA) or 64 (2CTA);
                             0 = choose. 2CTA tiles of 128 or 64 take 128-deep stages
                             (K % 64 == 0) */
    int tile_k;           /* K-elements per pipeline stage: 64 (1CTA), 64 or 128 (2CTA; SPLITK
                             with 128-wide tiles; 128 needs K % 64 == 0); block-scaled: 128 (the
                             one-CTA kernel) or 256 (the pair kernel); 0 = choose */
    int64_t lda;          /* elements between consecutive stored rows of A, B, C; 0 = dense (the */
    int64_t ldb;          /* row length: K or M for A, K or N for B, N for C). At least the row */
    int64_t ldc;          /* length, and rows must start 16 bytes apart (ld x element size %
                             16 == 0). Only the M x N region of C is written. */
    int mx_a_format;      /* block-scaled product only: element format of A: 0 = e4m3 (OCP FP8 */
    int mx_b_format;      /* E4M3, the default), 1 = e5m2 (OCP FP8 E5M2), 2 = e2m3 and 3 = e3m2
                             (OCP MX FP6), 4 = e2m1 (OCP MX FP4); likewise B. FP6 and FP4 rows
                             are packed: element k of a row is the 6- or 4-bit field at bit 6k or
                             4k of the row read as a little-endian bit stream (fp4: byte k/2, low
                             nibble for even k; fp6: 4 elements in 3 bytes). With an FP6 or FP4
                             operand K % 128 == 0, and that operand's base is 32-byte aligned
                             and its rows start a multiple of 32 bytes apart. */
    int mx_scale_block;   /* block-scaled product only: K-elements per E8M0 scale, 128 (0 = the
                             default, the pages' granularity) or 32 (the OCP MX block); the
                             scale arrays are then [rows, ceil(K / block)]. 32-element blocks run
                             on the one-CTA kernel. */
    void* workspace;      /* device scratch owned by the caller, 16-byte aligned; NULL = none
                             (see gemm_workspace_size). 16-bit products: stream-K; its first 1 KB
                             holds flags that must be zero before the first call that uses it;
                             every completed call leaves them zero again (after a
                             GEMM_ERR_TIMEOUT, zero them before reuse). Block-scaled product: a
                             large enough workspace receives the scale arrays repacked by a first
                             kernel of the call, from which the product kernel copies them into
                             Tensor Memory (see gemm_workspace_size for when); no initial contents
                             needed. Calls that may run at the same time (other streams) must not
                             share a workspace. */
    uint64_t workspace_bytes;
    int stream_k;         /* 0 = use stream-K when a large enough workspace is given and the
                             cost model prefers it; 1 = required (error if not possible); 2 = off.
                             Stream-K runs the pair kernel on 256 x 256 tiles with 128-deep
                             stages, or 64-deep ones when tile_k = 64. */
} gemm_options;

/*
 * bf16 operands, fp32 accumulation, bf16 output.
 *   A: [M,K] bf16 (NT, NN) or [K,M] (TN, TT). B: [N,K] bf16 (NT, TT) or [K,N] (NN, TN).
 *   C: [M,N] bf16.
 *   INVALID_ARG when: M, N or K is negative or above 2^31-1; layout is not NT, NN, TN or TT; a
 *   pointer needed for the sizes is NULL or not 16-byte aligned; a stored row is not a multiple
 *   of 16 bytes (its length % 8 != 0: K or M for A, K or N for B, N for C).
 * (TileLang SM100 Support (Preview), "Code Example" / "Compilation and Usage".)
 */
int gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int layout,
              dtc_stream_t stream);

/*
 * fp16 operands, fp32 accumulation, fp16 output (IEEE round to nearest even; overflow gives
 * +-inf). Same layouts and argument rules as gemm_bf16.
 * (tilelang (velog), section 1.1 Front-End DSL: dtype "float16", accum_dtype "float"; section 1.3
 * Generated Kernel Source: the fp32 accumulator is cast to half on output.)
 */
int gemm_f16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int layout,
             dtc_stream_t stream);

/*
 * MXFP8 block-scaled GEMM, NT only:
 *   C[m,n] = bf16( sum_k e4m3(A[m,k]) 2^(sfA[m,k/128]-127) * e4m3(B[n,k]) 2^(sfB[n,k/128]-127) )
 *   A: [M,K] e4m3 (OCP "fn" encoding). B: [N,K] e4m3. sfA: [M, ceil(K/128)] E8M0 bytes.
 *   sfB: [N, ceil(K/128)] E8M0 bytes. C: [M,N] bf16. One scale per row per 128 K-elements for
 *   both operands (05 Blackwell TCGEN05 GEMM tutorial, "Advanced": gemm_blockscaled with
 *   sf_a_granularity_k = sf_b_granularity_k = 128, the "1d1d" example).
 *   INVALID_ARG as for gemm_bf16, with K % 16 != 0 for the e4m3 rows; the scale arrays have no
 *   alignment rule.
 */
int gemm_mxfp8(const void* A, const void* B, const void* sfA, const void* sfB, void* C,
               int64_t M, int64_t N, int64_t K, dtc_stream_t stream);

/*
 * The same three operations with options (variant choice, leading dimensions, block-scaled
 * element formats and scale block, wait limit, test hook). dtype: 0 = bf16, 1 = fp16, 2 = mxfp8 (sfA/sfB are ignored for 0 and 1; layout must be
 * NT for 2; the scale arrays stay dense). opts may be NULL (all defaults). INVALID_ARG also when
 * a leading dimension is negative, below its row length, above 2^31-1 or not a multiple of 16
 * bytes.
 * (The products of gemm_bf16, gemm_f16 and gemm_mxfp8 with the options of the pages' GEMM call:
 * T.gemm's trans_A / trans_B in TileLang SM100 Support (Preview), "Code Example", and the block-
 * scaled variants of the 05 Blackwell TCGEN05 GEMM tutorial, "Advanced".)
 */
int gemm_ex(int dtype, const void* A, const void* B, const void* sfA, const void* sfB, void* C,
            int64_t M, int64_t N, int64_t K, int layout, const gemm_options* opts,
            dtc_stream_t stream);

/* What a call with these sizes and options would launch (gemm_plan, gemm_plan_model). */
typedef struct {
    int variant;  /* GEMM_VARIANT_1CTA, _2CTA or _SPLITK (never AUTO) */
    int tile_m;   /* rows of C per tile (per CTA pair for 2CTA) */
    int tile_n;   /* columns of C per tile */
    int tile_k;   /* K-elements per pipeline stage */
    int stages;   /* depth of the shared-memory ring */
    int split_k;  /* K-slices (1 unless SPLITK) */
    int ctas;     /* CTAs launched (persistent grid) */
    int tiles;    /* output tiles (times split_k work units for SPLITK) */
    int cluster;  /* CTAs per cluster */
    int sk_tiles; /* tiles shared out by stream-K (0 = none) */
    int sf_packed; /* block-scaled product: 1 = the scales are repacked into the workspace and
                      copied into Tensor Memory by the MMA thread (the pair kernel always; the
                      one-CTA kernel for 32-element blocks given a workspace; see
                      gemm_options.workspace); 0 = gathered by the one-CTA kernel's scale warps */
} gemm_plan_info;

/* Fills *info with the launch that gemm_ex would make for these sizes and options on the current
 * device. Returns GEMM_OK, or the status the call would fail with (sizes/layout/dtype only;
 * pointers are not part of the plan). Makes no CUDA call except device queries (the first call on
 * a device asks how many clusters of the pair and split-K kernels can be resident at once). The
 * pages have no counterpart: their kernels have one fixed tile. */
int gemm_plan(int dtype, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* opts,
              gemm_plan_info* info);

/* What the planner knows about a device. The pair kernel's stream-K mode makes pairs wait for
 * pieces other pairs compute, so it counts only on pairs that can be resident at once. */
typedef struct {
    int sm_count;         /* streaming multiprocessors (152 on GB300) */
    int pair_clusters;    /* clusters of 2 CTAs of the pair kernel resident at once (0 = half
                             the SMs) */
    int split2_clusters;  /* clusters of 2 CTAs of the split-K kernel resident at once (0 = half
                             the SMs) */
    int split4_clusters;  /* clusters of 4 CTAs of the split-K kernel resident at once (0 = a
                             quarter of the SMs) */
} gemm_device_model;

/* The current device's model (the first call asks the CUDA occupancy API). INVALID_ARG if out is
 * NULL. The pages have no counterpart. */
int gemm_device_model_query(gemm_device_model* out);

/* gemm_plan for a described device instead of the current one: a pure function of its arguments
 * (no CUDA call, so it also runs on a machine without a GPU). INVALID_ARG if model or info is
 * NULL, sm_count < 1 or a cluster count is negative; otherwise as gemm_plan. The pages have no
 * counterpart. */
int gemm_plan_model(const gemm_device_model* model, int dtype, int64_t M, int64_t N, int64_t K,
                    int layout, const gemm_options* opts, gemm_plan_info* info);

/*
 * gemm_ex, with the library's own workspace instead of a caller's: a 20 MiB region of module
 * memory (a file-scope device array, zero when the library is loaded), so this call allocates
 * nothing, on the host or the device. The pages have no counterpart.
 *   - opts->workspace must be NULL (INVALID_ARG otherwise); the other options are gemm_ex's.
 *   - The region serves as the stream-K workspace of the 16-bit products and as the home of the
 *     repacked scales of the block-scaled product (see gemm_options.workspace).
 *   - 20 MiB holds the stream-K workspace of up to 79 resident CTA pairs (devices of up to 158
 *     SMs). A plan that would need more runs without stream-K, or fails with INVALID_ARG when
 *     opts->stream_k = 1 (required); block-scaled scales that do not fit stay with the scale
 *     warps.
 *   - The first call on a device looks up the region's address with cudaGetSymbolAddress, a
 *     synchronous call.
 *   - The region's first 1 KB (flags) must be zero when a stream-K launch starts: a call whose
 *     plan uses stream-K clears it with cudaMemsetAsync on `stream` just before its launch (so a
 *     call after a GEMM_ERR_TIMEOUT starts clean); a call rejected by its argument checks
 *     enqueues nothing, one that takes whole tiles only its kernels.
 *   - There is one region per device: calls that may overlap (on different streams, or from
 *     different threads) race on it and may return wrong results. Serialise them.
 */
int gemm_ex_static_workspace(int dtype, const void* A, const void* B, const void* sfA,
                             const void* sfB, void* C, int64_t M, int64_t N, int64_t K,
                             int layout, const gemm_options* opts, dtc_stream_t stream);

/*
 * 2:4 structured-sparse A (the sparse GEMM, gemm_sp, that 05 Blackwell TCGEN05 GEMM tutorial, "An
 * API-level note", names among the exported forms; read as the 2:4 pattern along K):
 *   C[m,n] = round_out( sum_g sum_{j<2} vals[m,2g+j] * Bop[4g + pos_j(m,g), n] )
 * Each group g of 4 consecutive K-elements of a row of A keeps two values, stored in order in vals
 * [M, K/2] (bf16 for dtype 0, fp16 for 1), at two positions 0..3 given by meta [M, K/8] bytes:
 * group g's nibble is at bits 4*(g % 2) of byte g/2 of the row, its bits 0-1 the position of
 * vals[m, 2g] and bits 2-3 that of vals[m, 2g+1]. The two positions of a group must differ (the
 * 2:4 pattern); where they are equal the element is the two values' sum rounded to the element
 * type. B and C as for gemm_bf16 / gemm_f16 with layout NT or NN; opts as gemm_ex's (lda must be
 * 0; ldb, ldc, the variant and a stream-K workspace apply to the product).
 * The call expands A into `workspace` (device memory of the current device, 16-byte aligned, at
 * least gemm_sp_workspace_size bytes: M x K 16-bit elements, owned by the caller) with an
 * HBM-bound kernel, then runs the dense product on it; both are enqueued on `stream`.
 * INVALID_ARG also when K % 16 != 0, vals is NULL or not 16-byte aligned, meta is NULL, or the
 * workspace is missing or too small.
 */
int gemm_sp(int dtype, const void* vals, const void* meta, const void* B, void* C, int64_t M,
            int64_t N, int64_t K, int layout, const gemm_options* opts, void* workspace,
            uint64_t workspace_bytes, dtc_stream_t stream);

/* Bytes of workspace gemm_sp needs (M x K x 2). INVALID_ARG for a dtype other than 0 or 1, sizes
 * outside [0, 2^31-1] or a NULL bytes. (05 Blackwell TCGEN05 GEMM tutorial, "An API-level note":
 * gemm_sp.) */
int gemm_sp_workspace_size(int dtype, int64_t M, int64_t K, uint64_t* bytes);

/*
 * NVFP4 block-scaled GEMM, NT only (the NVFP4 member of the "other block-scaled formats" of the
 * 05 Blackwell TCGEN05 GEMM tutorial, "Advanced": gemm_blockscaled):
 *   C[m,n] = bf16( sum_k e2m1(A[m,k]) ue4m3(sfA[m,k/16]) * e2m1(B[n,k]) ue4m3(sfB[n,k/16]) )
 *   A: [M, K/2] bytes, B: [N, K/2] bytes: packed e2m1 (OCP MX FP4) codes, element k of a row in
 *   the low nibble of byte k/2 for even k, the high nibble for odd k. sfA: [M, K/16], sfB:
 *   [N, K/16] UE4M3 scale bytes (e4m3 codes with the sign bit clear; a code with the sign bit
 *   set, or the e4m3 NaN code, scales to NaN). C: [M,N] bf16.
 * The call writes A and B multiplied by their scales into `workspace` as bf16 (exact: at most 5
 * significant bits per product) with an HBM-bound kernel, then runs the bf16 product of the two on
 * the tensor cores; both are enqueued on `stream`. `workspace` is device memory of the current
 * device, 16-byte aligned, of at least gemm_nvfp4_workspace_size bytes, owned by the caller; its
 * contents need no initial value and are overwritten. opts may be NULL; the variant, tile, ldc,
 * wait limit and stream-K options (with opts->workspace as the stream-K workspace) apply to the
 * product; lda, ldb, mx_a_format, mx_b_format and mx_scale_block must be 0.
 * INVALID_ARG as for gemm_bf16, and also when K % 16 != 0, A or B is NULL or not 16-byte aligned,
 * sfA or sfB is NULL, or the workspace is NULL, misaligned or too small (the checks on A, B, the
 * scales and the workspace apply when M, N and K are all non-zero).
 */
int gemm_nvfp4(const void* A, const void* B, const void* sfA, const void* sfB, void* C,
               int64_t M, int64_t N, int64_t K, const gemm_options* opts, void* workspace,
               uint64_t workspace_bytes, dtc_stream_t stream);

/* Bytes of workspace gemm_nvfp4 needs: the expanded A (M x K bf16), padded to 256 bytes, then the
 * expanded B (N x K bf16). INVALID_ARG for sizes outside [0, 2^31-1] or a NULL bytes. (05 Blackwell
 * TCGEN05 GEMM tutorial, "Advanced": gemm_blockscaled.) */
int gemm_nvfp4_workspace_size(int64_t M, int64_t N, int64_t K, uint64_t* bytes);

/*
 * Bytes of workspace (gemm_options.workspace) with which the call would use stream-K on CTA pairs
 * (the last, part-full wave's tiles shared out over all pairs as equal runs of K-blocks, the
 * pieces summed through the workspace); 0 when it would not (or stream_k == 2). For the
 * block-scaled product (dtype 2): the bytes of the repacked scale arrays (about the size of sfA
 * and sfB together) when the call would use them -- AUTO with 128-element blocks, K % 128 == 0
 * and at least a wave of 256 x 224 tiles, or the pair kernel forced (the pair kernel with
 * 256-deep stages), and 32-element blocks (the one-CTA kernel) -- else 0; UNSUPPORTED when the
 * pair kernel is forced for a call it does not take. The pages have no counterpart:
 * their persistent 2-CTA variant (05 Blackwell TCGEN05 GEMM tutorial, "Advanced") takes whole
 * tiles. INVALID_ARG as gemm_ex; bytes must not be NULL.
 */
int gemm_workspace_size(int dtype, int64_t M, int64_t N, int64_t K, int layout,
                        const gemm_options* opts, uint64_t* bytes);

/* Message for the calling thread's most recent non-OK return ("" if none). Valid until that
 * thread's next call into the library. The convention of the generated host code of tilelang
 * (velog) section 1.3 (Generated Kernel Source, the host call()): every call returns an int status
 * and the text of the last error is kept in a buffer the caller reads afterwards (there one static
 * buffer, here one per thread). */
const char* gemm_last_error(void);

/*
 * The asynchronous half of the same convention (tilelang (velog) section 1.3, the host call():
 * the launch is enqueued and its status returned at once, and an error that happens later on the
 * stream is read afterwards from the error buffer; here device-side timeouts are added to it).
 * Synchronises `stream`, then reports and clears the device status word of the current device:
 * GEMM_ERR_TIMEOUT if a kernel's bounded wait gave up since the last check (the kernel then
 * released its tensor memory and returned early, so C is incomplete), GEMM_ERR_CUDA if the
 * stream reported an error, GEMM_OK otherwise.
 */
int gemm_stream_status(dtc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DTC_GEMM_H */
