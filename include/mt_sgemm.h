/*
 * mt_sgemm — tiled fp32 matrix multiply for one NVIDIA GB300 (sm_103a).
 *
 * C ABI of the library (libmtsgemm.so).  Plain pointers and 64-bit sizes
 * only.  Every entry point returns an mt_status; none of them aborts, traps
 * or prints.
 *
 * The operation (all entry points that compute):
 *
 *     C[M,N] = A[M,K] * B[K,N]            fp32 in, fp32 out
 *
 * with A, B and C dense row-major: element (i,k) of A at A[i*K + k],
 * (k,j) of B at B[k*N + j], (i,j) of C at C[i*N + j].  This is the product
 * `tl.dot` computes in "My Triton From Scratch, Part 14: Shared Memory Tiles"
 * (section "The canonical source pattern": a + rows*K + columns,
 * b + rows*N + columns, masks rows < bound & columns < bound, other = 0.0)
 * accumulated over the runtime K loop of section "Staging inside a runtime K
 * loop" starting from zeros.  Tiles that straddle M, N or K read 0.0 outside
 * the matrix, so any M, N, K >= 0 is accepted and C is overwritten (never
 * accumulated into).  K == 0 writes zeros.  M == 0 or N == 0 does nothing.
 *
 * Ownership: every matrix pointer is owned by the caller.  The device entry
 * points take device-accessible memory and return before the work finishes
 * (stream-ordered, no implicit synchronisation); errors of the launch itself
 * come back as MT_ERR_LAUNCH, errors during execution surface at the
 * caller's next synchronisation.  The library keeps no per-call state; the
 * only global state is a per-device record of kernel attributes set once.
 * All entry points are thread-safe.
 *
 * There is no CPU fallback: without a usable CUDA device the computing entry
 * points return MT_ERR_NO_DEVICE.
 */
#ifndef MT_SGEMM_H
#define MT_SGEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MT_API __attribute__((visibility("default")))
#else
#define MT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MT_OK = 0,
    MT_ERR_INVALID_ARG = 1,   /* negative or too-large size, NULL pointer, bad config */
    MT_ERR_ALIAS = 2,         /* C overlaps A or B */
    MT_ERR_NO_DEVICE = 3,     /* no usable CUDA device */
    MT_ERR_UNSUPPORTED = 4,   /* tile configuration not built into the library */
    MT_ERR_SMEM_BUDGET = 5,   /* staged tiles do not fit the shared-memory limit */
    MT_ERR_LAUNCH = 6,        /* the kernel launch was rejected */
    MT_ERR_TIMEOUT = 7,       /* a kernel gave up waiting (device status word) */
    MT_ERR_CUDA = 8,          /* a CUDA runtime call (copy, allocation, sync) failed */
    MT_ERR_SCRATCH_LIMIT = 9  /* problem too large for mt_sgemm_tf32x3_noalloc's scratch */
} mt_status;

typedef enum {
    MT_VARIANT_FFMA = 0,      /* CUDA-core FFMA register-tile kernel (default) */
    MT_VARIANT_TF32X3 = 1,    /* tcgen05 kind::tf32 with the 3xTF32 split */
    MT_VARIANT_P18 = 2,       /* one-warp kernel restating the pages' Version 18 */
    MT_VARIANT_TC16 = 3       /* tcgen05 kind::f16 on 16-bit inputs (mt_gemm_mixed* only) */
} mt_variant;

/* Storage type of A and B in the mt_gemm_mixed* entry points. */
typedef enum {
    MT_DTYPE_F16 = 1,         /* IEEE 754 binary16 */
    MT_DTYPE_BF16 = 2         /* bfloat16: the upper 16 bits of a binary32 */
} mt_dtype;

/* Optional launch choices.  Zero-initialise for "automatic". */
typedef struct {
    int variant;   /* mt_variant */
    int bm;        /* CTA tile rows (M); 0 = automatic */
    int bn;        /* CTA tile columns (N); 0 = automatic */
    int bk;        /* K depth of one staged tile; 0 = automatic */
    int stages;    /* shared-memory stages in the K pipeline; 0 = automatic.  1 = one
                      stage, no double buffering (copy, barrier, compute, barrier):
                      MT_VARIANT_P18 and the FFMA 128 x 128 x 16 tile, to measure
                      what the pipeline buys */
    int no_pad;    /* 1 = store rows unpadded (bank-conflict measurements); 0 = padding rule */
    int split_k;   /* K slices reduced in a second pass; 0 = automatic, 1 = none */
    int fma;       /* FFMA micro-kernel: 0 = automatic, 1 = scalar fma.rn.f32,
                      2 = packed fma.rn.f32x2 (same results, fewer issue slots) */
    int fault_inject; /* test hook, 0 = off.  1 (MT_VARIANT_TF32X3 and the
                         mt_gemm_mixed* kernel only): the copy thread issues
                         nothing, so every wait on its data runs out; the call
                         then leaves C unwritten and the next
                         mt_check_device_status returns MT_ERR_TIMEOUT. */
    int wm;        /* FFMA warp tile rows; 0 = automatic */
    int wn;        /* FFMA warp tile columns; 0 = automatic */
    int tm;        /* FFMA outputs per thread along M; 0 = automatic */
    int tn;        /* FFMA outputs per thread along N; 0 = automatic */
    int pack_a;    /* 0 = automatic.  MT_VARIANT_TF32X3: 1 = split A into a packed
                      copy by a separate kernel, 2 = split A inside the GEMM kernel
                      (A not transposed, 16-byte aligned, lda % 4 == 0).
                      MT_VARIANT_FFMA, row-major A tiles: 1 = copy operands the
                      16-byte staging cannot read as stored (transposed, rows not
                      whole float4s, unaligned) into zero-padded row-major scratch
                      first, 2 = stage them as stored (4-byte copies).
                      MT_VARIANT_FFMA, A tiles K-major (each k row holds BM rows of
                      A; the micro-kernel reads four rows with one float4): 3 =
                      source chosen automatically, 4 = gathered from A stored M x K
                      inside the kernel (A not transposed), 5 = from a K x M copy of
                      A (transposing A stored M x K); A stored K x M with M % 4 ==
                      0, lda % 4 == 0 and a 16-byte aligned base is read as stored.
                      B is copied into padded rows when the 16-byte staging cannot
                      read it.  Automatic (0): K-major A when padding is on and B
                      is 16-byte readable or M >= 512, from a copy when A is stored
                      K x M or N >= 1024 with 2^30 multiply-adds or more, else
                      gathered.  Every choice gives the same bits. */
    int group_m;   /* tile rows per group of the tile raster (tiles are walked
                      down a group's rows, then across); 0 = automatic */
    int schedule;  /* How tiles that do not fill a whole wave of resident CTAs
                      are run.  0 = automatic; 1 = whole tiles, with a grid
                      smaller than the SMs or a last wave under half full cut
                      into equal K slices (split tail); 2 = stream-K: those
                      tiles' K tiles spread evenly over one wave of CTAs (for
                      the persistent tensor-core kernels, over the grid after
                      each CTA's whole tiles), each taking a contiguous run
                      across tile boundaries, and the pieces of a tile added in
                      k order by a second kernel (deterministic).  split_k = 1
                      turns both off; split_k > 1 with 2, an explicit FFMA
                      tile whose warps form K groups (automatic tiles avoid
                      them) and MT_VARIANT_P18 are MT_ERR_UNSUPPORTED. */
} mt_config;

/* What a call with the same arguments would launch. */
typedef struct {
    int variant;
    int bm, bn, bk, stages;
    int pad_a, pad_b;         /* padding words appended to each shared row of A and B */
    int threads;              /* threads per CTA */
    int vec_ab;               /* 1: 16-byte staging of A and B; 0: 4-byte staging */
    int vec_c;                /* 1: 16-byte stores of C; 0: 4-byte stores */
    int split_k;              /* K slices (1 = none) */
    int fma;                  /* 1 scalar, 2 packed (FFMA variant; 0 otherwise) */
    int wm, wn;               /* warp tile (FFMA variant; 0 otherwise) */
    int tm, tn;               /* outputs per thread (FFMA variant; 0 otherwise) */
    int64_t grid;             /* CTAs of the main kernel */
    int64_t smem_bytes;       /* dynamic shared memory per CTA */
    int64_t workspace_bytes;  /* device scratch the call needs (0 = none) */
    int pack_a;               /* MT_VARIANT_TF32X3: 1 = A packed by its own kernel,
                                 2 = A split inside the GEMM kernel.  MT_VARIANT_FFMA:
                                 1 = operands copied into padded scratch first
                                 (row-major A tiles); 3 = A tiles K-major read as
                                 stored, 4 = gathered, 5 = from a K x M copy.
                                 0 otherwise */
    int stream_k;             /* CTAs running stream-K runs (the last ones of the
                                 grid; 0 = none) */
} mt_plan;

/*
 * C = A*B on `stream` with the default variant and automatic tiling.  The
 * default variant of every fp32 call made without a configuration (cfg ==
 * NULL here and in the _ex, general and host entry points) is FFMA, or the
 * one the environment variable MT_SGEMM_VARIANT names when the call is
 * made: "ffma", "tf32x3" or "p18" (unset or empty: "ffma"; any other value:
 * MT_ERR_INVALID_ARG, nothing launched).  A configuration's variant field
 * always wins.
 * A, B, C: device pointers, layouts above.  A and B may be NULL only when
 * the product has no element that reads them (M*K == 0 or K*N == 0).
 * Errors: MT_ERR_INVALID_ARG (size < 0 or > INT32_MAX per dimension,
 * NULL pointer), MT_ERR_ALIAS (C overlaps A or B), MT_ERR_NO_DEVICE,
 * MT_ERR_SMEM_BUDGET, MT_ERR_LAUNCH.  Nothing is launched on error.
 */
MT_API mt_status mt_sgemm(const float *A, const float *B, float *C,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* As mt_sgemm, with explicit choices (cfg == NULL: same as mt_sgemm).
 * A choice the library was not built for returns MT_ERR_UNSUPPORTED.
 * The product is the one cited for mt_sgemm; the choices themselves have no
 * counterpart on the pages, whose compiler picks one tile (BM = 4, BN = 8,
 * BK = 16 in "My Triton From Scratch, Part 14: Shared Memory Tiles",
 * section "Shared buffers are physical storage") and two stages ("Part 18",
 * section "One stage versus two stages"). */
MT_API mt_status mt_sgemm_ex(const float *A, const float *B, float *C,
                      int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                      const mt_config *cfg);

/*
 * The general form, BLAS-style:
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * op(A) is M x K: A[i*lda + k], or A[k*lda + i] when trans_a (A stored
 * K x M); op(B) is K x N: B[k*ldb + j], or B[j*ldb + k] when trans_b (B
 * stored N x K); C[i][j] is at C[i*ldc + j].  The pages' loads are the
 * row-major case with packed rows ("My Triton From Scratch, Part 14: Shared
 * Memory Tiles", section "Cooperative copy mapping" supports the order
 * (1, 0) alone); this entry point adds any leading dimension, transposed storage
 * and the alpha/beta update.  trans_a, trans_b: 0 or 1.  Leading dimensions
 * in elements: lda >= (trans_a ? M : K), ldb >= (trans_b ? K : N),
 * ldc >= N, each at least 1.  beta == 0: C is only written (NaN or Inf in
 * C do not propagate); alpha == 0 or K == 0: A and B are not read and
 * C = beta * C.  mt_sgemm(A, B, C, M, N, K, s) is the same as
 * mt_sgemm_general(0, 0, M, N, K, 1, A, K, B, N, 0, C, N, s, NULL).
 * Every variant supports every form; FFMA stages transposed operands with
 * 4-byte copies (the automatic tiles and 64 x 64 only — other explicit
 * tiles return MT_ERR_UNSUPPORTED).  Errors as mt_sgemm_ex (MT_ERR_ALIAS
 * compares the spans each view covers).
 */
MT_API mt_status mt_sgemm_general(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                  float alpha, const float *A, int64_t lda, const float *B,
                                  int64_t ldb, float beta, float *C, int64_t ldc,
                                  cudaStream_t stream, const mt_config *cfg);

/*
 * The general form with a bias row, fused into the epilogue:
 *
 *     C[i][j] = alpha * (op(A) * op(B))[i][j] + beta * C[i][j] + bias[j]
 *
 * bias: N floats in device memory (4-byte aligned), added to every row of C
 * after the alpha/beta update, in fp32; NULL is the same as
 * mt_sgemm_general.  The pages stop at the plain product; the bias epilogue
 * is the usual one of a linear layer (a per-output-column vector) and is
 * the plainest reading of "bias" for this product.  With alpha == 0 or
 * K == 0, C = beta * C + bias.  bias overlapping C is MT_ERR_ALIAS; a bias
 * not 4-byte aligned is MT_ERR_INVALID_ARG.  Every variant applies it,
 * including its K-slice reduce.  Other errors as mt_sgemm_general.
 */
MT_API mt_status mt_sgemm_general_bias(int trans_a, int trans_b, int64_t M, int64_t N,
                                       int64_t K, float alpha, const float *A, int64_t lda,
                                       const float *B, int64_t ldb, float beta,
                                       const float *bias, float *C, int64_t ldc,
                                       cudaStream_t stream, const mt_config *cfg);

/*
 * C = A*B with A, B, C in HOST memory (pageable or pinned).  Copies A and B
 * to the device, multiplies, copies C back and synchronises `stream` before
 * returning, so on MT_OK the host C holds the result.  Large products are
 * cut into row blocks of A and C: the copy in of one block and the copy out
 * of another run on the library's own copy streams while the product of a
 * third runs on `stream` (with pinned host memory the copies overlap the
 * products; the result is the same as mt_sgemm_ex's).  Device buffers come
 * from the stream-ordered pool of the current device and are returned to it
 * before the call ends.  Errors as mt_sgemm_ex, plus MT_ERR_CUDA when a
 * copy, allocation or the final synchronisation fails.
 */
MT_API mt_status mt_sgemm_host(const float *A, const float *B, float *C,
                        int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                        const mt_config *cfg);

/*
 * mt_sgemm_host without the final synchronisation: the copies in, products
 * and copies out are enqueued and the call returns; the result is in the
 * host C once `stream` has completed the work enqueued before the return
 * (for example after cudaStreamSynchronize(stream)).  A, B and C must stay
 * valid and A, B unchanged until then.  With pinned host memory successive
 * calls overlap: a call's copies in start while the products of the calls
 * before it still run.  With pageable C the copies out are synchronous, so
 * the call returns only when it is done.  Errors found before anything is
 * enqueued are returned; a failure of enqueued work shows at the
 * synchronisation, as for any stream work.
 */
MT_API mt_status mt_sgemm_host_async(const float *A, const float *B, float *C,
                                     int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                                     const mt_config *cfg);

/*
 * Allocation-free form of the MT_VARIANT_TF32X3 call, for callers that must
 * not allocate device memory while they run: code whose device memory is
 * owned by someone else (a host application or framework that hands it a
 * fixed budget, or a caching allocator it must not bypass) and real-time
 * loops that reserve everything at start-up, because cudaMalloc and
 * cudaFree can synchronise the device, take unbounded time or fail under
 * memory pressure in the middle of a step.  The paper has no counterpart:
 * its kernels need no scratch memory.
 *
 * Same arguments, layouts and result as mt_sgemm_ex with
 * cfg->variant = MT_VARIANT_TF32X3 (device pointers, stream-ordered).  The
 * packed copies of A and B that variant builds go to a static device array
 * of MT_NOALLOC_SCRATCH_BYTES (32 MiB) instead of memory allocated per call;
 * this call allocates nothing.  A problem needs the workspace_bytes that
 * mt_sgemm_plan reports for MT_VARIANT_TF32X3 (with the same A, B and C, as
 * the plan depends on their alignment); that figure is the exact test.  It
 * holds the packed big and small copies of B, about 8*N*K bytes, and of A,
 * about 8*M*K more, unless A is split inside the GEMM kernel (A row-major,
 * lda % 4 == 0, 16-byte aligned, and N <= 1024 or M*N*K <= 2^33: square
 * problems up to 2048^3 pack only B), plus the fp32 partial tiles of a
 * last round split over K (this call cannot turn that split off).  A
 * problem over the limit returns MT_ERR_SCRATCH_LIMIT and launches nothing.
 * Other errors as mt_sgemm_ex.
 *
 * The array is shared by every call in the process: calls that overlap on
 * the GPU (different streams, or host threads) race on it and must be
 * serialised by the caller.  Each call rewrites all of the scratch it reads,
 * so nothing needs clearing between calls.  Every device that loads the
 * library holds the array until the process exits.  The first call on a
 * device looks up the array's device address and sets the kernel's
 * shared-memory limit (no allocation); make that first call before any
 * stream capture.  The address is kept for the life of the process, like
 * the library's other per-device set-up: calls on a device after
 * cudaDeviceReset on it are not supported.
 */
#define MT_NOALLOC_SCRATCH_BYTES (32ll << 20)
MT_API mt_status mt_sgemm_tf32x3_noalloc(const float *A, const float *B, float *C,
                                         int64_t M, int64_t N, int64_t K,
                                         cudaStream_t stream);

/*
 * Mixed precision: A and B stored as 16-bit floating point (both fp16 or
 * both bf16, `dtype`), C in fp32, products and sums in fp32:
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * with the layouts, leading dimensions (in elements), transposes and
 * alpha/beta rules of mt_sgemm_general.  The pages announce mixed-precision
 * types as their next part ("My Triton From Scratch, Part 18: Shared Memory
 * Optimization", section "Next": Part 19, Mixed-Precision Types); this is
 * their product with 16-bit storage and fp32 accumulation.  A product of two
 * 16-bit values is exact in fp32; only the accumulation rounds.
 *
 * Runs on the tensor cores (tcgen05.mma kind::f16, MT_VARIANT_TC16) with
 * the operands read by TMA straight from A and B.  TMA needs a 16-byte
 * aligned base and a row pitch that is a multiple of 8 elements; an operand
 * without them is first copied into a padded scratch matrix from the
 * current device's stream-ordered pool (mt_gemm_mixed_plan reports the
 * bytes as workspace_bytes, vec_ab = 1 when no copy is needed).
 * A and B: 2-byte aligned device pointers.  cfg (NULL = automatic): variant
 * 0 or MT_VARIANT_TC16; bn 0, 256 or 128; bm 0 or 128; bk 0 or 64; stages 0
 * or the built count; split_k 0 (automatic tail split) or 1 (none);
 * fault_inject as for MT_VARIANT_TF32X3; other fields 0, else
 * MT_ERR_UNSUPPORTED.  dtype other than MT_DTYPE_F16 / MT_DTYPE_BF16:
 * MT_ERR_INVALID_ARG.  MT_ERR_CUDA when the driver's tensor-map encoder
 * cannot be found or scratch cannot be allocated.  Other errors as
 * mt_sgemm_general.
 */
MT_API mt_status mt_gemm_mixed_general(int dtype, int trans_a, int trans_b, int64_t M,
                                       int64_t N, int64_t K, float alpha, const void *A,
                                       int64_t lda, const void *B, int64_t ldb, float beta,
                                       float *C, int64_t ldc, cudaStream_t stream,
                                       const mt_config *cfg);

/* mt_gemm_mixed_general with the bias row of mt_sgemm_general_bias (N fp32
 * values added to every row of C after the alpha/beta update; NULL = none). */
MT_API mt_status mt_gemm_mixed_general_bias(int dtype, int trans_a, int trans_b, int64_t M,
                                            int64_t N, int64_t K, float alpha, const void *A,
                                            int64_t lda, const void *B, int64_t ldb,
                                            float beta, const float *bias, float *C,
                                            int64_t ldc, cudaStream_t stream,
                                            const mt_config *cfg);

/* C = A*B with 16-bit A (M x K, row stride K) and B (K x N, row stride N),
 * fp32 C (M x N): mt_gemm_mixed_general(dtype, 0, 0, M, N, K, 1, A, K, B, N,
 * 0, C, N, stream, NULL). */
MT_API mt_status mt_gemm_mixed(int dtype, const void *A, const void *B, float *C,
                               int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* The launch mt_gemm_mixed_general would make for these arguments, as
 * mt_sgemm_plan (pointers inspected for alignment only, may be NULL).  No
 * counterpart on the pages beyond the budget check cited for
 * mt_sgemm_plan. */
MT_API mt_status mt_gemm_mixed_plan(int dtype, int trans_a, int trans_b, int64_t M,
                                    int64_t N, int64_t K, const void *A, int64_t lda,
                                    const void *B, int64_t ldb, const float *C, int64_t ldc,
                                    const mt_config *cfg, int64_t smem_limit_bytes,
                                    mt_plan *out);

/* The launch mt_sgemm_general would make for these arguments, as
 * mt_sgemm_plan (pointers inspected for alignment only, may be NULL).  No
 * counterpart on the pages beyond the budget check cited for
 * mt_sgemm_plan. */
MT_API mt_status mt_sgemm_general_plan(int trans_a, int trans_b, int64_t M, int64_t N,
                                       int64_t K, const float *A, int64_t lda,
                                       const float *B, int64_t ldb, const float *C,
                                       int64_t ldc, const mt_config *cfg,
                                       int64_t smem_limit_bytes, mt_plan *out);

/*
 * Fills *out with the launch a call with these arguments would make,
 * without launching anything.  A, B, C are only inspected for 16-byte
 * alignment (they may be NULL, which counts as aligned).  smem_limit_bytes
 * is the per-CTA dynamic shared-memory limit to check against; <= 0 asks
 * the current device (MT_ERR_NO_DEVICE without one).  Returns the status the
 * call itself would return for these sizes and choices.  The pages check the
 * staged tiles' bytes against the device limit before a kernel is emitted
 * ("My Triton From Scratch, Part 18", section "Shared-memory budget checks
 * include stages and padding"; Part 14, section "Tracking the shared-memory
 * budget"); this is that check, plus the rest of the launch, made visible.
 */
MT_API mt_status mt_sgemm_plan(const float *A, const float *B, const float *C,
                        int64_t M, int64_t N, int64_t K, const mt_config *cfg,
                        int64_t smem_limit_bytes, mt_plan *out);

/*
 * The pages' padding rule ("My Triton From Scratch, Part 18: Shared Memory
 * Optimization", section "Choosing padding instead of hard-coding it"):
 * distinct_banks = 32 / gcd(columns, 32); returns 1 when simultaneous_rows
 * > distinct_banks, else 0.  Returns -1 when columns or simultaneous_rows
 * is not positive.  Pure host function.
 */
MT_API int mt_smem_row_padding(int columns, int simultaneous_rows);

/*
 * The same rule counted in 16-byte slots, for rows read with float4 loads:
 * 32 banks form 8 slots, a row of `columns` words spans columns/4 slots;
 * returns the padding in words (0 or 4).  -1 when columns is not a positive
 * multiple of 4 or simultaneous_rows is not positive.  Pure host function.
 */
MT_API int mt_smem_vector_row_padding(int columns, int simultaneous_rows);

/*
 * Physical layout of a staged shared tile ("My Triton From Scratch, Part 18",
 * section "A shared buffer needs a physical row stride"): row_stride =
 * columns + row_padding, stage_size = rows * row_stride, size = stage_count *
 * stage_size elements, nbytes = 4 * size.  The kernels address their shared
 * tiles through the same structure.
 */
typedef struct {
    int rows, columns, row_padding, stage_count;
    int row_stride, stage_size, size;
    int64_t nbytes;
} mt_smem_layout;

/* Fills *out; MT_ERR_INVALID_ARG for non-positive rows, columns or
 * stage_count, or negative padding.  Pure host function. */
MT_API mt_status mt_smem_layout_make(int rows, int columns, int row_padding,
                              int stage_count, mt_smem_layout *out);

/* Element offset stage*stage_size + row*row_stride + column, or -1 when the
 * coordinate lies outside the logical tile.  Pure host function. */
MT_API int64_t mt_smem_layout_offset(const mt_smem_layout *layout, int stage, int row,
                              int column);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: MT_ERR_TIMEOUT if a kernel gave up a bounded wait since
 * the last check, MT_ERR_CUDA if the synchronisation failed,
 * MT_ERR_NO_DEVICE without a usable device, else MT_OK.
 * No counterpart on the pages: their kernels never wait on a flag, and an
 * error of theirs surfaces at the caller's next synchronisation.  The
 * tensor-core kernels here wait on mbarriers with an iteration limit, and
 * this call is how a caller learns that a limit ran out.  Thread-safe; the
 * status word is per device and shared by every stream on it, so a check
 * clears what work on any stream of the device recorded.
 */
MT_API mt_status mt_check_device_status(cudaStream_t stream);

/* The same call under its earlier name (kept for existing callers). */
MT_API mt_status mt_device_status(cudaStream_t stream);

/*
 * The bounds-checked build.  libmtsgemm_checked.so is these sources built
 * with MT_BOUNDS_CHECK=1: the kernels of the FFMA path (the FFMA GEMM, its
 * operand copies, the K-slice reduce and C scaling, the one-warp kernel)
 * test every global and shared access against the extent of its buffer
 * before making it.  An access outside is skipped (a copy zero-fills, a
 * read gives 0, a store is dropped), so a checked kernel never touches
 * memory outside its buffers, and it is counted.  This stands in for a
 * memory checker where none can run; it is for tests and is slower than the
 * normal build.  No counterpart on the pages: they validate shared-memory
 * budgets before emitting a kernel ("My Triton From Scratch, Part 18",
 * section "Shared-memory budget checks include stages and padding") but
 * check no access at run time.  Sites of the first access found outside:
 */
typedef enum {
    MT_SITE_A_LOAD = 1,     /* global read of A by the staging copies */
    MT_SITE_B_LOAD = 2,     /* global read of B by the staging copies */
    MT_SITE_A_SMEM = 3,     /* shared write of a staged A tile */
    MT_SITE_B_SMEM = 4,     /* shared write of a staged B tile */
    MT_SITE_FRAG = 5,       /* shared read of an A or B fragment */
    MT_SITE_C_STORE = 6,    /* global read or write of C */
    MT_SITE_PARTIAL = 7,    /* global read or write of a K-slice partial tile */
    MT_SITE_BIAS = 8,       /* global read of the bias row */
    MT_SITE_SLICE_SUM = 9,  /* shared read or write of a K group's sum */
    MT_SITE_PREP_SRC = 10,  /* global read of an operand by the copy kernel */
    MT_SITE_PREP_DST = 11,  /* global write of an operand copy */
    MT_SITE_P18 = 12        /* any access of the one-warp kernel */
} mt_bounds_site;

/*
 * Checked build: synchronises the current device, then reads and clears its
 * record of accesses found outside their buffers: *count of them, and the
 * first one's *site (mt_bounds_site), element *offset within its buffer and
 * the buffer's *extent in elements (any pointer may be NULL).  Errors:
 * MT_ERR_NO_DEVICE, MT_ERR_CUDA.  The normal build checks nothing and
 * returns MT_ERR_UNSUPPORTED without touching the outputs.
 */
MT_API mt_status mt_bounds_status(int64_t *count, int *site, int64_t *offset, int64_t *extent);

/* Static English name of a status code.  No counterpart on the pages. */
MT_API const char *mt_status_string(mt_status status);

/* Library version: major*10000 + minor*100 + patch.  No counterpart on the
 * pages. */
MT_API int mt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MT_SGEMM_H */
