/*
 * gb300gemm.h - C ABI of the GB300 (sm_103a) dense NT GEMM library.
 *
 * All entry points:
 *  - take plain pointers and sizes; no framework types cross this boundary;
 *  - take DEVICE pointers for every matrix (memory the caller allocated on
 *    the current CUDA device); the library allocates no per-call memory and
 *    never takes ownership of a buffer;
 *  - enqueue their work on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and return without synchronising;
 *  - validate every argument on the host BEFORE launching anything and
 *    return a GEMM_ERR_* code without side effects when validation fails;
 *  - return GEMM_OK (0) when the work was enqueued.
 *
 * One-time set-up: the first call of any entry point on a device (with that
 * device current) reads its attributes and looks up the device addresses of
 * the library's own __device__ variables.  Make that first call outside any
 * stream capture; during a capture it returns GEMM_ERR_CAPTURE and does
 * nothing (a later call outside capture does the set-up).
 *
 * Threads: any host thread may call any entry point, concurrently with
 * others (the per-device set-up is serialised inside the library).  The
 * driver's tensor-map encoder needs a current context: a call from a thread
 * that has none makes the current device's primary context current there
 * (cudaSetDevice on the device that is already current).  A context the
 * caller made current is left as it is, and the current device is never
 * changed.
 *
 * Device-side wait limits: every wait inside a kernel is bounded (two
 * seconds).  A kernel that runs out of a wait stops, records a code in a
 * device status word and returns; gemm_get_device_status() reports it.
 *
 * Layouts are row-major.  "NT" means C[M,N] = A[M,K] . B[N,K]^T, i.e. B is
 * stored like a HuggingFace weight ([out_features, in_features]).
 */
#ifndef GB300GEMM_H
#define GB300GEMM_H

#include <stddef.h>

#if defined(__GNUC__)
#define GB300GEMM_API __attribute__((visibility("default")))
#else
#define GB300GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define GEMM_OK             0
#define GEMM_ERR_NULL       1  /* a required pointer is NULL */
#define GEMM_ERR_SHAPE      2  /* a dimension is <= 0, too large, or breaks a multiple-of rule */
#define GEMM_ERR_ALIGN      3  /* a pointer or a row pitch is not 16-byte aligned */
#define GEMM_ERR_ALIAS      4  /* an output buffer overlaps an input buffer */
#define GEMM_ERR_ARCH       5  /* the current device is not an sm_100-family (sm_103) GPU */
#define GEMM_ERR_LAUNCH     6  /* a CUDA call failed (launch, attribute, tensor-map encode) */
#define GEMM_ERR_TIMEOUT    7  /* a kernel ran out of a bounded device-side wait */
#define GEMM_ERR_NO_DEVICE  8  /* no usable CUDA device / driver */
#define GEMM_ERR_CAPTURE    9  /* the first call on a device was made during stream capture */

/*
 * gemm_bf16_nt - dense BF16 GEMM, C = bf16(A . B^T) with FP32 accumulation.
 *
 * Defined by: "gemm_dense.rs" (spark_model layers/ops), dense_gemm_tc doc
 * comment (A [M,K] activations, B [N,K] weights in HuggingFace layout, C
 * [M,N], all row-major); "sm121a_matmul.py", _sm121a_matmul_kernel (BF16
 * inputs, FP32 accumulator, BF16 store).
 *
 *   A  bf16 [M][K], row pitch K elements     (read)
 *   B  bf16 [N][K], row pitch K elements     (read)
 *   C  bf16 [M][N], row pitch N elements     (written; must not overlap A or B)
 *   M, N, K >= 1;  K % 8 == 0 and N % 8 == 0 (16-byte row pitches);
 *   A, B, C 16-byte aligned.
 * The order in which the tensor cores add the K products is the hardware's.
 * Errors: GEMM_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _ARCH, _LAUNCH.
 */
GB300GEMM_API int gemm_bf16_nt(const void* A, const void* B, void* C, int M, int N, int K, void* stream);

/*
 * gemm_bf16_nn - C[M,N] = bf16( A[M,K] . B[K,N] ), the NN layout: B stored
 * K rows of N (row-major [K][N]); FP32 accumulation on the tensor cores.
 *
 * Defined by: "sm121a_matmul.py", _sm121a_matmul_kernel and its docstring
 * (A [M,K], B [K,N], FP32 accumulator, BF16 store).
 *
 *   A bf16 [M][K], B bf16 [K][N], C bf16 [M][N] (written), row-major;
 *   M, N, K >= 1; K % 8 == 0 and N % 8 == 0 (16-byte row pitches); every
 *   pointer 16-byte aligned; C must not overlap A or B.
 * Results equal gemm_bf16_nt on the transposed B bit for bit (same tiles,
 * same K order).
 * Errors: GEMM_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _ARCH, _LAUNCH, _NO_DEVICE.
 */
GB300GEMM_API int gemm_bf16_nn(const void* A, const void* B, void* C, int M, int N, int K,
                               void* stream);

/*
 * gemm_bf16_nt_scaled_acc - fused LoRA expand+fold:
 *     C[m,n] = bf16( float(C[m,n]) + scale * float(bf16(sum_k A[m,k] B[n,k])) )
 * The GEMM result is rounded to BF16 first, then multiplied by `scale` in
 * FP32, then added in FP32 (separately rounded), then rounded to BF16, so the
 * result is bit-identical to gemm_bf16_nt into a BF16 scratch followed by
 * bf16_scaled_add.  C is read once and written once.
 *
 * Defined by: "gemm_dense.rs", dense_gemm_tc_scaled_acc doc comment (output
 * += scale * bf16(input @ weight^T) in one pass, bit-identical to the unfused
 * GEMM-into-scratch + bf16_scaled_add pair).
 *
 *   A, B, M, N, K as for gemm_bf16_nt;  C_inout bf16 [M][N] (read and written
 *   in place, must not overlap A or B);  scale any finite float.
 * Errors: as gemm_bf16_nt.
 */
GB300GEMM_API int gemm_bf16_nt_scaled_acc(const void* A, const void* B, void* C_inout, int M, int N, int K,
                            float scale, void* stream);

/*
 * gemm_w4a16 - BF16 activations times NVFP4 weights:
 *     w[n,k]  = e2m1(b[n,k]) * e4m3(sfb[n,k/16])          (exact in BF16)
 *     C[m,n]  = bf16( scale2 * sum_k A[m,k] * w[n,k] ), FP32 accumulation
 * The block-scaled weight has at most six significant bits, so its BF16
 * form is exact; the per-tensor scale multiplies the FP32 sum once, then the
 * result is rounded to BF16 (nearest, ties to even).  The weights are
 * dequantised on chip, stage by stage, and never written out.
 *
 * Defined by: "gemm_dense.rs", w4a16_gemm doc comment (C = A @ dequant(B);
 * A [M,K] BF16 activations; B NVFP4 packed weights: E2M1 codes, FP8 scales
 * and an FP32 per-tensor scale; C [M,N] BF16) and the doc comment of
 * w4a16_gemm_n128_m128_bf16 (FP4 dequantised to BF16, BF16 MMA, FP32
 * accumulation).  This entry point takes the weights as HuggingFace-
 * oriented rows (below); gemm_w4a16_t takes the page's transposed layout.
 * The page gives no place for the per-tensor scale; the library applies it
 * to the FP32 sum (C is linear in it).
 *
 *   A      bf16 [M][K], row pitch K                        (read)
 *   b      uint8 [N][K/2]: element k of row n in byte k/2, low nibble for
 *          even k, high nibble for odd k                   (read)
 *   sfb    uint8 [N][K/16] e4m3: byte j of row n scales elements
 *          16j .. 16j+15 of row n                          (read)
 *   scale2 the FP32 per-tensor scale
 *   C      bf16 [M][N] (written; must not overlap A, b or sfb)
 *   M, N, K >= 1; K % 256 == 0 and N % 8 == 0 (16-byte rows of sfb, b and
 *   C, which the tensor-memory-access copies need); every pointer 16-byte
 *   aligned.
 * Errors: GEMM_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _ARCH, _LAUNCH, _NO_DEVICE.
 */
GB300GEMM_API int gemm_w4a16(const void* A, const void* b, const void* sfb, float scale2, void* C,
                             int M, int N, int K, void* stream);

/*
 * gemm_w4a16_t - gemm_w4a16 with the weights in the transposed NVFP4 layout:
 *     w[n,k]  = e2m1(nibble k%2 of b_t[k/2][n]) * e4m3(sfb_t[k/16][n])
 *     C[m,n]  = bf16( scale2 * sum_k A[m,k] * w[n,k] ), FP32 accumulation
 * Same arithmetic, same result as gemm_w4a16 on the transposed bytes.
 *
 * Defined by: "gemm_dense.rs", w4a16_gemm_n128_m128_bf16 doc comment (the
 * lossless BF16 variant: same math as w4a16_gemm, weight layout "transposed
 * NVFP4"), w4a16_gemm_n128_ldb doc comment (transposed-B rows sit r * ldb
 * bytes apart; pass ldb = align_up(n, 128) when N is not a multiple of 16,
 * because 16-byte copies fault on misaligned rows) and w4a16_gemm_n128
 * (packed case: rows exactly N apart).  The library's reading: b_t is the
 * [N][K/2] code-byte matrix of gemm_w4a16 transposed, sfb_t the [N][K/16]
 * scale matrix transposed, both with row stride ldb.
 *
 *   A      bf16 [M][K], row pitch K                        (read)
 *   b_t    uint8 [K/2][ldb]: byte (j, n) holds element 2j of weight column
 *          n in its low nibble and element 2j+1 in its high nibble (read)
 *   sfb_t  uint8 [K/16][ldb] e4m3: byte (j, n) scales elements 16j .. 16j+15
 *          of column n                                     (read)
 *   ldb    row stride of b_t and sfb_t in bytes: ldb >= N, ldb % 16 == 0;
 *          bytes n >= N of a row are padding and never affect C
 *   scale2 the FP32 per-tensor scale
 *   C      bf16 [M][N], row pitch N (any N >= 1; written; must not overlap
 *          A, b_t or sfb_t)
 *   M, N, K >= 1; K % 128 == 0; every pointer 16-byte aligned.
 * Errors: GEMM_ERR_NULL, _SHAPE (also ldb < N), _ALIGN (also K % 128,
 * ldb % 16), _ALIAS, _ARCH, _LAUNCH, _NO_DEVICE.
 */
GB300GEMM_API int gemm_w4a16_t(const void* A, const void* b_t, const void* sfb_t, float scale2,
                               void* C, int M, int N, int K, int ldb, void* stream);

/*
 * gemm_w4a16_ws - gemm_w4a16 in two passes: the weights are first converted
 * once into `workspace` (BF16 [N][K], w = e2m1 * e4m3, exact), then the
 * dense CTA-pair GEMM multiplies A by them with the same tiles, K order and
 * epilogue (bf16(scale2 * sum)).  Results are bit-identical to gemm_w4a16.
 * For large M (prefill) this is faster: the fused kernel converts each
 * weight tile once per 256-row block of A; at small M the fused kernel
 * reads 3.6x fewer weight bytes and needs no workspace.
 *
 * Defined by: as gemm_w4a16.
 *
 *   A, b, sfb, scale2, C, M, N, K as for gemm_w4a16;  workspace: caller-owned
 *   device memory of at least gemm_w4a16_ws_workspace_bytes(N, K) bytes,
 *   16-byte aligned, not overlapping A, b, sfb or C; on return it holds the
 *   converted weights.
 * Errors: as gemm_w4a16; GEMM_ERR_NULL also for a NULL workspace,
 * GEMM_ERR_SHAPE for one that is too small.
 */
GB300GEMM_API int gemm_w4a16_ws(const void* A, const void* b, const void* sfb, float scale2,
                                void* C, void* workspace, size_t workspace_bytes, int M, int N,
                                int K, void* stream);

/* Workspace bytes gemm_w4a16_ws needs (N*K*2; 0 if N, K are invalid). */
GB300GEMM_API size_t gemm_w4a16_ws_workspace_bytes(int N, int K);

/*
 * gemm_bf16_nt_splitk - BF16 NT GEMM with the K dimension split into
 * `k_splits` chunks, for shapes with too few output tiles to fill the GPU:
 *     partial_s[m,n] = sum over the K blocks of split s of A[m,k] B[n,k]
 *     C[m,n]         = bf16( ((partial_0 + partial_1) + ...) + partial_{S-1} )
 * Each split's FP32 partial tile goes to `workspace`; a second kernel adds
 * the splits in split order (deterministic) and rounds once to BF16.  K is
 * split in 64-element blocks: S = min(k_splits, ceil(K/64)) reduced so that
 * no split is empty (gemm_bf16_nt_splitk_workspace_bytes gives the size).
 *
 * Defined by: "gemm_dense.rs", dense_gemm_splitk doc comment (partial
 * products over K_splits chunks into an FP32 workspace of
 * K_splits*M*N*4 bytes, then a reduce kernel writes BF16).
 *
 *   A, B, C, M, N, K as for gemm_bf16_nt;  workspace: caller-owned device
 *   memory of at least gemm_bf16_nt_splitk_workspace_bytes(M,N,K,k_splits)
 *   bytes, 16-byte aligned, not overlapping A, B or C; its contents on entry
 *   are ignored and on return are unspecified;  1 <= k_splits <= 64.
 * Errors: as gemm_bf16_nt; GEMM_ERR_SHAPE also for a bad k_splits or a
 * workspace that is too small.
 */
GB300GEMM_API int gemm_bf16_nt_splitk(const void* A, const void* B, void* C, void* workspace,
                                      size_t workspace_bytes, int M, int N, int K, int k_splits,
                                      void* stream);

/* Workspace bytes gemm_bf16_nt_splitk needs for these arguments (0 if invalid). */
GB300GEMM_API size_t gemm_bf16_nt_splitk_workspace_bytes(int M, int N, int K, int k_splits);

/*
 * gemm_bf16_nt_streamk - BF16 NT GEMM, C = bf16(A . B^T), scheduled for
 * shapes whose 256 x 256 tile count leaves part of the last wave idle.
 * One cluster of two CTAs (one CTA pair) runs per co-resident slot, P of
 * them.  The first floor(tiles / P) rounds of tiles are computed whole, as
 * gemm_bf16_nt computes them.  The remaining tiles' 128-deep K iterations
 * are dealt out evenly: pair p takes iterations [T*p/P, T*(p+1)/P) of the
 * T left.  A tile whose iterations span several pairs is summed from their
 * FP32 partial tiles in K order by a second kernel and rounded once to BF16;
 * every other tile equals gemm_bf16_nt's bit for bit.
 *
 * Defined by: "gemm_dense.rs", dense_gemm_tc doc comment (the product) and
 * dense_gemm_splitk doc comment (FP32 partial products over K chunks in a
 * workspace, reduced to BF16); the work loop of persistent_block_scaled_gemm
 * in "kernelbot-nvfp4-gemm-123329" (one program per slot striding over the
 * tiles).  Dividing the last round's K iterations over every slot is this
 * library's schedule; the pages have no such step.
 *
 *   A, B, C, M, N, K as for gemm_bf16_nt;  workspace: caller-owned device
 *   memory of at least gemm_bf16_nt_streamk_workspace_bytes() bytes (one
 *   size for every shape on the current device), 16-byte aligned, not
 *   overlapping A, B or C; contents on entry ignored, on return unspecified.
 * Errors: as gemm_bf16_nt; GEMM_ERR_SHAPE also for a workspace that is too
 * small; GEMM_ERR_NULL for a NULL workspace.
 */
GB300GEMM_API int gemm_bf16_nt_streamk(const void* A, const void* B, void* C, void* workspace,
                                       size_t workspace_bytes, int M, int N, int K, void* stream);

/* Workspace bytes gemm_bf16_nt_streamk needs on the current device: two FP32
 * 256 x 256 tiles per CTA pair of the device; 0 when no CUDA device is usable. */
GB300GEMM_API size_t gemm_bf16_nt_streamk_workspace_bytes(void);

/*
 * gemm_bf16_nt_splitk_static - gemm_bf16_nt_splitk without a workspace
 * argument, for callers that cannot allocate device memory: code whose host
 * framework owns the whole device pool and forbids other allocations,
 * serving loops that must not call the CUDA allocator after warm-up (an
 * allocation can synchronise the device), and plugins handed raw pointers
 * but no allocator.  The pages have no counterpart; it is a library
 * extension.
 *
 * The FP32 partial tiles go to a fixed scratch array of
 * GEMM_SPLITK_STATIC_SCRATCH_BYTES that is part of the library's device
 * image: every GPU that loads the library holds it until the process exits.
 * This call allocates nothing and frees nothing.  The caller still passes
 * A, B and C exactly as for gemm_bf16_nt_splitk, and the result is the same.
 *
 *   Limit: S * M * N * 4 <= GEMM_SPLITK_STATIC_SCRATCH_BYTES, with S the
 *   splits actually used (gemm_bf16_nt_splitk_workspace_bytes); larger
 *   problems are rejected with GEMM_ERR_SHAPE before anything is launched.
 *   The scratch array's device address is looked up (cudaGetSymbolAddress
 *   with that device current) in the library's one-time per-device set-up,
 *   i.e. by the first call of any entry point on the device; make that first
 *   call before any stream capture (during a capture it returns
 *   GEMM_ERR_CAPTURE).
 *   All calls share the one array and it keeps the last call's contents; no
 *   element needs to start at zero (each call writes every element it reads
 *   before reading it).  Calls whose executions overlap on the GPU (other
 *   streams, other host threads) race on the array and give wrong results:
 *   order them on one stream or with events.
 * Errors: GEMM_ERR_NULL, _SHAPE (dims, k_splits, or over the limit),
 * _ALIGN, _ALIAS, _ARCH, _NO_DEVICE, _CAPTURE, _LAUNCH.
 */
#define GEMM_SPLITK_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
GB300GEMM_API int gemm_bf16_nt_splitk_static(const void* A, const void* B, void* C, int M, int N,
                                             int K, int k_splits, void* stream);

/*
 * gemm_bf16_nt_ordered - order-preserving "router" GEMM with FP32 output:
 *     C[m,n] = (((0 + A[m,0]B[n,0]) + A[m,1]B[n,1]) + ... + A[m,K-1]B[n,K-1])
 * every product and every sum rounded to FP32 (round to nearest even), no
 * fused multiply-add, subnormals kept.  Runs on CUDA cores; the result is
 * bit-identical to the strict sequential loop.
 *
 * Defined by: "gemm_dense.rs", dense_gemm_router doc comment (same math and
 * same per-output FP32 accumulation order, strict k = 0..K-1, as the scalar
 * dense_gemm; bit-identical under --fmad=false) and dense_gemm.
 *
 *   A bf16 [M][K], B bf16 [N][K] (read);  C float [M][N] (written, must not
 *   overlap A or B);  M, N, K >= 1;  K % 8 == 0;  A, B, C 16-byte aligned.
 * Errors: GEMM_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _LAUNCH.
 */
GB300GEMM_API int gemm_bf16_nt_ordered(const void* A, const void* B, float* C, int M, int N, int K,
                         void* stream);

/*
 * gemm_nvfp4_bs - NVFP4 block-scaled GEMM with FP16 output, for each l < L:
 *     c[l][m][n] = fp16( sum_k  e2m1(a[l][m][k]) * e4m3(SFA(l,m,k/16))
 *                             * e2m1(b[l][n][k]) * e4m3(SFB(l,n,k/16)) )
 * accumulated in FP32 on the tensor cores (hardware order).
 *
 * Defined by: "kernelbot nvfp4 gemm submission 123329": module docstring
 * sections "SCALE FACTORS" (one scale per 16 consecutive K elements),
 * "NVIDIA Block layout" and "Layout semantics" (scale layout below), and
 * custom_kernel (a, b packed float4_e2m1fn_x2; c float16; mkl -> lmk
 * physical order; M % 128, N % 128, K % 256 asserts).
 *
 *   a    [L][M][K/2] bytes: two e2m1 codes per byte, element 2j in the low
 *        nibble of byte j and element 2j+1 in the high nibble.
 *   b    [L][N][K/2] bytes, same packing.
 *   sfa  L*M*K/16 e4m3 bytes in the hardware layout: logical
 *        [32,4,M/128,4,K/64,L] with dims [g,i_m,tile,i_k,tile_k,l], row
 *        r = tile*128 + i_m*32 + g, group j = tile_k*4 + i_k, stored in the
 *        order l, tile, tile_k, g, i_m, i_k; i.e. the byte of (r, j, l) is at
 *        ((l*(M/128) + r/128)*(K/64) + j/4)*512 + (r%32)*16 + ((r%128)/32)*4 + j%4.
 *   sfb  L*N*K/16 bytes, the same layout over N.
 *   c    fp16 [L][M][N] (written; must not overlap a, b, sfa, sfb).
 *   L >= 1, M % 128 == 0, N % 128 == 0, K % 256 == 0, all > 0;
 *   every pointer 16-byte aligned.  Scale bytes are read as unsigned e4m3
 *   (the sign bit must be clear).
 * Errors: GEMM_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _ARCH, _LAUNCH.
 */
GB300GEMM_API int gemm_nvfp4_bs(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                  int L, int M, int N, int K, void* stream);

/*
 * gemm_nvfp4_bs_splitk - gemm_nvfp4_bs with K split into `k_splits`
 * chunks, for problems with too few output tiles to fill the GPU
 * (decode-like M = 128): each chunk's FP32 partial product goes into
 * workspace[s][l][M][N], then the chunks are summed in split order in FP32
 * (deterministic) and rounded once to FP16.  With M <= 256 the kernel swaps
 * the operand roles (the weight rows b take the MMA's 256-row side of a CTA
 * pair, the activation rows the MMA N) and stores the partials transposed;
 * the result is the same product.
 *
 * Defined by: the operation is gemm_nvfp4_bs's ("kernelbot nvfp4 gemm
 * submission 123329", custom_kernel and the docstring's layout sections;
 * its benchmark shapes include M = 128 with K = 16384 and K = 7168); the
 * split-K scheme is "gemm_dense.rs", dense_gemm_splitk (FP32 partials over
 * K chunks, then a reduce).
 *
 *   a, b, sfa, sfb, c, L, M, N, K: as gemm_nvfp4_bs (L >= 1).
 *   K is split in 256-element blocks: S = min(k_splits, K/256), reduced so
 *   that every chunk is non-empty (gemm_nvfp4_bs_splitk_workspace_bytes
 *   gives S*M*N*4 for the S used, per batch).
 *   workspace: caller-owned device memory of at least
 *   L * gemm_nvfp4_bs_splitk_workspace_bytes(M,N,K,k_splits) bytes, 16-byte
 *   aligned, overlapping no operand; contents on entry are ignored, on
 *   return unspecified.  1 <= k_splits <= 64.
 * The FP32 sum order differs from gemm_nvfp4_bs (per chunk, then across
 * chunks), so results may differ from it in the last FP16 bit.
 * Errors: as gemm_nvfp4_bs; GEMM_ERR_SHAPE also for a bad k_splits or a
 * workspace that is too small; GEMM_ERR_NULL for a NULL workspace.
 */
GB300GEMM_API int gemm_nvfp4_bs_splitk(const void* a, const void* b, const void* sfa,
                                       const void* sfb, void* c, void* workspace,
                                       size_t workspace_bytes, int L, int M, int N, int K,
                                       int k_splits, void* stream);

/* Workspace bytes gemm_nvfp4_bs_splitk needs per batch (0 for invalid
 * arguments); an L-batch call needs L times this. */
GB300GEMM_API size_t gemm_nvfp4_bs_splitk_workspace_bytes(int M, int N, int K, int k_splits);

/*
 * bf16_scaled_add - out[i] = bf16( float(out[i]) + scale * float(d[i]) ),
 * product and sum each rounded to FP32.  The second kernel of the unfused
 * LoRA pair (GEMM into a BF16 scratch, then this), kept as the baseline the
 * fused gemm_bf16_nt_scaled_acc must match bit for bit.
 *
 * Defined by: "gemm_dense.rs", dense_gemm_tc_scaled_acc doc comment (the
 * unfused pair: GEMM into scratch, then bf16_scaled_add).
 *
 *   out bf16 [n] (read and written), d bf16 [n] (read), n >= 1;
 *   out and d 16-byte aligned and not overlapping.
 * Errors: GEMM_ERR_NULL, _SHAPE, _ALIGN, _ALIAS, _LAUNCH.
 */
GB300GEMM_API int bf16_scaled_add(void* out, const void* d, float scale, long n, void* stream);

/*
 * gemm_get_device_status - synchronise `stream`, then read and clear the
 * device status word of the current device.  Returns GEMM_OK, or
 * GEMM_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, or GEMM_ERR_LAUNCH if the stream reports a CUDA error.
 * Library extension (the pages define no such call).
 */
GB300GEMM_API int gemm_get_device_status(void* stream);

/*
 * gemm_selftest_wait_timeout - diagnostic of the failure path.  Launches one
 * CTA that waits, through the same bounded wait the GEMM kernels use, on a
 * barrier that nothing ever arrives on, with the limit `timeout_ms`
 * (1..10000).  The wait gives up, records a timeout in the device status
 * word and the kernel returns normally; the next gemm_get_device_status()
 * returns GEMM_ERR_TIMEOUT and the CUDA context stays usable.
 * Library extension (the pages define no such call).
 * Errors: GEMM_ERR_SHAPE (timeout out of range), _ARCH, _NO_DEVICE, _LAUNCH.
 */
GB300GEMM_API int gemm_selftest_wait_timeout(int timeout_ms, void* stream);

/*
 * gemm_testing_set_overrides - process-wide testing hook, not for production
 * use.  Forces choices the library otherwise makes from the shape, so that
 * tests can reach every kernel configuration:
 *   cta_group         0 = by shape; 1 or 2 = the single-CTA or the CTA-pair
 *                     configuration of gemm_bf16_nt, gemm_bf16_nn,
 *                     gemm_bf16_nt_scaled_acc and the BF16 split-K calls;
 *   streamk_clusters  0 = by shape; P >= 1 = gemm_bf16_nt_streamk divides the
 *                     last round's K iterations over min(P, pairs) CTA pairs.
 * Results stay within each call's documented accuracy whatever is forced.
 * Takes effect for calls made after it returns.  Library extension (the
 * pages define no such call).
 * Errors: GEMM_ERR_SHAPE (a value out of range).
 */
GB300GEMM_API int gemm_testing_set_overrides(int cta_group, int streamk_clusters);

/* gemm_status_string - static, human-readable name of a status code. */
GB300GEMM_API const char* gemm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_H */
