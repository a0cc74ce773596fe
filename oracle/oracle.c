/*
 * CPU oracle for the dense NT GEMM family and its three variants.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no code, header, table
 * or constant with the CUDA path.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -pthread.
 * -ffp-contract=off matters: aarch64 GCC would otherwise fuse a*b+c into an
 * FMA, which changes the rounding of every accumulation step below.
 *
 * Sources (page title, section):
 *  - "sm121a_matmul.py" (DGX Spark Unsloth kernels), _sm121a_matmul_kernel:
 *    BF16 x BF16 -> FP32 accumulator -> BF16 store.
 *  - "gemm_dense.rs" (spark_model layers/ops), dense_gemm_tc: C = A @ B^T
 *    with A [M,K] and B [N,K] row-major (HuggingFace weight layout).
 *  - "gemm_dense.rs", dense_gemm_tc_scaled_acc: out += scale * bf16(A @ B^T),
 *    with the delta rounded to BF16 before scaling, identical to the unfused
 *    "GEMM into BF16 scratch, then bf16_scaled_add" pair.
 *  - "gemm_dense.rs", dense_gemm / dense_gemm_router: per-output FP32 sum in
 *    strict k = 0..K-1 order, built with --fmad=false (no FMA contraction).
 *  - "kernelbot nvfp4 gemm submission 123329", module docstring sections
 *    "SCALE FACTORS", "NVIDIA Block layout" and "Layout semantics", plus
 *    custom_kernel: e2m1 values packed two per byte, one e4m3 scale per 16 K
 *    elements, scales stored as [32,4,rest_m,4,rest_k,L] with memory order
 *    l, tile_m, tile_k, g_m, i_m, i_k; FP16 output.
 *  - "gemm_dense.rs", w4a16_gemm / w4a16_gemm_n128_m128_bf16: BF16
 *    activations times NVFP4 weights dequantised to BF16, FP32 accumulation.
 *
 * Every function follows its definition literally: no blocking, no
 * reordering of the k sum, one output at a time.
 *
 * Parity pins: every exported function is pinned by the CPU tests
 * (tests/test_oracle_pins.py) against brute force FP64, closed forms,
 * library casts and hand-derived layout examples.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                          */
/* ------------------------------------------------------------------------ */

/* bfloat16 -> float: the bf16 bit pattern is the top half of an IEEE binary32. */
ORACLE_API float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float -> bfloat16, round to nearest, ties to even.  NaN stays a (quiet) NaN. */
ORACLE_API uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u) {
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t kept = u >> 16;              /* sign, exponent, 7 mantissa bits */
    uint32_t dropped = u & 0xffffu;       /* the 16 bits that are rounded away */
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) {
        kept += 1u;                       /* carries into the exponent as needed */
    }
    return (uint16_t)kept;
}

/*
 * double -> IEEE binary16, round to nearest, ties to even, with subnormals,
 * overflow to infinity, and NaN kept.  Works on the exact binary expansion
 * of the double: value = mant * 2^exp with a 53-bit integer mant.
 */
ORACLE_API uint16_t oracle_f64_to_f16(double x) {
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 48) & 0x8000u);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs(x);
    if (isinf(x)) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2);                  /* a = fr * 2^e2, fr in [0.5, 1) */
    /* binary16 normal range: a >= 2^-14, i.e. e2 >= -13.  The quantum
     * (value of one unit in the last place) is 2^(e2-11) for normals and
     * 2^-24 for subnormals. */
    int q = (e2 >= -13) ? (e2 - 11) : -24;
    double scaled = ldexp(a, -q);         /* exact: only the exponent changes */
    double fl = floor(scaled);
    double rem = scaled - fl;             /* exact: scaled < 2^53 */
    double r = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
    double v = ldexp(r, q);               /* the rounded magnitude */
    if (v >= 65536.0) return (uint16_t)(sign | 0x7c00u);  /* beyond max finite */
    /* encode v */
    if (v < ldexp(1.0, -14)) {            /* subnormal (or rounded up to min normal below) */
        uint32_t m = (uint32_t)ldexp(v, 24);
        return (uint16_t)(sign | m);      /* m == 1024 encodes the min normal exactly */
    }
    int ev;
    double fv = frexp(v, &ev);            /* v = fv * 2^ev, fv in [0.5,1) */
    uint32_t expf16 = (uint32_t)(ev - 1 + 15);
    uint32_t man = (uint32_t)ldexp(fv * 2.0 - 1.0, 10);
    if (expf16 >= 31u) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (expf16 << 10) | man);
}

ORACLE_API double oracle_f16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0x1f) v = (m == 0) ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

/*
 * e2m1 (FP4): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit, no
 * infinities or NaN.  Exponent field 0 is subnormal: m * 0.5.
 */
ORACLE_API double oracle_e2m1_decode(unsigned code) {
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double v = (e == 0u) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -v : v;
}

/*
 * e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN.  Exponent field 0 is subnormal:
 * (m/8) * 2^-6.
 */
ORACLE_API double oracle_e4m3_decode(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double v;
    if (e == 15u && m == 7u) v = NAN;
    else if (e == 0u) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/*
 * Byte offset of scale (row r, 16-element group j, batch l) in the
 * hardware scale layout: logical shape [32,4,rest_rows,4,rest_k,L] with dims
 * [g, i_m, tile, i_k, tile_k, l], where r = tile*128 + i_m*32 + g and
 * j = tile_k*4 + i_k, and memory order l, tile, tile_k, g, i_m, i_k
 * (sizes L, rest_rows, rest_k, 32, 4, 4).
 */
ORACLE_API long oracle_sf_offset(long r, long j, long l, long rest_rows, long rest_k) {
    long tile = r / 128;
    long i_m = (r % 128) / 32;
    long g = r % 32;
    long tile_k = j / 4;
    long i_k = j % 4;
    /* strides from the memory order: i_k 1, i_m 4, g 16, tile_k 512,
     * tile 512*rest_k, l 512*rest_k*rest_rows */
    return l * (512L * rest_k * rest_rows) + tile * (512L * rest_k) + tile_k * 512L
         + g * 16L + i_m * 4L + i_k;
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver: each worker takes whole output rows; every output   */
/* is still one sequential k loop.                                          */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(void* ctx, long out_row_index);

typedef struct {
    row_fn fn;
    void* ctx;
    long nrows;
    long next;
    pthread_mutex_t lock;
} row_pool;

static void* row_worker(void* arg) {
    row_pool* p = (row_pool*)arg;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        long i = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (i >= p->nrows) break;
        p->fn(p->ctx, i);
    }
    return NULL;
}

static void run_rows(row_fn fn, void* ctx, long nrows, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((long)threads > nrows) threads = (int)(nrows > 0 ? nrows : 1);
    row_pool p;
    p.fn = fn; p.ctx = ctx; p.nrows = nrows; p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    if (threads == 1) {
        row_worker(&p);
    } else {
        pthread_t tid[256];
        int started = 0;
        for (int t = 0; t < threads; ++t) {
            if (pthread_create(&tid[t], NULL, row_worker, &p) == 0) started++;
            else break;
        }
        if (started == 0) row_worker(&p);
        for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    }
    pthread_mutex_destroy(&p.lock);
}

/* ------------------------------------------------------------------------ */
/* BF16 NT GEMM family.                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t* A;   /* [M][K] bf16 */
    const float* Bf;     /* [N][K] B widened to float (exact) */
    long M, N, K;
    const long* rows;    /* which rows of C to produce (NULL: 0..nrows-1) */
    int mode;            /* 0: bf16 C, 1: scaled-acc, 2: fp32 router C, 3: bf16(scale * sum) */
    float scale;
    void* out;           /* [nrows][N] */
} bf16_ctx;

/* acc = +0.0f; for k = 0..K-1: acc = acc + a[m,k]*b[n,k], each op rounded to fp32 */
static float dot_fp32_strict(const float* a, const float* b, long K) {
    float acc = 0.0f;
    for (long k = 0; k < K; ++k) {
        float p = a[k] * b[k];
        acc = acc + p;
    }
    return acc;
}

static void bf16_row(void* vctx, long i) {
    bf16_ctx* c = (bf16_ctx*)vctx;
    long m = c->rows ? c->rows[i] : i;
    long K = c->K, N = c->N;
    float* arow = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
    for (long k = 0; k < K; ++k) arow[k] = oracle_bf16_to_f32(c->A[m * K + k]);
    for (long n = 0; n < N; ++n) {
        float acc = dot_fp32_strict(arow, c->Bf + n * K, K);
        if (c->mode == 0) {
            ((uint16_t*)c->out)[i * N + n] = oracle_f32_to_bf16(acc);
        } else if (c->mode == 1) {
            /* d = bf16(acc); out = bf16(float(out) + scale*float(d)),
             * product and sum each rounded to fp32 */
            uint16_t* o = (uint16_t*)c->out + i * N + n;
            float d = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));
            float t = c->scale * d;
            float r = oracle_bf16_to_f32(*o) + t;
            *o = oracle_f32_to_bf16(r);
        } else if (c->mode == 3) {
            /* one FP32 multiply of the sum, then one rounding to bf16 */
            float t = c->scale * acc;
            ((uint16_t*)c->out)[i * N + n] = oracle_f32_to_bf16(t);
        } else {
            ((float*)c->out)[i * N + n] = acc;
        }
    }
    free(arow);
}

/* The row loop over a B already widened to float (bf16 values, exact). */
static int run_bf16_widened(const uint16_t* A, const float* Bf, void* out, long M, long N,
                            long K, const long* rows, long nrows, int mode, float scale,
                            int threads) {
    if (!rows) nrows = M;
    for (long i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -2;
    bf16_ctx c = {A, Bf, M, N, K, rows, mode, scale, out};
    run_rows(bf16_row, &c, nrows, threads);
    return 0;
}

static int run_bf16(const uint16_t* A, const uint16_t* B, void* out, long M, long N, long K,
                    const long* rows, long nrows, int mode, float scale, int threads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    float* Bf = (float*)malloc(sizeof(float) * (size_t)(N * K > 0 ? N * K : 1));
    if (!Bf) return -3;
    for (long t = 0; t < N * K; ++t) Bf[t] = oracle_bf16_to_f32(B[t]);
    int rc = run_bf16_widened(A, Bf, out, M, N, K, rows, nrows, mode, scale, threads);
    free(Bf);
    return rc;
}

/*
 * C[i][n] = bf16( sum_k fp32 A[rows[i],k]*B[n,k] ) for i < nrows (rows == NULL:
 * every row, nrows ignored).  C is [nrows][N] bf16.
 */
ORACLE_API int oracle_gemm_bf16_nt(const uint16_t* A, const uint16_t* B, uint16_t* C,
                                   long M, long N, long K, const long* rows, long nrows,
                                   int threads) {
    return run_bf16(A, B, C, M, N, K, rows, nrows, 0, 0.0f, threads);
}

/*
 * out[i][n] = bf16( float(out[i][n]) + scale * float(bf16(acc)) ), the fused
 * LoRA expand+fold.  out holds the initial values of the selected rows.
 */
ORACLE_API int oracle_gemm_bf16_nt_scaled_acc(const uint16_t* A, const uint16_t* B,
                                              uint16_t* out, long M, long N, long K,
                                              float scale, const long* rows, long nrows,
                                              int threads) {
    return run_bf16(A, B, out, M, N, K, rows, nrows, 1, scale, threads);
}

/* Ordered FP32 "router" GEMM: the same strict k loop, FP32 output, no rounding. */
ORACLE_API int oracle_gemm_router(const uint16_t* A, const uint16_t* B, float* C,
                                  long M, long N, long K, const long* rows, long nrows,
                                  int threads) {
    return run_bf16(A, B, C, M, N, K, rows, nrows, 2, 0.0f, threads);
}

/* The second half of the unfused pair: out = bf16(float(out) + scale*float(d)). */
ORACLE_API void oracle_bf16_scaled_add(uint16_t* out, const uint16_t* d, float scale, long n) {
    for (long i = 0; i < n; ++i) {
        float t = scale * oracle_bf16_to_f32(d[i]);
        float r = oracle_bf16_to_f32(out[i]) + t;
        out[i] = oracle_f32_to_bf16(r);
    }
}

/* Elementwise casts over arrays (used by the codec pins). */
ORACLE_API void oracle_f32_to_bf16_array(const float* x, uint16_t* y, long n) {
    for (long i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]);
}
ORACLE_API void oracle_f64_to_f16_array(const double* x, uint16_t* y, long n) {
    for (long i = 0; i < n; ++i) y[i] = oracle_f64_to_f16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 block-scaled GEMM.                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* a;    /* [L][M][K/2] packed e2m1 */
    const uint8_t* b;    /* [L][N][K/2] packed e2m1 */
    const uint8_t* sfa;  /* hardware layout, rest_m = M/128, rest_k = K/64 */
    const uint8_t* sfb;  /* hardware layout, rest_n = N/128 */
    long L, M, N, K;
    const long* rows;    /* flat row ids l*M + m (NULL: all L*M rows) */
    uint16_t* c;         /* [nrows][N] fp16 */
} nvfp4_ctx;

/* Element k of a packed row: byte k/2, low nibble for even k, high for odd k. */
static unsigned fp4_code(const uint8_t* row, long k) {
    uint8_t byte = row[k / 2];
    return (k % 2 == 0) ? (byte & 0x0fu) : (byte >> 4);
}

static void nvfp4_row(void* vctx, long i) {
    nvfp4_ctx* c = (nvfp4_ctx*)vctx;
    long flat = c->rows ? c->rows[i] : i;
    long l = flat / c->M, m = flat % c->M;
    long K = c->K, N = c->N, Kh = K / 2;
    long rest_m = c->M / 128, rest_n = N / 128, rest_k = K / 64;
    const uint8_t* arow = c->a + (l * c->M + m) * Kh;
    /* dequantised A row: e2m1(a[m,k]) * e4m3(sfa[m, k/16]), exact in double */
    double* ad = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (long k = 0; k < K; ++k) {
        double s = oracle_e4m3_decode(c->sfa[oracle_sf_offset(m, k / 16, l, rest_m, rest_k)]);
        ad[k] = oracle_e2m1_decode(fp4_code(arow, k)) * s;
    }
    for (long n = 0; n < N; ++n) {
        const uint8_t* brow = c->b + (l * N + n) * Kh;
        double acc = 0.0;
        for (long k = 0; k < K; ++k) {
            double s = oracle_e4m3_decode(c->sfb[oracle_sf_offset(n, k / 16, l, rest_n, rest_k)]);
            double bv = oracle_e2m1_decode(fp4_code(brow, k)) * s;
            acc = acc + ad[k] * bv;
        }
        c->c[i * N + n] = oracle_f64_to_f16(acc);
    }
    free(ad);
}

/*
 * c[i][n] = fp16( sum_k e2m1(a)*sfa * e2m1(b)*sfb ) accumulated in FP64.
 * For the inputs the tests use (e2m1 magnitudes <= 6, scales 2^-4..2^2,
 * K <= 16384) every partial sum is an integer multiple of 2^-10 below 2^24,
 * so the FP64 sum is exact and the single rounding to FP16 is correct.
 * Requires M % 128 == 0, N % 128 == 0, K % 64 == 0.
 */
ORACLE_API int oracle_gemm_nvfp4_bs(const uint8_t* a, const uint8_t* b, const uint8_t* sfa,
                                    const uint8_t* sfb, uint16_t* c, long L, long M, long N,
                                    long K, const long* rows, long nrows, int threads) {
    if (L < 1 || M < 128 || N < 128 || K < 64) return -1;
    if (M % 128 || N % 128 || K % 64) return -1;
    if (!rows) nrows = L * M;
    for (long i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= L * M) return -2;
    nvfp4_ctx ctx = {a, b, sfa, sfb, L, M, N, K, rows, c};
    run_rows(nvfp4_row, &ctx, nrows, threads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* W4A16: BF16 activations x NVFP4 weights.                                 */
/* ------------------------------------------------------------------------ */

/*
 * "gemm_dense.rs", w4a16_gemm doc comment: C = A @ dequant(B) with A [M,K]
 * BF16 activations, B NVFP4 weights (e2m1 codes, FP8 e4m3 scales, an FP32
 * per-tensor scale) and C [M,N] BF16; the doc comment of its BF16 variant
 * (w4a16_gemm_n128_m128_bf16) names the math: FP4 dequantised to BF16, BF16
 * products accumulated in FP32.
 * Readings (the page gives no layout or rounding):
 *  - b: N rows of K/2 bytes, element k in byte k/2, low nibble for even k
 *    (the packing of the NVFP4 page); sfb: N rows of K/16 e4m3 bytes, byte
 *    j of row n scaling elements 16j .. 16j+15 of row n;
 *  - the BF16 weight is the block-scaled value w[n,k] = e2m1(b[n,k]) *
 *    e4m3(sfb[n,k/16]), which BF16 holds exactly (at most six significant
 *    bits, magnitude in [2^-10, 2688]): the dequantisation rounds nothing;
 *  - the per-tensor scale multiplies the FP32 sum once:
 *    C[m,n] = bf16( scale2 * (strict FP32 sum over k of A[m,k] * w[n,k]) ),
 *    the product rounded to FP32, then to BF16 (nearest, ties to even).
 *    C = A @ dequant(B) is linear in scale2, so this is the same product
 *    with one rounding where scaling every weight would add one per weight.
 * Requires K % 16 == 0.  C is [nrows][N] bf16.
 */
ORACLE_API int oracle_gemm_w4a16(const uint16_t* A, const uint8_t* b, const uint8_t* sfb,
                                 float scale2, uint16_t* C, long M, long N, long K,
                                 const long* rows, long nrows, int threads) {
    if (M < 0 || N < 0 || K < 0 || K % 16) return -1;
    float* W = (float*)malloc(sizeof(float) * (size_t)(N * K > 0 ? N * K : 1));
    if (!W) return -3;
    for (long n = 0; n < N; ++n) {
        const uint8_t* brow = b + n * (K / 2);
        for (long k = 0; k < K; ++k) {
            double q = oracle_e2m1_decode(fp4_code(brow, k))
                     * oracle_e4m3_decode(sfb[n * (K / 16) + k / 16]);
            W[n * K + k] = (float)q;        /* exact */
        }
    }
    int rc = run_bf16_widened(A, W, C, M, N, K, rows, nrows, 3, scale2, threads);
    free(W);
    return rc;
}

/*
 * W4A16 with the weights in the "transposed NVFP4" layout of "gemm_dense.rs"
 * (w4a16_gemm_n128_m128_bf16 doc comment: same math as w4a16_gemm, weight
 * layout "transposed NVFP4"; w4a16_gemm_n128_ldb doc comment: the
 * transposed-B rows sit at r * ldb, ldb = align_up(n, 128) with the pad
 * columns zero-filled; w4a16_gemm_n128: packed rows are exactly N apart).
 * Reading: the byte matrix [N][K/2] of the row-oriented form, transposed:
 *  - b_t: K/2 rows of ldb bytes; byte (j, n) holds elements k = 2j (low
 *    nibble) and k = 2j + 1 (high nibble) of weight column n, so that a
 *    byte stride of ldb per row makes odd N misalign 15 of every 16 rows;
 *  - sfb_t: K/16 rows of ldb e4m3 bytes; byte (j, n) scales elements
 *    16j .. 16j+15 of column n (the scales transposed the same way);
 *  - bytes n >= N of a row (the padding) are never read.
 * The arithmetic is oracle_gemm_w4a16's: w[n,k] = e2m1 * e4m3 (exact), the
 * strict FP32 sum over k, then C = bf16(scale2 * sum).
 * Requires K % 16 == 0 and ldb >= N.
 */
ORACLE_API int oracle_gemm_w4a16_t(const uint16_t* A, const uint8_t* b_t, const uint8_t* sfb_t,
                                   float scale2, uint16_t* C, long M, long N, long K, long ldb,
                                   const long* rows, long nrows, int threads) {
    if (M < 0 || N < 0 || K < 0 || K % 16 || ldb < N) return -1;
    float* W = (float*)malloc(sizeof(float) * (size_t)(N * K > 0 ? N * K : 1));
    if (!W) return -3;
    for (long n = 0; n < N; ++n) {
        for (long k = 0; k < K; ++k) {
            uint8_t byte = b_t[(k / 2) * ldb + n];
            unsigned code = (k % 2 == 0) ? (byte & 0x0fu) : (byte >> 4);
            double q = oracle_e2m1_decode(code) * oracle_e4m3_decode(sfb_t[(k / 16) * ldb + n]);
            W[n * K + k] = (float)q;        /* exact */
        }
    }
    int rc = run_bf16_widened(A, W, C, M, N, K, rows, nrows, 3, scale2, threads);
    free(W);
    return rc;
}
