/*
 * iq4xs_oracle.c -- plain, slow CPU oracle for the IQ4_XS x Q8_1 batched
 * matmul  y[M,N] = x[M,K] . W[N,K]^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the IQ4_XS layout, the codebook and the Q8_1 rule are restated
 * here from the format description on their own.
 *
 * Sources (V100TPS engine report, agent-report.daedalus.work/V100TPS/engine.html):
 *   - "tile geometry" passage after the new-kernel table: an IQ4_XS 32-element
 *     sub-block holds 4 ints of packed nibbles, low nibbles are elements 0-15
 *     and high nibbles 16-31; the per-sub-block scale is d*(ls-32) and a nibble
 *     is decoded through the kvalues_iq4nl table (not q-8).
 *   - kernel table (M=64): activations are quantized by quantize_q8_1 (Q8_1
 *     blocks of 32 int8 with scale d and sum term s).
 *   The super-block is 256 weights in 136 bytes: d (fp16), scales_h (u16),
 *   scales_l (u8[4]), qs (u8[128]); ls is 6 bits (4 from scales_l, 2 from
 *   scales_h).  Byte offsets follow the common GGUF order (d@0, scales_h@2,
 *   scales_l@4, qs@8) -- the pages list the fields but not their offsets, so
 *   this is a reading, and it is "parity unpinned" beyond self-consistency.
 *
 * Definitions written out here (no blocking, fusion or reordering):
 *   decode:   ls_j  = low/high nibble of scales_l[j/2] | ((scales_h >> 2j) & 3) << 4
 *             S_j   = float(d) * (ls_j - 32)                 (exact in fp32)
 *             w[16j+i]    = S_j * kv[qs[16j+i] & 15]          i < 16
 *             w[16j+16+i] = S_j * kv[qs[16j+i] >> 4]
 *   Q8_1:     amax = max|x| over 32;  d = amax/127 (fp32, IEEE RN);
 *             q = d == 0 ? 0 : roundf(x/d)  (fp32 IEEE division, ties away);
 *             stored d_h = half_rn(d), s_h = half_rn(d * (float)sum(q)).
 *   product:  y[m,n] = sum_b sum_j S_j * double(d_h[m,b,j]) * P[n,m,b,j],
 *             P = sum_i kv * q  (exact int32), accumulated in fp64 in natural
 *             (b, j) order.  Every term is an exact fp64 product.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread (no
 * intrinsics, no fast-math, no -march).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Format constants, restated from the IQ4_XS description.                   */
/* ------------------------------------------------------------------------ */
#define OR_QK          256   /* weights per super-block                      */
#define OR_SUB         32    /* weights per sub-block                        */
#define OR_NSUB        8     /* sub-blocks per super-block                   */
#define OR_BLOCK_BYTES 136   /* 2 + 2 + 4 + 128                              */
#define OR_OFF_D       0
#define OR_OFF_SCALES_H 2
#define OR_OFF_SCALES_L 4
#define OR_OFF_QS      8

/* kvalues_iq4nl: the 16-entry non-uniform codebook a nibble indexes. */
static const int or_kvalues[16] = {
    -127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};

int oracle_kvalue(int nibble) { return or_kvalues[nibble & 15]; }

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 / bfloat16 conversions written from the definitions.    */
/* Exact arithmetic is done in double (every float fits exactly).            */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double holding at most 53 significant bits to the
 * nearest integer, ties to even.  floor() and the comparisons are exact. */
static double or_rne_integer(double q) {
    double fl = floor(q);
    double r = q - fl; /* exact: q and fl share the exponent range */
    if (r > 0.5) return fl + 1.0;
    if (r < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

float oracle_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        if (m) return NAN;
        v = INFINITY;
    } else {
        v = ldexp((double)(m + 1024), e - 25); /* (1024+m) * 2^(e-15-10) */
    }
    return (float)(sign ? -v : v);
}

uint16_t oracle_f32_to_f16(float f) {
    if (isnan(f)) return 0x7E00;
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7C00;
    /* Values at or above 65520 (halfway between 65504 and 2^16) round to inf. */
    if (a >= 65520.0) return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {
        /* Subnormal range: quantum 2^-24.  m == 1024 lands on the smallest
         * normal, whose encoding (exponent 1, mantissa 0) is also 1024. */
        double m = or_rne_integer(a * ldexp(1.0, 24));
        return sign | (uint16_t)m;
    }
    int ex;
    (void)frexp(a, &ex);  /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;       /* a in [2^E, 2^(E+1)) */
    double m = or_rne_integer(a * ldexp(1.0, 10 - E)); /* in [1024, 2048] */
    if (m == 2048.0) { m = 1024.0; E += 1; }
    if (E > 15) return sign | 0x7C00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024));
}

float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t oracle_f32_to_bf16(float f) {
    /* bfloat16 keeps the fp32 exponent and 8 significant bits; round to
     * nearest even.  Done on the value, not on bit tricks. */
    if (isnan(f)) return 0x7FC0;
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int ex;
    (void)frexp(a, &ex);
    int E = ex - 1;
    if (E < -126) E = -126; /* fp32 subnormal range: fixed quantum 2^-133 */
    double m = or_rne_integer(a * ldexp(1.0, 7 - E)); /* significand, 8 bits */
    double v = ldexp(m, E - 7);
    if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
    float fv = (float)v; /* exact: v has <= 8 significant bits in range */
    uint32_t u;
    memcpy(&u, &fv, 4);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ------------------------------------------------------------------------ */
/* IQ4_XS decode.                                                            */
/* ------------------------------------------------------------------------ */

/* 6-bit scale of sub-block j (0..7) of one 136-byte super-block. */
int oracle_iq4xs_ls(const uint8_t* block, int j) {
    const uint8_t* scales_l = block + OR_OFF_SCALES_L;
    uint16_t scales_h = (uint16_t)(block[OR_OFF_SCALES_H] |
                                   (block[OR_OFF_SCALES_H + 1] << 8));
    int lo = (j & 1) ? (scales_l[j / 2] >> 4) : (scales_l[j / 2] & 0x0F);
    int hi = (scales_h >> (2 * j)) & 3;
    return lo | (hi << 4);
}

/* fp32 scale of sub-block j: float(d) * (ls - 32). */
float oracle_iq4xs_subblock_scale(const uint8_t* block, int j) {
    uint16_t dbits = (uint16_t)(block[OR_OFF_D] | (block[OR_OFF_D + 1] << 8));
    float d = oracle_f16_to_f32(dbits);
    return d * (float)(oracle_iq4xs_ls(block, j) - 32);
}

/* Codebook value (int) of element e (0..255) of a super-block. */
int oracle_iq4xs_code(const uint8_t* block, int e) {
    int j = e / OR_SUB;
    int i = e % OR_SUB;
    uint8_t byte = block[OR_OFF_QS + 16 * j + (i % 16)];
    int nib = (i < 16) ? (byte & 0x0F) : (byte >> 4);
    return or_kvalues[nib];
}

/* Decode the whole [N][K/256] block matrix to doubles, w[n*K + k]. */
int oracle_iq4xs_decode(const uint8_t* w, int64_t N, int64_t K, double* out) {
    if (K % OR_QK) return -1;
    int64_t nb = K / OR_QK;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* blk = w + (n * nb + b) * OR_BLOCK_BYTES;
            for (int e = 0; e < OR_QK; ++e) {
                float s = oracle_iq4xs_subblock_scale(blk, e / OR_SUB);
                out[n * K + b * OR_QK + e] = (double)s * (double)oracle_iq4xs_code(blk, e);
            }
        }
    }
    return 0;
}

/* Dequantize to fp32 (exact) and, if out_bf16 != NULL, to bfloat16 (RNE). */
int oracle_iq4xs_dequantize(const uint8_t* w, int64_t N, int64_t K, float* out_f32,
                            uint16_t* out_bf16) {
    if (K % OR_QK) return -1;
    int64_t nb = K / OR_QK;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* blk = w + (n * nb + b) * OR_BLOCK_BYTES;
            for (int e = 0; e < OR_QK; ++e) {
                float v = oracle_iq4xs_subblock_scale(blk, e / OR_SUB) *
                          (float)oracle_iq4xs_code(blk, e);
                if (out_f32) out_f32[n * K + b * OR_QK + e] = v;
                if (out_bf16) out_bf16[n * K + b * OR_QK + e] = oracle_f32_to_bf16(v);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Q8_1 activation quantization.                                             */
/* ------------------------------------------------------------------------ */

/* x: [M][ldx] fp32.  qs: [M][K] int8.  d_h, s_h: [M][K/32] fp16 bits.
 * Returns 0, or -1 on bad shape, -2 on a non-finite input, -3 if a code
 * falls outside [-127, 127] (cannot happen for finite input). */
int oracle_quantize_q8_1(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs,
                         uint16_t* d_h, uint16_t* s_h) {
    if (K % OR_SUB || ldx < K) return -1;
    int64_t nblk = K / OR_SUB;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < nblk; ++j) {
            const float* xb = x + m * ldx + j * OR_SUB;
            float amax = 0.0f;
            for (int i = 0; i < OR_SUB; ++i) {
                if (!isfinite(xb[i])) return -2;
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int i = 0; i < OR_SUB; ++i) {
                int q = 0;
                if (d != 0.0f) {
                    float t = xb[i] / d;
                    q = (int)roundf(t);
                }
                if (q < -127 || q > 127) return -3;
                qs[m * K + j * OR_SUB + i] = (int8_t)q;
                sum += q;
            }
            d_h[m * nblk + j] = oracle_f32_to_f16(d);
            s_h[m * nblk + j] = oracle_f32_to_f16(d * (float)sum);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Product, fp64 accumulation of exact per-sub-block integer dots.          */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* w;
    int64_t N, K;
    const int8_t* qs;
    const uint16_t* d_h;
    int64_t M;
    double* y;      /* [M][N] */
    int64_t n0, n1; /* row range of this worker */
    int status;
} or_mm_job;

static void* or_matmul_rows(void* arg) {
    or_mm_job* job = (or_mm_job*)arg;
    int64_t nb = job->K / OR_QK;
    int64_t nblk = job->K / OR_SUB;
    for (int64_t n = job->n0; n < job->n1; ++n) {
        for (int64_t m = 0; m < job->M; ++m) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* blk = job->w + (n * nb + b) * OR_BLOCK_BYTES;
                for (int j = 0; j < OR_NSUB; ++j) {
                    int64_t P = 0; /* accumulate wide, then check the int32 invariant */
                    for (int i = 0; i < OR_SUB; ++i) {
                        int e = j * OR_SUB + i;
                        P += (int64_t)oracle_iq4xs_code(blk, e) *
                             (int64_t)job->qs[m * job->K + b * OR_QK + e];
                    }
                    if (P > 516128 || P < -516128) { job->status = -3; return NULL; }
                    double sw = (double)oracle_iq4xs_subblock_scale(blk, j);
                    double dx = (double)oracle_f16_to_f32(job->d_h[m * nblk + b * OR_NSUB + j]);
                    acc += sw * dx * (double)P;
                }
            }
            job->y[m * job->N + n] = acc;
        }
    }
    return NULL;
}

/* y[M][N] (double) from IQ4_XS W [N][K/256] and Q8_1 (qs [M][K], d_h [M][K/32]).
 * nthreads <= 1 runs on the calling thread; otherwise rows n are split into
 * contiguous ranges, one POSIX thread each (the arithmetic per output is the
 * same either way). */
int oracle_matmul(const uint8_t* w, int64_t N, int64_t K, const int8_t* qs,
                  const uint16_t* d_h, int64_t M, double* y, int nthreads) {
    if (K % OR_QK || N < 0 || M < 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N && N > 0) nthreads = (int)N;
    if (nthreads <= 1) {
        or_mm_job job = {w, N, K, qs, d_h, M, y, 0, N, 0};
        or_matmul_rows(&job);
        return job.status;
    }
    or_mm_job* jobs = (or_mm_job*)calloc((size_t)nthreads, sizeof(or_mm_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -4; }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        or_mm_job j = {w, N, K, qs, d_h, M, y, N * t / nthreads, N * (t + 1) / nthreads, 0};
        jobs[t] = j;
        if (pthread_create(&th[t], NULL, or_matmul_rows, &jobs[t]) != 0) {
            or_matmul_rows(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        if (th[t]) pthread_join(th[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs);
    free(th);
    return status;
}

/* The per-sub-block integer dot P[n,m,b,j], exposed so tests can check the
 * int32 invariant (|P| <= 32*127*127) directly. */
int64_t oracle_subblock_dot(const uint8_t* w, int64_t K, const int8_t* qs, int64_t n,
                            int64_t m, int64_t b, int j) {
    int64_t nb = K / OR_QK;
    const uint8_t* blk = w + (n * nb + b) * OR_BLOCK_BYTES;
    int64_t P = 0;
    for (int i = 0; i < OR_SUB; ++i) {
        int e = j * OR_SUB + i;
        P += (int64_t)oracle_iq4xs_code(blk, e) * (int64_t)qs[m * K + b * OR_QK + e];
    }
    return P;
}

/* ------------------------------------------------------------------------ */
/* The 32-weight formats Q4_0 and IQ4_NL.                                    */
/*                                                                           */
/* V100TPS engine page, tile-geometry passage: one IQ4_XS sub-block is      */
/* exactly one Q4_0 block -- 4 ints of packed nibbles, low nibbles are       */
/* elements 0-15 and high nibbles 16-31 -- and the two formats differ only   */
/* in the scale (one d per 32 weights for Q4_0, d*(ls-32) per sub-block for  */
/* IQ4_XS) and in the value of a nibble (q-8 for Q4_0, kvalues_iq4nl for     */
/* IQ4_XS).  IQ4_NL is the kvalues_iq4nl codebook on blocks of 32 weights    */
/* in 18 bytes (forum page on the Qwen3.5 engine, the retracted TP claim:    */
/* the (32, 18) block shape of IQ4_NL).  Both blocks are 18 bytes: d (fp16)  */
/* at byte 0, then 16 bytes of nibbles (a reading: the pages give the sizes, */
/* not the offsets).                                                          */
/*   Q4_0:   w[i] = float(d) * (nib_i - 8)                                   */
/*   IQ4_NL: w[i] = float(d) * kv[nib_i]                                      */
/* with nib_i the low nibble of byte 2+i for i < 16, the high nibble of byte */
/* 2+(i-16) otherwise.                                                       */
/* ------------------------------------------------------------------------ */
#define OR_WT_IQ4XS 0
#define OR_WT_Q4_0  1
#define OR_WT_IQ4NL 2
#define OR_B18_BYTES 18
#define OR_B18_OFF_QS 2

/* Integer value of element i (0..31) of one 18-byte block. */
int oracle_b18_code(int wtype, const uint8_t* block, int i) {
    uint8_t byte = block[OR_B18_OFF_QS + (i % 16)];
    int nib = (i < 16) ? (byte & 0x0F) : (byte >> 4);
    return (wtype == OR_WT_Q4_0) ? nib - 8 : or_kvalues[nib];
}

/* fp32 scale of one 18-byte block: float(d). */
float oracle_b18_scale(const uint8_t* block) {
    return oracle_f16_to_f32((uint16_t)(block[0] | (block[1] << 8)));
}

/* Bytes of one weight row of K values in format wtype, or -1 if K does not
 * fit the format's block (256 for IQ4_XS, 32 for the others). */
int64_t oracle_row_bytes(int wtype, int64_t K) {
    if (wtype == OR_WT_IQ4XS) return (K % OR_QK) ? -1 : (K / OR_QK) * OR_BLOCK_BYTES;
    if (wtype == OR_WT_Q4_0 || wtype == OR_WT_IQ4NL)
        return (K % OR_SUB) ? -1 : (K / OR_SUB) * OR_B18_BYTES;
    return -1;
}

/* Code of element i and fp32 scale of 32-weight block c of row n. */
static int or_wt_code(int wtype, const uint8_t* w, int64_t row_bytes, int64_t n, int64_t c,
                      int i) {
    if (wtype == OR_WT_IQ4XS) {
        const uint8_t* blk = w + n * row_bytes + (c / OR_NSUB) * OR_BLOCK_BYTES;
        return oracle_iq4xs_code(blk, (int)(c % OR_NSUB) * OR_SUB + i);
    }
    return oracle_b18_code(wtype, w + n * row_bytes + c * OR_B18_BYTES, i);
}
static float or_wt_scale(int wtype, const uint8_t* w, int64_t row_bytes, int64_t n, int64_t c) {
    if (wtype == OR_WT_IQ4XS) {
        const uint8_t* blk = w + n * row_bytes + (c / OR_NSUB) * OR_BLOCK_BYTES;
        return oracle_iq4xs_subblock_scale(blk, (int)(c % OR_NSUB));
    }
    return oracle_b18_scale(w + n * row_bytes + c * OR_B18_BYTES);
}

/* Decode any format to doubles, out[n*K + k]. */
int oracle_decode_wt(int wtype, const uint8_t* w, int64_t N, int64_t K, double* out) {
    int64_t rb = oracle_row_bytes(wtype, K);
    if (rb < 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int64_t c = k / OR_SUB;
            out[n * K + k] = (double)or_wt_scale(wtype, w, rb, n, c) *
                             (double)or_wt_code(wtype, w, rb, n, c, (int)(k % OR_SUB));
        }
    return 0;
}

/* Dequantize any format to fp32 (exact) and, if out_bf16, to bfloat16 (RNE). */
int oracle_dequantize_wt(int wtype, const uint8_t* w, int64_t N, int64_t K, float* out_f32,
                         uint16_t* out_bf16) {
    int64_t rb = oracle_row_bytes(wtype, K);
    if (rb < 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int64_t c = k / OR_SUB;
            float v = or_wt_scale(wtype, w, rb, n, c) *
                      (float)or_wt_code(wtype, w, rb, n, c, (int)(k % OR_SUB));
            if (out_f32) out_f32[n * K + k] = v;
            if (out_bf16) out_bf16[n * K + k] = oracle_f32_to_bf16(v);
        }
    return 0;
}

typedef struct {
    int wtype;
    const uint8_t* w;
    int64_t row_bytes, N, K;
    const int8_t* qs;
    const uint16_t* d_h;
    int64_t M;
    double* y;
    int64_t n0, n1;
    int status;
} or_wt_job;

/* The same product as oracle_matmul, for any format: per 32-weight block an
 * exact integer dot P, then S_w * d_x * P accumulated in fp64 in block order. */
static void* or_matmul_wt_rows(void* arg) {
    or_wt_job* job = (or_wt_job*)arg;
    int64_t nblk = job->K / OR_SUB;
    for (int64_t n = job->n0; n < job->n1; ++n) {
        for (int64_t m = 0; m < job->M; ++m) {
            double acc = 0.0;
            for (int64_t c = 0; c < nblk; ++c) {
                int64_t P = 0;
                for (int i = 0; i < OR_SUB; ++i)
                    P += (int64_t)or_wt_code(job->wtype, job->w, job->row_bytes, n, c, i) *
                         (int64_t)job->qs[m * job->K + c * OR_SUB + i];
                if (P > 516128 || P < -516128) { job->status = -3; return NULL; }
                double sw = (double)or_wt_scale(job->wtype, job->w, job->row_bytes, n, c);
                double dx = (double)oracle_f16_to_f32(job->d_h[m * nblk + c]);
                acc += sw * dx * (double)P;
            }
            job->y[m * job->N + n] = acc;
        }
    }
    return NULL;
}

/* y[M][N] (double) for weights in format wtype; threads as oracle_matmul. */
int oracle_matmul_wt(int wtype, const uint8_t* w, int64_t N, int64_t K, const int8_t* qs,
                     const uint16_t* d_h, int64_t M, double* y, int nthreads) {
    int64_t rb = oracle_row_bytes(wtype, K);
    if (rb < 0 || N < 0 || M < 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N && N > 0) nthreads = (int)N;
    or_wt_job* jobs = (or_wt_job*)calloc((size_t)nthreads, sizeof(or_wt_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -4; }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        or_wt_job j = {wtype, w, rb, N, K, qs, d_h, M, y,
                       N * t / nthreads, N * (t + 1) / nthreads, 0};
        jobs[t] = j;
        if (nthreads == 1 || pthread_create(&th[t], NULL, or_matmul_wt_rows, &jobs[t]) != 0) {
            or_matmul_wt_rows(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        if (th[t]) pthread_join(th[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs);
    free(th);
    return status;
}
