/*
 * moe_oracle.c -- plain, slow CPU oracle for one routed quantized-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path loads this file; only the
 * tests, the package smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or constant generator with the CUDA library.
 *
 * Compiled with -O2 -ffp-contract=off (no silent FMA contraction): every float
 * operation below is the IEEE operation written, and fmaf() appears only where the
 * router's canonical summation order says "fused multiply-add".
 *
 * What it computes, and where each step comes from:
 *   - Q8_0 blocks (32 int8 + one fp16 scale, round half away from zero): the format
 *     the Xeon page runs ("Running Gemma 4 26B at 5 tokens/s on a 13-year-old Xeon
 *     without a GPU", amuse.peoplentools.com, opening summary and section "Compute
 *     paths broken in the non-AVX2 build"); the pages never spell out the block, so
 *     the widely used ggml convention is taken: d = amax/127, q = round(x/d).
 *   - NVFP4 (E2M1 values, one FP8-E4M3 scale per 16 consecutive values, one fp32
 *     scale per tensor) and the neuron-contiguous relayout of the down matrix:
 *     "Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU" (molayo1419.me),
 *     sections "The single most important number: bytes per token" and "How the
 *     engine works", steps 1 and 4.
 *   - Router + top-k + softmax over the selected logits, the permutation by expert
 *     (the grouping that an expert-indexed matmul presupposes), the fused gate/up
 *     with SwiGLU, the gateless ReLU^2 latent expert, the 16-neuron zero-group skip
 *     in the down projection, and the fixed-order combine: same Nemotron page, steps
 *     4 and section "How we check correctness" (per-(token, expert) buffers summed in
 *     a fixed order); Xeon page, section "A three-step fix", "Runtime graph fallback"
 *     (the [n_embd, 2*n_ff, n_experts] gate-first/up-second tensor split into two
 *     expert-indexed matmuls and a fused SiLU-multiply).
 *   - Per-channel int8 experts (one fp32 scale per output row): Inferentia page ("Squeezing
 *     a 26B MoE onto the cheapest Inferentia instance"), section "Wall 1: the memory math".
 *   - The activation-quantised Q8_0 path of the CPU engines (orc_layer_forward_ex with
 *     act_q8): each expert input quantised with the same Q8_0 codec, then Q8_0 x Q8_0
 *     block dots with exact integer code sums (Xeon page, "A three-step fix" and
 *     "Narrowing down the cause", which name the activation quantisers and the vector dot).
 *
 * Accumulation is fp64 throughout the expert path; quantisation decisions and router
 * logits are taken in fp32, the precision the method fixes for them.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_ACT_SWIGLU 0
#define ORC_ACT_RELU2 1
#define ORC_W_Q8_0 0
#define ORC_W_NVFP4 1
#define ORC_W_INT8PC 2

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (n >= 1); a no-op without OpenMP. */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------------------
 * Rounding to a small binary float format.
 *
 * A format with p significant bits (hidden bit included), smallest normal exponent
 * emin and largest finite value maxv.  The representable numbers near |x| are spaced
 * by quantum = 2^(max(floor(log2|x|), emin) - (p-1)); rounding to nearest-even is
 * rint(x / quantum) * quantum, computed exactly in double (division by a power of
 * two is exact, rint rounds ties to the even integer = even last significand bit).
 * ------------------------------------------------------------------------------------ */
static double round_to_format(double x, int p, int emin, double maxv, int saturate, int* overflow) {
    *overflow = 0;
    if (x == 0.0) return x;
    double a = fabs(x);
    int e;
    frexp(a, &e);           /* a = m * 2^e, m in [0.5, 1): floor(log2 a) = e - 1 */
    int ex = e - 1;
    if (ex < emin) ex = emin;
    double quantum = ldexp(1.0, ex - (p - 1));
    double r = rint(a / quantum) * quantum;
    if (r > maxv) {
        if (saturate) {
            r = maxv;
        } else {
            *overflow = 1;
            r = INFINITY;
        }
    }
    return x < 0 ? -r : r;
}

/* IEEE binary16: p = 11, emin = -14, max 65504; overflow rounds to infinity. */
uint16_t orc_f32_to_f16(float f) {
    int ovf;
    double r = round_to_format((double)f, 11, -14, 65504.0, 0, &ovf);
    uint16_t sign = signbit(r) ? 0x8000u : 0u;
    double a = fabs(r);
    if (ovf || isinf(a)) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < -14) { /* subnormal: a = frac * 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(a, 24));
    }
    uint16_t frac = (uint16_t)(ldexp(a, -ex) * 1024.0 - 1024.0);
    return (uint16_t)(sign | (uint16_t)((ex + 15) << 10) | frac);
}

double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (ex == 0) v = ldexp((double)frac, -24);
    else if (ex == 31) v = frac ? NAN : INFINITY;
    else v = ldexp(1024.0 + frac, ex - 25);
    return sign ? -v : v;
}

/* FP8 E4M3 (the "fn" variant: no infinities, 448 is the largest finite value):
 * p = 4, emin = -6, subnormal quantum 2^-9.  Saturating, as a block scale must be. */
uint8_t orc_f32_to_e4m3(float f) {
    int ovf;
    double r = round_to_format((double)f, 4, -6, 448.0, 1, &ovf);
    uint8_t sign = signbit(r) ? 0x80u : 0u;
    double a = fabs(r);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < -6) return (uint8_t)(sign | (uint8_t)ldexp(a, 9)); /* subnormal */
    uint8_t frac = (uint8_t)(ldexp(a, -ex) * 8.0 - 8.0);
    return (uint8_t)(sign | (uint8_t)((ex + 7) << 3) | frac);
}

double orc_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int ex = (b >> 3) & 0xf;
    int frac = b & 7;
    double v;
    if (ex == 0) v = ldexp((double)frac, -9);
    else if (ex == 15 && frac == 7) v = NAN;
    else v = ldexp(8.0 + frac, ex - 10);
    return sign ? -v : v;
}

/* FP4 E2M1: p = 2, emin = 0 (bias 1), magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
 * Saturating.  A zero result is always coded +0 (code 0x0). */
uint8_t orc_f32_to_e2m1(float f) {
    int ovf;
    double r = round_to_format((double)f, 2, 0, 6.0, 1, &ovf);
    double a = fabs(r);
    if (a == 0.0) return 0;
    uint8_t sign = r < 0 ? 0x8u : 0u;
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < 0) return (uint8_t)(sign | 0x1u); /* 0.5, the only subnormal */
    uint8_t frac = (uint8_t)(ldexp(a, -ex) * 2.0 - 2.0);
    return (uint8_t)(sign | (uint8_t)((ex + 1) << 1) | frac);
}

double orc_e2m1_to_f64(uint8_t c) {
    int sign = (c >> 3) & 1;
    int ex = (c >> 1) & 3;
    int frac = c & 1;
    double v = (ex == 0) ? 0.5 * frac : ldexp(2.0 + frac, ex - 2);
    return sign ? -v : v;
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------------------
 * Byte sizes.
 * ------------------------------------------------------------------------------------ */
int64_t orc_q8_0_bytes(int64_t rows, int64_t cols) { return rows * (cols / 32) * 34; }
int64_t orc_nvfp4_bytes(int64_t rows, int64_t cols) { return rows * cols / 2 + rows * cols / 16; }
int64_t orc_int8pc_bytes(int64_t rows, int64_t cols) { return rows * cols + 4 * rows; }

/* ------------------------------------------------------------------------------------
 * Q8_0.  Canonical byte layout: blocks in row-major order, each block = fp16 scale
 * (little endian) followed by 32 int8 codes.
 *   d = amax / 127 (fp32);  id = d != 0 ? 1/d : 0 (fp32);  q = roundf(x * id)
 * The scale is stored as fp16(d); the codes use the fp32 d.  roundf rounds half away
 * from zero.
 * ------------------------------------------------------------------------------------ */
void orc_q8_0_quantize(const float* src, int64_t rows, int64_t cols, uint8_t* dst) {
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* x = src + r * cols + b * 32;
            uint8_t* blk = dst + (r * nb + b) * 34;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(x[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            float id = (d != 0.0f) ? 1.0f / d : 0.0f;
            uint16_t dh = orc_f32_to_f16(d);
            blk[0] = (uint8_t)(dh & 0xff);
            blk[1] = (uint8_t)(dh >> 8);
            for (int i = 0; i < 32; ++i) {
                float v = x[i] * id;
                blk[2 + i] = (uint8_t)(int8_t)roundf(v);
            }
        }
    }
}

/* Exact dequantisation: q * fp16(d) in double. */
void orc_q8_0_dequant(const uint8_t* q, int64_t rows, int64_t cols, double* out) {
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* blk = q + (r * nb + b) * 34;
            double d = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int i = 0; i < 32; ++i) out[r * cols + b * 32 + i] = (double)(int8_t)blk[2 + i] * d;
        }
    }
}

/* ------------------------------------------------------------------------------------
 * Per-channel int8 (Inferentia page, "Wall 1: the memory math": the experts quantised
 * to int8 with one scale per output channel, numerically on par with fp32 for that model).
 * The page gives no recipe, so the plainest one is taken:
 *   s = amax(row) / 127 (fp32, one per row); q = roundf(x / s), half away from zero;
 *   an all-zero row has s = 0 and q = 0.
 * Bytes: the rows x cols codes row-major, then the rows' fp32 scales (little endian).
 * ------------------------------------------------------------------------------------ */
void orc_int8pc_quantize(const float* src, int64_t rows, int64_t cols, uint8_t* dst) {
    uint8_t* sb = dst + rows * cols;   /* the scales: byte offsets, no alignment assumed */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* x = src + r * cols;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            const float a = fabsf(x[c]);
            if (a > amax) amax = a;
        }
        const float sc = amax / 127.0f;
        for (int64_t c = 0; c < cols; ++c)
            dst[r * cols + c] = (uint8_t)(int8_t)(sc != 0.0f ? roundf(x[c] / sc) : 0.0f);
        memcpy(sb + 4 * r, &sc, sizeof(float));
    }
}

/* Exact dequantisation: q * s in double. */
void orc_int8pc_dequant(const uint8_t* q, int64_t rows, int64_t cols, double* out) {
    const uint8_t* sb = q + rows * cols;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float sc;
        memcpy(&sc, sb + 4 * r, sizeof(float));
        for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = (double)(int8_t)q[r * cols + c] * (double)sc;
    }
}

/* Q8_0 x Q8_0 dot product of two rows of nb canonical blocks each: the CPU engines'
 * activation-quantised path.  The Xeon page names its pieces: the Q8_0 / Q8_1 activation
 * quantisers its non-AVX2 fix rewrites (section "A three-step fix") and the Q8_0 x Q8_0
 * vector dot it checks (section "Narrowing down the cause").  It does not spell out the
 * arithmetic, so the plain reading is taken.  Per block, the 32 code products are summed
 * exactly as integers and scaled by both fp16 scales; the blocks are summed in fp64.  Each
 * block term is exact in fp64: at most 11 + 11 + 19 significant bits. */
double orc_q8_0_vec_dot(const uint8_t* a, const uint8_t* b, int64_t nb) {
    double acc = 0.0;
    for (int64_t i = 0; i < nb; ++i) {
        const uint8_t* ba = a + i * 34;
        const uint8_t* bb = b + i * 34;
        int32_t s = 0;
        for (int j = 0; j < 32; ++j) s += (int32_t)(int8_t)ba[2 + j] * (int32_t)(int8_t)bb[2 + j];
        const double da = orc_f16_to_f64((uint16_t)(ba[0] | (ba[1] << 8)));
        const double db = orc_f16_to_f64((uint16_t)(bb[0] | (bb[1] << 8)));
        acc += da * db * (double)s;
    }
    return acc;
}

/* Device layout for per-channel int8: a byte permutation of the canonical bytes.  First the
 * rows' fp32 scales (4 bytes each, rows in order), then panel b (columns 32b..32b+31): the 32
 * codes of every row (rows in order, 32 bytes each).  dir = +1 maps canonical -> device,
 * dir = -1 maps device -> canonical. */
void orc_int8pc_permute(const uint8_t* src, int64_t rows, int64_t cols, int dir, uint8_t* dst) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const int64_t canon = r * cols + c;
            const int64_t dev = 4 * rows + (c / 32) * (rows * 32) + r * 32 + (c % 32);
            if (dir > 0) dst[dev] = src[canon];
            else dst[canon] = src[dev];
        }
        for (int64_t i = 0; i < 4; ++i) {
            const int64_t canon = rows * cols + 4 * r + i, dev = 4 * r + i;
            if (dir > 0) dst[dev] = src[canon];
            else dst[canon] = src[dev];
        }
    }
}

/* Device layout for Q8_0: a byte permutation of the canonical blocks, panel by panel
 * along K.  Panel b (columns 32b..32b+31): the 32 codes of every row (rows in order,
 * 32 bytes each), then the fp16 scales of every row (2 bytes each).  dir = +1 maps
 * canonical -> device, dir = -1 maps device -> canonical. */
void orc_q8_0_permute(const uint8_t* src, int64_t rows, int64_t cols, int dir, uint8_t* dst) {
    const int64_t nb = cols / 32;
    for (int64_t b = 0; b < nb; ++b) {
        const int64_t panel = b * rows * 34;
        for (int64_t r = 0; r < rows; ++r) {
            const int64_t canon = (r * nb + b) * 34;
            const int64_t dev_q = panel + r * 32;
            const int64_t dev_s = panel + rows * 32 + r * 2;
            if (dir > 0) {
                memcpy(dst + dev_q, src + canon + 2, 32);
                memcpy(dst + dev_s, src + canon, 2);
            } else {
                memcpy(dst + canon + 2, src + dev_q, 32);
                memcpy(dst + canon, src + dev_s, 2);
            }
        }
    }
}

/* ------------------------------------------------------------------------------------
 * NVFP4.  Per matrix [rows, cols]:
 *   s_t = amax(|x|) / (6 * 448)  (fp32; s_t = 1 when the matrix is all zero)
 *   per 16 consecutive values along a row: sb = E4M3(amax_b / (6 * s_t))
 *   per value: q = E2M1(x / (dec(sb) * s_t)), q = 0 when dec(sb) = 0
 * Canonical layout: all codes row-major, two per byte (even element in the low
 * nibble), then all block scales row-major (one byte each).
 * ------------------------------------------------------------------------------------ */
float orc_nvfp4_tensor_scale(const float* src, int64_t rows, int64_t cols) {
    float amax = 0.0f;
    for (int64_t i = 0; i < rows * cols; ++i) {
        float a = fabsf(src[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) return 1.0f;
    return amax / 2688.0f;
}

void orc_nvfp4_quantize(const float* src, int64_t rows, int64_t cols, uint8_t* dst, float* tscale_out) {
    const float st = orc_nvfp4_tensor_scale(src, rows, cols);
    const int64_t nb = cols / 16;
    uint8_t* vals = dst;
    uint8_t* scales = dst + rows * cols / 2;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* x = src + r * cols + b * 16;
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(x[i]);
                if (a > amax) amax = a;
            }
            float six_st = 6.0f * st;
            uint8_t sb = orc_f32_to_e4m3(amax / six_st);
            scales[r * nb + b] = sb;
            float dec = (float)orc_e4m3_to_f64(sb);
            float denom = dec * st;
            for (int i = 0; i < 16; i += 2) {
                uint8_t lo = (dec == 0.0f) ? 0 : orc_f32_to_e2m1(x[i] / denom);
                uint8_t hi = (dec == 0.0f) ? 0 : orc_f32_to_e2m1(x[i + 1] / denom);
                vals[(r * cols + b * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    *tscale_out = st;
}

/* Exact dequantisation of the canonical layout: e2m1 * e4m3 * s_t in double. */
void orc_nvfp4_dequant(const uint8_t* q, int64_t rows, int64_t cols, float tscale, double* out) {
    const uint8_t* vals = q;
    const uint8_t* scales = q + rows * cols / 2;
    const int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = vals[(r * cols + c) / 2];
            uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xf);
            double s = orc_e4m3_to_f64(scales[r * nb + c / 16]);
            out[r * cols + c] = orc_e2m1_to_f64(code) * s * (double)tscale;
        }
    }
}

/* Device layout for NVFP4 (gate/up and up matrices): panels of 64 columns.  Panel P:
 * the 32 code bytes of every row (rows in order), then the 4 block-scale bytes of
 * every row.  dir = +1 canonical -> device, -1 device -> canonical. */
void orc_nvfp4_permute_panels(const uint8_t* src, int64_t rows, int64_t cols, int dir, uint8_t* dst) {
    const int64_t np = cols / 64;
    const int64_t scale_base = rows * cols / 2;
    for (int64_t p = 0; p < np; ++p) {
        const int64_t panel = p * rows * 36;
        for (int64_t r = 0; r < rows; ++r) {
            const int64_t cv = r * cols / 2 + p * 32;
            const int64_t cs = scale_base + r * (cols / 16) + p * 4;
            const int64_t dv = panel + r * 32;
            const int64_t ds = panel + rows * 32 + r * 4;
            if (dir > 0) {
                memcpy(dst + dv, src + cv, 32);
                memcpy(dst + ds, src + cs, 4);
            } else {
                memcpy(dst + cv, src + dv, 32);
                memcpy(dst + cs, src + ds, 4);
            }
        }
    }
}

/* Neuron-contiguous relayout of an NVFP4 down matrix [rows = d, cols = f]
 * (Nemotron page, "How the engine works", step 4: each neuron's 4-bit values
 * contiguous, scales grouped by 16 neurons; a pure byte permutation of equal size).
 * For each group g of 16 neurons (columns 16g..16g+15): for each neuron n of the
 * group, rows/2 bytes holding the codes of rows 0..rows-1 of column n (row r in the
 * low nibble of byte r/2 when r is even, the high nibble when odd); then the rows
 * block-scale bytes sb[r][g], r = 0..rows-1.  dir = +1 canonical -> neuron layout,
 * -1 neuron layout -> canonical. */
void orc_nvfp4_permute_neuron(const uint8_t* src, int64_t rows, int64_t cols, int dir, uint8_t* dst) {
    const int64_t ng = cols / 16;
    const int64_t scale_base = rows * cols / 2;
    const int64_t rec = 16 * (rows / 2) + rows;
    memset(dst, 0, (size_t)orc_nvfp4_bytes(rows, cols));
    for (int64_t g = 0; g < ng; ++g) {
        const int64_t base = g * rec;
        for (int64_t j = 0; j < 16; ++j) {
            const int64_t n = 16 * g + j;
            for (int64_t r = 0; r < rows; ++r) {
                /* canonical nibble of (r, n) */
                const int64_t cbyte = (r * cols + n) / 2;
                const int cshift = (int)((n & 1) * 4);
                /* neuron-layout nibble of (r, n) */
                const int64_t nbyte = base + j * (rows / 2) + r / 2;
                const int nshift = (int)((r & 1) * 4);
                if (dir > 0) {
                    uint8_t code = (uint8_t)((src[cbyte] >> cshift) & 0xf);
                    dst[nbyte] = (uint8_t)(dst[nbyte] | (code << nshift));
                } else {
                    uint8_t code = (uint8_t)((src[nbyte] >> nshift) & 0xf);
                    dst[cbyte] = (uint8_t)(dst[cbyte] | (code << cshift));
                }
            }
        }
        for (int64_t r = 0; r < rows; ++r) {
            const int64_t cs = scale_base + r * ng + g;
            const int64_t ns = base + 16 * (rows / 2) + r;
            if (dir > 0) dst[ns] = src[cs];
            else dst[cs] = src[ns];
        }
    }
}

/* ------------------------------------------------------------------------------------
 * Router.  logit[t][e] is an fp32 dot product of x[t][:] with W[:][e] (W is [d][E],
 * row-major) in one fixed ("canonical") order, so that every implementation rounds
 * identically:
 *   256 partial sums: s_l = 0, then s_l = fmaf(x[i], W[i][e], s_l) for
 *   i = l, l+256, l+512, ... < d in increasing i;
 *   then a halving tree: for h = 128, 64, ..., 1: s_l = s_l + s_{l+h} for l < h.
 *   The logit is s_0.
 * The pages do not state a summation order; this one is chosen for parallel hardware
 * and documented as the reading.
 * ------------------------------------------------------------------------------------ */
#define ORC_ROUTER_PARTIALS 256

static float router_dot(const float* x, const float* W, int64_t d, int64_t E, int64_t e) {
    float s[ORC_ROUTER_PARTIALS];
    for (int l = 0; l < ORC_ROUTER_PARTIALS; ++l) {
        float acc = 0.0f;
        for (int64_t i = l; i < d; i += ORC_ROUTER_PARTIALS) acc = fmaf(x[i], W[i * E + e], acc);
        s[l] = acc;
    }
    for (int h = ORC_ROUTER_PARTIALS / 2; h >= 1; h /= 2)
        for (int l = 0; l < h; ++l) s[l] = s[l] + s[l + h];
    return s[0];
}

/* x is fp32 (xt = 0) or bf16 bits (xt = 1), [T][d]. */
static void load_x_row(const void* x, int xt, int64_t d, int64_t t, float* row) {
    if (xt == 0) {
        memcpy(row, (const float*)x + t * d, (size_t)d * sizeof(float));
    } else {
        const uint16_t* xb = (const uint16_t*)x + t * d;
        for (int64_t i = 0; i < d; ++i) row[i] = bf16_to_f32(xb[i]);
    }
}

void orc_router_logits(const void* x, int xt, const float* W, int64_t T, int64_t d, int64_t E, float* logits) {
#pragma omp parallel
    {
        float* row = (float*)malloc((size_t)d * sizeof(float));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            load_x_row(x, xt, d, t, row);
            for (int64_t e = 0; e < E; ++e) logits[t * E + e] = router_dot(row, W, d, E, e);
        }
        free(row);
    }
}

/* Top-k by repeated selection: each round takes the largest remaining logit, the
 * lower expert index winning ties; slots are filled in selection order.  The
 * combine weights are a softmax over the k selected logits (computed in double with
 * the maximum, slot 0, subtracted; the sum runs in slot order). */
void orc_topk_softmax(const float* logits, int64_t T, int64_t E, int k, int32_t* idx, double* w) {
#pragma omp parallel
    {
        unsigned char* taken = (unsigned char*)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const float* l = logits + t * E;
            memset(taken, 0, (size_t)E);
            for (int j = 0; j < k; ++j) {
                int64_t best = -1;
                for (int64_t e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower index on ties */
                }
                taken[best] = 1;
                idx[t * k + j] = (int32_t)best;
            }
            double m = (double)l[idx[t * k]];
            double sum = 0.0;
            for (int j = 0; j < k; ++j) sum += exp((double)l[idx[t * k + j]] - m);
            for (int j = 0; j < k; ++j) w[t * k + j] = exp((double)l[idx[t * k + j]] - m) / sum;
        }
        free(taken);
    }
}

/* Stable counting sort of the T*k (token, slot) pairs by expert.  Pair p = t*k + j.
 * offsets[E+1]: exclusive prefix sum of the per-expert counts.  perm[r] = the pair at
 * sorted position r (pairs of one expert keep increasing p).  pos[p] = the sorted
 * position of pair p. */
void orc_permute(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* offsets, int32_t* perm, int32_t* pos) {
    const int64_t P = T * k;
    int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t p = 0; p < P; ++p) cnt[idx[p]]++;
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + (int32_t)cnt[e];
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t p = 0; p < P; ++p) {
        const int64_t e = idx[p];
        const int64_t r = offsets[e] + fill[e]++;
        perm[r] = (int32_t)p;
        pos[p] = (int32_t)r;
    }
    free(cnt);
    free(fill);
}

/* ------------------------------------------------------------------------------------
 * Expert arithmetic (fp64).
 * ------------------------------------------------------------------------------------ */
static void dequant_matrix(int wfmt, const uint8_t* q, int64_t rows, int64_t cols, float tscale, double* out) {
    if (wfmt == ORC_W_Q8_0) orc_q8_0_dequant(q, rows, cols, out);
    else if (wfmt == ORC_W_INT8PC) orc_int8pc_dequant(q, rows, cols, out);
    else orc_nvfp4_dequant(q, rows, cols, tscale, out);
}

/* Expert-indexed matmul on an already-dequantised stack of matrices:
 * for each (token t, slot j): out[t][j][r] = sum_c W[ids[t][j]][row0 + r][c] * x[t][c],
 * r < nrows, W[e] being [ld_rows][cols].  The rows row0..row0+nrows-1 are a view, as a
 * slice of the fused gate/up tensor would be. */
void orc_mul_mat_id(const double* const* W, int64_t ld_rows, int64_t cols, int64_t row0, int64_t nrows,
                    const double* x, int64_t T, int k, const int32_t* ids, double* out) {
    (void)ld_rows;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < T * k; ++p) {
        const int64_t t = p / k;
        const double* We = W[ids[p]];
        for (int64_t r = 0; r < nrows; ++r) {
            double acc = 0.0;
            for (int64_t c = 0; c < cols; ++c) acc += We[(row0 + r) * cols + c] * x[t * cols + c];
            out[p * nrows + r] = acc;
        }
    }
}

double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* SiLU(gate) * up, elementwise. */
void orc_fused_mul_silu(const double* gate, const double* up, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_silu(gate[i]) * up[i];
}

/* One expert, one token: h = act(W_gu x) over the fused rows (SwiGLU: rows 0..f-1 are
 * the gate, f..2f-1 the up projection; ReLU^2: rows 0..f-1 are the up projection). */
static void expert_gate_up(int act, const double* Wgu, int64_t f, int64_t d, const double* x, double* h) {
    if (act == ORC_ACT_SWIGLU) {
        for (int64_t n = 0; n < f; ++n) {
            double g = 0.0, u = 0.0;
            const double* wg = Wgu + n * d;
            const double* wu = Wgu + (f + n) * d;
            for (int64_t c = 0; c < d; ++c) {
                g += wg[c] * x[c];
                u += wu[c] * x[c];
            }
            h[n] = orc_silu(g) * u;
        }
    } else {
        for (int64_t n = 0; n < f; ++n) {
            double z = 0.0;
            const double* wu = Wgu + n * d;
            for (int64_t c = 0; c < d; ++c) z += wu[c] * x[c];
            double r = z > 0.0 ? z : 0.0;
            h[n] = r * r;
        }
    }
}

/* Down projection y = W_down h, W_down [d][f].  sparse = 1 skips every 16-neuron group
 * whose h values are all exactly zero (Nemotron page, step 4); the skipped terms are
 * exact zeros, so both forms agree. */
static void expert_down(const double* Wd, int64_t d, int64_t f, const double* h, int sparse, double* y) {
    const int64_t ng = f / 16;
    unsigned char* active = (unsigned char*)malloc((size_t)ng);
    for (int64_t g = 0; g < ng; ++g) {
        active[g] = 0;
        for (int64_t n = 16 * g; n < 16 * g + 16; ++n)
            if (h[n] != 0.0) active[g] = 1;
    }
    for (int64_t r = 0; r < d; ++r) {
        double acc = 0.0;
        for (int64_t g = 0; g < ng; ++g) {
            if (sparse && !active[g]) continue;
            for (int64_t n = 16 * g; n < 16 * g + 16; ++n) acc += Wd[r * f + n] * h[n];
        }
        y[r] = acc;
    }
    free(active);
}

/* The activation-quantised expert (Q8_0 weights only).  The expert's input vector (x for
 * gate.up; h, held in fp32, for down) is quantised with the same Q8_0 block codec as the
 * weights.  Every weight row is then dotted with it by orc_q8_0_vec_dot.  An all-zero
 * 16-neuron group of h quantises to zero codes, so the down projection needs no separate
 * skip: its terms are exact zeros. */
static void expert_q8act(int act, const uint8_t* Wgu, const uint8_t* Wd, int64_t f, int64_t d, const float* x,
                         double* h, double* y) {
    const int64_t nbd = d / 32, nbf = f / 32;
    uint8_t* xq = (uint8_t*)malloc((size_t)(nbd * 34));
    uint8_t* hq = (uint8_t*)malloc((size_t)(nbf * 34));
    float* hf = (float*)malloc((size_t)f * sizeof(float));
    orc_q8_0_quantize(x, 1, d, xq);
    for (int64_t n = 0; n < f; ++n) {
        if (act == ORC_ACT_SWIGLU) {
            const double g = orc_q8_0_vec_dot(Wgu + n * nbd * 34, xq, nbd);
            const double u = orc_q8_0_vec_dot(Wgu + (f + n) * nbd * 34, xq, nbd);
            h[n] = orc_silu(g) * u;
        } else {
            const double z = orc_q8_0_vec_dot(Wgu + n * nbd * 34, xq, nbd);
            const double r = z > 0.0 ? z : 0.0;
            h[n] = r * r;
        }
        hf[n] = (float)h[n];
    }
    orc_q8_0_quantize(hf, 1, f, hq);
    for (int64_t r = 0; r < d; ++r) y[r] = orc_q8_0_vec_dot(Wd + r * nbf * 34, hq, nbf);
    free(xq);
    free(hq);
    free(hf);
}

/* ------------------------------------------------------------------------------------
 * The layer.
 * ------------------------------------------------------------------------------------ */
typedef struct {
    int64_t d, f, E;
    int k, act, wfmt;
    const float* router_w;          /* [d][E] fp32 */
    const uint8_t* const* gate_up;  /* [E] canonical bytes of [rows_gu][d]; NULL where not needed */
    const uint8_t* const* down;     /* [E] canonical bytes of [d][f] */
    const float* gate_up_tscale;    /* [E], NVFP4 only */
    const float* down_tscale;       /* [E], NVFP4 only */
} orc_layer;

/* Outputs (each optional except out):
 *   logits [T][E] fp32, idx [T][k], w [T][k] (double), offsets [E+1], perm [T*k],
 *   pos [T*k], h [T*k][f] in pair order, y [T*k][d] in pair order, out [T][d] double.
 * idx_in / w_in: precomputed routing (both or neither); the router is skipped.
 * sparse_down: 1 = skip all-zero 16-neuron groups, 0 = dense down.
 * act_q8: 1 = the activation-quantised expert path (expert_q8act; Q8_0 weights, f a
 * multiple of 32), 0 = activations used as they are.
 * Returns 0, -1 when an expert needed by the routing has no weights, -2 when act_q8 is
 * asked of another format or shape. */
int orc_layer_forward_ex(const orc_layer* L, const void* x, int xt, int64_t T, const int32_t* idx_in,
                         const float* w_in, int sparse_down, int act_q8, float* logits_out, int32_t* idx_out,
                         double* w_out, int32_t* offsets_out, int32_t* perm_out, int32_t* pos_out, double* h_out,
                         double* y_out, double* out) {
    const int64_t d = L->d, f = L->f, E = L->E;
    const int k = L->k;
    const int64_t P = T * k;
    const int64_t rows_gu = (L->act == ORC_ACT_SWIGLU) ? 2 * f : f;
    if (act_q8 && (L->wfmt != ORC_W_Q8_0 || f % 32 != 0)) return -2;

    int32_t* idx = idx_out ? idx_out : (int32_t*)malloc((size_t)P * sizeof(int32_t));
    double* w = w_out ? w_out : (double*)malloc((size_t)P * sizeof(double));
    if (idx_in) {
        memcpy(idx, idx_in, (size_t)P * sizeof(int32_t));
        for (int64_t p = 0; p < P; ++p) w[p] = (double)w_in[p];
    } else {
        float* logits = logits_out ? logits_out : (float*)malloc((size_t)(T * E) * sizeof(float));
        orc_router_logits(x, xt, L->router_w, T, d, E, logits);
        orc_topk_softmax(logits, T, E, k, idx, w);
        if (!logits_out) free(logits);
    }
    int32_t* offsets = offsets_out ? offsets_out : (int32_t*)malloc((size_t)(E + 1) * sizeof(int32_t));
    int32_t* perm = perm_out ? perm_out : (int32_t*)malloc((size_t)P * sizeof(int32_t));
    int32_t* pos = pos_out ? pos_out : (int32_t*)malloc((size_t)P * sizeof(int32_t));
    orc_permute(idx, T, k, E, offsets, perm, pos);

    /* Check availability of the weights the routing needs. */
    for (int64_t p = 0; p < P; ++p)
        if (!L->gate_up[idx[p]] || !L->down[idx[p]]) return -1;

    /* Expert outputs, indexed by pair p, computed one expert at a time. */
    double* y = (double*)malloc((size_t)(P * d) * sizeof(double));
    double* hbuf = (double*)malloc((size_t)(P * f) * sizeof(double));
    double* Wgu = (double*)malloc((size_t)(rows_gu * d) * sizeof(double));
    double* Wd = (double*)malloc((size_t)(d * f) * sizeof(double));
    for (int64_t e = 0; e < E; ++e) {
        const int64_t r0 = offsets[e], r1 = offsets[e + 1];
        if (r0 == r1) continue;
        if (!act_q8) {
            dequant_matrix(L->wfmt, L->gate_up[e], rows_gu, d, L->gate_up_tscale ? L->gate_up_tscale[e] : 1.0f, Wgu);
            dequant_matrix(L->wfmt, L->down[e], d, f, L->down_tscale ? L->down_tscale[e] : 1.0f, Wd);
        }
#pragma omp parallel
        {
            float* xrow = (float*)malloc((size_t)d * sizeof(float));
            double* xd = (double*)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(static)
            for (int64_t r = r0; r < r1; ++r) {
                const int64_t p = perm[r];
                const int64_t t = p / k;
                load_x_row(x, xt, d, t, xrow);
                double* h = hbuf + p * f;
                if (act_q8) {
                    expert_q8act(L->act, L->gate_up[e], L->down[e], f, d, xrow, h, y + p * d);
                    continue;
                }
                for (int64_t c = 0; c < d; ++c) xd[c] = (double)xrow[c];
                expert_gate_up(L->act, Wgu, f, d, xd, h);
                expert_down(Wd, d, f, h, sparse_down, y + p * d);
            }
            free(xrow);
            free(xd);
        }
    }
    free(Wgu);
    free(Wd);

    /* Combine: out[t] = sum over slots j = 0..k-1, in slot order, of w[t][j] * y[pair]. */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) acc += w[t * k + j] * y[(t * k + j) * d + c];
            out[t * d + c] = acc;
        }
    }
    if (h_out) memcpy(h_out, hbuf, (size_t)(P * f) * sizeof(double));
    if (y_out) memcpy(y_out, y, (size_t)(P * d) * sizeof(double));
    free(y);
    free(hbuf);
    if (!idx_out) free(idx);
    if (!w_out) free(w);
    if (!offsets_out) free(offsets);
    if (!perm_out) free(perm);
    if (!pos_out) free(pos);
    return 0;
}

int orc_layer_forward(const orc_layer* L, const void* x, int xt, int64_t T, const int32_t* idx_in,
                      const float* w_in, int sparse_down, float* logits_out, int32_t* idx_out, double* w_out,
                      int32_t* offsets_out, int32_t* perm_out, int32_t* pos_out, double* h_out, double* y_out,
                      double* out) {
    return orc_layer_forward_ex(L, x, xt, T, idx_in, w_in, sparse_down, 0, logits_out, idx_out, w_out, offsets_out,
                                perm_out, pos_out, h_out, y_out, out);
}

/* The "DenseExperts" form (Inferentia page, "Honest caveats"): every expert is
 * evaluated for every token and weighted by wfull[t][e] (zero off the selected set),
 * summed in expert order.  Equal in value to the routed layer. */
void orc_layer_forward_dense_experts(const orc_layer* L, const void* x, int xt, int64_t T, const double* wfull,
                                     double* out) {
    const int64_t d = L->d, f = L->f, E = L->E;
    const int64_t rows_gu = (L->act == ORC_ACT_SWIGLU) ? 2 * f : f;
    double* Wgu = (double*)malloc((size_t)(rows_gu * d) * sizeof(double));
    double* Wd = (double*)malloc((size_t)(d * f) * sizeof(double));
    double* h = (double*)malloc((size_t)f * sizeof(double));
    double* y = (double*)malloc((size_t)d * sizeof(double));
    float* xrow = (float*)malloc((size_t)d * sizeof(float));
    double* xd = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t i = 0; i < T * d; ++i) out[i] = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        dequant_matrix(L->wfmt, L->gate_up[e], rows_gu, d, L->gate_up_tscale ? L->gate_up_tscale[e] : 1.0f, Wgu);
        dequant_matrix(L->wfmt, L->down[e], d, f, L->down_tscale ? L->down_tscale[e] : 1.0f, Wd);
        for (int64_t t = 0; t < T; ++t) {
            load_x_row(x, xt, d, t, xrow);
            for (int64_t c = 0; c < d; ++c) xd[c] = (double)xrow[c];
            expert_gate_up(L->act, Wgu, f, d, xd, h);
            expert_down(Wd, d, f, h, 0, y);
            for (int64_t c = 0; c < d; ++c) out[t * d + c] += wfull[t * E + e] * y[c];
        }
    }
    free(Wgu);
    free(Wd);
    free(h);
    free(y);
    free(xrow);
    free(xd);
}
