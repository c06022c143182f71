/*
 * KVarN CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision restatement of what the KVarN group seal and
 * the decode attention over sealed groups compute. It exists to check the CUDA
 * library; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it. It shares no code, header or table with the CUDA path.
 *
 * Sources (page title, section):
 *  - fig1.dev "KVarN: Variance-Normalized KV-Cache Quantization ...", "What it is":
 *    Hadamard rotation over channels, then Sinkhorn-style variance normalisation
 *    over both the token and the channel axis, then round-to-nearest.
 *  - anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", section 1:
 *    rotation per head on post-RoPE K and V; query rotated by the same matrix;
 *    attention in the rotated frame; output rotated back once per token;
 *    16 Sinkhorn iterations.
 *  - same page, section 2.1: first 128 tokens exact; groups of 128 tokens
 *    quantised when their last token arrives; payload stored with its scale
 *    metadata; the partial newest group stays exact.
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes of the repository):
 *  - H is the Sylvester Hadamard matrix scaled by 1/sqrt(d), no random signs.
 *  - "unit variance" is unit mean square (uncentred RMS), because the
 *    normalisation only rescales.
 *  - one Sinkhorn iteration = a token-axis step followed by a channel-axis step;
 *    a zero row or column keeps its factor (divides by 1).
 *  - stored scales: token scale a and channel scale c in fp16 (round to nearest
 *    even, saturating at 65504); one asymmetric grid (min m, step delta, both fp32)
 *    for the whole normalised group matrix.
 *  - codes: round half to even, clamped to [0, 2^b - 1].
 *  - record layout: delta f32 | m f32 | 8 zero bytes | a[T] f16 | c[d] f16 | codes;
 *    K codes token-major, V codes channel-major, packed LSB first into
 *    little-endian 32-bit words.
 *
 * Parity status: every function below is pinned by the tests under tests/
 * (closed forms, invariants, brute force, library routines); none is pinned to a
 * worked numeric example from the pages, which print none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16 <-> binary64, written from the format's definition:      */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                   */
/* ------------------------------------------------------------------------- */
double kvo_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 value, ties to even. Overflow goes to
 * +-infinity when saturate == 0, else to +-65504. */
static uint16_t half_from_double(double x, int saturate) {
    if (isnan(x)) return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    /* Find the binade: ax = m * 2^e with 1 <= m < 2. */
    int e2;
    double m = frexp(ax, &e2); /* ax = m * 2^e2, 0.5 <= m < 1 */
    int e = e2 - 1;            /* ax = (2m) * 2^e */
    double quantum;            /* spacing of representable halves near ax */
    if (e < -14) {
        quantum = ldexp(1.0, -24); /* subnormal spacing */
    } else {
        quantum = ldexp(1.0, e - 10);
    }
    double q = ax / quantum;           /* exact: division by a power of two */
    double r = nearbyint(q);           /* default rounding mode: ties to even */
    double rounded = r * quantum;
    if (rounded > 65504.0) {
        return saturate ? (uint16_t)(sign | 0x7bff) : (uint16_t)(sign | 0x7c00);
    }
    /* encode rounded */
    if (rounded < ldexp(1.0, -14)) {
        /* subnormal (or rounded up to the smallest normal, handled below) */
        uint32_t f = (uint32_t)(rounded / ldexp(1.0, -24));
        return (uint16_t)(sign | f); /* f == 1024 encodes 2^-14 correctly */
    }
    int re2;
    double rm = frexp(rounded, &re2);
    int re = re2 - 1;
    uint32_t frac = (uint32_t)((2.0 * rm - 1.0) * 1024.0);
    return (uint16_t)(sign | ((uint32_t)(re + 15) << 10) | frac);
}

uint16_t kvo_double_to_half(double x) { return half_from_double(x, 0); }
uint16_t kvo_double_to_half_sat(double x) { return half_from_double(x, 1); }

/* ------------------------------------------------------------------------- */
/* Rotation (fig1.dev "What it is"; anbeeld.com section 1).                   */
/* ------------------------------------------------------------------------- */

/* H[i*d + j] = (-1)^popcount(i & j) / sqrt(d), the normalised Sylvester matrix. */
void kvo_hadamard(int d, double* H) {
    double s = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            int p = __builtin_popcount((unsigned)(i & j)) & 1;
            H[(size_t)i * d + j] = p ? -s : s;
        }
}

/* Y = X * H for X of T rows and d columns (each token row rotated). The sum runs
 * over the +-1 entries of the Sylvester matrix and the result is divided by sqrt(d)
 * once: for fp16 inputs every partial sum is exact in binary64 (fp16 values are
 * multiples of 2^-24 below 2^16, so 128 of them need at most 47 significant bits),
 * hence Y is exact up to that single division and zero stays zero. */
void kvo_rotate(const double* X, int T, int d, double* Y) {
    double s = sqrt((double)d);
    for (int i = 0; i < T; ++i)
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int k = 0; k < d; ++k) {
                int neg = __builtin_popcount((unsigned)(k & j)) & 1;
                acc += neg ? -X[(size_t)i * d + k] : X[(size_t)i * d + k];
            }
            Y[(size_t)i * d + j] = acc / s;
        }
}

/* ------------------------------------------------------------------------- */
/* Sinkhorn-style variance normalisation (fig1.dev "What it is";              */
/* anbeeld.com section 1: 16 iterations).                                     */
/* Z starts as Y; each iteration divides every token row by its RMS (folding  */
/* the factor into a) and then every channel column by its RMS (folding it    */
/* into c). Y = diag(a) Z diag(c) holds throughout.                           */
/* row_dev[k], col_dev[k] (optional): after iteration k, the largest |RMS-1|  */
/* over rows and over columns of Z.                                           */
/* ------------------------------------------------------------------------- */
void kvo_sinkhorn(const double* Y, int T, int d, int iters, double* a, double* c,
                  double* Z_out, double* row_dev, double* col_dev) {
    double* Z = (double*)malloc(sizeof(double) * (size_t)T * d);
    memcpy(Z, Y, sizeof(double) * (size_t)T * d);
    for (int i = 0; i < T; ++i) a[i] = 1.0;
    for (int j = 0; j < d; ++j) c[j] = 1.0;
    for (int k = 0; k < iters; ++k) {
        /* token axis */
        for (int i = 0; i < T; ++i) {
            double ss = 0.0;
            for (int j = 0; j < d; ++j) ss += Z[(size_t)i * d + j] * Z[(size_t)i * d + j];
            double r = sqrt(ss / d);
            if (r == 0.0) r = 1.0;
            for (int j = 0; j < d; ++j) Z[(size_t)i * d + j] /= r;
            a[i] *= r;
        }
        /* channel axis */
        for (int j = 0; j < d; ++j) {
            double ss = 0.0;
            for (int i = 0; i < T; ++i) ss += Z[(size_t)i * d + j] * Z[(size_t)i * d + j];
            double g = sqrt(ss / T);
            if (g == 0.0) g = 1.0;
            for (int i = 0; i < T; ++i) Z[(size_t)i * d + j] /= g;
            c[j] *= g;
        }
        if (row_dev || col_dev) {
            double rd = 0.0, cd = 0.0;
            for (int i = 0; i < T; ++i) {
                double ss = 0.0;
                for (int j = 0; j < d; ++j) ss += Z[(size_t)i * d + j] * Z[(size_t)i * d + j];
                double dev = fabs(sqrt(ss / d) - 1.0);
                if (ss > 0.0 && dev > rd) rd = dev;
            }
            for (int j = 0; j < d; ++j) {
                double ss = 0.0;
                for (int i = 0; i < T; ++i) ss += Z[(size_t)i * d + j] * Z[(size_t)i * d + j];
                double dev = fabs(sqrt(ss / T) - 1.0);
                if (ss > 0.0 && dev > cd) cd = dev;
            }
            if (row_dev) row_dev[k] = rd;
            if (col_dev) col_dev[k] = cd;
        }
    }
    if (Z_out) memcpy(Z_out, Z, sizeof(double) * (size_t)T * d);
    free(Z);
}

/* ------------------------------------------------------------------------- */
/* Record layout (anbeeld.com section 2.1: "the layout stores the quantized   */
/* payload with its scale metadata").                                         */
/* ------------------------------------------------------------------------- */
size_t kvo_header_bytes(int T, int d) { return 16 + 2 * (size_t)T + 2 * (size_t)d; }

size_t kvo_payload_bytes(int T, int d, int bits) {
    size_t nbits = (size_t)T * d * bits;
    size_t words = (nbits + 31) / 32;
    return words * 4;
}

size_t kvo_record_bytes(int T, int d, int bits) {
    size_t r = kvo_header_bytes(T, d) + kvo_payload_bytes(T, d, bits);
    return (r + 15) / 16 * 16;
}

/* Stream position of logical code (i = token, j = channel). */
static size_t stream_index(int i, int j, int T, int d, int side) {
    return side == 0 ? (size_t)i * d + j /* K: token-major */
                     : (size_t)j * T + i; /* V: channel-major */
}

/* codes[i*d + j] -> payload. Element e of the stream occupies bits
 * (e*b) mod 32 .. of little-endian 32-bit word floor(e*b/32), least significant first,
 * spilling into the next word when it does not fit (b = 3). */
void kvo_pack(const uint8_t* codes, int T, int d, int bits, int side, uint8_t* payload) {
    size_t nbytes = kvo_payload_bytes(T, d, bits);
    memset(payload, 0, nbytes);
    for (int i = 0; i < T; ++i)
        for (int j = 0; j < d; ++j) {
            size_t e = stream_index(i, j, T, d, side);
            uint32_t v = codes[(size_t)i * d + j];
            for (int k = 0; k < bits; ++k) {
                size_t bit = e * bits + k;
                size_t word = bit / 32, off = bit % 32;
                if ((v >> k) & 1u) payload[word * 4 + off / 8] |= (uint8_t)(1u << (off % 8));
            }
        }
}

void kvo_unpack(const uint8_t* payload, int T, int d, int bits, int side, uint8_t* codes) {
    for (int i = 0; i < T; ++i)
        for (int j = 0; j < d; ++j) {
            size_t e = stream_index(i, j, T, d, side);
            uint32_t v = 0;
            for (int k = 0; k < bits; ++k) {
                size_t bit = e * bits + k;
                size_t word = bit / 32, off = bit % 32;
                if ((payload[word * 4 + off / 8] >> (off % 8)) & 1u) v |= 1u << k;
            }
            codes[(size_t)i * d + j] = (uint8_t)v;
        }
}

static void put_f32(uint8_t* p, float f) { memcpy(p, &f, 4); }
static float get_f32(const uint8_t* p) { float f; memcpy(&f, p, 4); return f; }
static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 255); p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Parse a record header into doubles. */
void kvo_read_header(const uint8_t* rec, int T, int d, double* delta, double* m, double* a, double* c) {
    *delta = get_f32(rec + 0);
    *m = get_f32(rec + 4);
    for (int i = 0; i < T; ++i) a[i] = kvo_half_to_double(get_u16(rec + 16 + 2 * i));
    for (int j = 0; j < d; ++j) c[j] = kvo_half_to_double(get_u16(rec + 16 + 2 * T + 2 * j));
}

/* ------------------------------------------------------------------------- */
/* Grid and round-to-nearest given the stored scales (fig1.dev "What it is":  */
/* round-to-nearest after the normalisation). Writes delta, m and codes.      */
/* a16/c16 are the stored fp16 scales (as doubles).                           */
/* ------------------------------------------------------------------------- */
void kvo_quantize(const double* Y, int T, int d, int bits, const double* a16, const double* c16,
                  float* delta_out, float* m_out, uint8_t* codes, double* t_out) {
    int L = (1 << bits) - 1;
    size_t n = (size_t)T * d;
    double* Zp = (double*)malloc(sizeof(double) * n);
    double mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < T; ++i)
        for (int j = 0; j < d; ++j) {
            double s = a16[i] * c16[j];
            double z = s != 0.0 ? Y[(size_t)i * d + j] / s : 0.0;
            Zp[(size_t)i * d + j] = z;
            if (z < mn) mn = z;
            if (z > mx) mx = z;
        }
    double delta = (mx - mn) / L;
    if (delta == 0.0) delta = 1.0;
    float d32 = (float)delta;
    float m32 = (float)mn;
    for (size_t e = 0; e < n; ++e) {
        double t = (Zp[e] - (double)m32) / (double)d32;
        if (t_out) t_out[e] = t;
        double q = nearbyint(t); /* ties to even */
        if (q < 0) q = 0;
        if (q > L) q = L;
        codes[e] = (uint8_t)q;
    }
    *delta_out = d32;
    *m_out = m32;
    free(Zp);
}

/* Codes for a given grid (m, delta) and stored scales: t = (Y/(a c) - m)/delta,
 * q = clamp(round-half-even(t), 0, 2^b-1). Used to check another implementation's
 * codes against its own metadata. */
void kvo_codes_for_grid(const double* Y, int T, int d, int bits, const double* a16, const double* c16,
                        double m, double delta, uint8_t* codes, double* t_out) {
    int L = (1 << bits) - 1;
    for (int i = 0; i < T; ++i)
        for (int j = 0; j < d; ++j) {
            size_t e = (size_t)i * d + j;
            double s = a16[i] * c16[j];
            double z = s != 0.0 ? Y[e] / s : 0.0;
            double t = (z - m) / delta;
            if (t_out) t_out[e] = t;
            double q = nearbyint(t);
            if (q < 0) q = 0;
            if (q > L) q = L;
            codes[e] = (uint8_t)q;
        }
}

/* ------------------------------------------------------------------------- */
/* The group seal: rotate, normalise, store scales, quantise, pack.           */
/* x: T x d fp16 bit patterns (token rows). side 0 = K, 1 = V.                */
/* Returns 0, or -1 on a bad argument. a_out/c_out (optional) receive the     */
/* unrounded fp64 Sinkhorn scales.                                            */
/* ------------------------------------------------------------------------- */
int kvo_seal(const uint16_t* x, int T, int d, int bits, int side, int iters,
             uint8_t* record, double* a_out, double* c_out) {
    if (bits < 1 || bits > 8 || T <= 0 || d <= 0 || (d & (d - 1)) != 0) return -1;
    size_t n = (size_t)T * d;
    double* X = (double*)malloc(sizeof(double) * n);
    double* Y = (double*)malloc(sizeof(double) * n);
    double* a = (double*)malloc(sizeof(double) * T);
    double* c = (double*)malloc(sizeof(double) * d);
    double* a16 = (double*)malloc(sizeof(double) * T);
    double* c16 = (double*)malloc(sizeof(double) * d);
    uint8_t* codes = (uint8_t*)malloc(n);
    for (size_t e = 0; e < n; ++e) X[e] = kvo_half_to_double(x[e]);
    kvo_rotate(X, T, d, Y);
    kvo_sinkhorn(Y, T, d, iters, a, c, NULL, NULL, NULL);
    size_t rb = kvo_record_bytes(T, d, bits);
    memset(record, 0, rb);
    for (int i = 0; i < T; ++i) {
        uint16_t h = kvo_double_to_half_sat(a[i]);
        a16[i] = kvo_half_to_double(h);
        put_u16(record + 16 + 2 * i, h);
    }
    for (int j = 0; j < d; ++j) {
        uint16_t h = kvo_double_to_half_sat(c[j]);
        c16[j] = kvo_half_to_double(h);
        put_u16(record + 16 + 2 * T + 2 * j, h);
    }
    float d32, m32;
    kvo_quantize(Y, T, d, bits, a16, c16, &d32, &m32, codes, NULL);
    put_f32(record + 0, d32);
    put_f32(record + 4, m32);
    kvo_pack(codes, T, d, bits, side, record + kvo_header_bytes(T, d));
    if (a_out) memcpy(a_out, a, sizeof(double) * T);
    if (c_out) memcpy(c_out, c, sizeof(double) * d);
    free(X); free(Y); free(a); free(c); free(a16); free(c16); free(codes);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Dequantisation ("convert to a standard cache layout", anbeeld.com 2.1):    */
/* yhat_ij = a_i c_j (m + delta q_ij) in the rotated frame; frame 0 rotates  */
/* back, xhat = yhat * H (H is symmetric and orthonormal, so H^-1 = H).       */
/* ------------------------------------------------------------------------- */
void kvo_dequant(const uint8_t* record, int T, int d, int bits, int side, int frame, double* out) {
    size_t n = (size_t)T * d;
    double delta, m;
    double* a = (double*)malloc(sizeof(double) * T);
    double* c = (double*)malloc(sizeof(double) * d);
    uint8_t* codes = (uint8_t*)malloc(n);
    kvo_read_header(record, T, d, &delta, &m, a, c);
    kvo_unpack(record + kvo_header_bytes(T, d), T, d, bits, side, codes);
    double* Yh = frame == 0 ? (double*)malloc(sizeof(double) * n) : out;
    for (int i = 0; i < T; ++i)
        for (int j = 0; j < d; ++j)
            Yh[(size_t)i * d + j] = a[i] * c[j] * (m + delta * codes[(size_t)i * d + j]);
    if (frame == 0) {
        kvo_rotate(Yh, T, d, out);
        free(Yh);
    }
    free(a); free(c); free(codes);
}

/* ------------------------------------------------------------------------- */
/* Decode attention for one (sequence, KV head) and its r query heads         */
/* (anbeeld.com section 1 and 2.1). Exact tokens (sink, tail) are scored with */
/* the unrotated query against their fp16 K; sealed tokens with the rotated   */
/* query q' = qH against the dequantised rotated K. Softmax over all tokens   */
/* in fp64. The sealed part of the output is accumulated in the rotated frame */
/* and rotated back once: o = (sum_exact p v + (sum_sealed p yhatV) H) / l.   */
/* krec/vrec: n_groups consecutive records each. out: [r][d]. lse (optional): */
/* log of the softmax denominator per head, including the max shift.          */
/* ------------------------------------------------------------------------- */
int kvo_attention(int d, int T, int r, int kbits, int vbits, const uint16_t* q, double scale,
                  int n_sink, const uint16_t* sink_k, const uint16_t* sink_v,
                  int n_groups, const uint8_t* krec, const uint8_t* vrec,
                  int n_tail, const uint16_t* tail_k, const uint16_t* tail_v,
                  double* out, double* lse) {
    if ((d & (d - 1)) != 0 || r <= 0) return -1;
    size_t kb = kvo_record_bytes(T, d, kbits), vb = kvo_record_bytes(T, d, vbits);
    size_t ns = (size_t)n_groups * T;
    int n_all = n_sink + (int)ns + n_tail;
    double* YK = (double*)malloc(sizeof(double) * (ns ? ns : 1) * d);
    double* YV = (double*)malloc(sizeof(double) * (ns ? ns : 1) * d);
    for (int g = 0; g < n_groups; ++g) {
        kvo_dequant(krec + (size_t)g * kb, T, d, kbits, 0, 1, YK + (size_t)g * T * d);
        kvo_dequant(vrec + (size_t)g * vb, T, d, vbits, 1, 1, YV + (size_t)g * T * d);
    }
    double* s = (double*)malloc(sizeof(double) * (n_all ? n_all : 1));
    double* qd = (double*)malloc(sizeof(double) * d);
    double* qr = (double*)malloc(sizeof(double) * d);
    double* oe = (double*)malloc(sizeof(double) * d);
    double* orot = (double*)malloc(sizeof(double) * d);
    double* ob = (double*)malloc(sizeof(double) * d);
    for (int h = 0; h < r; ++h) {
        for (int j = 0; j < d; ++j) qd[j] = kvo_half_to_double(q[(size_t)h * d + j]);
        kvo_rotate(qd, 1, d, qr);
        int t = 0;
        for (int i = 0; i < n_sink; ++i, ++t) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += qd[j] * kvo_half_to_double(sink_k[(size_t)i * d + j]);
            s[t] = scale * acc;
        }
        for (size_t i = 0; i < ns; ++i, ++t) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += qr[j] * YK[i * d + j];
            s[t] = scale * acc;
        }
        for (int i = 0; i < n_tail; ++i, ++t) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += qd[j] * kvo_half_to_double(tail_k[(size_t)i * d + j]);
            s[t] = scale * acc;
        }
        double mx = -INFINITY;
        for (t = 0; t < n_all; ++t) if (s[t] > mx) mx = s[t];
        double l = 0.0;
        for (t = 0; t < n_all; ++t) { s[t] = exp(s[t] - mx); l += s[t]; }
        for (int j = 0; j < d; ++j) { oe[j] = 0.0; orot[j] = 0.0; }
        t = 0;
        for (int i = 0; i < n_sink; ++i, ++t)
            for (int j = 0; j < d; ++j) oe[j] += s[t] * kvo_half_to_double(sink_v[(size_t)i * d + j]);
        for (size_t i = 0; i < ns; ++i, ++t)
            for (int j = 0; j < d; ++j) orot[j] += s[t] * YV[i * d + j];
        for (int i = 0; i < n_tail; ++i, ++t)
            for (int j = 0; j < d; ++j) oe[j] += s[t] * kvo_half_to_double(tail_v[(size_t)i * d + j]);
        kvo_rotate(orot, 1, d, ob);
        for (int j = 0; j < d; ++j) out[(size_t)h * d + j] = n_all ? (oe[j] + ob[j]) / l : 0.0;
        if (lse) lse[h] = n_all ? mx + log(l) : -INFINITY;
    }
    free(YK); free(YV); free(s); free(qd); free(qr); free(oe); free(orot); free(ob);
    return 0;
}
