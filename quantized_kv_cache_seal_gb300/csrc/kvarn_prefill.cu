// KVarN prefill (many-query) attention for sm_103a.
//
// Method (anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", sections 1 and
// 2.1): the cache is read the way the decode path reads it. The sink and the exact tail
// are fp16 and meet the unrotated query; every sealed group is read from its record with
// the query rotated by the record's Hadamard matrix, the sealed part of the output is
// summed in the rotated frame and rotated back once per output row. Each query token of
// a prompt chunk attends causally (keys at positions up to its own) to the cache as it
// stands after the chunk's append, so tokens of the chunk that already sit in a sealed
// group are read sealed.
//
// Work split. One CTA of 8 warps per (sequence, KV head, tile of 128 / r query tokens):
// its 128 query rows are (token, query head) pairs, token-major, and warp w owns rows
// 16 w .. 16 w + 15, the M side of mma.sync m16n8k16 (f16 in, f32 accumulate). Each key
// block is staged once in shared memory and read by all 8 warps:
//   * exact blocks of 64 fp16 tokens (the sink, then the tail), loaded cooperatively;
//   * sealed group pairs, copied with cp.async.bulk into a ring of stages and expanded
//     by all threads into f16 operand tiles: code c becomes the subnormal half c 2^-24
//     (exact), the K tile token-major and the V tile channel-major, as in the records.
// For a group with codes q, token scales a, channel scales c and grid (m, delta), the
// score of row i and token t is
//   scale * qm_i * a_t * (delta * sum_j (v_ij c_j) q_tj + m * sum_j v_ij c_j),
// v_i = q'_i / qm_i the rotated query scaled to |v| <= 1; v c enters as an f16 high
// part and an f16 low part (two MMAs into one accumulator), which keeps the logits at
// about fp32 accuracy. The rotated output of row i gains
//   c_j * (delta_V * sum_t w_it qV_tj + m_V * sum_t w_it),  w_it = p_it aV_t,
// with w scaled by a power of two rho into [0, 2) and rounded to f16. The row sums come
// from the same MMAs with an all-ones operand. The accumulator is unrotated over the
// exact blocks, rotated once into the record frame, summed over the groups and rotated
// back at the end (the scaled Sylvester matrix is its own inverse).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvarn_dev.cuh"

namespace kvarn {

namespace {

constexpr int kPfWarps = kPrefillThreads / 32;
constexpr int kPfRows = 16 * kPfWarps;  // query rows of a CTA
static_assert(kPfRows == kPrefillRows, "one 16-row MMA tile per warp");
constexpr int kPitch = 272;             // bytes per shared row of 128 halves (ldmatrix without bank conflicts)
constexpr int kTileBytes = 128 * kPitch;
constexpr int kExactBlock = 64;         // tokens of an exact block
constexpr int kQfragBytes = kPfWarps * 8 * 32 * 16;  // one query operand table (high or low parts)
constexpr uint32_t kOnes = 0x3c003c00u;  // half2(1, 1)
#define kNegInfP (-__int_as_float(0x7f800000))

// Shared memory (bytes):
//   [0, 2 T)            sealed phase: K operand tile, V operand tile (T = kTileBytes)
//                       exact phase: K rows [0, 64 pitch), V rows after them; the staged
//                       fp16 queries (128 rows) in [T, 2 T)
//   [2 T, 2 T + 2 Q)    query operand tables, high then low parts (Q = kQfragBytes)
//   ring                stages x (K record + V record), 16-byte aligned
//   bars, positions, query maxima
constexpr int kOffTiles = 0;
constexpr int kOffQraw = kTileBytes;
constexpr int kOffQhi = 2 * kTileBytes;
constexpr int kOffQlo = kOffQhi + kQfragBytes;
constexpr int kOffRing = kOffQlo + kQfragBytes;
static_assert(kOffRing % 128 == 0, "ring alignment");
static_assert(2 * kExactBlock * kPitch <= kTileBytes, "exact blocks fit below the staged queries");

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ldmatrix of four 8 x 8 b16 matrices; lanes 8 i .. 8 i + 7 give the row addresses of matrix i.
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t u32_of(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 h2_of(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ float2 f2_of(uint32_t u) { return __half22float2(h2_of(u)); }

// Bits pos .. pos + width - 1 (width <= 16) of a little-endian stream of N words.
template <int N>
__device__ __forceinline__ uint32_t bits_at(const uint32_t (&s)[N], int pos, int width) {
    const int lo = pos / 32, sh = pos % 32;
    uint32_t v = s[lo] >> sh;
    if (sh + width > 32) v |= s[lo + 1] << (32 - sh);
    return v & ((1u << width) - 1u);
}

// 32 codes of width B (LSB-first from src, 4-byte aligned) -> 16 words of two f16
// operands each: word k holds codes 2 k and 2 k + 1 as the subnormals code * 2^-24.
template <int B>
__device__ __forceinline__ void expand_chunk(const uint8_t* src, uint8_t* dst) {
    uint32_t s[B];
    if constexpr (B == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        s[0] = v.x; s[1] = v.y;
    } else if constexpr (B == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        s[0] = v.x; s[1] = v.y; s[2] = v.z; s[3] = v.w;
    } else if constexpr (B == 8) {
        const uint4 v0 = reinterpret_cast<const uint4*>(src)[0], v1 = reinterpret_cast<const uint4*>(src)[1];
        s[0] = v0.x; s[1] = v0.y; s[2] = v0.z; s[3] = v0.w;
        s[4] = v1.x; s[5] = v1.y; s[6] = v1.z; s[7] = v1.w;
    } else {
#pragma unroll
        for (int k = 0; k < B; ++k) s[k] = reinterpret_cast<const uint32_t*>(src)[k];
    }
    constexpr uint32_t m = (1u << B) - 1u;
    uint32_t o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint32_t f = bits_at(s, 2 * k * B, 2 * B);
        o[k] = (f & m) | ((f >> B) << 16);
    }
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int k = 0; k < 4; ++k) d[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
}

// 128-point Hadamard transform, scaled by 1/sqrt(128), of every row of a warp's 16 x 128
// accumulator in the m16n8 C layout: lane (g, tq) holds in x[nt][e] row g (e < 2) or
// g + 8 (e >= 2), column 8 nt + 2 tq + (e & 1). Column bit 0 is e & 1, bits 1-2 are
// lane bits 0-1, bits 3-6 the tile index. The lower column of a pair takes a + b.
__device__ __forceinline__ void rows_fwht128(float (&x)[16][4], int lane) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
        for (int rb = 0; rb < 4; rb += 2) {
            const float a = x[nt][rb], b = x[nt][rb + 1];
            x[nt][rb] = a + b;
            x[nt][rb + 1] = a - b;
        }
    }
#pragma unroll
    for (int bt = 1; bt < 4; bt <<= 1) {
        const bool upper = (lane & bt) != 0;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, x[nt][e], bt);
                x[nt][e] = upper ? o - x[nt][e] : x[nt][e] + o;
            }
        }
    }
#pragma unroll
    for (int len = 1; len < 16; len <<= 1) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            if (nt & len) continue;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = x[nt][e], b = x[nt + len][e];
                x[nt][e] = a + b;
                x[nt + len][e] = a - b;
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[nt][e] *= kInvSqrt128;
}

// Same transform of one 128-vector held by a warp, channel 4 lane + e in v[e].
__device__ __forceinline__ void vec_fwht128(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
    for (int b = 1; b < 32; b <<= 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[e], b);
            v[e] = (lane & b) ? (o - v[e]) : (v[e] + o);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] *= kInvSqrt128;
}

// Online-softmax state of the two rows a thread holds (g and g + 8 of its warp's tile).
struct RowState {
    float m[2], l[2];  // running maximum (log2 domain) and this thread's partial sum
    float acc[16][4];
};

// Row maxima of a score tile S (nt tiles) over the 4 lanes of a row, the new running
// maxima, the correction factors; p = 2^(S - m) in place; partial sums and accumulator
// rescaled.
template <int NT>
__device__ __forceinline__ void softmax_update(float (&S)[NT][4], RowState& st) {
    float mx0 = kNegInfP, mx1 = kNegInfP;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(S[nt][0], S[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(S[nt][2], S[nt][3]));
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    // the first block is the sink's first, which every row sees: st.m is finite after it
    const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
    const float c0 = ex2(st.m[0] - n0), c1 = ex2(st.m[1] - n1);
    st.m[0] = n0;
    st.m[1] = n1;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        S[nt][0] = ex2(S[nt][0] - n0);
        S[nt][1] = ex2(S[nt][1] - n0);
        S[nt][2] = ex2(S[nt][2] - n1);
        S[nt][3] = ex2(S[nt][3] - n1);
        s0 += S[nt][0] + S[nt][1];
        s1 += S[nt][2] + S[nt][3];
    }
    st.l[0] = fmaf(st.l[0], c0, s0);
    st.l[1] = fmaf(st.l[1], c1, s1);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
        st.acc[nt][0] *= c0;
        st.acc[nt][1] *= c0;
        st.acc[nt][2] *= c1;
        st.acc[nt][3] *= c1;
    }
}

struct Cta {
    const PrefillSeq* e;
    int kvh, r, t0;      // KV head, query heads per KV head, first query token of the tile
    int first_pos;       // position of query token 0 of the sequence's chunk
    int pmax;            // largest valid query position of the tile
    int n_vis;           // sealed groups with a token at or before pmax
    size_t blk;          // (sequence, layer, KV head) index of the exact regions
};

// One exact block: keys at positions kp0 .. kp0 + cnt - 1 (rows >= cnt are zeros),
// K rows at sK, V rows at sV (pitch kPitch), queries (unrotated fp16) at sQ.
__device__ __forceinline__ void exact_block(uint32_t sK, uint32_t sV, uint32_t sQ, int kp0, int cnt, int p0, int p1,
                                            float scale_log2, RowState& st, int lane) {
    const int tq = lane & 3;
    float S[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
    const uint32_t qa = sQ + (lane & 15) * kPitch + 16 * (lane >> 4);
    const uint32_t ka = sK + ((lane & 7) + 8 * (lane >> 4)) * kPitch + 16 * ((lane >> 3) & 1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldsm4(qa + 32 * ks, a);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b[4];
            ldsm4(ka + 16 * np * kPitch + 32 * ks, b);
            mma_f16(S[2 * np], a[0], a[1], a[2], a[3], b[0], b[1]);
            mma_f16(S[2 * np + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 8 * nt + 2 * tq + (e & 1);
            const int P = e < 2 ? p0 : p1;
            S[nt][e] = (j < cnt && kp0 + j <= P) ? S[nt][e] * scale_log2 : kNegInfP;
        }
    }
    softmax_update<8>(S, st);
    // P V with the weights split into f16 high and low parts
    uint32_t ph[4][4], pl[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float* s = S[2 * kk + h];
            const __half2 h01 = __floats2half2_rn(s[0], s[1]), h23 = __floats2half2_rn(s[2], s[3]);
            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
            ph[kk][2 * h] = u32_of(h01);
            ph[kk][2 * h + 1] = u32_of(h23);
            pl[kk][2 * h] = u32_of(__floats2half2_rn(s[0] - f01.x, s[1] - f01.y));
            pl[kk][2 * h + 1] = u32_of(__floats2half2_rn(s[2] - f23.x, s[3] - f23.y));
        }
    }
    // matrix i of an ldmatrix: keys 16 kk + 8 (i & 1), channels 8 nt + 8 (i >> 1), transposed
    const uint32_t va = sV + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kPitch + 16 * (lane >> 4);
#pragma unroll
    for (int np = 0; np < 8; ++np) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t b[4];
            ldsm4t(va + 16 * kk * kPitch + 32 * np, b);
            // A fragment order: (row g, k lo), (row g + 8, k lo), (row g, k hi), (row g + 8, k hi)
            mma_f16(st.acc[2 * np], ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3], b[0], b[1]);
            mma_f16(st.acc[2 * np], pl[kk][0], pl[kk][1], pl[kk][2], pl[kk][3], b[0], b[1]);
            mma_f16(st.acc[2 * np + 1], ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3], b[2], b[3]);
            mma_f16(st.acc[2 * np + 1], pl[kk][0], pl[kk][1], pl[kk][2], pl[kk][3], b[2], b[3]);
        }
    }
}

// One sealed group pair: operand tiles at sK (token-major) and sV (channel-major), the
// records' headers at krec / vrec, the warp's query tables at qhi / qlo.
__device__ __forceinline__ void sealed_group(uint32_t sK, uint32_t sV, const uint8_t* krec, const uint8_t* vrec,
                                             const uint4* qhi, const uint4* qlo, float qm0, float qm1, int gp0,
                                             bool masked, int p0, int p1, float scale_log2, RowState& st, int lane) {
    const int tq = lane & 3;
    const uint32_t* cK = reinterpret_cast<const uint32_t*>(krec + 272);
    float S[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
    float rs[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ka = sK + ((lane & 7) + 8 * (lane >> 4)) * kPitch + 16 * ((lane >> 3) & 1);
#pragma unroll 2
    for (int ks = 0; ks < 8; ++ks) {
        const uint4 vh = qhi[ks * 32 + lane], vl = qlo[ks * 32 + lane];
        const __half2 c01 = h2_of(cK[8 * ks + tq]), c89 = h2_of(cK[8 * ks + 4 + tq]);
        const uint32_t vhs[4] = {vh.x, vh.y, vh.z, vh.w}, vls[4] = {vl.x, vl.y, vl.z, vl.w};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 c = i < 2 ? c01 : c89;
            const __half2 hi = __hmul2(h2_of(vhs[i]), c);
            const __half2 res = __hfma2(h2_of(vhs[i]), c, __hneg2(hi));  // exact residual of the product
            ah[i] = u32_of(hi);
            al[i] = u32_of(__hfma2(h2_of(vls[i]), c, res));
        }
        mma_f16(rs, ah[0], ah[1], ah[2], ah[3], kOnes, kOnes);
        mma_f16(rs, al[0], al[1], al[2], al[3], kOnes, kOnes);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t b[4];
            ldsm4(ka + 16 * np * kPitch + 32 * ks, b);
            mma_f16(S[2 * np], ah[0], ah[1], ah[2], ah[3], b[0], b[1]);
            mma_f16(S[2 * np], al[0], al[1], al[2], al[3], b[0], b[1]);
            mma_f16(S[2 * np + 1], ah[0], ah[1], ah[2], ah[3], b[2], b[3]);
            mma_f16(S[2 * np + 1], al[0], al[1], al[2], al[3], b[2], b[3]);
        }
    }
    {
        const float dK = *reinterpret_cast<const float*>(krec);
        const float mK = *reinterpret_cast<const float*>(krec + 4);
        const uint32_t* aK = reinterpret_cast<const uint32_t*>(krec + 16);
        // codes entered as code * 2^-24
        const float al0 = scale_log2 * qm0 * dK * 16777216.0f, al1 = scale_log2 * qm1 * dK * 16777216.0f;
        const float be0 = scale_log2 * qm0 * mK * rs[0], be1 = scale_log2 * qm1 * mK * rs[2];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const float2 a = f2_of(aK[4 * nt + tq]);
            S[nt][0] = a.x * fmaf(al0, S[nt][0], be0);
            S[nt][1] = a.y * fmaf(al0, S[nt][1], be0);
            S[nt][2] = a.x * fmaf(al1, S[nt][2], be1);
            S[nt][3] = a.y * fmaf(al1, S[nt][3], be1);
        }
        if (masked) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int pos = gp0 + 8 * nt + 2 * tq;
                if (pos > p0) S[nt][0] = kNegInfP;
                if (pos + 1 > p0) S[nt][1] = kNegInfP;
                if (pos > p1) S[nt][2] = kNegInfP;
                if (pos + 1 > p1) S[nt][3] = kNegInfP;
            }
        }
    }
    softmax_update<16>(S, st);
    // weights w = p aV rho in f16; rho = 2^(15 - e) with e the biased exponent of the
    // group's largest aV, so that every aV rho lies in [0, 2)
    const uint32_t* aV = reinterpret_cast<const uint32_t*>(vrec + 16);
    float rho;
    {
        const uint2 ab = reinterpret_cast<const uint2*>(vrec + 16)[lane];
        uint32_t amaxb = __vmaxu2(ab.x, ab.y);
        amaxb = max(amaxb & 0xffffu, amaxb >> 16);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) amaxb = max(amaxb, __shfl_xor_sync(0xffffffffu, amaxb, o));
        const int ebits = max((int)(amaxb >> 10) & 31, 1);
        rho = __int_as_float((127 + 15 - ebits) << 23);
    }
    uint32_t pw[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nt = 2 * kk + h;
            const float2 a = f2_of(aV[4 * nt + tq]);
            const float wx = a.x * rho, wy = a.y * rho;
            pw[kk][2 * h] = u32_of(__floats2half2_rn(S[nt][0] * wx, S[nt][1] * wy));
            pw[kk][2 * h + 1] = u32_of(__floats2half2_rn(S[nt][2] * wx, S[nt][3] * wy));
        }
    }
    float ws[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_f16(ws, pw[kk][0], pw[kk][1], pw[kk][2], pw[kk][3], kOnes, kOnes);
    const float dV = *reinterpret_cast<const float*>(vrec);
    const float mV = *reinterpret_cast<const float*>(vrec + 4);
    const uint32_t* cV = reinterpret_cast<const uint32_t*>(vrec + 272);
    const float irho = 1.0f / rho;  // a power of two: exact
    const float gam = dV * 16777216.0f * irho;
    const float de0 = mV * ws[0] * irho, de1 = mV * ws[2] * irho;
    // matrix i of an ldmatrix: channels 16 np + 8 (i >> 1), tokens 16 kk + 8 (i & 1)
    const uint32_t va = sV + ((lane & 7) + 8 * (lane >> 4)) * kPitch + 16 * ((lane >> 3) & 1);
#pragma unroll
    for (int np = 0; np < 8; ++np) {
        float raw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t b[4];
            ldsm4(va + 16 * np * kPitch + 32 * kk, b);
            mma_f16(raw[0], pw[kk][0], pw[kk][1], pw[kk][2], pw[kk][3], b[0], b[1]);
            mma_f16(raw[1], pw[kk][0], pw[kk][1], pw[kk][2], pw[kk][3], b[2], b[3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nt = 2 * np + h;
            const float2 c = f2_of(cV[4 * nt + tq]);
            st.acc[nt][0] = fmaf(c.x, fmaf(gam, raw[h][0], de0), st.acc[nt][0]);
            st.acc[nt][1] = fmaf(c.y, fmaf(gam, raw[h][1], de0), st.acc[nt][1]);
            st.acc[nt][2] = fmaf(c.x, fmaf(gam, raw[h][2], de1), st.acc[nt][2]);
            st.acc[nt][3] = fmaf(c.y, fmaf(gam, raw[h][3], de1), st.acc[nt][3]);
        }
    }
}

__device__ __forceinline__ const uint8_t* group_src(const PrefillParams& p, const Cta& c, int g) {
    const int32_t* table = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table) +
                           ((size_t)c.e->seq * p.num_layers + p.layer) * p.max_groups;
    const int slot = table[g];
    return p.base + p.lay.pool + (size_t)slot * p.slot_bytes + (size_t)c.kvh * (p.rec_k + p.rec_v);
}

template <int KB, int VB>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int g = lane >> 2;
    const int pair = p.rec_k + p.rec_v;
    uint8_t* ring = smem + kOffRing;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)p.stages * pair);
    int* rowpos = reinterpret_cast<int*>(full + p.stages);
    float* rowqm = reinterpret_cast<float*>(rowpos + kPfRows);
    int32_t* err = reinterpret_cast<int32_t*>(p.base + p.lay.err);

    // the CTA's (sequence, KV head, tile): the heaviest tiles (latest tokens) first
    Cta c;
    {
        int lo = 0, up = p.n_seqs - 1;
        while (lo < up) {
            const int mid = (lo + up + 1) >> 1;
            if (p.seqs[mid].cta_begin <= (int)blockIdx.x) lo = mid; else up = mid - 1;
        }
        c.e = &p.seqs[lo];
        const int local = (int)blockIdx.x - c.e->cta_begin;
        c.kvh = local % p.hkv;
        const int tile = c.e->n_tiles - 1 - local / p.hkv;
        c.r = p.r;
        const int qt = kPfRows / p.r;
        c.t0 = tile * qt;
        c.first_pos = c.e->n - c.e->q_len;
        c.pmax = c.first_pos + min(c.t0 + qt, c.e->q_len) - 1;
        const int vis = c.pmax >= kSink ? (c.pmax - kSink) / kGroup + 1 : 0;
        c.n_vis = min(c.e->n_groups, vis);
        c.blk = ((size_t)c.e->seq * p.num_layers + p.layer) * p.hkv + c.kvh;
    }
    const int n_vis = c.n_vis;
    if (t == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(full + s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int gi = 0; gi < min(n_vis, p.stages); ++gi) {
            mbar_arrive_expect_tx(full + gi, (uint32_t)pair);
            bulk_g2s(ring + (size_t)gi * pair, group_src(p, c, gi), (uint32_t)pair, full + gi);
        }
    }
    // stage the tile's queries (fp16 rows; rows past the chunk are zeros) and positions
    {
        uint8_t* qraw = smem + kOffQraw;
#pragma unroll
        for (int it = 0; it < kPfRows * 16 / kPrefillThreads; ++it) {
            const int idx = t + kPrefillThreads * it;
            const int row = idx >> 4, col = idx & 15;
            const int tok = c.t0 + row / c.r;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (tok < c.e->q_len) {
                const size_t qrow = ((size_t)(c.e->q_row + tok) * p.hq + (size_t)c.kvh * c.r + row % c.r);
                v = reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim)[col];
            }
            *reinterpret_cast<uint4*>(qraw + row * kPitch + 16 * col) = v;
        }
        if (t < kPfRows) {
            const int tok = c.t0 + t / c.r;
            rowpos[t] = tok < c.e->q_len ? c.first_pos + tok : c.e->n - 1;
        }
    }
    RowState st;
    st.m[0] = st.m[1] = kNegInfP;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) st.acc[nt][0] = st.acc[nt][1] = st.acc[nt][2] = st.acc[nt][3] = 0.f;
    __syncthreads();
    const int p0 = rowpos[16 * w + g], p1 = rowpos[16 * w + g + 8];

    // ---- exact phase: the sink, then the tail, in blocks of 64 tokens
    {
        const int n_sink = min(c.e->n, kSink);
        const int sink_vis = min(n_sink, c.pmax + 1);
        const int tail_start = kSink + kGroup * c.e->n_groups;
        const int tail_vis = max(0, min(c.e->n, c.pmax + 1) - tail_start);
        const int nb_sink = (sink_vis + kExactBlock - 1) / kExactBlock;
        const int nb = nb_sink + (tail_vis + kExactBlock - 1) / kExactBlock;
        const uint32_t sK = smem_addr(smem + kOffTiles), sV = sK + kExactBlock * kPitch;
        const uint32_t sQ = smem_addr(smem + kOffQraw) + 16 * w * kPitch;
        for (int b = 0; b < nb; ++b) {
            const bool tail = b >= nb_sink;
            const int kp0 = tail ? tail_start + kExactBlock * (b - nb_sink) : kExactBlock * b;
            const int cnt = tail ? min(kExactBlock, tail_start + tail_vis - kp0) : min(kExactBlock, sink_vis - kp0);
            if (b > 0) __syncthreads();  // every warp is done with the previous block
#pragma unroll
            for (int it = 0; it < 2 * kExactBlock * 16 / kPrefillThreads; ++it) {
                const int idx = t + kPrefillThreads * it;
                const int side = idx / (kExactBlock * 16);
                const int row = (idx >> 4) % kExactBlock, col = idx & 15;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (row < cnt) {
                    const int pos = kp0 + row;
                    size_t off;
                    if (tail)
                        off = (side ? p.lay.tail_v : p.lay.tail_k) +
                              (c.blk * p.tail_cap + (size_t)((pos - kSink) % p.tail_cap)) * 256;
                    else
                        off = (side ? p.lay.sink_v : p.lay.sink_k) + (c.blk * kSink + pos) * 256;
                    v = reinterpret_cast<const uint4*>(p.base + off)[col];
                }
                *reinterpret_cast<uint4*>(smem + kOffTiles + (side * kExactBlock + row) * kPitch + 16 * col) = v;
            }
            __syncthreads();
            exact_block(sK, sV, sQ, kp0, cnt, p0, p1, p.scale_log2, st, lane);
        }
    }

    if (n_vis > 0) {
        // ---- the warp's query operand tables: v = q H / qm split into f16 high and low parts
        {
            const uint8_t* qraw = smem + kOffQraw;
            uint32_t* qhi = reinterpret_cast<uint32_t*>(smem + kOffQhi) + w * 8 * 32 * 4;
            uint32_t* qlo = reinterpret_cast<uint32_t*>(smem + kOffQlo) + w * 8 * 32 * 4;
            for (int rr = 0; rr < 16; ++rr) {
                const uint2 raw = *reinterpret_cast<const uint2*>(qraw + (16 * w + rr) * kPitch + 8 * lane);
                const float2 x01 = f2_of(raw.x), x23 = f2_of(raw.y);
                float v[4] = {x01.x, x01.y, x23.x, x23.y};
                vec_fwht128(v, lane);
                float qm = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
                const float inv = qm > 0.f ? 1.0f / qm : 0.f;
                if (lane == 0) rowqm[16 * w + rr] = qm;
                // channels 4 lane + 2 j, + 1 -> fragment (k-step ks, lane 4 (rr % 8) + tq, register rb + 2 h)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int ch = 4 * lane + 2 * j;
                    const int ks = ch >> 4, h = (ch >> 3) & 1, tq = (ch & 7) >> 1;
                    const int reg = (rr >> 3) + 2 * h;
                    const int dst = (ks * 32 + 4 * (rr & 7) + tq) * 4 + reg;
                    const float a = v[2 * j] * inv, b = v[2 * j + 1] * inv;
                    const __half2 hi = __floats2half2_rn(a, b);
                    const float2 hf = __half22float2(hi);
                    qhi[dst] = u32_of(hi);
                    qlo[dst] = u32_of(__floats2half2_rn(a - hf.x, b - hf.y));
                }
            }
        }
        rows_fwht128(st.acc, lane);  // into the records' frame
        __syncthreads();
        const float qm0 = rowqm[16 * w + g], qm1 = rowqm[16 * w + g + 8];
        const int pmin = __shfl_sync(0xffffffffu, min(p0, p1), 0);  // rows are in position order
        const uint4* qhi = reinterpret_cast<const uint4*>(smem + kOffQhi) + w * 8 * 32;
        const uint4* qlo = reinterpret_cast<const uint4*>(smem + kOffQlo) + w * 8 * 32;
        const uint32_t sK = smem_addr(smem + kOffTiles), sV = sK + kTileBytes;
        for (int gi = 0; gi < n_vis; ++gi) {
            const int s = gi % p.stages;
            const uint8_t* stage = ring + (size_t)s * pair;
            if (gi > 0) {
                __syncthreads();  // every warp is done with group gi - 1 (tiles and its stage)
                if (t == 0 && gi - 1 + p.stages < n_vis) {
                    const int sp = (gi - 1) % p.stages;
                    mbar_arrive_expect_tx(full + sp, (uint32_t)pair);
                    bulk_g2s(ring + (size_t)sp * pair, group_src(p, c, gi - 1 + p.stages), (uint32_t)pair, full + sp);
                }
            }
            mbar_wait(full + s, (uint32_t)((gi / p.stages) & 1), err);
            // expand the codes: 2 records x 128 rows x 4 chunks of 32 codes
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int idx = t + kPrefillThreads * it;
                const int side = idx >> 9, row = (idx >> 2) & 127, ch = idx & 3;
                uint8_t* dst = smem + kOffTiles + side * kTileBytes + row * kPitch + 64 * ch;
                if (side == 0)
                    expand_chunk<KB>(stage + 528 + row * 16 * KB + ch * 4 * KB, dst);
                else
                    expand_chunk<VB>(stage + p.rec_k + 528 + row * 16 * VB + ch * 4 * VB, dst);
            }
            __syncthreads();
            const int gp0 = kSink + kGroup * gi;
            sealed_group(sK, sV, stage, stage + p.rec_k, qhi, qlo, qm0, qm1, gp0, gp0 + kGroup - 1 > pmin, p0, p1,
                         p.scale_log2, st, lane);
        }
        rows_fwht128(st.acc, lane);  // back to the original frame
    }

    // ---- normalise and write the valid rows
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
    const int tq = lane & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int row = 16 * w + g + 8 * half;
        const int tok = c.t0 + row / c.r;
        if (tok < c.e->q_len) {
            const size_t orow = (size_t)(c.e->q_row + tok) * p.hq + (size_t)c.kvh * c.r + row % c.r;
            uint32_t* o = reinterpret_cast<uint32_t*>(p.out + orow * kHeadDim);
            const float inv = half ? i1 : i0;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                o[4 * nt + tq] = u32_of(__floats2half2_rn(st.acc[nt][2 * half] * inv, st.acc[nt][2 * half + 1] * inv));
        }
    }
    // Normally every copy was waited for. After a wait that gave up, let the copies in
    // flight land (bounded) before the CTA's shared memory goes away.
    __syncthreads();
    if (t == 0 && (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout)) {
        const uint64_t t0 = global_ns();
        for (int k = max(0, n_vis - p.stages); k < n_vis; ++k)  // every group below n_vis was issued
            while (!mbar_try_wait(full + (k % p.stages), (uint32_t)((k / p.stages) & 1)) &&
                   global_ns() - t0 < kWaitLimitNs) {
            }
    }
}

template <int KB, int VB>
int launch_pf(const PrefillParams& p, int smem, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             max_optin_smem());
        if (e != cudaSuccess) return (int)e;
        attr = true;
    }
    prefill_kernel<KB, VB><<<p.grid, kPrefillThreads, smem, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace

int prefill_smem_bytes(int k_bits, int v_bits, int stages) {
    const size_t pair = record_bytes(k_bits) + record_bytes(v_bits);
    return (int)(kOffRing + (size_t)stages * pair + (size_t)stages * 8 + kPrefillRows * 8);
}

int launch_prefill(const PrefillParams& p, int smem, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    switch (p.k_bits * 16 + p.v_bits) {
        case 0x22: return launch_pf<2, 2>(p, smem, s);
        case 0x24: return launch_pf<2, 4>(p, smem, s);
        case 0x28: return launch_pf<2, 8>(p, smem, s);
        case 0x42: return launch_pf<4, 2>(p, smem, s);
        case 0x44: return launch_pf<4, 4>(p, smem, s);
        case 0x48: return launch_pf<4, 8>(p, smem, s);
        case 0x82: return launch_pf<8, 2>(p, smem, s);
        case 0x84: return launch_pf<8, 4>(p, smem, s);
        case 0x88: return launch_pf<8, 8>(p, smem, s);
        case 0x33: return launch_pf<3, 3>(p, smem, s);
        case 0x55: return launch_pf<5, 5>(p, smem, s);
        case 0x66: return launch_pf<6, 6>(p, smem, s);
        case 0x65: return launch_pf<6, 5>(p, smem, s);
        case 0x54: return launch_pf<5, 4>(p, smem, s);
        case 0x32: return launch_pf<3, 2>(p, smem, s);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace kvarn
