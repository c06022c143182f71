// KVarN decode step for sm_103a: append, seal and split-K decode attention in one
// persistent launch.
//
// Method (anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", sections 1
// and 2.1): the first 128 tokens (sink) and the partial newest group (tail) are read
// exact in fp16 with the unrotated query; every sealed group is read straight from
// its packed record with the query rotated by the same Hadamard matrix; the sealed
// part of the output is accumulated in the rotated frame and rotated back once per
// output row. A group is sealed at the moment its last token arrives, so a step whose
// new token completes a group seals it first and attends to the sealed record.
//
// Work split. Every (sequence, KV head) pair is a block of scheduling units: one
// exact item, one seal item if the step seals a group, and one unit per sealed group.
// The units of all blocks are cut into equal contiguous ranges, one per CTA, so that
// every CTA streams the same number of records. Each CTA writes one partial softmax
// state (running max, sum, accumulator) per block it touches; the last CTA to finish a
// block (atomic ticket, no waiting) merges the partials, rotates the sealed
// accumulator back, adds the exact part and writes the fp16 output.
//
// Sealed-group stream. One producer thread copies whole group-pair records (K record
// then V record, contiguous in the pool) into a ring of shared-memory stages with
// cp.async.bulk; eight consumer warps take the stages round robin. For a group with
// codes q, token scales a, channel scales c and grid (m, delta), the score of token t
// is  scale * a_t * (delta * sum_j (q'_j c_j) q_tj + m * sum_j q'_j c_j)  with q' the
// rotated query, and the rotated output accumulates
//   c_j * (delta_V * sum_t w_t qV_jt + m_V * sum_t w_t),  w_t = p_t aV_t.
// Both inner sums are dense 128 x 128 x (4 heads) contractions on the raw integer
// codes, done with mma.sync m16n8k16 (f16 in, f32 accumulate). The codes become f16
// operands by masking alone: a code placed in the low mantissa bits of a half is
// the exact subnormal value code * 2^(e-24); the power of two is folded into the
// other operand. The query side is split into f16 high and low parts in the eight
// columns of the MMA (4 heads x 2), which keeps the logits at about fp32 accuracy.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kvarn_dev.cuh"

namespace kvarn {

namespace {

constexpr int kEV = 13;      // weight operand exponent: |B| < 2^14
constexpr int kXbHead = 88;  // exchange buffer words per head (bank-conflict-free stride)
constexpr int kXbWarp = 4 * kXbHead;
constexpr int kWarps = kDecodeThreads / 32;  // 12
constexpr int kMaxDevices = 64;
#define kNegInf (-__int_as_float(0x7f800000))

template <int B>
struct Codes {
    static constexpr int CPW = 32 / B;   // codes per 32-bit word
    static constexpr int HALF = CPW / 2; // partner code distance (low half -> high half)
    static constexpr int NWIN = 10 / B;  // codes of a 16-bit half that fit in the f16 mantissa
    __host__ __device__ static constexpr int sh(int x) { return (x / NWIN) * NWIN * B; }
    __host__ __device__ static constexpr int ex(int x) { return (x % NWIN) * B; }
    __host__ __device__ static constexpr uint32_t mask(int x) { return (((1u << B) - 1u) << ex(x)) * 0x10001u; }
};

template <int B>
__device__ __forceinline__ void load_chunk(const uint8_t* p, uint32_t (&w)[B]) {
    if constexpr (B == 2) {
        uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x;
        w[1] = v.y;
    } else if constexpr (B == 4) {
        uint4 v = *reinterpret_cast<const uint4*>(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
        uint4 v0 = reinterpret_cast<const uint4*>(p)[0];
        uint4 v1 = reinterpret_cast<const uint4*>(p)[1];
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
    }
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// QK row mapping: row g (0..7) of M tile mt holds token tok_row(mt, g) and row g + 8
// holds that token + HALF_V, so the two scores of a thread are a V code pair.
template <int VB>
__device__ __forceinline__ int tok_row(int mt, int g) {
    constexpr int CPW = 32 / VB, HALF = CPW / 2;
    return CPW * (mt * (16 / CPW) + g / HALF) + g % HALF;
}

__device__ __forceinline__ int64_t covering(int64_t u, int64_t U, int64_t P) { return ((u + 1) * P + U - 1) / U - 1; }

struct Item {
    int type;  // 1 exact, 2 seal, 3 chunk of sealed groups
    int ci;    // index of the sequence in the call
    int kvh;
    int g0, g1;
};

// Next item of this CTA's unit range [u, hi); advances u.
__device__ bool next_item(const DecodeParams& p, int64_t& u, int64_t hi, Item& it) {
    while (u < hi) {
        int lo = 0, up = p.n_seqs - 1;
        while (lo < up) {
            int mid = (lo + up + 1) >> 1;
            if (p.seqs[mid].unit_begin <= u) lo = mid; else up = mid - 1;
        }
        const SeqEntry& e = p.seqs[lo];
        const int per = e.w_exact + e.w_seal + e.n_groups;
        const int64_t rel = u - e.unit_begin;
        const int kvh = (int)(rel / per);
        const int off = (int)(rel % per);
        const int64_t blk0 = e.unit_begin + (int64_t)kvh * per;
        if (off < e.w_exact) {  // exact sub-item off / w_sub (g0 holds its index)
            const int sub = off / e.w_sub;
            u = blk0 + (int64_t)(sub + 1) * e.w_sub;
            if (off % e.w_sub == 0) { it = Item{1, lo, kvh, sub, 0}; return true; }
            continue;
        }
        if (off < e.w_exact + e.w_seal) {
            u = blk0 + e.w_exact + e.w_seal;
            if (off == e.w_exact) { it = Item{2, lo, kvh, e.seal_group, e.seal_group + 1}; return true; }
            continue;
        }
        const int gs = off - e.w_exact - e.w_seal;
        const int64_t end = min(hi, blk0 + per);
        it = Item{3, lo, kvh, gs, gs + (int)(end - u)};
        u = end;
        return true;
    }
    return false;
}

// Per-warp shared memory of a worker warp: exchange buffer, query operand table,
// rotated (or, in the exact part, raw) query, per-head query maxima.
constexpr int kWarpRegion = kXbWarp * 4 + 8 * 32 * 16 + 512 * 4 + 16;

struct WarpSmem {
    uint8_t* kstage;   // K record of the warp's current group
    uint8_t* vstage;   // V record of the warp's current group
    uint64_t* full_k;  // completes when a K record has landed
    uint64_t* full_v;
    float* xb;         // [4][kXbHead] half2 words
    float4* bqs;       // [8][32] lane operand bases
    float* qrot;       // [4][128]
    float* qmax;       // [4]
};

__device__ __forceinline__ float* partial_ptr(const DecodeParams& p, int blk, int slot) {
    return reinterpret_cast<float*>(p.base + p.lay.partials) + ((size_t)blk * kPartialSlots + slot) * kPartialFloats;
}

__device__ __forceinline__ int32_t* err_word(const DecodeParams& p) {
    return reinterpret_cast<int32_t*>(p.base + p.lay.err);
}

// 128-point Hadamard transform of a vector held by one warp, 4 consecutive values
// per lane; scaled by 1/sqrt(128).
__device__ __forceinline__ void warp_fwht128(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
    for (int b = 1; b < 32; b <<= 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float o = __shfl_xor_sync(0xffffffffu, v[e], b);
            v[e] = (lane & b) ? (o - v[e]) : (v[e] + o);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] *= kInvSqrt128;
}

__device__ __forceinline__ int64_t workers(const DecodeParams& p) { return (int64_t)p.grid * p.warps; }

// Expected number of partials of block (entry e, kvh) in this call; first worker of its groups.
__device__ int expected_partials(const DecodeParams& p, const SeqEntry& e, int kvh, int64_t* first_worker) {
    const int per = e.w_exact + e.w_seal + e.n_groups;
    const int64_t g0u = e.unit_begin + (int64_t)kvh * per + e.w_exact + e.w_seal;
    const int64_t W = workers(p);
    int n = e.w_exact / e.w_sub + (e.w_seal > 0 ? 1 : 0);
    const int64_t f = covering(g0u, p.units_total, W);
    if (e.n_groups > 0) n += (int)(covering(g0u + e.n_groups - 1, p.units_total, W) - f + 1);
    if (first_worker) *first_worker = f;
    return n;
}

// The last worker of a block merges every partial of this call, rotates the sealed
// accumulator back once and writes the fp16 output. One warp; lane l owns channels
// 4l..4l+3 of every head.
__device__ void final_merge_warp(const DecodeParams& p, int ci, int kvh, int lane) {
    const SeqEntry& e = p.seqs[ci];
    const int blk = e.seq * p.hkv + kvh;
    // headers of slots lane and 32 + lane
    float mh[2][4], lh[2][4];
    bool val[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int sidx = 32 * k + lane;
        val[k] = false;
#pragma unroll
        for (int h = 0; h < 4; ++h) { mh[k][h] = kNegInf; lh[k][h] = 0.f; }
        if (sidx < kPartialSlots) {
            const float* P = partial_ptr(p, blk, sidx);
            val[k] = (uint32_t)__float_as_int(__ldcg(P)) == p.epoch;
            if (val[k]) {
                const float4 m4 = __ldcg(reinterpret_cast<const float4*>(P + 4));
                const float4 l4 = __ldcg(reinterpret_cast<const float4*>(P + 8));
                mh[k][0] = m4.x; mh[k][1] = m4.y; mh[k][2] = m4.z; mh[k][3] = m4.w;
                lh[k][0] = l4.x; lh[k][1] = l4.y; lh[k][2] = l4.z; lh[k][3] = l4.w;
            }
        }
    }
    float M[4], L[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        float m = fmaxf(mh[0][h], mh[1][h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        M[h] = m;
    }
    float wt[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int h = 0; h < 4; ++h) wt[k][h] = (mh[k][h] == kNegInf) ? 0.f : exp2f(mh[k][h] - M[h]);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        float l = wt[0][h] * lh[0][h] + wt[1][h] * lh[1][h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        L[h] = l;
    }
    float ex[4][4], rot[4][4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) ex[h][c] = rot[h][c] = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        unsigned mask = __ballot_sync(0xffffffffu, val[k]);
        while (mask) {
            const int src = __ffs(mask) - 1;
            mask &= mask - 1;
            const int sidx = 32 * k + src;
            const float* P = partial_ptr(p, blk, sidx);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float w = __shfl_sync(0xffffffffu, wt[k][h], src);
                const float4 a = __ldcg(reinterpret_cast<const float4*>(P + 12 + 128 * h + 4 * lane));
                if (sidx < kMaxExactSubs) {
                    ex[h][0] = fmaf(w, a.x, ex[h][0]); ex[h][1] = fmaf(w, a.y, ex[h][1]);
                    ex[h][2] = fmaf(w, a.z, ex[h][2]); ex[h][3] = fmaf(w, a.w, ex[h][3]);
                } else {
                    rot[h][0] = fmaf(w, a.x, rot[h][0]); rot[h][1] = fmaf(w, a.y, rot[h][1]);
                    rot[h][2] = fmaf(w, a.z, rot[h][2]); rot[h][3] = fmaf(w, a.w, rot[h][3]);
                }
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        warp_fwht128(rot[h], lane);
        if (h < p.r) {
            const float inv = L[h] > 0.f ? 1.0f / L[h] : 0.f;
            const __half2 o0 = __floats2half2_rn((ex[h][0] + rot[h][0]) * inv, (ex[h][1] + rot[h][1]) * inv);
            const __half2 o1 = __floats2half2_rn((ex[h][2] + rot[h][2]) * inv, (ex[h][3] + rot[h][3]) * inv);
            uint16_t* out = p.out + ((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 + 4 * lane;
            *reinterpret_cast<uint2*>(out) = make_uint2(h2_bits(o0), h2_bits(o1));
        }
    }
}

// Publish a partial written by this warp; the last of the block's partials merges.
__device__ void publish_warp(const DecodeParams& p, int ci, int kvh, int lane) {
    __threadfence();
    __syncwarp();
    const SeqEntry& e = p.seqs[ci];
    const int blk = e.seq * p.hkv + kvh;
    int last = 0;
    if (lane == 0) {
        const int expect = expected_partials(p, e, kvh, nullptr);
        int32_t* tickets = reinterpret_cast<int32_t*>(p.base + p.lay.tickets);
        const int old = atomicAdd(tickets + blk, 1);
        last = (old == expect - 1);
        if (last) tickets[blk] = 0;
        __threadfence();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) final_merge_warp(p, ci, kvh, lane);
}

// Exact part (sink + tail) of one block, one sub-item of up to 64 tokens on one warp's
// CUDA cores. In a decode step the sub-item holding the new token first writes it to the
// sink or tail (unless it completes a group). Scores: lane = token, its K row read with
// sixteen 16-byte loads, the query from shared memory. P V: lane l owns channels
// 4l..4l+3; the V rows of a 32-token chunk are all requested before use, each a
// coalesced 256-byte warp load, and the probabilities come by shuffle.
__device__ void exact_item_warp(const DecodeParams& p, const WarpSmem& ws, int ci, int kvh, int sub, int lane) {
    const SeqEntry& e = p.seqs[ci];
    const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
    const size_t rows0 = (sl * p.hkv + kvh) * 128;
    const uint16_t* sink_k = reinterpret_cast<const uint16_t*>(p.base + p.lay.sink_k) + rows0 * 128;
    const uint16_t* sink_v = reinterpret_cast<const uint16_t*>(p.base + p.lay.sink_v) + rows0 * 128;
    const uint16_t* tail_k = reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_k) + rows0 * 128;
    const uint16_t* tail_v = reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_v) + rows0 * 128;
    const int n_ex = e.n_sink + e.n_tail;
    const int t_beg = kExactSub * sub, t_end = min(t_beg + kExactSub, n_ex);
    if (e.new_pos >= 0 && e.seal_group < 0) {
        const int x_new = e.new_pos < kSink ? e.new_pos : e.n_sink + (e.new_pos - kSink) % kGroup;
        if (x_new >= t_beg && x_new < t_end) {
            const int side = lane >> 4, chunk = lane & 15;
            const uint16_t* src = (side ? p.v_new : p.k_new) + ((size_t)ci * p.hkv + kvh) * 128;
            const size_t row = e.new_pos < kSink ? (size_t)e.new_pos : (size_t)((e.new_pos - kSink) % kGroup);
            const size_t off =
                (e.new_pos < kSink ? (side ? p.lay.sink_v : p.lay.sink_k) : (side ? p.lay.tail_v : p.lay.tail_k)) +
                (rows0 + row) * 256;
            reinterpret_cast<uint4*>(p.base + off)[chunk] = reinterpret_cast<const uint4*>(src)[chunk];
        }
    }
    float* qraw = ws.qrot;  // [4][128]
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (h < p.r) {
            const uint2 raw = *reinterpret_cast<const uint2*>(p.q + ((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 +
                                                                4 * lane);
            const float2 f0 = __half22float2(bits_h2(raw.x)), f1 = __half22float2(bits_h2(raw.y));
            v = make_float4(f0.x, f0.y, f1.x, f1.y);
        }
        reinterpret_cast<float4*>(qraw + 128 * h)[lane] = v;
    }
    __syncwarp();  // also orders the new token's global write before the reads below
    float m[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
    float lsum[4] = {0.f, 0.f, 0.f, 0.f};
    float acc[4][4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[h][c] = 0.f;
    for (int c0 = t_beg; c0 < t_end; c0 += 32) {
        const int t = c0 + lane;
        float s[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
        if (t < t_end) {
            const uint4* row = reinterpret_cast<const uint4*>(t < e.n_sink ? sink_k + (size_t)t * 128
                                                                          : tail_k + (size_t)(t - e.n_sink) * 128);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 kv[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) kv[c] = row[8 * half + c];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const __half2* hp = reinterpret_cast<const __half2*>(&kv[c]);
                    float kf[8];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const float2 f = __half22float2(hp[q2]);
                        kf[2 * q2] = f.x;
                        kf[2 * q2 + 1] = f.y;
                    }
                    const int cc = 8 * half + c;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float4 qa = reinterpret_cast<const float4*>(qraw + 128 * h + 8 * cc)[0];
                        const float4 qb = reinterpret_cast<const float4*>(qraw + 128 * h + 8 * cc)[1];
                        d[h] = fmaf(kf[0], qa.x, d[h]); d[h] = fmaf(kf[1], qa.y, d[h]);
                        d[h] = fmaf(kf[2], qa.z, d[h]); d[h] = fmaf(kf[3], qa.w, d[h]);
                        d[h] = fmaf(kf[4], qb.x, d[h]); d[h] = fmaf(kf[5], qb.y, d[h]);
                        d[h] = fmaf(kf[6], qb.z, d[h]); d[h] = fmaf(kf[7], qb.w, d[h]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) s[h] = d[h] * p.scale_log2;
        }
        float pr[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float cm = s[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            const float mn = fmaxf(m[h], cm);
            const float corr = (m[h] == kNegInf) ? 0.f : exp2f(m[h] - mn);
            m[h] = mn;
            pr[h] = (t < t_end) ? exp2f(s[h] - mn) : 0.f;
            lsum[h] = fmaf(lsum[h], corr, pr[h]);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[h][c] *= corr;
        }
        const int nt = min(32, t_end - c0);
        // V rows of the chunk, 16 requests in flight at a time
#pragma unroll
        for (int j0 = 0; j0 < 32; j0 += 16) {
            if (j0 >= nt) break;
            uint2 vv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int tt = c0 + j0 + j;
                vv[j] = make_uint2(0u, 0u);
                if (j0 + j < nt) {
                    const uint16_t* row =
                        tt < e.n_sink ? sink_v + (size_t)tt * 128 : tail_v + (size_t)(tt - e.n_sink) * 128;
                    vv[j] = reinterpret_cast<const uint2*>(row)[lane];
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float2 va = __half22float2(bits_h2(vv[j].x)), vb = __half22float2(bits_h2(vv[j].y));
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float pj = __shfl_sync(0xffffffffu, pr[h], j0 + j);
                    acc[h][0] = fmaf(pj, va.x, acc[h][0]);
                    acc[h][1] = fmaf(pj, va.y, acc[h][1]);
                    acc[h][2] = fmaf(pj, vb.x, acc[h][2]);
                    acc[h][3] = fmaf(pj, vb.y, acc[h][3]);
                }
            }
        }
    }
    float* P = partial_ptr(p, e.seq * p.hkv + kvh, sub);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        float l = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        reinterpret_cast<float4*>(P + 12 + 128 * h)[lane] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        if (lane == 0) {
            P[4 + h] = m[h];
            P[8 + h] = l;
        }
    }
    if (lane == 0) P[0] = __int_as_float((int)p.epoch);
    publish_warp(p, ci, kvh, lane);
}

// Rotate the query of a block (one warp): qrot = (q H) / max|q H| per head, qmax = that
// max; then the table of each lane's query operand base q_hat(head g>>1, channel) * 2^-ex
// in the pair order of its MMA fragments.
template <int KB>
__device__ void setup_query_warp(const DecodeParams& p, const WarpSmem& ws, int ci, int kvh, int lane) {
    using CK = Codes<KB>;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (h < p.r) {
            const uint16_t* q = p.q + ((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 + 4 * lane;
            const uint2 raw = *reinterpret_cast<const uint2*>(q);
            const float2 f0 = __half22float2(bits_h2(raw.x)), f1 = __half22float2(bits_h2(raw.y));
            v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
        }
        warp_fwht128(v, lane);
        float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (mx == 0.f) mx = 1.f;
        const float inv = 1.0f / mx;
        reinterpret_cast<float4*>(ws.qrot + 128 * h)[lane] = make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
        if (lane == 0) ws.qmax[h] = mx;
    }
    __syncwarp();
    const int g = lane >> 2, tq = lane & 3;
    const float* qh = ws.qrot + 128 * (g >> 1);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float vals[4];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
            const int P = 2 * q + e2;
            const int x = P % CK::HALF;
            const int c0 = 32 * tq + CK::CPW * (P / CK::HALF) + x;
            const float sc = __int_as_float((127 - CK::ex(x)) << 23);  // 2^-ex
            vals[2 * e2] = qh[c0] * sc;
            vals[2 * e2 + 1] = qh[c0 + CK::HALF] * sc;
        }
        ws.bqs[q * 32 + lane] = make_float4(vals[0], vals[1], vals[2], vals[3]);
    }
    __syncwarp();
}

struct WarpState {
    float m, l;
    float acc[8][2];
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Operand of pair P from a thread's code words (the pair of codes x, x + HALF of
// word P / HALF, masked into the low mantissa bits of two halves).
template <int B>
__device__ __forceinline__ uint32_t pair_operand(const uint32_t* w, int P) {
    using C = Codes<B>;
    const int word = P / C::HALF, x = P % C::HALF;
    return (w[word] >> C::sh(x)) & C::mask(x);
}

// Tiles processed together, k-step outer: TG independent MMA chains, TG * 2 * B
// code words live in registers.
template <int B>
struct TileGroup {
    static constexpr int TG = B == 8 ? 2 : 4;
};

// Process one sealed group: K record at krec, V record at vrec (both in shared memory).
// k_done() is called once the K record has been read completely (its stage may then be
// refilled); v_wait() waits for the V record before it is first read.
template <int KB, int VB, class KDone, class VWait>
__device__ __forceinline__ void process_group(const DecodeParams& p, const uint8_t* krec, const uint8_t* vrec,
                                              const float4* bqs, float qm, float* xb, WarpState& st, int g, int tq,
                                              int lane, KDone k_done, VWait v_wait) {
    using CK = Codes<KB>;
    using CV = Codes<VB>;
    const float dK = *reinterpret_cast<const float*>(krec);
    const float mK = *reinterpret_cast<const float*>(krec + 4);
    const uint16_t* aK = reinterpret_cast<const uint16_t*>(krec + 16);
    // ---- query operand of this group: q_hat * c_K * 2^-ex, split into f16 high / low parts.
    // |q_hat| <= 1, c_K <= 65504 and 2^-ex <= 1, so the operand can never overflow f16.
    uint32_t bk[16];
    float sumqc;
    {
        const uint4* cp = reinterpret_cast<const uint4*>(krec + 272 + 64 * tq);
        uint32_t cw[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 v = cp[k];
            cw[4 * k] = v.x; cw[4 * k + 1] = v.y; cw[4 * k + 2] = v.z; cw[4 * k + 3] = v.w;
        }
        float bq[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = bqs[q * 32 + lane];
            bq[4 * q] = v.x; bq[4 * q + 1] = v.y; bq[4 * q + 2] = v.z; bq[4 * q + 3] = v.w;
        }
        const bool lo_part = (g & 1) != 0;
        float sum = 0.f;
#pragma unroll
        for (int P = 0; P < 16; ++P) {
            const int x = P % CK::HALF;
            const int c0 = CK::CPW * (P / CK::HALF) + x;
            const int c1 = c0 + CK::HALF;
            const float f0 = bq[2 * P] * __half2float(reinterpret_cast<const __half*>(cw)[c0]);
            const float f1 = bq[2 * P + 1] * __half2float(reinterpret_cast<const __half*>(cw)[c1]);
            const __half2 hi = __floats2half2_rn(f0, f1);
            const float2 hf = __half22float2(hi);
            const uint32_t lo = h2_bits(__floats2half2_rn(f0 - hf.x, f1 - hf.y));
            bk[P] = lo_part ? lo : h2_bits(hi);
            const float sc = __int_as_float((127 + CK::ex(x)) << 23);  // 2^ex: back to q_hat * c_K
            sum = fmaf(f0 + f1, sc, sum);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        // lane 8 tq holds the sum of head tq (its column head is (2 tq) >> 1 = tq)
        sumqc = __shfl_sync(0xffffffffu, sum, 8 * tq);
    }
    // ---- scores of the 16 tokens this thread holds (head tq)
    float S[8][2];
    {
        constexpr int TG = TileGroup<KB>::TG;
#pragma unroll
        for (int t0g = 0; t0g < 8; t0g += TG) {
            uint32_t w0[TG][KB], w1[TG][KB];
#pragma unroll
            for (int i = 0; i < TG; ++i) {
                const int t0 = tok_row<VB>(t0g + i, g), t1 = t0 + CV::HALF;
                load_chunk<KB>(krec + 528 + t0 * 16 * KB + 4 * KB * tq, w0[i]);
                load_chunk<KB>(krec + 528 + t1 * 16 * KB + 4 * KB * tq, w1[i]);
            }
            float c[TG][4];
#pragma unroll
            for (int i = 0; i < TG; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int i = 0; i < TG; ++i)
                    mma16816(c[i], pair_operand<KB>(w0[i], 2 * ks), pair_operand<KB>(w1[i], 2 * ks),
                             pair_operand<KB>(w0[i], 2 * ks + 1), pair_operand<KB>(w1[i], 2 * ks + 1), bk[2 * ks],
                             bk[2 * ks + 1]);
            }
#pragma unroll
            for (int i = 0; i < TG; ++i) {
                S[t0g + i][0] = c[i][0] + c[i][1];
                S[t0g + i][1] = c[i][2] + c[i][3];
            }
        }
    }
    const float alpha = p.scale_log2 * qm * dK * 16777216.0f;  // codes enter as code * 2^(ex-24)
    const float beta = p.scale_log2 * qm * mK * sumqc;
    float gmax = kNegInf;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int t0 = tok_row<VB>(mt, g), t1 = t0 + CV::HALF;
        S[mt][0] = half_bits_to_float(aK[t0]) * fmaf(alpha, S[mt][0], beta);
        S[mt][1] = half_bits_to_float(aK[t1]) * fmaf(alpha, S[mt][1], beta);
        gmax = fmaxf(gmax, fmaxf(S[mt][0], S[mt][1]));
    }
    __syncwarp();
    k_done();   // the K record is no longer read
    v_wait();
    const float dV = *reinterpret_cast<const float*>(vrec);
    const float mV = *reinterpret_cast<const float*>(vrec + 4);
    const uint16_t* aV = reinterpret_cast<const uint16_t*>(vrec + 16);
    const uint16_t* cV = reinterpret_cast<const uint16_t*>(vrec + 272);
    float av[8][2];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int t0 = tok_row<VB>(mt, g), t1 = t0 + CV::HALF;
        av[mt][0] = half_bits_to_float(aV[t0]);
        av[mt][1] = half_bits_to_float(aV[t1]);
    }
    // largest V token scale of the group from its bit patterns (all >= 0): lane l reads 4
    uint32_t amaxb;
    {
        const uint2 ab = reinterpret_cast<const uint2*>(aV)[lane];
        amaxb = __vmaxu2(ab.x, ab.y);
        amaxb = max(amaxb & 0xffffu, amaxb >> 16);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amaxb = max(amaxb, __shfl_xor_sync(0xffffffffu, amaxb, o));
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    const float mnew = fmaxf(st.m, gmax);
    const float corr = fast_exp2(st.m - mnew);
    st.m = mnew;
    // rho = 2^(15 - e) puts every aV * rho in [0, 2): e = biased exponent of the largest aV
    const int ebits = max((int)(amaxb >> 10) & 31, 1);
    const float rho = __int_as_float((127 + 15 - ebits) << 23);
    const int xv = g % CV::HALF;
    const float sv = __int_as_float((127 + kEV - CV::ex(xv)) << 23) * rho;  // 2^(EV - ex) * rho
    const float svi = __int_as_float((127 - kEV + CV::ex(xv)) << 23);       // 2^(ex - EV)
    float lsum = 0.f, wsum = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const float p0 = fast_exp2(S[mt][0] - mnew), p1 = fast_exp2(S[mt][1] - mnew);
        lsum += p0 + p1;
        const __half2 wh = __floats2half2_rn(p0 * av[mt][0] * sv, p1 * av[mt][1] * sv);
        const float2 wf = __half22float2(wh);
        wsum = fmaf(wf.x + wf.y, svi, wsum);
        reinterpret_cast<uint32_t*>(xb)[kXbHead * tq + 20 * (mt >> 1) + 8 * (mt & 1) + g] = h2_bits(wh);
    }
    st.l = fmaf(st.l, corr, lsum);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    __syncwarp();
    uint32_t bv[16];
    {
        const uint4* src = reinterpret_cast<const uint4*>(xb + kXbHead * (g >> 1) + 20 * tq);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 v = src[k];
            bv[4 * k] = v.x; bv[4 * k + 1] = v.y; bv[4 * k + 2] = v.z; bv[4 * k + 3] = v.w;
        }
    }
    __syncwarp();
    // ---- P V in the rotated frame
    const float gam = dV * (float)(1 << (24 - kEV)) / rho;
    const float del = mV * wsum / rho;
    {
        constexpr int TG = TileGroup<VB>::TG;
#pragma unroll
        for (int m0 = 0; m0 < 8; m0 += TG) {
            uint32_t w0[TG][VB], w1[TG][VB];
#pragma unroll
            for (int i = 0; i < TG; ++i) {
                const int c0 = 16 * (m0 + i) + g;
                load_chunk<VB>(vrec + 528 + c0 * 16 * VB + 4 * VB * tq, w0[i]);
                load_chunk<VB>(vrec + 528 + (c0 + 8) * 16 * VB + 4 * VB * tq, w1[i]);
            }
            float d[TG][4];
#pragma unroll
            for (int i = 0; i < TG; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int i = 0; i < TG; ++i)
                    mma16816(d[i], pair_operand<VB>(w0[i], 2 * ks), pair_operand<VB>(w1[i], 2 * ks),
                             pair_operand<VB>(w0[i], 2 * ks + 1), pair_operand<VB>(w1[i], 2 * ks + 1), bv[2 * ks],
                             bv[2 * ks + 1]);
            }
#pragma unroll
            for (int i = 0; i < TG; ++i) {
                const int mt = m0 + i;
                const int c0 = 16 * mt + g;
                st.acc[mt][0] = fmaf(st.acc[mt][0], corr, half_bits_to_float(cV[c0]) * fmaf(gam, d[i][0], del));
                st.acc[mt][1] = fmaf(st.acc[mt][1], corr, half_bits_to_float(cV[c0 + 8]) * fmaf(gam, d[i][2], del));
            }
        }
    }
}

// Write one warp's softmax state of an item as a partial (lane (g, tq) holds head tq at
// channels 16 mt + g and 16 mt + g + 8).
__device__ void write_partial_warp(const DecodeParams& p, const WarpState& st, int blk, int slot, int lane) {
    const int g = lane >> 2, tq = lane & 3;
    float l = st.l;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    float* P = partial_ptr(p, blk, slot);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        P[12 + 128 * tq + 16 * mt + g] = st.acc[mt][0];
        P[12 + 128 * tq + 16 * mt + g + 8] = st.acc[mt][1];
    }
    if (g == 0) {
        P[4 + tq] = st.m;
        P[8 + tq] = l;
    }
    if (lane == 0) P[0] = __int_as_float((int)p.epoch);
}

__device__ __forceinline__ const uint8_t* group_src(const DecodeParams& p, int seq, int kvh, int g) {
    const int32_t* table = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table);
    int slot = table[((size_t)seq * p.num_layers + p.layer) * p.max_groups + g];
    if (slot < 0 || slot >= p.pool_slots) {
        atomicOr(err_word(p), kErrBadSlot);
        slot = 0;
    }
    return p.base + p.lay.pool + (size_t)slot * p.slot_bytes + (size_t)kvh * (p.rec_k + p.rec_v);
}

struct SealRows {
    const uint16_t* tail;  // rows 0..126
    const uint16_t* last;  // row 127: the new token
    __device__ const uint16_t* operator()(int i) const { return i < 127 ? tail + 128 * i : last; }
};

// Walks a worker's sealed groups in stream order to find the record of group number gn
// (0, 1, ... over the chunk and seal items of the worker's unit range, in item order).
struct GroupCursor {
    int64_t u;       // unit cursor of the item walk
    Item it;         // current chunk / seal item
    uint32_t base;   // group number of the item's first group
    bool valid;
    __device__ void init(int64_t lo) { u = lo; base = 0; valid = false; it.g0 = it.g1 = 0; }
    // record pair address of group gn (gn never decreases between calls); null past the end
    __device__ const uint8_t* src(const DecodeParams& p, int64_t hi, uint32_t gn) {
        for (;;) {
            if (valid && gn < base + (uint32_t)(it.g1 - it.g0)) break;
            if (valid) base += (uint32_t)(it.g1 - it.g0);
            valid = false;
            Item n;
            bool found = false;
            while (next_item(p, u, hi, n)) {
                if (n.type != 1) { found = true; break; }
            }
            if (!found) return nullptr;
            it = n;
            valid = true;
        }
        const SeqEntry& e = p.seqs[it.ci];
        const int pair = p.rec_k + p.rec_v;
        if (it.type == 2)
            return p.base + p.lay.pool + (size_t)e.seal_slot * p.slot_bytes + (size_t)it.kvh * pair;
        return group_src(p, e.seq, it.kvh, it.g0 + (int)(gn - base));
    }
};

// One CTA of up to 12 worker warps per SM. Every warp is an independent worker with its
// own contiguous range of scheduling units and a one-group stage split into a K half and
// a V half: the next group's K record is requested as soon as the current QK is done,
// its V record as soon as the current PV is done. The CTA only synchronises once, after
// the seal items of its range (run first by 8 warps, their scratch on the stage area).
template <int KB, int VB>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int pair = p.rec_k + p.rec_v;
    const int nw = p.warps;
    size_t ring = (size_t)nw * pair;
    if (ring < sizeof(SealSmem)) ring = sizeof(SealSmem);
    ring = (ring + 127) & ~(size_t)127;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + ring);  // full_k[12], full_v[12]
    uint8_t* regions = smem_raw + ring + 256;
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    if (t == 0) {
        for (int k = 0; k < 2 * kWarps; ++k) mbar_init(bars + k, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t U = p.units_total, W = workers(p), b = blockIdx.x;
    int32_t* err = err_word(p);

    // ---- 1. seal the groups completed by this step's tokens (before any prefetch)
    {
        const int64_t clo = b * nw * U / W, chi = (b + 1) * nw * U / W;
        SealSmem& S = *reinterpret_cast<SealSmem*>(smem_raw);
        bool sealed_any = false;
        int64_t u = clo;
        Item it;
        while (next_item(p, u, chi, it)) {
            if (it.type != 2) continue;
            const SeqEntry& e = p.seqs[it.ci];
            const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
            const size_t rows0 = (sl * p.hkv + it.kvh) * 128;
            uint8_t* dst = p.base + p.lay.pool + (size_t)e.seal_slot * p.slot_bytes + (size_t)it.kvh * pair;
            if (t < kSealThreads) {  // the seal runs on 8 warps (barrier 2)
                SealRows rk{reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_k) + rows0 * 128,
                            p.k_new + ((size_t)it.ci * p.hkv + it.kvh) * 128};
                seal_matrix(rk, p.k_bits, 0, p.iters, dst, nullptr, S, 2);
                SealRows rv{reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_v) + rows0 * 128,
                            p.v_new + ((size_t)it.ci * p.hkv + it.kvh) * 128};
                seal_matrix(rv, p.v_bits, 1, p.iters, dst + p.rec_k, nullptr, S, 2);
            }
            if (t == 0 && it.kvh == 0) {
                int32_t* table = reinterpret_cast<int32_t*>(p.base + p.lay.block_table);
                table[sl * p.max_groups + e.seal_group] = e.seal_slot;
            }
            sealed_any = true;
        }
        if (sealed_any) fence_proxy_async_global();  // the records just written are read by bulk copies
        __syncthreads();
    }
    if (w >= nw) return;

    // ---- 2. this warp's worker range
    const int64_t gw = b * nw + w;
    const int64_t lo = gw * U / W, hi = (gw + 1) * U / W;
    WarpSmem ws;
    ws.kstage = smem_raw + (size_t)w * pair;
    ws.vstage = ws.kstage + p.rec_k;
    ws.full_k = bars + w;
    ws.full_v = bars + kWarps + w;
    {
        uint8_t* r = regions + (size_t)w * kWarpRegion;
        ws.xb = reinterpret_cast<float*>(r);
        ws.bqs = reinterpret_cast<float4*>(r + kXbWarp * 4);
        ws.qrot = reinterpret_cast<float*>(r + kXbWarp * 4 + 8 * 32 * 16);
        ws.qmax = reinterpret_cast<float*>(r + kXbWarp * 4 + 8 * 32 * 16 + 512 * 4);
    }
    GroupCursor cur;
    cur.init(lo);
    const uint8_t* next_src = nullptr;  // lane 0: record pair of the next group to request
    if (lane == 0) {
        next_src = cur.src(p, hi, 0);
        if (next_src) {
            mbar_arrive_expect_tx(ws.full_k, p.rec_k);
            bulk_g2s(ws.kstage, next_src, p.rec_k, ws.full_k);
            mbar_arrive_expect_tx(ws.full_v, p.rec_v);
            bulk_g2s(ws.vstage, next_src + p.rec_k, p.rec_v, ws.full_v);
        }
    }

    const int g = lane >> 2, tq = lane & 3;
    int64_t u = lo;
    Item it;
    uint32_t n = 0;  // groups consumed by this warp
    while (next_item(p, u, hi, it)) {
        const SeqEntry& e = p.seqs[it.ci];
        const int blk = e.seq * p.hkv + it.kvh;
        if (it.type == 1) {
            exact_item_warp(p, ws, it.ci, it.kvh, it.g0, lane);
            continue;
        }
        int slot;
        if (it.type == 2) {
            slot = kSlotSeal;
        } else {
            int64_t first;
            expected_partials(p, e, it.kvh, &first);
            slot = kSlotChunk0 + (int)(gw - first);
            if (slot >= kPartialSlots) {  // cannot happen with the host's schedule
                if (lane == 0) atomicOr(err, kErrSpan);
                slot = kPartialSlots - 1;
            }
        }
        setup_query_warp<KB>(p, ws, it.ci, it.kvh, lane);
        const float qm = ws.qmax[tq];
        WarpState st;
        st.m = kNegInf;
        st.l = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) st.acc[mt][0] = st.acc[mt][1] = 0.f;
        const uint32_t cnt = (uint32_t)(it.g1 - it.g0);
        for (uint32_t k = 0; k < cnt; ++k, ++n) {
            const uint32_t par = n & 1;
            mbar_wait(ws.full_k, par, err);
            auto k_done = [&]() {
                if (lane == 0) {
                    next_src = cur.src(p, hi, n + 1);
                    if (next_src) {
                        mbar_arrive_expect_tx(ws.full_k, p.rec_k);
                        bulk_g2s(ws.kstage, next_src, p.rec_k, ws.full_k);
                    }
                }
            };
            auto v_wait = [&]() { mbar_wait(ws.full_v, par, err); };
            process_group<KB, VB>(p, ws.kstage, ws.vstage, ws.bqs, qm, ws.xb, st, g, tq, lane, k_done, v_wait);
            __syncwarp();
            if (lane == 0 && next_src) {
                mbar_arrive_expect_tx(ws.full_v, p.rec_v);
                bulk_g2s(ws.vstage, next_src + p.rec_k, p.rec_v, ws.full_v);
            }
        }
        write_partial_warp(p, st, blk, slot, lane);
        publish_warp(p, it.ci, it.kvh, lane);
    }
    // Normally every copy was waited for above. After a wait that gave up, let the
    // copies still in flight land (bounded) before the CTA's shared memory goes away.
    if (lane == 0 && (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout)) {
        const uint64_t t0 = global_ns();
        if (n > 0) {
            while (!mbar_try_wait(ws.full_k, (n - 1) & 1) && global_ns() - t0 < kWaitLimitNs) {
            }
            while (!mbar_try_wait(ws.full_v, (n - 1) & 1) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

template <int KB, int VB>
int launch_t(const DecodeParams& p, int smem, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             max_optin_smem());
        if (e != cudaSuccess) return (int)e;
        attr = true;
    }
    decode_kernel<KB, VB><<<p.grid, kDecodeThreads, smem, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace

int decode_smem_bytes(int k_bits, int v_bits, int warps, bool with_seal) {
    (void)with_seal;  // the seal scratch aliases the stage area
    size_t pair = record_bytes(k_bits) + record_bytes(v_bits);
    size_t ring = (size_t)warps * pair;
    if (ring < sizeof(SealSmem)) ring = sizeof(SealSmem);
    ring = (ring + 127) & ~(size_t)127;
    return (int)(ring + 256 + (size_t)warps * kWarpRegion);
}

// ---------------------------------------------------------------------------
// Static split-K workspace for kvarn_decode_attention_noalloc: partial softmax states
// and merge tickets of up to kStaticBlocks (sequence, KV head) blocks, 14.3 MB per GPU
// that loads the library, held until the process exits. Host code must not pass the
// symbol itself to a kernel (in host code it names a host-side shadow): the device
// address is fetched once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on it.
constexpr int kStaticBlocks = 128;
static __device__ __align__(256) float kvarn_static_partials[(size_t)kStaticBlocks * kPartialSlots * kPartialFloats];
static __device__ __align__(256) int32_t kvarn_static_tickets[kStaticBlocks];

int static_workspace_blocks() { return kStaticBlocks; }

int static_workspace(void** partials, void** tickets) {
    static std::mutex mu;
    static void* parts[kMaxDevices] = {};
    static void* ticks[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!parts[dev]) {
        void* pp = nullptr;
        void* tp = nullptr;
        e = cudaGetSymbolAddress(&pp, kvarn_static_partials);
        if (e != cudaSuccess) return (int)e;
        e = cudaGetSymbolAddress(&tp, kvarn_static_tickets);
        if (e != cudaSuccess) return (int)e;
        parts[dev] = pp;
        ticks[dev] = tp;
    }
    *partials = parts[dev];
    *tickets = ticks[dev];
    return 0;
}

int clear_static_tickets(void* tickets, void* stream) {
    return (int)cudaMemsetAsync(tickets, 0, sizeof(int32_t) * kStaticBlocks, (cudaStream_t)stream);
}

int launch_decode(const DecodeParams& p, int smem, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    switch (p.k_bits * 16 + p.v_bits) {
        case 0x22: return launch_t<2, 2>(p, smem, s);
        case 0x24: return launch_t<2, 4>(p, smem, s);
        case 0x28: return launch_t<2, 8>(p, smem, s);
        case 0x42: return launch_t<4, 2>(p, smem, s);
        case 0x44: return launch_t<4, 4>(p, smem, s);
        case 0x48: return launch_t<4, 8>(p, smem, s);
        case 0x82: return launch_t<8, 2>(p, smem, s);
        case 0x84: return launch_t<8, 4>(p, smem, s);
        case 0x88: return launch_t<8, 8>(p, smem, s);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace kvarn
