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
constexpr int kMrgFloats = 8 + 512;  // per warp: m[4], l[4], acc[4][128]
constexpr int kWarps = kDecodeThreads / 32;  // 12
constexpr int kConsumers = kDecodeThreads;
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

// pair P (0..15) of a thread's 32-code chunk: word P / HALF, position x = P % HALF;
// the pair holds codes x and x + HALF of that word.
template <int B>
__device__ __forceinline__ void unpack16(const uint32_t (&w)[B], uint32_t (&a)[16]) {
    using C = Codes<B>;
#pragma unroll
    for (int P = 0; P < 16; ++P) {
        const int word = P / C::HALF, x = P % C::HALF;
        a[P] = (w[word] >> C::sh(x)) & C::mask(x);
    }
}

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
        if (off < e.w_exact) {
            u = blk0 + e.w_exact;
            if (off == 0) { it = Item{1, lo, kvh, 0, 0}; return true; }
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

struct Smem {
    uint8_t* stages;
    uint64_t* full;
    float* qrot;    // [4][128] rotated query / its max
    uint4* qtab;    // [3 kinds][4][32 lanes]: query operand table (setup_query)
    float* qmax;    // [4]
    float* xbuf;    // [8 warps][kXbWarp] (half2 words)
    float* mrg;     // [8 warps][kMrgFloats], also exact-part and final-merge scratch
    int* flag;
    SealSmem* seal;
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

// Expected number of partials of block (entry e, kvh) in this call.
__device__ int expected_partials(const DecodeParams& p, const SeqEntry& e, int kvh, int64_t* first_cta) {
    const int per = e.w_exact + e.w_seal + e.n_groups;
    const int64_t g0u = e.unit_begin + (int64_t)kvh * per + e.w_exact + e.w_seal;
    int n = 1 + (e.w_seal > 0 ? 1 : 0);
    int64_t f = covering(g0u, p.units_total, p.grid);
    if (e.n_groups > 0) n += (int)(covering(g0u + e.n_groups - 1, p.units_total, p.grid) - f + 1);
    if (first_cta) *first_cta = f;
    return n;
}

// Last CTA of a block: merge every partial of this call, rotate back, write out.
// The partial headers are read in one parallel round (one thread per slot); the
// accumulators of the valid slots are then read with independent loads.
__device__ void final_merge(const DecodeParams& p, const Smem& sm, int ci, int kvh) {
    const int t = threadIdx.x;
    const SeqEntry& e = p.seqs[ci];
    const int blk = e.seq * p.hkv + kvh;
    float* hdr = sm.mrg + 1536;           // [kPartialSlots][8]: m[4], l[4]
    int* list = reinterpret_cast<int*>(sm.mrg + 1536 + 8 * kPartialSlots);  // [kPartialSlots + 1]
    bool valid = false;
    if (t < kPartialSlots) {
        const float* P = partial_ptr(p, blk, t);
        valid = (uint32_t)__float_as_int(__ldcg(P)) == p.epoch;
        const float4 m4 = __ldcg(reinterpret_cast<const float4*>(P + 4));
        const float4 l4 = __ldcg(reinterpret_cast<const float4*>(P + 8));
        float* H = hdr + 8 * t;
        H[0] = valid ? m4.x : kNegInf; H[1] = valid ? m4.y : kNegInf;
        H[2] = valid ? m4.z : kNegInf; H[3] = valid ? m4.w : kNegInf;
        H[4] = l4.x; H[5] = l4.y; H[6] = l4.z; H[7] = l4.w;
    }
    if (t < 32) {  // warp 0 lists the valid slots among 0..31
        const unsigned vm = __ballot_sync(0xffffffffu, valid);
        if (t == 0) {
            int n = 0;
            for (int k = 0; k < 32; ++k)
                if (vm >> k & 1) list[1 + n++] = k;
            list[0] = n;
        }
    }
    named_bar(1, kConsumers);
    if (t >= 32 && t < kPartialSlots && valid) {  // slots beyond the first warp (rare)
        const int k = atomicAdd(&list[0], 1);
        list[1 + k] = t;
    }
    named_bar(1, kConsumers);
    const int nv = list[0];
    const int h = (t >> 6) & 3, jj = 2 * (t & 63);
    float M = kNegInf;
    for (int k = 0; k < nv; ++k) M = fmaxf(M, hdr[8 * list[1 + k] + h]);
    float l = 0.f, r0 = 0.f, r1 = 0.f, x0 = 0.f, x1 = 0.f;
    if (M != kNegInf) {
#pragma unroll 4
        for (int k = 0; k < nv; ++k) {
            const int sl = list[1 + k];
            const float ms = hdr[8 * sl + h];
            const float w = ms == kNegInf ? 0.f : exp2f(ms - M);
            const float2 a = __ldcg(reinterpret_cast<const float2*>(partial_ptr(p, blk, sl) + 12 + 128 * h + jj));
            l = fmaf(w, hdr[8 * sl + 4 + h], l);
            if (sl == kSlotExact) {
                x0 = fmaf(w, a.x, x0);
                x1 = fmaf(w, a.y, x1);
            } else {
                r0 = fmaf(w, a.x, r0);
                r1 = fmaf(w, a.y, r1);
            }
        }
    }
    float* rot = sm.mrg;        // [4][128]
    float* ex = sm.mrg + 512;   // [4][128]
    float* ls = sm.mrg + 1024;  // [4]
    if (t < 256) {
        rot[128 * h + jj] = r0;
        rot[128 * h + jj + 1] = r1;
        ex[128 * h + jj] = x0;
        ex[128 * h + jj + 1] = x1;
        if ((t & 63) == 0) ls[h] = l;
    }
    named_bar(1, kConsumers);
    const int w = t >> 5, lane = t & 31;
    if (w < 4) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = rot[128 * w + 4 * lane + k];
        warp_fwht128(v, lane);
#pragma unroll
        for (int k = 0; k < 4; ++k) rot[128 * w + 4 * lane + k] = v[k];
    }
    named_bar(1, kConsumers);
    if (t < 256 && h < p.r) {
        const float lh = ls[h];
        const float inv = lh > 0.f ? 1.0f / lh : 0.f;
        __half2 o = __floats2half2_rn((ex[128 * h + jj] + rot[128 * h + jj]) * inv,
                                      (ex[128 * h + jj + 1] + rot[128 * h + jj + 1]) * inv);
        uint16_t* out = p.out + ((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 + jj;
        *reinterpret_cast<__half2*>(out) = o;
    }
}

// Publish a partial (written by all consumer threads before the call) and merge if last.
__device__ void publish(const DecodeParams& p, const Smem& sm, int ci, int kvh) {
    __threadfence();
    named_bar(1, kConsumers);
    const SeqEntry& e = p.seqs[ci];
    const int blk = e.seq * p.hkv + kvh;
    if (threadIdx.x == 0) {
        int expect = expected_partials(p, e, kvh, nullptr);
        int32_t* tickets = reinterpret_cast<int32_t*>(p.base + p.lay.tickets);
        int old = atomicAdd(tickets + blk, 1);
        int last = (old == expect - 1);
        if (last) tickets[blk] = 0;
        __threadfence();
        *sm.flag = last;
    }
    named_bar(1, kConsumers);
    if (*sm.flag) final_merge(p, sm, ci, kvh);
    named_bar(1, kConsumers);
}

// Exact part (sink + tail) of one block on CUDA cores; in a decode step the new token
// is first written to the sink or tail (unless it completes a group). Scores: one
// thread per token, sixteen independent 16-byte loads of its K row. P V: warp w takes
// tokens w, w+8, ...; lane l holds channels 4l..4l+3 of all four heads, so every V row
// is one coalesced 256-byte warp load; the eight warps' sums meet in shared memory.
__device__ void exact_item(const DecodeParams& p, const Smem& sm, int ci, int kvh) {
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const SeqEntry& e = p.seqs[ci];
    const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
    const size_t rows0 = (sl * p.hkv + kvh) * 128;  // first row of this (seq, layer, kv head)
    const uint16_t* sink_k = reinterpret_cast<const uint16_t*>(p.base + p.lay.sink_k) + rows0 * 128;
    const uint16_t* sink_v = reinterpret_cast<const uint16_t*>(p.base + p.lay.sink_v) + rows0 * 128;
    const uint16_t* tail_k = reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_k) + rows0 * 128;
    const uint16_t* tail_v = reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_v) + rows0 * 128;
    if (e.new_pos >= 0 && e.seal_group < 0 && t < 32) {
        const int side = t >> 4, chunk = t & 15;
        const uint16_t* src = (side ? p.v_new : p.k_new) + ((size_t)ci * p.hkv + kvh) * 128;
        size_t row = e.new_pos < kSink ? (size_t)e.new_pos : (size_t)((e.new_pos - kSink) % kGroup);
        size_t off = (e.new_pos < kSink ? (side ? p.lay.sink_v : p.lay.sink_k) : (side ? p.lay.tail_v : p.lay.tail_k)) +
                     (rows0 + row) * 256;
        reinterpret_cast<uint4*>(p.base + off)[chunk] = reinterpret_cast<const uint4*>(src)[chunk];
    }
    float* qraw = sm.xbuf;           // [4][128]
    float* sc = sm.xbuf + 512;       // [4][256]
    float* red = sm.xbuf + 1536;     // [16]
    float* part = sm.mrg;            // [kWarps][4][128]
    for (int k = t; k < 512; k += kConsumers) {
        const int h = k >> 7, j = k & 127;
        qraw[k] = h < p.r ? half_bits_to_float(p.q[((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 + j]) : 0.f;
    }
    named_bar(1, kConsumers);
    const int n_ex = e.n_sink + e.n_tail;
    float s[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
    if (t < n_ex) {
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
                    float2 f = __half22float2(hp[q2]);
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
    if (t < 256) {
#pragma unroll
        for (int h = 0; h < 4; ++h) sc[256 * h + t] = s[h];
    }
    named_bar(1, kConsumers);
    // per-head max and sum: 64 threads per head, 4 entries each (threads >= 256 idle)
    {
        const int h = (t >> 6) & 3, k0 = 4 * (t & 63);
        float m = fmaxf(fmaxf(sc[256 * h + k0], sc[256 * h + k0 + 1]), fmaxf(sc[256 * h + k0 + 2], sc[256 * h + k0 + 3]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0 && t < 256) red[2 * h + (w & 1)] = m;
        named_bar(1, kConsumers);
        m = fmaxf(red[2 * h], red[2 * h + 1]);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float v = sc[256 * h + k0 + k];
            float pv = (m == kNegInf) ? 0.f : exp2f(v - m);
            if (t < 256) sc[256 * h + k0 + k] = pv;
            sum += pv;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0 && t < 256) red[8 + 2 * h + (w & 1)] = sum;
        named_bar(1, kConsumers);
        if ((t & 63) == 0 && t < 256) {
            float* P = partial_ptr(p, e.seq * p.hkv + kvh, kSlotExact);
            P[4 + h] = m;
            P[8 + h] = red[8 + 2 * h] + red[8 + 2 * h + 1];
        }
    }
    // P V
    {
        float acc[4][4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[h][c] = 0.f;
        for (int k0 = w; k0 < n_ex; k0 += 4 * kWarps) {
            uint2 vv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = k0 + kWarps * u;
                vv[u] = make_uint2(0u, 0u);
                if (k < n_ex) {
                    const uint16_t* row = k < e.n_sink ? sink_v + (size_t)k * 128 : tail_v + (size_t)(k - e.n_sink) * 128;
                    vv[u] = reinterpret_cast<const uint2*>(row)[lane];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = k0 + kWarps * u;
                if (k < n_ex) {
                    const float2 va = __half22float2(bits_h2(vv[u].x)), vb = __half22float2(bits_h2(vv[u].y));
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float pk = sc[256 * h + k];
                        acc[h][0] = fmaf(pk, va.x, acc[h][0]);
                        acc[h][1] = fmaf(pk, va.y, acc[h][1]);
                        acc[h][2] = fmaf(pk, vb.x, acc[h][2]);
                        acc[h][3] = fmaf(pk, vb.y, acc[h][3]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 4; ++h)
            *reinterpret_cast<float4*>(part + (w * 4 + h) * 128 + 4 * lane) =
                make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        named_bar(1, kConsumers);
        if (t < 256) {
            const int h = t >> 6, jj = 2 * (t & 63);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < kWarps; ++k) {
                a0 += part[(k * 4 + h) * 128 + jj];
                a1 += part[(k * 4 + h) * 128 + jj + 1];
            }
            float* P = partial_ptr(p, e.seq * p.hkv + kvh, kSlotExact);
            *reinterpret_cast<float2*>(P + 12 + 128 * h + jj) = make_float2(a0, a1);
            if (t == 0) P[0] = __int_as_float((int)p.epoch);
        }
    }
    publish(p, sm, ci, kvh);
}

// Rotate the query of a block: qrot = (q H) / max|q H| per head, qmax = that max; then
// the table from which every lane builds its query operand for a group. Lane (g, tq)
// holds column g of the MMA (head g >> 1, part g & 1) for the channels of pair P of
// chunk tq; with v = q_hat * 2^-ex (the codes' power-of-two offset folded in) split
// into f16 parts v = vh + vl, the table holds per pair: vh, -vh on a low-part lane
// (0 on a high-part lane) and vl on a low-part lane (0 on a high-part lane).
template <int KB>
__device__ void setup_query(const DecodeParams& p, const Smem& sm, int ci, int kvh) {
    using CK = Codes<KB>;
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    if (w < 4) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (w < p.r) {
            const uint16_t* q = p.q + ((size_t)ci * p.hq + (size_t)kvh * p.r + w) * 128 + 4 * lane;
            uint2 raw = *reinterpret_cast<const uint2*>(q);
            float2 f0 = __half22float2(bits_h2(raw.x)), f1 = __half22float2(bits_h2(raw.y));
            v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
        }
        warp_fwht128(v, lane);
        float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (mx == 0.f) mx = 1.f;
        const float inv = 1.0f / mx;
#pragma unroll
        for (int k = 0; k < 4; ++k) sm.qrot[128 * w + 4 * lane + k] = v[k] * inv;
        if (lane == 0) sm.qmax[w] = mx;
    }
    named_bar(1, kConsumers);
    if (t < 256) {
        // thread (q, lane) writes pairs P = 2q, 2q + 1 of lane (g, tq)
        const int q = t >> 5, g = lane >> 2, tq = lane & 3;
        const bool lo_lane = (g & 1) != 0;
        const float* qh = sm.qrot + 128 * (g >> 1);
        uint32_t hi2[2], neg2[2], lo2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int P = 2 * q + e;
            const int x = P % CK::HALF;
            const int c0 = 32 * tq + CK::CPW * (P / CK::HALF) + x;
            const float sc = __int_as_float((127 - CK::ex(x)) << 23);  // 2^-ex
            const float v0 = qh[c0] * sc, v1 = qh[c0 + CK::HALF] * sc;
            const __half2 h = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(h);
            const __half2 l = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            hi2[e] = h2_bits(h);
            neg2[e] = lo_lane ? h2_bits(__hneg2(h)) : 0u;
            lo2[e] = lo_lane ? h2_bits(l) : 0u;
        }
        uint32_t* tab = reinterpret_cast<uint32_t*>(sm.qtab);
        const int word = 2 * (q & 1);  // pairs 4k .. 4k + 3 share one 16-byte entry
#pragma unroll
        for (int kind = 0; kind < 3; ++kind) {
            const uint32_t* src = kind == 0 ? hi2 : (kind == 1 ? neg2 : lo2);
            uint32_t* dst = tab + 4 * ((kind * 4 + (q >> 1)) * 32 + lane) + word;
            *reinterpret_cast<uint2*>(dst) = make_uint2(src[0], src[1]);
        }
    }
    named_bar(1, kConsumers);
}

struct WarpState {
    float m, l;
    float2 acc[8];  // channels 16 mt + g and 16 mt + g + 8 of head tq
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

// f16 pair (c[c0], c[c0 + HALF]) of the channel scales of pair P, from the scales of a
// 32-channel chunk held as 16 half2 words.
template <int B>
__device__ __forceinline__ __half2 pair_scales(const uint32_t* cw, int P) {
    using C = Codes<B>;
    const int c0 = C::CPW * (P / C::HALF) + P % C::HALF, c1 = c0 + C::HALF;
    const int b0 = 2 * (c0 & 1), b1 = 4 + 2 * (c1 & 1);
    return bits_h2(__byte_perm(cw[c0 >> 1], cw[c1 >> 1], b0 | (b0 + 1) << 4 | b1 << 8 | (b1 + 1) << 12));
}

// A operand whose every element is 2^e (rows identical): multiplies a B fragment into
// its per-column sum, undoing the power-of-two offsets folded into B.
__host__ __device__ constexpr uint32_t pow2_pair(int e) { return (uint32_t)((15 + e) << 10) * 0x10001u; }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Tiles processed together, k-step outer: TG independent MMA chains, TG * 2 * B
// code words live in registers.
template <int B>
struct TileGroup {
    static constexpr int TG = B == 8 ? 2 : 4;
};

// Process one sealed group pair held in shared memory (K record, then V record).
template <int KB, int VB>
__device__ __forceinline__ void process_group(const DecodeParams& p, const uint8_t* rec, const uint4* qtab,
                                              float qm, float* xb, WarpState& st, int g, int tq, int lane) {
    using CK = Codes<KB>;
    using CV = Codes<VB>;
    const uint8_t* krec = rec;
    const uint8_t* vrec = rec + p.rec_k;
    const float dK = *reinterpret_cast<const float*>(krec);
    const float mK = *reinterpret_cast<const float*>(krec + 4);
    const float dV = *reinterpret_cast<const float*>(vrec);
    const float mV = *reinterpret_cast<const float*>(vrec + 4);
    const uint16_t* aK = reinterpret_cast<const uint16_t*>(krec + 16);
    const uint16_t* aV = reinterpret_cast<const uint16_t*>(vrec + 16);
    const uint16_t* cV = reinterpret_cast<const uint16_t*>(vrec + 272);
    // ---- query operand of this group, (v c_K) split into f16 high / low parts:
    // high lane: RN(vh c); low lane: RN(vl c + (vh c - RN(vh c))), the residual being
    // exact in f16. |v| <= 1 and c_K <= 65504, so nothing overflows.
    uint32_t bk[16];
    {
        const uint4* cp = reinterpret_cast<const uint4*>(krec + 272 + 64 * tq);
        uint32_t cw[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 v = cp[k];
            cw[4 * k] = v.x; cw[4 * k + 1] = v.y; cw[4 * k + 2] = v.z; cw[4 * k + 3] = v.w;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 th = qtab[k * 32 + lane];
            const uint4 tn = qtab[(4 + k) * 32 + lane];
            const uint4 tl = qtab[(8 + k) * 32 + lane];
            const uint32_t vh[4] = {th.x, th.y, th.z, th.w};
            const uint32_t vn[4] = {tn.x, tn.y, tn.z, tn.w};
            const uint32_t vl[4] = {tl.x, tl.y, tl.z, tl.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 c2 = pair_scales<KB>(cw, 4 * k + e);
                const __half2 r = __hfma2(bits_h2(vh[e]), c2, __hmul2(bits_h2(vn[e]), c2));
                bk[4 * k + e] = h2_bits(__hfma2(bits_h2(vl[e]), c2, r));
            }
        }
    }
    // sum_j q_hat_j c_j of head tq: the high and low columns of the operand times 2^ex
    float sumqc;
    {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a0 = pow2_pair(CK::ex((2 * ks) % CK::HALF));
            const uint32_t a2 = pow2_pair(CK::ex((2 * ks + 1) % CK::HALF));
            mma16816(s4, a0, a0, a2, a2, bk[2 * ks], bk[2 * ks + 1]);
        }
        sumqc = s4[0] + s4[1];
    }
    // ---- raw scores of the 16 tokens this thread holds (head tq): high + low columns
    float2 S[8];
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
            for (int i = 0; i < TG; ++i) S[t0g + i] = make_float2(c[i][0] + c[i][1], c[i][2] + c[i][3]);
        }
    }
    // ---- scores: scale * a_t * (delta * raw + m * sum_j q_hat_j c_j), log2 domain
    const float alpha = p.scale_log2 * qm * dK * 16777216.0f;  // codes enter as code * 2^(ex-24)
    const float beta = p.scale_log2 * qm * mK * sumqc;
    const float2 alpha2 = make_float2(alpha, alpha), beta2 = make_float2(beta, beta);
    float gmax = kNegInf;
    float2 av[8];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int t0 = tok_row<VB>(mt, g), t1 = t0 + CV::HALF;
        const float2 ak = make_float2(half_bits_to_float(aK[t0]), half_bits_to_float(aK[t1]));
        S[mt] = __fmul2_rn(ak, __ffma2_rn(alpha2, S[mt], beta2));
        gmax = fmax3(gmax, S[mt].x, S[mt].y);
        av[mt] = make_float2(half_bits_to_float(aV[t0]), half_bits_to_float(aV[t1]));
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
    const float2 sv2 = make_float2(sv, sv), mneg = make_float2(-mnew, -mnew);
    float2 l2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const float2 d = __fadd2_rn(S[mt], mneg);
        const float2 pr = make_float2(fast_exp2(d.x), fast_exp2(d.y));
        l2 = __fadd2_rn(l2, pr);
        const __half2 wh = __float22half2_rn(__fmul2_rn(__fmul2_rn(pr, av[mt]), sv2));
        reinterpret_cast<uint32_t*>(xb)[kXbHead * tq + 20 * (mt >> 1) + 8 * (mt & 1) + g] = h2_bits(wh);
    }
    st.l = fmaf(st.l, corr, l2.x + l2.y);
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
    // sum_t w_t rho of head tq: the weight operand times 2^(ex - EV)
    float wsum;
    {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a0 = pow2_pair(CV::ex((2 * ks) % CV::HALF) - kEV);
            const uint32_t a2 = pow2_pair(CV::ex((2 * ks + 1) % CV::HALF) - kEV);
            mma16816(s4, a0, a0, a2, a2, bv[2 * ks], bv[2 * ks + 1]);
        }
        wsum = s4[0];
    }
    // ---- P V in the rotated frame
    const float gam = dV * (float)(1 << (24 - kEV)) / rho;
    const float del = mV * wsum / rho;
    const float2 corr2 = make_float2(corr, corr);
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
                const float2 cv = make_float2(half_bits_to_float(cV[c0]), half_bits_to_float(cV[c0 + 8]));
                const float2 x = make_float2(fmaf(gam, d[i][0], del), fmaf(gam, d[i][2], del));
                st.acc[mt] = __ffma2_rn(st.acc[mt], corr2, __fmul2_rn(cv, x));
            }
        }
    }
}

// Merge the eight warps' states of one item into a partial in global memory.
__device__ void write_item_partial(const DecodeParams& p, const Smem& sm, const WarpState& st, int blk, int slot) {
    const int t = threadIdx.x, w = t >> 5, lane = t & 31, g = lane >> 2, tq = lane & 3;
    float l = st.l;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    float* M = sm.mrg + w * kMrgFloats;
    if (g == 0) {
        M[tq] = st.m;
        M[4 + tq] = l;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        M[8 + 128 * tq + 16 * mt + g] = st.acc[mt].x;
        M[8 + 128 * tq + 16 * mt + g + 8] = st.acc[mt].y;
    }
    named_bar(1, kConsumers);
    if (t < 256) {
        const int h = t >> 6, jj = 2 * (t & 63);
        float mx = kNegInf;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) mx = fmaxf(mx, sm.mrg[k * kMrgFloats + h]);
        float ls = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) {
            const float* Mk = sm.mrg + k * kMrgFloats;
            const float mk = Mk[h];
            if (mk == kNegInf) continue;
            const float wgt = exp2f(mk - mx);
            ls = fmaf(wgt, Mk[4 + h], ls);
            a0 = fmaf(wgt, Mk[8 + 128 * h + jj], a0);
            a1 = fmaf(wgt, Mk[8 + 128 * h + jj + 1], a1);
        }
        float* P = partial_ptr(p, blk, slot);
        *reinterpret_cast<float2*>(P + 12 + 128 * h + jj) = make_float2(a0, a1);
        if ((t & 63) == 0) {
            P[4 + h] = mx;
            P[8 + h] = ls;
        }
        if (t == 0) P[0] = __int_as_float((int)p.epoch);
    }
}

struct SealRows {
    const uint16_t* tail;  // rows 0..126
    const uint16_t* last;  // row 127: the new token
    __device__ const uint16_t* operator()(int i) const { return i < 127 ? tail + 128 * i : last; }
};

// Source of a copy being resolved. For a sealed group the block-table entry is loaded
// one round ahead of the copy, so that its latency overlaps a group's processing.
struct PendingCopy {
    const uint8_t* base;  // seal record: its address; sealed group: pool + kv head offset
    int32_t slot;         // block-table entry of a sealed group (possibly still in flight)
    bool direct, valid;
};

// Walks the CTA's sealed groups in stream order to find the record of group number gn
// (0, 1, ... over the chunk and seal items of the CTA's unit range, in item order).
struct GroupCursor {
    int64_t u;       // unit cursor of the item walk
    Item it;         // current chunk / seal item
    uint32_t base;   // group number of the item's first group
    bool valid;
    __device__ void init(int64_t lo) { u = lo; base = 0; valid = false; it.g0 = it.g1 = 0; }
    // source of group gn (gn never decreases between calls); invalid past the end
    __device__ PendingCopy resolve(const DecodeParams& p, int64_t hi, uint32_t gn) {
        PendingCopy pc;
        pc.valid = false;
        pc.direct = false;
        pc.slot = 0;
        pc.base = nullptr;
        for (;;) {
            if (valid && gn < base + (uint32_t)(it.g1 - it.g0)) break;
            if (valid) base += (uint32_t)(it.g1 - it.g0);
            valid = false;
            Item n;
            bool found = false;
            while (next_item(p, u, hi, n)) {
                if (n.type != 1) { found = true; break; }
            }
            if (!found) return pc;
            it = n;
            valid = true;
        }
        const SeqEntry& e = p.seqs[it.ci];
        const size_t pair = (size_t)(p.rec_k + p.rec_v);
        pc.valid = true;
        if (it.type == 2) {
            pc.direct = true;
            pc.base = p.base + p.lay.pool + (size_t)e.seal_slot * p.slot_bytes + (size_t)it.kvh * pair;
        } else {
            const int32_t* table = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table);
            pc.base = p.base + p.lay.pool + (size_t)it.kvh * pair;
            pc.slot = table[((size_t)e.seq * p.num_layers + p.layer) * p.max_groups + it.g0 + (int)(gn - base)];
        }
        return pc;
    }
};

__device__ __forceinline__ void issue_copy(const DecodeParams& p, const Smem& sm, const PendingCopy& pc, uint32_t gn) {
    if (!pc.valid) return;
    const uint8_t* src = pc.base;
    if (!pc.direct) {
        int slot = pc.slot;
        if (slot < 0 || slot >= p.pool_slots) {
            atomicOr(err_word(p), kErrBadSlot);
            slot = 0;
        }
        src += (size_t)slot * p.slot_bytes;
    }
    const uint32_t pair = (uint32_t)(p.rec_k + p.rec_v);
    const uint32_t s = gn % p.stages;
    mbar_arrive_expect_tx(sm.full + s, pair);
    bulk_g2s(sm.stages + (size_t)s * pair, src, pair, sm.full + s);
}

// One CTA of 12 warps per SM. Stage ring: group gn lives in stage gn % S and is
// processed by warp gn % 12; the warp that finishes with a stage issues the copy of
// group gn + S into it, so no stage needs a release barrier. Seal items of the CTA run
// first, with their scratch aliased onto the (still empty) stage ring.
template <int KB, int VB>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem sm;
    const int pair = p.rec_k + p.rec_v;
    {
        size_t off = 0;
        sm.stages = smem_raw;
        size_t ring = (size_t)p.stages * pair;
        if (ring < sizeof(SealSmem)) ring = sizeof(SealSmem);
        off += ring;
        off = (off + 15) & ~(size_t)15;
        sm.full = reinterpret_cast<uint64_t*>(smem_raw + off);
        off += 32 * 8;
        sm.qrot = reinterpret_cast<float*>(smem_raw + off);
        off += 512 * 4;
        sm.qmax = reinterpret_cast<float*>(smem_raw + off);
        off += 16;
        sm.flag = reinterpret_cast<int*>(smem_raw + off);
        off += 16;
        sm.qtab = reinterpret_cast<uint4*>(smem_raw + off);
        off += 12 * 32 * 16;
        sm.xbuf = reinterpret_cast<float*>(smem_raw + off);
        off += kWarps * kXbWarp * 4;
        sm.mrg = reinterpret_cast<float*>(smem_raw + off);
        sm.seal = reinterpret_cast<SealSmem*>(smem_raw);
    }
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    if (t == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(sm.full + s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t U = p.units_total, P = p.grid, b = blockIdx.x;
    const int64_t lo = b * U / P, hi = (b + 1) * U / P;
    int32_t* err = err_word(p);

    // ---- 1. seal the groups completed by this step's tokens (before any prefetch)
    bool sealed_any = false;
    {
        int64_t u = lo;
        Item it;
        while (next_item(p, u, hi, it)) {
            if (it.type != 2) continue;
            const SeqEntry& e = p.seqs[it.ci];
            const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
            const size_t rows0 = (sl * p.hkv + it.kvh) * 128;
            uint8_t* dst = p.base + p.lay.pool + (size_t)e.seal_slot * p.slot_bytes + (size_t)it.kvh * pair;
            if (t < kSealThreads) {  // the seal runs on 8 warps (barrier 2); the others wait below
                SealRows rk{reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_k) + rows0 * 128,
                            p.k_new + ((size_t)it.ci * p.hkv + it.kvh) * 128};
                seal_matrix(rk, p.k_bits, 0, p.iters, dst, nullptr, *sm.seal, 2);
                SealRows rv{reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_v) + rows0 * 128,
                            p.v_new + ((size_t)it.ci * p.hkv + it.kvh) * 128};
                seal_matrix(rv, p.v_bits, 1, p.iters, dst + p.rec_k, nullptr, *sm.seal, 2);
            }
            if (t == 0 && it.kvh == 0) {
                int32_t* table = reinterpret_cast<int32_t*>(p.base + p.lay.block_table);
                table[sl * p.max_groups + e.seal_group] = e.seal_slot;
            }
            sealed_any = true;
        }
    }
    if (sealed_any) {
        fence_proxy_async_global();  // the records just written are read by bulk copies
        __syncthreads();
    }

    // ---- 2. prologue: the first S groups of the stream
    GroupCursor cur;
    cur.init(lo);
    PendingCopy pend;
    pend.valid = false;
    if (lane == 0) {
        for (uint32_t gn = w; gn < (uint32_t)p.stages; gn += kWarps) issue_copy(p, sm, cur.resolve(p, hi, gn), gn);
        pend = cur.resolve(p, hi, w + p.stages);  // this warp's first copy inside the loop
    }
    __syncwarp();

    // ---- 3. items in order
    const int g = lane >> 2, tq = lane & 3;
    int64_t u = lo;
    Item it;
    uint32_t n = 0;
    while (next_item(p, u, hi, it)) {
        const SeqEntry& e = p.seqs[it.ci];
        const int blk = e.seq * p.hkv + it.kvh;
        if (it.type == 1) {
            exact_item(p, sm, it.ci, it.kvh);
            continue;
        }
        int slot;
        if (it.type == 2) {
            slot = kSlotSeal;
        } else {
            int64_t first;
            expected_partials(p, e, it.kvh, &first);
            slot = kSlotChunk0 + (int)(b - first);
            if (slot >= kPartialSlots) {  // cannot happen with the host's schedule
                if (t == 0) atomicOr(err, kErrSpan);
                slot = kPartialSlots - 1;
            }
        }
        setup_query<KB>(p, sm, it.ci, it.kvh);
        const float qm = sm.qmax[tq];
        WarpState st;
        st.m = kNegInf;
        st.l = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) st.acc[mt] = make_float2(0.f, 0.f);
        float* xb = sm.xbuf + w * kXbWarp;
        const uint32_t cnt = (uint32_t)(it.g1 - it.g0);
        for (uint32_t k = (w + kWarps - (n % kWarps)) % kWarps; k < cnt; k += kWarps) {
            const uint32_t gn = n + k;
            const uint32_t s = gn % p.stages;
            mbar_wait(sm.full + s, (gn / p.stages) & 1, err);
            process_group<KB, VB>(p, sm.stages + (size_t)s * pair, sm.qtab, qm, xb, st, g, tq, lane);
            __syncwarp();
            if (lane == 0) {
                issue_copy(p, sm, pend, gn + p.stages);
                pend = cur.resolve(p, hi, gn + kWarps + p.stages);
            }
            __syncwarp();
        }
        n += cnt;
        write_item_partial(p, sm, st, blk, slot);
        publish(p, sm, it.ci, it.kvh);
    }
    // Normally every copy was waited for above. After a wait that gave up, let the
    // copies still in flight land (bounded) before the CTA's shared memory goes away.
    if (t == 0 && (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout)) {
        const uint64_t t0 = global_ns();
        for (uint32_t k = n > (uint32_t)p.stages ? n - p.stages : 0; k < n; ++k)
            while (!mbar_try_wait(sm.full + (k % p.stages), (k / p.stages) & 1) && global_ns() - t0 < kWaitLimitNs) {
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

int decode_smem_bytes(int k_bits, int v_bits, int stages, bool with_seal) {
    (void)with_seal;  // the seal scratch aliases the stage ring
    size_t pair = record_bytes(k_bits) + record_bytes(v_bits);
    size_t off = (size_t)stages * pair;
    if (off < sizeof(SealSmem)) off = sizeof(SealSmem);
    off = (off + 15) & ~(size_t)15;
    off += 32 * 8 + 512 * 4 + 16 + 16 + 12 * 32 * 16 + kWarps * kXbWarp * 4 + kWarps * kMrgFloats * 4;
    return (int)off;
}

// ---------------------------------------------------------------------------
// Static split-K workspace for kvarn_decode_attention_noalloc: partial softmax states
// and merge tickets of up to kStaticBlocks (sequence, KV head) blocks, 9.2 MB per GPU
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
