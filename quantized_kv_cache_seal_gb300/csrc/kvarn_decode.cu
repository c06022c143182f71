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
// Work split. Every (sequence, KV head) pair is a block of scheduling units: its exact
// part, the seal of a group this step completes, and one unit per sealed group. The
// units of all blocks are cut into contiguous ranges of near-equal size, one per CTA
// (a block's exact part and seal never split); the part of a
// block that a CTA covers is an item, whose stream entries are the block's exact
// sub-groups (16 fp16 tokens each, if the CTA owns the exact part), the record sealed in
// this step, then sealed groups. Each CTA writes one partial softmax state (running
// max, sum, rotated accumulator) per block it covers; merge_kernel, launched after the
// decode kernel, merges each block's partials, rotates back and writes fp16.
//
// Stream. Entries are copied with cp.async.bulk into a ring of shared-memory stages by
// one copy-issuing warp; entry n is processed by compute warp n mod 12, which releases
// its stage (an mbarrier arrive) for the copy of entry n + S. For a group with codes q, token scales a, channel scales c and
// grid (m, delta), the score of token t is
//   scale * a_t * (delta * sum_j (q'_j c_j) q_tj + m * sum_j q'_j c_j)
// with q' the rotated query, and the rotated output accumulates
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
constexpr int kWarps = 12;  // compute warps (warpgroups 0..2); warpgroup 3 issues the copies
static_assert(kDecodeThreads == 32 * (kWarps + 4), "three compute warpgroups and one copy-issuing warpgroup");
// Registers per thread after the split: the kernel is launched with 65536 / 512 = 128;
// the copy-issuing warpgroup gives back (128 - kRegsCopy) per thread, the compute
// warpgroups take (kRegsCompute - 128). Per CTA 12 * 32 * 24 = 9216 taken, 4 * 32 * 72 =
// 9216 given; per SM sub-partition (three compute warps, one copy warp) 2304 and 2304.
constexpr int kRegsCompute = 152, kRegsCopy = 56;
constexpr int kComputeThreads = 32 * kWarps;
static_assert(kWarps * 32 * (kRegsCompute - 128) <= 4 * 32 * (128 - kRegsCopy), "register split exceeds the launch");
static_assert(3 * 32 * (kRegsCompute - 128) <= 32 * (128 - kRegsCopy), "register split exceeds a sub-partition");
constexpr int kRowPitch = 272;                // shared-memory pitch of an exact fp16 row (conflict-free ldmatrix)
constexpr int kExactVOff = kExactRows * kRowPitch;  // V rows of an exact sub-group follow its K rows
constexpr int kTabWords = 12 * 32;            // uint4 entries of one query operand table
constexpr int kMaxDevices = 64;
#define kNegInf (-__int_as_float(0x7f800000))

// A thread's 32-code chunk is taken as NVW words of CPW codes, HALF in each 16-bit half
// at B-bit spacing from bit 0 of the half. For B = 2, 4, 8 these are the packed words
// themselves; for the odd widths (the stream has codes straddling words) load_chunk
// rebuilds them: 8 codes a word at 3 bits, 4 at 5 and 6 bits.
template <int B>
struct Codes {
    static constexpr int CPW = B == 3 ? 8 : (B == 5 || B == 6) ? 4 : 32 / B;  // codes per word
    static constexpr int NVW = 32 / CPW;  // words per 32-code chunk
    static constexpr int HALF = CPW / 2;  // partner code distance (low half -> high half)
    static constexpr int NWIN = 10 / B;   // codes of a 16-bit half that fit in the f16 mantissa
    __host__ __device__ static constexpr int sh(int x) { return (x / NWIN) * NWIN * B; }
    __host__ __device__ static constexpr int ex(int x) { return (x % NWIN) * B; }
    __host__ __device__ static constexpr uint32_t mask(int x) { return (((1u << B) - 1u) << ex(x)) * 0x10001u; }
};

// Bits pos .. pos + width - 1 (width <= 24) of a little-endian word stream.
template <int N>
__device__ __forceinline__ uint32_t stream_bits(const uint32_t (&s)[N], int pos, int width) {
    const int lo = pos / 32, sh = pos % 32;
    uint32_t v = s[lo] >> sh;
    if (sh + width > 32) v |= s[lo + 1] << (32 - sh);
    return v & ((1u << width) - 1u);
}

template <int B>
__device__ __forceinline__ void load_chunk(const uint8_t* p, uint32_t (&w)[Codes<B>::NVW]) {
    using C = Codes<B>;
    if constexpr (B == 3 || B == 5 || B == 6) {
        // 32 codes = B packed words (4-byte aligned); word v of the result holds codes
        // CPW v .. CPW v + CPW - 1: the first HALF in the low half, the others in the high
        uint32_t s[B];
#pragma unroll
        for (int k = 0; k < B; ++k) s[k] = reinterpret_cast<const uint32_t*>(p)[k];
        constexpr int HW = C::HALF * B;
#pragma unroll
        for (int v = 0; v < C::NVW; ++v) {
            const uint32_t f = stream_bits(s, v * C::CPW * B, C::CPW * B);
            w[v] = (f & ((1u << HW) - 1u)) | ((f >> HW) << 16);
        }
    } else if constexpr (B == 2) {
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
    constexpr int CPW = Codes<VB>::CPW, HALF = Codes<VB>::HALF;
    return CPW * (mt * (16 / CPW) + g / HALF) + g % HALF;
}

// CTA whose unit range holds unit u (the host's cut table: the last b with cta_begin[b] <= u).
__device__ __forceinline__ int64_t covering(const DecodeParams& p, int64_t u) {
    int lo = 0, hi = p.grid - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cta_begin[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The part of one (sequence, KV head) block that a CTA's unit range covers. Its stream
// entries, in order: n_ex exact sub-groups (the CTA that covers the block's first unit
// owns the exact part), the group sealed in this step (if the CTA covers the seal unit),
// then sealed groups g0 .. g1.
struct Item {
    int ci;    // index of the sequence in the call
    int kvh;
    int owner;  // covers the block's first unit (and so its exact part)
    int n_ex, seal;
    int g0, g1;
    __device__ int count() const { return n_ex + seal + g1 - g0; }
};

// Row (in units of 128 halves, from the tail region's start) of the first token of exact
// tail sub-group jt of block blk (sequence entry e): the tail is a ring of p.tail_cap rows
// per block whose tokens start at slot e.tail_first; a 16-row sub-group never wraps (the
// ring holds whole groups and the first slot is a multiple of 128).
__device__ __forceinline__ size_t tail_row(const DecodeParams& p, const SeqEntry& e, size_t blk, int jt) {
    return blk * (size_t)p.tail_cap + (size_t)((e.tail_first + jt * kExactRows) % p.tail_cap);
}

// Next item of this CTA's unit range [u, hi); advances u. Every block the range touches
// is an item, even one without stream entries: it still writes a (neutral) partial.
__device__ bool next_item(const DecodeParams& p, int64_t& u, int64_t hi, Item& it) {
    if (u >= hi) return false;
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
    const int end = (int)(min(hi, blk0 + per) - blk0);  // one past the last covered unit
    const int gu = e.w_exact + e.w_seal;                   // unit of group 0
    it.ci = lo;
    it.kvh = kvh;
    it.owner = off == 0;
    it.n_ex = off == 0 ? exact_subs(e.n_sink, e.n_tail) : 0;
    it.seal = (e.w_seal > 0 && off <= e.w_exact && e.w_exact < end) ? 1 : 0;
    it.g0 = max(off - gu, 0);
    it.g1 = max(end - gu, it.g0);
    u = blk0 + end;
    return true;
}

// The CTA's items, walked once at the start (the walk searches the sequence table in
// kernel-parameter memory); every later walk reads this list. A range with more items
// than fit walks the parameters again.
constexpr int kMaxItems = 8;
struct ItemList {
    int n;  // items; kMaxItems + 1 if the list overflowed
    int pad[3];
    Item it[kMaxItems];
};

// Sources of the CTA's first kMaxEntries stream entries, resolved once by the whole CTA:
// 8 bytes each, the low 48 bits an address (a record, or an exact sub-group's first K
// row), bits 48..57 the exact sub-group's rows (| 256 in the tail), bits 62..63 the kind.
constexpr int kMaxEntries = 256;

struct ItemWalk {
    int64_t u;  // unit cursor (overflowed list)
    int idx;    // next list entry
};

__device__ __forceinline__ bool walk_next(const DecodeParams& p, const ItemList& L, ItemWalk& wk, int64_t hi, Item& it) {
    if (L.n <= kMaxItems) {
        if (wk.idx >= L.n) return false;
        it = L.it[wk.idx++];
        return true;
    }
    return next_item(p, wk.u, hi, it);
}

struct WarpRegion {
    float2 acc[8][32];
    float m[4], l[4];
};

// Arrivals at the end of an item (two slots, by item parity).
struct ItemCtl {
    int tag;     // item number the slot currently takes
    int count;   // warps arrived
    int mask;    // warps that parked a state
    int pad;
};

struct Smem {
    uint8_t* stages;
    uint64_t* full;   // [32]: copy of the stage's group landed
    uint64_t* empty;  // [32]: the stage's group consumed (its stage may be refilled)
    uint32_t* gen;    // [32]: number of the group whose copy was last issued into each stage
    uint4* qtab;      // [2][kTabWords]: query operand tables (by block parity)
    float* qrot;      // [2][4][128]: rotated query of the table builder
    float* qmax;      // [2][4]
    uint32_t* qraw;   // [2][4][64]: the block's query as read (half2 words), for its exact part
    float* xbuf;      // [kWarps][kXbWarp] (half2 words)
    WarpRegion* region;  // [kWarps]
    ItemCtl* ictl;       // [2]
    int* busy;           // [kWarps]: item number parked in a warp's region, -1 if free
    int* ctl;            // [6]: table ready generation, claims and departures per table slot
    struct GroupCursor* cursor;  // [4]: each copy warp's cursor (all its lanes keep it in step)
    ItemList* items;
    unsigned long long* ent;  // [kMaxEntries]
    int* n_ent;               // entries in ent, or -1 if the stream does not fit
    SealSmem* seal;
};

__device__ __forceinline__ float* partial_ptr(const DecodeParams& p, int blk, int slot) {
    return p.partials + ((size_t)blk * kPartialSlots + slot) * kPartialFloats;
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

// CTAs whose unit ranges cover block (entry e, kvh) in this call (each writes one
// partial); the first of them in *first_cta.
__device__ int block_ctas(const DecodeParams& p, const SeqEntry& e, int kvh, int64_t* first_cta) {
    const int per = e.w_exact + e.w_seal + e.n_groups;
    const int64_t blk0 = e.unit_begin + (int64_t)kvh * per;
    const int64_t f = covering(p, blk0);
    if (first_cta) *first_cta = f;
    return (int)(covering(p, blk0 + per - 1) - f + 1);
}

// ldmatrix of four 8 x 8 b16 matrices (row addresses from lanes 8i .. 8i + 7 for matrix i).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}

// Bounded spin until *w == v (or >= v with at_least); records kErrTimeout on giving up.
__device__ __forceinline__ void spin_until(const int* w, int v, bool at_least, int32_t* err) {
    volatile const int* vw = w;
    auto ok = [&]() { return at_least ? (*vw >= v) : (*vw == v); };
    if (ok()) return;
    const uint64_t t0 = global_ns();
    while (!ok()) {
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            return;
        }
    }
}

// Query operand tables. For block (ci, kvh) the query is rotated per head:
// q_hat = (q H) / max|q H|, qmax = that max. Lane (g, tq) of a warp holds column g of
// the MMA (head g >> 1, part g & 1) for the channels of pair P of chunk tq; with
// v = q_hat * 2^-ex (the codes' power-of-two offset folded in) split into f16 parts
// v = vh + vl, the table holds per pair: vh, -vh on a low-part lane (0 on a high-part
// lane) and vl on a low-part lane (0 on a high-part lane).

// Lane's four query values of head h of block (ci, kvh) (zeros for a head the block's
// KV head does not have).
__device__ __forceinline__ uint2 load_query(const DecodeParams& p, int ci, int kvh, int h, int lane) {
    if (h >= p.r) return make_uint2(0u, 0u);
    return *reinterpret_cast<const uint2*>(p.q + ((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 + 4 * lane);
}

// Rotate head h (its values `raw` as load_query read them) into table slot b (one warp).
__device__ void rotate_loaded(const Smem& sm, int b, int h, int lane, uint2 raw) {
    float v[4];
    {
        const float2 f0 = __half22float2(bits_h2(raw.x)), f1 = __half22float2(bits_h2(raw.y));
        v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
    }
    *reinterpret_cast<uint2*>(sm.qraw + 256 * b + 64 * h + 2 * lane) = raw;
    warp_fwht128(v, lane);
    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (mx == 0.f) mx = 1.f;
    const float inv = 1.0f / mx;
    float* qrot = sm.qrot + 512 * b + 128 * h;
#pragma unroll
    for (int k = 0; k < 4; ++k) qrot[4 * lane + k] = v[k] * inv;
    if (lane == 0) sm.qmax[4 * b + h] = mx;
}

// Rotate head h of block (ci, kvh) into table slot b (one warp).
__device__ __forceinline__ void rotate_head(const DecodeParams& p, const Smem& sm, int b, int ci, int kvh, int h,
                                            int lane) {
    rotate_loaded(sm, b, h, lane, load_query(p, ci, kvh, h, lane));
}

// Table entries of pairs 2 q and 2 q + 1 of lane `lane` in slot b, from the rotated query.
template <int KB>
__device__ __forceinline__ void fill_table(const Smem& sm, int b, int q, int lane) {
    using CK = Codes<KB>;
    const int g = lane >> 2, tq = lane & 3;
    const bool lo_lane = (g & 1) != 0;
    const float* qh = sm.qrot + 512 * b + 128 * (g >> 1);
    uint32_t* tab = reinterpret_cast<uint32_t*>(sm.qtab + kTabWords * b);
    uint32_t hi2[2], neg2[2], lo2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int P = 2 * q + e;
        const int x = P % CK::HALF;
        const int c0 = 32 * tq + CK::CPW * (P / CK::HALF) + x;
        const float sc = __int_as_float((127 - CK::ex(x)) << 23);  // 2^-ex
        const float v0 = qh[c0] * sc, v1 = qh[c0 + CK::HALF] * sc;
        const __half2 hh = __floats2half2_rn(v0, v1);
        const float2 hf = __half22float2(hh);
        const __half2 l = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
        hi2[e] = h2_bits(hh);
        neg2[e] = lo_lane ? h2_bits(__hneg2(hh)) : 0u;
        lo2[e] = lo_lane ? h2_bits(l) : 0u;
    }
    const int word = 2 * (q & 1);  // pairs 4k .. 4k + 3 share one 16-byte entry
    *reinterpret_cast<uint2*>(tab + 4 * ((0 * 4 + (q >> 1)) * 32 + lane) + word) = make_uint2(hi2[0], hi2[1]);
    *reinterpret_cast<uint2*>(tab + 4 * ((1 * 4 + (q >> 1)) * 32 + lane) + word) = make_uint2(neg2[0], neg2[1]);
    *reinterpret_cast<uint2*>(tab + 4 * ((2 * 4 + (q >> 1)) * 32 + lane) + word) = make_uint2(lo2[0], lo2[1]);
}

// The whole table of block (ci, kvh) in slot b, by one warp.
template <int KB>
__device__ void build_table(const DecodeParams& p, const Smem& sm, int b, int ci, int kvh, int lane) {
#pragma unroll 1
    for (int h = 0; h < 4; ++h) rotate_head(p, sm, b, ci, kvh, h, lane);
    __syncwarp();
#pragma unroll 1
    for (int q = 0; q < 8; ++q) fill_table<KB>(sm, b, q, lane);
}

// Make the query table of the warp's kb-th table block available in slot kb & 1. The
// first `prebuilt` blocks were built by the whole CTA before the item loop. For a later
// block the first warp to reach it builds it once every warp has left block kb - 2 (the
// slot's previous user); the others wait for it.
template <int KB>
__device__ void acquire_table(const DecodeParams& p, const Smem& sm, int kb, int prebuilt, int ci, int kvh, int lane,
                              int32_t* err) {
    if (kb < prebuilt) return;
    const int b = kb & 1;
    int* ready = sm.ctl;
    int* claim = sm.ctl + 2;
    int* left = sm.ctl + 4;
    int old = 0;
    if (lane == 0) old = atomicAdd(claim + b, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == kWarps * ((kb >> 1) - 1)) {  // claims of slot b count from block 2 + b on
        if (lane == 0) spin_until(left + b, kWarps * (kb >> 1), true, err);
        __syncwarp();
        __threadfence_block();
        build_table<KB>(p, sm, b, ci, kvh, lane);
        __threadfence_block();
        __syncwarp();
        if (lane == 0) *reinterpret_cast<volatile int*>(ready + b) = kb + 1;
    } else {
        if (lane == 0) spin_until(ready + b, kb + 1, false, err);
        __syncwarp();
        __threadfence_block();
    }
}

// Exact query operand of a warp: column g holds head g >> 1 (both columns of a head
// carry it), k pairs are channels 16 ks + 2 tq (+ 8); read from the copy of the query
// kept with the block's table in slot b (zeros for heads the group does not have).
__device__ __forceinline__ void exact_query(const Smem& sm, int b, int g, int tq, uint32_t (&bq)[16]) {
    const uint32_t* qw = sm.qraw + 256 * b + 64 * (g >> 1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        bq[2 * ks] = qw[8 * ks + tq];
        bq[2 * ks + 1] = qw[8 * ks + 4 + tq];
    }
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
    static constexpr int TG = Codes<B>::NVW == 8 ? 2 : 4;
};

// One record's 128 x 128 code matrix times a B fragment (8 columns), k-step outer.
// Tile mt takes rows r = 16 mt + r0 and r + r1 of the matrix (the thread's row offset
// r0 and the row distance r1 are folded into `rows` and `off1`); out[mt] holds, for
// those two rows, the sum of the thread's columns 2 tq and 2 tq + 1. colsum is the
// same column sum of B itself with each pair weighted by 2^ex (the power-of-two
// offset of its codes), from eight MMAs with a constant A.
template <int B>
__device__ __forceinline__ void tiles_mma(const uint8_t* rows, int off1, const uint32_t (&bf)[16], float2 (&out)[8],
                                          float& colsum) {
    using C = Codes<B>;
    {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a0 = pow2_pair(C::ex((2 * ks) % C::HALF));
            const uint32_t a2 = pow2_pair(C::ex((2 * ks + 1) % C::HALF));
            mma16816(s4, a0, a0, a2, a2, bf[2 * ks], bf[2 * ks + 1]);
        }
        colsum = s4[0] + s4[1];
    }
    constexpr int TG = TileGroup<B>::TG;
#pragma unroll
    for (int t0g = 0; t0g < 8; t0g += TG) {
        uint32_t w0[TG][C::NVW], w1[TG][C::NVW];
#pragma unroll
        for (int i = 0; i < TG; ++i) {
            const uint8_t* r = rows + (t0g + i) * 16 * 16 * B;
            load_chunk<B>(r, w0[i]);
            load_chunk<B>(r + off1, w1[i]);
        }
        float c[TG][4];
#pragma unroll
        for (int i = 0; i < TG; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int i = 0; i < TG; ++i)
                mma16816(c[i], pair_operand<B>(w0[i], 2 * ks), pair_operand<B>(w1[i], 2 * ks),
                         pair_operand<B>(w0[i], 2 * ks + 1), pair_operand<B>(w1[i], 2 * ks + 1), bf[2 * ks],
                         bf[2 * ks + 1]);
        }
#pragma unroll
        for (int i = 0; i < TG; ++i) out[t0g + i] = make_float2(c[i][0] + c[i][1], c[i][2] + c[i][3]);
    }
}

// Query operand of a group: (v c_K) split into f16 high / low parts. High lane:
// RN(vh c); low lane: RN(vl c + (vh c - RN(vh c))), the residual being exact in f16.
// |v| <= 1 and c_K <= 65504, so nothing overflows.
template <int KB>
__device__ __forceinline__ void query_operand(const uint8_t* krec, const uint4* qtab, int tq, int lane,
                                              uint32_t (&bk)[16]) {
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

// Scores of the group from the raw QK sums, online-softmax update of the warp state,
// and the weight operand of P V: w = p * aV * rho * 2^(EV - ex) in f16, exchanged
// through the warp's buffer into the B fragment layout (bf). Returns the correction
// factor of the accumulator.
template <int VB>
__device__ __forceinline__ float softmax_weights(const DecodeParams& p, const uint8_t* krec, const uint8_t* vrec,
                                                 float qm, float sumqc, const float2 (&raw)[8], float* xb,
                                                 WarpState& st, int g, int tq, int lane, uint32_t (&bf)[16],
                                                 float& rho) {
    using CV = Codes<VB>;
    const float dK = *reinterpret_cast<const float*>(krec);
    const float mK = *reinterpret_cast<const float*>(krec + 4);
    const uint16_t* aK = reinterpret_cast<const uint16_t*>(krec + 16);
    const uint16_t* aV = reinterpret_cast<const uint16_t*>(vrec + 16);
    // scores: scale * a_t * (delta * raw + m * sum_j q_hat_j c_j), log2 domain
    const float alpha = p.scale_log2 * qm * dK * 16777216.0f;  // codes enter as code * 2^(ex-24)
    const float beta = p.scale_log2 * qm * mK * sumqc;
    const float2 alpha2 = make_float2(alpha, alpha), beta2 = make_float2(beta, beta);
    float gmax = kNegInf;
    float2 S[8];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int t0 = tok_row<VB>(mt, g), t1 = t0 + CV::HALF;
        const float2 ak = make_float2(half_bits_to_float(aK[t0]), half_bits_to_float(aK[t1]));
        S[mt] = __fmul2_rn(ak, __ffma2_rn(alpha2, raw[mt], beta2));
        gmax = fmax3(gmax, S[mt].x, S[mt].y);
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
    rho = __int_as_float((127 + 15 - ebits) << 23);
    const int xv = g % CV::HALF;
    const float sv = __int_as_float((127 + kEV - CV::ex(xv)) << 23) * rho;  // 2^(EV - ex) * rho
    const float2 sv2 = make_float2(sv, sv), mneg = make_float2(-mnew, -mnew);
    float2 l2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int t0 = tok_row<VB>(mt, g), t1 = t0 + CV::HALF;
        const float2 av = make_float2(half_bits_to_float(aV[t0]), half_bits_to_float(aV[t1]));
        const float2 d = __fadd2_rn(S[mt], mneg);
        const float2 pr = make_float2(fast_exp2(d.x), fast_exp2(d.y));
        l2 = __fadd2_rn(l2, pr);
        const __half2 wh = __float22half2_rn(__fmul2_rn(__fmul2_rn(pr, av), sv2));
        reinterpret_cast<uint32_t*>(xb)[kXbHead * tq + 20 * (mt >> 1) + 8 * (mt & 1) + g] = h2_bits(wh);
    }
    st.l = fmaf(st.l, corr, l2.x + l2.y);
    __syncwarp();
    {
        const uint4* src = reinterpret_cast<const uint4*>(xb + kXbHead * (g >> 1) + 20 * tq);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 v = src[k];
            bf[4 * k] = v.x; bf[4 * k + 1] = v.y; bf[4 * k + 2] = v.z; bf[4 * k + 3] = v.w;
        }
    }
    __syncwarp();
    return corr;
}

// Rotated-frame P V update of the warp state from the raw P V sums. Both B columns of
// a thread carry the same head's weights, so raw and colsum are twice the sums.
__device__ __forceinline__ void pv_update(const uint8_t* vrec, const float2 (&raw)[8], float colsum, float corr,
                                          float rho, WarpState& st, int g) {
    const float dV = *reinterpret_cast<const float*>(vrec);
    const float mV = *reinterpret_cast<const float*>(vrec + 4);
    const uint16_t* cV = reinterpret_cast<const uint16_t*>(vrec + 272);
    const float wsum = colsum * __int_as_float((127 - kEV - 1) << 23);  // sum_t w_t rho
    const float gam = dV * (float)(1 << (24 - kEV - 1)) / rho;
    const float del = mV * wsum / rho;
    const float2 gam2 = make_float2(gam, gam), del2 = make_float2(del, del), corr2 = make_float2(corr, corr);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int c0 = 16 * mt + g;
        const float2 cv = make_float2(half_bits_to_float(cV[c0]), half_bits_to_float(cV[c0 + 8]));
        st.acc[mt] = __ffma2_rn(st.acc[mt], corr2, __fmul2_rn(cv, __ffma2_rn(gam2, raw[mt], del2)));
    }
}

// Process one sealed group pair held in shared memory (K record, then V record).
template <int KB, int VB>
__device__ __forceinline__ void process_group(const DecodeParams& p, const uint8_t* rec, const uint4* qtab,
                                              float qm, float* xb, WarpState& st, int g, int tq, int lane) {
    using CV = Codes<VB>;
    const uint8_t* krec = rec;
    const uint8_t* vrec = rec + p.rec_k;
    const uint8_t* rows_k = krec + 528 + tok_row<VB>(0, g) * 16 * KB + 4 * KB * tq;
    const int off_k = CV::HALF * 16 * KB;
    const uint8_t* rows_v = vrec + 528 + g * 16 * VB + 4 * VB * tq;
    const int off_v = 8 * 16 * VB;
    uint32_t bf[16];
    query_operand<KB>(krec, qtab, tq, lane, bf);
    float2 raw[8];
    float colsum, corr, rho;
    if constexpr (KB == VB) {
        // One copy of the contraction code serves both records (a loop that is not
        // unrolled): the group loop then fits the instruction cache far better.
        const uint8_t* rows = rows_k;
        int off = off_k;
#pragma unroll 1
        for (int side = 0; side < 2; ++side) {
            tiles_mma<KB>(rows, off, bf, raw, colsum);
            if (side == 0) {
                corr = softmax_weights<VB>(p, krec, vrec, qm, colsum, raw, xb, st, g, tq, lane, bf, rho);
                rows = rows_v;
                off = off_v;
            }
        }
    } else {
        tiles_mma<KB>(rows_k, off_k, bf, raw, colsum);
        corr = softmax_weights<VB>(p, krec, vrec, qm, colsum, raw, xb, st, g, tq, lane, bf, rho);
        tiles_mma<VB>(rows_v, off_v, bf, raw, colsum);
    }
    pv_update(vrec, raw, colsum, corr, rho, st, g);
}

// 128-point Hadamard transform scaled by 1/sqrt(128) (the records' rotation) of a vector
// held in the P V output layout: lane (g, tq) holds x[mt] = (channel 16 mt + g, channel
// 16 mt + g + 8); channel bits 0..2 are lane bits 2..4, bit 3 the float2 half, bits 4..6
// the tile.
__device__ __forceinline__ void frag_fwht128(float2 (&x)[8], int lane) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) x[mt] = make_float2(x[mt].x + x[mt].y, x[mt].x - x[mt].y);
#pragma unroll
    for (int len = 1; len < 8; len <<= 1) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            if (mt & len) continue;
            const float2 a = x[mt], b = x[mt + len];
            x[mt] = make_float2(a.x + b.x, a.y + b.y);
            x[mt + len] = make_float2(a.x - b.x, a.y - b.y);
        }
    }
#pragma unroll 1
    for (int bt = 4; bt < 32; bt <<= 1) {
        const float sg = (lane & bt) ? -1.f : 1.f;  // the lane holding the higher channel takes lo - hi
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const float ox = __shfl_xor_sync(0xffffffffu, x[mt].x, bt), oy = __shfl_xor_sync(0xffffffffu, x[mt].y, bt);
            x[mt] = make_float2(fmaf(sg, x[mt].x, ox), fmaf(sg, x[mt].y, oy));
        }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) x[mt] = make_float2(x[mt].x * kInvSqrt128, x[mt].y * kInvSqrt128);
}

// One exact sub-group (16 fp16 tokens of the sink or the tail, rows at pitch kRowPitch,
// K rows then V rows; rows >= n_rows hold stale bytes) on the tensor cores: scores from
// the unrotated query, P V with the weights split into f16 high and low columns (both
// columns of a head), accumulated unrotated (the caller rotates the sum).
__device__ __forceinline__ void process_exact(const uint8_t* stage, int n_rows, const uint32_t (&bq)[16],
                                              float scale_log2, float* xb, WarpState& st, int g, int tq,
                                              int lane) {
    const uint32_t sK = smem_addr(stage), sV = sK + kExactVOff;
    const int i4 = lane >> 3, r8 = lane & 7;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    {
        // matrix i4: tokens r8 + 8 (i4 & 1), channels 16 ks + 8 (i4 >> 1)
        const uint32_t a = sK + (r8 + 8 * (i4 & 1)) * kRowPitch + 16 * (i4 >> 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(a + 32 * ks, a0, a1, a2, a3);
            mma16816(d, a0, a1, a2, a3, bq[2 * ks], bq[2 * ks + 1]);
        }
    }
    const float s0 = g < n_rows ? d[0] * scale_log2 : kNegInf;
    const float s1 = g + 8 < n_rows ? d[2] * scale_log2 : kNegInf;
    float gmax = fmaxf(s0, s1);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    const float mnew = fmaxf(st.m, gmax);  // finite: every sub-group has a valid token
    const float corr = fast_exp2(st.m - mnew);
    st.m = mnew;
    const float p0 = fast_exp2(s0 - mnew), p1 = fast_exp2(s1 - mnew);
    st.l = fmaf(st.l, corr, p0 + p1);
    {
        const __half h0 = __float2half_rn(p0), h1 = __float2half_rn(p1);
        const __half l0 = __float2half_rn(p0 - __half2float(h0)), l1 = __float2half_rn(p1 - __half2float(h1));
        __half* xe = reinterpret_cast<__half*>(xb);  // [head][part][16 tokens]
        xe[(2 * tq) * 16 + g] = h0;
        xe[(2 * tq + 1) * 16 + g] = l0;
        xe[(2 * tq) * 16 + g + 8] = h1;
        xe[(2 * tq + 1) * 16 + g + 8] = l1;
    }
    __syncwarp();
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(xb);
    const uint32_t b0 = xw[8 * g + tq], b1 = xw[8 * g + 4 + tq];  // column g: head g >> 1, part g & 1
    __syncwarp();
    uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;  // stale rows enter as zeros
    if (n_rows < kExactRows) {
        m01 = (2 * tq < n_rows ? 0x0000ffffu : 0u) | (2 * tq + 1 < n_rows ? 0xffff0000u : 0u);
        m23 = (2 * tq + 8 < n_rows ? 0x0000ffffu : 0u) | (2 * tq + 9 < n_rows ? 0xffff0000u : 0u);
    }
    const float2 corr2 = make_float2(corr, corr);
    // matrix i4 of tile mt: tokens r8 + 8 (i4 >> 1), channels 16 mt + 8 (i4 & 1), transposed
    const uint32_t av = sV + (r8 + 8 * (i4 >> 1)) * kRowPitch + 16 * (i4 & 1);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(av + 32 * mt, a0, a1, a2, a3);
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(e, a0 & m01, a1 & m01, a2 & m23, a3 & m23, b0, b1);
        st.acc[mt] = __ffma2_rn(st.acc[mt], corr2, make_float2(e[0] + e[1], e[2] + e[3]));
    }
}

// Merge the parked states of an item in warp order (deterministic whatever the order of
// arrival) and write the CTA's partial (one warp). The block's partials are merged by
// merge_kernel after this kernel.
__device__ __noinline__ void finalize_item(const DecodeParams& p, const Smem& sm, uint32_t mask, int ci, int kvh, int pslot,
                              int g, int tq, int lane) {
    float M = kNegInf;
    for (uint32_t mm = mask; mm; mm &= mm - 1) M = fmaxf(M, sm.region[__ffs(mm) - 1].m[tq]);
    float L = 0.f;
    float2 acc[8];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt] = make_float2(0.f, 0.f);
    for (uint32_t mm = mask; mm; mm &= mm - 1) {
        const WarpRegion& R = sm.region[__ffs(mm) - 1];
        const float mw = R.m[tq];
        const float wgt = mw == kNegInf ? 0.f : exp2f(mw - M);
        L = fmaf(wgt, R.l[tq], L);
        const float2 w2 = make_float2(wgt, wgt);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) acc[mt] = __ffma2_rn(w2, R.acc[mt][lane], acc[mt]);
    }
    const SeqEntry& e = p.seqs[ci];
    const int blk = e.seq * p.hkv + kvh;
    float* P = partial_ptr(p, blk, pslot);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        P[12 + 128 * tq + 16 * mt + g] = acc[mt].x;
        P[12 + 128 * tq + 16 * mt + g + 8] = acc[mt].y;
    }
    if (g == 0) {
        P[4 + tq] = M;
        P[8 + tq] = L;
    }
    if (lane == 0) P[0] = __int_as_float((int)p.epoch);
}

// End of item number i for a warp: park its state (if it processed any group of the item)
// in its region, then arrive; the warp that arrives last merges the parked states, writes
// the partial and frees the regions and the arrival slot.
__device__ void fold_item(const DecodeParams& p, const Smem& sm, const WarpState& st, uint32_t i, int ci, int kvh,
                          int pslot, int w, int g, int tq, int lane, int32_t* err) {
    ItemCtl& C = sm.ictl[i & 1];
    const bool has = __any_sync(0xffffffffu, st.m != kNegInf);
    if (has) {
        float l = st.l;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) spin_until(sm.busy + w, -1, false, err);  // freed by the previous item's merge
        __syncwarp();
        __threadfence_block();
        WarpRegion& R = sm.region[w];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) R.acc[mt][lane] = st.acc[mt];
        if (g == 0) {
            R.m[tq] = st.m;
            R.l[tq] = l;
        }
        if (lane == 0) sm.busy[w] = (int)i;
    }
    __threadfence_block();
    __syncwarp();
    int c = 0;
    if (lane == 0) {
        spin_until(&C.tag, (int)i, false, err);
        if (has) atomicOr(&C.mask, 1 << w);
        __threadfence_block();
        c = atomicAdd(&C.count, 1) + 1;
    }
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c == kWarps) {
        __threadfence_block();
        const uint32_t mask = (uint32_t)*reinterpret_cast<volatile int*>(&C.mask);
        finalize_item(p, sm, mask, ci, kvh, pslot, g, tq, lane);
        __syncwarp();
        if (lane < kWarps && (mask >> lane & 1)) *reinterpret_cast<volatile int*>(sm.busy + lane) = -1;
        if (lane == 0) {
            *reinterpret_cast<volatile int*>(&C.count) = 0;
            *reinterpret_cast<volatile int*>(&C.mask) = 0;
            __threadfence_block();
            *reinterpret_cast<volatile int*>(&C.tag) = (int)i + 2;
        }
    }
}

// Rows of the group sealed in a decode step: from the tail ring (contiguous there: the
// group starts at a multiple of 128 rows), the last one from the step's input when the
// step's token completes the group (no tail floor).
struct SealRows {
    const uint16_t* tail;  // row 0 of the group in the tail ring
    const uint16_t* last;  // the new token
    int from_tail;         // rows read from the ring: 127 (then row 127 is the new token) or 128
    __device__ const uint16_t* operator()(int i) const { return i < from_tail ? tail + 128 * i : last; }
};

// Source of a copy being resolved. For a sealed group the block-table entry is loaded
// one round ahead of the copy, so that its latency overlaps a group's processing.
struct PendingCopy {
    const uint8_t* base;  // seal record: its address; sealed group: pool + kv head offset;
                          // exact sub-group: its first K row
    int32_t aux;          // sealed group: its block-table entry (possibly still in flight);
                          // exact sub-group: valid rows | 256 if in the tail
    int32_t kind;         // 0 none, 1 exact sub-group, 2 seal record, 3 sealed group
};

// Walks the CTA's stream in order to find the source of entry number gn (0, 1, ... over
// the entries of the CTA's items, in item order). Per item it keeps what a sealed group
// needs, so that such an entry costs a compare, a subtraction and one load.
struct __align__(16) GroupCursor {
    ItemWalk wk;           // item walk
    uint32_t first, end;   // entry numbers of the current item's first entry and one past its last
    int32_t ci, kvh, n_ex, seal;
    bool valid;
    const uint8_t* base;   // pool + kv head offset
    const int32_t* row;    // block-table entry of the item's first group
    __device__ void init(int64_t lo) {
        wk.u = lo;
        wk.idx = 0;
        first = end = 0;
        ci = kvh = n_ex = seal = 0;
        valid = false;
        base = nullptr;
        row = nullptr;
    }
    // source of entry gn (gn never decreases between calls); kind 0 past the end
    __device__ __noinline__ PendingCopy resolve(const DecodeParams& p, const ItemList& L, int64_t hi, uint32_t gn) {
        PendingCopy pc;
        pc.kind = 0;
        pc.aux = 0;
        pc.base = nullptr;
        while (!valid || gn >= end) {
            first = valid ? end : first;
            valid = false;
            Item n;
            if (!walk_next(p, L, wk, hi, n)) return pc;
            const SeqEntry& e = p.seqs[n.ci];
            ci = n.ci;
            kvh = n.kvh;
            n_ex = n.n_ex;
            seal = n.seal;
            base = p.base + p.lay.pool + (size_t)n.kvh * (size_t)(p.rec_k + p.rec_v);
            row = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table) +
                  ((size_t)e.seq * p.num_layers + p.layer) * p.max_groups + n.g0;
            end = first + (uint32_t)n.count();
            valid = true;
        }
        const int j = (int)(gn - first);
        if (j >= n_ex + seal) {
            pc.kind = 3;
            pc.base = base;
            // issued here, first used when the copy is issued a group later: a volatile
            // load keeps the compiler from sinking it to that use
            asm volatile("ld.global.s32 %0, [%1];" : "=r"(pc.aux) : "l"(row + (j - n_ex - seal)));
        } else if (j >= n_ex) {
            const SeqEntry& e = p.seqs[ci];
            pc.kind = 2;
            pc.base = p.base + p.lay.pool + (size_t)e.seal_slot * p.slot_bytes + (size_t)kvh * (p.rec_k + p.rec_v);
        } else {
            // exact sub-group j: sink rows 16 j .. or tail rows 16 (j - sink sub-groups) ..
            const SeqEntry& e = p.seqs[ci];
            const size_t blk = ((size_t)e.seq * p.num_layers + p.layer) * p.hkv + kvh;
            const int js = (e.n_sink + kExactRows - 1) / kExactRows;
            pc.kind = 1;
            if (j < js) {
                pc.base = p.base + p.lay.sink_k + (blk * 128 + (size_t)j * kExactRows) * 256;
                pc.aux = min(kExactRows, e.n_sink - j * kExactRows);
            } else {
                pc.base = p.base + p.lay.tail_k + tail_row(p, e, blk, j - js) * 256;
                pc.aux = min(kExactRows, e.n_tail - (j - js) * kExactRows) | 256;
            }
        }
        return pc;
    }
};

// Copies of an exact sub-group's rows (whole warp) into rows padded to kRowPitch (so
// that the ldmatrix reads of process_exact are free of bank conflicts): 16-byte cp.async
// copies, two 256-byte rows per warp instruction (K rows, then V rows), tracked by the
// stage's full barrier (each lane's copies hold the barrier's phase open until they
// land; lane 0 makes the phase's one expected arrival). Many small bulk copies cost the
// copy warps far more issue time. Kept out of line: the group loop stays short.
__device__ __noinline__ void issue_exact_rows(const DecodeParams& p, uint64_t* bar, uint8_t* dst, const uint8_t* base,
                                              int aux, int lane) {
    const int rows = aux & 255;
    const size_t kv = (aux & 256) ? p.lay.tail_v - p.lay.tail_k : p.lay.sink_v - p.lay.sink_k;
    for (int i = lane; i < 2 * 16 * kExactRows; i += 32) {  // (side, row, 16-byte chunk)
        const int side = i / (16 * kExactRows), r = (i / 16) % kExactRows, c = i % 16;
        if (r < rows)
            cp_async_16(dst + (side ? kExactVOff : 0) + r * kRowPitch + 16 * c,
                        base + (side ? kv : 0) + (size_t)r * 256 + 16 * c);
    }
    cp_async_mbar_arrive(bar);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// Issue the copy of a group into stage s (whole warp). A record is one bulk copy by lane
// 0; an exact sub-group is copied by the whole warp (issue_exact_rows).
__device__ __forceinline__ void issue_copy(const DecodeParams& p, const Smem& sm, const PendingCopy& pc, uint32_t gn,
                                           uint32_t s, int lane) {
    if (pc.kind == 0) return;
    uint8_t* dst = sm.stages + (size_t)s * (uint32_t)(p.rec_k + p.rec_v);
    if (pc.kind == 1) {
        issue_exact_rows(p, sm.full + s, dst, pc.base, pc.aux, lane);
    } else if (lane == 0) {
        const uint8_t* src = pc.base;
        if (pc.kind == 3) {
            int slot = pc.aux;
            if (slot < 0 || slot >= p.pool_slots) {
                atomicOr(err_word(p), kErrBadSlot);
                slot = 0;
            }
            src += (size_t)slot * p.slot_bytes;
        }
        const uint32_t pair = (uint32_t)(p.rec_k + p.rec_v);
        mbar_arrive_expect_tx(sm.full + s, pair);
        bulk_g2s(dst, src, pair, sm.full + s);
    }
    if (lane == 0) *reinterpret_cast<volatile uint32_t*>(sm.gen + s) = gn;
}

// Source of stream entry gn from the CTA's entry table (kind 0 past the end).
__device__ __forceinline__ PendingCopy table_copy(const Smem& sm, int n_ent, uint32_t gn) {
    PendingCopy pc;
    pc.kind = 0;
    pc.aux = 0;
    pc.base = nullptr;
    if (gn < (uint32_t)n_ent) {
        const unsigned long long v = sm.ent[gn];
        pc.kind = (int)(v >> 62);
        pc.aux = (int)((v >> 48) & 0x3ff);
        pc.base = reinterpret_cast<const uint8_t*>(v & 0xffffffffffffull);
    }
    return pc;
}

// Wait until group gn has landed in its stage. A copy into a stage is issued only after
// the stage's previous group was consumed, so once the stage's group number reads gn the
// barrier's current phase is the one of gn and waiting on its parity is unambiguous; a
// parity wait alone could match the phase of the group two rounds earlier when a warp
// runs a full ring ahead of the copies.
__device__ __forceinline__ void wait_group(const Smem& sm, uint32_t gn, uint32_t s, uint32_t parity, int32_t* err) {
    volatile uint32_t* gp = sm.gen + s;
    if (*gp != gn) {
        const uint64_t t0 = global_ns();
        while (*gp != gn) {
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(err, kErrTimeout);
                return;
            }
        }
    }
    mbar_wait(sm.full + s, parity, err);
}

// One CTA of four warpgroups per SM: three compute warpgroups (12 warps, 152 registers
// per thread) and one copy-issuing warpgroup (56 registers; one warp issues). Stage
// ring: group gn lives in stage gn % S and is processed by compute warp gn % 12, which
// releases the stage; the copy warp then issues group gn + S into it. After the start
// the compute warps never wait for each other as a whole: an item's states are folded
// warp by warp and the last warp writes its partial.
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
        sm.empty = reinterpret_cast<uint64_t*>(smem_raw + off);
        off += 32 * 8;
        sm.gen = reinterpret_cast<uint32_t*>(smem_raw + off);
        off += 32 * 4;
        sm.qtab = reinterpret_cast<uint4*>(smem_raw + off);
        off += 2 * kTabWords * 16;
        sm.qrot = reinterpret_cast<float*>(smem_raw + off);
        off += 2 * 512 * 4;
        sm.qmax = reinterpret_cast<float*>(smem_raw + off);
        off += 2 * 4 * 4;
        sm.qraw = reinterpret_cast<uint32_t*>(smem_raw + off);
        off += 2 * 4 * 64 * 4;
        sm.region = reinterpret_cast<WarpRegion*>(smem_raw + off);
        off += kWarps * sizeof(WarpRegion);
        sm.ictl = reinterpret_cast<ItemCtl*>(smem_raw + off);
        off += 2 * sizeof(ItemCtl);
        sm.busy = reinterpret_cast<int*>(smem_raw + off);
        off += 16 * 4;
        sm.ctl = reinterpret_cast<int*>(smem_raw + off);
        off += 8 * 4;
        sm.cursor = reinterpret_cast<GroupCursor*>(smem_raw + off);
        off += 4 * sizeof(GroupCursor);
        sm.items = reinterpret_cast<ItemList*>(smem_raw + off);
        off += sizeof(ItemList);
        sm.n_ent = reinterpret_cast<int*>(smem_raw + off);
        off += 16;
        sm.ent = reinterpret_cast<unsigned long long*>(smem_raw + off);
        off += kMaxEntries * 8;

        sm.xbuf = reinterpret_cast<float*>(smem_raw + off);
        sm.seal = reinterpret_cast<SealSmem*>(smem_raw);
    }
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    if (t < 32) sm.gen[t] = 0xffffffffu;
    if (t < 8) sm.ctl[t] = 0;
    if (t < 16) sm.busy[t] = -1;
    if (t < 2) {
        sm.ictl[t].tag = t;
        sm.ictl[t].count = 0;
        sm.ictl[t].mask = 0;
    }
    const int64_t b = blockIdx.x;
    const int64_t lo = p.cta_begin[b], hi = p.cta_begin[b + 1];
    if (t == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(sm.full + s, 1);
            mbar_init(sm.empty + s, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        int64_t u = lo;
        int n = 0;
        Item it;
        while (n <= kMaxItems && next_item(p, u, hi, it)) {
            if (n < kMaxItems) sm.items->it[n] = it;
            ++n;
        }
        sm.items->n = n;
    }
    __syncthreads();
    // the merge kernel that follows may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int32_t* err = err_word(p);
    const ItemList& IL = *sm.items;
    uint32_t n = 0;  // stream entries of the CTA (counted by the compute warps)
    if (w >= kWarps) {
        // ---- 2. the copy-issuing warpgroup. It hands registers to the compute warpgroups;
        //      its warps issue every copy of the stream, entry n into stage n % S once the
        //      consumer of entry n - S has released that stage, from
        //      the moment the compute warps have written this step's tokens and seals and
        //      resolved the stream's sources (named barrier 3).
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCopy));
        asm volatile("griddepcontrol.wait;" ::: "memory");
        named_bar(3, kDecodeThreads);
        // copy warp k issues the entries of the stages s with s % 4 == k, in entry order
        // (a stage's entries all come from one warp, so each waits on the stage's release
        // of the entry before it and its phase parity is unambiguous)
        const uint32_t k = (uint32_t)(w - kWarps);
        const int n_ent = *sm.n_ent;
        GroupCursor& cur = sm.cursor[k];
        cur.init(lo);
        __syncwarp();
        uint32_t s = 0, round = 0;
        for (uint32_t gn = 0; k < (uint32_t)p.stages; ++gn) {  // (a ring of fewer than 4 stages idles some)
            if ((s & 3u) == k) {
                const PendingCopy pc = n_ent >= 0 ? table_copy(sm, n_ent, gn) : cur.resolve(p, IL, hi, gn);
                if (pc.kind == 0) break;
                if (round > 0) {
                    int ok = 1;
                    if (lane == 0) ok = mbar_wait(sm.empty + s, (round - 1) & 1u, err);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    __syncwarp();
                    if (!ok) break;  // a consumer stopped: the error word has the timeout
                }
                issue_copy(p, sm, pc, gn, s, lane);
            } else if (n_ent >= 0 && gn >= (uint32_t)n_ent) {
                break;
            }
            if (++s == (uint32_t)p.stages) {
                s = 0;
                ++round;
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
        // this grid is itself a programmatic dependent of the work before it in the stream
        // (the previous step's merge, or the kernel that wrote q, k or v): nothing above read
        // global memory, everything below may read that work's output
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (p.test_stall && b == 0) {  // a bounded wait on a word nothing sets (timeout path test)
            if (t == 0) spin_until(sm.ctl + 6, 1, false, err);
            named_bar(1, kComputeThreads);
        }
        // the CTA's first two blocks: their query tables are built by the whole CTA; the query
        // rows are loaded first, so that their latency overlaps the block-table loads below
        int prebuilt = 0;
        int bci[2] = {-1, -1}, bkv[2] = {-1, -1};
        {
            ItemWalk wk{lo, 0};
            Item it;
            while (prebuilt < 2 && walk_next(p, IL, wk, hi, it)) {
                bci[prebuilt] = it.ci;
                bkv[prebuilt] = it.kvh;
                ++prebuilt;
            }
        }
        const bool rotator = w < 4 * prebuilt;
        uint2 qrow = make_uint2(0u, 0u);
        if (rotator) qrow = load_query(p, bci[w >> 2], bkv[w >> 2], w & 3, lane);
        // ---- sources of the stream's entries, resolved once (block-table loads in parallel)
        {
            int total = 0;
            if (IL.n <= kMaxItems)
                for (int k = 0; k < IL.n; ++k) total += IL.it[k].count();
            const bool fits = IL.n <= kMaxItems && total <= kMaxEntries;
            if (fits) {
                for (int e = t; e < total; e += kComputeThreads) {
                    int k = 0, j = e;
                    while (j >= IL.it[k].count()) j -= IL.it[k++].count();
                    const Item& itm = IL.it[k];
                    const SeqEntry& se = p.seqs[itm.ci];
                    unsigned long long v;
                    if (j < itm.n_ex) {
                        const size_t blk = ((size_t)se.seq * p.num_layers + p.layer) * p.hkv + itm.kvh;
                        const int js = (se.n_sink + kExactRows - 1) / kExactRows;
                        uintptr_t a;
                        int aux;
                        if (j < js) {
                            a = (uintptr_t)(p.base + p.lay.sink_k + (blk * 128 + (size_t)j * kExactRows) * 256);
                            aux = min(kExactRows, se.n_sink - j * kExactRows);
                        } else {
                            a = (uintptr_t)(p.base + p.lay.tail_k + tail_row(p, se, blk, j - js) * 256);
                            aux = min(kExactRows, se.n_tail - (j - js) * kExactRows) | 256;
                        }
                        v = (1ull << 62) | ((unsigned long long)aux << 48) | (unsigned long long)a;
                    } else {
                        const uint8_t* src;
                        if (j < itm.n_ex + itm.seal) {
                            src = p.base + p.lay.pool + (size_t)se.seal_slot * p.slot_bytes;
                        } else {
                            const int32_t* table = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table);
                            int slot = table[((size_t)se.seq * p.num_layers + p.layer) * p.max_groups + itm.g0 +
                                             (j - itm.n_ex - itm.seal)];
                            if (slot < 0 || slot >= p.pool_slots) {
                                atomicOr(err, kErrBadSlot);
                                slot = 0;
                            }
                            src = p.base + p.lay.pool + (size_t)slot * p.slot_bytes;
                        }
                        src += (size_t)itm.kvh * (p.rec_k + p.rec_v);
                        v = (2ull << 62) | (unsigned long long)(uintptr_t)src;
                    }
                    sm.ent[e] = v;
                }
            }
            // addresses must fit the 48-bit field (they do on current GPUs; otherwise walk)
            const bool wide = ((uintptr_t)(p.base + p.lay.total) >> 48) != 0;
            if (t == 0) *sm.n_ent = (fits && !wide) ? total : -1;
        }
        if (rotator) rotate_loaded(sm, w >> 2, w & 3, lane, qrow);
        named_bar(1, kComputeThreads);
        const int n_ent = *sm.n_ent;

        // ---- 1. seal the groups completed by this step's tokens and write the other new
        //      tokens into the sink or the tail, before any copy reads them
        {
            ItemWalk wk{lo, 0};
            Item it;
            while (walk_next(p, IL, wk, hi, it)) {
                const SeqEntry& e = p.seqs[it.ci];
                const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
                const size_t blk = sl * p.hkv + it.kvh;
                const size_t rows0 = blk * (size_t)p.tail_cap;  // tail ring rows of the block
                // the new token goes to the sink or the tail ring, unless it completes the
                // group sealed now (no tail floor): then it is that group's last row
                const bool in_seal = e.seal_group >= 0 && p.tail_cap == kGroup;
                if (it.owner && e.new_pos >= 0 && !in_seal && t < 32) {
                    const int side = t >> 4, chunk = t & 15;
                    const uint16_t* src = (side ? p.v_new : p.k_new) + ((size_t)it.ci * p.hkv + it.kvh) * 128;
                    const size_t off = e.new_pos < kSink
                                           ? (side ? p.lay.sink_v : p.lay.sink_k) + (blk * 128 + e.new_pos) * 256
                                           : (side ? p.lay.tail_v : p.lay.tail_k) +
                                                 (rows0 + (size_t)((e.new_pos - kSink) % p.tail_cap)) * 256;
                    reinterpret_cast<uint4*>(p.base + off)[chunk] = reinterpret_cast<const uint4*>(src)[chunk];
                }
                if (!it.seal) continue;
                uint8_t* dst = p.base + p.lay.pool + (size_t)e.seal_slot * p.slot_bytes + (size_t)it.kvh * pair;
                if (t < kSealThreads) {  // the seal runs on 8 warps (barrier 2); the others wait below
                    const int first = (kGroup * e.seal_group) % p.tail_cap, from_tail = in_seal ? 127 : 128;
                    SealRows rk{reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_k) + (rows0 + first) * 128,
                                p.k_new + ((size_t)it.ci * p.hkv + it.kvh) * 128, from_tail};
                    seal_matrix(rk, p.k_bits, 0, p.iters, dst, nullptr, *sm.seal, 2);
                    SealRows rv{reinterpret_cast<const uint16_t*>(p.base + p.lay.tail_v) + (rows0 + first) * 128,
                                p.v_new + ((size_t)it.ci * p.hkv + it.kvh) * 128, from_tail};
                    seal_matrix(rv, p.v_bits, 1, p.iters, dst + p.rec_k, nullptr, *sm.seal, 2);
                }
                if (t == 0 && it.kvh == 0) {
                    int32_t* table = reinterpret_cast<int32_t*>(p.base + p.lay.block_table);
                    table[sl * p.max_groups + e.seal_group] = e.seal_slot;
                }
            }
        }
        // ---- query tables of the CTA's first two blocks (rotated above), by the whole CTA
        for (int k = t; k < 256 * prebuilt; k += kComputeThreads) fill_table<KB>(sm, k >> 8, (k >> 5) & 7, k & 31);
        fence_proxy_async_global();  // the rows and records just written are read by bulk copies
        named_bar(1, kComputeThreads);
        bar_arrive(3, kDecodeThreads);  // the copy-issuing warp may start

        // ---- 3. items in order, warp by warp
        const int g = lane >> 2, tq = lane & 3;
        // this warp processes group numbers w, w + kWarps, ...: stage and phase parity of the next
        uint32_t my_s = (uint32_t)w % (uint32_t)p.stages, my_par = ((uint32_t)w / (uint32_t)p.stages) & 1u;
        float* xb = sm.xbuf + w * kXbWarp;
        ItemWalk wk{lo, 0};
        Item it;
        uint32_t item_no = 0;
        int kb = -1;
        while (walk_next(p, IL, wk, hi, it)) {
            const SeqEntry& e = p.seqs[it.ci];
            ++kb;
            if (kb > 0 && lane == 0) atomicAdd(sm.ctl + 4 + ((kb - 1) & 1), 1);  // leaving block kb - 1
            acquire_table<KB>(p, sm, kb, prebuilt, it.ci, it.kvh, lane, err);
            const float qm = sm.qmax[4 * (kb & 1) + tq];
            const uint4* qtab = sm.qtab + kTabWords * (kb & 1);
            int64_t first;
            block_ctas(p, e, it.kvh, &first);
            int pslot = (int)(b - first);
            if (pslot >= kPartialSlots) {  // cannot happen with the host's schedule
                if (lane == 0) atomicOr(err, kErrSpan);
                pslot = kPartialSlots - 1;
            }
            WarpState st;
            st.m = kNegInf;
            st.l = 0.f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) st.acc[mt] = make_float2(0.f, 0.f);
            const uint32_t cnt = (uint32_t)it.count();
            uint32_t k = (uint32_t)((w + kWarps - (int)(n % kWarps)) % kWarps);
            if (k < (uint32_t)it.n_ex) {  // exact sub-groups come first
                uint32_t bq[16];
                exact_query(sm, kb & 1, g, tq, bq);
                const int js = (e.n_sink + kExactRows - 1) / kExactRows;
                for (; k < (uint32_t)it.n_ex; k += kWarps) {
                    const uint32_t gn = n + k;
                    wait_group(sm, gn, my_s, my_par, err);
                    const int j = (int)k;
                    const int rows = j < js ? min(kExactRows, e.n_sink - j * kExactRows)
                                            : min(kExactRows, e.n_tail - (j - js) * kExactRows);
                    process_exact(sm.stages + (size_t)my_s * pair, rows, bq, p.scale_log2, xb, st, g, tq, lane);
                    __syncwarp();  // every lane is done with the stage before it is released
                    if (lane == 0) mbar_arrive(sm.empty + my_s);
                    my_s += kWarps;
                    while (my_s >= (uint32_t)p.stages) {
                        my_s -= p.stages;
                        my_par ^= 1u;
                    }
                }
                // so far the state holds exact tokens only: rotate it like the records so that
                // the block's sealed groups accumulate onto it
                frag_fwht128(st.acc, lane);
            }
            for (; k < cnt; k += kWarps) {
                const uint32_t gn = n + k;
                wait_group(sm, gn, my_s, my_par, err);
                process_group<KB, VB>(p, sm.stages + (size_t)my_s * pair, qtab, qm, xb, st, g, tq, lane);
                __syncwarp();  // every lane is done with the stage before it is released
                if (lane == 0) mbar_arrive(sm.empty + my_s);
                my_s += kWarps;
                while (my_s >= (uint32_t)p.stages) {
                    my_s -= p.stages;
                    my_par ^= 1u;
                }
            }
            n += cnt;
            fold_item(p, sm, st, item_no, it.ci, it.kvh, pslot, w, g, tq, lane, err);
            ++item_no;
        }
    }
    // Normally every copy was waited for above. After a wait that gave up, let the
    // copies still in flight land (bounded) before the CTA's shared memory goes away.
    __syncthreads();
    if (t == 0 && (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout)) {
        const uint64_t t0 = global_ns();
        for (uint32_t k = n > (uint32_t)p.stages ? n - p.stages : 0; k < n; ++k)
            while (!mbar_try_wait(sm.full + (k % p.stages), (k / p.stages) & 1) && global_ns() - t0 < kWaitLimitNs) {
            }
    }
}

// Merge of every (sequence, KV head) block of a decode call: one CTA per block, one warp
// per query head. The partials of the CTAs that covered the block are merged (running
// maxima, sums and rotated accumulators), the sum is rotated back with the 128-point
// Hadamard transform and the fp16 output written. Launched right after the decode kernel
// (programmatic dependent launch); it waits for that grid's completion before reading.
__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ DecodeParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next decode launch may start its CTAs now (it waits for this grid before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int ci = blockIdx.x / p.hkv, kvh = blockIdx.x % p.hkv;
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (h >= p.r) return;
    const SeqEntry& e = p.seqs[ci];
    const int blk = e.seq * p.hkv + kvh;
    int64_t first;
    const int nsl = min(block_ctas(p, e, kvh, &first), kPartialSlots);
    // partials four at a time, every load of a round issued before any is used, combined
    // with the running maximum, sum and accumulator
    float M = kNegInf, L = 0.f, v[4] = {0.f, 0.f, 0.f, 0.f};
    bool stale = false;
    for (int s0 = 0; s0 < nsl; s0 += 4) {
        float ms[4], ls[4];
        float4 a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ms[k] = kNegInf;
            ls[k] = 0.f;
            a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s0 + k < nsl) {
                const float* P = partial_ptr(p, blk, s0 + k);
                const bool ok = (uint32_t)__float_as_int(__ldcg(P)) == p.epoch;
                const float m = __ldcg(P + 4 + h), l = __ldcg(P + 8 + h);
                const float4 av = __ldcg(reinterpret_cast<const float4*>(P + 12 + 128 * h) + lane);
                // a partial of another call (missing or overwritten) enters as nothing and
                // is reported; what its slot holds never reaches the sums
                ms[k] = ok ? m : kNegInf;
                ls[k] = ok ? l : 0.f;
                a[k] = ok ? av : make_float4(0.f, 0.f, 0.f, 0.f);
                stale |= !ok;
            }
        }
        float Mn = M;
#pragma unroll
        for (int k = 0; k < 4; ++k) Mn = fmaxf(Mn, ms[k]);
        if (Mn == kNegInf) continue;
        const float c = M == kNegInf ? 0.f : exp2f(M - Mn);
        L *= c;
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] *= c;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float wgt = ms[k] == kNegInf ? 0.f : exp2f(ms[k] - Mn);
            L = fmaf(wgt, ls[k], L);
            v[0] = fmaf(wgt, a[k].x, v[0]);
            v[1] = fmaf(wgt, a[k].y, v[1]);
            v[2] = fmaf(wgt, a[k].z, v[2]);
            v[3] = fmaf(wgt, a[k].w, v[3]);
        }
        M = Mn;
    }
    if (stale && lane == 0) atomicOr(err_word(p), kErrStalePartial);
    warp_fwht128(v, lane);
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    uint2 o;
    o.x = h2_bits(__floats2half2_rn(v[0] * inv, v[1] * inv));
    o.y = h2_bits(__floats2half2_rn(v[2] * inv, v[3] * inv));
    *reinterpret_cast<uint2*>(p.out + ((size_t)ci * p.hq + (size_t)kvh * p.r + h) * 128 + 4 * lane) = o;
}

int launch_merge(const DecodeParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_seqs * p.hkv));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, merge_kernel, p);
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
    // programmatic dependent of the work before it in the stream: the CTAs start (and
    // build their item lists) while that work drains, and wait for it before reading memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    const int rc = (int)cudaLaunchKernelEx(&cfg, decode_kernel<KB, VB>, p);
    if (rc) return rc;
    return launch_merge(p, s);
}

}  // namespace

int decode_smem_bytes(int k_bits, int v_bits, int stages, bool with_seal) {
    (void)with_seal;  // the seal scratch aliases the stage ring
    size_t pair = record_bytes(k_bits) + record_bytes(v_bits);
    size_t off = (size_t)stages * pair;
    if (off < sizeof(SealSmem)) off = sizeof(SealSmem);
    off = (off + 15) & ~(size_t)15;
    off += 2 * 32 * 8 + 32 * 4 + 2 * kTabWords * 16 + 2 * 512 * 4 + 2 * 4 * 4 + 2 * 4 * 64 * 4 + kWarps * sizeof(WarpRegion) + 2 * sizeof(ItemCtl) + 16 * 4 + 8 * 4 + 4 * sizeof(GroupCursor) + sizeof(ItemList) + 16 + kMaxEntries * 8 +
           kWarps * kXbWarp * 4;
    return (int)off;
}

// ---------------------------------------------------------------------------
// Static split-K workspace for kvarn_decode_attention_noalloc: the partial softmax
// states of up to kStaticBlocks (sequence, KV head) blocks, 8.7 MB per GPU
// that loads the library, held until the process exits. Host code must not pass the
// symbol itself to a kernel (in host code it names a host-side shadow): the device
// address is fetched once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on it.
constexpr int kStaticBlocks = 128;
static __device__ __align__(256) float kvarn_static_partials[(size_t)kStaticBlocks * kPartialSlots * kPartialFloats];

int static_workspace_blocks() { return kStaticBlocks; }

int static_workspace(void** partials) {
    static std::mutex mu;
    static void* parts[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!parts[dev]) {
        void* pp = nullptr;
        e = cudaGetSymbolAddress(&pp, kvarn_static_partials);
        if (e != cudaSuccess) return (int)e;
        parts[dev] = pp;
    }
    *partials = parts[dev];
    return 0;
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
        case 0x33: return launch_t<3, 3>(p, smem, s);
        case 0x55: return launch_t<5, 5>(p, smem, s);
        case 0x66: return launch_t<6, 6>(p, smem, s);
        case 0x65: return launch_t<6, 5>(p, smem, s);
        case 0x54: return launch_t<5, 4>(p, smem, s);
        case 0x32: return launch_t<3, 2>(p, smem, s);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace kvarn
