// KVarN prefill (many-query) attention for sm_103a on the 5th-generation tensor cores.
//
// Method (anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", sections 1 and
// 2.1): the cache is read the way the decode path reads it. Every sealed group is read
// from its record with the query rotated by the record's Hadamard matrix and the sealed
// part of the output is summed in the rotated frame; the sink and the exact tail are
// fp16 and meet the unrotated query, after the output has been rotated back (the scaled
// Sylvester matrix is its own inverse). Each query token of a prompt chunk attends
// causally (keys at positions up to its own) to the cache as it stands after the
// chunk's append.
//
// One CTA per (sequence, KV head, tile of 128 / r query tokens): 128 query rows
// (token, head), token-major, M = 128 of tcgen05.mma kind::f16 (f16 operands, f32
// accumulators in tensor memory). Adjacent tiles run as a cluster of two CTAs that walk
// the same units (those of the later tile): the visible sealed groups in order, then the
// exact blocks (the sink, then the tail, 128 tokens each). Each CTA of the pair expands
// half of every sealed group's K tile (64 channels) and V tile (64 tokens) and sends it
// to the same place in the other CTA's shared memory with one bulk copy, which completes
// on the other CTA's full barrier; the tensor cores release a tile in both CTAs
// (multicast commit), since both write it. For a
// group with codes q, token scales a, channel scales c and grid (m, delta):
//   QK  S_it = sum_j A_ij q_tj, A = v c_K as f16 high and low parts (two passes), v the
//       rotated query of row i over max|v|; the logit is
//       scale * qm_i * aK_t * (deltaK * S_it + mK * sum_j v_ij c_j).
//   PV  O_ij += sum_t W_it B_jt, W = p 2^e, B = 2^-e c_j aV_t (deltaV q_tj + mV) (the
//       dequantised value in the rotated frame; e = 0 unless it would reach 2^15): O
//       accumulates across groups in place. W and B are fp32 values carried as an f16
//       high part plus the f16 rounding of the residual; three passes (W high x B high,
//       W high x B low, W low x B high) keep the products to about 22 bits.
// Exact blocks: S = q . k on the raw fp16 query; W = p (high and low parts) against the
// fp16 values (transposed), two passes.
//
// Warp roles (640 threads, 5 warpgroups; warp w reaches tensor-memory lanes
// 32 (w % 4) .. 32 (w % 4) + 31, so thread 32 (w % 4) + lane of a warpgroup owns query
// row 32 (w % 4) + lane):
//   WG0  softmax: one thread per row; takes the unit's logits and row maximum, keeps the
//        running maximum (raised only when it grows by more than 8 in log2 units, with O
//        and l rescaled then), writes W (high and low f16 parts) over S in 32-column
//        chunks, and at the end normalises O and writes the output.
//   WG1  query operand: rotates and scales its row once, then per group writes A (high
//        and low parts) into tensor memory and the row sum sum_j v_ij c_j into shared
//        memory; before the exact blocks it writes the raw query and rotates O back.
//   WG2  K expansion: this CTA's half of the K codes of each group as f16 subnormals (or
//        the exact K rows) in a canonical K-major tile (no swizzle), the group's token
//        scales; and each unit's logits and row maxima, written over S.
//   WG3  V expansion: this CTA's half of the dequantised V values of each group as high
//        and low parts (or the exact V rows, transposed) in a canonical K-major tile.
//   WG4  warp 16 owns tensor memory and one of its threads issues every MMA, QK or PV,
//        whichever is ready first.
// Tensor memory (512 columns): A [0, 128), S0 [128, 256), S1 [256, 384), O [384, 512).
// QK of unit u + 1 runs while the softmax of unit u does; the K tiles, V tiles and S are
// double-buffered and released separately (a K tile when its QK completes, a V tile when
// its PV does). Every wait is bounded (2 s) and sets the error word when it gives up.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvarn_dev.cuh"

namespace kvarn {

namespace {

constexpr int kTcThreads = 640;      // five warpgroups
constexpr int kRows = kPrefillRows;  // 128 query rows per CTA
// registers a thread: 96 at launch (65536 / 640 rounded down to a multiple of 8), then
// re-split per warpgroup (per scheduler: one warp of each warpgroup)
constexpr int kRegsLaunch = 96, kRegsSoftmax = 112, kRegsQuery = 176, kRegsExpandK = 96, kRegsExpandV = 72,
              kRegsIssue = 24;
static_assert(kRegsSoftmax + kRegsQuery + kRegsExpandK + kRegsExpandV + kRegsIssue <= 5 * kRegsLaunch,
              "register split exceeds what a sub-partition holds at launch");
static_assert(kRegsLaunch * kTcThreads <= 65536, "launch registers");

// tensor memory columns
constexpr uint32_t kColA = 0, kColS = 128, kColO = 384;

// shared memory: two operand sets (K tile, V tile, the V expansion's token factors),
// the K-side tables of the last four units, then the small tables
constexpr int kKTile = 128 * 128 * 2;           // N = 128 tokens, K = 128 channels
constexpr int kVTile = 128 * 256 * 2;           // N = 128 channels, K = 128 tokens (high parts), 128 (low)
constexpr int kOffK = 0, kOffV = kKTile;
constexpr int kOffAlpha = kOffV + kVTile, kOffBeta = kOffAlpha + 512;  // deltaV aV_t, mV aV_t
constexpr int kSetBytes = kOffBeta + 512;
constexpr int kOffKtab = 2 * kSetBytes;         // [4][aK float[128], deltaK, mK, e, pad]
constexpr int kKtabBytes = 512 + 16;
constexpr int kOffRs = kOffKtab + 4 * kKtabBytes;  // float[4][128] row sums, ring by unit
constexpr int kOffRed = kOffRs + 4 * 128 * 4;   // float[2][2][8] expansion reductions (K, V warpgroups)
constexpr int kOffCq = kOffRed + 128;           // float[2][128] channel scales of the next query operand
constexpr int kOffMx = kOffCq + 1024;           // float[4][128] row maxima of the logits, ring by unit
constexpr int kOffPos = kOffMx + 2048;          // int[128] row positions
constexpr int kOffQm = kOffPos + 512;           // float[128] row maxima of the rotated query
constexpr int kOffVst = kOffQm + 512;           // uint32[32][128] the V expansion's code words (word k of thread t at k 128 + t)
constexpr int kOffBars = kOffVst + 32 * 128 * 4;
// barriers: k_full[4], k_empty[2], v_full[2], v_empty[2], a_full[4], a_empty, s_full[2],
// p_full[2], o_done[2], drain, m_full[4]
constexpr int kNumBars = 26;
constexpr int kOffTmem = kOffBars + 8 * kNumBars;
constexpr int kSmemTc = kOffTmem + 16;
static_assert(kSmemTc <= 227 * 1024, "shared memory of one CTA");
static_assert(kSetBytes % 128 == 0 && kOffV % 128 == 0 && kOffKtab % 16 == 0 && kKtabBytes % 16 == 0,
              "operand tiles stay 128-byte aligned");

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Canonical K-major operand without swizzle: 8-row x 16-byte core matrices, the two of
// a 16-element k-step 128 bytes apart (leading offset), 8-row groups 256 bytes apart
// (stride offset); a k-step of a tile of R rows spans R / 8 * 256 bytes.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(256 >> 4) << 32) |
           ((uint64_t)1 << 46);
}
// byte offset of element (row, k) in such a tile of 128 rows
__device__ __forceinline__ int tile_off(int row, int k) {
    return (((k >> 4) * 16 + (row >> 3)) * 2 + ((k >> 3) & 1)) * 128 + (row & 7) * 16 + (k & 7) * 2;
}
// kind::f16 instruction descriptor: f32 accumulator, f16 A and B, both K-major, M = 128, N = 128
constexpr uint32_t kIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// A from tensor memory
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}
// arrive on bar once every MMA issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
// the same, arriving on the barrier at bar's offset in both CTAs of the pair
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// ---- the CTA pair (a cluster of two: adjacent query tiles of one sequence and KV head) ----
__device__ __forceinline__ uint32_t pair_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// address in the other CTA's shared memory of the object at `local` in this one's
__device__ __forceinline__ uint32_t peer_addr(uint32_t local) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(pair_rank() ^ 1u));
    return a;
}
// every thread of both CTAs (also orders barrier initialisation before remote arrivals)
__device__ __forceinline__ void pair_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// bytes of this CTA's shared memory at `src` to the same offset in the other CTA's,
// completing (as transaction bytes) on the other CTA's barrier at bar's offset
__device__ __forceinline__ void copy_to_peer(const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     peer_addr(smem_addr(src))),
                 "r"(smem_addr(src)), "r"(bytes), "r"(peer_addr(smem_addr(bar)))
                 : "memory");
}

// 32 consecutive columns of the warp's 32 lanes: thread lane gets lane's row
__device__ __forceinline__ void tm_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
#define kNegInfT (-__int_as_float(0x7f800000))

// Bits pos .. pos + width - 1 (width <= 16) of a little-endian stream of N words.
template <int N>
__device__ __forceinline__ uint32_t bits_of(const uint32_t (&s)[N], int pos, int width) {
    const int lo = pos / 32, sh = pos % 32;
    uint32_t v = s[lo] >> sh;
    if (sh + width > 32 && lo + 1 < N) v |= s[lo + 1] << (32 - sh);
    return v & ((1u << width) - 1u);
}

// The codes enter the tensor cores as f16 subnormals: the bit pattern of a code c in
// the low bits of a half is c 2^-24, exact, so no conversion is needed; the 2^24 is
// folded into the group's scale (deltaK in the logits, deltaV aV_t in the V tile).
constexpr float kCodeUnit = 16777216.0f;  // 2^24

// Two codes at bits 0 .. B - 1 and B .. 2 B - 1 of f as a word of two f16 subnormals.
template <int B>
__device__ __forceinline__ uint32_t code_pair(uint32_t f) {
    constexpr uint32_t mask = (1u << B) - 1u;
    return (f & mask) | (((f >> B) & mask) << 16);
}

// Codes of one 16-bit field x (16 / B of them, B = 2, 4 or 8) as 8 / B words: with
// y = x | x << (16 - B), word k is (y >> 2 B k) masked to B bits in each half (the low
// half never reaches bit 16 - B, the high half reads only the shifted copy).
template <int B>
__device__ __forceinline__ void code_words16(uint32_t x, uint32_t* o) {
    constexpr uint32_t mask = ((1u << B) - 1u) * 0x00010001u;
    const uint32_t y = x | (x << (16 - B));
#pragma unroll
    for (int k = 0; k < 8 / B; ++k) o[k] = (y >> (2 * B * k)) & mask;
}

// Codes 8 m .. 8 m + 7 of a row of 128 B-bit codes held in s (4 B words) as four words
// of two f16 subnormals each.
template <int B>
__device__ __forceinline__ uint4 codes8(const uint32_t (&s)[4 * B], int m) {
    uint32_t o[4];
    if constexpr (B == 2 || B == 4 || B == 8) {
#pragma unroll
        for (int h = 0; h < B / 2; ++h) {
            const int pos = 8 * B * m + 16 * h;
            code_words16<B>((s[pos >> 5] >> (pos & 31)) & 0xffffu, o + h * (8 / B));
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = code_pair<B>(bits_of(s, (8 * m + 2 * k) * B, 2 * B));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Codes 8 m .. 8 m + 7 of a row of 128 B-bit codes staged as words k at col[128 k], as
// four words of two f16 subnormals each; m may vary at run time.
template <int B>
__device__ __forceinline__ uint4 codes8_staged(const uint32_t* col, int m) {
    const int pos = 8 * B * m, lo = pos >> 5, sh = pos & 31;
    uint64_t bits = col[128 * lo];
    if (sh + 8 * B > 32) bits |= (uint64_t)col[128 * (lo + 1)] << 32;
    bits >>= sh;
    uint32_t o[4];
    if constexpr (B == 2 || B == 4 || B == 8) {
#pragma unroll
        for (int h = 0; h < B / 2; ++h) code_words16<B>((uint32_t)(bits >> (16 * h)) & 0xffffu, o + h * (8 / B));
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = code_pair<B>((uint32_t)(bits >> (2 * B * k)));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

struct TcCta {
    const PrefillSeq* e;
    int kvh, t0;        // KV head, first query token of the tile
    int pmin, pmax;     // smallest and largest position among the tile's valid rows
    int n_sealed;       // sealed groups with a token at or before pmax
    int nb_sink;        // 1 when the sink has a visible token
    int sink_vis;       // visible sink tokens
    int tail_start, tail_vis;
    int units;          // n_sealed + exact blocks
    size_t blk;         // (sequence, layer, KV head) index of the exact regions
    int rank;           // in the CTA pair: expands K channel chunks and V token chunks 8 rank .. 8 rank + 7
};

struct Unit {
    bool sealed;
    int g;              // sealed group
    int kp0, cnt;       // exact block: first position, tokens
    bool tail;
};

__device__ __forceinline__ Unit unit_of(const TcCta& c, int u) {
    Unit x;
    x.sealed = u < c.n_sealed;
    x.g = u;
    x.tail = false;
    x.kp0 = 0;
    x.cnt = 0;
    if (!x.sealed) {
        const int e = u - c.n_sealed;
        if (e < c.nb_sink) {
            x.cnt = c.sink_vis;
        } else {
            x.tail = true;
            x.kp0 = c.tail_start + kGroup * (e - c.nb_sink);
            x.cnt = min(kGroup, c.tail_start + c.tail_vis - x.kp0);
        }
    }
    return x;
}

__device__ __forceinline__ const uint8_t* tc_group_src(const PrefillParams& p, const TcCta& c, int g) {
    const int32_t* table = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table) +
                           ((size_t)c.e->seq * p.num_layers + p.layer) * p.max_groups;
    const int slot = table[g];
    return p.base + p.lay.pool + (size_t)slot * p.slot_bytes + (size_t)c.kvh * (p.rec_k + p.rec_v);
}

// fp16 row of an exact block (side 0 = K, 1 = V) at position pos
__device__ __forceinline__ const uint4* exact_row(const PrefillParams& p, const TcCta& c, bool tail, int side, int pos) {
    size_t off;
    if (tail)
        off = (side ? p.lay.tail_v : p.lay.tail_k) + (c.blk * p.tail_cap + (size_t)((pos - kSink) % p.tail_cap)) * 256;
    else
        off = (side ? p.lay.sink_v : p.lay.sink_k) + (c.blk * kSink + pos) * 256;
    return reinterpret_cast<const uint4*>(p.base + off);
}

// bars: [0, 4) k_full (by unit % 4), [4, 6) k_empty, [6, 8) v_full, [8, 10) v_empty,
// [10, 14) a_full (by unit % 4), 14 a_empty, [15, 17) s_full, [17, 19) p_full,
// [19, 21) o_done (PV of unit v completes phase v / 2 of o_done[v % 2]), 21 drain (once),
// [22, 26) m_full (by unit % 4: the unit's logits and row maxima are in place).
// A barrier is indexed so that its previous phase has always completed when a thread
// waits for the next: a parity wait cannot then be satisfied by an older phase. For
// o_done this follows from tcgen05.mma completing in issue order: every wait for PV(v)
// comes after its thread has seen QK(v) or a later MMA complete, and PV(v - 2) is issued
// before QK(v) (QK(v) reuses the S buffer of PV(v - 2)'s weights).
constexpr int kBarKFull = 0, kBarKEmpty = 4, kBarVFull = 6, kBarVEmpty = 8, kBarAFull = 10, kBarAEmpty = 14,
              kBarSFull = 15, kBarPFull = 17, kBarODone = 19, kBarDrain = 21, kBarMFull = 22;

// wait until PV of unit v has completed
__device__ __forceinline__ void wait_pv(uint64_t* bars, int v, int32_t* err) {
    mbar_wait(bars + kBarODone + (v & 1), (uint32_t)((v >> 1) & 1), err);
}

// ---- WG4: the MMA issuer (one thread) ----
// QK(u) into S[u % 2] once the K tile and the query operand of unit u are in place and
// PV(u - 2), the last reader of that S buffer, has been issued; PV(u) into O once the
// weights of unit u and its V tile are in place. Whichever is ready is issued first.
__device__ __forceinline__ void issue_qk(const TcCta& c, uint32_t sbase, uint64_t* bars, uint32_t tmem, int u) {
    const int b = u & 1;
    const bool sealed = u < c.n_sealed;
    tc_fence_after();
    const uint32_t d = tmem + kColS + 128u * b;
    const uint32_t kt = sbase + b * kSetBytes + kOffK;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) mma_ts(d, tmem + kColA + 8 * ks, smem_desc(kt + ks * 4096), ks > 0);
    if (sealed) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_ts(d, tmem + kColA + 64 + 8 * ks, smem_desc(kt + ks * 4096), 1u);
    }
    mma_commit(bars + kBarSFull + b);
    mma_commit_pair(bars + kBarKEmpty + b);  // both CTAs write this CTA's K tile
    if (sealed) mma_commit(bars + kBarAEmpty);
}

__device__ __forceinline__ void issue_pv(const TcCta& c, uint32_t sbase, uint64_t* bars, uint32_t tmem, int v) {
    const int b = v & 1;
    tc_fence_after();
    const uint32_t a = tmem + kColS + 128u * b;
    const uint32_t vt = sbase + b * kSetBytes + kOffV;
    // W high x B high, W high x B low (sealed only), W low x B high; the weights of
    // k-step ks sit in columns 16 ks (high) and 16 ks + 8 (low)
    const int passes = v < c.n_sealed ? 3 : 2;
    for (int ps = 0; ps < passes; ++ps) {
        const uint32_t alo = ps == passes - 1 ? 8u : 0u;
        const uint32_t bks = ps == 1 && passes == 3 ? 8u : 0u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_ts(tmem + kColO, a + 16 * ks + alo, smem_desc(vt + (bks + ks) * 4096),
                   (v > 0 || ps > 0 || ks > 0) ? 1u : 0u);
    }
    mma_commit_pair(bars + kBarVEmpty + b);  // both CTAs write this CTA's V tile
    mma_commit(bars + kBarODone + b);
}

// non-blocking test of a barrier phase (try_wait may suspend the thread for a while)
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void issue_role(const TcCta& c, uint8_t* smem, uint64_t* bars, uint32_t tmem,
                                           int32_t* err) {
    const uint32_t sbase = smem_addr(smem);
    int nq = 0, np = 0;  // next QK, next PV
    uint64_t t0 = global_ns();
    while (np < c.units) {
        bool did = false;
        if (nq < c.units && nq <= np + 1 && mbar_test(bars + kBarKFull + (nq & 3), (uint32_t)((nq >> 2) & 1)) &&
            (nq > c.n_sealed || mbar_test(bars + kBarAFull + (nq & 3), (uint32_t)((nq >> 2) & 1)))) {
            issue_qk(c, sbase, bars, tmem, nq);
            ++nq;
            did = true;
        } else if (np < nq && mbar_test(bars + kBarPFull + (np & 1), (uint32_t)((np >> 1) & 1)) &&
                   mbar_test(bars + kBarVFull + (np & 1), (uint32_t)((np >> 1) & 1))) {
            issue_pv(c, sbase, bars, tmem, np);
            ++np;
            did = true;
        }
        if (did) {
            t0 = global_ns();
        } else if (global_ns() - t0 > kWaitLimitNs || (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout)) {
            atomicOr(err, kErrTimeout);
            return;
        } else {
            __nanosleep(32);  // leave the scheduler's issue slots to the softmax warp
        }
    }
}

__device__ __forceinline__ float wg_max(float x, float* red, int et, int id) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    if ((et & 31) == 0) red[et >> 5] = x;
    named_bar(id, 128);
    return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

// The group's power of two e (its dequantised values times 2^-e stay below 2^15; the
// weights take 2^e), computed alike by both expansion warpgroups from the V header.
template <int VB>
__device__ __forceinline__ int group_exponent(float aV, float cV, float dV, float mV, float* red, int et, int id) {
    const float amax = wg_max(aV, red, et, id);
    const float cmax = wg_max(cV, red + 4, et, id);
    const float bound = amax * cmax * (fabsf(mV) + fabsf(dV) * (float)((1 << VB) - 1));
    int e = 0;
    if (bound > 32768.f) frexpf(bound * (1.0f / 32768.f), &e);
    return e;
}

// What a thread of an expansion warpgroup reads of one record: its row of 128 codes
// (B bits each) and the scales of its token / channel index.
template <int B>
struct RecRow {
    uint32_t w[4 * B];
    float a, cV, aV, d, m, dV, mV;
};

// Loads of unit u's V record for thread et, issued a unit ahead of their use.
template <int VB>
__device__ __forceinline__ void load_v(const PrefillParams& p, const TcCta& c, int u, int et, RecRow<VB>& L) {
    if (u >= c.n_sealed) return;
    const uint8_t* vr = tc_group_src(p, c, u) + p.rec_k;
#pragma unroll
    for (int i = 0; i < VB; ++i) {
        const uint4 v4 = reinterpret_cast<const uint4*>(vr + 528 + et * 16 * VB)[i];
        L.w[4 * i] = v4.x; L.w[4 * i + 1] = v4.y; L.w[4 * i + 2] = v4.z; L.w[4 * i + 3] = v4.w;
    }
    L.aV = __half2float(reinterpret_cast<const __half*>(vr + 16)[et]);
    L.cV = __half2float(reinterpret_cast<const __half*>(vr + 272)[et]);
    L.dV = *reinterpret_cast<const float*>(vr);
    L.mV = *reinterpret_cast<const float*>(vr + 4);
}

// ---- WG3: the V tile of every unit (thread et = 0..127) ----
template <int VB>
__device__ __forceinline__ void expand_v_role(const PrefillParams& p, const TcCta& c, uint8_t* smem, uint64_t* bars,
                                              int32_t* err, int et) {
    const int lane = et & 31, wv = et >> 5;
    float* red_all = reinterpret_cast<float*>(smem + kOffRed) + 16;
    RecRow<VB> nx;
    load_v<VB>(p, c, 0, et, nx);
    for (int u = 0; u < c.units; ++u) {
        const int b = u & 1;
        const Unit x = unit_of(c, u);
        uint8_t* set = smem + b * kSetBytes;
        if (x.sealed) {
            const RecRow<VB> L = nx;
            load_v<VB>(p, c, u + 1, et, nx);
            const uint32_t(&vs_)[4 * VB] = L.w;
            const float aV = L.aV, cV = L.cV, dV = L.dV, mV = L.mV;
            if (u >= 2) mbar_wait(bars + kBarVEmpty + b, (uint32_t)(((u >> 1) - 1) & 1), err);
            // B = the dequantised value in the rotated frame, c_j aV_t (deltaV q_tj + mV), times 2^-e
            float* alpha = reinterpret_cast<float*>(set + kOffAlpha);
            float* beta = reinterpret_cast<float*>(set + kOffBeta);
            alpha[et] = dV * aV * kCodeUnit;  // the codes are c 2^-24
            beta[et] = mV * aV;
            // (the reductions' barriers also publish alpha and beta)
            const int e = group_exponent<VB>(aV, cV, dV, mV, red_all + 8 * b, et, 1);
            const float cs = ldexpf(cV, -e);
            const float2 cs2 = make_float2(cs, cs), m1 = make_float2(-1.f, -1.f);
            // row = channel et: f16 high parts in k-steps 0..7, the f16 rounding of the
            // residuals in k-steps 8..15
            const float2* al2 = reinterpret_cast<const float2*>(alpha);
            const float2* be2 = reinterpret_cast<const float2*>(beta);
            uint32_t* vst = reinterpret_cast<uint32_t*>(smem + kOffVst) + et;
#pragma unroll
            for (int k = 0; k < 4 * VB; ++k) vst[128 * k] = vs_[k];
            // this CTA's half: tokens 64 rank .. 64 rank + 63 (k-steps 4 rank .. 4 rank + 3 of
            // the high parts and 8 + 4 rank .. of the low parts); the other CTA sends the rest
#pragma unroll 1
            for (int m = 8 * c.rank; m < 8 * c.rank + 8; ++m) {
                const uint4 q4 = codes8_staged<VB>(vst, m);
                const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = __fmul2_rn(cs2, __ffma2_rn(__half22float2(u2h(qw[j])), al2[4 * m + j], be2[4 * m + j]));
                    const __half2 h = __float22half2_rn(x);
                    hi[j] = h2u(h);
                    lo[j] = h2u(__float22half2_rn(__ffma2_rn(__half22float2(h), m1, x)));
                }
                *reinterpret_cast<uint4*>(set + kOffV + tile_off(et, 8 * m)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(set + kOffV + tile_off(et, 128 + 8 * m)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        } else {
            // exact block: V rows transposed (movmatrix) into channel rows; core matrix
            // cm = (ks 16 + rg) 2 + kc holds channels 8 rg .., tokens 16 ks + 8 kc ..
            if (u >= 2) mbar_wait(bars + kBarVEmpty + b, (uint32_t)(((u >> 1) - 1) & 1), err);
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t a[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int cm = wv + 4 * (32 * hh + i);
                    const int ks = cm >> 5, rg = (cm >> 1) & 15, kc = cm & 1;
                    const int tt = 16 * ks + 8 * kc + (lane >> 2);
                    a[i] = 0u;
                    if (tt < x.cnt)
                        a[i] = reinterpret_cast<const uint32_t*>(exact_row(p, c, x.tail, 1, x.kp0 + tt))[4 * rg + (lane & 3)];
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int cm = wv + 4 * (32 * hh + i);
                    uint32_t d;
                    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a[i]));
                    *reinterpret_cast<uint32_t*>(set + kOffV + cm * 128 + 4 * lane) = d;
                }
            }
        }
        fence_proxy_async_smem();
        if (x.sealed) {
            named_bar(7, 128);
            if (et == 0) {
                copy_to_peer(set + kOffV + 4 * c.rank * 4096, 4 * 4096, bars + kBarVFull + b);
                copy_to_peer(set + kOffV + (8 + 4 * c.rank) * 4096, 4 * 4096, bars + kBarVFull + b);
                mbar_arrive_expect_tx(bars + kBarVFull + b, 8 * 4096);
            } else {
                mbar_arrive(bars + kBarVFull + b);
            }
        } else {
            mbar_arrive(bars + kBarVFull + b);
        }
    }
}

// 128-point Hadamard transform of a row held by one thread, scaled by 1 / sqrt(128);
// the lower index of each pair takes a + b (the Sylvester order of the records).
__device__ __forceinline__ void fwht_row(float (&v)[128]) {
#pragma unroll
    for (int len = 1; len < 128; len <<= 1) {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
            if (i & len) continue;
            const float a = v[i], b = v[i + len];
            v[i] = a + b;
            v[i + len] = a - b;
        }
    }
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] *= kInvSqrt128;
}

// Row i of the tile: its query vector (null when the row is past the chunk).
__device__ __forceinline__ const uint4* query_row(const PrefillParams& p, const TcCta& c, int i) {
    const int tok = c.t0 + i / p.r;
    if (tok >= c.e->q_len) return nullptr;
    const size_t qrow = (size_t)(c.e->q_row + tok) * p.hq + (size_t)c.kvh * p.r + i % p.r;
    return reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim);
}

// ---- WG1: the query operand in tensor memory (thread i = row i) ----
__device__ __forceinline__ void query_role(const PrefillParams& p, const TcCta& c, uint8_t* smem, uint64_t* bars,
                                           uint32_t tmem, int32_t* err, int i, uint32_t lane_off) {
    const uint4* qv = query_row(p, c, i);
    float* rowqm = reinterpret_cast<float*>(smem + kOffQm);
    float* rsring = reinterpret_cast<float*>(smem + kOffRs);
    float* cq = reinterpret_cast<float*>(smem + kOffCq);
    const uint32_t ta = tmem + lane_off + kColA;
    if (c.n_sealed > 0) {
        float v[128];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint4 r4 = qv ? qv[k] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w4[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(u2h(w4[j]));
                v[8 * k + 2 * j] = f.x;
                v[8 * k + 2 * j + 1] = f.y;
            }
        }
        fwht_row(v);
        float qm = 0.f;
#pragma unroll
        for (int k = 0; k < 128; ++k) qm = fmaxf(qm, fabsf(v[k]));
        const float inv = qm > 0.f ? 1.0f / qm : 0.f;
#pragma unroll
        for (int k = 0; k < 128; ++k) v[k] *= inv;
        rowqm[i] = qm;
        // channel i of the next group's c_K, fetched one group ahead
        float cnext = __half2float(reinterpret_cast<const __half*>(tc_group_src(p, c, 0) + 272)[i]);
        for (int u = 0; u < c.n_sealed; ++u) {
            const float cme = cnext;
            if (u + 1 < c.n_sealed)
                cnext = __half2float(reinterpret_cast<const __half*>(tc_group_src(p, c, u + 1) + 272)[i]);
            float* cu = cq + 128 * (u & 1);
            cu[i] = cme;
            named_bar(2, 128);
            if (u >= 1) mbar_wait(bars + kBarAEmpty, (uint32_t)((u - 1) & 1), err);
            tc_fence_after();
            float2 rs2 = make_float2(0.f, 0.f);
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    const float4 c4 = reinterpret_cast<const float4*>(cu)[4 * cc + qd];
                    const int ch = 16 * cc + 4 * qd;
                    const float2 x01 = __fmul2_rn(make_float2(v[ch], v[ch + 1]), make_float2(c4.x, c4.y));
                    const float2 x23 = __fmul2_rn(make_float2(v[ch + 2], v[ch + 3]), make_float2(c4.z, c4.w));
                    rs2 = __fadd2_rn(rs2, __fadd2_rn(x01, x23));
                    const __half2 h01 = __float22half2_rn(x01), h23 = __float22half2_rn(x23);
                    hi[2 * qd] = h2u(h01);
                    hi[2 * qd + 1] = h2u(h23);
                    lo[2 * qd] = h2u(__float22half2_rn(__ffma2_rn(__half22float2(h01), m1, x01)));
                    lo[2 * qd + 1] = h2u(__float22half2_rn(__ffma2_rn(__half22float2(h23), m1, x23)));
                }
                tm_st8(ta + 8 * cc, hi);
                tm_st8(ta + 64 + 8 * cc, lo);
            }
            tm_wait_st();
            rsring[128 * (u & 3) + i] = rs2.x + rs2.y;
            tc_fence_before();
            mbar_arrive(bars + kBarAFull + (u & 3));
        }
        mbar_wait(bars + kBarAEmpty, (uint32_t)((c.n_sealed - 1) & 1), err);
        tc_fence_after();
    }
    // the raw query for the exact blocks
    uint32_t raw[32];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 r4 = qv ? qv[8 * hh + k] : make_uint4(0u, 0u, 0u, 0u);
            raw[4 * k] = r4.x; raw[4 * k + 1] = r4.y; raw[4 * k + 2] = r4.z; raw[4 * k + 3] = r4.w;
        }
        tm_st32(ta + 32 * hh, raw);
    }
    tm_wait_st();
    tc_fence_before();
    mbar_arrive(bars + kBarAFull + (c.n_sealed & 3));
    if (c.n_sealed > 0) {
        // once the last sealed group is in O, rotate row i of O back to the original frame
        // for the exact blocks, then release the softmax warpgroups
        wait_pv(bars, c.n_sealed - 1, err);
        tc_fence_after();
        const uint32_t to = tmem + lane_off + kColO;
        float o[128];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t r[32];
            tm_ld32(to + 32 * ch, r);
            tm_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[32 * ch + j] = __uint_as_float(r[j]);
        }
        fwht_row(o);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(o[32 * ch + j]);
            tm_st32(to + 32 * ch, r);
        }
        tm_wait_st();
        tc_fence_before();
        named_bar(4, 256);
    }
}

// O *= f over the thread's row (O complete up to the last PV issued)
__device__ __forceinline__ void scale_o(uint32_t to, float f) {
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        tm_ld32(to + 32 * ch, r);
        tm_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
        tm_st32(to + 32 * ch, r);
    }
    tm_wait_st();
}

// Logits (log2 units) of 32 keys of a chunk, minus `sub`: sealed aK_t (al S + be) - sub,
// exact S al - sub; keys past the block's end or the row's position are -inf.
__device__ __forceinline__ void chunk_logits(const uint32_t (&r)[32], float (&w)[32], bool sealed, const float* aK,
                                             int ch, float al, float be, float sub, bool masked, int kcnt, int kbase,
                                             int pi) {
    const float2 al2 = make_float2(al, al), ns2 = make_float2(-sub, -sub);
    if (sealed) {
        const float2 be2 = make_float2(be, be);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
            const float4 a4 = reinterpret_cast<const float4*>(aK)[8 * ch + j4];
            const float2 s01 = __ffma2_rn(al2, make_float2(__uint_as_float(r[4 * j4]), __uint_as_float(r[4 * j4 + 1])), be2);
            const float2 s23 =
                __ffma2_rn(al2, make_float2(__uint_as_float(r[4 * j4 + 2]), __uint_as_float(r[4 * j4 + 3])), be2);
            const float2 w01 = __ffma2_rn(make_float2(a4.x, a4.y), s01, ns2);
            const float2 w23 = __ffma2_rn(make_float2(a4.z, a4.w), s23, ns2);
            w[4 * j4] = w01.x;
            w[4 * j4 + 1] = w01.y;
            w[4 * j4 + 2] = w23.x;
            w[4 * j4 + 3] = w23.y;
        }
    } else {
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) {
            const float2 w2 =
                __ffma2_rn(make_float2(__uint_as_float(r[2 * j2]), __uint_as_float(r[2 * j2 + 1])), al2, ns2);
            w[2 * j2] = w2.x;
            w[2 * j2 + 1] = w2.y;
        }
    }
    if (masked) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (32 * ch + j >= kcnt || kbase + 32 * ch + j > pi) w[j] = kNegInfT;
    }
}

// Weights of 16 keys (one k-step) as f16 high parts then the f16 rounding of the residuals.
__device__ __forceinline__ void split16(const float* w, uint32_t* o) {
    const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float2 x = make_float2(w[2 * q], w[2 * q + 1]);
        const __half2 hv = __float22half2_rn(x);
        o[q] = h2u(hv);
        o[8 + q] = h2u(__float22half2_rn(__ffma2_rn(__half22float2(hv), m1, x)));
    }
}

// Loads of unit u's K record (and the V header the group's power of two needs) for
// thread et, issued ahead of their use.
template <int KB>
__device__ __forceinline__ void load_k(const PrefillParams& p, const TcCta& c, int u, int et, RecRow<KB>& L) {
    if (u >= c.n_sealed) return;
    const uint8_t* kr = tc_group_src(p, c, u);
    const uint8_t* vr = kr + p.rec_k;
#pragma unroll
    for (int i = 0; i < KB; ++i) {
        const uint4 v4 = reinterpret_cast<const uint4*>(kr + 528 + et * 16 * KB)[i];
        L.w[4 * i] = v4.x; L.w[4 * i + 1] = v4.y; L.w[4 * i + 2] = v4.z; L.w[4 * i + 3] = v4.w;
    }
    L.a = __half2float(reinterpret_cast<const __half*>(kr + 16)[et]);
    L.d = *reinterpret_cast<const float*>(kr);
    L.m = *reinterpret_cast<const float*>(kr + 4);
    L.aV = __half2float(reinterpret_cast<const __half*>(vr + 16)[et]);
    L.cV = __half2float(reinterpret_cast<const __half*>(vr + 272)[et]);
    L.dV = *reinterpret_cast<const float*>(vr);
    L.mV = *reinterpret_cast<const float*>(vr + 4);
}

// ---- WG2: the K tile and the K-side tables of unit u (thread et = 0..127) ----
template <int KB, int VB>
__device__ __forceinline__ void expand_k_unit(const PrefillParams& p, const TcCta& c, uint8_t* smem, uint64_t* bars,
                                              int32_t* err, int et, int u, const RecRow<KB>& L) {
    float* red_all = reinterpret_cast<float*>(smem + kOffRed);
    const int b = u & 1;
    const Unit x = unit_of(c, u);
    uint8_t* set = smem + b * kSetBytes;
    float* kt = reinterpret_cast<float*>(smem + kOffKtab + (u & 3) * kKtabBytes);
    if (x.sealed) {
        // the set's K tile is free once QK(u - 2) has completed; the table slot u % 4 once
        // the softmax of unit u - 4 is done, which QK(u - 2) being issued implies
        if (u >= 2) mbar_wait(bars + kBarKEmpty + b, (uint32_t)(((u >> 1) - 1) & 1), err);
        const int e = group_exponent<VB>(L.aV, L.cV, L.dV, L.mV, red_all + 8 * b, et, 5);
        // this CTA's half of the tile: channels 64 rank .. 64 rank + 63 (k-steps 4 rank ..
        // 4 rank + 3, 16 KB in one piece); the other CTA sends the rest
        uint32_t hw[4 * KB];  // the half's code words first (selected, not indexed at run time)
#pragma unroll
        for (int k = 0; k < 4 * KB; ++k) hw[k] = k < 2 * KB ? (c.rank ? L.w[2 * KB + k] : L.w[k]) : 0u;
#pragma unroll
        for (int mm = 0; mm < 8; ++mm)
            *reinterpret_cast<uint4*>(set + kOffK + tile_off(et, 8 * (8 * c.rank + mm))) = codes8<KB>(hw, mm);
        kt[et] = L.a;
        if (et == 0) {
            kt[128] = L.d * kCodeUnit;  // the codes are c 2^-24
            kt[129] = L.m;
            kt[130] = (float)e;
        }
    } else {
        // exact block: the K rows as they are (rows past the block's end are zeros)
        const bool live = et < x.cnt;
        const uint4* src = live ? exact_row(p, c, x.tail, 0, x.kp0 + et) : nullptr;
        if (u >= 2) mbar_wait(bars + kBarKEmpty + b, (uint32_t)(((u >> 1) - 1) & 1), err);
#pragma unroll 1
        for (int i0 = 0; i0 < 16; i0 += 4) {
            uint4 kr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) kr[i] = live ? src[i0 + i] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(set + kOffK + tile_off(et, 8 * (i0 + i))) = kr[i];
        }
    }
    fence_proxy_async_smem();
    if (x.sealed) {
        // the half goes to the same place in the other CTA once all of it is written;
        // this CTA's k_full also waits for the 16 KB coming the other way
        named_bar(6, 128);
        if (et == 0) {
            copy_to_peer(set + kOffK + 4 * c.rank * 4096, 4 * 4096, bars + kBarKFull + (u & 3));
            mbar_arrive_expect_tx(bars + kBarKFull + (u & 3), 4 * 4096);
        } else {
            mbar_arrive(bars + kBarKFull + (u & 3));
        }
    } else {
        mbar_arrive(bars + kBarKFull + (u & 3));
    }
}

// ---- WG2: the logits of unit v for row i (once QK(v) has completed): written back
// over S as fp32 (log2 units, masked keys -inf), the row maximum into the ring ----
__device__ __forceinline__ void logits_unit(const PrefillParams& p, const TcCta& c, uint8_t* smem, uint64_t* bars,
                                            uint32_t tmem, int32_t* err, int i, uint32_t lane_off, int v) {
    const int b = v & 1;
    const Unit x = unit_of(c, v);
    const int pi = reinterpret_cast<const int*>(smem + kOffPos)[i];
    const float* kt = reinterpret_cast<const float*>(smem + kOffKtab + (v & 3) * kKtabBytes);
    mbar_wait(bars + kBarSFull + b, (uint32_t)((v >> 1) & 1), err);
    float al = p.scale_log2, be = 0.f;
    int kbase, kcnt;
    if (x.sealed) {
        mbar_wait(bars + kBarAFull + (v & 3), (uint32_t)((v >> 2) & 1), err);
        const float qm = reinterpret_cast<const float*>(smem + kOffQm)[i];
        al = p.scale_log2 * qm * kt[128];
        be = p.scale_log2 * qm * kt[129] * reinterpret_cast<const float*>(smem + kOffRs)[128 * (v & 3) + i];
        kbase = kSink + kGroup * x.g;
        kcnt = kGroup;
    } else {
        kbase = x.kp0;
        kcnt = x.cnt;
    }
    tc_fence_after();
    const uint32_t ts = tmem + lane_off + kColS + 128u * b;
    const bool masked = kcnt < kGroup || kbase + kGroup - 1 > c.pmin;
    float mx = kNegInfT;
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        tm_ld32(ts + 32 * ch, r);
        tm_wait_ld();
        float w[32];
        chunk_logits(r, w, x.sealed, kt, ch, al, be, 0.f, masked, kcnt, kbase, pi);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            mx = fmaxf(mx, w[j]);
            r[j] = __float_as_uint(w[j]);
        }
        tm_st32(ts + 32 * ch, r);
    }
    reinterpret_cast<float*>(smem + kOffMx)[128 * (v & 3) + i] = mx;
    tm_wait_st();
    tc_fence_before();
    mbar_arrive(bars + kBarMFull + (v & 3));
}

// WG2's loop: the K tiles of units 0 and 1, then per unit v the logits of v (as soon as
// QK(v) completes) followed by the K tile of v + 2 (whose slot QK(v) has just freed),
// that tile's loads issued before the logits.
template <int KB, int VB>
__device__ __forceinline__ void k_role(const PrefillParams& p, const TcCta& c, uint8_t* smem, uint64_t* bars,
                                       uint32_t tmem, int32_t* err, int et, uint32_t lane_off) {
    for (int u = 0; u < 2 && u < c.units; ++u) {
        RecRow<KB> L;
        load_k<KB>(p, c, u, et, L);
        expand_k_unit<KB, VB>(p, c, smem, bars, err, et, u, L);
    }
    for (int v = 0; v < c.units; ++v) {
        RecRow<KB> L;
        load_k<KB>(p, c, v + 2, et, L);
        logits_unit(p, c, smem, bars, tmem, err, et, lane_off, v);
        if (v + 2 < c.units) expand_k_unit<KB, VB>(p, c, smem, bars, err, et, v + 2, L);
    }
}

// ---- WG0: softmax, rescaling and the output (thread i = row i) ----
__device__ __forceinline__ void softmax_role(const PrefillParams& p, const TcCta& c, uint8_t* smem, uint64_t* bars,
                                             uint32_t tmem, int32_t* err, int i, uint32_t lane_off) {
    const uint32_t to = tmem + lane_off + kColO;
    float m_used = kNegInfT, l = 0.f;
    for (int u = 0; u < c.units; ++u) {
        const int b = u & 1;
        const Unit x = unit_of(c, u);
        if (!x.sealed && u == c.n_sealed && u > 0) {
            // all sealed groups are in O: the query warpgroup rotates it back to the
            // original frame before any thread here touches O again
            tc_fence_before();
            named_bar(4, 256);
            tc_fence_after();
        }
        // the unit's logits (over S) and row maximum, from the K warpgroup
        mbar_wait(bars + kBarMFull + (u & 3), (uint32_t)((u >> 2) & 1), err);
        const float e = x.sealed ? reinterpret_cast<const float*>(smem + kOffKtab + (u & 3) * kKtabBytes)[130] : 0.f;
        const float mx = reinterpret_cast<const float*>(smem + kOffMx)[128 * (u & 3) + i];
        tc_fence_after();
        const uint32_t ts = tmem + lane_off + kColS + 128u * b;
        // raise the reference maximum where it grew by more than 8; O and l follow (O
        // holds PV of every earlier unit). Tensor-memory accesses are warp-wide: the
        // whole warp rescales, by 1 in the rows that keep their maximum.
        const bool raise = mx > m_used + 8.0f;
        const float corr = raise ? ex2f(m_used - mx) : 1.0f;
        if (raise) {
            l *= corr;
            m_used = mx;
        }
        if (u > 0 && __any_sync(0xffffffffu, raise)) {
            wait_pv(bars, u - 1, err);
            tc_fence_after();
            scale_o(to, corr);
        }
        // weights W = 2^(logit - m + e) as f16 high and low parts, written over the
        // chunk's own columns: k-step ks (16 tokens) holds the high parts in columns
        // 16 ks .. 16 ks + 7 and the low parts in 16 ks + 8 .. 16 ks + 15
        const float sub = (m_used == kNegInfT ? 0.f : m_used) - e;
        const float2 ns2 = make_float2(-sub, -sub);
        float ws0 = 0.f, ws1 = 0.f;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t r[32];
            tm_ld32(ts + 32 * ch, r);
            tm_wait_ld();
            float w[32];
            float2 ws2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j2 = 0; j2 < 16; ++j2) {
                const float2 d = __fadd2_rn(make_float2(__uint_as_float(r[2 * j2]), __uint_as_float(r[2 * j2 + 1])), ns2);
                w[2 * j2] = ex2f(d.x);
                w[2 * j2 + 1] = ex2f(d.y);
                ws2 = __fadd2_rn(ws2, make_float2(w[2 * j2], w[2 * j2 + 1]));
            }
            ws0 += ws2.x;
            ws1 += ws2.y;
            uint32_t o[32];
            split16(w, o);
            split16(w + 16, o + 16);
            tm_st32(ts + 32 * ch, o);
        }
        l += ldexpf(ws0 + ws1, -(int)e);
        tm_wait_st();
        tc_fence_before();
        mbar_arrive(bars + kBarPFull + b);
    }
    // normalise and write the row
    wait_pv(bars, c.units - 1, err);
    tc_fence_after();
    const int tok = c.t0 + i / p.r;
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    uint4* dst = nullptr;
    if (tok < c.e->q_len) {
        const size_t orow = (size_t)(c.e->q_row + tok) * p.hq + (size_t)c.kvh * p.r + i % p.r;
        dst = reinterpret_cast<uint4*>(p.out + orow * kHeadDim);
    }
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        tm_ld32(to + 32 * ch, r);
        tm_wait_ld();
        if (dst) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t o4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o4[j] = h2u(__floats2half2_rn(__uint_as_float(r[8 * k + 2 * j]) * inv,
                                                  __uint_as_float(r[8 * k + 2 * j + 1]) * inv));
                dst[4 * ch + k] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
        }
    }
}

template <int KB, int VB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int t = threadIdx.x, w = t >> 5, lane = t & 31, wg = w >> 2;
    int32_t* err = reinterpret_cast<int32_t*>(p.base + p.lay.err);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);

    // the CTA's (sequence, KV head, tile): pairs of adjacent tiles (2 k, 2 k + 1) share a
    // cluster, the heaviest pairs (latest tokens) first; a sequence with an odd number of
    // tiles pads its last pair with a tile past its queries (no valid row). Both CTAs of a
    // pair walk the units of the later tile (the earlier one's rows mask what they do not
    // see), so that each expands half of every K and V tile for both.
    TcCta c;
    {
        int lo = 0, up = p.n_seqs - 1;
        while (lo < up) {
            const int mid = (lo + up + 1) >> 1;
            if (p.seqs[mid].cta_begin <= (int)blockIdx.x) lo = mid; else up = mid - 1;
        }
        c.e = &p.seqs[lo];
        const int local = (int)blockIdx.x - c.e->cta_begin;  // cta_begin is even
        c.rank = (int)pair_rank();
        c.kvh = (local >> 1) % p.hkv;
        const int pair = (c.e->n_tiles + 1) / 2 - 1 - (local >> 1) / p.hkv;
        const int qt = kRows / p.r;
        c.t0 = (2 * pair + c.rank) * qt;
        const int first_pos = c.e->n - c.e->q_len;
        c.pmin = first_pos + c.t0;
        c.pmax = first_pos + min((2 * pair + 2) * qt, c.e->q_len) - 1;  // the later tile's last row
        const int vis = c.pmax >= kSink ? (c.pmax - kSink) / kGroup + 1 : 0;
        c.n_sealed = min(c.e->n_groups, vis);
        c.blk = ((size_t)c.e->seq * p.num_layers + p.layer) * p.hkv + c.kvh;
        c.sink_vis = min(min(c.e->n, kSink), c.pmax + 1);
        c.nb_sink = c.sink_vis > 0 ? 1 : 0;
        c.tail_start = kSink + kGroup * c.e->n_groups;
        c.tail_vis = max(0, min(c.e->n, c.pmax + 1) - c.tail_start);
        c.units = c.n_sealed + c.nb_sink + (c.tail_vis + kGroup - 1) / kGroup;
        if (t < kRows) {
            const int tok = c.t0 + t / p.r;
            reinterpret_cast<int*>(smem + kOffPos)[t] = tok < c.e->q_len ? first_pos + tok : c.e->n - 1;
        }
    }
    if (t == 0) {
        for (int k = 0; k < 4; ++k) {
            mbar_init(bars + kBarKFull + k, 128);
            mbar_init(bars + kBarAFull + k, 128);
            mbar_init(bars + kBarMFull + k, 128);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(bars + kBarKEmpty + k, 2);  // the QK of both CTAs
            mbar_init(bars + kBarVFull + k, 128);
            mbar_init(bars + kBarVEmpty + k, 2);  // the PV of both CTAs
            mbar_init(bars + kBarSFull + k, 1);
            mbar_init(bars + kBarPFull + k, 128);
            mbar_init(bars + kBarODone + k, 1);
        }
        mbar_init(bars + kBarAEmpty, 1);
        mbar_init(bars + kBarDrain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 16) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_addr(smem + kOffTmem))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    pair_sync();  // the other CTA's barriers are initialised before anything arrives on them
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmem);
    const uint32_t lane_off = (uint32_t)(32 * (w & 3)) << 16;
    if (wg == 0) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        softmax_role(p, c, smem, bars, tmem, err, t, lane_off);
    } else if (wg == 1) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsQuery));
        query_role(p, c, smem, bars, tmem, err, t - 128, lane_off);
    } else if (wg == 2) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsExpandK));
        k_role<KB, VB>(p, c, smem, bars, tmem, err, t - 256, lane_off);
    } else if (wg == 3) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsExpandV));
        expand_v_role<VB>(p, c, smem, bars, err, t - 384);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
        if (w == 16 && lane == 0) {
            issue_role(c, smem, bars, tmem, err);
            // every MMA has completed before tensor memory is released (bounded even
            // after another wait gave up)
            mma_commit(bars + kBarDrain);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(bars + kBarDrain, 0u) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
    tc_fence_before();
    // neither CTA leaves while the other may still copy into it or commit to its barriers
    pair_sync();
    tc_fence_after();
    if (w == 16) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

template <int KB, int VB>
int launch_tc(const PrefillParams& p, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemTc);
        if (e != cudaSuccess) return (int)e;
        attr = true;
    }
    prefill_kernel<KB, VB><<<p.grid, kTcThreads, kSmemTc, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace

int prefill_smem_bytes() { return kSmemTc; }

int launch_prefill(const PrefillParams& p, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    switch (p.k_bits * 16 + p.v_bits) {
        case 0x22: return launch_tc<2, 2>(p, s);
        case 0x24: return launch_tc<2, 4>(p, s);
        case 0x28: return launch_tc<2, 8>(p, s);
        case 0x42: return launch_tc<4, 2>(p, s);
        case 0x44: return launch_tc<4, 4>(p, s);
        case 0x48: return launch_tc<4, 8>(p, s);
        case 0x82: return launch_tc<8, 2>(p, s);
        case 0x84: return launch_tc<8, 4>(p, s);
        case 0x88: return launch_tc<8, 8>(p, s);
        case 0x33: return launch_tc<3, 3>(p, s);
        case 0x55: return launch_tc<5, 5>(p, s);
        case 0x66: return launch_tc<6, 6>(p, s);
        case 0x65: return launch_tc<6, 5>(p, s);
        case 0x54: return launch_tc<5, 4>(p, s);
        case 0x32: return launch_tc<3, 2>(p, s);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace kvarn
