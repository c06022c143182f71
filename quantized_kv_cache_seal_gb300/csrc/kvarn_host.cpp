// Host side of the KVarN cache: argument checks, the host mirror of sequence
// lengths and pool slots, scheduling of the decode kernel, and the C ABI.
//
// Region rules (anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", 2.1):
// positions 0..127 form the sink; body group g covers positions [128 + 128 g,
// 256 + 128 g) and is sealed when its last token arrives; the partial newest group
// (the tail) stays exact. The host mirror decides every seal and slot without
// reading anything back from the device.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/kvarn.h"
#include "kvarn_internal.h"

using namespace kvarn;

namespace kvarn {
// host-side copy helpers of the snapshot calls (kvarn_seal.cu)
int memcpy_d2h_async(void* dst, const void* src, size_t bytes, void* stream);
int stream_sync(void* stream);
}  // namespace kvarn

namespace {
thread_local char g_last_error[256] = "";

void set_cuda_error(int code, const char* what) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cuda_error_string(code), code);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool bits_ok(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }

// K/V width pairs the decode kernel is built for: any of 2, 4, 8 with any; the odd widths
// 3, 5, 6 symmetric; and the presets K6/V5, K5/V4, K3/V2 (anbeeld.com section 6)
bool pair_ok(int kb, int vb) {
    const bool even = (kb == 2 || kb == 4 || kb == 8) && (vb == 2 || vb == 4 || vb == 8);
    const bool preset = (kb == 6 && vb == 5) || (kb == 5 && vb == 4) || (kb == 3 && vb == 2);
    return even || preset || (kb == vb && bits_ok(kb));
}

// Body groups sealed once a sequence holds n tokens: group g seals when group g + F
// fills (F = the tail floor in groups; 0 = the published design).
int64_t groups_sealed(int64_t n, int F) { return n > kSink ? std::max<int64_t>(0, (n - kSink) / kGroup - F) : 0; }
}  // namespace

struct kvarn_cache {
    kvarn_config cfg;
    Layout lay;
    uint8_t* base = nullptr;
    size_t bytes = 0;
    int r = 1;
    int max_groups = 0;
    size_t rec_k = 0, rec_v = 0, slot_bytes = 0;
    std::vector<int64_t> len;          // [max_seqs][num_layers]
    std::vector<int32_t> table;        // [max_seqs][num_layers][max_groups]
    std::vector<int32_t> free_slots;   // stack of free pool slots
    bool initialized = false;
    uint32_t epoch = 0;
    int sms = 152;
    int max_smem = 227 * 1024;
    bool host_only = false;
    bool test_stall = false;
    int tail_cap = kGroup;  // rows of the tail ring per (sequence, layer, KV head)
    int device = -1;        // CUDA device holding the block (set at create unless host-only)

    int64_t& L(int seq, int layer) { return len[(size_t)seq * cfg.num_layers + layer]; }
    int64_t Lc(int seq, int layer) const { return len[(size_t)seq * cfg.num_layers + layer]; }
    int32_t& T(int seq, int layer, int g) {
        return table[((size_t)seq * cfg.num_layers + layer) * max_groups + g];
    }
    int32_t Tc(int seq, int layer, int g) const {
        return table[((size_t)seq * cfg.num_layers + layer) * max_groups + g];
    }
};

namespace {

kvarn_status check_config(const kvarn_config* c) {
    if (!c) return KVARN_EINVAL;
    if (c->head_dim != kHeadDim || c->group_size != kGroup || c->sink_tokens != kSink) return KVARN_EINVAL;
    if (c->num_layers <= 0 || c->max_seqs <= 0 || c->num_kv_heads <= 0 || c->num_q_heads <= 0) return KVARN_EINVAL;
    if (c->num_q_heads % c->num_kv_heads) return KVARN_EINVAL;
    int r = c->num_q_heads / c->num_kv_heads;
    if (r != 1 && r != 2 && r != 4) return KVARN_EINVAL;
    if (!bits_ok(c->k_bits) || !bits_ok(c->v_bits) || !pair_ok(c->k_bits, c->v_bits)) return KVARN_EINVAL;
    if (c->sinkhorn_iters < 0 || c->sinkhorn_iters > 64) return KVARN_EINVAL;
    if (c->max_seq_len <= 0 || c->pool_groups < 0) return KVARN_EINVAL;
    if (c->tail_floor < 0 || c->tail_floor > 3) return KVARN_EINVAL;
    if ((int64_t)c->max_seqs * c->num_kv_heads > (1 << 24)) return KVARN_EINVAL;
    return KVARN_OK;
}

Layout make_layout(const kvarn_config& c, size_t* slot_bytes_out, int* max_groups_out) {
    Layout l{};
    int max_groups = (int)std::max<int64_t>(1, groups_sealed(c.max_seq_len, c.tail_floor));
    size_t rk = record_bytes(c.k_bits), rv = record_bytes(c.v_bits);
    size_t slot_bytes = align_up((size_t)c.num_kv_heads * (rk + rv), 256);
    size_t off = 0;
    auto take = [&](size_t n) { size_t o = off; off = align_up(off + n, 256); return o; };
    size_t seq_layers = (size_t)c.max_seqs * c.num_layers;
    size_t exact = seq_layers * c.num_kv_heads * kSink * kHeadDim * 2;
    l.err = take(16);
    l.block_table = take(seq_layers * max_groups * 4);
    l.sink_k = take(exact);
    l.sink_v = take(exact);
    l.tail_k = take(exact * (c.tail_floor + 1));  // a ring of 128 (F + 1) rows per head
    l.tail_v = take(exact * (c.tail_floor + 1));
    l.partials = take((size_t)c.max_seqs * c.num_kv_heads * kPartialSlots * kPartialFloats * 4);
    l.pool = take((size_t)c.pool_groups * slot_bytes);
    l.total = off;
    if (slot_bytes_out) *slot_bytes_out = slot_bytes;
    if (max_groups_out) *max_groups_out = max_groups;
    return l;
}

kvarn_status ensure_init(kvarn_cache* c, void* stream) {
    if (c->host_only || c->initialized) return KVARN_OK;
    int rc = launch_init(c->base, c->lay, stream);
    if (rc) { set_cuda_error(rc, "cache init"); return KVARN_ECUDA; }
    c->initialized = true;
    return KVARN_OK;
}

kvarn_status check_ids(const kvarn_cache* c, int32_t layer, int32_t n, const int32_t* ids) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers || n < 0 || (n > 0 && !ids)) return KVARN_EINVAL;
    std::vector<char> seen(c->cfg.max_seqs, 0);
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= c->cfg.max_seqs || seen[ids[i]]) return KVARN_EINVAL;
        seen[ids[i]] = 1;
    }
    return KVARN_OK;
}

// Costs of the decode schedule relative to one sealed group pair (one unit), fitted on the
// GPU from per-CTA times of decode steps over many blocks (ragged Phi-4 shape at 2 bits,
// CTAs covering 3 to 11 blocks): a 2-bit group pair 0.283 us, a 16-token exact sub-group
// 0.416 us (1.47 units), a block 3.86 us on average. A CTA's first two blocks have their
// query tables built by the whole CTA at its start; a later block has its table built by
// one warp while the others wait, so the fixed cost is charged per block beyond a CTA's
// second (item_units). Wider records make a group pair dearer; the other costs stay, so
// they shrink in units.
double pair_scale(const kvarn_cache* c) {
    return 2.0 * (528 + 2048 * 2) / (double)(c->rec_k + c->rec_v);
}

int exact_units(const kvarn_cache* c, int n_sink, int n_tail) {
    return std::max(1, (int)std::lround(1.47 * exact_subs(n_sink, n_tail) * pair_scale(c)));
}

int item_units(const kvarn_cache* c) { return (int)std::lround(16.0 * pair_scale(c)); }

int seal_units(const kvarn_cache* c) {
    // a K + V seal inside the decode kernel costs about as much as 140 group pairs of
    // 2-bit records on one SM (measured: ~43 us against ~0.31 us per group pair);
    // wider records make a group pair dearer
    const double pair2 = 2.0 * (528 + 2048 * 2);
    return std::max(1, (int)std::lround(140.0 * pair2 / (double)(c->rec_k + c->rec_v)));
}

// Greedy fill of the unit line with ranges of cost at most L, each cut as late as the
// indivisible block heads allow (a cut inside a head moves back to the head's start,
// which lies past the previous cut because L >= every head). A range's cost is its units
// plus item_cost for every block it touches beyond its first two. begin[k] = first unit
// of block k (begin[nb] = total). Stops once more than max_ranges ranges are needed.
// Returns the number of ranges (cuts in `cuts`, from 0 to the total).
int greedy_cuts(const std::vector<int64_t>& begin, const int32_t* head, int64_t L, int max_ranges, int item_cost,
                std::vector<int32_t>& cuts) {
    const int nb = (int)begin.size() - 1;
    const int64_t U = begin[nb];
    cuts.clear();
    cuts.push_back(0);
    int64_t start = 0;
    int k = 0;  // block holding the current cut position (cuts only move forward)
    while (start < U) {
        if ((int)cuts.size() > max_ranges) return max_ranges + 1;
        while (begin[k + 1] <= start) ++k;
        int64_t budget = L, pos = start, end = U;
        for (int kk = k, blocks = 1;; ++kk, ++blocks) {
            if (blocks > 2) budget -= item_cost;
            if (budget <= 0) {  // no room for another block (pos > start here)
                end = pos;
                break;
            }
            const int64_t bend = begin[kk + 1];
            if (bend - pos <= budget) {  // the rest of block kk fits
                budget -= bend - pos;
                pos = bend;
                if (pos >= U) {
                    end = U;
                    break;
                }
                continue;
            }
            end = pos + budget;  // cut inside block kk
            if (begin[kk] < end && end < begin[kk] + head[kk]) {
                end = begin[kk];
                if (end <= start) end = begin[kk] + head[kk];  // a range takes at least its first head
            }
            break;
        }
        cuts.push_back((int32_t)end);
        start = end;
    }
    return (int)cuts.size() - 1;
}

// Ranges covering each block at most max_span (one walk over blocks and cuts together).
bool spans_ok(const std::vector<int64_t>& begin, const std::vector<int32_t>& cuts, int max_span) {
    const int nb = (int)begin.size() - 1;
    const int n = (int)cuts.size() - 1;
    int c = 0;  // range holding the block's first unit
    for (int k = 0; k < nb; ++k) {
        while (c + 1 < n && cuts[c + 1] <= begin[k]) ++c;
        int z = c;  // range holding the block's last unit
        while (z + 1 < n && cuts[z + 1] <= begin[k + 1] - 1) ++z;
        if (z - c + 1 > max_span) return false;
    }
    return true;
}

kvarn_status partition_units(int nb, const int32_t* units, const int32_t* head, int max_ctas, int max_span,
                             int min_load, std::vector<int32_t>& cuts, int item_cost = 0) {
    if (nb < 1 || !units || !head || max_ctas < 1 || max_span < 1 || min_load < 1) return KVARN_EINVAL;
    std::vector<int64_t> begin(nb + 1, 0);
    int64_t lo = min_load, max_head = 1;
    for (int k = 0; k < nb; ++k) {
        if (units[k] < 1 || head[k] < 1 || head[k] > units[k]) return KVARN_EINVAL;
        begin[k + 1] = begin[k] + units[k];
        max_head = std::max<int64_t>(max_head, head[k]);
    }
    const int64_t U = begin[nb];
    if (U >= (1ll << 31)) return KVARN_ECAPACITY;
    lo = std::max(lo, max_head);
    lo = std::max<int64_t>(lo, (U + max_ctas - 1) / max_ctas);
    auto fits = [&](int64_t L) {
        return greedy_cuts(begin, head, L, max_ctas, item_cost, cuts) <= max_ctas && spans_ok(begin, cuts, max_span);
    };
    // Without block costs a bound of lo + max_head always fits the CTA count (a cut loses
    // less than one head, so every range but the last holds more than U / max_ctas units);
    // block costs or the span limit can ask for more, then the bound doubles until it fits
    // (the whole line, one range, does).
    // the whole line as one range costs its units plus the blocks beyond its second
    const int64_t whole = U + (int64_t)item_cost * std::max(0, nb - 2);
    int64_t hi = std::min(whole, lo + max_head);
    if (hi < lo) hi = lo;
    while (!fits(hi)) {
        if (hi >= whole) return KVARN_ECAPACITY;
        lo = hi + 1;
        hi = std::min(whole, 2 * hi);
    }
    // smallest bound that fits, by bisection (the range count of the greedy fill only
    // falls as L grows; the span limit, when it binds, is re-checked below)
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (fits(mid)) hi = mid; else lo = mid + 1;
    }
    while (!fits(lo)) ++lo;  // terminates: hi fitted
    return KVARN_OK;
}

// Fill the schedule of a decode call: per sequence unit offsets, the CTA ranges. The
// units of one (sequence, KV head) block are, in order: its exact part, the seal made
// in this call (if any), its sealed groups. The exact part and the seal go whole to the
// CTA that covers the block's first unit.
kvarn_status schedule(kvarn_cache* c, DecodeParams& p) {
    int64_t U = 0;
    std::vector<int32_t> units, head;
    units.reserve((size_t)p.n_seqs * p.hkv);
    head.reserve((size_t)p.n_seqs * p.hkv);
    for (int i = 0; i < p.n_seqs; ++i) {
        SeqEntry& e = p.seqs[i];
        e.unit_begin = (int32_t)U;
        int we = exact_units(c, e.n_sink, e.n_tail);
        int ws = e.seal_group >= 0 ? seal_units(c) : 0;
        e.w_exact = we;
        e.w_seal = ws;
        const int64_t per = (int64_t)we + ws + e.n_groups;
        if (U + (int64_t)p.hkv * per >= (1ll << 31)) return KVARN_ECAPACITY;
        for (int h = 0; h < p.hkv; ++h) {
            units.push_back((int32_t)per);
            head.push_back(we + ws);
        }
        U += (int64_t)p.hkv * per;
    }
    p.units_total = U;
    std::vector<int32_t> cuts;
    const int max_ctas = std::max(1, std::min(c->sms, kMaxGrid));
    // at least 24 units per CTA: fewer would make the per-CTA start and merge dominate
    kvarn_status st =
        partition_units((int)units.size(), units.data(), head.data(), max_ctas, kMaxSpan, 24, cuts, item_units(c));
    if (st) return st;
    p.grid = (int)cuts.size() - 1;
    for (size_t b = 0; b < cuts.size(); ++b) p.cta_begin[b] = cuts[b];
    return KVARN_OK;
}

// Split-K workspace placed outside the cache's device block (the allocation-free call).
struct WorkspaceOverride {
    void* partials;
    uint32_t epoch;
};

kvarn_status run_decode(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids, const void* k,
                        const void* v, const void* q, void* out, float scale, void* stream, bool step,
                        const WorkspaceOverride* ws = nullptr) {
    kvarn_status st = check_ids(c, layer, n_seqs, seq_ids);
    if (st) return st;
    if (n_seqs > kMaxBatch) return KVARN_ECAPACITY;
    if (n_seqs > 0 && (!q || !out)) return KVARN_EINVAL;
    if (step && n_seqs > 0 && (!k || !v)) return KVARN_EINVAL;
    if (!std::isfinite(scale)) return KVARN_EINVAL;
    if (n_seqs == 0) return KVARN_OK;
    const kvarn_config& cfg = c->cfg;
    // capacity checks before any state change
    int need_slots = 0;
    if (step) {
        for (int i = 0; i < n_seqs; ++i) {
            int64_t pos = c->Lc(seq_ids[i], layer);
            if (pos + 1 > cfg.max_seq_len) return KVARN_ECAPACITY;
            if (pos >= kSink && (pos - kSink) % kGroup == kGroup - 1 && (pos - kSink) / kGroup >= cfg.tail_floor)
                ++need_slots;
        }
        if ((size_t)need_slots > c->free_slots.size()) return KVARN_ECAPACITY;
    }
    static thread_local DecodeParams p;  // ~10 KB: keep it off the stack
    std::memset(&p, 0, sizeof(p));
    p.base = c->base;
    p.lay = c->lay;
    p.q = (const uint16_t*)q;
    p.out = (uint16_t*)out;
    p.k_new = step ? (const uint16_t*)k : nullptr;
    p.v_new = step ? (const uint16_t*)v : nullptr;
    p.n_seqs = n_seqs;
    p.hq = cfg.num_q_heads;
    p.hkv = cfg.num_kv_heads;
    p.r = c->r;
    p.k_bits = cfg.k_bits;
    p.v_bits = cfg.v_bits;
    p.iters = cfg.sinkhorn_iters;
    p.layer = layer;
    p.num_layers = cfg.num_layers;
    p.max_seqs = cfg.max_seqs;
    p.max_groups = c->max_groups;
    p.rec_k = (int32_t)c->rec_k;
    p.rec_v = (int32_t)c->rec_v;
    p.slot_bytes = (int32_t)c->slot_bytes;
    p.pool_slots = cfg.pool_groups;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.test_stall = c->test_stall ? 1 : 0;
    p.tail_cap = c->tail_cap;
    bool any_seal = false;
    std::vector<int32_t> taken;
    for (int i = 0; i < n_seqs; ++i) {
        SeqEntry& e = p.seqs[i];
        int s = seq_ids[i];
        int64_t n = c->Lc(s, layer);
        e.seq = s;
        e.new_pos = -1;
        e.seal_group = -1;
        e.seal_slot = -1;
        if (step) {
            e.new_pos = (int32_t)n;
            // the token completes group (n - 128) / 128; with a tail floor of F groups
            // the group F before it seals
            if (n >= kSink && (n - kSink) % kGroup == kGroup - 1 && (n - kSink) / kGroup >= cfg.tail_floor) {
                e.seal_group = (int32_t)((n - kSink) / kGroup - cfg.tail_floor);
                e.seal_slot = c->free_slots.back();
                c->free_slots.pop_back();
                taken.push_back(e.seal_slot);
                any_seal = true;
            }
            n += 1;
        }
        const int64_t sealed = groups_sealed(n, cfg.tail_floor);
        e.n_sink = (int32_t)std::min<int64_t>(n, kSink);
        e.n_groups = (int32_t)sealed - (e.seal_group >= 0 ? 1 : 0);
        e.n_tail = n > kSink ? (int32_t)(n - kSink - kGroup * sealed) : 0;
        e.tail_first = (int32_t)((kGroup * sealed) % c->tail_cap);
    }
    st = schedule(c, p);
    if (st) {
        for (int32_t s : taken) c->free_slots.push_back(s);
        return st;
    }
    int stages = 32;
    while (stages > 1 && decode_smem_bytes(cfg.k_bits, cfg.v_bits, stages, any_seal) > c->max_smem) --stages;
    if (decode_smem_bytes(cfg.k_bits, cfg.v_bits, stages, any_seal) > c->max_smem) {
        for (int32_t s : taken) c->free_slots.push_back(s);
        return KVARN_ECAPACITY;
    }
    // the decode kernel's four copy warps own the stages s % 4 == k: a ring of a multiple
    // of 4 stages gives each the same share, and entry n to warp n % 4 (measured faster
    // than one stage more)
    if (stages >= 8) stages &= ~3;
    p.stages = stages;
    if (ws) {
        p.partials = (float*)ws->partials;
        p.epoch = ws->epoch;
    } else {
        p.partials = (float*)(c->base + c->lay.partials);
        p.epoch = ++c->epoch;
    }
    if (!c->host_only) {
        st = ensure_init(c, stream);
        if (st) return st;
        int rc = launch_decode(p, decode_smem_bytes(cfg.k_bits, cfg.v_bits, stages, any_seal), stream);
        if (rc) { set_cuda_error(rc, "decode launch"); return KVARN_ECUDA; }
    }
    if (step) {
        for (int i = 0; i < n_seqs; ++i) {
            const SeqEntry& e = p.seqs[i];
            if (e.seal_group >= 0) c->T(e.seq, layer, e.seal_group) = e.seal_slot;
            c->L(e.seq, layer) += 1;
        }
    }
    return KVARN_OK;
}

// Checks of a prefill-attention call made before anything is enqueued. `added` (the
// tokens a fused call appends first, or null) extends each sequence's length.
kvarn_status check_prefill(const kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                           const int32_t* q_lens, const int32_t* added, const void* q, const void* out,
                           float scale) {
    kvarn_status st = check_ids(c, layer, n_seqs, seq_ids);
    if (st) return st;
    if (n_seqs > kMaxBatch) return KVARN_ECAPACITY;
    if (n_seqs > 0 && !q_lens) return KVARN_EINVAL;
    if (!std::isfinite(scale)) return KVARN_EINVAL;
    int64_t rows = 0, ctas = 0;
    const int qt = kPrefillRows / c->r;
    for (int i = 0; i < n_seqs; ++i) {
        const int64_t n = c->Lc(seq_ids[i], layer) + (added ? (int64_t)added[i] : 0);
        if (q_lens[i] < 0 || q_lens[i] > n) return KVARN_EINVAL;
        rows += q_lens[i];
        ctas += (int64_t)(q_lens[i] + qt - 1) / qt * c->cfg.num_kv_heads;
    }
    if (rows > 0 && (!q || !out)) return KVARN_EINVAL;
    if (rows * c->cfg.num_q_heads >= (1ll << 31) || ctas >= (1ll << 31)) return KVARN_ECAPACITY;
    if (!c->host_only && prefill_smem_bytes() > c->max_smem) return KVARN_ECAPACITY;
    return KVARN_OK;
}

// Prefill attention after check_prefill: one CTA per (sequence, KV head, query tile),
// adjacent tiles paired in clusters of two (a padding tile completes an odd count).
kvarn_status run_prefill(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                         const int32_t* q_lens, const void* q, void* out, float scale, void* stream) {
    const kvarn_config& cfg = c->cfg;
    static thread_local PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    p.base = c->base;
    p.lay = c->lay;
    p.q = (const uint16_t*)q;
    p.out = (uint16_t*)out;
    p.n_seqs = 0;
    p.hq = cfg.num_q_heads;
    p.hkv = cfg.num_kv_heads;
    p.r = c->r;
    p.k_bits = cfg.k_bits;
    p.v_bits = cfg.v_bits;
    p.layer = layer;
    p.num_layers = cfg.num_layers;
    p.max_groups = c->max_groups;
    p.rec_k = (int32_t)c->rec_k;
    p.rec_v = (int32_t)c->rec_v;
    p.slot_bytes = (int32_t)c->slot_bytes;
    p.tail_cap = c->tail_cap;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int qt = kPrefillRows / c->r;
    int64_t row = 0, ctas = 0;
    for (int i = 0; i < n_seqs; ++i) {
        const int64_t n = c->Lc(seq_ids[i], layer);
        if (q_lens[i] > 0) {  // sequences without queries take no CTA
            PrefillSeq& e = p.seqs[p.n_seqs++];
            e.seq = seq_ids[i];
            e.n = (int32_t)n;
            e.q_len = q_lens[i];
            e.q_row = (int32_t)row;
            e.n_groups = (int32_t)groups_sealed(n, cfg.tail_floor);
            e.n_tiles = (q_lens[i] + qt - 1) / qt;
            e.cta_begin = (int32_t)ctas;
            // CTA pairs of adjacent tiles (a cluster of two), so an even count per sequence
            ctas += (int64_t)((e.n_tiles + 1) / 2) * 2 * cfg.num_kv_heads;
        }
        row += q_lens[i];
    }
    if (ctas == 0) return KVARN_OK;
    p.grid = (int32_t)ctas;
    if (c->host_only) return KVARN_OK;
    kvarn_status st = ensure_init(c, stream);
    if (st) return st;
    const int rc = launch_prefill(p, stream);
    if (rc) { set_cuda_error(rc, "prefill launch"); return KVARN_ECUDA; }
    return KVARN_OK;
}

// ---- snapshot image: header, host bookkeeping, exact regions, used pool slots ----
constexpr char kSnapMagic[8] = {'K', 'V', 'A', 'R', 'N', 'S', 'N', '1'};
constexpr uint32_t kSnapVersion = 1;

struct SnapHeader {
    char magic[8];
    uint32_t version;
    uint32_t header_bytes;
    kvarn_config cfg;
    int32_t max_groups;
    int32_t reserved;
    uint64_t slot_bytes;
    uint64_t sink_bytes;   // one of the sink K / sink V regions
    uint64_t tail_bytes;   // one of the tail K / tail V regions
    uint64_t n_used;       // pool slots in the image
    uint64_t total_bytes;
};

struct SnapSizes {
    size_t seq_layers, len_bytes, table_bytes, sink_bytes, tail_bytes, total;
};

SnapSizes snap_sizes(const kvarn_cache* c, uint64_t n_used) {
    SnapSizes z{};
    z.seq_layers = (size_t)c->cfg.max_seqs * c->cfg.num_layers;
    z.len_bytes = z.seq_layers * sizeof(int64_t);
    z.table_bytes = z.seq_layers * (size_t)c->max_groups * sizeof(int32_t);
    z.sink_bytes = c->lay.sink_v - c->lay.sink_k;
    z.tail_bytes = c->lay.tail_v - c->lay.tail_k;
    z.total = sizeof(SnapHeader) + z.len_bytes + z.table_bytes + 2 * z.sink_bytes + 2 * z.tail_bytes +
              (size_t)n_used * c->slot_bytes;
    return z;
}

// Pool slots in use, ascending (every table entry of a sealed group).
std::vector<int32_t> used_slots(const kvarn_cache* c) {
    std::vector<int32_t> u;
    for (int s = 0; s < c->cfg.max_seqs; ++s)
        for (int l = 0; l < c->cfg.num_layers; ++l) {
            const int64_t ng = groups_sealed(c->Lc(s, l), c->cfg.tail_floor);
            for (int64_t g = 0; g < ng; ++g) u.push_back(c->Tc(s, l, (int)g));
        }
    std::sort(u.begin(), u.end());
    return u;
}

bool same_config(const kvarn_config& a, const kvarn_config& b) {
    return a.num_layers == b.num_layers && a.max_seqs == b.max_seqs && a.num_q_heads == b.num_q_heads &&
           a.num_kv_heads == b.num_kv_heads && a.head_dim == b.head_dim && a.k_bits == b.k_bits &&
           a.v_bits == b.v_bits && a.group_size == b.group_size && a.sink_tokens == b.sink_tokens &&
           a.sinkhorn_iters == b.sinkhorn_iters && a.max_seq_len == b.max_seq_len &&
           a.pool_groups == b.pool_groups && a.tail_floor == b.tail_floor;
}

}  // namespace

extern "C" {

size_t kvarn_record_bytes(int32_t bits) { return bits_ok(bits) ? record_bytes(bits) : 0; }

kvarn_status kvarn_device_accessible(const void* ptr, int32_t* accessible) {
    if (!accessible) return KVARN_EINVAL;
    int a = 0;
    const int rc = pointer_device_accessible(ptr, &a);
    if (rc) {
        set_cuda_error(rc, "cudaPointerGetAttributes");
        return KVARN_ECUDA;
    }
    *accessible = a;
    return KVARN_OK;
}

kvarn_status kvarn_partition_units(int32_t n_blocks, const int32_t* units, const int32_t* head, int32_t max_ctas,
                                   int32_t max_span, int32_t min_load, int32_t item_cost, int32_t* cuts,
                                   int32_t* n_ctas) {
    if (!cuts || !n_ctas || item_cost < 0) return KVARN_EINVAL;
    std::vector<int32_t> c;
    kvarn_status st = partition_units(n_blocks, units, head, max_ctas, max_span, min_load, c, item_cost);
    if (st) return st;
    std::copy(c.begin(), c.end(), cuts);
    *n_ctas = (int32_t)c.size() - 1;
    return KVARN_OK;
}

kvarn_status kvarn_cache_required_bytes(const kvarn_config* cfg, size_t* bytes) {
    kvarn_status st = check_config(cfg);
    if (st) return st;
    if (!bytes) return KVARN_EINVAL;
    *bytes = make_layout(*cfg, nullptr, nullptr).total;
    return KVARN_OK;
}

kvarn_status kvarn_cache_create(const kvarn_config* cfg, void* dev_mem, size_t bytes, kvarn_cache** out) {
    kvarn_status st = check_config(cfg);
    if (st) return st;
    if (!out || !dev_mem || ((uintptr_t)dev_mem & 255)) return KVARN_EINVAL;
    kvarn_cache* c = new (std::nothrow) kvarn_cache();
    if (!c) return KVARN_ENOMEM;
    c->cfg = *cfg;
    c->lay = make_layout(*cfg, &c->slot_bytes, &c->max_groups);
    if (bytes < c->lay.total) { delete c; return KVARN_ENOMEM; }
    c->base = (uint8_t*)dev_mem;
    c->bytes = bytes;
    c->r = cfg->num_q_heads / cfg->num_kv_heads;
    c->rec_k = record_bytes(cfg->k_bits);
    c->rec_v = record_bytes(cfg->v_bits);
    c->tail_cap = kGroup * (cfg->tail_floor + 1);
    c->host_only = (cfg->flags & KVARN_FLAG_HOST_ONLY) != 0;
    c->test_stall = (cfg->flags & KVARN_FLAG_TEST_STALL) != 0;
    c->len.assign((size_t)cfg->max_seqs * cfg->num_layers, 0);
    c->table.assign((size_t)cfg->max_seqs * cfg->num_layers * c->max_groups, -1);
    c->free_slots.resize(cfg->pool_groups);
    for (int i = 0; i < cfg->pool_groups; ++i) c->free_slots[i] = cfg->pool_groups - 1 - i;  // pop gives 0,1,2..
    if (!c->host_only) {
        c->sms = sm_count();
        c->max_smem = max_optin_smem();
        if (pointer_device(dev_mem, &c->device)) c->device = -1;
        if (c->sms <= 0 || c->max_smem <= 0 || c->device < 0) {
            std::snprintf(g_last_error, sizeof(g_last_error), "no CUDA device");
            delete c;
            return KVARN_ECUDA;
        }
    }
    *out = c;
    return KVARN_OK;
}

void kvarn_cache_destroy(kvarn_cache* cache) { delete cache; }

kvarn_status kvarn_append(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                          const int32_t* n_tokens, const void* k, const void* v, void* stream) {
    kvarn_status st = check_ids(c, layer, n_seqs, seq_ids);
    if (st) return st;
    if (n_seqs > kMaxBatch) return KVARN_ECAPACITY;
    if (n_seqs > 0 && !n_tokens) return KVARN_EINVAL;
    int64_t total = 0, new_groups = 0;
    for (int i = 0; i < n_seqs; ++i) {
        if (n_tokens[i] < 0) return KVARN_EINVAL;
        int64_t n0 = c->Lc(seq_ids[i], layer), n1 = n0 + n_tokens[i];
        if (n1 > c->cfg.max_seq_len) return KVARN_ECAPACITY;
        total += n_tokens[i];
        new_groups += groups_sealed(n1, c->cfg.tail_floor) - groups_sealed(n0, c->cfg.tail_floor);
    }
    if (total > 0 && (!k || !v)) return KVARN_EINVAL;
    if (total >= (1ll << 31) / (c->cfg.num_kv_heads * 32)) return KVARN_ECAPACITY;
    if ((size_t)new_groups > c->free_slots.size()) return KVARN_ECAPACITY;
    if (total == 0) return KVARN_OK;
    const kvarn_config& cfg = c->cfg;
    static thread_local SealParams sp;
    static thread_local AppendParams ap;
    std::memset(&sp, 0, sizeof(sp));
    std::memset(&ap, 0, sizeof(ap));
    sp.base = ap.base = c->base;
    sp.lay = ap.lay = c->lay;
    sp.k_in = ap.k_in = (const uint16_t*)k;
    sp.v_in = ap.v_in = (const uint16_t*)v;
    sp.n_seqs = ap.n_seqs = n_seqs;
    sp.hkv = ap.hkv = cfg.num_kv_heads;
    sp.k_bits = cfg.k_bits;
    sp.v_bits = cfg.v_bits;
    sp.iters = cfg.sinkhorn_iters;
    sp.layer = ap.layer = layer;
    sp.num_layers = ap.num_layers = cfg.num_layers;
    sp.max_groups = c->max_groups;
    sp.rec_k = (int32_t)c->rec_k;
    sp.rec_v = (int32_t)c->rec_v;
    sp.slot_bytes = (int32_t)c->slot_bytes;
    sp.tail_cap = ap.tail_cap = c->tail_cap;
    int64_t jobs = 0, row = 0, toks = 0;
    for (int i = 0; i < n_seqs; ++i) {
        int s = seq_ids[i];
        int64_t n0 = c->Lc(s, layer), n1 = n0 + n_tokens[i];
        int64_t g0 = groups_sealed(n0, cfg.tail_floor), g1 = groups_sealed(n1, cfg.tail_floor);
        SealJobSeq& j = sp.seqs[i];
        j.seq = s;
        j.g_first = (int32_t)g0;
        j.n_new = (int32_t)(g1 - g0);
        j.n_before = (int32_t)n0;
        j.in_row = (int32_t)row;
        j.job_begin = (int32_t)jobs;
        jobs += (g1 - g0) * cfg.num_kv_heads * 2;
        AppendSeq& a = ap.seqs[i];
        a.seq = s;
        a.n_before = (int32_t)n0;
        a.n_new = n_tokens[i];
        a.keep_from = (int32_t)(kSink + g1 * kGroup);
        a.in_row = (int32_t)row;
        a.tok_begin = (int32_t)toks;
        row += n_tokens[i];
        toks += n_tokens[i];
    }
    if (jobs >= (1ll << 31)) return KVARN_ECAPACITY;
    sp.jobs_total = (int32_t)jobs;
    ap.tokens_total = (int32_t)toks;
    if (!c->host_only) {
        st = ensure_init(c, stream);
        if (st) return st;
    }
    // take slots and publish the new block-table entries
    for (int i = 0; i < n_seqs; ++i) {
        const SealJobSeq& j = sp.seqs[i];
        for (int g = 0; g < j.n_new; ++g) {
            c->T(j.seq, layer, j.g_first + g) = c->free_slots.back();
            c->free_slots.pop_back();
        }
        if (j.n_new && !c->host_only) {
            size_t off = c->lay.block_table +
                         (((size_t)j.seq * cfg.num_layers + layer) * c->max_groups + j.g_first) * 4;
            int rc = memcpy_h2d_async(c->base + off, &c->T(j.seq, layer, j.g_first), (size_t)j.n_new * 4, stream);
            if (rc) { set_cuda_error(rc, "block table copy"); return KVARN_ECUDA; }
        }
    }
    if (!c->host_only) {
        if (jobs > 0) {
            int rc = launch_seal_jobs(sp, stream);
            if (rc) { set_cuda_error(rc, "seal launch"); return KVARN_ECUDA; }
        }
        int rc = launch_append(ap, stream);
        if (rc) { set_cuda_error(rc, "append launch"); return KVARN_ECUDA; }
    }
    for (int i = 0; i < n_seqs; ++i) c->L(seq_ids[i], layer) += n_tokens[i];
    return KVARN_OK;
}

kvarn_status kvarn_decode_attention(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                                    const void* q, void* out, float softmax_scale, void* stream) {
    return run_decode(c, layer, n_seqs, seq_ids, nullptr, nullptr, q, out, softmax_scale, stream, false);
}

kvarn_status kvarn_prefill_attention(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                                     const int32_t* q_lens, const void* q, void* out, float softmax_scale,
                                     void* stream) {
    kvarn_status st = check_prefill(c, layer, n_seqs, seq_ids, q_lens, nullptr, q, out, softmax_scale);
    if (st) return st;
    return run_prefill(c, layer, n_seqs, seq_ids, q_lens, q, out, softmax_scale, stream);
}

kvarn_status kvarn_prefill(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                           const int32_t* n_tokens, const void* k, const void* v, const void* q, void* out,
                           float softmax_scale, void* stream) {
    kvarn_status st = check_prefill(c, layer, n_seqs, seq_ids, n_tokens, n_tokens, q, out, softmax_scale);
    if (st) return st;
    st = kvarn_append(c, layer, n_seqs, seq_ids, n_tokens, k, v, stream);
    if (st) return st;
    return run_prefill(c, layer, n_seqs, seq_ids, n_tokens, q, out, softmax_scale, stream);
}

kvarn_status kvarn_decode_step(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                               const void* k, const void* v, const void* q, void* out, float softmax_scale,
                               void* stream) {
    return run_decode(c, layer, n_seqs, seq_ids, k, v, q, out, softmax_scale, stream, true);
}

// Decode attention whose split-K scratch lives in the library's static device array
// (see kvarn_decode_attention_noalloc in kvarn.h). Nothing is allocated: the array is
// fetched per device, and every call gets an epoch of its own so that partials left by
// earlier calls are never merged.
kvarn_status kvarn_decode_attention_noalloc(kvarn_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                                            const void* q, void* out, float softmax_scale, void* stream) {
    if (!c) return KVARN_EINVAL;
    int max_blocks = static_workspace_blocks();
    if ((int64_t)c->cfg.max_seqs * c->cfg.num_kv_heads > max_blocks) {
        std::snprintf(g_last_error, sizeof(g_last_error),
                      "max_seqs * num_kv_heads = %lld exceeds the static workspace (%d blocks)",
                      (long long)c->cfg.max_seqs * c->cfg.num_kv_heads, max_blocks);
        return KVARN_ECAPACITY;
    }
    if (c->host_only) return KVARN_EINVAL;
    // the array used is the current device's: it must be the device that holds the cache
    int cur = -1;
    int rc = current_device(&cur);
    if (rc) { set_cuda_error(rc, "current device"); return KVARN_ECUDA; }
    if (cur != c->device) {
        std::snprintf(g_last_error, sizeof(g_last_error),
                      "the current device (%d) is not the cache's device (%d)", cur, c->device);
        return KVARN_EINVAL;
    }
    WorkspaceOverride ws{};
    rc = static_workspace(&ws.partials);
    if (rc) { set_cuda_error(rc, "static workspace address"); return KVARN_ECUDA; }
    kvarn_status st = check_ids(c, layer, n_seqs, seq_ids);
    if (st) return st;
    static std::atomic<uint32_t> epochs{0x80000000u};
    ws.epoch = epochs.fetch_add(1) + 1;
    return run_decode(c, layer, n_seqs, seq_ids, nullptr, nullptr, q, out, softmax_scale, stream, false, &ws);
}

kvarn_status kvarn_group_record(const kvarn_cache* c, int32_t layer, int32_t seq_id, int32_t group,
                                int32_t kv_head, int32_t which, const void** dev_ptr, size_t* bytes) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers || seq_id < 0 || seq_id >= c->cfg.max_seqs) return KVARN_EINVAL;
    if (kv_head < 0 || kv_head >= c->cfg.num_kv_heads || (which != 0 && which != 1) || group < 0) return KVARN_EINVAL;
    if (group >= groups_sealed(c->Lc(seq_id, layer), c->cfg.tail_floor)) return KVARN_ESTATE;
    int32_t slot = c->Tc(seq_id, layer, group);
    if (slot < 0) return KVARN_ESTATE;
    size_t off = c->lay.pool + (size_t)slot * c->slot_bytes + (size_t)kv_head * (c->rec_k + c->rec_v) +
                 (which ? c->rec_k : 0);
    if (dev_ptr) *dev_ptr = c->base + off;
    if (bytes) *bytes = which ? c->rec_v : c->rec_k;
    return KVARN_OK;
}

kvarn_status kvarn_exact_regions(const kvarn_cache* c, int32_t layer, int32_t seq_id, const void** sink_k,
                                 const void** sink_v, const void** tail_k, const void** tail_v) {
    if (!c || layer < 0 || layer >= c->cfg.num_layers || seq_id < 0 || seq_id >= c->cfg.max_seqs) return KVARN_EINVAL;
    size_t per = (size_t)c->cfg.num_kv_heads * kSink * kHeadDim * 2;
    size_t off = ((size_t)seq_id * c->cfg.num_layers + layer) * per;
    size_t toff = off * (size_t)(c->cfg.tail_floor + 1);  // the tail ring is F + 1 groups long
    if (sink_k) *sink_k = c->base + c->lay.sink_k + off;
    if (sink_v) *sink_v = c->base + c->lay.sink_v + off;
    if (tail_k) *tail_k = c->base + c->lay.tail_k + toff;
    if (tail_v) *tail_v = c->base + c->lay.tail_v + toff;
    return KVARN_OK;
}

kvarn_status kvarn_dequant_group(kvarn_cache* c, int32_t layer, int32_t seq_id, int32_t group, int32_t kv_head,
                                 int32_t which, int32_t frame, int32_t out_fp32, void* out, void* stream) {
    const void* rec = nullptr;
    kvarn_status st = kvarn_group_record(c, layer, seq_id, group, kv_head, which, &rec, nullptr);
    if (st) return st;
    if (!out || (frame != 0 && frame != 1)) return KVARN_EINVAL;
    if (c->host_only) return KVARN_OK;
    st = ensure_init(c, stream);
    if (st) return st;
    int rc = launch_dequant((const uint8_t*)rec, which ? c->cfg.v_bits : c->cfg.k_bits, which, frame, out_fp32 != 0,
                            out, stream);
    if (rc) { set_cuda_error(rc, "dequant launch"); return KVARN_ECUDA; }
    return KVARN_OK;
}

kvarn_status kvarn_snapshot_bytes(const kvarn_cache* c, size_t* bytes) {
    if (!c || !bytes) return KVARN_EINVAL;
    *bytes = snap_sizes(c, used_slots(c).size()).total;
    return KVARN_OK;
}

kvarn_status kvarn_snapshot_save(kvarn_cache* c, void* dst, size_t bytes, void* stream) {
    if (!c || !dst) return KVARN_EINVAL;
    const std::vector<int32_t> used = used_slots(c);
    if (!used.empty() && (used.front() < 0 || used.back() >= c->cfg.pool_groups)) return KVARN_ESTATE;
    const SnapSizes z = snap_sizes(c, used.size());
    if (bytes < z.total) return KVARN_EINVAL;
    uint8_t* o = (uint8_t*)dst;
    SnapHeader h;
    std::memset(&h, 0, sizeof(h));
    std::memcpy(h.magic, kSnapMagic, sizeof(h.magic));
    h.version = kSnapVersion;
    h.header_bytes = (uint32_t)sizeof(SnapHeader);
    h.cfg = c->cfg;
    h.max_groups = c->max_groups;
    h.slot_bytes = c->slot_bytes;
    h.sink_bytes = z.sink_bytes;
    h.tail_bytes = z.tail_bytes;
    h.n_used = used.size();
    h.total_bytes = z.total;
    std::memcpy(o, &h, sizeof(h));
    size_t off = sizeof(h);
    std::memcpy(o + off, c->len.data(), z.len_bytes);
    off += z.len_bytes;
    std::memcpy(o + off, c->table.data(), z.table_bytes);
    off += z.table_bytes;
    if (c->host_only) {
        std::memset(o + off, 0, z.total - off);
        return KVARN_OK;
    }
    kvarn_status st = ensure_init(c, stream);
    if (st) return st;
    const size_t regions[4] = {c->lay.sink_k, c->lay.sink_v, c->lay.tail_k, c->lay.tail_v};
    const size_t sizes[4] = {z.sink_bytes, z.sink_bytes, z.tail_bytes, z.tail_bytes};
    for (int i = 0; i < 4; ++i) {
        int rc = memcpy_d2h_async(o + off, c->base + regions[i], sizes[i], stream);
        if (rc) { set_cuda_error(rc, "snapshot copy"); return KVARN_ECUDA; }
        off += sizes[i];
    }
    // used slots, runs of consecutive slots in one copy each
    for (size_t i = 0; i < used.size();) {
        size_t j = i + 1;
        while (j < used.size() && used[j] == used[j - 1] + 1) ++j;
        const size_t n = (j - i) * c->slot_bytes;
        int rc = memcpy_d2h_async(o + off, c->base + c->lay.pool + (size_t)used[i] * c->slot_bytes, n, stream);
        if (rc) { set_cuda_error(rc, "snapshot copy"); return KVARN_ECUDA; }
        off += n;
        i = j;
    }
    int rc = stream_sync(stream);
    if (rc) { set_cuda_error(rc, "snapshot copy"); return KVARN_ECUDA; }
    return KVARN_OK;
}

kvarn_status kvarn_snapshot_load(kvarn_cache* c, const void* src, size_t bytes, void* stream) {
    if (!c || !src || bytes < sizeof(SnapHeader)) return KVARN_EINVAL;
    const uint8_t* in = (const uint8_t*)src;
    SnapHeader h;
    std::memcpy(&h, in, sizeof(h));
    if (std::memcmp(h.magic, kSnapMagic, sizeof(h.magic)) || h.version != kSnapVersion ||
        h.header_bytes != sizeof(SnapHeader) || !same_config(h.cfg, c->cfg) || h.max_groups != c->max_groups ||
        h.slot_bytes != c->slot_bytes)
        return KVARN_EINVAL;
    if (h.n_used > (uint64_t)c->cfg.pool_groups) return KVARN_EINVAL;
    const SnapSizes z = snap_sizes(c, h.n_used);
    if (h.sink_bytes != z.sink_bytes || h.tail_bytes != z.tail_bytes || h.total_bytes != z.total || bytes < z.total)
        return KVARN_EINVAL;
    // the bookkeeping, checked in full before anything changes
    std::vector<int64_t> len(z.seq_layers);
    std::vector<int32_t> table(z.table_bytes / sizeof(int32_t));
    size_t off = sizeof(h);
    std::memcpy(len.data(), in + off, z.len_bytes);
    off += z.len_bytes;
    std::memcpy(table.data(), in + off, z.table_bytes);
    off += z.table_bytes;
    std::vector<char> seen(c->cfg.pool_groups, 0);
    std::vector<int32_t> used;
    for (size_t sl = 0; sl < z.seq_layers; ++sl) {
        if (len[sl] < 0 || len[sl] > c->cfg.max_seq_len) return KVARN_EINVAL;
        const int64_t ng = groups_sealed(len[sl], c->cfg.tail_floor);
        for (int g = 0; g < c->max_groups; ++g) {
            const int32_t v = table[sl * c->max_groups + g];
            if (g < ng) {
                if (v < 0 || v >= c->cfg.pool_groups || seen[v]) return KVARN_EINVAL;
                seen[v] = 1;
                used.push_back(v);
            } else if (v != -1) {
                return KVARN_EINVAL;
            }
        }
    }
    if (used.size() != h.n_used) return KVARN_EINVAL;
    std::sort(used.begin(), used.end());
    if (!c->host_only) {
        kvarn_status st = ensure_init(c, stream);
        if (st) return st;
        const size_t regions[4] = {c->lay.sink_k, c->lay.sink_v, c->lay.tail_k, c->lay.tail_v};
        const size_t sizes[4] = {z.sink_bytes, z.sink_bytes, z.tail_bytes, z.tail_bytes};
        size_t doff = off;
        for (int i = 0; i < 4; ++i) {
            int rc = memcpy_h2d_async(c->base + regions[i], in + doff, sizes[i], stream);
            if (rc) { set_cuda_error(rc, "snapshot copy"); return KVARN_ECUDA; }
            doff += sizes[i];
        }
        for (size_t i = 0; i < used.size();) {
            size_t j = i + 1;
            while (j < used.size() && used[j] == used[j - 1] + 1) ++j;
            const size_t n = (j - i) * c->slot_bytes;
            int rc = memcpy_h2d_async(c->base + c->lay.pool + (size_t)used[i] * c->slot_bytes, in + doff, n, stream);
            if (rc) { set_cuda_error(rc, "snapshot copy"); return KVARN_ECUDA; }
            doff += n;
            i = j;
        }
        int rc = memcpy_h2d_async(c->base + c->lay.block_table, table.data(), z.table_bytes, stream);
        if (rc == 0) rc = stream_sync(stream);  // `table` and the caller's image stay valid until here
        if (rc) { set_cuda_error(rc, "snapshot copy"); return KVARN_ECUDA; }
    }
    c->len = std::move(len);
    c->table = std::move(table);
    // free slots in the order a fresh cache hands them out (lowest first)
    c->free_slots.clear();
    for (int i = c->cfg.pool_groups - 1; i >= 0; --i)
        if (!seen[i]) c->free_slots.push_back(i);
    return KVARN_OK;
}

kvarn_status kvarn_seq_release(kvarn_cache* c, int32_t seq_id) {
    if (!c || seq_id < 0 || seq_id >= c->cfg.max_seqs) return KVARN_EINVAL;
    for (int l = 0; l < c->cfg.num_layers; ++l) {
        int64_t ng = groups_sealed(c->L(seq_id, l), c->cfg.tail_floor);
        for (int64_t g = 0; g < ng; ++g) {
            int32_t& s = c->T(seq_id, l, (int)g);
            if (s >= 0) c->free_slots.push_back(s);
            s = -1;
        }
        c->L(seq_id, l) = 0;
    }
    return KVARN_OK;
}

kvarn_status kvarn_seq_length(const kvarn_cache* c, int32_t layer, int32_t seq_id, int64_t* len) {
    if (!c || !len || layer < 0 || layer >= c->cfg.num_layers || seq_id < 0 || seq_id >= c->cfg.max_seqs)
        return KVARN_EINVAL;
    *len = c->Lc(seq_id, layer);
    return KVARN_OK;
}

kvarn_status kvarn_cache_stats(const kvarn_cache* c, kvarn_stats* o) {
    if (!c || !o) return KVARN_EINVAL;
    std::memset(o, 0, sizeof(*o));
    const kvarn_config& cfg = c->cfg;
    o->device_bytes = c->lay.total;
    o->record_bytes_k = c->rec_k;
    o->record_bytes_v = c->rec_v;
    o->slot_bytes = c->slot_bytes;
    o->pool_slots_total = cfg.pool_groups;
    o->pool_slots_used = cfg.pool_groups - c->free_slots.size();
    for (int s = 0; s < cfg.max_seqs; ++s)
        for (int l = 0; l < cfg.num_layers; ++l) {
            int64_t n = c->Lc(s, l);
            o->tokens_cached += n;
            o->sealed_tokens += groups_sealed(n, cfg.tail_floor) * kGroup;
        }
    o->exact_tokens = o->tokens_cached - o->sealed_tokens;
    double elems_per_token = (double)cfg.num_kv_heads * kHeadDim;  // per side
    o->sealed_bytes = (o->sealed_tokens / kGroup) * (uint64_t)cfg.num_kv_heads * (c->rec_k + c->rec_v);
    o->exact_bytes = o->exact_tokens * (uint64_t)cfg.num_kv_heads * kHeadDim * 2 * 2;
    o->body_bits_per_element = (double)(c->rec_k + c->rec_v) * 8.0 / (2.0 * kGroup * kHeadDim);
    o->all_in_bits_per_element =
        o->tokens_cached ? (double)(o->sealed_bytes + o->exact_bytes) * 8.0 / (o->tokens_cached * elems_per_token * 2)
                         : 0.0;
    return KVARN_OK;
}

kvarn_status kvarn_seal_groups(const void* x, int32_t n, int32_t bits, int32_t which, int32_t iters, void* records,
                               float* scales, void* stream) {
    if (n < 0 || !bits_ok(bits) || (which != 0 && which != 1) || iters < 0 || iters > 64) return KVARN_EINVAL;
    if (n == 0) return KVARN_OK;
    if (!x || !records || ((uintptr_t)x & 15) || ((uintptr_t)records & 15)) return KVARN_EINVAL;
    int rc = launch_seal_groups(x, n, bits, which, iters, records, scales, stream);
    if (rc) { set_cuda_error(rc, "seal launch"); return KVARN_ECUDA; }
    return KVARN_OK;
}

kvarn_status kvarn_check_device_error(kvarn_cache* c, void* stream) {
    if (!c) return KVARN_EINVAL;
    if (c->host_only || !c->initialized) return KVARN_OK;
    int32_t err[4] = {0, 0, 0, 0};
    int rc = memcpy_d2h_sync(err, c->base + c->lay.err, sizeof(err), stream);
    if (rc) { set_cuda_error(rc, "error word read"); return KVARN_ECUDA; }
    int32_t zero[4] = {0, 0, 0, 0};
    rc = memcpy_h2d_async(c->base + c->lay.err, zero, sizeof(zero), stream);
    if (rc) { set_cuda_error(rc, "error word clear"); return KVARN_ECUDA; }
    if (err[0] & kErrTimeout) return KVARN_ETIMEOUT;
    if (err[0]) return KVARN_ESTATE;
    return KVARN_OK;
}

const char* kvarn_status_string(kvarn_status s) {
    switch (s) {
        case KVARN_OK: return "ok";
        case KVARN_EINVAL: return "invalid argument";
        case KVARN_ENOMEM: return "device block too small";
        case KVARN_ECAPACITY: return "capacity exceeded";
        case KVARN_ECUDA: return "CUDA error";
        case KVARN_ESTATE: return "invalid state";
        case KVARN_ETIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char* kvarn_last_error(void) { return g_last_error; }

}  // extern "C"
