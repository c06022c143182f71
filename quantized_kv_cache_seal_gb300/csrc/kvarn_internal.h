// Internal declarations shared by the host side (kvarn_host.cpp) and the kernels.
// Plain structs passed by value as kernel parameters; no CUDA types in here so that
// the host file compiles with the host compiler alone.
#pragma once
#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define KVARN_HD __host__ __device__
#else
#define KVARN_HD
#endif

namespace kvarn {

constexpr int kHeadDim = 128;
constexpr int kGroup = 128;
constexpr int kSink = 128;
constexpr int kMaxBatch = 256;   // sequences per decode call (kernel parameter table size)
constexpr int kMaxSpan = 32;     // CTAs that may share the sealed groups of one (seq, kv head)
constexpr int kMaxGrid = 256;    // CTAs of a decode launch (at most one per SM)
constexpr int kPartialSlots = kMaxSpan;  // one partial per CTA covering a block
constexpr int kPartialFloats = 528;  // [0] epoch bits, [4..8) m, [8..12) l, [12..524) acc
constexpr int kDecodeThreads = 512;  // 3 compute warpgroups + 1 copy-issuing warpgroup
constexpr int kExactRows = 16;       // tokens of an exact (sink or tail) sub-group of the decode stream
constexpr int kSealThreads = 256;
constexpr int kPrefillRows = 128;     // query rows (token, head) of a prefill CTA

// device error word bits
constexpr int kErrTimeout = 1;
constexpr int kErrBadSlot = 2;
constexpr int kErrSpan = 4;
constexpr int kErrStalePartial = 8;  // a partial the merge needed carried another call's epoch

KVARN_HD inline size_t record_bytes(int bits) { return 528 + 2048 * (size_t)bits; }

// 16-token sub-groups of the exact part (sink then tail) of one (sequence, KV head).
KVARN_HD inline int exact_subs(int n_sink, int n_tail) {
    return (n_sink + kExactRows - 1) / kExactRows + (n_tail + kExactRows - 1) / kExactRows;
}

// Device memory layout of one cache (byte offsets into the caller's block).
struct Layout {
    size_t err;          // int32[4]
    size_t block_table;  // int32[max_seqs][num_layers][max_groups]
    size_t sink_k, sink_v, tail_k, tail_v;  // fp16[max_seqs][num_layers][Hkv][128][128]
    size_t partials;     // float[max_seqs][Hkv][kPartialSlots][kPartialFloats]
    size_t pool;         // slots * slot_bytes
    size_t total;
};

// One sequence of a decode call.
struct SeqEntry {
    int32_t seq;         // sequence id (index into the per-sequence buffers)
    int32_t n_groups;    // sealed groups read from records (excludes one sealed in this call)
    int32_t n_sink;      // exact sink tokens (after this call's append)
    int32_t n_tail;      // exact tail tokens (after this call's append)
    int32_t new_pos;     // position of the token appended by this call, -1 if none
    int32_t seal_group;  // group completed by the new token, -1 if none
    int32_t seal_slot;   // pool slot taken for it
    int32_t unit_begin;  // first scheduling unit of this sequence
    int32_t w_exact;     // units charged for the exact item of each (seq, kv head)
    int32_t w_seal;      // units charged for the seal item (0 if none)
    int32_t tail_first;  // tail ring slot of the first exact tail token
};

// Parameters of the decode kernel (append + seal + attention).
struct DecodeParams {
    uint8_t* base;              // cache device block
    Layout lay;
    float* partials;            // split-K partial states: the cache's own region or the static workspace
    const uint16_t* q;          // [n][Hq][128]
    uint16_t* out;              // [n][Hq][128]
    const uint16_t* k_new;      // [n][Hkv][128] or null
    const uint16_t* v_new;
    int32_t n_seqs, hq, hkv, r, k_bits, v_bits, iters, layer, num_layers, max_seqs, max_groups;
    int32_t rec_k, rec_v, slot_bytes, pool_slots;
    int32_t stages;             // smem ring stages
    int32_t grid;               // CTAs
    int64_t units_total;
    int32_t cta_begin[kMaxGrid + 1];  // first scheduling unit of each CTA; [grid] = units_total
    uint32_t epoch;
    int32_t test_stall;         // KVARN_FLAG_TEST_STALL: one bounded wait that runs out
    int32_t tail_cap;           // rows of the tail ring per (sequence, layer, KV head)
    float scale_log2;           // softmax_scale * log2(e)
    SeqEntry seqs[kMaxBatch];
};

// One sequence of a prefill-attention call: its queries are those of the last q_len
// tokens (positions n - q_len .. n - 1), rows q_row .. q_row + q_len - 1 of q and out.
struct PrefillSeq {
    int32_t seq;
    int32_t n;          // tokens in the cache
    int32_t q_len;
    int32_t q_row;
    int32_t n_groups;   // sealed groups of the sequence
    int32_t n_tiles;    // query tiles (kPrefillRows / r tokens each)
    int32_t cta_begin;  // first CTA of this sequence ((n_tiles + 1) / 2 * 2 * Hkv CTAs: tile pairs)
};

struct PrefillParams {
    uint8_t* base;
    Layout lay;
    const uint16_t* q;  // [rows][Hq][128]
    uint16_t* out;
    int32_t n_seqs, hq, hkv, r, k_bits, v_bits, layer, num_layers, max_groups;
    int32_t rec_k, rec_v, slot_bytes, tail_cap;
    int32_t grid;       // CTAs: one per (sequence, KV head, query tile), tiles padded to pairs
    float scale_log2;
    PrefillSeq seqs[kMaxBatch];
};

// Parameters of the bulk seal for kvarn_append.
struct SealJobSeq {
    int32_t seq;
    int32_t g_first;     // first group sealed by this call
    int32_t n_new;       // groups sealed by this call
    int32_t n_before;    // length before the call
    int32_t in_row;      // first input token row of this sequence
    int32_t job_begin;   // prefix over sequences of n_new * Hkv * 2
};

struct SealParams {
    uint8_t* base;
    Layout lay;
    const uint16_t* k_in;
    const uint16_t* v_in;
    int32_t n_seqs, hkv, k_bits, v_bits, iters, layer, num_layers, max_groups;
    int32_t rec_k, rec_v, slot_bytes;
    int32_t jobs_total;
    int32_t tail_cap;
    SealJobSeq seqs[kMaxBatch];
};

struct AppendSeq {
    int32_t seq;
    int32_t n_before;
    int32_t n_new;
    int32_t keep_from;   // first body position that stays in the tail after the call
    int32_t in_row;
    int32_t tok_begin;   // prefix over sequences of n_new
};

struct AppendParams {
    uint8_t* base;
    Layout lay;
    const uint16_t* k_in;
    const uint16_t* v_in;
    int32_t n_seqs, hkv, layer, num_layers, tokens_total;
    int32_t tail_cap;
    AppendSeq seqs[kMaxBatch];
};

// Launchers (defined in the .cu files). Return 0 on success, else a cudaError_t value.
int launch_decode(const DecodeParams& p, int smem_bytes, void* stream);
int launch_prefill(const PrefillParams& p, void* stream);
int prefill_smem_bytes();
int launch_seal_jobs(const SealParams& p, void* stream);
int launch_append(const AppendParams& p, void* stream);
int launch_seal_groups(const void* x, int n, int bits, int which, int iters, void* records, float* scales,
                       void* stream);
int launch_dequant(const uint8_t* rec, int bits, int which, int frame, int out_fp32, void* out, void* stream);
int launch_init(uint8_t* base, const Layout& lay, void* stream);
int decode_smem_bytes(int k_bits, int v_bits, int stages, bool with_seal);
int max_optin_smem();
int sm_count();
const char* cuda_error_string(int code);
int pointer_device_accessible(const void* ptr, int* accessible);  // 0 or a cudaError_t value
int current_device(int* device);                        // 0 or a cudaError_t value
int pointer_device(const void* ptr, int* device);       // device holding ptr (else the current one)
int memcpy_h2d_async(void* dst, const void* src, size_t bytes, void* stream);
int memcpy_d2h_sync(void* dst, const void* src, size_t bytes, void* stream);
// static split-K workspace for the allocation-free decode call (kvarn_decode.cu)
int static_workspace_blocks();
int static_workspace(void** partials);

}  // namespace kvarn
