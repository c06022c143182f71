// KVarN seal, append and dequantisation kernels (sm_103a).
//
//  - seal_groups_kernel: seal independent 128 x 128 fp16 matrices (bulk sealing,
//    parity checks).
//  - seal_jobs_kernel: seal the groups an append call completes, reading each token
//    row from the tail buffer (tokens cached before the call) or from the input.
//  - append_kernel: copy new tokens into the exact regions (sink, tail) of the
//    cache (anbeeld.com "KVarN KV Cache: Implementation and Benchmarks", 2.1).
//  - dequant_kernel: the "convert to a standard cache layout" path (same section):
//    yhat_ij = a_i c_j (m + delta q_ij), optionally rotated back by H.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvarn_dev.cuh"

namespace kvarn {

namespace {

struct PtrRows {
    const uint16_t* base;  // row i at base + 128 i
    __device__ const uint16_t* operator()(int i) const { return base + 128 * i; }
};

// Two CTAs per SM (at most 128 registers a thread; 73 KB of shared memory each): a
// prompt's few hundred group matrices then take two rounds of the GPU instead of four.
__global__ void __launch_bounds__(256, 2) seal_groups_kernel(const uint16_t* x, int bits, int which, int iters,
                                                          uint8_t* records, float* scales) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SealSmem& S = *reinterpret_cast<SealSmem*>(smem_raw);
    const size_t g = blockIdx.x;
    PtrRows rows{x + g * 128 * 128};
    seal_matrix(rows, bits, which, iters, records + g * record_bytes(bits), scales ? scales + g * 256 : nullptr, S,
                1);
}

struct JobRows {
    const uint16_t* tail;  // tail ring of (seq, layer, kv head)
    const uint16_t* in;    // input row of position n_before, this kv head
    int first_pos;         // position of row 0 of the group
    int n_before;
    int hkv;
    int cap;               // rows of the tail ring
    __device__ const uint16_t* operator()(int i) const {
        int p = first_pos + i;
        if (p < n_before) return tail + 128 * ((p - kSink) % cap);
        return in + (size_t)(p - n_before) * hkv * 128;
    }
};

__global__ void __launch_bounds__(256, 2) seal_jobs_kernel(const __grid_constant__ SealParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SealSmem& S = *reinterpret_cast<SealSmem*>(smem_raw);
    const int job = blockIdx.x;
    int lo = 0, hi = p.n_seqs - 1;
    while (lo < hi) {  // last sequence with job_begin <= job
        int mid = (lo + hi + 1) >> 1;
        if (p.seqs[mid].job_begin <= job) lo = mid; else hi = mid - 1;
    }
    const SealJobSeq& e = p.seqs[lo];
    int local = job - e.job_begin;
    const int side = local & 1;
    local >>= 1;
    const int kvh = local % p.hkv;
    const int g = e.g_first + local / p.hkv;
    const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
    const int32_t* table = reinterpret_cast<const int32_t*>(p.base + p.lay.block_table);
    const int slot = table[sl * p.max_groups + g];
    uint8_t* rec = p.base + p.lay.pool + (size_t)slot * p.slot_bytes + (size_t)kvh * (p.rec_k + p.rec_v) +
                   (side ? p.rec_k : 0);
    const uint16_t* tail = reinterpret_cast<const uint16_t*>(p.base + (side ? p.lay.tail_v : p.lay.tail_k)) +
                           (sl * p.hkv + kvh) * (size_t)p.tail_cap * 128;
    const uint16_t* in = (side ? p.v_in : p.k_in) + ((size_t)e.in_row * p.hkv + kvh) * 128;
    JobRows rows{tail, in, kSink + kGroup * g, e.n_before, p.hkv, p.tail_cap};
    seal_matrix(rows, side ? p.v_bits : p.k_bits, side, p.iters, rec, nullptr, S, 1);
}

// One thread per 16-byte chunk of a (token, kv head, side) row.
__global__ void append_kernel(const __grid_constant__ AppendParams p) {
    const int64_t total = (int64_t)p.tokens_total * p.hkv * 2 * 16;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int chunk = (int)(idx & 15);
        int64_t rest = idx >> 4;
        const int side = (int)(rest & 1);
        rest >>= 1;
        const int kvh = (int)(rest % p.hkv);
        const int tok = (int)(rest / p.hkv);
        int lo = 0, hi = p.n_seqs - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (p.seqs[mid].tok_begin <= tok) lo = mid; else hi = mid - 1;
        }
        const AppendSeq& e = p.seqs[lo];
        const int k = tok - e.tok_begin;
        const int pos = e.n_before + k;
        const size_t sl = (size_t)e.seq * p.num_layers + p.layer;
        size_t dst_off;
        if (pos < kSink) {
            dst_off = (side ? p.lay.sink_v : p.lay.sink_k) + ((sl * p.hkv + kvh) * 128 + pos) * 256;
        } else if (pos >= e.keep_from) {
            dst_off = (side ? p.lay.tail_v : p.lay.tail_k) +
                      ((sl * p.hkv + kvh) * (size_t)p.tail_cap + (pos - kSink) % p.tail_cap) * 256;
        } else {
            continue;  // sealed by this call
        }
        const uint16_t* src = (side ? p.v_in : p.k_in) + ((size_t)(e.in_row + k) * p.hkv + kvh) * 128;
        reinterpret_cast<uint4*>(p.base + dst_off)[chunk] = reinterpret_cast<const uint4*>(src)[chunk];
    }
}

template <int B>
__device__ __forceinline__ int code_at(const uint8_t* codes, int e) {
    // code e of the stream: bits e B .. e B + B - 1, least significant first
    const uint32_t* w = reinterpret_cast<const uint32_t*>(codes);
    const int bit = e * B, word = bit / 32, s = bit % 32;
    uint32_t v = w[word] >> s;
    if (s + B > 32) v |= w[word + 1] << (32 - s);
    return (int)(v & ((1u << B) - 1));
}

__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* rec, int bits, int which, int frame, int out_fp32,
                                                      void* out) {
    const int t = threadIdx.x, i = t >> 1, h = t & 1;
    const float delta = __uint_as_float(reinterpret_cast<const uint32_t*>(rec)[0]);
    const float m = __uint_as_float(reinterpret_cast<const uint32_t*>(rec)[1]);
    const uint16_t* r16 = reinterpret_cast<const uint16_t*>(rec);
    const float ai = half_bits_to_float(r16[8 + i]);
    const uint8_t* codes = rec + 528;
    float x[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        const int j = 64 * h + k;
        const int e = which == 0 ? i * 128 + j : j * 128 + i;
        int q;
        switch (bits) {
            case 2: q = code_at<2>(codes, e); break;
            case 3: q = code_at<3>(codes, e); break;
            case 4: q = code_at<4>(codes, e); break;
            case 5: q = code_at<5>(codes, e); break;
            case 6: q = code_at<6>(codes, e); break;
            default: q = code_at<8>(codes, e); break;
        }
        x[k] = ai * half_bits_to_float(r16[8 + 128 + j]) * fmaf(delta, (float)q, m);
    }
    if (frame == 0) {
#pragma unroll
        for (int len = 1; len < 64; len <<= 1) {
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                if (!(k & len)) {
                    float a = x[k], b = x[k + len];
                    x[k] = a + b;
                    x[k + len] = a - b;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 64; ++k) {
            float o = __shfl_xor_sync(0xffffffffu, x[k], 1);
            x[k] = (h ? (o - x[k]) : (x[k] + o)) * kInvSqrt128;
        }
    }
    if (out_fp32) {
        float* o = reinterpret_cast<float*>(out) + 128 * i + 64 * h;
#pragma unroll
        for (int k = 0; k < 64; ++k) o[k] = x[k];
    } else {
        __half* o = reinterpret_cast<__half*>(out) + 128 * i + 64 * h;
#pragma unroll
        for (int k = 0; k < 64; ++k) o[k] = __float2half_rn(x[k]);
    }
}

bool g_seal_attr_set = false;

int set_seal_attr() {
    if (g_seal_attr_set) return 0;
    cudaError_t e = cudaFuncSetAttribute(seal_groups_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(SealSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(seal_jobs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SealSmem));
    if (e == cudaSuccess) g_seal_attr_set = true;
    return (int)e;
}

}  // namespace

int launch_seal_groups(const void* x, int n, int bits, int which, int iters, void* records, float* scales,
                       void* stream) {
    int rc = set_seal_attr();
    if (rc) return rc;
    seal_groups_kernel<<<n, 256, sizeof(SealSmem), (cudaStream_t)stream>>>(
        (const uint16_t*)x, bits, which, iters, (uint8_t*)records, scales);
    return (int)cudaGetLastError();
}

int launch_seal_jobs(const SealParams& p, void* stream) {
    int rc = set_seal_attr();
    if (rc) return rc;
    seal_jobs_kernel<<<p.jobs_total, 256, sizeof(SealSmem), (cudaStream_t)stream>>>(p);
    return (int)cudaGetLastError();
}

int launch_append(const AppendParams& p, void* stream) {
    int64_t total = (int64_t)p.tokens_total * p.hkv * 2 * 16;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    append_kernel<<<(int)blocks, 256, 0, (cudaStream_t)stream>>>(p);
    return (int)cudaGetLastError();
}

int launch_dequant(const uint8_t* rec, int bits, int which, int frame, int out_fp32, void* out, void* stream) {
    dequant_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(rec, bits, which, frame, out_fp32, out);
    return (int)cudaGetLastError();
}

int launch_init(uint8_t* base, const Layout& lay, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(base + lay.err, 0, lay.block_table - lay.err, s);  // error word
    if (e == cudaSuccess) e = cudaMemsetAsync(base + lay.block_table, 0xff, lay.sink_k - lay.block_table, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + lay.partials, 0, lay.pool - lay.partials, s);
    return (int)e;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

int max_optin_smem() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
    return n;
}

const char* cuda_error_string(int code) { return cudaGetErrorString((cudaError_t)code); }

int current_device(int* device) { return (int)cudaGetDevice(device); }

int pointer_device(const void* ptr, int* device) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess || a.type != cudaMemoryTypeDevice) {
        cudaGetLastError();  // not a device allocation this runtime knows: take the current device
        return (int)cudaGetDevice(device);
    }
    *device = a.device;
    return 0;
}

int pointer_device_accessible(const void* ptr, int* accessible) {
    *accessible = 0;
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is an answer, not a sticky error
        return 0;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) *accessible = 1;
    // pinned host memory that kernels reach at the same address (unified addressing)
    if (a.type == cudaMemoryTypeHost && a.devicePointer == ptr) *accessible = 1;
    return 0;
}

int memcpy_h2d_async(void* dst, const void* src, size_t bytes, void* stream) {
    return (int)cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
}

int memcpy_d2h_async(void* dst, const void* src, size_t bytes, void* stream) {
    return (int)cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
}

int stream_sync(void* stream) { return (int)cudaStreamSynchronize((cudaStream_t)stream); }

int memcpy_d2h_sync(void* dst, const void* src, size_t bytes, void* stream) {
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return (int)e;
}

}  // namespace kvarn
