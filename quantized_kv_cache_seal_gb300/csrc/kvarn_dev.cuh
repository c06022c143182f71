// Device helpers and the KVarN group seal, shared by the kernels of this library.
//
// The seal follows fig1.dev "KVarN: Variance-Normalized KV-Cache Quantization ...",
// "What it is", and anbeeld.com "KVarN KV Cache: Implementation and Benchmarks",
// sections 1 and 2.1: rotate each token row of a 128 x 128 group by the Hadamard
// matrix, run 16 Sinkhorn iterations that rescale the token axis and then the
// channel axis to unit mean square, store the scales, round to nearest on one
// min/max grid and pack the codes next to the scale metadata.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvarn_internal.h"

namespace kvarn {

constexpr float kInvSqrt128 = 0.08838834764831845f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a bounded wait gives up after 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; give up after kWaitLimitNs,
// record kErrTimeout in the error word and return false.
// A wait that starts after any wait of the launch has given up returns at once, so a
// failure ends the kernel within one time limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int32_t*>(err) & kErrTimeout) return false;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// One-dimensional bulk copy global -> shared, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (through L2, not L1).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Make mbarrier `bar` track the completion of the calling thread's earlier cp.async
// copies: the barrier's current phase does not complete before they have landed (its
// expected arrival count is unchanged).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Arrive at named barrier id (n threads in all) without waiting for it.
__device__ __forceinline__ void bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint16_t f16_bits_sat(float x) {
    // round to nearest even; values beyond the largest finite half saturate
    return __half_as_ushort(__float2half_rn(fminf(x, 65504.0f)));
}

__device__ __forceinline__ float half_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// ---------------------------------------------------------------------------
// Seal of one 128 x 128 group matrix by 256 threads.
// ---------------------------------------------------------------------------
struct SealSmem {
    float Y[128 * 136];   // rotated group: row i at 136 i, channel j at j + 4 (j >= 64)
    float u[136];         // 1 / c^2, same padding as a row
    float v[136];         // 1 / a^2
    float ra[128];        // 1 / a16
    float rc[128];        // 1 / c16
    float red[2][8];
    uint16_t a16[128];
    uint16_t c16[128];
};

__device__ __forceinline__ int ypad(int j) { return j + ((j >> 6) << 2); }

// Bounds on the squared Sinkhorn scales kept in fp32. Rows of fp16 data have squared
// scales far inside them; only inputs on which the alternating normalisation diverges
// (every row with a single non-zero rotated entry) reach them, and there the stored
// fp16 scales saturate or flush either way. With A = Y^2 < 2^40, A / bound stays finite.
constexpr float kSqMax = 1.2089258196146292e24f;   // 2^80
constexpr float kSqMin = 8.271806125530277e-25f;   // 2^-80

template <int B>
__device__ __forceinline__ void pack64_store(const int (&q)[64], uint8_t* dst) {
    // 64 codes of B bits into 2B little-endian words: code e at bits e B .. e B + B - 1
    // of the stream, least significant first (a code may straddle two words)
    uint32_t w[2 * B];
#pragma unroll
    for (int k = 0; k < 2 * B; ++k) w[k] = 0;
#pragma unroll
    for (int e = 0; e < 64; ++e) {
        const int bit = e * B, word = bit / 32, s = bit % 32;
        w[word] |= (uint32_t)q[e] << s;
        if (s + B > 32) w[word + 1] |= (uint32_t)q[e] >> (32 - s);
    }
    if constexpr (B % 2 == 0) {  // 16-byte aligned (the stream of 64 codes starts at 8 B bytes)
        uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int k = 0; k < B / 2; ++k) d[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    } else {  // 8-byte aligned
        uint2* d = reinterpret_cast<uint2*>(dst);
#pragma unroll
        for (int k = 0; k < B; ++k) d[k] = make_uint2(w[2 * k], w[2 * k + 1]);
    }
}

// Row pointer functor: rows(i) returns a 16-byte aligned pointer to 128 fp16 values.
// which: 0 = K (token-major codes), 1 = V (channel-major codes).
// bar_id: named barrier used among the 256 participating threads (threads 0..255).
// Hardware reciprocal (rcp.approx.ftz.f32, within an ulp or so): the Sinkhorn
// iteration corrects its own rounding, and the squared scales stay inside
// [kSqMin, kSqMax] (no denormals to flush).
__device__ __forceinline__ float fast_rcp(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

template <class Rows>
__device__ void seal_matrix(const Rows& rows, int bits, int which, int iters, uint8_t* rec, float* dbg,
                            SealSmem& S, int bar_id) {
    const int t = threadIdx.x;
    const int i = t >> 1, h = t & 1;  // row role: token row i, channel half h
    const int j = t >> 1, hc = t & 1; // column role: channel j, token half hc
    // 1. rotation Y = X H of every token row: 6 butterfly stages in registers,
    //    the seventh across the partner thread, then the 1/sqrt(128) scaling.
    float x[64];
    {
        const uint4* src = reinterpret_cast<const uint4*>(rows(i) + 64 * h);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint4 w = src[q];
            const __half2* hp = reinterpret_cast<const __half2*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = __half22float2(hp[e]);
                x[8 * q + 2 * e] = f.x;
                x[8 * q + 2 * e + 1] = f.y;
            }
        }
    }
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
    float arow[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        float o = __shfl_xor_sync(0xffffffffu, x[k], 1);
        float y = (h ? (o - x[k]) : (x[k] + o)) * kInvSqrt128;
        x[k] = y;
        arow[k] = y * y;
    }
    {
        float4* dst = reinterpret_cast<float4*>(S.Y + 136 * i + 68 * h);
#pragma unroll
        for (int q = 0; q < 16; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    if (t < 128) S.u[ypad(t)] = 1.0f;
    named_bar(bar_id, 256);
    float acol[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        float y = S.Y[136 * (64 * hc + k) + ypad(j)];
        acol[k] = y * y;
    }
    // 2. Sinkhorn on A = Y*Y in its matrix-vector form: a_i^2 = mean_j A_ij / c_j^2,
    //    then c_j^2 = mean_i A_ij / a_i^2 (equal to rescaling the rows and columns of
    //    Y in turn; a zero row or column keeps the factor 1).
    float a2 = 1.0f, c2 = 1.0f;
    // (eight partial sums per pass keep the FMA chains short; the reciprocals are the
    // hardware approximation, fast_rcp)
    for (int it = 0; it < iters; ++it) {
        float pp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const float4* up = reinterpret_cast<const float4*>(S.u + 68 * h);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            float4 uu = up[q];
            const int o = 4 * (q & 1);
            pp[o] = fmaf(arow[4 * q], uu.x, pp[o]);
            pp[o + 1] = fmaf(arow[4 * q + 1], uu.y, pp[o + 1]);
            pp[o + 2] = fmaf(arow[4 * q + 2], uu.z, pp[o + 2]);
            pp[o + 3] = fmaf(arow[4 * q + 3], uu.w, pp[o + 3]);
        }
        float p = ((pp[0] + pp[4]) + (pp[2] + pp[6])) + ((pp[1] + pp[5]) + (pp[3] + pp[7]));
        p += __shfl_xor_sync(0xffffffffu, p, 1);
        a2 = p * (1.0f / 128.0f);
        // zero row keeps factor 1; the clamp only binds on divergent inputs (see kSqMax)
        a2 = a2 == 0.0f ? 1.0f : fminf(fmaxf(a2, kSqMin), kSqMax);
        if (h == 0) S.v[ypad(i)] = fast_rcp(a2);
        named_bar(bar_id, 256);
#pragma unroll
        for (int k = 0; k < 8; ++k) pp[k] = 0.f;
        const float4* vp = reinterpret_cast<const float4*>(S.v + 68 * hc);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            float4 vv = vp[q];
            const int o = 4 * (q & 1);
            pp[o] = fmaf(acol[4 * q], vv.x, pp[o]);
            pp[o + 1] = fmaf(acol[4 * q + 1], vv.y, pp[o + 1]);
            pp[o + 2] = fmaf(acol[4 * q + 2], vv.z, pp[o + 2]);
            pp[o + 3] = fmaf(acol[4 * q + 3], vv.w, pp[o + 3]);
        }
        p = ((pp[0] + pp[4]) + (pp[2] + pp[6])) + ((pp[1] + pp[5]) + (pp[3] + pp[7]));
        p += __shfl_xor_sync(0xffffffffu, p, 1);
        c2 = p * (1.0f / 128.0f);
        c2 = c2 == 0.0f ? 1.0f : fminf(fmaxf(c2, kSqMin), kSqMax);
        if (hc == 0) S.u[ypad(j)] = fast_rcp(c2);
        named_bar(bar_id, 256);
    }
    // 3. stored scales: fp16, round to nearest even, saturating
    if (h == 0) {
        float a = sqrtf(a2);
        uint16_t ab = f16_bits_sat(a);
        S.a16[i] = ab;
        const float af = half_bits_to_float(ab);
        S.ra[i] = af != 0.0f ? 1.0f / af : 0.0f;  // a zero scale maps the row to 0
        if (dbg) dbg[i] = a;
    }
    if (hc == 0) {
        float c = sqrtf(c2);
        uint16_t cb = f16_bits_sat(c);
        S.c16[j] = cb;
        const float cf = half_bits_to_float(cb);
        S.rc[j] = cf != 0.0f ? 1.0f / cf : 0.0f;
        if (dbg) dbg[128 + j] = c;
    }
    named_bar(bar_id, 256);
    // 4. normalised values Z' = Y / (a16 c16) from the packing perspective of this side
    float z[64];
    if (which == 0) {
        const float4* src = reinterpret_cast<const float4*>(S.Y + 136 * i + 68 * h);
        const float rai = S.ra[i];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            float4 y = src[q];
            z[4 * q + 0] = y.x * rai * S.rc[64 * h + 4 * q + 0];
            z[4 * q + 1] = y.y * rai * S.rc[64 * h + 4 * q + 1];
            z[4 * q + 2] = y.z * rai * S.rc[64 * h + 4 * q + 2];
            z[4 * q + 3] = y.w * rai * S.rc[64 * h + 4 * q + 3];
        }
    } else {
        const float rcj = S.rc[j];
#pragma unroll
        for (int k = 0; k < 64; ++k) z[k] = S.Y[136 * (64 * hc + k) + ypad(j)] * S.ra[64 * hc + k] * rcj;
    }
    float mn = z[0], mx = z[0];
#pragma unroll
    for (int k = 1; k < 64; ++k) {
        mn = fminf(mn, z[k]);
        mx = fmaxf(mx, z[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((t & 31) == 0) {
        S.red[0][t >> 5] = mn;
        S.red[1][t >> 5] = mx;
    }
    named_bar(bar_id, 256);
    mn = S.red[0][0];
    mx = S.red[1][0];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
        mn = fminf(mn, S.red[0][w]);
        mx = fmaxf(mx, S.red[1][w]);
    }
    const int L = (1 << bits) - 1;
    float delta = (mx - mn) / (float)L;
    if (delta == 0.0f) delta = 1.0f;
    const float inv = 1.0f / delta;
    // 5. round to nearest (ties to even), clamp, pack
    int qv[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        int c = __float2int_rn((z[k] - mn) * inv);
        qv[k] = min(max(c, 0), L);
    }
    const int row = (which == 0) ? i : j;  // token row (K) or channel row (V)
    const int half = (which == 0) ? h : hc;
    uint8_t* codes = rec + 528;
    uint8_t* dst = codes + 16 * bits * row + 8 * bits * half;  // 128 codes a row, 64 a half
    switch (bits) {
        case 2: pack64_store<2>(qv, dst); break;
        case 3: pack64_store<3>(qv, dst); break;
        case 4: pack64_store<4>(qv, dst); break;
        case 5: pack64_store<5>(qv, dst); break;
        case 6: pack64_store<6>(qv, dst); break;
        default: pack64_store<8>(qv, dst); break;
    }
    // 6. header: delta, m, zero, a16[128], c16[128]
    uint16_t* r16 = reinterpret_cast<uint16_t*>(rec);
    if (t == 0) {
        uint4 hdr = make_uint4(__float_as_uint(delta), __float_as_uint(mn), 0u, 0u);
        *reinterpret_cast<uint4*>(rec) = hdr;
    }
    if (t < 128)
        r16[8 + t] = S.a16[t];
    else
        r16[8 + 128 + (t - 128)] = S.c16[t - 128];
    named_bar(bar_id, 256);
}

}  // namespace kvarn
