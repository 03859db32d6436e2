// Device helpers shared by the verify, Markov-bias and pick-k kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

constexpr float kInf = __builtin_huge_valf();
constexpr double kLog2e = 1.4426950408889634073599246810019;
constexpr double kLn2 = 0.69314718055994530941723212145818;

// ---------------------------------------------------------------------------------------
// Scalar helpers
// ---------------------------------------------------------------------------------------

// 2^x on the special-function unit (relative error about 2^-22; subnormal results -> 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that returns NaN when either operand is NaN (so NaN rows are seen by the max alone).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): counter (4 words), key (2 words).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
        const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += W0;
        k.y += W1;
    }
    return c;
}

// U(x) = ((x >> 8) + 0.5) * 2^-24, exact in double, strictly inside (0, 1).
__device__ __forceinline__ double uniform24(uint32_t x) {
    return ((double)(x >> 8) + 0.5) * 0x1p-24;
}

// (acceptance uniform, sampling uniform) of (stream, slot) in step `step` under `seed`.
__device__ __forceinline__ double2 slot_uniforms(uint64_t seed, uint64_t step, uint32_t stream,
                                                 uint32_t slot) {
    const uint4 c = make_uint4(slot, stream, (uint32_t)step, (uint32_t)(step >> 32));
    const uint2 k = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
    const uint4 w = philox4x32_10(c, k);
    return make_double2(uniform24(w.x), uniform24(w.y));
}

// ---------------------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// inclusive prefix sum across the warp (lane order)
__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// ---------------------------------------------------------------------------------------
// Logit loaders: a "chunk" is E consecutive elements of one row.  E = 8 uses 16-byte loads
// (one for bf16, two for float) and needs 16-byte aligned rows; E = 1 is the plain path.
// ---------------------------------------------------------------------------------------
template <typename T, int E>
struct Chunk;

// A chunk of a row may also be gathered: element e of chunk k is row[t2d[8 k + e]], or -inf
// where t2d holds no index in [0, K) (a reduced draft vocabulary seen in target columns).
__device__ __forceinline__ bool in_vocab(int j, int32_t K) { return (unsigned)j < (unsigned)K; }

template <>
struct Chunk<__nv_bfloat16, 8> {
    uint4 raw;
    __device__ __forceinline__ void load(const void* row, int64_t chunk) {
        raw = __ldg(reinterpret_cast<const uint4*>(row) + chunk);
    }
    __device__ __forceinline__ void gather(const void* row, const int32_t* t2d, int32_t K, int64_t chunk) {
        const int4 a = __ldg(reinterpret_cast<const int4*>(t2d) + 2 * chunk);
        const int4 b = __ldg(reinterpret_cast<const int4*>(t2d) + 2 * chunk + 1);
        const int j[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = in_vocab(j[e], K) ? (uint32_t)__ldg(r + j[e]) : 0xff80u;   // bf16 -inf
        raw = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = bf16_lo(raw.x); x[1] = bf16_hi(raw.x);
        x[2] = bf16_lo(raw.y); x[3] = bf16_hi(raw.y);
        x[4] = bf16_lo(raw.z); x[5] = bf16_hi(raw.z);
        x[6] = bf16_lo(raw.w); x[7] = bf16_hi(raw.w);
    }
};

template <>
struct Chunk<float, 8> {
    float4 a, b;
    __device__ __forceinline__ void load(const void* row, int64_t chunk) {
        const float4* p = reinterpret_cast<const float4*>(row) + 2 * chunk;
        a = __ldg(p);
        b = __ldg(p + 1);
    }
    __device__ __forceinline__ void gather(const void* row, const int32_t* t2d, int32_t K, int64_t chunk) {
        const int4 ja = __ldg(reinterpret_cast<const int4*>(t2d) + 2 * chunk);
        const int4 jb = __ldg(reinterpret_cast<const int4*>(t2d) + 2 * chunk + 1);
        const float* r = reinterpret_cast<const float*>(row);
        const float ninf = __int_as_float(0xff800000);
        a = make_float4(in_vocab(ja.x, K) ? __ldg(r + ja.x) : ninf, in_vocab(ja.y, K) ? __ldg(r + ja.y) : ninf,
                        in_vocab(ja.z, K) ? __ldg(r + ja.z) : ninf, in_vocab(ja.w, K) ? __ldg(r + ja.w) : ninf);
        b = make_float4(in_vocab(jb.x, K) ? __ldg(r + jb.x) : ninf, in_vocab(jb.y, K) ? __ldg(r + jb.y) : ninf,
                        in_vocab(jb.z, K) ? __ldg(r + jb.z) : ninf, in_vocab(jb.w, K) ? __ldg(r + jb.w) : ninf);
    }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};

template <>
struct Chunk<__nv_bfloat16, 1> {
    uint16_t raw;
    __device__ __forceinline__ void load(const void* row, int64_t chunk) {
        raw = __ldg(reinterpret_cast<const unsigned short*>(row) + chunk);
    }
    __device__ __forceinline__ void gather(const void* row, const int32_t* t2d, int32_t K, int64_t chunk) {
        const int j = __ldg(t2d + chunk);
        raw = in_vocab(j, K) ? __ldg(reinterpret_cast<const unsigned short*>(row) + j) : (uint16_t)0xff80u;
    }
    __device__ __forceinline__ void unpack(float (&x)[1]) const {
        x[0] = __uint_as_float((uint32_t)raw << 16);
    }
};

template <>
struct Chunk<float, 1> {
    float v;
    __device__ __forceinline__ void load(const void* row, int64_t chunk) {
        v = __ldg(reinterpret_cast<const float*>(row) + chunk);
    }
    __device__ __forceinline__ void gather(const void* row, const int32_t* t2d, int32_t K, int64_t chunk) {
        const int j = __ldg(t2d + chunk);
        v = in_vocab(j, K) ? __ldg(reinterpret_cast<const float*>(row) + j) : __int_as_float(0xff800000);
    }
    __device__ __forceinline__ void unpack(float (&x)[1]) const { x[0] = v; }
};

// float32 rows written earlier by the same kernel (other CTAs, or the read-only path's cache
// from an earlier step): loaded through L2 (ld.global.cg), never through the read-only path.
struct f32_coherent {
    float v;
};
template <>
struct Chunk<f32_coherent, 8> {
    float4 a, b;
    __device__ __forceinline__ void load(const void* row, int64_t chunk) {
        const float4* p = reinterpret_cast<const float4*>(row) + 2 * chunk;
        a = __ldcg(p);
        b = __ldcg(p + 1);
    }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};
template <>
struct Chunk<f32_coherent, 1> {
    float v;
    __device__ __forceinline__ void load(const void* row, int64_t chunk) {
        v = __ldcg(reinterpret_cast<const float*>(row) + chunk);
    }
    __device__ __forceinline__ void unpack(float (&x)[1]) const { x[0] = v; }
};

// One element of a row (any alignment).
template <typename T>
__device__ __forceinline__ float load_elem(const void* row, int64_t i);
template <>
__device__ __forceinline__ float load_elem<float>(const void* row, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
}
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const void* row, int64_t i) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + i)
                           << 16);
}

template <typename T>
__device__ __forceinline__ const void* row_ptr(const void* base, int64_t row, int64_t V) {
    return reinterpret_cast<const T*>(base) + row * V;
}

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------------------------------
// Packed float32x2 arithmetic (one instruction for two lanes of data; compiler builtins)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------------------------------
// 1D bulk copies (TMA, cp.async.bulk) completing on a shared-memory mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

// Per-thread asynchronous 16-byte copies global -> shared (L2 only), grouped per thread.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's committed groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}


__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make the initialised barriers visible to the async proxy
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// order this thread's earlier generic shared-memory accesses before later async-proxy ones
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// global -> this CTA's shared memory, `bytes` a multiple of 16, both addresses 16-byte aligned
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// An L2 cache policy that evicts these lines before any other: for logits that are streamed
// through once, so that they do not push the kernels' code and workspace out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
// one poll of the barrier's phase `parity`; true once that phase has completed
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

}  // namespace sv
