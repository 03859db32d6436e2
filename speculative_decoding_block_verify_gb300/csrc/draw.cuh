// The inverse-CDF draw's fixed-point helpers shared by the verify and Markov-walk kernels
// (sm_103a): per-element weights of a residual max(0, c 2^(xp a - Kp) - 2^(xq a - Kq)) or of a
// softmax row 2^(xp a - Kp), converted to 64-bit fixed point with a power-of-two scale, summed
// and rescanned so that a draw reads each element of the drawn slice once more at most.
#pragma once

#include "common.cuh"
#include "df.cuh"

namespace sv {

// residual weights max(0, c 2^(xp a - Kp) - 2^(xq a - Kq)) of one chunk
template <int E>
__device__ __forceinline__ void resid_weights(const float (&xq)[E], const float (&xp)[E], float Kq, float Kp,
                                              float ah, float al, float c, float (&w)[E]) {
    if (E == 1) {
        const float ep = ex2(fmaf(xp[0], al, fmaf(xp[0], ah, -Kp)));
        const float eq = ex2(fmaf(xq[0], al, fmaf(xq[0], ah, -Kq)));
        w[0] = fmaxf(0.f, fmaf(c, ep, -eq));
    } else {
        const float2 a2h = make_float2(ah, ah), a2l = make_float2(al, al);
        const float2 nkp = make_float2(-Kp, -Kp), nkq = make_float2(-Kq, -Kq);
#pragma unroll
        for (int j = 0; j < E / 2; ++j) {
            const float2 pp = make_float2(xp[2 * j], xp[2 * j + 1]);
            const float2 qq = make_float2(xq[2 * j], xq[2 * j + 1]);
            const float2 e1 = ffma2(pp, a2l, ffma2(pp, a2h, nkp));
            const float2 e2 = ffma2(qq, a2l, ffma2(qq, a2h, nkq));
            w[2 * j] = fmaxf(0.f, fmaf(c, ex2(e1.x), -ex2(e2.x)));
            w[2 * j + 1] = fmaxf(0.f, fmaf(c, ex2(e1.y), -ex2(e2.y)));
        }
    }
}

// Draft chunk k: read from the draft row, or - over a reduced draft vocabulary (t2d given) -
// gathered through the column map.
template <typename DQ, int E>
__device__ __forceinline__ void load_q_chunk(Chunk<DQ, E>& c, const void* rq, int64_t k, const int32_t* t2d,
                                             int32_t Kv) {
    if (t2d) c.gather(rq, t2d, Kv, k);
    else c.load(rq, k);
}

// Fixed-point weight (times `scale`) of each element of one chunk pair.
template <typename DQ, typename DP, int E, bool BONUS>
__device__ __forceinline__ void rescan_weights(const Chunk<DQ, E>& cq, const Chunk<DP, E>& cp, float Kq, float Kp,
                                               float ah, float al, float c, float scale,
                                               unsigned long long (&qv)[E]) {
    float xp[E], w[E];
    cp.unpack(xp);
    if (BONUS) {
#pragma unroll
        for (int j = 0; j < E; ++j) w[j] = ex2(fmaf(xp[j], al, fmaf(xp[j], ah, -Kp)));
    } else {
        float xq[E];
        cq.unpack(xq);
        resid_weights<E>(xq, xp, Kq, Kp, ah, al, c, w);
    }
#pragma unroll
    for (int j = 0; j < E; ++j) qv[j] = __float2ull_rn(w[j] * scale);
}

// Inverse-CDF rescan of one warp segment in 64-bit fixed point (weights times `scale`): the
// first element whose running sum exceeds t, or - if rounding keeps the segment's sum at or
// below t - the segment's last positive element.  The segment is taken in groups of U chunks
// per lane (chunk base + 32 u + lane); the next group's loads are in flight while the current
// one is scanned, and the U cross-lane scans of a group are independent, so they overlap.
template <typename DQ, typename DP, int E, bool BONUS>
__device__ __noinline__ int rescan_segment(const void* rq, const void* rp, int64_t c0, int64_t c1, float Kq,
                                           float Kp, float ah, float al, float c, float scale, unsigned long long t,
                                           int lane, const int32_t* t2d, int32_t Kv) {
    // chunks per lane and group: bf16 rows 4, wider rows fewer (two groups stay in registers)
    constexpr int CB = E * (int)((BONUS ? 0 : sizeof(DQ)) + sizeof(DP));   // bytes per chunk (pair)
    constexpr int U = (E == 1) ? 4 : (CB <= 32 ? 2 : 1);
    constexpr int G = 32 * U;
    Chunk<DQ, E> qa[U], qb[U];
    Chunk<DP, E> pa[U], pb[U];
    auto load = [&](Chunk<DQ, E>(&cq)[U], Chunk<DP, E>(&cp)[U], int64_t base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                if (!BONUS) load_q_chunk(cq[u], rq, k, t2d, Kv);
                cp[u].load(rp, k);
            }
        }
    };
    unsigned long long run = 0;
    int ylast = -1;
    // one group: true once the token is found (y set)
    auto scan = [&](const Chunk<DQ, E>(&cq)[U], const Chunk<DP, E>(&cp)[U], int64_t base, int& y) -> bool {
        unsigned long long lsum[U], incl[U];
        int lpos[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            lsum[u] = 0;
            lpos[u] = -1;
            if (k < c1) {
                unsigned long long qv[E];
                rescan_weights<DQ, DP, E, BONUS>(cq[u], cp[u], Kq, Kp, ah, al, c, scale, qv);
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    lsum[u] += qv[j];
                    if (qv[j] > 0) lpos[u] = (int)(k * E + j);
                }
            }
            incl[u] = lsum[u];
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {   // U independent inclusive scans, interleaved
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned long long n = __shfl_up_sync(0xffffffffu, incl[u], o);
                if (lane >= o) incl[u] += n;
            }
        }
        int uh = -1, L = 0;
        unsigned long long before = 0;   // fixed-point mass before chunk slice uh
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned long long total = __shfl_sync(0xffffffffu, incl[u], 31);
            const unsigned hit = __ballot_sync(0xffffffffu, lsum[u] > 0 && run + incl[u] > t);
            const int lp_max = __reduce_max_sync(0xffffffffu, lpos[u]);
            if (uh < 0) {
                if (lp_max >= 0) ylast = lp_max;
                if (hit) {
                    uh = u;
                    L = __ffs(hit) - 1;
                    before = run;
                } else {
                    run += total;
                }
            }
        }
        if (uh < 0) return false;
        // lane L walks its chunk of slice uh
        int yl = -1;
        if (lane == L) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (u != uh) continue;
                const int64_t k = base + u * 32 + lane;
                unsigned long long qv[E];
                rescan_weights<DQ, DP, E, BONUS>(cq[u], cp[u], Kq, Kp, ah, al, c, scale, qv);
                unsigned long long acc = before + incl[u] - lsum[u];
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    acc += qv[j];
                    if (yl < 0 && qv[j] > 0 && acc > t) yl = (int)(k * E + j);
                }
                if (yl < 0) yl = lpos[u];
            }
        }
        y = __shfl_sync(0xffffffffu, yl, L);
        return true;
    };
    int y = -1;
    load(qa, pa, c0);
    for (int64_t base = c0; base < c1; base += 2 * G) {
        if (base + G < c1) load(qb, pb, base + G);
        if (scan(qa, pa, base, y)) break;
        if (base + G >= c1) break;
        if (base + 2 * G < c1) load(qa, pa, base + 2 * G);
        if (scan(qb, pb, base + G, y)) break;
    }
    return y >= 0 ? y : ylast;
}

// One warp's slice [k0, k1) (at most 64 chunks: two per lane) of the drawn segment, its
// fixed-point weights loaded once: sum() gives the slice's total and last positive element
// (every lane), rescan(t) - in the warp whose slice crosses the target - the first element
// whose running sum exceeds t, from the same registers.  Chunk order and arithmetic are those
// of segment_fixed_sum and rescan_segment (chunk k0 + 32 u + lane), so the token is the same.
template <typename DQ, typename DP, int E, bool BONUS>
struct DrawSlice {
    unsigned long long qv[2][E];
    unsigned long long lsum[2];
    int lpos[2];
    int64_t k0;
    __device__ __forceinline__ void load(const void* rq, const void* rp, int64_t a, int64_t b, float Kq, float Kp,
                                         float ah, float al, float c, float scale, int lane, const int32_t* t2d,
                                         int32_t Kv) {
        k0 = a;
        Chunk<DQ, E> cq[2];
        Chunk<DP, E> cp[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t k = a + u * 32 + lane;
            if (k < b) {
                if (!BONUS) load_q_chunk(cq[u], rq, k, t2d, Kv);
                cp[u].load(rp, k);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t k = a + u * 32 + lane;
            lsum[u] = 0;
            lpos[u] = -1;
#pragma unroll
            for (int j = 0; j < E; ++j) qv[u][j] = 0;
            if (k < b) {
                rescan_weights<DQ, DP, E, BONUS>(cq[u], cp[u], Kq, Kp, ah, al, c, scale, qv[u]);
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    lsum[u] += qv[u][j];
                    if (qv[u][j] > 0) lpos[u] = (int)(k * E + j);
                }
            }
        }
    }
    __device__ __forceinline__ void sum(unsigned long long& total, int& last) const {
        unsigned long long ls = lsum[0] + lsum[1];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
        total = ls;
        last = __reduce_max_sync(0xffffffffu, max(lpos[0], lpos[1]));
    }
    __device__ __forceinline__ int rescan(unsigned long long t, int lane) const {
        unsigned long long incl[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) incl[u] = lsum[u];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const unsigned long long n = __shfl_up_sync(0xffffffffu, incl[u], o);
                if (lane >= o) incl[u] += n;
            }
        unsigned long long run = 0;
        int ylast = -1;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const unsigned long long total = __shfl_sync(0xffffffffu, incl[u], 31);
            const unsigned hit = __ballot_sync(0xffffffffu, lsum[u] > 0 && run + incl[u] > t);
            const int lp_max = __reduce_max_sync(0xffffffffu, lpos[u]);
            if (lp_max >= 0) ylast = lp_max;
            if (hit) {
                const int L = __ffs(hit) - 1;
                int yl = -1;
                if (lane == L) {
                    unsigned long long acc = run + incl[u] - lsum[u];
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        acc += qv[u][j];
                        if (yl < 0 && qv[u][j] > 0 && acc > t) yl = (int)((k0 + u * 32 + lane) * E + j);
                    }
                    if (yl < 0) yl = lpos[u];
                }
                return __shfl_sync(0xffffffffu, yl, L);
            }
            run += total;
        }
        return ylast;
    }
};

// Fixed-point sum (weights times `scale`) of the chunks [k0, k1) and their last positive
// element, over the warp (every lane returns both).
template <typename DQ, typename DP, int E, bool BONUS>
__device__ __noinline__ void segment_fixed_sum(const void* rq, const void* rp, int64_t k0, int64_t k1, float Kq,
                                               float Kp, float ah, float al, float c, float scale, int lane,
                                               unsigned long long& sum, int& last, const int32_t* t2d, int32_t Kv) {
    constexpr int U = 2;
    unsigned long long ls = 0;
    int lp = -1;
    for (int64_t base = k0; base < k1; base += 32 * U) {
        Chunk<DQ, E> cq[U];
        Chunk<DP, E> cp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < k1) {
                if (!BONUS) load_q_chunk(cq[u], rq, k, t2d, Kv);
                cp[u].load(rp, k);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < k1) {
                unsigned long long qv[E];
                rescan_weights<DQ, DP, E, BONUS>(cq[u], cp[u], Kq, Kp, ah, al, c, scale, qv);
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    ls += qv[j];
                    if (qv[j] > 0) lp = (int)(k * E + j);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    sum = ls;
    last = __reduce_max_sync(0xffffffffu, lp);
}

// exponent l a - K as a df (a = ah + al), l finite
__device__ __forceinline__ df exponent_df(float l, float ah, float al, float K) {
    df e = two_prod(l, ah);
    e = df_add_f(e, __fmul_rn(l, al));
    return df_add_f(e, -K);
}

// power-of-two scale putting the largest weight just below 2^40
__device__ __forceinline__ float fixed_scale(float wmax) {
    int e;
    frexpf(wmax, &e);   // wmax = m 2^e, m in [0.5, 1)
    return pow2_int((float)(40 - e));
}

}  // namespace sv
