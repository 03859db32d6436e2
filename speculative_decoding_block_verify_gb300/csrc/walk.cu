// The Markov head's draft-side walk on sm_103a: bias slot i by the token sampled at slot i-1,
// sample t_i, left to right, in one launch.
//
// Method: "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com),
// §3 "The Markov fix-up" and Figure 2 ("slot 1 bias(t0)", the walk runs inside the draft
// pass's CUDA graph); "MTP Heads and Confidence Heads" (naphjohn.github.io), §6 "Why the Markov
// Head Helps" (B = W1 @ W2, default rank 256).
//
//   l~_i = l_i + W1[t_{i-1}] @ W2   (t_{-1} = the anchor),   t_i ~ softmax(l~_i / T)
//
// Design: one cooperative grid, one CTA per SM; CTA c owns a contiguous slice of the
// vocabulary for the whole walk.  Per slot: the CTA gathers W1[t_{i-1}] of up to WG (kWalkGroup, or 1 for a lone stream)
// streams into shared memory and computes the biased logits of its slice - W2 (66 MB for rank
// 256 at V = 129,280) is read once per slot for all streams of the group and stays in L2
// between slots; the CTA's 8 warps split it as 4 column groups x 2 rank halves - writes them (they are the rows the verify's q is taken from) and publishes
// one partial: (integer reference K, sum of 2^(l~ a - K)) for T > 0, (maximum, lowest index)
// for T = 0.  After a grid barrier every CTA reduces the same partials in the same order, so
// all agree on the draw: the 64-bit fixed-point CDF over the slices (the verify's scheme)
// picks the slice, and every CTA splits that slice over its warps and rescans one eighth, so
// every CTA holds t_i for the next slot without a second barrier (CTA 0 publishes it; the
// partials alternate between two buffers from slot to slot).  The barrier is a bounded spin
// (a cooperative launch keeps every CTA resident); one that gives up makes the walk's streams
// TIMEOUT.

#include <cooperative_groups.h>

#include <atomic>

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "df.cuh"
#include "draw.cuh"
#include "host_util.h"

namespace sv {

constexpr int kWalkThreads = 256;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kWalkGroup = 4;        // streams walked together (each W2 element feeds all of them)
constexpr int kWalkMaxRank = 1024;
constexpr int kWalkMaxCtas = 2048;
constexpr unsigned long long kWalkWaitNs = 4000000000ull;
constexpr float kWalkNoRef = -1e30f;

struct WalkParams {
    const void* draft;     // [B, N, V]
    const int32_t* anchor; // [B]
    const void* W1;        // [V, R]
    const void* W2;        // [R, V]
    const float* temp;     // [B]
    uint64_t seed, step;
    int32_t* tokens;       // [B, N]
    float* out;            // [B, N, V]
    int32_t* status;       // [B]
    char* ws;              // workspace: barrier counter, timeout flag, partials [2][B][kWalkMaxCtas]
    int32_t B, N, V, R;
    int64_t nchunk;        // chunks of E elements per row
    int64_t cw;            // chunks per CTA slice
};

struct WalkPart {
    float K;
    float s_hi, s_lo;
    int idx;
};

// The barrier counter and timeout flag, then the CTAs' partials in two buffers: slot i writes
// and reads buffer i mod 2, so a CTA already on slot i + 1 never overwrites partials that a
// slower CTA is still reading for slot i's draw.
__host__ __device__ inline size_t walk_workspace_bytes(int32_t B) {
    return 256 + 2 * (size_t)B * kWalkMaxCtas * sizeof(WalkPart);
}

__device__ __forceinline__ unsigned walk_now_load(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long walk_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid barrier: every CTA adds 1, then waits (bounded) for the count of this barrier.  Returns
// false once any CTA's wait has given up (then no later barrier waits either).
__device__ bool walk_barrier(unsigned* ctr, unsigned* timed_out, unsigned target) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        ok = 1;
        const unsigned long long t0 = walk_ns();
        for (int it = 0;; ++it) {
            if (walk_now_load(ctr) >= target) break;
            if (walk_now_load(timed_out) != 0u || walk_ns() - t0 > kWalkWaitNs || it > (1 << 26)) {
                atomicExch(timed_out, 1u);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
    }
    __syncthreads();
    return ok != 0;
}

// Dynamic shared memory of a walk CTA over groups of WG streams: the group's W1 rows [WG][R]
// floats, the rank halves' meeting area [4][32][WG][E] floats, then (16-byte aligned) one float4
// per CTA of the grid for the partials of the stream being drawn.
__host__ __device__ inline size_t walk_parts_offset(int R, int E, int WG) {
    const size_t b = sizeof(float) * ((size_t)WG * R + (size_t)4 * 32 * WG * E);
    return (b + 15) & ~(size_t)15;
}

// WG streams walked together (each W2 element feeds all of them): WG, or 1 for a lone
// stream, whose bias then issues a quarter of the FMAs.
template <typename DT, typename WT, int E, int WG>
__global__ void __launch_bounds__(kWalkThreads, 1) walk_kernel(const WalkParams p) {
    extern __shared__ __align__(16) float w1s[];   // [WG][R], the reduction area, the CTAs' partials
    __shared__ int s_prev[WG], s_alive[WG], s_greedy[WG], s_status[WG];
    __shared__ float s_ah[WG], s_al[WG];
    __shared__ float s_red[kWalkWarps][WG][4];
    __shared__ int s_draw_seg;
    __shared__ int s_tok[WG];   // the token each stream of the group drew at the current slot
    __shared__ unsigned long long s_sub[kWalkWarps], s_t, s_excl;
    __shared__ int s_sub_last[kWalkWarps];
    __shared__ float s_scale, s_K;
    const int c = blockIdx.x, ncta = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = p.V;
    const int64_t k0 = min(p.nchunk, (int64_t)c * p.cw), k1 = min(p.nchunk, k0 + p.cw);
    unsigned* ctr = reinterpret_cast<unsigned*>(p.ws);
    unsigned* timed_out = ctr + 1;
    WalkPart* parts = reinterpret_cast<WalkPart*>(p.ws + 256);
    // one stream's partials of every CTA, read from L2 once per draw by warp 0
    float4* s_parts = reinterpret_cast<float4*>(reinterpret_cast<char*>(w1s) + walk_parts_offset(p.R, E, WG));
    unsigned target = 0;
    bool live = true;   // no barrier has given up
    const float qnan = __int_as_float(0x7fffffff);

    for (int g0 = 0; g0 < p.B; g0 += WG) {
        const int gn = min(WG, p.B - g0);
        if (tid < WG) {
            const int b = g0 + tid;
            int st = SPEC_ST_OK;
            float ah = 0.f, al = 0.f;
            bool greedy = false;
            if (tid < gn) {
                const float T = p.temp[b];
                const int an = p.anchor[b];
                if (!(isfinite(T) && (T == 0.f || T >= FLT_MIN))) st = SPEC_ST_BAD_TEMPERATURE;
                else if (an < 0 || an >= p.V) st = SPEC_ST_BAD_TOKEN;
                greedy = (T == 0.f);
                if (st == SPEC_ST_OK && !greedy) {
                    const df a = temperature_scale(T);
                    ah = a.hi;
                    al = a.lo;
                }
            }
            s_status[tid] = (tid < gn) ? st : SPEC_ST_BAD_TOKEN;
            s_alive[tid] = (tid < gn && st == SPEC_ST_OK) ? 1 : 0;
            s_greedy[tid] = greedy ? 1 : 0;
            s_ah[tid] = ah;
            s_al[tid] = al;
        }
        __syncthreads();
        for (int i = 0; i < p.N; ++i) {
            // ---- the previous tokens and the gathered W1 rows; a stream that has stopped
            // reports -1 for the rest of its slots
            if (tid < WG) {
                const int b = g0 + tid;
                if (c == 0 && tid < gn && !s_alive[tid]) p.tokens[(int64_t)b * p.N + i] = -1;
                s_prev[tid] = (s_alive[tid] != 0) ? (i == 0 ? p.anchor[b] : s_tok[tid]) : 0;
            }
            __syncthreads();
            for (int t = tid; t < WG * p.R; t += kWalkThreads) {
                const int gi = t / p.R, j = t - gi * p.R;
                w1s[t] = (gi < gn && s_alive[gi]) ? load_elem<WT>(p.W1, (int64_t)s_prev[gi] * p.R + j) : 0.f;
            }
            __syncthreads();
            // ---- biased logits of this CTA's slice, and their maximum
            float mx[WG];
            int arg[WG];
#pragma unroll
            for (int g = 0; g < WG; ++g) {
                mx[g] = -kInf;
                arg[g] = INT_MAX;
            }
            // The 8 warps take (32 chunks, half of the rank): warp w sums ranks
            // [h R / 2, (h + 1) R / 2), h = w / 4, of chunks base + 32 (w % 4) + lane, a lane with 16
            // W2 loads in flight; the upper half's sums meet the lower half's in shared memory,
            // where the lower half's warps finish the chunks.
            const int half = warp >> 2, cgrp = warp & 3;
            const int jsplit = (p.R + 1) / 2;
            const int ja = half ? jsplit : 0, jb = half ? p.R : jsplit;
            float* red = w1s + WG * p.R;   // [4][32][WG][E]
            for (int64_t cb = k0; cb < k1; cb += 4 * 32) {
                const int64_t k = cb + cgrp * 32 + lane;
                const bool act = k < k1;
                float acc[WG][E];
#pragma unroll
                for (int g = 0; g < WG; ++g)
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
                if (act) {
#pragma unroll 16
                    for (int j = ja; j < jb; ++j) {
                        Chunk<WT, E> cwv;
                        cwv.load(row_ptr<WT>(p.W2, j, V), k);
                        float x[E];
                        cwv.unpack(x);
#pragma unroll
                        for (int g = 0; g < WG; ++g) {
                            const float wv = w1s[g * p.R + j];
#pragma unroll
                            for (int e = 0; e < E; ++e) acc[g][e] = fmaf(wv, x[e], acc[g][e]);
                        }
                    }
                }
                float* rl = red + ((cgrp * 32 + lane) * WG) * E;
                if (half) {
#pragma unroll
                    for (int g = 0; g < WG; ++g)
#pragma unroll
                        for (int e = 0; e < E; ++e) rl[g * E + e] = acc[g][e];
                }
                __syncthreads();   // the upper half's sums are in shared memory
                if (!half && act) {
#pragma unroll
                    for (int g = 0; g < WG; ++g)
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[g][e] += rl[g * E + e];
#pragma unroll
                    for (int g = 0; g < WG; ++g) {
                        if (g >= gn) continue;
                        const int64_t row = ((int64_t)(g0 + g) * p.N + i);
                        Chunk<DT, E> cd;
                        cd.load(row_ptr<DT>(p.draft, row, V), k);
                        float d[E];
                        cd.unpack(d);
                        float* o = p.out + row * V + k * E;
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float l = s_alive[g] ? d[e] + acc[g][e] : qnan;
                            o[e] = l;
                            const float key = s_greedy[g] ? l : l * s_ah[g];
                            if (!(key <= mx[g])) {   // a new maximum, NaN included (it then sticks)
                                if (!(key == mx[g])) arg[g] = (int)(k * E + e);
                                mx[g] = fmax_nan(mx[g], key);
                            }
                        }
                    }
                }
                __syncthreads();   // the lower half is done with the shared sums
            }
            // CTA maximum (NaN-aware) and its lowest index, per stream
#pragma unroll
            for (int g = 0; g < WG; ++g) {
                const float m = warp_max_nan(mx[g]);
                const int a = warp_min_i(mx[g] == m ? arg[g] : INT_MAX);
                if (lane == 0) {
                    s_red[warp][g][0] = m;
                    s_red[warp][g][1] = __int_as_float(a);
                }
            }
            __syncthreads();
            if (tid < WG) {
                float m = -kInf;
                for (int w = 0; w < kWalkWarps; ++w) m = fmax_nan(m, s_red[w][tid][0]);
                int a = INT_MAX;
                for (int w = 0; w < kWalkWarps; ++w)
                    if (s_red[w][tid][0] == m) a = min(a, __float_as_int(s_red[w][tid][1]));
                s_red[0][tid][2] = m;
                s_red[0][tid][3] = __int_as_float(a);
            }
            __syncthreads();
            // ---- T > 0: sum 2^(l~ a - K) over the slice (K = ceil of the slice maximum); the
            // biased values are read back from the output this CTA just wrote
            float kref[WG];
            df sum[WG];
#pragma unroll
            for (int g = 0; g < WG; ++g) {
                const float m = s_red[0][g][2];
                kref[g] = (isfinite(m)) ? ceilf(m) : kWalkNoRef;
                sum[g] = df{0.f, 0.f};
            }
            for (int64_t k = k0 + tid; k < k1; k += kWalkThreads) {
#pragma unroll
                for (int g = 0; g < WG; ++g) {
                    if (g >= gn || s_greedy[g] || !s_alive[g]) continue;
                    const float* o = p.out + ((int64_t)(g0 + g) * p.N + i) * V + k * E;
                    float t = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float l = __ldcg(o + e);
                        t += ex2(fmaf(l, s_al[g], fmaf(l, s_ah[g], -kref[g])));
                    }
                    sum[g] = df_add_f(sum[g], t);
                }
            }
#pragma unroll
            for (int g = 0; g < WG; ++g) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const df other{__shfl_xor_sync(0xffffffffu, sum[g].hi, o), __shfl_xor_sync(0xffffffffu, sum[g].lo, o)};
                    sum[g] = df_add(sum[g], other);
                }
                if (lane == 0) {
                    s_red[warp][g][0] = sum[g].hi;
                    s_red[warp][g][1] = sum[g].lo;
                }
            }
            __syncthreads();
            if (tid < gn) {
                df z{0.f, 0.f};
                for (int w = 0; w < kWalkWarps; ++w) z = df_add(z, df{s_red[w][tid][0], s_red[w][tid][1]});
                const int b = g0 + tid;
                const bool gr = s_greedy[tid] != 0;
                parts[((int64_t)(i & 1) * p.B + b) * kWalkMaxCtas + c] =
                    WalkPart{gr ? s_red[0][tid][2] : kref[tid], gr ? 0.f : z.hi, gr ? 0.f : z.lo,
                             gr ? __float_as_int(s_red[0][tid][3]) : INT_MAX};
            }
            live = live && walk_barrier(ctr, timed_out, target += ncta);

            // ---- the draw, stream by stream.  Every CTA reduces the same partials in the same
            // order and rescans the same drawn slice of the biased row (in L2 since the barrier),
            // so every CTA arrives at the same token, keeps it for the next slot's W1 row, and no
            // second barrier is needed.
            for (int g = 0; g < gn; ++g) {
                const int b = g0 + g;
                if (!s_alive[g]) continue;
                const WalkPart* pb = parts + ((int64_t)(i & 1) * p.B + b) * kWalkMaxCtas;
                if (s_greedy[g]) {
                    if (warp == 0) {
                        for (int q = lane; q < ncta; q += 32) s_parts[q] = __ldcg(reinterpret_cast<const float4*>(pb + q));
                        __syncwarp();
                        float m = -kInf;
                        for (int q = lane; q < ncta; q += 32) m = fmax_nan(m, s_parts[q].x);
                        m = warp_max_nan(m);
                        int a = INT_MAX;
                        for (int q = lane; q < ncta; q += 32)
                            if (s_parts[q].x == m) a = min(a, __float_as_int(s_parts[q].w));
                        a = warp_min_i(a);
                        if (lane == 0) {
                            const bool bad = !isfinite(m) || a == INT_MAX;
                            if (bad) s_status[g] = SPEC_ST_BAD_ROW;
                            if (c == 0) p.tokens[(int64_t)b * p.N + i] = bad ? -1 : a;
                            s_tok[g] = bad ? -1 : a;
                        }
                    }
                    __syncthreads();
                    if (tid == 0 && s_status[g] != SPEC_ST_OK) s_alive[g] = 0;
                    __syncthreads();
                    continue;
                }
                // global reference and the slices' weights in 64-bit fixed point (warp 0)
                if (warp == 0) {
                    for (int q = lane; q < ncta; q += 32) s_parts[q] = __ldcg(reinterpret_cast<const float4*>(pb + q));
                    __syncwarp();
                    float K = kWalkNoRef;
                    bool bad = false;
                    for (int q = lane; q < ncta; q += 32) {
                        const float kq = s_parts[q].x;
                        bad |= isnan(kq);
                        K = fmaxf(K, kq);
                    }
                    K = warp_max(K);
                    bad = __any_sync(0xffffffffu, bad) || !(K > kWalkNoRef) || !isfinite(K);
                    float wmax = 0.f;
                    for (int q = lane; q < ncta; q += 32) {
                        const float4 e = s_parts[q];
                        const float wq = (e.y + e.z) * (e.x == K ? 1.f : pow2_int(e.x - K));
                        bad |= !isfinite(wq);
                        wmax = fmaxf(wmax, wq);
                    }
                    wmax = warp_max(wmax);
                    bad = __any_sync(0xffffffffu, bad) || !(wmax > 0.f);
                    const float scale = bad ? 0.f : fixed_scale(wmax);
                    // total, then the first slice whose running sum passes t = floor(U R)
                    unsigned long long tot = 0;
                    for (int q = lane; q < ncta; q += 32) {
                        const float4 e = s_parts[q];
                        tot += __float2ull_rn((e.y + e.z) * (e.x == K ? 1.f : pow2_int(e.x - K)) * scale);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
                    const uint64_t stp = p.step;
                    const uint4 ctrv = make_uint4((uint32_t)i, (uint32_t)b, (uint32_t)stp, (uint32_t)(stp >> 32));
                    const uint4 wds = philox4x32_10(ctrv, make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
                    const unsigned long long odd = 2ull * (wds.z >> 8) + 1ull;
                    const unsigned long long t = (__umul64hi(odd, tot) << 39) | ((odd * tot) >> 25);
                    // scan the slices in lane-sized blocks, in order
                    unsigned long long before = 0;
                    int seg = -1;
                    for (int q0 = 0; q0 < ncta && seg < 0; q0 += 32) {
                        const int q = q0 + lane;
                        unsigned long long wq = 0;
                        if (q < ncta) {
                            const float4 e = s_parts[q];
                            wq = __float2ull_rn((e.y + e.z) * (e.x == K ? 1.f : pow2_int(e.x - K)) * scale);
                        }
                        unsigned long long incl = wq;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += n;
                        }
                        const unsigned hit = __ballot_sync(0xffffffffu, wq > 0 && before + incl > t);
                        if (hit) {
                            const int L = __ffs(hit) - 1;
                            seg = q0 + L;
                            const unsigned long long ex = __shfl_sync(0xffffffffu, incl - wq, L);
                            before += ex;
                        } else {
                            before += __shfl_sync(0xffffffffu, incl, 31);
                        }
                    }
                    if (lane == 0) {
                        if (bad || tot == 0 || seg < 0) {   // NaN, +inf or no finite logit in the row
                            s_status[g] = SPEC_ST_BAD_ROW;
                            s_draw_seg = -1;
                        } else {
                            s_draw_seg = seg;
                            s_t = t;
                            s_excl = before;
                            s_scale = scale;
                            s_K = K;
                        }
                    }
                }
                __syncthreads();
                if (s_status[g] != SPEC_ST_OK) {
                    __syncthreads();
                    if (tid == 0) {
                        if (c == 0) p.tokens[(int64_t)b * p.N + i] = -1;
                        s_alive[g] = 0;
                    }
                    __syncthreads();
                    continue;
                }
                {   // the drawn slice (CTA s_draw_seg's), split over the warps
                    const float* row = p.out + ((int64_t)b * p.N + i) * V;
                    const int64_t d0 = min(p.nchunk, (int64_t)s_draw_seg * p.cw), d1 = min(p.nchunk, d0 + p.cw);
                    const int64_t msub = (d1 - d0 + kWalkWarps - 1) / kWalkWarps;
                    const int64_t w0 = min(d1, d0 + warp * msub), w1 = min(d1, w0 + msub);
                    unsigned long long sub;
                    int last;
                    // an eighth of at most 64 chunks stays in registers between its sum and its rescan
                    const bool held = msub <= 64;
                    DrawSlice<float, f32_coherent, E, true> slice;
                    if (held) {
                        slice.load(nullptr, row, w0, w1, 0.f, s_K, s_ah[g], s_al[g], 0.f, s_scale, lane, nullptr, 0);
                        slice.sum(sub, last);
                    } else {
                        segment_fixed_sum<float, f32_coherent, E, true>(nullptr, row, w0, w1, 0.f, s_K, s_ah[g], s_al[g],
                                                                        0.f, s_scale, lane, sub, last, nullptr, 0);
                    }
                    if (lane == 0) {
                        s_sub[warp] = sub;
                        s_sub_last[warp] = last;
                    }
                    __syncthreads();
                    const unsigned long long tt = s_t - s_excl;
                    unsigned long long bef = 0;
                    int wsel = -1, lastpos = -1;
                    for (int w = 0; w < kWalkWarps; ++w) {
                        lastpos = max(lastpos, s_sub_last[w]);
                        if (wsel < 0) {
                            if (s_sub[w] > 0 && bef + s_sub[w] > tt) wsel = w;
                            else bef += s_sub[w];
                        }
                    }
                    int y = -1;
                    if (wsel < 0) y = lastpos;   // rounding kept the slice's sum at or below the target
                    else if (warp == wsel)
                        y = held ? slice.rescan(tt - bef, lane)
                                 : rescan_segment<float, f32_coherent, E, true>(nullptr, row, w0, w1, 0.f, s_K, s_ah[g],
                                                                                s_al[g], 0.f, s_scale, tt - bef, lane,
                                                                                nullptr, 0);
                    if ((wsel < 0 && tid == 0) || (warp == wsel && lane == 0)) {
                        if (c == 0) p.tokens[(int64_t)b * p.N + i] = y;
                        s_tok[g] = y;
                    }
                }
                __syncthreads();
            }
        }
        // ---- statuses of the group (CTA 0); a stream that stopped early pads its tokens
        if (c == 0 && tid < gn) {
            const int b = g0 + tid;
            p.status[b] = live ? s_status[tid] : SPEC_ST_TIMEOUT;
        }
        if (c == 0 && !live)
            for (int t = tid; t < gn * p.N; t += kWalkThreads)
                p.tokens[(int64_t)(g0 + t / p.N) * p.N + t % p.N] = -1;
        __syncthreads();
    }
}

template <typename DT, typename WT, int E, int WG>
static cudaError_t launch_walk_wg(WalkParams& p, cudaStream_t s) {
    static std::atomic<int> grid_cache[64];   // per device: the cooperative grid (0: not yet set up)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int grid = grid_cache[dev].load(std::memory_order_acquire);
    if (grid == 0) {
        cudaError_t e = cudaFuncSetAttribute(walk_kernel<DT, WT, E, WG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(walk_parts_offset(kWalkMaxRank, E, WG) + sizeof(float4) * kWalkMaxCtas));
        if (e != cudaSuccess) return e;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
        grid = sms < kWalkMaxCtas ? sms : kWalkMaxCtas;
        grid_cache[dev].store(grid, std::memory_order_release);
    }
    p.cw = (p.nchunk + grid - 1) / grid;
    const size_t smem = walk_parts_offset(p.R, E, WG) + sizeof(float4) * (size_t)grid;
    // the barrier counter and timeout flag start at zero in every launch
    cudaError_t e = cudaMemsetAsync(p.ws, 0, 8, s);
    if (e != cudaSuccess) return e;
    void* args[] = {&p};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(walk_kernel<DT, WT, E, WG>), dim3(grid),
                                       dim3(kWalkThreads), args, smem, s);
}

template <typename DT, typename WT, int E>
static cudaError_t launch_walk(WalkParams& p, cudaStream_t s) {
    return p.B == 1 ? launch_walk_wg<DT, WT, E, 1>(p, s) : launch_walk_wg<DT, WT, E, kWalkGroup>(p, s);
}

template <int E>
static cudaError_t dispatch_walk(WalkParams& p, int dt, int wt, cudaStream_t s) {
    if (dt == SPEC_DTYPE_BF16 && wt == SPEC_DTYPE_BF16) return launch_walk<__nv_bfloat16, __nv_bfloat16, E>(p, s);
    if (dt == SPEC_DTYPE_F32 && wt == SPEC_DTYPE_F32) return launch_walk<float, float, E>(p, s);
    if (dt == SPEC_DTYPE_F32 && wt == SPEC_DTYPE_BF16) return launch_walk<float, __nv_bfloat16, E>(p, s);
    return launch_walk<__nv_bfloat16, float, E>(p, s);
}

}  // namespace sv

extern "C" size_t dspark_markov_walk_workspace_bytes(int32_t B) {
    return B < 0 ? 0 : sv::walk_workspace_bytes(B);
}

extern "C" int dspark_markov_walk(const void* draft_logits, int32_t draft_dtype, int32_t B, int32_t N, int32_t V,
                                  const int32_t* anchor, const void* W1, const void* W2, int32_t w_dtype,
                                  int32_t rank, const float* temperature, uint64_t seed, uint64_t step,
                                  int32_t* out_tokens, float* out_logits, int32_t* status, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    const char* name = "dspark_markov_walk";
    if (!sv::valid_dtype(draft_dtype) || !sv::valid_dtype(w_dtype))
        return sv::set_error(SPEC_ERR_DTYPE, "%s: dtype must be SPEC_DTYPE_F32 or SPEC_DTYPE_BF16", name);
    if (B < 0 || N < 0 || N > SPEC_MAX_KMAX || V < 1 || V > SPEC_MAX_V || rank < 1 || rank > sv::kWalkMaxRank)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: B=%d N=%d V=%d rank=%d out of range", name, B, N, V, rank);
    if (B == 0) return sv::clear_error();
    if (!draft_logits && N > 0) return sv::set_error(SPEC_ERR_ARG, "%s: draft_logits is NULL", name);
    if (!anchor || !W1 || !W2 || !temperature || !status || (N > 0 && (!out_tokens || !out_logits)))
        return sv::set_error(SPEC_ERR_ARG, "%s: a pointer is NULL", name);
    const size_t need = sv::walk_workspace_bytes(B);
    if (workspace == nullptr || workspace_bytes < need || (uintptr_t)workspace % 16 != 0)
        return sv::set_error(SPEC_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", name,
                             need, workspace_bytes);
    sv::WalkParams p;
    p.draft = draft_logits;
    p.anchor = anchor;
    p.W1 = W1;
    p.W2 = W2;
    p.temp = temperature;
    p.seed = seed;
    p.step = step;
    p.tokens = out_tokens;
    p.out = out_logits;
    p.status = status;
    p.ws = reinterpret_cast<char*>(workspace);
    p.B = B;
    p.N = N;
    p.V = V;
    p.R = rank;
    const bool aligned = (V % 8 == 0) && ((uintptr_t)W2 % 16 == 0) && ((uintptr_t)draft_logits % 16 == 0) &&
                         ((uintptr_t)out_logits % 16 == 0);
    p.nchunk = aligned ? V / 8 : V;
    p.cw = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = aligned ? sv::dispatch_walk<8>(p, draft_dtype, w_dtype, s)
                                  : sv::dispatch_walk<1>(p, draft_dtype, w_dtype, s);
    if (e != cudaSuccess) return sv::set_cuda_error(e, name);
    return sv::clear_error();
}
