// Token-wise speculative sampling and block verification on sm_103a.
//
// Method: "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com),
// §4 "Verification: the guarantee" - "Token by token" (Leviathan et al. 2023), "Block
// verification" (Sun et al. 2024) with Figure 3, and "Greedy is a different code path".
//
// Design (one launch per call):
//   * one thread-block cluster of C CTAs per stream; CTA c owns a contiguous vocabulary slice
//     of every row of its stream, split into one contiguous segment per warp (C x 8 segments
//     per row, in vocabulary order);
//   * stats sweep: every logit of the stream is read from HBM exactly once (16-byte loads);
//     each lane keeps an online (max, sum 2^((l - max) a), argmax) per row, a = log2(e) / T;
//     warps publish per-segment partials in shared memory;
//   * one cluster barrier, then every CTA reduces all partials through distributed shared
//     memory in the same order, so every CTA holds bit-identical row statistics and takes the
//     same per-stream decisions (float64 scalars) without further communication;
//   * block verification evaluates tau top-down (i = N .. 1): h_N = w_N needs no sweep; an i
//     with eta_i > w_i fails without one (h_i <= w_i); otherwise a residual sweep of slot i
//     (re-read, mostly from L2) gives r_i and h_i; tau = 0 needs one sweep of slot 0;
//   * the draw: per-segment masses give a coarse CDF; the warp whose segment holds U*R
//     rescans that segment and writes the token.
// Slot 0 is the last pair read by the stats sweep so that its residual sweep (the common
// tau = 0 case at low acceptance) finds it in L2.

#include <cooperative_groups.h>

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "host_util.h"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxRows = 2 * SPEC_MAX_KMAX + 1;
constexpr int kMaxSeg = kMaxCluster * kWarps;

struct VerifyParams {
    int32_t B, V, kmax, rule;
    const int32_t* cu;
    const void* dq;
    const void* dp;
    const int32_t* tokens;
    const float* temp;
    uint64_t seed, step;
    int32_t* acc_len;
    int32_t* out_tok;
    int32_t* n_emit;
    int32_t* status;
    float* diag;
    int64_t nchunk;      // chunks per row
    int64_t seg_chunks;  // chunks per warp segment
};

struct Part {
    float m;
    float s;
    int idx;
};

struct Shared {
    Part part[kMaxRows][kWarps];
    float res_part[2][kWarps];
    float row_m[kMaxRows];
    double row_z[kMaxRows];
    int row_arg[kMaxRows];
    double seg_w[kMaxSeg];
    double bonus_w[kMaxSeg];
    double log2px[SPEC_MAX_KMAX];
    double log2qx[SPEC_MAX_KMAX];
    double rho[SPEC_MAX_KMAX];
    double log2w[SPEC_MAX_KMAX + 1];
    double w[SPEC_MAX_KMAX + 1];
    double h[SPEC_MAX_KMAX + 1];
    double r[SPEC_MAX_KMAX + 1];
    double u_acc[SPEC_MAX_KMAX + 1];
    double u_smp[SPEC_MAX_KMAX + 1];
    double resid_R;
    double sample_t;
    int x[SPEC_MAX_KMAX];
    int N, status, greedy, tau, pass_slot, done, sample_seg, sample_bonus;
    float a;
    float cc;
};

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <typename T, int E>
struct Unroll {
    static constexpr int value = (E == 1) ? 8 : (sizeof(T) == 2 ? 4 : 2);
};

// ---------------------------------------------------------------------------------------
// Per-lane online row statistics
// ---------------------------------------------------------------------------------------
template <int E, bool ARG, bool SUM>
struct LaneAcc {
    float m = -kInf;
    float s = 0.f;
    int idx = INT_MAX;
    __device__ __forceinline__ void add(const float (&x)[E], int64_t elem0, float a) {
        float vm = x[0];
#pragma unroll
        for (int j = 1; j < E; ++j) vm = fmax_nan(vm, x[j]);
        if (!(vm <= m)) {  // a new maximum (or a NaN)
            if (ARG) {
                int j0 = 0;
#pragma unroll
                for (int j = E - 1; j >= 0; --j)
                    if (x[j] == vm) j0 = j;
                idx = (int)(elem0 + j0);
            }
            if (SUM) s = (m == -kInf) ? 0.f : s * ex2((m - vm) * a);
            m = fmax_nan(m, vm);
        }
        if (SUM && m != -kInf) {
#pragma unroll
            for (int j = 0; j < E; ++j) s += ex2((x[j] - m) * a);
        }
    }
    // warp-combine and publish (lane 0)
    __device__ __forceinline__ void publish(Part* dst, float a, int lane) const {
        const float mw = warp_max_nan(m);
        float sw = 0.f;
        if (SUM) sw = warp_sum((m == -kInf) ? 0.f : s * ex2((m - mw) * a));
        const int iw = ARG ? warp_min_i((m == mw) ? idx : INT_MAX) : INT_MAX;
        if (lane == 0) *dst = Part{mw, sw, iw};
    }
};

// stats of one row pair (draft row q, target row p) over this warp's segment [c0, c1)
template <typename DQ, typename DP, int E>
__device__ __forceinline__ void stats_pair(const void* rq, const void* rp, int64_t c0, int64_t c1,
                                           float a, int lane, Part* dq, Part* dp) {
    constexpr int U = Unroll<DQ, E>::value < Unroll<DP, E>::value ? Unroll<DQ, E>::value
                                                                 : Unroll<DP, E>::value;
    LaneAcc<E, false, true> aq;
    LaneAcc<E, true, true> ap;
    for (int64_t base = c0; base < c1; base += 32 * U) {
        Chunk<DQ, E> cq[U];
        Chunk<DP, E> cp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                cq[u].load(rq, k);
                cp[u].load(rp, k);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                float x[E];
                cq[u].unpack(x);
                aq.add(x, k * E, a);
                cp[u].unpack(x);
                ap.add(x, k * E, a);
            }
        }
    }
    aq.publish(dq, a, lane);
    ap.publish(dp, a, lane);
}

// stats of one target row (bonus row: with sums; greedy rows: max/argmax only)
template <typename DP, int E, bool SUM>
__device__ __forceinline__ void stats_single(const void* rp, int64_t c0, int64_t c1, float a,
                                             int lane, Part* dp) {
    constexpr int U = 2 * Unroll<DP, E>::value;
    LaneAcc<E, true, SUM> ap;
    for (int64_t base = c0; base < c1; base += 32 * U) {
        Chunk<DP, E> cp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) cp[u].load(rp, k);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                float x[E];
                cp[u].unpack(x);
                ap.add(x, k * E, a);
            }
        }
    }
    ap.publish(dp, a, lane);
}

// residual weights max(0, cc * 2^((lp - mp) a) - 2^((lq - mq) a)) of one chunk
template <int E>
__device__ __forceinline__ void residual_weights(const float (&xq)[E], const float (&xp)[E],
                                                 float mq, float mp, float a, float cc,
                                                 float (&wt)[E]) {
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const float ep = ex2((xp[j] - mp) * a);
        const float eq = ex2((xq[j] - mq) * a);
        wt[j] = fmaxf(0.f, fmaf(cc, ep, -eq));
    }
}

// sum of residual weights over this warp's segment
template <typename DQ, typename DP, int E>
__device__ __forceinline__ float residual_sum(const void* rq, const void* rp, int64_t c0,
                                              int64_t c1, float mq, float mp, float a, float cc,
                                              int lane) {
    constexpr int U = Unroll<DQ, E>::value < Unroll<DP, E>::value ? Unroll<DQ, E>::value
                                                                 : Unroll<DP, E>::value;
    float s = 0.f;
    for (int64_t base = c0; base < c1; base += 32 * U) {
        Chunk<DQ, E> cq[U];
        Chunk<DP, E> cp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                cq[u].load(rq, k);
                cp[u].load(rp, k);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                float xq[E], xp[E], wt[E];
                cq[u].unpack(xq);
                cp[u].unpack(xp);
                residual_weights<E>(xq, xp, mq, mp, a, cc, wt);
#pragma unroll
                for (int j = 0; j < E; ++j) s += wt[j];
            }
        }
    }
    return warp_sum(s);
}

// Inverse-CDF rescan of one warp segment: the smallest element whose running mass reaches t
// (or, if rounding keeps the running mass below t, the segment's last positive element).
template <typename DQ, typename DP, int E, bool BONUS>
__device__ __forceinline__ int rescan_segment(const void* rq, const void* rp, int64_t c0,
                                              int64_t c1, float mq, float mp, float a, float cc,
                                              double t, int lane) {
    constexpr int U = Unroll<DQ, E>::value < Unroll<DP, E>::value ? Unroll<DQ, E>::value
                                                                 : Unroll<DP, E>::value;
    double run = 0.0;
    int y = -1, ylast = -1;
    for (int64_t base = c0; base < c1 && y < 0; base += 32 * U) {
        Chunk<DQ, E> cq[U];
        Chunk<DP, E> cp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                if (!BONUS) cq[u].load(rq, k);
                cp[u].load(rp, k);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            float wt[E];
            float lsum = 0.f;
            int lpos = -1;
            if (k < c1) {
                float xp[E];
                cp[u].unpack(xp);
                if (BONUS) {
#pragma unroll
                    for (int j = 0; j < E; ++j) wt[j] = ex2((xp[j] - mp) * a);
                } else {
                    float xq[E];
                    cq[u].unpack(xq);
                    residual_weights<E>(xq, xp, mq, mp, a, cc, wt);
                }
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    lsum += wt[j];
                    if (wt[j] > 0.f) lpos = (int)(k * E + j);
                }
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) wt[j] = 0.f;
            }
            const double incl = warp_incl_scan_d((double)lsum, lane);
            const double total = __shfl_sync(0xffffffffu, incl, 31);
            const unsigned hit = __ballot_sync(0xffffffffu, lsum > 0.f && run + incl >= t);
            // last positive element so far (the fallback)
            const int lp_max = __reduce_max_sync(0xffffffffu, lpos);
            if (lp_max >= 0) ylast = lp_max;
            if (hit && y < 0) {
                const int L = __ffs(hit) - 1;
                int yl = -1;
                if (lane == L) {
                    double acc = run + incl - (double)lsum;
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        acc += (double)wt[j];
                        if (yl < 0 && wt[j] > 0.f && acc >= t) yl = (int)(k * E + j);
                    }
                    if (yl < 0) yl = lpos;
                }
                y = __shfl_sync(0xffffffffu, yl, L);
            }
            run += total;
        }
    }
    return y >= 0 ? y : ylast;
}

// ---------------------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------------------
template <typename DQ, typename DP, int E>
__global__ void __launch_bounds__(kThreads, 3) verify_kernel(const VerifyParams p) {
    __shared__ Shared sh;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nseg = C * kWarps;
    const int64_t c0 = min(p.nchunk, (int64_t)(crank * kWarps + warp) * p.seg_chunks);
    const int64_t c1 = min(p.nchunk, c0 + p.seg_chunks);
    const int64_t V = p.V;

    // ---- stream header: offsets, temperature, tokens (identical in every CTA)
    if (tid == 0) {
        int st = SPEC_ST_OK;
        const int base = p.cu[b];
        const int n = p.cu[b + 1] - base;
        if (n < 0 || n > p.kmax) st = SPEC_ST_BAD_OFFSETS;
        const float T = p.temp[b];
        if (st == SPEC_ST_OK && !(isfinite(T) && (T == 0.f || T >= FLT_MIN)))
            st = SPEC_ST_BAD_TEMPERATURE;
        const int nn = (st == SPEC_ST_BAD_OFFSETS) ? 0 : n;
        if (st == SPEC_ST_OK) {
            for (int i = 0; i < nn; ++i) {
                const int xi = p.tokens[base + i];
                sh.x[i] = xi;
                if (xi < 0 || xi >= p.V) st = SPEC_ST_BAD_TOKEN;
            }
        }
        sh.N = nn;
        sh.status = st;
        sh.greedy = (st == SPEC_ST_OK && T == 0.f);
        sh.a = (st == SPEC_ST_OK && T > 0.f) ? (float)(kLog2e / (double)T) : 0.f;
        sh.tau = 0;
        sh.done = 0;
    }
    __syncthreads();
    const int N = sh.N;
    const float a = sh.a;
    const bool greedy = sh.greedy;
    const int64_t dbase = (sh.status == SPEC_ST_BAD_OFFSETS) ? 0 : p.cu[b];
    const int64_t tbase = dbase + b;
    auto qrow = [&](int i) { return row_ptr<DQ>(p.dq, dbase + i, V); };
    auto prow = [&](int i) { return row_ptr<DP>(p.dp, tbase + i, V); };
    const int nrows = 2 * N + 1;  // part index: draft row i -> i, target row i -> N + i

    if (sh.status == SPEC_ST_OK) {
        // ---- stats sweep: bonus row first, then pairs 1..N-1, then pair 0
        if (!greedy) {
            stats_single<DP, E, true>(prow(N), c0, c1, a, lane, &sh.part[2 * N][warp]);
            for (int j = 1; j <= N; ++j) {
                const int i = (j < N) ? j : 0;
                stats_pair<DQ, DP, E>(qrow(i), prow(i), c0, c1, a, lane, &sh.part[i][warp],
                                      &sh.part[N + i][warp]);
            }
        } else {
            for (int i = 0; i <= N; ++i)
                stats_single<DP, E, false>(prow(i), c0, c1, 0.f, lane, &sh.part[N + i][warp]);
        }
        __syncthreads();
        cluster_sync_all();

        // ---- cluster reduction of the per-segment partials (same order in every CTA)
        for (int r = (greedy ? N : 0) + warp; r < nrows; r += kWarps) {
            Part e[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int s = lane + 32 * k;
                if (s < nseg) {
                    const Part* src = cluster.map_shared_rank(&sh.part[r][s % kWarps], s / kWarps);
                    e[k] = *src;
                } else {
                    e[k] = Part{-kInf, 0.f, INT_MAX};
                }
            }
            const float M = warp_max_nan(fmax_nan(e[0].m, e[1].m));
            double z = 0.0;
            double sc[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                sc[k] = (e[k].m == -kInf || greedy) ? 0.0 : (double)(e[k].s * ex2((e[k].m - M) * a));
                z += sc[k];
            }
            z = warp_sum_d(z);
            const int arg = warp_min_i(min(e[0].m == M ? e[0].idx : INT_MAX,
                                           e[1].m == M ? e[1].idx : INT_MAX));
            if (lane == 0) {
                sh.row_m[r] = M;
                sh.row_z[r] = z;
                sh.row_arg[r] = arg;
            }
            if (r == 2 * N && !greedy) {
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (lane + 32 * k < nseg) sh.bonus_w[lane + 32 * k] = sc[k];
            }
        }
        __syncthreads();

        // ---- validity of the rows read, and q_i(x_i) > 0
        bool bad_row = false, zero_q = false;
        for (int r = (greedy ? N : 0) + tid; r < nrows; r += kThreads) {
            const float M = sh.row_m[r];
            bad_row |= !isfinite(M) || !isfinite(sh.row_z[r]) || !(greedy || sh.row_z[r] > 0.0);
        }
        if (!greedy && tid < N) {
            const int xi = sh.x[tid];
            const float lq = load_elem<DQ>(qrow(tid), xi);
            const float lp = load_elem<DP>(prow(tid), xi);
            zero_q = (lq == -kInf);
            const double a64 = (double)a;
            const double lzp = log2(sh.row_z[N + tid]);
            const double lzq = log2(sh.row_z[tid]);
            sh.log2px[tid] = ((double)lp - (double)sh.row_m[N + tid]) * a64 - lzp;
            sh.log2qx[tid] = ((double)lq - (double)sh.row_m[tid]) * a64 - lzq;
        }
        if (!greedy && tid <= N) {
            const double2 u = slot_uniforms(p.seed, p.step, (uint32_t)b, (uint32_t)tid);
            sh.u_acc[tid] = u.x;
            sh.u_smp[tid] = u.y;
        }
        bad_row = __syncthreads_or(bad_row);
        zero_q = __syncthreads_or(zero_q);
        if (tid == 0) {
            if (bad_row) sh.status = SPEC_ST_BAD_ROW;
            else if (zero_q) sh.status = SPEC_ST_ZERO_DRAFT_PROB;
        }
        if (!greedy && tid < N) sh.rho[tid] = exp2(sh.log2px[tid] - sh.log2qx[tid]);
        __syncthreads();
    }

    // ---- decisions
    if (sh.status == SPEC_ST_OK && greedy) {
        if (tid == 0) {
            int tau = N;
            for (int i = 0; i < N; ++i)
                if (sh.row_arg[N + i] != sh.x[i]) { tau = i; break; }
            sh.tau = tau;
        }
        __syncthreads();
    } else if (sh.status == SPEC_ST_OK) {
        const bool block = (p.rule == 1);
        if (tid <= N) {
            sh.h[tid] = nan("");
            sh.r[tid] = nan("");
        }
        if (block) {
            if (tid == 0) {
                sh.log2w[0] = 0.0;
                for (int i = 0; i < N; ++i)
                    sh.log2w[i + 1] = fmin(0.0, sh.log2w[i] + (sh.log2px[i] - sh.log2qx[i]));
            }
            __syncthreads();
            if (tid <= N) sh.w[tid] = exp2(sh.log2w[tid]);
            __syncthreads();
            if (tid == 0) {
                // u_acc[i-1] is eta_i
                if (N == 0) {
                    sh.tau = 0; sh.done = 1;       // bonus only
                } else {
                    sh.h[N] = sh.w[N];
                    if (sh.u_acc[N - 1] <= sh.h[N]) { sh.tau = N; sh.done = 1; }
                    else { sh.pass_slot = N; sh.done = 0; }
                }
            }
        } else if (tid == 0) {
            int tau = N;
            for (int i = 0; i < N; ++i)
                if (!(sh.u_acc[i] <= fmin(1.0, sh.rho[i]))) { tau = i; break; }
            sh.tau = tau;
            sh.done = (tau == N);
            sh.pass_slot = tau;
            if (tau < N) { sh.w[tau] = 1.0; }
        }
        __syncthreads();

        // ---- residual sweeps (cluster-wide, lazily, at most N + 1)
        int phase = 0;
        while (true) {
            if (tid == 0 && !sh.done && block) {
                // next candidate below the last one tried
                int i = sh.pass_slot - 1;
                while (i >= 1 && sh.u_acc[i - 1] > sh.w[i]) --i;
                sh.pass_slot = i;   // i == 0: tau = 0 and slot 0's residual is needed
            }
            __syncthreads();
            if (sh.done) break;
            const int i = sh.pass_slot;
            const float mq = sh.row_m[i], mp = sh.row_m[N + i];
            const float cc = (float)(sh.w[i] * sh.row_z[i] / sh.row_z[N + i]);
            const float ws = residual_sum<DQ, DP, E>(qrow(i), prow(i), c0, c1, mq, mp, a, cc, lane);
            if (lane == 0) sh.res_part[phase][warp] = ws;
            __syncthreads();
            cluster_sync_all();
            if (warp == 0) {
                double tot = 0.0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int s = lane + 32 * k;
                    double v = 0.0;
                    if (s < nseg)
                        v = (double)*cluster.map_shared_rank(&sh.res_part[phase][s % kWarps], s / kWarps);
                    if (s < kMaxSeg) sh.seg_w[s] = v;
                    tot += v;
                }
                tot = warp_sum_d(tot);
                if (lane == 0) {
                    sh.resid_R = tot;
                    const double ri = tot / sh.row_z[i];
                    sh.r[i] = ri;
                    if (!block || i == 0) {
                        sh.tau = i;
                        sh.done = 1;
                    } else {
                        const double den = ri + 1.0 - sh.w[i];
                        const double hi = (den == 0.0) ? 1.0 : ri / den;
                        sh.h[i] = hi;
                        if (sh.u_acc[i - 1] <= hi) { sh.tau = i; sh.done = 1; }
                    }
                }
            }
            __syncthreads();
            phase ^= 1;
            if (sh.done) break;
        }

        // ---- the draw: coarse CDF over segments, then the owner warp rescans
        if (tid == 0) {
            const int tau = sh.tau;
            const bool bonus = (tau == N);
            const double* wseg = bonus ? sh.bonus_w : sh.seg_w;
            double R = 0.0;
            for (int s = 0; s < nseg; ++s) R += wseg[s];
            sh.sample_bonus = bonus;
            if (!(R > 0.0) || !isfinite(R)) {
                sh.status = SPEC_ST_NUMERIC;
                sh.sample_seg = -1;
            } else {
                const double t = sh.u_smp[tau] * R;
                double cum = 0.0;
                int seg = -1, lastpos = -1;
                double tr = 0.0;
                for (int s = 0; s < nseg; ++s) {
                    if (wseg[s] > 0.0) {
                        lastpos = s;
                        if (seg < 0 && cum + wseg[s] >= t) { seg = s; tr = t - cum; }
                    }
                    cum += wseg[s];
                }
                if (seg < 0) { seg = lastpos; tr = wseg[lastpos]; }
                sh.sample_seg = seg;
                sh.sample_t = tr;
            }
        }
        __syncthreads();
        if (sh.status == SPEC_ST_OK && sh.sample_seg == crank * kWarps + warp) {
            const int tau = sh.tau;
            int y;
            if (sh.sample_bonus) {
                y = rescan_segment<DQ, DP, E, true>(nullptr, prow(N), c0, c1, 0.f, sh.row_m[2 * N],
                                                    a, 0.f, sh.sample_t, lane);
            } else {
                const float cc = (float)(sh.w[tau] * sh.row_z[tau] / sh.row_z[N + tau]);
                y = rescan_segment<DQ, DP, E, false>(qrow(tau), prow(tau), c0, c1, sh.row_m[tau],
                                                     sh.row_m[N + tau], a, cc, sh.sample_t, lane);
            }
            if (lane == 0) p.out_tok[(int64_t)b * (p.kmax + 1) + tau] = y;
        }
    }

    // ---- outputs (CTA rank 0)
    if (crank == 0) {
        const int st = sh.status;
        const int tau = sh.tau;
        const int64_t ob = (int64_t)b * (p.kmax + 1);
        for (int j = tid; j <= p.kmax; j += kThreads) {
            if (st != SPEC_ST_OK) p.out_tok[ob + j] = -1;
            else if (j < tau) p.out_tok[ob + j] = sh.x[j];
            else if (j > tau) p.out_tok[ob + j] = -1;
            else if (greedy) p.out_tok[ob + j] = sh.row_arg[N + tau];
        }
        if (tid == 0) {
            p.status[b] = st;
            p.acc_len[b] = (st == SPEC_ST_OK) ? tau : 0;
            p.n_emit[b] = (st == SPEC_ST_OK) ? tau + 1 : 0;
        }
        if (p.diag != nullptr && st != SPEC_ST_BAD_OFFSETS) {
            const float qnan = __int_as_float(0x7fffffff);
            const bool have = (!greedy) && (st == SPEC_ST_OK || st == SPEC_ST_NUMERIC);
            for (int i = tid; i <= N; i += kThreads) {
                float* d = p.diag + (tbase + i) * SPEC_DIAG_COLS;
                float v[SPEC_DIAG_COLS];
#pragma unroll
                for (int c = 0; c < SPEC_DIAG_COLS; ++c) v[c] = qnan;
                if (have) {
                    const double a64 = (double)a;
                    v[SPEC_DIAG_LOGZP] = (float)(kLn2 * ((double)sh.row_m[N + i] * a64 + log2(sh.row_z[N + i])));
                    if (i < N) {
                        v[SPEC_DIAG_PX] = (float)exp2(sh.log2px[i]);
                        v[SPEC_DIAG_QX] = (float)exp2(sh.log2qx[i]);
                        v[SPEC_DIAG_RHO] = (float)sh.rho[i];
                        v[SPEC_DIAG_LOGZQ] = (float)(kLn2 * ((double)sh.row_m[i] * a64 + log2(sh.row_z[i])));
                    }
                    if (p.rule == 1) {
                        v[SPEC_DIAG_W] = (float)sh.w[i];
                        if (i >= 1) v[SPEC_DIAG_H] = (float)sh.h[i];
                    }
                    v[SPEC_DIAG_R] = (float)sh.r[i];
                }
#pragma unroll
                for (int c = 0; c < SPEC_DIAG_COLS; ++c) d[c] = v[c];
            }
        }
    }
    // no CTA may leave while another can still read its shared memory
    cluster_sync_all();
}

// Uniforms exposed for checking: out[(s * n_slots + i) * 2 + {0, 1}]
__global__ void philox_uniforms_kernel(uint64_t seed, uint64_t step, int n_streams, int n_slots,
                                       double* out) {
    const int64_t total = (int64_t)n_streams * n_slots;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const double2 u = slot_uniforms(seed, step, (uint32_t)(t / n_slots), (uint32_t)(t % n_slots));
        out[2 * t] = u.x;
        out[2 * t + 1] = u.y;
    }
}

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------
template <typename DQ, typename DP, int E>
static cudaError_t launch_verify(const VerifyParams& p, int C, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_kernel<DQ, DP, E>, p);
}

// How many clusters of C CTAs fit on the device at once (queried once per kernel and C).
template <typename DQ, typename DP, int E>
static int resident_clusters(int C) {
    static int cache[kMaxCluster + 1][64] = {};   // [C][device]
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int& slot = cache[C][dev];
    if (slot == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)C);
        cfg.blockDim = dim3(kThreads);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, verify_kernel<DQ, DP, E>, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = 1;
        }
        slot = n;
    }
    return slot;
}

// Cluster size: each stream is one cluster; a larger cluster finishes its stream sooner, but
// streams beyond the resident cluster count run in extra waves.  Minimise waves / C, with at
// least 64 chunks per warp segment (small vocabularies use small clusters).
template <typename DQ, typename DP, int E>
static int pick_cluster(int B, int64_t nchunk) {
    int cmax = (int)(nchunk / (kWarps * 64));
    cmax = cmax < 1 ? 1 : (cmax > kMaxCluster ? kMaxCluster : cmax);
    int best = 1;
    double best_cost = 1e300;
    for (int C = 1; C <= cmax; ++C) {
        const int res = resident_clusters<DQ, DP, E>(C);
        const double waves = (double)((B + res - 1) / res);
        const double cost = waves / C;
        if (cost < best_cost * (1.0 - 1e-9)) {
            best_cost = cost;
            best = C;
        }
    }
    return best;
}

template <typename DQ, typename DP, int E>
static cudaError_t run_verify(VerifyParams& p, cudaStream_t s) {
    const int C = pick_cluster<DQ, DP, E>(p.B, p.nchunk);
    p.seg_chunks = (p.nchunk + (int64_t)C * kWarps - 1) / ((int64_t)C * kWarps);
    return launch_verify<DQ, DP, E>(p, C, s);
}

template <int E>
static cudaError_t dispatch_dtypes(VerifyParams& p, int dq, int dp, cudaStream_t s) {
    if (dq == SPEC_DTYPE_BF16 && dp == SPEC_DTYPE_BF16)
        return run_verify<__nv_bfloat16, __nv_bfloat16, E>(p, s);
    if (dq == SPEC_DTYPE_F32 && dp == SPEC_DTYPE_F32) return run_verify<float, float, E>(p, s);
    if (dq == SPEC_DTYPE_F32 && dp == SPEC_DTYPE_BF16)
        return run_verify<float, __nv_bfloat16, E>(p, s);
    return run_verify<__nv_bfloat16, float, E>(p, s);
}

static int verify_entry(const spec_verify_args* a, void* stream, int rule, const char* name) {
    if (a == nullptr) return set_error(SPEC_ERR_ARG, "%s: args is NULL", name);
    if (a->B < 0) return set_error(SPEC_ERR_SHAPE, "%s: B = %d < 0", name, a->B);
    if (a->V < 1 || a->V > SPEC_MAX_V)
        return set_error(SPEC_ERR_SHAPE, "%s: V = %d outside [1, %d]", name, a->V, SPEC_MAX_V);
    if (a->kmax < 0 || a->kmax > SPEC_MAX_KMAX)
        return set_error(SPEC_ERR_SHAPE, "%s: kmax = %d outside [0, %d]", name, a->kmax,
                         SPEC_MAX_KMAX);
    if (!valid_dtype(a->draft_dtype) || !valid_dtype(a->target_dtype))
        return set_error(SPEC_ERR_DTYPE, "%s: dtype must be SPEC_DTYPE_F32 or SPEC_DTYPE_BF16",
                         name);
    if (a->B == 0) return clear_error();
    if (!a->cu_drafts || !a->target_logits || !a->temperature || !a->accepted_len ||
        !a->out_tokens || !a->n_emitted || !a->status)
        return set_error(SPEC_ERR_ARG, "%s: a required pointer is NULL", name);
    if ((a->kmax > 0) && (!a->draft_logits || !a->draft_tokens))
        return set_error(SPEC_ERR_ARG, "%s: draft_logits / draft_tokens is NULL", name);
    VerifyParams p;
    p.B = a->B;
    p.V = a->V;
    p.kmax = a->kmax;
    p.rule = rule;
    p.cu = a->cu_drafts;
    p.dq = a->draft_logits;
    p.dp = a->target_logits;
    p.tokens = a->draft_tokens;
    p.temp = a->temperature;
    p.seed = a->seed;
    p.step = a->step;
    p.acc_len = a->accepted_len;
    p.out_tok = a->out_tokens;
    p.n_emit = a->n_emitted;
    p.status = a->status;
    p.diag = a->diag;
    const bool aligned = (a->V % 8 == 0) && ((uintptr_t)a->target_logits % 16 == 0) &&
                         ((uintptr_t)a->draft_logits % 16 == 0);
    p.nchunk = aligned ? a->V / 8 : a->V;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = aligned ? dispatch_dtypes<8>(p, a->draft_dtype, a->target_dtype, s)
                                  : dispatch_dtypes<1>(p, a->draft_dtype, a->target_dtype, s);
    if (e != cudaSuccess) return set_cuda_error(e, name);
    return clear_error();
}

}  // namespace sv

extern "C" int spec_verify_tokenwise(const spec_verify_args* args, void* stream) {
    return sv::verify_entry(args, stream, 0, "spec_verify_tokenwise");
}

extern "C" int spec_verify_block(const spec_verify_args* args, void* stream) {
    return sv::verify_entry(args, stream, 1, "spec_verify_block");
}

extern "C" int spec_philox_uniforms(uint64_t seed, uint64_t step, int32_t n_streams,
                                    int32_t n_slots, double* out, void* stream) {
    if (n_streams < 0 || n_slots < 0)
        return sv::set_error(SPEC_ERR_SHAPE, "spec_philox_uniforms: negative count");
    const int64_t total = (int64_t)n_streams * n_slots;
    if (total == 0) return sv::clear_error();
    if (out == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_philox_uniforms: out is NULL");
    const int64_t blocks64 = (total + 255) / 256;
    const int blocks = (int)(blocks64 < 4096 ? blocks64 : 4096);
    sv::philox_uniforms_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        seed, step, n_streams, n_slots, out);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_philox_uniforms");
    return sv::clear_error();
}
