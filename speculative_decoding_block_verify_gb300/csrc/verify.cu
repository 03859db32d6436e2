// Token-wise speculative sampling and block verification on sm_103a.
//
// Method: "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com),
// §4 "Verification: the guarantee" - "Token by token" (Leviathan et al. 2023), "Block
// verification" (Sun et al. 2024) with Figure 3, and "Greedy is a different code path".
//
// Design (two launches per call, on the caller's stream):
//   * stats_kernel - every logit of the batch is read from HBM once.  The chunks of all rows,
//     end to end, are cut into equal contiguous shares, one per warp of a persistent grid.
//     Each warp streams its share through a ring of shared-memory stages filled by TMA bulk
//     copies (one elected lane, one mbarrier per stage, bounded waits).  Each lane keeps, per
//     row piece, s = sum 2^(l a - K) against an integer reference K (a = log2(e)/T carried as
//     a_hi + a_lo, so every exponent is two FMAs with one rounding and the temperature is exact
//     to ~1e-14).  A full stage is taken at once: its maximum raises K at most once, then its
//     terms are independent and enter a Kahan sum once; NaN and +inf poison the row.  Greedy
//     rows keep the maximum and its lowest index instead.  One partial per (row, piece);
//     after writing it the warp adds 1 to the row's counter in the workspace (release).
//   * verify_kernel - one thread-block cluster of C CTAs per stream, launched with
//     programmatic dependent launch: its prologue (offsets, temperature, tokens, the logits
//     at the tokens, the uniforms) overlaps the stats kernel's tail, and each stream reads a
//     row's partials as soon as that row's counter (acquire, bounded wait) shows all its
//     pieces, so streams whose rows are done start while other rows are still being read; the
//     counters go back to zero when the stream is done.  Every CTA reduces the stream's
//     partials in the same order, so all hold bit-identical row statistics and take the same
//     decisions without communicating;
//     the per-stream scalars (rho, the running product w, h) are double-float on the float32
//     pipes.  CTA c owns a contiguous vocabulary slice of every row, one segment per warp.
//   * block verification: h_N = w_N needs no residual; slot i < N is a candidate only if
//     eta_i <= w_i (since h_i <= w_i); the residual masses of all candidates and of slot 0 are
//     computed in one cluster-wide sweep (a second read, partly from L2), then tau = the
//     largest candidate with eta_i <= h_i, else 0.  The token-wise rule needs one residual (at
//     tau); when every draft is accepted the sweep sums the bonus row p_N instead;
//   * the draw: a 64-bit fixed-point CDF over the segments (exact integer prefix sums through
//     distributed shared memory), then the CTA that owns the segment holding U*R sums its eight
//     warp slices in the same fixed point, and the warp whose slice crosses the target rescans
//     it and writes the token.  CTAs arrive at the final cluster barrier as soon as their last
//     distributed-shared-memory read is done, so the others do not wait for the rescan.

#include <cooperative_groups.h>

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "df.cuh"
#include "host_util.h"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxRows = 2 * SPEC_MAX_KMAX + 1;
constexpr int kRingBytesPerCta = 56 * 1024;
constexpr float kNoRef = -1e30f;     // reference of a lane that has seen no finite logit
constexpr int kPiecesMax = 64;       // stats partials per row

struct Part;

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
    int64_t nchunk;      // chunks of 8 (or 1) elements per row
    int64_t seg_chunks;  // chunks per warp segment of the cluster kernel's residual sweep
    char* ws;            // workspace: one block of kRowBytes per stats row (see row_block)
    int64_t stats_warps; // warps of the stats kernel's grid
};

// Per-warp partial of one row.  T > 0: K = integer reference, (s_hi, s_lo) = sum 2^(l a - K).
// T = 0: K = the segment maximum, idx = its lowest index.
struct Part {
    float K;
    float s_hi, s_lo;
    int idx;
};

// Workspace: stats row rho owns bytes [rho kRowBytes, (rho + 1) kRowBytes): a 32-bit counter
// of published partials (in a 16-byte slot), then its kPiecesMax partials.  A row's block sits
// at the same place for every batch size, and each call leaves the counters of the rows it
// used at zero, so a zero-filled workspace stays valid from call to call.  A stream has at
// most 2 kmax + 1 rows.
constexpr size_t kRowBytes = 16 + kPiecesMax * sizeof(Part);
static size_t workspace_rows(int32_t B, int32_t kmax) { return (size_t)B * (size_t)(2 * kmax + 1); }
static size_t workspace_bytes(int32_t B, int32_t kmax) { return workspace_rows(B, kmax) * kRowBytes; }
__device__ __forceinline__ unsigned* row_counter(const VerifyParams& p, int64_t rho) {
    return reinterpret_cast<unsigned*>(p.ws + rho * (int64_t)kRowBytes);
}
__device__ __forceinline__ Part* row_parts(const VerifyParams& p, int64_t rho) {
    return reinterpret_cast<Part*>(p.ws + rho * (int64_t)kRowBytes + 16);
}

struct Shared {
    float res_part[SPEC_MAX_KMAX + 1][kWarps];
    float rowK[kMaxRows];
    df rowZ[kMaxRows];
    int rowArg[kMaxRows];
    df rho[SPEC_MAX_KMAX];
    df w[SPEC_MAX_KMAX + 1];
    df h[SPEC_MAX_KMAX + 1];
    df r[SPEC_MAX_KMAX + 1];
    df u_acc[SPEC_MAX_KMAX + 1];
    uint32_t u_smp[SPEC_MAX_KMAX + 1];
    float cval[SPEC_MAX_KMAX + 1];     // residual weight scale w_i Z_q / Z_p per slot
    float lq[SPEC_MAX_KMAX], lp[SPEC_MAX_KMAX];
    int x[SPEC_MAX_KMAX];
    int pass_list[SPEC_MAX_KMAX + 1];
    int n_pass;
    int to_flag[kWarps];            // a bounded wait of this warp gave up
    int N, status, greedy, tau, sample_seg, sample_bonus;
    unsigned long long sample_t;   // in-segment target (fixed point)
    unsigned long long sub_sum[kWarps];   // the drawn segment split over the owning CTA's warps
    int sub_last[kWarps];
    float sample_scale;            // fixed-point scale of the draw's weights
    float a_hi, a_lo;
};

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    cluster_arrive();
    cluster_wait();
}

// ---------------------------------------------------------------------------------------
// Chunk feeds.  A stage is U chunks per lane of up to two rows (q and p): lane L of a warp
// takes chunks rel + u*32 + L, u < U.  The vector path (E = 8, 16-byte aligned rows) moves a
// stage with one TMA bulk copy per row into a per-warp shared-memory ring of D stages, each
// completing on its own mbarrier (one elected lane issues, every lane waits with a bounded
// poll); the plain path (E = 1) loads directly.
// ---------------------------------------------------------------------------------------
constexpr int kSpinLimit = 1 << 20;   // mbarrier polls before a wait gives up (status TIMEOUT)

// Row counters: a stats warp publishes a partial, then adds 1 to its row's counter with
// release semantics; a verify CTA reads the partials of a row once the counter (read with
// acquire semantics) equals the row's piece count.  The wait gives up after kRowWaitNs of
// device time (or a value above the count, which only a non-zero workspace can hold).
constexpr unsigned long long kRowWaitNs = 4000000000ull;

__device__ __forceinline__ void count_release(unsigned* c) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
}
__device__ __forceinline__ unsigned load_acquire(const unsigned* c) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool wait_count(const unsigned* c, unsigned want) {
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < (1 << 26); ++it) {
        const unsigned v = load_acquire(c);
        if (v == want) return true;
        if (v > want || global_ns() - t0 > kRowWaitNs) return false;
        __nanosleep(64);
    }
    return false;
}

template <typename DQ, typename DP, int E>
struct Feed;

template <typename DQ, typename DP>
struct Feed<DQ, DP, 8> {
    static constexpr int BQ = 8 * (int)sizeof(DQ);
    static constexpr int BP = 8 * (int)sizeof(DP);
    static constexpr int U = (2 * 32 * (BQ + BP) <= 2048) ? 2 : 1;
    static constexpr int GRP = 32 * U;                       // chunks per stage
    static constexpr int ROWQ = GRP * BQ, ROWP = GRP * BP;
    static constexpr int STAGE = ROWQ + ROWP;
    static constexpr int DR = (kRingBytesPerCta / kWarps - 64) / STAGE;
    static constexpr int D = DR < 2 ? 2 : (DR > 8 ? 8 : DR);
    static constexpr int RING = D * STAGE + 64;              // bytes per warp (stages + barriers)
    char* base;
    uint64_t* bar;
    int lane;
    unsigned phase;     // parity of the next completion of each slot
    unsigned pending;   // slots with a stage issued and not yet waited for
    bool timeout;
    __device__ __forceinline__ void init(char* b, int ln) {
        base = b;
        bar = reinterpret_cast<uint64_t*>(b + D * STAGE);
        lane = ln;
        phase = 0;
        pending = 0;
        timeout = false;
        if (lane == 0) {
            for (int i = 0; i < D; ++i) mbar_init(&bar[i], 1);
            mbar_init_fence();
        }
        __syncwarp();
    }
    // segment start of a row (bytes), or null
    __device__ __forceinline__ const char* seg_q(const void* row, int64_t c0) const {
        return row ? reinterpret_cast<const char*>(row) + c0 * BQ : nullptr;
    }
    __device__ __forceinline__ const char* seg_p(const void* row, int64_t c0) const {
        return reinterpret_cast<const char*>(row) + c0 * BP;
    }
    // stage of chunks [rel, rel + GRP) of the segment (nrel chunks long) into ring slot `slot`
    __device__ __forceinline__ void issue(int slot, const char* gq, const char* gp, int rel, int nrel) {
        if (timeout) return;   // after a failed wait nothing new is put in flight
        pending |= 1u << slot;
        __syncwarp();          // every lane is done reading this slot's previous stage
        if (lane == 0) {
            const int n = min(GRP, nrel - rel);
            fence_proxy_async_smem();
            mbar_expect_tx(&bar[slot], (unsigned)(n * ((gq ? BQ : 0) + BP)));
            if (gq) bulk_g2s(base + slot * STAGE, gq + (size_t)rel * BQ, (unsigned)(n * BQ), &bar[slot]);
            bulk_g2s(base + slot * STAGE + ROWQ, gp + (size_t)rel * BP, (unsigned)(n * BP), &bar[slot]);
        }
    }
    __device__ __forceinline__ void wait(int slot) {
        if (timeout) return;
        const unsigned parity = (phase >> slot) & 1u;
        int n = 0;
        while (!mbar_try_wait(&bar[slot], parity)) {
            if (++n > kSpinLimit) {
                timeout = true;   // the slot stays pending; drain() waits for it once more
                return;
            }
        }
        phase ^= 1u << slot;
        pending &= ~(1u << slot);
    }
    // before the CTA exits: wait (bounded) for any copy still in flight after a failed wait
    __device__ __forceinline__ void drain() {
        for (int slot = 0; slot < D; ++slot) {
            if (!((pending >> slot) & 1u)) continue;
            const unsigned parity = (phase >> slot) & 1u;
            for (int n = 0; n < kSpinLimit && !mbar_try_wait(&bar[slot], parity); ++n) {
            }
        }
    }
    __device__ __forceinline__ void get(int slot, int u, const void*, const void*, int64_t, bool has_q,
                                        float (&xq)[8], float (&xp)[8]) const {
        const char* sq = base + slot * STAGE + (u * 32 + lane) * BQ;
        const char* sp = base + slot * STAGE + ROWQ + (u * 32 + lane) * BP;
        if (has_q) unpack<DQ>(sq, xq);
        unpack<DP>(sp, xp);
    }
    template <typename T>
    __device__ __forceinline__ static void unpack(const char* s, float (&x)[8]) {
        if (sizeof(T) == 2) {
            const uint4 v = *reinterpret_cast<const uint4*>(s);
            x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
            x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
        } else {
            const float4 a = *reinterpret_cast<const float4*>(s);
            const float4 b = *reinterpret_cast<const float4*>(s + 16);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
    }
};

template <typename DQ, typename DP>
struct Feed<DQ, DP, 1> {
    static constexpr int U = 4;
    static constexpr int GRP = 32 * U;
    static constexpr int D = 1;
    static constexpr int RING = 0;
    int lane;
    bool timeout;
    __device__ __forceinline__ void init(char*, int ln) {
        lane = ln;
        timeout = false;
    }
    __device__ __forceinline__ const char* seg_q(const void*, int64_t) const { return nullptr; }
    __device__ __forceinline__ const char* seg_p(const void*, int64_t) const { return nullptr; }
    __device__ __forceinline__ void issue(int, const char*, const char*, int, int) {}
    __device__ __forceinline__ void wait(int) {}
    __device__ __forceinline__ void drain() {}
    __device__ __forceinline__ void get(int, int, const void* rq, const void* rp, int64_t k, bool has_q,
                                        float (&xq)[1], float (&xp)[1]) const {
        if (has_q) xq[0] = load_elem<DQ>(rq, k);
        xp[0] = load_elem<DP>(rp, k);
    }
};

// ---------------------------------------------------------------------------------------
// Per-lane accumulators
// ---------------------------------------------------------------------------------------
// Kahan-compensated running sum of chunk sums: the true sum is s - c.  Accumulating one
// float per chunk against a large running total would otherwise lose ~3e-8 of the total per
// addition when one token dominates the row.
struct Kahan {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float t) {
        const float y = __fsub_rn(t, c);
        const float u = __fadd_rn(s, y);
        c = __fsub_rn(__fsub_rn(u, s), y);
        s = u;
    }
    __device__ __forceinline__ df value() const { return fast_two_sum(s, -c); }
    __device__ __forceinline__ void scale(float f) {
        s *= f;
        c *= f;
    }
};

// sum 2^(x a - K) of one lane (T > 0 rows), with the reference K raised only when needed
struct LaneSum {
    float K = kNoRef;
    Kahan acc;

    template <int G>
    __device__ __forceinline__ float terms(const float (&x)[G], float ah, float al) const {
        if constexpr (G == 1) {
            return ex2(fmaf(x[0], al, fmaf(x[0], ah, -K)));
        } else {
            const float2 nk = make_float2(-K, -K), a2h = make_float2(ah, ah), a2l = make_float2(al, al);
            float2 e[G / 2];
#pragma unroll
            for (int j = 0; j < G / 2; ++j) {
                const float2 z = ffma2(make_float2(x[2 * j], x[2 * j + 1]), a2l,
                                       ffma2(make_float2(x[2 * j], x[2 * j + 1]), a2h, nk));
                e[j] = make_float2(ex2(z.x), ex2(z.y));
            }
#pragma unroll
            for (int w = G / 2; w > 1; w /= 2)
#pragma unroll
                for (int j = 0; j < w / 2; ++j) e[j] = fadd2(e[j], e[j + w / 2]);
            return e[0].x + e[0].y;
        }
    }
    // The fast path keeps every term of the load <= 16, i.e. its exponent x a - K <= 4, where
    // float32 rounds the exponent to 1.2e-7 (2^e to ~8e-8); a load with a larger sum (a new
    // maximum more than 4 above K, the first finite load, +inf or NaN) raises K to
    // ceil(max x a) and is recomputed.
    template <int G>
    __device__ __forceinline__ void add(const float (&x)[G], float ah, float al) {
        float t;
        for (int pass = 0;; ++pass) {   // one copy of the terms: the retry is rare
            t = terms<G>(x, ah, al);
            if (t <= 16.f || pass > 0) break;
            float vm = x[0];
#pragma unroll
            for (int j = 1; j < G; ++j) vm = fmaxf(vm, x[j]);   // NaN-ignoring
            const float kv = ceilf(vm * ah);
            if (kv > K) {
                acc.scale(pow2_int(K - kv));
                K = kv;
            }
        }
        acc.add(t);                     // NaN / inf stay and poison the row
    }
    // A group of U full chunks (x[u] = chunk u of this lane).  The group's maximum comes first,
    // the reference is raised at most once, and then all 8 U terms are independent: they are
    // summed as packed pairs and enter the Kahan sum once.  Every term stays <= 16 (exponent
    // <= 4), as in the per-chunk form, but without a data-dependent branch per chunk.
    template <int U>
    __device__ __forceinline__ void add_group(const float (&x)[U][8], float ah, float al) {
        float m = -kInf;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < 8; j += 2) m = fmax_nan(m, fmax_nan(x[u][j], x[u][j + 1]));
        if (!(m * ah <= K + 4.f)) {   // a new maximum (or NaN, which then poisons the sum)
            const float kv = ceilf(m * ah);
            if (kv > K) {
                acc.scale(pow2_int(K - kv));
                K = kv;
            }
        }
        const float2 nk = make_float2(-K, -K), a2h = make_float2(ah, ah), a2l = make_float2(al, al);
        float2 s4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 xx = make_float2(x[u][2 * j], x[u][2 * j + 1]);
                const float2 z = ffma2(xx, a2l, ffma2(xx, a2h, nk));
                s4[j] = fadd2(s4[j], make_float2(ex2(z.x), ex2(z.y)));
            }
        const float2 t = fadd2(fadd2(s4[0], s4[1]), fadd2(s4[2], s4[3]));
        acc.add(t.x + t.y);
    }
    // warp-combine and publish (lane 0)
    __device__ __forceinline__ void publish(Part* dst, int lane) const {
        const float Kw = warp_max(K);
        df sum = df_scale(acc.value(), K == Kw ? 1.f : pow2_int(K - Kw));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const df other{__shfl_xor_sync(0xffffffffu, sum.hi, o), __shfl_xor_sync(0xffffffffu, sum.lo, o)};
            sum = df_add(sum, other);
        }
        if (lane == 0) *dst = Part{Kw, sum.hi, sum.lo, INT_MAX};
    }
};

// max and its lowest index (T = 0 rows); NaN propagates
struct LaneMax {
    float m = -kInf;
    int idx = INT_MAX;
    template <int G>
    __device__ __forceinline__ void add(const float (&x)[G], int64_t elem0) {
        float vm = x[0];
#pragma unroll
        for (int j = 1; j < G; ++j) vm = fmax_nan(vm, x[j]);
        if (!(vm <= m)) {
            int j0 = 0;
#pragma unroll
            for (int j = G - 1; j >= 0; --j)
                if (x[j] == vm) j0 = j;
            idx = (int)(elem0 + j0);
            m = fmax_nan(m, vm);
        }
    }
    __device__ __forceinline__ void publish(Part* dst, int lane) const {
        const float mw = warp_max_nan(m);
        const int iw = warp_min_i((m == mw) ? idx : INT_MAX);
        if (lane == 0) *dst = Part{mw, 0.f, 0.f, iw};
    }
};

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

// sum of a chunk's residual weights (pairwise, packed)
template <int E>
__device__ __forceinline__ float resid_chunk_sum(const float (&xq)[E], const float (&xp)[E], float Kq, float Kp,
                                                 float ah, float al, float c) {
    if constexpr (E == 1) {
        float w[1];
        resid_weights<1>(xq, xp, Kq, Kp, ah, al, c, w);
        return w[0];
    } else {
        const float2 a2h = make_float2(ah, ah), a2l = make_float2(al, al);
        const float2 nkp = make_float2(-Kp, -Kp), nkq = make_float2(-Kq, -Kq);
        float2 d[E / 2];
#pragma unroll
        for (int j = 0; j < E / 2; ++j) {
            const float2 pp = make_float2(xp[2 * j], xp[2 * j + 1]);
            const float2 qq = make_float2(xq[2 * j], xq[2 * j + 1]);
            const float2 e1 = ffma2(pp, a2l, ffma2(pp, a2h, nkp));
            const float2 e2 = ffma2(qq, a2l, ffma2(qq, a2h, nkq));
            d[j] = make_float2(fmaxf(0.f, fmaf(c, ex2(e1.x), -ex2(e2.x))), fmaxf(0.f, fmaf(c, ex2(e1.y), -ex2(e2.y))));
        }
#pragma unroll
        for (int w = E / 2; w > 1; w /= 2)
#pragma unroll
            for (int j = 0; j < w / 2; ++j) d[j] = fadd2(d[j], d[j + w / 2]);
        return d[0].x + d[0].y;
    }
}

// sum of a chunk's target weights 2^(xp a - Kp) (the bonus slot's distribution)
template <int E>
__device__ __forceinline__ float target_chunk_sum(const float (&xp)[E], float Kp, float ah, float al) {
    LaneSum t;
    t.K = Kp;
    return t.terms<E>(xp, ah, al);
}

// ---------------------------------------------------------------------------------------
// Warp sweep over this warp's segment [c0, c1) of a list of items (a row or a row pair),
// each split into groups of U * 32 chunks; the ring runs D - 1 groups ahead of the consumer.
// rows(it, rq, rp) gives an item's rows; begin(it) / consume(k, xq, xp) / end(it) see the
// items in order.
// ---------------------------------------------------------------------------------------
template <typename DQ, typename DP, int E, typename RowsFn, typename BeginFn, typename ConsumeFn, typename EndFn,
          typename FlushFn>
__device__ __forceinline__ void sweep(Feed<DQ, DP, E>& feed, int items, int64_t c0, int64_t c1, int lane,
                                      RowsFn rows, BeginFn begin_item, ConsumeFn consume, EndFn end_item,
                                      FlushFn flush) {
    constexpr int D = Feed<DQ, DP, E>::D;
    constexpr int U = Feed<DQ, DP, E>::U;
    const int G = (c1 > c0) ? (int)((c1 - c0 + 32 * U - 1) / (32 * U)) : 0;
    const int nrel = (int)(c1 - c0);
    int ii = 0, gi = 0, slot_i = 0;
    const char *iq = nullptr, *ip = nullptr;
    auto load_rows = [&](int it) {
        const void *rq, *rp;
        rows(it, rq, rp);
        iq = feed.seg_q(rq, c0);
        ip = feed.seg_p(rp, c0);
    };
    if (G > 0 && items > 0) load_rows(0);
    auto issue_next = [&]() {
        if (ii < items) feed.issue(slot_i, iq, ip, gi * 32 * U, nrel);
        if (++slot_i == D) slot_i = 0;
        if (++gi == G) {
            gi = 0;
            ++ii;
            if (ii < items) load_rows(ii);
        }
    };
    if (G > 0)
        for (int s = 0; s < D - 1; ++s) issue_next();
    int slot_c = 0;
    for (int it = 0; it < items; ++it) {
        const void *cq, *cp;
        rows(it, cq, cp);
        begin_item(it);
        for (int g = 0; g < G; ++g) {
            issue_next();
            feed.wait(slot_c);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t k = c0 + ((int64_t)g * U + u) * 32 + lane;
                if (k < c1) {
                    float xq[E], xp[E];
                    feed.get(slot_c, u, cq, cp, k, cq != nullptr, xq, xp);
                    consume(k, xq, xp);
                }
            }
            flush();   // one group of chunks done
            if (++slot_c == D) slot_c = 0;
        }
        end_item(it);
    }
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
                                           int lane) {
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
                if (!BONUS) cq[u].load(rq, k);
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

// Fixed-point sum (weights times `scale`) of the chunks [k0, k1) and their last positive
// element, over the warp (every lane returns both).
template <typename DQ, typename DP, int E, bool BONUS>
__device__ __noinline__ void segment_fixed_sum(const void* rq, const void* rp, int64_t k0, int64_t k1, float Kq,
                                               float Kp, float ah, float al, float c, float scale, int lane,
                                               unsigned long long& sum, int& last) {
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
                if (!BONUS) cq[u].load(rq, k);
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

// stream j breaks the packed layout: its draft count is outside [0, kmax], or cu[0] != 0
__device__ __forceinline__ bool offsets_bad(const VerifyParams& p, int j) {
    const int n = p.cu[j + 1] - p.cu[j];
    return n < 0 || n > p.kmax || (j == 0 && p.cu[0] != 0);
}

// Streams [0, L) form the valid packed prefix (cu[0] = 0, every count in [0, kmax]); returns
// L.  Every thread of the block must call it.
__device__ int valid_prefix(const VerifyParams& p) {
    __shared__ int first_bad;
    if (threadIdx.x == 0) first_bad = p.B;
    __syncthreads();
    for (int j = threadIdx.x; j < p.B; j += blockDim.x)
        if (offsets_bad(p, j)) atomicMin(&first_bad, j);
    __syncthreads();
    const int L = first_bad;
    __syncthreads();
    return L;
}

// Chunks per warp of the stats kernel: equal shares of all rows' chunks, but at least
// ceil(n / (kPiecesMax - 2)) so that no row is cut into more than kPiecesMax pieces.
__device__ __forceinline__ int64_t stats_share(int64_t rows, int64_t n, int64_t nw) {
    const int64_t lw = (rows * n + nw - 1) / nw;
    const int64_t lmin = (n + kPiecesMax - 3) / (kPiecesMax - 2);
    return lw > lmin ? lw : (lmin > 0 ? lmin : 1);
}

// ---------------------------------------------------------------------------------------
// Stats kernel: every logit of the batch is read once.
//
// Rows are numbered stream by stream: stream b owns rows [g_b, g_b + 2 N_b + 1), g_b =
// 2 cu[b] + b; its target rows 0..N_b come first, then its draft rows 0..N_b-1.  The chunks
// of all these rows, end to end, are cut into equal contiguous shares, one per warp of a
// persistent grid, so every warp streams the same number of bytes, from one row or a few
// consecutive ones.  Per row piece a warp leaves one partial: (reference K, sum 2^(l a - K))
// for T > 0, (max, lowest argmax) for T = 0; the partial of piece k of row rho sits at
// rho * kPiecesMax + k.  Draft rows of greedy streams and all rows of a stream with an
// invalid temperature are skipped (never read).
// ---------------------------------------------------------------------------------------
template <typename T, int E, typename AddFn>
__device__ __forceinline__ void stream_piece(const void* row, int64_t c0, int64_t c1, int lane, AddFn add) {
    constexpr int U = (E == 8) ? (sizeof(T) == 2 ? 4 : 2) : 8;   // 64 bytes per lane and batch
    constexpr int G = 32 * U;
    Chunk<T, E> a[U], b[U];
    auto load = [&](Chunk<T, E>(&v)[U], int64_t base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) v[u].load(row, k);
        }
    };
    auto consume = [&](const Chunk<T, E>(&v)[U], int64_t base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = base + u * 32 + lane;
            if (k < c1) {
                float x[E];
                v[u].unpack(x);
                add(x, k * E);
            }
        }
    };
    // two register buffers: the next batch is in flight while the current one is summed
    load(a, c0);
    for (int64_t k = c0; k < c1; k += 2 * G) {
        if (k + G < c1) load(b, k + G);
        consume(a, k);
        if (k + G >= c1) break;
        if (k + 2 * G < c1) load(a, k + 2 * G);
        consume(b, k + G);
    }
}

// 16-byte rows (E = 8): each lane copies its own chunks into a per-warp ring of kStages
// stages of 2 KB with cp.async and later reads back only those chunks, so the ring needs no
// synchronisation beyond each thread's own wait_group; kStages - 1 stages are in flight while
// one is summed.  A float32 chunk (32 bytes) is stored as two 16-byte planes.
constexpr int kStages = 4;
constexpr int kStageBytes = 2048;
constexpr int kStatsRingBytes = kWarps * kStages * kStageBytes;
static size_t stats_smem_bytes(int E) { return E == 8 ? (size_t)kStatsRingBytes : 0; }

template <typename T, typename AddFn, typename GroupFn>
__device__ __forceinline__ void stream_piece_ring(char* ring, const void* row, int64_t c0, int64_t c1, int lane,
                                                  AddFn add, GroupFn add_full) {
    constexpr int BT = 8 * (int)sizeof(T);   // bytes per chunk
    constexpr int G = kStageBytes / BT;      // chunks per stage
    constexpr int U = G / 32;                // chunks per lane and stage
    constexpr int LPC = BT / 16;             // 16-byte copies per chunk
    const char* g = reinterpret_cast<const char*>(row);
    const int64_t nb = (c1 - c0 + G - 1) / G;
    auto issue = [&](int64_t i, int slot) {
        if (i < nb) {
            char* st = ring + slot * kStageBytes;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t k = c0 + i * G + u * 32 + lane;
                if (k < c1)
#pragma unroll
                    for (int l = 0; l < LPC; ++l) cp_async16(st + l * (G * 16) + (u * 32 + lane) * 16, g + k * BT + 16 * l);
            }
        }
        cp_async_commit();   // an empty group keeps the group count in step
    };
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) issue(i, i);
    int slot = 0;
    for (int64_t i = 0; i < nb; ++i) {
        issue(i + kStages - 1, slot == 0 ? kStages - 1 : slot - 1);
        cp_async_wait<kStages - 1>();
        const char* st = ring + slot * kStageBytes;
        if (c0 + (i + 1) * G <= c1) {   // a full stage: every lane has all U chunks
            float x[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if constexpr (sizeof(T) == 2) {
                    const uint4 v = *reinterpret_cast<const uint4*>(st + (u * 32 + lane) * 16);
                    x[u][0] = bf16_lo(v.x); x[u][1] = bf16_hi(v.x); x[u][2] = bf16_lo(v.y); x[u][3] = bf16_hi(v.y);
                    x[u][4] = bf16_lo(v.z); x[u][5] = bf16_hi(v.z); x[u][6] = bf16_lo(v.w); x[u][7] = bf16_hi(v.w);
                } else {
                    const float4 a = *reinterpret_cast<const float4*>(st + (u * 32 + lane) * 16);
                    const float4 b = *reinterpret_cast<const float4*>(st + G * 16 + (u * 32 + lane) * 16);
                    x[u][0] = a.x; x[u][1] = a.y; x[u][2] = a.z; x[u][3] = a.w;
                    x[u][4] = b.x; x[u][5] = b.y; x[u][6] = b.z; x[u][7] = b.w;
                }
            }
            add_full(x, c0 + i * G + lane);
            slot = (slot + 1 == kStages) ? 0 : slot + 1;
            continue;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = c0 + i * G + u * 32 + lane;
            if (k < c1) {
                float x[8];
                if constexpr (sizeof(T) == 2) {
                    const uint4 v = *reinterpret_cast<const uint4*>(st + (u * 32 + lane) * 16);
                    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
                    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
                } else {
                    const float4 a = *reinterpret_cast<const float4*>(st + (u * 32 + lane) * 16);
                    const float4 b = *reinterpret_cast<const float4*>(st + G * 16 + (u * 32 + lane) * 16);
                    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
                }
                add(x, k * 8);
            }
        }
        slot = (slot + 1 == kStages) ? 0 : slot + 1;
    }
}

// The stats kernel's per-warp ring: kStages stages of kStageBytes in shared memory, each
// filled by one TMA bulk copy (issued by lane 0) that completes on the stage's mbarrier; every
// lane waits with a bounded poll.  One instruction per stage moves the data, so the scan's
// issue slots go to the arithmetic.  Slots and phases persist from piece to piece.
struct StatsRing {
    char* base;
    uint64_t* bar;
    int lane;
    unsigned phase;     // parity of the next completion of each slot
    unsigned pending;   // slots with a copy issued and not yet waited for
    bool timeout;
    __device__ __forceinline__ void init(char* b, uint64_t* bars, int ln) {
        base = b;
        bar = bars;
        lane = ln;
        phase = 0;
        pending = 0;
        timeout = false;
        if (lane == 0) {
            for (int i = 0; i < kStages; ++i) mbar_init(&bar[i], 1);
            mbar_init_fence();
        }
        __syncwarp();
    }
    __device__ __forceinline__ void issue(int slot, const char* src, unsigned bytes) {
        if (timeout) return;   // after a failed wait nothing new is put in flight
        pending |= 1u << slot;
        __syncwarp();          // every lane is done with this slot's previous contents
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&bar[slot], bytes);
            bulk_g2s(base + slot * kStageBytes, src, bytes, &bar[slot]);
        }
    }
    __device__ __forceinline__ void wait(int slot) {
        if (timeout) return;
        const unsigned parity = (phase >> slot) & 1u;
        int n = 0;
        while (!mbar_try_wait(&bar[slot], parity)) {
            if (++n > kSpinLimit) {
                timeout = true;   // the slot stays pending; drain() waits for it once more
                return;
            }
        }
        phase ^= 1u << slot;
        pending &= ~(1u << slot);
    }
    __device__ __forceinline__ void drain() {
        for (int slot = 0; slot < kStages; ++slot) {
            if (!((pending >> slot) & 1u)) continue;
            const unsigned parity = (phase >> slot) & 1u;
            for (int n = 0; n < kSpinLimit && !mbar_try_wait(&bar[slot], parity); ++n) {
            }
        }
    }
};

// One piece [c0, c1) of a 16-byte aligned row through the bulk ring: full stages go to
// add_full (U chunks per lane), the ragged last stage chunk by chunk to add.
template <typename T, typename AddFn, typename GroupFn>
__device__ __forceinline__ void stream_piece_bulk(StatsRing& R, const void* row, int64_t c0, int64_t c1, int lane,
                                                  AddFn add, GroupFn add_full) {
    constexpr int BT = 8 * (int)sizeof(T);   // bytes per chunk
    constexpr int G = kStageBytes / BT;      // chunks per stage
    constexpr int U = G / 32;                // chunks per lane and stage
    const char* g = reinterpret_cast<const char*>(row) + c0 * BT;
    const int64_t n = c1 - c0;
    const int nb = (int)((n + G - 1) / G);
    auto issue = [&](int i) {
        if (i < nb) R.issue(i % kStages, g + (int64_t)i * G * BT, (unsigned)(min((int64_t)G, n - (int64_t)i * G) * BT));
    };
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) issue(i);
    for (int i = 0; i < nb; ++i) {
        issue(i + kStages - 1);
        const int slot = i % kStages;
        R.wait(slot);
        const char* st = R.base + slot * kStageBytes;
        if ((int64_t)(i + 1) * G <= n) {   // a full stage: every lane has all U chunks
            float x[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const char* c = st + (u * 32 + lane) * BT;
                if constexpr (sizeof(T) == 2) {
                    const uint4 v = *reinterpret_cast<const uint4*>(c);
                    x[u][0] = bf16_lo(v.x); x[u][1] = bf16_hi(v.x); x[u][2] = bf16_lo(v.y); x[u][3] = bf16_hi(v.y);
                    x[u][4] = bf16_lo(v.z); x[u][5] = bf16_hi(v.z); x[u][6] = bf16_lo(v.w); x[u][7] = bf16_hi(v.w);
                } else {
                    const float4 a = *reinterpret_cast<const float4*>(c);
                    const float4 b = *reinterpret_cast<const float4*>(c + 16);
                    x[u][0] = a.x; x[u][1] = a.y; x[u][2] = a.z; x[u][3] = a.w;
                    x[u][4] = b.x; x[u][5] = b.y; x[u][6] = b.z; x[u][7] = b.w;
                }
            }
            add_full(x, c0 + (int64_t)i * G + lane);
        } else {
            const int cnt = (int)(n - (int64_t)i * G);
            for (int kk = lane; kk < cnt; kk += 32) {
                float x[8];
                const char* c = st + kk * BT;
                if constexpr (sizeof(T) == 2) {
                    const uint4 v = *reinterpret_cast<const uint4*>(c);
                    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
                    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
                } else {
                    const float4 a = *reinterpret_cast<const float4*>(c);
                    const float4 b = *reinterpret_cast<const float4*>(c + 16);
                    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
                }
                add(x, (c0 + (int64_t)i * G + kk) * 8);
            }
        }
    }
}

constexpr int kStatsTimeout = -2;   // idx of a partial whose stats piece lost a bounded wait

template <typename T, int E>
__device__ __forceinline__ void stats_piece(StatsRing& ring, const void* row, int64_t c0, int64_t c1, bool greedy,
                                            float ah, float al, int lane, Part* dst) {
    constexpr int UG = kStageBytes / (8 * (int)sizeof(T)) / 32;   // chunks per lane and stage
    if (greedy) {
        LaneMax mx;
        auto f = [&](const float (&x)[E], int64_t e0) { mx.add<E>(x, e0); };
        // chunk u of the group is chunk k0 + 32 u of the row (this lane's chunks, ascending)
        auto g = [&](const float (&x)[UG][8], int64_t k0) {
#pragma unroll
            for (int u = 0; u < UG; ++u) mx.add<8>(x[u], (k0 + 32 * u) * 8);
        };
        if constexpr (E == 8) stream_piece_bulk<T>(ring, row, c0, c1, lane, f, g);
        else stream_piece<T, E>(row, c0, c1, lane, f);
        mx.publish(dst, lane);
        if (ring.timeout && lane == 0) dst->idx = kStatsTimeout;
    } else {
        LaneSum sum;
        auto f = [&](const float (&x)[E], int64_t) { sum.add<E>(x, ah, al); };
        auto g = [&](const float (&x)[UG][8], int64_t) { sum.add_group<UG>(x, ah, al); };
        if constexpr (E == 8) stream_piece_bulk<T>(ring, row, c0, c1, lane, f, g);
        else stream_piece<T, E>(row, c0, c1, lane, f);
        sum.publish(dst, lane);
        if (ring.timeout && lane == 0) dst->idx = kStatsTimeout;
    }
}

template <typename DQ, typename DP, int E>
__global__ void __launch_bounds__(kThreads, 3) stats_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) char stats_smem[];
    // the verify kernel may be scheduled now: it reads a row's partials once its counter is full
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ __align__(8) uint64_t stats_bars[kWarps][kStages];
    const int lane = threadIdx.x & 31;
    StatsRing ring;
    ring.init(stats_smem + (threadIdx.x >> 5) * (kStages * kStageBytes), stats_bars[threadIdx.x >> 5], lane);
    const int L = valid_prefix(p);
    if (L == 0) return;
    const int64_t n = p.nchunk;
    const int64_t rows = 2 * (int64_t)p.cu[L] + L;
    const int64_t lw = stats_share(rows, n, p.stats_warps);
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    int64_t f = gw * lw;
    const int64_t f1 = min(f + lw, rows * n);
    if (f >= f1) return;
    int64_t rho = f / n;
    int64_t c = f - rho * n;
    // the stream of the first row: largest b in [0, L) with g_b <= rho
    int lo = 0, hi = L - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (2 * (int64_t)p.cu[mid] + mid <= rho) lo = mid;
        else hi = mid - 1;
    }
    int b = lo;
    int64_t gb = 2 * (int64_t)p.cu[b] + b;
    int Nb = p.cu[b + 1] - p.cu[b];
    const int64_t V = p.V;
    while (f < f1) {
        const int64_t c_end = min(n, c + (f1 - f));
        while (rho - gb > 2 * (int64_t)Nb) {
            ++b;
            gb = 2 * (int64_t)p.cu[b] + b;
            Nb = p.cu[b + 1] - p.cu[b];
        }
        const int64_t j = rho - gb;
        const float T = p.temp[b];
        const bool greedy = (T == 0.f);
        const bool draft = j > Nb;
        const bool skip = !(isfinite(T) && (T == 0.f || T >= FLT_MIN)) || (draft && greedy);
        if (!skip) {
            float ah = 0.f, al = 0.f;
            if (!greedy) {
                const df l2e{1.4426950216293335f, 1.925963033500011e-08f};
                const df a = df_div(l2e, df_make(T));
                ah = a.hi;
                al = a.lo;
            }
            Part* dst = row_parts(p, rho) + (gw - rho * n / lw);
            if (draft)
                stats_piece<DQ, E>(ring, row_ptr<DQ>(p.dq, (int64_t)p.cu[b] + (j - Nb - 1), V), c, c_end, false,
                                   ah, al, lane, dst);
            else
                stats_piece<DP, E>(ring, row_ptr<DP>(p.dp, (int64_t)p.cu[b] + b + j, V), c, c_end, greedy, ah, al,
                                   lane, dst);
            if (lane == 0) count_release(row_counter(p, rho));   // lane 0 wrote the partial
        }
        f += c_end - c;
        c = 0;
        ++rho;
    }
    // no TMA copy of this warp may still be writing its ring when the CTA leaves
    ring.drain();
}

// ---------------------------------------------------------------------------------------
// The verify kernel (one cluster per stream)
// ---------------------------------------------------------------------------------------
template <typename DQ, typename DP, int E>
__global__ void __launch_bounds__(kThreads, 3) verify_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) char ring_smem[];
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
    Feed<DQ, DP, E> feed;
    feed.init(ring_smem + warp * Feed<DQ, DP, E>::RING, lane);

    // ---- stream header (identical in every CTA): offsets, temperature, tokens, and the draft
    // and target logits at each draft token (loaded now, consumed after the sweep)
    const int base = p.cu[b];
    const int n_raw = p.cu[b + 1] - base;
    const int Lv = valid_prefix(p);   // streams from the first broken count on are invalid
    const bool offsets_ok = b < Lv;
    const int N = offsets_ok ? n_raw : 0;
    const float T = p.temp[b];
    const bool temp_ok = isfinite(T) && (T == 0.f || T >= FLT_MIN);
    const bool greedy = (T == 0.f);
    const int64_t dbase = offsets_ok ? base : 0;
    const int64_t tbase = dbase + b;
    auto qrow = [&](int i) { return row_ptr<DQ>(p.dq, dbase + i, V); };
    auto prow = [&](int i) { return row_ptr<DP>(p.dp, tbase + i, V); };
    if (tid < kWarps) sh.to_flag[tid] = 0;
    bool bad_tok = false;
    if (offsets_ok && temp_ok && tid < N) {
        const int xi = p.tokens[base + tid];
        sh.x[tid] = xi;
        bad_tok = (xi < 0 || xi >= p.V);
        if (!bad_tok && !greedy) {
            sh.lq[tid] = load_elem<DQ>(qrow(tid), xi);
            sh.lp[tid] = load_elem<DP>(prow(tid), xi);
        }
    }
    bad_tok = __syncthreads_or(bad_tok);
    if (tid == 0) {
        int st = SPEC_ST_OK;
        if (!offsets_ok) st = SPEC_ST_BAD_OFFSETS;
        else if (!temp_ok) st = SPEC_ST_BAD_TEMPERATURE;
        else if (bad_tok) st = SPEC_ST_BAD_TOKEN;
        sh.N = N;
        sh.status = st;
        sh.greedy = (st == SPEC_ST_OK && greedy);
        float ah = 0.f, al = 0.f;
        if (st == SPEC_ST_OK && T > 0.f) {   // a = log2(e) / T as a df
            const df l2e{1.4426950216293335f, 1.925963033500011e-08f};
            const df q = df_div(l2e, df_make(T));
            ah = q.hi;
            al = q.lo;
        }
        sh.a_hi = ah;
        sh.a_lo = al;
        sh.tau = 0;
        sh.sample_seg = -1;
        sh.sample_bonus = 0;
        sh.n_pass = 0;
    }
    __syncthreads();
    const float ah = sh.a_hi, al = sh.a_lo;
    const int nrows = 2 * N + 1;   // part index: draft row i -> i, target row i -> N + i

    // Everything above read only the call's inputs.  The stats kernel writes every row of a
    // stream with valid offsets and temperature (target rows only when greedy); each row is
    // waited for here - also when the stream already failed, so that its counters can be reset
    // at the end - and its partials are read once the row's counter is full.
    // the per-slot uniforms depend on (seed, step, stream, slot) only
    if (sh.status == SPEC_ST_OK && !greedy && tid <= N) {
        const uint4 c = make_uint4((uint32_t)tid, (uint32_t)b, (uint32_t)p.step, (uint32_t)(p.step >> 32));
        const uint4 wds = philox4x32_10(c, make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
        sh.u_acc[tid] = uniform24_df(wds.x);
        sh.u_smp[tid] = wds.y;
        sh.h[tid] = df{__int_as_float(0x7fffffff), 0.f};
        sh.r[tid] = df{__int_as_float(0x7fffffff), 0.f};
    }
    const bool rows_written = offsets_ok && temp_ok;
    const int64_t nck = p.nchunk;
    const int64_t lw = stats_share(2 * (int64_t)p.cu[Lv] + Lv, nck, p.stats_warps);
    // stats row of part r: target row i at g_b + i, draft row i at g_b + N + 1 + i
    auto stats_row = [&](int r) { return 2 * (int64_t)base + b + (r < N ? N + 1 + r : r - N); };
    bool stats_to = false;
    if (rows_written) {
        // one row per half-warp (16 rows per pass): lane l of a half holds pieces l, l + 16, ...
        const bool ok = sh.status == SPEC_ST_OK;
        const int hl = lane & 15;
        for (int r0 = (greedy ? N : 0) + 2 * warp; r0 < nrows; r0 += 2 * kWarps) {
            const int r = r0 + (lane >> 4);
            const bool have = r < nrows;
            int cnt = 0;
            bool full = false;
            int64_t rho = 0;
            if (have) {
                rho = stats_row(r);
                const int64_t first = rho * nck / lw;
                cnt = (int)((rho * nck + nck - 1) / lw - first) + 1;   // pieces of this row
                full = wait_count(row_counter(p, rho), (unsigned)cnt);
                stats_to |= !full;
            }
            if (!ok) continue;
            // row statistics from the per-piece partials (same order in every CTA, so every
            // CTA holds bit-identical values)
            constexpr int kSlots = kPiecesMax / 16;
            Part e[kSlots];
#pragma unroll
            for (int k = 0; k < kSlots; ++k) {
                const int pk = hl + 16 * k;
                if (have && full && pk < cnt) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(row_parts(p, rho) + pk));
                    e[k] = Part{v.x, v.y, v.z, __float_as_int(v.w)};
                } else {
                    e[k] = Part{greedy ? -kInf : kNoRef, 0.f, 0.f, INT_MAX};
                }
                stats_to |= (e[k].idx == kStatsTimeout);   // that piece's bounded wait gave up
            }
            if (greedy) {
                float Kr = e[0].K;
#pragma unroll
                for (int k = 1; k < kSlots; ++k) Kr = fmax_nan(Kr, e[k].K);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) Kr = fmax_nan(Kr, __shfl_xor_sync(0xffffffffu, Kr, o));
                int arg = INT_MAX;
#pragma unroll
                for (int k = 0; k < kSlots; ++k) arg = min(arg, e[k].K == Kr ? e[k].idx : INT_MAX);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, o));
                if (have && hl == 0) {
                    sh.rowK[r] = Kr;
                    sh.rowArg[r] = arg;
                    sh.rowZ[r] = df{0.f, 0.f};
                }
                continue;
            }
            float Kr = e[0].K;
#pragma unroll
            for (int k = 1; k < kSlots; ++k) Kr = fmaxf(Kr, e[k].K);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) Kr = fmaxf(Kr, __shfl_xor_sync(0xffffffffu, Kr, o));
            df z{0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kSlots; ++k) {
                const float sc = (e[k].K == Kr) ? 1.f : pow2_int(e[k].K - Kr);
                z = df_add(z, df_scale(df{e[k].s_hi, e[k].s_lo}, sc));
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                const df other{__shfl_xor_sync(0xffffffffu, z.hi, o), __shfl_xor_sync(0xffffffffu, z.lo, o)};
                z = df_add(z, other);
            }
            if (have && hl == 0) {
                sh.rowK[r] = Kr;
                sh.rowZ[r] = z;
                sh.rowArg[r] = INT_MAX;
            }
        }
    }
    stats_to = __syncthreads_or(stats_to);
    if (tid == 0 && stats_to) {
        if (sh.status == SPEC_ST_OK) sh.status = SPEC_ST_TIMEOUT;
        sh.to_flag[0] = 1;   // the time-bounded waits of the cluster's CTAs may end differently
    }
    __syncthreads();
    if (sh.status == SPEC_ST_OK) {
        // ---- validity of the rows read, q_i(x_i) > 0, per-slot ratios
        bool bad_row = false, zero_q = false;
        for (int r = (greedy ? N : 0) + tid; r < nrows; r += kThreads) {
            const float K = sh.rowK[r];
            const df z = sh.rowZ[r];
            bad_row |= greedy ? !isfinite(K) : !(isfinite(K) && K > kNoRef && isfinite(z.hi) && z.hi > 0.f);
        }
        if (!greedy && tid < N) {
            const float lq = sh.lq[tid], lp = sh.lp[tid];
            zero_q = (lq == -kInf);
            const float Kq = sh.rowK[tid], Kp = sh.rowK[N + tid];
            df rho{0.f, 0.f};
            if (!zero_q && isfinite(lq) && isfinite(lp) && isfinite(Kq) && isfinite(Kp)) {
                const df e = df_sub(exponent_df(lp, ah, al, Kp), exponent_df(lq, ah, al, Kq));
                rho = df_div(df_mul(df_exp2(e), sh.rowZ[tid]), sh.rowZ[N + tid]);
            }
            sh.rho[tid] = rho;
        }
        bad_row = __syncthreads_or(bad_row);
        zero_q = __syncthreads_or(zero_q);
        if (tid == 0) {
            if (bad_row) sh.status = SPEC_ST_BAD_ROW;
            else if (zero_q) sh.status = SPEC_ST_ZERO_DRAFT_PROB;
        }
        __syncthreads();
    }

    const df one{1.f, 0.f};
    int np = 0;
    // ---- decisions
    if (sh.status == SPEC_ST_OK && greedy) {
        if (tid == 0) {
            int tau = N;
            for (int i = 0; i < N; ++i)
                if (sh.rowArg[N + i] != sh.x[i]) {
                    tau = i;
                    break;
                }
            sh.tau = tau;
        }
        __syncthreads();
    } else if (sh.status == SPEC_ST_OK) {
        const bool block = (p.rule == 1);
        if (tid == 0) {
            int n = 0;
            if (block) {
                sh.w[0] = one;
                for (int i = 0; i < N; ++i) sh.w[i + 1] = df_min(one, df_mul(sh.w[i], sh.rho[i]));
                sh.tau = 0;
                if (N > 0) sh.h[N] = sh.w[N];
                if (N > 0 && df_le(sh.u_acc[N - 1], sh.h[N])) {
                    sh.tau = N;   // eta_N <= w_N: accept everything, no residual needed
                } else {
                    for (int i = N - 1; i >= 1; --i)   // candidates: eta_i <= w_i (h_i <= w_i)
                        if (df_le(sh.u_acc[i - 1], sh.w[i])) sh.pass_list[n++] = i;
                    if (N > 0) sh.pass_list[n++] = 0;
                }
            } else {
                int tau = N;
                for (int i = 0; i < N; ++i)
                    if (!df_le(sh.u_acc[i], df_min(one, sh.rho[i]))) {
                        tau = i;
                        break;
                    }
                sh.tau = tau;
                if (tau < N) {
                    sh.w[tau] = one;
                    sh.pass_list[n++] = tau;
                }
            }
            if (sh.tau == N) {   // every draft accepted: the sweep sums the bonus row instead
                sh.pass_list[0] = N;
                n = 1;
                sh.sample_bonus = 1;
            }
            sh.n_pass = n;
        }
        __syncthreads();
        np = sh.n_pass;
        const bool bonus_sweep = sh.sample_bonus != 0;
        if (tid < np && !bonus_sweep) {
            const int i = sh.pass_list[tid];
            sh.cval[i] = df_to_f(df_div(df_mul(sh.w[i], sh.rowZ[i]), sh.rowZ[N + i]));
        }
        __syncthreads();

        // ---- one cluster-wide residual sweep over every slot that may be needed
        if (np > 0) {
            Kahan acc;
            float grp = 0.f;   // this lane's chunk sums of the current group (independent), added once
            float Kq = 0.f, Kp = 0.f, cc = 0.f;
            sweep<DQ, DP, E>(
                feed, np, c0, c1, lane,
                [&](int it, const void*& rq, const void*& rp) {
                    const int i = sh.pass_list[it];
                    rq = bonus_sweep ? nullptr : qrow(i);
                    rp = prow(i);
                },
                [&](int it) {
                    const int i = sh.pass_list[it];
                    Kq = bonus_sweep ? 0.f : sh.rowK[i];
                    Kp = sh.rowK[N + i];
                    cc = bonus_sweep ? 1.f : sh.cval[i];
                    acc = Kahan();
                },
                [&](int64_t, const float (&xq)[E], const float (&xp)[E]) {
                    if (bonus_sweep) grp += target_chunk_sum<E>(xp, Kp, ah, al);
                    else grp += resid_chunk_sum<E>(xq, xp, Kq, Kp, ah, al, cc);
                },
                [&](int it) {
                    df tot = acc.value();
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const df other{__shfl_xor_sync(0xffffffffu, tot.hi, o), __shfl_xor_sync(0xffffffffu, tot.lo, o)};
                        tot = df_add(tot, other);
                    }
                    if (lane == 0) sh.res_part[it][warp] = df_to_f(tot);
                },
                [&]() {
                    acc.add(grp);
                    grp = 0.f;
                });
            if (lane == 0 && feed.timeout) sh.to_flag[warp] = 1;
        }
    }

    // ---- every CTA of the cluster meets here exactly once, whatever its status, so the CTAs
    // cannot part ways at a cluster barrier; a bounded wait that gave up in any of them (their
    // statuses may differ only there) makes the stream TIMEOUT in all of them
    cluster_sync_all();
    {
        bool to = false;
        if (tid < nseg) to = *cluster.map_shared_rank(&sh.to_flag[tid % kWarps], tid / kWarps) != 0;
        to = __syncthreads_or(to);
        if (to && tid == 0 && sh.status == SPEC_ST_OK) sh.status = SPEC_ST_TIMEOUT;
        __syncthreads();
    }

    if (sh.status == SPEC_ST_OK && !greedy) {
        const bool block = (p.rule == 1);
        const bool bonus_sweep = sh.sample_bonus != 0;
        np = sh.n_pass;
        if (np > 0) {
            // per pass item: r_i = (sum over all segments) / Z_q
            for (int it = warp; it < np && !bonus_sweep; it += kWarps) {
                df tot{0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int s = lane + 32 * k;
                    const float v = (s < nseg) ? *cluster.map_shared_rank(&sh.res_part[it][s % kWarps], s / kWarps) : 0.f;
                    tot = df_add_f(tot, v);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const df other{__shfl_xor_sync(0xffffffffu, tot.hi, o), __shfl_xor_sync(0xffffffffu, tot.lo, o)};
                    tot = df_add(tot, other);
                }
                if (lane == 0) {
                    const int i = sh.pass_list[it];
                    const df ri = df_div(tot, sh.rowZ[i]);
                    sh.r[i] = ri;
                    if (block && i >= 1) {
                        const df den = df_add(ri, df_sub(one, sh.w[i]));
                        sh.h[i] = df_is_zero(den) ? one : df_div(ri, den);
                    }
                }
            }
            __syncthreads();
            if (tid == 0 && block) {
                int tau = 0;
                for (int it = 0; it < np; ++it) {   // candidates in descending order, then slot 0
                    const int i = sh.pass_list[it];
                    if (i >= 1 && df_le(sh.u_acc[i - 1], sh.h[i])) {
                        tau = i;
                        break;
                    }
                }
                sh.tau = tau;
            }
            __syncthreads();
        }

        // ---- the draw: 64-bit fixed-point CDF over the segments (warp 0)
        if (warp == 0) {
            const int tau = sh.tau;
            const bool bonus = (tau == N);
            int item = 0;
            for (int it = 0; it < np; ++it)
                if (sh.pass_list[it] == tau) item = it;
            float w0 = 0.f, w1 = 0.f;
            if (lane < nseg) w0 = *cluster.map_shared_rank(&sh.res_part[item][lane % kWarps], lane / kWarps);
            if (lane + 32 < nseg)
                w1 = *cluster.map_shared_rank(&sh.res_part[item][(lane + 32) % kWarps], (lane + 32) / kWarps);
            const float wmax = warp_max(fmaxf(w0, w1));
            const bool ok = isfinite(wmax) && wmax > 0.f;
            const float scale = ok ? fixed_scale(wmax) : 0.f;
            const unsigned long long q0 = ok ? __float2ull_rn(w0 * scale) : 0ull;
            const unsigned long long q1 = ok ? __float2ull_rn(w1 * scale) : 0ull;
            unsigned long long p0 = q0, p1 = q1;   // inclusive prefix sums
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long n0 = __shfl_up_sync(0xffffffffu, p0, o);
                const unsigned long long n1 = __shfl_up_sync(0xffffffffu, p1, o);
                if (lane >= o) {
                    p0 += n0;
                    p1 += n1;
                }
            }
            p1 += __shfl_sync(0xffffffffu, p0, 31);
            const unsigned long long R = __shfl_sync(0xffffffffu, p1, 31);
            // t = floor(U R), U = (2k + 1) 2^-25 with k the word's top 24 bits
            const unsigned long long odd = 2ull * (sh.u_smp[tau] >> 8) + 1ull;
            const unsigned long long t = (__umul64hi(odd, R) << 39) | ((odd * R) >> 25);
            const unsigned h0 = __ballot_sync(0xffffffffu, q0 > 0 && p0 > t);
            const unsigned h1 = __ballot_sync(0xffffffffu, q1 > 0 && p1 > t);
            const int seg = h0 ? __ffs(h0) - 1 : (h1 ? 32 + __ffs(h1) - 1 : -1);
            const int src = seg < 0 ? 0 : seg % 32;
            const unsigned long long i0 = __shfl_sync(0xffffffffu, p0, src);
            const unsigned long long i1 = __shfl_sync(0xffffffffu, p1, src);
            const unsigned long long qs0 = __shfl_sync(0xffffffffu, q0, src);
            const unsigned long long qs1 = __shfl_sync(0xffffffffu, q1, src);
            if (lane == 0) {
                if (ok && R > 0 && seg >= 0) {
                    const unsigned long long excl = (seg < 32) ? i0 - qs0 : i1 - qs1;
                    sh.sample_t = t - excl;
                    sh.sample_scale = scale;
                    sh.sample_seg = seg;
                    sh.sample_bonus = bonus;
                } else {
                    sh.status = SPEC_ST_NUMERIC;
                    sh.sample_seg = -1;
                }
            }
        }
        __syncthreads();
    }

    // every distributed-shared-memory read of this CTA is done: arrive now, wait at the end
    cluster_arrive();

    // ---- the rescan of the drawn segment, split over the warps of the CTA that owns it: each
    // warp sums an eighth in fixed point, the eighth that crosses the target is rescanned
    if (sh.status == SPEC_ST_OK && !greedy && sh.sample_seg >= 0 && crank == sh.sample_seg / kWarps) {
        const int tau = sh.tau;
        const bool bonus = sh.sample_bonus != 0;
        const void* rq = bonus ? nullptr : qrow(tau);
        const void* rp = bonus ? prow(N) : prow(tau);
        const float Kq = bonus ? 0.f : sh.rowK[tau], Kp = bonus ? sh.rowK[2 * N] : sh.rowK[N + tau];
        const float cc = bonus ? 0.f : sh.cval[tau];
        const int64_t s0 = min(p.nchunk, (int64_t)sh.sample_seg * p.seg_chunks);
        const int64_t s1 = min(p.nchunk, s0 + p.seg_chunks);
        const int64_t msub = (s1 - s0 + kWarps - 1) / kWarps;
        const int64_t w0 = min(s1, s0 + warp * msub), w1 = min(s1, w0 + msub);
        unsigned long long sub;
        int last;
        if (bonus)
            segment_fixed_sum<DQ, DP, E, true>(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, lane, sub, last);
        else
            segment_fixed_sum<DQ, DP, E, false>(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, lane, sub, last);
        if (lane == 0) {
            sh.sub_sum[warp] = sub;
            sh.sub_last[warp] = last;
        }
        __syncthreads();
        const unsigned long long t = sh.sample_t;
        unsigned long long before = 0;
        int wsel = -1, lastpos = -1;
        for (int w = 0; w < kWarps; ++w) {
            lastpos = max(lastpos, sh.sub_last[w]);
            if (wsel < 0) {
                if (sh.sub_sum[w] > 0 && before + sh.sub_sum[w] > t) wsel = w;
                else before += sh.sub_sum[w];
            }
        }
        int y = -1;
        if (wsel < 0) {
            y = lastpos;   // rounding kept the segment's sum at or below the target
        } else if (warp == wsel) {
            y = bonus ? rescan_segment<DQ, DP, E, true>(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, t - before, lane)
                      : rescan_segment<DQ, DP, E, false>(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, t - before,
                                                         lane);
        }
        if ((wsel < 0 && tid == 0) || (warp == wsel && lane == 0)) p.out_tok[(int64_t)b * (p.kmax + 1) + tau] = y;
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
            else if (sh.greedy) p.out_tok[ob + j] = sh.rowArg[N + tau];
        }
        if (tid == 0) {
            p.status[b] = st;
            p.acc_len[b] = (st == SPEC_ST_OK) ? tau : 0;
            p.n_emit[b] = (st == SPEC_ST_OK) ? tau + 1 : 0;
        }
        if (p.diag != nullptr && st != SPEC_ST_BAD_OFFSETS) {
            const float qnan = __int_as_float(0x7fffffff);
            const float ln2 = 0.6931471805599453f;
            const bool have = (!sh.greedy) && (st == SPEC_ST_OK || st == SPEC_ST_NUMERIC);
            for (int i = tid; i <= N; i += kThreads) {
                float* d = p.diag + (tbase + i) * SPEC_DIAG_COLS;
                float v[SPEC_DIAG_COLS];
#pragma unroll
                for (int c = 0; c < SPEC_DIAG_COLS; ++c) v[c] = qnan;
                if (have) {
                    // natural log of sum exp(l / T) = ln 2 (K + log2 Z)
                    const df zp = sh.rowZ[N + i];
                    v[SPEC_DIAG_LOGZP] = ln2 * (sh.rowK[N + i] + log2f(zp.hi)) + zp.lo / zp.hi;
                    if (i < N) {
                        const df zq = sh.rowZ[i];
                        const float lq = sh.lq[i], lp = sh.lp[i];
                        v[SPEC_DIAG_PX] =
                            isfinite(lp) ? df_to_f(df_div(df_exp2(exponent_df(lp, ah, al, sh.rowK[N + i])), zp)) : 0.f;
                        v[SPEC_DIAG_QX] =
                            isfinite(lq) ? df_to_f(df_div(df_exp2(exponent_df(lq, ah, al, sh.rowK[i])), zq)) : 0.f;
                        v[SPEC_DIAG_RHO] = df_to_f(sh.rho[i]);
                        v[SPEC_DIAG_LOGZQ] = ln2 * (sh.rowK[i] + log2f(zq.hi)) + zq.lo / zq.hi;
                    }
                    if (p.rule == 1) {
                        v[SPEC_DIAG_W] = df_to_f(sh.w[i]);
                        if (i >= 1) v[SPEC_DIAG_H] = df_to_f(sh.h[i]);
                    }
                    v[SPEC_DIAG_R] = df_to_f(sh.r[i]);
                }
#pragma unroll
                for (int c = 0; c < SPEC_DIAG_COLS; ++c) d[c] = v[c];
            }
        }
    }
    // no TMA copy of this warp may still be writing its ring when the CTA leaves
    feed.drain();
    // no CTA may leave while another can still read its shared memory
    cluster_wait();
    // The grid completes only after the stats grid (a stream with no rows, or whose wait gave
    // up, never waited for it).  Then every stats add has landed and every CTA of the cluster
    // has read its partials: the row counters go back to zero for the next call.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (crank == 0 && rows_written)
        for (int r = (greedy ? N : 0) + tid; r < nrows; r += kThreads) *row_counter(p, stats_row(r)) = 0u;
}

// Uniforms exposed for checking: out[(s * n_slots + i) * 2 + {0, 1}] (exact in double)
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
static size_t ring_bytes() {
    return (size_t)kWarps * Feed<DQ, DP, E>::RING;
}

template <typename DQ, typename DP, int E>
static cudaLaunchConfig_t make_config(int grid, int C, cudaStream_t s, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = ring_bytes<DQ, DP, E>();
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <typename DQ, typename DP, int E>
static cudaError_t prepare_kernel() {
    static int done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (done[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<DQ, DP, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ring_bytes<DQ, DP, E>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(stats_kernel<DQ, DP, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)stats_smem_bytes(E));
    if (e == cudaSuccess) done[dev] = 1;
    return e;
}

// How many clusters of C CTAs fit on the device at once (queried once per kernel, C, device).
template <typename DQ, typename DP, int E>
static int resident_clusters(int C) {
    static int cache[kMaxCluster + 1][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int& slot = cache[C][dev];
    if (slot == 0) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = make_config<DQ, DP, E>(C, C, nullptr, attr);
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

// Persistent grid of the stats kernel: every SM filled to its occupancy.
template <typename DQ, typename DP, int E>
static int stats_grid() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (cache[dev] == 0) {
        int sms = 0, occ = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, stats_kernel<DQ, DP, E>, kThreads,
                                                          stats_smem_bytes(E)) != cudaSuccess ||
            occ < 1) {
            cudaGetLastError();
            occ = 1;
        }
        cache[dev] = sms * occ;
    }
    return cache[dev];
}

template <typename DQ, typename DP, int E>
static cudaError_t run_verify(VerifyParams& p, cudaStream_t s, int* info) {
    cudaError_t e = prepare_kernel<DQ, DP, E>();
    if (e != cudaSuccess) return e;
    const int C = pick_cluster<DQ, DP, E>(p.B, p.nchunk);
    p.seg_chunks = (p.nchunk + (int64_t)C * kWarps - 1) / ((int64_t)C * kWarps);
    if (info) {
        info[0] = C;
        info[1] = resident_clusters<DQ, DP, E>(C);
        return cudaSuccess;
    }
    const int grid = stats_grid<DQ, DP, E>();
    p.stats_warps = (int64_t)grid * kWarps;
    stats_kernel<DQ, DP, E><<<grid, kThreads, stats_smem_bytes(E), s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config<DQ, DP, E>(p.B * C, C, s, attr);
    // programmatic dependent launch: the verify kernel's CTAs start while the stats kernel
    // drains; each stream waits only for its own rows' counters
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, verify_kernel<DQ, DP, E>, p);
    if (e != cudaSuccess)   // the stats kernel ran: its counts must not reach the next call
        cudaMemsetAsync(p.ws, 0, workspace_bytes(p.B, p.kmax), s);
    return e;
}

template <int E>
static cudaError_t dispatch_dtypes(VerifyParams& p, int dq, int dp, cudaStream_t s, int* info) {
    if (dq == SPEC_DTYPE_BF16 && dp == SPEC_DTYPE_BF16) return run_verify<__nv_bfloat16, __nv_bfloat16, E>(p, s, info);
    if (dq == SPEC_DTYPE_F32 && dp == SPEC_DTYPE_F32) return run_verify<float, float, E>(p, s, info);
    if (dq == SPEC_DTYPE_F32 && dp == SPEC_DTYPE_BF16) return run_verify<float, __nv_bfloat16, E>(p, s, info);
    return run_verify<__nv_bfloat16, float, E>(p, s, info);
}

static int verify_entry(const spec_verify_args* a, void* stream, int rule, const char* name, int* info) {
    if (a == nullptr) return set_error(SPEC_ERR_ARG, "%s: args is NULL", name);
    if (a->B < 0) return set_error(SPEC_ERR_SHAPE, "%s: B = %d < 0", name, a->B);
    if (a->V < 1 || a->V > SPEC_MAX_V)
        return set_error(SPEC_ERR_SHAPE, "%s: V = %d outside [1, %d]", name, a->V, SPEC_MAX_V);
    if (a->kmax < 0 || a->kmax > SPEC_MAX_KMAX)
        return set_error(SPEC_ERR_SHAPE, "%s: kmax = %d outside [0, %d]", name, a->kmax, SPEC_MAX_KMAX);
    if (!valid_dtype(a->draft_dtype) || !valid_dtype(a->target_dtype))
        return set_error(SPEC_ERR_DTYPE, "%s: dtype must be SPEC_DTYPE_F32 or SPEC_DTYPE_BF16", name);
    if (info == nullptr) {
        if (a->B == 0) return clear_error();
        if (!a->cu_drafts || !a->target_logits || !a->temperature || !a->accepted_len || !a->out_tokens ||
            !a->n_emitted || !a->status)
            return set_error(SPEC_ERR_ARG, "%s: a required pointer is NULL", name);
        if ((a->kmax > 0) && (!a->draft_logits || !a->draft_tokens))
            return set_error(SPEC_ERR_ARG, "%s: draft_logits / draft_tokens is NULL", name);
    }
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
    p.ws = reinterpret_cast<char*>(a->workspace);
    if (info == nullptr) {
        const size_t need = workspace_bytes(a->B, a->kmax);
        if (a->workspace == nullptr || a->workspace_bytes < need || (uintptr_t)a->workspace % 16 != 0)
            return set_error(SPEC_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", name,
                             need, a->workspace_bytes);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = aligned ? dispatch_dtypes<8>(p, a->draft_dtype, a->target_dtype, s, info)
                                  : dispatch_dtypes<1>(p, a->draft_dtype, a->target_dtype, s, info);
    if (e != cudaSuccess) return set_cuda_error(e, name);
    if (info) info[2] = aligned ? 8 : 1;
    return clear_error();
}

}  // namespace sv

extern "C" int spec_verify_tokenwise(const spec_verify_args* args, void* stream) {
    return sv::verify_entry(args, stream, 0, "spec_verify_tokenwise", nullptr);
}

extern "C" int spec_verify_block(const spec_verify_args* args, void* stream) {
    return sv::verify_entry(args, stream, 1, "spec_verify_block", nullptr);
}

// ---------------------------------------------------------------------------------------
// Block verification with a fixed, device-resident workspace.  Some callers cannot allocate
// device memory at the point where they verify (an allocator that is not theirs to touch, a
// memory budget fixed at start-up); for them the stats partials live in one array reserved
// when the library's module is loaded, so this call allocates nothing.  The array holds
// kStaticWorkspaceBytes: B (2 kmax + 1) row blocks (a counter and kPiecesMax 16-byte partials
// each), i.e. up to 8192 rows (for example B = 256 at kmax = 15); larger batches are refused.
// Like every device variable it starts zero-filled, which is the state each call leaves its
// row counters in.  All calls share the one array, so calls that may overlap in time
// (different streams, threads) race on it and must be ordered by the caller.
// ---------------------------------------------------------------------------------------
namespace sv {
constexpr size_t kStaticWorkspaceBytes = (size_t)8192 * kRowBytes;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// device address of g_static_workspace on the current device, looked up once per device
static cudaError_t static_workspace(void** ptr) {
    static void* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (addr[dev] == nullptr) {
        void* a = nullptr;
        e = cudaGetSymbolAddress(&a, g_static_workspace);
        if (e != cudaSuccess) return e;
        addr[dev] = a;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}
}  // namespace sv

extern "C" int spec_verify_block_static(const spec_verify_args* args, void* stream) {
    const char* name = "spec_verify_block_static";
    if (args == nullptr) return sv::set_error(SPEC_ERR_ARG, "%s: args is NULL", name);
    spec_verify_args a = *args;
    const bool shape_ok = a.B >= 0 && a.kmax >= 0 && a.kmax <= SPEC_MAX_KMAX;
    if (shape_ok && a.B > 0) {   // bad shapes and empty batches are reported by the common path
        const size_t need = sv::workspace_bytes(a.B, a.kmax);
        if (need > sv::kStaticWorkspaceBytes)
            return sv::set_error(SPEC_ERR_WORKSPACE,
                                 "%s: B = %d, kmax = %d needs %zu workspace bytes; the static workspace "
                                 "holds %zu (use spec_verify_block with a caller workspace)",
                                 name, a.B, a.kmax, need, sv::kStaticWorkspaceBytes);
        void* ws = nullptr;
        const cudaError_t e = sv::static_workspace(&ws);
        if (e != cudaSuccess) return sv::set_cuda_error(e, name);
        a.workspace = ws;
        a.workspace_bytes = sv::kStaticWorkspaceBytes;
    }
    return sv::verify_entry(&a, stream, 1, name, nullptr);
}

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t kmax) {
    if (B < 0 || kmax < 0 || kmax > SPEC_MAX_KMAX) return 0;
    return sv::workspace_bytes(B, kmax);
}

extern "C" int spec_verify_launch_info(const spec_verify_args* args, int32_t* cluster_size,
                                       int32_t* resident_clusters, int32_t* elems_per_load) {
    if (!cluster_size || !resident_clusters || !elems_per_load)
        return sv::set_error(SPEC_ERR_ARG, "spec_verify_launch_info: an output pointer is NULL");
    int info[3] = {0, 0, 0};
    const int rc = sv::verify_entry(args, nullptr, 1, "spec_verify_launch_info", info);
    if (rc != SPEC_OK) return rc;
    *cluster_size = info[0];
    *resident_clusters = info[1];
    *elems_per_load = info[2];
    return SPEC_OK;
}

extern "C" int spec_philox_uniforms(uint64_t seed, uint64_t step, int32_t n_streams, int32_t n_slots,
                                    double* out, void* stream) {
    if (n_streams < 0 || n_slots < 0) return sv::set_error(SPEC_ERR_SHAPE, "spec_philox_uniforms: negative count");
    const int64_t total = (int64_t)n_streams * n_slots;
    if (total == 0) return sv::clear_error();
    if (out == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_philox_uniforms: out is NULL");
    const int64_t blocks64 = (total + 255) / 256;
    const int blocks = (int)(blocks64 < 4096 ? blocks64 : 4096);
    sv::philox_uniforms_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(seed, step, n_streams,
                                                                                        n_slots, out);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_philox_uniforms");
    return sv::clear_error();
}
