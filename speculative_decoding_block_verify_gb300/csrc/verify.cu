// Token-wise speculative sampling and block verification on sm_103a.
//
// Method: "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com),
// §4 "Verification: the guarantee" - "Token by token" (Leviathan et al. 2023), "Block
// verification" (Sun et al. 2024) with Figure 3, and "Greedy is a different code path".
//
// Design: four launches per call on the caller's stream, chained by programmatic dependent
// launch (each kernel's prologue overlaps its predecessor's tail; griddepcontrol.wait orders
// the data).  No kernel waits for another kernel's CTAs, so none can deadlock.
//   * stats_kernel (persistent): every logit of the batch is read from HBM once.  The chunks of
//     all rows, end to end, are cut into equal contiguous shares, one per warp, so every warp
//     streams the same bytes without any claim or hand-off; a share goes through a ring of
//     shared-memory stages filled by TMA bulk copies and leaves one partial per row it touches:
//     (integer reference K, sum of 2^(l a - K)) for T > 0, (maximum, lowest index) for T = 0.
//     a = log2(e) / T is carried as a_hi + a_lo, so each exponent is two FMAs and the
//     temperature is exact to ~1e-14.
//   * decide_kernel (one CTA per stream): the row normalisers from the partials, the ratios
//     rho_i and the clipped running product w_i in double-float, the statuses, and the
//     decision - greedy tau, token-wise tau, or block verification's candidate slots (eta_i <=
//     w_i, since h_i <= w_i) plus slot 0; every slot whose residual may be needed becomes a
//     sweep item, and the items' segments are appended to the sweep's work list.
//   * sweep_kernel (persistent): the residual masses sum_v max(0, c 2^(lp a - Kp) -
//     2^(lq a - Kq)), c = w_i Z_q / Z_p, of every item, one sum per segment, with the warps of
//     the whole GPU claiming runs of segments - a stream with many candidates no longer waits
//     for a few SMs.  These reads are the only ones beyond the algorithmic bytes.
//   * finish_kernel (one CTA per stream): r_i, h_i = r_i / (r_i + 1 - w_i), tau, then the draw:
//     a 64-bit fixed-point CDF over the drawn item's segment sums picks the segment, its eight
//     slices are summed in the same fixed point by the CTA's warps, and the warp whose slice
//     crosses the target rescans it.
// Every bounded wait that gives up turns the stream to SPEC_ST_TIMEOUT; nothing traps.

#include <cfloat>
#include <climits>

#include <atomic>

#include "common.cuh"
#include "df.cuh"
#include "draw.cuh"
#include "host_util.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 2 * SPEC_MAX_KMAX + 1;
constexpr float kNoRef = -1e30f;     // reference of a lane that has seen no finite logit
constexpr int kSegs = 64;            // residual segments per row: the draw's CDF resolution
constexpr int kSegLanes = kSegs / 32;   // segments a lane holds in the per-row warp steps
static_assert(kSegs % 32 == 0, "segments come in whole warps");
constexpr int kPiecesMax = 64;       // stats partials per row
constexpr int kSegsPerClaim = 1;     // a sweep claim is one segment of one row pair (2 took 2 us more: coarser balance)
constexpr int kStatsThreads = 256;   // threads of a stats CTA
constexpr int kStatsWarps = kStatsThreads / 32;

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
    int64_t seg_chunks;  // chunks per residual segment
    int32_t nseg;        // segments per row (<= kSegs)
    int64_t stats_warps; // warps of the stats grid
    char* ws;            // workspace (layout below)
    char* list;          // the sweep's work list: the end of the workspace the caller passed
    int32_t dense;       // 1: logits and tokens in the dense [B, kmax (+1)] layout (see below)
    const uint64_t* step_dev;   // non-null: the Philox step is read from here (graph replays)
    // draft rows over a reduced draft vocabulary: Kq logits per draft row, target column v
    // holds draft id t2d[v] (none when t2d[v] lies outside [0, Kq)); t2d null: Kq = V
    const int32_t* t2d;
    int32_t Kq;
    int64_t nchunk_q;    // chunks per draft row (= nchunk unless t2d is given)
};

// Logit rows of (stream b, slot i).  Packed layout (the public verify calls): draft row
// cu[b] + i, target row cu[b] + b + i.  Dense layout (the adaptive pipeline, where the drafter
// always fills kmax slots and the controller picks how many are verified): draft row
// b kmax + i, target row b (kmax + 1) + i; draft tokens follow the draft rows.
__device__ __forceinline__ int64_t qrow_of(const VerifyParams& p, int b, int base, int i) {
    return p.dense ? (int64_t)b * p.kmax + i : (int64_t)base + i;
}
__device__ __forceinline__ int64_t prow_of(const VerifyParams& p, int b, int base, int i) {
    return p.dense ? (int64_t)b * (p.kmax + 1) + i : (int64_t)base + b + i;
}
__device__ __forceinline__ uint64_t step_of(const VerifyParams& p) { return p.step_dev ? *p.step_dev : p.step; }

// Draft logit of target column x in draft row `row` (-inf outside a reduced draft vocabulary).
template <typename DQ>
__device__ __forceinline__ float draft_logit_at(const VerifyParams& p, const void* row, int x) {
    if (p.t2d == nullptr) return load_elem<DQ>(row, x);
    const int j = __ldg(p.t2d + x);
    return in_vocab(j, p.Kq) ? load_elem<DQ>(row, j) : -__int_as_float(0x7f800000);
}

// Geometry of the stats pass: the chunks of all stats rows, stream by stream (target rows of
// nchunk chunks, then draft rows of nchunk_q), enumerated in one range.  Offset of stream b's
// first row: cu[b] + b target rows and cu[b] draft rows lie before it.
__device__ __forceinline__ int64_t stream_off(const VerifyParams& p, int b) {
    return ((int64_t)p.cu[b] + b) * p.nchunk + (int64_t)p.cu[b] * p.nchunk_q;
}
// Offset and length of stats row j of stream b (j <= N: target row j, else draft row j - N - 1).
__device__ __forceinline__ int64_t row_off(const VerifyParams& p, int b, int N, int j) {
    const int64_t o = stream_off(p, b);
    return j <= N ? o + (int64_t)j * p.nchunk : o + (int64_t)(N + 1) * p.nchunk + (int64_t)(j - N - 1) * p.nchunk_q;
}
__device__ __forceinline__ int64_t row_len(const VerifyParams& p, int N, int j) {
    return j <= N ? p.nchunk : p.nchunk_q;
}

// Per-piece partial of one row.  T > 0: K = integer reference, (s_hi, s_lo) = sum 2^(l a - K).
// T = 0: K = the piece maximum, idx = its lowest index.
struct Part {
    float K;
    float s_hi, s_lo;
    int idx;
};

// ---------------------------------------------------------------------------------------
// Workspace.  A 256-byte header (the two claim tickets, the valid stream prefix, the number of
// sweep claims), then one block of kRowBytes per stats row; the sweep's work list sits at the
// very end of the buffer the caller passed, so that it never lands on the row counters of a
// call with a larger batch on the same buffer.
// Stream b owns stats rows g_b = 2 cu[b] + b .. g_b + 2 N_b: its target rows 0..N_b, then its
// draft rows 0..N_b-1.  A row's block holds its piece counter and partials, its statistics
// (decide_kernel), and - in target row i's block - slot i's scalars and the segment sums of
// slot i's sweep item; the stream's own scalars sit in its first row's block.  The state that
// must be zero between calls (tickets, counters) sits at the same place for every B, and every
// call returns it to zero, so a zero-filled workspace stays valid from call to call.
// ---------------------------------------------------------------------------------------
constexpr int kTailTickets = 8;        // the stats tail is cut into this many claim ranges
struct WsHeader {
    unsigned long long ticket_sweep;   // next sweep claim
    unsigned long long sweep_total;    // sweep claims appended by decide_kernel
    unsigned long long ticket_stats[kTailTickets];   // next piece of each range of the stats tail
    int32_t L;                         // streams [0, L) have valid offsets
};
struct RowStat {
    float K;          // reference exponent (T > 0) or maximum (T = 0)
    float zhi, zlo;   // sum 2^(l a - K) as a df
    int arg;          // lowest argmax (T = 0)
};
struct SlotRec {
    df rho, w, h, r;
    float cval;       // residual scale c = w_i Z_q / Z_p of slot i's sweep item
    int x;
    float lq, lp;     // the draft and target logits at x_i
};
struct StreamRec {
    int32_t status, N, greedy, tau, n_pass, bonus;
    float a_hi, a_lo;
    uint8_t pass[SPEC_MAX_KMAX + 4];   // sweep items: slots, candidates in descending order, then 0
};
struct SweepItem {   // one claim of the residual sweep, self-contained (32 bytes)
    int32_t b;        // stream
    int16_t slot;     // slot i of the item (N: the bonus row)
    int16_t s0;       // first segment of the claim
    float Kq, Kp;     // reference exponents of the draft and target rows at slot i
    float cc;         // residual scale c = w_i Z_q / Z_p (1 for the bonus row)
    float ah, al;     // a = log2(e) / T
    int32_t bonus;    // 1: the bonus row's own mass, not a residual
};
constexpr size_t kHeaderBytes = 256;
constexpr size_t kRowBytes = 1536;
constexpr int kOffStatsCount = 0;    // u32: stats pieces published for this row
constexpr int kOffSweepCount = 4;    // u32 (stream's first row): sweep segments published
constexpr int kOffSweepTimeout = 8;  // u32 (stream's first row): a sweep wait gave up
constexpr int kOffParts = 16;
constexpr int kOffSeg = kOffParts + kPiecesMax * (int)sizeof(Part);
constexpr int kOffRow = kOffSeg + kSegs * (int)sizeof(float);
constexpr int kOffSlot = kOffRow + (int)sizeof(RowStat);
constexpr int kOffStream = kOffSlot + (int)sizeof(SlotRec);
static_assert(sizeof(WsHeader) <= kHeaderBytes, "header");
static_assert(kOffStream + sizeof(StreamRec) <= kRowBytes, "row block");
static_assert(kOffSlot % 8 == 0 && kOffRow % 16 == 0 && kOffParts % 16 == 0, "alignment");

__host__ __device__ inline size_t workspace_rows(int32_t B, int32_t kmax) {
    return (size_t)B * (size_t)(2 * kmax + 1);
}
__host__ __device__ inline size_t work_list_claims(int32_t B, int32_t kmax) {
    return (size_t)B * (size_t)(kmax + 1) * (size_t)((kSegs + kSegsPerClaim - 1) / kSegsPerClaim);
}
__host__ __device__ inline size_t workspace_bytes(int32_t B, int32_t kmax) {
    if (B == 0) return 0;   // nothing is launched
    return kHeaderBytes + workspace_rows(B, kmax) * kRowBytes + work_list_claims(B, kmax) * sizeof(SweepItem);
}
__device__ __forceinline__ WsHeader* ws_header(const VerifyParams& p) { return reinterpret_cast<WsHeader*>(p.ws); }
__device__ __forceinline__ char* row_block(const VerifyParams& p, int64_t rho) {
    return p.ws + kHeaderBytes + rho * (int64_t)kRowBytes;
}
template <typename T>
__device__ __forceinline__ T* blk_at(char* blk, int off) {
    return reinterpret_cast<T*>(blk + off);
}
__device__ __forceinline__ SweepItem* work_list(const VerifyParams& p) { return reinterpret_cast<SweepItem*>(p.list); }

constexpr int kSpinLimit = 1 << 20;   // mbarrier polls before a wait gives up (status TIMEOUT)
constexpr int kStatsTimeout = -2;     // idx of a partial whose piece lost a bounded wait

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

// ---------------------------------------------------------------------------------------
// stats_kernel
// ---------------------------------------------------------------------------------------
// 16-byte rows (E = 8): each warp owns a ring of kStages stages of kStageBytes in shared
// memory, each filled by one TMA bulk copy (issued by lane 0) that completes on the stage's
// mbarrier; every lane waits with a bounded poll.  Large stages keep the per-stage work (the
// wait, the next copy, the reference check) small next to the per-element arithmetic: the
// scan is bound by issue slots as much as by HBM, about four instructions per logit.
#ifndef SV_STATS_STAGES
#define SV_STATS_STAGES 3
#endif
#ifndef SV_STATS_STAGE_BYTES
#define SV_STATS_STAGE_BYTES 4096
#endif
#ifndef SV_STATS_MIN_BLOCKS
#define SV_STATS_MIN_BLOCKS 2
#endif
constexpr int kStages = SV_STATS_STAGES;
constexpr int kStageBytes = SV_STATS_STAGE_BYTES;
constexpr int kStatsMinBlocks = SV_STATS_MIN_BLOCKS;   // resident CTAs per SM the registers allow
constexpr int kStatsRingBytes = kStatsWarps * kStages * kStageBytes;
static size_t stats_smem_bytes(int E) { return E == 8 ? (size_t)kStatsRingBytes : 0; }

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

// The stats kernel's per-warp ring: kStages stages of kStageBytes in shared memory, each
// filled by one TMA bulk copy (issued by lane 0, with an evict-first L2 policy: the logits are
// streamed through once and must not push the kernels' code and workspace out of L2) that
// completes on the stage's mbarrier; every lane waits with a bounded poll.  Copies are
// numbered over every piece of the warp: copy q uses slot q mod kStages, and its wait is that
// slot's (q div kStages)-th completion, so the parity is that count's low bit.
struct StatsRing {
    char* base;
    uint64_t* bar;
    uint64_t policy;
    uint32_t issued, done;   // copies issued / waited for
    int lane;
    bool timeout;
    __device__ __forceinline__ void init(char* b, uint64_t* bars, int ln) {
        base = b;
        bar = bars;
        lane = ln;
        issued = done = 0;
        timeout = false;
        policy = l2_evict_first_policy();
        if (lane == 0) {
            for (int i = 0; i < kStages; ++i) mbar_init(&bar[i], 1);
            mbar_init_fence();
        }
        __syncwarp();
    }
    __device__ __forceinline__ void issue(const char* src, unsigned bytes) {
        if (timeout) return;   // after a failed wait nothing new is put in flight
        const uint32_t slot = issued % kStages;
        ++issued;
        __syncwarp();          // every lane is done with this slot's previous contents
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&bar[slot], bytes);
            bulk_g2s_hint(base + slot * kStageBytes, src, bytes, &bar[slot], policy);
        }
    }
    // Waits for the oldest copy in flight and returns its stage.  The outcome is decided for the
    // whole warp (every lane takes the same path afterwards).
    __device__ __forceinline__ const char* wait() {
        const uint32_t slot = done % kStages;
        if (!timeout) {
            const uint32_t parity = (done / kStages) & 1u;
            bool ok = true;
            for (int n = 0; !mbar_try_wait(&bar[slot], parity);)
                if (++n > kSpinLimit) {
                    ok = false;
                    break;
                }
            timeout = !__all_sync(0xffffffffu, ok);   // a copy that timed out stays outstanding: drain() waits once more
            if (!timeout) ++done;
        }
        return base + slot * kStageBytes;
    }
    __device__ __forceinline__ void drain() {
        for (uint32_t q = done; q != issued; ++q) {
            const uint32_t slot = q % kStages, parity = (q / kStages) & 1u;
            for (int n = 0; n < kSpinLimit && !mbar_try_wait(&bar[slot], parity); ++n) {
            }
        }
    }
};

// One piece [c0, c1) of a 16-byte aligned row through the bulk ring: full stages go to
// add_full (U chunks per lane), the ragged last stage chunk by chunk to add.  after_last() runs
// (in every lane) right after the piece's last copy has been issued, while kStages - 1 stages
// are still to be consumed: the next claim is fired there, so its round trip overlaps this tail.
template <typename T, typename AddFn, typename GroupFn, typename AfterFn>
__device__ __forceinline__ void stream_piece_bulk(StatsRing& R, const void* row, int64_t c0, int64_t c1, int lane,
                                                  AddFn add, GroupFn add_full, AfterFn after_last) {
    constexpr int BT = 8 * (int)sizeof(T);   // bytes per chunk
    constexpr int G = kStageBytes / BT;      // chunks per stage
    constexpr int U = G / 32;                // chunks per lane and stage
    const char* src = reinterpret_cast<const char*>(row) + c0 * BT;
    const int64_t n = c1 - c0;
    const int nb = (int)((n + G - 1) / G);
    const int nfull = (int)(n / G);
    const unsigned last_bytes = (unsigned)((n - (int64_t)(nb - 1) * G) * BT);
    int next = 0;   // the next stage of the piece to issue
    auto issue_next = [&]() {
        R.issue(src, next == nb - 1 ? last_bytes : (unsigned)kStageBytes);
        src += kStageBytes;
        if (++next == nb) after_last();
    };
    const int prime = min(nb, kStages - 1);
    for (int i = 0; i < prime; ++i) issue_next();
    int64_t k0 = c0 + lane;   // this lane's first chunk of the stage
    for (int i = 0; i < nb; ++i, k0 += G) {
        if (next < nb) issue_next();   // into the slot of stage i - 1, consumed
        const char* st = R.wait();
        if (i < nfull) {   // a full stage: every lane has all U chunks
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
            add_full(x, k0);
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
                add(x, (k0 - lane + kk) * 8);
            }
        }
    }
}

template <typename T, int E, typename AfterFn>
__device__ __forceinline__ void stats_piece(StatsRing& ring, const void* row, int64_t c0, int64_t c1, bool greedy,
                                            float ah, float al, int lane, Part* dst, AfterFn after_last) {
    constexpr int UG = kStageBytes / (8 * (int)sizeof(T)) / 32;   // chunks per lane and stage
    if (greedy) {
        LaneMax mx;
        auto f = [&](const float (&x)[E], int64_t e0) { mx.add<E>(x, e0); };
        // chunk u of the group is chunk k0 + 32 u of the row (this lane's chunks, ascending)
        auto g = [&](const float (&x)[UG][8], int64_t k0) {
#pragma unroll
            for (int u = 0; u < UG; ++u) mx.add<8>(x[u], (k0 + 32 * u) * 8);
        };
        if constexpr (E == 8) {
            stream_piece_bulk<T>(ring, row, c0, c1, lane, f, g, after_last);
        } else {
            after_last();
            stream_piece<T, E>(row, c0, c1, lane, f);
        }
        mx.publish(dst, lane);
        if (ring.timeout && lane == 0) dst->idx = kStatsTimeout;
    } else {
        LaneSum sum;
        auto f = [&](const float (&x)[E], int64_t) { sum.add<E>(x, ah, al); };
        auto g = [&](const float (&x)[UG][8], int64_t) { sum.add_group<UG>(x, ah, al); };
        if constexpr (E == 8) {
            stream_piece_bulk<T>(ring, row, c0, c1, lane, f, g, after_last);
        } else {
            after_last();
            stream_piece<T, E>(row, c0, c1, lane, f);
        }
        sum.publish(dst, lane);
        if (ring.timeout && lane == 0) dst->idx = kStatsTimeout;
    }
}

// a = log2(e) / T as a df
__device__ __forceinline__ df scale_of_temperature(float T) { return temperature_scale(T); }

__device__ __forceinline__ bool temperature_ok(float T) { return isfinite(T) && (T == 0.f || T >= FLT_MIN); }

// The stream owning stats row rho: the largest b in [lo, L) with g_b = 2 cu[b] + b <= rho.
__device__ __forceinline__ int stream_of_row(const VerifyParams& p, int64_t rho, int lo, int L) {
    int hi = L - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (2 * (int64_t)p.cu[mid] + mid <= rho) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The stats kernel's work: the first rows (the static rows) in equal contiguous shares, one per
// warp; the remaining rows in fixed pieces of two segments, claimed by whichever warp is free
// (so SMs that run slower, or whose CTAs started later, simply take fewer of them).  The claimed
// tail pays a ramp and a claim per piece, which only a long share amortises: measured on the
// batch-64 bf16 call (~75 KB per warp) a twentieth, a tenth or a fifth of the rows as tail cost
// 4, 6 and 9 us more than none (75 us); on the batch-256 fp32 call (~1 MB per warp) a tenth
// takes 510 us, a twentieth 516 us, a fifth 533 us.  So the tail is a tenth of the rows when a
// warp's share is at least kTailMinChunks chunks, else empty.
// Draft rows over a reduced draft vocabulary are shorter than target rows; their calls take
// every row static (the tail's fixed pieces assume one row length).
constexpr int64_t kTailMinChunks = 16384;
__host__ __device__ inline int64_t static_rows(int64_t rows, int64_t n, int64_t warps, bool reduced) {
    if (reduced) return rows;
    return (rows * n >= kTailMinChunks * warps) ? rows * 9 / 10 : rows;
}
__host__ __device__ inline int64_t tail_pieces_per_row(int64_t n, int64_t seg_chunks) {
    const int64_t pc = 2 * seg_chunks;
    return (n + pc - 1) / pc;
}
// Chunks per warp of the static range (`total` chunks): equal shares, but at least
// ceil(nmax / (kPiecesMax - 2)) (nmax the longest row) so that no row is cut into more than
// kPiecesMax pieces.
__host__ __device__ inline int64_t stats_share(int64_t total, int64_t nmax, int64_t nw) {
    const int64_t lw = (total + nw - 1) / nw;
    const int64_t lmin = (nmax + kPiecesMax - 3) / (kPiecesMax - 2);
    return lw > lmin ? lw : (lmin > 0 ? lmin : 1);
}
// The pieces of a stats row at offset `off` with `len` chunks.  A static row: warps
// first .. first + count - 1, warp gw's partial is piece gw - first; a tail row:
// tail_pieces_per_row fixed pieces.
__device__ __forceinline__ int row_piece_count(bool tail, int64_t off, int64_t len, int64_t lw, int64_t seg_chunks) {
    if (tail) return (int)tail_pieces_per_row(len, seg_chunks);
    const int64_t first = off / lw;
    return (int)((off + len - 1) / lw - first) + 1;
}
// The static range of a call: rs rows of nchunk chunks, or every row (reduced vocabulary).
__device__ __forceinline__ int64_t static_total(const VerifyParams& p, int L, int64_t rs) {
    return p.t2d ? stream_off(p, L) : rs * p.nchunk;
}

template <typename DQ, typename DP, int E>
__global__ void __launch_bounds__(kStatsThreads, kStatsMinBlocks) stats_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) char stats_smem[];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ __align__(8) uint64_t stats_bars[kStatsWarps][kStages];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    StatsRing ring;
    ring.init(stats_smem + warp * (kStages * kStageBytes), stats_bars[warp], lane);
    const int L = valid_prefix(p);
    WsHeader* hdr = ws_header(p);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->L = L;
        // the sweep's work list starts empty in every call, whatever the workspace held (the
        // decide kernel appends only after this grid has completed)
        hdr->ticket_sweep = 0ull;
        hdr->sweep_total = 0ull;
    }
    if (L == 0) return;
    const int64_t n = p.nchunk;
    const bool reduced = p.t2d != nullptr;
    const int64_t rows = 2 * (int64_t)p.cu[L] + L;
    const int64_t rs = static_rows(rows, n, p.stats_warps, reduced);
    const int64_t stot = static_total(p, L, rs);
    const int64_t lw = stats_share(stot, max(n, p.nchunk_q), p.stats_warps);
    const int64_t gw = (int64_t)blockIdx.x * kStatsWarps + warp;
    const int64_t V = p.V;
    int b = 0;
    int64_t gb = 0;
    int Nb = p.cu[1] - p.cu[0];
    // one piece [c, c_end) of row rho into partial slot `slot`
    auto piece = [&](int64_t rho, int64_t c, int64_t c_end, int slot, auto after_last) {
        // a warp's static rows only move forward, but its tail claims wrap around from the last
        // ticket range to the first, so a claimed row may lie before the current stream
        if (rho < gb || rho > gb + 2 * (int64_t)Nb) {
            b = stream_of_row(p, rho, rho < gb ? 0 : b, L);
            gb = 2 * (int64_t)p.cu[b] + b;
            Nb = p.cu[b + 1] - p.cu[b];
        }
        const int64_t j = rho - gb;
        const float T = p.temp[b];
        const bool greedy = (T == 0.f);
        const bool draft = j > Nb;
        if (!temperature_ok(T) || (draft && greedy)) {   // never read
            after_last();
            return;
        }
        float ah = 0.f, al = 0.f;
        if (!greedy) {
            const df a = scale_of_temperature(T);
            ah = a.hi;
            al = a.lo;
        }
        char* blk = row_block(p, rho);
        Part* dst = blk_at<Part>(blk, kOffParts) + slot;
        if (draft)
            stats_piece<DQ, E>(ring, row_ptr<DQ>(p.dq, qrow_of(p, b, p.cu[b], (int)(j - Nb - 1)), p.Kq), c, c_end, false, ah, al,
                               lane, dst, after_last);
        else
            stats_piece<DP, E>(ring, row_ptr<DP>(p.dp, prow_of(p, b, p.cu[b], (int)j), V), c, c_end, greedy, ah, al, lane,
                               dst, after_last);
        if (lane == 0) atomicAdd(blk_at<unsigned>(blk, kOffStatsCount), 1u);   // after lane 0's partial
    };
    auto nothing = []() {};
    // ---- this warp's static share
    int64_t f = gw * lw;
    const int64_t f1 = min(f + lw, stot);
    if (f < f1 && !reduced) {   // rows of one length: row f / n
        int64_t rho = f / n;
        int64_t c = f - rho * n;
        while (f < f1) {
            const int64_t c_end = min(n, c + (f1 - f));
            piece(rho, c, c_end, (int)(gw - rho * n / lw), nothing);
            f += c_end - c;
            c = 0;
            ++rho;
        }
    } else if (f < f1) {        // target and draft rows of different lengths, stream by stream
        int lo = 0, hi = L - 1;   // the stream holding chunk f: the last sb with stream_off(sb) <= f
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (stream_off(p, mid) <= f) lo = mid;
            else hi = mid - 1;
        }
        int sb = lo;
        int Ns = p.cu[sb + 1] - p.cu[sb];
        const int64_t d = f - stream_off(p, sb), tp = (int64_t)(Ns + 1) * n;
        int j = d < tp ? (int)(d / n) : Ns + 1 + (int)((d - tp) / p.nchunk_q);
        int64_t roff = row_off(p, sb, Ns, j);
        int64_t c = f - roff;
        while (f < f1) {
            const int64_t len = row_len(p, Ns, j);
            const int64_t c_end = min(len, c + (f1 - f));
            piece(2 * (int64_t)p.cu[sb] + sb + j, c, c_end, (int)(gw - roff / lw), nothing);
            f += c_end - c;
            c = 0;
            roff += len;
            if (++j > 2 * Ns) {   // the stream's last row: on to the next stream's first
                j = 0;
                if (++sb < L) Ns = p.cu[sb + 1] - p.cu[sb];
            }
        }
    }
    // ---- the tail: fixed pieces claimed one by one from kTailTickets ranges (a warp starts on
    // its own range and moves on when it is used up, so no single counter takes every claim; a
    // plain read skips a used-up range without an atomic).  The next claim is fired once the
    // current piece's last copy is issued, so its round trip overlaps the piece's last stages.
    const int64_t pc = 2 * p.seg_chunks;
    const int64_t npd = tail_pieces_per_row(n, p.seg_chunks);
    const unsigned long long total = (unsigned long long)(rows - rs) * (unsigned long long)npd;
    const unsigned long long per_range = (total + kTailTickets - 1) / kTailTickets;
    const int home = (int)(gw % kTailTickets);
    unsigned long long next = total;
    auto claim = [&]() {   // all lanes: lanes 0..kTailTickets-1 read one ticket each (one round trip)
        const int rg = (home + lane) % kTailTickets;
        const unsigned long long lo = (unsigned long long)rg * per_range;
        const unsigned long long span = (lo < total) ? min(per_range, total - lo) : 0ull;
        const bool open = lane < kTailTickets && __ldcg(&hdr->ticket_stats[rg]) < span;
        unsigned mask = __ballot_sync(0xffffffffu, open);
        next = total;
        while (mask) {   // the first open range, from this warp's home range on
            const int l = __ffs(mask) - 1;
            unsigned long long got = 0;
            if (lane == l) got = atomicAdd(&hdr->ticket_stats[rg], 1ull);
            got = __shfl_sync(0xffffffffu, got, l);
            const unsigned long long lo_l = __shfl_sync(0xffffffffu, lo, l);
            const unsigned long long span_l = __shfl_sync(0xffffffffu, span, l);
            if (got < span_l) {
                next = lo_l + got;
                break;
            }
            mask &= mask - 1;
        }
    };
    claim();
    unsigned long long cur = __shfl_sync(0xffffffffu, next, 0);
    while (cur < total) {
        const int64_t rho = rs + (int64_t)(cur / (unsigned long long)npd);
        const int k = (int)(cur % (unsigned long long)npd);
        const int64_t c = (int64_t)k * pc;
        piece(rho, c, min(n, c + pc), k, claim);
        cur = __shfl_sync(0xffffffffu, next, 0);
    }
    // no TMA copy of this warp may still be writing its ring when the CTA leaves
    ring.drain();
}

// ---------------------------------------------------------------------------------------
// decide_kernel: one CTA per stream
// ---------------------------------------------------------------------------------------
// Part index of a stream's rows inside the per-stream kernels: draft row i -> i (i < N),
// target row i -> N + i (i <= N); stats row of part r: g_b + N + 1 + r (draft), g_b + r - N
// (target).
__device__ __forceinline__ int64_t stats_row_of_part(int64_t gb, int N, int r) {
    return gb + (r < N ? N + 1 + r : r - N);
}

struct DecideShared {
    float rowK[kMaxRows];
    df rowZ[kMaxRows];
    int rowArg[kMaxRows];
    df rho[SPEC_MAX_KMAX];
    df w[SPEC_MAX_KMAX + 1];
    df u_acc[SPEC_MAX_KMAX + 1];
    float cval[SPEC_MAX_KMAX + 1];
    float lq[SPEC_MAX_KMAX], lp[SPEC_MAX_KMAX];
    int x[SPEC_MAX_KMAX];
    int pass_list[SPEC_MAX_KMAX + 1];
    int n_pass, status, tau, bonus;
    unsigned long long claim0;
};

template <typename DQ, typename DP>
__global__ void __launch_bounds__(kThreads) decide_kernel(const VerifyParams p) {
    __shared__ DecideShared sh;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // ---- prologue (inputs only, overlaps the stats kernel): temperature, uniforms, and -
    // once the stream's offsets are known to be valid - its tokens and the logits at them
    const float T = p.temp[b];
    const bool temp_ok = temperature_ok(T);
    const bool greedy = (T == 0.f);
    const df a = (temp_ok && !greedy) ? scale_of_temperature(T) : df{0.f, 0.f};
    if (tid <= p.kmax && temp_ok && !greedy) {
        const uint64_t stp = step_of(p);
        const uint4 c = make_uint4((uint32_t)tid, (uint32_t)b, (uint32_t)stp, (uint32_t)(stp >> 32));
        const uint4 wds = philox4x32_10(c, make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
        sh.u_acc[tid] = uniform24_df(wds.x);
    }
    if (tid <= SPEC_MAX_KMAX) sh.w[tid] = df{__int_as_float(0x7fffffff), 0.f};
    // the valid stream prefix [0, L) (the stats grid computes the same from the same inputs) and,
    // from it, the stats partition: all before the wait, while the stats grid streams
    const int L = valid_prefix(p);
    const bool offsets_ok = b < L;   // no stream j <= b breaks the packed layout
    const int64_t rs = static_rows(2 * (int64_t)p.cu[L] + L, p.nchunk, p.stats_warps, p.t2d != nullptr);
    const int64_t lw = stats_share(static_total(p, L, rs), max(p.nchunk, p.nchunk_q), p.stats_warps);
    const int base = p.cu[b];
    const int N = offsets_ok ? p.cu[b + 1] - base : 0;
    const int64_t V = p.V;
    bool bad_tok = false;
    if (offsets_ok && temp_ok && tid < N) {
        const int xi = p.tokens[qrow_of(p, b, base, tid)];
        sh.x[tid] = xi;
        bad_tok = (xi < 0 || xi >= p.V);
        if (!bad_tok && !greedy) {
            sh.lq[tid] = draft_logit_at<DQ>(p, row_ptr<DQ>(p.dq, qrow_of(p, b, base, tid), p.Kq), xi);
            sh.lp[tid] = load_elem<DP>(row_ptr<DP>(p.dp, prow_of(p, b, base, tid), V), xi);
        }
    }
    bad_tok = __syncthreads_or(bad_tok);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    WsHeader* hdr = ws_header(p);
    if (!offsets_ok) return;   // finish_kernel reports BAD_OFFSETS
    const int64_t gb = 2 * (int64_t)base + b;
    const int nrows = 2 * N + 1;
    const bool reduce_rows = temp_ok && !bad_tok;

    // ---- row statistics from the pieces' partials: one warp per row, lane l holds piece l
    // (same order every time, so the result is reproducible bit for bit)
    bool stats_to = false;
    if (temp_ok) {
        for (int r = (greedy ? N : 0) + warp; r < nrows; r += kWarps) {
            const int64_t rho = stats_row_of_part(gb, N, r);
            char* blk = row_block(p, rho);
            const int cnt_want = row_piece_count(rho >= rs, row_off(p, b, N, (int)(rho - gb)), row_len(p, N, (int)(rho - gb)),
                                                 lw, p.seg_chunks);
            const unsigned cnt = __ldcg(blk_at<unsigned>(blk, kOffStatsCount));
            Part e[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int pk = lane + 32 * k;
                e[k] = Part{greedy ? -kInf : kNoRef, 0.f, 0.f, INT_MAX};
                if (pk < cnt_want) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(blk_at<Part>(blk, kOffParts) + pk));
                    e[k] = Part{v.x, v.y, v.z, __float_as_int(v.w)};
                }
            }
            const bool full = (cnt == (unsigned)cnt_want);
            stats_to |= __any_sync(0xffffffffu, !full || e[0].idx == kStatsTimeout || e[1].idx == kStatsTimeout);
            if (!reduce_rows || !full) continue;
            if (greedy) {
                const float Kr = warp_max_nan(fmax_nan(e[0].K, e[1].K));
                const int arg = warp_min_i(min(e[0].K == Kr ? e[0].idx : INT_MAX, e[1].K == Kr ? e[1].idx : INT_MAX));
                if (lane == 0) {
                    sh.rowK[r] = Kr;
                    sh.rowArg[r] = arg;
                    sh.rowZ[r] = df{0.f, 0.f};
                }
                continue;
            }
            const float Kr = warp_max(fmaxf(e[0].K, e[1].K));
            df z{0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 2; ++k)
                z = df_add(z, df_scale(df{e[k].s_hi, e[k].s_lo}, (e[k].K == Kr) ? 1.f : pow2_int(e[k].K - Kr)));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const df other{__shfl_xor_sync(0xffffffffu, z.hi, o), __shfl_xor_sync(0xffffffffu, z.lo, o)};
                z = df_add(z, other);
            }
            if (lane == 0) {
                sh.rowK[r] = Kr;
                sh.rowZ[r] = z;
                sh.rowArg[r] = INT_MAX;
            }
        }
    }
    stats_to = __syncthreads_or(stats_to);
    // the stream's counters go back to zero for the next call (every row, read or not)
    for (int r = tid; r < nrows; r += kThreads) *blk_at<unsigned>(row_block(p, gb + r), kOffStatsCount) = 0u;
    if (tid == 0) {
        *blk_at<unsigned>(row_block(p, gb), kOffSweepCount) = 0u;
        *blk_at<unsigned>(row_block(p, gb), kOffSweepTimeout) = 0u;
        int st = SPEC_ST_OK;
        if (!temp_ok) st = SPEC_ST_BAD_TEMPERATURE;
        else if (bad_tok) st = SPEC_ST_BAD_TOKEN;
        else if (stats_to) st = SPEC_ST_TIMEOUT;
        sh.status = st;
        sh.tau = 0;
        sh.n_pass = 0;
        sh.bonus = 0;
    }
    __syncthreads();

    // ---- validity of the rows read, q_i(x_i) > 0, per-slot ratios
    if (sh.status == SPEC_ST_OK) {
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
                const df e = df_sub(exponent_df(lp, a.hi, a.lo, Kp), exponent_df(lq, a.hi, a.lo, Kq));
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

    // ---- decisions
    const df one{1.f, 0.f};
    if (tid == 0 && sh.status == SPEC_ST_OK) {
        int n = 0, tau = 0;
        if (greedy) {
            tau = N;
            for (int i = 0; i < N; ++i)
                if (sh.rowArg[N + i] != sh.x[i]) {
                    tau = i;
                    break;
                }
        } else if (p.rule == 1) {
            sh.w[0] = one;
            for (int i = 0; i < N; ++i) sh.w[i + 1] = df_min(one, df_mul(sh.w[i], sh.rho[i]));
            if (N > 0 && df_le(sh.u_acc[N - 1], sh.w[N])) {
                tau = N;   // eta_N <= w_N = h_N: accept everything, no residual needed
            } else {
                for (int i = N - 1; i >= 1; --i)   // candidates: eta_i <= w_i (h_i <= w_i)
                    if (df_le(sh.u_acc[i - 1], sh.w[i])) sh.pass_list[n++] = i;
                if (N > 0) sh.pass_list[n++] = 0;
            }
        } else {
            tau = N;
            for (int i = 0; i < N; ++i)
                if (!df_le(sh.u_acc[i], df_min(one, sh.rho[i]))) {
                    tau = i;
                    break;
                }
            if (tau < N) {
                sh.w[tau] = one;
                sh.pass_list[n++] = tau;
            }
        }
        if (!greedy && tau == N) {   // every draft accepted: the sweep sums the bonus row instead
            sh.pass_list[0] = N;
            n = 1;
            sh.bonus = 1;
        }
        sh.tau = tau;
        sh.n_pass = n;
    }
    __syncthreads();
    int np = sh.n_pass;
    if (tid < np && !sh.bonus) {
        const int i = sh.pass_list[tid];
        sh.cval[i] = df_to_f(df_div(df_mul(sh.w[i], sh.rowZ[i]), sh.rowZ[N + i]));
    }
    // this stream's sweep claims: np items x ncl runs of kSegsPerClaim segments
    const int ncl = (p.nseg + kSegsPerClaim - 1) / kSegsPerClaim;
    if (tid == 0) {
        sh.claim0 = np > 0 ? atomicAdd(&hdr->sweep_total, (unsigned long long)(np * ncl)) : 0ull;
        // every stream appends at most (kmax + 1) ncl claims, so the list never overflows; the
        // bound is kept anyway, and a stream that would cross it reports TIMEOUT
        if (np > 0 && sh.claim0 + (unsigned long long)(np * ncl) > work_list_claims(p.B, p.kmax)) {
            sh.status = SPEC_ST_TIMEOUT;
            sh.n_pass = 0;
        }
    }
    __syncthreads();

    // ---- records for the sweep and finish kernels
    const bool ok = sh.status == SPEC_ST_OK;
    np = sh.n_pass;
    if (ok) {
        for (int r = (greedy ? N : 0) + tid; r < nrows; r += kThreads) {
            RowStat* rs = blk_at<RowStat>(row_block(p, stats_row_of_part(gb, N, r)), kOffRow);
            *rs = RowStat{sh.rowK[r], sh.rowZ[r].hi, sh.rowZ[r].lo, sh.rowArg[r]};
        }
        if (tid <= N) {
            SlotRec* sr = blk_at<SlotRec>(row_block(p, gb + tid), kOffSlot);
            const df qnan{__int_as_float(0x7fffffff), 0.f};
            sr->rho = (!greedy && tid < N) ? sh.rho[tid] : qnan;
            sr->w = sh.w[tid];
            sr->h = qnan;
            sr->r = qnan;
            sr->cval = sh.cval[tid];
            sr->x = tid < N ? sh.x[tid] : -1;
            sr->lq = (!greedy && tid < N) ? sh.lq[tid] : 0.f;
            sr->lp = (!greedy && tid < N) ? sh.lp[tid] : 0.f;
        }
        SweepItem* list = work_list(p);
        for (int t = tid; t < np * ncl; t += kThreads) {
            const int i = sh.pass_list[t / ncl];
            const bool bonus = sh.bonus != 0;
            list[sh.claim0 + t] = SweepItem{b,
                                            (int16_t)i,
                                            (int16_t)((t % ncl) * kSegsPerClaim),
                                            bonus ? 0.f : sh.rowK[i],
                                            sh.rowK[N + i],
                                            bonus ? 1.f : sh.cval[i],
                                            a.hi,
                                            a.lo,
                                            bonus ? 1 : 0};
        }
    }
    if (tid == 0) {
        StreamRec* srec = blk_at<StreamRec>(row_block(p, gb), kOffStream);
        srec->status = sh.status;
        srec->N = N;
        srec->greedy = greedy ? 1 : 0;
        srec->tau = sh.tau;
        srec->n_pass = ok ? np : 0;
        srec->bonus = sh.bonus;
        srec->a_hi = a.hi;
        srec->a_lo = a.lo;
        for (int i = 0; i < np; ++i) srec->pass[i] = (uint8_t)sh.pass_list[i];
    }
}

// ---------------------------------------------------------------------------------------
// sweep_kernel: residual (or bonus) sums of every stream's sweep items, spread over the GPU
// ---------------------------------------------------------------------------------------
// A stage is G chunks of both rows of an item (q and p; p alone for the bonus row).  The
// vector path (E = 8, 16-byte aligned rows) moves a stage with one TMA bulk copy per row into a
// per-warp ring of D stages, each completing on its own mbarrier (lane 0 issues, every lane
// waits with a bounded poll); the plain path (E = 1) loads chunk by chunk.
template <typename DQ, typename DP, int E>
struct SweepRing;

template <typename DQ, typename DP>
struct SweepRing<DQ, DP, 8> {
    static constexpr int BQ = 8 * (int)sizeof(DQ);
    static constexpr int BP = 8 * (int)sizeof(DP);
    static constexpr int G = 2048 / (BQ > BP ? BQ : BP);   // chunks per stage and row
    static constexpr int ROWQ = G * BQ;
    static constexpr int STAGE = G * (BQ + BP);
    static constexpr int D = 3;
    static constexpr int RING = D * STAGE + 64;   // bytes per warp (stages + barriers)
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
    // chunks [c0, c0 + n) of both rows into ring slot `slot` (rq null: p only)
    __device__ __forceinline__ void issue(int slot, const void* rq, const void* rp, int64_t c0, int n) {
        if (timeout || n <= 0) return;   // after a failed wait nothing new is put in flight
        pending |= 1u << slot;
        __syncwarp();                    // every lane is done reading this slot's previous stage
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&bar[slot], (unsigned)(n * ((rq ? BQ : 0) + BP)));
            if (rq)
                bulk_g2s_hint(base + slot * STAGE, reinterpret_cast<const char*>(rq) + c0 * BQ, (unsigned)(n * BQ),
                              &bar[slot], l2_evict_first_policy());
            bulk_g2s_hint(base + slot * STAGE + ROWQ, reinterpret_cast<const char*>(rp) + c0 * BP, (unsigned)(n * BP),
                          &bar[slot], l2_evict_first_policy());
        }
    }
    __device__ __forceinline__ void wait(int slot, int n) {
        if (timeout || n <= 0) return;
        const unsigned parity = (phase >> slot) & 1u;
        bool ok = true;
        for (int k = 0; !mbar_try_wait(&bar[slot], parity);)
            if (++k > kSpinLimit) {
                ok = false;
                break;
            }
        timeout = !__all_sync(0xffffffffu, ok);   // one decision for the whole warp
        if (timeout) return;                       // the slot stays pending; drain() waits for it once more
        phase ^= 1u << slot;
        pending &= ~(1u << slot);
    }
    // before the CTA exits: wait (bounded) for any copy still in flight after a failed wait
    __device__ __forceinline__ void drain() {
        for (int slot = 0; slot < D; ++slot) {
            if (!((pending >> slot) & 1u)) continue;
            const unsigned parity = (phase >> slot) & 1u;
            for (int k = 0; k < kSpinLimit && !mbar_try_wait(&bar[slot], parity); ++k) {
            }
        }
    }
    __device__ __forceinline__ void get(int slot, int kk, const void*, const void*, int64_t, bool has_q,
                                        float (&xq)[8], float (&xp)[8]) const {
        if (has_q) unpack<DQ>(base + slot * STAGE + kk * BQ, xq);
        unpack<DP>(base + slot * STAGE + ROWQ + kk * BP, xp);
    }
    template <typename T>
    __device__ __forceinline__ static void unpack(const char* s, float (&x)[8]) {
        if constexpr (sizeof(T) == 2) {
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
struct SweepRing<DQ, DP, 1> {
    static constexpr int G = 128;
    static constexpr int D = 1;
    static constexpr int RING = 0;
    bool timeout;
    __device__ __forceinline__ void init(char*, int) { timeout = false; }
    __device__ __forceinline__ void issue(int, const void*, const void*, int64_t, int) {}
    __device__ __forceinline__ void wait(int, int) {}
    __device__ __forceinline__ void drain() {}
    __device__ __forceinline__ void get(int, int kk, const void* rq, const void* rp, int64_t c0, bool has_q,
                                        float (&xq)[1], float (&xp)[1]) const {
        if (has_q) xq[0] = load_elem<DQ>(rq, c0 + kk);
        xp[0] = load_elem<DP>(rp, c0 + kk);
    }
};

// Sums of segments [s0, s1) of one item into seg_out[s0 .. s1): max(0, c 2^(lp a - Kp) -
// 2^(lq a - Kq)) for a residual item, 2^(lp a - Kp) for the bonus row.  Stages never straddle
// a segment; each segment's lane sums enter a Kahan sum stage by stage and are combined across
// the warp in double-float.  after_last() runs in every lane right after the last copy.
template <typename DQ, typename DP, int E, typename AfterFn>
__device__ __forceinline__ void sweep_segments(SweepRing<DQ, DP, E>& R, const VerifyParams& p, const void* rq,
                                               const void* rp, int s0, int s1, float Kq, float Kp, float ah,
                                               float al, float cc, bool bonus, int lane, float* seg_out,
                                               AfterFn after_last) {
    using Ring = SweepRing<DQ, DP, E>;
    constexpr int G = Ring::G, D = Ring::D;
    const int64_t sc = p.seg_chunks;
    const int mps = (int)((sc + G - 1) / G);   // stages per segment
    const int nst = (s1 - s0) * mps;
    auto stage = [&](int t, int64_t& c0, int& n) {
        const int s = s0 + t / mps, m = t % mps;
        const int64_t seg_end = min(p.nchunk, (int64_t)(s + 1) * sc);
        c0 = (int64_t)s * sc + (int64_t)m * G;
        const int64_t left = seg_end - c0;
        n = left <= 0 ? 0 : (int)(left < G ? left : G);
    };
    const bool gather_q = !bonus && p.t2d != nullptr;   // reduced draft vocabulary: q is gathered
    const void* q = (bonus || gather_q) ? nullptr : rq;
    auto issue = [&](int t) {
        if (t < nst) {
            int64_t c0;
            int n;
            stage(t, c0, n);
            R.issue(t % D, q, rp, c0, n);
            if (t == nst - 1) after_last();
        }
    };
    for (int t = 0; t < D - 1; ++t) issue(t);
    // reduced draft vocabulary: the draft chunks of a stage are gathered through the column
    // map, all of a lane's at once, one stage ahead (in flight while the stage before is summed)
    constexpr int UQ = (G + 31) / 32;
    Chunk<DQ, E> cq_cur[UQ], cq_nxt[UQ];
    auto gather_stage = [&](int t, Chunk<DQ, E>(&cq)[UQ]) {
        int64_t c0;
        int n;
        stage(t, c0, n);
#pragma unroll
        for (int u = 0; u < UQ; ++u)
            if (lane + 32 * u < n) cq[u].gather(rq, p.t2d, p.Kq, c0 + lane + 32 * u);
    };
    if (gather_q && nst > 0) gather_stage(0, cq_cur);
    Kahan acc;
    for (int t = 0; t < nst; ++t) {
        issue(t + D - 1);
        int64_t c0;
        int n;
        stage(t, c0, n);
        if (gather_q && t + 1 < nst) gather_stage(t + 1, cq_nxt);
        R.wait(t % D, n);
        float grp = 0.f;   // this lane's chunk sums of the stage (independent), added once
        if (gather_q) {
#pragma unroll
            for (int u = 0; u < UQ; ++u) {
                const int kk = lane + 32 * u;
                if (kk < n) {
                    float xq[E], xp[E];
                    R.get(t % D, kk, rq, rp, c0, false, xq, xp);
                    cq_cur[u].unpack(xq);
                    grp += resid_chunk_sum<E>(xq, xp, Kq, Kp, ah, al, cc);
                }
            }
#pragma unroll
            for (int u = 0; u < UQ; ++u) cq_cur[u] = cq_nxt[u];
        } else {
            for (int kk = lane; kk < n; kk += 32) {
                float xq[E], xp[E];
                R.get(t % D, kk, rq, rp, c0, !bonus, xq, xp);
                grp += bonus ? target_chunk_sum<E>(xp, Kp, ah, al) : resid_chunk_sum<E>(xq, xp, Kq, Kp, ah, al, cc);
            }
        }
        acc.add(grp);
        if (t % mps == mps - 1) {   // the segment is complete
            df tot = acc.value();
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const df other{__shfl_xor_sync(0xffffffffu, tot.hi, o), __shfl_xor_sync(0xffffffffu, tot.lo, o)};
                tot = df_add(tot, other);
            }
            if (lane == 0) seg_out[s0 + t / mps] = df_to_f(tot);
            acc = Kahan();
        }
    }
    if (nst == 0) after_last();
}

template <typename DQ, typename DP, int E>
__global__ void __launch_bounds__(kThreads, 2) sweep_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) char ring_smem[];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    SweepRing<DQ, DP, E> ring;
    ring.init(ring_smem + warp * SweepRing<DQ, DP, E>::RING, lane);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    WsHeader* hdr = ws_header(p);
    const unsigned long long cap = work_list_claims(p.B, p.kmax);
    const unsigned long long appended = __ldcg(&hdr->sweep_total);
    const unsigned long long total = appended < cap ? appended : cap;
    const SweepItem* list = work_list(p);
    const int64_t V = p.V;
    // a claim's entry: 32 bytes, lanes 0..7 hold one 32-bit word each
    auto load_entry = [&](unsigned long long id) -> int {
        return (lane < 8 && id < total) ? __ldcg(reinterpret_cast<const int*>(list + id) + lane) : 0;
    };
    // warp gw's first claim is gw itself; later claims come from the ticket, offset by the
    // number of warps
    const unsigned long long W = (unsigned long long)gridDim.x * kWarps;
    unsigned long long claim = 0;
    unsigned long long cur = (unsigned long long)blockIdx.x * kWarps + warp;
    int word = load_entry(cur);
    while (cur < total) {
        const int b = __shfl_sync(0xffffffffu, word, 0);
        const int w1 = __shfl_sync(0xffffffffu, word, 1);
        const int i = (int)(int16_t)(w1 & 0xffff), s0 = (w1 >> 16) & 0xffff;
        const float Kq = __int_as_float(__shfl_sync(0xffffffffu, word, 2));
        const float Kp = __int_as_float(__shfl_sync(0xffffffffu, word, 3));
        const float cc = __int_as_float(__shfl_sync(0xffffffffu, word, 4));
        const float ah = __int_as_float(__shfl_sync(0xffffffffu, word, 5));
        const float al = __int_as_float(__shfl_sync(0xffffffffu, word, 6));
        const bool bonus = __shfl_sync(0xffffffffu, word, 7) != 0;
        if (lane == 0) claim = W + atomicAdd(&hdr->ticket_sweep, 1ull);   // the next claim, in flight
        unsigned long long nxt = total;
        int nword = 0;
        const int64_t gb = 2 * (int64_t)p.cu[b] + b;
        const void* rq = bonus ? nullptr : row_ptr<DQ>(p.dq, qrow_of(p, b, p.cu[b], i), p.Kq);
        const void* rp = row_ptr<DP>(p.dp, prow_of(p, b, p.cu[b], i), V);
        const int s1 = min(p.nseg, s0 + kSegsPerClaim);
        // once this claim's last copy is issued: the next claim's entry is loaded while the
        // rest of this one is summed
        sweep_segments<DQ, DP, E>(ring, p, rq, rp, s0, s1, Kq, Kp, ah, al, cc, bonus, lane,
                                  blk_at<float>(row_block(p, gb + i), kOffSeg), [&]() {
                                      nxt = __shfl_sync(0xffffffffu, claim, 0);
                                      nword = load_entry(nxt);
                                  });
        if (lane == 0) {
            char* sblk = row_block(p, gb);
            if (ring.timeout) atomicExch(blk_at<unsigned>(sblk, kOffSweepTimeout), 1u);
            atomicAdd(blk_at<unsigned>(sblk, kOffSweepCount), (unsigned)(s1 - s0));
        }
        cur = nxt;
        word = nword;
    }
    // no TMA copy of this warp may still be writing its ring when the CTA leaves
    ring.drain();
}

// ---------------------------------------------------------------------------------------
// finish_kernel: one CTA per stream - r_i, h_i, tau, the draw, the outputs
// ---------------------------------------------------------------------------------------
struct FinishShared {
    float rowK[kMaxRows];
    df rowZ[kMaxRows];
    int rowArg[kMaxRows];
    df rho[SPEC_MAX_KMAX];
    df w[SPEC_MAX_KMAX + 1];
    df h[SPEC_MAX_KMAX + 1];
    df r[SPEC_MAX_KMAX + 1];
    df u_acc[SPEC_MAX_KMAX + 1];
    uint32_t u_smp[SPEC_MAX_KMAX + 1];
    float cval[SPEC_MAX_KMAX + 1];
    float lq[SPEC_MAX_KMAX], lp[SPEC_MAX_KMAX];
    int x[SPEC_MAX_KMAX];
    int pass_list[SPEC_MAX_KMAX + 1];
    int N, n_pass, status, greedy, tau, bonus, sample_seg;
    unsigned long long sample_t;                 // in-segment target (fixed point)
    unsigned long long sub_sum[kWarps];          // the drawn segment split over the warps
    int sub_last[kWarps];
    float sample_scale;                          // fixed-point scale of the draw's weights
    float a_hi, a_lo;
    unsigned sweep_count, sweep_timeout;
    float seg[SPEC_MAX_KMAX + 1][kSegs];         // every slot's segment sums (swept slots hold data)
};

// The draw's last two steps over the drawn segment [s0, s1): every warp sums an eighth of it
// in fixed point, and the warp whose eighth crosses the target rescans that eighth (from the
// weights it already holds when the eighth is at most 64 chunks, else by reading it again).
// The token is written to out_tok[slot_out] by the thread that found it.
template <typename DQ, typename DP, int E, bool BONUS>
__device__ __forceinline__ void draw_in_segment(const VerifyParams& p, FinishShared& sh, const void* rq, const void* rp,
                                                int64_t s0, int64_t s1, float Kq, float Kp, float ah, float al,
                                                float cc, int warp, int lane, int64_t slot_out) {
    const int64_t msub = (s1 - s0 + kWarps - 1) / kWarps;
    const int64_t w0 = min(s1, s0 + warp * msub), w1 = min(s1, w0 + msub);
    const bool held = msub <= 64;
    DrawSlice<DQ, DP, E, BONUS> slice;
    unsigned long long sub;
    int last;
    if (held) {
        slice.load(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, lane, p.t2d, p.Kq);
        slice.sum(sub, last);
    } else {
        segment_fixed_sum<DQ, DP, E, BONUS>(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, lane, sub, last,
                                            p.t2d, p.Kq);
    }
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
        y = held ? slice.rescan(t - before, lane)
                 : rescan_segment<DQ, DP, E, BONUS>(rq, rp, w0, w1, Kq, Kp, ah, al, cc, sh.sample_scale, t - before,
                                                    lane, p.t2d, p.Kq);
    }
    if ((wsel < 0 && threadIdx.x == 0) || (warp == wsel && lane == 0)) p.out_tok[slot_out] = y;
}

template <typename DQ, typename DP, int E>
__global__ void __launch_bounds__(kThreads) finish_kernel(const VerifyParams p) {
    __shared__ FinishShared sh;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = p.V;
    const int64_t ob = (int64_t)b * (p.kmax + 1);
    // ---- prologue (inputs only): the per-slot uniforms and the stream's offsets
    if (tid <= p.kmax) {
        const uint64_t stp = step_of(p);
        const uint4 c = make_uint4((uint32_t)tid, (uint32_t)b, (uint32_t)stp, (uint32_t)(stp >> 32));
        const uint4 wds = philox4x32_10(c, make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
        sh.u_acc[tid] = uniform24_df(wds.x);
        sh.u_smp[tid] = wds.y;
        sh.h[tid] = df{__int_as_float(0x7fffffff), 0.f};
        sh.r[tid] = df{__int_as_float(0x7fffffff), 0.f};
    }
    const int base = p.cu[b];
    const int n_raw = p.cu[b + 1] - base;
    const int L = valid_prefix(p);   // as the stats grid computed it, from the same inputs
    asm volatile("griddepcontrol.wait;" ::: "memory");
    WsHeader* hdr = ws_header(p);
    if (b == 0 && tid == 0) {   // every earlier grid of the call has finished: tickets back to zero
        for (int i = 0; i < kTailTickets; ++i) hdr->ticket_stats[i] = 0ull;
        hdr->ticket_sweep = 0ull;
        hdr->sweep_total = 0ull;
    }
    if (b >= L) {
        for (int j = tid; j <= p.kmax; j += kThreads) p.out_tok[ob + j] = -1;
        if (tid == 0) {
            p.status[b] = SPEC_ST_BAD_OFFSETS;
            p.acc_len[b] = 0;
            p.n_emit[b] = 0;
        }
        return;
    }
    const int N = n_raw;
    const int64_t gb = 2 * (int64_t)base + b;
    const int nrows = 2 * N + 1;
    char* sblk = row_block(p, gb);
    // ---- one round of loads: the stream's record, every row's statistics, every slot's
    // scalars and segment sums (decide_kernel wrote the records of every OK stream; the
    // segment sums of slots that were not swept are not used)
    if (tid == 0) {
        const StreamRec* sr = blk_at<StreamRec>(sblk, kOffStream);
        sh.status = __ldcg(&sr->status);
        sh.N = N;
        sh.greedy = __ldcg(&sr->greedy);
        sh.tau = __ldcg(&sr->tau);
        sh.n_pass = __ldcg(&sr->n_pass);
        sh.bonus = __ldcg(&sr->bonus);
        sh.a_hi = __ldcg(&sr->a_hi);
        sh.a_lo = __ldcg(&sr->a_lo);
        const int4 pl[3] = {__ldcg(reinterpret_cast<const int4*>(sr->pass)),
                            __ldcg(reinterpret_cast<const int4*>(sr->pass) + 1),
                            __ldcg(reinterpret_cast<const int4*>(sr->pass) + 2)};
        const unsigned char* pb = reinterpret_cast<const unsigned char*>(pl);
        for (int i = 0; i <= SPEC_MAX_KMAX; ++i) sh.pass_list[i] = pb[i];
        sh.sweep_count = __ldcg(blk_at<unsigned>(sblk, kOffSweepCount));
        sh.sweep_timeout = __ldcg(blk_at<unsigned>(sblk, kOffSweepTimeout));
        sh.sample_seg = -1;
    }
    for (int r = tid; r < nrows; r += kThreads) {
        const RowStat* rs = blk_at<RowStat>(row_block(p, stats_row_of_part(gb, N, r)), kOffRow);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(rs));
        sh.rowK[r] = v.x;
        sh.rowZ[r] = df{v.y, v.z};
        sh.rowArg[r] = __float_as_int(v.w);
    }
    if (tid <= N) {
        const SlotRec* sr = blk_at<SlotRec>(row_block(p, gb + tid), kOffSlot);
        if (tid < N) {
            sh.rho[tid] = df{__ldcg(&sr->rho.hi), __ldcg(&sr->rho.lo)};
            sh.x[tid] = __ldcg(&sr->x);
            sh.lq[tid] = __ldcg(&sr->lq);
            sh.lp[tid] = __ldcg(&sr->lp);
        }
        sh.w[tid] = df{__ldcg(&sr->w.hi), __ldcg(&sr->w.lo)};
        sh.cval[tid] = __ldcg(&sr->cval);
    }
    for (int t = tid; t < (N + 1) * p.nseg; t += kThreads) {
        const int i = t / p.nseg, sg = t - i * p.nseg;
        sh.seg[i][sg] = __ldcg(blk_at<const float>(row_block(p, gb + i), kOffSeg) + sg);
    }
    __syncthreads();
    if (tid == 0) {
        if (sh.status == SPEC_ST_OK && !sh.greedy && sh.n_pass > 0) {
            if (sh.sweep_timeout != 0u || sh.sweep_count != (unsigned)(sh.n_pass * p.nseg))
                sh.status = SPEC_ST_TIMEOUT;
            *blk_at<unsigned>(sblk, kOffSweepCount) = 0u;   // back to zero for the next call
            *blk_at<unsigned>(sblk, kOffSweepTimeout) = 0u;
        }
    }
    __syncthreads();
    const bool greedy = sh.greedy != 0;
    const float ah = sh.a_hi, al = sh.a_lo;
    const df one{1.f, 0.f};
    const bool block = (p.rule == 1);
    auto qrow = [&](int i) { return row_ptr<DQ>(p.dq, qrow_of(p, b, base, i), p.Kq); };
    auto prow = [&](int i) { return row_ptr<DP>(p.dp, prow_of(p, b, base, i), V); };

    if (sh.status == SPEC_ST_OK && !greedy && sh.n_pass > 0) {
        const int np = sh.n_pass;
        const bool bonus_sweep = sh.bonus != 0;
        // ---- r_i = (sum of the item's segment sums) / Z_q, per item (same order every time)
        for (int it = warp; it < np && !bonus_sweep; it += kWarps) {
            const int i = sh.pass_list[it];
            df tot{0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kSegLanes; ++k) {
                const int sg = lane + 32 * k;
                tot = df_add_f(tot, sg < p.nseg ? sh.seg[i][sg] : 0.f);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const df other{__shfl_xor_sync(0xffffffffu, tot.hi, o), __shfl_xor_sync(0xffffffffu, tot.lo, o)};
                tot = df_add(tot, other);
            }
            if (lane == 0) {
                const df ri = df_div(tot, sh.rowZ[i]);
                sh.r[i] = ri;
                if (block && i >= 1) {
                    const df den = df_add(ri, df_sub(one, sh.w[i]));
                    sh.h[i] = df_is_zero(den) ? one : df_div(ri, den);
                }
            }
        }
        __syncthreads();
        if (tid == 0 && block && !bonus_sweep) {
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

        // ---- the draw: 64-bit fixed-point CDF over the drawn item's segments (warp 0); lane l
        // holds segments l, l + 32, ...: the scan runs block by block, each block's inclusive
        // prefix plus the total of the blocks before it
        if (warp == 0) {
            const int tau = sh.tau;
            float wv[kSegLanes];
            float wm = 0.f;
#pragma unroll
            for (int k = 0; k < kSegLanes; ++k) {
                const int sg = lane + 32 * k;
                wv[k] = sg < p.nseg ? sh.seg[tau][sg] : 0.f;
                wm = fmaxf(wm, wv[k]);
            }
            const float wmax = warp_max(wm);
            const bool ok = isfinite(wmax) && wmax > 0.f;
            const float scale = ok ? fixed_scale(wmax) : 0.f;
            unsigned long long q[kSegLanes], pre[kSegLanes];   // weights, inclusive prefix sums
            unsigned long long carry = 0;
#pragma unroll
            for (int k = 0; k < kSegLanes; ++k) {
                q[k] = ok ? __float2ull_rn(wv[k] * scale) : 0ull;
                unsigned long long v = q[k];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += n;
                }
                pre[k] = v + carry;
                carry = __shfl_sync(0xffffffffu, pre[k], 31);
            }
            const unsigned long long R = carry;
            // t = floor(U R), U = (2k + 1) 2^-25 with k the word's top 24 bits
            const unsigned long long odd = 2ull * (sh.u_smp[tau] >> 8) + 1ull;
            const unsigned long long t = (__umul64hi(odd, R) << 39) | ((odd * R) >> 25);
            int sg = -1;
            unsigned long long excl = 0;
#pragma unroll
            for (int k = 0; k < kSegLanes; ++k) {
                const unsigned hit = __ballot_sync(0xffffffffu, q[k] > 0 && pre[k] > t);
                if (sg < 0 && hit) {
                    const int src = __ffs(hit) - 1;
                    sg = 32 * k + src;
                    excl = __shfl_sync(0xffffffffu, pre[k] - q[k], src);
                }
            }
            if (lane == 0) {
                if (ok && R > 0 && sg >= 0) {
                    sh.sample_t = t - excl;
                    sh.sample_scale = scale;
                    sh.sample_seg = sg;
                } else {
                    sh.status = SPEC_ST_NUMERIC;
                    sh.sample_seg = -1;
                }
            }
        }
        __syncthreads();

        // ---- the rescan of the drawn segment, split over the warps: each warp sums an eighth in
        // fixed point, the eighth that crosses the target is rescanned
        if (sh.status == SPEC_ST_OK && sh.sample_seg >= 0) {
            const int tau = sh.tau;
            const bool bonus = (tau == N);
            const void* rq = bonus ? nullptr : qrow(tau);
            const void* rp = prow(tau);
            const float Kq = bonus ? 0.f : sh.rowK[tau], Kp = sh.rowK[N + tau];
            const float cc = bonus ? 0.f : sh.cval[tau];
            const int64_t s0 = min(p.nchunk, (int64_t)sh.sample_seg * p.seg_chunks);
            const int64_t s1 = min(p.nchunk, s0 + p.seg_chunks);
            if (bonus)
                draw_in_segment<DQ, DP, E, true>(p, sh, rq, rp, s0, s1, Kq, Kp, ah, al, cc, warp, lane, ob + tau);
            else
                draw_in_segment<DQ, DP, E, false>(p, sh, rq, rp, s0, s1, Kq, Kp, ah, al, cc, warp, lane, ob + tau);
        }
    }

    // ---- outputs
    const int st = sh.status;
    const int tau = sh.tau;
    for (int j = tid; j <= p.kmax; j += kThreads) {
        if (st != SPEC_ST_OK) p.out_tok[ob + j] = -1;
        else if (j < tau) p.out_tok[ob + j] = sh.x[j];
        else if (j > tau) p.out_tok[ob + j] = -1;
        else if (greedy) p.out_tok[ob + j] = sh.rowArg[N + tau];
    }
    if (tid == 0) {
        p.status[b] = st;
        p.acc_len[b] = (st == SPEC_ST_OK) ? tau : 0;
        p.n_emit[b] = (st == SPEC_ST_OK) ? tau + 1 : 0;
    }
    if (p.diag != nullptr) {
        const float qnan = __int_as_float(0x7fffffff);
        const float ln2 = 0.6931471805599453f;
        const bool have = (!greedy) && (st == SPEC_ST_OK || st == SPEC_ST_NUMERIC);
        const int64_t tbase = prow_of(p, b, base, 0);
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
                if (block) {
                    v[SPEC_DIAG_W] = df_to_f(sh.w[i]);
                    if (i >= 1) v[SPEC_DIAG_H] = df_to_f(i == N ? sh.w[N] : sh.h[i]);
                }
                v[SPEC_DIAG_R] = df_to_f(sh.r[i]);
            }
#pragma unroll
            for (int c = 0; c < SPEC_DIAG_COLS; ++c) d[c] = v[c];
        }
    }
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
static size_t sweep_smem_bytes() {
    return (size_t)kWarps * SweepRing<DQ, DP, E>::RING;
}

static int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    return dev;
}

// Per kernel instantiation and device, set once: the dynamic shared memory limits and the two
// persistent grid sizes (every SM filled to its occupancy).
template <typename DQ, typename DP, int E>
struct LaunchCache {
    static std::atomic<int> stats_grid[64];
    static std::atomic<int> sweep_grid[64];
};
template <typename DQ, typename DP, int E>
std::atomic<int> LaunchCache<DQ, DP, E>::stats_grid[64];
template <typename DQ, typename DP, int E>
std::atomic<int> LaunchCache<DQ, DP, E>::sweep_grid[64];

template <typename DQ, typename DP, int E>
static cudaError_t prepare(int* stats_grid, int* sweep_grid) {
    using C = LaunchCache<DQ, DP, E>;
    const int dev = current_device();
    int g1 = C::stats_grid[dev].load(std::memory_order_acquire);
    int g3 = C::sweep_grid[dev].load(std::memory_order_acquire);
    if (g1 == 0 || g3 == 0) {
        cudaError_t e = cudaFuncSetAttribute(stats_kernel<DQ, DP, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)stats_smem_bytes(E));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sweep_kernel<DQ, DP, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sweep_smem_bytes<DQ, DP, E>());
        if (e != cudaSuccess) return e;
        int sms = 0, occ1 = 0, occ3 = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, stats_kernel<DQ, DP, E>, kStatsThreads,
                                                          stats_smem_bytes(E)) != cudaSuccess || occ1 < 1)
            occ1 = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ3, sweep_kernel<DQ, DP, E>, kThreads,
                                                          sweep_smem_bytes<DQ, DP, E>()) != cudaSuccess || occ3 < 1)
            occ3 = 1;
        cudaGetLastError();
        g1 = sms * occ1;
        g3 = sms * occ3;
        C::stats_grid[dev].store(g1, std::memory_order_release);
        C::sweep_grid[dev].store(g3, std::memory_order_release);
    }
    *stats_grid = g1;
    *sweep_grid = g3;
    return cudaSuccess;
}

// A launch that may begin while the previous kernel on the stream is still running (its
// griddepcontrol.wait orders the data).
template <typename Kernel>
static cudaError_t launch_dependent(Kernel kernel, int grid, size_t smem, cudaStream_t s, const VerifyParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename DQ, typename DP, int E>
static cudaError_t run_verify(VerifyParams& p, cudaStream_t s, int* info) {
    int g1 = 0, g3 = 0;
    cudaError_t e = prepare<DQ, DP, E>(&g1, &g3);
    if (e != cudaSuccess) return e;
    if (info) {
        info[0] = 1;
        info[1] = g3;
        return cudaSuccess;
    }
    p.stats_warps = (int64_t)g1 * kStatsWarps;
    stats_kernel<DQ, DP, E><<<g1, kStatsThreads, stats_smem_bytes(E), s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_dependent(decide_kernel<DQ, DP>, p.B, 0, s, p);
    if (e == cudaSuccess) e = launch_dependent(sweep_kernel<DQ, DP, E>, g3, sweep_smem_bytes<DQ, DP, E>(), s, p);
    if (e == cudaSuccess) e = launch_dependent(finish_kernel<DQ, DP, E>, p.B, 0, s, p);
    if (e != cudaSuccess)   // a kernel ran whose tickets and counters the next call must not see
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

// Argument checks shared by every verify entry point (no pointer is dereferenced).
static int check_args(const spec_verify_args* a, const char* name, bool need_pointers) {
    if (a == nullptr) return set_error(SPEC_ERR_ARG, "%s: args is NULL", name);
    if (a->B < 0) return set_error(SPEC_ERR_SHAPE, "%s: B = %d < 0", name, a->B);
    if (a->V < 1 || a->V > SPEC_MAX_V)
        return set_error(SPEC_ERR_SHAPE, "%s: V = %d outside [1, %d]", name, a->V, SPEC_MAX_V);
    if (a->kmax < 0 || a->kmax > SPEC_MAX_KMAX)
        return set_error(SPEC_ERR_SHAPE, "%s: kmax = %d outside [0, %d]", name, a->kmax, SPEC_MAX_KMAX);
    if (!valid_dtype(a->draft_dtype) || !valid_dtype(a->target_dtype))
        return set_error(SPEC_ERR_DTYPE, "%s: dtype must be SPEC_DTYPE_F32 or SPEC_DTYPE_BF16", name);
    if (need_pointers && a->B > 0) {
        if (!a->cu_drafts || !a->target_logits || !a->temperature || !a->accepted_len || !a->out_tokens ||
            !a->n_emitted || !a->status)
            return set_error(SPEC_ERR_ARG, "%s: a required pointer is NULL", name);
        if ((a->kmax > 0) && (!a->draft_logits || !a->draft_tokens))
            return set_error(SPEC_ERR_ARG, "%s: draft_logits / draft_tokens is NULL", name);
    }
    return SPEC_OK;
}

static int verify_entry(const spec_verify_args* a, void* stream, int rule, const char* name, int* info,
                        const int32_t* t2d = nullptr, int32_t Kq = 0) {
    int rc = check_args(a, name, info == nullptr);
    if (rc != SPEC_OK) return rc;
    const bool reduced = t2d != nullptr;
    if (reduced && (Kq < 1 || Kq > a->V))
        return set_error(SPEC_ERR_SHAPE, "%s: draft vocabulary K = %d outside [1, V = %d]", name, Kq, a->V);
    if (info == nullptr && a->B == 0) return clear_error();
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
    p.dense = 0;
    p.step_dev = nullptr;
    p.t2d = t2d;
    p.Kq = reduced ? Kq : a->V;
    const bool aligned = (a->V % 8 == 0) && ((uintptr_t)a->target_logits % 16 == 0) &&
                         ((uintptr_t)a->draft_logits % 16 == 0) &&
                         (!reduced || (Kq % 8 == 0 && (uintptr_t)t2d % 16 == 0));
    p.nchunk = aligned ? a->V / 8 : a->V;
    p.nchunk_q = aligned ? p.Kq / 8 : p.Kq;
    p.seg_chunks = (p.nchunk + kSegs - 1) / kSegs;
    p.nseg = (int32_t)((p.nchunk + p.seg_chunks - 1) / p.seg_chunks);
    p.ws = reinterpret_cast<char*>(a->workspace);
    p.list = p.ws + ((a->workspace_bytes - work_list_claims(a->B, a->kmax) * sizeof(SweepItem)) & ~(size_t)15);
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

// The verify over the dense layout (draft row b kmax + i, target row b (kmax + 1) + i, N_b =
// cu[b + 1] - cu[b] of them used), the Philox step read from device memory: the adaptive
// pipeline's verify, whose counts come from the controller on the device.  `prepare_only`
// sets the kernels' attributes and grid sizes and launches nothing (before a graph capture).
int verify_dense_launch(int rule, const spec_verify_args* a, const uint64_t* step_dev, void* stream,
                        bool prepare_only) {
    const char* name = "spec_pipeline (verify)";
    int rc = check_args(a, name, !prepare_only);
    if (rc != SPEC_OK) return rc;
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
    p.step = 0;
    p.acc_len = a->accepted_len;
    p.out_tok = a->out_tokens;
    p.n_emit = a->n_emitted;
    p.status = a->status;
    p.diag = a->diag;
    p.dense = 1;
    p.step_dev = step_dev;
    p.t2d = nullptr;
    p.Kq = a->V;
    const bool aligned = (a->V % 8 == 0) && ((uintptr_t)a->target_logits % 16 == 0) &&
                         ((uintptr_t)a->draft_logits % 16 == 0);
    p.nchunk = aligned ? a->V / 8 : a->V;
    p.nchunk_q = p.nchunk;
    p.seg_chunks = (p.nchunk + kSegs - 1) / kSegs;
    p.nseg = (int32_t)((p.nchunk + p.seg_chunks - 1) / p.seg_chunks);
    p.ws = reinterpret_cast<char*>(a->workspace);
    if (!prepare_only) {
        const size_t need = workspace_bytes(a->B, a->kmax);
        if (a->workspace == nullptr || a->workspace_bytes < need || (uintptr_t)a->workspace % 16 != 0)
            return set_error(SPEC_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", name,
                             need, a->workspace_bytes);
        p.list = p.ws + ((a->workspace_bytes - work_list_claims(a->B, a->kmax) * sizeof(SweepItem)) & ~(size_t)15);
    }
    int info[3];
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = aligned ? dispatch_dtypes<8>(p, a->draft_dtype, a->target_dtype, s, prepare_only ? info : nullptr)
                                  : dispatch_dtypes<1>(p, a->draft_dtype, a->target_dtype, s, prepare_only ? info : nullptr);
    if (e != cudaSuccess) return set_cuda_error(e, name);
    return SPEC_OK;
}

}  // namespace sv

extern "C" int spec_verify_tokenwise(const spec_verify_args* args, void* stream) {
    return sv::verify_entry(args, stream, 0, "spec_verify_tokenwise", nullptr);
}

extern "C" int spec_verify_block(const spec_verify_args* args, void* stream) {
    return sv::verify_entry(args, stream, 1, "spec_verify_block", nullptr);
}

extern "C" int spec_verify_tokenwise_reduced(const spec_verify_args* args, const int32_t* t2d, int32_t K,
                                             void* stream) {
    if (t2d == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_verify_tokenwise_reduced: t2d is NULL");
    return sv::verify_entry(args, stream, 0, "spec_verify_tokenwise_reduced", nullptr, t2d, K);
}

extern "C" int spec_verify_block_reduced(const spec_verify_args* args, const int32_t* t2d, int32_t K,
                                         void* stream) {
    if (t2d == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_verify_block_reduced: t2d is NULL");
    return sv::verify_entry(args, stream, 1, "spec_verify_block_reduced", nullptr, t2d, K);
}

// ---------------------------------------------------------------------------------------
// Block verification with a fixed, device-resident workspace.  Some callers cannot allocate
// device memory at the point where they verify (an allocator that is not theirs to touch, a
// memory budget fixed at start-up); for them the workspace lives in one array reserved when
// the library's module is loaded, so this call allocates nothing.  The array holds
// kStaticWorkspaceBytes; a batch whose workspace_bytes(B, kmax) is larger is refused.  Like
// every device variable it starts zero-filled, which is the state each call leaves it in.
// All calls share the one array, so calls that may overlap in time (different streams,
// threads) race on it and must be ordered by the caller.
// ---------------------------------------------------------------------------------------
namespace sv {
constexpr size_t kStaticWorkspaceBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of g_static_workspace on the current device, looked up once per device and
// kept for the life of the process (a context reset is not noticed: see the header).
static cudaError_t static_workspace(void** ptr) {
    static std::atomic<void*> addr[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void* a = addr[dev].load(std::memory_order_acquire);
    if (a == nullptr) {
        e = cudaGetSymbolAddress(&a, g_static_workspace);
        if (e != cudaSuccess) return e;
        addr[dev].store(a, std::memory_order_release);   // racing first calls store the same value
    }
    *ptr = a;
    return cudaSuccess;
}
}  // namespace sv

extern "C" int spec_verify_block_static(const spec_verify_args* args, void* stream) {
    const char* name = "spec_verify_block_static";
    // the common checks first, so that a bad shape or dtype gets the same code as in
    // spec_verify_block; only the workspace check is this call's own
    int rc = sv::check_args(args, name, true);
    if (rc != SPEC_OK) return rc;
    spec_verify_args a = *args;
    if (a.B > 0) {
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
