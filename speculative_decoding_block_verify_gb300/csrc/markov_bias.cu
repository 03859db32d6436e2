// The Markov head's previous-token logit bias on sm_103a.
//
// Method: "MTP Heads and Confidence Heads: Linking Three Self-Drafting Routes into One Chain"
// (naphjohn.github.io), §6 "Why the Markov Head Helps": a low-rank logit bias B = W1 @ W2
// (default rank 256) added to the draft logits by the previous token; "MTP, DSpark and Block
// Verification, Explained" (al-engr.com), §3 "The Markov fix-up" and Figure 2.
//
//   out[r, v] = draft[r, v] + sum_j W1[prev_r, j] * W2[j, v]
//
// At the draft-side shapes (a handful of rows per W2 pass) this is a skinny GEMM whose bound is
// W2's bytes (66 MB at rank 256, V = 129,280): every W2 element is read once per row group and
// feeds every row of the group.  Three kernels, by operand layout:
//   * bf16 W1 and W2, 16-byte rows: markov_bias_mma_kernel - W2 by 2-D TMA boxes, the products
//     on the tensor cores (warp-level mma.sync); on CUDA cores five rows cost ~2.5 FFMA2 per W2
//     element, which with their issue slots made the scan instruction-bound even from L2;
//   * float32 W2, 16-byte rows: markov_bias_tma_kernel - W2 by 2-D TMA boxes, FFMA2;
//   * other shapes: markov_bias_kernel - a CTA owns a 32 x E column tile, its 4 warps split the
//     rank dimension with register-held loads, and the partial sums meet in shared memory.

#include <atomic>
#include <cfloat>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host_util.h"

namespace sv {

constexpr int kBiasThreads = 128;
constexpr int kBiasWarps = kBiasThreads / 32;
constexpr int kRowGroup = 8;
constexpr int kMaxRank = 1024;

struct BiasParams {
    const void* draft;
    const int32_t* prev;
    const void* W1;
    const void* W2;
    float* out;
    int32_t rows, V, R;
    int64_t nchunk;  // chunks per W2 row
};

template <typename DT, typename WT, int E>
__global__ void __launch_bounds__(kBiasThreads, 4) markov_bias_kernel(const BiasParams p) {
    extern __shared__ float smem[];
    constexpr int kTile = 32 * E;
    // W2 rows per load group; two groups per lane alternate (one in flight while the other is
    // multiplied), 64 bytes of registers per group
    constexpr int UJ = (E == 1) ? 8 : (sizeof(WT) == 2 ? 4 : 2);
    float* w1s = smem;                          // [kRowGroup][R]
    float* red = smem + kRowGroup * p.R;        // [kBiasWarps][kRowGroup][kTile]
    __shared__ int row_ok[kRowGroup];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = p.V;
    const int64_t col0 = (int64_t)blockIdx.x * kTile;
    const int r0 = blockIdx.y * kRowGroup;
    const int nr = min(kRowGroup, p.rows - r0);

    // gather the group's W1 rows (float32) - an invalid prev zeroes its row and marks it.  The
    // prev tokens first, then the gather unrolled so that its loads are in flight together.
    __shared__ int s_prev[kRowGroup];
    if (tid < kRowGroup) {
        int pv = -1;
        if (tid < nr) pv = p.prev[r0 + tid];
        const int ok = (pv >= 0 && pv < p.V);
        s_prev[tid] = ok ? pv : -1;
        row_ok[tid] = ok;
    }
    __syncthreads();
#pragma unroll 8
    for (int t = tid; t < kRowGroup * p.R; t += kBiasThreads) {
        const int r = t / p.R, j = t - r * p.R;
        const int pv = s_prev[r];
        w1s[t] = (pv >= 0) ? load_elem<WT>(p.W1, (int64_t)pv * p.R + j) : 0.f;
    }
    __syncthreads();

    const int jper = (p.R + kBiasWarps - 1) / kBiasWarps;
    const int j0 = min(p.R, warp * jper), j1 = min(p.R, j0 + jper);
    const int64_t chunk = col0 / E + lane;
    const bool active = chunk < p.nchunk;
    float acc[kRowGroup][E];
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[r][e] = 0.f;

    Chunk<WT, E> ca[UJ], cb[UJ];
    auto load = [&](Chunk<WT, E>(&c)[UJ], int j) {
#pragma unroll
        for (int u = 0; u < UJ; ++u)
            if (active && j + u < j1) c[u].load(row_ptr<WT>(p.W2, j + u, V), chunk);
    };
    auto fma_group = [&](const Chunk<WT, E>(&c)[UJ], int j) {
#pragma unroll
        for (int u = 0; u < UJ; ++u) {
            if (active && j + u < j1) {
                float x[E];
                c[u].unpack(x);
#pragma unroll
                for (int r = 0; r < kRowGroup; ++r) {
                    if (r < nr) {
                        const float wv = w1s[r * p.R + j + u];
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[r][e] = fmaf(wv, x[e], acc[r][e]);
                    }
                }
            }
        }
    };
    if (j0 < j1) load(ca, j0);
    for (int j = j0; j < j1; j += 2 * UJ) {
        if (j + UJ < j1) load(cb, j + UJ);
        fma_group(ca, j);
        if (j + UJ >= j1) break;
        if (j + 2 * UJ < j1) load(ca, j + 2 * UJ);
        fma_group(cb, j + UJ);
    }
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int e = 0; e < E; ++e) red[(warp * kRowGroup + r) * kTile + lane * E + e] = acc[r][e];
    __syncthreads();

    // epilogue: this thread's outputs o = tid + k * threads; the draft logits are loaded first,
    // all together, then the warps' partial sums are added
    const float qnan = __int_as_float(0x7fffffff);
    constexpr int KO = kRowGroup * kTile / kBiasThreads;
    float d[KO];
#pragma unroll
    for (int k = 0; k < KO; ++k) {
        const int o = tid + k * kBiasThreads;
        const int r = o / kTile, ci = o % kTile;
        const int64_t v = col0 + ci;
        d[k] = (r < nr && v < V) ? load_elem<DT>(p.draft, (int64_t)(r0 + r) * V + v) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < KO; ++k) {
        const int o = tid + k * kBiasThreads;
        const int r = o / kTile, ci = o % kTile;
        const int64_t v = col0 + ci;
        if (r < nr && v < V) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kBiasWarps; ++w) sum += red[(w * kRowGroup + r) * kTile + ci];
            p.out[(int64_t)(r0 + r) * V + v] = row_ok[r] ? d[k] + sum : qnan;
        }
    }
}

// ---------------------------------------------------------------------------------------
// 16-byte rows: W2 streamed by the tensor memory accelerator.  A CTA owns a 256-column tile (a
// lane, 8 columns) of a group of NR rows; its 4 warps split the rank into slices of whole
// boxes, each streaming its slice through a 2-stage ring in which one cp.async.bulk.tensor.2d
// brings a [8 W2 rows x 256 columns] box (rows past the rank and columns past V arrive as
// zeros).  The group's gathered W1 rows sit in shared memory as duplicated pairs (w, w) per
// (rank index, row), so that each W2 element feeds the NR rows through packed FFMA2 (two
// columns per instruction).  After the scan the ring and the W1 area hold the warps' partial
// sums, which the epilogue adds to the draft logits.  At ~48 KB of shared memory four CTAs
// share an SM, so the 505 tiles of a 129,280-token vocabulary run as one wave.
// ---------------------------------------------------------------------------------------
constexpr int kTmaMinBlocks = 4;             // resident CTAs per SM the registers allow
constexpr int kTmaCols = 256;                // columns per tile
constexpr int kLaneCols = kTmaCols / 32;     // columns per lane
constexpr int kTmaJS = 8;                    // W2 rows per box (one stage)
constexpr int kTmaStages = 2;
constexpr int kTmaMaxRows = 8;
constexpr int kBiasSpinLimit = 1 << 20;   // mbarrier polls before a wait gives up (the tile is written as NaN)

template <typename WT, int NR>
struct TmaLayout {
    static constexpr int kStageBytes = kTmaJS * kTmaCols * (int)sizeof(WT);
    static constexpr int kRingBytes = kBiasWarps * kTmaStages * kStageBytes;
    static constexpr int kRedBytes = kBiasWarps * NR * kTmaCols * (int)sizeof(float);
    static size_t smem(int R) {
        const size_t scan = (size_t)kRingBytes + (size_t)R * NR * sizeof(float2);
        return scan > (size_t)kRedBytes ? scan : (size_t)kRedBytes;
    }
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

template <typename DT, typename WT, int NR>
__global__ void __launch_bounds__(kBiasThreads, kTmaMinBlocks) markov_bias_tma_kernel(const BiasParams p,
                                                                         const __grid_constant__ CUtensorMap w2map) {
    using Lay = TmaLayout<WT, NR>;
    extern __shared__ __align__(128) char bsm[];
    __shared__ __align__(8) uint64_t bars[kBiasWarps][kTmaStages];
    __shared__ int s_prev[NR], s_ok[NR];
    float2* w1d = reinterpret_cast<float2*>(bsm + Lay::kRingBytes);   // [R][NR], (w, w)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = p.V;
    const int64_t col0 = (int64_t)blockIdx.x * kTmaCols;
    const int ncol = (int)min((int64_t)kTmaCols, V - col0);
    const int r0 = blockIdx.y * NR;
    const int nr = min(NR, p.rows - r0);
    // rank slices of whole boxes: warp w takes rows [j0, j1)
    const int jper = ((p.R + kBiasWarps - 1) / kBiasWarps + kTmaJS - 1) / kTmaJS * kTmaJS;
    const int j0 = min(p.R, warp * jper), j1 = min(p.R, j0 + jper);
    const int nst = (j1 - j0 + kTmaJS - 1) / kTmaJS;
    char* ring = bsm + warp * kTmaStages * Lay::kStageBytes;
    uint64_t* wb = bars[warp];
    if (lane == 0) {
        for (int s = 0; s < kTmaStages; ++s) mbar_init(&wb[s], 1);
        mbar_init_fence();
    }
    __syncwarp();
    int issued = 0;
    auto issue = [&](int q) {   // stage q: the box at W2 rows j0 + q kTmaJS, columns col0
        if (q >= nst) return;
        const int slot = q % kTmaStages;
        __syncwarp();   // every lane is done with the slot's previous stage (stage q - kTmaStages)
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&wb[slot], (unsigned)Lay::kStageBytes);
            tma_load_2d(ring + slot * Lay::kStageBytes, &w2map, (int)col0, j0 + q * kTmaJS, &wb[slot]);
        }
        issued = q + 1;
    };
    // the whole ring is in flight while the group's W1 rows are gathered
    for (int q = 0; q < kTmaStages; ++q) issue(q);
    if (tid < NR) {
        int pv = -1;
        if (tid < nr) pv = p.prev[r0 + tid];
        const int ok = (pv >= 0 && pv < p.V);
        s_prev[tid] = ok ? pv : -1;
        s_ok[tid] = ok;
    }
    __syncthreads();
    for (int t = tid; t < NR * p.R; t += kBiasThreads) {   // row-major reads of W1 (coalesced)
        const int r = t / p.R, j = t - r * p.R;
        const int pv = s_prev[r];
        const float w = (pv >= 0) ? load_elem<WT>(p.W1, (int64_t)pv * p.R + j) : 0.f;
        w1d[j * NR + r] = make_float2(w, w);
    }
    __syncthreads();

    // this thread's draft logits for the epilogue (outputs o = tid + k threads), in flight
    // during the scan
    constexpr int KO = NR * kTmaCols / kBiasThreads;
    float d[KO];
#pragma unroll
    for (int k = 0; k < KO; ++k) {
        const int o = tid + k * kBiasThreads;
        const int r = o / kTmaCols, ci = o % kTmaCols;
        d[k] = (r < nr && ci < ncol) ? load_elem<DT>(p.draft, (int64_t)(r0 + r) * V + col0 + ci) : 0.f;
    }
    constexpr int LP = kLaneCols / 2;   // column pairs per lane
    float2 acc[NR][LP];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int c = 0; c < LP; ++c) acc[r][c] = make_float2(0.f, 0.f);
    const bool has_cols = lane * kLaneCols < ncol;
    bool timeout = false;
    int waited = 0;
    for (int q = 0; q < nst; ++q) {
        if (q > 0) issue(q + kTmaStages - 1);   // into the slot of stage q - 1, consumed
        const int slot = q % kTmaStages;
        const unsigned parity = (unsigned)(q / kTmaStages) & 1u;
        bool ok = true;
        for (int n = 0; !mbar_try_wait(&wb[slot], parity);)
            if (++n > kBiasSpinLimit) {
                ok = false;
                break;
            }
        timeout = !__all_sync(0xffffffffu, ok);   // one decision for the whole warp
        if (timeout) break;
        waited = q + 1;
        const int ja = j0 + q * kTmaJS;
        const int jn = min(kTmaJS, j1 - ja);
        const char* st = ring + slot * Lay::kStageBytes + lane * kLaneCols * (int)sizeof(WT);
        if (has_cols) {
#pragma unroll
            for (int jj = 0; jj < kTmaJS; ++jj) {
                if (jj < jn) {
                    float2 x[LP];
                    const char* c = st + jj * kTmaCols * (int)sizeof(WT);
                    if constexpr (sizeof(WT) == 2 && LP == 4) {
                        const uint4 v = *reinterpret_cast<const uint4*>(c);
                        x[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
                        x[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
                        x[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
                        x[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
                    } else if constexpr (sizeof(WT) == 2) {
                        const uint2 v = *reinterpret_cast<const uint2*>(c);
                        x[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
                        x[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
                    } else {
#pragma unroll
                        for (int h = 0; h < LP / 2; ++h) {
                            const float4 a = *reinterpret_cast<const float4*>(c + 16 * h);
                            x[2 * h] = make_float2(a.x, a.y);
                            x[2 * h + 1] = make_float2(a.z, a.w);
                        }
                    }
                    const float4* wv = reinterpret_cast<const float4*>(w1d + (ja + jj) * NR);
#pragma unroll
                    for (int rp = 0; rp < NR / 2; ++rp) {
                        const float4 w = wv[rp];   // (w_2rp, w_2rp, w_2rp+1, w_2rp+1)
                        const float2 wa = make_float2(w.x, w.y), wc = make_float2(w.z, w.w);
#pragma unroll
                        for (int cc = 0; cc < LP; ++cc) {
                            acc[2 * rp][cc] = ffma2(wa, x[cc], acc[2 * rp][cc]);
                            acc[2 * rp + 1][cc] = ffma2(wc, x[cc], acc[2 * rp + 1][cc]);
                        }
                    }
                }
            }
        }
    }
    // a failed wait: the copies still in flight land before the CTA reuses or leaves the ring
    for (int q = waited; q < issued; ++q) {
        const unsigned parity = (unsigned)(q / kTmaStages) & 1u;
        for (int n = 0; n < kBiasSpinLimit && !mbar_try_wait(&wb[q % kTmaStages], parity); ++n) {
        }
    }
    const bool any_timeout = __syncthreads_or(timeout);   // every warp is done with the ring and W1
    float* red = reinterpret_cast<float*>(bsm);            // [kBiasWarps][NR][kTmaCols]
    if (has_cols) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float4* dst = reinterpret_cast<float4*>(red + (warp * NR + r) * kTmaCols + lane * kLaneCols);
#pragma unroll
            for (int h = 0; h < LP / 2; ++h)
                dst[h] = make_float4(acc[r][2 * h].x, acc[r][2 * h].y, acc[r][2 * h + 1].x, acc[r][2 * h + 1].y);
        }
    }
    __syncthreads();
    // epilogue: the warps' partial sums added to the draft logits
    const float qnan = __int_as_float(0x7fffffff);
#pragma unroll
    for (int k = 0; k < KO; ++k) {
        const int o = tid + k * kBiasThreads;
        const int r = o / kTmaCols, ci = o % kTmaCols;
        if (r < nr && ci < ncol) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kBiasWarps; ++w) sum += red[(w * NR + r) * kTmaCols + ci];
            p.out[(int64_t)(r0 + r) * V + col0 + ci] = (s_ok[r] && !any_timeout) ? d[k] + sum : qnan;
        }
    }
}

// ---------------------------------------------------------------------------------------
// bf16 W1 and W2 with 16-byte rows: the products on the tensor cores.  The rank is the
// contraction dimension of a skinny GEMM out[r, v] = sum_j W1[prev_r, j] W2[j, v], M = 16
// vocabulary columns, N = 8 rows, K = 16 rank indices per warp-level mma.sync (bf16 inputs,
// float32 accumulation); the bound stays W2's bytes, and the tensor cores take the ~2.5 FFMA2
// per W2 element (and their issue slots) off the SMs.  A warp streams whole 64-column strips of
// W2 (all ranks), strip after strip, through a 3-stage ring of 8 KB stages, each [rank rows x
// strip columns] brought by cp.async.bulk.tensor.2d as 64-column boxes with the 128-byte
// swizzle (so that the ldmatrix.trans reads of the A fragments are free of bank conflicts, and
// each rank row's columns are read from HBM in one contiguous run); the group's W1 rows sit
// in shared memory with rows 16 bytes apart from a bank boundary.  No partial sums cross warps:
// each strip's outputs go out from the warp's accumulators, the draft logits added.
// ---------------------------------------------------------------------------------------
constexpr int kMmaCols = 128;                 // columns per strip
constexpr int kMmaSub = kMmaCols / 64;        // 64-column sub-boxes (128-byte swizzled rows) per stage
constexpr int kMmaBoxBytes = 8192;            // one stage
constexpr int kMmaKB = kMmaBoxBytes / (kMmaCols * 2);   // rank rows per stage (a multiple of 16)
constexpr int kMmaGroups = kMmaCols / 16;     // 16-column mma groups per strip
constexpr int kMmaStages = 3;
constexpr int kMmaRows = 8;                   // rows per group: the mma's N

static size_t mma_smem_bytes(int R) {   // ranks padded to a whole stage
    const int Rp = (R + kMmaKB - 1) / kMmaKB * kMmaKB;
    return 1024 + (size_t)kBiasWarps * kMmaStages * kMmaBoxBytes + (size_t)kMmaRows * (Rp + 8) * 2;
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
// d += a b: a the 16 x 16 (M x K) fragment, b the 16 x 8 (K x N) fragment, d 16 x 8 float32
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <typename DT>
__global__ void __launch_bounds__(kBiasThreads, 2) markov_bias_mma_kernel(const BiasParams p,
                                                                         const __grid_constant__ CUtensorMap w2map,
                                                                         int nstrips) {
    constexpr int SC = kMmaCols;   // strip columns
    constexpr int KB = kMmaKB;     // ranks per stage
    constexpr int NG = SC / 16;    // 16-column mma groups
    extern __shared__ __align__(1024) char msm[];
    __shared__ __align__(8) uint64_t bars[kBiasWarps][kMmaStages];
    __shared__ int s_prev[kMmaRows], s_ok[kMmaRows];
    // the swizzle pattern repeats every 1024 bytes: the ring starts on such a boundary
    char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(msm) + 1023) & ~static_cast<uintptr_t>(1023));
    const int Rp = (p.R + KB - 1) / KB * KB;
    const int ldw = Rp + 8;   // W1 row stride in elements: rows 16 bytes off a bank boundary
    uint16_t* w1s = reinterpret_cast<uint16_t*>(base + kBiasWarps * kMmaStages * kMmaBoxBytes);   // [8][ldw]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = p.V;
    const int r0 = blockIdx.y * kMmaRows;
    const int nr = min(kMmaRows, p.rows - r0);
    const int nkb = Rp / KB;
    // strip s goes to warp s / gridDim.x of CTA s % gridDim.x (then every W-th): with the grid at
    // the resident CTA count, the CTAs sharing an SM get strip counts that differ by at most one
    const int W = gridDim.x * kBiasWarps;
    const int s_first = blockIdx.x + warp * gridDim.x;
    const int nmine = s_first < nstrips ? (nstrips - s_first + W - 1) / W : 0;
    const int total = nmine * nkb;   // boxes this warp streams: its strips in order, each over all ranks
    char* ring = base + warp * kMmaStages * kMmaBoxBytes;
    uint64_t* wb = bars[warp];
    if (lane == 0) {
        for (int s = 0; s < kMmaStages; ++s) mbar_init(&wb[s], 1);
        mbar_init_fence();
    }
    __syncwarp();
    int issued = 0;
    auto issue = [&](int q) {   // stage q: strip s_first + (q / nkb) W, ranks (q % nkb) KB ..
        if (q >= total) return;
        const int slot = q % kMmaStages;
        const int strip = s_first + (q / nkb) * W, kb = q % nkb;
        __syncwarp();   // every lane is done with the slot's previous stage
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&wb[slot], (unsigned)kMmaBoxBytes);
#pragma unroll
            for (int sb = 0; sb < kMmaSub; ++sb)   // each rank row arrives as kMmaCols contiguous columns
                tma_load_2d(ring + slot * kMmaBoxBytes + sb * (kMmaKB * 128), &w2map, strip * kMmaCols + sb * 64,
                            kb * kMmaKB, &wb[slot]);
        }
        issued = q + 1;
    };
    // the whole ring is in flight while the group's W1 rows are gathered
    for (int q = 0; q < kMmaStages; ++q) issue(q);
    if (tid < kMmaRows) {
        int pv = -1;
        if (tid < nr) pv = p.prev[r0 + tid];
        const int ok = (pv >= 0 && pv < p.V);
        s_prev[tid] = ok ? pv : -1;
        s_ok[tid] = ok;
    }
    __syncthreads();
    const uint16_t* w1g = static_cast<const uint16_t*>(p.W1);
    for (int t = tid; t < kMmaRows * Rp; t += kBiasThreads) {   // row-major reads of W1 (coalesced)
        const int r = t / Rp, j = t - r * Rp;
        const int pv = s_prev[r];
        w1s[r * ldw + j] = (pv >= 0 && j < p.R) ? __ldg(w1g + (int64_t)pv * p.R + j) : (uint16_t)0;
    }
    __syncthreads();
    // ldmatrix row addresses of this lane: B (x2) rows n = lane & 7, k half (lane >> 3) & 1;
    // A (x4.trans) box row a_j of the k16 step, 8-column block a_cb of the 16-column group
    const uint32_t w1_addr = smem_u32(w1s) + (uint32_t)(((lane & 7) * ldw + ((lane >> 3) & 1) * 8) * 2);
    // the x4.trans matrices are (ranks 0-7 | 8-15) x (columns 0-7 | 8-15) of the 16-column group
    const int a_j = (lane & 7) + ((lane >> 4) << 3);
    const int a_cb = (lane >> 3) & 1;
    const int g = lane >> 2, t4 = lane & 3;   // accumulator fragment: columns g, g + 8; rows 2 t4, 2 t4 + 1
    const float qnan = __int_as_float(0x7fffffff);
    bool timeout = false;
    int q = 0, si = 0;
    for (; si < nmine && !timeout; ++si) {
        const int strip = s_first + si * W;
        float acc[NG][4];
#pragma unroll
        for (int gg = 0; gg < NG; ++gg)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[gg][e] = 0.f;
        for (int kb = 0; kb < nkb; ++kb, ++q) {
            if (q > 0) issue(q + kMmaStages - 1);   // into the slot of box q - 1, consumed
            const int slot = q % kMmaStages;
            const unsigned parity = (unsigned)(q / kMmaStages) & 1u;
            bool ok = true;
            for (int n = 0; !mbar_try_wait(&wb[slot], parity);)
                if (++n > kBiasSpinLimit) {
                    ok = false;
                    break;
                }
            timeout = !__all_sync(0xffffffffu, ok);   // one decision for the whole warp (mma.sync below)
            if (timeout) break;
            const uint32_t box = smem_u32(ring + slot * kMmaBoxBytes);
#pragma unroll
            for (int ks = 0; ks < KB / 16; ++ks) {
                uint32_t b[2];
                ldsm_x2(b, w1_addr + (uint32_t)((kb * KB + ks * 16) * 2));
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) {
                    uint32_t a[4];
                    const int j = ks * 16 + a_j;          // box row = rank (128 bytes of columns)
                    const int c16 = (gg & 3) * 2 + a_cb;  // 16-byte chunk = 8 columns, swizzled by the row
                    ldsm_x4_trans(a, box + (uint32_t)((gg >> 2) * (kMmaKB * 128) + j * 128 + ((c16 ^ (j & 7)) << 4)));
                    mma_16816_bf16(acc[gg], a, b);
                }
            }
        }
        if (timeout) break;
        // this strip's outputs: acc[gg][e] is row 2 t4 + (e & 1), column strip 64 + 16 gg + g + 8 (e >> 1)
        float d[NG][4];
#pragma unroll
        for (int gg = 0; gg < NG; ++gg)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = 2 * t4 + (e & 1);
                const int64_t col = (int64_t)strip * SC + 16 * gg + g + 8 * (e >> 1);
                d[gg][e] = (n < nr && col < V) ? load_elem<DT>(p.draft, (int64_t)(r0 + n) * V + col) : 0.f;
            }
#pragma unroll
        for (int gg = 0; gg < NG; ++gg)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = 2 * t4 + (e & 1);
                const int64_t col = (int64_t)strip * SC + 16 * gg + g + 8 * (e >> 1);
                if (n < nr && col < V) p.out[(int64_t)(r0 + n) * V + col] = s_ok[n] ? d[gg][e] + acc[gg][e] : qnan;
            }
    }
    if (timeout) {   // the strip that could not be summed and every later one read as NaN
        for (int sj = si; sj < nmine; ++sj) {
            const int64_t c0 = (int64_t)(s_first + sj * W) * SC;
            for (int k = lane; k < nr * SC; k += 32) {
                const int n = k / SC;
                const int64_t col = c0 + k % SC;
                if (col < V) p.out[(int64_t)(r0 + n) * V + col] = qnan;
            }
        }
    }
    // the copies still in flight land before the CTA leaves
    for (int qq = q; qq < issued; ++qq) {
        const unsigned parity = (unsigned)(qq / kMmaStages) & 1u;
        for (int n = 0; n < kBiasSpinLimit && !mbar_try_wait(&wb[qq % kMmaStages], parity); ++n) {
        }
    }
}

template <int E>
constexpr size_t bias_smem_bytes(int R) {
    return sizeof(float) * ((size_t)kRowGroup * R + (size_t)kBiasWarps * kRowGroup * 32 * E);
}

// The shared-memory opt-in is set once per device and kernel instance, for the largest rank;
// later launches skip the driver call.
template <typename DT, typename WT, int E>
struct BiasAttr {
    static std::atomic<int> set[64];
};
template <typename DT, typename WT, int E>
std::atomic<int> BiasAttr<DT, WT, E>::set[64];

template <typename DT, typename WT, int E>
static cudaError_t launch_bias(const BiasParams& p, cudaStream_t s) {
    constexpr int kTile = 32 * E;
    const size_t smem = bias_smem_bytes<E>(p.R);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !BiasAttr<DT, WT, E>::set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(markov_bias_kernel<DT, WT, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bias_smem_bytes<E>(kMaxRank));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) BiasAttr<DT, WT, E>::set[dev].store(1, std::memory_order_release);
    }
    const dim3 grid((unsigned)((p.V + kTile - 1) / kTile),
                    (unsigned)((p.rows + kRowGroup - 1) / kRowGroup));
    markov_bias_kernel<DT, WT, E><<<grid, kBiasThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename DT, typename WT, int NR>
struct TmaAttr {
    static std::atomic<int> set[64];
};
template <typename DT, typename WT, int NR>
std::atomic<int> TmaAttr<DT, WT, NR>::set[64];

// cuTensorMapEncodeTiled from the driver, looked up once (the library links the runtime only).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

template <typename DT, typename WT, int NR>
static cudaError_t launch_bias_tma_nr(const BiasParams& p, const CUtensorMap& map, cudaStream_t s) {
    using Lay = TmaLayout<WT, NR>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !TmaAttr<DT, WT, NR>::set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(markov_bias_tma_kernel<DT, WT, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Lay::smem(kMaxRank));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) TmaAttr<DT, WT, NR>::set[dev].store(1, std::memory_order_release);
    }
    const dim3 grid((unsigned)((p.V + kTmaCols - 1) / kTmaCols), (unsigned)((p.rows + NR - 1) / NR));
    markov_bias_tma_kernel<DT, WT, NR><<<grid, kBiasThreads, Lay::smem(p.R), s>>>(p, map);
    return cudaGetLastError();
}

// W2 [R, V] (V a multiple of 8, 16-byte aligned) as a 2-D tensor of boxes [8 rows x 256
// columns]; rows past R and columns past V read as zeros.  Rows go in groups of the smallest of
// 2, 4, 6, 8 that holds them (8 for more than 8 rows).
template <typename DT, typename WT>
static cudaError_t launch_bias_tma(const BiasParams& p, cudaStream_t s, bool* unavailable) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) {
        *unavailable = true;
        return cudaSuccess;
    }
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.V, (cuuint64_t)p.R};
    const cuuint64_t strides[1] = {(cuuint64_t)p.V * sizeof(WT)};
    const cuuint32_t box[2] = {(cuuint32_t)kTmaCols, (cuuint32_t)kTmaJS};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = encode(&map, sizeof(WT) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                              const_cast<void*>(p.W2), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *unavailable = true;
        return cudaSuccess;
    }
    if (p.rows <= 2) return launch_bias_tma_nr<DT, WT, 2>(p, map, s);
    if (p.rows <= 4) return launch_bias_tma_nr<DT, WT, 4>(p, map, s);
    if (p.rows <= 6) return launch_bias_tma_nr<DT, WT, 6>(p, map, s);
    return launch_bias_tma_nr<DT, WT, kTmaMaxRows>(p, map, s);
}

template <typename DT>
struct MmaAttr {
    static std::atomic<int> grid[64];   // resident CTAs of the device (0: not yet set up)
};
template <typename DT>
std::atomic<int> MmaAttr<DT>::grid[64];

// bf16 W1 and W2 on the tensor cores: W2 [R, V] as a 2-D tensor of [rank rows x 64 columns] boxes
// with the 128-byte swizzle (elements past the tensor's edges read as zeros).
template <typename DT>
static cudaError_t launch_bias_mma(const BiasParams& p, cudaStream_t s, bool* unavailable) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) {
        *unavailable = true;
        return cudaSuccess;
    }
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.V, (cuuint64_t)p.R};
    const cuuint64_t strides[1] = {(cuuint64_t)p.V * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)kMmaKB};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.W2), dims, strides, box,
                              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *unavailable = true;
        return cudaSuccess;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int resident = (dev >= 0 && dev < 64) ? MmaAttr<DT>::grid[dev].load(std::memory_order_acquire) : 0;
    if (resident == 0) {
        e = cudaFuncSetAttribute(markov_bias_mma_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mma_smem_bytes(kMaxRank));
        if (e != cudaSuccess) return e;
        int sms = 0, occ = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, markov_bias_mma_kernel<DT>, kBiasThreads,
                                                          mma_smem_bytes(256)) != cudaSuccess || occ < 1)
            occ = 1;
        cudaGetLastError();
        resident = sms * occ;
        if (dev >= 0 && dev < 64) MmaAttr<DT>::grid[dev].store(resident, std::memory_order_release);
    }
    const int nstrips = (int)((p.V + kMmaCols - 1) / kMmaCols);
    const dim3 grid((unsigned)(nstrips < resident ? nstrips : resident), (unsigned)((p.rows + kMmaRows - 1) / kMmaRows));
    markov_bias_mma_kernel<DT><<<grid, kBiasThreads, mma_smem_bytes(p.R), s>>>(p, map, nstrips);
    return cudaGetLastError();
}

template <int E>
static cudaError_t dispatch_bias(const BiasParams& p, int dt, int wt, cudaStream_t s) {
    if constexpr (E == 8) {   // 16-byte rows: W2 through the tensor memory accelerator
        bool unavailable = false;   // no tensor-map encoder in the driver: the plain kernel below
        cudaError_t e;
        if (wt == SPEC_DTYPE_BF16)   // bf16 weights: the products on the tensor cores
            e = dt == SPEC_DTYPE_F32 ? launch_bias_mma<float>(p, s, &unavailable)
                                     : launch_bias_mma<__nv_bfloat16>(p, s, &unavailable);
        else if (dt == SPEC_DTYPE_F32) e = launch_bias_tma<float, float>(p, s, &unavailable);
        else e = launch_bias_tma<__nv_bfloat16, float>(p, s, &unavailable);
        if (!unavailable) return e;
    }
    if (dt == SPEC_DTYPE_F32 && wt == SPEC_DTYPE_BF16) return launch_bias<float, __nv_bfloat16, E>(p, s);
    if (dt == SPEC_DTYPE_BF16 && wt == SPEC_DTYPE_BF16)
        return launch_bias<__nv_bfloat16, __nv_bfloat16, E>(p, s);
    if (dt == SPEC_DTYPE_F32 && wt == SPEC_DTYPE_F32) return launch_bias<float, float, E>(p, s);
    return launch_bias<__nv_bfloat16, float, E>(p, s);
}

}  // namespace sv

extern "C" int dspark_markov_bias(const void* draft_logits, int32_t draft_dtype, int32_t rows,
                                  int32_t V, const int32_t* prev_tokens, const void* W1,
                                  const void* W2, int32_t w_dtype, int32_t rank,
                                  float* out_logits, void* stream) {
    const char* name = "dspark_markov_bias";
    if (!sv::valid_dtype(draft_dtype) || !sv::valid_dtype(w_dtype))
        return sv::set_error(SPEC_ERR_DTYPE, "%s: dtype must be SPEC_DTYPE_F32 or SPEC_DTYPE_BF16",
                             name);
    if (rows < 0 || V < 1 || V > SPEC_MAX_V || rank < 1 || rank > sv::kMaxRank)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: rows=%d V=%d rank=%d out of range", name, rows,
                             V, rank);
    if (rows == 0) return sv::clear_error();
    if (!draft_logits || !prev_tokens || !W1 || !W2 || !out_logits)
        return sv::set_error(SPEC_ERR_ARG, "%s: a pointer is NULL", name);
    if ((const void*)out_logits == draft_logits && draft_dtype != SPEC_DTYPE_F32)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: in-place needs float32 draft logits", name);
    sv::BiasParams p;
    p.draft = draft_logits;
    p.prev = prev_tokens;
    p.W1 = W1;
    p.W2 = W2;
    p.out = out_logits;
    p.rows = rows;
    p.V = V;
    p.R = rank;
    const bool aligned = (V % 8 == 0) && ((uintptr_t)W2 % 16 == 0);
    const int E = aligned ? 8 : 1;
    p.nchunk = V / E;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = aligned ? sv::dispatch_bias<8>(p, draft_dtype, w_dtype, s)
                                  : sv::dispatch_bias<1>(p, draft_dtype, w_dtype, s);
    if (e != cudaSuccess) return sv::set_cuda_error(e, name);
    return sv::clear_error();
}
