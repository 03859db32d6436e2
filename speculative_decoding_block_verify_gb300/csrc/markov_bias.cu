// The Markov head's previous-token logit bias on sm_103a.
//
// Method: "MTP Heads and Confidence Heads: Linking Three Self-Drafting Routes into One Chain"
// (naphjohn.github.io), §6 "Why the Markov Head Helps": a low-rank logit bias B = W1 @ W2
// (default rank 256) added to the draft logits by the previous token; "MTP, DSpark and Block
// Verification, Explained" (al-engr.com), §3 "The Markov fix-up" and Figure 2.
//
//   out[r, v] = draft[r, v] + sum_j W1[prev_r, j] * W2[j, v]
//
// At the draft-side shapes (a handful of rows per W2 pass) this is a gather-GEMV: W2 (rank x V)
// is streamed from HBM once per row group and every loaded W2 element feeds every row of the
// group from registers, so the bound is W2's bytes, not the FMAs; tensor cores would only
// add operand staging here.  Layout: a CTA owns a 32 x E column tile; its 4 warps split the
// rank dimension (a warp streams rank / 4 rows of the tile, eight 16-byte loads in flight per
// lane), each lane keeps (rows x E) float32 accumulators, and the warps' partial sums are added
// in shared memory in the epilogue.  Small CTAs let four of them share an SM, so the ~500
// column tiles of a 129,280-token vocabulary run as one wave with ~64 KB of W2 in flight per SM.

#include <atomic>
#include <cfloat>

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

template <int E>
static cudaError_t dispatch_bias(const BiasParams& p, int dt, int wt, cudaStream_t s) {
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
