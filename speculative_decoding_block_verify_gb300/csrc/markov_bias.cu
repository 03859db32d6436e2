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
// add operand staging here.  Layout: a CTA owns a 32 x E column tile; its 8 warps split the
// rank dimension, each lane keeps (rows x E) float32 accumulators, and the warps' partial sums
// are added in shared memory in the epilogue.

#include <cfloat>

#include "common.cuh"
#include "host_util.h"

namespace sv {

constexpr int kBiasThreads = 256;
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
__global__ void __launch_bounds__(kBiasThreads) markov_bias_kernel(const BiasParams p) {
    extern __shared__ float smem[];
    constexpr int kTile = 32 * E;
    constexpr int UJ = (E == 1) ? 8 : 4;
    float* w1s = smem;                          // [kRowGroup][R]
    float* red = smem + kRowGroup * p.R;        // [kBiasWarps][kRowGroup][kTile]
    __shared__ int row_ok[kRowGroup];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = p.V;
    const int64_t col0 = (int64_t)blockIdx.x * kTile;
    const int r0 = blockIdx.y * kRowGroup;
    const int nr = min(kRowGroup, p.rows - r0);

    // gather the group's W1 rows (float32) - an invalid prev zeroes its row and marks it
    for (int t = tid; t < kRowGroup * p.R; t += kBiasThreads) {
        const int r = t / p.R, j = t % p.R;
        float v = 0.f;
        if (r < nr) {
            const int pv = p.prev[r0 + r];
            if (pv >= 0 && pv < p.V) v = load_elem<WT>(p.W1, (int64_t)pv * p.R + j);
        }
        w1s[t] = v;
    }
    if (tid < kRowGroup) {
        int ok = 0;
        if (tid < nr) {
            const int pv = p.prev[r0 + tid];
            ok = (pv >= 0 && pv < p.V);
        }
        row_ok[tid] = ok;
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

    for (int j = j0; j < j1; j += UJ) {
        Chunk<WT, E> c[UJ];
#pragma unroll
        for (int u = 0; u < UJ; ++u)
            if (active && j + u < j1) c[u].load(row_ptr<WT>(p.W2, j + u, V), chunk);
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
    }
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int e = 0; e < E; ++e) red[(warp * kRowGroup + r) * kTile + lane * E + e] = acc[r][e];
    __syncthreads();

    const float qnan = __int_as_float(0x7fffffff);
    for (int o = tid; o < kRowGroup * kTile; o += kBiasThreads) {
        const int r = o / kTile, ci = o % kTile;
        const int64_t v = col0 + ci;
        if (r < nr && v < V) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kBiasWarps; ++w) s += red[(w * kRowGroup + r) * kTile + ci];
            const int64_t idx = (int64_t)(r0 + r) * V + v;
            const float d = load_elem<DT>(p.draft, idx);
            p.out[idx] = row_ok[r] ? d + s : qnan;
        }
    }
}

template <typename DT, typename WT, int E>
static cudaError_t launch_bias(const BiasParams& p, cudaStream_t s) {
    constexpr int kTile = 32 * E;
    const size_t smem = sizeof(float) * ((size_t)kRowGroup * p.R +
                                         (size_t)kBiasWarps * kRowGroup * kTile);
    cudaError_t e = cudaFuncSetAttribute(markov_bias_kernel<DT, WT, E>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
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
