// Confidence head and adaptive verification (pick how many drafts to verify) on sm_103a.
//
// Method: "MTP Heads and Confidence Heads" (naphjohn.github.io), §7 (c_k = sigmoid(Linear(h))),
// §9 (prefix survival a_j = c_1 ... c_j) and the figure text after §9 (the scheduler adds
// candidates in descending a_j); "MTP, DSpark and Block Verification, Explained" (al-engr.com),
// §6 (tokens per step = 1 + sum of a); "Teaching the Speculator What a Draft Costs"
// (al-engr.com), "The controller, and the table it reads from" (best expected tokens per
// millisecond, cost from verify_ms[num_tokens]).
//
// Kernel 1: one CTA (16 warps) per stream, `split` warps per draft slot (up to 4, as many as
// 16 warps allow; with more than 16 slots a warp takes two): each warp takes a contiguous
// share of the dot h . w with all of a lane's 16-byte loads in flight at once (float32
// accumulation; at H = 7168 a lane's share is 7 chunks, so the hidden state streams in one
// round trip), the shares are added in a fixed order, then one warp takes sigmoid, cumulative
// product and - in per-stream mode - the stream's own pick, with scans across its lanes.
// Kernel 2: one CTA, launched as a programmatic dependent of kernel 1 (its launch overlaps
// kernel 1): batch mode's ordering of all (stream, slot) entries and its pick, then the
// exclusive prefix sum that gives cu_drafts.

#include <atomic>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "df.cuh"
#include "host_util.h"

namespace sv {

constexpr int kPickThreads = 1024;
constexpr int kMaxBatchEntries = 4096;
constexpr int kConfMaxSplit = 4;   // warps per dot product
constexpr int kConfWarps = 16;     // warps of a confidence CTA: items (slot, share) go round them

struct PickParams {
    const void* hidden;
    const void* w;
    double bias;
    int32_t B, kmax, H, mode, n_max;
    const float* verify_ms;
    float* c_out;
    float* a_out;
    int32_t* k_out;
    int32_t* cu_out;
    int64_t nchunk;
    int32_t split;   // warps per dot product
};

template <typename T, int E>
__global__ void __launch_bounds__(kConfWarps * 32) confidence_kernel(const PickParams p) {
    __shared__ float part_s[SPEC_MAX_KMAX * kConfMaxSplit];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t per = (p.nchunk + p.split - 1) / p.split;
    // chunks per lane in flight at once: 10 (bf16) cover a warp's third of H = 7168 (299
    // chunks) in one round of loads, where 8 took two (6.1 -> 5.8 us at B = 128, kmax = 5)
    constexpr int U = (sizeof(T) == 2) ? 10 : 5;
    for (int item = warp; item < p.kmax * p.split; item += kConfWarps) {
        const int slot = item / p.split, part = item - slot * p.split;
        const int64_t k0 = min(p.nchunk, (int64_t)part * per), k1 = min(p.nchunk, k0 + per);
        const void* hrow = row_ptr<T>(p.hidden, (int64_t)b * p.kmax + slot, p.H);
        float acc = 0.f;
        for (int64_t base = k0; base < k1; base += 32 * U) {
            Chunk<T, E> ch[U], cw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t k = base + u * 32 + lane;
                if (k < k1) {
                    ch[u].load(hrow, k);
                    cw[u].load(p.w, k);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t k = base + u * 32 + lane;
                if (k < k1) {
                    float xh[E], xw[E];
                    ch[u].unpack(xh);
                    cw[u].unpack(xw);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc = fmaf(xh[e], xw[e], acc);
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) part_s[item] = acc;
    }
    __syncthreads();
    // the stream's tail in one warp (float32, exact-rounding exp and divide): lane j holds slot
    // j: c_j, the prefix product a_j, E_{j+1} = 1 + a_0 + ... + a_j (scans across the lanes),
    // and the controller's best n by E_n / verify_ms[n + 1] (ties -> the smaller n)
    if (warp == 0) {
        const int j = lane;
        float cj = 1.f;
        if (j < p.kmax) {
            float dot = 0.f;
            for (int q = 0; q < p.split; ++q) dot += part_s[j * p.split + q];   // a fixed order
            const float x = dot + (float)p.bias;
            cj = (x >= 0.f) ? 1.f / (1.f + expf(-x)) : expf(x) / (1.f + expf(x));
        }
        float a = cj;   // inclusive prefix product
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, a, o);
            if (lane >= o) a *= n;
        }
        float sa = (j < p.kmax) ? a : 0.f;   // inclusive prefix sum of a
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, sa, o);
            if (lane >= o) sa += n;
        }
        if (j < p.kmax) {
            p.c_out[(int64_t)b * p.kmax + j] = cj;
            p.a_out[(int64_t)b * p.kmax + j] = a;
        }
        // candidate n = j + 1 (lane j), n = 0 (lane 0 also holds it)
        float best = (j < p.kmax) ? (1.f + sa) / p.verify_ms[j + 2] : -1.f;
        int best_n = j + 1;
        if (lane == 0) {
            const float r0 = 1.f / p.verify_ms[1];
            if (!(best > r0)) {
                best = r0;
                best_n = 0;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int on = __shfl_xor_sync(0xffffffffu, best_n, o);
            if (ob > best || (ob == best && on < best_n)) {
                best = ob;
                best_n = on;
            }
        }
        if (p.mode == 0 && lane == 0) p.k_out[b] = best_n;
    }
}

// exclusive prefix sum of k over the batch (one CTA)
__device__ void write_cu(const int32_t* k, int32_t* cu, int B) {
    __shared__ int carry;
    __shared__ int warp_tot[kPickThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < B; base += kPickThreads) {
        const int i = base + tid;
        int v = (i < B) ? k[i] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int wofs = 0;
        for (int w = 0; w < warp; ++w) wofs += warp_tot[w];
        if (i < B) cu[i] = carry + wofs + incl - v;
        __syncthreads();
        if (tid == kPickThreads - 1) carry += wofs + incl;
        __syncthreads();
    }
    if (tid == 0) cu[B] = carry;
}

// Batch mode's ordering as a bitonic sort of 64-bit keys in shared memory: key = (~bits of
// a) << 32 | entry, entry = b kmax + j.  Sorting the keys ascending orders a descending (a is
// in [0, 1], where the float bits are monotone) and equal a by (stream, slot) ascending, the
// order the pages' scheduler adds candidates in.  Padding keys (all ones) sort last.
__device__ __forceinline__ float key_a(unsigned long long key) { return __uint_as_float(~(uint32_t)(key >> 32)); }
__device__ __forceinline__ int key_entry(unsigned long long key) { return (int)(uint32_t)key; }

__global__ void __launch_bounds__(kPickThreads) pick_batch_kernel(const PickParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // every confidence CTA has finished
    extern __shared__ __align__(16) unsigned long long keys[];   // [npow2], then k_s [B] int
    __shared__ df best_v[kPickThreads / 32];
    __shared__ int best_m[kPickThreads / 32];
    __shared__ df seg_tot[kPickThreads / 32];
    __shared__ df seg_ofs[kPickThreads / 32];
    __shared__ int m_star;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.B * p.kmax;
    if (p.mode == 1) {
        int npow2 = 1;
        while (npow2 < n) npow2 <<= 1;
        int* k_s = reinterpret_cast<int*>(keys + npow2);
        for (int e = tid; e < npow2; e += kPickThreads)
            keys[e] = e < n ? ((unsigned long long)(~__float_as_uint(p.a_out[e])) << 32) | (unsigned)e : ~0ull;
        for (int b = tid; b < p.B; b += kPickThreads) k_s[b] = 0;
        __syncthreads();
        for (int kk = 2; kk <= npow2; kk <<= 1)
            for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                for (int i = tid; i < npow2; i += kPickThreads) {
                    const int ixj = i ^ jj;
                    if (ixj > i) {
                        const unsigned long long x = keys[i], y = keys[ixj];
                        if ((x > y) == ((i & kk) == 0)) {
                            keys[i] = y;
                            keys[ixj] = x;
                        }
                    }
                }
                __syncthreads();
            }
        // S_m for m = 1..n: each thread owns a contiguous run of ranks.  Double-float scalars
        // (~48 bits; this part's float64 pipe is narrow): the run sums, one scan across the lanes,
        // one across the warps' totals, then every m's ratio (B + S_m) / verify_ms[B + m].
        const int per = (n + kPickThreads - 1) / kPickThreads;
        const int m0 = min(n, tid * per), m1 = min(n, m0 + per);
        df run{0.f, 0.f};
        for (int m = m0; m < m1; ++m) run = df_add_f(run, key_a(keys[m]));
        df incl = run;   // inclusive scan of the runs across the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const df nb{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
            if (lane >= o) incl = df_add(incl, nb);
        }
        if (lane == 31) seg_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {   // exclusive scan of the warps' totals
            df t = lane < kPickThreads / 32 ? seg_tot[lane] : df{0.f, 0.f};
            df inc = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const df nb{__shfl_up_sync(0xffffffffu, inc.hi, o), __shfl_up_sync(0xffffffffu, inc.lo, o)};
                if (lane >= o) inc = df_add(inc, nb);
            }
            if (lane < kPickThreads / 32) seg_ofs[lane] = df_sub(inc, t);
        }
        __syncthreads();
        df sm = df_sub(df_add(seg_ofs[warp], incl), run);   // the sum of the ranks before m0
        // best ratio over this thread's m (m = number chosen, 1-based); m = 0 handled below
        df bv{-1.f, 0.f};
        int bm = INT_MAX;
        const df Bd = df_make((float)p.B);
        for (int m = m0; m < m1; ++m) {
            sm = df_add_f(sm, key_a(keys[m]));
            const df v = df_div(df_add(Bd, sm), df_make(p.verify_ms[p.B + m + 1]));
            if (df_lt(bv, v)) {
                bv = v;
                bm = m + 1;
            }
        }
        if (tid == 0) {
            const df v0 = df_div(Bd, df_make(p.verify_ms[p.B]));
            if (!df_lt(v0, bv)) {   // ties go to the smaller m
                bv = v0;
                bm = 0;
            }
        }
        // block argmax (larger value, then smaller m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const df ov{__shfl_xor_sync(0xffffffffu, bv.hi, o), __shfl_xor_sync(0xffffffffu, bv.lo, o)};
            const int om = __shfl_xor_sync(0xffffffffu, bm, o);
            if (df_lt(bv, ov) || (!df_lt(ov, bv) && om < bm)) {
                bv = ov;
                bm = om;
            }
        }
        if (lane == 0) {
            best_v[warp] = bv;
            best_m[warp] = bm;
        }
        __syncthreads();
        if (tid == 0) {
            df v = best_v[0];
            int m = best_m[0];
            for (int w = 1; w < kPickThreads / 32; ++w)
                if (df_lt(v, best_v[w]) || (!df_lt(best_v[w], v) && best_m[w] < m)) {
                    v = best_v[w];
                    m = best_m[w];
                }
            m_star = m;
        }
        __syncthreads();
        for (int r = tid; r < m_star; r += kPickThreads) atomicAdd(&k_s[key_entry(keys[r]) / p.kmax], 1);
        __syncthreads();
        for (int b = tid; b < p.B; b += kPickThreads) p.k_out[b] = k_s[b];
        __syncthreads();
        write_cu(k_s, p.cu_out, p.B);
    } else {
        write_cu(p.k_out, p.cu_out, p.B);
    }
}

template <typename T, int E>
static cudaError_t launch_pick(PickParams p, cudaStream_t s) {
    p.split = kConfWarps / p.kmax < kConfMaxSplit ? kConfWarps / p.kmax : kConfMaxSplit;
    if (p.split < 1) p.split = 1;
    confidence_kernel<T, E><<<p.B, kConfWarps * 32, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    size_t smem = 0;
    if (p.mode == 1) {   // the sort keys and the per-stream counts
        int npow2 = 1;
        while (npow2 < p.B * p.kmax) npow2 <<= 1;
        smem = (size_t)npow2 * sizeof(unsigned long long) + (size_t)p.B * sizeof(int);
        static std::atomic<int> attr_set[64];
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
            e = cudaFuncSetAttribute(pick_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kMaxBatchEntries * (sizeof(unsigned long long) + sizeof(int))));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev].store(1, std::memory_order_release);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPickThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pick_batch_kernel, p);
}

}  // namespace sv

extern "C" int adaptive_pick_k(const void* hidden, const void* w, int32_t dtype, float bias,
                               int32_t B, int32_t kmax, int32_t H, const float* verify_ms,
                               int32_t n_max, int32_t mode, float* c_out, float* a_out,
                               int32_t* k_out, int32_t* cu_drafts_out, void* stream) {
    const char* name = "adaptive_pick_k";
    if (mode != 0 && mode != 1) return sv::set_error(SPEC_ERR_ARG, "%s: mode must be 0 or 1", name);
    if (!sv::valid_dtype(dtype))
        return sv::set_error(SPEC_ERR_DTYPE, "%s: dtype must be SPEC_DTYPE_F32 or SPEC_DTYPE_BF16",
                             name);
    if (B < 1 || kmax < 1 || kmax > SPEC_MAX_KMAX || H < 1)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: B=%d kmax=%d H=%d out of range", name, B, kmax, H);
    if (mode == 0 && n_max < kmax + 1)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: verify_ms needs n_max >= kmax + 1", name);
    if (mode == 1 && ((int64_t)B * (kmax + 1) > n_max || (int64_t)B * kmax > sv::kMaxBatchEntries))
        return sv::set_error(SPEC_ERR_SHAPE,
                             "%s: batch mode needs n_max >= B*(kmax+1) and B*kmax <= %d", name,
                             sv::kMaxBatchEntries);
    if (!hidden || !w || !verify_ms || !c_out || !a_out || !k_out || !cu_drafts_out)
        return sv::set_error(SPEC_ERR_ARG, "%s: a pointer is NULL", name);
    sv::PickParams p;
    p.hidden = hidden;
    p.w = w;
    p.bias = (double)bias;
    p.B = B;
    p.kmax = kmax;
    p.H = H;
    p.mode = mode;
    p.n_max = n_max;
    p.verify_ms = verify_ms;
    p.c_out = c_out;
    p.a_out = a_out;
    p.k_out = k_out;
    p.cu_out = cu_drafts_out;
    const bool aligned = (H % 8 == 0) && ((uintptr_t)hidden % 16 == 0) && ((uintptr_t)w % 16 == 0);
    p.nchunk = aligned ? H / 8 : H;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == SPEC_DTYPE_BF16)
        e = aligned ? sv::launch_pick<__nv_bfloat16, 8>(p, s) : sv::launch_pick<__nv_bfloat16, 1>(p, s);
    else
        e = aligned ? sv::launch_pick<float, 8>(p, s) : sv::launch_pick<float, 1>(p, s);
    if (e != cudaSuccess) return sv::set_cuda_error(e, name);
    return sv::clear_error();
}
