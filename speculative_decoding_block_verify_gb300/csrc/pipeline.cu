// Acceptance counters and the adaptive verify step as one CUDA graph, on sm_103a.
//
// Method: "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com),
// §6 "The arithmetic you need before tuning k": the per-position acceptance rates a_p (the
// share of steps whose p-th draft was accepted) and tokens per step = 1 + sum_p a_p; §3 "The
// Markov fix-up" (the drafter's sampling runs inside the same CUDA graph as its forward pass)
// and "Two cliffs, not one" (a graph per batch size).  "Teaching the Speculator What a Draft
// Costs" (al-engr.com), "The controller, and the table it reads from": the controller picks
// how many drafts each stream verifies before the target runs.
//
// accept_counters_kernel: one pass over the batch's results; each CTA counts in shared memory
// and adds its counts to the caller's 64-bit accumulators once.
// The pipeline captures, once, on a private stream: adaptive_pick_k (confidence head,
// prefix survival, k per stream and the offsets) -> the verify over the dense draft/target
// layout with those counts -> the acceptance counters -> the step counter's increment; each
// launch then replays the whole step with one cudaGraphLaunch.

#include <cstdlib>
#include <new>

#include "common.cuh"
#include "host_util.h"

namespace sv {

constexpr int kCountThreads = 256;

// counts[0] += streams with status OK; counts[p] += OK streams with tau >= p (p = 1..kmax);
// counts[kmax + p] += OK streams that offered a p-th draft (N_b >= p).
__global__ void __launch_bounds__(kCountThreads) accept_counters_kernel(const int32_t* acc_len, const int32_t* status,
                                                                        const int32_t* cu, int B, int kmax,
                                                                        unsigned long long* counts) {
    __shared__ unsigned int c[2 * SPEC_MAX_KMAX + 1];
    for (int i = threadIdx.x; i < 2 * kmax + 1; i += blockDim.x) c[i] = 0u;
    __syncthreads();
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
        if (status[b] != SPEC_ST_OK) continue;
        atomicAdd(&c[0], 1u);
        const int tau = min(acc_len[b], kmax);
        const int n = min(cu[b + 1] - cu[b], kmax);
        for (int q = 1; q <= tau; ++q) atomicAdd(&c[q], 1u);
        for (int q = 1; q <= n; ++q) atomicAdd(&c[kmax + q], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * kmax + 1; i += blockDim.x)
        if (c[i]) atomicAdd(&counts[i], (unsigned long long)c[i]);
}

__global__ void step_increment_kernel(unsigned long long* step) { *step += 1ull; }

static cudaError_t launch_counters(const int32_t* acc_len, const int32_t* status, const int32_t* cu, int B, int kmax,
                                   uint64_t* counts, cudaStream_t s) {
    const int blocks = (B + kCountThreads - 1) / kCountThreads < 256 ? (B + kCountThreads - 1) / kCountThreads : 256;
    accept_counters_kernel<<<blocks, kCountThreads, 0, s>>>(acc_len, status, cu, B, kmax,
                                                            reinterpret_cast<unsigned long long*>(counts));
    return cudaGetLastError();
}

struct Pipeline {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

}  // namespace sv

extern "C" int spec_accept_counters(const int32_t* accepted_len, const int32_t* status, const int32_t* cu_drafts,
                                    int32_t B, int32_t kmax, uint64_t* counts, void* stream) {
    const char* name = "spec_accept_counters";
    if (B < 0 || kmax < 0 || kmax > SPEC_MAX_KMAX)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: B = %d, kmax = %d out of range", name, B, kmax);
    if (B == 0) return sv::clear_error();
    if (!accepted_len || !status || !cu_drafts || !counts)
        return sv::set_error(SPEC_ERR_ARG, "%s: a pointer is NULL", name);
    const cudaError_t e = sv::launch_counters(accepted_len, status, cu_drafts, B, kmax, counts,
                                              reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return sv::set_cuda_error(e, name);
    return sv::clear_error();
}

extern "C" int spec_pipeline_create(const spec_pipeline_args* a, void** pipeline) {
    const char* name = "spec_pipeline_create";
    if (a == nullptr || pipeline == nullptr) return sv::set_error(SPEC_ERR_ARG, "%s: NULL argument", name);
    *pipeline = nullptr;
    if (a->rule != 0 && a->rule != 1) return sv::set_error(SPEC_ERR_ARG, "%s: rule must be 0 or 1", name);
    if (a->B < 1 || a->kmax < 1 || a->kmax > SPEC_MAX_KMAX)
        return sv::set_error(SPEC_ERR_SHAPE, "%s: B = %d, kmax = %d out of range", name, a->B, a->kmax);
    if (!a->step || !a->k_out || !a->cu_drafts_out || !a->c_out || !a->a_out)
        return sv::set_error(SPEC_ERR_ARG, "%s: a required pointer is NULL", name);
    spec_verify_args v = {};
    v.B = a->B;
    v.V = a->V;
    v.kmax = a->kmax;
    v.cu_drafts = a->cu_drafts_out;
    v.draft_logits = a->draft_logits;
    v.draft_dtype = a->draft_dtype;
    v.target_logits = a->target_logits;
    v.target_dtype = a->target_dtype;
    v.draft_tokens = a->draft_tokens;
    v.temperature = a->temperature;
    v.seed = a->seed;
    v.accepted_len = a->accepted_len;
    v.out_tokens = a->out_tokens;
    v.n_emitted = a->n_emitted;
    v.status = a->status;
    v.diag = a->diag;
    v.workspace = a->workspace;
    v.workspace_bytes = a->workspace_bytes;
    const uint64_t* step = a->step;
    // every attribute, occupancy query and argument check before the capture
    const int rc = sv::verify_dense_launch(a->rule, &v, step, nullptr, true);
    if (rc != SPEC_OK) return rc;
    const size_t need = spec_verify_workspace_bytes(a->B, a->kmax);
    if (a->workspace == nullptr || a->workspace_bytes < need || (uintptr_t)a->workspace % 16 != 0)
        return sv::set_error(SPEC_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", name,
                             need, a->workspace_bytes);
    if (!a->accepted_len || !a->out_tokens || !a->n_emitted || !a->status || !a->draft_logits ||
        !a->target_logits || !a->draft_tokens || !a->temperature)
        return sv::set_error(SPEC_ERR_ARG, "%s: a required pointer is NULL", name);

    cudaStream_t s = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return sv::set_cuda_error(e, name);
    sv::Pipeline* pl = new (std::nothrow) sv::Pipeline();
    if (pl == nullptr) {
        cudaStreamDestroy(s);
        return sv::set_error(SPEC_ERR_ARG, "%s: out of host memory", name);
    }
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    int step_rc = SPEC_OK;
    if (e == cudaSuccess) {
        step_rc = adaptive_pick_k(a->hidden, a->w, a->head_dtype, a->bias, a->B, a->kmax, a->H, a->verify_ms,
                                  a->n_max, a->mode, a->c_out, a->a_out, a->k_out, a->cu_drafts_out, s);
        if (step_rc == SPEC_OK) step_rc = sv::verify_dense_launch(a->rule, &v, step, s, false);
        if (step_rc == SPEC_OK && a->accept_counts != nullptr) {
            const cudaError_t ce = sv::launch_counters(a->accepted_len, a->status, a->cu_drafts_out, a->B, a->kmax,
                                                       a->accept_counts, s);
            if (ce != cudaSuccess) step_rc = sv::set_cuda_error(ce, name);
        }
        if (step_rc == SPEC_OK) {
            sv::step_increment_kernel<<<1, 1, 0, s>>>(reinterpret_cast<unsigned long long*>(a->step));
            const cudaError_t ce = cudaGetLastError();
            if (ce != cudaSuccess) step_rc = sv::set_cuda_error(ce, name);
        }
        const cudaError_t ee = cudaStreamEndCapture(s, &pl->graph);
        if (step_rc == SPEC_OK && ee != cudaSuccess) e = ee;
    }
    if (e == cudaSuccess && step_rc == SPEC_OK) e = cudaGraphInstantiate(&pl->exec, pl->graph, 0);
    cudaStreamDestroy(s);
    if (e != cudaSuccess || step_rc != SPEC_OK) {
        if (pl->exec) cudaGraphExecDestroy(pl->exec);
        if (pl->graph) cudaGraphDestroy(pl->graph);
        delete pl;
        return step_rc != SPEC_OK ? step_rc : sv::set_cuda_error(e, name);
    }
    *pipeline = pl;
    return sv::clear_error();
}

extern "C" int spec_pipeline_launch(void* pipeline, void* stream) {
    if (pipeline == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_pipeline_launch: NULL pipeline");
    sv::Pipeline* pl = static_cast<sv::Pipeline*>(pipeline);
    const cudaError_t e = cudaGraphLaunch(pl->exec, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_pipeline_launch");
    return sv::clear_error();
}

extern "C" int spec_pipeline_destroy(void* pipeline) {
    if (pipeline == nullptr) return sv::clear_error();
    sv::Pipeline* pl = static_cast<sv::Pipeline*>(pipeline);
    if (pl->exec) cudaGraphExecDestroy(pl->exec);
    if (pl->graph) cudaGraphDestroy(pl->graph);
    delete pl;
    return sv::clear_error();
}
