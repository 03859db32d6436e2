// The online verify-cost curve for adaptive_pick_k (host code).
//
// Method: "Teaching the Speculator What a Draft Costs" (al-engr.com), "What we changed" and
// "Reproduce": around every real verification step a pair of CUDA events is recorded; the
// elapsed time is read later, without ever making the host wait for the GPU, and filed under
// the step's token count; every rebuild_every observations the controller's table is rebuilt
// from the boot curve with the live medians laid on top (knobs: window 32, min samples 3,
// rebuild every 32).  Readings where the page is terse: the median of an even number of samples
// is the mean of the two middle ones; a token count with fewer than min_samples live samples
// keeps its boot value; an event pair that has not completed stays pending (pairs are folded in
// in the order they were recorded), and a begin with every pair slot pending records nothing.
//
// The token count of a step may live on the device (the controller picks it there): end() then
// launches a one-thread kernel after the end event that stores it into mapped pinned memory (no
// copy-engine round trip on the stream), so the timed region holds the verify alone and the
// count is read on the host only once that store has completed.
//
// The table the controller reads lives in device memory; upload() copies the current table
// there asynchronously on the caller's stream from one of two pinned host buffers, so a copy
// in flight is never overwritten by the next rebuild.

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "host_util.h"

namespace sv {

struct CostCurve {
    int n_max = 0, window = 32, min_samples = 3, rebuild_every = 32;
    std::vector<float> boot, table;
    std::vector<std::vector<float>> samples;   // per token count: circular, at most `window`
    std::vector<int> next;                     // per token count: next slot of the circle
    long long observations = 0, dropped = 0;
    int rebuilds = 0, since_rebuild = 0;
    bool dirty = false;                        // the table changed since the last upload
    // event pairs in flight (a ring): start, end, "count read", token count
    static constexpr int kPairs = 64;
    cudaEvent_t ev_start[kPairs] = {}, ev_end[kPairs] = {}, ev_ready[kPairs] = {};
    int pair_tokens[kPairs] = {};
    int32_t* pinned_count = nullptr;           // [kPairs] device counts read back (mapped)
    int32_t* mapped_count = nullptr;           // the device address of pinned_count
    bool from_device[kPairs] = {};
    int head = 0, count = 0;                   // oldest pending pair, pending pairs
    int open = -1;                             // the pair whose end is still to be recorded
    float* pinned[2] = {nullptr, nullptr};
    cudaEvent_t copied[2] = {};
    int next_buffer = 0;

    void observe(int n, float ms) {
        if (n < 0 || n > n_max || !(ms >= 0.f)) {
            ++dropped;
            return;
        }
        std::vector<float>& s = samples[n];
        if ((int)s.size() < window) s.push_back(ms);
        else s[next[n]] = ms;
        next[n] = (next[n] + 1) % window;
        ++observations;
        if (++since_rebuild >= rebuild_every) rebuild();
    }
    void rebuild() {
        since_rebuild = 0;
        ++rebuilds;
        for (int n = 0; n <= n_max; ++n) {
            const std::vector<float>& s = samples[n];
            float v = boot[n];
            if ((int)s.size() >= min_samples) {
                std::vector<float> t(s);
                std::sort(t.begin(), t.end());
                const size_t m = t.size() / 2;
                v = (t.size() % 2) ? t[m] : 0.5f * (t[m - 1] + t[m]);
            }
            if (v != table[n]) dirty = true;
            table[n] = v;
        }
    }
};

__global__ void read_count_kernel(const int32_t* src, int32_t* dst) { *dst = *src; }

}  // namespace sv

extern "C" void* spec_cost_curve_create(const float* boot_ms, int32_t n_max, int32_t window, int32_t min_samples,
                                        int32_t rebuild_every) {
    if (boot_ms == nullptr || n_max < 1 || window < 1 || min_samples < 1 || min_samples > window || rebuild_every < 1) {
        sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_create: invalid argument");
        return nullptr;
    }
    sv::CostCurve* c = new (std::nothrow) sv::CostCurve();
    if (c == nullptr) {
        sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_create: out of host memory");
        return nullptr;
    }
    c->n_max = n_max;
    c->window = window;
    c->min_samples = min_samples;
    c->rebuild_every = rebuild_every;
    c->boot.assign(boot_ms, boot_ms + n_max + 1);
    c->table = c->boot;
    c->samples.assign(n_max + 1, std::vector<float>());
    c->next.assign(n_max + 1, 0);
    sv::clear_error();
    return c;
}

static cudaError_t ensure_events(sv::CostCurve* c) {
    if (c->mapped_count != nullptr) return cudaSuccess;
    for (int i = 0; i < sv::CostCurve::kPairs; ++i) {   // (what a failed earlier call made is kept)
        cudaError_t e = cudaSuccess;
        if (c->ev_start[i] == nullptr) e = cudaEventCreate(&c->ev_start[i]);
        if (e == cudaSuccess && c->ev_end[i] == nullptr) e = cudaEventCreate(&c->ev_end[i]);
        if (e == cudaSuccess && c->ev_ready[i] == nullptr)
            e = cudaEventCreateWithFlags(&c->ev_ready[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    if (c->pinned_count != nullptr)
        return cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->mapped_count), c->pinned_count, 0);
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&c->pinned_count), sizeof(int32_t) * sv::CostCurve::kPairs,
                                  cudaHostAllocMapped);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->mapped_count), c->pinned_count, 0);
    return e;
}

// Event pairs must go on a stream that is not being captured: a captured record is a graph
// dependency, not a timestamp.
static int refuse_capture(cudaStream_t s, const char* where) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &st);
    if (e != cudaSuccess) return sv::set_cuda_error(e, where);
    if (st != cudaStreamCaptureStatusNone) return sv::set_error(SPEC_ERR_ARG, "%s: the stream is capturing", where);
    return SPEC_OK;
}

extern "C" int spec_cost_curve_begin(void* curve, void* stream) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_begin: NULL curve");
    if (c->open != -1) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_begin: the previous begin has no end");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = refuse_capture(s, "spec_cost_curve_begin");
    if (rc != SPEC_OK) return rc;
    cudaError_t e = ensure_events(c);
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_cost_curve_begin");
    if (c->count == sv::CostCurve::kPairs) {   // every pair still pending: this step goes unobserved
        ++c->dropped;
        c->open = -2;
        return sv::clear_error();
    }
    const int slot = (c->head + c->count) % sv::CostCurve::kPairs;
    e = cudaEventRecord(c->ev_start[slot], s);
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_cost_curve_begin");
    c->open = slot;
    return sv::clear_error();
}

extern "C" int spec_cost_curve_end(void* curve, int32_t num_tokens, const int32_t* device_count, void* stream) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_end: NULL curve");
    if (c->open == -2) {   // its begin had no free pair
        c->open = -1;
        return sv::clear_error();
    }
    if (c->open < 0) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_end: no matching begin");
    const int slot = c->open;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(c->ev_end[slot], s);
    if (e == cudaSuccess && device_count != nullptr) {
        sv::read_count_kernel<<<1, 1, 0, s>>>(device_count, c->mapped_count + slot);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_ready[slot], s);
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_cost_curve_end");
    c->pair_tokens[slot] = num_tokens;
    c->from_device[slot] = device_count != nullptr;
    c->open = -1;
    ++c->count;
    return sv::clear_error();
}

extern "C" int spec_cost_curve_observe(void* curve, int32_t num_tokens, float ms) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_observe: NULL curve");
    c->observe(num_tokens, ms);
    return sv::clear_error();
}

extern "C" int spec_cost_curve_poll(void* curve) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_poll: NULL curve");
    while (c->count > 0) {
        const int slot = c->head;
        const cudaError_t q = cudaEventQuery(c->ev_ready[slot]);
        if (q == cudaErrorNotReady) break;   // never wait: this pair and later ones fold in on a later poll
        if (q != cudaSuccess) return sv::set_cuda_error(q, "spec_cost_curve_poll");
        float ms = 0.f;
        const cudaError_t e = cudaEventElapsedTime(&ms, c->ev_start[slot], c->ev_end[slot]);
        if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_cost_curve_poll");
        c->observe(c->pair_tokens[slot] + (c->from_device[slot] ? c->pinned_count[slot] : 0), ms);
        c->head = (c->head + 1) % sv::CostCurve::kPairs;
        --c->count;
    }
    return sv::clear_error();
}

extern "C" int spec_cost_curve_table(void* curve, float* out, int64_t* counters) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr || out == nullptr) return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_table: NULL argument");
    std::memcpy(out, c->table.data(), sizeof(float) * (c->n_max + 1));
    if (counters != nullptr) {
        counters[0] = c->observations;
        counters[1] = c->rebuilds;
        counters[2] = c->dropped;
        counters[3] = c->count;
    }
    return sv::clear_error();
}

extern "C" int spec_cost_curve_upload(void* curve, float* device_table, void* stream) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr || device_table == nullptr)
        return sv::set_error(SPEC_ERR_ARG, "spec_cost_curve_upload: NULL argument");
    if (!c->dirty) return sv::clear_error();
    const size_t bytes = sizeof(float) * (c->n_max + 1);
    const int b = c->next_buffer;
    cudaError_t e = cudaSuccess;
    if (c->pinned[b] == nullptr) {
        e = cudaMallocHost(reinterpret_cast<void**>(&c->pinned[b]), bytes);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->copied[b], cudaEventDisableTiming);
        if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_cost_curve_upload");
    } else {
        const cudaError_t q = cudaEventQuery(c->copied[b]);
        if (q == cudaErrorNotReady) return sv::clear_error();   // its last copy is in flight: next time
        if (q != cudaSuccess) return sv::set_cuda_error(q, "spec_cost_curve_upload");
    }
    std::memcpy(c->pinned[b], c->table.data(), bytes);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(device_table, c->pinned[b], bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaEventRecord(c->copied[b], s);
    if (e != cudaSuccess) return sv::set_cuda_error(e, "spec_cost_curve_upload");
    c->dirty = false;
    c->next_buffer = 1 - b;
    return sv::clear_error();
}

extern "C" void spec_cost_curve_destroy(void* curve) {
    sv::CostCurve* c = static_cast<sv::CostCurve*>(curve);
    if (c == nullptr) return;
    for (int i = 0; i < sv::CostCurve::kPairs; ++i) {
        if (c->ev_start[i]) cudaEventDestroy(c->ev_start[i]);
        if (c->ev_end[i]) cudaEventDestroy(c->ev_end[i]);
        if (c->ev_ready[i]) {
            cudaEventSynchronize(c->ev_ready[i]);
            cudaEventDestroy(c->ev_ready[i]);
        }
    }
    if (c->pinned_count) cudaFreeHost(c->pinned_count);
    for (int b = 0; b < 2; ++b) {
        if (c->copied[b]) {
            cudaEventSynchronize(c->copied[b]);
            cudaEventDestroy(c->copied[b]);
        }
        if (c->pinned[b]) cudaFreeHost(c->pinned[b]);
    }
    delete c;
}
