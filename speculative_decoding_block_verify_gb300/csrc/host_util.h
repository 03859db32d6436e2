// Host-side error reporting shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "specverify.h"

namespace sv {

// one message per host thread; defined in api.cu
char* error_buffer();
constexpr int kErrLen = 512;

inline int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(error_buffer(), kErrLen, fmt, ap);
    va_end(ap);
    return code;
}

inline int clear_error() {
    error_buffer()[0] = '\0';
    return SPEC_OK;
}

inline int set_cuda_error(cudaError_t e, const char* where) {
    return set_error(SPEC_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e),
                     cudaGetErrorName(e));
}

inline bool valid_dtype(int d) { return d == SPEC_DTYPE_F32 || d == SPEC_DTYPE_BF16; }

// The verify over the dense [B, kmax (+1), V] layout with the step read from device memory
// (defined in verify.cu; used by the adaptive pipeline).
int verify_dense_launch(int rule, const spec_verify_args* a, const uint64_t* step_dev, void* stream,
                        bool prepare_only);

}  // namespace sv
