// es_jit.h -- run-time compilation of body-program kernels (host code).
//
// A kernel source (a skeleton header, a generated functor) is compiled once
// with NVRTC for sm_103a, loaded into each device's context with the driver
// API and cached by its text, so a body program pays the compile on its
// first call and launches like a built-in kernel afterwards.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

namespace es {

struct JitKernel {
    CUfunction fn = nullptr;
};

// Compile `source` into the cache unless it is there (no device needed).
bool jit_compile(const std::string& source, const std::string& name_expr, std::string* err);

// Compile (or find in the cache) `source`, which includes skeleton headers by
// name and instantiates the kernel `name_expr` (e.g.
// "&es::k_body_lane<EsBody, 128, 32>"), and return it for the current
// device.  On failure returns false with a message (the NVRTC log for a
// compile error).
bool jit_kernel(const std::string& source, const std::string& name_expr, JitKernel* out, std::string* err);

// cuLaunchKernel on `stream` with `dyn_smem` bytes of dynamic shared memory
// (raising the kernel's limit first when above the default 48 KB).  Returns
// false with a message when the driver refuses the launch.
bool jit_launch(const JitKernel& k, unsigned grid, unsigned block, size_t dyn_smem, cudaStream_t stream, void** args,
                std::string* err);

// Number of NVRTC compilations so far (cache misses), for tests.
unsigned long long jit_compile_count();

}  // namespace es
