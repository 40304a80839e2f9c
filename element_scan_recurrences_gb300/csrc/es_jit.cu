// es_jit.cu -- NVRTC compilation and driver-API loading of body-program
// kernels (see es_jit.h).
//
// The skeleton headers are compiled into the library as text (the build
// writes them into es_jit_headers.inc) and handed to NVRTC as in-memory
// headers, so nothing is read from disk at run time.  The driver entry points
// are fetched through the runtime, like cuTensorMapEncodeTiled, so the
// library still loads on machines without a GPU driver.
#include "es_jit.h"

#include <nvrtc.h>

#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

#include "es_jit_headers.inc"   // kJitHeaderCount, kJitHeaderNames[], kJitHeaderSources[]

namespace es {
namespace {

typedef CUresult (*ModuleLoadDataFn)(CUmodule*, const void*);
typedef CUresult (*ModuleGetFunctionFn)(CUfunction*, CUmodule, const char*);
typedef CUresult (*FuncSetAttributeFn)(CUfunction, CUfunction_attribute, int);
typedef CUresult (*LaunchKernelFn)(CUfunction, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned,
                                   CUstream, void**, void**);
typedef CUresult (*GetErrorStringFn)(CUresult, const char**);

struct Driver {
    ModuleLoadDataFn module_load_data = nullptr;
    ModuleGetFunctionFn module_get_function = nullptr;
    FuncSetAttributeFn func_set_attribute = nullptr;
    LaunchKernelFn launch_kernel = nullptr;
    GetErrorStringFn get_error_string = nullptr;
    bool ok = false;
};

Driver& driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, []() {
        auto get = [](const char* name) -> void* {
            void* p = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess)
                return nullptr;
            return p;
        };
        d.module_load_data = reinterpret_cast<ModuleLoadDataFn>(get("cuModuleLoadData"));
        d.module_get_function = reinterpret_cast<ModuleGetFunctionFn>(get("cuModuleGetFunction"));
        d.func_set_attribute = reinterpret_cast<FuncSetAttributeFn>(get("cuFuncSetAttribute"));
        d.launch_kernel = reinterpret_cast<LaunchKernelFn>(get("cuLaunchKernel"));
        d.get_error_string = reinterpret_cast<GetErrorStringFn>(get("cuGetErrorString"));
        d.ok = d.module_load_data && d.module_get_function && d.func_set_attribute && d.launch_kernel &&
               d.get_error_string;
    });
    return d;
}

std::string driver_error(const char* what, CUresult r) {
    const char* s = nullptr;
    if (driver().get_error_string == nullptr || driver().get_error_string(r, &s) != CUDA_SUCCESS || s == nullptr)
        s = "unknown driver error";
    return std::string(what) + ": " + s;
}

constexpr int kMaxDevices = 64;

struct Entry {
    std::string cubin;
    std::string lowered;          // mangled kernel name
    CUmodule module[kMaxDevices] = {};
    CUfunction fn[kMaxDevices] = {};
};

std::mutex g_mu;
std::map<std::string, std::unique_ptr<Entry>> g_cache;
std::atomic<unsigned long long> g_compiles{0};

bool compile(const std::string& source, const std::string& name_expr, Entry* e, std::string* err) {
    nvrtcProgram prog;
    nvrtcResult r = nvrtcCreateProgram(&prog, source.c_str(), "es_body_kernel.cu", kJitHeaderCount,
                                       kJitHeaderSources, kJitHeaderNames);
    if (r != NVRTC_SUCCESS) {
        *err = std::string("nvrtcCreateProgram: ") + nvrtcGetErrorString(r);
        return false;
    }
    nvrtcAddNameExpression(prog, name_expr.c_str());
    const char* opts[] = {"--gpu-architecture=sm_103a", "-std=c++17", "-lineinfo"};
    r = nvrtcCompileProgram(prog, 3, opts);
    if (r != NVRTC_SUCCESS) {
        size_t n = 0;
        nvrtcGetProgramLogSize(prog, &n);
        std::string log(n, '\0');
        if (n > 0) nvrtcGetProgramLog(prog, &log[0]);
        *err = std::string("NVRTC could not compile the body kernel: ") + nvrtcGetErrorString(r) + "\n" + log;
        nvrtcDestroyProgram(&prog);
        return false;
    }
    const char* lowered = nullptr;
    size_t n = 0;
    if (nvrtcGetLoweredName(prog, name_expr.c_str(), &lowered) != NVRTC_SUCCESS || lowered == nullptr ||
        nvrtcGetCUBINSize(prog, &n) != NVRTC_SUCCESS) {
        *err = "NVRTC produced no kernel " + name_expr;
        nvrtcDestroyProgram(&prog);
        return false;
    }
    e->lowered = lowered;
    e->cubin.assign(n, '\0');
    nvrtcGetCUBIN(prog, &e->cubin[0]);
    nvrtcDestroyProgram(&prog);
    g_compiles.fetch_add(1);
    return true;
}

// the cache entry of a source, compiled on first use; call with g_mu held
Entry* cached(const std::string& source, const std::string& name_expr, std::string* err) {
    const std::string key = name_expr + '\n' + source;
    auto it = g_cache.find(key);
    if (it == g_cache.end()) {
        std::unique_ptr<Entry> e(new Entry());
        if (!compile(source, name_expr, e.get(), err)) return nullptr;
        it = g_cache.emplace(key, std::move(e)).first;
    }
    return it->second.get();
}

}  // namespace

bool jit_compile(const std::string& source, const std::string& name_expr, std::string* err) {
    std::lock_guard<std::mutex> lock(g_mu);
    return cached(source, name_expr, err) != nullptr;
}

bool jit_kernel(const std::string& source, const std::string& name_expr, JitKernel* out, std::string* err) {
    Driver& d = driver();
    if (!d.ok) {
        *err = "the CUDA driver does not provide the module API";
        return false;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = "no usable current device";
        return false;
    }
    // the runtime's primary context must be current for the driver calls
    if (cudaSetDevice(dev) != cudaSuccess) {
        *err = "cudaSetDevice failed";
        return false;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    Entry* found = cached(source, name_expr, err);
    if (found == nullptr) return false;
    Entry& e = *found;
    if (e.fn[dev] == nullptr) {
        CUresult r = d.module_load_data(&e.module[dev], e.cubin.data());
        if (r != CUDA_SUCCESS) {
            *err = driver_error("cuModuleLoadData", r);
            return false;
        }
        r = d.module_get_function(&e.fn[dev], e.module[dev], e.lowered.c_str());
        if (r != CUDA_SUCCESS) {
            *err = driver_error("cuModuleGetFunction", r);
            return false;
        }
    }
    out->fn = e.fn[dev];
    return true;
}

bool jit_launch(const JitKernel& k, unsigned grid, unsigned block, size_t dyn_smem, cudaStream_t stream, void** args,
                std::string* err) {
    Driver& d = driver();
    if (dyn_smem > 48 * 1024) {
        CUresult r = d.func_set_attribute(k.fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES,
                                          static_cast<int>(dyn_smem));
        if (r != CUDA_SUCCESS) {
            *err = driver_error("cuFuncSetAttribute", r);
            return false;
        }
    }
    CUresult r = d.launch_kernel(k.fn, grid, 1, 1, block, 1, 1, static_cast<unsigned>(dyn_smem),
                                 reinterpret_cast<CUstream>(stream), args, nullptr);
    if (r != CUDA_SUCCESS) {
        *err = driver_error("cuLaunchKernel", r);
        return false;
    }
    return true;
}

unsigned long long jit_compile_count() { return g_compiles.load(); }

}  // namespace es
