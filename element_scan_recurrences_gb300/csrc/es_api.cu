// es_api.cu -- the C ABI of libes.so (declared in include/es.h): argument
// validation, canonicalisation to [O, T, J, W], kernel-path choice and launch.
//
// Argument contract: "Nonlinear element scans", "Arguments and body" table
// (initial = sequence shape minus the axis; sequences share one shape, under
// a state axis except for their own last width; the axis may be negative and
// its length is at least one; the state axis is the last axis and holds 1 to
// 16 values).  Error classes: "Tensor operations", "Errors" (E-DIM-001 shapes
// do not fit, E-DIM-002 dtypes; messages name both operands with their shapes).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "es.h"
#include "es_internal.h"

// One status word per device, in the library's own device memory (module
// scope), so no call allocates anything.  Kernels OR in ES_DEVICE_TIMEOUT.
static __device__ unsigned int g_es_device_status;

namespace {

thread_local std::string t_error;

std::atomic<int> g_path_override{ES_PATH_AUTO};
std::atomic<uint64_t> g_wait_ns{2000000000ull};
std::atomic<int64_t> g_drop_tile{-1};
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
using es::DeviceState;
DeviceState g_dev[kMaxDevices];

std::once_flag g_encode_once;
es::EncodeTiledFn g_encode = nullptr;

es_status fail(es_status st, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_error = buf;
    return st;
}

std::string shape_str(const int64_t* shape, int rank, int replace_last = -1, int64_t last = 0) {
    std::string s = "[";
    for (int d = 0; d < rank; ++d) {
        if (d) s += ", ";
        s += std::to_string((d == rank - 1 && replace_last >= 0) ? last : shape[d]);
    }
    return s + "]";
}

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

struct Plan {
    int64_t O, T, J, W;
    int64_t sw[2];
    int64_t n_out, n_init, n_seq[2];
    int path;
};

const char* kSeqName[3][2] = {{"x", "a"}, {"x", "a"}, {"x", "c"}};

es_status plan_impl(es_body body, const float* initial, const float* const* seqs, int n_seqs, const int64_t* shape,
                    int rank, int axis, int state_width, const int64_t* seq_widths, const float* out, int forced,
                    Plan* P) {
    if (body != ES_TANH_DECAY && body != ES_NORMCAP && body != ES_MAXPLUS)
        return fail(ES_E_ARG, "es_scan_f32: unknown body id %d", static_cast<int>(body));
    if (n_seqs != 2)
        return fail(ES_E_ARG, "es_scan_f32: body %d takes the state and 2 sequences, got %d sequences",
                    static_cast<int>(body), n_seqs);
    if (state_width == 0 && body == ES_NORMCAP && shape != nullptr && seqs != nullptr)
        return fail(ES_E_UNSUPPORTED, "es_scan_f32: NORMCAP reduces over its state and needs a state axis "
                    "(state_width >= 1); a scalar state cannot reduce");
    es::ShapePlan S{};
    es_status st = es::plan_shapes("es_scan_f32", kSeqName[body], initial, seqs, n_seqs, shape, rank, axis,
                                   state_width, seq_widths, out, &S);
    if (st != ES_OK) return st;
    P->O = S.O;
    P->T = S.T;
    P->J = S.J;
    P->W = S.W;
    P->n_out = S.n_out;
    P->n_init = S.n_init;
    for (int k = 0; k < 2; ++k) {
        P->sw[k] = S.sw[k];
        P->n_seq[k] = S.n_seq[k];
    }
    if (S.empty) {      // no lanes: nothing to read or write
        P->path = ES_PATH_EMPTY;
        return ES_OK;
    }
    const void* ptrs[4] = {initial, seqs[0], seqs[1], out};
    const bool vec_ok = es::vec_tma_ok(body, S.O, S.T, S.J, S.W, P->sw, ptrs);
    const bool time_ok = es::time_tma_ok(body, S.O, S.T, S.J, S.W, P->sw, ptrs);
    const bool lane_ok = es::lane_tma_ok(body, S.O, S.T, S.J, S.W, P->sw, ptrs);
    if (forced == ES_PATH_AUTO) {
        P->path = vec_ok ? ES_PATH_VEC_TMA : time_ok ? ES_PATH_TIME_TMA : lane_ok ? ES_PATH_LANE_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    const bool ok = forced == ES_PATH_GENERIC || (forced == ES_PATH_VEC_TMA && vec_ok) ||
                    (forced == ES_PATH_TIME_TMA && time_ok) || (forced == ES_PATH_LANE_TMA && lane_ok);
    if (!ok) return fail(ES_E_UNSUPPORTED, "es_scan_f32: the forced kernel path %d cannot serve this call", forced);
    P->path = forced;
    return ES_OK;
}

// Backward call: the forward plan for the shapes (the saved states have the
// output shape), then the gradient buffers: present, aligned, and disjoint
// from every input and from each other.
es_status plan_backward_impl(es_body body, const float* initial, const float* const* seqs, int n_seqs,
                             const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                             const float* states, const float* grad_out, const float* grad_initial,
                             float* const* grad_seqs, Plan* P) {
    // the forced-path choice happens below, once the gradient buffers are known
    const int forced = g_path_override.load();
    es_status st = plan_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, states,
                             ES_PATH_AUTO, P);
    if (st != ES_OK) return st;
    if (P->path == ES_PATH_EMPTY) return ES_OK;
    if (grad_seqs == nullptr || grad_out == nullptr || grad_initial == nullptr || grad_seqs[0] == nullptr ||
        grad_seqs[1] == nullptr)
        return fail(ES_E_ARG, "es_scan_backward_f32: null gradient pointer");
    const void* bufs[7] = {initial, seqs[0], seqs[1], states, grad_out, grad_initial, grad_seqs[0]};
    const void* g1 = grad_seqs[1];
    const int64_t n[8] = {P->n_init, P->n_seq[0], P->n_seq[1], P->n_out, P->n_out, P->n_init, P->n_seq[0], P->n_seq[1]};
    const void* all[8] = {bufs[0], bufs[1], bufs[2], bufs[3], bufs[4], bufs[5], bufs[6], g1};
    const char* nm[8] = {"initial", "x", kSeqName[body][1], "states", "grad_out", "grad_initial", "grad_x",
                         body == ES_MAXPLUS ? "grad_c" : "grad_a"};
    for (int k = 0; k < 8; ++k)
        if (reinterpret_cast<uintptr_t>(all[k]) % 4 != 0)
            return fail(ES_E_ARG, "es_scan_backward_f32: `%s` is not 4-byte aligned", nm[k]);
    // outputs (k >= 5) may overlap nothing else
    for (int k = 5; k < 8; ++k) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(all[k]), hi = lo + static_cast<uintptr_t>(n[k]) * 4;
        for (int q = 0; q < 8; ++q) {
            if (q == k) continue;
            const uintptr_t l2 = reinterpret_cast<uintptr_t>(all[q]), h2 = l2 + static_cast<uintptr_t>(n[q]) * 4;
            if (lo < h2 && l2 < hi) return fail(ES_E_ARG, "es_scan_backward_f32: `%s` overlaps `%s`", nm[k], nm[q]);
        }
    }
    const void* ptrs[4] = {initial, seqs[0], seqs[1], states};
    bool grads_aligned = true;
    for (int k = 4; k < 8; ++k)
        if (reinterpret_cast<uintptr_t>(all[k]) % 16 != 0) grads_aligned = false;
    const bool lane_ok = grads_aligned && es::lane_tma_ok(body, P->O, P->T, P->J, P->W, P->sw, ptrs);
    const bool vec_ok = grads_aligned && es::vec_tma_ok(body, P->O, P->T, P->J, P->W, P->sw, ptrs);
    // the time-innermost backward reads 36-trip state boxes: at least two tiles of trips
    const bool time_ok = grads_aligned && P->T >= 64 && es::time_tma_ok(body, P->O, P->T, P->J, P->W, P->sw, ptrs);
    if (forced == ES_PATH_AUTO) {
        P->path = vec_ok ? ES_PATH_VEC_TMA : time_ok ? ES_PATH_TIME_TMA : lane_ok ? ES_PATH_LANE_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    if (forced == ES_PATH_GENERIC || (forced == ES_PATH_LANE_TMA && lane_ok) || (forced == ES_PATH_VEC_TMA && vec_ok) ||
        (forced == ES_PATH_TIME_TMA && time_ok)) {
        P->path = forced;
        return ES_OK;
    }
    return fail(ES_E_UNSUPPORTED, "es_scan_backward_f32: the forced kernel path %d cannot serve this call", forced);
}

es_status device_state(int* dev_out, DeviceState** st_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ES_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(ES_E_UNSUPPORTED, "device ordinal %d too large", dev);
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, [&]() {
        void* p = nullptr;
        st.err = cudaGetSymbolAddress(&p, g_es_device_status);
        if (st.err == cudaSuccess) st.status = static_cast<unsigned int*>(p);
        if (st.err == cudaSuccess) st.err = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    });
    if (st.err != cudaSuccess) return fail(ES_E_CUDA, "device set-up: %s", cudaGetErrorString(st.err));
    *dev_out = dev;
    *st_out = &st;
    return ES_OK;
}

es_status encoder(es::EncodeTiledFn* fn) {
    std::call_once(g_encode_once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<es::EncodeTiledFn>(p);
    });
    if (g_encode == nullptr) return fail(ES_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    *fn = g_encode;
    return ES_OK;
}

}  // namespace

namespace es {

es_status api_fail(es_status st, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_error = buf;
    return st;
}

es_status plan_shapes(const char* fn, const char* const* names, const float* initial, const float* const* seqs,
                      int n_seqs, const int64_t* shape, int rank, int axis, int state_width,
                      const int64_t* seq_widths, const float* out, ShapePlan* P, bool zero_initial) {
    if (shape == nullptr || seqs == nullptr) return fail(ES_E_ARG, "%s: null shape or sequence list", fn);
    if (n_seqs < 1 || n_seqs > ES_MAX_SEQS)
        return fail(ES_E_UNSUPPORTED, "%s: %d sequences; 1..%d are supported", fn, n_seqs, ES_MAX_SEQS);
    if (rank < 1 || rank > ES_MAX_RANK)
        return fail(ES_E_UNSUPPORTED, "%s: rank %d outside 1..%d", fn, rank, ES_MAX_RANK);
    for (int d = 0; d < rank; ++d)
        if (shape[d] < 0)
            return fail(ES_E_DIM_001, "E-DIM-001 %s: negative dimension in %s", fn, shape_str(shape, rank).c_str());
    const std::string xs = shape_str(shape, rank);
    if (axis < -rank || axis >= rank)
        return fail(ES_E_DIM_001, "E-DIM-001 %s: axis %d out of range for `%s` %s f32", fn, axis, names[0],
                    xs.c_str());
    const int ax = axis < 0 ? axis + rank : axis;
    if (shape[ax] < 1)
        return fail(ES_E_DIM_001, "E-DIM-001 %s: sequence axis %d of `%s` %s f32 has length %lld; it must be "
                    "at least one", fn, ax, names[0], xs.c_str(), static_cast<long long>(shape[ax]));
    int64_t W = 1;
    if (state_width != 0) {
        if (rank < 2 || ax == rank - 1)
            return fail(ES_E_DIM_001, "E-DIM-001 %s: the state axis is the last axis of `%s` %s f32 and "
                        "cannot also be the sequence axis %d", fn, names[0], xs.c_str(), ax);
        if (state_width < 1 || state_width > ES_MAX_STATE || shape[rank - 1] != state_width)
            return fail(ES_E_DIM_001, "E-DIM-001 %s: state width %d does not fit the last axis of `%s` %s "
                        "f32 (1..%d values)", fn, state_width, names[0], xs.c_str(), ES_MAX_STATE);
        W = state_width;
    }
    int64_t O = 1, after = 1;
    for (int d = 0; d < ax; ++d)
        if (!mul_ok(O, shape[d], &O)) return fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    for (int d = ax + 1; d < rank; ++d)
        if (!mul_ok(after, shape[d], &after)) return fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    const int64_t T = shape[ax];
    P->O = O;
    P->T = T;
    P->W = W;
    P->J = after / W;
    P->n_seqs = n_seqs;
    for (int k = 0; k < n_seqs; ++k) {
        int64_t w = W;
        if (seq_widths != nullptr) {
            w = seq_widths[k];
            const bool fits = state_width != 0 ? (w == 1 || w == W) : (w == shape[rank - 1]);
            if (!fits)
                return fail(ES_E_DIM_001, "E-DIM-001 %s: `%s` %s f32 does not fit `%s` %s f32%s", fn, names[k],
                            shape_str(shape, rank, 1, w).c_str(), names[0], xs.c_str(),
                            state_width != 0 ? " (its last width must be 1 or the state width)" : "");
        }
        P->sw[k] = state_width != 0 ? w : 1;
    }
    int64_t rows, tmp;
    if (!mul_ok(O, T, &rows) || !mul_ok(rows, after, &P->n_out) || !mul_ok(O, after, &P->n_init))
        return fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    for (int k = 0; k < n_seqs; ++k)
        if (!mul_ok(rows, P->J, &tmp) || !mul_ok(tmp, P->sw[k], &P->n_seq[k]))
            return fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    if (P->n_out > (int64_t(1) << 60)) return fail(ES_E_UNSUPPORTED, "%s: too many elements", fn);
    P->empty = O * P->J == 0;
    if (P->empty) return ES_OK;

    if ((initial == nullptr) != zero_initial || out == nullptr) return fail(ES_E_ARG, "%s: null data pointer", fn);
    for (int k = 0; k < n_seqs; ++k)
        if (seqs[k] == nullptr) return fail(ES_E_ARG, "%s: null data pointer", fn);
    if (reinterpret_cast<uintptr_t>(initial) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return fail(ES_E_ARG, "%s: `initial` or `out` is not 4-byte aligned", fn);
    for (int k = 0; k < n_seqs; ++k)
        if (reinterpret_cast<uintptr_t>(seqs[k]) % 4 != 0)
            return fail(ES_E_ARG, "%s: `%s` is not 4-byte aligned", fn, names[k]);
    // the result is a new value: `out` may not overlap any input
    const uintptr_t olo = reinterpret_cast<uintptr_t>(out), ohi = olo + static_cast<uintptr_t>(P->n_out) * 4;
    for (int k = zero_initial ? 0 : -1; k < n_seqs; ++k) {
        const void* p = k < 0 ? static_cast<const void*>(initial) : static_cast<const void*>(seqs[k]);
        const int64_t n = k < 0 ? P->n_init : P->n_seq[k];
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p), hi = lo + static_cast<uintptr_t>(n) * 4;
        if (lo < ohi && olo < hi) return fail(ES_E_ARG, "%s: `out` overlaps `%s`", fn, k < 0 ? "initial" : names[k]);
    }
    return ES_OK;
}

es_status api_device(int* dev, DeviceState** st) { return device_state(dev, st); }

es_status api_encoder(EncodeTiledFn* fn) { return encoder(fn); }

void count_launch(int kernels) { g_launches.fetch_add(static_cast<uint64_t>(kernels)); }

uint64_t api_wait_ns() { return g_wait_ns.load(); }

int64_t api_drop_tile() { return g_drop_tile.load(); }

int api_path_override() { return g_path_override.load(); }

}  // namespace es

extern "C" {

es_status es_plan_f32(es_body body, const float* initial, const float* const* seqs, int n_seqs,
                      const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                      int reverse, const float* out, es_plan_info* info) {
    Plan P{};
    es_status st = plan_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, out,
                             g_path_override.load(), &P);
    if (st != ES_OK) return st;
    if (info != nullptr) {
        std::memset(info, 0, sizeof(*info));
        info->O = P.O;
        info->T = P.T;
        info->J = P.J;
        info->W = P.W;
        info->seq_width[0] = P.sw[0];
        info->seq_width[1] = P.sw[1];
        info->elements = P.n_out;
        info->path = P.path;
        info->reverse = reverse ? 1 : 0;
    }
    return ES_OK;
}

es_status es_scan_f32(es_body body, const float* initial, const float* const* seqs, int n_seqs,
                      const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                      int reverse, float* out, es_stream_t stream) {
    Plan P{};
    es_status st = plan_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, out,
                             g_path_override.load(), &P);
    if (st != ES_OK) return st;
    if (P.path == ES_PATH_EMPTY) return ES_OK;

    int dev = 0;
    DeviceState* ds = nullptr;
    if ((st = device_state(&dev, &ds)) != ES_OK) return st;

    es::Launch L{};
    L.body = static_cast<int>(body);
    L.init = initial;
    L.x = seqs[0];
    L.a = seqs[1];
    L.out = out;
    L.O = P.O;
    L.T = P.T;
    L.J = P.J;
    L.W = P.W;
    L.sw[0] = P.sw[0];
    L.sw[1] = P.sw[1];
    L.reverse = reverse ? 1 : 0;
    L.status = ds->status;
    L.wait_ns = g_wait_ns.load();
    L.drop_tile = g_drop_tile.load();
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.num_sms = ds->num_sms;
    L.device = dev;

    const char* msg = nullptr;
    cudaError_t e;
    if (P.path == ES_PATH_GENERIC) {
        e = es::launch_generic(L);
    } else {
        if ((st = encoder(&L.encode)) != ES_OK) return st;
        if (P.path == ES_PATH_LANE_TMA) e = es::launch_lane_tma(L, &msg);
        else if (P.path == ES_PATH_TIME_TMA) e = es::launch_time_tma(L, &msg);
        else e = es::launch_vec_tma(L, &msg);
    }
    if (e != cudaSuccess) {
        if (msg != nullptr) return fail(ES_E_CUDA, "es_scan_f32: %s", msg);
        return fail(ES_E_CUDA, "es_scan_f32: kernel launch: %s", cudaGetErrorString(e));
    }
    g_launches.fetch_add(1);
    return ES_OK;
}

es_status es_plan_backward_f32(es_body body, const float* initial, const float* const* seqs, int n_seqs,
                               const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                               int reverse, const float* states, const float* grad_out, const float* grad_initial,
                               float* const* grad_seqs, es_plan_info* info) {
    Plan P{};
    es_status st = plan_backward_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths,
                                      states, grad_out, grad_initial, grad_seqs, &P);
    if (st != ES_OK) return st;
    if (info != nullptr) {
        std::memset(info, 0, sizeof(*info));
        info->O = P.O;
        info->T = P.T;
        info->J = P.J;
        info->W = P.W;
        info->seq_width[0] = P.sw[0];
        info->seq_width[1] = P.sw[1];
        info->elements = P.n_out;
        info->path = P.path;
        info->reverse = reverse ? 1 : 0;
    }
    return ES_OK;
}

es_status es_scan_backward_f32(es_body body, const float* initial, const float* const* seqs, int n_seqs,
                               const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                               int reverse, const float* states, const float* grad_out, float* grad_initial,
                               float* const* grad_seqs, es_stream_t stream) {
    Plan P{};
    es_status st = plan_backward_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths,
                                      states, grad_out, grad_initial, grad_seqs, &P);
    if (st != ES_OK) return st;
    if (P.path == ES_PATH_EMPTY) return ES_OK;
    int dev = 0;
    DeviceState* ds = nullptr;
    if ((st = device_state(&dev, &ds)) != ES_OK) return st;
    es::BackwardLaunch B{};
    es::Launch& L = B.fwd;
    L.body = static_cast<int>(body);
    L.init = initial;
    L.x = seqs[0];
    L.a = seqs[1];
    L.out = nullptr;
    L.O = P.O;
    L.T = P.T;
    L.J = P.J;
    L.W = P.W;
    L.sw[0] = P.sw[0];
    L.sw[1] = P.sw[1];
    L.reverse = reverse ? 1 : 0;
    L.status = ds->status;
    L.wait_ns = g_wait_ns.load();
    L.drop_tile = g_drop_tile.load();
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.num_sms = ds->num_sms;
    L.device = dev;
    B.states = states;
    B.gout = grad_out;
    B.ginit = grad_initial;
    B.gx = grad_seqs[0];
    B.ga = grad_seqs[1];
    const char* msg = nullptr;
    cudaError_t e;
    if (P.path == ES_PATH_GENERIC) {
        e = es::launch_generic_bwd(B);
    } else {
        if ((st = encoder(&L.encode)) != ES_OK) return st;
        if (P.path == ES_PATH_VEC_TMA) e = es::launch_vec_tma_bwd(B, &msg);
        else if (P.path == ES_PATH_TIME_TMA) e = es::launch_time_tma_bwd(B, &msg);
        else e = es::launch_lane_tma_bwd(B, &msg);
    }
    if (e != cudaSuccess) {
        if (msg != nullptr) return fail(ES_E_CUDA, "es_scan_backward_f32: %s", msg);
        return fail(ES_E_CUDA, "es_scan_backward_f32: kernel launch: %s", cudaGetErrorString(e));
    }
    g_launches.fetch_add(1);
    return ES_OK;
}

es_status es_device_status(es_stream_t stream) {
    int dev = 0;
    DeviceState* ds = nullptr;
    es_status st = device_state(&dev, &ds);
    if (st != ES_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(ES_E_CUDA, "es_device_status: %s", cudaGetErrorString(e));
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_es_device_status, sizeof(word));
    if (e == cudaSuccess && word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_es_device_status, &zero, sizeof(zero));
    }
    if (e != cudaSuccess) return fail(ES_E_CUDA, "es_device_status: %s", cudaGetErrorString(e));
    if (word & ES_DEVICE_TIMEOUT)
        return fail(ES_E_TIMEOUT, "es_device_status: a kernel gave up a bounded wait; its output is incomplete");
    return ES_OK;
}

const char* es_last_error(void) { return t_error.c_str(); }

const char* es_status_string(es_status status) {
    switch (status) {
        case ES_OK: return "ES_OK";
        case ES_E_DIM_001: return "ES_E_DIM_001";
        case ES_E_DIM_002: return "ES_E_DIM_002";
        case ES_E_ARG: return "ES_E_ARG";
        case ES_E_UNSUPPORTED: return "ES_E_UNSUPPORTED";
        case ES_E_CUDA: return "ES_E_CUDA";
        case ES_E_TIMEOUT: return "ES_E_TIMEOUT";
        case ES_E_BODY: return "ES_E_BODY";
    }
    return "ES_UNKNOWN_STATUS";
}

uint64_t es_launch_count(void) { return g_launches.load(); }

es_status es_set_path_override(int path) {
    if (path != ES_PATH_AUTO && path != ES_PATH_GENERIC && path != ES_PATH_LANE_TMA && path != ES_PATH_TIME_TMA &&
        path != ES_PATH_VEC_TMA && path != ES_PATH_MAT_TMA && path != ES_PATH_MAT_CHUNKED &&
        path != ES_PATH_MAT_CHUNKED_TMA)
        return fail(ES_E_ARG, "es_set_path_override: unknown path %d", path);
    g_path_override.store(path);
    return ES_OK;
}

es_status es_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return fail(ES_E_ARG, "es_set_wait_limit_ns: the limit must be positive");
    g_wait_ns.store(ns);
    return ES_OK;
}

es_status es_set_drop_tile(int64_t k) {
    g_drop_tile.store(k < 0 ? -1 : k);
    return ES_OK;
}

}  // extern "C"
