// es_matrix_api.cu -- the matrix-scan and linear-scan entry points of the C
// ABI (es.h): shape checks, broadcasting of the leading dims, kernel choice.
//
// Contract ("Tensor operations": the `matrix-scan` row and section): a is
// lead_a + [n, n] and b lead_b + [n, m], n <= 16; lead_a and lead_b
// broadcast NumPy-style (right-aligned, each dim equal or 1) to one leading
// shape, among whose dims `axis` counts (negative from the end, so -1 is the
// one before the matrices); the result is that shape + [n, m].  linear-scan
// takes a and b broadcast to one shape, numbers included: the same scan over
// one-by-one matrices.  Shape errors are E-DIM-001.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>

#include "es.h"
#include "es_internal.h"
#include "es_matrix.h"

// Scratch the library owns for es_matrix_scan_static_f32: module scope, so no
// call allocates device memory.  In host code this name stands for the array
// but is no device address; the address comes from cudaGetSymbolAddress, once
// per device, with that device current.
static __device__ __align__(256) unsigned char g_es_static_scratch[ES_STATIC_SCRATCH_BYTES];

// Tuning override: trip windows of a matrix-scan gradient on the TMA path (1:
// one cotangent launch, then one da launch).
#ifndef ES_MAT_BWD_WINDOWS
#define ES_MAT_BWD_WINDOWS 8
#endif

namespace es {
namespace {

// the static scratch of one device: its address, fetched once, and the event
// that orders successive uses
struct StaticScratch {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void* ptr = nullptr;
    cudaEvent_t released = nullptr;
    bool used = false;
    std::mutex mu;
};
constexpr int kScratchDevices = 64;
StaticScratch g_scratch[kScratchDevices];

std::string dims_str(const int64_t* d, int r) {
    std::string s = "[";
    for (int i = 0; i < r; ++i) {
        if (i) s += ", ";
        s += std::to_string(d[i]);
    }
    return s + "]";
}

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

struct MatPlan {
    MatLaunch L;
    int64_t lead[ES_MAX_RANK];
    int lead_rank;
    int ax;
    int64_t n_out, n_a, n_b;     // element counts
    bool dense;                  // a and b both have the full leading shape
    bool empty;
    int path;
};

// `linear`: a and b have no matrix dims (n = m = 1)
es_status plan_matrix(const char* fn, const float* a, const int64_t* a_shape, int a_rank, const float* b,
                      const int64_t* b_shape, int b_rank, int axis, int reverse, int projective, const float* out,
                      bool linear, MatPlan* P) {
    if ((a_shape == nullptr && a_rank > 0) || (b_shape == nullptr && b_rank > 0))
        return api_fail(ES_E_ARG, "%s: null shape", fn);
    const int mat = linear ? 0 : 2;
    if (a_rank < mat || b_rank < mat || a_rank - mat > ES_MAX_RANK || b_rank - mat > ES_MAX_RANK)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: a %s and b %s: ranks outside %d..%d", fn,
                        dims_str(a_shape, a_rank).c_str(), dims_str(b_shape, b_rank).c_str(), mat,
                        mat + ES_MAX_RANK);
    for (int d = 0; d < a_rank; ++d)
        if (a_shape[d] < 0) return api_fail(ES_E_DIM_001, "E-DIM-001 %s: negative dimension in a", fn);
    for (int d = 0; d < b_rank; ++d)
        if (b_shape[d] < 0) return api_fail(ES_E_DIM_001, "E-DIM-001 %s: negative dimension in b", fn);
    int n = 1, m = 1;
    if (!linear) {
        const int64_t na = a_shape[a_rank - 1];
        if (a_shape[a_rank - 2] != na || b_shape[b_rank - 2] != na)
            return api_fail(ES_E_DIM_001, "E-DIM-001 %s: a %s f32 must be [.., n, n] and b %s f32 [.., n, m]", fn,
                            dims_str(a_shape, a_rank).c_str(), dims_str(b_shape, b_rank).c_str());
        if (na < 1 || na > 16)
            return api_fail(ES_E_DIM_001, "E-DIM-001 %s: n = %lld; matrix-scan takes n from 1 to 16", fn,
                            static_cast<long long>(na));
        if (b_shape[b_rank - 1] < 1 || b_shape[b_rank - 1] > (int64_t(1) << 20))
            return api_fail(ES_E_DIM_001, "E-DIM-001 %s: m = %lld", fn, static_cast<long long>(b_shape[b_rank - 1]));
        n = static_cast<int>(na);
        m = static_cast<int>(b_shape[b_rank - 1]);
    }
    // NumPy broadcast of the leading shapes
    const int ra = a_rank - mat, rb = b_rank - mat;
    const int r = ra > rb ? ra : rb;
    if (r < 1) return api_fail(ES_E_DIM_001, "E-DIM-001 %s: no leading axis to scan along", fn);
    int64_t la[ES_MAX_RANK], lb[ES_MAX_RANK];
    for (int d = 0; d < r; ++d) {
        la[d] = d < r - ra ? 1 : a_shape[d - (r - ra)];
        lb[d] = d < r - rb ? 1 : b_shape[d - (r - rb)];
        if (la[d] != lb[d] && la[d] != 1 && lb[d] != 1)
            return api_fail(ES_E_DIM_001, "E-DIM-001 %s: the leading dims of a %s and b %s do not broadcast", fn,
                            dims_str(a_shape, a_rank).c_str(), dims_str(b_shape, b_rank).c_str());
        P->lead[d] = la[d] == 1 ? lb[d] : la[d];
    }
    P->lead_rank = r;
    if (axis < -r || axis >= r)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: axis %d out of range for the leading shape %s", fn, axis,
                        dims_str(P->lead, r).c_str());
    const int ax = axis < 0 ? axis + r : axis;
    P->ax = ax;
    const int64_t T = P->lead[ax];
    if (T < 1) return api_fail(ES_E_DIM_001, "E-DIM-001 %s: the scanned axis has length %lld", fn,
                               static_cast<long long>(T));

    MatLaunch& L = P->L;
    L = MatLaunch{};
    L.a = a;
    L.b = b;
    L.out = const_cast<float*>(out);
    L.n = n;
    L.m = m;
    L.projective = projective != 0;
    L.reverse = reverse ? 1 : 0;
    int C = m + (L.projective ? n : 0);
    L.gp = 1;
    while (L.gp < C && L.gp < 64) L.gp *= 2;
    if (L.projective && C > 32)
        return api_fail(ES_E_UNSUPPORTED, "%s: a projective scan carries n + m = %d columns; at most 32", fn, C);
    // strides in matrices: dense row-major over each operand's own leading shape
    int64_t sa_all[ES_MAX_RANK], sb_all[ES_MAX_RANK], so_all[ES_MAX_RANK];
    int64_t ca = 1, cb = 1, co = 1;
    for (int d = r - 1; d >= 0; --d) {
        sa_all[d] = la[d] == 1 ? 0 : ca;
        sb_all[d] = lb[d] == 1 ? 0 : cb;
        so_all[d] = co;
        if (!mul_ok(ca, la[d], &ca) || !mul_ok(cb, lb[d], &cb) || !mul_ok(co, P->lead[d], &co))
            return api_fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    }
    MatGeom& g = L.g;
    g.T = T;
    g.nd = 0;
    g.lanes = 1;
    for (int d = 0; d < r; ++d) {
        if (d == ax) continue;
        g.dim[g.nd] = P->lead[d];
        g.sa[g.nd] = sa_all[d];
        g.sb[g.nd] = sb_all[d];
        g.so[g.nd] = so_all[d];
        ++g.nd;
        if (!mul_ok(g.lanes, P->lead[d], &g.lanes)) return api_fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    }
    g.ta = sa_all[ax];
    g.tb = sb_all[ax];
    g.to = so_all[ax];
    L.O = 1;
    for (int d = 0; d < ax; ++d) L.O *= P->lead[d];
    L.T = T;
    L.J = 1;
    for (int d = ax + 1; d < r; ++d) L.J *= P->lead[d];
    if (!mul_ok(co, static_cast<int64_t>(n) * m, &P->n_out) || !mul_ok(ca, static_cast<int64_t>(n) * n, &P->n_a) ||
        !mul_ok(cb, static_cast<int64_t>(n) * m, &P->n_b) || P->n_out > (int64_t(1) << 60))
        return api_fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    P->dense = true;
    for (int d = 0; d < r; ++d)
        if (la[d] != P->lead[d] || lb[d] != P->lead[d]) P->dense = false;
    P->empty = g.lanes == 0;
    if (P->empty) {
        P->path = ES_PATH_EMPTY;
        return ES_OK;
    }
    if (a == nullptr || b == nullptr || out == nullptr) return api_fail(ES_E_ARG, "%s: null data pointer", fn);
    if (reinterpret_cast<uintptr_t>(a) % 4 || reinterpret_cast<uintptr_t>(b) % 4 ||
        reinterpret_cast<uintptr_t>(out) % 4)
        return api_fail(ES_E_ARG, "%s: a data pointer is not 4-byte aligned", fn);
    // the result is a new value: `out` may not overlap a or b
    const uintptr_t olo = reinterpret_cast<uintptr_t>(out), ohi = olo + static_cast<uintptr_t>(P->n_out) * 4;
    const uintptr_t alo = reinterpret_cast<uintptr_t>(a), ahi = alo + static_cast<uintptr_t>(P->n_a) * 4;
    const uintptr_t blo = reinterpret_cast<uintptr_t>(b), bhi = blo + static_cast<uintptr_t>(P->n_b) * 4;
    if ((alo < ohi && olo < ahi) || (blo < ohi && olo < bhi))
        return api_fail(ES_E_ARG, "%s: `out` overlaps an input", fn);
    return ES_OK;
}

es_status choose_matrix_path(const char* fn, MatPlan* P) {
    if (P->empty) return ES_OK;
    const MatLaunch& L = P->L;
    const bool tma = mat_tma_ok(L.n, L.m, L.gp, L.projective, L.O, L.T, L.J, P->dense, L.a, L.b) &&
                     reinterpret_cast<uintptr_t>(L.out) % 16 == 0;
    const int forced = api_path_override();
    if (forced == ES_PATH_AUTO) {
        P->path = tma ? ES_PATH_MAT_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    if (forced == ES_PATH_GENERIC || (forced == ES_PATH_MAT_TMA && tma)) {
        P->path = forced;
        return ES_OK;
    }
    return api_fail(ES_E_UNSUPPORTED, "%s: the forced kernel path %d cannot serve this call", fn, forced);
}

// the chunked scan: few lanes (a lane-by-lane run would leave the GPU
// idle), many trips, no projective normalisation
bool chunked_applies(const MatPlan& P) {
    const MatLaunch& L = P.L;
    return !P.empty && !L.projective && L.g.lanes * L.m < 8192 && L.T >= 256;
}

size_t chunked_workspace(const MatPlan& P, int64_t* chunks, int64_t* chunk) {
    mat_chunk_shape(P.L.n, P.L.m, P.dense, P.L.g.lanes, P.L.T, chunks, chunk);
    return mat_chunk_workspace_bytes(P.L.n, P.L.m, P.L.g.lanes, *chunks);
}

void fill_matrix_info(const MatPlan& P, es_plan_info* info) {
    if (info == nullptr) return;
    std::memset(info, 0, sizeof(*info));
    info->O = P.L.O;
    info->T = P.L.T;
    info->J = P.L.J;
    info->W = static_cast<int64_t>(P.L.n) * P.L.m;
    info->seq_width[0] = static_cast<int64_t>(P.L.n) * P.L.n;
    info->seq_width[1] = static_cast<int64_t>(P.L.n) * P.L.m;
    info->elements = P.n_out;
    info->path = P.path;
    info->reverse = P.L.reverse;
}

es_status launch_matrix(const char* fn, MatPlan* P, cudaStream_t stream) {
    int dev = 0;
    DeviceState* ds = nullptr;
    es_status st = api_device(&dev, &ds);
    if (st != ES_OK) return st;
    MatLaunch& L = P->L;
    L.status = ds->status;
    L.wait_ns = api_wait_ns();
    L.drop_tile = api_drop_tile();
    L.stream = stream;
    L.num_sms = ds->num_sms;
    const char* msg = nullptr;
    cudaError_t e;
    if (P->path == ES_PATH_MAT_TMA) {
        if ((st = api_encoder(&L.encode)) != ES_OK) return st;
        e = launch_mat_tma(L, &msg);
    } else {
        e = launch_mat_generic(L);
    }
    if (e != cudaSuccess)
        return api_fail(ES_E_CUDA, "%s: %s", fn, msg != nullptr ? msg : cudaGetErrorString(e));
    count_launch();
    return ES_OK;
}

// linear-scan of operands that share one shape runs as the element scan of
// the body (+ (* a h) b) from a zero state: per trip one product and one
// sum, rounded, in that order -- the one-by-one matrix-scan's arithmetic --
// on the element-scan skeletons
es_body_t linear_body() {
    static es_body_t body = nullptr;
    static std::once_flag once;
    std::call_once(once, []() { es_body_create("(lambda (h a b) (+ (* a h) b))", &body); });
    return body;
}

bool same_shape(const int64_t* a_shape, int a_rank, const int64_t* b_shape, int b_rank) {
    if (a_rank != b_rank) return false;
    for (int d = 0; d < a_rank; ++d)
        if (a_shape[d] != b_shape[d]) return false;
    return true;
}

bool overlaps(const void* p, int64_t n, const void* q, int64_t k) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + static_cast<uintptr_t>(k) * 4 && b < a + static_cast<uintptr_t>(n) * 4;
}

// ---------------------------------------------------------------------------
// gradients ("matrix-scan": "its gradient is the same scan run backwards on
// a's transposes"; a projective scan "has no gradient")
//
// The cotangent lam[t] = a[t+1]^T lam[t+1] + g[t] (a reverse scan: a[t-1],
// lam[t-1]) is the matrix-scan kernel run in the opposite direction on the
// state gradients with the transposed coefficient one trip off (the zero
// matrix past the end); it is db.  A second kernel forms
// da[t] = lam[t] h[t-1]^T from it and the saved states.

struct MatBwdPlan {
    MatPlan P;           // the cotangent scan: b = grad_out, out = grad_b
    const float* states;
    float* grad_a;
};

es_status plan_matrix_backward(const char* fn, const float* a, const int64_t* a_shape, int a_rank, const float* b,
                               const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                               const float* states, const float* grad_out, const float* grad_a,
                               const float* grad_b, MatBwdPlan* Q, bool chunk_forcible = false) {
    if (projective) return api_fail(ES_E_ARG, "%s: a projective matrix-scan has no gradient", fn);
    MatPlan& P = Q->P;
    es_status st = plan_matrix(fn, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, 0, states, false, &P);
    if (st != ES_OK) return st;
    if (!P.dense)
        return api_fail(ES_E_UNSUPPORTED,
                        "%s: a %s and b %s: the gradient wants one leading shape (broadcast the operands first)", fn,
                        dims_str(a_shape, a_rank).c_str(), dims_str(b_shape, b_rank).c_str());
    Q->states = states;
    Q->grad_a = const_cast<float*>(grad_a);
    if (P.empty) return ES_OK;
    if (grad_out == nullptr || grad_a == nullptr || grad_b == nullptr)
        return api_fail(ES_E_ARG, "%s: null gradient pointer", fn);
    const void* buf[6] = {a, b, states, grad_out, grad_a, grad_b};
    const int64_t cnt[6] = {P.n_a, P.n_b, P.n_out, P.n_out, P.n_a, P.n_b};
    const char* nm[6] = {"a", "b", "states", "grad_out", "grad_a", "grad_b"};
    for (int k = 3; k < 6; ++k)
        if (reinterpret_cast<uintptr_t>(buf[k]) % 4 != 0)
            return api_fail(ES_E_ARG, "%s: `%s` is not 4-byte aligned", fn, nm[k]);
    for (int k = 4; k < 6; ++k)
        for (int q = 0; q < 6; ++q)
            if (q != k && overlaps(buf[k], cnt[k], buf[q], cnt[q]))
                return api_fail(ES_E_ARG, "%s: `%s` overlaps `%s`", fn, nm[k], nm[q]);
    // the cotangent scan
    MatLaunch& L = P.L;
    L.b = grad_out;
    L.out = const_cast<float*>(grad_b);
    L.trans = true;
    L.a_shift = reverse ? -1 : 1;       // the trip after t in the forward's order
    L.reverse = reverse ? 0 : 1;        // the opposite direction
    const bool tma = mat_tma_ok(L.n, L.m, L.gp, false, L.O, L.T, L.J, true, L.a, L.b) &&
                     reinterpret_cast<uintptr_t>(L.out) % 16 == 0;
    const int forced = api_path_override();
    // a forced chunked path is decided by the workspace entry (its sequential
    // choice is then the automatic one)
    if (forced == ES_PATH_AUTO || (chunk_forcible && forced == ES_PATH_MAT_CHUNKED_TMA)) {
        P.path = tma ? ES_PATH_MAT_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    if (forced == ES_PATH_GENERIC || (forced == ES_PATH_MAT_TMA && tma)) {
        P.path = forced;
        return ES_OK;
    }
    return api_fail(ES_E_UNSUPPORTED, "%s: the forced kernel path %d cannot serve this call", fn, forced);
}

// es_matrix_scan_backward_ws_f32's path: the cotangent scan chunked on the TMA
// passes (the forward's chunks and workspace size: the geometry is the same)
// when the lanes are few, the operands suit it and the workspace suffices;
// else the sequential path of es_matrix_scan_backward_f32.  ws_chunked set
// for the former.
es_status plan_matrix_backward_ws(const char* fn, MatBwdPlan* Q, const float* b, const float* grad_out,
                                  const void* workspace, size_t workspace_bytes, int64_t* chunks, int64_t* chunk,
                                  bool* ws_chunked) {
    *ws_chunked = false;
    MatPlan& P = Q->P;
    if (P.empty) return ES_OK;
    const int forced = api_path_override();
    if (forced == ES_PATH_MAT_CHUNKED)
        return api_fail(ES_E_UNSUPPORTED, "%s: the direct-load chunk kernels have no gradient", fn);
    const size_t need = chunked_applies(P) ? chunked_workspace(P, chunks, chunk) : 0;
    const bool tma = need > 0 && mat_chunked_tma_ok(P.L, P.dense, *chunks, *chunk);
    if (!(tma && workspace != nullptr && workspace_bytes >= need)) {
        if (forced == ES_PATH_MAT_CHUNKED_TMA)
            return api_fail(ES_E_UNSUPPORTED,
                            "%s: the chunked gradient needs few long lanes, operands the TMA passes take and %zu "
                            "workspace bytes", fn, need);
        return ES_OK;
    }
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return api_fail(ES_E_ARG, "%s: workspace not 16-byte aligned", fn);
    const void* ops[6] = {P.L.a, b, Q->states, grad_out, Q->grad_a, P.L.out};
    const int64_t cnt[6] = {P.n_a, P.n_b, P.n_out, P.n_out, P.n_a, P.n_b};
    const uintptr_t wlo = reinterpret_cast<uintptr_t>(workspace), whi = wlo + need;
    for (int k = 0; k < 6; ++k) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(ops[k]), hi = lo + static_cast<uintptr_t>(cnt[k]) * 4;
        if (lo < whi && wlo < hi) return api_fail(ES_E_ARG, "%s: the workspace overlaps an operand", fn);
    }
    P.path = ES_PATH_MAT_CHUNKED_TMA;
    *ws_chunked = true;
    return ES_OK;
}

// The two launches of the gradient overlap in windows of trips.  The
// cotangent scan is bound by its chain and leaves bandwidth that the da
// kernel, bound by bandwidth, can use: the scan runs window by window on the
// caller's stream (each window started from the states the previous one left
// next to it), and each window's da runs on a library-owned stream as soon as
// its scan window is done, beside the next scan window.  Same operations in
// the same order as one scan then one da launch, so the same bits.
constexpr int kBwdWindows = ES_MAT_BWD_WINDOWS;
constexpr int kBwdDevices = 64;

struct BwdPipe {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    cudaStream_t side = nullptr;
    cudaEvent_t scanned[kBwdWindows > 1 ? kBwdWindows : 1] = {};
    cudaEvent_t done = nullptr;
    std::mutex mu;        // one call at a time enqueues on the side stream
};
BwdPipe g_bwd[kBwdDevices];

cudaError_t bwd_pipe_init(BwdPipe* p) {
    cudaError_t e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking);
    for (int k = 0; k < kBwdWindows && e == cudaSuccess; ++k)
        e = cudaEventCreateWithFlags(&p->scanned[k], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming);
    return e;
}

// windows for a gradient: the TMA scan with at least 128 trips a window
int bwd_windows(const MatPlan& P) {
    if (P.path != ES_PATH_MAT_TMA || kBwdWindows < 2) return 1;
    const int64_t k = P.L.T / 128;
    return static_cast<int>(k < 2 ? 1 : k > kBwdWindows ? kBwdWindows : k);
}

es_status launch_matrix_backward(const char* fn, MatBwdPlan* Q, int reverse, cudaStream_t stream) {
    const int K = bwd_windows(Q->P);
    if (K <= 1) {
        es_status st = launch_matrix(fn, &Q->P, stream);
        if (st != ES_OK) return st;
        const MatLaunch& L = Q->P.L;
        cudaError_t e = launch_mat_da(L.out, Q->states, Q->grad_a, L.n, L.O, L.T, L.J, L.m, reverse ? 1 : 0, stream);
        if (e != cudaSuccess) return api_fail(ES_E_CUDA, "%s: %s", fn, cudaGetErrorString(e));
        count_launch();
        return ES_OK;
    }
    int dev = 0;
    DeviceState* ds = nullptr;
    es_status st = api_device(&dev, &ds);
    if (st != ES_OK) return st;
    if (dev >= kBwdDevices) return api_fail(ES_E_CUDA, "%s: device %d beyond the library's table", fn, dev);
    BwdPipe* p = &g_bwd[dev];
    std::call_once(p->once, [p]() { p->err = bwd_pipe_init(p); });
    if (p->err != cudaSuccess) return api_fail(ES_E_CUDA, "%s: %s", fn, cudaGetErrorString(p->err));
    std::lock_guard<std::mutex> lock(p->mu);
    auto check = [&](cudaError_t e) -> es_status {
        return e == cudaSuccess ? ES_OK : api_fail(ES_E_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    };
    MatLaunch& L = Q->P.L;
    L.status = ds->status;
    L.wait_ns = api_wait_ns();
    L.drop_tile = api_drop_tile();
    L.stream = stream;
    L.num_sms = ds->num_sms;
    if ((st = api_encoder(&L.encode)) != ES_OK) return st;
    const int64_t T = L.T, span = (T + K - 1) / K;
    const int64_t trip_floats = L.J * L.n * L.m;      // one trip of the dense [O, T, J] view
    // the cotangent runs descending for a forward scan's gradient
    const bool desc = L.reverse != 0;
    for (int w = 0; w < K; ++w) {
        const int64_t t1 = desc ? T - w * span : std::min<int64_t>(T, (w + 1) * span);
        const int64_t t0 = desc ? std::max<int64_t>(0, t1 - span) : w * span;
        if (t1 <= t0) break;
        MatLaunch Lw = L;
        Lw.win0 = t0;
        Lw.win_len = t1 - t0;
        const int64_t tc = desc ? t1 : t0 - 1;            // the trip whose states start this window
        Lw.carry = (tc >= 0 && tc < T) ? L.out + tc * trip_floats : nullptr;
        const char* msg = nullptr;
        cudaError_t e = launch_mat_tma(Lw, &msg);
        if (e != cudaSuccess) return api_fail(ES_E_CUDA, "%s: %s", fn, msg != nullptr ? msg : cudaGetErrorString(e));
        count_launch();
        if ((st = check(cudaEventRecord(p->scanned[w], stream))) != ES_OK) return st;
        if ((st = check(cudaStreamWaitEvent(p->side, p->scanned[w], 0))) != ES_OK) return st;
        e = launch_mat_da(L.out, Q->states, Q->grad_a, L.n, L.O, T, L.J, L.m, reverse ? 1 : 0, p->side, t0, t1 - t0);
        if ((st = check(e)) != ES_OK) return st;
        count_launch();
    }
    // later work on the caller's stream waits for the last da window
    if ((st = check(cudaEventRecord(p->done, p->side))) != ES_OK) return st;
    return check(cudaStreamWaitEvent(stream, p->done, 0));
}

}  // namespace
}  // namespace es

extern "C" {

es_status es_plan_matrix_scan_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                  const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                                  const float* out, es_plan_info* info) {
    es::MatPlan P{};
    es_status st = es::plan_matrix("es_matrix_scan_f32", a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse,
                                   projective, out, false, &P);
    if (st == ES_OK) st = es::choose_matrix_path("es_matrix_scan_f32", &P);
    if (st != ES_OK) return st;
    es::fill_matrix_info(P, info);
    return ES_OK;
}

es_status es_matrix_scan_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                             const int64_t* b_shape, int b_rank, int axis, int reverse, int projective, float* out,
                             es_stream_t stream) {
    es::MatPlan P{};
    es_status st = es::plan_matrix("es_matrix_scan_f32", a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse,
                                   projective, out, false, &P);
    if (st == ES_OK) st = es::choose_matrix_path("es_matrix_scan_f32", &P);
    if (st != ES_OK || P.empty) return st;
    return es::launch_matrix("es_matrix_scan_f32", &P, reinterpret_cast<cudaStream_t>(stream));
}

es_status es_matrix_scan_workspace_f32(const int64_t* a_shape, int a_rank, const int64_t* b_shape, int b_rank,
                                       int axis, int projective, size_t* bytes) {
    if (bytes == nullptr) return es::api_fail(ES_E_ARG, "es_matrix_scan_workspace_f32: null result pointer");
    es::MatPlan P{};
    // shapes only: stand-in pointers that pass the pointer checks
    const float* pa = reinterpret_cast<const float*>(uintptr_t(1) << 44);
    const float* pb = reinterpret_cast<const float*>(uintptr_t(2) << 44);
    float* po = reinterpret_cast<float*>(uintptr_t(3) << 44);
    es_status st = es::plan_matrix("es_matrix_scan_workspace_f32", pa, a_shape, a_rank, pb, b_shape, b_rank, axis, 0,
                                   projective, po, false, &P);
    if (st != ES_OK) return st;
    int64_t chunks = 0, chunk = 0;
    *bytes = es::chunked_applies(P) ? es::chunked_workspace(P, &chunks, &chunk) : 0;
    return ES_OK;
}

}  // extern "C"

namespace es {

// the path es_matrix_scan_ws_f32 takes with this workspace: the chunked scan
// (on the TMA kernel where it takes the operands, else the direct-load chunk
// kernels, the same arithmetic) or the sequential choice of
// es_matrix_scan_f32; ws_chunked set for the former
es_status plan_matrix_ws(const char* fn, MatPlan* P, const void* workspace, size_t workspace_bytes,
                         int64_t* chunks, int64_t* chunk, bool* ws_chunked) {
    *ws_chunked = false;
    if (P->empty) return ES_OK;
    const size_t need = chunked_applies(*P) ? chunked_workspace(*P, chunks, chunk) : 0;
    const int forced = api_path_override();
    const bool want = forced == ES_PATH_AUTO || forced == ES_PATH_MAT_CHUNKED || forced == ES_PATH_MAT_CHUNKED_TMA;
    if (!(need > 0 && workspace != nullptr && workspace_bytes >= need && want)) {
        if (forced == ES_PATH_MAT_CHUNKED || forced == ES_PATH_MAT_CHUNKED_TMA)
            return api_fail(ES_E_UNSUPPORTED, "%s: the chunked path needs few long lanes and %zu workspace bytes",
                            fn, need);
        return choose_matrix_path(fn, P);
    }
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return api_fail(ES_E_ARG, "%s: workspace not 16-byte aligned", fn);
    const uintptr_t wlo = reinterpret_cast<uintptr_t>(workspace), whi = wlo + need;
    const void* ops[3] = {P->L.a, P->L.b, P->L.out};
    const int64_t cnt[3] = {P->n_a, P->n_b, P->n_out};
    for (int k = 0; k < 3; ++k) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(ops[k]), hi = lo + static_cast<uintptr_t>(cnt[k]) * 4;
        if (lo < whi && wlo < hi) return api_fail(ES_E_ARG, "%s: the workspace overlaps an operand", fn);
    }
    const bool tma = forced != ES_PATH_MAT_CHUNKED && mat_chunked_tma_ok(P->L, P->dense, *chunks, *chunk);
    if (forced == ES_PATH_MAT_CHUNKED_TMA && !tma)
        return api_fail(ES_E_UNSUPPORTED, "%s: the forced kernel path %d cannot serve this call", fn, forced);
    P->path = tma ? ES_PATH_MAT_CHUNKED_TMA : ES_PATH_MAT_CHUNKED;
    *ws_chunked = true;
    return ES_OK;
}

}  // namespace es

extern "C" {

es_status es_plan_matrix_scan_ws_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                     const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                                     const float* out, const void* workspace, size_t workspace_bytes,
                                     es_plan_info* info) {
    const char* fn = "es_matrix_scan_ws_f32";
    es::MatPlan P{};
    es_status st = es::plan_matrix(fn, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, projective,
                                   const_cast<float*>(out), false, &P);
    int64_t chunks = 0, chunk = 0;
    bool ws_chunked = false;
    if (st == ES_OK) st = es::plan_matrix_ws(fn, &P, workspace, workspace_bytes, &chunks, &chunk, &ws_chunked);
    if (st != ES_OK) return st;
    es::fill_matrix_info(P, info);
    return ES_OK;
}

es_status es_matrix_scan_ws_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                const int64_t* b_shape, int b_rank, int axis, int reverse, int projective, float* out,
                                void* workspace, size_t workspace_bytes, es_stream_t stream) {
    const char* fn = "es_matrix_scan_ws_f32";
    es::MatPlan P{};
    es_status st = es::plan_matrix(fn, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, projective, out, false,
                                   &P);
    if (st != ES_OK || P.empty) return st;
    int64_t chunks = 0, chunk = 0;
    bool ws_chunked = false;
    if ((st = es::plan_matrix_ws(fn, &P, workspace, workspace_bytes, &chunks, &chunk, &ws_chunked)) != ES_OK)
        return st;
    if (!ws_chunked) return es::launch_matrix(fn, &P, reinterpret_cast<cudaStream_t>(stream));
    int dev = 0;
    es::DeviceState* ds = nullptr;
    if ((st = es::api_device(&dev, &ds)) != ES_OK) return st;
    es::MatLaunch& L = P.L;
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.status = ds->status;
    L.wait_ns = es::api_wait_ns();
    L.drop_tile = es::api_drop_tile();
    L.num_sms = ds->num_sms;
    const char* msg = nullptr;
    cudaError_t e;
    if (P.path == ES_PATH_MAT_CHUNKED_TMA) {
        if ((st = es::api_encoder(&L.encode)) != ES_OK) return st;
        e = es::launch_mat_chunked_tma(L, static_cast<float*>(workspace), chunks, chunk, &msg);
    } else {
        e = es::launch_mat_chunked(L, static_cast<float*>(workspace), chunks, chunk);
    }
    if (e != cudaSuccess) return es::api_fail(ES_E_CUDA, "%s: %s", fn, msg != nullptr ? msg : cudaGetErrorString(e));
    es::count_launch(3);
    return ES_OK;
}

es_status es_matrix_scan_static_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                    const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                                    float* out, es_stream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return es::api_fail(ES_E_CUDA, "es_matrix_scan_static_f32: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= es::kScratchDevices)
        return es::api_fail(ES_E_UNSUPPORTED, "es_matrix_scan_static_f32: device ordinal %d too large", dev);
    es::StaticScratch& sc = es::g_scratch[dev];
    std::call_once(sc.once, [&]() {
        sc.err = cudaGetSymbolAddress(&sc.ptr, g_es_static_scratch);
        if (sc.err == cudaSuccess) sc.err = cudaEventCreateWithFlags(&sc.released, cudaEventDisableTiming);
    });
    if (sc.err != cudaSuccess)
        return es::api_fail(ES_E_CUDA, "es_matrix_scan_static_f32: scratch set-up: %s", cudaGetErrorString(sc.err));
    // the chunked scan of this call must fit the library's array
    size_t need = 0;
    es_status st = es_matrix_scan_workspace_f32(a_shape, a_rank, b_shape, b_rank, axis, projective, &need);
    if (st != ES_OK) return st;
    if (need > ES_STATIC_SCRATCH_BYTES)
        return es::api_fail(ES_E_UNSUPPORTED,
                            "es_matrix_scan_static_f32: this scan needs %zu bytes of scratch, more than the %zu "
                            "bytes (ES_STATIC_SCRATCH_BYTES) the library holds; call es_matrix_scan_ws_f32 with a "
                            "workspace of es_matrix_scan_workspace_f32 bytes instead",
                            need, static_cast<size_t>(ES_STATIC_SCRATCH_BYTES));
    std::lock_guard<std::mutex> lock(sc.mu);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the previous user of the scratch, on whatever stream, comes first
    if (sc.used && (e = cudaStreamWaitEvent(s, sc.released, 0)) != cudaSuccess)
        return es::api_fail(ES_E_CUDA, "es_matrix_scan_static_f32: %s", cudaGetErrorString(e));
    st = es_matrix_scan_ws_f32(a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, projective, out, sc.ptr,
                               ES_STATIC_SCRATCH_BYTES, stream);
    if (st != ES_OK) return st;
    if ((e = cudaEventRecord(sc.released, s)) != cudaSuccess)
        return es::api_fail(ES_E_CUDA, "es_matrix_scan_static_f32: %s", cudaGetErrorString(e));
    sc.used = true;
    return ES_OK;
}

es_status es_plan_linear_scan_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                  const int64_t* b_shape, int b_rank, int axis, int reverse, const float* out,
                                  es_plan_info* info) {
    es::MatPlan P{};
    es_status st = es::plan_matrix("es_linear_scan_f32", a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, 0,
                                   out, true, &P);
    if (st != ES_OK) return st;
    if (!P.empty && es::same_shape(a_shape, a_rank, b_shape, b_rank) && es::api_path_override() != ES_PATH_MAT_TMA) {
        const float* seqs[2] = {a, b};
        return es::plan_body_impl(es::linear_body(), nullptr, seqs, 2, a_shape, a_rank, axis, 0, nullptr, reverse,
                                  out, info, true);
    }
    if ((st = es::choose_matrix_path("es_linear_scan_f32", &P)) != ES_OK) return st;
    es::fill_matrix_info(P, info);
    return ES_OK;
}

es_status es_linear_scan_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                             const int64_t* b_shape, int b_rank, int axis, int reverse, float* out,
                             es_stream_t stream) {
    es::MatPlan P{};
    es_status st = es::plan_matrix("es_linear_scan_f32", a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, 0,
                                   out, true, &P);
    if (st != ES_OK || P.empty) return st;
    if (es::same_shape(a_shape, a_rank, b_shape, b_rank) && es::api_path_override() != ES_PATH_MAT_TMA) {
        const float* seqs[2] = {a, b};
        return es::scan_body_impl(es::linear_body(), nullptr, seqs, 2, a_shape, a_rank, axis, 0, nullptr, reverse,
                                  out, reinterpret_cast<cudaStream_t>(stream), true);
    }
    if ((st = es::choose_matrix_path("es_linear_scan_f32", &P)) != ES_OK) return st;
    return es::launch_matrix("es_linear_scan_f32", &P, reinterpret_cast<cudaStream_t>(stream));
}

es_status es_plan_matrix_scan_backward_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                           const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                                           const float* states, const float* grad_out, const float* grad_a,
                                           const float* grad_b, es_plan_info* info) {
    es::MatBwdPlan Q{};
    es_status st = es::plan_matrix_backward("es_matrix_scan_backward_f32", a, a_shape, a_rank, b, b_shape, b_rank,
                                            axis, reverse, projective, states, grad_out, grad_a, grad_b, &Q);
    if (st != ES_OK) return st;
    es::fill_matrix_info(Q.P, info);
    if (info != nullptr) info->reverse = reverse ? 1 : 0;
    return ES_OK;
}

es_status es_matrix_scan_backward_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                      const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                                      const float* states, const float* grad_out, float* grad_a, float* grad_b,
                                      es_stream_t stream) {
    const char* fn = "es_matrix_scan_backward_f32";
    es::MatBwdPlan Q{};
    es_status st = es::plan_matrix_backward(fn, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, projective,
                                            states, grad_out, grad_a, grad_b, &Q);
    if (st != ES_OK || Q.P.empty) return st;
    return es::launch_matrix_backward(fn, &Q, reverse, reinterpret_cast<cudaStream_t>(stream));
}

es_status es_plan_matrix_scan_backward_ws_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                              const int64_t* b_shape, int b_rank, int axis, int reverse,
                                              int projective, const float* states, const float* grad_out,
                                              const float* grad_a, const float* grad_b, const void* workspace,
                                              size_t workspace_bytes, es_plan_info* info) {
    const char* fn = "es_matrix_scan_backward_ws_f32";
    es::MatBwdPlan Q{};
    es_status st = es::plan_matrix_backward(fn, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, projective,
                                            states, grad_out, grad_a, grad_b, &Q, true);
    int64_t chunks = 0, chunk = 0;
    bool ws_chunked = false;
    if (st == ES_OK)
        st = es::plan_matrix_backward_ws(fn, &Q, b, grad_out, workspace, workspace_bytes, &chunks, &chunk,
                                         &ws_chunked);
    if (st != ES_OK) return st;
    es::fill_matrix_info(Q.P, info);
    if (info != nullptr) info->reverse = reverse ? 1 : 0;
    return ES_OK;
}

es_status es_matrix_scan_backward_ws_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                         const int64_t* b_shape, int b_rank, int axis, int reverse, int projective,
                                         const float* states, const float* grad_out, float* grad_a, float* grad_b,
                                         void* workspace, size_t workspace_bytes, es_stream_t stream) {
    const char* fn = "es_matrix_scan_backward_ws_f32";
    es::MatBwdPlan Q{};
    es_status st = es::plan_matrix_backward(fn, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, projective,
                                            states, grad_out, grad_a, grad_b, &Q, true);
    if (st != ES_OK || Q.P.empty) return st;
    int64_t chunks = 0, chunk = 0;
    bool ws_chunked = false;
    if ((st = es::plan_matrix_backward_ws(fn, &Q, b, grad_out, workspace, workspace_bytes, &chunks, &chunk,
                                          &ws_chunked)) != ES_OK)
        return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!ws_chunked) return es::launch_matrix_backward(fn, &Q, reverse, s);
    int dev = 0;
    es::DeviceState* ds = nullptr;
    if ((st = es::api_device(&dev, &ds)) != ES_OK) return st;
    es::MatLaunch& L = Q.P.L;
    L.stream = s;
    L.status = ds->status;
    L.wait_ns = es::api_wait_ns();
    L.drop_tile = es::api_drop_tile();
    L.num_sms = ds->num_sms;
    if ((st = es::api_encoder(&L.encode)) != ES_OK) return st;
    const char* msg = nullptr;
    // the cotangent scan, chunked (grad_b), then grad_a from it and the states
    cudaError_t e = es::launch_mat_chunked_tma(L, static_cast<float*>(workspace), chunks, chunk, &msg);
    if (e == cudaSuccess)
        e = es::launch_mat_da(L.out, Q.states, Q.grad_a, L.n, L.O, L.T, L.J, L.m, reverse ? 1 : 0, s);
    if (e != cudaSuccess) return es::api_fail(ES_E_CUDA, "%s: %s", fn, msg != nullptr ? msg : cudaGetErrorString(e));
    es::count_launch(4);
    return ES_OK;
}

// linear-scan's gradient is the element-scan backward of its body, from zero
static es_status linear_backward(bool plan_only, const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                 const int64_t* b_shape, int b_rank, int axis, int reverse, const float* states,
                                 const float* grad_out, float* grad_a, float* grad_b, es_plan_info* info,
                                 cudaStream_t stream) {
    const char* fn = "es_linear_scan_backward_f32";
    if (a_shape == nullptr || b_shape == nullptr) return es::api_fail(ES_E_ARG, "%s: null shape", fn);
    if (!es::same_shape(a_shape, a_rank, b_shape, b_rank))
        return es::api_fail(ES_E_UNSUPPORTED,
                            "%s: a %s and b %s: the gradient wants one shape (broadcast the operands first)", fn,
                            es::dims_str(a_shape, a_rank).c_str(), es::dims_str(b_shape, b_rank).c_str());
    const float* seqs[2] = {a, b};
    float* gseqs[2] = {grad_a, grad_b};
    if (plan_only)
        return es::plan_body_backward_impl(es::linear_body(), nullptr, seqs, 2, a_shape, a_rank, axis, 0, nullptr,
                                           reverse, states, grad_out, nullptr, gseqs, info, true);
    return es::scan_body_backward_impl(es::linear_body(), nullptr, seqs, 2, a_shape, a_rank, axis, 0, nullptr,
                                       reverse, states, grad_out, nullptr, gseqs, stream, true);
}

es_status es_plan_linear_scan_backward_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                           const int64_t* b_shape, int b_rank, int axis, int reverse,
                                           const float* states, const float* grad_out, const float* grad_a,
                                           const float* grad_b, es_plan_info* info) {
    return linear_backward(true, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, states, grad_out,
                           const_cast<float*>(grad_a), const_cast<float*>(grad_b), info, nullptr);
}

es_status es_linear_scan_backward_f32(const float* a, const int64_t* a_shape, int a_rank, const float* b,
                                      const int64_t* b_shape, int b_rank, int axis, int reverse, const float* states,
                                      const float* grad_out, float* grad_a, float* grad_b, es_stream_t stream) {
    return linear_backward(false, a, a_shape, a_rank, b, b_shape, b_rank, axis, reverse, states, grad_out, grad_a,
                           grad_b, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
