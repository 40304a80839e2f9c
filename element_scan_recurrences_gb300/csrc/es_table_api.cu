// es_table_api.cu -- the table-scan entry points of the C ABI (es.h).
//
// Contract ("Tensor operations": the `table-scan` row and section): `table`
// is [states symbols] and `symbols` any shape, both i32 (the typed pointers
// fix the dtype); a table with no states or no symbols, an axis out of range
// or a start that is not a state is E-DIM-001.  The result has `symbols`'
// shape.
#include <cstring>
#include <string>

#include "es.h"
#include "es_internal.h"
#include "es_table.h"

namespace es {
namespace {

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

struct TablePlan {
    TableLaunch L;
    int64_t elements;
    int path;
};

es_status plan_table(const int32_t* table, int64_t n_states, int64_t n_syms, const int32_t* sym,
                     const int64_t* shape, int rank, int axis, int32_t start, const int32_t* out, TablePlan* P) {
    const char* fn = "es_table_scan_i32";
    if (shape == nullptr) return api_fail(ES_E_ARG, "%s: null shape", fn);
    if (n_states < 1 || n_syms < 1)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: the table is [%lld %lld]; it needs at least one state and one "
                        "symbol", fn, static_cast<long long>(n_states), static_cast<long long>(n_syms));
    int64_t entries;
    if (!mul_ok(n_states, n_syms, &entries) || entries >= (int64_t(1) << 31))
        return api_fail(ES_E_UNSUPPORTED, "%s: a table of %lld x %lld entries is too large", fn,
                        static_cast<long long>(n_states), static_cast<long long>(n_syms));
    if (start < 0 || start >= n_states)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: start %d is not a state of a %lld-state table", fn, start,
                        static_cast<long long>(n_states));
    if (rank < 1 || rank > ES_MAX_RANK)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: symbols of rank %d (1..%d)", fn, rank, ES_MAX_RANK);
    for (int d = 0; d < rank; ++d)
        if (shape[d] < 0) return api_fail(ES_E_DIM_001, "E-DIM-001 %s: a negative dimension", fn);
    if (axis < -rank || axis >= rank)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: axis %d out of range for rank %d", fn, axis, rank);
    const int ax = axis < 0 ? axis + rank : axis;
    TableLaunch& L = P->L;
    L = TableLaunch{};
    L.table = table;
    L.sym = sym;
    L.out = const_cast<int*>(out);
    L.O = 1;
    L.J = 1;
    for (int d = 0; d < ax; ++d)
        if (!mul_ok(L.O, shape[d], &L.O)) return api_fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    for (int d = ax + 1; d < rank; ++d)
        if (!mul_ok(L.J, shape[d], &L.J)) return api_fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    L.T = shape[ax];
    L.n_states = static_cast<int>(n_states);
    L.n_syms = static_cast<int>(n_syms);
    L.start = start;
    int64_t tmp;
    if (!mul_ok(L.O, L.T, &tmp) || !mul_ok(tmp, L.J, &P->elements) || P->elements > (int64_t(1) << 60))
        return api_fail(ES_E_UNSUPPORTED, "%s: element count overflows", fn);
    if (P->elements == 0) {
        P->path = ES_PATH_EMPTY;
        return ES_OK;
    }
    if (table == nullptr || sym == nullptr || out == nullptr) return api_fail(ES_E_ARG, "%s: null data pointer", fn);
    if (reinterpret_cast<uintptr_t>(table) % 4 || reinterpret_cast<uintptr_t>(sym) % 4 ||
        reinterpret_cast<uintptr_t>(out) % 4)
        return api_fail(ES_E_ARG, "%s: a data pointer is not 4-byte aligned", fn);
    const uintptr_t olo = reinterpret_cast<uintptr_t>(out), ohi = olo + static_cast<uintptr_t>(P->elements) * 4;
    const uintptr_t slo = reinterpret_cast<uintptr_t>(sym), shi = slo + static_cast<uintptr_t>(P->elements) * 4;
    const uintptr_t tlo = reinterpret_cast<uintptr_t>(table), thi = tlo + static_cast<uintptr_t>(entries) * 4;
    if ((slo < ohi && olo < shi) || (tlo < ohi && olo < thi))
        return api_fail(ES_E_ARG, "%s: `out` overlaps an input", fn);
    const bool time_ok = table_time_ok(L.O, L.T, L.J, sym, out);
    const bool lane_ok = table_lane_ok(L.O, L.T, L.J, sym, out);
    const int forced = api_path_override();
    if (forced == ES_PATH_AUTO) {
        P->path = time_ok ? ES_PATH_TIME_TMA : lane_ok ? ES_PATH_LANE_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    if (forced == ES_PATH_GENERIC || (forced == ES_PATH_TIME_TMA && time_ok) || (forced == ES_PATH_LANE_TMA && lane_ok)) {
        P->path = forced;
        return ES_OK;
    }
    return api_fail(ES_E_UNSUPPORTED, "%s: the forced kernel path %d cannot serve this call", fn, forced);
}

}  // namespace
}  // namespace es

extern "C" {

es_status es_plan_table_scan_i32(const int32_t* table, int64_t n_states, int64_t n_syms, const int32_t* symbols,
                                 const int64_t* shape, int rank, int axis, int32_t start, const int32_t* out,
                                 es_plan_info* info) {
    es::TablePlan P{};
    es_status st = es::plan_table(table, n_states, n_syms, symbols, shape, rank, axis, start, out, &P);
    if (st != ES_OK) return st;
    if (info != nullptr) {
        std::memset(info, 0, sizeof(*info));
        info->O = P.L.O;
        info->T = P.L.T;
        info->J = P.L.J;
        info->W = 1;
        info->seq_width[0] = 1;
        info->elements = P.elements;
        info->path = P.path;
    }
    return ES_OK;
}

es_status es_table_scan_i32(const int32_t* table, int64_t n_states, int64_t n_syms, const int32_t* symbols,
                            const int64_t* shape, int rank, int axis, int32_t start, int32_t* out,
                            es_stream_t stream) {
    es::TablePlan P{};
    es_status st = es::plan_table(table, n_states, n_syms, symbols, shape, rank, axis, start, out, &P);
    if (st != ES_OK || P.path == ES_PATH_EMPTY) return st;
    int dev = 0;
    es::DeviceState* ds = nullptr;
    if ((st = es::api_device(&dev, &ds)) != ES_OK) return st;
    es::TableLaunch& L = P.L;
    L.status = ds->status;
    L.wait_ns = es::api_wait_ns();
    L.drop_tile = es::api_drop_tile();
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.num_sms = ds->num_sms;
    const char* msg = nullptr;
    cudaError_t e;
    if (P.path == ES_PATH_GENERIC) {
        e = es::launch_table_generic(L);
    } else {
        if ((st = es::api_encoder(&L.encode)) != ES_OK) return st;
        e = P.path == ES_PATH_TIME_TMA ? es::launch_table_time(L, &msg) : es::launch_table_lane(L, &msg);
    }
    if (e != cudaSuccess)
        return es::api_fail(ES_E_CUDA, "es_table_scan_i32: %s", msg != nullptr ? msg : cudaGetErrorString(e));
    es::count_launch();
    return ES_OK;
}

}  // extern "C"
