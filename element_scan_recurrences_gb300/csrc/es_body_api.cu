// es_body_api.cu -- the body-program entry points of the C ABI (es.h):
// checking a call, choosing a kernel skeleton, generating the body's functor
// and launching the kernel compiled from them at run time.
//
// Paths ("Nonlinear element scans": lanes in parallel, trips in sequence):
//   * ES_PATH_LANE_TMA  scalar state (or width one), lanes innermost: the
//     TMA time-tile pipeline of skel_lane.cuh;
//   * ES_PATH_TIME_TMA  scalar state with the sequence axis last: TMA tiles
//     transposed in shared memory (skel_time.cuh);
//   * ES_PATH_VEC_TMA   vector state of 2, 4, 8 or 16 values: the TMA
//     pipeline with a lane's state over G threads (skel_vec.cuh);
//   * ES_PATH_GENERIC   any shape or alignment (skel_generic.cuh).
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "es.h"
#include "es_body_compiler.h"
#include "es_internal.h"
#include "es_jit.h"
#include "skel_common.cuh"

struct es_body_program {
    std::unique_ptr<es::body::Program> prog;
    std::mutex mu;
    // generated functor per (state width, vector state, wide mask, with the
    // vector-Jacobian product)
    std::map<std::tuple<int, bool, unsigned, bool>, std::string> functors;
};

namespace es {
namespace {

using body::Error;

es_status body_fail(const Error& e) { return api_fail(ES_E_BODY, "%s: %s", e.code.c_str(), e.msg.c_str()); }

// the functor for a signature, generated once per program
es_status functor_for(es_body_program* b, int W, bool vector, unsigned wide_mask, std::string* out,
                      bool with_vjp = false) {
    std::lock_guard<std::mutex> lock(b->mu);
    const auto key = std::make_tuple(W, vector, wide_mask, with_vjp);
    auto it = b->functors.find(key);
    if (it == b->functors.end()) {
        try {
            it = b->functors.emplace(key, b->prog->generate(W, vector, wide_mask, with_vjp)).first;
        } catch (const Error& e) {
            return body_fail(e);
        }
    }
    *out = it->second;
    return ES_OK;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

struct BodyCall {
    ShapePlan S;
    bool vector;          // `:state-axis` given
    unsigned wide_mask;   // bit k: sequence k is as wide as the state
    int reverse;
    int path;
    std::string functor;  // the body's generated functor for this signature
};

// lanes innermost: I = J contiguous lanes per trip row, 16-byte rows
bool body_lane_ok(const ShapePlan& S, const float* const* seqs, const float* out) {
    if (S.W != 1) return false;
    const int64_t I = S.J;
    if (I < 32 || I % 4 != 0) return false;
    if (S.O >= (int64_t(1) << 31) || S.T >= (int64_t(1) << 31) || I >= (int64_t(1) << 31)) return false;
    if (S.O * ((I + 31) / 32) >= (int64_t(1) << 31)) return false;
    if (!aligned16(out)) return false;
    for (int k = 0; k < S.n_seqs; ++k)
        if (!aligned16(seqs[k])) return false;
    return true;
}

// sequence axis innermost: one row of T values per lane, 16-byte rows
bool body_time_ok(const ShapePlan& S, const float* const* seqs, const float* out) {
    if (S.W != 1 || S.J != 1) return false;
    if (S.T % 4 != 0 || S.T < 32) return false;
    if (S.O >= (int64_t(1) << 31) || S.T >= (int64_t(1) << 31)) return false;
    if (!aligned16(out)) return false;
    for (int k = 0; k < S.n_seqs; ++k)
        if (!aligned16(seqs[k])) return false;
    return true;
}

// vector state of 2, 4, 8 or 16 values: 128 values per CTA and trip, 16-byte
// rows and boxes for every sequence
bool body_vec_ok(const ShapePlan& S, const float* const* seqs, const float* out) {
    const int64_t W = S.W;
    if (W != 2 && W != 4 && W != 8 && W != 16) return false;
    const int64_t LV = 128 / W;
    if (S.J < LV || (S.J * W) % 4 != 0) return false;
    for (int k = 0; k < S.n_seqs; ++k)
        if (S.sw[k] == 1 && S.J % 4 != 0) return false;
    if (S.O >= (int64_t(1) << 31) || S.T >= (int64_t(1) << 31) || S.J * W >= (int64_t(1) << 31)) return false;
    if (S.O * ((S.J + LV - 1) / LV) >= (int64_t(1) << 31)) return false;
    if (!aligned16(out)) return false;
    for (int k = 0; k < S.n_seqs; ++k)
        if (!aligned16(seqs[k])) return false;
    return true;
}

es_status plan_body(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                    const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                    int reverse, const float* out, BodyCall* C, bool zero_initial = false) {
    if (body == nullptr || !body->prog) return api_fail(ES_E_ARG, "es_scan_body_f32: null body program");
    const body::Program& p = *body->prog;
    if (n_seqs != p.n_seqs())
        return api_fail(ES_E_BODY, "arity: the body takes %d sequence(s), the call passes %d", p.n_seqs(), n_seqs);
    static const char* const kNames[ES_MAX_SEQS] = {"seq 0", "seq 1", "seq 2", "seq 3",
                                                    "seq 4", "seq 5", "seq 6", "seq 7"};
    es_status st = plan_shapes("es_scan_body_f32", kNames, initial, seqs, n_seqs, shape, rank, axis, state_width,
                               seq_widths, out, &C->S, zero_initial);
    if (st != ES_OK) return st;
    C->vector = state_width != 0;
    C->reverse = reverse ? 1 : 0;
    C->wide_mask = 0;
    for (int k = 0; k < n_seqs; ++k)
        if (C->S.sw[k] == C->S.W) C->wide_mask |= 1u << k;
    // the body must fit the signature (checked before any path choice)
    if ((st = functor_for(body, static_cast<int>(C->S.W), C->vector, C->wide_mask, &C->functor)) != ES_OK)
        return st;
    if (C->S.empty) {
        C->path = ES_PATH_EMPTY;
        return ES_OK;
    }
    const bool lane_ok = body_lane_ok(C->S, seqs, out);
    const bool time_ok = body_time_ok(C->S, seqs, out);
    const bool vec_ok = body_vec_ok(C->S, seqs, out);
    const int forced = api_path_override();
    if (forced == ES_PATH_AUTO) {
        C->path = vec_ok ? ES_PATH_VEC_TMA : time_ok ? ES_PATH_TIME_TMA : lane_ok ? ES_PATH_LANE_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    if (forced == ES_PATH_GENERIC || (forced == ES_PATH_LANE_TMA && lane_ok) || (forced == ES_PATH_TIME_TMA && time_ok) ||
        (forced == ES_PATH_VEC_TMA && vec_ok)) {
        C->path = forced;
        return ES_OK;
    }
    return api_fail(ES_E_UNSUPPORTED, "es_scan_body_f32: the forced kernel path %d cannot serve this call", forced);
}

// ---------------------------------------------------------------------------
// launchers (one kernel each)

struct BodyLaunch {
    const BodyCall* C;
    const float* init;
    const float* const* seqs;
    float* out;
    cudaStream_t stream;
    DeviceState* dev;
    EncodeTiledFn encode;
};

// Kernel sources: a skeleton header, the functor, and the instantiation to
// compile (template arguments of the launch configuration).
struct KernelText {
    std::string source;
    std::string name;
};

KernelText generic_text(const std::string& functor, int W) {
    return {"#include \"skel_generic.cuh\"\n" + functor, "&es::k_body_generic<EsBody, " + std::to_string(W) + ">"};
}

KernelText lane_text(const std::string& functor, int LI, int TT) {
    return {"#include \"skel_lane.cuh\"\n" + functor,
            "&es::k_body_lane<EsBody, " + std::to_string(LI) + ", " + std::to_string(TT) + ">"};
}

constexpr int kTimeLO = 64;   // rows (lanes) per CTA of the time-innermost skeleton

KernelText time_text(const std::string& functor) {
    return {"#include \"skel_time.cuh\"\n" + functor, "&es::k_body_time<EsBody, " + std::to_string(kTimeLO) + ">"};
}

// Values of a lane's state per thread in the vector-state skeleton: one.  A
// trip is a serial chain whose operations on the thread's own values run one
// after another (an IEEE division or square root is tens of cycles each),
// while a lane-group shuffle adds about 30 cycles per halving; on GB300 the
// NORMCAP body took 0.47 / 0.38 / 0.34 ms (2048 trips) at 4 / 2 / 1 values
// per thread, 0.73 at 8 and 2.1 at 16.
int vec_values(int) { return 1; }

KernelText vec_text(const std::string& functor, int W, int TT) {
    return {"#include \"skel_vec.cuh\"\n" + functor, "&es::k_body_vec<EsBody, " + std::to_string(W) + ", " +
                                                           std::to_string(vec_values(W)) + ", " +
                                                           std::to_string(TT) + ">"};
}

// bytes of one vector-state pipeline stage (every sequence's TT-trip tile)
int64_t vec_stage_bytes(int W, int TT, int n_wide, int n_narrow) {
    return static_cast<int64_t>(TT) * (n_wide * 128LL * 4 + n_narrow * (128LL / W) * 4);
}

// bytes of one forward vector-state stage: the sequences' tiles, then the
// tile of states the store warp sends out (as laid out by k_body_vec)
int64_t vec_fwd_stage_bytes(int W, int TT, int n_wide, int n_narrow) {
    const int64_t in = (vec_stage_bytes(W, TT, n_wide, n_narrow) + 127) & ~int64_t(127);
    return (in + static_cast<int64_t>(TT) * 128 * 4 + 1023) & ~int64_t(1023);
}

// trips per vector-state tile: 32 unless a stage of every sequence would
// pass 64 KB
int vec_trips(int W, int n_wide, int n_narrow) {
    int TT = 32;
    while (TT > 8 && vec_stage_bytes(W, TT, n_wide, n_narrow) > 64 * 1024) TT /= 2;
    return TT;
}

// trips per tile of the lanes-innermost skeleton: every sequence's tile sits
// in registers
int lane_trips(int n_seqs) { return n_seqs <= 2 ? 32 : n_seqs <= 4 ? 16 : 8; }

bool launch_body_generic(const BodyLaunch& L, std::string* err) {
    const BodyCall& C = *L.C;
    JitKernel k;
    const KernelText kt = generic_text(C.functor, static_cast<int>(C.S.W));
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    SeqPtrs sp{};
    for (int q = 0; q < C.S.n_seqs; ++q) sp.p[q] = L.seqs[q];
    const int64_t lanes = C.S.O * C.S.J;
    const int threads = 128;
    const int64_t blocks = (lanes + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) {
        *err = "too many lanes for one launch";
        return false;
    }
    const float* init = L.init;
    float* out = L.out;
    int64_t O = C.S.O, T = C.S.T, J = C.S.J;
    int reverse = C.reverse;
    void* args[] = {&sp, &init, &out, &O, &T, &J, &reverse};
    return jit_launch(k, static_cast<unsigned>(blocks), threads, 0, L.stream, args, err);
}

// a 3-D map over [O, T, I] with box {LI, TT, 1}
bool encode_rows(EncodeTiledFn encode, CUtensorMap* m, const float* base, int64_t O, int64_t T, int64_t I, int LI,
                 int TT) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(O)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(I) * 4, static_cast<cuuint64_t>(I) * T * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(LI), static_cast<cuuint32_t>(TT), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool launch_body_lane(const BodyLaunch& L, std::string* err) {
    const BodyCall& C = *L.C;
    const int NS = C.S.n_seqs;
    const int64_t I = C.S.J;
    // lanes per CTA: the widest tile (the longest contiguous row segment per
    // TMA box row) that still puts a CTA on most SMs
    int LI = 32;
    for (int cand : {256, 128, 64}) {
        if (I >= cand && 5 * C.S.O * ((I + cand - 1) / cand) >= 4LL * L.dev->num_sms) {
            LI = cand;
            break;
        }
    }
    const int TT = lane_trips(NS);
    // about 96 trips in flight; when there are more CTAs than SMs, at most
    // about 100 KB of shared memory each, so that two CTAs share an SM (one
    // consumer group alone cannot keep the serial chains' latency covered)
    const int64_t stage_bytes = static_cast<int64_t>(NS) * TT * LI * 4;
    const int64_t tiles_i = (I + LI - 1) / LI;
    const int64_t smem_cap = C.S.O * tiles_i > L.dev->num_sms ? 100 * 1024 : 200 * 1024;
    int stages = 96 / TT;
    if (stages > 8) stages = 8;
    while (stages > 2 && stages * stage_bytes > smem_cap) --stages;
    alignas(64) CUtensorMap maps[ES_MAX_SEQS];
    for (int q = 0; q < NS; ++q) {
        if (!encode_rows(L.encode, &maps[q], L.seqs[q], C.S.O, C.S.T, I, LI, TT)) {
            *err = "cuTensorMapEncodeTiled failed for a lane-innermost tile map";
            return false;
        }
    }
    JitKernel k;
    const KernelText kt = lane_text(C.functor, LI, TT);
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    const float* init = L.init;
    float* out = L.out;
    int T = static_cast<int>(C.S.T), Ii = static_cast<int>(I), ti = static_cast<int>(tiles_i);
    int reverse = C.reverse;
    unsigned int* status = L.dev->status;
    uint64_t wait_ns = api_wait_ns();
    int64_t drop = api_drop_tile();
    void* args[] = {maps, &init, &out, &T, &Ii, &ti, &stages, &reverse, &status, &wait_ns, &drop};
    const size_t smem = static_cast<size_t>(stages * stage_bytes) + 1024;
    return jit_launch(k, static_cast<unsigned>(C.S.O * tiles_i), 32 + LI, smem, L.stream, args, err);
}

// the functor of a signature given by widths (no shapes)
es_status signature_functor(const char* fn, es_body_t body, int state_width, int n_seqs, const int64_t* seq_widths,
                            std::string* functor, int* W_out, bool with_vjp = false) {
    if (body == nullptr || !body->prog) return api_fail(ES_E_ARG, "%s: null body program", fn);
    if (n_seqs != body->prog->n_seqs())
        return api_fail(ES_E_BODY, "arity: the body takes %d sequence(s), not %d", body->prog->n_seqs(), n_seqs);
    if (state_width < 0 || state_width > ES_MAX_STATE)
        return api_fail(ES_E_DIM_001, "E-DIM-001 %s: state width %d outside 0..%d", fn, state_width, ES_MAX_STATE);
    const int W = state_width == 0 ? 1 : state_width;
    unsigned mask = 0;
    for (int k = 0; k < n_seqs; ++k) {
        const int64_t w = seq_widths == nullptr ? W : seq_widths[k];
        if (state_width != 0 && w != 1 && w != W)
            return api_fail(ES_E_DIM_001, "E-DIM-001 %s: sequence %d has width %lld", fn, k,
                            static_cast<long long>(w));
        if (w == W) mask |= 1u << k;
    }
    *W_out = W;
    return functor_for(body, W, state_width != 0, mask, functor, with_vjp);
}

bool launch_body_time(const BodyLaunch& L, std::string* err) {
    const BodyCall& C = *L.C;
    const int NS = C.S.n_seqs;
    constexpr int LO = kTimeLO;
    const int64_t ctas = (C.S.O + LO - 1) / LO;
    int64_t per_sm = (ctas + L.dev->num_sms - 1) / L.dev->num_sms;
    per_sm = per_sm < 1 ? 1 : per_sm > 3 ? 3 : per_sm;
    const int64_t budget = (210 * 1024) / per_sm - 3 * LO * 128 - 1024;
    const int64_t stage_bytes = static_cast<int64_t>(NS) * LO * 128;
    int64_t st = budget / stage_bytes;
    const int stages = static_cast<int>(st < 2 ? 2 : st > 6 ? 6 : st);
    alignas(64) CUtensorMap maps[ES_MAX_SEQS + 1];
    for (int q = 0; q <= NS; ++q) {
        const float* basep = q < NS ? L.seqs[q] : L.out;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(C.S.T), static_cast<cuuint64_t>(C.S.O)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(C.S.T) * 4};
        const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(LO)};
        const cuuint32_t estr[2] = {1, 1};
        if (L.encode(&maps[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(basep), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled failed for a time-innermost tile map";
            return false;
        }
    }
    JitKernel k;
    const KernelText kt = time_text(C.functor);
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    const float* init = L.init;
    int O = static_cast<int>(C.S.O), T = static_cast<int>(C.S.T);
    int stg = stages, reverse = C.reverse;
    unsigned int* status = L.dev->status;
    uint64_t wait_ns = api_wait_ns();
    int64_t drop = api_drop_tile();
    void* args[] = {maps, &init, &O, &T, &stg, &reverse, &status, &wait_ns, &drop};
    const size_t smem = static_cast<size_t>(stages * stage_bytes) + 3 * LO * 128 + 1024;
    return jit_launch(k, static_cast<unsigned>(ctas), 32 + LO, smem, L.stream, args, err);
}

bool launch_body_vec(const BodyLaunch& L, std::string* err) {
    const BodyCall& C = *L.C;
    const int NS = C.S.n_seqs;
    const int W = static_cast<int>(C.S.W);
    const int LV = 128 / W;
    int n_wide = 0;
    for (int q = 0; q < NS; ++q) n_wide += C.S.sw[q] == W ? 1 : 0;
    const int TT = vec_trips(W, n_wide, NS - n_wide);
    const int64_t stage_bytes = vec_fwd_stage_bytes(W, TT, n_wide, NS - n_wide);
    const int64_t tiles_j = (C.S.J + LV - 1) / LV;
    const int64_t ctas = C.S.O * tiles_j;
    int64_t per_sm = (ctas + L.dev->num_sms - 1) / L.dev->num_sms;
    per_sm = per_sm < 1 ? 1 : per_sm > 8 ? 8 : per_sm;
    // a stage is held from its load through the chain to the store of its
    // states: three or more where shared memory allows
    int64_t budget = (200 * 1024) / per_sm;
    if (budget > 160 * 1024) budget = 160 * 1024;
    int64_t st = budget / stage_bytes;
    st = st < 3 ? 3 : st > 8 ? 8 : st;
    const int64_t fit = (222 * 1024) / stage_bytes;     // beside the reductions' static shared memory
    if (st > fit) st = fit < 2 ? 2 : fit;
    const int stages = static_cast<int>(st);
    alignas(64) CUtensorMap maps[ES_MAX_SEQS];
    for (int q = 0; q < NS; ++q) {
        const bool wide = C.S.sw[q] == W;
        const int64_t row = wide ? C.S.J * W : C.S.J;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row), static_cast<cuuint64_t>(C.S.T),
                                    static_cast<cuuint64_t>(C.S.O)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row) * 4, static_cast<cuuint64_t>(row) * C.S.T * 4};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(wide ? 128 : LV), static_cast<cuuint32_t>(TT), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (L.encode(&maps[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(L.seqs[q]), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled failed for a vector-state tile map";
            return false;
        }
    }
    alignas(64) CUtensorMap omap;
    {
        const int64_t row = C.S.J * W;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row), static_cast<cuuint64_t>(C.S.T),
                                    static_cast<cuuint64_t>(C.S.O)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row) * 4, static_cast<cuuint64_t>(row) * C.S.T * 4};
        const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(TT), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (L.encode(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, L.out, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled failed for the vector-state output map";
            return false;
        }
    }
    JitKernel k;
    const KernelText kt = vec_text(C.functor, W, TT);
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    const float* init = L.init;
    int T = static_cast<int>(C.S.T), J = static_cast<int>(C.S.J), tj = static_cast<int>(tiles_j);
    int stg = stages, reverse = C.reverse;
    unsigned int* status = L.dev->status;
    uint64_t wait_ns = api_wait_ns();
    int64_t drop = api_drop_tile();
    void* args[] = {maps, &omap, &init, &T, &J, &tj, &stg, &reverse, &status, &wait_ns, &drop};
    const size_t smem = static_cast<size_t>(stages * stage_bytes) + 1024;
    const int consumer_threads = 128 / vec_values(W);
    return jit_launch(k, static_cast<unsigned>(ctas), 32 * ((consumer_threads + 31) / 32) + 64, smem, L.stream, args,
                      err);
}

// ---------------------------------------------------------------------------
// backward ("Precision and gradients"): the body's vector-Jacobian product
// scanned in the opposite trip order, one thread per lane

KernelText generic_bwd_text(const std::string& functor, int W) {
    return {"#include \"skel_generic_bwd.cuh\"\n" + functor,
            "&es::k_body_generic_bwd<EsBody, " + std::to_string(W) + ">"};
}

KernelText lane_bwd_text(const std::string& functor, int LI, int TT) {
    return {"#include \"skel_lane_bwd.cuh\"\n" + functor,
            "&es::k_body_lane_bwd<EsBody, " + std::to_string(LI) + ", " + std::to_string(TT) + ">"};
}

// Trips per tile of the lanes-innermost backward: the sequences, the shifted
// states and the output gradient of a tile sit in registers.  With at most
// one CTA per SM (four consumer warps, one per SM sub-partition) the longer
// tile of the forward's size pays off: the per-tile barrier and wait are
// latency no other warp hides (GB300, 128 lanes x 128 rows x 16384 trips of
// the MAXPLUS body: 0.70 -> 0.77 of HBM peak; with two CTAs per SM the
// shorter tile stays ahead, 0.997 vs 0.948 on 64 x 1024 lanes).
int lane_bwd_trips(int n_seqs, bool one_cta_per_sm) {
    return one_cta_per_sm ? lane_trips(n_seqs) : lane_trips(n_seqs + 2);
}

// rows per CTA of the time-innermost backward: 64, or 32 with more than three
// sequences (every sequence's tile and its gradient's stay in shared memory)
int time_bwd_rows(int n_seqs) { return n_seqs <= 3 ? 64 : 32; }

KernelText time_bwd_text(const std::string& functor, int n_seqs) {
    return {"#include \"skel_time_bwd.cuh\"\n" + functor,
            "&es::k_body_time_bwd<EsBody, " + std::to_string(time_bwd_rows(n_seqs)) + ">"};
}

// values of a lane's state per thread in the vector-state backward
int vec_bwd_values(int) { return 1; }

KernelText vec_bwd_text(const std::string& functor, int W, int TT) {
    return {"#include \"skel_vec_bwd.cuh\"\n" + functor, "&es::k_body_vec_bwd<EsBody, " + std::to_string(W) + ", " +
                                                               std::to_string(vec_bwd_values(W)) + ", " +
                                                               std::to_string(TT) + ">"};
}

// bytes of one vector-state backward stage: the tiles of the sequences the
// VJP reads (n_wide, n_narrow of them), the output gradient's and TT+1 rows
// of the saved states
int64_t vec_bwd_stage_bytes(int W, int TT, int n_wide, int n_narrow) {
    return vec_stage_bytes(W, TT, n_wide + 1, n_narrow) + (TT + 1) * 128LL * 4;
}

// trips per vector-state backward tile: 32 unless a stage would pass 32 KB
// (two or three CTAs share an SM)
int vec_bwd_trips(int W, int n_wide, int n_narrow) {
    int TT = 32;
    while (TT > 8 && vec_bwd_stage_bytes(W, TT, n_wide, n_narrow) > 32 * 1024) TT /= 2;
    return TT;
}

// the sequences a backward functor's VJP reads (its kVjpSeqs)
unsigned vjp_live_mask(const std::string& functor) {
    const std::string key = "kVjpSeqs = 0x";
    const size_t at = functor.find(key);
    if (at == std::string::npos) return ~0u;
    return static_cast<unsigned>(std::strtoul(functor.c_str() + at + key.size(), nullptr, 16));
}

int popcount(unsigned x) {
    int n = 0;
    for (; x != 0; x &= x - 1) ++n;
    return n;
}

// the live sequences of a signature, wide and width-one
void live_counts(unsigned live, int n_seqs, const int64_t* widths, int W, int* n_wide, int* n_narrow) {
    *n_wide = *n_narrow = 0;
    for (int k = 0; k < n_seqs; ++k) {
        if (!((live >> k) & 1u)) continue;
        if (widths == nullptr || widths[k] == W) ++*n_wide;
        else ++*n_narrow;
    }
}

struct BodyBwdCall {
    BodyCall C;           // the forward call's plan (shapes, signature)
    std::string functor;  // the functor with its `vjp`
};

// The forward plan for the shapes (the saved states have the output shape),
// then the gradient buffers: present, 4-byte aligned, disjoint from every
// input and from each other.
es_status plan_body_backward(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                             const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                             int reverse, const float* states, const float* grad_out, const float* grad_initial,
                             float* const* grad_seqs, BodyBwdCall* B, bool zero_initial = false) {
    static const char* const kFn = "es_scan_body_backward_f32";
    // the forced-path check comes after the plan (any forward path is fine)
    BodyCall& C = B->C;
    es_status st = plan_body(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, reverse, states,
                             &C, zero_initial);
    if (st != ES_OK) return st;
    if ((st = functor_for(body, static_cast<int>(C.S.W), C.vector, C.wide_mask, &B->functor, true)) != ES_OK)
        return st;
    const int forced = api_path_override();
    if (forced != ES_PATH_AUTO && forced != ES_PATH_GENERIC && forced != ES_PATH_LANE_TMA && forced != ES_PATH_VEC_TMA &&
        forced != ES_PATH_TIME_TMA)
        return api_fail(ES_E_UNSUPPORTED, "%s: the forced kernel path %d cannot serve this call", kFn, forced);
    if (C.S.empty) {
        C.path = ES_PATH_EMPTY;
        return ES_OK;
    }
    // from zero (an internal caller): no initial and no initial gradient
    if (grad_out == nullptr || (grad_initial == nullptr) != zero_initial || grad_seqs == nullptr)
        return api_fail(ES_E_ARG, "%s: null gradient pointer", kFn);
    for (int k = 0; k < n_seqs; ++k)
        if (grad_seqs[k] == nullptr) return api_fail(ES_E_ARG, "%s: null gradient pointer", kFn);
    // every buffer of the call: inputs first, then the written gradients
    const int nb = 2 * n_seqs + 4;
    std::vector<const void*> ptr(nb);
    std::vector<int64_t> cnt(nb);
    std::vector<std::string> nm(nb);
    ptr[0] = initial, cnt[0] = C.S.n_init, nm[0] = "initial";
    for (int k = 0; k < n_seqs; ++k) ptr[1 + k] = seqs[k], cnt[1 + k] = C.S.n_seq[k], nm[1 + k] = "seq " + std::to_string(k);
    ptr[n_seqs + 1] = states, cnt[n_seqs + 1] = C.S.n_out, nm[n_seqs + 1] = "states";
    ptr[n_seqs + 2] = grad_out, cnt[n_seqs + 2] = C.S.n_out, nm[n_seqs + 2] = "grad_out";
    ptr[n_seqs + 3] = grad_initial, cnt[n_seqs + 3] = C.S.n_init, nm[n_seqs + 3] = "grad_initial";
    for (int k = 0; k < n_seqs; ++k)
        ptr[n_seqs + 4 + k] = grad_seqs[k], cnt[n_seqs + 4 + k] = C.S.n_seq[k], nm[n_seqs + 4 + k] = "grad seq " + std::to_string(k);
    for (int k = 0; k < nb; ++k)
        if (reinterpret_cast<uintptr_t>(ptr[k]) % 4 != 0)
            return api_fail(ES_E_ARG, "%s: `%s` is not 4-byte aligned", kFn, nm[k].c_str());
    for (int k = n_seqs + 3; k < nb; ++k) {
        if (ptr[k] == nullptr) continue;        // no initial gradient (a scan from zero)
        const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr[k]), hi = lo + static_cast<uintptr_t>(cnt[k]) * 4;
        for (int q = 0; q < nb; ++q) {
            if (q == k || ptr[q] == nullptr) continue;
            const uintptr_t l2 = reinterpret_cast<uintptr_t>(ptr[q]), h2 = l2 + static_cast<uintptr_t>(cnt[q]) * 4;
            if (lo < h2 && l2 < hi)
                return api_fail(ES_E_ARG, "%s: `%s` overlaps `%s`", kFn, nm[k].c_str(), nm[q].c_str());
        }
    }
    // the forward's tile rules for every buffer TMA reads or writes
    bool grads16 = aligned16(grad_out);
    for (int k = 0; k < n_seqs; ++k) grads16 = grads16 && aligned16(grad_seqs[k]);
    const bool lane_ok = grads16 && body_lane_ok(C.S, seqs, states);
    const bool vec_ok = grads16 && body_vec_ok(C.S, seqs, states);
    // the 36-trip state boxes want at least two tiles of trips
    const bool time_ok = grads16 && C.S.T >= 64 && body_time_ok(C.S, seqs, states);
    if (forced == ES_PATH_AUTO) {
        C.path = vec_ok ? ES_PATH_VEC_TMA : time_ok ? ES_PATH_TIME_TMA : lane_ok ? ES_PATH_LANE_TMA : ES_PATH_GENERIC;
        return ES_OK;
    }
    if (forced == ES_PATH_GENERIC || (forced == ES_PATH_LANE_TMA && lane_ok) || (forced == ES_PATH_VEC_TMA && vec_ok) ||
        (forced == ES_PATH_TIME_TMA && time_ok)) {
        C.path = forced;
        return ES_OK;
    }
    return api_fail(ES_E_UNSUPPORTED, "%s: the forced kernel path %d cannot serve this call", kFn, forced);
}

bool launch_body_generic_bwd(const BodyBwdCall& B, const float* init, const float* const* seqs, const float* states,
                             const float* gout, float* ginit, float* const* gseqs, cudaStream_t stream,
                             std::string* err) {
    const BodyCall& C = B.C;
    JitKernel k;
    const KernelText kt = generic_bwd_text(B.functor, static_cast<int>(C.S.W));
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    SeqPtrs sp{};
    GradPtrs gp{};
    for (int q = 0; q < C.S.n_seqs; ++q) {
        sp.p[q] = seqs[q];
        gp.p[q] = gseqs[q];
    }
    const int64_t lanes = C.S.O * C.S.J;
    const int threads = 128;
    const int64_t blocks = (lanes + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) {
        *err = "too many lanes for one launch";
        return false;
    }
    int64_t O = C.S.O, T = C.S.T, J = C.S.J;
    int reverse = C.reverse;
    void* args[] = {&sp, &init, &states, &gout, &gp, &ginit, &O, &T, &J, &reverse};
    return jit_launch(k, static_cast<unsigned>(blocks), threads, 0, stream, args, err);
}

bool launch_body_lane_bwd(const BodyBwdCall& B, const float* init, const float* const* seqs, const float* states,
                          const float* gout, float* ginit, float* const* gseqs, cudaStream_t stream,
                          DeviceState* dev, EncodeTiledFn encode, std::string* err) {
    const BodyCall& C = B.C;
    const int NS = C.S.n_seqs;
    const int NM = NS + 2;
    const int64_t I = C.S.J;
    int LI = 32;
    for (int cand : {128, 64}) {
        if (I >= cand && 5 * C.S.O * ((I + cand - 1) / cand) >= 4LL * dev->num_sms) {
            LI = cand;
            break;
        }
    }
    const int64_t tiles_i = (I + LI - 1) / LI;
    const bool one_per_sm = C.S.O * tiles_i <= dev->num_sms;
    const int NL = popcount(vjp_live_mask(B.functor) & ((1u << NS) - 1u));   // sequences streamed
    const int TT = lane_bwd_trips(NL, one_per_sm);
    // the live sequences' tiles, the output gradient's, TT+1 rows of states
    const int64_t stage_bytes = ((NL + 1) * static_cast<int64_t>(TT) + TT + 1) * LI * 4;
    const int64_t out_bytes = 2LL * NS * TT * LI * 4;       // two gradient tiles
    const int64_t smem_cap = one_per_sm ? 200 * 1024 : 100 * 1024;
    int stages = 96 / TT;
    if (stages > 8) stages = 8;
    while (stages > 2 && stages * stage_bytes + out_bytes > smem_cap) --stages;
    // the sequences, the saved states, the output gradient, then the gradients
    alignas(64) CUtensorMap maps[2 * ES_MAX_SEQS + 2];
    for (int q = 0; q < 2 * NS + 2; ++q) {
        const float* base = q < NS ? seqs[q] : q == NS ? states : q == NS + 1 ? gout : gseqs[q - NM];
        if (!encode_rows(encode, &maps[q], base, C.S.O, C.S.T, I, LI, q == NS ? TT + 1 : TT)) {
            *err = "cuTensorMapEncodeTiled failed for a lane-innermost backward tile map";
            return false;
        }
    }
    JitKernel k;
    const KernelText kt = lane_bwd_text(B.functor, LI, TT);
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    int T = static_cast<int>(C.S.T), Ii = static_cast<int>(I), ti = static_cast<int>(tiles_i);
    int reverse = C.reverse;
    unsigned int* status = dev->status;
    uint64_t wait_ns = api_wait_ns();
    int64_t drop = api_drop_tile();
    void* args[] = {maps, &init, &ginit, &T, &Ii, &ti, &stages, &reverse, &status, &wait_ns, &drop};
    const size_t smem = static_cast<size_t>(stages * stage_bytes + out_bytes) + 1024;
    return jit_launch(k, static_cast<unsigned>(C.S.O * tiles_i), 32 + LI, smem, stream, args, err);
}

bool launch_body_vec_bwd(const BodyBwdCall& B, const float* init, const float* const* seqs, const float* states,
                         const float* gout, float* ginit, float* const* gseqs, cudaStream_t stream, DeviceState* dev,
                         EncodeTiledFn encode, std::string* err) {
    const BodyCall& C = B.C;
    const int NS = C.S.n_seqs;
    const int W = static_cast<int>(C.S.W);
    const int LV = 128 / W;
    int n_wide = 0;
    for (int q = 0; q < NS; ++q) n_wide += C.S.sw[q] == W ? 1 : 0;
    int lw = 0, ln = 0;
    live_counts(vjp_live_mask(B.functor), NS, C.S.sw, W, &lw, &ln);
    const int TT = vec_bwd_trips(W, lw, ln);
    const int64_t stage_bytes = vec_bwd_stage_bytes(W, TT, lw, ln);
    const int64_t out_bytes = 2 * vec_stage_bytes(W, TT, n_wide, NS - n_wide);   // two gradient tiles
    const int64_t tiles_j = (C.S.J + LV - 1) / LV;
    const int64_t ctas = C.S.O * tiles_j;
    int64_t per_sm = (ctas + dev->num_sms - 1) / dev->num_sms;
    per_sm = per_sm < 1 ? 1 : per_sm > 8 ? 8 : per_sm;
    int64_t budget = (200 * 1024) / per_sm;
    if (budget > 160 * 1024) budget = 160 * 1024;
    int64_t st = (budget - out_bytes) / stage_bytes;
    const int stages = static_cast<int>(st < 2 ? 2 : st > 8 ? 8 : st);
    // the sequences, the saved states, the output gradient, then the gradients
    alignas(64) CUtensorMap maps[2 * ES_MAX_SEQS + 2];
    for (int q = 0; q < 2 * NS + 2; ++q) {
        const int qs = q < NS ? q : q >= NS + 2 ? q - NS - 2 : -1;   // the sequence a map follows
        const bool wide = qs < 0 || C.S.sw[qs] == W;
        const float* basep = q < NS ? seqs[q] : q == NS ? states : q == NS + 1 ? gout : gseqs[q - NS - 2];
        const int64_t row = wide ? C.S.J * W : C.S.J;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row), static_cast<cuuint64_t>(C.S.T),
                                    static_cast<cuuint64_t>(C.S.O)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row) * 4, static_cast<cuuint64_t>(row) * C.S.T * 4};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(wide ? 128 : LV),
                                   static_cast<cuuint32_t>(q == NS ? TT + 1 : TT), 1};   // states: TT+1 rows
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&maps[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(basep), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled failed for a vector-state backward tile map";
            return false;
        }
    }
    JitKernel k;
    const KernelText kt = vec_bwd_text(B.functor, W, TT);
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    int T = static_cast<int>(C.S.T), J = static_cast<int>(C.S.J), tj = static_cast<int>(tiles_j);
    int stg = stages, reverse = C.reverse;
    unsigned int* status = dev->status;
    uint64_t wait_ns = api_wait_ns();
    int64_t drop = api_drop_tile();
    void* args[] = {maps, &init, &ginit, &T, &J, &tj, &stg, &reverse, &status, &wait_ns, &drop};
    const size_t smem = static_cast<size_t>(stages * stage_bytes + out_bytes) + 1024;
    return jit_launch(k, static_cast<unsigned>(ctas), 32 + 128 / vec_bwd_values(W), smem, stream, args, err);
}

bool launch_body_time_bwd(const BodyBwdCall& B, const float* init, const float* const* seqs, const float* states,
                          const float* gout, float* ginit, float* const* gseqs, cudaStream_t stream,
                          DeviceState* dev, EncodeTiledFn encode, std::string* err) {
    const BodyCall& C = B.C;
    const int NS = C.S.n_seqs;
    const int LO = time_bwd_rows(NS);
    const int NL = popcount(vjp_live_mask(B.functor) & ((1u << NS) - 1u));   // sequences streamed
    const int64_t stage_bytes = ((NL + 1) * LO * 128LL + LO * 144LL + 1023) & ~1023LL;
    const int64_t out_bytes = 2LL * NS * LO * 128;
    const int64_t ctas = (C.S.O + LO - 1) / LO;
    int64_t per_sm = (ctas + dev->num_sms - 1) / dev->num_sms;
    per_sm = per_sm < 1 ? 1 : per_sm > 2 ? 2 : per_sm;
    const int64_t budget = (220 * 1024) / per_sm - out_bytes - 2048;
    int64_t st = budget / stage_bytes;
    const int stages = static_cast<int>(st < 2 ? 2 : st > 4 ? 4 : st);
    // the sequences, the saved states (36-trip unswizzled boxes), the output
    // gradient, then the gradients
    alignas(64) CUtensorMap maps[2 * ES_MAX_SEQS + 2];
    for (int q = 0; q < 2 * NS + 2; ++q) {
        const bool hbox = q == NS;
        const float* basep = q < NS ? seqs[q] : q == NS ? states : q == NS + 1 ? gout : gseqs[q - NS - 2];
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(C.S.T), static_cast<cuuint64_t>(C.S.O)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(C.S.T) * 4};
        const cuuint32_t box[2] = {hbox ? 36u : 32u, static_cast<cuuint32_t>(LO)};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&maps[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(basep), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, hbox ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled failed for a time-innermost backward tile map";
            return false;
        }
    }
    JitKernel k;
    const KernelText kt = time_bwd_text(B.functor, NS);
    if (!jit_kernel(kt.source, kt.name, &k, err)) return false;
    int O = static_cast<int>(C.S.O), T = static_cast<int>(C.S.T);
    int stg = stages, reverse = C.reverse;
    unsigned int* status = dev->status;
    uint64_t wait_ns = api_wait_ns();
    int64_t drop = api_drop_tile();
    void* args[] = {maps, &init, &ginit, &O, &T, &stg, &reverse, &status, &wait_ns, &drop};
    const size_t smem = static_cast<size_t>(stages * stage_bytes + out_bytes) + 1024;
    return jit_launch(k, static_cast<unsigned>(ctas), 32 + LO, smem, stream, args, err);
}

void fill_info(const BodyCall& C, es_plan_info* info) {
    if (info == nullptr) return;
    std::memset(info, 0, sizeof(*info));
    info->O = C.S.O;
    info->T = C.S.T;
    info->J = C.S.J;
    info->W = C.S.W;
    for (int k = 0; k < C.S.n_seqs; ++k) info->seq_width[k] = C.S.sw[k];
    info->elements = C.S.n_out;
    info->path = C.path;
    info->reverse = C.reverse;
}

}  // namespace
}  // namespace es

extern "C" {

es_status es_body_create(const char* text, es_body_t* body) {
    if (text == nullptr || body == nullptr) return es::api_fail(ES_E_ARG, "es_body_create: null argument");
    *body = nullptr;
    try {
        std::unique_ptr<es_body_program> b(new es_body_program());
        b->prog = es::body::Program::parse(text);
        *body = b.release();
    } catch (const es::body::Error& e) {
        return es::body_fail(e);
    } catch (const std::bad_alloc&) {
        return es::api_fail(ES_E_ARG, "es_body_create: out of host memory");
    }
    return ES_OK;
}

es_status es_body_destroy(es_body_t body) {
    delete body;
    return ES_OK;
}

int es_body_n_seqs(es_body_t body) { return body != nullptr && body->prog ? body->prog->n_seqs() : -1; }

es_status es_body_source(es_body_t body, int state_width, int n_seqs, const int64_t* seq_widths, char* buf,
                         size_t cap, size_t* needed) {
    std::string src;
    int W = 1;
    es_status st = es::signature_functor("es_body_source", body, state_width, n_seqs, seq_widths, &src, &W);
    if (st != ES_OK) return st;
    if (needed != nullptr) *needed = src.size();
    if (buf != nullptr && cap > 0) {
        const size_t n = src.size() < cap - 1 ? src.size() : cap - 1;
        std::memcpy(buf, src.data(), n);
        buf[n] = '\0';
    }
    return ES_OK;
}

es_status es_body_prepare(es_body_t body, int state_width, int n_seqs, const int64_t* seq_widths, int path) {
    std::string functor;
    int W = 1;
    es_status st = es::signature_functor("es_body_prepare", body, state_width, n_seqs, seq_widths, &functor, &W);
    if (st != ES_OK) return st;
    std::vector<es::KernelText> todo;
    if (path == ES_PATH_AUTO || path == ES_PATH_GENERIC) todo.push_back(es::generic_text(functor, W));
    if ((path == ES_PATH_AUTO || path == ES_PATH_LANE_TMA) && W == 1)
        for (int LI : {32, 64, 128, 256}) todo.push_back(es::lane_text(functor, LI, es::lane_trips(n_seqs)));
    if ((path == ES_PATH_AUTO || path == ES_PATH_TIME_TMA) && W == 1) todo.push_back(es::time_text(functor));
    if ((path == ES_PATH_AUTO || path == ES_PATH_VEC_TMA) && (W == 2 || W == 4 || W == 8 || W == 16)) {
        int n_wide = 0;
        for (int k = 0; k < n_seqs; ++k) n_wide += (seq_widths == nullptr || seq_widths[k] == W) ? 1 : 0;
        todo.push_back(es::vec_text(functor, W, es::vec_trips(W, n_wide, n_seqs - n_wide)));
    }
    if (todo.empty())
        return es::api_fail(ES_E_UNSUPPORTED, "es_body_prepare: path %d cannot serve this signature", path);
    for (const es::KernelText& kt : todo) {
        std::string err;
        if (!es::jit_compile(kt.source, kt.name, &err)) return es::api_fail(ES_E_CUDA, "es_body_prepare: %s", err.c_str());
    }
    return ES_OK;
}

es_status es_body_prepare_backward(es_body_t body, int state_width, int n_seqs, const int64_t* seq_widths) {
    std::string functor;
    int W = 1;
    es_status st = es::signature_functor("es_body_prepare_backward", body, state_width, n_seqs, seq_widths, &functor,
                                         &W, true);
    if (st != ES_OK) return st;
    std::vector<es::KernelText> todo = {es::generic_bwd_text(functor, W)};
    const unsigned live = es::vjp_live_mask(functor);
    const int NL = es::popcount(live & ((1u << n_seqs) - 1u));
    if (W == 1)
        for (int LI : {32, 64, 128})
            for (bool one : {false, true}) {
                const int TT = es::lane_bwd_trips(NL, one);
                if (one && TT == es::lane_bwd_trips(NL, false)) continue;
                todo.push_back(es::lane_bwd_text(functor, LI, TT));
            }
    if (W == 1) todo.push_back(es::time_bwd_text(functor, n_seqs));
    if (W == 2 || W == 4 || W == 8 || W == 16) {
        int lw = 0, ln = 0;
        std::vector<int64_t> widths(n_seqs);
        for (int k = 0; k < n_seqs; ++k) widths[k] = seq_widths == nullptr ? W : seq_widths[k];
        es::live_counts(live, n_seqs, widths.data(), W, &lw, &ln);
        todo.push_back(es::vec_bwd_text(functor, W, es::vec_bwd_trips(W, lw, ln)));
    }
    for (const es::KernelText& kt : todo) {
        std::string err;
        if (!es::jit_compile(kt.source, kt.name, &err))
            return es::api_fail(ES_E_CUDA, "es_body_prepare_backward: %s", err.c_str());
    }
    return ES_OK;
}

es_status es_body_source_backward(es_body_t body, int state_width, int n_seqs, const int64_t* seq_widths, char* buf,
                                  size_t cap, size_t* needed) {
    std::string src;
    int W = 1;
    es_status st = es::signature_functor("es_body_source_backward", body, state_width, n_seqs, seq_widths, &src, &W,
                                         true);
    if (st != ES_OK) return st;
    if (needed != nullptr) *needed = src.size();
    if (buf != nullptr && cap > 0) {
        const size_t n = src.size() < cap - 1 ? src.size() : cap - 1;
        std::memcpy(buf, src.data(), n);
        buf[n] = '\0';
    }
    return ES_OK;
}

es_status es_plan_body_backward_f32(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                                    const int64_t* shape, int rank, int axis, int state_width,
                                    const int64_t* seq_widths, int reverse, const float* states,
                                    const float* grad_out, const float* grad_initial, float* const* grad_seqs,
                                    es_plan_info* info) {
    return es::plan_body_backward_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths,
                                       reverse, states, grad_out, grad_initial, grad_seqs, info, false);
}

es_status es_scan_body_backward_f32(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                                    const int64_t* shape, int rank, int axis, int state_width,
                                    const int64_t* seq_widths, int reverse, const float* states,
                                    const float* grad_out, float* grad_initial, float* const* grad_seqs,
                                    es_stream_t stream) {
    return es::scan_body_backward_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths,
                                       reverse, states, grad_out, grad_initial, grad_seqs,
                                       reinterpret_cast<cudaStream_t>(stream), false);
}

}  // extern "C"

namespace es {

es_status plan_body_backward_impl(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                                  const int64_t* shape, int rank, int axis, int state_width,
                                  const int64_t* seq_widths, int reverse, const float* states, const float* grad_out,
                                  const float* grad_initial, float* const* grad_seqs, es_plan_info* info,
                                  bool zero_initial) {
    BodyBwdCall B{};
    es_status st = plan_body_backward(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths,
                                      reverse, states, grad_out, grad_initial, grad_seqs, &B, zero_initial);
    if (st != ES_OK) return st;
    fill_info(B.C, info);
    return ES_OK;
}

es_status scan_body_backward_impl(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                                  const int64_t* shape, int rank, int axis, int state_width,
                                  const int64_t* seq_widths, int reverse, const float* states, const float* grad_out,
                                  float* grad_initial, float* const* grad_seqs, cudaStream_t stream,
                                  bool zero_initial) {
    es::BodyBwdCall B{};
    es_status st = es::plan_body_backward(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths,
                                          reverse, states, grad_out, grad_initial, grad_seqs, &B, zero_initial);
    if (st != ES_OK) return st;
    if (B.C.path == ES_PATH_EMPTY) return ES_OK;
    int dev = 0;
    es::DeviceState* ds = nullptr;
    if ((st = es::api_device(&dev, &ds)) != ES_OK) return st;
    std::string err;
    bool ok;
    const cudaStream_t s = stream;
    if (B.C.path != ES_PATH_GENERIC) {
        es::EncodeTiledFn encode = nullptr;
        if ((st = es::api_encoder(&encode)) != ES_OK) return st;
        if (B.C.path == ES_PATH_LANE_TMA)
            ok = es::launch_body_lane_bwd(B, initial, seqs, states, grad_out, grad_initial, grad_seqs, s, ds, encode,
                                          &err);
        else if (B.C.path == ES_PATH_TIME_TMA)
            ok = es::launch_body_time_bwd(B, initial, seqs, states, grad_out, grad_initial, grad_seqs, s, ds, encode,
                                          &err);
        else
            ok = es::launch_body_vec_bwd(B, initial, seqs, states, grad_out, grad_initial, grad_seqs, s, ds, encode,
                                         &err);
    } else {
        ok = es::launch_body_generic_bwd(B, initial, seqs, states, grad_out, grad_initial, grad_seqs, s, &err);
    }
    if (!ok) return es::api_fail(ES_E_CUDA, "es_scan_body_backward_f32: %s", err.c_str());
    es::count_launch();
    return ES_OK;
}

}  // namespace es

extern "C" {

uint64_t es_body_compile_count(void) { return es::jit_compile_count(); }

es_status es_plan_body_f32(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                           const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                           int reverse, const float* out, es_plan_info* info) {
    es::BodyCall C{};
    es_status st = es::plan_body(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, reverse,
                                 out, &C);
    if (st != ES_OK) return st;
    es::fill_info(C, info);
    return ES_OK;
}

es_status es_scan_body_f32(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                           const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                           int reverse, float* out, es_stream_t stream) {
    return es::scan_body_impl(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, reverse, out,
                              reinterpret_cast<cudaStream_t>(stream), false);
}

}  // extern "C"

namespace es {

es_status scan_body_impl(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                         const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                         int reverse, float* out, cudaStream_t stream, bool zero_initial) {
    es::BodyCall C{};
    es_status st = es::plan_body(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, reverse,
                                 out, &C, zero_initial);
    if (st != ES_OK) return st;
    if (C.path == ES_PATH_EMPTY) return ES_OK;
    es::BodyLaunch L{};
    L.C = &C;
    L.init = initial;
    L.seqs = seqs;
    L.out = out;
    L.stream = stream;
    int dev = 0;
    if ((st = es::api_device(&dev, &L.dev)) != ES_OK) return st;
    std::string err;
    bool ok;
    if (C.path == ES_PATH_GENERIC) {
        ok = es::launch_body_generic(L, &err);
    } else {
        if ((st = es::api_encoder(&L.encode)) != ES_OK) return st;
        if (C.path == ES_PATH_LANE_TMA) ok = es::launch_body_lane(L, &err);
        else if (C.path == ES_PATH_TIME_TMA) ok = es::launch_body_time(L, &err);
        else ok = es::launch_body_vec(L, &err);
    }
    if (!ok) return es::api_fail(ES_E_CUDA, "es_scan_body_f32: %s", err.c_str());
    es::count_launch();
    return ES_OK;
}

es_status plan_body_impl(es_body_t body, const float* initial, const float* const* seqs, int n_seqs,
                         const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                         int reverse, const float* out, es_plan_info* info, bool zero_initial) {
    es::BodyCall C{};
    es_status st = es::plan_body(body, initial, seqs, n_seqs, shape, rank, axis, state_width, seq_widths, reverse,
                                 out, &C, zero_initial);
    if (st != ES_OK) return st;
    es::fill_info(C, info);
    return ES_OK;
}

}  // namespace es
