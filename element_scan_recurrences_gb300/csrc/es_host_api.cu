// es_host_api.cu -- end-to-end entry points on host buffers: the inputs are
// copied into caller-owned device buffers, scanned, and the states copied
// back, in pieces that overlap.
//
// Lanes are independent ("Storage and execution": lanes run in parallel,
// trips in sequence), so a call whose sequence axis is not the first splits
// along its first dimension into row chunks, each a complete smaller scan.
// Three library-owned streams per device then pipeline the chunks: chunk k's
// host-to-device copies, chunk k-1's scan and chunk k-2's device-to-host copy
// run at the same time (the link carries both directions at once).  The call
// is ordered after earlier work on the caller's stream, and later work there
// waits for it, through events; nothing is allocated per call.
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "es.h"
#include "es_internal.h"

namespace es {
namespace {

constexpr int kMaxChunks = 64;
constexpr int kDefaultChunks = 8;
constexpr int kHostDevices = 64;

// per device: the pipeline's streams and events, created on first use
struct HostPipe {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr, tail_in = nullptr, tail_comp = nullptr;
    cudaEvent_t loaded[kMaxChunks] = {};
    cudaEvent_t scanned[kMaxChunks] = {};
    std::mutex mu;       // one call at a time uses the pipeline
};
HostPipe g_pipes[kHostDevices];

cudaError_t pipe_init(HostPipe* p) {
    cudaError_t e = cudaSuccess;
    for (cudaStream_t* s : {&p->in, &p->comp, &p->out})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&p->start, &p->end, &p->tail_in, &p->tail_comp})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int k = 0; k < kMaxChunks && e == cudaSuccess; ++k) {
        e = cudaEventCreateWithFlags(&p->loaded[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->scanned[k], cudaEventDisableTiming);
    }
    return e;
}

// one chunk's scan on the compute stream: device pointers already offset,
// the shape with its first dimension cut to the chunk's rows
using ChunkScan = std::function<es_status(const float* init, const float* const* seqs, const int64_t* shape,
                                          float* out, cudaStream_t stream)>;

es_status host_pipeline(const char* fn, const float* initial_h, const float* const* seqs_h, int n_seqs,
                        const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                        float* out_h, float* initial_d, float* const* seqs_d, float* out_d, int chunks,
                        cudaStream_t stream, const ChunkScan& scan) {
    if (initial_h == nullptr || seqs_h == nullptr || out_h == nullptr)
        return api_fail(ES_E_ARG, "%s: null host pointer", fn);
    for (int k = 0; k < n_seqs; ++k)
        if (seqs_h[k] == nullptr) return api_fail(ES_E_ARG, "%s: null host pointer", fn);
    if (chunks < 0 || chunks > kMaxChunks) return api_fail(ES_E_ARG, "%s: chunks %d outside 0..%d", fn, chunks, kMaxChunks);
    // the whole call's shapes (validated by the device scan's planner first)
    const int ax = axis < 0 ? axis + rank : axis;
    ShapePlan S{};
    static const char* const kNames[ES_MAX_SEQS] = {"seq 0", "seq 1", "seq 2", "seq 3",
                                                    "seq 4", "seq 5", "seq 6", "seq 7"};
    es_status st = plan_shapes(fn, kNames, initial_d, seqs_d, n_seqs, shape, rank, axis, state_width, seq_widths,
                               out_d, &S);
    if (st != ES_OK) return st;
    if (S.empty) return ES_OK;
    // rows of the first dimension and the elements of one row of each buffer
    const bool split = ax > 0;
    const int64_t rows = split ? shape[0] : 1;
    int n = chunks == 0 ? kDefaultChunks : chunks;
    if (n > rows) n = static_cast<int>(rows);
    if (n < 1) n = 1;
    const int64_t out_row = S.n_out / rows, init_row = S.n_init / rows;
    int64_t seq_row[ES_MAX_SEQS];
    for (int k = 0; k < n_seqs; ++k) seq_row[k] = S.n_seq[k] / rows;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostDevices)
        return api_fail(ES_E_CUDA, "%s: no usable CUDA device", fn);
    HostPipe* p = &g_pipes[dev];
    std::call_once(p->once, [p]() { p->err = pipe_init(p); });
    if (p->err != cudaSuccess) return api_fail(ES_E_CUDA, "%s: %s", fn, cudaGetErrorString(p->err));
    std::lock_guard<std::mutex> lock(p->mu);

    auto check = [&](cudaError_t e) -> es_status {
        return e == cudaSuccess ? ES_OK : api_fail(ES_E_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    };
    // after the caller's earlier work
    if ((st = check(cudaEventRecord(p->start, stream))) != ES_OK) return st;
    for (cudaStream_t s : {p->in, p->comp, p->out})
        if ((st = check(cudaStreamWaitEvent(s, p->start, 0))) != ES_OK) return st;

    std::vector<int64_t> sub(shape, shape + rank);
    int64_t r0 = 0;
    for (int c = 0; c < n; ++c) {
        const int64_t r1 = rows * (c + 1) / n;
        const int64_t nr = r1 - r0;
        // copies in: one cudaMemcpyAsync per buffer
        st = check(cudaMemcpyAsync(initial_d + r0 * init_row, initial_h + r0 * init_row,
                                   static_cast<size_t>(nr * init_row) * 4, cudaMemcpyHostToDevice, p->in));
        for (int k = 0; k < n_seqs && st == ES_OK; ++k)
            st = check(cudaMemcpyAsync(seqs_d[k] + r0 * seq_row[k], seqs_h[k] + r0 * seq_row[k],
                                       static_cast<size_t>(nr * seq_row[k]) * 4, cudaMemcpyHostToDevice, p->in));
        if (st == ES_OK) st = check(cudaEventRecord(p->loaded[c], p->in));
        // the chunk's scan
        if (st == ES_OK) st = check(cudaStreamWaitEvent(p->comp, p->loaded[c], 0));
        if (st == ES_OK) {
            const float* sp[ES_MAX_SEQS];
            for (int k = 0; k < n_seqs; ++k) sp[k] = seqs_d[k] + r0 * seq_row[k];
            if (split) sub[0] = nr;
            st = scan(initial_d + r0 * init_row, sp, sub.data(), out_d + r0 * out_row, p->comp);
        }
        if (st == ES_OK) st = check(cudaEventRecord(p->scanned[c], p->comp));
        // the copy out
        if (st == ES_OK) st = check(cudaStreamWaitEvent(p->out, p->scanned[c], 0));
        if (st == ES_OK)
            st = check(cudaMemcpyAsync(out_h + r0 * out_row, out_d + r0 * out_row,
                                       static_cast<size_t>(nr * out_row) * 4, cudaMemcpyDeviceToHost, p->out));
        if (st != ES_OK) break;
        r0 = r1;
    }
    // later work on the caller's stream waits for all three streams (also
    // after a failure, so that no enqueued piece outlives the call's order)
    es_status st2 = check(cudaEventRecord(p->tail_in, p->in));
    if (st2 == ES_OK) st2 = check(cudaEventRecord(p->tail_comp, p->comp));
    if (st2 == ES_OK) st2 = check(cudaStreamWaitEvent(p->out, p->tail_in, 0));
    if (st2 == ES_OK) st2 = check(cudaStreamWaitEvent(p->out, p->tail_comp, 0));
    if (st2 == ES_OK) st2 = check(cudaEventRecord(p->end, p->out));
    if (st2 == ES_OK) st2 = check(cudaStreamWaitEvent(stream, p->end, 0));
    return st != ES_OK ? st : st2;
}

}  // namespace
}  // namespace es

extern "C" {

es_status es_scan_host_f32(es_body body, const float* initial_h, const float* const* seqs_h, int n_seqs,
                           const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                           int reverse, float* out_h, float* initial_d, float* const* seqs_d, float* out_d,
                           int chunks, es_stream_t stream) {
    const int sw = state_width;
    auto scan = [&](const float* init, const float* const* seqs, const int64_t* shp, float* out,
                    cudaStream_t s) -> es_status {
        return es_scan_f32(body, init, seqs, n_seqs, shp, rank, axis, sw, seq_widths, reverse, out,
                           reinterpret_cast<es_stream_t>(s));
    };
    return es::host_pipeline("es_scan_host_f32", initial_h, seqs_h, n_seqs, shape, rank, axis, state_width,
                             seq_widths, out_h, initial_d, seqs_d, out_d, chunks,
                             reinterpret_cast<cudaStream_t>(stream), scan);
}

es_status es_scan_body_host_f32(es_body_t body, const float* initial_h, const float* const* seqs_h, int n_seqs,
                                const int64_t* shape, int rank, int axis, int state_width,
                                const int64_t* seq_widths, int reverse, float* out_h, float* initial_d,
                                float* const* seqs_d, float* out_d, int chunks, es_stream_t stream) {
    if (body == nullptr) return es::api_fail(ES_E_ARG, "es_scan_body_host_f32: null body program");
    auto scan = [&](const float* init, const float* const* seqs, const int64_t* shp, float* out,
                    cudaStream_t s) -> es_status {
        return es_scan_body_f32(body, init, seqs, n_seqs, shp, rank, axis, state_width, seq_widths, reverse, out,
                                reinterpret_cast<es_stream_t>(s));
    };
    return es::host_pipeline("es_scan_body_host_f32", initial_h, seqs_h, n_seqs, shape, rank, axis, state_width,
                             seq_widths, out_h, initial_d, seqs_d, out_d, chunks,
                             reinterpret_cast<cudaStream_t>(stream), scan);
}

}  // extern "C"
