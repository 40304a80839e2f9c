// es_internal.h -- declarations shared by the host dispatcher (es_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "es.h"

#define ES_BODY_TANH_DECAY 0
#define ES_BODY_NORMCAP 1
#define ES_BODY_MAXPLUS 2

// bits of the per-device status word
#define ES_DEVICE_TIMEOUT 1u

namespace es {

// cuTensorMapEncodeTiled, fetched from the driver at run time
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// One validated call in canonical form: output [O, T, J, W] and sequence k
// as [O, T, J, sw[k]] (sw[k] == 1 broadcasts over the state).
struct Launch {
    int body;
    const float* init;
    const float* x;
    const float* a;
    float* out;
    int64_t O, T, J, W;
    int64_t sw[2];
    int reverse;
    unsigned int* status;   // device status word
    uint64_t wait_ns;       // bounded-wait limit
    int64_t drop_tile;      // testing hook: producers skip this tile (-1: off)
    cudaStream_t stream;
    int num_sms;
    int device;
    EncodeTiledFn encode;
};

// A backward call: the forward call's arguments plus the saved states, the
// output gradient and the gradients to produce (same canonical layouts).
struct BackwardLaunch {
    Launch fwd;
    const float* states;    // forward output [O, T, J, W]
    const float* gout;      // dL/d states    [O, T, J, W]
    float* ginit;           // dL/d initial   [O, J, W]
    float* gx;              // dL/d x         [O, T, J, sw0]
    float* ga;              // dL/d a or c    [O, T, J, sw1]
};

// Per-device state of the library: the device status word and the SM count.
struct DeviceState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    unsigned int* status = nullptr;
    int num_sms = 0;
};

// A validated call's shapes in canonical form (shared by every entry point).
struct ShapePlan {
    int64_t O, T, J, W;
    int n_seqs;
    int64_t sw[ES_MAX_SEQS];
    int64_t n_out, n_init, n_seq[ES_MAX_SEQS];
    bool empty;       // no lanes: nothing to read or write
};

// Check the arguments every scan shares ("Arguments and body": shapes, axis,
// state axis, sequence widths) and the data pointers (present, 4-byte
// aligned, `out` disjoint from every input); `names` name the sequences in
// messages.  Returns ES_OK or the status with es_last_error() set.
// `zero_initial`: the scan starts from zero and `initial` must be null.
es_status plan_shapes(const char* fn, const char* const* names, const float* initial, const float* const* seqs,
                      int n_seqs, const int64_t* shape, int rank, int axis, int state_width,
                      const int64_t* seq_widths, const float* out, ShapePlan* P, bool zero_initial = false);

// set es_last_error() and return `st`
es_status api_fail(es_status st, const char* fmt, ...);
es_status api_device(int* dev, DeviceState** st);
es_status api_encoder(EncodeTiledFn* fn);
void count_launch(int kernels = 1);
uint64_t api_wait_ns();
int64_t api_drop_tile();
int api_path_override();

// The body-program scan (es_scan_body_f32) and its plan, with an optional
// zero initial state (then `initial` is null), for operations built on it.
es_status scan_body_impl(struct es_body_program* body, const float* initial, const float* const* seqs, int n_seqs,
                         const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                         int reverse, float* out, cudaStream_t stream, bool zero_initial);
es_status plan_body_impl(struct es_body_program* body, const float* initial, const float* const* seqs, int n_seqs,
                         const int64_t* shape, int rank, int axis, int state_width, const int64_t* seq_widths,
                         int reverse, const float* out, es_plan_info* info, bool zero_initial);

// Gradients of a body-program scan (es_scan_body_backward_f32); with
// `zero_initial` the forward started from zero: `initial` and
// `grad_initial` are null.
es_status scan_body_backward_impl(struct es_body_program* body, const float* initial, const float* const* seqs, int n_seqs,
                                  const int64_t* shape, int rank, int axis, int state_width,
                                  const int64_t* seq_widths, int reverse, const float* states, const float* grad_out,
                                  float* grad_initial, float* const* grad_seqs, cudaStream_t stream,
                                  bool zero_initial);
es_status plan_body_backward_impl(struct es_body_program* body, const float* initial, const float* const* seqs, int n_seqs,
                                  const int64_t* shape, int rank, int axis, int state_width,
                                  const int64_t* seq_widths, int reverse, const float* states, const float* grad_out,
                                  const float* grad_initial, float* const* grad_seqs, es_plan_info* info,
                                  bool zero_initial);

// Each launcher enqueues exactly one kernel; it returns cudaSuccess or the
// launch error.  `err` receives a message for non-CUDA failures (tensor-map
// encoding).
cudaError_t launch_generic(const Launch& L);
cudaError_t launch_lane_tma(const Launch& L, const char** err);
cudaError_t launch_time_tma(const Launch& L, const char** err);
cudaError_t launch_vec_tma(const Launch& L, const char** err);
cudaError_t launch_generic_bwd(const BackwardLaunch& B);
cudaError_t launch_lane_tma_bwd(const BackwardLaunch& B, const char** err);
cudaError_t launch_vec_tma_bwd(const BackwardLaunch& B, const char** err);
cudaError_t launch_time_tma_bwd(const BackwardLaunch& B, const char** err);

// eligibility of the TMA paths (pure host logic, also used by planning)
bool lane_tma_ok(int body, int64_t O, int64_t T, int64_t J, int64_t W, const int64_t sw[2],
                 const void* const ptrs[4]);
bool time_tma_ok(int body, int64_t O, int64_t T, int64_t J, int64_t W, const int64_t sw[2],
                 const void* const ptrs[4]);
bool vec_tma_ok(int body, int64_t O, int64_t T, int64_t J, int64_t W, const int64_t sw[2],
                const void* const ptrs[4]);

}  // namespace es
