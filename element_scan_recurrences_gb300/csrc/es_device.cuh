// es_device.cuh -- device code shared by the element-scan kernels built into
// the library: the three fixed bodies and the MAXPLUS vector-Jacobian
// product, on top of the PTX building blocks of es_ptx.cuh.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "es_internal.h"
#include "es_ptx.cuh"

namespace es {

// ---------------------------------------------------------------------------
// bodies ("Nonlinear element scans": intro, :state-axis and :reverse examples)
//
// Each body operation is one f32 operation rounded to nearest in the order the
// body is written; the _rn intrinsics keep the compiler from contracting a
// multiply and an add into one fused operation.

// h = tanh(x + a*h)
__device__ __forceinline__ float step_tanh_decay(float h, float x, float a) {
    return tanhf(__fadd_rn(x, __fmul_rn(a, h)));
}

// h = maximum(h - c, x)
__device__ __forceinline__ float step_maxplus(float h, float x, float c) {
    return ieee_maximum(__fsub_rn(h, c), x);
}

template <int BODY>
__device__ __forceinline__ float step_pointwise(float h, float x, float s) {
    if constexpr (BODY == ES_BODY_TANH_DECAY) {
        return step_tanh_decay(h, x, s);
    } else {
        return step_maxplus(h, x, s);
    }
}

// Vector-Jacobian product of one MAXPLUS trip h = maximum(v, x), v = p - c,
// for the state cotangent `lam`: the larger operand takes it, a tie (or a
// NaN) splits it evenly (the usual tie rule for maximum).  Writes dx and dc
// and leaves in `lam` the cotangent of the previous state.  Selects only, so
// lanes that take different sides do not diverge.
__device__ __forceinline__ void maxplus_vjp(float v, float xv, float& lam, float& dx, float& dc) {
    const bool to_state = v > xv;
    const bool to_x = xv > v;
    const float half = __fmul_rn(lam, 0.5f);
    const float keep = to_state ? lam : (to_x ? 0.0f : half);
    dx = to_x ? lam : (to_state ? 0.0f : half);
    dc = to_state ? -lam : (to_x ? 0.0f : -half);
    lam = keep;
}

}  // namespace es
