// k_generic.cu -- the any-layout element-scan kernel (ES_PATH_GENERIC).
//
// One thread per lane (o, j) of the canonical view [O, T, J, W]; the thread
// keeps the lane's W state values in registers and walks the trips in order
// ("Nonlinear element scans": lanes run in parallel, trips in sequence),
// reading each trip's sequence values straight from global memory.  Adjacent
// threads hold adjacent lanes, so with W == 1 every trip is one coalesced row.
// It serves shapes and alignments the TMA paths do not, and tiny problems.
// NORMCAP adds the squares in state order w = 0..W-1.
#include "es_device.cuh"

namespace es {
namespace {

template <int BODY, int WMAX>
__global__ void __launch_bounds__(128)
k_generic(const float* __restrict__ init, const float* __restrict__ x, const float* __restrict__ a,
          float* __restrict__ out, int64_t O, int64_t T, int64_t J, int W, int sx, int sa, int reverse) {
    const int64_t lane = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (lane >= O * J) return;
    const int64_t o = lane / J;
    const int64_t j = lane - o * J;

    float h[WMAX];
#pragma unroll
    for (int w = 0; w < WMAX; ++w)
        if (w < W) h[w] = init[lane * W + w];

    for (int64_t s = 0; s < T; ++s) {
        const int64_t t = reverse ? T - 1 - s : s;
        const int64_t row = (o * T + t) * J + j;
        const float* xp = x + row * sx;
        const float* ap = a + row * sa;
        float* op = out + row * W;
        if constexpr (BODY == ES_BODY_NORMCAP) {
            // y = a*h + x;  h = y / maximum(1, sqrt(sum y^2))
            float y[WMAX];
            float ss = 0.0f;
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (w < W) {
                    const float xv = __ldg(xp + (sx == 1 ? 0 : w));
                    const float av = __ldg(ap + (sa == 1 ? 0 : w));
                    y[w] = __fadd_rn(__fmul_rn(av, h[w]), xv);
                }
            }
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) ss = __fadd_rn(ss, __fmul_rn(y[w], y[w]));
            const float d = ieee_maximum(1.0f, __fsqrt_rn(ss));
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) h[w] = __fdiv_rn(y[w], d);
        } else {
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (w < W) {
                    const float xv = __ldg(xp + (sx == 1 ? 0 : w));
                    const float av = __ldg(ap + (sa == 1 ? 0 : w));
                    h[w] = step_pointwise<BODY>(h[w], xv, av);
                }
            }
        }
#pragma unroll
        for (int w = 0; w < WMAX; ++w)
            if (w < W) __stcs(op + w, h[w]);
    }
}

template <int BODY>
cudaError_t launch_body(const Launch& L) {
    const int64_t lanes = L.O * L.J;
    const int threads = 128;
    const int64_t blocks = (lanes + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int sx = static_cast<int>(L.sw[0]);
    const int sa = static_cast<int>(L.sw[1]);
    if (L.W == 1) {
        k_generic<BODY, 1><<<static_cast<unsigned>(blocks), threads, 0, L.stream>>>(
            L.init, L.x, L.a, L.out, L.O, L.T, L.J, 1, sx, sa, L.reverse);
    } else {
        k_generic<BODY, 16><<<static_cast<unsigned>(blocks), threads, 0, L.stream>>>(
            L.init, L.x, L.a, L.out, L.O, L.T, L.J, static_cast<int>(L.W), sx, sa, L.reverse);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic(const Launch& L) {
    switch (L.body) {
        case ES_BODY_TANH_DECAY: return launch_body<ES_BODY_TANH_DECAY>(L);
        case ES_BODY_NORMCAP: return launch_body<ES_BODY_NORMCAP>(L);
        default: return launch_body<ES_BODY_MAXPLUS>(L);
    }
}

}  // namespace es

// ---------------------------------------------------------------------------
// Backward pass, any layout ("Precision and gradients": the gradient of a scan
// is another scan in the opposite trip order applying the body's
// vector-Jacobian product once a trip).  One thread per lane walks the trips
// in reverse scan order carrying the state's cotangent `lam`; the operations
// and their order are those of the plain definition, so the result is exact
// against a sequential CPU loop: TANH_DECAY and MAXPLUS use no transcendental,
// NORMCAP's correctly rounded sqrt and division are IEEE operations.  A
// width-one sequence receives the sum over the state, added in state order.
namespace es {
namespace {

template <int BODY, int WMAX>
__global__ void __launch_bounds__(128)
k_generic_bwd(const float* __restrict__ init, const float* __restrict__ x, const float* __restrict__ a,
              const float* __restrict__ states, const float* __restrict__ gout, float* __restrict__ ginit,
              float* __restrict__ gx, float* __restrict__ ga, int64_t O, int64_t T, int64_t J, int W, int sx, int sa,
              int reverse) {
    const int64_t lane = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (lane >= O * J) return;
    const int64_t o = lane / J;
    const int64_t j = lane - o * J;
    float lam[WMAX], h[WMAX], p[WMAX];
#pragma unroll
    for (int w = 0; w < WMAX; ++w) {
        lam[w] = 0.0f;
        if (w < W) h[w] = states[((o * T + (reverse ? 0 : T - 1)) * J + j) * W + w];
    }
    for (int64_t s = T - 1; s >= 0; --s) {
        const int64_t t = reverse ? T - 1 - s : s;
        const int64_t row = (o * T + t) * J + j;
        // the state before this trip: initial for the first trip in scan order
        if (s == 0) {
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) p[w] = init[lane * W + w];
        } else {
            const int64_t tp = reverse ? t + 1 : t - 1;
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) p[w] = states[((o * T + tp) * J + j) * W + w];
        }
#pragma unroll
        for (int w = 0; w < WMAX; ++w)
            if (w < W) lam[w] = __fadd_rn(lam[w], gout[row * W + w]);
        const float* xp = x + row * sx;
        const float* ap = a + row * sa;
        float dx[WMAX], da[WMAX];
        if constexpr (BODY == ES_BODY_TANH_DECAY) {
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (w < W) {
                    const float av = ap[sa == 1 ? 0 : w];
                    const float m = __fmul_rn(lam[w], __fsub_rn(1.0f, __fmul_rn(h[w], h[w])));
                    dx[w] = m;
                    da[w] = __fmul_rn(m, p[w]);
                    lam[w] = __fmul_rn(m, av);
                }
            }
        } else if constexpr (BODY == ES_BODY_MAXPLUS) {
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (w < W) {
                    const float v = __fsub_rn(p[w], ap[sa == 1 ? 0 : w]);
                    const float xv = xp[sx == 1 ? 0 : w];
                    maxplus_vjp(v, xv, lam[w], dx[w], da[w]);
                }
            }
        } else {
            float y[WMAX], mu[WMAX];
            float ss = 0.0f;
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) y[w] = __fadd_rn(__fmul_rn(ap[sa == 1 ? 0 : w], p[w]), xp[sx == 1 ? 0 : w]);
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) ss = __fadd_rn(ss, __fmul_rn(y[w], y[w]));
            const float nrm = __fsqrt_rn(ss);
            if (nrm <= 1.0f) {
#pragma unroll
                for (int w = 0; w < WMAX; ++w)
                    if (w < W) mu[w] = lam[w];
            } else {
                float hl = 0.0f;
#pragma unroll
                for (int w = 0; w < WMAX; ++w)
                    if (w < W) hl = __fadd_rn(hl, __fmul_rn(h[w], lam[w]));
#pragma unroll
                for (int w = 0; w < WMAX; ++w)
                    if (w < W) mu[w] = __fdiv_rn(__fsub_rn(lam[w], __fmul_rn(h[w], hl)), nrm);
            }
#pragma unroll
            for (int w = 0; w < WMAX; ++w) {
                if (w < W) {
                    dx[w] = mu[w];
                    da[w] = __fmul_rn(mu[w], p[w]);
                    lam[w] = __fmul_rn(ap[sa == 1 ? 0 : w], mu[w]);
                }
            }
        }
        if (sx == 1 && W > 1) {
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) acc = __fadd_rn(acc, dx[w]);
            gx[row] = acc;
        } else {
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) gx[row * sx + w] = dx[w];
        }
        if (sa == 1 && W > 1) {
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) acc = __fadd_rn(acc, da[w]);
            ga[row] = acc;
        } else {
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (w < W) ga[row * sa + w] = da[w];
        }
        // the state before this trip is the output of the next one visited
#pragma unroll
        for (int w = 0; w < WMAX; ++w)
            if (w < W) h[w] = p[w];
    }
#pragma unroll
    for (int w = 0; w < WMAX; ++w)
        if (w < W) ginit[lane * W + w] = lam[w];
}

template <int BODY>
cudaError_t launch_bwd_body(const BackwardLaunch& B) {
    const Launch& L = B.fwd;
    const int64_t lanes = L.O * L.J;
    const int threads = 128;
    const int64_t blocks = (lanes + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int sx = static_cast<int>(L.sw[0]);
    const int sa = static_cast<int>(L.sw[1]);
    if (L.W == 1) {
        k_generic_bwd<BODY, 1><<<static_cast<unsigned>(blocks), threads, 0, L.stream>>>(
            L.init, L.x, L.a, B.states, B.gout, B.ginit, B.gx, B.ga, L.O, L.T, L.J, 1, sx, sa, L.reverse);
    } else {
        k_generic_bwd<BODY, 16><<<static_cast<unsigned>(blocks), threads, 0, L.stream>>>(
            L.init, L.x, L.a, B.states, B.gout, B.ginit, B.gx, B.ga, L.O, L.T, L.J, static_cast<int>(L.W), sx, sa,
            L.reverse);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic_bwd(const BackwardLaunch& B) {
    switch (B.fwd.body) {
        case ES_BODY_TANH_DECAY: return launch_bwd_body<ES_BODY_TANH_DECAY>(B);
        case ES_BODY_NORMCAP: return launch_bwd_body<ES_BODY_NORMCAP>(B);
        default: return launch_bwd_body<ES_BODY_MAXPLUS>(B);
    }
}

}  // namespace es
