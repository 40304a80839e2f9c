// skel_generic_bwd.cuh -- the backward skeleton for body programs.
//
// "Nonlinear element scans", "Precision and gradients": the gradient of an
// element scan is another element scan over the same lanes, in the opposite
// trip order, applying the body's vector-Jacobian product once a trip.  One
// thread per lane (o, j) of the canonical view [O, T, J, W] carries the
// state's cotangent lam (W values).  At trip t it adds the output gradient of
// t to lam, takes the state before the trip (the saved state of the previous
// trip in scan order, or `init` at the first), evaluates the body's `vjp`
// there, writes the sequences' cotangents of trip t and carries the previous
// state's cotangent on.  After the last trip lam is the gradient of `init`.
// A forward scan's gradient walks t = T-1 .. 0, a reverse scan's t = 0 ..
// T-1.  One thread holds the whole state (G = 1), so the sums over the state
// run w = 0..W-1 in order.  Only the sequences the VJP reads are loaded, and
// the trip's result comes from the saved states where the VJP reads it.
// Loads for the next trip are issued one trip ahead when the registers
// allow.
#pragma once

#include "skel_common.cuh"

namespace es {

template <class Body, int W>
__global__ void __launch_bounds__(128)
k_body_generic_bwd(const SeqPtrs seqs, const float* __restrict__ init, const float* __restrict__ states,
                   const float* __restrict__ gout, const GradPtrs gseqs, float* __restrict__ ginit, int64_t O,
                   int64_t T, int64_t J, int reverse) {
    constexpr int NS = Body::kNS;
    constexpr int kSW = Body::kSW, kSN = Body::kSN;
    // one trip ahead while a trip's loads take at most 64 registers
    constexpr bool kAhead = W * (kSW + 3) + kSN <= 64;
    const int64_t lane = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (lane >= O * J) return;
    const int64_t o = lane / J;
    const int64_t j = lane - o * J;

    struct Trip {
        float sw[kSW][W];
        float sn[kSN];
        float p[W];    // the state before the trip
        float res[W];  // the trip's result (its saved state)
        float g[W];    // the output gradient of the trip
    };
    auto load = [&](int64_t t, Trip& d) {
        const int64_t row = (o * T + t) * J + j;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            if (!is_live(Body::kVjpSeqs, k)) {
                if (is_wide(Body::kWideMask, k)) {
#pragma unroll
                    for (int w = 0; w < W; ++w) d.sw[wide_slot(Body::kWideMask, k)][w] = 0.0f;
                } else {
                    d.sn[narrow_slot(Body::kWideMask, k)] = 0.0f;
                }
            } else if (is_wide(Body::kWideMask, k)) {
#pragma unroll
                for (int w = 0; w < W; ++w) d.sw[wide_slot(Body::kWideMask, k)][w] = __ldg(seqs.p[k] + row * W + w);
            } else {
                d.sn[narrow_slot(Body::kWideMask, k)] = __ldg(seqs.p[k] + row);
            }
        }
        const int64_t tp = reverse ? t + 1 : t - 1;
        const bool first = tp < 0 || tp >= T;
        const int64_t prow = (o * T + tp) * J + j;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            d.p[w] = first ? (init != nullptr ? __ldg(init + lane * W + w) : 0.0f) : __ldg(states + prow * W + w);
            d.res[w] = Body::kVjpRes ? __ldg(states + row * W + w) : 0.0f;
            d.g[w] = __ldcs(gout + row * W + w);
        }
    };

    float lam[W];
#pragma unroll
    for (int w = 0; w < W; ++w) lam[w] = 0.0f;
    Trip cur;
    load(reverse ? 0 : T - 1, cur);
    for (int64_t s = 0; s < T; ++s) {
        const int64_t t = reverse ? s : T - 1 - s;
        Trip nxt;
        if constexpr (kAhead) {
            // the next trip's values (the last trip reloads its own: in bounds)
            const int64_t tn = s + 1 < T ? (reverse ? t + 1 : t - 1) : t;
            load(tn, nxt);
        }
#pragma unroll
        for (int w = 0; w < W; ++w) lam[w] = __fadd_rn(lam[w], cur.g[w]);
        float dp[W];
        float dsw[kSW][W];
        float dsn[kSN];
        Body::template vjp<W, 1>(dp, dsw, dsn, lam, cur.p, cur.res, cur.sw, cur.sn, 0xffffffffu);
        const int64_t row = (o * T + t) * J + j;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            if (is_wide(Body::kWideMask, k)) {
#pragma unroll
                for (int w = 0; w < W; ++w) __stcs(gseqs.p[k] + row * W + w, dsw[wide_slot(Body::kWideMask, k)][w]);
            } else {
                __stcs(gseqs.p[k] + row, dsn[narrow_slot(Body::kWideMask, k)]);
            }
        }
#pragma unroll
        for (int w = 0; w < W; ++w) lam[w] = dp[w];
        if constexpr (kAhead) {
            cur = nxt;
        } else if (s + 1 < T) {
            load(reverse ? t + 1 : t - 1, cur);
        }
    }
    if (ginit != nullptr) {   // null: the scan started from zero and wants no initial gradient
#pragma unroll
        for (int w = 0; w < W; ++w) ginit[lane * W + w] = lam[w];
    }
}

}  // namespace es
