// skel_generic.cuh -- the any-layout skeleton for body programs.
//
// One thread per lane (o, j) of the canonical view [O, T, J, W] holds the
// lane's whole state (W values, so a `sum` adds w = 0..W-1 in order) and
// walks the trips in order ("Nonlinear element scans": lanes in parallel,
// trips in sequence), loading each trip's sequence values straight from
// global memory one trip ahead of its use.  It serves every shape and
// alignment, and tiny problems.
#pragma once

#include "skel_common.cuh"

namespace es {

template <class Body, int W>
__global__ void __launch_bounds__(128)
k_body_generic(const SeqPtrs seqs, const float* __restrict__ init, float* __restrict__ out, int64_t O, int64_t T,
               int64_t J, int reverse) {
    constexpr int NS = Body::kNS;
    const int64_t lane = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (lane >= O * J) return;
    const int64_t o = lane / J;
    const int64_t j = lane - o * J;

    float h[W];
#pragma unroll
    for (int w = 0; w < W; ++w) h[w] = init != nullptr ? init[lane * W + w] : 0.0f;   // null: from zero

    float sw[Body::kSW][W];
    float sn[Body::kSN];
    auto load = [&](int64_t t, float (&dw)[Body::kSW][W], float (&dn)[Body::kSN]) {
        const int64_t row = (o * T + t) * J + j;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            if (is_wide(Body::kWideMask, k)) {
#pragma unroll
                for (int w = 0; w < W; ++w) dw[wide_slot(Body::kWideMask, k)][w] = __ldg(seqs.p[k] + row * W + w);
            } else {
                dn[narrow_slot(Body::kWideMask, k)] = __ldg(seqs.p[k] + row);
            }
        }
    };
    load(reverse ? T - 1 : 0, sw, sn);
    for (int64_t s = 0; s < T; ++s) {
        const int64_t t = reverse ? T - 1 - s : s;
        float nw[Body::kSW][W];
        float nn[Body::kSN];
        // the next trip's values (the last trip reloads its own: in bounds)
        const int64_t tn = s + 1 < T ? (reverse ? t - 1 : t + 1) : t;
        load(tn, nw, nn);
        float r[W];
        Body::template step<W, 1>(r, h, sw, sn, 0xffffffffu);
        float* op = out + ((o * T + t) * J + j) * W;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            h[w] = r[w];
            __stcs(op + w, r[w]);
        }
#pragma unroll
        for (int q = 0; q < Body::kSW; ++q)
#pragma unroll
            for (int w = 0; w < W; ++w) sw[q][w] = nw[q][w];
#pragma unroll
        for (int q = 0; q < Body::kSN; ++q) sn[q] = nn[q];
    }
}

}  // namespace es
