// skel_common.cuh -- what every body-program kernel skeleton shares.
//
// A body program ("Nonlinear element scans", "Arguments and body": a body
// made of pointwise arithmetic, transcendental functions, comparisons,
// `where`, constants, booleans and casts; with `:state-axis` also `sum` and
// `max` over the state) is translated on the host into a functor type
//
//   struct Body {
//       static constexpr int kNS;            // sequences after the state
//       static constexpr unsigned kWideMask; // bit k: sequence k is as wide
//                                            // as the state (else width one)
//       static constexpr int kSW, kSN;       // array extents (>= 1) for the
//                                            // wide and the width-one ones
//       template <int E, int G>
//       static void step(float (&r)[E], const float (&h)[E],
//                        const float (&sw)[kSW][E], const float (&sn)[kSN],
//                        unsigned mask);
//   };
//
// A lane's state of W values is held by G threads with E = W / G values each
// (G = 1: one thread holds the whole state).  `sw` holds this thread's E
// values of each wide sequence in order, `sn` each width-one sequence's
// value; `mask` names the warp's active threads for the reductions, which
// combine a lane's G threads with xor shuffles.  The skeletons (generic,
// lanes innermost, time innermost, vector state) stream the sequences and
// call `step` once a trip; they are compiled with the functor at run time.
#pragma once

#include "es_ptx.cuh"

namespace es {

constexpr int kMaxBodySeqs = 8;

// sequence base pointers of a plain-load launch
struct SeqPtrs {
    const float* p[kMaxBodySeqs];
};

// gradient outputs of a backward launch, one per sequence
struct GradPtrs {
    float* p[kMaxBodySeqs];
};

// one TMA descriptor per sequence, passed by value (__grid_constant__)
template <int NS>
struct TmaMaps {
    CUtensorMap m[NS];
};

// position of sequence k among the wide (or the width-one) sequences
__host__ __device__ constexpr int wide_slot(unsigned wide_mask, int k) {
    int n = 0;
    for (int q = 0; q < k; ++q) n += (wide_mask >> q) & 1u;
    return n;
}
__host__ __device__ constexpr int narrow_slot(unsigned wide_mask, int k) { return k - wide_slot(wide_mask, k); }
__host__ __device__ constexpr bool is_wide(unsigned wide_mask, int k) { return ((wide_mask >> k) & 1u) != 0; }

// the sequences a backward kernel streams (those the body's vector-Jacobian
// product reads): their number, and sequence k's place among them
__host__ __device__ constexpr int live_count(unsigned live_mask, int ns) {
    int n = 0;
    for (int q = 0; q < ns; ++q) n += (live_mask >> q) & 1u;
    return n;
}
__host__ __device__ constexpr int live_slot(unsigned live_mask, int k) { return live_count(live_mask, k); }
__host__ __device__ constexpr bool is_live(unsigned live_mask, int k) { return ((live_mask >> k) & 1u) != 0; }

// threads of a block that may call group_sum with G >= 8 (the vector-state
// skeletons launch at most 192)
constexpr int kGroupSumThreads = 256;

// `sum` over a lane's state: this thread's E values in order, then over the
// lane's G threads.  With G >= 8 the partials meet in shared memory and
// every thread adds its group's G partials as one pairwise tree (the same
// order in all of them): a store and one 16-byte read per four partials
// instead of log2(G) dependent shuffles on the chain; with G = 2 or 4 a
// butterfly.  Every thread of the group ends with the same bits.  With G = 1
// the order is w = 0..W-1.
template <int E, int G>
__device__ __forceinline__ float group_sum(const float (&v)[E], unsigned mask) {
    float s = v[0];
#pragma unroll
    for (int e = 1; e < E; ++e) s = __fadd_rn(s, v[e]);
    if constexpr (G >= 8) {
        __shared__ __align__(16) float partial[kGroupSumThreads];
        const int tid = threadIdx.x;
        __syncwarp(mask);            // the group's reads of the previous call are done
        partial[tid] = s;
        __syncwarp(mask);
        const float4* g4 = reinterpret_cast<const float4*>(partial + (tid & ~(G - 1)));
        float p[G];
#pragma unroll
        for (int q = 0; q < G / 4; ++q) {
            const float4 w = g4[q];
            p[4 * q] = w.x;
            p[4 * q + 1] = w.y;
            p[4 * q + 2] = w.z;
            p[4 * q + 3] = w.w;
        }
#pragma unroll
        for (int span = 1; span < G; span *= 2)
#pragma unroll
            for (int q = 0; q < G; q += 2 * span) p[q] = __fadd_rn(p[q], p[q + span]);
        return p[0];
    } else {
#pragma unroll
        for (int off = G / 2; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(mask, s, off));
        return s;
    }
}

// `max` over a lane's state (IEEE maximum: exact, so the order is free)
template <int E, int G>
__device__ __forceinline__ float group_max(const float (&v)[E], unsigned mask) {
    float s = v[0];
#pragma unroll
    for (int e = 1; e < E; ++e) s = ieee_maximum(s, v[e]);
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) s = ieee_maximum(s, __shfl_xor_sync(mask, s, off));
    return s;
}

}  // namespace es
