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

// `sum` over a lane's state: this thread's E values in order, then a
// butterfly over the lane's G threads.  Every thread of the group ends with
// the same bits (each level adds the same two operands).  With G = 1 the
// order is w = 0..W-1.
template <int E, int G>
__device__ __forceinline__ float group_sum(const float (&v)[E], unsigned mask) {
    float s = v[0];
#pragma unroll
    for (int e = 1; e < E; ++e) s = __fadd_rn(s, v[e]);
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(mask, s, off));
    return s;
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
