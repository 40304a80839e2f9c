// skel_lane.cuh -- body-program skeleton with the lanes innermost.
//
// Canonical view [O, T, I] (scalar state, I contiguous lanes per trip row).
// One CTA owns LI adjacent lanes of one o and walks all T trips:
//   * warp 0, lane 0 is the producer: it streams time tiles of TT trips of
//     every sequence (box {LI, TT, 1} of a 3-D tensor map per sequence) into
//     an S-stage SMEM ring with TMA, each stage guarded by a full / empty
//     mbarrier pair;
//   * LI consumer threads (one per lane) copy a whole tile into registers,
//     hand the stage back at once, then run the body over the tile with the
//     state in a register: one coalesced 4*LI-byte store per trip and warp.
// Reverse scans walk the tiles from last to first and each tile bottom-up
// (no flipped copy).  A ragged last tile is zero-filled by TMA and only its
// valid rows are used.  Every wait is bounded: on give-up the CTA records
// ES_DEVICE_TIMEOUT, the producer waits (bounded) for its copies in flight,
// and all threads return.
#pragma once

#include "skel_common.cuh"

namespace es {

constexpr int kLaneMaxStages = 8;

template <class Body, int LI, int TT>
__global__ void __launch_bounds__(32 + LI)
k_body_lane(const __grid_constant__ TmaMaps<Body::kNS> maps, const float* __restrict__ init,
            float* __restrict__ out, int T, int I, int tiles_i, int stages, int reverse, unsigned int* status,
            uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    static_assert(Body::kWideMask == (1u << NS) - 1u, "a scalar state has no width-one sequences");
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kLaneMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kLaneMaxStages];
    __shared__ int abort_flag;

    float* tiles = reinterpret_cast<float*>(smem_raw + smem_align_pad(smem_raw));
    constexpr int kTileFloats = TT * LI;            // one sequence, one stage
    constexpr uint32_t kStageBytes = NS * kTileFloats * 4u;

    const int o = blockIdx.x / tiles_i;
    const int i0 = (blockIdx.x % tiles_i) * LI;
    const int ntiles = (T + TT - 1) / TT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], LI / 32);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            for (int q = 0; q < NS; ++q) tma_prefetch_desc(&maps.m[q]);
            const uint64_t pol = l2_policy_stream();
            int issued = 0;
            for (int k = 0; k < ntiles; ++k) {
                const int s = k % stages;
                const int round = k / stages;
                if (round > 0 && !mbar_wait_bounded(&empty_bar[s], (round - 1) & 1, wait_ns, &abort_flag)) {
                    report_timeout(status, &abort_flag);
                    break;
                }
                issued = k + 1;
                if (k == drop_tile) continue;   // testing hook: this tile never arrives
                const int j = reverse ? ntiles - 1 - k : k;
                float* st = tiles + s * NS * kTileFloats;
                mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    tma_load_3d(st + q * kTileFloats, &maps.m[q], i0, j * TT, o, &full_bar[s], pol);
            }
            // no copy may still target SMEM when the CTA exits
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    // consumers: one lane each
    const int c = threadIdx.x - 32;
    const int i = i0 + c;
    const bool valid = i < I;
    float h = valid && init != nullptr ? init[static_cast<int64_t>(o) * I + i] : 0.0f;   // null: from zero
    float* obase = out + static_cast<int64_t>(o) * T * I + i;

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        // the whole warp leaves together, so __syncwarp never misses a lane
        if (!__all_sync(0xffffffffu, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int j = reverse ? ntiles - 1 - k : k;
        const int t0 = j * TT;
        const int n = min(TT, T - t0);          // < TT only for the last time tile
        const float* st = tiles + s * NS * kTileFloats + c;
        // the whole tile goes to registers first: the loads overlap each other
        // and the serial chain below only waits on arithmetic
        float vr[NS][TT];
#pragma unroll
        for (int q = 0; q < NS; ++q)
#pragma unroll
            for (int tt = 0; tt < TT; ++tt) vr[q][tt] = st[q * kTileFloats + tt * LI];
        // the stage is free as soon as the tile sits in registers
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        float* op = obase + static_cast<int64_t>(t0) * I;
        // The state alternates between two registers (by trip parity), so a
        // trip never overwrites the register the previous trip's store may
        // still be reading.
        float hv[2] = {h, h};
        auto trip = [&](const int tt) {
            float r[1];
            const float hp[1] = {hv[(tt & 1) ^ 1]};
            float sw[Body::kSW][1];
            const float sn[Body::kSN] = {};
#pragma unroll
            for (int q = 0; q < NS; ++q) sw[q][0] = vr[q][tt];
            Body::template step<1, 1>(r, hp, sw, sn, 0xffffffffu);
            hv[tt & 1] = r[0];
            if (valid) __stcs(op + static_cast<int64_t>(tt) * I, r[0]);
        };
        // full tiles run unguarded (one basic block, so consecutive trips
        // overlap); only the ragged last tile checks every trip
        if (n == TT) {
            if (!reverse) {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) trip(tt);
            } else {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt) trip(tt);
            }
        } else {
            if (!reverse) {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    if (tt < n) trip(tt);
            } else {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt)
                    if (tt < n) trip(tt);
            }
        }
        h = reverse ? hv[0] : hv[(n - 1) & 1];
    }
}

}  // namespace es
