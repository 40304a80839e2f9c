// skel_vec.cuh -- body-program skeleton for a vector state of W = 2, 4, 8 or
// 16 values ("Nonlinear element scans", `:state-axis`).
//
// Canonical view: the output and every full-width sequence are [O, T, J*W],
// a width-one sequence is [O, T, J].  One CTA owns LV = 128 / W adjacent
// lanes of one o (128 contiguous values per trip) and walks all T trips.
// Warp 0's lane 0 streams time tiles of TT trips of every sequence (box
// {128, TT} of a full-width sequence, {LV, TT} of a width-one one) into an
// S-stage SMEM ring with TMA, each stage guarded by a full / empty mbarrier
// pair.  Each of the 128 / E consumer threads holds E consecutive values of
// one lane's state; a lane is G = W / E threads, and the body's reductions
// combine them with xor shuffles.  A consumer reads a trip's operands from
// SMEM one trip ahead of its use, runs the body, and stores its E values with
// one vector store (a coalesced 512-byte row per trip and CTA); the stage goes
// back to the producer after the tile.  Waits are bounded as in the other
// pipelines.
#pragma once

#include "skel_common.cuh"

namespace es {

constexpr int kVecRow = 128;        // state values per CTA per trip
constexpr int kVecMaxStages = 8;

template <int E>
__device__ __forceinline__ void vec_load(float (&d)[E], const float* p) {
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int i = 0; i < E; i += 4) {
            const float4 t = *reinterpret_cast<const float4*>(p + i);
            d[i] = t.x;
            d[i + 1] = t.y;
            d[i + 2] = t.z;
            d[i + 3] = t.w;
        }
    } else if constexpr (E == 2) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        d[0] = t.x;
        d[1] = t.y;
    } else {
        d[0] = p[0];
    }
}

template <int E>
__device__ __forceinline__ void vec_store(float* p, const float (&v)[E]) {
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int i = 0; i < E; i += 4)
            __stcs(reinterpret_cast<float4*>(p + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
    } else if constexpr (E == 2) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
    } else {
        __stcs(p, v[0]);
    }
}

template <class Body, int W, int E, int TT>
__global__ void __launch_bounds__(32 + kVecRow / E)
k_body_vec(const __grid_constant__ TmaMaps<Body::kNS> maps, const float* __restrict__ init, float* __restrict__ out,
           int T, int J, int tiles_j, int stages, int reverse, unsigned int* status, uint64_t wait_ns,
           int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    constexpr unsigned kWide = Body::kWideMask;
    constexpr int LV = kVecRow / W;                // lanes per CTA
    constexpr int NC = kVecRow / E;                // consumer threads
    constexpr int G = W / E;                       // threads per lane
    constexpr unsigned kMask = NC >= 32 ? 0xffffffffu : ((1u << NC) - 1u);
    constexpr uint32_t kWideBytes = TT * kVecRow * 4u;
    constexpr uint32_t kNarrowBytes = TT * LV * 4u;   // a multiple of 128 bytes
    // byte offset of sequence q's tile inside a stage, and the stage size
    auto tile_off = [](int q) -> uint32_t {
        uint32_t off = 0;
        for (int k = 0; k < q; ++k) off += is_wide(kWide, k) ? kWideBytes : kNarrowBytes;
        return off;
    };
    const uint32_t stage_bytes = tile_off(NS);

    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kVecMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kVecMaxStages];
    __shared__ int abort_flag;
    unsigned char* base = smem_raw + smem_align_pad(smem_raw);

    const int o = blockIdx.x / tiles_j;
    const int j0 = (blockIdx.x % tiles_j) * LV;
    const int ntiles = (T + TT - 1) / TT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], (NC + 31) / 32);
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
                unsigned char* st = base + static_cast<size_t>(s) * stage_bytes;
                mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    tma_load_3d(st + tile_off(q), &maps.m[q], is_wide(kWide, q) ? j0 * W : j0, j * TT, o,
                                &full_bar[s], pol);
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    // consumers: thread c holds values w0 .. w0+E-1 of lane j0 + v
    const int c = threadIdx.x - 32;
    const int v = (c * E) / W;
    const int w0 = (c * E) % W;
    const bool valid = j0 + v < J;
    const int64_t row = static_cast<int64_t>(J) * W;
    float h[E];
#pragma unroll
    for (int e = 0; e < E; ++e)   // a null `init`: from zero
        h[e] = valid && init != nullptr ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] : 0.0f;
    float* obase = out + static_cast<int64_t>(o) * T * row + static_cast<int64_t>(j0) * W + c * E;

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(kMask, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int j = reverse ? ntiles - 1 - k : k;
        const int t0 = j * TT;
        const int n = min(TT, T - t0);
        const unsigned char* st = base + static_cast<size_t>(s) * stage_bytes;
        float* op = obase + static_cast<int64_t>(t0) * row;
        auto load = [&](const int tt, float (&dw)[Body::kSW][E], float (&dn)[Body::kSN]) {
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                const float* tile = reinterpret_cast<const float*>(st + tile_off(q));
                if (is_wide(kWide, q))
                    vec_load<E>(dw[wide_slot(kWide, q)], tile + tt * kVecRow + c * E);
                else
                    dn[narrow_slot(kWide, q)] = tile[tt * LV + v];
            }
        };
        float aw[Body::kSW][E], an[Body::kSN], bw[Body::kSW][E], bn[Body::kSN];
        // The state alternates between two register sets by trip parity, so a
        // trip never overwrites the registers the previous trip's store may
        // still be reading (consecutive trips alternate parity both ways).
        float hr[2][E];
#pragma unroll
        for (int e = 0; e < E; ++e) hr[0][e] = hr[1][e] = h[e];
        auto trip = [&](const int tt, const float (&dw)[Body::kSW][E], const float (&dn)[Body::kSN]) {
            Body::template step<E, G>(hr[tt & 1], hr[(tt & 1) ^ 1], dw, dn, kMask);
            if (valid) vec_store<E>(op + static_cast<int64_t>(tt) * row, hr[tt & 1]);
        };
        // the next trip's operands are read while a trip runs; rows past the
        // valid trips of a ragged tile hold TMA's zero fill and are not used
        if (!reverse) {
            load(0, aw, an);
#pragma unroll
            for (int tt = 0; tt < TT; tt += 2) {
                load(tt + 1, bw, bn);
                if (tt < n) trip(tt, aw, an);
                if (tt + 2 < TT) load(tt + 2, aw, an);
                if (tt + 1 < n) trip(tt + 1, bw, bn);
            }
        } else {
            load(TT - 1, aw, an);
#pragma unroll
            for (int tt = TT - 1; tt >= 0; tt -= 2) {
                load(tt - 1, bw, bn);
                if (tt < n) trip(tt, aw, an);
                if (tt - 2 >= 0) load(tt - 2, aw, an);
                if (tt - 1 < n) trip(tt - 1, bw, bn);
            }
        }
        // the last trip of the tile: n - 1 forward, 0 in reverse
        const int last = reverse ? 0 : n - 1;
#pragma unroll
        for (int e = 0; e < E; ++e) h[e] = hr[last & 1][e];
        __syncwarp(kMask);
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
}

}  // namespace es
