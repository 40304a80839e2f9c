// skel_vec.cuh -- body-program skeleton for a vector state of W = 2, 4, 8 or
// 16 values ("Nonlinear element scans", `:state-axis`).
//
// Canonical view: the output and every full-width sequence are [O, T, J*W],
// a width-one sequence is [O, T, J].  One CTA owns LV = 128 / W adjacent
// lanes of one o (128 contiguous values per trip) and walks all T trips.
// Warp roles: the consumer warps first (one per scheduler), then a producer
// and a store warp.  The producer streams time tiles of TT trips of every
// sequence (box {128, TT} of a full-width sequence, {LV, TT} of a width-one
// one) into an S-stage SMEM ring with TMA.  Each of the 128 / E consumer
// threads holds E consecutive values of one lane's state; a lane is G = W / E
// threads, and the body's reductions combine them with xor shuffles.  A
// consumer reads a trip's operands from SMEM one trip ahead of its use, runs
// the body, and writes its E values into the stage's tile of states; the
// store warp sends each finished tile out with one TMA tensor store and hands
// the stage back to the producer once the store has read it (full, done and
// empty mbarriers; the consumers issue no global store).  Waits are bounded
// as in the other pipelines.
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

// E values into shared memory (16-byte pieces where E allows)
template <int E>
__device__ __forceinline__ void vec_put(float* p, const float (&v)[E]) {
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int i = 0; i < E; i += 4)
            *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else if constexpr (E == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    } else {
        p[0] = v[0];
    }
}

template <class Body, int W, int E, int TT>
__global__ void __launch_bounds__(32 * ((kVecRow / E + 31) / 32) + 64)
k_body_vec(const __grid_constant__ TmaMaps<Body::kNS> maps, const __grid_constant__ CUtensorMap map_out,
           const float* __restrict__ init, int T, int J, int tiles_j, int stages, int reverse, unsigned int* status,
           uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    constexpr unsigned kWide = Body::kWideMask;
    constexpr int LV = kVecRow / W;                // lanes per CTA
    constexpr int NC = kVecRow / E;                // consumer threads
    constexpr int CWN = (NC + 31) / 32;            // consumer warps
    constexpr int G = W / E;                       // threads per lane
    constexpr unsigned kMask = NC >= 32 ? 0xffffffffu : ((1u << NC) - 1u);
    constexpr uint32_t kWideBytes = TT * kVecRow * 4u;
    constexpr uint32_t kNarrowBytes = TT * LV * 4u;   // a multiple of 128 bytes
    // byte offset of sequence q's tile inside a stage (the states' tile
    // follows the sequences'), and the stage size
    auto tile_off = [](int q) -> uint32_t {
        uint32_t off = 0;
        for (int k = 0; k < q; ++k) off += is_wide(kWide, k) ? kWideBytes : kNarrowBytes;
        return off;
    };
    const uint32_t in_bytes = tile_off(NS);
    const uint32_t out_off = (in_bytes + 127u) & ~127u;
    const uint32_t stage_bytes = (out_off + kWideBytes + 1023u) & ~1023u;

    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kVecMaxStages];
    __shared__ __align__(8) uint64_t done_bar[kVecMaxStages];
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
            mbar_init(&done_bar[s], CWN);
            mbar_init(&empty_bar[s], 1);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == CWN) {
        // producer: time tiles of every sequence into the stage ring
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
                mbar_arrive_expect_tx(&full_bar[s], in_bytes);
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
    if (warp == CWN + 1) {
        // storer: each tile of states leaves shared memory as one TMA tensor
        // store (rows past T and lanes past J clipped by the tensor map); the
        // stage goes back to the producer once the store has read it
        if (lane == 0) {
            tma_prefetch_desc(&map_out);
            for (int k = 0; k < ntiles; ++k) {
                const int s = k % stages;
                if (!mbar_wait_bounded(&done_bar[s], (k / stages) & 1, wait_ns, &abort_flag)) {
                    report_timeout(status, &abort_flag);
                    break;
                }
                const int j = reverse ? ntiles - 1 - k : k;
                tma_store_3d(&map_out, j0 * W, j * TT, o, base + static_cast<size_t>(s) * stage_bytes + out_off);
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(&empty_bar[s]);
            }
            bulk_wait_all();
        }
        return;
    }

    // consumers (the first warps, one per scheduler): thread c holds values
    // w0 .. w0+E-1 of lane j0 + v
    const int c = threadIdx.x;
    if (c >= NC) return;
    const int v = (c * E) / W;
    const int w0 = (c * E) % W;
    const bool valid = j0 + v < J;
    float h[E];
#pragma unroll
    for (int e = 0; e < E; ++e)   // a null `init`: from zero
        h[e] = valid && init != nullptr ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] : 0.0f;

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
        unsigned char* st = base + static_cast<size_t>(s) * stage_bytes;
        float* op = reinterpret_cast<float*>(st + out_off) + c * E;
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
            vec_put<E>(op + tt * kVecRow, hr[tt & 1]);
        };
        // the next trip's operands are read while a trip runs; rows past the
        // valid trips of a ragged tile hold TMA's zero fill and are not used
        // (full tiles run unguarded: one basic block, so the loads and stores
        // of neighbouring trips overlap the chain)
        if (!reverse) {
            load(0, aw, an);
            if (n == TT) {
#pragma unroll
                for (int tt = 0; tt < TT; tt += 2) {
                    load(tt + 1, bw, bn);
                    trip(tt, aw, an);
                    if (tt + 2 < TT) load(tt + 2, aw, an);
                    trip(tt + 1, bw, bn);
                }
            } else {
#pragma unroll
                for (int tt = 0; tt < TT; tt += 2) {
                    load(tt + 1, bw, bn);
                    if (tt < n) trip(tt, aw, an);
                    if (tt + 2 < TT) load(tt + 2, aw, an);
                    if (tt + 1 < n) trip(tt + 1, bw, bn);
                }
            }
        } else {
            load(TT - 1, aw, an);
            if (n == TT) {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; tt -= 2) {
                    load(tt - 1, bw, bn);
                    trip(tt, aw, an);
                    if (tt - 2 >= 0) load(tt - 2, aw, an);
                    trip(tt - 1, bw, bn);
                }
            } else {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; tt -= 2) {
                    load(tt - 1, bw, bn);
                    if (tt < n) trip(tt, aw, an);
                    if (tt - 2 >= 0) load(tt - 2, aw, an);
                    if (tt - 1 < n) trip(tt - 1, bw, bn);
                }
            }
        }
        // the last trip of the tile: n - 1 forward, 0 in reverse
        const int last = reverse ? 0 : n - 1;
#pragma unroll
        for (int e = 0; e < E; ++e) h[e] = hr[last & 1][e];
        // the tile's states are in shared memory: visible to the tensor
        // store, then handed to the storer
        fence_proxy_async_smem();
        __syncwarp(kMask);
        if (lane == 0) mbar_arrive(&done_bar[s]);
    }
}

}  // namespace es
