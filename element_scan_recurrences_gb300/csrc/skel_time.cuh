// skel_time.cuh -- body-program skeleton with the sequence axis innermost
// (a scalar state on a [lanes, T] layout, e.g. `:axis -1`).
//
// Each lane is one contiguous row of T values.  The CTA stages tiles of LO
// rows x 32 trips of every sequence (box {32, LO} of a 2-D tensor map, one
// 128-byte segment per row) through an S-stage TMA/mbarrier ring, with the
// 128-byte swizzle, so that a thread reading its own row four trips at a time
// (one 16-byte vector) is conflict-free across the warp.  Each consumer
// thread owns one row: it reads its 32-trip segments (all of them into
// registers first when the body has at most three sequences, so the stage
// goes back to the producer before the chain runs; else four trips ahead),
// runs the body over the segment and writes the states into a swizzled
// output tile, which one thread stores with a TMA tensor store (three output
// buffers, so the stores overlap the next tiles).  Reverse scans take the
// tiles last-first and each group of four trips in descending order.  Waits
// are bounded as in the other pipelines.
#pragma once

#include "skel_common.cuh"

namespace es {

constexpr int kTimeTT = 32;          // trips per tile: 128 bytes per row (the swizzle span)
constexpr int kTimeMaxStages = 6;
constexpr int kTimeOutBufs = 3;

template <class Body, int LO>
__global__ void __launch_bounds__(32 + LO)
k_body_time(const __grid_constant__ TmaMaps<Body::kNS + 1> maps, const float* __restrict__ init, int O, int T,
            int stages, int reverse, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    static_assert(Body::kWideMask == (1u << NS) - 1u, "a scalar state has no width-one sequences");
    constexpr bool kStage = NS <= 3;          // the whole segment of every sequence in registers
    constexpr uint32_t kTileBytes = LO * 128u;
    const CUtensorMap* map_out = &maps.m[NS];   // the output map follows the sequences'

    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kTimeMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kTimeMaxStages];
    __shared__ int abort_flag;

    // every tile is LO rows x 128 bytes and starts on a 1024-byte boundary
    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    unsigned char* in_tiles = base;                                             // [stages][NS][LO][128 B]
    unsigned char* out_tiles = base + static_cast<size_t>(stages) * NS * kTileBytes;   // [3][LO][128 B]

    const int o0 = blockIdx.x * LO;
    const int ntiles = (T + kTimeTT - 1) / kTimeTT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], LO / 32);
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
                unsigned char* st = in_tiles + static_cast<size_t>(s) * NS * kTileBytes;
                mbar_arrive_expect_tx(&full_bar[s], NS * kTileBytes);
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    tma_load_2d(st + q * kTileBytes, &maps.m[q], j * kTimeTT, o0, &full_bar[s], pol);
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    // consumers: thread r owns row o0 + r
    const int r = threadIdx.x - 32;
    const bool valid = o0 + r < O;
    float h = valid && init != nullptr ? init[o0 + r] : 0.0f;   // null: from zero
    const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
    const uint32_t swz = static_cast<uint32_t>(r & 7);   // 128-byte swizzle: chunk q lives at q ^ (row % 8)
    const bool storer = (threadIdx.x == 32);

    // One consumer barrier per tile votes on whether any consumer gave up its
    // wait (all leave together) and marks the previous tile's output complete.
    for (int k = 0; k <= ntiles; ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (k > 0) fence_proxy_async_smem();     // this thread's writes of tile k-1
        if (consumer_vote_any_failed(!ok, LO)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        if (storer && k > 0) {
            const int jp = reverse ? ntiles - k : k - 1;
            tma_store_2d(map_out, jp * kTimeTT, o0,
                         out_tiles + static_cast<size_t>((k - 1) % kTimeOutBufs) * kTileBytes);
            bulk_commit();
            // the buffer written at the next tile was read out by an older store
            bulk_wait_read<1>();
        }
        if (k == ntiles) break;
        const int j = reverse ? ntiles - 1 - k : k;
        const int t0 = j * kTimeTT;
        const int nq = min(kTimeTT, T - t0) >> 2;     // T % 4 == 0 on this path
        const unsigned char* srow = in_tiles + static_cast<size_t>(s) * NS * kTileBytes + row_off;
        unsigned char* orow = out_tiles + static_cast<size_t>(k % kTimeOutBufs) * kTileBytes + row_off;
        auto chunk = [&](int q) { return (static_cast<uint32_t>(q) ^ swz) << 4; };
        auto read4 = [&](int q, float4 (&d)[NS]) {
#pragma unroll
            for (int p = 0; p < NS; ++p) d[p] = *reinterpret_cast<const float4*>(srow + p * kTileBytes + chunk(q));
        };
        // four trips of the row from one 16-byte vector of every sequence
        auto quad = [&](const int q, const float4 (&d)[NS], const bool rev) {
            float res[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = rev ? 3 - i : i;
                float sw[Body::kSW][1];
                const float sn[Body::kSN] = {};
#pragma unroll
                for (int p = 0; p < NS; ++p) sw[p][0] = m == 0 ? d[p].x : m == 1 ? d[p].y : m == 2 ? d[p].z : d[p].w;
                const float hp[1] = {h};
                float rr[1];
                Body::template step<1, 1>(rr, hp, sw, sn, 0xffffffffu);
                h = rr[0];
                res[m] = h;
            }
            *reinterpret_cast<float4*>(orow + chunk(q)) = make_float4(res[0], res[1], res[2], res[3]);
        };
        if constexpr (kStage) {
            float4 seg[kTimeTT / 4][NS];
#pragma unroll
            for (int q = 0; q < kTimeTT / 4; ++q) read4(q, seg[q]);
            // the input stage is free as soon as the segment sits in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            // full tiles run unguarded (one basic block, so the quads' loads,
            // stores and address arithmetic overlap the chain); only a ragged
            // last tile checks every quad
            if (nq == kTimeTT / 4) {
                if (!reverse) {
#pragma unroll
                    for (int q = 0; q < kTimeTT / 4; ++q) quad(q, seg[q], false);
                } else {
#pragma unroll
                    for (int q = kTimeTT / 4 - 1; q >= 0; --q) quad(q, seg[q], true);
                }
            } else if (!reverse) {
#pragma unroll
                for (int q = 0; q < kTimeTT / 4; ++q)
                    if (q < nq) quad(q, seg[q], false);
            } else {
#pragma unroll
                for (int q = kTimeTT / 4 - 1; q >= 0; --q)
                    if (q < nq) quad(q, seg[q], true);
            }
        } else {
            float4 cur[NS], nxt[NS];
            if (!reverse) {
                read4(0, cur);
#pragma unroll
                for (int q = 0; q < kTimeTT / 4; ++q) {
                    if (q + 1 < kTimeTT / 4) read4(q + 1, nxt);
                    if (q < nq) quad(q, cur, false);
#pragma unroll
                    for (int p = 0; p < NS; ++p) cur[p] = nxt[p];
                }
            } else {
                read4(kTimeTT / 4 - 1, cur);
#pragma unroll
                for (int q = kTimeTT / 4 - 1; q >= 0; --q) {
                    if (q > 0) read4(q - 1, nxt);
                    if (q < nq) quad(q, cur, true);
#pragma unroll
                    for (int p = 0; p < NS; ++p) cur[p] = nxt[p];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
    }
    if (storer) bulk_wait_all();
}

}  // namespace es
