// skel_vec_bwd.cuh -- backward skeleton for body programs with a vector
// state of W = 2, 4, 8 or 16 values.
//
// "Nonlinear element scans", "Precision and gradients": the gradient is an
// element scan in the opposite trip order applying the body's
// vector-Jacobian product once a trip.  The layout is the forward vector
// skeleton's: the saved states, the output gradient and every full-width
// sequence are [O, T, J*W], a width-one sequence is [O, T, J]; one CTA owns
// LV = 128 / W adjacent lanes of one o (128 contiguous values per trip).
// Warp 0's lane 0 streams time tiles of TT trips, last tile first for a
// forward scan, of every sequence the VJP reads (`kVjpSeqs`), of the output
// gradient and TT+1 rows of the saved states (rows t0-1 .. t0+TT-1 of a
// forward scan, t0 .. t0+TT of a reverse one: every trip's previous state
// and its result; the row outside [0, T) arrives zero-filled and the scan's
// first trip takes `init`) into an S-stage SMEM ring with TMA.  Each of the 128 / E consumer threads holds E
// consecutive values of one lane's cotangent (a lane is G = W / E threads;
// the VJP's sums over the state combine them with xor shuffles).  Per trip
// it reads its operands from SMEM, adds the trip's output gradient to the
// cotangent, runs the VJP and writes its share of the gradients into an
// SMEM output tile (a width-one sequence's gradient, the same in the lane's
// G threads after the butterfly, by the lane's first thread).  After a
// consumer barrier one thread stores the tile with TMA tensor stores, which
// clip a ragged lane or time tile (two output buffers alternate).  Waits are
// bounded as in the other pipelines.
#pragma once

#include "skel_vec.cuh"   // vec_load, kVecRow

namespace es {

constexpr int kVecBwdMaxStages = 8;

template <class Body, int W, int E, int TT>
__global__ void __launch_bounds__(32 + kVecRow / E)
k_body_vec_bwd(const __grid_constant__ TmaMaps<2 * Body::kNS + 2> maps, const float* __restrict__ init,
               float* __restrict__ ginit, int T, int J, int tiles_j, int stages, int reverse, unsigned int* status,
               uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    constexpr int kP = NS, kG = NS + 1;           // map slots of the states and the output gradient
    constexpr unsigned kWide = Body::kWideMask;
    constexpr int LV = kVecRow / W;            // lanes per CTA
    constexpr int NC = kVecRow / E;            // consumer threads
    constexpr int G = W / E;                      // threads per lane
    constexpr unsigned kMask = 0xffffffffu;
    static_assert(NC % 32 == 0, "the consumer barrier counts whole warps");
    constexpr unsigned kLive = Body::kVjpSeqs;
    constexpr uint32_t kWideBytes = TT * kVecRow * 4u;
    constexpr uint32_t kNarrowBytes = TT * LV * 4u;   // a multiple of 128 bytes
    constexpr uint32_t kHBytes = (TT + 1) * kVecRow * 4u;
    auto seq_bytes = [](int q) -> uint32_t { return is_wide(kWide, q) ? kWideBytes : kNarrowBytes; };
    // byte offsets in a stage: the live sequences' tiles, the output
    // gradient's, then TT+1 rows of the saved states
    auto in_off = [&](int q) -> uint32_t {
        uint32_t off = 0;
        for (int k = 0; k < q; ++k)
            if (is_live(kLive, k)) off += seq_bytes(k);
        return off;
    };
    const uint32_t off_g = in_off(NS);
    const uint32_t off_h = off_g + kWideBytes;
    const uint32_t stage_bytes = off_h + kHBytes;
    // byte offset of sequence q's gradient tile in an output buffer
    auto out_off = [&](int q) -> uint32_t {
        uint32_t off = 0;
        for (int k = 0; k < q; ++k) off += seq_bytes(k);
        return off;
    };
    const uint32_t out_bytes = out_off(NS);

    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kVecBwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kVecBwdMaxStages];
    __shared__ int abort_flag;
    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    unsigned char* outs = base + static_cast<size_t>(stages) * stage_bytes;    // [2][out_bytes]
    const CUtensorMap* gmaps = &maps.m[NS + 2];

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
            for (int q = 0; q < NS + 2; ++q)
                if (q >= NS || is_live(kLive, q)) tma_prefetch_desc(&maps.m[q]);
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
                const int j = reverse ? k : ntiles - 1 - k;
                const int t0 = j * TT;
                unsigned char* st = base + static_cast<size_t>(s) * stage_bytes;
                mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    if (is_live(kLive, q))
                        tma_load_3d(st + in_off(q), &maps.m[q], is_wide(kWide, q) ? j0 * W : j0, t0, o, &full_bar[s],
                                    pol);
                tma_load_3d(st + off_g, &maps.m[kG], j0 * W, t0, o, &full_bar[s], pol);
                // the states from the row before the tile (forward) or from the tile's first (reverse)
                tma_load_3d(st + off_h, &maps.m[kP], j0 * W, reverse ? t0 : t0 - 1, o, &full_bar[s], pol);
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
    const int t_first = reverse ? T - 1 : 0;     // the scan's first trip starts from init
    const bool storer = (threadIdx.x == 32);
    float h0[E];
#pragma unroll
    for (int e = 0; e < E; ++e)   // a null `init`: from zero
        h0[e] = valid && init != nullptr ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] : 0.0f;
    float lam[E];
#pragma unroll
    for (int e = 0; e < E; ++e) lam[e] = 0.0f;

    for (int k = 0; k <= ntiles; ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        // the buffer this tile writes was last read by the store issued a tile
        // ago (long done): the storer waits for that read before the barrier
        // rather than for each store right after issuing it
        if (storer) bulk_wait_read<0>();
        if (k > 0) fence_proxy_async_smem();     // this thread's gradient writes of tile k-1
        if (consumer_vote_any_failed(!ok, NC)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        if (storer && k > 0) {
            const int jp = reverse ? k - 1 : ntiles - k;
            const unsigned char* ob = outs + static_cast<size_t>((k - 1) & 1) * out_bytes;
#pragma unroll
            for (int q = 0; q < NS; ++q)
                tma_store_3d(&gmaps[q], is_wide(kWide, q) ? j0 * W : j0, jp * TT, o, ob + out_off(q));
            bulk_commit();
        }
        if (k == ntiles) break;
        const int j = reverse ? k : ntiles - 1 - k;
        const int t0 = j * TT;
        const int n = min(TT, T - t0);
        const unsigned char* st = base + static_cast<size_t>(s) * stage_bytes;
        unsigned char* ob = outs + static_cast<size_t>(k & 1) * out_bytes;
        auto trip = [&](const int tt) {
            float dw[Body::kSW][E], dn[Body::kSN], p[E], hr[E], g[E];
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                const float* tile = reinterpret_cast<const float*>(st + in_off(q));
                if (is_wide(kWide, q)) {
                    if (is_live(kLive, q)) {
                        vec_load<E>(dw[wide_slot(kWide, q)], tile + tt * kVecRow + c * E);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) dw[wide_slot(kWide, q)][e] = 0.0f;
                    }
                } else {
                    dn[narrow_slot(kWide, q)] = is_live(kLive, q) ? tile[tt * LV + v] : 0.0f;
                }
            }
            // rows of the states box: the previous state and the trip's result
            const float* hb = reinterpret_cast<const float*>(st + off_h) + c * E;
            vec_load<E>(p, hb + (tt + reverse) * kVecRow);
            vec_load<E>(hr, hb + (tt + 1 - reverse) * kVecRow);
            vec_load<E>(g, reinterpret_cast<const float*>(st + off_g) + tt * kVecRow + c * E);
            const bool first = t0 + tt == t_first;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if (first) p[e] = h0[e];
                lam[e] = __fadd_rn(lam[e], g[e]);
            }
            float dp[E], dsw[Body::kSW][E], dsn[Body::kSN];
            Body::template vjp<E, G>(dp, dsw, dsn, lam, p, hr, dw, dn, kMask);
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                float* tile = reinterpret_cast<float*>(ob + out_off(q));
                if (is_wide(kWide, q)) {
                    float* d = tile + tt * kVecRow + c * E;
#pragma unroll
                    for (int e = 0; e < E; ++e) d[e] = dsw[wide_slot(kWide, q)][e];
                } else if (w0 == 0) {
                    tile[tt * LV + v] = dsn[narrow_slot(kWide, q)];
                }
            }
#pragma unroll
            for (int e = 0; e < E; ++e) lam[e] = dp[e];
        };
        // trips past T in a ragged tile (zero-filled) must not touch the
        // cotangent; the TMA store clips them
        if (n == TT) {
            if (!reverse) {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt) trip(tt);
            } else {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) trip(tt);
            }
        } else {
            if (!reverse) {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt)
                    if (tt < n) trip(tt);
            } else {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    if (tt < n) trip(tt);
            }
        }
        // every operand of the stage has been read
        __syncwarp(kMask);
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    if (storer) bulk_wait_all();
    if (valid && ginit != nullptr) {   // null: not wanted
#pragma unroll
        for (int e = 0; e < E; ++e) ginit[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] = lam[e];
    }
}

}  // namespace es
