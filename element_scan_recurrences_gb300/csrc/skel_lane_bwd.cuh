// skel_lane_bwd.cuh -- backward skeleton for body programs with the lanes
// innermost (scalar state, canonical view [O, T, I]).
//
// "Nonlinear element scans", "Precision and gradients": the gradient is an
// element scan in the opposite trip order applying the body's
// vector-Jacobian product once a trip.  One CTA owns LI adjacent lanes of
// one o and walks the time tiles of TT trips backwards in scan order:
//   * warp 0, lane 0 streams, per tile, TT trips of every sequence the VJP
//     reads (`kVjpSeqs`), of the output gradient, and TT+1 rows of the saved
//     states (rows t0-1 .. t0+TT-1 of a forward scan, t0 .. t0+TT of a
//     reverse one: every trip's previous state and its own result; the row
//     outside [0, T) arrives zero-filled and the scan's first trip takes
//     `init`) into an S-stage SMEM ring with TMA;
//   * LI consumer threads (one per lane) copy the tile into registers, hand
//     the stage back, then run the VJP over the tile with the cotangent in a
//     register.  The serial chain is only the cotangent's (the body itself
//     is evaluated from loaded states), so trips overlap freely.  Each trip
//     writes the sequences' gradients into an SMEM output tile (fixed
//     offsets, no address arithmetic); after a consumer barrier one thread
//     stores the tile with TMA tensor stores, which also clip a ragged lane
//     or time tile (two output buffers alternate).
// Waits are bounded as in the forward skeletons.
#pragma once

#include "skel_common.cuh"

namespace es {

constexpr int kLaneBwdMaxStages = 8;

template <class Body, int LI, int TT>
__global__ void __launch_bounds__(32 + LI)
k_body_lane_bwd(const __grid_constant__ TmaMaps<2 * Body::kNS + 2> maps, const float* __restrict__ init,
                float* __restrict__ ginit, int T, int I, int tiles_i, int stages, int reverse, unsigned int* status,
                uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    constexpr unsigned kLive = Body::kVjpSeqs;
    constexpr int NL = live_count(kLive, NS);    // sequences streamed
    constexpr int kP = NS, kG = NS + 1;          // map slots of the states and the output gradient
    static_assert(Body::kWideMask == (1u << NS) - 1u, "a scalar state has no width-one sequences");
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kLaneBwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kLaneBwdMaxStages];
    __shared__ int abort_flag;

    // a stage: the live sequences' tiles, the output gradient's, then TT+1
    // rows of the saved states
    constexpr int kTileFloats = TT * LI;
    constexpr int kOffG = NL * kTileFloats, kOffH = (NL + 1) * kTileFloats;
    constexpr int kStageFloats = kOffH + (TT + 1) * LI;
    constexpr uint32_t kStageBytes = kStageFloats * 4u;
    float* tiles = reinterpret_cast<float*>(smem_raw + smem_align_pad(smem_raw));   // [stages][kStageFloats]
    float* outs = tiles + static_cast<size_t>(stages) * kStageFloats;               // [2][NS][TT][LI]
    const CUtensorMap* gmaps = &maps.m[NS + 2];                                      // the gradients' maps

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
                float* st = tiles + static_cast<size_t>(s) * kStageFloats;
                mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    if (is_live(kLive, q))
                        tma_load_3d(st + live_slot(kLive, q) * kTileFloats, &maps.m[q], i0, t0, o, &full_bar[s], pol);
                tma_load_3d(st + kOffG, &maps.m[kG], i0, t0, o, &full_bar[s], pol);
                // the states from the row before the tile (forward) or from the tile's first (reverse)
                tma_load_3d(st + kOffH, &maps.m[kP], i0, reverse ? t0 : t0 - 1, o, &full_bar[s], pol);
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    const int c = threadIdx.x - 32;
    const int i = i0 + c;
    const bool valid = i < I;
    const float h0 = valid && init != nullptr ? init[static_cast<int64_t>(o) * I + i] : 0.0f;   // null: zero
    const int t_first = reverse ? T - 1 : 0;     // the scan's first trip starts from init
    const bool storer = (threadIdx.x == 32);
    float lam = 0.0f;

    // One consumer barrier per tile votes on whether any consumer gave up its
    // wait and marks the previous tile's gradients complete in SMEM.
    for (int k = 0; k <= ntiles; ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        // the buffer this tile writes was last read by the store issued a tile
        // ago (long done): the storer waits for that read before the barrier
        // rather than for each store right after issuing it
        if (storer) bulk_wait_read<0>();
        if (k > 0) fence_proxy_async_smem();     // this thread's gradient writes of tile k-1
        if (consumer_vote_any_failed(!ok, LI)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        if (storer && k > 0) {
            const int jp = reverse ? k - 1 : ntiles - k;
            const float* ob = outs + static_cast<size_t>((k - 1) & 1) * NS * kTileFloats;
#pragma unroll
            for (int q = 0; q < NS; ++q) tma_store_3d(&gmaps[q], i0, jp * TT, o, ob + q * kTileFloats);
            bulk_commit();
        }
        if (k == ntiles) break;
        const int j = reverse ? k : ntiles - 1 - k;
        const int t0 = j * TT;
        const int n = min(TT, T - t0);
        const float* st = tiles + static_cast<size_t>(s) * kStageFloats + c;
        float vr[NL > 0 ? NL : 1][TT], vg[TT], vh[TT + 1];
#pragma unroll
        for (int q = 0; q < NL; ++q)
#pragma unroll
            for (int tt = 0; tt < TT; ++tt) vr[q][tt] = st[q * kTileFloats + tt * LI];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) vg[tt] = st[kOffG + tt * LI];
#pragma unroll
        for (int tt = 0; tt <= TT; ++tt) vh[tt] = st[kOffH + tt * LI];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        // the scan's first trip takes `init` as its previous state (one tile;
        // the row it replaces is outside [0, T), no trip's result)
        if (t_first >= t0 && t_first < t0 + TT) {
#pragma unroll
            for (int tt = 0; tt < TT; ++tt)
                if (t0 + tt == t_first) {
                    if (!reverse)
                        vh[tt] = h0;
                    else
                        vh[tt + 1] = h0;
                }
        }
        float* ob = outs + static_cast<size_t>(k & 1) * NS * kTileFloats + c;
        // trip tt with its previous state in row pi and its result in row ri
        auto trip = [&](const int tt, const int pi, const int ri) {
            lam = __fadd_rn(lam, vg[tt]);
            const float lm[1] = {lam};
            const float hp[1] = {vh[pi]};
            const float hr[1] = {vh[ri]};
            float sw[Body::kSW][1];
            const float sn[Body::kSN] = {};
#pragma unroll
            for (int q = 0; q < NS; ++q) sw[q][0] = is_live(kLive, q) ? vr[live_slot(kLive, q)][tt] : 0.0f;
            float dp[1];
            float dsw[Body::kSW][1];
            float dsn[Body::kSN];
            Body::template vjp<1, 1>(dp, dsw, dsn, lm, hp, hr, sw, sn, 0xffffffffu);
#pragma unroll
            for (int q = 0; q < NS; ++q) ob[q * kTileFloats + tt * LI] = dsw[q][0];
            lam = dp[0];
        };
        // trips past T in a ragged tile (zero-filled) must not touch the
        // cotangent; the TMA store clips them
        if (n == TT) {
            if (!reverse) {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt) trip(tt, tt, tt + 1);
            } else {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) trip(tt, tt + 1, tt);
            }
        } else {
            if (!reverse) {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt)
                    if (tt < n) trip(tt, tt, tt + 1);
            } else {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    if (tt < n) trip(tt, tt + 1, tt);
            }
        }
    }
    if (storer) bulk_wait_all();
    if (valid && ginit != nullptr) ginit[static_cast<int64_t>(o) * I + i] = lam;   // null: not wanted
}

}  // namespace es
