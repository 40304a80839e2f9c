// skel_time_bwd.cuh -- backward skeleton for body programs with the sequence
// axis innermost (scalar state on a [lanes, T] layout, e.g. `:axis -1`).
//
// "Nonlinear element scans", "Precision and gradients": the gradient is an
// element scan in the opposite trip order applying the body's
// vector-Jacobian product once a trip.  Each lane is one row of T values.
// Per tile of LO rows x 32 trips the producer streams, with TMA, every
// sequence the VJP reads (`kVjpSeqs`) and the output gradient as
// 128-byte-swizzled boxes {32, LO}
// (conflict-free 16-byte reads of a thread's own row) and the saved states as
// an unswizzled box {36, LO} whose 144-byte rows also read conflict-free:
// trips t0-4 .. t0+31 for a forward scan, t0 .. t0+35 for a reverse one, so
// the state before every trip of the tile, and its result, are in the same
// box (columns outside 0..T-1 are zero-filled and `init` takes the scan's
// first trip's place).
// Each consumer thread owns one row.  It walks its 32 trips in backward order
// four at a time (one 16-byte vector of every tile, read one group ahead),
// runs the VJP with the cotangent in a register, and writes the sequences'
// gradients into swizzled output tiles that one thread stores with TMA tensor
// stores after a consumer barrier (two buffers alternate).  Waits are bounded
// as in the other pipelines.
#pragma once

#include "skel_common.cuh"

namespace es {

constexpr int kTimeBwdTT = 32;          // trips per tile: 128 bytes per row (the swizzle span)
constexpr int kTimeBwdHCols = 36;       // state columns per tile row
constexpr int kTimeBwdMaxStages = 4;

template <class Body, int LO>
__global__ void __launch_bounds__(32 + LO)
k_body_time_bwd(const __grid_constant__ TmaMaps<2 * Body::kNS + 2> maps, const float* __restrict__ init,
                float* __restrict__ ginit, int O, int T, int stages, int reverse, unsigned int* status,
                uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NS = Body::kNS;
    constexpr unsigned kLive = Body::kVjpSeqs;
    constexpr int NL = live_count(kLive, NS);   // sequences streamed
    constexpr int kP = NS, kG = NS + 1;      // map slots of the states and the output gradient
    static_assert(Body::kWideMask == (1u << NS) - 1u, "a scalar state has no width-one sequences");
    constexpr uint32_t kTile = LO * 128u;                          // one swizzled {32, LO} tile
    constexpr uint32_t kHTile = LO * kTimeBwdHCols * 4u;
    constexpr uint32_t kOffG = NL * kTile;                         // the live sequences, then the output gradient
    constexpr uint32_t kOffH = (NL + 1) * kTile;
    constexpr uint32_t kStage = (kOffH + kHTile + 1023u) & ~1023u;
    constexpr uint32_t kOut = NS * kTile;                           // one output buffer
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kTimeBwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kTimeBwdMaxStages];
    __shared__ int abort_flag;

    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    unsigned char* outs = base + static_cast<size_t>(stages) * kStage;    // [2][NS][LO rows x 128 B]
    const CUtensorMap* gmaps = &maps.m[NS + 2];
    const int o0 = blockIdx.x * LO;
    const int ntiles = (T + kTimeBwdTT - 1) / kTimeBwdTT;
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
                const int t0 = (reverse ? k : ntiles - 1 - k) * kTimeBwdTT;
                unsigned char* st = base + static_cast<size_t>(s) * kStage;
                mbar_arrive_expect_tx(&full_bar[s], kOffH + kHTile);
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    if (is_live(kLive, q))
                        tma_load_2d(st + live_slot(kLive, q) * kTile, &maps.m[q], t0, o0, &full_bar[s], pol);
                tma_load_2d(st + kOffG, &maps.m[kG], t0, o0, &full_bar[s], pol);
                // the states four trips back (forward) or from the tile (reverse): x stays 16-byte aligned
                tma_load_2d(st + kOffH, &maps.m[kP], reverse ? t0 : t0 - 4, o0, &full_bar[s], pol);
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
    const float h0 = valid && init != nullptr ? init[o0 + r] : 0.0f;   // null: from zero
    const int t_first = reverse ? T - 1 : 0;
    const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
    const uint32_t swz = static_cast<uint32_t>(r & 7);   // 128-byte swizzle: chunk q lives at q ^ (row % 8)
    const bool storer = (threadIdx.x == 32);
    float lam = 0.0f;

    struct Quad {
        float4 s[NS];   // four trips of every sequence
        float4 g;       // and of the output gradient
        float4 h0, h1;  // the state columns 4q .. 4q+7 of the 36-column box
    };

    for (int k = 0; k <= ntiles; ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        // the buffer this tile writes was last read by the store issued a tile
        // ago (long done): the storer waits for that read before the barrier
        // rather than for each store right after issuing it
        if (storer) bulk_wait_read<0>();
        if (k > 0) fence_proxy_async_smem();     // this thread's gradient writes of tile k-1
        if (consumer_vote_any_failed(!ok, LO)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        if (storer && k > 0) {
            const int tp = (reverse ? k - 1 : ntiles - k) * kTimeBwdTT;
            const unsigned char* ob = outs + static_cast<size_t>((k - 1) & 1) * kOut;
#pragma unroll
            for (int q = 0; q < NS; ++q) tma_store_2d(&gmaps[q], tp, o0, ob + q * kTile);
            bulk_commit();
        }
        if (k == ntiles) break;
        const int t0 = (reverse ? k : ntiles - 1 - k) * kTimeBwdTT;
        const int nq = min(kTimeBwdTT, T - t0) >> 2;      // T % 4 == 0 on this path
        const unsigned char* st = base + static_cast<size_t>(s) * kStage;
        const unsigned char* hrow = st + kOffH + static_cast<uint32_t>(r) * (kTimeBwdHCols * 4);
        unsigned char* ob = outs + static_cast<size_t>(k & 1) * kOut + row_off;
        auto chunk = [&](int q) { return (static_cast<uint32_t>(q) ^ swz) << 4; };
        auto readq = [&](int q, Quad& d) {
#pragma unroll
            for (int p = 0; p < NS; ++p)
                d.s[p] = is_live(kLive, p)
                             ? *reinterpret_cast<const float4*>(st + live_slot(kLive, p) * kTile + row_off + chunk(q))
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            d.g = *reinterpret_cast<const float4*>(st + kOffG + row_off + chunk(q));
            d.h0 = *reinterpret_cast<const float4*>(hrow + 16 * q);
            d.h1 = *reinterpret_cast<const float4*>(hrow + 16 * (q + 1));
        };
        auto comp = [](const float4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; };
        // four trips of the row, in backward order
        auto quad = [&](const int q, const Quad& d) {
            float res[NS][4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = reverse ? m : 3 - m;
                // the state before trip 4q+i: column 4q+i+3 of the box (forward), 4q+i+1 (reverse)
                const int hc = reverse ? i + 1 : i + 3;
                float p = hc < 4 ? comp(d.h0, hc) : comp(d.h1, hc - 4);
                if (t0 + 4 * q + i == t_first) p = h0;
                // the trip's result: column 4q+i+4 (forward), 4q+i (reverse)
                const float hr[1] = {reverse ? comp(d.h0, i) : comp(d.h1, i)};
                lam = __fadd_rn(lam, comp(d.g, i));
                const float lm[1] = {lam};
                const float hp[1] = {p};
                float sw[Body::kSW][1];
                const float sn[Body::kSN] = {};
#pragma unroll
                for (int pq = 0; pq < NS; ++pq) sw[pq][0] = comp(d.s[pq], i);
                float dp[1];
                float dsw[Body::kSW][1];
                float dsn[Body::kSN];
                Body::template vjp<1, 1>(dp, dsw, dsn, lm, hp, hr, sw, sn, 0xffffffffu);
#pragma unroll
                for (int pq = 0; pq < NS; ++pq) res[pq][i] = dsw[pq][0];
                lam = dp[0];
            }
#pragma unroll
            for (int pq = 0; pq < NS; ++pq)
                *reinterpret_cast<float4*>(ob + pq * kTile + chunk(q)) =
                    make_float4(res[pq][0], res[pq][1], res[pq][2], res[pq][3]);
        };
        // groups past T in a ragged tile (zero-filled) must not touch the
        // cotangent; the TMA store clips them
        // (full tiles run unguarded: one basic block, so the next group's
        // reads and this group's stores overlap the chain)
        Quad cur, nxt;
        const bool full = nq == kTimeBwdTT / 4;
        if (!reverse) {
            readq(kTimeBwdTT / 4 - 1, cur);
            if (full) {
#pragma unroll
                for (int q = kTimeBwdTT / 4 - 1; q >= 0; --q) {
                    if (q > 0) readq(q - 1, nxt);
                    quad(q, cur);
                    cur = nxt;
                }
            } else {
#pragma unroll
                for (int q = kTimeBwdTT / 4 - 1; q >= 0; --q) {
                    if (q > 0) readq(q - 1, nxt);
                    if (q < nq) quad(q, cur);
                    cur = nxt;
                }
            }
        } else {
            readq(0, cur);
            if (full) {
#pragma unroll
                for (int q = 0; q < kTimeBwdTT / 4; ++q) {
                    if (q + 1 < kTimeBwdTT / 4) readq(q + 1, nxt);
                    quad(q, cur);
                    cur = nxt;
                }
            } else {
#pragma unroll
                for (int q = 0; q < kTimeBwdTT / 4; ++q) {
                    if (q + 1 < kTimeBwdTT / 4) readq(q + 1, nxt);
                    if (q < nq) quad(q, cur);
                    cur = nxt;
                }
            }
        }
        // every operand of the stage has been read
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    if (storer) bulk_wait_all();
    if (valid && ginit != nullptr) ginit[o0 + r] = lam;   // null: not wanted
}

}  // namespace es
