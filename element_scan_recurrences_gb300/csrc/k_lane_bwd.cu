// k_lane_bwd.cu -- backward pass of TANH_DECAY / MAXPLUS with the lanes
// innermost (ES_PATH_LANE_TMA for es_scan_backward_f32).
//
// "Nonlinear element scans", "Precision and gradients": the gradient of a scan
// is another scan over the same lanes in the opposite trip order, applying
// the body's vector-Jacobian product once a trip; a forward scan's gradient
// runs from the last trip to the first, a reverse scan's from the first to the
// last.  Per trip, with h the trip's output, p the state before it and lam
// the state's cotangent (lam += dL/dh first):
//   TANH_DECAY  m = lam * (1 - h*h):  dx = m, da = m * p, lam = m * a
//   MAXPLUS     v = p - c: the larger of v and x takes lam (a tie splits it)
//
// Layout as in the forward lane kernel: canonical [O, T, I], one CTA per tile
// of LI lanes of one o.  The producer streams, per time tile of TT trips, the
// output gradient, the second sequence (a or c), x (MAXPLUS only) and TT+1
// rows of saved states: the tile's own outputs plus the state before its
// first trip in scan order (a TMA box that may start at row -1 or end at row
// T; TMA fills those rows with zeros and the consumer takes `initial` there).
// Consumers copy the tile to registers, free the stage, then run the chain.
// Gradients go either straight to global memory (one coalesced row store of
// dx and da per trip and warp) or, staged, into a shared-memory tile that one
// thread sends out with two TMA tensor stores after a consumer barrier (two
// tiles alternate; the stores also clip ragged lane and time tiles).  Waits
// are bounded as in the forward kernels.
#include <algorithm>

#include "es_device.cuh"

// Tuning overrides (0, or -1 for the flag: chosen per shape in
// launch_lane_tma_bwd).
#ifndef ES_LANE_BWD_TT
#define ES_LANE_BWD_TT 0        // trips per tile: 16 or 32
#endif
#ifndef ES_LANE_BWD_STAGES
#define ES_LANE_BWD_STAGES 0    // pipeline depth
#endif
#ifndef ES_LANE_BWD_STAGED
#define ES_LANE_BWD_STAGED -1   // 1: gradients staged for TMA stores, 0: direct row stores
#endif

namespace es {
namespace {

constexpr int kMaxStages = 8;

template <int BODY, int LI, int TT, bool kStaged>
__global__ void __launch_bounds__(32 + LI)
k_lane_bwd(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_h,
           const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_x,
           const __grid_constant__ CUtensorMap map_gx, const __grid_constant__ CUtensorMap map_ga,
           const float* __restrict__ init, float* __restrict__ ginit, float* __restrict__ gx,
           float* __restrict__ ga, int T, int I, int tiles_i, int stages, int reverse, unsigned int* status,
           uint64_t wait_ns, int64_t drop_tile) {
    constexpr bool kNeedX = BODY == ES_BODY_MAXPLUS;
    constexpr int kRows = TT + 1;                        // state rows per tile
    constexpr int kTile = TT * LI;                       // floats of one per-trip stream
    constexpr int kStageFloats = (kNeedX ? 3 : 2) * kTile + kRows * LI;
    constexpr uint32_t kStageBytes = kStageFloats * 4u;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;

    float* tiles = reinterpret_cast<float*>(smem_raw + smem_align_pad(smem_raw));
    float* outs = tiles + static_cast<size_t>(stages) * kStageFloats;   // staged: [2][dx, da][TT][LI]
    const int o = blockIdx.x / tiles_i;
    const int i0 = (blockIdx.x % tiles_i) * LI;
    const int ntiles = (T + TT - 1) / TT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // backward visits time descending for a forward scan, ascending for a reverse one
    const bool desc = !reverse;

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
            tma_prefetch_desc(&map_g);
            tma_prefetch_desc(&map_h);
            tma_prefetch_desc(&map_a);
            if (kNeedX) tma_prefetch_desc(&map_x);
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
                const int j = desc ? ntiles - 1 - k : k;
                const int t0 = j * TT;
                float* st = tiles + s * kStageFloats;
                mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
                tma_load_3d(st, &map_g, i0, t0, o, &full_bar[s], pol);
                tma_load_3d(st + kTile, &map_a, i0, t0, o, &full_bar[s], pol);
                if (kNeedX) tma_load_3d(st + 2 * kTile, &map_x, i0, t0, o, &full_bar[s], pol);
                // states: rows t0-1 .. t0+TT-1 (forward scan) or t0 .. t0+TT (reverse scan)
                tma_load_3d(st + (kNeedX ? 3 : 2) * kTile, &map_h, i0, reverse ? t0 : t0 - 1, o, &full_bar[s], pol);
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
    const float p0 = valid ? init[static_cast<int64_t>(o) * I + i] : 0.0f;
    const int t_first = reverse ? T - 1 : 0;            // first trip in scan order: its p is initial
    const bool storer = kStaged && threadIdx.x == 32;
    float lam = 0.0f;
    const int64_t base = static_cast<int64_t>(o) * T * I + i;

    // Staged: one consumer barrier per tile votes on whether any consumer gave
    // up its wait and marks the previous tile's gradients complete in SMEM.
    // Direct: each warp leaves on its own vote.
    for (int k = 0; k < ntiles + (kStaged ? 1 : 0); ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if constexpr (kStaged) {
            // the buffer this tile writes was last read by the store issued a
            // tile ago: the storer waits for that read before the barrier
            if (storer) bulk_wait_read<0>();
            if (k > 0) fence_proxy_async_smem();     // this thread's gradient writes of tile k-1
            if (consumer_vote_any_failed(!ok, LI)) {
                if (!ok) report_timeout(status, &abort_flag);
                break;
            }
            if (storer && k > 0) {
                const int jp = desc ? ntiles - k : k - 1;
                const float* ob = outs + static_cast<size_t>((k - 1) & 1) * 2 * kTile;
                tma_store_3d(&map_gx, i0, jp * TT, o, ob);
                tma_store_3d(&map_ga, i0, jp * TT, o, ob + kTile);
                bulk_commit();
            }
            if (k == ntiles) break;
        } else {
            if (!__all_sync(0xffffffffu, ok)) {
                if (!ok) report_timeout(status, &abort_flag);
                break;
            }
        }
        const int j = desc ? ntiles - 1 - k : k;
        const int t0 = j * TT;
        const int n = min(TT, T - t0);
        const float* st = tiles + s * kStageFloats + c;
        float gr[TT], ar[TT], xr[kNeedX ? TT : 1], hr[kRows];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            gr[tt] = st[tt * LI];
            ar[tt] = st[kTile + tt * LI];
            if constexpr (kNeedX) xr[tt] = st[2 * kTile + tt * LI];
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) hr[r] = st[(kNeedX ? 3 : 2) * kTile + r * LI];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);

        // state row of trip tt is hr[tt + 1] (forward scan) or hr[tt] (reverse
        // scan); the state before it is the row next to it
        float* dxp = gx + base + static_cast<int64_t>(t0) * I;
        float* dap = ga + base + static_cast<int64_t>(t0) * I;
        float* ob = outs + static_cast<size_t>(k & 1) * 2 * kTile + c;
        auto trip = [&](const int tt) {
            const float h = reverse ? hr[tt] : hr[tt + 1];
            float p = reverse ? hr[tt + 1] : hr[tt];
            p = (t0 + tt == t_first) ? p0 : p;
            lam = __fadd_rn(lam, gr[tt]);
            float dx, da;
            if constexpr (BODY == ES_BODY_TANH_DECAY) {
                const float m = __fmul_rn(lam, __fsub_rn(1.0f, __fmul_rn(h, h)));
                dx = m;
                da = __fmul_rn(m, p);
                lam = __fmul_rn(m, ar[tt]);
            } else {
                maxplus_vjp(__fsub_rn(p, ar[tt]), xr[tt], lam, dx, da);
            }
            if constexpr (kStaged) {
                ob[tt * LI] = dx;
                ob[kTile + tt * LI] = da;
            } else if (valid) {
                __stcs(dxp + static_cast<int64_t>(tt) * I, dx);
                __stcs(dap + static_cast<int64_t>(tt) * I, da);
            }
        };
        // trips past T in a ragged tile (zero-filled) must not touch the
        // cotangent; a staged tile's TMA store clips them
        if (n == TT) {
            if (desc) {
#pragma unroll
                for (int tt = TT - 1; tt >= 0; --tt) trip(tt);
            } else {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) trip(tt);
            }
        } else if (desc) {
#pragma unroll
            for (int tt = TT - 1; tt >= 0; --tt)
                if (tt < n) trip(tt);
        } else {
#pragma unroll
            for (int tt = 0; tt < TT; ++tt)
                if (tt < n) trip(tt);
        }
    }
    if (storer) bulk_wait_all();
    if (valid) ginit[static_cast<int64_t>(o) * I + i] = lam;
}

// the launch's shape: lanes per CTA, trips per tile, stages, staged stores
struct BwdCfg {
    int LI, TT, stages;
    bool staged;
};

size_t bwd_smem(int body, const BwdCfg& c) {
    const size_t tile = static_cast<size_t>(c.TT) * c.LI;
    const size_t stage = (body == ES_BODY_MAXPLUS ? 3 : 2) * tile + static_cast<size_t>(c.TT + 1) * c.LI;
    return (c.stages * stage + (c.staged ? 4 * tile : 0)) * 4 + 1024;
}

template <int BODY, int LI, int TT, bool kStaged>
cudaError_t launch_bwd_cfg(const BackwardLaunch& B, const CUtensorMap* maps, int I, int tiles_i, int stages) {
    const Launch& L = B.fwd;
    const size_t smem = bwd_smem(BODY, BwdCfg{LI, TT, stages, kStaged});
    auto kern = k_lane_bwd<BODY, LI, TT, kStaged>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = L.O * tiles_i;
    kern<<<static_cast<unsigned>(grid), 32 + LI, smem, L.stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], L.init, B.ginit, B.gx, B.ga, static_cast<int>(L.T), I,
        tiles_i, stages, L.reverse, L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

template <int BODY, int LI>
cudaError_t launch_bwd_li(const BackwardLaunch& B, const CUtensorMap* maps, int I, int tiles_i, const BwdCfg& c) {
    if (c.staged) {
        if (c.TT == 32) return launch_bwd_cfg<BODY, LI, 32, true>(B, maps, I, tiles_i, c.stages);
        return launch_bwd_cfg<BODY, LI, 16, true>(B, maps, I, tiles_i, c.stages);
    }
    if (c.TT == 32) return launch_bwd_cfg<BODY, LI, 32, false>(B, maps, I, tiles_i, c.stages);
    return launch_bwd_cfg<BODY, LI, 16, false>(B, maps, I, tiles_i, c.stages);
}

template <int BODY>
cudaError_t launch_bwd_body(const BackwardLaunch& B, const CUtensorMap* maps, int I, int tiles_i, const BwdCfg& c) {
    if (c.LI == 128) return launch_bwd_li<BODY, 128>(B, maps, I, tiles_i, c);
    if (c.LI == 64) return launch_bwd_li<BODY, 64>(B, maps, I, tiles_i, c);
    return launch_bwd_li<BODY, 32>(B, maps, I, tiles_i, c);
}

bool encode_bwd(const Launch& L, CUtensorMap* m, const float* base, int64_t I, int LI, int rows, const char** err) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(L.T),
                                static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(I) * 4, static_cast<cuuint64_t>(I) * L.T * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(LI), static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = L.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for a backward tile map";
        return false;
    }
    return true;
}

}  // namespace

cudaError_t launch_lane_tma_bwd(const BackwardLaunch& B, const char** err) {
    const Launch& L = B.fwd;
    const int64_t I = L.J * L.W;
    int LI = 32;
    for (int cand : {128, 64}) {
        if (I >= cand && 5 * L.O * ((I + cand - 1) / cand) >= 4LL * L.num_sms) {
            LI = cand;
            break;
        }
    }
    const int64_t tiles_i = (I + LI - 1) / LI;
    const bool one_per_sm = L.O * tiles_i <= L.num_sms;
    // Where several CTAs share an SM, 16-trip tiles with the gradients staged
    // for TMA stores, as many stages as keep a CTA within about 100 KB (two a
    // SM); where there is at most one CTA a SM, direct row stores and four
    // 16-trip stages.
    BwdCfg c{LI, 16, 4, !one_per_sm};
    if (c.staged) {
        c.stages = 6;
        while (c.stages > 2 && bwd_smem(L.body, c) > 100 * 1024) --c.stages;
    }
    if (ES_LANE_BWD_TT != 0) c.TT = ES_LANE_BWD_TT;
    if (ES_LANE_BWD_STAGES != 0) c.stages = ES_LANE_BWD_STAGES;
    if (ES_LANE_BWD_STAGED >= 0) c.staged = ES_LANE_BWD_STAGED != 0;
    CUtensorMap maps[6];
    const float* x = L.body == ES_BODY_MAXPLUS ? L.x : L.a;   // TANH needs no x: map something valid
    if (!encode_bwd(L, &maps[0], B.gout, I, LI, c.TT, err) ||
        !encode_bwd(L, &maps[1], B.states, I, LI, c.TT + 1, err) || !encode_bwd(L, &maps[2], L.a, I, LI, c.TT, err) ||
        !encode_bwd(L, &maps[3], x, I, LI, c.TT, err) || !encode_bwd(L, &maps[4], B.gx, I, LI, c.TT, err) ||
        !encode_bwd(L, &maps[5], B.ga, I, LI, c.TT, err))
        return cudaErrorInvalidValue;
    const int Ii = static_cast<int>(I), ti = static_cast<int>(tiles_i);
    if (L.body == ES_BODY_TANH_DECAY) return launch_bwd_body<ES_BODY_TANH_DECAY>(B, maps, Ii, ti, c);
    return launch_bwd_body<ES_BODY_MAXPLUS>(B, maps, Ii, ti, c);
}

}  // namespace es
