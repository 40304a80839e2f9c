// k_lane_tma.cu -- element scan with the lanes innermost (ES_PATH_LANE_TMA).
//
// Canonical view [O, T, I] with I = J*W contiguous lanes per trip row
// ("Nonlinear element scans": every lane is an independent recurrence; lanes
// run in parallel and trips in sequence).  One CTA owns a tile of LI adjacent
// lanes of one o and walks all T trips:
//   * warp 0, lane 0 is the producer: it streams time tiles of TT trips of
//     both sequences (box {LI, TT, 1} of a 3-D tensor map) into an S-stage
//     SMEM ring with TMA, each stage guarded by a full / empty mbarrier pair;
//   * LI consumer threads (one per lane) copy a whole tile into registers
//     (conflict-free SMEM reads), hand the stage back to the producer at
//     once, then run the serial body over the tile with the state in a
//     register, one coalesced 4*LI-byte store per trip and warp.
// Handing the stage back before the serial chain runs keeps all S stages in
// flight while the warp computes, so HBM latency hides behind the chain.
// Reverse scans walk the tiles from last to first and each tile bottom-up, so
// no flipped copy is ever made (reverse paragraph of the page).  A ragged
// last tile is zero-filled by TMA and only its valid rows are used.  Every
// wait is bounded: on give-up the CTA records ES_DEVICE_TIMEOUT, the producer
// waits (bounded) for its copies in flight, and all threads return.
#include <algorithm>

#include "es_device.cuh"

// Tuning overrides (0: chosen per shape in launch_lane_tma).
#ifndef ES_LANE_TT
#define ES_LANE_TT 0        // trips per tile: 16 or 32
#endif
#ifndef ES_LANE_LI
#define ES_LANE_LI 0        // lanes per CTA: 32, 64 or 128
#endif
#ifndef ES_LANE_STAGES
#define ES_LANE_STAGES 0    // pipeline depth
#endif

namespace es {
namespace {

constexpr int kMaxStages = 8;

template <int BODY, int LI, int TT>
__global__ void __launch_bounds__(32 + LI)
k_lane_tma(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_a,
           const float* __restrict__ init, float* __restrict__ out, int T, int I, int tiles_i,
           int stages, int reverse, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;

    float* tiles = reinterpret_cast<float*>(smem_raw + smem_align_pad(smem_raw));
    constexpr int kTileFloats = TT * LI;            // one sequence, one stage
    constexpr uint32_t kStageBytes = 2u * kTileFloats * 4u;

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
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_a);
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
                float* xs = tiles + s * 2 * kTileFloats;
                mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
                tma_load_3d(xs, &map_x, i0, j * TT, o, &full_bar[s], pol);
                tma_load_3d(xs + kTileFloats, &map_a, i0, j * TT, o, &full_bar[s], pol);
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
    float h = valid ? init[static_cast<int64_t>(o) * I + i] : 0.0f;
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
        const float* xs = tiles + s * 2 * kTileFloats + c;
        const float* as = xs + kTileFloats;
        // the whole tile goes to registers first: the loads overlap each other
        // and the serial chain below only waits on arithmetic
        float xr[TT], ar[TT];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            xr[tt] = xs[tt * LI];
            ar[tt] = as[tt * LI];
        }
        // the stage is free as soon as the tile sits in registers, so the
        // producer refills it while this warp runs the chain
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        float* op = obase + static_cast<int64_t>(t0) * I;
        // The state alternates between two registers (by trip parity), so a
        // trip never overwrites the register the previous trip's store may
        // still be reading.  Consecutive trips alternate parity in both
        // directions; the last trip is n-1 forward and 0 in reverse.
        float hv[2] = {h, h};
        auto trip = [&](const int tt) {
            hv[tt & 1] = step_pointwise<BODY>(hv[(tt & 1) ^ 1], xr[tt], ar[tt]);
            if (valid) __stcs(op + static_cast<int64_t>(tt) * I, hv[tt & 1]);
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

template <int BODY, int LI, int TT>
cudaError_t launch_cfg(const Launch& L, const CUtensorMap& mx, const CUtensorMap& ma, int I, int tiles_i,
                       int stages) {
    const size_t smem = static_cast<size_t>(stages) * 2 * TT * LI * 4 + 1024;
    auto kern = k_lane_tma<BODY, LI, TT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = L.O * tiles_i;
    kern<<<static_cast<unsigned>(grid), 32 + LI, smem, L.stream>>>(
        mx, ma, L.init, L.out, static_cast<int>(L.T), I, tiles_i, stages, L.reverse, L.status, L.wait_ns,
        L.drop_tile);
    return cudaGetLastError();
}

template <int BODY, int TT>
cudaError_t launch_tt(const Launch& L, const CUtensorMap& mx, const CUtensorMap& ma, int I, int tiles_i,
                      int stages, int LI) {
    if (LI == 256) return launch_cfg<BODY, 256, TT>(L, mx, ma, I, tiles_i, stages);
    if (LI == 128) return launch_cfg<BODY, 128, TT>(L, mx, ma, I, tiles_i, stages);
    if (LI == 64) return launch_cfg<BODY, 64, TT>(L, mx, ma, I, tiles_i, stages);
    return launch_cfg<BODY, 32, TT>(L, mx, ma, I, tiles_i, stages);
}

template <int BODY>
cudaError_t launch_body(const Launch& L, const CUtensorMap& mx, const CUtensorMap& ma, int I, int tiles_i,
                        int stages, int LI, int TT) {
    if (TT == 32) return launch_tt<BODY, 32>(L, mx, ma, I, tiles_i, stages, LI);
    return launch_tt<BODY, 16>(L, mx, ma, I, tiles_i, stages, LI);
}

bool encode_rows(const Launch& L, CUtensorMap* m, const float* base, int64_t I, int LI, int TT, const char** err) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(L.T),
                                static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(I) * 4, static_cast<cuuint64_t>(I) * L.T * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(LI), static_cast<cuuint32_t>(TT), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = L.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for the lane-innermost tile map";
        return false;
    }
    return true;
}

}  // namespace

bool lane_tma_ok(int body, int64_t O, int64_t T, int64_t J, int64_t W, const int64_t sw[2],
                 const void* const ptrs[4]) {
    if (body == ES_BODY_NORMCAP) return false;
    if (W > 1 && (sw[0] != W || sw[1] != W)) return false;   // broadcast sequences: generic path
    const int64_t I = J * W;
    if (I < 32 || I % 4 != 0) return false;                  // 16-byte row stride, box <= row
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || I >= (int64_t(1) << 31)) return false;
    if (O * ((I + 31) / 32) >= (int64_t(1) << 31)) return false;
    for (int k = 1; k < 4; ++k)
        if (reinterpret_cast<uintptr_t>(ptrs[k]) % 16 != 0) return false;
    return true;
}

cudaError_t launch_lane_tma(const Launch& L, const char** err) {
    const int64_t I = L.J * L.W;
    // Lanes per CTA: the widest tile (longest contiguous row segment per TMA
    // box row, the friendliest pattern for HBM) that still puts a CTA on most
    // SMs.
    int LI = 32;
    for (int cand : {256, 128, 64}) {
        if (I >= cand && 5 * L.O * ((I + cand - 1) / cand) >= 4LL * L.num_sms) {
            LI = cand;
            break;
        }
    }
    if (ES_LANE_LI != 0 && I >= ES_LANE_LI) LI = ES_LANE_LI;
    const int64_t tiles_i = (I + LI - 1) / LI;
    // Pipeline depth: about 96 trips of both sequences in flight per CTA
    // (three 32-trip stages), measured best on GB300 for both one CTA per
    // SM (few lanes) and several (many lanes, even when not all CTAs fit at
    // once); 16-trip tiles only when 32-trip stages would not fit twice.
    // 256-lane tiles (1 KB row segments, one CTA a SM) measured best with two
    // 32-trip stages: 0.502 against 0.517 ms for 128-lane tiles on
    // [64, 4096, 1024], three stages 0.511.
    int TT = 32;
    int stages = 3;
    if (LI == 256) {
        stages = 2;
    } else if (2LL * 32 * LI * 4 * 3 > 200 * 1024) {
        TT = 16;
        stages = 6;
    }
    if (ES_LANE_TT != 0) TT = ES_LANE_TT;
    if (ES_LANE_STAGES != 0) stages = ES_LANE_STAGES;
    CUtensorMap mx, ma;
    if (!encode_rows(L, &mx, L.x, I, LI, TT, err) || !encode_rows(L, &ma, L.a, I, LI, TT, err))
        return cudaErrorInvalidValue;
    const int Ii = static_cast<int>(I), ti = static_cast<int>(tiles_i);
    if (L.body == ES_BODY_TANH_DECAY) return launch_body<ES_BODY_TANH_DECAY>(L, mx, ma, Ii, ti, stages, LI, TT);
    return launch_body<ES_BODY_MAXPLUS>(L, mx, ma, Ii, ti, stages, LI, TT);
}

}  // namespace es
