// k_time_tma.cu -- element scan with the sequence axis innermost
// (ES_PATH_TIME_TMA, e.g. `:axis -1` on a [lanes, T] tensor).
//
// Each lane is one contiguous row of T values, so a warp reading "trip t of
// 32 lanes" directly would touch 32 rows.  Instead the CTA stages a tile of
// LO rows x 32 trips (box {32, LO} of a 2-D tensor map, one 128-byte segment
// per row) in SMEM through an S-stage TMA/mbarrier ring, with the 128-byte
// swizzle so that a thread reading its own row four trips at a time (one
// 16-byte vector) is conflict-free across the warp.  Each consumer thread owns
// one row: it copies its 32-trip segment of both sequences into registers,
// hands the input stage back to the producer at once (so every stage stays
// in flight while the chain runs), runs the serial body over the segment,
// and writes the states into a swizzled output tile; one thread stores the
// tile back with a TMA tensor store (three output buffers, so the stores
// overlap the next tiles).  Reverse scans take the tiles last-first and the
// four values of every vector in descending order.  Waits are bounded as in
// the other pipelines.
#include <algorithm>

#include "es_device.cuh"

namespace es {
namespace {

constexpr int kTT = 32;            // trips per tile: 128 bytes per row (swizzle span)
constexpr int kMaxStages = 6;

// Tuning overrides (0: chosen per shape in launch_time_tma).
#ifndef ES_TIME_LO
#define ES_TIME_LO 64       // rows (lanes) per CTA: 64 or 128
#endif
#ifndef ES_TIME_STAGES
#define ES_TIME_STAGES 0    // pipeline depth
#endif
constexpr int kOutBufs = 3;

template <int BODY>
__device__ __forceinline__ void run_vec(float& h, const float4 xv, const float4 av, float4& ov, bool reverse) {
    if (!reverse) {
        h = step_pointwise<BODY>(h, xv.x, av.x); ov.x = h;
        h = step_pointwise<BODY>(h, xv.y, av.y); ov.y = h;
        h = step_pointwise<BODY>(h, xv.z, av.z); ov.z = h;
        h = step_pointwise<BODY>(h, xv.w, av.w); ov.w = h;
    } else {
        h = step_pointwise<BODY>(h, xv.w, av.w); ov.w = h;
        h = step_pointwise<BODY>(h, xv.z, av.z); ov.z = h;
        h = step_pointwise<BODY>(h, xv.y, av.y); ov.y = h;
        h = step_pointwise<BODY>(h, xv.x, av.x); ov.x = h;
    }
}

template <int BODY, int LO>
__global__ void __launch_bounds__(32 + LO)
k_time_tma(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_a,
           const __grid_constant__ CUtensorMap map_out, const float* __restrict__ init, int O, int T, int stages,
           int reverse, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;

    // every tile is LO rows x 128 bytes and starts on a 1024-byte boundary
    constexpr uint32_t kTileBytes = LO * 128u;
    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    unsigned char* in_tiles = base;                                   // [stages][2][LO][128 B]
    unsigned char* out_tiles = base + static_cast<size_t>(stages) * 2 * kTileBytes;  // [3][LO][128 B]

    const int o0 = blockIdx.x * LO;
    const int ntiles = (T + kTT - 1) / kTT;
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
                unsigned char* xs = in_tiles + static_cast<size_t>(s) * 2 * kTileBytes;
                mbar_arrive_expect_tx(&full_bar[s], 2 * kTileBytes);
                tma_load_2d(xs, &map_x, j * kTT, o0, &full_bar[s], pol);
                tma_load_2d(xs + kTileBytes, &map_a, j * kTT, o0, &full_bar[s], pol);
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
    float h = valid ? init[o0 + r] : 0.0f;
    const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
    const uint32_t sw = static_cast<uint32_t>(r & 7);   // 128-byte swizzle: chunk q lives at q ^ (row % 8)
    const bool storer = (threadIdx.x == 32);

    // One consumer barrier per tile does two jobs: it is the vote on whether
    // any consumer gave up its wait (so all leave together and no barrier is
    // left waiting), and it marks the previous tile's output as complete.
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
            tma_store_2d(&map_out, jp * kTT, o0, out_tiles + static_cast<size_t>((k - 1) % kOutBufs) * kTileBytes);
            bulk_commit();
            // the buffer written at the next tile was read out by an older store
            bulk_wait_read<1>();
        }
        if (k == ntiles) break;
        const int j = reverse ? ntiles - 1 - k : k;
        const int t0 = j * kTT;
        const int nq = min(kTT, T - t0) >> 2;     // T % 4 == 0 on this path
        const unsigned char* xrow = in_tiles + static_cast<size_t>(s) * 2 * kTileBytes + row_off;
        const unsigned char* arow = xrow + kTileBytes;
        unsigned char* orow = out_tiles + static_cast<size_t>(k % kOutBufs) * kTileBytes + row_off;
        // the row's whole segment goes to registers first, then the serial chain
        float4 xv[kTT / 4], av[kTT / 4];
#pragma unroll
        for (int q = 0; q < kTT / 4; ++q) {
            const uint32_t off = ((static_cast<uint32_t>(q) ^ sw) << 4);
            xv[q] = *reinterpret_cast<const float4*>(xrow + off);
            av[q] = *reinterpret_cast<const float4*>(arow + off);
        }
        // the input stage is free as soon as the segment sits in registers
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        auto quad = [&](const int q, const bool rev) {
            float4 ov;
            run_vec<BODY>(h, xv[q], av[q], ov, rev);
            *reinterpret_cast<float4*>(orow + ((static_cast<uint32_t>(q) ^ sw) << 4)) = ov;
        };
        // full tiles run unguarded (one basic block); only a ragged last tile
        // checks every group of four trips
        if (nq == kTT / 4) {
            if (!reverse) {
#pragma unroll
                for (int q = 0; q < kTT / 4; ++q) quad(q, false);
            } else {
#pragma unroll
                for (int q = kTT / 4 - 1; q >= 0; --q) quad(q, true);
            }
        } else if (!reverse) {
#pragma unroll
            for (int q = 0; q < kTT / 4; ++q)
                if (q < nq) quad(q, false);
        } else {
#pragma unroll
            for (int q = kTT / 4 - 1; q >= 0; --q)
                if (q < nq) quad(q, true);
        }
    }
    if (storer) bulk_wait_all();
}

template <int BODY, int LO>
cudaError_t launch_lo(const Launch& L, const CUtensorMap& mx, const CUtensorMap& ma, const CUtensorMap& mo,
                      int stages) {
    const size_t smem = (static_cast<size_t>(stages) * 2 + kOutBufs) * LO * 128 + 1024;
    auto kern = k_time_tma<BODY, LO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = (L.O + LO - 1) / LO;
    kern<<<static_cast<unsigned>(grid), 32 + LO, smem, L.stream>>>(mx, ma, mo, L.init, static_cast<int>(L.O),
                                                                   static_cast<int>(L.T), stages, L.reverse,
                                                                   L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

bool encode_time_rows(const Launch& L, CUtensorMap* m, const float* base, int LO, const char** err) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.T), static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.T) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTT), static_cast<cuuint32_t>(LO)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = L.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for the time-innermost tile map";
        return false;
    }
    return true;
}

}  // namespace

bool time_tma_ok(int body, int64_t O, int64_t T, int64_t J, int64_t W, const int64_t sw[2],
                 const void* const ptrs[4]) {
    if (body == ES_BODY_NORMCAP) return false;
    if (J * W != 1 || sw[0] != 1 || sw[1] != 1) return false;
    if (T % 4 != 0 || T < kTT) return false;                   // 16-byte row stride
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31)) return false;
    for (int k = 1; k < 4; ++k)
        if (reinterpret_cast<uintptr_t>(ptrs[k]) % 16 != 0) return false;
    return true;
}

cudaError_t launch_time_tma(const Launch& L, const char** err) {
    constexpr int LO = ES_TIME_LO;
    const int64_t ctas = (L.O + LO - 1) / LO;
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(3, (ctas + L.num_sms - 1) / L.num_sms));
    const int64_t budget = (210 * 1024) / per_sm - kOutBufs * LO * 128 - 1024;
    const int64_t stage_bytes = 2LL * LO * 128;
    int stages = static_cast<int>(std::max<int64_t>(2, std::min<int64_t>(kMaxStages, budget / stage_bytes)));
    if (ES_TIME_STAGES != 0) stages = ES_TIME_STAGES;
    CUtensorMap mx, ma, mo;
    if (!encode_time_rows(L, &mx, L.x, LO, err) || !encode_time_rows(L, &ma, L.a, LO, err) ||
        !encode_time_rows(L, &mo, L.out, LO, err))
        return cudaErrorInvalidValue;
    if (L.body == ES_BODY_TANH_DECAY) return launch_lo<ES_BODY_TANH_DECAY, LO>(L, mx, ma, mo, stages);
    return launch_lo<ES_BODY_MAXPLUS, LO>(L, mx, ma, mo, stages);
}

}  // namespace es
