// k_time_bwd.cu -- backward pass of TANH_DECAY / MAXPLUS with the sequence
// axis innermost (ES_PATH_TIME_TMA for es_scan_backward_f32).
//
// "Nonlinear element scans", "Precision and gradients": the gradient is an
// element scan in the opposite trip order applying the body's
// vector-Jacobian product once a trip (TANH_DECAY: m = lam (1 - h^2),
// dx = m, da = m p, lam <- m a; MAXPLUS: the larger of p - c and x takes lam,
// a tie splits it).
//
// Each lane is a row of T values.  Per tile of 64 rows x 32 trips the
// producer streams, with TMA, the output gradient, the second sequence and
// (MAXPLUS) x as 128-byte-swizzled boxes {32, 64} (conflict-free 16-byte
// reads of a thread's own row), and the saved states as an unswizzled box
// {36, 64} whose 144-byte rows also read conflict-free: trips t0-4 .. t0+31
// for a forward scan, t0 .. t0+35 for a reverse one, so the state before
// each trip of the tile is in the same box (columns outside 0..T-1 are
// zero-filled and `initial` takes the first trip's place).  Each thread owns
// one row: it copies its segments to registers, frees the input stage, runs
// the chain over its 32 trips in backward order and writes dx and da into
// swizzled output tiles that one thread stores with TMA tensor stores (three
// buffers each).  One consumer barrier per tile votes on give-ups and marks
// the previous tile's outputs complete, as in the forward time kernel.
#include <algorithm>

#include "es_device.cuh"

namespace es {
namespace {

constexpr int kTT = 32;
constexpr int kHCols = 36;          // state columns per tile row
constexpr int kLO = 64;             // rows per CTA
constexpr int kOutBufs = 3;
constexpr int kMaxStages = 4;

template <int BODY>
__global__ void __launch_bounds__(32 + kLO)
k_time_bwd(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_a,
           const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_h,
           const __grid_constant__ CUtensorMap map_gx, const __grid_constant__ CUtensorMap map_ga,
           const float* __restrict__ init, float* __restrict__ ginit, int O, int T, int stages, int reverse,
           unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    constexpr bool kNeedX = BODY == ES_BODY_MAXPLUS;
    constexpr uint32_t kTile = kLO * 128u;                      // one swizzled {32, 64} tile
    constexpr uint32_t kHTile = kLO * kHCols * 4u;              // 9216 bytes
    constexpr uint32_t kOffH = (kNeedX ? 3u : 2u) * kTile;
    constexpr uint32_t kStage = (kOffH + kHTile + 1023u) & ~1023u;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;

    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    unsigned char* out_tiles = base + static_cast<size_t>(stages) * kStage;   // [2][3][64 rows x 128 B]
    const int o0 = blockIdx.x * kLO;
    const int ntiles = (T + kTT - 1) / kTT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool desc = !reverse;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kLO / 32);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&map_g);
            tma_prefetch_desc(&map_a);
            tma_prefetch_desc(&map_h);
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
                const int t0 = (desc ? ntiles - 1 - k : k) * kTT;
                unsigned char* st = base + static_cast<size_t>(s) * kStage;
                mbar_arrive_expect_tx(&full_bar[s], kOffH + kHTile);
                tma_load_2d(st, &map_g, t0, o0, &full_bar[s], pol);
                tma_load_2d(st + kTile, &map_a, t0, o0, &full_bar[s], pol);
                if (kNeedX) tma_load_2d(st + 2 * kTile, &map_x, t0, o0, &full_bar[s], pol);
                tma_load_2d(st + kOffH, &map_h, reverse ? t0 : t0 - 4, o0, &full_bar[s], pol);
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    const int r = threadIdx.x - 32;
    const bool valid = o0 + r < O;
    const float p0 = valid ? init[o0 + r] : 0.0f;
    const int t_first = reverse ? T - 1 : 0;
    float lam = 0.0f;
    const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    const bool storer = (threadIdx.x == 32);

    for (int k = 0; k <= ntiles; ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (k > 0) fence_proxy_async_smem();
        if (consumer_vote_any_failed(!ok, kLO)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        if (storer && k > 0) {
            const int tp = (desc ? ntiles - k : k - 1) * kTT;
            const size_t b = static_cast<size_t>((k - 1) % kOutBufs) * kTile;
            tma_store_2d(&map_gx, tp, o0, out_tiles + b);
            tma_store_2d(&map_ga, tp, o0, out_tiles + kOutBufs * kTile + b);
            bulk_commit();
            bulk_wait_read<1>();
        }
        if (k == ntiles) break;
        const int t0 = (desc ? ntiles - 1 - k : k) * kTT;
        const int n = min(kTT, T - t0);
        const unsigned char* st = base + static_cast<size_t>(s) * kStage;
        float gr[kTT], ar[kTT], xr[kNeedX ? kTT : 1], hr[kHCols];
#pragma unroll
        for (int q = 0; q < kTT / 4; ++q) {
            const uint32_t off = row_off + ((static_cast<uint32_t>(q) ^ sw) << 4);
            const float4 g4 = *reinterpret_cast<const float4*>(st + off);
            const float4 a4 = *reinterpret_cast<const float4*>(st + kTile + off);
            gr[4 * q] = g4.x; gr[4 * q + 1] = g4.y; gr[4 * q + 2] = g4.z; gr[4 * q + 3] = g4.w;
            ar[4 * q] = a4.x; ar[4 * q + 1] = a4.y; ar[4 * q + 2] = a4.z; ar[4 * q + 3] = a4.w;
            if constexpr (kNeedX) {
                const float4 x4 = *reinterpret_cast<const float4*>(st + 2 * kTile + off);
                xr[4 * q] = x4.x; xr[4 * q + 1] = x4.y; xr[4 * q + 2] = x4.z; xr[4 * q + 3] = x4.w;
            }
        }
#pragma unroll
        for (int q = 0; q < kHCols / 4; ++q) {
            const float4 h4 = *reinterpret_cast<const float4*>(st + kOffH + static_cast<uint32_t>(r) * (kHCols * 4) + 16 * q);
            hr[4 * q] = h4.x; hr[4 * q + 1] = h4.y; hr[4 * q + 2] = h4.z; hr[4 * q + 3] = h4.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);

        unsigned char* ox = out_tiles + static_cast<size_t>(k % kOutBufs) * kTile + row_off;
        unsigned char* oa = out_tiles + static_cast<size_t>(kOutBufs + k % kOutBufs) * kTile + row_off;
        float dxr[kTT], dar[kTT];
        auto trip = [&](const int tt) {
            // own state and the state before the trip inside the 36-column box
            const float h = reverse ? hr[tt] : hr[tt + 4];
            float p = reverse ? hr[tt + 1] : hr[tt + 3];
            p = (t0 + tt == t_first) ? p0 : p;
            lam = __fadd_rn(lam, gr[tt]);
            if constexpr (BODY == ES_BODY_TANH_DECAY) {
                const float m = __fmul_rn(lam, __fsub_rn(1.0f, __fmul_rn(h, h)));
                dxr[tt] = m;
                dar[tt] = __fmul_rn(m, p);
                lam = __fmul_rn(m, ar[tt]);
            } else {
                maxplus_vjp(__fsub_rn(p, ar[tt]), xr[tt], lam, dxr[tt], dar[tt]);
            }
        };
        if (n == kTT) {
            if (desc) {
#pragma unroll
                for (int tt = kTT - 1; tt >= 0; --tt) trip(tt);
            } else {
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt) trip(tt);
            }
        } else if (desc) {
#pragma unroll
            for (int tt = kTT - 1; tt >= 0; --tt)
                if (tt < n) trip(tt);
        } else {
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt)
                if (tt < n) trip(tt);
        }
#pragma unroll
        for (int q = 0; q < kTT / 4; ++q) {
            const uint32_t off = ((static_cast<uint32_t>(q) ^ sw) << 4);
            *reinterpret_cast<float4*>(ox + off) = make_float4(dxr[4 * q], dxr[4 * q + 1], dxr[4 * q + 2], dxr[4 * q + 3]);
            *reinterpret_cast<float4*>(oa + off) = make_float4(dar[4 * q], dar[4 * q + 1], dar[4 * q + 2], dar[4 * q + 3]);
        }
    }
    if (storer) bulk_wait_all();
    if (valid) ginit[o0 + r] = lam;
}

bool encode_tb(const Launch& L, CUtensorMap* m, const void* base, int cols, bool swizzle, const char** err) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.T), static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.T) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), static_cast<cuuint32_t>(kLO)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = L.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for a time-innermost backward tile map";
        return false;
    }
    return true;
}

template <int BODY>
cudaError_t launch_tb(const BackwardLaunch& B, const CUtensorMap* maps, int stages) {
    const Launch& L = B.fwd;
    constexpr bool kNeedX = BODY == ES_BODY_MAXPLUS;
    constexpr size_t kTile = kLO * 128;
    constexpr size_t kStage = (((kNeedX ? 3 : 2) * kTile + kLO * kHCols * 4) + 1023) & ~size_t(1023);
    const size_t smem = static_cast<size_t>(stages) * kStage + 2 * kOutBufs * kTile + 1024;
    auto kern = k_time_bwd<BODY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = (L.O + kLO - 1) / kLO;
    kern<<<static_cast<unsigned>(grid), 32 + kLO, smem, L.stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], L.init, B.ginit, static_cast<int>(L.O),
        static_cast<int>(L.T), stages, L.reverse, L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_time_tma_bwd(const BackwardLaunch& B, const char** err) {
    const Launch& L = B.fwd;
    const int stages = 2;
    CUtensorMap maps[6];
    const float* x = L.body == ES_BODY_MAXPLUS ? L.x : L.a;   // TANH reads no x: map something valid
    if (!encode_tb(L, &maps[0], B.gout, kTT, true, err) || !encode_tb(L, &maps[1], L.a, kTT, true, err) ||
        !encode_tb(L, &maps[2], x, kTT, true, err) || !encode_tb(L, &maps[3], B.states, kHCols, false, err) ||
        !encode_tb(L, &maps[4], B.gx, kTT, true, err) || !encode_tb(L, &maps[5], B.ga, kTT, true, err))
        return cudaErrorInvalidValue;
    if (L.body == ES_BODY_TANH_DECAY) return launch_tb<ES_BODY_TANH_DECAY>(B, maps, stages);
    return launch_tb<ES_BODY_MAXPLUS>(B, maps, stages);
}

}  // namespace es
