// k_vec_tma.cu -- NORMCAP with a vector state (ES_PATH_VEC_TMA).
//
// "Nonlinear element scans", :state-axis example: each lane carries W values
// (W in {2, 4, 8, 16}) and every trip computes y = a*h + x with a per-trip
// gate `a` (width 1, broadcast over the state, or width W), then
// h = y / max(1, ||y||_2).
//
// Canonical view: x and out are [O, T, J*W], the gate is [O, T, J*gw].  One
// CTA owns LV = 128 / W adjacent lanes of one o (128 contiguous values per
// trip) and walks all T trips.  Warp 0's lane 0 streams time tiles of TT
// trips of x and of the gate into an S-stage SMEM ring with TMA (full/empty
// mbarrier pairs); each of the 128 consumer threads holds one state value.
// The norm is a butterfly of W/2 .. 1 xor-shuffles inside each W-thread group
// (every thread of a group ends with the same bitwise sum, because each level
// adds the same two operands), then a correctly rounded sqrt, the floor at
// one, and a correctly rounded division.  Stores are one coalesced 512-byte
// row per trip.  Waits are bounded as in the other pipelines.
#include <algorithm>

#include "es_device.cuh"

namespace es {
namespace {

constexpr int kTT = 16;
constexpr int kMaxStages = 8;
constexpr int kThreads = 128;     // consumer threads = values per CTA row

template <int W>
__global__ void __launch_bounds__(32 + kThreads)
k_vec_tma(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_g,
          const float* __restrict__ init, float* __restrict__ out, int T, int J, int gw, int tiles_j, int stages,
          int reverse, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    constexpr int LV = kThreads / W;               // lanes per CTA
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;

    const int gl = LV * gw;                        // gate floats per trip row
    const uint32_t x_bytes = kTT * kThreads * 4;
    const uint32_t g_bytes = static_cast<uint32_t>(kTT * gl * 4);
    const uint32_t g_pad = (g_bytes + 1023u) & ~1023u;
    const uint32_t stage_bytes = x_bytes + g_pad;
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int o = blockIdx.x / tiles_j;
    const int j0 = (blockIdx.x % tiles_j) * LV;
    const int ntiles = (T + kTT - 1) / kTT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kThreads / 32);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_g);
            const uint64_t pol = l2_policy_evict_first();
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
                unsigned char* xs = base + static_cast<size_t>(s) * stage_bytes;
                mbar_arrive_expect_tx(&full_bar[s], x_bytes + g_bytes);
                tma_load_3d(xs, &map_x, j0 * W, j * kTT, o, &full_bar[s], pol);
                tma_load_3d(xs + x_bytes, &map_g, j0 * gw, j * kTT, o, &full_bar[s], pol);
            }
            volatile int never = 0;
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, &never))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    // consumers: thread c holds value w of lane j0 + v
    const int c = threadIdx.x - 32;
    const int v = c / W;
    const int w = c % W;
    const bool valid = j0 + v < J;
    const int64_t row = static_cast<int64_t>(J) * W;           // values per trip row
    float h = valid ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w] : 0.0f;
    float* obase = out + static_cast<int64_t>(o) * T * row + static_cast<int64_t>(j0) * W + c;
    const int gi = v * gw + (gw == 1 ? 0 : w);

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int j = reverse ? ntiles - 1 - k : k;
        const int t0 = j * kTT;
        const int n = min(kTT, T - t0);
        const float* xs = reinterpret_cast<const float*>(base + static_cast<size_t>(s) * stage_bytes) + c;
        const float* gs = reinterpret_cast<const float*>(base + static_cast<size_t>(s) * stage_bytes + x_bytes) + gi;
        float* op = obase + static_cast<int64_t>(t0) * row;
        for (int q = 0; q < n; ++q) {
            const int tt = reverse ? n - 1 - q : q;
            const float xv = xs[tt * kThreads];
            const float g = gs[tt * gl];
            const float y = __fadd_rn(__fmul_rn(g, h), xv);
            float ss = __fmul_rn(y, y);
#pragma unroll
            for (int off = W / 2; off >= 1; off >>= 1)
                ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
            const float d = ieee_maximum(1.0f, __fsqrt_rn(ss));
            h = __fdiv_rn(y, d);
            if (valid) __stcs(op + static_cast<int64_t>(tt) * row, h);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
}

template <int W>
cudaError_t launch_w(const Launch& L, const CUtensorMap& mx, const CUtensorMap& mg, int gw, int tiles_j,
                     int stages, size_t stage_bytes) {
    const size_t smem = static_cast<size_t>(stages) * stage_bytes + 1024;
    auto kern = k_vec_tma<W>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = L.O * tiles_j;
    kern<<<static_cast<unsigned>(grid), 32 + kThreads, smem, L.stream>>>(
        mx, mg, L.init, L.out, static_cast<int>(L.T), static_cast<int>(L.J), gw, tiles_j, stages, L.reverse,
        L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

bool encode_vec(const Launch& L, CUtensorMap* m, const float* base, int64_t row, int box_inner, const char** err) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row), static_cast<cuuint64_t>(L.T),
                                static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row) * 4, static_cast<cuuint64_t>(row) * L.T * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(kTT), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = L.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for the vector-state tile map";
        return false;
    }
    return true;
}

}  // namespace

bool vec_tma_ok(int body, int64_t O, int64_t T, int64_t J, int64_t W, const int64_t sw[2],
                const void* const ptrs[4]) {
    if (body != ES_BODY_NORMCAP) return false;
    if (W != 2 && W != 4 && W != 8 && W != 16) return false;
    if (sw[0] != W || (sw[1] != 1 && sw[1] != W)) return false;
    const int64_t LV = kThreads / W;
    if (J < LV) return false;                               // a tile never exceeds the row
    if ((J * sw[1]) % 4 != 0 || (LV * sw[1]) % 4 != 0) return false;   // 16-byte strides and boxes
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || J * W >= (int64_t(1) << 31)) return false;
    if (O * ((J + LV - 1) / LV) >= (int64_t(1) << 31)) return false;
    for (int k = 1; k < 4; ++k)
        if (reinterpret_cast<uintptr_t>(ptrs[k]) % 16 != 0) return false;
    return true;
}

cudaError_t launch_vec_tma(const Launch& L, const char** err) {
    const int W = static_cast<int>(L.W);
    const int gw = static_cast<int>(L.sw[1]);
    const int LV = kThreads / W;
    const int64_t tiles_j = (L.J + LV - 1) / LV;
    const int64_t ctas = L.O * tiles_j;
    const size_t x_bytes = static_cast<size_t>(kTT) * kThreads * 4;
    const size_t g_bytes = static_cast<size_t>(kTT) * LV * gw * 4;
    const size_t stage_bytes = x_bytes + ((g_bytes + 1023) & ~size_t(1023));
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(8, (ctas + L.num_sms - 1) / L.num_sms));
    const int64_t budget = std::min<int64_t>(96 * 1024, (200 * 1024) / per_sm);
    const int stages = static_cast<int>(
        std::max<int64_t>(2, std::min<int64_t>(kMaxStages, budget / static_cast<int64_t>(stage_bytes))));
    CUtensorMap mx, mg;
    if (!encode_vec(L, &mx, L.x, L.J * W, kThreads, err) || !encode_vec(L, &mg, L.a, L.J * gw, LV * gw, err))
        return cudaErrorInvalidValue;
    const int tj = static_cast<int>(tiles_j);
    switch (W) {
        case 2: return launch_w<2>(L, mx, mg, gw, tj, stages, stage_bytes);
        case 4: return launch_w<4>(L, mx, mg, gw, tj, stages, stage_bytes);
        case 8: return launch_w<8>(L, mx, mg, gw, tj, stages, stage_bytes);
        default: return launch_w<16>(L, mx, mg, gw, tj, stages, stage_bytes);
    }
}

}  // namespace es
