// k_vec_bwd.cu -- backward pass of NORMCAP with a vector state
// (ES_PATH_VEC_TMA for es_scan_backward_f32).
//
// "Nonlinear element scans", "Precision and gradients": the gradient is an
// element scan in the opposite trip order applying the body's
// vector-Jacobian product once a trip.  For y = a*p + x, h = y / max(1, |y|)
// and the state cotangent lam (after lam += dL/dh):
//   |y| <= 1:  mu = lam
//   |y| >  1:  mu = (lam - h (h . lam)) / |y|
//   dx = mu,  da = mu * p (summed over the state for a width-one gate),
//   lam <- a * mu.
// Only (h . lam) sits on the serial chain: |y| and the gate gradient depend
// on the saved states, the inputs and mu alone.  1/|y| comes from the
// hardware reciprocal square root of |y|^2 (relative error below 2^-22) and
// is multiplied in, the same value as the division up to rounding; sums over
// a lane are pairwise within a thread, then xor-shuffles across the lane's
// W/E threads, as in the forward vector kernel.
//
// Layout as in the forward vector kernel (x, states, grad_out, grad_x are
// [O, T, J*W]; the gate and its gradient [O, T, J*gw]).  A CTA owns the
// lanes of CW consumer warps (E values a thread, 32*CW*E values a trip row)
// and its warps split the work of each time tile of TT trips:
//   * the producer streams grad_out, x, the gate and TT+1 rows of saved
//     states (the tile's outputs and the state before its first trip in scan
//     order, from a box that may start at row -1 or end at row T, zero-filled
//     there; `initial` replaces it) into a stage ring with TMA;
//   * a helper warp per chain warp forms each trip's 1/|y| and cap flag ahead
//     of the chain (written over the trip's x values in the stage), and after
//     the chain the gate gradients sum(mu * p) (written over the gate);
//   * the chain warps run the cotangent recurrence alone, reading each trip's
//     operands one trip ahead and writing mu over the trip's grad_out;
//   * a store warp sends the tile's grad_x and grad_gate out with two TMA
//     tensor stores (rows past T and lanes past J are clipped by the tensor
//     maps) and hands the stage back once they have read it.
// The roles hand a stage on with mbarriers only.  Waits are bounded.
#include <algorithm>

#include "es_device.cuh"

namespace es {
namespace {

constexpr int kTT = 16;
constexpr int kMaxStages = 6;

template <int E>
__device__ __forceinline__ void ld_vec(float* d, const float* p) {
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
__device__ __forceinline__ void put_vec(float* p, const float* v) {
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

// shared-memory layout of one stage, in bytes
template <int W, int E, bool GW, int CW>
struct VbLayout {
    static constexpr int R = 32 * CW * E;          // values of a trip row per CTA
    static constexpr int LV = R / W;               // lanes per CTA
    static constexpr int GW_ = GW ? W : 1;         // gate width
    static constexpr uint32_t kSeq = kTT * R * 4;  // grad_out or x
    static constexpr uint32_t kH = (kTT + 1) * R * 4;
    static constexpr uint32_t kA = kTT * LV * GW_ * 4;
    static constexpr uint32_t kOffX = kSeq;
    static constexpr uint32_t kOffH = 2 * kSeq;
    static constexpr uint32_t kOffA = (kOffH + kH + 1023u) & ~1023u;
    static constexpr uint32_t kStage = (kOffA + kA + 1023u) & ~1023u;
};

template <int W, int E, bool GW, int CW>
__global__ void __launch_bounds__(32 * (2 * CW + 2))
k_vec_bwd(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_x,
          const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_h,
          const __grid_constant__ CUtensorMap map_gx, const __grid_constant__ CUtensorMap map_ga,
          const float* __restrict__ init, float* __restrict__ ginit, int T, int J, int tiles_j, int stages,
          int reverse, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    using Lay = VbLayout<W, E, GW, CW>;
    constexpr int R = Lay::R;
    constexpr int LV = Lay::LV;
    constexpr int gw = Lay::GW_;
    constexpr int G = W / E;
    constexpr int GE = GW ? E : 1;
    constexpr unsigned kMask = 0xffffffffu;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t rn_bar[kMaxStages];    // helpers: the tile's 1/|y| are in place
    __shared__ __align__(8) uint64_t mu_bar[kMaxStages];    // chain warps: the tile's mu are in place
    __shared__ __align__(8) uint64_t done_bar[kMaxStages];  // helpers: the gate gradients are in place
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages]; // storer: the stores have read the stage
    __shared__ int abort_flag;

    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    const int o = blockIdx.x / tiles_j;
    const int j0 = (blockIdx.x % tiles_j) * LV;
    const int ntiles = (T + kTT - 1) / kTT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool desc = !reverse;                      // the gradient runs the trips backwards

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&rn_bar[s], CW);
            mbar_init(&mu_bar[s], CW);
            mbar_init(&done_bar[s], CW);
            mbar_init(&empty_bar[s], 1);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    auto tile_t0 = [&](int k) { return (desc ? ntiles - 1 - k : k) * kTT; };

    if (warp == 2 * CW) {
        // producer
        if (lane == 0) {
            tma_prefetch_desc(&map_g);
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_a);
            tma_prefetch_desc(&map_h);
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
                const int t0 = tile_t0(k);
                unsigned char* st = base + static_cast<size_t>(s) * Lay::kStage;
                mbar_arrive_expect_tx(&full_bar[s], 2 * Lay::kSeq + Lay::kH + Lay::kA);
                tma_load_3d(st, &map_g, j0 * W, t0, o, &full_bar[s], pol);
                tma_load_3d(st + Lay::kOffX, &map_x, j0 * W, t0, o, &full_bar[s], pol);
                tma_load_3d(st + Lay::kOffH, &map_h, j0 * W, reverse ? t0 : t0 - 1, o, &full_bar[s], pol);
                tma_load_3d(st + Lay::kOffA, &map_a, j0 * gw, t0, o, &full_bar[s], pol);
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }
    if (warp == 2 * CW + 1) {
        // storer: grad_x from the grad_out rows, grad_gate from the gate rows
        if (lane == 0) {
            tma_prefetch_desc(&map_gx);
            tma_prefetch_desc(&map_ga);
            for (int k = 0; k < ntiles; ++k) {
                const int s = k % stages;
                if (!mbar_wait_bounded(&done_bar[s], (k / stages) & 1, wait_ns, &abort_flag)) {
                    report_timeout(status, &abort_flag);
                    break;
                }
                const int t0 = tile_t0(k);
                unsigned char* st = base + static_cast<size_t>(s) * Lay::kStage;
                tma_store_3d(&map_gx, j0 * W, t0, o, st);
                tma_store_3d(&map_ga, j0 * gw, t0, o, st + Lay::kOffA);
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(&empty_bar[s]);
            }
            bulk_wait_all();
        }
        return;
    }

    // chain warp w (< CW) and helper warp CW + w own the same lanes: thread c
    // holds values w0 .. w0+E-1 of lane j0 + v
    const bool helper = warp >= CW;
    const int c = (helper ? warp - CW : warp) * 32 + lane;
    const int v = (c * E) / W;
    const int w0 = (c * E) % W;
    const bool valid = j0 + v < J;
    const int t_first = reverse ? T - 1 : 0;
    const int gi = v * gw + (GW ? w0 : 0);
    float p0[E];
#pragma unroll
    for (int e = 0; e < E; ++e) p0[e] = valid ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] : 0.0f;

    auto lane_sum = [&](float s) {
#pragma unroll
        for (int off = G / 2; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(kMask, s, off));
        return s;
    };
    auto local_sum = [&](float* q) {
#pragma unroll
        for (int span = 1; span < E; span *= 2)
#pragma unroll
            for (int e = 0; e + span < E; e += 2 * span) q[e] = __fadd_rn(q[e], q[e + span]);
        return q[0];
    };
    struct Rows {
        float* g;          // grad_out; mu replaces it
        float* x;          // x; the signed 1/|y| replaces its first value
        const float* h;    // states
        float* a;          // gate; its gradient replaces it
    };
    auto rows = [&](int s) {
        unsigned char* st = base + static_cast<size_t>(s) * Lay::kStage;
        return Rows{reinterpret_cast<float*>(st) + c * E, reinterpret_cast<float*>(st + Lay::kOffX) + c * E,
                    reinterpret_cast<const float*>(st + Lay::kOffH) + c * E,
                    reinterpret_cast<float*>(st + Lay::kOffA) + gi};
    };
    // the state before trip tt of the tile starting at t0 (initial before the first trip)
    auto before = [&](const Rows& rw, int t0, int tt, float* p) {
        if (t0 + tt == t_first) {
#pragma unroll
            for (int e = 0; e < E; ++e) p[e] = p0[e];
        } else {
            ld_vec<E>(p, rw.h + (reverse ? tt + 1 : tt) * R);
        }
    };

    if (helper) {
        // pass 1 of tile k: 1/|y| with its cap flag for every trip, the lane
        // sums level by level over all trips so their shuffles overlap
        auto norms = [&](int k) -> bool {
            const int s = k % stages;
            const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
            if (!__all_sync(kMask, ok)) {
                if (!ok) report_timeout(status, &abort_flag);
                return false;
            }
            const int t0 = tile_t0(k);
            const Rows rw = rows(s);
            float ss[kTT];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {
                float p[E], x[E], a[GE], q[E];
                before(rw, t0, tt, p);
                ld_vec<E>(x, rw.x + tt * R);
#pragma unroll
                for (int e = 0; e < GE; ++e) a[e] = rw.a[tt * LV * gw + e];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float y = __fadd_rn(__fmul_rn(a[GW ? e : 0], p[e]), x[e]);
                    q[e] = __fmul_rn(y, y);
                }
                ss[tt] = local_sum(q);
            }
#pragma unroll
            for (int off = G / 2; off >= 1; off >>= 1)
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt) ss[tt] = __fadd_rn(ss[tt], __shfl_xor_sync(kMask, ss[tt], off));
            // a positive value is 1/|y| of a capped trip; -1 marks |y| <= 1
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) rw.x[tt * R] = ss[tt] > 1.0f ? rsqrt_approx(ss[tt]) : -1.0f;
            __syncwarp(kMask);
            if (lane == 0) mbar_arrive(&rn_bar[s]);
            return true;
        };
        // pass 3 of tile k: the gate gradients sum(mu * p), over the lane for
        // a width-one gate, written over the gate
        auto gate_grads = [&](int k) -> bool {
            const int s = k % stages;
            const bool ok = mbar_wait_bounded(&mu_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
            if (!__all_sync(kMask, ok)) {
                if (!ok) report_timeout(status, &abort_flag);
                return false;
            }
            const int t0 = tile_t0(k);
            const Rows rw = rows(s);
            float dl[kTT];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {
                float mu[E], p[E], da[E];
                ld_vec<E>(mu, rw.g + tt * R);
                before(rw, t0, tt, p);
#pragma unroll
                for (int e = 0; e < E; ++e) da[e] = __fmul_rn(mu[e], p[e]);
                if constexpr (GW) {
                    put_vec<E>(rw.a + tt * LV * gw, da);
                } else {
                    dl[tt] = local_sum(da);
                }
            }
            if constexpr (!GW) {
#pragma unroll
                for (int off = G / 2; off >= 1; off >>= 1)
#pragma unroll
                    for (int tt = 0; tt < kTT; ++tt) dl[tt] = __fadd_rn(dl[tt], __shfl_xor_sync(kMask, dl[tt], off));
                if (w0 == 0) {
#pragma unroll
                    for (int tt = 0; tt < kTT; ++tt) rw.a[tt * LV] = dl[tt];
                }
            }
            fence_proxy_async_smem();
            __syncwarp(kMask);
            if (lane == 0) mbar_arrive(&done_bar[s]);
            return true;
        };
        // the norms run one tile ahead of the chain, the gate gradients one behind
        if (!norms(0)) return;
        for (int k = 0; k < ntiles; ++k) {
            if (k + 1 < ntiles && !norms(k + 1)) return;
            if (!gate_grads(k)) return;
        }
        return;
    }

    // chain warp: lam -> (h . lam) -> mu -> a * mu, trip after trip
    float lam[E];
#pragma unroll
    for (int e = 0; e < E; ++e) lam[e] = 0.0f;
    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&rn_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(kMask, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int t0 = tile_t0(k);
        const int n = min(kTT, T - t0);
        const Rows rw = rows(s);
        // the next trip's operands are read while a trip runs
        float gn[E], hn[E], an[GE], rnn;
        auto fetch = [&](const int tt) {
            ld_vec<E>(gn, rw.g + tt * R);
            ld_vec<E>(hn, rw.h + (reverse ? tt : tt + 1) * R);
#pragma unroll
            for (int e = 0; e < GE; ++e) an[e] = rw.a[tt * LV * gw + e];
            rnn = rw.x[tt * R];
        };
        auto chain = [&](const int tt, const int next) {
            float g[E], h[E], a[GE], q[E], mu[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                g[e] = gn[e];
                h[e] = hn[e];
            }
#pragma unroll
            for (int e = 0; e < GE; ++e) a[e] = an[e];
            const float rn = rnn;
            if (next >= 0) fetch(next);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                lam[e] = __fadd_rn(lam[e], g[e]);
                q[e] = __fmul_rn(h[e], lam[e]);
            }
            const float hl = lane_sum(local_sum(q));
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float m = __fmul_rn(__fsub_rn(lam[e], __fmul_rn(h[e], hl)), rn);
                mu[e] = rn > 0.0f ? m : lam[e];
                lam[e] = __fmul_rn(a[GW ? e : 0], mu[e]);
            }
            put_vec<E>(rw.g + tt * R, mu);
        };
        if (n == kTT) {
            // full tile: one basic block, so consecutive trips overlap (with
            // the whole tile's operands staged in registers instead, the
            // burst of loads at each tile start measured slower)
            if (desc) {
                fetch(kTT - 1);
#pragma unroll
                for (int tt = kTT - 1; tt >= 0; --tt) chain(tt, tt - 1);
            } else {
                fetch(0);
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt) chain(tt, tt + 1 < kTT ? tt + 1 : -1);
            }
        } else if (desc) {
            fetch(n - 1);
            for (int tt = n - 1; tt >= 0; --tt) chain(tt, tt - 1);
        } else {
            fetch(0);
            for (int tt = 0; tt < n; ++tt) chain(tt, tt + 1 < n ? tt + 1 : -1);
        }
        fence_proxy_async_smem();
        __syncwarp(kMask);
        if (lane == 0) mbar_arrive(&mu_bar[s]);
    }
    if (valid) {
#pragma unroll
        for (int e = 0; e < E; ++e) ginit[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] = lam[e];
    }
}

// consumer warps per CTA: two where the row of lanes is wide enough
int vb_consumer_warps(int W, int64_t J) {
    const int E = W >= 4 ? 4 : W;
    return J >= 2 * (32 * E / W) ? 2 : 1;
}

template <int W, int E, bool GW, int CW>
cudaError_t launch_vb(const BackwardLaunch& B, const CUtensorMap* maps, int stages) {
    using Lay = VbLayout<W, E, GW, CW>;
    const Launch& L = B.fwd;
    const int64_t tiles_j = (L.J + Lay::LV - 1) / Lay::LV;
    const size_t smem = static_cast<size_t>(stages) * Lay::kStage + 1024;
    auto kern = k_vec_bwd<W, E, GW, CW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = L.O * tiles_j;
    kern<<<static_cast<unsigned>(grid), 32 * (2 * CW + 2), smem, L.stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], L.init, B.ginit, static_cast<int>(L.T),
        static_cast<int>(L.J), static_cast<int>(tiles_j), stages, L.reverse, L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

template <int W, int CW>
cudaError_t launch_vb_wc(const BackwardLaunch& B, const CUtensorMap* maps, int stages) {
    constexpr int E = W >= 4 ? 4 : W;
    if (B.fwd.sw[1] == 1) return launch_vb<W, E, false, CW>(B, maps, stages);
    return launch_vb<W, E, true, CW>(B, maps, stages);
}

template <int W>
cudaError_t launch_vb_w(const BackwardLaunch& B, const CUtensorMap* maps, int CW, int stages) {
    if (CW == 2) return launch_vb_wc<W, 2>(B, maps, stages);
    return launch_vb_wc<W, 1>(B, maps, stages);
}

bool encode_vb(const Launch& L, CUtensorMap* m, const float* base, int64_t row, int box_inner, int rows,
               const char** err) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row), static_cast<cuuint64_t>(L.T),
                                static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row) * 4, static_cast<cuuint64_t>(row) * L.T * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = L.encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for a vector-state backward tile map";
        return false;
    }
    return true;
}

}  // namespace

cudaError_t launch_vec_tma_bwd(const BackwardLaunch& B, const char** err) {
    const Launch& L = B.fwd;
    const int W = static_cast<int>(L.W);
    const int gw = static_cast<int>(L.sw[1]);
    const int E = W >= 4 ? 4 : W;
    const int CW = vb_consumer_warps(W, L.J);
    const int R = 32 * CW * E;
    const int LV = R / W;
    const int64_t tiles_j = (L.J + LV - 1) / LV;
    const int64_t ctas = L.O * tiles_j;
    // a stage is held from its load through the norms, the chain and the
    // gate gradients to its stores: four stages where one CTA a SM runs,
    // fewer where more CTAs share a SM
    const size_t seq = static_cast<size_t>(kTT) * R * 4;
    const size_t stage_bytes = ((2 * seq + (kTT + 1) * R * 4 + 1023) & ~size_t(1023)) +
                               ((static_cast<size_t>(kTT) * LV * gw * 4 + 1023) & ~size_t(1023));
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(8, (ctas + L.num_sms - 1) / L.num_sms));
    const int stages = static_cast<int>(std::max<int64_t>(
        3, std::min<int64_t>(std::min<int64_t>(4, kMaxStages),
                             static_cast<int64_t>(210 * 1024 / per_sm) / static_cast<int64_t>(stage_bytes))));
    CUtensorMap maps[6];
    if (!encode_vb(L, &maps[0], B.gout, L.J * W, R, kTT, err) ||
        !encode_vb(L, &maps[1], L.x, L.J * W, R, kTT, err) ||
        !encode_vb(L, &maps[2], L.a, L.J * gw, LV * gw, kTT, err) ||
        !encode_vb(L, &maps[3], B.states, L.J * W, R, kTT + 1, err) ||
        !encode_vb(L, &maps[4], B.gx, L.J * W, R, kTT, err) ||
        !encode_vb(L, &maps[5], B.ga, L.J * gw, LV * gw, kTT, err))
        return cudaErrorInvalidValue;
    switch (W) {
        case 2: return launch_vb_w<2>(B, maps, CW, stages);
        case 4: return launch_vb_w<4>(B, maps, CW, stages);
        case 8: return launch_vb_w<8>(B, maps, CW, stages);
        default: return launch_vb_w<16>(B, maps, CW, stages);
    }
}

}  // namespace es
