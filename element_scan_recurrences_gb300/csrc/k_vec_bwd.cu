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
// on the saved states and inputs alone.  1/|y| comes from the hardware
// reciprocal square root of |y|^2 (relative error below 2^-22) and is
// multiplied in, the same value as the division up to rounding; sums over a
// lane are pairwise within a thread, then xor-shuffles across the lane's W/E
// threads, as in the forward vector kernel.
//
// Layout as in the forward vector kernel (x, states, grad_out, grad_x are
// [O, T, J*W]; the gate and its gradient [O, T, J*gw]); one CTA owns
// LV = 128/W lanes of one o.  Per time tile of TT trips the producer streams
// grad_out, x, the gate and TT+1 rows of saved states (the tile's outputs and
// the state before its first trip in scan order, from a box that may start
// at row -1 or end at row T, zero-filled there; `initial` replaces it).
// Consumers prefetch each trip's operands one trip ahead from SMEM and hand
// the stage back at the end of the tile.  Waits are bounded.
#include <algorithm>

#include "es_device.cuh"

namespace es {
namespace {

constexpr int kTT = 16;
constexpr int kMaxStages = 8;
constexpr int kRow = 128;        // values per CTA per trip

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
__device__ __forceinline__ void st_vec(float* p, const float* v) {
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int i = 0; i < E; i += 4) __stcs(reinterpret_cast<float4*>(p + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
    } else if constexpr (E == 2) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
    } else {
        __stcs(p, v[0]);
    }
}

template <int W, int E, bool GW>
__global__ void __launch_bounds__(32 + kRow / E)
k_vec_bwd(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_x,
          const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_h,
          const float* __restrict__ init, float* __restrict__ ginit, float* __restrict__ gx, float* __restrict__ ga,
          int T, int J, int tiles_j, int stages, int reverse, unsigned int* status, uint64_t wait_ns,
          int64_t drop_tile) {
    constexpr int LV = kRow / W;
    constexpr int NC = kRow / E;
    constexpr int G = W / E;
    constexpr int GE = GW ? E : 1;
    constexpr int gw = GW ? W : 1;
    constexpr unsigned kMask = NC >= 32 ? 0xffffffffu : ((1u << NC) - 1u);
    constexpr uint32_t kSeqBytes = kTT * kRow * 4;                 // grad_out or x
    constexpr uint32_t kHBytes = (kTT + 1) * kRow * 4;             // states
    constexpr uint32_t kABytes = kTT * LV * gw * 4;                // gate
    constexpr uint32_t kOffX = kSeqBytes;
    constexpr uint32_t kOffH = 2 * kSeqBytes;
    constexpr uint32_t kOffA = (kOffH + kHBytes + 1023u) & ~1023u;
    constexpr uint32_t kStageBytes = (kOffA + kABytes + 1023u) & ~1023u;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int abort_flag;

    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    const int o = blockIdx.x / tiles_j;
    const int j0 = (blockIdx.x % tiles_j) * LV;
    const int ntiles = (T + kTT - 1) / kTT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool desc = !reverse;

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
                const int t0 = (desc ? ntiles - 1 - k : k) * kTT;
                unsigned char* st = base + static_cast<size_t>(s) * kStageBytes;
                mbar_arrive_expect_tx(&full_bar[s], 2 * kSeqBytes + kHBytes + kABytes);
                tma_load_3d(st, &map_g, j0 * W, t0, o, &full_bar[s], pol);
                tma_load_3d(st + kOffX, &map_x, j0 * W, t0, o, &full_bar[s], pol);
                tma_load_3d(st + kOffH, &map_h, j0 * W, reverse ? t0 : t0 - 1, o, &full_bar[s], pol);
                tma_load_3d(st + kOffA, &map_a, j0 * gw, t0, o, &full_bar[s], pol);
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
    const bool lead = (w0 == 0);                       // writes the lane's summed gate gradient
    const int64_t row = static_cast<int64_t>(J) * W;
    const int64_t grow = static_cast<int64_t>(J) * gw;
    float p0[E], lam[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        p0[e] = valid ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] : 0.0f;
        lam[e] = 0.0f;
    }
    const int t_first = reverse ? T - 1 : 0;
    const int gi = v * gw + (GW ? w0 : 0);

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

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(kMask, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int t0 = (desc ? ntiles - 1 - k : k) * kTT;
        const int n = min(kTT, T - t0);
        const unsigned char* st = base + static_cast<size_t>(s) * kStageBytes;
        const float* gs = reinterpret_cast<const float*>(st) + c * E;
        const float* xs = reinterpret_cast<const float*>(st + kOffX) + c * E;
        const float* hs = reinterpret_cast<const float*>(st + kOffH) + c * E;
        const float* as = reinterpret_cast<const float*>(st + kOffA) + gi;
        float* gxp = gx + static_cast<int64_t>(o) * T * row + static_cast<int64_t>(j0) * W + c * E;
        float* gap = ga + static_cast<int64_t>(o) * T * grow + static_cast<int64_t>(j0) * gw + gi;

        struct Ops {
            float g[E], x[E], h[E], p[E], a[GE];
        };
        // operands of trip tt: its own state row and the row of the state before it
        auto load = [&](const int tt, Ops& d) {
            ld_vec<E>(d.g, gs + tt * kRow);
            ld_vec<E>(d.x, xs + tt * kRow);
            const int hr = reverse ? tt : tt + 1;
            const int pr = reverse ? tt + 1 : tt;
            ld_vec<E>(d.h, hs + hr * kRow);
            ld_vec<E>(d.p, hs + pr * kRow);
            if (t0 + tt == t_first) {
#pragma unroll
                for (int e = 0; e < E; ++e) d.p[e] = p0[e];
            }
#pragma unroll
            for (int e = 0; e < GE; ++e) d.a[e] = as[tt * LV * gw + e];
        };
        auto trip = [&](const int tt, const Ops& d) {
            // off the chain: |y| from the saved state before the trip
            float y[E], q[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                y[e] = __fadd_rn(__fmul_rn(d.a[GW ? e : 0], d.p[e]), d.x[e]);
                q[e] = __fmul_rn(y[e], y[e]);
            }
            const float ss = lane_sum(local_sum(q));
            const bool capped = ss > 1.0f;
            const float rn = rsqrt_approx(ss);
            // the chain: lam -> (h . lam) -> mu -> a * mu
#pragma unroll
            for (int e = 0; e < E; ++e) {
                lam[e] = __fadd_rn(lam[e], d.g[e]);
                q[e] = __fmul_rn(d.h[e], lam[e]);
            }
            const float hl = lane_sum(local_sum(q));
            float mu[E], da[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float m = __fmul_rn(__fsub_rn(lam[e], __fmul_rn(d.h[e], hl)), rn);
                mu[e] = capped ? m : lam[e];
                da[e] = __fmul_rn(mu[e], d.p[e]);
                lam[e] = __fmul_rn(d.a[GW ? e : 0], mu[e]);
            }
            if (valid) {
                st_vec<E>(gxp + static_cast<int64_t>(t0 + tt) * row, mu);
                if constexpr (GW) {
                    st_vec<E>(gap + static_cast<int64_t>(t0 + tt) * grow, da);
                }
            }
            if constexpr (!GW) {
                const float dsum = lane_sum(local_sum(da));
                if (valid && lead) __stcs(gap + static_cast<int64_t>(t0 + tt) * grow, dsum);
            }
        };
        Ops A;
        if (n == kTT) {
            // Full tile in three passes so the serial chain runs alone:
            // (1) every trip's 1/|y| and cap flag (they need only saved states
            //     and inputs), (2) the cotangent chain, keeping each mu,
            // (3) the gate gradients sum(mu * p) over each lane.  The lane
            // sums of passes 1 and 3 go level by level over all trips of the
            // tile, so their shuffles overlap instead of forming 16 chains.
            float rn[kTT], ssl[kTT];
            bool capped[kTT];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {
                Ops d;
                load(tt, d);
                float q[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float y = __fadd_rn(__fmul_rn(d.a[GW ? e : 0], d.p[e]), d.x[e]);
                    q[e] = __fmul_rn(y, y);
                }
                ssl[tt] = local_sum(q);
            }
#pragma unroll
            for (int off = G / 2; off >= 1; off >>= 1)
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt) ssl[tt] = __fadd_rn(ssl[tt], __shfl_xor_sync(kMask, ssl[tt], off));
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {
                capped[tt] = ssl[tt] > 1.0f;
                rn[tt] = rsqrt_approx(ssl[tt]);
            }
            float mus[kTT][E];
            float gn[E], hn[E];            // the next trip's operands, read one trip ahead
            auto fetch = [&](const int tt) {
                ld_vec<E>(gn, gs + tt * kRow);
                ld_vec<E>(hn, hs + (reverse ? tt : tt + 1) * kRow);
            };
            auto chain = [&](const int tt, const int next) {
                float g[E], h[E], q[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    g[e] = gn[e];
                    h[e] = hn[e];
                }
                if (next >= 0) fetch(next);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    lam[e] = __fadd_rn(lam[e], g[e]);
                    q[e] = __fmul_rn(h[e], lam[e]);
                }
                const float hl = lane_sum(local_sum(q));
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float m = __fmul_rn(__fsub_rn(lam[e], __fmul_rn(h[e], hl)), rn[tt]);
                    mus[tt][e] = capped[tt] ? m : lam[e];
                    lam[e] = __fmul_rn(as[tt * LV * gw + (GW ? e : 0)], mus[tt][e]);
                }
                if (valid) st_vec<E>(gxp + static_cast<int64_t>(t0 + tt) * row, mus[tt]);
            };
            if (desc) {
                fetch(kTT - 1);
#pragma unroll
                for (int tt = kTT - 1; tt >= 0; --tt) chain(tt, tt - 1);
            } else {
                fetch(0);
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt) chain(tt, tt + 1 < kTT ? tt + 1 : -1);
            }
            float dl[kTT][GW ? E : 1];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) {
                Ops d;
                load(tt, d);
                float da[E];
#pragma unroll
                for (int e = 0; e < E; ++e) da[e] = __fmul_rn(mus[tt][e], d.p[e]);
                if constexpr (GW) {
                    if (valid) st_vec<E>(gap + static_cast<int64_t>(t0 + tt) * grow, da);
                } else {
                    dl[tt][0] = local_sum(da);
                }
            }
            if constexpr (!GW) {
#pragma unroll
                for (int off = G / 2; off >= 1; off >>= 1)
#pragma unroll
                    for (int tt = 0; tt < kTT; ++tt)
                        dl[tt][0] = __fadd_rn(dl[tt][0], __shfl_xor_sync(kMask, dl[tt][0], off));
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt)
                    if (valid && lead) __stcs(gap + static_cast<int64_t>(t0 + tt) * grow, dl[tt][0]);
            }
        } else if (desc) {
            for (int tt = n - 1; tt >= 0; --tt) {
                load(tt, A);
                trip(tt, A);
            }
        } else {
            for (int tt = 0; tt < n; ++tt) {
                load(tt, A);
                trip(tt, A);
            }
        }
        __syncwarp(kMask);
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    if (valid) {
#pragma unroll
        for (int e = 0; e < E; ++e) ginit[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] = lam[e];
    }
}

template <int W, int E, bool GW>
cudaError_t launch_vb(const BackwardLaunch& B, const CUtensorMap* maps, int tiles_j, int stages) {
    const Launch& L = B.fwd;
    constexpr int LV = kRow / W;
    constexpr uint32_t kSeqBytes = kTT * kRow * 4;
    constexpr uint32_t kHBytes = (kTT + 1) * kRow * 4;
    constexpr uint32_t kABytes = kTT * LV * (GW ? W : 1) * 4;
    constexpr uint32_t kOffA = (2 * kSeqBytes + kHBytes + 1023u) & ~1023u;
    constexpr uint32_t kStageBytes = (kOffA + kABytes + 1023u) & ~1023u;
    const size_t smem = static_cast<size_t>(stages) * kStageBytes + 1024;
    auto kern = k_vec_bwd<W, E, GW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = L.O * tiles_j;
    kern<<<static_cast<unsigned>(grid), 32 + kRow / E, smem, L.stream>>>(
        maps[0], maps[1], maps[2], maps[3], L.init, B.ginit, B.gx, B.ga, static_cast<int>(L.T), static_cast<int>(L.J),
        tiles_j, stages, L.reverse, L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

template <int W>
cudaError_t launch_vb_w(const BackwardLaunch& B, const CUtensorMap* maps, int tiles_j, int stages) {
    constexpr int E = W >= 4 ? 4 : W;
    if (B.fwd.sw[1] == 1) return launch_vb<W, E, false>(B, maps, tiles_j, stages);
    return launch_vb<W, E, true>(B, maps, tiles_j, stages);
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
    const int LV = kRow / W;
    const int64_t tiles_j = (L.J + LV - 1) / LV;
    // four stages of the four streams (about 100 KB): two CTAs per SM
    const int stages = 4;
    CUtensorMap maps[4];
    if (!encode_vb(L, &maps[0], B.gout, L.J * W, kRow, kTT, err) ||
        !encode_vb(L, &maps[1], L.x, L.J * W, kRow, kTT, err) ||
        !encode_vb(L, &maps[2], L.a, L.J * gw, LV * gw, kTT, err) ||
        !encode_vb(L, &maps[3], B.states, L.J * W, kRow, kTT + 1, err))
        return cudaErrorInvalidValue;
    const int tj = static_cast<int>(tiles_j);
    switch (W) {
        case 2: return launch_vb_w<2>(B, maps, tj, stages);
        case 4: return launch_vb_w<4>(B, maps, tj, stages);
        case 8: return launch_vb_w<8>(B, maps, tj, stages);
        default: return launch_vb_w<16>(B, maps, tj, stages);
    }
}

}  // namespace es
