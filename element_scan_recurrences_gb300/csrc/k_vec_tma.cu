// k_vec_tma.cu -- NORMCAP with a vector state (ES_PATH_VEC_TMA).
//
// "Nonlinear element scans", :state-axis example: each lane carries W values
// (W in {2, 4, 8, 16}) and every trip computes y = a*h + x with a per-trip
// gate `a` (width 1, broadcast over the state, or width W), then
// h = y / max(1, ||y||_2).
//
// Canonical view: x and out are [O, T, J*W], the gate is [O, T, J*gw].  One
// CTA owns LV = 128 / W adjacent lanes of one o (128 contiguous values per
// trip) and walks all T trips.  Warp 0's lane 0 streams time tiles of 32
// trips of x and of the gate into an S-stage SMEM ring with TMA (full/empty
// mbarrier pairs).  Each of the 128 / E consumer threads holds E consecutive
// values of one lane's state (E in {1, 2, 4, 8, 16}); a lane is G = W / E
// threads.  A trip is a serial chain, so its latency bounds the kernel when
// lanes are few; the chain is kept short:
//   * the squared norm adds each thread's E squares pairwise, then a
//     butterfly of G/2 .. 1 xor-shuffles inside the lane's group (every
//     thread of a group ends with the same bitwise sum: each level adds the
//     same two operands); E = 4 (two shuffles for W = 16) measured best;
//   * the division by max(1, ||y||) is a multiplication by
//     min(1, 1/sqrt(ss)) from the hardware reciprocal square root: the same
//     value up to rounding (exactly y inside the unit ball), one multiply on
//     the chain instead of a square root followed by a division;
//   * a tile's inputs go to registers before its chain starts and the stage
//     is handed back to the producer at once.
// Stores are one coalesced 512-byte row per trip.  Waits are bounded as in
// the other pipelines.
#include <algorithm>
#include <type_traits>

#include "es_device.cuh"

// Tuning overrides.
#ifndef ES_VEC_VALUES_PER_THREAD
#define ES_VEC_VALUES_PER_THREAD 0      // 0: min(W, 4)
#endif
#ifndef ES_VEC_STAGE_TILE
#define ES_VEC_STAGE_TILE -1            // -1: chosen from the operand count per trip
#endif

namespace es {
namespace {

constexpr int kTT = 32;       // trips per tile
constexpr int kMaxStages = 8;

template <int E>
struct Vec;
template <>
struct Vec<1> {
    static __device__ __forceinline__ void load(float* d, const float* p) { d[0] = p[0]; }
    static __device__ __forceinline__ void store(float* p, const float* v) { __stcs(p, v[0]); }
    static __device__ __forceinline__ void put(float* p, const float* v) { p[0] = v[0]; }
};
template <>
struct Vec<2> {
    static __device__ __forceinline__ void load(float* d, const float* p) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        d[0] = t.x;
        d[1] = t.y;
    }
    static __device__ __forceinline__ void store(float* p, const float* v) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
    }
    static __device__ __forceinline__ void put(float* p, const float* v) {
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    }
};
template <>
struct Vec<4> {
    static __device__ __forceinline__ void load(float* d, const float* p) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        d[0] = t.x;
        d[1] = t.y;
        d[2] = t.z;
        d[3] = t.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* v) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
    static __device__ __forceinline__ void put(float* p, const float* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <int E>
struct VecN {   // E = 8 or 16 values as 16-byte pieces
    static __device__ __forceinline__ void load(float* d, const float* p) {
#pragma unroll
        for (int i = 0; i < E; i += 4) Vec<4>::load(d + i, p + i);
    }
    static __device__ __forceinline__ void store(float* p, const float* v) {
#pragma unroll
        for (int i = 0; i < E; i += 4) Vec<4>::store(p + i, v + i);
    }
    static __device__ __forceinline__ void put(float* p, const float* v) {
#pragma unroll
        for (int i = 0; i < E; i += 4) Vec<4>::put(p + i, v + i);
    }
};
template <>
struct Vec<8> : VecN<8> {};
template <>
struct Vec<16> : VecN<16> {};

// 1 / max(1, sqrt(ss)) for ss >= 0, i.e. min(1, 1/sqrt(ss)): the hardware
// reciprocal square root (relative error below 2^-22) and an IEEE minimum
// with one.  Inside the unit ball the result is exactly one, so h = y as with
// the division.  A NaN propagates.
__device__ __forceinline__ float normcap_scale(float ss) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(ss));
    return ieee_minimum(r, 1.0f);
}

template <int W, int E, bool GW, int CW>
__global__ void __launch_bounds__(32 * (CW + 2))
k_vec_tma(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_g,
          const __grid_constant__ CUtensorMap map_o, const float* __restrict__ init, int T, int J, int gw,
          int tiles_j, int stages, int reverse, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    constexpr int NC = 32 * CW;                    // consumer threads
    constexpr int R = NC * E;                      // values of x per CTA per trip
    constexpr int LV = R / W;                      // lanes per CTA
    constexpr int G = W / E;                       // threads per lane
    constexpr int GE = GW ? E : 1;                 // staged gate values per trip
    // whole-tile staging while the tile's operands fit in about 160 registers
    constexpr bool kStageTile = ES_VEC_STAGE_TILE < 0 ? (kTT * (E + GE) <= 160) : (ES_VEC_STAGE_TILE != 0);
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t done_bar[kMaxStages];
    __shared__ int abort_flag;

    const int gl = LV * gw;                        // gate floats per trip row
    const uint32_t x_bytes = kTT * R * 4;
    const uint32_t g_bytes = static_cast<uint32_t>(kTT * gl * 4);
    const uint32_t g_pad = (g_bytes + 1023u) & ~1023u;
    const uint32_t stage_bytes = x_bytes + g_pad;
    unsigned char* base = smem_raw + smem_align_pad(smem_raw);

    const int o = blockIdx.x / tiles_j;
    const int j0 = (blockIdx.x % tiles_j) * LV;
    const int ntiles = (T + kTT - 1) / kTT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&done_bar[s], CW);
            mbar_init(&empty_bar[s], 1);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == CW) {
        // producer: time tiles of x and of the gate into the stage ring
        if (lane == 0) {
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_g);
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
                unsigned char* xs = base + static_cast<size_t>(s) * stage_bytes;
                mbar_arrive_expect_tx(&full_bar[s], x_bytes + g_bytes);
                tma_load_3d(xs, &map_x, j0 * W, j * kTT, o, &full_bar[s], pol);
                tma_load_3d(xs + x_bytes, &map_g, j0 * gw, j * kTT, o, &full_bar[s], pol);
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }
    if (warp == CW + 1) {
        // storer: the consumers leave each tile's states in place of its x
        // values; the tile leaves shared memory as one TMA tensor store (rows
        // past T and lanes past J are clipped by the tensor map), and the
        // stage goes back to the producer once the store has read it
        if (lane == 0) {
            tma_prefetch_desc(&map_o);
            for (int k = 0; k < ntiles; ++k) {
                const int s = k % stages;
                if (!mbar_wait_bounded(&done_bar[s], (k / stages) & 1, wait_ns, &abort_flag)) {
                    report_timeout(status, &abort_flag);
                    break;
                }
                const int j = reverse ? ntiles - 1 - k : k;
                tma_store_3d(&map_o, j0 * W, j * kTT, o, base + static_cast<size_t>(s) * stage_bytes);
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(&empty_bar[s]);
            }
            bulk_wait_all();
        }
        return;
    }

    // consumers: thread c holds values w0 .. w0+E-1 of lane j0 + v
    constexpr unsigned kMask = 0xffffffffu;
    const int c = threadIdx.x;
    const int v = (c * E) / W;
    const int w0 = (c * E) % W;
    const bool valid = j0 + v < J;
    float h[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        h[e] = valid ? init[(static_cast<int64_t>(o) * J + j0 + v) * W + w0 + e] : 0.0f;
    const int gi = v * gw + (GW ? w0 : 0);

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(kMask, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int j = reverse ? ntiles - 1 - k : k;
        const int t0 = j * kTT;
        const int n = min(kTT, T - t0);
        // a thread writes each state over its own x values of that trip,
        // after it has read them
        float* xs = reinterpret_cast<float*>(base + static_cast<size_t>(s) * stage_bytes) + c * E;
        const float* gs = reinterpret_cast<const float*>(base + static_cast<size_t>(s) * stage_bytes + x_bytes) + gi;
        float* op = xs;
        auto load = [&](const int tt, float* xd, float* gd) {
            Vec<E>::load(xd, xs + tt * R);
#pragma unroll
            for (int e = 0; e < GE; ++e) gd[e] = gs[tt * gl + e];
        };
        // one trip from operands already in registers
        auto trip = [&](const int tt, const float* xv, const float* gv) {
            float y[E];
#pragma unroll
            for (int e = 0; e < E; ++e) y[e] = __fadd_rn(__fmul_rn(gv[GW ? e : 0], h[e]), xv[e]);
            float sq[E];
#pragma unroll
            for (int e = 0; e < E; ++e) sq[e] = __fmul_rn(y[e], y[e]);
#pragma unroll
            for (int span = 1; span < E; span *= 2)
#pragma unroll
                for (int e = 0; e + span < E; e += 2 * span) sq[e] = __fadd_rn(sq[e], sq[e + span]);
            float ss = sq[0];
#pragma unroll
            for (int off = G / 2; off >= 1; off >>= 1)
                ss = __fadd_rn(ss, __shfl_xor_sync(kMask, ss, off));
            const float scale = normcap_scale(ss);
#pragma unroll
            for (int e = 0; e < E; ++e) h[e] = __fmul_rn(y[e], scale);
            Vec<E>::put(op + tt * R, h);
        };
        // Sum over the lane's W values of u[e]*v[e]: this thread's E products
        // pairwise, then the xor-shuffle butterfly of the lane's group.
        auto local_dot = [&](const float* u, const float* v) {
            float p[E];
#pragma unroll
            for (int e = 0; e < E; ++e) p[e] = __fmul_rn(u[e], v[e]);
#pragma unroll
            for (int span = 1; span < E; span *= 2)
#pragma unroll
                for (int e = 0; e + span < E; e += 2 * span) p[e] = __fadd_rn(p[e], p[e + span]);
            return p[0];
        };
        // the same sum with the products folded into two fused partial sums
        auto fused_dot = [&](const float* u, const float* v) {
            float p0 = __fmul_rn(u[0], v[0]);
            if constexpr (E == 1) {
                return p0;
            } else {
                float p1 = __fmul_rn(u[1], v[1]);
#pragma unroll
                for (int e = 2; e < E; e += 2) {
                    p0 = __fmaf_rn(u[e], v[e], p0);
                    p1 = __fmaf_rn(u[e + 1], v[e + 1], p1);
                }
                return __fadd_rn(p0, p1);
            }
        };
        if constexpr (kStageTile) {
            // the whole tile goes to registers before the chain starts
            float xr[kTT][E], gr[kTT][GE];
#pragma unroll
            for (int tt = 0; tt < kTT; ++tt) load(tt, xr[tt], gr[tt]);
            // A full tile with a width-one gate, trips in scan order.  With
            // h = s*y and a = g'*s, the next trip's y' = g'*h + x' has
            //     ||y'||^2 = a^2 ||y||^2 + 2a (y . x') + ||x'||^2.
            // ||y||^2 is the value this trip's scale s came from, and the two
            // dot products depend only on this trip's y and the staged x', so
            // they are reduced while s is still being formed: the next scale
            // needs a few scalar operations after s instead of a whole
            // y' -> ||y'||^2 reduction.  While the cap acts, a^2 ||y||^2 is
            // g'^2 whatever the rounding of ||y||^2, so rounding errors do not
            // build up along the tile; the sum is clamped at zero (rounding
            // could make a vanishing norm slightly negative), and each tile's
            // first trip reduces its ||y||^2 directly.  The dot products fold
            // their products into two fused partial sums.
            auto propagated_tile = [&](auto fwd_tag) {
                constexpr bool FWD = decltype(fwd_tag)::value;
                constexpr int first = FWD ? 0 : kTT - 1;
                float y[E];
#pragma unroll
                for (int e = 0; e < E; ++e) y[e] = __fadd_rn(__fmul_rn(gr[first][0], h[e]), xr[first][e]);
                float qf = local_dot(y, y);
#pragma unroll
                for (int off = G / 2; off >= 1; off >>= 1) qf = __fadd_rn(qf, __shfl_xor_sync(kMask, qf, off));
#pragma unroll
                for (int q = 0; q < kTT; ++q) {
                    const int tt = FWD ? q : kTT - 1 - q;
                    const float sc = normcap_scale(qf);
                    if (q + 1 < kTT) {
                        const int tn = FWD ? tt + 1 : tt - 1;
                        float D = fused_dot(y, xr[tn]);
                        float P = fused_dot(xr[tn], xr[tn]);
#pragma unroll
                        for (int off = G / 2; off >= 1; off >>= 1) {
                            D = __fadd_rn(D, __shfl_xor_sync(kMask, D, off));
                            P = __fadd_rn(P, __shfl_xor_sync(kMask, P, off));
                        }
#pragma unroll
                        for (int e = 0; e < E; ++e) h[e] = __fmul_rn(y[e], sc);
                        // the state replaces this trip's x, no longer read
#pragma unroll
                        for (int e = 0; e < E; ++e) xr[tt][e] = h[e];
                        const float gn = gr[tn][0];
#pragma unroll
                        for (int e = 0; e < E; ++e) y[e] = __fadd_rn(__fmul_rn(gn, h[e]), xr[tn][e]);
                        const float a = __fmul_rn(gn, sc);
                        qf = __fmaf_rn(__fmul_rn(a, a), qf, __fmaf_rn(__fadd_rn(a, a), D, P));
                        qf = ieee_maximum(qf, 0.0f);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) h[e] = __fmul_rn(y[e], sc);
#pragma unroll
                        for (int e = 0; e < E; ++e) xr[tt][e] = h[e];
                    }
                }
                // the tile's states leave the registers in one burst, off the
                // chain (shared-memory stores queue with the shuffles)
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt) Vec<E>::put(op + tt * R, xr[tt]);
            };
            // full tiles run unguarded (one basic block, so consecutive trips
            // overlap); only the ragged last tile checks every trip
            if (n == kTT) {
                if constexpr (!GW) {
                    // width-one gate: the squared norm of the next trip's y
                    // follows from this trip's (see propagated_tile)
                    if (!reverse) propagated_tile(std::true_type{});
                    else propagated_tile(std::false_type{});
                } else if (!reverse) {
#pragma unroll
                    for (int tt = 0; tt < kTT; ++tt) trip(tt, xr[tt], gr[tt]);
                } else {
#pragma unroll
                    for (int tt = kTT - 1; tt >= 0; --tt) trip(tt, xr[tt], gr[tt]);
                }
            } else if (!reverse) {
#pragma unroll
                for (int tt = 0; tt < kTT; ++tt)
                    if (tt < n) trip(tt, xr[tt], gr[tt]);
            } else {
#pragma unroll
                for (int tt = kTT - 1; tt >= 0; --tt)
                    if (tt < n) trip(tt, xr[tt], gr[tt]);
            }
        } else {
            // wide threads: the next trip's operands are read while a trip runs
            float xa[E], ga[GE], xb[E], gb[GE];
            if (!reverse) {
                load(0, xa, ga);
#pragma unroll
                for (int tt = 0; tt < kTT; tt += 2) {
                    load(tt + 1, xb, gb);
                    if (tt < n) trip(tt, xa, ga);
                    if (tt + 2 < kTT) load(tt + 2, xa, ga);
                    if (tt + 1 < n) trip(tt + 1, xb, gb);
                }
            } else {
                load(kTT - 1, xa, ga);
#pragma unroll
                for (int tt = kTT - 1; tt >= 0; tt -= 2) {
                    load(tt - 1, xb, gb);
                    if (tt < n) trip(tt, xa, ga);
                    if (tt - 2 >= 0) load(tt - 2, xa, ga);
                    if (tt - 1 < n) trip(tt - 1, xb, gb);
                }
            }
        }
        // the tile's states are in shared memory: make them visible to the
        // tensor store and hand the stage to the storer
        fence_proxy_async_smem();
        __syncwarp(kMask);
        if (lane == 0) mbar_arrive(&done_bar[s]);
    }
}

// values per consumer thread and consumer warps per CTA for a state width
struct VecShape {
    int E, CW;
};

template <int W, int E, int CW>
cudaError_t launch_wec(const Launch& L, const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mo,
                       int gw, int tiles_j, int stages, size_t smem) {
    auto kern = gw == 1 ? k_vec_tma<W, E, false, CW> : k_vec_tma<W, E, true, CW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = L.O * tiles_j;
    kern<<<static_cast<unsigned>(grid), 32 * (CW + 2), smem, L.stream>>>(
        mx, mg, mo, L.init, static_cast<int>(L.T), static_cast<int>(L.J), gw, tiles_j, stages, L.reverse, L.status,
        L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

template <int W, int E>
cudaError_t launch_we(const Launch& L, const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mo, int gw,
                      int tiles_j, int stages, size_t smem, int CW) {
    if (CW == 2) return launch_wec<W, E, 2>(L, mx, mg, mo, gw, tiles_j, stages, smem);
    return launch_wec<W, E, 1>(L, mx, mg, mo, gw, tiles_j, stages, smem);
}

// values per thread: each halving of a lane's thread group takes one shuffle
// off the serial chain and adds one add to the thread's own tree
int vec_values_per_thread(int W) {
    int E = ES_VEC_VALUES_PER_THREAD;
    if (E == 0) E = W >= 4 ? 4 : W;
    return E > W ? W : E;
}

// Consumer warps per CTA: two (on two schedulers of the SM) where the row of
// lanes is wide enough, so that one CTA a SM drives two independent chains.
int vec_consumer_warps(int W, int64_t J) {
    const int lanes_per_warp = 32 * vec_values_per_thread(W) / W;
    return J >= 2 * lanes_per_warp ? 2 : 1;
}

template <int W>
cudaError_t launch_w(const Launch& L, const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mo, int gw,
                     int tiles_j, int stages, size_t smem, int CW) {
    const int E = vec_values_per_thread(W);
    if constexpr (W >= 16) {
        if (E == 16) return launch_we<W, 16>(L, mx, mg, mo, gw, tiles_j, stages, smem, CW);
    }
    if constexpr (W >= 8) {
        if (E == 8) return launch_we<W, 8>(L, mx, mg, mo, gw, tiles_j, stages, smem, CW);
    }
    if constexpr (W >= 4) {
        if (E == 4) return launch_we<W, 4>(L, mx, mg, mo, gw, tiles_j, stages, smem, CW);
    }
    if (E == 2) return launch_we<W, 2>(L, mx, mg, mo, gw, tiles_j, stages, smem, CW);
    return launch_we<W, 1>(L, mx, mg, mo, gw, tiles_j, stages, smem, CW);
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
    const int64_t LV = 32 * vec_values_per_thread(static_cast<int>(W)) / W;     // lanes of one consumer warp
    if (J < LV) return false;                               // a tile never exceeds the row
    if ((J * W) % 4 != 0 || (J * sw[1]) % 4 != 0 || (LV * sw[1]) % 4 != 0) return false;   // 16-byte strides, boxes
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || J * W >= (int64_t(1) << 31)) return false;
    if (O * ((J + LV - 1) / LV) >= (int64_t(1) << 31)) return false;
    for (int k = 1; k < 4; ++k)
        if (reinterpret_cast<uintptr_t>(ptrs[k]) % 16 != 0) return false;
    return true;
}

cudaError_t launch_vec_tma(const Launch& L, const char** err) {
    const int W = static_cast<int>(L.W);
    const int gw = static_cast<int>(L.sw[1]);
    const int E = vec_values_per_thread(W);
    const int CW = vec_consumer_warps(W, L.J);
    const int R = 32 * CW * E;                  // values of a trip row per CTA
    const int LV = R / W;                       // lanes per CTA
    const int64_t tiles_j = (L.J + LV - 1) / LV;
    const int64_t ctas = L.O * tiles_j;
    const size_t x_bytes = static_cast<size_t>(kTT) * R * 4;
    const size_t g_bytes = static_cast<size_t>(kTT) * LV * gw * 4;
    const size_t stage_bytes = x_bytes + ((g_bytes + 1023) & ~size_t(1023));
    // a stage is held from its load through the chain to the store of its
    // states: 3 or more stages, as many as the CTAs a SM holds leave room for
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(8, (ctas + L.num_sms - 1) / L.num_sms));
    const int64_t budget = (200 * 1024) / per_sm;
    const int stages = static_cast<int>(
        std::max<int64_t>(3, std::min<int64_t>(kMaxStages, budget / static_cast<int64_t>(stage_bytes))));
    const size_t smem = static_cast<size_t>(stages) * stage_bytes + 1024;
    CUtensorMap mx, mg, mo;
    if (!encode_vec(L, &mx, L.x, L.J * W, R, err) || !encode_vec(L, &mg, L.a, L.J * gw, LV * gw, err) ||
        !encode_vec(L, &mo, L.out, L.J * W, R, err))
        return cudaErrorInvalidValue;
    const int tj = static_cast<int>(tiles_j);
    switch (W) {
        case 2: return launch_w<2>(L, mx, mg, mo, gw, tj, stages, smem, CW);
        case 4: return launch_w<4>(L, mx, mg, mo, gw, tj, stages, smem, CW);
        case 8: return launch_w<8>(L, mx, mg, mo, gw, tj, stages, smem, CW);
        default: return launch_w<16>(L, mx, mg, mo, gw, tj, stages, smem, CW);
    }
}

}  // namespace es
