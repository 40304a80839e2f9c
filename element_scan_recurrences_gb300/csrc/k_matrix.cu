// k_matrix.cu -- matrix-scan kernels ("Tensor operations": the `matrix-scan`
// row of the operations table and the section "matrix-scan").
//
//     h[t] = a[t] @ h[t-1] + b[t]      from h = 0 (h[T] = 0 in reverse)
//
// with a [.., n, n] (n <= 16) and b, h [.., n, m].  "Every column of h is its
// own recurrence on the shared a", so a lane (one leading position off the
// axis) is m independent column recurrences: each column is one thread,
// holding its n values in registers.  A product is the plain definition in
// f32: for row i the terms a[i][j] * h[j] are rounded and added in the order
// j = 0..n-1, then b[i] is added (no fused multiply-add), which is also the
// oracle's order, so the results match it bit for bit.
//
// `:projective` (same section): the running product P of a, from the
// identity, is divided by its largest magnitude after every step, and h by
// the same number.  P's n columns are n more column recurrences on the same
// a (no b), carried by n more threads of the lane's group; the largest
// magnitude is an xor-shuffle maximum over the group (IEEE maximum, so a NaN
// propagates), and every column is divided by it (IEEE division).
//
// Kernels:
//   * k_mat_generic: any broadcast of the leading dims (per-dim strides, a
//     stride of 0 repeats an operand), loads straight from global memory;
//   * k_mat_tma: dense operands; a producer thread streams {lanes x trips}
//     tiles of a and b with TMA into an mbarrier ring, the lane's column
//     threads read a's rows from shared memory (broadcast reads) and their own
//     column of b, and store their column of h.  Waits are bounded as in the
//     element-scan pipelines.  Its chunk modes are the two scan passes of the
//     chunked scan for few long lanes, linked by k_mat_chunk_link; the
//     direct-load chunk kernels (k_mat_chunk_*) serve other operands;
//   * the gradient ("its gradient is the same scan run backwards on a's
//     transposes"): the same kernels with a transposed, one-trip-shifted
//     coefficient for the cotangent, then k_mat_da / k_mat_da16 for grad_a.
#include <algorithm>

#include "es_device.cuh"
#include "es_matrix.h"

namespace es {
namespace {

// this column's update hn = a @ h, row by row: the products a[i][j] * h[j]
// rounded and added in the order j = 0..N-1.  ROW(i, r) fills r with row i.
template <int N, class Row>
__device__ __forceinline__ void column_step(float (&hn)[N], const float (&h)[N], Row row) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float r[N];
        row(i, r);
        float acc = __fmul_rn(r[0], h[0]);
#pragma unroll
        for (int j = 1; j < N; ++j) acc = __fadd_rn(acc, __fmul_rn(r[j], h[j]));
        hn[i] = acc;
    }
}

// row i of an N x N block in shared memory (16-byte aligned when N is even)
template <int N>
__device__ __forceinline__ void smem_row(const float* A, int i, float (&r)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N; q += 4) {
            const float4 v = *reinterpret_cast<const float4*>(A + i * N + q);
            r[q] = v.x;
            r[q + 1] = v.y;
            r[q + 2] = v.z;
            r[q + 3] = v.w;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int q = 0; q < N; q += 2) {
            const float2 v = *reinterpret_cast<const float2*>(A + i * N + q);
            r[q] = v.x;
            r[q + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) r[q] = A[i * N + q];
    }
}

// two IEEE products in one packed instruction (sm_100 and later):
// (p0, p1) = (a0 * b0, a1 * b1), each rounded to nearest on its own, so the
// result is that of two __fmul_rn
__device__ __forceinline__ void mul2_rn(float& p0, float& p1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(p0), "=f"(p1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// two IEEE fused multiply-adds in one packed instruction (sm_100 and
// later): (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1), each rounded once, so the
// result is that of two __fmaf_rn
__device__ __forceinline__ void fma2_rn(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                        float c1) {
    asm("{\n\t.reg .b64 x, y, z, w;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "mov.b64 z, {%6, %7};\n\tfma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// K consecutive floats of shared memory (16-byte aligned when K % 4 == 0,
// 8-byte when K % 2 == 0)
template <int K>
__device__ __forceinline__ void smem_seg(const float* p, float (&d)[K]) {
    if constexpr (K % 4 == 0) {
#pragma unroll
        for (int q = 0; q < K; q += 4) {
            const float4 v = *reinterpret_cast<const float4*>(p + q);
            d[q] = v.x;
            d[q + 1] = v.y;
            d[q + 2] = v.z;
            d[q + 3] = v.w;
        }
    } else if constexpr (K % 2 == 0) {
#pragma unroll
        for (int q = 0; q < K; q += 2) {
            const float2 v = *reinterpret_cast<const float2*>(p + q);
            d[q] = v.x;
            d[q + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int q = 0; q < K; ++q) d[q] = p[q];
    }
}

// the largest |value| over the lane group of `gp` threads (a power of two)
__device__ __forceinline__ float group_max_abs(float v, int gp, unsigned mask) {
    for (int off = gp / 2; off >= 1; off >>= 1) v = ieee_maximum(v, __shfl_xor_sync(mask, v, off));
    return v;
}

// ---------------------------------------------------------------------------
// any layout

// TRANS (the gradient's cotangent scan): the step's coefficient is
// a[t + a_shift]^T, the zero matrix where t + a_shift falls outside the axis.
template <int N, bool PROJ, bool TRANS>
__global__ void __launch_bounds__(128)
k_mat_generic(const float* __restrict__ a, const float* __restrict__ b, float* __restrict__ out, const MatGeom g,
              int m, int gp, int reverse, int a_shift) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // projective: a lane is a group of gp threads (columns of h, then of P);
    // else one thread per column of h
    const int64_t lane = PROJ ? tid / gp : tid / m;
    const int c = static_cast<int>(PROJ ? tid % gp : tid % m);
    const bool live = lane < g.lanes;
    const bool is_h = c < m;
    const bool is_p = PROJ && !is_h && c < m + N;
    // offsets of this lane (in matrices) in a, b and out
    int64_t oa = 0, ob = 0, oo = 0;
    {
        int64_t rem = live ? lane : 0;
        for (int d = g.nd - 1; d >= 0; --d) {
            const int64_t q = rem % g.dim[d];
            rem /= g.dim[d];
            oa += q * g.sa[d];
            ob += q * g.sb[d];
            oo += q * g.so[d];
        }
    }
    float h[N];
#pragma unroll
    for (int i = 0; i < N; ++i) h[i] = (is_p && i == c - m) ? 1.0f : 0.0f;
    for (int64_t s = 0; s < g.T; ++s) {
        const int64_t t = reverse ? g.T - 1 - s : s;
        float hn[N];
        if (live) {
            const int64_t tc = t + a_shift;
            const bool a_in = tc >= 0 && tc < g.T;
            const float* A = a + (oa + (a_in ? tc : 0) * g.ta) * N * N;
            column_step<N>(hn, h, [&](int i, float (&r)[N]) {
#pragma unroll
                for (int q = 0; q < N; ++q) {
                    if constexpr (TRANS)
                        r[q] = a_in ? __ldg(A + q * N + i) : 0.0f;
                    else
                        r[q] = __ldg(A + i * N + q);
                }
            });
            if (is_h) {
                const float* B = b + (ob + t * g.tb) * N * m + c;
#pragma unroll
                for (int i = 0; i < N; ++i) hn[i] = __fadd_rn(hn[i], __ldg(B + i * m));
            }
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) hn[i] = 0.0f;
        }
        if constexpr (PROJ) {
            float mx = 0.0f;
            if (is_p) {
#pragma unroll
                for (int i = 0; i < N; ++i) mx = ieee_maximum(mx, fabsf(hn[i]));
            }
            const float sc = group_max_abs(mx, gp, 0xffffffffu);
#pragma unroll
            for (int i = 0; i < N; ++i) hn[i] = __fdiv_rn(hn[i], sc);
        }
#pragma unroll
        for (int i = 0; i < N; ++i) h[i] = hn[i];
        if (live && is_h) {
            float* O = out + (oo + t * g.to) * N * m + c;
#pragma unroll
            for (int i = 0; i < N; ++i) __stcs(O + i * m, h[i]);
        }
    }
}

// ---------------------------------------------------------------------------
// dense operands, TMA pipeline
//
// A lane's C carried columns (of h, then of P) are gp threads (gp a power of
// two >= C), and each column's N rows are split over R row groups, so a lane
// is TPL = gp * R threads (R = min(32 / gp, N): one warp per lane for the
// wide columns, twice the warps of one thread per column).  Thread (g, c)
// forms rows i = r * R + g of column c (rows interleaved by group, so the
// groups' broadcast reads of a's rows fall in different banks), then N
// shuffles give every thread of the column the whole new column.  Products
// are formed two at a time with the packed f32x2 multiply (each still one
// rounded product) and summed in order.  On GB300 the delta-rule workload
// went from 0.89 ms (one thread per column) to 0.67 ms (two row groups) and
// 0.65 ms (packed products).

constexpr int kMatMaxStages = 4;
constexpr int kMatConsumers = 128;

// What a launch of the row-group kernel computes:
//   kMatFull   the whole scan of each lane, every state stored;
//   kMatLocal  the first pass of the chunked scan: each CTA lane is one
//              chunk of trips of one scan lane, scanned from zero, with its
//              transition product (the chunk's a, from the identity, no b) in
//              n more column threads; only the chunk's last state and product
//              are written, to the workspace;
//   kMatFinal  the last pass: each chunk scanned again from its carry (read
//              from the workspace), every state stored.
// In the chunk modes a CTA's LPC lanes are LPC consecutive chunks of one scan
// lane, each streamed as its own {block, 1, TT} box.  A chunk's trips that
// fall outside the axis (the short chunk) arrive zero-filled and leave the
// state as it was.
enum : int { kMatFull = 0, kMatLocal = 1, kMatFinal = 2 };

// TRANS (the gradient's cotangent scan): the step's coefficient is
// a[t + a_shift]^T; the a tile is loaded a_shift trips off the b tile, and
// TMA's zero fill past either end of the axis is the zero matrix.  The chunk
// modes run it too (a chunk's product is then the product of the transposed,
// shifted coefficients).
template <int N, int R, bool PROJ, bool TRANS, int MODE>
__global__ void __launch_bounds__(32 + kMatConsumers, 1)
k_mat_tma(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
          float* __restrict__ out, float* __restrict__ ws, int T, int J, int m, int gp, int LPC, int tiles_j, int TT,
          int stages, int reverse, int a_shift, int chunks, int chunk, int chunk_off, int win0, int win_len,
          const float* __restrict__ carry, unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    constexpr bool kChunk = MODE != kMatFull;
    constexpr bool kIdent = PROJ || MODE == kMatLocal;     // columns that carry a product from the identity
    static_assert(!(PROJ && TRANS), "a projective scan has no gradient");
    static_assert(!kChunk || !PROJ, "a projective scan is not chunked");
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMatMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMatMaxStages];
    __shared__ int abort_flag;

    const int TPL = gp * R;                                 // threads per lane
    const int consumers = LPC * TPL;                        // a multiple of 32, at most kMatConsumers
    // a stage: the a region, then the b region, each on a 128-byte boundary;
    // in the chunk modes each lane's box also starts on one
    const uint32_t la = kChunk ? (static_cast<uint32_t>(TT) * N * N + 31u) & ~31u : 0u;
    const uint32_t lb = kChunk ? (static_cast<uint32_t>(TT) * N * m + 31u) & ~31u : 0u;
    const uint32_t a_region = kChunk ? LPC * la : static_cast<uint32_t>(TT) * LPC * N * N;
    const uint32_t b_region = kChunk ? LPC * lb : static_cast<uint32_t>(TT) * LPC * N * m;
    const uint32_t a_pad = (a_region + 31u) & ~31u;
    const uint32_t stage_floats = (a_pad + b_region + 31u) & ~31u;
    const uint32_t stage_bytes = static_cast<uint32_t>(TT) * LPC * (N * N + N * m) * 4u;   // bytes the copies bring
    float* tiles = reinterpret_cast<float*>(smem_raw + smem_align_pad(smem_raw));

    // full: CTA = (o, a tile of LPC lanes along J); chunk modes: CTA = (scan
    // lane o * J + j, a group of LPC chunks)
    int o, jj, c0;
    if constexpr (kChunk) {
        const int lane_id = blockIdx.x / tiles_j;
        o = lane_id / J;
        jj = lane_id % J;
        c0 = (blockIdx.x % tiles_j) * LPC;
    } else {
        o = blockIdx.x / tiles_j;
        jj = (blockIdx.x % tiles_j) * LPC;
        c0 = 0;
    }
    // trips a CTA lane scans: a chunk, or (full scan) the window [win0,
    // win0 + win_len) of the axis, the whole axis unless the scan is cut into
    // windows
    const int span = kChunk ? chunk : win_len;
    const int ntiles = (span + TT - 1) / TT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], consumers / 32);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&map_a);
            tma_prefetch_desc(&map_b);
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
                const int jt = reverse ? ntiles - 1 - k : k;
                float* st = tiles + static_cast<size_t>(s) * stage_floats;
                mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
                if constexpr (kChunk) {
                    for (int l = 0; l < LPC; ++l) {
                        // the chunk's trips from jt * TT; past the axis (and
                        // for lanes past the last chunk) the box is zero-filled
                        const int64_t t = static_cast<int64_t>(c0 + l) * chunk - chunk_off + jt * TT;
                        const int ct = static_cast<int>(t < T ? t : T);
                        tma_load_4d(st + l * la, &map_a, 0, jj, ct + a_shift, o, &full_bar[s], pol);
                        tma_load_4d(st + a_pad + l * lb, &map_b, 0, jj, ct, o, &full_bar[s], pol);
                    }
                } else {
                    tma_load_4d(st, &map_a, 0, jj, win0 + jt * TT + a_shift, o, &full_bar[s], pol);
                    tma_load_4d(st + a_pad, &map_b, 0, jj, win0 + jt * TT, o, &full_bar[s], pol);
                }
            }
            for (int k = max(0, issued - stages); k < issued; ++k) {
                if (k == drop_tile) continue;
                if (!mbar_wait_bounded(&full_bar[k % stages], (k / stages) & 1, wait_ns, nullptr))
                    atomicOr(status, ES_DEVICE_TIMEOUT);
            }
        }
        return;
    }

    // consumers: thread (l, g, c) is row group g of column c of CTA lane l
    const int ct = threadIdx.x - 32;
    const int l = ct / TPL;
    const int w = ct % TPL;
    const int g = w / gp;
    const int c = w % gp;
    const bool valid = kChunk ? c0 + l < chunks : jj + l < J;
    const bool is_h = c < m;
    const bool is_p = kIdent && !is_h && c < m + N;
    constexpr int RPT = N / R;                              // rows per thread
    // warp lane of this column's row group 0
    const int col_base = (lane & ~(TPL - 1)) + c;
    const int64_t lane_block = static_cast<int64_t>(N) * m;          // floats of h per lane and trip
    float* obase = out + (static_cast<int64_t>(o) * T * J + (kChunk ? jj : jj + l)) * lane_block + c;
    const int64_t trip_stride = static_cast<int64_t>(J) * lane_block;
    // chunk modes: the chunk's first trip on the axis and its workspace unit
    // (units of a scan lane in scan order)
    const int64_t tbase = kChunk ? static_cast<int64_t>(c0 + l) * chunk - chunk_off : 0;
    const int64_t unit = static_cast<int64_t>(blockIdx.x / tiles_j) * chunks + (reverse ? chunks - 1 - (c0 + l) : c0 + l);
    const int64_t unit_floats = static_cast<int64_t>(N) * N + 2LL * N * m;
    // the column's whole state (every row), the same in all its row groups
    float h[N];
    if constexpr (MODE == kMatFinal) {
        const float* cin = ws + unit * unit_floats + N * N + N * m;
#pragma unroll
        for (int i = 0; i < N; ++i) h[i] = (valid && is_h) ? cin[i * m + c] : 0.0f;
    } else if constexpr (MODE == kMatFull) {
        // a window after the first starts from the state the previous window
        // left at the trip next to it (`carry` points at that trip's states)
        const float* cin = carry != nullptr ? carry + (static_cast<int64_t>(o) * T * J + jj + l) * lane_block + c
                                            : nullptr;
#pragma unroll
        for (int i = 0; i < N; ++i)
            h[i] = (cin != nullptr && valid && is_h) ? cin[i * m] : (is_p && i == c - m) ? 1.0f : 0.0f;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) h[i] = (is_p && i == c - m) ? 1.0f : 0.0f;
    }

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int jt = reverse ? ntiles - 1 - k : k;
        const int t0 = jt * TT;
        const int n = min(TT, span - t0);
        const float* sa = tiles + static_cast<size_t>(s) * stage_floats;
        const float* sb = sa + a_pad;
        // one trip: this thread's rows of a @ h + b (scaled when projective),
        // stored, then the whole new column gathered into h
        auto trip = [&](const int tt, float (&mine)[RPT]) {
            const float* A = kChunk ? sa + l * la + tt * (N * N) : sa + (static_cast<uint32_t>(tt) * LPC + l) * (N * N);
            // columns past m (a product's) read no b: their pointer stays in the block
            const float* B = (kChunk ? sb + l * lb + tt * (N * m) : sb + (static_cast<uint32_t>(tt) * LPC + l) * (N * m)) +
                             (is_h ? c : 0);
            const int64_t t = kChunk ? tbase + t0 + tt : win0 + t0 + tt;
            const bool live = !kChunk || (t >= 0 && t < T);
            if constexpr (kChunk && TRANS) {
                // the chunked passes: row i of a^T h + b as one fused sum
                // started from b (0 for a product column), j in order; two
                // rows a packed instruction
                float acc[RPT];
#pragma unroll
                for (int r = 0; r < RPT; ++r) acc[r] = is_h ? B[(g * RPT + r) * m] : 0.0f;
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    float seg[RPT];
                    smem_seg<RPT>(A + j * N + g * RPT, seg);
#pragma unroll
                    for (int r = 0; r + 1 < RPT; r += 2)
                        fma2_rn(acc[r], acc[r + 1], seg[r], seg[r + 1], h[j], h[j], acc[r], acc[r + 1]);
                    if constexpr (RPT % 2 == 1) acc[RPT - 1] = __fmaf_rn(seg[RPT - 1], h[j], acc[RPT - 1]);
                }
#pragma unroll
                for (int r = 0; r < RPT; ++r) mine[r] = acc[r];
            } else if constexpr (kChunk) {
                // the chunked passes: row i of a h + b as two fused partial
                // sums over the even and the odd j (the even one started
                // from b, 0 for a product column), j in order within each,
                // one packed instruction a pair of j, then their sum
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int i = r * R + g;
                    float row[N];
                    smem_row<N>(A, i, row);
                    float p0 = is_h ? B[i * m] : 0.0f, p1 = 0.0f;
#pragma unroll
                    for (int j = 0; j < N; j += 2) fma2_rn(p0, p1, row[j], row[j + 1], h[j], h[j + 1], p0, p1);
                    mine[r] = __fadd_rn(p0, p1);
                }
            } else if constexpr (TRANS) {
                // row i of a^T h is sum_j a[j][i] h[j]: over j in order, this
                // thread's contiguous rows i = g*RPT + r take the segment
                // a[j][g*RPT ..] of row j (vector loads) times h[j], the
                // same rounded products added in the same order as a dot
                // product of column i
                float acc[RPT];
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    float seg[RPT], prod[RPT];
                    smem_seg<RPT>(A + j * N + g * RPT, seg);
#pragma unroll
                    for (int r = 0; r + 1 < RPT; r += 2) mul2_rn(prod[r], prod[r + 1], seg[r], seg[r + 1], h[j], h[j]);
                    if constexpr (RPT % 2 == 1) prod[RPT - 1] = __fmul_rn(seg[RPT - 1], h[j]);
#pragma unroll
                    for (int r = 0; r < RPT; ++r) acc[r] = j == 0 ? prod[r] : __fadd_rn(acc[r], prod[r]);
                }
#pragma unroll
                for (int r = 0; r < RPT; ++r) mine[r] = is_h ? __fadd_rn(acc[r], B[(g * RPT + r) * m]) : acc[r];
            } else {
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int i = r * R + g;
                    float row[N];
                    smem_row<N>(A, i, row);
                    float prod[N];
#pragma unroll
                    for (int j = 0; j < N; j += 2) mul2_rn(prod[j], prod[j + 1], row[j], row[j + 1], h[j], h[j + 1]);
                    float acc = prod[0];
#pragma unroll
                    for (int j = 1; j < N; ++j) acc = __fadd_rn(acc, prod[j]);
                    mine[r] = is_h ? __fadd_rn(acc, B[i * m]) : acc;
                }
            }
            if constexpr (PROJ) {
                float mx = 0.0f;
                if (is_p) {
#pragma unroll
                    for (int r = 0; r < RPT; ++r) mx = ieee_maximum(mx, fabsf(mine[r]));
                }
                const float sc = group_max_abs(mx, TPL, 0xffffffffu);
#pragma unroll
                for (int r = 0; r < RPT; ++r) mine[r] = __fdiv_rn(mine[r], sc);
            }
            if (MODE != kMatLocal && valid && is_h && live) {
                float* op = obase + t * trip_stride;
#pragma unroll
                for (int r = 0; r < RPT; ++r) __stcs(op + (TRANS ? g * RPT + r : r * R + g) * m, mine[r]);
            }
            // row i lives in row group i % R at position i / R (TRANS: group
            // i / RPT at position i % RPT); a trip off the axis keeps the
            // state (the same for the whole lane group)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                float v;
                if constexpr (R == 1)
                    v = mine[i];    // the thread holds its whole column
                else
                    v = TRANS ? __shfl_sync(0xffffffffu, mine[i % RPT], col_base + (i / RPT) * gp)
                              : __shfl_sync(0xffffffffu, mine[i / R], col_base + (i % R) * gp);
                h[i] = live ? v : h[i];
            }
        };
        // two register sets by trip parity: a trip never overwrites the
        // registers the previous trip's stores may still be reading
        float ma[RPT], mb[RPT];
        int q = 0;
        for (; q + 1 < n; q += 2) {
            trip(reverse ? n - 1 - q : q, ma);
            trip(reverse ? n - 2 - q : q + 1, mb);
        }
        if (q < n) trip(reverse ? n - 1 - q : q, ma);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    if constexpr (MODE == kMatLocal) {
        // the chunk's last state (u) and transition product (Phi), written
        // once by row group 0
        if (valid && g == 0 && (is_h || is_p)) {
            float* wu = ws + unit * unit_floats;
#pragma unroll
            for (int i = 0; i < N; ++i) {
                if (is_h) wu[N * N + i * m + c] = h[i];
                else wu[i * N + (c - m)] = h[i];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// the gradient of a: da[t] = lam[t] @ h_prev^T
//
// One unit is one (lane, trip) of the dense view [O, T, J]; h_prev is the
// state before the trip in scan order (zero before the first).  Each thread
// forms a B x B block of da, every entry the sum over k = 0..m-1 in order of
// lam[i][k] * h_prev[j][k], each product and sum rounded (the first product
// starts the sum).  Rows come straight from global memory (16-byte loads when
// m is a multiple of 4); the rows a unit's threads share meet in L1.  MC > 0
// is m known at compile time: the loop over k unrolls and every load of the
// unit can be in flight at once.
// Unit v of a window of trips [t_lo, t_lo + t_cnt) of the dense view
// [O, T, J]: its index u in the whole view and its trip t (32-bit divisions
// while the view's units fit).
__device__ __forceinline__ void window_unit(int64_t v, int64_t T, int64_t J, int64_t t_lo, int64_t t_cnt, bool small,
                                            int64_t* u, int64_t* t) {
    const int64_t per_o = t_cnt * J;
    int64_t ob, r, tr;
    if (small) {
        ob = static_cast<uint32_t>(v) / static_cast<uint32_t>(per_o);
        r = v - ob * per_o;
        tr = static_cast<uint32_t>(r) / static_cast<uint32_t>(J);
    } else {
        ob = v / per_o;
        r = v - ob * per_o;
        tr = r / J;
    }
    *u = (ob * T + t_lo) * J + r;
    *t = t_lo + tr;
}

template <int N, int B, int KV, int MC>
__global__ void __launch_bounds__(128)
k_mat_da(const float* __restrict__ lam, const float* __restrict__ states, float* __restrict__ da, int64_t O,
         int64_t T, int64_t J, int m_rt, int reverse, int64_t t_lo, int64_t t_cnt) {
    const int m = MC > 0 ? MC : m_rt;
    constexpr int NB = N / B;
    constexpr int TPU = NB * NB;                 // threads per unit
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t v = tid / TPU;
    if (v >= O * t_cnt * J) return;
    const int w = static_cast<int>(tid % TPU);
    const int bi = w / NB, bj = w % NB;
    // the unit u of the whole view and its trip t (the state before it is
    // unit u - J, or u + J in reverse)
    int64_t u, t;
    window_unit(v, T, J, t_lo, t_cnt, O * T * J < (int64_t(1) << 31), &u, &t);
    const bool has_prev = reverse ? t + 1 < T : t > 0;
    const float* Lr = lam + (u * N + bi * B) * m;
    const float* Hr = states + ((has_prev ? (reverse ? u + J : u - J) : u) * N + bj * B) * m;
    float acc[B][B];
    auto load = [&](const float* p, int k, float (&d)[KV]) {
        if constexpr (KV == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p + k));
            d[0] = v.x;
            d[1] = v.y;
            d[2] = v.z;
            d[3] = v.w;
        } else {
            d[0] = __ldg(p + k);
        }
    };
#pragma unroll(MC > 0 ? MC / KV : 1)
    for (int k = 0; k < m; k += KV) {
        float lv[B][KV], hv[B][KV];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            load(Lr + b * m, k, lv[b]);
            if (has_prev) {
                load(Hr + b * m, k, hv[b]);
            } else {
#pragma unroll
                for (int q = 0; q < KV; ++q) hv[b][q] = 0.0f;
            }
        }
        if constexpr (KV % 2 == 0) {
            // two consecutive k of one entry per packed multiply (each still
            // one rounded product; the operands sit side by side as loaded)
#pragma unroll
            for (int q = 0; q < KV; q += 2)
#pragma unroll
                for (int x = 0; x < B; ++x)
#pragma unroll
                    for (int y = 0; y < B; ++y) {
                        float p0, p1;
                        mul2_rn(p0, p1, lv[x][q], lv[x][q + 1], hv[y][q], hv[y][q + 1]);
                        const float a = (k + q == 0) ? p0 : __fadd_rn(acc[x][y], p0);
                        acc[x][y] = __fadd_rn(a, p1);
                    }
        } else {
#pragma unroll
            for (int q = 0; q < KV; ++q) {
#pragma unroll
                for (int x = 0; x < B; ++x) {
                    float p[B];
                    if constexpr (B % 2 == 0) {
                        // two products at a time (each still one rounded product)
#pragma unroll
                        for (int y = 0; y < B; y += 2)
                            mul2_rn(p[y], p[y + 1], lv[x][q], lv[x][q], hv[y][q], hv[y + 1][q]);
                    } else {
#pragma unroll
                        for (int y = 0; y < B; ++y) p[y] = __fmul_rn(lv[x][q], hv[y][q]);
                    }
#pragma unroll
                    for (int y = 0; y < B; ++y) acc[x][y] = (k + q == 0) ? p[y] : __fadd_rn(acc[x][y], p[y]);
                }
            }
        }
    }
    float* D = da + u * N * N + (bi * B) * N + bj * B;
#pragma unroll
    for (int x = 0; x < B; ++x) {
        if constexpr (B % 4 == 0) {
#pragma unroll
            for (int y = 0; y < B; y += 4)
                __stcs(reinterpret_cast<float4*>(D + x * N + y),
                       make_float4(acc[x][y], acc[x][y + 1], acc[x][y + 2], acc[x][y + 3]));
        } else {
#pragma unroll
            for (int y = 0; y < B; ++y) __stcs(D + x * N + y, acc[x][y]);
        }
    }
}

// n = m = 16 (the delta rule's blocks): one warp per unit.  Reading rows of
// lam and of the state straight from global memory left each 16-byte load
// of a warp spread over 8 rows, one L1 wavefront per 16 bytes, and L1 bound
// the kernel (ncu: L1TEX throughput 93%).  Here the warp reads the unit's two
// 1 KB blocks with coalesced 16-byte loads into shared memory, each row's
// four 16-byte chunks XOR-swizzled (da16_off) so that the reads below are
// free of bank conflicts.  Lane (ri, cj) forms rows ri and ri + 8, columns
// 4cj .. 4cj + 3 of da, each entry the sum over k = 0..15 in order of
// lam[i][k] * h_prev[j][k] (the same rounded products and sums as k_mat_da).
// A packed multiply takes two consecutive k of one entry, whose operands sit
// side by side in the 16-byte chunks read, and each finished row of four
// entries leaves in one 16-byte store (a warp's store covers 512 contiguous
// bytes).
constexpr int kDa16Warps = 4;

// chunk slot of (row, chunk): XOR by ((row >> 1) + (row >> 3)) % 4.  Rows 0..7
// (or 8..15) read at one chunk land on eight different bank groups, and so do
// rows {y, y + 4, y + 8, y + 12} (row parity picks the half of the banks).
__device__ __forceinline__ int da16_off(int row, int chunk) {
    return row * 16 + ((chunk ^ (((row >> 1) + (row >> 3)) & 3)) << 2);
}

__global__ void __launch_bounds__(32 * kDa16Warps)
k_mat_da16(const float* __restrict__ lam, const float* __restrict__ states, float* __restrict__ da, int64_t units,
           int64_t T, int64_t J, int reverse, int64_t t_lo, int64_t t_cnt, bool small) {
    __shared__ __align__(16) float sm[kDa16Warps][2][256];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * kDa16Warps + warp;
    if (v >= units) return;   // the whole warp
    int64_t u, t;
    window_unit(v, T, J, t_lo, t_cnt, small, &u, &t);
    const bool has_prev = reverse ? t + 1 < T : t > 0;
    const float4* L4 = reinterpret_cast<const float4*>(lam + u * 256);
    const float4* H4 = reinterpret_cast<const float4*>(states + (has_prev ? (reverse ? u + J : u - J) : u) * 256);
    float* sl = sm[warp][0];
    float* sh = sm[warp][1];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int f = lane + 32 * q;             // 16-byte piece: row f / 4, chunk f % 4
        const float4 lv = __ldg(L4 + f);
        const float4 hv = has_prev ? __ldg(H4 + f) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        *reinterpret_cast<float4*>(sl + da16_off(f >> 2, f & 3)) = lv;
        *reinterpret_cast<float4*>(sh + da16_off(f >> 2, f & 3)) = hv;
    }
    __syncwarp();
    const int ri = lane & 7, cj = lane >> 3;
    float acc[2][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float4 lv[2], hv[4];
#pragma unroll
        for (int x = 0; x < 2; ++x) lv[x] = *reinterpret_cast<const float4*>(sl + da16_off(ri + 8 * x, c));
#pragma unroll
        for (int y = 0; y < 4; ++y) hv[y] = *reinterpret_cast<const float4*>(sh + da16_off(4 * cj + y, c));
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                float p0, p1, p2, p3;
                mul2_rn(p0, p1, lv[x].x, lv[x].y, hv[y].x, hv[y].y);
                mul2_rn(p2, p3, lv[x].z, lv[x].w, hv[y].z, hv[y].w);
                float a = c == 0 ? p0 : __fadd_rn(acc[x][y], p0);
                a = __fadd_rn(a, p1);
                a = __fadd_rn(a, p2);
                acc[x][y] = __fadd_rn(a, p3);
            }
    }
    float* D = da + u * 256;
#pragma unroll
    for (int x = 0; x < 2; ++x)
        __stcs(reinterpret_cast<float4*>(D + (ri + 8 * x) * 16 + 4 * cj),
               make_float4(acc[x][0], acc[x][1], acc[x][2], acc[x][3]));
}

template <int N>
cudaError_t launch_da_n(const float* lam, const float* states, float* da, int64_t O, int64_t T, int64_t J, int m,
                        int reverse, int64_t t_lo, int64_t t_cnt, cudaStream_t stream) {
    const int64_t units = O * t_cnt * J;
    if (units == 0) return cudaSuccess;
    auto go = [&](auto kern, int tpu) {
        const int64_t blocks = (units * tpu + 127) / 128;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        kern<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(lam, states, da, O, T, J, m, reverse, t_lo, t_cnt);
        return cudaGetLastError();
    };
    const bool vec = m % 4 == 0 && reinterpret_cast<uintptr_t>(lam) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(states) % 16 == 0;
    if constexpr (N == 16) {
        if (m == 16 && vec && reinterpret_cast<uintptr_t>(da) % 16 == 0) {
            const int64_t blocks = (units + kDa16Warps - 1) / kDa16Warps;
            if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
            k_mat_da16<<<static_cast<unsigned>(blocks), 32 * kDa16Warps, 0, stream>>>(
                lam, states, da, units, T, J, reverse, t_lo, t_cnt, O * T * J < (int64_t(1) << 31));
            return cudaGetLastError();
        }
    }
    if constexpr (N % 4 == 0) {
        if (vec && reinterpret_cast<uintptr_t>(da) % 16 == 0) {
            if (m == 16) return go(k_mat_da<N, 4, 4, 16>, (N / 4) * (N / 4));
            return go(k_mat_da<N, 4, 4, 0>, (N / 4) * (N / 4));
        }
        return go(k_mat_da<N, 4, 1, 0>, (N / 4) * (N / 4));
    } else if constexpr (N % 2 == 0) {
        if (vec) return go(k_mat_da<N, 2, 4, 0>, (N / 2) * (N / 2));
        return go(k_mat_da<N, 2, 1, 0>, (N / 2) * (N / 2));
    } else {
        if (vec) return go(k_mat_da<N, 1, 4, 0>, N * N);
        return go(k_mat_da<N, 1, 1, 0>, N * N);
    }
}

template <int N>
cudaError_t launch_generic_n(const MatLaunch& L) {
    const int gp = L.gp;
    const int64_t threads_total = L.projective ? L.g.lanes * gp : L.g.lanes * L.m;
    const int64_t blocks = (threads_total + 127) / 128;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const unsigned grid = static_cast<unsigned>(blocks);
    if (L.projective)
        k_mat_generic<N, true, false><<<grid, 128, 0, L.stream>>>(L.a, L.b, L.out, L.g, L.m, gp, L.reverse, 0);
    else if (L.trans)
        k_mat_generic<N, false, true><<<grid, 128, 0, L.stream>>>(L.a, L.b, L.out, L.g, L.m, gp, L.reverse,
                                                                   L.a_shift);
    else
        k_mat_generic<N, false, false><<<grid, 128, 0, L.stream>>>(L.a, L.b, L.out, L.g, L.m, gp, L.reverse, 0);
    return cudaGetLastError();
}

// the chunk modes' extra arguments (unused by a full scan), and the full
// scan's window of the axis with the state it starts from (unused by the
// chunk modes)
struct MatChunkArgs {
    float* ws;
    int chunks, chunk, chunk_off;
    int win0, win_len;
    const float* carry;
};

template <int N, int R, int MODE>
cudaError_t launch_tma_nr(const MatLaunch& L, const CUtensorMap& ma, const CUtensorMap& mb, int gp, int lpc,
                          int tiles_j, int TT, int stages, size_t smem, const MatChunkArgs& C) {
    auto kern = MODE != kMatFull ? (L.trans ? k_mat_tma<N, R, false, true, MODE> : k_mat_tma<N, R, false, false, MODE>)
                : L.projective   ? k_mat_tma<N, R, true, false, kMatFull>
                : L.trans        ? k_mat_tma<N, R, false, true, kMatFull>
                                 : k_mat_tma<N, R, false, false, kMatFull>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = (MODE != kMatFull ? L.g.lanes : L.O) * tiles_j;
    kern<<<static_cast<unsigned>(grid), 32 + lpc * gp * R, smem, L.stream>>>(
        ma, mb, L.out, C.ws, static_cast<int>(L.T), static_cast<int>(L.J), L.m, gp, lpc, tiles_j, TT, stages,
        L.reverse, L.trans ? L.a_shift : 0, C.chunks, C.chunk, C.chunk_off, C.win0, C.win_len, C.carry, L.status,
        L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

template <int N, int MODE>
cudaError_t launch_tma_n(const MatLaunch& L, const CUtensorMap& ma, const CUtensorMap& mb, int gp, int R, int lpc,
                         int tiles_j, int TT, int stages, size_t smem, const MatChunkArgs& C) {
    if constexpr (N >= 16) {
        if (R == 16) return launch_tma_nr<N, 16, MODE>(L, ma, mb, gp, lpc, tiles_j, TT, stages, smem, C);
    }
    if constexpr (N >= 8) {
        if (R == 8) return launch_tma_nr<N, 8, MODE>(L, ma, mb, gp, lpc, tiles_j, TT, stages, smem, C);
    }
    if constexpr (N >= 4) {
        if (R == 4) return launch_tma_nr<N, 4, MODE>(L, ma, mb, gp, lpc, tiles_j, TT, stages, smem, C);
    }
    if (R == 2) return launch_tma_nr<N, 2, MODE>(L, ma, mb, gp, lpc, tiles_j, TT, stages, smem, C);
    return launch_tma_nr<N, 1, MODE>(L, ma, mb, gp, lpc, tiles_j, TT, stages, smem, C);
}

template <int MODE>
cudaError_t launch_tma_mode(const MatLaunch& L, const CUtensorMap& ma, const CUtensorMap& mb, int gp, int R, int lpc,
                            int tiles_j, int TT, int stages, size_t smem, const MatChunkArgs& C) {
    switch (L.n) {
        case 2: return launch_tma_n<2, MODE>(L, ma, mb, gp, R, lpc, tiles_j, TT, stages, smem, C);
        case 4: return launch_tma_n<4, MODE>(L, ma, mb, gp, R, lpc, tiles_j, TT, stages, smem, C);
        case 8: return launch_tma_n<8, MODE>(L, ma, mb, gp, R, lpc, tiles_j, TT, stages, smem, C);
        default: return launch_tma_n<16, MODE>(L, ma, mb, gp, R, lpc, tiles_j, TT, stages, smem, C);
    }
}

// Row groups per column: enough to fill a warp with one lane's threads (at
// most one row per thread).  Lanes per CTA: 128 consumer threads, fewer (down
// to one warp) while one trip of the tile would pass 32 KB; trips per stage:
// about 32 KB of operands.
void mat_tile_shape(int n, int m, int gp, int* R, int* lpc, int* TT) {
    *R = std::min(32 / gp, n);
    const int tpl = gp * *R;
    auto per_trip = [&](int l) { return static_cast<int64_t>(l) * (n * n + n * m) * 4; };
    int l = std::max(1, kMatConsumers / tpl);
    while (l * tpl > 32 && per_trip(l) > 32 * 1024) l /= 2;
    *lpc = l;
    *TT = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(64, (32 * 1024) / per_trip(l))));
}

// floats of one pipeline stage as the kernel lays it out (the a region, then
// the b region, each on a 128-byte boundary; per lane in the chunk modes)
int64_t mat_stage_floats(int n, int m, int lpc, int TT, bool chunked) {
    auto up = [](int64_t v) { return (v + 31) & ~int64_t(31); };
    const int64_t na = static_cast<int64_t>(TT) * n * n, nb = static_cast<int64_t>(TT) * n * m;
    const int64_t a_region = chunked ? lpc * up(na) : lpc * na;
    const int64_t b_region = chunked ? lpc * up(nb) : lpc * nb;
    return up(up(a_region) + b_region);
}

bool encode_blocks(EncodeTiledFn encode, CUtensorMap* map, const float* base, int64_t block, int64_t J, int64_t T,
                   int64_t O, int LPC, int TT) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(block), static_cast<cuuint64_t>(J),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(O)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(block) * 4, static_cast<cuuint64_t>(block * J) * 4,
                                   static_cast<cuuint64_t>(block * J * T) * 4};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(block), static_cast<cuuint32_t>(LPC),
                               static_cast<cuuint32_t>(TT), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_mat_da(const float* lam, const float* states, float* da, int n, int64_t O, int64_t T,
                          int64_t J, int m, int reverse, cudaStream_t stream, int64_t t_lo, int64_t t_cnt) {
    if (t_cnt < 0) t_cnt = T;
    switch (n) {
#define ES_DA_CASE(K) \
    case K: return launch_da_n<K>(lam, states, da, O, T, J, m, reverse, t_lo, t_cnt, stream);
        ES_DA_CASE(1) ES_DA_CASE(2) ES_DA_CASE(3) ES_DA_CASE(4) ES_DA_CASE(5) ES_DA_CASE(6) ES_DA_CASE(7)
        ES_DA_CASE(8) ES_DA_CASE(9) ES_DA_CASE(10) ES_DA_CASE(11) ES_DA_CASE(12) ES_DA_CASE(13)
        ES_DA_CASE(14) ES_DA_CASE(15) ES_DA_CASE(16)
#undef ES_DA_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_mat_generic(const MatLaunch& L) {
    switch (L.n) {
#define ES_MAT_CASE(K) \
    case K: return launch_generic_n<K>(L);
        ES_MAT_CASE(1) ES_MAT_CASE(2) ES_MAT_CASE(3) ES_MAT_CASE(4) ES_MAT_CASE(5) ES_MAT_CASE(6) ES_MAT_CASE(7)
        ES_MAT_CASE(8) ES_MAT_CASE(9) ES_MAT_CASE(10) ES_MAT_CASE(11) ES_MAT_CASE(12) ES_MAT_CASE(13)
        ES_MAT_CASE(14) ES_MAT_CASE(15) ES_MAT_CASE(16)
#undef ES_MAT_CASE
    }
    return cudaErrorInvalidValue;
}

bool mat_tma_ok(int n, int m, int gp, bool projective, int64_t O, int64_t T, int64_t J, bool dense,
                const void* a, const void* b) {
    if (!dense) return false;
    if (n != 2 && n != 4 && n != 8 && n != 16) return false;
    if ((static_cast<int64_t>(n) * m) % 4 != 0 || static_cast<int64_t>(n) * m > 256) return false;   // boxes, strides
    if (gp > 32 || (!projective && m > 32)) return false;
    (void)projective;
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || J >= (int64_t(1) << 31)) return false;
    int R = 0, LPC = 0, TT = 0;
    mat_tile_shape(n, m, gp, &R, &LPC, &TT);
    if (O * ((J + LPC - 1) / LPC) >= (int64_t(1) << 31)) return false;
    return reinterpret_cast<uintptr_t>(a) % 16 == 0 && reinterpret_cast<uintptr_t>(b) % 16 == 0;
}

cudaError_t launch_mat_tma(const MatLaunch& L, const char** err) {
    const int n = L.n, m = L.m;
    int R = 0, LPC = 0, TT = 0;
    mat_tile_shape(n, m, L.gp, &R, &LPC, &TT);
    // a scan cut into windows shares the SMs with the grad_a windows: two
    // stages leave them room (delta-rule gradient 1.082 -> 1.062 ms on GB300)
    const int stages = L.win_len > 0 ? 2 : 3;
    const int64_t tiles_j = (L.J + LPC - 1) / LPC;
    CUtensorMap ma, mb;
    if (!encode_blocks(L.encode, &ma, L.a, static_cast<int64_t>(n) * n, L.J, L.T, L.O, LPC, TT) ||
        !encode_blocks(L.encode, &mb, L.b, static_cast<int64_t>(n) * m, L.J, L.T, L.O, LPC, TT)) {
        *err = "cuTensorMapEncodeTiled failed for a matrix-scan tile map";
        return cudaErrorInvalidValue;
    }
    const size_t smem = static_cast<size_t>(stages) * mat_stage_floats(n, m, LPC, TT, false) * 4 + 1024;
    return launch_tma_mode<kMatFull>(L, ma, mb, L.gp, R, LPC, static_cast<int>(tiles_j), TT, stages, smem,
                                     MatChunkArgs{nullptr, 0, 0, 0, static_cast<int>(L.win0),
                                                  static_cast<int>(L.win_len > 0 ? L.win_len : L.T), L.carry});
}


// ---------------------------------------------------------------------------
// few long lanes: a chunked scan in three launches
//
// The recurrence composes: over a chunk of trips s..e, h[e] = Phi h[s-1] + u[e]
// with Phi = a[e] ... a[s] and u the chunk's scan from zero.  With few lanes
// the sequential kernels leave most of the GPU idle, so the trips are cut
// into chunks:
//   1. k_mat_chunk_local, one thread per column of every (lane, chunk): the
//      chunk's scan from zero (its last state u[e]) and, in n more column
//      threads, its transition product Phi (the scan of the identity with no
//      b); both go to the workspace;
//   2. k_mat_chunk_carry, one thread per (lane, column): the chunks in scan
//      order, carry = Phi_k carry + u_k, recording the carry into each chunk;
//   3. k_mat_chunk_final, one thread per column of every (lane, chunk): the
//      chunk scanned again from its carry, writing the states.
// Every step keeps the definition's order inside a product, but the carries
// reassociate the chain (Phi_k applied to a carry rather than step by step),
// so results agree with the sequential scan to rounding, not bit for bit.
// Workspace per (lane, chunk): Phi (n x n), u[e] and the carry (n x m each).

namespace {

// the trips of chunk k in scan order: first trip, step
struct ChunkTrips {
    int64_t first;
    int64_t count;
    int64_t step;
};

__device__ __forceinline__ ChunkTrips chunk_trips(int64_t k, int64_t chunk, int64_t T, int reverse) {
    // chunks count in scan order: chunk 0 holds the first trips scanned
    const int64_t lo = k * chunk;
    const int64_t cnt = min(chunk, T - lo);
    return reverse ? ChunkTrips{T - 1 - lo, cnt, -1} : ChunkTrips{lo, cnt, 1};
}

__device__ __forceinline__ void lane_offsets(const MatGeom& g, int64_t lane, int64_t* oa, int64_t* ob, int64_t* oo) {
    int64_t rem = lane;
    *oa = *ob = *oo = 0;
    for (int d = g.nd - 1; d >= 0; --d) {
        const int64_t q = rem % g.dim[d];
        rem /= g.dim[d];
        *oa += q * g.sa[d];
        *ob += q * g.sb[d];
        *oo += q * g.so[d];
    }
}

// one step of a chunked pass for one column: hn[i] = sum_j a[i][j] h[j]
// + b[i] as two fused partial sums over the even and the odd j (the even
// one started from b[i], 0 without b), j in order within each, then their
// sum; an odd N's last term joins the even sum.  The arithmetic of the TMA
// kernel's chunk modes.  hn may alias h.
template <int N>
__device__ __forceinline__ void chunk_step(float (&hn)[N], const float (&h)[N], const float* A, const float* B,
                                           int m) {
    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float p0 = B != nullptr ? __ldg(B + i * m) : 0.0f, p1 = 0.0f;
#pragma unroll
        for (int j = 0; j + 1 < N; j += 2) {
            p0 = __fmaf_rn(__ldg(A + i * N + j), h[j], p0);
            p1 = __fmaf_rn(__ldg(A + i * N + j + 1), h[j + 1], p1);
        }
        if constexpr (N % 2 == 1) p0 = __fmaf_rn(__ldg(A + i * N + N - 1), h[N - 1], p0);
        acc[i] = N == 1 ? p0 : __fadd_rn(p0, p1);
    }
#pragma unroll
    for (int i = 0; i < N; ++i) hn[i] = acc[i];
}

template <int N>
__global__ void __launch_bounds__(128)
k_mat_chunk_local(const float* __restrict__ a, const float* __restrict__ b, float* __restrict__ ws, const MatGeom g,
                  int m, int64_t chunks, int64_t chunk, int reverse) {
    const int cols = m + N;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t unit = tid / cols;                      // (lane, chunk)
    const int c = static_cast<int>(tid % cols);
    if (unit >= g.lanes * chunks) return;
    const int64_t lane = unit / chunks, k = unit % chunks;
    int64_t oa, ob, oo;
    lane_offsets(g, lane, &oa, &ob, &oo);
    const bool is_h = c < m;
    float h[N];
#pragma unroll
    for (int i = 0; i < N; ++i) h[i] = (!is_h && i == c - m) ? 1.0f : 0.0f;
    const ChunkTrips ct = chunk_trips(k, chunk, g.T, reverse);
    for (int64_t q = 0; q < ct.count; ++q) {
        const int64_t t = ct.first + q * ct.step;
        const float* A = a + (oa + t * g.ta) * N * N;
        const float* B = b + (ob + t * g.tb) * N * m + c;
        float hn[N];
        chunk_step<N>(hn, h, A, is_h ? B : nullptr, m);
#pragma unroll
        for (int i = 0; i < N; ++i) h[i] = hn[i];
    }
    // workspace unit: Phi [N][N] (column c - m), then u [N][m] (column c)
    float* wu = ws + unit * (static_cast<int64_t>(N) * N + 2LL * N * m);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (is_h) wu[N * N + i * m + c] = h[i];
        else wu[i * N + (c - m)] = h[i];
    }
}

template <int N>
__global__ void __launch_bounds__(128)
k_mat_chunk_carry(float* __restrict__ ws, int64_t lanes, int m, int64_t chunks) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid >= lanes * m) return;
    const int64_t lane = tid / m;
    const int c = static_cast<int>(tid % m);
    const int64_t unit_floats = static_cast<int64_t>(N) * N + 2LL * N * m;
    float carry[N];
#pragma unroll
    for (int i = 0; i < N; ++i) carry[i] = 0.0f;
    for (int64_t k = 0; k < chunks; ++k) {
        float* wu = ws + (lane * chunks + k) * unit_floats;
        float* carry_in = wu + N * N + N * m;
#pragma unroll
        for (int i = 0; i < N; ++i) carry_in[i * m + c] = carry[i];
        const float* Phi = wu;
        float hn[N];
        column_step<N>(hn, carry, [&](int i, float (&r)[N]) {
#pragma unroll
            for (int j = 0; j < N; ++j) r[j] = Phi[i * N + j];
        });
#pragma unroll
        for (int i = 0; i < N; ++i) carry[i] = __fadd_rn(hn[i], wu[N * N + i * m + c]);
    }
}

template <int N>
__global__ void __launch_bounds__(128)
k_mat_chunk_final(const float* __restrict__ a, const float* __restrict__ b, const float* __restrict__ ws,
                  float* __restrict__ out, const MatGeom g, int m, int64_t chunks, int64_t chunk, int reverse) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t unit = tid / m;
    const int c = static_cast<int>(tid % m);
    if (unit >= g.lanes * chunks) return;
    const int64_t lane = unit / chunks, k = unit % chunks;
    int64_t oa, ob, oo;
    lane_offsets(g, lane, &oa, &ob, &oo);
    const float* carry_in = ws + unit * (static_cast<int64_t>(N) * N + 2LL * N * m) + N * N + N * m;
    float h[N];
#pragma unroll
    for (int i = 0; i < N; ++i) h[i] = carry_in[i * m + c];
    const ChunkTrips ct = chunk_trips(k, chunk, g.T, reverse);
    for (int64_t q = 0; q < ct.count; ++q) {
        const int64_t t = ct.first + q * ct.step;
        const float* A = a + (oa + t * g.ta) * N * N;
        const float* B = b + (ob + t * g.tb) * N * m + c;
        float* O = out + (oo + t * g.to) * N * m + c;
        chunk_step<N>(h, h, A, B, m);
#pragma unroll
        for (int i = 0; i < N; ++i) __stcs(O + i * m, h[i]);
    }
}

template <int N>
cudaError_t launch_chunked_n(const MatLaunch& L, float* ws, int64_t chunks, int64_t chunk) {
    const int64_t units = L.g.lanes * chunks;
    const int64_t t1 = units * (L.m + N), t2 = L.g.lanes * L.m, t3 = units * L.m;
    for (int64_t t : {t1, t2, t3})
        if ((t + 127) / 128 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    k_mat_chunk_local<N><<<static_cast<unsigned>((t1 + 127) / 128), 128, 0, L.stream>>>(L.a, L.b, ws, L.g, L.m,
                                                                                       chunks, chunk, L.reverse);
    k_mat_chunk_carry<N><<<static_cast<unsigned>((t2 + 127) / 128), 128, 0, L.stream>>>(ws, L.g.lanes, L.m, chunks);
    k_mat_chunk_final<N><<<static_cast<unsigned>((t3 + 127) / 128), 128, 0, L.stream>>>(L.a, L.b, ws, L.out, L.g,
                                                                                       L.m, chunks, chunk, L.reverse);
    return cudaGetLastError();
}

// The link pass of the chunked scan on the TMA kernels: one CTA per scan
// lane, thread (i, c) holding row i of column c of the carry.  The chunks'
// Phi and u (contiguous at the head of each workspace unit) stream into a
// ring of kLinkDepth shared-memory slots with 16-byte cp.async copies issued
// kLinkDepth - 1 chunks ahead; the carry's columns are exchanged through
// shared memory (two buffers alternate), one CTA barrier per chunk.  The
// arithmetic is k_mat_chunk_carry's: row i of Phi times the column, products
// rounded and added in order, then u.
constexpr int kLinkDepth = 16;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int K>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}

template <int N>
__global__ void __launch_bounds__(256)
k_mat_chunk_link(float* __restrict__ ws, int m, int chunks) {
    extern __shared__ float4 link_smem[];
    const int head = N * N + N * m;                        // Phi and u: the part read (a multiple of 4)
    const int64_t unit_floats = head + static_cast<int64_t>(N) * m;
    float* wl = ws + static_cast<int64_t>(blockIdx.x) * chunks * unit_floats;
    float* ring = reinterpret_cast<float*>(link_smem);     // [kLinkDepth][head]
    float* cb = ring + kLinkDepth * head;                  // [2][N][m]
    const int tid = threadIdx.x, nt = blockDim.x;          // N * m threads
    const int i = tid / m, c = tid % m;
    auto issue = [&](int k) {
        if (k < chunks) {
            const float* src = wl + k * unit_floats;
            float* dst = ring + (k % kLinkDepth) * head;
            for (int q = tid; q < head / 4; q += nt) cp_async16(dst + 4 * q, src + 4 * q);
        }
        cp_async_commit();   // an empty group past the end keeps the count uniform
    };
    for (int k = 0; k < kLinkDepth - 1; ++k) issue(k);
    float cv = 0.0f;
    cb[tid] = 0.0f;          // the carry into the first chunk
    for (int k = 0; k < chunks; ++k) {
        cp_async_wait<kLinkDepth - 2>();   // this thread's copies of chunk k
        __syncthreads();                   // everyone's, and the carry of chunk k - 1
        issue(k + kLinkDepth - 1);         // into the slot chunk k - 1 used
        const float* Phi = ring + (k % kLinkDepth) * head;
        const float* cur = cb + (k & 1) * (N * m);
        wl[k * unit_floats + head + tid] = cv;   // the carry into chunk k
        float acc = __fmul_rn(Phi[i * N], cur[c]);
#pragma unroll
        for (int j = 1; j < N; ++j) acc = __fadd_rn(acc, __fmul_rn(Phi[i * N + j], cur[j * m + c]));
        cv = __fadd_rn(acc, Phi[N * N + tid]);
        cb[((k + 1) & 1) * (N * m) + tid] = cv;
    }
    cp_async_wait<0>();
}

template <int N>
cudaError_t launch_chunked_tma_n(const MatLaunch& L, float* ws, int64_t chunks, int64_t chunk, const char** err) {
    const int m = L.m;
    const int stages = 3;
    MatChunkArgs C{ws, static_cast<int>(chunks), static_cast<int>(chunk),
                   static_cast<int>(L.reverse ? chunks * chunk - L.T : 0), 0, static_cast<int>(L.T), nullptr};
    // pass 1 carries the m state columns and the product's N; pass 3 the m
    int gp1 = 1;
    while (gp1 < m + N) gp1 <<= 1;
    const int gp3 = L.gp;
    int R1 = 0, lpc1 = 0, TT1 = 0, R3 = 0, lpc3 = 0, TT3 = 0;
    mat_tile_shape(N, m, gp1, &R1, &lpc1, &TT1);
    mat_tile_shape(N, m, gp3, &R3, &lpc3, &TT3);
    CUtensorMap ma1, mb1, ma3, mb3;
    if (!encode_blocks(L.encode, &ma1, L.a, N * N, L.J, L.T, L.O, 1, TT1) ||
        !encode_blocks(L.encode, &mb1, L.b, static_cast<int64_t>(N) * m, L.J, L.T, L.O, 1, TT1) ||
        !encode_blocks(L.encode, &ma3, L.a, N * N, L.J, L.T, L.O, 1, TT3) ||
        !encode_blocks(L.encode, &mb3, L.b, static_cast<int64_t>(N) * m, L.J, L.T, L.O, 1, TT3)) {
        *err = "cuTensorMapEncodeTiled failed for a matrix-scan chunk map";
        return cudaErrorInvalidValue;
    }
    const size_t smem1 = static_cast<size_t>(stages) * mat_stage_floats(N, m, lpc1, TT1, true) * 4 + 1024;
    const size_t smem3 = static_cast<size_t>(stages) * mat_stage_floats(N, m, lpc3, TT3, true) * 4 + 1024;
    const int groups1 = static_cast<int>((chunks + lpc1 - 1) / lpc1);
    const int groups3 = static_cast<int>((chunks + lpc3 - 1) / lpc3);
    cudaError_t e = launch_tma_n<N, kMatLocal>(L, ma1, mb1, gp1, R1, lpc1, groups1, TT1, stages, smem1, C);
    if (e != cudaSuccess) return e;
    const size_t smem_link = (static_cast<size_t>(kLinkDepth) * (N * N + N * m) + 2 * N * m) * 4;
    e = cudaFuncSetAttribute(k_mat_chunk_link<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_link));
    if (e != cudaSuccess) return e;
    k_mat_chunk_link<N><<<static_cast<unsigned>(L.g.lanes), N * m, smem_link, L.stream>>>(ws, m,
                                                                                     static_cast<int>(chunks));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_tma_n<N, kMatFinal>(L, ma3, mb3, gp3, R3, lpc3, groups3, TT3, stages, smem3, C);
}

}  // namespace

namespace {

// The TMA passes take the chunked scan's operands by shape: n in
// {2, 4, 8, 16}, n*m a multiple of 4 and at most 256, n + m <= 32 (pass 1
// carries m state columns and n product columns), dense leading dims.
bool chunked_tma_shape(int n, int m, bool dense) {
    return dense && (n == 2 || n == 4 || n == 8 || n == 16) && (n * m) % 4 == 0 && n * m <= 256 && n + m <= 32;
}

// GB300: 152 SMs of 228 KB shared memory.  Plan-time constants, so that the
// chunk shape (and with it the workspace size) needs no GPU to compute.
constexpr int64_t kPlanSMs = 152;
constexpr int64_t kPlanSmemPerSM = 228 * 1024;

// CTAs of one chunk pass resident per SM: shared memory (with the 1 KB the
// runtime reserves per CTA), and registers at up to 128 per thread
int64_t chunk_pass_ctas_per_sm(int n, int m, int gp) {
    int R = 0, lpc = 0, TT = 0;
    mat_tile_shape(n, m, gp, &R, &lpc, &TT);
    const int64_t smem = 3 * mat_stage_floats(n, m, lpc, TT, true) * 4 + 1024 + 1024;
    const int64_t threads = 32 + static_cast<int64_t>(lpc) * gp * R;
    return std::max<int64_t>(1, std::min(kPlanSmemPerSM / smem, 65536 / (threads * 128)));
}

}  // namespace

void mat_chunk_shape(int n, int m, bool dense, int64_t lanes, int64_t T, int64_t* chunks, int64_t* chunk) {
    const int64_t max_chunks = T / 64 > 1 ? T / 64 : 1;      // chunks of at least 64 trips
    int64_t c;
    if (chunked_tma_shape(n, m, dense)) {
        // the TMA passes: one CTA scans LPC chunks of one lane, so
        // lanes * ceil(chunks / LPC) CTAs; as many chunks as fill one wave of
        // resident CTAs, which leaves no ragged last wave and keeps the link
        // pass (one step per chunk) short
        int gp1 = 1, gp3 = 1;
        while (gp1 < m + n) gp1 <<= 1;
        while (gp3 < m) gp3 <<= 1;
        int R = 0, lpc1 = 0, lpc3 = 0, TT = 0;
        mat_tile_shape(n, m, gp1, &R, &lpc1, &TT);
        mat_tile_shape(n, m, gp3, &R, &lpc3, &TT);
        const int64_t lpc = std::min(lpc1, lpc3);
        const int64_t slots = kPlanSMs * std::min(chunk_pass_ctas_per_sm(n, m, gp1), chunk_pass_ctas_per_sm(n, m, gp3));
        const int64_t groups = std::max<int64_t>(1, slots / lanes);
        c = groups * lpc;
    } else {
        // the direct-load kernels: about 4096 (lane, chunk) units
        c = lanes >= 4096 ? 1 : (4096 + lanes - 1) / lanes;
    }
    if (c > max_chunks) c = max_chunks;
    *chunk = (T + c - 1) / c;
    *chunks = (T + *chunk - 1) / *chunk;
}

size_t mat_chunk_workspace_bytes(int n, int m, int64_t lanes, int64_t chunks) {
    return static_cast<size_t>(lanes) * static_cast<size_t>(chunks) *
           (static_cast<size_t>(n) * n + 2 * static_cast<size_t>(n) * m) * 4;
}

bool mat_chunked_tma_ok(const MatLaunch& L, bool dense, int64_t chunks, int64_t chunk) {
    int gp1 = 1;
    while (gp1 < L.m + L.n) gp1 <<= 1;
    if (L.projective || !chunked_tma_shape(L.n, L.m, dense)) return false;
    if (!mat_tma_ok(L.n, L.m, gp1, false, L.O, L.T, L.J, dense, L.a, L.b)) return false;
    if (reinterpret_cast<uintptr_t>(L.out) % 16 != 0) return false;
    // chunk coordinates, counts and grids in 32-bit
    const int64_t lim = int64_t(1) << 30;
    return chunks * chunk < lim && L.T < lim && L.g.lanes * chunks < lim && L.g.lanes == L.O * L.J;
}

cudaError_t launch_mat_chunked_tma(const MatLaunch& L, float* ws, int64_t chunks, int64_t chunk, const char** err) {
    switch (L.n) {
        case 2: return launch_chunked_tma_n<2>(L, ws, chunks, chunk, err);
        case 4: return launch_chunked_tma_n<4>(L, ws, chunks, chunk, err);
        case 8: return launch_chunked_tma_n<8>(L, ws, chunks, chunk, err);
        case 16: return launch_chunked_tma_n<16>(L, ws, chunks, chunk, err);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_mat_chunked(const MatLaunch& L, float* ws, int64_t chunks, int64_t chunk) {
    switch (L.n) {
#define ES_MAT_CASE(K) \
    case K: return launch_chunked_n<K>(L, ws, chunks, chunk);
        ES_MAT_CASE(1) ES_MAT_CASE(2) ES_MAT_CASE(3) ES_MAT_CASE(4) ES_MAT_CASE(5) ES_MAT_CASE(6) ES_MAT_CASE(7)
        ES_MAT_CASE(8) ES_MAT_CASE(9) ES_MAT_CASE(10) ES_MAT_CASE(11) ES_MAT_CASE(12) ES_MAT_CASE(13)
        ES_MAT_CASE(14) ES_MAT_CASE(15) ES_MAT_CASE(16)
#undef ES_MAT_CASE
    }
    return cudaErrorInvalidValue;
}

}  // namespace es
