// k_table.cu -- table-scan kernels ("Tensor operations": the `table-scan` row
// of the operations table and the section "table-scan").
//
//     h[t] = table[h[t-1], symbols[t]]        from h[-1] = start
//
// a deterministic automaton run along one axis of an i32 tensor of symbols,
// every state kept.  On CUDA a symbol outside [0, symbols) and a table entry
// outside [0, states) are clamped into range (as `gather` clamps an index);
// the clamped entry is the state, so every state stays a valid row.  Each
// step is one dependent lookup, so the pages' design is kept: one thread per
// sequence and the table in shared memory when it fits (it is copied there
// once per CTA); a table too large for shared memory is read through the
// read-only path from L2.  Around it, the GB300 pipelines of the element-scan
// kernels stream the symbols:
//   * k_table_lane: the sequence axis not last -- [O, T, I] with I sequences
//     side by side; a producer thread streams {LI sequences x TT trips} tiles
//     with TMA into an mbarrier ring, each thread copies its column of the
//     tile to registers, frees the stage, runs the lookups and stores one
//     coalesced row per trip and warp;
//   * k_table_time: the sequence axis last -- one row of T symbols per
//     sequence; {32 trips x 64 rows} tiles loaded with the 128-byte swizzle
//     (a thread reads its own row four trips at a time, conflict-free), the
//     states written into a swizzled tile and stored with a TMA tensor store;
//   * k_table_generic: any shape or alignment, one thread per sequence.
// Waits are bounded as in the other pipelines.
#include <algorithm>

#include "es_device.cuh"
#include "es_table.h"

namespace es {
namespace {

__device__ __forceinline__ int clamp_symbol(int s, int n_syms) { return min(max(s, 0), n_syms - 1); }

// The automaton's state is carried as its row offset, state * n_syms.  A
// table in shared memory is staged once per CTA as two arrays over the
// entries q = row * n_syms + symbol: the next state, clamped (`state_of`),
// and that state's row offset (`next_off`).  A step is then
//     off' = next_off[off + s]      (one add and one load on the chain)
// with the state read beside it, off the chain: state_of[off + s].  When
// n_syms is a power of two the state is off' >> log2(n_syms) and only
// next_off is staged: one shared-memory lookup a step, not two (the lookups,
// at random rows, are what the kernels' shared-memory traffic is made of).
//
// TAB: 0 the table read from global memory, 1 staged as both arrays, 2
// staged as next_off alone (n_syms a power of two).
struct TableSmem {
    const int* next_off;
    const int* state_of;
};

// copy and prepare the table (every thread of the CTA takes part)
template <int TAB>
__device__ __forceinline__ TableSmem stage_table(int* dst, const int* __restrict__ src, int n_states, int n_syms) {
    const int entries = n_states * n_syms;
    int* next_off = dst;
    int* state_of = dst + entries;
    for (int q = threadIdx.x; q < entries; q += blockDim.x) {
        const int e = min(max(__ldg(src + q), 0), n_states - 1);
        if constexpr (TAB == 1) state_of[q] = e;
        next_off[q] = e * n_syms;
    }
    return TableSmem{next_off, state_of};
}

// One step of a row-offset-carrying run: returns the state after symbol `s`
// (already clamped) and advances `off`.  A table left in global memory is
// read through the read-only path and clamped on the way.  `sh` is
// log2(n_syms) (TAB 2).
template <int TAB>
__device__ __forceinline__ int table_step(int& off, int s, const TableSmem& ts, const int* __restrict__ table,
                                          int n_syms, int hi, int sh) {
    const int q = off + s;
    if constexpr (TAB == 2) {
        off = ts.next_off[q];
        return off >> sh;
    } else if constexpr (TAB == 1) {
        off = ts.next_off[q];
        return ts.state_of[q];
    } else {
        const int e = min(max(__ldg(table + q), 0), hi);
        off = e * n_syms;
        return e;
    }
}

// shared memory a staged table takes (both arrays)
__host__ __device__ constexpr size_t staged_table_bytes(int64_t n_states, int64_t n_syms) {
    return static_cast<size_t>(n_states) * static_cast<size_t>(n_syms) * 8;
}

// the staging a launch uses, and the shared memory it takes
int table_mode(bool smem, int n_syms) { return !smem ? 0 : (n_syms & (n_syms - 1)) == 0 ? 2 : 1; }
size_t table_mode_bytes(int tab, int64_t n_states, int64_t n_syms) {
    return tab == 0 ? 0 : tab == 2 ? staged_table_bytes(n_states, n_syms) / 2 : staged_table_bytes(n_states, n_syms);
}

// ---------------------------------------------------------------------------
// any layout

template <int TAB>
__global__ void __launch_bounds__(128)
k_table_generic(const int* __restrict__ table, const int* __restrict__ sym, int* __restrict__ out, int64_t O,
                int64_t T, int64_t J, int n_states, int n_syms, int start) {
    extern __shared__ int tab_s[];
    TableSmem ts{};
    if constexpr (TAB > 0) {
        ts = stage_table<TAB>(tab_s, table, n_states, n_syms);
        __syncthreads();
    }
    const int64_t lane = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (lane >= O * J) return;
    const int64_t o = lane / J;
    const int64_t j = lane - o * J;
    int off = start * n_syms;
    const int hi = n_states - 1;
    const int sh = __ffs(n_syms) - 1;
    const int* sp = sym + o * T * J + j;
    int* op = out + o * T * J + j;
    for (int64_t t = 0; t < T; ++t) {
        const int h = table_step<TAB>(off, clamp_symbol(__ldg(sp + t * J), n_syms), ts, table, n_syms, hi, sh);
        __stcs(op + t * J, h);
    }
}

// ---------------------------------------------------------------------------
// sequences side by side (the axis not last)

constexpr int kTabMaxStages = 6;
constexpr int kTabTT = 32;

template <int LI, int TAB>
__global__ void __launch_bounds__(32 + LI)
k_table_lane(const __grid_constant__ CUtensorMap map_s, const int* __restrict__ table, int* __restrict__ out, int T,
             int I, int tiles_i, int stages, int n_states, int n_syms, int start, unsigned int* status,
             uint64_t wait_ns, int64_t drop_tile) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kTabMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kTabMaxStages];
    __shared__ int abort_flag;
    constexpr int kTileInts = kTabTT * LI;
    int* tiles = reinterpret_cast<int*>(smem_raw + smem_align_pad(smem_raw));
    TableSmem ts{};
    if constexpr (TAB > 0) ts = stage_table<TAB>(tiles + stages * kTileInts, table, n_states, n_syms);

    const int o = blockIdx.x / tiles_i;
    const int i0 = (blockIdx.x % tiles_i) * LI;
    const int ntiles = (T + kTabTT - 1) / kTabTT;
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
    __syncthreads();   // barriers and the staged table

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&map_s);
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
                mbar_arrive_expect_tx(&full_bar[s], kTileInts * 4u);
                tma_load_3d(tiles + s * kTileInts, &map_s, i0, k * kTabTT, o, &full_bar[s], pol);
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
    const int hi = n_states - 1;
    const int sh = __ffs(n_syms) - 1;
    int off = start * n_syms;
    int* obase = out + static_cast<int64_t>(o) * T * I + i;
    for (int k = 0; k < ntiles; ++k) {
        const int s = k % stages;
        const bool ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        const int t0 = k * kTabTT;
        const int n = min(kTabTT, T - t0);
        const int* st = tiles + s * kTileInts + c;
        // the tile's symbols go to registers (clamped) and the stage is freed
        int sr[kTabTT];
#pragma unroll
        for (int tt = 0; tt < kTabTT; ++tt) sr[tt] = clamp_symbol(st[tt * LI], n_syms);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        int* op = obase + static_cast<int64_t>(t0) * I;
        // the state stored goes to one of two registers by trip parity: a
        // lookup never overwrites the register the previous trip's store may
        // still be reading
        int hv[2];
        auto trip = [&](const int tt) {
            hv[tt & 1] = table_step<TAB>(off, sr[tt], ts, table, n_syms, hi, sh);
            if (valid) __stcs(op + static_cast<int64_t>(tt) * I, hv[tt & 1]);
        };
        if (n == kTabTT) {
#pragma unroll
            for (int tt = 0; tt < kTabTT; ++tt) trip(tt);
        } else {
#pragma unroll
            for (int tt = 0; tt < kTabTT; ++tt)
                if (tt < n) trip(tt);
        }
    }
}

// ---------------------------------------------------------------------------
// the sequence axis last

constexpr int kTabLO = 64;
constexpr int kTabOutBufs = 3;

template <int TAB>
__global__ void __launch_bounds__(32 + kTabLO)
k_table_time(const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_out,
             const int* __restrict__ table, int O, int T, int stages, int n_states, int n_syms, int start,
             unsigned int* status, uint64_t wait_ns, int64_t drop_tile) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kTabMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kTabMaxStages];
    __shared__ int abort_flag;
    constexpr uint32_t kTileBytes = kTabLO * 128u;
    unsigned char* base = smem_raw + smem_align_pad(smem_raw);
    unsigned char* in_tiles = base;
    unsigned char* out_tiles = base + static_cast<size_t>(stages) * kTileBytes;
    TableSmem ts{};
    if constexpr (TAB > 0)
        ts = stage_table<TAB>(reinterpret_cast<int*>(out_tiles + kTabOutBufs * kTileBytes), table, n_states, n_syms);

    const int o0 = blockIdx.x * kTabLO;
    const int ntiles = (T + 31) / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kTabLO / 32);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();   // barriers and the staged table

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&map_s);
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
                mbar_arrive_expect_tx(&full_bar[s], kTileBytes);
                tma_load_2d(in_tiles + static_cast<size_t>(s) * kTileBytes, &map_s, k * 32, o0, &full_bar[s], pol);
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
    const int hi = n_states - 1;
    const int sh = __ffs(n_syms) - 1;
    int off = start * n_syms;
    const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
    const uint32_t swz = static_cast<uint32_t>(r & 7);   // 128-byte swizzle: chunk q lives at q ^ (row % 8)
    const bool storer = (threadIdx.x == 32);
    for (int k = 0; k <= ntiles; ++k) {
        const int s = k % stages;
        bool ok = true;
        if (k < ntiles) ok = mbar_wait_bounded(&full_bar[s], (k / stages) & 1, wait_ns, &abort_flag);
        if (k > 0) fence_proxy_async_smem();     // this thread's writes of tile k-1
        if (consumer_vote_any_failed(!ok, kTabLO)) {
            if (!ok) report_timeout(status, &abort_flag);
            break;
        }
        if (storer && k > 0) {
            tma_store_2d(&map_out, (k - 1) * 32, o0,
                         out_tiles + static_cast<size_t>((k - 1) % kTabOutBufs) * kTileBytes);
            bulk_commit();
            bulk_wait_read<1>();
        }
        if (k == ntiles) break;
        const int nq = min(32, T - k * 32) >> 2;     // T % 4 == 0 on this path
        const unsigned char* srow = in_tiles + static_cast<size_t>(s) * kTileBytes + row_off;
        unsigned char* orow = out_tiles + static_cast<size_t>(k % kTabOutBufs) * kTileBytes + row_off;
        int4 seg[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) seg[q] = *reinterpret_cast<const int4*>(srow + ((static_cast<uint32_t>(q) ^ swz) << 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        auto quad = [&](const int q) {
            int4 v;
            v.x = table_step<TAB>(off, clamp_symbol(seg[q].x, n_syms), ts, table, n_syms, hi, sh);
            v.y = table_step<TAB>(off, clamp_symbol(seg[q].y, n_syms), ts, table, n_syms, hi, sh);
            v.z = table_step<TAB>(off, clamp_symbol(seg[q].z, n_syms), ts, table, n_syms, hi, sh);
            v.w = table_step<TAB>(off, clamp_symbol(seg[q].w, n_syms), ts, table, n_syms, hi, sh);
            *reinterpret_cast<int4*>(orow + ((static_cast<uint32_t>(q) ^ swz) << 4)) = v;
        };
        // full tiles run unguarded (one basic block); only a ragged last tile
        // checks every group of four trips
        if (nq == 8) {
#pragma unroll
            for (int q = 0; q < 8; ++q) quad(q);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < nq) quad(q);
        }
    }
    if (storer) bulk_wait_all();
}

template <int TAB>
cudaError_t launch_generic_t(const TableLaunch& L, size_t table_bytes) {
    const int64_t lanes = L.O * L.J;
    const int64_t blocks = (lanes + 127) / 128;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = table_bytes;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_table_generic<TAB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    k_table_generic<TAB><<<static_cast<unsigned>(blocks), 128, smem, L.stream>>>(
        L.table, L.sym, L.out, L.O, L.T, L.J, L.n_states, L.n_syms, L.start);
    return cudaGetLastError();
}

template <int LI, int TAB>
cudaError_t launch_lane_t(const TableLaunch& L, const CUtensorMap& ms, int tiles_i, int stages, size_t smem) {
    auto kern = k_table_lane<LI, TAB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(L.O * tiles_i), 32 + LI, smem, L.stream>>>(
        ms, L.table, L.out, static_cast<int>(L.T), static_cast<int>(L.J), tiles_i, stages, L.n_states, L.n_syms,
        L.start, L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

template <int TAB>
cudaError_t launch_time_t(const TableLaunch& L, const CUtensorMap& ms, const CUtensorMap& mo, int stages,
                          size_t smem) {
    auto kern = k_table_time<TAB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>((L.O + kTabLO - 1) / kTabLO), 32 + kTabLO, smem, L.stream>>>(
        ms, mo, L.table, static_cast<int>(L.O), static_cast<int>(L.T), stages, L.n_states, L.n_syms, L.start,
        L.status, L.wait_ns, L.drop_tile);
    return cudaGetLastError();
}

}  // namespace

// a table of at most 32 KB (64 KB staged) goes to shared memory
bool table_in_smem(int64_t n_states, int64_t n_syms) { return staged_table_bytes(n_states, n_syms) <= 64 * 1024; }

bool table_lane_ok(int64_t O, int64_t T, int64_t J, const void* sym, const void* out) {
    if (J < 32 || J % 4 != 0) return false;
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || J >= (int64_t(1) << 31)) return false;
    if (O * ((J + 31) / 32) >= (int64_t(1) << 31)) return false;
    return reinterpret_cast<uintptr_t>(sym) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
}

bool table_time_ok(int64_t O, int64_t T, int64_t J, const void* sym, const void* out) {
    if (J != 1 || T % 4 != 0 || T < 32) return false;
    if (O >= (int64_t(1) << 31) || T >= (int64_t(1) << 31)) return false;
    return reinterpret_cast<uintptr_t>(sym) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
}

cudaError_t launch_table_generic(const TableLaunch& L) {
    const int tab = table_mode(table_in_smem(L.n_states, L.n_syms), L.n_syms);
    const size_t tb = table_mode_bytes(tab, L.n_states, L.n_syms);
    return tab == 2 ? launch_generic_t<2>(L, tb) : tab == 1 ? launch_generic_t<1>(L, tb) : launch_generic_t<0>(L, tb);
}

cudaError_t launch_table_lane(const TableLaunch& L, const char** err) {
    const int tab = table_mode(table_in_smem(L.n_states, L.n_syms), L.n_syms);
    const size_t tb = table_mode_bytes(tab, L.n_states, L.n_syms);
    // 64 sequences per CTA and two stages: a lookup chain per thread leaves
    // latency that more CTAs per SM cover (on GB300 the lanes workload took
    // 0.49 / 0.47 / 0.41 ms at 4 / 3 / 2 stages with 128 sequences per CTA,
    // 0.38 ms with 64)
    const int64_t I = L.J;
    const int LI = I >= 64 && 5 * L.O * ((I + 63) / 64) >= 4LL * L.num_sms ? 64 : 32;
    const int64_t tiles_i = (I + LI - 1) / LI;
    const int stages = 2;
    const size_t smem = static_cast<size_t>(stages) * kTabTT * LI * 4 + tb + 1024;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(L.T), static_cast<cuuint64_t>(L.O)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(I) * 4, static_cast<cuuint64_t>(I) * L.T * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(LI), static_cast<cuuint32_t>(kTabTT), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap ms;
    if (L.encode(&ms, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, const_cast<int*>(L.sym), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for the table-scan symbol map";
        return cudaErrorInvalidValue;
    }
    const int ti = static_cast<int>(tiles_i);
    if (tab == 2) return LI == 64 ? launch_lane_t<64, 2>(L, ms, ti, stages, smem)
                                  : launch_lane_t<32, 2>(L, ms, ti, stages, smem);
    if (tab == 1) return LI == 64 ? launch_lane_t<64, 1>(L, ms, ti, stages, smem)
                                  : launch_lane_t<32, 1>(L, ms, ti, stages, smem);
    return LI == 64 ? launch_lane_t<64, 0>(L, ms, ti, stages, smem) : launch_lane_t<32, 0>(L, ms, ti, stages, smem);
}

cudaError_t launch_table_time(const TableLaunch& L, const char** err) {
    const int tab = table_mode(table_in_smem(L.n_states, L.n_syms), L.n_syms);
    const size_t tb = table_mode_bytes(tab, L.n_states, L.n_syms);
    const int stages = 2;   // more CTAs per SM beat a deeper ring (0.43 ms at 4 stages, 0.38 at 2)
    const size_t smem = (static_cast<size_t>(stages) + kTabOutBufs) * kTabLO * 128 + tb + 1024;
    CUtensorMap maps[2];
    const int* bases[2] = {L.sym, L.out};
    for (int q = 0; q < 2; ++q) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.T), static_cast<cuuint64_t>(L.O)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.T) * 4};
        const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kTabLO)};
        const cuuint32_t estr[2] = {1, 1};
        if (L.encode(&maps[q], CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int*>(bases[q]), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled failed for a time-innermost table-scan map";
            return cudaErrorInvalidValue;
        }
    }
    return tab == 2 ? launch_time_t<2>(L, maps[0], maps[1], stages, smem)
           : tab == 1 ? launch_time_t<1>(L, maps[0], maps[1], stages, smem)
                      : launch_time_t<0>(L, maps[0], maps[1], stages, smem);
}

}  // namespace es
