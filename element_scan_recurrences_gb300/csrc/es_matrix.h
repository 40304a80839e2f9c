// es_matrix.h -- matrix-scan launch descriptions shared by the entry points
// (es_matrix_api.cu) and the kernels (k_matrix.cu).  Not part of the ABI.
#pragma once

#include "es_internal.h"

namespace es {

// Lanes of a matrix-scan with broadcast leading dims: a lane index splits
// into the non-axis leading coordinates (row-major over dim[0..nd)); each
// operand advances by its own stride per coordinate and along the axis, in
// matrices (0 where the operand is broadcast).
struct MatGeom {
    int64_t lanes;
    int64_t T;
    int nd;
    int64_t dim[ES_MAX_RANK];
    int64_t sa[ES_MAX_RANK], sb[ES_MAX_RANK], so[ES_MAX_RANK];
    int64_t ta, tb, to;
};

struct MatLaunch {
    const float* a;
    const float* b;
    float* out;
    int n, m;
    int gp;              // threads per lane group: a power of two >= the columns carried
    bool projective;
    int reverse;
    bool trans;          // the gradient's cotangent scan: a[t + a_shift]^T (zero off the axis)
    int a_shift;
    MatGeom g;           // any layout (generic kernel)
    int64_t O, T, J;     // dense canonical view [O, T, J] of the leading dims (TMA kernel)
    // TMA full scan only: the trips [win0, win0 + win_len) of the axis (0
    // length: all of it), started from the states at `carry` (the dense
    // [O, J] view of one trip of `out`; null: from zero)
    int64_t win0 = 0, win_len = 0;
    const float* carry = nullptr;
    unsigned int* status;
    uint64_t wait_ns;
    int64_t drop_tile;
    cudaStream_t stream;
    int num_sms;
    EncodeTiledFn encode;
};

cudaError_t launch_mat_generic(const MatLaunch& L);

// da[t] = lam[t] @ h_prev^T over the dense view [O, T, J] of n x m blocks
// (h_prev: the state before trip t in scan order, zero before the first), for
// the trips [t_lo, t_lo + t_cnt) (t_cnt < 0: all of them).
cudaError_t launch_mat_da(const float* lam, const float* states, float* da, int n, int64_t O, int64_t T,
                          int64_t J, int m, int reverse, cudaStream_t stream, int64_t t_lo = 0, int64_t t_cnt = -1);
cudaError_t launch_mat_tma(const MatLaunch& L, const char** err);

// The chunked scan for few long lanes (three launches, a caller workspace):
// how to cut T, the workspace it needs, and the launch.
void mat_chunk_shape(int n, int m, bool dense, int64_t lanes, int64_t T, int64_t* chunks, int64_t* chunk);
size_t mat_chunk_workspace_bytes(int n, int m, int64_t lanes, int64_t chunks);
cudaError_t launch_mat_chunked(const MatLaunch& L, float* ws, int64_t chunks, int64_t chunk);
// The same chunked scan with its two scan passes on the TMA kernel (dense
// operands as the TMA kernel takes them, n + m <= 32) and a pipelined link
// pass; the same workspace layout, the same results bit for bit.  With
// `trans` set it runs the gradient's cotangent scan, chunked the same way.
bool mat_chunked_tma_ok(const MatLaunch& L, bool dense, int64_t chunks, int64_t chunk);
cudaError_t launch_mat_chunked_tma(const MatLaunch& L, float* ws, int64_t chunks, int64_t chunk, const char** err);

// The TMA kernel serves dense operands with n in {2, 4, 8, 16}, 16-byte
// aligned bases, n*m a multiple of 4 and at most 256, and a lane group of at
// most 32 threads.
bool mat_tma_ok(int n, int m, int gp, bool projective, int64_t O, int64_t T, int64_t J, bool dense, const void* a,
                const void* b);

}  // namespace es
