// es_table.h -- table-scan launch description shared by the entry points
// (es_table_api.cu) and the kernels (k_table.cu).  Not part of the ABI.
#pragma once

#include "es_internal.h"

namespace es {

// One validated call in canonical form: symbols and states [O, T, J].
struct TableLaunch {
    const int* table;    // [n_states, n_syms]
    const int* sym;
    int* out;
    int64_t O, T, J;
    int n_states, n_syms, start;
    unsigned int* status;
    uint64_t wait_ns;
    int64_t drop_tile;
    cudaStream_t stream;
    int num_sms;
    EncodeTiledFn encode;
};

bool table_in_smem(int64_t n_states, int64_t n_syms);
bool table_lane_ok(int64_t O, int64_t T, int64_t J, const void* sym, const void* out);
bool table_time_ok(int64_t O, int64_t T, int64_t J, const void* sym, const void* out);
cudaError_t launch_table_generic(const TableLaunch& L);
cudaError_t launch_table_lane(const TableLaunch& L, const char** err);
cudaError_t launch_table_time(const TableLaunch& L, const char** err);

}  // namespace es
