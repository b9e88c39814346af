// Internal interface between the C-ABI front end (pa_api.cu) and the kernel
// translation units (pa_kv.cu, pa_decode.cu).  Not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "pa.h"

struct pa_pool {
    int device = 0;
    int num_blocks = 0, block_size = 0, kv_heads = 0, head_dim = 0;
    pa_dtype dtype = PA_BF16;
    void* k = nullptr;          // K [num_blocks][kv_heads][block_size][head_dim]
    void* v = nullptr;          // V [num_blocks][kv_heads][head_dim][block_size]
    int* err = nullptr;         // device error word (first recorded PA_ERR_*)
    void* ws = nullptr;         // decode workspace: counters, then partials
    size_t ws_bytes = 0;
    int num_sms = 0;
};

// Everything one decode launch needs, passed by value to the kernels.
struct DecodeParams {
    const void* q;              // [S][Hq][D]
    const void* k;              // pool K
    const void* v;              // pool V (transposed tiles)
    const int32_t* tables;      // [S][max_blocks]
    const int32_t* lens;        // [S]
    void* out;                  // [S][Hq][D]
    float* part_acc;            // [max_items][G][D]  un-normalised partial sums
    float* part_ml;             // [max_items][G][2]  (running max, sum) in log2 units
    int* counters;              // [S][Hkv] arrival counters, zero between launches
    int* err;
    float scale_log2;           // scale * log2(e)
    int S, Hq, Hkv, G, D, B, num_blocks, max_blocks;
    int out_bf16;
    int items_target;           // wanted number of work items (fast path)
    int pt_min;                 // smallest partition, tokens (multiple of B)
    int pt_fixed;               // > 0: use exactly this partition size
};

// Sizes of the decode workspace for a launch shape.
struct DecodeWorkspace {
    size_t counters_bytes;      // S * Hkv ints, rounded to 256
    size_t max_items;
    size_t bytes;               // total
};

namespace pa_detail {

void count_launch();

// Launchers; each returns PA_OK or PA_ERR_CUDA (launch failure).
int launch_append(const pa_pool* p, const void* k, const void* v, const int64_t* slots,
                  int T, cudaStream_t st);
int launch_copy(const pa_pool* p, const int64_t* pairs, int P, cudaStream_t st);

// Decode: how the launch is shaped for a pool and batch.
struct DecodePlan {
    bool fast;                  // bf16 tensor-core path
    bool bf16;                  // pool element type is bf16
    int grid, threads;
    size_t smem;
    int items_target, pt_min, pt_fixed;
    size_t max_items;
};
int plan_decode(const pa_pool* p, int S, int Hq, int max_blocks, DecodePlan* plan);
int launch_decode(const DecodePlan& plan, const DecodeParams& prm, cudaStream_t st);

}  // namespace pa_detail
