// Internal interface between the C-ABI front end (pa_api.cu) and the kernel
// translation units (pa_kv.cu, pa_decode.cu).  Not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

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
    int* ticket;                // [2] work ticket and retired-CTA count, zero between launches
    int* sched;                 // [S + 3] PT, item count, first item of each sequence
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

// Decode workspace header: ticket[2], 2 spare ints, then the published
// schedule (PT, item count, S + 1 item offsets); zeroed before first use.
inline size_t decode_header_bytes(int S) {
    return ((static_cast<size_t>(S) + 8) * sizeof(int) + 255) / 256 * 256;
}

namespace pa_detail {

void count_launch();

// Launch `kernel` on `st` allowing programmatic dependent launch (the kernel
// must call pa_dev::wait_prior_grid() before reading any input).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

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
