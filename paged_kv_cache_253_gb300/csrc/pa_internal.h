// Internal interface between the C-ABI front end (pa_api.cu) and the kernel
// translation units (pa_kv.cu, pa_decode.cu).  Not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pa.h"

struct pa_pool {
    int device = 0;
    int num_blocks = 0, block_size = 0, kv_heads = 0, head_dim = 0;
    pa_dtype dtype = PA_BF16;
    float k_scale = 1.f, v_scale = 1.f;   // fp8 pools: a code stands for e4m3(code) * scale
    void* k = nullptr;          // K [num_blocks][kv_heads][block_size][head_dim]
    void* v = nullptr;          // V [num_blocks][kv_heads][head_dim][block_size]
    int* err = nullptr;         // device error word (first recorded PA_ERR_*)
    void* ws = nullptr;         // decode workspace: header, then partials
    size_t ws_bytes = 0;
    int num_sms = 0;
    int smem_optin = 0;         // largest dynamic shared memory a CTA may opt in to
    // TMA descriptors of K (boxes 64 d x 16 tokens, 128-byte swizzle) and of V^T
    // (boxes 16 tokens x 128 d, 32-byte swizzle), made on first use
    CUtensorMap kmap;
    CUtensorMap vmap;
    bool tmaps_ready = false;
    // kernel-choice options (pa_pool_set_option)
    int opt_partition_cap = -1;     // decode partition cap, tokens; -1 automatic, 0 none
    int opt_shared_kernel = 0;      // 0 tcgen05 where eligible, 1 mma.sync
    int opt_prefill_kernel = 0;     // 0 tcgen05 where eligible, 1 mma.sync
    // shared-prefix descriptor last uploaded by pa_decode_shared (host copy + device copy)
    std::vector<int> desc_host;
    int* desc_dev = nullptr;
    size_t desc_cap = 0;        // ints
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
    float scale_log2;           // scale * log2(e) (* k_scale for an fp8 pool)
    float v_scale;              // factor on the value sums (fp8 pool's v_scale, else 1)
    float k_scale;              // fp8 pool's k_scale (quantizing a fused append), else 1
    int S, Hq, Hkv, G, D, B, num_blocks, max_blocks;
    int out_bf16;
    int items_target;           // wanted number of work items (fast path)
    int pt_min;                 // smallest partition, tokens (multiple of B)
    int pt_soft;                // > pt_min: the smallest partition grows towards this many
                                // tokens (multiple of B) while at least items_floor items remain
    int items_floor;            // (both zero: pt_min alone)
    int wave_items;             // > 0: the item target is whole waves of this many items,
    int wave_tokens;            // one wave per wave_tokens token-heads per item, at most
                                // items_target
    int pt_max;                 // largest partition, tokens (multiple of B; 0: no cap)
    int max_items;              // partial slots the workspace holds (fast path)
    int pt_fixed;               // > 0: use exactly this partition size
    // Shared-prefix description (pa_decode_shared); all zero / null otherwise.
    int n_shared_items;         // shared work items, heads included (K * Hkv)
    int chunk_tokens;           // shared tokens per item (multiple of B)
    int members_per_tile;       // group members per item (16-row tiles of members x G)
    const int* sh_items;        // [K][4] (group, member tile, chunk, 0)
    const int* seq_group;       // [S] group of each sequence, -1 if none
    const int* seq_member;      // [S] index of the sequence inside its group
    const int* seq_start;       // [S] first private token (the shared span precedes it)
    const int* g_members_off;   // [Ng + 1]
    const int* g_members;       // batch indices, grouped
    const int* g_nchunks;       // [Ng] shared chunks of each group
    const int* g_spart_base;    // [Ng] first shared-partial slot of each group
    const int* g_shared_tokens; // [Ng] shared tokens of each group
    float* spart_acc;           // [slots][Hkv][G][D] shared-span partial sums
    float* spart_ml;            // [slots][Hkv][G][2]
    // Fused append (pa_append_decode): each sequence's new token, written by
    // the warp that reads the sequence's last block; null otherwise.
    const void* new_k;          // [S][Hkv][D]
    const void* new_v;          // [S][Hkv][D]
    const int64_t* new_slots;   // [S] slot of position L-1 of each sequence, or < 0
    // 1: the preceding kernel is the tcgen05 shared-prefix kernel, which already
    // waited for the work before it; the split kernel then runs alongside it and
    // waits for it only before exiting (so the merge after it sees both).
    int defer_wait;
};

// Everything one prefill launch needs (pa_prefill), passed by value.
struct PrefillParams {
    const uint16_t* q;          // [T][Hq][D] bf16
    const void* k;              // pool K (bf16 values or e4m3 codes)
    const void* v;              // pool V^T tiles
    const int32_t* cu_q;        // [S + 1] first query row of each sequence
    const int32_t* tables;      // [S][max_blocks]
    const int32_t* lens;        // [S] context length after the chunk's append
    void* out;                  // [T][Hq][D]
    int* err;
    float scale_log2;           // scale * log2(e) (* k_scale for an fp8 pool)
    float v_scale;              // factor on the outputs (fp8 pool's v_scale, else 1)
    int T, S, Hq, Hkv, G, B, num_blocks, max_blocks;
    int max_q;                  // longest chunk the launch was sized for
    int out_bf16;
};

// Bytes of one K or V element of the pool.
inline size_t pool_elem_size(pa_dtype t) { return t == PA_FP8E4M3 ? 1 : t == PA_BF16 ? 2 : 4; }

// Score factor of a decode in log2 units (an fp8 pool's k_scale folded in)
// and the factor on the value sums.
inline void decode_scales(const pa_pool* pool, float scale, DecodeParams* p) {
    const bool f8 = pool->dtype == PA_FP8E4M3;
    p->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 *
                                       (f8 ? static_cast<double>(pool->k_scale) : 1.0));
    p->v_scale = f8 ? pool->v_scale : 1.f;
    p->k_scale = f8 ? pool->k_scale : 1.f;
}

// Decode workspace header: ticket[2], 2 spare ints, the published schedule
// (S + 3 ints used of S + 4); zeroed before first use (the kernels reset the
// tickets they count).
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
    bool shared = false;        // shared-prefix items present (fast path only)
    bool fuse = false;          // the decode kernel also appends each sequence's new token
    bool tc = false;            // shared items run in the tcgen05 kernel before the split pass
    pa_pool* pool = nullptr;
    bool fast;                  // tensor-core path (bf16 pool, or fp8 codes widened to f16)
    bool bf16;                  // pool element type is bf16
    bool fp8;                   // pool element type is e4m3
    int grid, threads;
    size_t smem;
    int items_target, pt_min, pt_max = 0, pt_fixed;
    int pt_soft = 0, items_floor = 0;
    int wave_items = 0, wave_tokens = 0;
    size_t max_items;
    size_t min_items;           // fewest partial slots the kernel can work with (fast path)
};
int plan_decode(pa_pool* p, int S, int Hq, int max_blocks, DecodePlan* plan);
// Host checks of pa_decode's arguments (shared by every decode entry point).
int check_decode_args(const pa_pool* pool, const void* q, int S, int Hq, const int32_t* tables,
                      int max_blocks, const int32_t* lens, const void* out, pa_dtype out_dtype);
int launch_decode(const DecodePlan& plan, const DecodeParams& prm, cudaStream_t st);

// TMA descriptors of the pool's K and V^T (16-token blocks), made once per pool.
int ensure_tensor_maps(pa_pool* pool);

// tcgen05 shared-prefix items (pa_shared_tc.cu).
bool shared_tc_eligible(const pa_pool* pool, int G);
int shared_tc_rows();
int shared_tc_chunk_tokens();     // shared tokens per item (a multiple of 16)
int launch_shared_tc(pa_pool* pool, const DecodeParams& p, cudaStream_t st);

// tcgen05 prefill (pa_shared_tc.cu): one CTA per (128 query rows, KV head,
// sequence); bf16 pools of 16-token blocks, head_dim 128.
bool prefill_tc_eligible(const pa_pool* pool);
int prefill_tc_rows();
int launch_prefill_tc(pa_pool* pool, const PrefillParams& p, dim3 grid, cudaStream_t st);

}  // namespace pa_detail
