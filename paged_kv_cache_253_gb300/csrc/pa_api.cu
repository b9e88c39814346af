// C-ABI front end of libpagedattn: pool lifetime, argument checks, decode
// workspace and the device error word.  Semantics are documented in pa.h.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa_detail {

static std::atomic<uint64_t> g_launch_counter{0};
void count_launch() { g_launch_counter.fetch_add(1, std::memory_order_relaxed); }

}  // namespace pa_detail

namespace {

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

size_t elem_size(pa_dtype t) { return pool_elem_size(t); }

// Workspace: [header: ticket + schedule, 256-aligned][part_acc][part_ml]
size_t workspace_bytes(const pa_detail::DecodePlan& plan, int S, int G, int D,
                       size_t* counters_bytes) {
    const size_t cb = decode_header_bytes(S);
    const size_t acc = round256(plan.max_items * G * D * sizeof(float));
    const size_t ml = round256(plan.max_items * G * 2 * sizeof(float));
    if (counters_bytes) *counters_bytes = cb;
    return cb + acc + ml;
}

// Grow the pool's workspace to at least `bytes`; new memory is zeroed (the
// work ticket must start at zero; the kernel resets it after use).
int ensure_workspace(pa_pool* pool, size_t bytes) {
    if (pool->ws_bytes >= bytes) return PA_OK;
    if (pool->ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
        cudaFree(pool->ws);
        pool->ws = nullptr;
        pool->ws_bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemset(p, 0, bytes) != cudaSuccess) {
        cudaFree(p);
        return PA_ERR_CUDA;
    }
    pool->ws = p;
    pool->ws_bytes = bytes;
    return PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

int pa_pool_create(int num_blocks, int block_size, int kv_heads, int head_dim, pa_dtype dtype,
                   pa_pool** out) {
    if (!out || num_blocks <= 0 || block_size <= 0 || block_size > 1024 || kv_heads <= 0 ||
        head_dim <= 0 || head_dim > 256 || head_dim % 4 != 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8E4M3) return PA_ERR_DTYPE;
    *out = nullptr;
    pa_pool* p = new (std::nothrow) pa_pool();
    if (!p) return PA_ERR_OUT_OF_MEMORY;
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&p->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               p->device) != cudaSuccess) {
        delete p;
        return PA_ERR_CUDA;
    }
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->kv_heads = kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    const size_t bytes =
        static_cast<size_t>(num_blocks) * kv_heads * block_size * head_dim * elem_size(dtype);
    if (cudaMalloc(&p->k, bytes) != cudaSuccess || cudaMalloc(&p->v, bytes) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&p->err), sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->k);
        cudaFree(p->v);
        cudaFree(p->err);
        delete p;
        return PA_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemset(p->k, 0, bytes) != cudaSuccess || cudaMemset(p->v, 0, bytes) != cudaSuccess ||
        cudaMemset(p->err, 0, sizeof(int)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(p->k);
        cudaFree(p->v);
        cudaFree(p->err);
        delete p;
        return PA_ERR_CUDA;
    }
    *out = p;
    return PA_OK;
}

int pa_pool_destroy(pa_pool* pool) {
    if (!pool) return PA_OK;
    DeviceGuard g(pool->device);
    cudaDeviceSynchronize();
    cudaFree(pool->k);
    cudaFree(pool->v);
    cudaFree(pool->err);
    cudaFree(pool->ws);
    cudaFree(pool->desc_dev);
    delete pool;
    return PA_OK;
}

int pa_pool_kv_ptrs(pa_pool* pool, void** k, void** v) {
    if (!pool) return PA_ERR_INVALID_ARG;
    if (k) *k = pool->k;
    if (v) *v = pool->v;
    return PA_OK;
}

static int pool_copy(pa_pool* pool, void* k_dst, const void* k_src, void* v_dst,
                     const void* v_src, void* stream) {
    DeviceGuard g(pool->device);
    if (!g.ok) return PA_ERR_CUDA;
    const size_t bytes = static_cast<size_t>(pool->num_blocks) * pool->kv_heads *
                         pool->block_size * pool->head_dim * elem_size(pool->dtype);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(k_dst, k_src, bytes, cudaMemcpyDefault, st) != cudaSuccess ||
        cudaMemcpyAsync(v_dst, v_src, bytes, cudaMemcpyDefault, st) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

int pa_pool_export(pa_pool* pool, void* k_dst, void* v_dst, void* stream) {
    if (!pool || !k_dst || !v_dst) return PA_ERR_INVALID_ARG;
    return pool_copy(pool, k_dst, pool->k, v_dst, pool->v, stream);
}

int pa_pool_import(pa_pool* pool, const void* k_src, const void* v_src, void* stream) {
    if (!pool || !k_src || !v_src) return PA_ERR_INVALID_ARG;
    return pool_copy(pool, pool->k, k_src, pool->v, v_src, stream);
}

int pa_pool_info(const pa_pool* pool, int* num_blocks, int* block_size, int* kv_heads,
                 int* head_dim, int* dtype) {
    if (!pool) return PA_ERR_INVALID_ARG;
    if (num_blocks) *num_blocks = pool->num_blocks;
    if (block_size) *block_size = pool->block_size;
    if (kv_heads) *kv_heads = pool->kv_heads;
    if (head_dim) *head_dim = pool->head_dim;
    if (dtype) *dtype = pool->dtype;
    return PA_OK;
}

int pa_pool_set_kv_scales(pa_pool* pool, float k_scale, float v_scale) {
    if (!pool) return PA_ERR_INVALID_ARG;
    if (pool->dtype != PA_FP8E4M3) return PA_ERR_DTYPE;
    // finite and positive (NaN fails both comparisons)
    if (!(k_scale > 0.f && k_scale <= 3.4028235e38f) || !(v_scale > 0.f && v_scale <= 3.4028235e38f))
        return PA_ERR_INVALID_ARG;
    pool->k_scale = k_scale;
    pool->v_scale = v_scale;
    return PA_OK;
}

int pa_pool_kv_scales(const pa_pool* pool, float* k_scale, float* v_scale) {
    if (!pool) return PA_ERR_INVALID_ARG;
    if (k_scale) *k_scale = pool->k_scale;
    if (v_scale) *v_scale = pool->v_scale;
    return PA_OK;
}

int pa_pool_set_option(pa_pool* pool, pa_option option, int value) {
    if (!pool) return PA_ERR_INVALID_ARG;
    switch (option) {
        case PA_OPT_PARTITION_CAP:
            if (value < -1) return PA_ERR_INVALID_ARG;
            pool->opt_partition_cap = value;
            return PA_OK;
        case PA_OPT_SHARED_KERNEL:
            if (value != 0 && value != 1) return PA_ERR_INVALID_ARG;
            pool->opt_shared_kernel = value;
            return PA_OK;
        case PA_OPT_PREFILL_KERNEL:
            if (value != 0 && value != 1) return PA_ERR_INVALID_ARG;
            pool->opt_prefill_kernel = value;
            return PA_OK;
        default:
            return PA_ERR_INVALID_ARG;
    }
}

int pa_pool_get_option(const pa_pool* pool, pa_option option, int* value) {
    if (!pool || !value) return PA_ERR_INVALID_ARG;
    switch (option) {
        case PA_OPT_PARTITION_CAP: *value = pool->opt_partition_cap; return PA_OK;
        case PA_OPT_SHARED_KERNEL: *value = pool->opt_shared_kernel; return PA_OK;
        case PA_OPT_PREFILL_KERNEL: *value = pool->opt_prefill_kernel; return PA_OK;
        default: return PA_ERR_INVALID_ARG;
    }
}

int pa_append_kv(pa_pool* pool, const void* k, const void* v, const int64_t* slot_mapping,
                 int num_tokens, void* stream) {
    if (!pool || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !aligned(slot_mapping, 8)) return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_tokens) * pool->kv_heads * 32 > (int64_t{1} << 31) * 256)
        return PA_ERR_UNSUPPORTED;
    DeviceGuard g(pool->device);
    if (!g.ok) return PA_ERR_CUDA;
    return pa_detail::launch_append(pool, k, v, slot_mapping, num_tokens,
                                    static_cast<cudaStream_t>(stream));
}

int pa_copy_blocks(pa_pool* pool, const int64_t* pairs, int num_pairs, void* stream) {
    if (!pool || num_pairs < 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!pairs || !aligned(pairs, 8)) return PA_ERR_INVALID_ARG;
    DeviceGuard g(pool->device);
    if (!g.ok) return PA_ERR_CUDA;
    return pa_detail::launch_copy(pool, pairs, num_pairs, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pa_detail {

int check_decode_args(const pa_pool* pool, const void* q, int S, int Hq, const int32_t* tables,
                      int max_blocks, const int32_t* lens, const void* out, pa_dtype out_dtype) {
    if (!pool || S < 0 || Hq <= 0 || max_blocks < 0) return PA_ERR_INVALID_ARG;
    if (Hq % pool->kv_heads != 0 || Hq / pool->kv_heads > 16) return PA_ERR_UNSUPPORTED;
    if (out_dtype != PA_F32 && out_dtype != PA_BF16) return PA_ERR_DTYPE;
    if (S > 16384) return PA_ERR_UNSUPPORTED;
    if (S == 0) return PA_OK;
    if (!q || !tables || !lens || !out || max_blocks == 0) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16)) return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_blocks) * pool->block_size > (int64_t{1} << 30))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace pa_detail

extern "C" {

int pa_decode_reserve(pa_pool* pool, int max_seqs, int max_q_heads) {
    if (!pool || max_seqs <= 0 || max_q_heads <= 0 || max_q_heads % pool->kv_heads)
        return PA_ERR_INVALID_ARG;
    DeviceGuard g(pool->device);
    if (!g.ok) return PA_ERR_CUDA;
    pa_detail::DecodePlan plan;
    // the fp32 path's partial count grows with the table width; reserve for the fast path
    int rc = pa_detail::plan_decode(pool, max_seqs, max_q_heads, 1, &plan);
    if (rc != PA_OK) return rc;
    return ensure_workspace(pool, workspace_bytes(plan, max_seqs, max_q_heads / pool->kv_heads,
                                                  pool->head_dim, nullptr));
}

// Host plan of the shared-prefix items (see pa_decode_shared).
struct SharedPlan {
    bool tc = false;            // shared items on the tcgen05 kernel (128-row tiles)
    int num_groups = 0;
    int K = 0;                  // items before expanding over KV heads
    int slots = 0;              // shared-partial slots (members x chunks)
    int chunk_tokens = 0, members_per_tile = 0;
    std::vector<int> desc;      // packed device descriptor
    size_t off_items, off_sgroup, off_smember, off_sstart, off_goff, off_gmem, off_gnc, off_gbase, off_gtok;
};

// Fused append: the new token of each sequence (k, v [S][Hkv][D], slots [S]).
struct NewTokens {
    const void* k;
    const void* v;
    const int64_t* slots;
};

static int decode_impl(pa_pool* pool, const void* q, int num_seqs, int num_q_heads,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, float scale, void* out, pa_dtype out_dtype,
                       void* stream, const SharedPlan* sh, const NewTokens* nt = nullptr) {
    int rc = pa_detail::check_decode_args(pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                               context_lens, out, out_dtype);
    if (rc != PA_OK || num_seqs == 0) return rc;
    DeviceGuard g(pool->device);
    if (!g.ok) return PA_ERR_CUDA;
    const int G = num_q_heads / pool->kv_heads;
    pa_detail::DecodePlan plan;
    plan.shared = sh != nullptr;
    plan.fuse = nt != nullptr && sh == nullptr;
    plan.tc = sh != nullptr && sh->tc;
    rc = pa_detail::plan_decode(pool, num_seqs, num_q_heads, max_blocks_per_seq, &plan);
    if (rc != PA_OK) return rc;
    if (sh && !plan.fast) return PA_ERR_UNSUPPORTED;
    if (nt && !(plan.fast && plan.fuse)) {         // no fused form: append first, then decode
        rc = pa_detail::launch_append(pool, nt->k, nt->v, nt->slots, num_seqs,
                                      static_cast<cudaStream_t>(stream));
        if (rc != PA_OK) return rc;
        plan.fuse = false;
    }
    size_t cb = 0;
    size_t need = workspace_bytes(plan, num_seqs, G, pool->head_dim, &cb);
    const size_t sacc_off = need;
    const size_t sacc_bytes = sh ? round256(static_cast<size_t>(sh->slots) * pool->kv_heads * G *
                                            pool->head_dim * sizeof(float)) : 0;
    const size_t sml_bytes = sh ? round256(static_cast<size_t>(sh->slots) * pool->kv_heads * G * 2 *
                                           sizeof(float)) : 0;
    need += sacc_bytes + sml_bytes;
    rc = ensure_workspace(pool, need);
    if (rc != PA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (sh && sh->desc != pool->desc_host) {       // upload only a changed description
        if (sh->desc.size() > pool->desc_cap) {
            if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
            cudaFree(pool->desc_dev);
            pool->desc_dev = nullptr;
            pool->desc_cap = 0;
            if (cudaMalloc(&pool->desc_dev, sh->desc.size() * sizeof(int)) != cudaSuccess) {
                cudaGetLastError();
                return PA_ERR_OUT_OF_MEMORY;
            }
            pool->desc_cap = sh->desc.size();
        }
        // pageable source: the runtime stages it before returning, after prior work on st
        if (cudaMemcpyAsync(pool->desc_dev, sh->desc.data(), sh->desc.size() * sizeof(int),
                            cudaMemcpyHostToDevice, st) != cudaSuccess)
            return PA_ERR_CUDA;
        pool->desc_host = sh->desc;
    }
    DecodeParams p{};
    if (sh) {
        const int* d = pool->desc_dev;
        p.n_shared_items = sh->K * pool->kv_heads;
        p.chunk_tokens = sh->chunk_tokens;
        p.members_per_tile = sh->members_per_tile;
        p.sh_items = d + sh->off_items;
        p.seq_group = d + sh->off_sgroup;
        p.seq_member = d + sh->off_smember;
        p.seq_start = d + sh->off_sstart;
        p.g_members_off = d + sh->off_goff;
        p.g_members = d + sh->off_gmem;
        p.g_nchunks = d + sh->off_gnc;
        p.g_spart_base = d + sh->off_gbase;
        p.g_shared_tokens = d + sh->off_gtok;
        p.spart_acc = reinterpret_cast<float*>(static_cast<char*>(pool->ws) + sacc_off);
        p.spart_ml = reinterpret_cast<float*>(static_cast<char*>(pool->ws) + sacc_off + sacc_bytes);
    }
    p.q = q;
    p.k = pool->k;
    p.v = pool->v;
    p.tables = block_tables;
    p.lens = context_lens;
    p.out = out;
    p.ticket = static_cast<int*>(pool->ws);
    p.sched = p.ticket + 4;
    p.part_acc = reinterpret_cast<float*>(static_cast<char*>(pool->ws) + cb);
    p.part_ml = reinterpret_cast<float*>(
        static_cast<char*>(pool->ws) + cb + round256(plan.max_items * G * pool->head_dim * sizeof(float)));
    p.err = pool->err;
    decode_scales(pool, scale, &p);
    p.S = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = pool->kv_heads;
    p.G = G;
    p.D = pool->head_dim;
    p.B = pool->block_size;
    p.num_blocks = pool->num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.out_bf16 = out_dtype == PA_BF16;
    if (plan.fast && plan.fuse) {
        p.new_k = nt->k;
        p.new_v = nt->v;
        p.new_slots = nt->slots;
    }
    return pa_detail::launch_decode(plan, p, st);
}

int pa_append_decode(pa_pool* pool, const void* k, const void* v, const int64_t* slot_mapping,
                     const void* q, int num_seqs, int num_q_heads, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, float scale, void* out,
                     pa_dtype out_dtype, void* stream) {
    if (num_seqs > 0 && (!k || !v || !slot_mapping || !aligned(slot_mapping, 8) ||
                         !aligned(k, 16) || !aligned(v, 16)))
        return PA_ERR_INVALID_ARG;
    const NewTokens nt{k, v, slot_mapping};
    return decode_impl(pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                       context_lens, scale, out, out_dtype, stream, nullptr, &nt);
}

int pa_decode(pa_pool* pool, const void* q, int num_seqs, int num_q_heads,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              float scale, void* out, pa_dtype out_dtype, void* stream) {
    return decode_impl(pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                       context_lens, scale, out, out_dtype, stream, nullptr);
}

int pa_decode_shared(pa_pool* pool, const void* q, int num_seqs, int num_q_heads,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, float scale, void* out, pa_dtype out_dtype,
                     const int32_t* group_seq_offsets, const int32_t* group_seqs,
                     const int32_t* group_shared_blocks, int num_groups, void* stream) {
    int rc = pa_detail::check_decode_args(pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                               context_lens, out, out_dtype);
    if (rc != PA_OK || num_seqs == 0) return rc;
    if (num_groups < 0 || (num_groups > 0 && (!group_seq_offsets || !group_seqs ||
                                               !group_shared_blocks)))
        return PA_ERR_INVALID_ARG;
    const int Hkv = pool->kv_heads, G = num_q_heads / Hkv, B = pool->block_size;
    const bool tensor_path = (pool->dtype == PA_BF16 || pool->dtype == PA_FP8E4M3) && B % 16 == 0 && G <= 8 &&
                             (pool->head_dim == 64 || pool->head_dim == 128 || pool->head_dim == 256);
    // validate and keep groups of at least two members with a shared span
    std::vector<char> seen(num_seqs, 0);
    std::vector<int> keep;
    if (num_groups > 0 && group_seq_offsets[0] != 0) return PA_ERR_INVALID_ARG;
    for (int gi = 0; gi < num_groups; ++gi) {
        const int a = group_seq_offsets[gi], b = group_seq_offsets[gi + 1];
        if (b < a) return PA_ERR_INVALID_ARG;
        if (group_shared_blocks[gi] < 0 || group_shared_blocks[gi] > max_blocks_per_seq)
            return PA_ERR_INVALID_ARG;
        for (int i = a; i < b; ++i) {
            const int s = group_seqs[i];
            if (s < 0 || s >= num_seqs || seen[s]) return PA_ERR_INVALID_ARG;
            seen[s] = 1;
        }
        if (b - a >= 2 && group_shared_blocks[gi] > 0) keep.push_back(gi);
    }
    if (keep.empty() || !tensor_path)
        return decode_impl(pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                           context_lens, scale, out, out_dtype, stream, nullptr);
    SharedPlan sh;
    sh.num_groups = static_cast<int>(keep.size());
    // tcgen05 items take 128 query rows; the mma.sync variant 64 (the pool's
    // PA_OPT_SHARED_KERNEL option selects it)
    sh.tc = pa_detail::shared_tc_eligible(pool, G) && pool->opt_shared_kernel == 0;
    sh.members_per_tile = std::max(1, (sh.tc ? pa_detail::shared_tc_rows() : 64) / G);
    // shared tokens per item: the tcgen05 kernel stages a 1024-token table slice,
    // the mma.sync variant one block id per lane (32 blocks)
    sh.chunk_tokens = sh.tc ? pa_detail::shared_tc_chunk_tokens() : std::max(B, 512 / B * B);
    const int Ng = sh.num_groups;
    std::vector<int> items, sgroup(num_seqs, -1), smember(num_seqs, 0), sstart(num_seqs, 0);
    std::vector<int> goff(Ng + 1, 0), gmem, gnc(Ng), gbase(Ng), gtok(Ng);
    int slots = 0;
    for (int k = 0; k < Ng; ++k) {
        const int gi = keep[k];
        const int a = group_seq_offsets[gi], b = group_seq_offsets[gi + 1], M = b - a;
        const int tok = group_shared_blocks[gi] * B;
        const int nc = (tok + sh.chunk_tokens - 1) / sh.chunk_tokens;
        const int tiles = (M + sh.members_per_tile - 1) / sh.members_per_tile;
        for (int i = a; i < b; ++i) {
            const int s = group_seqs[i];
            sgroup[s] = k;
            smember[s] = i - a;
            sstart[s] = tok;
            gmem.push_back(s);
        }
        goff[k + 1] = goff[k] + M;
        gnc[k] = nc;
        gbase[k] = slots;
        gtok[k] = tok;
        slots += M * nc;
        for (int c = 0; c < nc; ++c)          // chunk-major: spread a group's tiles over CTAs
            for (int t = 0; t < tiles; ++t) {
                items.push_back(k);
                items.push_back(t);
                items.push_back(c);
                items.push_back(0);
            }
    }
    sh.K = static_cast<int>(items.size() / 4);
    sh.slots = slots;
    auto& d = sh.desc;
    auto put = [&d](const std::vector<int>& v) {
        const size_t off = d.size();
        d.insert(d.end(), v.begin(), v.end());
        while (d.size() % 4) d.push_back(0);        // keep int4 alignment of each section
        return off;
    };
    sh.off_items = put(items);
    sh.off_sgroup = put(sgroup);
    sh.off_smember = put(smember);
    sh.off_sstart = put(sstart);
    sh.off_goff = put(goff);
    sh.off_gmem = put(gmem);
    sh.off_gnc = put(gnc);
    sh.off_gbase = put(gbase);
    sh.off_gtok = put(gtok);
    return decode_impl(pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                       context_lens, scale, out, out_dtype, stream, &sh);
}

int pa_get_error(pa_pool* pool, void* stream) {
    if (!pool) return PA_ERR_INVALID_ARG;
    DeviceGuard g(pool->device);
    if (!g.ok) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, pool->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PA_ERR_CUDA;
    if (code != 0 && cudaMemset(pool->err, 0, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
    return code;
}

const char* pa_error_string(int code) {
    switch (code) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_DTYPE: return "unsupported dtype";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_NO_FREE_BLOCK: return "no free block in the pool";
        case PA_ERR_BAD_BLOCK_ID: return "block id outside the pool";
        case PA_ERR_BAD_SLOT: return "slot outside the pool";
        case PA_ERR_REFCOUNT: return "reference count underflow";
        case PA_ERR_UNKNOWN_REQUEST: return "unknown request";
        case PA_ERR_OUT_OF_MEMORY: return "out of memory";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_OVERLAP: return "copy pairs overlap";
        case PA_ERR_BAD_LENGTH: return "context length beyond the block table";
        default: return "unknown error";
    }
}

uint64_t pa_launch_count(void) {
    return pa_detail::g_launch_counter.load(std::memory_order_relaxed);
}

}  // extern "C"
