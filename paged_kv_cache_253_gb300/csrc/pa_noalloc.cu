// pa_decode_noalloc: the decode entry point for callers that must not allocate
// device memory.
//
// pa_decode keeps its split partials and work counters in a workspace that
// the pool grows with cudaMalloc on demand.  Some callers cannot let a library
// do that: processes whose device memory is already owned by another allocator
// (a framework's caching allocator that has reserved the GPU, or a fixed
// memory budget the application enforces), and serving loops that cannot pay
// for cudaMalloc's implicit device-wide synchronisation.  This variant runs the
// same decode kernel with its scratch in a fixed array that is part of the
// library image itself, so the call never allocates.
//
// The array is a file-scope __device__ object.  Host code cannot use the
// array's name as a device address; the address is looked up once per device
// with cudaGetSymbolAddress (on the first call made on that device, with that
// device current) and cached.  Under lazy module loading (the CUDA default)
// that lookup is also what loads this library's device code onto the device,
// so the array's kScratchBytes are reserved then, on the first call on each
// device, and held until the process exits.  A cudaDeviceReset of the device
// unloads the module: the cached address is then stale and the process must
// not call this entry point on that device again.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t{32} << 20;   // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t round_up256(size_t n) { return (n + 255) / 256 * 256; }

// Device address of this device's copy of g_decode_scratch (looked up once,
// with that device current).
int scratch_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            // loading the module (and the array with it) needs device memory
            return e == cudaErrorMemoryAllocation ? PA_ERR_OUT_OF_MEMORY : PA_ERR_CUDA;
        }
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(pa_pool* pool, const void* q, int num_seqs, int num_q_heads,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, float scale, void* out,
                                 pa_dtype out_dtype, void* stream) {
    // the same argument rules as pa_decode
    const int arc = pa_detail::check_decode_args(pool, q, num_seqs, num_q_heads, block_tables,
                                                 max_blocks_per_seq, context_lens, out, out_dtype);
    if (arc != PA_OK || num_seqs == 0) return arc;

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return PA_ERR_CUDA;
    if (prev != pool->device && cudaSetDevice(pool->device) != cudaSuccess) return PA_ERR_CUDA;
    struct Restore {
        int dev, was;
        ~Restore() { if (dev != was) cudaSetDevice(was); }
    } restore{pool->device, prev};

    const int Hkv = pool->kv_heads, D = pool->head_dim;
    const int G = num_q_heads / Hkv;
    pa_detail::DecodePlan plan;
    int rc = pa_detail::plan_decode(pool, num_seqs, num_q_heads, max_blocks_per_seq, &plan);
    if (rc != PA_OK) return rc;
    const size_t counters = decode_header_bytes(num_seqs);
    // partial slots: as many as the plan asks for, or as fit in the array (the
    // kernel lengthens its partitions to stay within what it is given)
    const size_t per_item = static_cast<size_t>(G) * (D + 2) * sizeof(float);
    const size_t fit = kScratchBytes > counters + 512 ? (kScratchBytes - counters - 512) / per_item : 0;
    if (fit < plan.min_items) return PA_ERR_UNSUPPORTED;                // batch too large
    if (plan.max_items > fit) plan.max_items = fit;
    const size_t acc = round_up256(plan.max_items * G * D * sizeof(float));
    const size_t ml = round_up256(plan.max_items * G * 2 * sizeof(float));
    if (counters + acc + ml > kScratchBytes) return PA_ERR_UNSUPPORTED;

    void* base = nullptr;
    rc = scratch_address(pool->device, &base);
    if (rc != PA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the work tickets must start at zero; the array keeps the previous call's bytes
    if (cudaMemsetAsync(base, 0, counters, st) != cudaSuccess) return PA_ERR_CUDA;

    DecodeParams p{};
    p.q = q;
    p.k = pool->k;
    p.v = pool->v;
    p.tables = block_tables;
    p.lens = context_lens;
    p.out = out;
    p.ticket = static_cast<int*>(base);
    p.sched = p.ticket + 4;
    p.part_acc = reinterpret_cast<float*>(static_cast<char*>(base) + counters);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(base) + counters + acc);
    p.err = pool->err;
    decode_scales(pool, scale, &p);
    p.S = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = Hkv;
    p.G = G;
    p.D = D;
    p.B = pool->block_size;
    p.num_blocks = pool->num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.out_bf16 = out_dtype == PA_BF16;
    return pa_detail::launch_decode(plan, p, st);
}
