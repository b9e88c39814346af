// KV append and copy-on-write block copy kernels.
//
// append: each new token's keys and values go to its (physical block,
// offset) slot (kgptalkie "Day 28: PagedAttention / vLLM", "Follow One Token
// Address", "Growth Needs Only Another Free Block"; zenaique prefix-sharing
// answer: the new token's data goes into its request's slot).
// copy:   copy-on-write duplicates a whole shared block before the diverging
// write (kgptalkie "Shared Blocks Must Not Be Changed in Place"; zenaique
// "Most common mistake": only the divergent block is copied).
//
// Both are pure data movement, elements moved as raw bits, except the append
// into an fp8 pool, which quantizes its bf16 input.
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

// One warp per (token, KV head).  The key row is contiguous in the pool and is
// written with whole-row vector stores; the value row lands in a column of the
// transposed (head_dim x block_size) value tile, one element per dimension.
template <typename E>
__global__ void __launch_bounds__(256) append_kv_kernel(
    E* __restrict__ kpool, E* __restrict__ vpool, const E* __restrict__ k,
    const E* __restrict__ v, const int64_t* __restrict__ slots, int T, int Hkv, int D, int B,
    int64_t num_slots, int* err) {
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();
    const int warp = static_cast<int>((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= T * Hkv) return;
    const int t = warp / Hkv;
    const int h = warp - t * Hkv;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0) pa_dev::record_error(err, PA_ERR_BAD_SLOT);
        return;
    }
    const int64_t blk = slot / B;
    const int off = static_cast<int>(slot - blk * B);
    const int64_t tile = (blk * Hkv + h) * static_cast<int64_t>(B) * D;
    const E* ksrc = k + (static_cast<int64_t>(t) * Hkv + h) * D;
    const E* vsrc = v + (static_cast<int64_t>(t) * Hkv + h) * D;
    E* kdst = kpool + tile + static_cast<int64_t>(off) * D;
    constexpr int kVec = 16 / sizeof(E);
    const bool vec = (D % kVec == 0) &&
                     ((reinterpret_cast<uintptr_t>(ksrc) | reinterpret_cast<uintptr_t>(kdst)) % 16 == 0);
    if (vec) {
        for (int i = lane; i < D / kVec; i += 32)
            reinterpret_cast<uint4*>(kdst)[i] = reinterpret_cast<const uint4*>(ksrc)[i];
    } else {
        for (int d = lane; d < D; d += 32) kdst[d] = ksrc[d];
    }
    E* vdst = vpool + tile + off;
    for (int d = lane; d < D; d += 32) vdst[static_cast<int64_t>(d) * B] = vsrc[d];
}

// fp8 pool: the same walk, with each bf16 input element quantized on the
// way, code = e4m3(fl32(x / scale)) (IEEE division, then the hardware
// conversion: nearest, ties to even, saturating at 448).  Lanes take element
// pairs; the key row is written two codes at a time.
__global__ void __launch_bounds__(256) append_kv_fp8_kernel(
    uint8_t* __restrict__ kpool, uint8_t* __restrict__ vpool, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const int64_t* __restrict__ slots, int T, int Hkv, int D,
    int B, int64_t num_slots, float k_scale, float v_scale, int* err) {
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();
    const int warp = static_cast<int>((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= T * Hkv) return;
    const int t = warp / Hkv;
    const int h = warp - t * Hkv;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0) pa_dev::record_error(err, PA_ERR_BAD_SLOT);
        return;
    }
    const int64_t blk = slot / B;
    const int off = static_cast<int>(slot - blk * B);
    const int64_t tile = (blk * Hkv + h) * static_cast<int64_t>(B) * D;
    const uint16_t* ksrc = k + (static_cast<int64_t>(t) * Hkv + h) * D;
    const uint16_t* vsrc = v + (static_cast<int64_t>(t) * Hkv + h) * D;
    uint8_t* kdst = kpool + tile + static_cast<int64_t>(off) * D;   // even: D % 4 == 0
    uint8_t* vdst = vpool + tile + off;
    auto bf = [](uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); };
    for (int i = lane; i < D / 2; i += 32) {
        const uint32_t kc = pa_dev::e4m3x2_from_f32(__fdiv_rn(bf(ksrc[2 * i]), k_scale),
                                                    __fdiv_rn(bf(ksrc[2 * i + 1]), k_scale));
        reinterpret_cast<uint16_t*>(kdst)[i] = static_cast<uint16_t>(kc);
        const uint32_t vc = pa_dev::e4m3x2_from_f32(__fdiv_rn(bf(vsrc[2 * i]), v_scale),
                                                    __fdiv_rn(bf(vsrc[2 * i + 1]), v_scale));
        vdst[static_cast<int64_t>(2 * i) * B] = static_cast<uint8_t>(vc);
        vdst[static_cast<int64_t>(2 * i + 1) * B] = static_cast<uint8_t>(vc >> 8);
    }
}

// One CTA per (src, dst) pair.  The pair is checked against every other pair
// of the call first; a conflicting or out-of-range pair copies nothing.
__global__ void __launch_bounds__(256) copy_blocks_kernel(
    uint8_t* __restrict__ kpool, uint8_t* __restrict__ vpool, const int64_t* __restrict__ pairs,
    int P, int64_t num_blocks, int64_t block_bytes, int* err) {
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();
    const int i = blockIdx.x;
    const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    const bool range_bad = src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks;
    int conflict = (src == dst);
    for (int j = threadIdx.x; j < P; j += blockDim.x) {
        if (j == i) continue;
        const int64_t s2 = pairs[2 * j], d2 = pairs[2 * j + 1];
        conflict |= (dst == s2) | (dst == d2) | (src == d2);
    }
    conflict = __syncthreads_or(conflict);
    if (range_bad || conflict) {
        if (threadIdx.x == 0)
            pa_dev::record_error(err, range_bad ? PA_ERR_BAD_BLOCK_ID : PA_ERR_OVERLAP);
        return;
    }
    for (int which = 0; which < 2; ++which) {
        uint8_t* base = which == 0 ? kpool : vpool;
        const uint8_t* s = base + src * block_bytes;
        uint8_t* d = base + dst * block_bytes;
        if (block_bytes % 16 == 0) {
            const int64_t n = block_bytes / 16;
            for (int64_t e = threadIdx.x; e < n; e += blockDim.x)
                reinterpret_cast<uint4*>(d)[e] = reinterpret_cast<const uint4*>(s)[e];
        } else {
            const int64_t n = block_bytes / 4;      // head_dim % 4 == 0: whole words
            for (int64_t e = threadIdx.x; e < n; e += blockDim.x)
                reinterpret_cast<uint32_t*>(d)[e] = reinterpret_cast<const uint32_t*>(s)[e];
        }
    }
}

}  // namespace

namespace pa_detail {

int launch_append(const pa_pool* p, const void* k, const void* v, const int64_t* slots, int T,
                  cudaStream_t st) {
    const int64_t warps = static_cast<int64_t>(T) * p->kv_heads;
    const int threads = 256;
    const int64_t grid = (warps * 32 + threads - 1) / threads;
    const int64_t num_slots = static_cast<int64_t>(p->num_blocks) * p->block_size;
    cudaError_t e;
    if (p->dtype == PA_FP8E4M3)
        e = launch_pdl(append_kv_fp8_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0,
                       st, static_cast<uint8_t*>(p->k), static_cast<uint8_t*>(p->v),
                       static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), slots, T,
                       p->kv_heads, p->head_dim, p->block_size, num_slots, p->k_scale, p->v_scale,
                       p->err);
    else if (p->dtype == PA_BF16)
        e = launch_pdl(append_kv_kernel<uint16_t>, dim3(static_cast<unsigned>(grid)), dim3(threads),
                       0, st, static_cast<uint16_t*>(p->k), static_cast<uint16_t*>(p->v),
                       static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), slots, T,
                       p->kv_heads, p->head_dim, p->block_size, num_slots, p->err);
    else
        e = launch_pdl(append_kv_kernel<uint32_t>, dim3(static_cast<unsigned>(grid)), dim3(threads),
                       0, st, static_cast<uint32_t*>(p->k), static_cast<uint32_t*>(p->v),
                       static_cast<const uint32_t*>(k), static_cast<const uint32_t*>(v), slots, T,
                       p->kv_heads, p->head_dim, p->block_size, num_slots, p->err);
    count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_copy(const pa_pool* p, const int64_t* pairs, int P, cudaStream_t st) {
    const int64_t esz = static_cast<int64_t>(pool_elem_size(p->dtype));
    const int64_t block_bytes =
        static_cast<int64_t>(p->kv_heads) * p->block_size * p->head_dim * esz;
    const cudaError_t e = launch_pdl(copy_blocks_kernel, dim3(P), dim3(256), 0, st,
                                     static_cast<uint8_t*>(p->k), static_cast<uint8_t*>(p->v),
                                     pairs, P, static_cast<int64_t>(p->num_blocks), block_bytes,
                                     p->err);
    count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
