// Paged decode attention.
//
// What it computes (kgptalkie "Day 28: PagedAttention / vLLM": "The Block
// Table Is the Map", "Follow One Token Address", "Batching Becomes More
// Flexible"): for each sequence s and query head h, the query scores every
// cached key of s, found through s's block table in logical order, and mixes
// the matching values by the softmax of the scores.  Query head h reads KV
// head h / G (G = Hq / Hkv).
//
// How (designed for sm_103a; the pages give no kernel):
//   * Work item = (sequence, KV head, partition of PT tokens).  PT is chosen
//     on the device from the batch's total length so that the items number a
//     few per CTA; long contexts are split over block ranges and merged by
//     log-sum-exp.  The grid is persistent (a few CTAs per SM); every CTA
//     builds the same item list from context_lens in shared memory.
//   * Each item is served by the CTA's 4 warps, which take the partition's
//     blocks round-robin and keep their own online-softmax state; the warps
//     are merged in shared memory at the end of the item.
//   * bf16 pools: a 16-token block tile of one KV head is one tensor-core
//     M tile.  Scores S^T[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8] and
//     O^T[D x 8] += V^T[D x 16] . P^T[16 x 8] with mma.sync m16n8k16 (bf16 in,
//     fp32 accumulate): every key/value byte is loaded once for all G <= 8
//     query heads of its group.  Operand fragments are loaded straight from
//     HBM into registers with 16-byte (K) and 8-byte (V) streaming loads; the
//     token order inside a tile is permuted so these loads are contiguous.
//     P^T reaches the B-operand layout through movmatrix; P is split into a
//     bf16 high part and a bf16 low part so the value product keeps ~16 bits
//     of the fp32 probabilities.
//   * f32 pools (and bf16 shapes outside the tensor-core tile) use a plain
//     fp32 CUDA-core item: scores to shared memory, softmax, value mix.
//   * An item whose sequence has one partition writes the normalised output.
//     Otherwise it writes (acc, max, sum) to the workspace; the CTA that
//     completes a (sequence, head)'s last partition (arrival counter, no
//     waiting) merges them and resets the counter.
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

using pa_dev::record_error;

// ------------------------------------------------------------- schedule ---

__device__ __forceinline__ int seq_len(const DecodeParams& p, int s, bool report) {
    int L = __ldg(p.lens + s);
    const int cap = p.max_blocks * p.B;
    if (L < 0 || L > cap) {
        if (report) record_error(p.err, PA_ERR_BAD_LENGTH);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

struct Sched {
    int PT;
    int total_items;
};

// Every CTA derives the same item list: per sequence nP = max(1, ceil(L/PT))
// partitions, each of Hkv items; s_start[s] = first item of sequence s.
__device__ Sched build_schedule(const DecodeParams& p, int* s_start, long long* s_red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.S + kThreads - 1) / kThreads;
    const int lo = min(p.S, tid * per), hi = min(p.S, lo + per);
    const bool report = blockIdx.x == 0;
    long long tok = 0;
    for (int s = lo; s < hi; ++s) tok += seq_len(p, s, report);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tok += __shfl_xor_sync(0xffffffffu, tok, o);
    if (lane == 0) s_red[warp] = tok;
    __syncthreads();
    long long total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) total += s_red[w];
    int PT;
    if (p.pt_fixed > 0) {
        PT = p.pt_fixed;
    } else {
        long long need = (total * p.Hkv + p.items_target - 1) / p.items_target;
        need = (need + p.B - 1) / p.B * p.B;
        PT = static_cast<int>(max(need, static_cast<long long>(p.pt_min)));
    }
    int cnt = 0;
    for (int s = lo; s < hi; ++s) {
        const int L = seq_len(p, s, false);
        cnt += max(1, (L + PT - 1) / PT) * p.Hkv;
    }
    int inc = cnt;                                  // inclusive scan over the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();                                // s_red reuse
    if (lane == 31) s_red[warp] = inc;
    __syncthreads();
    int base = inc - cnt;
    for (int w = 0; w < warp; ++w) base += static_cast<int>(s_red[w]);
    int total_items = 0;
    for (int w = 0; w < kWarps; ++w) total_items += static_cast<int>(s_red[w]);
    for (int s = lo; s < hi; ++s) {
        s_start[s] = base;
        base += max(1, (seq_len(p, s, false) + PT - 1) / PT) * p.Hkv;
    }
    if (tid == 0) s_start[p.S] = total_items;
    __syncthreads();
    return Sched{PT, total_items};
}

__device__ __forceinline__ int find_seq(const int* s_start, int S, int item) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= item) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// --------------------------------------------------------- item results ---

__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float x) {
    if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float*>(p.out)[idx] = x;
}

// res_m/res_l: [G] (log2-domain running max, sum); res_acc: [G][stride].
__device__ void finish_item(const DecodeParams& p, int item, int s, int h, int nP,
                            int seq_item0, const float* res_m, const float* res_l,
                            const float* res_acc, int stride, int* s_flag) {
    const int tid = threadIdx.x;
    const int GD = p.G * p.D;
    const size_t out0 = (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G) * p.D;
    if (nP == 1) {
        for (int idx = tid; idx < GD; idx += kThreads) {
            const int n = idx / p.D, d = idx - n * p.D;
            const float l = res_l[n];
            store_out(p, out0 + idx, l > 0.f ? res_acc[n * stride + d] / l : 0.f);
        }
        return;
    }
    float* pacc = p.part_acc + static_cast<size_t>(item) * GD;
    for (int idx = tid; idx < GD; idx += kThreads) {
        const int n = idx / p.D, d = idx - n * p.D;
        pacc[idx] = res_acc[n * stride + d];
    }
    if (tid < p.G) {
        p.part_ml[(static_cast<size_t>(item) * p.G + tid) * 2 + 0] = res_m[tid];
        p.part_ml[(static_cast<size_t>(item) * p.G + tid) * 2 + 1] = res_l[tid];
    }
    __threadfence();
    __syncthreads();
    int* counter = p.counters + static_cast<size_t>(s) * p.Hkv + h;
    if (tid == 0) *s_flag = (atomicAdd(counter, 1) == nP - 1);
    __syncthreads();
    if (!*s_flag) return;
    __threadfence();
    for (int idx = tid; idx < GD; idx += kThreads) {
        const int n = idx / p.D;
        float M = -INFINITY;
        for (int q = 0; q < nP; ++q) {
            const size_t it = static_cast<size_t>(seq_item0) + static_cast<size_t>(q) * p.Hkv + h;
            M = fmaxf(M, __ldcg(p.part_ml + (it * p.G + n) * 2));
        }
        float acc = 0.f, l = 0.f;
        if (M != -INFINITY) {
            for (int q = 0; q < nP; ++q) {
                const size_t it = static_cast<size_t>(seq_item0) + static_cast<size_t>(q) * p.Hkv + h;
                const float mq = __ldcg(p.part_ml + (it * p.G + n) * 2);
                const float f = pa_dev::ex2(mq - M);
                l += f * __ldcg(p.part_ml + (it * p.G + n) * 2 + 1);
                acc += f * __ldcg(p.part_acc + it * GD + idx);
            }
        }
        store_out(p, out0 + idx, l > 0.f ? acc / l : 0.f);
    }
    if (tid == 0) *counter = 0;
}

// ------------------------------------------------ bf16 tensor-core item ---
//
// Lane layout of one warp (g = lane / 4, c = lane % 4), per 16-token tile:
//   A rows of the score product are tokens; row r holds token pi(r) with
//   pi(2c'+e) = 4c'+e and pi(8+2c'+e) = 4c'+2+e (e in {0,1}), so the two
//   tokens thread c needs for a P^T fragment are the 4 adjacent tokens
//   4c..4c+3 of the transposed value tile (one 8-byte load per value row).
//   The contraction index d is split in 16-byte chunks: thread c owns chunks
//   c, c+4, ... of each row; chunk elements 0-1 / 2-3 feed the low / high k
//   half of one k-step and elements 4-7 the next k-step, identically for K
//   and Q, so every product q[d]*k[d] is formed exactly once.
template <int D>
__device__ __forceinline__ void fast_item(const DecodeParams& p, int s, int h, int tok0,
                                          int tok1, int L, float* sm_o, float* sm_m,
                                          float* sm_l) {
    constexpr int NJ = D / 32;        // 16-byte chunks per thread per row
    constexpr int NT = D / 16;        // m-tiles of the value product
    constexpr int OS = D + 4;         // padded row stride of the merge buffer
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int B = p.B;

    uint4 qf[NJ];
    {
        const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                               (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G + g) * D;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            qf[j] = g < p.G ? __ldg(reinterpret_cast<const uint4*>(qrow + (4 * j + c) * 8))
                            : make_uint4(0u, 0u, 0u, 0u);
    }
    float o[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl = p.scale_log2;
    const int r0 = 4 * (g >> 1) + (g & 1), r1 = r0 + 2;
    const int lb0 = tok0 / B, lb1 = (tok1 + B - 1) / B;
    const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
    const uint16_t* kpool = static_cast<const uint16_t*>(p.k);
    const uint16_t* vpool = static_cast<const uint16_t*>(p.v);

    for (int lb = lb0 + warp; lb < lb1; lb += kWarps) {
        const int phys = __ldg(table + lb);
        if (phys < 0 || phys >= p.num_blocks) {
            if (lane == 0) record_error(p.err, PA_ERR_BAD_BLOCK_ID);
            continue;
        }
        const size_t tile = (static_cast<size_t>(phys) * p.Hkv + h) * static_cast<size_t>(B) * D;
        for (int sub = 0; sub * 16 < B; ++sub) {
            const int nvalid = min(16, L - (lb * B + sub * 16));
            if (nvalid <= 0) break;
            const uint16_t* kt = kpool + tile + static_cast<size_t>(sub) * 16 * D;
            const uint16_t* vt = vpool + tile + sub * 16 + 4 * c;
            uint4 k0[NJ], k1[NJ];
            uint2 v0[NT], v1[NT];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                k0[j] = pa_dev::ld_stream16(kt + r0 * D + (4 * j + c) * 8);
                k1[j] = pa_dev::ld_stream16(kt + r1 * D + (4 * j + c) * 8);
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                v0[t] = pa_dev::ld_stream8(vt + static_cast<size_t>(16 * t + g) * B);
                v1[t] = pa_dev::ld_stream8(vt + static_cast<size_t>(16 * t + g + 8) * B);
            }
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                pa_dev::mma_bf16_16816(sc, k0[j].x, k1[j].x, k0[j].y, k1[j].y, qf[j].x, qf[j].y);
                pa_dev::mma_bf16_16816(sc, k0[j].z, k1[j].z, k0[j].w, k1[j].w, qf[j].z, qf[j].w);
            }
            float x0 = sc[0] * sl, x1 = sc[1] * sl, x2 = sc[2] * sl, x3 = sc[3] * sl;
            if (nvalid < 16) {                        // partly filled last tile
                if (r0 >= nvalid) x0 = x1 = -INFINITY;
                if (r1 >= nvalid) x2 = x3 = -INFINITY;
                const uint32_t mlo = (4 * c < nvalid ? 0x0000ffffu : 0u) |
                                     (4 * c + 1 < nvalid ? 0xffff0000u : 0u);
                const uint32_t mhi = (4 * c + 2 < nvalid ? 0x0000ffffu : 0u) |
                                     (4 * c + 3 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    v0[t].x &= mlo; v0[t].y &= mhi;
                    v1[t].x &= mlo; v1[t].y &= mhi;
                }
            }
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
            const float cr0 = pa_dev::ex2(m0 - ms0), cr1 = pa_dev::ex2(m1 - ms1);
            const float p0 = pa_dev::ex2(x0 - ms0), p1 = pa_dev::ex2(x1 - ms1);
            const float p2 = pa_dev::ex2(x2 - ms0), p3 = pa_dev::ex2(x3 - ms1);
            l0 = l0 * cr0 + (p0 + p2);
            l1 = l1 * cr1 + (p1 + p3);
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                o[t][0] *= cr0; o[t][1] *= cr1;
                o[t][2] *= cr0; o[t][3] *= cr1;
            }
            const uint32_t h01 = pa_dev::pack_bf16(p0, p1), h23 = pa_dev::pack_bf16(p2, p3);
            const uint32_t e01 = pa_dev::pack_bf16(p0 - pa_dev::bf16_lo(h01), p1 - pa_dev::bf16_hi(h01));
            const uint32_t e23 = pa_dev::pack_bf16(p2 - pa_dev::bf16_lo(h23), p3 - pa_dev::bf16_hi(h23));
            const uint32_t bh0 = pa_dev::movmatrix_trans(h01), bh1 = pa_dev::movmatrix_trans(h23);
            const uint32_t be0 = pa_dev::movmatrix_trans(e01), be1 = pa_dev::movmatrix_trans(e23);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                pa_dev::mma_bf16_16816(o[t], v0[t].x, v1[t].x, v0[t].y, v1[t].y, bh0, bh1);
                pa_dev::mma_bf16_16816(o[t], v0[t].x, v1[t].x, v0[t].y, v1[t].y, be0, be1);
            }
        }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* mo = sm_o + warp * 8 * OS;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        mo[(2 * c) * OS + 16 * t + g] = o[t][0];
        mo[(2 * c + 1) * OS + 16 * t + g] = o[t][1];
        mo[(2 * c) * OS + 16 * t + g + 8] = o[t][2];
        mo[(2 * c + 1) * OS + 16 * t + g + 8] = o[t][3];
    }
    if (g == 0) {
        sm_m[warp * 8 + 2 * c] = m0;
        sm_m[warp * 8 + 2 * c + 1] = m1;
        sm_l[warp * 8 + 2 * c] = l0;
        sm_l[warp * 8 + 2 * c + 1] = l1;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 3) decode_fast_kernel(const DecodeParams p) {
    constexpr int OS = D + 4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* sm_o = reinterpret_cast<float*>(smem_raw);        // [kWarps][8][OS]
    float* sm_m = sm_o + kWarps * 8 * OS;                     // [kWarps][8]
    float* sm_l = sm_m + kWarps * 8;                          // [kWarps][8]
    float* res_m = sm_l + kWarps * 8;                         // [8]
    float* res_l = res_m + 8;                                 // [8]
    long long* s_red = reinterpret_cast<long long*>(res_l + 8);   // [kWarps]
    int* s_flag = reinterpret_cast<int*>(s_red + kWarps);
    int* s_start = s_flag + 4;                                // [S + 1]

    const Sched sc = build_schedule(p, s_start, s_red);
    for (int item = blockIdx.x; item < sc.total_items; item += gridDim.x) {
        const int s = find_seq(s_start, p.S, item);
        const int local = item - s_start[s];
        const int part = local / p.Hkv, h = local - part * p.Hkv;
        const int L = seq_len(p, s, false);
        const int nP = max(1, (L + sc.PT - 1) / sc.PT);
        const int tok0 = part * sc.PT, tok1 = min(L, tok0 + sc.PT);
        fast_item<D>(p, s, h, tok0, tok1, L, sm_o, sm_m, sm_l);
        __syncthreads();
        // merge the warps' softmax states (in place into warp 0's buffer)
        for (int idx = threadIdx.x; idx < p.G * D; idx += kThreads) {
            const int n = idx / D, d = idx - n * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 8 + n]);
            float acc = 0.f, l = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float f = pa_dev::ex2(sm_m[w * 8 + n] - M);
                    acc += f * sm_o[(w * 8 + n) * OS + d];
                    l += f * sm_l[w * 8 + n];
                }
            }
            sm_o[n * OS + d] = acc;
            if (d == 0) {
                res_m[n] = M;
                res_l[n] = l;
            }
        }
        __syncthreads();
        finish_item(p, item, s, h, nP, s_start[s], res_m, res_l, sm_o, OS, s_flag);
        __syncthreads();
    }
}

// ------------------------------------------------ fp32 CUDA-core item ---

template <typename E>
__device__ __forceinline__ float load_elem(const E* base, size_t i);
template <>
__device__ __forceinline__ float load_elem<float>(const float* base, size_t i) {
    return __ldg(base + i);
}
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t* base, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(base + i)) << 16);
}

// Items of at most pt_fixed tokens.  Shared memory: q [G][D], scores/probs
// [G][PT], result [G][D+4].
template <typename E>
__global__ void __launch_bounds__(kThreads) decode_simple_kernel(const DecodeParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int PTm = p.pt_fixed;
    const int OS = p.D + 4;
    float* qs = reinterpret_cast<float*>(smem_raw);           // [G][D]
    float* sc = qs + p.G * p.D;                               // [G][PTm]
    float* res = sc + p.G * PTm;                              // [G][OS]
    float* res_m = res + p.G * OS;                            // [16]
    float* res_l = res_m + 16;                                // [16]
    const int used = p.G * p.D + p.G * PTm + p.G * OS + 32;   // floats so far
    long long* s_red = reinterpret_cast<long long*>(qs + (used + 3) / 4 * 4);
    int* s_flag = reinterpret_cast<int*>(s_red + kWarps);
    int* s_start = s_flag + 4;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const E* q = static_cast<const E*>(p.q);
    const E* kp = static_cast<const E*>(p.k);
    const E* vp = static_cast<const E*>(p.v);
    const Sched sched = build_schedule(p, s_start, s_red);
    for (int item = blockIdx.x; item < sched.total_items; item += gridDim.x) {
        const int s = find_seq(s_start, p.S, item);
        const int local = item - s_start[s];
        const int part = local / p.Hkv, h = local - part * p.Hkv;
        const int L = seq_len(p, s, false);
        const int nP = max(1, (L + sched.PT - 1) / sched.PT);
        const int tok0 = part * sched.PT, nt = max(0, min(L, tok0 + sched.PT) - tok0);
        const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
        for (int i = tid; i < p.G * p.D; i += kThreads)
            qs[i] = load_elem<E>(q, (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G) * p.D + i);
        __syncthreads();
        for (int i = tid; i < p.G * nt; i += kThreads) {
            const int n = i / nt, j = i - n * nt;
            const int tok = tok0 + j, lb = tok / p.B, off = tok - lb * p.B;
            const int phys = __ldg(table + lb);
            float x = -INFINITY;
            if (phys >= 0 && phys < p.num_blocks) {
                const size_t row = ((static_cast<size_t>(phys) * p.Hkv + h) * p.B + off) * p.D;
                float dot = 0.f;
                for (int d = 0; d < p.D; ++d) dot = fmaf(qs[n * p.D + d], load_elem<E>(kp, row + d), dot);
                x = dot * p.scale_log2;
            } else if (n == 0) {
                record_error(p.err, PA_ERR_BAD_BLOCK_ID);
            }
            sc[n * PTm + j] = x;
        }
        __syncthreads();
        for (int n = warp; n < p.G; n += kWarps) {
            float m = -INFINITY;
            for (int j = lane; j < nt; j += 32) m = fmaxf(m, sc[n * PTm + j]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float ms = m == -INFINITY ? 0.f : m;
            float l = 0.f;
            for (int j = lane; j < nt; j += 32) {
                const float e = pa_dev::ex2(sc[n * PTm + j] - ms);
                sc[n * PTm + j] = e;
                l += e;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane == 0) {
                res_m[n] = m;
                res_l[n] = l;
            }
        }
        __syncthreads();
        for (int i = tid; i < p.G * p.D; i += kThreads) {
            const int n = i / p.D, d = i - n * p.D;
            float acc = 0.f;
            for (int j = 0; j < nt; ++j) {
                const int tok = tok0 + j, lb = tok / p.B, off = tok - lb * p.B;
                const int phys = __ldg(table + lb);
                if (phys < 0 || phys >= p.num_blocks) continue;
                const size_t vt = (static_cast<size_t>(phys) * p.Hkv + h) * p.B * static_cast<size_t>(p.D);
                acc = fmaf(sc[n * PTm + j], load_elem<E>(vp, vt + static_cast<size_t>(d) * p.B + off), acc);
            }
            res[n * OS + d] = acc;
        }
        __syncthreads();
        finish_item(p, item, s, h, nP, s_start[s], res_m, res_l, res, OS, s_flag);
        __syncthreads();
    }
}

size_t fast_smem(int D, int S) {
    return static_cast<size_t>(kWarps * 8 * (D + 4) + kWarps * 16 + 16) * sizeof(float) +
           kWarps * sizeof(long long) + 4 * sizeof(int) + static_cast<size_t>(S + 1) * sizeof(int);
}

size_t simple_smem(int G, int D, int PT, int S) {
    return static_cast<size_t>((G * D + G * PT + G * (D + 4) + 32 + 3) / 4 * 4) * sizeof(float) +
           kWarps * sizeof(long long) + 4 * sizeof(int) + static_cast<size_t>(S + 1) * sizeof(int);
}

template <typename K>
int occupancy(K kernel, size_t smem) {
    int n = 0;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, smem) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

namespace pa_detail {

int plan_decode(const pa_pool* pool, int S, int Hq, int max_blocks, DecodePlan* plan) {
    const int Hkv = pool->kv_heads, D = pool->head_dim, B = pool->block_size;
    const int G = Hq / Hkv;
    const bool fast = pool->dtype == PA_BF16 && (D == 64 || D == 128 || D == 256) &&
                      B % 16 == 0 && G <= 8;
    plan->fast = fast;
    plan->bf16 = pool->dtype == PA_BF16;
    plan->threads = kThreads;
    int occ = 0;
    if (fast) {
        plan->smem = fast_smem(D, S);
        plan->pt_fixed = 0;
        plan->pt_min = std::max(B, (64 + B - 1) / B * B);
        if (D == 64) occ = occupancy(decode_fast_kernel<64>, plan->smem);
        else if (D == 128) occ = occupancy(decode_fast_kernel<128>, plan->smem);
        else occ = occupancy(decode_fast_kernel<256>, plan->smem);
    } else {
        const int PT = B >= 256 ? B : (256 / B) * B;
        plan->pt_fixed = PT;
        plan->pt_min = PT;
        plan->smem = simple_smem(G, D, PT, S);
        occ = pool->dtype == PA_BF16 ? occupancy(decode_simple_kernel<uint16_t>, plan->smem)
                                     : occupancy(decode_simple_kernel<float>, plan->smem);
    }
    if (occ <= 0) return PA_ERR_UNSUPPORTED;
    plan->grid = pool->num_sms * occ;
    if (fast) {
        plan->items_target = plan->grid * 4;
        plan->max_items = static_cast<size_t>(plan->items_target) + static_cast<size_t>(Hkv) * S;
    } else {
        plan->items_target = 0;
        const size_t per_seq = (static_cast<size_t>(max_blocks) * B + plan->pt_fixed - 1) / plan->pt_fixed;
        plan->max_items = static_cast<size_t>(Hkv) * S * std::max<size_t>(1, per_seq);
    }
    if (static_cast<size_t>(plan->grid) > plan->max_items)
        plan->grid = static_cast<int>(plan->max_items);
    return PA_OK;
}

int launch_decode(const DecodePlan& plan, const DecodeParams& prm, cudaStream_t st) {
    DecodeParams p = prm;
    p.items_target = plan.items_target;
    p.pt_min = plan.pt_min;
    p.pt_fixed = plan.pt_fixed;
    if (plan.fast) {
        if (p.D == 64) decode_fast_kernel<64><<<plan.grid, plan.threads, plan.smem, st>>>(p);
        else if (p.D == 128) decode_fast_kernel<128><<<plan.grid, plan.threads, plan.smem, st>>>(p);
        else decode_fast_kernel<256><<<plan.grid, plan.threads, plan.smem, st>>>(p);
    } else if (plan.bf16) {
        decode_simple_kernel<uint16_t><<<plan.grid, plan.threads, plan.smem, st>>>(p);
    } else {
        decode_simple_kernel<float><<<plan.grid, plan.threads, plan.smem, st>>>(p);
    }
    count_launch();
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
