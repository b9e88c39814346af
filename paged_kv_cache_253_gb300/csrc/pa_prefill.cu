// Paged prefill attention: the queries of a chunk of new tokens per sequence
// attend, through the sequence's block table, to the cached prefix and to the
// chunk causally up to themselves (kgptalkie "Day 28: PagedAttention / vLLM",
// "Prefix Sharing Is a Natural Extension" and the zenaique prefix-sharing
// answer name the step through what a cache hit saves: the cached span needs
// no prefill).  The chunk's keys and values are appended before the
// call (pa_append_kv), so chunk token i of a sequence with context length L
// after the append sits at position L-n+i and sees keys 0 .. L-n+i.
//
// One CTA per (query tile, KV head, sequence): 4 warps x 16 query rows, a row
// being one (chunk token, query head of the KV head's group) pair, so a tile
// holds 64/G chunk tokens.  The tile's keys [0, last position] are streamed
// as 16-token K / V^T units through an 8-stage cp.async ring in shared memory
// that all four warps read (one HBM/L2 read per unit for 64 rows), with the
// fragment layout of the shared-prefix decode items (token permutation pi,
// 16-byte d chunks): S = Q K^T by mma.sync m16n8k16 (bf16, fp32 accumulate),
// causal and length masks, online softmax per row, O += P V with P as a bf16
// high + low pair.  Each row's normalised output is written directly.
//
// fp8 (e4m3) pools (F8): the units hold codes (one byte per element, half the
// bytes), staged the same way; each thread widens its fragments to f16 pairs
// in registers (exact: every e4m3 value is an f16 value), the queries are
// re-rounded to f16 once (exact for bf16 magnitudes 2^-17 .. 65504), the
// products run as f16 mma.sync with fp32 accumulation and P enters as an f16
// high + low pair; k_scale is folded into the score factor and v_scale
// multiplies the outputs.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

constexpr int kWarpsP = 4;
constexpr int kThreadsP = kWarpsP * 32;
constexpr int kRowsP = kWarpsP * 16;      // query rows per CTA
constexpr int kStagesP = 8;               // staged 16-token units
constexpr int kPerSyncP = 4;              // units consumed per barrier (even: 32-token steps)
static_assert(kStagesP > kPerSyncP && kPerSyncP % 2 == 0, "prefill pipeline shape");

// Eight e4m3 codes widened to four f16 pairs, four to two, and eight bf16
// values re-rounded to f16.
__device__ __forceinline__ uint4 f8_widen8(uint2 c) {
    return make_uint4(pa_dev::e4m3x2_to_f16x2(c.x), pa_dev::e4m3x2_to_f16x2(c.x >> 16),
                      pa_dev::e4m3x2_to_f16x2(c.y), pa_dev::e4m3x2_to_f16x2(c.y >> 16));
}
__device__ __forceinline__ uint2 f8_widen4(uint32_t c) {
    return make_uint2(pa_dev::e4m3x2_to_f16x2(c), pa_dev::e4m3x2_to_f16x2(c >> 16));
}
__device__ __forceinline__ uint32_t bf16x2_f16x2(uint32_t x) {
    return pa_dev::pack_f16(pa_dev::bf16_lo(x), pa_dev::bf16_hi(x));
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreadsP, 2) prefill_kernel(const PrefillParams p) {
    constexpr int NJ = D / 32, ND = D / 8;
    constexpr int ES = F8 ? 1 : 2;                    // bytes per pool element
    constexpr int UNIT = 32 * ES * D;                 // K 16 x D + V^T D x 16
    constexpr int KB = 16 * ES * D;                   // K part of a unit
    constexpr int NCH = ES * D / 16;                  // 16-byte chunks per key row
    constexpr int SWZ = NCH < 8 ? NCH - 1 : 7;        // fp8 key rows: chunk c of row r at c ^ (r & SWZ)
    extern __shared__ __align__(128) unsigned char stage_mem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gi = lane >> 2, c = lane & 3;
    const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const bool reporter = tid == 0 && tile == 0 && h == 0;
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();

    const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
    const int n = q1 - q0;
    const int L = __ldg(p.lens + s);
    if (q0 < 0 || n < 0 || q1 > p.T || L < n) {       // malformed chunk description
        if (reporter) pa_dev::record_error(p.err, PA_ERR_INVALID_ARG);
        return;
    }
    if (L > p.max_blocks * p.B) {                      // context beyond the table
        if (reporter) pa_dev::record_error(p.err, PA_ERR_BAD_LENGTH);
        return;
    }
    const int G = p.G;
    if (n > p.max_q) {                                 // chunk above max_q_len
        if (reporter) pa_dev::record_error(p.err, PA_ERR_INVALID_ARG);
        return;
    }
    const int r_lo = tile * kRowsP;
    if (r_lo >= n * G) return;                         // past this sequence's chunk
    const int P0 = L - n;                              // position of the chunk's first token

    // this thread's two query rows (A: gi, B: gi + 8 of the warp's 16)
    const int rA = r_lo + warp * 16 + gi, rB = rA + 8;
    const int qiA = rA / G, qiB = rB / G;
    const bool okA = qiA < n, okB = qiB < n;
    const int posA = okA ? P0 + qiA : -1, posB = okB ? P0 + qiB : -1;
    const int rows_end = min(n * G, r_lo + kRowsP);
    const int kv_end = P0 + (rows_end - 1) / G + 1;    // keys [0, kv_end) reach some row
    const int nunits = (kv_end + 15) / 16;

    uint4 qa[NJ], qb[NJ];
    {
        const uint16_t* rowA = okA ? p.q + (static_cast<size_t>(q0 + qiA) * p.Hq +
                                            static_cast<size_t>(h) * G + rA % G) * D : nullptr;
        const uint16_t* rowB = okB ? p.q + (static_cast<size_t>(q0 + qiB) * p.Hq +
                                            static_cast<size_t>(h) * G + rB % G) * D : nullptr;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            qa[j] = okA ? __ldg(reinterpret_cast<const uint4*>(rowA + (4 * j + c) * 8)) : make_uint4(0u, 0u, 0u, 0u);
            qb[j] = okB ? __ldg(reinterpret_cast<const uint4*>(rowB + (4 * j + c) * 8)) : make_uint4(0u, 0u, 0u, 0u);
            if constexpr (F8) {
                qa[j] = make_uint4(bf16x2_f16x2(qa[j].x), bf16x2_f16x2(qa[j].y), bf16x2_f16x2(qa[j].z),
                                   bf16x2_f16x2(qa[j].w));
                qb[j] = make_uint4(bf16x2_f16x2(qb[j].x), bf16x2_f16x2(qb[j].y), bf16x2_f16x2(qb[j].z),
                                   bf16x2_f16x2(qb[j].w));
            }
        }
    }
    float o[ND][4];
#pragma unroll
    for (int t = 0; t < ND; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    const float sl = p.scale_log2;
    const int r0 = 4 * (gi >> 1) + (gi & 1), r1 = r0 + 2;      // token rows pi(gi), pi(gi + 8)

    const int B = p.B;
    const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
    const size_t tile_elems = static_cast<size_t>(B) * D;
    const uint32_t stage_s = static_cast<uint32_t>(__cvta_generic_to_shared(stage_mem));
    unsigned valid = 0;                                 // bit (u % stages): unit u staged
    auto issue = [&](int u) {
        const int tok = u * 16, lbk = tok / B, sub = (tok - lbk * B) / 16;
        const int phys = __ldg(table + lbk);
        const int st = u % kStagesP;
        valid &= ~(1u << st);
        if (phys < 0 || phys >= p.num_blocks) {
            if (tid == 0) pa_dev::record_error(p.err, PA_ERR_BAD_BLOCK_ID);
        } else {
            const size_t tl = (static_cast<size_t>(phys) * p.Hkv + h) * tile_elems * ES;
            const char* kg = static_cast<const char*>(p.k) + tl + static_cast<size_t>(sub) * 16 * D * ES;
            const char* vg = static_cast<const char*>(p.v) + tl + sub * 16 * ES;
            const uint32_t ks = stage_s + st * UNIT, vs = ks + KB;
            if constexpr (F8) {
                for (int q = tid; q < 16 * NCH; q += kThreadsP) {    // K: 16 rows x D/16 chunks
                    const int r = q / NCH, ch = q - r * NCH;
                    pa_dev::cp_async16(ks + r * D + ((ch ^ (r & SWZ)) << 4), kg + r * D + ch * 16);
                }
                for (int d = tid; d < D; d += kThreadsP)             // V^T: D rows of 16 codes
                    pa_dev::cp_async16(vs + d * 16, vg + static_cast<size_t>(d) * B);
            } else {
                for (int q = tid; q < 2 * D; q += kThreadsP) {       // K: 16 rows x D/8 chunks
                    const int r = q / (D / 8), ch = q - r * (D / 8);
                    pa_dev::cp_async16(ks + r * (2 * D) + ((ch ^ ((r & 1) << 2)) << 4), kg + r * D * 2 + ch * 16);
                }
                for (int q = tid; q < 2 * D; q += kThreadsP) {       // V^T: D rows x 2 halves
                    const int d = q >> 1, half = q & 1;
                    pa_dev::cp_async16(vs + d * 32 + half * 16, vg + static_cast<size_t>(d) * B * 2 + half * 16);
                }
            }
            valid |= 1u << st;
        }
        pa_dev::cp_async_commit();
    };
    for (int u = 0; u < kStagesP - kPerSyncP; ++u) {
        if (u < nunits) issue(u);
        else pa_dev::cp_async_commit();
    }
    for (int u0 = 0; u0 < nunits; u0 += kPerSyncP) {
#pragma unroll
        for (int k = 0; k < kPerSyncP; ++k) {
            if (u0 + kStagesP - kPerSyncP + k < nunits) issue(u0 + kStagesP - kPerSyncP + k);
            else pa_dev::cp_async_commit();
        }
        pa_dev::cp_async_wait<kStagesP - kPerSyncP>();
        __syncthreads();
        for (int u = u0; u < min(nunits, u0 + kPerSyncP); u += 2) {
            // two 16-token units form one 32-token step: 4 token n-tiles
            const bool v0ok = (valid >> (u % kStagesP)) & 1u;
            const bool v1ok = u + 1 < nunits && ((valid >> ((u + 1) % kStagesP)) & 1u);
            float sA[4][4], sB[4][4];               // [n-tile][frag], even / odd d-chunk chains
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) sA[nt][i] = sB[nt][i] = 0.f;
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                if (!(w == 0 ? v0ok : v1ok)) continue;
                const unsigned char* ks = stage_mem + ((u + w) % kStagesP) * UNIT;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int ch = 4 * j + c;
                    if constexpr (F8) {
                        // 8 codes: half (ch & 1) of 16-byte chunk ch >> 1 of the row
                        const uint4 ka = f8_widen8(*reinterpret_cast<const uint2*>(
                            ks + r0 * D + (((ch >> 1) ^ (r0 & SWZ)) << 4) + (ch & 1) * 8));
                        const uint4 kb = f8_widen8(*reinterpret_cast<const uint2*>(
                            ks + r1 * D + (((ch >> 1) ^ (r1 & SWZ)) << 4) + (ch & 1) * 8));
                        pa_dev::mma_f16_16816(sA[2 * w], qa[j].x, qb[j].x, qa[j].y, qb[j].y, ka.x, ka.y);
                        pa_dev::mma_f16_16816(sB[2 * w], qa[j].z, qb[j].z, qa[j].w, qb[j].w, ka.z, ka.w);
                        pa_dev::mma_f16_16816(sA[2 * w + 1], qa[j].x, qb[j].x, qa[j].y, qb[j].y, kb.x, kb.y);
                        pa_dev::mma_f16_16816(sB[2 * w + 1], qa[j].z, qb[j].z, qa[j].w, qb[j].w, kb.z, kb.w);
                    } else {
                        const uint4 ka = *reinterpret_cast<const uint4*>(ks + r0 * (2 * D) + ((ch ^ ((r0 & 1) << 2)) << 4));
                        const uint4 kb = *reinterpret_cast<const uint4*>(ks + r1 * (2 * D) + ((ch ^ ((r1 & 1) << 2)) << 4));
                        pa_dev::mma_bf16_16816(sA[2 * w], qa[j].x, qb[j].x, qa[j].y, qb[j].y, ka.x, ka.y);
                        pa_dev::mma_bf16_16816(sB[2 * w], qa[j].z, qb[j].z, qa[j].w, qb[j].w, ka.z, ka.w);
                        pa_dev::mma_bf16_16816(sA[2 * w + 1], qa[j].x, qb[j].x, qa[j].y, qb[j].y, kb.x, kb.y);
                        pa_dev::mma_bf16_16816(sB[2 * w + 1], qa[j].z, qb[j].z, qa[j].w, qb[j].w, kb.z, kb.w);
                    }
                }
            }
            // score (row, n-tile nt, column e) is the key at position
            // 16 (u + nt/2) + 4c + 2 (nt % 2) + e; a row sees keys up to its own position
            float xa[8], xb[8];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const bool ok = (nt < 2) ? v0ok : v1ok;
                const int kp = 16 * (u + (nt >> 1)) + 4 * c + 2 * (nt & 1);
                xa[2 * nt] = ok && kp <= posA ? (sA[nt][0] + sB[nt][0]) * sl : -INFINITY;
                xa[2 * nt + 1] = ok && kp + 1 <= posA ? (sA[nt][1] + sB[nt][1]) * sl : -INFINITY;
                xb[2 * nt] = ok && kp <= posB ? (sA[nt][2] + sB[nt][2]) * sl : -INFINITY;
                xb[2 * nt + 1] = ok && kp + 1 <= posB ? (sA[nt][3] + sB[nt][3]) * sl : -INFINITY;
            }
            float mxa = xa[0], mxb = xb[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                mxa = fmaxf(mxa, xa[i]);
                mxb = fmaxf(mxb, xb[i]);
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
                mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
            }
            const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
            const float sa = na == -INFINITY ? 0.f : na, sb = nb == -INFINITY ? 0.f : nb;
            const float cra = pa_dev::ex2(ma - sa), crb = pa_dev::ex2(mb - sb);
            float pa[8], pb[8], suma = 0.f, sumb = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pa[i] = pa_dev::ex2(xa[i] - sa);
                pb[i] = pa_dev::ex2(xb[i] - sb);
                suma += pa[i];
                sumb += pb[i];
            }
            la = la * cra + suma;
            lb = lb * crb + sumb;
            ma = na;
            mb = nb;
            // A fragments of P for the two 16-token k-steps (high and low parts:
            // bf16, or f16 for an fp8 pool's f16 products)
            uint32_t ah[2][4], al[2][4];
            if constexpr (F8) {
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int n0 = 2 * w, n1 = 2 * w + 1;
                    ah[w][0] = pa_dev::pack_f16(pa[2 * n0], pa[2 * n0 + 1]);
                    ah[w][1] = pa_dev::pack_f16(pb[2 * n0], pb[2 * n0 + 1]);
                    ah[w][2] = pa_dev::pack_f16(pa[2 * n1], pa[2 * n1 + 1]);
                    ah[w][3] = pa_dev::pack_f16(pb[2 * n1], pb[2 * n1 + 1]);
                    al[w][0] = pa_dev::pack_f16(pa[2 * n0] - pa_dev::f16_lo(ah[w][0]), pa[2 * n0 + 1] - pa_dev::f16_hi(ah[w][0]));
                    al[w][1] = pa_dev::pack_f16(pb[2 * n0] - pa_dev::f16_lo(ah[w][1]), pb[2 * n0 + 1] - pa_dev::f16_hi(ah[w][1]));
                    al[w][2] = pa_dev::pack_f16(pa[2 * n1] - pa_dev::f16_lo(ah[w][2]), pa[2 * n1 + 1] - pa_dev::f16_hi(ah[w][2]));
                    al[w][3] = pa_dev::pack_f16(pb[2 * n1] - pa_dev::f16_lo(ah[w][3]), pb[2 * n1 + 1] - pa_dev::f16_hi(ah[w][3]));
                }
            } else {
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int n0 = 2 * w, n1 = 2 * w + 1;
                ah[w][0] = pa_dev::pack_bf16(pa[2 * n0], pa[2 * n0 + 1]);
                ah[w][1] = pa_dev::pack_bf16(pb[2 * n0], pb[2 * n0 + 1]);
                ah[w][2] = pa_dev::pack_bf16(pa[2 * n1], pa[2 * n1 + 1]);
                ah[w][3] = pa_dev::pack_bf16(pb[2 * n1], pb[2 * n1 + 1]);
                al[w][0] = pa_dev::pack_bf16(pa[2 * n0] - pa_dev::bf16_lo(ah[w][0]), pa[2 * n0 + 1] - pa_dev::bf16_hi(ah[w][0]));
                al[w][1] = pa_dev::pack_bf16(pb[2 * n0] - pa_dev::bf16_lo(ah[w][1]), pb[2 * n0 + 1] - pa_dev::bf16_hi(ah[w][1]));
                al[w][2] = pa_dev::pack_bf16(pa[2 * n1] - pa_dev::bf16_lo(ah[w][2]), pa[2 * n1 + 1] - pa_dev::bf16_hi(ah[w][2]));
                al[w][3] = pa_dev::pack_bf16(pb[2 * n1] - pa_dev::bf16_lo(ah[w][3]), pb[2 * n1 + 1] - pa_dev::bf16_hi(ah[w][3]));
            }
            }
#pragma unroll
            for (int t = 0; t < ND; ++t) {
                o[t][0] *= cra; o[t][1] *= cra; o[t][2] *= crb; o[t][3] *= crb;
            }
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                if (!(w == 0 ? v0ok : v1ok)) continue;
                const unsigned char* vs = stage_mem + ((u + w) % kStagesP) * UNIT + KB;
                // value columns at or past the context length hold whatever the
                // block held before: zero them so that 0 * (garbage) stays 0
                const int tb = 16 * (u + w) + 4 * c;
                const bool tail = 16 * (u + w) + 16 > L;
                const uint32_t mlo = (tb < L ? 0x0000ffffu : 0u) | (tb + 1 < L ? 0xffff0000u : 0u);
                const uint32_t mhi = (tb + 2 < L ? 0x0000ffffu : 0u) | (tb + 3 < L ? 0xffff0000u : 0u);
#pragma unroll
                for (int t = 0; t < ND; ++t) {
                    uint2 v;
                    if constexpr (F8)                          // 4 codes: tokens 4c .. 4c+3 of row d
                        v = f8_widen4(*reinterpret_cast<const uint32_t*>(vs + (8 * t + gi) * 16 + 4 * c));
                    else
                        v = *reinterpret_cast<const uint2*>(vs + (8 * t + gi) * 32 + 8 * c);
                    if (tail) {
                        v.x &= mlo;
                        v.y &= mhi;
                    }
                    if constexpr (F8) {
                        pa_dev::mma_f16_16816(o[t], ah[w][0], ah[w][1], ah[w][2], ah[w][3], v.x, v.y);
                        pa_dev::mma_f16_16816(o[t], al[w][0], al[w][1], al[w][2], al[w][3], v.x, v.y);
                    } else {
                        pa_dev::mma_bf16_16816(o[t], ah[w][0], ah[w][1], ah[w][2], ah[w][3], v.x, v.y);
                        pa_dev::mma_bf16_16816(o[t], al[w][0], al[w][1], al[w][2], al[w][3], v.x, v.y);
                    }
                }
            }
        }
        __syncthreads();                             // the consumed stages are refilled next
    }
    pa_dev::cp_async_wait<0>();
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    auto write_row = [&](int qi, int hq, int which, float l) {
        const size_t row = (static_cast<size_t>(q0 + qi) * p.Hq + hq) * D;
        const float inv = l > 0.f ? p.v_scale / l : 0.f;
#pragma unroll
        for (int t = 0; t < ND; ++t) {
            const int d = 8 * t + 2 * c;
            const float x0 = o[t][which] * inv, x1 = o[t][which + 1] * inv;
            if (p.out_bf16)
                *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + row + d) = pa_dev::pack_bf16(x0, x1);
            else
                *reinterpret_cast<float2*>(static_cast<float*>(p.out) + row + d) = make_float2(x0, x1);
        }
    };
    if (okA) write_row(qiA, h * G + rA % G, 0, la);
    if (okB) write_row(qiB, h * G + rB % G, 2, lb);
}

template <int D, bool F8>
int launch_prefill_d(const PrefillParams& prm, dim3 grid, cudaStream_t st) {
    const size_t smem = static_cast<size_t>(kStagesP) * (F8 ? 32 : 64) * D;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(prefill_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PA_ERR_CUDA;
    const cudaError_t e = pa_detail::launch_pdl(prefill_kernel<D, F8>, grid, dim3(kThreadsP), smem, st, prm);
    pa_detail::count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" int pa_prefill(pa_pool* pool, const void* q, int num_tokens, int num_q_heads,
                          const int32_t* cu_seqlens_q, int num_seqs, int max_q_len,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, float scale, void* out,
                          pa_dtype out_dtype, void* stream) {
    if (!pool || num_tokens < 0 || num_seqs < 0 || max_q_len < 0 || num_q_heads <= 0 ||
        max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (pool->dtype != PA_BF16 && pool->dtype != PA_FP8E4M3) return PA_ERR_DTYPE;
    if (out_dtype != PA_F32 && out_dtype != PA_BF16) return PA_ERR_DTYPE;
    const int D = pool->head_dim, B = pool->block_size, Hkv = pool->kv_heads;
    if (num_q_heads % Hkv != 0 || B % 16 != 0 || (D != 64 && D != 128 && D != 256) ||
        num_seqs > 65535)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0 || max_q_len == 0) return PA_OK;
    if (!q || !cu_seqlens_q || !block_tables || !context_lens || !out || max_blocks_per_seq == 0)
        return PA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 8 != 0)
        return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_blocks_per_seq) * B > (int64_t{1} << 30)) return PA_ERR_UNSUPPORTED;
    const int G = num_q_heads / Hkv;
    const int64_t tiles = (static_cast<int64_t>(max_q_len) * G + kRowsP - 1) / kRowsP;
    if (tiles > (int64_t{1} << 30)) return PA_ERR_UNSUPPORTED;

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return PA_ERR_CUDA;
    if (prev != pool->device && cudaSetDevice(pool->device) != cudaSuccess) return PA_ERR_CUDA;
    struct Restore {
        int dev, was;
        ~Restore() { if (dev != was) cudaSetDevice(was); }
    } restore{pool->device, prev};

    PrefillParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.k = pool->k;
    p.v = pool->v;
    p.cu_q = cu_seqlens_q;
    p.tables = block_tables;
    p.lens = context_lens;
    p.out = out;
    p.err = pool->err;
    const bool f8 = pool->dtype == PA_FP8E4M3;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 *
                                      (f8 ? static_cast<double>(pool->k_scale) : 1.0));
    p.v_scale = f8 ? pool->v_scale : 1.f;
    p.T = num_tokens;
    p.S = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = Hkv;
    p.G = G;
    p.B = B;
    p.num_blocks = pool->num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.max_q = max_q_len;
    p.out_bf16 = out_dtype == PA_BF16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // tcgen05 form (128 rows per CTA, TMA-staged K/V^T) where the pool's TMA
    // views apply; the pool's PA_OPT_PREFILL_KERNEL option selects the
    // mma.sync form instead
    if (pa_detail::prefill_tc_eligible(pool) && reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
        pool->opt_prefill_kernel == 0) {
        const int rows = pa_detail::prefill_tc_rows();
        const dim3 tgrid(static_cast<unsigned>((static_cast<int64_t>(max_q_len) * G + rows - 1) / rows),
                         static_cast<unsigned>(Hkv), static_cast<unsigned>(num_seqs));
        return pa_detail::launch_prefill_tc(pool, p, tgrid, st);
    }
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(Hkv),
                    static_cast<unsigned>(num_seqs));
    if (f8) {
        if (D == 64) return launch_prefill_d<64, true>(p, grid, st);
        if (D == 128) return launch_prefill_d<128, true>(p, grid, st);
        return launch_prefill_d<256, true>(p, grid, st);
    }
    if (D == 64) return launch_prefill_d<64, false>(p, grid, st);
    if (D == 128) return launch_prefill_d<128, false>(p, grid, st);
    return launch_prefill_d<256, false>(p, grid, st);
}
