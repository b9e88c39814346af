// Paged decode attention, stream-K split pass (bf16 pools, 16-token blocks).
//
// What it computes is the same as the other decode kernels (kgptalkie "Day 28:
// PagedAttention / vLLM", "The Block Table Is the Map", "Follow One Token
// Address"): for each sequence s and query head, softmax-weighted values of
// every cached key of s, found through s's block table in logical order.
//
// How:
//   * Work is the list of tiles (sequence, KV head, logical block) in that
//     order; T tiles in all.  Warp w of the Wt warps in the grid takes tiles
//     [T*w/Wt, T*(w+1)/Wt): every warp gets the same number of blocks (+-1), so
//     no warp waits for a long sequence at the end of the launch.  A warp's
//     range covers the tail of one (sequence, head) unit, whole units, and the
//     head of another; each piece of a unit is a segment.  A segment that is a
//     whole unit writes the normalised output; any other writes (acc, max, sum)
//     to partial slot unit + w and counts itself in the unit's arrival counter;
//     the warp that completes the count combines the pieces by log-sum-exp
//     (no second launch; nothing waits on another warp).
//   * Each warp runs its own ring of NS shared-memory stages.  Lane 0 issues
//     TMA copies of a tile's keys (64-wide boxes, 128-byte swizzle) and
//     transposed values (one box of 128-byte lines, 128-byte swizzle) into a stage, plus the
//     unit's query rows (a bulk copy) when the tile starts a segment, and the
//     new token's key and value rows when the tile holds the appended position
//     (fused append).  An mbarrier per stage counts the bytes in.  The next NS-1
//     tiles are in flight while a tile is computed, across unit boundaries, and
//     block-table entries are read 32 tiles ahead.
//   * Per tile and warp (mma.sync m16n8k16, bf16 in, fp32 accumulate; operand
//     fragments by ldmatrix from the swizzled stages; two tiles of a unit at a
//     time when they follow each other):
//       S^T[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8]
//       online softmax per head in fp32 (exp2 domain) against a reference
//       maximum that is raised only when a score passes it by 2^8
//       O^T[D x 8] += V^T[D x 16] . P^T[16 x 8], P as a bf16 high part plus a
//       bf16 low part, P^T reaching the operand layout through movmatrix.
#include <cstdint>
#include <cstdlib>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

#ifndef PA_SK_WARPS
#define PA_SK_WARPS 4           // independent warps per CTA (one CTA per SM)
#endif
#ifndef PA_SK_MAX_STAGES
#define PA_SK_MAX_STAGES 6      // ring depth cap per warp
#endif

namespace {

constexpr int kW = PA_SK_WARPS;
constexpr int kT = kW * 32;
constexpr int kMaxStages = PA_SK_MAX_STAGES;
static_assert(kMaxStages >= 3 && kMaxStages <= 32, "stage bits live in 32-bit masks");
constexpr uint32_t kSpin = 1u << 22;     // bounded mbarrier polls (each poll may suspend)

using pa_dev::record_error;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// global -> shared, counted on the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(pa_tc::smem_u32(bar))
        : "memory");
}

// Counter access with explicit ordering: a piece's partial is published by a
// release increment; a warp that sees the count through an acquire load (or
// that fences after its own increment) then reads the other partials.
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int atom_add_release(int* p, int x) {
    int v;
    asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(v) : "l"(p), "r"(x) : "memory");
    return v;
}

// Largest s with s_tiles[s] <= t (s_tiles non-decreasing, s_tiles[0] = 0 <= t < s_tiles[S]).
__device__ __forceinline__ int seq_of_tile(const int* s_tiles, int S, int t) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tiles[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Position in the tile list: sequence, KV head, logical block, blocks of the sequence.
struct Cursor {
    int s, h, j, nb;
};

__device__ __forceinline__ Cursor cursor_at(const int* s_tiles, int S, int Hkv, int t) {
    Cursor c;
    c.s = seq_of_tile(s_tiles, S, t);
    c.nb = (s_tiles[c.s + 1] - s_tiles[c.s]) / Hkv;
    const int local = t - s_tiles[c.s];
    c.h = local / c.nb;
    c.j = local - c.h * c.nb;
    return c;
}

__device__ __forceinline__ void advance(Cursor& c, const int* s_tiles, int S, int Hkv) {
    if (++c.j < c.nb) return;
    c.j = 0;
    if (++c.h < Hkv) return;
    c.h = 0;
    do {
        ++c.s;
    } while (c.s < S && s_tiles[c.s + 1] == s_tiles[c.s]);
    c.nb = c.s < S ? (s_tiles[c.s + 1] - s_tiles[c.s]) / Hkv : 0;
}

// Warp w of Wt has a non-empty tile range [T*w/Wt, T*(w+1)/Wt).
__device__ __forceinline__ bool warp_has_tiles(int T, int Wt, int w) {
    return static_cast<long long>(T) * (w + 1) / Wt > static_cast<long long>(T) * w / Wt;
}

// Combine the pieces of unit u (written by warps w0..w1 to partial slots
// u + w) by log-sum-exp and write the normalised output:
//   M = max m_w,  L = sum l_w 2^(m_w - M),  out = sum acc_w 2^(m_w - M) / L.
// Run by one warp; lane owns D/32 consecutive elements of every head.  The
// pieces come from other SMs, so they are read from L2, two pieces (all heads)
// per round so that a round costs one memory latency.
template <int D>
__device__ void merge_unit(const DecodeParams& p, int u, int s, int h, int w0, int w1, int T,
                           int Wt, int lane) {
    constexpr int E = D / 32;                           // elements per lane per head
    static_assert(E == 2 || E == 4, "head_dim 64 or 128");
    const int G = p.G;
    float M[8], L[8], acc[8][E];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        M[n] = -INFINITY;
        L[n] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[n][e] = 0.f;
    }
    for (int w = w0; w <= w1; w += 2) {
        float2 ml[2][8];
        float x[2][8][E];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const bool okq = w + q <= w1 && warp_has_tiles(T, Wt, w + q);
            const size_t slot = static_cast<size_t>(u) + w + q;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                ml[q][n] = make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int e = 0; e < E; ++e) x[q][n][e] = 0.f;
                if (okq && n < G) {
                    ml[q][n] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (slot * G + n) * 2));
                    const float* src = p.part_acc + (slot * G + n) * D + lane * E;
#pragma unroll
                    for (int e = 0; e < E; e += 2) {
                        const float2 v = __ldcg(reinterpret_cast<const float2*>(src + e));
                        x[q][n][e] = v.x;
                        x[q][n][e + 1] = v.y;
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                if (ml[q][n].x == -INFINITY) continue;  // absent piece (or nothing seen)
                const float nm = fmaxf(M[n], ml[q][n].x);
                const float fo = M[n] == -INFINITY ? 0.f : pa_dev::ex2(M[n] - nm);
                const float fn = pa_dev::ex2(ml[q][n].x - nm);
                L[n] = L[n] * fo + ml[q][n].y * fn;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[n][e] = acc[n][e] * fo + x[q][n][e] * fn;
                M[n] = nm;
            }
    }
    const size_t out0 = (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * G) * D;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        if (n >= G) break;
        const float inv = L[n] > 0.f ? 1.f / L[n] : 0.f;
        const size_t o = out0 + static_cast<size_t>(n) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            if (p.out_bf16) {
                __nv_bfloat162 v = __floats2bfloat162_rn(acc[n][e] * inv, acc[n][e + 1] * inv);
                *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + o + e) = v;
            } else {
                *reinterpret_cast<float2*>(static_cast<float*>(p.out) + o + e) =
                    make_float2(acc[n][e] * inv, acc[n][e + 1] * inv);
            }
        }
    }
}

// A warp's online-softmax state for the unit it is working on.
template <int D>
struct Acc {
    uint32_t qf[D / 16][2];      // Q^T B-fragments per 16-wide k-step
    float o[D / 16][4];          // O^T: rows d = 16t + g (+8), columns heads 2c, 2c+1
    float m0, m1, l0, l1;        // reference max / partial sum, heads 2c, 2c+1 (log2 units)
};

// Stage layout (bytes from the stage base, 1024-aligned):
//   [0, 32D)     K tile: D/64 boxes of 16 rows x 128 B, 128-byte swizzle
//   [32D, 64D)   V^T tile: D/4 lines of 128 B (4 d rows x 16 tokens), 128-byte swizzle
//   [64D, 80D)   query rows of the unit (G rows of 2D bytes; rows G..7 zero)
//   [80D, 84D)   fused append: the new token's key row, then its value row
// The softmax reference maximum of a head is raised only when a score exceeds
// it by more than kRaise (log2 units), so probabilities 2^(x - ref) stay below
// 2^kRaise and the common tile needs no cross-lane maximum and no rescale.
constexpr float kRaise = 8.f;

// NTL consecutive tiles of one unit (stage bases kb0, kb1; V^T at +32D).  Only
// the last of them may be partly filled (nvalid_last tokens).
template <int D, int NTL>
__device__ __forceinline__ void tiles_compute(Acc<D>& a, uint32_t kb0, uint32_t kb1, int nvalid_last,
                                              float sl, int lane) {
    constexpr int KS = D / 16;
    const int g = lane >> 2, c = lane & 3;
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;   // ldmatrix row of this lane
    const int hi = lane >> 4;                           // ldmatrix column half
    const uint32_t kbs[2] = {kb0, kb1};
    float sc[NTL][2][4];                                // [tile][chain][fragment]
#pragma unroll
    for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[tl][0][i] = sc[tl][1][i] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        const int cd = 2 * kk + hi;                     // 16-byte chunk along d
        const uint32_t off = (cd >> 3) * 2048 + r * 128 + (((cd & 7) ^ (r & 7)) << 4);
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kbs[tl] + off, a0, a1, a2, a3);
            pa_dev::mma_bf16_16816(sc[tl][kk & 1], a0, a1, a2, a3, a.qf[kk][0], a.qf[kk][1]);
        }
    }
    // x[tl]: tokens g ([0], [1]) and g + 8 ([2], [3]) of tile tl; heads 2c, 2c + 1
    float x[NTL][4];
#pragma unroll
    for (int tl = 0; tl < NTL; ++tl)
#pragma unroll
        for (int i = 0; i < 4; ++i) x[tl][i] = (sc[tl][0][i] + sc[tl][1][i]) * sl;
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (nvalid_last < 16) {                             // partly filled last block
        if (g >= nvalid_last) x[NTL - 1][0] = x[NTL - 1][1] = -INFINITY;
        if (g + 8 >= nvalid_last) x[NTL - 1][2] = x[NTL - 1][3] = -INFINITY;
        mlo = (2 * c < nvalid_last ? 0x0000ffffu : 0u) | (2 * c + 1 < nvalid_last ? 0xffff0000u : 0u);
        mhi = (2 * c + 8 < nvalid_last ? 0x0000ffffu : 0u) | (2 * c + 9 < nvalid_last ? 0xffff0000u : 0u);
    }
    bool need = false;
#pragma unroll
    for (int tl = 0; tl < NTL; ++tl)
        need |= x[tl][0] > a.m0 + kRaise || x[tl][2] > a.m0 + kRaise ||
                x[tl][1] > a.m1 + kRaise || x[tl][3] > a.m1 + kRaise;
    if (__any_sync(0xffffffffu, need)) {                // raise the references to the true maxima
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            mx0 = fmaxf(mx0, fmaxf(x[tl][0], x[tl][2]));
            mx1 = fmaxf(mx1, fmaxf(x[tl][1], x[tl][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float n0 = fmaxf(a.m0, mx0), n1 = fmaxf(a.m1, mx1);
        const float cr0 = a.m0 == -INFINITY ? 0.f : pa_dev::ex2(a.m0 - n0);
        const float cr1 = a.m1 == -INFINITY ? 0.f : pa_dev::ex2(a.m1 - n1);
        a.l0 *= cr0;
        a.l1 *= cr1;
#pragma unroll
        for (int t = 0; t < KS; ++t) {
            a.o[t][0] *= cr0; a.o[t][1] *= cr1;
            a.o[t][2] *= cr0; a.o[t][3] *= cr1;
        }
        a.m0 = n0;
        a.m1 = n1;
    }
    const float ref0 = a.m0 == -INFINITY ? 0.f : a.m0, ref1 = a.m1 == -INFINITY ? 0.f : a.m1;
    // P rows (token g / g + 8, heads 2c, 2c+1) -> P^T B-fragments (tokens 2c.., head g),
    // each as a bf16 high part and a bf16 low part
    uint32_t bh[NTL][2], be[NTL][2];
#pragma unroll
    for (int tl = 0; tl < NTL; ++tl) {
        const float p0 = pa_dev::ex2(x[tl][0] - ref0), p1 = pa_dev::ex2(x[tl][1] - ref1);
        const float p2 = pa_dev::ex2(x[tl][2] - ref0), p3 = pa_dev::ex2(x[tl][3] - ref1);
        a.l0 += p0 + p2;
        a.l1 += p1 + p3;
        const uint32_t h01 = pa_dev::pack_bf16(p0, p1), h23 = pa_dev::pack_bf16(p2, p3);
        const uint32_t e01 = pa_dev::pack_bf16(p0 - pa_dev::bf16_lo(h01), p1 - pa_dev::bf16_hi(h01));
        const uint32_t e23 = pa_dev::pack_bf16(p2 - pa_dev::bf16_lo(h23), p3 - pa_dev::bf16_hi(h23));
        bh[tl][0] = pa_dev::movmatrix_trans(h01);
        bh[tl][1] = pa_dev::movmatrix_trans(h23);
        be[tl][0] = pa_dev::movmatrix_trans(e01);
        be[tl][1] = pa_dev::movmatrix_trans(e23);
    }
#pragma unroll
    for (int t = 0; t < KS; ++t) {
        const int d = 16 * t + r;                       // V^T row; line d/4, chunk 2(d%4) + hi
        const uint32_t off = 32 * D + (d >> 2) * 128 + (((((d & 3) << 1) | hi) ^ ((d >> 2) & 7)) << 4);
#pragma unroll
        for (int tl = 0; tl < NTL; ++tl) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4(kbs[tl] + off, v0, v1, v2, v3);
            if (tl == NTL - 1) {
                v0 &= mlo; v1 &= mlo; v2 &= mhi; v3 &= mhi;
            }
            pa_dev::mma_bf16_16816(a.o[t], v0, v1, v2, v3, bh[tl][0], bh[tl][1]);
            pa_dev::mma_bf16_16816(a.o[t], v0, v1, v2, v3, be[tl][0], be[tl][1]);
        }
    }
}

template <int D, bool FUSE>
__global__ void __launch_bounds__(kT, 1)
decode_stream_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap) {
    constexpr int KS = D / 16;
    extern __shared__ unsigned char sk_raw[];
    const uint32_t raw_s = pa_tc::smem_u32(sk_raw);
    unsigned char* base = sk_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const int NS = p.sk_stages;
    const uint32_t SB = static_cast<uint32_t>(p.sk_stage_bytes);
    const int S = p.S, Hkv = p.Hkv, G = p.G;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + static_cast<size_t>(kW) * NS * SB);
    int* s_phys = reinterpret_cast<int*>(bars + kW * NS);      // [kW][kMaxStages] block id of each stage
    int* s_tiles = s_phys + kW * kMaxStages;                    // [S + 1] first tile of each sequence
    int* s_len = s_tiles + S + 1;                               // [S] context lengths
    int* s_red = s_len + S;                                     // [kW] scan scratch

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t wbase = pa_tc::smem_u32(base) + static_cast<uint32_t>(warp) * NS * SB;
    uint64_t* wbar = bars + warp * NS;

    // ---- set-up that reads no input: barriers, zeroed query regions
    if (lane == 0) {
        for (int i = 0; i < NS; ++i) pa_tc::mbar_init(wbar + i, 1);
        pa_tc::mbar_init_fence();
    }
    for (int i = 0; i < NS; ++i)
        for (int o = lane * 16; o < 16 * D; o += 32 * 16)
            *reinterpret_cast<uint4*>(base + (static_cast<size_t>(warp) * NS + i) * SB + 64 * D + o) =
                make_uint4(0u, 0u, 0u, 0u);
    pa_tc::fence_smem_to_async();
    pa_dev::wait_prior_grid();

    // ---- tile prefix over sequences (every CTA builds the same one)
    {
        const int per = (S + kT - 1) / kT;
        const int lo = min(S, tid * per), hi = min(S, lo + per);
        const int cap = p.max_blocks * 16;
        int cnt = 0;
        for (int s = lo; s < hi; ++s) {
            int L = __ldg(p.lens + s);
            if (L < 0 || L > cap) {
                if (blockIdx.x == 0) record_error(p.err, PA_ERR_BAD_LENGTH);
                L = L < 0 ? 0 : cap;
            }
            s_len[s] = L;
            cnt += ((L + 15) >> 4) * Hkv;
        }
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) s_red[warp] = inc;
        __syncthreads();
        int b = inc - cnt;
        for (int w = 0; w < warp; ++w) b += s_red[w];
        for (int s = lo; s < hi; ++s) {
            s_tiles[s] = b;
            b += ((s_len[s] + 15) >> 4) * Hkv;
        }
        if (tid == kT - 1) s_tiles[S] = b;              // the last thread's end is the total
        __syncthreads();
    }
    const int T = s_tiles[S];
    const int Wt = static_cast<int>(gridDim.x) * kW;
    if (blockIdx.x == 0) {                               // schedule, published for inspection
        if (tid == 0) {
            p.sched[0] = T;
            p.sched[1] = Wt;
        }
        for (int i = tid; i <= S; i += kT) p.sched[2 + i] = s_tiles[i];
    }
    pa_dev::allow_next_grid();
    // a sequence with no cached position attends to nothing: zeros
    for (int s0 = blockIdx.x; s0 < S; s0 += gridDim.x) {
        if (s_len[s0] != 0) continue;
        const size_t o0 = static_cast<size_t>(s0) * p.Hq * D;
        for (int e = tid; e < p.Hq * D; e += kT) {
            if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[o0 + e] = __float2bfloat16_rn(0.f);
            else static_cast<float*>(p.out)[o0 + e] = 0.f;
        }
    }

    const int gw = static_cast<int>(blockIdx.x) * kW + warp;
    const int t0 = static_cast<int>(static_cast<long long>(T) * gw / Wt);
    const int t1 = static_cast<int>(static_cast<long long>(T) * (gw + 1) / Wt);
    const int n = t1 - t0;
    if (n <= 0) return;

    const uint16_t* kpool = static_cast<const uint16_t*>(p.k);
    const uint16_t* vpool = static_cast<const uint16_t*>(p.v);
    const char* qg = static_cast<const char*>(p.q);
    const float sl = p.scale_log2;

    // Block ids of 32 consecutive tiles of this warp's list, one per lane.  The
    // loads are started one window (32 tiles) before use and checked only when
    // the window becomes current, so no wait on them sits in the pipeline.
    struct Window {
        int phys;               // raw table entry
        int off;                // fused form: offset of position L-1 when this is a unit's last tile, else -1
        long long slot;         // fused form: the sequence's new-token slot (raw)
        bool has;               // the lane's tile exists
    };
    auto load_window = [&](int k) {
        Window w{-1, -1, -1, false};
        const int idx = 32 * k + lane;
        if (idx >= n) return w;
        const Cursor c = cursor_at(s_tiles, S, Hkv, t0 + idx);
        w.has = true;
        w.phys = __ldg(p.tables + static_cast<size_t>(c.s) * p.max_blocks + c.j);
        if (FUSE && c.j == c.nb - 1) {
            w.off = (s_len[c.s] - 1) - 16 * c.j;
            w.slot = __ldg(p.new_slots + c.s);
        }
        return w;
    };
    // checked block id (-1 if none or outside the pool) and "receives the new token"
    int wcur_p = -1, wcur_f = 0;
    auto take_window = [&](const Window& w) {
        int phys = w.has ? w.phys : -1;
        if (w.has && (phys < 0 || phys >= p.num_blocks)) {
            record_error(p.err, PA_ERR_BAD_BLOCK_ID);
            phys = -1;
        }
        wcur_p = phys;
        wcur_f = 0;
        if (FUSE && phys >= 0 && w.off >= 0 && w.slot >= 0) {
            if (w.slot == static_cast<long long>(phys) * 16 + w.off) wcur_f = 1;
            else record_error(p.err, PA_ERR_INVALID_ARG);        // not this sequence's slot
        }
    };
    Window wnxt = load_window(0);
    take_window(wnxt);
    wnxt = load_window(1);

    // ---- issue side: tile i of the list into stage i % NS
    Cursor ic = cursor_at(s_tiles, S, Hkv, t0);
    uint32_t valid = 0, app = 0;                         // per stage (bit = stage), warp-uniform
    int ist = 0;
    auto issue = [&](int i) {
        if (i > 0 && (i & 31) == 0) {
            take_window(wnxt);
            wnxt = load_window((i >> 5) + 1);
        }
        const int phys = __shfl_sync(0xffffffffu, wcur_p, i & 31);
        const int ap = __shfl_sync(0xffffffffu, wcur_f, i & 31);
        const bool first = i == 0 || ic.j == 0;
        const uint32_t bytes = (phys >= 0 ? 64u * D : 0u) + (first ? 2u * G * D : 0u) + (ap ? 4u * D : 0u);
        const uint32_t st = wbase + ist * SB;
        if (lane == 0) {
            s_phys[warp * kMaxStages + ist] = phys;
            pa_tc::fence_smem_to_async();                // earlier reads of this stage come first
            pa_tc::mbar_expect_tx(wbar + ist, bytes);
            if (phys >= 0) {
                const int row = phys * Hkv + ic.h;
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    pa_tc::tma_load_2d(st + b * 2048, &kmap, 64 * b, row * 16, wbar + ist);
                pa_tc::tma_load_2d(st + 32 * D, &vmap, 0, row * (D / 4), wbar + ist);
            }
            if (first)
                bulk_load(st + 64 * D,
                          qg + (static_cast<size_t>(ic.s) * p.Hq + static_cast<size_t>(ic.h) * G) * D * 2,
                          2u * G * D, wbar + ist);
            if (FUSE && ap) {
                const size_t row = (static_cast<size_t>(ic.s) * Hkv + ic.h) * D * 2;
                bulk_load(st + 80 * D, static_cast<const char*>(p.new_k) + row, 2u * D, wbar + ist);
                bulk_load(st + 82 * D, static_cast<const char*>(p.new_v) + row, 2u * D, wbar + ist);
            }
        }
        valid = phys >= 0 ? (valid | (1u << ist)) : (valid & ~(1u << ist));
        app = ap ? (app | (1u << ist)) : (app & ~(1u << ist));
        advance(ic, s_tiles, S, Hkv);
        if (++ist == NS) ist = 0;
    };

    const int npro = n < NS ? n : NS;
    for (int i = 0; i < npro; ++i) issue(i);

    // ---- consume side
    Cursor cc = cursor_at(s_tiles, S, Hkv, t0);
    Acc<D> a;
    int seg_j0 = 0;
    int cst = 0;
    uint32_t phase = 0;                                  // bit per stage
    const int g = lane >> 2, c = lane & 3;
    bool ok = true;
    int fail_at = 0;
    // The warp's first piece, when another warp shares its unit: published
    // mid-range by a release increment whose result is looked at only at the
    // end of the range (so no wait on it sits in the stream).
    int pend_u = -1, pend_prev = 0;
    // The warp's last piece, when shared: a few tiles before its end the
    // unit's counter is read (acquire); if every other piece is published by
    // then, this warp merges at once, without an increment.
    constexpr int kSoleLead = 4;
    int sole_cnt = -1;
    bool sole_read = false;
    for (int i = 0; i < n;) {
        // two consecutive tiles of one unit are computed together
        const bool pair = i + 1 < n && cc.j + 1 < cc.nb;
        const int c0 = cst, c1 = cst + 1 == NS ? 0 : cst + 1;
        bool w = pa_tc::mbar_wait(wbar + c0, (phase >> c0) & 1u, kSpin);
        if (pair) w = w && pa_tc::mbar_wait(wbar + c1, (phase >> c1) & 1u, kSpin);
        if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            fail_at = i;
            break;
        }
        phase ^= (1u << c0) | (pair ? (1u << c1) : 0u);
        const uint32_t st0 = wbase + c0 * SB, st1 = wbase + c1 * SB;
        const int s = cc.s, h = cc.h;
        const int L = s_len[s];
        const bool first = i == 0 || cc.j == 0;
        if (first) {
            const uint32_t qb = st0 + 64 * D + (lane & 7) * (2 * D);
#pragma unroll
            for (int k2 = 0; k2 < D / 32; ++k2)
                ldsm_x4(qb + ((4 * k2 + (lane >> 3)) << 4), a.qf[2 * k2][0], a.qf[2 * k2][1],
                        a.qf[2 * k2 + 1][0], a.qf[2 * k2 + 1][1]);
#pragma unroll
            for (int t = 0; t < KS; ++t) a.o[t][0] = a.o[t][1] = a.o[t][2] = a.o[t][3] = 0.f;
            a.m0 = a.m1 = -INFINITY;
            a.l0 = a.l1 = 0.f;
            seg_j0 = cc.j;
        }
        // the last tile of this step (only it can be a unit's last block)
        const int jl = pair ? cc.j + 1 : cc.j, cl = pair ? c1 : c0;
        if (FUSE && ((app >> cl) & 1u)) {
            // the appended position: the new key row and value column go into
            // the staged tile (which the copy filled with the old contents) and
            // into the pool
            const int phys = s_phys[warp * kMaxStages + cl];
            const int off = (L - 1) - 16 * jl;
            const size_t tile = (static_cast<size_t>(phys) * Hkv + h) * 16 * D;
            uint16_t* kw = const_cast<uint16_t*>(kpool) + tile + static_cast<size_t>(off) * D;
            uint16_t* vw = const_cast<uint16_t*>(vpool) + tile + off;
            unsigned char* sb = base + (static_cast<size_t>(warp) * NS + cl) * SB;
            for (int ch = lane; ch < D / 8; ch += 32) {
                const uint4 val = *reinterpret_cast<const uint4*>(sb + 80 * D + ch * 16);
                *reinterpret_cast<uint4*>(sb + (ch >> 3) * 2048 + off * 128 + (((ch & 7) ^ (off & 7)) << 4)) = val;
                *reinterpret_cast<uint4*>(kw + ch * 8) = val;
            }
            for (int d = lane; d < D; d += 32) {
                const uint16_t val = *reinterpret_cast<const uint16_t*>(sb + 82 * D + d * 2);
                *reinterpret_cast<uint16_t*>(sb + 32 * D + (d >> 2) * 128 +
                                             (((((d & 3) << 1) | (off >> 3)) ^ ((d >> 2) & 7)) << 4) +
                                             (off & 7) * 2) = val;
                vw[static_cast<size_t>(d) * 16] = val;
            }
            __syncwarp();
        }
        const bool v0 = (valid >> c0) & 1u, v1 = pair && ((valid >> c1) & 1u);
        const int nv_last = min(16, L - 16 * jl);
        if (pair && v0 && v1) {
            tiles_compute<D, 2>(a, st0, st1, nv_last, sl, lane);
        } else {
            if (v0) tiles_compute<D, 1>(a, st0, st0, pair ? 16 : nv_last, sl, lane);
            if (v1) tiles_compute<D, 1>(a, st1, st1, nv_last, sl, lane);
        }
        if (pair) advance(cc, s_tiles, S, Hkv);         // cc: the last tile of this step
        const int il = pair ? i + 1 : i;
        if (!sole_read && n - 1 - il <= kSoleLead) {
            // this step lies in the range's last kSoleLead tiles: if its unit
            // reaches the range end (the range's final piece) and is shared with
            // another warp, start reading the unit's counter
            const int U0 = s_tiles[s] + h * cc.nb, U1 = U0 + cc.nb;
            if (U1 >= t1 && (U0 < t0 || U1 > t1)) {
                sole_read = true;
                if (lane == 0) sole_cnt = ld_acquire(p.unit_cnt + s * Hkv + h);
            }
        }
        const bool last = cc.j == cc.nb - 1 || il == n - 1;
        if (last) {
            float l0 = a.l0, l1 = a.l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            const bool whole = seg_j0 == 0 && cc.j == cc.nb - 1;
            const int n0 = 2 * c, n1 = 2 * c + 1;
            if (whole) {
                const size_t o0 = (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * G) * D;
                const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
                for (int t = 0; t < KS; ++t) {
                    const int d = 16 * t + g;
                    if (p.out_bf16) {
                        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + o0;
                        if (n0 < G) {
                            out[n0 * D + d] = __float2bfloat16_rn(a.o[t][0] * i0);
                            out[n0 * D + d + 8] = __float2bfloat16_rn(a.o[t][2] * i0);
                        }
                        if (n1 < G) {
                            out[n1 * D + d] = __float2bfloat16_rn(a.o[t][1] * i1);
                            out[n1 * D + d + 8] = __float2bfloat16_rn(a.o[t][3] * i1);
                        }
                    } else {
                        float* out = static_cast<float*>(p.out) + o0;
                        if (n0 < G) {
                            out[n0 * D + d] = a.o[t][0] * i0;
                            out[n0 * D + d + 8] = a.o[t][2] * i0;
                        }
                        if (n1 < G) {
                            out[n1 * D + d] = a.o[t][1] * i1;
                            out[n1 * D + d + 8] = a.o[t][3] * i1;
                        }
                    }
                }
            } else {
                const int u = s * Hkv + h;
                const size_t slot = static_cast<size_t>(u) + gw;
                float* acc = p.part_acc + slot * G * D;
#pragma unroll
                for (int t = 0; t < KS; ++t) {
                    const int d = 16 * t + g;
                    if (n0 < G) {
                        acc[n0 * D + d] = a.o[t][0];
                        acc[n0 * D + d + 8] = a.o[t][2];
                    }
                    if (n1 < G) {
                        acc[n1 * D + d] = a.o[t][1];
                        acc[n1 * D + d + 8] = a.o[t][3];
                    }
                }
                if (g == 0) {
                    if (n0 < G) {
                        p.part_ml[(slot * G + n0) * 2] = a.m0;
                        p.part_ml[(slot * G + n0) * 2 + 1] = l0;
                    }
                    if (n1 < G) {
                        p.part_ml[(slot * G + n1) * 2] = a.m1;
                        p.part_ml[(slot * G + n1) * 2 + 1] = l1;
                    }
                }
                // The last warp to finish a piece of this unit merges the pieces.
                __syncwarp();
                const long long T0 = s_tiles[s] + static_cast<long long>(h) * cc.nb, T1 = T0 + cc.nb;
                const int w0 = static_cast<int>(((T0 + 1) * Wt - 1) / T);
                const int w1 = static_cast<int>((T1 * Wt - 1) / T);
                int parts = 0;
                for (int w = w0 + lane; w <= w1; w += 32) parts += warp_has_tiles(T, Wt, w);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) parts += __shfl_xor_sync(0xffffffffu, parts, off);
                const bool final_piece = il == n - 1;
                const int seen = __shfl_sync(0xffffffffu, sole_cnt, 0);
                if (final_piece && sole_read && seen == parts - 1) {
                    // every other piece was published before the read: merge now
                    merge_unit<D>(p, u, s, h, w0, w1, T, Wt, lane);
                    if (lane == 0) p.unit_cnt[u] = 0;     // ready for the next launch
                } else if (final_piece) {
                    int prev = 0;
                    if (lane == 0) prev = atom_add_release(p.unit_cnt + u, 1);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    if (prev == parts - 1) {
                        __threadfence();
                        merge_unit<D>(p, u, s, h, w0, w1, T, Wt, lane);
                        if (lane == 0) p.unit_cnt[u] = 0;
                    }
                } else {
                    // the range's first piece: publish now, look at the count at the end
                    if (lane == 0) pend_prev = atom_add_release(p.unit_cnt + u, 1);
                    pend_u = u;
                }
            }
        }
        advance(cc, s_tiles, S, Hkv);
        cst = c1;
        if (pair && ++cst == NS) cst = 0;
        __syncwarp();                                    // every lane is done with these stages
        if (i + NS < n) issue(i + NS);
        if (pair && i + 1 + NS < n) issue(i + 1 + NS);
        i = il + 1;
    }
    if (ok && pend_u >= 0) {
        // the first piece's increment: if it completed its unit's count, merge it
        const int su = pend_u / Hkv, hu = pend_u - su * Hkv;
        const int nbu = (s_tiles[su + 1] - s_tiles[su]) / Hkv;
        const long long T0 = s_tiles[su] + static_cast<long long>(hu) * nbu, T1 = T0 + nbu;
        const int w0 = static_cast<int>(((T0 + 1) * Wt - 1) / T);
        const int w1 = static_cast<int>((T1 * Wt - 1) / T);
        int parts = 0;
        for (int w = w0 + lane; w <= w1; w += 32) parts += warp_has_tiles(T, Wt, w);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) parts += __shfl_xor_sync(0xffffffffu, parts, off);
        const int prev = __shfl_sync(0xffffffffu, pend_prev, 0);
        if (prev == parts - 1) {
            __threadfence();
            merge_unit<D>(p, pend_u, su, hu, w0, w1, T, Wt, lane);
            if (lane == 0) p.unit_cnt[pend_u] = 0;
        }
    }
    if (!ok) {
        // a copy did not arrive in time: record it and wait (bounded) for the
        // copies still in flight into this warp's stages (tiles fail_at ..
        // min(n, fail_at + NS) - 1, from stage cst on) before leaving
        if (lane == 0) {
            record_error(p.err, PA_ERR_CUDA);
            const int pending = min(n - fail_at, NS);
            int k = cst;
            for (int q = 0; q < pending; ++q) {
                pa_tc::mbar_wait(wbar + k, (phase >> k) & 1u, kSpin);
                if (++k == NS) k = 0;
            }
        }
        __syncwarp();
    }
}

}  // namespace

namespace pa_detail {

namespace {

size_t stream_stage_bytes(int D, bool fuse) {
    const size_t b = static_cast<size_t>(fuse ? 84 : 80) * D;
    return (b + 1023) / 1024 * 1024;
}

size_t stream_smem(int S, int stages, size_t stage_bytes) {
    return 1024 + static_cast<size_t>(kW) * stages * stage_bytes + static_cast<size_t>(kW) * stages * 8 +
           static_cast<size_t>(kW) * kMaxStages * 4 + static_cast<size_t>(2 * S + 1) * 4 + kW * 4 + 16;
}

template <int D, bool FUSE>
cudaError_t launch_split(const DecodeParams& p, const pa_pool* pool, int grid, size_t smem,
                         cudaStream_t st) {
    // largest dynamic size set on the kernel so far, per device
    static size_t configured[64] = {};
    const int dev = pool->device >= 0 && pool->device < 64 ? pool->device : 0;
    if (smem > configured[dev] || pool->device >= 64) {
        const cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<D, FUSE>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = smem;
    }
    return launch_pdl(decode_stream_kernel<D, FUSE>, dim3(grid), dim3(kT), smem, st, p, pool->kmap,
                      pool->vmap_lines);
}

}  // namespace

bool plan_stream(pa_pool* pool, int S, int Hq, int max_blocks, DecodePlan* plan) {
    // Opt-in (PA_DECODE_STREAM=1): on GB300 the ticketed split kernel measures as
    // fast or faster on every workload but the smallest batches.
    const char* env = std::getenv("PA_DECODE_STREAM");
    if (!env || env[0] != '1') return false;
    const int Hkv = pool->kv_heads, D = pool->head_dim, G = Hq / Hkv;
    if (pool->dtype != PA_BF16 || pool->block_size != 16 || G < 1 || G > 8 || S < 1 || S > 4096)
        return false;
    if (D != 64 && D != 128) return false;         // D = 256 leaves room for fewer than 3 stages
    // TMA coordinates and the tile count are 32-bit
    if (static_cast<long long>(pool->num_blocks) * Hkv * (D > 16 ? D : 16) >= (1LL << 31)) return false;
    if (static_cast<long long>(S) * max_blocks * Hkv >= (1LL << 31)) return false;
    const size_t sb = stream_stage_bytes(D, plan->fuse);
    int stages = PA_SK_MAX_STAGES;
    while (stages >= 3 && stream_smem(S, stages, sb) > static_cast<size_t>(pool->smem_optin)) --stages;
    if (stages < 3) return false;
    if (ensure_tensor_maps(pool) != PA_OK) return false;
    plan->stream = true;
    plan->fast = true;
    plan->bf16 = true;
    plan->pool = pool;
    plan->threads = kT;
    plan->grid = pool->num_sms;
    plan->smem = stream_smem(S, stages, sb);
    plan->sk_stages = stages;
    plan->sk_stage_bytes = static_cast<int>(sb);
    plan->items_target = 0;
    plan->pt_min = 0;
    plan->pt_fixed = 0;
    plan->max_items = static_cast<size_t>(S) * Hkv + static_cast<size_t>(plan->grid) * kW;
    plan->min_items = plan->max_items;
    return true;
}

int launch_stream(const DecodePlan& plan, const DecodeParams& prm, cudaStream_t st) {
    DecodeParams p = prm;
    p.sk_stages = plan.sk_stages;
    p.sk_stage_bytes = plan.sk_stage_bytes;
    cudaError_t e;
    const pa_pool* pool = plan.pool;
    if (p.D == 64) e = plan.fuse ? launch_split<64, true>(p, pool, plan.grid, plan.smem, st)
                                 : launch_split<64, false>(p, pool, plan.grid, plan.smem, st);
    else e = plan.fuse ? launch_split<128, true>(p, pool, plan.grid, plan.smem, st)
                       : launch_split<128, false>(p, pool, plan.grid, plan.smem, st);
    count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
