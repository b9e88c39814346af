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
//     on the device from the batch's total length so that the items fill
//     whole waves of one item per resident CTA: one wave for a small batch,
//     up to about twelve items per SM for a large one; long contexts are
//     split over block ranges and merged by log-sum-exp.  The grid is
//     persistent (a few CTAs per SM);
//     every CTA builds the same item list from context_lens in shared memory
//     and takes items by a global ticket.
//   * Each item is served by the CTA's 4 warps, which take the partition's
//     blocks round-robin and keep their own online-softmax state; at the end
//     of the item each head's warp weights are computed once and every thread
//     writes its merged columns out.
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
//   * fp8 (e4m3) pools: the same tiles with half the bytes; each thread's
//     codes are widened to f16 pairs (exact) just before the MMA that reads
//     them, queries are re-rounded to f16 and P is an f16 pair.  With G <= 4
//     the score columns 4..7 repeat heads 0..3 and carry P's remainders, so
//     one value MMA per m-tile takes both parts.  The walk fits 128 registers,
//     four CTAs per SM.
//   * f32 pools (and shapes outside the tensor-core tile) use a plain fp32
//     CUDA-core item: scores to shared memory, softmax, value mix.
//   * An item whose sequence has one partition writes the normalised output.
//     Otherwise it writes (acc, max, sum) to the workspace, and the merge
//     kernel, launched behind the split pass with programmatic dependent
//     launch, combines each (sequence, head)'s partials by log-sum-exp.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

// Tuning constants (the measured best on GB300).
namespace {

constexpr int kItemsPerSm = 12;         // most work items per SM (12 beat 9 and 15 on GB300)
constexpr int kWarps = 4;               // warps per CTA sharing one item
constexpr int kMinCtas = 3;             // resident CTAs per SM the register budget aims at (bf16)
constexpr int kMinCtasF8 = 4;           // the same for the fp8 walk (one tile in flight per warp)
constexpr int kPtMax = 2048;            // partition cap in tokens for batches of many sequences
constexpr int kPtSoftF8 = 256;          // fp8 pools: smallest partition while items allow, tokens
constexpr size_t kWaveBytes = 1u << 20;  // cache bytes per item that justify another wave of items
constexpr int kBlockPrefetch = 1;       // L2 prefetch of the block a warp reads this many blocks ahead
constexpr int kGuideMinPT = 256;        // shortest partition of the guided tail, tokens
constexpr int kSharedStages = 8;        // staged 16-token tiles per CTA for shared-prefix items
constexpr int kSharedUnitsPerSync = 2;  // tiles consumed per barrier by shared-prefix items
static_assert(kSharedStages > kSharedUnitsPerSync, "shared pipeline needs copies in flight");
static_assert(kSharedUnitsPerSync % 2 == 0, "shared items consume 32-token tiles");
constexpr int kThreads = kWarps * 32;
constexpr int kMergeThreads = 512;      // merge kernel: four groups of 128 threads share a (sequence, KV head)

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

// First token of a sequence's private span: tokens before it are a shared
// prefix that pa_decode_shared serves with its shared items.
__device__ __forceinline__ int priv_start(const DecodeParams& p, int s) {
    return p.seq_start ? __ldg(p.seq_start + s) : 0;
}

__device__ __forceinline__ int priv_len(const DecodeParams& p, int s, bool report) {
    return max(0, seq_len(p, s, report) - priv_start(p, s));
}

__device__ __forceinline__ bool in_group(const DecodeParams& p, int s) {
    return p.seq_group && __ldg(p.seq_group + s) >= 0;
}

struct Sched {
    int PT;
    int total_items;    // private items (the shared ones come first in the item order)
    int PTs;            // partition of sequences s >= S_split (the launch's last items)
    int S_split;
    __device__ __forceinline__ int pt(int s) const { return s >= S_split ? PTs : PT; }
};

// Every CTA derives the same private item list: per sequence nP =
// max(1, ceil(Lp/PT)) partitions of its private span (length Lp), each of Hkv
// items; s_start[s] = first private item of sequence s.
__device__ Sched build_schedule(const DecodeParams& p, int* s_start, long long* s_red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.S + kThreads - 1) / kThreads;
    const int lo = min(p.S, tid * per), hi = min(p.S, lo + per);
    const bool report = blockIdx.x == 0;
    // tokens before this thread's sequences (exclusive scan) and in all
    long long tok = 0;
    for (int s = lo; s < hi; ++s) tok += priv_len(p, s, report);
    long long tinc = tok;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, tinc, o);
        if (lane >= o) tinc += y;
    }
    if (lane == 31) s_red[warp] = tinc;
    __syncthreads();
    long long total = 0, tbase = tinc - tok;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        total += s_red[w];
        if (w < warp) tbase += s_red[w];
    }
    int PT, PTs;
    long long split_at = LLONG_MAX;
    if (p.pt_fixed > 0) {
        PT = PTs = p.pt_fixed;
    } else {
        // Item target: whole waves of wave_items (one item per resident CTA),
        // as many as the token-heads fill at wave_tokens per item, at most
        // items_target.  Small batches run in one wave: a second, partial wave
        // of short items costs more in per-item work than it saves in balance
        // (measured on GB300: 16 sequences 33.3 -> 29.1 us bf16, 28.9 -> 24.6
        // us fp8; 2 long sequences fp8 80.8 -> 71.5 us); large ones keep
        // items_target for balance (8 long sequences fp8: 229 us at three
        // waves, 237 us at one).
        long long target = p.items_target;
        if (p.wave_items > 0 && p.wave_tokens > 0) {
            const long long per_wave = static_cast<long long>(p.wave_items) * p.wave_tokens;
            const long long waves = (total * p.Hkv + per_wave - 1) / per_wave;
            target = min(target, max(1LL, waves) * p.wave_items);
        }
        long long need = (total * p.Hkv + target - 1) / target;
        need = (need + p.B - 1) / p.B * p.B;
        // Smallest partition: pt_min, raised towards pt_soft tokens as far as
        // that still leaves items_floor items.  fp8 pools use it: an item's
        // fixed work (its queries, the warps' merge, its partial) weighs more
        // against tiles of half the bytes, and at pt_soft the guided tail
        // below is allowed again for batches of a few thousand tokens.
        long long pmin = p.pt_min;
        if (p.pt_soft > p.pt_min && p.items_floor > 0) {
            const long long cap = total * p.Hkv / p.items_floor / p.B * p.B;
            pmin = max(pmin, min(static_cast<long long>(p.pt_soft), cap));
            if (p.pt_max > 0) pmin = min(pmin, static_cast<long long>(p.pt_max));
        }
        // cap the partition so the launch's last items are short (long
        // sequences split into more items; the merge combines them), but never
        // below the length that keeps the item count within the workspace:
        // items <= Hkv * (total / PT + S) <= max_items
        if (p.pt_max > 0) {
            const long long room = static_cast<long long>(p.max_items) - static_cast<long long>(p.Hkv) * p.S;
            long long lo = room > 0 ? (total * p.Hkv + room - 1) / room : need;
            lo = (lo + p.B - 1) / p.B * p.B;
            need = min(need, max(static_cast<long long>(p.pt_max), lo));
        }
        PT = static_cast<int>(max(need, pmin));
        // Guided tail: sequences that start in the last quarter of the tokens
        // (they are the last items handed out) use partitions a quarter as long,
        // so the launch ends on short items.  Their tokens are at most a quarter
        // of the total, so items <= Hkv * (total/PT + total/(4 PTs) + S); used
        // only when that fits the workspace, and only when the short partitions
        // still hold kGuideMinPT tokens (shorter items cost more to start than
        // they save at the end: measured on GB300).
        PTs = max(static_cast<int>(pmin), (PT / 4 + p.B - 1) / p.B * p.B);
        const long long bound = static_cast<long long>(p.Hkv) *
            ((total + PT - 1) / PT + (total + 4LL * PTs - 1) / (4LL * PTs) + p.S);
        if (PTs < PT && PTs >= kGuideMinPT && bound <= p.max_items) split_at = total - total / 4;
        else PTs = PT;
    }
    // first sequence starting at or after split_at (every thread of the CTA
    // has the same split_at, so the branch is uniform)
    int S_split = p.S;
    __syncthreads();                                // s_red reuse
    if (split_at != LLONG_MAX) {
        int* s_split = reinterpret_cast<int*>(s_red);
        if (tid == 0) *s_split = p.S;
        __syncthreads();
        long long c = tbase;
        for (int s = lo; s < hi; ++s) {
            if (c >= split_at) {
                atomicMin(s_split, s);
                break;
            }
            c += priv_len(p, s, false);
        }
        __syncthreads();
        S_split = *s_split;
        __syncthreads();                            // s_red reuse below
    }
    int cnt = 0;
    for (int s = lo; s < hi; ++s) {
        const int L = priv_len(p, s, false), pts = s >= S_split ? PTs : PT;
        cnt += max(1, (L + pts - 1) / pts) * p.Hkv;
    }
    int inc = cnt;                                  // inclusive scan over the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_red[warp] = inc;
    __syncthreads();
    int base = inc - cnt;
    for (int w = 0; w < warp; ++w) base += static_cast<int>(s_red[w]);
    int total_items = 0;
    for (int w = 0; w < kWarps; ++w) total_items += static_cast<int>(s_red[w]);
    for (int s = lo; s < hi; ++s) {
        const int pts = s >= S_split ? PTs : PT;
        s_start[s] = base;
        base += max(1, (priv_len(p, s, false) + pts - 1) / pts) * p.Hkv;
    }
    if (tid == 0) s_start[p.S] = total_items;
    __syncthreads();
    return Sched{PT, total_items, PTs, S_split};
}

__device__ __forceinline__ int find_seq(const int* s_start, int S, int item) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= item) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Next item for this CTA.  Dynamic: every CTA starts at blockIdx.x and then
// takes gridDim.x + (a global ticket), so CTAs that finish early keep working
// and the launch ends about one item after the average CTA.  The ticket
// counter lives in the workspace header.
__device__ __forceinline__ int next_item(const DecodeParams& p, int* s_next) {
    if (threadIdx.x == 0) *s_next = static_cast<int>(gridDim.x) + atomicAdd(p.ticket, 1);
    __syncthreads();
    const int it = *s_next;
    __syncthreads();
    return it;
}

// The last CTA to stop resets the ticket counters for the next launch.  Every
// other CTA has taken its last ticket before it counts itself out, so nothing
// reads the counters after the reset.
__device__ __forceinline__ void retire_cta(const DecodeParams& p) {
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.ticket + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            p.ticket[0] = 0;
            p.ticket[1] = 0;
            __threadfence();
        }
    }
}

// --------------------------------------------------------- item results ---

__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float x) {
    if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float*>(p.out)[idx] = x;
}

// res_m/res_l: [G] (log2-domain running max, sum); res_acc: [G][stride].
// A sequence with one partition gets its normalised output here; otherwise the
// item's partial goes to the workspace for the merge kernel.
__device__ void finish_item(const DecodeParams& p, int item, int s, int h, int nP,
                            const float* res_m, const float* res_l, const float* res_acc,
                            int stride) {
    const int tid = threadIdx.x;
    const int GD = p.G * p.D;
    if (nP == 1 && !in_group(p, s)) {
        const size_t out0 = (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G) * p.D;
        for (int idx = tid; idx < GD; idx += kThreads) {
            const int n = idx / p.D, d = idx - n * p.D;
            const float l = res_l[n];
            store_out(p, out0 + idx, l > 0.f ? res_acc[n * stride + d] * p.v_scale / l : 0.f);
        }
        return;
    }
    float* pacc = p.part_acc + static_cast<size_t>(item) * GD;
    for (int idx = tid; idx < GD; idx += kThreads) {
        const int n = idx / p.D, d = idx - n * p.D;
        pacc[idx] = res_acc[n * stride + d] * p.v_scale;
    }
    if (tid < p.G) {
        p.part_ml[(static_cast<size_t>(item) * p.G + tid) * 2 + 0] = res_m[tid];
        p.part_ml[(static_cast<size_t>(item) * p.G + tid) * 2 + 1] = res_l[tid];
    }
}

// CTA 0 publishes the schedule (PT, item count, first item of each sequence)
// for the merge kernel.
__device__ void publish_schedule(const DecodeParams& p, const Sched& sc, const int* s_start) {
    if (blockIdx.x != 0) return;
    if (threadIdx.x == 0) {
        p.sched[0] = sc.PT;
        p.ticket[2] = sc.PTs;                       // the header's two spare ints
        p.ticket[3] = sc.S_split;
        p.sched[1] = sc.total_items;
    }
    for (int i = threadIdx.x; i <= p.S; i += kThreads) p.sched[2 + i] = s_start[i];
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
struct WarpAcc {
    static constexpr int NJ = D / 32;     // 16-byte chunks per thread per row
    static constexpr int NT = D / 16;     // m-tiles of the value product
    uint4 qf[NJ];                         // Q^T B-fragments (bf16 pairs)
    float o[NT][4];                       // O^T accumulators: rows d, columns heads 2c, 2c+1
    float m0, m1, l0, l1;                 // running max / sum (log2 units), heads 2c, 2c+1
};

// Online-softmax update of one 16-token tile.  sc holds this thread's four
// scores (token rows r0 / r1 x heads 2c / 2c+1); rows at or past nvalid are
// masked.  Returns the tile's probabilities as the value product's B
// fragments: the rounded pair (bh) and the remainder (be), bf16 or (F8) f16.
template <int D, bool F8>
__device__ __forceinline__ void softmax_tile(WarpAcc<D>& a, const float (&sc)[4], int nvalid, float sl,
                                             int r0, int r1, uint32_t& bh0, uint32_t& bh1, uint32_t& be0,
                                             uint32_t& be1) {
    constexpr int NT = D / 16;
    float x0 = sc[0] * sl, x1 = sc[1] * sl, x2 = sc[2] * sl, x3 = sc[3] * sl;
    if (nvalid < 16) {                        // partly filled last tile
        if (r0 >= nvalid) x0 = x1 = -INFINITY;
        if (r1 >= nvalid) x2 = x3 = -INFINITY;
    }
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // Each head keeps a reference, not the running maximum: it is raised only
    // when a score passes it by more than 2^8 (log2 units), so the weights
    // 2^(x - ref) stay below 2^8 and the sums are rescaled only then (a lane
    // rescales 2 NT + 2 values).  A partial carries its reference in place of
    // its maximum; the log-sum-exp merges are exact for any reference.  With
    // the running maximum itself the sums were rescaled on most tiles, since
    // a warp sees only a few tiles of each item.
    const bool up0 = mx0 > a.m0 + 8.f, up1 = mx1 > a.m1 + 8.f;   // also: reference still unset
    const float mn0 = up0 ? mx0 : a.m0, mn1 = up1 ? mx1 : a.m1;
    const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
    const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
    const float p0 = pa_dev::ex2(x0 - ms0), p1 = pa_dev::ex2(x1 - ms1);
    const float p2 = pa_dev::ex2(x2 - ms0), p3 = pa_dev::ex2(x3 - ms1);
    if (__any_sync(0xffffffffu, up0 || up1)) {
        // factor 1 for a head that kept its reference; 0 for one that had none
        // (its sums are still 0)
        const float cr0 = up0 ? pa_dev::ex2(a.m0 - ms0) : 1.f;
        const float cr1 = up1 ? pa_dev::ex2(a.m1 - ms1) : 1.f;
        a.l0 *= cr0;
        a.l1 *= cr1;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            a.o[t][0] *= cr0; a.o[t][1] *= cr1;
            a.o[t][2] *= cr0; a.o[t][3] *= cr1;
        }
    }
    a.l0 += p0 + p2;
    a.l1 += p1 + p3;
    a.m0 = mn0;
    a.m1 = mn1;
    uint32_t h01, h23, e01, e23;          // probabilities as a rounded pair plus the remainder
    if constexpr (F8) {
        h01 = pa_dev::pack_f16(p0, p1);
        h23 = pa_dev::pack_f16(p2, p3);
        e01 = pa_dev::pack_f16(p0 - pa_dev::f16_lo(h01), p1 - pa_dev::f16_hi(h01));
        e23 = pa_dev::pack_f16(p2 - pa_dev::f16_lo(h23), p3 - pa_dev::f16_hi(h23));
    } else {
        h01 = pa_dev::pack_bf16(p0, p1);
        h23 = pa_dev::pack_bf16(p2, p3);
        e01 = pa_dev::pack_bf16(p0 - pa_dev::bf16_lo(h01), p1 - pa_dev::bf16_hi(h01));
        e23 = pa_dev::pack_bf16(p2 - pa_dev::bf16_lo(h23), p3 - pa_dev::bf16_hi(h23));
    }
    bh0 = pa_dev::movmatrix_trans(h01);
    bh1 = pa_dev::movmatrix_trans(h23);
    be0 = pa_dev::movmatrix_trans(e01);
    be1 = pa_dev::movmatrix_trans(e23);
}

// O^T += V^T . P^T for one tile.  pack (G <= 4): the score columns 4..7
// repeat heads 0..3, so those columns carry the probabilities' remainders
// and one MMA per m-tile takes both parts (the two halves of the sums are
// added once per item); otherwise the rounded pair and the remainder go
// through two MMAs into the same accumulators.
// afrag(t, x) fills the A fragment of m-tile t (value rows 16t..16t+15).
template <int D, bool F16, typename AFrag>
__device__ __forceinline__ void value_product(WarpAcc<D>& a, AFrag&& afrag, bool pack, uint32_t bh0,
                                              uint32_t bh1, uint32_t be0, uint32_t be1) {
    constexpr int NT = D / 16;
    auto mma = [](float (&d)[4], const uint32_t (&x)[4], uint32_t b0, uint32_t b1) {
        if constexpr (F16) pa_dev::mma_f16_16816(d, x[0], x[1], x[2], x[3], b0, b1);
        else pa_dev::mma_bf16_16816(d, x[0], x[1], x[2], x[3], b0, b1);
    };
    if (pack) {
        const bool upper = (threadIdx.x & 31) >= 16;          // columns 4..7
        const uint32_t b0 = upper ? be0 : bh0, b1 = upper ? be1 : bh1;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            uint32_t x[4];
            afrag(t, x);
            mma(a.o[t], x, b0, b1);
        }
    } else {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            uint32_t x[4];
            afrag(t, x);
            mma(a.o[t], x, bh0, bh1);
            mma(a.o[t], x, be0, be1);
        }
    }
}

// One bf16 16-token tile: scores, online-softmax update, value product.
template <int D>
__device__ __forceinline__ void tile_update(WarpAcc<D>& a, const uint4 (&k0)[D / 32],
                                            const uint4 (&k1)[D / 32], uint2 (&v0)[D / 16],
                                            uint2 (&v1)[D / 16], int nvalid, float sl, int r0,
                                            int r1, int c, bool pack) {
    constexpr int NJ = D / 32, NT = D / 16;
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};   // two chains
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        pa_dev::mma_bf16_16816(sc, k0[j].x, k1[j].x, k0[j].y, k1[j].y, a.qf[j].x, a.qf[j].y);
        pa_dev::mma_bf16_16816(sd, k0[j].z, k1[j].z, k0[j].w, k1[j].w, a.qf[j].z, a.qf[j].w);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] += sd[i];
    if (nvalid < 16) {                        // 0 * Inf is NaN: clear the values past the tile's end
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
    uint32_t bh0, bh1, be0, be1;
    softmax_tile<D, false>(a, sc, nvalid, sl, r0, r1, bh0, bh1, be0, be1);
    value_product<D, false>(
        a,
        [&](int t, uint32_t (&x)[4]) {
            x[0] = v0[t].x; x[1] = v1[t].x; x[2] = v0[t].y; x[3] = v1[t].y;
        },
        pack, bh0, bh1, be0, be1);
}

// Eight e4m3 codes (8 bytes) widened to four f16 pairs, and four to two.
__device__ __forceinline__ uint2 widen4(uint32_t c) {
    uint2 y;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(y.x), "=r"(y.y) : "r"(c));
    return y;
}
__device__ __forceinline__ uint4 widen8(uint2 c) {
    const uint2 a = widen4(c.x), b = widen4(c.y);
    return make_uint4(a.x, a.y, b.x, b.y);
}

// One 16-token tile of an fp8 pool from its raw codes: K as 8-byte pieces
// (token rows r0 / r1, 16-byte chunk j of the bf16 layout), V^T as 4-byte
// pieces (value rows 16t+g / 16t+g+8, tokens 4c..4c+3).  Each piece is
// widened to f16 pairs just before the MMA that reads it, so only a few
// widened fragments are live at once; the codes of tokens past the tile's end
// are cleared before widening (code 0 is +0).
template <int D>
__device__ __forceinline__ void tile_update_f8(WarpAcc<D>& a, const uint2 (&k0)[D / 32],
                                               const uint2 (&k1)[D / 32], uint32_t (&v0)[D / 16],
                                               uint32_t (&v1)[D / 16], int nvalid, float sl,
                                               int r0, int r1, int c, bool pack) {
    constexpr int NJ = D / 32, NT = D / 16;
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};   // two chains
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const uint4 a0 = widen8(k0[j]), a1 = widen8(k1[j]);
        pa_dev::mma_f16_16816(sc, a0.x, a1.x, a0.y, a1.y, a.qf[j].x, a.qf[j].y);
        pa_dev::mma_f16_16816(sd, a0.z, a1.z, a0.w, a1.w, a.qf[j].z, a.qf[j].w);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] += sd[i];
    if (nvalid < 16) {                        // partly filled last tile
        const int nv4 = min(max(nvalid - 4 * c, 0), 4);  // this thread's valid tokens of 4
        const uint32_t vm = nv4 >= 4 ? 0xffffffffu : (1u << (8 * nv4)) - 1u;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            v0[t] &= vm;
            v1[t] &= vm;
        }
    }
    uint32_t bh0, bh1, be0, be1;
    softmax_tile<D, true>(a, sc, nvalid, sl, r0, r1, bh0, bh1, be0, be1);
    value_product<D, true>(
        a,
        [&](int t, uint32_t (&x)[4]) {
            const uint2 a0 = widen4(v0[t]), a1 = widen4(v1[t]);
            x[0] = a0.x; x[1] = a1.x; x[2] = a0.y; x[3] = a1.y;
        },
        pack, bh0, bh1, be0, be1);
}
// Eight bf16 values re-rounded to f16 (exact for magnitudes 2^-17 .. 65504).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
    return pa_dev::pack_f16(pa_dev::bf16_lo(x), pa_dev::bf16_hi(x));
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x) {
    return make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                      bf16x2_to_f16x2(x.w));
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The warp's share of one item: blocks lb0 + warp + kWarps*i of the
// partition, each block cut into 16-token units whose K and V^T fragments are
// loaded straight from memory into registers.
//
// F8 (fp8 pool): the same fragments are read as e4m3
// codes, half the bytes (8 per K chunk, 4 per V^T row piece), and widened to
// f16 pairs in registers; the queries are re-rounded to f16 once per item.
// BS > 0: the pool's block size is known to be BS at compile time (16-token
// blocks: one 16-token tile per block, constant value-row strides).
// AHEAD (fp8): load each tile's codes one tile ahead of the tile being
// computed, for kernels whose register budget holds a second tile's codes.
template <int D, bool FUSE, bool F8 = false, int BS = 0, bool AHEAD = false>
__device__ __forceinline__ void fast_item(const DecodeParams& p, int s, int h, int tok0,
                                          int tok1, int L, float* sm_o, float* sm_m,
                                          float* sm_l) {
    constexpr int NJ = D / 32, NT = D / 16;
    constexpr int ES = F8 ? 1 : 2;        // bytes per pool element
    constexpr int OS = D + 4;             // padded row stride of the merge buffer
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int B = BS > 0 ? BS : p.B, nsub = B / 16;

    // fp8 pool, G <= 4: the score columns 4..7 repeat heads 0..3 (their
    // queries loaded twice), which lets the value product carry the
    // probabilities' remainders there (value_product): 8 instead of 16 value
    // MMAs per tile for the instruction-bound fp8 walk (long context 248 ->
    // 236 us on GB300); the bf16 walk, bound by load latency, ran 1.3 us
    // slower with it on the decode batch
    const bool pack = F8 && p.G <= 4;
    const int hq = pack ? (g & 3) : g;    // the query head of score column g
    WarpAcc<D> a;
    {
        const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                               (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G + hq) * D;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            a.qf[j] = hq < p.G ? __ldg(reinterpret_cast<const uint4*>(qrow + (4 * j + c) * 8))
                               : make_uint4(0u, 0u, 0u, 0u);
            if constexpr (F8) a.qf[j] = bf16x8_to_f16x8(a.qf[j]);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) a.o[t][0] = a.o[t][1] = a.o[t][2] = a.o[t][3] = 0.f;
    a.m0 = a.m1 = -INFINITY;
    a.l0 = a.l1 = 0.f;
    const float sl = p.scale_log2;
    const int r0 = 4 * (g >> 1) + (g & 1), r1 = r0 + 2;
    const int lb0 = tok0 / B, lb1 = (tok1 + B - 1) / B;
    const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
    const uint16_t* kpool = static_cast<const uint16_t*>(p.k);
    const uint16_t* vpool = static_cast<const uint16_t*>(p.v);
    const size_t tile_elems = static_cast<size_t>(B) * D;
    const int nblk = lb1 > lb0 + warp ? (lb1 - lb0 - warp + kWarps - 1) / kWarps : 0;

    // Fused append: the warp that reads the block holding position L-1 first
    // writes the sequence's new token there (key row, value column), then
    // reads that block through L2 so it sees its own writes.
    constexpr int VPL = D / 32;                   // value elements per lane
    const int lb_last = L > 0 ? (L - 1) / B : -1;
    const bool own_new = FUSE && lb_last >= lb0 && lb_last < lb1 &&
                         (lb_last - lb0) % kWarps == warp;
    const size_t new_row = (static_cast<size_t>(s) * p.Hkv + h) * D;
    if (own_new && lane < 2 * D * 2 / 128) {      // start the new token's rows towards L2
        const char* src = static_cast<const char*>(lane < D * 2 / 128 ? p.new_k : p.new_v) +
                          new_row * 2 + (lane % (D * 2 / 128)) * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
    }
    auto walk = [&](auto cg_tag) {
        constexpr bool CG = decltype(cg_tag)::value;
        int my_phys = -1;
        for (int i = 0; i < nblk; ++i) {
            const int lb = lb0 + warp + kWarps * i;
            if ((i & 31) == 0) {
                const int mine = lb + lane * kWarps;
                my_phys = mine < lb1 ? __ldg(table + mine) : -1;
            }
            const int phys = __shfl_sync(0xffffffffu, my_phys, i & 31);
            // start the block this warp reads kBlockPrefetch blocks from now
            // towards L2 (bulk prefetch: no registers, no shared memory)
            if (i + kBlockPrefetch < nblk && (i & 31) + kBlockPrefetch < 32) {
                const int pphys = __shfl_sync(0xffffffffu, my_phys, (i + kBlockPrefetch) & 31);
                if (lane == 0 && pphys >= 0 && pphys < p.num_blocks) {
                    const size_t ptile = (static_cast<size_t>(pphys) * p.Hkv + h) * tile_elems * ES;
                    pa_dev::prefetch_l2(static_cast<const char*>(p.k) + ptile,
                                        static_cast<uint32_t>(tile_elems * ES));
                    pa_dev::prefetch_l2(static_cast<const char*>(p.v) + ptile,
                                        static_cast<uint32_t>(tile_elems * ES));
                }
            }
            if (phys < 0 || phys >= p.num_blocks) {
                if (lane == 0) record_error(p.err, PA_ERR_BAD_BLOCK_ID);
                continue;
            }
            const size_t tile = (static_cast<size_t>(phys) * p.Hkv + h) * tile_elems;
            if (own_new && lb == lb_last) {
                const int64_t new_slot = __ldg(p.new_slots + s);
                const int off = (L - 1) - lb * B;
                if (new_slot >= 0 && new_slot != static_cast<int64_t>(phys) * B + off) {
                    if (lane == 0) record_error(p.err, PA_ERR_INVALID_ARG);   // not this sequence's slot
                } else if (new_slot >= 0) {
                    const uint16_t* ks = static_cast<const uint16_t*>(p.new_k) + new_row;
                    const uint16_t* vs = static_cast<const uint16_t*>(p.new_v) + new_row;
                    uint16_t* kw = const_cast<uint16_t*>(kpool) + tile + static_cast<size_t>(off) * D;
                    uint16_t* vw = const_cast<uint16_t*>(vpool) + tile + off;
                    if (lane < D / 8)
                        *reinterpret_cast<uint4*>(kw + lane * 8) = __ldg(reinterpret_cast<const uint4*>(ks + lane * 8));
    #pragma unroll
                    for (int e = 0; e < VPL; ++e)
                        vw[static_cast<size_t>(lane * VPL + e) * B] = __ldg(vs + lane * VPL + e);
                }
                __syncwarp();
            }
            for (int sub = 0; sub < nsub; ++sub) {
                const int nvalid = min(16, L - (lb * B + sub * 16));
                if (nvalid <= 0) break;
                const uint16_t* kt = kpool + tile + static_cast<size_t>(sub) * 16 * D;
                const uint16_t* vt = vpool + tile + sub * 16 + 4 * c;
                uint4 k0[NJ], k1[NJ];
                uint2 v0[NT], v1[NT];
                // the warp that wrote the new token loads through L2 (ld.global.cg) so
                // it sees its own writes; every other warp uses the read-only path
    #pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    k0[j] = CG ? pa_dev::ld_cg16(kt + r0 * D + (4 * j + c) * 8)
                                 : pa_dev::ld_stream16(kt + r0 * D + (4 * j + c) * 8);
                    k1[j] = CG ? pa_dev::ld_cg16(kt + r1 * D + (4 * j + c) * 8)
                                 : pa_dev::ld_stream16(kt + r1 * D + (4 * j + c) * 8);
                }
    #pragma unroll
                for (int t = 0; t < NT; ++t) {
                    v0[t] = CG ? pa_dev::ld_cg8(vt + static_cast<size_t>(16 * t + g) * B)
                                 : pa_dev::ld_stream8(vt + static_cast<size_t>(16 * t + g) * B);
                    v1[t] = CG ? pa_dev::ld_cg8(vt + static_cast<size_t>(16 * t + g + 8) * B)
                                 : pa_dev::ld_stream8(vt + static_cast<size_t>(16 * t + g + 8) * B);
                }
                tile_update<D>(a, k0, k1, v0, v1, nvalid, sl, r0, r1, c, pack);
            }
        }
    };
    // fp8 pool: the warp's 16-token tiles one after another, each tile's raw
    // codes (K: 8-byte pieces, V^T: 4-byte pieces, 32 registers) loaded, then
    // widened piece by piece just before the MMAs that read them (walk_f8
    // below).  Holding one tile's codes instead of two lets the walk fit 128
    // registers, four CTAs (16 warps) per SM: more loads in flight per SM than
    // three CTAs with a one-tile lookahead (on GB300, with the merge below,
    // 48-50 against 52 us on the decode batch, 246-250 against 251 us on long
    // context).  The mma.sync shared-prefix kernel runs two CTAs per SM, whose
    // register budget holds a second tile: it loads one tile ahead (AHEAD).
    //
    // Fused append into an fp8 pool: the warp that owns the block holding
    // position L-1 quantizes the new token's bf16 key row and value column
    // (code = e4m3(fl32(x / scale)), the arithmetic of the quantizing append)
    // and writes the codes before its first load; its tiles are then loaded
    // through L2 (ld.global.cg), so it reads its own writes.
    auto append_f8 = [&]() {
        const int phys = __ldg(table + lb_last);
        const int64_t new_slot = __ldg(p.new_slots + s);
        const int off = (L - 1) - lb_last * B;
        if (phys < 0 || phys >= p.num_blocks || new_slot < 0) return;   // the walk records a bad id
        if (new_slot != static_cast<int64_t>(phys) * B + off) {
            if (lane == 0) record_error(p.err, PA_ERR_INVALID_ARG);     // not this sequence's slot
            return;
        }
        const size_t tile = (static_cast<size_t>(phys) * p.Hkv + h) * tile_elems;
        unsigned char* kw = const_cast<unsigned char*>(static_cast<const unsigned char*>(p.k)) + tile +
                            static_cast<size_t>(off) * D;
        unsigned char* vw = const_cast<unsigned char*>(static_cast<const unsigned char*>(p.v)) + tile + off;
        const uint16_t* ks = static_cast<const uint16_t*>(p.new_k) + new_row;
        const uint16_t* vs = static_cast<const uint16_t*>(p.new_v) + new_row;
        auto bf = [](uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); };
        for (int i = lane; i < D / 2; i += 32) {
            const uint32_t kc = pa_dev::e4m3x2_from_f32(__fdiv_rn(bf(__ldg(ks + 2 * i)), p.k_scale),
                                                        __fdiv_rn(bf(__ldg(ks + 2 * i + 1)), p.k_scale));
            reinterpret_cast<uint16_t*>(kw)[i] = static_cast<uint16_t>(kc);
            const uint32_t vc = pa_dev::e4m3x2_from_f32(__fdiv_rn(bf(__ldg(vs + 2 * i)), p.v_scale),
                                                        __fdiv_rn(bf(__ldg(vs + 2 * i + 1)), p.v_scale));
            vw[static_cast<size_t>(2 * i) * B] = static_cast<unsigned char>(vc);
            vw[static_cast<size_t>(2 * i + 1) * B] = static_cast<unsigned char>(vc >> 8);
        }
    };
    auto walk_f8 = [&](auto cg_tag) {
        constexpr bool CG = decltype(cg_tag)::value;
        const unsigned char* kb = static_cast<const unsigned char*>(p.k);
        const unsigned char* vb = static_cast<const unsigned char*>(p.v);
        const int nunits = nblk * nsub;
        int my_phys = -1;
        // unit u's raw codes into (rk0, rk1, rv0, rv1); returns its valid
        // tokens (0: nothing to compute)
        auto load = [&](int u, uint2 (&rk0)[NJ], uint2 (&rk1)[NJ], uint32_t (&rv0)[NT],
                        uint32_t (&rv1)[NT]) -> int {
            const int i = u / nsub, sub = u - i * nsub;
            if (sub == 0 && (i & 31) == 0) {
                const int mine = lb0 + warp + kWarps * (i + lane);
                my_phys = mine < lb1 ? __ldg(table + mine) : -1;
            }
            const int phys = __shfl_sync(0xffffffffu, my_phys, i & 31);
            if (sub == 0 && i + kBlockPrefetch < nblk && (i & 31) + kBlockPrefetch < 32) {
                const int pphys = __shfl_sync(0xffffffffu, my_phys, (i + kBlockPrefetch) & 31);
                if (lane == 0 && pphys >= 0 && pphys < p.num_blocks) {
                    const size_t ptile = (static_cast<size_t>(pphys) * p.Hkv + h) * tile_elems;
                    pa_dev::prefetch_l2(kb + ptile, static_cast<uint32_t>(tile_elems));
                    pa_dev::prefetch_l2(vb + ptile, static_cast<uint32_t>(tile_elems));
                }
            }
            const int lb = lb0 + warp + kWarps * i;
            const int nv = min(16, L - (lb * B + sub * 16));
            if (phys < 0 || phys >= p.num_blocks) {
                if (lane == 0 && sub == 0) record_error(p.err, PA_ERR_BAD_BLOCK_ID);
                return 0;
            }
            if (nv <= 0) return 0;
            const size_t tile = (static_cast<size_t>(phys) * p.Hkv + h) * tile_elems;
            const unsigned char* kt = kb + tile + static_cast<size_t>(sub) * 16 * D;
            const unsigned char* vt = vb + tile + sub * 16 + 4 * c;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                rk0[j] = CG ? pa_dev::ld_cg8(kt + r0 * D + (4 * j + c) * 8)
                            : pa_dev::ld_stream8(kt + r0 * D + (4 * j + c) * 8);
                rk1[j] = CG ? pa_dev::ld_cg8(kt + r1 * D + (4 * j + c) * 8)
                            : pa_dev::ld_stream8(kt + r1 * D + (4 * j + c) * 8);
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                rv0[t] = CG ? pa_dev::ld_cg4(vt + static_cast<size_t>(16 * t + g) * B)
                            : pa_dev::ld_stream4(vt + static_cast<size_t>(16 * t + g) * B);
                rv1[t] = CG ? pa_dev::ld_cg4(vt + static_cast<size_t>(16 * t + g + 8) * B)
                            : pa_dev::ld_stream4(vt + static_cast<size_t>(16 * t + g + 8) * B);
            }
            return nv;
        };
        uint2 ak0[NJ], ak1[NJ];
        uint32_t av0[NT], av1[NT];
        if constexpr (AHEAD) {
            // the next tile's codes load while the current tile is computed
            int na = nunits > 0 ? load(0, ak0, ak1, av0, av1) : 0;
            for (int u = 0; u < nunits; ++u) {
                uint2 bk0[NJ], bk1[NJ];
                uint32_t bv0[NT], bv1[NT];
#pragma unroll
                for (int j = 0; j < NJ; ++j) { bk0[j] = ak0[j]; bk1[j] = ak1[j]; }
#pragma unroll
                for (int t = 0; t < NT; ++t) { bv0[t] = av0[t]; bv1[t] = av1[t]; }
                const int nb = na;
                na = u + 1 < nunits ? load(u + 1, ak0, ak1, av0, av1) : 0;
                if (nb > 0) tile_update_f8<D>(a, bk0, bk1, bv0, bv1, nb, sl, r0, r1, c, pack);
            }
        } else {
            for (int u = 0; u < nunits; ++u) {   // one tile's codes at a time (see above)
                const int na = load(u, ak0, ak1, av0, av1);
                if (na > 0) tile_update_f8<D>(a, ak0, ak1, av0, av1, na, sl, r0, r1, c, pack);
            }
        }
    };
    if constexpr (F8) {
        // with a fused append every warp of the kernel loads through L2 (one
        // walk compiled instead of two: the fp8 walk has no registers to spare)
        if (own_new) {
            append_f8();
            __syncwarp();                         // the codes are written before any lane loads them
        }
        walk_f8(std::integral_constant<bool, FUSE>{});
    } else {
        // only the warp that writes the new token needs loads that see it
        if (own_new) walk(std::true_type{});
        else walk(std::false_type{});
    }
    float l0 = a.l0, l1 = a.l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (pack) {
        // the sums of the remainders (columns 4..7, lanes c + 2) join those of
        // the rounded pairs (columns 0..3)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) a.o[t][i] += __shfl_down_sync(0xffffffffu, a.o[t][i], 2);
    }
    float* mo = sm_o + warp * 8 * OS;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        mo[(2 * c) * OS + 16 * t + g] = a.o[t][0];
        mo[(2 * c + 1) * OS + 16 * t + g] = a.o[t][1];
        mo[(2 * c) * OS + 16 * t + g + 8] = a.o[t][2];
        mo[(2 * c + 1) * OS + 16 * t + g + 8] = a.o[t][3];
    }
    if (g == 0) {
        sm_m[warp * 8 + 2 * c] = a.m0;
        sm_m[warp * 8 + 2 * c + 1] = a.m1;
        sm_l[warp * 8 + 2 * c] = l0;
        sm_l[warp * 8 + 2 * c + 1] = l1;
    }
}

// ------------------------------------------------- shared-prefix item ---
//
// One item = (group, KV head, tile of members, chunk of the shared span).  The
// CTA's 4 warps each own 16 query rows (row r = member r / G, head r % G of
// the tile); the chunk's 16-token K and V^T tiles are staged once in shared
// memory (cp.async, double-buffered, all threads copying) and read by every
// warp, so each shared block is read from memory once per item for up to 64
// queries instead of once per query.  Per 16-token tile and warp:
//   S[16 rows x 16 tokens] = Q[16 x D] . K^T   (2 n-tiles x D/16 k-steps)
//   O[16 x D] += P[16 x 16] . V[16 x D]         (D/8 n-tiles, P as bf16 hi+lo)
// with the same token permutation and d-chunk split as the private path, so
// K and V^T fragments are read with 16-byte / 8-byte loads.  The item's
// (acc, max, sum) per (member, head) go to the shared-partial slots.
//
// F8 (fp8 pool): the staged tiles hold e4m3 codes (half the bytes; key rows
// with 16-byte chunk c of row r at c ^ (r & 7)), widened to f16 pairs as each
// fragment is read; the queries are re-rounded to f16, the products are f16
// mma.sync, P enters as an f16 pair, and v_scale multiplies the partial sums.
template <int D, bool F8 = false>
__device__ void shared_item(const DecodeParams& p, int grp, int h, int tile, int chunk,
                            unsigned char* stage_mem) {
    constexpr int NJ = D / 32, NT = D / 16, ND = D / 8;
    constexpr int ES = F8 ? 1 : 2;                  // bytes per pool element
    constexpr int UNIT = 32 * ES * D;               // bytes per staged tile pair
    constexpr int KB = 16 * ES * D;                 // K part of a pair
    constexpr int NCH = ES * D / 16;                // 16-byte chunks per key row (fp8)
    constexpr int SWZ = NCH < 8 ? NCH - 1 : 7;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gi = lane >> 2, c = lane & 3;
    const int G = p.G, B = p.B;
    const int moff = p.g_members_off[grp];
    const int M = p.g_members_off[grp + 1] - moff;
    const int m0 = tile * p.members_per_tile, m1 = min(M, m0 + p.members_per_tile);
    const int shared_tok = p.g_shared_tokens[grp];
    const int t0 = chunk * p.chunk_tokens, t1 = min(shared_tok, t0 + p.chunk_tokens);
    const int nunits = (t1 - t0) / 16;
    const int nC = p.g_nchunks[grp];

    // every member must have these leading blocks in its context
    if (chunk == 0 && tid < m1 - m0 && seq_len(p, p.g_members[moff + m0 + tid], false) < shared_tok)
        record_error(p.err, PA_ERR_INVALID_ARG);
    static_assert(kThreads >= 64, "one thread per member of a tile");

    // query rows of this warp
    const int rA = warp * 16 + gi, rB = rA + 8;
    const int memA = m0 + rA / G, memB = m0 + rB / G;
    const bool okA = memA < m1, okB = memB < m1;
    uint4 qa[NJ], qb[NJ];
    {
        const uint16_t* q = static_cast<const uint16_t*>(p.q);
        const uint16_t* rowA = okA ? q + (static_cast<size_t>(p.g_members[moff + memA]) * p.Hq +
                                          static_cast<size_t>(h) * G + rA % G) * D : nullptr;
        const uint16_t* rowB = okB ? q + (static_cast<size_t>(p.g_members[moff + memB]) * p.Hq +
                                          static_cast<size_t>(h) * G + rB % G) * D : nullptr;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            qa[j] = okA ? __ldg(reinterpret_cast<const uint4*>(rowA + (4 * j + c) * 8)) : make_uint4(0u, 0u, 0u, 0u);
            qb[j] = okB ? __ldg(reinterpret_cast<const uint4*>(rowB + (4 * j + c) * 8)) : make_uint4(0u, 0u, 0u, 0u);
            if constexpr (F8) {
                qa[j] = bf16x8_to_f16x8(qa[j]);
                qb[j] = bf16x8_to_f16x8(qb[j]);
            }
        }
    }
    float o[ND][4];
#pragma unroll
    for (int t = 0; t < ND; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb_ = 0.f;
    const float sl = p.scale_log2;
    const int r0 = 4 * (gi >> 1) + (gi & 1), r1 = r0 + 2;

    const int32_t* table = p.tables + static_cast<size_t>(p.g_members[moff]) * p.max_blocks;
    const char* kpool = static_cast<const char*>(p.k);
    const char* vpool = static_cast<const char*>(p.v);
    const size_t tile_bytes = static_cast<size_t>(B) * D * ES;
    const uint32_t stage_s = static_cast<uint32_t>(__cvta_generic_to_shared(stage_mem));
    constexpr int NS = kSharedStages, CH = kSharedUnitsPerSync;
    unsigned valid = 0;
    // the chunk's block ids, one per lane (a chunk spans at most 32 blocks)
    const int lbc = t0 / B, nbc = (t1 - t0) / B;
    const int chunk_phys = lane < nbc ? __ldg(table + lbc + lane) : -1;
    auto issue = [&](int u) {
        const int tok = t0 + u * 16, lb = tok / B, sub = (tok - lb * B) / 16;
        const int phys = __shfl_sync(0xffffffffu, chunk_phys, lb - lbc);
        const int st = u % NS;
        valid &= ~(1u << st);
        (void)sub;
        if (phys < 0 || phys >= p.num_blocks) {
            if (tid == 0) record_error(p.err, PA_ERR_BAD_BLOCK_ID);
        } else {
            const size_t tl = (static_cast<size_t>(phys) * p.Hkv + h) * tile_bytes;
            const char* kg = kpool + tl + static_cast<size_t>(sub) * 16 * D * ES;
            const char* vg = vpool + tl + sub * 16 * ES;
            const uint32_t ks = stage_s + st * UNIT, vs = ks + KB;
            if constexpr (F8) {
                for (int q = tid; q < 16 * NCH; q += kThreads) {     // K: 16 rows x D/16 chunks
                    const int r = q / NCH, ch = q - r * NCH;
                    cp_async16(ks + r * D + ((ch ^ (r & SWZ)) << 4), kg + r * D + ch * 16);
                }
                for (int d = tid; d < D; d += kThreads)              // V^T: D rows of 16 codes
                    cp_async16(vs + d * 16, vg + static_cast<size_t>(d) * B);
            } else {
                for (int q = tid; q < 2 * D; q += kThreads) {
                    const int r = q / (D / 8), ch = q - r * (D / 8);
                    cp_async16(ks + r * (2 * D) + ((ch ^ ((r & 1) << 2)) << 4), kg + r * D * 2 + ch * 16);
                }
                for (int q = tid; q < 2 * D; q += kThreads) {
                    const int d = q >> 1, half = q & 1;
                    cp_async16(vs + d * 32 + half * 16, vg + static_cast<size_t>(d) * B * 2 + half * 16);
                }
            }
            valid |= 1u << st;
        }
        cp_async_commit();
    };
    // NS stages; each step consumes CH units after one barrier, while the
    // copies of the next NS - CH units are in flight.
    for (int u = 0; u < NS - CH; ++u) {
        if (u < nunits) issue(u);
        else cp_async_commit();
    }
    // every member's table must hold the same blocks here (checked once per
    // item while the first copies are in flight)
    for (int e = tid; e < (m1 - m0) * nbc; e += kThreads) {
        const int mi = e / nbc, bi = e - mi * nbc;
        const int32_t* mt = p.tables + static_cast<size_t>(p.g_members[moff + m0 + mi]) * p.max_blocks;
        if (__ldg(mt + lbc + bi) != __ldg(table + lbc + bi)) record_error(p.err, PA_ERR_INVALID_ARG);
    }
    for (int u0 = 0; u0 < nunits; u0 += CH) {
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            if (u0 + NS - CH + k < nunits) issue(u0 + NS - CH + k);
            else cp_async_commit();
        }
        cp_async_wait<NS - CH>();
        __syncthreads();
      for (int u = u0; u < min(nunits, u0 + CH); u += 2) {
        // two 16-token units form one 32-token tile: 4 token n-tiles
        const bool v0ok = (valid >> (u % NS)) & 1u;
        const bool v1ok = u + 1 < nunits && ((valid >> ((u + 1) % NS)) & 1u);
        float sA[4][4], sB[4][4];                   // [n-tile][frag], even / odd k-step chains
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) sA[nt][i] = sB[nt][i] = 0.f;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            if (!(w == 0 ? v0ok : v1ok)) continue;
            const unsigned char* ks = stage_mem + ((u + w) % NS) * UNIT;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int ch = 4 * j + c;
                if constexpr (F8) {
                    const uint4 ka = widen8(*reinterpret_cast<const uint2*>(
                        ks + r0 * D + (((ch >> 1) ^ (r0 & SWZ)) << 4) + (ch & 1) * 8));
                    const uint4 kb = widen8(*reinterpret_cast<const uint2*>(
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
        // rows gi ([0], [1]) and gi + 8 ([2], [3]) of each n-tile
        float xa[8], xb[8];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const bool ok = (nt < 2) ? v0ok : v1ok;
            xa[2 * nt] = ok ? (sA[nt][0] + sB[nt][0]) * sl : -INFINITY;
            xa[2 * nt + 1] = ok ? (sA[nt][1] + sB[nt][1]) * sl : -INFINITY;
            xb[2 * nt] = ok ? (sA[nt][2] + sB[nt][2]) * sl : -INFINITY;
            xb[2 * nt + 1] = ok ? (sA[nt][3] + sB[nt][3]) * sl : -INFINITY;
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
        lb_ = lb_ * crb + sumb;
        ma = na;
        mb = nb;
        // A fragments of P for the two 16-token k-steps (high and low parts:
        // bf16, or f16 for the f16 products of an fp8 pool)
        uint32_t ah[2][4], al[2][4];
        auto pk = [](float x, float y) { return F8 ? pa_dev::pack_f16(x, y) : pa_dev::pack_bf16(x, y); };
        auto lo16 = [](uint32_t v) { return F8 ? pa_dev::f16_lo(v) : pa_dev::bf16_lo(v); };
        auto hi16 = [](uint32_t v) { return F8 ? pa_dev::f16_hi(v) : pa_dev::bf16_hi(v); };
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const int n0 = 2 * w, n1 = 2 * w + 1;
            ah[w][0] = pk(pa[2 * n0], pa[2 * n0 + 1]);
            ah[w][1] = pk(pb[2 * n0], pb[2 * n0 + 1]);
            ah[w][2] = pk(pa[2 * n1], pa[2 * n1 + 1]);
            ah[w][3] = pk(pb[2 * n1], pb[2 * n1 + 1]);
            al[w][0] = pk(pa[2 * n0] - lo16(ah[w][0]), pa[2 * n0 + 1] - hi16(ah[w][0]));
            al[w][1] = pk(pb[2 * n0] - lo16(ah[w][1]), pb[2 * n0 + 1] - hi16(ah[w][1]));
            al[w][2] = pk(pa[2 * n1] - lo16(ah[w][2]), pa[2 * n1 + 1] - hi16(ah[w][2]));
            al[w][3] = pk(pb[2 * n1] - lo16(ah[w][3]), pb[2 * n1 + 1] - hi16(ah[w][3]));
        }
#pragma unroll
        for (int t = 0; t < ND; ++t) {
            o[t][0] *= cra; o[t][1] *= cra; o[t][2] *= crb; o[t][3] *= crb;
        }
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            if (!(w == 0 ? v0ok : v1ok)) continue;
            const unsigned char* vs = stage_mem + ((u + w) % NS) * UNIT + KB;
#pragma unroll
            for (int t = 0; t < ND; ++t) {
                if constexpr (F8) {
                    const uint2 v = widen4(*reinterpret_cast<const uint32_t*>(vs + (8 * t + gi) * 16 + 4 * c));
                    pa_dev::mma_f16_16816(o[t], ah[w][0], ah[w][1], ah[w][2], ah[w][3], v.x, v.y);
                    pa_dev::mma_f16_16816(o[t], al[w][0], al[w][1], al[w][2], al[w][3], v.x, v.y);
                } else {
                    const uint2 v = *reinterpret_cast<const uint2*>(vs + (8 * t + gi) * 32 + 8 * c);
                    pa_dev::mma_bf16_16816(o[t], ah[w][0], ah[w][1], ah[w][2], ah[w][3], v.x, v.y);
                    pa_dev::mma_bf16_16816(o[t], al[w][0], al[w][1], al[w][2], al[w][3], v.x, v.y);
                }
            }
        }
      }
        __syncthreads();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb_ += __shfl_xor_sync(0xffffffffu, lb_, off);
    }
    const int GD = G * D;
    auto write_row = [&](int mem, int n, int which, float m, float l) {
        const size_t slot = (static_cast<size_t>(p.g_spart_base[grp]) + static_cast<size_t>(mem) * nC + chunk) * p.Hkv + h;
        float* acc = p.spart_acc + slot * GD + static_cast<size_t>(n) * D;
#pragma unroll
        for (int t = 0; t < ND; ++t)
            *reinterpret_cast<float2*>(acc + 8 * t + 2 * c) =
                make_float2(o[t][which] * p.v_scale, o[t][which + 1] * p.v_scale);
        if (c == 0) {
            p.spart_ml[(slot * G + n) * 2] = m;
            p.spart_ml[(slot * G + n) * 2 + 1] = l;
        }
    };
    if (okA) write_row(memA, rA % G, 0, ma, la);
    if (okB) write_row(memB, rB % G, 2, mb, lb_);
    __syncthreads();                                // the stages are reused by the next item
}

// Bytes at the front of the fast kernel's shared memory: the warps' merge
// buffer, which shared-prefix items (mma.sync form) reuse for their staged tiles.
__host__ __device__ constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }
__host__ __device__ constexpr size_t fast_front_bytes(int D, bool shared) {
    return cmax(static_cast<size_t>(kWarps) * 8 * (D + 4) * 4,
                shared ? static_cast<size_t>(kSharedStages) * 64 * D : 0);
}


template <int D, bool SHARED, bool FUSE, bool F8 = false>
__global__ void __launch_bounds__(kThreads, SHARED || (F8 && D > 128) ? 2 : (F8 ? kMinCtasF8 : kMinCtas))
decode_fast_kernel(const DecodeParams p) {
    constexpr int OS = D + 4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // [merge buffer | shared-prefix stages][m, l, ...][s_start]
    unsigned char* ring = smem_raw;
    float* sm_o = reinterpret_cast<float*>(smem_raw);        // [kWarps][8][OS]
    float* sm_m = reinterpret_cast<float*>(smem_raw + fast_front_bytes(D, SHARED));  // [kWarps][8]
    float* sm_l = sm_m + kWarps * 8;                          // [kWarps][8]
    float* res_m = sm_l + kWarps * 8;                         // [8]
    float* res_l = res_m + 8;                                 // [8]
    long long* s_red = reinterpret_cast<long long*>(res_l + 8);   // [kWarps]
    int* s_flag = reinterpret_cast<int*>(s_red + kWarps);
    int* s_start = s_flag + 4;                                // [S + 1]

    if (!p.defer_wait) pa_dev::wait_prior_grid();
    const Sched sc = build_schedule(p, s_start, s_red);
    publish_schedule(p, sc, s_start);
    const int n_sh = SHARED ? p.n_shared_items : 0;
    for (int item = blockIdx.x; item < n_sh + sc.total_items;) {
        if (SHARED && item < n_sh) {
            const int k = item / p.Hkv, hh = item - k * p.Hkv;
            shared_item<D, F8>(p, p.sh_items[4 * k], hh, p.sh_items[4 * k + 1], p.sh_items[4 * k + 2],
                               ring);
            item = next_item(p, s_flag + 1);
            continue;
        }
        const int pitem = item - n_sh;
        const int s = find_seq(s_start, p.S, pitem);
        const int local = pitem - s_start[s];
        const int part = local / p.Hkv, h = local - part * p.Hkv;
        const int L = seq_len(p, s, false);
        const int start = priv_start(p, s);
        const int PTq = sc.pt(s);
        const int nP = max(1, (max(0, L - start) + PTq - 1) / PTq);
        const int tok0 = start + part * PTq, tok1 = min(L, tok0 + PTq);
        // the compile-time 16-token walk pays off for fp8 codes (13 % fewer
        // instructions, 5 % faster); the bf16 walk, bound by load latency, ran
        // 1.5 us slower with it on the decode batch (measured on GB300)
        if (F8 && p.B == 16)
            fast_item<D, FUSE, F8, 16, SHARED && D <= 128>(p, s, h, tok0, tok1, L, sm_o, sm_m, sm_l);
        else
            fast_item<D, FUSE, F8>(p, s, h, tok0, tok1, L, sm_o, sm_m, sm_l);
        // the next item's ticket, taken as soon as warp 0 is done with this
        // item's blocks: its round trip overlaps the merge of the warps below
        // (62.2 against 63.0 us on the decode batch, measured on GB300)
        int ticket = 0;
        if (threadIdx.x == 0) ticket = atomicAdd(p.ticket, 1);
        __syncthreads();
        // merge the warps' softmax states: first, per head n, the weight of
        // each warp's sums (2^(m_w - M), written over sm_m) and the combined
        // (M, l); then every thread combines its (head, column) elements and
        // writes them out: the normalised output row when the sequence has one
        // partition, else the item's partial for the merge kernel
        if (threadIdx.x < p.G) {
            const int n = threadIdx.x;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 8 + n]);
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = M != -INFINITY ? pa_dev::ex2(sm_m[w * 8 + n] - M) : 0.f;
                l += f * sm_l[w * 8 + n];
                sm_m[w * 8 + n] = f;
            }
            res_m[n] = M;
            res_l[n] = l;
        }
        __syncthreads();
        const bool single = nP == 1 && !in_group(p, s);
        const size_t dst0 = single ? (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G) * D
                                   : static_cast<size_t>(pitem) * p.G * D;
        for (int idx = threadIdx.x; idx < p.G * D; idx += kThreads) {
            const int n = idx / D, d = idx - n * D;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += sm_m[w * 8 + n] * sm_o[(w * 8 + n) * OS + d];
            if (single) {
                const float l = res_l[n];
                store_out(p, dst0 + idx, l > 0.f ? acc * p.v_scale / l : 0.f);
            } else {
                p.part_acc[dst0 + idx] = acc * p.v_scale;
            }
        }
        if (!single && threadIdx.x < p.G) {
            p.part_ml[(static_cast<size_t>(pitem) * p.G + threadIdx.x) * 2 + 0] = res_m[threadIdx.x];
            p.part_ml[(static_cast<size_t>(pitem) * p.G + threadIdx.x) * 2 + 1] = res_l[threadIdx.x];
        }
        if (threadIdx.x == 0) s_flag[1] = static_cast<int>(gridDim.x) + ticket;
        __syncthreads();
        item = s_flag[1];
        // s_flag[1] is written again only after the next item's first barrier
    }
    if (p.defer_wait) pa_dev::wait_prior_grid();        // the shared-prefix kernel is done too
    pa_dev::allow_next_grid();
    retire_cta(p);
}

// ------------------------------------------------ fp32 CUDA-core item ---

template <typename E>
__device__ __forceinline__ float load_elem(const E* base, size_t i);
template <>
__device__ __forceinline__ float load_elem<uint8_t>(const uint8_t* base, size_t i) {   // e4m3 code
    return pa_dev::f16_lo(pa_dev::e4m3x2_to_f16x2(__ldg(base + i)));
}
template <>
__device__ __forceinline__ float load_elem<float>(const float* base, size_t i) {
    return __ldg(base + i);
}
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t* base, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(base + i)) << 16);
}

// Items of at most pt_fixed tokens.  Shared memory: q [G][D], scores/probs
// [G][PT], result [G][D+4].  QE: query element type; E: pool element type
// (an fp8 pool's codes are read as their e4m3 values; its scales are folded
// into scale_log2 and v_scale).
template <typename QE, typename E>
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
    const QE* q = static_cast<const QE*>(p.q);
    const E* kp = static_cast<const E*>(p.k);
    const E* vp = static_cast<const E*>(p.v);
    pa_dev::wait_prior_grid();
    const Sched sched = build_schedule(p, s_start, s_red);
    publish_schedule(p, sched, s_start);
    for (int item = blockIdx.x; item < sched.total_items; item = next_item(p, s_flag + 1)) {
        const int s = find_seq(s_start, p.S, item);
        const int local = item - s_start[s];
        const int part = local / p.Hkv, h = local - part * p.Hkv;
        const int L = seq_len(p, s, false);
        const int PTq = sched.pt(s);
        const int nP = max(1, (L + PTq - 1) / PTq);
        const int tok0 = part * PTq, nt = max(0, min(L, tok0 + PTq) - tok0);
        const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
        for (int i = tid; i < p.G * p.D; i += kThreads)
            qs[i] = load_elem<QE>(q, (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G) * p.D + i);
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
        finish_item(p, item, s, h, nP, res_m, res_l, res, OS);
        __syncthreads();
    }
    pa_dev::allow_next_grid();
    retire_cta(p);
}

// --------------------------------------------------------------- merge ---
//
// One CTA per (sequence, KV head) with more than one partition: combine the
// partitions' (acc, max, sum) by log-sum-exp,
//   M = max_q m_q,  L = sum_q l_q 2^(m_q - M),  out = sum_q acc_q 2^(m_q - M) / L.
// Launched as a programmatic dependent of the split kernel: it may start while
// the split kernel drains and waits (griddepcontrol.wait) for it to finish.
template <bool WIDE>
__global__ void __launch_bounds__(WIDE ? kMergeThreads : kThreads, WIDE ? 2 : 1)
decode_merge_kernel(const DecodeParams p) {
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();
    const int s = blockIdx.x / p.Hkv, h = blockIdx.x - s * p.Hkv;
    const int PT = s >= p.ticket[3] ? p.ticket[2] : p.sched[0];     // this sequence's partition
    const int nP = max(1, (priv_len(p, s, false) + PT - 1) / PT);
    const int grp = p.seq_group ? p.seq_group[s] : -1;
    if (nP == 1 && grp < 0) return;                        // written by the split kernel
    const int item0 = p.sched[2 + s] + h;                   // item of partition q: item0 + q*Hkv
    // the sequence's shared-span partials (one per chunk of its group)
    const int nC = grp >= 0 ? p.g_nchunks[grp] : 0;
    const size_t slot0 = grp >= 0 ? (static_cast<size_t>(p.g_spart_base[grp]) +
                                     static_cast<size_t>(p.seq_member[s]) * nC) * p.Hkv + h
                                  : 0;
    const int nAll = nP + nC;
    const int GD = p.G * p.D;
    // partial q < nP: private item; q >= nP: shared chunk q - nP
    auto part = [&](int q) -> size_t {
        return q < nP ? static_cast<size_t>(item0) + static_cast<size_t>(q) * p.Hkv
                      : slot0 + static_cast<size_t>(q - nP) * p.Hkv;
    };
    // Each thread owns 4 consecutive elements of one head (D % 4 == 0).  The
    // CTA's threads form R groups of nqt threads; group r folds partials r,
    // r + R, ... by an online log-sum-exp, loading a batch of kBatch partials
    // (their (max, sum) and its 4 values) at once so that a batch costs one
    // memory latency; the groups' states then combine through shared memory.
    // WIDE (many partials per (sequence, head); long contexts: ~30):
    // kMergeThreads threads, whose groups shorten each thread's chain of
    // batches R-fold; otherwise kThreads threads, one group.
    constexpr int kBatch = WIDE ? 4 : 8;
    constexpr int kT = WIDE ? kMergeThreads : kThreads;
    __shared__ float4 red_acc[WIDE ? kMergeThreads : 1];
    __shared__ float2 red_ml[WIDE ? kMergeThreads : 1];
    const int nq = GD / 4;                                  // element quads of the (sequence, head)
    const int nqt = min(nq, kT);                            // threads per group
    const int R = WIDE ? kT / nqt : 1;                      // groups (the narrow form: one)
    const int r = static_cast<int>(threadIdx.x) / nqt, qd = static_cast<int>(threadIdx.x) - r * nqt;
    const size_t out0 = (static_cast<size_t>(s) * p.Hq + static_cast<size_t>(h) * p.G) * p.D;
    for (int quad0 = 0; quad0 < nq; quad0 += nqt) {
        const int quad = quad0 + qd;
        const bool mine = r < R && quad < nq;
        float M = -INFINITY, L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mine) {
            const int e = quad * 4, n = e / p.D;
            for (int q0 = r; q0 < nAll; q0 += kBatch * R) {
                float2 ml[kBatch];
                float4 x[kBatch];
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int q = q0 + k * R;
                    ml[k] = make_float2(-INFINITY, 0.f);
                    x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (q < nAll) {
                        const size_t it = part(q);
                        const bool pr = q < nP;
                        ml[k] = __ldcg(reinterpret_cast<const float2*>((pr ? p.part_ml : p.spart_ml) + (it * p.G + n) * 2));
                        x[k] = __ldcg(reinterpret_cast<const float4*>((pr ? p.part_acc : p.spart_acc) + it * GD + e));
                    }
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    if (ml[k].x == -INFINITY) continue;     // absent, or a partial that saw nothing
                    const float nm = fmaxf(M, ml[k].x);
                    const float fo = M == -INFINITY ? 0.f : pa_dev::ex2(M - nm);
                    const float fn = pa_dev::ex2(ml[k].x - nm);
                    L = L * fo + ml[k].y * fn;
                    acc.x = acc.x * fo + x[k].x * fn;
                    acc.y = acc.y * fo + x[k].y * fn;
                    acc.z = acc.z * fo + x[k].z * fn;
                    acc.w = acc.w * fo + x[k].w * fn;
                    M = nm;
                }
            }
        }
        if (WIDE && R > 1) {
            red_acc[threadIdx.x] = acc;
            red_ml[threadIdx.x] = make_float2(M, L);
            __syncthreads();
            if (r == 0 && mine) {
                for (int g2 = 1; g2 < R; ++g2) {
                    const float2 o = red_ml[g2 * nqt + qd];
                    if (o.x == -INFINITY) continue;
                    const float4 y = red_acc[g2 * nqt + qd];
                    const float nm = fmaxf(M, o.x);
                    const float fo = M == -INFINITY ? 0.f : pa_dev::ex2(M - nm);
                    const float fn = pa_dev::ex2(o.x - nm);
                    L = L * fo + o.y * fn;
                    acc.x = acc.x * fo + y.x * fn;
                    acc.y = acc.y * fo + y.y * fn;
                    acc.z = acc.z * fo + y.z * fn;
                    acc.w = acc.w * fo + y.w * fn;
                    M = nm;
                }
            }
            __syncthreads();                                // red_* reuse by the next quads
        }
        if (r == 0 && mine) {
            const int e = quad * 4;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            store_out(p, out0 + e + 0, acc.x * inv);
            store_out(p, out0 + e + 1, acc.y * inv);
            store_out(p, out0 + e + 2, acc.z * inv);
            store_out(p, out0 + e + 3, acc.w * inv);
        }
    }
}

size_t fast_smem(int D, int S, bool shared) {
    return fast_front_bytes(D, shared) + static_cast<size_t>(kWarps * 16 + 16) * sizeof(float) +
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

int plan_decode(pa_pool* pool, int S, int Hq, int max_blocks, DecodePlan* plan) {
    const int Hkv = pool->kv_heads, D = pool->head_dim, B = pool->block_size;
    const int G = Hq / Hkv;
    const bool fp8 = pool->dtype == PA_FP8E4M3;
    const bool tc_shape = (D == 64 || D == 128 || D == 256) && B % 16 == 0 && G <= 8;
    const bool fast = tc_shape && (pool->dtype == PA_BF16 || fp8);
    plan->fast = fast;
    plan->pool = pool;
    plan->bf16 = pool->dtype == PA_BF16;
    plan->fp8 = fp8;
    plan->threads = kThreads;
    int occ = 0;
    if (fast) {
        plan->smem = fast_smem(D, S, plan->shared && !plan->tc);
        plan->pt_fixed = 0;
        plan->pt_min = std::max(B, (64 + B - 1) / B * B);
        // Batches of more sequences than SMs are mostly one item per sequence,
        // of uneven sizes; partitions of at most kPtMax tokens then shorten the
        // launch's tail (measured on GB300: mixed lengths 473 -> 455 us; a few
        // long sequences, already many equal items, are better uncapped).
        // The pool's PA_OPT_PARTITION_CAP option overrides the choice (0: no cap).
        const int pt_max = pool->opt_partition_cap >= 0 ? pool->opt_partition_cap
                                                         : (S > pool->num_sms ? kPtMax : 0);
        plan->pt_max = pt_max > 0 ? std::max(plan->pt_min, pt_max / B * B) : 0;
        if (plan->shared && !plan->tc && fp8) {
            if (D == 64) occ = occupancy(decode_fast_kernel<64, true, false, true>, plan->smem);
            else if (D == 128) occ = occupancy(decode_fast_kernel<128, true, false, true>, plan->smem);
            else occ = occupancy(decode_fast_kernel<256, true, false, true>, plan->smem);
        } else if (plan->shared && !plan->tc) {
            if (D == 64) occ = occupancy(decode_fast_kernel<64, true, false>, plan->smem);
            else if (D == 128) occ = occupancy(decode_fast_kernel<128, true, false>, plan->smem);
            else occ = occupancy(decode_fast_kernel<256, true, false>, plan->smem);
        } else if (fp8 && plan->fuse) {
            if (D == 64) occ = occupancy(decode_fast_kernel<64, false, true, true>, plan->smem);
            else if (D == 128) occ = occupancy(decode_fast_kernel<128, false, true, true>, plan->smem);
            else occ = occupancy(decode_fast_kernel<256, false, true, true>, plan->smem);
        } else if (fp8) {
            if (D == 64) occ = occupancy(decode_fast_kernel<64, false, false, true>, plan->smem);
            else if (D == 128) occ = occupancy(decode_fast_kernel<128, false, false, true>, plan->smem);
            else occ = occupancy(decode_fast_kernel<256, false, false, true>, plan->smem);
        } else if (plan->fuse) {
            if (D == 64) occ = occupancy(decode_fast_kernel<64, false, true>, plan->smem);
            else if (D == 128) occ = occupancy(decode_fast_kernel<128, false, true>, plan->smem);
            else occ = occupancy(decode_fast_kernel<256, false, true>, plan->smem);
        } else {
            if (D == 64) occ = occupancy(decode_fast_kernel<64, false, false>, plan->smem);
            else if (D == 128) occ = occupancy(decode_fast_kernel<128, false, false>, plan->smem);
            else occ = occupancy(decode_fast_kernel<256, false, false>, plan->smem);
        }
    } else {
        const int PT = B >= 256 ? B : (256 / B) * B;
        plan->pt_fixed = PT;
        plan->pt_min = PT;
        plan->smem = simple_smem(G, D, PT, S);
        occ = fp8 ? occupancy(decode_simple_kernel<uint16_t, uint8_t>, plan->smem)
              : pool->dtype == PA_BF16 ? occupancy(decode_simple_kernel<uint16_t, uint16_t>, plan->smem)
                                       : occupancy(decode_simple_kernel<float, float>, plan->smem);
    }
    if (occ <= 0) return PA_ERR_UNSUPPORTED;
    plan->grid = pool->num_sms * occ;
    if (fast) {
        // the mma.sync shared-prefix kernel (two CTAs per SM) keeps four items per
        // CTA (faster on the fp8 prefix batch than twelve per SM, measured on GB300)
        plan->items_target = plan->shared && !plan->tc ? plan->grid * 4 : pool->num_sms * kItemsPerSm;
        if (fp8 && !(plan->shared && !plan->tc)) {
            // fp8 pools: partitions of at least kPtSoftF8 tokens while that
            // leaves two items per SM, so that the guided tail's short
            // partitions reach kGuideMinPT in a one-wave batch (measured on
            // GB300, 64 sequences of 128-2048 tokens: 45.2 -> 41.4 us)
            plan->pt_soft = std::max(plan->pt_min, kPtSoftF8 / B * B);
            plan->items_floor = pool->num_sms * 2;
        }
        // items <= Hkv * (total / PT + S); PT >= total * Hkv / items_target keeps
        // that below min_items.  The extra items_target of room lets the
        // partition cap and the guided tail take effect; the kernel never
        // exceeds max_items.
        plan->min_items = static_cast<size_t>(plan->items_target) + static_cast<size_t>(Hkv) * S;
        plan->max_items = plan->min_items + static_cast<size_t>(plan->items_target);
    } else {
        plan->items_target = 0;
        const size_t per_seq = (static_cast<size_t>(max_blocks) * B + plan->pt_fixed - 1) / plan->pt_fixed;
        plan->max_items = static_cast<size_t>(Hkv) * S * std::max<size_t>(1, per_seq);
        plan->min_items = plan->max_items;
    }
    if (static_cast<size_t>(plan->grid) > plan->max_items)
        plan->grid = static_cast<int>(plan->max_items);
    if (fast && !(plan->shared && !plan->tc)) {
        // whole waves of one item per resident CTA, one wave per
        // kWaveBytes of cache each CTA reads
        plan->wave_items = plan->grid;
        plan->wave_tokens = static_cast<int>(kWaveBytes / (2 * static_cast<size_t>(D) * (fp8 ? 1 : 2)));
    }
    return PA_OK;
}

int launch_decode(const DecodePlan& plan, const DecodeParams& prm, cudaStream_t st) {
    DecodeParams p = prm;
    p.items_target = plan.items_target;
    p.pt_soft = plan.pt_soft;
    p.items_floor = plan.items_floor;
    p.wave_items = plan.wave_items;
    p.wave_tokens = plan.wave_tokens;
    p.pt_min = plan.pt_min;
    p.pt_max = plan.pt_max;
    p.max_items = static_cast<int>(std::min<size_t>(plan.max_items, 1u << 30));
    p.pt_fixed = plan.pt_fixed;
    const dim3 grid(plan.grid), block(plan.threads);
    cudaError_t e;
    if (plan.fast && plan.shared && plan.tc) {
        // shared items on tcgen05 first, then the private spans on the plain split kernel
        const int rc = launch_shared_tc(plan.pool, p, st);
        if (rc != PA_OK) return rc;
        DecodeParams q = p;
        q.n_shared_items = 0;
        q.defer_wait = 1;
        if (plan.fp8) {
            if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, false, false, true>, grid, block, plan.smem, st, q);
            else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, false, false, true>, grid, block, plan.smem, st, q);
            else e = launch_pdl(decode_fast_kernel<256, false, false, true>, grid, block, plan.smem, st, q);
        } else {
            if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, false, false>, grid, block, plan.smem, st, q);
            else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, false, false>, grid, block, plan.smem, st, q);
            else e = launch_pdl(decode_fast_kernel<256, false, false>, grid, block, plan.smem, st, q);
        }
    } else if (plan.fast && plan.shared && plan.fp8) {
        if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, true, false, true>, grid, block, plan.smem, st, p);
        else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, true, false, true>, grid, block, plan.smem, st, p);
        else e = launch_pdl(decode_fast_kernel<256, true, false, true>, grid, block, plan.smem, st, p);
    } else if (plan.fast && plan.shared) {
        if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, true, false>, grid, block, plan.smem, st, p);
        else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, true, false>, grid, block, plan.smem, st, p);
        else e = launch_pdl(decode_fast_kernel<256, true, false>, grid, block, plan.smem, st, p);
    } else if (plan.fast && plan.fp8 && plan.fuse) {
        if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, false, true, true>, grid, block, plan.smem, st, p);
        else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, false, true, true>, grid, block, plan.smem, st, p);
        else e = launch_pdl(decode_fast_kernel<256, false, true, true>, grid, block, plan.smem, st, p);
    } else if (plan.fast && plan.fp8) {
        if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, false, false, true>, grid, block, plan.smem, st, p);
        else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, false, false, true>, grid, block, plan.smem, st, p);
        else e = launch_pdl(decode_fast_kernel<256, false, false, true>, grid, block, plan.smem, st, p);
    } else if (plan.fast && plan.fuse) {
        if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, false, true>, grid, block, plan.smem, st, p);
        else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, false, true>, grid, block, plan.smem, st, p);
        else e = launch_pdl(decode_fast_kernel<256, false, true>, grid, block, plan.smem, st, p);
    } else if (plan.fast) {
        if (p.D == 64) e = launch_pdl(decode_fast_kernel<64, false, false>, grid, block, plan.smem, st, p);
        else if (p.D == 128) e = launch_pdl(decode_fast_kernel<128, false, false>, grid, block, plan.smem, st, p);
        else e = launch_pdl(decode_fast_kernel<256, false, false>, grid, block, plan.smem, st, p);
    } else if (plan.fp8) {
        e = launch_pdl(decode_simple_kernel<uint16_t, uint8_t>, grid, block, plan.smem, st, p);
    } else if (plan.bf16) {
        e = launch_pdl(decode_simple_kernel<uint16_t, uint16_t>, grid, block, plan.smem, st, p);
    } else {
        e = launch_pdl(decode_simple_kernel<float, float>, grid, block, plan.smem, st, p);
    }
    count_launch();
    if (e != cudaSuccess) return PA_ERR_CUDA;
    // many partials per (sequence, KV head): split each one's partials over
    // four thread groups (long context 424 -> 416 us, on an fp8 pool 238 ->
    // 229 us, on GB300)
    const dim3 mgrid(static_cast<unsigned>(p.S) * static_cast<unsigned>(p.Hkv));
    if (plan.fast && plan.items_target >= 8 * p.S * p.Hkv)
        e = launch_pdl(decode_merge_kernel<true>, mgrid, dim3(kMergeThreads), 0, st, p);
    else
        e = launch_pdl(decode_merge_kernel<false>, mgrid, dim3(kThreads), 0, st, p);
    count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
