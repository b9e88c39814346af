// Work schedule of the decode split kernels (shared by the mma.sync and the
// tcgen05 forms): every CTA derives the same list of work items, (sequence,
// KV head, partition of PT tokens), from context_lens; CTA 0 publishes it for
// the merge kernel; items are handed out by a global ticket.  Run by the first
// 128 threads of a CTA (named barrier 1), so kernels with more warps can give
// the other warps other roles.
#pragma once

#include <climits>
#include <cstdint>

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa_sched {

constexpr int kSchedThreads = 128;      // threads that build the schedule
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kGuideMinPT = 256;        // shortest partition of the guided tail, tokens

// Barrier among the kSchedThreads schedule threads only.
__device__ __forceinline__ void sched_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }


__device__ __forceinline__ int seq_len(const DecodeParams& p, int s, bool report) {
    int L = __ldg(p.lens + s);
    const int cap = p.max_blocks * p.B;
    if (L < 0 || L > cap) {
        if (report) pa_dev::record_error(p.err, PA_ERR_BAD_LENGTH);
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
static __device__ Sched build_schedule(const DecodeParams& p, int* s_start, long long* s_red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.S + kSchedThreads - 1) / kSchedThreads;
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
    sched_sync();
    long long total = 0, tbase = tinc - tok;
#pragma unroll
    for (int w = 0; w < kSchedWarps; ++w) {
        total += s_red[w];
        if (w < warp) tbase += s_red[w];
    }
    int PT, PTs;
    long long split_at = LLONG_MAX;
    if (p.pt_fixed > 0) {
        PT = PTs = p.pt_fixed;
    } else {
        long long need = (total * p.Hkv + p.items_target - 1) / p.items_target;
        need = (need + p.B - 1) / p.B * p.B;
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
        PT = static_cast<int>(max(need, static_cast<long long>(p.pt_min)));
        // Guided tail: sequences that start in the last quarter of the tokens
        // (they are the last items handed out) use partitions a quarter as long,
        // so the launch ends on short items.  Their tokens are at most a quarter
        // of the total, so items <= Hkv * (total/PT + total/(4 PTs) + S); used
        // only when that fits the workspace, and only when the short partitions
        // still hold kGuideMinPT tokens (shorter items cost more to start than
        // they save at the end: measured on GB300).
        PTs = max(p.pt_min, (PT / 4 + p.B - 1) / p.B * p.B);
        const long long bound = static_cast<long long>(p.Hkv) *
            ((total + PT - 1) / PT + (total + 4LL * PTs - 1) / (4LL * PTs) + p.S);
        if (PTs < PT && PTs >= kGuideMinPT && bound <= p.max_items) split_at = total - total / 4;
        else PTs = PT;
    }
    // first sequence starting at or after split_at (every thread of the CTA
    // has the same split_at, so the branch is uniform)
    int S_split = p.S;
    sched_sync();                                // s_red reuse
    if (split_at != LLONG_MAX) {
        int* s_split = reinterpret_cast<int*>(s_red);
        if (tid == 0) *s_split = p.S;
        sched_sync();
        long long c = tbase;
        for (int s = lo; s < hi; ++s) {
            if (c >= split_at) {
                atomicMin(s_split, s);
                break;
            }
            c += priv_len(p, s, false);
        }
        sched_sync();
        S_split = *s_split;
        sched_sync();                            // s_red reuse below
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
    sched_sync();
    int base = inc - cnt;
    for (int w = 0; w < warp; ++w) base += static_cast<int>(s_red[w]);
    int total_items = 0;
    for (int w = 0; w < kSchedWarps; ++w) total_items += static_cast<int>(s_red[w]);
    for (int s = lo; s < hi; ++s) {
        const int pts = s >= S_split ? PTs : PT;
        s_start[s] = base;
        base += max(1, (priv_len(p, s, false) + pts - 1) / pts) * p.Hkv;
    }
    if (tid == 0) s_start[p.S] = total_items;
    sched_sync();
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
    sched_sync();
    const int it = *s_next;
    sched_sync();
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

__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float x) {
    if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float*>(p.out)[idx] = x;
}

// CTA 0 publishes the schedule (PT, item count, first item of each sequence)
// for the merge kernel (called by the schedule threads).
static __device__ void publish_schedule(const DecodeParams& p, const Sched& sc, const int* s_start) {
    if (blockIdx.x != 0) return;
    if (threadIdx.x == 0) {
        p.sched[0] = sc.PT;
        p.ticket[2] = sc.PTs;                       // the header's two spare ints
        p.ticket[3] = sc.S_split;
        p.sched[1] = sc.total_items;
    }
    for (int i = threadIdx.x; i <= p.S; i += kSchedThreads) p.sched[2 + i] = s_start[i];
}

}  // namespace pa_sched
