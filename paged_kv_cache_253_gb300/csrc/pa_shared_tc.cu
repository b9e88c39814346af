// Shared-prefix decode items on the 5th-generation tensor cores (tcgen05).
//
// For a group of requests whose block tables start with the same physical
// blocks (zenaique prefix-sharing answer: requests with one prefix point at one
// copy; kgptalkie "Day 28", "Prefix Sharing Is a Natural Extension"), every
// query of every member attends to the shared span.  Stacked, those queries
// form a real dense contraction: 128 query rows (members x their G heads) of
// one KV head against the span's keys, read once per 128 rows.
//
// The shared-prefix kernel takes an item = (group, KV head, tile of 128 / G
// members, chunk of 1024 shared tokens) and walks it in 64-token steps:
//   S[128 x 64]   = Q[128 x 128] . K^T           tcgen05.mma, fp32 in TMEM
//   softmax       thread t owns query row t = TMEM lane t (tcgen05.ld), exp2 in
//                 fp32 with a reference maximum that is raised only when a row's
//                 maximum grows by more than 2^8 (then O is rescaled in TMEM)
//   O[128 x 128] += P[128 x 64] . V[64 x 128]    tcgen05.mma, fp32 in TMEM,
//                 P entering from TMEM as a high part plus a low part
// with its warps specialised: a producer (Q by cp.async, K and V^T by TMA into
// four swizzled K-major stages), a Q.K^T issuer, a P.V issuer and four softmax
// warps, handing work to each other through mbarriers with S, P and O double
// buffered in TMEM (one CTA per SM).  Each row's (acc, max, sum) goes to the
// shared-partial slot the merge kernel reads.  fp8 pools: the producer copies
// the codes and four more warps widen them to f16 (shared_tc_kernel<true>).
//
// The chunked-prefill kernel runs the same step on a (128 rows = 128 / G chunk
// tokens x G heads, KV head, sequence) item with one warpgroup: one thread
// issues the MMAs and commits them to mbarriers the others wait on, two K/V
// stages, ~99 KB of shared memory so that two CTAs share an SM, causal masks.
// Value columns that get zero weight (block slots a step did not load,
// positions past a context) are zeroed before the value product, so stale
// non-finite bits never reach it.  Every mbarrier wait is bounded: on timeout
// the kernel records PA_ERR_CUDA and the CTA stops.
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kD = 128;                  // head_dim of this path
constexpr int kRows = 128;               // M: query rows per item
constexpr int kStep = 64;                // tokens per step (N of S, K of P.V)
constexpr int kTmemCols = 256;           // S [0,64), O [64,192), P hi [192,224), P lo [224,256)
constexpr uint32_t kWaitLimit = 1u << 20;      // polls; milliseconds, far beyond any copy or MMA

// shared-memory map (offsets from a 1024-aligned base); ~99 KB, two CTAs per SM
constexpr uint32_t kQOff = 0;                            // 2 regions x [128 rows][128 B]
constexpr uint32_t kStageOff = 32768;                    // stage s: K (2 x [64][128 B]) then V^T ([128][128 B])
constexpr uint32_t kStageBytes = 32768;
constexpr uint32_t kMiscOff = kStageOff + 2 * kStageBytes;   // mbarriers, TMEM slot, table slice
constexpr int kChunkBlocks = 64;                         // shared blocks per item (1024 tokens)
constexpr uint32_t kSmemBytes = kMiscOff + 64 + 4 * kChunkBlocks + 1024;   // + alignment slack

constexpr uint32_t kIdescQK = pa_tc::idesc_bf16_f32(kRows, kStep);
constexpr uint32_t kIdescPV = pa_tc::idesc_bf16_f32(kRows, kD);

__device__ __forceinline__ float exp2_approx(float x) { return pa_dev::ex2(x); }

__device__ __forceinline__ int seq_len(const DecodeParams& p, int s) {
    const int L = __ldg(p.lens + s);
    return L < 0 ? 0 : min(L, p.max_blocks * p.B);
}

// ------------------------------------------------- shared-prefix items ---
//
// Warp roles of one CTA (224 threads; one CTA per SM, so that the split pass
// of the private suffixes runs beside it on every SM):
//   warps 0-3  softmax: thread t owns query row t, which is TMEM lane t; they
//              also check an item's sharing description and write each
//              finished item's partial rows
//   warp 4     producer: the item's Q rows by cp.async, then each 64-token
//              step's K and V^T by TMA into a ring of kWsStages stages
//   warp 5     Q.K^T issue (lane 0): S into one of two S buffers in TMEM
//   warp 6     P.V issue (lane 0): O += P.V with P read from one of two P
//              buffers in TMEM, into one of two O buffers (one per item)
// Items go to CTAs statically (item = blockIdx.x + k * gridDim.x), so every
// role walks the same items and steps without telling the others which; the
// roles hand each other work through mbarriers only.  Q.K^T(j) is issued as
// soon as the step's keys have landed and an S buffer is free, P.V(j) once the
// softmax warps have written P(j): the tensor pipe computes the next step's
// scores while the softmax warps work on this one, and the two kinds of MMA
// are issued by two threads (one thread issuing both was the step's limit).
// An item's partial rows are written while the next item's first step runs
// (its O buffer is not touched again until the item after that).
// Every mbarrier wait is bounded; a role that gives up raises a shared abort
// flag that ends the others' waits at once, records PA_ERR_CUDA, and the CTA
// drains its own copies and MMAs before it frees TMEM and exits.
constexpr int kWsThreads = 224;
constexpr int kWsThreadsF8 = 352;                        // fp8 pools: + 4 converter warps (7-10)
constexpr int kWsStages = 4;
constexpr uint32_t kWsStageOff = 32768;                  // after Q (2 x [128][128 B])
constexpr uint32_t kWsCodeOff = kWsStageOff + kWsStages * kStageBytes;   // fp8: each stage's raw codes
constexpr uint32_t kWsCodeBytes = 16384;                  // 4 blocks x (K 2 KB, then V^T 2 KB) of e4m3 codes
enum WsBar {
    kQFull, kQEmpty, kSFull0, kSFull1, kSEmpty0, kSEmpty1, kPFull0, kPFull1, kPEmpty0, kPEmpty1,
    kOFull0, kOFull1, kMmaDone, kKvFull0, kKvEmpty0 = kKvFull0 + kWsStages,
    kKvConv0 = kKvEmpty0 + kWsStages,        // fp8: the stage's codes are widened (4 converter warps)
    kQConv = kKvConv0 + kWsStages,           // fp8: the Q tile is in f16
    kNumWsBars
};
// after the stages (and, for fp8 pools, the code staging): mbarriers, then TMEM
// slot, abort flag and stage masks, then the batch index of each row's member
__host__ __device__ constexpr uint32_t ws_bar_off(bool f8) {
    return kWsCodeOff + (f8 ? kWsStages * kWsCodeBytes : 0);
}
__host__ __device__ constexpr uint32_t ws_misc_off(bool f8) { return ws_bar_off(f8) + kNumWsBars * 8; }
__host__ __device__ constexpr uint32_t ws_members_off(bool f8) { return ws_misc_off(f8) + 64; }
__host__ __device__ constexpr uint32_t ws_smem_bytes(bool f8) {
    return ws_members_off(f8) + 4 * kRows + 1024;             // + alignment slack
}
static_assert(ws_smem_bytes(true) <= 232448, "fp8 shared-prefix CTA beyond the opt-in shared memory");
constexpr uint32_t kIdescQK16 = pa_tc::idesc_f16_f32(kRows, kStep);
constexpr uint32_t kIdescPV16 = pa_tc::idesc_f16_f32(kRows, kD);

// Eight bf16 values (16 bytes) re-rounded to f16 in place (exact for
// magnitudes 2^-17 .. 65504: every such bf16 value is an f16 value).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x) {
    auto cv = [](uint32_t w) { return pa_dev::pack_f16(pa_dev::bf16_lo(w), pa_dev::bf16_hi(w)); };
    return make_uint4(cv(x.x), cv(x.y), cv(x.z), cv(x.w));
}
// Eight e4m3 codes (8 bytes, first element in the low byte) widened to f16 (exact).
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 c) {
    return make_uint4(pa_dev::e4m3x2_to_f16x2(c.x), pa_dev::e4m3x2_to_f16x2(c.x >> 16),
                      pa_dev::e4m3x2_to_f16x2(c.y), pa_dev::e4m3x2_to_f16x2(c.y >> 16));
}
// TMEM columns: S0 [0,64), S1 [64,128), O0 [128,256), O1 [256,384), then two
// P buffers of 64 columns at 384 and 448, P hi (bf16 pairs) in the first 32
// and P lo in the next 32
constexpr int kWsTmemCols = 512;

// Bounded wait on an mbarrier phase that also gives up when another role has
// raised the abort flag; a timeout raises it.
__device__ __forceinline__ bool ws_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    const uint32_t a = pa_tc::smem_u32(bar);
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 31) == 31 && *abort_flag) return false;
    }
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ void ws_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(pa_tc::smem_u32(bar)) : "memory");
}

// What every role derives from an item index.
struct WsItem {
    int grp, h, chunk, m0, m1, moff, t0, t1, nsteps, nC, lbc, nbc;
    const int32_t* table;       // the first member's table (the shared blocks)
};

__device__ __forceinline__ WsItem ws_item(const DecodeParams& p, int item) {
    WsItem it;
    const int k = item / p.Hkv;
    it.h = item - k * p.Hkv;
    it.grp = p.sh_items[4 * k];
    const int tile = p.sh_items[4 * k + 1];
    it.chunk = p.sh_items[4 * k + 2];
    it.moff = p.g_members_off[it.grp];
    const int M = p.g_members_off[it.grp + 1] - it.moff;
    it.m0 = tile * p.members_per_tile;
    it.m1 = min(M, it.m0 + p.members_per_tile);
    const int shared_tok = p.g_shared_tokens[it.grp];
    it.t0 = it.chunk * p.chunk_tokens;
    it.t1 = min(shared_tok, it.t0 + p.chunk_tokens);
    it.nsteps = (it.t1 - it.t0 + kStep - 1) / kStep;
    it.nC = p.g_nchunks[it.grp];
    it.lbc = it.t0 / p.B;
    it.nbc = (it.t1 - it.t0) / p.B;
    it.table = p.tables + static_cast<size_t>(p.g_members[it.moff]) * p.max_blocks;
    return it;
}

// The sharing description must match the tables: every member covers the
// shared span, and every member's table holds the first member's blocks on
// this item's chunk (recorded, never trapped).  The tables do not depend on
// the head, so the Hkv items of one (group, tile, chunk) split the checks
// between them: the item of head h takes every Hkv-th entry, starting at h.
// Run by the 128 softmax threads, eight table entries in flight per thread.
__device__ __forceinline__ void ws_validate(const DecodeParams& p, const WsItem& it, int t) {
    const int nm = it.m1 - it.m0, step = 128 * p.Hkv;
    if (it.chunk == 0)
        for (int mi = it.h + t * p.Hkv; mi < nm; mi += step)
            if (seq_len(p, p.g_members[it.moff + it.m0 + mi]) < p.g_shared_tokens[it.grp])
                pa_dev::record_error(p.err, PA_ERR_INVALID_ARG);
    const int n = nm * it.nbc;
    for (int e0 = it.h + t * p.Hkv; e0 < n; e0 += 8 * step) {
        int mine[8], ref[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * step;
            mine[u] = ref[u] = 0;
            if (e < n) {
                const int mi = e / it.nbc, bi = e - mi * it.nbc;
                mine[u] = __ldg(p.tables + static_cast<size_t>(p.g_members[it.moff + it.m0 + mi]) * p.max_blocks +
                                it.lbc + bi);
                ref[u] = __ldg(it.table + it.lbc + bi);
            }
        }
        bool bad = false;
#pragma unroll
        for (int u = 0; u < 8; ++u) bad |= mine[u] != ref[u];
        if (bad) pa_dev::record_error(p.err, PA_ERR_INVALID_ARG);
    }
}

// F8 (fp8 pool): the producer copies each block's raw e4m3 codes (K and V^T,
// 2 KB each per KV head) into the stage's code area; four converter warps
// widen them to f16 (exact) in the layouts the MMAs read (K: 128-byte swizzle;
// V^T: 32-byte swizzle; blocks without keys get zero values), re-round each
// item's Q tile to f16 in place, and release the stage to the MMA issuers; the
// MMAs are f16, P is an f16 pair, k_scale sits in the score factor and v_scale
// is applied to the partial sums.  kmap / vmap are unused then.
template <bool F8>
__global__ void __launch_bounds__(F8 ? kWsThreadsF8 : kWsThreads, F8 ? 1 : 2)
shared_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ unsigned char tc_raw[];
    const uint32_t raw_s = pa_tc::smem_u32(tc_raw);
    unsigned char* base = tc_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = pa_tc::smem_u32(base);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + ws_bar_off(F8));
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + ws_misc_off(F8));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + ws_misc_off(F8) + 4);
    volatile int* stage_mask = reinterpret_cast<volatile int*>(base + ws_misc_off(F8) + 8);   // [kWsStages]
    int* s_members = reinterpret_cast<int*>(base + ws_members_off(F8));   // [kRows], producer only

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();       // the private-span split kernel runs alongside
    if (tid == 0) {
        pa_tc::mbar_init(&bars[kQFull], 32);                 // the producer's 32 lanes
        pa_tc::mbar_init(&bars[kQEmpty], 1);
        pa_tc::mbar_init(&bars[kSFull0], 1);
        pa_tc::mbar_init(&bars[kSFull1], 1);
        pa_tc::mbar_init(&bars[kSEmpty0], 4);                // one arrival per softmax warp
        pa_tc::mbar_init(&bars[kSEmpty1], 4);
        pa_tc::mbar_init(&bars[kPFull0], 4);
        pa_tc::mbar_init(&bars[kPFull1], 4);
        pa_tc::mbar_init(&bars[kPEmpty0], 1);
        pa_tc::mbar_init(&bars[kPEmpty1], 1);
        pa_tc::mbar_init(&bars[kOFull0], 1);
        pa_tc::mbar_init(&bars[kOFull1], 1);
        pa_tc::mbar_init(&bars[kMmaDone], 2);                // both MMA-issuing warps
        for (int s = 0; s < kWsStages; ++s) {
            pa_tc::mbar_init(&bars[kKvFull0 + s], 1);
            pa_tc::mbar_init(&bars[kKvEmpty0 + s], 1);
            pa_tc::mbar_init(&bars[kKvConv0 + s], 4);        // one arrival per converter warp
        }
        pa_tc::mbar_init(&bars[kQConv], 4);
        *abort_flag = 0;
        pa_tc::mbar_init_fence();
    }
    if (warp == 0) pa_tc::tmem_alloc<kWsTmemCols>(tslot);
    pa_tc::fence_before_sync();
    __syncthreads();
    pa_tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tO = tmem + 128, tP = tmem + 384;     // O buffer b at tO + 128 b, P buffer b at tP + 64 b
    const int G = p.G, Hkv = p.Hkv;
    bool ok = true;

    if (warp == 4) {
        // ------------------------------------------------------ producer
        const uint16_t* qg = static_cast<const uint16_t*>(p.q);
        uint32_t kv_it = 0, fills[kWsStages] = {};
        int kk = 0;
        for (int item = blockIdx.x; ok && item < p.n_shared_items; item += gridDim.x, ++kk) {
            const WsItem it = ws_item(p, item);
            // the chunk's block ids (at most 64): lane b holds blocks b and b + 32
            auto block_id = [&](int bi) {
                int b = bi < it.nbc ? __ldg(it.table + it.lbc + bi) : -1;
                if (bi < it.nbc && (b < 0 || b >= p.num_blocks)) {
                    pa_dev::record_error(p.err, PA_ERR_BAD_BLOCK_ID);
                    b = -1;
                }
                return b;
            };
            const int tb0 = block_id(lane), tb1 = block_id(lane + 32);
            // the tile's members (batch indices), read once for the row loop below
            for (int mi = lane; mi < it.m1 - it.m0; mi += 32) s_members[mi] = p.g_members[it.moff + it.m0 + mi];
            __syncwarp();
            // Q rows, once the previous item's last Q.K^T is done with the Q tile
            if (kk > 0 && !ws_wait(&bars[kQEmpty], (kk - 1) & 1, abort_flag)) { ok = false; break; }
            for (int idx = lane; idx < kRows * 16; idx += 32) {
                const int r = idx >> 4, c16 = idx & 15;
                const int rmi = r / G, rn = r - rmi * G;
                const bool v = r < p.members_per_tile * G && it.m0 + rmi < it.m1;
                const uint16_t* src = qg + (v ? ((static_cast<size_t>(s_members[rmi]) * p.Hq +
                                                  static_cast<size_t>(it.h) * G + rn) * kD + c16 * 8)
                                              : 0);
                pa_tc::cp16(sbase + kQOff + (c16 >> 3) * 16384 + pa_tc::sw128_off(r, c16 & 7), src,
                            v ? 16u : 0u);
            }
            pa_tc::cp_commit();
            pa_tc::cp_wait<0>();
            pa_tc::fence_smem_to_async();                    // cp.async writes -> tensor core reads
            ws_arrive(&bars[kQFull]);
            for (int j = 0; j < it.nsteps; ++j, ++kv_it) {
                const int st = kv_it % kWsStages;
                const uint32_t use = kv_it / kWsStages;
                if (use > 0 && !ws_wait(&bars[kKvEmpty0 + st], (use - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                unsigned char* stage = base + kWsStageOff + st * kStageBytes;
                int phys[kStep / 16], loaded = 0;
#pragma unroll
                for (int b = 0; b < kStep / 16; ++b) {
                    const int rel = j * kStep + 16 * b, bi = rel >> 4;
                    const int id = bi < 32 ? __shfl_sync(0xffffffffu, tb0, bi & 31)
                                           : __shfl_sync(0xffffffffu, tb1, bi & 31);
                    phys[b] = it.t0 + rel < it.t1 ? id : -1;
                    if (phys[b] >= 0) loaded |= 1 << b;
                }
                // slots without keys keep what an earlier step left: their scores
                // are masked, and zero values keep 0 * Inf out of P.V (fp8: the
                // converter warps write those zeros)
                if (!F8 && loaded != (1 << (kStep / 16)) - 1) {
#pragma unroll
                    for (int b = 0; b < kStep / 16; ++b)
                        if (!((loaded >> b) & 1))
                            for (int o = lane * 16; o < 4096; o += 32 * 16)
                                *reinterpret_cast<uint4*>(stage + 16384 + b * 4096 + o) = make_uint4(0u, 0u, 0u, 0u);
                    pa_tc::fence_smem_to_async();
                }
                __syncwarp();
                if (lane == 0) {
                    stage_mask[st] = loaded;
                    const uint32_t kst = sbase + kWsStageOff + st * kStageBytes;
                    pa_tc::mbar_expect_tx(&bars[kKvFull0 + st],
                                          static_cast<uint32_t>(__popc(loaded)) * (F8 ? 2 * 2048 : 2 * 2048 + 4096));
#pragma unroll
                    for (int b = 0; b < kStep / 16; ++b) {
                        if (phys[b] < 0) continue;
                        if constexpr (F8) {
                            // one block's codes for this KV head: K [16][128] then V^T [128][16]
                            const uint32_t cst = sbase + kWsCodeOff + st * kWsCodeBytes;
                            const size_t tile = (static_cast<size_t>(phys[b]) * Hkv + it.h) * 2048;
                            pa_tc::bulk_load(cst + b * 2048, static_cast<const unsigned char*>(p.k) + tile, 2048,
                                             &bars[kKvFull0 + st]);
                            pa_tc::bulk_load(cst + 8192 + b * 2048, static_cast<const unsigned char*>(p.v) + tile,
                                             2048, &bars[kKvFull0 + st]);
                        } else {
                            const int yk = (phys[b] * Hkv + it.h) * 16, yv = (phys[b] * Hkv + it.h) * kD;
                            pa_tc::tma_load_2d(kst + b * 2048, &kmap, 0, yk, &bars[kKvFull0 + st]);
                            pa_tc::tma_load_2d(kst + 8192 + b * 2048, &kmap, 64, yk, &bars[kKvFull0 + st]);
                            pa_tc::tma_load_2d(kst + 16384 + b * 4096, &vmap, 0, yv, &bars[kKvFull0 + st]);
                        }
                    }
                }
                __syncwarp();
                ++fills[st];
            }
        }
        // every copy issued must have landed before the CTA's shared memory is released
        for (int s = 0; s < kWsStages; ++s)
            if (fills[s] > 0) pa_tc::mbar_wait(&bars[kKvFull0 + s], (fills[s] - 1) & 1, kWaitLimit);
    } else if (warp == 5) {
        // ----------------------------------------------- Q.K^T issue
        uint32_t kv_it = 0, s_it = 0;
        int kk = 0;
        for (int item = blockIdx.x; ok && item < p.n_shared_items; item += gridDim.x, ++kk) {
            const WsItem it = ws_item(p, item);
            if (!ws_wait(&bars[F8 ? kQConv : kQFull], kk & 1, abort_flag)) { ok = false; break; }
            for (int j = 0; j < it.nsteps; ++j, ++kv_it, ++s_it) {
                const int st = kv_it % kWsStages, sb = s_it & 1;
                if (!ws_wait(&bars[(F8 ? kKvConv0 : kKvFull0) + st], (kv_it / kWsStages) & 1, abort_flag) ||
                    ((s_it >> 1) > 0 && !ws_wait(&bars[kSEmpty0 + sb], ((s_it >> 1) - 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                pa_tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kst = sbase + kWsStageOff + st * kStageBytes;
#pragma unroll
                    for (int q = 0; q < kD / 16; ++q) {
                        const uint64_t a = pa_tc::sw128_desc(sbase + kQOff + (q >> 2) * 16384 + (q & 3) * 32);
                        const uint64_t b = pa_tc::sw128_desc(kst + (q >> 2) * 8192 + (q & 3) * 32);
                        pa_tc::mma_bf16(tmem + sb * 64, a, b, F8 ? kIdescQK16 : kIdescQK, q > 0);
                    }
                    pa_tc::commit(&bars[kSFull0 + sb]);
                    if (j == it.nsteps - 1) pa_tc::commit(&bars[kQEmpty]);   // Q tile free
                }
                __syncwarp();
            }
        }
        // every MMA issued must be complete before TMEM is freed
        if (lane == 0) pa_tc::commit(&bars[kMmaDone]);
        __syncwarp();
        pa_tc::mbar_wait(&bars[kMmaDone], 0, kWaitLimit);
    } else if (warp == 6) {
        // ------------------------------------------------- P.V issue
        // P.V(j) needs P(j) from the softmax warps, which took S(j), which
        // needed the step's keys: so its Q.K^T is done and its values landed
        // (the wait on the stage below is already complete).
        uint32_t kv_it = 0, p_it = 0;
        int kk = 0;
        for (int item = blockIdx.x; ok && item < p.n_shared_items; item += gridDim.x, ++kk) {
            const WsItem it = ws_item(p, item);
            const int ob = kk & 1;
            for (int j = 0; j < it.nsteps; ++j, ++kv_it, ++p_it) {
                const int st = kv_it % kWsStages, pb = p_it & 1;
                if (!ws_wait(&bars[kPFull0 + pb], (p_it >> 1) & 1, abort_flag) ||
                    !ws_wait(&bars[(F8 ? kKvConv0 : kKvFull0) + st], (kv_it / kWsStages) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                pa_tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kst = sbase + kWsStageOff + st * kStageBytes;
                    const uint32_t ph = tP + pb * 64, pl = ph + 32, od = tO + ob * 128;
#pragma unroll
                    for (int q = 0; q < kStep / 16; ++q) {
                        const uint64_t b = pa_tc::sw32_desc(kst + 16384 + q * 4096);   // block q's V^T
                        pa_tc::mma_bf16_ta(od, ph + q * 8, b, F8 ? kIdescPV16 : kIdescPV, !(j == 0 && q == 0));
                        pa_tc::mma_bf16_ta(od, pl + q * 8, b, F8 ? kIdescPV16 : kIdescPV, true);
                    }
                    pa_tc::commit(&bars[kKvEmpty0 + st]);    // the stage may be refilled
                    pa_tc::commit(&bars[kPEmpty0 + pb]);     // P buffer free, O settled up to here
                    if (j == it.nsteps - 1) pa_tc::commit(&bars[kOFull0 + ob]);
                }
                __syncwarp();
            }
        }
        if (lane == 0) pa_tc::commit(&bars[kMmaDone]);
        __syncwarp();
        pa_tc::mbar_wait(&bars[kMmaDone], 0, kWaitLimit);
    } else if (F8 && warp >= 7) {
        // ----------------------------------------------- fp8: converters
        // thread ct of 128: the item's Q tile re-rounded to f16 in place, then
        // every step's codes widened into the stage's f16 layouts
        const int ct = tid - 7 * 32;
        uint32_t kv_it = 0;
        int kk = 0;
        for (int item = blockIdx.x; ok && item < p.n_shared_items; item += gridDim.x, ++kk) {
            const WsItem it = ws_item(p, item);
            if (!ws_wait(&bars[kQFull], kk & 1, abort_flag)) { ok = false; break; }
            for (int i = ct; i < kRows * 16; i += 128) {            // 16-byte chunks of the Q tile
                uint4* q16 = reinterpret_cast<uint4*>(base + kQOff + i * 16);
                *q16 = bf16x8_to_f16x8(*q16);
            }
            pa_tc::fence_smem_to_async();                           // generic writes -> tensor core reads
            __syncwarp();
            if (lane == 0) ws_arrive(&bars[kQConv]);
            for (int j = 0; j < it.nsteps; ++j, ++kv_it) {
                const int st = kv_it % kWsStages;
                if (!ws_wait(&bars[kKvFull0 + st], (kv_it / kWsStages) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int loaded = stage_mask[st];
                const unsigned char* codes = base + kWsCodeOff + st * kWsCodeBytes;
                unsigned char* stage = base + kWsStageOff + st * kStageBytes;
                // K: key row `key` of the step (block key / 16), 8-value chunk c of
                // its 128 values, into half c / 8 (values 0-63 / 64-127) of the
                // 128-byte-swizzled tile, at 16-byte chunk c % 8 of the row
                for (int gi = ct; gi < kStep * 16; gi += 128) {
                    const int key = gi >> 4, c = gi & 15, b = key >> 4;
                    uint4 y = make_uint4(0u, 0u, 0u, 0u);
                    if ((loaded >> b) & 1)
                        y = e4m3x8_to_f16x8(
                            *reinterpret_cast<const uint2*>(codes + b * 2048 + (key & 15) * 128 + c * 8));
                    *reinterpret_cast<uint4*>(stage + (c >> 3) * 8192 + pa_tc::sw128_off(key, c & 7)) = y;
                }
                // V^T: block b, value row d, tokens 8k..8k+7, into the 32-byte-swizzled
                // tile (row d at d * 32, its two halves swapped when bit 2 of d is set);
                // blocks without keys get zeros (0 * Inf stays out of P.V)
                for (int gi = ct; gi < (kStep / 16) * kD * 2; gi += 128) {
                    const int b = gi >> 8, d = (gi >> 1) & (kD - 1), k = gi & 1;
                    uint4 y = make_uint4(0u, 0u, 0u, 0u);
                    if ((loaded >> b) & 1)
                        y = e4m3x8_to_f16x8(*reinterpret_cast<const uint2*>(codes + 8192 + b * 2048 + d * 16 + k * 8));
                    *reinterpret_cast<uint4*>(stage + 16384 + b * 4096 + d * 32 + ((k ^ ((d >> 2) & 1)) << 4)) = y;
                }
                pa_tc::fence_smem_to_async();
                __syncwarp();
                if (lane == 0) ws_arrive(&bars[kKvConv0 + st]);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;   // this warp's TMEM lanes
        const float sl = p.scale_log2;
        uint32_t kv_it = 0, s_it = 0, p_it = 0;
        int kk = 0;
        // the previous item's partial rows, written during this item's first step
        struct Pending {
            bool live;
            int kk;
            size_t slot;            // this thread's partial slot (valid when row_ok)
            bool row_ok;
            int row_n;
            float m, l;
        } pend = {false, 0, 0, false, 0, 0.f, 0.f};
        auto write_partial = [&]() {
            if (!ws_wait(&bars[kOFull0 + (pend.kk & 1)], (pend.kk >> 1) & 1, abort_flag)) return false;
            pa_tc::fence_after_sync();
            float* acc = p.spart_acc + (pend.slot * G + pend.row_n) * kD;
            const uint32_t od = tO + (pend.kk & 1) * 128 + lane_sel;
#pragma unroll 1
            for (int cc = 0; cc < kD / 32; ++cc) {
                float o[32];
                pa_tc::tmem_ld32(od + cc * 32, o);
                pa_tc::tmem_wait_ld();
                if (pend.row_ok) {
                    const float vs = F8 ? p.v_scale : 1.f;            // fp8: the sums of codes * v_scale
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(acc + cc * 32 + i) =
                            make_float4(o[i] * vs, o[i + 1] * vs, o[i + 2] * vs, o[i + 3] * vs);
                }
            }
            if (pend.row_ok) {
                p.spart_ml[(pend.slot * G + pend.row_n) * 2] = pend.m;
                p.spart_ml[(pend.slot * G + pend.row_n) * 2 + 1] = pend.l;
            }
            pa_tc::fence_before_sync();
            pend.live = false;
            return true;
        };
        for (int item = blockIdx.x; ok && item < p.n_shared_items; item += gridDim.x, ++kk) {
            const WsItem it = ws_item(p, item);
            ws_validate(p, it, tid);
            const int row_m = it.m0 + tid / G, row_n = tid - (tid / G) * G;
            const bool row_ok = tid < p.members_per_tile * G && row_m < it.m1;
            const uint32_t od = tO + (kk & 1) * 128 + lane_sel;   // this item's O rows
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < it.nsteps; ++j, ++kv_it, ++s_it, ++p_it) {
                const int st = kv_it % kWsStages, sb = s_it & 1;
                // the stage's keys have landed (and its slot mask is written)
                if (!ws_wait(&bars[kKvFull0 + st], (kv_it / kWsStages) & 1, abort_flag) ||
                    !ws_wait(&bars[kSFull0 + sb], (s_it >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int loaded = stage_mask[st];
                pa_tc::fence_after_sync();
                // scores of this row in two halves of 32 keys (TMEM columns)
                float sa[32], sb32[32];
                pa_tc::tmem_ld32(tmem + sb * 64 + lane_sel, sa);
                pa_tc::tmem_ld32(tmem + sb * 64 + lane_sel + 32, sb32);
                pa_tc::tmem_wait_ld();
                pa_tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ws_arrive(&bars[kSEmpty0 + sb]);   // S buffer free
                // Fast path (every key slot loaded, positive scale): the maximum of
                // the scaled scores is scale times the raw maximum, and each weight
                // is one FFMA and one exp2.  Otherwise: scale, mask, then exp2.
                const bool fast = loaded == (1 << (kStep / 16)) - 1 && sl > 0.f;
                float mx = -INFINITY;
                if (fast) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fmaxf(sa[i], sb32[i]));
                    mx *= sl;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        sa[i] = (loaded >> (i >> 4)) & 1 ? sa[i] * sl : -INFINITY;
                        sb32[i] = (loaded >> (2 + (i >> 4))) & 1 ? sb32[i] * sl : -INFINITY;
                        mx = fmaxf(mx, fmaxf(sa[i], sb32[i]));
                    }
                }
                // raise the reference maximum only when it is far behind (or unset)
                const bool first = m_ref == -INFINITY;
                const bool raise = !first && mx > m_ref + 8.f;
                const float old_ref = m_ref;
                if (first || raise) m_ref = mx;
                const float ref = m_ref == -INFINITY ? 0.f : m_ref;
                if (__any_sync(0xffffffffu, raise)) {
                    // O holds the sums up to the previous step once its P.V is done;
                    // rescale this warp's rows of O to the new reference
                    if (p_it > 0 &&
                        !ws_wait(&bars[kPEmpty0 + ((p_it - 1) & 1)], ((p_it - 1) >> 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    pa_tc::fence_after_sync();
                    const float corr = raise ? exp2_approx(old_ref - m_ref) : 1.f;
                    if (raise) l *= corr;
#pragma unroll 1
                    for (int cc = 0; cc < kD / 32; ++cc) {
                        float o[32];
                        pa_tc::tmem_ld32(od + cc * 32, o);
                        pa_tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= corr;
                        pa_tc::tmem_st32(od + cc * 32, o);
                    }
                }
                // this step's P buffer was last read by the P.V two steps back
                const int pb = p_it & 1;
                if (p_it >= 2 && !ws_wait(&bars[kPEmpty0 + pb], ((p_it >> 1) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                pa_tc::fence_after_sync();
                const uint32_t ph = tP + pb * 64 + lane_sel, pl = ph + 32;
                // weight = exp2(x * xs - ref): raw scores with xs = scale on the
                // fast path, already scaled (and masked) scores with xs = 1 otherwise
                const float nref = -ref, xs = fast ? sl : 1.f;
                float sum = 0.f;
                auto weights = [&](const float (&x)[32], uint32_t col) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = exp2_approx(fmaf(x[2 * e], xs, nref));
                        const float p1 = exp2_approx(fmaf(x[2 * e + 1], xs, nref));
                        sum += p0 + p1;
                        if constexpr (F8) {
                            hi[e] = pa_dev::pack_f16(p0, p1);
                            lo[e] = pa_dev::pack_f16(p0 - pa_dev::f16_lo(hi[e]), p1 - pa_dev::f16_hi(hi[e]));
                        } else {
                            hi[e] = pa_dev::pack_bf16(p0, p1);
                            lo[e] = pa_dev::pack_bf16(p0 - pa_dev::bf16_lo(hi[e]), p1 - pa_dev::bf16_hi(hi[e]));
                        }
                    }
                    pa_tc::tmem_st16u(ph + col, hi);
                    pa_tc::tmem_st16u(pl + col, lo);
                };
                weights(sa, 0);                                 // keys 0..31 of the step
                weights(sb32, 16);                              // keys 32..63
                pa_tc::tmem_wait_st();
                l += sum;
                pa_tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) ws_arrive(&bars[kPFull0 + pb]);
                // the previous item's rows, while this item's P.V runs
                if (j == 0 && pend.live && !write_partial()) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            pend.live = true;
            pend.kk = kk;
            pend.row_ok = row_ok;
            pend.row_n = row_n;
            pend.slot = row_ok ? (static_cast<size_t>(p.g_spart_base[it.grp]) +
                                  static_cast<size_t>(row_m) * it.nC + it.chunk) * Hkv + it.h : 0;
            pend.m = m_ref;
            pend.l = l;
        }
        if (ok && pend.live && !write_partial()) ok = false;
    }
    if (!ok) {
        *abort_flag = 1;
        if (lane == 0) pa_dev::record_error(p.err, PA_ERR_CUDA);
    }
    pa_tc::fence_before_sync();
    __syncthreads();
    pa_tc::fence_after_sync();
    if (warp == 0) pa_tc::tmem_free<kWsTmemCols>(tmem);
}

// ------------------------------------------------------------ prefill ---
//
// Chunked prefill on the same machinery: one CTA per (128 query rows, KV
// head, sequence), a row being one (chunk token, query head of the group)
// pair, so a tile holds 128/G chunk tokens.  The tile's keys [0, last row's
// position] stream through the two TMA stages in 64-token steps exactly as a
// shared span does (S in TMEM, per-row softmax by the thread owning the TMEM
// lane, P as bf16 high + low in TMEM, O += P.V in TMEM); the causal mask is
// applied to the scores (a row at position p keeps keys 0 .. p), and each row's
// normalised output is written directly.  Block ids come from the sequence's
// table as each step is staged.
// F8 (fp8 pool): a step's e4m3 codes (K [16][128] and V^T [128][16] per
// block, 2 KB each) are copied by bulk copy into the V^T half of the stage;
// once they land every thread reads its 16 groups of 8 codes into registers
// and, after a block-wide barrier, writes them widened to f16 (exact) into the
// stage's K and V^T layouts; the Q tile is re-rounded to f16 in place (each
// thread the chunks it copied), the MMAs are f16, P is an f16 pair, k_scale
// sits in the score factor and v_scale in the rows' normaliser.  kmap / vmap
// are unused then.
template <bool F8>
__global__ void __launch_bounds__(kThreads, 2)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ unsigned char tc_raw[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const bool reporter = tid == 0 && tile == 0 && h == 0;
    pa_dev::wait_prior_grid();
    pa_dev::allow_next_grid();

    // the item (uniform over the CTA: every early return happens before any
    // barrier, mbarrier or TMEM is touched)
    const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
    const int n = q1 - q0;
    const int L = __ldg(p.lens + s);
    if (q0 < 0 || n < 0 || q1 > p.T || L < n || n > p.max_q) {
        if (reporter) pa_dev::record_error(p.err, PA_ERR_INVALID_ARG);
        return;
    }
    if (L > p.max_blocks * 16) {
        if (reporter) pa_dev::record_error(p.err, PA_ERR_BAD_LENGTH);
        return;
    }
    const int G = p.G, Hkv = p.Hkv;
    const int r_lo = tile * kRows;
    if (r_lo >= n * G) return;
    const int P0 = L - n;
    const int rows_end = min(n * G, r_lo + kRows);
    const int kv_end = P0 + (rows_end - 1) / G + 1;        // keys [0, kv_end) reach some row
    const int nsteps = (kv_end + kStep - 1) / kStep;

    const uint32_t raw_s = pa_tc::smem_u32(tc_raw);
    unsigned char* base = tc_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = pa_tc::smem_u32(base);
    uint64_t* bar_s = reinterpret_cast<uint64_t*>(base + kMiscOff);
    uint64_t* bar_pv = bar_s + 1;
    uint64_t* bar_full = bar_s + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + kMiscOff + 32);
    volatile int* s_skip = reinterpret_cast<volatile int*>(base + kMiscOff + 48);   // [2] per stage
    // a thread whose bounded wait gave up raises this; the CTA leaves the step
    // loop together at the next block barrier
    volatile int* s_abort = reinterpret_cast<volatile int*>(base + kMiscOff + 56);
    if (tid == 0) {
        *s_abort = 0;
        pa_tc::mbar_init(bar_s, 1);
        pa_tc::mbar_init(bar_pv, 1);
        pa_tc::mbar_init(bar_full, 1);
        pa_tc::mbar_init(bar_full + 1, 1);
        pa_tc::mbar_init_fence();
    }
    if (warp == 0) pa_tc::tmem_alloc<kTmemCols>(tslot);
    pa_tc::fence_before_sync();
    __syncthreads();
    pa_tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem, tO = tmem + 64, tPh = tmem + 192, tPl = tmem + 224;
    const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t ph_s = 0, ph_pv = 0, ph_full0 = 0, ph_full1 = 0;
    int pending = 0;                    // thread 0: stages with copies issued and not yet waited for
    bool ok = true;

    // this thread's row: TMEM lane tid
    const int r = r_lo + tid;
    const int qi = r / G;
    const bool row_ok = r < rows_end;
    const int pos = row_ok ? P0 + qi : -1;
    const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
    const float sl = p.scale_log2;

    // Q tile: 128 rows x 16 chunks of 16 B, zero rows past the chunk
    for (int idx = tid; idx < kRows * 16; idx += kThreads) {
        const int rr = idx >> 4, c16 = idx & 15;
        const int gr = r_lo + rr;
        const bool v = gr < rows_end;
        const uint16_t* src = p.q + (v ? ((static_cast<size_t>(q0 + gr / G) * p.Hq +
                                           static_cast<size_t>(h) * G + gr % G) * kD + c16 * 8)
                                       : 0);
        pa_tc::cp16(sbase + kQOff + (c16 >> 3) * 16384 + pa_tc::sw128_off(rr, c16 & 7), src,
                    v ? 16u : 0u);
    }
    pa_tc::cp_commit();

    // One thread stages step j: its (up to) four 16-token blocks, K as two
    // 64-d boxes and V^T as one box each, on the stage's mbarrier; the block
    // slots it leaves unloaded go to s_skip[stage] (read after the wait).
    auto load_step = [&](int j) {
        if (tid != 0) return;
        const int st = j & 1;
        pending |= 1 << st;
        const uint32_t kst = sbase + kStageOff + st * kStageBytes;
        int phys[kStep / 16], skip = 0;
        uint32_t bytes = 0;
#pragma unroll
        for (int b = 0; b < kStep / 16; ++b) {
            const int tok = j * kStep + 16 * b;
            phys[b] = -1;
            if (tok < kv_end) {
                const int x = __ldg(table + tok / 16);
                if (x < 0 || x >= p.num_blocks) pa_dev::record_error(p.err, PA_ERR_BAD_BLOCK_ID);
                else phys[b] = x;
            }
            if (phys[b] >= 0) bytes += F8 ? 2 * 2048 : 2 * 2048 + 4096;
            else skip |= 1 << b;
        }
        s_skip[st] = skip;
        pa_tc::mbar_expect_tx(bar_full + st, bytes);
#pragma unroll
        for (int b = 0; b < kStep / 16; ++b) {
            if (phys[b] < 0) continue;
            if constexpr (F8) {
                // codes: K at 16 KB + 2 KB b, V^T at 24 KB + 2 KB b of the stage
                const size_t tile = (static_cast<size_t>(phys[b]) * Hkv + h) * 2048;
                pa_tc::bulk_load(kst + 16384 + b * 2048, static_cast<const unsigned char*>(p.k) + tile, 2048,
                                 bar_full + st);
                pa_tc::bulk_load(kst + 24576 + b * 2048, static_cast<const unsigned char*>(p.v) + tile, 2048,
                                 bar_full + st);
            } else {
                const int yk = (phys[b] * Hkv + h) * 16, yv = (phys[b] * Hkv + h) * kD;
                pa_tc::tma_load_2d(kst + b * 2048, &kmap, 0, yk, bar_full + st);
                pa_tc::tma_load_2d(kst + 8192 + b * 2048, &kmap, 64, yk, bar_full + st);
                pa_tc::tma_load_2d(kst + 16384 + b * 4096, &vmap, 0, yv, bar_full + st);
            }
        }
    };

    load_step(0);
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nsteps && ok; ++j) {
        const int st = j & 1;
        // S = Q.K^T of this step is issued as soon as its keys have landed,
        // behind the previous step's P.V in the tensor pipe: it writes only the
        // S columns (read out before that P.V was issued) and reads this
        // step's stage, so it need not wait for that P.V to finish
        if (j == 0) {
            pa_tc::cp_wait<0>();
            if constexpr (F8) {
                // this thread's own Q chunks (those it copied), bf16 -> f16 in place
                for (int idx = tid; idx < kRows * 16; idx += kThreads) {
                    const int rr = idx >> 4, c16 = idx & 15;
                    uint4* q16 = reinterpret_cast<uint4*>(base + kQOff + (c16 >> 3) * 16384 +
                                                          pa_tc::sw128_off(rr, c16 & 7));
                    *q16 = bf16x8_to_f16x8(*q16);
                }
            }
        }
        {
            // each thread waits for the stage itself (its codes, its V^T rows):
            // no block barrier here
            const bool w = pa_tc::mbar_wait(bar_full + st, st ? ph_full1 : ph_full0, kWaitLimit);
            if (st) ph_full1 ^= 1u; else ph_full0 ^= 1u;
            if (w) pending &= ~(1 << st);
            if (!w) *s_abort = 1;
        }
        if constexpr (F8) {
            // the step's codes into registers (8 K groups, 8 V^T groups of 8 codes),
            // then, once every thread has read its own, widened into the stage
            unsigned char* stg = base + kStageOff + st * kStageBytes;
            uint2 kc[8], vc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int gi = tid + kThreads * k;
                const int key = gi >> 4, c = gi & 15, b = key >> 4;
                kc[k] = *reinterpret_cast<const uint2*>(stg + 16384 + b * 2048 + (key & 15) * 128 + c * 8);
                const int vb = gi >> 8, d = (gi >> 1) & (kD - 1), kh = gi & 1;
                vc[k] = *reinterpret_cast<const uint2*>(stg + 24576 + vb * 2048 + d * 16 + kh * 8);
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int gi = tid + kThreads * k;
                const int key = gi >> 4, c = gi & 15;
                *reinterpret_cast<uint4*>(stg + (c >> 3) * 8192 + pa_tc::sw128_off(key, c & 7)) = e4m3x8_to_f16x8(kc[k]);
                const int vb = gi >> 8, d = (gi >> 1) & (kD - 1), kh = gi & 1;
                *reinterpret_cast<uint4*>(stg + 16384 + vb * 4096 + d * 32 + ((kh ^ ((d >> 2) & 1)) << 4)) =
                    e4m3x8_to_f16x8(vc[k]);
            }
            __syncthreads();                               // before the tails are zeroed row by row
        }
        // Keys that no row of the tile may weigh: block slots this step did not
        // load (past the tile's last key, or a block id outside the pool),
        // which hold what an earlier step left there, and positions at or past
        // the context length in the sequence's last block, which hold whatever
        // the block held before.  Their scores are masked below, but a
        // zero-weight value still enters P.V and 0 * Inf or 0 * NaN is NaN:
        // zero those V^T columns (thread t clears row t of each tile).
        const int kbase = j * kStep;
        const int skip = s_skip[st];                       // bit b: block slot b not loaded
#pragma unroll
        for (int b = 0; b < kStep / 16; ++b) {
            const int tok = kbase + 16 * b;
            const int zero_from = (skip >> b) & 1 ? 0 : tok + 16 > L ? L - tok : 16;
            if (zero_from < 16)
                pa_tc::zero_vt_row_tail(base + kStageOff + st * kStageBytes + 16384 + b * 4096, tid,
                                        zero_from);
        }
        pa_tc::fence_smem_to_async();
        pa_tc::fence_before_sync();
        if (__syncthreads_or(*s_abort)) { ok = false; break; }   // Q (every thread's copies) and the stage
        pa_tc::fence_after_sync();
        const uint32_t kst = sbase + kStageOff + st * kStageBytes;
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t a = pa_tc::sw128_desc(sbase + kQOff + (kk >> 2) * 16384 + (kk & 3) * 32);
                const uint64_t b = pa_tc::sw128_desc(kst + (kk >> 2) * 8192 + (kk & 3) * 32);
                pa_tc::mma_bf16(tS, a, b, F8 ? kIdescQK16 : kIdescQK, kk > 0);
            }
            pa_tc::commit(bar_s);
        }
        // the previous P.V must be done before its stage is refilled, before P
        // is overwritten and before O is rescaled
        // (every thread waits for itself: the stage refill, its P columns and
        // its O row each need only their own view of these phases)
        if (j > 0) {
            const bool w = pa_tc::mbar_wait(bar_pv, ph_pv, kWaitLimit);
            if (!w) *s_abort = 1;
            ph_pv ^= 1u;
        }
        if (j + 1 < nsteps && !*s_abort) load_step(j + 1);
        {
            const bool w = pa_tc::mbar_wait(bar_s, ph_s, kWaitLimit);
            if (!w) *s_abort = 1;
        }
        ph_s ^= 1u;
        pa_tc::fence_after_sync();
        float sc[64];
        {
            float a32[32], b32[32];
            pa_tc::tmem_ld32(tS + lane_sel, a32);
            pa_tc::tmem_ld32(tS + lane_sel + 32, b32);
            pa_tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                sc[i] = a32[i];
                sc[32 + i] = b32[i];
            }
        }
        // causal mask: key j*64 + i is visible to this row iff it is at or
        // before the row's position (pos < kv_end, so this also ends the keys);
        // a block whose id is outside the pool was not loaded and is skipped
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            sc[i] = kbase + i <= pos && !((skip >> (i >> 4)) & 1) ? sc[i] * sl : -INFINITY;
            mx = fmaxf(mx, sc[i]);
        }
        const bool first = m_ref == -INFINITY;
        const bool raise = !first && mx > m_ref + 8.f;
        if (first) m_ref = mx;
        if (__any_sync(0xffffffffu, raise)) {
            const float corr = raise ? exp2_approx(m_ref - mx) : 1.f;
            if (raise) {
                l *= corr;
                m_ref = mx;
            }
#pragma unroll
            for (int cc = 0; cc < kD / 32; ++cc) {
                float o[32];
                pa_tc::tmem_ld32(tO + lane_sel + cc * 32, o);
                pa_tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= corr;
                pa_tc::tmem_st32(tO + lane_sel + cc * 32, o);
            }
            pa_tc::tmem_wait_st();
        }
        const float ref = m_ref == -INFINITY ? 0.f : m_ref;
        float sum = 0.f;
        {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float p0 = exp2_approx(sc[2 * e] - ref);
                const float p1 = exp2_approx(sc[2 * e + 1] - ref);
                sum += p0 + p1;
                if constexpr (F8) {
                    hi[e] = pa_dev::pack_f16(p0, p1);
                    lo[e] = pa_dev::pack_f16(p0 - pa_dev::f16_lo(hi[e]), p1 - pa_dev::f16_hi(hi[e]));
                } else {
                    hi[e] = pa_dev::pack_bf16(p0, p1);
                    lo[e] = pa_dev::pack_bf16(p0 - pa_dev::bf16_lo(hi[e]), p1 - pa_dev::bf16_hi(hi[e]));
                }
            }
            pa_tc::tmem_st32u(tPh + lane_sel, hi);
            pa_tc::tmem_st32u(tPl + lane_sel, lo);
            pa_tc::tmem_wait_st();
        }
        l += sum;
        pa_tc::fence_before_sync();
        if (__syncthreads_or(*s_abort)) { ok = false; break; }   // every row's P is in TMEM
        pa_tc::fence_after_sync();
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < kStep / 16; ++kk) {
                const uint64_t b = pa_tc::sw32_desc(kst + 16384 + kk * 4096);
                pa_tc::mma_bf16_ta(tO, tPh + kk * 8, b, F8 ? kIdescPV16 : kIdescPV, j > 0 || kk > 0);
                pa_tc::mma_bf16_ta(tO, tPl + kk * 8, b, F8 ? kIdescPV16 : kIdescPV, true);
            }
            pa_tc::commit(bar_pv);
        }
    }
    if (ok) {
        const bool w = pa_tc::mbar_wait(bar_pv, ph_pv, kWaitLimit);
        ok = __syncthreads_and(w);
        ph_pv ^= 1u;
    }
    if (ok) {
        pa_tc::fence_after_sync();
        const float inv = l > 0.f ? (F8 ? p.v_scale : 1.f) / l : 0.f;
        const size_t orow = row_ok ? (static_cast<size_t>(q0 + qi) * p.Hq +
                                      static_cast<size_t>(h) * G + r % G) * kD : 0;
#pragma unroll
        for (int cc = 0; cc < kD / 32; ++cc) {
            float o[32];
            pa_tc::tmem_ld32(tO + lane_sel + cc * 32, o);
            pa_tc::tmem_wait_ld();
            if (!row_ok) continue;
            if (p.out_bf16) {
                uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + orow + cc * 32);
#pragma unroll
                for (int i = 0; i < 32; i += 8)
                    *reinterpret_cast<uint4*>(dst + i / 2) =
                        make_uint4(pa_dev::pack_bf16(o[i] * inv, o[i + 1] * inv),
                                   pa_dev::pack_bf16(o[i + 2] * inv, o[i + 3] * inv),
                                   pa_dev::pack_bf16(o[i + 4] * inv, o[i + 5] * inv),
                                   pa_dev::pack_bf16(o[i + 6] * inv, o[i + 7] * inv));
            } else {
                float* dst = static_cast<float*>(p.out) + orow + cc * 32;
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(dst + i) =
                        make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
            }
        }
    }
    if (!ok && tid == 0) {
        pa_dev::record_error(p.err, PA_ERR_CUDA);
        // copies still in flight land before the CTA's shared memory is released
        // (bounded again)
        if (pending & 1) pa_tc::mbar_wait(bar_full, ph_full0, kWaitLimit);
        if (pending & 2) pa_tc::mbar_wait(bar_full + 1, ph_full1, kWaitLimit);
    }
    pa_tc::cp_wait<0>();
    pa_tc::fence_before_sync();
    __syncthreads();
    pa_tc::fence_after_sync();
    if (warp == 0) pa_tc::tmem_free<kTmemCols>(tmem);
}

}  // namespace

namespace pa_detail {

bool prefill_tc_eligible(const pa_pool* pool) {
    // bf16: 32-bit TMA coordinates (value rows num_blocks * Hkv * D); fp8: bulk copies of codes
    return (pool->dtype == PA_BF16 || pool->dtype == PA_FP8E4M3) && pool->head_dim == kD &&
           pool->block_size == 16 &&
           (pool->dtype == PA_FP8E4M3 || static_cast<long long>(pool->num_blocks) * pool->kv_heads * kD < (1LL << 31));
}

int prefill_tc_rows() { return kRows; }

int launch_prefill_tc(pa_pool* pool, const PrefillParams& p, dim3 grid, cudaStream_t st) {
    const bool f8 = pool->dtype == PA_FP8E4M3;
    if (!f8) {
        const int rc = ensure_tensor_maps(pool);
        if (rc != PA_OK) return rc;
    }
    auto kernel = f8 ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
        return PA_ERR_CUDA;
    const cudaError_t e = launch_pdl(kernel, grid, dim3(kThreads), kSmemBytes, st, p,
                                     pool->kmap, pool->vmap);
    count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

bool shared_tc_eligible(const pa_pool* pool, int G) {
    // bf16: TMA coordinates are 32-bit, so value rows num_blocks * Hkv * D stay
    // below 2^31; fp8: bulk copies of codes, and a CTA that needs nearly all of
    // the opt-in shared memory
    const bool f8 = pool->dtype == PA_FP8E4M3;
    return (pool->dtype == PA_BF16 || f8) && pool->head_dim == kD && G >= 1 && G <= 8 &&
           pool->block_size == 16 &&
           (f8 ? static_cast<uint32_t>(pool->smem_optin) >= ws_smem_bytes(true)
               : static_cast<long long>(pool->num_blocks) * pool->kv_heads * kD < (1LL << 31));
}

// TMA descriptors over the pool (16-token blocks): K as
// [num_blocks*Hkv*16 rows][D] with 64 x 16 boxes (128-byte swizzle); V^T as
// [num_blocks*Hkv*D rows][16 tokens] with 16 x D boxes (32-byte swizzle).
int ensure_tensor_maps(pa_pool* pool) {
    if (pool->tmaps_ready) return PA_OK;
    const int D = pool->head_dim;
    if (pool->dtype != PA_BF16 || pool->block_size != 16 || D % 64 != 0 || D > 256)
        return PA_ERR_UNSUPPORTED;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return PA_ERR_CUDA;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    const cuuint64_t rows_k = static_cast<cuuint64_t>(pool->num_blocks) * pool->kv_heads * 16;
    const cuuint64_t rows_v = static_cast<cuuint64_t>(pool->num_blocks) * pool->kv_heads * D;
    const cuuint64_t kdim[2] = {static_cast<cuuint64_t>(D), rows_k};
    const cuuint64_t kstr[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t kbox[2] = {64, 16};
    const cuuint64_t vdim[2] = {16, rows_v};
    const cuuint64_t vstr[1] = {16 * 2};
    const cuuint32_t vbox[2] = {16, static_cast<cuuint32_t>(D)};
    const cuuint32_t one[2] = {1, 1};
    if (encode(&pool->kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool->k, kdim, kstr, kbox, one,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    if (encode(&pool->vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool->v, vdim, vstr, vbox, one,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    pool->tmaps_ready = true;
    return PA_OK;
}

int shared_tc_rows() { return kRows; }
int shared_tc_chunk_tokens() { return kChunkBlocks * 16; }

int launch_shared_tc(pa_pool* pool, const DecodeParams& p, cudaStream_t st) {
    if (p.n_shared_items <= 0) return PA_OK;
    const bool f8 = pool->dtype == PA_FP8E4M3;
    if (!f8) {
        const int rc = ensure_tensor_maps(pool);
        if (rc != PA_OK) return rc;
    }
    auto kernel = f8 ? shared_tc_kernel<true> : shared_tc_kernel<false>;
    const uint32_t smem = ws_smem_bytes(f8);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    // one CTA per SM: the split pass of the private suffixes fills the rest of each SM
    const int grid = p.n_shared_items < pool->num_sms ? p.n_shared_items : pool->num_sms;
    const cudaError_t e = launch_pdl(kernel, dim3(grid), dim3(f8 ? kWsThreadsF8 : kWsThreads), smem,
                                     st, p, pool->kmap, pool->vmap);
    count_launch();
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
