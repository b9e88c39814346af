// Paged decode on the 5th-generation tensor cores (tcgen05), the cached tokens
// as the MMA's M dimension.
//
// What it computes is what the split kernels of pa_decode.cu compute
// (kgptalkie "Day 28: PagedAttention / vLLM", "The Block Table Is the Map",
// "Follow One Token Address"): per work item = (sequence, KV head, partition
// of PT tokens) the online-softmax partial of the group's G query heads over
// the partition's keys, found through the sequence's block table in logical
// order; the items come from the same schedule and the same merge kernel
// combines partitions.  Only the engine differs.
//
// A tile is 128 consecutive tokens of an item (eight 16-token blocks):
//   S^T[128 tokens x 16]  = K[128 x 128 d] . Q^T          M=128, N=16, fp32 in TMEM
//   softmax               thread t owns tile row t (TMEM lane t): its token's
//                         scores for the G heads, masked, exp2 against a
//                         per-head reference that is raised only when a tile's
//                         maximum passes it by 2^8 (O^T is rescaled then)
//   O^T[128 d x 32]      += V^T[128 d x 128 tokens] . P^T   M=128, N=32, fp32 in TMEM,
//                         P^T's rows: the weights' high parts, then their low parts
// The group's heads are the N columns (zero queries pad G up to 16), so every
// key and value byte enters the tensor core once for all heads of its group,
// and the MMA's 128 rows are filled by tokens (scores) and by head_dim
// (values) instead of by the few query heads of one sequence.
//
// Roles of one CTA (one per SM, persistent):
//   warps 0-3   softmax and item results (thread t = TMEM lane t)
//   warps 4-11  fp8 pools only: widen the stage's e4m3 codes to f16 straight
//               into TMEM, where they are the A operands of both products
//               (warps 4-7 key row t in lane t, warps 8-11 value row d in
//               lane d, zeroing the codes of tokens that must weigh nothing)
//   producer    takes work tickets into a small item ring, stages each item's
//               queries (f16 for an fp8 pool) and streams its tiles by TMA
//               into a ring of shared-memory stages (block ids read four
//               tiles at a time, a batch ahead; one box per lane)
//   S issuer    one thread: S^T of a tile into one of two S buffers
//   P.V issuer  one thread: O^T += V^T . P^T into the item's O buffer, the
//               high and low parts of P^T stacked as N = 32 (one read of
//               each value tile serves both)
// bf16 pools give both products their A operands from shared memory (keys in
// the 128-byte swizzle, value tiles in the 32-byte swizzle, as TMA lays them
// down); value columns of tokens past the item's end or of blocks left
// unloaded are zeroed there by the softmax threads before the value product,
// so stale non-finite bits never reach it.
// Every hand-off is an mbarrier wait with a poll limit; a role that gives up
// raises a CTA-wide abort flag that ends the other roles' waits, records
// PA_ERR_CUDA, and the CTA drains its own copies and MMAs, frees TMEM and exits.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_sched.cuh"
#include "pa_tc.cuh"

namespace {

using namespace pa_sched;

constexpr int kD = 128;                  // head_dim of this path
constexpr int kTile = 128;               // tokens per tile: M of the score product
constexpr int kTileBlocks = kTile / 16;  // 16-token blocks per tile
constexpr int kN = 16;                   // N of the score product: the group's heads (G <= 8), padded
constexpr int kRing = 4;                 // entries of the item ring
constexpr int kMaxStages = 6;
constexpr int kMaskRing = 16;            // tile masks kept (the producer runs at most kMaxStages + 2 tiles ahead)
constexpr int kItemsPerCta = 8;          // work items per CTA the schedule aims at
constexpr int kPtCap = 2048;             // longest partition, tokens
constexpr uint32_t kWaitLimit = 1u << 20;   // polls; milliseconds, far beyond any copy or MMA

constexpr uint32_t kIdescSbf = pa_tc::idesc_bf16_f32(128, kN);       // scores: N = 16 heads
constexpr uint32_t kIdescS16 = pa_tc::idesc_f16_f32(128, kN);
constexpr uint32_t kIdescPVbf = pa_tc::idesc_bf16_f32(128, 2 * kN);  // values: N = 16 high + 16 low
constexpr uint32_t kIdescPV16 = pa_tc::idesc_f16_f32(128, 2 * kN);

// shared memory (offsets from a 1024-byte-aligned base)
constexpr uint32_t kQOff = 0;                        // 2 buffers: Q^T [16 heads][128 d], 128-byte swizzle
constexpr uint32_t kQBytes = 4096;
constexpr uint32_t kPOff = 2 * kQBytes;              // 2 buffers: P^T [16 high + 16 low rows][128 tokens]
constexpr uint32_t kPBytes = 8192;
constexpr uint32_t kMiscOff = kPOff + 2 * kPBytes;   // mbarriers, then the slots below
constexpr uint32_t kSlotOff = kMiscOff + 512;        // TMEM slot, abort flag, rings, schedule
constexpr uint32_t kWmaxOff = kMiscOff + 1024;       // [2][4 warps][16] tile maxima
constexpr uint32_t kWlOff = kMiscOff + 1536;         // [2][4 warps][16] row sums
constexpr uint32_t kStageOff = kMiscOff + 2048;      // stages, then the schedule's s_start
// bf16 stage: K [2 x 64 d][128 tokens][128 B] (32 KB), V^T [8 blocks][128 d][32 B] (32 KB)
// fp8 stage:  K codes [128 tokens][128 B] (16 KB), V^T codes [8 blocks][128 d][16 B] (16 KB)
__host__ __device__ constexpr uint32_t stage_bytes(bool f8) { return f8 ? 32768u : 65536u; }
__host__ __device__ constexpr int tc_threads(bool f8) { return f8 ? 480 : 224; }

enum Bar : int {
    kItemFull = 0,                       // [kRing]
    kItemEmpty = kItemFull + kRing,      // [kRing]
    kQFull = kItemEmpty + kRing,         // [2] each
    kQEmpty = kQFull + 2,
    kSFull = kQEmpty + 2,
    kSEmpty = kSFull + 2,
    kPFull = kSEmpty + 2,
    kPEmpty = kPFull + 2,
    kOFull = kPEmpty + 2,
    kKwFull = kOFull + 2,                // fp8: widened keys in TMEM
    kKwEmpty = kKwFull + 2,
    kVwFull = kKwEmpty + 2,              // fp8: widened values in TMEM
    kVwEmpty = kVwFull + 2,
    kMxFull = kVwEmpty + 2,              // tile maxima exchanged among the softmax warps
    kLFull = kMxFull + 2,                // row sums exchanged at an item's end
    kMmaDone = kLFull + 2,
    kKvFull = kMmaDone + 1,              // [kMaxStages]
    kKvEmpty = kKvFull + kMaxStages,     // [kMaxStages]
    kNumBars = kKvEmpty + kMaxStages
};
static_assert(kNumBars * 8 <= 512, "mbarriers overflow their region");

// What every role derives from an item index.
struct TcItem {
    int s, h, tok0, tok1, ntiles, L;
    bool direct;        // the sequence's only partition: normalised output, no merge
};

__device__ __forceinline__ TcItem tc_item(const DecodeParams& p, const Sched& sc, const int* s_start,
                                          int item) {
    TcItem it;
    it.s = find_seq(s_start, p.S, item);
    const int local = item - s_start[it.s];
    const int part = local / p.Hkv;
    it.h = local - part * p.Hkv;
    const int L = seq_len(p, it.s, false), start = priv_start(p, it.s), PTq = sc.pt(it.s);
    const int nP = max(1, (max(0, L - start) + PTq - 1) / PTq);
    it.tok0 = start + part * PTq;
    it.tok1 = min(L, it.tok0 + PTq);
    it.ntiles = it.tok1 > it.tok0 ? (it.tok1 - it.tok0 + kTile - 1) / kTile : 0;
    it.direct = nP == 1 && !in_group(p, it.s);
    it.L = L;
    return it;
}

// Maximum over the warp's lanes: floats mapped to order-preserving integers
// for one redux.sync, and back.
__device__ __forceinline__ float warp_max(float x) {
    int i = __float_as_int(x);
    i ^= (i >> 31) & 0x7fffffff;
    i = __reduce_max_sync(0xffffffffu, i);
    i ^= (i >> 31) & 0x7fffffff;
    return __int_as_float(i);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
    return pa_dev::pack_f16(pa_dev::bf16_lo(x), pa_dev::bf16_hi(x));
}

// 16 e4m3 codes widened to 8 f16 pairs (code 2i in the low half of pair i).
__device__ __forceinline__ void widen16(uint4 r, uint32_t* o) {
    o[0] = pa_dev::e4m3x2_to_f16x2(r.x);
    o[1] = pa_dev::e4m3x2_to_f16x2(r.x >> 16);
    o[2] = pa_dev::e4m3x2_to_f16x2(r.y);
    o[3] = pa_dev::e4m3x2_to_f16x2(r.y >> 16);
    o[4] = pa_dev::e4m3x2_to_f16x2(r.z);
    o[5] = pa_dev::e4m3x2_to_f16x2(r.z >> 16);
    o[6] = pa_dev::e4m3x2_to_f16x2(r.w);
    o[7] = pa_dev::e4m3x2_to_f16x2(r.w >> 16);
}

// Codes nv..15 of a 16-code row replaced by +0.
__device__ __forceinline__ uint4 keep_codes(uint4 r, int nv) {
    if (nv >= 16) return r;
    uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = nv - 4 * i;
        w[i] = k <= 0 ? 0u : k >= 4 ? w[i] : (w[i] & ((1u << (8 * k)) - 1u));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// pa_append_decode's write of one sequence's new token, KV head h, into
// (block phys, offset off), by one warp: the key row (contiguous) and the
// value column of the transposed tile, as pa_append_kv writes them (an fp8
// pool's codes quantized exactly as there: e4m3 of fl32(x / scale)).
template <bool F8>
__device__ __forceinline__ void append_token(const DecodeParams& p, int s, int h, int phys, int off,
                                             int lane) {
    const size_t row = (static_cast<size_t>(s) * p.Hkv + h) * kD;
    const size_t tile = (static_cast<size_t>(phys) * p.Hkv + h) * 16 * kD;
    const uint16_t* ks = static_cast<const uint16_t*>(p.new_k) + row;
    const uint16_t* vs = static_cast<const uint16_t*>(p.new_v) + row;
    if (F8) {
        unsigned char* kw = static_cast<unsigned char*>(const_cast<void*>(p.k)) + tile + static_cast<size_t>(off) * kD;
        unsigned char* vw = static_cast<unsigned char*>(const_cast<void*>(p.v)) + tile + off;
        auto bf = [](uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); };
#pragma unroll
        for (int i = lane; i < kD / 2; i += 32) {
            const uint32_t kc = pa_dev::e4m3x2_from_f32(__fdiv_rn(bf(__ldg(ks + 2 * i)), p.k_scale),
                                                        __fdiv_rn(bf(__ldg(ks + 2 * i + 1)), p.k_scale));
            reinterpret_cast<uint16_t*>(kw)[i] = static_cast<uint16_t>(kc);
            const uint32_t vc = pa_dev::e4m3x2_from_f32(__fdiv_rn(bf(__ldg(vs + 2 * i)), p.v_scale),
                                                        __fdiv_rn(bf(__ldg(vs + 2 * i + 1)), p.v_scale));
            vw[static_cast<size_t>(2 * i) * 16] = static_cast<unsigned char>(vc);
            vw[static_cast<size_t>(2 * i + 1) * 16] = static_cast<unsigned char>(vc >> 8);
        }
    } else {
        uint16_t* kw = static_cast<uint16_t*>(const_cast<void*>(p.k)) + tile + static_cast<size_t>(off) * kD;
        uint16_t* vw = static_cast<uint16_t*>(const_cast<void*>(p.v)) + tile + off;
        if (lane < kD / 8)
            *reinterpret_cast<uint4*>(kw + lane * 8) = __ldg(reinterpret_cast<const uint4*>(ks + lane * 8));
#pragma unroll
        for (int e = 0; e < kD / 32; ++e)
            vw[static_cast<size_t>(lane * (kD / 32) + e) * 16] = __ldg(vs + lane * (kD / 32) + e);
    }
}

template <bool F8, int NG>
__global__ void __launch_bounds__(tc_threads(F8), 1)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
    constexpr uint32_t SB = stage_bytes(F8);
    constexpr int kWidenK = 4, kWidenV = 8;                     // fp8: first warp of each widening group
    constexpr int kProd = F8 ? 12 : 4, kIssS = kProd + 1, kIssPV = kProd + 2;
    constexpr int kTmemCols = F8 ? 512 : 128;
    constexpr uint32_t kItemConsumers = F8 ? 14 : 6;            // warps that read each ring entry
    constexpr int kTmaPerBlock = F8 ? 2 : 3;                    // boxes per 16-token block
    static_assert(NG == 4 || NG == 8, "heads per group padded to 4 or 8");

    extern __shared__ unsigned char tc_raw[];
    const uint32_t raw_s = pa_tc::smem_u32(tc_raw);
    unsigned char* base = tc_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = pa_tc::smem_u32(base);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kMiscOff);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + kSlotOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + kSlotOff + 4);
    volatile int* s_item = reinterpret_cast<volatile int*>(base + kSlotOff + 16);      // [kRing]
    int* s_sched = reinterpret_cast<int*>(base + kSlotOff + 32);                        // PT, items, PTs, S_split
    long long* s_red = reinterpret_cast<long long*>(base + kSlotOff + 64);             // [4]
    volatile int* s_mask = reinterpret_cast<volatile int*>(base + kSlotOff + 128);     // [kMaskRing]
    float* s_wmax = reinterpret_cast<float*>(base + kWmaxOff);
    float* s_wl = reinterpret_cast<float*>(base + kWlOff);
    const int R = p.tc_stages;
    int* s_start = reinterpret_cast<int*>(base + kStageOff + static_cast<uint32_t>(R) * SB);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pa_dev::wait_prior_grid();
    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) {
            pa_tc::mbar_init(&bars[kItemFull + i], 1);
            pa_tc::mbar_init(&bars[kItemEmpty + i], kItemConsumers);
        }
        for (int i = 0; i < 2; ++i) {
            pa_tc::mbar_init(&bars[kQFull + i], 32);            // the producer's lanes
            pa_tc::mbar_init(&bars[kQEmpty + i], 1);
            pa_tc::mbar_init(&bars[kSFull + i], 1);
            pa_tc::mbar_init(&bars[kSEmpty + i], 4);            // one arrival per softmax warp
            pa_tc::mbar_init(&bars[kPFull + i], 4);
            pa_tc::mbar_init(&bars[kPEmpty + i], 1);
            pa_tc::mbar_init(&bars[kOFull + i], 1);
            pa_tc::mbar_init(&bars[kKwFull + i], 4);            // one arrival per widening warp
            pa_tc::mbar_init(&bars[kKwEmpty + i], 1);
            pa_tc::mbar_init(&bars[kVwFull + i], 4);
            pa_tc::mbar_init(&bars[kVwEmpty + i], 1);
            pa_tc::mbar_init(&bars[kMxFull + i], 4);
            pa_tc::mbar_init(&bars[kLFull + i], 4);
        }
        pa_tc::mbar_init(&bars[kMmaDone], 2);                   // both MMA-issuing warps
        for (int i = 0; i < kMaxStages; ++i) {
            pa_tc::mbar_init(&bars[kKvFull + i], 1);
            pa_tc::mbar_init(&bars[kKvEmpty + i], F8 ? 8 : 1);  // both widening groups / the P.V commit
        }
        *abort_flag = 0;
        pa_tc::mbar_init_fence();
    }
    // the Q and P buffers start zeroed: rows past the group's heads stay zero
    for (int i = tid; i < static_cast<int>(kMiscOff / 16); i += blockDim.x)
        reinterpret_cast<uint4*>(base)[i] = make_uint4(0u, 0u, 0u, 0u);
    pa_tc::fence_smem_to_async();
    if (warp == 0) pa_tc::tmem_alloc<kTmemCols>(tslot);
    if (warp == kProd && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&kmap) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&vmap) : "memory");
    }
    if (warp < kSchedWarps) {
        const Sched sc = build_schedule(p, s_start, s_red);
        publish_schedule(p, sc, s_start);
        if (tid == 0) {
            s_sched[0] = sc.PT;
            s_sched[1] = sc.total_items;
            s_sched[2] = sc.PTs;
            s_sched[3] = sc.S_split;
        }
    }
    pa_tc::fence_before_sync();
    __syncthreads();
    pa_tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    const Sched sc{s_sched[0], s_sched[1], s_sched[2], s_sched[3]};
    // TMEM: S buffer b at tS + 16 b; O buffer b at tO + 32 b (16 columns of the
    // high part's sums, then 16 of the low part's); fp8: widened K and V^T
    // tiles, 64 columns per buffer, two of each
    const uint32_t tS = tmem, tO = tmem + 32;
    const uint32_t tKw = tmem + 128, tVw = tmem + 256;
    bool ok = true;

    auto wait = [&](int bar, uint32_t parity) {
        return pa_tc::wait_or_abort(&bars[bar], parity, abort_flag, kWaitLimit);
    };
    // The next ring entry, for the warps that consume items.
    auto take_item = [&](uint32_t kk, int& item) {
        const int slot = static_cast<int>(kk % kRing);
        if (!wait(kItemFull + slot, (kk / kRing) & 1)) return false;
        item = s_item[slot];
        __syncwarp();
        if (lane == 0) pa_tc::arrive(&bars[kItemEmpty + slot]);
        return true;
    };

    if (warp == kProd) {
        // ------------------------------------------------------------ producer
        const uint16_t* qg = static_cast<const uint16_t*>(p.q);
        uint32_t kk = 0, ne = 0, kv_it = 0;
        int next = blockIdx.x;
        for (;;) {
            const int item = next < sc.total_items ? next : -1;
            const int slot = static_cast<int>(kk % kRing);
            if (kk >= kRing && !wait(kItemEmpty + slot, ((kk / kRing) - 1) & 1)) { ok = false; break; }
            if (lane == 0) s_item[slot] = item;
            __syncwarp();
            if (lane == 0) pa_tc::arrive(&bars[kItemFull + slot]);
            ++kk;
            if (item < 0) break;
            // the next ticket now: its round trip overlaps this item's loads
            int tk = 0;
            if (lane == 0) tk = atomicAdd(p.ticket, 1);
            const TcItem it = tc_item(p, sc, s_start, item);
            next = static_cast<int>(gridDim.x) + __shfl_sync(0xffffffffu, tk, 0);
            if (it.ntiles == 0) continue;
            // block ids of the item, 32 (four tiles) per load, each batch loaded
            // one batch ahead; INT_MIN marks slots past the item
            const int32_t* table = p.tables + static_cast<size_t>(it.s) * p.max_blocks;
            const int lb0 = it.tok0 >> 4, nblk = (it.tok1 - it.tok0 + 15) >> 4;
            auto load_ids = [&](int g) {
                const int bi = g * 32 + lane;
                return bi < nblk ? __ldg(table + lb0 + bi) : INT_MIN;
            };
            int ids_cur = load_ids(0);
            int ids_next = it.ntiles > 4 ? load_ids(1) : INT_MIN;
            // the group's query rows, once the item two back is done with the buffer
            const int qb = ne & 1;
            if (ne >= 2 && !wait(kQEmpty + qb, ((ne >> 1) - 1) & 1)) { ok = false; break; }
            unsigned char* qs = base + kQOff + qb * kQBytes;
            const uint16_t* qrow = qg + (static_cast<size_t>(it.s) * p.Hq + static_cast<size_t>(it.h) * p.G) * kD;
            for (int idx = lane; idx < p.G * 16; idx += 32) {
                const int n = idx >> 4, c16 = idx & 15;
                uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + n * kD + c16 * 8));
                if (F8) v = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                                       bf16x2_to_f16x2(v.w));
                *reinterpret_cast<uint4*>(qs + (c16 >> 3) * 2048 + pa_tc::sw128_off(n, c16 & 7)) = v;
            }
            pa_tc::fence_smem_to_async();                      // generic writes -> tensor core reads
            pa_tc::arrive(&bars[kQFull + qb]);
            ++ne;
            // the item's tiles: lane l stages box l / 8 of block l % 8 of each tile
            for (int j = 0; j < it.ntiles; ++j, ++kv_it) {
                if (j > 0 && (j & 3) == 0) {
                    ids_cur = ids_next;
                    ids_next = (j >> 2) + 1 < (it.ntiles + 3) >> 2 ? load_ids((j >> 2) + 1) : INT_MIN;
                }
                const int st = static_cast<int>(kv_it % static_cast<uint32_t>(R));
                const uint32_t use = kv_it / static_cast<uint32_t>(R);
                if (use > 0 && !wait(kKvEmpty + st, (use - 1) & 1)) { ok = false; break; }
                const int b = lane & 7;
                int id = __shfl_sync(0xffffffffu, ids_cur, (j & 3) * 8 + b);
                if (id != INT_MIN && (id < 0 || id >= p.num_blocks)) {
                    if (lane < 8) pa_dev::record_error(p.err, PA_ERR_BAD_BLOCK_ID);
                    id = INT_MIN;
                }
                const uint32_t loaded = __ballot_sync(0xffffffffu, lane < 8 && id != INT_MIN);
                if (p.new_slots && j == it.ntiles - 1 && it.tok1 == it.L) {
                    // pa_append_decode: this tile holds position L - 1, so the
                    // producer writes the sequence's new token (head h) first
                    const int lb = ((it.L - 1) >> 4) - lb0 - j * kTileBlocks;
                    const int phys = __shfl_sync(0xffffffffu, id, lb);
                    const int64_t new_slot = __ldg(p.new_slots + it.s);
                    const int off = (it.L - 1) & 15;
                    if (phys != INT_MIN && new_slot >= 0) {
                        if (new_slot != static_cast<int64_t>(phys) * 16 + off) {
                            if (lane == 0) pa_dev::record_error(p.err, PA_ERR_INVALID_ARG);
                        } else {
                            append_token<F8>(p, it.s, it.h, phys, off, lane);
                        }
                    }
                    // generic writes to global memory -> the TMA reads below
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                }
                uint64_t* full = &bars[kKvFull + st];
                if (lane == 0) {
                    s_mask[kv_it % kMaskRing] = static_cast<int>(loaded);
                    pa_tc::mbar_expect_tx(full, static_cast<uint32_t>(__popc(loaded)) * (F8 ? 4096u : 8192u));
                }
                __syncwarp();
                const int box = lane >> 3;
                if (box < kTmaPerBlock && id != INT_MIN) {
                    const uint32_t kst = sbase + kStageOff + static_cast<uint32_t>(st) * SB;
                    const int yk = (id * p.Hkv + it.h) * 16, yv = (id * p.Hkv + it.h) * kD;
                    if (F8) {
                        if (box == 0) pa_tc::tma_load_2d(kst + b * 2048, &kmap, 0, yk, full);            // 16 key rows
                        else pa_tc::tma_load_2d(kst + 16384 + b * 2048, &vmap, 0, yv, full);            // 128 value rows
                    } else {
                        if (box < 2) pa_tc::tma_load_2d(kst + box * 16384 + b * 2048, &kmap, box * 64, yk, full);
                        else pa_tc::tma_load_2d(kst + 32768 + b * 4096, &vmap, 0, yv, full);
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        // every copy issued must have landed before the CTA's shared memory is released
        for (int st = 0; st < R; ++st)
            if (kv_it > static_cast<uint32_t>(st))
                pa_tc::mbar_wait(&bars[kKvFull + st], ((kv_it - 1 - st) / static_cast<uint32_t>(R)) & 1,
                                 kWaitLimit);
    } else if (warp == kIssS) {
        // --------------------------------------------------------- S issue
        uint32_t kk = 0, ne = 0, kv_it = 0;
        for (;;) {
            int item;
            if (!take_item(kk, item)) { ok = false; break; }
            ++kk;
            if (item < 0) break;
            const TcItem it = tc_item(p, sc, s_start, item);
            if (it.ntiles == 0) continue;
            const int qb = ne & 1;
            if (!wait(kQFull + qb, (ne >> 1) & 1)) { ok = false; break; }
            ++ne;
            for (int j = 0; j < it.ntiles; ++j, ++kv_it) {
                const int sb = kv_it & 1;
                const int st = static_cast<int>(kv_it % static_cast<uint32_t>(R));
                const bool ready = F8 ? wait(kKwFull + sb, (kv_it >> 1) & 1)
                                      : wait(kKvFull + st, (kv_it / static_cast<uint32_t>(R)) & 1);
                if (!ready || (kv_it >= 2 && !wait(kSEmpty + sb, ((kv_it >> 1) - 1) & 1))) {
                    ok = false;
                    break;
                }
                pa_tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t qaddr = sbase + kQOff + qb * kQBytes;
                    const uint32_t kst = sbase + kStageOff + static_cast<uint32_t>(st) * SB;
#pragma unroll
                    for (int q = 0; q < kD / 16; ++q) {
                        const uint64_t b = pa_tc::sw128_desc(qaddr + (q >> 2) * 2048 + (q & 3) * 32);
                        if (F8)
                            pa_tc::mma_bf16_ta(tS + sb * kN, tKw + sb * 64 + q * 8, b, kIdescS16, q > 0);
                        else
                            pa_tc::mma_bf16(tS + sb * kN, pa_tc::sw128_desc(kst + (q >> 2) * 16384 + (q & 3) * 32),
                                            b, kIdescSbf, q > 0);
                    }
                    pa_tc::commit(&bars[kSFull + sb]);
                    if (F8) pa_tc::commit(&bars[kKwEmpty + sb]);
                    if (j == it.ntiles - 1) pa_tc::commit(&bars[kQEmpty + qb]);
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        // every MMA issued must be complete before TMEM is freed
        if (lane == 0) pa_tc::commit(&bars[kMmaDone]);
        __syncwarp();
        pa_tc::mbar_wait(&bars[kMmaDone], 0, kWaitLimit);
    } else if (warp == kIssPV) {
        // ------------------------------------------------------- P.V issue
        // One MMA per 16 tokens with N = 32: P^T's high part in rows 0-15 and
        // its low part in rows 16-31, so O^T gets both sums from one read of
        // the value tile.
        uint32_t kk = 0, ne = 0, kv_it = 0;
        for (;;) {
            int item;
            if (!take_item(kk, item)) { ok = false; break; }
            ++kk;
            if (item < 0) break;
            const TcItem it = tc_item(p, sc, s_start, item);
            if (it.ntiles == 0) continue;
            const int ob = ne & 1;
            ++ne;
            for (int j = 0; j < it.ntiles; ++j, ++kv_it) {
                const int pb = kv_it & 1;
                const int st = static_cast<int>(kv_it % static_cast<uint32_t>(R));
                bool ready = wait(kPFull + pb, (kv_it >> 1) & 1);
                ready = ready && (F8 ? wait(kVwFull + pb, (kv_it >> 1) & 1)
                                     : wait(kKvFull + st, (kv_it / static_cast<uint32_t>(R)) & 1));
                if (!ready) { ok = false; break; }
                pa_tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t pbuf = sbase + kPOff + pb * kPBytes;
                    const uint32_t vst = sbase + kStageOff + static_cast<uint32_t>(st) * SB + 32768;
#pragma unroll
                    for (int q = 0; q < kTile / 16; ++q) {
                        const uint64_t b = pa_tc::sw128_desc(pbuf + (q >> 2) * 4096 + (q & 3) * 32);
                        const bool acc = j > 0 || q > 0;
                        if (F8)
                            pa_tc::mma_bf16_ta(tO + ob * 32, tVw + pb * 64 + q * 8, b, kIdescPV16, acc);
                        else
                            pa_tc::mma_bf16(tO + ob * 32, pa_tc::sw32_desc(vst + q * 4096), b, kIdescPVbf, acc);
                    }
                    pa_tc::commit(F8 ? &bars[kVwEmpty + pb] : &bars[kKvEmpty + st]);
                    pa_tc::commit(&bars[kPEmpty + pb]);
                    if (j == it.ntiles - 1) pa_tc::commit(&bars[kOFull + ob]);
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (lane == 0) pa_tc::commit(&bars[kMmaDone]);
        __syncwarp();
        pa_tc::mbar_wait(&bars[kMmaDone], 0, kWaitLimit);
    } else if (F8 && warp >= kWidenK && warp < kWidenV + 4) {
        // ----------------------------------------------- widening (fp8 pool)
        // warps 4-7 widen key rows, warps 8-11 value rows; each group covers
        // the 128 TMEM lanes (a warp reaches the lane quarter warp % 4)
        const bool keys = warp < kWidenV;
        const int r = (warp & 3) * 32 + lane;                               // tile row = TMEM lane
        const uint32_t lane_sel = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int full_bar = keys ? kKwFull : kVwFull, empty_bar = keys ? kKwEmpty : kVwEmpty;
        const uint32_t tdst = keys ? tKw : tVw;
        uint32_t kk = 0, kv_it = 0;
        for (;;) {
            int item;
            if (!take_item(kk, item)) { ok = false; break; }
            ++kk;
            if (item < 0) break;
            const TcItem it = tc_item(p, sc, s_start, item);
            for (int j = 0; j < it.ntiles; ++j, ++kv_it) {
                const int st = static_cast<int>(kv_it % static_cast<uint32_t>(R));
                const int wb = kv_it & 1;
                if (!wait(kKvFull + st, (kv_it / static_cast<uint32_t>(R)) & 1) ||
                    (kv_it >= 2 && !wait(empty_bar + wb, ((kv_it >> 1) - 1) & 1))) {
                    ok = false;
                    break;
                }
                pa_tc::fence_after_sync();
                const unsigned char* stage = base + kStageOff + static_cast<uint32_t>(st) * SB;
                uint32_t w0[32], w1[32];
                if (keys) {
                    // key row r: 128 codes in the 128-byte swizzle (chunk c at c ^ (r % 8));
                    // codes of unloaded slots are left as they are: their scores are masked
                    const unsigned char* krow = stage + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        widen16(*reinterpret_cast<const uint4*>(krow + ((c ^ (r & 7)) << 4)), w0 + 8 * c);
#pragma unroll
                    for (int c = 4; c < 8; ++c)
                        widen16(*reinterpret_cast<const uint4*>(krow + ((c ^ (r & 7)) << 4)), w1 + 8 * (c - 4));
                } else {
                    // value row r (= head_dim index): tokens outside the item, or in
                    // blocks left unloaded, get +0 so that 0 * Inf never enters P.V
                    const int loaded = s_mask[kv_it % kMaskRing];
                    const int tb = it.tok0 + j * kTile;
#pragma unroll
                    for (int b = 0; b < kTileBlocks; ++b) {
                        const int nv = (loaded >> b) & 1 ? min(16, it.tok1 - (tb + 16 * b)) : 0;
                        const uint4 raw = *reinterpret_cast<const uint4*>(stage + 16384 + b * 2048 + r * 16);
                        if (b < 4) widen16(keep_codes(raw, nv), w0 + 8 * b);
                        else widen16(keep_codes(raw, nv), w1 + 8 * (b - 4));
                    }
                }
                pa_tc::tmem_st32u(tdst + wb * 64 + lane_sel, w0);
                pa_tc::tmem_st32u(tdst + wb * 64 + 32 + lane_sel, w1);
                pa_tc::tmem_wait_st();
                pa_tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    pa_tc::arrive(&bars[full_bar + wb]);
                    pa_tc::arrive(&bars[kKvEmpty + st]);              // this group is done with the raw stage
                }
            }
            if (!ok) break;
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------- softmax
        const int t = tid;                                                  // tile row = TMEM lane
        const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
        const float sl = p.scale_log2;
        uint32_t kk = 0, ne = 0, kv_it = 0, ex = 0;
        for (;;) {
            int item;
            if (!take_item(kk, item)) { ok = false; break; }
            ++kk;
            if (item < 0) break;
            const TcItem it = tc_item(p, sc, s_start, item);
            const int ob = ne & 1;
            const uint32_t od = tO + ob * 32 + lane_sel;
            float ref[NG], l[NG];
#pragma unroll
            for (int n = 0; n < NG; ++n) {
                ref[n] = -INFINITY;
                l[n] = 0.f;
            }
            for (int j = 0; j < it.ntiles; ++j, ++kv_it) {
                const int sb = kv_it & 1;
                const int st = static_cast<int>(kv_it % static_cast<uint32_t>(R));
                if (!wait(kSFull + sb, (kv_it >> 1) & 1) ||
                    (!F8 && !wait(kKvFull + st, (kv_it / static_cast<uint32_t>(R)) & 1))) {
                    ok = false;
                    break;
                }
                pa_tc::fence_after_sync();
                const int loaded = s_mask[kv_it % kMaskRing];
                float x[NG];
                pa_tc::tmem_ldn<NG>(tS + sb * kN + lane_sel, x);
                pa_tc::tmem_wait_ld();
                pa_tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) pa_tc::arrive(&bars[kSEmpty + sb]);      // S buffer free
                const int tok = it.tok0 + j * kTile + t;
                const bool valid = tok < it.tok1 && ((loaded >> (t >> 4)) & 1);
#pragma unroll
                for (int n = 0; n < NG; ++n) x[n] = valid ? x[n] * sl : -INFINITY;
                // the tile's maximum of each head: this warp's, then the four warps'
                float m[NG];
#pragma unroll
                for (int n = 0; n < NG; ++n) m[n] = warp_max(x[n]);
                float* wm = s_wmax + (kv_it & 1) * 64;
                if (lane == 0) {
#pragma unroll
                    for (int n = 0; n < NG; n += 4)
                        *reinterpret_cast<float4*>(wm + warp * 16 + n) = make_float4(m[n], m[n + 1], m[n + 2], m[n + 3]);
                    pa_tc::arrive(&bars[kMxFull + (kv_it & 1)]);
                }
                if (!wait(kMxFull + (kv_it & 1), (kv_it >> 1) & 1)) { ok = false; break; }
#pragma unroll
                for (int n = 0; n < NG; n += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(wm + n);
                    const float4 b = *reinterpret_cast<const float4*>(wm + 16 + n);
                    const float4 c = *reinterpret_cast<const float4*>(wm + 32 + n);
                    const float4 d = *reinterpret_cast<const float4*>(wm + 48 + n);
                    m[n] = fmaxf(fmaxf(a.x, b.x), fmaxf(c.x, d.x));
                    m[n + 1] = fmaxf(fmaxf(a.y, b.y), fmaxf(c.y, d.y));
                    m[n + 2] = fmaxf(fmaxf(a.z, b.z), fmaxf(c.z, d.z));
                    m[n + 3] = fmaxf(fmaxf(a.w, b.w), fmaxf(c.w, d.w));
                }
                // raise a head's reference only when it is unset or far behind
                // (every thread holds the same maxima, so the branch is uniform)
                bool raise_any = false;
                float corr[NG];
#pragma unroll
                for (int n = 0; n < NG; ++n) {
                    const bool first = ref[n] == -INFINITY;
                    const bool raise = !first && m[n] > ref[n] + 8.f;
                    corr[n] = raise ? pa_dev::ex2(ref[n] - m[n]) : 1.f;
                    if (first || raise) ref[n] = m[n];
                    raise_any |= raise;
                }
                if (raise_any) {
                    // O^T holds this item's sums up to the previous tile once its P.V is done
                    const uint32_t prev = kv_it - 1;
                    if (!wait(kPEmpty + (prev & 1), (prev >> 1) & 1)) { ok = false; break; }
                    pa_tc::fence_after_sync();
                    float oh[NG], ol[NG];
                    pa_tc::tmem_ldn<NG>(od, oh);
                    pa_tc::tmem_ldn<NG>(od + 16, ol);
                    pa_tc::tmem_wait_ld();
#pragma unroll
                    for (int n = 0; n < NG; ++n) {
                        oh[n] *= corr[n];
                        ol[n] *= corr[n];
                        l[n] *= corr[n];
                    }
                    pa_tc::tmem_stn<NG>(od, oh);
                    pa_tc::tmem_stn<NG>(od + 16, ol);
                    pa_tc::tmem_wait_st();
                }
                // this tile's P buffer was last read by the P.V two tiles back
                const int pb = kv_it & 1;
                if (kv_it >= 2 && !wait(kPEmpty + pb, ((kv_it >> 1) - 1) & 1)) { ok = false; break; }
                pa_tc::fence_after_sync();
                // weights into P^T (column t = token): the high part in row n, the low part in row 16 + n
                unsigned char* pbuf = base + kPOff + pb * kPBytes;
                const uint32_t col = static_cast<uint32_t>((t >> 6) * 4096 + (t & 7) * 2);
#pragma unroll
                for (int n = 0; n < NG; ++n) {
                    const float pr = pa_dev::ex2(x[n] - (ref[n] == -INFINITY ? 0.f : ref[n]));
                    l[n] += pr;
                    uint16_t hi, lo;
                    if (F8) {
                        const __half h = __float2half_rn(pr);
                        hi = __half_as_ushort(h);
                        lo = __half_as_ushort(__float2half_rn(pr - __half2float(h)));
                    } else {
                        const __nv_bfloat16 h = __float2bfloat16_rn(pr);
                        hi = __bfloat16_as_ushort(h);
                        lo = __bfloat16_as_ushort(__float2bfloat16_rn(pr - __bfloat162float(h)));
                    }
                    *reinterpret_cast<uint16_t*>(pbuf + col + pa_tc::sw128_off(n, (t & 63) >> 3)) = hi;
                    *reinterpret_cast<uint16_t*>(pbuf + col + pa_tc::sw128_off(16 + n, (t & 63) >> 3)) = lo;
                }
                // bf16: value columns of tokens outside the item or of unloaded
                // blocks get zeros (thread t clears value row t of each block)
                if (!F8 && (loaded != (1 << kTileBlocks) - 1 || it.tok0 + (j + 1) * kTile > it.tok1)) {
                    unsigned char* vt = base + kStageOff + static_cast<uint32_t>(st) * SB + 32768;
                    const int tb = it.tok0 + j * kTile;
#pragma unroll 1
                    for (int b = 0; b < kTileBlocks; ++b) {
                        const int zf = (loaded >> b) & 1 ? min(16, max(0, it.tok1 - (tb + 16 * b))) : 0;
                        if (zf < 16) pa_tc::zero_vt_row_tail(vt + b * 4096, t, zf);
                    }
                }
                pa_tc::fence_smem_to_async();
                pa_tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) pa_tc::arrive(&bars[kPFull + pb]);
            }
            if (!ok) break;
            // row sums: this warp's, then the four warps'
            float* wl = s_wl + (ex & 1) * 64;
            float lt[NG];
#pragma unroll
            for (int n = 0; n < NG; ++n) lt[n] = warp_sum(l[n]);
            if (lane == 0) {
#pragma unroll
                for (int n = 0; n < NG; n += 4)
                    *reinterpret_cast<float4*>(wl + warp * 16 + n) = make_float4(lt[n], lt[n + 1], lt[n + 2], lt[n + 3]);
                pa_tc::arrive(&bars[kLFull + (ex & 1)]);
            }
            if (!wait(kLFull + (ex & 1), (ex >> 1) & 1)) { ok = false; break; }
            ++ex;
#pragma unroll
            for (int n = 0; n < NG; n += 4) {
                const float4 a = *reinterpret_cast<const float4*>(wl + n);
                const float4 b = *reinterpret_cast<const float4*>(wl + 16 + n);
                const float4 c = *reinterpret_cast<const float4*>(wl + 32 + n);
                const float4 d = *reinterpret_cast<const float4*>(wl + 48 + n);
                lt[n] = (a.x + b.x) + (c.x + d.x);
                lt[n + 1] = (a.y + b.y) + (c.y + d.y);
                lt[n + 2] = (a.z + b.z) + (c.z + d.z);
                lt[n + 3] = (a.w + b.w) + (c.w + d.w);
            }
            float o[NG];
#pragma unroll
            for (int n = 0; n < NG; ++n) o[n] = 0.f;
            if (it.ntiles > 0) {
                if (!wait(kOFull + ob, (ne >> 1) & 1)) { ok = false; break; }
                pa_tc::fence_after_sync();
                float ol[NG];
                pa_tc::tmem_ldn<NG>(od, o);
                pa_tc::tmem_ldn<NG>(od + 16, ol);
                pa_tc::tmem_wait_ld();
                pa_tc::fence_before_sync();
#pragma unroll
                for (int n = 0; n < NG; ++n) o[n] += ol[n];
                ++ne;
            }
            // thread t holds O^T row d = t: element d of every head
            if (it.direct) {
                const size_t out0 =
                    (static_cast<size_t>(it.s) * p.Hq + static_cast<size_t>(it.h) * p.G) * kD + t;
#pragma unroll
                for (int n = 0; n < NG; ++n)
                    if (n < p.G) store_out(p, out0 + static_cast<size_t>(n) * kD, lt[n] > 0.f ? o[n] * p.v_scale / lt[n] : 0.f);
            } else {
                float* pacc = p.part_acc + static_cast<size_t>(item) * p.G * kD + t;
#pragma unroll
                for (int n = 0; n < NG; ++n)
                    if (n < p.G) pacc[static_cast<size_t>(n) * kD] = o[n] * p.v_scale;
#pragma unroll
                for (int n = 0; n < NG; ++n)
                    if (n < p.G && t == n) {
                        p.part_ml[(static_cast<size_t>(item) * p.G + n) * 2] = ref[n];
                        p.part_ml[(static_cast<size_t>(item) * p.G + n) * 2 + 1] = lt[n];
                    }
            }
        }
    }
    if (!ok) {
        *abort_flag = 1;
        if (lane == 0) pa_dev::record_error(p.err, PA_ERR_CUDA);
    }
    pa_tc::fence_before_sync();
    __syncthreads();
    pa_tc::fence_after_sync();
    if (warp == 0) pa_tc::tmem_free<kTmemCols>(tmem);
    pa_dev::allow_next_grid();
    retire_cta(p);
}

size_t tc_smem(bool f8, int stages, int S) {
    return 1024 + kStageOff + static_cast<size_t>(stages) * stage_bytes(f8) +
           static_cast<size_t>(S + 1) * sizeof(int);
}

template <bool F8>
int launch_ng(const DecodeParams& p, int G, dim3 grid, size_t smem, const CUtensorMap& km,
              const CUtensorMap& vm, cudaStream_t st) {
    void (*k)(DecodeParams, CUtensorMap, CUtensorMap) = G <= 4 ? decode_tc_kernel<F8, 4> : decode_tc_kernel<F8, 8>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    const cudaError_t e = pa_detail::launch_pdl(k, grid, dim3(tc_threads(F8)), smem, st, p, km, vm);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

namespace pa_detail {

bool decode_tc_eligible(const pa_pool* pool, int G) {
    // TMA coordinates are 32-bit: value rows num_blocks * Hkv * D must stay below 2^31
    return (pool->dtype == PA_BF16 || pool->dtype == PA_FP8E4M3) && pool->head_dim == kD &&
           pool->block_size == 16 && G >= 1 && G <= 8 &&
           static_cast<long long>(pool->num_blocks) * pool->kv_heads * kD < (1LL << 31);
}

// Stages that fit beside the schedule of S sequences (0: none do).
int decode_tc_stages(const pa_pool* pool, int S) {
    const bool f8 = pool->dtype == PA_FP8E4M3;
    for (int r = kMaxStages; r >= 2; --r) {
        if (!f8 && r > 3) continue;              // 3 bf16 stages already keep 192 KB in flight
        if (tc_smem(f8, r, S) <= static_cast<size_t>(pool->smem_optin)) return r;
    }
    return 0;
}

void plan_decode_tc(const pa_pool* pool, int S, int stages, DecodePlan* plan) {
    const bool f8 = pool->dtype == PA_FP8E4M3;
    plan->tcd = true;
    plan->tc_stages = stages;
    plan->grid = pool->num_sms;
    plan->threads = tc_threads(f8);
    // at least half an SM's shared memory, so that one CTA holds each SM (the
    // fp8 form's 512 TMEM columns are the whole SM's)
    plan->smem = std::max(tc_smem(f8, stages, S), static_cast<size_t>(pool->smem_optin) / 2 + 1024);
    plan->items_target = plan->grid * kItemsPerCta;
    plan->pt_min = kTile;                        // no partition shorter than one tile
    // partitions of at most 2048 tokens (16 tiles) whatever the batch: with one
    // CTA per SM, longer items leave the launch a long tail
    plan->pt_max = pool->opt_partition_cap >= 0 ? (pool->opt_partition_cap > 0 ? std::max(kTile, pool->opt_partition_cap / 16 * 16) : 0)
                                                : kPtCap;
}

size_t decode_tc_extra_items(const DecodePlan& plan) {
    // room for the partition cap and the guided tail on long contexts
    return static_cast<size_t>(3) * plan.items_target;
}

// TMA descriptors over an fp8 pool (16-token blocks): K codes as
// [num_blocks*Hkv*16 rows][128] with 128 x 16 boxes (128-byte swizzle); V^T
// codes as [num_blocks*Hkv*128 rows][16] with 16 x 128 boxes.
static int ensure_tensor_maps_f8(pa_pool* pool) {
    if (pool->tmaps8_ready) return PA_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return PA_ERR_CUDA;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    const cuuint64_t rows_k = static_cast<cuuint64_t>(pool->num_blocks) * pool->kv_heads * 16;
    const cuuint64_t rows_v = static_cast<cuuint64_t>(pool->num_blocks) * pool->kv_heads * kD;
    const cuuint64_t kdim[2] = {static_cast<cuuint64_t>(kD), rows_k};
    const cuuint64_t kstr[1] = {static_cast<cuuint64_t>(kD)};
    const cuuint32_t kbox[2] = {static_cast<cuuint32_t>(kD), 16};
    const cuuint64_t vdim[2] = {16, rows_v};
    const cuuint64_t vstr[1] = {16};
    const cuuint32_t vbox[2] = {16, static_cast<cuuint32_t>(kD)};
    const cuuint32_t one[2] = {1, 1};
    if (encode(&pool->kmap8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pool->k, kdim, kstr, kbox, one,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    if (encode(&pool->vmap8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pool->v, vdim, vstr, vbox, one,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    pool->tmaps8_ready = true;
    return PA_OK;
}

int launch_decode_tc(pa_pool* pool, const DecodePlan& plan, const DecodeParams& prm, cudaStream_t st) {
    DecodeParams p = prm;
    p.tc_stages = plan.tc_stages;
    const bool f8 = pool->dtype == PA_FP8E4M3;
    const int rc = f8 ? ensure_tensor_maps_f8(pool) : ensure_tensor_maps(pool);
    if (rc != PA_OK) return rc;
    const int e = f8 ? launch_ng<true>(p, p.G, dim3(plan.grid), plan.smem, pool->kmap8, pool->vmap8, st)
                     : launch_ng<false>(p, p.G, dim3(plan.grid), plan.smem, pool->kmap, pool->vmap, st);
    count_launch();
    return e;
}

}  // namespace pa_detail
