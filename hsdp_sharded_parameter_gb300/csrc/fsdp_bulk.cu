// The fused gradient sync on a capped grid, fed by TMA bulk loads.
//
// What it computes is the fused reduce's definition ([FS-RFC §2.1.3 item 3,
// §3.3]: ReduceScatter over the shard group, then AllReduce over the
// replicate group, into the 512-byte-aligned fused regions of [OVERLAP
// §二.1]; with the apply folded in, [OVERLAP §二.3] SUM-then-divide and the
// back-fill of the actual shard rows of [RAGGED §6.4]): for every element of
// every shard row, the W gradients summed in fp32, shard group first, from
// the first term, in ascending order, written to all D replicas.
//
// When the backward's GEMMs keep most SMs (fsdp_plan_set_grid_limit caps
// the sync at a few blocks), the sync must pull HBM bandwidth from few SMs.
// One block per SM is split by role:
//   * a producer warp walks the plan's run table chunk by chunk (a chunk is
//     one 2048-element warp tile of a run); per chunk each of its lanes
//     announces and issues one `cp.async.bulk` global -> shared copy, of its
//     own source, completing on the stage's mbarrier (transaction bytes);
//   * one or two groups of eight consumer warps wait for the stage, fold
//     one 8-element granule per thread straight from shared memory into
//     registers, release the stage to the producer through a second
//     mbarrier, then store the fp32 sums (and the applied, rounded shard
//     gradients) from registers; a chunk's record (pointers, shifts) lives
//     in a ring of its own, so it outlasts the data slot.
// The shared memory holds as many stages as fit (3 for 16 bf16 sources, 6
// for 8), so up to ~200 KB per SM stay in flight without registers. On one
// GB300, a probe of this layout (8 bf16 sources into 2 fp32 destinations,
// contiguous, nothing but the fold) measured ~90-97 GB/s per SM with the
// copies issued by 8 lanes, against ~60 GB/s per SM with one issuing thread
// and ~61 GB/s per SM with cp.async from the producer warp; this kernel
// moves ~76 GB/s per SM with 8 sources and ~92 with 16 (64 SMs: 0.72 and
// 0.87 of the measured copy peak), against ~30-67 for per-warp cp.async
// rings.
//
// Every wait is bounded: a wait that runs past KArgs::wait_ns sets a bit in
// the plan's status word (fsdp_plan_status reads it), raises the block's
// abort flag, and the block leaves after the producer has waited (bounded
// too) for the copies it issued, so no copy lands in a block that has
// exited.
//
// Sources, by page title + section:
//   [OVERLAP] "Hyper通信掩盖方案" (hyper-parallel issue 184), PR #758 write-up
//   [RAGGED]  FSDP dim-0 uneven-sharding RFC (hyper-parallel issue 319)
//   [FS-RFC]  "【RFC】FullyShard 多维并行适配设计方案" (hyper-parallel issue 1)
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <set>
#include <unordered_map>
#include <utility>

#include "fsdp_device.cuh"

namespace fsdp {
namespace {

// A block is one producer warp plus G groups of 8 consumer warps (one
// granule per thread per chunk); with two groups they take alternate
// chunks. Two groups where at least 4 stages fit (up to 8 bf16 sources)
// and at most 2 replicas: measured on one GB300 at 64 SMs, the one-pass
// sync of the HSDP (2,4) layer 0.503 -> 0.658 of the measured copy peak;
// with 16 sources only two stages would be left (large (2,8) layer 0.744 ->
// 0.582), so one group.
constexpr int kBulkConsumers = 8;  // warps of one group
template <int G>
__host__ __device__ constexpr int bulk_threads() {
    return (G * kBulkConsumers + 1) * 32;
}
static_assert(kBulkConsumers * 32 * kGran == kWarpTile, "a chunk is one warp tile");
constexpr size_t kBulkSmem = 224 * 1024;  // ring + chunk records + barriers
constexpr int kBulkMaxStages = 12;
constexpr int kBulkMaxSources = 32;  // one issuing lane per source
constexpr int kBulkMaxDests = 32;    // one lane per replica

// What the producer tells the consumers about one chunk.
struct alignas(16) ChunkRecord {
    int64_t t;     // the chunk (checked by the consumers before they store)
    int64_t n;     // elements of the run
    int64_t rel0;  // run-relative element of thread 0's first granule (< 0 by the destination's phase)
    int64_t lo;    // first element of the run the stage holds (max(rel0, 0))
    int32_t p;     // parameter, < 0 for a run of zeros
    int32_t ushift;  // the shift every source shares (0..15), or -1
    int32_t pad[2];
    int32_t shift[kBulkMaxSources];  // bytes from source i's slot to element lo
    float* dst[kBulkMaxDests];       // replica j's fused row at the run's first element
    void* grad[kBulkMaxDests];       // replica j's actual-shard gradient (apply folded in)
};

// One source's slot of a stage: a chunk, one 16-byte block wider when
// shifted, rounded to 128 bytes so every slot (the bulk copies' destination)
// starts on a 128-byte boundary.
template <typename S>
__host__ __device__ constexpr size_t bulk_slot() {
    return ((size_t)kWarpTile * sizeof(S) + 16 + 127) / 128 * 128;
}
// The ring: per stage its data slots (one per source) and two mbarriers;
// nst + 2 chunk records (a chunk's record outlives its data slot, see the
// consumer loop).
template <typename S>
__host__ __device__ constexpr int bulk_stages_fit(int ns) {
    return (int)((kBulkSmem - 2 * sizeof(ChunkRecord)) / ((size_t)ns * bulk_slot<S>() + sizeof(ChunkRecord) + 16));
}
// As many stages as fit (at most kBulkMaxStages), a multiple of the number
// of consumer groups G: stage s then always serves group s % G, so a group
// waits on each of its stages' phases in order. (A parity wait can only
// tell a phase from the one before it; with alternating groups on an odd
// ring a group could wait on a stage whose previous phase, the other
// group's chunk, had not completed, and pass at once.)
template <typename S, int G>
__host__ __device__ constexpr int bulk_stages(int ns) {
    return ((bulk_stages_fit<S>(ns) > kBulkMaxStages ? kBulkMaxStages : bulk_stages_fit<S>(ns)) / G) * G;
}
template <typename S>
__host__ __device__ constexpr size_t bulk_smem(int ns, int nst) {
    return (size_t)nst * ((size_t)ns * bulk_slot<S>() + 16) + (size_t)(nst + 2) * sizeof(ChunkRecord);
}

// --------------------------------------------------------------- mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(b)) : "memory");
}
// One arrival that also announces `tx` bytes the stage's copies will bring.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t tx) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(b)),
                 "r"(tx)
                 : "memory");
}
// Whether the phase of parity `par` has completed (one bounded hardware
// wait, no spinning inside).
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(par)
        : "memory");
    return ok != 0;
}
// Waits for the phase of parity `par`: false once `limit_ns` has passed or
// the block's abort flag is raised.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t par, const volatile int* abort, uint64_t limit_ns) {
    if (mbar_test(b, par)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_test(b, par)) return true;
        if (*abort || global_ns() - t0 > limit_ns) return false;
    }
    return false;
}
// Global -> shared bulk copy completing on mbarrier b (both addresses and
// the size multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(sdst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(b))
                 : "memory");
}

__device__ __forceinline__ void fail(const KArgs& a, int bit, volatile int* abort) {
    atomicOr(a.status, bit);
    *abort = 1;
}

// ------------------------------------------------------------------ fold

// The 8 elements at byte offset `off` of a stage slot (any element-aligned
// offset; the slot holds every byte read).
template <typename S>
__device__ __forceinline__ void slot_read(const char* slot, uint32_t off, Raw<S>& r) {
    const uint4* q = reinterpret_cast<const uint4*>(slot + (off & ~15u));
    const unsigned sh = off & 15u;
    if (sh == 0) {
#pragma unroll
        for (int v = 0; v < Raw<S>::kVec; ++v) put(r.w + 4 * v, q[v]);
    } else {
        uint4 blk[Raw<S>::kVec + 1];
#pragma unroll
        for (int v = 0; v <= Raw<S>::kVec; ++v) blk[v] = q[v];
#pragma unroll
        for (int v = 0; v < Raw<S>::kVec; ++v) put(r.w + 4 * v, funnel(blk[v], blk[v + 1], sh));
    }
}

// part = the granule of the group's first term, widened.
__device__ __forceinline__ void fold_first(const Raw<uint16_t>& r, float (&part)[8]) { widen(r, part); }
__device__ __forceinline__ void fold_first(const Raw<float>& r, float (&part)[8]) { widen(r, part); }
// part[e] += term e: one IEEE binary32 round-to-nearest-even addition each.
// For bf16 terms the mixed-precision add takes the bf16 operand directly
// (it is widened exactly, so the sum is the same as with the fp32 operand).
__device__ __forceinline__ void fold_add(const Raw<uint16_t>& r, float (&part)[8]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        unsigned short lo, hi;
        asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(r.w[q]));
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(part[2 * q]) : "h"(lo));
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(part[2 * q + 1]) : "h"(hi));
    }
}
__device__ __forceinline__ void fold_add(const Raw<float>& r, float (&part)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) part[e] = __fadd_rn(part[e], __uint_as_float(r.w[e]));
}


// The fixed-order fold of one granule: d_out groups of s_in terms (source
// i = d * s_in + s at `shift[i] + eoff` bytes into its slot; shift ==
// nullptr: at eoff, a multiple of 16), each group summed from its first
// term, then the groups from the first group. Compile-time counts (DOUT,
// SIN > 0) unroll it; 0 reads the arguments.
template <typename S, int DOUT, int SIN>
__device__ __forceinline__ void fold_granule(const char* slots, const int32_t* shift, uint32_t eoff, int d_out,
                                             int s_in, float (&total)[8]) {
    constexpr size_t kSlot = bulk_slot<S>();
    if constexpr (DOUT > 0) {
        if (shift == nullptr) {
            // every source at the same 16-byte phase as the granule: aligned
            // reads at fixed offsets from slot 0
#pragma unroll
            for (int d = 0; d < DOUT; ++d) {
                float part[8];
#pragma unroll
                for (int s = 0; s < SIN; ++s) {
                    const uint4* q = reinterpret_cast<const uint4*>(slots + (size_t)(d * SIN + s) * kSlot + eoff);
                    Raw<S> r;
#pragma unroll
                    for (int v = 0; v < Raw<S>::kVec; ++v) put(r.w + 4 * v, q[v]);
                    if (s == 0)
                        fold_first(r, part);
                    else
                        fold_add(r, part);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) total[e] = d == 0 ? part[e] : __fadd_rn(total[e], part[e]);
            }
            return;
        }
#pragma unroll
        for (int d = 0; d < DOUT; ++d) {
            float part[8];
#pragma unroll
            for (int s = 0; s < SIN; ++s) {
                const int i = d * SIN + s;
                Raw<S> r;
                slot_read<S>(slots + (size_t)i * kSlot, (uint32_t)shift[i] + eoff, r);
                if (s == 0)
                    fold_first(r, part);
                else
                    fold_add(r, part);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) total[e] = d == 0 ? part[e] : __fadd_rn(total[e], part[e]);
        }
    } else {
#pragma unroll 1
        for (int d = 0; d < d_out; ++d) {
            float part[8];
#pragma unroll 1
            for (int s = 0; s < s_in; ++s) {
                const int i = d * s_in + s;
                Raw<S> r;
                slot_read<S>(slots + (size_t)i * kSlot, (uint32_t)shift[i] + eoff, r);
                if (s == 0)
                    fold_first(r, part);
                else
                    fold_add(r, part);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) total[e] = d == 0 ? part[e] : __fadd_rn(total[e], part[e]);
        }
    }
}

template <typename S, int NS, int SIN, int ND, bool AP, int G>
__global__ void __launch_bounds__(bulk_threads<G>(), 1) rs_ar_reduce_bulk_kernel(const KArgs a, int nst) {
    extern __shared__ __align__(128) char smem[];
    __shared__ int abort_flag;
    const int ns = NS > 0 ? NS : a.W;
    const int s_in = SIN > 0 ? SIN : a.S;
    const int nd = ND > 0 ? ND : a.D;
    const int d_out = ns / s_in;
    constexpr size_t kSlot = bulk_slot<S>();
    char* ring = smem;
    // chunk q's record is records[q % (nst + 2)]
    ChunkRecord* records = reinterpret_cast<ChunkRecord*>(smem + (size_t)nst * ns * kSlot);
    uint64_t* full = reinterpret_cast<uint64_t*>(records + nst + 2);
    uint64_t* empty = full + nst;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < nst; ++s) {
            mbar_init(full + s, ns);  // one arrival per source lane
            mbar_init(empty + s, kBulkConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    const uint64_t limit = a.wait_ns;

    if (warp == G * kBulkConsumers) {
        // ---------------------------------------------------- producer warp
        // The run of the current chunk stays in registers (its tile range,
        // record, and each lane's source, fused-row and gradient pointer,
        // and the sources' 16-byte phases): consecutive chunks of a block
        // mostly share a run, and a chunk of a known run then needs no
        // global load and no exchange between lanes. Each source lane
        // announces its own copy's bytes on the stage's barrier (it counts
        // one arrival per source) and issues the copy.
        int stage = 0, k = 0, rec = 0;
        uint32_t ph = 0, armed = 0, armed_par = 0;  // per stage: copies issued, and their phase
        bool first = true;
        int64_t run_first = 0, run_end = -1, n = 0, src_off = 0, phase = 0;
        int p = -1;
        const char* my_src = nullptr;  // source `lane` of the run
        float* my_dst = nullptr;       // replica `lane`'s fused row at the run
        void* my_grad = nullptr;       // replica `lane`'s actual-shard gradient
        // the shift every source shares (or -1), at the run's first chunk
        // (which starts at element 0) and at its later chunks (which start
        // whole 16-byte blocks apart)
        int32_t u_first = 0, u_rest = 0;
        for (int64_t t = blockIdx.x; t < a.ntiles; t += gridDim.x) {
            if (t >= run_end) {
                k = find_seg(a.tile_begin, a.tile_run, a.nseg, k, t);
                const Seg sg = a.segs[k];
                run_first = __ldg(a.tile_begin + k);
                run_end = __ldg(a.tile_begin + k + 1);
                n = sg.n;
                src_off = sg.src_off;
                p = sg.p;
                phase = ((sg.dst_off * 4) & 15) / 4;  // the fused row's 16-byte phase at the run
                my_src = (p >= 0 && lane < ns) ? static_cast<const char*>(a.src_tab[(int64_t)lane * a.P + p]) : nullptr;
                my_dst = lane < nd ? static_cast<float*>(a.dst_tab[lane * a.S + sg.row]) + sg.dst_off : nullptr;
                my_grad = (AP && p >= 0 && lane < nd) ? a.sg_tab[(int64_t)(lane * a.S + sg.row) * a.P + p] : nullptr;
                const uint32_t sf = my_src ? (uint32_t)((reinterpret_cast<uintptr_t>(my_src) +
                                                         (uintptr_t)(src_off * (int64_t)sizeof(S))) & 15u)
                                           : 0u;
                const uint32_t sr = my_src ? (uint32_t)((reinterpret_cast<uintptr_t>(my_src) +
                                                         (uintptr_t)((src_off - phase) * (int64_t)sizeof(S))) & 15u)
                                           : 0u;
                const uint32_t sf0 = __shfl_sync(kFull, sf, 0), sr0 = __shfl_sync(kFull, sr, 0);
                u_first = __all_sync(kFull, lane >= ns || sf == sf0) ? (int32_t)sf0 : -1;
                u_rest = __all_sync(kFull, lane >= ns || sr == sr0) ? (int32_t)sr0 : -1;
            }
            const int64_t rel0 = (t - run_first) * kWarpTile - phase;
            const int64_t lo = rel0 < 0 ? 0 : rel0;
            const int64_t hi = rel0 + kWarpTile < n ? rel0 + kWarpTile : n;
            uintptr_t g0 = 0;
            uint32_t bytes = 0, shift = 0;
            if (my_src) {
                // the 16-byte blocks holding elements [lo, hi) of source `lane`
                const uintptr_t b = reinterpret_cast<uintptr_t>(my_src) + (uintptr_t)((src_off + lo) * (int64_t)sizeof(S));
                g0 = b & ~(uintptr_t)15;
                bytes = (uint32_t)(((b + (uintptr_t)((hi - lo) * (int64_t)sizeof(S)) + 15) & ~(uintptr_t)15) - g0);
                shift = (uint32_t)(b - g0);
            }
            if (!mbar_wait(empty + stage, ph ^ 1u, abort, limit)) {
                if (lane == 0) fail(a, kStatusProducerWait, abort);
                break;
            }
            ChunkRecord& m = records[rec];
            if (++rec == nst + 2) rec = 0;
            if (lane < ns) m.shift[lane] = (int32_t)shift;
            if (lane < nd) {
                m.dst[lane] = my_dst;
                m.grad[lane] = my_grad;
            }
            if (lane == 0) {
                m.t = t;
                m.n = n;
                m.rel0 = rel0;
                m.lo = lo;
                m.p = p;
                m.ushift = t == run_first ? u_first : u_rest;
            }
            // the failure-detection hook: block 0 never announces its first
            // chunk, so the consumers' wait for it runs out
            const bool hold = a.stall && first && blockIdx.x == 0;
            first = false;
            if (!hold) {
                // each source lane's arrival releases its own writes of the
                // record (lane 0 wrote the scalars; every replica lane is a
                // source lane, nd <= ns)
                if (lane < ns) {
                    if (bytes) {
                        mbar_arrive_tx(full + stage, bytes);
                        bulk_load(ring + ((size_t)stage * ns + lane) * kSlot, reinterpret_cast<const void*>(g0), bytes,
                                  full + stage);
                    } else {
                        mbar_arrive(full + stage);
                    }
                }
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (ph << stage);
            }
            if (++stage == nst) {
                stage = 0;
                ph ^= 1u;
            }
        }
        // After an abort the consumers may not take what was issued: wait
        // (bounded) until every issued copy has landed before leaving.
        if (*abort && lane == 0) {
            for (int s = 0; s < nst; ++s) {
                if (!((armed >> s) & 1u)) continue;
                const uint64_t t0 = global_ns();
                for (uint32_t it = 0; it < (1u << 30); ++it)
                    if (mbar_test(full + s, (armed_par >> s) & 1u) || global_ns() - t0 > limit) break;
            }
        }
        return;
    }

    // ------------------------------------------------------ consumer warps
    // Each thread folds its granule of the chunk into registers, then the
    // warp releases the data slot and stores. The chunk's record (pointers)
    // is still read after the release: the producer rewrites record q % (nst
    // + 2) for chunk q + nst + 2 only once chunk q + 2 (the stage's previous
    // chunk) has been released, by the group that took chunk q, which had
    // finished chunk q by then.
    // Group g takes the block's chunks g, g + G, ...: stages g, g + G, ...
    // of the ring (nst is a multiple of G).
    const int group = warp / kBulkConsumers;
    const int tid = threadIdx.x - group * kBulkConsumers * 32;  // 0 .. 255: granule of the chunk
    int stage = group, rec = group;
    uint32_t ph = 0;
    for (int64_t t = blockIdx.x + (int64_t)group * gridDim.x; t < a.ntiles; t += (int64_t)G * gridDim.x) {
        if (!mbar_wait(full + stage, ph, abort, limit)) {
            if (lane == 0) fail(a, kStatusConsumerWait, abort);
            break;
        }
        const ChunkRecord& m = records[rec];
        if ((rec += G) >= nst + 2) rec -= nst + 2;
        if (m.t != t) {
            // not this chunk's record: stop before storing anything
            if (lane == 0) fail(a, kStatusOrder, abort);
            break;
        }
        const char* slots = ring + (size_t)stage * ns * kSlot;
        const int64_t n = m.n, lo = m.lo;
        const int64_t rel = m.rel0 + (int64_t)tid * kGran;
        const int pm = m.p;
        // 0: nothing of the run here; 1: a full granule to 16-byte aligned
        // destinations; 2: element by element (a run's head or tail, or
        // unaligned destinations)
        const int kind = (rel >= n || rel + kGran <= 0) ? 0 : ((a.vec && rel >= 0 && rel + kGran <= n) ? 1 : 2);
        const int64_t e0 = rel < 0 ? 0 : rel;
        const int64_t e1 = rel + kGran < n ? rel + kGran : n;
        float total[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) total[e] = 0.0f;
        if (kind == 1 && pm >= 0) {
            const uint32_t eoff = (uint32_t)((rel - lo) * (int64_t)sizeof(S));
            // (rel - lo) is a whole number of granules unless the chunk
            // starts a run whose destination is off the 16-byte grid
            const bool aligned = m.ushift == 0 && (eoff & 15u) == 0;
            if constexpr (ND > 0 && SIN > 0)
                fold_granule<S, ND, SIN>(slots, aligned ? nullptr : m.shift, eoff, ND, SIN, total);
            else
                fold_granule<S, 0, 0>(slots, m.shift, eoff, d_out, s_in, total);
        } else if (kind == 2 && pm >= 0) {
#pragma unroll
            for (int q = 0; q < kGran; ++q) {
                const int64_t e = rel + q;
                if (e < e0 || e >= e1) continue;
                const uint32_t eoff = (uint32_t)((e - lo) * (int64_t)sizeof(S));
                float v = 0.0f;
                for (int d = 0; d < d_out; ++d) {
                    float part = 0.0f;
                    for (int s = 0; s < s_in; ++s) {
                        const int i = d * s_in + s;
                        const float x = load_f32(
                            reinterpret_cast<const S*>(slots + (size_t)i * kSlot + (uint32_t)m.shift[i] + eoff), 0);
                        part = s == 0 ? x : __fadd_rn(part, x);
                    }
                    v = d == 0 ? part : __fadd_rn(v, part);
                }
                total[q] = v;
            }
        }
        // every lane's reads of the slot are done: release it
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + stage);
        if ((stage += G) >= nst) {
            stage -= nst;
            ph ^= 1u;
        }
        if (kind == 1) {
            if constexpr (AP) {
                if (pm >= 0)
                    for (int j = 0; j < nd; ++j) store_applied(a, total, static_cast<S*>(m.grad[j]) + rel);
            }
            Raw<float> o;
            narrow(total, o);
            for (int j = 0; j < nd; ++j) store_raw(m.dst[j] + rel, o);
        } else if (kind == 2) {
#pragma unroll
            for (int q = 0; q < kGran; ++q) {
                const int64_t e = rel + q;
                if (e < e0 || e >= e1) continue;
                const float v = total[q];
                if constexpr (AP) {
                    if (pm >= 0) {
                        const float q = a.div != 1.0f ? scaled(v, a) : v;
                        for (int j = 0; j < nd; ++j) {
                            S* g = static_cast<S*>(m.grad[j]);
                            float x = q;
                            if (a.accumulate) x = __fadd_rn(load_f32(g, e), x);
                            store_f32(g, e, x);
                        }
                    }
                }
                for (int j = 0; j < nd; ++j) m.dst[j][e] = v;
            }
        }
    }
}

// SM count of the current device, cached per device (the same query as the
// step kernels' launcher makes; kept here so this file stands alone).
int bulk_sm_count() {
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return cache.emplace(dev, v > 0 ? v : 1).first->second;
}

template <typename S, int NS, int SIN, int ND, bool AP, int G>
cudaError_t go_bulk(const KArgs& a, cudaStream_t st) {
    auto kernel = rs_ar_reduce_bulk_kernel<S, NS, SIN, ND, AP, G>;
    const int nst = bulk_stages<S, G>(a.W);
    const size_t smem = bulk_smem<S>(a.W, nst);
    {
        // the dynamic shared memory limit, raised once per device and kernel
        static std::mutex mu;
        static std::set<std::pair<int, const void*>> done;
        int dev = 0;
        cudaGetDevice(&dev);
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_pair(dev, reinterpret_cast<const void*>(kernel));
        if (!done.count(key)) {
            const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem);
            if (e != cudaSuccess) return e;
            done.insert(key);
        }
    }
    int64_t grid = a.max_grid < bulk_sm_count() ? a.max_grid : bulk_sm_count();
    if (grid > a.ntiles) grid = a.ntiles;
    kernel<<<(int)grid, bulk_threads<G>(), smem, st>>>(a, nst);
    return cudaGetLastError();
}

// Two consumer groups where the ring holds at least two stages per group
// and there are at most two replicas (with 8 replicas, the pure-TP layer,
// one group measured faster: 0.529 against 0.408 of the measured copy peak
// on 64 SMs).
#ifndef FSDP_BULK_GROUPS
#define FSDP_BULK_GROUPS 0  // 0: by the rule above; 1 or 2: always that many
#endif
template <typename S, int NS, int SIN, int ND, bool AP>
cudaError_t go_bulk_shape(const KArgs& a, cudaStream_t st) {
    const bool two = FSDP_BULK_GROUPS == 2 || (FSDP_BULK_GROUPS == 0 && bulk_stages<S, 2>(a.W) >= 4 && a.D <= 2);
    return two && bulk_stages<S, 2>(a.W) >= 2 ? go_bulk<S, NS, SIN, ND, AP, 2>(a, st)
                                               : go_bulk<S, NS, SIN, ND, AP, 1>(a, st);
}

}  // namespace

bool bulk_reduce_fits(int sdt, int W, int D) {
    if (W > kBulkMaxSources || D > kBulkMaxDests) return false;
    if (sdt == FSDP_F32) return bulk_stages<float, 1>(W) >= 2;
    if (sdt == FSDP_BF16) return bulk_stages<uint16_t, 1>(W) >= 2;
    return false;
}

cudaError_t launch_bulk_reduce(int sdt, const KArgs& a, cudaStream_t st, bool* used) {
    *used = false;
    const bool sf = sdt == FSDP_F32;
    if (!a.status || a.max_grid <= 0 || a.reps != 1 || !bulk_reduce_fits(sdt, a.W, a.D)) return cudaSuccess;
    *used = true;
    const bool ap = a.sg_tab != nullptr;
    if (sf) return ap ? go_bulk_shape<float, 0, 0, 0, true>(a, st) : go_bulk_shape<float, 0, 0, 0, false>(a, st);
#define FSDP_BULK(W_, S_)                                                                    \
    if (a.W == W_ && a.S == S_)                                                              \
        return ap ? go_bulk_shape<uint16_t, W_, S_, W_ / S_, true>(a, st)                     \
                  : go_bulk_shape<uint16_t, W_, S_, W_ / S_, false>(a, st);
    FSDP_BULK(16, 8) FSDP_BULK(8, 4) FSDP_BULK(8, 8) FSDP_BULK(8, 1)
#undef FSDP_BULK
    return ap ? go_bulk_shape<uint16_t, 0, 0, 0, true>(a, st) : go_bulk_shape<uint16_t, 0, 0, 0, false>(a, st);
}

}  // namespace fsdp
