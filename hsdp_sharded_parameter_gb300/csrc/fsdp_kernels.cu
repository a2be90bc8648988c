// Kernels of the GB300 HSDP data path (sm_103a). Every kernel is HBM-bound
// data movement plus, for the gradient sync, an fp32 sum over ranks: no
// tensor cores. All of them share one work model:
//
//   * A plan-time table lists runs ("segments") of contiguous elements; a
//     prefix array gives each run's first warp tile (2048 elements: 8 steps
//     of 32 lanes x 8 elements).
//   * A grid of warps strides over (tile, repetition) pairs, repetition
//     fastest (the ranks or replicas the table is repeated for); each kernel
//     family has its own measured grid size (see FSDP_GRID_*). A warp finds
//     its run with a cooperative search over the prefix array (a ballot over
//     32 probes narrows the range 32-fold per round), moving only forward;
//     the next tile's run is looked up while the current tile's loads are in
//     flight.
//   * Granules are anchored at 16-byte boundaries of the destination, so
//     every full granule is written with aligned 16-byte stores. A tile whose
//     granules are all full (a whole tile, or the whole steps left of a short
//     run) loads every step before storing; partial granules (run heads and
//     tails) and destinations that are not 16-byte aligned go element by
//     element.
//   * Copy kernels read with aligned 16-byte loads into registers; a source
//     run shifted against its destination (ragged offsets) is realigned with
//     funnel shifts, each lane taking its neighbour block from the next lane
//     by a warp shuffle. Kernels that write one tile to several destinations
//     (fused copy-in, gather, direct unshard) stage it in shared memory once
//     and fan it out with TMA bulk stores.
//   * The apply kernel reads the fp32 fused region; a shifted source is off
//     by whole elements, so it switches to a strided lane mapping (lane l
//     takes elements l, l+32, ...) whose loads need no realignment.
//   * Reduce kernels (W sources per output) stage each warp step's source
//     windows in shared memory with cp.async (16-byte copies, one aligned
//     window per source, one block wider when shifted) two steps deep, so
//     the bytes in flight do not depend on registers, then fold from shared
//     memory in the fixed order. With several replicas to write, a step's
//     result goes to shared memory once and out to every replica by TMA bulk
//     stores (see fan_out).
//   * Every staged or loaded 16-byte block holds at least one byte of its
//     source run, so no access leaves the source allocation's pages.
//   * On a capped grid (fsdp_plan_set_grid_limit) the fused sync takes the
//     TMA-bulk-fed kernel of fsdp_bulk.cu instead, where its ring fits.
//
// Sources, by page title + section:
//   [OVERLAP] "Hyper通信掩盖方案" (hyper-parallel issue 184), PR #758 write-up
//   [RAGGED]  FSDP dim-0 uneven-sharding RFC (hyper-parallel issue 319)
//   [FS-RFC]  "【RFC】FullyShard 多维并行适配设计方案" (hyper-parallel issue 1)
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <unordered_map>

#include "fsdp_device.cuh"

namespace fsdp {
namespace {

constexpr int kMaxStagedSources = 32;
// The fused reduce fans a step's result out with TMA bulk stores (one
// shared-memory image, one bulk store per destination) instead of having
// each lane store its granule to every replica: with 4 or more replicas
// (pure-TP layer, 8: 0.855 -> 0.903 of the measured copy peak), and with 2
// when there are at most 8 sources (HSDP (2,4): 0.948 -> 0.961); the (2,8)
// mesh's 16 sources measured slower with it (0.939 -> 0.924).
// One reduce step of RG granules per lane (RG * 256 elements) of fp32.
template <int RG>
__host__ __device__ constexpr size_t fan_img_bytes() { return (size_t)RG * kStepElems * sizeof(float); }
// The unfused AllReduce fans out from 4 replicas on (pure-TP, 8: 0.84 ->
// 0.90; with 2 it measured slower, 0.878 -> 0.841).
template <int KIND, int NS, int ND>
__host__ __device__ constexpr bool fan_out() {
    return (KIND == K_RSAR && NS > 0 && (ND >= 4 || (ND >= 2 && NS <= 8))) ||
           (KIND == K_AR && NS > 0 && ND >= 4);
}
// Resident blocks of the staged reduce its shared memory allows for 16 bf16
// sources (69 KB each); telling the compiler so lets it keep the unrolled
// fold in registers (up to 170 each) instead of spilling.
constexpr int kStagedBlocksPerSm = 3;


// ------------------------------------------------------------ copy kernels

// K_AGIN  : shards[(d,s),p] -> ag[(d,s)] row s (+ every shard-group member
//           with fuse); zero runs pad the rows. rep = d.
// K_GATHER: ag[(d,s)] slice s -> ag[(d,s')] slice s, s' != s. rep = d.
// K_AGOUT : ag[w] at s*slice + o_p -> full[w,p] rows [off, off+len). rep = w.
// K_RSIN  : grads[w,p] rows [off, off+len) -> rs_in[w] row s. rep = w.
// K_RS    : (shard groups of one rank only) rs_in[(d,0)] row 0 -> fused[(d,0)],
//           widened to fp32: the ReduceScatter of one term. rep = d.
template <int KIND, typename S>
__device__ __forceinline__ const S* copy_src(const KArgs& a, const Tile& ti) {
    if (KIND == K_AGIN)
        return ti.p >= 0 ? static_cast<const S*>(a.src_tab[(int64_t)(ti.rep * a.S + ti.row) * a.P + ti.p])
                         : nullptr;
    if (KIND == K_GATHER) return static_cast<const S*>(a.src_tab[ti.rep * a.S + ti.row]);
    if (KIND == K_AGOUT) return static_cast<const S*>(a.src_tab[ti.rep]);
    if (KIND == K_UNSHARD)
        return static_cast<const S*>(a.src_tab[(int64_t)(ti.rep * a.S + ti.row) * a.P + ti.p]);
    if (KIND == K_RS) return static_cast<const S*>(a.src_tab[ti.rep * a.S + ti.row]);
    return ti.p >= 0 ? static_cast<const S*>(a.src_tab[(int64_t)ti.rep * a.P + ti.p]) : nullptr;
}

template <int KIND>
__device__ __forceinline__ int copy_ndst(const KArgs& a) {
    if (KIND == K_AGIN) return a.fuse ? a.S : 1;
    if (KIND == K_GATHER) return a.S - 1;
    if (KIND == K_UNSHARD) return a.S;
    return 1;
}

template <int KIND, typename D>
__device__ __forceinline__ D* copy_dst(const KArgs& a, const Tile& ti, int j) {
    D* d;
    if (KIND == K_AGIN)
        d = static_cast<D*>(a.dst_tab[ti.rep * a.S + (a.fuse ? j : ti.row)]);
    else if (KIND == K_GATHER)
        d = static_cast<D*>(a.dst_tab[ti.rep * a.S + j + (j >= ti.row ? 1 : 0)]);
    else if (KIND == K_AGOUT)
        d = static_cast<D*>(a.dst_tab[(int64_t)ti.rep * a.P + ti.p]);
    else if (KIND == K_UNSHARD)  // shard-group member j of replica rep
        d = static_cast<D*>(a.dst_tab[(int64_t)(ti.rep * a.S + j) * a.P + ti.p]);
    else if (KIND == K_RS)
        d = static_cast<D*>(a.dst_tab[ti.rep * a.S + ti.row]);
    else
        d = static_cast<D*>(a.dst_tab[ti.rep]);
    return d + ti.dst_off;
}

// TMA bulk copies shared -> global (bulk-group completion; the waits are
// hardware waits, no polling).
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory"); }
// Waits until every bulk store of this thread has read its shared-memory
// source (the wait before a block exits and its shared memory is reused);
// their global writes complete on their own, and the kernel's end orders
// them before later work on the stream. Waiting for the writes too at every
// block's exit measured slower once grids run many short waves (HSDP (2,4)
// fused reduce 0.959 -> 1.032 with this wait and many waves).
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// Orders this thread's shared-memory writes before later async-proxy
// (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// Dynamic shared memory of a multi-destination copy: two tile images per warp.
template <typename D>
constexpr size_t copy_img_bytes() {
    return (size_t)(kThreads / 32) * 2 * kWarpTile * sizeof(D);
}

// MULTI: the kernel writes one source to several destinations (fused
// all-gather copy-in, the gather) and has copy_img_bytes<D>() of dynamic
// shared memory for bulk stores. ALIGNED: the plan's runs and the buffers
// put every source on its destination's 16-byte phase (KArgs::aligned_runs):
// the realigning path of interior tiles is left out (71-75 instead of
// 98-106 registers: three resident blocks per SM instead of two), and a
// shifted tile, should one come, takes the per-granule path, which
// realigns too.
template <int KIND, typename S, typename D, bool MULTI, bool ALIGNED = false>
__device__ __forceinline__ void copy_body(const KArgs& a) {
    extern __shared__ __align__(128) uint4 copy_smem[];
    const int lane = threadIdx.x & 31;
    const int64_t stride = warp_count(), total = a.ntiles * a.reps;
    uint4* tile_img = MULTI ? copy_smem + (size_t)(threadIdx.x >> 5) * 2 * (kWarpTile * sizeof(D) / 16) : nullptr;
    int parity = 0;
    int64_t t = warp_id();
    int k = 0;
    Tile cur;
    if (t < total) lookup(a, t, k, (int)sizeof(D), cur);
    const int nd = copy_ndst<KIND>(a);
    while (t < total) {
        const int64_t tn = t + stride;
        const S* src = copy_src<KIND, S>(a, cur);
        Tile nxt;
        // whole steps of the run from lane 0's first granule on (a short
        // run, or a run's last tile, whose length is a multiple of a step
        // also takes the interior path with fewer steps)
        const int64_t ext = cur.n - cur.rel0;
        const int nsteps = ext >= kWarpTile ? kSteps : (int)(ext / kStepElems);
        bool interior = a.vec && cur.rel0 >= 0 && (ext >= kWarpTile || ext % kStepElems == 0);
        if constexpr (ALIGNED) {
            if (interior && src != nullptr)
                interior = (reinterpret_cast<uintptr_t>(src + cur.src_off + cur.rel0) & 15u) == 0;
        }
        if (interior) {
            // interior tile: nsteps steps, every granule full, destination aligned
            Raw<D> val[kSteps];
            if (src == nullptr) {
#pragma unroll
                for (int u = 0; u < kSteps; ++u) zero_raw(val[u]);
            } else {
                const uintptr_t t0 = reinterpret_cast<uintptr_t>(src + cur.src_off + cur.rel0);
                const unsigned sh = (unsigned)(t0 & 15u);
                if (ALIGNED || sh == 0) {
                    const uintptr_t b = t0 + (uintptr_t)(lane * kGran * (int)sizeof(S));
#pragma unroll
                    for (int u = 0; u < kSteps; ++u) {
                        Raw<S> r;
                        if (u < nsteps)
                            load_raw_at(r, b + (uintptr_t)(u * kStepElems * (int)sizeof(S)));
                        else
                            zero_raw(r);
                        convert(r, val[u]);
                    }
                } else if constexpr (!ALIGNED) {
                    Raw<S> r[kSteps];
                    load_tile_shifted(r, t0 - sh, (uintptr_t)(kStepElems * (int)sizeof(S)), sh, lane, nsteps);
#pragma unroll
                    for (int u = 0; u < kSteps; ++u) convert(r[u], val[u]);
                }
            }
            if (tn < total) lookup(a, tn, k, (int)sizeof(D), nxt);
            if (MULTI && nd > 1) {
                // one tile image in shared memory, written to every
                // destination by TMA bulk stores issued from lane 0; the
                // warp's two images alternate, and an image is rewritten
                // only after the bulk stores of two tiles ago have read it
                uint4* img = tile_img + (size_t)parity * (kWarpTile * sizeof(D) / 16);
                if (lane == 0) bulk_wait_read_1();
                __syncwarp();
#pragma unroll
                for (int u = 0; u < kSteps; ++u)
#pragma unroll
                    for (int v = 0; v < Raw<D>::kVec; ++v)
                        if (u < nsteps)
                            img[(u * 32 + lane) * Raw<D>::kVec + v] = make_uint4(
                                val[u].w[4 * v], val[u].w[4 * v + 1], val[u].w[4 * v + 2], val[u].w[4 * v + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(img));
                    for (int j = 0; j < nd; ++j)
                        bulk_store(copy_dst<KIND, D>(a, cur, j) + cur.rel0, s,
                                   (uint32_t)(nsteps * kStepElems) * (uint32_t)sizeof(D));
                    bulk_commit();
                }
                parity ^= 1;
            } else {
                for (int j = 0; j < nd; ++j) {
                    D* d = copy_dst<KIND, D>(a, cur, j) + cur.rel0 + lane * kGran;
#pragma unroll
                    for (int u = 0; u < kSteps; ++u)
                        if (u < nsteps) store_raw(d + u * kStepElems, val[u]);
                }
            }
        } else {
            // edge tile: per-granule checks, element-wise where partial
            for (int j = 0; j < nd; ++j) {
                D* d = copy_dst<KIND, D>(a, cur, j);
#pragma unroll 1
                for (int u = 0; u < kSteps; ++u) {
                    const int64_t rel = cur.rel0 + (int64_t)(u * kStepElems + lane * kGran);
                    if (rel >= cur.n || rel + kGran <= 0) continue;
                    if (a.vec && rel >= 0 && rel + kGran <= cur.n) {
                        Raw<D> v;
                        if (src) {
                            Raw<S> r;
                            load_raw_at(r, reinterpret_cast<uintptr_t>(src + cur.src_off + rel));
                            convert(r, v);
                        } else {
                            zero_raw(v);
                        }
                        store_raw(d + rel, v);
                    } else {
                        const int64_t lo = rel < 0 ? 0 : rel;
                        const int64_t hi = rel + kGran < cur.n ? rel + kGran : cur.n;
                        for (int64_t e = lo; e < hi; ++e) {
                            if (src)
                                copy_elem<S, D>(d, e, src, cur.src_off + e);
                            else
                                d[e] = D(0);
                        }
                    }
                }
            }
            if (tn < total) lookup(a, tn, k, (int)sizeof(D), nxt);
        }
        cur = nxt;
        t = tn;
    }
    // bulk stores must have read the tile images before the block exits
    if (MULTI && lane == 0) bulk_wait_read_all();
}

// ------------------------------------------------------------ apply kernel

// fused[(d,s)] at o_p -> shard_grads[(d,s),p] (actual rows only), divided
// by a.div (W for AVG), optionally added to the gradient already there,
// rounded once to the gradient dtype. rep = d.
template <typename D>
__device__ __forceinline__ void apply_granule(const KArgs& a, const Raw<float>& r, D* dst, bool scale) {
    float x[8];
    widen(r, x);
    if (scale) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = scaled(x[e], a);
    }
    if (a.accumulate) {
        Raw<D> old;
        load_aligned(old, dst);
        float y[8];
        widen(old, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fadd_rn(y[e], x[e]);
    }
    Raw<D> o;
    narrow(x, o);
    store_raw(dst, o);
}

template <typename D>
__device__ __forceinline__ void apply_body(const KArgs& a) {
    const int lane = threadIdx.x & 31;
    const int64_t stride = warp_count(), total = a.ntiles * a.reps;
    const bool scale = a.div != 1.0f;
    int64_t t = warp_id();
    int k = 0;
    Tile cur;
    if (t < total) lookup(a, t, k, (int)sizeof(D), cur);
    while (t < total) {
        const int64_t tn = t + stride;
        const int w = cur.rep * a.S + cur.row;
        const float* src = static_cast<const float*>(a.src_tab[w]) + cur.src_off;
        D* dst = static_cast<D*>(a.dst_tab[(int64_t)w * a.P + cur.p]) + cur.dst_off;
        Tile nxt;
        if (a.vec && cur.rel0 >= 0 && cur.rel0 + kWarpTile <= cur.n) {
            // interior tile: all loads first, then the next lookup, then stores
            Raw<float> r[kSteps];
            const uintptr_t t0 = reinterpret_cast<uintptr_t>(src + cur.rel0);
            const unsigned sh = (unsigned)(t0 & 15u);
            if (sh == 0) {
                const uintptr_t b = t0 + (uintptr_t)(lane * kGran * 4);
#pragma unroll
                for (int u = 0; u < kSteps; ++u) load_raw_at(r[u], b + (uintptr_t)(u * kStepElems * 4));
            } else {
                // fp32 source off the 16-byte grid by k = 1..3 whole
                // elements: lane l loads its two aligned blocks of each step
                // (bytes 32l .. 32l+31 past the step's aligned start), takes
                // the third from lane l+1 by a warp shuffle (lane 31 takes
                // lane 0's first block of the next step, or loads it on the
                // last step: it holds the step's last elements, so it lies in
                // the run), and keeps words k..k+7: 16-byte loads and one
                // 16-byte store per granule instead of element-wise accesses
                const int kw = (int)(sh >> 2);
                const uint4* q = reinterpret_cast<const uint4*>(t0 - sh) + lane * 2;
                uint4 b[kSteps][2];
#pragma unroll
                for (int u = 0; u < kSteps; ++u) {
                    b[u][0] = ld_stream(q + u * 64);
                    b[u][1] = ld_stream(q + u * 64 + 1);
                }
                const uint4 tail = lane == 31 ? ld_stream(q + (kSteps - 1) * 64 + 2) : make_uint4(0, 0, 0, 0);
                if (tn < total) lookup(a, tn, k, (int)sizeof(D), nxt);
#pragma unroll
                for (int u = 0; u < kSteps; ++u) {
                    // lanes 1..31 hand their first block down one lane; lane 0
                    // hands lane 31 its first block of the next step
                    const uint4 give = (lane == 0 && u + 1 < kSteps) ? b[u + 1 < kSteps ? u + 1 : u][0] : b[u][0];
                    uint4 nx;
                    nx.x = __shfl_sync(kFull, give.x, (lane + 1) & 31);
                    nx.y = __shfl_sync(kFull, give.y, (lane + 1) & 31);
                    nx.z = __shfl_sync(kFull, give.z, (lane + 1) & 31);
                    nx.w = __shfl_sync(kFull, give.w, (lane + 1) & 31);
                    if (lane == 31 && u + 1 == kSteps) nx = tail;
                    const uint32_t wd[12] = {b[u][0].x, b[u][0].y, b[u][0].z, b[u][0].w, b[u][1].x, b[u][1].y,
                                             b[u][1].z, b[u][1].w, nx.x,      nx.y,      nx.z,      nx.w};
                    Raw<float> rr;
                    if (kw == 1) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) rr.w[i] = wd[i + 1];
                    } else if (kw == 2) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) rr.w[i] = wd[i + 2];
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) rr.w[i] = wd[i + 3];
                    }
                    apply_granule<D>(a, rr, dst + cur.rel0 + u * kStepElems + lane * kGran, scale);
                }
                cur = nxt;
                t = tn;
                continue;
            }
            if (tn < total) lookup(a, tn, k, (int)sizeof(D), nxt);
#pragma unroll
            for (int u = 0; u < kSteps; ++u)
                apply_granule<D>(a, r[u], dst + cur.rel0 + u * kStepElems + lane * kGran, scale);
            cur = nxt;
            t = tn;
            continue;
        }
        if (tn < total) lookup(a, tn, k, (int)sizeof(D), nxt);
#pragma unroll 2
        for (int u = 0; u < kSteps; ++u) {
            const int64_t rel = cur.rel0 + (int64_t)(u * kStepElems + lane * kGran);
            if (rel >= cur.n || rel + kGran <= 0) continue;
            if (a.vec && rel >= 0 && rel + kGran <= cur.n) {
                Raw<float> r;
                load_raw_at(r, reinterpret_cast<uintptr_t>(src + rel));
                apply_granule<D>(a, r, dst + rel, scale);
            } else {
                const int64_t lo = rel < 0 ? 0 : rel;
                const int64_t hi = rel + kGran < cur.n ? rel + kGran : cur.n;
                for (int64_t e = lo; e < hi; ++e) {
                    float q = src[e];
                    if (scale) q = scaled(q, a);
                    if (a.accumulate) q = __fadd_rn(load_f32(dst, e), q);
                    store_f32(dst, e, q);
                }
            }
        }
        cur = nxt;
        t = tn;
    }
}

// ---------------------------------------------------------- reduce kernels

// K_RSAR: sources grads[w',p] (w' = 0..W-1, grouped S per replica);
//         D destinations fused[(d,s)] at o_p; zero runs write +0. reps = 1.
// K_RS  : sources rs_in[(d,s'')] row s (s'' = 0..S-1); destination
//         fused[(d,s)]; AVG divides by S. rep = d.
// K_AR  : sources fused[(d',s)] (d' = 0..D-1); destinations all fused[(d,s)]
//         in place; AVG divides by D. reps = 1.
//
// The fold ([FS-RFC §2.1.3 item 3, §3.3]: ReduceScatter over the shard
// group, then AllReduce over the replicate group): sources come in groups
// of s_in (a shard group); each group is summed from its first term in
// ascending order (part), then the groups are summed from the first group
// in ascending order (total). Every '+' is one IEEE binary32 RN addition.
template <int KIND>
struct ReduceShape {
    __device__ static int ns(const KArgs& a) { return KIND == K_RSAR ? a.W : (KIND == K_RS ? a.S : a.D); }
    __device__ static int s_in(const KArgs& a) { return KIND == K_AR ? 1 : a.S; }
    __device__ static int nd(const KArgs& a) { return KIND == K_RS ? 1 : a.D; }
    template <typename S>
    __device__ static const S* src(const KArgs& a, int p, int row, int rep, int i) {
        if (KIND == K_RSAR) return static_cast<const S*>(a.src_tab[(int64_t)i * a.P + p]);
        if (KIND == K_RS) return static_cast<const S*>(a.src_tab[rep * a.S + i]);
        return static_cast<const S*>(a.src_tab[i * a.S + row]);
    }
    __device__ static float* dst(const KArgs& a, int row, int rep, int j) {
        if (KIND == K_RS) return static_cast<float*>(a.dst_tab[rep * a.S + row]);
        return static_cast<float*>(a.dst_tab[j * a.S + row]);
    }
};

// Element-wise fold of one element (partial granules).
template <int KIND, typename S>
__device__ __forceinline__ float fold_elem(const KArgs& a, const S* const* sp, int64_t e) {
    const int s_in = ReduceShape<KIND>::s_in(a), d_out = ReduceShape<KIND>::ns(a) / s_in;
    float total = 0.0f;
    for (int d = 0; d < d_out; ++d) {
        float part = load_f32(sp[d * s_in], e);
        for (int s = 1; s < s_in; ++s) part = __fadd_rn(part, load_f32(sp[d * s_in + s], e));
        total = d == 0 ? part : __fadd_rn(total, part);
    }
    return total;
}

// The staged reduce works in steps of RG * 256 elements: each lane folds
// RG granules of 8 elements per step (granule g of lane l starts at element
// g*256 + l*8 of the step). RG = 1 on the full grid; RG = 2 on a capped
// grid (one block per SM), where the reduce is issue-bound and the
// per-step work (staging the pointers, checking the sources' alignment,
// issuing the copies, stepping through the table) is then paid once per
// 512 elements. A step that repeats the run of the step staged last in the
// same stage slot reuses the pointers and the alignment found then (they
// are per-run constants).
// Per-warp shared-memory layout of the staged reduce: per stage, one window
// of kWin 16-byte blocks per source (a step of RG * 256 elements spans RG *
// 32 blocks of bf16 or RG * 64 of fp32, plus one when the source is
// shifted), then the step's source and destination pointers.
template <typename S, int RG = 1>
struct Staging {
    static constexpr int kWin = RG * kStepElems * (int)sizeof(S) / 16 + 1;
    __host__ __device__ static constexpr size_t window_bytes(int ns) { return (size_t)ns * kWin * 16; }
    __host__ __device__ static constexpr size_t stage_bytes(int ns, int nd) {
        return window_bytes(ns) + (size_t)(ns + nd) * sizeof(void*) + 15 & ~(size_t)15;
    }
    __host__ __device__ static constexpr size_t warp_bytes(int ns, int nd) { return 2 * stage_bytes(ns, nd); }
};

struct Step {
    int64_t n, dst_off, src_off, rel;  // rel: run-relative element of lane 0's first granule
    int p, row, rep;
    bool valid;
    bool fast;       // interior data step whose sources all share one 16-byte shift
    unsigned shift;  // that shift in bytes (0 = aligned)
};

// What a stage slot last staged: the run's key (p, row, rep), whether its
// sources share one 16-byte shift, and that shift. Warp-uniform.
// Which reduces use the slot cache and the packed (f32x2) adds: both cut
// instructions, which pays on a capped grid, where the reduce is
// issue-bound; on the full grid (HBM-bound) they measured slower (ragged
// layer 0.999 -> 0.912 of the copy peak with both).
#ifndef FSDP_SLOT_CACHE_FULL
#define FSDP_SLOT_CACHE_FULL 0
#endif
#ifndef FSDP_PACKED_ADDS_FULL
#define FSDP_PACKED_ADDS_FULL 0
#endif
#ifndef FSDP_SLOT_CACHE_SM
#define FSDP_SLOT_CACHE_SM 1
#endif
#ifndef FSDP_PACKED_ADDS_SM
#define FSDP_PACKED_ADDS_SM 1
#endif
template <int RG>
__host__ __device__ constexpr bool slot_cache() { return RG == 1 ? FSDP_SLOT_CACHE_FULL != 0 : FSDP_SLOT_CACHE_SM != 0; }
template <int RG>
__host__ __device__ constexpr bool packed_adds() { return RG == 1 ? FSDP_PACKED_ADDS_FULL != 0 : FSDP_PACKED_ADDS_SM != 0; }

struct SlotCache {
    int64_t dst_off = -1;
    int p = -2, row = -1, rep = -1;
    bool uniform = false;
    unsigned shift = 0;
};

// Yields a warp's steps in order: its tiles (grid stride), kWarpTile /
// (RG * 256) steps each, skipping steps past the end of their run.
// Warp-uniform.
template <int RG>
struct StepGen {
    static constexpr int kStep = RG * kStepElems, kPerTile = kWarpTile / kStep;
    static_assert(kWarpTile % kStep == 0, "a warp tile is a whole number of reduce steps");
    int64_t t, stride, total;
    int u, k;
    Tile tile;
    __device__ void init(const KArgs& a) {
        stride = warp_count();
        total = a.ntiles * a.reps;
        t = warp_id();
        u = -1;
        k = 0;
        if (t < total) lookup(a, t, k, 4, tile);
    }
    __device__ Step next(const KArgs& a) {
        Step s;
        s.valid = false;
        s.fast = false;
        s.shift = 0;
        for (;;) {
            if (t >= total) return s;
            if (++u == kPerTile) {
                t += stride;
                u = 0;
                if (t >= total) return s;
                lookup(a, t, k, 4, tile);
            }
            const int64_t rel = tile.rel0 + (int64_t)u * kStep;
            if (rel < tile.n) {
                s.n = tile.n;
                s.dst_off = tile.dst_off;
                s.src_off = tile.src_off;
                s.rel = rel;
                s.p = tile.p;
                s.row = tile.row;
                s.rep = tile.rep;
                s.valid = true;
                return s;
            }
        }
    }
};

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

// The reduce's shape: sources, their grouping and destinations. Template
// values > 0 fix them at compile time (common meshes, fully unrolled);
// 0 reads them from the arguments.
template <int KIND, int NS, int SIN, int ND>
struct Shape {
    int ns, s_in, d_out, nd;
    __device__ explicit Shape(const KArgs& a) {
        ns = NS > 0 ? NS : ReduceShape<KIND>::ns(a);
        s_in = SIN > 0 ? SIN : ReduceShape<KIND>::s_in(a);
        nd = ND > 0 ? ND : ReduceShape<KIND>::nd(a);
        d_out = (NS > 0 && SIN > 0) ? NS / SIN : ns / s_in;
    }
};

// Stage one step: pointers into the stage's pointer area (unless the slot
// holds this run's already), and for a data run with aligned destinations,
// each source's window via cp.async (only blocks that hold bytes of the
// step's valid range). An interior step whose sources are all 16-byte
// aligned copies exactly the RG * 256 elements of each source, RG blocks per
// lane per 16-byte vector. Always commits one group (possibly empty) so the
// group count stays in step with the ring.
template <int KIND, typename S, int NS, int SIN, int ND, int RG, bool AP = false>
__device__ __forceinline__ void stage_step(const KArgs& a, Step& st, char* stage, SlotCache& c,
                                           const Shape<KIND, NS, SIN, ND>& sh) {
    const int lane = threadIdx.x & 31;
    constexpr int kWin = Staging<S, RG>::kWin;
    constexpr int kStep = RG * kStepElems;
    uint4* win = reinterpret_cast<uint4*>(stage);
    const S** sp = reinterpret_cast<const S**>(stage + Staging<S, RG>::window_bytes(sh.ns));
    float** dp = reinterpret_cast<float**>(stage + Staging<S, RG>::window_bytes(sh.ns) + sh.ns * sizeof(void*));
    const bool same = slot_cache<RG>() && st.valid && st.p == c.p && st.row == c.row && st.rep == c.rep &&
                      st.dst_off == c.dst_off;
    if (st.valid && !same) {
        if (st.p >= 0)
            for (int i = lane; i < sh.ns; i += 32) sp[i] = ReduceShape<KIND>::template src<S>(a, st.p, st.row, st.rep, i);
        for (int j = lane; j < sh.nd; j += 32) dp[j] = ReduceShape<KIND>::dst(a, st.row, st.rep, j) + st.dst_off;
        if constexpr (AP) {
            // replica j's actual-shard gradient of this run's parameter
            S** gp = reinterpret_cast<S**>(stage + Staging<S, RG>::window_bytes(sh.ns) + (sh.ns + sh.nd) * sizeof(void*));
            if (st.p >= 0)
                for (int j = lane; j < sh.nd; j += 32)
                    gp[j] = static_cast<S*>(a.sg_tab[(int64_t)(j * a.S + st.row) * a.P + st.p]);
        }
    }
    __syncwarp();
    if (st.valid && st.p >= 0 && a.vec) {
        const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(win));
        const int64_t byte0 = (st.src_off + st.rel) * (int64_t)sizeof(S);  // may precede the run: address only
        bool uniform;
        unsigned shift;
        if (!same) {
            // one shift for every source? (a per-run constant: steps of a run
            // are whole multiples of 256 elements apart)
            const unsigned sh0 = (unsigned)((reinterpret_cast<uintptr_t>(sp[0]) + (uintptr_t)byte0) & 15u);
            bool ok = true;
            for (int i = lane; i < sh.ns; i += 32)
                ok = ok && ((reinterpret_cast<uintptr_t>(sp[i]) + (uintptr_t)byte0) & 15u) == sh0;
            uniform = __all_sync(kFull, ok);
            shift = sh0;
            if constexpr (slot_cache<RG>()) {
                c.uniform = uniform;
                c.shift = sh0;
                c.p = st.p;
                c.row = st.row;
                c.rep = st.rep;
                c.dst_off = st.dst_off;
            }
        } else {
            uniform = c.uniform;
            shift = c.shift;
        }
        if (uniform && st.rel >= 0 && st.rel + kStep <= st.n) {
            // every source window starts `shift` bytes before its first
            // element; a shifted window needs one block more, copied by lane 0
            st.fast = true;
            st.shift = shift;
#pragma unroll
            for (int i = 0; i < sh.ns; ++i) {
                const char* g = reinterpret_cast<const char*>(sp[i]) + byte0 - shift;
#pragma unroll
                for (int v = 0; v < RG * Raw<S>::kVec; ++v)
                    cp_async16(sbase + (uint32_t)((i * kWin + lane + 32 * v) * 16), g + (lane + 32 * v) * 16);
                if (shift != 0 && lane == 0)
                    cp_async16(sbase + (uint32_t)((i * kWin + kWin - 1) * 16), g + (kWin - 1) * 16);
            }
        } else {
            const int64_t e_lo = st.rel < 0 ? 0 : st.rel;
            const int64_t e_hi = st.rel + kStep < st.n ? st.rel + kStep : st.n;
            for (int i = 0; i < sh.ns; ++i) {
                const uintptr_t base = reinterpret_cast<uintptr_t>(sp[i]) + (uintptr_t)(st.src_off * (int64_t)sizeof(S));
                const uintptr_t wst = (base + (uintptr_t)(st.rel * (int64_t)sizeof(S))) & ~(uintptr_t)15;
                const uintptr_t vlo = base + (uintptr_t)(e_lo * (int64_t)sizeof(S));
                const uintptr_t vhi = base + (uintptr_t)(e_hi * (int64_t)sizeof(S));
                for (int blk = lane; blk < kWin; blk += 32) {
                    const uintptr_t g = wst + 16 * (uintptr_t)blk;
                    if (g < vhi && g + 16 > vlo)
                        cp_async16(sbase + (uint32_t)((i * kWin + blk) * 16), reinterpret_cast<const void*>(g));
                }
            }
        }
    } else if (slot_cache<RG>() && st.valid && !same) {
        // zero runs and unaligned destinations stage no windows; the slot
        // now holds this run's pointers
        c.p = st.p;
        c.row = st.row;
        c.rep = st.rep;
        c.dst_off = st.dst_off;
        c.uniform = false;
    }
    cp_async_commit();
}

// Reads granule g of a lane's 8 elements of source i from its staged window.
template <typename S, int RG>
__device__ __forceinline__ void read_window(const uint4* win, int i, int lane, int g, unsigned sh, Raw<S>& r) {
    const uint4* w = win + i * Staging<S, RG>::kWin + (g * 32 + lane) * Raw<S>::kVec;
    if (sh == 0) {
#pragma unroll
        for (int v = 0; v < Raw<S>::kVec; ++v) put(r.w + 4 * v, w[v]);
    } else {
        uint4 blk[Raw<S>::kVec + 1];
#pragma unroll
        for (int v = 0; v <= Raw<S>::kVec; ++v) blk[v] = w[v];
#pragma unroll
        for (int v = 0; v < Raw<S>::kVec; ++v) put(r.w + 4 * v, funnel(blk[v], blk[v + 1], sh));
    }
}

// x[2k..2k+1] += y[2k..2k+1] as packed pairs: each element one IEEE binary32
// round-to-nearest-even addition, as __fadd_rn would do it.
__device__ __forceinline__ void add_pairs(float (&x)[8], const float (&y)[8]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint64_t a = (uint64_t)__float_as_uint(x[2 * k]) | ((uint64_t)__float_as_uint(x[2 * k + 1]) << 32);
        const uint64_t b = (uint64_t)__float_as_uint(y[2 * k]) | ((uint64_t)__float_as_uint(y[2 * k + 1]) << 32);
        asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
        x[2 * k] = __uint_as_float((uint32_t)a);
        x[2 * k + 1] = __uint_as_float((uint32_t)(a >> 32));
    }
}

// Interior step whose sources share one shift: granule g of the lane is
// full; source i of lane l starts `shift` bytes into its window's block
// (g*32 + l)*kVec.
template <bool SHIFTED, typename S, int RG, int NS, int SIN, int ND, int KIND>
__device__ __forceinline__ void fold_fast(const uint4* win, int lane, int g, unsigned shift,
                                          const Shape<KIND, NS, SIN, ND>& sh, float (&total)[8]) {
#pragma unroll
    for (int d = 0; d < sh.d_out; ++d) {
        float part[8];
#pragma unroll
        for (int s = 0; s < sh.s_in; ++s) {
            Raw<S> r;
            read_window<S, RG>(win, d * sh.s_in + s, lane, g, SHIFTED ? shift : 0u, r);
            float x[8];
            widen(r, x);
            if (s == 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) part[e] = x[e];
            } else if constexpr (packed_adds<RG>()) {
                add_pairs(part, x);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) part[e] = __fadd_rn(part[e], x[e]);
            }
        }
        if (d == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) total[e] = part[e];
        } else if constexpr (packed_adds<RG>()) {
            add_pairs(total, part);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) total[e] = __fadd_rn(total[e], part[e]);
        }
    }
}


template <int KIND, typename S, int NS, int SIN, int ND, int RG, bool AP = false>
__device__ __forceinline__ void consume_step(const KArgs& a, const Step& st, const char* stage,
                                             const Shape<KIND, NS, SIN, ND>& sh, uint4* img, int& parity) {
    if (!st.valid) return;
    const int lane = threadIdx.x & 31;
    const uint4* win = reinterpret_cast<const uint4*>(stage);
    const S* const* sp = reinterpret_cast<const S* const*>(stage + Staging<S, RG>::window_bytes(sh.ns));
    float* const* dp =
        reinterpret_cast<float* const*>(stage + Staging<S, RG>::window_bytes(sh.ns) + sh.ns * sizeof(void*));
    // with the apply folded in: the replicas' actual-shard gradients
    S* const* gp = reinterpret_cast<S* const*>(stage + Staging<S, RG>::window_bytes(sh.ns) +
                                               (sh.ns + sh.nd) * sizeof(void*));
    constexpr size_t kImg = fan_img_bytes<RG>();
    // the fused region holds the raw sum; with the apply folded in, a.div
    // is the apply's divisor
    const bool scale = !AP && a.div != 1.0f;
    if (st.fast) {
        Raw<float> o[RG];
#pragma unroll
        for (int g = 0; g < RG; ++g) {
            float total[8];
            if (st.shift == 0)
                fold_fast<false, S, RG>(win, lane, g, 0u, sh, total);
            else
                fold_fast<true, S, RG>(win, lane, g, st.shift, sh, total);
            if (scale) {
#pragma unroll
                for (int e = 0; e < 8; ++e) total[e] = scaled(total[e], a);
            }
            if constexpr (AP) {
#pragma unroll
                for (int j = 0; j < sh.nd; ++j) store_applied(a, total, gp[j] + st.rel + g * kStepElems + lane * kGran);
            }
            narrow(total, o[g]);
        }
        if constexpr (fan_out<KIND, NS, ND>()) {
            // the step's results as one image (two per warp, in turn; an
            // image is rewritten only after the bulk stores of two fast steps
            // ago have read it), written to every replica by lane 0
            uint4* im = img + parity * (int)(kImg / 16);
            if (lane == 0) bulk_wait_read_1();
            __syncwarp();
#pragma unroll
            for (int g = 0; g < RG; ++g) {
                im[2 * (g * 32 + lane)] = make_uint4(o[g].w[0], o[g].w[1], o[g].w[2], o[g].w[3]);
                im[2 * (g * 32 + lane) + 1] = make_uint4(o[g].w[4], o[g].w[5], o[g].w[6], o[g].w[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(im));
#pragma unroll
                for (int j = 0; j < sh.nd; ++j) bulk_store(dp[j] + st.rel, s, (uint32_t)kImg);
                bulk_commit();
            }
            parity ^= 1;
        } else {
#pragma unroll
            for (int j = 0; j < sh.nd; ++j)
#pragma unroll
                for (int g = 0; g < RG; ++g) store_raw(dp[j] + st.rel + g * kStepElems + lane * kGran, o[g]);
        }
        return;
    }
#pragma unroll 1
    for (int g = 0; g < RG; ++g) {
        const int64_t rel = st.rel + g * kStepElems + lane * kGran;
        if (rel >= st.n || rel + kGran <= 0) continue;
        if (a.vec && rel >= 0 && rel + kGran <= st.n) {
            float total[8];
            if (st.p < 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) total[e] = 0.0f;
            } else {
                for (int d = 0; d < sh.d_out; ++d) {
                    float part[8];
                    for (int s = 0; s < sh.s_in; ++s) {
                        const int i = d * sh.s_in + s;
                        const unsigned shift = (unsigned)((reinterpret_cast<uintptr_t>(sp[i]) +
                                                           (uintptr_t)((st.src_off + st.rel) * (int64_t)sizeof(S))) & 15u);
                        Raw<S> r;
                        read_window<S, RG>(win, i, lane, g, shift, r);
                        float x[8];
                        widen(r, x);
                        if (s == 0) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) part[e] = x[e];
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) part[e] = __fadd_rn(part[e], x[e]);
                        }
                    }
                    if (d == 0) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) total[e] = part[e];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) total[e] = __fadd_rn(total[e], part[e]);
                    }
                }
                if (scale) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) total[e] = scaled(total[e], a);
                }
                if constexpr (AP) {
                    for (int j = 0; j < sh.nd; ++j) store_applied(a, total, gp[j] + rel);
                }
            }
            Raw<float> o;
            narrow(total, o);
            for (int j = 0; j < sh.nd; ++j) store_raw(dp[j] + rel, o);
        } else {
            const int64_t lo = rel < 0 ? 0 : rel;
            const int64_t hi = rel + kGran < st.n ? rel + kGran : st.n;
            for (int64_t e = lo; e < hi; ++e) {
                float v = 0.0f;
                if (st.p >= 0) {
                    v = fold_elem<KIND, S>(a, sp, st.src_off + e);
                    if (scale) v = scaled(v, a);
                    if constexpr (AP) {
                        float q = a.div != 1.0f ? scaled(v, a) : v;
                        for (int j = 0; j < sh.nd; ++j) {
                            float x = q;
                            if (a.accumulate) x = __fadd_rn(load_f32(gp[j], e), x);
                            store_f32(gp[j], e, x);
                        }
                    }
                }
                for (int j = 0; j < sh.nd; ++j) dp[j][e] = v;
            }
        }
    }
}

// Two-stage ring per warp: while step i is folded from shared memory, the
// copies of step i+1 are in flight. Each lane waits for its own copies;
// __syncwarp then makes every lane's copies visible to the whole warp.
template <int KIND, typename S, int NS, int SIN, int ND, int RG = 1, bool AP = false>
__device__ __forceinline__ void staged_reduce_body(const KArgs& a) {
    extern __shared__ __align__(16) char smem_raw[];
    const Shape<KIND, NS, SIN, ND> sh(a);
    // with the apply folded in, each stage also holds the replicas'
    // shard-gradient pointers
    const size_t sb = Staging<S, RG>::stage_bytes(sh.ns, AP ? 2 * sh.nd : sh.nd);
    constexpr bool kFan = fan_out<KIND, NS, ND>();
    char* base = smem_raw + (threadIdx.x >> 5) * (2 * sb + (kFan ? 2 * fan_img_bytes<RG>() : 0));
    char* here = base;        // stage of the step being folded
    char* there = base + sb;  // stage of the step in flight
    SlotCache c_here, c_there;
    uint4* img = kFan ? reinterpret_cast<uint4*>(base + 2 * sb) : nullptr;  // fan-out images
    int parity = 0;
    StepGen<RG> gen;
    gen.init(a);
    Step cur = gen.next(a);
    stage_step<KIND, S, NS, SIN, ND, RG, AP>(a, cur, here, c_here, sh);
    while (cur.valid) {
        Step nxt = gen.next(a);
        stage_step<KIND, S, NS, SIN, ND, RG, AP>(a, nxt, there, c_there, sh);
        cp_async_wait1();
        __syncwarp();
        consume_step<KIND, S, NS, SIN, ND, RG, AP>(a, cur, here, sh, img, parity);
        __syncwarp();
        cur = nxt;
        char* t = here;
        here = there;
        there = t;
        const SlotCache tc = c_here;
        c_here = c_there;
        c_there = tc;
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    // bulk stores must have read the images before the block exits
    if (kFan && (threadIdx.x & 31) == 0) bulk_wait_read_all();
}

// Register path for more than kMaxStagedSources sources: each lane loads
// its granule of every source straight into registers, 8 at a time.
template <int KIND, typename S>
__device__ __forceinline__ void direct_reduce_body(const KArgs& a) {
    const int lane = threadIdx.x & 31;
    const int ns = ReduceShape<KIND>::ns(a), nd = ReduceShape<KIND>::nd(a);
    const int s_in = ReduceShape<KIND>::s_in(a);
    const bool scale = a.div != 1.0f;
    const int64_t stride = warp_count(), total_t = a.ntiles * a.reps;
    int k = 0;
    for (int64_t t = warp_id(); t < total_t; t += stride) {
        Tile ti;
        lookup(a, t, k, 4, ti);
#pragma unroll 1
        for (int u = 0; u < kSteps; ++u) {
            const int64_t rel = ti.rel0 + (int64_t)(u * kStepElems + lane * kGran);
            if (rel >= ti.n || rel + kGran <= 0) continue;
            const bool full = a.vec && rel >= 0 && rel + kGran <= ti.n;
            if (full) {
                float total[8], part[8];
                if (ti.p < 0) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) total[e] = 0.0f;
                } else {
                    for (int i = 0; i < ns; ++i) {
                        const S* sp = ReduceShape<KIND>::template src<S>(a, ti.p, ti.row, ti.rep, i);
                        Raw<S> r;
                        load_raw_at(r, reinterpret_cast<uintptr_t>(sp + ti.src_off + rel));
                        float x[8];
                        widen(r, x);
                        const int s = i % s_in;
#pragma unroll
                        for (int e = 0; e < 8; ++e) part[e] = s == 0 ? x[e] : __fadd_rn(part[e], x[e]);
                        if (s == s_in - 1) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) total[e] = i < s_in ? part[e] : __fadd_rn(total[e], part[e]);
                        }
                    }
                    if (scale) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) total[e] = scaled(total[e], a);
                    }
                }
                Raw<float> o;
                narrow(total, o);
                for (int j = 0; j < nd; ++j) store_raw(ReduceShape<KIND>::dst(a, ti.row, ti.rep, j) + ti.dst_off + rel, o);
            } else {
                const int64_t lo = rel < 0 ? 0 : rel;
                const int64_t hi = rel + kGran < ti.n ? rel + kGran : ti.n;
                for (int64_t e = lo; e < hi; ++e) {
                    float v = 0.0f;
                    if (ti.p >= 0) {
                        float tot = 0.0f, part = 0.0f;
                        for (int i = 0; i < ns; ++i) {
                            const S* sp = ReduceShape<KIND>::template src<S>(a, ti.p, ti.row, ti.rep, i);
                            const float x = load_f32(sp, ti.src_off + e);
                            const int s = i % s_in;
                            part = s == 0 ? x : __fadd_rn(part, x);
                            if (s == s_in - 1) tot = i < s_in ? part : __fadd_rn(tot, part);
                        }
                        v = scale ? scaled(tot, a) : tot;
                    }
                    for (int j = 0; j < nd; ++j) ReduceShape<KIND>::dst(a, ti.row, ti.rep, j)[ti.dst_off + e] = v;
                }
            }
        }
    }
}

// ----------------------------------------------------------- entry kernels
// One named kernel per C-ABI call (the names show in profiles).

template <typename S, typename D, bool AL = false>
__global__ void __launch_bounds__(kThreads) ag_copy_in_kernel(const KArgs a) { copy_body<K_AGIN, S, D, true, AL>(a); }
template <typename T>
__global__ void __launch_bounds__(kThreads) ag_gather_kernel(const KArgs a) { copy_body<K_GATHER, T, T, true>(a); }
template <typename T, bool AL = false>
__global__ void __launch_bounds__(kThreads) ag_copy_out_kernel(const KArgs a) { copy_body<K_AGOUT, T, T, false, AL>(a); }
template <typename T>
__global__ void __launch_bounds__(kThreads) rs_copy_in_kernel(const KArgs a) { copy_body<K_RSIN, T, T, false>(a); }
template <typename S, typename D>
__global__ void __launch_bounds__(kThreads) ag_unshard_kernel(const KArgs a) { copy_body<K_UNSHARD, S, D, true>(a); }
// The unfused ReduceScatter over a shard group of one rank: a widening copy
// (the sum of one term, divided by 1).
template <typename S>
__global__ void __launch_bounds__(kThreads) rs_reduce_copy_kernel(const KArgs a) { copy_body<K_RS, S, float, false>(a); }
template <typename S, int NS, int SIN, int ND>
__global__ void __launch_bounds__(kStagedWarps * 32, kStagedBlocksPerSm)rs_ar_reduce_kernel(const KArgs a) {
    staged_reduce_body<K_RSAR, S, NS, SIN, ND>(a);
}
// The fused reduce with the apply folded in (fsdp_rs_ar_reduce_apply).
template <typename S, int NS, int SIN, int ND>
__global__ void __launch_bounds__(kStagedWarps * 32, kStagedBlocksPerSm) rs_ar_reduce_apply_kernel(const KArgs a) {
    staged_reduce_body<K_RSAR, S, NS, SIN, ND, 1, true>(a);
}
template <typename S, int NS>
__global__ void __launch_bounds__(kStagedWarps * 32, kStagedBlocksPerSm)rs_reduce_kernel(const KArgs a) {
    staged_reduce_body<K_RS, S, NS, NS, 1>(a);
}
template <int NS>
__global__ void __launch_bounds__(kStagedWarps * 32, kStagedBlocksPerSm)ar_reduce_kernel(const KArgs a) {
    staged_reduce_body<K_AR, float, NS, 1, NS>(a);
}
// The same reduces on a capped grid (fsdp_plan_set_grid_limit): one block
// per SM, as many warps as the SM's shared memory holds staging rings for
// (11 to 23 on the common meshes), so a few SMs keep as many bytes in
// flight as many SMs do with the 4-warp blocks. On one GB300, cp.async
// reads from one 1024-thread block per SM reach 130-180 GB/s per SM, and 48
// SMs 6.3-6.7 TB/s; a 4-warp block keeps ~34 KB in flight and reached ~30
// GB/s per SM. The block's warp count is fixed at compile time for the
// compiled meshes and is an upper bound for the others (the launch then
// picks it). These run 512-element steps (kSmRG granules per lane).
constexpr size_t kSmBlockSmem = 220 * 1024;
// Steps of 512 elements (two granules per lane) on a capped grid.
constexpr int kSmRG = 2;
template <int KIND, typename S, int NS, int ND>
__host__ __device__ constexpr size_t staged_warp_bytes() {
    return Staging<S, kSmRG>::warp_bytes(NS, ND) + (fan_out<KIND, NS, ND>() ? 2 * fan_img_bytes<kSmRG>() : 0);
}
// Warps of the one-block-per-SM reduce: as many as the shared memory holds,
// at most 16 (the fold keeps up to ~128 registers per thread; more warps
// would force spills).
constexpr int kSmMaxWarps = 16;
template <int KIND, typename S, int NS, int ND>
__host__ __device__ constexpr int sm_warps() {
    return NS == 0 ? 8
                   : (kSmBlockSmem / staged_warp_bytes<KIND, S, NS, ND>() > kSmMaxWarps
                          ? kSmMaxWarps
                          : (int)(kSmBlockSmem / staged_warp_bytes<KIND, S, NS, ND>()));
}
template <typename S, int NS, int SIN, int ND>
__global__ void __launch_bounds__(sm_warps<K_RSAR, S, NS, ND>() * 32, 1) rs_ar_reduce_sm_kernel(const KArgs a) {
    staged_reduce_body<K_RSAR, S, NS, SIN, ND, kSmRG>(a);
}
// Per SM, with the apply folded in: each stage also holds D gradient
// pointers, sized like a reduce with twice the destinations.
template <typename S, int NS, int SIN, int ND>
__global__ void __launch_bounds__(sm_warps<K_RSAR, S, NS, 2 * ND>() * 32, 1)
    rs_ar_reduce_apply_sm_kernel(const KArgs a) {
    staged_reduce_body<K_RSAR, S, NS, SIN, ND, kSmRG, true>(a);
}
template <typename S, int NS>
__global__ void __launch_bounds__(sm_warps<K_RS, S, NS, 1>() * 32, 1) rs_reduce_sm_kernel(const KArgs a) {
    staged_reduce_body<K_RS, S, NS, NS, 1, kSmRG>(a);
}
template <int NS>
__global__ void __launch_bounds__(sm_warps<K_AR, float, NS, NS>() * 32, 1) ar_reduce_sm_kernel(const KArgs a) {
    staged_reduce_body<K_AR, float, NS, 1, NS, kSmRG>(a);
}
template <typename S>
__global__ void __launch_bounds__(kThreads) rs_ar_reduce_wide_kernel(const KArgs a) {
    direct_reduce_body<K_RSAR, S>(a);
}
template <typename S>
__global__ void __launch_bounds__(kThreads) rs_reduce_wide_kernel(const KArgs a) {
    direct_reduce_body<K_RS, S>(a);
}
__global__ void __launch_bounds__(kThreads) ar_reduce_wide_kernel(const KArgs a) {
    direct_reduce_body<K_AR, float>(a);
}
template <typename D>
__global__ void __launch_bounds__(kThreads) apply_grads_kernel(const KArgs a) { apply_body<D>(a); }

// ------------------------------------------------------------------ launch

struct LaunchShape {
    int per_sm;
};

// SM count of the current device, cached per device (a process may launch
// on several GPUs).
int sm_count() {
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

// Resident blocks per SM for (kernel, block size, dynamic shared memory),
// cached. Raises the kernel's dynamic shared memory limit when needed.
// See go(): run count above which a short launch keeps one wave.
constexpr int kWaveMaxRuns = 256;



int blocks_per_sm(const void* fn, int threads, size_t smem) {
    static std::mutex mu;
    // keyed by (device, kernel): function attributes are set per device
    static std::map<std::pair<int, const void*>, std::unordered_map<size_t, int>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    auto fit = cache.find({dev, fn});
    if (fit == cache.end()) {
        // allow the device's whole opt-in shared memory (less the kernel's
        // static shared memory) once per kernel and device, so any later
        // launch of it (any table size) fits
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, fn) == cudaSuccess) {
            const int dyn = optin - (int)fa.sharedSizeBytes;
            if (dyn > 48 * 1024 && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
                (void)cudaGetLastError();  // keep the launch's own status clean
        } else {
            (void)cudaGetLastError();
        }
        fit = cache.emplace(std::make_pair(dev, fn), std::unordered_map<size_t, int>()).first;
    }
    auto& per = fit->second;
    auto it = per.find(smem);
    if (it != per.end()) return it->second;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem) != cudaSuccess || b < 1) b = 1;
    per.emplace(smem, b);
    return b;
}

// Blocks per SM of each kernel family's grid: 0 = as many as fit at once
// (one persistent wave). A value above what fits gives many waves of
// short-lived blocks; each warp still strides over the whole table, but it
// handles few tiles, so the tiles in flight at any time form one
// contiguous window of the table, and that measured faster than a
// persistent grid. Each family has the value its sweep chose (large (2,8)
// layer unless noted; fraction of the measured copy peak):
//   copy-out 128 (one wave 0.955, 16: 1.006, 128: 1.019; 256 was no better
//     there), 16 when most of the plan's copy-out data is shifted
//     (FSDP_GRID_COPY_SHIFTED),
//   fused copy-in 256 (one wave 0.889, 32: 0.981, 256: 0.998),
//   direct unshard 256 (one wave 0.90, 32: 0.983, 256: 0.999),
//   apply 64 (16: 0.998, 64: 1.02; ragged 0.884 -> 0.913),
//   unfused all-gather 256 (one wave 0.89, 32: 0.98, 256: 1.01-1.03).
// The fused reduce's value is in rsar_grid(); the unfused reduces take
// KArgs::staged_blocks, which the plan derives from its layout, or
// rs_grid().
#ifndef FSDP_GRID_COPY
#define FSDP_GRID_COPY 128
#endif
// Copy-out of a plan whose data sits mostly in shifted runs (the ragged
// layer: 0.960 at 128, 0.980 at 16; 32 and 64 in between).
#ifndef FSDP_GRID_COPY_SHIFTED
#define FSDP_GRID_COPY_SHIFTED 16
#endif
// Copy-out over a table with a tile -> run map (thousands of runs), many
// waves: 32 (2000-parameter layer, timed inside the step: one wave 0.94,
// 16: 0.960, 32: 0.965, 128: 0.899).
#ifndef FSDP_GRID_COPY_MAPPED
#define FSDP_GRID_COPY_MAPPED 32
#endif
#ifndef FSDP_GRID_MULTI
#define FSDP_GRID_MULTI 256
#endif
// bf16 copy-in and copy-out launches whose runs and buffers are all on
// their destination's 16-byte phase (KArgs::aligned_runs) take a build of
// the copy without the realigning path: 71-75 registers instead of 98-106,
// three blocks per SM instead of two (2000-parameter pure-TP layer, timed
// inside the step: copy-in 0.931 -> 0.943, copy-out 0.963 -> 0.976 of the
// measured copy peak; the other layers unchanged). The direct unshard keeps
// its one build: without the realigning path it measured slower (HSDP (2,4)
// 1.021 -> 0.991, large 1.012 -> 0.984).
#ifndef FSDP_ALIGNED_COPIES
#define FSDP_ALIGNED_COPIES 1
#endif
#ifndef FSDP_GRID_APPLY
#define FSDP_GRID_APPLY 64
#endif
#ifndef FSDP_GRID_STAGED
#define FSDP_GRID_STAGED 0
#endif
#ifndef FSDP_GRID_UNSHARD
#define FSDP_GRID_UNSHARD 256
#endif
// The direct unshard over a table with a tile -> run map (thousands of
// runs), many waves of 32 blocks per SM like the copy-out (2000-parameter
// layer, timed alone: 256: 0.897, 64: 0.958, 32: 0.960, 16: 0.959).
#ifndef FSDP_GRID_UNSHARD_MAPPED
#define FSDP_GRID_UNSHARD_MAPPED 32
#endif
#ifndef FSDP_GRID_GATHER
#define FSDP_GRID_GATHER 256
#endif
// The unfused copy-in of the own slice only (one destination): 32 (large
// 0.999, ragged 0.80; at 256 the ragged layer measured 0.71).
#ifndef FSDP_GRID_OWN
#define FSDP_GRID_OWN 32
#endif
// The unfused RS copy-in (large 0.956 -> 1.013, HSDP (2,4) 0.952 -> 1.015
// at 128 against one wave).
#ifndef FSDP_GRID_RSIN
#define FSDP_GRID_RSIN 128
#endif

// fallback_per_sm: blocks per SM when the launch stays at one wave (0 = as
// many as fit). map_waves: a table with a tile -> run map is exempt from
// the one-wave rule below.
// Copy and apply launches over a table with a tile -> run map take many
// waves too when set (as the staged reduces do). Off by default: the
// copy-out, the direct unshard and the one-destination copy-in pass it
// themselves (2000-parameter layer, timed inside the step: copy-out 0.94 ->
// 0.965 with its own grid, one-destination copy-in 0.930 -> 0.941; unshard
// timed alone 0.91 -> 0.924); the apply measured slower with it (0.941 ->
// 0.934).
#ifndef FSDP_COPY_MAP_WAVES
#define FSDP_COPY_MAP_WAVES 0
#endif
#ifndef FSDP_AGOUT_MAP_WAVES
#define FSDP_AGOUT_MAP_WAVES 1
#endif
#ifndef FSDP_OWN_MAP_WAVES
#define FSDP_OWN_MAP_WAVES 1
#endif
#ifndef FSDP_UNSHARD_MAP_WAVES
#define FSDP_UNSHARD_MAP_WAVES 1
#endif
// A fused copy-in whose shard group has one rank writes one destination:
// it takes the own-slice copy-in's grid.
#ifndef FSDP_ONE_DEST_OWN
#define FSDP_ONE_DEST_OWN 1
#endif
template <typename F>
cudaError_t go(F kernel, const KArgs& a, cudaStream_t st, int threads = kThreads, size_t smem = 0,
               int grid_per_sm = 0, int fallback_per_sm = 0, bool map_waves = FSDP_COPY_MAP_WAVES != 0) {
    const void* fn = reinterpret_cast<const void*>(kernel);
    sm_count();
    const int resident = blocks_per_sm(fn, threads, smem);  // also raises the smem limit once
    const int64_t warps = a.ntiles * a.reps;
    int per_sm = grid_per_sm > 0 ? grid_per_sm : resident;
    // Many waves pay off unless a launch is short AND its table is long: a
    // warp's first lookup searches the runs from the start, and with few
    // tiles per warp that search is paid over and over. A launch with fewer
    // than 100 tiles per resident warp over more than kWaveMaxRuns runs
    // (the 2000-parameter pure-TP layer: copy-in 0.884 at one wave, 0.759
    // with many) stays at one wave; a short launch over few runs takes many
    // (HSDP (2,4) apply, 36 runs: 0.967 -> 1.000). A tile written to several
    // destinations counts once per destination.
    const int64_t dests = a.fuse ? a.S : (a.dests > 1 ? a.dests : 1);
    if (per_sm > resident && !(map_waves && a.tile_run) && a.nseg > kWaveMaxRuns &&
        warps * dests < (int64_t)resident * sm_count() * (threads / 32) * 100)
        per_sm = fallback_per_sm > 0 && fallback_per_sm < resident ? fallback_per_sm : resident;
    const int64_t want = (warps + threads / 32 - 1) / (threads / 32);
    int64_t cap = (int64_t)sm_count() * per_sm;
    if (a.max_grid > 0 && a.max_grid < cap) cap = a.max_grid;
    const int grid = (int)(want < cap ? want : cap);
    kernel<<<grid, threads, smem, st>>>(a);
    return cudaGetLastError();
}

// Blocks per SM of the fused reduce: many waves of short-lived blocks (the
// tiles in flight at any time then form one contiguous window of the
// table): large (2,8) layer 0.948 -> 1.046 of the measured copy peak,
// ragged 0.918 -> 1.001 at 256 blocks per SM (64: 1.025 / 0.988, 128:
// 1.037 / 0.998); with the read-only exit wait the shapes that fan out to
// their replicas gain too (HSDP (2,4) 0.959 -> 1.032). A launch that stays
// at one wave (the 2000-parameter layer) uses the plan's staged_blocks.
#ifndef FSDP_GRID_RSAR
#define FSDP_GRID_RSAR 256
#endif
int rsar_grid(bool) { return FSDP_GRID_RSAR; }

// Blocks per SM of the unfused ReduceScatter: with 4 sources or fewer a
// step moves few bytes and one wave of 4 blocks per SM measured best (HSDP
// (2,4): 0.758 -> 0.992 of the measured copy peak; many waves 0.935); with
// 8 or more, many waves like the fused reduce (large 0.94 -> 1.02, ragged
// 0.93 -> 1.03).
int rs_grid(int ns) { return ns <= 4 ? 4 : FSDP_GRID_RSAR; }
// The unfused AllReduce also runs many waves (large layer, 2 replicas:
// 0.886 -> 1.012; pure-TP, 8 replicas with fan-out: 0.90 -> 0.99).
int ar_grid(bool) { return FSDP_GRID_RSAR; }
// per_sm < 0: the plan's staged_blocks (the fused reduce's policy); 0: as
// many blocks as fit; > 0: that many.
template <typename S, typename F>
cudaError_t go_staged(F kernel, const KArgs& a, cudaStream_t st, int ns, int nd, bool fan = false,
                      int per_sm = -1) {
    const size_t per_warp = Staging<S>::warp_bytes(ns, nd) + (fan ? 2 * fan_img_bytes<1>() : 0);
    const int policy = FSDP_GRID_STAGED > 0 ? FSDP_GRID_STAGED : a.staged_blocks;
    // a staged reduce over a table with a tile -> run map takes many waves
    // even when short (2000-parameter layer: fused reduce 0.927 -> 0.996)
    return go(kernel, a, st, kStagedWarps * 32, kStagedWarps * per_warp, per_sm >= 0 ? per_sm : policy, policy,
              true);
}

// A staged reduce on a capped grid: one block per SM with `warps_max` warps
// (fewer if their staging rings do not fit), at most a.max_grid blocks.
template <typename S, typename F>
cudaError_t go_sm(F kernel, const KArgs& a, cudaStream_t st, int ns, int nd, bool fan, int warps_max) {
    const size_t per_warp = Staging<S, kSmRG>::warp_bytes(ns, nd) + (fan ? 2 * fan_img_bytes<kSmRG>() : 0);
    int warps = (int)(kSmBlockSmem / per_warp);
    if (warps > warps_max) warps = warps_max;
    if (warps < 1) warps = 1;
    const size_t smem = (size_t)warps * per_warp;
    blocks_per_sm(reinterpret_cast<const void*>(kernel), warps * 32, smem);  // raises the smem limit once
    const int64_t want = (a.ntiles * a.reps + warps - 1) / warps;
    const int64_t cap = a.max_grid > 0 ? a.max_grid : sm_count();
    const int grid = (int)(want < cap ? want : cap);
    kernel<<<grid, warps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

// The staged reduce fits when its per-block shared memory stays well inside
// one SM's 227 KB (up to 32 bf16 or ~26 fp32 sources).
template <typename S>
bool staged_fits(int ns, int nd) {
    return ns <= kMaxStagedSources && nd <= kMaxStagedSources &&
           kStagedWarps * Staging<S>::warp_bytes(ns, nd) <= 200 * 1024;
}

}  // namespace

cudaError_t launch(Kind kind, int sdt, int ddt, const KArgs& a, cudaStream_t st) {
    const bool sf = sdt == FSDP_F32, df = ddt == FSDP_F32;
    switch (kind) {
        case K_AGIN:
            if (sf && df) return go(ag_copy_in_kernel<float, float>, a, st, kThreads, copy_img_bytes<float>());
            if (sf) return go(ag_copy_in_kernel<float, uint16_t>, a, st, kThreads, copy_img_bytes<uint16_t>());
            // one destination (the own slice, or a shard group of one rank):
            // the own-slice policy, many waves over a mapped table too
            // (2000-parameter pure-TP layer: fused copy-in 0.92 -> 0.965)
            if (!a.fuse || (FSDP_ONE_DEST_OWN && a.S == 1))
                return FSDP_ALIGNED_COPIES && a.aligned_runs
                           ? go(ag_copy_in_kernel<uint16_t, uint16_t, true>, a, st, kThreads,
                                copy_img_bytes<uint16_t>(), FSDP_GRID_OWN, 0, FSDP_OWN_MAP_WAVES != 0)
                           : go(ag_copy_in_kernel<uint16_t, uint16_t>, a, st, kThreads, copy_img_bytes<uint16_t>(),
                                FSDP_GRID_OWN, 0, FSDP_OWN_MAP_WAVES != 0);
            return FSDP_ALIGNED_COPIES && a.aligned_runs
                       ? go(ag_copy_in_kernel<uint16_t, uint16_t, true>, a, st, kThreads, copy_img_bytes<uint16_t>(),
                            FSDP_GRID_MULTI)
                       : go(ag_copy_in_kernel<uint16_t, uint16_t>, a, st, kThreads, copy_img_bytes<uint16_t>(),
                            FSDP_GRID_MULTI);
        case K_GATHER:
            return sf ? go(ag_gather_kernel<float>, a, st, kThreads, copy_img_bytes<float>())
                      : go(ag_gather_kernel<uint16_t>, a, st, kThreads, copy_img_bytes<uint16_t>(), FSDP_GRID_GATHER);
        case K_UNSHARD:
            if (sf && df) return go(ag_unshard_kernel<float, float>, a, st, kThreads, copy_img_bytes<float>());
            if (sf) return go(ag_unshard_kernel<float, uint16_t>, a, st, kThreads, copy_img_bytes<uint16_t>());
            return go(ag_unshard_kernel<uint16_t, uint16_t>, a, st, kThreads, copy_img_bytes<uint16_t>(),
                      a.tile_run ? FSDP_GRID_UNSHARD_MAPPED : FSDP_GRID_UNSHARD, 0, FSDP_UNSHARD_MAP_WAVES != 0);
        case K_AGOUT:
            if (sf) return go(ag_copy_out_kernel<float>, a, st);
            return FSDP_ALIGNED_COPIES && a.aligned_runs
                       ? go(ag_copy_out_kernel<uint16_t, true>, a, st, kThreads, 0,
                            a.tile_run ? FSDP_GRID_COPY_MAPPED : FSDP_GRID_COPY, 0, FSDP_AGOUT_MAP_WAVES != 0)
                       : go(ag_copy_out_kernel<uint16_t>, a, st, kThreads, 0,
                            a.shifted ? FSDP_GRID_COPY_SHIFTED
                                      : (a.tile_run ? FSDP_GRID_COPY_MAPPED : FSDP_GRID_COPY),
                            0, FSDP_AGOUT_MAP_WAVES != 0);
        case K_RSIN:
            return sf ? go(rs_copy_in_kernel<float>, a, st)
                      : go(rs_copy_in_kernel<uint16_t>, a, st, kThreads, 0, FSDP_GRID_RSIN);
        case K_RSAR:
            if (a.max_grid > 0) {
                // a capped grid: the bulk-fed reduce where its ring fits
                bool used = false;
                const cudaError_t e = launch_bulk_reduce(sdt, a, st, &used);
                if (used) return e;
            }
            if (a.sg_tab && a.max_grid > 0) {
                // the apply folded in, on a capped grid: one block per SM
                if (sf)
                    return go_sm<float>(rs_ar_reduce_apply_sm_kernel<float, 0, 0, 0>, a, st, a.W, 2 * a.D, false,
                                        sm_warps<K_RSAR, float, 0, 0>());
#define FSDP_RSAR_AP_SM(W_, S_)                                                                               \
    if (a.W == W_ && a.S == S_)                                                                               \
        return go_sm<uint16_t>(rs_ar_reduce_apply_sm_kernel<uint16_t, W_, S_, W_ / S_>, a, st, W_, 2 * (W_ / S_), \
                               fan_out<K_RSAR, W_, W_ / S_>(), sm_warps<K_RSAR, uint16_t, W_, 2 * (W_ / S_)>());
                FSDP_RSAR_AP_SM(16, 8) FSDP_RSAR_AP_SM(8, 4) FSDP_RSAR_AP_SM(8, 8) FSDP_RSAR_AP_SM(8, 1)
#undef FSDP_RSAR_AP_SM
                return go_sm<uint16_t>(rs_ar_reduce_apply_sm_kernel<uint16_t, 0, 0, 0>, a, st, a.W, 2 * a.D, false,
                                       sm_warps<K_RSAR, uint16_t, 0, 0>());
            }
            if (a.sg_tab) {
                // the apply folded in (can_fold_apply said the shape fits);
                // each stage holds 2 * D destination pointers
                if (sf) {
                    if (a.W == 4 && a.S == 4)
                        return go_staged<float>(rs_ar_reduce_apply_kernel<float, 4, 4, 1>, a, st, 4, 2, false,
                                                rsar_grid(false));
                    return go_staged<float>(rs_ar_reduce_apply_kernel<float, 0, 0, 0>, a, st, a.W, 2 * a.D, false,
                                            rsar_grid(false));
                }
#define FSDP_RSAR_AP(W_, S_)                                                                                \
    if (a.W == W_ && a.S == S_)                                                                             \
        return go_staged<uint16_t>(rs_ar_reduce_apply_kernel<uint16_t, W_, S_, W_ / S_>, a, st, W_, 2 * (W_ / S_), \
                                   fan_out<K_RSAR, W_, W_ / S_>(), rsar_grid(fan_out<K_RSAR, W_, W_ / S_>()));
                FSDP_RSAR_AP(16, 8) FSDP_RSAR_AP(8, 4) FSDP_RSAR_AP(8, 8) FSDP_RSAR_AP(8, 1) FSDP_RSAR_AP(4, 4)
#undef FSDP_RSAR_AP
                return go_staged<uint16_t>(rs_ar_reduce_apply_kernel<uint16_t, 0, 0, 0>, a, st, a.W, 2 * a.D, false,
                                           rsar_grid(false));
            }
            if (a.max_grid > 0 && (sf ? staged_fits<float>(a.W, a.D) : staged_fits<uint16_t>(a.W, a.D))) {
                if (sf) {
                    if (a.W == 4 && a.S == 4)
                        return go_sm<float>(rs_ar_reduce_sm_kernel<float, 4, 4, 1>, a, st, 4, 1, false,
                                            sm_warps<K_RSAR, float, 4, 1>());
                    return go_sm<float>(rs_ar_reduce_sm_kernel<float, 0, 0, 0>, a, st, a.W, a.D, false,
                                        sm_warps<K_RSAR, float, 0, 0>());
                }
#define FSDP_RSAR_SM(W_, S_)                                                                                    \
    if (a.W == W_ && a.S == S_)                                                                                 \
        return go_sm<uint16_t>(rs_ar_reduce_sm_kernel<uint16_t, W_, S_, W_ / S_>, a, st, W_, W_ / S_,           \
                               fan_out<K_RSAR, W_, W_ / S_>(), sm_warps<K_RSAR, uint16_t, W_, W_ / S_>());
                FSDP_RSAR_SM(16, 8) FSDP_RSAR_SM(8, 4) FSDP_RSAR_SM(8, 8) FSDP_RSAR_SM(8, 1) FSDP_RSAR_SM(4, 4)
#undef FSDP_RSAR_SM
                return go_sm<uint16_t>(rs_ar_reduce_sm_kernel<uint16_t, 0, 0, 0>, a, st, a.W, a.D, false,
                                       sm_warps<K_RSAR, uint16_t, 0, 0>());
            }
            if (sf) {
                if (!staged_fits<float>(a.W, a.D)) return go(rs_ar_reduce_wide_kernel<float>, a, st);
                if (a.W == 4 && a.S == 4)
                    return go_staged<float>(rs_ar_reduce_kernel<float, 4, 4, 1>, a, st, 4, 1, false, rsar_grid(false));
                return go_staged<float>(rs_ar_reduce_kernel<float, 0, 0, 0>, a, st, a.W, a.D, false, rsar_grid(false));
            }
            if (!staged_fits<uint16_t>(a.W, a.D)) return go(rs_ar_reduce_wide_kernel<uint16_t>, a, st);
#define FSDP_RSAR(W_, S_)                                                                               \
    if (a.W == W_ && a.S == S_)                                                                         \
        return go_staged<uint16_t>(rs_ar_reduce_kernel<uint16_t, W_, S_, W_ / S_>, a, st, W_, W_ / S_, \
                                   fan_out<K_RSAR, W_, W_ / S_>(), rsar_grid(fan_out<K_RSAR, W_, W_ / S_>()));
            FSDP_RSAR(16, 8) FSDP_RSAR(8, 4) FSDP_RSAR(8, 8) FSDP_RSAR(8, 1) FSDP_RSAR(16, 16)
            FSDP_RSAR(16, 4) FSDP_RSAR(4, 4) FSDP_RSAR(4, 2) FSDP_RSAR(4, 1) FSDP_RSAR(2, 2) FSDP_RSAR(2, 1)
#undef FSDP_RSAR
            return go_staged<uint16_t>(rs_ar_reduce_kernel<uint16_t, 0, 0, 0>, a, st, a.W, a.D, false,
                                       rsar_grid(false));
        case K_RS:
            // one rank per shard group: a widening copy
            if (a.S == 1)
                return sf ? go(rs_reduce_copy_kernel<float>, a, st)
                          : go(rs_reduce_copy_kernel<uint16_t>, a, st, kThreads, 0, FSDP_GRID_COPY);
            if (a.max_grid > 0 && (sf ? staged_fits<float>(a.S, 1) : staged_fits<uint16_t>(a.S, 1))) {
                if (sf) return go_sm<float>(rs_reduce_sm_kernel<float, 0>, a, st, a.S, 1, false, sm_warps<K_RS, float, 0, 1>());
                if (a.S == 8)
                    return go_sm<uint16_t>(rs_reduce_sm_kernel<uint16_t, 8>, a, st, 8, 1, false,
                                           sm_warps<K_RS, uint16_t, 8, 1>());
                if (a.S == 4)
                    return go_sm<uint16_t>(rs_reduce_sm_kernel<uint16_t, 4>, a, st, 4, 1, false,
                                           sm_warps<K_RS, uint16_t, 4, 1>());
                return go_sm<uint16_t>(rs_reduce_sm_kernel<uint16_t, 0>, a, st, a.S, 1, false,
                                       sm_warps<K_RS, uint16_t, 0, 1>());
            }
            if (sf)
                return staged_fits<float>(a.S, 1)
                           ? go_staged<float>(rs_reduce_kernel<float, 0>, a, st, a.S, 1, false, rs_grid(a.S))
                           : go(rs_reduce_wide_kernel<float>, a, st);
            if (!staged_fits<uint16_t>(a.S, 1)) return go(rs_reduce_wide_kernel<uint16_t>, a, st);
            if (a.S == 8) return go_staged<uint16_t>(rs_reduce_kernel<uint16_t, 8>, a, st, 8, 1, false, rs_grid(8));
            if (a.S == 4) return go_staged<uint16_t>(rs_reduce_kernel<uint16_t, 4>, a, st, 4, 1, false, rs_grid(4));
            return go_staged<uint16_t>(rs_reduce_kernel<uint16_t, 0>, a, st, a.S, 1, false, rs_grid(a.S));
        case K_AR:
            if (!staged_fits<float>(a.D, a.D)) return go(ar_reduce_wide_kernel, a, st);
            if (a.max_grid > 0) {
                if (a.D == 2)
                    return go_sm<float>(ar_reduce_sm_kernel<2>, a, st, 2, 2, fan_out<K_AR, 2, 2>(),
                                        sm_warps<K_AR, float, 2, 2>());
                if (a.D == 8)
                    return go_sm<float>(ar_reduce_sm_kernel<8>, a, st, 8, 8, fan_out<K_AR, 8, 8>(),
                                        sm_warps<K_AR, float, 8, 8>());
                return go_sm<float>(ar_reduce_sm_kernel<0>, a, st, a.D, a.D, false, sm_warps<K_AR, float, 0, 0>());
            }
            if (a.D == 2)
                return go_staged<float>(ar_reduce_kernel<2>, a, st, 2, 2, fan_out<K_AR, 2, 2>(),
                                        ar_grid(fan_out<K_AR, 2, 2>()));
            if (a.D == 8)
                return go_staged<float>(ar_reduce_kernel<8>, a, st, 8, 8, fan_out<K_AR, 8, 8>(),
                                        ar_grid(fan_out<K_AR, 8, 8>()));
            return go_staged<float>(ar_reduce_kernel<0>, a, st, a.D, a.D, false, ar_grid(false));
        case K_APPLY:
            return df ? go(apply_grads_kernel<float>, a, st)
                      : go(apply_grads_kernel<uint16_t>, a, st, kThreads, 0, FSDP_GRID_APPLY);
    }
    return cudaErrorInvalidValue;
}

bool can_fold_apply(int src_dt, int W, int D) {
    return src_dt == FSDP_F32 ? staged_fits<float>(W, 2 * D) : staged_fits<uint16_t>(W, 2 * D);
}

}  // namespace fsdp
