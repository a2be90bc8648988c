// Device helpers shared by the kernels of the GB300 HSDP data path: bf16
// conversions, 16-byte vector moves and realignment, the work-table search
// and the apply's rounded store. Included by the kernel translation units
// only (each gets its own inline copies).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "fsdp_internal.h"

namespace fsdp {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------------ scalars

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// Round to nearest even by adding half an ulp of the kept part minus one,
// plus the kept part's lowest bit (ties go to the even neighbour); the
// carry propagates into the exponent, up to infinity. NaN -> 0x7FC0|sign.
__device__ __forceinline__ uint32_t f32_to_bf16(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return ((u >> 16) & 0x8000u) | 0x7fc0u;
    u += 0x7fffu + ((u >> 16) & 1u);
    return u >> 16;
}

// ------------------------------------------------------- vector memory ops

// 8 elements of T as raw 32-bit words: 4 for bf16, 8 for fp32.
template <typename T>
struct Raw {
    static constexpr int kWords = kGran * (int)sizeof(T) / 4;
    static constexpr int kVec = kWords / 4;  // 16-byte vectors
    uint32_t w[kWords];
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ uint4 ld_reuse(const uint4* p) { return __ldg(p); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }

__device__ __forceinline__ void put(uint32_t* w, uint4 x) {
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
}

// Bytes [sh, sh + 16) of the 32-byte string lo:hi (little endian).
__device__ __forceinline__ uint4 funnel(uint4 lo, uint4 hi, unsigned sh) {
    const unsigned r = (sh & 3u) * 8u;
    uint32_t a0, a1, a2, a3, a4;
    switch (sh >> 2) {
        case 0: a0 = lo.x; a1 = lo.y; a2 = lo.z; a3 = lo.w; a4 = hi.x; break;
        case 1: a0 = lo.y; a1 = lo.z; a2 = lo.w; a3 = hi.x; a4 = hi.y; break;
        case 2: a0 = lo.z; a1 = lo.w; a2 = hi.x; a3 = hi.y; a4 = hi.z; break;
        default: a0 = lo.w; a1 = hi.x; a2 = hi.y; a3 = hi.z; a4 = hi.w; break;
    }
    uint4 v;
    v.x = __funnelshift_r(a0, a1, r);
    v.y = __funnelshift_r(a1, a2, r);
    v.z = __funnelshift_r(a2, a3, r);
    v.w = __funnelshift_r(a3, a4, r);
    return v;
}

// Loads the 8 elements at byte address a (all inside the source run) from
// any element-aligned address.
template <typename T>
__device__ __forceinline__ void load_raw_at(Raw<T>& r, uintptr_t a) {
    const unsigned sh = (unsigned)(a & 15u);
    const uint4* q = reinterpret_cast<const uint4*>(a - sh);
    if (sh == 0) {
#pragma unroll
        for (int v = 0; v < Raw<T>::kVec; ++v) put(r.w + 4 * v, ld_stream(q + v));
    } else {
        uint4 blk[Raw<T>::kVec + 1];
#pragma unroll
        for (int v = 0; v <= Raw<T>::kVec; ++v) blk[v] = ld_reuse(q + v);
#pragma unroll
        for (int v = 0; v < Raw<T>::kVec; ++v) put(r.w + 4 * v, funnel(blk[v], blk[v + 1], sh));
    }
}

// One warp step (256 elements) whose source is shifted by sh (1..15) bytes
// against the destination granules. w0 is the aligned start of the step's
// source window (33 or 65 blocks). Lane l loads its own aligned blocks and
// takes the next one from lane l+1 (lane 31 loads it), so every source
// block is loaded once; all 32 lanes must take part.
// All kSteps steps of an interior tile are loaded first and shuffled after:
// a warp-synchronous shuffle keeps later loads from being issued ahead of
// it, so interleaving them would expose one memory latency per step. step
// is the byte distance between consecutive steps' windows. Only the first
// nsteps steps (warp-uniform) are loaded.
template <typename T>
__device__ __forceinline__ void load_tile_shifted(Raw<T> (&r)[kSteps], uintptr_t w0, uintptr_t step,
                                                  unsigned sh, int lane, int nsteps) {
    constexpr int kV = Raw<T>::kVec;
    uint4 blk[kSteps][kV];
    uint4 last[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
        const uint4* q = reinterpret_cast<const uint4*>(w0 + u * step) + lane * kV;
#pragma unroll
        for (int v = 0; v < kV; ++v) blk[u][v] = u < nsteps ? ld_stream(q + v) : make_uint4(0, 0, 0, 0);
        last[u] = lane == 31 && u < nsteps ? ld_stream(q + kV) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
        uint4 nx;
        nx.x = __shfl_down_sync(kFull, blk[u][0].x, 1);
        nx.y = __shfl_down_sync(kFull, blk[u][0].y, 1);
        nx.z = __shfl_down_sync(kFull, blk[u][0].z, 1);
        nx.w = __shfl_down_sync(kFull, blk[u][0].w, 1);
        if (lane == 31) nx = last[u];
#pragma unroll
        for (int v = 0; v < kV; ++v) put(r[u].w + 4 * v, funnel(blk[u][v], v + 1 < kV ? blk[u][v + 1] : nx, sh));
    }
}

template <typename T>
__device__ __forceinline__ void load_aligned(Raw<T>& r, const T* src) {
    const uint4* q = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int v = 0; v < Raw<T>::kVec; ++v) put(r.w + 4 * v, ld_stream(q + v));
}

// Stores 8 elements at a 16-byte aligned address.
template <typename T>
__device__ __forceinline__ void store_raw(T* dst, const Raw<T>& r) {
    uint4* q = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < Raw<T>::kVec; ++v)
        st_stream(q + v, make_uint4(r.w[4 * v], r.w[4 * v + 1], r.w[4 * v + 2], r.w[4 * v + 3]));
}

template <typename T>
__device__ __forceinline__ void zero_raw(Raw<T>& r) {
#pragma unroll
    for (int i = 0; i < Raw<T>::kWords; ++i) r.w[i] = 0u;
}

// Raw granule <-> 8 floats.
__device__ __forceinline__ void widen(const Raw<uint16_t>& r, float (&x)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(r.w[i] << 16);
        x[2 * i + 1] = __uint_as_float(r.w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void widen(const Raw<float>& r, float (&x)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(r.w[i]);
}
// Two floats to a packed bf16 pair (lo in bits 0-15) with the conversion
// instruction's round to nearest even (subnormals kept). Its NaN result is
// replaced by this library's NaN rule (0x7FC0 | sign).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    if (lo != lo || hi != hi) d = f32_to_bf16(lo) | (f32_to_bf16(hi) << 16);
    return d;
}

__device__ __forceinline__ void narrow(const float (&x)[8], Raw<uint16_t>& r) {
#pragma unroll
    for (int i = 0; i < 4; ++i) r.w[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
}

// The AVG divisor, applied as KArgs::scale_mode says.
__device__ __forceinline__ float scaled(float x, const KArgs& a) {
    if (a.scale_mode == 1) return __fmul_rn(x, a.recip);
    if (a.scale_mode == 2) return __fdiv_rn(x, a.div);
    return x;
}
__device__ __forceinline__ void narrow(const float (&x)[8], Raw<float>& r) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r.w[i] = __float_as_uint(x[i]);
}

// Element-wise forms for partial granules.
__device__ __forceinline__ float load_f32(const uint16_t* p, int64_t i) { return bf16_to_f32(p[i]); }
__device__ __forceinline__ float load_f32(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ void store_f32(uint16_t* p, int64_t i, float v) { p[i] = (uint16_t)f32_to_bf16(v); }
__device__ __forceinline__ void store_f32(float* p, int64_t i, float v) { p[i] = v; }

// Same-type copy keeps the bits (no float round trip); f32 -> bf16 rounds.
template <typename S, typename D>
__device__ __forceinline__ void convert(const Raw<S>& in, Raw<D>& out) {
    if constexpr (sizeof(S) == sizeof(D)) {
#pragma unroll
        for (int i = 0; i < Raw<D>::kWords; ++i) out.w[i] = in.w[i];
    } else {
        float x[8];
        widen(in, x);
        narrow(x, out);
    }
}
template <typename S, typename D>
__device__ __forceinline__ void copy_elem(D* dst, int64_t di, const S* src, int64_t si) {
    if constexpr (sizeof(S) == sizeof(D)) {
        dst[di] = *reinterpret_cast<const D*>(src + si);
    } else {
        store_f32(dst, di, load_f32(src, si));
    }
}

// ----------------------------------------------------------- work search

// Largest k with tb[k] <= tile, searching forward from k (tb strictly
// increasing, tb[k] <= tile < tb[nseg]). Warp-uniform; all 32 lanes take
// part. The common case (same or next run) costs one or two loads; a longer
// jump reads the plan's tile -> run map (one load) or, without one, narrows
// [lo, hi) 32-fold per round: lane i probes lo + i*step and a ballot counts
// the probes at or below the tile (they form a prefix).
__device__ __forceinline__ int find_seg(const int64_t* __restrict__ tb, const int32_t* __restrict__ run, int nseg,
                                        int k, int64_t tile) {
    if (tile < __ldg(tb + k + 1)) return k;
    if (k + 2 > nseg || tile < __ldg(tb + k + 2)) return k + 1;
    if (run) return __ldg(run + tile);  // a longer jump: the plan's tile -> run map
    const int lane = threadIdx.x & 31;
    int lo = k + 1, hi = nseg;  // tb[lo] <= tile < tb[hi]
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int idx = lo + lane * step;
        const bool le = idx < hi && __ldg(tb + idx) <= tile;
        const int c = __popc(__ballot_sync(kFull, le));  // >= 1: lane 0 probes lo
        const int nlo = lo + (c - 1) * step;
        const int nhi = lo + c * step;
        lo = nlo;
        hi = nhi < hi ? nhi : hi;
    }
    return lo;
}

// One warp tile: a window of up to kWarpTile elements of one run. rel0 is
// the run-relative element of lane 0's first granule (negative by the
// destination's 16-byte phase on a run's first tile).
struct Tile {
    int64_t n, dst_off, src_off, rel0;
    int p, row, rep;
};

__device__ __forceinline__ void lookup(const KArgs& a, int64_t t, int& k, int dst_es, Tile& ti) {
    const int64_t tile = t / a.reps;
    ti.rep = (int)(t - tile * a.reps);
    k = find_seg(a.tile_begin, a.tile_run, a.nseg, k, tile);
    const Seg sg = a.segs[k];
    ti.n = sg.n;
    ti.dst_off = sg.dst_off;
    ti.src_off = sg.src_off;
    ti.p = sg.p;
    ti.row = sg.row;
    ti.rel0 = (tile - __ldg(a.tile_begin + k)) * kWarpTile - ((sg.dst_off * dst_es) & 15) / dst_es;
}

__device__ __forceinline__ int64_t warp_id() { return ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; }
__device__ __forceinline__ int64_t warp_count() { return ((int64_t)gridDim.x * blockDim.x) >> 5; }

// The apply folded into the fused reduce: the 8 fused sums of a granule,
// divided as KArgs says (W for AVG), added to the gradient already there
// when accumulating, rounded once to the gradient dtype and stored at g,
// the granule's first actual-shard element of one replica. The same
// operations in the same order as the apply kernel; g may sit at any
// element alignment (16-, 8- or 2/4-byte stores).
template <typename G>
__device__ __forceinline__ void store_applied(const KArgs& a, const float (&sum)[8], G* g) {
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = a.div != 1.0f ? scaled(sum[e], a) : sum[e];
    const uintptr_t addr = reinterpret_cast<uintptr_t>(g);
    if (a.accumulate) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fadd_rn(load_f32(g, e), x[e]);
    }
    Raw<G> r;
    narrow(x, r);
    if ((addr & 15u) == 0) {
        store_raw(g, r);
    } else if ((addr & 7u) == 0) {
        uint2* q = reinterpret_cast<uint2*>(g);
#pragma unroll
        for (int v = 0; v < Raw<G>::kWords / 2; ++v) q[v] = make_uint2(r.w[2 * v], r.w[2 * v + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) store_f32(g, e, x[e]);
    }
}

}  // namespace
}  // namespace fsdp
