// Kernels of the GB300 HSDP data path (sm_103a). Every kernel is HBM-bound
// data movement plus, for the gradient sync, an fp32 sum over ranks: no
// tensor cores. All of them share one work model:
//
//   * A plan-time table lists runs ("segments") of contiguous elements; a
//     prefix array gives each run's first warp tile. Tiles are 1024
//     elements: a lane moves 8 consecutive elements per step, 4 steps.
//   * A persistent grid of warps strides over (tile, repetition) pairs,
//     repetition fastest (the ranks or replicas the table is repeated for).
//     A warp finds its run with a cooperative forward search (each lane
//     tests one tile boundary; a ballot picks the run), so the cursor only
//     moves forward.
//   * Granules are anchored at 16-byte boundaries of the destination, so
//     every full granule is written with aligned 16-byte stores. Sources
//     are read with aligned 16-byte loads; when a source run is shifted
//     against its destination (ragged offsets), two neighbouring aligned
//     blocks are loaded and funnel-shifted into place. Each loaded block
//     holds at least one byte of the source run, so no load leaves the
//     source allocation's pages. Partial granules (run heads/tails) and
//     destinations that are not 16-byte aligned go element by element.
//
// Sources, by page title + section:
//   [OVERLAP] "Hyper通信掩盖方案" (hyper-parallel issue 184), PR #758 write-up
//   [RAGGED]  FSDP dim-0 uneven-sharding RFC (hyper-parallel issue 319)
//   [FS-RFC]  "【RFC】FullyShard 多维并行适配设计方案" (hyper-parallel issue 1)
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

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

// Loads the 8 elements base[e .. e+8), all inside the source run, from any
// element-aligned address.
template <typename T>
__device__ __forceinline__ void load_raw(Raw<T>& r, const T* base, int64_t e) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(base) + (uintptr_t)(e * (int64_t)sizeof(T));
    const unsigned sh = (unsigned)(a & 15u);
    const uint4* q = reinterpret_cast<const uint4*>(a - sh);
    if (sh == 0) {
#pragma unroll
        for (int v = 0; v < Raw<T>::kVec; ++v) {
            uint4 x = ld_stream(q + v);
            r.w[4 * v] = x.x; r.w[4 * v + 1] = x.y; r.w[4 * v + 2] = x.z; r.w[4 * v + 3] = x.w;
        }
    } else {
        uint4 blk[Raw<T>::kVec + 1];
#pragma unroll
        for (int v = 0; v <= Raw<T>::kVec; ++v) blk[v] = ld_reuse(q + v);
#pragma unroll
        for (int v = 0; v < Raw<T>::kVec; ++v) {
            uint4 x = funnel(blk[v], blk[v + 1], sh);
            r.w[4 * v] = x.x; r.w[4 * v + 1] = x.y; r.w[4 * v + 2] = x.z; r.w[4 * v + 3] = x.w;
        }
    }
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
__device__ __forceinline__ void load_aligned(Raw<T>& r, const T* src) {
    const uint4* q = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int v = 0; v < Raw<T>::kVec; ++v) {
        uint4 x = ld_stream(q + v);
        r.w[4 * v] = x.x; r.w[4 * v + 1] = x.y; r.w[4 * v + 2] = x.z; r.w[4 * v + 3] = x.w;
    }
}

// Raw granule <-> 8 floats.
__device__ __forceinline__ void widen(const Raw<uint16_t>& r, float (&x)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_to_f32(r.w[i] & 0xffffu);
        x[2 * i + 1] = bf16_to_f32(r.w[i] >> 16);
    }
}
__device__ __forceinline__ void widen(const Raw<float>& r, float (&x)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(r.w[i]);
}
__device__ __forceinline__ void narrow(const float (&x)[8], Raw<uint16_t>& r) {
#pragma unroll
    for (int i = 0; i < 4; ++i) r.w[i] = f32_to_bf16(x[2 * i]) | (f32_to_bf16(x[2 * i + 1]) << 16);
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

template <typename T>
__device__ __forceinline__ int phase_of(int64_t dst_off) {
    return (int)(((dst_off * (int64_t)sizeof(T)) & 15) / (int64_t)sizeof(T));
}

// ----------------------------------------------------------- work search

// Largest k with tb[k] <= tile, searching forward from k (tb strictly
// increasing, tb[nseg] > tile). Warp-uniform; all 32 lanes take part.
__device__ __forceinline__ int find_seg(const int64_t* __restrict__ tb, int nseg, int k, int64_t tile) {
    if (tile < __ldg(tb + k + 1)) return k;
    const int lane = threadIdx.x & 31;
    for (;;) {
        const int idx = k + 1 + lane;
        const bool le = idx < nseg && __ldg(tb + idx) <= tile;
        const unsigned m = __ballot_sync(kFull, le);
        if (m != kFull) return k + __popc(m);
        k += 32;
    }
}

struct WarpCursor {
    int64_t t, stride, total;
    __device__ WarpCursor(const KArgs& a) {
        t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
        stride = ((int64_t)gridDim.x * kThreads) >> 5;
        total = a.ntiles * a.reps;
    }
};

// ------------------------------------------------------------ copy kernels

// K_AGIN  : shards[(d,s),p] -> ag[(d,s)] row s (+ every shard-group member
//           with fuse); zero runs pad the rows. rep = d.
// K_GATHER: ag[(d,s)] slice s -> ag[(d,s')] slice s, s' != s. rep = d.
// K_AGOUT : ag[w] at s*slice + o_p -> full[w,p] rows [off, off+len). rep = w.
// K_RSIN  : grads[w,p] rows [off, off+len) -> rs_in[w] row s. rep = w.
template <int KIND, typename S, typename D>
__global__ void __launch_bounds__(kThreads) copy_kernel(const KArgs a) {
    const int lane = threadIdx.x & 31;
    WarpCursor c(a);
    int k = 0;
    for (int64_t t = c.t; t < c.total; t += c.stride) {
        const int64_t tile = t / a.reps;
        const int rep = (int)(t - tile * a.reps);
        k = find_seg(a.tile_begin, a.nseg, k, tile);
        const Seg sg = a.segs[k];
        const int64_t rel0 = (tile - __ldg(a.tile_begin + k)) * kWarpTile - phase_of<D>(sg.dst_off);

        const S* src = nullptr;
        int nd = 1;
        if (KIND == K_AGIN) {
            if (sg.p >= 0) src = static_cast<const S*>(a.src_tab[(int64_t)(rep * a.S + sg.row) * a.P + sg.p]);
            nd = a.fuse ? a.S : 1;
        } else if (KIND == K_GATHER) {
            src = static_cast<const S*>(a.src_tab[rep * a.S + sg.row]);
            nd = a.S - 1;
        } else if (KIND == K_AGOUT) {
            src = static_cast<const S*>(a.src_tab[rep]);
        } else {  // K_RSIN
            if (sg.p >= 0) src = static_cast<const S*>(a.src_tab[(int64_t)rep * a.P + sg.p]);
        }

        Raw<D> val[kSteps];
        bool full[kSteps];
        int64_t rel[kSteps];
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            rel[u] = rel0 + (int64_t)(u * 32 + lane) * kGran;
            full[u] = a.vec && rel[u] >= 0 && rel[u] + kGran <= sg.n;
            if (full[u]) {
                if (src) {
                    Raw<S> r;
                    load_raw(r, src, sg.src_off + rel[u]);
                    convert(r, val[u]);
                } else {
#pragma unroll
                    for (int i = 0; i < Raw<D>::kWords; ++i) val[u].w[i] = 0u;
                }
            }
        }
        for (int j = 0; j < nd; ++j) {
            D* dst;
            if (KIND == K_AGIN)
                dst = static_cast<D*>(a.dst_tab[rep * a.S + (a.fuse ? j : sg.row)]);
            else if (KIND == K_GATHER)
                dst = static_cast<D*>(a.dst_tab[rep * a.S + j + (j >= sg.row ? 1 : 0)]);
            else if (KIND == K_AGOUT)
                dst = static_cast<D*>(a.dst_tab[(int64_t)rep * a.P + sg.p]);
            else
                dst = static_cast<D*>(a.dst_tab[rep]);
            dst += sg.dst_off;
#pragma unroll
            for (int u = 0; u < kSteps; ++u) {
                if (full[u]) {
                    store_raw(dst + rel[u], val[u]);
                } else if (rel[u] < sg.n && rel[u] + kGran > 0) {
                    const int64_t lo = rel[u] < 0 ? 0 : rel[u];
                    const int64_t hi = rel[u] + kGran < sg.n ? rel[u] + kGran : sg.n;
                    for (int64_t e = lo; e < hi; ++e) {
                        if (src)
                            copy_elem<S, D>(dst, e, src, sg.src_off + e);
                        else
                            dst[e] = D(0);
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------- reduce kernels

// Folds sources in ascending index order: sources are grouped in runs of
// s_in (the shard group); each run is summed from its first term (part),
// and the runs are summed from the first run (total). [FS-RFC §2.1.3 item
// 3, §3.3]: ReduceScatter over the shard group, then AllReduce over the
// replicate group.
struct Fold {
    int s_in, i_in, n_out;
    __device__ Fold(int s) : s_in(s), i_in(0), n_out(0) {}
    template <int N>
    __device__ __forceinline__ void add(const float (&x)[N], float (&part)[N], float (&total)[N]) {
#pragma unroll
        for (int e = 0; e < N; ++e) part[e] = i_in == 0 ? x[e] : __fadd_rn(part[e], x[e]);
        if (++i_in == s_in) {
            i_in = 0;
#pragma unroll
            for (int e = 0; e < N; ++e) total[e] = n_out == 0 ? part[e] : __fadd_rn(total[e], part[e]);
            ++n_out;
        }
    }
};

constexpr int kChunk = 8;  // sources loaded together per granule

// K_RSAR: sources grads[w',p] (w' = 0..W-1, nested S x D); D destinations
//         fused[(d,s)] at o_p; zero runs write +0. reps = 1.
// K_RS  : sources rs_in[(d,s'')] row s (s'' = 0..S-1); destination
//         fused[(d,s)]; AVG divides by S. rep = d.
// K_AR  : sources fused[(d',s)] (d' = 0..D-1); destinations all fused[(d,s)]
//         in place; AVG divides by D. reps = 1.
template <int KIND, typename S>
__global__ void __launch_bounds__(kThreads) reduce_kernel(const KArgs a) {
    const int lane = threadIdx.x & 31;
    WarpCursor c(a);
    int k = 0;
    const int ns = KIND == K_RSAR ? a.W : (KIND == K_RS ? a.S : a.D);
    const int s_in = KIND == K_RSAR ? a.S : (KIND == K_RS ? a.S : 1);
    const int nd = KIND == K_RS ? 1 : a.D;
    const bool scale = a.div != 1.0f;
    for (int64_t t = c.t; t < c.total; t += c.stride) {
        const int64_t tile = t / a.reps;
        const int rep = (int)(t - tile * a.reps);
        k = find_seg(a.tile_begin, a.nseg, k, tile);
        const Seg sg = a.segs[k];
        const int64_t rel0 = (tile - __ldg(a.tile_begin + k)) * kWarpTile - phase_of<float>(sg.dst_off);

        auto src_of = [&](int i) -> const S* {
            if (KIND == K_RSAR) return static_cast<const S*>(a.src_tab[(int64_t)i * a.P + sg.p]);
            if (KIND == K_RS) return static_cast<const S*>(a.src_tab[rep * a.S + i]);
            return static_cast<const S*>(a.src_tab[i * a.S + sg.row]);
        };
        auto dst_of = [&](int j) -> float* {
            if (KIND == K_RS) return static_cast<float*>(a.dst_tab[rep * a.S + sg.row]) + sg.dst_off;
            return static_cast<float*>(a.dst_tab[j * a.S + sg.row]) + sg.dst_off;
        };

#pragma unroll 1
        for (int u = 0; u < kSteps; ++u) {
            const int64_t rel = rel0 + (int64_t)(u * 32 + lane) * kGran;
            if (rel >= sg.n || rel + kGran <= 0) continue;
            const bool full = a.vec && rel >= 0 && rel + kGran <= sg.n;
            if (full) {
                float part[8], total[8];
                if (sg.p < 0) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) total[e] = 0.0f;
                } else {
                    Fold f(s_in);
#pragma unroll 1
                    for (int i0 = 0; i0 < ns; i0 += kChunk) {
                        Raw<S> r[kChunk];
#pragma unroll
                        for (int q = 0; q < kChunk; ++q)
                            if (i0 + q < ns) load_raw(r[q], src_of(i0 + q), sg.src_off + rel);
#pragma unroll
                        for (int q = 0; q < kChunk; ++q) {
                            if (i0 + q < ns) {
                                float x[8];
                                widen(r[q], x);
                                f.add(x, part, total);
                            }
                        }
                    }
                    if (scale) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) total[e] = __fdiv_rn(total[e], a.div);
                    }
                }
                Raw<float> o;
                narrow(total, o);
                for (int j = 0; j < nd; ++j) store_raw(dst_of(j) + rel, o);
            } else {
                const int64_t lo = rel < 0 ? 0 : rel;
                const int64_t hi = rel + kGran < sg.n ? rel + kGran : sg.n;
                for (int64_t e = lo; e < hi; ++e) {
                    float v[1] = {0.0f};
                    if (sg.p >= 0) {
                        float part[1], total[1];
                        Fold f(s_in);
                        for (int i = 0; i < ns; ++i) {
                            float x[1] = {load_f32(src_of(i), sg.src_off + e)};
                            f.add(x, part, total);
                        }
                        v[0] = scale ? __fdiv_rn(total[0], a.div) : total[0];
                    }
                    for (int j = 0; j < nd; ++j) dst_of(j)[e] = v[0];
                }
            }
        }
    }
}

// ------------------------------------------------------------ apply kernel

// fused[(d,s)] at o_p -> shard_grads[(d,s),p] (actual rows only), divided
// by a.div (W for AVG), optionally added to the gradient already there,
// rounded once to the gradient dtype. rep = d.
template <typename D>
__global__ void __launch_bounds__(kThreads) apply_kernel(const KArgs a) {
    const int lane = threadIdx.x & 31;
    WarpCursor c(a);
    int k = 0;
    const bool scale = a.div != 1.0f;
    for (int64_t t = c.t; t < c.total; t += c.stride) {
        const int64_t tile = t / a.reps;
        const int rep = (int)(t - tile * a.reps);
        k = find_seg(a.tile_begin, a.nseg, k, tile);
        const Seg sg = a.segs[k];
        const int64_t rel0 = (tile - __ldg(a.tile_begin + k)) * kWarpTile - phase_of<D>(sg.dst_off);
        const int w = rep * a.S + sg.row;
        const float* src = static_cast<const float*>(a.src_tab[w]) + sg.src_off;
        D* dst = static_cast<D*>(a.dst_tab[(int64_t)w * a.P + sg.p]) + sg.dst_off;
#pragma unroll
        for (int u = 0; u < kSteps; ++u) {
            const int64_t rel = rel0 + (int64_t)(u * 32 + lane) * kGran;
            if (rel >= sg.n || rel + kGran <= 0) continue;
            if (a.vec && rel >= 0 && rel + kGran <= sg.n) {
                Raw<float> r;
                load_raw(r, src, rel);
                float x[8];
                widen(r, x);
                if (scale) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __fdiv_rn(x[e], a.div);
                }
                if (a.accumulate) {
                    Raw<D> old;
                    load_aligned(old, dst + rel);
                    float y[8];
                    widen(old, y);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __fadd_rn(y[e], x[e]);
                }
                Raw<D> o;
                narrow(x, o);
                store_raw(dst + rel, o);
            } else {
                const int64_t lo = rel < 0 ? 0 : rel;
                const int64_t hi = rel + kGran < sg.n ? rel + kGran : sg.n;
                for (int64_t e = lo; e < hi; ++e) {
                    float q = src[e];
                    if (scale) q = __fdiv_rn(q, a.div);
                    if (a.accumulate) q = __fadd_rn(load_f32(dst, e), q);
                    store_f32(dst, e, q);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ launch

int grid_for(const void* fn, int64_t warps_needed) {
    static std::mutex mu;
    static std::unordered_map<const void*, int> cache;  // resident blocks per SM
    static int sm_count = 0;
    int per_sm;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sm_count == 0) {
            int dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
            if (sm_count <= 0) sm_count = 1;
        }
        auto it = cache.find(fn);
        if (it == cache.end()) {
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, kThreads, 0) != cudaSuccess || b < 1) b = 1;
            it = cache.emplace(fn, b).first;
        }
        per_sm = it->second;
    }
    const int64_t want = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t cap = (int64_t)sm_count * per_sm;
    return (int)(want < cap ? want : cap);
}

template <typename F>
cudaError_t go(F kernel, const KArgs& a, cudaStream_t st) {
    const int grid = grid_for(reinterpret_cast<const void*>(kernel), a.ntiles * a.reps);
    kernel<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch(Kind kind, int sdt, int ddt, const KArgs& a, cudaStream_t st) {
    const bool sf = sdt == FSDP_F32, df = ddt == FSDP_F32;
    switch (kind) {
        case K_AGIN:
            if (sf && df) return go(copy_kernel<K_AGIN, float, float>, a, st);
            if (sf) return go(copy_kernel<K_AGIN, float, uint16_t>, a, st);
            return go(copy_kernel<K_AGIN, uint16_t, uint16_t>, a, st);
        case K_GATHER:
            return sf ? go(copy_kernel<K_GATHER, float, float>, a, st)
                      : go(copy_kernel<K_GATHER, uint16_t, uint16_t>, a, st);
        case K_AGOUT:
            return sf ? go(copy_kernel<K_AGOUT, float, float>, a, st)
                      : go(copy_kernel<K_AGOUT, uint16_t, uint16_t>, a, st);
        case K_RSIN:
            return sf ? go(copy_kernel<K_RSIN, float, float>, a, st)
                      : go(copy_kernel<K_RSIN, uint16_t, uint16_t>, a, st);
        case K_RSAR:
            return sf ? go(reduce_kernel<K_RSAR, float>, a, st) : go(reduce_kernel<K_RSAR, uint16_t>, a, st);
        case K_RS:
            return sf ? go(reduce_kernel<K_RS, float>, a, st) : go(reduce_kernel<K_RS, uint16_t>, a, st);
        case K_AR:
            return go(reduce_kernel<K_AR, float>, a, st);
        case K_APPLY:
            return df ? go(apply_kernel<float>, a, st) : go(apply_kernel<uint16_t>, a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fsdp
