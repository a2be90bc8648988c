// Allocation-free variant of the fused gradient sync (fsdp_rs_ar_reduce).
//
// The regular path keeps its work tables (the runs of the fused region and
// the tables of buffer pointers) in device memory that fsdp_plan_upload and
// fsdp_bind allocate. Some callers cannot allocate device memory at all: a
// framework whose caching allocator owns every byte of the device (side
// allocations would break its accounting and fragmentation control), or a
// job running so close to the memory limit that a surprise allocation may
// fail in the middle of a step. This entry point serves them: it needs only
// a host-side plan (fsdp_plan_create) and the caller's buffers, and keeps
// its work tables in one fixed device array that is part of the library
// image, loaded with the library on every GPU that uses it and held until
// the process exits.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "fsdp_internal.h"

namespace {

constexpr size_t kScratchBytes = FSDP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The device-side work area. In host code this name is only a stand-in for
// the symbol: the kernel must be given the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host staging of the tables (static storage, no heap), guarded by g_mu.
alignas(256) unsigned char g_host_stage[kScratchBytes];
std::mutex g_mu;
void* g_dev_addr[kMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Device address of the scratch array on the current device; looked up once
// per device, with that device current.
int scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices)
        return fsdp::set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_noalloc: device index out of range");
    if (!g_dev_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fsdp::set_error(FSDP_ERR_CUDA, std::string("rs_ar_reduce_noalloc: cudaGetSymbolAddress: ") +
                                                      cudaGetErrorString(e));
        g_dev_addr[dev] = p;
    }
    *out = g_dev_addr[dev];
    return FSDP_OK;
}

// The runs of the fused region, shard row by shard row: the same builder,
// in the same order, as the uploaded table of the regular fused sync
// (fsdp::for_each_row_run). Writes up to `cap` runs; returns how many there
// are.
int64_t fused_runs(const fsdp_plan_s& pl, fsdp::Seg* out, int64_t cap) {
    const int64_t sf = pl.slice(FSDP_F32);
    int64_t n = 0;
    for (int s = 0; s < pl.S; ++s)
        fsdp::for_each_row_run(pl, s, 0, sf, true, [&](int64_t cnt, int64_t dst_off, int64_t src_off, int p, int row) {
            if (n < cap) {
                out[n].n = cnt;
                out[n].dst_off = dst_off;
                out[n].src_off = src_off;
                out[n].p = p;
                out[n].row = row;
            }
            ++n;
        });
    return n;
}

}  // namespace

extern "C" int fsdp_rs_ar_reduce_noalloc(fsdp_plan_t pl, int grad_dtype, const void* const* grads,
                                         float* const* fused, fsdp_stream_t stream) {
    using namespace fsdp;
    clear_error();
    if (!pl) return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_noalloc: plan is NULL");
    const int es = elem_size(grad_dtype);
    if (es == 0) return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_noalloc: unknown gradient dtype");
    const int W = pl->W, P = pl->P;
    if ((W * P > 0 && !grads) || !fused)
        return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_noalloc: pointer table is NULL");
    const int64_t sf = pl->slice(FSDP_F32);
    for (int i = 0; i < W * P; ++i) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(grads[i]);
        const int64_t need = pl->d0[i % P] * pl->inner[i % P];
        if ((need > 0 && a == 0) || a % (uintptr_t)es != 0)
            return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_noalloc: gradient " + std::to_string(i) +
                                                       " is NULL or not element aligned");
    }
    bool vec = true;
    for (int w = 0; w < W; ++w) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(fused[w]);
        if ((sf > 0 && a == 0) || a % 4u != 0)
            return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_noalloc: fused region " + std::to_string(w) +
                                                       " is NULL or not 4-byte aligned");
        if (a & 15u) vec = false;
    }

    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The tables are staged through host memory that the next call reuses,
    // so a copy recorded into a graph would replay another call's tables.
    cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cap_status);
    if (e != cudaSuccess) return set_error(FSDP_ERR_CUDA, std::string("rs_ar_reduce_noalloc: ") + cudaGetErrorString(e));
    if (cap_status != cudaStreamCaptureStatusNone)
        return set_error(FSDP_ERR_INVALID_ARG,
                         "rs_ar_reduce_noalloc: the stream is being captured; this call stages its tables through "
                         "a host buffer that later calls overwrite, so it is refused during capture");

    std::lock_guard<std::mutex> lock(g_mu);
    // layout: runs | tile prefix | gradient pointers [W][P] | fused pointers [W]
    Seg* runs = reinterpret_cast<Seg*>(g_host_stage);
    const int64_t cap = (int64_t)(kScratchBytes / sizeof(Seg));
    const int64_t nseg = fused_runs(*pl, runs, cap);
    const size_t off_tiles = up256((size_t)nseg * sizeof(Seg));
    const size_t off_src = off_tiles + up256((size_t)(nseg + 1) * sizeof(int64_t));
    const size_t off_dst = off_src + up256((size_t)W * P * sizeof(void*));
    const size_t bytes = off_dst + up256((size_t)W * sizeof(void*));
    if (nseg > cap || bytes > kScratchBytes)
        return set_error(FSDP_ERR_INVALID_ARG,
                         "rs_ar_reduce_noalloc: the plan needs " + std::to_string(bytes) +
                             " bytes of work tables, more than the fixed " + std::to_string(kScratchBytes) +
                             " (use fsdp_rs_ar_reduce)");
    if (nseg == 0) return FSDP_OK;  // empty fused region: nothing to write
    int64_t* tiles = reinterpret_cast<int64_t*>(g_host_stage + off_tiles);
    tiles[0] = 0;
    for (int64_t k = 0; k < nseg; ++k) {
        const int64_t phase = ((runs[k].dst_off * 4) & 15) / 4;
        tiles[k + 1] = tiles[k] + (runs[k].n + phase + kWarpTile - 1) / kWarpTile;
    }
    std::memcpy(g_host_stage + off_src, grads, (size_t)W * P * sizeof(void*));
    std::memcpy(g_host_stage + off_dst, fused, (size_t)W * sizeof(void*));

    int dev = -1;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(FSDP_ERR_CUDA, std::string("rs_ar_reduce_noalloc: ") + cudaGetErrorString(e));
    void* scratch = nullptr;
    if (int rc = scratch_address(dev, &scratch)) return rc;
    // Pageable source: the call returns once the bytes are staged, so the
    // host buffer may be reused right after; the copy is ordered before the
    // kernel on the same stream.
    e = cudaMemcpyAsync(scratch, g_host_stage, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return set_error(FSDP_ERR_CUDA, std::string("rs_ar_reduce_noalloc: ") + cudaGetErrorString(e));

    unsigned char* base = static_cast<unsigned char*>(scratch);
    KArgs a;
    std::memset(&a, 0, sizeof a);
    a.segs = reinterpret_cast<const Seg*>(base);
    a.tile_begin = reinterpret_cast<const int64_t*>(base + off_tiles);
    a.nseg = (int)nseg;
    a.ntiles = tiles[nseg];
    a.reps = 1;
    a.P = P;
    a.S = pl->S;
    a.D = pl->D;
    a.W = W;
    a.src_tab = reinterpret_cast<void* const*>(base + off_src);
    a.dst_tab = reinterpret_cast<void* const*>(base + off_dst);
    a.vec = vec ? 1 : 0;
    // the plan's grid cap (fsdp_plan_set_grid_limit) and the staged reduce's
    // blocks per SM, derived from the runs as fsdp_plan_upload derives them
    a.max_grid = pl->max_grid;
    a.staged_blocks = staged_blocks_for(runs, (size_t)nseg);
    set_divisor(a, 1);
    e = launch(K_RSAR, grad_dtype, FSDP_F32, a, st);
    if (e != cudaSuccess) return set_error(FSDP_ERR_CUDA, std::string("rs_ar_reduce_noalloc: ") + cudaGetErrorString(e));
    count_launch();
    return FSDP_OK;
}
