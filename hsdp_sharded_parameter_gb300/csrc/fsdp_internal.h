// Internal definitions shared by the host plan code, the C-ABI entry points
// and the kernels of the GB300 HSDP data path. Not installed; the public
// interface is include/hsdp_fsdp.h.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "hsdp_fsdp.h"

namespace fsdp {

// One contiguous run of work: n elements written at dst_off of the
// destination buffer(s), read from src_off of the source buffer(s). p < 0
// marks a run of zeros (padding rows, slice tails). `row` is the shard rank
// s the run belongs to; how src/dst buffers are picked from (row, p, rep)
// depends on the kernel.
struct Seg {
    int64_t n;
    int64_t dst_off;
    int64_t src_off;
    int32_t p;
    int32_t row;
};
static_assert(sizeof(Seg) == 32, "Seg is 32 bytes on host and device");

// Work is cut into warp tiles: 32 lanes x 8 steps x 8 elements. A lane
// moves 8 consecutive elements per step (16 B of bf16, 32 B of fp32), so a
// warp step covers 256 consecutive elements. Granules are anchored at
// 16-byte boundaries of the destination: a run whose first destination
// element is not 16-byte aligned starts with a partial granule.
constexpr int kGran = 8;
constexpr int kSteps = 8;
constexpr int kStepElems = 32 * kGran;            // 256 elements
constexpr int kWarpTile = kSteps * kStepElems;    // 2048 elements
constexpr int kThreads = 256;                     // copy and apply kernels
constexpr int kStagedWarps = 4;                   // warps per block, staged reduce

// Work tables. Each kernel walks one: a list of runs plus, per run, the
// index of its first warp tile (prefix sum, nseg + 1 entries).
enum TableId {
    T_RSAR = 0,        // fused RS+AR: rows of the fp32 fused region, per s
    T_AGIN_F32,        // copy-in: rows of the ag slice, per s (f32 ag dtype)
    T_AGIN_BF16,       //          (bf16 ag dtype)
    T_GATHER_F32,      // all-gather: whole slice s, per s
    T_GATHER_BF16,
    T_AGOUT_F32,       // copy-out: (p, s) pieces of the full parameters
    T_AGOUT_BF16,
    T_RSIN_F32,        // RS copy-in: rows of the RS input, per s
    T_RSIN_BF16,
    T_APPLY,           // apply: (s, p) actual-shard pieces of the fused region
    T_RS_F32,          // unfused RS: row s of an f32 RS input
    T_RS_BF16,         //             row s of a bf16 RS input
    T_AR,              // unfused AR: fp32 fused region, per s
    T_UNSHARD_F32,     // direct unshard: (p, s) shards into the full parameters
    T_UNSHARD_BF16,
    T_COUNT
};

struct Table {
    const Seg* segs = nullptr;           // device
    const int64_t* tile_begin = nullptr; // device, nseg + 1
    const int32_t* tile_run = nullptr;   // device, ntiles: the run of each tile
    int nseg = 0;
    int64_t ntiles = 0;
    // some data run's source is off its destination's 16-byte phase (with
    // 16-byte aligned buffers): the copies then need their realigning path
    bool any_shifted = true;
};

inline int elem_size(int dt) { return dt == FSDP_F32 ? 4 : (dt == FSDP_BF16 ? 2 : 0); }

// Arguments of every kernel (passed by value).
struct KArgs {
    const Seg* segs;
    const int64_t* tile_begin;
    // The run of every tile (ntiles entries), or nullptr: a lookup that
    // jumps past the next run reads it here instead of searching the prefix.
    const int32_t* tile_run;
    int nseg;
    int64_t ntiles;  // tiles of one repetition
    int reps;        // repetitions of the table (ranks or replicas)
    int P, S, D, W;
    void* const* src_tab;  // device table of source pointers
    void* const* dst_tab;  // device table of destination pointers
    int fuse;              // copy-in: also write every shard-group member
    int vec;               // 1: every destination is 16-byte aligned
    int op;                // FSDP_AVG / FSDP_SUM
    int accumulate;        // apply: add to the gradient already there
    float div;             // divisor applied after the sum (1 = none)
    // How the divisor is applied: 0 = not at all (div == 1); 1 = multiply by
    // recip = 1/div, an exact power of two (the exact quotient and the exact
    // product are the same real number, so the correctly rounded results
    // agree bit for bit, subnormals included); 2 = IEEE division.
    int scale_mode;
    float recip;
    int max_grid;  // upper bound on the launch's blocks (0 = the kernel's own grid)
    // Blocks per SM for the staged reduce (0 = as many as fit): 2 when most
    // of the fused region's data sits in runs aligned with their sources,
    // 3 when most runs are shifted (their steps do more work per byte, so
    // more warps are needed to keep the same bytes in flight).
    int staged_blocks;
    // Most of the table's data sits in runs whose source is shifted against
    // the destination's 16-byte grid (copy-out picks its grid by it).
    int shifted;
    int dests;  // destinations written per tile when more than one (the gather)
    // Copies: no run's source is shifted against its destination and both
    // bindings are 16-byte aligned, so the kernel without the realigning
    // path (fewer registers, more resident warps) may run (it still routes
    // any shifted tile through its per-granule path).
    int aligned_runs;
    // The fused reduce with the apply folded in: the [W][P] table of
    // actual-shard gradients it also writes (nullptr: not folded in).
    void* const* sg_tab;
    // Kernels that wait inside (the bulk-fed reduce of a capped grid): the
    // plan's device status word (nullptr: such kernels are not used), the
    // limit of any one wait in nanoseconds, and the failure-detection test
    // hook (nonzero: block 0 never announces its first chunk, so that waits
    // for it run out).
    int* status;
    uint64_t wait_ns;
    int stall;
};

// Fills div, scale_mode and recip for a divisor d >= 1.
inline void set_divisor(KArgs& a, int d) {
    a.div = (float)d;
    a.scale_mode = d == 1 ? 0 : ((d & (d - 1)) == 0 ? 1 : 2);
    a.recip = 1.0f / (float)d;
}

enum Kind {
    K_AGIN = 0,
    K_GATHER,
    K_AGOUT,
    K_RSIN,
    K_RSAR,
    K_RS,
    K_AR,
    K_APPLY,
    K_UNSHARD
};

// Launches the kernel of `kind` for the given element types. Returns a
// cudaError_t of the launch.
cudaError_t launch(Kind kind, int src_dt, int dst_dt, const KArgs& a, cudaStream_t stream);

// Whether the fused reduce of W sources (D replicas) of this dtype can fold
// the apply in (its staged form fits with the replicas' gradient pointers).
bool can_fold_apply(int src_dt, int W, int D);

// The fused reduce (K_RSAR, with the apply folded in when a.sg_tab is set)
// on a capped grid, fed by TMA bulk loads (fsdp_bulk.cu). Sets *used to
// false, launching nothing, when the shape does not fit its shared-memory
// ring (the caller then takes the staged kernels).
cudaError_t launch_bulk_reduce(int src_dt, const KArgs& a, cudaStream_t stream, bool* used);
// Whether that kernel's shared-memory ring fits W sources of this dtype
// (and D replicas).
bool bulk_reduce_fits(int src_dt, int W, int D);

// Status bits a kernel with internal waits sets in the plan's status word.
constexpr int kStatusProducerWait = 1;  // a stage was not released in time
constexpr int kStatusConsumerWait = 2;  // a stage's data did not arrive in time
constexpr int kStatusOrder = 4;         // a consumer found another chunk's record (internal error)

}  // namespace fsdp

struct fsdp_plan_s {
    int P = 0, W = 1, S = 1, D = 1;
    std::vector<int64_t> d0, inner, chunk, off, len, o;  // off/len: [P*S]
    int64_t sum_padded = 0;
    int device = -1;
    bool uploaded = false;
    int max_grid = 0;  // fsdp_plan_set_grid_limit
    uint64_t wait_ns = 1000000000ull;  // fsdp_plan_set_wait_limit
    int stall = 0;                     // fsdp_plan_inject_stall
    int* dev_status = nullptr;         // inside dev_block
    int sm_count = 0;                  // of the plan's device, set by fsdp_plan_upload
    int staged_blocks = 2;  // see KArgs::staged_blocks, set by fsdp_plan_upload
    bool agout_shifted = false;  // see KArgs::shifted (bf16 copy-out), set by fsdp_plan_upload
    void* dev_block = nullptr;
    fsdp::Table tables[fsdp::T_COUNT];
    int64_t slice(int dt) const {
        int64_t per = 512 / fsdp::elem_size(dt);
        return (sum_padded + per - 1) / per * per;
    }
};

struct fsdp_binding_s {
    fsdp_plan_s* plan = nullptr;
    int role = -1;
    int dt = -1;
    int count = 0;
    void** dev_table = nullptr;
    bool aligned16 = true;
};

namespace fsdp {

// Runs of one slice row s: for every parameter with a non-empty shard s, its
// actual elements at o_p, and zero runs for the padding rows between them
// and for the tail up to row_len ([RAGGED §6.4]: padding is zero); adjacent
// zero runs come out merged. data_src_full: a data run reads the full tensor
// at off_{p,s} * inner (gradients); otherwise the shard from 0. Calls
// emit(n, dst_off, src_off, p, row) once per run, in order, and allocates
// nothing (the allocation-free entry point builds its table with it too).
template <typename Emit>
void for_each_row_run(const fsdp_plan_s& pl, int s, int64_t row_base, int64_t row_len, bool data_src_full,
                      Emit&& emit) {
    int64_t zero_from = 0;
    for (int p = 0; p < pl.P; ++p) {
        const int64_t n = pl.len[(size_t)p * pl.S + s] * pl.inner[p];
        if (n == 0) continue;
        if (pl.o[p] > zero_from) emit(pl.o[p] - zero_from, row_base + zero_from, (int64_t)0, -1, s);
        const int64_t src = data_src_full ? pl.off[(size_t)p * pl.S + s] * pl.inner[p] : 0;
        emit(n, row_base + pl.o[p], src, p, s);
        zero_from = pl.o[p] + n;
    }
    if (row_len > zero_from) emit(row_len - zero_from, row_base + zero_from, (int64_t)0, -1, s);
}

// Blocks per SM of the staged fused reduce for its run table (see
// KArgs::staged_blocks): 3 when most of the data sits in runs whose bf16
// source is shifted against the fp32 destination's 16-byte grid (16-byte
// aligned buffers assumed), else 2.
inline int staged_blocks_for(const Seg* segs, size_t nseg) {
    int64_t shifted = 0, total = 0;
    for (size_t k = 0; k < nseg; ++k) {
        const Seg& g = segs[k];
        if (g.p < 0) continue;
        total += g.n;
        if ((((g.src_off - (g.dst_off & 3)) * 2) & 15) != 0) shifted += g.n;
    }
    return 2 * shifted > total ? 3 : 2;
}

int set_error(int code, const std::string& msg);
void clear_error();
void count_launch();
// Builds the host-side work tables of a plan (used by fsdp_plan_upload).
void build_tables(const fsdp_plan_s& plan, std::vector<Seg> segs[T_COUNT],
                  std::vector<int64_t> tiles[T_COUNT]);
}  // namespace fsdp
