// C-ABI entry points of the GB300 HSDP data path: plan construction and
// queries (host only), device upload of the work tables, pointer-table
// bindings, and argument checking for the data calls, which each enqueue one
// kernel (fsdp_kernels.cu).
//
// Sources, by page title + section:
//   [FS-RFC]  "【RFC】FullyShard 多维并行适配设计方案" (hyper-parallel issue 1)
//   [OVERLAP] "Hyper通信掩盖方案" (hyper-parallel issue 184), PR #758 write-up
//   [RAGGED]  FSDP dim-0 uneven-sharding RFC (hyper-parallel issue 319)
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <utility>

#include "fsdp_internal.h"

namespace fsdp {

namespace {
thread_local std::string g_error;
std::atomic<uint64_t> g_launches{0};
}  // namespace

int set_error(int code, const std::string& msg) {
    g_error = msg;
    return code;
}
void clear_error() { g_error.clear(); }
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

Seg make_seg(int64_t n, int64_t dst_off, int64_t src_off, int p, int row) {
    Seg g;
    g.n = n;
    g.dst_off = dst_off;
    g.src_off = src_off;
    g.p = p;
    g.row = row;
    return g;
}

// The runs of one slice row (for_each_row_run) appended to out.
void row_runs(const fsdp_plan_s& pl, int s, int64_t row_base, int64_t row_len, bool data_src_full,
              std::vector<Seg>& out) {
    for_each_row_run(pl, s, row_base, row_len, data_src_full,
                     [&](int64_t n, int64_t dst_off, int64_t src_off, int p, int row) {
                         out.push_back(make_seg(n, dst_off, src_off, p, row));
                     });
}

void tile_prefix(const std::vector<Seg>& segs, int dst_es, std::vector<int64_t>& tiles) {
    tiles.assign(segs.size() + 1, 0);
    for (size_t k = 0; k < segs.size(); ++k) {
        int64_t phase = ((segs[k].dst_off * dst_es) & 15) / dst_es;
        tiles[k + 1] = tiles[k] + (segs[k].n + phase + kWarpTile - 1) / kWarpTile;
    }
}

#ifndef FSDP_SPREAD_SHORT_RUNS
#define FSDP_SPREAD_SHORT_RUNS 1
#endif
// Spreads a table's short runs (fewer than 4 warp tiles: latency-bound, a
// lookup and a few loads per tile) evenly among its long runs, each list
// keeping its order, so that short tiles are always mixed with streaming
// ones instead of filling one end of the launch. The kernels take runs in
// any order; the long runs keep theirs (the apply and copy-out list them
// last first, see below). Used for the copy-out and apply tables of more
// than 1024 runs: on the 2000-parameter layer (1912 short parameters after
// 88 long ones) copy-out 0.948 -> 0.962 and apply 0.943 -> 0.952 of the
// measured copy peak, inside the step on one GB300; its copy-in did not
// move (0.932 / 0.930), and the 64-parameter ragged layer's copy-out lost
// (0.988 -> 0.969), so shorter tables keep their order.
void spread_short_runs(std::vector<Seg>& segs, int dst_es) {
    constexpr size_t kSpreadMinRuns = 1024;
    if (!FSDP_SPREAD_SHORT_RUNS || segs.size() <= kSpreadMinRuns) return;
    constexpr int64_t kShortTiles = 4;
    auto tiles_of = [&](const Seg& g) {
        const int64_t phase = ((g.dst_off * dst_es) & 15) / dst_es;
        return (g.n + phase + kWarpTile - 1) / kWarpTile;
    };
    std::vector<Seg> lng, sht;
    int64_t lt = 0, st = 0;
    for (const Seg& g : segs) {
        if (tiles_of(g) >= kShortTiles) {
            lng.push_back(g);
            lt += tiles_of(g);
        } else {
            sht.push_back(g);
            st += tiles_of(g);
        }
    }
    if (lng.empty() || sht.empty()) return;
    segs.clear();
    size_t j = 0;
    int64_t lt_done = 0, st_done = 0;
    for (const Seg& g : lng) {
        segs.push_back(g);
        lt_done += tiles_of(g);
        // short tiles so far : long tiles so far = st : lt
        while (j < sht.size() && (st_done + tiles_of(sht[j])) * lt <= lt_done * st) {
            st_done += tiles_of(sht[j]);
            segs.push_back(sht[j++]);
        }
    }
    while (j < sht.size()) segs.push_back(sht[j++]);
}

}  // namespace

void build_tables(const fsdp_plan_s& pl, std::vector<Seg> segs[T_COUNT],
                  std::vector<int64_t> tiles[T_COUNT]) {
    const int64_t sf = pl.slice(FSDP_F32);
    for (int s = 0; s < pl.S; ++s) row_runs(pl, s, 0, sf, true, segs[T_RSAR]);
    tile_prefix(segs[T_RSAR], 4, tiles[T_RSAR]);

    const int dts[2] = {FSDP_F32, FSDP_BF16};
    for (int i = 0; i < 2; ++i) {
        const int dt = dts[i], es = elem_size(dt);
        const int64_t sl = pl.slice(dt);
        // copy-in: row s of the all-gather buffer, from the local shards
        for (int s = 0; s < pl.S; ++s) row_runs(pl, s, s * sl, sl, false, segs[T_AGIN_F32 + i]);
        tile_prefix(segs[T_AGIN_F32 + i], es, tiles[T_AGIN_F32 + i]);
        // all-gather: whole slice s
        for (int s = 0; s < pl.S; ++s)
            if (sl > 0) segs[T_GATHER_F32 + i].push_back(make_seg(sl, s * sl, s * sl, 0, s));
        tile_prefix(segs[T_GATHER_F32 + i], es, tiles[T_GATHER_F32 + i]);
        // copy-out: shard s of parameter p goes to rows [off, off+len) of p.
        // Listed last parameter first: the copy-in before it in a step
        // writes the gathered rows in the opposite order, so the copy-out
        // starts on the rows still in L2 (runs may come in any order).
        for (int p = pl.P - 1; p >= 0; --p)
            for (int s = pl.S - 1; s >= 0; --s) {
                int64_t n = pl.len[(size_t)p * pl.S + s] * pl.inner[p];
                if (n == 0) continue;
                segs[T_AGOUT_F32 + i].push_back(
                    make_seg(n, pl.off[(size_t)p * pl.S + s] * pl.inner[p], s * sl + pl.o[p], p, s));
            }
        spread_short_runs(segs[T_AGOUT_F32 + i], es);
        tile_prefix(segs[T_AGOUT_F32 + i], es, tiles[T_AGOUT_F32 + i]);
        // direct unshard: shard s of parameter p (held by shard-group member
        // s) goes to rows [off, off+len) of p, no gathered buffer in between
        for (int p = 0; p < pl.P; ++p)
            for (int s = 0; s < pl.S; ++s) {
                int64_t n = pl.len[(size_t)p * pl.S + s] * pl.inner[p];
                if (n == 0) continue;
                segs[T_UNSHARD_F32 + i].push_back(make_seg(n, pl.off[(size_t)p * pl.S + s] * pl.inner[p], 0, p, s));
            }
        tile_prefix(segs[T_UNSHARD_F32 + i], es, tiles[T_UNSHARD_F32 + i]);
        // RS copy-in: row s of the RS input, from the full gradients
        for (int s = 0; s < pl.S; ++s) row_runs(pl, s, s * sl, sl, true, segs[T_RSIN_F32 + i]);
        tile_prefix(segs[T_RSIN_F32 + i], es, tiles[T_RSIN_F32 + i]);
        // unfused RS: row s of an RS input of this dtype into the f32 region
        for (int s = 0; s < pl.S; ++s)
            if (sf > 0) segs[T_RS_F32 + i].push_back(make_seg(sf, 0, s * sl, 0, s));
        tile_prefix(segs[T_RS_F32 + i], 4, tiles[T_RS_F32 + i]);
    }
    // apply: actual shard s of parameter p, from o_p of the fused region.
    // Listed last shard row and parameter first: the fused reduce before it
    // writes the fused rows in the opposite order, so the apply starts on
    // the fused elements still in L2.
    for (int s = pl.S - 1; s >= 0; --s)
        for (int p = pl.P - 1; p >= 0; --p) {
            int64_t n = pl.len[(size_t)p * pl.S + s] * pl.inner[p];
            if (n > 0) segs[T_APPLY].push_back(make_seg(n, 0, pl.o[p], p, s));
        }
    spread_short_runs(segs[T_APPLY], 4);
    tile_prefix(segs[T_APPLY], 4, tiles[T_APPLY]);
    // unfused AR: the whole fused region of shard rank s
    for (int s = 0; s < pl.S; ++s)
        if (sf > 0) segs[T_AR].push_back(make_seg(sf, 0, 0, 0, s));
    tile_prefix(segs[T_AR], 4, tiles[T_AR]);
}

namespace {

// One table's runs against the buffers its kernel reads and writes:
// dst_len(g) / src_len(g) give the element count of the buffer a run writes
// / reads (-1: the run reads nothing); rows_of(g) the destination extent the
// runs of that row must tile exactly (each element written once), keyed by
// key(g). Returns "" or the first violation.
template <typename DstLen, typename SrcLen, typename Key>
std::string check_runs(const char* name, const std::vector<Seg>& segs, const std::vector<int64_t>& tiles,
                       int dst_es, DstLen dst_len, SrcLen src_len, Key key,
                       const std::vector<std::pair<int64_t, int64_t>>& extents) {
    char buf[256];
    if (tiles.size() != segs.size() + 1 || tiles[0] != 0) return std::string(name) + ": bad tile prefix size";
    // destination coverage per key: sorted runs must tile [lo, hi) exactly
    std::vector<std::vector<std::pair<int64_t, int64_t>>> cover(extents.size());
    for (size_t k = 0; k < segs.size(); ++k) {
        const Seg& g = segs[k];
        const int64_t phase = ((g.dst_off * dst_es) & 15) / dst_es;
        if (g.n <= 0) {
            snprintf(buf, sizeof buf, "%s: run %zu is empty", name, k);
            return buf;
        }
        if (tiles[k + 1] - tiles[k] != (g.n + phase + kWarpTile - 1) / kWarpTile) {
            snprintf(buf, sizeof buf, "%s: run %zu has a wrong tile count", name, k);
            return buf;
        }
        const int64_t dl = dst_len(g), sl = src_len(g);
        if (g.dst_off < 0 || g.dst_off + g.n > dl) {
            snprintf(buf, sizeof buf, "%s: run %zu writes [%lld, %lld) of a %lld-element buffer", name, k,
                     (long long)g.dst_off, (long long)(g.dst_off + g.n), (long long)dl);
            return buf;
        }
        if (sl >= 0 && (g.src_off < 0 || g.src_off + g.n > sl)) {
            snprintf(buf, sizeof buf, "%s: run %zu reads [%lld, %lld) of a %lld-element buffer", name, k,
                     (long long)g.src_off, (long long)(g.src_off + g.n), (long long)sl);
            return buf;
        }
        const size_t c = key(g);
        if (c >= cover.size()) {
            snprintf(buf, sizeof buf, "%s: run %zu has an out-of-range key", name, k);
            return buf;
        }
        cover[c].push_back({g.dst_off, g.dst_off + g.n});
    }
    for (size_t c = 0; c < cover.size(); ++c) {
        auto& v = cover[c];
        std::sort(v.begin(), v.end());
        int64_t at = extents[c].first;
        for (const auto& r : v) {
            if (r.first != at) {
                snprintf(buf, sizeof buf, "%s: destination %zu %s at element %lld", name, c,
                         r.first > at ? "has a gap" : "is written twice", (long long)at);
                return buf;
            }
            at = r.second;
        }
        if (at != extents[c].second) {
            snprintf(buf, sizeof buf, "%s: destination %zu ends at %lld, not %lld", name, c, (long long)at,
                     (long long)extents[c].second);
            return buf;
        }
    }
    return "";
}

}  // namespace

}  // namespace fsdp

using namespace fsdp;

namespace {

#define FSDP_CHECK_PLAN(pl)                                                     \
    do {                                                                        \
        if (!(pl)) return set_error(FSDP_ERR_INVALID_ARG, "plan is NULL");      \
    } while (0)

int cuda_fail(cudaError_t e, const char* what) {
    return set_error(FSDP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool role_is_per_param(int role) {
    return role == FSDP_ROLE_SHARDS || role == FSDP_ROLE_FULL_PARAMS || role == FSDP_ROLE_GRADS ||
           role == FSDP_ROLE_SHARD_GRADS;
}

// Element count a buffer of `role` at table index i must hold.
int64_t required_numel(const fsdp_plan_s& pl, int role, int dt, int i) {
    switch (role) {
        case FSDP_ROLE_SHARDS:
        case FSDP_ROLE_SHARD_GRADS: {
            int w = i / pl.P, p = i % pl.P;
            return pl.len[(size_t)p * pl.S + (w % pl.S)] * pl.inner[p];
        }
        case FSDP_ROLE_FULL_PARAMS:
        case FSDP_ROLE_GRADS: {
            int p = i % pl.P;
            return pl.d0[p] * pl.inner[p];
        }
        case FSDP_ROLE_AG_OUTPUT:
        case FSDP_ROLE_RS_INPUT:
            return pl.S * pl.slice(dt);
        case FSDP_ROLE_FUSED:
            return pl.slice(FSDP_F32);
    }
    return -1;
}

const char* role_name(int role) {
    static const char* names[] = {"SHARDS", "AG_OUTPUT", "FULL_PARAMS", "GRADS",
                                  "RS_INPUT", "FUSED", "SHARD_GRADS"};
    return role >= 0 && role <= 6 ? names[role] : "?";
}

int check_binding(const fsdp_plan_s* pl, fsdp_binding_t b, int role, const char* what) {
    if (!b) return set_error(FSDP_ERR_INVALID_ARG, std::string(what) + ": binding is NULL");
    if (b->plan != pl)
        return set_error(FSDP_ERR_INVALID_ARG, std::string(what) + ": binding belongs to another plan");
    if (b->role != role)
        return set_error(FSDP_ERR_INVALID_ARG, std::string(what) + ": expected a " + role_name(role) +
                                                   " binding, got " + role_name(b->role));
    return FSDP_OK;
}

int check_ready(const fsdp_plan_s* pl, const char* what) {
    if (!pl) return set_error(FSDP_ERR_INVALID_ARG, std::string(what) + ": plan is NULL");
    if (!pl->uploaded)
        return set_error(FSDP_ERR_INVALID_ARG, std::string(what) + ": plan not uploaded (fsdp_plan_upload)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, what);
    if (dev != pl->device)
        return set_error(FSDP_ERR_INVALID_ARG, std::string(what) + ": current device " +
                                                   std::to_string(dev) + " is not the plan's device " +
                                                   std::to_string(pl->device));
    return FSDP_OK;
}

KArgs base_args(const fsdp_plan_s* pl, TableId t, int reps) {
    KArgs a;
    std::memset(&a, 0, sizeof a);
    a.segs = pl->tables[t].segs;
    a.tile_begin = pl->tables[t].tile_begin;
    a.tile_run = pl->tables[t].tile_run;
    a.nseg = pl->tables[t].nseg;
    a.ntiles = pl->tables[t].ntiles;
    a.reps = reps;
    a.P = pl->P;
    a.S = pl->S;
    a.D = pl->D;
    a.W = pl->W;
    a.max_grid = pl->max_grid;
    a.staged_blocks = pl->staged_blocks;
    a.status = pl->dev_status;
    a.wait_ns = pl->wait_ns;
    a.stall = pl->stall;
    set_divisor(a, 1);
    return a;
}

int run(Kind kind, int sdt, int ddt, const KArgs& a, fsdp_stream_t stream, const char* what) {
    if (a.ntiles == 0 || a.reps == 0) return FSDP_OK;  // nothing to do, no launch
    cudaError_t e = launch(kind, sdt, ddt, a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, what);
    count_launch();
    return FSDP_OK;
}

}  // namespace

extern "C" {

const char* fsdp_last_error(void) { return g_error.c_str(); }

uint64_t fsdp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int fsdp_plan_create(int n_params, const int64_t* dim0, const int64_t* inner, int rank_size,
                     int shard_size, int enable_param_shard, int shard_dim, fsdp_plan_t* out) {
    return fsdp_plan_create_bucketed(n_params, dim0, inner, nullptr, rank_size, shard_size,
                                     enable_param_shard, shard_dim, out);
}

int fsdp_plan_create_bucketed(int n_params, const int64_t* dim0, const int64_t* inner, const int* bucket,
                              int rank_size, int shard_size, int enable_param_shard, int shard_dim,
                              fsdp_plan_t* out) {
    clear_error();
    if (!out) return set_error(FSDP_ERR_INVALID_ARG, "plan_create: out is NULL");
    *out = nullptr;
    if (n_params < 0 || (n_params > 0 && (!dim0 || !inner)))
        return set_error(FSDP_ERR_INVALID_ARG, "plan_create: bad parameter list");
    if (rank_size < 1) return set_error(FSDP_ERR_INVALID_ARG, "plan_create: rank_size must be >= 1");
    // [FS-RFC §2.2.3 option A, §2.2.5 item 3]: sharding disabled -> shard_size 1.
    const int S = enable_param_shard ? shard_size : 1;
    if (S < 1 || rank_size % S != 0)
        return set_error(FSDP_ERR_INVALID_ARG,
                         "plan_create: shard_size must be >= 1 and divide rank_size");
    // [RAGGED §3.2]: uneven sharding of a dim other than 0 is out of scope.
    if (shard_dim != 0)
        return set_error(FSDP_ERR_NOT_IMPLEMENTED, "plan_create: only shard_dim 0 is supported");
    fsdp_plan_s* pl = new (std::nothrow) fsdp_plan_s;
    if (!pl) return set_error(FSDP_ERR_NOMEM, "plan_create: out of host memory");
    pl->P = n_params;
    pl->W = rank_size;
    pl->S = S;
    pl->D = rank_size / S;  // dp_size = rank_size // shard_size [FS-RFC §2.2.5]
    pl->d0.assign(dim0, dim0 + n_params);
    pl->inner.assign(inner, inner + n_params);
    pl->chunk.resize(n_params);
    pl->off.resize((size_t)n_params * S);
    pl->len.resize((size_t)n_params * S);
    pl->o.assign(n_params + 1, 0);
    int64_t end = 0;  // end of the previous parameter's padded region
    for (int p = 0; p < n_params; ++p) {
        if (dim0[p] < 0 || inner[p] < 1) {
            delete pl;
            return set_error(FSDP_ERR_INVALID_ARG, "plan_create: parameter " + std::to_string(p) +
                                                       " needs dim0 >= 0 and inner >= 1");
        }
        if (bucket && (bucket[p] < 0 || (p > 0 && bucket[p] < bucket[p - 1]))) {
            delete pl;
            return set_error(FSDP_ERR_INVALID_ARG,
                             "plan_create: bucket ids must be >= 0 and follow the registration order");
        }
        // [OVERLAP PR #758 §二.1, AllReduceParamGroup]: a new bucket starts
        // at the next multiple of 256 elements (512 B in bf16 and in fp32).
        if (bucket && p > 0 && bucket[p] != bucket[p - 1]) end = (end + 255) / 256 * 256;
        pl->o[p] = end;
        // [RAGGED §6.4]: chunk = ceil(dim0 / S); shard s starts at
        // min(s * chunk, dim0) and holds min(chunk, dim0 - start) rows.
        const int64_t c = (dim0[p] + S - 1) / S;
        pl->chunk[p] = c;
        for (int s = 0; s < S; ++s) {
            const int64_t start = std::min<int64_t>((int64_t)s * c, dim0[p]);
            pl->off[(size_t)p * S + s] = start;
            pl->len[(size_t)p * S + s] = std::min<int64_t>(c, dim0[p] - start);
        }
        // The slice offset advances by padded_sharded_param_size.numel().
        end = pl->o[p] + c * inner[p];
    }
    pl->o[n_params] = end;
    pl->sum_padded = end;
    *out = pl;
    return FSDP_OK;
}

int fsdp_plan_destroy(fsdp_plan_t pl) {
    clear_error();
    if (!pl) return FSDP_OK;
    if (pl->dev_block) cudaFree(pl->dev_block);
    delete pl;
    return FSDP_OK;
}

int fsdp_plan_upload(fsdp_plan_t pl) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (pl->uploaded) return FSDP_OK;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "plan_upload");
    std::vector<Seg> segs[T_COUNT];
    std::vector<int64_t> tiles[T_COUNT];
    build_tables(*pl, segs, tiles);
    // Share of the fused region's data in runs whose bf16 source is shifted
    // against the fp32 destination's 16-byte grid (16-byte aligned buffers
    // assumed): picks the staged reduce's blocks per SM.
    {
        pl->staged_blocks = staged_blocks_for(segs[T_RSAR].data(), segs[T_RSAR].size());
        // the same measure for the bf16 copy-out (16-byte aligned buffers)
        int64_t shifted = 0, total = 0;
        for (const Seg& g : segs[T_AGOUT_BF16]) {
            total += g.n;
            if ((((g.src_off - g.dst_off) * 2) & 15) != 0) shifted += g.n;
        }
        pl->agout_shifted = 2 * shifted > total;
    }
    // Per table: the runs, the tile prefix and, for tables of more than
    // kMapMinRuns runs, the run of every tile, so that a lookup that jumps
    // far costs one load instead of three or more rounds of search. Shorter
    // tables search their prefix, which stays in the L1 cache; there the map
    // (one entry per tile) measured slower (HSDP (2,4) copy-in 1.012 ->
    // 0.994 of the measured copy peak; 2000-parameter layer 0.89 -> 0.92).
    constexpr size_t kMapMinRuns = 1024;
    size_t bytes = 0;
    size_t seg_at[T_COUNT], tile_at[T_COUNT], run_at[T_COUNT];
    bool mapped[T_COUNT];
    for (int t = 0; t < T_COUNT; ++t) {
        seg_at[t] = bytes;
        bytes += (segs[t].size() * sizeof(Seg) + 255) / 256 * 256;
        tile_at[t] = bytes;
        bytes += (tiles[t].size() * sizeof(int64_t) + 255) / 256 * 256;
        run_at[t] = bytes;
        mapped[t] = segs[t].size() > kMapMinRuns;
        if (mapped[t]) bytes += ((size_t)tiles[t].back() * sizeof(int32_t) + 255) / 256 * 256;
    }
    // the status word of the kernels that wait inside (zero: nothing ran out)
    const size_t status_at = bytes;
    bytes += 256;
    std::vector<unsigned char> host(bytes, 0);
    for (int t = 0; t < T_COUNT; ++t) {
        if (!segs[t].empty()) std::memcpy(&host[seg_at[t]], segs[t].data(), segs[t].size() * sizeof(Seg));
        std::memcpy(&host[tile_at[t]], tiles[t].data(), tiles[t].size() * sizeof(int64_t));
        if (!mapped[t]) continue;
        int32_t* run = reinterpret_cast<int32_t*>(&host[run_at[t]]);
        for (size_t k = 0; k < segs[t].size(); ++k)
            for (int64_t i = tiles[t][k]; i < tiles[t][k + 1]; ++i) run[i] = (int32_t)k;
    }
    void* block = nullptr;
    e = cudaMalloc(&block, bytes);
    if (e != cudaSuccess) return set_error(FSDP_ERR_NOMEM, std::string("plan_upload: ") + cudaGetErrorString(e));
    e = cudaMemcpy(block, host.data(), bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(block);
        return cuda_fail(e, "plan_upload");
    }
    pl->dev_block = block;
    pl->dev_status = reinterpret_cast<int*>(static_cast<char*>(block) + status_at);
    for (int t = 0; t < T_COUNT; ++t) {
        pl->tables[t].segs = reinterpret_cast<const Seg*>(static_cast<char*>(block) + seg_at[t]);
        pl->tables[t].tile_begin = reinterpret_cast<const int64_t*>(static_cast<char*>(block) + tile_at[t]);
        pl->tables[t].tile_run =
            mapped[t] ? reinterpret_cast<const int32_t*>(static_cast<char*>(block) + run_at[t]) : nullptr;
        pl->tables[t].nseg = (int)segs[t].size();
        pl->tables[t].ntiles = tiles[t].back();
        if (t == T_AGIN_BF16 || t == T_AGOUT_BF16) {
            bool any = false;
            for (const Seg& g : segs[t])
                if (g.p >= 0 && (((g.src_off - g.dst_off) * 2) & 15) != 0) any = true;
            pl->tables[t].any_shifted = any;
        }
    }
    pl->device = dev;
    if (cudaDeviceGetAttribute(&pl->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        pl->sm_count = 0;
    }
    pl->uploaded = true;
    return FSDP_OK;
}

int fsdp_plan_check_tables(fsdp_plan_t pl) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    std::vector<Seg> segs[T_COUNT];
    std::vector<int64_t> tiles[T_COUNT];
    build_tables(*pl, segs, tiles);
    const int S = pl->S, P = pl->P;
    auto shard_n = [&](int p, int s) { return pl->len[(size_t)p * S + s] * pl->inner[p]; };
    auto full_n = [&](int p) { return pl->d0[p] * pl->inner[p]; };
    const int64_t sf = pl->slice(FSDP_F32);
    const std::vector<std::pair<int64_t, int64_t>> none;
    std::string err;
    // one extent per shard row s of a slice-sized region
    auto rows = [&](int64_t sl, bool stacked) {
        std::vector<std::pair<int64_t, int64_t>> v;
        for (int s = 0; s < S; ++s) v.push_back({stacked ? s * sl : 0, stacked ? (s + 1) * sl : sl});
        return v;
    };
    std::vector<std::pair<int64_t, int64_t>> per_param;
    for (int p = 0; p < P; ++p) per_param.push_back({0, full_n(p)});
    std::vector<std::pair<int64_t, int64_t>> per_shard;  // key p*S + s
    for (int p = 0; p < P; ++p)
        for (int s = 0; s < S; ++s) per_shard.push_back({0, shard_n(p, s)});
    auto row_key = [](const Seg& g) { return (size_t)g.row; };
    auto param_key = [](const Seg& g) { return (size_t)g.p; };

    err = check_runs("fused RS+AR", segs[T_RSAR], tiles[T_RSAR], 4, [&](const Seg&) { return sf; },
                     [&](const Seg& g) { return g.p < 0 ? (int64_t)-1 : full_n(g.p); }, row_key, rows(sf, false));
    for (int i = 0; i < 2 && err.empty(); ++i) {
        const int dt = i == 0 ? FSDP_F32 : FSDP_BF16, es = elem_size(dt);
        const int64_t sl = pl->slice(dt);
        const char* tag = i == 0 ? " (f32)" : " (bf16)";
        err = check_runs((std::string("all-gather copy-in") + tag).c_str(), segs[T_AGIN_F32 + i], tiles[T_AGIN_F32 + i],
                         es, [&](const Seg&) { return S * sl; },
                         [&](const Seg& g) { return g.p < 0 ? (int64_t)-1 : shard_n(g.p, g.row); }, row_key,
                         rows(sl, true));
        if (err.empty())
            err = check_runs((std::string("all-gather") + tag).c_str(), segs[T_GATHER_F32 + i],
                             tiles[T_GATHER_F32 + i], es, [&](const Seg&) { return S * sl; },
                             [&](const Seg&) { return S * sl; }, row_key, rows(sl, true));
        if (err.empty())
            err = check_runs((std::string("copy-out") + tag).c_str(), segs[T_AGOUT_F32 + i], tiles[T_AGOUT_F32 + i],
                             es, [&](const Seg& g) { return full_n(g.p); }, [&](const Seg&) { return S * sl; },
                             param_key, per_param);
        if (err.empty())
            err = check_runs((std::string("direct unshard") + tag).c_str(), segs[T_UNSHARD_F32 + i],
                             tiles[T_UNSHARD_F32 + i], es, [&](const Seg& g) { return full_n(g.p); },
                             [&](const Seg& g) { return shard_n(g.p, g.row); }, param_key, per_param);
        if (err.empty())
            err = check_runs((std::string("RS copy-in") + tag).c_str(), segs[T_RSIN_F32 + i], tiles[T_RSIN_F32 + i],
                             es, [&](const Seg&) { return S * sl; },
                             [&](const Seg& g) { return g.p < 0 ? (int64_t)-1 : full_n(g.p); }, row_key,
                             rows(sl, true));
        if (err.empty())
            err = check_runs((std::string("unfused RS") + tag).c_str(), segs[T_RS_F32 + i], tiles[T_RS_F32 + i], 4,
                             [&](const Seg&) { return sf; }, [&](const Seg&) { return S * sl; }, row_key,
                             rows(sf, false));
    }
    if (err.empty())
        err = check_runs("apply", segs[T_APPLY], tiles[T_APPLY], 4,
                         [&](const Seg& g) { return shard_n(g.p, g.row); }, [&](const Seg&) { return sf; },
                         [&](const Seg& g) { return (size_t)g.p * S + g.row; }, per_shard);
    if (err.empty())
        err = check_runs("unfused AR", segs[T_AR], tiles[T_AR], 4, [&](const Seg&) { return sf; },
                         [&](const Seg&) { return sf; }, row_key, rows(sf, false));
    if (!err.empty()) return set_error(FSDP_ERR_INVALID_ARG, "plan_check_tables: " + err);
    return FSDP_OK;
}

int fsdp_plan_set_grid_limit(fsdp_plan_t pl, int max_blocks) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (max_blocks < 0) return set_error(FSDP_ERR_INVALID_ARG, "plan_set_grid_limit: max_blocks must be >= 0");
    pl->max_grid = max_blocks;
    return FSDP_OK;
}

int fsdp_plan_set_wait_limit(fsdp_plan_t pl, uint64_t nanoseconds) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    pl->wait_ns = nanoseconds ? nanoseconds : 1000000000ull;
    return FSDP_OK;
}

int fsdp_plan_inject_stall(fsdp_plan_t pl, int on) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    pl->stall = on ? 1 : 0;
    return FSDP_OK;
}

int fsdp_plan_status(fsdp_plan_t pl, fsdp_stream_t stream, int* status) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "plan_status"))) return rc;
    if (!status) return set_error(FSDP_ERR_INVALID_ARG, "plan_status: status is NULL");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, pl->dev_status, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(pl->dev_status, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "plan_status");
    *status = v;
    return FSDP_OK;
}

int fsdp_plan_info(fsdp_plan_t pl, int* rank_size, int* shard_size, int* dp_size, int* n_params,
                   int64_t* sum_padded) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (rank_size) *rank_size = pl->W;
    if (shard_size) *shard_size = pl->S;
    if (dp_size) *dp_size = pl->D;
    if (n_params) *n_params = pl->P;
    if (sum_padded) *sum_padded = pl->sum_padded;
    return FSDP_OK;
}

int fsdp_slice_numel(fsdp_plan_t pl, int dt, int64_t* out) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (!out || elem_size(dt) == 0) return set_error(FSDP_ERR_INVALID_ARG, "slice_numel: bad argument");
    *out = pl->slice(dt);
    return FSDP_OK;
}

int fsdp_sharded_size(fsdp_plan_t pl, int p, int s, int64_t* offset_rows, int64_t* length_rows) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (p < 0 || p >= pl->P || s < 0 || s >= pl->S)
        return set_error(FSDP_ERR_INVALID_ARG, "sharded_size: parameter or shard rank out of range");
    if (offset_rows) *offset_rows = pl->off[(size_t)p * pl->S + s];
    if (length_rows) *length_rows = pl->len[(size_t)p * pl->S + s];
    return FSDP_OK;
}

int fsdp_padded_sharded_param_size(fsdp_plan_t pl, int p, int64_t* chunk_rows) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (p < 0 || p >= pl->P || !chunk_rows)
        return set_error(FSDP_ERR_INVALID_ARG, "padded_sharded_param_size: bad argument");
    *chunk_rows = pl->chunk[p];
    return FSDP_OK;
}

int fsdp_offsets(fsdp_plan_t pl, int64_t* offsets) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (!offsets) return set_error(FSDP_ERR_INVALID_ARG, "offsets: out is NULL");
    std::copy(pl->o.begin(), pl->o.end(), offsets);
    return FSDP_OK;
}

int fsdp_group_ranks(fsdp_plan_t pl, int w, int* shard_group, int* replicate_group) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    if (w < 0 || w >= pl->W) return set_error(FSDP_ERR_INVALID_ARG, "group_ranks: rank out of range");
    const int d = w / pl->S, s = w % pl->S;
    if (shard_group)
        for (int k = 0; k < pl->S; ++k) shard_group[k] = d * pl->S + k;
    if (replicate_group)
        for (int k = 0; k < pl->D; ++k) replicate_group[k] = k * pl->S + s;
    return FSDP_OK;
}

int fsdp_comm_calls(fsdp_plan_t pl, int* rs_group_size, int* ar_group_size) {
    clear_error();
    FSDP_CHECK_PLAN(pl);
    // [FS-RFC §2.2.2]: RS over the shard group iff S > 1; AR over the
    // replicate group iff dp_size > 1.
    if (rs_group_size) *rs_group_size = pl->S > 1 ? pl->S : 0;
    if (ar_group_size) *ar_group_size = pl->D > 1 ? pl->D : 0;
    return FSDP_OK;
}

int fsdp_bind(fsdp_plan_t pl, int role, int dt, const void* const* dev_ptrs, const int64_t* numels,
              fsdp_binding_t* out) {
    clear_error();
    if (!out) return set_error(FSDP_ERR_INVALID_ARG, "bind: out is NULL");
    *out = nullptr;
    FSDP_CHECK_PLAN(pl);
    if (!pl->uploaded) return set_error(FSDP_ERR_INVALID_ARG, "bind: plan not uploaded");
    if (role < FSDP_ROLE_SHARDS || role > FSDP_ROLE_SHARD_GRADS)
        return set_error(FSDP_ERR_INVALID_ARG, "bind: unknown role");
    const int es = elem_size(dt);
    if (es == 0) return set_error(FSDP_ERR_INVALID_ARG, "bind: unknown dtype");
    if (role == FSDP_ROLE_FUSED && dt != FSDP_F32)
        return set_error(FSDP_ERR_INVALID_ARG, "bind: FUSED buffers are fp32");
    const int count = role_is_per_param(role) ? pl->W * pl->P : pl->W;
    if (count > 0 && !dev_ptrs) return set_error(FSDP_ERR_INVALID_ARG, "bind: dev_ptrs is NULL");
    bool aligned16 = true;
    for (int i = 0; i < count; ++i) {
        const int64_t need = required_numel(*pl, role, dt, i);
        const uintptr_t a = reinterpret_cast<uintptr_t>(dev_ptrs[i]);
        if (numels && numels[i] < need)
            return set_error(FSDP_ERR_INVALID_ARG, std::string("bind: ") + role_name(role) + " buffer " +
                                                       std::to_string(i) + " holds " + std::to_string(numels[i]) +
                                                       " elements, needs " + std::to_string(need));
        if (need > 0 && a == 0)
            return set_error(FSDP_ERR_INVALID_ARG, std::string("bind: ") + role_name(role) + " buffer " +
                                                       std::to_string(i) + " is NULL");
        if (a % (uintptr_t)es != 0)
            return set_error(FSDP_ERR_INVALID_ARG, std::string("bind: ") + role_name(role) + " buffer " +
                                                       std::to_string(i) + " is not element aligned");
        if (need > 0 && (a & 15u) != 0) aligned16 = false;
    }
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "bind");
    if (dev != pl->device) return set_error(FSDP_ERR_INVALID_ARG, "bind: current device is not the plan's device");
    fsdp_binding_s* b = new (std::nothrow) fsdp_binding_s;
    if (!b) return set_error(FSDP_ERR_NOMEM, "bind: out of host memory");
    b->plan = pl;
    b->role = role;
    b->dt = dt;
    b->count = count;
    b->aligned16 = aligned16;
    if (count > 0) {
        e = cudaMalloc(reinterpret_cast<void**>(&b->dev_table), sizeof(void*) * count);
        if (e != cudaSuccess) {
            delete b;
            return set_error(FSDP_ERR_NOMEM, std::string("bind: ") + cudaGetErrorString(e));
        }
        e = cudaMemcpy(b->dev_table, dev_ptrs, sizeof(void*) * count, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cudaFree(b->dev_table);
            delete b;
            return cuda_fail(e, "bind");
        }
    }
    *out = b;
    return FSDP_OK;
}

int fsdp_binding_destroy(fsdp_binding_t b) {
    clear_error();
    if (!b) return FSDP_OK;
    if (b->dev_table) cudaFree(b->dev_table);
    delete b;
    return FSDP_OK;
}

int fsdp_ag_copy_in(fsdp_plan_t pl, fsdp_binding_t shards, fsdp_binding_t ag_out, int fuse_gather,
                    fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "ag_copy_in"))) return rc;
    if ((rc = check_binding(pl, shards, FSDP_ROLE_SHARDS, "ag_copy_in"))) return rc;
    if ((rc = check_binding(pl, ag_out, FSDP_ROLE_AG_OUTPUT, "ag_copy_in"))) return rc;
    // the all-gather dtype may narrow the parameter dtype, never widen it
    if (shards->dt == FSDP_BF16 && ag_out->dt == FSDP_F32)
        return set_error(FSDP_ERR_INVALID_ARG, "ag_copy_in: bf16 shards cannot be gathered as f32");
    KArgs a = base_args(pl, ag_out->dt == FSDP_F32 ? T_AGIN_F32 : T_AGIN_BF16, pl->D);
    a.src_tab = shards->dev_table;
    a.dst_tab = ag_out->dev_table;
    a.fuse = fuse_gather ? 1 : 0;
    a.vec = ag_out->aligned16;
    a.aligned_runs = !pl->tables[ag_out->dt == FSDP_F32 ? T_AGIN_F32 : T_AGIN_BF16].any_shifted &&
                     shards->aligned16 && ag_out->aligned16;
    return run(K_AGIN, shards->dt, ag_out->dt, a, stream, "ag_copy_in");
}

int fsdp_ag_gather(fsdp_plan_t pl, fsdp_binding_t ag_out, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "ag_gather"))) return rc;
    if ((rc = check_binding(pl, ag_out, FSDP_ROLE_AG_OUTPUT, "ag_gather"))) return rc;
    if (pl->S == 1) return FSDP_OK;  // a one-member group has nothing to gather
    KArgs a = base_args(pl, ag_out->dt == FSDP_F32 ? T_GATHER_F32 : T_GATHER_BF16, pl->D);
    a.src_tab = ag_out->dev_table;
    a.dst_tab = ag_out->dev_table;
    a.vec = ag_out->aligned16;
    a.dests = pl->S - 1;
    return run(K_GATHER, ag_out->dt, ag_out->dt, a, stream, "ag_gather");
}

int fsdp_ag_copy_out(fsdp_plan_t pl, fsdp_binding_t ag_out, fsdp_binding_t full, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "ag_copy_out"))) return rc;
    if ((rc = check_binding(pl, ag_out, FSDP_ROLE_AG_OUTPUT, "ag_copy_out"))) return rc;
    if ((rc = check_binding(pl, full, FSDP_ROLE_FULL_PARAMS, "ag_copy_out"))) return rc;
    if (ag_out->dt != full->dt)
        return set_error(FSDP_ERR_INVALID_ARG, "ag_copy_out: gathered and full dtypes differ");
    KArgs a = base_args(pl, full->dt == FSDP_F32 ? T_AGOUT_F32 : T_AGOUT_BF16, pl->W);
    a.src_tab = ag_out->dev_table;
    a.dst_tab = full->dev_table;
    a.vec = full->aligned16;
    a.shifted = pl->agout_shifted ? 1 : 0;
    a.aligned_runs = !pl->tables[full->dt == FSDP_F32 ? T_AGOUT_F32 : T_AGOUT_BF16].any_shifted &&
                     ag_out->aligned16 && full->aligned16;
    return run(K_AGOUT, ag_out->dt, full->dt, a, stream, "ag_copy_out");
}

int fsdp_ag_unshard(fsdp_plan_t pl, fsdp_binding_t shards, fsdp_binding_t full, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "ag_unshard"))) return rc;
    if ((rc = check_binding(pl, shards, FSDP_ROLE_SHARDS, "ag_unshard"))) return rc;
    if ((rc = check_binding(pl, full, FSDP_ROLE_FULL_PARAMS, "ag_unshard"))) return rc;
    if (shards->dt == FSDP_BF16 && full->dt == FSDP_F32)
        return set_error(FSDP_ERR_INVALID_ARG, "ag_unshard: bf16 shards cannot be gathered as f32");
    // one repetition per replica: each shard tile is read once and written
    // to every shard-group member's full parameter
    KArgs a = base_args(pl, full->dt == FSDP_F32 ? T_UNSHARD_F32 : T_UNSHARD_BF16, pl->D);
    a.dests = pl->S;
    a.src_tab = shards->dev_table;
    a.dst_tab = full->dev_table;
    a.vec = full->aligned16;
    return run(K_UNSHARD, shards->dt, full->dt, a, stream, "ag_unshard");
}

int fsdp_rs_copy_in(fsdp_plan_t pl, fsdp_binding_t grads, fsdp_binding_t rs_in, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "rs_copy_in"))) return rc;
    if ((rc = check_binding(pl, grads, FSDP_ROLE_GRADS, "rs_copy_in"))) return rc;
    if ((rc = check_binding(pl, rs_in, FSDP_ROLE_RS_INPUT, "rs_copy_in"))) return rc;
    if (grads->dt != rs_in->dt)
        return set_error(FSDP_ERR_INVALID_ARG, "rs_copy_in: gradient and RS input dtypes differ");
    KArgs a = base_args(pl, rs_in->dt == FSDP_F32 ? T_RSIN_F32 : T_RSIN_BF16, pl->W);
    a.src_tab = grads->dev_table;
    a.dst_tab = rs_in->dev_table;
    a.vec = rs_in->aligned16;
    return run(K_RSIN, grads->dt, rs_in->dt, a, stream, "rs_copy_in");
}

int fsdp_rs_ar_reduce(fsdp_plan_t pl, fsdp_binding_t grads, fsdp_binding_t fused, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "rs_ar_reduce"))) return rc;
    if ((rc = check_binding(pl, grads, FSDP_ROLE_GRADS, "rs_ar_reduce"))) return rc;
    if ((rc = check_binding(pl, fused, FSDP_ROLE_FUSED, "rs_ar_reduce"))) return rc;
    KArgs a = base_args(pl, T_RSAR, 1);
    a.src_tab = grads->dev_table;
    a.dst_tab = fused->dev_table;
    a.vec = fused->aligned16;
    return run(K_RSAR, grads->dt, FSDP_F32, a, stream, "rs_ar_reduce");
}

int fsdp_apply_grads(fsdp_plan_t pl, fsdp_binding_t fused, int op, int accumulate,
                     fsdp_binding_t shard_grads, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "apply_grads"))) return rc;
    if ((rc = check_binding(pl, fused, FSDP_ROLE_FUSED, "apply_grads"))) return rc;
    if ((rc = check_binding(pl, shard_grads, FSDP_ROLE_SHARD_GRADS, "apply_grads"))) return rc;
    if (op != FSDP_AVG && op != FSDP_SUM) return set_error(FSDP_ERR_INVALID_ARG, "apply_grads: unknown op");
    KArgs a = base_args(pl, T_APPLY, pl->D);
    a.src_tab = fused->dev_table;
    a.dst_tab = shard_grads->dev_table;
    a.vec = shard_grads->aligned16;
    a.op = op;
    a.accumulate = accumulate ? 1 : 0;
    // [OVERLAP PR #758 §二.3]: the fused buffer holds the SUM; AVG divides
    // once here, by the number of ranks that contributed (W).
    set_divisor(a, op == FSDP_AVG ? pl->W : 1);
    return run(K_APPLY, FSDP_F32, shard_grads->dt, a, stream, "apply_grads");
}

int fsdp_rs_ar_reduce_apply(fsdp_plan_t pl, fsdp_binding_t grads, fsdp_binding_t fused, int op, int accumulate,
                            fsdp_binding_t shard_grads, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "rs_ar_reduce_apply"))) return rc;
    if ((rc = check_binding(pl, grads, FSDP_ROLE_GRADS, "rs_ar_reduce_apply"))) return rc;
    if ((rc = check_binding(pl, fused, FSDP_ROLE_FUSED, "rs_ar_reduce_apply"))) return rc;
    if ((rc = check_binding(pl, shard_grads, FSDP_ROLE_SHARD_GRADS, "rs_ar_reduce_apply"))) return rc;
    if (op != FSDP_AVG && op != FSDP_SUM) return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_apply: unknown op");
    if (shard_grads->dt != grads->dt)
        return set_error(FSDP_ERR_INVALID_ARG, "rs_ar_reduce_apply: shard gradients must have the gradient dtype");
    if (!can_fold_apply(grads->dt, pl->W, pl->D)) {
        // too many sources for the staged reduce: the two calls it stands for
        if ((rc = fsdp_rs_ar_reduce(pl, grads, fused, stream))) return rc;
        return fsdp_apply_grads(pl, fused, op, accumulate, shard_grads, stream);
    }
    KArgs a = base_args(pl, T_RSAR, 1);
    a.src_tab = grads->dev_table;
    a.dst_tab = fused->dev_table;
    a.sg_tab = shard_grads->dev_table;
    a.vec = fused->aligned16;
    a.op = op;
    a.accumulate = accumulate ? 1 : 0;
    // the fused buffer keeps the raw sum; the shard gradients divide by W
    // for AVG, as fsdp_apply_grads does [OVERLAP PR #758 §二.3]
    set_divisor(a, op == FSDP_AVG ? pl->W : 1);
    // Sources mostly shifted against the fused rows (staged_blocks 3, the
    // ragged layer): the TMA-bulk-fed kernel on every SM (one block per SM)
    // measured faster than the staged one there (0.868 -> 0.967 of the
    // measured copy peak on one GB300) and slower on unshifted layers (HSDP
    // (2,4) 1.027 -> 0.927, pure-TP 0.957 -> 0.858), which keep it.
    if (a.max_grid == 0 && pl->staged_blocks == 3 && pl->sm_count > 0 &&
        bulk_reduce_fits(grads->dt, pl->W, pl->D))
        a.max_grid = pl->sm_count;
    return run(K_RSAR, grads->dt, FSDP_F32, a, stream, "rs_ar_reduce_apply");
}

int fsdp_rs_reduce(fsdp_plan_t pl, fsdp_binding_t rs_in, int op, fsdp_binding_t fused, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "rs_reduce"))) return rc;
    if ((rc = check_binding(pl, rs_in, FSDP_ROLE_RS_INPUT, "rs_reduce"))) return rc;
    if ((rc = check_binding(pl, fused, FSDP_ROLE_FUSED, "rs_reduce"))) return rc;
    if (op != FSDP_AVG && op != FSDP_SUM) return set_error(FSDP_ERR_INVALID_ARG, "rs_reduce: unknown op");
    KArgs a = base_args(pl, rs_in->dt == FSDP_F32 ? T_RS_F32 : T_RS_BF16, pl->D);
    a.src_tab = rs_in->dev_table;
    a.dst_tab = fused->dev_table;
    a.vec = fused->aligned16;
    a.op = op;
    set_divisor(a, op == FSDP_AVG ? pl->S : 1);
    return run(K_RS, rs_in->dt, FSDP_F32, a, stream, "rs_reduce");
}

int fsdp_ar_reduce(fsdp_plan_t pl, fsdp_binding_t fused, int op, fsdp_stream_t stream) {
    clear_error();
    int rc;
    if ((rc = check_ready(pl, "ar_reduce"))) return rc;
    if ((rc = check_binding(pl, fused, FSDP_ROLE_FUSED, "ar_reduce"))) return rc;
    if (op != FSDP_AVG && op != FSDP_SUM) return set_error(FSDP_ERR_INVALID_ARG, "ar_reduce: unknown op");
    // [FS-RFC §2.2.2]: no AllReduce is issued for a single replica.
    if (pl->D == 1) return FSDP_OK;
    KArgs a = base_args(pl, T_AR, 1);
    a.src_tab = fused->dev_table;
    a.dst_tab = fused->dev_table;
    a.vec = fused->aligned16;
    a.op = op;
    set_divisor(a, op == FSDP_AVG ? pl->D : 1);
    return run(K_AR, FSDP_F32, FSDP_F32, a, stream, "ar_reduce");
}

}  // extern "C"
