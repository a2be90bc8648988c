/*
 * hsdp_fsdp.h -- C ABI of the GB300 HSDP fully_shard data path with dim-0
 * ragged (uneven) parameter shards.
 *
 * All rank_size = W virtual ranks live in ONE GPU's HBM. Virtual rank w sits
 * at mesh coordinate (d, s) = (w / S, w % S): d is the replicate index
 * (0 <= d < D = dp_size), s the shard rank (0 <= s < S = shard_size). The
 * shard group of w is {d*S + k : k < S} (the ReduceScatter / AllGather
 * group); its replicate group is {k*S + s : k < D} (the AllReduce group).
 * The collectives of the pages become kernels that read and write the ranks'
 * buffers in place; there is no second GPU and no NCCL.
 *
 * Sources (page title + section):
 *   [FS-RFC]  "【RFC】FullyShard 多维并行适配设计方案" (hyper-parallel issue 1)
 *   [OVERLAP] "Hyper通信掩盖方案" (hyper-parallel issue 184) and its PR #758
 *             write-up ("方案落地说明")
 *   [RAGGED]  FSDP dim-0 uneven-sharding RFC (hyper-parallel issue 319)
 *
 * Layout (all element offsets, row-major tensors):
 *   parameter p has shape (d0_p, rest...), inner_p = prod(rest) (1 for a
 *   vector). chunk_p = ceil(d0_p / S) ("padded_sharded_param_size" rows);
 *   shard s of p holds rows [off_{p,s}, off_{p,s} + len_{p,s}) with
 *   off = min(s*chunk, d0), len = min(chunk, d0 - off) ("sharded_size",
 *   possibly 0) [RAGGED §6.4]. Inside a per-rank slice parameter p starts at
 *   o_p = sum_{q<p} chunk_q * inner_q (one bucket; several buckets: see
 *   fsdp_plan_create_bucketed) and occupies chunk_p * inner_p
 *   elements; the rows past len are zero. A slice holds slice(dt) elements:
 *   sum_p chunk_p*inner_p rounded up to a multiple of 512 bytes [OVERLAP
 *   PR #758 §二.1, the 512B-aligned fused buffer].
 *
 * Conventions for every call:
 *   - Return value: FSDP_OK (0) or an error code; the message of the last
 *     failure on the calling thread is fsdp_last_error().
 *   - Memory: the caller allocates and frees every data buffer (PyTorch
 *     here). The library owns only plans and bindings (small device tables
 *     allocated by fsdp_plan_upload / fsdp_bind and freed by the matching
 *     destroy). Data calls never allocate, never free, never synchronise.
 *   - Streams: data calls enqueue exactly one kernel on `stream` (NULL = the
 *     legacy default stream; fsdp_rs_ar_reduce_apply on a mesh too wide for
 *     its one-pass kernel enqueues the two it stands for) and return;
 *     launch failures come back as FSDP_ERR_CUDA. Calls on different streams are safe when the buffers
 *     they write are disjoint from the buffers the others touch.
 *   - Waits: no kernel waits on another kernel or on the host. The one
 *     kernel that waits inside (the fused sync on a capped grid, and the
 *     one-pass sync of a mostly shifted plan; between its own warps) bounds
 *     every wait and reports one that ran out through the plan's status
 *     word (fsdp_plan_status), not the return value.
 *   - Pointers: device pointers aligned to their element size; NULL only
 *     for a buffer of 0 elements. 16-byte-aligned pointers (every PyTorch
 *     allocation) take the vectorised path; others take an element-wise
 *     path with identical results.
 *   - Numerics: sums are IEEE binary32 additions, round to nearest even,
 *     subnormals kept, folded in ascending rank order: first over the shard
 *     group, then over the replicas. float -> bf16 rounds to nearest even;
 *     a NaN becomes the quiet NaN 0x7FC0 with its sign.
 */
#ifndef HSDP_FSDP_H
#define HSDP_FSDP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fsdp_plan_s* fsdp_plan_t;
typedef struct fsdp_binding_s* fsdp_binding_t;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* fsdp_stream_t;

enum fsdp_status {
    FSDP_OK = 0,
    FSDP_ERR_INVALID_ARG = 1,     /* bad argument, size, dtype or state */
    FSDP_ERR_NOT_IMPLEMENTED = 2, /* uneven sharding of a dim other than 0 */
    FSDP_ERR_CUDA = 3,            /* a CUDA runtime call failed */
    FSDP_ERR_NOMEM = 4            /* host or device allocation failed */
};

enum fsdp_dtype { FSDP_F32 = 0, FSDP_BF16 = 1 };

/* AVG and SUM as in [OVERLAP] PR #758 §二.3 (_resolve_default_reduce_op:
 * AVG by default, SUM for DTensor-managed parameters). */
enum fsdp_reduce_op { FSDP_AVG = 0, FSDP_SUM = 1 };

/* What a binding's pointers are. "[W][P]" tables hold one pointer per
 * (rank, parameter), index w*P + p; "[W]" tables one pointer per rank.
 * Required element counts (checked by fsdp_bind when numels is given):
 *   SHARDS       [W][P] local actual shard of p on rank w:  len_{p,s} * inner_p
 *   AG_OUTPUT    [W]    all-gather buffer of rank w:        S * slice(dt)
 *   FULL_PARAMS  [W][P] unsharded parameter p on rank w:    d0_p * inner_p
 *   GRADS        [W][P] unsharded gradient p on rank w:     d0_p * inner_p
 *   RS_INPUT     [W]    reduce-scatter input of rank w:     S * slice(dt)
 *   FUSED        [W]    fused fp32 gradient region of w:    slice(F32)   (F32 only)
 *   SHARD_GRADS  [W][P] actual-shard gradient p on rank w:  len_{p,s} * inner_p
 */
enum fsdp_role {
    FSDP_ROLE_SHARDS = 0,
    FSDP_ROLE_AG_OUTPUT = 1,
    FSDP_ROLE_FULL_PARAMS = 2,
    FSDP_ROLE_GRADS = 3,
    FSDP_ROLE_RS_INPUT = 4,
    FSDP_ROLE_FUSED = 5,
    FSDP_ROLE_SHARD_GRADS = 6
};

/* Message of the last failed call on this thread ("" if none). The string
 * stays valid until the next call on this thread. */
const char* fsdp_last_error(void);

/* Number of kernels this library has enqueued in this process. */
uint64_t fsdp_launch_count(void);

/* ---------------------------------------------------------------- plan */

/* Creates a host-only plan for n_params parameters registered in order.
 * dim0[p] >= 0 is the dim-0 length, inner[p] >= 1 the product of the other
 * dims (1 for a vector; a 0-dim scalar is passed as dim0 = 1, inner = 1).
 * rank_size = W >= 1. shard_size = S must divide W; dp_size = W / S
 * [FS-RFC §2.2.5]. enable_param_shard = 0 switches parameter sharding off
 * and forces S = 1 (AllReduce only, the pure-TP compatibility path)
 * [FS-RFC §2.2.3 option A, §4.1]. shard_dim must be 0: uneven sharding of
 * another dim is a non-goal [RAGGED §3.2] -> FSDP_ERR_NOT_IMPLEMENTED.
 * Needs no GPU. *out receives a handle owned by the caller. */
int fsdp_plan_create(int n_params, const int64_t* dim0, const int64_t* inner, int rank_size,
                     int shard_size, int enable_param_shard, int shard_dim, fsdp_plan_t* out);

/* As fsdp_plan_create, for several buckets sharing one fused buffer: the
 * AllReduceParamGroup of [OVERLAP PR #758 §二.1], which gathers the buckets
 * of one replicate group into a single 512-byte-aligned fused all-reduce.
 * bucket[p] >= 0 is parameter p's bucket, non-decreasing in registration
 * order (NULL = one bucket). Every per-rank slice holds the buckets in
 * order; a bucket starts at the next multiple of 256 elements (512 bytes
 * in bf16, 1024 in fp32), its parameters packed as in a one-bucket plan,
 * the gaps zero. One call of each data function then covers all buckets. */
int fsdp_plan_create_bucketed(int n_params, const int64_t* dim0, const int64_t* inner,
                              const int* bucket, int rank_size, int shard_size,
                              int enable_param_shard, int shard_dim, fsdp_plan_t* out);

/* Frees the plan and its device tables. The caller must ensure no enqueued
 * work still uses them (e.g. synchronise the streams first). NULL is a no-op. */
int fsdp_plan_destroy(fsdp_plan_t plan);

/* Uploads the plan's work tables to the current CUDA device (synchronous,
 * allocates device memory once: 40 bytes per run of each kernel's table,
 * plus, for tables of more than 1024 runs, 4 bytes per 2048 elements the
 * table covers, plus the plan's 4-byte status word, see fsdp_plan_status).
 * Required before any data call; data calls must then run with that device
 * current. Calling it again is a no-op. */
int fsdp_plan_upload(fsdp_plan_t plan);

/* Caps the number of thread blocks every later data call of this plan
 * launches (0, the default: each kernel's own grid, many short waves of
 * blocks on long launches). The kernels stride over their work, so any cap
 * gives the same results; a small cap leaves the other SMs to kernels
 * running beside them, e.g. the backward compute the gradient sync overlaps
 * with, the way the pages' communication streams run beside compute
 * [OVERLAP §二.2]. Under a cap the reductions run one block per SM, so
 * max_blocks is the number of SMs they occupy: the fused RS+AR (with or
 * without the apply folded in) as a producer warp feeding eight folding
 * warps through TMA bulk loads into a shared-memory ring (up to 32 sources
 * of bf16, 16 of fp32; its waits are bounded, see fsdp_plan_status), the
 * unfused ReduceScatter and AllReduce (and a fused reduce with more
 * sources) with up to 16 warps of per-warp cp.async rings. May be changed
 * between calls. */
int fsdp_plan_set_grid_limit(fsdp_plan_t plan, int max_blocks);

/* Failure detection of the kernels that wait inside (the bulk-fed fused
 * reduce of a capped grid; no counterpart in the pages, whose collectives
 * report errors through HCCL). Each such wait gives up after `nanoseconds`
 * (default 1 s; 0 restores the default): the block then records why in
 * the plan's status word, stops, waits (bounded too) for its copies in
 * flight, and the kernel returns, so the CUDA context stays usable and the
 * outputs of that call are undefined. */
int fsdp_plan_set_wait_limit(fsdp_plan_t plan, uint64_t nanoseconds);

/* Reads the plan's status word after every call enqueued on `stream` so far
 * (synchronises the stream), stores it in *status and clears it. 0: no
 * wait ran out; otherwise FSDP_STATUS_PRODUCER_WAIT (a stage of the ring was
 * not released in time), FSDP_STATUS_CONSUMER_WAIT (a stage's data did not
 * arrive in time) and/or FSDP_STATUS_ORDER (a folding warp found the record
 * of another chunk than the one it waited for and stopped before storing:
 * an internal error). Returns FSDP_ERR_CUDA if the copy fails. */
#define FSDP_STATUS_PRODUCER_WAIT 1
#define FSDP_STATUS_CONSUMER_WAIT 2
#define FSDP_STATUS_ORDER 4
int fsdp_plan_status(fsdp_plan_t plan, fsdp_stream_t stream, int* status);

/* Test hook of that failure detection: with on != 0, every later bulk-fed
 * reduce of this plan withholds the first chunk of its first block, so the
 * waits for it run out after the wait limit and set the status word (the
 * call's outputs are then undefined). No fault, trap or endless wait is
 * involved. 0 switches it off. */
int fsdp_plan_inject_stall(fsdp_plan_t plan, int on);

/* Diagnostic, with no counterpart in the pages: builds the plan's work
 * tables on the host, as fsdp_plan_upload does, and checks every run
 * against the buffers its kernel touches, at the sizes fsdp_bind requires:
 * each run reads and writes inside those buffers, the runs of every
 * destination (a slice row, a full parameter, an actual shard) cover it
 * exactly once, and each run's tile count matches the prefix the kernels
 * search. Needs no GPU and changes nothing. Returns FSDP_OK, or
 * FSDP_ERR_INVALID_ARG with the first violation in fsdp_last_error(). */
int fsdp_plan_check_tables(fsdp_plan_t plan);

/* Mesh sizes and the unpadded total sum_p chunk_p * inner_p. Any output
 * pointer may be NULL. */
int fsdp_plan_info(fsdp_plan_t plan, int* rank_size, int* shard_size, int* dp_size,
                   int* n_params, int64_t* sum_padded);

/* Elements of one per-rank slice for dtype dt: sum_padded rounded up to a
 * multiple of 512 bytes [OVERLAP PR #758 §二.1]. */
int fsdp_slice_numel(fsdp_plan_t plan, int dt, int64_t* out);

/* "sharded_size" of parameter p on shard rank s [RAGGED §6.4]: the first
 * row and the number of rows it holds (possibly 0). */
int fsdp_sharded_size(fsdp_plan_t plan, int p, int shard_rank, int64_t* offset_rows,
                      int64_t* length_rows);

/* "padded_sharded_param_size" of parameter p: chunk_p = ceil(d0_p / S)
 * rows [RAGGED §6.4]; its numel is chunk_p * inner_p. */
int fsdp_padded_sharded_param_size(fsdp_plan_t plan, int p, int64_t* chunk_rows);

/* Element offsets o_0 .. o_P of the parameters inside a slice (n_params+1
 * values; o_P = sum_padded). */
int fsdp_offsets(fsdp_plan_t plan, int64_t* offsets);

/* Rank lists of rank w: shard_group[S] (ReduceScatter/AllGather group) and
 * replicate_group[D] (AllReduce group) [FS-RFC §2.2.1]. Either may be NULL. */
int fsdp_group_ranks(fsdp_plan_t plan, int w, int* shard_group, int* replicate_group);

/* Collectives the gradient sync issues [FS-RFC §2.2.2]: *rs_group_size = S
 * if a ReduceScatter over the shard group is issued (S > 1), else 0;
 * *ar_group_size = D if an AllReduce over the replicate group is issued
 * (D > 1), else 0. */
int fsdp_comm_calls(fsdp_plan_t plan, int* rs_group_size, int* ar_group_size);

/* ------------------------------------------------------------- bindings */

/* Uploads a pointer table for `role` (see enum fsdp_role) with element type
 * dt to the plan's device. dev_ptrs: host array of W*P or W device pointers.
 * numels: optional host array (same length) of the buffers' element counts,
 * checked against the role's requirement; NULL skips the check and makes
 * the caller responsible for the sizes. Pointers are checked for element
 * alignment. The plan must be uploaded. *out receives a handle owned by the
 * caller; the pointed-to buffers stay owned by the caller. */
int fsdp_bind(fsdp_plan_t plan, int role, int dt, const void* const* dev_ptrs,
              const int64_t* numels, fsdp_binding_t* out);

/* Frees a binding's device table (same caveat as fsdp_plan_destroy). */
int fsdp_binding_destroy(fsdp_binding_t binding);

/* --------------------------------------------------- forward (unshard) */

/* All-gather copy-in [OVERLAP PR #758 §二.1, §四.1; RAGGED §6.4]: rank w =
 * (d, s) packs its shards (SHARDS, dtype F32 or BF16) into ITS OWN slice of
 * its all-gather buffer (AG_OUTPUT, elements [s*slice, (s+1)*slice)), cast
 * F32->F32, F32->BF16 (round to nearest even) or BF16->BF16; padding rows
 * and the slice tail become 0. With fuse_gather != 0 the same slice is also
 * written into every shard-group member's buffer at the same place, so the
 * AllGather needs no separate pass. */
int fsdp_ag_copy_in(fsdp_plan_t plan, fsdp_binding_t shards, fsdp_binding_t ag_out,
                    int fuse_gather, fsdp_stream_t stream);

/* The AllGather over each shard group [OVERLAP §四.1]: copies slice s of
 * rank (d, s) into slice s of every other member (d, s'). */
int fsdp_ag_gather(fsdp_plan_t plan, fsdp_binding_t ag_out, fsdp_stream_t stream);

/* All-gather copy-out [OVERLAP PR #758 §二.1; RAGGED §6.4]: unpacks each
 * rank's gathered buffer into its full parameters (FULL_PARAMS, same dtype):
 * row r of parameter p comes from slice r / chunk_p, local row
 * r % chunk_p; padding rows are dropped. */
int fsdp_ag_copy_out(fsdp_plan_t plan, fsdp_binding_t ag_out, fsdp_binding_t full_params,
                     fsdp_stream_t stream);

/* Direct unshard, all three forward steps in one pass without the gathered
 * buffer (the follow-up "option 2" of [OVERLAP PR #758 §四, on ag_output]:
 * unsharded parameters filled straight from the shards): rank (d, s)'s
 * full parameter p gets, at rows [off_{p,s'}, off_{p,s'} + len_{p,s'}),
 * shard s' of p held by shard-group member (d, s'), cast as in
 * fsdp_ag_copy_in. The result equals fsdp_ag_copy_in + fsdp_ag_gather +
 * fsdp_ag_copy_out bit for bit; no AG_OUTPUT buffer is needed. */
int fsdp_ag_unshard(fsdp_plan_t plan, fsdp_binding_t shards, fsdp_binding_t full_params,
                    fsdp_stream_t stream);

/* ------------------------------------------------- backward (grad sync) */

/* Reduce-scatter copy-in [RAGGED §6.4; OVERLAP PR #758 §二.1]: row s' of
 * rank w's RS input (RS_INPUT, same dtype as GRADS) holds rows
 * [off_{p,s'}, off+len) of every gradient p at o_p, zeros to the padded
 * size and in the slice tail. Used by the unfused path. */
int fsdp_rs_copy_in(fsdp_plan_t plan, fsdp_binding_t grads, fsdp_binding_t rs_in,
                    fsdp_stream_t stream);

/* Fused gradient sync: reduce-scatter copy-in + ReduceScatter (SUM over the
 * shard group) + AllReduce (SUM over the replicate group) into the fused
 * fp32 regions, in one pass that reads every unpadded gradient once
 * [OVERLAP PR #758 §二.1 AllReduceParamGroup zero-copy fused buffer, §二.3
 * fused AllReduce uses SUM]. For rank (d, s) and element j < slice(F32):
 * fused_{d,s}[j] = sum_{d'} sum_{s''} grads_{(d',s''),p}[off_{p,s}*inner_p +
 * j - o_p] when j lies in the actual rows of parameter p's region, +0
 * otherwise. GRADS: F32 or BF16; FUSED: F32. No scaling happens here. */
int fsdp_rs_ar_reduce(fsdp_plan_t plan, fsdp_binding_t grads, fsdp_binding_t fused,
                      fsdp_stream_t stream);

/* Applies synced gradients [OVERLAP PR #758 §二.3 wait_and_apply_grads;
 * RAGGED §6.4 back-fill by sharded_size]: for rank (d, s) and parameter p,
 * shard_grads[k] = round(fused[o_p + k] / div) for k < len_{p,s}*inner_p,
 * div = W for FSDP_AVG (the fused buffer holds the SUM over all W ranks),
 * 1 for FSDP_SUM. With accumulate != 0 the result is added, in fp32, to the
 * gradient already in shard_grads and rounded once (grad accumulation,
 * [FS-RFC §5.2 item 9]). SHARD_GRADS: F32 or BF16. Zero-length shards are
 * not touched. */
int fsdp_apply_grads(fsdp_plan_t plan, fsdp_binding_t fused, int op, int accumulate,
                     fsdp_binding_t shard_grads, fsdp_stream_t stream);

/* Unfused path, ReduceScatter half [OVERLAP PR #758 §二.3-§二.4]: for rank
 * (d, s), fused[j] = sum_{s''} rs_in_{(d,s'')}[s*slice(dt_in) + j] for
 * j < slice(F32), divided by S for FSDP_AVG. */
int fsdp_rs_reduce(fsdp_plan_t plan, fsdp_binding_t rs_in, int op, fsdp_binding_t fused,
                   fsdp_stream_t stream);

/* Unfused path, AllReduce half, in place over each replicate group
 * [OVERLAP PR #758 §二.4 fix 1: the replicate-dim AllReduce is scaled by
 * replicate_world_size]: fused_{(d,s)}[j] = sum_{d'} fused_{(d',s)}[j] for
 * every d, divided by D for FSDP_AVG. With power-of-two S and D, rs_reduce
 * (AVG) + ar_reduce (AVG) + apply_grads (SUM) equals rs_ar_reduce +
 * apply_grads (AVG) bit for bit. */
int fsdp_ar_reduce(fsdp_plan_t plan, fsdp_binding_t fused, int op, fsdp_stream_t stream);

/* fsdp_rs_ar_reduce followed by fsdp_apply_grads, in one pass: the fused
 * regions get exactly the bits fsdp_rs_ar_reduce writes (the raw SUM) and
 * the actual-shard gradients exactly the bits fsdp_apply_grads would write
 * from them (op, accumulate as there), without reading the fused regions
 * back: the apply's divide, back-fill of the actual rows and rounding
 * ([OVERLAP] PR #758 §二.3, [RAGGED] §6.4) happen where the sum is formed.
 * No counterpart as one call in the pages (which apply after the fused
 * AllReduce). shard_grads must have the gradient dtype. One kernel when the
 * staged reduce fits the mesh (up to 32 bf16 or ~26 fp32 sources);
 * otherwise the two calls it stands for, in order on `stream`. When most of
 * the plan's gradient runs are shifted against the fused rows' 16-byte grid
 * (a ragged layout) and no grid cap is set, the kernel is the TMA-bulk-fed
 * one on every SM (as under a cap; its waits report through
 * fsdp_plan_status). */
int fsdp_rs_ar_reduce_apply(fsdp_plan_t plan, fsdp_binding_t grads, fsdp_binding_t fused, int op,
                            int accumulate, fsdp_binding_t shard_grads, fsdp_stream_t stream);

/* ------------------------------------------------ allocation-free call */

/* Size of the fixed device work area of fsdp_rs_ar_reduce_noalloc. */
#define FSDP_NOALLOC_SCRATCH_BYTES (1 << 20)

/* The fused gradient sync of fsdp_rs_ar_reduce, computing the same bits,
 * for callers that cannot allocate device memory. The pages have no
 * counterpart: it exists for this library's users. Who needs it: a caller
 * whose device memory is owned wholly by its own allocator (a training
 * framework's caching allocator, whose accounting and fragmentation control
 * break if a library allocates on the side), or a job so close to the
 * device's memory limit that an allocation in the middle of a step could
 * fail. fsdp_plan_upload and fsdp_bind allocate; this call does not.
 *
 * plan: from fsdp_plan_create; it need not be uploaded. grad_dtype:
 * FSDP_F32 or FSDP_BF16. grads: HOST array of W*P device pointers (index
 * w*P + p) to the unsharded gradients, d0_p * inner_p elements each,
 * element aligned. fused: HOST array of W device pointers to fp32 fused
 * regions of fsdp_slice_numel(plan, FSDP_F32) elements, 4-byte aligned.
 * Both arrays are read before the call returns.
 *
 * The work tables (the runs of the fused region and the two pointer tables)
 * go to one device array of FSDP_NOALLOC_SCRATCH_BYTES that is part of the
 * library image: every GPU that loads the library holds it until the
 * process exits. The tables take about 40 bytes per run of the fused
 * region (at most S * (2P + 1) runs) plus 8 bytes per buffer pointer
 * (W * (P + 1)); a plan that needs more than FSDP_NOALLOC_SCRATCH_BYTES is
 * refused with FSDP_ERR_INVALID_ARG and a message saying how many bytes it
 * needs (use fsdp_rs_ar_reduce for it). The first call on a device
 * looks up the array's device address (with that device current); make
 * that first call before any stream capture. Every call copies its tables
 * into the array on `stream` ahead of the kernel and rewrites everything it
 * reads, so nothing in the array needs to start at zero; the array is
 * shared by all calls, so calls that overlap on the GPU (different streams,
 * no ordering between them) race on it and must not be issued. The tables
 * are staged through one host buffer that the next call overwrites, so a
 * call while `stream` is being captured is refused (FSDP_ERR_INVALID_ARG).
 * A grid cap set with fsdp_plan_set_grid_limit applies here too. Host calls
 * are serialised by a lock. The caller sizes both pointer arrays (W*P and
 * W entries) and the buffers they point to; the library cannot check a
 * buffer's size here. Returns as fsdp_rs_ar_reduce does. */
int fsdp_rs_ar_reduce_noalloc(fsdp_plan_t plan, int grad_dtype, const void* const* grads,
                              float* const* fused, fsdp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HSDP_FSDP_H */
