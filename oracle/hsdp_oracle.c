/*
 * hsdp_oracle.c -- plain, slow, single-threaded CPU oracle of the HSDP
 * fully_shard parameter / gradient data path with dim-0 ragged shards.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * calls it and shares no code, header, table or helper with it.
 *
 * Every function is the plain definition of one step written as loops over
 * (rank, param, shard, element), in the order the pages describe the step.
 * Sources, cited as page title + section:
 *   [FS-RFC]  "【RFC】FullyShard 多维并行适配设计方案" (hyper-parallel issue 1)
 *   [OVERLAP] "Hyper通信掩盖方案" (hyper-parallel issue 184) and the PR #758
 *             write-up under it ("方案落地说明")
 *   [RAGGED]  FSDP dim-0 uneven-sharding RFC (hyper-parallel issue 319)
 *
 * Readings taken where the pages are silent:
 *   - rank w of the W = rank_size ranks sits at mesh coordinate
 *     (d, s) = (w / S, w % S): replicate index outer, shard rank inner;
 *   - the fused buffer holds the raw SUM over all W ranks; AVG divides once
 *     by W when gradients are applied;
 *   - sums are IEEE binary32 round-to-nearest-even additions folded in
 *     ascending order from the first term: inner fold over the shard group,
 *     outer fold over the replicas;
 *   - every per-rank slice is rounded up to 512 bytes; parameters inside it
 *     are packed back to back at their padded sizes;
 *   - float -> bf16 is round-to-nearest-even; a NaN becomes the quiet NaN
 *     0x7FC0 with its sign kept.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (no FMA
 * contraction, no flush-to-zero), so every float operation below is one
 * IEEE binary32 operation.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "hsdp_oracle.h"

/* ------------------------------------------------------------------ */
/* Scalar conversions                                                  */
/* ------------------------------------------------------------------ */

float hor_bf16_to_f32(uint16_t h)
{
    /* bf16 is the upper half of a binary32: widening is exact. */
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t hor_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) {
        /* NaN: quiet NaN, sign kept (reading; the pages fix no NaN rule). */
        return (uint16_t)((sign >> 16) | 0x7FC0u);
    }
    /* Sign-magnitude: the bf16 candidates bracketing |x| are the magnitude
     * truncated to its upper 16 bits and the next magnitude up. The 16
     * discarded bits say how far |x| lies above the lower candidate, in
     * units of 2^-16 of the candidates' spacing. Round to nearest; on an
     * exact tie pick the candidate whose last bit is 0. Incrementing the
     * magnitude carries into the exponent correctly, up to infinity. */
    uint32_t upper = mag >> 16;
    uint32_t rest = mag & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)((sign >> 16) | upper);
}

static int elem_bytes(int dt)
{
    return dt == HOR_F32 ? 4 : (dt == HOR_BF16 ? 2 : 0);
}

static float load_as_f32(const void* base, int dt, int64_t i)
{
    if (dt == HOR_F32)
        return ((const float*)base)[i];
    return hor_bf16_to_f32(((const uint16_t*)base)[i]);
}

static void store_from_f32(void* base, int dt, int64_t i, float v)
{
    if (dt == HOR_F32)
        ((float*)base)[i] = v;
    else
        ((uint16_t*)base)[i] = hor_f32_to_bf16(v);
}

/* One element moved from src[si] (type sdt) to dst[di] (type ddt): the same
 * type is a bit copy; f32 -> bf16 rounds to nearest even; bf16 -> f32 widens. */
static void move_elem(void* dst, int ddt, int64_t di, const void* src, int sdt, int64_t si)
{
    if (sdt == ddt) {
        int es = elem_bytes(sdt);
        memcpy((char*)dst + di * es, (const char*)src + si * es, (size_t)es);
    } else {
        store_from_f32(dst, ddt, di, load_as_f32(src, sdt, si));
    }
}

static void zero_elems(void* dst, int dt, int64_t first, int64_t count)
{
    int es = elem_bytes(dt);
    if (count > 0)
        memset((char*)dst + first * es, 0, (size_t)(count * es));
}

/* ------------------------------------------------------------------ */
/* Planning                                                            */
/* ------------------------------------------------------------------ */

int hor_effective_shard_size(int shard_size, int enable_param_shard)
{
    /* [FS-RFC] §2.2.3 option A / §4.1: enable_param_shard=False switches
     * parameter sharding off; §2.2.5 item 3: shard_size is then fixed at 1. */
    return enable_param_shard ? shard_size : 1;
}

int hor_plan(int P, const int64_t* d0, const int64_t* inner, int rank_size,
             int shard_size, int enable_param_shard, int shard_dim,
             int64_t* dss, int64_t* off, int64_t* len, int64_t* o)
{
    return hor_plan_bucketed(P, d0, inner, NULL, rank_size, shard_size, enable_param_shard,
                             shard_dim, dss, off, len, o);
}

int hor_plan_bucketed(int P, const int64_t* d0, const int64_t* inner, const int* bucket,
                      int rank_size, int shard_size, int enable_param_shard, int shard_dim,
                      int64_t* dss, int64_t* off, int64_t* len, int64_t* o)
{
    if (P < 0 || rank_size < 1 || (P > 0 && (!d0 || !inner)))
        return HOR_EINVAL;
    int S = hor_effective_shard_size(shard_size, enable_param_shard);
    /* [FS-RFC] §2.2.5: dp_size = rank_size // shard_size; the shard group
     * must tile the rank domain. */
    if (S < 1 || rank_size % S != 0)
        return HOR_EINVAL;
    /* [RAGGED] §3.2 non-goal 1 / §5.1: only dim 0 may be sharded unevenly;
     * this layout describes dim 0 only. */
    if (shard_dim != 0)
        return HOR_ENOTIMPL;
    int64_t end = 0; /* end of the previous parameter's padded region */
    for (int p = 0; p < P; ++p) {
        if (d0[p] < 0 || inner[p] < 1)
            return HOR_EINVAL;
        /* [OVERLAP] PR #758 write-up §二.1 (AllReduceParamGroup): several
         * buckets share one fused buffer. Reading: bucket ids rise with the
         * registration order and a new bucket starts at the next multiple of
         * 256 elements, a 512-byte boundary in bf16 and in fp32 alike. */
        if (bucket && (bucket[p] < 0 || (p > 0 && bucket[p] < bucket[p - 1])))
            return HOR_EINVAL;
        if (bucket && p > 0 && bucket[p] != bucket[p - 1])
            end = (end + 255) / 256 * 256;
        o[p] = end;
        /* [RAGGED] §6.4: fixed-size chunks of ceil(dim0 / S) rows; shard s
         * starts at min(s * chunk, dim0) and holds min(chunk, dim0 - start)
         * rows, which may be 0. */
        int64_t chunk = (d0[p] + S - 1) / S;
        dss[p] = chunk;
        for (int s = 0; s < S; ++s) {
            int64_t start = (int64_t)s * chunk;
            if (start > d0[p])
                start = d0[p];
            int64_t rows = d0[p] - start;
            if (rows > chunk)
                rows = chunk;
            off[(int64_t)p * S + s] = start;
            len[(int64_t)p * S + s] = rows;
        }
        /* [RAGGED] §6.4 "AllGather 和 ReduceScatter": the offset inside the
         * fused buffer advances by padded_sharded_param_size.numel(). */
        end = o[p] + chunk * inner[p];
    }
    o[P] = end;
    return HOR_OK;
}

int64_t hor_slice_numel(int64_t sum_padded, int dt)
{
    /* [OVERLAP] PR #758 write-up §二.1: the fused buffer is 512-byte aligned;
     * every per-rank slice is rounded up to a whole number of 512 bytes. */
    int64_t per = 512 / elem_bytes(dt);
    return (sum_padded + per - 1) / per * per;
}

void hor_group_ranks(int W, int S, int w, int* shard_group, int* replicate_group)
{
    /* [FS-RFC] §2.2.1: each rank has a shard group (the ReduceScatter group)
     * and a replicate group (the AllReduce group). Reading: w = d*S + s. */
    int D = W / S, d = w / S, s = w % S;
    for (int k = 0; k < S; ++k)
        shard_group[k] = d * S + k;
    for (int k = 0; k < D; ++k)
        replicate_group[k] = k * S + s;
}

void hor_comm_calls(int S, int D, int* rs_group_size, int* ar_group_size)
{
    /* [FS-RFC] §2.2.2 decision matrix: ReduceScatter over the shard group
     * when shard_size > 1; AllReduce over the replicate group when
     * dp_size > 1; neither keeps the local gradient. 0 = not issued. */
    *rs_group_size = S > 1 ? S : 0;
    *ar_group_size = D > 1 ? D : 0;
}

/* ------------------------------------------------------------------ */
/* Forward: all-gather copy-in, the all-gather itself, copy-out        */
/* ------------------------------------------------------------------ */

int hor_ag_copy_in(const hor_layout* L, int src_dt, const void* const* shards,
                   int dst_dt, int64_t slice, void* const* ag_out)
{
    /* [OVERLAP] PR #758 write-up §二.1 and §四.1: each rank packs its local
     * shards, cast to the all-gather dtype, into ITS OWN slice of ag_output
     * (send = ag_output.narrow(rank * input_numel, input_numel)).
     * [RAGGED] §6.4: each parameter occupies padded_sharded_param_size
     * elements; the rows past the actual shard are zero. The slice tail past
     * the last parameter is zero too. Other ranks' slices are not touched. */
    int P = L->P, S = L->S;
    if (elem_bytes(src_dt) == 0 || elem_bytes(dst_dt) == 0)
        return HOR_EINVAL;
    if (src_dt == HOR_BF16 && dst_dt == HOR_F32)
        return HOR_EINVAL; /* the cast narrows or keeps, never widens */
#pragma omp parallel for schedule(dynamic)
    for (int w = 0; w < L->W; ++w) {
        int s = w % S;
        int64_t base = (int64_t)s * slice;
        zero_elems(ag_out[w], dst_dt, base, slice);
        for (int p = 0; p < P; ++p) {
            int64_t n = L->len[(int64_t)p * S + s] * L->inner[p];
            for (int64_t k = 0; k < n; ++k)
                move_elem(ag_out[w], dst_dt, base + L->o[p] + k,
                          shards[(int64_t)w * P + p], src_dt, k);
        }
    }
    return HOR_OK;
}

int hor_ag_gather(const hor_layout* L, int dt, int64_t slice, void* const* ag_out)
{
    /* [OVERLAP] §四.1: AllGather within the shard group; afterwards every
     * member holds every member's slice, slice s' at offset s' * slice. */
    int S = L->S, es = elem_bytes(dt);
    if (es == 0)
        return HOR_EINVAL;
#pragma omp parallel for schedule(dynamic)
    for (int w = 0; w < L->W; ++w) {
        int d = w / S;
        for (int sp = 0; sp < S; ++sp) {
            int src = d * S + sp;
            if (src == w)
                continue;
            memcpy((char*)ag_out[w] + (int64_t)sp * slice * es,
                   (const char*)ag_out[src] + (int64_t)sp * slice * es,
                   (size_t)(slice * es));
        }
    }
    return HOR_OK;
}

int hor_ag_copy_out(const hor_layout* L, int dt, int64_t slice,
                    const void* const* ag_out, void* const* full)
{
    /* [OVERLAP] §二.1 (foreach copy-out) and [RAGGED] §6.4: the gathered
     * buffer is unpacked into each parameter's full tensor; only the logical
     * (dim0, ...) shape is exposed, padding rows are dropped. Row r of
     * parameter p comes from shard r / dss, local row r % dss. */
    int P = L->P;
    if (elem_bytes(dt) == 0)
        return HOR_EINVAL;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int w = 0; w < L->W; ++w) {
        for (int p = 0; p < P; ++p) {
            int64_t dss = L->dss[p], in = L->inner[p];
            for (int64_t r = 0; r < L->d0[p]; ++r)
                for (int64_t c = 0; c < in; ++c)
                    move_elem(full[(int64_t)w * P + p], dt, r * in + c, ag_out[w], dt,
                              (r / dss) * slice + L->o[p] + (r % dss) * in + c);
        }
    }
    return HOR_OK;
}

/* ------------------------------------------------------------------ */
/* Backward: reduce-scatter copy-in, the reductions, applying grads    */
/* ------------------------------------------------------------------ */

int hor_rs_copy_in(const hor_layout* L, int dt, int64_t slice,
                   const void* const* grads, void* const* rs_in)
{
    /* [RAGGED] §6.4: the reduce-scatter input of each rank is S rows, one per
     * destination shard; row s' holds, for every parameter at offset o_p, the
     * rows [off, off + len) of its gradient followed by zeros up to the
     * padded size. [OVERLAP] §二.1: one packed buffer per rank. */
    int P = L->P, S = L->S;
    if (elem_bytes(dt) == 0)
        return HOR_EINVAL;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int w = 0; w < L->W; ++w) {
        for (int sp = 0; sp < S; ++sp) {
            int64_t row = (int64_t)sp * slice;
            zero_elems(rs_in[w], dt, row, slice);
            for (int p = 0; p < P; ++p) {
                int64_t in = L->inner[p];
                int64_t first = L->off[(int64_t)p * S + sp];
                for (int64_t i = 0; i < L->len[(int64_t)p * S + sp]; ++i)
                    for (int64_t c = 0; c < in; ++c)
                        move_elem(rs_in[w], dt, row + L->o[p] + i * in + c,
                                  grads[(int64_t)w * P + p], dt, (first + i) * in + c);
            }
        }
    }
    return HOR_OK;
}

float hor_fold_nested(int S, int D, const float* vals)
{
    /* ReduceScatter over the shard group, then AllReduce over the replicate
     * group ([FS-RFC] §2.1.3 item 3, §3.3): part_d = sum over s of
     * vals[d*S + s], total = sum over d of part_d, each a left fold in
     * ascending order that starts from its first term. */
    float total = 0.0f;
    for (int d = 0; d < D; ++d) {
        float part = vals[d * S];
        for (int s = 1; s < S; ++s)
            part = part + vals[d * S + s];
        total = d == 0 ? part : total + part;
    }
    return total;
}

int hor_rs_ar_reduce(const hor_layout* L, int dt, int64_t slice_g,
                     const void* const* rs_in, int64_t slice_f32, float* const* fused)
{
    /* [OVERLAP] PR #758 write-up §二.1 and §二.3: the ReduceScatter outputs
     * land in views of one contiguous fused buffer which is then all-reduced
     * with SUM. Result for rank (d, s), element j: the nested fold of element
     * j of row s of every rank's reduce-scatter input. */
    int S = L->S, D = L->D, W = L->W;
    if (elem_bytes(dt) == 0 || slice_g < slice_f32)
        return HOR_EINVAL;
    /* one scratch row of W values per rank */
    float* vals_all = (float*)malloc(sizeof(float) * (size_t)(W > 0 ? W * W : 1));
    if (!vals_all)
        return HOR_ENOMEM;
#pragma omp parallel for schedule(dynamic)
    for (int w = 0; w < W; ++w) {
        int s = w % S;
        float* vals = vals_all + (int64_t)w * W;
        for (int64_t j = 0; j < slice_f32; ++j) {
            for (int v = 0; v < W; ++v)
                vals[v] = load_as_f32(rs_in[v], dt, (int64_t)s * slice_g + j);
            fused[w][j] = hor_fold_nested(S, D, vals);
        }
    }
    free(vals_all);
    return HOR_OK;
}

int hor_rs_reduce(const hor_layout* L, int dt, int64_t slice_g, const void* const* rs_in,
                  int op, int64_t slice_f32, float* const* out)
{
    /* Unfused path, ReduceScatter half ([OVERLAP] §二.3, §二.4): the native
     * collective sums row s over the shard group; AVG divides by S. */
    int S = L->S;
    if (elem_bytes(dt) == 0 || slice_g < slice_f32)
        return HOR_EINVAL;
#pragma omp parallel for schedule(dynamic)
    for (int w = 0; w < L->W; ++w) {
        int d = w / S, s = w % S;
        for (int64_t j = 0; j < slice_f32; ++j) {
            float part = load_as_f32(rs_in[d * S], dt, (int64_t)s * slice_g + j);
            for (int sp = 1; sp < S; ++sp)
                part = part + load_as_f32(rs_in[d * S + sp], dt, (int64_t)s * slice_g + j);
            out[w][j] = op == HOR_AVG ? part / (float)S : part;
        }
    }
    return HOR_OK;
}

int hor_ar_reduce(const hor_layout* L, int op, int64_t slice_f32, float* const* buf)
{
    /* Unfused path, AllReduce half ([OVERLAP] §二.4 fix 1): the replicate-dim
     * all-reduce is scaled by replicate_world_size = D for AVG. In place:
     * every member of the replicate group gets the same result. */
    int S = L->S, D = L->D;
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        for (int64_t j = 0; j < slice_f32; ++j) {
            float total = buf[s][j];
            for (int d = 1; d < D; ++d)
                total = total + buf[d * S + s][j];
            if (op == HOR_AVG)
                total = total / (float)D;
            for (int d = 0; d < D; ++d)
                buf[d * S + s][j] = total;
        }
    }
    return HOR_OK;
}

int hor_apply_grads(const hor_layout* L, const float* const* fused, int op, int dt,
                    int accumulate, void* const* shard_grads)
{
    /* [OVERLAP] §二.3: the fused all-reduce sums and wait_and_apply_grads
     * divides afterwards (reading: once, by W, for AVG; SUM divides by 1).
     * [RAGGED] §6.4: only sharded_size rows go back; the optimizer never sees
     * padding. A zero-length shard writes nothing. [FS-RFC] §5.2 item 9
     * (requires_grad_sync): accumulate adds the new value to the gradient
     * already held, in fp32, and rounds once. */
    int P = L->P, S = L->S;
    if (elem_bytes(dt) == 0)
        return HOR_EINVAL;
    float div = op == HOR_AVG ? (float)L->W : 1.0f;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int w = 0; w < L->W; ++w) {
        for (int p = 0; p < P; ++p) {
            int s = w % S;
            int64_t n = L->len[(int64_t)p * S + s] * L->inner[p];
            void* g = shard_grads[(int64_t)w * P + p];
            for (int64_t k = 0; k < n; ++k) {
                float q = fused[w][L->o[p] + k] / div;
                if (accumulate)
                    q = load_as_f32(g, dt, k) + q;
                store_from_f32(g, dt, k, q);
            }
        }
    }
    return HOR_OK;
}

/* ------------------------------------------------------------------ */
/* Element locators for sampled checks on full-size problems           */
/* ------------------------------------------------------------------ */

int hor_locate_fused(const hor_layout* L, int s, int64_t j, int64_t* e)
{
    /* Which gradient element feeds fused element j of shard row s: find the
     * parameter whose padded region holds j, then the row inside shard s.
     * Returns the parameter index, or -1 when j is padding. */
    for (int p = 0; p < L->P; ++p) {
        if (j >= L->o[p] && j < L->o[p] + L->dss[p] * L->inner[p]) {
            int64_t rel = j - L->o[p];
            int64_t i = rel / L->inner[p], c = rel % L->inner[p];
            if (i >= L->len[(int64_t)p * L->S + s])
                return -1;
            *e = (L->off[(int64_t)p * L->S + s] + i) * L->inner[p] + c;
            return p;
        }
    }
    return -1;
}

int64_t hor_locate_gathered(const hor_layout* L, int64_t slice, int p, int64_t e,
                            int* shard, int64_t* k)
{
    /* Where element e of parameter p's full tensor sits after the
     * all-gather: shard r / dss (returned in *shard), element *k of that
     * shard, and the returned index inside the gathered buffer. */
    int64_t in = L->inner[p], r = e / in, c = e % in, dss = L->dss[p];
    *shard = (int)(r / dss);
    *k = (r % dss) * in + c;
    return (r / dss) * slice + L->o[p] + (r % dss) * in + c;
}

void hor_locate_fused_many(const hor_layout* L, int64_t n, const int* s, const int64_t* j,
                           int* p, int64_t* e)
{
    for (int64_t i = 0; i < n; ++i) {
        e[i] = -1;
        p[i] = hor_locate_fused(L, s[i], j[i], &e[i]);
    }
}

void hor_locate_gathered_many(const hor_layout* L, int64_t slice, int64_t n, const int* p,
                              const int64_t* e, int* shard, int64_t* k, int64_t* idx)
{
    for (int64_t i = 0; i < n; ++i)
        idx[i] = hor_locate_gathered(L, slice, p[i], e[i], &shard[i], &k[i]);
}

void hor_fold_nested_many(int S, int D, int64_t n, const float* vals, float* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = hor_fold_nested(S, D, vals + i * (int64_t)S * D);
}

void hor_f32_to_bf16_many(int64_t n, const float* x, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = hor_f32_to_bf16(x[i]);
}

void hor_div_many(int64_t n, const float* x, float div, float* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = x[i] / div;
}
