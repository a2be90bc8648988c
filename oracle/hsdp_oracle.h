/*
 * hsdp_oracle.h -- interface of the CPU oracle (test infrastructure only).
 * The product library has its own header and shares nothing with this one.
 * All pointers are host pointers. dtype codes: HOR_F32 = 0, HOR_BF16 = 1
 * (bf16 stored as its 16 raw bits). Reduce ops: HOR_AVG = 0, HOR_SUM = 1.
 */
#ifndef HSDP_ORACLE_H
#define HSDP_ORACLE_H

#include <stdint.h>

enum { HOR_OK = 0, HOR_EINVAL = 1, HOR_ENOTIMPL = 2, HOR_ENOMEM = 3 };
enum { HOR_F32 = 0, HOR_BF16 = 1 };
enum { HOR_AVG = 0, HOR_SUM = 1 };

typedef struct {
    int P, W, S, D;
    const int64_t* d0;    /* [P] dim-0 length of each parameter */
    const int64_t* inner; /* [P] product of the other dims (1 for a vector) */
    const int64_t* dss;   /* [P] padded shard rows = ceil(d0 / S) */
    const int64_t* off;   /* [P*S] first row of shard s of param p (p*S + s) */
    const int64_t* len;   /* [P*S] rows held by shard s of param p */
    const int64_t* o;     /* [P+1] element offset of param p inside a slice; o[P] = end */
} hor_layout;

float hor_bf16_to_f32(uint16_t h);
uint16_t hor_f32_to_bf16(float x);

int hor_effective_shard_size(int shard_size, int enable_param_shard);
int hor_plan(int P, const int64_t* d0, const int64_t* inner, int rank_size,
             int shard_size, int enable_param_shard, int shard_dim,
             int64_t* dss, int64_t* off, int64_t* len, int64_t* o);
int hor_plan_bucketed(int P, const int64_t* d0, const int64_t* inner, const int* bucket,
                      int rank_size, int shard_size, int enable_param_shard, int shard_dim,
                      int64_t* dss, int64_t* off, int64_t* len, int64_t* o);
int64_t hor_slice_numel(int64_t sum_padded, int dt);
void hor_group_ranks(int W, int S, int w, int* shard_group, int* replicate_group);
void hor_comm_calls(int S, int D, int* rs_group_size, int* ar_group_size);

int hor_ag_copy_in(const hor_layout* L, int src_dt, const void* const* shards,
                   int dst_dt, int64_t slice, void* const* ag_out);
int hor_ag_gather(const hor_layout* L, int dt, int64_t slice, void* const* ag_out);
int hor_ag_copy_out(const hor_layout* L, int dt, int64_t slice,
                    const void* const* ag_out, void* const* full);
int hor_rs_copy_in(const hor_layout* L, int dt, int64_t slice,
                   const void* const* grads, void* const* rs_in);
float hor_fold_nested(int S, int D, const float* vals);
int hor_rs_ar_reduce(const hor_layout* L, int dt, int64_t slice_g,
                     const void* const* rs_in, int64_t slice_f32, float* const* fused);
int hor_rs_reduce(const hor_layout* L, int dt, int64_t slice_g, const void* const* rs_in,
                  int op, int64_t slice_f32, float* const* out);
int hor_ar_reduce(const hor_layout* L, int op, int64_t slice_f32, float* const* buf);
int hor_apply_grads(const hor_layout* L, const float* const* fused, int op, int dt,
                    int accumulate, void* const* shard_grads);

int hor_locate_fused(const hor_layout* L, int s, int64_t j, int64_t* e);
int64_t hor_locate_gathered(const hor_layout* L, int64_t slice, int p, int64_t e,
                            int* shard, int64_t* k);
void hor_locate_fused_many(const hor_layout* L, int64_t n, const int* s, const int64_t* j,
                           int* p, int64_t* e);
void hor_locate_gathered_many(const hor_layout* L, int64_t slice, int64_t n, const int* p,
                              const int64_t* e, int* shard, int64_t* k, int64_t* idx);
void hor_fold_nested_many(int S, int D, int64_t n, const float* vals, float* out);
void hor_f32_to_bf16_many(int64_t n, const float* x, uint16_t* out);
void hor_div_many(int64_t n, const float* x, float div, float* out);

#endif
