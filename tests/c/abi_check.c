/*
 * abi_check.c -- drives the C ABI (include/hsdp_fsdp.h) from plain C11 with
 * cudaMalloc'd buffers, no Python and no PyTorch: plan queries, the forward
 * unshard (gathered and direct), the fused gradient sync and apply, and an
 * error path. Values are small integers, exact in bf16, so every expected
 * result has a closed form:
 *   mesh rank_size 4, shard_size 2 (dp_size 2), params (5,3), (4,), (7,2);
 *   parameter p element e = 100p + e (every replica holds the same shards);
 *   gradient of rank w, parameter p, element e = (w+1) * (1 + e % 3),
 *   so the sum over ranks is 10 * (1 + e % 3) and AVG divides it by 4.
 * Exit status 0 when every check passes.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "hsdp_fsdp.h"

#define W 4
#define S 2
#define P 3

static const int64_t DIM0[P] = {5, 4, 7};
static const int64_t INNER[P] = {3, 1, 2};
static int failures = 0;

#define CHECK(cond, ...)                          \
    do {                                          \
        if (!(cond)) {                            \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);         \
            fprintf(stderr, "\n");                \
            ++failures;                           \
        }                                         \
    } while (0)

#define OK(call)                                                                      \
    do {                                                                              \
        int rc_ = (call);                                                             \
        if (rc_ != FSDP_OK) {                                                         \
            fprintf(stderr, "FAIL %s:%d: %s -> %d (%s)\n", __FILE__, __LINE__, #call, \
                    rc_, fsdp_last_error());                                          \
            exit(1);                                                                  \
        }                                                                             \
    } while (0)

#define CUDA(call)                                                                     \
    do {                                                                               \
        cudaError_t e_ = (call);                                                       \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "FAIL %s:%d: %s -> %s\n", __FILE__, __LINE__, #call,        \
                    cudaGetErrorString(e_));                                           \
            exit(1);                                                                   \
        }                                                                              \
    } while (0)

/* bf16 bits of a value that bf16 holds exactly (integers up to 256, halves) */
static uint16_t bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

static void* dev_alloc(size_t bytes) {
    void* p = NULL;
    CUDA(cudaMalloc(&p, bytes ? bytes : 16));
    CUDA(cudaMemset(p, 0xFF, bytes ? bytes : 16)); /* dirty: every output must be written */
    return p;
}

static int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

int main(void) {
    fsdp_plan_t plan = NULL;
    int64_t chunk[P], off[P][S], len[P][S], o[P + 1];
    int64_t sum_padded = 0, sl_bf16 = 0, sl_f32 = 0;

    /* uneven sharding of a dim other than 0 is refused with a message */
    int rc = fsdp_plan_create(P, DIM0, INNER, W, S, 1, 1, &plan);
    CHECK(rc == FSDP_ERR_NOT_IMPLEMENTED, "shard_dim 1 returned %d", rc);
    CHECK(strlen(fsdp_last_error()) > 0, "no message for the refused plan");

    /* plan queries against the closed forms */
    OK(fsdp_plan_create(P, DIM0, INNER, W, S, 1, 0, &plan));
    {
        int rs, ss, ds, np;
        int64_t expect = 0;
        OK(fsdp_plan_info(plan, &rs, &ss, &ds, &np, &sum_padded));
        CHECK(rs == W && ss == S && ds == W / S && np == P, "plan_info %d %d %d %d", rs, ss, ds, np);
        for (int p = 0; p < P; ++p) {
            int64_t c;
            chunk[p] = (DIM0[p] + S - 1) / S;
            OK(fsdp_padded_sharded_param_size(plan, p, &c));
            CHECK(c == chunk[p], "chunk of param %d: %lld", p, (long long)c);
            for (int s = 0; s < S; ++s) {
                int64_t ro, rl;
                off[p][s] = min64(s * chunk[p], DIM0[p]);
                len[p][s] = min64(chunk[p], DIM0[p] - off[p][s]);
                OK(fsdp_sharded_size(plan, p, s, &ro, &rl));
                CHECK(ro == off[p][s] && rl == len[p][s], "sharded_size(%d, %d) = (%lld, %lld)", p, s,
                      (long long)ro, (long long)rl);
            }
            expect += chunk[p] * INNER[p];
        }
        CHECK(sum_padded == expect, "sum_padded %lld", (long long)sum_padded);
        OK(fsdp_offsets(plan, o));
        for (int p = 0, acc = 0; p <= P; ++p) {
            CHECK(o[p] == acc, "o[%d] = %lld", p, (long long)o[p]);
            if (p < P) acc += (int)(chunk[p] * INNER[p]);
        }
        OK(fsdp_slice_numel(plan, FSDP_BF16, &sl_bf16));
        OK(fsdp_slice_numel(plan, FSDP_F32, &sl_f32));
        CHECK(sl_bf16 == (sum_padded + 255) / 256 * 256, "bf16 slice %lld", (long long)sl_bf16);
        CHECK(sl_f32 == (sum_padded + 127) / 128 * 128, "f32 slice %lld", (long long)sl_f32);
        for (int w = 0; w < W; ++w) {
            int sg[S], rg[W / S];
            OK(fsdp_group_ranks(plan, w, sg, rg));
            for (int k = 0; k < S; ++k) CHECK(sg[k] == (w / S) * S + k, "shard group of %d", w);
            for (int k = 0; k < W / S; ++k) CHECK(rg[k] == k * S + w % S, "replicate group of %d", w);
        }
        OK(fsdp_comm_calls(plan, &rs, &ds));
        CHECK(rs == S && ds == W / S, "comm calls %d %d", rs, ds);
    }
    OK(fsdp_plan_upload(plan));

    /* buffers: caller-owned device memory, one allocation per (rank, param) */
    void *shards[W * P], *full[W * P], *full2[W * P], *grads[W * P], *sgrad[W * P];
    void *ag[W], *fused[W];
    int64_t n_shard[W * P], n_full[W * P], n_ag[W], n_fused[W];
    for (int w = 0; w < W; ++w) {
        for (int p = 0; p < P; ++p) {
            const int s = w % S, i = w * P + p;
            n_shard[i] = len[p][s] * INNER[p];
            n_full[i] = DIM0[p] * INNER[p];
            shards[i] = dev_alloc((size_t)n_shard[i] * 2);
            sgrad[i] = dev_alloc((size_t)n_shard[i] * 2);
            full[i] = dev_alloc((size_t)n_full[i] * 2);
            full2[i] = dev_alloc((size_t)n_full[i] * 2);
            grads[i] = dev_alloc((size_t)n_full[i] * 2);
            uint16_t* h = (uint16_t*)malloc((size_t)(n_full[i] ? n_full[i] : 1) * 2);
            for (int64_t k = 0; k < n_shard[i]; ++k) h[k] = bf16((float)(100 * p + off[p][s] * INNER[p] + k));
            CUDA(cudaMemcpy(shards[i], h, (size_t)n_shard[i] * 2, cudaMemcpyHostToDevice));
            for (int64_t e = 0; e < n_full[i]; ++e) h[e] = bf16((float)((w + 1) * (1 + e % 3)));
            CUDA(cudaMemcpy(grads[i], h, (size_t)n_full[i] * 2, cudaMemcpyHostToDevice));
            free(h);
        }
        n_ag[w] = S * sl_bf16;
        n_fused[w] = sl_f32;
        ag[w] = dev_alloc((size_t)n_ag[w] * 2);
        fused[w] = dev_alloc((size_t)n_fused[w] * 4);
    }
    fsdp_binding_t b_shards, b_ag, b_full, b_full2, b_grads, b_fused, b_sgrad;
    OK(fsdp_bind(plan, FSDP_ROLE_SHARDS, FSDP_BF16, (const void* const*)shards, n_shard, &b_shards));
    OK(fsdp_bind(plan, FSDP_ROLE_AG_OUTPUT, FSDP_BF16, (const void* const*)ag, n_ag, &b_ag));
    OK(fsdp_bind(plan, FSDP_ROLE_FULL_PARAMS, FSDP_BF16, (const void* const*)full, n_full, &b_full));
    OK(fsdp_bind(plan, FSDP_ROLE_FULL_PARAMS, FSDP_BF16, (const void* const*)full2, n_full, &b_full2));
    OK(fsdp_bind(plan, FSDP_ROLE_GRADS, FSDP_BF16, (const void* const*)grads, n_full, &b_grads));
    OK(fsdp_bind(plan, FSDP_ROLE_FUSED, FSDP_F32, (const void* const*)fused, n_fused, &b_fused));
    OK(fsdp_bind(plan, FSDP_ROLE_SHARD_GRADS, FSDP_BF16, (const void* const*)sgrad, n_shard, &b_sgrad));

    /* the step: each data call enqueues exactly one kernel */
    const uint64_t l0 = fsdp_launch_count();
    OK(fsdp_ag_copy_in(plan, b_shards, b_ag, 1, NULL));
    OK(fsdp_ag_copy_out(plan, b_ag, b_full, NULL));
    OK(fsdp_ag_unshard(plan, b_shards, b_full2, NULL));
    OK(fsdp_rs_ar_reduce(plan, b_grads, b_fused, NULL));
    OK(fsdp_apply_grads(plan, b_fused, FSDP_AVG, 0, b_sgrad, NULL));
    CUDA(cudaDeviceSynchronize());
    CHECK(fsdp_launch_count() - l0 == 5, "launches %llu", (unsigned long long)(fsdp_launch_count() - l0));

    /* forward: every rank holds every full parameter, by both routes */
    for (int i = 0; i < W * P; ++i) {
        const int p = i % P;
        uint16_t* h = (uint16_t*)malloc((size_t)n_full[i] * 2);
        uint16_t* h2 = (uint16_t*)malloc((size_t)n_full[i] * 2);
        CUDA(cudaMemcpy(h, full[i], (size_t)n_full[i] * 2, cudaMemcpyDeviceToHost));
        CUDA(cudaMemcpy(h2, full2[i], (size_t)n_full[i] * 2, cudaMemcpyDeviceToHost));
        for (int64_t e = 0; e < n_full[i]; ++e) {
            const uint16_t want = bf16((float)(100 * p + e));
            CHECK(h[e] == want, "full[%d][%lld] = %04x, want %04x", i, (long long)e, h[e], want);
            CHECK(h2[e] == want, "unshard full[%d][%lld] = %04x, want %04x", i, (long long)e, h2[e], want);
        }
        free(h);
        free(h2);
    }

    /* gradient sync: the fused region holds the sum over all ranks at o_p,
     * +0 in padding rows and the tail; AVG divides by rank_size once */
    for (int w = 0; w < W; ++w) {
        const int s = w % S;
        float* f = (float*)malloc((size_t)n_fused[w] * 4);
        CUDA(cudaMemcpy(f, fused[w], (size_t)n_fused[w] * 4, cudaMemcpyDeviceToHost));
        for (int64_t j = 0; j < n_fused[w]; ++j) {
            float want = 0.0f;
            for (int p = 0; p < P; ++p)
                if (j >= o[p] && j < o[p] + len[p][s] * INNER[p]) {
                    const int64_t e = off[p][s] * INNER[p] + (j - o[p]);
                    want = (float)(10 * (1 + e % 3));
                }
            uint32_t got_bits, want_bits;
            memcpy(&got_bits, &f[j], 4);
            memcpy(&want_bits, &want, 4);
            CHECK(got_bits == want_bits, "fused[%d][%lld] = %g, want %g", w, (long long)j, f[j], want);
        }
        free(f);
    }
    for (int op = FSDP_AVG; op <= FSDP_SUM; ++op) {
        if (op == FSDP_SUM) {
            OK(fsdp_apply_grads(plan, b_fused, FSDP_SUM, 0, b_sgrad, NULL));
            CUDA(cudaDeviceSynchronize());
        }
        for (int i = 0; i < W * P; ++i) {
            const int w = i / P, p = i % P, s = w % S;
            uint16_t* h = (uint16_t*)malloc((size_t)(n_shard[i] ? n_shard[i] : 1) * 2);
            CUDA(cudaMemcpy(h, sgrad[i], (size_t)n_shard[i] * 2, cudaMemcpyDeviceToHost));
            for (int64_t k = 0; k < n_shard[i]; ++k) {
                const int64_t e = off[p][s] * INNER[p] + k;
                const float sum = (float)(10 * (1 + e % 3));
                const uint16_t want = bf16(op == FSDP_AVG ? sum / W : sum);
                CHECK(h[k] == want, "%s shard grad[%d][%lld] = %04x, want %04x", op == FSDP_AVG ? "AVG" : "SUM",
                      i, (long long)k, h[k], want);
            }
            free(h);
        }
    }

    /* the sync in one pass: the same fused regions and shard gradients from
     * one kernel, on buffers dirtied first; the last round on a grid capped
     * at 3 blocks (the bulk-fed kernel, whose waits report through the
     * plan's status word) */
    for (int round = 0; round < 3; ++round) {
        const int op = round == 1 ? FSDP_SUM : FSDP_AVG;
        OK(fsdp_plan_set_grid_limit(plan, round == 2 ? 3 : 0));
        for (int w = 0; w < W; ++w) CUDA(cudaMemset(fused[w], 0xFF, (size_t)n_fused[w] * 4));
        for (int i = 0; i < W * P; ++i)
            if (n_shard[i]) CUDA(cudaMemset(sgrad[i], 0xFF, (size_t)n_shard[i] * 2));
        const uint64_t l1 = fsdp_launch_count();
        OK(fsdp_rs_ar_reduce_apply(plan, b_grads, b_fused, op, 0, b_sgrad, NULL));
        CUDA(cudaDeviceSynchronize());
        CHECK(fsdp_launch_count() - l1 == 1, "one-pass launches %llu", (unsigned long long)(fsdp_launch_count() - l1));
        for (int w = 0; w < W; ++w) {
            const int s = w % S;
            float* f = (float*)malloc((size_t)n_fused[w] * 4);
            CUDA(cudaMemcpy(f, fused[w], (size_t)n_fused[w] * 4, cudaMemcpyDeviceToHost));
            for (int64_t j = 0; j < n_fused[w]; ++j) {
                float want = 0.0f;
                for (int p = 0; p < P; ++p)
                    if (j >= o[p] && j < o[p] + len[p][s] * INNER[p])
                        want = (float)(10 * (1 + (off[p][s] * INNER[p] + (j - o[p])) % 3));
                CHECK(memcmp(&f[j], &want, 4) == 0, "one-pass fused[%d][%lld] = %g, want %g", w, (long long)j, f[j],
                      want);
            }
            free(f);
        }
        for (int i = 0; i < W * P; ++i) {
            const int w = i / P, p = i % P, s = w % S;
            uint16_t* h = (uint16_t*)malloc((size_t)(n_shard[i] ? n_shard[i] : 1) * 2);
            CUDA(cudaMemcpy(h, sgrad[i], (size_t)n_shard[i] * 2, cudaMemcpyDeviceToHost));
            for (int64_t k = 0; k < n_shard[i]; ++k) {
                const float sum = (float)(10 * (1 + (off[p][s] * INNER[p] + k) % 3));
                const uint16_t want = bf16(op == FSDP_AVG ? sum / W : sum);
                CHECK(h[k] == want, "one-pass %s shard grad[%d][%lld] = %04x, want %04x",
                      op == FSDP_AVG ? "AVG" : "SUM", i, (long long)k, h[k], want);
            }
            free(h);
        }
        int status = -1;
        OK(fsdp_plan_status(plan, NULL, &status));
        CHECK(status == 0, "plan status %d after the one-pass sync (round %d)", status, round);
    }
    OK(fsdp_plan_set_grid_limit(plan, 0));

    OK(fsdp_binding_destroy(b_shards));
    OK(fsdp_binding_destroy(b_ag));
    OK(fsdp_binding_destroy(b_full));
    OK(fsdp_binding_destroy(b_full2));
    OK(fsdp_binding_destroy(b_grads));
    OK(fsdp_binding_destroy(b_fused));
    OK(fsdp_binding_destroy(b_sgrad));
    OK(fsdp_plan_destroy(plan));
    for (int i = 0; i < W * P; ++i) {
        CUDA(cudaFree(shards[i]));
        CUDA(cudaFree(full[i]));
        CUDA(cudaFree(full2[i]));
        CUDA(cudaFree(grads[i]));
        CUDA(cudaFree(sgrad[i]));
    }
    for (int w = 0; w < W; ++w) {
        CUDA(cudaFree(ag[w]));
        CUDA(cudaFree(fused[w]));
    }
    if (failures) {
        fprintf(stderr, "abi_check: %d failures\n", failures);
        return 1;
    }
    printf("abi_check: ok\n");
    return 0;
}
