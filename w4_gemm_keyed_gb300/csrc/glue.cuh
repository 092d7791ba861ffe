// MoE routing / combine and synthetic-decoder glue kernels: declarations.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace tfk {

constexpr int kMaxExperts = 256;
constexpr int kMaxRouteK = 8;

constexpr int kMaxRows = 16;
// Per row: experts ranked by (router logit desc, id asc), first top_k kept,
// renormalised weights computed in fp64 and stored as fp32; then the touched
// experts in ascending id: expert_ids[0..U), *n_problems = U, and
// slot_of[r][j] = index u of ids[r][j].  One CTA, R <= kMaxRows.
cudaError_t launch_route_list(const float *router, int R, int E, int top_k, int32_t *ids, float *w,
                              int32_t *expert_ids, int32_t *n_problems, int32_t *slot_of, int *err, cudaStream_t s);
// drafts[i] = table[*pos + i] (0 outside the table), i < n.
cudaError_t launch_gather_drafts(const int32_t *table, long long table_len, const int64_t *pos, int n,
                                 int32_t *drafts, cudaStream_t s);
// After a verify pass that advanced *pos by a + 1: log[*pos - (a + 1) - 1 + i] = tokens[i], i <= a.
cudaError_t launch_commit_tokens(const int32_t *tokens, const int32_t *accepted, const int64_t *pos, int32_t *log,
                                 long long log_len, cudaStream_t s);
// out[r][n] = sum_j w[r][j] * Y[slot_of[r][j]][r][n], j ascending (fp32 FMA chain).
cudaError_t launch_combine(const float *Y, const int32_t *slot_of, const float *w, int R, int H, int top_k,
                           float *out, cudaStream_t s);

// y[r][n] = bf16(x[r][n]), round to nearest even.
cudaError_t launch_cast_bf16(const float *x, int R, int N, int ldx, uint16_t *y, int ldy, cudaStream_t s);
// *first = min(*first, code_base + r) over rows r < R whose N fp32 values differ in any bit.
cudaError_t launch_rows_differ(const float *a, const float *b, int R, int N, int ld, int code_base, int *first,
                               cudaStream_t s);

// x[r][:] = emb[token_r][:] (bf16 -> fp32); token_0 = *last_token, token_r = drafts[r-1].
cudaError_t launch_embed(const uint16_t *emb, int V, int H, const int32_t *last_token, const int32_t *drafts,
                         int R, float *x, int *err, cudaStream_t s);
// out[r][:] = bf16(x[r][:] / sqrt(mean(x[r]^2) + eps)), fixed-order fp32 reduction per row.
cudaError_t launch_rmsnorm_bf16(const float *x, int R, int H, float eps, uint16_t *out, cudaStream_t s);

}  // namespace tfk
