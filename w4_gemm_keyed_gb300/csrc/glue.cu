// Small kernels around the W4 GEMM: MoE routing and combine, and the synthetic
// decoder's embedding gather and RMSNorm.  All are per-row (one CTA or one
// fixed reduction tree per row), so no row's bits depend on R.
#include <cuda_bf16.h>

#include "glue.cuh"
#include "tf_keys.cuh"
#include "tf_ptx.cuh"

namespace tfk {

namespace {

// MoE routing (TensorFold README: MoE kernels over 4-bit group-32 weights; the
// 30B-A3B class routes each token to its top-8 of 128 experts), followed by the
// list of touched experts, in one CTA of R + 1 warps.
//   1. Warp r routes row r: the k-th largest of the lanes' largest keys bounds
//      the row's k-th best from below (k lanes hold a key at or above it), so
//      only the few keys at or above it are ranked; their ranks give the
//      row's k best in order (key = (logit desc, expert id asc)).
//   2. Warp r forms row r's renormalised weights in fp32 (summed in rank
//      order) while warp R numbers the touched experts in ascending id and
//      maps every (row, rank) to its expert's slot.
__global__ void route_list_kernel(const float *router, int R, int E, int top_k, int32_t *ids, float *w,
                                  int32_t *expert_ids, int32_t *n_problems, int32_t *slot_of, int *err) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    constexpr int KE = kMaxExperts / 32;   // experts per lane
    __shared__ int s_ids[kMaxRows][kMaxRouteK];
    __shared__ int s_bad[kMaxRows];
    __shared__ uint64_t s_surv[kMaxRows][kMaxExperts];
    __shared__ int touched[kMaxExperts];
    __shared__ int pos[kMaxExperts];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned lt = (1u << lane) - 1u;
    if (warp < R) {
        const int r = warp;
        const float *z = router + (long long)r * E;
        uint64_t key[KE];
        bool bad = false;
        uint64_t lmax = 0ull;
#pragma unroll
        for (int i = 0; i < KE; ++i) {
            const int e = lane + 32 * i;
            key[i] = 0ull;
            if (e < E) {
                const float v = z[e];
                bad |= !isfinite(v);
                key[i] = composite(order_key(v), e);
                lmax = key[i] > lmax ? key[i] : lmax;
            }
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) s_bad[r] = bad ? 1 : 0;
        if (bad) {
            if (lane == 0) set_error(err, 2);
            if (lane < top_k) s_ids[r][lane] = lane;
        } else {
            const uint64_t L = __shfl_sync(0xFFFFFFFFu, warp_sort_desc(lmax), top_k - 1);
            int ns = 0;
#pragma unroll
            for (int i = 0; i < KE; ++i) {
                const bool sv = key[i] != 0ull && key[i] >= L;
                const unsigned m = __ballot_sync(0xFFFFFFFFu, sv);
                if (sv) s_surv[r][ns + __popc(m & lt)] = key[i];
                ns += __popc(m);
            }
            __syncwarp();
            for (int j = lane; j < ns; j += 32) {
                const uint64_t v = s_surv[r][j];
                int rank = 0;
                for (int t = 0; t < ns; ++t) rank += s_surv[r][t] > v;
                if (rank < top_k) s_ids[r][rank] = composite_id(v);
            }
        }
    }
    __syncthreads();
    if (warp < R) {
        const int r = warp;
        if (s_bad[r]) {
            if (lane < top_k) {
                ids[r * kMaxRouteK + lane] = lane;
                w[r * kMaxRouteK + lane] = 0.f;
            }
        } else {
            // renormalised weights over the kept experts, fp32, summed in rank
            // order (within a few ulp of the exact softmax; the row warps of
            // one CTA share the SM's few fp64 units, where this took ~1 us a row)
            const float *z = router + (long long)r * E;
            float ej = 0.f;
            if (lane < top_k) ej = expf(z[s_ids[r][lane]] - z[s_ids[r][0]]);
            // every lane forms the same left-to-right sum; lane j divides its own term
            float tot = 0.f;
            for (int j = 0; j < top_k; ++j) tot += __shfl_sync(0xFFFFFFFFu, ej, j);
            if (lane < top_k) {
                ids[r * kMaxRouteK + lane] = s_ids[r][lane];
                w[r * kMaxRouteK + lane] = __fdiv_rn(ej, tot);
            }
        }
    } else if (warp == R) {
        for (int e = lane; e < kMaxExperts; e += 32) touched[e] = 0;
        __syncwarp();
        for (int i = lane; i < R * top_k; i += 32) touched[s_ids[i / top_k][i % top_k]] = 1;
        __syncwarp();
        int base = 0;
        for (int c = 0; c < KE; ++c) {
            const int e = c * 32 + lane;
            const int f = e < E ? touched[e] : 0;
            const unsigned b = __ballot_sync(0xFFFFFFFFu, f);
            pos[e] = base + __popc(b & lt);
            if (f) expert_ids[base + __popc(b & lt)] = e;
            base += __popc(b);
        }
        if (lane == 0) *n_problems = base;
        __syncwarp();
        for (int i = lane; i < R * top_k; i += 32) {
            const int r = i / top_k, j = i % top_k;
            slot_of[r * kMaxRouteK + j] = pos[s_ids[r][j]];
        }
    }
}

__global__ void combine_kernel(const float *Y, const int32_t *slot_of, const float *w, int R, int H, int top_k,
                               float *out) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    const int r = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= H) return;
    float acc = 0.f;
    for (int j = 0; j < top_k; ++j) {
        const long long u = slot_of[r * kMaxRouteK + j];
        acc = fmaf(w[r * kMaxRouteK + j], Y[(u * R + r) * H + n], acc);
    }
    out[(long long)r * H + n] = acc;
}

__global__ void embed_kernel(const uint16_t *emb, int V, int H, const int32_t *last_token, const int32_t *drafts,
                             float *x, int *err) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    const int r = blockIdx.x;
    int tok = r == 0 ? *last_token : drafts[r - 1];
    if (tok < 0 || tok >= V) {
        if (threadIdx.x == 0) set_error(err, 3);
        tok = 0;
    }
    const uint16_t *src = emb + (long long)tok * H;
    for (int h = threadIdx.x; h < H; h += blockDim.x)
        x[(long long)r * H + h] = __uint_as_float(uint32_t(src[h]) << 16);
}

__global__ void rmsnorm_bf16_kernel(const float *x, int H, float eps, uint16_t *out) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    __shared__ float s_part[32];
    const int r = blockIdx.x, tid = threadIdx.x;
    const float *xr = x + (long long)r * H;
    float ss = 0.f;
    for (int h = tid; h < H; h += blockDim.x) ss = fmaf(xr[h], xr[h], ss);
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    if (tid < 32) {
        float v = tid < int(blockDim.x >> 5) ? s_part[tid] : 0.f;
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (tid == 0) s_part[0] = v;
    }
    __syncthreads();
    const float inv = 1.0f / sqrtf(s_part[0] / float(H) + eps);
    for (int h = tid; h < H; h += blockDim.x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(xr[h] * inv);
        out[(long long)r * H + h] = __bfloat16_as_ushort(b);
    }
}

// Device-side decode loop helpers: the next verify pass's drafts come from a
// table of proposals indexed by position, and each pass's committed tokens are
// written into a log indexed by position, so consecutive passes chain on the
// device (and can be captured in one CUDA graph).
__global__ void gather_drafts_kernel(const int32_t *table, long long table_len, const int64_t *pos, int n,
                                     int32_t *drafts) {
    grid_dependency_wait();     // *pos comes from the preceding pass
    grid_launch_dependents();
    const int i = threadIdx.x;
    if (i < n) {
        const long long q = *pos + i;   // draft i proposes position *pos + i
        drafts[i] = (q >= 0 && q < table_len) ? table[q] : 0;
    }
}

__global__ void commit_tokens_kernel(const int32_t *tokens, const int32_t *accepted, const int64_t *pos,
                                     int32_t *log, long long log_len) {
    grid_dependency_wait();     // tokens, accepted and the advanced *pos come from the pass
    grid_launch_dependents();
    const int a = *accepted;
    const long long first = *pos - (a + 1);   // position of t[0]; *pos was advanced by a + 1
    const int i = threadIdx.x;
    if (i <= a) {
        const long long q = first - 1 + i;  // position 1 is the first generated token
        if (q >= 0 && q < log_len) log[q] = tokens[i];
    }
}

__global__ void cast_bf16_kernel(const float *x, int N, int ldx, uint16_t *y, int ldy) {
    grid_dependency_wait();     // x comes from the preceding grid
    grid_launch_dependents();
    const int r = blockIdx.y, n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n < N) y[(long long)r * ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(x[(long long)r * ldx + n]));
}

// *first = min(*first, code_base + r) for every row r whose bytes differ
// between a and b (grid-stride over R x N).
__global__ void rows_differ_kernel(const float *a, const float *b, int R, int N, int ld, int code_base, int *first) {
    grid_dependency_wait();     // both outputs come from preceding grids
    grid_launch_dependents();
    const long long total = (long long)R * N;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int r = int(i / N), n = int(i % N);
        if (__float_as_uint(a[(long long)r * ld + n]) != __float_as_uint(b[(long long)r * ld + n]))
            atomicMin(first, code_base + r);
    }
}

}  // namespace

cudaError_t launch_cast_bf16(const float *x, int R, int N, int ldx, uint16_t *y, int ldy, cudaStream_t s) {
    return launch_pdl(cast_bf16_kernel, dim3((N + 255) / 256, R), dim3(256), 0, s, x, N, ldx, y, ldy);
}

cudaError_t launch_rows_differ(const float *a, const float *b, int R, int N, int ld, int code_base, int *first,
                               cudaStream_t s) {
    return launch_pdl(rows_differ_kernel, dim3(256), dim3(256), 0, s, a, b, R, N, ld, code_base, first);
}

cudaError_t launch_gather_drafts(const int32_t *table, long long table_len, const int64_t *pos, int n,
                                 int32_t *drafts, cudaStream_t s) {
    return launch_pdl(gather_drafts_kernel, dim3(1), dim3(32), 0, s, table, table_len, pos, n, drafts);
}

cudaError_t launch_commit_tokens(const int32_t *tokens, const int32_t *accepted, const int64_t *pos, int32_t *log,
                                 long long log_len, cudaStream_t s) {
    return launch_pdl(commit_tokens_kernel, dim3(1), dim3(32), 0, s, tokens, accepted, pos, log, log_len);
}

cudaError_t launch_route_list(const float *router, int R, int E, int top_k, int32_t *ids, float *w,
                              int32_t *expert_ids, int32_t *n_problems, int32_t *slot_of, int *err, cudaStream_t s) {
    return launch_pdl(route_list_kernel, dim3(1), dim3(32 * (R + 1)), 0, s, router, R, E, top_k, ids, w, expert_ids,
                      n_problems, slot_of, err);
}

cudaError_t launch_combine(const float *Y, const int32_t *slot_of, const float *w, int R, int H, int top_k,
                           float *out, cudaStream_t s) {
    return launch_pdl(combine_kernel, dim3((H + 255) / 256, R), dim3(256), 0, s, Y, slot_of, w, R, H, top_k, out);
}

cudaError_t launch_embed(const uint16_t *emb, int V, int H, const int32_t *last_token, const int32_t *drafts,
                         int R, float *x, int *err, cudaStream_t s) {
    return launch_pdl(embed_kernel, dim3(R), dim3(256), 0, s, emb, V, H, last_token, drafts, x, err);
}

cudaError_t launch_rmsnorm_bf16(const float *x, int R, int H, float eps, uint16_t *out, cudaStream_t s) {
    return launch_pdl(rmsnorm_bf16_kernel, dim3(R), dim3(256), 0, s, x, H, eps, out);
}

}  // namespace tfk
