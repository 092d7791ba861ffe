// Small kernels around the W4 GEMM: MoE routing and combine, and the synthetic
// decoder's embedding gather and RMSNorm.  All are per-row (one CTA or one
// fixed reduction tree per row), so no row's bits depend on R.
#include <cuda_bf16.h>

#include "glue.cuh"
#include "tf_ptx.cuh"

namespace tfk {

namespace {

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// MoE routing (TensorFold README: MoE kernels over 4-bit group-32 weights; the
// 30B-A3B class routes each token to its top-8 of 128 experts).
__global__ void route_kernel(const float *router, int E, int top_k, int32_t *ids, float *w, int *err) {
    __shared__ unsigned long long s_best[32];
    __shared__ int s_sel[kMaxRouteK];
    __shared__ int s_bad;
    const int r = blockIdx.x, tid = threadIdx.x;
    const float z = tid < E ? router[(long long)r * E + tid] : 0.f;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    if (tid < E && !isfinite(z)) atomicOr(&s_bad, 1);
    __syncthreads();
    if (s_bad) {
        if (tid == 0) set_error(err, 2);
        if (tid < top_k) {
            ids[r * kMaxRouteK + tid] = tid;
            w[r * kMaxRouteK + tid] = 0.f;
        }
        return;
    }
    // composite key: (logit desc, id asc); distinct for distinct ids
    unsigned long long key =
        tid < E ? ((unsigned long long)order_key(z) << 32) | (0xFFFFFFFFull - (unsigned)tid) : 0ull;
    for (int j = 0; j < top_k; ++j) {
        unsigned long long m = key;
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long v = __shfl_xor_sync(0xFFFFFFFFu, m, o);
            m = v > m ? v : m;
        }
        if ((tid & 31) == 0) s_best[tid >> 5] = m;
        __syncthreads();
        if (tid == 0) {
            unsigned long long b = 0;
            for (int i = 0; i < int(blockDim.x + 31) / 32; ++i) b = s_best[i] > b ? s_best[i] : b;
            s_sel[j] = int(0xFFFFFFFFull - (b & 0xFFFFFFFFull));
        }
        __syncthreads();
        if (tid == s_sel[j]) key = 0ull;  // remove the chosen expert
    }
    if (tid == 0) {
        double e[kMaxRouteK];
        const double z0 = double(router[(long long)r * E + s_sel[0]]);
        double tot = 0.0;
        for (int j = 0; j < top_k; ++j) {
            e[j] = exp(double(router[(long long)r * E + s_sel[j]]) - z0);
            tot += e[j];
        }
        for (int j = 0; j < top_k; ++j) {
            ids[r * kMaxRouteK + j] = s_sel[j];
            w[r * kMaxRouteK + j] = float(e[j] / tot);
        }
    }
}

__global__ void expert_list_kernel(const int32_t *ids, int R, int E, int top_k, int32_t *expert_ids,
                                   int32_t *n_problems, int32_t *slot_of) {
    __shared__ int touched[kMaxExperts];
    __shared__ int pos[kMaxExperts];
    const int tid = threadIdx.x;
    for (int e = tid; e < kMaxExperts; e += blockDim.x) touched[e] = 0;
    __syncthreads();
    for (int i = tid; i < R * top_k; i += blockDim.x) touched[ids[(i / top_k) * kMaxRouteK + i % top_k]] = 1;
    __syncthreads();
    if (tid == 0) {
        int n = 0;
        for (int e = 0; e < E; ++e) {
            pos[e] = n;
            if (touched[e]) expert_ids[n++] = e;
        }
        *n_problems = n;
    }
    __syncthreads();
    for (int i = tid; i < R * top_k; i += blockDim.x) {
        const int r = i / top_k, j = i % top_k;
        slot_of[r * kMaxRouteK + j] = pos[ids[r * kMaxRouteK + j]];
    }
}

__global__ void combine_kernel(const float *Y, const int32_t *slot_of, const float *w, int R, int H, int top_k,
                               float *out) {
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

}  // namespace

cudaError_t launch_route(const float *router, int R, int E, int top_k, int32_t *ids, float *w, int *err,
                         cudaStream_t s) {
    route_kernel<<<R, kMaxExperts, 0, s>>>(router, E, top_k, ids, w, err);
    return cudaGetLastError();
}

cudaError_t launch_expert_list(const int32_t *ids, int R, int E, int top_k, int32_t *expert_ids,
                               int32_t *n_problems, int32_t *slot_of, cudaStream_t s) {
    expert_list_kernel<<<1, 256, 0, s>>>(ids, R, E, top_k, expert_ids, n_problems, slot_of);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *Y, const int32_t *slot_of, const float *w, int R, int H, int top_k,
                           float *out, cudaStream_t s) {
    combine_kernel<<<dim3((H + 255) / 256, R), 256, 0, s>>>(Y, slot_of, w, R, H, top_k, out);
    return cudaGetLastError();
}

cudaError_t launch_embed(const uint16_t *emb, int V, int H, const int32_t *last_token, const int32_t *drafts,
                         int R, float *x, int *err, cudaStream_t s) {
    embed_kernel<<<R, 256, 0, s>>>(emb, V, H, last_token, drafts, x, err);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const float *x, int R, int H, float eps, uint16_t *out, cudaStream_t s) {
    rmsnorm_bf16_kernel<<<R, 256, 0, s>>>(x, H, eps, out);
    return cudaGetLastError();
}

}  // namespace tfk
