// Row-exact attention of verify rows over a KV cache.
//
// The TensorFold README's note on drafting: starting from one cache, a run
// with drafts emits exactly the tokens of a run without them.  With attention
// in the pass, that needs each row's result to depend only on its own query,
// its own position p and the cache entries 0..p -- never on how many rows
// share the launch or where the launch starts.
// The arithmetic here is fixed by absolute positions alone:
//
//   * keys are cut into partitions of 256 positions (c*256 .. c*256+255) and
//     each partition into 4 steps of 64 keys; a row folds the steps of a
//     partition in ascending order with an online softmax (running max m,
//     weight sum l, unnormalised output o, all fp32);
//   * the partitions 0..p/256 of a row are combined against their common
//     max in an order fixed by p (four contiguous groups, each ascending);
//   * steps past a row's position are exact no-ops for that row (scale 1,
//     weights 0), so rows of one launch may run more steps than they need;
//   * scores and P.V run on mma.sync with the queries as MMA rows; MMA rows
//     never mix, so a row's bits do not depend on its slot.  P is split into
//     bf16 hi + lo parts (two MMAs), keeping ~16 bits of each weight.
#include <atomic>

#include <cuda_bf16.h>

#include "attention.cuh"
#include "tf_ptx.cuh"
#include "w4_gemm.cuh"

namespace tfk {

namespace {

constexpr int kRowBytes = kHeadDim * 2;                 // 256 B per key
constexpr int kSubBytes = kKvSub * kRowBytes;           // 16 KB of K (or V) per step
constexpr int kStageBytes = 2 * kSubBytes;              // K then V
constexpr size_t attn_smem(int ns) { return size_t(ns) * kStageBytes + 2 * ns * sizeof(uint64_t); }
constexpr float kScoreLog2 = 0.12751743074439720f;      // log2(e) / sqrt(128)

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 b) { return *reinterpret_cast<uint32_t *>(&b); }

// (a, b) -> bf16 hi parts and bf16 lo parts (a - hi, exact in fp32), low half = a.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = bf16x2_bits(h);
    lo = bf16x2_bits(__floats2bfloat162_rn(a - hf.x, b - hf.y));
}

__device__ __forceinline__ bool bad_position(long long pos0, int R, int max_len) {
    return pos0 < 0 || pos0 + R > max_len;
}

// Persistent CTAs over items (KV head j, partition c), j-major; each CTA takes
// a contiguous run of items.  Warp w takes 16 query vectors (query vector
// v = row * group + head-in-group).  Thread 0 also streams the items' 64-key
// steps of K and V through a ring of NS stages with bulk copies (NS = 2 where
// three CTAs share an SM, else 3), running ahead across item boundaries; it
// refills a stage once every warp has released it.  Each item's state starts
// afresh, so its partial result is the same whichever CTA computes it.
template <int NS>
__global__ void __launch_bounds__(32 * kAttnMaxGroup, 1) attn_partial_kernel(AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    grid_dependency_wait();     // the cache entries and queries come from the preceding grids
    grid_launch_dependents();
    const long long pos0 = *a.pos;
    if (bad_position(pos0, a.R, a.max_len)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, kDevBadPosition);
        return;
    }
    const long long p_max = pos0 + a.R - 1;
    const int n_parts = int(p_max / kKvPart) + 1;
    const int n_items = n_parts * a.n_kv;
    const int P = int(gridDim.x);
    const int q_it = n_items / P, rem = n_items % P;
    const int it_begin = int(blockIdx.x) * q_it + min(int(blockIdx.x), rem);
    const int it_end = it_begin + q_it + (int(blockIdx.x) < rem ? 1 : 0);
    if (it_begin >= it_end) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_cw = int(blockDim.x >> 5);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * kStageBytes);
    uint64_t *empty = full + NS;

    // V rows past the copied prefix of a step must hold finite values (their
    // weight is 0, and 0 * finite = 0): zero the V halves once.
    for (int i = threadIdx.x; i < NS * kSubBytes / 16; i += blockDim.x) {
        const int st = i / (kSubBytes / 16), o = i % (kSubBytes / 16);
        reinterpret_cast<uint4 *>(smem + st * kStageBytes + kSubBytes)[o] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < NS; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], n_cw);
        }
        fence_mbar_init();
    }
    fence_proxy_async_smem();   // the zero fill precedes the bulk copies into the same bytes
    __syncthreads();

    // steps of partition c: 64-key steps up to the last position any row needs
    auto steps_of = [&](int c) { return int(min((long long)(kKvPart / kKvSub), (p_max - (long long)c * kKvPart) / kKvSub + 1)); };

    // producer cursor (thread 0 only): next item / step to copy, steps issued
    int p_it = it_begin, p_sub = 0, n_issued = 0;
    const uint64_t pol = l2_policy_evict_first();
    auto issue_next = [&]() {
        const int j = p_it / n_parts, c = p_it % n_parts;
        const int st = n_issued % NS;
        const long long t0 = (long long)c * kKvPart + (long long)p_sub * kKvSub;
        const uint32_t bytes = uint32_t(min((long long)kKvSub, p_max - t0 + 1)) * kRowBytes;
        const size_t off = ((size_t)j * a.max_len + (size_t)t0) * kHeadDim;
        mbar_arrive_expect_tx(&full[st], 2 * bytes);
        bulk_g2s_hint(smem + st * kStageBytes, a.k + off, bytes, &full[st], pol);
        bulk_g2s_hint(smem + st * kStageBytes + kSubBytes, a.v + off, bytes, &full[st], pol);
        ++n_issued;
        if (++p_sub == steps_of(c)) {
            p_sub = 0;
            ++p_it;
        }
    };
    if (threadIdx.x == 0)
        for (int i = 0; i < NS && p_it < it_end; ++i) issue_next();

    // ------------------------------------------------------------------ consumers
    const int gq = lane >> 2, tq = lane & 3;
    const int g = a.group, n_q = a.n_kv * g, nqv = a.R * g;
    const int v0 = 16 * warp + gq, v1 = v0 + 8;
    const bool ok0 = v0 < nqv, ok1 = v1 < nqv;
    const int r0 = v0 / g, r1 = v1 / g;
    // positions of the slot's two rows (-1: the slot holds no row)
    const long long p0 = ok0 ? pos0 + r0 : -1, p1 = ok1 ? pos0 + r1 : -1;
    const uint32_t sbase = smem_u32(smem);
    const int sw = lane & 7;    // key & 7 of the rows this lane addresses (steps start at multiples of 8)

    uint32_t qa[8][4];
    int q_head = -1;            // KV head whose queries qa holds
    int s = 0;                  // steps consumed
    for (int it = it_begin; it < it_end; ++it) {
        const int j = it / n_parts, c = it % n_parts;
        const int h0 = j * g + v0 % g, h1 = j * g + v1 % g;
        if (j != q_head) {
            q_head = j;
            const uint32_t *q0 = ok0 ? reinterpret_cast<const uint32_t *>(a.q + (size_t)r0 * a.ldq + h0 * kHeadDim)
                                     : nullptr;
            const uint32_t *q1 = ok1 ? reinterpret_cast<const uint32_t *>(a.q + (size_t)r1 * a.ldq + h1 * kHeadDim)
                                     : nullptr;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qa[ks][0] = ok0 ? q0[8 * ks + tq] : 0u;
                qa[ks][1] = ok1 ? q1[8 * ks + tq] : 0u;
                qa[ks][2] = ok0 ? q0[8 * ks + 4 + tq] : 0u;
                qa[ks][3] = ok1 ? q1[8 * ks + 4 + tq] : 0u;
            }
        }
        const long long t_begin = (long long)c * kKvPart;
        const int n_sub = steps_of(c);

        float o[16][4];
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int i = 0; i < n_sub; ++i, ++s) {
            const int st = s % NS;
            if (!mbar_wait(&full[st], (s / NS) & 1)) {
                set_error(a.err, kDevTimeout);
                return;
            }
            const uint32_t kaddr = sbase + st * kStageBytes, vaddr = kaddr + kSubBytes;
            const long long t0 = t_begin + (long long)i * kKvSub;
            const int lim0 = int(max(-1LL, min((long long)kKvSub, p0 - t0)));
            const int lim1 = int(max(-1LL, min((long long)kKvSub, p1 - t0)));

            // scores S[query][key] = q . k over 64 keys (8 n-tiles), fp32
            float sc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                const uint32_t row = kaddr + (nt * 8 + sw) * kRowBytes;
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    const int chunk = 4 * kp + (lane >> 3);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(row + ((chunk ^ sw) << 4), b0, b1, b2, b3);
                    mma_bf16_16816(sc[nt], qa[2 * kp], b0, b1);
                    mma_bf16_16816(sc[nt], qa[2 * kp + 1], b2, b3);
                }
            }
            // causal mask, then the step's row max (exact, any order)
            float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int kk = nt * 8 + 2 * tq;
                sc[nt][0] = kk <= lim0 ? sc[nt][0] : -INFINITY;
                sc[nt][1] = kk + 1 <= lim0 ? sc[nt][1] : -INFINITY;
                sc[nt][2] = kk <= lim1 ? sc[nt][2] : -INFINITY;
                sc[nt][3] = kk + 1 <= lim1 ? sc[nt][3] : -INFINITY;
                mt0 = fmaxf(mt0, fmaxf(sc[nt][0], sc[nt][1]));
                mt1 = fmaxf(mt1, fmaxf(sc[nt][2], sc[nt][3]));
            }
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xFFFFFFFFu, mt0, 1));
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xFFFFFFFFu, mt0, 2));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xFFFFFFFFu, mt1, 1));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xFFFFFFFFu, mt1, 2));
            const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
            // rescale of the running state: exactly 1 when the max did not move
            const float al0 = mn0 == m0 ? 1.f : exp2f(__fmul_rn(__fsub_rn(m0, mn0), kScoreLog2));
            const float al1 = mn1 == m1 ? 1.f : exp2f(__fmul_rn(__fsub_rn(m1, mn1), kScoreLog2));
            m0 = mn0;
            m1 = mn1;
            const float mc0 = mn0 == -INFINITY ? 0.f : __fmul_rn(mn0, kScoreLog2);
            const float mc1 = mn1 == -INFINITY ? 0.f : __fmul_rn(mn1, kScoreLog2);
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                sc[nt][0] = exp2f(fmaf(sc[nt][0], kScoreLog2, -mc0));
                sc[nt][1] = exp2f(fmaf(sc[nt][1], kScoreLog2, -mc0));
                sc[nt][2] = exp2f(fmaf(sc[nt][2], kScoreLog2, -mc1));
                sc[nt][3] = exp2f(fmaf(sc[nt][3], kScoreLog2, -mc1));
                sum0 += sc[nt][0];
                sum0 += sc[nt][1];
                sum1 += sc[nt][2];
                sum1 += sc[nt][3];
            }
            l0 = fmaf(l0, al0, sum0);
            l1 = fmaf(l1, al1, sum1);
#pragma unroll
            for (int dn = 0; dn < 16; ++dn) {
                o[dn][0] *= al0;
                o[dn][1] *= al0;
                o[dn][2] *= al1;
                o[dn][3] *= al1;
            }
            // o += P.V, 16 keys per k step; P as bf16 hi + lo
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t ah[4], alo[4];
                split_bf16x2(sc[2 * kk][0], sc[2 * kk][1], ah[0], alo[0]);
                split_bf16x2(sc[2 * kk][2], sc[2 * kk][3], ah[1], alo[1]);
                split_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ah[2], alo[2]);
                split_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ah[3], alo[3]);
                const int mi = lane >> 3;
                const uint32_t row = vaddr + (16 * kk + ((mi & 1) << 3) + sw) * kRowBytes;
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    const int chunk = 2 * dp + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(row + ((chunk ^ sw) << 4), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * dp], ah, b0, b1);
                    mma_bf16_16816(o[2 * dp], alo, b0, b1);
                    mma_bf16_16816(o[2 * dp + 1], ah, b2, b3);
                    mma_bf16_16816(o[2 * dp + 1], alo, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (threadIdx.x == 0 && p_it < it_end) {
                // every issued step is consumed by every warp before it exits, so no
                // copy is left in flight; a refill that cannot start makes the
                // warps' next full-barrier waits run out instead
                if (mbar_wait(&empty[st], (s / NS) & 1))
                    issue_next();
                else
                    set_error(a.err, kDevTimeout);
            }
        }

        // weight sums over the quad (same order on all four lanes)
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
        if (ok0 && t_begin <= p0) {
            const size_t b = ((size_t)c * a.R + r0) * n_q + h0;
            float *op = a.opart + b * kHeadDim + 2 * tq;
#pragma unroll
            for (int dn = 0; dn < 16; ++dn) *reinterpret_cast<float2 *>(op + 8 * dn) = make_float2(o[dn][0], o[dn][1]);
            if (tq == 0) *reinterpret_cast<float2 *>(a.ml + 2 * b) = make_float2(m0, l0);
        }
        if (ok1 && t_begin <= p1) {
            const size_t b = ((size_t)c * a.R + r1) * n_q + h1;
            float *op = a.opart + b * kHeadDim + 2 * tq;
#pragma unroll
            for (int dn = 0; dn < 16; ++dn) *reinterpret_cast<float2 *>(op + 8 * dn) = make_float2(o[dn][2], o[dn][3]);
            if (tq == 0) *reinterpret_cast<float2 *>(a.ml + 2 * b) = make_float2(m1, l1);
        }
    }
}

// One CTA per (query head, row): the row's partitions 0..n_c-1 (n_c = p/256 + 1)
// weighted against their common max.  Four groups of 128 threads (one per
// output dimension) each sum a contiguous quarter of every chunk of up to 512
// partitions in ascending order; the group sums are then added in group
// order.  The grouping is a function of n_c alone, i.e. of the row's position.
constexpr int kCombThreads = 512;
constexpr int kCombGroups = kCombThreads / kHeadDim;
constexpr int kCombUnroll = 16;

__global__ void __launch_bounds__(kCombThreads) attn_combine_kernel(AttnArgs a) {
    __shared__ float s_w[kCombThreads], s_l[kCombThreads], s_red[kCombThreads / 32];
    __shared__ float s_o[kCombGroups][kHeadDim], s_lg[kCombGroups];
    grid_dependency_wait();     // partials come from the preceding grid
    grid_launch_dependents();
    const long long pos0 = *a.pos;
    if (bad_position(pos0, a.R, a.max_len)) return;
    const int h = blockIdx.x, r = blockIdx.y, tid = threadIdx.x, d = tid % kHeadDim, grp = tid / kHeadDim;
    const int n_q = a.n_kv * a.group;
    const int n_c = int((pos0 + r) / kKvPart) + 1;
    const size_t stride = (size_t)a.R * n_q, base = (size_t)r * n_q + h;
    float M = -INFINITY;
    for (int c = tid; c < n_c; c += kCombThreads) M = fmaxf(M, a.ml[2 * (c * stride + base)]);
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    if ((tid & 31) == 0) s_red[tid >> 5] = M;
    __syncthreads();
    M = s_red[0];
    for (int w = 1; w < kCombThreads / 32; ++w) M = fmaxf(M, s_red[w]);
    float L = 0.f, O = 0.f;
    for (int c0 = 0; c0 < n_c; c0 += kCombThreads) {
        const int n = min(kCombThreads, n_c - c0);
        __syncthreads();        // the previous chunk's weights are no longer read
        if (tid < n) {
            const float2 mlc = *reinterpret_cast<const float2 *>(a.ml + 2 * ((c0 + tid) * stride + base));
            s_w[tid] = exp2f(__fmul_rn(__fsub_rn(mlc.x, M), kScoreLog2));
            s_l[tid] = mlc.y;
        }
        __syncthreads();
        const int qn = n / kCombGroups, rn = n % kCombGroups;
        const int k0 = grp * qn + min(grp, rn), k1 = k0 + qn + (grp < rn ? 1 : 0);
        const size_t step = stride * kHeadDim;
        const float *op = a.opart + ((c0 + k0) * stride + base) * kHeadDim + d;
        int k = k0;
        for (; k + kCombUnroll <= k1; k += kCombUnroll, op += kCombUnroll * step) {
            float v[kCombUnroll];
#pragma unroll
            for (int u = 0; u < kCombUnroll; ++u) v[u] = op[u * step];
#pragma unroll
            for (int u = 0; u < kCombUnroll; ++u) {
                L = fmaf(s_l[k + u], s_w[k + u], L);
                O = fmaf(v[u], s_w[k + u], O);
            }
        }
        for (; k < k1; ++k, op += step) {
            L = fmaf(s_l[k], s_w[k], L);
            O = fmaf(*op, s_w[k], O);
        }
    }
    s_o[grp][d] = O;
    if (d == 0) s_lg[grp] = L;
    __syncthreads();
    if (grp == 0) {
        float Ot = s_o[0][d], Lt = s_lg[0];
#pragma unroll
        for (int g2 = 1; g2 < kCombGroups; ++g2) {
            Ot += s_o[g2][d];
            Lt += s_lg[g2];
        }
        a.out[(size_t)r * a.ldo + h * kHeadDim + d] = __fdiv_rn(Ot, Lt);
    }
}

// 8 (row, KV head) items per CTA, one warp each: 16 lanes copy the K row and
// 16 the V row, 16 B per lane, into the position's swizzled chunks.
__global__ void kv_append_kernel(const uint16_t *k_new, const uint16_t *v_new, int ld, int R, const int64_t *pos,
                                 uint16_t *k_cache, uint16_t *v_cache, int n_kv, int max_len, int *err) {
    grid_dependency_wait();     // the new entries come from the preceding grid
    grid_launch_dependents();
    const long long pos0 = *pos;
    if (bad_position(pos0, R, max_len)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, kDevBadPosition);
        return;
    }
    const long long item = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (item >= (long long)R * n_kv) return;
    const int r = int(item / n_kv), j = int(item % n_kv);
    const int lane = threadIdx.x & 31, which = lane >> 4, chunk = lane & 15;
    const long long t = pos0 + r;
    const uint16_t *src = (which ? v_new : k_new) + (size_t)r * ld + j * kHeadDim + chunk * 8;
    uint16_t *dst = (which ? v_cache : k_cache) + ((size_t)j * max_len + (size_t)t) * kHeadDim +
                    ((chunk ^ int(t & 7)) << 3);
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
}

}  // namespace

size_t attn_opart_bytes(int n_kv, int group, int max_len, int R) {
    const size_t b = size_t(max_len / kKvPart) * R * n_kv * group * kHeadDim * sizeof(float);
    return (b + 255) / 256 * 256;
}

size_t attn_ml_bytes(int n_kv, int group, int max_len, int R) {
    const size_t b = size_t(max_len / kKvPart) * R * n_kv * group * 2 * sizeof(float);
    return (b + 255) / 256 * 256;
}

cudaError_t launch_kv_append(const uint16_t *k_new, const uint16_t *v_new, int ld, int R, const int64_t *pos,
                             uint16_t *k_cache, uint16_t *v_cache, int n_kv, int max_len, int *err,
                             cudaStream_t s) {
    const long long items = (long long)R * n_kv;
    return launch_pdl(kv_append_kernel, dim3(unsigned((items + 7) / 8)), dim3(256), 0, s, k_new, v_new, ld, R, pos,
                      k_cache, v_cache, n_kv, max_len, err);
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s) {
    static std::atomic<bool> opted_in[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !opted_in[dev]) {
        e = cudaFuncSetAttribute(attn_partial_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(attn_smem(2)));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_partial_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(attn_smem(3)));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) opted_in[dev] = true;
    }
    // CTAs resident per SM: three with a 2-stage ring (64 KB) for up to two warps,
    // else two (3-stage ring, 96 KB) up to four warps, else one (registers)
    const int n_cw = (a.R * a.group + 15) / 16;
    const int per_sm = n_cw <= 2 ? 3 : (n_cw <= kAttnMaxGroup / 2 ? 2 : 1);
    const long long items_max = (long long)(a.max_len / kKvPart) * a.n_kv;
    const int grid = int(min(items_max, (long long)per_sm * device_sm_count()));
    if (n_cw <= 2)
        e = launch_pdl(attn_partial_kernel<2>, dim3(grid), dim3(32 * n_cw), attn_smem(2), s, a);
    else
        e = launch_pdl(attn_partial_kernel<3>, dim3(grid), dim3(32 * n_cw), attn_smem(3), s, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_combine_kernel, dim3(a.n_kv * a.group, a.R), dim3(kCombThreads), 0, s, a);
}

}  // namespace tfk
