// W4 lane GEMM for the speculative-decoding verify pass (sm_103a).
//
// TensorFold README, "A row of a multi-row verify pass gets the same bits as a
// one-row step": up to 16 drafted rows share one launch that streams every
// 4-bit weight once, and row r's bits never depend on how many rows there are.
//
// Structure of one CTA (9 warps, one CTA per SM):
//   * warp 8 (producer): one elected lane streams, per iteration (tile t,
//     k-slice kc), the contiguous packed weight stage with a bulk TMA copy
//     (L2 evict-first) plus the R activation rows of that k-slice, into a
//     14-deep shared-memory ring guarded by full/empty mbarriers;
//   * warps 0-7 (consumers): warp (kg, b) handles feature block b of the tile
//     for the iterations of parity kg.  Per 16-wide k step it turns one 32-bit
//     packed word into the m16n8k16 A fragment with one LOP3 + one bf16x2 FMA
//     per register (exact: integer codes -8..7), loads the activation B
//     fragment with ldmatrix and issues one mma per 8 rows.  Each quantisation
//     group's partial sum is formed in a fresh fp32 fragment and folded into the
//     running sum as  acc = fma(scale, partial, acc).
// Row invariance: rows are MMA columns; a column's result depends only on its
// own activations, the rows 8..15 MMA is simply skipped when R <= 8, and the
// stream-K cut, the k-group parity split and the fixed-order partial sums all
// depend on (T, Kc, Pv) only.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tf_ptx.cuh"
#include "w4_gemm.cuh"

namespace tfk {

namespace {

constexpr uint32_t kBf16One2 = 0x3F803F80u;    // (1.0, 1.0)
constexpr uint32_t kBf16Neg136x2 = 0xC308C308u; // (-136, -136)
constexpr uint32_t kNibMask = 0x000F000Fu;
constexpr uint32_t kBf16Magic = 0x43004300u;    // (128, 128): OR-ing u in gives 128 + u

__device__ __forceinline__ uint32_t word_of(const uint4 &q, int j) {
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

// One 64-wide k slice of one 64-feature block for this warp.
template <int G>
__device__ __forceinline__ void consume_stage(const uint8_t *cb, uint32_t xaddr, int lane, int gq, bool hi,
                                              float (&acc)[4][2][4]) {
    constexpr int NG = kKChunk / G;
    constexpr int KS = G / 16;
    uint4 q[4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) q[mt] = *reinterpret_cast<const uint4 *>(cb + (mt * 32 + lane) * 16);
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
        const uint4 sv = *reinterpret_cast<const uint4 *>(cb + 2048 + grp * 128 + gq * 16);
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        float part[4][2][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) part[mt][n][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const int j = grp * KS + kk;
            uint32_t b0, b1, b2 = 0, b3 = 0;
            if (hi)
                ldsm_x4(xaddr + j * 32, b0, b1, b2, b3);
            else
                ldsm_x2(xaddr + j * 32, b0, b1);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const uint32_t w = word_of(q[mt], j);
                uint32_t af[4];
                af[0] = fma_bf16x2(lop3_and_or(w, kNibMask, kBf16Magic), kBf16One2, kBf16Neg136x2);
                af[1] = fma_bf16x2(lop3_and_or(w >> 4, kNibMask, kBf16Magic), kBf16One2, kBf16Neg136x2);
                af[2] = fma_bf16x2(lop3_and_or(w >> 8, kNibMask, kBf16Magic), kBf16One2, kBf16Neg136x2);
                af[3] = fma_bf16x2(lop3_and_or(w >> 12, kNibMask, kBf16Magic), kBf16One2, kBf16Neg136x2);
                mma_bf16_16816(part[mt][0], af, b0, b1);
                if (hi) mma_bf16_16816(part[mt][1], af, b2, b3);
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const float s_lo = half_lo(sw[mt]);   // feature mt*16 + g
            const float s_hi = half_hi(sw[mt]);   // feature mt*16 + g + 8
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                if (n == 1 && !hi) continue;
                acc[mt][n][0] = fmaf(s_lo, part[mt][n][0], acc[mt][n][0]);
                acc[mt][n][1] = fmaf(s_lo, part[mt][n][1], acc[mt][n][1]);
                acc[mt][n][2] = fmaf(s_hi, part[mt][n][2], acc[mt][n][2]);
                acc[mt][n][3] = fmaf(s_hi, part[mt][n][3], acc[mt][n][3]);
            }
        }
    }
}

__device__ __forceinline__ void put(const GemmArgs &a, void *yb, int r, int f, float v) {
    float *y = static_cast<float *>(yb) + (long long)r * a.ldy + f;
    if (a.mode == kAccumulateF32)
        *y = *y + v;
    else
        *y = v;
}

__device__ __forceinline__ void store_tile(const GemmArgs &a, void *yb, int t, int b, int gq, int tq, bool hi,
                                           const float (&v)[4][2][4]) {
    if (a.mode == kSwiGluBf16) {
        // sub-tiles (0,1) and (2,3) are (gate, up) of the same 16 h columns
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                if (n == 1 && !hi) continue;
                const int j = t * (kTileN / 2) + b * 32 + pr * 16 + gq;
                const int r = n * 8 + tq * 2;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int jj = j + (c >= 2 ? 8 : 0);
                    const int rr = r + (c & 1);
                    if (jj < a.F && rr < a.R) {
                        const float g = v[2 * pr][n][c];
                        const float up = v[2 * pr + 1][n][c];
                        const float h = g / (1.0f + expf(-g)) * up;
                        static_cast<__nv_bfloat16 *>(yb)[(long long)rr * a.ldy + jj] = __float2bfloat16_rn(h);
                    }
                }
            }
        }
        return;
    }
    const int f0 = t * kTileN + b * 64;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (n == 1 && !hi) continue;
            const int f = f0 + mt * 16 + gq;
            const int r = n * 8 + tq * 2;
            if (f < a.N) {
                if (r < a.R) put(a, yb, r, f, v[mt][n][0]);
                if (r + 1 < a.R) put(a, yb, r + 1, f, v[mt][n][1]);
            }
            if (f + 8 < a.N) {
                if (r < a.R) put(a, yb, r, f + 8, v[mt][n][2]);
                if (r + 1 < a.R) put(a, yb, r + 1, f + 8, v[mt][n][3]);
            }
        }
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) w4_lane_gemm_kernel(const __grid_constant__ GemmArgs a) {
    constexpr int CB = chunk_bytes(G);
    constexpr int SWB = stage_w_bytes(G);

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sw = smem;
    uint8_t *sx = sw + kStages * SWB;
    float *red = reinterpret_cast<float *>(sx + kStages * kXStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(red + kBlocks * kWarpAccFloats);
    uint64_t *empty = full + kStages;

    const int u = blockIdx.y;
    const int nprob = a.n_problems ? *a.n_problems : 1;
    if (u >= nprob) return;
    const long long tot = (long long)a.T * a.Kc;
    const int vp = blockIdx.x;
    const long long i0 = (long long)vp * tot / a.Pv;
    const long long i1 = (long long)(vp + 1) * tot / a.Pv;
    if (i0 >= i1) return;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kStages * kXStageBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(sx)[i] = make_uint4(0u, 0u, 0u, 0u);  // rows >= R stay zero
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBlocks);
        }
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    __syncthreads();

    const int e = a.expert_ids ? a.expert_ids[u] : u;
    const uint8_t *wb = a.w + (long long)e * a.w_stride;
    const uint16_t *xb = a.x + (long long)u * a.x_stride;
    const int R = a.R;

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const uint32_t tx = SWB + R * 128;
            long long n_issued = 0;
            for (long long i = i0; i < i1; ++i) {
                const int it = int(i - i0);
                const int s = it % kStages;
                if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1)) {
                    set_error(a.err, 1);
                    break;
                }
                const int kc = int(i % a.Kc);
                mbar_arrive_expect_tx(&full[s], tx);
                bulk_g2s_hint(sw + s * SWB, wb + i * SWB, SWB, &full[s], pol);
                const uint16_t *xs = xb + kc * kKChunk;
                for (int r = 0; r < R; ++r)
                    bulk_g2s(sx + s * kXStageBytes + r * kXRowStride, xs + (long long)r * a.ldx, 128, &full[s]);
                ++n_issued;
            }
            // Leave only once every issued copy has landed (bounded).
            for (long long k = (n_issued > kStages ? n_issued - kStages : 0); k < n_issued; ++k)
                mbar_wait(&full[k % kStages], uint32_t(k / kStages) & 1);
        }
        return;
    }

    // ---------------- consumers ----------------
    const int kg = warp / kBlocks;
    const int b = warp % kBlocks;
    const int gq = lane >> 2, tq = lane & 3;
    const bool hi = R > 8;
    const int lrow = (lane & 7) + ((lane >> 4) << 3);
    const int lcol = (lane >> 3) & 1;
    const uint32_t sx_lane = smem_u32(sx) + lrow * kXRowStride + lcol * 16;
    const size_t ysz = a.mode == kSwiGluBf16 ? sizeof(__nv_bfloat16) : sizeof(float);
    void *yb = static_cast<char *>(a.y) + (long long)u * a.y_stride * (long long)ysz;
    float *rb = red + b * kWarpAccFloats;
    bool failed = false;

    long long i = i0;
    while (i < i1) {
        const int t = int(i / a.Kc);
        const long long seg_b = i;
        const long long seg_e = min(i1, (long long)(t + 1) * a.Kc);
        float acc[4][2][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][n][c] = 0.f;

        if (!failed) {
            for (long long j = seg_b; j < seg_e; ++j) {
                const int it = int(j - i0);
                if ((it & 1) != kg) continue;
                const int s = it % kStages;
                if (!mbar_wait(&full[s], uint32_t(it / kStages) & 1)) {
                    set_error(a.err, 1);
                    failed = true;
                    break;
                }
                consume_stage<G>(sw + s * SWB + b * CB, sx_lane + s * kXStageBytes, lane, gq, hi, acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        }

        // Combine the two k-parity groups in a fixed order (group 0 + group 1).
        named_bar_sync(1, kConsumerWarps * 32);
        if (kg == 1) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int n = 0; n < 2; ++n)
                    reinterpret_cast<float4 *>(rb)[(mt * 2 + n) * 32 + lane] =
                        make_float4(acc[mt][n][0], acc[mt][n][1], acc[mt][n][2], acc[mt][n][3]);
        }
        named_bar_sync(1, kConsumerWarps * 32);
        if (kg == 0) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const float4 o = reinterpret_cast<const float4 *>(rb)[(mt * 2 + n) * 32 + lane];
                    acc[mt][n][0] += o.x;
                    acc[mt][n][1] += o.y;
                    acc[mt][n][2] += o.z;
                    acc[mt][n][3] += o.w;
                }
            const long long tb = (long long)t * a.Kc;
            const long long te = tb + a.Kc;
            if (seg_b == tb && seg_e == te) {
                store_tile(a, yb, t, b, gq, tq, hi, acc);
            } else {
                // Stream-K partial: publish, count, and let the last arriver sum
                // every segment of this tile in k order.
                const int which = (t == int(i0 / a.Kc)) ? 0 : 1;
                float4 *slot = a.partials + ((((long long)u * a.Pv + vp) * 2 + which) * kBlocks + b) * 256;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        if (n == 1 && !hi) continue;
                        __stcg(slot + (mt * 2 + n) * 32 + lane,
                               make_float4(acc[mt][n][0], acc[mt][n][1], acc[mt][n][2], acc[mt][n][3]));
                    }
                __threadfence();
                __syncwarp();
                const int p_lo = int(((tb + 1) * a.Pv - 1) / tot);
                const int p_hi = int((te * a.Pv - 1) / tot);
                int nseg = 0;
                for (int p2 = p_lo; p2 <= p_hi; ++p2)
                    if ((long long)p2 * tot / a.Pv < (long long)(p2 + 1) * tot / a.Pv) ++nseg;
                unsigned *ctr = a.counters + ((long long)u * a.T + t) * kBlocks + b;
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(ctr, 1u);
                old = __shfl_sync(0xFFFFFFFFu, old, 0);
                if (old == unsigned(nseg - 1)) {
                    __threadfence();
                    float sum[4][2][4];
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                        for (int n = 0; n < 2; ++n)
#pragma unroll
                            for (int c = 0; c < 4; ++c) sum[mt][n][c] = 0.f;
                    for (int p2 = p_lo; p2 <= p_hi; ++p2) {
                        const long long r0 = (long long)p2 * tot / a.Pv;
                        const long long r1 = (long long)(p2 + 1) * tot / a.Pv;
                        if (r0 >= r1) continue;
                        const int which2 = (t == int(r0 / a.Kc)) ? 0 : 1;
                        const float4 *src =
                            a.partials + ((((long long)u * a.Pv + p2) * 2 + which2) * kBlocks + b) * 256;
#pragma unroll
                        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                            for (int n = 0; n < 2; ++n) {
                                if (n == 1 && !hi) continue;
                                const float4 v = __ldcg(src + (mt * 2 + n) * 32 + lane);
                                sum[mt][n][0] += v.x;
                                sum[mt][n][1] += v.y;
                                sum[mt][n][2] += v.z;
                                sum[mt][n][3] += v.w;
                            }
                    }
                    if (lane == 0) *ctr = 0u;  // leave the counter zero for the next launch
                    store_tile(a, yb, t, b, gq, tq, hi, sum);
                }
            }
        }
        i = seg_e;
    }
}

// ---- load-time repack: canonical [N][K/2] nibbles + [N][K/G] fp16 -> kernel layout
// Canonical row of packed feature p (interleave: gate/up pairs per 32 features).
__device__ __forceinline__ long long canonical_row(long long p, int N, bool inter) {
    if (!inter) return p < N ? p : -1;
    const int F = N / 2;
    const long long t = p / kTileN;
    const int w = int(p % kTileN);
    const int b = w / 64, mt = (w % 64) / 16, row = w % 16;
    const long long j = t * (kTileN / 2) + b * 32 + (mt >> 1) * 16 + row;
    if (j >= F) return -1;
    return (mt & 1) ? F + j : j;
}

template <int G>
__global__ void pack_codes_kernel(const uint8_t *codes, int K, int N, uint8_t *out, long long n_entries, int Kc,
                                  bool inter) {
    constexpr int CB = chunk_bytes(G);
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int lane = int(idx % 32);
    long long r = idx / 32;
    const int mt = int(r % 4);
    r /= 4;
    const int b = int(r % kBlocks);
    r /= kBlocks;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t words[4];
    for (int j = 0; j < 4; ++j) {
        uint32_t w = 0;
        for (int i = 0; i < 4; ++i)
            for (int h = 0; h < 2; ++h) {
                const long long f =
                    canonical_row(t * kTileN + b * 64 + mt * 16 + gq + ((i & 1) ? 8 : 0), N, inter);
                const int k = kc * kKChunk + j * 16 + 2 * tq + h + ((i & 2) ? 8 : 0);
                uint32_t nib = 0;  // code 0
                if (f >= 0) {
                    const uint8_t byte = codes[f * (K / 2) + k / 2];
                    nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
                }
                w |= ((nib ^ 8u) & 0xFu) << (4 * i + 16 * h);   // two's complement -> offset binary
            }
        words[j] = w;
    }
    uint8_t *dst = out + ((t * Kc + kc) * kBlocks + b) * (long long)CB + (mt * 32 + lane) * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

template <int G>
__global__ void pack_scales_kernel(const uint16_t *scales, int K, int N, uint8_t *out, long long n_entries, int Kc,
                                   bool inter) {
    constexpr int CB = chunk_bytes(G);
    constexpr int NG = kKChunk / G;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int mt = int(idx % 4);
    long long r = idx / 4;
    const int g = int(r % 8);
    r /= 8;
    const int grp = int(r % NG);
    r /= NG;
    const int b = int(r % kBlocks);
    r /= kBlocks;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const long long p = t * kTileN + b * 64 + mt * 16 + g;
    const long long f_lo = canonical_row(p, N, inter);
    const long long f_hi = canonical_row(p + 8, N, inter);
    const int gi = kc * NG + grp;
    const int ngroups = K / G;
    const uint32_t lo = f_lo >= 0 ? scales[f_lo * ngroups + gi] : 0u;
    const uint32_t hi = f_hi >= 0 ? scales[f_hi * ngroups + gi] : 0u;
    uint8_t *dst = out + ((t * Kc + kc) * kBlocks + b) * (long long)CB + 2048 + grp * 128 + g * 16 + mt * 4;
    *reinterpret_cast<uint32_t *>(dst) = lo | (hi << 16);
}

template <int G>
cudaError_t launch_gemm_g(const GemmArgs &a, int u_max, cudaStream_t s) {
    const size_t smem = gemm_smem_bytes(G);
    cudaError_t err = cudaFuncSetAttribute(w4_lane_gemm_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(smem));
    if (err != cudaSuccess) return err;
    dim3 grid(a.Pv, u_max);
    w4_lane_gemm_kernel<G><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_pack_g(const uint8_t *codes, const uint16_t *scales, int K, int N, void *packed, bool inter,
                          cudaStream_t s) {
    const int T = (N + kTileN - 1) / kTileN;
    const int Kc = K / kKChunk;
    const long long n_codes = (long long)T * Kc * kBlocks * 4 * 32;
    const long long n_scales = (long long)T * Kc * kBlocks * (kKChunk / G) * 8 * 4;
    const int th = 256;
    pack_codes_kernel<G><<<unsigned((n_codes + th - 1) / th), th, 0, s>>>(codes, K, N, (uint8_t *)packed, n_codes, Kc,
                                                                                        inter);
    pack_scales_kernel<G><<<unsigned((n_scales + th - 1) / th), th, 0, s>>>(scales, K, N, (uint8_t *)packed, n_scales,
                                                                           Kc, inter);
    return cudaGetLastError();
}

}  // namespace

size_t gemm_workspace_bytes(int K, int N, int G, int u_max, int Pv) {
    (void)K;
    (void)N;
    (void)G;
    return 256 + kCounterBytes + size_t(u_max) * size_t(Pv) * 2 * kSlotBytes;
}

void gemm_bind_workspace(GemmArgs &a, void *ws, int u_max) {
    (void)u_max;
    char *base = static_cast<char *>(ws);
    a.err = reinterpret_cast<int *>(base);
    a.counters = reinterpret_cast<unsigned *>(base + 256);
    a.partials = reinterpret_cast<float4 *>(base + 256 + kCounterBytes);
}

cudaError_t launch_w4_gemm(const GemmArgs &a, int u_max, cudaStream_t s) {
    return a.G == 64 ? launch_gemm_g<64>(a, u_max, s) : launch_gemm_g<32>(a, u_max, s);
}

cudaError_t launch_pack_w4(const uint8_t *codes, const uint16_t *scales, int K, int N, int G, void *packed,
                           bool interleave_gate_up, cudaStream_t s) {
    return G == 64 ? launch_pack_g<64>(codes, scales, K, N, packed, interleave_gate_up, s)
                   : launch_pack_g<32>(codes, scales, K, N, packed, interleave_gate_up, s);
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace tfk
