// W4 lane GEMM for the speculative-decoding verify pass (sm_103a, tcgen05).
//
// TensorFold README, "A row of a multi-row verify pass gets the same bits as a
// one-row step": up to 16 drafted rows share one launch that streams every
// 4-bit weight once, and row r's bits never depend on how many rows there are.
//
// One CTA per SM, 10 warps:
//   warp 0  producer: per pipeline stage (up to 4 consecutive 64-wide k slices
//           of one 256-feature tile, never crossing a tile boundary) lane 0
//           issues ONE bulk TMA copy of the packed weights (~35 KB, L2
//           evict-first) and ONE 4-D tensor TMA of the activation slices
//           ([16 rows][64 k] bf16 each, 128-byte swizzled, rows >= R
//           zero-filled by the copy engine's out-of-bounds fill).
//   warp 1  MMA issuer (lane 0) and TMEM owner.  For each slice and M-tile it
//           issues tcgen05.mma kind::f16, M=128 (weight rows), N=16 (verify
//           rows), K=16, A from tensor memory, B (activations) from shared
//           memory, fp32 accumulator in tensor memory.
//   warps 2-9  two warpgroups, one per 128-row M-tile.  Each thread owns one
//           weight row: it turns the row's 64 packed codes of a slice into
//           bf16 (16 + u, u = code + 8; exact) with one shift + LOP3 per pair, stores
//           them to tensor memory as the MMA's A operand, and later reads back
//           the group's fp32 partial sums (tcgen05.ld) and folds them in as
//           acc = fma(scale, partial, acc).
// Exactness: the A operand holds 16 + u; for every k step a second MMA adds
// (-24) x the same activations from a constant A block, so the tensor core
// accumulates  sum (16 + u - 24) x = sum code * x  of the group; every product
// is exact and the partial carries only the fp32 accumulation error (the bias
// of 24 is the smallest this OR-into-the-mantissa conversion allows: u sits in
// mantissa bits 3..6 under the implicit leading one of 16).
// Row invariance: rows are MMA columns (N = 16 for every R); the cut of the
// iteration space, the stage schedule and the fixed-order split-K sums depend
// on (T, Kc, Pv) only.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "tf_ptx.cuh"
#include "w4_gemm.cuh"

namespace tfk {

namespace {

constexpr uint32_t kNibMask = 0x00780078u;    // mantissa bits 3..6 of both bf16 halves
constexpr uint32_t kBf16Magic = 0x41804180u;  // (16, 16): u in mantissa bits 3..6 gives 16 + u
constexpr uint32_t kBf16Neg24x2 = 0xC1C0C1C0u;  // (-24, -24)
// tcgen05 instruction descriptor, kind::f16: D fp32, A bf16, B bf16, both
// K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(kRows) >> 3) << 17) |
                            ((uint32_t(kMTile) >> 4) << 24);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;        // A buffers: [mt][2] x 32 columns
constexpr uint32_t kColConst = 128;  // 8 columns of -24
constexpr uint32_t kColD = 160;      // D buffers: [mt][2*NG] x 16 columns

__device__ __forceinline__ float half_at(const uint8_t *p) {
    return __half2float(*reinterpret_cast<const __half *>(p));
}

// Shared-memory descriptor of a [16 rows][64 k] bf16 slice, K-major, 128-byte
// swizzle (8-row atoms of 1024 B), starting `koff` bytes into each row.
__device__ __forceinline__ uint64_t x_desc(uint32_t slice_smem, uint32_t koff) {
    const uint32_t start = (slice_smem + koff) >> 4;
    return uint64_t(start & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) |
           (uint64_t(2) << 61);
}

struct Sync {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t a_full[kMTiles][2];
    uint64_t a_free[kMTiles][2];
    uint64_t d_full[kMTiles][4];
    uint64_t d_free[kMTiles][4];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

// Bounded wait that gives up at once after any wait of this CTA timed out.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Sync *sy, int *err) {
    for (uint32_t i = 0; i < kSpinPolls; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *reinterpret_cast<volatile int *>(&sy->abort)) return false;
    }
    *reinterpret_cast<volatile int *>(&sy->abort) = 1;
    set_error(err, 1);
    return false;
}

// Iteration-space walker shared by every role so all agree on the schedule:
// segments end at tile boundaries, stages are runs of <= kStageIters
// iterations from the segment start.
struct Walk {
    long long gi;     // global iteration index (tile * Kc + kc)
    long long seg_b, seg_e;
    int pos;          // position inside the stage
    int st;           // stage counter
    int n_in_stage;
};

__device__ __forceinline__ void walk_begin(Walk &w, long long i0, long long i1, int Kc) {
    w.gi = i0;
    w.seg_b = i0;
    w.seg_e = min(i1, (i0 / Kc + 1) * (long long)Kc);
    w.pos = 0;
    w.st = 0;
    w.n_in_stage = int(min((long long)kStageIters, w.seg_e - w.seg_b));
}

__device__ __forceinline__ void walk_next(Walk &w, long long i1, int Kc) {
    ++w.gi;
    if (w.gi == w.seg_e) {
        w.seg_b = w.gi;
        w.seg_e = min(i1, (w.gi / Kc + 1) * (long long)Kc);
    }
    const int pos = int((w.gi - w.seg_b) % kStageIters);
    if (pos == 0) {
        ++w.st;
        w.n_in_stage = int(min((long long)kStageIters, w.seg_e - w.gi));
    }
    w.pos = pos;
}

__device__ __forceinline__ void dequant_slice(const uint4 &c0, const uint4 &c1, uint32_t (&v)[32]) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        // pair p (bits 4p / 16+4p) moves to mantissa bits 3..6 of each half
        v[4 * e + 0] = lop3_and_or(w[e] << 3, kNibMask, kBf16Magic);
#pragma unroll
        for (int p = 1; p < 4; ++p) v[4 * e + p] = lop3_and_or(w[e] >> (4 * p - 3), kNibMask, kBf16Magic);
    }
}

// Writes one thread's 16 results (its weight row, verify rows 0..15).
__device__ __forceinline__ void store_row(const GemmArgs &a, void *yb, int t, int mt, int quarter, int lane,
                                          const float (&v)[kRows]) {
    if (a.mode == kSwiGluBf16) {
        // lanes 0-15 hold gate rows, lanes 16-31 the matching up rows
        const int j = t * (kTileN / 2) + mt * (kMTile / 2) + quarter * 16 + (lane & 15);
        __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(yb);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float up = __shfl_down_sync(0xFFFFFFFFu, v[r], 16);
            if (lane < 16 && j < a.F && r < a.R) {
                const float g = v[r];
                h[(long long)r * a.ldy + j] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * up);
            }
        }
        return;
    }
    const int f = t * kTileN + mt * kMTile + quarter * 32 + lane;
    if (f >= a.N) return;
    float *y = static_cast<float *>(yb);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (r < a.R) {
            float *p = y + (long long)r * a.ldy + f;
            *p = a.mode == kAccumulateF32 ? *p + v[r] : v[r];
        }
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) w4_lane_gemm_kernel(const __grid_constant__ GemmArgs a) {
    constexpr int NG = kKChunk / G;   // quantisation groups per slice
    constexpr int KS = G / 16;        // k16 steps per group
    constexpr int MB = mtile_bytes(G);
    constexpr int CB = chunk_bytes(G);
    constexpr int STW = kStageIters * CB;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sx = smem;                                  // [kStages][kXStageBytes], 1024-B aligned
    uint8_t *sw = sx + kStages * kXStageBytes;           // [kStages][STW]
    Sync *sy = reinterpret_cast<Sync *>(sw + kStages * STW);

    const int u = blockIdx.y;
    const int nprob = a.n_problems ? *a.n_problems : 1;
    if (u >= nprob) return;
    const long long tot = (long long)a.T * a.Kc;
    const int vp = blockIdx.x;
    const long long i0 = (long long)vp * tot / a.Pv;
    const long long i1 = (long long)(vp + 1) * tot / a.Pv;
    if (i0 >= i1) return;
    const int n_it = int(i1 - i0);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sy->full[s], 1);
            mbar_init(&sy->empty[s], kDequantWarps + 1);
        }
        for (int m = 0; m < kMTiles; ++m) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&sy->a_full[m][b], 4);
                mbar_init(&sy->a_free[m][b], 1);
            }
            for (int b = 0; b < 4; ++b) {
                mbar_init(&sy->d_full[m][b], 1);
                mbar_init(&sy->d_free[m][b], 4);
            }
        }
        mbar_init(&sy->done, 1);
        sy->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sy->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sy->tmem_base;

    const int e = a.expert_ids ? a.expert_ids[u] : u;
    const uint8_t *wb = a.w + (long long)e * a.w_stride;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            Walk w;
            walk_begin(w, i0, i1, a.Kc);
            int issued = 0;
            for (int j = 0; j < n_it; ++j, walk_next(w, i1, a.Kc)) {
                if (w.pos != 0) continue;
                const int s = w.st % kStages;
                if (w.st >= kStages && !wait_bar(&sy->empty[s], uint32_t((w.st / kStages) - 1) & 1, sy, a.err))
                    break;
                mbar_arrive_expect_tx(&sy->full[s], uint32_t(w.n_in_stage * CB + kXStageBytes));
                bulk_g2s_hint(sw + s * STW, wb + w.gi * CB, uint32_t(w.n_in_stage * CB), &sy->full[s], pol);
                tma_load_4d(sx + s * kXStageBytes, &a.xmap, 0, 0, int(w.gi % a.Kc), a.x_per_problem ? u : 0,
                            &sy->full[s]);
                issued = w.st + 1;
            }
            // leave only once every issued copy has landed (bounded)
            for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
                wait_bar(&sy->full[k % kStages], uint32_t(k / kStages) & 1, sy, a.err);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            Walk w;
            walk_begin(w, i0, i1, a.Kc);
            bool ok = true;
            for (int j = 0; j < n_it && ok; ++j, walk_next(w, i1, a.Kc)) {
                const int s = w.st % kStages;
                if (w.pos == 0) ok = wait_bar(&sy->full[s], uint32_t(w.st / kStages) & 1, sy, a.err);
                const uint32_t slice = smem_u32(sx + s * kXStageBytes + w.pos * kXSliceBytes);
                for (int m = 0; m < kMTiles && ok; ++m) {
                    ok = wait_bar(&sy->a_full[m][j & 1], uint32_t(j >> 1) & 1, sy, a.err);
                    tc_fence_after();
                    const uint32_t acol = tbase + kColA + uint32_t(m * 2 + (j & 1)) * 32;
                    for (int g = 0; g < NG && ok; ++g) {
                        const int gi = j * NG + g;
                        const int db = gi % (2 * NG);
                        if (gi >= 2 * NG)
                            ok = wait_bar(&sy->d_free[m][db], uint32_t(gi / (2 * NG) - 1) & 1, sy, a.err);
                        tc_fence_after();
                        const uint32_t dcol = tbase + kColD + uint32_t(m * 2 * NG + db) * 16;
#pragma unroll
                        for (int kk = 0; kk < KS; ++kk) {
                            const int ks = g * KS + kk;
                            const uint64_t bd = x_desc(slice, uint32_t(ks) * 32);
                            umma_tmem_a(dcol, acol + uint32_t(ks) * 8, bd, kIdesc, kk > 0 ? 1u : 0u);
                            umma_tmem_a(dcol, tbase + kColConst, bd, kIdesc, 1u);
                        }
                        umma_commit(&sy->d_full[m][db]);
                    }
                    umma_commit(&sy->a_free[m][j & 1]);
                }
                if (w.pos == w.n_in_stage - 1) umma_commit(&sy->empty[s]);
            }
            // every MMA has completed before TMEM is released (bounded)
            umma_commit(&sy->done);
            wait_bar(&sy->done, 0, sy, a.err);
        }
    } else {
        // ---------------- dequant + epilogue warpgroups ----------------
        const int wid = warp - 2;                 // 0..7
        const int mt = wid / 4;                   // M-tile of this warpgroup
        const int quarter = warp & 3;             // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;      // weight row within the M-tile
        const uint32_t tl = uint32_t(quarter * 32) << 16;
        const size_t ysz = a.mode == kSwiGluBf16 ? sizeof(__nv_bfloat16) : sizeof(float);
        void *yb = static_cast<char *>(a.y) + (long long)u * a.y_stride * (long long)ysz;

        if (mt == 0) {  // the constant A block: -24 in every lane
            uint32_t cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) cv[i] = kBf16Neg24x2;
            tmem_st_x8(tbase + tl + kColConst, cv);
            tmem_wait_st();
        }

        float acc[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) acc[r] = 0.f;
        float sc_prev[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) sc_prev[g] = 0.f;
        long long prev_gi = -1, prev_seg_b = 0, prev_seg_e = 0;
        bool ok = true;

        // Reads back the group partials of iteration jj.
        auto readback = [&](int jj) {
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const int gi = jj * NG + g;
                const int db = gi % (2 * NG);
                if (ok) ok = wait_bar(&sy->d_full[mt][db], uint32_t(gi / (2 * NG)) & 1, sy, a.err);
                tc_fence_after();
                uint32_t d[16];
                tmem_ld_x16(tbase + tl + kColD + uint32_t(mt * 2 * NG + db) * 16, d);
                tmem_wait_ld();
#pragma unroll
                for (int r = 0; r < kRows; ++r) acc[r] = fmaf(sc_prev[g], __uint_as_float(d[r]), acc[r]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sy->d_free[mt][db]);
            }
        };

        // Publishes the segment ending with iteration gi_last.
        auto finish_segment = [&](long long gi_last, long long sb, long long se) {
            const int t = int(gi_last / a.Kc);
            const long long tb = (long long)t * a.Kc, te = tb + a.Kc;
            if (sb == tb && se == te) {
                store_row(a, yb, t, mt, quarter, lane, acc);
            } else {
                // stream-K partial: publish; the last arriver sums every
                // segment of this tile in ascending k order
                const int which = (t == int(i0 / a.Kc)) ? 0 : 1;
                float4 *slot = a.partials +
                               ((((long long)u * a.Pv + vp) * 2 + which) * kDequantWarps + wid) * 128 + lane * 4;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    __stcg(slot + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
                __threadfence();
                __syncwarp();
                const int p_lo = int(((tb + 1) * a.Pv - 1) / tot);
                const int p_hi = int((te * a.Pv - 1) / tot);
                int nseg = 0;
                for (int p2 = p_lo; p2 <= p_hi; ++p2)
                    if ((long long)p2 * tot / a.Pv < (long long)(p2 + 1) * tot / a.Pv) ++nseg;
                unsigned *ctr = a.counters + ((long long)u * a.T + t) * kDequantWarps + wid;
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(ctr, 1u);
                old = __shfl_sync(0xFFFFFFFFu, old, 0);
                if (old == unsigned(nseg - 1)) {
                    __threadfence();
                    float sum[kRows];
#pragma unroll
                    for (int r = 0; r < kRows; ++r) sum[r] = 0.f;
                    int p2 = p_lo;
                    while (p2 <= p_hi) {
                        // up to 4 segments' loads in flight, summed in k order
                        const float4 *src[4];
                        int ns = 0;
                        while (ns < 4 && p2 <= p_hi) {
                            const long long r0 = (long long)p2 * tot / a.Pv;
                            const long long r1 = (long long)(p2 + 1) * tot / a.Pv;
                            if (r0 < r1) {
                                const int w2 = (t == int(r0 / a.Kc)) ? 0 : 1;
                                src[ns++] = a.partials +
                                            ((((long long)u * a.Pv + p2) * 2 + w2) * kDequantWarps + wid) * 128 +
                                            lane * 4;
                            }
                            ++p2;
                        }
                        float4 v[4][4];
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                v[s2][q] = s2 < ns ? __ldcg(src[s2] + q) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) {
                            if (s2 >= ns) continue;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                sum[4 * q] += v[s2][q].x;
                                sum[4 * q + 1] += v[s2][q].y;
                                sum[4 * q + 2] += v[s2][q].z;
                                sum[4 * q + 3] += v[s2][q].w;
                            }
                        }
                    }
                    if (lane == 0) *ctr = 0u;  // leave the counter zero for the next launch
                    store_row(a, yb, t, mt, quarter, lane, sum);
                }
            }
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r] = 0.f;
        };

        Walk w;
        walk_begin(w, i0, i1, a.Kc);
        for (int j = 0; j < n_it; ++j, walk_next(w, i1, a.Kc)) {
            const int s = w.st % kStages;
            if (w.pos == 0 && ok) ok = wait_bar(&sy->full[s], uint32_t(w.st / kStages) & 1, sy, a.err);
            const uint8_t *blk = sw + s * STW + w.pos * CB + mt * MB;
            const uint4 c0 = *reinterpret_cast<const uint4 *>(blk + row * 16);
            const uint4 c1 = *reinterpret_cast<const uint4 *>(blk + 2048 + row * 16);
            float sc[NG];
#pragma unroll
            for (int g = 0; g < NG; ++g) sc[g] = half_at(blk + 4096 + (row * NG + g) * 2);
            __syncwarp();
            if (w.pos == w.n_in_stage - 1 && lane == 0) mbar_arrive(&sy->empty[s]);
            uint32_t v[32];
            dequant_slice(c0, c1, v);
            if (j >= 2 && ok) ok = wait_bar(&sy->a_free[mt][j & 1], uint32_t((j >> 1) - 1) & 1, sy, a.err);
            tc_fence_after();
            tmem_st_x32(tbase + tl + kColA + uint32_t(mt * 2 + (j & 1)) * 32, v);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sy->a_full[mt][j & 1]);
            // software pipeline: fold in the previous slice while this one multiplies
            if (j > 0) {
                readback(j - 1);
                if (prev_gi + 1 == prev_seg_e) finish_segment(prev_gi, prev_seg_b, prev_seg_e);
            }
#pragma unroll
            for (int g = 0; g < NG; ++g) sc_prev[g] = sc[g];
            prev_gi = w.gi;
            prev_seg_b = w.seg_b;
            prev_seg_e = w.seg_e;
        }
        readback(n_it - 1);
        finish_segment(prev_gi, prev_seg_b, prev_seg_e);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ---- load-time repack: canonical [N][K/2] nibbles + [N][K/G] fp16 -> kernel layout
// Canonical row of packed feature p (interleave: per 32-row warp slice, 16 gate
// rows then the 16 matching up rows).
__device__ __forceinline__ long long canonical_row(long long p, int N, bool inter) {
    if (!inter) return p < N ? p : -1;
    const int F = N / 2;
    const long long t = p / kTileN;
    const int wtile = int(p % kTileN);
    const int mt = wtile / kMTile, row = wtile % kMTile;
    const int quarter = row / 32, lane = row % 32;
    const long long j = t * (kTileN / 2) + mt * (kMTile / 2) + quarter * 16 + (lane & 15);
    if (j >= F) return -1;
    return lane < 16 ? j : F + j;
}

template <int G>
__global__ void pack_codes_kernel(const uint8_t *codes, int K, int N, uint8_t *out, long long n_entries, int Kc,
                                  bool inter) {
    constexpr int MB = mtile_bytes(G);
    constexpr int CB = chunk_bytes(G);
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int row = int(idx % kMTile);
    long long r = idx / kMTile;
    const int half = int(r % 2);
    r /= 2;
    const int mt = int(r % kMTiles);
    r /= kMTiles;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const long long f = canonical_row(t * kTileN + mt * kMTile + row, N, inter);
    uint32_t words[4];
    for (int e = 0; e < 4; ++e) {
        uint32_t w = 0;
        for (int q = 0; q < 8; ++q) {
            const int k = kc * kKChunk + half * 32 + e * 8 + q;
            uint32_t nib = 0;  // code 0
            if (f >= 0) {
                const uint8_t byte = codes[f * (K / 2) + k / 2];
                nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
            }
            w |= ((nib ^ 8u) & 0xFu) << (4 * (q / 2) + 16 * (q % 2));   // two's complement -> offset binary
        }
        words[e] = w;
    }
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + mt * MB + half * 2048 + row * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

template <int G>
__global__ void pack_scales_kernel(const uint16_t *scales, int K, int N, uint8_t *out, long long n_entries, int Kc,
                                   bool inter) {
    constexpr int MB = mtile_bytes(G);
    constexpr int CB = chunk_bytes(G);
    constexpr int NG = kKChunk / G;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int g = int(idx % NG);
    long long r = idx / NG;
    const int row = int(r % kMTile);
    r /= kMTile;
    const int mt = int(r % kMTiles);
    r /= kMTiles;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const long long f = canonical_row(t * kTileN + mt * kMTile + row, N, inter);
    const int ngroups = K / G;
    const uint16_t v = f >= 0 ? scales[f * ngroups + kc * NG + g] : uint16_t(0);
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + mt * MB + 4096 + (row * NG + g) * 2;
    *reinterpret_cast<uint16_t *>(dst) = v;
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
    const long long n_codes = (long long)T * Kc * kMTiles * 2 * kMTile;
    const long long n_scales = (long long)T * Kc * kMTiles * kMTile * (kKChunk / G);
    const int th = 256;
    pack_codes_kernel<G><<<unsigned((n_codes + th - 1) / th), th, 0, s>>>(codes, K, N, (uint8_t *)packed, n_codes,
                                                                        Kc, inter);
    pack_scales_kernel<G><<<unsigned((n_scales + th - 1) / th), th, 0, s>>>(scales, K, N, (uint8_t *)packed,
                                                                          n_scales, Kc, inter);
    return cudaGetLastError();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
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

bool gemm_encode_x(GemmArgs &a, const uint16_t *x, int ldx, long long x_stride, int u_max, const char **why) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) {
        *why = "cuTensorMapEncodeTiled is unavailable";
        return false;
    }
    const bool per = x_stride != 0 && u_max > 1;
    // dims (innermost first): k within a 64-wide slice, row, slice, problem
    cuuint64_t dims[4] = {cuuint64_t(kKChunk), cuuint64_t(a.R), cuuint64_t(a.Kc), cuuint64_t(per ? u_max : 1)};
    cuuint64_t strides[3] = {cuuint64_t(ldx) * 2, cuuint64_t(kKChunk) * 2,
                             per ? cuuint64_t(x_stride) * 2 : cuuint64_t(ldx) * 2 * cuuint64_t(a.R)};
    cuuint32_t box[4] = {cuuint32_t(kKChunk), cuuint32_t(kRows), cuuint32_t(kStageIters), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(&a.xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(x), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    a.x_per_problem = per ? 1 : 0;
    if (r != CUDA_SUCCESS) {
        *why = "cuTensorMapEncodeTiled rejected the activation layout";
        return false;
    }
    return true;
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
