// W4 lane GEMM for the speculative-decoding verify pass (sm_103a).
//
// TensorFold README, section on the two guarantees (row invariance): up to 16
// drafted rows share one launch that streams every 4-bit weight once, and row
// r's bits never depend on how many rows there are.
//
// At most one CTA per SM, 17 warps, persistent over work items (problem,
// range of the tile x k-slice iteration space):
//   warp 16 producer: per pipeline stage (up to 8 consecutive 64-wide k slices
//           of one 128-feature tile, never crossing a tile boundary) one lane
//           issues ONE bulk TMA copy of the packed weights (~35 KB, L2
//           evict-first; the bulk engine only reaches HBM rate with copies of
//           this size) and ONE 4-D tensor TMA of the activation slices
//           ([8 or 16 rows][64 k] bf16 each, 128-byte swizzled, rows >= R
//           zero-filled by the copy engine's out-of-bounds fill).
//   warps 0-15 consumers: warp (kg, fw) owns the 32 weight rows of feature
//           block fw and every fourth k slice (k-group kg).  Per 16-wide k step
//           it turns one packed 32-bit word per 16-row sub-tile into the
//           m16n8k16 A fragment (shift + LOP3 + bf16x2 FMA per register: exact
//           integer codes -8..7), loads the activation B fragment with a
//           swizzle-aware ldmatrix and issues one mma.sync per 8 rows.  Each
//           quantisation group's partial is formed in a fresh fp32 fragment and
//           folded in as acc = fma(scale, partial, acc).  At the end of a
//           whole tile the four k-groups of a feature block trade partial sums
//           through shared memory (one named barrier) and each adds and stores
//           one quarter of the block; a split tile's sums go to k-group 0,
//           which runs the split-K fixup.
// The grid signals its dependents at once (programmatic dependent launch): the
// next launch in the stream lands on every SM this one frees and requests its
// first weight stages before it waits for this grid to finish.
// Why mma.sync and not tcgen05: the verify pass multiplies a weight tile by at
// most 16 rows.  Measured on sm_103a, a tcgen05.mma of M = 128, K = 16 costs
// ~46 cycles at any N up to 32 (44 weights per cycle per SM, the rate HBM
// delivers at peak, with no room for the rest), while mma.sync.m16n8k16 runs
// at 0.5 per cycle per SM: 127 weights per cycle per SM at R <= 8, 63 at
// R = 16.  Per 256 weights a consumer warp issues about 18 instructions of
// which the MMA is one (R <= 8) or two (R > 8); the rest turn the 4-bit codes
// into exact bf16 operands and apply the group scales, work either path needs.
// Row invariance: rows are MMA columns (a column's result depends only on its
// own activations; the rows 8..15 MMA is skipped when R <= 8), and the cut of
// the iteration space, the stage schedule, the k-group split, the fixed-order
// k-group combine and the fixed-order split-K sums depend on (T, Kc, Pv) only.
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "tf_keys.cuh"
#include "tf_ptx.cuh"
#include "w4_gemm.cuh"

namespace tfk {

namespace {

constexpr uint32_t kBf16One2 = 0x3F803F80u;     // (1.0, 1.0)
constexpr uint32_t kBf16Neg136x2 = 0xC308C308u; // (-136, -136): symmetric codes c = u - 8
constexpr uint32_t kBf16Neg128x2 = 0xC300C300u; // (-128, -128): affine codes q = u
constexpr uint32_t kNibMask = 0x000F000Fu;
constexpr uint32_t kBf16Magic = 0x43004300u;    // (128, 128): OR-ing u in gives 128 + u

__device__ __forceinline__ uint32_t word_of(const uint4 &q, int j) {
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
}

struct Sync {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort;
};

// Bounded wait: non-suspending polls for short hand-offs, then try_wait; gives
// up at once after any wait of this CTA timed out.
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

// Balanced split of a problem's tot = T * Kc iterations into Pv contiguous
// ranges: the first rem ranges hold q + 1 iterations, the others q
// (q = tot / Pv, rem = tot % Pv, Pv <= tot).  Range p starts at p*q + min(p, rem).
struct Split {
    unsigned q, rem;
    __device__ __forceinline__ unsigned start(unsigned p) const { return p * q + (p < rem ? p : rem); }
    __device__ __forceinline__ unsigned owner(unsigned i) const {
        const unsigned big = rem * (q + 1);
        return i < big ? i / (q + 1) : rem + (i - big) / q;
    }
};

// bf16 pair -> two floats (low half, high half).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// One 64-wide k slice of one 32-row feature block for this warp.  HI: the
// launch has more than 8 rows (a second n8 MMA per sub-tile); rows 0..7 run the
// identical instruction sequence in both instantiations.  AFF: MLX-style affine
// weights (unsigned codes, bf16 scale and bias per group): the group's partial
// sum_k q x is scaled and the bias is added times the group's activation sum,
// which one extra MMA per k step with an all-ones A operand delivers in the
// accumulator layout.
template <int G, bool HI, bool AFF>
__device__ __forceinline__ void consume_slice(const uint8_t *blk, uint32_t xslice, int lane, int gq,
                                              const uint32_t (&xoff)[4], float (&acc)[2][2][4]) {
    constexpr int NG = kKChunk / G;
    constexpr int KS = G / 16;
    constexpr uint32_t kOffset = AFF ? kBf16Neg128x2 : kBf16Neg136x2;
    constexpr int kGroupBytes = AFF ? 128 : 64;
    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + lane * 16);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 512 + lane * 16);
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
        const uint2 sv = *reinterpret_cast<const uint2 *>(blk + 1024 + grp * kGroupBytes + gq * 8);
        float part[2][2][4];
        float xs[2][4];   // AFF: group activation sums (element c: verify row 2q + (c & 1))
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const int j = grp * KS + kk;
            const uint32_t xa = xslice + xoff[j];
            uint32_t b0, b1, b2 = 0, b3 = 0;
            if (HI)
                ldsm_x4(xa, b0, b1, b2, b3);
            else
                ldsm_x2(xa, b0, b1);
            if (AFF) {
                const uint32_t ones[4] = {kBf16One2, kBf16One2, kBf16One2, kBf16One2};
                if (kk == 0) {
                    mma_bf16_16816_zero(xs[0], ones, b0, b1);
                    if (HI) mma_bf16_16816_zero(xs[1], ones, b2, b3);
                } else {
                    mma_bf16_16816(xs[0], ones, b0, b1);
                    if (HI) mma_bf16_16816(xs[1], ones, b2, b3);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint32_t w = word_of(mt ? q1 : q0, j);
                uint32_t af[4];
                af[0] = fma_bf16x2(lop3_and_or(w, kNibMask, kBf16Magic), kBf16One2, kOffset);
                af[1] = fma_bf16x2(lop3_and_or(w >> 4, kNibMask, kBf16Magic), kBf16One2, kOffset);
                af[2] = fma_bf16x2(lop3_and_or(w >> 8, kNibMask, kBf16Magic), kBf16One2, kOffset);
                af[3] = fma_bf16x2(lop3_and_or(w >> 12, kNibMask, kBf16Magic), kBf16One2, kOffset);
                if (kk == 0) {
                    mma_bf16_16816_zero(part[mt][0], af, b0, b1);
                    if (HI) mma_bf16_16816_zero(part[mt][1], af, b2, b3);
                } else {
                    mma_bf16_16816(part[mt][0], af, b0, b1);
                    if (HI) mma_bf16_16816(part[mt][1], af, b2, b3);
                }
            }
        }
        uint2 bv = make_uint2(0, 0);
        if (AFF) bv = *reinterpret_cast<const uint2 *>(blk + 1024 + grp * kGroupBytes + 64 + gq * 8);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            // sc.x: row mt*16 + g, sc.y: row mt*16 + g + 8
            const float2 sc = AFF ? bf16x2_to_float2(mt ? sv.y : sv.x)
                                  : __half22float2(*reinterpret_cast<const __half2 *>(mt ? &sv.y : &sv.x));
#pragma unroll
            for (int n = 0; n < (HI ? 2 : 1); ++n) {
                acc[mt][n][0] = fmaf(sc.x, part[mt][n][0], acc[mt][n][0]);
                acc[mt][n][1] = fmaf(sc.x, part[mt][n][1], acc[mt][n][1]);
                acc[mt][n][2] = fmaf(sc.y, part[mt][n][2], acc[mt][n][2]);
                acc[mt][n][3] = fmaf(sc.y, part[mt][n][3], acc[mt][n][3]);
            }
            if (AFF) {
                const float2 bi = bf16x2_to_float2(mt ? bv.y : bv.x);
#pragma unroll
                for (int n = 0; n < (HI ? 2 : 1); ++n) {
                    acc[mt][n][0] = fmaf(bi.x, xs[n][0], acc[mt][n][0]);
                    acc[mt][n][1] = fmaf(bi.x, xs[n][1], acc[mt][n][1]);
                    acc[mt][n][2] = fmaf(bi.y, xs[n][2], acc[mt][n][2]);
                    acc[mt][n][3] = fmaf(bi.y, xs[n][3], acc[mt][n][3]);
                }
            }
        }
    }
}

// NVFP4 helpers.  e2m1x2 / e4m3x2: the low nibble (byte) goes to the low
// fp16 half, the high one to the high half.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&a)[4]) {
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\tmov.b32 {t0, t1, t2, t3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t0;\n\tcvt.rn.f16x2.e2m1x2 %1, t1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, t2;\n\tcvt.rn.f16x2.e2m1x2 %3, t3;\n\t}"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
        : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t s16) {
    uint32_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(d) : "r"(s16));
    return d;
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// bf16 pair -> fp16 pair (exact within the fp16 range; larger values overflow to inf)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t b) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(__uint_as_float(b & 0xFFFF0000u)), "f"(__uint_as_float(b << 16)));
    return d;
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 64-wide k slice of NVFP4 weights for this warp's 32-row feature block.
// Each 16-wide k step is one scale block: the E2M1 codes become exact fp16
// values and are multiplied by their rows' E4M3 block scales (the product has
// at most 6 significant bits and stays a normal fp16: exact), so the MMA adds
// sum_k w x straight into the fp32 accumulator; the tensor scale is applied
// once at the store.  Activations are taken to fp16 (exact within its range).
// Rows 0..7 run the identical instruction sequence whatever R is.
template <bool HI>
__device__ __forceinline__ void consume_slice_nvfp4(const uint8_t *blk, uint32_t xslice, int lane, int gq,
                                                    const uint32_t (&xoff)[4], float (&acc)[2][2][4]) {
    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + lane * 16);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 512 + lane * 16);
    const uint4 sc = *reinterpret_cast<const uint4 *>(blk + 1024 + gq * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t xa = xslice + xoff[j];
        uint32_t b0, b1, b2 = 0, b3 = 0;
        if (HI)
            ldsm_x4(xa, b0, b1, b2, b3);
        else
            ldsm_x2(xa, b0, b1);
        b0 = bf16x2_to_f16x2(b0);
        b1 = bf16x2_to_f16x2(b1);
        if (HI) {
            b2 = bf16x2_to_f16x2(b2);
            b3 = bf16x2_to_f16x2(b3);
        }
        const uint32_t sw = word_of(sc, j);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const uint32_t s2 = e4m3x2_to_f16x2(mt ? (sw >> 16) : (sw & 0xFFFFu));   // (s[row g], s[row g+8])
            const uint32_t sg = __byte_perm(s2, 0, 0x1010), sg8 = __byte_perm(s2, 0, 0x3232);
            uint32_t af[4];
            e2m1x8_to_f16x2(word_of(mt ? q1 : q0, j), af);
            af[0] = mul_f16x2(af[0], sg);
            af[1] = mul_f16x2(af[1], sg8);
            af[2] = mul_f16x2(af[2], sg);
            af[3] = mul_f16x2(af[3], sg8);
            mma_f16_16816(acc[mt][0], af, b0, b1);
            if (HI) mma_f16_16816(acc[mt][1], af, b2, b3);
        }
    }
}

template <bool NV>
__device__ __forceinline__ void put(const GemmArgs &a, void *yb, int r, int f, float v) {
    if (NV) v *= a.gscale;   // the NVFP4 tensor scale, once per output
    float *y = static_cast<float *>(yb) + (long long)r * a.ldy + f;
    if (a.mode == kAccumulateF32)
        *y = *y + v;
    else
        *y = v;
}

// Stores a lane's 16 results: element (mt, n, c) is weight row mt*16 + g (+8
// for c >= 2) of the feature block and verify row n*8 + 2q + (c & 1).
template <bool NV>
__device__ __forceinline__ void store_block(const GemmArgs &a, void *yb, int t, int fw, int gq, int tq, bool hi,
                                            const float (&v)[2][2][4]) {
    if (a.mode == kSwiGluBf16) {
        // sub-tile 0 holds gate rows, sub-tile 1 the matching up rows; silu
        // through the fast exponential and divide (relative error ~1e-6, far
        // inside the bf16 rounding of h)
        __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(yb);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (n == 1 && !hi) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = t * (kTileN / 2) + fw * 16 + gq + (c >= 2 ? 8 : 0);
                const int r = n * 8 + tq * 2 + (c & 1);
                if (j < a.F && r < a.R) {
                    const float g = v[0][n][c];
                    const float up = v[1][n][c];
                    h[(long long)r * a.ldy + j] = __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * up);
                }
            }
        }
        return;
    }
    const int f0 = t * kTileN + fw * kBlockRows;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (n == 1 && !hi) continue;
            const int f = f0 + mt * 16 + gq;
            const int r = n * 8 + tq * 2;
            if (f < a.N) {
                if (r < a.R) put<NV>(a, yb, r, f, v[mt][n][0]);
                if (r + 1 < a.R) put<NV>(a, yb, r + 1, f, v[mt][n][1]);
            }
            if (f + 8 < a.N) {
                if (r < a.R) put<NV>(a, yb, r, f + 8, v[mt][n][2]);
                if (r + 1 < a.R) put<NV>(a, yb, r + 1, f + 8, v[mt][n][3]);
            }
        }
    }
}

// Stores k-group q's quarter of a lane's results after the whole-tile combine:
// v[mt][n] is element (mt, n, q) of the block, i.e. weight row mt*16 + g (+8
// when q >= 2) of the feature block and verify row n*8 + 2tq + (q & 1).  The
// arithmetic per output is store_block's.
template <bool NV>
__device__ __forceinline__ void store_quarter(const GemmArgs &a, void *yb, int t, int fw, int gq, int tq, int q,
                                              bool hi, const float (&v)[2][2]) {
    const int r0 = tq * 2 + (q & 1);
    if (a.mode == kSwiGluBf16) {
        __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(yb);
        const int j = t * (kTileN / 2) + fw * 16 + gq + (q >= 2 ? 8 : 0);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (n == 1 && !hi) continue;
            const int r = n * 8 + r0;
            if (j < a.F && r < a.R) {
                const float g = v[0][n];
                const float up = v[1][n];
                h[(long long)r * a.ldy + j] = __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * up);
            }
        }
        return;
    }
    const int fb = t * kTileN + fw * kBlockRows + gq + (q >= 2 ? 8 : 0);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (n == 1 && !hi) continue;
            const int f = fb + mt * 16, r = n * 8 + r0;
            if (f < a.N && r < a.R) put<NV>(a, yb, r, f, v[mt][n]);
        }
    }
}

// Shared-memory view of the candidate epilogue (selector launches only).
template <bool HI>
struct SelView {
    static constexpr int SR = x_rows(HI);
    float *ring;          // [kSelSlots][SR][kSelStride]
    int *f0;              // [kSelSlots]: first feature of the block, -1 = the sender's last
    int *tail;            // tickets handed out
    uint64_t *full;       // [kSelSlots]
    uint64_t *empty;      // [kSelSlots]: one arrival per selector warp
    uint64_t *lists;      // [SR][kSelList], descending, 0-padded
    uint64_t *pend;       // [SR][32]: words above the list's k'-th best, not yet merged
    int *npend;           // [SR]
    __device__ SelView(uint8_t *base) {
        ring = reinterpret_cast<float *>(base);
        f0 = reinterpret_cast<int *>(base + sel_ring_bytes(HI));
        tail = f0 + kSelSlots;
        full = reinterpret_cast<uint64_t *>(base + sel_ring_bytes(HI) + 256);
        empty = full + kSelSlots;
        lists = empty + kSelSlots;
        pend = lists + SR * kSelList;
        npend = reinterpret_cast<int *>(pend + SR * 32);
    }
};

// Merges row r's pending words into its list.
__device__ __forceinline__ void sel_flush(uint64_t *L, uint64_t *P, int *np, int lane) {
    const int n = *np;
    if (n == 0) return;
    warp_merge_rank(L, P, n);
    if (lane == 0) *np = 0;
    __syncwarp();
}

// A selector warp: takes the blocks the storing warps hand over, in ticket
// order, and for each of its rows (r % kSelWarps == sw) queues the words above
// the row's current k'-th best; a full queue is merged into the row's list
// (each word placed by its rank in the merged order).  Once every storing
// warp has sent its last block it merges what is queued and writes the lists.
// The kept set of a CTA is exact (its sel_k best over the blocks it stored),
// whatever the arrival order.  Waits poll with short sleeps (a suspended warp
// wakes late; a polling one takes few issue slots from the consumers) and
// give up after kWaitLimit polls.
template <bool HI>
__device__ void run_selector(const GemmArgs &a, SelView<HI> v, Sync *sy, int sw) {
    constexpr int SR = SelView<HI>::SR;
    const int lane = threadIdx.x & 31;
    const int kk = a.sel_k;
    for (int r = sw; r < SR; r += kSelWarps) {
        for (int i = lane; i < kSelList; i += 32) v.lists[r * kSelList + i] = 0ull;
        if (lane == 0) v.npend[r] = 0;
    }
    __syncwarp();
    unsigned bad = 0;
    const unsigned lt = (1u << lane) - 1u;
    constexpr int RW = (SR + kSelWarps - 1) / kSelWarps;   // rows of this warp
    uint64_t gb[RW];   // the shared bound of each row, as read during the previous block
#pragma unroll
    for (int q = 0; q < RW; ++q) gb[q] = 0ull;
    bool timed_out = false;
    for (int t = 0, done = 0; done < kFeatWarps && !timed_out; ++t) {
        const int slot = t % kSelSlots;
        const uint32_t par = uint32_t(t / kSelSlots) & 1u;
        for (uint32_t i = 0;; ++i) {
            if (__all_sync(0xFFFFFFFFu, mbar_test_wait(&v.full[slot], par))) break;
            __nanosleep(128);
            if (i >= kWaitLimit || ((i & 1023u) == 1023u && *reinterpret_cast<volatile int *>(&sy->abort))) {
                *reinterpret_cast<volatile int *>(&sy->abort) = 1;
                set_error(a.err, 1);
                timed_out = true;
                break;
            }
        }
        if (timed_out) break;
        const int f0 = v.f0[slot];
        if (f0 < 0) {
            ++done;
        } else {
            const float *src = v.ring + slot * SR * kSelStride;
            const int fi = f0 + lane;
            const bool fv = fi < a.N;
            // this warp's rows: every value and every threshold first (the row's
            // own k'-th best, or the shared bound if higher); the shared bounds
            // for the next block are requested now and arrive meanwhile
            float xv[RW];
            uint64_t th[RW], gn[RW];
#pragma unroll
            for (int q = 0; q < RW; ++q) {
                const int r = sw + q * kSelWarps;
                xv[q] = r < a.R ? src[r * kSelStride + lane] : 0.f;
                const uint64_t own = r < a.R ? v.lists[r * kSelList + kk - 1] : 0ull;
                th[q] = own > gb[q] ? own : gb[q];
                gn[q] = r < a.R ? __ldcg(&a.sel_bound[r]) : 0ull;
            }
#pragma unroll
            for (int q = 0; q < RW; ++q) {
                const int r = sw + q * kSelWarps;
                if (r >= a.R) break;
                const float x = xv[q];
                if (__any_sync(0xFFFFFFFFu, fv && !isfinite(x))) bad |= 1u << r;
                const uint64_t key = fv ? composite(order_key(x), fi) : 0ull;
                uint64_t *L = v.lists + r * kSelList;
                uint64_t *P = v.pend + r * 32;
                bool s = key > th[q];
                unsigned m = __ballot_sync(0xFFFFFFFFu, s);
                if (!m) continue;
                int np = v.npend[r];
                if (np + __popc(m) > 32) {   // queue full: merge it, publish, then re-test against the new k'-th best
                    sel_flush(L, P, &v.npend[r], lane);
                    const uint64_t own = L[kk - 1];
                    if (lane == 0 && own) atomicMax(reinterpret_cast<unsigned long long *>(&a.sel_bound[r]),
                                                    (unsigned long long)own);
                    np = 0;
                    th[q] = own > th[q] ? own : th[q];
                    s = key > th[q];
                    m = __ballot_sync(0xFFFFFFFFu, s);
                }
                if (s) P[np + __popc(m & lt)] = key;
                __syncwarp();
                if (lane == 0) v.npend[r] = np + __popc(m);
                __syncwarp();
            }
#pragma unroll
            for (int q = 0; q < RW; ++q) gb[q] = gn[q];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&v.empty[slot]);
    }
    const long long c = blockIdx.x;
    for (int r = sw; r < a.R; r += kSelWarps) {
        uint64_t *L = v.lists + r * kSelList;
        sel_flush(L, v.pend + r * 32, &v.npend[r], lane);
        const long long slot = r * (long long)a.sel_nc + c;
        for (int i = lane; i < kk; i += 32) {
            const uint64_t w = L[i];
            a.sel_val[slot * kSelList + i] = w ? key_value(uint32_t(w >> 32)) : __uint_as_float(0xFFFFFFFFu);
            a.sel_id[slot * kSelList + i] = w ? composite_id(w) : -1;
        }
        if (lane == 0) {
            a.sel_cnt[slot] = kk;
            a.sel_kth[slot] = L[kk - 1];
            if ((bad >> r) & 1u) {
                atomicOr(&a.sel_bad[r], 1);
                set_error(a.err, 2);
            }
        }
    }
}

template <int G, bool HI, int FMT, bool SEL = false>
__global__ void __launch_bounds__(SEL ? kThreads + 32 * kSelWarps : kThreads, 1)
    w4_lane_gemm_kernel(const __grid_constant__ GemmArgs a) {
    constexpr bool AFF = FMT == kFmtAffine;
    constexpr int BB = block_bytes(G, FMT);
    constexpr int CB = chunk_bytes(G, FMT);
    constexpr int STW = kStageIters * CB;
    constexpr int NS = num_stages(G, HI, FMT);
    constexpr int XSL = x_slice_bytes(HI);
    constexpr int XST = x_stage_bytes(HI);
    constexpr int NQ = lane_vals(HI) / 4;   // float4 per lane in the combine and the fixup

    extern __shared__ uint8_t smem_raw[];
    // 1024-B aligned start, derived by pointer arithmetic so that the compiler
    // keeps every access below in the shared state space
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sx = smem;                                  // [NS][XST], 1024-B aligned
    uint8_t *sw = sx + NS * XST;                         // [NS][STW]
    constexpr int CBF = comb_buf_floats(HI);
    static_assert(2 * 32 * 4 * NQ <= CBF / kFeatWarps, "the split-tile combine must fit in a feature block's part");
    float *red = reinterpret_cast<float *>(sw + NS * STW);   // [2][CBF]: the k-group combine buffers
    Sync *sy = reinterpret_cast<Sync *>(red + 2 * CBF);
    uint8_t *selb = reinterpret_cast<uint8_t *>(sy) + 256;   // SEL: SelView<HI> region

    // Work items are (problem u, range vp) pairs, u-major; CTA b takes items
    // b, b + gridDim.x, ...  A grouped launch whose problem list comes from the
    // preceding grid waits for it here; one whose list was complete before the
    // preceding grid started (list_ready) reads it at once and, like a dense
    // launch, streams its first weight stages while that grid finishes.
    if ((a.n_problems || a.expert_ids) && !a.list_ready) grid_dependency_wait();
    const int nprob = a.n_problems ? *a.n_problems : 1;
    const int n_items = nprob * a.Pv;
    if (int(blockIdx.x) >= n_items) return;
    const unsigned tot = unsigned(a.T) * unsigned(a.Kc);
    const Split split{tot / unsigned(a.Pv), tot % unsigned(a.Pv)};   // Pv <= tot: no empty range
    const unsigned Kc = unsigned(a.Kc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sy->full[s], 1);
            mbar_init(&sy->empty[s], kConsumerWarps);
        }
        sy->abort = 0;
        if constexpr (SEL) {
            SelView<HI> v(selb);
            for (int i = 0; i < kSelSlots; ++i) {
                mbar_init(&v.full[i], 1);
                mbar_init(&v.empty[i], kSelWarps);
            }
            *v.tail = 0;
        }
        fence_mbar_init();
    }
    __syncthreads();
    // The next grid in the stream may start now: its CTAs land on every SM this
    // grid frees and stream their first weight stages while it finishes.  It
    // reads nothing this grid writes before its own grid_dependency_wait().
    grid_launch_dependents();

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            // Weights are read-only model data: the first NP stages are
            // requested before waiting for the preceding grid (programmatic
            // dependent launch), their activation slices only after it.  Two,
            // not the whole ring: the copies of CTAs that land early compete
            // with the preceding grid's last L2 round trips (its split-K sums),
            // and a smaller burst there shortens that grid's tail by more than
            // it delays this one.
            constexpr int NP = NS < kPreWaitStages ? NS : kPreWaitStages;
            int st = 0, x_issued = 0;
            int stage_kc[NP], stage_u[NP];
            bool ok = true;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const int u = int(idx_div(unsigned(item), unsigned(a.Pv))), vp = item - u * a.Pv;
            const int xu = a.x_per_problem ? u : 0;
            const uint8_t *wb = a.w + (long long)(a.expert_ids ? a.expert_ids[u] : u) * a.w_stride;
            const unsigned i0 = split.start(vp);
            const int n_it = int(split.start(vp + 1) - i0);
            for (int j = 0; j < n_it && ok;) {
                const unsigned gi = i0 + unsigned(j);
                const int kc0 = int(gi - idx_div(gi, Kc) * Kc);
                const int seg_len = min(n_it - j, a.Kc - kc0);
                for (int sj = 0; sj < seg_len; sj += kStageIters, ++st) {
                    const int n_here = min(kStageIters, seg_len - sj);
                    const int s = st % NS;
                    if (st == NP) {
                        grid_dependency_wait();
                        for (; x_issued < NP; ++x_issued)
                            tma_load_4d(sx + x_issued * XST, &a.xmap, 0, 0, stage_kc[x_issued],
                                        stage_u[x_issued], &sy->full[x_issued]);
                    }
                    if (st >= NS && !wait_bar(&sy->empty[s], uint32_t(st / NS - 1) & 1, sy, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sy->full[s], uint32_t(n_here * CB + XST));
                    bulk_g2s_hint(sw + s * STW, wb + (long long)(gi + sj) * CB, uint32_t(n_here * CB), &sy->full[s],
                                  pol);
                    if (st < NP) {
                        stage_kc[st] = kc0 + sj;
                        stage_u[st] = xu;
                    } else {
                        tma_load_4d(sx + s * XST, &a.xmap, 0, 0, kc0 + sj, xu, &sy->full[s]);
                    }
                }
                j += seg_len;
            }
            }
            if (x_issued < min(st, NP)) {  // short ranges: fewer than NP stages
                grid_dependency_wait();
                for (; x_issued < min(st, NP); ++x_issued)
                    tma_load_4d(sx + x_issued * XST, &a.xmap, 0, 0, stage_kc[x_issued], stage_u[x_issued],
                                &sy->full[x_issued]);
            }
            const int issued = st;
            // leave only once every issued copy has landed (bounded)
            for (int k = (issued > NS ? issued - NS : 0); k < issued; ++k)
                wait_bar(&sy->full[k % NS], uint32_t(k / NS) & 1, sy, a.err);
        }
        return;
    }

    if constexpr (SEL) {
        if (warp > kConsumerWarps) {
            grid_dependency_wait();   // the candidate arrays may still be read by a preceding grid
            run_selector<HI>(a, SelView<HI>(selb), sy, warp - kConsumerWarps - 1);
            return;
        }
    }

    // ---------------- consumers ----------------
    const int kg = warp / kFeatWarps;   // k-group: slices kg, kg + 4, ... of each stage
    const int fw = warp % kFeatWarps;   // feature block
    const int gq = lane >> 2, tq = lane & 3;
    constexpr bool hi = HI;
    // ldmatrix row addresses: lane l supplies row (l & 7) + 8 * (l >> 4), 16-byte
    // chunk (l >> 3) & 1 of k step j; with the 128-byte swizzle, chunk c of row r
    // sits at chunk c ^ (r % 8)
    uint32_t xoff[4];
    {
        const int lrow = (lane & 7) + ((lane >> 4) << 3);
        const int lcol = (lane >> 3) & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) xoff[j] = uint32_t(lrow * 128 + (((2 * j + lcol) ^ (lrow & 7)) << 4));
    }
    const size_t ysz = a.mode == kSwiGluBf16 ? sizeof(__nv_bfloat16) : sizeof(float);
    // the split-tile combine of feature block fw stays inside fw's part of
    // buffer 0, which only fw's four warps touch
    float4 *rb_a = reinterpret_cast<float4 *>(red + fw * (CBF / kFeatWarps)) + lane * NQ;
    float4 *rb_b = rb_a + 32 * NQ;
    bool ok = true;

    float acc[2][2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][n][c] = 0.f;

    // SEL: a storing warp (kg == 0) hands each finished block to the selectors
    // through the shared ring; f0 < 0 signals its last block
    auto sel_push = [&](int f0, const float (&v)[2][2][4]) {
        SelView<HI> sv(selb);
        int ticket = 0;
        if (lane == 0) ticket = atomicAdd(sv.tail, 1);
        ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
        const int slot = ticket % kSelSlots;
        bool free_slot = true;
        if (ticket >= kSelSlots)
            free_slot = wait_bar(&sv.empty[slot], uint32_t(ticket / kSelSlots - 1) & 1u, sy, a.err);
        if (free_slot) {
            if (f0 >= 0) {
                float *dst = sv.ring + slot * SelView<HI>::SR * kSelStride;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        if (n == 1 && !HI) continue;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            dst[(n * 8 + tq * 2 + (c & 1)) * kSelStride + mt * 16 + gq + (c >= 2 ? 8 : 0)] =
                                v[mt][n][c];
                    }
            }
            if (lane == 0) sv.f0[slot] = f0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sv.full[slot]);
    };

    grid_dependency_wait();  // activations, workspace and outputs come from earlier grids
    int st = 0;  // stage counter, identical to the producer's
    int cpar = 0;   // combine buffer of the next whole-tile segment end (the same in every warp)
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int u = int(idx_div(unsigned(item), unsigned(a.Pv))), vp = item - u * a.Pv;
    void *yb = static_cast<char *>(a.y) + (long long)u * a.y_stride * (long long)ysz;
    const unsigned i0 = split.start(vp);
    const int n_it = int(split.start(vp + 1) - i0);
    for (int j = 0; j < n_it;) {
        const unsigned gi = i0 + unsigned(j);
        const int t = int(idx_div(gi, Kc));
        const int kc0 = int(gi - unsigned(t) * Kc);
        const int seg_len = min(n_it - j, a.Kc - kc0);
        for (int sj = 0; sj < seg_len; sj += kStageIters, ++st) {
            const int n_here = min(kStageIters, seg_len - sj);
            const int s = st % NS;
            if (ok) ok = wait_bar(&sy->full[s], uint32_t(st / NS) & 1, sy, a.err);
            if (ok) {
                const uint8_t *stage_w = sw + s * STW + fw * BB;
                const uint32_t stage_x = smem_u32(sx + s * XST);
                // slices of this stage whose index within the range is kg mod kKGroups
                const int p0 = (kg - (j + sj)) & (kKGroups - 1);
                if (!HI && n_here == kStageIters) {
#pragma unroll
                    for (int p = 0; p < kStageIters; p += kKGroups) {
                        if constexpr (FMT == kFmtNvfp4)
                            consume_slice_nvfp4<HI>(stage_w + (p0 + p) * CB, stage_x + (p0 + p) * XSL, lane, gq, xoff,
                                                    acc);
                        else
                            consume_slice<G, HI, AFF>(stage_w + (p0 + p) * CB, stage_x + (p0 + p) * XSL, lane, gq,
                                                      xoff, acc);
                    }
                } else {
                    for (int p = p0; p < n_here; p += kKGroups) {
                        if constexpr (FMT == kFmtNvfp4)
                            consume_slice_nvfp4<HI>(stage_w + p * CB, stage_x + p * XSL, lane, gq, xoff, acc);
                        else
                            consume_slice<G, HI, AFF>(stage_w + p * CB, stage_x + p * XSL, lane, gq, xoff, acc);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sy->empty[s]);
        }
        const unsigned seg_b = gi, seg_e = gi + unsigned(seg_len);
        j += seg_len;

        // ---- segment end: combine the k-groups in a fixed order, (0 + 1) + (2 + 3);
        // the four warps of feature block fw meet at their own named barrier
        auto put_rb = [&](float4 *rb) {
#pragma unroll
            for (int jq = 0; jq < NQ; ++jq) {
                const int q = HI ? jq : 2 * jq;
                rb[jq] = make_float4(acc[q >> 1][q & 1][0], acc[q >> 1][q & 1][1], acc[q >> 1][q & 1][2],
                                     acc[q >> 1][q & 1][3]);
            }
        };
        auto add_rb = [&](const float4 *rb) {
#pragma unroll
            for (int jq = 0; jq < NQ; ++jq) {
                const int q = HI ? jq : 2 * jq;
                const float4 o = rb[jq];
                acc[q >> 1][q & 1][0] += o.x;
                acc[q >> 1][q & 1][1] += o.y;
                acc[q >> 1][q & 1][2] += o.z;
                acc[q >> 1][q & 1][3] += o.w;
            }
        };
        const unsigned tb = unsigned(t) * Kc, te = tb + Kc;
        if (!SEL && seg_b == tb && seg_e == te) {
            // Whole tile: a reduce-scatter.  k-group q keeps element c = q of
            // every accumulator; the others hand it their values through buffer
            // cpar, and it adds the four in the order (0 + 1) + (2 + 3) and
            // stores that quarter, so the four warps share the epilogue.  The
            // buffers alternate: a warp writes buffer b again only after the
            // barrier of the segment end in between, which every warp reaches
            // after reading b.
            constexpr int QV = lane_vals(HI) / kKGroups;
            float *cb = red + cpar * CBF;
#pragma unroll
            for (int q = 0; q < kKGroups; ++q) {
                if (q == kg) continue;
                float *dst = cb + (((fw * kKGroups + q) * 3 + (((kg - q) & 3) - 1)) * 32 + lane) * QV;
                if (HI)
                    *reinterpret_cast<float4 *>(dst) = make_float4(acc[0][0][q], acc[1][0][q], acc[0][1][q], acc[1][1][q]);
                else
                    *reinterpret_cast<float2 *>(dst) = make_float2(acc[0][0][q], acc[1][0][q]);
            }
            float own[2][2];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    float o = acc[mt][n][0];
                    if (kg == 1) o = acc[mt][n][1];
                    if (kg == 2) o = acc[mt][n][2];
                    if (kg == 3) o = acc[mt][n][3];
                    own[mt][n] = o;
                }
            bar_sync_named(1 + fw, 32 * kKGroups);
            // k-group w's values of this warp's quarter
            auto fetch = [&](int w, float (&o)[2][2]) {
                if (w == kg) {
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                        for (int n = 0; n < 2; ++n) o[mt][n] = own[mt][n];
                    return;
                }
                const float *src = cb + (((fw * kKGroups + kg) * 3 + (((w - kg) & 3) - 1)) * 32 + lane) * QV;
                if (HI) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    o[0][0] = v.x;
                    o[1][0] = v.y;
                    o[0][1] = v.z;
                    o[1][1] = v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    o[0][0] = v.x;
                    o[1][0] = v.y;
                    o[0][1] = o[1][1] = 0.f;
                }
            };
            float sum[2][2], pa[2][2], pb[2][2];
            fetch(0, pa);
            fetch(1, pb);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int n = 0; n < 2; ++n) sum[mt][n] = pa[mt][n] + pb[mt][n];
            fetch(2, pa);
            fetch(3, pb);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int n = 0; n < 2; ++n) sum[mt][n] = sum[mt][n] + (pa[mt][n] + pb[mt][n]);
            store_quarter<FMT == kFmtNvfp4>(a, yb, t, fw, gq, tq, kg, hi, sum);
            cpar ^= 1;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[mt][n][c] = 0.f;
            continue;
        }
        cpar = 1;   // the split-tile combine below uses fw's part of buffer 0
        bar_sync_named(1 + fw, 32 * kKGroups);
        if (kg == 1) put_rb(rb_a);
        if (kg == 3) put_rb(rb_b);
        bar_sync_named(1 + fw, 32 * kKGroups);
        if (kg == 0) add_rb(rb_a);          // 0 + 1
        if (kg == 2) {
            add_rb(rb_b);                   // 2 + 3, written back over the slot it came from
            put_rb(rb_b);
        }
        bar_sync_named(1 + fw, 32 * kKGroups);
        if (kg == 0) {
            add_rb(rb_b);                   // (0 + 1) + (2 + 3)
            if (seg_b == tb && seg_e == te) {
                if (!SEL || a.y) store_block<FMT == kFmtNvfp4>(a, yb, t, fw, gq, tq, hi, acc);
                if constexpr (SEL) sel_push(t * kTileN + fw * kBlockRows, acc);
            } else {
                // stream-K partial.  A split tile's first k-slice lies in the
                // range p_lo, and the tile is the last segment of that range (a
                // range holding the tile's first and last slices holds all of
                // it), so p_lo owns the sum: every other segment publishes its
                // partial and bumps the tile's counter without waiting, and the
                // owner, at the end of its range, waits (bounded) until all of
                // them are in and adds them to its own in ascending k order.  No
                // range stalls on a round trip in its middle.  The waits rely on
                // every range running at once: a dense launch has one range per
                // CTA and at most one CTA per SM (grouped launches never split a
                // tile).  Rows 8..15 (accumulator half n = 1) travel only when
                // the launch has them.
                constexpr int NB = HI ? 2 : 4;   // segments loaded per round
                const int p_lo = int(split.owner(tb));
                const int p_hi = int(split.owner(te - 1));
                const int nseg = p_hi - p_lo + 1;
                // slot of segment p: index 0 if the tile is the first of p's range, else 1
                auto slot_of = [&](int p) -> float4 * {
                    const int which = split.start(unsigned(p)) >= tb ? 0 : 1;
                    return a.partials + ((((long long)u * a.Pv + p) * 2 + which) * kFeatWarps + fw) * 128 + lane * 4;
                };
                unsigned *ctr = a.counters + ((long long)u * a.T + t) * kFeatWarps + fw;
                if (n_items > int(gridDim.x)) {
                    if (lane == 0) set_error(a.err, 3);   // ranges not all resident: never launched so
                } else if (vp != p_lo) {
                    float4 *slot = slot_of(vp);
#pragma unroll
                    for (int jq = 0; jq < NQ; ++jq) {
                        const int q = HI ? jq : 2 * jq;
                        __stcg(slot + q, make_float4(acc[q >> 1][q & 1][0], acc[q >> 1][q & 1][1],
                                                     acc[q >> 1][q & 1][2], acc[q >> 1][q & 1][3]));
                    }
                    // the warp barrier orders every lane's stores before lane 0's release
                    __syncwarp();
                    if (lane == 0) red_add_release_gpu(ctr, 1u);
                } else {
                    bool in = true;
                    if (lane == 0) {
                        uint32_t it = 0;
                        while (ld_acquire_gpu(ctr) != unsigned(nseg - 1)) {
                            if (++it == kWaitLimit) {
                                in = false;
                                set_error(a.err, 1);
                                break;
                            }
                        }
                    }
                    in = __shfl_sync(0xFFFFFFFFu, in ? 1 : 0, 0) != 0;
                    __syncwarp();     // every lane's reads after lane 0's acquire
                    if (in) {
                        float sum[2][2][4];
#pragma unroll
                        for (int q = 0; q < 16; ++q) sum[q >> 3][(q >> 2) & 1][q & 3] = 0.f;
                        for (int pb = p_lo; pb <= p_hi; pb += NB) {
                            float4 v[NB][NQ];
#pragma unroll
                            for (int b = 0; b < NB; ++b) {
                                const int p = pb + b;
                                const float4 *src = (p <= p_hi && p != vp) ? slot_of(p) : nullptr;
#pragma unroll
                                for (int jq = 0; jq < NQ; ++jq) {
                                    const int q = HI ? jq : 2 * jq;
                                    v[b][jq] = src ? __ldcg(src + q)
                                                   : make_float4(acc[q >> 1][q & 1][0], acc[q >> 1][q & 1][1],
                                                                 acc[q >> 1][q & 1][2], acc[q >> 1][q & 1][3]);
                                }
                            }
                            // add in ascending k order
#pragma unroll
                            for (int b = 0; b < NB; ++b) {
                                if (pb + b > p_hi) break;
#pragma unroll
                                for (int jq = 0; jq < NQ; ++jq) {
                                    const int q = HI ? jq : 2 * jq;
                                    sum[q >> 1][q & 1][0] += v[b][jq].x;
                                    sum[q >> 1][q & 1][1] += v[b][jq].y;
                                    sum[q >> 1][q & 1][2] += v[b][jq].z;
                                    sum[q >> 1][q & 1][3] += v[b][jq].w;
                                }
                            }
                        }
                        if (lane == 0) *ctr = 0u;  // leave the counter zero for the next launch
                        if (!SEL || a.y) store_block<FMT == kFmtNvfp4>(a, yb, t, fw, gq, tq, hi, sum);
                        if constexpr (SEL) sel_push(t * kTileN + fw * kBlockRows, sum);
                    }
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][n][c] = 0.f;
    }
    }
    if constexpr (SEL) {
        if (kg == 0) sel_push(-1, acc);
    }
}

// ---- load-time repack: canonical [N][K/2] nibbles + [N][K/G] fp16 -> kernel layout
// Canonical row of packed feature p (interleave: per 32-row feature block, 16
// gate rows then the 16 matching up rows).
__device__ __forceinline__ long long canonical_row(long long p, int N, bool inter) {
    if (!inter) return p < N ? p : -1;
    const int F = N / 2;
    const long long t = p / kTileN;
    const int fw = int(p % kTileN) / kBlockRows;
    const int r32 = int(p % kBlockRows);
    const long long j = t * (kTileN / 2) + fw * 16 + (r32 & 15);
    if (j >= F) return -1;
    return r32 < 16 ? j : F + j;
}

template <int G>
__global__ void pack_codes_kernel(const uint8_t *codes, int K, int N, uint8_t *out, long long n_entries, int Kc,
                                  bool inter) {
    constexpr int BB = block_bytes(G);
    constexpr int CB = chunk_bytes(G);
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int lane = int(idx % 32);
    long long r = idx / 32;
    const int mt = int(r % 2);
    r /= 2;
    const int fw = int(r % kFeatWarps);
    r /= kFeatWarps;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t words[4];
    for (int j = 0; j < 4; ++j) {
        uint32_t w = 0;
        for (int i = 0; i < 4; ++i)
            for (int h = 0; h < 2; ++h) {
                const long long f = canonical_row(
                    t * kTileN + fw * kBlockRows + mt * 16 + gq + ((i & 1) ? 8 : 0), N, inter);
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
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + fw * BB + mt * 512 + lane * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

template <int G>
__global__ void pack_scales_kernel(const uint16_t *scales, int K, int N, uint8_t *out, long long n_entries, int Kc,
                                   bool inter) {
    constexpr int BB = block_bytes(G);
    constexpr int CB = chunk_bytes(G);
    constexpr int NG = kKChunk / G;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int mt = int(idx % 2);
    long long r = idx / 2;
    const int g = int(r % 8);
    r /= 8;
    const int grp = int(r % NG);
    r /= NG;
    const int fw = int(r % kFeatWarps);
    r /= kFeatWarps;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const long long p = t * kTileN + fw * kBlockRows + mt * 16 + g;
    const long long f_lo = canonical_row(p, N, inter);
    const long long f_hi = canonical_row(p + 8, N, inter);
    const int gi = kc * NG + grp;
    const int ngroups = K / G;
    const uint32_t lo = f_lo >= 0 ? scales[f_lo * ngroups + gi] : 0u;
    const uint32_t hi = f_hi >= 0 ? scales[f_hi * ngroups + gi] : 0u;
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + fw * BB + 1024 + grp * 64 + g * 8 + mt * 4;
    *reinterpret_cast<uint32_t *>(dst) = lo | (hi << 16);
}

// Affine (MLX-style) packing: same chunk geometry; codes are taken as they are
// (unsigned, no offset), and each group carries bf16 scales then bf16 biases.
template <int G>
__global__ void pack_codes_affine_kernel(const uint32_t *codes, int K, int N, uint8_t *out, long long n_entries,
                                         int Kc) {
    constexpr int BB = block_bytes(G, true);
    constexpr int CB = chunk_bytes(G, true);
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int lane = int(idx % 32);
    long long r = idx / 32;
    const int mt = int(r % 2);
    r /= 2;
    const int fw = int(r % kFeatWarps);
    r /= kFeatWarps;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t words[4];
    for (int j = 0; j < 4; ++j) {
        uint32_t w = 0;
        for (int i = 0; i < 4; ++i)
            for (int h = 0; h < 2; ++h) {
                const long long f = t * kTileN + fw * kBlockRows + mt * 16 + gq + ((i & 1) ? 8 : 0);
                const int k = kc * kKChunk + j * 16 + 2 * tq + h + ((i & 2) ? 8 : 0);
                uint32_t q = 0;  // rows past N: zero codes (and zero scale and bias)
                if (f < N) q = (codes[f * (K / 8) + k / 8] >> (4 * (k % 8))) & 0xFu;
                w |= q << (4 * i + 16 * h);
            }
        words[j] = w;
    }
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + fw * BB + mt * 512 + lane * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

template <int G>
__global__ void pack_scales_affine_kernel(const uint16_t *scales, const uint16_t *biases, int K, int N, uint8_t *out,
                                          long long n_entries, int Kc) {
    constexpr int BB = block_bytes(G, true);
    constexpr int CB = chunk_bytes(G, true);
    constexpr int NG = kKChunk / G;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int mt = int(idx % 2);
    long long r = idx / 2;
    const int g = int(r % 8);
    r /= 8;
    const int grp = int(r % NG);
    r /= NG;
    const int fw = int(r % kFeatWarps);
    r /= kFeatWarps;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const long long f_lo = t * kTileN + fw * kBlockRows + mt * 16 + g;
    const long long f_hi = f_lo + 8;
    const int gi = kc * NG + grp;
    const int ngroups = K / G;
    const uint32_t s_lo = f_lo < N ? scales[f_lo * ngroups + gi] : 0u;
    const uint32_t s_hi = f_hi < N ? scales[f_hi * ngroups + gi] : 0u;
    const uint32_t b_lo = f_lo < N ? biases[f_lo * ngroups + gi] : 0u;
    const uint32_t b_hi = f_hi < N ? biases[f_hi * ngroups + gi] : 0u;
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + fw * BB + 1024 + grp * 128 + g * 8 + mt * 4;
    *reinterpret_cast<uint32_t *>(dst) = s_lo | (s_hi << 16);
    *reinterpret_cast<uint32_t *>(dst + 64) = b_lo | (b_hi << 16);
}

template <int G>
cudaError_t launch_pack_affine_g(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases, int K, int N,
                                 void *packed, cudaStream_t s) {
    const int T = (N + kTileN - 1) / kTileN;
    const int Kc = K / kKChunk;
    const long long n_codes = (long long)T * Kc * kFeatWarps * 2 * 32;
    const long long n_scales = (long long)T * Kc * kFeatWarps * (kKChunk / G) * 8 * 2;
    const int th = 256;
    pack_codes_affine_kernel<G><<<unsigned((n_codes + th - 1) / th), th, 0, s>>>(codes, K, N, (uint8_t *)packed,
                                                                               n_codes, Kc);
    pack_scales_affine_kernel<G><<<unsigned((n_scales + th - 1) / th), th, 0, s>>>(scales, biases, K, N,
                                                                                 (uint8_t *)packed, n_scales, Kc);
    return cudaGetLastError();
}

// NVFP4 packing: same chunk geometry.  Byte i of word j of a lane's 16-byte
// entry is its A register i for k step j: the canonical byte of row (g or
// g + 8) holding elements k, k + 1 (k = 16 j + 2 q (+ 8)), low nibble first --
// exactly the canonical storage byte.  Rows past N get code 0 and scale 0.
__global__ void pack_codes_nvfp4_kernel(const uint8_t *codes, int K, int N, uint8_t *out, long long n_entries,
                                        int Kc) {
    constexpr int BB = block_bytes(16, kFmtNvfp4);
    constexpr int CB = chunk_bytes(16, kFmtNvfp4);
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int lane = int(idx % 32);
    long long r = idx / 32;
    const int mt = int(r % 2);
    r /= 2;
    const int fw = int(r % kFeatWarps);
    r /= kFeatWarps;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t words[4];
    for (int j = 0; j < 4; ++j) {
        uint32_t w = 0;
        for (int i = 0; i < 4; ++i) {
            const long long f = t * kTileN + fw * kBlockRows + mt * 16 + gq + ((i & 1) ? 8 : 0);
            const int k = kc * kKChunk + j * 16 + 2 * tq + ((i & 2) ? 8 : 0);
            const uint32_t byte = f < N ? codes[f * (K / 2) + k / 2] : 0u;
            w |= byte << (8 * i);
        }
        words[j] = w;
    }
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + fw * BB + mt * 512 + lane * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

// Scale entry of (tile t, slice kc, feature block fw, lane group g): 16 bytes
// [j 0..3][mt 0..1] (s[row g][4 kc + j], s[row g + 8][4 kc + j]).
__global__ void pack_scales_nvfp4_kernel(const uint8_t *scales, int K, int N, uint8_t *out, long long n_entries,
                                         int Kc) {
    constexpr int BB = block_bytes(16, kFmtNvfp4);
    constexpr int CB = chunk_bytes(16, kFmtNvfp4);
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_entries) return;
    const int g = int(idx % 8);
    long long r = idx / 8;
    const int fw = int(r % kFeatWarps);
    r /= kFeatWarps;
    const int kc = int(r % Kc);
    const long long t = r / Kc;
    const int nb = K / 16;
    uint32_t words[4];
    for (int j = 0; j < 4; ++j) {
        uint32_t w = 0;
        for (int mt = 0; mt < 2; ++mt)
            for (int h = 0; h < 2; ++h) {
                const long long f = t * kTileN + fw * kBlockRows + mt * 16 + g + (h ? 8 : 0);
                const uint32_t b = f < N ? scales[f * nb + kc * 4 + j] : 0u;
                w |= b << (8 * (mt * 2 + h));
            }
        words[j] = w;
    }
    uint8_t *dst = out + (t * Kc + kc) * (long long)CB + fw * BB + 1024 + g * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

int grid_of(const GemmArgs &a, int u_max) {
    // persistent over work items: at most one CTA per SM
    const long long items = (long long)a.Pv * u_max;
    int sms = device_sm_count();
    if (sms <= 0) sms = 1;
    return int(items < sms ? items : sms);
}

template <int G, bool HI, int FMT, bool SEL = false>
cudaError_t launch_gemm_g(const GemmArgs &a, int u_max, cudaStream_t s) {
    const size_t smem = gemm_smem_bytes(G, HI, FMT, SEL);
    // the shared-memory opt-in is a per-device property of the kernel: set it once
    static std::atomic<bool> opted_in[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(w4_lane_gemm_kernel<G, HI, FMT, SEL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   int(smem));
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid_of(a, u_max)));
    cfg.blockDim = dim3(SEL ? kThreads + 32 * kSelWarps : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w4_lane_gemm_kernel<G, HI, FMT, SEL>, a);
}

template <int G>
cudaError_t launch_pack_g(const uint8_t *codes, const uint16_t *scales, int K, int N, void *packed, bool inter,
                          cudaStream_t s) {
    const int T = (N + kTileN - 1) / kTileN;
    const int Kc = K / kKChunk;
    const long long n_codes = (long long)T * Kc * kFeatWarps * 2 * 32;
    const long long n_scales = (long long)T * Kc * kFeatWarps * (kKChunk / G) * 8 * 2;
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
    cuuint32_t box[4] = {cuuint32_t(kKChunk), cuuint32_t(x_rows(a.R > 8)), cuuint32_t(kStageIters), 1};
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
    const bool hi = a.R > 8;
    if (a.fmt == kFmtNvfp4) return hi ? launch_gemm_g<16, true, kFmtNvfp4>(a, u_max, s)
                                      : launch_gemm_g<16, false, kFmtNvfp4>(a, u_max, s);
    if (a.fmt == kFmtAffine) {
        if (hi) return a.G == 64 ? launch_gemm_g<64, true, kFmtAffine>(a, u_max, s)
                                 : launch_gemm_g<32, true, kFmtAffine>(a, u_max, s);
        return a.G == 64 ? launch_gemm_g<64, false, kFmtAffine>(a, u_max, s)
                         : launch_gemm_g<32, false, kFmtAffine>(a, u_max, s);
    }
    if (hi) return a.G == 64 ? launch_gemm_g<64, true, kFmtSym>(a, u_max, s) : launch_gemm_g<32, true, kFmtSym>(a, u_max, s);
    return a.G == 64 ? launch_gemm_g<64, false, kFmtSym>(a, u_max, s) : launch_gemm_g<32, false, kFmtSym>(a, u_max, s);
}

int gemm_grid(const GemmArgs &a, int u_max) { return grid_of(a, u_max); }

cudaError_t launch_w4_gemm_select(const GemmArgs &a, cudaStream_t s) {
    if (a.fmt != kFmtSym || a.n_problems || a.expert_ids || a.mode != kStoreF32 || a.sel_k < 1 ||
        a.sel_k > kSelList || a.sel_nc != grid_of(a, 1) || !a.sel_val || !a.sel_id || !a.sel_cnt || !a.sel_kth ||
        !a.sel_bad || !a.sel_bound)
        return cudaErrorInvalidValue;
    if (a.R > kSelMaxRows) return cudaErrorInvalidValue;
    return a.G == 64 ? launch_gemm_g<64, false, kFmtSym, true>(a, 1, s) : launch_gemm_g<32, false, kFmtSym, true>(a, 1, s);
}

cudaError_t launch_pack_w4_affine(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases, int K, int N,
                                  int G, void *packed, cudaStream_t s) {
    return G == 64 ? launch_pack_affine_g<64>(codes, scales, biases, K, N, packed, s)
                   : launch_pack_affine_g<32>(codes, scales, biases, K, N, packed, s);
}

cudaError_t launch_pack_w4(const uint8_t *codes, const uint16_t *scales, int K, int N, int G, void *packed,
                           bool interleave_gate_up, cudaStream_t s) {
    return G == 64 ? launch_pack_g<64>(codes, scales, K, N, packed, interleave_gate_up, s)
                   : launch_pack_g<32>(codes, scales, K, N, packed, interleave_gate_up, s);
}

cudaError_t launch_pack_nvfp4(const uint8_t *codes, const uint8_t *scales, int K, int N, void *packed,
                              cudaStream_t s) {
    const int T = (N + kTileN - 1) / kTileN;
    const int Kc = K / kKChunk;
    const long long n_codes = (long long)T * Kc * kFeatWarps * 2 * 32;
    const long long n_scales = (long long)T * Kc * kFeatWarps * 8;
    const int th = 256;
    pack_codes_nvfp4_kernel<<<unsigned((n_codes + th - 1) / th), th, 0, s>>>(codes, K, N, (uint8_t *)packed, n_codes,
                                                                           Kc);
    pack_scales_nvfp4_kernel<<<unsigned((n_scales + th - 1) / th), th, 0, s>>>(scales, K, N, (uint8_t *)packed,
                                                                             n_scales, Kc);
    return cudaGetLastError();
}

int device_sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace tfk
