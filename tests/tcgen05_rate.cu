// Rate probe for the two tensor-core paths an sm_103a lane GEMM could use.
//
//  * tc05_rate_kernel: one thread per CTA issues a chain of `tcgen05.mma
//    .cta_group::1.kind::f16` (M = 128, N = n, K = 16, bf16 operands in shared
//    memory without swizzle, fp32 accumulator in tensor memory), commits it to
//    an mbarrier and waits (bounded); the CTA then reads the accumulator back
//    with `tcgen05.ld`, so a caller can check the product before trusting the
//    timing.
//  * mma_sync_rate_kernel: every warp issues chains of `mma.sync.m16n8k16`
//    (bf16, fp32 accumulate) with `chains` independent accumulators.
//
// Both record clock64() cycles per CTA.  C ABI only; built by the test that
// uses it.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

constexpr int kM = 128;
constexpr int kK = 16;
constexpr int kMaxN = 256;
constexpr int kTmemCols = 512;   // accumulator (up to 256 columns) + the tensor-memory copy of A
constexpr uint32_t kWaitPolls = 1u << 24;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Operand tile in the no-swizzle K-major layout: core matrices of 8 rows x
// 16 bytes (8 bf16 along K) stored as 128 contiguous bytes; the two core
// matrices of a row group (K = 0..7, 8..15) are `lbo` bytes apart, successive
// 8-row groups `sbo` bytes apart.
__device__ __forceinline__ int core_offset(int row, int k, int lbo, int sbo) {
    return (row >> 3) * sbo + (k >> 3) * lbo + (row & 7) * 16 + (k & 7) * 2;
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (each >> 4), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, int lbo, int sbo) {
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);
    d |= uint64_t((uint32_t(lbo) >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((uint32_t(sbo) >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same with A read from tensor memory (lane m holds row m, two bf16 per
// 32-bit column along K).
__device__ __forceinline__ void tc_mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t db, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(tmem_d), "r"(tmem_a), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}
template <bool TA>
__device__ __forceinline__ void mma_one(uint32_t d, uint32_t ta, uint64_t da, uint64_t db, uint32_t idesc,
                                        uint32_t accumulate) {
    if (TA)
        tc_mma_ta(d, ta, db, idesc, accumulate);
    else
        tc_mma(d, da, db, idesc, accumulate);
}

// n_mma MMAs in rounds of n_acc (one per accumulator), the first round
// overwriting, eight rounds per loop trip.
template <bool TA>
__device__ __forceinline__ void issue_chain(uint32_t tmem, uint32_t ta, uint64_t da, uint64_t db, uint32_t idesc,
                                            int n_mma, int n_acc) {
    const int rounds = n_mma / n_acc;
    if (n_acc == 1) {
        mma_one<TA>(tmem, ta, da, db, idesc, 0u);
        int r = 1;
        for (; r + 8 <= rounds; r += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) mma_one<TA>(tmem, ta, da, db, idesc, 1u);
        }
        for (; r < rounds; ++r) mma_one<TA>(tmem, ta, da, db, idesc, 1u);
    } else {
        const uint32_t d1 = tmem + 64u, d2 = tmem + 128u, d3 = tmem + 192u;
        mma_one<TA>(tmem, ta, da, db, idesc, 0u);
        mma_one<TA>(d1, ta, da, db, idesc, 0u);
        mma_one<TA>(d2, ta, da, db, idesc, 0u);
        mma_one<TA>(d3, ta, da, db, idesc, 0u);
        int r = 1;
        for (; r + 2 <= rounds; r += 2) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mma_one<TA>(tmem, ta, da, db, idesc, 1u);
                mma_one<TA>(d1, ta, da, db, idesc, 1u);
                mma_one<TA>(d2, ta, da, db, idesc, 1u);
                mma_one<TA>(d3, ta, da, db, idesc, 1u);
            }
        }
        for (; r < rounds; ++r) {
            mma_one<TA>(tmem, ta, da, db, idesc, 1u);
            mma_one<TA>(d1, ta, da, db, idesc, 1u);
            mma_one<TA>(d2, ta, da, db, idesc, 1u);
            mma_one<TA>(d3, ta, da, db, idesc, 1u);
        }
    }
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__global__ void __launch_bounds__(128, 1)
    tc05_rate_kernel(int n, int n_mma, int n_acc, int lbo, int sbo, int a_tmem, long long *cycles, float *dout,
                     int *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sa = smem;                  // A: 128 x 16 bf16, 4 KB
    uint8_t *sb = smem + 16384;          // B: n x 16 bf16, up to 8 KB
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // operands: small integers, exact in bf16 and in the fp32 sums
    for (int i = tid; i < kM * kK; i += blockDim.x) {
        const int r = i / kK, k = i % kK;
        *reinterpret_cast<__nv_bfloat16 *>(sa + core_offset(r, k, lbo, sbo)) =
            __float2bfloat16(float((7 * r + 3 * k) % 11 - 5));
    }
    for (int i = tid; i < n * kK; i += blockDim.x) {
        const int r = i / kK, k = i % kK;
        *reinterpret_cast<__nv_bfloat16 *>(sb + core_offset(r, k, lbo, sbo)) =
            __float2bfloat16(float((5 * r + 13 * k) % 9 - 4));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (tid == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t tmem_a = tmem + uint32_t(kMaxN);   // A copy: columns 256..263
    if (a_tmem) {
        // thread t of warp w writes row 32 w + t: column j holds k = 2j (low half), 2j + 1
        const int r = 32 * warp + lane;
        uint32_t v[8];
        for (int j = 0; j < 8; ++j) {
            const float lo = float((7 * r + 3 * (2 * j)) % 11 - 5), hi = float((7 * r + 3 * (2 * j + 1)) % 11 - 5);
            const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
            v[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                         tmem_a + (uint32_t(32 * warp) << 16)),
                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                     : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    bool done = true;
    if (tid == 0) {
        const uint64_t da = smem_desc(smem_addr(sa), lbo, sbo);
        const uint64_t db = smem_desc(smem_addr(sb), lbo, sbo);
        const uint32_t idesc = instr_desc(kM, n);
        const long long t0 = clock64();
        // n_acc independent accumulators, 64 columns apart (N <= 64 when n_acc > 1),
        // taken in turn; the issue loop is unrolled so that the one issuing
        // thread's own instructions stay off the measured rate
        if (a_tmem)
            issue_chain<true>(tmem, tmem_a, da, db, idesc, n_mma, n_acc);
        else
            issue_chain<false>(tmem, tmem_a, da, db, idesc, n_mma, n_acc);
        tc_commit(&bar);
        uint32_t it = 0;
        while (!mbar_test(&bar, 0) && ++it < kWaitPolls) {
        }
        const long long t1 = clock64();
        done = it < kWaitPolls;
        if (!done) atomicExch(status, 1);
        cycles[blockIdx.x] = t1 - t0;
    }
    // everyone waits for the chain before reading the accumulator
    if (tid != 0) {
        uint32_t it = 0;
        while (!mbar_test(&bar, 0) && ++it < kWaitPolls) {
        }
    }
    tc_fence_after();
    if (blockIdx.x == 0) {
        // 32x32b.x16: thread t of warp w reads lane 32 w + t, 16 columns at a time
        for (int c0 = 0; c0 < n; c0 += 16) {
            uint32_t v[16];
            const uint32_t taddr = tmem + (uint32_t(32 * warp) << 16) + uint32_t(c0);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                "[%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            for (int j = 0; j < 16; ++j) dout[(32 * warp + lane) * kMaxN + c0 + j] = __uint_as_float(v[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <int CH>
__global__ void __launch_bounds__(512, 1) mma_sync_rate_kernel(int iters, long long *cycles, float *sink) {
    uint32_t a[4], b0, b1;
    const uint32_t one = 0x3F803F80u;   // bf16 (1, 1)
    for (int i = 0; i < 4; ++i) a[i] = one ^ (threadIdx.x & 1u);
    b0 = one;
    b1 = one;
    float d[CH][4];
    for (int c = 0; c < CH; ++c)
        for (int j = 0; j < 4; ++j) d[c][j] = 0.f;
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < CH; ++c)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __syncthreads();
    const long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    float s = 0.f;
    for (int c = 0; c < CH; ++c)
        for (int j = 0; j < 4; ++j) s += d[c][j];
    if (s == 12345.f) sink[threadIdx.x] = s;   // keeps the chains live
}

}  // namespace

extern "C" {

// One launch of `grid` CTAs, each issuing n_mma tcgen05.mma of M = 128, N = n,
// K = 16, A from shared memory or (a_tmem != 0) from tensor memory, cycling
// over n_acc accumulators (1 or 4, N <= 64 for 4; n_mma a multiple of n_acc).  cycles[grid] (device) gets each CTA's issue-to-completion cycles;
// dout[128 * 256] (device) gets CTA 0's accumulator (row-major, 256 columns);
// status (device int) becomes 1 if a wait gave up.  Returns a cudaError_t.
// lbo, sbo: multiples of 16 with every operand byte inside its 16 KB half of
// the 32 KB the kernel uses (whichever way the descriptor's two offsets are
// read); 120 KB of dynamic shared memory keep one CTA per SM.
int tc05_rate(int grid, int n, int n_mma, int n_acc, int lbo, int sbo, int a_tmem, long long *cycles, float *dout,
              int *status) {
    if (n < 16 || n > kMaxN || n % 16 || n_mma < 1 || grid < 1) return int(cudaErrorInvalidValue);
    if ((n_acc != 1 && n_acc != 4) || (n_acc > 1 && n > 64) || n_mma % n_acc) return int(cudaErrorInvalidValue);
    if (lbo < 16 || sbo < 16 || lbo % 16 || sbo % 16) return int(cudaErrorInvalidValue);
    const int hi = lbo > sbo ? lbo : sbo;
    if ((kMaxN / 8 - 1) * hi + hi + 128 > 16384) return int(cudaErrorInvalidValue);
    constexpr int kSmem = 120 * 1024;
    cudaError_t e = cudaFuncSetAttribute(tc05_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return int(e);
    tc05_rate_kernel<<<grid, 128, kSmem>>>(n, n_mma, n_acc, lbo, sbo, a_tmem, cycles, dout, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return int(e);
    return int(cudaDeviceSynchronize());
}

// One launch of `grid` CTAs of `warps` warps, each warp issuing iters x chains
// mma.sync.m16n8k16 (chains = 1, 2, 4 or 8 independent accumulators).
int mma_sync_rate(int grid, int warps, int chains, int iters, long long *cycles, float *sink) {
    if (warps < 1 || warps > 16 || grid < 1 || iters < 1) return int(cudaErrorInvalidValue);
    switch (chains) {
        case 1: mma_sync_rate_kernel<1><<<grid, 32 * warps>>>(iters, cycles, sink); break;
        case 2: mma_sync_rate_kernel<2><<<grid, 32 * warps>>>(iters, cycles, sink); break;
        case 4: mma_sync_rate_kernel<4><<<grid, 32 * warps>>>(iters, cycles, sink); break;
        case 8: mma_sync_rate_kernel<8><<<grid, 32 * warps>>>(iters, cycles, sink); break;
        default: return int(cudaErrorInvalidValue);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return int(e);
    return int(cudaDeviceSynchronize());
}
}
