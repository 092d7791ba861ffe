// Device check of tfk::idx_div, the lane GEMM's reciprocal quotient, against
// the integer division it replaces: n = n_begin, n_begin + n_step, ... below
// n_end for each divisor d = d_lo, d_lo + d_step, ... up to d_hi.  Counts
// mismatches and keeps the first one.  C ABI only; built by the test that
// uses it.
#include <cstdint>
#include <cuda_runtime.h>

#include "../w4_gemm_keyed_gb300/csrc/tf_ptx.cuh"

namespace {

__global__ void idx_div_kernel(unsigned d_lo, unsigned d_hi, unsigned d_step, unsigned n_begin, unsigned n_end,
                               unsigned n_step,
                               unsigned long long *bad, unsigned *first) {
    const unsigned long long nd = (unsigned long long)((d_hi - d_lo) / d_step + 1);
    const unsigned long long nn = (unsigned long long)((n_end - n_begin + n_step - 1) / n_step);
    const unsigned long long total = nd * nn;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (unsigned long long)gridDim.x * blockDim.x) {
        const unsigned d = d_lo + unsigned(i / nn) * d_step;
        const unsigned n = n_begin + unsigned(i % nn) * n_step;
        if (tfk::idx_div(n, d) != n / d) {
            if (atomicAdd(bad, 1ull) == 0ull) {
                first[0] = n;
                first[1] = d;
            }
        }
    }
}

}  // namespace

extern "C" int idx_div_check(unsigned d_lo, unsigned d_hi, unsigned d_step, unsigned n_begin, unsigned n_end,
                             unsigned n_step,
                             unsigned long long *bad, unsigned *first) {
    if (d_lo < 1 || d_hi < d_lo || d_step < 1 || n_step < 1 || n_end <= n_begin) return 1;
    idx_div_kernel<<<1024, 256>>>(d_lo, d_hi, d_step, n_begin, n_end, n_step, bad, first);
    if (cudaGetLastError() != cudaSuccess) return 2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
