// Row-exact attention of verify rows over a KV cache: declarations.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tfk {

constexpr int kHeadDim = 128;
constexpr int kKvPart = 256;     // keys per partition: a fixed grid of absolute positions
constexpr int kKvSub = 64;       // keys per pipeline stage
constexpr int kAttnMaxGroup = 8;
constexpr int kDevTimeout = 1;        // device status: a bounded wait ran out
constexpr int kDevBadPosition = 4;    // device status: *pos < 0 or *pos + R > max_len

struct AttnArgs {
    const uint16_t *k;      // cache, bf16 [n_kv][max_len][128], 16-B chunks XOR-swizzled by position
    const uint16_t *v;
    const uint16_t *q;      // bf16 [R][ldq], query head h at columns h*128
    int ldq;
    int R, group, n_kv, max_len;
    const int64_t *pos;     // row r sits at position *pos + r
    float *opart;           // [max_len/256][R][n_q][128] unnormalised partial outputs
    float *ml;              // [max_len/256][R][n_q][2] (raw score max, weight sum)
    float *out;             // fp32 [R][ldo]
    int ldo;
    int *err;
};

// Bytes of the partial-output arrays for R rows (each rounded to 256 B).
size_t attn_opart_bytes(int n_kv, int group, int max_len, int R);
size_t attn_ml_bytes(int n_kv, int group, int max_len, int R);

// cache[j][*pos + r] = new[r][j*128 .. j*128+127] for K and V, r < R.
cudaError_t launch_kv_append(const uint16_t *k_new, const uint16_t *v_new, int ld, int R, const int64_t *pos,
                             uint16_t *k_cache, uint16_t *v_cache, int n_kv, int max_len, int *err,
                             cudaStream_t s);
// Partials per (partition, KV head), then the fixed-order combine per (row, query head).
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s);

}  // namespace tfk
