// W4 lane GEMM: shared declarations between the kernel file and the C ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tfk {

// ---- packed weight layout --------------------------------------------------
// Output features are grouped in tiles of 256 = two "M-tiles" of 128 rows (one
// tcgen05 MMA's M).  For every tile t and every 64-wide slice kc of the input
// features there is one contiguous "chunk", and consecutive kc of a tile are
// consecutive in memory, so any run of iterations of one tile is one bulk copy.
// A chunk is two M-tile blocks; an M-tile block holds
//   codes : [half 0..1][row 0..127][16 B]   4096 B   row's k = 32*half .. +31
//   scales: [row 0..127][64/G] fp16          256 B per group
// Inside a row's 16 bytes, word e (k = 32*half + 8*e .. +7, e = 0..3) keeps the
// code of k offset q (0..7) as offset binary (code + 8) at bits
// 4*(q/2) + 16*(q%2): one shift + LOP3 per pair turns it into bf16 (16 + u).
constexpr int kMTile = 128;                // rows per tcgen05 MMA (M)
constexpr int kMTiles = 2;                 // M-tiles per tile
constexpr int kTileN = kMTile * kMTiles;   // 256 output features per tile
constexpr int kKChunk = 64;                // k per iteration
constexpr int kRows = 16;                  // MMA N: verify rows, zero-padded
constexpr int kStageIters = 4;             // iterations per pipeline stage (one weight copy of ~35 KB)
constexpr int kStages = 4;
constexpr int kDequantWarps = 8;           // two warpgroups, one per M-tile
constexpr int kThreads = 32 * (2 + kDequantWarps);  // producer + MMA + dequant/epilogue warps
constexpr int kXSliceBytes = kRows * kKChunk * 2;   // [16 rows][64 k] bf16, 128-byte swizzled
constexpr int kXStageBytes = kStageIters * kXSliceBytes;

__host__ __device__ constexpr int mtile_bytes(int G) { return 4096 + 256 * (kKChunk / G); }
__host__ __device__ constexpr int chunk_bytes(int G) { return kMTiles * mtile_bytes(G); }
// One partial tile of the split-K fixup: 8 warps x 32 lanes x 16 floats.
constexpr size_t kSlotBytes = size_t(kDequantWarps) * 32 * kRows * 4;

inline size_t gemm_smem_bytes(int G) {
    return 1024                                                         // alignment slack
           + size_t(kStages) * kXStageBytes                             // activation slices (1024-B aligned)
           + size_t(kStages) * kStageIters * chunk_bytes(G)            // weight stages
           + 256;                                                       // barriers, TMEM base
}

inline bool packed_shape_ok(int K, int N, int G) {
    return K > 0 && N > 0 && (G == 32 || G == 64) && K % kKChunk == 0;
}
inline size_t packed_bytes(int K, int N, int G) {
    if (!packed_shape_ok(K, N, G)) return 0;
    size_t T = (size_t(N) + kTileN - 1) / kTileN;
    return T * size_t(K / kKChunk) * size_t(chunk_bytes(G));
}

// ---- launch description ------------------------------------------------------
// A launch runs U problems (U = 1 for a plain linear layer; U = touched experts
// for the MoE layer).  Problem u uses weights at w + expert(u) * w_stride,
// activations from the tensor map (problem coordinate u when x_per_problem)
// and writes y + u * y_stride.  Each problem's tile x k-slice iteration space
// is cut into Pv contiguous ranges ("virtual CTAs", stream-K style); the cut
// depends only on (T, Kc, Pv).
enum EpilogueMode : int {
    kStoreF32 = 0,      // y (fp32) = result
    kAccumulateF32 = 1, // y (fp32) += result          (residual update)
    kSwiGluBf16 = 2,    // y (bf16 [R][F]) = bf16(silu(gate) * up), weights packed gate/up-interleaved
};

struct GemmArgs {
    CUtensorMap xmap;          // activations: dims {64, R, K/64, U}, box {64, 16, kStageIters, 1}, 128B swizzle
    const uint8_t *w;
    long long w_stride;        // bytes between experts
    const int *expert_ids;     // dev [U_max] or nullptr (expert = u)
    const int *n_problems;     // dev count or nullptr (1)
    int x_per_problem;         // activations differ per problem (use coordinate u)
    void *y;                   // fp32, or bf16 for kSwiGluBf16
    long long y_stride;        // elements between problems
    int ldy;
    int mode;                  // EpilogueMode
    int F;                     // kSwiGluBf16: width of h (N = 2F)
    int R, K, N, G;
    int T, Kc, Pv;
    unsigned *counters;        // [U_max][T][kDequantWarps], zero between launches
    float4 *partials;          // [U_max][Pv][2][kDequantWarps][32][4]
    int *err;
};

// GEMM workspace: [0, 256) status word | [256, 256 + kCounterBytes) split-K
// counters | partial tiles.  The counter region has a fixed size so that every
// GEMM sharing one workspace (the launches of a verify step, the two MoE
// projections) finds its counters at the same place, left zero by the last
// launch; partial tiles are always written before they are read.
constexpr size_t kCounterBytes = size_t(1) << 18;      // 65536 counters
constexpr size_t kMaxCounters = kCounterBytes / sizeof(unsigned);
size_t gemm_workspace_bytes(int K, int N, int G, int u_max, int Pv);
void gemm_bind_workspace(GemmArgs &a, void *ws, int u_max);
// Encodes a.xmap for activations x (bf16) [U][R][ldx] with problem stride
// x_stride elements (0: shared by all problems).  Returns false (with a message)
// if the driver rejects the description.
bool gemm_encode_x(GemmArgs &a, const uint16_t *x, int ldx, long long x_stride, int u_max, const char **why);
cudaError_t launch_w4_gemm(const GemmArgs &a, int u_max, cudaStream_t s);
// interleave_gate_up: rows [0, N/2) are gate rows, [N/2, N) up rows; they are
// packed so that lanes 0-15 of every 32-row warp slice hold 16 gate rows and
// lanes 16-31 the matching up rows (the layout kSwiGluBf16 expects).
cudaError_t launch_pack_w4(const uint8_t *codes, const uint16_t *scales, int K, int N, int G, void *packed,
                           bool interleave_gate_up, cudaStream_t s);
int device_sm_count();

}  // namespace tfk
