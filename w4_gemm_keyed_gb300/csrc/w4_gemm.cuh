// W4 lane GEMM: shared declarations between the kernel file and the C ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tfk {

// ---- packed weight layout --------------------------------------------------
// A "tile" is 256 output features = 4 feature blocks of 64.  For every tile t
// and every 64-wide slice kc of the input features there is one contiguous
// "stage" of 4 chunks (one per feature block).  A chunk holds
//   codes : [mt 0..3][lane 0..31][4 x u32]   2048 B
//   scales: [grp][g 0..7][mt 0..3] half2     128 B per group (64/G groups)
// Lane (g = lane/4, q = lane%4) of a warp owns, for the 16-feature sub-tile mt
// and the 16-wide k step j, the 32-bit word j of its 16-byte entry.  Its nibble
// i (bits 4i..4i+3) / 16+4i.. holds, as offset-binary (code + 8):
//   i=0: (f=g,   k=2q | 2q+1)      i=1: (f=g+8, k=2q | 2q+1)
//   i=2: (f=g,   k=2q+8 | 2q+9)    i=3: (f=g+8, k=2q+8 | 2q+9)
// low half = the even k, high half = the odd k: exactly the m16n8k16 A
// fragment, so one LOP3 per register turns it into bf16 (128 + u).
constexpr int kBlocks = 4;                 // feature blocks per tile
constexpr int kTileN = 64 * kBlocks;       // 256
constexpr int kKChunk = 64;                // k per stage
constexpr int kKGroups = 2;                // consumer warp groups splitting the stages
constexpr int kConsumerWarps = kBlocks * kKGroups;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + one producer warp
constexpr int kStages = 14;
constexpr int kXRowStride = 144;           // staged activation row: 128 B + 16 B pad (conflict-free ldmatrix)
constexpr int kXStageBytes = 16 * kXRowStride;
constexpr int kMaxRows = 16;

__host__ __device__ constexpr int chunk_bytes(int G) { return 2048 + 128 * (kKChunk / G); }
__host__ __device__ constexpr int stage_w_bytes(int G) { return kBlocks * chunk_bytes(G); }
// Per consumer warp: 4 sub-tiles x 2 row-halves x 32 lanes x float4.
constexpr int kWarpAccFloats = 4 * 2 * 32 * 4;
constexpr size_t kSlotBytes = size_t(kBlocks) * kWarpAccFloats * 4;   // one partial tile, 16 KB

inline size_t gemm_smem_bytes(int G) {
    return size_t(kStages) * (stage_w_bytes(G) + kXStageBytes)   // weight + activation stages
           + size_t(kBlocks) * kWarpAccFloats * 4                 // cross-group reduction buffer
           + size_t(2 * kStages) * 8;                             // full / empty barriers
}

inline bool packed_shape_ok(int K, int N, int G) {
    return K > 0 && N > 0 && (G == 32 || G == 64) && K % kKChunk == 0;
}
inline size_t packed_bytes(int K, int N, int G) {
    if (!packed_shape_ok(K, N, G)) return 0;
    size_t T = (size_t(N) + kTileN - 1) / kTileN;
    return T * size_t(K / kKChunk) * size_t(stage_w_bytes(G));
}

// ---- launch description ------------------------------------------------------
// A launch runs U problems (U = 1 for a plain linear layer; U = touched experts
// for the MoE layer).  Problem u uses weights at w + expert(u) * w_stride,
// activations x + u * x_stride and writes y + u * y_stride.  Each problem's
// tile x k-slice iteration space is cut into Pv contiguous ranges ("virtual
// CTAs", stream-K style); the cut depends only on (T, Kc, Pv).
// Epilogue of a launch.
enum EpilogueMode : int {
    kStoreF32 = 0,      // y (fp32) = result
    kAccumulateF32 = 1, // y (fp32) += result          (residual update)
    kSwiGluBf16 = 2,    // y (bf16 [R][F]) = bf16(silu(gate) * up), weights packed gate/up-interleaved
};

struct GemmArgs {
    const uint8_t *w;
    long long w_stride;        // bytes between experts
    const int *expert_ids;     // dev [U_max] or nullptr (expert = u)
    const int *n_problems;     // dev count or nullptr (1)
    const uint16_t *x;
    long long x_stride;        // elements between problems
    int ldx;
    void *y;                   // fp32, or bf16 for kSwiGluBf16
    long long y_stride;        // elements between problems
    int ldy;
    int mode;                  // EpilogueMode
    int F;                     // kSwiGluBf16: width of h (N = 2F)
    int R, K, N, G;
    int T, Kc, Pv;
    unsigned *counters;        // [U_max][T][kBlocks], zero between launches
    float4 *partials;          // [U_max][Pv][2][kBlocks][8][32]
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
// Fills counters/partials pointers inside `a` from a workspace region.
void gemm_bind_workspace(GemmArgs &a, void *ws, int u_max);
cudaError_t launch_w4_gemm(const GemmArgs &a, int u_max, cudaStream_t s);
// interleave_gate_up: rows [0, N/2) are gate rows, [N/2, N) up rows; they are
// packed so that each 32-feature group holds 16 gate rows then the 16 matching
// up rows (the layout kSwiGluBf16 expects).
cudaError_t launch_pack_w4(const uint8_t *codes, const uint16_t *scales, int K, int N, int G, void *packed,
                           bool interleave_gate_up, cudaStream_t s);
int device_sm_count();

}  // namespace tfk
