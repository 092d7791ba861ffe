// W4 lane GEMM: shared declarations between the kernel file and the C ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tfk {

// ---- packed weight layout --------------------------------------------------
// Output features are grouped in tiles of 128 = 4 "feature blocks" of 32 rows
// (one consumer warp per k-group each).  For every tile t and every 64-wide
// slice kc of the input features there is one contiguous "chunk", and
// consecutive kc of a tile are consecutive in memory, so any run of iterations
// of one tile is one bulk copy.  A chunk is 4 feature blocks; a block holds
//   codes : [mt 0..1][lane 0..31][16 B]       1024 B
//   scales: [grp][g 0..7][mt 0..1] half2      64 B per quantisation group
// Lane (g = lane/4, q = lane%4) of the warp owns, for the 16-row sub-tile mt and
// the 16-wide k step j, word j of its 16-byte entry.  Its nibble pairs
// (bits 4i / 16+4i, offset binary code + 8) are the m16n8k16 A fragment:
//   i=0: (row g,   k 2q | 2q+1)      i=1: (row g+8, k 2q | 2q+1)
//   i=2: (row g,   k 2q+8 | 2q+9)    i=3: (row g+8, k 2q+8 | 2q+9)
// and the half2 (s[row g], s[row g+8]) of each sub-tile are the lane's scales.
constexpr int kBlockRows = 32;             // weight rows per consumer warp
constexpr int kFeatWarps = 4;              // feature blocks per tile
constexpr int kTileN = kBlockRows * kFeatWarps;   // 128 output features per tile
constexpr int kKChunk = 64;                // k per iteration
constexpr int kRows = 16;                  // verify rows (MMA columns), zero-padded
constexpr int kKGroups = 4;                // consumer warp groups taking every fourth k slice
constexpr int kConsumerWarps = kFeatWarps * kKGroups;
constexpr int kThreads = 32 * (kConsumerWarps + 1);   // + one producer warp
constexpr int kStageIters = 8;             // iterations per pipeline stage (one weight copy of ~35 KB)
constexpr int kStages = 3;
constexpr int kPreWaitStages = 2;   // weight stages requested before the grid-dependency wait

// Activation slice in shared memory: [rows][64 k] bf16, 128-byte swizzled; 16
// rows when the launch has more than 8, else 8 (rows >= R are zero-filled).
__host__ __device__ constexpr int x_rows(bool hi) { return hi ? kRows : kRows / 2; }
__host__ __device__ constexpr int x_slice_bytes(bool hi) { return x_rows(hi) * kKChunk * 2; }
__host__ __device__ constexpr int x_stage_bytes(bool hi) { return kStageIters * x_slice_bytes(hi); }
constexpr int kLaneAccHi = 16;             // fp32 accumulators per lane: 2 sub-tiles x 2 row-halves x 4
// fp32 values per lane exchanged by the k-group combine and the split-K fixup:
// rows 8..15 (accumulator half n = 1) only when the launch has them
__host__ __device__ constexpr int lane_vals(bool hi) { return hi ? kLaneAccHi : kLaneAccHi / 2; }
// k-group combine of a whole tile: each k-group ends with one quarter of every
// lane's sums (accumulator element c = its k-group) and stores it.  A lane
// writes the three quarters it does not keep: per buffer [fw][quarter][3][32]
// of lane_vals / 4 floats; two buffers alternate between segment ends.  The
// split-tile combine of feature block fw (all sums to k-group 0) uses the
// start of fw's part of buffer 0.
__host__ __device__ constexpr int comb_buf_floats(bool hi) {
    return kFeatWarps * kKGroups * (kKGroups - 1) * 32 * (lane_vals(hi) / kKGroups);
}

// Weight formats of a packed matrix.
enum WeightFormat : int {
    kFmtSym = 0,     // symmetric int4 codes, one fp16 scale per (row, group of G)
    kFmtAffine = 1,  // MLX-style affine: unsigned codes, bf16 scale and bias per (row, group of G)
    kFmtNvfp4 = 2,   // NVFP4: E2M1 codes, one E4M3 scale per (row, 16 features), fp32 tensor scale
};
// Affine (MLX-style) blocks also carry one bf16 bias per row and group after the
// bf16 scales: [grp][scales 64 B][biases 64 B].  NVFP4 blocks carry the E4M3
// scale bytes of the block's four 16-wide k steps: [g 0..7][j 0..3][mt 0..1]
// (s[row g], s[row g+8]), 128 B.
__host__ __device__ constexpr int block_bytes(int G, int fmt = kFmtSym) {
    return fmt == kFmtNvfp4 ? 1024 + 128 : 1024 + (fmt == kFmtAffine ? 128 : 64) * (kKChunk / G);
}
__host__ __device__ constexpr int chunk_bytes(int G, int fmt = kFmtSym) { return kFeatWarps * block_bytes(G, fmt); }
// One partial tile of the split-K fixup: 4 feature warps x 32 lanes x 16 floats.
constexpr size_t kSlotBytes = size_t(kFeatWarps) * 32 * kLaneAccHi * 4;

// Pipeline depth: three stages of ~35 KB (measured faster than four, and than
// smaller copies in more stages).
__host__ __device__ constexpr int num_stages(int, bool, int) { return kStages; }

// Candidate epilogue (LM head): kSelWarps extra warps, the selectors, keep
// for every row the kSelList best (logit, id) words of the feature blocks its
// CTA stores.  A storing consumer warp takes a ticket, waits for slot
// ticket % kSelSlots of one shared ring to be free, writes its finished
// 32-feature block there ([rows][kSelStride] fp32; the stride keeps the
// lanes' stores on distinct banks) and signals the slot's barrier; the
// selectors take the slots in ticket order.
constexpr int kSelSlots = 16;
constexpr int kSelStride = 36;
constexpr int kSelList = 64;
constexpr int kSelMaxRows = 8;             // launches of up to 8 rows only: at 16 rows the consumers are
                                           // issue-bound and the selectors' scan slows them (measured)
constexpr int kSelWarps = 3;               // selector warps; row r belongs to warp r % kSelWarps (20 warps
                                           // in all keep 96 registers a thread; 21 cap them at 80)
__host__ __device__ constexpr int sel_ring_bytes(bool hi) { return kSelSlots * x_rows(hi) * kSelStride * 4; }
__host__ __device__ constexpr int sel_smem_bytes(bool hi) {
    return sel_ring_bytes(hi) + 256                   // ring + slot headers and the ticket counter
           + 2 * kSelSlots * 8                        // full / empty barriers
           + x_rows(hi) * kSelList * 8                // per-row lists
           + x_rows(hi) * 32 * 8                      // per-row pending words
           + 64;                                      // pending counts
}

inline size_t gemm_smem_bytes(int G, bool hi, int fmt = kFmtSym, bool sel = false) {
    const int ns = num_stages(G, hi, fmt);
    return 1024                                                         // alignment slack
           + size_t(ns) * x_stage_bytes(hi)                             // activation slices (1024-B aligned)
           + size_t(ns) * kStageIters * chunk_bytes(G, fmt)            // weight stages
           + 2 * size_t(comb_buf_floats(hi)) * 4                        // k-group combine buffers
           + 256                                                        // barriers
           + (sel ? size_t(sel_smem_bytes(hi)) : 0);
}

inline bool packed_shape_ok(int K, int N, int G) {
    return K > 0 && N > 0 && (G == 32 || G == 64) && K % kKChunk == 0;
}
inline size_t packed_bytes(int K, int N, int G, int fmt = kFmtSym) {
    if (fmt == kFmtNvfp4 ? !(K > 0 && N > 0 && K % kKChunk == 0) : !packed_shape_ok(K, N, G)) return 0;
    size_t T = (size_t(N) + kTileN - 1) / kTileN;
    return T * size_t(K / kKChunk) * size_t(chunk_bytes(G, fmt));
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
    int list_ready;            // expert_ids / n_problems were written before the preceding grid started
    int x_per_problem;         // activations differ per problem (use coordinate u)
    void *y;                   // fp32, or bf16 for kSwiGluBf16
    long long y_stride;        // elements between problems
    int ldy;
    int mode;                  // EpilogueMode
    int F;                     // kSwiGluBf16: width of h (N = 2F)
    int R, K, N, G;
    int fmt;                   // WeightFormat of the packed weights
    float gscale;              // kFmtNvfp4: tensor scale applied to every output (else 1)
    int T, Kc, Pv;
    unsigned *counters;        // [U_max][T][kFeatWarps], zero between launches
    float4 *partials;          // [U_max][Pv][2][kFeatWarps][32][4]
    int *err;
    // candidate epilogue (launch_w4_gemm_select; dense launches only): CTA c
    // writes, for every row r, its sel_k best (logit, id) in descending order
    // at [r][c][0..sel_k) of sel_val / sel_id (padded with value bits
    // 0xFFFFFFFF and id -1), sel_cnt[r][c] = sel_k and sel_kth[r][c] = its
    // sel_k-th best word (0 if it saw fewer); rows with a non-finite logit
    // set sel_bad[r].  y may be null (no logits stored).  CTAs share, per
    // row, the largest k'-th best any of them has reached (sel_bound): a
    // word at or below it cannot be among the row's k' best, so no CTA keeps
    // it; a list may then hold fewer than sel_k words (padded).
    int sel_k;
    int sel_nc;                // chunk stride of the candidate arrays = the launch's grid size
    float *sel_val;
    int32_t *sel_id;
    int32_t *sel_cnt;
    uint64_t *sel_kth;
    int32_t *sel_bad;
    uint64_t *sel_bound;       // [R], zero before the launch: the largest k'-th best any CTA has published
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
// Grid size of a launch of a (one CTA per work item, at most one per SM).
int gemm_grid(const GemmArgs &a, int u_max);
// Dense symmetric-int4 launch with the candidate epilogue (a.sel_* set, sel_nc
// = gemm_grid(a, 1), 1 <= sel_k <= kSelList, R <= kSelMaxRows).
cudaError_t launch_w4_gemm_select(const GemmArgs &a, cudaStream_t s);
// interleave_gate_up: rows [0, N/2) are gate rows, [N/2, N) up rows; they are
// packed so that each 32-row feature block holds 16 gate rows (sub-tile 0) and
// the 16 matching up rows (sub-tile 1), the layout kSwiGluBf16 expects.
// MLX-style affine weights: codes uint32 [N][K/8] (element i of a word in bits
// 4i..4i+3, unsigned), scales and biases bf16 [N][K/G].
// NVFP4 weights: codes uint8 [N][K/2] (E2M1, element 2j in the low nibble of
// byte j), block scales uint8 [N][K/16] (E4M3 bit patterns).
cudaError_t launch_pack_nvfp4(const uint8_t *codes, const uint8_t *scales, int K, int N, void *packed,
                              cudaStream_t s);
cudaError_t launch_pack_w4_affine(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases, int K, int N,
                                  int G, void *packed, cudaStream_t s);
cudaError_t launch_pack_w4(const uint8_t *codes, const uint16_t *scales, int K, int N, int G, void *packed,
                           bool interleave_gate_up, cudaStream_t s);
int device_sm_count();

}  // namespace tfk
