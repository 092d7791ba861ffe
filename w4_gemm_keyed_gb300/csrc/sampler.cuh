// Keyed sampler and acceptance: declarations shared with the C ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tfk {

constexpr int kSampleChunk = 4096;     // vocabulary entries per top-k CTA
constexpr int kSampleThreads = 256;
constexpr int kMaxTopK = 64;

struct SampleArgs {
    const float *logits;
    int ldl;
    int R, V;
    int k_eff;            // 1 for greedy, else k' = min(top_k or V, V); > 64 takes the general path
    float temperature;
    float top_p;
    uint64_t seed;
    const int64_t *pos;   // dev [R] (or pos_base when pos_scalar)
    const int64_t *pos_base;  // dev [1]: row r at *pos_base + r (used when pos == nullptr)
    int32_t *tokens;
    // workspace
    float *cand_val;      // [R][n_chunks][64]
    int32_t *cand_id;     // [R][n_chunks][64]
    int32_t *cand_cnt;    // [R][n_chunks]
    uint64_t *cand_kth;   // [R][n_chunks]: (key, id) of the chunk's k-th best when it kept k_eff, else 0
    int32_t *row_bad;     // [R]
    // general candidate path (k' > kMaxTopK)
    uint64_t *gen_cmax;   // [R][n_chunks] largest composite key of each chunk
    uint64_t *gen_thr;    // [R] smallest composite key kept
    uint64_t *gen_q;      // [R][V] floor(2^53 exp((l_i - l_0) / T)) of the k' candidates, else 0
    uint64_t *gen_zp;     // [R][n_sub] sum of gen_q over each 1024-entry sub-chunk (exact)
    void *gen_walk;       // [3][R][256] top-p walk bins
    void *gen_state;      // [R] top-p walk state
    double *gen_bscore;   // [R][n_sub] best score of each sub-chunk
    int32_t *gen_bid;     // [R][n_sub] its token id
    int n_sub;            // 1024-entry sub-chunks of the vocabulary
    int *err;
    int n_chunks;
    // acceptance (accepted non-null): a = first i < R - 1 with drafts[i] !=
    // tokens[i], else R - 1; *accepted = a, *bonus = tokens[a] (bonus may be
    // null), *acc_pos += a + 1 (acc_pos may be null)
    const int32_t *drafts;
    int32_t *accepted;
    int32_t *bonus;
    int64_t *acc_pos;
    unsigned *done;       // workspace counter of finished rows, zero between calls
    uint64_t *bound;      // [R] candidate epilogue's shared bounds: zeroed by finalize_lists
};

size_t sample_workspace_bytes(int R, int V);
void sample_bind_workspace(SampleArgs &a, void *ws_region, int R, int V);
cudaError_t launch_keyed_sample(const SampleArgs &a, cudaStream_t s);
int sample_max_vocab();

// Candidates from the LM head's epilogue: nc lists of k_eff (logit, id) per row
// (every list padded to k_eff with the empty entry: value bits 0xFFFFFFFF, id
// -1) in the cand_* arrays with chunk stride nc.  finalize alone then merges
// them, applies top-p and draws the token.
size_t sample_candidate_bytes(int R, int nc);
void sample_bind_candidates(SampleArgs &a, void *region, int R, int nc);
bool sample_candidates_fit(int nc, int k_eff);
cudaError_t launch_sample_finalize(const SampleArgs &a, cudaStream_t s);
// Acceptance; if last_token / pos are non-null also writes the bonus to
// *last_token and advances *pos by a + 1 (device-side chaining of steps).
cudaError_t launch_accept(const int32_t *drafts, const int32_t *sampled, int R, int32_t *accepted,
                          int32_t *bonus, int64_t *pos, cudaStream_t s);

// Key and Gumbel noise of n (seed, position, token) triples, by the functions
// the sampler uses (h_out or g_out may be null).
cudaError_t launch_keyed_hash(const uint64_t *seed, const int64_t *pos, const int32_t *token, long long n,
                              uint64_t *h_out, double *g_out, cudaStream_t s);

}  // namespace tfk
