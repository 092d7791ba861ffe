// extern "C" entry points of libtf: argument validation, workspace layout and
// launch sequencing.  Every step of the verify pass runs in this library's own
// kernels (w4_gemm.cu, sampler.cu, glue.cu, attention.cu); nothing here computes
// on the host.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/tf.h"
#include "attention.cuh"
#include "glue.cuh"
#include "sampler.cuh"
#include "w4_gemm.cuh"

using namespace tfk;

namespace {

thread_local std::string g_error;

tf_status fail(tf_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_error = buf;
    return st;
}

tf_status ok() {
    g_error.clear();
    return TF_OK;
}

tf_status cuda_fail(cudaError_t e, const char *what) {
    return fail(TF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round256(size_t b) { return (b + 255) / 256 * 256; }


// Ranges of a dense launch.  When an even share of m whole tiles per CTA
// (m = 1..4) nearly fills the SMs, no tile is split (no split-K fixup);
// otherwise a stream-K split over all SMs.  The choice depends on the shape
// only, never on R.
int dense_pv(int T, int Kc) {
    const long long tot = (long long)T * Kc;
    int sms = device_sm_count();
    if (sms <= 0) sms = 1;
    for (int m = 1; m <= 4; ++m)
        if (T % m == 0 && T / m <= sms && 8LL * (T / m) >= 7LL * sms) return T / m;
    return int(tot < sms ? tot : sms);
}

// Ranges of a grouped (MoE) launch: one whole tile each, so no expert tile is
// split and no split-K fixup runs; the persistent CTAs spread the
// experts x tiles items.  Depends on the shape only, never on R.
int grouped_pv(int T, int Kc) {
    (void)Kc;
    return T;
}

tf_status check_matrix(const tf_w4_matrix *W, const char *name) {
    if (!W) return fail(TF_ERR_INVALID_ARG, "%s: null matrix", name);
    if (!W->packed) return fail(TF_ERR_INVALID_ARG, "%s: null packed pointer", name);
    if (!aligned(W->packed, 256)) return fail(TF_ERR_INVALID_ARG, "%s: packed pointer not 256-B aligned", name);
    if (W->group != 32 && W->group != 64) return fail(TF_ERR_UNSUPPORTED, "%s: group %d not in {32, 64}", name, W->group);
    if (W->K <= 0 || W->K % kKChunk) return fail(TF_ERR_UNSUPPORTED, "%s: K=%d is not a positive multiple of 64", name, W->K);
    if (W->N <= 0) return fail(TF_ERR_INVALID_ARG, "%s: N=%d must be >= 1", name, W->N);
    if (W->affine != 0 && W->affine != 1) return fail(TF_ERR_INVALID_ARG, "%s: affine must be 0 or 1", name);
    if ((long long)((W->N + kTileN - 1) / kTileN) * (W->K / kKChunk) > 0x7FFFFFFFLL)
        return fail(TF_ERR_UNSUPPORTED, "%s: K x N too large for the split-K index space", name);
    return TF_OK;
}

tf_status check_ws(const void *ws, size_t ws_bytes, size_t need) {
    if (!ws) return fail(TF_ERR_WORKSPACE, "null workspace");
    if (!aligned(ws, 256)) return fail(TF_ERR_WORKSPACE, "workspace not 256-B aligned");
    if (ws_bytes < need) return fail(TF_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    return TF_OK;
}

tf_status check_sampling(const tf_sampling *p, int V, int *k_eff) {
    if (!p) return fail(TF_ERR_INVALID_ARG, "null sampling parameters");
    if (!std::isfinite(p->temperature) || p->temperature < 0.f)
        return fail(TF_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (std::isnan(p->top_p)) return fail(TF_ERR_INVALID_ARG, "top_p is NaN");
    if (p->temperature == 0.f) {
        *k_eff = 1;
        return TF_OK;
    }
    // k' <= kMaxTopK takes the fast candidate path, larger k' the general one
    *k_eff = (p->top_k <= 0 || p->top_k >= V) ? V : p->top_k;
    return TF_OK;
}

GemmArgs dense_args(const tf_w4_matrix &W, int R, void *y, int ldy, int mode) {
    GemmArgs a{};
    a.w = static_cast<const uint8_t *>(W.packed);
    a.y = y;
    a.ldy = ldy;
    a.mode = mode;
    a.F = W.N / 2;
    a.R = R;
    a.K = W.K;
    a.N = W.N;
    a.G = W.group;
    a.fmt = W.affine ? kFmtAffine : kFmtSym;
    a.gscale = 1.0f;
    a.T = (W.N + kTileN - 1) / kTileN;
    a.Kc = W.K / kKChunk;
    a.Pv = dense_pv(a.T, a.Kc);
    return a;
}

// Binds the workspace, encodes the activation tensor map and launches.
cudaError_t bind_and_launch(GemmArgs &a, const uint16_t *x, int ldx, long long x_stride, int u_max, void *ws,
                            cudaStream_t s, const char **why) {
    gemm_bind_workspace(a, ws, u_max);
    if (!gemm_encode_x(a, x, ldx, x_stride, u_max, why)) return cudaErrorInvalidValue;
    return launch_w4_gemm(a, u_max, s);
}

size_t dense_gemm_ws(const tf_w4_matrix &W) {
    const int T = (W.N + kTileN - 1) / kTileN;
    return gemm_workspace_bytes(W.K, W.N, W.group, 1, dense_pv(T, W.K / kKChunk));
}

// ---- LM head + keyed sampling ----
// Fused when the matrix is symmetric int4, R <= 8 and every CTA's k'
// candidates fit the finaliser's pool: the GEMM's selector warps leave
// per-CTA candidate lists, and the finaliser alone merges them.  Otherwise the GEMM writes the
// logits and the whole sampler runs on them.  Both give the same tokens: the
// finaliser sees the same k' best (logit, id) in the same order.
struct LmLayout {
    size_t gemm, sample, logits, total;
};

int lmhead_grid(const tf_w4_matrix &W) {
    GemmArgs a = dense_args(W, 1, nullptr, W.N, kStoreF32);
    return gemm_grid(a, 1);
}

LmLayout lm_layout(const tf_w4_matrix &W, int R) {
    LmLayout l{};
    size_t off = round256(dense_gemm_ws(W));
    l.gemm = 0;
    l.sample = off;
    const size_t full = sample_workspace_bytes(R, W.N), cand = sample_candidate_bytes(R, lmhead_grid(W));
    off += round256(full > cand ? full : cand);
    l.logits = off;
    off += round256(size_t(R) * W.N * 4);
    l.total = off;
    return l;
}

bool lmhead_fused(const tf_w4_matrix &W, int R, int k_eff) {
    return !W.affine && R <= kSelMaxRows && sample_candidates_fit(lmhead_grid(W), k_eff);
}

// gemm_ws: a GEMM workspace (status word first, also the sampler's);
// sample_ws: >= max(sample_workspace_bytes, sample_candidate_bytes) bytes;
// logits: where to store the logits (may be null when fused; then the
// unfused path uses scratch).  pos per row, or pos_base + r when pos is null.
// accepted non-null: the finaliser also accepts (drafts, bonus, acc_pos as in
// SampleArgs).
cudaError_t run_lmhead_sample(const tf_w4_matrix &W, const uint16_t *x, int ldx, int R, const tf_sampling &p,
                              int k_eff, uint64_t seed, const int64_t *pos, const int64_t *pos_base, int32_t *tokens,
                              float *logits, int ldl, float *scratch, void *gemm_ws, void *sample_ws,
                              const int32_t *drafts, int32_t *accepted, int32_t *bonus, int64_t *acc_pos,
                              cudaStream_t s, const char **why) {
    int *err = static_cast<int *>(gemm_ws);
    SampleArgs sa{};
    sa.drafts = drafts;
    sa.accepted = accepted;
    sa.bonus = bonus;
    sa.acc_pos = acc_pos;
    sa.R = R;
    sa.V = W.N;
    sa.k_eff = k_eff;
    sa.temperature = p.temperature;
    sa.top_p = p.top_p;
    sa.seed = seed;
    sa.pos = pos;
    sa.pos_base = pos_base;
    sa.tokens = tokens;
    sa.err = err;
    if (!sa.pos && !sa.pos_base) sa.pos = reinterpret_cast<const int64_t *>(gemm_ws);   // greedy: never read
    if (lmhead_fused(W, R, k_eff)) {
        GemmArgs a = dense_args(W, R, logits, logits ? ldl : W.N, kStoreF32);
        const int nc = gemm_grid(a, 1);
        sample_bind_candidates(sa, sample_ws, R, nc);
        a.sel_k = k_eff;
        a.sel_nc = nc;
        a.sel_val = sa.cand_val;
        a.sel_id = sa.cand_id;
        a.sel_cnt = sa.cand_cnt;
        a.sel_kth = sa.cand_kth;
        a.sel_bad = sa.row_bad;
        a.sel_bound = sa.bound;
        gemm_bind_workspace(a, gemm_ws, 1);
        if (!gemm_encode_x(a, x, ldx, 0, 1, why)) return cudaErrorInvalidValue;
        cudaError_t e = launch_w4_gemm_select(a, s);
        if (e == cudaSuccess) e = launch_sample_finalize(sa, s);
        return e;
    }
    float *lg = logits ? logits : scratch;
    const int ld = logits ? ldl : W.N;
    GemmArgs a = dense_args(W, R, lg, ld, kStoreF32);
    cudaError_t e = bind_and_launch(a, x, ldx, 0, 1, gemm_ws, s, why);
    if (e != cudaSuccess) return e;
    sa.logits = lg;
    sa.ldl = ld;
    sample_bind_workspace(sa, sample_ws, R, W.N);
    return launch_keyed_sample(sa, s);
}

// ---- MoE workspace layout ----
struct MoeLayout {
    size_t gemm, ids, w, expert_ids, nprob, slot_of, h, Y, total;
    int u_max;
};

MoeLayout moe_layout(const tf_moe_layer &L, int R) {
    MoeLayout m{};
    m.u_max = L.n_experts < L.top_k * R ? L.n_experts : L.top_k * R;
    const int Tgu = (2 * L.ffn + kTileN - 1) / kTileN, Td = (L.hidden + kTileN - 1) / kTileN;
    const size_t g1 = gemm_workspace_bytes(L.hidden, 2 * L.ffn, L.group, m.u_max, grouped_pv(Tgu, L.hidden / kKChunk));
    const size_t g2 = gemm_workspace_bytes(L.ffn, L.hidden, L.group, m.u_max, grouped_pv(Td, L.ffn / kKChunk));
    size_t off = round256(g1 > g2 ? g1 : g2);
    m.gemm = 0;
    m.ids = off;
    off += round256(size_t(R) * kMaxRouteK * 4);
    m.w = off;
    off += round256(size_t(R) * kMaxRouteK * 4);
    m.expert_ids = off;
    off += round256(size_t(kMaxExperts) * 4);
    m.nprob = off;
    off += 256;
    m.slot_of = off;
    off += round256(size_t(R) * kMaxRouteK * 4);
    m.h = off;
    off += round256(size_t(m.u_max) * R * L.ffn * 2);
    m.Y = off;
    off += round256(size_t(m.u_max) * R * L.hidden * 4);
    m.total = off;
    return m;
}

tf_status check_moe(const tf_moe_layer *L) {
    if (!L) return fail(TF_ERR_INVALID_ARG, "null MoE layer");
    {
        const size_t T = size_t((2 * size_t(L->ffn > 0 ? L->ffn : 0) + kTileN - 1) / kTileN) +
                         size_t((L->hidden > 0 ? L->hidden : 0) + kTileN - 1) / kTileN;
        if (T * kFeatWarps * size_t(kMaxExperts) > kMaxCounters)
            return fail(TF_ERR_UNSUPPORTED, "MoE layer too large for the split-K counter region");
    }
    if (!L->gate_up || !L->down) return fail(TF_ERR_INVALID_ARG, "null MoE weights");
    if (!aligned(L->gate_up, 256) || !aligned(L->down, 256))
        return fail(TF_ERR_INVALID_ARG, "MoE weights not 256-B aligned");
    if (L->group != 32 && L->group != 64) return fail(TF_ERR_UNSUPPORTED, "group %d not in {32, 64}", L->group);
    if (L->hidden <= 0 || L->hidden % kKChunk || L->ffn <= 0 || L->ffn % kKChunk)
        return fail(TF_ERR_UNSUPPORTED, "hidden and ffn must be positive multiples of 64");
    if (L->n_experts < 1 || L->n_experts > kMaxExperts)
        return fail(TF_ERR_UNSUPPORTED, "n_experts must be in [1, %d]", kMaxExperts);
    if (L->top_k < 1 || L->top_k > kMaxRouteK || L->top_k > L->n_experts)
        return fail(TF_ERR_UNSUPPORTED, "top_k must be in [1, min(8, n_experts)]");
    return TF_OK;
}

// ---- verify-step workspace layout ----
struct StepLayout {
    size_t gemm, sample, x, n, h, logits, total;
};

StepLayout step_layout(const tf_model &m, int R) {
    StepLayout s{};
    size_t g = dense_gemm_ws(m.lm_head);
    for (int b = 0; b < m.n_blocks; ++b) {
        const size_t g1 = dense_gemm_ws(m.gate_up[b]), g2 = dense_gemm_ws(m.down[b]);
        g = g1 > g ? g1 : g;
        g = g2 > g ? g2 : g;
    }
    size_t off = round256(g);
    s.gemm = 0;
    s.sample = off;
    {
        const size_t full = sample_workspace_bytes(R, m.vocab), cand = sample_candidate_bytes(R, lmhead_grid(m.lm_head));
        off += round256(full > cand ? full : cand);
    }
    s.x = off;
    off += round256(size_t(R) * m.hidden * 4);
    s.n = off;
    off += round256(size_t(R) * m.hidden * 2);
    s.h = off;
    off += round256(size_t(R) * m.ffn * 2);
    s.logits = off;
    off += round256(size_t(R) * m.vocab * 4);
    s.total = off;
    return s;
}

tf_status check_model(const tf_model *m) {
    if (!m) return fail(TF_ERR_INVALID_ARG, "null model");
    if (!m->embedding || !m->gate_up || !m->down) return fail(TF_ERR_INVALID_ARG, "null model pointer");
    if (m->n_blocks < 0) return fail(TF_ERR_INVALID_ARG, "n_blocks < 0");
    if (m->vocab < 1 || m->vocab > sample_max_vocab())
        return fail(TF_ERR_UNSUPPORTED, "vocab must be in [1, %d]", sample_max_vocab());
    if (!(m->rms_eps >= 0.f) || !std::isfinite(m->rms_eps)) return fail(TF_ERR_INVALID_ARG, "bad rms_eps");
    for (int b = 0; b < m->n_blocks; ++b) {
        tf_status st = check_matrix(&m->gate_up[b], "gate_up");
        if (st) return st;
        if ((st = check_matrix(&m->down[b], "down"))) return st;
        if (m->gate_up[b].affine || m->down[b].affine)
            return fail(TF_ERR_UNSUPPORTED, "block %d: the decoder takes symmetric matrices", b);
        if (m->gate_up[b].K != m->hidden || m->gate_up[b].N != 2 * m->ffn || m->down[b].K != m->ffn ||
            m->down[b].N != m->hidden || m->gate_up[b].group != m->group || m->down[b].group != m->group)
            return fail(TF_ERR_INVALID_ARG, "block %d: matrix shapes do not match the model", b);
    }
    tf_status st = check_matrix(&m->lm_head, "lm_head");
    if (st) return st;
    if (m->lm_head.affine) return fail(TF_ERR_UNSUPPORTED, "lm_head: the decoder takes symmetric matrices");
    if (m->lm_head.K != m->hidden || m->lm_head.N != m->vocab)
        return fail(TF_ERR_INVALID_ARG, "lm_head shape does not match the model");
    if (m->hidden % kKChunk || m->ffn % kKChunk) return fail(TF_ERR_UNSUPPORTED, "hidden, ffn must be multiples of 64");
    if (size_t((m->vocab + kTileN - 1) / kTileN) * kFeatWarps > kMaxCounters ||
        size_t((2 * size_t(m->ffn) + kTileN - 1) / kTileN) * kFeatWarps > kMaxCounters)
        return fail(TF_ERR_UNSUPPORTED, "model too large for the split-K counter region");
    return TF_OK;
}

cudaError_t run_block(const tf_model &m, int b, float *x, int R, uint16_t *n, uint16_t *h, void *ws,
                      cudaStream_t s, const char **why) {
    cudaError_t e = launch_rmsnorm_bf16(x, R, m.hidden, m.rms_eps, n, s);
    if (e != cudaSuccess) return e;
    GemmArgs g1 = dense_args(m.gate_up[b], R, h, m.ffn, kSwiGluBf16);
    e = bind_and_launch(g1, n, m.hidden, 0, 1, ws, s, why);
    if (e != cudaSuccess) return e;
    GemmArgs g2 = dense_args(m.down[b], R, x, m.hidden, kAccumulateF32);
    return bind_and_launch(g2, h, m.ffn, 0, 1, ws, s, why);
}

size_t block_gemm_ws(const tf_model &m) {
    size_t g = 256;
    for (int b = 0; b < m.n_blocks; ++b) {
        const size_t g1 = dense_gemm_ws(m.gate_up[b]), g2 = dense_gemm_ws(m.down[b]);
        g = g1 > g ? g1 : g;
        g = g2 > g ? g2 : g;
    }
    return g;
}

}  // namespace

extern "C" {

const char *tf_last_error(void) { return g_error.c_str(); }

const char *tf_status_string(tf_status s) {
    switch (s) {
        case TF_OK: return "ok";
        case TF_ERR_INVALID_ARG: return "invalid argument";
        case TF_ERR_UNSUPPORTED: return "unsupported";
        case TF_ERR_CUDA: return "CUDA error";
        case TF_ERR_TIMEOUT: return "device wait timed out";
        case TF_ERR_WORKSPACE: return "bad workspace";
    }
    return "unknown status";
}

int tf_version(void) { return 300; }  // 0.3.0: NVFP4 lane GEMM, device key hash

int32_t tf_device_sm_count(void) { return device_sm_count(); }

tf_status tf_workspace_status(void *ws, void *stream, int32_t *code) {
    if (!ws || !code) return fail(TF_ERR_INVALID_ARG, "null argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof v, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "tf_workspace_status");
    *code = v;
    return ok();
}

size_t tf_w4_packed_bytes(int32_t K, int32_t N, int32_t group) { return packed_bytes(K, N, group); }

size_t tf_w4_affine_packed_bytes(int32_t K, int32_t N, int32_t group) { return packed_bytes(K, N, group, true); }

tf_status tf_pack_w4_affine(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases, int32_t K, int32_t N,
                            int32_t group, void *packed, size_t bytes, void *stream) {
    if (!codes || !scales || !biases || !packed) return fail(TF_ERR_INVALID_ARG, "null pointer");
    if (!packed_shape_ok(K, N, group)) return fail(TF_ERR_UNSUPPORTED, "unsupported shape K=%d N=%d group=%d", K, N, group);
    if (!aligned(packed, 256)) return fail(TF_ERR_INVALID_ARG, "packed buffer not 256-B aligned");
    if (bytes < packed_bytes(K, N, group, true)) return fail(TF_ERR_INVALID_ARG, "packed buffer too small");
    cudaError_t e = launch_pack_w4_affine(codes, scales, biases, K, N, group, packed, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_pack_w4_affine");
    return ok();
}

static tf_status pack_common(const uint8_t *codes, const uint16_t *scales, int32_t K, int32_t N, int32_t group,
                             void *packed, size_t bytes, void *stream, bool inter) {
    if (!codes || !scales || !packed) return fail(TF_ERR_INVALID_ARG, "null pointer");
    if (!packed_shape_ok(K, N, group)) return fail(TF_ERR_UNSUPPORTED, "unsupported shape K=%d N=%d group=%d", K, N, group);
    if (inter && N % 2) return fail(TF_ERR_INVALID_ARG, "gate/up matrix needs an even N");
    if (!aligned(packed, 256)) return fail(TF_ERR_INVALID_ARG, "packed pointer not 256-B aligned");
    if (bytes < packed_bytes(K, N, group)) return fail(TF_ERR_INVALID_ARG, "packed buffer too small");
    cudaError_t e = launch_pack_w4(codes, scales, K, N, group, packed, inter, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_pack_w4");
    return ok();
}

tf_status tf_pack_w4(const uint8_t *codes, const uint16_t *scales, int32_t K, int32_t N, int32_t group, void *packed,
                     size_t packed_bytes_, void *stream) {
    return pack_common(codes, scales, K, N, group, packed, packed_bytes_, stream, false);
}

tf_status tf_pack_w4_gate_up(const uint8_t *codes, const uint16_t *scales, int32_t K, int32_t ffn, int32_t group,
                             void *packed, size_t packed_bytes_, void *stream) {
    if (ffn <= 0) return fail(TF_ERR_INVALID_ARG, "ffn must be >= 1");
    return pack_common(codes, scales, K, 2 * ffn, group, packed, packed_bytes_, stream, true);
}

size_t tf_nvfp4_packed_bytes(int32_t K, int32_t N) { return packed_bytes(K, N, 16, kFmtNvfp4); }

tf_status tf_pack_nvfp4(const uint8_t *codes, const uint8_t *scales, int32_t K, int32_t N, void *packed, size_t bytes,
                        void *stream) {
    if (!codes || !scales || !packed) return fail(TF_ERR_INVALID_ARG, "null pointer");
    if (tf_nvfp4_packed_bytes(K, N) == 0) return fail(TF_ERR_UNSUPPORTED, "unsupported shape K=%d N=%d", K, N);
    if (!aligned(packed, 256)) return fail(TF_ERR_INVALID_ARG, "packed buffer not 256-B aligned");
    if (bytes < tf_nvfp4_packed_bytes(K, N)) return fail(TF_ERR_INVALID_ARG, "packed buffer too small");
    cudaError_t e = launch_pack_nvfp4(codes, scales, K, N, packed, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_pack_nvfp4");
    return ok();
}

size_t tf_lane_gemm_nvfp4_workspace_bytes(int32_t K, int32_t N) {
    if (tf_nvfp4_packed_bytes(K, N) == 0) return 0;
    const int T = (N + kTileN - 1) / kTileN;
    return gemm_workspace_bytes(K, N, 16, 1, dense_pv(T, K / kKChunk));
}

tf_status tf_lane_gemm_nvfp4(const tf_nvfp4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y,
                             int32_t ldy, void *ws, size_t ws_bytes, void *stream) {
    if (!W || !W->packed) return fail(TF_ERR_INVALID_ARG, "W: null matrix or packed pointer");
    if (!aligned(W->packed, 256)) return fail(TF_ERR_INVALID_ARG, "W: packed pointer not 256-B aligned");
    if (tf_nvfp4_packed_bytes(W->K, W->N) == 0)
        return fail(TF_ERR_UNSUPPORTED, "W: K=%d must be a positive multiple of 64 and N=%d >= 1", W->K, W->N);
    if (!std::isfinite(W->global_scale)) return fail(TF_ERR_INVALID_ARG, "W: global_scale must be finite");
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!x || !aligned(x, 16)) return fail(TF_ERR_INVALID_ARG, "x must be non-null and 16-B aligned");
    if (ldx < W->K || ldx % 8) return fail(TF_ERR_INVALID_ARG, "ldx=%d must be >= K and a multiple of 8", ldx);
    if (!y || !aligned(y, 4)) return fail(TF_ERR_INVALID_ARG, "y must be non-null and 4-B aligned");
    if (ldy < W->N) return fail(TF_ERR_INVALID_ARG, "ldy=%d must be >= N", ldy);
    tf_status st = check_ws(ws, ws_bytes, tf_lane_gemm_nvfp4_workspace_bytes(W->K, W->N));
    if (st) return st;
    if (size_t((W->N + kTileN - 1) / kTileN) * kFeatWarps > kMaxCounters)
        return fail(TF_ERR_UNSUPPORTED, "N=%d too large for the split-K counter region", W->N);
    tf_w4_matrix M{W->packed, W->K, W->N, 64, 0};
    GemmArgs a = dense_args(M, R, y, ldy, kStoreF32);
    a.G = 16;
    a.fmt = kFmtNvfp4;
    a.gscale = W->global_scale;
    const char *why = "";
    cudaError_t e = bind_and_launch(a, x, ldx, 0, 1, ws, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "tf_lane_gemm_nvfp4: %s (%s)", cudaGetErrorString(e), why);
    return ok();
}

size_t tf_lane_gemm_workspace_bytes(int32_t K, int32_t N, int32_t group) {
    if (!packed_shape_ok(K, N, group)) return 0;
    tf_w4_matrix W{nullptr, K, N, group};
    return dense_gemm_ws(W);
}

namespace {
tf_status lane_gemm(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y, int32_t ldy,
                    void *ws, size_t ws_bytes, void *stream, int mode, const char *name);
}  // namespace

tf_status tf_lane_gemm_w4(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y, int32_t ldy,
                          void *ws, size_t ws_bytes, void *stream) {
    return lane_gemm(W, x, ldx, R, y, ldy, ws, ws_bytes, stream, kStoreF32, "tf_lane_gemm_w4");
}

tf_status tf_lane_gemm_w4_accumulate(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y,
                                     int32_t ldy, void *ws, size_t ws_bytes, void *stream) {
    return lane_gemm(W, x, ldx, R, y, ldy, ws, ws_bytes, stream, kAccumulateF32, "tf_lane_gemm_w4_accumulate");
}

tf_status tf_cast_bf16(const float *x, int32_t R, int32_t N, int32_t ldx, uint16_t *y, int32_t ldy, void *stream) {
    if (!x || !y) return fail(TF_ERR_INVALID_ARG, "null x or y");
    if (R < 1 || R > 65535 || N < 1) return fail(TF_ERR_INVALID_ARG, "R=%d (1..65535) or N=%d (>= 1) out of range", R, N);
    if (ldx < N || ldy < N) return fail(TF_ERR_INVALID_ARG, "ldx=%d and ldy=%d must be >= N=%d", ldx, ldy, N);
    cudaError_t e = launch_cast_bf16(x, R, N, ldx, y, ldy, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_cast_bf16");
    return ok();
}

namespace {
tf_status lane_gemm(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y, int32_t ldy,
                    void *ws, size_t ws_bytes, void *stream, int mode, const char *name) {
    tf_status st = check_matrix(W, "W");
    if (st) return st;
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!x || !aligned(x, 16)) return fail(TF_ERR_INVALID_ARG, "x must be non-null and 16-B aligned");
    if (ldx < W->K || ldx % 8) return fail(TF_ERR_INVALID_ARG, "ldx=%d must be >= K and a multiple of 8", ldx);
    if (!y || !aligned(y, 4)) return fail(TF_ERR_INVALID_ARG, "y must be non-null and 4-B aligned");
    if (ldy < W->N) return fail(TF_ERR_INVALID_ARG, "ldy=%d must be >= N", ldy);
    if ((st = check_ws(ws, ws_bytes, dense_gemm_ws(*W)))) return st;
    if (size_t((W->N + kTileN - 1) / kTileN) * kFeatWarps > kMaxCounters)
        return fail(TF_ERR_UNSUPPORTED, "N=%d too large for the split-K counter region", W->N);
    GemmArgs a = dense_args(*W, R, y, ldy, mode);
    const char *why = "";
    cudaError_t e = bind_and_launch(a, x, ldx, 0, 1, ws, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "%s: %s (%s)", name, cudaGetErrorString(e), why);
    return ok();
}
}  // namespace

// ---- tf_selfcheck_row_invariance / tf_workspace_size ----
namespace {
size_t selfcheck_ld(int N) { return (size_t(N) + 63) / 64 * 64; }
}  // namespace

size_t tf_selfcheck_scratch_bytes(int32_t N) {
    if (N <= 0) return 0;
    return 256 + 2 * size_t(TF_MAX_ROWS) * selfcheck_ld(N) * sizeof(float);
}

tf_status tf_selfcheck_row_invariance(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, void *scratch,
                                      size_t scratch_bytes, void *ws, size_t ws_bytes, void *stream,
                                      int32_t *result) {
    if (!result) return fail(TF_ERR_INVALID_ARG, "null result");
    tf_status st = check_matrix(W, "W");
    if (st) return st;
    if (!scratch || !aligned(scratch, 256) || scratch_bytes < tf_selfcheck_scratch_bytes(W->N))
        return fail(TF_ERR_INVALID_ARG, "scratch must be 256-B aligned and >= %zu bytes",
                    tf_selfcheck_scratch_bytes(W->N));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ld = int(selfcheck_ld(W->N));
    int *flag = static_cast<int *>(scratch);
    float *single = reinterpret_cast<float *>(static_cast<char *>(scratch) + 256);
    float *multi = single + size_t(TF_MAX_ROWS) * ld;
    constexpr int kNone = 0x7F7F7F7F;
    cudaError_t e = cudaMemsetAsync(flag, 0x7F, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "tf_selfcheck_row_invariance");
    for (int r = 0; r < TF_MAX_ROWS; ++r)
        if ((st = tf_lane_gemm_w4(W, x + size_t(r) * ldx, ldx, 1, single + size_t(r) * ld, ld, ws, ws_bytes, stream)))
            return st;
    for (int R = 1; R <= TF_MAX_ROWS; ++R) {
        if ((st = tf_lane_gemm_w4(W, x, ldx, R, multi, ld, ws, ws_bytes, stream))) return st;
        if ((e = launch_rows_differ(multi, single, R, W->N, ld, R * 256, flag, s)) != cudaSuccess)
            return cuda_fail(e, "tf_selfcheck_row_invariance");
    }
    int v = 0;
    if ((e = cudaMemcpyAsync(&v, flag, sizeof v, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return cuda_fail(e, "tf_selfcheck_row_invariance");
    *result = v == kNone ? 0 : v;
    return ok();
}

size_t tf_workspace_size(int32_t op, const int64_t *dims, int32_t n_dims) {
    if (!dims) return 0;
    for (int i = 0; i < n_dims; ++i)
        if (dims[i] <= 0 || dims[i] > 0x7FFFFFFF) return 0;
    switch (op) {
    case TF_OP_LANE_GEMM:
        return n_dims == 3 ? tf_lane_gemm_workspace_bytes(int32_t(dims[0]), int32_t(dims[1]), int32_t(dims[2])) : 0;
    case TF_OP_KEYED_SAMPLE:
        return n_dims == 2 ? tf_keyed_sample_workspace_bytes(int32_t(dims[0]), int32_t(dims[1])) : 0;
    case TF_OP_ATTENTION: {
        if (n_dims != 4) return 0;
        tf_kv_cache c{};
        c.n_kv = int32_t(dims[0]);
        c.max_len = int32_t(dims[1]);
        return tf_attention_workspace_bytes(&c, int32_t(dims[2]), int32_t(dims[3]));
    }
    default:
        return 0;
    }
}

// ---- tf_lane_gemm_w4_noalloc: the lane GEMM on library-owned scratch ----
// The split-K status word, counters and partial tiles live in one fixed array
// of this module instead of a caller workspace.  Each device that loads the
// library has its own copy; its device address is looked up on every call
// (with the caller's device current), so a context rebuilt after a device
// reset is never handed a stale address.  All calls on a device share the copy.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
tf_status noalloc_scratch(void **out) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "tf_lane_gemm_w4_noalloc: cudaGetSymbolAddress");
    if (!p || !aligned(p, 256)) return fail(TF_ERR_CUDA, "tf_lane_gemm_w4_noalloc: scratch address unusable");
    *out = p;
    return TF_OK;
}
}  // namespace

tf_status tf_lane_gemm_w4_noalloc(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y,
                                  int32_t ldy, int32_t *status, void *stream) {
    tf_status st = check_matrix(W, "W");
    if (st) return st;
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!x || !aligned(x, 16)) return fail(TF_ERR_INVALID_ARG, "x must be non-null and 16-B aligned");
    if (ldx < W->K || ldx % 8) return fail(TF_ERR_INVALID_ARG, "ldx=%d must be >= K and a multiple of 8", ldx);
    if (!y || !aligned(y, 4)) return fail(TF_ERR_INVALID_ARG, "y must be non-null and 4-B aligned");
    if (ldy < W->N) return fail(TF_ERR_INVALID_ARG, "ldy=%d must be >= N", ldy);
    if (status && !aligned(status, 4)) return fail(TF_ERR_INVALID_ARG, "status must be 4-B aligned");
    if (size_t((W->N + kTileN - 1) / kTileN) * kFeatWarps > kMaxCounters)
        return fail(TF_ERR_UNSUPPORTED, "N=%d too large for the split-K counter region", W->N);
    GemmArgs a = dense_args(*W, R, y, ldy, kStoreF32);
    const size_t need = gemm_workspace_bytes(a.K, a.N, a.G, 1, a.Pv);
    if (need > kNoAllocScratchBytes)
        return fail(TF_ERR_UNSUPPORTED,
                    "tf_lane_gemm_w4_noalloc: this launch needs %zu bytes of scratch, the built-in array holds %zu "
                    "(use tf_lane_gemm_w4 with a workspace)",
                    need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch))) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left.  The status word and this
    // launch's split-K counters must start at zero; partial tiles are always
    // written before they are read.
    cudaError_t e = cudaMemsetAsync(scratch, 0, 256 + size_t(a.T) * kFeatWarps * sizeof(unsigned), s);
    if (e != cudaSuccess) return cuda_fail(e, "tf_lane_gemm_w4_noalloc: clearing scratch");
    gemm_bind_workspace(a, scratch, 1);
    if (status) a.err = status;
    const char *why = "";
    if (!gemm_encode_x(a, x, ldx, 0, 1, &why))
        return fail(TF_ERR_CUDA, "tf_lane_gemm_w4_noalloc: %s", why);
    e = launch_w4_gemm(a, 1, s);
    if (e != cudaSuccess) return cuda_fail(e, "tf_lane_gemm_w4_noalloc");
    return ok();
}

size_t tf_keyed_sample_workspace_bytes(int32_t R, int32_t V) {
    if (R < 1 || V < 1) return 0;
    return 256 + sample_workspace_bytes(R, V);
}

tf_status tf_keyed_sample(const float *logits, int32_t ldl, int32_t R, int32_t V, const tf_sampling *p, uint64_t seed,
                          const int64_t *pos, int32_t *tokens, void *ws, size_t ws_bytes, void *stream) {
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (V < 1) return fail(TF_ERR_INVALID_ARG, "V must be >= 1");
    if (V > sample_max_vocab()) return fail(TF_ERR_UNSUPPORTED, "V=%d exceeds %d", V, sample_max_vocab());
    if (!logits || !aligned(logits, 4)) return fail(TF_ERR_INVALID_ARG, "logits must be non-null");
    if (ldl < V) return fail(TF_ERR_INVALID_ARG, "ldl must be >= V");
    if (!tokens) return fail(TF_ERR_INVALID_ARG, "tokens must be non-null");
    int k_eff = 0;
    tf_status st = check_sampling(p, V, &k_eff);
    if (st) return st;
    if (p->temperature > 0.f && !pos) return fail(TF_ERR_INVALID_ARG, "pos must be non-null when T > 0");
    if ((st = check_ws(ws, ws_bytes, tf_keyed_sample_workspace_bytes(R, V)))) return st;
    SampleArgs a{};
    a.logits = logits;
    a.ldl = ldl;
    a.R = R;
    a.V = V;
    a.k_eff = k_eff;
    a.temperature = p->temperature;
    a.top_p = p->top_p;
    a.seed = seed;
    a.pos = pos;
    a.pos_base = nullptr;
    a.tokens = tokens;
    a.err = static_cast<int *>(ws);
    sample_bind_workspace(a, static_cast<char *>(ws) + 256, R, V);
    if (!a.pos) {  // greedy without positions: never read
        a.pos = reinterpret_cast<const int64_t *>(ws);
    }
    cudaError_t e = launch_keyed_sample(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_keyed_sample");
    return ok();
}

size_t tf_lmhead_sample_workspace_bytes(const tf_w4_matrix *W, int32_t R) {
    if (R < 1 || R > TF_MAX_ROWS || check_matrix(W, "W") != TF_OK) return 0;
    return lm_layout(*W, R).total;
}

tf_status tf_lmhead_sample(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, const tf_sampling *p,
                           uint64_t seed, const int64_t *pos, int32_t *tokens, float *logits, int32_t ldl,
                           const int32_t *drafts, int32_t *accepted, int32_t *bonus, void *ws, size_t ws_bytes,
                           void *stream) {
    tf_status st = check_matrix(W, "W");
    if (st) return st;
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (W->N > sample_max_vocab()) return fail(TF_ERR_UNSUPPORTED, "N=%d exceeds %d", W->N, sample_max_vocab());
    if (!x || !aligned(x, 16)) return fail(TF_ERR_INVALID_ARG, "x must be non-null and 16-B aligned");
    if (ldx < W->K || ldx % 8) return fail(TF_ERR_INVALID_ARG, "ldx=%d must be >= K and a multiple of 8", ldx);
    if (!tokens) return fail(TF_ERR_INVALID_ARG, "tokens must be non-null");
    if (logits && (!aligned(logits, 4) || ldl < W->N))
        return fail(TF_ERR_INVALID_ARG, "logits must be 4-B aligned with ldl >= N");
    if (accepted && R > 1 && !drafts) return fail(TF_ERR_INVALID_ARG, "drafts must be non-null when accepting R > 1 rows");
    int k_eff = 0;
    if ((st = check_sampling(p, W->N, &k_eff))) return st;
    if (p->temperature > 0.f && !pos) return fail(TF_ERR_INVALID_ARG, "pos must be non-null when T > 0");
    if (size_t((W->N + kTileN - 1) / kTileN) * kFeatWarps > kMaxCounters)
        return fail(TF_ERR_UNSUPPORTED, "N=%d too large for the split-K counter region", W->N);
    const LmLayout L = lm_layout(*W, R);
    if ((st = check_ws(ws, ws_bytes, L.total))) return st;
    char *base = static_cast<char *>(ws);
    const char *why = "";
    cudaError_t e = run_lmhead_sample(*W, x, ldx, R, *p, k_eff, seed, pos, nullptr, tokens, logits, ldl,
                                      reinterpret_cast<float *>(base + L.logits), ws, base + L.sample, drafts,
                                      accepted, bonus, nullptr, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "tf_lmhead_sample: %s (%s)", cudaGetErrorString(e), why);
    return ok();
}

tf_status tf_keyed_hash(const uint64_t *seed, const int64_t *pos, const int32_t *token, int64_t n, uint64_t *h_out,
                        double *g_out, void *stream) {
    if (n < 0) return fail(TF_ERR_INVALID_ARG, "n=%lld must be >= 0", (long long)n);
    if (n == 0) return ok();
    if (!seed || !pos || !token) return fail(TF_ERR_INVALID_ARG, "null seed, pos or token");
    cudaError_t e = launch_keyed_hash(seed, pos, token, (long long)n, h_out, g_out, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_keyed_hash");
    return ok();
}

tf_status tf_accept(const int32_t *drafts, const int32_t *sampled, int32_t R, int32_t *accepted, int32_t *bonus,
                    void *stream) {
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (R > 1 && !drafts) return fail(TF_ERR_INVALID_ARG, "drafts must be non-null when R > 1");
    if (!sampled || !accepted || !bonus) return fail(TF_ERR_INVALID_ARG, "null pointer");
    cudaError_t e = launch_accept(drafts, sampled, R, accepted, bonus, nullptr, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_accept");
    return ok();
}

tf_status tf_gather_drafts(const int32_t *table, int64_t table_len, const int64_t *pos, int32_t R, int32_t *drafts,
                           void *stream) {
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (R == 1) return ok();  // a one-row pass has no drafts
    if (!table || table_len < 0 || !pos || !drafts) return fail(TF_ERR_INVALID_ARG, "null pointer or negative length");
    cudaError_t e = launch_gather_drafts(table, table_len, pos, R - 1, drafts, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_gather_drafts");
    return ok();
}

namespace {

tf_status check_cache(const tf_kv_cache *c) {
    if (!c) return fail(TF_ERR_INVALID_ARG, "null KV cache");
    if (!c->k || !c->v) return fail(TF_ERR_INVALID_ARG, "KV cache: null k or v");
    if (!aligned(c->k, 16) || !aligned(c->v, 16)) return fail(TF_ERR_INVALID_ARG, "KV cache: k, v not 16-B aligned");
    if (c->n_kv < 1 || c->n_kv > 128) return fail(TF_ERR_UNSUPPORTED, "KV cache: n_kv=%d outside [1, 128]", c->n_kv);
    if (c->max_len <= 0 || c->max_len % kKvPart)
        return fail(TF_ERR_UNSUPPORTED, "KV cache: max_len=%d is not a positive multiple of %d", c->max_len, kKvPart);
    return TF_OK;
}

}  // namespace

tf_status tf_kv_append(const tf_kv_cache *c, const uint16_t *k_new, const uint16_t *v_new, int32_t ld, int32_t R,
                       const int64_t *pos, void *ws, size_t ws_bytes, void *stream) {
    tf_status st = check_cache(c);
    if (st != TF_OK) return st;
    if (R < 1 || R > c->max_len) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, max_len=%d]", R, c->max_len);
    if (((long long)R * c->n_kv + 7) / 8 > 0x7FFFFFFFLL)
        return fail(TF_ERR_UNSUPPORTED, "R=%d x n_kv=%d entries exceed one launch", R, c->n_kv);
    if (!k_new || !v_new || !pos) return fail(TF_ERR_INVALID_ARG, "null k_new, v_new or pos");
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(TF_ERR_INVALID_ARG, "k_new, v_new not 16-B aligned");
    if (ld < c->n_kv * kHeadDim || ld % 8)
        return fail(TF_ERR_INVALID_ARG, "ld=%d must be a multiple of 8 and >= n_kv * 128", ld);
    if ((st = check_ws(ws, ws_bytes, 256)) != TF_OK) return st;
    cudaError_t e = launch_kv_append(k_new, v_new, ld, R, pos, c->k, c->v, c->n_kv, c->max_len,
                                     static_cast<int *>(ws), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_kv_append");
    return ok();
}

size_t tf_attention_workspace_bytes(const tf_kv_cache *c, int32_t group, int32_t R) {
    if (!c || c->n_kv < 1 || c->max_len <= 0 || c->max_len % kKvPart || R < 1 || R > TF_MAX_ROWS) return 0;
    if (group != 1 && group != 2 && group != 4 && group != 8) return 0;
    return 256 + attn_opart_bytes(c->n_kv, group, c->max_len, R) + attn_ml_bytes(c->n_kv, group, c->max_len, R);
}

tf_status tf_attention_verify(const tf_kv_cache *c, int32_t group, const uint16_t *q, int32_t ldq, int32_t R,
                              const int64_t *pos, float *out, int32_t ldo, void *ws, size_t ws_bytes, void *stream) {
    tf_status st = check_cache(c);
    if (st != TF_OK) return st;
    if (group != 1 && group != 2 && group != 4 && group != 8)
        return fail(TF_ERR_UNSUPPORTED, "group=%d not in {1, 2, 4, 8}", group);
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!q || !pos || !out) return fail(TF_ERR_INVALID_ARG, "null q, pos or out");
    const int n_q = c->n_kv * group;
    if (!aligned(q, 16) || ldq < n_q * kHeadDim || ldq % 8)
        return fail(TF_ERR_INVALID_ARG, "q must be 16-B aligned with ldq a multiple of 8 and >= %d", n_q * kHeadDim);
    if (!aligned(out, 4) || ldo < n_q * kHeadDim)
        return fail(TF_ERR_INVALID_ARG, "out must be 4-B aligned with ldo >= %d", n_q * kHeadDim);
    if ((st = check_ws(ws, ws_bytes, tf_attention_workspace_bytes(c, group, R))) != TF_OK) return st;
    AttnArgs a{};
    a.k = c->k;
    a.v = c->v;
    a.q = q;
    a.ldq = ldq;
    a.R = R;
    a.group = group;
    a.n_kv = c->n_kv;
    a.max_len = c->max_len;
    a.pos = pos;
    a.err = static_cast<int *>(ws);
    a.opart = reinterpret_cast<float *>(static_cast<char *>(ws) + 256);
    a.ml = reinterpret_cast<float *>(static_cast<char *>(ws) + 256 + attn_opart_bytes(c->n_kv, group, c->max_len, R));
    a.out = out;
    a.ldo = ldo;
    cudaError_t e = launch_attention(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_attention_verify");
    return ok();
}

tf_status tf_commit_tokens(const int32_t *tokens, const int32_t *accepted, const int64_t *pos, int32_t *log,
                           int64_t log_len, void *stream) {
    if (!tokens || !accepted || !pos || !log || log_len < 0)
        return fail(TF_ERR_INVALID_ARG, "null pointer or negative length");
    cudaError_t e = launch_commit_tokens(tokens, accepted, pos, log, log_len, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_commit_tokens");
    return ok();
}

size_t tf_moe_workspace_bytes(const tf_moe_layer *L, int32_t R) {
    if (!L || R < 1 || R > TF_MAX_ROWS || L->n_experts < 1 || L->top_k < 1 || L->hidden <= 0 || L->ffn <= 0)
        return 0;
    return moe_layout(*L, R).total;
}

tf_status tf_moe_w4(const tf_moe_layer *L, const uint16_t *x, const float *router_logits, int32_t R, float *out,
                    void *ws, size_t ws_bytes, void *stream) {
    tf_status st = check_moe(L);
    if (st) return st;
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!x || !aligned(x, 16) || !router_logits || !out) return fail(TF_ERR_INVALID_ARG, "null or misaligned pointer");
    const MoeLayout m = moe_layout(*L, R);
    if ((st = check_ws(ws, ws_bytes, m.total))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    int32_t *ids = reinterpret_cast<int32_t *>(base + m.ids);
    float *w = reinterpret_cast<float *>(base + m.w);
    int32_t *expert_ids = reinterpret_cast<int32_t *>(base + m.expert_ids);
    int32_t *nprob = reinterpret_cast<int32_t *>(base + m.nprob);
    int32_t *slot_of = reinterpret_cast<int32_t *>(base + m.slot_of);
    uint16_t *h = reinterpret_cast<uint16_t *>(base + m.h);
    float *Y = reinterpret_cast<float *>(base + m.Y);
    int *err = reinterpret_cast<int *>(base);

    cudaError_t e = launch_route_list(router_logits, R, L->n_experts, L->top_k, ids, w, expert_ids, nprob,
                                      slot_of, err, s);
    if (e != cudaSuccess) return cuda_fail(e, "tf_moe_w4 routing");

    // gate/up (+ SwiGLU) for every touched expert, all R rows
    const char *why = "";
    tf_w4_matrix Wgu{L->gate_up, L->hidden, 2 * L->ffn, L->group};
    GemmArgs g1 = dense_args(Wgu, R, h, L->ffn, kSwiGluBf16);
    g1.Pv = grouped_pv(g1.T, g1.Kc);
    g1.w_stride = (long long)packed_bytes(L->hidden, 2 * L->ffn, L->group);
    g1.expert_ids = expert_ids;
    g1.n_problems = nprob;
    g1.y_stride = (long long)R * L->ffn;
    e = bind_and_launch(g1, x, L->hidden, 0, m.u_max, ws, s, &why);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "tf_moe_w4 gate/up: %s (%s)", cudaGetErrorString(e), why);

    tf_w4_matrix Wd{L->down, L->ffn, L->hidden, L->group};
    GemmArgs g2 = dense_args(Wd, R, Y, L->hidden, kStoreF32);
    g2.Pv = grouped_pv(g2.T, g2.Kc);
    g2.w_stride = (long long)packed_bytes(L->ffn, L->hidden, L->group);
    g2.expert_ids = expert_ids;
    g2.n_problems = nprob;
    g2.list_ready = 1;   // routed by the grid before gate/up, which has passed its own wait
    g2.y_stride = (long long)R * L->hidden;
    e = bind_and_launch(g2, h, L->ffn, (long long)R * L->ffn, m.u_max, ws, s, &why);
    if (e == cudaSuccess) e = launch_combine(Y, slot_of, w, R, L->hidden, L->top_k, out, s);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "tf_moe_w4 down/combine: %s (%s)", cudaGetErrorString(e), why);
    return ok();
}

size_t tf_verify_step_workspace_bytes(const tf_model *m, int32_t R) {
    if (R < 1 || R > TF_MAX_ROWS || check_model(m) != TF_OK) return 0;
    return step_layout(*m, R).total;
}

tf_status tf_verify_step(const tf_model *m, int32_t R, int32_t *last_token, int64_t *pos, const int32_t *drafts,
                         const tf_sampling *p, uint64_t seed, int32_t *tokens, int32_t *accepted, float *logits,
                         void *ws, size_t ws_bytes, void *stream) {
    tf_status st = check_model(m);
    if (st) return st;
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!last_token || !pos || !tokens || !accepted) return fail(TF_ERR_INVALID_ARG, "null pointer");
    if (R > 1 && !drafts) return fail(TF_ERR_INVALID_ARG, "drafts must be non-null when R > 1");
    int k_eff = 0;
    if ((st = check_sampling(p, m->vocab, &k_eff))) return st;
    const StepLayout L = step_layout(*m, R);
    if ((st = check_ws(ws, ws_bytes, L.total))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    int *err = reinterpret_cast<int *>(base);
    float *x = reinterpret_cast<float *>(base + L.x);
    uint16_t *n = reinterpret_cast<uint16_t *>(base + L.n);
    uint16_t *h = reinterpret_cast<uint16_t *>(base + L.h);

    const char *why = "";
    cudaError_t e = launch_embed(m->embedding, m->vocab, m->hidden, last_token, drafts, R, x, err, s);
    for (int b = 0; b < m->n_blocks && e == cudaSuccess; ++b) e = run_block(*m, b, x, R, n, h, ws, s, &why);
    if (e == cudaSuccess) e = launch_rmsnorm_bf16(x, R, m->hidden, m->rms_eps, n, s);
    if (e == cudaSuccess)
        e = run_lmhead_sample(m->lm_head, n, m->hidden, R, *p, k_eff, seed, nullptr, pos, tokens, logits, m->vocab,
                              reinterpret_cast<float *>(base + L.logits), ws, base + L.sample, drafts, accepted,
                              last_token, pos, s, &why);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "tf_verify_step: %s %s", cudaGetErrorString(e), why);
    return ok();
}

tf_status tf_embed_rows(const tf_model *m, const int32_t *last_token, const int32_t *drafts, int32_t R, float *x,
                        void *ws, void *stream) {
    if (!m || !m->embedding) return fail(TF_ERR_INVALID_ARG, "null model");
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!last_token || !x || (R > 1 && !drafts)) return fail(TF_ERR_INVALID_ARG, "null pointer");
    tf_status st = check_ws(ws, 256, 256);
    if (st) return st;
    cudaError_t e = launch_embed(m->embedding, m->vocab, m->hidden, last_token, drafts, R, x, static_cast<int *>(ws),
                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_embed_rows");
    return ok();
}

tf_status tf_rmsnorm_bf16(const float *x, int32_t R, int32_t H, float eps, uint16_t *out, void *stream) {
    if (!x || !out) return fail(TF_ERR_INVALID_ARG, "null pointer");
    if (R < 1 || H < 1) return fail(TF_ERR_INVALID_ARG, "R and H must be >= 1");
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(TF_ERR_INVALID_ARG, "bad eps");
    cudaError_t e = launch_rmsnorm_bf16(x, R, H, eps, out, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tf_rmsnorm_bf16");
    return ok();
}

size_t tf_decoder_block_workspace_bytes(const tf_model *m) {
    if (check_model(m) != TF_OK) return 0;
    return block_gemm_ws(*m);
}

tf_status tf_decoder_block(const tf_model *m, int32_t block, float *x, int32_t R, uint16_t *n_out, uint16_t *h_out,
                           void *ws, size_t ws_bytes, void *stream) {
    tf_status st = check_model(m);
    if (st) return st;
    if (block < 0 || block >= m->n_blocks) return fail(TF_ERR_INVALID_ARG, "block %d outside the model", block);
    if (R < 1 || R > TF_MAX_ROWS) return fail(TF_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, TF_MAX_ROWS);
    if (!x || !n_out || !h_out) return fail(TF_ERR_INVALID_ARG, "null pointer");
    if (!aligned(n_out, 16) || !aligned(h_out, 16)) return fail(TF_ERR_INVALID_ARG, "n_out / h_out not 16-B aligned");
    if ((st = check_ws(ws, ws_bytes, block_gemm_ws(*m)))) return st;
    const char *why = "";
    cudaError_t e = run_block(*m, block, x, R, n_out, h_out, ws, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) return fail(TF_ERR_CUDA, "tf_decoder_block: %s %s", cudaGetErrorString(e), why);
    return ok();
}

}  // extern "C"
