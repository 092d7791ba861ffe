/*
 * tf.h -- C ABI of the exact speculative-decoding verify pass for GB300 (sm_103a).
 *
 * The method (TensorFold README, section on its two guarantees):
 *   1. keyed sampling: the token chosen for position p maximises
 *      logit / T + g(seed, p, token) over the top-k / top-p candidates, where g
 *      is Gumbel noise derived by hashing seed, position and token id;
 *   2. row invariance: each row of a verify pass over several drafted rows
 *      comes out bit for bit as it would in a pass of one row;
 * hence a draft survives only if it matches what one-row decoding samples at
 * that position, and a drafted run emits exactly the serial run's tokens.  Weights are 4-bit codes with one fp16 scale per group of 64
 * (dense model) or 32 (MoE model) input features (README, "What each
 * checkpoint needs").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers marked "dev" are CUDA device pointers owned by the caller.
 *   The library never allocates, frees or retains device memory, and it keeps
 *   no global state besides a thread-local error message, with one exception:
 *   tf_lane_gemm_w4_noalloc works on a fixed scratch array that the library
 *   itself holds on every device that loads it (see that entry point).
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every compute call only enqueues work on that stream and returns;
 *   outputs are valid once the stream has reached that point.
 * - `ws` is caller-provided device scratch ("workspace") of at least the size
 *   the matching *_workspace_bytes() query returns, 256-byte aligned, and
 *   zero-filled before its first use (the kernels leave the parts they
 *   need zeroed when they finish, so a workspace can be reused by later calls
 *   on the same stream without clearing it again).  Calls that overlap in time
 *   must not share a workspace.
 * - Host-side argument errors return TF_ERR_INVALID_ARG / TF_ERR_UNSUPPORTED
 *   before anything is enqueued; tf_last_error() then describes the problem.
 *   Errors that only the device can see (a non-finite logit, an out-of-range
 *   token id, a bounded wait that ran out) are recorded in the first word of
 *   the workspace; read them with tf_workspace_status().  Nothing traps,
 *   aborts or throws across this boundary.
 * - Row counts R are 1..TF_MAX_ROWS.  R = 1 is the serial reference
 *   (README: "draft": false decodes one token a round).
 * - bf16 / fp16 values are passed as their 16-bit IEEE bit patterns (uint16_t).
 */
#ifndef TF_H
#define TF_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TF_API __attribute__((visibility("default")))
#else
#define TF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define TF_MAX_ROWS 16
#define TF_MAX_TOP_K 64   /* largest k' of the fast candidate path */

typedef enum tf_status {
    TF_OK = 0,
    TF_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or value */
    TF_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
    TF_ERR_CUDA = 3,          /* a CUDA runtime call failed (message in tf_last_error) */
    TF_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out (device status) */
    TF_ERR_WORKSPACE = 5      /* workspace missing, misaligned or too small */
} tf_status;

/* Device-status codes stored in the first 32-bit word of a workspace. */
#define TF_DEV_OK 0
#define TF_DEV_TIMEOUT 1          /* an mbarrier wait exceeded its iteration limit */
#define TF_DEV_NONFINITE_LOGIT 2  /* a logit was NaN or +-inf (its row's token is -1) */
#define TF_DEV_BAD_TOKEN 3        /* a token id outside [0, vocab) reached the embedding */
#define TF_DEV_BAD_POSITION 4     /* a KV-cache call saw *pos < 0 or *pos + R > max_len (nothing written) */

/* Thread-local description of the last host-side error ("" when none). */
TF_API const char *tf_last_error(void);
TF_API const char *tf_status_string(tf_status s);
/* Library ABI version (major * 10000 + minor * 100 + patch). */
TF_API int tf_version(void);

/*
 * Read and clear the device-status word of a workspace.  Synchronises `stream`
 * first.  *code receives one of the TF_DEV_* values.  Returns TF_OK, or
 * TF_ERR_CUDA if the copy failed.
 */
TF_API tf_status tf_workspace_status(void *ws, void *stream, int32_t *code);

/* ------------------------------------------------------------------------
 * W4 weights
 * ------------------------------------------------------------------------
 * Canonical layout (the input of tf_pack_w4), for a linear layer with K
 * input and N output features and group size G (32 or 64):
 *   codes  uint8  [N][K/2]  element (n, k) is the low nibble of byte k/2 when k
 *                           is even and the high nibble when k is odd; each
 *                           nibble is a two's-complement integer in [-8, 7];
 *   scales uint16 [N][K/G]  fp16 scale of group g = k / G of row n;
 *   w[n][k] = code(n, k) * scale(n, k / G)   (symmetric, no zero point).
 * The kernels read a private "packed" layout produced on the device by
 * tf_pack_w4 (a load-time step).  Its size is tf_w4_packed_bytes(); N is padded
 * up to a multiple of 128 with zero weights inside it.
 */
typedef struct tf_w4_matrix {
    const void *packed;   /* dev, tf_w4_packed_bytes(K, N, group) bytes, 256-B aligned */
    int32_t K;            /* input features, a positive multiple of 64 */
    int32_t N;            /* output features, >= 1 */
    int32_t group;        /* 32 or 64 */
    int32_t affine;       /* 0: symmetric (tf_pack_w4); 1: MLX-style affine (tf_pack_w4_affine) */
} tf_w4_matrix;

/* Bytes of the packed layout, or 0 if (K, N, group) is unsupported. */
TF_API size_t tf_w4_packed_bytes(int32_t K, int32_t N, int32_t group);

/* MLX-style affine 4-bit weights (the format of MLX 4-bit checkpoints, which the
 * README says the engine serves; its layout follows MLX's public quantisation):
 *   codes  uint32 [N][K/8]  word j of row n holds q(n, 8j + i) in bits 4i..4i+3,
 *                           q an unsigned integer in [0, 15];
 *   scales uint16 [N][K/G]  bf16 scale of group g = k / G of row n;
 *   biases uint16 [N][K/G]  bf16 bias of that group;
 *   w[n][k] = scale(n, k / G) * q(n, k) + bias(n, k / G).
 * tf_pack_w4_affine produces the packed layout of a matrix with affine = 1
 * (size tf_w4_affine_packed_bytes); tf_lane_gemm_w4 and tf_lane_gemm_w4_noalloc
 * accept it: each group's partial sum_k q x is scaled, and the bias is added
 * times the group's activation sum sum_k x (fp32, formed by the tensor core),
 * bits of row r still independent of R.  The MoE and decoder entry points take
 * symmetric matrices only. */
TF_API size_t tf_w4_affine_packed_bytes(int32_t K, int32_t N, int32_t group);
TF_API tf_status tf_pack_w4_affine(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                                   int32_t K, int32_t N, int32_t group, void *packed, size_t packed_bytes,
                                   void *stream);

/* ------------------------------------------------------------------------
 * NVFP4 weights and their lane GEMM
 * ------------------------------------------------------------------------
 * Context Studios, "TensorFold: The engine that makes local LLMs 2-3x faster":
 * the engine reads NVFP4 checkpoints on Blackwell.  The pages do not give the
 * format; this follows NVIDIA's public description of NVFP4:
 *   codes  uint8 [N][K/2]   4-bit E2M1 codes (bit 3 sign, bits 2..1 exponent
 *                           with bias 1, bit 0 mantissa; values 0, 0.5, 1,
 *                           1.5, 2, 3, 4, 6 and negatives), element 2j in the
 *                           low nibble of byte j;
 *   scales uint8 [N][K/16]  E4M3 bit pattern of the scale of the 16 features
 *                           16b .. 16b + 15 of row n (NaN pattern 0x7F/0xFF
 *                           not allowed);
 *   global_scale            fp32, one per tensor;
 *   w[n][k] = e2m1(n, k) * e4m3(n, k / 16) * global_scale.
 * tf_pack_nvfp4 repacks (codes, scales) into `packed` (dev, 256-B aligned,
 * tf_nvfp4_packed_bytes(K, N) bytes; K a positive multiple of 64, N >= 1).
 * tf_lane_gemm_nvfp4 computes y[r][n] = sum_k w[n][k] x[r][k] with the same
 * argument conventions, workspace rules and row invariance as
 * tf_lane_gemm_w4.  Arithmetic: each weight times its block scale is formed
 * exactly in fp16, the activations are taken to fp16 (exact for bf16 values
 * with |x| <= 65504; larger values overflow to inf, values below 2^-14 round
 * to fp16 subnormals), products accumulate in fp32 in a fixed k order, and
 * the output is multiplied by global_scale once.
 */
typedef struct tf_nvfp4_matrix {
    const void *packed;   /* dev, tf_nvfp4_packed_bytes(K, N) bytes, 256-B aligned */
    int32_t K;            /* input features, a positive multiple of 64 */
    int32_t N;            /* output features, >= 1 */
    float global_scale;   /* the tensor's fp32 scale, finite */
} tf_nvfp4_matrix;

TF_API size_t tf_nvfp4_packed_bytes(int32_t K, int32_t N);
TF_API tf_status tf_pack_nvfp4(const uint8_t *codes, const uint8_t *scales, int32_t K, int32_t N, void *packed,
                               size_t packed_bytes, void *stream);
TF_API size_t tf_lane_gemm_nvfp4_workspace_bytes(int32_t K, int32_t N);
TF_API tf_status tf_lane_gemm_nvfp4(const tf_nvfp4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R, float *y,
                                    int32_t ldy, void *ws, size_t ws_bytes, void *stream);

/*
 * Repack canonical codes + scales (dev) into the kernel layout `packed` (dev,
 * packed_bytes >= tf_w4_packed_bytes).  Not on the hot path.  Pure
 * permutation: the codes and the scale bits are preserved exactly.
 */
TF_API tf_status tf_pack_w4(const uint8_t *codes, const uint16_t *scales, int32_t K, int32_t N,
                     int32_t group, void *packed, size_t packed_bytes, void *stream);

/*
 * Pack the fused gate/up projection of a SwiGLU layer: canonical rows
 * 0..ffn-1 are the gate rows, ffn..2*ffn-1 the up rows (N = 2*ffn).  The packed
 * layout interleaves each 16 gate rows with the matching 16 up rows so the
 * kernel can apply silu(gate) * up in its epilogue.  Matrices packed this way
 * are consumed by tf_moe_w4 and tf_verify_step (not by tf_lane_gemm_w4).
 * Size: tf_w4_packed_bytes(K, 2 * ffn, group).
 */
TF_API tf_status tf_pack_w4_gate_up(const uint8_t *codes, const uint16_t *scales, int32_t K, int32_t ffn,
                             int32_t group, void *packed, size_t packed_bytes, void *stream);

/* ------------------------------------------------------------------------
 * tf_lane_gemm_w4 -- the verify pass's linear layer
 * ------------------------------------------------------------------------
 * README, the two guarantees (row invariance): all R drafted rows go through
 * one launch that reads each weight once, and row r's result is bit-identical
 * whatever R is.
 *
 *   y[r][n] = sum_g scale(n, g) * ( sum_{k in g} code(n, k) * x[r][k] )
 *
 * x   dev bf16 [R][ldx]   (ldx >= K, ldx % 8 == 0, 16-B aligned)
 * y   dev fp32 [R][ldy]   (ldy >= N)
 * Each group's partial sum is formed exactly (integer codes times bf16
 * activations, fp32 accumulation) and then scaled in fp32; groups, and the
 * fixed split-K partials, are added in an order that depends only on
 * (K, N, group) and the GPU's SM count -- never on R.
 */
TF_API size_t tf_lane_gemm_workspace_bytes(int32_t K, int32_t N, int32_t group);
TF_API tf_status tf_lane_gemm_w4(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R,
                          float *y, int32_t ldy, void *ws, size_t ws_bytes, void *stream);

/*
 * tf_lane_gemm_w4_accumulate: y[r][n] += (the tf_lane_gemm_w4 result), one
 * fp32 add per element in the epilogue -- the residual update of a layer whose
 * output joins the residual stream.  Arguments, layouts and row invariance as
 * tf_lane_gemm_w4.
 * tf_cast_bf16: y[r][n] = bf16(x[r][n]), rounded to nearest, ties to even, for
 * r < R (1..65535) and n < N; x dev fp32 [R][ldx], y dev bf16 [R][ldy]
 * (ldx, ldy >= N).  The bf16 operand of the next layer (queries, keys and
 * values for the KV cache, the attention output for its projection).
 */
TF_API tf_status tf_lane_gemm_w4_accumulate(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R,
                                            float *y, int32_t ldy, void *ws, size_t ws_bytes, void *stream);
TF_API tf_status tf_cast_bf16(const float *x, int32_t R, int32_t N, int32_t ldx, uint16_t *y, int32_t ldy,
                              void *stream);

/* ------------------------------------------------------------------------
 * tf_lane_gemm_w4_noalloc -- tf_lane_gemm_w4 without a caller workspace
 * ------------------------------------------------------------------------
 * No counterpart in the pages: an integration convenience.  Same operation,
 * arguments (minus ws / ws_bytes), layouts and bits as tf_lane_gemm_w4.
 *
 * For callers that cannot hand in device memory: code that runs inside an
 * allocator or an out-of-memory handler (allocating there would re-enter the
 * allocator or fail), and hosts that own no device memory pool and must not
 * call cudaMalloc, which can synchronise the device.  This call allocates
 * nothing: its split-K scratch is a fixed 8 MiB array inside libtf, one copy
 * per device.
 *
 * - Every call looks up the array's address on the current device (a
 *   cudaGetSymbolAddress, no allocation), so the address stays right after a
 *   device reset; the first call on a device loads the array there, so make
 *   it before any stream capture.
 * - A launch whose scratch need exceeds the array (it grows with the device's
 *   SM count: 256 B + 256 KiB + 16 KiB per SM) returns TF_ERR_UNSUPPORTED and
 *   launches nothing.
 * - Every call on a device shares the one array, which keeps what the last call
 *   left; each call clears the parts that must start at zero on `stream`
 *   before its kernel.  Calls that can overlap in time on one device (different
 *   streams, or several host threads) race on the array and give undefined
 *   results: serialise them, or use tf_lane_gemm_w4 with one workspace each.
 * status  dev int32 or NULL.  When given (zeroed by the caller), the kernel
 *         records there the first device-side error of this call
 *         (TF_DEV_TIMEOUT); when NULL, such an error goes to the shared array
 *         and is cleared, unread, by the next call.
 */
TF_API tf_status tf_lane_gemm_w4_noalloc(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R,
                                         float *y, int32_t ldy, int32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * tf_keyed_sample -- keyed Gumbel-max sampling over top-k / top-p
 * ------------------------------------------------------------------------
 * README, the two guarantees (keyed sampling), and the CLI options table
 * (a temperature of 0 selects greedy decoding).  Per row r, at position pos[r]:
 *   T == 0: token = argmax_i logit_i (ties: lower id);
 *   T  > 0: order the V tokens by (logit desc, id asc); keep the first
 *           k' = (top_k <= 0 || top_k >= V) ? V : top_k; if top_p < 1 keep the
 *           shortest prefix whose renormalised mass q_i = exp((l_i-l_0)/T)/Z
 *           (fp64, summed left to right in rank order) reaches top_p;
 *           token = argmax over the kept ids of (double)l/(double)T + g,
 *           g = -ln(-ln u), u = ((h >> 11) + 0.5) / 2^53 (fp64),
 *           h = sm(sm(sm(seed) ^ pos) ^ (uint32)token), sm = SplitMix64
 *           finaliser; ties: lower id.
 * logits dev fp32 [R][ldl] (ldl >= V); pos dev int64 [R]; tokens dev int32 [R].
 * Supported: 1 <= V <= tf's vocabulary limit (524288), any top_k, T >= 0
 * finite.  k' <= TF_MAX_TOP_K takes the fast path (per-chunk top-k', one
 * finaliser summing the top-p mass left to right in rank order); larger k'
 * (top_k <= 0 included) take a general path: a radix select of the k'-th key,
 * the fp64 weights exp((l_i - l_0)/T) kept as exact 53-bit fixed-point masses
 * (floor(2^53 w)), Z and the top-p boundary from exact integer sums of them,
 * so the boundary matches the left-to-right fp64 sum except where the mass
 * reaching it lies within about V * 2^-53 (relative to Z) of top_p; then the
 * Gumbel argmax over the kept candidates (fp64 for every score that an fp32
 * estimate with a stated error bound cannot rule out).  Both paths are deterministic and
 * give each row the same token whatever R is.  A non-finite logit sets
 * TF_DEV_NONFINITE_LOGIT and that row's token to -1.
 */
typedef struct tf_sampling {
    float temperature;  /* 0 = greedy */
    int32_t top_k;      /* <= 0: no top-k limit */
    float top_p;        /* >= 1: no top-p limit */
} tf_sampling;

TF_API size_t tf_keyed_sample_workspace_bytes(int32_t R, int32_t V);
TF_API tf_status tf_keyed_sample(const float *logits, int32_t ldl, int32_t R, int32_t V, const tf_sampling *p,
                          uint64_t seed, const int64_t *pos, int32_t *tokens, void *ws,
                          size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * tf_lmhead_sample -- LM head and keyed sampling in one call
 * ------------------------------------------------------------------------
 * README, the two guarantees (keyed sampling over the top-k / top-p
 * candidates of the LM head's logits).  Per row r:
 *   tokens[r] = tf_keyed_sample(tf_lane_gemm_w4(W, x)[r], p, seed, pos[r])
 * with the same bits as those two calls in a row (same logits, same candidate
 * set and order, same finaliser).  When W is symmetric int4, R <= 8 and every
 * CTA of the GEMM can keep k' = (T == 0 ? 1 : k') candidates in the
 * finaliser's pool (k' * grid <= 8192 with grid = the GEMM's CTA count, at
 * most the SM count; k' <= 53 on 152 SMs), the GEMM's epilogue keeps each CTA's k' best
 * (logit, id) per row as it stores them and the finaliser alone merges
 * them: no logits are re-read and no vocabulary-wide pass runs.  Otherwise
 * (R > 8, larger k', top_k <= 0, affine weights) the GEMM stores the logits
 * and the sampler runs on them.
 * W       symmetric or affine int4 matrix, K x N with N = the vocabulary V
 *         (V <= 524288).
 * x       dev bf16 [R][ldx] (ldx >= K, a multiple of 8; 16-B aligned).
 * p, seed, pos, tokens: as tf_keyed_sample (pos dev int64 [R], may be NULL
 *         for T == 0).
 * logits  dev fp32 [R][ldl] (ldl >= V) or NULL: when given, also receives the
 *         logits (bit-identical to tf_lane_gemm_w4's).
 * drafts, accepted, bonus: when accepted (dev int32 [1]) is non-NULL, the
 *         finaliser also runs tf_accept(drafts, tokens, R) on this call's
 *         tokens: the last row to finish writes *accepted and, if bonus is
 *         non-NULL, *bonus (drafts dev int32 [R-1], may be NULL for R == 1).
 * ws      >= tf_lmhead_sample_workspace_bytes(W, R) bytes (GEMM scratch, the
 *         sampler's, and logits scratch for the unfused path).
 * Device errors as tf_lane_gemm_w4 and tf_keyed_sample (a non-finite logit
 * sets TF_DEV_NONFINITE_LOGIT and that row's token to -1).
 */
TF_API size_t tf_lmhead_sample_workspace_bytes(const tf_w4_matrix *W, int32_t R);
TF_API tf_status tf_lmhead_sample(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, int32_t R,
                                  const tf_sampling *p, uint64_t seed, const int64_t *pos, int32_t *tokens,
                                  float *logits, int32_t ldl, const int32_t *drafts, int32_t *accepted,
                                  int32_t *bonus, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * tf_keyed_hash -- the sampler's key and Gumbel noise for given triples
 * ------------------------------------------------------------------------
 * README, the two guarantees (keyed sampling): g is Gumbel noise derived from
 * a hash of the seed, the position and the token id.  For i < n:
 *   h[i] = sm(sm(sm(seed[i]) ^ (uint64)pos[i]) ^ (uint32)token[i])
 *   g[i] = -ln(-ln u),  u = ((h[i] >> 11) + 0.5) / 2^53 in fp64
 * computed by the same device functions tf_keyed_sample uses, so a caller can
 * check the sampler's noise bit for bit.  seed dev uint64 [n], pos dev int64
 * [n], token dev int32 [n]; h_out dev uint64 [n] and g_out dev fp64 [n] (either
 * may be NULL).  n = 0 does nothing; n < 0 or a NULL input with n > 0 is
 * TF_ERR_INVALID_ARG.
 */
TF_API tf_status tf_keyed_hash(const uint64_t *seed, const int64_t *pos, const int32_t *token, int64_t n,
                               uint64_t *h_out, double *g_out, void *stream);

/* ------------------------------------------------------------------------
 * tf_accept -- longest-prefix acceptance
 * ------------------------------------------------------------------------
 * README, the two guarantees: a draft counts only if one-row decoding would
 * sample that same token at its position.  Row i samples position pos0 + i;
 * draft d[i] (i < R-1) proposes position pos0 + i.
 *   a = first i with d[i] != t[i], else R-1;  commit t[0..a];  bonus = t[a].
 * drafts dev int32 [R-1] (may be NULL when R == 1); sampled dev int32 [R];
 * accepted, bonus dev int32 [1].
 */
TF_API tf_status tf_accept(const int32_t *drafts, const int32_t *sampled, int32_t R, int32_t *accepted,
                    int32_t *bonus, void *stream);

/* ------------------------------------------------------------------------
 * tf_moe_w4 -- top-k routed W4 SwiGLU experts (30B-A3B-class MoE layer)
 * ------------------------------------------------------------------------
 * README, "What each checkpoint needs" (the MoE model is served from 4-bit
 * weights quantised in groups of 32) and source layout (fused MoE kernels).
 * Per row r:
 *   experts ranked by (router logit desc, id asc), the first top_k kept,
 *   weights w_j = exp(z_j - z_0) / sum_{i<top_k} exp(z_i - z_0) (fp64, then fp32);
 *   for each kept expert e: h = bf16(silu(x Wg_e) * (x Wu_e)), y_e = h Wd_e;
 *   out[r] = sum_j w_j * y_{e_j} in rank order (fp32).
 * Every touched expert's weights are read once for all R rows, and each row's
 * y_e is bit-identical to the one its 1-row launch produces.
 * gate_up: n_experts matrices of K = hidden, N = 2*ffn, each packed with
 *          tf_pack_w4_gate_up, back to back: expert e at byte
 *          e * tf_w4_packed_bytes(hidden, 2*ffn, group);
 * down:    n_experts matrices of K = ffn, N = hidden, packed likewise.
 * x dev bf16 [R][hidden]; router dev fp32 [R][n_experts]; out dev fp32 [R][hidden].
 */
typedef struct tf_moe_layer {
    const void *gate_up;   /* dev */
    const void *down;      /* dev */
    int32_t hidden;        /* multiple of 64 */
    int32_t ffn;           /* multiple of 64 */
    int32_t n_experts;     /* 1..256 */
    int32_t top_k;         /* 1..8, <= n_experts */
    int32_t group;         /* 32 or 64 */
} tf_moe_layer;

TF_API size_t tf_moe_workspace_bytes(const tf_moe_layer *L, int32_t R);
TF_API tf_status tf_moe_w4(const tf_moe_layer *L, const uint16_t *x, const float *router_logits, int32_t R,
                    float *out, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * tf_verify_step -- one verify pass of the attention-free synthetic decoder
 * ------------------------------------------------------------------------
 * Stand-in for the pages' 27B-class dense model (weights not available):
 *   x = emb[token];  n_blocks x { n = bf16(rms(x)); h = bf16(silu(n Wg) * (n Wu));
 *   x += h Wd };  logits = bf16(rms(x)) Wlm;  then keyed sampling and acceptance.
 * rms(x) = x / sqrt(mean(x^2) + eps); residual kept in fp32.
 * Inputs of row 0: *last_token at position *pos; row i > 0: drafts[i-1] at
 * position *pos + i.  On completion tokens[0..R-1] hold the samples,
 * *accepted = a, *last_token = bonus t[a] and *pos += a + 1, so consecutive
 * steps chain on the device.  logits (dev fp32 [R][vocab]) may be NULL.
 */
typedef struct tf_model {
    int32_t vocab, hidden, ffn, n_blocks, group;
    float rms_eps;
    const uint16_t *embedding;     /* dev bf16 [vocab][hidden] */
    const tf_w4_matrix *gate_up;   /* host array [n_blocks]: K = hidden, N = 2*ffn (tf_pack_w4_gate_up) */
    const tf_w4_matrix *down;      /* host array [n_blocks]: K = ffn, N = hidden */
    tf_w4_matrix lm_head;          /* K = hidden, N = vocab */
} tf_model;

TF_API size_t tf_verify_step_workspace_bytes(const tf_model *m, int32_t R);
TF_API tf_status tf_verify_step(const tf_model *m, int32_t R, int32_t *last_token, int64_t *pos,
                         const int32_t *drafts, const tf_sampling *p, uint64_t seed, int32_t *tokens,
                         int32_t *accepted, float *logits, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Device-side decode loop: drafts in, committed tokens out
 * ------------------------------------------------------------------------
 * README, the paragraph on the two guarantees (drafted and serial decoding
 * write the same tokens): a decode loop is verify passes chained on the device
 * (tf_verify_step advances *last_token and *pos itself).  With these two calls no pass needs the host,
 * so a run of passes can be captured in one CUDA graph and the host
 * synchronises only between runs.
 *
 * tf_gather_drafts: drafts[i] = table[*pos + i] for i < R - 1 -- the proposals
 *   for the positions the next pass verifies (draft i proposes position
 *   *pos + i); entries outside [0, table_len) read as token 0.  table dev int32
 *   [table_len], pos dev int64 [1], drafts dev int32 [R - 1].  R == 1: no-op.
 * tf_commit_tokens: after a pass that advanced *pos by a + 1 (a = *accepted),
 *   log[p - 1] = t for each committed token t at position p, i.e.
 *   log[*pos - a - 2 + i] = tokens[i] for i <= a; entries outside
 *   [0, log_len) are skipped.  tokens dev int32 [R], accepted dev int32 [1],
 *   pos dev int64 [1], log dev int32 [log_len].
 */
TF_API tf_status tf_gather_drafts(const int32_t *table, int64_t table_len, const int64_t *pos, int32_t R,
                                  int32_t *drafts, void *stream);
TF_API tf_status tf_commit_tokens(const int32_t *tokens, const int32_t *accepted, const int64_t *pos, int32_t *log,
                                  int64_t log_len, void *stream);

/* ------------------------------------------------------------------------
 * Attention of the verify rows over a KV cache.
 *
 * By the README's note on drafting, runs with and without drafts emit the same
 * tokens when they start from one cache; the 0.3.4.1 release note
 * ("TensorFold: the contract is what it does not change", section "The
 * regression it published against itself") keeps cached bits independent of
 * where a conversation resumed.  The
 * pages do not spell out the attention; these calls compute causal scaled
 * dot-product attention with grouped key/value heads (head dimension 128,
 * query head h reads KV head h / group), and make each row's bits depend only
 * on its own query, its own position p and cache entries 0..p:
 *   s_t = q . k_t / sqrt(128),  out = sum_{t <= p} exp(s_t - max s) v_t / sum exp(s_t - max s).
 * Keys are processed on a fixed grid of absolute positions (partitions of 256,
 * steps of 64), never relative to the launch, so a verify pass of R rows gives
 * every row the bits of a one-row pass at that position.  Rolling back
 * rejected rows needs no call: the next pass starts at the advanced *pos and
 * rewrites those entries before any row can read them.
 * ------------------------------------------------------------------------
 * tf_kv_cache: k and v are dev bf16 arrays [n_kv][max_len][128]; the element
 *   (head j, position t, dimension d) is stored at
 *     (j * max_len + t) * 128 + 8 * ((d / 8) XOR (t % 8)) + d % 8
 *   (the 16-byte chunks of each entry permuted by its position, so that one
 *   contiguous copy of 64 entries reads without shared-memory bank conflicts).
 *   Only tf_kv_append writes entries.  Caller-owned, 16-B aligned; n_kv in
 *   1..128; max_len a positive multiple of 256.  Entries at positions past
 *   *pos + R - 1 are never read; entries a call reads must be finite.
 * tf_kv_append: writes k_new[r] and v_new[r] (dev bf16 [R][ld], KV head j at
 *   columns j*128 .. j*128+127; ld a multiple of 8, rows 16-B aligned) as the
 *   entries at position *pos + r, r < R, R in 1..max_len (a whole prompt may be
 *   appended in one call).  pos: dev int64 [1], read on the device.  A bad
 *   position records TF_DEV_BAD_POSITION in ws (>= 256 B) and writes nothing.
 * tf_attention_verify: out[r][h*128 + d] (dev fp32 [R][ldo], ldo >= n_kv*group*128)
 *   for rows r < R (R in 1..16) at positions *pos + r, over the entries
 *   already appended (append the pass's own rows first).  q: dev bf16 [R][ldq],
 *   query head h at columns h*128 (ldq a multiple of 8, 16-B aligned).  group
 *   in {1, 2, 4, 8}.  ws: tf_attention_workspace_bytes(c, group, R) bytes of
 *   scratch for per-partition partial results.  A bad position records
 *   TF_DEV_BAD_POSITION and leaves out unwritten.
 */
typedef struct tf_kv_cache {
    uint16_t *k;
    uint16_t *v;
    int32_t n_kv;
    int32_t max_len;
} tf_kv_cache;

TF_API tf_status tf_kv_append(const tf_kv_cache *c, const uint16_t *k_new, const uint16_t *v_new, int32_t ld,
                              int32_t R, const int64_t *pos, void *ws, size_t ws_bytes, void *stream);
TF_API size_t tf_attention_workspace_bytes(const tf_kv_cache *c, int32_t group, int32_t R);
TF_API tf_status tf_attention_verify(const tf_kv_cache *c, int32_t group, const uint16_t *q, int32_t ldq,
                                     int32_t R, const int64_t *pos, float *out, int32_t ldo, void *ws,
                                     size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Pieces of the synthetic decoder (the steps tf_verify_step chains), public so
 * a caller can compose or check them one layer at a time.
 * ------------------------------------------------------------------------
 * tf_embed_rows: x[r][:] = float(embedding[token_r][:]) with token_0 =
 *   *last_token and token_r = drafts[r-1]; x dev fp32 [R][hidden].  An id
 *   outside [0, vocab) records TF_DEV_BAD_TOKEN in ws and uses id 0.
 * tf_rmsnorm_bf16: out[r][:] = bf16(x[r][:] / sqrt(mean(x[r]^2) + eps)), one
 *   fixed-order fp32 reduction per row; x dev fp32 [R][H], out dev bf16 [R][H].
 * tf_decoder_block: one residual SwiGLU block b of the model, in place on the
 *   fp32 residual x [R][hidden]:  n = bf16(rms(x)); h = bf16(silu(n Wg) * (n Wu));
 *   x += h Wd.  n_out (dev bf16 [R][hidden]) and h_out (dev bf16 [R][ffn]) receive
 *   the block's intermediate activations.  ws: tf_decoder_block_workspace_bytes.
 */
TF_API tf_status tf_embed_rows(const tf_model *m, const int32_t *last_token, const int32_t *drafts, int32_t R,
                               float *x, void *ws, void *stream);
TF_API tf_status tf_rmsnorm_bf16(const float *x, int32_t R, int32_t H, float eps, uint16_t *out, void *stream);
TF_API size_t tf_decoder_block_workspace_bytes(const tf_model *m);
TF_API tf_status tf_decoder_block(const tf_model *m, int32_t block, float *x, int32_t R, uint16_t *n_out,
                                  uint16_t *h_out, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Self-check and generic workspace query.
 * ------------------------------------------------------------------------
 * tf_selfcheck_row_invariance: the row-invariance guarantee (README, the two
 *   guarantees: each row of a verify pass comes out as it would alone), checked
 *   on the caller's matrix and rows.  Runs tf_lane_gemm_w4 on x[0..R-1] for every
 *   R in 1..16 and compares every row's output bytes with the one-row launch of
 *   that row.  x: dev bf16 [16][ldx]; scratch: dev, 256-B aligned, at least
 *   tf_selfcheck_scratch_bytes(W->N) bytes; ws: as for tf_lane_gemm_w4.
 *   Synchronises `stream`.  *result (host) = 0 when every row matched, else
 *   R * 256 + row of the first mismatch (smallest R, then smallest row).
 * tf_workspace_size: the workspace bytes of one operation by code, for callers
 *   that size buffers generically: TF_OP_LANE_GEMM dims {K, N, group},
 *   TF_OP_KEYED_SAMPLE dims {R, V}, TF_OP_ATTENTION dims {n_kv, max_len, group, R}.
 *   0 for an unknown code, a wrong dims count or unsupported dims.  The MoE layer
 *   and the decoder step take their descriptors: tf_moe_workspace_bytes,
 *   tf_verify_step_workspace_bytes.
 */
#define TF_OP_LANE_GEMM 1
#define TF_OP_KEYED_SAMPLE 2
#define TF_OP_ATTENTION 3
TF_API size_t tf_selfcheck_scratch_bytes(int32_t N);
TF_API tf_status tf_selfcheck_row_invariance(const tf_w4_matrix *W, const uint16_t *x, int32_t ldx, void *scratch,
                                             size_t scratch_bytes, void *ws, size_t ws_bytes, void *stream,
                                             int32_t *result);
TF_API size_t tf_workspace_size(int32_t op, const int64_t *dims, int32_t n_dims);

/* Number of SMs the split-K decomposition is sized for on the current device. */
TF_API int32_t tf_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* TF_H */
