// Keyed Gumbel-max sampling over top-k / top-p candidates, and acceptance.
//
// TensorFold README, section on the two guarantees (keyed sampling): position
// p gets the top-k/top-p candidate maximising logit/T + g(seed, p, token), g
// Gumbel noise computed from a hash of (seed, p, token); the CLI options table
// makes temperature 0 greedy.  Acceptance keeps a draft only while it matches
// what one-row decoding samples at its position.
//
// Two launches per call.  Candidates are ordered by the composite key
// (logit desc, id asc), unique per token.
//   1. topk_partial: grid (ceil(V/4096), R).  Each CTA keeps 16 logits per
//      thread in registers (coalesced loads).  The k-th largest of the 256
//      per-thread maxima bounds the chunk's k-th largest from below (k threads
//      hold an element at or above it), so only the few elements at or above it
//      survive; each survivor's rank among them gives the chunk's top k in
//      order.  When ties leave too many survivors, a 4-pass 8-bit radix select
//      over a shared histogram (ties at the threshold broken by a second select
//      on the ids) picks them instead.  Non-finite logits flag the row.
//   2. finalize: one CTA per row.  The largest of the chunks' k-th best keys
//      bounds the row's k-th best from below; the candidates at or above it are
//      ranked the same way (radix select as the fallback), giving the k' best in
//      order; then the top-p prefix in fp64 left to right and the Gumbel argmax.
// Every decision depends on the row's own logits only, so a row's token is the
// same whatever R is.
#include <atomic>

#include <cuda_runtime.h>

#include "sampler.cuh"
#include "tf_keys.cuh"
#include "tf_ptx.cuh"

namespace tfk {

namespace {

constexpr int kE1 = kSampleChunk / kSampleThreads;  // 16 logits per thread in a chunk
constexpr int kE2 = 32;                             // pool entries per thread in finalize
constexpr int kMaxChunks = kE2 * kSampleThreads / kMaxTopK;  // 128
constexpr int kSurvMax = 1024;                      // survivors ranked directly (else radix select)

// A lower bound on the k-th largest element held by the block, from each
// thread's largest key (0 for a thread that holds none).  Threads below
// n_thr hold at least one element, so warps below n_thr / 32 are full.  In
// each full warp the c-th largest thread maximum, c = ceil(k / full warps),
// has c elements at or above it; the smallest of these over the full warps
// therefore has at least k elements at or above it.  0 (every element
// survives) when no warp is full or c > 32.  Call with the whole block.
__device__ uint64_t kth_bound(uint64_t tmax, int k, int n_thr, uint64_t *s_wb) {
    const int n_full = min(n_thr, int(blockDim.x)) >> 5;
    const uint64_t v = warp_sort_desc(tmax);
    const int c = n_full > 0 ? (k + n_full - 1) / n_full : 33;
    const uint64_t vc = __shfl_sync(0xFFFFFFFFu, v, c <= 32 ? c - 1 : 0);
    if ((threadIdx.x & 31) == 0) s_wb[threadIdx.x >> 5] = vc;
    __syncthreads();
    if (c > 32) return 0ull;
    uint64_t L = ~0ull;
    for (int w = 0; w < n_full; ++w) L = s_wb[w] < L ? s_wb[w] : L;
    return L;
}

// SplitMix64 output function (Steele, Lea & Flood 2014): advance by the golden
// gamma, then the two xor-shift-multiply rounds and a final xor-shift.
__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Key of (seed, position, token id): sm(sm(sm(seed) ^ pos) ^ token), the
// position as a 64-bit two's-complement word, the token id zero-extended.
__device__ __forceinline__ uint64_t key_hash(uint64_t seed, int64_t pos, int32_t token) {
    uint64_t h = splitmix64(seed);
    h = splitmix64(h ^ static_cast<uint64_t>(pos));
    return splitmix64(h ^ static_cast<uint64_t>(static_cast<uint32_t>(token)));
}

// Gumbel noise of a key: u = ((h >> 11) + 0.5) / 2^53 in fp64 (the top value
// rounds to u = 1 and gives +inf), g = -ln(-ln u).
__device__ __forceinline__ double gumbel_of_hash(uint64_t h) {
    const double u = (__ull2double_rn(h >> 11) + 0.5) * (1.0 / 9007199254740992.0);
    return -log(-log(u));
}

// fp32 estimate of the Gumbel noise of key h, g = -ln(-ln u) with
// u = ((h >> 11) + 1/2) / 2^53.  -ln u is formed from u itself when u <= 1/2
// and as -log1p(-(1 - u)) from the exact integer 1 - u otherwise, so every
// step is well conditioned: -ln u comes out within a few 2^-24 relative and g
// within 6e-6 absolute (|g| < 23; logf and log1pf are within 1 ulp).  Keys
// with 1 - u below 2^-33 (g above ~22, and u rounding to 1 in fp64) are
// flagged for the fp64 formula.
__device__ __forceinline__ float gumbel_f32(uint64_t h, bool &needs_fp64) {
    const uint64_t k = h >> 11;
    float x;
    if (k >= (1ull << 52)) {
        const uint64_t m = ((1ull << 53) - 1ull) - k;   // 1 - u = (m + 1/2) / 2^53
        needs_fp64 = m < (1ull << 20);
        x = -log1pf(-((__ull2float_rn(m) + 0.5f) * 0x1p-53f));
    } else {
        needs_fp64 = false;
        x = -logf((__ull2float_rn(k) + 0.5f) * 0x1p-53f);
    }
    return -logf(x);
}

// Bound on the error of the fp32 top-p pass below: every candidate's
// exp((l_i - l_0) / T) comes within 2^-22 relative plus 2^-23 |x| e^x <= 4.4e-8
// absolute of the exact value (two roundings in the argument, expf within
// 2 ulp), and the sums of at most 64 such terms within 64 * 2^-24 relative, so
// the cumulative mass C_i / Z is within 1.5e-5 of the exact one; twice that
// also covers the roundings of (p +- eps) * Z.
constexpr float kTopPEps = 3e-5f;

struct Sel {
    uint32_t thr;  // key of the k-th largest element
    int need;      // how many elements equal to thr belong to the top k
    int n_eq;      // how many elements equal thr
};

// Block-wide: k-th largest of the valid keys (k >= 1 and <= number of valid).
template <int E>
__device__ Sel radix_select(const uint32_t (&key)[E], uint32_t valid, int k, uint32_t *hist, int *sh) {
    uint32_t prefix = 0, mask = 0;
    int remaining = k, n_eq = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (((valid >> e) & 1u) && (key[e] & mask) == prefix) atomicAdd(&hist[(key[e] >> shift) & 0xFFu], 1u);
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            uint32_t c[8], s = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - lane * 8 - j];
                s += c[j];
            }
            uint32_t incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const uint32_t excl = incl - s;
            if (excl < uint32_t(remaining) && uint32_t(remaining) <= incl) {
                uint32_t run = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + c[j] >= uint32_t(remaining)) {
                        sh[0] = 255 - lane * 8 - j;
                        sh[1] = int(run);
                        sh[2] = int(c[j]);
                        break;
                    }
                    run += c[j];
                }
            }
        }
        __syncthreads();
        const uint32_t d = uint32_t(sh[0]);
        remaining -= sh[1];
        n_eq = sh[2];
        prefix |= d << shift;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    return Sel{prefix, remaining, n_eq};
}

// Selects the top-k by (key desc, id asc) among valid entries; returns, per
// entry, whether it is selected (bit mask).
template <int E>
__device__ uint32_t select_top(const uint32_t (&key)[E], const int32_t (&id)[E], uint32_t valid, int k,
                               uint32_t *hist, int *sh) {
    const Sel s = radix_select<E>(key, valid, k, hist, sh);
    uint32_t id_max = 0xFFFFFFFFu;  // ties at the threshold are taken up to this id
    if (s.need < s.n_eq) {
        uint32_t key2[E];
        uint32_t v2 = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            key2[e] = ~uint32_t(id[e]);  // larger key2 = smaller id
            if (((valid >> e) & 1u) && key[e] == s.thr) v2 |= 1u << e;
        }
        const Sel s2 = radix_select<E>(key2, v2, s.need, hist, sh);
        id_max = ~s2.thr;
    }
    uint32_t chosen = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (!((valid >> e) & 1u)) continue;
        if (key[e] > s.thr || (key[e] == s.thr && uint32_t(id[e]) <= id_max)) chosen |= 1u << e;
    }
    return chosen;
}

__global__ void __launch_bounds__(kSampleThreads) topk_partial_kernel(const SampleArgs a) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    __shared__ uint32_t hist[256];
    __shared__ int sh[4];
    __shared__ int s_cnt, s_bad;
    const int c = blockIdx.x, r = blockIdx.y;
    const float *row = a.logits + (long long)r * a.ldl;
    const int base = c * kSampleChunk;
    uint32_t key[kE1];
    int32_t id[kE1];
    uint32_t valid = 0;
    bool bad = false;
#pragma unroll
    for (int e = 0; e < kE1; ++e) {
        const int idx = base + e * kSampleThreads + threadIdx.x;
        id[e] = idx;
        key[e] = 0;
        if (idx < a.V) {
            const float f = row[idx];
            bad |= !isfinite(f);
            key[e] = order_key(f);
            valid |= 1u << e;
        }
    }
    if (threadIdx.x == 0) {
        s_cnt = 0;
        s_bad = 0;
    }
    __syncthreads();
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();
    const int slot0 = r * a.n_chunks + c;
    if (s_bad) {
        if (threadIdx.x == 0) {
            atomicOr(&a.row_bad[r], 1);
            set_error(a.err, 2);
            a.cand_cnt[slot0] = 0;
        }
        return;
    }
    const int n_valid = min(kSampleChunk, a.V - base);
    const int k = min(a.k_eff, n_valid);
    float *out_val = a.cand_val + (long long)slot0 * kMaxTopK;
    int32_t *out_id = a.cand_id + (long long)slot0 * kMaxTopK;

    // lower bound on the chunk's k-th best from the per-thread maxima
    __shared__ uint64_t s_wb[kSampleThreads / 32];
    __shared__ uint64_t s_surv[kSurvMax];
    __shared__ int s_ns;
    uint64_t ck[kE1];
    uint64_t tmax = 0;
#pragma unroll
    for (int e = 0; e < kE1; ++e) {
        ck[e] = ((valid >> e) & 1u) ? composite(key[e], id[e]) : 0ull;
        tmax = ck[e] > tmax ? ck[e] : tmax;
    }
    if (threadIdx.x == 0) s_ns = 0;
    const uint64_t L = kth_bound(tmax, k, n_valid, s_wb);   // its barrier also publishes s_ns = 0
#pragma unroll
    for (int e = 0; e < kE1; ++e)
        if (ck[e] != 0ull && ck[e] >= L) {
            const int q = atomicAdd(&s_ns, 1);
            if (q < kSurvMax) s_surv[q] = ck[e];
        }
    __syncthreads();
    const int ns = s_ns;
    if (ns <= kSurvMax) {
        // the k best survivors, written in order
        for (int i = threadIdx.x; i < ns; i += kSampleThreads) {
            const uint64_t v = s_surv[i];
            int rank = 0;
            for (int j = 0; j < ns; ++j) rank += s_surv[j] > v;
            if (rank < k) {
                out_val[rank] = key_value(uint32_t(v >> 32));
                out_id[rank] = composite_id(v);
                if (rank == k - 1) a.cand_kth[slot0] = k == a.k_eff ? v : 0ull;
            }
        }
    } else {
        const uint32_t chosen = select_top<kE1>(key, id, valid, k, hist, sh);
        uint64_t kmin = ~0ull;
#pragma unroll
        for (int e = 0; e < kE1; ++e) {
            if ((chosen >> e) & 1u) {
                const int q = atomicAdd(&s_cnt, 1);
                if (q < kMaxTopK) {
                    out_val[q] = key_value(key[e]);
                    out_id[q] = id[e];
                }
                kmin = ck[e] < kmin ? ck[e] : kmin;
            }
        }
        // the k-th best is the smallest chosen key
        __shared__ unsigned long long s_kmin;
        if (threadIdx.x == 0) s_kmin = ~0ull;
        __syncthreads();
        if (kmin != ~0ull) atomicMin(&s_kmin, (unsigned long long)kmin);
        __syncthreads();
        if (threadIdx.x == 0) a.cand_kth[slot0] = k == a.k_eff ? uint64_t(s_kmin) : 0ull;
    }
    if (threadIdx.x == 0) a.cand_cnt[slot0] = k;
}

// Acceptance by the last row to finish (a.accepted set): the rows' tokens are
// published with a fence before the count, and read after it.  One row needs
// no count: it accepts nothing and its token is the bonus.
__device__ void accept_by_last_row(const SampleArgs &a, int32_t token) {
    if (a.R == 1) {   // one row: nothing to compare, it is its own bonus
        if (threadIdx.x == 0) {
            *a.accepted = 0;
            if (a.bonus) *a.bonus = token;
            if (a.acc_pos) *a.acc_pos += 1;
        }
        return;
    }
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.done, 1u) == unsigned(a.R - 1);
    }
    __syncthreads();
    if (!s_last || threadIdx.x >= 32) return;
    __threadfence();
    const int lane = threadIdx.x, R = a.R;
    const bool mismatch = lane < R - 1 && __ldcg(&a.drafts[lane]) != __ldcg(&a.tokens[lane]);
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, mismatch);
    const int acc = m ? __ffs(m) - 1 : R - 1;
    if (lane == 0) {
        const int32_t t = __ldcg(&a.tokens[acc]);
        *a.accepted = acc;
        if (a.bonus) *a.bonus = t;
        if (a.acc_pos) *a.acc_pos += acc + 1;
        *a.done = 0u;   // leave the counter zero for the next call
    }
}

__device__ __forceinline__ bool better(double s, int id, double bs, int bid) {
    return s > bs || (s == bs && id < bid);
}

// One row's token from a pool of candidate words (E per thread of NT, index
// e * NT + tid, 0 = none; n_total pool entries) holding the row's k best, L, a
// lower bound on the k-th best (0: none known), and per thread a word tmax of
// the pool such that threads below n_thr hold distinct ones (kth_bound turns
// them into a second bound).  The candidates at or above the larger bound are
// ranked (radix select when too many survive), giving the k best in order;
// then the top-p prefix in fp64 summed left to right in rank order, and the
// Gumbel argmax over it.  Call with the whole block.
template <int NT, int E>
__device__ void finalize_row(const SampleArgs &a, const int r, const uint64_t (&ck)[E], uint64_t L, uint64_t tmax,
                             int n_thr, const int k, const int n_total, const bool bad,
                             const uint64_t *wmax = nullptr) {
    __shared__ uint32_t hist[256];
    __shared__ int sh[4];
    __shared__ int s_cnt, s_m, s_ns, s_token;
    __shared__ float sel_val[kMaxTopK], srt_val[kMaxTopK];
    __shared__ int32_t sel_id[kMaxTopK], srt_id[kMaxTopK];
    __shared__ double ex[kMaxTopK], score[kMaxTopK], gsc[kMaxTopK], g_lo[kMaxTopK], g_hi[kMaxTopK];
    __shared__ float e32[kMaxTopK];
    __shared__ uint64_t g_hash[kMaxTopK];
    __shared__ int8_t g_exact[kMaxTopK];
    __shared__ uint64_t s_surv[kSurvMax];
    __shared__ uint64_t s_wb[NT / 32];
    const int tid = threadIdx.x;
    if (tid == 0) {   // published by the next barrier (kth_bound's, or the one before the token)
        s_ns = 0;
        s_cnt = 0;
        s_token = -1;
    }
    if (!bad && n_total > 0) {   // uniform over the block
        const uint64_t L2 = kth_bound(tmax, k, n_thr, s_wb);
        L = L > L2 ? L : L2;
        if (wmax)   // per-warp maxima of a third bound, written before the call
            for (int w = 0; w < NT / 32; ++w) L = wmax[w] > L ? wmax[w] : L;
        // candidates at or above the bound
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (ck[e] != 0ull && ck[e] >= L) {
                const int q = atomicAdd(&s_ns, 1);
                if (q < kSurvMax) s_surv[q] = ck[e];
            }
        __syncthreads();
        const int ns = s_ns;
        const double T = double(a.temperature);
        const double p = double(a.top_p);
        const int64_t pos = a.pos ? a.pos[r] : (*a.pos_base + r);
        const bool ranked_direct = ns <= kSurvMax;   // uniform over the block
        if (ranked_direct) {
            for (int i = tid; i < ns; i += NT) {
                const uint64_t v = s_surv[i];
                int rank = 0;
                for (int j = 0; j < ns; ++j) rank += s_surv[j] > v;
                if (rank < k) {
                    srt_val[rank] = key_value(uint32_t(v >> 32));
                    srt_id[rank] = composite_id(v);
                }
            }
            if (tid == 0) s_cnt = k;
        } else {
            uint32_t key[E];
            int32_t id[E];
            uint32_t valid = 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                key[e] = uint32_t(ck[e] >> 32);
                id[e] = composite_id(ck[e]);
                if (ck[e] != 0ull) valid |= 1u << e;
            }
            const uint32_t chosen = select_top<E>(key, id, valid, k, hist, sh);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if ((chosen >> e) & 1u) {
                    const int q = atomicAdd(&s_cnt, 1);
                    if (q < kMaxTopK) {
                        sel_val[q] = key_value(key[e]);
                        sel_id[q] = id[e];
                    }
                }
            }
            __syncthreads();
            const int n_sel = min(s_cnt, kMaxTopK);
            if (tid < n_sel) {  // rank sort by (logit desc, id asc)
                const uint64_t ki = composite(order_key(sel_val[tid]), sel_id[tid]);
                int rank = 0;
                for (int j = 0; j < n_sel; ++j) rank += composite(order_key(sel_val[j]), sel_id[j]) > ki;
                srt_val[rank] = sel_val[tid];
                srt_id[rank] = sel_id[tid];
            }
        }
        __syncthreads();
        const int n_sel = min(s_cnt, kMaxTopK);
        if (a.temperature == 0.0f) {
            if (tid == 0) s_token = srt_id[0];
        } else {
            // fp32 first, fp64 where fp32 cannot decide.  Warps 2-3 form
            // every candidate's fp32 score l/T + g with an error bound (fp64 at
            // once for a key whose 1 - u is below 2^-33), while warps 0-1 find
            // the top-p prefix from fp32 masses, falling back to the fp64 sums
            // when the cumulative mass lies within kTopPEps of p at the cut.
            // Then warp 0 takes the kept candidates whose upper bound reaches
            // the best lower bound; a single one is the token, several are
            // decided by their fp64 scores (ties to the lower id).
            if (tid >= 64 && tid < 128) {
                const int i = tid - 64;
                if (i < n_sel) {
                    const uint64_t h = key_hash(a.seed, pos, srt_id[i]);
                    const float lt = __fdiv_rn(srt_val[i], a.temperature);
                    bool exact = false;
                    const float sf = lt + gumbel_f32(h, exact);
                    g_hash[i] = h;
                    g_exact[i] = exact ? 1 : 0;
                    if (exact) {
                        gsc[i] = double(srt_val[i]) / T + gumbel_of_hash(h);
                    } else {
                        const double e = double(3e-5f + 2.4e-7f * (fabsf(lt) + fabsf(sf)));
                        g_lo[i] = double(sf) - e;
                        g_hi[i] = double(sf) + e;
                    }
                }
            }
            if (tid < 64) {
                if (p < 1.0) {
                    __shared__ double s_Z;
                    __shared__ int s_sure;
                    const float pf = a.top_p;
                    if (tid < n_sel) e32[tid] = expf(__fdiv_rn(srt_val[tid] - srt_val[0], a.temperature));
                    bar_sync_named(1, 64);
                    if (tid == 0) {
                        float Z = 0.f;
                        for (int i = 0; i < n_sel; ++i) Z += e32[i];
                        float C = 0.f, Cprev = 0.f;
                        int m = n_sel, sure = 0;
                        for (int i = 0; i < n_sel; ++i) {   // the same left-to-right cut as the fp64 sums
                            C += e32[i];
                            if (C >= pf * Z) {
                                m = i + 1;
                                sure = C >= (pf + kTopPEps) * Z && (i == 0 || Cprev < (pf - kTopPEps) * Z);
                                break;
                            }
                            Cprev = C;
                        }
                        s_m = m;
                        s_sure = sure;
                    }
                    bar_sync_named(1, 64);
                    if (!s_sure) {
                        if (tid < n_sel) ex[tid] = exp((double(srt_val[tid]) - double(srt_val[0])) / T);
                        bar_sync_named(1, 64);
                        if (tid == 0) {
                            double Z = 0.0;
                            for (int i = 0; i < n_sel; ++i) Z += ex[i];
                            s_Z = Z;
                        }
                        bar_sync_named(1, 64);
                        if (tid < n_sel) score[tid] = ex[tid] / s_Z;   // q_i, each term on its own thread
                        bar_sync_named(1, 64);
                        if (tid == 0) {
                            double S = 0.0;
                            int m = n_sel;
                            for (int i = 0; i < n_sel; ++i) {   // renormalised mass summed left to right
                                S += score[i];
                                if (S >= p) {
                                    m = i + 1;
                                    break;
                                }
                            }
                            s_m = m;
                        }
                    }
                } else if (tid == 0) {
                    s_m = n_sel;
                }
            }
            __syncthreads();
            if (tid < 32) {
                const int m = s_m;
                double lo = -1.0 / 0.0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i = tid + 32 * h;
                    if (i < m) lo = fmax(lo, g_exact[i] ? gsc[i] : g_lo[i]);
                }
                for (int o = 16; o > 0; o >>= 1) lo = fmax(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
                bool surv[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i = tid + 32 * h;
                    surv[h] = i < m && (g_exact[i] ? gsc[i] : g_hi[i]) >= lo;
                }
                const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, surv[0]), b1 = __ballot_sync(0xFFFFFFFFu, surv[1]);
                if (__popc(b0) + __popc(b1) == 1) {
                    if (tid == 0) s_token = srt_id[b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1];
                } else {
                    double bs = -1.0 / 0.0;
                    int bd = 0x7FFFFFFF;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int i = tid + 32 * h;
                        if (surv[h]) {
                            const double sc = g_exact[i] ? gsc[i] : double(srt_val[i]) / T + gumbel_of_hash(g_hash[i]);
                            if (better(sc, srt_id[i], bs, bd)) {
                                bs = sc;
                                bd = srt_id[i];
                            }
                        }
                    }
                    for (int o = 16; o > 0; o >>= 1) {
                        const double os = __shfl_xor_sync(0xFFFFFFFFu, bs, o);
                        const int od = __shfl_xor_sync(0xFFFFFFFFu, bd, o);
                        if (better(os, od, bs, bd)) {
                            bs = os;
                            bd = od;
                        }
                    }
                    if (tid == 0) s_token = bd;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        a.tokens[r] = s_token;           // -1 for a row with a non-finite logit
        if (bad) a.row_bad[r] = 0;       // leave the workspace clean for the next call
    }
    if (a.accepted) accept_by_last_row(a, s_token);
}

// Finaliser over the per-chunk candidates of topk_partial.
__global__ void __launch_bounds__(kSampleThreads) finalize_kernel(const SampleArgs a) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int nc = a.n_chunks;
    __shared__ unsigned long long s_L;
    __shared__ int s_total;
    if (tid == 0) {
        s_L = 0ull;
        s_total = 0;
    }
    __syncthreads();
    // chunk counts, their total, and the bound: the largest chunk k-th best
    for (int c = tid; c < nc; c += kSampleThreads) {
        atomicAdd(&s_total, a.cand_cnt[r * nc + c]);
        const unsigned long long kth = a.cand_kth[r * nc + c];
        if (kth) atomicMax(&s_L, kth);
    }
    __syncthreads();
    const int n_total = s_total;
    const bool bad = a.row_bad[r] != 0;
    const int k = min(a.k_eff, n_total);
    // Every chunk but the last kept exactly k_eff candidates (it had 4096 >= k_eff
    // valid logits), so candidate i of the row sits in chunk i / k_eff, slot
    // i % k_eff; the float quotient is exact here ((i + 0.5) / k_eff never lies
    // within 1/128 of an integer for i < 8192), and the loads carry no
    // data-dependent branch.
    const int ke = a.k_eff;
    const float inv_ke = 1.0f / float(ke);
    uint64_t ck[kE2];
    uint64_t tmax = 0ull;
#pragma unroll
    for (int e = 0; e < kE2; ++e) {
        const int i = e * kSampleThreads + tid;
        ck[e] = 0ull;
        if (!bad && i < n_total) {
            const int c = int((float(i) + 0.5f) * inv_ke);
            const long long q = (long long)(r * nc + c) * kMaxTopK + (i - c * ke);
            ck[e] = composite(order_key(a.cand_val[q]), a.cand_id[q]);
        }
        tmax = ck[e] > tmax ? ck[e] : tmax;
    }
    // the second bound from the per-thread maxima of the pool
    finalize_row<kSampleThreads, kE2>(a, r, ck, s_L, tmax, n_total, k, n_total, bad);
}

// Finaliser over the LM head epilogue's lists: n_chunks lists of exactly
// k_eff words per row (padded with the empty word).  Every load is issued
// before any is used: the k-th best words of the lists (their maximum bounds
// the row's k-th best from below) and the pool, E words per thread.
constexpr int kListThreads = 512;
constexpr int kE3 = 16;
__global__ void __launch_bounds__(kListThreads) finalize_lists_kernel(const SampleArgs a) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int nc = a.n_chunks, ke = a.k_eff;
    const int n_total = nc * ke;
    __shared__ uint64_t s_wmax[kListThreads / 32];
    const uint64_t kth = tid < nc ? a.cand_kth[r * nc + tid] : 0ull;
    // each list's best word (entry 0: the lists are in descending order)
    const long long q0 = (long long)(r * nc + (tid < nc ? tid : 0)) * kMaxTopK;
    const float v0 = a.cand_val[q0];
    const int32_t id0 = a.cand_id[q0];
    const float inv_ke = 1.0f / float(ke);
    float v[kE3];
    int32_t id[kE3];
#pragma unroll
    for (int e = 0; e < kE3; ++e) {
        const int i = e * kListThreads + tid;
        const int ii = i < n_total ? i : 0;
        const int c = int((float(ii) + 0.5f) * inv_ke);
        const long long q = (long long)(r * nc + c) * kMaxTopK + (ii - c * ke);
        v[e] = a.cand_val[q];
        id[e] = a.cand_id[q];
    }
    const bool bad = a.row_bad[r] != 0;
    uint64_t wm = kth;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t x = __shfl_xor_sync(0xFFFFFFFFu, wm, o);
        wm = x > wm ? x : wm;
    }
    if ((tid & 31) == 0) s_wmax[tid >> 5] = wm;   // the largest list k-th best: a bound on the row's
    uint64_t ck[kE3];
#pragma unroll
    for (int e = 0; e < kE3; ++e)
        ck[e] = (!bad && e * kListThreads + tid < n_total) ? composite(order_key(v[e]), id[e]) : 0ull;
    // the second bound from the lists' best words: thread c < nc holds list c's
    const uint64_t lmax = (!bad && tid < nc) ? composite(order_key(v0), id0) : 0ull;
    if (tid == 0) a.bound[r] = 0ull;   // the GEMM that shared it has finished
    finalize_row<kListThreads, kE3>(a, r, ck, 0ull, lmax, nc, ke, n_total, bad, s_wmax);
}

// ---- general candidate path: T > 0 with k' > 64 candidates ----
// Same candidate set and selection as the fast path (rank order by (logit
// desc, id asc), the first k', then the top-p prefix, then the Gumbel argmax),
// for any k' up to V.  Every reduction runs in a fixed order or on integers,
// so a row's token depends on its own logits only:
//   gen_prep   (chunk, row): the chunk's largest key; non-finite logits flag the row.
//   gen_select (row): the k'-th largest key tau by an 8-bit radix select,
//              most significant digit first; once the digit's bin is small
//              its keys are gathered into shared memory and the remaining
//              digits are read there.  (tau = 0 when k' = V.)
//   gen_exp    (sub-chunk of 1024, row; top_p < 1): e_i = exp((l_i - l_0) / T)
//              in fp64 for the candidates (key >= tau), kept as the 53-bit
//              fixed-point mass q_i = floor(2^53 e_i) (e_i <= 1), and the
//              sub-chunk's sum of them.
//   gen_walk   (sub-chunk, row; top_p < 1; passes 1..7, then gen_walk_final):
//              the top-p boundary b, the largest key with sum_{key >= b} q >=
//              top_p * Z (Z = sum q), by an 8-bit radix walk, most significant
//              digit first.  Pass k adds the masses, counts and largest keys of
//              the digit at bit 56 - 8k of the keys inside the bins chosen so
//              far into global bins (integer atomics: exact in any order);
//              every CTA of pass k + 1 reads them and takes the same decision
//              (a scan over the bins from the top), so the walk needs no grid
//              barrier.  gen_exp is pass 0.  It stops at a bin of one key.
//   gen_score  (sub-chunk, row): the best (l / T + g, id) among keys >= b; an
//              fp32 estimate of every score with a bound on its error leaves
//              fp64 only to the scores that can still be the best.
//   gen_final  (row): the best over the sub-chunks.
// The masses are exact sums of weights truncated to multiples of 2^-53, so
// the boundary agrees with the left-to-right fp64 sum of the definition
// except when the mass reaching it lies within about V * 2^-53 (~2e-11 for
// V = 151936) of top_p * Z, relative to Z >= 1.
constexpr int kGenThreads = 512;
constexpr int kGenSub = 1024;                        // sub-chunk of gen_exp / gen_score
constexpr int kGenSubThreads = 256;
constexpr int kGenE = kGenSub / kGenSubThreads;      // 4 elements a thread
constexpr int kSelectCompact = 8192;                 // keys gen_select gathers (64 KB)
constexpr int kWalkPasses = 8;                       // 8-bit digits of the 64-bit keys

__device__ __forceinline__ uint64_t row_composite(const float *row, int i) { return composite(order_key(row[i]), i); }

// 128-bit unsigned sums of the 53-bit fixed-point masses (at most 2^19
// entries of at most 2^53 each).
struct U128 {
    unsigned long long lo, hi;
};
__device__ __forceinline__ U128 add128(U128 a, U128 b) {
    U128 r;
    r.lo = a.lo + b.lo;
    r.hi = a.hi + b.hi + (r.lo < a.lo ? 1ull : 0ull);
    return r;
}
__device__ __forceinline__ U128 warp_sum128(U128 v) {
    for (int o = 16; o > 0; o >>= 1) {
        U128 x;
        x.lo = __shfl_xor_sync(0xFFFFFFFFu, v.lo, o);
        x.hi = __shfl_xor_sync(0xFFFFFFFFu, v.hi, o);
        v = add128(v, x);
    }
    return v;
}
__device__ __forceinline__ double to_double(U128 a) { return double(a.hi) * 18446744073709551616.0 + double(a.lo); }

// Walk bins of one pass and row: 256 digits of (mass as 128 bits, count,
// largest key).  Buffer (pass % 3) is written by pass `pass`, read by pass
// + 1 and cleared by pass - 1 (gen_prep clears buffer 0).
struct WalkBin {
    unsigned long long lo, hi, maxkey;
    unsigned cnt, pad;
};
__device__ __forceinline__ WalkBin *walk_bins(const SampleArgs &a, int pass, int r) {
    return reinterpret_cast<WalkBin *>(a.gen_walk) + ((long long)(pass % 3) * a.R + r) * 256;
}

// The row's walk state after a decision: prefix / mask of the digits chosen,
// the mass of the candidates above the current bin, the target top_p * Z,
// and once done the boundary.
struct WalkState {
    unsigned long long prefix, mask, acc_lo, acc_hi, beta;
    double target;
    int done, pad;
};

// Clears this CTA's share of the buffer of `pass` for row r (blocks of the
// grid's x dimension split the 256 bins).
__device__ __forceinline__ void walk_clear(const SampleArgs &a, int pass, int r) {
    WalkBin *b = walk_bins(a, pass, r);
    for (int d = blockIdx.x * blockDim.x + threadIdx.x; d < 256; d += gridDim.x * blockDim.x) b[d] = WalkBin{0, 0, 0, 0, 0};
}

// Adds this CTA's keys (candidate, inside prefix / mask) to the bins of the
// digit at `shift`: shared-memory bins first, then one global update per
// bin that was hit.
__device__ void walk_histogram(const SampleArgs &a, int pass, int r, int shift, uint64_t prefix, uint64_t mask,
                               const uint64_t (&key)[kGenE], const uint64_t (&q)[kGenE], bool (&in)[kGenE]) {
    __shared__ unsigned long long s_m[256], s_k[256];
    __shared__ unsigned s_c[256];
    for (int d = threadIdx.x; d < 256; d += blockDim.x) {
        s_m[d] = 0ull;
        s_k[d] = 0ull;
        s_c[d] = 0u;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kGenE; ++e)
        if (in[e] && (key[e] & mask) == prefix) {
            const int d = int((key[e] >> shift) & 0xFFu);
            atomicAdd(&s_m[d], (unsigned long long)q[e]);   // < 1024 * 2^53 per CTA
            atomicAdd(&s_c[d], 1u);
            atomicMax(&s_k[d], (unsigned long long)key[e]);
        }
    __syncthreads();
    WalkBin *b = walk_bins(a, pass, r);
    for (int d = threadIdx.x; d < 256; d += blockDim.x) {
        if (!s_c[d]) continue;
        const unsigned long long old = atomicAdd(&b[d].lo, s_m[d]);
        if (old + s_m[d] < old) atomicAdd(&b[d].hi, 1ull);   // the carries add up to the same in any order
        atomicAdd(&b[d].cnt, s_c[d]);
        atomicMax(&b[d].maxkey, s_k[d]);
    }
}

// The decision on the bins of the digit at `shift` (buffer of `pass`): the
// highest non-empty digit whose mass, added to the mass above it, reaches the
// target.  256 threads, one digit each; the same result in every CTA.
__device__ void walk_decide(const SampleArgs &a, int pass, int r, int shift, WalkState &st, uint64_t tau) {
    __shared__ unsigned long long s_lo[8], s_hi[8];
    __shared__ int s_pick;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int d = 255 - t;   // thread t: digit 255 - t, so the scan runs from the top
    const WalkBin bn = walk_bins(a, pass, r)[d];
    // inclusive scan of the masses from digit 255 down to d
    U128 v{bn.lo, bn.hi};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        U128 x;
        x.lo = __shfl_up_sync(0xFFFFFFFFu, v.lo, o);
        x.hi = __shfl_up_sync(0xFFFFFFFFu, v.hi, o);
        if (lane >= o) v = add128(v, x);
    }
    if (lane == 31) {
        s_lo[w] = v.lo;
        s_hi[w] = v.hi;
    }
    if (t == 0) s_pick = 256;
    __syncthreads();
    for (int k = 0; k < w; ++k) v = add128(v, U128{s_lo[k], s_hi[k]});
    const U128 reach = add128(U128{st.acc_lo, st.acc_hi}, v);
    if (bn.cnt && to_double(reach) >= st.target) atomicMin(&s_pick, t);   // the first from the top
    __syncthreads();
    const int pick = s_pick;
    if (pick == 256) {   // the whole mass stays below top_p * Z: keep all k'
        st.done = 1;
        st.beta = tau;
    } else {
        __shared__ WalkBin s_bin;
        __shared__ U128 s_acc;
        if (t == pick) {
            s_bin = bn;
            // the mass above the chosen digit: reach minus its own
            U128 above = reach;
            above.hi -= bn.hi + (above.lo < bn.lo ? 1ull : 0ull);
            above.lo -= bn.lo;
            s_acc = above;
        }
        __syncthreads();
        st.prefix |= uint64_t(255 - pick) << shift;
        st.mask |= 0xFFull << shift;
        st.acc_lo = s_acc.lo;
        st.acc_hi = s_acc.hi;
        if (s_bin.cnt == 1u || shift == 0) {
            st.done = 1;
            st.beta = s_bin.maxkey;
        }
    }
    __syncthreads();
}

// Loads this CTA's keys and masses (the candidates of sub-chunk c of row r).
__device__ __forceinline__ void walk_load(const SampleArgs &a, int r, int c, uint64_t tau, uint64_t (&key)[kGenE],
                                          uint64_t (&q)[kGenE], bool (&in)[kGenE]) {
    const float *row = a.logits + (long long)r * a.ldl;
#pragma unroll
    for (int e = 0; e < kGenE; ++e) {
        const int i = c * kGenSub + e * kGenSubThreads + threadIdx.x;
        in[e] = i < a.V;
        key[e] = in[e] ? row_composite(row, i) : 0ull;
        q[e] = in[e] ? a.gen_q[(long long)r * a.V + i] : 0ull;
        in[e] = in[e] && key[e] >= tau;
    }
}

__global__ void __launch_bounds__(kSampleThreads) gen_prep_kernel(const SampleArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    __shared__ unsigned long long s_max;
    __shared__ int s_bad;
    const int c = blockIdx.x, r = blockIdx.y;
    const float *row = a.logits + (long long)r * a.ldl;
    if (threadIdx.x == 0) {
        s_max = 0ull;
        s_bad = 0;
    }
    __syncthreads();
    uint64_t m = 0ull;
    bool bad = false;
    for (int e = 0; e < kE1; ++e) {
        const int i = c * kSampleChunk + e * kSampleThreads + threadIdx.x;
        if (i < a.V) {
            bad |= !isfinite(row[i]);
            const uint64_t v = row_composite(row, i);
            m = v > m ? v : m;
        }
    }
    atomicMax(&s_max, (unsigned long long)m);
    if (bad) atomicOr(&s_bad, 1);
    if (a.top_p < 1.0f) walk_clear(a, 0, r);   // the top-p walk's first bins
    __syncthreads();
    if (threadIdx.x == 0) {
        a.gen_cmax[r * a.n_chunks + c] = s_max;
        if (s_bad) {
            atomicOr(&a.row_bad[r], 1);
            set_error(a.err, 2);
        }
    }
}

// Counts key into hist[digit] with one shared atomic per distinct digit of the warp.
__device__ __forceinline__ void hist_add(unsigned *hist, bool take, unsigned digit) {
    const unsigned act = __ballot_sync(0xFFFFFFFFu, take);
    if (!act) return;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, take ? digit : 0xFFFFFFFFu);
    const int lane = threadIdx.x & 31;
    if (take && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], unsigned(__popc(peers)));
}

__global__ void __launch_bounds__(kGenThreads) gen_select_kernel(const SampleArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    extern __shared__ uint64_t gsel[];   // [kSelectCompact] gathered keys
    __shared__ unsigned hist[256];
    __shared__ int s_int[3];
    __shared__ int s_n;
    const int r = blockIdx.x, tid = threadIdx.x;
    const float *row = a.logits + (long long)r * a.ldl;
    const int V = a.V;
    if (a.row_bad[r]) {
        if (tid == 0) a.gen_thr[r] = ~0ull;   // no candidates: gen_final writes -1
        return;
    }
    uint64_t tau = 0ull;   // k' = V: every key
    if (a.k_eff < V) {
        uint64_t prefix = 0ull, mask = 0ull;
        int remaining = a.k_eff, n_c = -1;   // n_c >= 0: the bin's keys sit in gsel[0, n_c)
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kGenThreads) hist[i] = 0u;
            __syncthreads();
            if (n_c < 0) {
                for (int i0 = 0; i0 < V; i0 += kGenThreads) {   // whole warps, for the vote
                    const int i = i0 + tid;
                    const uint64_t cv = i < V ? row_composite(row, i) : 0ull;
                    hist_add(hist, i < V && (cv & mask) == prefix, unsigned(cv >> shift) & 0xFFu);
                }
            } else {
                for (int j0 = 0; j0 < n_c; j0 += kGenThreads) {
                    const int j = j0 + tid;
                    const uint64_t cv = j < n_c ? gsel[j] : 0ull;
                    hist_add(hist, j < n_c && (cv & mask) == prefix, unsigned(cv >> shift) & 0xFFu);
                }
            }
            __syncthreads();
            if (tid == 0) {
                int run = 0, d = 255;
                for (; d > 0; --d) {
                    if (run + int(hist[d]) >= remaining) break;
                    run += int(hist[d]);
                }
                s_int[0] = d;
                s_int[1] = run;
                s_int[2] = int(hist[d]);
            }
            __syncthreads();
            prefix |= uint64_t(s_int[0]) << shift;
            mask |= 0xFFull << shift;
            remaining -= s_int[1];
            if (n_c < 0 && shift > 0 && s_int[2] <= kSelectCompact) {   // gather the bin (any order: counts only)
                if (tid == 0) s_n = 0;
                __syncthreads();
                for (int i = tid; i < V; i += kGenThreads) {
                    const uint64_t cv = row_composite(row, i);
                    if ((cv & mask) == prefix) gsel[atomicAdd(&s_n, 1)] = cv;
                }
                __syncthreads();
                n_c = s_n;
            }
            __syncthreads();
        }
        tau = prefix;
    }
    if (tid == 0) a.gen_thr[r] = tau;
}

__global__ void __launch_bounds__(kGenSubThreads) gen_exp_kernel(const SampleArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    __shared__ unsigned long long s_top;
    __shared__ unsigned long long s_w[kGenSubThreads / 32];
    const int c = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const uint64_t tau = a.gen_thr[r];
    if (tid == 0) s_top = 0ull;
    __syncthreads();
    for (int k = tid; k < a.n_chunks; k += kGenSubThreads) atomicMax(&s_top, (unsigned long long)a.gen_cmax[r * a.n_chunks + k]);
    __syncthreads();
    if (tau == ~0ull) {   // row with a non-finite logit: no walk
        walk_clear(a, 1, r);
        return;
    }
    const float *row = a.logits + (long long)r * a.ldl;
    const double l0 = double(key_value(uint32_t(s_top >> 32)));
    const double T = double(a.temperature);
    unsigned long long part = 0ull;   // < 1024 * 2^53: no overflow
    uint64_t key[kGenE], q[kGenE];
    bool in[kGenE];
#pragma unroll
    for (int e = 0; e < kGenE; ++e) {
        const int i = c * kGenSub + e * kGenSubThreads + tid;
        key[e] = 0ull;
        q[e] = 0ull;
        in[e] = false;
        if (i < a.V) {
            key[e] = row_composite(row, i);
            in[e] = key[e] >= tau;
            // e <= 1 (l_0 is the largest logit), so 2^53 e is at most 2^53
            q[e] = in[e] ? __double2ull_rz(9007199254740992.0 * exp((double(row[i]) - l0) / T)) : 0ull;
            a.gen_q[(long long)r * a.V + i] = q[e];
            part += q[e];
        }
    }
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
    if ((tid & 31) == 0) s_w[tid >> 5] = part;
    __syncthreads();
    if (tid == 0) {
        unsigned long long z = 0ull;
        for (int w = 0; w < kGenSubThreads / 32; ++w) z += s_w[w];
        a.gen_zp[r * a.n_sub + c] = z;
    }
    // walk pass 0: the top digit of every candidate key
    walk_clear(a, 1, r);
    walk_histogram(a, 0, r, 56, 0ull, 0ull, key, q, in);
}



// Pass `pass` (1..7): decide on the previous pass's bins, then (if the walk
// goes on) histogram the next digit.
__global__ void __launch_bounds__(kGenSubThreads) gen_walk_kernel(const SampleArgs a, int pass) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int c = blockIdx.x, r = blockIdx.y;
    const uint64_t tau = a.gen_thr[r];
    WalkState *gst = reinterpret_cast<WalkState *>(a.gen_state) + r;
    WalkState st;
    if (pass == 1) {
        st = WalkState{0ull, 0ull, 0ull, 0ull, 0ull, 0.0, tau == ~0ull ? 1 : 0, 0};
        if (!st.done) {   // Z = the sub-chunk sums (integers: any order gives the same)
            __shared__ U128 s_z;
            if (threadIdx.x < 32) {
                U128 z{0ull, 0ull};
                for (int k = threadIdx.x; k < a.n_sub; k += 32) z = add128(z, U128{a.gen_zp[r * a.n_sub + k], 0ull});
                z = warp_sum128(z);
                if (threadIdx.x == 0) s_z = z;
            }
            __syncthreads();
            st.target = double(a.top_p) * to_double(s_z);
        }
    } else {
        st = *gst;
    }
    if (!st.done) walk_decide(a, pass - 1, r, 56 - 8 * (pass - 1), st, tau);
    if (c == 0 && threadIdx.x == 0) *gst = st;
    walk_clear(a, pass + 1, r);
    if (st.done) return;
    uint64_t key[kGenE], q[kGenE];
    bool in[kGenE];
    walk_load(a, r, c, tau, key, q, in);
    walk_histogram(a, pass, r, 56 - 8 * pass, st.prefix, st.mask, key, q, in);
}

// The last decision (digit at bit 0): the boundary is then one key.
__global__ void gen_walk_final_kernel(const SampleArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int r = blockIdx.x;
    const uint64_t tau = a.gen_thr[r];
    WalkState st = reinterpret_cast<WalkState *>(a.gen_state)[r];
    if (!st.done) walk_decide(a, kWalkPasses - 1, r, 0, st, tau);
    if (threadIdx.x == 0 && tau != ~0ull) a.gen_thr[r] = st.beta;
}

__global__ void __launch_bounds__(kGenSubThreads) gen_score_kernel(const SampleArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    __shared__ double s_sc[kGenSubThreads / 32];
    __shared__ int s_id[kGenSubThreads / 32];
    __shared__ float s_lb[kGenSubThreads / 32];
    const int c = blockIdx.x, r = blockIdx.y, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float *row = a.logits + (long long)r * a.ldl;
    const uint64_t thr = a.gen_thr[r];
    const float Tf = a.temperature;
    const double T = double(Tf);
    const int64_t pos = a.pos ? a.pos[r] : (*a.pos_base + r);
    // fp32 scores s with an error bound: s + err bounds the exact l / T + g
    // from above, s - err from below; only a score whose upper bound reaches
    // the chunk's best lower bound can be the chunk's best
    float s32[kGenE], err[kGenE];
    uint64_t hk[kGenE];
    bool cand[kGenE], exact[kGenE];
    float lb = -1.0f / 0.0f;
#pragma unroll
    for (int e = 0; e < kGenE; ++e) {
        const int i = c * kGenSub + e * kGenSubThreads + threadIdx.x;
        cand[e] = i < a.V && row_composite(row, i) >= thr;
        exact[e] = false;
        s32[e] = -1.0f / 0.0f;
        err[e] = 0.f;
        hk[e] = 0ull;
        if (cand[e]) {
            hk[e] = key_hash(a.seed, pos, i);
            const float lt = __fdiv_rn(row[i], Tf);
            s32[e] = lt + gumbel_f32(hk[e], exact[e]);
            err[e] = 3e-5f + 2.4e-7f * (fabsf(lt) + fabsf(s32[e]));
            if (!exact[e]) lb = fmaxf(lb, s32[e] - err[e]);
        }
    }
    for (int o = 16; o > 0; o >>= 1) lb = fmaxf(lb, __shfl_xor_sync(0xFFFFFFFFu, lb, o));
    if (lane == 0) s_lb[w] = lb;
    __syncthreads();
    lb = s_lb[0];
    for (int k = 1; k < kGenSubThreads / 32; ++k) lb = fmaxf(lb, s_lb[k]);
    double best = -1.0 / 0.0;
    int best_id = 0x7FFFFFFF;
#pragma unroll
    for (int e = 0; e < kGenE; ++e) {
        const int i = c * kGenSub + e * kGenSubThreads + threadIdx.x;
        if (cand[e] && (exact[e] || s32[e] + err[e] >= lb)) {
            const double sc = double(row[i]) / T + gumbel_of_hash(hk[e]);
            if (better(sc, i, best, best_id)) {
                best = sc;
                best_id = i;
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const double ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int oid = __shfl_xor_sync(0xFFFFFFFFu, best_id, o);
        if (better(ob, oid, best, best_id)) {
            best = ob;
            best_id = oid;
        }
    }
    if (lane == 0) {
        s_sc[w] = best;
        s_id[w] = best_id;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < kGenSubThreads / 32; ++k)
            if (better(s_sc[k], s_id[k], best, best_id)) {
                best = s_sc[k];
                best_id = s_id[k];
            }
        a.gen_bscore[r * a.n_sub + c] = best;
        a.gen_bid[r * a.n_sub + c] = best_id;
    }
}

__global__ void gen_final_kernel(const SampleArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int r = blockIdx.x, lane = threadIdx.x;
    double best = -1.0 / 0.0;
    int best_id = 0x7FFFFFFF;
    for (int c = lane; c < a.n_sub; c += 32)
        if (better(a.gen_bscore[r * a.n_sub + c], a.gen_bid[r * a.n_sub + c], best, best_id)) {
            best = a.gen_bscore[r * a.n_sub + c];
            best_id = a.gen_bid[r * a.n_sub + c];
        }
    for (int o = 16; o > 0; o >>= 1) {
        const double ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int oid = __shfl_xor_sync(0xFFFFFFFFu, best_id, o);
        if (better(ob, oid, best, best_id)) {
            best = ob;
            best_id = oid;
        }
    }
    if (lane == 0) {
        if (a.row_bad[r]) {
            a.tokens[r] = -1;
            a.row_bad[r] = 0;   // leave the workspace clean for the next call
        } else {
            a.tokens[r] = best_id;
        }
    }
}

__global__ void accept_kernel(const int32_t *drafts, const int32_t *sampled, int R, int32_t *accepted,
                              int32_t *bonus, int64_t *pos) {
    grid_dependency_wait();     // inputs come from the preceding grid
    grid_launch_dependents();
    const int lane = threadIdx.x;
    const bool mismatch = lane < R - 1 && drafts[lane] != sampled[lane];
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, mismatch);
    const int acc = m ? __ffs(m) - 1 : R - 1;
    if (lane == 0) {
        const int32_t t = sampled[acc];
        if (accepted) *accepted = acc;
        if (bonus) *bonus = t;
        if (pos) *pos += acc + 1;
    }
}

}  // namespace

static int n_chunks_of(int V) { return (V + kSampleChunk - 1) / kSampleChunk; }

// The 256-B header both layouts start with, every word left zero by the calls
// that use it: row_bad[kMaxRows] at 0, the finished-row counter at 64, the
// candidate epilogue's shared bounds [kMaxRows] at 128.  A workspace can
// serve calls of either path and any R.
static void bind_header(SampleArgs &a, char *p) {
    a.row_bad = reinterpret_cast<int32_t *>(p);
    a.done = reinterpret_cast<unsigned *>(p + 64);
    a.bound = reinterpret_cast<uint64_t *>(p + 128);
}

// Region layout: the header (bind_header) at a fixed offset and sized for the
// largest R, so a workspace reused by calls with different R never sees stale
// flags; the candidate arrays that follow are always written before read.
size_t sample_workspace_bytes(int R, int V) {
    const size_t nc = size_t(n_chunks_of(V));
    size_t b = 256;  // header (bind_header)
    b += size_t(R) * nc * sizeof(uint64_t);
    b += size_t(R) * nc * kMaxTopK * (sizeof(float) + sizeof(int32_t));
    b += size_t(R) * nc * sizeof(int32_t);
    b = (b + 255) / 256 * 256;
    // general path: chunk maxima, per-row boundary, e_i, sub-chunk sums and bests
    const size_t ns = size_t((V + kGenSub - 1) / kGenSub);
    b += size_t(R) * nc * sizeof(uint64_t) + size_t(R) * sizeof(uint64_t);
    b = (b + 255) / 256 * 256;
    b += size_t(R) * size_t(V) * sizeof(double);
    b += size_t(R) * ns * (2 * sizeof(double) + sizeof(int32_t));
    b = (b + 255) / 256 * 256;
    b += size_t(3) * R * 256 * sizeof(WalkBin) + size_t(R) * sizeof(WalkState);   // top-p walk
    return (b + 255) / 256 * 256;
}

void sample_bind_workspace(SampleArgs &a, void *ws_region, int R, int V) {
    const size_t nc = size_t(n_chunks_of(V));
    char *p = static_cast<char *>(ws_region);
    bind_header(a, p);
    p += 256;
    a.cand_kth = reinterpret_cast<uint64_t *>(p);
    p += size_t(R) * nc * sizeof(uint64_t);
    a.cand_val = reinterpret_cast<float *>(p);
    p += size_t(R) * nc * kMaxTopK * sizeof(float);
    a.cand_id = reinterpret_cast<int32_t *>(p);
    p += size_t(R) * nc * kMaxTopK * sizeof(int32_t);
    a.cand_cnt = reinterpret_cast<int32_t *>(p);
    p += size_t(R) * nc * sizeof(int32_t);
    p = static_cast<char *>(ws_region) + (size_t(p - static_cast<char *>(ws_region)) + 255) / 256 * 256;
    a.gen_cmax = reinterpret_cast<uint64_t *>(p);
    p += size_t(R) * nc * sizeof(uint64_t);
    a.gen_thr = reinterpret_cast<uint64_t *>(p);
    p += size_t(R) * sizeof(uint64_t);
    p = static_cast<char *>(ws_region) + (size_t(p - static_cast<char *>(ws_region)) + 255) / 256 * 256;
    a.gen_q = reinterpret_cast<uint64_t *>(p);
    p += size_t(R) * size_t(V) * sizeof(uint64_t);
    const size_t ns = size_t((V + kGenSub - 1) / kGenSub);
    a.gen_zp = reinterpret_cast<uint64_t *>(p);
    p += size_t(R) * ns * sizeof(uint64_t);
    a.gen_bscore = reinterpret_cast<double *>(p);
    p += size_t(R) * ns * sizeof(double);
    a.gen_bid = reinterpret_cast<int32_t *>(p);
    p += size_t(R) * ns * sizeof(int32_t);
    p = static_cast<char *>(ws_region) + (size_t(p - static_cast<char *>(ws_region)) + 255) / 256 * 256;
    a.gen_walk = p;
    p += size_t(3) * R * 256 * sizeof(WalkBin);
    a.gen_state = p;
    a.n_chunks = int(nc);
    a.n_sub = int(ns);
}

// The general path's shared-memory opt-in, once per device.
cudaError_t gen_opt_in() {
    static std::atomic<bool> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(gen_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSelectCompact * sizeof(uint64_t)));
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
    return e;
}

cudaError_t launch_keyed_sample(const SampleArgs &a, cudaStream_t s) {
    if (a.n_chunks > kMaxChunks) return cudaErrorInvalidValue;
    if (a.temperature > 0.0f && a.k_eff > kMaxTopK) {   // general candidate path
        cudaError_t e = gen_opt_in();
        if (e == cudaSuccess) e = launch_pdl(gen_prep_kernel, dim3(a.n_chunks, a.R), dim3(kSampleThreads), 0, s, a);
        if (e == cudaSuccess)
            e = launch_pdl(gen_select_kernel, dim3(a.R), dim3(kGenThreads), kSelectCompact * sizeof(uint64_t), s, a);
        if (a.top_p < 1.0f) {
            if (e == cudaSuccess) e = launch_pdl(gen_exp_kernel, dim3(a.n_sub, a.R), dim3(kGenSubThreads), 0, s, a);
            for (int pass = 1; pass < kWalkPasses && e == cudaSuccess; ++pass)
                e = launch_pdl(gen_walk_kernel, dim3(a.n_sub, a.R), dim3(kGenSubThreads), 0, s, a, pass);
            if (e == cudaSuccess) e = launch_pdl(gen_walk_final_kernel, dim3(a.R), dim3(256), 0, s, a);
        }
        if (e == cudaSuccess) e = launch_pdl(gen_score_kernel, dim3(a.n_sub, a.R), dim3(kGenSubThreads), 0, s, a);
        if (e == cudaSuccess) e = launch_pdl(gen_final_kernel, dim3(a.R), dim3(32), 0, s, a);
        if (e == cudaSuccess && a.accepted) e = launch_accept(a.drafts, a.tokens, a.R, a.accepted, a.bonus, a.acc_pos, s);
        return e;
    }
    cudaError_t e = launch_pdl(topk_partial_kernel, dim3(a.n_chunks, a.R), dim3(kSampleThreads), 0, s, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(finalize_kernel, dim3(a.R), dim3(kSampleThreads), 0, s, a);   // accepts too
}

// ---- candidates written by the LM head's epilogue ----
size_t sample_candidate_bytes(int R, int nc) {
    size_t b = 256;  // the header of sample_workspace_bytes
    b += size_t(R) * nc * sizeof(uint64_t);
    b += size_t(R) * nc * kMaxTopK * (sizeof(float) + sizeof(int32_t));
    b += size_t(R) * nc * sizeof(int32_t);
    return (b + 255) / 256 * 256;
}

void sample_bind_candidates(SampleArgs &a, void *region, int R, int nc) {
    char *p = static_cast<char *>(region);
    bind_header(a, p);
    p += 256;
    a.cand_kth = reinterpret_cast<uint64_t *>(p);
    p += size_t(R) * nc * sizeof(uint64_t);
    a.cand_val = reinterpret_cast<float *>(p);
    p += size_t(R) * nc * kMaxTopK * sizeof(float);
    a.cand_id = reinterpret_cast<int32_t *>(p);
    p += size_t(R) * nc * kMaxTopK * sizeof(int32_t);
    a.cand_cnt = reinterpret_cast<int32_t *>(p);
    a.n_chunks = nc;
}

bool sample_candidates_fit(int nc, int k_eff) {
    return nc >= 1 && nc <= kListThreads && k_eff >= 1 && k_eff <= kMaxTopK &&
           (long long)nc * k_eff <= (long long)kE3 * kListThreads;
}

cudaError_t launch_sample_finalize(const SampleArgs &a, cudaStream_t s) {
    if (!sample_candidates_fit(a.n_chunks, a.k_eff)) return cudaErrorInvalidValue;
    return launch_pdl(finalize_lists_kernel, dim3(a.R), dim3(kListThreads), 0, s, a);
}

cudaError_t launch_accept(const int32_t *drafts, const int32_t *sampled, int R, int32_t *accepted, int32_t *bonus,
                          int64_t *pos, cudaStream_t s) {
    return launch_pdl(accept_kernel, dim3(1), dim3(32), 0, s, drafts, sampled, R, accepted, bonus, pos);
}

int sample_max_vocab() { return kMaxChunks * kSampleChunk; }

namespace {
// The sampler's own key and Gumbel functions, evaluated for a list of
// (seed, position, token) triples.
__global__ void keyed_hash_kernel(const uint64_t *seed, const int64_t *pos, const int32_t *token, long long n,
                                  uint64_t *h_out, double *g_out) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const uint64_t h = key_hash(seed[i], pos[i], token[i]);
        if (h_out) h_out[i] = h;
        if (g_out) g_out[i] = gumbel_of_hash(h);
    }
}
}  // namespace

cudaError_t launch_keyed_hash(const uint64_t *seed, const int64_t *pos, const int32_t *token, long long n,
                              uint64_t *h_out, double *g_out, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    keyed_hash_kernel<<<unsigned(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(seed, pos, token, n, h_out, g_out);
    return cudaGetLastError();
}

}  // namespace tfk
