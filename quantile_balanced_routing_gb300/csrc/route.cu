// Router scores, Quantile Balancing and biased top-k (fp32, bit-reproducible).
//
// [K3-width] = "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club).
//   Q&A on Quantile Balancing: per-expert bias = (1 - k/n) quantile over the
//     batch of the expert's margin, minus a common offset; target load T*k/n.
//   延伸解读 "QB vs DeepSeek-V3": the bias is the exact coordinate minimiser of
//     the balanced-assignment dual (no step size).
//   Q&A on routing: sigmoid scores, top-k on score + bias, mixture weights =
//     raw scores renormalised over the chosen k, bias frozen at inference.
//
// Kernels (one sweep = token pass + expert select):
//   k_scores        s = score_of_logit(logit), elementwise (only when no sweep
//                   runs; otherwise the first token pass computes s)
//   k_token_pass    per token: top-(k+1) of v = s + b (threshold gather and a
//                   warp sort, or ranking rounds); margins m = s - tau written
//                   transposed [n, T] via SMEM
//   k_expert_select per expert: exact r-th and (r+1)-th largest margin by a
//                   4-pass 8-bit radix select with warp-aggregated SMEM
//                   histograms (later passes over the first bucket's keys);
//                   b'_j = -midpoint
//   k_topk          per token: top-k of s + b, rank-order weights, per-block
//                   expert counts
//   k_block_scan    per expert: exclusive prefix of block counts, loads
// The common offset b = b' - (pairwise-tree sum of b') / n is applied by every
// CTA of the kernel that reads the biases next (stage_bias).
#include "common.cuh"

#include <algorithm>
#include <climits>
#include <cstdio>

namespace {

using namespace qb;

constexpr int kTokPassTokens = 8;    // tokens per CTA in the token pass (one per warp)
constexpr int kTokPassWarps = 8;
constexpr int kTopkWarps = 8;
constexpr int kSelectThreads = 256;
constexpr int kSelectSmemMaxT = 48 * 1024;   // margins staged in SMEM up to this T
constexpr int kSelectCand = 1024;            // candidate words after the first digit pass (6 CTAs per SM at T = 4096)

__global__ void k_scores(const float* __restrict__ logits, float* __restrict__ scores, long long count,
                         int32_t* __restrict__ zero, int nzero) {
    if (zero && blockIdx.x == 0)
        for (int j = threadIdx.x; j < nzero; j += blockDim.x) zero[j] = 0;   // for the top-k's load counts
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (; i < count; i += stride) scores[i] = score_of_logit(logits[i]);
}

// Ranking of one token's n values v (lane owns slots j = lane + 32 c) under
// (value desc, index asc).  Values are compared through order keys
// (f32_order_key of v with -0 folded into +0, 0 for padding slots), so a
// warp's next-ranked entry is one max-reduce over the lanes' head keys plus
// one min-reduce over the indices of the heads that tie with it.  Each lane
// caches its two best remaining slots and rescans its NPL slots only when a
// third one is taken.
QB_DEV uint32_t value_key(float v) { return f32_order_key(v == 0.0f ? 0.0f : v); }

template <int NPL>
struct WarpRanker {
    uint32_t removed = 0;   // slots already ranked
    uint32_t k0 = 0, k1 = 0;
    int c0 = 0, c1 = 0;
    bool have1 = false;

    QB_DEV void scan(const uint32_t (&key)[NPL]) {
        k0 = k1 = 0;
        c0 = c1 = 0;
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const uint32_t kc = ((removed >> c) & 1u) ? 0u : key[c];
            if (kc > k0) { k1 = k0; c1 = c0; k0 = kc; c0 = c; }
            else if (kc > k1) { k1 = kc; c1 = c; }
        }
        have1 = true;
    }
    // Key and index of the next-ranked entry, which leaves the ranking.
    QB_DEV void next(const uint32_t (&key)[NPL], int lane, uint32_t& K, int& j) {
        K = __reduce_max_sync(0xffffffffu, k0);
        const unsigned mine = (unsigned)(lane + 32 * c0);
        j = (int)__reduce_min_sync(0xffffffffu, k0 == K ? mine : 0xFFFFFFFFu);
        if ((unsigned)j == mine) {
            removed |= 1u << c0;
            if (have1) { k0 = k1; c0 = c1; have1 = false; }
            else scan(key);
        }
    }
    // Key of the next-ranked entry, left in the ranking.
    QB_DEV uint32_t peek() const { return __reduce_max_sync(0xffffffffu, k0); }
};

// Descending bitonic sort of one value per lane across the warp.
template <typename U>
QB_DEV U warp_sort_desc(U x, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const U o = __shfl_xor_sync(0xffffffffu, x, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
            x = keep_max ? (x > o ? x : o) : (x < o ? x : o);
        }
    }
    return x;
}

// (key desc, index asc) as one descending 64-bit order.
QB_DEV unsigned long long rank_word(uint32_t key, int j) {
    return ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)j;
}
QB_DEV uint32_t rank_word_key(unsigned long long w) { return (uint32_t)(w >> 32); }
QB_DEV int rank_word_index(unsigned long long w) { return (int)~(uint32_t)w; }

// Fast path of a token's ranking: the first `need` (<= 32) ranked entries,
// lane r ending with the r-th as a rank word.  The need-th largest of the 32
// lane maxima is a threshold that at least `need` values reach, so every
// ranked entry up to `need` is among the values at or above it; when those
// are at most 32 they are gathered one per lane (through buf, 32 words of
// this warp's shared memory) and sorted.  Returns false (warp-uniform) when
// more than 32 values reach the threshold; the caller then ranks by rounds.
template <int NPL>
QB_DEV bool warp_top_sorted(const uint32_t (&key)[NPL], int need, int lane, unsigned long long* buf,
                            unsigned long long& mine) {
    if (need > 32) return false;
    uint32_t mx = 0;
#pragma unroll
    for (int c = 0; c < NPL; ++c) mx = max(mx, key[c]);
    const uint32_t sorted_max = warp_sort_desc<uint32_t>(mx, lane);
    const uint32_t theta = __shfl_sync(0xffffffffu, sorted_max, need - 1);
    int cnt = 0;
#pragma unroll
    for (int c = 0; c < NPL; ++c) cnt += (key[c] != 0u && key[c] >= theta) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total > 32) return false;
    int pos = incl - cnt;
#pragma unroll
    for (int c = 0; c < NPL; ++c)
        if (key[c] != 0u && key[c] >= theta) buf[pos++] = rank_word(key[c], lane + 32 * c);
    __syncwarp();
    const unsigned long long w = lane < total ? buf[lane] : 0ull;
    __syncwarp();
    mine = warp_sort_desc<unsigned long long>(w, lane);
    return true;
}

// One token's ranking rounds (warp-uniform): V_k and V_{k+1} are the values of
// the k-th and (k+1)-th ranked experts; mask_k marks this lane's slots that
// are in the token's top k.
template <int NPL>
QB_DEV void rank_rounds(const uint32_t (&key)[NPL], int k, int lane, unsigned long long* buf, float& Vk, float& Vk1,
                        uint32_t& mask_k) {
    unsigned long long w;
    if (warp_top_sorted<NPL>(key, k + 1, lane, buf, w)) {
        const unsigned long long wk = __shfl_sync(0xffffffffu, w, k - 1);
        const unsigned long long wk1 = __shfl_sync(0xffffffffu, w, k);
        Vk = f32_from_order_key(rank_word_key(wk));
        Vk1 = f32_from_order_key(rank_word_key(wk1));
        mask_k = 0;
#pragma unroll
        for (int c = 0; c < NPL; ++c)
            if (key[c] != 0u && rank_word(key[c], lane + 32 * c) >= wk) mask_k |= 1u << c;
        return;
    }
    WarpRanker<NPL> rk;
    rk.scan(key);
    uint32_t K = 0;
    int j = 0;
    for (int r = 0; r < k; ++r) rk.next(key, lane, K, j);
    Vk = f32_from_order_key(K);
    Vk1 = f32_from_order_key(rk.peek());
    mask_k = rk.removed;
}

// Common offset of raw coordinate biases b' (one warp): the pairwise-tree sum
// of b' (zero-padded to a power of two P; each lane reduces P/32 contiguous
// leaves, then the lanes combine by halving strides) divided by n.
template <bool kFromL2 = false>
QB_DEV float common_offset_warp(const float* __restrict__ raw, int n, int lane) {
    int P = 1;
    while (P < n) P <<= 1;
    const int L = P >= 32 ? P / 32 : 1;     // leaves per lane
    const int A = P / L;                    // lanes holding a subtree
    float x = 0.0f;
    if (lane < A) {
        float a[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = lane * L + i;
            a[i] = (i < L && j < n) ? (kFromL2 ? __ldcg(raw + j) : raw[j]) : 0.0f;
        }
#pragma unroll
        for (int w = 32; w > 1; w >>= 1)
            if (w <= L)
#pragma unroll
                for (int i = 0; i < w / 2; ++i) a[i] = __fadd_rn(a[2 * i], a[2 * i + 1]);
        x = a[0];
    }
    for (int off = 1; off < A; off <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, x, off);
        if ((lane % (2 * off)) == 0) x = __fadd_rn(x, o);
    }
    return __fdiv_rn(__shfl_sync(0xffffffffu, x, 0), (float)n);
}

// Where a kernel takes the biases b from: b' - offset(b') when raw is set,
// else b (NULL = zeros).  Block 0 also stores the biases it used in out
// (may be NULL).
struct BiasArg {
    const float* b;
    const float* raw;
    float* out;
};

// Stage the n biases in shared memory (sb[QBMOE_MAX_EXPERTS]); ends with a
// block barrier.
QB_DEV void stage_bias(const BiasArg& ba, int n, float* sb) {
    __shared__ float s_off;
    if (ba.raw) {
        if (threadIdx.x < 32) {
            const float c = common_offset_warp(ba.raw, n, threadIdx.x);
            if (threadIdx.x == 0) s_off = c;
        }
        __syncthreads();
        const float c = s_off;
        for (int j = threadIdx.x; j < n; j += blockDim.x) sb[j] = __fsub_rn(ba.raw[j], c);
    } else {
        for (int j = threadIdx.x; j < n; j += blockDim.x) sb[j] = ba.b ? ba.b[j] : 0.0f;
    }
    __syncthreads();
    if (blockIdx.x == 0 && ba.out)
        for (int j = threadIdx.x; j < n; j += blockDim.x) ba.out[j] = sb[j];
}

// Token pass of a QB sweep: per token, tau_j (the k-th best biased score among
// the experts other than j) and the margin m_tj = s_tj - tau_j, written
// transposed [n, T] through a shared-memory tile.  With kFromLogits the
// scores are computed here from the router logits and stored.
template <int NPL, bool kFromLogits>
__global__ void __launch_bounds__(kTokPassWarps * 32, 4)
k_token_pass(int T, int n, int k, const float* __restrict__ logits, float* __restrict__ scores, BiasArg ba,
             float* __restrict__ margins, unsigned* __restrict__ ticket, int32_t* __restrict__ loads_zero) {
    extern __shared__ float tile[];   // [n][kTokPassTokens + 1]: scores, then margins
    __shared__ unsigned long long rank_buf[kTokPassWarps][32];
    __shared__ float sb[QBMOE_MAX_EXPERTS];
    static_assert(kTokPassTokens == kTokPassWarps, "one token per warp");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * kTokPassTokens;
    constexpr int LD = kTokPassTokens + 1;
    const int tl = warp;
    const int t = t0 + tl;
    pdl_wait();
    pdl_trigger();
    if (ticket && blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;   // for the select that follows
    if (loads_zero && blockIdx.x == 0)                                   // for the top-k's load counts
        for (int j = threadIdx.x; j < n; j += blockDim.x) loads_zero[j] = 0;
    // the token's row is requested before the biases are staged
    const float* src = kFromLogits ? logits + (size_t)t * n : scores + (size_t)t * n;
    float x[NPL];
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        x[c] = (t < T && j < n) ? src[j] : 0.0f;
    }
    stage_bias(ba, n, sb);
    if (t < T) {
        uint32_t key[NPL];
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int j = lane + 32 * c;
            key[c] = 0u;
            if (j < n) {
                const float sc = kFromLogits ? score_of_logit(x[c]) : x[c];
                if (kFromLogits) scores[(size_t)t * n + j] = sc;
                tile[j * LD + tl] = sc;   // kept for the margin below
                key[c] = value_key(__fadd_rn(sc, sb[j]));
            }
        }
        float Vk = 0.0f, Vk1 = 0.0f;
        uint32_t mask_k = 0;
        rank_rounds<NPL>(key, k, lane, rank_buf[warp], Vk, Vk1, mask_k);
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int j = lane + 32 * c;
            if (j < n) {
                const float tau = ((mask_k >> c) & 1u) ? Vk1 : Vk;
                float m = __fsub_rn(tile[j * LD + tl], tau);
                if (m == 0.0f) m = 0.0f;   // canonical +0
                tile[j * LD + tl] = m;
            }
        }
    }
    __syncthreads();
    // transposed write: each group of kTokPassTokens threads stores one
    // expert's consecutive tokens
    const int wl = threadIdx.x % kTokPassTokens;
    const int wt = t0 + wl;
    constexpr int kRowsPerPass = kTokPassWarps * 32 / kTokPassTokens;
    for (int j = threadIdx.x / kTokPassTokens; j < n; j += kRowsPerPass) {
        if (wt < T) margins[(size_t)j * T + wt] = tile[j * LD + wl];
    }
}

// Radix select of the rank-th largest margin of one expert's column: the
// rank-th smallest descending key (~order_key(margin), rank 1-based), in
// three digit passes of 12, 10 and 10 bits.  A 12-bit first digit (sign,
// exponent and three mantissa bits) splits QB margins finely: at 4096 tokens
// and 896 experts the bucket holding the target rank keeps a few dozen keys,
// where an 8-bit digit (sign and exponent only) often keeps the whole
// column.  With the column staged in shared memory, the keys of the first
// pass's chosen bucket are compacted (when they fit kSelectCand words) and
// the later passes run over them alone.
constexpr int kSelectMaxBits = 12;
struct SelectShared {
    unsigned hist[1 << kSelectMaxBits];
    unsigned wsum[kSelectThreads / 32];
    int digit, rank, cnt, ncand;
    uint32_t next;
    float red[kSelectThreads / 32];
};

// One digit pass over src[0..count) (keys matching prefix under mask): the
// BITS-wide digit at `shift` that holds rank; leaves the digit, the rank
// within it and the bucket's size in sh.  kFromCol: keys come from the
// margin column (and are stored to stage[] when stage is set), else from
// src[] in shared memory.
template <bool kFromCol, int BITS>
QB_DEV void radix_pass(const uint32_t* src, const float* col, uint32_t* stage, int count, uint32_t prefix,
                       uint32_t mask, int shift, int rank, SelectShared& sh) {
    constexpr int kBins = 1 << BITS;
    constexpr int kPer = kBins / kSelectThreads;   // bins per thread in the scan
    static_assert(kPer >= 1 && kBins % kSelectThreads == 0, "bins per thread");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kBins; i += kSelectThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < count; base += kSelectThreads) {
        const int i = base + tid;
        uint32_t key = 0;
        bool pred = false;
        if (i < count) {
            if (kFromCol) {
                key = ~f32_order_key(col[i]);
                if (stage) stage[i] = key;
            } else {
                key = src[i];
            }
            pred = (key & mask) == prefix;
        }
        const unsigned active = __ballot_sync(0xffffffffu, pred);
        if (pred) {
            const unsigned digit = (key >> shift) & (unsigned)(kBins - 1);
            const unsigned peers = __match_any_sync(active, digit);
            if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], (unsigned)__popc(peers));
        }
    }
    __syncthreads();
    // each thread scans kPer consecutive bins; warp and block prefixes on top
    unsigned c[kPer];
    unsigned tot = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        c[q] = sh.hist[tid * kPer + q];
        tot += c[q];
    }
    unsigned incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) sh.wsum[warp] = incl;
    __syncthreads();
    unsigned before = 0;
    for (int w = 0; w < warp; ++w) before += sh.wsum[w];
    unsigned excl = before + incl - tot;
    if ((int)excl < rank && rank <= (int)(excl + tot)) {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            if ((int)excl < rank && rank <= (int)(excl + c[q])) {
                sh.digit = tid * kPer + q;
                sh.rank = rank - (int)excl;
                sh.cnt = (int)c[q];
            }
            excl += c[q];
        }
    }
    __syncthreads();
}

// With kSmem the first pass also stages the keys in keys[0..T); returns the
// selected key and leaves in sh.ncand the number of compacted candidates at
// keys + T (0 when the later passes ran over all keys).
template <bool kSmem>
QB_DEV uint32_t radix_select(uint32_t* keys, uint32_t* cand, const float* col, int T, int rank,
                             SelectShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31;
    radix_pass<true, 12>(nullptr, col, kSmem ? keys : nullptr, T, 0u, 0u, 20, rank, sh);
    uint32_t prefix = (uint32_t)sh.digit << 20, mask = 0xFFF00000u;
    rank = sh.rank;
    const uint32_t* src = keys;
    int count = T;
    if (tid == 0) sh.ncand = 0;
    if (kSmem && sh.cnt <= kSelectCand && sh.cnt < T / 2) {
        __syncthreads();
        for (int base = 0; base < T; base += blockDim.x) {
            const int i = base + tid;
            const uint32_t key = i < T ? keys[i] : 0u;
            const bool pred = i < T && (key & mask) == prefix;
            const unsigned bal = __ballot_sync(0xffffffffu, pred);
            int wbase = 0;
            if (lane == 0 && bal) wbase = atomicAdd(&sh.ncand, __popc(bal));
            wbase = __shfl_sync(0xffffffffu, wbase, 0);
            if (pred) cand[wbase + __popc(bal & ((1u << lane) - 1u))] = key;
        }
        __syncthreads();
        src = cand;
        count = sh.ncand;
    }
    for (int shift = 10; shift >= 0; shift -= 10) {
        if (kSmem) radix_pass<false, 10>(src, col, nullptr, count, prefix, mask, shift, rank, sh);
        else radix_pass<true, 10>(nullptr, col, nullptr, count, prefix, mask, shift, rank, sh);
        prefix |= (uint32_t)sh.digit << shift;
        mask |= 0x3FFu << shift;
        rank = sh.rank;
        __syncthreads();
    }
    return prefix;
}

// Coordinate step of expert j (QB): with margins M (descending) and target
// load r, the bias is minus the midpoint of M_r and M_{r+1}; r = 0 and r >= T
// step just past the largest / smallest margin.
template <bool kSmem>
QB_DEV float coordinate_bias(int T, int r, const float* col, uint32_t* keys, SelectShared& sh) {
    const int tid = threadIdx.x;
    float q = 0.0f;
    if (r <= 0 || r >= T) {
        // max margin (r = 0) or min margin (r >= T)
        const bool want_max = r <= 0;
        float acc = want_max ? -INFINITY : INFINITY;
        for (int i = tid; i < T; i += blockDim.x) acc = want_max ? fmaxf(acc, col[i]) : fminf(acc, col[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, acc, off);
            acc = want_max ? fmaxf(acc, o) : fminf(acc, o);
        }
        if ((tid & 31) == 0) sh.red[tid >> 5] = acc;
        __syncthreads();
        if (tid == 0) {
            float a = sh.red[0];
            for (int w = 1; w < (int)(blockDim.x / 32); ++w) a = want_max ? fmaxf(a, sh.red[w]) : fminf(a, sh.red[w]);
            q = want_max ? __fadd_rn(a, 1.0f) : __fsub_rn(a, 1.0f);
        }
        return -q;
    }
    uint32_t* cand = keys + (kSmem ? T : 0);
    const uint32_t kr = radix_select<kSmem>(keys, cand, col, T, r, sh);
    // (r+1)-th largest: equal to the r-th when its final bucket holds another
    // copy, else the next larger descending key: the smallest candidate above
    // kr when the first digit's bucket holds one (every key outside it is
    // larger than all of them), else a min pass over all keys.
    uint32_t kr1 = kr;
    if (sh.cnt - sh.rank < 1) {
        const int nc = sh.ncand;
        for (int round = nc > 0 ? 0 : 1; round < 2; ++round) {
            const uint32_t* src = round == 0 ? cand : keys;
            const int count = round == 0 ? nc : T;
            uint32_t mn = 0xFFFFFFFFu;
            for (int i = tid; i < count; i += blockDim.x) {
                const uint32_t key = (kSmem || round == 0) ? src[i] : ~f32_order_key(col[i]);
                if (key > kr && key < mn) mn = key;
            }
            mn = __reduce_min_sync(0xffffffffu, mn);
            if (tid == 0) sh.next = 0xFFFFFFFFu;
            __syncthreads();
            if ((tid & 31) == 0) atomicMin(&sh.next, mn);
            __syncthreads();
            kr1 = sh.next;
            __syncthreads();
            if (kr1 != 0xFFFFFFFFu) break;
        }
    }
    if (tid == 0) {
        const float Mr = f32_from_order_key(~kr);
        const float Mr1 = f32_from_order_key(~kr1);
        q = __fmul_rn(__fadd_rn(Mr, Mr1), 0.5f);
    }
    return -q;
}

// Target load r_j: T*k routes split as evenly as possible, the first
// (T*k mod n) experts taking one more.
QB_DEV int target_load(int T, int n, int k, int j) {
    const long long total = (long long)T * k;
    return (int)(total / n) + (j < (int)(total % n) ? 1 : 0);
}

// Fast path of the coordinate step for 2 <= r <= T - 1 and T <= kSelectThreads
// * KPT: each thread holds KPT keys of the column in registers (all loads in
// flight at once), one 12-bit histogram pass locates the bins of ranks r and
// r + 1, and the keys of those bins (a few dozen on QB margins) are ranked
// exactly by counting.  Returns false (CTA-uniform) when the bins hold more
// than kRankCand keys; the caller then runs the general radix select.
constexpr int kRankCand = 256;

template <int KPT>
QB_DEV bool select_by_bins(int T, int r, const float* __restrict__ col, uint32_t* keys, uint32_t* cand,
                           SelectShared& sh, float& q_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kBins = 1 << 12;
    constexpr int kPer = kBins / kSelectThreads;
    for (int i = tid; i < kBins; i += kSelectThreads) sh.hist[i] = 0;
    if (tid == 0) sh.ncand = 0;
    {
        float m[KPT];   // every load of the column in flight at once
#pragma unroll
        for (int c = 0; c < KPT; ++c) {
            const int i = tid + kSelectThreads * c;
            m[c] = i < T ? col[i] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < KPT; ++c) {
            const int i = tid + kSelectThreads * c;
            if (i < T) {
                const uint32_t key = ~f32_order_key(m[c]);
                keys[i] = key;
                atomicAdd(&sh.hist[key >> 20], 1u);
            }
        }
    }
    __syncthreads();
    // bins of ranks r and r + 1 and the keys before the first of them
    unsigned cb[kPer];
    unsigned tot = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        cb[q] = sh.hist[tid * kPer + q];
        tot += cb[q];
    }
    unsigned incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) sh.wsum[warp] = incl;
    __syncthreads();
    unsigned excl = incl - tot;
    for (int w = 0; w < warp; ++w) excl += sh.wsum[w];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        if ((int)excl < r && r <= (int)(excl + cb[q])) {
            sh.digit = tid * kPer + q;   // bin of rank r
            sh.rank = (int)excl;         // keys before it
        }
        if ((int)excl < r + 1 && r + 1 <= (int)(excl + cb[q])) sh.cnt = tid * kPer + q;   // bin of rank r + 1
        excl += cb[q];
    }
    __syncthreads();
    const uint32_t bin_a = (uint32_t)sh.digit, bin_b = (uint32_t)sh.cnt;
    const int before = sh.rank;
    // gather the keys of bins [bin_a, bin_b]
#pragma unroll 4
    for (int c = 0; c < KPT; ++c) {
        const int i = tid + kSelectThreads * c;
        const uint32_t key = i < T ? keys[i] : 0xFFFFFFFFu;
        const uint32_t b = key >> 20;
        const bool pred = i < T && b >= bin_a && b <= bin_b;
        const unsigned bal = __ballot_sync(0xffffffffu, pred);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&sh.ncand, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (pred && pos < kRankCand) cand[pos] = key;
    }
    __syncthreads();
    const int nc = sh.ncand;
    if (nc > kRankCand) return false;
    // rank of each candidate among them: keys below and equal
    if (tid < nc) {
        const uint32_t me = cand[tid];
        int less = 0, eq = 0;
        for (int i = 0; i < nc; ++i) {
            const uint32_t o = cand[i];
            less += o < me ? 1 : 0;
            eq += o == me ? 1 : 0;
        }
        const int lo = before + less + 1, hi = before + less + eq;
        if (lo <= r && r <= hi) sh.next = me;            // key of rank r
        if (lo <= r + 1 && r + 1 <= hi) sh.wsum[0] = me;  // key of rank r + 1
    }
    __syncthreads();
    if (tid == 0) {
        const float Mr = f32_from_order_key(~sh.next);
        const float Mr1 = f32_from_order_key(~sh.wsum[0]);
        q_out = -__fmul_rn(__fadd_rn(Mr, Mr1), 0.5f);
    }
    return true;
}

// Thread 0 holds expert j's coordinate bias b': store it, and let the last
// CTA of the launch to finish (ticket) subtract the common offset from all n
// once, into fin, so that the kernels reading the biases next only copy them.
QB_DEV void publish_bias(int j, float b, int n, float* __restrict__ raw, float* __restrict__ fin,
                         unsigned* __restrict__ ticket) {
    __shared__ int s_last;
    __shared__ float s_off;
    if (threadIdx.x == 0) {
        raw[j] = b;
        __threadfence();
        s_last = atomicAdd(ticket, 1u) == (unsigned)(n - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < 32) {
        const float c = common_offset_warp<true>(raw, n, threadIdx.x);
        if (threadIdx.x == 0) s_off = c;
    }
    __syncthreads();
    for (int jj = threadIdx.x; jj < n; jj += blockDim.x) fin[jj] = __fsub_rn(__ldcg(raw + jj), s_off);
    if (threadIdx.x == 0) *ticket = 0u;
}

// One CTA per expert: the fast path when it applies, else the general
// radix select (coordinate_bias) over the column staged in shared memory.
template <int KPT>
__global__ void __launch_bounds__(kSelectThreads, KPT <= 16 ? 6 : 2)
k_expert_select_reg(int T, int n, int k, const float* __restrict__ margins, float* __restrict__ bias_raw,
                    float* __restrict__ bias_fin, unsigned* __restrict__ ticket) {
    extern __shared__ uint32_t keys[];   // [T] keys, then [min(T, kSelectCand)] candidates
    __shared__ SelectShared sh;
    const int j = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int r = target_load(T, n, k, j);
    const float* col = margins + (size_t)j * T;
    float b = 0.0f;
    if (!(r >= 1 && r <= T - 1 && select_by_bins<KPT>(T, r, col, keys, keys + T, sh, b))) {
        __syncthreads();
        b = coordinate_bias<true>(T, r, col, keys, sh);
    }
    publish_bias(j, b, n, bias_raw, bias_fin, ticket);
}

template <bool kSmem>
__global__ void __launch_bounds__(kSelectThreads)
k_expert_select(int T, int n, int k, const float* __restrict__ margins, float* __restrict__ bias_raw,
                float* __restrict__ bias_fin, unsigned* __restrict__ ticket) {
    extern __shared__ uint32_t keys[];   // [T] keys, then [min(T, kSelectCand)] candidates
    __shared__ SelectShared sh;
    const int j = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const float b = coordinate_bias<kSmem>(T, target_load(T, n, k, j), margins + (size_t)j * T, keys, sh);
    publish_bias(j, b, n, bias_raw, bias_fin, ticket);
}


template <int NPL>
__global__ void __launch_bounds__(kTopkWarps * 32, 3)
k_topk(int T, int n, int k, int tpw, const float* __restrict__ s, BiasArg ba, int32_t* __restrict__ idx,
       float* __restrict__ w, int* __restrict__ blk_cnt, int32_t* __restrict__ loads_acc, int early) {
    extern __shared__ int cnt[];   // [n]
    __shared__ unsigned long long rank_buf[kTopkWarps][32];
    __shared__ float sb[QBMOE_MAX_EXPERTS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j = threadIdx.x; j < n; j += blockDim.x) cnt[j] = 0;
    const int blk_tokens = kTopkWarps * tpw;
    const int t0 = blockIdx.x * blk_tokens + warp * tpw;
    // The first token's row is requested before the biases are staged.  With
    // `early` set the scores were written two kernels back (by the QB token
    // pass, which had finished before the preceding select kernel got past
    // its own dependency wait and let this one start), so the row is read
    // before this kernel's dependency wait.
    float x[NPL];
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        x[c] = (t0 < T && j < n) ? s[(size_t)t0 * n + j] : 0.0f;
    }
    if (early) {
        pdl_wait();
        pdl_trigger();
    }
    stage_bias(ba, n, sb);
    for (int q = 0; q < tpw; ++q) {
        const int t = t0 + q;
        if (t >= T) break;
        if (q > 0) {
#pragma unroll
            for (int c = 0; c < NPL; ++c) {
                const int j = lane + 32 * c;
                x[c] = j < n ? s[(size_t)t * n + j] : 0.0f;
            }
        }
        uint32_t key[NPL];
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int j = lane + 32 * c;
            key[c] = j < n ? value_key(__fadd_rn(x[c], sb[j])) : 0u;
        }
        int my_j = 0;
        unsigned long long wr;
        if (warp_top_sorted<NPL>(key, k, lane, rank_buf[warp], wr)) {
            my_j = rank_word_index(wr);
        } else {
            WarpRanker<NPL> rk;
            rk.scan(key);
            for (int r = 0; r < k; ++r) {
                uint32_t K;
                int wj;
                rk.next(key, lane, K, wj);
                if (lane == r) my_j = wj;
            }
        }
        // weights use the raw (unbiased) scores of the chosen experts
        const float my_s = lane < k ? s[(size_t)t * n + my_j] : 0.0f;
        float sum = 0.0f;
        for (int r = 0; r < k; ++r) {
            const float sr = __shfl_sync(0xffffffffu, my_s, r);
            sum = r == 0 ? sr : __fadd_rn(sum, sr);
        }
        if (lane < k) {
            idx[(size_t)t * k + lane] = my_j;
            w[(size_t)t * k + lane] = __fdiv_rn(my_s, sum);
            atomicAdd(&cnt[my_j], 1);
        }
    }
    __syncthreads();
    // expert-major [n, nblk]: expert j's counts of all blocks are contiguous
    if (blk_cnt)
        for (int j = threadIdx.x; j < n; j += blockDim.x) blk_cnt[(size_t)j * gridDim.x + blockIdx.x] = cnt[j];
    // or the loads themselves (integer sums: the same in any order)
    if (loads_acc)
        for (int j = threadIdx.x; j < n; j += blockDim.x)
            if (cnt[j]) atomicAdd(&loads_acc[j], cnt[j]);
}

// Per expert (one warp each): exclusive prefix over blocks of the expert's
// per-block counts (in place, expert-major [n, nblk]) and the expert's load.
// Each lane takes 8 consecutive blocks of a 256-block chunk, so a chunk's
// loads are issued together and coalesced.
__global__ void k_block_scan(int nblk, int n, int* __restrict__ blk_cnt, int32_t* __restrict__ loads) {
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (j >= n) return;
    int* row = blk_cnt + (size_t)j * nblk;
    int running = 0;
    for (int b0 = 0; b0 < nblk; b0 += 256) {
        const int first = b0 + lane * 8;
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = first + i < nblk ? row[first + i] : 0;
        int tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) tot += v[i];
        int incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int acc = running + incl - tot;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (first + i < nblk) row[first + i] = acc;
            acc += v[i];
        }
        running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0 && loads) loads[j] = running;
}

// ---------------------------------------------------------------------------
// Cyclic (Gauss-Seidel) QB sweep: experts updated one after another, each
// coordinate step seeing the latest biases.  Per token the top-(k+1) list of
// v = s + b is kept; expert j's step reads tau from it, and the next step
// refreshes only the lists that expert j's new bias can change (j in the
// list, or j's new value ranking before the list's last entry).

// Full top-(k1) list of one token (warp): lane r < k1 ends with the r-th
// ranked (value, index).
template <int NPL>
QB_DEV void top_list(const uint32_t (&key)[NPL], int k1, int lane, unsigned long long* buf, float& my_v,
                     int& my_j) {
    unsigned long long w;
    if (warp_top_sorted<NPL>(key, k1, lane, buf, w)) {
        if (lane < k1) { my_v = f32_from_order_key(rank_word_key(w)); my_j = rank_word_index(w); }
        return;
    }
    WarpRanker<NPL> rk;
    rk.scan(key);
    for (int r = 0; r < k1; ++r) {
        uint32_t K;
        int wj;
        rk.next(key, lane, K, wj);
        if (lane == r) { my_v = f32_from_order_key(K); my_j = wj; }
    }
}

template <int NPL>
QB_DEV void biased_row(const float* __restrict__ s_row, const float* __restrict__ b, int n, int lane,
                       uint32_t (&key)[NPL]) {
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        key[c] = j < n ? value_key(__fadd_rn(s_row[j], b[j])) : 0u;
    }
}

template <int NPL>
__global__ void __launch_bounds__(256)
k_gs_lists(int T, int n, int k, const float* __restrict__ s, const float* __restrict__ b, float* __restrict__ lv,
           int* __restrict__ li, const int* __restrict__ done) {
    __shared__ unsigned long long rank_buf[8][32];
    if (*done) return;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int K1 = k + 1;
    uint32_t key[NPL];
    biased_row<NPL>(s + (size_t)t * n, b, n, lane, key);
    float my_v = 0.0f;
    int my_j = 0;
    top_list<NPL>(key, K1, lane, rank_buf[threadIdx.x >> 5], my_v, my_j);
    if (lane < K1) {
        lv[(size_t)t * K1 + lane] = my_v;
        li[(size_t)t * K1 + lane] = my_j;
    }
}

template <int NPL>
__global__ void __launch_bounds__(256)
k_gs_token(int T, int n, int k, int j, int prev, const float* __restrict__ s, const float* __restrict__ b,
           float* __restrict__ lv, int* __restrict__ li, float* __restrict__ mj, const int* __restrict__ done) {
    __shared__ unsigned long long rank_buf[8][32];
    if (*done) return;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int K1 = k + 1;
    float ev = lane < K1 ? lv[(size_t)t * K1 + lane] : 0.0f;
    int ej = lane < K1 ? li[(size_t)t * K1 + lane] : -1;
    if (prev >= 0) {
        const float vn = __fadd_rn(s[(size_t)t * n + prev], b[prev]);
        const bool in_list = __any_sync(0xffffffffu, lane < K1 && ej == prev);
        const float lastv = __shfl_sync(0xffffffffu, ev, k);
        const int lastj = __shfl_sync(0xffffffffu, ej, k);
        if (in_list || ranks_before(vn, prev, lastv, lastj)) {
            uint32_t key[NPL];
            biased_row<NPL>(s + (size_t)t * n, b, n, lane, key);
            top_list<NPL>(key, K1, lane, rank_buf[threadIdx.x >> 5], ev, ej);
            if (lane < K1) {
                lv[(size_t)t * K1 + lane] = ev;
                li[(size_t)t * K1 + lane] = ej;
            }
        }
    }
    // tau: the k-th best biased score among the experts other than j
    const bool in_top = __any_sync(0xffffffffu, lane < k && ej == j);
    const float tau = __shfl_sync(0xffffffffu, ev, in_top ? k : k - 1);
    if (lane == 0) {
        float m = __fsub_rn(s[(size_t)t * n + j], tau);
        if (m == 0.0f) m = 0.0f;
        mj[t] = m;
    }
}

template <bool kSmem>
__global__ void __launch_bounds__(kSelectThreads)
k_gs_select(int T, int n, int k, int j, const float* __restrict__ mj, float* __restrict__ b,
            const int* __restrict__ done) {
    if (*done) return;
    extern __shared__ uint32_t keys[];   // [T] keys, then [min(T, kSelectCand)] candidates
    __shared__ SelectShared sh;
    const float bj = coordinate_bias<kSmem>(T, target_load(T, n, k, j), mj, keys, sh);
    if (threadIdx.x == 0) b[j] = bj;
}

// In-place common offset of a sweep (skipped once the loads are balanced).
__global__ void k_gs_offset(int n, float* __restrict__ b, const int* __restrict__ done) {
    if (*done) return;
    const int lane = threadIdx.x & 31;
    int P = 1;
    while (P < n) P <<= 1;
    const int L = P >= 32 ? P / 32 : 1;
    const int A = P / L;
    float a[32];
    float x = 0.0f;
    if (lane < A) {
        for (int i = 0; i < L; ++i) {
            const int jj = lane * L + i;
            a[i] = jj < n ? b[jj] : 0.0f;
        }
        for (int w = L; w > 1; w >>= 1)
            for (int i = 0; i < w / 2; ++i) a[i] = __fadd_rn(a[2 * i], a[2 * i + 1]);
        x = a[0];
    }
    for (int off = 1; off < A; off <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, x, off);
        if ((lane % (2 * off)) == 0) x = __fadd_rn(x, o);
    }
    const float c = __fdiv_rn(__shfl_sync(0xffffffffu, x, 0), (float)n);
    __syncwarp();
    for (int jj = lane; jj < n; jj += 32) b[jj] = __fsub_rn(b[jj], c);
}

// After a sweep: record the sweep count; stop further sweeps once every
// expert's load equals its target (when asked to).
__global__ void __launch_bounds__(1024)
k_gs_check(int T, int n, int k, const int32_t* __restrict__ loads, int* __restrict__ done,
           int32_t* __restrict__ sweeps_done, int sweep, int stop_when_balanced) {
    if (*done) return;
    const int j = threadIdx.x;
    const int bad = (j < n) && loads[j] != target_load(T, n, k, j);
    const int any_bad = __syncthreads_or(bad);
    if (j == 0) {
        if (sweeps_done) *sweeps_done = sweep + 1;
        if (stop_when_balanced && !any_bad) *done = 1;
    }
}

template <int NPL>
struct GsListsLaunch {
    static int run(int T, int n, int k, const float* s, const float* b, float* lv, int* li, const int* done,
                   cudaStream_t st) {
        k_gs_lists<NPL><<<(T + 7) / 8, 256, 0, st>>>(T, n, k, s, b, lv, li, done);
        return qbh::cuda_err(cudaGetLastError());
    }
};

template <int NPL>
struct GsTokenLaunch {
    static int run(int T, int n, int k, int j, int prev, const float* s, const float* b, float* lv, int* li,
                   float* mj, const int* done, cudaStream_t st) {
        k_gs_token<NPL><<<(T + 7) / 8, 256, 0, st>>>(T, n, k, j, prev, s, b, lv, li, mj, done);
        return qbh::cuda_err(cudaGetLastError());
    }
};

int npl_for(int n) {
    const int need = (n + 31) / 32;
    const int opts[] = {1, 2, 4, 8, 16, 28, 32};
    for (int o : opts)
        if (o >= need) return o;
    return -1;
}

template <template <int> class F, typename... Args>
int dispatch_npl(int npl, Args... args) {
    switch (npl) {
        case 1: return F<1>::run(args...);
        case 2: return F<2>::run(args...);
        case 4: return F<4>::run(args...);
        case 8: return F<8>::run(args...);
        case 16: return F<16>::run(args...);
        case 28: return F<28>::run(args...);
        case 32: return F<32>::run(args...);
        default: return QBMOE_EINVAL;
    }
}

// Kernel attributes are set once per device (route_init_attributes) to the
// largest size any call uses, never per call: a per-call set could lower the
// limit between another host thread's set and its launch.
template <int NPL>
struct TokenPassAttr {
    static int run() {
        const int smem = QBMOE_MAX_EXPERTS * (kTokPassTokens + 1) * (int)sizeof(float);
        for (auto kern : {k_token_pass<NPL, true>, k_token_pass<NPL, false>}) {
            // the largest shared-memory carveout lets several tiles share an SM
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                return QBMOE_ECUDA;
        }
        return QBMOE_OK;
    }
};

template <int NPL>
struct TokenPassLaunch {
    static int run(int T, int n, int k, const float* logits, float* scores, BiasArg ba, float* margins,
                   unsigned* ticket, int32_t* loads_zero, cudaStream_t st) {
        const size_t smem = (size_t)n * (kTokPassTokens + 1) * sizeof(float);
        auto kern = logits ? k_token_pass<NPL, true> : k_token_pass<NPL, false>;
        const int grid = (T + kTokPassTokens - 1) / kTokPassTokens;
        return qbh::launch_pdl(kern, dim3(grid), dim3(kTokPassWarps * 32), smem, st, T, n, k, logits, scores, ba,
                               margins, ticket, loads_zero);
    }
};

template <int NPL>
struct TopkLaunch {
    static int run(int T, int n, int k, int tpw, const float* s, BiasArg ba, int32_t* idx, float* w,
                   int* blk_cnt, int32_t* loads_acc, int early, cudaStream_t st) {
        const size_t smem = (size_t)n * sizeof(int);
        const int grid = (T + kTopkWarps * tpw - 1) / (kTopkWarps * tpw);
        return qbh::launch_pdl(k_topk<NPL>, dim3(grid), dim3(kTopkWarps * 32), smem, st, T, n, k, tpw, s, ba, idx, w,
                               blk_cnt, loads_acc, early);
    }
};

size_t select_smem_bytes(int T) { return (size_t)(T + std::min(T, kSelectCand)) * sizeof(uint32_t); }

int launch_select(int T, int n, int k, const float* margins, float* bias_raw, float* bias_fin, unsigned* ticket,
                  cudaStream_t st) {
    if (T <= 16 * kSelectThreads) {
        const size_t smem = select_smem_bytes(T);
        if (T <= 4 * kSelectThreads)
            return qbh::launch_pdl(k_expert_select_reg<4>, dim3(n), dim3(kSelectThreads), smem, st, T, n, k, margins,
                                   bias_raw, bias_fin, ticket);
        return qbh::launch_pdl(k_expert_select_reg<16>, dim3(n), dim3(kSelectThreads), smem, st, T, n, k, margins,
                               bias_raw, bias_fin, ticket);
    }
    if (T <= 64 * kSelectThreads) {
        const size_t smem = select_smem_bytes(T);
        return qbh::launch_pdl(k_expert_select_reg<64>, dim3(n), dim3(kSelectThreads), smem, st, T, n, k, margins,
                               bias_raw, bias_fin, ticket);
    }
    if (T <= kSelectSmemMaxT) {
        const size_t smem = select_smem_bytes(T);
        return qbh::launch_pdl(k_expert_select<true>, dim3(n), dim3(kSelectThreads), smem, st, T, n, k, margins,
                               bias_raw, bias_fin, ticket);
    }
    return qbh::launch_pdl(k_expert_select<false>, dim3(n), dim3(kSelectThreads), 0, st, T, n, k, margins, bias_raw,
                           bias_fin, ticket);
}

}  // namespace

namespace {

// ---------------------------------------------------------------------------
// DeepSeek-V3's fixed-step sign rule (the comparator of QB): every expert's
// bias moves by -gamma when its load exceeds its target and +gamma when it
// falls short ([K3-width] 延伸解读 "QB vs DeepSeek-V3": SignSGD on the dual
// that QB minimises exactly).
__global__ void k_sign_step(int T, int n, int k, const int32_t* __restrict__ loads, float gamma,
                            float* __restrict__ b) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const int r = target_load(T, n, k, j);
    const int l = loads[j];
    if (l > r) b[j] = __fsub_rn(b[j], gamma);
    else if (l < r) b[j] = __fadd_rn(b[j], gamma);
}

// ---------------------------------------------------------------------------
// Token-sharded QB: the r_j-th and (r_j+1)-th largest margins of every
// expert over a batch split into shards that exchange only per-expert digit
// histograms ([K3-width] Q&A on Quantile Balancing: histogram estimates keep
// the communication cheap).  Margins are compared through descending order
// keys (~f32_order_key); each of four passes fixes one 8-bit digit of both
// order statistics from the histogram of that digit among the keys that
// match the digits already fixed, summed over the shards.
struct HistSel {
    uint32_t prefix[2];   // digits fixed so far of the two tracked keys
    int rank[2];          // 1-based rank within the keys matching prefix
    int r;                // target load r_j
    int T;                // tokens of the whole batch
    int pad[2];
};
static_assert(sizeof(HistSel) == 32, "state layout");
constexpr int kHistBins = 256;
constexpr int kHistThreads = 256;
constexpr int kHistKeysPerThread = 8;

__global__ void k_hist_init(int T, int n, int k, HistSel* __restrict__ st, int* __restrict__ hist) {
    const long long total = (long long)n * 2 * kHistBins;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x)
        hist[i] = 0;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < n) {
        const int r = target_load(T, n, k, j);
        HistSel s;
        s.prefix[0] = s.prefix[1] = 0u;
        // r = 0: the largest margin (twice); r >= T: the smallest (twice)
        s.rank[0] = min(max(r, 1), T);
        s.rank[1] = (r >= 1 && r <= T - 1) ? r + 1 : s.rank[0];
        s.r = r;
        s.T = T;
        s.pad[0] = s.pad[1] = 0;
        st[j] = s;
    }
}

// One shard's histogram of pass `pass` added into hist [n][2][256]: CTA
// (chunk, expert), keys counted through warp-aggregated shared-memory atomics.
__global__ void __launch_bounds__(kHistThreads)
k_hist_count(int Ts, int pass, const float* __restrict__ margins, const HistSel* __restrict__ st,
             int* __restrict__ hist) {
    __shared__ unsigned h[2][kHistBins];
    const int j = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < 2 * kHistBins; i += blockDim.x) (&h[0][0])[i] = 0u;
    __syncthreads();
    const HistSel s = st[j];
    const int shift = 24 - 8 * pass;
    const uint32_t hi = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    const bool same = s.prefix[0] == s.prefix[1];
    const float* col = margins + (size_t)j * Ts;
    const int per_cta = kHistThreads * kHistKeysPerThread;
    const int end = min(Ts, (blockIdx.x + 1) * per_cta);
    for (int base = blockIdx.x * per_cta; base < end; base += kHistThreads) {
        const int i = base + tid;
        uint32_t key = 0u;
        if (i < end) key = ~f32_order_key(col[i]);
        const unsigned dg = (key >> shift) & 0xFFu;
        const bool pa = i < end && (key & hi) == s.prefix[0];
        const bool pb = i < end && !same && (key & hi) == s.prefix[1];
        const unsigned ma = __ballot_sync(0xffffffffu, pa);
        if (pa) {
            const unsigned peers = __match_any_sync(ma, dg);
            if (lane == __ffs(peers) - 1) atomicAdd(&h[0][dg], (unsigned)__popc(peers));
        }
        const unsigned mb = __ballot_sync(0xffffffffu, pb);
        if (pb) {
            const unsigned peers = __match_any_sync(mb, dg);
            if (lane == __ffs(peers) - 1) atomicAdd(&h[1][dg], (unsigned)__popc(peers));
        }
    }
    __syncthreads();
    int* out = hist + (size_t)j * 2 * kHistBins;
    for (int i = tid; i < kHistBins; i += blockDim.x) {
        const unsigned a = h[0][i];
        const unsigned b = same ? a : h[1][i];
        if (a) atomicAdd(out + i, (int)a);
        if (b) atomicAdd(out + kHistBins + i, (int)b);
    }
}

// After the exchange: fix pass `pass`'s digit of both tracked keys of every
// expert (one warp each) from the summed histogram, then clear it for the
// next pass.
__global__ void k_hist_advance(int n, int pass, int* __restrict__ hist, HistSel* __restrict__ st) {
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (j >= n) return;
    HistSel s = st[j];
    const int shift = 24 - 8 * pass;
    int* row = hist + (size_t)j * 2 * kHistBins;
    for (int a = 0; a < 2; ++a) {
        int v[8];
        int tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = row[a * kHistBins + lane * 8 + i];
            tot += v[i];
        }
        int incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const int rank = s.rank[a];
        int digit = -1, within = 0;
        int c = incl - tot;
        if (c < rank && rank <= incl) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (digit < 0 && c + v[i] >= rank) {
                    digit = lane * 8 + i;
                    within = rank - c;
                }
                c += v[i];
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, digit >= 0);
        const int src = m ? __ffs(m) - 1 : 0;
        digit = __shfl_sync(0xffffffffu, digit, src);
        within = __shfl_sync(0xffffffffu, within, src);
        if (m) {
            s.prefix[a] |= (uint32_t)digit << shift;
            s.rank[a] = within;
        }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 2 * kHistBins / 32; ++i) row[lane + 32 * i] = 0;
    if (lane == 0) st[j] = s;
}

// After the last pass: b'_j = -(midpoint of the two order statistics), or the
// end cases of the coordinate step, then the common offset (one CTA).
__global__ void __launch_bounds__(1024) k_hist_bias(int n, const HistSel* __restrict__ st, float* __restrict__ bias) {
    __shared__ float raw[QBMOE_MAX_EXPERTS];
    __shared__ float s_off;
    const int j = threadIdx.x;
    if (j < n) {
        const HistSel s = st[j];
        const float Ma = f32_from_order_key(~s.prefix[0]);
        const float Mb = f32_from_order_key(~s.prefix[1]);
        float q;
        if (s.r <= 0) q = __fadd_rn(Ma, 1.0f);
        else if (s.r >= s.T) q = __fsub_rn(Ma, 1.0f);
        else q = __fmul_rn(__fadd_rn(Ma, Mb), 0.5f);
        raw[j] = -q;
    }
    __syncthreads();
    if (j < 32) {
        const float c = common_offset_warp(raw, n, j);
        if (j == 0) s_off = c;
    }
    __syncthreads();
    if (j < n) bias[j] = __fsub_rn(raw[j], s_off);
}

}  // namespace

namespace qbh {

int route_tokens_per_warp(int T) {
    // about four 8-warp CTAs per SM before a warp takes a second token
    const int per = (T + kTopkWarps * 608 - 1) / (kTopkWarps * 608);
    return std::min(8, std::max(1, per));
}

size_t route_ws_layout(int T, int n, int k, RouteBuffers* rb, void* base) {
    (void)k;
    // Per-block count rows for any T' <= T: tokens_per_warp(T') is 1 while
    // T' <= 8*608 (then at most ceil(T'/8) blocks, never more than 608),
    // between 2 and 7 (at most 608 blocks), or 8 (ceil(T'/64) blocks).
    const int nblk = std::max(std::min((T + 7) / 8, 608), (T + 63) / 64);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_m = take((size_t)n * T * sizeof(float));
    const size_t o_raw = take((size_t)n * sizeof(float));
    const size_t o_fin = take((size_t)n * sizeof(float));
    const size_t o_tick = take(sizeof(unsigned));
    const size_t o_cnt = take((size_t)nblk * n * sizeof(int));
    if (rb && base) {
        char* p = static_cast<char*>(base);
        rb->margins = reinterpret_cast<float*>(p + o_m);
        rb->bias_raw = reinterpret_cast<float*>(p + o_raw);
        rb->bias_fin = reinterpret_cast<float*>(p + o_fin);
        rb->ticket = reinterpret_cast<unsigned*>(p + o_tick);
        rb->blk_cnt = reinterpret_cast<int*>(p + o_cnt);
    }
    return off;
}

int launch_scores(const float* logits, float* scores, long long count, cudaStream_t s, int* nl, int32_t* zero,
                  int nzero) {
    const int threads = 256;
    long long blocks = (count + threads - 1) / threads;
    blocks = std::min<long long>(blocks, 152LL * 16);
    k_scores<<<(int)std::max<long long>(blocks, 1), threads, 0, s>>>(logits, scores, count, zero, nzero);
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

// QB sweeps (if any) then the final top-k.  bias_in may be NULL (zeros).
// With logits set, the scores are computed from them first (inside the first
// token pass when there is a sweep).
int launch_qb_and_topk(int T, int n, int k, int sweeps, const float* logits, float* scores, const float* bias_in,
                       float* bias_out, int32_t* idx, float* w, int* blk_cnt, const RouteBuffers& rb,
                       cudaStream_t s, int* nl, int32_t* loads) {
    const int npl = npl_for(n);
    if (npl < 0) return QBMOE_EINVAL;
    int rc;
    if (logits && sweeps == 0 && (rc = launch_scores(logits, scores, (long long)T * n, s, nl, loads, n))) return rc;
    if (loads && sweeps == 0 && !logits && cudaMemsetAsync(loads, 0, (size_t)n * sizeof(int32_t), s) != cudaSuccess)
        return QBMOE_ECUDA;
    BiasArg ba{bias_in, nullptr, nullptr};
    for (int it = 0; it < sweeps; ++it) {
        rc = dispatch_npl<TokenPassLaunch>(npl, T, n, k, it == 0 ? logits : nullptr, scores, ba, rb.margins,
                                           rb.ticket, loads, s);
        if (rc) return rc;
        rc = launch_select(T, n, k, rb.margins, rb.bias_raw, rb.bias_fin, rb.ticket, s);
        if (rc) return rc;
        ba = BiasArg{rb.bias_fin, nullptr, nullptr};
        if (nl) *nl += 2;
    }
    ba.out = bias_out;
    const int tpw = route_tokens_per_warp(T);
    rc = dispatch_npl<TopkLaunch>(npl, T, n, k, tpw, scores, ba, idx, w, blk_cnt, loads, sweeps > 0 ? 1 : 0, s);
    if (nl) ++*nl;
    return rc;
}

int launch_loads_from_counts(int T, int n, int tpw, const int* blk_cnt, int32_t* loads, cudaStream_t s,
                             int* nl) {
    const int nblk = (T + kTopkWarps * tpw - 1) / (kTopkWarps * tpw);
    const int warps = 8;
    if (nl) ++*nl;
    return launch_pdl(k_block_scan, dim3((n + warps - 1) / warps), dim3(warps * 32), 0, s, nblk, n,
                      const_cast<int*>(blk_cnt), loads);
}

int route_init_attributes() {
    int rc;
    for (int npl : {1, 2, 4, 8, 16, 28, 32})
        if ((rc = dispatch_npl<TokenPassAttr>(npl))) return rc;
    const int sel = (int)select_smem_bytes(kSelectSmemMaxT);
    for (auto kern : {k_expert_select_reg<4>, k_expert_select_reg<16>, k_expert_select_reg<64>})
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)select_smem_bytes(64 * kSelectThreads)) != cudaSuccess)
            return QBMOE_ECUDA;
    if (cudaFuncSetAttribute(k_expert_select<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sel) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_gs_select<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sel) != cudaSuccess)
        return QBMOE_ECUDA;
    return QBMOE_OK;
}

}  // namespace qbh

// ---------------------------------------------------------------------------
// C ABI: moe_route_qb
// ---------------------------------------------------------------------------
static int g_route_launches = 0;

extern "C" size_t qbmoe_route_workspace_bytes(int T, int n, int k) {
    if (T < 1 || n < 2 || k < 1) return 0;
    return qbh::route_ws_layout(T, n, k, nullptr, nullptr);
}

extern "C" int qbmoe_route_last_launch_count(void) { return g_route_launches; }

extern "C" int moe_route_qb(int T, int n, int k, int qb_sweeps, const float* logits, const float* bias_in,
                            float* bias_out, float* scores, int32_t* topk_idx, float* topk_w, int32_t* loads,
                            void* workspace, size_t workspace_bytes, qbmoe_stream_t stream) {
    if (T < 1 || n < 2 || n > QBMOE_MAX_EXPERTS || k < 1 || k >= n || k > QBMOE_MAX_TOPK || qb_sweeps < 0)
        return QBMOE_EINVAL;
    if (!logits || !scores || !topk_idx || !topk_w || !loads || !workspace) return QBMOE_EINVAL;
    const void* ptrs[] = {logits, bias_in, bias_out, scores, topk_idx, topk_w, loads};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QBMOE_EINVAL;
    if (workspace_bytes < qbmoe_route_workspace_bytes(T, n, k)) return QBMOE_EWORKSPACE;
    int rc = qbh::device_init();
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qbh::RouteBuffers rb;
    qbh::route_ws_layout(T, n, k, &rb, workspace);
    int nl = 0;
    // the loads come from the top-k's per-CTA counts, added atomically (no
    // per-block prefix is needed without a dispatch)
    rc = qbh::launch_qb_and_topk(T, n, k, qb_sweeps, logits, scores, bias_in, bias_out, topk_idx, topk_w, nullptr,
                                 rb, s, &nl, loads);
    g_route_launches = nl;
    return rc;
}

// ---------------------------------------------------------------------------
// C ABI: moe_route_qb_gs (cyclic coordinate-descent QB)
// ---------------------------------------------------------------------------
namespace qbh {

size_t route_gs_ws_layout(int T, int n, int k, RouteBuffers* rb, GsBuffers* gb, void* base) {
    char* p = static_cast<char*>(base);
    size_t off = align_up(route_ws_layout(T, n, k, rb, base), 256);
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return p ? p + o : nullptr;
    };
    char* p_lv = take((size_t)T * (k + 1) * sizeof(float));
    char* p_li = take((size_t)T * (k + 1) * sizeof(int));
    char* p_mj = take((size_t)T * sizeof(float));
    char* p_b = take((size_t)n * sizeof(float));
    char* p_done = take(sizeof(int));
    if (gb && p) {
        gb->lv = reinterpret_cast<float*>(p_lv);
        gb->li = reinterpret_cast<int*>(p_li);
        gb->mj = reinterpret_cast<float*>(p_mj);
        gb->b = reinterpret_cast<float*>(p_b);
        gb->done = reinterpret_cast<int*>(p_done);
    }
    return off;
}

// Scores, max_sweeps cyclic sweeps (each followed by the loads under the new
// biases, for the sweep count and the balance test), then the final biased
// top-k; blk_cnt is left holding the final top-k's per-block counts (the
// caller turns them into loads).  `loads` is scratch for the balance test.
int launch_qb_gs(int T, int n, int k, int max_sweeps, int stop_when_balanced, const float* logits, float* scores,
                 const float* bias_in, float* bias_out, int32_t* topk_idx, float* topk_w, int32_t* loads,
                 int32_t* sweeps_done, const RouteBuffers& rb, const GsBuffers& gb, cudaStream_t s, int* nl) {
    const int npl = npl_for(n);
    if (npl < 0) return QBMOE_EINVAL;
    int rc;
    if ((rc = launch_scores(logits, scores, (long long)T * n, s, nl))) return rc;
    if (bias_in) {
        if (cudaMemcpyAsync(gb.b, bias_in, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return QBMOE_ECUDA;
    } else if (cudaMemsetAsync(gb.b, 0, (size_t)n * sizeof(float), s) != cudaSuccess) {
        return QBMOE_ECUDA;
    }
    if (cudaMemsetAsync(gb.done, 0, sizeof(int), s) != cudaSuccess) return QBMOE_ECUDA;
    if (sweeps_done && cudaMemsetAsync(sweeps_done, 0, sizeof(int32_t), s) != cudaSuccess) return QBMOE_ECUDA;
    const bool smem_sel = T <= kSelectSmemMaxT;
    const size_t sel_smem = smem_sel ? select_smem_bytes(T) : 0;
    const int tpw = route_tokens_per_warp(T);
    for (int sweep = 0; sweep < max_sweeps; ++sweep) {
        if ((rc = dispatch_npl<GsListsLaunch>(npl, T, n, k, (const float*)scores, (const float*)gb.b, gb.lv, gb.li,
                                              (const int*)gb.done, s)))
            return rc;
        for (int j = 0; j < n; ++j) {
            if ((rc = dispatch_npl<GsTokenLaunch>(npl, T, n, k, j, j - 1, (const float*)scores, (const float*)gb.b,
                                                  gb.lv, gb.li, gb.mj, (const int*)gb.done, s)))
                return rc;
            if (smem_sel) k_gs_select<true><<<1, kSelectThreads, sel_smem, s>>>(T, n, k, j, gb.mj, gb.b, gb.done);
            else k_gs_select<false><<<1, kSelectThreads, 0, s>>>(T, n, k, j, gb.mj, gb.b, gb.done);
            if ((rc = cuda_err(cudaGetLastError()))) return rc;
        }
        k_gs_offset<<<1, 32, 0, s>>>(n, gb.b, gb.done);
        if ((rc = cuda_err(cudaGetLastError()))) return rc;
        if (nl) *nl += 2 * n + 2;
        // loads under the new biases, for the sweep count and the balance test
        if ((rc = launch_qb_and_topk(T, n, k, 0, nullptr, scores, gb.b, nullptr, topk_idx, topk_w, rb.blk_cnt, rb, s,
                                     nl)))
            return rc;
        if ((rc = launch_loads_from_counts(T, n, tpw, rb.blk_cnt, loads, s, nl))) return rc;
        k_gs_check<<<1, 1024, 0, s>>>(T, n, k, loads, gb.done, sweeps_done, sweep, stop_when_balanced);
        if ((rc = cuda_err(cudaGetLastError()))) return rc;
        if (nl) ++*nl;
    }
    // final routing with the final biases
    return launch_qb_and_topk(T, n, k, 0, nullptr, scores, gb.b, bias_out, topk_idx, topk_w, rb.blk_cnt, rb, s, nl);
}

}  // namespace qbh

extern "C" size_t qbmoe_route_gs_workspace_bytes(int T, int n, int k) {
    if (T < 1 || n < 2 || k < 1) return 0;
    return qbh::route_gs_ws_layout(T, n, k, nullptr, nullptr, nullptr);
}

extern "C" int moe_route_qb_gs(int T, int n, int k, int max_sweeps, int stop_when_balanced, const float* logits,
                               const float* bias_in, float* bias_out, float* scores, int32_t* topk_idx,
                               float* topk_w, int32_t* loads, int32_t* sweeps_done, void* workspace,
                               size_t workspace_bytes, qbmoe_stream_t stream) {
    if (T < 1 || n < 2 || n > QBMOE_MAX_EXPERTS || k < 1 || k >= n || k > QBMOE_MAX_TOPK || max_sweeps < 0)
        return QBMOE_EINVAL;
    if (!logits || !scores || !topk_idx || !topk_w || !loads || !workspace) return QBMOE_EINVAL;
    const void* ptrs[] = {logits, bias_in, bias_out, scores, topk_idx, topk_w, loads, sweeps_done};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QBMOE_EINVAL;
    if (workspace_bytes < qbmoe_route_gs_workspace_bytes(T, n, k)) return QBMOE_EWORKSPACE;
    int rc = qbh::device_init();
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qbh::RouteBuffers rb;
    qbh::GsBuffers gb;
    qbh::route_gs_ws_layout(T, n, k, &rb, &gb, workspace);
    int nl = 0;
    rc = qbh::launch_qb_gs(T, n, k, max_sweeps, stop_when_balanced, logits, scores, bias_in, bias_out, topk_idx,
                           topk_w, loads, sweeps_done, rb, gb, s, &nl);
    if (!rc) rc = qbh::launch_loads_from_counts(T, n, qbh::route_tokens_per_warp(T), rb.blk_cnt, loads, s, &nl);
    g_route_launches = nl;
    return rc;
}

// ---------------------------------------------------------------------------
// C ABI: moe_route_signsgd (DeepSeek-V3's sign rule, the comparator of QB)
// ---------------------------------------------------------------------------
namespace {

size_t signsgd_ws_layout(int T, int n, int k, qbh::RouteBuffers* rb, float** b, void* base) {
    size_t off = qbh::align_up(qbh::route_ws_layout(T, n, k, rb, base), 256);
    if (b && base) *b = reinterpret_cast<float*>(static_cast<char*>(base) + off);
    return qbh::align_up(off + (size_t)n * sizeof(float), 256);
}

}  // namespace

extern "C" size_t qbmoe_route_signsgd_workspace_bytes(int T, int n, int k) {
    if (T < 1 || n < 2 || k < 1) return 0;
    return signsgd_ws_layout(T, n, k, nullptr, nullptr, nullptr);
}

extern "C" int moe_route_signsgd(int T, int n, int k, int steps, float gamma, const float* logits,
                                 const float* bias_in, float* bias_out, float* scores, int32_t* topk_idx,
                                 float* topk_w, int32_t* loads, void* workspace, size_t workspace_bytes,
                                 qbmoe_stream_t stream) {
    if (T < 1 || n < 2 || n > QBMOE_MAX_EXPERTS || k < 1 || k >= n || k > QBMOE_MAX_TOPK || steps < 0)
        return QBMOE_EINVAL;
    if (!(gamma > 0.0f) || !(gamma < INFINITY)) return QBMOE_EINVAL;
    if (!logits || !scores || !topk_idx || !topk_w || !loads || !workspace) return QBMOE_EINVAL;
    const void* ptrs[] = {logits, bias_in, bias_out, scores, topk_idx, topk_w, loads};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QBMOE_EINVAL;
    if (workspace_bytes < qbmoe_route_signsgd_workspace_bytes(T, n, k)) return QBMOE_EWORKSPACE;
    int rc = qbh::device_init();
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qbh::RouteBuffers rb;
    float* b = nullptr;
    signsgd_ws_layout(T, n, k, &rb, &b, workspace);
    int nl = 0;
    const int tpw = qbh::route_tokens_per_warp(T);
    if ((rc = qbh::launch_scores(logits, scores, (long long)T * n, s, &nl))) return rc;
    if (bias_in) {
        if (cudaMemcpyAsync(b, bias_in, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return QBMOE_ECUDA;
    } else if (cudaMemsetAsync(b, 0, (size_t)n * sizeof(float), s) != cudaSuccess) {
        return QBMOE_ECUDA;
    }
    for (int it = 0; it < steps; ++it) {
        // loads under the current biases, then one sign step
        if ((rc = qbh::launch_qb_and_topk(T, n, k, 0, nullptr, scores, b, nullptr, topk_idx, topk_w, rb.blk_cnt, rb,
                                          s, &nl)) ||
            (rc = qbh::launch_loads_from_counts(T, n, tpw, rb.blk_cnt, loads, s, &nl)))
            return rc;
        k_sign_step<<<(n + 255) / 256, 256, 0, s>>>(T, n, k, loads, gamma, b);
        if ((rc = qbh::cuda_err(cudaGetLastError()))) return rc;
        ++nl;
    }
    rc = qbh::launch_qb_and_topk(T, n, k, 0, nullptr, scores, b, bias_out, topk_idx, topk_w, rb.blk_cnt, rb, s, &nl);
    if (!rc) rc = qbh::launch_loads_from_counts(T, n, tpw, rb.blk_cnt, loads, s, &nl);
    g_route_launches = nl;
    return rc;
}

// ---------------------------------------------------------------------------
// C ABI: token-sharded QB with a histogram exchange
// ---------------------------------------------------------------------------
extern "C" size_t qbmoe_qb_hist_state_bytes(int n) {
    return n < 2 ? 0 : qbh::align_up((size_t)n * sizeof(HistSel), 256);
}

extern "C" size_t qbmoe_qb_hist_bytes(int n) { return n < 2 ? 0 : (size_t)n * 2 * kHistBins * sizeof(int); }

extern "C" size_t qbmoe_qb_shard_workspace_bytes(int T_shard, int n, int k) {
    if (T_shard < 1 || n < 2 || k < 1) return 0;
    return qbh::align_up((size_t)n * T_shard * sizeof(float), 256);
}

namespace {

int hist_common_checks(int n, const void* state, const void* hist) {
    if (n < 2 || n > QBMOE_MAX_EXPERTS || !state || !hist) return QBMOE_EINVAL;
    if (!qbh::aligned16(state) || !qbh::aligned16(hist)) return QBMOE_EINVAL;
    return qbh::device_init();
}

}  // namespace

extern "C" int moe_qb_hist_init(int T_total, int n, int k, void* state, int32_t* hist, qbmoe_stream_t stream) {
    if (T_total < 1 || k < 1 || k >= n || k > QBMOE_MAX_TOPK) return QBMOE_EINVAL;
    if ((long long)T_total * k >= (1LL << 31)) return QBMOE_EINVAL;
    int rc = hist_common_checks(n, state, hist);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    k_hist_init<<<(n * 2 * kHistBins + 255) / 256, 256, 0, s>>>(T_total, n, k, static_cast<HistSel*>(state), hist);
    return qbh::cuda_err(cudaGetLastError());
}

extern "C" int moe_qb_shard_margins(int T_shard, int n, int k, const float* logits, const float* bias_in,
                                    float* scores, void* workspace, size_t workspace_bytes, qbmoe_stream_t stream) {
    if (T_shard < 1 || n < 2 || n > QBMOE_MAX_EXPERTS || k < 1 || k >= n || k > QBMOE_MAX_TOPK) return QBMOE_EINVAL;
    if (!logits || !scores || !workspace) return QBMOE_EINVAL;
    const void* ptrs[] = {logits, bias_in, scores};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QBMOE_EINVAL;
    if (workspace_bytes < qbmoe_qb_shard_workspace_bytes(T_shard, n, k)) return QBMOE_EWORKSPACE;
    int rc = qbh::device_init();
    if (rc) return rc;
    const int npl = npl_for(n);
    if (npl < 0) return QBMOE_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dispatch_npl<TokenPassLaunch>(npl, T_shard, n, k, logits, scores, BiasArg{bias_in, nullptr, nullptr},
                                         static_cast<float*>(workspace), (unsigned*)nullptr, (int32_t*)nullptr, s);
}

extern "C" int moe_qb_shard_hist(int T_shard, int n, int pass, const void* state, const void* workspace,
                                 int32_t* hist, qbmoe_stream_t stream) {
    if (T_shard < 1 || pass < 0 || pass >= 4 || !workspace) return QBMOE_EINVAL;
    int rc = hist_common_checks(n, state, hist);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int per_cta = kHistThreads * kHistKeysPerThread;
    const dim3 grid((T_shard + per_cta - 1) / per_cta, n);
    k_hist_count<<<grid, kHistThreads, 0, s>>>(T_shard, pass, static_cast<const float*>(workspace),
                                               static_cast<const HistSel*>(state), hist);
    return qbh::cuda_err(cudaGetLastError());
}

extern "C" int moe_qb_hist_advance(int n, int pass, int32_t* hist, void* state, qbmoe_stream_t stream) {
    if (pass < 0 || pass >= 4) return QBMOE_EINVAL;
    int rc = hist_common_checks(n, state, hist);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    k_hist_advance<<<(n + 7) / 8, 256, 0, s>>>(n, pass, hist, static_cast<HistSel*>(state));
    return qbh::cuda_err(cudaGetLastError());
}

extern "C" int moe_qb_hist_bias(int n, const void* state, float* bias_out, qbmoe_stream_t stream) {
    if (!bias_out || !qbh::aligned16(bias_out)) return QBMOE_EINVAL;
    int rc = hist_common_checks(n, state, state);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    k_hist_bias<<<1, 1024, 0, s>>>(n, static_cast<const HistSel*>(state), bias_out);
    return qbh::cuda_err(cudaGetLastError());
}
