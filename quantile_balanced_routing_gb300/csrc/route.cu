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
// Kernels (one sweep = token pass + expert select + offset):
//   k_scores        s = score_of_logit(logit), elementwise
//   k_token_pass    per token: top-(k+1) of v = s + b by warp argmax rounds;
//                   margins m = s - tau written transposed [n, T] via SMEM
//   k_expert_select per expert: exact r-th and (r+1)-th largest margin by a
//                   4-pass 8-bit radix select with warp-aggregated SMEM
//                   histograms; b'_j = -midpoint
//   k_offset        b = b' - (pairwise-tree sum of b') / n   (one warp)
//   k_topk          per token: top-k of s + b, rank-order weights, per-block
//                   expert counts
//   k_block_scan    per expert: exclusive prefix of block counts, loads
#include "common.cuh"

#include <algorithm>
#include <climits>
#include <cstdio>

namespace {

using namespace qb;

constexpr int kTokPassTokens = 32;   // tokens per CTA in the token pass
constexpr int kTokPassWarps = 16;
constexpr int kTopkWarps = 8;
constexpr int kSelectThreads = 512;
constexpr int kSelectSmemMaxT = 50 * 1024;   // margins staged in SMEM up to this T

__global__ void k_scores(const float* __restrict__ logits, float* __restrict__ scores, long long count) {
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (; i < count; i += stride) scores[i] = score_of_logit(logits[i]);
}

// Warp-wide argmax under (value desc, index asc).
QB_DEV void warp_best(float& v, int& j) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oj = __shfl_xor_sync(0xffffffffu, j, off);
        if (ranks_before(ov, oj, v, j)) { v = ov; j = oj; }
    }
}

template <int NPL>
QB_DEV void lane_best(const float (&v)[NPL], uint32_t removed, int lane, float& bv, int& bj) {
    bv = -INFINITY;
    bj = INT_MAX;
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        if (!((removed >> c) & 1u) && ranks_before(v[c], j, bv, bj)) { bv = v[c]; bj = j; }
    }
}

// One token's ranking rounds (warp-uniform): V_k and V_{k+1} are the values of
// the k-th and (k+1)-th ranked experts; mask_k marks this lane's slots that
// are in the token's top k.
template <int NPL>
QB_DEV void rank_rounds(const float (&v)[NPL], int k, int lane, float& Vk, float& Vk1, uint32_t& mask_k) {
    uint32_t removed = 0;
    float bv;
    int bj;
    lane_best<NPL>(v, removed, lane, bv, bj);
    for (int r = 0; r <= k; ++r) {
        float wv = bv;
        int wj = bj;
        warp_best(wv, wj);
        if (r == k - 1) Vk = wv;
        if (r == k) { Vk1 = wv; break; }
        if ((wj & 31) == lane) {
            removed |= 1u << (wj >> 5);
            lane_best<NPL>(v, removed, lane, bv, bj);
        }
        if (r == k - 1) mask_k = removed;
    }
}

template <int NPL>
__global__ void __launch_bounds__(kTokPassWarps * 32)
k_token_pass(int T, int n, int k, const float* __restrict__ s, const float* __restrict__ b,
             float* __restrict__ margins) {
    extern __shared__ float tile[];   // [n][kTokPassTokens + 1]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * kTokPassTokens;
    constexpr int LD = kTokPassTokens + 1;
    float bj_[NPL];
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        bj_[c] = j < n ? b[j] : 0.0f;
    }
    for (int tl = warp; tl < kTokPassTokens; tl += kTokPassWarps) {
        const int t = t0 + tl;
        if (t >= T) break;
        float sv[NPL], v[NPL];
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int j = lane + 32 * c;
            sv[c] = j < n ? s[(size_t)t * n + j] : 0.0f;
            v[c] = j < n ? __fadd_rn(sv[c], bj_[c]) : -INFINITY;
        }
        float Vk = 0.0f, Vk1 = 0.0f;
        uint32_t mask_k = 0;
        rank_rounds<NPL>(v, k, lane, Vk, Vk1, mask_k);
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int j = lane + 32 * c;
            if (j < n) {
                const float tau = ((mask_k >> c) & 1u) ? Vk1 : Vk;
                float m = __fsub_rn(sv[c], tau);
                if (m == 0.0f) m = 0.0f;   // canonical +0
                tile[j * LD + tl] = m;
            }
        }
    }
    __syncthreads();
    const int tl = threadIdx.x & 31;
    const int t = t0 + tl;
    for (int j = threadIdx.x >> 5; j < n; j += kTokPassWarps) {
        if (t < T) margins[(size_t)j * T + t] = tile[j * LD + tl];
    }
}

// Radix select of the rank-th smallest descending key (rank 1-based) among
// keys[0..T).  Descending key = ~order_key(margin): the rank-th smallest
// descending key is the rank-th largest margin.
template <bool kSmem>
QB_DEV uint32_t radix_select(const uint32_t* keys_smem, const float* col, int T, int rank,
                             unsigned* hist, int* shared_digit, int* shared_rank) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0, mask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < T; base += blockDim.x) {
            const int i = base + tid;
            uint32_t key = 0;
            bool pred = false;
            if (i < T) {
                key = kSmem ? keys_smem[i] : ~f32_order_key(col[i]);
                pred = (key & mask) == prefix;
            }
            const unsigned active = __ballot_sync(0xffffffffu, pred);
            if (pred) {
                const unsigned digit = (key >> shift) & 0xFFu;
                const unsigned peers = __match_any_sync(active, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (unsigned)__popc(peers));
            }
        }
        __syncthreads();
        // inclusive scan of the 256 bins by warps 0..7 (one bin per thread)
        if (warp < 8) {
            const int bin = tid;
            const unsigned c = hist[bin];
            unsigned incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            // per-warp totals, combined across the 8 scanning warps
            __shared__ unsigned wsum[8];
            if (lane == 31) wsum[warp] = incl;
            __syncwarp();
            asm volatile("bar.sync 1, 256;");
            unsigned before = 0;
            for (int w = 0; w < warp; ++w) before += wsum[w];
            incl += before;
            const unsigned excl = incl - c;
            if ((int)excl < rank && rank <= (int)incl) {
                *shared_digit = bin;
                *shared_rank = rank - (int)excl;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)(*shared_digit) << shift;
        mask |= 0xFFu << shift;
        rank = *shared_rank;
        __syncthreads();
    }
    return prefix;
}

// Exact coordinate minimiser of one expert from its T margins `col` (keys
// staged in SMEM when kSmem): returns -q, q the midpoint of the r-th and
// (r+1)-th largest margins (r = 0: M_1 + 1; r >= T: M_T - 1).  Result valid
// in thread 0; every thread of the CTA must call it.
template <bool kSmem>
QB_DEV float coordinate_bias(int T, int r, const float* col, uint32_t* keys, unsigned* hist, int* s_digit,
                             int* s_rank, float* red) {
    const int tid = threadIdx.x;
    if (kSmem) {
        for (int i = tid; i < T; i += blockDim.x) keys[i] = ~f32_order_key(col[i]);
        __syncthreads();
    }
    float q = 0.0f;
    if (r <= 0 || r >= T) {
        // max margin (r = 0) or min margin (r >= T)
        const bool want_max = r <= 0;
        float acc = want_max ? -INFINITY : INFINITY;
        for (int i = tid; i < T; i += blockDim.x) {
            const float m = kSmem ? f32_from_order_key(~keys[i]) : col[i];
            acc = want_max ? fmaxf(acc, m) : fminf(acc, m);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, acc, off);
            acc = want_max ? fmaxf(acc, o) : fminf(acc, o);
        }
        if ((tid & 31) == 0) red[tid >> 5] = acc;
        __syncthreads();
        if (tid == 0) {
            float a = red[0];
            for (int w = 1; w < (int)(blockDim.x / 32); ++w) a = want_max ? fmaxf(a, red[w]) : fminf(a, red[w]);
            q = want_max ? __fadd_rn(a, 1.0f) : __fsub_rn(a, 1.0f);
        }
        return -q;
    }
    const uint32_t kr = radix_select<kSmem>(keys, col, T, r, hist, s_digit, s_rank);
    const uint32_t kr1 = radix_select<kSmem>(keys, col, T, r + 1, hist, s_digit, s_rank);
    if (tid == 0) {
        const float Mr = f32_from_order_key(~kr);
        const float Mr1 = f32_from_order_key(~kr1);
        q = __fmul_rn(__fadd_rn(Mr, Mr1), 0.5f);
    }
    return -q;
}

QB_DEV int target_load(int T, int n, int k, int j) {
    const long long total = (long long)T * k;
    return (int)(total / n) + (j < (int)(total % n) ? 1 : 0);
}

template <bool kSmem>
__global__ void __launch_bounds__(kSelectThreads)
k_expert_select(int T, int n, int k, const float* __restrict__ margins, float* __restrict__ bias_raw) {
    extern __shared__ uint32_t keys[];
    __shared__ unsigned hist[256];
    __shared__ int s_digit, s_rank;
    __shared__ float red[kSelectThreads / 32];
    const int j = blockIdx.x;
    const float b = coordinate_bias<kSmem>(T, target_load(T, n, k, j), margins + (size_t)j * T, keys, hist,
                                           &s_digit, &s_rank, red);
    if (threadIdx.x == 0) bias_raw[j] = b;
}

// b = fl(b' - c), c = fl(tree(b') / n); one warp.  Optionally also writes out2.
__global__ void k_offset(int n, const float* __restrict__ bias_raw, float* __restrict__ bias_cur,
                         float* __restrict__ out2) {
    const int lane = threadIdx.x & 31;
    int P = 1;
    while (P < n) P <<= 1;
    const int L = P >= 32 ? P / 32 : 1;     // leaves per lane
    const int A = P / L;                    // lanes holding a subtree
    float a[32];
    float x = 0.0f;
    if (lane < A) {
        for (int i = 0; i < L; ++i) {
            const int j = lane * L + i;
            a[i] = j < n ? bias_raw[j] : 0.0f;
        }
        for (int w = L; w > 1; w >>= 1)
            for (int i = 0; i < w / 2; ++i) a[i] = __fadd_rn(a[2 * i], a[2 * i + 1]);
        x = a[0];
    }
    for (int off = 1; off < A; off <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, x, off);
        if ((lane % (2 * off)) == 0) x = __fadd_rn(x, o);
    }
    const float sum = __shfl_sync(0xffffffffu, x, 0);
    const float c = __fdiv_rn(sum, (float)n);
    for (int j = lane; j < n; j += 32) {
        const float bj = __fsub_rn(bias_raw[j], c);
        bias_cur[j] = bj;
        if (out2) out2[j] = bj;
    }
}

template <int NPL>
__global__ void __launch_bounds__(kTopkWarps * 32)
k_topk(int T, int n, int k, int tpw, const float* __restrict__ s, const float* __restrict__ b,
       int32_t* __restrict__ idx, float* __restrict__ w, int* __restrict__ blk_cnt) {
    extern __shared__ int cnt[];   // [n]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j = threadIdx.x; j < n; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    float bj_[NPL];
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        bj_[c] = j < n ? b[j] : 0.0f;
    }
    const int blk_tokens = kTopkWarps * tpw;
    const int t0 = blockIdx.x * blk_tokens + warp * tpw;
    for (int q = 0; q < tpw; ++q) {
        const int t = t0 + q;
        if (t >= T) break;
        float sv[NPL], v[NPL];
#pragma unroll
        for (int c = 0; c < NPL; ++c) {
            const int j = lane + 32 * c;
            sv[c] = j < n ? s[(size_t)t * n + j] : 0.0f;
            v[c] = j < n ? __fadd_rn(sv[c], bj_[c]) : -INFINITY;
        }
        uint32_t removed = 0;
        float bv;
        int bjx;
        lane_best<NPL>(v, removed, lane, bv, bjx);
        int my_j = 0;
        float my_s = 0.0f;
        for (int r = 0; r < k; ++r) {
            float wv = bv;
            int wj = bjx;
            warp_best(wv, wj);
            const int owner = wj & 31;
            float ws = 0.0f;
            if (owner == lane) {
#pragma unroll
                for (int c = 0; c < NPL; ++c)
                    if (c == (wj >> 5)) ws = sv[c];
                removed |= 1u << (wj >> 5);
                lane_best<NPL>(v, removed, lane, bv, bjx);
            }
            ws = __shfl_sync(0xffffffffu, ws, owner);
            if (lane == r) { my_j = wj; my_s = ws; }
        }
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
    for (int j = threadIdx.x; j < n; j += blockDim.x) blk_cnt[(size_t)blockIdx.x * n + j] = cnt[j];
}

// Per expert (one warp each): exclusive prefix of per-block counts (in place)
// and the expert's load.
__global__ void k_block_scan(int nblk, int n, int* __restrict__ blk_cnt, int32_t* __restrict__ loads) {
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (j >= n) return;
    int running = 0;
    for (int b0 = 0; b0 < nblk; b0 += 32) {
        const int bb = b0 + lane;
        const int v = bb < nblk ? blk_cnt[(size_t)bb * n + j] : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (bb < nblk) blk_cnt[(size_t)bb * n + j] = running + incl - v;
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
QB_DEV void top_list(const float (&v)[NPL], int k1, int lane, float& my_v, int& my_j) {
    uint32_t removed = 0;
    float bv;
    int bj;
    lane_best<NPL>(v, removed, lane, bv, bj);
    for (int r = 0; r < k1; ++r) {
        float wv = bv;
        int wj = bj;
        warp_best(wv, wj);
        if (lane == r) { my_v = wv; my_j = wj; }
        if ((wj & 31) == lane) {
            removed |= 1u << (wj >> 5);
            lane_best<NPL>(v, removed, lane, bv, bj);
        }
    }
}

template <int NPL>
QB_DEV void biased_row(const float* __restrict__ s_row, const float* __restrict__ b, int n, int lane, float (&v)[NPL]) {
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int j = lane + 32 * c;
        v[c] = j < n ? __fadd_rn(s_row[j], b[j]) : -INFINITY;
    }
}

template <int NPL>
__global__ void __launch_bounds__(256)
k_gs_lists(int T, int n, int k, const float* __restrict__ s, const float* __restrict__ b, float* __restrict__ lv,
           int* __restrict__ li, const int* __restrict__ done) {
    if (*done) return;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int K1 = k + 1;
    float v[NPL];
    biased_row<NPL>(s + (size_t)t * n, b, n, lane, v);
    float my_v = 0.0f;
    int my_j = 0;
    top_list<NPL>(v, K1, lane, my_v, my_j);
    if (lane < K1) {
        lv[(size_t)t * K1 + lane] = my_v;
        li[(size_t)t * K1 + lane] = my_j;
    }
}

template <int NPL>
__global__ void __launch_bounds__(256)
k_gs_token(int T, int n, int k, int j, int prev, const float* __restrict__ s, const float* __restrict__ b,
           float* __restrict__ lv, int* __restrict__ li, float* __restrict__ mj, const int* __restrict__ done) {
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
            float v[NPL];
            biased_row<NPL>(s + (size_t)t * n, b, n, lane, v);
            top_list<NPL>(v, K1, lane, ev, ej);
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
    extern __shared__ uint32_t keys[];
    __shared__ unsigned hist[256];
    __shared__ int s_digit, s_rank;
    __shared__ float red[kSelectThreads / 32];
    const float bj = coordinate_bias<kSmem>(T, target_load(T, n, k, j), mj, keys, hist, &s_digit, &s_rank, red);
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

template <int NPL>
struct TokenPassLaunch {
    static int run(int T, int n, int k, const float* s, const float* b, float* margins, cudaStream_t st) {
        const size_t smem = (size_t)n * (kTokPassTokens + 1) * sizeof(float);
        auto kern = k_token_pass<NPL>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QBMOE_ECUDA;
        const int grid = (T + kTokPassTokens - 1) / kTokPassTokens;
        kern<<<grid, kTokPassWarps * 32, smem, st>>>(T, n, k, s, b, margins);
        return qbh::cuda_err(cudaGetLastError());
    }
};

template <int NPL>
struct TopkLaunch {
    static int run(int T, int n, int k, int tpw, const float* s, const float* b, int32_t* idx, float* w,
                   int* blk_cnt, cudaStream_t st) {
        const size_t smem = (size_t)n * sizeof(int);
        const int grid = (T + kTopkWarps * tpw - 1) / (kTopkWarps * tpw);
        k_topk<NPL><<<grid, kTopkWarps * 32, smem, st>>>(T, n, k, tpw, s, b, idx, w, blk_cnt);
        return qbh::cuda_err(cudaGetLastError());
    }
};

int launch_select(int T, int n, int k, const float* margins, float* bias_raw, cudaStream_t st) {
    if (T <= kSelectSmemMaxT) {
        const size_t smem = (size_t)T * sizeof(uint32_t);
        if (cudaFuncSetAttribute(k_expert_select<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)std::max<size_t>(smem, 1)) != cudaSuccess)
            return QBMOE_ECUDA;
        k_expert_select<true><<<n, kSelectThreads, smem, st>>>(T, n, k, margins, bias_raw);
    } else {
        k_expert_select<false><<<n, kSelectThreads, 0, st>>>(T, n, k, margins, bias_raw);
    }
    return qbh::cuda_err(cudaGetLastError());
}

}  // namespace

namespace qbh {

int route_tokens_per_warp(int T) {
    const int per = (T + kTopkWarps * 304 - 1) / (kTopkWarps * 304);
    return std::min(8, std::max(1, per));
}

size_t route_ws_layout(int T, int n, int k, RouteBuffers* rb, void* base) {
    (void)k;
    // Per-block count rows for any T' <= T: tokens_per_warp(T') is 1 while
    // T' <= 8*304 (then at most ceil(T'/8) blocks, never more than 304),
    // between 2 and 7 (at most 304 blocks), or 8 (ceil(T'/64) blocks).
    const int nblk = std::max(std::min((T + 7) / 8, 304), (T + 63) / 64);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_m = take((size_t)n * T * sizeof(float));
    const size_t o_raw = take((size_t)n * sizeof(float));
    const size_t o_cur = take((size_t)n * sizeof(float));
    const size_t o_cnt = take((size_t)nblk * n * sizeof(int));
    if (rb && base) {
        char* p = static_cast<char*>(base);
        rb->margins = reinterpret_cast<float*>(p + o_m);
        rb->bias_raw = reinterpret_cast<float*>(p + o_raw);
        rb->bias_cur = reinterpret_cast<float*>(p + o_cur);
        rb->blk_cnt = reinterpret_cast<int*>(p + o_cnt);
    }
    return off;
}

int launch_scores(const float* logits, float* scores, long long count, cudaStream_t s, int* nl) {
    const int threads = 256;
    long long blocks = (count + threads - 1) / threads;
    blocks = std::min<long long>(blocks, 152LL * 16);
    k_scores<<<(int)std::max<long long>(blocks, 1), threads, 0, s>>>(logits, scores, count);
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

// QB sweeps (if any) then the final top-k.  bias_in may be NULL (zeros).
int launch_qb_and_topk(int T, int n, int k, int sweeps, const float* scores, const float* bias_in,
                       float* bias_out, int32_t* idx, float* w, int* blk_cnt, const RouteBuffers& rb,
                       cudaStream_t s, int* nl) {
    const int npl = npl_for(n);
    if (npl < 0) return QBMOE_EINVAL;
    const float* b = bias_in;
    if (!b) {
        if (cudaMemsetAsync(rb.bias_cur, 0, (size_t)n * sizeof(float), s) != cudaSuccess) return QBMOE_ECUDA;
        b = rb.bias_cur;
    }
    int rc;
    for (int it = 0; it < sweeps; ++it) {
        rc = dispatch_npl<TokenPassLaunch>(npl, T, n, k, scores, b, rb.margins, s);
        if (rc) return rc;
        rc = launch_select(T, n, k, rb.margins, rb.bias_raw, s);
        if (rc) return rc;
        const bool last = it == sweeps - 1;
        k_offset<<<1, 32, 0, s>>>(n, rb.bias_raw, rb.bias_cur, last ? bias_out : nullptr);
        if ((rc = cuda_err(cudaGetLastError()))) return rc;
        b = rb.bias_cur;
        if (nl) *nl += 3;
    }
    if (sweeps == 0 && bias_out && bias_out != b) {
        if (cudaMemcpyAsync(bias_out, b, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return QBMOE_ECUDA;
    }
    const int tpw = route_tokens_per_warp(T);
    rc = dispatch_npl<TopkLaunch>(npl, T, n, k, tpw, scores, b, idx, w, blk_cnt, s);
    if (nl) ++*nl;
    return rc;
}

int launch_loads_from_counts(int T, int n, int tpw, const int* blk_cnt, int32_t* loads, cudaStream_t s,
                             int* nl) {
    const int nblk = (T + kTopkWarps * tpw - 1) / (kTopkWarps * tpw);
    const int warps = 8;
    k_block_scan<<<(n + warps - 1) / warps, warps * 32, 0, s>>>(nblk, n, const_cast<int*>(blk_cnt), loads);
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
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

int qbmoe_check_device_arch();   // api.cu

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
    int rc = qbmoe_check_device_arch();
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qbh::RouteBuffers rb;
    qbh::route_ws_layout(T, n, k, &rb, workspace);
    int nl = 0;
    rc = qbh::launch_scores(logits, scores, (long long)T * n, s, &nl);
    if (!rc) rc = qbh::launch_qb_and_topk(T, n, k, qb_sweeps, scores, bias_in, bias_out, topk_idx, topk_w,
                                          rb.blk_cnt, rb, s, &nl);
    if (!rc) rc = qbh::launch_loads_from_counts(T, n, qbh::route_tokens_per_warp(T), rb.blk_cnt, loads, s, &nl);
    g_route_launches = nl;
    return rc;
}

// ---------------------------------------------------------------------------
// C ABI: moe_route_qb_gs (cyclic coordinate-descent QB)
// ---------------------------------------------------------------------------
namespace {

struct GsBuffers {
    float* lv;     // [T, k+1] top-(k+1) values per token
    int* li;       // [T, k+1] their experts
    float* mj;     // [T] margins of the expert being updated
    float* b;      // [n] current biases
    int* done;     // balanced flag
};

size_t gs_ws_layout(int T, int n, int k, qbh::RouteBuffers* rb, GsBuffers* gb, void* base) {
    char* p = static_cast<char*>(base);
    size_t off = qbh::align_up(qbh::route_ws_layout(T, n, k, rb, base), 256);
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = qbh::align_up(off + bytes, 256);
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

}  // namespace

extern "C" size_t qbmoe_route_gs_workspace_bytes(int T, int n, int k) {
    if (T < 1 || n < 2 || k < 1) return 0;
    return gs_ws_layout(T, n, k, nullptr, nullptr, nullptr);
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
    int rc = qbmoe_check_device_arch();
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qbh::RouteBuffers rb;
    GsBuffers gb;
    gs_ws_layout(T, n, k, &rb, &gb, workspace);
    const int npl = npl_for(n);
    if (npl < 0) return QBMOE_EINVAL;
    int nl = 0;
    if ((rc = qbh::launch_scores(logits, scores, (long long)T * n, s, &nl))) return rc;
    if (bias_in) {
        if (cudaMemcpyAsync(gb.b, bias_in, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return QBMOE_ECUDA;
    } else if (cudaMemsetAsync(gb.b, 0, (size_t)n * sizeof(float), s) != cudaSuccess) {
        return QBMOE_ECUDA;
    }
    if (cudaMemsetAsync(gb.done, 0, sizeof(int), s) != cudaSuccess) return QBMOE_ECUDA;
    if (sweeps_done && cudaMemsetAsync(sweeps_done, 0, sizeof(int32_t), s) != cudaSuccess) return QBMOE_ECUDA;
    const bool smem_sel = T <= kSelectSmemMaxT;
    const size_t sel_smem = smem_sel ? (size_t)T * sizeof(uint32_t) : 0;
    if (smem_sel && cudaFuncSetAttribute(k_gs_select<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)std::max<size_t>(sel_smem, 1)) != cudaSuccess)
        return QBMOE_ECUDA;
    const int tpw = qbh::route_tokens_per_warp(T);
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
            if ((rc = qbh::cuda_err(cudaGetLastError()))) return rc;
        }
        k_gs_offset<<<1, 32, 0, s>>>(n, gb.b, gb.done);
        if ((rc = qbh::cuda_err(cudaGetLastError()))) return rc;
        // loads under the new biases, for the sweep count and the balance test
        if ((rc = qbh::launch_qb_and_topk(T, n, k, 0, scores, gb.b, nullptr, topk_idx, topk_w, rb.blk_cnt, rb, s,
                                          &nl)))
            return rc;
        if ((rc = qbh::launch_loads_from_counts(T, n, tpw, rb.blk_cnt, loads, s, &nl))) return rc;
        k_gs_check<<<1, 1024, 0, s>>>(T, n, k, loads, gb.done, sweeps_done, sweep, stop_when_balanced);
        if ((rc = qbh::cuda_err(cudaGetLastError()))) return rc;
    }
    // final routing with the final biases
    rc = qbh::launch_qb_and_topk(T, n, k, 0, scores, gb.b, bias_out, topk_idx, topk_w, rb.blk_cnt, rb, s, &nl);
    if (!rc) rc = qbh::launch_loads_from_counts(T, n, tpw, rb.blk_cnt, loads, s, &nl);
    return rc;
}
