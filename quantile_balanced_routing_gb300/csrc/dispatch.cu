// Token dispatch (expert offsets, stable permutation) and the fused
// combine + RMSNorm of the routed branch.
//
// [K3-width] = "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club).
//   Q&A on RMSNorm: RMSNorm sits after the latent aggregation of the k expert
//   outputs and before the up-projection.
#include "common.cuh"
#include "dispatch.cuh"

#include <algorithm>

namespace {

using namespace qb;

// One CTA (<= 1024 threads, one per expert): offsets = exclusive scan of
// loads; tile_off = exclusive scan of ceil(load / tile_rows).
__global__ void __launch_bounds__(1024)
k_expert_offsets(int n, const int32_t* __restrict__ loads, int* __restrict__ offsets,
                 int tile_rows, int* __restrict__ tile_off) {
    __shared__ int wsum[2][32];
    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const int v = j < n ? loads[j] : 0;
    const int tv = j < n ? (v + tile_rows - 1) / tile_rows : 0;
    int a = v, b = tv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int oa = __shfl_up_sync(0xffffffffu, a, off);
        const int ob = __shfl_up_sync(0xffffffffu, b, off);
        if (lane >= off) { a += oa; b += ob; }
    }
    if (lane == 31) { wsum[0][warp] = a; wsum[1][warp] = b; }
    __syncthreads();
    int pa = 0, pb = 0;
    for (int w = 0; w < warp; ++w) { pa += wsum[0][w]; pb += wsum[1][w]; }
    a += pa;
    b += pb;
    if (j < n) {
        offsets[j] = a - v;
        tile_off[j] = b - tv;
    }
    if (j == n - 1) {
        offsets[n] = a;
        tile_off[n] = b;
    }
}

// Stable scatter: route (t, i) of expert e goes to
//   pos = offsets[e] + blk_base[e][blk] + #(tokens of this block before t routed to e).
// One thread per token of the block (block = 8 * tpw <= 64 tokens).
__global__ void k_scatter(int T, int n, int k, int tpw, const int32_t* __restrict__ idx,
                          const int* __restrict__ blk_base, const int* __restrict__ offsets,
                          int* __restrict__ perm, int* __restrict__ route_pos) {
    extern __shared__ unsigned long long masks[];   // [n]
    const int blk_tokens = 8 * tpw;
    const int tl = threadIdx.x;
    const int t = blockIdx.x * blk_tokens + tl;
    for (int j = tl; j < n; j += blockDim.x) masks[j] = 0ull;
    __syncthreads();
    if (t < T)
        for (int i = 0; i < k; ++i) atomicOr(&masks[idx[(size_t)t * k + i]], 1ull << tl);
    __syncthreads();
    if (t >= T) return;
    const unsigned long long below = (tl == 0) ? 0ull : ((1ull << tl) - 1ull);
    for (int i = 0; i < k; ++i) {
        const int e = idx[(size_t)t * k + i];
        const int pos = offsets[e] + blk_base[(size_t)e * gridDim.x + blockIdx.x] + __popcll(masks[e] & below);
        perm[pos] = t;
        route_pos[(size_t)t * k + i] = pos;
    }
}

// Row copy in token order: dst[route_pos[t * k + i]] = src[t] for each of
// token t's k routes (16-byte vectors).  Each source row is read once and
// written k times; walking the destination rows instead re-reads every source
// row k times, from DRAM once the rows have left L2.
__global__ void k_scatter_rows(const uint4* __restrict__ src, int vec_per_row, const int* __restrict__ route_pos,
                               int T, int k, uint4* __restrict__ dst) {
    const long long total = (long long)T * vec_per_row;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long t = i / vec_per_row;
        const int c = (int)(i - t * vec_per_row);
        const uint4 v = src[i];
        const int* rp = route_pos + t * k;
        for (int r = 0; r < k; ++r) dst[(long long)__ldg(rp + r) * vec_per_row + c] = v;
    }
}

// y = sum_i w[t,i] * e[route_pos[t,i]] (fp32); z = y / sqrt(mean(y^2) + eps) * gamma.
// One CTA per token; each thread owns VPT 16-byte vectors of the row and
// reads its k expert rows eight at a time, so that many loads are in flight
// (the kernel streams the T*k expert rows once).
constexpr int kCombMaxThreads = 1024;
constexpr int kCombUnroll = 8;

template <typename TA, int VPT>
__global__ void __launch_bounds__(kCombMaxThreads)
k_combine_rmsnorm(int T, int k, int latent, const TA* __restrict__ e, const float* __restrict__ w,
                  const int* __restrict__ route_pos, const float* __restrict__ gamma, float eps,
                  TA* __restrict__ z, long long ldz) {
    constexpr int V = 16 / sizeof(TA);             // elements per vector
    __shared__ float s_w[QBMOE_MAX_TOPK];
    __shared__ int s_pos[QBMOE_MAX_TOPK];
    __shared__ float red[kCombMaxThreads / 32];
    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const int nvec = latent / V;
    if (tid < k) {
        s_w[tid] = w[(size_t)t * k + tid];
        s_pos[tid] = route_pos[(size_t)t * k + tid];
    }
    __syncthreads();
    float y[VPT][V];
#pragma unroll
    for (int q = 0; q < VPT; ++q)
#pragma unroll
        for (int u = 0; u < V; ++u) y[q][u] = 0.0f;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
        const int c = tid + q * blockDim.x;
        if (c >= nvec) break;
        for (int i0 = 0; i0 < k; i0 += kCombUnroll) {
            uint4 raw[kCombUnroll];
#pragma unroll
            for (int u = 0; u < kCombUnroll; ++u)
                if (i0 + u < k)
                    raw[u] = __ldg(reinterpret_cast<const uint4*>(e + (size_t)s_pos[i0 + u] * latent) + c);
#pragma unroll
            for (int u = 0; u < kCombUnroll; ++u) {
                if (i0 + u < k) {
                    const float wi = s_w[i0 + u];
                    const TA* vals = reinterpret_cast<const TA*>(&raw[u]);
#pragma unroll
                    for (int x = 0; x < V; ++x) y[q][x] = fmaf(wi, to_f32(vals[x]), y[q][x]);
                }
            }
        }
    }
    float ss = 0.0f;
#pragma unroll
    for (int q = 0; q < VPT; ++q)
        if (tid + q * (int)blockDim.x < nvec)
#pragma unroll
            for (int u = 0; u < V; ++u) ss = fmaf(y[q][u], y[q][u], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) tot += red[q];
    const float inv = 1.0f / sqrtf(tot / (float)latent + eps);
    uint4* zr = reinterpret_cast<uint4*>(z + (size_t)t * ldz);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
        const int c = tid + q * blockDim.x;
        if (c < nvec) {
            __align__(16) TA o[V];
#pragma unroll
            for (int u = 0; u < V; u += 4) {
                const float4 g = __ldg(g4 + (c * V + u) / 4);
                o[u + 0] = from_f32<TA>(y[q][u + 0] * inv * g.x);
                o[u + 1] = from_f32<TA>(y[q][u + 1] * inv * g.y);
                o[u + 2] = from_f32<TA>(y[q][u + 2] * inv * g.z);
                o[u + 3] = from_f32<TA>(y[q][u + 3] * inv * g.w);
            }
            zr[c] = *reinterpret_cast<const uint4*>(o);
        }
    }
}

template <typename TA>
int launch_combine_t(int T, int k, int latent, const TA* e, const float* w, const int* route_pos,
                     const float* gamma, float eps, TA* z, long long ldz, cudaStream_t s) {
    constexpr int V = 16 / sizeof(TA);
    const int nvec = latent / V;
    const int vpt = nvec <= kCombMaxThreads ? 1 : (nvec <= 2 * kCombMaxThreads ? 2 : 4);
    if (nvec > 4 * kCombMaxThreads) return QBMOE_EINVAL;
    const int threads = std::min(kCombMaxThreads, ((nvec + vpt - 1) / vpt + 31) & ~31);
    if (vpt == 1)
        k_combine_rmsnorm<TA, 1><<<T, threads, 0, s>>>(T, k, latent, e, w, route_pos, gamma, eps, z, ldz);
    else if (vpt == 2)
        k_combine_rmsnorm<TA, 2><<<T, threads, 0, s>>>(T, k, latent, e, w, route_pos, gamma, eps, z, ldz);
    else
        k_combine_rmsnorm<TA, 4><<<T, threads, 0, s>>>(T, k, latent, e, w, route_pos, gamma, eps, z, ldz);
    return QBMOE_OK;
}

}  // namespace

namespace qbh {

int launch_expert_offsets(int n, const int32_t* loads, int* offsets, int tile_rows, int* tile_off,
                          cudaStream_t s, int* nl) {
    k_expert_offsets<<<1, 1024, 0, s>>>(n, loads, offsets, tile_rows, tile_off);
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

int launch_scatter(int T, int n, int k, int tpw, const int32_t* idx, const int* blk_base, const int* offsets,
                   int* perm, int* route_pos, cudaStream_t s, int* nl) {
    const int bt = 8 * tpw;
    const int nblk = (T + bt - 1) / bt;
    k_scatter<<<nblk, bt, (size_t)n * sizeof(unsigned long long), s>>>(T, n, k, tpw, idx, blk_base, offsets,
                                                                        perm, route_pos);
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

int launch_scatter_rows(const void* src, int row_bytes, const int* route_pos, int T, int k, void* dst,
                        cudaStream_t s, int* nl) {
    if (row_bytes % 16 || !aligned16(src) || !aligned16(dst)) return QBMOE_EINVAL;
    const int vpr = row_bytes / 16;
    const long long total = (long long)T * vpr;
    const int grid = (int)std::min<long long>((total + 255) / 256, 152LL * 8);
    k_scatter_rows<<<std::max(grid, 1), 256, 0, s>>>(static_cast<const uint4*>(src), vpr, route_pos, T, k,
                                                     static_cast<uint4*>(dst));
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

int launch_combine_rmsnorm(int act_dtype, int T, int k, int latent, const void* e, const float* w,
                           const int* route_pos, const float* gamma, float eps, void* z, long long ldz,
                           cudaStream_t s, int* nl) {
    const int V = act_dtype == QBMOE_BF16 ? 8 : 4;
    if (latent % V || k > QBMOE_MAX_TOPK || !aligned16(gamma)) return QBMOE_EINVAL;
    int rc;
    if (act_dtype == QBMOE_BF16)
        rc = launch_combine_t<__nv_bfloat16>(T, k, latent, (const __nv_bfloat16*)e, w, route_pos, gamma, eps,
                                             (__nv_bfloat16*)z, ldz, s);
    else
        rc = launch_combine_t<float>(T, k, latent, (const float*)e, w, route_pos, gamma, eps, (float*)z, ldz, s);
    if (rc) return rc;
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

}  // namespace qbh
