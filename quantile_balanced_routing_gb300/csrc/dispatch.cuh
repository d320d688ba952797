// Host-side launchers of the dispatch / GEMM kernels (internal to the library).
#pragma once

#include "common.cuh"

namespace qbh {

int launch_expert_offsets(int n, const int32_t* loads, int* offsets, int tile_rows, int* tile_off,
                          cudaStream_t s, int* nl);
int launch_scatter(int T, int n, int k, int tpw, const int32_t* idx, const int* blk_base, const int* offsets,
                   int* perm, int* route_pos, cudaStream_t s, int* nl);
// Token rows into expert order: dst[route_pos[t * k + i]] = src[t] for
// t < T, i < k (rows of row_bytes, a multiple of 16; 16-byte aligned bases).
int launch_scatter_rows(const void* src, int row_bytes, const int* route_pos, int T, int k, void* dst,
                        cudaStream_t s, int* nl);
int launch_combine_rmsnorm(int act_dtype, int T, int k, int latent, const void* e, const float* w,
                           const int* route_pos, const float* gamma, float eps, void* z, long long ldz,
                           cudaStream_t s, int* nl);

// Epilogues of the GEMMs.
enum GemmEpi { EPI_STORE = 0, EPI_ROUTER = 1, EPI_SITU = 2 };

// out[r, f] = epi( sum_k A[r, k] * W[f, k] ), f < F.
//   A: [rows, K1 + K2] activations (act dtype), row stride lda; in grouped
//      mode rows are taken through a_rows (if given) within each expert's
//      segment [seg_off[g], seg_off[g+1]).
//   W: for k < K1 from W1 [F, K1], for k >= K1 from W2 [F, K2] (dense, act
//      dtype).  Grouped: expert g's weights start at W1 + g * F * K1 (wfmt);
//      MXFP4 weights use S1 (scales).  EPI_SITU also reads Wu/Su (up branch).
//   out: row r at out + r * ldo (act dtype; for EPI_ROUTER the fp32 logit
//        plus col_bias, from which the QB token pass takes the score).
struct GemmArgs {
    const void* A = nullptr;
    long long lda = 0;
    const int* a_rows = nullptr;
    int rows = 0;
    int K1 = 0, K2 = 0;
    const void* W1 = nullptr;
    const uint8_t* S1 = nullptr;
    const void* W2 = nullptr;
    const void* Wu = nullptr;
    const uint8_t* Su = nullptr;
    int F = 0;
    const int* seg_off = nullptr;
    const int* tile_off = nullptr;
    int n_groups = 0;
    int max_tiles = 0;           // grouped: upper bound of token tiles
    void* out = nullptr;
    long long ldo = 0;
    const float* col_bias = nullptr;
    float beta1 = 4.0f, beta2 = 25.0f;
};

constexpr int kSimtBM = 64;   // token rows per SIMT tile (grouped tile_off granularity)

// act_dtype: QBMOE_F32 | QBMOE_BF16; wfmt: QBMOE_W_* of W1/Wu (W2 is dense act dtype).
int launch_gemm_simt(int act_dtype, int wfmt, GemmEpi epi, const GemmArgs& a, cudaStream_t s, int* nl);

}  // namespace qbh
