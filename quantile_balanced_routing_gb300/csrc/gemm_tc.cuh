// tcgen05 / TMA tensor-core GEMMs of the layer (bf16 and MXFP4 weights).
#pragma once

#include "common.cuh"

namespace qbh {

struct TcPlan;

TcPlan* tc_plan_create(const qbmoe_config& cfg);
void tc_plan_destroy(TcPlan* p);
int tc_plan_set_weights(TcPlan* p, const qbmoe_config& cfg, const qbmoe_weights& w);
bool tc_enabled(const TcPlan* p);
// token rows per grouped tile for T tokens (the tile_off granularity)
int tc_token_tile(const TcPlan* p, int T);

void tc_set_wait_limit(TcPlan* p, long long iterations);
void tc_set_stall(TcPlan* p, int on);

// The layer's tensor-core launches.  Each tc_prepare_* call builds one
// launch's parameters (every tensor map encoded, tile and kernel variant
// chosen) without touching the device; tc_launch enqueues a prepared launch.
// moe_latent_forward prepares all of them before its first launch, so that
// a failure to prepare leaves nothing launched.
enum { TC_XSIDE = 0, TC_GATE_UP = 1, TC_DOWN = 2, TC_UP_SHARED = 3, TC_STAGES = 4 };

// A token row of K activations in E4M3 for the block-scaled MMA: K hi bytes,
// K lo bytes, then K / 32 E8M0 block scales (K % 512 == 0 keeps every part
// 16-byte aligned), the row padded to a multiple of 128 bytes so that every
// 128-byte K block of a row is one aligned line.
__host__ __device__ constexpr long long mx_row_bytes(long long K) { return (2 * K + K / 32 + 127) / 128 * 128; }

// Router logits (optional; fp32 x W_r^T + o) + latent down-projection +
// shared gate/up in one launch.  h is bf16 [T, latent], or E4M3 rows of
// mx_row_bytes(latent) when the expert GEMMs run on the block-scaled MMA.
int tc_prepare_xside(TcPlan* p, int T, const void* x, bool with_router, float* logits, void* h, void* zcat,
                     long long ldz, int* status);
// Whether the MXFP4 expert GEMMs run on the block-scaled MMA: their token
// inputs (h_perm, act) are then E4M3 bytes.
bool tc_mx_scaled(const TcPlan* p);
// Expert gate/up.  With h and perm given, bf16 launches on the one-CTA
// kernel gather their token rows from h [T, latent] through perm (token of
// each route position) and set *gathered; otherwise they read h_perm, the
// rows already in expert order.
int tc_prepare_gate_up(TcPlan* p, int T, const void* h_perm, const int* offsets, const int* tile_off, void* act,
                       int* status, const void* h = nullptr, const int* perm = nullptr, bool* gathered = nullptr);
int tc_prepare_down(TcPlan* p, int T, const void* act, const int* offsets, const int* tile_off, void* e,
                    int* status);
int tc_prepare_up_shared(TcPlan* p, int T, const void* zcat, long long ldz, void* out, int* status);
int tc_launch(TcPlan* p, int stage, cudaStream_t s, int* nl);

}  // namespace qbh
