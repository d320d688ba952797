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

// Router logits (optional; fp32 x W_r^T + o) + latent down-projection +
// shared gate/up in one launch.  h is bf16 [T, latent], or E4M3 pairs (hi
// plane, then lo plane: 2 x latent bytes a row) when the expert GEMMs run on
// the block-scaled MMA.
int tc_xside(TcPlan* p, int T, const void* x, bool with_router, float* logits, void* h, void* zcat, long long ldz,
             int* status, cudaStream_t s, int* nl);
// Whether the MXFP4 expert GEMMs run on the block-scaled MMA: their token
// inputs (h_perm, act) are then E4M3 bytes.
bool tc_mx_scaled(const TcPlan* p);
int tc_expert_gate_up(TcPlan* p, int T, const void* h_perm, const int* offsets, const int* tile_off, void* act,
                      int* status, cudaStream_t s, int* nl);
int tc_expert_down(TcPlan* p, int T, const void* act, const int* offsets, const int* tile_off, void* e,
                   int* status, cudaStream_t s, int* nl);
int tc_up_shared(TcPlan* p, int T, const void* zcat, long long ldz, void* out, int* status, cudaStream_t s,
                 int* nl);

}  // namespace qbh
