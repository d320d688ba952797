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

int tc_router(TcPlan* p, int T, const void* x, float* scores, cudaStream_t s, int* nl);
int tc_xside(TcPlan* p, int T, const void* x, void* h, void* zcat, long long ldz, cudaStream_t s, int* nl);
int tc_expert_gate_up(TcPlan* p, int T, const void* h, const int* perm, const int* offsets, const int* tile_off,
                      int max_tiles, void* act, cudaStream_t s, int* nl);
int tc_expert_down(TcPlan* p, int T, const void* act, const int* offsets, const int* tile_off, int max_tiles,
                   void* e, cudaStream_t s, int* nl);
int tc_up_shared(TcPlan* p, int T, const void* zcat, long long ldz, void* out, cudaStream_t s, int* nl);

}  // namespace qbh
