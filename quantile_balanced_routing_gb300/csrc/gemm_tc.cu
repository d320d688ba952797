// tcgen05 / TMA tensor-core GEMMs (bf16 activations; bf16 or MXFP4 weights).
#include "gemm_tc.cuh"

namespace qbh {

struct TcPlan {
    bool enabled = false;
};

TcPlan* tc_plan_create(const qbmoe_config&) { return new TcPlan(); }
void tc_plan_destroy(TcPlan* p) { delete p; }
int tc_plan_set_weights(TcPlan*, const qbmoe_config&, const qbmoe_weights&) { return QBMOE_OK; }
bool tc_enabled(const TcPlan* p) { return p && p->enabled; }
int tc_token_tile(const TcPlan*, int) { return 64; }
int tc_router(TcPlan*, int, const void*, float*, cudaStream_t, int*) { return QBMOE_EINVAL; }
int tc_xside(TcPlan*, int, const void*, void*, void*, long long, cudaStream_t, int*) { return QBMOE_EINVAL; }
int tc_expert_gate_up(TcPlan*, int, const void*, const int*, const int*, const int*, int, void*, cudaStream_t, int*) {
    return QBMOE_EINVAL;
}
int tc_expert_down(TcPlan*, int, const void*, const int*, const int*, int, void*, cudaStream_t, int*) {
    return QBMOE_EINVAL;
}
int tc_up_shared(TcPlan*, int, const void*, long long, void*, cudaStream_t, int*) { return QBMOE_EINVAL; }

}  // namespace qbh
