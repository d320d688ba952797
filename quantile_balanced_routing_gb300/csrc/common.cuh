// Shared device helpers of the qbmoe CUDA path (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/qbmoe.h"

#define QB_DEV __device__ __forceinline__

namespace qb {

// ---------------------------------------------------------------------------
// Router score: the exactly specified fp32 sigmoid of the routing contract.
// Every step is one IEEE fp32 operation (explicit _rn intrinsics: no FMA
// contraction), so any conforming implementation of the recipe reproduces
// the bits.  Recipe: Cody-Waite reduction of e^-x by ln 2 split in a 15-bit
// head and a tail, degree-7 Taylor polynomial in Horner form, exact 2^j
// scaling, then 1/(1+e).
// ---------------------------------------------------------------------------
QB_DEV float score_of_logit(float x) {
    const float kLog2e = 0x1.715476p+0f;
    const float kLn2Hi = 0x1.62e4p-1f;
    const float kLn2Lo = 0x1.7f7d1cp-20f;
    x = fminf(fmaxf(x, -80.0f), 80.0f);
    const float y = -x;
    const float j = rintf(__fmul_rn(y, kLog2e));
    const float r = __fsub_rn(__fsub_rn(y, __fmul_rn(j, kLn2Hi)), __fmul_rn(j, kLn2Lo));
    float p = 0x1.a01a02p-13f;                       // 1/5040
    p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);  // 1/720
    p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);   // 1/120
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);   // 1/24
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);   // 1/6
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    const float two_j = __int_as_float(((int)j + 127) << 23);
    const float e = __fmul_rn(p, two_j);
    // the correctly rounded reciprocal is the IEEE quotient 1 / (1 + e)
    return __frcp_rn(__fadd_rn(1.0f, e));
}

// SiTU-GLU: a = b1 tanh(g/b1), b = b2 tanh(u/b2), out = a sigmoid(a) b.
QB_DEV float situ_glu(float g, float u, float beta1, float beta2) {
    const float a = beta1 * tanhf(g / beta1);
    const float b = beta2 * tanhf(u / beta2);
    return a / (1.0f + expf(-a)) * b;
}

// (value desc, index asc) order: true when (va, ja) ranks before (vb, jb).
QB_DEV bool ranks_before(float va, int ja, float vb, int jb) {
    return va > vb || (va == vb && ja < jb);
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key).
QB_DEV uint32_t f32_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
QB_DEV float f32_from_order_key(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

template <typename T> QB_DEV float to_f32(T v);
template <> QB_DEV float to_f32<float>(float v) { return v; }
template <> QB_DEV float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> QB_DEV T from_f32(float v);
template <> QB_DEV float from_f32<float>(float v) { return v; }
template <> QB_DEV __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

QB_DEV void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// scheduled while the kernel before it on the stream is still running;
// pdl_wait blocks until that kernel has completed and its writes are
// visible, so it comes before the first read of anything the earlier kernel
// writes.  pdl_trigger lets the next kernel's CTAs be scheduled once every
// CTA of this kernel has called it (or exited).  Both are no-ops for a
// kernel launched without the attribute.
QB_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QB_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace qb

// Host-side launch helpers shared by the .cu files.
namespace qbh {
inline int cuda_err(cudaError_t e) { return e == cudaSuccess ? QBMOE_OK : QBMOE_ECUDA; }

// Launch with programmatic stream serialisation (see qb::pdl_wait): the
// kernel may start while the previous kernel on the stream drains.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cuda_err(cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...));
}
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Once per device (api.cu): checks that the current device is sm_103 and sets
// every kernel's dynamic shared-memory limit to the largest size any call
// uses, so that no launch sequence sets an attribute between its launches.
int device_init();
int route_init_attributes();   // route.cu
int tc_init_attributes();      // gemm_tc.cu

// Route kernels (route.cu)
struct RouteBuffers {
    float* margins;      // [n, T]
    float* bias_raw;     // [n] coordinate biases b' of the last sweep
    float* bias_fin;     // [n] b' minus the common offset (written by the sweep's last select CTA)
    unsigned* ticket;    // select CTAs finished (zeroed by the sweep's token pass)
    int* blk_cnt;        // [n, nblk] per-block expert counts (expert-major)
};
size_t route_ws_layout(int T, int n, int k, RouteBuffers* rb, void* base);
int route_tokens_per_warp(int T);
// zero (may be NULL): nzero int32 set to 0 by the same launch.
int launch_scores(const float* logits, float* scores, long long count, cudaStream_t s, int* nl,
                  int32_t* zero = nullptr, int nzero = 0);
// logits may be NULL (scores already computed); bias_in may be NULL (zeros).
// blk_cnt (may be NULL): the top-k's per-CTA expert counts, expert-major;
// loads (may be NULL): zeroed, then the expert loads accumulated atomically.
int launch_qb_and_topk(int T, int n, int k, int sweeps, const float* logits, float* scores, const float* bias_in,
                       float* bias_out, int32_t* idx, float* w, int* blk_cnt, const RouteBuffers& rb,
                       cudaStream_t s, int* nl, int32_t* loads = nullptr);
int launch_loads_from_counts(int T, int n, int tpw, const int* blk_cnt, int32_t* loads, cudaStream_t s,
                             int* nl);

// Cyclic (Gauss-Seidel) QB (route.cu): the route buffers plus the sweep's own.
struct GsBuffers {
    float* lv;     // [T, k+1] top-(k+1) values per token
    int* li;       // [T, k+1] their experts
    float* mj;     // [T] margins of the expert being updated
    float* b;      // [n] current biases
    int* done;     // balanced flag
};
size_t route_gs_ws_layout(int T, int n, int k, RouteBuffers* rb, GsBuffers* gb, void* base);
int launch_qb_gs(int T, int n, int k, int max_sweeps, int stop_when_balanced, const float* logits, float* scores,
                 const float* bias_in, float* bias_out, int32_t* topk_idx, float* topk_w, int32_t* loads,
                 int32_t* sweeps_done, const RouteBuffers& rb, const GsBuffers& gb, cudaStream_t s, int* nl);
}  // namespace qbh
