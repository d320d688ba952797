// moe_route_qb_noalloc: the QB router with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they route:
// engines that plan every buffer up front and forbid allocation on the
// serving path, and plug-ins that are handed only their inputs and outputs
// by a host program that owns all memory.  This
// entry point serves them: it takes only inputs and outputs and keeps its
// scratch (the margin matrix, raw biases, per-block counts) in a file-scope
// __device__ array of kNoAllocScratchBytes, which every GPU that loads the
// library holds until the process exits.
#include "common.cuh"

#include <mutex>

namespace {

// 32 MiB: enough for T * n up to about 8.3 million (e.g. 8192 tokens x 1024 experts).
constexpr size_t kNoAllocScratchBytes = 32u << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once per
// device).  The array's name in host code is only a host-side stand-in, so
// the kernels must be given this address instead.
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QBMOE_ECUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return QBMOE_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QBMOE_OK;
}

}  // namespace

extern "C" size_t qbmoe_route_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int moe_route_qb_noalloc(int T, int n, int k, int qb_sweeps, const float* logits, const float* bias_in,
                                    float* bias_out, float* scores, int32_t* topk_idx, float* topk_w,
                                    int32_t* loads, qbmoe_stream_t stream) {
    if (T < 1 || n < 2 || n > QBMOE_MAX_EXPERTS || k < 1 || k >= n || k > QBMOE_MAX_TOPK || qb_sweeps < 0)
        return QBMOE_EINVAL;
    if (!logits || !scores || !topk_idx || !topk_w || !loads) return QBMOE_EINVAL;
    const void* ptrs[] = {logits, bias_in, bias_out, scores, topk_idx, topk_w, loads};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    // Sizes whose scratch does not fit the fixed array are refused.
    if (qbmoe_route_workspace_bytes(T, n, k) > kNoAllocScratchBytes) return QBMOE_EWORKSPACE;
    int rc = qbh::device_init();
    if (rc) return rc;
    void* scratch = nullptr;
    if ((rc = scratch_for_current_device(&scratch))) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qbh::RouteBuffers rb;
    qbh::route_ws_layout(T, n, k, &rb, scratch);
    // Every scratch region is fully written before it is read, so stale
    // contents from an earlier call cannot leak into this one.
    int nl = 0;
    rc = qbh::launch_qb_and_topk(T, n, k, qb_sweeps, logits, scores, bias_in, bias_out, topk_idx, topk_w,
                                 rb.blk_cnt, rb, s, &nl);
    if (!rc) rc = qbh::launch_loads_from_counts(T, n, qbh::route_tokens_per_warp(T), rb.blk_cnt, loads, s, &nl);
    return rc;
}
