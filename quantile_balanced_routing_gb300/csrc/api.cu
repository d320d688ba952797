// C ABI of the layer: context, workspace and the forward orchestration.
//
// [K3-width] = "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club).
// The stages follow the pages' layer: full-width sigmoid router (Q&A on
// routing), QB bias (Q&A on Quantile Balancing), latent down-projection
// (延伸解读 "why a half-width latent space"), per-expert SiTU-GLU in latent
// space (Q&A on SiTU-GLU), weighted combine + RMSNorm (Q&A on RMSNorm),
// up-projection plus the merged full-width shared expert (Q&A on the shared
// expert).
#include "common.cuh"
#include "dispatch.cuh"
#include "gemm_tc.cuh"

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

namespace {

int check_device_arch(int dev) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return QBMOE_ECUDA;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return QBMOE_ECUDA;
    return (major == 10 && minor == 3) ? QBMOE_OK : QBMOE_EARCH;
}

constexpr int kMaxDevices = 64;
std::mutex g_init_mu;
bool g_init_done[kMaxDevices] = {};

}  // namespace

int qbh::device_init() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QBMOE_ECUDA;
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (g_init_done[dev]) return QBMOE_OK;
    int rc = check_device_arch(dev);
    if (!rc) rc = qbh::route_init_attributes();
    if (!rc) rc = qbh::tc_init_attributes();
    if (rc) {
        cudaGetLastError();
        return rc;
    }
    g_init_done[dev] = true;
    return QBMOE_OK;
}

namespace {

constexpr int kMaxStages = 16;

struct Stage {
    const char* name;
};

}  // namespace

struct qbmoe_ctx {
    qbmoe_config cfg{};
    int max_tokens = 0;
    int device = 0;
    qbmoe_weights w{};
    bool have_weights = false;
    void* packed = nullptr;    // weights copied by qbmoe_pack_weights (owned)
    void* ws = nullptr;
    size_t ws_bytes = 0;
    // workspace views
    float* scores = nullptr;
    float* logits = nullptr;   // router GEMM output (logit + offset) [T, n] fp32
    qbh::RouteBuffers rb{};
    qbh::GsBuffers gb{};       // cyclic QB (qb_mode = QBMOE_QB_GAUSS_SEIDEL)
    int32_t* idx = nullptr;
    float* wts = nullptr;
    int32_t* loads = nullptr;
    int* offsets = nullptr;
    int* tile_off_simt = nullptr;
    int* tile_off_tc = nullptr;
    int* perm = nullptr;
    int* route_pos = nullptr;
    void* h = nullptr;
    void* h_perm = nullptr;
    void* act = nullptr;
    void* e = nullptr;
    void* zcat = nullptr;
    int* status = nullptr;
    long long wait_limit = 0;
    // timing: a ring of `slots` forwards, each with kMaxStages + 1 events
    int slots = 0;
    std::vector<cudaEvent_t> ev;
    const char* stage_names[kMaxStages] = {};
    int n_stages = 0;
    long long recorded = 0;
    int launches = 0;
    qbh::TcPlan* tc = nullptr;
};

namespace {

size_t elt(int dtype) { return dtype == QBMOE_BF16 ? 2 : 4; }

size_t layout(const qbmoe_config& c, int T, qbmoe_ctx* x, char* base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = qbh::align_up(off + bytes, 256);
        return base ? base + o : nullptr;
    };
    const int n = c.n_experts, k = c.top_k;
    const size_t routes = (size_t)T * k;
    const size_t a = elt(c.act_dtype);
    char* p_scores = take((size_t)T * n * 4);
    char* p_logits = take((size_t)T * n * 4);
    const bool gs = c.qb_mode == QBMOE_QB_GAUSS_SEIDEL;
    const size_t rbytes = gs ? qbh::route_gs_ws_layout(T, n, k, nullptr, nullptr, nullptr)
                             : qbh::route_ws_layout(T, n, k, nullptr, nullptr);
    char* p_route = take(rbytes);
    char* p_idx = take(routes * 4);
    char* p_w = take(routes * 4);
    char* p_loads = take((size_t)n * 4);
    char* p_off = take((size_t)(n + 1) * 4);
    char* p_toff = take((size_t)(n + 1) * 4);
    char* p_toff2 = take((size_t)(n + 1) * 4);
    char* p_perm = take(routes * 4);
    char* p_rpos = take(routes * 4);
    // h, h_perm and act rows: bf16 or fp32, or, for MXFP4 experts on the
    // block-scaled MMA, E4M3 rows with their block scales (the larger size)
    const bool mx = c.expert_wfmt == QBMOE_W_MXFP4;
    const size_t h_row = mx ? (size_t)qbh::mx_row_bytes(c.latent) : c.latent * a;
    const size_t act_row = mx ? (size_t)qbh::mx_row_bytes(c.expert_inter) : c.expert_inter * a;
    char* p_h = take((size_t)T * h_row);
    char* p_hp = take(routes * h_row);
    char* p_act = take(routes * act_row);
    char* p_e = take(routes * c.latent * a);
    char* p_z = take((size_t)T * (c.latent + c.shared_inter) * a);
    char* p_status = take(256);
    if (x && base) {
        x->scores = (float*)p_scores;
        x->logits = (float*)p_logits;
        if (gs) qbh::route_gs_ws_layout(T, n, k, &x->rb, &x->gb, p_route);
        else qbh::route_ws_layout(T, n, k, &x->rb, p_route);
        x->idx = (int32_t*)p_idx;
        x->wts = (float*)p_w;
        x->loads = (int32_t*)p_loads;
        x->offsets = (int*)p_off;
        x->tile_off_simt = (int*)p_toff;
        x->tile_off_tc = (int*)p_toff2;
        x->perm = (int*)p_perm;
        x->route_pos = (int*)p_rpos;
        x->h = p_h;
        x->h_perm = p_hp;
        x->act = p_act;
        x->e = p_e;
        x->zcat = p_z;
        x->status = (int*)p_status;
    }
    return off;
}

int validate(const qbmoe_config* c, int max_tokens) {
    if (!c) return QBMOE_EINVAL;
    if (c->d < 1 || c->latent < 1 || c->expert_inter < 1 || c->shared_inter < 0) return QBMOE_EINVAL;
    if (c->n_experts < 2 || c->n_experts > QBMOE_MAX_EXPERTS) return QBMOE_EINVAL;
    if (c->top_k < 1 || c->top_k >= c->n_experts || c->top_k > QBMOE_MAX_TOPK) return QBMOE_EINVAL;
    if (c->qb_sweeps < 0 || max_tokens < 1) return QBMOE_EINVAL;
    if (c->qb_mode != QBMOE_QB_JACOBI && c->qb_mode != QBMOE_QB_GAUSS_SEIDEL) return QBMOE_EINVAL;
    if (c->act_dtype != QBMOE_F32 && c->act_dtype != QBMOE_BF16) return QBMOE_EINVAL;
    if (c->act_dtype == QBMOE_F32 && c->expert_wfmt != QBMOE_W_F32) return QBMOE_EINVAL;
    if (c->act_dtype == QBMOE_BF16 && c->expert_wfmt != QBMOE_W_BF16 && c->expert_wfmt != QBMOE_W_MXFP4)
        return QBMOE_EINVAL;
    if (c->expert_wfmt == QBMOE_W_MXFP4 && (c->latent % 32 || c->expert_inter % 32)) return QBMOE_EINVAL;
    if (c->latent > 128 * 8 * 4) return QBMOE_EINVAL;   // combine kernel: 128 threads x 8 vectors
    if (!(c->situ_beta1 > 0.0f) || !(c->situ_beta2 > 0.0f) || !(c->rms_eps >= 0.0f)) return QBMOE_EINVAL;
    // 16-byte rows of every activation matrix (vector and TMA access)
    const int a = c->act_dtype == QBMOE_BF16 ? 8 : 4;
    if (c->d % a || c->latent % a || c->expert_inter % a || c->shared_inter % a) return QBMOE_EINVAL;
    if ((long long)max_tokens * c->top_k > (1LL << 30)) return QBMOE_EINVAL;
    return QBMOE_OK;
}

struct StageClock {
    qbmoe_ctx* c;
    cudaStream_t s;
    int i = 0;
    cudaEvent_t* slot() { return c->ev.data() + (size_t)(c->recorded % c->slots) * (kMaxStages + 1); }
    void mark(const char* name) {
        if (!c->slots || i >= kMaxStages) return;
        cudaEventRecord(slot()[i], s);
        c->stage_names[i] = name;
        ++i;
    }
    void end() {
        if (!c->slots || i == 0) return;
        cudaEventRecord(slot()[i], s);
        c->n_stages = i;
        ++c->recorded;
    }
};

}  // namespace

extern "C" size_t qbmoe_layer_workspace_bytes(const qbmoe_config* cfg, int max_tokens) {
    if (validate(cfg, max_tokens)) return 0;
    return layout(*cfg, max_tokens, nullptr, nullptr);
}

extern "C" int qbmoe_create(qbmoe_ctx** out, const qbmoe_config* cfg, int max_tokens) {
    if (!out) return QBMOE_EINVAL;
    *out = nullptr;
    int rc = validate(cfg, max_tokens);
    if (rc) return rc;
    if ((rc = qbh::device_init())) return rc;
    qbmoe_ctx* c = new (std::nothrow) qbmoe_ctx();
    if (!c) return QBMOE_ENOMEM;
    c->cfg = *cfg;
    c->max_tokens = max_tokens;
    cudaGetDevice(&c->device);
    c->ws_bytes = layout(*cfg, max_tokens, nullptr, nullptr);
    if (cudaMalloc(&c->ws, c->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return QBMOE_ENOMEM;
    }
    layout(*cfg, max_tokens, c, static_cast<char*>(c->ws));
    if (cudaMemset(c->status, 0, 4) != cudaSuccess) {
        cudaFree(c->ws);
        delete c;
        return QBMOE_ECUDA;
    }
    c->tc = qbh::tc_plan_create(c->cfg);
    *out = c;
    return QBMOE_OK;
}

extern "C" int qbmoe_destroy(qbmoe_ctx* c) {
    if (!c) return QBMOE_OK;
    cudaDeviceSynchronize();
    for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
    qbh::tc_plan_destroy(c->tc);
    cudaFree(c->ws);
    if (c->packed) cudaFree(c->packed);
    delete c;
    return QBMOE_OK;
}

extern "C" int qbmoe_set_weights(qbmoe_ctx* c, const qbmoe_weights* w) {
    if (!c || !w) return QBMOE_EINVAL;
    const qbmoe_config& g = c->cfg;
    if (!w->w_router || !w->w_down || !w->w_gate || !w->w_up || !w->w_out || !w->rms_gamma || !w->w_proj_up)
        return QBMOE_EINVAL;
    if (g.shared_inter > 0 && (!w->w_shared_gate || !w->w_shared_up || !w->w_shared_out)) return QBMOE_EINVAL;
    if (g.expert_wfmt == QBMOE_W_MXFP4 && (!w->s_gate || !w->s_up || !w->s_out)) return QBMOE_EINVAL;
    const void* ptrs[] = {w->w_router, w->router_offset, w->w_down, w->w_gate, w->w_up, w->w_out,
                          w->rms_gamma, w->w_proj_up, w->w_shared_gate, w->w_shared_up, w->w_shared_out};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    // Packed E2M1 weights are read by TMA copies that unpack 4-bit codes,
    // which need 32-byte aligned bases.
    if (g.expert_wfmt == QBMOE_W_MXFP4)
        for (const void* p : {w->w_gate, w->w_up, w->w_out})
            if ((reinterpret_cast<uintptr_t>(p) & 31u) != 0) return QBMOE_EINVAL;
    c->w = *w;
    c->have_weights = true;
    int rc = qbh::tc_plan_set_weights(c->tc, c->cfg, *w);
    return rc;
}

namespace {

// Flags E8M0 scale bytes of 0xFF (NaN: not a weight scale) in [n] bytes.
__global__ void k_check_e8m0(const uint8_t* __restrict__ sc, long long n, int* __restrict__ bad) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        if (sc[i] == 0xFFu) atomicExch(bad, 1);
}

struct PackItem {
    const void* src;
    size_t bytes;
    const void** dst;
    bool scales;
};

}  // namespace

extern "C" int qbmoe_pack_weights(qbmoe_ctx* c, const qbmoe_weights* w, qbmoe_stream_t stream) {
    if (!c || !w) return QBMOE_EINVAL;
    const qbmoe_config& g = c->cfg;
    const size_t a = elt(g.act_dtype);
    const size_t n = g.n_experts, d = g.d, L = g.latent, m = g.expert_inter, ms = g.shared_inter;
    const bool mx = g.expert_wfmt == QBMOE_W_MXFP4;
    const size_t we = mx ? 0 : elt(g.expert_wfmt);
    // expert tensor bytes: MXFP4 packs two codes a byte with one scale byte per 32
    auto ex = [&](size_t rows, size_t K) { return mx ? rows * K / 2 : rows * K * we; };
    qbmoe_weights nw{};
    std::vector<PackItem> items = {
        {w->w_router, n * d * a, &nw.w_router, false},
        {w->router_offset, w->router_offset ? n * 4 : 0, (const void**)&nw.router_offset, false},
        {w->w_down, L * d * a, &nw.w_down, false},
        {w->w_gate, ex(n * m, L), &nw.w_gate, false},
        {w->w_up, ex(n * m, L), &nw.w_up, false},
        {w->w_out, ex(n * L, m), &nw.w_out, false},
        {w->rms_gamma, L * 4, (const void**)&nw.rms_gamma, false},
        {w->w_proj_up, d * L * a, &nw.w_proj_up, false},
    };
    if (ms > 0) {
        items.push_back({w->w_shared_gate, ms * d * a, &nw.w_shared_gate, false});
        items.push_back({w->w_shared_up, ms * d * a, &nw.w_shared_up, false});
        items.push_back({w->w_shared_out, d * ms * a, &nw.w_shared_out, false});
    }
    if (mx) {
        items.push_back({w->s_gate, n * m * L / 32, (const void**)&nw.s_gate, true});
        items.push_back({w->s_up, n * m * L / 32, (const void**)&nw.s_up, true});
        items.push_back({w->s_out, n * L * m / 32, (const void**)&nw.s_out, true});
    }
    size_t total = 256;   // the first 256 bytes hold the scale check's flag
    for (const PackItem& it : items) {
        if (it.bytes && !it.src) return QBMOE_EINVAL;
        total = qbh::align_up(total + it.bytes, 256);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device) return QBMOE_EINVAL;
    void* buf = nullptr;
    if (cudaMalloc(&buf, total) != cudaSuccess) {
        cudaGetLastError();
        return QBMOE_ENOMEM;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(buf);
    int* bad = reinterpret_cast<int*>(base);
    bool ok = cudaMemsetAsync(bad, 0, sizeof(int), s) == cudaSuccess;
    size_t off = 256;
    for (const PackItem& it : items) {
        if (!it.bytes) continue;
        char* dst = base + off;
        ok = ok && cudaMemcpyAsync(dst, it.src, it.bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
        if (ok && it.scales) {
            k_check_e8m0<<<1216, 256, 0, s>>>(reinterpret_cast<const uint8_t*>(dst), (long long)it.bytes, bad);
            ok = cudaGetLastError() == cudaSuccess;
        }
        *it.dst = dst;
        off = qbh::align_up(off + it.bytes, 256);
    }
    int flag = 0;
    ok = ok && cudaMemcpyAsync(&flag, bad, sizeof(int), cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaStreamSynchronize(s) == cudaSuccess;
    int rc = !ok ? QBMOE_ECUDA : (flag ? QBMOE_EINVAL : QBMOE_OK);
    if (!rc) {
        const qbmoe_weights prev = c->w;
        const bool had = c->have_weights;
        rc = qbmoe_set_weights(c, &nw);
        if (rc) {
            c->w = prev;
            c->have_weights = had;
            if (had) qbh::tc_plan_set_weights(c->tc, c->cfg, prev);
        }
    }
    if (rc) {
        cudaGetLastError();
        cudaFree(buf);
        return rc;
    }
    if (c->packed) cudaFree(c->packed);
    c->packed = buf;
    return QBMOE_OK;
}

extern "C" int qbmoe_set_timing(qbmoe_ctx* c, int slots) {
    if (!c || slots < 0 || slots > 4096) return QBMOE_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return QBMOE_ECUDA;
    for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
    c->ev.assign((size_t)slots * (kMaxStages + 1), nullptr);
    for (auto& e : c->ev)
        if (cudaEventCreate(&e) != cudaSuccess) return QBMOE_ECUDA;
    c->slots = slots;
    c->recorded = 0;
    c->n_stages = 0;
    return QBMOE_OK;
}

extern "C" int qbmoe_stage_times(qbmoe_ctx* c, float* ms, const char** names, int max) {
    if (!c || !ms) return QBMOE_EINVAL;
    if (!c->slots || c->recorded == 0) return 0;
    const long long have = c->recorded < c->slots ? c->recorded : c->slots;
    const int n = c->n_stages < max ? c->n_stages : max;
    for (int i = 0; i < n; ++i) ms[i] = 0.0f;
    for (long long q = c->recorded - have; q < c->recorded; ++q) {
        cudaEvent_t* e = c->ev.data() + (size_t)(q % c->slots) * (kMaxStages + 1);
        if (cudaEventSynchronize(e[c->n_stages]) != cudaSuccess) return QBMOE_ECUDA;
        for (int i = 0; i < n; ++i) {
            float t = 0.0f;
            if (cudaEventElapsedTime(&t, e[i], e[i + 1]) != cudaSuccess) return QBMOE_ECUDA;
            ms[i] += t / (float)have;
        }
    }
    if (names)
        for (int i = 0; i < n; ++i) names[i] = c->stage_names[i];
    return n;
}

extern "C" int qbmoe_last_launch_count(qbmoe_ctx* c) { return c ? c->launches : 0; }

extern "C" int qbmoe_set_wait_limit(qbmoe_ctx* c, long long iterations) {
    if (!c) return QBMOE_EINVAL;
    c->wait_limit = iterations > 0 ? iterations : 0;
    qbh::tc_set_wait_limit(c->tc, c->wait_limit);
    return QBMOE_OK;
}

extern "C" int qbmoe_debug_stall(qbmoe_ctx* c, int enable) {
    if (!c) return QBMOE_EINVAL;
    qbh::tc_set_stall(c->tc, enable != 0);
    return QBMOE_OK;
}

extern "C" int qbmoe_uses_tensor_cores(qbmoe_ctx* c) { return c && qbh::tc_enabled(c->tc) ? 1 : 0; }

extern "C" int qbmoe_status(qbmoe_ctx* c, qbmoe_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return QBMOE_ECUDA;
    if (cudaGetLastError() != cudaSuccess) return QBMOE_ECUDA;
    if (!c) return QBMOE_OK;
    int v = 0;
    if (cudaMemcpy(&v, c->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return QBMOE_ECUDA;
    if (v != 0 && cudaMemset(c->status, 0, 4) != cudaSuccess) return QBMOE_ECUDA;
    return v;
}

extern "C" const char* qbmoe_strerror(int code) {
    switch (code) {
        case QBMOE_OK: return "ok";
        case QBMOE_EINVAL: return "invalid argument";
        case QBMOE_ENOMEM: return "device allocation failed";
        case QBMOE_ECUDA: return "CUDA error";
        case QBMOE_EARCH: return "device is not sm_103 (GB300)";
        case QBMOE_EWORKSPACE: return "workspace too small";
        case QBMOE_ETIMEOUT: return "bounded device wait expired";
        case QBMOE_EDEVICE: return "device-side check failed";
        default: return "unknown status";
    }
}

extern "C" int moe_latent_forward(qbmoe_ctx* c, int T, const void* x, const float* logits_in, const float* bias_in,
                                  float* bias_out, void* out, float* scores_opt, int32_t* idx_opt, float* w_opt,
                                  int32_t* loads_opt, qbmoe_stream_t stream) {
    // ---- every check, and every launch's parameters, before the first launch
    if (!c || !c->have_weights || !x || !out) return QBMOE_EINVAL;
    if (T < 1) return QBMOE_EINVAL;
    if (T > c->max_tokens) return QBMOE_EWORKSPACE;
    const void* ptrs[] = {x, logits_in, bias_in, bias_out, out, scores_opt, idx_opt, w_opt, loads_opt};
    for (const void* p : ptrs)
        if (p && !qbh::aligned16(p)) return QBMOE_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device) return QBMOE_EINVAL;
    int rc = qbh::device_init();
    if (rc) return rc;

    const qbmoe_config& g = c->cfg;
    const int n = g.n_experts, k = g.top_k, L = g.latent, m = g.expert_inter, ms = g.shared_inter, d = g.d;
    const int ad = g.act_dtype;
    const int dense_wf = ad == QBMOE_BF16 ? QBMOE_W_BF16 : QBMOE_W_F32;
    const long long ldz = (long long)L + ms;
    const size_t a = elt(ad);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int nl = 0;
    StageClock clk{c, s};
    const bool use_tc = qbh::tc_enabled(c->tc);
    const float* logits = logits_in ? logits_in : c->logits;
    const int tpw = qbh::route_tokens_per_warp(T);
    const int tile_rows = use_tc ? qbh::tc_token_tile(c->tc, T) : qbh::kSimtBM;
    const size_t routes = (size_t)T * k;
    const int max_tiles = (int)((routes + tile_rows - 1) / tile_rows) + n;
    bool gathered = false;   // expert gate/up gathers h rows by route: no expert-ordered copy
    if (use_tc) {
        if ((rc = qbh::tc_prepare_xside(c->tc, T, x, logits_in == nullptr, c->logits, c->h, c->zcat, ldz,
                                        c->status)) ||
            (rc = qbh::tc_prepare_gate_up(c->tc, T, c->h_perm, c->offsets, c->tile_off_simt, c->act, c->status,
                                          c->h, c->perm, &gathered)) ||
            (rc = qbh::tc_prepare_down(c->tc, T, c->act, c->offsets, c->tile_off_simt, c->e, c->status)) ||
            (rc = qbh::tc_prepare_up_shared(c->tc, T, c->zcat, ldz, out, c->status)))
            return rc;
    }

    // ---- launches (a failure from here on may leave outputs partly written)
    // 1. router logits x W_r^T + o (tensor-core path: fused with the other
    //    x-side GEMMs), unless the caller gives them
    if (use_tc) {
        clk.mark("xside_gemm");
        rc = qbh::tc_launch(c->tc, qbh::TC_XSIDE, s, &nl);
    } else if (!logits_in) {
        clk.mark("router");
        qbh::GemmArgs ga;
        ga.A = x; ga.lda = d; ga.rows = T; ga.K1 = d; ga.W1 = c->w.w_router; ga.F = n;
        ga.out = c->logits; ga.ldo = n; ga.col_bias = c->w.router_offset;
        rc = qbh::launch_gemm_simt(ad, dense_wf, qbh::EPI_ROUTER, ga, s, &nl);
    }
    if (rc) return rc;

    // 2-3. scores (in the first QB token pass), QB sweeps and biased top-k
    clk.mark("qb_topk");
    if (g.qb_mode == QBMOE_QB_GAUSS_SEIDEL)
        rc = qbh::launch_qb_gs(T, n, k, g.qb_sweeps, 0, logits, c->scores, bias_in, bias_out, c->idx, c->wts,
                               c->loads, nullptr, c->rb, c->gb, s, &nl);
    else
        rc = qbh::launch_qb_and_topk(T, n, k, g.qb_sweeps, logits, c->scores, bias_in, bias_out, c->idx, c->wts,
                                     c->rb.blk_cnt, c->rb, s, &nl);
    if (rc) return rc;

    // 4. dispatch: loads, offsets, stable permutation
    clk.mark("dispatch");
    if ((rc = qbh::launch_loads_from_counts(T, n, tpw, c->rb.blk_cnt, c->loads, s, &nl))) return rc;
    if ((rc = qbh::launch_expert_offsets(n, c->loads, c->offsets, tile_rows, c->tile_off_simt, s, &nl))) return rc;
    if ((rc = qbh::launch_scatter(T, n, k, tpw, c->idx, c->rb.blk_cnt, c->offsets, c->perm, c->route_pos, s, &nl)))
        return rc;

    if (use_tc) {
        // h rows are bf16, or E4M3 rows with block scales for block-scaled experts
        const int h_row = qbh::tc_mx_scaled(c->tc) ? (int)qbh::mx_row_bytes(L) : 2 * L;
        if (!gathered && (rc = qbh::launch_scatter_rows(c->h, h_row, c->route_pos, T, k, c->h_perm, s, &nl)))
            return rc;
        clk.mark("expert_gate_up");
        if ((rc = qbh::tc_launch(c->tc, qbh::TC_GATE_UP, s, &nl))) return rc;
        clk.mark("expert_down");
        if ((rc = qbh::tc_launch(c->tc, qbh::TC_DOWN, s, &nl))) return rc;
    } else {
        // 5. latent down-projection h = x W_down^T
        clk.mark("down_proj");
        {
            qbh::GemmArgs ga;
            ga.A = x; ga.lda = d; ga.rows = T; ga.K1 = d; ga.W1 = c->w.w_down; ga.F = L;
            ga.out = c->h; ga.ldo = L;
            if ((rc = qbh::launch_gemm_simt(ad, dense_wf, qbh::EPI_STORE, ga, s, &nl))) return rc;
        }
        // 5b. shared expert gate/up at full width -> act_s (right half of zcat)
        if (ms > 0) {
            clk.mark("shared_gate_up");
            qbh::GemmArgs ga;
            ga.A = x; ga.lda = d; ga.rows = T; ga.K1 = d; ga.W1 = c->w.w_shared_gate; ga.Wu = c->w.w_shared_up;
            ga.F = ms; ga.out = static_cast<char*>(c->zcat) + (size_t)L * a; ga.ldo = ldz;
            ga.beta1 = g.situ_beta1; ga.beta2 = g.situ_beta2;
            if ((rc = qbh::launch_gemm_simt(ad, dense_wf, qbh::EPI_SITU, ga, s, &nl))) return rc;
        }
        // 6. expert gate/up with SiTU-GLU, rows gathered through perm
        clk.mark("expert_gate_up");
        {
            qbh::GemmArgs ga;
            ga.A = c->h; ga.lda = L; ga.a_rows = c->perm; ga.K1 = L; ga.W1 = c->w.w_gate; ga.S1 = c->w.s_gate;
            ga.Wu = c->w.w_up; ga.Su = c->w.s_up; ga.F = m; ga.seg_off = c->offsets; ga.tile_off = c->tile_off_simt;
            ga.n_groups = n; ga.max_tiles = max_tiles; ga.out = c->act; ga.ldo = m;
            ga.beta1 = g.situ_beta1; ga.beta2 = g.situ_beta2;
            if ((rc = qbh::launch_gemm_simt(ad, g.expert_wfmt, qbh::EPI_SITU, ga, s, &nl))) return rc;
        }
        // 7. expert down e = act W_o^T
        clk.mark("expert_down");
        {
            qbh::GemmArgs ga;
            ga.A = c->act; ga.lda = m; ga.K1 = m; ga.W1 = c->w.w_out; ga.S1 = c->w.s_out; ga.F = L;
            ga.seg_off = c->offsets; ga.tile_off = c->tile_off_simt; ga.n_groups = n; ga.max_tiles = max_tiles;
            ga.out = c->e; ga.ldo = L;
            if ((rc = qbh::launch_gemm_simt(ad, g.expert_wfmt, qbh::EPI_STORE, ga, s, &nl))) return rc;
        }
    }
    // 8. combine + RMSNorm -> z (left part of zcat)
    clk.mark("combine_rmsnorm");
    rc = qbh::launch_combine_rmsnorm(ad, T, k, L, c->e, c->wts, c->route_pos, c->w.rms_gamma, g.rms_eps, c->zcat,
                                     ldz, s, &nl);
    if (rc) return rc;
    // 9. out = [z | act_s] [W_proj_up | W_shared_out]^T
    clk.mark("up_proj_shared");
    if (use_tc) {
        rc = qbh::tc_launch(c->tc, qbh::TC_UP_SHARED, s, &nl);
    } else {
        qbh::GemmArgs ga;
        ga.A = c->zcat; ga.lda = ldz; ga.rows = T; ga.K1 = L; ga.W1 = c->w.w_proj_up; ga.K2 = ms;
        ga.W2 = c->w.w_shared_out; ga.F = d; ga.out = out; ga.ldo = d;
        rc = qbh::launch_gemm_simt(ad, dense_wf, qbh::EPI_STORE, ga, s, &nl);
    }
    if (rc) return rc;
    clk.end();
    // optional outputs
    auto cp = [&](void* dst, const void* src, size_t bytes) {
        if (!dst) return true;
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
    };
    if (!cp(scores_opt, c->scores, (size_t)T * n * 4) || !cp(idx_opt, c->idx, routes * 4) ||
        !cp(w_opt, c->wts, routes * 4) || !cp(loads_opt, c->loads, (size_t)n * 4))
        return QBMOE_ECUDA;
    c->launches = nl;
    return QBMOE_OK;
}
