// Tensor-core GEMMs of the layer on sm_103a: TMA -> SMEM (128-byte swizzle)
// -> tcgen05.mma (bf16, fp32 accumulator in TMEM) -> tcgen05.ld epilogue.
//
// [K3-width] = "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club).
// The contractions are the layer's: full-width router (Q&A on routing), the
// latent down-projection (延伸解读 "half-width latent space"), the per-expert
// SiTU-GLU experts in latent space (Q&A on SiTU-GLU), the up-projection and
// the merged shared expert (Q&A on the shared expert).
//
// Orientation: every GEMM is out[t, f] = sum_k W[f, k] X[t, k] with the
// weights as the MMA's A operand (M = 128 weight rows) and the tokens as its
// B operand (N = 16..256 token rows), so a decode step with ~5 tokens per
// expert still issues full-height MMAs while streaming the weights.
//
// One persistent, warp-specialised kernel (192 threads, one CTA per SM):
//   warp 0      TMA producer (one lane): A (weights) and B (tokens) tiles
//               into a STAGES-deep ring, mbarrier complete_tx
//   warp 1      TMEM owner and MMA issuer (one lane): 4 x (128 x N x 16)
//               MMAs per 64-wide K block, commit frees the stage; a tile's
//               last commit hands the accumulator to the epilogue
//   warps 2-5   epilogue: tcgen05.ld 32 lanes x 16 columns, stage through
//               SMEM, epilogue math, 16-byte stores
// Two TMEM accumulators alternate so a tile's epilogue overlaps the next
// tile's main loop.  Every mbarrier wait is bounded: on expiry the kernel
// records QBMOE_ETIMEOUT, stops, drains its own TMA/MMA work (bounded) and
// frees TMEM.
//
// Epilogues per sub-GEMM: STORE (bf16), ROUTER (fp32 score of logit + offset)
// and SITU (A tile = 64 gate rows over 64 up rows of the same features;
// act = SiTU-GLU(gate, up)).
#include "gemm_tc.cuh"
#include "dispatch.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace {

using namespace qb;

constexpr int kProdAWarp = 0, kProdBWarp = 1, kMmaWarp = 2, kEpiFirstWarp = 3;
constexpr int kThreads = (kEpiFirstWarp + 4) * 32;   // 224
constexpr int kBK = 64;                        // K elements per block (128 bytes of bf16)
constexpr int kATileBytes = 128 * kBK * 2;     // 16 KB
constexpr int kMaxSub = 3;
constexpr int kStLd = 17;                      // epilogue staging row stride (floats)
constexpr long long kDefaultWait = 1LL << 17;  // polls (<= 20 us each) before a wait expires

enum { SUB_STORE = 0, SUB_ROUTER = 1, SUB_SITU = 2 };

struct SubGemm {
    int epi;
    int F;              // output features (rows of W per group)
    int m_tiles;        // tiles over F (128 rows, or 64 features for SITU)
    int m_begin;        // first global m index of this sub-GEMM
    int k_split;        // K blocks read from a0; the rest from a1 (ignored for SITU)
    int pad;
    void* out;
    long long ldo;
    const float* col_bias;
};

struct TcParams {
    CUtensorMap a0[kMaxSub];
    CUtensorMap a1[kMaxSub];
    CUtensorMap bx[5];  // activations, boxes {64, 16 << i} rows, i = 0..4 (16..256)
    SubGemm sub[kMaxSub];
    int n_sub;
    int m_total;
    int nkb;            // K blocks
    int rows;           // dense: token rows
    int n_groups;       // grouped: experts; 0 = dense
    int raster_g;       // dense: m-tiles per raster group
    const int* seg_off;
    const int* tile_off;
    float beta1, beta2;
    int* status;
    long long wait_limit;
    int stall_first_tile;   // test hook: withhold the first accumulator hand-off
};

struct TileInfo {
    int sub, mt, g, row0, nrows;
};

// Tile -> (sub-GEMM, m-tile, expert, token rows).  Grouped launches read the
// expert offsets from the CTA's shared-memory copy (s_toff, s_seg).
template <int BN>
__device__ __forceinline__ void decode_tile(const TcParams& p, int tile, int n_tiles_dense, const int* s_toff,
                                            const int* s_seg, TileInfo& ti) {
    int m;
    if (p.n_groups > 0) {
        const int ntg = tile / p.m_total;
        m = tile - ntg * p.m_total;
        int lo = 0, hi = p.n_groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_toff[mid] <= ntg) lo = mid; else hi = mid - 1;
        }
        ti.g = lo;
        // The expert's rows are split into equal tiles (multiples of 16 rows),
        // so the tiles that share a weight tile run at the same pace.
        const int nt = ntg - s_toff[lo];
        const int ntiles = s_toff[lo + 1] - s_toff[lo];
        const int seg0 = s_seg[lo], seg1 = s_seg[lo + 1];
        const int per = (((seg1 - seg0 + ntiles - 1) / ntiles) + 15) & ~15;
        ti.row0 = seg0 + nt * per;
        ti.nrows = min(per, seg1 - ti.row0);
    } else {
        const int G = p.raster_g;
        const int per = G * n_tiles_dense;
        const int grp = tile / per;
        const int rem = tile - grp * per;
        const int gsz = min(G, p.m_total - grp * G);
        const int nt = rem / gsz;
        m = grp * G + (rem - nt * gsz);
        ti.g = 0;
        ti.row0 = nt * BN;
        ti.nrows = min(BN, p.rows - ti.row0);
    }
    int s = 0;
    while (s + 1 < p.n_sub && m >= p.sub[s + 1].m_begin) ++s;
    ti.sub = s;
    ti.mt = m - p.sub[s].m_begin;
}

template <int BN, int SA, int SB>
__global__ void __launch_bounds__(kThreads, 1) k_tc_gemm(const __grid_constant__ TcParams p) {
    constexpr int kBBytes = BN * kBK * 2;
    constexpr uint32_t kCols = (2 * BN <= 32) ? 32 : (2 * BN <= 128 ? 128 : 512);   // two accumulators, power of two
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_ring = smem;                                  // SA x 16 KB weight tiles
    uint8_t* b_ring = smem + SA * kATileBytes;               // SB x BN*128 B token tiles
    uint64_t* fullA = reinterpret_cast<uint64_t*>(b_ring + SB * kBBytes);
    uint64_t* emptyA = fullA + SA;
    uint64_t* fullB = emptyA + SA;
    uint64_t* emptyB = fullB + SB;
    uint64_t* accf = emptyB + SB;
    uint64_t* acce = accf + 2;
    uint64_t* drain = acce + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* st = reinterpret_cast<float*>(tmem_slot + 4);   // [128][kStLd]
    int* s_toff = reinterpret_cast<int*>(st + 128 * kStLd);   // [n_groups + 1] (grouped only)
    int* s_seg = s_toff + (QBMOE_MAX_EXPERTS + 1);            // [n_groups + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit > 0 ? p.wait_limit : kDefaultWait;
    if (p.n_groups > 0) {
        for (int i = threadIdx.x; i <= p.n_groups; i += blockDim.x) {
            s_toff[i] = __ldg(p.tile_off + i);
            s_seg[i] = __ldg(p.seg_off + i);
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            tc::mbar_init(&fullA[s], 1);
            tc::mbar_init(&emptyA[s], 1);
        }
        for (int s = 0; s < SB; ++s) {
            tc::mbar_init(&fullB[s], 1);
            tc::mbar_init(&emptyB[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&accf[a], 1);
            tc::mbar_init(&acce[a], 4);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::fence_proxy_async_smem();
        for (int i = 0; i < 5; ++i) tc::prefetch_tmap(&p.bx[i]);
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, kCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    const int n_tiles_dense = p.n_groups > 0 ? 0 : (p.rows + BN - 1) / BN;
    const int n_tiles = p.n_groups > 0 ? s_toff[p.n_groups] * p.m_total : n_tiles_dense * p.m_total;

    if (warp == kProdAWarp || warp == kProdBWarp) {
        // ------------------------------------------------- producers (one lane each)
        // Warp kProdAWarp streams the weight tiles through the deep A ring,
        // warp kProdBWarp the token tiles through the B ring, so the weight
        // stream can run SA blocks ahead whatever the token-tile size.
        const bool is_a = warp == kProdAWarp;
        const int S = is_a ? SA : SB;
        uint64_t* fullx = is_a ? fullA : fullB;
        uint64_t* emptyx = is_a ? emptyA : emptyB;
        uint32_t issued = 0, last_par = 0;
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                TileInfo ti;
                decode_tile<BN>(p, tile, n_tiles_dense, s_toff, s_seg, ti);
                const SubGemm& sg = p.sub[ti.sub];
                const int n_eff = (ti.nrows + 15) & ~15;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!tc::mbar_wait(&emptyx[s], ph ^ 1u, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                    if (is_a) {
                        uint8_t* A = a_ring + s * kATileBytes;
                        tc::mbar_expect_tx(&fullx[s], kATileBytes);
                        if (sg.epi == SUB_SITU) {
                            const int y = ti.g * sg.F + ti.mt * 64;
                            tc::tma_load_2d(A, &p.a0[ti.sub], &fullx[s], kb * kBK, y);
                            tc::tma_load_2d(A + kATileBytes / 2, &p.a1[ti.sub], &fullx[s], kb * kBK, y);
                        } else {
                            const int y = ti.g * sg.F + ti.mt * 128;
                            if (kb < sg.k_split)
                                tc::tma_load_2d(A, &p.a0[ti.sub], &fullx[s], kb * kBK, y);
                            else
                                tc::tma_load_2d(A, &p.a1[ti.sub], &fullx[s], (kb - sg.k_split) * kBK, y);
                        }
                    } else {
                        uint8_t* B = b_ring + s * kBBytes;
                        tc::mbar_expect_tx(&fullx[s], n_eff * kBK * 2);
                        // n_eff rows as a sum of power-of-two boxes (largest first): <= 5 TMA issues
                        int r = 0;
#pragma unroll
                        for (int i = 4; i >= 0; --i) {
                            const int h = 16 << i;
                            if (h <= BN && (n_eff - r) >= h) {
                                tc::tma_load_2d(B + r * kBK * 2, &p.bx[i], &fullx[s], kb * kBK, ti.row0 + r);
                                r += h;
                            }
                        }
                    }
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
        }
        __syncthreads();
        // drain: every TMA this thread issued has landed before SMEM is released
        if (lane == 0 && *abort_flag) {
            for (int s = 0; s < S; ++s)
                if ((issued >> s) & 1u) tc::mbar_wait(&fullx[s], (last_par >> s) & 1u, kDefaultWait);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int sa = 0, sb = 0;
            uint32_t pha = 0, phb = 0;
            int ab = 0;
            uint32_t aph = 0;
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                TileInfo ti;
                decode_tile<BN>(p, tile, n_tiles_dense, s_toff, s_seg, ti);
                const uint32_t n_eff = (ti.nrows + 15) & ~15;
                const uint32_t idesc = tc::idesc_bf16_m128(n_eff);
                if (!tc::mbar_wait(&acce[ab], aph ^ 1u, lim)) {
                    set_status(p.status, QBMOE_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d = tbase + ab * BN;
                bool ok = true;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!tc::mbar_wait(&fullA[sa], pha, lim) || !tc::mbar_wait(&fullB[sb], phb, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a_addr = tc::smem_u32(a_ring + sa * kATileBytes);
                    const uint32_t b_addr = tc::smem_u32(b_ring + sb * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::tc_mma_bf16(d, tc::desc_sw128(a_addr + kk * 32), tc::desc_sw128(b_addr + kk * 32), idesc,
                                        (kb | kk) != 0);
                    tc::tc_commit(&emptyA[sa]);
                    tc::tc_commit(&emptyB[sb]);
                    if (++sa == SA) { sa = 0; pha ^= 1u; }
                    if (++sb == SB) { sb = 0; phb ^= 1u; }
                }
                if (!ok) break;
                if (!(p.stall_first_tile && tile == (int)blockIdx.x)) tc::tc_commit(&accf[ab]);
                ab ^= 1;
                if (ab == 0) aph ^= 1u;
            }
            // all MMAs issued by this thread complete before TMEM is freed
            tc::tc_commit(drain);
            tc::mbar_wait(drain, 0, kDefaultWait);
        }
        __syncwarp();
        __syncthreads();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int et = threadIdx.x - kEpiFirstWarp * 32;   // 0..127
        int ab = 0;
        uint32_t aph = 0;
        volatile int* ok_slot = abort_flag + 1;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            TileInfo ti;
            decode_tile<BN>(p, tile, n_tiles_dense, s_toff, s_seg, ti);
            const SubGemm& sg = p.sub[ti.sub];
            const int n_eff = (ti.nrows + 15) & ~15;
            // one thread waits; the verdict is shared so the 128 threads stay uniform
            if (et == 0) {
                const bool ok = tc::mbar_wait(&accf[ab], aph, lim);
                if (!ok) {
                    set_status(p.status, QBMOE_ETIMEOUT);
                    *abort_flag = 1;
                }
                *ok_slot = ok ? 1 : 0;
            }
            tc::named_bar_sync(1, 128);
            const bool ok = *ok_slot != 0;
            tc::named_bar_sync(1, 128);
            if (!ok) break;
            tc::tc_fence_after();
            for (int c0 = 0; c0 < n_eff; c0 += 16) {
                float v[16];
                tc::tmem_ld16(tbase + (static_cast<uint32_t>(32 * q) << 16) + ab * BN + c0, v);
                tc::named_bar_sync(1, 128);   // previous chunk's readers are done
#pragma unroll
                for (int j = 0; j < 16; ++j) st[(32 * q + lane) * kStLd + j] = v[j];
                tc::named_bar_sync(1, 128);
                const int tok_left = ti.nrows - c0;
                if (sg.epi == SUB_STORE) {
                    // 16 tokens x 16 groups of 8 features: two items per thread
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
#pragma unroll
                    for (int it = 0; it < 2; ++it) {
                        const int item = et + 128 * it;
                        const int j = item >> 4, fg = item & 15;
                        const int f = ti.mt * 128 + fg * 8;
                        if (j < tok_left && f < sg.F) {
                            __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) o[u] = __float2bfloat16_rn(st[(fg * 8 + u) * kStLd + j]);
                            *reinterpret_cast<uint4*>(out + (long long)(ti.row0 + c0 + j) * sg.ldo + f) =
                                *reinterpret_cast<const uint4*>(o);
                        }
                    }
                } else if (sg.epi == SUB_ROUTER) {
                    // 16 tokens x 32 groups of 4 features (fp32)
                    float* out = static_cast<float*>(sg.out);
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int item = et + 128 * it;
                        const int j = item >> 5, fg = item & 31;
                        const int f = ti.mt * 128 + fg * 4;
                        if (j < tok_left && f < sg.F) {
                            float4 o;
                            float* op = &o.x;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                float lg = st[(fg * 4 + u) * kStLd + j];
                                if (sg.col_bias) lg = __fadd_rn(lg, sg.col_bias[f + u]);
                                op[u] = score_of_logit(lg);
                            }
                            *reinterpret_cast<float4*>(out + (long long)(ti.row0 + c0 + j) * sg.ldo + f) = o;
                        }
                    }
                } else {
                    // SITU: 16 tokens x 8 groups of 8 features, gate rows 0..63, up rows 64..127
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
                    const int j = et >> 3, fg = et & 7;
                    const int f = ti.mt * 64 + fg * 8;
                    if (j < tok_left && f < sg.F) {
                        __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const float g = st[(fg * 8 + u) * kStLd + j];
                            const float up = st[(64 + fg * 8 + u) * kStLd + j];
                            o[u] = __float2bfloat16_rn(situ_glu(g, up, p.beta1, p.beta2));
                        }
                        *reinterpret_cast<uint4*>(out + (long long)(ti.row0 + c0 + j) * sg.ldo + f) =
                            *reinterpret_cast<const uint4*>(o);
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acce[ab]);
            ab ^= 1;
            if (ab == 0) aph ^= 1u;
        }
        __syncthreads();
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, kCols);
    }
}

// ---------------------------------------------------------------------------
// Row gather: dst[r] = src[rows[r]] (16-byte vectors), r < n_rows.
__global__ void k_gather_rows(const uint4* __restrict__ src, int vec_per_row, const int* __restrict__ rows,
                              int n_rows, uint4* __restrict__ dst) {
    const long long total = (long long)n_rows * vec_per_row;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / vec_per_row;
        const int c = (int)(i - r * vec_per_row);
        dst[i] = src[(long long)__ldg(rows + r) * vec_per_row + c];
    }
}

// Ring depths (weight tiles A, token tiles B), chosen by measurement on
// GB300: the token ring must cover its own load latency, the weight ring the
// DRAM latency of the streamed weights.
template <int BN> struct Rings;
template <> struct Rings<16> { static constexpr int SA = 11, SB = 11; };
template <> struct Rings<64> { static constexpr int SA = 9, SB = 7; };
template <> struct Rings<160> { static constexpr int SA = 6, SB = 5; };
template <> struct Rings<256> { static constexpr int SA = 5, SB = 4; };
template <int BN>
constexpr size_t smem_for() {
    return 1024 + (size_t)Rings<BN>::SA * kATileBytes + (size_t)Rings<BN>::SB * BN * kBK * 2 + 512 + 128 * kStLd * 4 +
           2 * (QBMOE_MAX_EXPERTS + 1) * 4;
}

}  // namespace

namespace qbh {

struct TcPlan {
    bool enabled = false;
    qbmoe_config cfg{};
    qbmoe_weights w{};
    bool have_w = false;
    int num_sms = 0;
    long long wait_limit = 0;
    int stall = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous, row stride ld elements), box {64, box_rows}.
bool make_map(TcPlan* P, CUtensorMap* m, const void* base, long long rows, long long cols, long long ld,
              int box_rows) {
    if (!P->encode || rows <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = P->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Token-tile maps with box heights 16, 32, 64, 128, 256 (those above BN unused).
bool make_token_maps(TcPlan* P, TcParams& prm, const void* x, long long rows, long long K, long long ld, int BN) {
    for (int i = 0; i < 5; ++i) {
        const int h = std::min(16 << i, BN);
        if (!make_map(P, &prm.bx[i], x, rows, K, ld, h)) return false;
    }
    return true;
}

template <int BN>
int launch_bn(TcParams& prm, int grid, cudaStream_t s) {
    constexpr size_t smem = smem_for<BN>();
    static_assert(smem <= 232448, "shared memory per CTA");
    auto kern = k_tc_gemm<BN, Rings<BN>::SA, Rings<BN>::SB>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err != cudaSuccess) return QBMOE_ECUDA;
    kern<<<grid, kThreads, smem, s>>>(prm);
    return cuda_err(cudaGetLastError());
}

int launch_any(int BN, TcParams& prm, int grid, cudaStream_t s) {
    switch (BN) {
        case 16: return launch_bn<16>(prm, grid, s);
        case 64: return launch_bn<64>(prm, grid, s);
        case 160: return launch_bn<160>(prm, grid, s);
        case 256: return launch_bn<256>(prm, grid, s);
        default: return QBMOE_EINVAL;
    }
}

void base_params(TcPlan* P, TcParams& prm, int* status) {
    std::memset(&prm, 0, sizeof(prm));
    prm.beta1 = P->cfg.situ_beta1;
    prm.beta2 = P->cfg.situ_beta2;
    prm.status = status;
    prm.wait_limit = P->wait_limit;
    prm.stall_first_tile = P->stall;
}

// Dense launch over T token rows; n_tiles x m_total tiles.
int launch_dense(TcPlan* P, TcParams& prm, int T, const void* x, long long ldx, long long K, cudaStream_t s,
                 int* nl) {
    int BN = 256;
    if ((long long)prm.m_total * ((T + 255) / 256) < 64) BN = T <= 16 ? 16 : 64;
    if (!make_token_maps(P, prm, x, T, K, ldx, BN)) return QBMOE_ECUDA;
    prm.rows = T;
    prm.nkb = (int)((K + kBK - 1) / kBK);
    prm.n_groups = 0;
    prm.raster_g = std::min(prm.m_total, 16);
    const long long tiles = (long long)prm.m_total * ((T + BN - 1) / BN);
    const int grid = (int)std::min<long long>(tiles, P->num_sms);
    if (nl) ++*nl;
    return launch_any(BN, prm, std::max(grid, 1), s);
}

}  // namespace

TcPlan* tc_plan_create(const qbmoe_config& cfg) {
    TcPlan* P = new TcPlan();
    P->cfg = cfg;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, dev);
    P->encode = get_encode();
    const bool shapes_ok = cfg.act_dtype == QBMOE_BF16 && cfg.expert_wfmt == QBMOE_W_BF16 && cfg.d % kBK == 0 &&
                           cfg.latent % kBK == 0 && cfg.expert_inter % kBK == 0 && cfg.shared_inter % kBK == 0 &&
                           cfg.n_experts % 4 == 0 && cfg.latent % 128 == 0 && cfg.d % 128 == 0;
    const char* env = getenv("QBMOE_DISABLE_TC");
    P->enabled = shapes_ok && P->encode != nullptr && !(env && env[0] == '1');
    return P;
}

void tc_plan_destroy(TcPlan* p) { delete p; }

int tc_plan_set_weights(TcPlan* P, const qbmoe_config&, const qbmoe_weights& w) {
    if (!P) return QBMOE_EINVAL;
    P->w = w;
    P->have_w = true;
    return QBMOE_OK;
}

bool tc_enabled(const TcPlan* p) { return p && p->enabled; }

void tc_set_wait_limit(TcPlan* p, long long lim) {
    if (p) p->wait_limit = lim;
}

void tc_set_stall(TcPlan* p, int on) {
    if (p) p->stall = on;
}

int tc_token_tile(const TcPlan* P, int T) {
    // Token rows per grouped tile: each expert's rows are split into equal
    // tiles of at most this many rows (e.g. 293 -> 160 + 133).
    const long long avg = (long long)T * P->cfg.top_k / P->cfg.n_experts;
    return avg <= 16 ? 16 : (avg <= 64 ? 64 : 160);
}

int tc_xside(TcPlan* P, int T, const void* x, bool with_router, float* scores, void* h, void* zcat, long long ldz,
             int* status, cudaStream_t s, int* nl) {
    const qbmoe_config& c = P->cfg;
    TcParams prm;
    base_params(P, prm, status);
    int m = 0, ns = 0;
    if (with_router) {
        SubGemm& r = prm.sub[ns];
        r.epi = SUB_ROUTER; r.F = c.n_experts; r.m_tiles = (c.n_experts + 127) / 128; r.m_begin = m;
        r.k_split = 1 << 30; r.out = scores; r.ldo = c.n_experts; r.col_bias = P->w.router_offset;
        if (!make_map(P, &prm.a0[ns], P->w.w_router, c.n_experts, c.d, c.d, 128)) return QBMOE_ECUDA;
        prm.a1[ns] = prm.a0[ns];
        m += r.m_tiles;
        ++ns;
    }
    {
        SubGemm& g = prm.sub[ns];
        g.epi = SUB_STORE; g.F = c.latent; g.m_tiles = (c.latent + 127) / 128; g.m_begin = m;
        g.k_split = 1 << 30; g.out = h; g.ldo = c.latent;
        if (!make_map(P, &prm.a0[ns], P->w.w_down, c.latent, c.d, c.d, 128)) return QBMOE_ECUDA;
        prm.a1[ns] = prm.a0[ns];
        m += g.m_tiles;
        ++ns;
    }
    if (c.shared_inter > 0) {
        SubGemm& g = prm.sub[ns];
        g.epi = SUB_SITU; g.F = c.shared_inter; g.m_tiles = (c.shared_inter + 63) / 64; g.m_begin = m;
        g.k_split = 1 << 30;
        g.out = static_cast<__nv_bfloat16*>(zcat) + c.latent; g.ldo = ldz;
        if (!make_map(P, &prm.a0[ns], P->w.w_shared_gate, c.shared_inter, c.d, c.d, 64) ||
            !make_map(P, &prm.a1[ns], P->w.w_shared_up, c.shared_inter, c.d, c.d, 64))
            return QBMOE_ECUDA;
        m += g.m_tiles;
        ++ns;
    }
    prm.n_sub = ns;
    prm.m_total = m;
    return launch_dense(P, prm, T, x, c.d, c.d, s, nl);
}

int tc_gather(const void* src, int cols, const int* perm, int n_rows, void* dst, cudaStream_t s, int* nl) {
    const int vpr = cols * 2 / 16;
    const long long total = (long long)n_rows * vpr;
    const int grid = (int)std::min<long long>((total + 255) / 256, 152LL * 8);
    k_gather_rows<<<std::max(grid, 1), 256, 0, s>>>(static_cast<const uint4*>(src), vpr, perm, n_rows,
                                                    static_cast<uint4*>(dst));
    if (nl) ++*nl;
    return cuda_err(cudaGetLastError());
}

static int launch_grouped(TcPlan* P, TcParams& prm, const void* act, long long routes, long long K,
                          const int* offsets, const int* tile_off, int BN, cudaStream_t s, int* nl) {
    if (!make_token_maps(P, prm, act, routes, K, K, BN)) return QBMOE_ECUDA;
    prm.nkb = (int)((K + kBK - 1) / kBK);
    prm.n_groups = P->cfg.n_experts;
    prm.seg_off = offsets;
    prm.tile_off = tile_off;
    prm.rows = 0;
    prm.raster_g = 1;
    if (nl) ++*nl;
    return launch_any(BN, prm, P->num_sms, s);
}

int tc_expert_gate_up(TcPlan* P, int T, const void* h_perm, const int* offsets, const int* tile_off, void* act,
                      int* status, cudaStream_t s, int* nl) {
    const qbmoe_config& c = P->cfg;
    const long long routes = (long long)T * c.top_k;
    TcParams prm;
    base_params(P, prm, status);
    prm.n_sub = 1;
    SubGemm& g = prm.sub[0];
    g.epi = SUB_SITU; g.F = c.expert_inter; g.m_tiles = (c.expert_inter + 63) / 64; g.m_begin = 0;
    g.k_split = 1 << 30; g.out = act; g.ldo = c.expert_inter;
    const long long wrows = (long long)c.n_experts * c.expert_inter;
    if (!make_map(P, &prm.a0[0], P->w.w_gate, wrows, c.latent, c.latent, 64) ||
        !make_map(P, &prm.a1[0], P->w.w_up, wrows, c.latent, c.latent, 64))
        return QBMOE_ECUDA;
    prm.m_total = g.m_tiles;
    return launch_grouped(P, prm, h_perm, routes, c.latent, offsets, tile_off, tc_token_tile(P, T), s, nl);
}

int tc_expert_down(TcPlan* P, int T, const void* act, const int* offsets, const int* tile_off, void* e,
                   int* status, cudaStream_t s, int* nl) {
    const qbmoe_config& c = P->cfg;
    const long long routes = (long long)T * c.top_k;
    TcParams prm;
    base_params(P, prm, status);
    prm.n_sub = 1;
    SubGemm& g = prm.sub[0];
    g.epi = SUB_STORE; g.F = c.latent; g.m_tiles = (c.latent + 127) / 128; g.m_begin = 0;
    g.k_split = 1 << 30; g.out = e; g.ldo = c.latent;
    const long long wrows = (long long)c.n_experts * c.latent;
    if (!make_map(P, &prm.a0[0], P->w.w_out, wrows, c.expert_inter, c.expert_inter, 128)) return QBMOE_ECUDA;
    prm.a1[0] = prm.a0[0];
    prm.m_total = g.m_tiles;
    return launch_grouped(P, prm, act, routes, c.expert_inter, offsets, tile_off, tc_token_tile(P, T), s, nl);
}

int tc_up_shared(TcPlan* P, int T, const void* zcat, long long ldz, void* out, int* status, cudaStream_t s,
                 int* nl) {
    const qbmoe_config& c = P->cfg;
    TcParams prm;
    base_params(P, prm, status);
    prm.n_sub = 1;
    SubGemm& g = prm.sub[0];
    g.epi = SUB_STORE; g.F = c.d; g.m_tiles = (c.d + 127) / 128; g.m_begin = 0;
    g.k_split = c.latent / kBK; g.out = out; g.ldo = c.d;
    if (!make_map(P, &prm.a0[0], P->w.w_proj_up, c.d, c.latent, c.latent, 128)) return QBMOE_ECUDA;
    if (c.shared_inter > 0) {
        if (!make_map(P, &prm.a1[0], P->w.w_shared_out, c.d, c.shared_inter, c.shared_inter, 128))
            return QBMOE_ECUDA;
    } else {
        prm.a1[0] = prm.a0[0];
    }
    prm.m_total = g.m_tiles;
    return launch_dense(P, prm, T, zcat, ldz, (long long)c.latent + c.shared_inter, s, nl);
}

}  // namespace qbh
