// Tensor-core GEMMs of the layer on sm_103a: TMA -> SMEM (128-byte swizzle)
// -> tcgen05.mma (fp32 accumulator in TMEM) -> tcgen05.ld epilogue.
//
// [K3-width] = "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club).
// The contractions are the layer's: full-width router (Q&A on routing), the
// latent down-projection (延伸解读 "half-width latent space"), the per-expert
// SiTU-GLU experts in latent space (Q&A on SiTU-GLU), the up-projection and
// the merged shared expert (Q&A on the shared expert); MXFP4 expert weights
// follow 延伸解读 on deployment (OCP MX: E2M1 codes, an E8M0 scale per 32).
//
// Orientation: every GEMM is out[t, f] = sum_k W[f, k] X[t, k] with the
// weights as the MMA's A operand (M = 128 weight rows) and the tokens as its
// B operand (N = 16..256 token rows), so a decode step with ~5 tokens per
// expert still issues full-height MMAs while streaming the weights.
//
// One persistent, warp-specialised kernel (one CTA per SM):
//   warps 0, 7  weight producers (one lane each; warp 7 takes the odd K
//               blocks): TMA of A tiles into a STAGES-deep ring (and the
//               E8M0 scales for MXFP4)
//   warps 1, 8  token producers (one lane each; or, on 16-row bf16 tiles,
//               the whole warp gathering the tile's rows by route with
//               tile::gather4)
//   warp 2      TMEM owner and MMA issuer (one lane); one commit per stage
//               frees it, a tile's last commit hands the accumulator over
//   warps 3-6   epilogue: tcgen05.ld 32 lanes x 16 columns, stage through
//               SMEM, epilogue math, 16-byte stores
//   warps 7+    MXFP4 decode only (one producer pair): converter warps that
//               decode E2M1 to bf16 in SMEM for the kind::f16 MMA
//   warps 9-12  block-scaled only: scale writers (E8M0 weight and token
//               scale words into TMEM); warps 13-16 a second epilogue group
//   last warp   the MMA issuer's waiter: every mbarrier wait of the issuer,
//               handed over through a named barrier
// Modes: bf16 weights (kind::f16, 4 x K=16 MMAs per 64-wide K stage);
// MXFP4 decoded to bf16; MXFP4 block-scaled (E2M1 unpacked by TMA, tokens
// as exact E4M3 hi/lo pairs with per-32 E8M0 scales stacked in one N = 2n
// MMA, 4 x K=32 MMAs per 128-wide K sub-tile, two sub-tiles per stage on
// 16-row token tiles).
// Two TMEM accumulators alternate so a tile's epilogue overlaps the next
// tile's main loop.  The bf16 gate/up at 160-row token tiles runs units of
// two m-tiles that share each stage's token tile, their accumulators taken
// from a ring of three TMEM slots.  Every mbarrier wait is bounded: on
// expiry the kernel records QBMOE_ETIMEOUT, stops, drains its own TMA/MMA
// work (bounded) and frees TMEM.
//
// Epilogues per sub-GEMM: STORE (bf16), ROUTER (fp32 logit + offset)
// and SITU (A tile = 64 gate rows over 64 up rows of the same features;
// act = SiTU-GLU(gate, up), stored as bf16 or as E4M3 pairs).
#include "gemm_tc.cuh"
#include "dispatch.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace {

using namespace qb;

// (MXFP4-decode mode has one producer pair; its converter warps start at 7.)
constexpr int kProdAWarp = 0, kProdBWarp = 1, kMmaWarp = 2, kEpiFirstWarp = 3, kConvFirstWarp = 7;
// Second producer pair (bf16 and block-scaled modes, and the 2-SM kernel):
// producer pair p issues the weight and token tiles of the K blocks with
// kb % 2 == p, so twice as many threads issue TMA copies.
constexpr int kProdA1Warp = 7, kProdB1Warp = 8;
constexpr int kConvWarps = 8;                          // MXFP4 converter warps (two threads per weight row)
constexpr int kThreadsMx = (kConvFirstWarp + kConvWarps) * 32;  // 480
constexpr int kSfWarps = 4;                            // block-scaled MXFP4: scale writers, one per TMEM lane quarter
constexpr int kSfFirstWarp = kProdB1Warp + 1;          // 9
// block-scaled MXFP4: a second epilogue group (one warp per lane quarter)
// takes every other 16-token chunk of a tile (its stacked hi and lo
// accumulators make the epilogue twice as long per token)
constexpr int kEpi2FirstWarp = kSfFirstWarp + kSfWarps;      // 13
constexpr int kThreadsMxS = (kEpi2FirstWarp + 4) * 32;       // 544
constexpr int kThreadsBf16 = (kProdB1Warp + 1) * 32;   // 288
constexpr int kBKS = 128;                      // block-scaled: K elements per stage (128 bytes of E4M3 per row)
constexpr int kScaleGroupS = 4;                // block-scaled: stages per E8M0 scale load (16 scale bytes per row)
constexpr int kBK = 64;                        // K elements per block (128 bytes of bf16)
constexpr int kATileBytes = 128 * kBK * 2;     // 16 KB
constexpr int kPackBytes = 128 * kBK / 2;              // packed E2M1 bytes of one 128 x 64 weight block
constexpr int kScaleGroup = 8;                         // K blocks per E8M0 scale load (16 scale bytes per row)
constexpr int kScaleBytes = 128 * 2 * kScaleGroup;     // 2 KB
constexpr int kMaxSub = 3;
constexpr int kTokMaps = 16;                   // token-tile heights per launch (see TcParams::bx)
constexpr int kStRow = 132;                    // epilogue staging: 16 token rows of 128 features (+4 pad)
constexpr int kStBytes = 16 * kStRow * 4;
constexpr long long kDefaultWait = 1LL << 17;  // polls (<= 20 us each) before a wait expires
constexpr long long kDrainWait = 1LL << 12;    // polls per stage when draining after an expiry

enum { SUB_STORE = 0, SUB_ROUTER = 1, SUB_SITU = 2 };

// Kernel modes: bf16 weights; MXFP4 weights decoded to bf16 in SMEM by
// converter warps (kind::f16 MMA); MXFP4 weights fed to the block-scaled MMA
// (kind::mxf8f6f4) with E4M3 tokens.
enum { MODE_BF16 = 0, MODE_MX_DECODE = 1, MODE_MX_SCALED = 2 };

// Block-scaled MMAs take fp8 tokens with an E8M0 scale per 32 K elements.
// A token row's bf16 activations are cut into blocks of 32; block b gets the
// scale 2^e_b with e_b = floor(log2 max|a|) - 7, so that every scaled value
// c = a 2^-e_b has |c| < 256, inside E4M3's finite range (448).  c enters as
// two E4M3 terms, c = hi + lo / 16 with hi = e4m3(c) and lo = e4m3(16 (c -
// hi)); the lo rows are stacked under the hi rows in one MMA, both with the
// block's scale, and the epilogue combines the two accumulators as
// hi + lo / 16.  For 2^-6 <= |c| < 256 both terms are exact (a bf16 residual
// has at most four significant bits), so the product is that of the bf16
// activation; smaller values of the block keep an absolute error below
// 2^(e_b - 14).  Nothing saturates.
constexpr int kLoShift = 4;
constexpr int kTokScaleHeadroom = 7;   // e_b = floor(log2 amax) - 7
__device__ __forceinline__ void e4m3_pair(float a, uint8_t& hi, uint8_t& lo) {
    hi = __nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
    const float h = __half2float(__half(__nv_cvt_fp8_to_halfraw(hi, __NV_E4M3)));
    lo = __nv_cvt_float_to_fp8(__fmul_rn(__fsub_rn(a, h), float(1 << kLoShift)), __NV_SATFINITE, __NV_E4M3);
}
// The E8M0 scale of the 32-value block spread over four consecutive lanes
// (8 values each, every lane of the warp calling): x8 is scaled by 2^-e in
// place and e + 127 returned (127, i.e. 2^0, for an all-zero block).  The
// exponent is read from amax's bits: a subnormal amax takes the smallest
// scale, 2^-127.
__device__ __forceinline__ uint8_t mx_block_scale(float (&x8)[8]) {
    float m = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) m = fmaxf(m, fabsf(x8[u]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    int e = 0;
    if (m > 0.f) e = max(((__float_as_int(m) >> 23) & 0xff) - 127 - kTokScaleHeadroom, -127);
    e = min(e, 126);
    const float inv = __int_as_float((127 - e) << 23);   // 2^-e, a normal float for -127 <= e <= 126
#pragma unroll
    for (int u = 0; u < 8; ++u) x8[u] = __fmul_rn(x8[u], inv);
    return static_cast<uint8_t>(e + 127);
}
struct SubGemm {
    int epi;
    int F;              // output features (rows of W per group)
    int m_tiles;        // tiles over F (128 rows, or 64 features for SITU)
    int m_begin;        // first global m index of this sub-GEMM
    int k_split;        // K blocks read from a0; the rest from a1 (ignored for SITU)
    int out_e4m3;       // STORE/SITU output stored as an E4M3 pair (hi bytes at column f, lo at F + f)
    void* out;
    long long ldo;
    const float* col_bias;
};

struct TcParams {
    CUtensorMap a0[kMaxSub];
    CUtensorMap a1[kMaxSub];
    // token rows, one map per tile height: box {64 K, kTokUnit * (i + 1)} rows
    // (one-CTA kernel: 16-row steps up to 256; 2-SM kernel: each CTA's half,
    // 8-row steps up to 128), so that a token tile is one TMA copy
    CUtensorMap bx[kTokMaps];
    CUtensorMap sc0, sc1;   // MXFP4 weights: E8M0 scales of a0 / a1 (box {16, rows})
    CUtensorMap bsc;        // block-scaled: the token rows' E8M0 scales (box {16, BN rows})
    CUtensorMap bg;         // gathered tokens: the unordered token rows, box {64 K, 1 row}
    SubGemm sub[kMaxSub];
    int n_sub;
    int m_total;
    int nkb;            // K blocks
    int rows;           // dense: token rows
    int n_groups;       // grouped: experts; 0 = dense
    int raster_g;       // dense: m-tiles per raster group
    const int* seg_off;
    const int* tile_off;
    // grouped bf16: token row of each route position (the tile's B rows are
    // gathered from bg through it), or NULL (B rows read in order through bx)
    const int* gather_rows;
    float beta1, beta2;
    int* status;
    long long wait_limit;
    int stall_first_tile;   // test hook: withhold the first accumulator hand-off
};

struct TileInfo {
    int sub, mt, g, row0, nrows;
};

// Tile -> (sub-GEMM, m-tile, expert, token rows).  Grouped launches read the
// expert offsets (tile_off, seg_off: a few KB, L1-resident) from global
// memory, which leaves the shared memory to the pipeline stages.
template <int BN>
__device__ __forceinline__ void decode_tile(const TcParams& p, int tile, int n_tiles_dense, TileInfo& ti) {
    const int* __restrict__ s_toff = p.tile_off;
    const int* __restrict__ s_seg = p.seg_off;
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

// Walks a grouped launch's tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// without a division or a search per tile: the (token tile, m-tile) pair
// steps by gridDim.x and the expert of a token tile is found by scanning
// forward from the previous one, since a CTA's tiles only move forward.
// (decode_tile's division and binary search sat on the MMA thread's path
// between tiles.)  Dense launches fall back to decode_tile.
template <int BN>
struct TileWalker {
    int ntg = 0, m = 0, g = 0;
    __device__ __forceinline__ void seek(const TcParams& p) {
        const int* __restrict__ s_toff = p.tile_off;
        while (g + 8 < p.n_groups && __ldg(s_toff + g + 8) <= ntg) g += 8;
        while (g + 1 < p.n_groups && __ldg(s_toff + g + 1) <= ntg) ++g;
    }
    __device__ __forceinline__ void start(const TcParams& p) {
        if (p.n_groups > 0) {
            ntg = blockIdx.x / p.m_total;
            m = blockIdx.x - ntg * p.m_total;
            g = 0;
            seek(p);
        }
    }
    __device__ __forceinline__ void next(const TcParams& p) {
        if (p.n_groups > 0) {
            m += gridDim.x;
            while (m >= p.m_total) { m -= p.m_total; ++ntg; }
            seek(p);
        }
    }
    __device__ __forceinline__ void get(const TcParams& p, int tile, int n_tiles_dense, TileInfo& ti) const {
        if (p.n_groups == 0) {
            decode_tile<BN>(p, tile, n_tiles_dense, ti);
            return;
        }
        // the expert's rows split into equal tiles (multiples of 16 rows), as in decode_tile
        ti.g = g;
        const int t0 = __ldg(p.tile_off + g), t1 = __ldg(p.tile_off + g + 1);
        const int nt = ntg - t0;
        const int ntiles = t1 - t0;
        const int seg0 = __ldg(p.seg_off + g), seg1 = __ldg(p.seg_off + g + 1);
        const int len = seg1 - seg0;
        const int per = ((ntiles == 1 ? len : (len + ntiles - 1) / ntiles) + 15) & ~15;
        ti.row0 = seg0 + nt * per;
        ti.nrows = min(per, seg1 - ti.row0);
        int sb = 0;
        while (sb + 1 < p.n_sub && m >= p.sub[sb + 1].m_begin) ++sb;
        ti.sub = sb;
        ti.mt = m - p.sub[sb].m_begin;
    }
};

// Epilogue of one accumulator tile by the 128 epilogue threads: TMEM lane
// quarter q of this warp, 16-column chunks staged through SMEM, epilogue
// math, 16-byte global stores.  f_base is the output feature of TMEM lane 0;
// tacc the accumulator's TMEM column base.
// SiTU-GLU for the tensor-core epilogues, whose results are stored as bf16
// (or E4M3 pairs of bf16): a = b1 tanh(g / b1), b = b2 tanh(u / b2),
// out = a sigmoid(a) b with sigmoid(a) = (1 + tanh(a / 2)) / 2, the three
// tanh on the hardware approximation (tanh.approx.f32, relative error about
// 2^-11, below the bf16 rounding that follows).
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float situ_glu_hw(float g, float u, float b1, float inv_b1, float b2, float inv_b2) {
    const float a = b1 * tanh_hw(g * inv_b1);
    const float b = b2 * tanh_hw(u * inv_b2);
    return a * fmaf(0.5f, tanh_hw(0.5f * a), 0.5f) * b;
}

// Word i of a 16-byte vector (i a compile-time constant after unrolling).
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One lane's 8 scaled activations (features f .. f + 7 of an E4M3 row of F
// features) as hi and lo bytes; the first lane of a 32-feature block also
// stores the block's scale byte.
__device__ __forceinline__ void store_e4m3_block(uint8_t* row, int F, int f, const float (&c8)[8], uint8_t sc) {
    __align__(8) uint8_t oh[8];
    __align__(8) uint8_t ol[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) e4m3_pair(c8[u], oh[u], ol[u]);
    *reinterpret_cast<uint2*>(row + f) = *reinterpret_cast<const uint2*>(oh);
    *reinterpret_cast<uint2*>(row + F + f) = *reinterpret_cast<const uint2*>(ol);
    if ((f & 31) == 0) row[2 * F + f / 32] = sc;
}

// Eight consecutive staged floats at row + 8 fg as two float4 loads.  The
// threads of a quarter-warp (fg = 0..7 or 8..15) read their two halves in
// alternating order (fg % 8 >= 4 takes the upper half first), so each of the
// two loads covers all 32 banks once instead of half of them twice.
__device__ __forceinline__ void ld_staged8(const float* row, int fg, float (&x8)[8]) {
    const int sw = fg & 4;
    const float4 p0 = *reinterpret_cast<const float4*>(row + fg * 8 + sw);
    const float4 p1 = *reinterpret_cast<const float4*>(row + fg * 8 + (4 - sw));
    const float4 a = sw ? p1 : p0, b = sw ? p0 : p1;
    x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w;
    x8[4] = b.x; x8[5] = b.y; x8[6] = b.z; x8[7] = b.w;
}

// lo_col > 0 (block-scaled, stacked token planes): the accumulator holds
// W * hi in columns [0, n) and W * lo in [lo_col, lo_col + n); the result is
// hi + lo * 2^-kLoShift.
// grp / n_grp: this group's share of the chunks (chunk c of the tile goes to
// group c % n_grp); bar: the group's named barrier; st: its staging buffer.
__device__ __forceinline__ void epilogue_tile(const TcParams& p, const TileInfo& ti, const SubGemm& sg, int f_base,
                                              uint32_t tacc, int lo_col, int q, int lane, int et, float* st,
                                              int grp = 0, int n_grp = 1, int bar = 1) {
    const int n_eff = (ti.nrows + 15) & ~15;
    // Staging: st[j * kStRow + f] holds token j (of a 16-token chunk) of the
    // tile's feature row f.  Each thread writes its feature row's 16 tokens
    // (consecutive lanes, consecutive words: no bank conflict); the stores
    // then read a token's consecutive features as float4 vectors.
    for (int c0 = 16 * grp; c0 < n_eff; c0 += 16 * n_grp) {
        float v[16];
        tc::tmem_ld16(tacc + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
        if (lo_col > 0) {
            float lo[16];
            tc::tmem_ld16(tacc + (static_cast<uint32_t>(32 * q) << 16) + lo_col + c0, lo);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = fmaf(lo[j], 1.0f / float(1 << kLoShift), v[j]);
        }
        tc::named_bar_sync(bar, 128);   // previous chunk's readers are done
#pragma unroll
        for (int j = 0; j < 16; ++j) st[j * kStRow + 32 * q + lane] = v[j];
        tc::named_bar_sync(bar, 128);
        const int tok_left = ti.nrows - c0;
        if (sg.epi == SUB_STORE) {
            // 16 tokens x 16 groups of 8 features: two items per thread
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int item = et + 128 * it;
                const int j = item >> 4, fg = item & 15;
                const int f = f_base + fg * 8;
                const bool ok = j < tok_left && f < sg.F;
                if (sg.out_e4m3) {
                    // E4M3 row: hi plane, lo plane, block scales.  Four consecutive
                    // lanes hold one token's 32-feature block (F % 32 == 0, so they
                    // agree on ok); rows past the tile's end are read but not stored.
                    float x8[8];
                    ld_staged8(st + j * kStRow, fg, x8);
#pragma unroll
                    for (int u = 0; u < 8; ++u) x8[u] = __bfloat162float(__float2bfloat16_rn(x8[u]));
                    const uint8_t sc = mx_block_scale(x8);
                    if (ok) store_e4m3_block(static_cast<uint8_t*>(sg.out) + (long long)(ti.row0 + c0 + j) * sg.ldo,
                                             sg.F, f, x8, sc);
                } else if (ok) {
                    float x8[8];
                    ld_staged8(st + j * kStRow, fg, x8);
                    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) o[u] = __float2bfloat16_rn(x8[u]);
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
                const int f = f_base + fg * 4;
                if (j < tok_left && f < sg.F) {
                    float4 o = *reinterpret_cast<const float4*>(st + j * kStRow + fg * 4);
                    if (sg.col_bias) {
                        // the score is taken from this logit by the QB token pass
                        o.x = __fadd_rn(o.x, sg.col_bias[f + 0]);
                        o.y = __fadd_rn(o.y, sg.col_bias[f + 1]);
                        o.z = __fadd_rn(o.z, sg.col_bias[f + 2]);
                        o.w = __fadd_rn(o.w, sg.col_bias[f + 3]);
                    }
                    *reinterpret_cast<float4*>(out + (long long)(ti.row0 + c0 + j) * sg.ldo + f) = o;
                }
            }
        } else {
            // SITU: 16 tokens x 8 groups of 8 features, gate rows 0..63, up rows 64..127
            const int j = et >> 3, fg = et & 7;
            const int f = f_base + fg * 8;
            const bool ok = j < tok_left && f < sg.F;
            // E4M3 output: every lane takes part in the block-scale exchange
            // (four consecutive lanes hold one 32-feature block)
            if (ok || sg.out_e4m3) {
                const float inv_b1 = 1.0f / p.beta1, inv_b2 = 1.0f / p.beta2;
                const float* row = st + j * kStRow;
                float g8[8], u8[8];
                ld_staged8(row, fg, g8);
                ld_staged8(row + 64, fg, u8);
                float a[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) a[u] = situ_glu_hw(g8[u], u8[u], p.beta1, inv_b1, p.beta2, inv_b2);
                const long long r = (long long)(ti.row0 + c0 + j) * sg.ldo;
                if (sg.out_e4m3) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) a[u] = __bfloat162float(__float2bfloat16_rn(a[u]));
                    const uint8_t sc = mx_block_scale(a);
                    if (ok) store_e4m3_block(static_cast<uint8_t*>(sg.out) + r, sg.F, f, a, sc);
                } else {
                    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) o[u] = __float2bfloat16_rn(a[u]);
                    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(sg.out) + r + f) =
                        *reinterpret_cast<const uint4*>(o);
                }
            }
        }
    }
}

// ---- MXFP4 (OCP MX: E2M1 elements, E8M0 scale per 32) -> bf16 ----------------
// E2M1 magnitude index i = code & 7 has value {0, .5, 1, 1.5, 2, 3, 4, 6}[i].
// Times 2^d its bf16 has exponent field f_i + d with f = {-, 126, 127, 127,
// 128, 128, 129, 129} and mantissa {0, 0, 0, 0x40, 0, 0x40, 0, 0x40}; the
// decode is exact while every field stays in [1, 254] (|d| <= 125).
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
    const uint32_t ex = (code >> 1) & 3u, man = code & 1u;
    const float v = ex == 0u ? 0.5f * (float)man : __int_as_float((int)(ex + 126u) << 23) * (1.0f + 0.5f * (float)man);
    return (code & 8u) ? -v : v;
}

// High and low bytes of the eight magnitudes' bf16 at scale 2^d, packed four
// per register for byte-permute lookups (h[0]/l[0]: indices 0-3, h[1]/l[1]: 4-7).
__device__ __forceinline__ void mx_tables(int d, uint32_t (&h)[2], uint32_t (&l)[2]) {
    const uint32_t a = 126 + d, b = a + 1, c = a + 2, e = a + 3;   // exponent fields
    h[0] = ((a >> 1) << 8) | ((b >> 1) << 16) | ((b >> 1) << 24);
    h[1] = (c >> 1) | ((c >> 1) << 8) | ((e >> 1) << 16) | ((e >> 1) << 24);
    l[0] = ((a & 1u) << 15) | ((b & 1u) << 23) | (((b & 1u) << 31) | (0x40u << 24));
    l[1] = ((c & 1u) << 7) | ((((c & 1u) << 7) | 0x40u) << 8) | ((e & 1u) << 23) | ((((e & 1u) << 7) | 0x40u) << 24);
}

// Eight E2M1 codes of one 32-bit word (code j in bits 4j..4j+3) -> four bf16
// pairs (elements 2q and 2q+1 in o[q]).
__device__ __forceinline__ void mx_decode_word(uint32_t w, const uint32_t (&h)[2], const uint32_t (&l)[2],
                                               uint32_t (&o)[4]) {
    const uint32_t sel0 = w & 0x7777u, sel1 = (w >> 16) & 0x7777u;     // magnitudes of codes 0-3, 4-7
    const uint32_t h0 = __byte_perm(h[0], h[1], sel0), l0 = __byte_perm(l[0], l[1], sel0);
    const uint32_t h1 = __byte_perm(h[0], h[1], sel1), l1 = __byte_perm(l[0], l[1], sel1);
    o[0] = __byte_perm(l0, h0, 0x5140);
    o[1] = __byte_perm(l0, h0, 0x7362);
    o[2] = __byte_perm(l1, h1, 0x5140);
    o[3] = __byte_perm(l1, h1, 0x7362);
    // sign of code 2q is bit 3 of byte q (-> bit 15), of code 2q+1 bit 7 (-> bit 31)
    const uint32_t w4 = w << 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] |= __byte_perm(w, w4, (q << 12) | ((4 + q) << 4)) & 0x80008000u;
}

// Every mode adds one warp after its others: the MMA waiter (see the MMA
// issuer below).
template <int MODE>
constexpr int base_threads_of() {
    return MODE == MODE_MX_DECODE ? kThreadsMx : (MODE == MODE_MX_SCALED ? kThreadsMxS : kThreadsBf16);
}
template <int MODE>
constexpr int threads_of() {
    return base_threads_of<MODE>() + 32;
}
constexpr int kHandoffBar = 2;   // named barrier of the MMA warp and its waiter (64 threads)
constexpr uint32_t pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

// 128-K sub-tiles per stage: two for the block-scaled kernel on 16-row token
// tiles, whose short MMAs (N = 32) leave the per-stage hand-off, commit and
// barrier costs comparable to the MMAs themselves, so a stage carries eight
// MMAs instead of four; one elsewhere.
template <int BN, int MODE>
constexpr int ksub_of() { return MODE == MODE_MX_SCALED && BN == 16 ? 2 : 1; }

template <int BN, int S, int MODE, int MP>
__global__ void __launch_bounds__(threads_of<MODE>(), 1) k_tc_gemm(const __grid_constant__ TcParams p) {
    constexpr bool MX = MODE == MODE_MX_DECODE;    // MXFP4 decoded to bf16 by converter warps
    constexpr bool MXS = MODE == MODE_MX_SCALED;   // MXFP4 on the block-scaled MMA, E4M3 tokens
    constexpr bool kTestFirst = MODE == MODE_BF16;  // waits start with a non-blocking test
    constexpr int kKS = MXS ? kBKS : kBK;          // K elements per stage
    constexpr int kPlane = BN * 128;               // token tile: BN rows of 128 bytes
    constexpr int kBBytes = MXS ? 2 * kPlane : kPlane;   // block-scaled: hi and lo planes
    // Block-scaled: the lo rows of a token tile are stacked under its hi rows
    // so one MMA (N = 2 n) serves both planes; the epilogue adds lo * 2^-4.
    // (The MMA's cost per instruction is mostly reading the weight tile from
    // SMEM, so one N = 2n MMA is much cheaper than two N = n ones.)
    static_assert(!MXS || 2 * BN <= 256, "stacked token planes need N = 2 BN <= 256");
    constexpr int kAccCols = MXS ? 2 * BN : BN;   // TMEM columns per accumulator
    constexpr int kSub = ksub_of<BN, MODE>();     // 128-K sub-tiles per stage
    // MP m-tiles per work unit (bf16): the unit's MP weight tiles share each
    // stage's token tile, so the token rows cross shared memory once per MP
    // MMAs.  Its MP accumulators come from a ring of kSlots TMEM slots (MP = 2:
    // three, so the next unit can start once the epilogue has drained the
    // first accumulator of this one).
    static_assert(MP == 1 || (MODE == MODE_BF16 && 3 * BN <= 512), "paired m-tiles: bf16, three accumulators");
    constexpr int kSlots = MP == 1 ? 2 : 3;
    constexpr int kAStage = kATileBytes * kSub * MP;   // a stage's weight tiles
    constexpr int kBStage = kBBytes * kSub;       // a stage's token tiles
    static_assert(kScaleGroupS % kSub == 0, "whole stages per scale group");
    constexpr int kGrpStages = kScaleGroupS / kSub;   // block-scaled: stages per scale group
    // TMEM columns: two accumulators; block-scaled adds, per stage and 128-K
    // sub-tile, an 8-column token-scale slot (N = 2 BN <= 256 rows) and a
    // 4-column weight-scale slot.
    constexpr int kSfbCol = 2 * kAccCols, kSfaCol = 2 * kAccCols + 8 * kSub * S;
    constexpr uint32_t kCols = MXS ? pow2_cols(kSfaCol + 4 * kSub * S) : pow2_cols(kSlots * BN);
    static_assert(!MXS || kSfaCol + 4 * kSub * S <= 512, "TMEM columns");
    constexpr int kTokScBytes = MXS ? BN * 16 : 0;   // token scales of one scale group (16 per row)
    constexpr bool kScaleAhead = MXS && BN >= 64;     // scale groups issued one group ahead
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // S stages, each a 16 KB weight tile and a BN-row token tile that share
    // one "full" barrier (both producers arrive) and one "empty" barrier (one
    // MMA commit per stage).
    // MXFP4 weights add: a ring of packed E2M1 blocks (S x 4 KB) and two
    // scale slots (2 x 2 KB, 8 K blocks each).
    uint8_t* a_ring = smem;
    uint8_t* b_ring = smem + S * kAStage;
    uint8_t* p_ring = b_ring + S * kBStage;
    uint8_t* sc_ring = p_ring + (MX ? S * kPackBytes : 0);
    uint8_t* tsc_ring = sc_ring + (MX || MXS ? 2 * kScaleBytes : 0);   // block-scaled: 2 token-scale slots
    uint64_t* full = reinterpret_cast<uint64_t*>(tsc_ring + 2 * kTokScBytes);
    uint64_t* empty = full + S;
    uint64_t* fullP = empty + S;                       // MX: packed block landed
    uint64_t* fullS = fullP + (MX ? S : 0);            // MX, MXS: scale group landed
    uint64_t* emptyS = fullS + (MX || MXS ? 2 : 0);    // MX, MXS: scale group consumed
    uint64_t* accf = emptyS + (MX || MXS ? 2 : 0);
    uint64_t* acce = accf + kSlots;
    uint64_t* drain = acce + kSlots;
    // words after the barriers: [0] TMEM base, [1] abort flag, [2, 3] the
    // epilogue groups' per-tile ok words, [4, 5] the MMA issuer's per-tile go/stop
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* go_flag = reinterpret_cast<volatile int*>(tmem_slot + 4);   // [2]: per-tile MMA go/stop
    // [16][kStRow] epilogue staging, read and written as float4: 16-byte aligned
    float* st = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_slot + 6) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit > 0 ? p.wait_limit : kDefaultWait;
    constexpr int kWaitWarp = base_threads_of<MODE>() / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // token producer + weight producer (bf16), + the converter warps
            // (MXFP4 decode) or + the scale writers (block-scaled)
            tc::mbar_init(&full[s], MX ? 1 + kConvWarps : (MXS ? 2 + kSfWarps : 2));
            tc::mbar_init(&empty[s], 1);   // one MMA commit per stage
            if (MX) tc::mbar_init(&fullP[s], 1);
        }
        if (MX || MXS) {
            for (int g = 0; g < 2; ++g) {
                tc::mbar_init(&fullS[g], 1);
                tc::mbar_init(&emptyS[g], MX ? kConvWarps : kSfWarps);
            }
        }
        for (int a = 0; a < kSlots; ++a) {
            tc::mbar_init(&accf[a], 1);
            tc::mbar_init(&acce[a], MXS ? 8 : 4);   // every epilogue warp arrives
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::fence_proxy_async_smem();
        for (int i = 0; i < BN / 16; ++i) tc::prefetch_tmap(&p.bx[i]);
        if (p.gather_rows) tc::prefetch_tmap(&p.bg);
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
    const int n_tiles = p.n_groups > 0 ? __ldg(p.tile_off + p.n_groups) * p.m_total : n_tiles_dense * p.m_total;

    constexpr int kNProd = MX ? 1 : 2;   // producer pairs
    const bool is_prod = warp == kProdAWarp || warp == kProdBWarp ||
                         (kNProd == 2 && (warp == kProdA1Warp || warp == kProdB1Warp));
    if (is_prod) {
        // ------------------------------------------------- producers (one lane each)
        // A weight producer and a token producer per pair load into the same
        // stage in parallel (up to 5 TMA issues each); pair p takes the K
        // blocks with kb % kNProd == p.
        const bool is_a = warp == kProdAWarp || warp == kProdA1Warp;
        const int pair = (warp == kProdAWarp || warp == kProdBWarp) ? 0 : 1;
        uint64_t* fullx = (MX && is_a) ? fullP : full;
        uint32_t issued = 0, last_par = 0;
        uint32_t sc_issued = 0, sc_par = 0;
        int gidx = 0;
        const bool gather_b = MODE == MODE_BF16 && !is_a && p.gather_rows != nullptr;
        if (gather_b) {
            // Token rows gathered by route: the whole warp issues a stage's
            // n_eff / 4 four-row gathers (lane l: rows 4 l .. 4 l + 3 and
            // 4 (l + 32) .. 4 (l + 32) + 3); lane 0 waits and sets the byte
            // count first.  Rows past the tile's routes repeat its last route.
            int s = 0;
            uint32_t ph = 0;
            TileWalker<BN> tw;
            tw.start(p);
            TileInfo tn;
            if ((int)blockIdx.x < n_tiles) tw.get(p, blockIdx.x, n_tiles_dense, tn);
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                const TileInfo ti = tn;
                if (tile + (int)gridDim.x < n_tiles) {
                    tw.next(p);
                    tw.get(p, tile + gridDim.x, n_tiles_dense, tn);
                }
                const int n_eff = (ti.nrows + 15) & ~15;
                int rr[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int r = 4 * (lane + 32 * (j >> 2)) + (j & 3);
                    rr[j] = r < n_eff ? __ldg(p.gather_rows + ti.row0 + min(r, ti.nrows - 1)) : 0;
                }
                bool ok = true;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (kNProd == 2 && (kb & 1) != pair) {   // the other pair's K block
                        if (++s == S) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    int w = 1;
                    if (lane == 0) {
                        w = tc::mbar_wait<kTestFirst>(&empty[s], ph ^ 1u, lim);
                        if (w) {
                            tc::mbar_expect_tx(&full[s], n_eff * 128);
                            issued |= 1u << s;
                            last_par = (last_par & ~(1u << s)) | (ph << s);
                        } else {
                            set_status(p.status, QBMOE_ETIMEOUT);
                            *abort_flag = 1;
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
                    uint8_t* B = b_ring + s * kBBytes;
                    if (4 * lane < n_eff)
                        tc::tma_gather4(B + 512 * lane, &p.bg, &full[s], kb * kBK, rr[0], rr[1], rr[2], rr[3]);
                    if (4 * (lane + 32) < n_eff)
                        tc::tma_gather4(B + 512 * (lane + 32), &p.bg, &full[s], kb * kBK, rr[4], rr[5], rr[6], rr[7]);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
        } else if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            // The walker runs one tile ahead: the next tile's bookkeeping loads
            // are issued while this tile's K blocks go out (and block-scaled
            // kernels issue the next tile's first scale group from it).
            TileWalker<BN> tw;
            tw.start(p);
            TileInfo tn;
            if ((int)blockIdx.x < n_tiles) tw.get(p, blockIdx.x, n_tiles_dense, tn);
            int gstart = 0;   // block-scaled: scale groups begun by this thread
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                const TileInfo ti = tn;
                const bool has_next = tile + (int)gridDim.x < n_tiles;
                if (has_next) {
                    tw.next(p);
                    tw.get(p, tile + gridDim.x, n_tiles_dense, tn);
                }
                const SubGemm& sg = p.sub[ti.sub];
                const int n_eff = (ti.nrows + 15) & ~15;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (kNProd == 2 && (kb & 1) != pair) {   // the other pair's K block
                        if (++s == S) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    if (!tc::mbar_wait<kTestFirst>(&empty[s], ph ^ 1u, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                    if ((MX || MXS) && is_a) {
                        // MX: packed E2M1 block for the converters; MXS: E2M1
                        // tile unpacked by TMA into the stage.  Every sgrp K
                        // blocks also the E8M0 scales (16 bytes per row).
                        const bool situ = sg.epi == SUB_SITU;
                        const int y = ti.g * sg.F + ti.mt * (situ ? 64 : 128);
                        constexpr int sgrp = MX ? kScaleGroup : kGrpStages;   // stages per scale group
                        if (MXS && kb % sgrp == 0) {
                            // Weight and token scales of a group go out one group
                            // ahead (two slots) on prefill-sized tiles, so that the
                            // scale writers find a group's scales landed when its
                            // first stage is due.  (Measured on GB300: 3% faster at
                            // 112-row tiles, 5-7% slower at 16-row decode tiles,
                            // which then issue each group with its first stage.)
                            auto issue_scales = [&](const TileInfo& t, int kbg) -> bool {
                                const SubGemm& gs = p.sub[t.sub];
                                const bool gsitu = gs.epi == SUB_SITU;
                                const int gy = t.g * gs.F + t.mt * (gsitu ? 64 : 128);
                                const int slot = gidx & 1;
                                if (!tc::mbar_wait<kTestFirst>(&emptyS[slot], ((gidx >> 1) & 1) ^ 1u, lim)) return false;
                                uint8_t* SC = sc_ring + slot * kScaleBytes;
                                tc::mbar_expect_tx(&fullS[slot], kScaleBytes + kTokScBytes);
                                const int xs = (kbg / sgrp) * 16;
                                if (gsitu) {
                                    tc::tma_load_2d(SC, &p.sc0, &fullS[slot], xs, gy);
                                    tc::tma_load_2d(SC + kScaleBytes / 2, &p.sc1, &fullS[slot], xs, gy);
                                } else {
                                    tc::tma_load_2d(SC, &p.sc0, &fullS[slot], xs, gy);
                                }
                                tc::tma_load_2d(tsc_ring + slot * kTokScBytes, &p.bsc, &fullS[slot], xs, t.row0);
                                sc_issued |= 1u << slot;
                                sc_par = (sc_par & ~(1u << slot)) | (((gidx >> 1) & 1u) << slot);
                                ++gidx;
                                return true;
                            };
                            bool iss = true;
                            if (gidx == gstart) iss = issue_scales(ti, kb);   // the thread's first group
                            if (kScaleAhead && iss && gidx == gstart + 1) {
                                if (kb + sgrp < p.nkb) iss = issue_scales(ti, kb + sgrp);
                                else if (has_next) iss = issue_scales(tn, 0);
                            }
                            ++gstart;
                            if (!iss) {
                                set_status(p.status, QBMOE_ETIMEOUT);
                                *abort_flag = 1;
                                break;
                            }
                        } else if (MX && kb % sgrp == 0) {
                            const int slot = gidx & 1;
                            if (!tc::mbar_wait<kTestFirst>(&emptyS[slot], ((gidx >> 1) & 1) ^ 1u, lim)) {
                                set_status(p.status, QBMOE_ETIMEOUT);
                                *abort_flag = 1;
                                break;
                            }
                            uint8_t* SC = sc_ring + slot * kScaleBytes;
                            tc::mbar_expect_tx(&fullS[slot], kScaleBytes);
                            const int xs = (kb / sgrp) * 16;
                            if (situ) {
                                tc::tma_load_2d(SC, &p.sc0, &fullS[slot], xs, y);
                                tc::tma_load_2d(SC + kScaleBytes / 2, &p.sc1, &fullS[slot], xs, y);
                            } else {
                                tc::tma_load_2d(SC, &p.sc0, &fullS[slot], xs, y);
                            }
                            sc_issued |= 1u << slot;
                            sc_par = (sc_par & ~(1u << slot)) | (((gidx >> 1) & 1u) << slot);
                            ++gidx;
                        }
                        if (MX) {
                            uint8_t* PK = p_ring + s * kPackBytes;
                            tc::mbar_expect_tx(&fullP[s], kPackBytes);
                            if (situ) {
                                tc::tma_load_2d(PK, &p.a0[ti.sub], &fullP[s], kb * (kBK / 2), y);
                                tc::tma_load_2d(PK + kPackBytes / 2, &p.a1[ti.sub], &fullP[s], kb * (kBK / 2), y);
                            } else {
                                tc::tma_load_2d(PK, &p.a0[ti.sub], &fullP[s], kb * (kBK / 2), y);
                            }
                        } else {
                            // 128 rows x 128 codes, each 16-code chunk landing as 8 bytes + 8 unused;
                            // the transaction counts the 8 KB of packed codes read
                            uint8_t* A = a_ring + s * kAStage;
                            tc::mbar_expect_tx(&full[s], kSub * kATileBytes / 2);
#pragma unroll
                            for (int u = 0; u < kSub; ++u) {
                                const int xk = (kb * kSub + u) * kBKS;
                                uint8_t* Au = A + u * kATileBytes;
                                if (situ) {
                                    tc::tma_load_2d(Au, &p.a0[ti.sub], &full[s], xk, y);
                                    tc::tma_load_2d(Au + kATileBytes / 2, &p.a1[ti.sub], &full[s], xk, y);
                                } else {
                                    tc::tma_load_2d(Au, &p.a0[ti.sub], &full[s], xk, y);
                                }
                            }
                        }
                    } else if (is_a) {
                        uint8_t* A0 = a_ring + s * kAStage;
                        tc::mbar_expect_tx(&fullx[s], kAStage);
#pragma unroll
                        for (int hm = 0; hm < MP; ++hm) {   // the unit's m-tiles
                            uint8_t* A = A0 + hm * kATileBytes;
                            const int mt = ti.mt * MP + hm;
                            if (sg.epi == SUB_SITU) {
                                const int y = ti.g * sg.F + mt * 64;
                                tc::tma_load_2d(A, &p.a0[ti.sub], &fullx[s], kb * kBK, y);
                                tc::tma_load_2d(A + kATileBytes / 2, &p.a1[ti.sub], &fullx[s], kb * kBK, y);
                            } else {
                                const int y = ti.g * sg.F + mt * 128;
                                if (kb < sg.k_split)
                                    tc::tma_load_2d(A, &p.a0[ti.sub], &fullx[s], kb * kBK, y);
                                else
                                    tc::tma_load_2d(A, &p.a1[ti.sub], &fullx[s], (kb - sg.k_split) * kBK, y);
                            }
                        }
                    } else {
                        uint8_t* B = b_ring + s * kBStage;
                        tc::mbar_expect_tx(&fullx[s], (MXS ? 2 : 1) * n_eff * 128 * kSub);
                        // the n_eff token rows as one box per 128-K sub-tile (block-scaled:
                        // hi columns k, lo columns K + k, the lo rows stacked under the hi rows)
                        const CUtensorMap* bmap = &p.bx[(n_eff >> 4) - 1];
#pragma unroll
                        for (int u = 0; u < kSub; ++u) {
                            const int kk128 = kb * kSub + u;
                            tc::tma_load_2d(B + u * kBBytes, bmap, &fullx[s], kk128 * kKS, ti.row0);
                            if (MXS)
                                tc::tma_load_2d(B + u * kBBytes + n_eff * 128, bmap, &fullx[s],
                                                (p.nkb * kSub + kk128) * kKS, ti.row0);
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
                if ((issued >> s) & 1u) tc::mbar_wait<kTestFirst>(&fullx[s], (last_par >> s) & 1u, kDrainWait);
            for (int g = 0; g < 2; ++g)
                if ((sc_issued >> g) & 1u) tc::mbar_wait<kTestFirst>(&fullS[g], (sc_par >> g) & 1u, kDrainWait);
        }
    } else if (MX && warp >= kConvFirstWarp && warp < kConvFirstWarp + kConvWarps) {
        // ------------------------------------------------- MXFP4 converters
        // Two threads per weight row: thread (r, hh) decodes elements
        // 32*hh .. 32*hh+31 of row r of each 128 x 64 block (16 packed bytes,
        // one E8M0 scale) into bf16 in the stage's swizzled A tile.
        const int ct = threadIdx.x - kConvFirstWarp * 32;
        const int r = ct >> 1, hh = ct & 1;
        int s = 0, gidx = 0;
        uint32_t ph = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            bool ok = true;
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int slot = gidx & 1;
                int w = 1;
                if (lane == 0) {
                    if (kb % kScaleGroup == 0) w = tc::mbar_wait<kTestFirst>(&fullS[slot], (gidx >> 1) & 1u, lim);
                    if (w) w = tc::mbar_wait<kTestFirst>(&fullP[s], ph, lim);
                    if (!w) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                    }
                }
                if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
                const uint4 q = *reinterpret_cast<const uint4*>(p_ring + s * kPackBytes + r * (kBK / 2) + hh * 16);
                const int sc = sc_ring[slot * kScaleBytes + r * 16 + (kb % kScaleGroup) * 2 + hh];
                uint8_t* dst = a_ring + s * kATileBytes + r * 128;
                const uint32_t words[4] = {q.x, q.y, q.z, q.w};
                if (sc >= 2 && sc <= 252) {
                    uint32_t th[2], tl[2];
                    mx_tables(sc - 127, th, tl);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int c = hh * 4 + j;
                        uint32_t o[4];
                        mx_decode_word(words[j], th, tl, o);
                        *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else {
                    const float m = __int_as_float(sc == 0 ? 0x00400000 : (sc << 23));   // 2^(sc-127)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int c = hh * 4 + j;
                        uint32_t o[4];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            uint32_t pr = 0;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const float v = e2m1_to_f32((words[j] >> (8 * b + 4 * h)) & 15u) * m;
                                pr |= (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v)) << (16 * h);
                            }
                            o[b] = pr;
                        }
                        *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                tc::fence_proxy_async_smem();   // generic-proxy writes -> tcgen05.mma reads
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&full[s]);
                if (kb % kScaleGroup == kScaleGroup - 1 || kb == p.nkb - 1) {
                    if (lane == 0) tc::mbar_arrive(&emptyS[slot]);
                    ++gidx;
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            const int stop = __shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0);
            if (!ok || stop) break;
        }
        __syncthreads();
    } else if (MXS && warp >= kSfFirstWarp && warp < kSfFirstWarp + kSfWarps) {
        // ------------------------------------------------- scales -> TMEM
        // Warp w writes TMEM lane quarter w % 4 (each quarter holds a full
        // copy).  A stage's scale words (four E8M0 bytes per row, one per
        // 32-wide K slice) go to its slots in the layout the block-scaled MMA
        // reads: lane i column j holds row i + 32 j.  Weights: a 4-column slot
        // for the M = 128 rows.  Tokens: an 8-column slot for the N = 2 n_eff
        // stacked rows, lo row n_eff + r taking hi row r's scale.  A scale
        // group (4 stages) holds 16 bytes per row, one word per stage, so each
        // lane reads its rows' groups once as 16-byte vectors (4 weight rows,
        // 8 stacked token rows) and releases the group's slot right away.
        static_assert(!MXS || kScaleGroupS == 4, "one 16-byte vector per row and scale group");
        const int q = warp & 3;
        const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
        int s = 0, gidx = 0;
        uint32_t ph = 0;
        TileWalker<BN> tw;   // one tile ahead, as in the producers
        tw.start(p);
        TileInfo tn;
        if ((int)blockIdx.x < n_tiles) tw.get(p, blockIdx.x, n_tiles_dense, tn);
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            const int n_eff = (tn.nrows + 15) & ~15;
            if (tile + (int)gridDim.x < n_tiles) {
                tw.next(p);
                tw.get(p, tile + gridDim.x, n_tiles_dense, tn);
            }
            bool ok = true;
            for (int kb0 = 0; kb0 < p.nkb && ok; kb0 += kGrpStages) {
                uint4 wa[4], wt[8];
#pragma unroll
                for (int kq = 0; kq < kGrpStages; ++kq) {
                    int w = 1;
                    if (lane == 0) {
                        if (kq == 0) w = tc::mbar_wait<kTestFirst>(&fullS[gidx & 1], (gidx >> 1) & 1u, lim);
                        // the slots are free once the MMAs of the stage's last use completed
                        if (w) w = tc::mbar_wait<kTestFirst>(&empty[s], ph ^ 1u, lim);
                        if (!w) {
                            set_status(p.status, QBMOE_ETIMEOUT);
                            *abort_flag = 1;
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
                    tc::tc_fence_after();
                    if (kq == 0) {
                        const int slot = gidx & 1;
                        const uint8_t* SC = sc_ring + slot * kScaleBytes;
                        const uint8_t* TS = tsc_ring + slot * kTokScBytes;
#pragma unroll
                        for (int j = 0; j < 4; ++j) wa[j] = *reinterpret_cast<const uint4*>(SC + (lane + 32 * j) * 16);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // stacked row lane + 32 j: hi row n, lo row n - n_eff, or past the rows
                            const int n = lane + 32 * j;
                            const int r = n < n_eff ? n : n - n_eff;
                            wt[j] = r < n_eff ? *reinterpret_cast<const uint4*>(TS + r * 16)
                                              : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
                        }
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&emptyS[slot]);   // the group is in registers
                        ++gidx;
                    }
#pragma unroll
                    for (int u = 0; u < kSub; ++u) {
                        const int wi = kq * kSub + u;   // the sub-tile's word of the group's 16 bytes
                        const uint32_t ca = tbase + lanes + kSfaCol + 4 * (kSub * s + u);
                        const uint32_t cb = tbase + lanes + kSfbCol + 8 * (kSub * s + u);
                        tc::tmem_st4(ca, word_of(wa[0], wi), word_of(wa[1], wi), word_of(wa[2], wi),
                                     word_of(wa[3], wi));
                        tc::tmem_st4(cb, word_of(wt[0], wi), word_of(wt[1], wi), word_of(wt[2], wi),
                                     word_of(wt[3], wi));
                        tc::tmem_st4(cb + 4, word_of(wt[4], wi), word_of(wt[5], wi), word_of(wt[6], wi),
                                     word_of(wt[7], wi));
                    }
                    tc::tmem_wait_st();
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&full[s]);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            const int stop = __shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0);
            if (!ok || stop) break;
        }
        __syncthreads();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 issues the MMAs and never touches an mbarrier itself in the
        // main loop: measured on GB300, an mbarrier wait by the thread that
        // issues tcgen05.mma stalls its MMA stream (45% of the tensor rate at
        // N = 160, even when the barrier has long completed), while a named
        // barrier with a waiter warp that does the mbarrier waits keeps it at
        // 84% (N = 160) to 100% (N = 256).  So the waiter warp below waits
        // for "accumulator free" and "stage landed" and releases this warp
        // through named barrier kHandoffBar; once per tile it also passes the
        // go/stop decision in go_flag.
        int sa = 0;
        int z0 = 0;   // TMEM slot of the unit's first accumulator
        int h = 0;
        TileWalker<BN> tw;
        tw.start(p);
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, tw.next(p)) {
            TileInfo ti;
            tw.get(p, tile, n_tiles_dense, ti);
            const uint32_t n_eff = (ti.nrows + 15) & ~15;
            const uint32_t idesc = tc::idesc_bf16_m128(n_eff);
            tc::named_bar_sync(kHandoffBar, 64);   // the unit's accumulators are free (or stop)
            const bool go = go_flag[h & 1] != 0;
            ++h;
            if (!go) break;
            uint32_t dm[MP];
#pragma unroll
            for (int hm = 0; hm < MP; ++hm) dm[hm] = tbase + ((z0 + hm) % kSlots) * kAccCols;
            const uint32_t d = dm[0];
            // Descriptors step by plain adds: the start-address field holds
            // address / 16, so a 32-byte K step is +2 and a stage is
            // +stage_bytes / 16 (addresses stay below 256 KB, inside the
            // 14-bit field).
            const uint64_t a_desc0 = tc::desc_sw128(tc::smem_u32(a_ring));
            const uint64_t b_desc0 = tc::desc_sw128(tc::smem_u32(b_ring));
            uint32_t id_k[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                id_k[kk] = MXS ? tc::idesc_mx_e2m1_e4m3_m128(2 * n_eff, kk, kk) : idesc;
            for (int kb = 0; kb < p.nkb; ++kb) {
                tc::named_bar_sync(kHandoffBar, 64);   // stage sa has landed
                if (lane == 0) {
                    tc::tc_fence_after();
                    const uint64_t ad = a_desc0 + (uint64_t)(sa * (kAStage >> 4));
                    const uint64_t bd = b_desc0 + (uint64_t)(sa * (kBStage >> 4));
#pragma unroll
                    for (int kk = 0; kk < 4 * kSub; ++kk) {
                        if (MXS) {
                            // 128-K sub-tile u, 32-wide K slice kq (byte kq of the weight and
                            // token scale words) against the stacked hi and lo rows
                            const int u = kk >> 2, kq = kk & 3;
                            const uint32_t sfa = tbase + kSfaCol + 4 * (kSub * sa + u);
                            const uint32_t sfb = tbase + kSfbCol + 8 * (kSub * sa + u);
                            tc::tc_mma_mxf8f6f4(d, ad + (uint64_t)(u * (kATileBytes >> 4)) + 2 * kq,
                                                bd + (uint64_t)(u * (kBBytes >> 4)) + 2 * kq, id_k[kq], sfa, sfb,
                                                (kb | kk) != 0);
                        } else {
#pragma unroll
                            for (int hm = 0; hm < MP; ++hm)
                                tc::tc_mma_bf16(dm[hm], ad + (uint64_t)(hm * (kATileBytes >> 4)) + 2 * kk,
                                                bd + 2 * kk, id_k[kk], (kb | kk) != 0);
                        }
                    }
                    tc::tc_commit(&empty[sa]);
                }
                __syncwarp();
                if (++sa == S) sa = 0;
            }
            if (lane == 0 && !(p.stall_first_tile && tile == (int)blockIdx.x))
#pragma unroll
                for (int hm = 0; hm < MP; ++hm) tc::tc_commit(&accf[(z0 + hm) % kSlots]);
            __syncwarp();
            z0 = (z0 + MP) % kSlots;
        }
        // all MMAs issued by this thread complete before TMEM is freed
        if (lane == 0) {
            tc::tc_commit(drain);
            tc::mbar_wait<kTestFirst>(drain, 0, kDefaultWait);
        }
        __syncwarp();
        __syncthreads();
    } else if (warp == kWaitWarp) {
        // ------------------------------------------------------------ MMA waiter
        // Mirrors the issuer's loop: lane 0 waits (bounded) for the tile's
        // accumulator and for each stage, then the warp meets the issuer at
        // kHandoffBar.  After an expiry or an abort it stops waiting and only
        // releases the issuer, whose MMAs then read stale tiles (outputs are
        // undefined after an expiry), until the next tile boundary stops both.
        int sa = 0;
        uint32_t pha = 0;
        int z0 = 0;
        uint32_t eph = 0;    // per TMEM slot: parity of its releases so far
        int h = 0;
        bool dead = false;   // lane 0: stop waiting
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            if (lane == 0) {
                if (!dead && *abort_flag) dead = true;
#pragma unroll
                for (int hm = 0; hm < MP; ++hm) {
                    const int z = (z0 + hm) % kSlots;
                    if (!dead && !tc::mbar_wait<kTestFirst>(&acce[z], ((eph >> z) & 1u) ^ 1u, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        dead = true;
                    }
                }
                go_flag[h & 1] = dead ? 0 : 1;
            }
#pragma unroll
            for (int hm = 0; hm < MP; ++hm) eph ^= 1u << ((z0 + hm) % kSlots);
            z0 = (z0 + MP) % kSlots;
            __syncwarp();
            tc::named_bar_sync(kHandoffBar, 64);
            const bool go = go_flag[h & 1] != 0;
            ++h;
            if (!go) break;
            for (int kb = 0; kb < p.nkb; ++kb) {
                if (lane == 0) {
                    if (!dead && *abort_flag) dead = true;
                    if (!dead && !tc::mbar_wait<kTestFirst>(&full[sa], pha, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        dead = true;
                    }
                }
                __syncwarp();
                tc::named_bar_sync(kHandoffBar, 64);
                if (++sa == S) { sa = 0; pha ^= 1u; }
            }
        }
        __syncwarp();
        __syncthreads();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter of this warp
        // block-scaled: two groups of four warps (3-6, 13-16), each with its
        // own barrier, ok word and staging buffer
        const int grp = MXS && warp >= kEpi2FirstWarp ? 1 : 0;
        constexpr int kGroups = MXS ? 2 : 1;
        const int bar = grp ? 3 : 1;
        const int et = threadIdx.x - (grp ? kEpi2FirstWarp : kEpiFirstWarp) * 32;   // 0..127
        float* stg = st + grp * (kStBytes / 4);
        int z = 0;           // TMEM slot of the next accumulator
        uint32_t fph = 0;    // per slot: parity of its hand-offs so far
        bool ok = true;
        volatile int* ok_slot = abort_flag + 1 + grp;
        TileWalker<BN> tw;
        tw.start(p);
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, tw.next(p)) {
            TileInfo ti;
            tw.get(p, tile, n_tiles_dense, ti);
            const SubGemm& sg = p.sub[ti.sub];
            for (int hm = 0; hm < MP; ++hm) {   // the unit's accumulators, in hand-off order
                // one thread waits; its result is shared so the 128 threads stay uniform
                if (et == 0) {
                    const bool okw = tc::mbar_wait<kTestFirst>(&accf[z], (fph >> z) & 1u, lim);
                    if (!okw) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                    }
                    *ok_slot = okw ? 1 : 0;
                }
                tc::named_bar_sync(bar, 128);
                ok = *ok_slot != 0;
                tc::named_bar_sync(bar, 128);
                if (!ok) break;
                tc::tc_fence_after();
                const int mt = ti.mt * MP + hm;
                epilogue_tile(p, ti, sg, sg.epi == SUB_SITU ? mt * 64 : mt * 128, tbase + z * kAccCols,
                              MXS ? (ti.nrows + 15) & ~15 : 0, q, lane, et, stg, grp, kGroups, bar);
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&acce[z]);
                fph ^= 1u << z;
                if (++z == kSlots) z = 0;
            }
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
// 2-SM variant for the large (prefill-size) GEMMs: a cluster of two CTAs
// computes a 256-row weight tile x N tokens with tcgen05.mma.cta_group::2.
// Each CTA loads its own 128 weight rows and half of the N token rows, so
// per SM the tile moves 16 KB + N*64 B per K block for twice the MMA work of
// the one-CTA kernel.  The leader CTA (rank 0) issues the MMAs; both CTAs'
// TMA loads complete on the leader's "full" barriers; the MMA commits are
// multicast to both CTAs' "empty" and accumulator-ready barriers; each CTA's
// epilogue drains its own TMEM lanes (weight rows) and arrives on the
// leader's accumulator-free barrier.
template <int BN, int S>
__global__ void __launch_bounds__(kThreadsBf16 + 32, 1) k_tc_gemm2(const __grid_constant__ TcParams p) {
    constexpr int kHalf = BN / 2;                            // token rows per CTA per stage
    constexpr int kBBytes = kHalf * kBK * 2;
    constexpr uint32_t kCols = (2 * BN <= 128) ? 128 : 512;  // two accumulators of BN columns
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_ring = smem;
    uint8_t* b_ring = smem + S * kATileBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(b_ring + S * kBBytes);
    uint64_t* empty = full + S;
    uint64_t* accf = empty + S;
    uint64_t* acce = accf + 2;
    uint64_t* drain = acce + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* go_flag = reinterpret_cast<volatile int*>(tmem_slot + 4);   // [2]: per-tile MMA go/stop
    // [16][kStRow] epilogue staging, read and written as float4: 16-byte aligned
    float* st = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_slot + 6) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWaitWarp = kThreadsBf16 / 32;   // the leader's MMA waiter
    const uint32_t rank = tc::cluster_ctarank();
    const bool leader = rank == 0;
    const long long lim = p.wait_limit > 0 ? p.wait_limit : kDefaultWait;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(&full[s], 2);    // the leader's two producers arrive; both CTAs' copies complete on it
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&accf[a], 1);
            tc::mbar_init(&acce[a], 8);   // 4 epilogue warps in each CTA of the pair
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::fence_proxy_async_smem();
        for (int i = 0; i < kHalf / 8; ++i) tc::prefetch_tmap(&p.bx[i]);
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc_pair(tmem_slot, kCols);
        tc::tmem_relinquish_pair();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();   // both CTAs' barriers are initialised before any cross-CTA signal
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const int n_tiles_dense = p.n_groups > 0 ? 0 : (p.rows + BN - 1) / BN;
    const int n_tiles = p.n_groups > 0 ? __ldg(p.tile_off + p.n_groups) * p.m_total : n_tiles_dense * p.m_total;

    const bool is_prod = warp == kProdAWarp || warp == kProdBWarp || warp == kProdA1Warp || warp == kProdB1Warp;
    if (is_prod) {
        // two producer pairs per CTA, pair p taking the K blocks with kb % 2 == p
        const bool is_a = warp == kProdAWarp || warp == kProdA1Warp;
        const int pair = (warp == kProdAWarp || warp == kProdBWarp) ? 0 : 1;
        uint64_t* fullx = full;
        uint64_t* emptyx = empty;
        uint32_t issued = 0, last_par = 0;
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int tile = cl; tile < n_tiles && !*abort_flag; tile += ncl) {
                TileInfo ti;
                decode_tile<BN>(p, tile, n_tiles_dense, ti);
                const SubGemm& sg = p.sub[ti.sub];
                const int n_eff = (ti.nrows + 15) & ~15;
                const int half = n_eff >> 1;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if ((kb & 1) != pair) {   // the other pair's K block
                        if (++s == S) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    if (!tc::mbar_wait<true>(&emptyx[s], ph ^ 1u, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                    const uint32_t bar = tc::mapa_cluster(&fullx[s], 0);   // the leader's barrier
                    if (is_a) {
                        uint8_t* A = a_ring + s * kATileBytes;
                        if (leader) tc::mbar_expect_tx(&fullx[s], 2 * kATileBytes);
                        if (sg.epi == SUB_SITU) {
                            const int y = ti.g * sg.F + ti.mt * 128 + (int)rank * 64;
                            tc::tma_load_2d_pair(A, &p.a0[ti.sub], bar, kb * kBK, y);
                            tc::tma_load_2d_pair(A + kATileBytes / 2, &p.a1[ti.sub], bar, kb * kBK, y);
                        } else {
                            const int y = ti.g * sg.F + ti.mt * 256 + (int)rank * 128;
                            if (kb < sg.k_split)
                                tc::tma_load_2d_pair(A, &p.a0[ti.sub], bar, kb * kBK, y);
                            else
                                tc::tma_load_2d_pair(A, &p.a1[ti.sub], bar, (kb - sg.k_split) * kBK, y);
                        }
                    } else {
                        uint8_t* B = b_ring + s * kBBytes;
                        if (leader) tc::mbar_expect_tx(&fullx[s], n_eff * kBK * 2);
                        const int row0 = ti.row0 + (int)rank * half;
                        tc::tma_load_2d_pair(B, &p.bx[(half >> 3) - 1], bar, kb * kBK, row0);
                    }
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
        }
        __syncthreads();
        if (lane == 0 && *abort_flag) {
            if (leader) {
                for (int s = 0; s < S; ++s)
                    if ((issued >> s) & 1u) tc::mbar_wait<true>(&fullx[s], (last_par >> s) & 1u, kDrainWait);
            } else {
                // this CTA's copies signal the leader's barriers: give them time to land
                for (int i = 0; i < 200; ++i) __nanosleep(10000);
            }
        }
    } else if (warp == kMmaWarp) {
        // The leader's lane 0 issues the pair's MMAs; as in the one-CTA
        // kernel, a waiter warp does its mbarrier waits and releases it
        // through named barrier kHandoffBar (go/stop once per tile).
        if (leader) {
            int sa = 0;
            int ab = 0;
            int h = 0;
            for (int tile = cl; tile < n_tiles; tile += ncl) {
                TileInfo ti;
                decode_tile<BN>(p, tile, n_tiles_dense, ti);
                const uint32_t n_eff = (ti.nrows + 15) & ~15;
                const uint32_t idesc = tc::idesc_bf16_m256(n_eff);
                tc::named_bar_sync(kHandoffBar, 64);   // accumulator ab is free (or stop)
                const bool go = go_flag[h & 1] != 0;
                ++h;
                if (!go) break;
                const uint32_t d = tbase + ab * BN;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    tc::named_bar_sync(kHandoffBar, 64);   // both CTAs' halves of stage sa have landed
                    if (lane == 0) {
                        tc::tc_fence_after();
                        const uint32_t a_addr = tc::smem_u32(a_ring + sa * kATileBytes);
                        const uint32_t b_addr = tc::smem_u32(b_ring + sa * kBBytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            tc::tc_mma_bf16_pair(d, tc::desc_sw128(a_addr + kk * 32),
                                                 tc::desc_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
                        }
                        tc::tc_commit_pair(&empty[sa], 0x3);
                    }
                    __syncwarp();
                    if (++sa == S) sa = 0;
                }
                if (lane == 0) tc::tc_commit_pair(&accf[ab], 0x3);
                __syncwarp();
                ab ^= 1;
            }
            if (lane == 0) {
                tc::tc_commit_pair(drain, 0x1);
                tc::mbar_wait<true>(drain, 0, kDefaultWait);
            }
        }
        __syncwarp();
        __syncthreads();
    } else if (warp == kWaitWarp) {
        if (leader) {
            int sa = 0;
            uint32_t pha = 0;
            int ab = 0;
            uint32_t aph = 0;
            int h = 0;
            bool dead = false;
            for (int tile = cl; tile < n_tiles; tile += ncl) {
                if (lane == 0) {
                    if (!dead && *abort_flag) dead = true;
                    if (!dead && !tc::mbar_wait<true>(&acce[ab], aph ^ 1u, lim)) {
                        set_status(p.status, QBMOE_ETIMEOUT);
                        *abort_flag = 1;
                        dead = true;
                    }
                    go_flag[h & 1] = dead ? 0 : 1;
                }
                __syncwarp();
                tc::named_bar_sync(kHandoffBar, 64);
                const bool go = go_flag[h & 1] != 0;
                ++h;
                if (!go) break;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (lane == 0) {
                        if (!dead && *abort_flag) dead = true;
                        if (!dead && !tc::mbar_wait<true>(&full[sa], pha, lim)) {
                            set_status(p.status, QBMOE_ETIMEOUT);
                            *abort_flag = 1;
                            dead = true;
                        }
                    }
                    __syncwarp();
                    tc::named_bar_sync(kHandoffBar, 64);
                    if (++sa == S) { sa = 0; pha ^= 1u; }
                }
                ab ^= 1;
                if (ab == 0) aph ^= 1u;
            }
        }
        __syncwarp();
        __syncthreads();
    } else {
        const int q = warp & 3;
        const int et = threadIdx.x - kEpiFirstWarp * 32;
        int ab = 0;
        uint32_t aph = 0;
        volatile int* ok_slot = abort_flag + 1;
        for (int tile = cl; tile < n_tiles; tile += ncl) {
            TileInfo ti;
            decode_tile<BN>(p, tile, n_tiles_dense, ti);
            const SubGemm& sg = p.sub[ti.sub];
            if (et == 0) {
                const bool ok = tc::mbar_wait<true>(&accf[ab], aph, lim);
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
            const int f_base = sg.epi == SUB_SITU ? ti.mt * 128 + (int)rank * 64 : ti.mt * 256 + (int)rank * 128;
            epilogue_tile(p, ti, sg, f_base, tbase + ab * BN, 0, q, lane, et, st);
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) tc::mbar_arrive(&acce[ab]);
                else tc::mbar_arrive_cluster(tc::mapa_cluster(&acce[ab], 0));
            }
            ab ^= 1;
            if (ab == 0) aph ^= 1u;
        }
        __syncthreads();
    }
    __syncthreads();
    tc::tc_fence_before();
    tc::cluster_sync();   // the pair's MMAs and remote signals are done before TMEM and SMEM go
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tbase, kCols);
    }
}

// Pipeline depths (stages of one weight tile + one token tile), chosen by
// measurement on GB300 within the 227 KB of shared memory per CTA.
template <int BN> struct Stages;
template <> struct Stages<16> { static constexpr int S = 12; };
template <> struct Stages<64> { static constexpr int S = 9; };
template <> struct Stages<128> { static constexpr int S = 6; };
template <> struct Stages<160> { static constexpr int S = 6; };
template <> struct Stages<256> { static constexpr int S = 4; };

// 2-SM kernel: per-CTA token stages hold BN/2 rows.
template <int BN> struct Stages2;
template <> struct Stages2<160> { static constexpr int S = 8; };
template <> struct Stages2<256> { static constexpr int S = 6; };
template <int BN>
constexpr size_t smem2_for() {
    return 1024 + (size_t)Stages2<BN>::S * (kATileBytes + (BN / 2) * kBK * 2) + 512 + kStBytes;
}

// MXFP4 weights: each stage also holds a 4 KB packed block.
template <int BN> struct StagesMx;
template <> struct StagesMx<16> { static constexpr int S = 9; };
template <> struct StagesMx<64> { static constexpr int S = 7; };
template <> struct StagesMx<160> { static constexpr int S = 5; };

// Block-scaled MXFP4: stages as for bf16 (a 16 KB E2M1 tile and a token tile
// of BN x 128 E4M3 bytes) plus two 2 KB scale slots.
template <int BN> struct StagesMxS;
template <> struct StagesMxS<16> { static constexpr int S = 5; };   // stages of two 128-K sub-tiles
template <> struct StagesMxS<64> { static constexpr int S = 6; };
template <> struct StagesMxS<112> { static constexpr int S = 4; };

// Paired m-tiles (bf16, 160-row token tiles): two 16 KB weight tiles and one
// token tile per stage.
template <int BN> struct StagesMp2;
template <> struct StagesMp2<160> { static constexpr int S = 4; };

template <int BN, int MODE> struct StagesOf { static constexpr int S = Stages<BN>::S; };
template <int BN> struct StagesOf<BN, MODE_MX_DECODE> { static constexpr int S = StagesMx<BN>::S; };
template <int BN> struct StagesOf<BN, MODE_MX_SCALED> { static constexpr int S = StagesMxS<BN>::S; };

template <int BN, int MODE, int MP = 1>
constexpr int stages_of() {
    if constexpr (MP == 2) return StagesMp2<BN>::S;
    else return StagesOf<BN, MODE>::S;
}

template <int BN, int MODE, int MP = 1>
constexpr size_t smem_for() {
    constexpr int S = stages_of<BN, MODE, MP>();
    constexpr bool MX = MODE == MODE_MX_DECODE, MXS = MODE == MODE_MX_SCALED;
    constexpr int kSub = ksub_of<BN, MODE>();
    return 1024 + (size_t)S * (MP * kSub * kATileBytes + kSub * (MXS ? 2 : 1) * BN * 128 + (MX ? kPackBytes : 0)) +
           (MX || MXS ? 2 * kScaleBytes : 0) + (MXS ? 2 * BN * 16 : 0) + 768 + (MXS ? 2 : 1) * kStBytes;
}

}  // namespace

namespace qbh {

// One prepared launch: parameters with every tensor map encoded, the token
// tile and the kernel variant.  Filled by the tc_prepare_* calls, consumed
// by tc_launch.
struct TcLaunch {
    TcParams prm;
    int BN = 0;
    bool pair = false;
    int mode = MODE_BF16;
    int mp = 1;   // m-tiles per work unit (one-CTA bf16 kernel)
    bool grouped = false;
    long long tiles = 0;
    bool ready = false;
};

struct TcPlan {
    bool enabled = false;
    qbmoe_config cfg{};
    qbmoe_weights w{};
    bool have_w = false;
    int num_sms = 0;
    long long wait_limit = 0;
    int stall = 0;
    bool pair_dense = false;     // dense 256-row launches on the 2-SM kernel (default; QBMOE_DISABLE_2SM=1 turns off)
    bool pair_grouped = false;   // grouped launches on the 2-SM kernel (QBMOE_ENABLE_2SM=1)
    bool mx_scaled = false;  // MXFP4 experts on the block-scaled MMA (else decoded to bf16 in SMEM)
    bool no_gather = false;  // bf16 expert gate/up reads an expert-ordered copy of h (QBMOE_NO_GATHER=1)
    bool no_mpair = false;   // bf16 prefill gate/up on single m-tiles (QBMOE_NO_MPAIR=1)
    int pair_clusters[2] = {0, 0};   // co-resident clusters of the 160 / 256 variants
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    TcLaunch stage[TC_STAGES];       // the forward's launches, prepared before the first one
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

// Token-tile maps with box heights unit, 2 unit, ..., max_rows (one per
// tile height the launch can meet; unit 16 for the one-CTA kernel's tiles,
// 8 for the 2-SM kernel's per-CTA halves).
bool make_token_maps(TcPlan* P, TcParams& prm, const void* x, long long rows, long long K, long long ld, int unit,
                     int max_rows) {
    for (int i = 0; i < kTokMaps && unit * (i + 1) <= max_rows; ++i)
        if (!make_map(P, &prm.bx[i], x, rows, K, ld, unit * (i + 1))) return false;
    return true;
}

// 2-D E4M3 tensor [rows, cols] (row stride ld bytes), box {128, box_rows}, 128-byte swizzle.
bool make_map_e4m3(TcPlan* P, CUtensorMap* m, const void* base, long long rows, long long cols, long long ld,
                   int box_rows) {
    if (!P->encode || rows <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)kBKS, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = P->encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_u8(TcPlan* P, CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_x,
                 int box_rows);

// E4M3 token rows of K activations (mx_row_bytes(K) bytes each): the hi and
// lo planes as one [rows, 2K] map per tile height, and the block scales
// [rows, K/32] (box {16, BN rows}).
bool make_token_maps_e4m3(TcPlan* P, TcParams& prm, const void* x, long long rows, long long K, int BN) {
    const long long ld = mx_row_bytes(K);
    for (int i = 0; i < kTokMaps && 16 * (i + 1) <= BN; ++i)
        if (!make_map_e4m3(P, &prm.bx[i], x, rows, 2 * K, ld, 16 * (i + 1))) return false;
    return make_map_u8(P, &prm.bsc, static_cast<const uint8_t*>(x) + 2 * K, rows, K / 32, ld, 16, BN);
}

// Packed E2M1 weights [rows, K] (K codes per row, two per byte, row stride
// K/2 bytes), box {128 codes, box_rows}: each 16-code chunk lands in SMEM as
// 8 bytes followed by 8 unused bytes, the operand layout of the block-scaled
// MMA, with the 128-byte swizzle.  Needs K % 128 == 0, a row stride that is a
// multiple of 32 bytes and a 32-byte aligned base.
bool make_map_e2m1(TcPlan* P, CUtensorMap* m, const void* base, long long rows, long long K, int box_rows) {
    if (!P->encode || rows <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {(cuuint32_t)kBKS, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = P->encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box,
                           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D uint8 tensor [rows, cols] (row stride ld bytes), box {box_x, box_rows}, no swizzle.
bool make_map_u8(TcPlan* P, CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_x,
                 int box_rows) {
    if (!P->encode || rows <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = P->encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Dynamic shared memory limits are set once per device by
// tc_init_attributes (before any launch of the library on that device).
template <int BN, int MODE, int MP = 1>
int attr_bn() {
    constexpr size_t smem = smem_for<BN, MODE, MP>();
    static_assert(smem <= 232448, "shared memory per CTA");
    return cuda_err(cudaFuncSetAttribute(k_tc_gemm<BN, stages_of<BN, MODE, MP>(), MODE, MP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
}

template <int BN>
int attr_bn2() {
    constexpr size_t smem = smem2_for<BN>();
    static_assert(smem <= 232448, "shared memory per CTA");
    return cuda_err(cudaFuncSetAttribute(k_tc_gemm2<BN, Stages2<BN>::S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem));
}

template <int BN, int MODE, int MP = 1>
int launch_bn(TcParams& prm, int grid, cudaStream_t s) {
    constexpr size_t smem = smem_for<BN, MODE, MP>();
    constexpr int S = stages_of<BN, MODE, MP>();
    k_tc_gemm<BN, S, MODE, MP><<<grid, threads_of<MODE>(), smem, s>>>(prm);
    return cuda_err(cudaGetLastError());
}

// Co-resident clusters of the 2-SM kernel (queried once per plan).
template <int BN>
int pair_occupancy(int num_sms, int* out) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsBf16 + 32, 1, 1);
    cfg.dynamicSmemBytes = smem2_for<BN>();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(num_sms & ~1, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_tc_gemm2<BN, Stages2<BN>::S>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return QBMOE_ECUDA;
    }
    *out = n;
    return QBMOE_OK;
}

template <int BN>
int launch_bn2(TcPlan* P, TcParams& prm, int tiles, cudaStream_t s) {
    constexpr size_t smem = smem2_for<BN>();
    auto kern = k_tc_gemm2<BN, Stages2<BN>::S>;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsBf16 + 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int maxc = P->pair_clusters[BN == 256 ? 1 : 0];
    if (maxc <= 0) return QBMOE_ECUDA;
    const int clusters = std::max(1, std::min(maxc, tiles));
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return QBMOE_ECUDA;
    return cuda_err(cudaGetLastError());
}

int launch_mx_decode(int BN, TcParams& prm, int grid, cudaStream_t s) {
    switch (BN) {
        case 16: return launch_bn<16, MODE_MX_DECODE>(prm, grid, s);
        case 64: return launch_bn<64, MODE_MX_DECODE>(prm, grid, s);
        case 160: return launch_bn<160, MODE_MX_DECODE>(prm, grid, s);
        default: return QBMOE_EINVAL;
    }
}

int launch_mx_scaled(int BN, TcParams& prm, int grid, cudaStream_t s) {
    switch (BN) {
        case 16: return launch_bn<16, MODE_MX_SCALED>(prm, grid, s);
        case 64: return launch_bn<64, MODE_MX_SCALED>(prm, grid, s);
        case 112: return launch_bn<112, MODE_MX_SCALED>(prm, grid, s);
        default: return QBMOE_EINVAL;
    }
}

int launch_any(int BN, TcParams& prm, int grid, cudaStream_t s) {
    switch (BN) {
        case 16: return launch_bn<16, MODE_BF16>(prm, grid, s);
        case 64: return launch_bn<64, MODE_BF16>(prm, grid, s);
        case 128: return launch_bn<128, MODE_BF16>(prm, grid, s);
        case 160: return launch_bn<160, MODE_BF16>(prm, grid, s);
        case 256: return launch_bn<256, MODE_BF16>(prm, grid, s);
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

// Token tile of a dense launch.  With many waves of tiles (prefill) 256 rows
// move the fewest bytes per flop.  Otherwise the launch is a weight stream
// (decode): take the tile that still fits one wave with the most tiles, so
// that as many SMs as possible stream weights.
int dense_bn(long long m_tiles_128, int T, int num_sms) {
    const auto tiles = [&](int bn) { return m_tiles_128 * ((T + bn - 1) / bn); };
    if (tiles(256) >= 2LL * num_sms) return 256;
    int best = 256;
    for (int bn : {128, 64})
        if (tiles(bn) <= num_sms && tiles(bn) > tiles(best)) best = bn;
    if (T <= 16) return 16;
    return best;
}

// Whether a launch with token tile BN runs on the 2-SM kernel.
bool use_pair(const TcPlan* P, int BN, bool grouped) {
    return grouped ? P->pair_grouped && (BN == 256 || BN == 160) : P->pair_dense && BN == 256;
}

// Dense launch over T token rows; n_tiles x m_total tiles.
int prep_dense(TcPlan* P, TcLaunch& L, int BN, bool pair, int T, const void* x, long long ldx, long long K) {
    TcParams& prm = L.prm;
    if (!make_token_maps(P, prm, x, T, K, ldx, pair ? 8 : 16, pair ? BN / 2 : BN)) return QBMOE_ECUDA;
    prm.rows = T;
    prm.nkb = (int)((K + kBK - 1) / kBK);
    prm.n_groups = 0;
    prm.raster_g = std::min(prm.m_total, pair ? 8 : 16);
    L.BN = BN;
    L.pair = pair;
    L.mode = MODE_BF16;
    L.mp = 1;
    L.grouped = false;
    L.tiles = (long long)prm.m_total * ((T + BN - 1) / BN);
    if (pair && BN != 256) return QBMOE_EINVAL;
    L.ready = true;
    return QBMOE_OK;
}

int launch_prepared(TcPlan* P, TcLaunch& L, cudaStream_t s) {
    if (!L.ready) return QBMOE_EINVAL;
    L.ready = false;
    if (!L.grouped) {
        if (L.pair) return launch_bn2<256>(P, L.prm, (int)std::min<long long>(L.tiles, 1 << 30), s);
        const int grid = (int)std::min<long long>(L.tiles, P->num_sms);
        return launch_any(L.BN, L.prm, std::max(grid, 1), s);
    }
    if (L.mode == MODE_MX_SCALED) return launch_mx_scaled(L.BN, L.prm, P->num_sms, s);
    if (L.mode == MODE_MX_DECODE) return launch_mx_decode(L.BN, L.prm, P->num_sms, s);
    if (L.pair)
        return L.BN == 160 ? launch_bn2<160>(P, L.prm, 1 << 30, s) : launch_bn2<256>(P, L.prm, 1 << 30, s);
    if (L.mp == 2) return L.BN == 160 ? launch_bn<160, MODE_BF16, 2>(L.prm, P->num_sms, s) : QBMOE_EINVAL;
    return launch_any(L.BN, L.prm, P->num_sms, s);
}

}  // namespace

TcPlan* tc_plan_create(const qbmoe_config& cfg) {
    TcPlan* P = new TcPlan();
    P->cfg = cfg;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, dev);
    P->encode = get_encode();
    // MXFP4 expert weights: the scale rows (K/32 bytes) must be TMA-aligned (16 B), so K % 512 == 0.
    const bool wfmt_ok = cfg.expert_wfmt == QBMOE_W_BF16 ||
                         (cfg.expert_wfmt == QBMOE_W_MXFP4 && cfg.latent % 512 == 0 && cfg.expert_inter % 512 == 0);
    const bool shapes_ok = cfg.act_dtype == QBMOE_BF16 && wfmt_ok && cfg.d % kBK == 0 &&
                           cfg.latent % kBK == 0 && cfg.expert_inter % kBK == 0 && cfg.shared_inter % kBK == 0 &&
                           cfg.n_experts % 4 == 0 && cfg.latent % 128 == 0 && cfg.d % 128 == 0;
    const char* env = getenv("QBMOE_DISABLE_TC");
    P->enabled = shapes_ok && P->encode != nullptr && !(env && env[0] == '1');
    // Measured on GB300 at the prefill shape: the 2-SM kernel runs the dense
    // 256-row GEMMs 7-13% faster than the one-CTA kernel (each SM stages half
    // the token tile) and the grouped expert GEMMs no faster, so dense
    // launches use it by default and grouped ones only on request.
    const char* env2 = getenv("QBMOE_ENABLE_2SM");
    const char* env4 = getenv("QBMOE_DISABLE_2SM");
    P->pair_grouped = env2 && env2[0] == '1';
    P->pair_dense = !(env4 && env4[0] == '1');
    // MXFP4 experts use the block-scaled MMA unless QBMOE_MX_DECODE=1 asks for
    // the in-SMEM decode to bf16.
    const char* env3 = getenv("QBMOE_MX_DECODE");
    P->mx_scaled = cfg.expert_wfmt == QBMOE_W_MXFP4 && !(env3 && env3[0] == '1');
    // bf16 expert gate/up gathers its token rows by route with TMA (no
    // expert-ordered copy of h) unless QBMOE_NO_GATHER=1 asks for the copy.
    const char* env5 = getenv("QBMOE_NO_GATHER");
    P->no_gather = env5 && env5[0] == '1';
    const char* env6 = getenv("QBMOE_NO_MPAIR");
    P->no_mpair = env6 && env6[0] == '1';
    if (P->enabled && (pair_occupancy<160>(P->num_sms, &P->pair_clusters[0]) ||
                       pair_occupancy<256>(P->num_sms, &P->pair_clusters[1]))) {
        // the 2-SM kernel cannot be placed: run everything on the one-CTA kernel
        P->pair_dense = P->pair_grouped = false;
    }
    return P;
}

int tc_init_attributes() {
    int rc;
    if ((rc = attr_bn<16, MODE_BF16>()) || (rc = attr_bn<64, MODE_BF16>()) || (rc = attr_bn<128, MODE_BF16>()) ||
        (rc = attr_bn<160, MODE_BF16>()) || (rc = attr_bn<256, MODE_BF16>()) || (rc = attr_bn<160, MODE_BF16, 2>()) ||
        (rc = attr_bn<16, MODE_MX_DECODE>()) || (rc = attr_bn<64, MODE_MX_DECODE>()) ||
        (rc = attr_bn<160, MODE_MX_DECODE>()) || (rc = attr_bn<16, MODE_MX_SCALED>()) ||
        (rc = attr_bn<64, MODE_MX_SCALED>()) || (rc = attr_bn<112, MODE_MX_SCALED>()) ||
        (rc = attr_bn2<160>()) || (rc = attr_bn2<256>()))
        return rc;
    return QBMOE_OK;
}

void tc_plan_destroy(TcPlan* p) { delete p; }

int tc_plan_set_weights(TcPlan* P, const qbmoe_config&, const qbmoe_weights& w) {
    if (!P) return QBMOE_EINVAL;
    P->w = w;
    P->have_w = true;
    return QBMOE_OK;
}

bool tc_enabled(const TcPlan* p) { return p && p->enabled; }

bool tc_mx_scaled(const TcPlan* p) { return p && p->enabled && p->mx_scaled; }

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
    // the block-scaled MXFP4 kernel stacks two token planes in one MMA
    // (N = 2 x rows <= 256) and keeps two accumulators plus the scale slots
    // in TMEM, so its largest tile is 112 rows
    const int big = tc_mx_scaled(P) ? 112 : 160;
    return avg <= 16 ? 16 : (avg <= 64 ? 64 : big);
}

// m-tiles of a sub-GEMM over F outputs: the one-CTA kernel covers 128 weight
// rows per tile (64 features for SiTU, whose tile stacks gate over up rows),
// the 2-SM kernel twice that.
static int m_tiles_of(int F, bool situ, bool pair) {
    const int rows = (situ ? 64 : 128) * (pair ? 2 : 1);
    return (F + rows - 1) / rows;
}

int tc_prepare_xside(TcPlan* P, int T, const void* x, bool with_router, float* logits, void* h, void* zcat,
                     long long ldz, int* status) {
    const qbmoe_config& c = P->cfg;
    const long long m128 = (with_router ? (c.n_experts + 127) / 128 : 0) + (c.latent + 127) / 128 +
                           (c.shared_inter + 63) / 64;
    const int BN = dense_bn(m128, T, P->num_sms);
    const bool pair = use_pair(P, BN, false);
    TcLaunch& L = P->stage[TC_XSIDE];
    L.ready = false;
    TcParams& prm = L.prm;
    base_params(P, prm, status);
    int m = 0, ns = 0;
    if (with_router) {
        SubGemm& r = prm.sub[ns];
        r.epi = SUB_ROUTER; r.F = c.n_experts; r.m_tiles = m_tiles_of(c.n_experts, false, pair); r.m_begin = m;
        r.k_split = 1 << 30; r.out = logits; r.ldo = c.n_experts; r.col_bias = P->w.router_offset;
        if (!make_map(P, &prm.a0[ns], P->w.w_router, c.n_experts, c.d, c.d, 128)) return QBMOE_ECUDA;
        prm.a1[ns] = prm.a0[ns];
        m += r.m_tiles;
        ++ns;
    }
    {
        SubGemm& g = prm.sub[ns];
        g.epi = SUB_STORE; g.F = c.latent; g.m_tiles = m_tiles_of(c.latent, false, pair); g.m_begin = m;
        g.k_split = 1 << 30; g.out = h; g.ldo = c.latent;
        if (tc_mx_scaled(P)) {
            // block-scaled experts read h as E4M3 rows: converted here once
            // per token, then copied into expert order as plain bytes
            g.out_e4m3 = 1;
            g.ldo = mx_row_bytes(c.latent);
        }
        if (!make_map(P, &prm.a0[ns], P->w.w_down, c.latent, c.d, c.d, 128)) return QBMOE_ECUDA;
        prm.a1[ns] = prm.a0[ns];
        m += g.m_tiles;
        ++ns;
    }
    if (c.shared_inter > 0) {
        SubGemm& g = prm.sub[ns];
        g.epi = SUB_SITU; g.F = c.shared_inter; g.m_tiles = m_tiles_of(c.shared_inter, true, pair); g.m_begin = m;
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
    return prep_dense(P, L, BN, pair, T, x, c.d, c.d);
}

static int prep_grouped(TcPlan* P, TcLaunch& L, bool pair, const void* act, long long routes, long long K,
                        const int* offsets, const int* tile_off, int BN, int mode) {
    TcParams& prm = L.prm;
    if (mode == MODE_MX_SCALED) {
        // E4M3 rows: hi plane, lo plane, block scales
        if (K % 512 != 0) return QBMOE_EINVAL;   // whole scale groups: the scale writers take stage pairs
        if (!make_token_maps_e4m3(P, prm, act, routes, K, BN)) return QBMOE_ECUDA;
        prm.nkb = (int)(K / (kBKS * (BN == 16 ? 2 : 1)));   // stages of ksub_of<BN, MODE_MX_SCALED> sub-tiles
    } else {
        if (!make_token_maps(P, prm, act, routes, K, K, pair ? 8 : 16, pair ? BN / 2 : BN)) return QBMOE_ECUDA;
        prm.nkb = (int)((K + kBK - 1) / kBK);
    }
    prm.n_groups = P->cfg.n_experts;
    prm.seg_off = offsets;
    prm.tile_off = tile_off;
    prm.rows = 0;
    prm.raster_g = 1;
    L.BN = BN;
    L.pair = pair;
    L.mode = mode;
    L.mp = 1;
    L.grouped = true;
    L.tiles = 0;
    if (pair && BN != 160 && BN != 256) return QBMOE_EINVAL;
    L.ready = true;
    return QBMOE_OK;
}

int tc_prepare_gate_up(TcPlan* P, int T, const void* h_perm, const int* offsets, const int* tile_off, void* act,
                       int* status, const void* h, const int* perm, bool* gathered) {
    const qbmoe_config& c = P->cfg;
    const long long routes = (long long)T * c.top_k;
    const int BN = tc_token_tile(P, T);
    const bool mx = c.expert_wfmt == QBMOE_W_MXFP4;
    const bool pair = !mx && use_pair(P, BN, true);
    TcLaunch& L = P->stage[TC_GATE_UP];
    L.ready = false;
    TcParams& prm = L.prm;
    base_params(P, prm, status);
    prm.n_sub = 1;
    SubGemm& g = prm.sub[0];
    g.epi = SUB_SITU; g.F = c.expert_inter; g.m_tiles = m_tiles_of(c.expert_inter, true, pair); g.m_begin = 0;
    g.k_split = 1 << 30; g.out = act; g.ldo = c.expert_inter;
    const long long wrows = (long long)c.n_experts * c.expert_inter;
    const int mode = !mx ? MODE_BF16 : (P->mx_scaled ? MODE_MX_SCALED : MODE_MX_DECODE);
    if (mode == MODE_MX_SCALED) {
        // E2M1 tiles unpacked by TMA (box 128 codes x 64 rows), E8M0 scales
        // [rows, K/32] (box 16 x 64); the output act is E4M3 for the down GEMM
        const long long K = c.latent;
        g.out_e4m3 = 1;
        g.ldo = mx_row_bytes(c.expert_inter);   // act as E4M3 rows for the down GEMM
        if (!make_map_e2m1(P, &prm.a0[0], P->w.w_gate, wrows, K, 64) ||
            !make_map_e2m1(P, &prm.a1[0], P->w.w_up, wrows, K, 64) ||
            !make_map_u8(P, &prm.sc0, P->w.s_gate, wrows, K / 32, K / 32, 16, 64) ||
            !make_map_u8(P, &prm.sc1, P->w.s_up, wrows, K / 32, K / 32, 16, 64))
            return QBMOE_ECUDA;
    } else if (mx) {
        // packed E2M1 [rows, K/2] (box 32 bytes x 64 rows) and E8M0 scales [rows, K/32] (box 16 x 64)
        const long long K = c.latent;
        if (!make_map_u8(P, &prm.a0[0], P->w.w_gate, wrows, K / 2, K / 2, kBK / 2, 64) ||
            !make_map_u8(P, &prm.a1[0], P->w.w_up, wrows, K / 2, K / 2, kBK / 2, 64) ||
            !make_map_u8(P, &prm.sc0, P->w.s_gate, wrows, K / 32, K / 32, 16, 64) ||
            !make_map_u8(P, &prm.sc1, P->w.s_up, wrows, K / 32, K / 32, 16, 64))
            return QBMOE_ECUDA;
    } else if (!make_map(P, &prm.a0[0], P->w.w_gate, wrows, c.latent, c.latent, 64) ||
               !make_map(P, &prm.a1[0], P->w.w_up, wrows, c.latent, c.latent, 64)) {
        return QBMOE_ECUDA;
    }
    prm.m_total = g.m_tiles;
    // bf16 decode-sized tiles (16 rows) on the one-CTA kernel: the token rows
    // are gathered from h through the route order (no expert-ordered copy);
    // else read from h_perm.  Measured on GB300: at decode (T = 256) the
    // gather saves the copy and 1.5% of the gate/up launch; at prefill (160-row
    // tiles, 40 four-row gathers per stage) the gate/up launch took 8.1 ms
    // instead of 3.3 ms, bound by the gather issue rate.
    const bool gather = mode == MODE_BF16 && !pair && BN == 16 && h && perm && !P->no_gather;
    if (gathered) *gathered = gather;
    if (gather) {
        int rc = prep_grouped(P, L, pair, h, T, c.latent, offsets, tile_off, BN, mode);
        if (rc) return rc;
        if (!make_map(P, &prm.bg, h, T, c.latent, c.latent, 1)) return QBMOE_ECUDA;
        prm.gather_rows = perm;
        return QBMOE_OK;
    }
    int rc = prep_grouped(P, L, pair, h_perm, routes, c.latent, offsets, tile_off, BN, mode);
    if (rc) return rc;
    // Prefill-sized bf16 tiles: pairs of m-tiles share each stage's token
    // tile (units of two m-tiles; QBMOE_NO_MPAIR=1 keeps single m-tiles).
    if (mode == MODE_BF16 && !pair && BN == 160 && g.m_tiles % 2 == 0 && !P->no_mpair) {
        L.mp = 2;
        g.m_tiles /= 2;
        prm.m_total = g.m_tiles;
    }
    return QBMOE_OK;
}

int tc_prepare_down(TcPlan* P, int T, const void* act, const int* offsets, const int* tile_off, void* e,
                    int* status) {
    const qbmoe_config& c = P->cfg;
    const long long routes = (long long)T * c.top_k;
    const int BN = tc_token_tile(P, T);
    const bool mx = c.expert_wfmt == QBMOE_W_MXFP4;
    const bool pair = !mx && use_pair(P, BN, true);
    TcLaunch& L = P->stage[TC_DOWN];
    L.ready = false;
    TcParams& prm = L.prm;
    base_params(P, prm, status);
    prm.n_sub = 1;
    SubGemm& g = prm.sub[0];
    g.epi = SUB_STORE; g.F = c.latent; g.m_tiles = m_tiles_of(c.latent, false, pair); g.m_begin = 0;
    g.k_split = 1 << 30; g.out = e; g.ldo = c.latent;
    const long long wrows = (long long)c.n_experts * c.latent;
    const int mode = !mx ? MODE_BF16 : (P->mx_scaled ? MODE_MX_SCALED : MODE_MX_DECODE);
    if (mode == MODE_MX_SCALED) {
        const long long K = c.expert_inter;
        if (!make_map_e2m1(P, &prm.a0[0], P->w.w_out, wrows, K, 128) ||
            !make_map_u8(P, &prm.sc0, P->w.s_out, wrows, K / 32, K / 32, 16, 128))
            return QBMOE_ECUDA;
    } else if (mx) {
        const long long K = c.expert_inter;
        if (!make_map_u8(P, &prm.a0[0], P->w.w_out, wrows, K / 2, K / 2, kBK / 2, 128) ||
            !make_map_u8(P, &prm.sc0, P->w.s_out, wrows, K / 32, K / 32, 16, 128))
            return QBMOE_ECUDA;
    } else if (!make_map(P, &prm.a0[0], P->w.w_out, wrows, c.expert_inter, c.expert_inter, 128)) {
        return QBMOE_ECUDA;
    }
    prm.a1[0] = prm.a0[0];
    prm.m_total = g.m_tiles;
    return prep_grouped(P, L, pair, act, routes, c.expert_inter, offsets, tile_off, BN, mode);
}

int tc_prepare_up_shared(TcPlan* P, int T, const void* zcat, long long ldz, void* out, int* status) {
    const qbmoe_config& c = P->cfg;
    const int BN = dense_bn((c.d + 127) / 128, T, P->num_sms);
    const bool pair = use_pair(P, BN, false);
    TcLaunch& L = P->stage[TC_UP_SHARED];
    L.ready = false;
    TcParams& prm = L.prm;
    base_params(P, prm, status);
    prm.n_sub = 1;
    SubGemm& g = prm.sub[0];
    g.epi = SUB_STORE; g.F = c.d; g.m_tiles = m_tiles_of(c.d, false, pair); g.m_begin = 0;
    g.k_split = c.latent / kBK; g.out = out; g.ldo = c.d;
    if (!make_map(P, &prm.a0[0], P->w.w_proj_up, c.d, c.latent, c.latent, 128)) return QBMOE_ECUDA;
    if (c.shared_inter > 0) {
        if (!make_map(P, &prm.a1[0], P->w.w_shared_out, c.d, c.shared_inter, c.shared_inter, 128))
            return QBMOE_ECUDA;
    } else {
        prm.a1[0] = prm.a0[0];
    }
    prm.m_total = g.m_tiles;
    return prep_dense(P, L, BN, pair, T, zcat, ldz, (long long)c.latent + c.shared_inter);
}

int tc_launch(TcPlan* P, int stage, cudaStream_t s, int* nl) {
    if (!P || stage < 0 || stage >= TC_STAGES) return QBMOE_EINVAL;
    if (nl) ++*nl;
    return launch_prepared(P, P->stage[stage], s);
}

}  // namespace qbh
