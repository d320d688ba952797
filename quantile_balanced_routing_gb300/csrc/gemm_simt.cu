// CUDA-core (FFMA) GEMMs of the layer, dense and grouped by expert.
//
// This is the fp32 path (the tiny fp32 layer: tensor cores would round fp32
// operands to tf32) and the reference-grade path for every format; the
// bf16/MXFP4 hot path is the tcgen05 kernel in gemm_tc.cu.
//
// [K3-width] = "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club).
//   Q&A on SiTU-GLU (epilogue), 延伸解读 "Parameter scale and deployment"
//   (MXFP4 routed-expert weights, decoded here on load).
#include "common.cuh"
#include "dispatch.cuh"

namespace {

using namespace qb;
using qbh::GemmArgs;

constexpr int BM = qbh::kSimtBM, BN = 64, BK = 16;

// E2M1 code -> value (OCP MX): bit 3 sign, bits 2-1 exponent (bias 1), bit 0
// mantissa; exponent 0 is subnormal (0 or 0.5).
QB_DEV float e2m1_value(uint32_t code) {
    const uint32_t ex = (code >> 1) & 3u, man = code & 1u;
    const float v = ex == 0u ? 0.5f * (float)man : __int_as_float((int)(ex + 126u) << 23) * (1.0f + 0.5f * (float)man);
    return (code & 8u) ? -v : v;
}

// E8M0 scale byte -> 2^(s - 127) (s = 255, NaN, is rejected on the host).
QB_DEV float e8m0_scale(uint8_t s) { return s == 0 ? __int_as_float(0x00400000) : __int_as_float((int)s << 23); }

template <int WF>
struct WLoad;
template <>
struct WLoad<QBMOE_W_F32> {
    QB_DEV static float at(const void* W, const uint8_t*, long long expert_base, long long f, int K, int k) {
        return static_cast<const float*>(W)[expert_base + f * K + k];
    }
};
template <>
struct WLoad<QBMOE_W_BF16> {
    QB_DEV static float at(const void* W, const uint8_t*, long long expert_base, long long f, int K, int k) {
        return __bfloat162float(static_cast<const __nv_bfloat16*>(W)[expert_base + f * K + k]);
    }
};
template <>
struct WLoad<QBMOE_W_MXFP4> {
    // expert_base counts elements (F*K per expert).
    QB_DEV static float at(const void* W, const uint8_t* S, long long expert_base, long long f, int K, int k) {
        const long long e = expert_base + f * K + k;
        const uint8_t byte = static_cast<const uint8_t*>(W)[e >> 1];
        const uint32_t code = (e & 1) ? (byte >> 4) : (byte & 15u);
        return e2m1_value(code) * e8m0_scale(S[e >> 5]);
    }
};

template <typename TA, int WF, typename TO, int EPI>
__global__ void __launch_bounds__(256) k_gemm_simt(GemmArgs p) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Ws[BK][BN + 4];
    __shared__ float Us[EPI == qbh::EPI_SITU ? BK : 1][BN + 4];
    const int tid = threadIdx.x;
    int g = 0, row0, nrows;
    if (p.seg_off) {
        const int tile = blockIdx.x;
        if (tile >= p.tile_off[p.n_groups]) return;
        int lo = 0, hi = p.n_groups - 1;   // last g with tile_off[g] <= tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        g = lo;
        row0 = p.seg_off[g] + (tile - p.tile_off[g]) * BM;
        nrows = min(BM, p.seg_off[g + 1] - row0);
    } else {
        row0 = blockIdx.x * BM;
        nrows = min(BM, p.rows - row0);
    }
    if (nrows <= 0) return;
    const int f0 = blockIdx.y * BN;
    const int K = p.K1 + p.K2;
    const long long wbase = (long long)g * p.F * p.K1;
    const TA* A = static_cast<const TA*>(p.A);

    const int tr = tid / 16, tc = tid % 16;   // 16x16 threads, 4x4 outputs each
    float acc[4][4] = {}, accu[4][4] = {};

    // load mapping: 256 threads x 4 elements = 64 x 16 tile
    const int lr = tid / 4, lk = (tid % 4) * 4;
    long long arow = -1;
    if (lr < nrows) arow = p.a_rows ? p.a_rows[row0 + lr] : row0 + lr;
    const long long fl = f0 + lr;

    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = k0 + lk + q;
            float av = 0.0f, wv = 0.0f, uv = 0.0f;
            if (arow >= 0 && k < K) av = to_f32(A[arow * p.lda + k]);
            if (fl < p.F && k < K) {
                if (k < p.K1) {
                    wv = WLoad<WF>::at(p.W1, p.S1, wbase, fl, p.K1, k);
                    if (EPI == qbh::EPI_SITU) uv = WLoad<WF>::at(p.Wu, p.Su, wbase, fl, p.K1, k);
                } else {
                    wv = to_f32(static_cast<const TA*>(p.W2)[fl * p.K2 + (k - p.K1)]);
                }
            }
            As[lk + q][lr] = av;
            Ws[lk + q][lr] = wv;
            if (EPI == qbh::EPI_SITU) Us[lk + q][lr] = uv;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], w[4], u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][tr * 4 + i];
                w[i] = Ws[kk][tc * 4 + i];
                if (EPI == qbh::EPI_SITU) u[i] = Us[kk][tc * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
                    if (EPI == qbh::EPI_SITU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
                }
        }
        __syncthreads();
    }
    TO* out = static_cast<TO*>(p.out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = tr * 4 + i;
        if (r >= nrows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = f0 + tc * 4 + j;
            if (f >= p.F) continue;
            float v;
            if (EPI == qbh::EPI_ROUTER) {
                // router logit + offset; the QB token pass takes the score from it
                v = p.col_bias ? __fadd_rn(acc[i][j], p.col_bias[f]) : acc[i][j];
            } else if (EPI == qbh::EPI_SITU) {
                v = situ_glu(acc[i][j], accu[i][j], p.beta1, p.beta2);
            } else {
                v = acc[i][j];
            }
            out[(long long)(row0 + r) * p.ldo + f] = from_f32<TO>(v);
        }
    }
}

template <typename TA, int WF, typename TO, int EPI>
int go(const GemmArgs& a, cudaStream_t s) {
    const int gx = a.seg_off ? a.max_tiles : (a.rows + BM - 1) / BM;
    const int gy = (a.F + BN - 1) / BN;
    if (gx <= 0 || gy <= 0) return QBMOE_OK;
    k_gemm_simt<TA, WF, TO, EPI><<<dim3(gx, gy), 256, 0, s>>>(a);
    return qbh::cuda_err(cudaGetLastError());
}

}  // namespace

namespace qbh {

int launch_gemm_simt(int act_dtype, int wfmt, GemmEpi epi, const GemmArgs& a, cudaStream_t s, int* nl) {
    int rc = QBMOE_EINVAL;
    using bf = __nv_bfloat16;
    if (act_dtype == QBMOE_F32) {
        if (wfmt != QBMOE_W_F32) return QBMOE_EINVAL;
        if (epi == EPI_STORE) rc = go<float, QBMOE_W_F32, float, EPI_STORE>(a, s);
        else if (epi == EPI_ROUTER) rc = go<float, QBMOE_W_F32, float, EPI_ROUTER>(a, s);
        else rc = go<float, QBMOE_W_F32, float, EPI_SITU>(a, s);
    } else if (act_dtype == QBMOE_BF16) {
        if (wfmt == QBMOE_W_BF16) {
            if (epi == EPI_STORE) rc = go<bf, QBMOE_W_BF16, bf, EPI_STORE>(a, s);
            else if (epi == EPI_ROUTER) rc = go<bf, QBMOE_W_BF16, float, EPI_ROUTER>(a, s);
            else rc = go<bf, QBMOE_W_BF16, bf, EPI_SITU>(a, s);
        } else if (wfmt == QBMOE_W_MXFP4) {
            if (epi == EPI_STORE) rc = go<bf, QBMOE_W_MXFP4, bf, EPI_STORE>(a, s);
            else if (epi == EPI_SITU) rc = go<bf, QBMOE_W_MXFP4, bf, EPI_SITU>(a, s);
        }
    }
    if (nl) ++*nl;
    return rc;
}

}  // namespace qbh
