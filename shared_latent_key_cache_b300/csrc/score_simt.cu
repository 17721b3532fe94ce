// score_simt.cu -- group scoring on the CUDA cores (fp32 FMA, no TF32).
//
// The same eq. (8) as the tensor-core scorer ("LatentIndex: Cross-Layer
// Sharing with Layer-Specific Selection for Sparse Attention", summary page,
// Methodology):  u_l(t) = sum_h w_{l,h} ReLU(q~_{l,h} . c_t + beta_{l,h}),
// for any storage type pair and small shapes.  This is the path for fp32
// caches, whose scores are checked to a relative 1e-5, and for shapes the
// tensor-core tiles do not cover.
//
// One CTA scores 128 positions of one query: the query's absorbed rows and
// the 128 latent rows are decoded (with their scales) to fp32 in shared
// memory; thread i then evaluates every (layer, head) dot product of its
// position in plain fp32 FMA order and writes one score per layer.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kTok = 128;

__device__ __forceinline__ float decode(const void *p, int dtype, int64_t i)
{
    if (dtype == LI_F32)
        return static_cast<const float *>(p)[i];
    if (dtype == LI_BF16)
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    const __nv_fp8_storage_t code = static_cast<const uint8_t *>(p)[i];
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(code, __NV_E4M3)));
}

__global__ void __launch_bounds__(kTok) score_simt_kernel(const ScoreParams p)
{
    extern __shared__ float sm[];
    griddep_wait();
    griddep_launch_dependents();
    const int N = p.Gs * p.H;
    const int rp = p.r + 1;
    float *qs = sm;                     // [N][r]
    float *ws = qs + N * p.r;           // [N]
    float *bs = ws + N;                 // [N]
    float *cs = bs + N;                 // [kTok][r+1]

    const int64_t bt = blockIdx.y;
    const int b = static_cast<int>(bt / p.T);
    const int t = static_cast<int>(bt % p.T);
    const bool gather = p.gather_idx != nullptr;
    int Lv = p.L_lat;
    if (gather)
        Lv = p.n_gather;
    else if (p.q_pos != nullptr)
        Lv = min(p.L_lat, p.q_pos[t] + 1);
    const int pos0 = blockIdx.x * kTok;
    if (pos0 >= Lv)
        return;

    const int64_t row0 = (bt * p.Gtot + p.g0) * p.H;   // first absorbed row of the query
    for (int e = threadIdx.x; e < N * p.r; e += kTok) {
        const int j = e / p.r;
        const float s = p.q_abs_scale ? p.q_abs_scale[row0 + j] : 1.f;
        qs[e] = s * decode(p.q_abs, p.abs_t, row0 * p.r + e);
    }
    for (int j = threadIdx.x; j < N; j += kTok) {
        ws[j] = p.w[row0 + j];
        bs[j] = p.beta ? p.beta[row0 + j] : 0.f;
    }
    for (int e = threadIdx.x; e < kTok * p.r; e += kTok) {
        const int i = e / p.r, k = e % p.r;
        const int pos = pos0 + i;
        float v = 0.f;
        if (pos < Lv) {
            int tok = pos;
            if (gather)
                tok = p.gather_idx[static_cast<int64_t>(b) * p.L_out + pos];
            if (tok >= 0 && tok < p.L_lat) {
                const int64_t n = static_cast<int64_t>(b) * p.L_lat + tok;
                const float s = p.lat_scale ? p.lat_scale[n] : 1.f;
                v = s * decode(p.latent, p.lat_t, n * p.r + k);
            } else if (k == 0) {
                atomicCAS(p.status, 0, -7 /* LI_ERR_DEVICE_BOUNDS */);
            }
        }
        cs[i * rp + k] = v;
    }
    __syncthreads();

    const int pos = pos0 + threadIdx.x;
    if (pos >= Lv)
        return;
    const float *c = cs + threadIdx.x * rp;
    float *out = p.scores + (static_cast<int64_t>(bt) * (p.Gout ? p.Gout : p.Gs) + p.gout0) * p.L_out + pos;
    for (int l = 0; l < p.Gs; ++l) {
        float u = 0.f;
        for (int h = 0; h < p.H; ++h) {
            const int j = l * p.H + h;
            const float *q = qs + j * p.r;
            float dot = 0.f;
            for (int k = 0; k < p.r; ++k)
                dot = fmaf(q[k], c[k], dot);
            dot += bs[j];
            u = fmaf(ws[j], fmaxf(dot, 0.f), u);
        }
        out[static_cast<int64_t>(l) * p.L_out] = u;
    }
}

} // namespace

cudaError_t launch_score_simt(const ScoreParams &p, cudaStream_t s)
{
    const int N = p.Gs * p.H;
    const size_t smem = sizeof(float) * (static_cast<size_t>(N) * p.r + 2 * N +
                                         static_cast<size_t>(kTok) * (p.r + 1));
    if (smem > 227 * 1024)
        return cudaErrorInvalidValue;
    static std::atomic<int> attr_set{0};
    if (smem > 48 * 1024 && !attr_set.load()) {
        cudaError_t e = cudaFuncSetAttribute(score_simt_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess)
            return e;
        attr_set.store(1);
    }
    const int Lrow = p.gather_idx ? p.n_gather : p.L_lat;
    const int gx = (Lrow + kTok - 1) / kTok;
    const int64_t gy = static_cast<int64_t>(p.B) * p.T;
    if (gx <= 0 || gy <= 0)
        return cudaSuccess;
    if (gy > 65535)
        return cudaErrorInvalidValue;
    return launch_pdl(score_simt_kernel, dim3(gx, static_cast<unsigned>(gy)), dim3(kTok),
                      static_cast<size_t>(smem), s, p);
}

} // namespace li
