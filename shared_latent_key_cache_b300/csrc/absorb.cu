// absorb.cu -- query-side decoder absorption, q~_{n,l,h} = D_l q_{n,l,h}
// ("LatentIndex: Cross-Layer Sharing with Layer-Specific Selection for Sparse
// Attention", summary page, eq. (6); the decoder is stored r x d, so this is
// the page's (D^(l))^T q).  Optionally rounds each output row to FP8 E4M3 with
// one fp32 scale per row (max|row| / 448), which is the operand format of the
// fp8 tensor-core scorer.
//
// One CTA computes 64 query rows of one layer against all r outputs: the
// rows' queries and the layer's decoder stream through shared memory in
// 32-wide K chunks and each thread keeps a 4 x 16 register tile (fp32 FMA).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "li_internal.cuh"

namespace li {
namespace {

constexpr int kRows = 64;      // query rows per CTA
constexpr int kKC = 32;        // K chunk
constexpr int kMaxR = 256;     // 16 column slots x 16 lanes
constexpr int kThreads = 256;  // 16 (rows) x 16 (cols)

__device__ __forceinline__ float load_val(const void *p, int dtype, int64_t i)
{
    if (dtype == LI_BF16)
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    return static_cast<const float *>(p)[i];
}

__global__ void __launch_bounds__(kThreads) absorb_kernel(AbsorbParams p)
{
    __shared__ float qs[kRows][kKC + 1];
    __shared__ float Ds[kMaxR][kKC + 1];

    const int l = blockIdx.y;
    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int64_t nrows = static_cast<int64_t>(p.N) * p.H;   // rows of this layer
    const int64_t rho0 = static_cast<int64_t>(blockIdx.x) * kRows;

    float acc[4][16];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 16; ++c)
            acc[i][c] = 0.f;

    // element offset of row (rho = n*H + h) of layer l in a [N][G][H][width] tensor
    auto row_off = [&](int64_t rho, int width) -> int64_t {
        int64_t n = rho / p.H, h = rho % p.H;
        return ((n * p.G + l) * p.H + h) * static_cast<int64_t>(width);
    };

    if (p.D == nullptr) {
        // identity decoder (r == d): conversion / quantisation only
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int64_t rho = rho0 + ty * 4 + i;
            if (rho >= nrows)
                continue;
            int64_t off = row_off(rho, p.d);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                int col = tx + 16 * c;
                if (col < p.r)
                    acc[i][c] = load_val(p.q, p.q_t, off + col);
            }
        }
    } else {
        for (int k0 = 0; k0 < p.d; k0 += kKC) {
            for (int e = tid; e < kRows * kKC; e += kThreads) {
                int i = e / kKC, kk = e % kKC;
                int64_t rho = rho0 + i;
                float v = 0.f;
                if (rho < nrows && k0 + kk < p.d)
                    v = load_val(p.q, p.q_t, row_off(rho, p.d) + k0 + kk);
                qs[i][kk] = v;
            }
            for (int e = tid; e < p.r * kKC; e += kThreads) {
                int j = e / kKC, kk = e % kKC;
                float v = 0.f;
                if (k0 + kk < p.d)
                    v = load_val(p.D, p.D_t, (static_cast<int64_t>(l) * p.r + j) * p.d + k0 + kk);
                Ds[j][kk] = v;
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < kKC; ++kk) {
                float a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    a[i] = qs[ty * 4 + i][kk];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    int col = tx + 16 * c;
                    float b = (col < p.r) ? Ds[col][kk] : 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[i][c] = fmaf(a[i], b, acc[i][c]);
                }
            }
            __syncthreads();
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int64_t rho = rho0 + ty * 4 + i;
        bool live = rho < nrows;       // uniform across the 16 lanes of a row
        int64_t off = live ? row_off(rho, p.r) : 0;
        if (p.abs_t == LI_FP8_E4M3) {
            float amax = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (tx + 16 * c < p.r)
                    amax = fmaxf(amax, fabsf(acc[i][c]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            float inv = amax > 0.f ? 448.f / amax : 0.f;
            if (live) {
                uint8_t *out = static_cast<uint8_t *>(p.q_abs);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    int col = tx + 16 * c;
                    if (col < p.r)
                        out[off + col] = static_cast<uint8_t>(
                            __nv_cvt_float_to_fp8(acc[i][c] * inv, __NV_SATFINITE, __NV_E4M3));
                }
                if (tx == 0)
                    p.q_abs_scale[off / p.r] = amax / 448.f;
            }
        } else if (live) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                int col = tx + 16 * c;
                if (col >= p.r)
                    continue;
                if (p.abs_t == LI_BF16)
                    static_cast<__nv_bfloat16 *>(p.q_abs)[off + col] = __float2bfloat16_rn(acc[i][c]);
                else
                    static_cast<float *>(p.q_abs)[off + col] = acc[i][c];
            }
        }
    }
}

} // namespace

cudaError_t launch_absorb(const AbsorbParams &p, cudaStream_t s)
{
    int64_t nrows = static_cast<int64_t>(p.N) * p.H;
    int64_t gx = (nrows + kRows - 1) / kRows;
    if (gx > 0x7FFFFFFF || p.G > 65535)
        return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(p.G));
    absorb_kernel<<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

} // namespace li
