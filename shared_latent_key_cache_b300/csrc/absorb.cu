// absorb.cu -- query-side decoder absorption, q~_{n,l,h} = D_l q_{n,l,h}
// ("LatentIndex: Cross-Layer Sharing with Layer-Specific Selection for Sparse
// Attention", summary page, eq. (6); the decoder is stored r x d, so this is
// the page's (D^(l))^T q).  Optionally rounds each output row to FP8 E4M3 with
// one fp32 scale per row (max|row| / 448), the operand format of the fp8
// tensor-core scorer, or to bf16.
//
// One CTA computes 32 query rows of one layer against all r <= 256 outputs.
// Query and decoder chunks (32 of the d inputs at a time) are staged k-major
// in shared memory with 16-byte global loads, so a thread reads its two rows
// with one 8-byte load and four consecutive outputs with one 16-byte load;
// each thread keeps a 2 rows x (4 x ceil(r/64)) register tile and accumulates
// the two rows as one packed fp32 pair (FFMA2).  A row's outputs live in the
// 16 lanes that share its row pair, so the fp8 row maximum is a 16-lane
// shuffle reduction.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kRows = 32;      // query rows per CTA
constexpr int kKC = 32;        // K chunk
constexpr int kMaxR = 256;     // 4 column groups of 64
constexpr int kThreads = 256;  // 16 row pairs x 16 column lanes
constexpr int kQPad = 36;      // qs row stride (floats)
constexpr int kDPad = kMaxR + 4;

__device__ __forceinline__ float load_val(const void *p, int dtype, int64_t i)
{
    if (dtype == LI_BF16)
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    return static_cast<const float *>(p)[i];
}

// Loads 16 bytes (8 bf16 or 4 fp32 values) at element offset `off` as floats;
// off < 0 yields zeros.
__device__ __forceinline__ void load16(const void *p, int dtype, int64_t off, float (&v)[8])
{
#pragma unroll
    for (int t = 0; t < 8; ++t)
        v[t] = 0.f;
    if (off < 0)
        return;
    if (dtype == LI_BF16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + off));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            v[2 * t] = __uint_as_float(w[t] << 16);
            v[2 * t + 1] = __uint_as_float(w[t] & 0xFFFF0000u);
        }
    } else {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + off));
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
    }
}

__global__ void __launch_bounds__(kThreads) absorb_kernel(AbsorbParams p)
{
    __shared__ __align__(16) float qs[kKC][kQPad];
    __shared__ __align__(16) float Ds[kKC][kDPad];

    griddep_wait();
    griddep_launch_dependents();
    const int l = blockIdx.y;
    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int64_t nrows = static_cast<int64_t>(p.N) * p.H;   // rows of this layer
    const int64_t rho0 = static_cast<int64_t>(blockIdx.x) * kRows;
    const int NJ = (p.r + 63) / 64;

    // element offset of row rho (= n*H + h) of layer l in a [N][G][H][width] tensor
    auto row_off = [&](int64_t rho, int width) -> int64_t {
        const int64_t n = rho / p.H, h = rho % p.H;
        return ((n * p.G + l) * p.H + h) * static_cast<int64_t>(width);
    };

    float2 acc[16];   // [j*4 + c]: rows (2ty, 2ty+1) x column 64j + 4tx + c
#pragma unroll
    for (int i = 0; i < 16; ++i)
        acc[i] = make_float2(0.f, 0.f);

    if (p.D == nullptr) {
        // identity decoder (r == d): conversion / quantisation only
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t rho = rho0 + 2 * ty + rr;
            if (rho >= nrows)
                continue;
            const int64_t off = row_off(rho, p.d);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col = 64 * j + 4 * tx + c;
                    if (col < p.r) {
                        const float v = load_val(p.q, p.q_t, off + col);
                        if (rr == 0)
                            acc[j * 4 + c].x = v;
                        else
                            acc[j * 4 + c].y = v;
                    }
                }
        }
    } else {
        // 16-byte staging loads need rows whose length is a multiple of 8 elements
        const bool vec = (p.d % 8) == 0;
        const int epl = p.q_t == LI_BF16 ? 8 : 4;    // elements per 16-byte load
        const int lpr = kKC / epl;                   // loads per row per chunk
        const int epl_d = p.D_t == LI_BF16 ? 8 : 4;
        const int lpr_d = kKC / epl_d;
        for (int k0 = 0; k0 < p.d; k0 += kKC) {
            if (vec) {
                for (int e = tid; e < kRows * lpr; e += kThreads) {
                    const int i = e / lpr, part = e % lpr;
                    const int64_t rho = rho0 + i;
                    const bool in = rho < nrows && k0 + part * epl < p.d;
                    float v[8];
                    load16(p.q, p.q_t, in ? row_off(rho, p.d) + k0 + part * epl : -1, v);
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        if (t < epl)
                            qs[part * epl + t][i] = v[t];
                }
                for (int e = tid; e < kMaxR * lpr_d; e += kThreads) {
                    const int j = e / lpr_d, part = e % lpr_d;
                    const bool in = j < p.r && k0 + part * epl_d < p.d;
                    float v[8];
                    load16(p.D, p.D_t, in ? (static_cast<int64_t>(l) * p.r + j) * p.d + k0 + part * epl_d : -1, v);
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        if (t < epl_d)
                            Ds[part * epl_d + t][j] = v[t];
                }
            } else {
                for (int e = tid; e < kRows * kKC; e += kThreads) {
                    const int i = e / kKC, kk = e % kKC;
                    const int64_t rho = rho0 + i;
                    float v = 0.f;
                    if (rho < nrows && k0 + kk < p.d)
                        v = load_val(p.q, p.q_t, row_off(rho, p.d) + k0 + kk);
                    qs[kk][i] = v;
                }
                for (int e = tid; e < kMaxR * kKC; e += kThreads) {
                    const int j = e / kKC, kk = e % kKC;
                    float v = 0.f;
                    if (j < p.r && k0 + kk < p.d)
                        v = load_val(p.D, p.D_t, (static_cast<int64_t>(l) * p.r + j) * p.d + k0 + kk);
                    Ds[kk][j] = v;
                }
            }
            __syncthreads();
#pragma unroll 2
            for (int kk = 0; kk < kKC; ++kk) {
                const float2 a = *reinterpret_cast<const float2 *>(&qs[kk][2 * ty]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j < NJ) {
                        const float4 b = *reinterpret_cast<const float4 *>(&Ds[kk][64 * j + 4 * tx]);
                        acc[j * 4 + 0] = __ffma2_rn(a, make_float2(b.x, b.x), acc[j * 4 + 0]);
                        acc[j * 4 + 1] = __ffma2_rn(a, make_float2(b.y, b.y), acc[j * 4 + 1]);
                        acc[j * 4 + 2] = __ffma2_rn(a, make_float2(b.z, b.z), acc[j * 4 + 2]);
                        acc[j * 4 + 3] = __ffma2_rn(a, make_float2(b.w, b.w), acc[j * 4 + 3]);
                    }
                }
            }
            __syncthreads();
        }
    }

    const bool vec = (p.r % 4) == 0;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int64_t rho = rho0 + 2 * ty + rr;
        const bool live = rho < nrows;        // uniform across the 16 lanes of a row
        const int64_t off = live ? row_off(rho, p.r) : 0;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = rr == 0 ? acc[i].x : acc[i].y;
        if (p.abs_t == LI_FP8_E4M3) {
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (64 * j + 4 * tx + c < p.r)
                        amax = fmaxf(amax, fabsf(v[j * 4 + c]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float inv = amax > 0.f ? 448.f / amax : 0.f;
            if (live) {
                uint8_t *out = static_cast<uint8_t *>(p.q_abs) + off;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = 64 * j + 4 * tx;
                    if (col >= p.r)
                        continue;
                    uint32_t code[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        code[c] = static_cast<uint8_t>(
                            __nv_cvt_float_to_fp8(v[j * 4 + c] * inv, __NV_SATFINITE, __NV_E4M3));
                    if (vec) {
                        *reinterpret_cast<uint32_t *>(out + col) =
                            code[0] | (code[1] << 8) | (code[2] << 16) | (code[3] << 24);
                    } else {
                        for (int c = 0; c < 4; ++c)
                            if (col + c < p.r)
                                out[col + c] = static_cast<uint8_t>(code[c]);
                    }
                }
                if (tx == 0)
                    p.q_abs_scale[off / p.r] = amax / 448.f;
            }
        } else if (live) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = 64 * j + 4 * tx;
                if (col >= p.r)
                    continue;
                if (p.abs_t == LI_BF16) {
                    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.q_abs) + off + col;
                    if (vec) {
                        __nv_bfloat162 lo = __floats2bfloat162_rn(v[j * 4 + 0], v[j * 4 + 1]);
                        __nv_bfloat162 hi = __floats2bfloat162_rn(v[j * 4 + 2], v[j * 4 + 3]);
                        uint2 pk;
                        pk.x = *reinterpret_cast<uint32_t *>(&lo);
                        pk.y = *reinterpret_cast<uint32_t *>(&hi);
                        *reinterpret_cast<uint2 *>(out) = pk;
                    } else {
                        for (int c = 0; c < 4; ++c)
                            if (col + c < p.r)
                                out[c] = __float2bfloat16_rn(v[j * 4 + c]);
                    }
                } else {
                    float *out = static_cast<float *>(p.q_abs) + off + col;
                    if (vec) {
                        *reinterpret_cast<float4 *>(out) =
                            make_float4(v[j * 4 + 0], v[j * 4 + 1], v[j * 4 + 2], v[j * 4 + 3]);
                    } else {
                        for (int c = 0; c < 4; ++c)
                            if (col + c < p.r)
                                out[c] = v[j * 4 + c];
                    }
                }
            }
        }
    }
}

} // namespace

cudaError_t launch_absorb(const AbsorbParams &p, cudaStream_t s)
{
    if (absorb_tc_supported(p))
        return launch_absorb_tc(p, s);
    const int64_t nrows = static_cast<int64_t>(p.N) * p.H;
    const int64_t gx = (nrows + kRows - 1) / kRows;
    if (gx > 0x7FFFFFFF || p.G > 65535 || p.r > kMaxR)
        return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(p.G));
    return launch_pdl(absorb_kernel, grid, dim3(kThreads), 0, s, p);
}

} // namespace li
