// append.cu -- latent-cache append: the shared latent of one new token per
// sequence, written into the cache.
//
// Eqs. (1)-(2) of "LatentIndex: Cross-Layer Sharing with Layer-Specific
// Selection for Sparse Attention" (summary page, Methodology, "Shared Latent
// Cache"): from the anchor layer's hidden state x of token t,
//     z^N = P_N^T x,   z^R = Q_t P_R^T x,   c = [z^R ; z^N],
// with Q_t the rotary position encoding of the RoPE branch, applied as
// complex multiplications within each rotary frequency: pair i of z^R is
// multiplied by exp(i t theta_i), theta_i = base^(-2i/rR).
//
// A token's r outputs are split over a cluster of ceil(r / 32) CTAs, 32
// outputs each (RoPE pairs never straddle two CTAs).  A CTA's eight warps
// take four outputs each; the lanes of a warp share the dm-long dot products
// (16-byte loads of x and of the four P rows, fp32 accumulation) and reduce
// them with shuffles.  The rotation angle is formed and turned into cos/sin
// in double precision (t * theta reaches 10^5 rad).  For an fp8 cache the
// row scale max|c| / 448 needs the whole row: each CTA publishes its partial
// maximum in shared memory and reads its cluster peers' through distributed
// shared memory between two cluster barriers.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kThreads = 256;
constexpr int kOutPerCta = 32;
constexpr int kOutPerWarp = kOutPerCta / (kThreads / 32);   // 4

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// The float at `local` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_peer(const float *local, uint32_t rank)
{
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// 8 consecutive elements starting at e (16-byte aligned for bf16; two
// 16-byte loads for fp32) into fp32.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, int64_t e, float (&o)[8])
{
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p + e));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void load8(const float *p, int64_t e, float (&o)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p + e));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p + e + 4));
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

template <typename TX, typename TP>
__global__ void __launch_bounds__(kThreads, 2) append_kernel(const AppendParams p)
{
    __shared__ float c_s[kOutPerCta];
    __shared__ float amax_s;
    const int b = blockIdx.x;
    const int blk = blockIdx.y;                  // = rank in the cluster
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const TX *x = static_cast<const TX *>(p.x) + static_cast<int64_t>(b) * p.dm;
    const TP *P = static_cast<const TP *>(p.P);
    griddep_wait();
    griddep_launch_dependents();

    // ---- four dot products per warp
    const int i0 = blk * kOutPerCta + warp * kOutPerWarp;
    float acc[kOutPerWarp] = {0.f, 0.f, 0.f, 0.f};
    const bool vec = p.vec;
    if (vec) {
        // unrolled so that several iterations' loads are in flight (the loop
        // is bound by load latency, with one CTA of eight warps per token slice)
#pragma unroll 4
        for (int64_t e = 8 * lane; e < p.dm; e += 8 * 32) {
            float xv[8];
            load8(x, e, xv);
#pragma unroll
            for (int o = 0; o < kOutPerWarp; ++o) {
                if (i0 + o < p.r) {
                    float pv[8];
                    load8(P, static_cast<int64_t>(i0 + o) * p.dm + e, pv);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[o] = fmaf(pv[j], xv[j], acc[o]);
                }
            }
        }
    } else {
#pragma unroll 4
        for (int64_t e = lane; e < p.dm; e += 32) {
            const float xv = to_f(x[e]);
#pragma unroll
            for (int o = 0; o < kOutPerWarp; ++o)
                if (i0 + o < p.r)
                    acc[o] = fmaf(to_f(P[static_cast<int64_t>(i0 + o) * p.dm + e]), xv, acc[o]);
        }
    }
#pragma unroll
    for (int o = 0; o < kOutPerWarp; ++o) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc[o] += __shfl_xor_sync(0xffffffffu, acc[o], off);
    }
    if (lane == 0) {
#pragma unroll
        for (int o = 0; o < kOutPerWarp; ++o)
            c_s[warp * kOutPerWarp + o] = acc[o];
    }
    __syncthreads();

    // ---- rotary encoding of the RoPE branch (pairs 2i, 2i+1 with 2i < rR)
    const int t = p.pos[b];
    const int i = blk * kOutPerCta + threadIdx.x;     // this thread's output (threads < 32)
    float c = 0.f;
    if (threadIdx.x < kOutPerCta && i < p.r) {
        c = c_s[threadIdx.x];
        if (i < p.rR) {
            const int pr = i >> 1;
            const double ang = static_cast<double>(t) * pow(static_cast<double>(p.base), -2.0 * pr / p.rR);
            double sn, cs;
            sincos(ang, &sn, &cs);
            const double re = c_s[threadIdx.x & ~1], im = c_s[threadIdx.x | 1];
            c = static_cast<float>((i & 1) ? re * sn + im * cs : re * cs - im * sn);
        }
    }

    // ---- row scale (fp8): the maximum over the cluster's CTAs
    float scale = 1.f;
    if (p.lat_t == LI_FP8_E4M3) {
        float m = fabsf(c);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (threadIdx.x == 0)
            amax_s = m;
        cluster_sync();                              // every CTA's partial is written
        float amax = 0.f;
        if (threadIdx.x < 32)
            for (int rk = 0; rk < static_cast<int>(gridDim.y); ++rk)
                amax = fmaxf(amax, ld_peer(&amax_s, static_cast<uint32_t>(rk)));
        cluster_sync();                              // no CTA leaves while peers read it
        scale = amax / 448.f;
        if (threadIdx.x < kOutPerCta)
            c = amax > 0.f ? c * (448.f / amax) : 0.f;
    }

    // ---- store into row pos[b] of sequence b
    if (t < 0 || t >= p.L) {
        if (threadIdx.x == 0 && blk == 0)
            atomicCAS(p.status, 0, LI_ERR_DEVICE_BOUNDS);
        return;
    }
    if (threadIdx.x < kOutPerCta && i < p.r) {
        const int64_t row = static_cast<int64_t>(b) * p.L + t;
        if (p.lat_t == LI_FP8_E4M3) {
            const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3);
            static_cast<uint8_t *>(p.latent)[row * p.r + i] = q;
            if (i == 0)
                p.lat_scale[row] = scale;
        } else if (p.lat_t == LI_BF16) {
            static_cast<__nv_bfloat16 *>(p.latent)[row * p.r + i] = __float2bfloat16_rn(c);
        } else {
            static_cast<float *>(p.latent)[row * p.r + i] = c;
        }
    }
}

template <typename TX, typename TP>
cudaError_t launch_t(const AppendParams &p, cudaStream_t s)
{
    const int nblk = (p.r + kOutPerCta - 1) / kOutPerCta;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.B), static_cast<unsigned>(nblk));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(nblk);
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, append_kernel<TX, TP>, p);
}

} // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t s)
{
    if (p.B <= 0)
        return cudaSuccess;
    if (p.x_t == LI_BF16 && p.P_t == LI_BF16)
        return launch_t<__nv_bfloat16, __nv_bfloat16>(p, s);
    if (p.x_t == LI_F32 && p.P_t == LI_BF16)
        return launch_t<float, __nv_bfloat16>(p, s);
    if (p.x_t == LI_BF16 && p.P_t == LI_F32)
        return launch_t<__nv_bfloat16, float>(p, s);
    return launch_t<float, float>(p, s);
}

} // namespace li
