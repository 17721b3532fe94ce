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
// The projection is the contraction [B x dm] x [dm x r] (B new tokens, dm
// the hidden size): split over the hidden dimension.  A thread-block
// cluster of KS CTAs (up to 16) takes kTok tokens; CTA s of the cluster
// takes the hidden slice [s kc, (s + 1) kc), so that P is read
// ceil(B / kTok) times (from L2 after the first) instead of once per token.
// With bf16 P and dm % 8 == 0 the CTA brings its slice of all r rows of P
// into shared memory with 2D TMA copies (boxes of 64 hidden elements x r
// rows), kw elements at a time; the lanes of a warp then run along the
// hidden dimension (each holding its eight hidden elements of the kTok
// tokens' x in registers) and the warp's partial sums for eight rows x kTok
// tokens are combined by a transposing butterfly reduction (31 shuffles for
// 32 sums).  Other input types read P row by row, one thread per row.
//
// The KS partial sums of each output are added in a fixed order (CTA 0
// first) by the CTA that owns the output, reading its peers' partials
// through distributed shared memory; the same CTA applies the rotation.
// The frequencies theta_i come from the host in double precision; the angle
// t * theta_i (up to 10^5 rad) is formed and reduced modulo 2 pi in double
// precision (two-term 2 pi), and the reduced angle's sine and cosine are
// taken in fp32.  For an fp8 cache the row scale max|c| / 448 needs the
// whole row: each CTA folds its outputs' magnitudes into per-token maxima in
// CTA 0's shared memory (an atomic max on the float's bits, exact for
// non-negative floats) and reads them back after a cluster barrier.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kThreads = 256;     // eight warps; r <= 256 latent rows
constexpr int kTok = 4;           // tokens per cluster
constexpr int kSub = 256;         // staged P: hidden elements per step at most (one group of 8 per lane)
constexpr int kXs = 512;          // hidden elements of x staged at a time
constexpr int kMaxKS = 16;        // CTAs per cluster (hidden-dimension split)
constexpr int kBox = 64;          // hidden elements per TMA box of P (128 bytes of bf16)

__device__ __forceinline__ uint32_t cl_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cl_nrank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// Address of `local` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    return a;
}

__device__ __forceinline__ float ld_peer_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void max_peer_u32(uint32_t addr, uint32_t v)
{
    asm volatile("red.relaxed.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
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

struct AppendSmem {
    float xs[kTok][kXs];         // slice of x, fp32; after the partial sums: finished outputs
    float part[kTok][kThreads];  // this CTA's partial sums, [token][latent row]
    uint32_t amax_l[kTok];       // this CTA's row maxima, then the cluster's (float bits)
    uint32_t amax_s[kTok];       // CTA 0: the cluster's row maxima
    uint64_t bar;                // staged path: P copies
    int abort_s;
};

// Stages x[t][s0, s0 + n) of this cluster's tokens (n <= kXs; zero past n
// and past the last token) as fp32.  Every load of a thread is issued before
// its first store, so the slice costs one memory round trip.
template <typename TX>
__device__ __forceinline__ void stage_x(AppendSmem &sm, const TX *x, int64_t dm, int nt, int64_t s0, int n)
{
    constexpr int kPer = kTok * kXs / kThreads;
    float v[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int j = threadIdx.x + q * kThreads;
        const int t = j / kXs, e = j % kXs;
        v[q] = (t < nt && e < n) ? to_f(x[t * dm + s0 + e]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int j = threadIdx.x + q * kThreads;
        sm.xs[j / kXs][j % kXs] = v[q];
    }
}

// After every CTA's partial sums are in part[][]: the outputs this CTA owns
// (elements [ks per, (ks + 1) per) of [nt][r]) are summed over the cluster
// in a fixed order, rotated, scaled and stored.  Every CTA of the cluster
// must call it (it contains cluster barriers).
__device__ void finish_outputs(AppendSmem &sm, const AppendParams &p, int tok0, int nt, bool drain,
                               uint32_t drain_parity)
{
    const uint32_t ks = cl_rank(), nks = cl_nrank();
    const int tid = threadIdx.x;
    float *cval = &sm.xs[0][0];                       // finished outputs, flat: per <= kTok * 256
    cluster_sync();                                   // every CTA's partials are written
    const int tot = nt * p.r;
    const int per = (kTok * p.r + static_cast<int>(nks) - 1) / static_cast<int>(nks);
    const int e0 = static_cast<int>(ks) * per;
    const int e1 = min(tot, e0 + per);
    auto full_sum = [&](int t, int i) {
        float v[kMaxKS];
#pragma unroll
        for (int q = 0; q < kMaxKS; ++q)                // all peers' loads in flight together
            v[q] = q < static_cast<int>(nks) ? ld_peer_f32(peer_addr(&sm.part[t][i], q)) : 0.f;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxKS; ++q)                // fixed order: CTA 0 first
            s += v[q];
        return s;
    };
    for (int e = e0 + tid; e < e1; e += kThreads) {
        const int t = e / p.r, i = e % p.r;
        float c = full_sum(t, i);
        if (i < p.rR) {
            // rotate the complex pair (2 pr, 2 pr + 1) by t * theta_pr
            const float o = full_sum(t, i ^ 1);
            const float re = (i & 1) ? o : c, im = (i & 1) ? c : o;
            const double ang = static_cast<double>(p.pos[tok0 + t]) * p.theta[i >> 1];
            const double kq = rint(ang * 0.15915494309189535);          // 1 / (2 pi)
            double red = fma(-kq, 6.283185307179586, ang);              // 2 pi, high part
            red = fma(-kq, 2.4492935982947064e-16, red);                // 2 pi, low part
            float sn, cs;
            sincosf(static_cast<float>(red), &sn, &cs);
            c = (i & 1) ? re * sn + im * cs : re * cs - im * sn;
        }
        cval[e - e0] = c;
        if (p.lat_t == LI_FP8_E4M3)
            atomicMax(&sm.amax_l[t], __float_as_uint(fabsf(c)));
    }
    if (p.lat_t == LI_FP8_E4M3) {
        __syncthreads();
        if (tid < nt && sm.amax_l[tid] != 0u)
            max_peer_u32(peer_addr(&sm.amax_s[tid], 0), sm.amax_l[tid]);
        cluster_sync();                               // the row maxima are complete
        if (tid < nt)
            sm.amax_l[tid] = ld_peer_u32(peer_addr(&sm.amax_s[tid], 0));
        __syncthreads();
    }
    // This CTA reads no peer from here on (its loads have returned): a
    // relaxed arrival now and the wait before leaving keep every CTA's shared
    // memory alive while peers read it, and no release waits for the stores.
    cluster_arrive_relaxed();

    // ---- store into row pos[b] of sequence b
    for (int e = e0 + tid; e < e1; e += kThreads) {
        const int t = e / p.r, i = e % p.r;
        const int b = tok0 + t;
        const int pt = p.pos[b];
        if (pt < 0 || pt >= p.L) {
            if (i == 0)
                atomicCAS(p.status, 0, LI_ERR_DEVICE_BOUNDS);
            continue;
        }
        const int64_t row = static_cast<int64_t>(b) * p.L + pt;
        float c = cval[e - e0];
        if (p.lat_t == LI_FP8_E4M3) {
            const float am = __uint_as_float(sm.amax_l[t]);
            c = am > 0.f ? c * (448.f / am) : 0.f;
            static_cast<uint8_t *>(p.latent)[row * p.r + i] = __nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3);
            if (i == 0)
                p.lat_scale[row] = am / 448.f;
        } else if (p.lat_t == LI_BF16) {
            static_cast<__nv_bfloat16 *>(p.latent)[row * p.r + i] = __float2bfloat16_rn(c);
        } else {
            static_cast<float *>(p.latent)[row * p.r + i] = c;
        }
    }
    if (drain) {
        // a copy phase was given up on: let it land (bounded) before the
        // shared memory it writes goes away
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&sm.bar, drain_parity) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
    }
    cluster_wait();                                   // peers no longer read this CTA
}

// bf16 P with dm % 8 == 0: the CTA's slice of P comes into shared memory by
// TMA, kw hidden elements at a time as kw / kBox boxes of [r][kBox].
template <typename TX>
__global__ void __launch_bounds__(kThreads)
    append_staged_kernel(const __grid_constant__ CUtensorMap tmP, const AppendParams p)
{
    extern __shared__ uint8_t dyn_raw[];
    __shared__ AppendSmem sm;
    const uint32_t ks = cl_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok0 = blockIdx.y * kTok;
    const int nt = min(kTok, p.B - tok0);
    const int64_t dm = p.dm;
    const int64_t k0 = static_cast<int64_t>(ks) * p.kc;
    const int64_t k1 = min(dm, k0 + p.kc);
    const TX *x = static_cast<const TX *>(p.x) + static_cast<int64_t>(tok0) * dm;
    // box j of the slice: [r][kBox] bf16 at Ps + j r kBox (128-byte aligned)
    uint8_t *dyn = dyn_raw + ((128u - (smem_u32(dyn_raw) & 127u)) & 127u);
    const __nv_bfloat16 *Ps = reinterpret_cast<const __nv_bfloat16 *>(dyn);
    for (int i = tid; i < kTok * kThreads; i += kThreads)
        (&sm.part[0][0])[i] = 0.f;
    if (tid < kTok) {
        sm.amax_l[tid] = 0u;
        sm.amax_s[tid] = 0u;
    }
    if (tid == 0) {
        sm.abort_s = 0;
        mbar_init(&sm.bar, 1);
        mbar_fence_init();
        tma_prefetch_desc(&tmP);
    }
    __syncthreads();
    griddep_wait();

    const int nbatch = (p.r + 7) / 8;                 // eight latent rows per warp step
    const uint32_t box_bytes = static_cast<uint32_t>(p.r) * kBox * 2u;
    // x of the whole slice is staged once when it fits, else per step
    const bool x_once = k1 - k0 <= kXs;
    uint32_t phase = 0;
    bool pending = false;
    for (int64_t s0 = k0; s0 < k1; s0 += p.kw) {
        const int n = static_cast<int>(min(static_cast<int64_t>(p.kw), k1 - s0));
        const int nb = (n + kBox - 1) / kBox;
        __syncthreads();                              // the previous slice is used up
        if (tid == 0) {
            fence_proxy_async_smem();                 // earlier reads of the boxes before the copies
            mbar_arrive_expect_tx(&sm.bar, static_cast<uint32_t>(nb) * box_bytes);
            for (int j = 0; j < nb; ++j)
                tma_load_2d(dyn + j * box_bytes, &tmP, &sm.bar, static_cast<int>(s0) + j * kBox, 0);
        }
        if (!x_once)
            stage_x(sm, x, dm, nt, s0, n);
        else if (s0 == k0)
            stage_x(sm, x, dm, nt, k0, static_cast<int>(k1 - k0));
        const int xo = x_once ? static_cast<int>(s0 - k0) : 0;
        __syncthreads();
        pending = true;
        if (mbar_wait(&sm.bar, phase, &sm.abort_s, p.status, kWaitLimitNs))
            pending = false;
        phase ^= 1u;

        // lane: hidden elements [8 lane, 8 lane + 8) of the slice (kw <= 256),
        // x of the kTok tokens there in registers
        const bool gv = lane < nb * (kBox / 8);
        float xr[kTok][8];
#pragma unroll
        for (int t = 0; t < kTok; ++t)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                xr[t][j] = gv ? sm.xs[t][xo + 8 * lane + j] : 0.f;
        const __nv_bfloat16 *pg = Ps + static_cast<int64_t>(lane >> 3) * p.r * kBox + (lane & 7) * 8;
        for (int bt = warp; bt < nbatch; bt += kThreads / 32) {
            float v[32];                              // [row of the eight][token]
#pragma unroll
            for (int rb = 0; rb < 8; ++rb) {
                const int row = bt * 8 + rb;
                float pv[8];
                if (gv && row < p.r) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(pg + row * kBox);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        pv[2 * q] = __uint_as_float(wd[q] << 16);
                        pv[2 * q + 1] = __uint_as_float(wd[q] & 0xFFFF0000u);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        pv[q] = 0.f;
                }
#pragma unroll
                for (int t = 0; t < kTok; ++t) {
                    float a = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        a = fmaf(pv[j], xr[t][j], a);
                    v[rb * kTok + t] = a;
                }
            }
            // butterfly over the lanes: afterwards lane l holds the warp's sum
            // of value l = (row bt 8 + l / 4, token l % 4)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < o; ++i) {
                    const float send = up ? v[i] : v[i + o];
                    const float keep = up ? v[i + o] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            const int row = bt * 8 + (lane >> 2);
            if (row < p.r)
                sm.part[lane & 3][row] += v[0];
        }
    }
    finish_outputs(sm, p, tok0, nt, pending, phase ^ 1u);
    // the next kernel may start only once this CTA's latent rows are visible
    // (a scan issues its first latent loads before waiting for this grid)
    __threadfence();
    griddep_launch_dependents();
}

// Any other input types: one thread per latent row, P read from global memory.
template <typename TX, typename TP, bool VEC>
__global__ void __launch_bounds__(kThreads) append_direct_kernel(const AppendParams p)
{
    __shared__ AppendSmem sm;
    const uint32_t ks = cl_rank();
    const int tid = threadIdx.x;
    const int tok0 = blockIdx.y * kTok;
    const int nt = min(kTok, p.B - tok0);
    const int64_t dm = p.dm;
    const int64_t k0 = static_cast<int64_t>(ks) * p.kc;
    const int64_t k1 = min(dm, k0 + p.kc);
    const TX *x = static_cast<const TX *>(p.x) + static_cast<int64_t>(tok0) * dm;
    const TP *Prow = static_cast<const TP *>(p.P) + static_cast<int64_t>(tid) * dm;
    if (tid < kTok) {
        sm.amax_l[tid] = 0u;
        sm.amax_s[tid] = 0u;
    }
    griddep_wait();
    float acc[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t)
        acc[t] = 0.f;
    for (int64_t s0 = k0; s0 < k1; s0 += kXs) {
        const int n = static_cast<int>(min(static_cast<int64_t>(kXs), k1 - s0));
        __syncthreads();                              // the previous slice is used up
        stage_x(sm, x, dm, nt, s0, n);
        __syncthreads();
        if (tid < p.r) {
            if (VEC) {
                // n is a multiple of 8 (slices start at multiples of 8, dm % 8 == 0)
#pragma unroll 4
                for (int e = 0; e < n; e += 8) {
                    float pv[8];
                    load8(Prow, s0 + e, pv);
#pragma unroll
                    for (int t = 0; t < kTok; ++t) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            acc[t] = fmaf(pv[j], sm.xs[t][e + j], acc[t]);
                    }
                }
            } else {
#pragma unroll 4
                for (int e = 0; e < n; ++e) {
                    const float pv = to_f(Prow[s0 + e]);
#pragma unroll
                    for (int t = 0; t < kTok; ++t)
                        acc[t] = fmaf(pv, sm.xs[t][e], acc[t]);
                }
            }
        }
    }
    if (tid < p.r) {
#pragma unroll
        for (int t = 0; t < kTok; ++t)
            sm.part[t][tid] = acc[t];
    }
    finish_outputs(sm, p, tok0, nt, false, 0u);
    __threadfence();
    griddep_launch_dependents();
}

constexpr int kMaxDev = 64;
constexpr int kStageBytes = 96 * 1024;               // staged P boxes per CTA at most (two CTAs per SM)

// Largest cluster the device holds for `kern` (16 when a 16-CTA cluster is
// resident: a non-portable size, else 8), found once per device and kernel;
// the kernel's dynamic shared memory limit is raised on the first call.
template <typename Kern>
int cluster_limit(Kern kern, std::atomic<int> (&cache)[kMaxDev], size_t dyn_smem)
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDev)
        dev = 0;
    int c = cache[dev].load(std::memory_order_relaxed);
    if (c != 0)
        return c;
    if (dyn_smem > 0 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn_smem)) !=
            cudaSuccess)
        return -1;
    c = 8;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kMaxKS, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = dyn_smem;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = kMaxKS;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0)
            c = kMaxKS;
    }
    cudaGetLastError();
    cache[dev].store(c, std::memory_order_relaxed);
    return c;
}

// Hidden slices: at least 448 elements, at most `cmax` of them, each a
// multiple of 8 elements.  Returns the cluster size.
int split_hidden(AppendParams &p, int cmax)
{
    int ks = p.dm / 448;
    ks = ks < 1 ? 1 : (ks > cmax ? cmax : ks);
    p.kc = ((p.dm + ks - 1) / ks + 7) / 8 * 8;
    return (p.dm + p.kc - 1) / p.kc;
}

template <typename Kern, typename... Args>
cudaError_t launch_cluster(Kern kern, const AppendParams &p, int ks, size_t dyn_smem, cudaStream_t s,
                           Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks), static_cast<unsigned>((p.B + kTok - 1) / kTok));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename TX>
cudaError_t launch_staged(AppendParams p, cudaStream_t s)
{
    static std::atomic<int> cache[kMaxDev];
    const int cmax = cluster_limit(append_staged_kernel<TX>, cache, kStageBytes + 128);
    if (cmax < 0)
        return cudaErrorInvalidConfiguration;
    const int ks = split_hidden(p, cmax);
    // kw: a multiple of kBox, at most kSub, r rows of it within kStageBytes
    int kw = kSub;
    while (kw > kBox && static_cast<int64_t>(p.r) * kw * 2 > kStageBytes)
        kw -= kBox;
    p.kw = kw;
    // P is a weight: its tensor map is kept per thread for the last (P, dm, r)
    struct MapKey {
        const void *P;
        int dm, r;
    };
    thread_local MapKey key{nullptr, 0, 0};
    thread_local CUtensorMap tmP;
    if (key.P != p.P || key.dm != p.dm || key.r != p.r) {
        EncodeTiledFn enc = encode_fn();
        if (!enc)
            return cudaErrorInvalidConfiguration;
        memset(&tmP, 0, sizeof tmP);
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.dm), static_cast<cuuint64_t>(p.r)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.dm) * 2};
        cuuint32_t box[2] = {static_cast<cuuint32_t>(kBox), static_cast<cuuint32_t>(p.r)};
        cuuint32_t estr[2] = {1, 1};
        key = MapKey{nullptr, 0, 0};
        if (enc(&tmP, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.P), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        key = MapKey{p.P, p.dm, p.r};
    }
    const size_t dyn = static_cast<size_t>(kw / kBox) * p.r * kBox * 2 + 128;
    return launch_cluster(append_staged_kernel<TX>, p, ks, dyn, s, tmP, p);
}

template <typename TX, typename TP, bool VEC>
cudaError_t launch_direct(AppendParams p, cudaStream_t s)
{
    static std::atomic<int> cache[kMaxDev];
    const int cmax = cluster_limit(append_direct_kernel<TX, TP, VEC>, cache, 0);
    const int ks = split_hidden(p, cmax);
    return launch_cluster(append_direct_kernel<TX, TP, VEC>, p, ks, 0, s, p);
}

template <typename TX, typename TP>
cudaError_t launch_v(const AppendParams &p, cudaStream_t s)
{
    return p.vec ? launch_direct<TX, TP, true>(p, s) : launch_direct<TX, TP, false>(p, s);
}

} // namespace

cudaError_t launch_append(const AppendParams &p0, cudaStream_t s)
{
    if (p0.B <= 0)
        return cudaSuccess;
    if (p0.r > kThreads || p0.rR > 2 * kMaxRopePairs)
        return cudaErrorInvalidValue;
    AppendParams p = p0;
    // rotary frequencies theta_i = base^(-2i / rR), in double precision
    for (int i = 0; 2 * i < p.rR; ++i)
        p.theta[i] = std::pow(static_cast<double>(p.base), -2.0 * i / p.rR);
    if (p.x_t == LI_BF16 && p.P_t == LI_BF16)
        return p.vec ? launch_staged<__nv_bfloat16>(p, s) : launch_direct<__nv_bfloat16, __nv_bfloat16, false>(p, s);
    if (p.x_t == LI_F32 && p.P_t == LI_BF16)
        return p.vec ? launch_staged<float>(p, s) : launch_direct<float, __nv_bfloat16, false>(p, s);
    if (p.x_t == LI_BF16 && p.P_t == LI_F32)
        return launch_v<__nv_bfloat16, float>(p, s);
    return launch_v<float, float>(p, s);
}

} // namespace li
