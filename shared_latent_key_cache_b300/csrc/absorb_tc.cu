// absorb_tc.cu -- query-side decoder absorption on the tensor cores.
//
// Eq. (6) of "LatentIndex: Cross-Layer Sharing with Layer-Specific Selection
// for Sparse Attention" (summary page, Methodology): every indexer-head query
// of layer l is folded into that layer's decoder once,  q~ = D_l q  (D_l stored
// r x d), so that the score needs one r-dot per cached latent instead of a
// reconstructed d-dimensional key per token.  For one layer this is the dense
// contraction  [query rows x d] x [d x r]:  one CTA takes a tile of 128 query
// rows (128/H queries x H heads, loaded by TMA as a 4D box) and the layer's
// decoder, issues kind::f16 tcgen05 MMAs (M = 128 rows, N = r, fp32
// accumulation in tensor memory), and eight warps read the result back: two
// per TMEM lane quarter, each thread holding one output row's half (r/2
// columns) in registers after a single round of loads.  The fp8 per-row scale
// (max|row| / 448) combines the two halves' maxima through shared memory;
// the thread then converts (E4M3, round to nearest even, saturating) and
// stores its half.  bf16 and fp32 outputs are converted and stored directly.
//
// Operands are K-major bf16 in 64-element (128-byte) K chunks with the
// 128-byte swizzle, as TMA writes them; both fit in shared memory at once
// (d <= 256, r <= 256), so a CTA has a single load phase and a single MMA
// phase.  Waits are bounded (LI_ERR_TIMEOUT) like every wait of this library.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <atomic>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

constexpr int kThreads = 256;       // 8 warps: two per TMEM lane quarter (128 rows)
constexpr int kTileRows = 128;
constexpr int kChunk = 64;          // bf16 elements per 128-byte K chunk
constexpr int kMaxDev = 64;

struct AbsTcCfg {
    int qpt;            // queries per tile (128 / H)
    int nchunk;         // d / 64
    int a_chunk_bytes;  // 128 rows x 128 B
    int b_chunk_bytes;  // r rows x 128 B
    int off_b;          // byte offset of the decoder operand (1024-aligned)
    int off_bar;
    int tmem_cols;
};

// Ties the registers of a finished 16-column tcgen05.ld to the preceding
// wait::ld (which covers every outstanding load of the thread).
__device__ __forceinline__ void regs_ready16(uint32_t (&v)[16])
{
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                   "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                   "+r"(v[14]), "+r"(v[15])
                 :
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    absorb_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmD,
                     const AbsorbParams p, const AbsTcCfg c, int *status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ float amax_part[2][kTileRows];     // fp8: row maxima of the two column halves
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    uint8_t *smA = base;
    uint8_t *smB = base + c.off_b;
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(base + c.off_bar);
    uint64_t *bar_mma = bar_full + 1;
    volatile int *abort_flag = &abort_s;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int tile = blockIdx.x;
    const int l = blockIdx.y;

    if (threadIdx.x == 0) {
        mbar_init(bar_full, 1u);
        mbar_init(bar_mma, 1u);
        abort_s = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, static_cast<uint32_t>(c.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    griddep_wait();
    griddep_launch_dependents();

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmD);
            mbar_arrive_expect_tx(bar_full,
                                  static_cast<uint32_t>(c.nchunk * (c.a_chunk_bytes + c.b_chunk_bytes)));
            for (int ch = 0; ch < c.nchunk; ++ch) {
                tma_load_4d(smA + ch * c.a_chunk_bytes, &tmQ, bar_full, ch * kChunk, 0, l, tile * c.qpt);
                tma_load_2d(smB + ch * c.b_chunk_bytes, &tmD, bar_full, ch * kChunk, l * p.r);
            }
        }
        __syncwarp();
        ok = __all_sync(0xffffffffu, mbar_wait(bar_full, 0, abort_flag, status, kWaitLimitNs));
        tc_fence_after();
        if (ok && lane == 0) {
            const uint32_t idesc = umma_idesc(false, kTileRows, p.r);
            const uint32_t a0 = smem_u32(smA), b0 = smem_u32(smB);
            for (int ch = 0; ch < c.nchunk; ++ch) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {      // 4 K steps of 16 bf16 (32 B) per chunk
                    const uint64_t ad = umma_sdesc(a0 + static_cast<uint32_t>(ch * c.a_chunk_bytes + ks * 32), 1024u, 2u);
                    const uint64_t bd = umma_sdesc(b0 + static_cast<uint32_t>(ch * c.b_chunk_bytes + ks * 32), 1024u, 2u);
                    umma_bf16(tmem_base, ad, bd, idesc, (ch | ks) != 0 ? 1u : 0u);
                }
            }
        }
        if (lane == 0)
            umma_commit(bar_mma);   // arrives even when nothing was issued
        __syncwarp();
    }
    // ---------------------------------------------------------------- epilogue
    ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 0, abort_flag, status, kWaitLimitNs)) &&
         *abort_flag == 0;
    tc_fence_after();
    // Two warps per TMEM lane quarter (warp % 4): warp w reads its quarter's
    // rows, columns [half * r/2, (half + 1) * r/2) with half = w / 4, all in
    // one round of loads, so every value is read from TMEM once.
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int hc = p.r / 2;                           // columns per thread (16 ... 128)
    const int n16 = hc / 16;
    const int row = quarter * 32 + lane;              // TMEM lane = tile row
    const int qi = row / p.H;
    const int h = row % p.H;
    const int64_t n = static_cast<int64_t>(tile) * c.qpt + qi;
    const bool live = ok && n < p.N;
    const int64_t orow = (n * p.G + l) * p.H + h;      // output row index
    const uint32_t tcol = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                          static_cast<uint32_t>(half * hc);
    uint32_t v[8][16];
    if (ok) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < n16)
                tmem_ld16(tcol + static_cast<uint32_t>(16 * j), v[j]);
        tmem_ld_wait16(v[0]);
#pragma unroll
        for (int j = 1; j < 8; ++j)
            regs_ready16(v[j]);
    }
    if (p.abs_t == LI_FP8_E4M3) {
        // the row maximum: this thread's half, then the partner warp's
        float amax = 0.f;
        if (ok) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n16) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        amax = fmaxf(amax, fabsf(__uint_as_float(v[j][i])));
                }
        }
        amax_part[half][row] = amax;
        __syncthreads();
        amax = fmaxf(amax_part[0][row], amax_part[1][row]);
        const float inv = amax > 0.f ? 448.f / amax : 0.f;
        if (ok) {
            uint8_t *out = static_cast<uint8_t *>(p.q_abs) + orow * p.r + half * hc;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < n16) {
                    uint32_t packed[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                            make_float2(__uint_as_float(v[j][4 * i]) * inv, __uint_as_float(v[j][4 * i + 1]) * inv),
                            __NV_SATFINITE, __NV_E4M3);
                        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                            make_float2(__uint_as_float(v[j][4 * i + 2]) * inv, __uint_as_float(v[j][4 * i + 3]) * inv),
                            __NV_SATFINITE, __NV_E4M3);
                        packed[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
                    }
                    if (live)
                        reinterpret_cast<uint4 *>(out)[j] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                }
            if (live && half == 0)
                p.q_abs_scale[orow] = amax / 448.f;
        }
    } else if (ok && p.abs_t == LI_BF16) {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.q_abs) + orow * p.r + half * hc;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < n16) {
                uint32_t packed[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const __nv_bfloat162 b2 =
                        __floats2bfloat162_rn(__uint_as_float(v[j][2 * i]), __uint_as_float(v[j][2 * i + 1]));
                    packed[i] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                if (live) {
                    uint4 *o4 = reinterpret_cast<uint4 *>(out + 16 * j);
                    o4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                    o4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                }
            }
    } else if (ok) {
        float *out = static_cast<float *>(p.q_abs) + orow * p.r + half * hc;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < n16 && live) {
                uint4 *o4 = reinterpret_cast<uint4 *>(out + 16 * j);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o4[i] = make_uint4(v[j][4 * i], v[j][4 * i + 1], v[j][4 * i + 2], v[j][4 * i + 3]);
            }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(c.tmem_cols));
    }
}

bool make_cfg(const AbsorbParams &p, AbsTcCfg &c, int &smem)
{
    c.qpt = kTileRows / p.H;
    c.nchunk = p.d / kChunk;
    c.a_chunk_bytes = kTileRows * kChunk * 2;
    c.b_chunk_bytes = p.r * kChunk * 2;
    c.off_b = c.nchunk * c.a_chunk_bytes;
    c.off_bar = c.off_b + ((c.nchunk * c.b_chunk_bytes + 1023) & ~1023);
    int cols = 32;
    while (cols < p.r)
        cols <<= 1;
    c.tmem_cols = cols;
    smem = c.off_bar + 16 + 1024;
    return smem <= 227 * 1024 - 2048;   // the kernel's static shared memory comes on top
}

} // namespace

bool absorb_tc_supported(const AbsorbParams &p)
{
    if (p.D == nullptr || p.q_t != LI_BF16 || p.D_t != LI_BF16)
        return false;
    if (p.d % kChunk != 0 || p.d > 256 || p.r % 32 != 0 || p.r < 32 || p.r > 256)
        return false;
    if (p.H != 16 && p.H != 32 && p.H != 64 && p.H != 128)
        return false;
    if (p.G > 65535 || static_cast<int64_t>(p.N) * p.G * p.H > 0x7FFFFFFFll)
        return false;
    AbsTcCfg c;
    int smem = 0;
    return make_cfg(p, c, smem) && encode_fn() != nullptr;
}

cudaError_t launch_absorb_tc(const AbsorbParams &p, cudaStream_t s)
{
    AbsTcCfg c;
    int smem = 0;
    if (!make_cfg(p, c, smem))
        return cudaErrorInvalidValue;
    EncodeTiledFn enc = encode_fn();
    int *status = device_status_ptr();
    if (enc == nullptr || status == nullptr)
        return cudaErrorNotSupported;
    CUtensorMap tmQ, tmD;
    // q [N][G][H][d] as a 4D map {d, H, G, N}; box {64, H, 1, 128 / H}
    {
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.H),
                              static_cast<cuuint64_t>(p.G), static_cast<cuuint64_t>(p.N)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.d) * 2, static_cast<cuuint64_t>(p.H) * p.d * 2,
                                 static_cast<cuuint64_t>(p.G) * p.H * p.d * 2};
        cuuint32_t box[4] = {kChunk, static_cast<cuuint32_t>(p.H), 1, static_cast<cuuint32_t>(c.qpt)};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p.q), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // D [G][r][d] as a 2D map {d, G*r}; box {64, r}
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.G) * p.r};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.d) * 2};
        cuuint32_t box[2] = {kChunk, static_cast<cuuint32_t>(p.r)};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.D), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // The attribute covers the dynamic part only (the kernel also has a few
    // bytes of static shared memory), so it is raised to what this launch
    // needs, never to the whole 227 KB.
    static std::atomic<int> attr_bytes[kMaxDev];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDev)
        dev = 0;
    if (attr_bytes[dev].load(std::memory_order_relaxed) < smem) {
        cudaError_t e = cudaFuncSetAttribute(absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_bytes[dev].store(smem, std::memory_order_relaxed);
    }
    const int64_t tiles = (static_cast<int64_t>(p.N) + c.qpt - 1) / c.qpt;
    if (tiles > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(p.G));
    return launch_pdl(absorb_tc_kernel, grid, dim3(kThreads), static_cast<size_t>(smem), s, tmQ, tmD, p, c,
                      status);
}

} // namespace li
